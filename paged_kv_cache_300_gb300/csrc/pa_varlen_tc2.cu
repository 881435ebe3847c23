// bf16 varlen attention on pairs of SMs: tcgen05.mma.cta_group::2, M = 256.
//
// What it computes: "Perhatian berhalaman" (HF transformers docs), section
// "Jalur Varlen": packed requests located by cu_seq_lens_q / cu_seq_lens_k;
// query i of request r (lengths ql, kl) attends key j (j <= i + kl - ql when
// causal), softmax(q k^T * scale) v; a query with no visible key gives 0.
// With PAGED the keys of request r are its positions 0..kl-1 read through
// block_table row r from the pool ("Jalur Varlen" -> "Perilaku cache";
// "39 · PagedAttention", "Ghi chú": attention kernels can take the table).
//
// Work item: one cluster of two CTAs per (group of `pack` query heads, tile
// of 256 rows, request).  Rows are (query, head) pairs, query-major: the
// `pack` heads of one GQA group times 256 / pack consecutive queries; CTA
// rank c of the pair owns rows [128 c, 128 c + 128), i.e. queries
// [c 128/pack, (c+1) 128/pack) of the tile.  All rows use the same kv head.
//
// The pair computes, per tile of 128 keys,
//   S = Q K^T   (M = 256, N = 128, K = 128): each CTA holds its 128 rows of Q
//               and 64 of the 128 keys of K (CTA c: keys 64 c .. 64 c + 63),
//               both K-major; each CTA's tensor memory receives its 128 rows
//               x 128 key columns of S;
//   O += P V    (M = 256, N = 128 dims, K = 128 keys): P from each CTA's
//               tensor memory (its rows), V split by dims: CTA c holds the
//               64-dim half c of all 128 keys (MN-major); each CTA's O holds
//               its rows x all 128 dims.
// So each SM loads 16 KB of K and 16 KB of V per 128 keys (half of what a
// single-SM M = 128 tile with the same keys needs), and each MMA streams half
// of B from each SM's shared memory.
//
// Warp roles (224 threads, one CTA per SM: 166 KB of shared memory, all 512
// TMEM columns):
//   warps 0-3  softmax, thread r <-> TMEM lane r <-> tile row r.  It reads its
//              row of S_j (128 fp32), masks, keeps the running max / sum
//              (exp2 domain), writes P_j (bf16 pairs) over the first half of
//              the S_j columns, rescales its O row lazily (only when the
//              running max grew by more than 2^8; the final division by the
//              same running sum cancels the stale max exactly) and finally
//              divides O by the sum and stores the row.
//   warp 4     lane 0: TMA loads of this CTA's Q tile, then its K tiles.
//   warp 5     TMEM allocation (both CTAs, collectively).  Even CTA, lane 0:
//              the MMA issuer of the pair.  Odd CTA, lane 0: forwards the
//              arrival of its Q and K tiles to the even CTA's barriers.
//   warp 6     lane 0: TMA loads of this CTA's V tiles.
// The even CTA's MMA thread waits until both CTAs' operands have landed and
// both CTAs' softmax warps have written P; tcgen05.commit with a multicast
// mask signals S-ready, stage-free, O-done and all-done in both CTAs.
//
// TMEM columns: [0,128) S_0, [128,256) S_1 (P over the first 64 of each),
// [256,384) O.  Every mbarrier wait is bounded; after a timeout the kernel
// flags PA_DEVERR_TIMEOUT and still reaches the final cluster barrier, so
// neither CTA of a pair leaves while the other may touch its memory.
#include "pa_common.cuh"
#include "pa_internal.h"

#include <math.h>

namespace pa {
namespace {

constexpr int BM = 128;               // query rows per CTA (TMEM lanes)
constexpr int BN = kVarlenPairKeys;   // keys per S tile (N of the pair)
constexpr int KH = BN / 2;            // keys of a K tile held by one CTA
constexpr int HD = 128;               // head_dim
constexpr int QBOX = BM * 128;        // 128 rows x 64 dims, 128-byte swizzled
constexpr int Q_BYTES = 2 * QBOX;     // the Q tile: two 64-dim boxes
constexpr int KBOX = KH * 128;        // 64 keys x 64 dims
constexpr int K_STAGE = 2 * KBOX;     // this CTA's 64 keys, both 64-dim halves
constexpr int V_STAGE = BN * 128;     // 128 keys x this CTA's 64-dim half
constexpr int NK = 4;                 // K ring stages
constexpr int NV = 4;                 // V ring stages
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + Q_BYTES;
constexpr int OFF_V = OFF_K + NK * K_STAGE;
constexpr int OFF_BAR = OFF_V + NV * V_STAGE;
constexpr int TAB_CAP = 512;          // block-table entries staged in smem (paged)
constexpr int OFF_TAB = OFF_BAR + 512;
constexpr int SMEM_BYTES = OFF_TAB + 2 * 4 * TAB_CAP + 1024;
constexpr int kThreads = 224;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 2 * BN;
constexpr float kRescaleThreshold = 8.0f; // log2 units

struct Barriers {
    uint64_t q_full;        // even CTA: its own load + the odd CTA's forward
    uint64_t k_full[NK];    // likewise
    uint64_t k_empty[NK];   // S_j computed: the K stage may be reloaded
    uint64_t v_full[NV];    // this CTA's V tile landed (local only)
    uint64_t v_empty[NV];   // P V_j computed
    uint64_t s_full[2];
    uint64_t p_full[2];     // even CTA: 4 local + 4 remote softmax warps
    uint64_t o_done;        // one phase per P V_j
    uint64_t all_done;      // one phase: every MMA of the pair completed
    uint32_t tmem_base;
    int bad_block;          // a needed table entry was not a valid block (either CTA)
};
static_assert(sizeof(Barriers) <= 512, "barrier block");

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk, uint32_t box_bytes)
{
    // kk-th 16-element slice of the reduction dimension of a K-major tile made
    // of 64-element boxes of `box_bytes`: box kk / 4, 32 bytes per slice
    // inside a 128-byte row; 8-row groups are 1024 bytes apart
    return umma_desc_sw128(tile + (uint32_t)(kk >> 2) * box_bytes + (uint32_t)(kk & 3) * 32u, 16u,
                           1024u);
}

__device__ __forceinline__ uint64_t v_desc(uint32_t tile, int kk)
{
    // this CTA's V tile [128 keys][64 dims] as its half of the MN-major B
    // operand: 16 keys per instruction = two 8-row groups (SBO 1024 B); the
    // 64 dims are one swizzle atom, so the leading offset is not used
    return umma_desc_sw128(tile + (uint32_t)kk * 2048u, (uint32_t)V_STAGE, 1024u);
}

__device__ __forceinline__ void store_cluster_u32(uint32_t cluster_addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// One TMA box per pool block for `nkeys` keys starting at logical position
// `pos0` (a multiple of block_size), 64-dim half `half`, landing at `dst` in
// rows of 128 bytes.  Blocks whose first position is not below `kl` read
// the zero fill past the end of the pool; a needed entry that is not a
// valid block is flagged (in both CTAs) and read as zero fill.
__device__ __forceinline__ void load_paged_rows(uint32_t dst, const CUtensorMap *map, uint64_t *full,
                                                const VarlenArgs &a, int b, int kvh, int half,
                                                int pos0, int nkeys, int kl, const int *tab,
                                                Barriers *bar, uint32_t peer_bad)
{
    const int bs = a.block_size;
    const int oob = a.num_blocks * bs;
    for (int i = 0; i < nkeys / bs; ++i) {
        const int pos = pos0 + i * bs;
        int row = oob;
        if (pos < kl) {
            const int e = pos / bs;
            const int p = e < TAB_CAP ? tab[e]
                                      : __ldg(a.block_table + (size_t)b * a.max_blocks_per_seq + e);
            if (p >= 0 && p < a.num_blocks) {
                row = p * bs;
            } else {
                bar->bad_block = 1;
                store_cluster_u32(peer_bad, 1u);
            }
        }
        tma_load_3d(dst + i * bs * 128, map, full, 0, kvh * 2 + half, row);
    }
}

template <bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    varlen_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const VarlenArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers *bar = reinterpret_cast<Barriers *>(smem + OFF_BAR);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank(); // 0: issues the MMAs of the pair
    const uint32_t peer = rank ^ 1u;
    const int pack = a.pack, QPT = BM / pack; // queries per CTA tile
    const int h0 = (int)(blockIdx.x >> 1) * pack, b = blockIdx.z;
    const int m = gridDim.y - 1 - blockIdx.y; // heavy (late) tiles first
    const int G = a.num_heads / a.num_kv_heads, kvh = h0 / G;

    // ---- decisions that depend only on the pair's work item: both CTAs of
    // the pair take the same branch, before they touch each other
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    int k0 = 0, kl = 0;
    bool bad_cu = q0 < 0 || q1 < q0 || q1 > a.total_q || q1 - q0 > (int)gridDim.y * 2 * QPT;
    if constexpr (PAGED) {
        kl = __ldg(a.seqlens_k + b);
        if (kl < 0 || (long long)kl > (long long)a.max_blocks_per_seq * a.block_size) {
            if (tid == 0 && rank == 0 && h0 == 0 && m == 0) flag_error(a.dev_err, PA_DEVERR_OVERFLOW);
            kl = 0; // no keys: the rows below come out as zeros
        }
    } else {
        k0 = __ldg(a.cu_k + b);
        const int k1 = __ldg(a.cu_k + b + 1);
        bad_cu |= k0 < 0 || k1 < k0 || k1 > a.total_k;
        kl = k1 - k0;
    }
    if (bad_cu) {
        if (tid == 0 && rank == 0 && h0 == 0 && m == 0) flag_error(a.dev_err, PA_DEVERR_BAD_CU);
        return;
    }
    const int ql = q1 - q0;
    const int rp = m * 2 * QPT; // first query of the pair's tile
    if (rp >= ql) return;
    const int pq = min(2 * QPT, ql - rp);          // queries of the pair's tile
    const int r0 = rp + (int)rank * QPT;          // first query of this CTA's rows
    const int qrows = max(0, min(QPT, ql - r0));  // this CTA's valid queries
    const int rows_here = qrows * pack;
    int n_keys = kl;
    if (a.causal) n_keys = max(0, min(kl, rp + pq - 1 + kl - ql + 1));
    const int n_tiles = (n_keys + BN - 1) / BN;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
    auto out_row = [&](int r) -> size_t {
        return ((size_t)(q0 + r0 + r / pack) * a.num_heads + h0 + r % pack) * HD;
    };
    if (n_tiles == 0) { // no visible key for any row of the pair
        if (tid < rows_here) {
            uint4 *o = reinterpret_cast<uint4 *>(out + out_row(tid));
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        return;
    }

    // ---- set-up: barriers, TMEM (collective over the pair), then a cluster
    // barrier so that every barrier is initialised before the peer uses it
    if (tid == 0) {
        mbar_init(&bar->q_full, rank == 0 ? 2 : 1);
        for (int s = 0; s < NK; ++s) {
            mbar_init(&bar->k_full[s], rank == 0 ? 2 : 1);
            mbar_init(&bar->k_empty[s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&bar->v_full[s], 1);
            mbar_init(&bar->v_empty[s], 1);
        }
        mbar_init(&bar->s_full[0], 1);
        mbar_init(&bar->s_full[1], 1);
        mbar_init(&bar->p_full[0], 8);
        mbar_init(&bar->p_full[1], 8);
        mbar_init(&bar->o_done, 1);
        mbar_init(&bar->all_done, 1);
        bar->bad_block = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem2_alloc(&bar->tmem_base, TMEM_COLS);
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = bar->tmem_base;
    const uint32_t peer_bad = mapa_shared(smem_u32(&bar->bad_block), peer);
    bool ok = true;

    if (warp == 4 || warp == 6) {
        // ================= TMA producers =================
        int *tab = reinterpret_cast<int *>(smem + OFF_TAB + (warp == 6 ? 4 * TAB_CAP : 0));
        if constexpr (PAGED) {
            const int need = min(TAB_CAP, (min(kl, n_tiles * BN) + a.block_size - 1) / a.block_size);
            for (int e = lane; e < need; e += 32)
                tab[e] = __ldg(a.block_table + (size_t)b * a.max_blocks_per_seq + e);
            __syncwarp();
        }
        if (lane == 0) {
            if (warp == 4) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
                mbar_arrive_expect_tx(&bar->q_full, Q_BYTES);
                for (int c = 0; c < 2; ++c)
                    tma_load_4d(sbase + OFF_Q + c * QBOX, &tm_q, &bar->q_full, 0, c, h0, q0 + r0);
                for (int j = 0; j < n_tiles; ++j) {
                    const int st = j % NK;
                    if (j >= NK && !mbar_wait_cluster(&bar->k_empty[st], ((j / NK) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sbase + OFF_K + st * K_STAGE;
                    const int kb = j * BN + (int)rank * KH; // this CTA's 64 keys
                    mbar_arrive_expect_tx(&bar->k_full[st], K_STAGE);
                    for (int c = 0; c < 2; ++c) {
                        if constexpr (PAGED)
                            load_paged_rows(dst + c * KBOX, &tm_k, &bar->k_full[st], a, b, kvh, c, kb,
                                            KH, kl, tab, bar, peer_bad);
                        else
                            tma_load_3d(dst + c * KBOX, &tm_k, &bar->k_full[st], 0, kvh * 2 + c,
                                        k0 + kb);
                    }
                }
            } else {
                prefetch_tmap(&tm_v);
                for (int j = 0; j < n_tiles; ++j) {
                    const int st = j % NV;
                    if (j >= NV && !mbar_wait_cluster(&bar->v_empty[st], ((j / NV) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sbase + OFF_V + st * V_STAGE;
                    mbar_arrive_expect_tx(&bar->v_full[st], V_STAGE);
                    if constexpr (PAGED)
                        load_paged_rows(dst, &tm_v, &bar->v_full[st], a, b, kvh, (int)rank, j * BN,
                                        BN, kl, tab, bar, peer_bad);
                    else
                        tma_load_3d(dst, &tm_v, &bar->v_full[st], 0, kvh * 2 + (int)rank,
                                    k0 + j * BN);
                }
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0 && rank == 0) {
            // ================= MMA issuer of the pair =================
            constexpr uint32_t idesc_qk = umma_idesc_bf16(2 * BM, BN, 0, 0);
            constexpr uint32_t idesc_pv = umma_idesc_bf16(2 * BM, HD, 0, 1);
            const uint32_t qs = sbase + OFF_Q;
            ok = mbar_wait_cluster(&bar->q_full, 0);
            auto issue_qk = [&](int j) -> bool {
                const int st = j % NK, sb = j & 1;
                if (!mbar_wait_cluster(&bar->k_full[st], (j / NK) & 1)) return false;
                tc_fence_after();
                const uint32_t ks = sbase + OFF_K + st * K_STAGE;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    umma2_bf16(tmem + sb * BN, kmajor_desc(qs, kk, QBOX), kmajor_desc(ks, kk, KBOX),
                               idesc_qk, kk > 0);
                umma2_commit_both(&bar->s_full[sb]);
                umma2_commit_both(&bar->k_empty[st]);
                return true;
            };
            // S_0 and S_1 first; then S_(j+2) right after P V_j, which reads
            // P_j from the same columns (the pair's MMAs execute in order)
            if (ok) ok = issue_qk(0);
            if (ok && n_tiles > 1) ok = issue_qk(1);
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int sb = j & 1, sv = j % NV;
                if (!mbar_wait_cluster(&bar->p_full[sb], (j >> 1) & 1) ||
                    !mbar_wait(&bar->v_full[sv], (j / NV) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pt = tmem + sb * BN;
                const uint32_t vs = sbase + OFF_V + sv * V_STAGE;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma2_bf16_tmem_a(tmem + COL_O, pt + kk * 8, v_desc(vs, kk), idesc_pv,
                                      (j > 0 || kk > 0) ? 1u : 0u);
                umma2_commit_both(&bar->o_done);
                umma2_commit_both(&bar->v_empty[sv]);
                if (j + 2 < n_tiles && !(ok = issue_qk(j + 2))) break;
            }
            if (ok) umma2_commit_both(&bar->all_done);
        } else if (lane == 0) {
            // ============ odd CTA: Q and K landed -> the even CTA's barriers
            const uint32_t q_remote = mapa_shared(smem_u32(&bar->q_full), 0);
            ok = mbar_wait(&bar->q_full, 0);
            if (ok) mbar_arrive_cluster(q_remote);
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int st = j % NK;
                if (!mbar_wait(&bar->k_full[st], (j / NK) & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_cluster(mapa_shared(smem_u32(&bar->k_full[st]), 0));
            }
        }
        // before the CTA may leave, every commit arrival addressed to this
        // CTA's barriers has landed: the last phases no loader waits for
        if (lane == 0) {
            if (ok) ok = mbar_wait_cluster(&bar->all_done, 0) &&
                         mbar_wait_cluster(&bar->o_done, (n_tiles - 1) & 1);
            for (int t = max(0, n_tiles - NK); t < n_tiles && ok; ++t)
                ok = mbar_wait_cluster(&bar->k_empty[t % NK], (t / NK) & 1);
            for (int t = max(0, n_tiles - NV); t < n_tiles && ok; ++t)
                ok = mbar_wait_cluster(&bar->v_empty[t % NV], (t / NV) & 1);
        }
        __syncwarp();
    } else {
        // ================= softmax: thread r <-> row r =================
        const int r = tid;
        const int i = r0 + r / pack; // query of this row inside the request
        const int lim = a.causal ? min(i + kl - ql, kl - 1) : kl - 1; // last visible key
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float sl2 = a.scale_log2;
        const uint32_t p_remote0 = mapa_shared(smem_u32(&bar->p_full[0]), 0);
        const uint32_t p_remote1 = mapa_shared(smem_u32(&bar->p_full[1]), 0);
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1, sv = j % NV;
            if (!warp_wait_cluster(&bar->s_full[sb], (j >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int kb = j * BN;
            float sv_[BN];
#pragma unroll
            for (int ch = 0; ch < BN / 32; ++ch)
                tmem_ld32(trow + sb * BN + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv_[ch * 32]));
            tmem_ld_wait();
            if (kb + BN - 1 > lim) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (kb + c > lim) sv_[c] = -INFINITY;
            }
            // row max as 8 independent chains (short critical path)
            float mx8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx8[u] = sv_[u];
#pragma unroll
            for (int c = 8; c < BN; c += 8)
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(mx8[u], sv_[c + u]);
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            const float m_new = fmaxf(m_run, mx * sl2);
            const bool need = m_new > m_run + kRescaleThreshold;
            float alpha = 1.f;
            if (need) {
                alpha = exp2_approx(m_run - m_new);
                m_run = m_new;
            }
            const float mu = m_run == -INFINITY ? 0.f : m_run;
            // P = 2^(s * scale - m) as bf16 pairs over the first half of the
            // S_j columns (every S value is in registers by now)
            float sum4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                const float p0 = exp2_approx(fmaf(sv_[c], sl2, -mu));
                const float p1 = exp2_approx(fmaf(sv_[c + 1], sl2, -mu));
                sum4[(c >> 1) & 3] += p0 + p1;
                pk[c >> 1] = pack_bf16(p0, p1);
            }
            tmem_st32(trow + sb * BN, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
            tmem_st32(trow + sb * BN + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
            l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
            // This CTA's V tile of P V_j must have landed before the pair's
            // MMA may use it (the even CTA's MMA thread sees only its own
            // V barrier; the odd CTA's arrival on p_full carries its V).
            // The tile holding the request's last key also holds rows that
            // are not keys of this request (the unwritten tail of a pool
            // block -- any bits, NaN included -- or the next request's rows):
            // their weights are 0, but 0 * NaN is NaN, so their V rows are
            // zeroed first (rows of blocks wholly past the keys were
            // zero-filled by the TMA).
            const bool tail = j == n_tiles - 1 && kl - kb < BN;
            if (rank == 1 || tail) {
                if (!warp_wait(&bar->v_full[sv], (j / NV) & 1)) {
                    ok = false;
                    break;
                }
            }
            if (tail) {
                const int z0 = kl - kb;
                const int z1 = PAGED ? min(BN, (kl + a.block_size - 1) / a.block_size * a.block_size - kb)
                                     : BN;
                uint8_t *vt = smem + OFF_V + sv * V_STAGE;
                for (int c = r; c < (z1 - z0) * 8; c += BM)
                    *reinterpret_cast<uint4 *>(vt + (z0 + c / 8) * 128 + (c % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
            }
            // O is rescaled only by a warp with a row whose max grew past the
            // threshold, after P V_(j-1) is done and before P V_j (which waits
            // for this warp).  S_j ready implies P V_(j-2) is done, so o_done
            // is at most one phase behind and its parity is unambiguous.
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                if (!warp_wait_cluster(&bar->o_done, (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(trow + COL_O + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(trow + COL_O + c * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0)
                    mbar_arrive(&bar->p_full[sb]);
                else
                    mbar_arrive_cluster(sb ? p_remote1 : p_remote0);
            }
        }
        if (ok && warp_wait_cluster(&bar->all_done, 0)) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            uint4 *orow = reinterpret_cast<uint4 *>(out + out_row(r));
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(trow + COL_O + c * 32, o);
                tmem_ld_wait();
                if (r < rows_here) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        orow[(c * 32 + e) / 8] = make_uint4(
                            pack_bf16(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                            pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                            pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                            pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                }
            }
        } else {
            ok = false;
        }
    }
    if (!ok) flag_error(a.dev_err, PA_DEVERR_TIMEOUT);
    // neither CTA leaves (or frees its tensor memory) while the pair's MMAs,
    // commits or remote arrivals may still reach it
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 5) tmem2_dealloc(tmem, TMEM_COLS);
    if constexpr (PAGED) {
        // a needed block was missing in either CTA's loads: zero the rows
        if (bar->bad_block) {
            if (tid == 0) flag_error(a.dev_err, PA_DEVERR_BAD_BLOCK);
            if (tid < rows_here) {
                uint4 *o = reinterpret_cast<uint4 *>(out + out_row(tid));
                for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
}

template <bool PAGED>
int launch_pair(const VarlenArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                const CUtensorMap &tm_v, cudaStream_t s)
{
    if (a.head_dim != HD) return PA_ERR_UNSUPPORTED;
    if (a.max_q <= 0) return PA_OK;
    // the shared-memory limit is an attribute of the kernel in each device's
    // context: raise it once per device
    constexpr int kMaxDev = 64;
    static int attr_set[kMaxDev] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return PA_ERR_DEVICE;
    if (__atomic_load_n(&attr_set[dev], __ATOMIC_ACQUIRE) == 0) {
        if (cudaFuncSetAttribute(varlen_pair_kernel<PAGED>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return PA_ERR_LAUNCH;
        __atomic_store_n(&attr_set[dev], 1, __ATOMIC_RELEASE);
    }
    const int qpt2 = 2 * BM / a.pack; // queries per pair tile
    const unsigned tiles = (unsigned)((a.max_q + qpt2 - 1) / qpt2);
    if (tiles > 65535u || a.batch > 65535) return PA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)(2 * (a.num_heads / a.pack)), tiles, (unsigned)a.batch);
    varlen_pair_kernel<PAGED><<<grid, kThreads, SMEM_BYTES, s>>>(tm_q, tm_k, tm_v, a);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

}  // namespace

int varlen_pair_bf16_launch(const VarlenArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                            const CUtensorMap &tm_v, cudaStream_t s)
{
    return launch_pair<false>(a, tm_q, tm_k, tm_v, s);
}

int varlen_pair_paged_bf16_launch(const VarlenArgs &a, const CUtensorMap &tm_q,
                                  const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                  cudaStream_t s)
{
    return launch_pair<true>(a, tm_q, tm_k, tm_v, s);
}

}  // namespace pa
