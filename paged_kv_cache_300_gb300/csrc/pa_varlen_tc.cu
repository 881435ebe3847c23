// bf16 varlen attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// What it computes: "Perhatian berhalaman" (HF transformers docs), section
// "Jalur Varlen": packed requests located by cu_seq_lens_q / cu_seq_lens_k;
// query i of request r (lengths ql, kl) attends key j (j <= i + kl - ql when
// causal), softmax(q k^T * scale) v; a query with no visible key gives 0.
//
// One CTA per (group of `pack` query heads, 128-row tile, request).  The
// rows of a tile are (query, head) pairs, query-major: the `pack` heads of one
// GQA group (the largest power of two dividing the group size) times
// 128 / pack consecutive queries, loaded by one 4-D TMA box per 64-dim half
// (the heads of a query are adjacent in memory).  All rows of a tile use the
// same kv head, so every K/V tile feeds 128 rows, while the ragged last tile
// of a request and the causal diagonal band shrink by `pack`.  grid.x runs
// over the head groups so the CTAs of one GQA group run side by side.  Tiles
// are issued from the last (most keys under the causal mask) to the first.
//
// Warp roles (192 threads, 256 for paged keys; two CTAs share an SM, 103 KB
// of shared memory and 256 TMEM columns each, so one CTA's softmax overlaps
// the other's MMAs):
//   warps 0-3  softmax: thread r owns query row r of the tile, which is TMEM
//              lane r.  It reads its row of S_j from TMEM, masks, keeps the
//              running max/sum in registers (exp2 domain), writes P_j as bf16
//              pairs back over the first half of its S_j row (the tensor core
//              reads it from there as the A operand), rescales its row of O in
//              TMEM when the running max grew by more than 2^8 (lazy rescale:
//              P is then computed against a max up to 8 below the true one,
//              which the final division by the same running sum cancels
//              exactly), and in the end divides O by the sum and stores the row.
//   warp 4     TMA producers: lane 0 loads the Q tile (128 rows) once.
//              Contiguous keys: lane 0 loads the K tiles of 64 keys (two 64-dim
//              swizzled boxes each) and lane 1 the V tiles, into one ring whose
//              stage i % 2 holds {V_(i-1), K_(i+1)} as a single TMA transaction
//              (see NSTAGE below).  Paged keys: the same ring, but a tile is
//              one box per pool block and 64-dim half, and warps 4, 6 and 7
//              (4 and 6 for blocks of 32 or 64 keys) share each transaction's
//              boxes, one box per lane.
//   warp 5     TMEM allocator and MMA issuer (one thread): S_j = Q K_j^T into
//              one of two TMEM S buffers (M=128, N=64, K=16 per instruction,
//              both operands K-major from shared memory), then O += P_j V_j
//              (M=128, N=128) with P_j from TMEM and V read MN-major straight
//              from its TMA tile; tcgen05.commit signals the mbarriers.  S_0
//              and S_1 are issued first, then S_{j+2} right after PV_j, so
//              S_{j+1} is ready while the softmax warps work on S_j.
//
// TMEM: columns [0,64) and [64,128) hold the two S (then P) buffers,
// [128,256) O.  Every mbarrier wait is bounded; on timeout the kernel flags
// PA_DEVERR_TIMEOUT, frees its TMEM and returns.
#include "pa_common.cuh"
#include "pa_internal.h"

#include <math.h>

namespace pa {
namespace {

constexpr int BM = kVarlenQRows;              // query rows per tile (TMEM lanes)
constexpr int BN = kVarlenKRows;              // keys per tile
constexpr int HD = 128;                       // head_dim
constexpr int QBOX = BM * 128;                // 128 rows x 64 dims bf16, 128-byte swizzled
constexpr int KBOX = BN * 128;                // 64 keys x 64 dims
constexpr int Q_BYTES = 2 * QBOX;             // the query tile: two 64-dim boxes
constexpr int KV_BYTES = 2 * KBOX;            // one K (or V) tile of 64 keys
// Key/value ring: stage i % 2 holds transaction T_i, T_0 = {K_0, K_1} and
// T_i = {V_(i-1), K_(i+1)} for i >= 1: the V tile of P V_(i-1) and the K tile
// of S_(i+1), which the MMA thread issues back to back.  One transaction of
// two tiles instead of one per tile halves the TMA transactions per key (a
// TMA transaction costs a few hundred cycles whatever its size, and the
// per-tile rings kept the SM's TMA unit busy all the time; giving V its own
// barrier in the same ring measured 4.6% slower on the prefill workload).
// Paged keys use the same transactions, each filled by two or three warps
// that issue in parallel, one box per lane (one warp issuing all 16 boxes at
// block size 16 measured 0.79 ms against 0.68 ms for two; a K ring and a V
// ring, each with its own warp and barriers, measured 1.5% slower at block
// size 16 and 4.1% at block size 64).
constexpr int NSTAGE = 2;
constexpr int STAGE_BYTES = 2 * KV_BYTES;     // slot A (V, or K_0) + slot B (K)
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + Q_BYTES;
constexpr int OFF_BAR = OFF_KV + NSTAGE * STAGE_BYTES;
constexpr int TAB_CAP = 512;                  // block-table entries staged in smem (paged)
constexpr int OFF_TAB = OFF_BAR + 256;
// three staged copies of the table slice (one per loader warp), + alignment
// slack: still two CTAs per SM
constexpr int SMEM_BYTES = OFF_TAB + 3 * 4 * TAB_CAP + 1024;
// warps 0-3 softmax, 4 TMA (Q + K; contiguous keys: V too), 5 MMA; paged
// keys: warps 6 and 7 issue TMA boxes too, in parallel with warp 4 (a ninth
// warp would cap the kernel below the registers the softmax needs at two
// CTAs per SM)
template <bool PAGED> constexpr int kThreads = PAGED ? 256 : 192;

// Paged keys: the loader warps that share a transaction's boxes.  A warp
// issues its lanes' boxes one after another, so with small blocks more warps
// issue faster: 3 warps against 2 measured 0.690 -> 0.635 ms at block size 8
// and 0.605 -> 0.602 at 16 on the prefill workload, but 0.582 -> 0.584 at 64.
__device__ __forceinline__ int paged_loaders(int block_size) { return block_size <= 16 ? 3 : 2; }
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_O = 2 * BN;
constexpr float kRescaleThreshold = 8.0f; // log2 units

struct Barriers {
    uint64_t q_full;
    uint64_t kv_full[NSTAGE];  // transaction T_i in stage i % 2 (paged keys: both loader warps arrive)
    uint64_t kv_empty[NSTAGE];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done;   // one phase per PV_j (waited only before an O rescale)
    uint64_t all_done; // one phase: every MMA of the CTA has completed
    uint64_t o_staged; // one phase: the four softmax warps wrote the output tile to smem
    uint32_t tmem_base;
    int bad_block; // paged variant: a needed table entry was not a valid block
};

__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk, uint32_t box_bytes)
{
    // kk-th 16-element slice of the reduction dimension inside a K-major tile
    // made of 64-element boxes of `box_bytes`: box kk / 4, 32 bytes per slice
    // inside a 128-byte row; 8-row groups are 1024 bytes apart.
    return umma_desc_sw128(tile + (uint32_t)(kk >> 2) * box_bytes + (uint32_t)(kk & 3) * 32u, 16u,
                           1024u);
}

__device__ __forceinline__ uint64_t v_desc(uint32_t tile, int kk)
{
    // V tile [64 keys][128 dims] read as the MN-major B operand (N = dims):
    // 16 keys per instruction = two 8-row groups (SBO 1024 B); the second
    // 64-dim box is LBO = KBOX bytes away.
    return umma_desc_sw128(tile + (uint32_t)kk * 2048u, (uint32_t)KBOX, 1024u);
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {

// Loads contiguous key/value tile j (64 keys, both 64-dim halves: one box
// each, at row k0 + 64 j of the packed tensor) into `dst`.
__device__ __forceinline__ void load_kv_tile(uint32_t dst, const CUtensorMap *map, uint64_t *full,
                                             int kvh, int k0, int j)
{
    for (int c = 0; c < 2; ++c) tma_load_3d(dst + c * KBOX, map, full, 0, kvh * 2 + c, k0 + j * BN);
}

template <bool PAGED>
__global__ void __launch_bounds__(kThreads<PAGED>, 2)
    varlen_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const VarlenArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers *bar = reinterpret_cast<Barriers *>(smem + OFF_BAR);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // tile rows are (query, head) pairs, query-major: `pack` query heads of
    // one GQA group times QPT consecutive queries
    const int pack = a.pack, QPT = BM / pack;
    const int h0 = blockIdx.x * pack, b = blockIdx.z;
    const int m = gridDim.y - 1 - blockIdx.y; // heavy (late) tiles first
    const int G = a.num_heads / a.num_kv_heads, kvh = h0 / G;

    // Paged keys: the loader warps read the first 32 entries of the
    // request's table row now, alongside the length loads below, so that the
    // first tiles' boxes do not wait for a table round trip of their own.
    int tab_head = -1;
    if (PAGED && (warp == 4 || warp >= 6) && lane < a.max_blocks_per_seq)
        tab_head = __ldg(a.block_table + (size_t)b * a.max_blocks_per_seq + lane);

    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    int k0 = 0, kl = 0;
    bool bad_cu = q0 < 0 || q1 < q0 || q1 > a.total_q || q1 - q0 > (int)gridDim.y * QPT;
    if constexpr (PAGED) {
        kl = __ldg(a.seqlens_k + b);
        if (kl < 0 || (long long)kl > (long long)a.max_blocks_per_seq * a.block_size) {
            if (tid == 0 && h0 == 0 && m == 0) flag_error(a.dev_err, PA_DEVERR_OVERFLOW);
            kl = 0; // no keys: the rows below come out as zeros
        }
    } else {
        k0 = __ldg(a.cu_k + b);
        const int k1 = __ldg(a.cu_k + b + 1);
        bad_cu |= k0 < 0 || k1 < k0 || k1 > a.total_k;
        kl = k1 - k0;
    }
    if (bad_cu) {
        if (tid == 0 && h0 == 0 && m == 0) flag_error(a.dev_err, PA_DEVERR_BAD_CU);
        return;
    }
    const int ql = q1 - q0;
    const int r0 = m * QPT; // first query of the tile inside the request
    if (r0 >= ql) return;
    const int qrows = min(QPT, ql - r0);
    const int rows_here = qrows * pack; // valid tile rows
    int n_keys = kl;
    if (a.causal) n_keys = max(0, min(kl, r0 + qrows - 1 + kl - ql + 1));
    const int n_tiles = (n_keys + BN - 1) / BN;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
    // output row of tile row r
    auto out_row = [&](int r) -> size_t {
        return ((size_t)(q0 + r0 + r / pack) * a.num_heads + h0 + r % pack) * HD;
    };

    if (n_tiles == 0) { // no visible key for any row of the tile
        if (tid < rows_here) {
            uint4 *o = reinterpret_cast<uint4 *>(out + out_row(tid));
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        return;
    }

    // The K loader sets up the barriers of its first loads itself and issues
    // them now (Q and T_0 = {K_0, K_1}), so that their latency overlaps the
    // TMEM allocation and the block-wide barrier below; every other thread
    // touches those barriers only after that barrier.  Paged keys: the whole
    // warp issues T_0's boxes, one per lane, each reading its pool block from
    // the table entries read at entry (T_0 issued after the barrier reached
    // the MMA thread ~700 cycles later per CTA at block size 64, ~1300 at 16).
    const bool k_lane = warp == 4 && lane == 0;
    if (warp == 4) {
        if (k_lane) {
            mbar_init(&bar->q_full, 1);
            for (int s = 0; s < NSTAGE; ++s) mbar_init(&bar->kv_full[s], PAGED ? paged_loaders(a.block_size) : 1);
            bar->bad_block = 0;
            fence_mbar_init();
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            mbar_arrive_expect_tx(&bar->q_full, Q_BYTES);
            for (int c = 0; c < 2; ++c)
                tma_load_4d(sbase + OFF_Q + c * QBOX, &tm_q, &bar->q_full, 0, c, h0, q0 + r0);
            mbar_arrive_expect_tx(&bar->kv_full[0], min(2, n_tiles) * KV_BYTES);
            if constexpr (!PAGED)
                for (int t = 0; t < min(2, n_tiles); ++t)
                    load_kv_tile(sbase + OFF_KV + t * KV_BYTES, &tm_k, &bar->kv_full[0], kvh, k0, t);
        }
        if constexpr (PAGED) {
            // lane 2 i + c (+ one tile's boxes for K_1): the 64-dim half c of
            // pool block i of the tile; entry e < 2 * (64 / block_size) <= 16
            const int bpt = BN / a.block_size, nbox = 2 * bpt;
            const int tt = lane / nbox, rem = lane % nbox, blk = rem >> 1, c = rem & 1;
            const int e = tt * bpt + blk;
            const int p = __shfl_sync(0xffffffffu, tab_head, e & 31);
            __syncwarp(); // the barrier init and the byte count come first
            if (tt < min(2, n_tiles)) {
                int row = a.num_blocks * a.block_size; // past the keys: zero fill
                if (e * a.block_size < kl) {
                    if (p >= 0 && p < a.num_blocks)
                        row = p * a.block_size;
                    else
                        bar->bad_block = 1;
                }
                tma_load_3d(sbase + OFF_KV + tt * KV_BYTES + c * KBOX + blk * a.block_size * 128, &tm_k,
                            &bar->kv_full[0], 0, kvh * 2 + c, row);
            }
        }
    }
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bar->kv_empty[s], 1);
        mbar_init(&bar->s_full[0], 1);
        mbar_init(&bar->s_full[1], 1);
        mbar_init(&bar->p_full[0], 4);
        mbar_init(&bar->p_full[1], 4);
        mbar_init(&bar->o_done, 1);
        mbar_init(&bar->all_done, 1);
        mbar_init(&bar->o_staged, 4);
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(&bar->tmem_base, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bar->tmem_base;
    bool ok = true;

    if (warp == 4 || warp >= 6) {
        // ================= TMA producers =================
        // each loader warp stages its own copy of the table slice
        const int w = warp == 4 ? 0 : warp - 5; // paged keys: loader 0, 1 or 2
        int *tab = reinterpret_cast<int *>(smem + OFF_TAB + w * 4 * TAB_CAP);
        if constexpr (PAGED) {
            // The loader warps fill transaction T_i of the ring above
            // together (warp 4 issued T_0 = {K_0, K_1} alone, before the
            // block-wide barrier): box g of T_i, counting V_(i-1)'s boxes
            // (slot A) and then K_(i+1)'s (slot B), goes to loader g % W,
            // lane g / W.  A tile has one box per pool block and 64-dim half:
            // box 2 i + c of a tile loads the 64-dim half c of its block i.
            // Each warp announces its own boxes' bytes, so the barrier takes
            // W arrivals a phase.  With 2 KB boxes (block size 16) a single
            // issuing thread, not the TMA unit, set the loaders' pace
            // (prefill workload: 0.92 -> 0.68 ms with one box per lane).
            const int W = paged_loaders(a.block_size);
            if (w < W) {
                // T_0 is warp 4's alone: the others' arrivals on it come
                // first, ahead of the table reads (arriving after the table
                // staging put its latency before T_0: ~750 cycles of MMA
                // wait per CTA at block size 16 against ~290 for contiguous
                // keys)
                if (w > 0 && lane == 0) mbar_arrive(&bar->kv_full[0]);
                if (w == 1 && lane == 0) prefetch_tmap(&tm_v);
                const int bpt = BN / a.block_size, nbox = 2 * bpt;
                // The table slice this CTA reads: the first 32 entries were
                // read at entry and cover the boxes of T_0 and T_1 (at most 3
                // tiles = 24 blocks of 8 keys); the rest is staged while those
                // load.  (Staging pool rows, validated once, instead of block
                // ids measured 0.4-1% slower.)
                const int need = min(TAB_CAP, (min(kl, n_tiles * BN) + a.block_size - 1) / a.block_size);
                if (lane < need) tab[lane] = tab_head;
                __syncwarp();
                // This lane's box g: half c of block blk of the V tile
                // (tt = 0, V_(i-1), slot A) or of the K tile (tt = 1,
                // K_(i+1), slot B), landing at its row offset inside the tile
                // (a multiple of 8 rows, so the 128-byte swizzle phase is the
                // same as for a packed tile).  Its table entry at step i is
                // e0 + i bpt; a V box loads at every step, a K box while
                // K_(i+1) exists (i < ilim).
                const int g = lane * W + w;
                const bool gv = g < 2 * nbox;
                const int tt = g / nbox, rem = g % nbox, blk = rem >> 1, c = rem & 1;
                const CUtensorMap *map = tt == 0 ? &tm_v : &tm_k;
                const uint32_t dst0 = sbase + OFF_KV + tt * KV_BYTES + c * KBOX + blk * a.block_size * 128;
                const int e0 = tt == 0 ? blk - bpt : blk + bpt;
                const int ilim = tt == 0 ? n_tiles + 1 : n_tiles - 1;
                const int nblk = (kl + a.block_size - 1) / a.block_size; // entries holding keys
                // a row past the end of the pool: its box reads the TMA's zero fill
                const int oob = a.num_blocks * a.block_size;
                const int vbytes = __popc(__ballot_sync(0xffffffffu, gv && tt == 0)) * a.block_size * 128;
                const int kbytes = __popc(__ballot_sync(0xffffffffu, gv && tt == 1)) * a.block_size * 128;
                for (int i = 1; i <= n_tiles; ++i) {
                    const int st = i & 1;
                    if (i == NSTAGE) {
                        for (int e = 32 + lane; e < need; e += 32)
                            tab[e] = __ldg(a.block_table + (size_t)b * a.max_blocks_per_seq + e);
                        __syncwarp();
                    }
                    // The box's pool row.  Entries past the request's keys
                    // load zeros; a needed entry that is not a valid block is
                    // flagged and loads zeros.  A loaded tile's entries below
                    // TAB_CAP are all staged; later ones come from the table.
                    const int e = e0 + i * bpt;
                    const bool mine = gv && i < ilim;
                    int row = oob;
                    if (mine && e < nblk) {
                        const int p = e < TAB_CAP ? tab[e]
                                                  : __ldg(a.block_table + (size_t)b * a.max_blocks_per_seq + e);
                        if ((unsigned)p < (unsigned)a.num_blocks)
                            row = p * a.block_size;
                        else
                            bar->bad_block = 1;
                    }
                    int go = 1;
                    if (i >= NSTAGE && lane == 0) go = mbar_wait(&bar->kv_empty[st], ((i >> 1) - 1) & 1);
                    if (!__shfl_sync(0xffffffffu, go, 0)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0)
                        mbar_arrive_expect_tx(&bar->kv_full[st], vbytes + (i + 1 < n_tiles ? kbytes : 0));
                    __syncwarp();
                    if (mine) tma_load_3d(dst0 + st * STAGE_BYTES, map, &bar->kv_full[st], 0, kvh * 2 + c, row);
                }
            }
        } else {
            // Contiguous keys: two threads load, one the K tiles (it announces
            // each transaction's bytes, V included), the other the V tiles, so
            // that neither waits behind the other's issue loop.
            const bool v_lane = warp == 4 && lane == 1;
            if (v_lane) prefetch_tmap(&tm_v);
            if (k_lane || v_lane) {
                // T_0 went out before the block-wide barrier
                for (int i = k_lane ? 1 : 0; i <= n_tiles; ++i) {
                    const int st = i & 1;
                    // T_i's stage frees when the MMAs reading T_(i-2) are done
                    if (i >= NSTAGE && !mbar_wait(&bar->kv_empty[st], ((i >> 1) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t slot_a = sbase + OFF_KV + st * STAGE_BYTES;
                    const uint32_t slot_b = slot_a + KV_BYTES;
                    if (k_lane) {
                        // announces the whole transaction: K tile and V tile
                        const int kb = i + 1; // K tile in slot B
                        const int tiles = 1 + (kb < n_tiles ? 1 : 0);
                        mbar_arrive_expect_tx(&bar->kv_full[st], tiles * KV_BYTES);
                        if (kb < n_tiles) load_kv_tile(slot_b, &tm_k, &bar->kv_full[st], kvh, k0, kb);
                    } else if (i >= 1) {
                        load_kv_tile(slot_a, &tm_v, &bar->kv_full[st], kvh, k0, i - 1);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 5) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, BN, 0, 0);
            constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, HD, 0, 1);
            const uint32_t qs = sbase + OFF_Q;
            ok = mbar_wait(&bar->q_full, 0);
            // S_j = Q K_j^T into S buffer j % 2, K_j read from `ks`
            auto issue_qk = [&](int j, uint32_t ks) {
                const int sb = j & 1;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    umma_bf16(tmem + sb * BN, kmajor_desc(qs, kk, QBOX), kmajor_desc(ks, kk, KBOX),
                              idesc_qk, kk > 0);
                umma_commit(&bar->s_full[sb]);
            };
            // S_0 and S_1 (both from T_0) go first; afterwards P V_j and
            // S_(j+2), both from T_(j+1), go back to back (P V_j reads P_j
            // from the TMEM columns that S_(j+2) overwrites; the tensor pipe
            // executes one thread's MMAs in order)
            if (ok) ok = mbar_wait(&bar->kv_full[0], 0);
            if (ok) {
                tc_fence_after();
                issue_qk(0, sbase + OFF_KV);
                if (n_tiles > 1) issue_qk(1, sbase + OFF_KV + KV_BYTES);
                umma_commit(&bar->kv_empty[0]);
            }
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int sb = j & 1, i = j + 1, st = i & 1;
                if (!mbar_wait(&bar->p_full[sb], (j >> 1) & 1) ||
                    !mbar_wait(&bar->kv_full[st], (i >> 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // P_j (bf16, 32 columns) overwrote the first half of S_j in TMEM
                const uint32_t pt = tmem + sb * BN;
                const uint32_t vs = sbase + OFF_KV + st * STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_bf16_tmem_a(tmem + COL_O, pt + kk * 8, v_desc(vs, kk), idesc_pv,
                                     (j > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bar->o_done);
                if (j + 2 < n_tiles) issue_qk(j + 2, vs + KV_BYTES);
                umma_commit(&bar->kv_empty[st]);
            }
            if (ok) umma_commit(&bar->all_done); // tracks every MMA issued above
            // and the last o_done arrival lands before the CTA leaves (every
            // MMA is complete once all_done is, so the parity is unambiguous)
            if (ok) ok = mbar_wait(&bar->all_done, 0) && mbar_wait(&bar->o_done, (n_tiles - 1) & 1);
            // the loaders never wait for the last two stage releases: wait
            // here so that no commit arrives after the CTA has left
            for (int t = max(0, n_tiles - 1); t <= n_tiles && ok; ++t)
                ok = mbar_wait(&bar->kv_empty[t & 1], (t >> 1) & 1);
        }
        __syncwarp();
    } else {
        // ================= softmax: thread r <-> query row r =================
        const int r = tid;
        const int i = r0 + r / pack; // query of this row inside the request
        const int lim = a.causal ? min(i + kl - ql, kl - 1) : kl - 1; // last visible key
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float sl2 = a.scale_log2;
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            if (!mbar_wait(&bar->s_full[st], (j >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
                tmem_ld32(trow + st * BN + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
            tmem_ld_wait();
            const int kb = j * BN;
            if (kb + BN - 1 > lim) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (kb + c > lim) s[c] = -INFINITY;
            }
            // row max as 8 independent chains (short critical path; four
            // chains of the three-input max measured slower)
            float mx8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx8[u] = s[u];
#pragma unroll
            for (int c = 8; c < BN; c += 8)
#pragma unroll
                for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(mx8[u], s[c + u]);
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
            // the scale-and-offset and the running sums take the paired fp32
            // instructions (two lanes of arithmetic per instruction): the
            // softmax phase is issue-bound, not bound by the exponentials
            const float2 sl2x2 = make_float2(sl2, sl2), nmu = make_float2(-mu, -mu);
            float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}; // 4 partial sums
            uint32_t pk[BN / 2];
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2x2, nmu);
                const float p0 = exp2_approx(x.x), p1 = exp2_approx(x.y);
                sum2[(c >> 1) & 1] = __fadd2_rn(sum2[(c >> 1) & 1], make_float2(p0, p1));
                pk[c >> 1] = pack_bf16(p0, p1);
            }
            const float sum = (sum2[0].x + sum2[1].x) + (sum2[0].y + sum2[1].y);
            l_run = l_run * alpha + sum;
            // P row (bf16 pairs) over the S_j row it came from; PV_j reads it
            // as the TMEM A operand.  Its own buffer: no wait on PV_{j-1}.
            tmem_st32(trow + st * BN, pk);
            // The key tile that holds the request's last key also holds rows
            // that are not keys of this request: the unwritten tail of a pool
            // block (paged keys; any bits at all, NaN included) or the next
            // request's rows.  Their weights are 0, but the tensor core
            // multiplies 0 by whatever is there and 0 * NaN is NaN, so their
            // V rows are zeroed before P V_j may start (rows whose whole block
            // lies past the keys were zero-filled by the TMA already).
            if (j == n_tiles - 1 && kl - kb < BN) {
                const int z0 = kl - kb;
                const int z1 = PAGED ? min(BN, (kl + a.block_size - 1) / a.block_size * a.block_size - kb)
                                     : BN;
                const int ti = j + 1; // V_j travels in transaction T_(j+1)
                uint64_t *vbar = &bar->kv_full[ti & 1];
                const uint32_t vpar = (ti >> 1) & 1;
                uint8_t *vt = smem + OFF_KV + (ti & 1) * STAGE_BYTES;
                if (z1 > z0) {
                    if (!mbar_wait(vbar, vpar)) {
                        ok = false;
                        break;
                    }
                    const int per_half = (z1 - z0) * 8; // 16-byte chunks per 64-dim half
                    for (int c = r; c < 2 * per_half; c += BM) {
                        const int hf = c / per_half, rem = c % per_half;
                        *reinterpret_cast<uint4 *>(vt + hf * KBOX + (z0 + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
            }
            // O is rescaled only by a warp with a row whose max grew past the
            // threshold, after PV_{j-1} is done and before PV_j (which needs
            // this warp's arrival).  Otherwise P_j is released at once and
            // PV_j queues behind PV_{j-1} without a round trip.
            // (S_j being ready implies PV_{j-2} is done -- its commit covers
            // every earlier MMA -- so o_done is at most one phase behind and
            // its parity is unambiguous)
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                if (!mbar_wait(&bar->o_done, (j - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
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
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->p_full[st]);
        }
        // two PVs may still be in flight here, so the epilogue waits on the
        // single-phase barrier committed after the last one
        if (ok && mbar_wait(&bar->all_done, 0)) {
            tc_fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            if (a.out_tma && rows_here == BM) {
                // A full tile leaves through the TMA: every thread writes its
                // bf16 row into the Q buffer (no MMA reads it any more) in
                // the layout the Q load used, and one thread stores the two
                // 64-dim boxes.  Thread stores of 16-byte pieces of 128
                // different rows took ~1.5 us of the ~1.8 us epilogue.
                uint8_t *qs = smem + OFF_Q;
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(trow + COL_O + c * 32, o);
                    tmem_ld_wait();
                    uint8_t *box = qs + (c >> 1) * QBOX + r * 128;
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        const int chunk = ((c & 1) * 32 + e) >> 3; // 16-byte chunk in the 128-byte row
                        *reinterpret_cast<uint4 *>(box + ((chunk ^ (r & 7)) << 4)) = make_uint4(
                            pack_bf16(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                            pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                            pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                            pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->o_staged);
                if (r == 0) {
                    if (mbar_wait(&bar->o_staged, 0)) {
                        for (int c = 0; c < 2; ++c)
                            tma_store_4d(&tm_o, sbase + OFF_Q + c * QBOX, 0, c, h0, q0 + r0);
                        bulk_commit();
                        bulk_wait_read(); // the Q buffer is read before the CTA leaves
                    } else {
                        ok = false;
                    }
                }
            } else {
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
            }
        } else {
            ok = false;
        }
    }
    if (!ok) flag_error(a.dev_err, PA_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, TMEM_COLS);
    if constexpr (PAGED) {
        // a needed block was missing: flag it and zero the tile's rows (after
        // the tile's TMA store, if it took one, has written them: thread 0
        // issued it)
        if (bar->bad_block) {
            if (tid == 0) {
                flag_error(a.dev_err, PA_DEVERR_BAD_BLOCK);
                bulk_wait_all_global();
            }
            __syncthreads();
            if (tid < rows_here) {
                uint4 *o = reinterpret_cast<uint4 *>(out + out_row(tid));
                for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
}

template <bool PAGED>
int launch_varlen(const VarlenArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                  const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t s)
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
        if (cudaFuncSetAttribute(varlen_tc_kernel<PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return PA_ERR_LAUNCH;
        __atomic_store_n(&attr_set[dev], 1, __ATOMIC_RELEASE);
    }
    const int qpt = BM / a.pack;
    const unsigned tiles = (unsigned)((a.max_q + qpt - 1) / qpt);
    if (tiles > 65535u || a.batch > 65535) return PA_ERR_UNSUPPORTED;
    dim3 grid((unsigned)(a.num_heads / a.pack), tiles, (unsigned)a.batch);
    varlen_tc_kernel<PAGED><<<grid, kThreads<PAGED>, SMEM_BYTES, s>>>(tm_q, tm_k, tm_v, tm_o, a);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

}  // namespace

int varlen_bf16_launch(const VarlenArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                       const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t s)
{
    return launch_varlen<false>(a, tm_q, tm_k, tm_v, tm_o, s);
}

int varlen_paged_bf16_launch(const VarlenArgs &a, const CUtensorMap &tm_q,
                             const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const CUtensorMap &tm_o, cudaStream_t s)
{
    return launch_varlen<true>(a, tm_q, tm_k, tm_v, tm_o, s);
}

}  // namespace pa
