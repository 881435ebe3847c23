// Paged decode attention (one query per sequence) for GB300.
//
// What it computes ("Perhatian berhalaman", HF transformers docs, section
// "Jalur decode"; "39 · PagedAttention", inference-notes, sections 1-3):
// for every sequence b the new token's K/V is written in place at logical
// position L = cache_seqlens[b] (block block_table[b][L / bs], slot L % bs),
// then the query attends over positions 0..L walked in logical order through
// the block table: score per key, one softmax, weighted sum of V.
//
// bf16 design (HBM-bound):
//  * Stream-K over the flattened work list.  A "unit" is one logical block
//    of one sequence for one group of HS kv heads; units are ordered (head
//    group, sequence, logical block) and the persistent grid of P CTAs takes
//    contiguous ranges of about equal cost (a unit, plus a fixed overhead
//    per sequence when most sequences are split; see kSeqCost), so every SM
//    streams about the same number of bytes whatever the length mix.  Every
//    CTA derives the ranges itself from cache_seqlens (block-wide scan), so
//    the host needs no lengths and no device-to-host copy.
//  * A producer warp resolves logical -> physical blocks through the table
//    (32 entries per coalesced load) and issues TMA tensor loads of the K and
//    V tiles of each physical block (one 128-byte-swizzled box per kv head
//    and 64 dims) into a ring of NST shared-memory stages (mbarrier
//    full/empty pairs).  KV bytes are read exactly once.
//  * HS consumer warps, one per kv head.  The GQA group of query heads is
//    packed into the N=8 side of mma.sync m16n8k16: S^T[token, head] = K q^T
//    with K straight from swizzled shared memory (ldmatrix), online softmax
//    in registers (exp2), then O^T[dim, head] += V^T P^T with P moved into
//    the B layout by movmatrix.  Each KV element is touched once by the
//    tensor pipe instead of G times by the FMA pipe.
//  * A sequence split across CTAs leaves partial (acc, m, l) per CTA; the
//    last CTA to finish it (atomic ticket, no spin) merges the partials in
//    logical order with m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m)
//    (inference-notes, "3. Trên GPU"), the accumulator merged with the same
//    weights, then normalises.  Merge order depends only on the lengths, so
//    the output is bitwise independent of the physical block placement.
//  * The CTA that owns a sequence's last block performs the append: it
//    copies k_new/v_new into the pool slot and into its staged tile, so the
//    new token is attended without waiting on its own global write.
//
// fp32 path: one warp per (sequence, query head), CUDA-core FMA with expf;
// kept simple, it serves fp32 inputs (tolerance 1e-5) only.
#include "pa_common.cuh"
#include "pa_internal.h"

#include <math.h>

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int D, int BS, int HS>
struct Geom {
    static constexpr int KB = D / 64;                 // 128-byte boxes per head row
    static constexpr int BOX_BYTES = BS * 128;        // one box: BS rows x 64 dims
    static constexpr int HEAD_BYTES = KB * BOX_BYTES; // one head's K (or V) tile
    static constexpr int KV_BYTES = HS * HEAD_BYTES;  // the K (or V) half of a stage
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int MT = BS / 16; // 16-token m-tiles per block
    static constexpr int KS = D / 16;  // k-steps of QK^T = 16-dim tiles of PV
    static constexpr int THREADS = (HS + 1) * 32;
    static constexpr int NW = HS + 1;
};

// Position of the walk over units (head group, sequence, logical block).
struct SeqWalk {
    int hg, b, j;
    int nblk; // logical blocks of sequence b (>= 1)
    int len;  // cache_seqlens[b], or -1 for an invalid length
    long long sb; // units of sequences 0..b-1 within the head group
};

// Blocks of a sequence with L cached tokens once the new token is appended;
// `cap` is the positions a sequence can hold (the table's blocks times the
// block size, or the rows of a contiguous cache).
__device__ __forceinline__ int seq_blocks(int L, long long cap, int bs, bool *ok)
{
    *ok = L >= 0 && (long long)L + 1 <= cap;
    return *ok ? (L + bs) / bs : 1;
}

__device__ __forceinline__ void walk_load(SeqWalk &w, const int32_t *seqlens, long long cap, int bs)
{
    bool ok;
    int L = __ldg(seqlens + w.b);
    w.nblk = seq_blocks(L, cap, bs, &ok);
    w.len = ok ? L : -1;
}

__device__ __forceinline__ void walk_next(SeqWalk &w, const int32_t *seqlens, long long cap, int bs,
                                          int batch)
{
    if (++w.j == w.nblk) {
        w.sb += w.nblk;
        w.j = 0;
        if (++w.b == batch) {
            w.b = 0;
            w.sb = 0;
            ++w.hg;
        }
        walk_load(w, seqlens, cap, bs);
    }
}

// Work split.  Units are weighed in "cost": unit (hg, b, j) sits at cost
// position hg * cblk + sc_b + cs + j, where sc_b = (units of sequences
// 0..b-1) + cs * b, i.e. every sequence carries an overhead of cs
// unit-equivalents before its first unit (cblk = units + cs * B per head
// group).  CTA c takes the units whose positions fall in
// [c Ctot / P, (c+1) Ctot / P).  Starting or ending a sequence costs a CTA a
// fixed time (q load, partial write, fence, ticket): measured on GB300 as
// ~3 us, about two units of 64 KB, so a CTA whose range crosses sequence
// starts gets fewer units and the CTAs finish together (B=64 GQA workload:
// 102-104 -> 100.4 us).  With cs = 0 this is the plain equal split of units.
constexpr int kSeqCost = 2;

// CTA whose cost range contains position pos.
__device__ __forceinline__ int cta_of(long long pos, int P, long long Ctot)
{
    return (int)(((pos + 1) * P - 1) / Ctot);
}

// CONTIG = false: the paged cache [num_blocks, BS, Hkv, D] through the block
// table.  CONTIG = true: the contiguous-cache twin, a cache [batch,
// max_seqlen, Hkv, D] whose sequence b holds position t at row
// b * max_seqlen + t; it has no table, and a unit is BS consecutive rows.
// Everything after the address of a unit's rows is the same code, so for the
// same logical cache and the same split both give the same bits.
template <int D, int BS, int HS, bool CONTIG>
__global__ void __launch_bounds__((HS + 1) * 32, 1)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a)
{
    using Gm = Geom<D, BS, HS>;
    constexpr int NT = Gm::THREADS, NW = Gm::NW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int nst = a.nstages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + nst * Gm::STAGE_BYTES);
    uint64_t *empty = full + nst;
    int *stage_phys = reinterpret_cast<int *>(empty + nst);
    __shared__ int s_warp[NW];
    __shared__ int s_total;
    __shared__ long long s_start[2]; // first sequence, its unit offset sb
    __shared__ long long s_u[2];     // first and one-past-last unit of this CTA

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.batch, mbps = a.max_blocks_per_seq;
    const long long cap = CONTIG ? (long long)a.max_seqlen : (long long)mbps * BS;
    const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(a.q);

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], HS);
        }
        fence_mbar_init();
    }
    if (warp == HS && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    // The next kernel on the stream (when it was launched for programmatic
    // dependence, e.g. the next decode step) is launched once every CTA of
    // this grid has passed here, so it never takes an SM one of ours still
    // needs; its CTAs take SMs as ours leave them and run their own start-up
    // during this grid's merge tail, then wait for this grid to finish.
    grid_dep_trigger();
    // L2 prefetches are hints, and L2 is where every write lands, so they may
    // run before the predecessor has finished: a line it rewrites later is
    // simply updated.  The lengths are prefetched for the scan below, and a
    // small block table, each CTA taking a slice, so that the producer's
    // first table read after the scan hits in L2 instead of waiting on HBM.
    for (int b = tid * 32; b < B; b += NT * 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.cache_seqlens + b));
    if constexpr (!CONTIG) {
        const size_t tbytes = (size_t)B * mbps * 4;
        if (tbytes <= ((size_t)4 << 20)) {
            const size_t lines = (tbytes + 127) / 128;
            const size_t l0 = lines * blockIdx.x / gridDim.x, l1 = lines * (blockIdx.x + 1) / gridDim.x;
            const char *tb = reinterpret_cast<const char *>(a.block_table);
            for (size_t l = l0 + tid; l < l1; l += NT)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(tb + l * 128));
        }
    }
    // Nothing above read or wrote memory a predecessor may write.
    grid_dep_wait();

    // ---- block-wide exclusive scan of the per-sequence block counts
    const int per = (B + NT - 1) / NT;
    const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
    int local = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        bool ok;
        local += seq_blocks(__ldg(a.cache_seqlens + b), cap, BS, &ok);
        if (!ok && blockIdx.x == 0) flag_error(a.dev_err, PA_DEVERR_OVERFLOW);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < NW ? s_warp[lane] : 0;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += t;
        }
        if (lane < NW) s_warp[lane] = inc - v;
        if (lane == NW - 1) s_total = inc;
    }
    __syncthreads();
    const long long ublk = s_total;
    const long long U = ublk * a.head_groups;
    const int P = gridDim.x;
    // Sequence overhead only when sequences are long against a CTA's share
    // (the average sequence spans at least half of one), so that most are
    // split across CTAs and their starts and ends are the expensive kind
    // (partials, fence, ticket); sequences that fit whole inside a CTA cost
    // little (workload of 1028 short sequences: 934 us with cs = 0, 946 us
    // with cs = 2).  Also only when every CTA has several units, so that each
    // CTA strictly inside a sequence's range still holds units of it.
    const bool split_heavy = 2 * ublk * P >= (long long)B * U;
    const int cs = (U >= 4ll * P && split_heavy) ? kSeqCost : 0;
    const long long cblk = ublk + (long long)cs * B;
    const long long Ctot = cblk * a.head_groups;
    {
        // first unit at or after cost positions c0 and c1
        const long long sbt = (long long)s_warp[warp] + incl - local; // units before b_lo
        const long long sct = sbt + (long long)cs * b_lo;             // cost before b_lo
        const long long span = local + (long long)cs * (b_hi - b_lo);
        for (int e = 0; e < 2; ++e) {
            const long long cc = (long long)(blockIdx.x + e) * Ctot / P;
            if (cc >= Ctot) {
                if (tid == 0) s_u[e] = U;
                continue;
            }
            const long long r = cc % cblk;
            if (r < sct || r >= sct + span) continue;
            long long sb = sbt, sc = sct;
            for (int b = b_lo; b < b_hi; ++b) {
                bool ok;
                const int n = seq_blocks(__ldg(a.cache_seqlens + b), cap, BS, &ok);
                if (r < sc + cs + n) {
                    const long long j = r < sc + cs ? 0 : r - sc - cs;
                    s_u[e] = (cc / cblk) * ublk + sb + j;
                    if (e == 0) {
                        s_start[0] = b;
                        s_start[1] = sb;
                    }
                    break;
                }
                sb += n;
                sc += cs + n;
            }
        }
    }
    __syncthreads();
    const long long u0 = s_u[0], u1 = s_u[1];
    if (u0 >= u1) return;

    SeqWalk w;
    w.hg = (int)(u0 / ublk);
    w.b = (int)s_start[0];
    w.sb = s_start[1];
    walk_load(w, a.cache_seqlens, cap, BS);
    w.j = (int)(u0 % ublk - w.sb);

    if (warp == HS) {
        // ================= producer: unit rows -> TMA =================
        // One box per unit for K and one for V: the cache is viewed as
        // (64 dims, rows, kv-head halves), so a box of BS rows x the HS*KB
        // halves of this head group lands as HS*KB slabs of BS 128-byte rows,
        // slab (head, half) at (head * KB + half) * BOX_BYTES: the layout the
        // consumers read, with the 128-byte swizzle phase = row % 8.
        int tab_b = -1, tab_hg = -1, tab_j0 = 0, tab_entry = -1;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long u = u0; u < u1; ++u) {
            int row0 = -1; // cache row of the unit's first token, -1: nothing to load
            if constexpr (CONTIG) {
                if (w.len >= 0) row0 = w.b * a.max_seqlen + w.j * BS;
            } else {
                if (w.b != tab_b || w.hg != tab_hg || w.j >= tab_j0 + 32) {
                    tab_b = w.b;
                    tab_hg = w.hg;
                    tab_j0 = w.j;
                    const int jj = w.j + lane;
                    tab_entry = (w.len >= 0 && jj < w.nblk)
                                    ? __ldg(a.block_table + (size_t)w.b * mbps + jj)
                                    : -1;
                }
                const int p = __shfl_sync(kFull, tab_entry, w.j - tab_j0);
                const bool valid = w.len >= 0 && p >= 0 && p < a.num_blocks;
                if (w.len >= 0 && !valid && lane == 0) flag_error(a.dev_err, PA_DEVERR_BAD_BLOCK);
                row0 = valid ? p * BS : -1;
            }
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                stage_phys[stage] = row0;
                if (row0 >= 0)
                    mbar_arrive_expect_tx(&full[stage], Gm::STAGE_BYTES);
                else
                    mbar_arrive(&full[stage]);
            }
            __syncwarp();
            if (row0 >= 0 && lane < 2) {
                const uint32_t dst = smem_u32(smem + stage * Gm::STAGE_BYTES + lane * Gm::KV_BYTES);
                tma_load_3d(dst, lane ? &tm_v : &tm_k, &full[stage], 0, row0, w.hg * HS * Gm::KB);
            }
            if (++stage == nst) {
                stage = 0;
                phase ^= 1;
            }
            walk_next(w, a.cache_seqlens, cap, BS, B);
        }
        if (!ok && lane == 0) flag_error(a.dev_err, PA_DEVERR_TIMEOUT);
        return;
    }

    // ================= consumers: one warp per kv head =================
    const int hw = warp;
    const int G = a.group;
    const int Hkv = a.num_kv_heads, Hq = a.num_heads;
    const int trow = lane >> 2;        // C-fragment row (token / dim) within 8
    const int g0 = 2 * (lane & 3);     // C-fragment columns g0, g0 + 1 (query heads)
    const int mi = lane >> 3, mr = lane & 7;
    const int k_toff = (mi & 1) * 8 + mr, k_doff = (mi >> 1) * 8; // ldmatrix A = K
    const int v_toff = (mi >> 1) * 8 + mr, v_doff = (mi & 1) * 8; // ldmatrix.trans A = V^T
    const size_t slot_floats = (size_t)HS * G * (D + 2);

    uint32_t qf[Gm::KS][2];
    float acc[Gm::KS][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool bad = false, open = false;
    int seg_j0 = 0;
    int stage = 0;
    uint32_t phase = 0;

    // q fragments of the sequence after this one, fetched during this one's
    // last unit so that a new segment does not start on a dependent load
    uint32_t qn[Gm::KS][2];
    bool qn_ok = false;
    const int gq = lane >> 2;
    auto load_q = [&](int b, int kvh_, uint32_t(&dst)[Gm::KS][2]) {
        const __nv_bfloat16 *qrow = qp + ((size_t)b * Hq + (size_t)kvh_ * G + gq) * D + 2 * (lane & 3);
#pragma unroll
        for (int ks = 0; ks < Gm::KS; ++ks) {
            dst[ks][0] = gq < G ? __ldg(reinterpret_cast<const unsigned int *>(qrow + ks * 16)) : 0u;
            dst[ks][1] = gq < G ? __ldg(reinterpret_cast<const unsigned int *>(qrow + ks * 16 + 8)) : 0u;
        }
    };

    for (long long u = u0; u < u1; ++u) {
        const int kvh = w.hg * HS + hw;
        if (!open) {
            if (qn_ok) {
#pragma unroll
                for (int ks = 0; ks < Gm::KS; ++ks) {
                    qf[ks][0] = qn[ks][0];
                    qf[ks][1] = qn[ks][1];
                }
            } else {
                load_q(w.b, kvh, qf);
            }
            qn_ok = false;
#pragma unroll
            for (int i = 0; i < Gm::KS; ++i)
                acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            bad = w.len < 0;
            seg_j0 = w.j;
            open = true;
        }
        if (w.j == w.nblk - 1 && u + 1 < u1) {
            // the next unit starts sequence b + 1 (or sequence 0 of the next
            // head group): its q is in flight while this unit is computed
            const bool wrap = w.b + 1 == B;
            load_q(wrap ? 0 : w.b + 1, (wrap ? w.hg + 1 : w.hg) * HS + hw, qn);
            qn_ok = true;
        }
        if (!mbar_wait(&full[stage], phase)) {
            if (lane == 0) flag_error(a.dev_err, PA_DEVERR_TIMEOUT);
            return;
        }
        const int p = stage_phys[stage]; // first cache row of the unit, or -1
        const int L = w.len;
        bad |= (p < 0);
        uint8_t *kst = smem + stage * Gm::STAGE_BYTES + hw * Gm::HEAD_BYTES;
        uint8_t *vst = kst + Gm::KV_BYTES;

        // in-place append: the block holding position L
        if (p >= 0 && L >= 0 && w.j == L / BS) {
            constexpr int EPL = D / 32;
            const int slot = L % BS, d0 = lane * EPL;
            const size_t src = ((size_t)w.b * Hkv + kvh) * D + d0;
            const size_t dst = ((size_t)(p + slot) * Hkv + kvh) * D + d0;
            const uint32_t so = (d0 >> 6) * Gm::BOX_BYTES + sw128_offset(slot, d0 & 63);
            const __nv_bfloat16 *kn = static_cast<const __nv_bfloat16 *>(a.k_new);
            const __nv_bfloat16 *vn = static_cast<const __nv_bfloat16 *>(a.v_new);
            __nv_bfloat16 *kc = static_cast<__nv_bfloat16 *>(a.k_cache);
            __nv_bfloat16 *vc = static_cast<__nv_bfloat16 *>(a.v_cache);
            if constexpr (EPL == 4) {
                const uint2 kx = *reinterpret_cast<const uint2 *>(kn + src);
                const uint2 vx = *reinterpret_cast<const uint2 *>(vn + src);
                *reinterpret_cast<uint2 *>(kc + dst) = kx;
                *reinterpret_cast<uint2 *>(vc + dst) = vx;
                *reinterpret_cast<uint2 *>(kst + so) = kx;
                *reinterpret_cast<uint2 *>(vst + so) = vx;
            } else {
                const uint32_t kx = *reinterpret_cast<const uint32_t *>(kn + src);
                const uint32_t vx = *reinterpret_cast<const uint32_t *>(vn + src);
                *reinterpret_cast<uint32_t *>(kc + dst) = kx;
                *reinterpret_cast<uint32_t *>(vc + dst) = vx;
                *reinterpret_cast<uint32_t *>(kst + so) = kx;
                *reinterpret_cast<uint32_t *>(vst + so) = vx;
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // slots past the last position of the sequence: zero their V rows so
        // that whatever the pool holds there (even NaN) meets a zero weight
        // as a zero, not as NaN
        if (p >= 0 && L >= 0 && w.j == w.nblk - 1 && L % BS != BS - 1) {
            const int r0 = L % BS + 1;
            const int chunks = (BS - r0) * 8 * Gm::KB;
            for (int ci = lane; ci < chunks; ci += 32) {
                const int box = ci / ((BS - r0) * 8), rem = ci % ((BS - r0) * 8);
                *reinterpret_cast<uint4 *>(vst + box * Gm::BOX_BYTES + (r0 + rem / 8) * 128 +
                                           (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
        }

        // ---- S^T[token, head] = K q^T (fp32 accumulators)
        const uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);
        float s[Gm::MT][4];
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
            const int t = mt * 16 + k_toff;
#pragma unroll
            for (int ks = 0; ks < Gm::KS; ++ks) {
                const int d = ks * 16 + k_doff;
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kbase + (d >> 6) * Gm::BOX_BYTES + sw128_offset(t, d & 63), r0, r1, r2, r3);
                mma_bf16_16816(s[mt], r0, r1, r2, r3, qf[ks][0], qf[ks][1]);
            }
        }
        // ---- mask, scale (log2 domain), online softmax
        const int pos0 = w.j * BS + trow;
        float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pos = pos0 + mt * 16 + ((i >> 1) << 3);
                const bool vis = p >= 0 && pos <= L;
                s[mt][i] = vis ? s[mt][i] * a.scale_log2 : -INFINITY;
                if (i & 1)
                    t1 = fmaxf(t1, s[mt][i]);
                else
                    t0 = fmaxf(t0, s[mt][i]);
            }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, o));
            t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, o));
        }
        const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2_approx(m0 - mu0), al1 = exp2_approx(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            s[mt][0] = exp2_approx(s[mt][0] - mu0);
            s[mt][1] = exp2_approx(s[mt][1] - mu1);
            s[mt][2] = exp2_approx(s[mt][2] - mu0);
            s[mt][3] = exp2_approx(s[mt][3] - mu1);
            ps0 += s[mt][0] + s[mt][2];
            ps1 += s[mt][1] + s[mt][3];
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int dm = 0; dm < Gm::KS; ++dm) {
            acc[dm][0] *= al0;
            acc[dm][1] *= al1;
            acc[dm][2] *= al0;
            acc[dm][3] *= al1;
        }
        // ---- O^T[dim, head] += V^T P^T
#pragma unroll
        for (int mt = 0; mt < Gm::MT; ++mt) {
            const uint32_t b0 = movmatrix_trans(pack_bf16(s[mt][0], s[mt][1]));
            const uint32_t b1 = movmatrix_trans(pack_bf16(s[mt][2], s[mt][3]));
            const int t = mt * 16 + v_toff;
#pragma unroll
            for (int dm = 0; dm < Gm::KS; ++dm) {
                const int d = dm * 16 + v_doff;
                uint32_t r0, r1, r2, r3;
                ldsm_x4_trans(vbase + (d >> 6) * Gm::BOX_BYTES + sw128_offset(t, d & 63), r0, r1,
                              r2, r3);
                mma_bf16_16816(acc[dm], r0, r1, r2, r3, b0, b1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == nst) {
            stage = 0;
            phase ^= 1;
        }

        // ---- end of this CTA's share of the sequence
        if (w.j == w.nblk - 1 || u == u1 - 1) {
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                l0 += __shfl_xor_sync(kFull, l0, o);
                l1 += __shfl_xor_sync(kFull, l1, o);
            }
            __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);
            const size_t orow = ((size_t)w.b * Hq + (size_t)kvh * G) * D;
            if (seg_j0 == 0 && w.j == w.nblk - 1) {
                // the whole sequence was here: normalise and store
                const float i0 = (bad || !(l0 > 0.f)) ? 0.f : 1.f / l0;
                const float i1 = (bad || !(l1 > 0.f)) ? 0.f : 1.f / l1;
#pragma unroll
                for (int dm = 0; dm < Gm::KS; ++dm)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int d = dm * 16 + trow + ((i >> 1) << 3), g = g0 + (i & 1);
                        if (g < G)
                            out[orow + (size_t)g * D + d] =
                                __float2bfloat16_rn(acc[dm][i] * ((i & 1) ? i1 : i0));
                    }
            } else {
                // partial (acc, m, l) into slot (CTA + segment row)
                // cost position of the sequence's first unit
                const long long F = (long long)w.hg * cblk + w.sb + (long long)cs * w.b + cs;
                const int cfirst = cta_of(F, P, Ctot), clast = cta_of(F + w.nblk - 1, P, Ctot);
                const long long segrow = (long long)w.hg * B + w.b;
                float *slot = a.part + (size_t)(blockIdx.x + segrow) * slot_floats;
                float *pacc = slot + (size_t)hw * G * D;
                float *pml = slot + (size_t)HS * G * D + (size_t)hw * G * 2;
#pragma unroll
                for (int dm = 0; dm < Gm::KS; ++dm)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int d = dm * 16 + trow + ((i >> 1) << 3), g = g0 + (i & 1);
                        if (g < G) pacc[(size_t)g * D + d] = acc[dm][i];
                    }
                if (trow == 0) {
                    if (g0 < G) {
                        pml[g0 * 2] = m0;
                        pml[g0 * 2 + 1] = bad ? -1.f : l0;
                    }
                    if (g0 + 1 < G) {
                        pml[g0 * 2 + 2] = m1;
                        pml[g0 * 2 + 3] = bad ? -1.f : l1;
                    }
                }
                // The warp's partial writes are ordered before lane 0's ticket
                // increment by the warp barrier, and the increment is an
                // acquire-release at GPU scope: it publishes them, and the
                // last arriver acquires every other segment's partial through
                // it (then the warp barrier orders its lanes' loads after
                // that).  One round trip instead of a fence in every lane
                // before the increment and another after it.
                __syncwarp();
                int last = 0;
                int32_t *ticket = a.tickets + (size_t)w.b * Hkv + kvh;
                // segments of this sequence: every CTA in [cfirst, clast] has units
                // when U >= P; when U < P a CTA holds at most one unit, so the
                // sequence has exactly nblk segments, one per unit
                const bool dense = U >= P;
                const int nseg = dense ? clast - cfirst + 1 : w.nblk;
                if (lane == 0) {
                    int old;
                    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(ticket) : "memory");
                    last = old == nseg - 1;
                }
                last = __shfl_sync(kFull, last, 0);
                if (last) {
                    __syncwarp();
                    // fold the partials in logical (CTA) order.  Each
                    // partial's (m, l) and accumulator rows for every head of
                    // the group are loaded together before any of them is
                    // folded: one L2 round trip per partial instead of one
                    // per (head, partial) -- this fold runs at the very end
                    // of the launch, so its latency is the launch's tail.
                    // Heads go in pairs (G <= 8, checked by the plan): 12 to
                    // 20 loads in flight per round trip, and few enough
                    // registers that the 9-warp variant (at most 168 per
                    // thread) does not spill; chunks of 4 spilled there.
                    constexpr int GC = 2, DL = D / 32;
                    for (int gb = 0; gb < G; gb += GC) {
                        float m[GC], l[GC], o[GC][DL];
                        bool gbad[GC];
#pragma unroll
                        for (int g = 0; g < GC; ++g) {
                            m[g] = -INFINITY;
                            l[g] = 0.f;
                            gbad[g] = false;
#pragma unroll
                            for (int k = 0; k < DL; ++k) o[g][k] = 0.f;
                        }
                        for (int k = 0; k < nseg; ++k) {
                            const int c = dense ? cfirst + k : cta_of(F + k, P, Ctot);
                            const float *sc = a.part + (size_t)(c + segrow) * slot_floats;
                            const float *ml = sc + (size_t)HS * G * D + ((size_t)hw * G + gb) * 2;
                            const float *pc = sc + ((size_t)hw * G + gb) * D;
                            float mc[GC], lc[GC], oc[GC][DL];
#pragma unroll
                            for (int g = 0; g < GC; ++g) {
                                if (gb + g < G) {
                                    mc[g] = __ldcg(ml + g * 2);
                                    lc[g] = __ldcg(ml + g * 2 + 1);
#pragma unroll
                                    for (int kk = 0; kk < DL; ++kk)
                                        oc[g][kk] = __ldcg(pc + (size_t)g * D + lane + 32 * kk);
                                }
                            }
#pragma unroll
                            for (int g = 0; g < GC; ++g) {
                                if (gb + g < G) {
                                    gbad[g] |= lc[g] < 0.f;
                                    const float mn = fmaxf(m[g], mc[g]);
                                    const float mu = mn == -INFINITY ? 0.f : mn;
                                    const float wa = exp2_approx(m[g] - mu);
                                    const float wb = exp2_approx(mc[g] - mu);
                                    l[g] = l[g] * wa + lc[g] * wb;
#pragma unroll
                                    for (int kk = 0; kk < DL; ++kk)
                                        o[g][kk] = o[g][kk] * wa + oc[g][kk] * wb;
                                    m[g] = mn;
                                }
                            }
                        }
#pragma unroll
                        for (int g = 0; g < GC; ++g) {
                            if (gb + g < G) {
                                const float inv = (gbad[g] || !(l[g] > 0.f)) ? 0.f : 1.f / l[g];
#pragma unroll
                                for (int k = 0; k < DL; ++k)
                                    out[orow + (size_t)(gb + g) * D + lane + 32 * k] =
                                        __float2bfloat16_rn(o[g][k] * inv);
                            }
                        }
                    }
                    if (lane == 0) *ticket = 0;
                }
            }
            open = false;
        }
        walk_next(w, a.cache_seqlens, cap, BS, B);
    }
}

// ------------------------------------------------------------------ fp32
template <int D>
__global__ void __launch_bounds__(128) decode_f32_kernel(const DecodeArgs a, int bs)
{
    constexpr int EPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 4 + warp;
    if (gw >= (long long)a.batch * a.num_heads) return;
    const int b = (int)(gw / a.num_heads), h = (int)(gw % a.num_heads);
    const int G = a.group, kvh = h / G, Hkv = a.num_kv_heads;
    const float *q = static_cast<const float *>(a.q);
    const float *kc = static_cast<const float *>(a.k_cache);
    const float *vc = static_cast<const float *>(a.v_cache);
    const float *kn = static_cast<const float *>(a.k_new);
    const float *vn = static_cast<const float *>(a.v_new);
    float *out = static_cast<float *>(a.out) + ((size_t)b * a.num_heads + h) * D + lane * EPL;
    const int L = a.cache_seqlens[b];
    const int mbps = a.max_blocks_per_seq;
    if (L < 0 || (long long)L + 1 > (long long)mbps * bs) {
        if (lane == 0) flag_error(a.dev_err, PA_DEVERR_OVERFLOW);
#pragma unroll
        for (int k = 0; k < EPL; ++k) out[k] = 0.f;
        return;
    }
    float qv[EPL], acc[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) {
        qv[k] = q[((size_t)b * a.num_heads + h) * D + lane * EPL + k];
        acc[k] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    int p_app = -1;
    for (int j = 0; j <= L; ++j) {
        const int p = a.block_table[(size_t)b * mbps + j / bs];
        if (p < 0 || p >= a.num_blocks) {
            bad = true;
            break;
        }
        const float *krow, *vrow;
        if (j == L) {
            p_app = p;
            krow = kn + ((size_t)b * Hkv + kvh) * D;
            vrow = vn + ((size_t)b * Hkv + kvh) * D;
        } else {
            const size_t off = (((size_t)p * bs + j % bs) * Hkv + kvh) * D;
            krow = kc + off;
            vrow = vc + off;
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < EPL; ++k) dot = fmaf(qv[k], krow[lane * EPL + k], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
        const float sc = dot * a.scale;
        const float mn = fmaxf(m, sc);
        const float alpha = expf(m - mn), pj = expf(sc - mn);
        l = l * alpha + pj;
#pragma unroll
        for (int k = 0; k < EPL; ++k) acc[k] = acc[k] * alpha + pj * vrow[lane * EPL + k];
        m = mn;
    }
    if (bad) {
        if (lane == 0) flag_error(a.dev_err, PA_DEVERR_BAD_BLOCK);
#pragma unroll
        for (int k = 0; k < EPL; ++k) out[k] = 0.f;
        return;
    }
    if (h % G == 0) { // one warp per kv head performs the append
        const size_t dst = (((size_t)p_app * bs + L % bs) * Hkv + kvh) * D + lane * EPL;
        const size_t src = ((size_t)b * Hkv + kvh) * D + lane * EPL;
#pragma unroll
        for (int k = 0; k < EPL; ++k) {
            const_cast<float *>(kc)[dst + k] = kn[src + k];
            const_cast<float *>(vc)[dst + k] = vn[src + k];
        }
    }
    const float inv = 1.f / l;
#pragma unroll
    for (int k = 0; k < EPL; ++k) out[k] = acc[k] * inv;
}

template <int D, int BS, int HS, bool CONTIG>
int launch_bf16(const DecodeArgs &a, const DecodePlan &plan, const CUtensorMap &tm_k,
                const CUtensorMap &tm_v, cudaStream_t s)
{
    // The shared-memory attribute was set when the plan was made.  The
    // launch allows programmatic dependence: the kernel's start-up (barrier
    // set-up, descriptor and L2 prefetches) may overlap the end of the kernel
    // before it on the stream, and it reads nothing before that kernel is done.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ctas);
    cfg.blockDim = dim3(Geom<D, BS, HS>::THREADS);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_bf16_kernel<D, BS, HS, CONTIG>, tm_k, tm_v, a);
    return e == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

// Resident CTAs per SM of one instantiation on the current device.  The
// first query per (device, instantiation) also raises the kernel's dynamic
// shared-memory limit; later calls read the cached answer, so the per-call
// host cost of a decode launch is a few table lookups.
constexpr int kMaxDev = 64;
int g_occ_cache[kMaxDev][2][2][2][4];

template <int D, int BS, int HS, bool CONTIG>
int occupancy_of(size_t smem)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    int &slot =
        g_occ_cache[dev][CONTIG][D == 128][BS == 32][HS == 8 ? 3 : HS == 4 ? 2 : HS == 2 ? 1 : 0];
    const int cached = __atomic_load_n(&slot, __ATOMIC_ACQUIRE);
    if (cached > 0) return cached;
    auto kern = decode_bf16_kernel<D, BS, HS, CONTIG>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Geom<D, BS, HS>::THREADS, smem) !=
        cudaSuccess)
        return 0;
    __atomic_store_n(&slot, n, __ATOMIC_RELEASE);
    return n;
}

}  // namespace

// Runs __VA_ARGS__ with constexpr D, BS, HS set to the runtime values.
#define PA_DECODE_HS(D_, BS_, HS_, ...)                                                      \
    do {                                                                                      \
        if (HS_ == 8) { constexpr int D = D_, BS = BS_, HS = 8; __VA_ARGS__; }               \
        if (HS_ == 4) { constexpr int D = D_, BS = BS_, HS = 4; __VA_ARGS__; }               \
        if (HS_ == 2) { constexpr int D = D_, BS = BS_, HS = 2; __VA_ARGS__; }               \
        if (HS_ == 1) { constexpr int D = D_, BS = BS_, HS = 1; __VA_ARGS__; }               \
    } while (0)
// Paged kernels: every supported (head_dim, block_size).  Contiguous-cache
// kernels: only the unit contig_unit(head_dim).
#define PA_DECODE_SWITCH(CONTIG_, D_, BS_, HS_, ...)                                         \
    do {                                                                                      \
        if (CONTIG_) {                                                                        \
            constexpr bool CONTIG = true;                                                     \
            if (D_ == 128 && BS_ == contig_unit(128)) PA_DECODE_HS(128, contig_unit(128), HS_, __VA_ARGS__); \
            else if (D_ == 64 && BS_ == contig_unit(64)) PA_DECODE_HS(64, contig_unit(64), HS_, __VA_ARGS__); \
        } else {                                                                              \
            constexpr bool CONTIG = false;                                                    \
            if (D_ == 128 && BS_ == 16) PA_DECODE_HS(128, 16, HS_, __VA_ARGS__);             \
            else if (D_ == 128 && BS_ == 32) PA_DECODE_HS(128, 32, HS_, __VA_ARGS__);        \
            else if (D_ == 64 && BS_ == 16) PA_DECODE_HS(64, 16, HS_, __VA_ARGS__);          \
            else if (D_ == 64 && BS_ == 32) PA_DECODE_HS(64, 32, HS_, __VA_ARGS__);          \
        }                                                                                     \
    } while (0)

int decode_bf16_plan(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     DecodePlan *plan, bool contig)
{
    if (!((head_dim == 64 || head_dim == 128) && (block_size == 16 || block_size == 32)))
        return PA_ERR_UNSUPPORTED;
    if (contig && block_size != contig_unit(head_dim)) return PA_ERR_UNSUPPORTED;
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
    const int G = num_heads / num_kv_heads;
    if (G > 8) return PA_ERR_UNSUPPORTED;
    int hs = 8;
    while (num_kv_heads % hs != 0) hs >>= 1;
    const size_t stage = (size_t)2 * hs * head_dim * block_size * 2;
    int nst = (int)(196608 / stage);
    nst = nst < 2 ? 2 : (nst > 8 ? 8 : nst);
    plan->heads_per_cta = hs;
    plan->head_groups = num_kv_heads / hs;
    plan->nstages = nst;
    plan->smem_bytes = nst * stage + 1024 + (size_t)nst * 20 + 64;
    int occ = 0;
    PA_DECODE_SWITCH(contig, head_dim, block_size, hs,
                     { occ = occupancy_of<D, BS, HS, CONTIG>(plan->smem_bytes); });
    if (occ <= 0) return PA_ERR_LAUNCH;
    const int sms = num_sms();
    if (sms <= 0) return PA_ERR_DEVICE;
    plan->ctas = sms * occ;
    plan->part_floats = ((size_t)plan->ctas + (size_t)plan->head_groups * batch) *
                        (size_t)hs * G * (head_dim + 2);
    plan->ticket_ints = (size_t)batch * num_kv_heads;
    if (plan->ticket_ints * 4 > kTicketRegionBytes) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

size_t decode_workspace_bytes(const DecodePlan &plan)
{
    return kTicketRegionBytes + plan.part_floats * 4;
}

int decode_bf16_launch(const DecodeArgs &a, int head_dim, int block_size, const DecodePlan &plan,
                       const CUtensorMap &tm_k, const CUtensorMap &tm_v, cudaStream_t s,
                       bool contig)
{
    int rc = PA_ERR_UNSUPPORTED;
    PA_DECODE_SWITCH(contig, head_dim, block_size, plan.heads_per_cta,
                     { rc = launch_bf16<D, BS, HS, CONTIG>(a, plan, tm_k, tm_v, s); });
    return rc;
}

int decode_f32_launch(const DecodeArgs &a, int head_dim, int block_size, cudaStream_t s)
{
    const long long warps = (long long)a.batch * a.num_heads;
    const unsigned grid = (unsigned)((warps + 3) / 4);
    if (head_dim == 64)
        decode_f32_kernel<64><<<grid, 128, 0, s>>>(a, block_size);
    else if (head_dim == 128)
        decode_f32_kernel<128><<<grid, 128, 0, s>>>(a, block_size);
    else
        return PA_ERR_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

}  // namespace pa
