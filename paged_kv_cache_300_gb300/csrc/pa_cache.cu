// Varlen cache update: scatter a packed chunk of new K/V rows into the paged
// pool and, optionally, gather each request's whole key sequence (cached
// prefix + chunk) into packed k/v for the varlen attention.
//
// "Perhatian berhalaman" (HF transformers docs), section "Jalur Varlen" ->
// "Perilaku cache": the varlen kernel has no way to reach the paged cache,
// so the cache is read and written by a separate update step.  Row i of
// request b's chunk belongs at logical position cache_seqlens[b] + i, i.e.
// block block_table[b][pos / bs], slot pos % bs ("Jalur decode" indexing).
//
// HBM-bound copy: one warp per packed row; a pool row of one token is
// num_kv_heads * head_dim contiguous elements in both the packed tensors and
// the pool ([num_blocks, block_size, num_kv_heads, head_dim]), so every warp
// moves whole rows with 16-byte vector loads and stores.  Rows are mapped to
// requests by binary search over the cumulative lengths.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Largest r in [0, n) with cu[r] <= x (cu has n + 1 entries).
__device__ __forceinline__ int owner_of(const int32_t *cu, int n, long long x)
{
    int lo = 0, hi = n; // invariant: cu[lo] <= x (if any), answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= x)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void copy_row(uint8_t *dst, const uint8_t *src, int bytes, int lane)
{
    for (int off = lane * 16; off < bytes; off += 32 * 16)
        *reinterpret_cast<uint4 *>(dst + off) = __ldg(reinterpret_cast<const uint4 *>(src + off));
}

__device__ __forceinline__ void copy_row2(uint8_t *dst0, uint8_t *dst1, const uint8_t *src,
                                          int bytes, int lane)
{
    for (int off = lane * 16; off < bytes; off += 32 * 16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src + off));
        *reinterpret_cast<uint4 *>(dst0 + off) = v;
        *reinterpret_cast<uint4 *>(dst1 + off) = v;
    }
}

// Physical pool row of logical position pos of request b, or -1 (error flagged).
__device__ __forceinline__ long long pool_row(const CacheUpdateArgs &a, int b, int pos)
{
    const int lb = pos / a.block_size;
    if (pos < 0 || lb >= a.max_blocks_per_seq) {
        flag_error(a.dev_err, PA_DEVERR_OVERFLOW);
        return -1;
    }
    const int p = __ldg(a.block_table + (size_t)b * a.max_blocks_per_seq + lb);
    if (p < 0 || p >= a.num_blocks) {
        flag_error(a.dev_err, PA_DEVERR_BAD_BLOCK);
        return -1;
    }
    return (long long)p * a.block_size + pos % a.block_size;
}

__global__ void __launch_bounds__(256) cache_update_kernel(const CacheUpdateArgs a)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + warp;
    const bool gather = a.k_full != nullptr;
    const int rb = a.row_bytes;
    const uint8_t *kch = static_cast<const uint8_t *>(a.k_chunk);
    const uint8_t *vch = static_cast<const uint8_t *>(a.v_chunk);
    uint8_t *kc = static_cast<uint8_t *>(a.k_cache);
    uint8_t *vc = static_cast<uint8_t *>(a.v_cache);

    if (!gather) {
        if (row >= a.total_q) return;
        const int b = owner_of(a.cu_q, a.batch, row);
        const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
        if (row < q0 || row >= q1) {
            if (lane == 0) flag_error(a.dev_err, PA_DEVERR_BAD_CU);
            return;
        }
        const int pos = __ldg(a.prefix + b) + (int)(row - q0);
        const long long pr = pool_row(a, b, pos);
        if (pr < 0) return;
        copy_row(kc + pr * rb, kch + row * rb, rb, lane);
        copy_row(vc + pr * rb, vch + row * rb, rb, lane);
        return;
    }

    if (row >= a.total_k) return;
    const int b = owner_of(a.cu_k, a.batch, row);
    const int k0 = __ldg(a.cu_k + b), k1 = __ldg(a.cu_k + b + 1);
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    const int prefix = __ldg(a.prefix + b);
    if (row < k0 || row >= k1 || q1 < q0 || prefix < 0 || k1 - k0 != prefix + (q1 - q0) ||
        q1 > a.total_q) {
        if (lane == 0) flag_error(a.dev_err, PA_DEVERR_BAD_CU);
        return;
    }
    const int pos = (int)(row - k0);
    uint8_t *kf = static_cast<uint8_t *>(a.k_full) + row * rb;
    uint8_t *vf = static_cast<uint8_t *>(a.v_full) + row * rb;
    const long long pr = pool_row(a, b, pos);
    if (pr < 0) return;
    if (pos < prefix) { // cached prefix: pool -> packed
        copy_row(kf, kc + pr * rb, rb, lane);
        copy_row(vf, vc + pr * rb, rb, lane);
    } else { // new token: chunk -> pool and packed
        const long long src = q0 + (pos - prefix);
        copy_row2(kc + pr * rb, kf, kch + src * rb, rb, lane);
        copy_row2(vc + pr * rb, vf, vch + src * rb, rb, lane);
    }
}

}  // namespace

int cache_update_launch(const CacheUpdateArgs &a, cudaStream_t s)
{
    const long long rows = a.k_full != nullptr ? a.total_k : a.total_q;
    if (rows <= 0) return PA_OK;
    const unsigned grid = (unsigned)((rows + 7) / 8);
    cache_update_kernel<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

}  // namespace pa
