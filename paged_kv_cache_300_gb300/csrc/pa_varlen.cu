// Varlen (packed, variable-length) attention.
//
// "Perhatian berhalaman" (HF transformers docs), section "Jalur Varlen" ->
// "Mekanisme pengindeksan" / "Contoh": requests are packed along the token
// axis; request r owns q rows [cu_seq_lens_q[r], cu_seq_lens_q[r+1]) and k/v
// rows [cu_seq_lens_k[r], cu_seq_lens_k[r+1]); max_length_q/k size the
// launch.  Causal masking is bottom-right aligned: query i of a request with
// lengths (ql, kl) sees key j iff j <= i + kl - ql.  A query with no visible
// key (for instance every query of the example's request r0, which has no
// key tokens) gets a zero row.
//
// This file holds the fp32 CUDA-core kernel (one warp per query row and
// head, online softmax with expf).  The bf16 tensor-core kernel lives in
// pa_varlen_tc.cu.
#include "pa_common.cuh"
#include "pa_internal.h"

#include <math.h>

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int owner_of(const int32_t *cu, int n, long long x)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= x)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

template <int D>
__global__ void __launch_bounds__(128) varlen_f32_kernel(const VarlenArgs a)
{
    constexpr int EPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 4 + warp;
    if (gw >= (long long)a.total_q * a.num_heads) return;
    const long long row = gw / a.num_heads;
    const int h = (int)(gw % a.num_heads);
    const int G = a.num_heads / a.num_kv_heads, kvh = h / G;
    float *out = static_cast<float *>(a.out) + (row * a.num_heads + h) * D + lane * EPL;
    const int b = owner_of(a.cu_q, a.batch, row);
    const int q0 = __ldg(a.cu_q + b), q1 = __ldg(a.cu_q + b + 1);
    const int k0 = __ldg(a.cu_k + b), k1 = __ldg(a.cu_k + b + 1);
    if (row < q0 || row >= q1 || k1 < k0 || k0 < 0 || k1 > a.total_k) {
        if (lane == 0) flag_error(a.dev_err, PA_DEVERR_BAD_CU);
#pragma unroll
        for (int k = 0; k < EPL; ++k) out[k] = 0.f;
        return;
    }
    const int ql = q1 - q0, kl = k1 - k0, i = (int)(row - q0);
    int n = kl;
    if (a.causal) n = max(0, min(kl, i + kl - ql + 1));
    const float *q = static_cast<const float *>(a.q) + (row * a.num_heads + h) * D + lane * EPL;
    const float *kp = static_cast<const float *>(a.k);
    const float *vp = static_cast<const float *>(a.v);
    float qv[EPL], acc[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) {
        qv[k] = q[k];
        acc[k] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n; ++j) {
        const size_t off = ((size_t)(k0 + j) * a.num_kv_heads + kvh) * D + lane * EPL;
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < EPL; ++k) dot = fmaf(qv[k], kp[off + k], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
        const float sc = dot * a.scale;
        const float mn = fmaxf(m, sc);
        const float alpha = expf(m - mn), pj = expf(sc - mn);
        l = l * alpha + pj;
#pragma unroll
        for (int k = 0; k < EPL; ++k) acc[k] = acc[k] * alpha + pj * vp[off + k];
        m = mn;
    }
    const float inv = n > 0 ? 1.f / l : 0.f;
#pragma unroll
    for (int k = 0; k < EPL; ++k) out[k] = acc[k] * inv;
}

}  // namespace

int varlen_f32_launch(const VarlenArgs &a, cudaStream_t s)
{
    const long long warps = (long long)a.total_q * a.num_heads;
    if (warps == 0) return PA_OK;
    const unsigned grid = (unsigned)((warps + 3) / 4);
    if (a.head_dim == 64)
        varlen_f32_kernel<64><<<grid, 128, 0, s>>>(a);
    else if (a.head_dim == 128)
        varlen_f32_kernel<128><<<grid, 128, 0, s>>>(a);
    else
        return PA_ERR_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_LAUNCH;
}

}  // namespace pa
