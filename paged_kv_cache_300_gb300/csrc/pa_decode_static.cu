// pa_decode_static_scratch: the bf16 decode step without a caller-supplied
// workspace, for callers that cannot allocate device memory at call time
// (an allocator-free runtime, a plugin that only receives input and output
// pointers, code running where cudaMalloc is forbidden or would
// synchronise).  Its split-K partials and merge counters live in a
// fixed-size array in this file, allocated once when the library's module
// is loaded on a device and held until the process exits.
#include "pa_internal.h"

#include <mutex>

namespace pa {
namespace {

// 16 MiB: the 1 MiB counter region plus 15 MiB of partials.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static_assert(kStaticScratchBytes > kTicketRegionBytes, "scratch must hold the counters");

// Zero-initialised at module load; one copy per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (set-up once
// per device; in host code the symbol itself is only a host-side stand-in).
int scratch_address(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
            return PA_ERR_LAUNCH;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_static_scratch(const void *q, void *k_cache, void *v_cache,
                                        const int32_t *block_table, const int32_t *cache_seqlens,
                                        const void *k_new, const void *v_new, void *out,
                                        int batch, int num_heads, int num_kv_heads, int head_dim,
                                        int num_blocks, int block_size, int max_blocks_per_seq,
                                        float softmax_scale, int32_t *dev_err, void *stream)
{
    using namespace pa;
    if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || num_heads % num_kv_heads != 0)
        return PA_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (batch == 0) return PA_OK;
    // every check pa_decode makes on the host comes first: a call refused
    // with a status must not have cleared the counters of a call in flight
    if (!block_table || !cache_seqlens) return PA_ERR_NULL;
    int rc = decode_check_pointers(q, k_cache, v_cache, k_new, v_new, out);
    if (rc != PA_OK) return rc;
    if ((long long)num_blocks * block_size >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    DecodePlan plan;
    rc = decode_bf16_plan(batch, num_heads, num_kv_heads, head_dim, block_size, &plan);
    if (rc != PA_OK) return rc;
    const size_t need = decode_workspace_bytes(plan);
    if (need > kStaticScratchBytes) return PA_ERR_WORKSPACE; // beyond the fixed maximum
    void *scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != PA_OK) return rc;
    // The array keeps the previous call's contents: clear the counters this
    // call uses (a memset, no allocation) so that even a call that ended
    // with PA_DEVERR_TIMEOUT leaves nothing behind.
    if (cudaMemsetAsync(scratch, 0, plan.ticket_ints * sizeof(int32_t),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_LAUNCH;
    return pa_decode(q, k_cache, v_cache, block_table, cache_seqlens, k_new, v_new, out, batch,
                     num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                     max_blocks_per_seq, PA_BF16, softmax_scale, scratch, need, dev_err, stream);
}
