/*
 * pa.h -- C ABI of the paged-attention forward library (GB300, sm_103a).
 *
 * The library computes attention over a key/value cache that is stored in
 * fixed-size physical blocks and reached through a per-sequence block table.
 * The operations follow these passages:
 *
 *   pa_decode        "Perhatian berhalaman" (HF transformers docs), section
 *                    "Jalur decode": one query token per sequence; the cache
 *                    is indexed through block_table[batch, max_blocks_per_seq]
 *                    and updated in place; cache_seqlens gives each
 *                    sequence's cached length.  "39 · PagedAttention"
 *                    (inference-notes), sections 1-3: score every key of the
 *                    sequence in logical order, one softmax, weighted sum of
 *                    the values; partial results merge with
 *                    m = max(m1, m2), l = l1 e^(m1-m) + l2 e^(m2-m).
 *   pa_cache_update  "Perhatian berhalaman", section "Jalur Varlen" ->
 *                    "Perilaku cache": the varlen kernel cannot reach the
 *                    paged cache, so the cache is written and read by a
 *                    separate update step.
 *   pa_varlen        "Perhatian berhalaman", section "Jalur Varlen" ->
 *                    "Mekanisme pengindeksan" / "Contoh": packed requests,
 *                    cumulative lengths cu_seq_lens_q / cu_seq_lens_k,
 *                    maxima max_length_q / max_length_k.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is DEVICE memory owned by the caller, unless a
 *    parameter says otherwise.  The library allocates and frees nothing and
 *    keeps no pointer after a call returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream) and never synchronises the host.
 *  - Tensors are dense and row-major (C order), with the shapes given below.
 *    q/k/v/out element type is selected by `dtype` and is the same for all of
 *    them.  Index arrays are int32.
 *      KV pool  k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *      decode   q, out            [batch, num_heads, head_dim]
 *               k_new, v_new      [batch, num_kv_heads, head_dim]
 *      varlen   q, out            [total_q, num_heads, head_dim]
 *               k, v              [total_k, num_kv_heads, head_dim]
 *  - Query head h reads kv head h / (num_heads / num_kv_heads).
 *  - softmax_scale <= 0 selects 1 / sqrt(head_dim).
 *  - Return value: PA_OK, or a negative PA_ERR_* code for misuse the host can
 *    see (null pointer, unsupported shape or dtype, short workspace).  On a
 *    negative return nothing was launched and no memory was touched.
 *  - Problems only the device can see (a needed block_table entry that is
 *    not a valid block, a length beyond the table, inconsistent cumulative
 *    lengths) set bits PA_DEVERR_* in *dev_err with an atomic OR, if dev_err
 *    is not NULL; the affected outputs are written as zeros and no
 *    out-of-range address is touched.  The kernels never trap and every
 *    wait inside them is bounded (PA_DEVERR_TIMEOUT).  The caller clears
 *    *dev_err when it wants to.
 *
 * Supported: dtype PA_BF16 or PA_F32; head_dim 64 or 128; for PA_BF16
 * decode, block_size 16 or 32 and num_heads / num_kv_heads <= 8.  The bf16
 * varlen calls (pa_varlen, pa_varlen_paged) run the tensor-core kernel, built
 * for head_dim 128 only: head_dim 64 returns PA_ERR_UNSUPPORTED there.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F32 = 0, PA_BF16 = 1 } pa_dtype;

enum {
    PA_OK = 0,
    PA_ERR_NULL = -1,        /* a required pointer is NULL */
    PA_ERR_DTYPE = -2,       /* dtype not PA_F32 / PA_BF16 */
    PA_ERR_SHAPE = -3,       /* inconsistent or negative sizes */
    PA_ERR_UNSUPPORTED = -4, /* valid but not built: head_dim, block_size, group size */
    PA_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than the query says */
    PA_ERR_LAUNCH = -6,      /* the CUDA runtime refused a launch or a setup call */
    PA_ERR_DEVICE = -7       /* no usable CUDA device / not an sm_103 GPU */
};

/* bits of *dev_err */
#define PA_DEVERR_BAD_BLOCK 1 /* a needed block_table entry is < 0 or >= num_blocks */
#define PA_DEVERR_OVERFLOW 2  /* a position lies beyond max_blocks_per_seq * block_size,
                                 or a length is negative */
#define PA_DEVERR_BAD_CU 4    /* cu_seq_lens not non-decreasing, or cu_seq_lens_k does not
                                 equal cache_seqlens + q lengths in pa_cache_update */
#define PA_DEVERR_TIMEOUT 8   /* a bounded wait inside a kernel gave up */

/*
 * Bytes of scratch workspace pa_decode needs for these sizes on the current
 * device (split-K partials and per-sequence merge counters).  0 for PA_F32.
 */
size_t pa_decode_workspace_size(int batch, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, pa_dtype dtype);

/*
 * Decode step: one query per sequence ("Jalur decode").
 *
 * For every sequence b, with L = cache_seqlens[b]:
 *  1. append: k_new[b], v_new[b] are copied bit for bit into the pool at
 *     logical position L, i.e. physical block block_table[b][L / block_size],
 *     slot L % block_size (the worked example: 30 -> block 2 slot 30,
 *     32 -> second block slot 0, 70 -> third block slot 6);
 *  2. attend: out[b, h] = softmax(q[b, h] . K_j * scale) V_j over the
 *     L + 1 positions j = 0..L in logical order, the new token included.
 * cache_seqlens is read only: the caller advances it.  Only the append slot
 * of each sequence is written in the pool; the caller must not map an
 * append slot into a block shared with another sequence.
 *
 * block_table   [batch, max_blocks_per_seq]; entries past the needed blocks
 *               may be -1.  The needed blocks are 0 .. L / block_size.
 * workspace     device scratch of at least pa_decode_workspace_size(...)
 *               bytes (ignored for PA_F32), 16-byte aligned.  It must be
 *               zero-filled before its first use; every call leaves it in a
 *               state the next call accepts (its merge counters back at
 *               zero, whatever the sizes of the call), so one zero fill at
 *               allocation is enough.  After a call that reported
 *               PA_DEVERR_TIMEOUT, zero it again.  Calls that share one
 *               workspace must be ordered on the GPU.  batch * num_kv_heads
 *               may not exceed 262144 (PA_ERR_UNSUPPORTED).
 * Result is independent of where the blocks sit in the pool (bitwise).
 *
 * Host buffers: q, block_table, cache_seqlens, k_new, v_new and out may be
 * page-locked host memory (cudaHostAlloc / cudaMallocHost, or
 * cudaHostRegister-ed), passed as the host pointer.  GB300 reaches such
 * memory in place over NVLink-C2C (unified addressing), so the kernel reads
 * the step's inputs and writes its output there during the call, with no
 * separate copy; a caller that keeps its per-step tensors on the host saves
 * two transfers per step.  k_cache, v_cache, workspace and dev_err must be
 * device memory.  The caller reads `out` after the stream reaches the call.
 */
int pa_decode(const void *q, void *k_cache, void *v_cache, const int32_t *block_table,
              const int32_t *cache_seqlens, const void *k_new, const void *v_new, void *out,
              int batch, int num_heads, int num_kv_heads, int head_dim, int num_blocks,
              int block_size, int max_blocks_per_seq, pa_dtype dtype, float softmax_scale,
              void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * pa_decode without a workspace argument, for callers that cannot allocate
 * device memory when they call: a runtime with its own fixed memory budget
 * and no allocator at hand, a plugin handed only its input and output
 * buffers, or code on a path where cudaMalloc is not allowed or would
 * stall the device.  The pages have no counterpart to this entry point; it
 * is a deployment convenience.
 *
 * Same arguments and results as pa_decode with dtype PA_BF16 (bf16 only).
 * The split-K scratch is a 16 MiB array inside the library (device memory
 * reserved on every GPU that loads the library, held until the process
 * exits); the caller still passes every input and output.  Sizes whose
 * scratch need (pa_decode_workspace_size) exceeds 16 MiB are rejected with
 * PA_ERR_WORKSPACE before anything is launched.  The call allocates nothing
 * (no cudaMalloc/cudaFree, no allocating library routine); it clears the
 * merge counters it uses with cudaMemsetAsync on `stream`.
 *
 * The first call on each device looks up the array's device address with
 * that device current (cudaGetSymbolAddress); make that first call before
 * any stream capture.  All calls share the one array per device, which keeps
 * the previous call's contents: calls that may overlap on the GPU (different
 * streams without ordering) race on it and must be serialised by the caller.
 */
int pa_decode_static_scratch(const void *q, void *k_cache, void *v_cache,
                             const int32_t *block_table, const int32_t *cache_seqlens,
                             const void *k_new, const void *v_new, void *out, int batch,
                             int num_heads, int num_kv_heads, int head_dim, int num_blocks,
                             int block_size, int max_blocks_per_seq, float softmax_scale,
                             int32_t *dev_err, void *stream);

/*
 * The contiguous-cache twin of pa_decode, for measuring what paging costs:
 * "39 · PagedAttention" (inference-notes), sections "Ghi chú" and
 * "4. Có miễn phí không?", compares a paged attention kernel with one over a
 * contiguous cache.  This call is that contiguous kernel: the same decode
 * kernel with the block table taken out.
 *
 * k_cache, v_cache  [batch, max_seqlen, num_kv_heads, head_dim]: sequence b
 *                   holds its position t at [b, t].  Nothing is shared
 *                   between sequences and no table is read.
 * For every sequence b, with L = cache_seqlens[b] (read only):
 *  1. append: k_new[b], v_new[b] are copied bit for bit to [b, L];
 *  2. attend: out[b, h] = softmax(q[b, h] . K_j * scale) V_j over positions
 *     j = 0..L of row b.
 * L + 1 > max_seqlen (or L < 0) sets PA_DEVERR_OVERFLOW and zeroes the
 * sequence's output.  Positions past L of a row are never used in the
 * result (whatever they hold).  bf16 only (dtype PA_BF16 implied); head_dim
 * 64 or 128; num_heads / num_kv_heads <= 8; batch * max_seqlen < 2^31.
 * workspace: as pa_decode, at least pa_decode_contiguous_workspace_size(...)
 * bytes, zero-filled before first use.  For the same logical cache contents,
 * the result equals pa_decode's with block_size 16 (head_dim 128) or 32
 * (head_dim 64) bit for bit.
 */
size_t pa_decode_contiguous_workspace_size(int batch, int num_heads, int num_kv_heads,
                                           int head_dim);
int pa_decode_contiguous(const void *q, void *k_cache, void *v_cache,
                         const int32_t *cache_seqlens, const void *k_new, const void *v_new,
                         void *out, int batch, int num_heads, int num_kv_heads, int head_dim,
                         int max_seqlen, float softmax_scale, void *workspace,
                         size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * Varlen cache update ("Jalur Varlen" -> "Perilaku cache").
 *
 * k_chunk, v_chunk [total_q, num_kv_heads, head_dim]: the new tokens of all
 * requests, packed by cu_seq_lens_q [batch + 1].  Row i of request b is
 * copied bit for bit into the pool at logical position cache_seqlens[b] + i
 * (cache_seqlens = tokens already cached, read only).
 *
 * If k_full, v_full and cu_seq_lens_k are all non-NULL, request b's rows
 * [cu_seq_lens_k[b], cu_seq_lens_k[b+1]) of k_full/v_full [total_k,
 * num_kv_heads, head_dim] also receive its whole key sequence in logical
 * order: the cached prefix read from the pool, then the chunk.  That
 * requires cu_seq_lens_k[b+1] - cu_seq_lens_k[b] == cache_seqlens[b] +
 * (cu_seq_lens_q[b+1] - cu_seq_lens_q[b]) (PA_DEVERR_BAD_CU otherwise).
 * All three NULL: scatter only.  total_k is ignored then.
 */
int pa_cache_update(const void *k_chunk, const void *v_chunk, const int32_t *cu_seq_lens_q,
                    const int32_t *cache_seqlens, const int32_t *block_table, void *k_cache,
                    void *v_cache, void *k_full, void *v_full, const int32_t *cu_seq_lens_k,
                    int batch, int total_q, int total_k, int num_kv_heads, int head_dim,
                    int num_blocks, int block_size, int max_blocks_per_seq, pa_dtype dtype,
                    int32_t *dev_err, void *stream);

/*
 * Varlen attention ("Jalur Varlen").  Request r owns q rows
 * [cu_seq_lens_q[r], cu_seq_lens_q[r+1]) and k/v rows [cu_seq_lens_k[r],
 * cu_seq_lens_k[r+1]); max_length_q / max_length_k must be at least the
 * largest q / k length (they size the launch).  causal != 0 masks
 * bottom-right: query i of a request with lengths (ql, kl) sees key j iff
 * j <= i + kl - ql.  A query that sees no key gets a zero output row.
 * PA_BF16 runs on the tcgen05 tensor cores and needs head_dim 128
 * (head_dim 64 returns PA_ERR_UNSUPPORTED); PA_F32 runs on CUDA cores with
 * head_dim 64 or 128.
 */
int pa_varlen(const void *q, const void *k, const void *v, const int32_t *cu_seq_lens_q,
              const int32_t *cu_seq_lens_k, int max_length_q, int max_length_k, int causal,
              void *out, int batch, int total_q, int total_k, int num_heads, int num_kv_heads,
              int head_dim, pa_dtype dtype, float softmax_scale, int32_t *dev_err, void *stream);

/*
 * Varlen attention that reads each request's keys straight from the paged
 * pool through its block_table row, with no packed copy: "Perhatian
 * berhalaman", section "Jalur Varlen" -> "Perilaku cache" names the manual
 * cache read of the varlen path as a bottleneck at long lengths, and
 * "39 · PagedAttention" (inference-notes), section "Ghi chú", notes that
 * attention kernels can take the block table directly.  Typical use: scatter
 * the new chunk with pa_cache_update (k_full/v_full NULL), then call this.
 *
 * Request r owns q rows [cu_seq_lens_q[r], cu_seq_lens_q[r+1]) of q/out
 * [total_q, num_heads, head_dim]; its keys are logical positions
 * 0 .. seqlens_k[r]-1 of block_table row r in k_cache/v_cache
 * [num_blocks, block_size, num_kv_heads, head_dim].  Masking, scaling, GQA
 * mapping and empty rows as pa_varlen; for equal inputs the result equals
 * pa_varlen on the gathered keys bit for bit.  seqlens_k[r] beyond
 * max_blocks_per_seq * block_size sets PA_DEVERR_OVERFLOW and zeroes the
 * request's rows; a needed entry that is not a valid block sets
 * PA_DEVERR_BAD_BLOCK and zeroes the affected query tiles.
 * Supported: PA_BF16, head_dim 128, block_size 8, 16, 32 or 64.
 */
int pa_varlen_paged(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_table, const int32_t *cu_seq_lens_q,
                    const int32_t *seqlens_k, int max_length_q, int max_length_k, int causal,
                    void *out, int batch, int total_q, int num_heads, int num_kv_heads,
                    int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
                    pa_dtype dtype, float softmax_scale, int32_t *dev_err, void *stream);

/* Static description of a status code (never NULL). */
const char *pa_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
