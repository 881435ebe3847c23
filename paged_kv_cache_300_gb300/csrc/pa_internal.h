// Host-side interface between the C ABI (pa_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// ------------------------------------------------------------------ decode
struct DecodeArgs {
    const void *q;
    void *k_cache;
    void *v_cache;
    const int32_t *block_table;
    const int32_t *cache_seqlens;
    const void *k_new;
    const void *v_new;
    void *out;
    float *part;      // split-K partials (bf16 path)
    int32_t *tickets; // per (sequence, kv head) arrival counters (bf16 path)
    int32_t *dev_err;
    int batch, num_heads, num_kv_heads, num_blocks, max_blocks_per_seq;
    int max_seqlen;  // contiguous cache: rows per sequence (paged: unused)
    int group;       // num_heads / num_kv_heads
    int head_groups; // num_kv_heads / kv heads per CTA
    int nstages;
    float scale;      // softmax scale
    float scale_log2; // softmax scale * log2(e)
};

// Launch geometry of the bf16 decode kernel for one problem shape.
struct DecodePlan {
    int heads_per_cta; // kv heads handled by one CTA (one consumer warp each)
    int head_groups;
    int nstages;
    int ctas;          // persistent grid size (stream-K partitions)
    size_t smem_bytes;
    size_t part_floats; // partial buffer size in floats
    size_t ticket_ints;
};

// The decode workspace starts with a fixed-size region of merge counters
// (one int per sequence and kv head).  Only counter operations ever touch it
// and every call leaves its counters at zero, so a workspace zero-filled once
// stays valid for calls of any shape; the split-K partials follow it.
constexpr size_t kTicketRegionBytes = size_t(1) << 20;

// `contig`: the kernel variant over a contiguous cache [batch, max_seqlen,
// Hkv, D] with no block table (block_size is then its unit of tokens).
int decode_bf16_plan(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     DecodePlan *plan, bool contig = false);
size_t decode_workspace_bytes(const DecodePlan &plan);
int decode_bf16_launch(const DecodeArgs &a, int head_dim, int block_size, const DecodePlan &plan,
                       const CUtensorMap &tm_k, const CUtensorMap &tm_v, cudaStream_t s,
                       bool contig = false);
// Tokens per work unit of the contiguous decode variant: 16 for head_dim 128,
// 32 for head_dim 64 (a 64 KB ring stage for 8 kv heads either way).
constexpr int contig_unit(int head_dim) { return head_dim == 128 ? 16 : 32; }
// Host checks shared by the decode entry points: PA_OK, or the status the
// call must return before anything is launched.
int decode_check_pointers(const void *q, const void *k_cache, const void *v_cache,
                          const void *k_new, const void *v_new, const void *out);
int decode_f32_launch(const DecodeArgs &a, int head_dim, int block_size, cudaStream_t s);

// ------------------------------------------------------------------ cache update
struct CacheUpdateArgs {
    const void *k_chunk;
    const void *v_chunk;
    const int32_t *cu_q;
    const int32_t *prefix;
    const int32_t *block_table;
    void *k_cache;
    void *v_cache;
    void *k_full;
    void *v_full;
    const int32_t *cu_k;
    int32_t *dev_err;
    int batch, total_q, total_k, num_kv_heads, head_dim, num_blocks, block_size,
        max_blocks_per_seq;
    int row_bytes; // num_kv_heads * head_dim * element size
};
int cache_update_launch(const CacheUpdateArgs &a, cudaStream_t s);

// ------------------------------------------------------------------ varlen
struct VarlenArgs {
    const void *q;
    const void *k;
    const void *v;
    const int32_t *cu_q;
    const int32_t *cu_k;
    void *out;
    int32_t *dev_err;
    int batch, total_q, total_k, num_heads, num_kv_heads, head_dim, max_q, max_k, causal;
    float scale, scale_log2;
    // paged variant: keys of request r are logical positions 0..seqlens_k[r)-1
    // of block_table row r in the pool [num_blocks, block_size, Hkv, D]
    const int32_t *block_table;
    const int32_t *seqlens_k;
    int num_blocks, block_size, max_blocks_per_seq;
    // tensor-core kernel: query heads packed per 128-row tile (a power of two
    // dividing num_heads / num_kv_heads); a tile holds 128 / pack queries
    int pack;
    // 1 when the output tensor map was encoded, so that full tiles leave
    // through a TMA store
    int out_tma;
};
// Rows of one TMA box of the tensor-core varlen kernel: query tiles are 128
// rows, key/value tiles 64 rows.
constexpr int kVarlenQRows = 128;
constexpr int kVarlenKRows = 64;
int varlen_f32_launch(const VarlenArgs &a, cudaStream_t s);
int varlen_bf16_launch(const VarlenArgs &a, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                       const CUtensorMap &tm_v, const CUtensorMap &tm_o, cudaStream_t s);
int varlen_paged_bf16_launch(const VarlenArgs &a, const CUtensorMap &tm_q,
                             const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const CUtensorMap &tm_o, cudaStream_t s);

// ------------------------------------------------------------------ helpers
int num_sms();
int encode_rows_map(CUtensorMap *map, const void *base, uint64_t rows, int heads, int head_dim,
                    int box_rows);
int encode_unit_map(CUtensorMap *map, const void *base, uint64_t rows, int heads, int head_dim,
                    int box_rows, int box_heads);
int encode_packed_q_map(CUtensorMap *map, const void *base, uint64_t rows, int heads, int pack,
                        int box_queries);
int varlen_pack_factor(int num_heads, int num_kv_heads);

}  // namespace pa
