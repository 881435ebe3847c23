/*
 * pa_blocks.h -- host-side block manager for the paged KV pool (C ABI).
 *
 * Keeps, on the host, which physical blocks of a pool of `num_blocks`
 * blocks belong to which sequence, and produces the block_table and
 * cache_seqlens arrays that pa_decode / pa_cache_update / pa_varlen_paged
 * read.  What it implements:
 *  - a sequence's logical block i maps to any physical block; a sequence of
 *    n cached tokens holds ceil(n / block_size) blocks, and one more block is
 *    taken only when a token no longer fits ("Perhatian berhalaman", HF
 *    transformers docs, section "Jalur decode" -> "Contoh": 30 + 1 fits one
 *    block of 32, 32 + 1 needs a second; "PagedAttention", paweldubiel.com,
 *    "Mechanizm i szczegóły": with 4 tokens per block the 5th token needs a
 *    second block and the prefix never moves);
 *  - a free list and per-block reference counts, so that full blocks of a
 *    common prefix are shared by several sequences and return to the free
 *    list only when the last user releases them ("Paged Attention", notes
 *    repo, sections 块分配策略 and 共享前缀; its Python sketches are not
 *    followed: they count blocks from capacity instead of tokens).
 *
 * Blocks are handed out lowest-index-first from the free list; the order
 * carries no meaning for the kernels (their results do not depend on where
 * blocks sit).  Only full blocks are ever shared, so every sequence's next
 * write position lies in a block it owns alone.
 *
 * Not thread safe: one manager per thread, or external locking.  All
 * functions return PA_BM_OK (0) or a negative PA_BM_ERR_* code and leave the
 * manager unchanged on error.
 */
#ifndef PA_BLOCKS_H_
#define PA_BLOCKS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

enum {
    PA_BM_OK = 0,
    PA_BM_ERR_ARGS = -1,     /* bad sizes or NULL pointers */
    PA_BM_ERR_NO_SEQ = -2,   /* unknown sequence id */
    PA_BM_ERR_EXISTS = -3,   /* sequence id already in use */
    PA_BM_ERR_NO_SPACE = -4, /* not enough free blocks */
    PA_BM_ERR_TOO_LONG = -5  /* more than max_blocks_per_seq blocks needed */
};

/* A manager for a pool of num_blocks blocks of block_size tokens; a sequence
 * may hold at most max_blocks_per_seq blocks.  NULL on bad sizes. */
pa_block_manager *pa_bm_create(int num_blocks, int block_size, int max_blocks_per_seq);
void pa_bm_destroy(pa_block_manager *bm);

/* New sequence holding num_tokens tokens (ceil(num_tokens / block_size)
 * fresh blocks). */
int pa_bm_add(pa_block_manager *bm, int64_t seq_id, int num_tokens);

/* New sequence `child` sharing the first shared_tokens tokens of `parent`:
 * the parent's full blocks inside that prefix are shared (reference count
 * + 1); shared_tokens must be a multiple of block_size and at most the
 * parent's length.  The child's length is shared_tokens. */
int pa_bm_fork(pa_block_manager *bm, int64_t parent, int64_t child, int shared_tokens);

/* Room for num_tokens more tokens at the end of the sequence: takes fresh
 * blocks as needed and advances the sequence's length by num_tokens.  The
 * new tokens occupy logical positions old_length .. old_length+n-1. */
int pa_bm_append(pa_block_manager *bm, int64_t seq_id, int num_tokens);

/* Drops the sequence; blocks whose reference count reaches 0 are freed. */
int pa_bm_free(pa_block_manager *bm, int64_t seq_id);

/* Free blocks, and the reference count of one block (0 = free, negative =
 * bad index). */
int pa_bm_num_free(const pa_block_manager *bm);
int pa_bm_refcount(const pa_block_manager *bm, int block);

/* Length (tokens) of a sequence, or a negative error. */
int pa_bm_length(const pa_block_manager *bm, int64_t seq_id);

/* Rows of block_table [n, max_blocks_per_seq] (int32, -1 padded) and the
 * lengths [n] of the sequences seq_ids[0..n-1], in that order (host
 * buffers owned by the caller). */
int pa_bm_tables(const pa_block_manager *bm, const int64_t *seq_ids, int n, int32_t *block_table,
                 int32_t *lengths);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCKS_H_ */
