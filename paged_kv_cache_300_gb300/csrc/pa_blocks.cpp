// Host block manager for the paged KV pool: free list, reference counts,
// shared-prefix forks and block-table export (see include/pa_blocks.h).
#include "../../include/pa_blocks.h"

#include <cstring>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

struct pa_block_manager {
    struct Seq {
        std::vector<int> blocks;
        int length = 0;
    };
    int num_blocks, block_size, max_blocks;
    std::set<int> free_blocks;   // lowest index first
    std::vector<int> refcount;   // 0 = free
    std::unordered_map<int64_t, Seq> seqs;

    int blocks_for(long long tokens) const
    {
        return (int)((tokens + block_size - 1) / block_size);
    }

    // Takes n fresh blocks (caller checked availability).
    void take(int n, std::vector<int> &dst)
    {
        for (int i = 0; i < n; ++i) {
            const int b = *free_blocks.begin();
            free_blocks.erase(free_blocks.begin());
            refcount[b] = 1;
            dst.push_back(b);
        }
    }
};

extern "C" {

pa_block_manager *pa_bm_create(int num_blocks, int block_size, int max_blocks_per_seq)
{
    if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0) return nullptr;
    auto *bm = new (std::nothrow) pa_block_manager();
    if (bm == nullptr) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_blocks = max_blocks_per_seq;
    bm->refcount.assign(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) bm->free_blocks.insert(bm->free_blocks.end(), i);
    return bm;
}

void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

int pa_bm_add(pa_block_manager *bm, int64_t seq_id, int num_tokens)
{
    if (bm == nullptr || num_tokens < 0) return PA_BM_ERR_ARGS;
    if (bm->seqs.count(seq_id)) return PA_BM_ERR_EXISTS;
    const int need = bm->blocks_for(num_tokens);
    if (need > bm->max_blocks) return PA_BM_ERR_TOO_LONG;
    if (need > (int)bm->free_blocks.size()) return PA_BM_ERR_NO_SPACE;
    pa_block_manager::Seq s;
    bm->take(need, s.blocks);
    s.length = num_tokens;
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_BM_OK;
}

int pa_bm_fork(pa_block_manager *bm, int64_t parent, int64_t child, int shared_tokens)
{
    if (bm == nullptr || shared_tokens < 0 || shared_tokens % bm->block_size != 0)
        return PA_BM_ERR_ARGS;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return PA_BM_ERR_NO_SEQ;
    if (bm->seqs.count(child)) return PA_BM_ERR_EXISTS;
    if (shared_tokens > it->second.length) return PA_BM_ERR_ARGS;
    pa_block_manager::Seq s;
    const int nb = shared_tokens / bm->block_size;
    s.blocks.assign(it->second.blocks.begin(), it->second.blocks.begin() + nb);
    for (int b : s.blocks) ++bm->refcount[b];
    s.length = shared_tokens;
    bm->seqs.emplace(child, std::move(s));
    return PA_BM_OK;
}

int pa_bm_append(pa_block_manager *bm, int64_t seq_id, int num_tokens)
{
    if (bm == nullptr || num_tokens < 0) return PA_BM_ERR_ARGS;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_BM_ERR_NO_SEQ;
    auto &s = it->second;
    const int total = bm->blocks_for((long long)s.length + num_tokens);
    if (total > bm->max_blocks) return PA_BM_ERR_TOO_LONG;
    const int need = total - (int)s.blocks.size();
    if (need > (int)bm->free_blocks.size()) return PA_BM_ERR_NO_SPACE;
    if (need > 0) bm->take(need, s.blocks);
    s.length += num_tokens;
    return PA_BM_OK;
}

int pa_bm_free(pa_block_manager *bm, int64_t seq_id)
{
    if (bm == nullptr) return PA_BM_ERR_ARGS;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_BM_ERR_NO_SEQ;
    for (int b : it->second.blocks)
        if (--bm->refcount[b] == 0) bm->free_blocks.insert(b);
    bm->seqs.erase(it);
    return PA_BM_OK;
}

int pa_bm_num_free(const pa_block_manager *bm)
{
    return bm == nullptr ? PA_BM_ERR_ARGS : (int)bm->free_blocks.size();
}

int pa_bm_refcount(const pa_block_manager *bm, int block)
{
    if (bm == nullptr || block < 0 || block >= bm->num_blocks) return PA_BM_ERR_ARGS;
    return bm->refcount[block];
}

int pa_bm_length(const pa_block_manager *bm, int64_t seq_id)
{
    if (bm == nullptr) return PA_BM_ERR_ARGS;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? PA_BM_ERR_NO_SEQ : it->second.length;
}

int pa_bm_tables(const pa_block_manager *bm, const int64_t *seq_ids, int n, int32_t *block_table,
                 int32_t *lengths)
{
    if (bm == nullptr || n < 0 || (n > 0 && (seq_ids == nullptr || block_table == nullptr)))
        return PA_BM_ERR_ARGS;
    for (int i = 0; i < n; ++i)
        if (!bm->seqs.count(seq_ids[i])) return PA_BM_ERR_NO_SEQ;
    for (int i = 0; i < n; ++i) {
        const auto &s = bm->seqs.at(seq_ids[i]);
        int32_t *row = block_table + (size_t)i * bm->max_blocks;
        for (int j = 0; j < bm->max_blocks; ++j)
            row[j] = j < (int)s.blocks.size() ? s.blocks[j] : -1;
        if (lengths != nullptr) lengths[i] = s.length;
    }
    return PA_BM_OK;
}

}  // extern "C"
