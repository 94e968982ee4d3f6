// pa_block_manager.cpp -- host-side KV block manager: free list, reference
// counts, on-demand allocation and copy-on-write (include/pa_block_manager.h).
#include <new>
#include <stdint.h>
#include <unordered_map>
#include <vector>

#include "pa_block_manager.h"
#include "pagedattn.h"

struct pa_block_manager {
    struct Seq {
        std::vector<int32_t> blocks;   // logical -> physical
        int64_t len = 0;               // tokens
    };
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_list;    // stack; back() is handed out next
    std::vector<int32_t> refs;         // per block
    std::unordered_map<int64_t, Seq> seqs;
    int64_t allocations = 0, releases = 0, cow_copies = 0;

    int32_t take()
    {
        const int32_t b = free_list.back();
        free_list.pop_back();
        refs[b] = 1;
        ++allocations;
        return b;
    }

    void drop(int32_t b)
    {
        if (--refs[b] == 0) {
            free_list.push_back(b);
            ++releases;
        }
    }
};

extern "C" {

pa_block_manager *pa_bm_create(int num_blocks, int block_size)
{
    if (num_blocks <= 0 || block_size <= 0)
        return nullptr;
    pa_block_manager *bm = new (std::nothrow) pa_block_manager;
    if (!bm)
        return nullptr;
    try {
        bm->num_blocks = num_blocks;
        bm->block_size = block_size;
        bm->refs.assign(num_blocks, 0);
        bm->free_list.reserve(num_blocks);
        for (int b = num_blocks - 1; b >= 0; --b)   // lowest id on top
            bm->free_list.push_back(b);
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

int pa_bm_add_sequence(pa_block_manager *bm, int64_t seq_id)
{
    if (!bm || bm->seqs.count(seq_id))
        return PA_ERR_INVALID_ARG;
    bm->seqs.emplace(seq_id, pa_block_manager::Seq{});
    return PA_OK;
}

int pa_bm_fork(pa_block_manager *bm, int64_t parent, int64_t child)
{
    if (!bm || bm->seqs.count(child))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq copy = it->second;
    for (int32_t b : copy.blocks)
        ++bm->refs[b];
    bm->seqs.emplace(child, std::move(copy));
    return PA_OK;
}

int pa_bm_append(pa_block_manager *bm, int64_t seq_id, int num_tokens, int64_t *slots,
                 int64_t *cow_pairs, int *num_cow)
{
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !slots))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq &s = it->second;
    const int bs = bm->block_size;
    if (num_cow)
        *num_cow = 0;
    if (num_tokens == 0)
        return PA_OK;
    // blocks needed: one per block boundary crossed, plus a copy when the
    // first token goes into a shared, partially filled last block
    const int64_t first = s.len, last = s.len + num_tokens - 1;
    const bool partial = first % bs != 0;
    const bool cow = partial && bm->refs[s.blocks.back()] > 1;
    const int64_t fresh = last / bs - (partial ? first / bs : first / bs - 1);
    if (fresh + (cow ? 1 : 0) > (int64_t)bm->free_list.size())
        return PA_ERR_OUT_OF_BLOCKS;
    if (cow && !cow_pairs)
        return PA_ERR_INVALID_ARG;
    if (cow) {
        const int32_t src = s.blocks.back();
        const int32_t dst = bm->take();
        bm->drop(src);
        s.blocks.back() = dst;
        cow_pairs[0] = src;
        cow_pairs[1] = dst;
        if (num_cow)
            *num_cow = 1;
        ++bm->cow_copies;
    }
    for (int i = 0; i < num_tokens; ++i) {
        const int64_t pos = s.len;
        if (pos % bs == 0)
            s.blocks.push_back(bm->take());
        slots[i] = (int64_t)s.blocks[pos / bs] * bs + pos % bs;
        ++s.len;
    }
    return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager *bm, int64_t seq_id)
{
    if (!bm)
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    // release in reverse order, so the blocks a sequence took last are
    // handed out first again
    for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b)
        bm->drop(*b);
    bm->seqs.erase(it);
    return PA_OK;
}

int pa_bm_block_table(const pa_block_manager *bm, int64_t seq_id, int32_t *table, int max_blocks,
                      int *num_blocks, int64_t *seq_len)
{
    if (!bm || max_blocks < 0 || (max_blocks > 0 && !table))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID_ARG;
    const auto &blocks = it->second.blocks;
    if ((int64_t)blocks.size() > max_blocks)
        return PA_ERR_INVALID_ARG;
    for (int i = 0; i < max_blocks; ++i)
        table[i] = i < (int)blocks.size() ? blocks[i] : -1;
    if (num_blocks)
        *num_blocks = (int)blocks.size();
    if (seq_len)
        *seq_len = it->second.len;
    return PA_OK;
}

int pa_bm_ref_count(const pa_block_manager *bm, int block)
{
    if (!bm || block < 0 || block >= bm->num_blocks)
        return -1;
    return bm->refs[block];
}

int pa_bm_get_stats(const pa_block_manager *bm, pa_bm_stats *st)
{
    if (!bm || !st)
        return PA_ERR_INVALID_ARG;
    st->num_blocks = bm->num_blocks;
    st->free_blocks = (int64_t)bm->free_list.size();
    st->num_sequences = (int64_t)bm->seqs.size();
    st->allocations = bm->allocations;
    st->releases = bm->releases;
    st->cow_copies = bm->cow_copies;
    int64_t shared = 0;
    for (int32_t r : bm->refs)
        shared += r > 1;
    st->shared_blocks = shared;
    return PA_OK;
}

}  // extern "C"
