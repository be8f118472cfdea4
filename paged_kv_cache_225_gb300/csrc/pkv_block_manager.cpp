// Host-side paged KV-cache block manager (declared in include/pkv.h).
//
// The "Inference optimization" lesson (section "PagedAttention") and section
// 3 of "Continuous Batching e PagedAttention no vLLM" describe the cache as a
// pool of fixed 16-token pages placed anywhere in memory, one page table per
// request, pages of a shared prompt stored once and referenced by every
// request that shares it, and a private copy made only when a request
// diverges (copy-on-write).  This file keeps that bookkeeping on the host and
// hands the GPU what it needs per step: slot ids for the cache write, (src,
// dst) page pairs for pkv_copy_blocks, and dense block tables for attention.
//
// Choices the pages leave open: the lowest free page id is taken first (any
// free page is valid; a fixed choice makes tables reproducible); a fork
// shares every page of the parent, the partly filled last page included, so
// only that page can need a copy (appends never touch earlier pages).  Every
// call either succeeds completely or changes nothing.
#include <climits>
#include <cstdint>
#include <functional>
#include <mutex>
#include <new>
#include <queue>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_manager {
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
    };
    int num_blocks = 0, block_size = 0, max_blocks = 0;
    std::vector<int32_t> ref;
    std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_ids;
    std::unordered_map<int32_t, Seq> seqs;
    std::mutex mu;

    int32_t take()
    {
        const int32_t b = free_ids.top();
        free_ids.pop();
        ref[b] = 1;
        return b;
    }
    void drop(int32_t b)
    {
        if (--ref[b] == 0)
            free_ids.push(b);
    }
    int64_t slot(const Seq &q, int64_t t) const
    {
        return static_cast<int64_t>(q.table[t / block_size]) * block_size + t % block_size;
    }
    // Appends one token to q (the caller checked the pool); the copy, if any,
    // goes to pair[0..1].  Returns whether a copy was recorded.
    bool append(Seq &q, int64_t *slot_out, int32_t *pair)
    {
        bool copied = false;
        if (q.len % block_size == 0) {
            q.table.push_back(take());
        } else {
            const int32_t last = q.table.back();
            if (ref[last] > 1) {
                const int32_t fresh = take();
                pair[0] = last;
                pair[1] = fresh;
                drop(last);
                q.table.back() = fresh;
                copied = true;
            }
        }
        *slot_out = slot(q, q.len);
        ++q.len;
        return copied;
    }
};

extern "C" {

pkv_status pkv_bm_create(int num_blocks, int block_size, int max_blocks_per_seq,
                         pkv_block_manager **out)
{
    if (!out || num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0)
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
    if (!bm)
        return PKV_ERR_NO_BLOCKS;
    try {
        bm->num_blocks = num_blocks;
        bm->block_size = block_size;
        bm->max_blocks = max_blocks_per_seq;
        bm->ref.assign(num_blocks, 0);
        std::vector<int32_t> ids(num_blocks);
        for (int i = 0; i < num_blocks; ++i)
            ids[i] = i;
        bm->free_ids = decltype(bm->free_ids)(std::greater<int32_t>(), std::move(ids));
    } catch (...) {
        delete bm;
        return PKV_ERR_NO_BLOCKS;
    }
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int pkv_bm_num_free(pkv_block_manager *bm)
{
    if (!bm)
        return -1;
    std::lock_guard<std::mutex> lock(bm->mu);
    return static_cast<int>(bm->free_ids.size());
}

int pkv_bm_ref_count(pkv_block_manager *bm, int block)
{
    if (!bm || block < 0 || block >= bm->num_blocks)
        return -1;
    std::lock_guard<std::mutex> lock(bm->mu);
    return bm->ref[block];
}

pkv_status pkv_bm_add(pkv_block_manager *bm, int seq_id, int num_tokens, int64_t *slots)
{
    if (!bm || num_tokens < 0)
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    if (bm->seqs.count(seq_id))
        return PKV_ERR_INVALID_ARG;
    const int64_t need = (static_cast<int64_t>(num_tokens) + bm->block_size - 1) / bm->block_size;
    if (need > bm->max_blocks)
        return PKV_ERR_INVALID_ARG;
    if (need > static_cast<int64_t>(bm->free_ids.size()))
        return PKV_ERR_NO_BLOCKS;
    try {
        pkv_block_manager::Seq q;
        q.table.reserve(static_cast<size_t>(need));
        for (int64_t i = 0; i < need; ++i)
            q.table.push_back(bm->take());
        q.len = num_tokens;
        if (slots)
            for (int64_t t = 0; t < num_tokens; ++t)
                slots[t] = bm->slot(q, t);
        bm->seqs.emplace(seq_id, std::move(q));
    } catch (...) {
        return PKV_ERR_NO_BLOCKS;
    }
    return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager *bm, int parent_id, int child_id)
{
    if (!bm)
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end() || bm->seqs.count(child_id))
        return PKV_ERR_INVALID_ARG;
    try {
        pkv_block_manager::Seq q = it->second;
        for (int32_t b : q.table)
            ++bm->ref[b];
        bm->seqs.emplace(child_id, std::move(q));
    } catch (...) {
        return PKV_ERR_NO_BLOCKS;
    }
    return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager *bm, const int32_t *seq_ids, int n, int64_t *slots,
                         int32_t *copy_pairs, int *num_copies)
{
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots || !copy_pairs)) || !num_copies)
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    // Validate everything and count the pages the appends take, in order, before
    // changing state.  An earlier append can drop a shared last page to one
    // reference (its sibling then writes in place), hence the running deltas.
    int64_t need = 0;
    try {
        std::unordered_map<int32_t, int> seen;
        std::unordered_map<int32_t, int32_t> dropped;
        for (int i = 0; i < n; ++i) {
            auto it = bm->seqs.find(seq_ids[i]);
            if (it == bm->seqs.end() || seen[seq_ids[i]]++)
                return PKV_ERR_INVALID_ARG;  // unknown or listed twice
            const pkv_block_manager::Seq &q = it->second;
            if (q.len % bm->block_size == 0) {
                if (static_cast<int64_t>(q.table.size()) + 1 > bm->max_blocks)
                    return PKV_ERR_INVALID_ARG;
                ++need;
            } else {
                const int32_t last = q.table.back();
                if (bm->ref[last] - dropped[last] > 1) {
                    ++need;
                    ++dropped[last];
                }
            }
        }
    } catch (...) {
        return PKV_ERR_NO_BLOCKS;
    }
    if (need > static_cast<int64_t>(bm->free_ids.size()))
        return PKV_ERR_NO_BLOCKS;
    int copies = 0;
    for (int i = 0; i < n; ++i) {
        pkv_block_manager::Seq &q = bm->seqs[seq_ids[i]];
        if (bm->append(q, slots + i, copy_pairs + 2 * copies))
            ++copies;
    }
    *num_copies = copies;
    return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager *bm, int seq_id)
{
    if (!bm)
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PKV_ERR_INVALID_ARG;
    for (int32_t b : it->second.table)
        bm->drop(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_bm_tables(pkv_block_manager *bm, const int32_t *seq_ids, int n,
                         int max_blocks_per_seq, int32_t *tables, int32_t *seq_lens)
{
    if (!bm || n < 0 || max_blocks_per_seq <= 0 || (n > 0 && (!seq_ids || !tables)))
        return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(bm->mu);
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() ||
            static_cast<int64_t>(it->second.table.size()) > max_blocks_per_seq ||
            it->second.len > INT32_MAX)
            return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i) {
        const pkv_block_manager::Seq &q = bm->seqs[seq_ids[i]];
        int32_t *row = tables + static_cast<size_t>(i) * max_blocks_per_seq;
        const int nb = static_cast<int>(q.table.size());
        for (int j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < nb ? q.table[j] : -1;
        if (seq_lens)
            seq_lens[i] = static_cast<int32_t>(q.len);
    }
    return PKV_OK;
}

}  // extern "C"
