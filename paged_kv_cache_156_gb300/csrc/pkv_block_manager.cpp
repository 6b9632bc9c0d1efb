// Host block manager: the allocator that owns a pool's physical blocks and
// produces the decode step's inputs (block tables, sequence lengths, slots)
// and copy-on-write pairs.
//
// "LLM 推理引擎内部原理" §2.3 (BlockEngine: a FIFO list of free blocks; allocate
// takes ceil(tokens / block_size) blocks from its front; append_slot returns
// the slot of a sequence's next token, taking a new block when the last one
// is full, or reports that none is left so the scheduler can preempt; free
// returns a sequence's blocks to the back of the list) and §3.3 (forked
// samples share their prefix blocks); "vLLM核心概念" §4.2.2 (a writer to a
// shared block copies it first); tbr8.org PagedAttention article §五 (shared
// blocks carry a reference count and are not freed while it is above 1).
//
// Not thread-safe: one manager is driven by one host thread.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <deque>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pkv.h"
#include "pkv_internal.h"

struct pkv_block_manager {
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t num_tokens = 0;
    };
    int64_t num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Seq> seqs;
};

namespace {

pkv_status err(pkv_status st, const char* msg) { return static_cast<pkv_status>(pkv::set_error_message(st, msg)); }

// ceil(tokens / bs) without forming tokens + bs - 1, which overflows near INT64_MAX
int64_t blocks_for(int64_t tokens, int bs) { return tokens / bs + (tokens % bs != 0); }

}  // namespace

extern "C" {

pkv_block_manager* pkv_bm_create(int64_t num_blocks, int block_size, const int64_t* free_order) {
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
    if (free_order) {
        std::vector<char> seen(static_cast<size_t>(num_blocks), 0);
        for (int64_t i = 0; i < num_blocks; ++i) {
            const int64_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete bm;
                return nullptr;                  // not a permutation of the pool
            }
            seen[b] = 1;
            bm->free_list.push_back(static_cast<int32_t>(b));
        }
    } else {
        for (int64_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(static_cast<int32_t>(b));
    }
    return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) {
    return bm ? static_cast<int64_t>(bm->free_list.size()) : -1;
}

int64_t pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : it->second.num_tokens;
}

int pkv_bm_refcount(const pkv_block_manager* bm, int64_t block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    return bm->refcount[static_cast<size_t>(block)];
}

pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, int64_t num_tokens) {
    if (!bm) return err(PKV_ERR_INVALID, "null block manager");
    if (num_tokens < 0) return err(PKV_ERR_INVALID, "allocate: num_tokens < 0");
    if (bm->seqs.count(seq_id)) return err(PKV_ERR_INVALID, "allocate: sequence id already present");
    const int64_t nb = blocks_for(num_tokens, bm->block_size);
    if (nb > static_cast<int64_t>(bm->free_list.size())) return err(PKV_ERR_OOM, "allocate: not enough free blocks");
    pkv_block_manager::Seq sq;
    sq.num_tokens = num_tokens;
    sq.blocks.reserve(static_cast<size_t>(nb));
    for (int64_t i = 0; i < nb; ++i) {
        const int32_t b = bm->free_list.front();
        bm->free_list.pop_front();
        bm->refcount[b] = 1;
        sq.blocks.push_back(b);
    }
    bm->seqs.emplace(seq_id, std::move(sq));
    return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
    if (!bm) return err(PKV_ERR_INVALID, "null block manager");
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return err(PKV_ERR_INVALID, "fork: unknown parent sequence");
    if (bm->seqs.count(child_id)) return err(PKV_ERR_INVALID, "fork: child id already present");
    pkv_block_manager::Seq child = it->second;   // shares every block
    for (int32_t b : child.blocks) ++bm->refcount[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PKV_OK;
}

pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return err(PKV_ERR_INVALID, "null block manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return err(PKV_ERR_INVALID, "free: unknown sequence");
    for (int32_t b : it->second.blocks)
        if (--bm->refcount[b] == 0) bm->free_list.push_back(b);
    bm->seqs.erase(it);
    return PKV_OK;
}

pkv_status pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int64_t n, int64_t* slots,
                               int64_t* cow_pairs, int64_t cow_capacity, int64_t* num_cow) {
    if (!bm) return err(PKV_ERR_INVALID, "null block manager");
    if (n < 0 || (n > 0 && (!seq_ids || !slots)) || !num_cow)
        return err(PKV_ERR_INVALID, "append_slots: bad arguments");
    const int bs = bm->block_size;
    // check first, change nothing unless every sequence can take its token
    std::unordered_set<int64_t> seen;
    std::unordered_map<int32_t, int64_t> writers;               // shared partly filled last block -> listed holders
    int64_t need_blocks = 0, need_cow = 0;
    for (int64_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return err(PKV_ERR_INVALID, "append_slots: unknown sequence");
        if (!seen.insert(seq_ids[i]).second) return err(PKV_ERR_INVALID, "append_slots: sequence listed twice");
        const auto& sq = it->second;
        if (sq.num_tokens % bs == 0) {
            ++need_blocks;                                       // the last block is full (or none yet)
        } else if (bm->refcount[sq.blocks.back()] > 1) {
            ++writers[sq.blocks.back()];
        }
    }
    // A shared partly filled block with r holders, k of them listed: each listed
    // holder copies it while another sequence still holds it, so the last of all
    // r holders writes in place: min(k, r - 1) copies.
    for (const auto& w : writers) {
        const int64_t copies = std::min<int64_t>(w.second, bm->refcount[w.first] - 1);
        need_blocks += copies;
        need_cow += copies;
    }
    if (need_cow > 0 && (!cow_pairs || cow_capacity < need_cow))
        return err(PKV_ERR_INVALID, "append_slots: cow_pairs buffer too small");
    if (need_blocks > static_cast<int64_t>(bm->free_list.size()))
        return err(PKV_ERR_OOM, "append_slots: not enough free blocks (preempt a sequence)");
    int64_t ncow = 0;
    for (int64_t i = 0; i < n; ++i) {
        auto& sq = bm->seqs[seq_ids[i]];
        const int64_t off = sq.num_tokens % bs;
        if (off == 0) {
            const int32_t b = bm->free_list.front();
            bm->free_list.pop_front();
            bm->refcount[b] = 1;
            sq.blocks.push_back(b);
        } else if (bm->refcount[sq.blocks.back()] > 1) {
            const int32_t src = sq.blocks.back();
            const int32_t dst = bm->free_list.front();
            bm->free_list.pop_front();
            bm->refcount[dst] = 1;
            --bm->refcount[src];
            sq.blocks.back() = dst;
            cow_pairs[2 * ncow] = src;
            cow_pairs[2 * ncow + 1] = dst;
            ++ncow;
        }
        slots[i] = static_cast<int64_t>(sq.blocks.back()) * bs + off;
        ++sq.num_tokens;
    }
    *num_cow = ncow;
    return PKV_OK;
}

pkv_status pkv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int64_t n, int32_t* tables,
                               int max_blocks_per_seq, int32_t pad, int32_t* seq_lens) {
    if (!bm) return err(PKV_ERR_INVALID, "null block manager");
    if (n < 0 || (n > 0 && (!seq_ids || !tables || !seq_lens)) || max_blocks_per_seq < 0)
        return err(PKV_ERR_INVALID, "block_tables: bad arguments");
    for (int64_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return err(PKV_ERR_INVALID, "block_tables: unknown sequence");
        if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks_per_seq)
            return err(PKV_ERR_INVALID, "block_tables: max_blocks_per_seq too small");
        if (it->second.num_tokens > INT32_MAX)
            return err(PKV_ERR_INVALID, "block_tables: a sequence length does not fit int32 seq_lens");
    }
    for (int64_t i = 0; i < n; ++i) {
        const auto& sq = bm->seqs.find(seq_ids[i])->second;
        int32_t* row = tables + i * max_blocks_per_seq;
        const size_t nb = sq.blocks.size();
        if (nb) memcpy(row, sq.blocks.data(), nb * sizeof(int32_t));
        for (int j = static_cast<int>(nb); j < max_blocks_per_seq; ++j) row[j] = pad;
        seq_lens[i] = static_cast<int32_t>(sq.num_tokens);
    }
    return PKV_OK;
}

}  // extern "C"
