// Host-side pool of KV-cache blocks ("Fast Attention Kernels and Operator
// Fusion", section "Paged Attention Kernels": blocks are allocated on
// demand, returned to a pool when a request ends, and shared when sequences
// have a common prefix; a logical sequence is a block table).
//
// Bookkeeping only: the pool hands out block ids and slot numbers for
// fa_cache_append and builds the block tables fa_paged_attn reads; it never
// touches device memory.  Every block has a reference count.  A block shared
// by several sequences (a common prefix) is always full, so nobody writes to
// it again: a fork shares the full blocks of the prefix and copies on write
// the block that holds a partial prefix tail (the caller performs that copy
// on the device with fa_copy_blocks before writing into the new sequence).
#include <mutex>
#include <new>
#include <vector>

#include "../../include/fattn.h"

namespace {
constexpr int kBS = 16;

struct Seq {
    bool live = false;
    int len = 0;
    std::vector<int> blocks;
};
}  // namespace

struct fa_block_pool {
    int num_blocks = 0, max_blocks = 0;
    std::vector<int> ref;       // reference count per block
    std::vector<int> free_list; // blocks with ref == 0 (taken from the back)
    std::vector<Seq> seqs;
    std::vector<int> free_ids;  // released sequence ids, reused first
    mutable std::mutex mu;

    int new_seq_id() {
        int id;
        if (!free_ids.empty()) {
            id = free_ids.back();
            free_ids.pop_back();
        } else {
            id = (int)seqs.size();
            seqs.emplace_back();
        }
        seqs[id] = Seq();
        seqs[id].live = true;
        return id;
    }
    bool valid(int s) const { return s >= 0 && s < (int)seqs.size() && seqs[s].live; }
    int take_block() {
        const int b = free_list.back();
        free_list.pop_back();
        ref[b] = 1;
        return b;
    }
    void drop_block(int b) {
        if (--ref[b] == 0) free_list.push_back(b);
    }
};

extern "C" {

fa_status fa_pool_create(fa_block_pool** pool, int num_blocks, int max_blocks_per_seq) {
    if (!pool) return FA_ERR_INVALID_ARG;
    *pool = nullptr;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0) return FA_ERR_INVALID_ARG;
    fa_block_pool* p = new (std::nothrow) fa_block_pool;
    if (!p) return FA_ERR_NO_BLOCKS;
    p->num_blocks = num_blocks;
    p->max_blocks = max_blocks_per_seq;
    p->ref.assign(num_blocks, 0);
    p->free_list.reserve(num_blocks);
    for (int b = num_blocks - 1; b >= 0; --b) p->free_list.push_back(b);  // block 0 is handed out first
    *pool = p;
    return FA_OK;
}

void fa_pool_destroy(fa_block_pool* pool) { delete pool; }

int fa_pool_num_free(const fa_block_pool* pool) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> lk(pool->mu);
    return (int)pool->free_list.size();
}

int fa_pool_refcount(const fa_block_pool* pool, int block) {
    if (!pool || block < 0 || block >= pool->num_blocks) return -1;
    std::lock_guard<std::mutex> lk(pool->mu);
    return pool->ref[block];
}

int fa_pool_seq_len(const fa_block_pool* pool, int seq) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> lk(pool->mu);
    return pool->valid(seq) ? pool->seqs[seq].len : -1;
}

fa_status fa_pool_add_seq(fa_block_pool* pool, int* seq) {
    if (!pool || !seq) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    *seq = pool->new_seq_id();
    return FA_OK;
}

fa_status fa_pool_fork(fa_block_pool* pool, int parent, int prefix_len, int* child, int* copy_src, int* copy_dst) {
    if (!pool || !child || !copy_src || !copy_dst) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    if (!pool->valid(parent) || prefix_len < 0 || prefix_len > pool->seqs[parent].len) return FA_ERR_INVALID_ARG;
    const int full = prefix_len / kBS, tail = prefix_len % kBS;
    if (tail && pool->free_list.empty()) return FA_ERR_NO_BLOCKS;
    const int id = pool->new_seq_id();
    Seq& c = pool->seqs[id];
    const Seq& par = pool->seqs[parent];  // (re-read: new_seq_id may have grown the vector)
    c.len = prefix_len;
    for (int i = 0; i < full; ++i) {
        c.blocks.push_back(par.blocks[i]);
        ++pool->ref[par.blocks[i]];
    }
    *copy_src = *copy_dst = -1;
    if (tail) {  // the prefix tail shares a block with tokens the child must not see written over
        const int b = pool->take_block();
        *copy_src = pool->seqs[parent].blocks[full];
        *copy_dst = b;
        pool->seqs[id].blocks.push_back(b);
    }
    *child = id;
    return FA_OK;
}

fa_status fa_pool_append(fa_block_pool* pool, int seq, int n, int32_t* slots) {
    if (!pool || n < 0 || (n > 0 && !slots)) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    if (!pool->valid(seq)) return FA_ERR_INVALID_ARG;
    Seq& s = pool->seqs[seq];
    const long new_len = (long)s.len + n;
    const long need_blocks = (new_len + kBS - 1) / kBS;
    if (need_blocks > pool->max_blocks) return FA_ERR_INVALID_ARG;
    const long extra = need_blocks - (long)s.blocks.size();
    if (extra > (long)pool->free_list.size()) return FA_ERR_NO_BLOCKS;  // all or nothing
    for (long i = 0; i < extra; ++i) s.blocks.push_back(pool->take_block());
    for (int i = 0; i < n; ++i) {
        const int t = s.len + i;
        slots[i] = s.blocks[t / kBS] * kBS + t % kBS;
    }
    s.len = (int)new_len;
    return FA_OK;
}

fa_status fa_pool_release(fa_block_pool* pool, int seq) {
    if (!pool) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    if (!pool->valid(seq)) return FA_ERR_INVALID_ARG;
    Seq& s = pool->seqs[seq];
    for (int b : s.blocks) pool->drop_block(b);
    s = Seq();
    pool->free_ids.push_back(seq);
    return FA_OK;
}

fa_status fa_pool_tables(const fa_block_pool* pool, const int* seqs, int n, int32_t* table, int32_t* ctx_lens) {
    if (!pool || n < 0 || (n > 0 && (!seqs || !table || !ctx_lens))) return FA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    for (int i = 0; i < n; ++i)
        if (!pool->valid(seqs[i])) return FA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const Seq& s = pool->seqs[seqs[i]];
        for (int j = 0; j < pool->max_blocks; ++j)
            table[(long)i * pool->max_blocks + j] = j < (int)s.blocks.size() ? s.blocks[j] : -1;
        ctx_lens[i] = s.len;
    }
    return FA_OK;
}

}  // extern "C"
