// pkv_pool.cpp -- host-side pool of physical KV blocks with reference counts.
//
// PagedAttention keeps each sequence's KV cache in fixed-size blocks reached
// through a block table; blocks are handed out on demand, and several
// sequences can share a block -- a common prompt prefix, or the prompt of
// several sampled continuations -- with copy-on-write when one of them has to
// write into a shared block ("Inference Engines", The Breakthrough,
// PagedAttention paragraph; CS336 lecture-10 notes, PagedAttention (vLLM);
// "Transformer inference mechanics", FlashAttention versus PagedAttention:
// on-demand allocation, sharing and copy-on-write).
//
// This is plain host bookkeeping: a LIFO free list and one reference count
// per block.  It never touches device memory; the copies it asks for are done
// by pkv_copy_blocks on the device.  Every call either succeeds completely or
// changes nothing.  A pool is not thread-safe: callers serialise access.
#include <cstdint>
#include <new>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_pool {
    int block_size;
    std::vector<int32_t> refcount;  // 0 = free
    std::vector<int32_t> free_list; // stack of free block ids
};

extern "C" {

pkv_block_pool* pkv_pool_create(int num_blocks, int block_size) {
    if (num_blocks < 1 || block_size < 1) return nullptr;
    pkv_block_pool* p = new (std::nothrow) pkv_block_pool;
    if (!p) return nullptr;
    p->block_size = block_size;
    p->refcount.assign(num_blocks, 0);
    p->free_list.reserve(num_blocks);
    for (int b = num_blocks - 1; b >= 0; --b) p->free_list.push_back(b);  // hands out 0, 1, ...
    return p;
}

void pkv_pool_destroy(pkv_block_pool* pool) { delete pool; }

int pkv_pool_num_free(const pkv_block_pool* pool) {
    return pool ? static_cast<int>(pool->free_list.size()) : -1;
}

int pkv_pool_refcount(const pkv_block_pool* pool, int block) {
    if (!pool || block < 0 || block >= static_cast<int>(pool->refcount.size())) return -1;
    return pool->refcount[block];
}

int pkv_pool_alloc(pkv_block_pool* pool, int n, int32_t* out_blocks) {
    if (!pool || n < 0 || (n > 0 && !out_blocks)) return PKV_ERR_INVALID_ARG;
    if (n > static_cast<int>(pool->free_list.size())) return PKV_ERR_OUT_OF_BLOCKS;
    for (int i = 0; i < n; ++i) {
        const int32_t b = pool->free_list.back();
        pool->free_list.pop_back();
        pool->refcount[b] = 1;
        out_blocks[i] = b;
    }
    return PKV_OK;
}

static bool valid_in_use(const pkv_block_pool* pool, const int32_t* blocks, int n) {
    for (int i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < 0 || b >= static_cast<int>(pool->refcount.size()) || pool->refcount[b] <= 0)
            return false;
    }
    return true;
}

int pkv_pool_share(pkv_block_pool* pool, const int32_t* blocks, int n) {
    if (!pool || n < 0 || (n > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
    if (!valid_in_use(pool, blocks, n)) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) ++pool->refcount[blocks[i]];
    return PKV_OK;
}

int pkv_pool_release(pkv_block_pool* pool, const int32_t* blocks, int n) {
    if (!pool || n < 0 || (n > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
    // O(n) work and no allocation: drop the counts one by one (the same id
    // may appear several times); if one would go below zero, put back the
    // drops already made and fail.
    const int num_blocks = static_cast<int>(pool->refcount.size());
    for (int i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < 0 || b >= num_blocks || pool->refcount[b] == 0) {
            for (int k = 0; k < i; ++k) ++pool->refcount[blocks[k]];
            return PKV_ERR_INVALID_ARG;
        }
        --pool->refcount[b];
    }
    // Blocks whose count reached zero join the free list once each (-1 marks
    // "already pushed" during this pass and is reset to 0 afterwards).
    for (int i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (pool->refcount[b] == 0) {
            pool->free_list.push_back(b);
            pool->refcount[b] = -1;
        }
    }
    for (int i = 0; i < n; ++i)
        if (pool->refcount[blocks[i]] < 0) pool->refcount[blocks[i]] = 0;
    return PKV_OK;
}

int pkv_pool_append_slots(pkv_block_pool* pool, int32_t* table, int* nblocks, int max_blocks,
                          int ctx, int n_new, int32_t* slot_out, int32_t* copy_pairs,
                          int* num_pairs) {
    if (!pool || !table || !nblocks || !slot_out || !num_pairs || max_blocks < 0 || ctx < 0 ||
        n_new < 0)
        return PKV_ERR_INVALID_ARG;
    const int bs = pool->block_size;
    const int have = *nblocks;
    // The table must hold every resident token (it may hold spare blocks too).
    if (have < 0 || have > max_blocks || (long long)have * bs < ctx) return PKV_ERR_INVALID_ARG;
    if (!valid_in_use(pool, table, have)) return PKV_ERR_INVALID_ARG;
    *num_pairs = 0;
    if (n_new == 0) return PKV_OK;
    const long long need_total = ((long long)ctx + n_new + bs - 1) / bs;
    if (need_total > max_blocks) return PKV_ERR_INVALID_ARG;
    // Blocks that receive a new token: [ctx / bs, need_total).  Those already
    // in the table must be owned exclusively (copy-on-write); the rest are new.
    const int first = ctx / bs;
    const int last = have < need_total ? have : static_cast<int>(need_total);  // existing, written
    int fresh = static_cast<int>(need_total) - have;  // blocks appended to the table
    int cow = 0;
    for (int j = first; j < last; ++j)
        if (pool->refcount[table[j]] > 1) ++cow;
    if (fresh < 0) fresh = 0;
    if (fresh + cow > static_cast<int>(pool->free_list.size())) return PKV_ERR_OUT_OF_BLOCKS;
    if (cow > 0 && !copy_pairs) return PKV_ERR_INVALID_ARG;
    // Apply: copy-on-write first, then new blocks, then the slots.
    for (int j = first; j < last; ++j) {
        const int32_t src = table[j];
        if (pool->refcount[src] > 1) {
            const int32_t dst = pool->free_list.back();
            pool->free_list.pop_back();
            pool->refcount[dst] = 1;
            --pool->refcount[src];
            copy_pairs[2 * *num_pairs] = src;
            copy_pairs[2 * *num_pairs + 1] = dst;
            ++*num_pairs;
            table[j] = dst;
        }
    }
    for (int j = have; j < need_total; ++j) {
        const int32_t b = pool->free_list.back();
        pool->free_list.pop_back();
        pool->refcount[b] = 1;
        table[j] = b;
    }
    *nblocks = static_cast<int>(need_total > have ? need_total : have);
    for (int i = 0; i < n_new; ++i) {
        const long long pos = (long long)ctx + i;
        slot_out[i] = table[pos / bs] * bs + static_cast<int32_t>(pos % bs);
    }
    return PKV_OK;
}

}  // extern "C"
