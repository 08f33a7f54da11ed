// Host block pool: fixed-size physical blocks, per-sequence block tables,
// reference counts and copy-on-write of a shared last block.
//
// Behaviour follows "大模型部署.md" §2.1 "3. vLLM 调度策略与显存块管理"
// (can_allocate with a watermark; one physical block per logical block;
// append_slots: new block only when the last is full, copy-on-write when the
// last block is shared) and "【自用】AI infra相关" 二、vLLM (global free block
// list; block table; fork shares blocks by reference count).
//
// The pool plans; it never touches device memory.  Slots it returns are
// block * block_size + row, fed to paged_kv_append; copy pairs it returns are
// fed to pkv_copy_blocks.
#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pkv_pool {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    int32_t watermark = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> refs;        // reference count per physical block
    struct Seq {
        std::vector<int32_t> table;   // logical block -> physical block
        int64_t len = 0;              // tokens
    };
    std::unordered_map<int64_t, Seq> seqs;

    int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }

    int32_t take() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        refs[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--refs[b] == 0) free_stack.push_back(b);
    }
    int admission(int64_t need) const {
        if (int64_t(num_blocks) - need < watermark) return PKV_ERR_NEVER;
        if (int64_t(free_stack.size()) - need >= watermark) return PKV_OK;
        return PKV_ERR_NO_BLOCKS;
    }
};

#define PKV_GUARD_BEGIN try {
#define PKV_GUARD_END                      \
    }                                      \
    catch (const std::bad_alloc&) {        \
        return PKV_ERR_HOST;               \
    }                                      \
    catch (...) {                          \
        return PKV_ERR_INVALID;            \
    }

extern "C" {

int pkv_pool_create(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                    const int32_t* free_order, pkv_pool** out) {
    if (!out || num_blocks < 1 || block_size < 1 || watermark_blocks < 0) return PKV_ERR_INVALID;
    *out = nullptr;
    PKV_GUARD_BEGIN
    pkv_pool* p = new pkv_pool;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->watermark = watermark_blocks;
    p->refs.assign(num_blocks, 0);
    p->free_stack.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return PKV_ERR_INVALID;
            }
            seen[b] = 1;
            // first listed is handed out first: it sits at the back of the stack
            p->free_stack[num_blocks - 1 - i] = b;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) p->free_stack[num_blocks - 1 - i] = i;
    }
    *out = p;
    return PKV_OK;
    PKV_GUARD_END
}

int pkv_pool_destroy(pkv_pool* pool) {
    delete pool;
    return PKV_OK;
}

int pkv_pool_num_free(const pkv_pool* pool, int32_t* out) {
    if (!pool || !out) return PKV_ERR_INVALID;
    *out = int32_t(pool->free_stack.size());
    return PKV_OK;
}

int pkv_pool_can_allocate(const pkv_pool* pool, int32_t num_tokens) {
    if (!pool || num_tokens < 1) return PKV_ERR_INVALID;
    return pool->admission(pool->blocks_for(num_tokens));
}

int pkv_seq_add(pkv_pool* pool, int64_t seq_id, int32_t num_tokens, int64_t* slots_out) {
    if (!pool || num_tokens < 1) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    if (pool->seqs.count(seq_id)) return PKV_ERR_INVALID;
    const int64_t need = pool->blocks_for(num_tokens);
    const int st = pool->admission(need);
    if (st != PKV_OK) return st;
    pkv_pool::Seq s;
    s.table.reserve(need);
    s.len = num_tokens;
    auto& slot = pool->seqs[seq_id];  // may throw before any block is taken
    for (int64_t j = 0; j < need; ++j) s.table.push_back(pool->take());
    if (slots_out) {
        for (int64_t p = 0; p < num_tokens; ++p)
            slots_out[p] = int64_t(s.table[p / pool->block_size]) * pool->block_size +
                           p % pool->block_size;
    }
    slot = std::move(s);
    return PKV_OK;
    PKV_GUARD_END
}

int pkv_seq_fork(pkv_pool* pool, int64_t parent, int64_t child) {
    if (!pool) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    auto it = pool->seqs.find(parent);
    if (it == pool->seqs.end() || pool->seqs.count(child)) return PKV_ERR_INVALID;
    pkv_pool::Seq copy = it->second;
    pool->seqs.emplace(child, std::move(copy));
    for (int32_t b : pool->seqs[child].table) pool->refs[b] += 1;
    return PKV_OK;
    PKV_GUARD_END
}

int pkv_seq_append_slot(pkv_pool* pool, int64_t seq_id, int64_t* slot_out, int32_t* cow_src,
                        int32_t* cow_dst) {
    if (!pool || !slot_out) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return PKV_ERR_INVALID;
    pkv_pool::Seq& s = it->second;
    const int64_t pos = s.len;  // logical position of the new token
    const int32_t bs = pool->block_size;
    int32_t src = -1, dst = -1;
    if (pos % bs == 0) {
        // every existing block is full: the token opens a new logical block
        if (pool->free_stack.empty()) return PKV_ERR_NO_BLOCKS;
        s.table.reserve(s.table.size() + 1);
        s.table.push_back(pool->take());
    } else {
        const int32_t last = s.table.back();
        if (pool->refs[last] > 1) {
            // shared partial block: this sequence gets a private copy
            if (pool->free_stack.empty()) return PKV_ERR_NO_BLOCKS;
            const int32_t fresh = pool->take();
            s.table.back() = fresh;
            pool->release(last);
            src = last;
            dst = fresh;
        }
    }
    s.len = pos + 1;
    *slot_out = int64_t(s.table[pos / bs]) * bs + pos % bs;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PKV_OK;
    PKV_GUARD_END
}

int pkv_seq_free(pkv_pool* pool, int64_t seq_id) {
    if (!pool) return PKV_ERR_INVALID;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return PKV_ERR_INVALID;
    for (int32_t b : it->second.table) pool->release(b);
    pool->seqs.erase(it);
    return PKV_OK;
}

int pkv_seq_len(const pkv_pool* pool, int64_t seq_id, int32_t* len_out) {
    if (!pool || !len_out) return PKV_ERR_INVALID;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return PKV_ERR_INVALID;
    *len_out = int32_t(it->second.len);
    return PKV_OK;
}

int pkv_block_ref_count(const pkv_pool* pool, int32_t block, int32_t* out) {
    if (!pool || !out || block < 0 || block >= pool->num_blocks) return PKV_ERR_INVALID;
    *out = pool->refs[block];
    return PKV_OK;
}

int pkv_block_tables(const pkv_pool* pool, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                     int32_t* tables_out, int32_t* ctx_lens_out) {
    if (!pool || n < 0 || max_blocks < 1 || (n > 0 && (!seq_ids || !tables_out)))
        return PKV_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end()) return PKV_ERR_INVALID;
        if (int64_t(it->second.table.size()) > max_blocks) return PKV_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        const pkv_pool::Seq& s = pool->seqs.find(seq_ids[i])->second;
        int32_t* row = tables_out + int64_t(i) * max_blocks;
        std::fill(row, row + max_blocks, -1);
        std::copy(s.table.begin(), s.table.end(), row);
        if (ctx_lens_out) ctx_lens_out[i] = int32_t(s.len);
    }
    return PKV_OK;
}

}  // extern "C"
