// Host block pool: fixed-size physical blocks, per-sequence block tables,
// reference counts and copy-on-write of a shared last block.
//
// Behaviour follows "大模型部署.md" §2.1 "3. vLLM 调度策略与显存块管理"
// (can_allocate with a watermark; one physical block per logical block;
// append_slots: new block only when the last is full, copy-on-write when the
// last block is shared) and "【自用】AI infra相关" 二、vLLM (global free block
// list; block table; fork shares blocks by reference count).
//
// Two variants from the same section (BlockSpaceManager options): prefix
// caching (CachedBlockAllocator: full blocks shared by a hash of the whole
// token prefix, freed hashed blocks parked in an LRU evictor, a block filled
// by decoding promoted to an existing identical block) and a sliding window
// (logical block j >= W_b reuses table[j % W_b]).  The pages allow one or the
// other.
//
// The pool plans; it never touches device memory.  Slots it returns are
// block * block_size + row, fed to paged_kv_append; copy pairs it returns are
// fed to pkv_copy_blocks.
#include <algorithm>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

// FNV-1a, 64 bit (published offset basis and prime), over the bytes of the
// previous block's hash (8, little-endian) and the block's token ids (4 each,
// little-endian): the hash of a full block covers its whole prefix.
uint64_t chained_block_hash(uint64_t prev, const int32_t* tokens, int32_t n) {
    uint64_t h = 0xcbf29ce484222325ull;
    auto mix = [&h](uint8_t byte) {
        h ^= byte;
        h *= 0x100000001b3ull;
    };
    for (int i = 0; i < 8; ++i) mix(uint8_t(prev >> (8 * i)));
    for (int32_t t = 0; t < n; ++t) {
        const uint32_t v = uint32_t(tokens[t]);
        for (int i = 0; i < 4; ++i) mix(uint8_t(v >> (8 * i)));
    }
    return h;
}

}  // namespace

struct pkv_pool {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    int32_t watermark = 0;
    bool caching = false;
    int32_t ring = 0;                 // ring of a sliding-window pool in blocks (0: off)
    int32_t window = 0;               // the window in tokens (a multiple of block_size)
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> refs;        // reference count per physical block
    struct Seq {
        std::vector<int32_t> table;   // logical block -> physical block (ring with a window)
        int64_t len = 0;              // tokens
        std::vector<int32_t> tokens;  // prefix caching: token ids
        std::vector<uint64_t> hashes; // prefix caching: hash of each full block
    };
    std::unordered_map<int64_t, Seq> seqs;

    // ---- prefix caching state ----
    struct BlockInfo {
        bool hashed = false;
        uint64_t hash = 0;
        int64_t hashed_tokens = 0;
        int64_t last_accessed = 0;
        uint64_t parked = 0;          // order in which it entered the evictor
    };
    std::vector<BlockInfo> info;
    std::unordered_map<uint64_t, int32_t> cached;   // hash -> block (in use or parked)
    // evictor: oldest access first, then most hashed tokens, then parked first
    using EvictKey = std::tuple<int64_t, int64_t, uint64_t, int32_t>;
    std::set<EvictKey> evictor;
    int64_t clock = 0;
    uint64_t park_counter = 0;

    int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
    int64_t need_for(int64_t tokens) const {
        const int64_t b = blocks_for(tokens);
        return ring ? std::min<int64_t>(b, ring) : b;
    }
    int64_t num_free() const { return int64_t(free_stack.size()) + int64_t(evictor.size()); }

    EvictKey key_of(int32_t b) const {
        const BlockInfo& i = info[b];
        return EvictKey(i.last_accessed, -i.hashed_tokens, i.parked, b);
    }
    // a block with one reference: free list first, else the evictor gives one up
    int32_t take() {
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {
            b = std::get<3>(*evictor.begin());
            evictor.erase(evictor.begin());
            cached.erase(info[b].hash);
            info[b].hashed = false;
            info[b].hash = 0;
            info[b].hashed_tokens = 0;
        }
        refs[b] = 1;
        if (caching) info[b].last_accessed = clock;
        return b;
    }
    void release(int32_t b) {
        if (--refs[b] > 0) return;
        if (caching && info[b].hashed) {
            info[b].last_accessed = clock;
            info[b].parked = park_counter++;
            evictor.insert(key_of(b));
        } else {
            free_stack.push_back(b);
        }
    }
    // the block registered under h with one more reference, or -1
    int32_t lookup(uint64_t h) {
        auto it = cached.find(h);
        if (it == cached.end()) return -1;
        const int32_t b = it->second;
        if (refs[b] == 0) evictor.erase(key_of(b));
        refs[b] += 1;
        info[b].last_accessed = clock;
        return b;
    }
    void register_block(int32_t b, uint64_t h, int64_t tokens) {
        info[b].hashed = true;
        info[b].hash = h;
        info[b].hashed_tokens = tokens;
        cached[h] = b;
    }
    int admission(int64_t need) const {
        if (int64_t(num_blocks) - need < watermark) return PKV_ERR_NEVER;
        if (num_free() - need >= watermark) return PKV_OK;
        return PKV_ERR_NO_BLOCKS;
    }
    int64_t slot(const Seq& s, int64_t pos) const {
        int64_t j = pos / block_size;
        if (ring) j %= ring;
        return int64_t(s.table[j]) * block_size + pos % block_size;
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

static int create_pool(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                       const int32_t* free_order, int32_t flags, int32_t sliding_window,
                       int32_t max_chunk, pkv_pool** out) {
    if (!out || num_blocks < 1 || block_size < 1 || watermark_blocks < 0 || sliding_window < 0 ||
        max_chunk < 1 || (flags & ~PKV_POOL_PREFIX_CACHING))
        return PKV_ERR_INVALID;
    *out = nullptr;
    if ((flags & PKV_POOL_PREFIX_CACHING) && sliding_window > 0) return PKV_ERR_UNSUPPORTED;
    if (sliding_window > 0 && sliding_window % block_size) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    pkv_pool* p = new pkv_pool;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->watermark = watermark_blocks;
    p->caching = (flags & PKV_POOL_PREFIX_CACHING) != 0;
    p->window = sliding_window;
    // the window's blocks, plus room for the keys a chunk of max_chunk queries
    // needs beyond the window of its first query
    p->ring = sliding_window > 0
                  ? sliding_window / block_size + (max_chunk - 1 + block_size - 1) / block_size
                  : 0;
    p->refs.assign(num_blocks, 0);
    if (p->caching) p->info.assign(num_blocks, pkv_pool::BlockInfo());
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

int pkv_pool_create_ex(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                       const int32_t* free_order, int32_t flags, int32_t sliding_window,
                       pkv_pool** out) {
    return create_pool(num_blocks, block_size, watermark_blocks, free_order, flags,
                       sliding_window, 1, out);
}

int pkv_pool_create_window(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                           const int32_t* free_order, int32_t sliding_window, int32_t max_chunk,
                           pkv_pool** out) {
    if (sliding_window < 1) return PKV_ERR_INVALID;
    return create_pool(num_blocks, block_size, watermark_blocks, free_order, 0, sliding_window,
                       max_chunk, out);
}

int pkv_pool_create(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                    const int32_t* free_order, pkv_pool** out) {
    return create_pool(num_blocks, block_size, watermark_blocks, free_order, 0, 0, 1, out);
}

int pkv_pool_destroy(pkv_pool* pool) {
    delete pool;
    return PKV_OK;
}

int pkv_pool_num_free(const pkv_pool* pool, int32_t* out) {
    if (!pool || !out) return PKV_ERR_INVALID;
    *out = int32_t(pool->num_free());
    return PKV_OK;
}

int pkv_pool_num_evictable(const pkv_pool* pool, int32_t* out) {
    if (!pool || !out) return PKV_ERR_INVALID;
    *out = int32_t(pool->evictor.size());
    return PKV_OK;
}

int pkv_pool_set_clock(pkv_pool* pool, int64_t now) {
    if (!pool) return PKV_ERR_INVALID;
    pool->clock = now;
    return PKV_OK;
}

int pkv_pool_can_allocate(const pkv_pool* pool, int32_t num_tokens) {
    if (!pool || num_tokens < 1) return PKV_ERR_INVALID;
    return pool->admission(pool->need_for(num_tokens));
}

static int add_sequence(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                        int32_t num_tokens, int64_t* slots_out, int32_t* num_cached_out) {
    if (pool->seqs.count(seq_id)) return PKV_ERR_INVALID;
    const int64_t need = pool->need_for(num_tokens);
    const int st = pool->admission(need);
    if (st != PKV_OK) return st;
    const int32_t bs = pool->block_size;
    pkv_pool::Seq s;
    s.table.reserve(need);
    s.len = num_tokens;
    if (pool->caching) {
        s.tokens.assign(token_ids, token_ids + num_tokens);
        s.hashes.reserve(num_tokens / bs);
    }
    auto& entry = pool->seqs[seq_id];  // may throw before any block is taken
    int64_t leading = 0;
    bool run = true;
    for (int64_t j = 0; j < need; ++j) {
        int32_t b;
        if (pool->caching && (j + 1) * bs <= num_tokens) {
            const uint64_t prev = j > 0 ? s.hashes[j - 1] : 0;
            const uint64_t h = chained_block_hash(prev, token_ids + j * bs, bs);
            s.hashes.push_back(h);
            b = pool->lookup(h);
            if (b < 0) {
                run = false;
                b = pool->take();
                pool->register_block(b, h, (j + 1) * bs);
            } else if (run) {
                ++leading;
            }
        } else {
            run = false;
            b = pool->take();
        }
        s.table.push_back(b);
    }
    if (slots_out) {
        // a token whose ring slot a later token of the same prompt takes is skipped
        const int64_t capacity = int64_t(pool->ring) * bs;
        for (int64_t p = 0; p < num_tokens; ++p)
            slots_out[p] = (capacity && p + capacity < num_tokens) ? -1 : pool->slot(s, p);
    }
    if (num_cached_out) *num_cached_out = int32_t(leading * bs);
    entry = std::move(s);
    return PKV_OK;
}

int pkv_seq_add(pkv_pool* pool, int64_t seq_id, int32_t num_tokens, int64_t* slots_out) {
    if (!pool || num_tokens < 1) return PKV_ERR_INVALID;
    if (pool->caching) return PKV_ERR_UNSUPPORTED;   // prefix caching needs the token ids
    PKV_GUARD_BEGIN
    return add_sequence(pool, seq_id, nullptr, num_tokens, slots_out, nullptr);
    PKV_GUARD_END
}

int pkv_seq_add_tokens(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                       int32_t num_tokens, int64_t* slots_out, int32_t* num_cached_out) {
    if (!pool || num_tokens < 1 || !token_ids) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    return add_sequence(pool, seq_id, token_ids, num_tokens, slots_out, num_cached_out);
    PKV_GUARD_END
}

int pkv_seq_fork(pkv_pool* pool, int64_t parent, int64_t child) {
    if (!pool) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    auto it = pool->seqs.find(parent);
    if (it == pool->seqs.end() || pool->seqs.count(child)) return PKV_ERR_INVALID;
    pkv_pool::Seq copy = it->second;
    auto& c = pool->seqs.emplace(child, std::move(copy)).first->second;
    for (int32_t b : c.table) pool->refs[b] += 1;
    return PKV_OK;
    PKV_GUARD_END
}

static int append_one(pkv_pool* pool, int64_t seq_id, int32_t token_id, int64_t* slot_out,
                      int32_t* cow_src, int32_t* cow_dst) {
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return PKV_ERR_INVALID;
    pkv_pool::Seq& s = it->second;
    const int64_t pos = s.len;  // logical position of the new token
    const int32_t bs = pool->block_size;
    const int64_t j = pos / bs;
    const int64_t r = pool->ring ? j % pool->ring : j;   // table entry the token goes to
    int32_t src = -1, dst = -1;
    if (pool->caching) {
        s.tokens.reserve(s.tokens.size() + 1);
        s.hashes.reserve(s.hashes.size() + 1);
    }
    if (pos % bs == 0 && r == int64_t(s.table.size())) {
        // every existing block is full: the token opens a new block
        if (pool->num_free() == 0) return PKV_ERR_NO_BLOCKS;
        s.table.reserve(s.table.size() + 1);
        s.table.push_back(pool->take());
    } else {
        const int32_t cur = s.table[r];
        if (pool->refs[cur] > 1) {
            // shared block: this sequence gets a private copy
            if (pool->num_free() == 0) return PKV_ERR_NO_BLOCKS;
            const int32_t fresh = pool->take();
            s.table[r] = fresh;
            pool->release(cur);
            src = cur;
            dst = fresh;
        }
    }
    s.len = pos + 1;
    if (pool->caching) {
        s.tokens.push_back(token_id);
        if ((pos + 1) % bs == 0) {
            // the block is full: share an identical one, or register this one
            const uint64_t prev = j > 0 ? s.hashes[j - 1] : 0;
            const uint64_t h = chained_block_hash(prev, s.tokens.data() + j * bs, bs);
            s.hashes.push_back(h);
            const int32_t found = pool->lookup(h);
            if (found >= 0) {
                pool->release(s.table[j]);
                s.table[j] = found;
                src = dst = -1;   // the found block already holds these tokens
            } else {
                pool->register_block(s.table[j], h, (j + 1) * bs);
            }
        }
    }
    *slot_out = pool->slot(s, pos);
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PKV_OK;
}

int pkv_seq_append_slot(pkv_pool* pool, int64_t seq_id, int64_t* slot_out, int32_t* cow_src,
                        int32_t* cow_dst) {
    if (!pool || !slot_out) return PKV_ERR_INVALID;
    if (pool->caching) return PKV_ERR_UNSUPPORTED;   // prefix caching needs the token id
    PKV_GUARD_BEGIN
    return append_one(pool, seq_id, 0, slot_out, cow_src, cow_dst);
    PKV_GUARD_END
}

int pkv_seq_append_token(pkv_pool* pool, int64_t seq_id, int32_t token_id, int64_t* slot_out,
                         int32_t* cow_src, int32_t* cow_dst) {
    if (!pool || !slot_out) return PKV_ERR_INVALID;
    PKV_GUARD_BEGIN
    return append_one(pool, seq_id, token_id, slot_out, cow_src, cow_dst);
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

int pkv_block_hash(const pkv_pool* pool, int32_t block, uint64_t* hash_out,
                   int32_t* hashed_out) {
    if (!pool || !hash_out || !hashed_out || block < 0 || block >= pool->num_blocks)
        return PKV_ERR_INVALID;
    const bool h = pool->caching && pool->info[block].hashed;
    *hashed_out = h ? 1 : 0;
    *hash_out = h ? pool->info[block].hash : 0;
    return PKV_OK;
}

int pkv_block_tables(const pkv_pool* pool, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                     int32_t* tables_out, int32_t* ctx_lens_out) {
    if (!pool || n < 0 || max_blocks < 1 || (n > 0 && (!seq_ids || !tables_out)))
        return PKV_ERR_INVALID;
    // the rotated export holds exactly the last `window` tokens only on a ring of
    // exactly the window's blocks
    if (pool->ring && pool->ring != pool->window / pool->block_size) return PKV_ERR_UNSUPPORTED;
    for (int32_t i = 0; i < n; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end()) return PKV_ERR_INVALID;
        if (int64_t(it->second.table.size()) > max_blocks) return PKV_ERR_INVALID;
    }
    const int32_t bs = pool->block_size;
    for (int32_t i = 0; i < n; ++i) {
        const pkv_pool::Seq& s = pool->seqs.find(seq_ids[i])->second;
        int32_t* row = tables_out + int64_t(i) * max_blocks;
        std::fill(row, row + max_blocks, -1);
        if (pool->ring) {
            // the last W_b logical blocks, in logical order, over the last `window` tokens
            const int64_t nb = pool->blocks_for(s.len);
            const int64_t first = std::max<int64_t>(0, nb - pool->ring);
            for (int64_t j = first; j < nb; ++j) row[j - first] = s.table[j % pool->ring];
            if (ctx_lens_out)
                ctx_lens_out[i] = int32_t(std::min<int64_t>(s.len, int64_t(pool->ring) * bs));
        } else {
            std::copy(s.table.begin(), s.table.end(), row);
            if (ctx_lens_out) ctx_lens_out[i] = int32_t(s.len);
        }
    }
    return PKV_OK;
}

int pkv_window_tables(const pkv_pool* pool, const int64_t* seq_ids, const int32_t* query_lens,
                      int32_t n, int32_t max_blocks, int32_t* tables_out, int32_t* ctx_lens_out) {
    if (!pool || n < 0 || max_blocks < 1 ||
        (n > 0 && (!seq_ids || !query_lens || !tables_out || !ctx_lens_out)))
        return PKV_ERR_INVALID;
    if (!pool->ring) return PKV_ERR_UNSUPPORTED;
    const int64_t bs = pool->block_size, capacity = int64_t(pool->ring) * bs;
    // validate everything before writing anything
    for (int32_t i = 0; i < n; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end()) return PKV_ERR_INVALID;
        const int64_t len = it->second.len, q = query_lens[i];
        if (q < 1 || q > len || q + pool->window - 1 > capacity) return PKV_ERR_INVALID;
        const int64_t first = std::max<int64_t>(0, len - q - pool->window + 1) / bs;
        if (pool->blocks_for(len) - first > max_blocks) return PKV_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        const pkv_pool::Seq& s = pool->seqs.find(seq_ids[i])->second;
        const int64_t first = std::max<int64_t>(0, s.len - query_lens[i] - pool->window + 1) / bs;
        const int64_t nb = pool->blocks_for(s.len);
        int32_t* row = tables_out + int64_t(i) * max_blocks;
        std::fill(row, row + max_blocks, -1);
        for (int64_t j = first; j < nb; ++j) row[j - first] = s.table[j % pool->ring];
        ctx_lens_out[i] = int32_t(s.len - first * bs);
    }
    return PKV_OK;
}

}  // extern "C"
