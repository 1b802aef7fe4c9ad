// pa_block_manager.cpp -- host block manager: the paged pool's allocator and
// prefix cache, producing the block tables the kernels consume.
//
// What it implements [NV12 §12.8 "BlockManager: 分页 KV Cache + Prefix
// Caching"; VS §1.1 and §1.2.4-1.2.5]:
//  * Blocks carry a reference count, the chained hash of the prefix up to and
//    including the block (or none) and the block's token ids.
//  * Free block ids form a FIFO queue (taken from the front, returned to the
//    back); used ids a set; a map goes from prefix hash to block id.
//  * Allocating a block takes the front of the queue, drops the map entry
//    that still names it (its content is about to change) and resets it.
//    Releasing a block keeps its hash and tokens, so a later request with the
//    same prefix can take it back while nobody has overwritten it.
//  * can_allocate walks the full blocks of a sequence except the last, while
//    the chained hash is in the map and the block there holds the same
//    tokens; blocks found in use need no free block.  allocate reuses those
//    blocks (a used one gains a reference; a free one leaves the queue), then
//    takes fresh blocks for the rest.  deallocate drops one reference per
//    block, last block first, releasing blocks that reach zero.
//  * A decode step needs a new block exactly when the sequence length is one
//    past a multiple of the block size (can_append / may_append).
//  * hash_blocks registers the blocks a step filled: blocks
//    [cached / B, (cached + scheduled) / B), chained from the hash of the
//    block before.
// The chained hash of a block is XXH64 (seed 0) over the previous block's
// 64-bit hash as 8 little-endian bytes (omitted for the first block) followed
// by the block's token ids as 64-bit little-endian integers.  XXH64 is written
// here from its published specification (xxHash, Y. Collet).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <deque>
#include <memory>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa.h"

namespace pa {
pa_status fail(pa_status s, const char *fmt, ...);
}

namespace {

// ---------------------------------------------------------------- XXH64
constexpr uint64_t P1 = 0x9E3779B185EBCA87ull, P2 = 0xC2B2AE3D27D4EB4Full, P3 = 0x165667B19E3779F9ull,
                   P4 = 0x85EBCA77C2B2AE63ull, P5 = 0x27D4EB2F165667C5ull;

inline uint64_t rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }
inline uint64_t rd64(const uint8_t *p) {
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];  // little-endian on any host
    return v;
}
inline uint32_t rd32(const uint8_t *p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
inline uint64_t round_(uint64_t acc, uint64_t lane) { return rotl(acc + lane * P2, 31) * P1; }
inline uint64_t merge_(uint64_t acc, uint64_t v) { return (acc ^ round_(0, v)) * P1 + P4; }

uint64_t xxh64(const uint8_t *p, size_t n, uint64_t seed) {
    const uint8_t *end = p + n;
    uint64_t h;
    if (n >= 32) {
        uint64_t v1 = seed + P1 + P2, v2 = seed + P2, v3 = seed, v4 = seed - P1;
        const uint8_t *limit = end - 32;
        do {
            v1 = round_(v1, rd64(p));
            v2 = round_(v2, rd64(p + 8));
            v3 = round_(v3, rd64(p + 16));
            v4 = round_(v4, rd64(p + 24));
            p += 32;
        } while (p <= limit);
        h = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
        h = merge_(h, v1);
        h = merge_(h, v2);
        h = merge_(h, v3);
        h = merge_(h, v4);
    } else {
        h = seed + P5;
    }
    h += (uint64_t)n;
    while (p + 8 <= end) {
        h ^= round_(0, rd64(p));
        h = rotl(h, 27) * P1 + P4;
        p += 8;
    }
    if (p + 4 <= end) {
        h ^= (uint64_t)rd32(p) * P1;
        h = rotl(h, 23) * P2 + P3;
        p += 4;
    }
    while (p < end) {
        h ^= (uint64_t)(*p) * P5;
        h = rotl(h, 11) * P1;
        ++p;
    }
    h ^= h >> 33;
    h *= P2;
    h ^= h >> 29;
    h *= P3;
    h ^= h >> 32;
    return h;
}

// The chained hash of one block's tokens after the prefix hash `prev`.
uint64_t block_hash(const int64_t *tokens, int32_t n, bool has_prev, uint64_t prev) {
    std::vector<uint8_t> bytes((has_prev ? 8 : 0) + 8 * (size_t)n);
    size_t o = 0;
    if (has_prev)
        for (int i = 0; i < 8; ++i) bytes[o++] = (uint8_t)(prev >> (8 * i));
    for (int32_t t = 0; t < n; ++t) {
        const uint64_t v = (uint64_t)tokens[t];
        for (int i = 0; i < 8; ++i) bytes[o++] = (uint8_t)(v >> (8 * i));
    }
    return xxh64(bytes.data(), bytes.size(), 0);
}

// ---------------------------------------------------------------- state
struct Block {
    int32_t ref_count = 0;
    bool has_hash = false;
    uint64_t hash = 0;
    std::vector<int64_t> token_ids;
};

struct Seq {
    bool live = false;
    std::vector<int64_t> tokens;
    std::vector<int32_t> block_table;
    int32_t num_cached_tokens = 0;
    int32_t num_blocks(int32_t B) const { return (int32_t)((tokens.size() + B - 1) / B); }
    // Tokens of logical block i (the last one may be partial).
    const int64_t *block(int32_t i, int32_t B, int32_t *n) const {
        const size_t s = (size_t)i * B;
        *n = (int32_t)std::min<size_t>((size_t)B, tokens.size() - s);
        return tokens.data() + s;
    }
};

}  // namespace

struct pa_block_manager {
    int32_t B = 0;
    std::vector<Block> blocks;
    std::deque<int32_t> free_ids;
    std::unordered_set<int32_t> used_ids;
    std::unordered_map<uint64_t, int32_t> hash_to_block;
    std::vector<Seq> seqs;

    int32_t allocate_block() {
        const int32_t id = free_ids.front();
        free_ids.pop_front();
        Block &b = blocks[id];
        if (b.has_hash) {
            auto it = hash_to_block.find(b.hash);
            if (it != hash_to_block.end() && it->second == id) hash_to_block.erase(it);  // content about to change
        }
        b.ref_count = 1;
        b.has_hash = false;
        b.hash = 0;
        b.token_ids.clear();
        used_ids.insert(id);
        return id;
    }
    void deallocate_block(int32_t id) {  // keeps hash and tokens for a later prefix hit
        used_ids.erase(id);
        free_ids.push_back(id);
    }
    // Cached blocks of s, and how many of them are in use (need no free block).
    int32_t cached_prefix(const Seq &s, int32_t *in_use) const {
        bool has = false;
        uint64_t h = 0;
        int32_t cached = 0, used = 0;
        const int32_t nb = s.num_blocks(B);
        for (int32_t i = 0; i + 1 < nb; ++i) {  // never the last block (it may be partial)
            int32_t n;
            const int64_t *t = s.block(i, B, &n);
            h = block_hash(t, n, has, h);
            has = true;
            auto it = hash_to_block.find(h);
            if (it == hash_to_block.end()) break;
            const Block &b = blocks[it->second];
            if (b.token_ids.size() != (size_t)n || std::memcmp(b.token_ids.data(), t, sizeof(int64_t) * n) != 0)
                break;  // a hash collision: the content differs
            ++cached;
            if (used_ids.count(it->second)) ++used;
        }
        *in_use = used;
        return cached;
    }
};

namespace {

pa_status check_seq(const pa_block_manager *bm, int32_t seq) {
    if (!bm) return pa::fail(PA_ERR_INVALID_ARG, "null block manager");
    if (seq < 0 || seq >= (int32_t)bm->seqs.size() || !bm->seqs[seq].live)
        return pa::fail(PA_ERR_INVALID_ARG, "no sequence %d", seq);
    return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_bm_create(int32_t num_blocks, int32_t block_size, pa_block_manager **out) {
    if (!out) return pa::fail(PA_ERR_INVALID_ARG, "null out");
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0) return pa::fail(PA_ERR_INVALID_ARG, "num_blocks and block_size must be positive");
    pa_block_manager *bm = new (std::nothrow) pa_block_manager;
    if (!bm) return pa::fail(PA_ERR_INVALID_ARG, "out of host memory");
    bm->B = block_size;
    bm->blocks.resize(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) bm->free_ids.push_back(i);
    *out = bm;
    return PA_OK;
}

void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

pa_status pa_bm_seq_add(pa_block_manager *bm, const int64_t *token_ids, int32_t num_tokens, int32_t *seq_id) {
    if (!bm || !seq_id || (num_tokens > 0 && !token_ids)) return pa::fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_tokens < 0) return pa::fail(PA_ERR_INVALID_ARG, "num_tokens < 0");
    Seq s;
    s.live = true;
    s.tokens.assign(token_ids, token_ids + num_tokens);
    bm->seqs.push_back(std::move(s));
    *seq_id = (int32_t)bm->seqs.size() - 1;
    return PA_OK;
}

pa_status pa_bm_seq_append_token(pa_block_manager *bm, int32_t seq, int64_t token_id) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    bm->seqs[seq].tokens.push_back(token_id);
    return PA_OK;
}

pa_status pa_bm_seq_set_num_cached_tokens(pa_block_manager *bm, int32_t seq, int32_t num_cached_tokens) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    if (num_cached_tokens < 0 || num_cached_tokens > (int32_t)bm->seqs[seq].tokens.size())
        return pa::fail(PA_ERR_INVALID_ARG, "num_cached_tokens out of range");
    bm->seqs[seq].num_cached_tokens = num_cached_tokens;
    return PA_OK;
}

pa_status pa_bm_seq_info(const pa_block_manager *bm, int32_t seq, int32_t *num_tokens, int32_t *num_cached_tokens,
                         int32_t *num_table_blocks) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    const Seq &s = bm->seqs[seq];
    if (num_tokens) *num_tokens = (int32_t)s.tokens.size();
    if (num_cached_tokens) *num_cached_tokens = s.num_cached_tokens;
    if (num_table_blocks) *num_table_blocks = (int32_t)s.block_table.size();
    return PA_OK;
}

int32_t pa_bm_can_allocate(const pa_block_manager *bm, int32_t seq) {
    if (check_seq(bm, seq) != PA_OK) return -2;
    const Seq &s = bm->seqs[seq];
    int32_t in_use = 0;
    const int32_t cached = bm->cached_prefix(s, &in_use);
    const int32_t need = s.num_blocks(bm->B) - in_use;
    return (int32_t)bm->free_ids.size() < need ? -1 : cached;
}

pa_status pa_bm_allocate(pa_block_manager *bm, int32_t seq, int32_t num_cached_blocks) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    Seq &s = bm->seqs[seq];
    if (!s.block_table.empty()) return pa::fail(PA_ERR_INVALID_ARG, "sequence %d already holds blocks", seq);
    int32_t in_use = 0;
    const int32_t cached = bm->cached_prefix(s, &in_use);
    if (num_cached_blocks < 0 || num_cached_blocks > cached)
        return pa::fail(PA_ERR_INVALID_ARG, "num_cached_blocks %d but %d blocks are cached", num_cached_blocks, cached);
    const int32_t nb = s.num_blocks(bm->B);
    // The reused blocks, in order (cached_prefix confirmed every one).
    std::vector<int32_t> reuse;
    {
        bool has = false;
        uint64_t h = 0;
        for (int32_t i = 0; i < num_cached_blocks; ++i) {
            int32_t n;
            const int64_t *t = s.block(i, bm->B, &n);
            h = block_hash(t, n, has, h);
            has = true;
            auto it = bm->hash_to_block.find(h);
            if (it == bm->hash_to_block.end()) return pa::fail(PA_ERR_INVALID_ARG, "prefix cache changed");
            reuse.push_back(it->second);
        }
    }
    // Free blocks needed: the fresh ones plus reused ones still in the queue.
    int32_t need = nb - num_cached_blocks;
    for (int32_t id : reuse)
        if (!bm->used_ids.count(id)) ++need;
    if ((int32_t)bm->free_ids.size() < need) return pa::fail(PA_ERR_INVALID_ARG, "not enough free blocks");
    for (int32_t id : reuse) {
        Block &b = bm->blocks[id];
        if (bm->used_ids.count(id)) {
            ++b.ref_count;  // shared with another sequence
        } else {
            b.ref_count = 1;  // released earlier, content intact: take it back
            for (auto it = bm->free_ids.begin(); it != bm->free_ids.end(); ++it)
                if (*it == id) {
                    bm->free_ids.erase(it);
                    break;
                }
            bm->used_ids.insert(id);
        }
        s.block_table.push_back(id);
    }
    for (int32_t i = num_cached_blocks; i < nb; ++i) s.block_table.push_back(bm->allocate_block());
    s.num_cached_tokens = num_cached_blocks * bm->B;
    return PA_OK;
}

pa_status pa_bm_deallocate(pa_block_manager *bm, int32_t seq) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    Seq &s = bm->seqs[seq];
    for (auto it = s.block_table.rbegin(); it != s.block_table.rend(); ++it) {
        Block &b = bm->blocks[*it];
        if (--b.ref_count == 0) bm->deallocate_block(*it);
    }
    s.num_cached_tokens = 0;
    s.block_table.clear();
    return PA_OK;
}

int32_t pa_bm_can_append(const pa_block_manager *bm, int32_t seq) {
    if (check_seq(bm, seq) != PA_OK) return -2;
    const size_t len = bm->seqs[seq].tokens.size();
    const size_t need = (len % (size_t)bm->B == 1) ? 1 : 0;
    return bm->free_ids.size() >= need ? 1 : 0;
}

pa_status pa_bm_may_append(pa_block_manager *bm, int32_t seq) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    Seq &s = bm->seqs[seq];
    if (s.tokens.size() % (size_t)bm->B == 1) {
        if (bm->free_ids.empty()) return pa::fail(PA_ERR_INVALID_ARG, "no free block (check can_append first)");
        s.block_table.push_back(bm->allocate_block());
    }
    return PA_OK;
}

pa_status pa_bm_hash_blocks(pa_block_manager *bm, int32_t seq, int32_t num_scheduled_tokens) {
    pa_status st = check_seq(bm, seq);
    if (st != PA_OK) return st;
    Seq &s = bm->seqs[seq];
    if (num_scheduled_tokens < 0 || (size_t)s.num_cached_tokens + num_scheduled_tokens > s.tokens.size())
        return pa::fail(PA_ERR_INVALID_ARG, "num_scheduled_tokens out of range");
    const int32_t start = s.num_cached_tokens / bm->B;
    const int32_t end = (s.num_cached_tokens + num_scheduled_tokens) / bm->B;
    if (start == end) return PA_OK;
    if (end > (int32_t)s.block_table.size()) return pa::fail(PA_ERR_INVALID_ARG, "block table too short");
    bool has = false;
    uint64_t h = 0;
    if (start > 0) {
        const Block &prev = bm->blocks[s.block_table[start - 1]];
        has = prev.has_hash;
        h = prev.hash;
    }
    for (int32_t i = start; i < end; ++i) {
        Block &b = bm->blocks[s.block_table[i]];
        int32_t n;
        const int64_t *t = s.block(i, bm->B, &n);
        h = block_hash(t, n, has, h);
        has = true;
        b.has_hash = true;
        b.hash = h;
        b.token_ids.assign(t, t + n);
        bm->hash_to_block[h] = s.block_table[i];
    }
    return PA_OK;
}

int32_t pa_bm_seq_block_table(const pa_block_manager *bm, int32_t seq, int32_t *out, int32_t capacity) {
    if (check_seq(bm, seq) != PA_OK) return -2;
    const auto &t = bm->seqs[seq].block_table;
    const int32_t n = (int32_t)t.size();
    if (out)
        for (int32_t i = 0; i < n && i < capacity; ++i) out[i] = t[i];
    return n;
}

pa_status pa_bm_block_tables(const pa_block_manager *bm, const int32_t *seq_ids, int32_t num_seqs, int32_t *out,
                             int32_t max_blocks_per_seq) {
    if (!bm || (num_seqs > 0 && (!seq_ids || !out))) return pa::fail(PA_ERR_INVALID_ARG, "null pointer");
    if (num_seqs < 0 || max_blocks_per_seq <= 0) return pa::fail(PA_ERR_INVALID_ARG, "bad sizes");
    for (int32_t r = 0; r < num_seqs; ++r) {
        pa_status st = check_seq(bm, seq_ids[r]);
        if (st != PA_OK) return st;
        const auto &t = bm->seqs[seq_ids[r]].block_table;
        if ((int32_t)t.size() > max_blocks_per_seq)
            return pa::fail(PA_ERR_INVALID_ARG, "sequence %d holds %d blocks > %d", seq_ids[r], (int)t.size(),
                            max_blocks_per_seq);
        for (int32_t i = 0; i < max_blocks_per_seq; ++i)
            out[(int64_t)r * max_blocks_per_seq + i] = i < (int32_t)t.size() ? t[i] : -1;
    }
    return PA_OK;
}

int32_t pa_bm_free_block_ids(const pa_block_manager *bm, int32_t *out, int32_t capacity) {
    if (!bm) return -2;
    int32_t i = 0;
    if (out)
        for (int32_t id : bm->free_ids) {
            if (i >= capacity) break;
            out[i++] = id;
        }
    return (int32_t)bm->free_ids.size();
}

pa_status pa_bm_block_info(const pa_block_manager *bm, int32_t block_id, int32_t *ref_count, int32_t *has_hash,
                           uint64_t *hash, int32_t *num_token_ids) {
    if (!bm) return pa::fail(PA_ERR_INVALID_ARG, "null block manager");
    if (block_id < 0 || block_id >= (int32_t)bm->blocks.size()) return pa::fail(PA_ERR_INVALID_ARG, "no block %d", block_id);
    const Block &b = bm->blocks[block_id];
    if (ref_count) *ref_count = b.ref_count;
    if (has_hash) *has_hash = b.has_hash ? 1 : 0;
    if (hash) *hash = b.hash;
    if (num_token_ids) *num_token_ids = (int32_t)b.token_ids.size();
    return PA_OK;
}

int32_t pa_bm_lookup_hash(const pa_block_manager *bm, uint64_t hash) {
    if (!bm) return -2;
    auto it = bm->hash_to_block.find(hash);
    return it == bm->hash_to_block.end() ? -1 : it->second;
}

int32_t pa_bm_num_hashes(const pa_block_manager *bm) { return bm ? (int32_t)bm->hash_to_block.size() : -2; }

uint64_t pa_bm_block_hash(const int64_t *token_ids, int32_t num_tokens, int32_t has_prefix, uint64_t prefix) {
    return block_hash(token_ids, num_tokens < 0 ? 0 : num_tokens, has_prefix != 0, prefix);
}

uint64_t pa_bm_xxh64(const void *data, size_t len, uint64_t seed) {
    return xxh64(static_cast<const uint8_t *>(data), data ? len : 0, seed);
}

}  // extern "C"
