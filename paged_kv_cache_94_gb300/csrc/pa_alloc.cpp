// Host block manager of the paged KV cache: reference counts, chained-hash
// prefix caching with an LRU evictable pool, fork and copy-on-write.
//
// Behaviour: "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度",
// section "Prefix Caching 与 Copy-on-Write" (H_k = Hash(H_{k-1}, tokens),
// hits bump the reference count, released blocks stay hashed in an LRU
// pool, a shared partly filled tail is copied on write); "KV Cache 显存管理全景",
// 考点 4 (branches share blocks, one reference each). Every operation either
// succeeds or leaves the state as it was: its checks come before any change.
//
// Data structures: per block a reference count, a fill count, a hash and
// the links of an intrusive doubly linked LRU list (head = next to evict);
// token ids of all blocks in one flat array; an open hash map from chained
// hash to block.
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa_alloc.h"

namespace {

// ----------------------------------------------------------------------------
// BLAKE2b (RFC 7693), unkeyed, digest length nn <= 64 bytes.
// ----------------------------------------------------------------------------
constexpr uint64_t kIV[8] = {0x6a09e667f3bcc908ull, 0xbb67ae8584caa73bull, 0x3c6ef372fe94f82bull,
                             0xa54ff53a5f1d36f1ull, 0x510e527fade682d1ull, 0x9b05688c2b3e6c1full,
                             0x1f83d9abfb41bd6bull, 0x5be0cd19137e2179ull};

constexpr uint8_t kSigma[10][16] = {
    {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15},
    {14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3},
    {11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4},
    {7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8},
    {9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13},
    {2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9},
    {12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11},
    {13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10},
    {6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5},
    {10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0},
};

inline uint64_t rotr64(uint64_t x, int n) { return (x >> n) | (x << (64 - n)); }

inline uint64_t load_le64(const uint8_t *p)
{
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i)
        v = (v << 8) | p[i];
    return v;
}

struct Blake2b {
    uint64_t h[8];
    uint8_t buf[128];
    size_t fill = 0;     // bytes in buf
    uint64_t total = 0;  // bytes compressed so far (the counter t; < 2^64 here)
    int nn;

    explicit Blake2b(int out_bytes) : nn(out_bytes)
    {
        for (int i = 0; i < 8; ++i)
            h[i] = kIV[i];
        h[0] ^= 0x01010000ull ^ (uint64_t)nn; // parameter block: depth 1, fanout 1, no key
    }

    static void mix(uint64_t *v, int a, int b, int c, int d, uint64_t x, uint64_t y)
    {
        v[a] = v[a] + v[b] + x;
        v[d] = rotr64(v[d] ^ v[a], 32);
        v[c] = v[c] + v[d];
        v[b] = rotr64(v[b] ^ v[c], 24);
        v[a] = v[a] + v[b] + y;
        v[d] = rotr64(v[d] ^ v[a], 16);
        v[c] = v[c] + v[d];
        v[b] = rotr64(v[b] ^ v[c], 63);
    }

    void compress(bool last)
    {
        uint64_t m[16], v[16];
        for (int i = 0; i < 16; ++i)
            m[i] = load_le64(buf + 8 * i);
        for (int i = 0; i < 8; ++i) {
            v[i] = h[i];
            v[i + 8] = kIV[i];
        }
        v[12] ^= total; // low word of t; the high word stays 0
        if (last)
            v[14] = ~v[14];
        for (int r = 0; r < 12; ++r) {
            const uint8_t *s = kSigma[r % 10];
            mix(v, 0, 4, 8, 12, m[s[0]], m[s[1]]);
            mix(v, 1, 5, 9, 13, m[s[2]], m[s[3]]);
            mix(v, 2, 6, 10, 14, m[s[4]], m[s[5]]);
            mix(v, 3, 7, 11, 15, m[s[6]], m[s[7]]);
            mix(v, 0, 5, 10, 15, m[s[8]], m[s[9]]);
            mix(v, 1, 6, 11, 12, m[s[10]], m[s[11]]);
            mix(v, 2, 7, 8, 13, m[s[12]], m[s[13]]);
            mix(v, 3, 4, 9, 14, m[s[14]], m[s[15]]);
        }
        for (int i = 0; i < 8; ++i)
            h[i] ^= v[i] ^ v[i + 8];
    }

    void update(const uint8_t *p, size_t n)
    {
        while (n > 0) {
            if (fill == 128) { // a full block is compressed only once more input follows
                total += 128;
                compress(false);
                fill = 0;
            }
            const size_t take = n < 128 - fill ? n : 128 - fill;
            std::memcpy(buf + fill, p, take);
            fill += take;
            p += take;
            n -= take;
        }
    }

    uint64_t final_le64()
    {
        total += fill;
        std::memset(buf + fill, 0, 128 - fill);
        compress(true);
        uint8_t out[8];
        for (int i = 0; i < 8; ++i)
            out[i] = (uint8_t)(h[0] >> (8 * i));
        uint64_t r = 0;
        for (int i = nn < 8 ? nn - 1 : 7; i >= 0; --i)
            r = (r << 8) | out[i];
        return r;
    }
};

uint64_t chain_hash(uint64_t parent, const int32_t *tok, int32_t n)
{
    Blake2b b(8);
    uint8_t w[8];
    for (int i = 0; i < 8; ++i)
        w[i] = (uint8_t)(parent >> (8 * i));
    b.update(w, 8);
    for (int32_t j = 0; j < n; ++j) {
        const uint32_t t = (uint32_t)tok[j];
        for (int i = 0; i < 4; ++i)
            w[i] = (uint8_t)(t >> (8 * i));
        b.update(w, 4);
    }
    return b.final_le64();
}

} // namespace

// ----------------------------------------------------------------------------
struct pa_allocator {
    struct Block {
        int32_t ref = 0;
        int32_t ntok = 0;
        uint64_t hash = 0;
        bool has_hash = false;
        bool in_pool = false;
        int32_t prev = -1, next = -1; // LRU links while in the pool
    };

    int32_t bs;
    std::vector<Block> blk;
    std::vector<int32_t> tokens; // [num_blocks][bs]
    std::unordered_map<uint64_t, int32_t> by_hash;
    int32_t head = -1, tail = -1; // head: least recently released
    int64_t pool_size = 0;

    pa_allocator(int64_t nb, int32_t block_size) : bs(block_size), blk((size_t)nb),
        tokens((size_t)nb * (size_t)block_size)
    {
        for (int32_t i = 0; i < (int32_t)nb; ++i)
            push_tail(i);
    }

    void push_tail(int32_t b)
    {
        Block &x = blk[b];
        x.prev = tail;
        x.next = -1;
        x.in_pool = true;
        if (tail >= 0)
            blk[tail].next = b;
        else
            head = b;
        tail = b;
        ++pool_size;
    }

    void unlink(int32_t b)
    {
        Block &x = blk[b];
        if (x.prev >= 0)
            blk[x.prev].next = x.next;
        else
            head = x.next;
        if (x.next >= 0)
            blk[x.next].prev = x.prev;
        else
            tail = x.prev;
        x.prev = x.next = -1;
        x.in_pool = false;
        --pool_size;
    }

    // Head of the LRU pool, wiped for new data, reference count 1.
    int32_t take()
    {
        const int32_t b = head;
        unlink(b);
        Block &x = blk[b];
        if (x.has_hash) {
            by_hash.erase(x.hash);
            x.has_hash = false;
        }
        x.ntok = 0;
        x.ref = 1;
        return b;
    }

    int32_t find(uint64_t h) const
    {
        auto it = by_hash.find(h);
        return it == by_hash.end() ? -1 : it->second;
    }

    bool held(int32_t b) const { return b >= 0 && (size_t)b < blk.size() && blk[b].ref > 0; }
};

namespace {

bool tokens_ok(const int32_t *t, int32_t n)
{
    for (int32_t i = 0; i < n; ++i)
        if (t[i] < 0)
            return false;
    return true;
}

} // namespace

extern "C" {

uint64_t pa_block_hash(uint64_t parent, const int32_t *token_ids, int32_t n)
{
    return chain_hash(parent, token_ids, n > 0 && token_ids ? n : 0);
}

pa_status pa_allocator_create(int64_t num_blocks, int32_t block_size, pa_allocator **out)
{
    if (!out)
        return PA_ERR_NULL;
    *out = nullptr;
    if (num_blocks < 1 || num_blocks > INT32_MAX || block_size < 1 ||
        num_blocks * (int64_t)block_size > ((int64_t)1 << 40))
        return PA_ERR_SHAPE;
    try {
        *out = new pa_allocator(num_blocks, block_size);
    } catch (const std::bad_alloc &) {
        return PA_ERR_SHAPE;
    }
    return PA_OK;
}

void pa_allocator_destroy(pa_allocator *a) { delete a; }

pa_status pa_allocator_allocate_prompt(pa_allocator *a, const int32_t *token_ids,
                                       int32_t n_tokens, int32_t *block_table, int32_t capacity,
                                       int32_t *n_blocks, int32_t *cached_tokens)
{
    if (!a || !n_blocks || !cached_tokens || (n_tokens > 0 && (!token_ids || !block_table)))
        return PA_ERR_NULL;
    if (n_tokens < 0 || capacity < 0 || !tokens_ok(token_ids, n_tokens))
        return PA_ERR_SHAPE;
    const int32_t bs = a->bs;
    const int32_t nchunk = (int32_t)(((int64_t)n_tokens + bs - 1) / bs);
    if (nchunk > capacity)
        return PA_ERR_SHAPE;

    // Dry run: hits and the hit blocks sitting in the pool (nothing changes).
    const int32_t nfull = n_tokens / bs;
    int32_t n_hit = 0;
    int64_t hits_in_pool = 0;
    uint64_t parent = 0;
    for (; n_hit < nfull; ++n_hit) {
        const uint64_t h = chain_hash(parent, token_ids + (size_t)n_hit * bs, bs);
        const int32_t b = a->find(h);
        if (b < 0)
            break;
        hits_in_pool += a->blk[b].ref == 0;
        parent = h;
    }
    if ((int64_t)(nchunk - n_hit) > a->pool_size - hits_in_pool)
        return PA_ERR_OUT_OF_BLOCKS;

    parent = 0;
    for (int32_t k = 0; k < nchunk; ++k) {
        const int32_t *chunk = token_ids + (size_t)k * bs;
        const int32_t len = k < nfull ? bs : n_tokens - k * bs;
        if (k < n_hit) { // the dry run found it: share it
            parent = chain_hash(parent, chunk, bs);
            const int32_t b = a->find(parent);
            if (a->blk[b].ref == 0)
                a->unlink(b);
            ++a->blk[b].ref;
            block_table[k] = b;
            continue;
        }
        const int32_t b = a->take();
        pa_allocator::Block &x = a->blk[b];
        std::memcpy(a->tokens.data() + (size_t)b * bs, chunk, sizeof(int32_t) * (size_t)len);
        x.ntok = len;
        if (len == bs) {
            parent = chain_hash(parent, chunk, bs);
            // One block per hash: an older holder of this hash gives it up
            // (blocks leave the pool oldest first, so the older copies of a
            // prefix are recycled before this point; the check keeps the map
            // exact regardless).
            const int32_t old = a->find(parent);
            if (old >= 0)
                a->blk[old].has_hash = false;
            x.hash = parent;
            x.has_hash = true;
            a->by_hash[parent] = b;
        }
        block_table[k] = b;
    }
    *n_blocks = nchunk;
    *cached_tokens = n_hit * bs;
    return PA_OK;
}

pa_status pa_allocator_append_slots(pa_allocator *a, int32_t *block_tables, int32_t capacity,
                                    int32_t *n_blocks, const int32_t *token_ids,
                                    int32_t num_seqs, int64_t *slots, int32_t *cow_pairs,
                                    int32_t *num_cow, int32_t *num_done)
{
    if (!a || !num_cow || !num_done)
        return PA_ERR_NULL;
    *num_cow = 0;
    *num_done = 0;
    if (num_seqs < 0 || capacity < 0)
        return PA_ERR_SHAPE;
    if (num_seqs > 0 && (!block_tables || !n_blocks || !token_ids || !slots || !cow_pairs))
        return PA_ERR_NULL;
    const int32_t bs = a->bs;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int32_t *table = block_tables + (size_t)i * capacity;
        const int32_t n = n_blocks[i];
        if (n < 0 || n > capacity || token_ids[i] < 0)
            return PA_ERR_SHAPE;
        const int32_t last = n > 0 ? table[n - 1] : -1;
        if (n > 0 && !a->held(last))
            return PA_ERR_STATE;
        const bool fresh = n == 0 || a->blk[last].ntok == bs;
        if (fresh && n == capacity)
            return PA_ERR_SHAPE;
        if ((fresh || a->blk[last].ref > 1) && a->pool_size == 0)
            return PA_ERR_OUT_OF_BLOCKS;

        if (fresh) {
            const int32_t b = a->take();
            a->tokens[(size_t)b * bs] = token_ids[i];
            a->blk[b].ntok = 1;
            table[n] = b;
            n_blocks[i] = n + 1;
            slots[i] = (int64_t)b * bs;
        } else if (a->blk[last].ref > 1) { // copy-on-write of the shared tail
            const int32_t b = a->take();
            --a->blk[last].ref;
            const int32_t nt = a->blk[last].ntok;
            std::memcpy(a->tokens.data() + (size_t)b * bs, a->tokens.data() + (size_t)last * bs,
                        sizeof(int32_t) * (size_t)nt);
            a->tokens[(size_t)b * bs + nt] = token_ids[i];
            a->blk[b].ntok = nt + 1;
            table[n - 1] = b;
            slots[i] = (int64_t)b * bs + nt;
            cow_pairs[2 * *num_cow] = last;
            cow_pairs[2 * *num_cow + 1] = b;
            ++*num_cow;
        } else {
            const int32_t nt = a->blk[last].ntok;
            a->tokens[(size_t)last * bs + nt] = token_ids[i];
            a->blk[last].ntok = nt + 1;
            slots[i] = (int64_t)last * bs + nt;
        }
        *num_done = i + 1;
    }
    return PA_OK;
}

pa_status pa_allocator_fork(pa_allocator *a, const int32_t *block_table, int32_t n_blocks)
{
    if (!a || (n_blocks > 0 && !block_table))
        return PA_ERR_NULL;
    if (n_blocks < 0)
        return PA_ERR_SHAPE;
    for (int32_t k = 0; k < n_blocks; ++k)
        if (!a->held(block_table[k]))
            return PA_ERR_STATE;
    for (int32_t k = 0; k < n_blocks; ++k)
        ++a->blk[block_table[k]].ref;
    return PA_OK;
}

pa_status pa_allocator_free(pa_allocator *a, const int32_t *block_table, int32_t n_blocks)
{
    if (!a || (n_blocks > 0 && !block_table))
        return PA_ERR_NULL;
    if (n_blocks < 0)
        return PA_ERR_SHAPE;
    // A block named m times must hold at least m references.
    std::unordered_map<int32_t, int32_t> uses;
    for (int32_t k = 0; k < n_blocks; ++k) {
        const int32_t b = block_table[k];
        if (!a->held(b) || ++uses[b] > a->blk[b].ref)
            return PA_ERR_STATE;
    }
    for (int32_t k = 0; k < n_blocks; ++k) {
        const int32_t b = block_table[k];
        if (--a->blk[b].ref == 0)
            a->push_tail(b);
    }
    return PA_OK;
}

int64_t pa_allocator_num_free(const pa_allocator *a) { return a ? a->pool_size : 0; }

pa_status pa_allocator_block_info(const pa_allocator *a, int64_t block, int32_t *ref_count,
                                  int32_t *num_tokens, uint64_t *hash, int32_t *has_hash)
{
    if (!a)
        return PA_ERR_NULL;
    if (block < 0 || (size_t)block >= a->blk.size())
        return PA_ERR_SHAPE;
    const pa_allocator::Block &x = a->blk[(size_t)block];
    if (ref_count)
        *ref_count = x.ref;
    if (num_tokens)
        *num_tokens = x.ntok;
    if (hash)
        *hash = x.has_hash ? x.hash : 0;
    if (has_hash)
        *has_hash = x.has_hash ? 1 : 0;
    return PA_OK;
}

pa_status pa_allocator_free_order(const pa_allocator *a, int32_t *out, int64_t capacity,
                                  int64_t *n)
{
    if (!a || !n || (capacity > 0 && !out))
        return PA_ERR_NULL;
    int64_t i = 0;
    for (int32_t b = a->head; b >= 0; b = a->blk[b].next, ++i)
        if (i < capacity)
            out[i] = b;
    *n = a->pool_size;
    return PA_OK;
}

} // extern "C"
