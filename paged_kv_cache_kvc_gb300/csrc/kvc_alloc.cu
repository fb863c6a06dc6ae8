// Host block allocator (free queue, reference counts, copy-on-write, retention
// of evictable prefix blocks, block-hash prefix lookup) and the device block copy.
//
// "KV cache: Generation state, latency, and allocation" 21.5 and Table 21.1:
// blocks are allocated as a sequence grows; a block shared by several
// requests carries a reference count; full shared blocks stay immutable and
// a shared, partly filled block is copied before a write (copy-on-write);
// releasing a request drops its references, and a block whose count reaches
// zero returns to the free pool or, under a retention policy, stays as an
// evictable cached entry.  21.4: a block's identity chains the previous
// block's identity, its exact token ids and configuration identity (salt).
// "KV Cache Explained", "Follow the 32 GiB pool ...": the allocator takes free
// blocks first, then reclaims unreferenced cached blocks, and reports the
// moment it cannot provide one more block.
#include <algorithm>
#include <cstring>
#include <deque>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "kvc_internal.h"

namespace {

constexpr int32_t kFree = 0, kUsed = 1, kCached = 2;

struct Seq {
    bool live = false;
    uint32_t version = 0;            // table entries replaced by copy-on-write since the sequence began
    int64_t len = 0;                 // tokens written (committed); capacity is blocks.size() * bs
    std::vector<int32_t> blocks;
    std::vector<uint64_t> hashes;    // identity of each published full block
};

struct CachedKey {
    std::vector<int32_t> tokens;     // exact token ids of the block (collision check)
    uint64_t parent;                 // identity of the previous block (or the salt seed)
};

inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// h_i = hash(h_{i-1}, tokens_i); h_0 = hash(salt)
uint64_t chain_hash(uint64_t parent, const int32_t *tok, int32_t n)
{
    uint64_t h = mix64(parent ^ 0x9E3779B97F4A7C15ULL);
    for (int32_t i = 0; i < n; ++i) h = mix64(h + static_cast<uint32_t>(tok[i]) + 0x632BE59BD9B4E019ULL * (i + 1));
    return h;
}

uint64_t salt_seed(uint64_t salt) { return mix64(salt + 0xD1B54A32D192ED03ULL); }

}  // namespace

struct kvc_alloc {
    int64_t N = 0;
    int32_t bs = 0;
    bool retain = false;
    std::vector<int32_t> ref;
    std::vector<int32_t> state;
    std::deque<int32_t> free_q;                         // FIFO
    std::list<int32_t> lru;                             // evictable cached blocks, least recent first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<uint64_t> block_hash;                   // published identity of a block (0 = none)
    std::vector<CachedKey> block_key;
    std::unordered_multimap<uint64_t, int32_t> by_hash; // identity -> block
    std::vector<Seq> seqs;
    std::vector<uint32_t> incarnation;                  // per sequence id: times it was handed out
};

namespace {

kvc_status take_block(kvc_alloc *a, int32_t *out)
{
    if (!a->free_q.empty()) {
        *out = a->free_q.front();
        a->free_q.pop_front();
    } else if (!a->lru.empty()) {                       // reclaim the least recently used cached block
        const int32_t b = a->lru.front();
        a->lru.pop_front();
        auto range = a->by_hash.equal_range(a->block_hash[b]);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second == b) {
                a->by_hash.erase(it);
                break;
            }
        a->block_hash[b] = 0;
        a->block_key[b] = CachedKey{};
        *out = b;
    } else {
        return KVC_ERR_OOM;
    }
    a->state[*out] = kUsed;
    a->ref[*out] = 1;
    return KVC_OK;
}

void drop_ref(kvc_alloc *a, int32_t b)
{
    if (--a->ref[b] > 0) return;
    if (a->retain && a->block_hash[b] != 0) {           // a full, published block stays as an evictable entry
        a->state[b] = kCached;
        a->lru_pos[b] = a->lru.insert(a->lru.end(), b);
    } else {
        a->state[b] = kFree;
        if (a->block_hash[b] != 0) {
            auto range = a->by_hash.equal_range(a->block_hash[b]);
            for (auto it = range.first; it != range.second; ++it)
                if (it->second == b) {
                    a->by_hash.erase(it);
                    break;
                }
            a->block_hash[b] = 0;
            a->block_key[b] = CachedKey{};
        }
        a->free_q.push_back(b);
    }
}

void add_ref(kvc_alloc *a, int32_t b)
{
    if (a->state[b] == kCached) {                       // a hit revives an evictable entry
        a->lru.erase(a->lru_pos[b]);
        a->state[b] = kUsed;
        a->ref[b] = 0;
    }
    ++a->ref[b];
}

Seq *get_seq(kvc_alloc *a, int32_t s)
{
    if (!a || s < 0 || s >= static_cast<int32_t>(a->seqs.size()) || !a->seqs[s].live) return nullptr;
    return &a->seqs[s];
}

int32_t new_seq_slot(kvc_alloc *a)
{
    for (size_t i = 0; i < a->seqs.size(); ++i)
        if (!a->seqs[i].live) {
            a->seqs[i] = Seq{};
            a->seqs[i].live = true;
            ++a->incarnation[i];
            return static_cast<int32_t>(i);
        }
    a->seqs.push_back(Seq{});
    a->seqs.back().live = true;
    a->incarnation.push_back(1);
    return static_cast<int32_t>(a->seqs.size() - 1);
}

// (times the id was handed out, copy-on-write replacements of its table entries)
uint64_t lease_stamp(const kvc_alloc *a, int32_t s)
{
    return (static_cast<uint64_t>(a->incarnation[s]) << 32) | a->seqs[s].version;
}

}  // namespace

using namespace kvc;

extern "C" kvc_status kvc_alloc_create(int64_t num_blocks, int32_t block_size, const int32_t *free_order,
                                       int32_t retain_cached, kvc_alloc **out)
{
    if (!out) return KVC_ERR_ARG;
    *out = nullptr;
    if (num_blocks < 1 || num_blocks > (int64_t(1) << 31) - 1 || block_size < 1) return KVC_ERR_ARG;
    kvc_alloc *a = new (std::nothrow) kvc_alloc();
    if (!a) return KVC_ERR_OOM;
    a->N = num_blocks;
    a->bs = block_size;
    a->retain = retain_cached != 0;
    a->ref.assign(num_blocks, 0);
    a->state.assign(num_blocks, kFree);
    a->lru_pos.resize(num_blocks);
    a->block_hash.assign(num_blocks, 0);
    a->block_key.resize(num_blocks);
    if (free_order) {                                   // a permutation of [0, N): the initial queue order
        std::vector<char> seen(num_blocks, 0);
        for (int64_t i = 0; i < num_blocks; ++i) {
            const int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete a;
                return KVC_ERR_ARG;
            }
            seen[b] = 1;
            a->free_q.push_back(b);
        }
    } else {
        for (int64_t i = 0; i < num_blocks; ++i) a->free_q.push_back(static_cast<int32_t>(i));
    }
    *out = a;
    return KVC_OK;
}

extern "C" void kvc_alloc_destroy(kvc_alloc *a) { delete a; }

extern "C" kvc_status kvc_alloc_new_seq(kvc_alloc *a, int32_t *seq)
{
    if (!a || !seq) return KVC_ERR_ARG;
    *seq = new_seq_slot(a);
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_fork(kvc_alloc *a, int32_t src, int32_t n_tokens, int32_t *seq)
{
    Seq *s = get_seq(a, src);
    if (!s || !seq || n_tokens < 0 || n_tokens > s->len) return KVC_ERR_ARG;
    const int32_t nb = static_cast<int32_t>((static_cast<int64_t>(n_tokens) + a->bs - 1) / a->bs);
    const int32_t id = new_seq_slot(a);
    Seq &d = a->seqs[id];
    s = &a->seqs[src];                                  // (the vector may have grown)
    d.blocks.assign(s->blocks.begin(), s->blocks.begin() + nb);
    d.hashes.assign(s->hashes.begin(), s->hashes.begin() + std::min<size_t>(s->hashes.size(), n_tokens / a->bs));
    d.len = n_tokens;
    for (int32_t b : d.blocks) add_ref(a, b);
    *seq = id;
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_reserve(kvc_alloc *a, int32_t seq, int32_t n_tokens, int32_t *cow_pairs,
                                        int32_t max_cow, int32_t *n_cow)
{
    Seq *s = get_seq(a, seq);
    if (!s || n_tokens < 0) return KVC_ERR_ARG;
    if (n_cow) *n_cow = 0;
    const int64_t target = s->len + n_tokens;
    const int64_t have = static_cast<int64_t>(s->blocks.size());
    const int64_t need_blocks = std::max<int64_t>(0, (target + a->bs - 1) / a->bs - have);
    // copy-on-write: the next write lands in a shared, partly filled block (the one holding position len)
    const int64_t w = s->len / a->bs;
    const bool cow = n_tokens > 0 && s->len % a->bs != 0 && w < have && a->ref[s->blocks[w]] > 1;
    if (!cow && need_blocks == 0) return KVC_OK;
    if (static_cast<int64_t>(a->free_q.size() + a->lru.size()) < need_blocks + (cow ? 1 : 0))
        return KVC_ERR_OOM;                              // nothing changed
    if (cow) {
        if (!cow_pairs || max_cow < 1) return KVC_ERR_ARG;
        int32_t fresh;
        (void)take_block(a, &fresh);
        const int32_t old = s->blocks[w];
        cow_pairs[0] = old;
        cow_pairs[1] = fresh;
        if (n_cow) *n_cow = 1;
        s->blocks[w] = fresh;
        ++s->version;                                   // tables handed out before now map the old block
        drop_ref(a, old);
    }
    for (int64_t i = 0; i < need_blocks; ++i) {
        int32_t b;
        (void)take_block(a, &b);
        s->blocks.push_back(b);
    }
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_commit(kvc_alloc *a, int32_t seq, int32_t n_tokens)
{
    Seq *s = get_seq(a, seq);
    if (!s || n_tokens < 0 || s->len + n_tokens > static_cast<int64_t>(s->blocks.size()) * a->bs) return KVC_ERR_ARG;
    // every written position must sit in a private block: reserve copies shared ones first
    for (int64_t t = s->len; t < s->len + n_tokens; t += a->bs - (t % a->bs))
        if (a->ref[s->blocks[t / a->bs]] > 1) return KVC_ERR_ALIAS;
    s->len += n_tokens;
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_release(kvc_alloc *a, int32_t seq)
{
    Seq *s = get_seq(a, seq);
    if (!s) return KVC_ERR_ARG;
    for (int32_t b : s->blocks) drop_ref(a, b);
    *s = Seq{};
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_publish(kvc_alloc *a, int32_t seq, const int32_t *tokens, int32_t n_tokens,
                                        uint64_t salt)
{
    Seq *s = get_seq(a, seq);
    if (!s || (n_tokens > 0 && !tokens) || n_tokens < 0 || n_tokens > s->len) return KVC_ERR_ARG;
    const int32_t full = n_tokens / a->bs;
    uint64_t parent = salt_seed(salt);
    for (int32_t i = 0; i < full; ++i) {
        const int32_t *t = tokens + static_cast<int64_t>(i) * a->bs;
        const uint64_t h = chain_hash(parent, t, a->bs);
        if (static_cast<int32_t>(s->hashes.size()) <= i) s->hashes.push_back(h);
        const int32_t b = s->blocks[i];
        // one block per exact identity: a second block with the same prefix stays unpublished
        bool known = false;
        auto range = a->by_hash.equal_range(h);
        for (auto it = range.first; it != range.second && !known; ++it) {
            const CachedKey &k = a->block_key[it->second];
            known = k.parent == parent && std::memcmp(k.tokens.data(), t, sizeof(int32_t) * a->bs) == 0;
        }
        if (a->block_hash[b] == 0 && !known) {
            a->block_hash[b] = h;
            a->block_key[b] = CachedKey{std::vector<int32_t>(tokens + static_cast<int64_t>(i) * a->bs,
                                                             tokens + static_cast<int64_t>(i + 1) * a->bs),
                                        parent};
            a->by_hash.emplace(h, b);
        }
        parent = h;
    }
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_match(kvc_alloc *a, const int32_t *tokens, int32_t n_tokens, uint64_t salt,
                                      int32_t *seq_out, int32_t *hit_tokens)
{
    if (!a || !seq_out || !hit_tokens || n_tokens < 0 || (n_tokens > 0 && !tokens)) return KVC_ERR_ARG;
    std::vector<int32_t> hit;
    uint64_t parent = salt_seed(salt);
    const int32_t full = n_tokens / a->bs;
    for (int32_t i = 0; i < full; ++i) {
        const int32_t *t = tokens + static_cast<int64_t>(i) * a->bs;
        const uint64_t h = chain_hash(parent, t, a->bs);
        int32_t found = -1;
        auto range = a->by_hash.equal_range(h);
        for (auto it = range.first; it != range.second && found < 0; ++it) {
            const CachedKey &k = a->block_key[it->second];
            if (k.parent == parent && static_cast<int32_t>(k.tokens.size()) == a->bs &&
                std::memcmp(k.tokens.data(), t, sizeof(int32_t) * a->bs) == 0)
                found = it->second;                     // exact ids and parent: not a collision
        }
        if (found < 0) break;
        hit.push_back(found);
        parent = h;
    }
    const int32_t id = new_seq_slot(a);
    Seq &d = a->seqs[id];
    d.blocks = hit;
    for (int32_t b : hit) {
        add_ref(a, b);
        d.hashes.push_back(a->block_hash[b]);
    }
    d.len = static_cast<int64_t>(hit.size()) * a->bs;
    *seq_out = id;
    *hit_tokens = static_cast<int32_t>(d.len);
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_seq_info(const kvc_alloc *a, int32_t seq, int64_t *len, int32_t *n_blocks)
{
    Seq *s = get_seq(const_cast<kvc_alloc *>(a), seq);
    if (!s) return KVC_ERR_ARG;
    if (len) *len = s->len;
    if (n_blocks) *n_blocks = static_cast<int32_t>(s->blocks.size());
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_block_tables(const kvc_alloc *a, const int32_t *seqs, int32_t n, int32_t max_blocks,
                                             int32_t *table, int32_t *lens)
{
    if (!a || (n > 0 && (!seqs || !table)) || n < 0 || max_blocks < 1) return KVC_ERR_ARG;
    for (int32_t i = 0; i < n; ++i) {
        Seq *s = get_seq(const_cast<kvc_alloc *>(a), seqs[i]);
        if (!s || static_cast<int32_t>(s->blocks.size()) > max_blocks) return KVC_ERR_ARG;
        for (int32_t j = 0; j < max_blocks; ++j)
            table[static_cast<int64_t>(i) * max_blocks + j] = j < static_cast<int32_t>(s->blocks.size()) ? s->blocks[j] : -1;
        if (lens) lens[i] = static_cast<int32_t>(s->len);
    }
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_lease(const kvc_alloc *a, int32_t seq, uint64_t *stamp)
{
    Seq *s = get_seq(const_cast<kvc_alloc *>(a), seq);
    if (!s || !stamp) return KVC_ERR_ARG;
    *stamp = lease_stamp(a, seq);
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_check(const kvc_alloc *a, int32_t seq, uint64_t stamp)
{
    if (!a || seq < 0 || seq >= static_cast<int32_t>(a->seqs.size())) return KVC_ERR_ARG;
    if (!a->seqs[seq].live || lease_stamp(a, seq) != stamp) return KVC_ERR_STALE;
    return KVC_OK;
}

extern "C" kvc_status kvc_alloc_counts(const kvc_alloc *a, int64_t *n_free, int64_t *n_used, int64_t *n_cached)
{
    if (!a) return KVC_ERR_ARG;
    if (n_free) *n_free = static_cast<int64_t>(a->free_q.size());
    if (n_cached) *n_cached = static_cast<int64_t>(a->lru.size());
    if (n_used) *n_used = a->N - static_cast<int64_t>(a->free_q.size() + a->lru.size());
    return KVC_OK;
}

extern "C" int32_t kvc_alloc_refcount(const kvc_alloc *a, int32_t block)
{
    if (!a || block < 0 || block >= a->N) return -1;
    return a->ref[block];
}

// ------------------------------------------------------------------ device block copy (copy-on-write)
namespace kvc {

// Copy every layer's keys and values of block src to block dst: per layer the
// block is one contiguous run of block_bytes (layout [l][p][h][kv][slot][c]).
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t *base, const int32_t *pairs, int64_t N,
                                                          int64_t layer_bytes, int64_t block_bytes, uint32_t *err)
{
    const int i = blockIdx.x, layer = blockIdx.y;
    const int32_t src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || dst < 0 || src >= N || dst >= N) {
        if (threadIdx.x == 0 && layer == 0) atomicOr(err, KVC_EBIT_BAD_BLOCK);
        return;
    }
    const uint4 *s = reinterpret_cast<const uint4 *>(base + layer * layer_bytes + src * block_bytes);
    uint4 *d = reinterpret_cast<uint4 *>(base + layer * layer_bytes + dst * block_bytes);
    for (int64_t k = threadIdx.x; k < block_bytes / 16; k += blockDim.x) d[k] = s[k];
}

}  // namespace kvc

extern "C" kvc_status kvc_copy_blocks(kvc_pool *pool, const int32_t *pairs, int32_t n, kvc_stream_t stream)
{
    if (!pool || n < 0 || n > 65535 || (n > 0 && !pairs)) return KVC_ERR_ARG;
    if (n == 0) return KVC_OK;
    if ((reinterpret_cast<uintptr_t>(pairs) & 3) != 0) return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    const int64_t block_bytes = 2ll * pool->H_KV * pool->bs * pool->D * pool->bits / 8;
    copy_blocks_kernel<<<dim3(n, pool->L), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        pool->base, pairs, pool->N, static_cast<int64_t>(pool->layer_bytes), block_bytes, pool->err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return KVC_OK;
}
