// pa_prefix.cpp -- radix-tree prefix cache over the block pool.
//
// "KV Cache Optimization and Management", section "RadixAttention: caching,
// not just packing, the prefix": cached token sequences are kept in a radix
// tree whose edges are labelled with runs of tokens; a new request walks the
// tree and reuses the K/V blocks of every matched token; when memory runs low,
// least-recently-used leaves are evicted, and reference counting protects
// branches a running request still uses.  Only whole blocks are cached and
// reused ("PagedAttention: Virtual Memory for the KV Cache", "Sharing a prefix
// and copying a partial block": implementations may restrict reuse to complete
// blocks; answer A3 of the same chapter counts shareable full blocks).
//
// Semantics (mirrored by the oracle model used in the tests):
//  - the cache holds a prefix-closed set of block-aligned token prefixes, each
//    mapped to one physical block on which it holds one pool reference;
//  - match(tokens) returns the blocks of the longest cached prefix and stamps
//    those prefixes with a new clock value;
//  - insert(tokens, blocks) caches every missing prefix of the first
//    min(n_blocks, n_tokens / B) blocks (existing entries keep their block) and
//    stamps all of them;
//  - evict(n) repeatedly removes a leaf prefix (no cached extension) whose
//    block only the cache holds (pool refcount 1), smallest (stamp, block id)
//    first, until n blocks are free or none qualifies.
//  - a physical block is cached under at most one prefix: insert rejects, and
//    changes nothing, when a block it would newly cache is cached already or
//    appears twice among the new ones.
// Edges are runs of whole blocks (path compression), split at block
// boundaries when a sequence diverges inside an edge; stamps are per block.
// The tails of childless nodes are kept in one ordered set keyed by
// (stamp, block).  Stamps never increase along a root-to-leaf path (match and
// insert stamp a prefix of it), so eviction scans that set from its smallest
// key, skipping tails that running sequences still hold.

#include <cstdint>
#include <map>
#include <memory>
#include <new>
#include <vector>

#include "pa_pool.h"

namespace {

struct RNode {
    std::vector<int32_t> tokens;  // edge label: k * B tokens
    std::vector<int32_t> blocks;  // k physical blocks
    std::vector<uint64_t> stamp;  // k last-use stamps
    std::map<std::vector<int32_t>, std::unique_ptr<RNode>> children;  // by the child's first block of tokens
    RNode *parent = nullptr;
};

std::vector<int32_t> key_at(const int32_t *tokens, int64_t pos, int32_t B) {
    return std::vector<int32_t>(tokens + pos, tokens + pos + B);
}

// Leading blocks of `node`'s edge equal to tokens[pos ...], at most `limit`.
int64_t match_blocks(const RNode *node, const int32_t *tokens, int64_t pos, int64_t limit, int32_t B) {
    int64_t k = 0;
    const int64_t nb = (int64_t)node->blocks.size();
    while (k < nb && k < limit) {
        for (int32_t i = 0; i < B; ++i)
            if (node->tokens[k * B + i] != tokens[pos + k * B + i]) return k;
        ++k;
    }
    return k;
}

}  // namespace

using TailKey = std::pair<uint64_t, int32_t>;  // (stamp, block) of a childless node's last block

struct pa_prefix_cache {
    pa_pool *pool = nullptr;
    RNode root;
    uint64_t clock = 0;
    int64_t cached = 0;
    std::vector<uint8_t> in_cache;      // per pool block: cached under some prefix
    std::map<TailKey, RNode *> leaves;  // every childless non-root node, by its tail
};

namespace {

// Split `child` after its first k blocks; returns the new upper node.
RNode *split(RNode *child, int64_t k, int32_t B) {
    RNode *parent = child->parent;
    auto it = parent->children.find(std::vector<int32_t>(child->tokens.begin(), child->tokens.begin() + B));
    std::unique_ptr<RNode> owned = std::move(it->second);
    auto mid = std::make_unique<RNode>();
    mid->parent = parent;
    mid->tokens.assign(child->tokens.begin(), child->tokens.begin() + k * B);
    mid->blocks.assign(child->blocks.begin(), child->blocks.begin() + k);
    mid->stamp.assign(child->stamp.begin(), child->stamp.begin() + k);
    child->tokens.erase(child->tokens.begin(), child->tokens.begin() + k * B);
    child->blocks.erase(child->blocks.begin(), child->blocks.begin() + k);
    child->stamp.erase(child->stamp.begin(), child->stamp.begin() + k);
    child->parent = mid.get();
    RNode *m = mid.get();
    m->children.emplace(std::vector<int32_t>(child->tokens.begin(), child->tokens.begin() + B), std::move(owned));
    it->second = std::move(mid);
    return m;
}

void release_all(pa_pool *pool, RNode *n) {
    for (int32_t b : n->blocks) pa_pool_detail::release_block(pool, b);
    for (auto &c : n->children) release_all(pool, c.second.get());
}

bool is_leaf(const pa_prefix_cache *c, const RNode *n) {
    return n != &c->root && n->children.empty() && !n->blocks.empty();
}

TailKey tail_of(const RNode *n) { return {n->stamp.back(), n->blocks.back()}; }

// Bracket every change to a node's stamps, blocks or children with these two.
void leaf_out(pa_prefix_cache *c, RNode *n) {
    if (is_leaf(c, n)) c->leaves.erase(tail_of(n));
}

void leaf_in(pa_prefix_cache *c, RNode *n) {
    if (is_leaf(c, n)) c->leaves.emplace(tail_of(n), n);
}

// Leading blocks of tokens[0 .. m*B) already cached (a walk without stamping).
int64_t cached_prefix_blocks(const RNode *root, const int32_t *tokens, int64_t m, int32_t B) {
    const RNode *node = root;
    int64_t j = 0;
    while (j < m) {
        auto it = node->children.find(key_at(tokens, j * B, B));
        if (it == node->children.end()) break;
        const RNode *child = it->second.get();
        const int64_t k = match_blocks(child, tokens, j * B, m - j, B);
        j += k;
        if (k < (int64_t)child->blocks.size()) break;
        node = child;
    }
    return j;
}

}  // namespace

extern "C" {

pa_prefix_cache *pa_prefix_cache_create(pa_pool *pool) {
    if (!pool) return nullptr;
    pa_prefix_cache *c = new (std::nothrow) pa_prefix_cache();
    if (!c) return nullptr;
    c->pool = pool;
    try {
        c->in_cache.assign((size_t)pool->num_blocks, 0);
    } catch (const std::bad_alloc &) {
        delete c;
        return nullptr;
    }
    return c;
}

void pa_prefix_cache_destroy(pa_prefix_cache *cache) {
    if (!cache) return;
    for (auto &c : cache->root.children) release_all(cache->pool, c.second.get());
    delete cache;
}

int32_t pa_prefix_match(pa_prefix_cache *cache, const int32_t *tokens, int32_t n_tokens, int32_t *blocks_out,
                        int32_t cap) {
    if (!cache || n_tokens < 0 || (n_tokens > 0 && !tokens) || cap < 0 || (cap > 0 && !blocks_out))
        return -PA_ERR_INVALID;
    const int32_t B = cache->pool->B;
    const uint64_t now = ++cache->clock;
    RNode *node = &cache->root;
    int64_t pos = 0;
    int32_t found = 0;
    while (pos + B <= n_tokens) {
        auto it = node->children.find(key_at(tokens, pos, B));
        if (it == node->children.end()) break;
        RNode *child = it->second.get();
        const int64_t k = match_blocks(child, tokens, pos, (n_tokens - pos) / B, B);
        leaf_out(cache, child);
        for (int64_t j = 0; j < k; ++j) {
            child->stamp[j] = now;
            if (found < cap) blocks_out[found] = child->blocks[j];
            ++found;
        }
        leaf_in(cache, child);
        pos += k * B;
        if (k < (int64_t)child->blocks.size()) break;
        node = child;
    }
    return found;
}

int32_t pa_prefix_insert(pa_prefix_cache *cache, const int32_t *tokens, int32_t n_tokens, const int32_t *blocks,
                         int32_t n_blocks) {
    if (!cache || n_tokens < 0 || n_blocks < 0 || (n_tokens > 0 && !tokens) || (n_blocks > 0 && !blocks))
        return -PA_ERR_INVALID;
    pa_pool *pool = cache->pool;
    const int32_t B = pool->B;
    const int64_t m = n_blocks < n_tokens / B ? n_blocks : n_tokens / B;
    for (int64_t j = 0; j < m; ++j)
        if (blocks[j] < 0 || blocks[j] >= pool->num_blocks || pool->ref[blocks[j]] < 1) return -PA_ERR_BAD_INDEX;
    // prefixes are cached closed under shortening, so the new entries are exactly blocks [j0, m)
    const int64_t j0 = cached_prefix_blocks(&cache->root, tokens, m, B);
    int64_t marked = j0;
    for (; marked < m; ++marked) {
        if (cache->in_cache[blocks[marked]]) break;
        cache->in_cache[blocks[marked]] = 1;
    }
    if (marked < m) {
        for (int64_t q = j0; q < marked; ++q) cache->in_cache[blocks[q]] = 0;
        return -PA_ERR_INVALID;
    }
    const uint64_t now = ++cache->clock;
    RNode *node = &cache->root;
    int64_t pos = 0, j = 0;
    int32_t added = 0;
    while (j < m) {
        auto it = node->children.find(key_at(tokens, pos, B));
        if (it == node->children.end()) {
            auto leaf = std::make_unique<RNode>();
            leaf->parent = node;
            leaf->tokens.assign(tokens + pos, tokens + m * B);
            leaf->blocks.assign(blocks + j, blocks + m);
            leaf->stamp.assign((size_t)(m - j), now);
            for (int32_t b : leaf->blocks) ++pool->ref[b];
            added += (int32_t)(m - j);
            cache->cached += m - j;
            RNode *l = leaf.get();
            leaf_out(cache, node);
            node->children.emplace(key_at(tokens, pos, B), std::move(leaf));
            leaf_in(cache, l);
            break;
        }
        RNode *child = it->second.get();
        const int64_t k = match_blocks(child, tokens, pos, m - j, B);
        leaf_out(cache, child);
        for (int64_t q = 0; q < k; ++q) child->stamp[q] = now;
        pos += k * B;
        j += k;
        if (k < (int64_t)child->blocks.size()) {
            if (j < m) split(child, k, B);  // diverges inside the edge: the upper part gets a child
            leaf_in(cache, child);          // the lower part keeps its tail
            if (j == m) break;              // the sequence ends inside this edge
            node = child->parent;
            continue;
        }
        leaf_in(cache, child);
        node = child;
    }
    return added;
}

int32_t pa_prefix_evict(pa_prefix_cache *cache, int32_t n_blocks) {
    if (!cache || n_blocks < 0) return -PA_ERR_INVALID;
    pa_pool *pool = cache->pool;
    const int32_t B = pool->B;
    int32_t freed = 0;
    // Entries before `it` are tails a sequence still holds; eviction does not
    // change those references, so they stay ineligible for this whole call.
    auto it = cache->leaves.begin();
    auto reinsert = [&](RNode *n) {
        if (!is_leaf(cache, n)) return;
        auto pos = cache->leaves.emplace(tail_of(n), n).first;
        if (it == cache->leaves.end() || pos->first < it->first) it = pos;
    };
    while (freed < n_blocks && it != cache->leaves.end()) {
        RNode *best = it->second;
        const int32_t b = best->blocks.back();
        if (pool->ref[b] != 1) {
            ++it;
            continue;
        }
        it = cache->leaves.erase(it);
        cache->in_cache[b] = 0;
        pa_pool_detail::release_block(pool, b);
        best->blocks.pop_back();
        best->stamp.pop_back();
        best->tokens.resize(best->tokens.size() - B);
        --cache->cached;
        ++freed;
        if (!best->blocks.empty()) {
            reinsert(best);
            continue;
        }
        RNode *parent = best->parent;
        for (auto c = parent->children.begin(); c != parent->children.end(); ++c)
            if (c->second.get() == best) {
                parent->children.erase(c);
                break;
            }
        reinsert(parent);
    }
    return freed;
}

int32_t pa_prefix_cached_blocks(const pa_prefix_cache *cache) {
    return cache ? (int32_t)cache->cached : -PA_ERR_INVALID;
}

int32_t pa_seq_create_from_prefix(pa_pool *pool, const int32_t *blocks, int32_t n_blocks) {
    if (!pool || n_blocks < 0 || (n_blocks > 0 && !blocks)) return -PA_ERR_INVALID;
    for (int32_t j = 0; j < n_blocks; ++j)
        if (blocks[j] < 0 || blocks[j] >= pool->num_blocks || pool->ref[blocks[j]] < 1) return -PA_ERR_BAD_INDEX;
    const int32_t s = pa_seq_create(pool);
    pa_seq_rec &r = pool->seqs[s];
    r.table.assign(blocks, blocks + n_blocks);
    r.len = (int64_t)n_blocks * pool->B;
    for (int32_t j = 0; j < n_blocks; ++j) ++pool->ref[blocks[j]];
    return s;
}

}  // extern "C"
