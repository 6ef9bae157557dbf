// Host-side prefix index for recurrent-state checkpoints.
//
// Prefix caching keeps the DeltaNet state next to the attention context so that a later
// turn restores it instead of recomputing the prompt, and conversations with identical
// opening turns share that state across requests ("HyperQwen: 1,000 tok/s on a Single
// RTX 3090 ...", Technical Insight: 22.4 s -> 0.56 s to first token on a ~25,000-token
// document). dn_prefill_checkpoint writes the state after every 64 tokens; this index
// maps token content to the slot where the caller keeps each such checkpoint, so the
// caller can restore the longest cached 64-token boundary and prefill only the tail.
//
// Structure: a trie whose nodes are chunks of `chunk` tokens. A child is found by the
// hash of its chunk (64-bit), and its tokens are compared exactly, so a hash collision
// can never return a wrong state. Nodes that hold a slot are kept in least-recently-used
// order; inserting into a full index evicts the least recently used slot and reports it.
#include <cstdint>
#include <cstring>
#include <list>
#include <memory>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "dn.h"

namespace dn {
namespace {

uint64_t mix64(uint64_t x) {  // splitmix64 finaliser
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

uint64_t chunk_hash(const int32_t *t, int n) {
    uint64_t h = 0x6a09e667f3bcc909ull;
    for (int i = 0; i < n; ++i) h = mix64(h ^ (uint64_t)(uint32_t)t[i]);
    return h;
}

struct Node {
    std::vector<int32_t> tokens;                     // this chunk's tokens
    std::unordered_multimap<uint64_t, Node *> kids;  // child chunks by hash
    Node *parent = nullptr;
    int32_t slot = -1;                               // checkpoint slot, -1 if none
    std::list<Node *>::iterator lru;                 // position in the LRU list when slot >= 0
};

}  // namespace
}  // namespace dn

struct dn_prefix_cache {
    int chunk = 64;
    int capacity = 0;
    dn::Node root;
    std::vector<std::unique_ptr<dn::Node>> nodes;
    std::list<dn::Node *> lru;  // front = most recently used
    std::mutex mu;
};

namespace dn {
namespace {

Node *find_child(Node *p, const int32_t *t, int n) {
    const uint64_t h = chunk_hash(t, n);
    auto range = p->kids.equal_range(h);
    for (auto it = range.first; it != range.second; ++it)
        if (std::memcmp(it->second->tokens.data(), t, sizeof(int32_t) * n) == 0) return it->second;
    return nullptr;
}

void touch(dn_prefix_cache *c, Node *x) {
    c->lru.erase(x->lru);
    c->lru.push_front(x);
    x->lru = c->lru.begin();
}

}  // namespace
}  // namespace dn

extern "C" dn_prefix_cache *dn_prefix_cache_create(int chunk, int capacity) {
    if (chunk < 1 || capacity < 1) return nullptr;
    dn_prefix_cache *c = new (std::nothrow) dn_prefix_cache();
    if (!c) return nullptr;
    c->chunk = chunk;
    c->capacity = capacity;
    return c;
}

extern "C" void dn_prefix_cache_destroy(dn_prefix_cache *c) { delete c; }

extern "C" dn_status dn_prefix_cache_insert(dn_prefix_cache *c, const int32_t *tokens, int position,
                                            int32_t slot, int32_t *evicted_slot) {
    using namespace dn;
    if (!c || !tokens || !evicted_slot || slot < 0 || position < c->chunk || position % c->chunk)
        return DN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(c->mu);
    *evicted_slot = -1;
    Node *p = &c->root;
    for (int p0 = 0; p0 < position; p0 += c->chunk) {
        Node *x = find_child(p, tokens + p0, c->chunk);
        if (!x) {
            c->nodes.emplace_back(new Node());
            x = c->nodes.back().get();
            x->tokens.assign(tokens + p0, tokens + p0 + c->chunk);
            x->parent = p;
            p->kids.emplace(chunk_hash(tokens + p0, c->chunk), x);
        }
        p = x;
    }
    if (p->slot >= 0) {  // replace this prefix's slot
        *evicted_slot = (p->slot != slot) ? p->slot : -1;
        p->slot = slot;
        touch(c, p);
        return DN_OK;
    }
    if ((int)c->lru.size() >= c->capacity) {
        Node *old = c->lru.back();
        c->lru.pop_back();
        *evicted_slot = old->slot;
        old->slot = -1;
    }
    p->slot = slot;
    c->lru.push_front(p);
    p->lru = c->lru.begin();
    return DN_OK;
}

extern "C" dn_status dn_prefix_cache_lookup(dn_prefix_cache *c, const int32_t *tokens, int n,
                                            int *position, int32_t *slot) {
    using namespace dn;
    if (!c || !position || !slot || n < 0 || (n > 0 && !tokens)) return DN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(c->mu);
    *position = 0;
    *slot = -1;
    Node *p = &c->root, *best = nullptr;
    int best_pos = 0;
    for (int p0 = 0; p0 + c->chunk <= n; p0 += c->chunk) {
        Node *x = find_child(p, tokens + p0, c->chunk);
        if (!x) break;
        p = x;
        if (x->slot >= 0) {
            best = x;
            best_pos = p0 + c->chunk;
        }
    }
    if (best) {
        touch(c, best);
        *position = best_pos;
        *slot = best->slot;
    }
    return DN_OK;
}

extern "C" int dn_prefix_cache_size(dn_prefix_cache *c) {
    if (!c) return -1;
    std::lock_guard<std::mutex> lock(c->mu);
    return (int)c->lru.size();
}
