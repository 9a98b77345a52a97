// Radix-tree prefix cache over the pool's blocks ("SGLang RadixAttention",
// sections on the node and edge structure, on match / split / insert and on
// reference counting with LRU eviction; "Trellis", section "RadixAttention in
// Trellis").  Host only.
//
// Nodes live in a vector (index 0 is the root; freed indices are reused).
// A node's children are keyed by the tokens of their first block: siblings
// always differ there, because an insert that agrees with an edge's first
// block walks into that edge (splitting it if it agrees only in part).
// Evictable leaves (no children, no locks) are found through a min-heap of
// (stamp, node) entries that is validated lazily: an entry is pushed
// whenever a node may have become an evictable leaf or was re-stamped, and
// an entry whose node is gone, has children, is locked or carries a newer
// stamp is dropped when it reaches the top.  Stamps come from a logical
// clock, one tick per match or insert, so the nodes sharing a stamp lie on
// one root path and at most one of them is a leaf: the eviction order is a
// strict order.
#include <algorithm>
#include <functional>
#include <map>
#include <new>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/kvp.h"
#include "kvp_internal.h"

namespace {

struct Node {
    int32_t parent = -1;
    std::vector<int32_t> run;      // token ids: blocks.size() * bs of them
    std::vector<int32_t> blocks;   // pool block ids of this edge
    std::map<std::vector<int32_t>, int32_t> kids;   // first block's tokens -> child
    int32_t locks = 0;
    int64_t stamp = 0;
    bool alive = false;
};

}  // namespace

struct kvp_radix {
    kvp_pool *pool = nullptr;
    int32_t bs = 0;
    int64_t clock = 0;
    std::vector<Node> nodes;
    std::vector<int32_t> spare;    // free node indices
    std::priority_queue<std::pair<int64_t, int32_t>, std::vector<std::pair<int64_t, int32_t>>,
                        std::greater<std::pair<int64_t, int32_t>>>
        leaves;
    std::vector<int32_t> path;     // scratch
};

namespace {

using kvp::pool_block_in_use;
using kvp::pool_drop_block;
using kvp::pool_free_count;
using kvp::pool_hold_block;

std::vector<int32_t> key_at(const int32_t *tokens, int64_t at, int32_t bs) {
    return std::vector<int32_t>(tokens + at, tokens + at + bs);
}

// Whole blocks of node's run that equal tokens[at, end), from the run's start.
int32_t agree(const Node &n, const int32_t *tokens, int64_t at, int64_t end, int32_t bs) {
    int32_t k = 0;
    const int32_t nb = (int32_t)n.blocks.size();
    while (k < nb && at + (int64_t)(k + 1) * bs <= end &&
           std::equal(n.run.begin() + (size_t)k * bs, n.run.begin() + (size_t)(k + 1) * bs,
                      tokens + at + (int64_t)k * bs))
        ++k;
    return k;
}

bool evictable(const kvp_radix *c, int32_t i) {
    const Node &n = c->nodes[i];
    return i != 0 && n.alive && n.kids.empty() && n.locks == 0;
}

void note_leaf(kvp_radix *c, int32_t i) {
    if (evictable(c, i)) c->leaves.push({c->nodes[i].stamp, i});
}

int32_t new_node(kvp_radix *c) {
    int32_t i;
    if (!c->spare.empty()) {
        i = c->spare.back();
        c->spare.pop_back();
        c->nodes[i] = Node{};
    } else {
        i = (int32_t)c->nodes.size();
        c->nodes.emplace_back();
    }
    c->nodes[i].alive = true;
    return i;
}

void release_blocks(kvp_radix *c, Node &n, int32_t *freed) {
    for (auto it = n.blocks.rbegin(); it != n.blocks.rend(); ++it)
        if (pool_drop_block(c->pool, *it) && freed) ++*freed;
    n.blocks.clear();
}

void dump_node(const kvp_radix *c, int32_t i, int32_t depth, std::vector<int32_t> &out) {
    for (const auto &kv : c->nodes[i].kids) {
        const Node &n = c->nodes[kv.second];
        out.push_back(depth);
        out.push_back(n.locks);
        out.push_back((int32_t)n.stamp);
        out.push_back((int32_t)n.run.size());
        out.insert(out.end(), n.run.begin(), n.run.end());
        out.push_back((int32_t)n.blocks.size());
        out.insert(out.end(), n.blocks.begin(), n.blocks.end());
        dump_node(c, kv.second, depth + 1, out);
    }
}

void release_subtree(kvp_radix *c, int32_t i) {
    for (const auto &kv : c->nodes[i].kids) release_subtree(c, kv.second);
    release_blocks(c, c->nodes[i], nullptr);
}

}  // namespace

extern "C" {

int kvp_radix_create(kvp_pool *pool, kvp_radix **out) {
    if (!pool || !out) return KVP_ERR_INVALID;
    kvp_radix *c = new (std::nothrow) kvp_radix;
    if (!c) return KVP_ERR_OOM;
    c->pool = pool;
    c->bs = kvp::pool_block_size(pool);
    c->nodes.emplace_back();
    c->nodes[0].alive = true;
    *out = c;
    return KVP_OK;
}

int kvp_radix_destroy(kvp_radix *c) {
    if (!c) return KVP_ERR_INVALID;
    release_subtree(c, 0);
    delete c;
    return KVP_OK;
}

int kvp_radix_match(kvp_radix *c, const int32_t *tokens, int32_t n_tokens, int32_t *blocks_out,
                    int32_t cap, int32_t *n_blocks_out, int32_t *lock_out) {
    if (!c || n_tokens < 0 || (n_tokens > 0 && !tokens) || !n_blocks_out || !lock_out) return KVP_ERR_INVALID;
    const int32_t bs = c->bs;
    const int64_t end = (int64_t)n_tokens / bs * bs;
    if (end > 0 && (!blocks_out || cap < n_tokens / bs)) return KVP_ERR_INVALID;
    c->clock += 1;
    c->path.clear();
    int32_t node = 0, got = 0;
    int64_t at = 0;
    while (at < end) {
        const auto it = c->nodes[node].kids.find(key_at(tokens, at, bs));
        if (it == c->nodes[node].kids.end()) break;
        const int32_t kid = it->second;
        const Node &kn = c->nodes[kid];
        const int32_t k = agree(kn, tokens, at, end, bs);
        std::copy(kn.blocks.begin(), kn.blocks.begin() + k, blocks_out + got);
        got += k;
        c->path.push_back(kid);
        at += (int64_t)k * bs;
        if (k < (int32_t)kn.blocks.size()) break;
        node = kid;
    }
    for (int32_t i : c->path) {
        c->nodes[i].locks += 1;
        c->nodes[i].stamp = c->clock;
    }
    *n_blocks_out = got;
    *lock_out = c->path.empty() ? -1 : c->path.back();
    return KVP_OK;
}

int kvp_radix_unlock(kvp_radix *c, int32_t lock) {
    if (!c) return KVP_ERR_INVALID;
    if (lock == -1) return KVP_OK;
    if (lock <= 0 || lock >= (int32_t)c->nodes.size() || !c->nodes[lock].alive) return KVP_ERR_INVALID;
    for (int32_t i = lock; i != 0; i = c->nodes[i].parent)
        if (c->nodes[i].locks <= 0) return KVP_ERR_STATE;
    for (int32_t i = lock; i != 0; i = c->nodes[i].parent) {
        c->nodes[i].locks -= 1;
        note_leaf(c, i);
    }
    return KVP_OK;
}

int kvp_radix_insert(kvp_radix *c, const int32_t *tokens, int32_t n_tokens, const int32_t *blocks,
                     int32_t n_blocks) {
    if (!c || n_tokens < 0 || n_blocks < 0 || (n_tokens > 0 && !tokens) || (n_blocks > 0 && !blocks))
        return KVP_ERR_INVALID;
    const int32_t bs = c->bs;
    const int32_t nblk = std::min(n_tokens / bs, n_blocks);
    for (int32_t j = 0; j < nblk; ++j)
        if (!pool_block_in_use(c->pool, blocks[j])) return KVP_ERR_INVALID;
    const int64_t end = (int64_t)nblk * bs;
    c->clock += 1;
    int32_t node = 0;
    int64_t at = 0;
    while (at < end) {
        std::vector<int32_t> key = key_at(tokens, at, bs);
        auto it = c->nodes[node].kids.find(key);
        if (it == c->nodes[node].kids.end()) {
            const int32_t leaf = new_node(c);   // may reallocate nodes
            Node &ln = c->nodes[leaf];
            ln.parent = node;
            ln.run.assign(tokens + at, tokens + end);
            ln.blocks.assign(blocks + at / bs, blocks + nblk);
            ln.stamp = c->clock;
            for (int32_t b : ln.blocks) pool_hold_block(c->pool, b);
            c->nodes[node].kids.emplace(std::move(key), leaf);
            note_leaf(c, leaf);
            return KVP_OK;
        }
        int32_t kid = it->second;
        const int32_t k = agree(c->nodes[kid], tokens, at, end, bs);
        if (k < (int32_t)c->nodes[kid].blocks.size()) {
            // split: the upper node takes the agreeing blocks and the lower
            // node's locks; the lower node keeps the rest and its stamp
            const int32_t up = new_node(c);
            Node &un = c->nodes[up];
            Node &kn = c->nodes[kid];
            un.parent = node;
            un.run.assign(kn.run.begin(), kn.run.begin() + (size_t)k * bs);
            un.blocks.assign(kn.blocks.begin(), kn.blocks.begin() + k);
            un.locks = kn.locks;
            kn.run.erase(kn.run.begin(), kn.run.begin() + (size_t)k * bs);
            kn.blocks.erase(kn.blocks.begin(), kn.blocks.begin() + k);
            kn.parent = up;
            un.kids.emplace(std::vector<int32_t>(kn.run.begin(), kn.run.begin() + bs), kid);
            c->nodes[node].kids[key] = up;
            kid = up;
        }
        c->nodes[kid].stamp = c->clock;
        note_leaf(c, kid);
        node = kid;
        at += (int64_t)k * bs;
    }
    return KVP_OK;
}

int kvp_radix_evict(kvp_radix *c, int32_t need_free, int32_t *freed_out) {
    if (!c || !freed_out) return KVP_ERR_INVALID;
    int32_t freed = 0;
    while (pool_free_count(c->pool) < need_free) {
        int32_t v = -1;
        while (!c->leaves.empty()) {
            const auto top = c->leaves.top();
            c->leaves.pop();
            if (evictable(c, top.second) && c->nodes[top.second].stamp == top.first) {
                v = top.second;
                break;
            }
        }
        if (v < 0) {
            *freed_out = freed;
            return KVP_ERR_OOM;
        }
        Node &n = c->nodes[v];
        const int32_t parent = n.parent;
        c->nodes[parent].kids.erase(std::vector<int32_t>(n.run.begin(), n.run.begin() + c->bs));
        release_blocks(c, n, &freed);
        n = Node{};
        c->spare.push_back(v);
        note_leaf(c, parent);
    }
    *freed_out = freed;
    return KVP_OK;
}

int kvp_radix_dump(const kvp_radix *c, int32_t *out, int64_t cap, int64_t *n_out) {
    if (!c || !n_out) return KVP_ERR_INVALID;
    std::vector<int32_t> words;
    dump_node(c, 0, 0, words);
    *n_out = (int64_t)words.size();
    if ((int64_t)words.size() > cap || (!out && !words.empty())) return KVP_ERR_INVALID;
    std::copy(words.begin(), words.end(), out);
    return KVP_OK;
}

}  // extern "C"
