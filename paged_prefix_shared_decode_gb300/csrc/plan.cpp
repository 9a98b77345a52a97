// Host planner for decode and tree-verify attention, and the attention entry
// points.
//
// Decode plan (cascade over shared blocks):
//  1. A trie over the batch's block tables, keyed at table position j by
//     (physical block id, valid tokens in that block).  Sequences that share a
//     key path share those blocks (prefix sharing from fork / RadixAttention:
//     "Trellis" page, section "RadixAttention in Trellis"; "SGLang
//     RadixAttention" page, radix-tree section).  Chains with one member set
//     are merged into one segment.
//  2. Sequences are ordered by a pre-order walk of the trie so that every
//     segment's members are contiguous, then cut into row tiles of
//     floor(64 / G) sequences (at most 64 query rows: sequences x GQA group).
//  3. A row tile's KV list is every segment any of its members touches, each
//     cut into 64-token tiles tagged with the member interval that sees it.
//     A segment shared by all of a tile's sequences is therefore read once
//     for all of them.
//  4. Long lists are cut into chunks so the grid covers the GPU; chunks of a
//     row tile write partial (o, lse) rows that a merge kernel combines.
// With use_sharing = 0 every sequence is its own row tile over its own table.
//
// Verify plan: row tiles of floor(64 / G) draft nodes of one sequence; the
// context is read in 64-token tiles seen by every node, then one tree-masked
// tile with the draft tokens up to the tile's last node.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "../../include/kvp.h"
#include "kvp_internal.h"

namespace kvp {
namespace {

struct Seg {
    int32_t j0, j1;          // block range [j0, j1)
    int32_t tok0, tok1;      // token range
    int32_t row;             // a member's table row
    int32_t lo, hi;          // members (positions in DFS order) [lo, hi)
};

struct Builder {
    const int32_t *tables;
    const int32_t *lens;
    int32_t S, MB, bs;
    std::vector<int32_t> nblk;
    std::vector<int32_t> order;   // DFS order of sequences
    std::vector<Seg> segs;

    int32_t valid(int32_t s, int32_t j) const { return std::min(bs, lens[s] - j * bs); }
    int64_t key(int32_t s, int32_t j) const {
        return ((int64_t)tables[(size_t)s * MB + j] << 8) | (int64_t)(valid(s, j) & 0xFF);
    }

    // members share blocks [0, j); emit their subtree
    void build(const std::vector<int32_t> &members, int32_t j) {
        // members whose path ends here come first in the order
        std::vector<int32_t> rest;
        for (int32_t s : members) {
            if (nblk[s] <= j) order.push_back(s);
            else rest.push_back(s);
        }
        // group by key at j, first-seen order
        std::vector<std::vector<int32_t>> groups;
        std::vector<int64_t> keys;
        for (int32_t s : rest) {
            int64_t k = key(s, j);
            size_t g = 0;
            while (g < keys.size() && keys[g] != k) ++g;
            if (g == keys.size()) { keys.push_back(k); groups.emplace_back(); }
            groups[g].push_back(s);
        }
        for (auto &g : groups) {
            int32_t j1 = j + 1;
            if (g.size() == 1) {
                j1 = nblk[g[0]];
            } else {
                for (;; ++j1) {
                    bool same = true;
                    for (int32_t s : g) {
                        if (nblk[s] <= j1 || key(s, j1) != key(g[0], j1)) { same = false; break; }
                    }
                    if (!same) break;
                }
            }
            size_t seg_index = segs.size();
            segs.push_back(Seg{j, j1, j * bs, std::min(j1 * bs, lens[g[0]]), g[0], 0, 0});
            int32_t lo = (int32_t)order.size();
            build(g, j1);
            segs[seg_index].lo = lo;
            segs[seg_index].hi = (int32_t)order.size();
        }
    }
};

int sm_count_cached() {
    static int sms = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            sms = v;
        else
            sms = 152;
    });
    return sms;
}

struct HostPlan {
    std::vector<WorkItem> items;
    std::vector<KvTile> tiles;
    std::vector<int32_t> members;
    std::vector<MergeDesc> merge;
    int32_t n_row_tiles = 0, n_partial_rows = 0, ts = 1;
    int64_t unique_kv_bytes = 0;
};

// A row tile: members (query tokens) + its 64-token KV tiles (before chunking).
struct RowTile {
    std::vector<int32_t> members;
    std::vector<KvTile> kv;
};

void push_range(std::vector<KvTile> &kv, int32_t row, int32_t t0, int32_t t1, int32_t lo,
                int32_t hi, int32_t flags) {
    for (int32_t t = t0; t < t1; t += kTileTokens) {
        int32_t n = std::min(kTileTokens, t1 - t);
        kv.push_back(KvTile{row, t, n | (flags << 16), lo | (hi << 16)});
    }
}

// Chunk row tiles into work items and lay out partial rows and merge info.
void finish(HostPlan &hp, std::vector<RowTile> &rts, int32_t G, int32_t nq, int32_t layers_heads,
            int sms) {
    int64_t total_tiles = 0;
    int32_t max_rows = 0;
    for (auto &rt : rts) {
        total_tiles += (int64_t)rt.kv.size();
        max_rows = std::max(max_rows, (int32_t)rt.members.size() * G);
    }
    // aim for about 4 CTAs per SM over all (layer, kv head) pairs
    int64_t target_items = std::max<int64_t>(1, (4LL * sms + layers_heads - 1) / layers_heads);
    int64_t chunk = std::max<int64_t>(4, (total_tiles + target_items - 1) / target_items);
    hp.merge.assign(nq, MergeDesc{0, 0, 0, 0});
    hp.n_row_tiles = (int32_t)rts.size();
    int32_t P = 0;
    struct Pending { WorkItem it; int64_t cost; };
    std::vector<Pending> pend;
    for (auto &rt : rts) {
        int32_t nm = (int32_t)rt.members.size();
        int32_t rows = nm * G;
        int32_t moff = (int32_t)hp.members.size();
        hp.members.insert(hp.members.end(), rt.members.begin(), rt.members.end());
        int64_t nt = (int64_t)rt.kv.size();
        int64_t nchunks = std::max<int64_t>(1, (nt + chunk - 1) / chunk);
        int32_t base = -1;
        if (nchunks > 1) {
            base = P;
            P += (int32_t)nchunks * rows;
            for (int32_t m = 0; m < nm; ++m)
                hp.merge[rt.members[m]] = MergeDesc{base, rows, (int32_t)nchunks, m};
        }
        int32_t tbase = (int32_t)hp.tiles.size();
        hp.tiles.insert(hp.tiles.end(), rt.kv.begin(), rt.kv.end());
        for (int64_t c = 0; c < nchunks; ++c) {
            int64_t b = nt * c / nchunks, e = nt * (c + 1) / nchunks;
            WorkItem it{};
            it.tile_begin = tbase + (int32_t)b;
            it.tile_end = tbase + (int32_t)e;
            it.member_off = moff;
            it.n_members = nm;
            it.out_base = nchunks > 1 ? base + (int32_t)c * rows : -1;
            pend.push_back(Pending{it, (e - b) * (64 + rows)});
        }
    }
    std::stable_sort(pend.begin(), pend.end(),
                     [](const Pending &a, const Pending &b) { return a.cost > b.cost; });
    for (auto &p : pend) hp.items.push_back(p.it);
    hp.n_partial_rows = P;
    int32_t rg = (max_rows + 15) / 16;
    hp.ts = rg <= 1 ? 4 : (rg <= 2 ? 2 : 1);
}

int build_decode(const kvp_attn_desc &d, const int32_t *tables, const int32_t *lens, int32_t S,
                 int32_t MB, int sms, HostPlan &hp) {
    const int32_t bs = d.block_size, G = d.num_q_heads / d.num_kv_heads;
    Builder b{tables, lens, S, MB, bs, std::vector<int32_t>(S), {}, {}};
    for (int32_t s = 0; s < S; ++s) {
        if (lens[s] <= 0) return KVP_ERR_INVALID;
        int64_t nb = ((int64_t)lens[s] + bs - 1) / bs;
        if (nb > MB) return KVP_ERR_INVALID;
        b.nblk[s] = (int32_t)nb;
        for (int32_t j = 0; j < nb; ++j) {
            int32_t id = tables[(size_t)s * MB + j];
            if (id < 0 || id >= d.num_blocks) return KVP_ERR_INVALID;
        }
    }
    std::vector<RowTile> rts;
    const int64_t tok_bytes = 2LL * d.num_kv_heads * d.head_dim * 2 * d.num_layers;
    if (d.use_sharing) {
        std::vector<int32_t> all(S);
        std::iota(all.begin(), all.end(), 0);
        b.build(all, 0);
        for (auto &sg : b.segs) hp.unique_kv_bytes += (int64_t)(sg.tok1 - sg.tok0) * tok_bytes;
        const int32_t per_tile = std::max(1, 64 / G);
        for (int32_t lo = 0; lo < S; lo += per_tile) {
            int32_t hi = std::min(S, lo + per_tile);
            RowTile rt;
            rt.members.assign(b.order.begin() + lo, b.order.begin() + hi);
            for (auto &sg : b.segs) {   // pre-order: a segment precedes its subtree
                int32_t a = std::max(lo, sg.lo), e = std::min(hi, sg.hi);
                if (a >= e) continue;
                push_range(rt.kv, sg.row, sg.tok0, sg.tok1, a - lo, e - lo, 0);
            }
            rts.push_back(std::move(rt));
        }
    } else {
        for (int32_t s = 0; s < S; ++s) {
            hp.unique_kv_bytes += (int64_t)lens[s] * tok_bytes;
            RowTile rt;
            rt.members.push_back(s);
            push_range(rt.kv, s, 0, lens[s], 0, 1, 0);
            rts.push_back(std::move(rt));
        }
    }
    finish(hp, rts, G, S, d.num_layers * d.num_kv_heads, sms);
    return KVP_OK;
}

int build_verify(const kvp_attn_desc &d, const int32_t *ctx, int32_t B, int32_t n, int32_t MB,
                 int sms, HostPlan &hp) {
    const int32_t bs = d.block_size, G = d.num_q_heads / d.num_kv_heads;
    if (n <= 0 || n > 64) return KVP_ERR_INVALID;
    const int64_t tok_bytes = 2LL * d.num_kv_heads * d.head_dim * 2 * d.num_layers;
    std::vector<RowTile> rts;
    const int32_t per_tile = std::max(1, 64 / G);
    for (int32_t b = 0; b < B; ++b) {
        if (ctx[b] < 0 || ((int64_t)ctx[b] + n + bs - 1) / bs > MB) return KVP_ERR_INVALID;
        hp.unique_kv_bytes += (int64_t)(ctx[b] + n) * tok_bytes;
        for (int32_t i0 = 0; i0 < n; i0 += per_tile) {
            int32_t i1 = std::min(n, i0 + per_tile);
            RowTile rt;
            for (int32_t i = i0; i < i1; ++i) rt.members.push_back(b * n + i);
            push_range(rt.kv, b, 0, ctx[b], 0, i1 - i0, 0);
            // draft tokens 0 .. i1-1 (ancestors have smaller indices), tree-masked
            push_range(rt.kv, b, ctx[b], ctx[b] + i1, 0, i1 - i0, kTileTree);
            rts.push_back(std::move(rt));
        }
    }
    finish(hp, rts, G, B * n, d.num_layers * d.num_kv_heads, sms);
    return KVP_OK;
}

bool desc_ok(const kvp_attn_desc *d) {
    return d && d->num_layers > 0 && d->num_q_heads > 0 && d->num_kv_heads > 0 &&
           d->num_q_heads % d->num_kv_heads == 0 && d->num_q_heads / d->num_kv_heads <= 64 &&
           (d->head_dim == 64 || d->head_dim == 128) && d->block_size > 0 && d->num_blocks > 0;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    size_t items, tiles, members, merge, part_o, part_lse, total, plan_bytes;
};

WsLayout layout(const HostPlan &hp, const kvp_attn_desc &d) {
    WsLayout w{};
    size_t off = sizeof(WsHeader);
    w.items = off;   off = align256(off + sizeof(WorkItem) * hp.items.size());
    w.tiles = off;   off = align256(off + sizeof(KvTile) * hp.tiles.size());
    w.members = off; off = align256(off + sizeof(int32_t) * hp.members.size());
    w.merge = off;   off = align256(off + sizeof(MergeDesc) * hp.merge.size());
    w.plan_bytes = off;
    const size_t lh = (size_t)d.num_layers * d.num_kv_heads * (size_t)hp.n_partial_rows;
    w.part_o = off;  off = align256(off + sizeof(float) * lh * d.head_dim);
    w.part_lse = off; off = align256(off + sizeof(float) * lh);
    w.total = off;
    return w;
}

// Host image of the plan region, reused across calls on the same thread.
thread_local std::vector<unsigned char> t_image;

int run(const HostPlan &hp, const kvp_attn_desc &d, const void *q, const void *k_pool,
        const void *v_pool, const int32_t *tables, int32_t MB, int32_t nq, const int32_t *parent,
        int32_t n_draft, void *out, float *lse, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!q || !k_pool || !v_pool || !tables || !out || !ws) return KVP_ERR_INVALID;
    if (((uintptr_t)ws & 255) != 0) return KVP_ERR_INVALID;
    if (((uintptr_t)q | (uintptr_t)k_pool | (uintptr_t)v_pool | (uintptr_t)out) & 15)
        return KVP_ERR_INVALID;
    WsLayout w = layout(hp, d);
    if (ws_bytes < w.total) return KVP_ERR_INVALID;
    t_image.assign(w.plan_bytes, 0);
    unsigned char *img = t_image.data();
    WsHeader h{};
    h.n_items = (int32_t)hp.items.size();
    h.n_tiles = (int32_t)hp.tiles.size();
    h.n_members = (int32_t)hp.members.size();
    h.n_merge = (int32_t)hp.merge.size();
    h.n_partial_rows = hp.n_partial_rows;
    std::memcpy(img, &h, sizeof h);
    std::memcpy(img + w.items, hp.items.data(), sizeof(WorkItem) * hp.items.size());
    std::memcpy(img + w.tiles, hp.tiles.data(), sizeof(KvTile) * hp.tiles.size());
    std::memcpy(img + w.members, hp.members.data(), sizeof(int32_t) * hp.members.size());
    std::memcpy(img + w.merge, hp.merge.data(), sizeof(MergeDesc) * hp.merge.size());
    // pageable source: staged before the call returns
    if (cudaMemcpyAsync(ws, img, w.plan_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return KVP_ERR_CUDA;
    unsigned char *base = (unsigned char *)ws;
    AttnLaunch a{};
    a.q = q; a.k_pool = k_pool; a.v_pool = v_pool; a.tables = tables;
    a.MB = MB; a.NB = d.num_blocks; a.bs = d.block_size;
    a.Hq = d.num_q_heads; a.Hkv = d.num_kv_heads; a.G = d.num_q_heads / d.num_kv_heads;
    a.nq = nq; a.L = d.num_layers; a.D = d.head_dim;
    float scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt((float)d.head_dim);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.tree_parent = parent; a.n_draft = n_draft;
    a.out = out; a.lse = lse;
    a.err = (int32_t *)base;
    a.items = (const WorkItem *)(base + w.items);
    a.tiles = (const KvTile *)(base + w.tiles);
    a.members = (const int32_t *)(base + w.members);
    a.merge = (const MergeDesc *)(base + w.merge);
    a.part_o = (float *)(base + w.part_o);
    a.part_lse = (float *)(base + w.part_lse);
    a.n_items = (int32_t)hp.items.size();
    a.n_merge_q = hp.n_partial_rows > 0 ? nq : 0;
    a.P = hp.n_partial_rows;
    a.ts = hp.ts;
    return launch_attention(a, stream) == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" {

size_t kvp_decode_workspace_size(const kvp_attn_desc *desc, const int32_t *h_block_tables,
                                 const int32_t *h_seq_lens, int32_t num_seqs, int32_t max_blocks) {
    if (!desc_ok(desc) || num_seqs <= 0 || max_blocks <= 0 || !h_block_tables || !h_seq_lens) return 0;
    HostPlan hp;
    if (build_decode(*desc, h_block_tables, h_seq_lens, num_seqs, max_blocks, sm_count_cached(), hp))
        return 0;
    return layout(hp, *desc).total;
}

int paged_decode_attention(const void *q, const void *k_pool, const void *v_pool,
                           const int32_t *block_tables, const int32_t *h_block_tables,
                           const int32_t *h_seq_lens, int32_t num_seqs, int32_t max_blocks,
                           const kvp_attn_desc *desc, void *out, float *lse, void *workspace,
                           size_t ws_bytes, void *stream) {
    if (!desc_ok(desc) || num_seqs <= 0 || max_blocks <= 0 || !h_block_tables || !h_seq_lens)
        return KVP_ERR_INVALID;
    HostPlan hp;
    int rc = build_decode(*desc, h_block_tables, h_seq_lens, num_seqs, max_blocks, sm_count_cached(), hp);
    if (rc) return rc;
    return run(hp, *desc, q, k_pool, v_pool, block_tables, max_blocks, num_seqs, nullptr, 0, out,
               lse, workspace, ws_bytes, (cudaStream_t)stream);
}

size_t kvp_verify_workspace_size(const kvp_attn_desc *desc, const int32_t *h_ctx_lens,
                                 int32_t batch, int32_t n_draft) {
    if (!desc_ok(desc) || batch <= 0 || !h_ctx_lens) return 0;
    HostPlan hp;
    if (build_verify(*desc, h_ctx_lens, batch, n_draft, INT32_MAX / 2, sm_count_cached(), hp)) return 0;
    return layout(hp, *desc).total;
}

int tree_verify_attention(const void *q, const int32_t *tree_parent, int32_t n_draft,
                          const void *k_pool, const void *v_pool, const int32_t *block_tables,
                          const int32_t *h_ctx_lens, int32_t batch, int32_t max_blocks,
                          const kvp_attn_desc *desc, void *out, float *lse, void *workspace,
                          size_t ws_bytes, void *stream) {
    if (!desc_ok(desc) || batch <= 0 || max_blocks <= 0 || !h_ctx_lens || !tree_parent)
        return KVP_ERR_INVALID;
    HostPlan hp;
    int rc = build_verify(*desc, h_ctx_lens, batch, n_draft, max_blocks, sm_count_cached(), hp);
    if (rc) return rc;
    return run(hp, *desc, q, k_pool, v_pool, block_tables, max_blocks, batch * n_draft, tree_parent,
               n_draft, out, lse, workspace, ws_bytes, (cudaStream_t)stream);
}

int kvp_device_error(void *workspace, void *stream, int32_t *err_out) {
    if (!workspace || !err_out) return KVP_ERR_INVALID;
    int32_t v = 0;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
    if (v != 0 && cudaMemsetAsync(workspace, 0, sizeof v, st) != cudaSuccess) return KVP_ERR_CUDA;
    *err_out = v;
    return KVP_OK;
}

int kvp_decode_plan_stats(const kvp_attn_desc *desc, const int32_t *h_block_tables,
                          const int32_t *h_seq_lens, int32_t num_seqs, int32_t max_blocks,
                          int32_t sm_count, int32_t *n_items, int32_t *n_row_tiles,
                          int32_t *n_kv_tiles, int32_t *n_partial_rows, int64_t *unique_kv_bytes) {
    if (!desc_ok(desc) || num_seqs <= 0 || max_blocks <= 0 || !h_block_tables || !h_seq_lens ||
        sm_count <= 0)
        return KVP_ERR_INVALID;
    HostPlan hp;
    int rc = build_decode(*desc, h_block_tables, h_seq_lens, num_seqs, max_blocks, sm_count, hp);
    if (rc) return rc;
    if (n_items) *n_items = (int32_t)hp.items.size();
    if (n_row_tiles) *n_row_tiles = hp.n_row_tiles;
    if (n_kv_tiles) *n_kv_tiles = (int32_t)hp.tiles.size();
    if (n_partial_rows) *n_partial_rows = hp.n_partial_rows;
    if (unique_kv_bytes) *unique_kv_bytes = hp.unique_kv_bytes;
    return KVP_OK;
}

}  // extern "C"
