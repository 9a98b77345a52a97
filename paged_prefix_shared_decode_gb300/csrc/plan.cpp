// Host planner for decode and tree-verify attention, and the attention entry
// points.
//
// Decode plan (cascade over shared blocks):
//  1. A trie over the batch's block tables, keyed at table position j by
//     (physical block id, valid tokens in that block).  Sequences that share
//     a key path share those blocks -- the prefix sharing that fork and
//     RadixAttention create ("Trellis" page, section "RadixAttention in
//     Trellis"; "SGLang RadixAttention" page, radix-tree section).  Chains
//     with one member set are merged into one segment.
//  2. Sequences are ordered by a pre-order walk of the trie, so every
//     segment's members are contiguous, and cut into row tiles of
//     floor(64 / G) sequences (at most 64 query rows: sequences x GQA group).
//  3. Within a row tile, every segment that two or more of its sequences see
//     goes into the tile's shared item as 64-token KV tiles tagged with the
//     member interval that sees them: one read of such a tile serves all of
//     those sequences.  Tokens that only one sequence of the tile sees go
//     into a per-sequence private item (G rows, four warps splitting tokens).
//  4. Items longer than needed to fill the GPU are cut into chunks.  A query
//     row whose keys span several item chunks gets partial (o, lse) rows that
//     the merge kernel combines by log-sum-exp; otherwise it is written
//     directly.
// With use_sharing = 0 every sequence is one private item over its own table.
//
// Verify plan: row tiles of floor(64 / G) draft nodes of one sequence; each
// reads the context in 64-token tiles seen by every node, then one
// tree-masked tile with the draft tokens up to the tile's last node.
//
// The plan carries each tile's physical block ids, so the kernels read no
// device block table; block tables are consumed here, on the host.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <numeric>
#include <unordered_map>
#include <vector>

#include "../../include/kvp.h"
#include "kvp_internal.h"

namespace kvp {
namespace {

struct Seg {
    int32_t tok0, tok1;   // token range
    int32_t row;          // a member's table row
    int32_t lo, hi;       // members (positions in pre-order) [lo, hi)
};

struct HostPlan {
    std::vector<WorkItem> items;      // mma.sync kernel
    std::vector<WorkItem> tc_items;   // tcgen05 kernel
    std::vector<KvTile> tiles;
    std::vector<int32_t> members;
    std::vector<MergeDesc> merge;
    std::vector<int32_t> entries;
    int32_t n_row_tiles = 0, n_partial_rows = 0, n_units = 0, n_tc_units = 0;
    int32_t n_tree_q = 0;   // query tokens with a draft-tree mask (verify)
    int64_t unique_kv_bytes = 0;

    void clear() {
        items.clear();
        tc_items.clear();
        tiles.clear();
        members.clear();
        merge.clear();
        entries.clear();
        n_row_tiles = n_partial_rows = n_units = n_tc_units = n_tree_q = 0;
        unique_kv_bytes = 0;
    }
};

// Items before chunking, stored flat: item i has members [m0, m1) of `mem`
// (query tokens) and KV tiles [t0, t1) of `kv`.
struct Protos {
    struct Item {
        int32_t m0, m1, t0, t1;
    };
    std::vector<int32_t> mem;
    std::vector<KvTile> kv;
    std::vector<Item> items;
    void clear() {
        mem.clear();
        kv.clear();
        items.clear();
    }
    int32_t n_mem(const Item &it) const { return it.m1 - it.m0; }
    int32_t n_kv(const Item &it) const { return it.t1 - it.t0; }
};

// Working storage of the planner, kept per thread so that planning a batch
// allocates nothing once the buffers have grown to its size.
struct Scratch {
    std::vector<int32_t> nblk, order, members, gid, tmp, gcount, bounds, priv_seg, priv_cnt;
    std::vector<int64_t> gkeys;
    std::unordered_map<int64_t, int32_t> gmap;
    std::vector<Seg> segs;
    Protos protos, packed;
    std::vector<int32_t> cur_mem;
    std::vector<KvTile> cur_kv;
    std::vector<int32_t> cover, ent_cnt, ent_pos;
    struct Chunked {
        WorkItem it;
        int64_t cost;
        int32_t idx;
        bool tc;
    };
    std::vector<Chunked> cs;
};

struct Builder {
    const int32_t *tables;
    const int32_t *lens;
    int32_t S, MB, bs;
    Scratch &sc;

    int32_t valid(int32_t s, int32_t j) const { return std::min(bs, lens[s] - j * bs); }
    int64_t key(int32_t s, int32_t j) const {
        return ((int64_t)tables[(size_t)s * MB + j] << 24) | (int64_t)valid(s, j);
    }

    // First block index >= from where rows s0 and s1 differ in block id or
    // valid tokens, or where either row ends.  Below the shorter row's last
    // block both hold full blocks, so only that block's valid count needs
    // comparing.
    int32_t agree(int32_t s0, int32_t s1, int32_t from) const {
        const int32_t lim = std::min(sc.nblk[s0], sc.nblk[s1]);
        const int32_t *r0 = tables + (size_t)s0 * MB, *r1 = tables + (size_t)s1 * MB;
        int32_t x = from;
        while (x < lim && r0[x] == r1[x]) ++x;
        if (x == lim && lim > from && valid(s0, lim - 1) != valid(s1, lim - 1)) x = lim - 1;
        return x;
    }

    // The n members at m (rows of the tables) share blocks [0, j); emit their
    // subtree.  Members whose rows end at j come first in pre-order; the rest
    // are regrouped in place by the key of block j, groups in order of first
    // appearance (a linear scan while there are few distinct keys, a hash map
    // after), and each group is handled in turn.
    void build(int32_t *m, int32_t n, int32_t j) {
        int32_t nr = 0;
        for (int32_t i = 0; i < n; ++i) {
            if (sc.nblk[m[i]] <= j) sc.order.push_back(m[i]);
            else m[nr++] = m[i];
        }
        if (nr == 0) return;
        sc.gkeys.clear();
        sc.gmap.clear();
        sc.gid.resize(nr);
        for (int32_t i = 0; i < nr; ++i) {
            const int64_t k = key(m[i], j);
            int32_t g = (int32_t)sc.gkeys.size();
            if (sc.gmap.empty()) {
                for (int32_t x = 0; x < (int32_t)sc.gkeys.size(); ++x)
                    if (sc.gkeys[x] == k) { g = x; break; }
                if (g == (int32_t)sc.gkeys.size() && sc.gkeys.size() == 16)
                    for (int32_t x = 0; x < 16; ++x) sc.gmap.emplace(sc.gkeys[x], x);
            }
            if (!sc.gmap.empty()) g = sc.gmap.emplace(k, (int32_t)sc.gkeys.size()).first->second;
            if (g == (int32_t)sc.gkeys.size()) sc.gkeys.push_back(k);
            sc.gid[i] = g;
        }
        const int32_t ng = (int32_t)sc.gkeys.size();
        // group boundaries of this call sit on a shared stack: the recursion
        // below reuses every other scratch buffer
        const size_t base = sc.bounds.size();
        sc.bounds.resize(base + ng + 1, 0);
        for (int32_t i = 0; i < nr; ++i) sc.bounds[base + sc.gid[i] + 1] += 1;
        for (int32_t g = 0; g < ng; ++g) sc.bounds[base + g + 1] += sc.bounds[base + g];
        sc.gcount.assign(sc.bounds.begin() + base, sc.bounds.begin() + base + ng);
        sc.tmp.resize(nr);
        for (int32_t i = 0; i < nr; ++i) sc.tmp[sc.gcount[sc.gid[i]]++] = m[i];
        std::copy(sc.tmp.begin(), sc.tmp.begin() + nr, m);
        for (int32_t g = 0; g < ng; ++g) {
            int32_t *gm = m + sc.bounds[base + g];
            const int32_t gn = sc.bounds[base + g + 1] - sc.bounds[base + g];
            if (gn == 1) {   // a single member: its whole remaining row is one segment
                const int32_t s0 = gm[0];
                sc.segs.push_back(Seg{j * bs, lens[s0], s0, (int32_t)sc.order.size(), (int32_t)sc.order.size() + 1});
                sc.order.push_back(s0);
                continue;
            }
            // the group shares blocks [j, j1): j1 is the first block where
            // some member's key differs from the first member's (or a row
            // ends), found row by row
            int32_t j1 = sc.nblk[gm[0]];
            for (int32_t i = 1; i < gn && j1 > j + 1; ++i) j1 = std::min(j1, agree(gm[0], gm[i], j + 1));
            const size_t si = sc.segs.size();
            sc.segs.push_back(Seg{j * bs, std::min(j1 * bs, lens[gm[0]]), gm[0], 0, 0});
            const int32_t lo = (int32_t)sc.order.size();
            build(gm, gn, j1);
            sc.segs[si].lo = lo;
            sc.segs[si].hi = (int32_t)sc.order.size();
        }
        sc.bounds.resize(base);
    }
};

thread_local Scratch t_scratch;
thread_local HostPlan t_plan;

}  // namespace

// Items with more rows than this run on the tcgen05 kernel.  By default that
// is every many-row item for head dim 128 (verify, MCTS: measured 1.9x and
// 1.25x faster than mma.sync) and none for head dim 64, where the mma.sync
// kernel measured faster on the shared-prefix decode shapes.
// KVP_ATTN_PATH=tc / =mma in the environment forces one path (ablations).
int tc_row_threshold(int head_dim) {
    static int mode = [] {
        const char *e = std::getenv("KVP_ATTN_PATH");
        if (e && std::strcmp(e, "tc") == 0) return 1;
        if (e && std::strcmp(e, "mma") == 0) return 2;
        return 0;
    }();
    if (mode == 2) return INT32_MAX;
    if (mode == 1 || head_dim == 128) return 32;
    return INT32_MAX;
}

namespace {

bool tc_usable(const kvp_attn_desc &d) {
    return tc_row_threshold(d.head_dim) != INT32_MAX &&
           tc_path_supported(d.num_layers, d.num_blocks, d.num_kv_heads, d.block_size);
}

// Query rows per row tile on the mma.sync kernel.  Fewer rows per tile means
// more tiles read the same shared blocks (from L2, since their units run back
// to back) for cheaper per-tile work; 64 rows measured fastest on the decode
// shapes.  KVP_MMA_ROWS (16, 32 or 64) overrides it for ablations.
int32_t mma_tile_rows() {
    static int rows = [] {
        const char *e = std::getenv("KVP_MMA_ROWS");
        int v = e ? std::atoi(e) : 64;
        return (v == 16 || v == 32 || v == 64) ? v : 64;
    }();
    return rows;
}

// Members per row tile: 128 query rows when the tcgen05 kernel is in use.
int32_t members_per_tile(int32_t G, bool tc) {
    return std::max(1, (tc ? kTcRows : mma_tile_rows()) / G);
}

struct TileSrc {
    const int32_t *tables;
    int32_t MB, bs;
};

void push_range(std::vector<KvTile> &kv, const TileSrc &src, int32_t row, int32_t t0, int32_t t1,
                int32_t lo, int32_t hi, int32_t flags) {
    const int32_t *tr = src.tables + (size_t)row * src.MB;
    for (int32_t t = t0; t < t1; t += kTileTokens) {
        int32_t n = std::min(kTileTokens, t1 - t);
        KvTile k{};
        k.tok0 = t;
        k.ntok_flags = n | (flags << 16);
        k.members = lo | (hi << 16);
        int32_t jb = t / src.bs, je = (t + n - 1) / src.bs;
        for (int32_t j = jb; j <= je; ++j) k.blk[j - jb] = tr[j];
        for (int32_t j = je - jb + 1; j < kTileBlocks; ++j) k.blk[j] = 0;
        kv.push_back(k);
    }
}

// Opens an item of `protos` whose members are given; tiles are then pushed
// to protos.kv and close_item() ends it (an item without tiles is dropped).
void open_item(Protos &pr, const int32_t *mem, int32_t n) {
    pr.items.push_back(Protos::Item{(int32_t)pr.mem.size(), 0, (int32_t)pr.kv.size(), 0});
    pr.mem.insert(pr.mem.end(), mem, mem + n);
    pr.items.back().m1 = (int32_t)pr.mem.size();
}
void close_item(Protos &pr) {
    Protos::Item &it = pr.items.back();
    it.t1 = (int32_t)pr.kv.size();
    if (it.t1 == it.t0) {
        pr.mem.resize(it.m0);
        pr.items.pop_back();
    }
}

// Chunk items into work items, lay out partial rows and merge lists.  Items
// with more than `thr` rows go to the tcgen05 kernel (one CTA per SM), the
// rest to the mma.sync kernel (`mma_ctas` CTAs per SM).
// Items of at most 16 rows and a few tiles cost more in per-unit start-up
// than in work; pack them into items of up to 32 rows, each tile keeping the
// member interval of the item it came from.  (A tile of one member leaves
// the warps of the other members' rows idle, so packs stay small: 32 rows
// measured 8% faster than 64 on Trellis phi = 0.9 and equal on MCTS; no
// packing made MCTS 43% slower.  With a GQA group of 8 or more, packs of 16
// rows -- at most two members, whose tiles the four warps split four ways --
// measured 2% faster on Dendrite and 3% on Trellis phi = 0.75, and 16 rows
// for small groups made MCTS 3% slower.)
void pack_small(Scratch &sc, int32_t G, int thr) {
    // stay on the mma.sync kernel: at most 32 rows and at most the threshold
    const int kPackRows = G >= 8 ? 16 : (thr < 32 ? thr : 32);
    constexpr int kPackTiles = 4, kPackMaxTiles = 64;
    const Protos &in = sc.protos;
    Protos &out = sc.packed;
    out.clear();
    sc.cur_mem.clear();
    sc.cur_kv.clear();
    auto flush = [&]() {
        if (sc.cur_mem.empty()) return;
        open_item(out, sc.cur_mem.data(), (int32_t)sc.cur_mem.size());
        out.kv.insert(out.kv.end(), sc.cur_kv.begin(), sc.cur_kv.end());
        close_item(out);
        sc.cur_mem.clear();
        sc.cur_kv.clear();
    };
    for (const auto &p : in.items) {
        const int rows = in.n_mem(p) * G;
        const bool small = rows <= 16 && rows <= thr && in.n_kv(p) <= kPackTiles;
        if (!small) {
            open_item(out, in.mem.data() + p.m0, in.n_mem(p));
            out.kv.insert(out.kv.end(), in.kv.begin() + p.t0, in.kv.begin() + p.t1);
            close_item(out);
            continue;
        }
        if ((int)(sc.cur_mem.size() + in.n_mem(p)) * G > kPackRows ||
            (int)(sc.cur_kv.size() + in.n_kv(p)) > kPackMaxTiles)
            flush();
        const int32_t off = (int32_t)sc.cur_mem.size();
        sc.cur_mem.insert(sc.cur_mem.end(), in.mem.begin() + p.m0, in.mem.begin() + p.m1);
        for (int32_t t = p.t0; t < p.t1; ++t) {
            KvTile k = in.kv[t];
            const int32_t lo = (k.members & 0xFFFF) + off, hi = (k.members >> 16) + off;
            k.members = lo | (hi << 16);
            sc.cur_kv.push_back(k);
        }
    }
    flush();
}

void finish(HostPlan &hp, Scratch &sc, int32_t G, int32_t nq, int32_t layers_heads, int32_t sms,
            int32_t mma_ctas, int thr, bool kv4 = false) {
    pack_small(sc, G, thr);
    const Protos &pr = sc.packed;
    auto &cs = sc.cs;
    cs.clear();
    sc.cover.assign(nq, 0);
    for (int pass = 0; pass < 2; ++pass) {
        const bool tc = pass == 1;
        int64_t total_tiles = 0, n_protos = 0;
        for (const auto &p : pr.items) {
            if ((pr.n_mem(p) * G > thr) != tc) continue;
            total_tiles += pr.n_kv(p);
            n_protos += 1;
        }
        if (n_protos == 0) continue;
        // about one work unit per resident CTA: longest first off the atomic
        // queue balances them, and fewer, longer units pay fewer unit
        // start-ups and leave fewer partial rows to merge (two per CTA
        // measured 8% slower on Dendrite, 3/4 per CTA 11% slower)
        // (4-bit pages: a quarter more, since their tiles cost more to expand
        // than to load; measured 2.6% faster on Dendrite, and 0.75 / 1.25 /
        // 1.5 per CTA slower on bf16 pages)
        const int64_t target_units = tc ? 1LL * sms : (kv4 ? 5LL * sms * mma_ctas / 4 : 1LL * sms * mma_ctas);
        int64_t chunk = kMaxItemTiles;
        if (n_protos * layers_heads < target_units) {
            int64_t want = (total_tiles * layers_heads + target_units - 1) / target_units;
            chunk = std::max<int64_t>(4, std::min<int64_t>(chunk, want));
        }
        for (const auto &p : pr.items) {
            if ((pr.n_mem(p) * G > thr) != tc) continue;
            const int32_t moff = (int32_t)hp.members.size();
            hp.members.insert(hp.members.end(), pr.mem.begin() + p.m0, pr.mem.begin() + p.m1);
            const int64_t nt = pr.n_kv(p);
            const int64_t nchunks = std::max<int64_t>(1, (nt + chunk - 1) / chunk);
            const int32_t tbase = (int32_t)hp.tiles.size();
            hp.tiles.insert(hp.tiles.end(), pr.kv.begin() + p.t0, pr.kv.begin() + p.t1);
            const int32_t nm = pr.n_mem(p), rows = nm * G;
            for (int64_t c = 0; c < nchunks; ++c) {
                const int64_t b = nt * c / nchunks, e = nt * (c + 1) / nchunks;
                WorkItem it{};
                it.tile_begin = tbase + (int32_t)b;
                it.tile_end = tbase + (int32_t)e;
                it.member_off = moff;
                it.n_members = nm;
                it.out_base = 0;
                // rows beyond 16 cost tensor and exp work per tile
                cs.push_back(Scratch::Chunked{it, (e - b) * (64 + std::max(16, rows)), (int32_t)cs.size(), tc});
                for (int32_t x = p.m0; x < p.m1; ++x) sc.cover[pr.mem[x]] += 1;
            }
        }
    }
    // partial rows for every chunk whose members are not all covered once;
    // each query's merge entries in chunk order
    int32_t P = 0;
    sc.ent_cnt.assign(nq + 1, 0);
    for (auto &c : cs) {
        bool direct = true;
        for (int32_t m = 0; m < c.it.n_members; ++m)
            if (sc.cover[hp.members[c.it.member_off + m]] != 1) direct = false;
        if (direct) {
            c.it.out_base = -1;
        } else {
            c.it.out_base = P;
            for (int32_t m = 0; m < c.it.n_members; ++m) sc.ent_cnt[hp.members[c.it.member_off + m] + 1] += 1;
            P += c.it.n_members * G;
        }
    }
    for (int32_t q = 0; q < nq; ++q) sc.ent_cnt[q + 1] += sc.ent_cnt[q];
    hp.entries.resize(sc.ent_cnt[nq]);
    sc.ent_pos.assign(sc.ent_cnt.begin(), sc.ent_cnt.end() - 1);
    for (const auto &c : cs) {
        if (c.it.out_base < 0) continue;
        for (int32_t m = 0; m < c.it.n_members; ++m)
            hp.entries[sc.ent_pos[hp.members[c.it.member_off + m]]++] = c.it.out_base + m * G;
    }
    hp.merge.resize(nq);
    for (int32_t q = 0; q < nq; ++q) hp.merge[q] = MergeDesc{sc.ent_cnt[q], sc.ent_cnt[q + 1] - sc.ent_cnt[q]};
    // longest first; equal costs keep their order
    std::sort(cs.begin(), cs.end(), [](const Scratch::Chunked &a, const Scratch::Chunked &b) {
        return a.cost != b.cost ? a.cost > b.cost : a.idx < b.idx;
    });
    for (const auto &c : cs) (c.tc ? hp.tc_items : hp.items).push_back(c.it);
    hp.n_partial_rows = P;
    hp.n_units = (int32_t)hp.items.size() * layers_heads;
    hp.n_tc_units = (int32_t)hp.tc_items.size() * layers_heads;
}


int build_decode(const kvp_attn_desc &d, const int32_t *tables, const int32_t *lens, int32_t S,
                 int32_t MB, int sms, HostPlan &hp) {
    const int32_t bs = d.block_size, G = d.num_q_heads / d.num_kv_heads;
    Scratch &sc = t_scratch;
    sc.nblk.resize(S);
    for (int32_t s = 0; s < S; ++s) {
        if (lens[s] <= 0) return KVP_ERR_INVALID;
        int64_t nb = ((int64_t)lens[s] + bs - 1) / bs;
        if (nb > MB) return KVP_ERR_INVALID;
        sc.nblk[s] = (int32_t)nb;
        for (int32_t j = 0; j < nb; ++j) {
            int32_t id = tables[(size_t)s * MB + j];
            if (id < 0 || id >= d.num_blocks) return KVP_ERR_INVALID;
        }
    }
    TileSrc src{tables, MB, bs};
    Protos &pr = sc.protos;
    pr.clear();
    // K and V rows in the pool's format: d bf16 values, or d / 2 code bytes and
    // one exponent byte
    const int64_t tok_bytes = 2LL * d.num_kv_heads * d.num_layers *
                              (d.kv_format == KVP_KV_4BIT ? d.head_dim / 2 + 1 : d.head_dim * 2);
    if (d.use_sharing) {
        sc.order.clear();
        sc.segs.clear();
        sc.bounds.clear();
        sc.members.resize(S);
        std::iota(sc.members.begin(), sc.members.end(), 0);
        Builder b{tables, lens, S, MB, bs, sc};
        b.build(sc.members.data(), S, 0);
        for (const auto &sg : sc.segs) hp.unique_kv_bytes += (int64_t)(sg.tok1 - sg.tok0) * tok_bytes;
        const int32_t per_tile = members_per_tile(G, tc_usable(d));
        for (int32_t lo = 0; lo < S; lo += per_tile) {
            const int32_t hi = std::min(S, lo + per_tile);
            hp.n_row_tiles += 1;
            // the tile's shared item: segments that two or more of its members see
            open_item(pr, sc.order.data() + lo, hi - lo);
            sc.priv_seg.clear();
            for (int32_t i = 0; i < (int32_t)sc.segs.size(); ++i) {   // pre-order: a segment precedes its subtree
                const Seg &sg = sc.segs[i];
                const int32_t a = std::max(lo, sg.lo), e = std::min(hi, sg.hi);
                if (a >= e) continue;
                if (e - a >= 2) push_range(pr.kv, src, sg.row, sg.tok0, sg.tok1, a - lo, e - lo, 0);
                else sc.priv_seg.push_back(((a - lo) << 20) | i);   // a member's own segment
            }
            close_item(pr);
            // one private item per member, its segments in pre-order
            sc.priv_cnt.assign(hi - lo + 1, 0);
            for (int32_t x : sc.priv_seg) sc.priv_cnt[(x >> 20) + 1] += 1;
            for (int32_t m = 0; m < hi - lo; ++m) sc.priv_cnt[m + 1] += sc.priv_cnt[m];
            sc.tmp.resize(sc.priv_seg.size());
            sc.gcount.assign(sc.priv_cnt.begin(), sc.priv_cnt.end() - 1);
            for (int32_t x : sc.priv_seg) sc.tmp[sc.gcount[x >> 20]++] = x & 0xFFFFF;
            for (int32_t m = 0; m < hi - lo; ++m) {
                if (sc.priv_cnt[m] == sc.priv_cnt[m + 1]) continue;
                open_item(pr, sc.order.data() + lo + m, 1);
                for (int32_t k = sc.priv_cnt[m]; k < sc.priv_cnt[m + 1]; ++k) {
                    const Seg &sg = sc.segs[sc.tmp[k]];
                    push_range(pr.kv, src, sg.row, sg.tok0, sg.tok1, 0, 1, 0);
                }
                close_item(pr);
            }
        }
    } else {
        for (int32_t s = 0; s < S; ++s) {
            hp.unique_kv_bytes += (int64_t)lens[s] * tok_bytes;
            hp.n_row_tiles += 1;
            open_item(pr, &s, 1);
            push_range(pr.kv, src, s, 0, lens[s], 0, 1, 0);
            close_item(pr);
        }
    }
    finish(hp, sc, G, S, d.num_layers * d.num_kv_heads, sms, attention_ctas_per_sm(d.head_dim),
           tc_usable(d) ? tc_row_threshold(d.head_dim) : INT32_MAX, d.kv_format == KVP_KV_4BIT);
    return KVP_OK;
}

int build_verify(const kvp_attn_desc &d, const int32_t *tables, const int32_t *ctx, int32_t B,
                 int32_t n, int32_t MB, int sms, HostPlan &hp) {
    const int32_t bs = d.block_size, G = d.num_q_heads / d.num_kv_heads;
    if (n <= 0 || n > kMaxDraft) return KVP_ERR_INVALID;
    const int64_t tok_bytes = 2LL * d.num_kv_heads * d.head_dim * 2 * d.num_layers;
    TileSrc src{tables, MB, bs};
    Scratch &sc = t_scratch;
    Protos &pr = sc.protos;
    pr.clear();
    const int32_t per_tile = members_per_tile(G, tc_usable(d));
    for (int32_t b = 0; b < B; ++b) {
        if (ctx[b] < 0) return KVP_ERR_INVALID;
        int64_t nb = ((int64_t)ctx[b] + n + bs - 1) / bs;
        if (nb > MB) return KVP_ERR_INVALID;
        for (int32_t j = 0; j < nb; ++j) {
            int32_t id = tables[(size_t)b * MB + j];
            if (id < 0 || id >= d.num_blocks) return KVP_ERR_INVALID;
        }
        hp.unique_kv_bytes += (int64_t)(ctx[b] + n) * tok_bytes;
        for (int32_t i0 = 0; i0 < n; i0 += per_tile) {
            int32_t i1 = std::min(n, i0 + per_tile);
            hp.n_row_tiles += 1;
            sc.members.clear();
            for (int32_t i = i0; i < i1; ++i) sc.members.push_back(b * n + i);
            open_item(pr, sc.members.data(), i1 - i0);
            push_range(pr.kv, src, b, 0, ctx[b], 0, i1 - i0, 0);
            // draft tokens 0 .. i1-1 (ancestors have smaller indices), tree-masked
            push_range(pr.kv, src, b, ctx[b], ctx[b] + i1, 0, i1 - i0, kTileTree);
            close_item(pr);
        }
    }
    finish(hp, sc, G, B * n, d.num_layers * d.num_kv_heads, sms, attention_ctas_per_sm(d.head_dim),
           tc_usable(d) ? tc_row_threshold(d.head_dim) : INT32_MAX);
    hp.n_tree_q = B * n;
    return KVP_OK;
}

bool desc_ok(const kvp_attn_desc *d) {
    if (!d || d->num_layers <= 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 ||
        d->num_q_heads % d->num_kv_heads != 0 || d->num_q_heads / d->num_kv_heads > 64 ||
        (d->head_dim != 64 && d->head_dim != 128) || d->num_blocks <= 0)
        return false;
    // power-of-two block sizes >= 16: a 64-token tile touches at most 5 blocks
    const int32_t bs = d->block_size;
    return bs >= 16 && bs <= (1 << 20) && (bs & (bs - 1)) == 0 &&
           (d->kv_format == KVP_KV_BF16 || d->kv_format == KVP_KV_4BIT);
}

int log2_int(int32_t x) {
    int r = 0;
    while ((1 << r) < x) ++r;
    return r;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    size_t items, tc_items, tiles, members, merge, entries, part_o, part_lse, tree_mask, total, plan_bytes;
};

WsLayout layout(const HostPlan &hp, const kvp_attn_desc &d) {
    WsLayout w{};
    size_t off = sizeof(WsHeader);
    w.items = off;   off = align256(off + sizeof(WorkItem) * hp.items.size());
    w.tc_items = off; off = align256(off + sizeof(WorkItem) * hp.tc_items.size());
    w.tiles = off;   off = align256(off + sizeof(KvTile) * hp.tiles.size());
    w.members = off; off = align256(off + sizeof(int32_t) * hp.members.size());
    w.merge = off;   off = align256(off + sizeof(MergeDesc) * hp.merge.size());
    w.entries = off; off = align256(off + sizeof(int32_t) * hp.entries.size());
    w.plan_bytes = off;
    const size_t lh = (size_t)d.num_layers * d.num_kv_heads * (size_t)hp.n_partial_rows;
    w.part_o = off;  off = align256(off + sizeof(float) * lh * d.head_dim);
    w.part_lse = off; off = align256(off + sizeof(float) * lh);
    w.tree_mask = off; off = align256(off + sizeof(uint64_t) * (size_t)hp.n_tree_q);
    w.total = off;
    return w;
}

// A plan packed for upload: the host image of the workspace's plan region
// and what the launch takes from the plan.  The image is pageable on
// purpose: a small pageable copy travels with the copy command itself, which
// measured faster than a copy from page-locked memory.
struct Packed {
    std::vector<unsigned char> image;
    WsLayout w{};
    int32_t n_units = 0, n_tc_units = 0, n_partial_rows = 0;
};

void pack(const HostPlan &hp, const kvp_attn_desc &d, Packed &pk) {
    pk.w = layout(hp, d);
    const WsLayout &w = pk.w;
    pk.image.assign(w.plan_bytes, 0);
    unsigned char *img = pk.image.data();
    WsHeader h{};
    h.n_items = (int32_t)hp.items.size();
    h.n_tc_items = (int32_t)hp.tc_items.size();
    h.n_units = hp.n_units;
    h.n_tiles = (int32_t)hp.tiles.size();
    h.n_members = (int32_t)hp.members.size();
    h.n_entries = (int32_t)hp.entries.size();
    h.n_partial_rows = hp.n_partial_rows;
    std::memcpy(img, &h, sizeof h);
    std::memcpy(img + w.items, hp.items.data(), sizeof(WorkItem) * hp.items.size());
    std::memcpy(img + w.tc_items, hp.tc_items.data(), sizeof(WorkItem) * hp.tc_items.size());
    std::memcpy(img + w.tiles, hp.tiles.data(), sizeof(KvTile) * hp.tiles.size());
    std::memcpy(img + w.members, hp.members.data(), sizeof(int32_t) * hp.members.size());
    std::memcpy(img + w.merge, hp.merge.data(), sizeof(MergeDesc) * hp.merge.size());
    std::memcpy(img + w.entries, hp.entries.data(), sizeof(int32_t) * hp.entries.size());
    pk.n_units = hp.n_units;
    pk.n_tc_units = hp.n_tc_units;
    pk.n_partial_rows = hp.n_partial_rows;
}

thread_local Packed t_packed;
thread_local cudaEvent_t t_ev_before = nullptr, t_ev_after = nullptr;
std::atomic<long long> g_launches{0};

// An append whose bookkeeping is done and whose device write is issued
// between the plan upload and the attention launch, so that the attention
// kernel follows the write kernel directly in the stream (and may start
// while it finishes).
struct StagedAppend {
    kvp_pool *pool;
    const std::vector<int32_t> *slots, *cow;
    const void *k, *v;
};

// Uploads a packed plan into the workspace, issues a staged append, and
// launches the attention kernels (and the merge).
// (uploaded: the kernel right before wrote the plan into the workspace.)
int launch_packed(const Packed &pk, const kvp_attn_desc &d, const void *q, const void *k_pool,
                  const void *v_pool, int32_t nq, const int32_t *parent, int32_t n_draft, void *out,
                  float *lse, void *ws, size_t ws_bytes, cudaStream_t stream, const void *k_exp = nullptr,
                  const void *v_exp = nullptr, const StagedAppend *append = nullptr, bool uploaded = false) {
    if (!q || !k_pool || !v_pool || !out || !ws) return KVP_ERR_INVALID;
    const bool kv4 = d.kv_format == KVP_KV_4BIT;
    if (kv4 && (!k_exp || !v_exp || (((uintptr_t)k_exp | (uintptr_t)v_exp) & 15))) return KVP_ERR_INVALID;
    if (((uintptr_t)ws & 255) != 0) return KVP_ERR_INVALID;
    if (((uintptr_t)q | (uintptr_t)k_pool | (uintptr_t)v_pool | (uintptr_t)out) & 15)
        return KVP_ERR_INVALID;
    if ((uintptr_t)lse & 3) return KVP_ERR_INVALID;
    const WsLayout &w = pk.w;
    if (ws_bytes < w.total) return KVP_ERR_INVALID;
    // pageable source: the copy is staged before the call returns
    if (!uploaded &&
        cudaMemcpyAsync(ws, pk.image.data(), w.plan_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return KVP_ERR_CUDA;
    if (append) {
        const int rc = append_issue_lists(append->pool, *append->slots, *append->cow, append->k, append->v, stream);
        if (rc) return rc;
    }
    unsigned char *base = (unsigned char *)ws;
    AttnLaunch a{};
    a.q = q; a.k_pool = k_pool; a.v_pool = v_pool;
    a.k_exp = k_exp; a.v_exp = v_exp; a.kv4 = kv4 ? 1 : 0;
    a.NB = d.num_blocks; a.bs_log2 = log2_int(d.block_size);
    a.Hq = d.num_q_heads; a.Hkv = d.num_kv_heads; a.G = d.num_q_heads / d.num_kv_heads;
    a.nq = nq; a.L = d.num_layers; a.D = d.head_dim;
    float scale = d.scale > 0.f ? d.scale : 1.0f / std::sqrt((float)d.head_dim);
    a.scale_log2 = scale * 1.4426950408889634f;
    a.tree_parent = parent; a.n_draft = n_draft;
    a.out = out; a.lse = lse;
    a.err = (int32_t *)base;
    a.counter = (int32_t *)base + 1;
    a.tc_counter = (int32_t *)base + 2;
    a.items = (const WorkItem *)(base + w.items);
    a.tc_items = (const WorkItem *)(base + w.tc_items);
    a.tiles = (const KvTile *)(base + w.tiles);
    a.members = (const int32_t *)(base + w.members);
    a.merge = (const MergeDesc *)(base + w.merge);
    a.entries = (const int32_t *)(base + w.entries);
    a.part_o = (float *)(base + w.part_o);
    a.part_lse = (float *)(base + w.part_lse);
    a.tree_mask = parent ? (uint64_t *)(base + w.tree_mask) : nullptr;
    a.n_units = pk.n_units;
    a.n_tc_units = pk.n_tc_units;
    a.n_merge_q = pk.n_partial_rows > 0 ? nq : 0;
    a.P = pk.n_partial_rows;
    a.wait_first = uploaded ? 1 : 0;
    return launch_attention(a, stream, t_ev_before, t_ev_after) == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

int run(const HostPlan &hp, const kvp_attn_desc &d, const void *q, const void *k_pool,
        const void *v_pool, int32_t nq, const int32_t *parent, int32_t n_draft, void *out,
        float *lse, void *ws, size_t ws_bytes, cudaStream_t stream, const void *k_exp = nullptr,
        const void *v_exp = nullptr) {
    pack(hp, d, t_packed);
    return launch_packed(t_packed, d, q, k_pool, v_pool, nq, parent, n_draft, out, lse, ws, ws_bytes, stream,
                         k_exp, v_exp);
}

// The plan's own invariants, for the host-side stats call: every item's
// tiles lie inside the tile list and fit the kernels' descriptor stage, its
// rows fit its kernel's unit, and every tile holds 1..64 tokens and a member
// interval inside its item.
bool plan_consistent(const HostPlan &hp, int32_t G) {
    const int32_t nt = (int32_t)hp.tiles.size();
    auto item_ok = [&](const WorkItem &it, int32_t max_rows) {
        if (it.tile_begin < 0 || it.tile_end <= it.tile_begin || it.tile_end > nt) return false;
        if (it.tile_end - it.tile_begin > kMaxItemTiles || it.n_members <= 0 || it.n_members * G > max_rows)
            return false;
        for (int32_t t = it.tile_begin; t < it.tile_end; ++t) {
            const KvTile &k = hp.tiles[t];
            const int32_t lo = k.members & 0xFFFF, hi = k.members >> 16, n = k.ntok_flags & 0xFFFF;
            if (n < 1 || n > kTileTokens || hi <= lo || hi > it.n_members) return false;
        }
        return true;
    };
    for (const WorkItem &it : hp.items)
        if (!item_ok(it, kMmaMaxRows)) return false;
    for (const WorkItem &it : hp.tc_items)
        if (!item_ok(it, kTcRows)) return false;
    return true;
}

bool desc_matches_pool(const kvp_attn_desc &d, const PoolView &pv) {
    return d.num_layers == pv.L && d.num_kv_heads == pv.Hkv && d.head_dim == pv.d &&
           d.block_size == pv.bs && d.num_blocks == pv.NB &&
           d.kv_format == (pv.kv4 ? KVP_KV_4BIT : KVP_KV_BF16);
}

// The decode plan of pool sequences at their current lengths.
int plan_pool(const kvp_pool *pool, const int32_t *seqs, int32_t n, const kvp_attn_desc &d,
              HostPlan &hp) {
    int32_t width = 0, *tables = nullptr, *lens = nullptr;
    int rc = pool_tables(pool, seqs, n, &width, &tables, &lens);
    if (rc) return rc;
    return build_decode(d, tables, lens, n, width, device_sm_count(), hp);
}

int run_pool(const HostPlan &hp, const kvp_attn_desc &d, const PoolView &pv, const void *q, int32_t n,
             void *out, float *lse, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return run(hp, d, q, pv.k, pv.v, n, nullptr, 0, out, lse, ws, ws_bytes, stream,
               pv.kv4 ? pv.k_exp : nullptr, pv.kv4 ? pv.v_exp : nullptr);
}

}  // namespace

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int device_sm_count() {
    static std::atomic<int> cache[kMaxDevices] = {};
    const int dev = current_device();
    if (dev < 0) return 152;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

}  // namespace kvp

using namespace kvp;

extern "C" {

size_t kvp_decode_workspace_size(const kvp_attn_desc *desc, const int32_t *block_tables,
                                 const int32_t *seq_lens, int32_t num_seqs, int32_t max_blocks) {
    if (!desc_ok(desc) || num_seqs <= 0 || max_blocks <= 0 || !block_tables || !seq_lens) return 0;
    HostPlan &hp = t_plan;
    hp.clear();
    if (build_decode(*desc, block_tables, seq_lens, num_seqs, max_blocks, device_sm_count(), hp))
        return 0;
    return layout(hp, *desc).total;
}

int paged_decode_attention(const void *q, const void *k_pool, const void *v_pool,
                           const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                           int32_t max_blocks, const kvp_attn_desc *desc, void *out, float *lse,
                           void *workspace, size_t ws_bytes, void *stream) {
    if (!desc_ok(desc) || desc->kv_format != KVP_KV_BF16 || num_seqs <= 0 || max_blocks <= 0 ||
        !block_tables || !seq_lens)
        return KVP_ERR_INVALID;
    HostPlan &hp = t_plan;
    hp.clear();
    int rc = build_decode(*desc, block_tables, seq_lens, num_seqs, max_blocks, device_sm_count(), hp);
    if (rc) return rc;
    return run(hp, *desc, q, k_pool, v_pool, num_seqs, nullptr, 0, out, lse, workspace, ws_bytes,
               (cudaStream_t)stream);
}

int paged_decode_attention_kv4(const void *q, const void *k_codes, const void *k_exps,
                               const void *v_codes, const void *v_exps, const int32_t *block_tables,
                               const int32_t *seq_lens, int32_t num_seqs, int32_t max_blocks,
                               const kvp_attn_desc *desc, void *out, float *lse, void *workspace,
                               size_t ws_bytes, void *stream) {
    if (!desc_ok(desc) || desc->kv_format != KVP_KV_4BIT || num_seqs <= 0 || max_blocks <= 0 ||
        !block_tables || !seq_lens)
        return KVP_ERR_INVALID;
    HostPlan &hp = t_plan;
    hp.clear();
    int rc = build_decode(*desc, block_tables, seq_lens, num_seqs, max_blocks, device_sm_count(), hp);
    if (rc) return rc;
    return run(hp, *desc, q, k_codes, v_codes, num_seqs, nullptr, 0, out, lse, workspace, ws_bytes,
               (cudaStream_t)stream, k_exps, v_exps);
}

size_t kvp_pool_decode_workspace_size(const kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs,
                                      const kvp_attn_desc *desc) {
    if (!pool || !desc_ok(desc) || !desc_matches_pool(*desc, pool_view(pool))) return 0;
    HostPlan &hp = t_plan;
    hp.clear();
    if (plan_pool(pool, seq_ids, num_seqs, *desc, hp)) return 0;
    return layout(hp, *desc).total;
}

int paged_decode_attention_pool(const kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs,
                                const void *q, void *out, float *lse, const kvp_attn_desc *desc,
                                void *workspace, size_t ws_bytes, void *stream) {
    if (!pool || !desc_ok(desc)) return KVP_ERR_INVALID;
    const PoolView pv = pool_view(pool);
    if (!desc_matches_pool(*desc, pv)) return KVP_ERR_INVALID;
    HostPlan &hp = t_plan;
    hp.clear();
    int rc = plan_pool(pool, seq_ids, num_seqs, *desc, hp);
    if (rc) return rc;
    return run_pool(hp, *desc, pv, q, num_seqs, out, lse, workspace, ws_bytes, (cudaStream_t)stream);
}

}  // extern "C"

// A decode step planned ahead of its launch: the append's bookkeeping is
// done (the sequences hold the new tokens), its device write is staged as
// slot and copy-on-write lists, and the attention plan over the grown
// sequences is packed for upload.
struct kvp_step_plan {
    kvp_pool *pool = nullptr;
    kvp_attn_desc desc{};
    int32_t num_seqs = 0, ntok = 0;
    bool ready = false;                // planned and not yet run
    std::vector<int32_t> slots, cow;   // the append's device write
    Packed pk;
};

namespace {

bool a16(const void *p) { return ((uintptr_t)p & 15) == 0; }

struct StepBytes {
    size_t kv, q, lse;
};
StepBytes step_bytes(const kvp_attn_desc &d, int32_t num_seqs, int32_t ntok) {
    const size_t rows = (size_t)d.num_layers * num_seqs * d.num_q_heads;
    return StepBytes{(size_t)d.num_layers * num_seqs * ntok * d.num_kv_heads * d.head_dim * 2,
                     rows * d.head_dim * 2, rows * sizeof(float)};
}

// Everything about a step's buffers that the launch would reject.
int check_io(const kvp_step_io *io, int32_t ntok) {
    if (!io || (io->flags & ~(uint32_t)KVP_STEP_HOST_MAPPED)) return KVP_ERR_INVALID;
    const bool mapped = (io->flags & KVP_STEP_HOST_MAPPED) != 0;
    const void *out = mapped && io->h_out ? io->h_out : io->d_out;
    const float *lse = mapped && io->h_lse ? io->h_lse : io->d_lse;
    if (!io->d_q || !out || !a16(io->d_q) || !a16(out) || ((uintptr_t)lse & 3)) return KVP_ERR_INVALID;
    if (!mapped && ((io->h_out && !io->d_out) || (io->h_lse && !io->d_lse))) return KVP_ERR_INVALID;
    if (mapped && !(a16(io->h_k_new) && a16(io->h_v_new) && a16(io->h_q))) return KVP_ERR_INVALID;
    if (ntok > 0 && (!io->d_k_new || !io->d_v_new || !a16(io->d_k_new) || !a16(io->d_v_new)))
        return KVP_ERR_INVALID;
    return KVP_OK;
}

// Step 1: the inputs to the device buffers (copy-engine transfers, or one
// copy kernel over all of them from mapped host memory).
int step_inputs(const kvp_step_io *io, const StepBytes &b, int32_t ntok, cudaStream_t st) {
    if (io->flags & KVP_STEP_HOST_MAPPED) {
        const void *src[3];
        void *dst[3];
        int64_t len[3];
        int n = 0;
        if (io->h_k_new && ntok > 0) {
            src[n] = io->h_k_new, dst[n] = io->d_k_new, len[n++] = (int64_t)b.kv;
            src[n] = io->h_v_new, dst[n] = io->d_v_new, len[n++] = (int64_t)b.kv;
        }
        if (io->h_q) src[n] = io->h_q, dst[n] = io->d_q, len[n++] = (int64_t)b.q;
        return launch_copy_segments(src, dst, len, n, st) == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
    }
    if (io->h_k_new && ntok > 0 &&
        (cudaMemcpyAsync(io->d_k_new, io->h_k_new, b.kv, cudaMemcpyHostToDevice, st) != cudaSuccess ||
         cudaMemcpyAsync(io->d_v_new, io->h_v_new, b.kv, cudaMemcpyHostToDevice, st) != cudaSuccess))
        return KVP_ERR_CUDA;
    if (io->h_q && cudaMemcpyAsync(io->d_q, io->h_q, b.q, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    return KVP_OK;
}

// The host half: the append's bookkeeping and the plan over the grown
// sequences (the append was checked to fit).  For a pool whose tables are
// consistent, planning after a committed append cannot fail.
int plan_step(kvp_step_plan &sp, kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs, int32_t ntok,
              const kvp_attn_desc &d, const int32_t *ntoks) {
    sp.pool = pool;
    sp.desc = d;
    sp.num_seqs = num_seqs;
    sp.ntok = ntok;
    sp.slots.clear();
    sp.cow.clear();
    if (ntok > 0) {
        int32_t total = 0;
        const int rc = append_batch_commit_lists(pool, num_seqs, seq_ids, ntoks, sp.slots, sp.cow, &total);
        if (rc) return rc;
    }
    HostPlan &hp = t_plan;
    hp.clear();
    const int rc = plan_pool(pool, seq_ids, num_seqs, d, hp);
    if (rc) return rc;
    pack(hp, d, sp.pk);
    sp.ready = true;
    return KVP_OK;
}

// The device half after the inputs: plan upload, the append's write,
// attention, merge, then the outputs' copies.  With too small a workspace
// only the append is written.
int launch_step(kvp_step_plan &sp, const kvp_step_io *io, void *ws, size_t ws_bytes, cudaStream_t st) {
    sp.ready = false;
    const PoolView pv = pool_view(sp.pool);
    const bool mapped = (io->flags & KVP_STEP_HOST_MAPPED) != 0;
    void *out = mapped && io->h_out ? io->h_out : io->d_out;
    float *lse = mapped && io->h_lse ? io->h_lse : io->d_lse;
    if (ws_bytes < sp.pk.w.total) {   // the pool already holds the new tokens: write them
        if (!sp.slots.empty() &&
            append_issue_lists(sp.pool, sp.slots, sp.cow, io->d_k_new, io->d_v_new, st) != KVP_OK)
            return KVP_ERR_CUDA;
        return KVP_ERR_WORKSPACE;
    }
    const StagedAppend staged{sp.pool, &sp.slots, &sp.cow, io->d_k_new, io->d_v_new};
    int rc = launch_packed(sp.pk, sp.desc, io->d_q, pv.k, pv.v, sp.num_seqs, nullptr, 0, out, lse, ws, ws_bytes,
                           st, pv.kv4 ? pv.k_exp : nullptr, pv.kv4 ? pv.v_exp : nullptr,
                           sp.slots.empty() ? nullptr : &staged);
    if (rc || mapped) return rc;
    const StepBytes b = step_bytes(sp.desc, sp.num_seqs, sp.ntok);
    if (io->h_out && cudaMemcpyAsync(io->h_out, io->d_out, b.q, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    if (io->h_lse && cudaMemcpyAsync(io->h_lse, io->d_lse, b.lse, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    return KVP_OK;
}

// The planned step with its inputs already on the device or in mapped host
// memory, on a bf16 pool with a small append and plan: one kernel writes the
// append (new K/V from d_k_new, or straight from h_k_new when mapped), q
// (from h_q when mapped) and the plan image into the workspace; attention and
// merge follow, then (unmapped) the outputs' copies.  *launched = false when
// the step does not qualify (nothing enqueued).
int launch_fused(kvp_step_plan &sp, const kvp_step_io *io, void *ws, size_t ws_bytes, cudaStream_t st,
                 bool *launched) {
    *launched = false;
    const bool mapped = (io->flags & KVP_STEP_HOST_MAPPED) != 0;
    if (!mapped && (io->h_k_new || io->h_v_new || io->h_q)) return KVP_OK;
    const PoolView pv = pool_view(sp.pool);
    if (pv.kv4 || ws_bytes < sp.pk.w.total) return KVP_OK;
    KvWrite w{};
    w.k_pool = const_cast<void *>(pv.k);
    w.v_pool = const_cast<void *>(pv.v);
    w.k = mapped && io->h_k_new ? io->h_k_new : io->d_k_new;
    w.v = mapped && io->h_v_new ? io->h_v_new : io->d_v_new;
    w.L = pv.L; w.NB = pv.NB; w.Hkv = pv.Hkv; w.bs = pv.bs; w.d = pv.d;
    w.ntok = (int32_t)sp.slots.size();
    w.slots = sp.slots.data();
    w.ncow = (int32_t)(sp.cow.size() / 3);
    w.cow = sp.cow.data();
    if (!step_write_fits(w, sp.pk.w.plan_bytes)) return KVP_OK;
    *launched = true;
    sp.ready = false;
    const StepBytes b = step_bytes(sp.desc, sp.num_seqs, sp.ntok);
    if (launch_step_write(w, mapped ? io->h_q : nullptr, io->d_q, b.q, sp.pk.image.data(), ws, sp.pk.w.plan_bytes,
                          st) != cudaSuccess)
        return KVP_ERR_CUDA;
    void *out = mapped && io->h_out ? io->h_out : io->d_out;
    float *lse = mapped && io->h_lse ? io->h_lse : io->d_lse;
    int rc = launch_packed(sp.pk, sp.desc, io->d_q, pv.k, pv.v, sp.num_seqs, nullptr, 0, out, lse, ws, ws_bytes, st,
                           nullptr, nullptr, nullptr, true);
    if (rc || mapped) return rc;
    if (io->h_out && cudaMemcpyAsync(io->h_out, io->d_out, b.q, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    if (io->h_lse && cudaMemcpyAsync(io->h_lse, io->d_lse, b.lse, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KVP_ERR_CUDA;
    return KVP_OK;
}

// The checks shared by kvp_decode_step and kvp_decode_step_plan; fills the
// per-sequence token counts.
int check_step(kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs, int32_t ntok, const kvp_attn_desc *desc,
               std::vector<int32_t> &ntoks) {
    if (!pool || !desc_ok(desc) || num_seqs <= 0 || !seq_ids || ntok < 0) return KVP_ERR_INVALID;
    if (!desc_matches_pool(*desc, pool_view(pool))) return KVP_ERR_INVALID;
    if ((int64_t)num_seqs * ntok > INT32_MAX / 2) return KVP_ERR_INVALID;
    ntoks.assign(num_seqs, ntok);
    if (ntok > 0) return append_batch_check(pool, num_seqs, seq_ids, ntoks.data());
    return KVP_OK;
}

thread_local kvp_step_plan t_step;
thread_local std::vector<int32_t> t_ntoks;

}  // namespace

extern "C" {

int kvp_decode_step(kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs, int32_t ntok,
                    const kvp_step_io *io, const kvp_attn_desc *desc, void *workspace,
                    size_t ws_bytes, size_t *ws_needed, void *stream) {
    if (!workspace || ((uintptr_t)workspace & 255)) return KVP_ERR_INVALID;
    int rc = check_io(io, ntok);
    if (rc) return rc;
    rc = check_step(pool, seq_ids, num_seqs, ntok, desc, t_ntoks);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const StepBytes b = step_bytes(*desc, num_seqs, ntok);
    const bool mapped = (io->flags & KVP_STEP_HOST_MAPPED) != 0;
    if (mapped || !(io->h_k_new || io->h_v_new || io->h_q)) {
        // inputs on the device or mapped: plan first, then (when the step
        // qualifies) inputs, append and plan in one kernel
        rc = plan_step(t_step, pool, seq_ids, num_seqs, ntok, *desc, t_ntoks.data());
        if (rc) return rc;
        if (ws_needed) *ws_needed = t_step.pk.w.total;
        bool launched = false;
        rc = launch_fused(t_step, io, workspace, ws_bytes, st, &launched);
        if (rc || launched) return rc;
        rc = step_inputs(io, b, ntok, st);
        if (rc) return rc;
        return launch_step(t_step, io, workspace, ws_bytes, st);
    }
    // copy-engine inputs first, so that they run while the host plans
    rc = step_inputs(io, b, ntok, st);
    if (rc) return rc;
    rc = plan_step(t_step, pool, seq_ids, num_seqs, ntok, *desc, t_ntoks.data());
    if (rc) return rc;
    if (ws_needed) *ws_needed = t_step.pk.w.total;
    return launch_step(t_step, io, workspace, ws_bytes, st);
}

kvp_step_plan *kvp_step_plan_create(void) { return new (std::nothrow) kvp_step_plan(); }

void kvp_step_plan_destroy(kvp_step_plan *plan) { delete plan; }

int kvp_decode_step_plan(kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs, int32_t ntok,
                         const kvp_attn_desc *desc, kvp_step_plan *plan, size_t *ws_needed) {
    if (!plan || plan->ready) return KVP_ERR_INVALID;
    int rc = check_step(pool, seq_ids, num_seqs, ntok, desc, t_ntoks);
    if (rc) return rc;
    rc = plan_step(*plan, pool, seq_ids, num_seqs, ntok, *desc, t_ntoks.data());
    if (rc) return rc;
    if (ws_needed) *ws_needed = plan->pk.w.total;
    return KVP_OK;
}

int kvp_decode_step_run(kvp_step_plan *plan, const kvp_step_io *io, void *workspace, size_t ws_bytes,
                        void *stream) {
    if (!plan || !plan->ready || !workspace || ((uintptr_t)workspace & 255)) return KVP_ERR_INVALID;
    int rc = check_io(io, plan->ntok);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const StepBytes b = step_bytes(plan->desc, plan->num_seqs, plan->ntok);
    bool launched = false;
    rc = launch_fused(*plan, io, workspace, ws_bytes, st, &launched);
    if (rc || launched) return rc;
    rc = step_inputs(io, b, plan->ntok, st);
    if (rc) return rc;
    return launch_step(*plan, io, workspace, ws_bytes, st);
}

size_t kvp_verify_workspace_size(const kvp_attn_desc *desc, const int32_t *block_tables,
                                 const int32_t *ctx_lens, int32_t batch, int32_t n_draft,
                                 int32_t max_blocks) {
    if (!desc_ok(desc) || batch <= 0 || !ctx_lens || !block_tables || max_blocks <= 0) return 0;
    HostPlan &hp = t_plan;
    hp.clear();
    if (build_verify(*desc, block_tables, ctx_lens, batch, n_draft, max_blocks, device_sm_count(), hp))
        return 0;
    return layout(hp, *desc).total;
}

int tree_verify_attention(const void *q, const int32_t *tree_parent, int32_t n_draft,
                          const void *k_pool, const void *v_pool, const int32_t *block_tables,
                          const int32_t *ctx_lens, int32_t batch, int32_t max_blocks,
                          const kvp_attn_desc *desc, void *out, float *lse, void *workspace,
                          size_t ws_bytes, void *stream) {
    if (!desc_ok(desc) || desc->kv_format != KVP_KV_BF16 || batch <= 0 || max_blocks <= 0 || !ctx_lens ||
        !block_tables || !tree_parent)
        return KVP_ERR_INVALID;
    HostPlan &hp = t_plan;
    hp.clear();
    int rc = build_verify(*desc, block_tables, ctx_lens, batch, n_draft, max_blocks, device_sm_count(), hp);
    if (rc) return rc;
    return run(hp, *desc, q, k_pool, v_pool, batch * n_draft, tree_parent, n_draft, out, lse,
               workspace, ws_bytes, (cudaStream_t)stream);
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

int kvp_decode_plan_stats(const kvp_attn_desc *desc, const int32_t *block_tables,
                          const int32_t *seq_lens, int32_t num_seqs, int32_t max_blocks,
                          int32_t sm_count, int32_t *n_items, int32_t *n_row_tiles,
                          int32_t *n_kv_tiles, int32_t *n_partial_rows, int64_t *unique_kv_bytes) {
    if (!desc_ok(desc) || num_seqs <= 0 || max_blocks <= 0 || !block_tables || !seq_lens ||
        sm_count <= 0)
        return KVP_ERR_INVALID;
    HostPlan &hp = t_plan;
    hp.clear();
    int rc = build_decode(*desc, block_tables, seq_lens, num_seqs, max_blocks, sm_count, hp);
    if (rc) return rc;
    if (!plan_consistent(hp, desc->num_q_heads / desc->num_kv_heads)) return KVP_ERR_STATE;
    if (n_items) *n_items = (int32_t)(hp.items.size() + hp.tc_items.size());
    if (n_row_tiles) *n_row_tiles = hp.n_row_tiles;
    if (n_kv_tiles) *n_kv_tiles = (int32_t)hp.tiles.size();
    if (n_partial_rows) *n_partial_rows = hp.n_partial_rows;
    if (unique_kv_bytes) *unique_kv_bytes = hp.unique_kv_bytes;
    return KVP_OK;
}

int kvp_set_kernel_events(void *before, void *after) {
    if ((before == nullptr) != (after == nullptr)) return KVP_ERR_INVALID;
    t_ev_before = (cudaEvent_t)before;
    t_ev_after = (cudaEvent_t)after;
    return KVP_OK;
}

int kvp_kernel_launches(int64_t *n_out) {
    if (!n_out) return KVP_ERR_INVALID;
    *n_out = launch_count();
    return KVP_OK;
}

}  // extern "C"
