// Internal declarations shared by the library's host code and its kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace kvp {

// One 64-token KV tile of a work item: tokens [tok0, tok0 + ntok) of the
// sequence in table row `row`, seen by the item's members with local index in
// [m_lo, m_hi).  TREE: token j of the tile is visible to a draft-node row only
// if bit j of that node's ancestor-or-self mask is set.
struct KvTile {
    int32_t row;
    int32_t tok0;
    int32_t ntok_flags;   // ntok | flags << 16
    int32_t members;      // m_lo | m_hi << 16
};
constexpr int kTileTokens = 64;
constexpr int kTileTree = 1;

// A CTA's work: KV tiles [tile_begin, tile_end) for up to 64 query rows
// (n_members sequences or draft nodes times the GQA group).  out_base < 0:
// the item sees every key of its rows and writes out/lse directly; otherwise
// it writes partial rows out_base + m * G + g for the merge kernel.
struct WorkItem {
    int32_t tile_begin, tile_end;
    int32_t member_off, n_members;
    int32_t out_base;
    int32_t pad[3];
};

// Per query token: partial rows base + c * stride + m_pos * G + g for chunks
// c < n_chunks; n_chunks == 0 means the query was written directly.
struct MergeDesc {
    int32_t base, stride, n_chunks, m_pos;
};

// Layout of the workspace: [header | items | tiles | members | merge | partials].
struct WsHeader {
    int32_t err;
    int32_t n_items, n_tiles, n_members, n_merge, n_partial_rows;
    int32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct Plan {
    int32_t n_items = 0, n_row_tiles = 0, n_partial_rows = 0, n_merge_q = 0;
    int32_t ts = 1;               // warps that split one tile's tokens (1, 2, 4)
    int64_t unique_kv_bytes = 0;  // distinct (block, valid tokens) bytes, all layers
    // host images of the uploaded arrays
    WorkItem *items = nullptr;
    KvTile *tiles = nullptr;
    int32_t *members = nullptr;
    MergeDesc *merge = nullptr;
    int32_t n_tiles = 0, n_members = 0, n_merge = 0;
};

struct AttnLaunch {
    const void *q;
    const void *k_pool;
    const void *v_pool;
    const int32_t *tables;
    int32_t MB, NB, bs, Hq, Hkv, G, nq, L, D;
    float scale_log2;
    const int32_t *tree_parent;   // null for decode
    int32_t n_draft;
    void *out;
    float *lse;
    // workspace views
    int32_t *err;
    const WorkItem *items;
    const KvTile *tiles;
    const int32_t *members;
    const MergeDesc *merge;
    float *part_o;
    float *part_lse;
    int32_t n_items, n_merge_q, P, ts;
};

cudaError_t launch_attention(const AttnLaunch &a, cudaStream_t stream);

// K/V write: copy-on-write copies (src, dst, used slots) then token scatter.
struct KvWrite {
    void *k_pool;
    void *v_pool;
    const void *k;
    const void *v;
    int32_t L, NB, Hkv, bs, d;
    int32_t ntok;          // tokens in k / v
    const int32_t *slots;  // host: block*bs + slot per token
    int32_t ncow;
    const int32_t *cow;    // host: (src, dst, used) triples
};

cudaError_t launch_kv_write(const KvWrite &w, cudaStream_t stream);

}  // namespace kvp
