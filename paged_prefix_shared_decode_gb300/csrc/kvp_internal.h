// Internal declarations shared by the library's host code and its kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

struct kvp_pool;

namespace kvp {

constexpr int kTileTokens = 64;    // tokens per KV tile (one pipeline stage)
constexpr int kTileBlocks = 5;     // blocks a 64-token tile can touch when bs >= 16
constexpr int kMaxItemTiles = 128; // KV tiles per work item (descriptors staged in smem)
constexpr int kTileTree = 1;       // tile flag: draft tokens under a tree mask
constexpr int kMmaMaxRows = 64;    // rows of an mma.sync unit (4 warps x 16)
constexpr int kTcRows = 256;       // rows of a tcgen05 unit: one 128-row tile or a pair
constexpr int kMaxDraft = 64;      // draft tokens per sequence (64-bit ancestor masks)

// One KV tile of a work item: tokens [tok0, tok0 + ntok) of one sequence,
// whose physical blocks (in order) are blk[0..]: token t of the tile lives in
// blk[(tok0 + t) / bs - tok0 / bs], slot (tok0 + t) % bs.  The tile is seen
// by the item's members with local index in [m_lo, m_hi).  TREE: token t is
// visible to draft node i only if bit t of i's ancestor-or-self mask is set.
struct KvTile {
    int32_t tok0;
    int32_t ntok_flags;   // ntok | flags << 16
    int32_t members;      // m_lo | m_hi << 16
    int32_t blk[kTileBlocks];
};
static_assert(sizeof(KvTile) == 32, "KvTile is 32 bytes");

// A work item: KV tiles [tile_begin, tile_end) against the query rows of
// n_members members (decode sequences or draft nodes) x the GQA group.
// out_base < 0: the item covers every key of its rows and writes out / lse;
// otherwise row r goes to partial row out_base + r.
struct WorkItem {
    int32_t tile_begin, tile_end;
    int32_t member_off, n_members;
    int32_t out_base;
    int32_t pad[3];
};

// Per query token: merge entries[off .. off + cnt) are partial-row bases
// (add the head's index within its group); cnt == 0 means written directly.
struct MergeDesc {
    int32_t off, cnt;
};

// Workspace: [header | items | tiles | members | merge | entries | partials].
struct WsHeader {
    int32_t err;         // KVP_DEVERR_* bits
    int32_t counter;     // next work unit of the mma.sync kernel
    int32_t tc_counter;  // next work unit of the tcgen05 kernel
    int32_t n_items, n_tc_items, n_units, n_tiles, n_members, n_entries, n_partial_rows;
    int32_t pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct AttnLaunch {
    const void *q;
    const void *k_pool;           // bf16 K, or the 4-bit codes (kv4)
    const void *v_pool;
    const void *k_exp;            // kv4: row exponents
    const void *v_exp;
    int32_t kv4;
    int32_t NB, bs_log2, Hq, Hkv, G, nq, L, D;
    float scale_log2;
    const int32_t *tree_parent;   // null for decode
    int32_t n_draft;
    uint64_t *tree_mask;          // per query token: ancestor-or-self bits (verify only)
    void *out;
    float *lse;
    // workspace views
    int32_t *err;
    int32_t *counter;
    int32_t *tc_counter;
    const WorkItem *items;      // mma.sync items (at most 32 query rows)
    const WorkItem *tc_items;   // tcgen05 items (up to 128 query rows)
    const KvTile *tiles;
    const int32_t *members;
    const MergeDesc *merge;
    const int32_t *entries;
    float *part_o;
    float *part_lse;
    int32_t n_units, n_tc_units, n_merge_q, P;
    int32_t wait_first;   // 1: the kernel before wrote the plan too; wait before reading anything
};

// before/after: optional events recorded around the work-item kernel.
cudaError_t launch_attention(const AttnLaunch &a, cudaStream_t stream, cudaEvent_t before,
                             cudaEvent_t after);
// tcgen05 kernel over a.tc_items (no-op when there are none); at most
// `ctas_per_sm` CTAs per SM (0: as many as fit).
cudaError_t launch_attention_tc(const AttnLaunch &a, cudaStream_t stream, int ctas_per_sm);
// Whether the tcgen05 kernel can address this pool (32-bit TMA row index).
bool tc_path_supported(int L, int NB, int Hkv, int bs);
// TMA view of a K or V pool as rows = L*NB*Hkv*bs token rows of D bf16
// (box: 64 columns x box_rows rows, 128-byte swizzle), from a small
// per-thread cache.  False when the driver's encoder is unavailable or
// rejects the view.
bool make_pool_map(CUtensorMap *m, const void *pool, int D, long long rows, int box_rows);
// TMA view of the queries [ntok][Hq][D] (box: 64 columns x G heads x
// max(1, 8 / G) tokens, 128-byte swizzle), cached the same way.  False when
// q is not 16-byte aligned, the view is too large or the encoder rejects it.
bool make_q_map(CUtensorMap *m, const void *q, int D, int Hq, long long ntok, int G);
// CTAs of the mma.sync work-item kernel that fit on one SM for head dim D.
int attention_ctas_per_sm(int D);
// Rows above which items of head dim D run on the tcgen05 kernel
// (INT32_MAX: never).
int tc_row_threshold(int head_dim);

// Pool access for other holders of blocks (the prefix cache).  b must be
// in use (refcount > 0) for hold and drop; drop returns true when the block
// went back to the front of the free list.
int32_t pool_block_size(const kvp_pool *p);
int32_t pool_num_blocks(const kvp_pool *p);
int32_t pool_free_count(const kvp_pool *p);
bool pool_block_in_use(const kvp_pool *p, int32_t b);
void pool_hold_block(kvp_pool *p, int32_t b);
bool pool_drop_block(kvp_pool *p, int32_t b);

// The checks of seq_append_batch with no change to the pool: KVP_OK when
// every append fits; *total_out (may be null) = the tokens appended.
int append_batch_check(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks,
                       int64_t *total_out = nullptr);

// seq_append_batch's checks and bookkeeping, the slots and copy-on-write
// triples staged in the pool for its device write.
int append_batch_commit(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks, const void *k,
                        const void *v, int32_t *total_out);

// seq_append_batch in two halves: the checks and the bookkeeping, whose
// token slots and copy-on-write triples go to the caller's lists (the
// sequences grow at once), then the device write of those lists, with the
// new tokens' K/V [L][slots.size()][Hkv][d].  No call that frees or
// reallocates the lists' blocks may come in between.
int append_batch_commit_lists(kvp_pool *p, int32_t nseq, const int32_t *seqs, const int32_t *ntoks,
                              std::vector<int32_t> &slots, std::vector<int32_t> &cow, int32_t *total_out);
int append_issue_lists(kvp_pool *p, const std::vector<int32_t> &slots, const std::vector<int32_t> &cow,
                       const void *k, const void *v, void *stream);

// A pool's shape and device storage (codes and exponents for 4-bit pages).
struct PoolView {
    int32_t L, NB, bs, Hkv, d;
    const void *k, *v, *k_exp, *v_exp;
    bool kv4;
};
PoolView pool_view(const kvp_pool *p);

// Block tables of seqs[0..n) as rows of `width` (the longest table; padded
// with -1) and their lengths, into caller vectors.  KVP_ERR_INVALID for a
// sequence that is not live.
int pool_tables(const kvp_pool *p, const int32_t *seqs, int32_t n, int32_t *width, int32_t **tables,
                int32_t **lens);

// Devices the library keeps per-device state for (SM counts, kernel
// attributes, side streams); ids at or above this fail their launches.
constexpr int kMaxDevices = 64;
// Current device id, or -1 when there is none or it is >= kMaxDevices.
int current_device();
// SM count of the current device, looked up once per device (152 if the
// query fails).
int device_sm_count();

// Counts every kernel launch the library makes.
void count_launch();
long long launch_count();

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

// A decode step's inputs in one launch (the append of w, q_bytes of q from
// q_src to q_dst when q_src is given, and plan_bytes of a host plan image,
// carried in the kernel parameters, to plan_dst), letting the kernel launched
// behind it with programmatic serialisation start at once.  For appends of at
// most 64 tokens and 16 copy-on-write blocks and plans of at most
// kStepPlanMax bytes (step_write_fits); cudaErrorInvalidValue otherwise.
constexpr size_t kStepPlanMax = 24576;
bool step_write_fits(const KvWrite &w, size_t plan_bytes);
cudaError_t launch_step_write(const KvWrite &w, const void *q_src, void *q_dst, size_t q_bytes, const void *plan,
                              void *plan_dst, size_t plan_bytes, cudaStream_t stream);

// Speculative accept on the device: copy-on-write block copies (all slots),
// then kept draft tokens moved from src to dst slots in order.
struct KvMove {
    void *k_pool;
    void *v_pool;
    int32_t L, NB, Hkv, bs, d;
    int32_t ncow;
    const int32_t *cow;    // host: (source block, copy block) pairs
    int32_t nmove;
    const int32_t *src;    // host: block*bs + slot per kept token
    const int32_t *dst;
};

cudaError_t launch_kv_move(const KvMove &m, cudaStream_t stream);

// One launch copying n <= 4 buffers (16-byte aligned, sizes multiples of 4)
// through the SMs.
cudaError_t launch_copy_segments(const void *const *src, void *const *dst, const int64_t *bytes, int n,
                                 cudaStream_t stream);

// The same two for a pool of 4-bit pages: codes [L][NB][Hkv][bs][d/2] bytes
// (two signed 4-bit codes per byte, element 2i in the low nibble) and one
// int8 power-of-two exponent per (token, kv head) row [L][NB][Hkv][bs].
// Appended rows (bf16) are quantised on the device.
struct Kv4Write {
    void *k_codes, *v_codes, *k_exp, *v_exp;
    const void *k, *v;     // appended bf16 [L][ntok][Hkv][d]
    int32_t L, NB, Hkv, bs, d;
    int32_t ntok;
    const int32_t *slots;  // host: block*bs + slot per token
    int32_t ncow;
    const int32_t *cow;    // host: (src, dst, used) triples
};
cudaError_t launch_kv4_write(const Kv4Write &w, cudaStream_t stream);

struct Kv4Move {
    void *k_codes, *v_codes, *k_exp, *v_exp;
    int32_t L, NB, Hkv, bs, d;
    int32_t ncow;
    const int32_t *cow;    // host: (source block, copy block) pairs
    int32_t nmove;
    const int32_t *src;    // host: block*bs + slot per kept token
    const int32_t *dst;
};
cudaError_t launch_kv4_move(const Kv4Move &m, cudaStream_t stream);

}  // namespace kvp
