/*
 * kvp.h -- C ABI of the paged, prefix-shared KV pool, its prefix cache and its
 * attention kernels (GB300 / sm_103a).
 *
 * Conventions for every entry point:
 *   - returns KVP_OK (0) or a negative KVP_ERR_* code; out-parameters are
 *     written only on success and state is left unchanged on failure, except
 *     where a function says otherwise (kvp_radix_evict reports how far it
 *     got; seq_accept_draft's bookkeeping stands when its launch fails);
 *   - "device" pointers are CUDA global memory on the current device, owned by
 *     the caller; "host" pointers are ordinary host memory owned by the caller;
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream);
 *     device work is enqueued on it and the call returns without synchronising,
 *     except where a function says it synchronises;
 *   - bf16 tensors are IEEE bfloat16 bit patterns, 16-byte aligned;
 *   - a pool handle is not thread-safe: serialise calls on one pool.
 *
 * Layouts (row-major, innermost last):
 *   K pool, V pool   [L][NB][Hkv][bs][d]  bf16   (one (block, kv head) tile is
 *                                                  a contiguous bs*d run)
 *   block tables     [S][MB] int32 (host), entries past a sequence's blocks ignored
 *   decode q, out    [L][S][Hq][d] bf16;   lse [L][S][Hq] fp32, natural log
 *   verify q, out    [L][B*n][Hq][d] bf16; lse [L][B*n][Hq] fp32
 *   appended k, v    [L][ntok][Hkv][d] bf16
 * Query head h reads kv head h / (Hq / Hkv).
 */
#ifndef KVP_H
#define KVP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    KVP_OK = 0,
    KVP_ERR_INVALID = -1, /* bad argument, unknown sequence, capacity exceeded */
    KVP_ERR_OOM = -2,     /* no free block or sequence slot                   */
    KVP_ERR_STATE = -3,   /* operation not possible in the object's state     */
    KVP_ERR_CUDA = -4,    /* a CUDA runtime call failed                        */
    KVP_ERR_DEVICE = -5,  /* a kernel's own bounds check tripped (see below)  */
    KVP_ERR_WORKSPACE = -6 /* kvp_decode_step: workspace too small (see there) */
};

/* Device error word bits (kvp_device_error). */
enum {
    KVP_DEVERR_BLOCK_ID = 1,     /* a planned block id outside [0, NB): those tokens read as 0 */
    KVP_DEVERR_TREE_PARENT = 2,  /* a parent pointer not in [-1, i): treated as a root       */
    KVP_DEVERR_WAIT_TIMEOUT = 4  /* a tcgen05 pipeline wait ran out: that CTA stopped early  */
};

/* ------------------------------------------------------------------ pool */

/*
 * A block-paged KV pool: NB blocks of bs token slots per layer, shared by many
 * sequences through per-sequence block tables with per-block refcounts.
 * Paper: "Dendrite: O(1) fork latency agent-native inference engine", section
 * details (16-token paged blocks; tree-shaped KV cache with reference
 * counting); "Trellis: RadixAttention", section "RadixAttention in Trellis"
 * (a session holds an ordered list of block ids into one shared pool).
 */
typedef struct kvp_pool kvp_pool;

typedef struct {
    int32_t num_layers;         /* L   */
    int32_t num_blocks;         /* NB  */
    int32_t block_size;         /* bs, tokens per block (16 and 32 are the pages' sizes) */
    int32_t num_kv_heads;       /* Hkv */
    int32_t head_dim;           /* d, a multiple of 8 */
    int32_t max_seqs;           /* sequence ids are 0 .. max_seqs-1, lowest free id first */
    int32_t max_blocks_per_seq; /* MB, block table capacity */
    uint64_t alloc_seed;        /* free-list order: splitmix64-driven Fisher-Yates
                                   shuffle of [0, NB); 0 = identity order */
} kvp_pool_desc;

/* Create a pool over caller-owned device storage k_storage / v_storage, each
 * [L][NB][Hkv][bs][d] bf16.  Both may be NULL for a bookkeeping-only pool, in
 * which case seq_append / seq_append_batch return KVP_ERR_STATE (use
 * seq_reserve).  The pool never allocates or frees KV storage. */
int kv_pool_create(const kvp_pool_desc *desc, void *k_storage, void *v_storage, kvp_pool **out);

/*
 * A pool of 4-bit pages ("Dendrite", section on FlashInfer kernels and
 * TurboQuant integration: 4-bit KV compression that cuts KV memory 3.88x and
 * is computed on directly; the quantiser is not given there).  Each (token,
 * kv head) row of d values is kept as d signed 4-bit codes in [-7, 7] and one
 * power-of-two scale 2^e, e an int8 in [-127, 127]:
 *   e = the smallest integer with max|x| <= 7 * 2^e (-127 for a zero row),
 *   code = x / 2^e rounded half to even, value = code * 2^e,
 * 4 + 8/d bits per value (16 / 4.125 = 3.88x less than bf16 at d = 64).
 * Storage, all device memory owned by the caller, 16-byte aligned:
 *   k_codes, v_codes  [L][NB][Hkv][bs][d/2] bytes: element 2i of a row in
 *                     the low nibble of byte i, 2i+1 in the high nibble
 *                     (two's complement);
 *   k_exps, v_exps    [L][NB][Hkv][bs] int8.
 * Needs d = 64 or 128 and bs a multiple of 16, else KVP_ERR_INVALID.
 * seq_append / seq_append_batch take bf16 K/V as for any pool and quantise
 * them on the device (copy-on-write copies codes and exponents);
 * seq_accept_draft moves codes and exponents.  Attention over such a pool:
 * paged_decode_attention_kv4 with desc->kv_format = KVP_KV_4BIT.
 */
int kv_pool_create_kv4(const kvp_pool_desc *desc, void *k_codes, void *k_exps, void *v_codes,
                       void *v_exps, kvp_pool **out);
int kv_pool_destroy(kvp_pool *pool);

/* New empty sequence ("allocate_sequence" in Dendrite's API example). */
int seq_alloc(kvp_pool *pool, int32_t *seq_out);

/* Copy-on-write fork ("fork_sequence(parent)?" in Dendrite's API example):
 * the child gets a copy of the parent's block table and every block's
 * refcount goes up by one.  No KV bytes move and no device work is issued;
 * cost is O(number of blocks) host integer work, independent of KV size. */
int seq_fork(kvp_pool *pool, int32_t parent, int32_t *child_out);

/* Release a sequence: every block's refcount drops by one and blocks that
 * reach zero go back to the free list, last table entry first ("SGLang
 * RadixAttention", reference-counting section: referenced blocks are never
 * reclaimed). */
int seq_free(kvp_pool *pool, int32_t seq);

/* Speculative accept after tree verify ("CAST", section on speculative
 * decoding: the target model accepts one path of the draft tree).  The
 * sequence holds ctx_len context tokens followed by n_draft draft tokens,
 * draft node i at position ctx_len + i with parent[i] in [-1, i) (-1: a
 * root), n_draft <= 64.  The path from a root down to node `accepted` (-1:
 * none) is kept: its tokens move, in order, to positions ctx_len,
 * ctx_len + 1, ... (K and V, every layer and kv head); the length becomes
 * ctx_len + path length and the blocks past the new end are released, last
 * first.  A block that receives a moved token and is shared with another
 * sequence is copied first (copy-on-write).  Device work is one
 * kv_move_kernel launch on `stream` (none when nothing moves; a pool without
 * K/V storage updates its bookkeeping only).  path_out (n_draft entries,
 * may be NULL) receives the kept node ids, root first, *n_path_out their
 * count.  KVP_ERR_INVALID (bad sequence, lengths or parents) or
 * KVP_ERR_OOM (no block to copy into) change nothing; KVP_ERR_CUDA: the
 * bookkeeping is done but the launch failed. */
int seq_accept_draft(kvp_pool *pool, int32_t seq, int32_t ctx_len, const int32_t *parent, int32_t n_draft,
                     int32_t accepted, int32_t *path_out, int32_t *n_path_out, void *stream);

/* A new sequence that starts from blocks someone already holds (a prefix
 * found in the prefix cache below): its table is blocks[0..n_blocks), one
 * more reference on each, and its length n_blocks * block_size ("Trellis",
 * section "RadixAttention in Trellis": a session acquires the existing
 * prefix blocks, raising their refcount, instead of allocating and
 * recomputing them).  Every block must be in use (refcount > 0), else
 * KVP_ERR_INVALID and nothing changes; KVP_ERR_OOM when no sequence slot is
 * free. */
int seq_alloc_prefix(kvp_pool *pool, const int32_t *blocks, int32_t n_blocks, int32_t *seq_out);

/* Append ntok tokens' K and V (device, [L][ntok][Hkv][d] bf16 each) to a
 * sequence.  Copy-on-write ("Dendrite", section details: data is shared until
 * modified and copied only on write): if the last block is partially filled
 * and other live sequences also hold it, the sequence first gets a fresh
 * block with the used slots copied on the device; a full last block just
 * gets a new block; a block held only by this sequence is written in place.
 * Enqueues at most one kernel.  k and v must stay valid until it has run. */
int seq_append(kvp_pool *pool, int32_t seq, const void *k, const void *v, int32_t ntok,
               void *stream);

/* Append to several distinct sequences in one launch: ntoks[i] tokens to
 * seqs[i] (host arrays), processed in order with the semantics of seq_append;
 * k, v: device [L][sum ntoks][Hkv][d], sequence-major.  All or nothing: if the
 * pool cannot hold every append, nothing changes and KVP_ERR_OOM returns. */
int seq_append_batch(kvp_pool *pool, int32_t nseq, const int32_t *seqs, const int32_t *ntoks,
                     const void *k, const void *v, void *stream);

/* Bookkeeping half of seq_append with no device work: reserves slots for ntok
 * tokens and reports where they go.  slots_out (host, ntok entries, may be
 * NULL) receives block*bs + slot per token; cow_out (host, 3 entries, may be
 * NULL) receives {source block, copy block, used slots} or {-1, -1, 0} when no
 * copy-on-write happened.  The caller is then responsible for the data. */
int seq_reserve(kvp_pool *pool, int32_t seq, int32_t ntok, int32_t *slots_out, int32_t *cow_out);

/* Host queries. */
int seq_block_table(const kvp_pool *pool, int32_t seq, int32_t *host_out, int32_t cap,
                    int32_t *nblocks_out);
int seq_len(const kvp_pool *pool, int32_t seq, int32_t *len_out);
int block_refcount(const kvp_pool *pool, int32_t block, int32_t *rc_out);
int kvp_free_block_count(const kvp_pool *pool, int32_t *n_out);
int kvp_cow_count(const kvp_pool *pool, int64_t *n_out);

/* Block tables and lengths of n sequences into host arrays h_tables
 * [n][width] (padded with -1) and h_lens [n]. */
int kvp_gather_tables(const kvp_pool *pool, const int32_t *seqs, int32_t n, int32_t width,
                      int32_t *h_tables, int32_t *h_lens);

/* Same, written to device arrays d_tables [n][width] and d_lens [n] (either
 * may be NULL) with an asynchronous host-to-device copy on `stream`. */
int kvp_export_tables(kvp_pool *pool, const int32_t *seqs, int32_t n, int32_t width,
                      int32_t *d_tables, int32_t *d_lens, void *stream);

/* ---------------------------------------------------------- prefix cache */

/*
 * A radix-tree prefix cache over a pool's blocks ("SGLang RadixAttention",
 * sections on the node and edge structure, on the three operations match /
 * split / insert, and on reference counting with LRU eviction; "Trellis",
 * section "RadixAttention in Trellis").  The root is the empty sequence; the
 * edge into a node holds a run of token ids and the ids of the blocks that
 * store them.  Everything is in whole blocks of block_size tokens: a run is
 * a whole number of blocks, a match is rounded down to whole agreeing
 * blocks, and edges split on block boundaries.  The cache holds one pool
 * reference on every block in the tree, so a block goes back to the pool
 * only when neither the cache nor a sequence holds it.  "Last used" is a
 * logical clock advanced by every match and insert and stamped on every node
 * of the path it used.  Not thread-safe; destroy the cache before its pool.
 */
typedef struct kvp_radix kvp_radix;

/* KVP_ERR_INVALID on a null pool; KVP_ERR_OOM if memory runs out. */
int kvp_radix_create(kvp_pool *pool, kvp_radix **out);

/* Drops the cache's references (each node's blocks last to first, children
 * before parents) and frees the cache. */
int kvp_radix_destroy(kvp_radix *cache);

/* Longest cached prefix of tokens[0..n_tokens) in whole blocks: its block
 * ids go to blocks_out (cap >= n_tokens / block_size) and their count to
 * *n_blocks_out.  Every node whose blocks were returned (including one whose
 * edge agreed only in part) is locked, i.e. not evictable, until
 * kvp_radix_unlock(cache, *lock_out); *lock_out = -1 when nothing matched. */
int kvp_radix_match(kvp_radix *cache, const int32_t *tokens, int32_t n_tokens, int32_t *blocks_out,
                    int32_t cap, int32_t *n_blocks_out, int32_t *lock_out);

/* Releases a lock from kvp_radix_match (-1: nothing to release).
 * KVP_ERR_STATE, with nothing changed, if that path is not locked. */
int kvp_radix_unlock(kvp_radix *cache, int32_t lock);

/* Caches a sequence's whole blocks: tokens[0..n_tokens) are stored in
 * blocks[0..n_blocks) (block j holds tokens [j*bs, (j+1)*bs)); only the
 * first min(n_tokens / bs, n_blocks) blocks count.  The tree is walked as in
 * match, splitting an edge that agrees for only part of its run (the upper
 * part inherits the lower part's locks); what is not cached yet becomes a
 * new leaf on which the cache takes one reference per block.  Blocks already
 * cached for an equal prefix are kept.  Every new block must be in use, else
 * KVP_ERR_INVALID and nothing changes. */
int kvp_radix_insert(kvp_radix *cache, const int32_t *tokens, int32_t n_tokens, const int32_t *blocks,
                     int32_t n_blocks);

/* Until the pool has need_free free blocks: the unlocked leaf used longest
 * ago gives its blocks back (last to first) and leaves the tree; a parent
 * left childless and unlocked is then a leaf like any other.  *freed_out =
 * blocks that went back to the pool.  KVP_OK when met, KVP_ERR_OOM when
 * nothing more is evictable. */
int kvp_radix_evict(kvp_radix *cache, int32_t need_free, int32_t *freed_out);

/* Canonical dump for tests and tools: depth first from the root, children
 * in increasing order of their first block's tokens; per node the int32
 * words depth, locks, stamp, n_tokens, tokens..., n_blocks, blocks...
 * *n_out = words needed; KVP_ERR_INVALID (nothing written) when cap is too
 * small. */
int kvp_radix_dump(const kvp_radix *cache, int32_t *out, int64_t cap, int64_t *n_out);

/* ------------------------------------------------------------- attention */

typedef struct {
    int32_t num_layers;    /* L: q/out/lse and both pools carry a leading layer axis */
    int32_t num_q_heads;   /* Hq */
    int32_t num_kv_heads;  /* Hkv; Hq % Hkv == 0 and Hq / Hkv <= 64 */
    int32_t head_dim;      /* d: 64 or 128 */
    int32_t block_size;    /* bs: a power of two >= 16 */
    int32_t num_blocks;    /* NB */
    float scale;           /* softmax scale; <= 0 selects 1/sqrt(d) */
    int32_t use_sharing;   /* 1: blocks that several sequences share are read once per
                              tile of up to 64 query rows (cascade); 0: every sequence
                              reads its own blocks (the unshared baseline) */
    int32_t kv_format;     /* KVP_KV_BF16 (0) or KVP_KV_4BIT (1): the pool's page format */
} kvp_attn_desc;

enum { KVP_KV_BF16 = 0, KVP_KV_4BIT = 1 };

/* Device workspace bytes that paged_decode_attention (or, with
 * desc->kv_format = KVP_KV_4BIT, paged_decode_attention_kv4) needs for this
 * batch (same host tables and lengths as the call).  Returns 0 on invalid
 * input. */
size_t kvp_decode_workspace_size(const kvp_attn_desc *desc, const int32_t *block_tables,
                                 const int32_t *seq_lens, int32_t num_seqs, int32_t max_blocks);

/*
 * Decode attention over the paged pool: for each layer, sequence s and query
 * head h, out = softmax(q k^T * scale) v over the first seq_lens[s] tokens of
 * sequence s, and lse = the natural-log log-sum-exp of the scaled scores.
 * (Decode is one new token attending to the cached keys and values: "SGLang
 * RadixAttention", section on the KV-cache lifecycle; the pool is the paged
 * cache of "Dendrite", section details.)  The call attends to exactly
 * seq_len tokens; append the new token's K/V first to include it.
 *
 * block_tables [num_seqs][max_blocks] and seq_lens [num_seqs] are HOST arrays
 * (kvp_gather_tables gives them for pool sequences).  The call plans on the
 * host: sequences whose tables hold the same physical blocks at the same
 * positions are grouped so that a shared block is read from HBM once per
 * group of up to 64 query rows instead of once per sequence; long key ranges
 * are split across CTAs and merged by log-sum-exp.  The plan, which carries
 * the physical block ids, is copied into the workspace with an asynchronous
 * copy from host memory on `stream`; no device block table is read, and the
 * host arrays may be reused as soon as the call returns.
 *
 * q: device [L][num_seqs][Hq][d] bf16; k_pool / v_pool: the pool's device
 * storage; out: device [L][num_seqs][Hq][d] bf16; lse: device
 * [L][num_seqs][Hq] fp32 or NULL.  workspace: device, 256-byte aligned,
 * ws_bytes >= kvp_decode_workspace_size(); one call at a time per workspace.
 * Errors: KVP_ERR_INVALID for an empty sequence, a table entry outside
 * [0, NB), a too-small or misaligned workspace, misaligned tensors or
 * unsupported shapes; KVP_ERR_CUDA if a launch fails.
 */
int paged_decode_attention(const void *q, const void *k_pool, const void *v_pool,
                           const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                           int32_t max_blocks, const kvp_attn_desc *desc, void *out, float *lse,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * Decode attention over a pool of 4-bit pages (kv_pool_create_kv4): the same
 * call and results as paged_decode_attention, with the keys and values being
 * the pages' values code * 2^e.  k_codes / k_exps / v_codes / v_exps are the
 * pool's storage; desc->kv_format must be KVP_KV_4BIT (paged_decode_attention
 * rejects such a descriptor).  HBM traffic per token is (d/2 + 1) bytes per
 * kv head for K and for V instead of 2d.
 */
int paged_decode_attention_kv4(const void *q, const void *k_codes, const void *k_exps,
                               const void *v_codes, const void *v_exps, const int32_t *block_tables,
                               const int32_t *seq_lens, int32_t num_seqs, int32_t max_blocks,
                               const kvp_attn_desc *desc, void *out, float *lse, void *workspace,
                               size_t ws_bytes, void *stream);

size_t kvp_verify_workspace_size(const kvp_attn_desc *desc, const int32_t *block_tables,
                                 const int32_t *ctx_lens, int32_t batch, int32_t n_draft,
                                 int32_t max_blocks);

/*
 * Speculative tree-verify attention ("Inference-Cost-Aware Dynamic Tree
 * Construction for Efficient Inference in Large Language Models" (CAST),
 * technical summary sections 1-2: the target model checks a dynamic draft
 * tree of candidate tokens, EAGLE-2/3 style, in one forward pass).
 * Sequence b has ctx_lens[b] context tokens followed, in its pages, by
 * n_draft <= 64 draft tokens.  Draft node i (query row b*n_draft + i) attends
 * to every context token and to the draft tokens of its ancestors and itself,
 * anc*(i) = {i, parent(i), parent(parent(i)), ...}.
 * tree_parent: DEVICE [batch][n_draft] int32, parent < i or -1 for a root
 * (a forest is allowed).  block_tables / ctx_lens: HOST [batch][max_blocks] /
 * [batch].  Other arguments as for paged_decode_attention with
 * num_seqs = batch * n_draft query rows.  A bad parent pointer sets
 * KVP_DEVERR_TREE_PARENT in the workspace error word and that node is
 * treated as a root.  Pages must be bf16 (desc->kv_format = KVP_KV_BF16).
 */
int tree_verify_attention(const void *q, const int32_t *tree_parent, int32_t n_draft,
                          const void *k_pool, const void *v_pool, const int32_t *block_tables,
                          const int32_t *ctx_lens, int32_t batch, int32_t max_blocks,
                          const kvp_attn_desc *desc, void *out, float *lse, void *workspace,
                          size_t ws_bytes, void *stream);

/*
 * Decode attention for callers that cannot allocate device memory -- e.g. a
 * serving process whose memory manager has already given (nearly) all device
 * memory to its own pools, or a plug-in that cannot reach its host program's
 * allocator and must not bypass it.  Same arguments and results as
 * paged_decode_attention, without workspace: the scratch space is a
 * KVP_STATIC_WORKSPACE_BYTES array inside the library, present on every GPU
 * that loads it until the process exits.  The pages have no counterpart; this
 * is an interface for such callers.
 *   - Returns KVP_ERR_INVALID, before enqueuing anything, when the batch's plan
 *     needs more than KVP_STATIC_WORKSPACE_BYTES (see
 *     kvp_decode_workspace_size).
 *   - All calls on a device share the array: calls that overlap on the GPU
 *     race; serialise them.  Each call rewrites the words that must start at
 *     zero (error word, work counters) before its kernels run.
 *   - The first call on each device looks up the array's device address; make
 *     it before any stream capture.  No call allocates device memory.
 * kvp_device_error cannot read this call's error word (there is no caller
 * workspace); bounds violations still skip the access.
 */
#define KVP_STATIC_WORKSPACE_BYTES (32u << 20)
int paged_decode_attention_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, const int32_t *seq_lens,
                                   int32_t num_seqs, int32_t max_blocks, const kvp_attn_desc *desc,
                                   void *out, float *lse, void *stream);

/*
 * Decode attention over pool sequences: paged_decode_attention with the block
 * tables and lengths read from the pool itself, so the caller keeps no host
 * tables.  Row s of q / out / lse is sequence seq_ids[s] (host array) at its
 * current length.  desc must describe the pool (layers, kv heads, head dim,
 * block size, block count and page format); 4-bit pools read their codes and
 * exponents.  kvp_pool_decode_workspace_size returns the workspace bytes for
 * the sequences as they are now (0 on invalid input).
 */
size_t kvp_pool_decode_workspace_size(const kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs,
                                      const kvp_attn_desc *desc);
int paged_decode_attention_pool(const kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs,
                                const void *q, void *out, float *lse, const kvp_attn_desc *desc,
                                void *workspace, size_t ws_bytes, void *stream);

/*
 * One decode step, host buffers in and out ("Dendrite", API example: every
 * branch appends its new token and attends over its own blocks, the shared
 * prefix included).  In stream order on `stream`:
 *   1. host-to-device copies h_k_new -> d_k_new, h_v_new -> d_v_new and
 *      h_q -> d_q (each skipped when its host pointer is NULL: the data is
 *      already on the device);
 *   2. seq_append_batch of ntok tokens to every sequence (skipped for ntok 0):
 *      its bookkeeping and the plan of step 3 are done on the host first, and
 *      its write kernel is enqueued right before the attention kernels, which
 *      are launched programmatically behind it (they start while it
 *      finishes and wait for it before reading K/V);
 *   3. paged_decode_attention_pool over the sequences at their new lengths,
 *      d_q -> d_out, d_lse;
 *   4. device-to-host copies d_out -> h_out and d_lse -> h_lse (each skipped
 *      when its host pointer is NULL).
 * The call returns once all of it is enqueued; host outputs are valid after
 * the stream synchronises, and host inputs must stay untouched until then.
 * Page-locked host buffers make the copies asynchronous; pageable ones work,
 * but the driver then stages each copy before returning.  With
 * KVP_STEP_HOST_MAPPED in io->flags the host buffers must be page-locked and
 * addressable by the device (cudaHostAlloc, or registered with
 * cudaHostRegisterMapped; under unified addressing any page-locked memory)
 * and 16-byte aligned: the inputs then cross in one copy kernel into the d_*
 * buffers, and the attention kernels write out and lse straight into h_out /
 * h_lse (d_out and d_lse are then neither read nor written and may be NULL),
 * instead of one copy-engine transfer per buffer.
 *
 * Shapes: k_new, v_new [L][num_seqs * ntok][Hkv][d] bf16, sequence-major;
 * q, out [L][num_seqs][Hq][d] bf16; lse [L][num_seqs][Hq] fp32 (d_lse may be
 * NULL, then h_lse must be NULL too).  seq_ids: host, distinct live
 * sequences.  *ws_needed (may be NULL) receives the workspace bytes the
 * attention needed.
 * Errors: KVP_ERR_INVALID (bad arguments, descriptor not matching the pool,
 * unknown flags, misaligned mapped buffers) and KVP_ERR_OOM (the appends do
 * not fit) before anything is enqueued; KVP_ERR_WORKSPACE when ws_bytes <
 * *ws_needed: the copies and the append of steps 1-2 are enqueued and the
 * pool holds the new tokens, nothing else ran; grow the workspace and finish
 * the step with paged_decode_attention_pool.
 */
typedef struct {
    const void *h_k_new, *h_v_new, *h_q; /* host inputs, or NULL */
    void *h_out;                         /* host outputs, or NULL */
    float *h_lse;
    void *d_k_new, *d_v_new, *d_q;       /* device inputs / staging */
    void *d_out;                         /* device outputs */
    float *d_lse;
    uint32_t flags;                      /* KVP_STEP_* */
} kvp_step_io;

enum { KVP_STEP_HOST_MAPPED = 1 };

int kvp_decode_step(kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs, int32_t ntok,
                    const kvp_step_io *io, const kvp_attn_desc *desc, void *workspace,
                    size_t ws_bytes, size_t *ws_needed, void *stream);

/*
 * kvp_decode_step in two halves, so that the host work of step i + 1 can run
 * while the device runs step i (each sequence appending ntok tokens per step
 * is known before the step's K/V and q are):
 *
 *   kvp_decode_step_plan: the checks of kvp_decode_step that involve the pool,
 *     then the append's bookkeeping (the sequences grow by ntok tokens at once:
 *     slots and copy-on-write copies are assigned) and the attention plan over
 *     the grown sequences, packed into `plan`.  No device work.  *ws_needed
 *     (may be NULL) receives the workspace bytes the run will need.
 *   kvp_decode_step_run: steps 1-4 of kvp_decode_step for that plan, with the
 *     plan's upload into `workspace` right before the append's write.
 *
 * Both kvp_decode_step and kvp_decode_step_run, when the step's inputs are
 * already on the device or in mapped host memory (KVP_STEP_HOST_MAPPED), the
 * pool holds bf16 pages, the append has at most 64 tokens and 16
 * copy-on-write blocks and the plan at most 24 KB, make steps 1-2 and the
 * plan upload one kernel: the new K/V go straight into their pool slots (from
 * host memory when mapped; d_k_new / d_v_new are then left unwritten), q to
 * d_q, and the plan, carried in the kernel's parameters, into the workspace;
 * attention and merge follow.
 *
 * A plan object (kvp_step_plan_create; kvp_step_plan_destroy frees it) holds
 * one planned step at a time and is reused from step to step.  Planning a
 * plan that is still waiting for its run is KVP_ERR_INVALID, since its
 * tokens are already in the sequences.  Between plan and run no call may
 * change the planned sequences or free blocks; appends and attention on other
 * sequences may run.  `workspace` belongs to the run until the stream passes
 * its kernels, as for every attention call.  The run takes its device
 * buffers from io as kvp_decode_step does (num_seqs and ntok are the plan's).
 * Errors: the plan call as kvp_decode_step's (KVP_ERR_INVALID, KVP_ERR_OOM;
 * nothing changed); the run returns KVP_ERR_INVALID for a plan that is not
 * waiting for its run or bad buffers (the plan then stays ready), and
 * KVP_ERR_WORKSPACE when ws_bytes is short: the inputs' copies and the
 * append's write are enqueued, nothing else; the plan is used up.
 */
typedef struct kvp_step_plan kvp_step_plan;

kvp_step_plan *kvp_step_plan_create(void);
void kvp_step_plan_destroy(kvp_step_plan *plan);
int kvp_decode_step_plan(kvp_pool *pool, const int32_t *seq_ids, int32_t num_seqs, int32_t ntok,
                         const kvp_attn_desc *desc, kvp_step_plan *plan, size_t *ws_needed);
int kvp_decode_step_run(kvp_step_plan *plan, const kvp_step_io *io, void *workspace, size_t ws_bytes,
                        void *stream);

/* Reads (and clears) the device error word that the last attention call on
 * this workspace left; synchronises `stream`.  *err_out = 0 when clean. */
int kvp_device_error(void *workspace, void *stream, int32_t *err_out);

/* Host-side view of the decode plan (no device work; for tests and tools):
 * work items, row tiles, 64-token KV tiles and partial rows per (layer, kv
 * head), and the bytes of distinct (block, valid tokens) one call reads over
 * all layers (K and V rows in the pool's format: d bf16 values, or d/2 code
 * bytes and one exponent byte), planned for a GPU with sm_count SMs.  Any out-pointer may be
 * NULL.  The plan's internal invariants (tile ranges inside the tile list
 * and within the kernels' descriptor stage, rows within each kernel's unit,
 * member intervals inside their items) are checked: KVP_ERR_STATE if one
 * fails, which would be a planner defect. */
int kvp_decode_plan_stats(const kvp_attn_desc *desc, const int32_t *block_tables,
                          const int32_t *seq_lens, int32_t num_seqs, int32_t max_blocks,
                          int32_t sm_count, int32_t *n_items, int32_t *n_row_tiles,
                          int32_t *n_kv_tiles, int32_t *n_partial_rows, int64_t *unique_kv_bytes);

/* Measurement hooks.  kvp_set_kernel_events: cudaEvent_t handles (as void*)
 * that every later attention call on this thread records on its stream
 * immediately before and after its main attention kernel (the work-item
 * kernel), so a caller can time that kernel alone; NULL, NULL turns it off.
 * kvp_kernel_launches: total kernels this library has launched in the
 * process (all threads). */
int kvp_set_kernel_events(void *before, void *after);
int kvp_kernel_launches(int64_t *n_out);

const char *kvp_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* KVP_H */
