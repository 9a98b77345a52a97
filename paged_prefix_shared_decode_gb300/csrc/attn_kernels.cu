// Paged attention work-item kernel and log-sum-exp merge (sm_103a).
//
// A persistent grid (up to four CTAs of 4 warps per SM) pulls work units --
// (work item, layer, kv head) -- from an atomic counter, longest first.  A
// unit is up to 64 query rows (sequences or draft nodes x the GQA group that
// shares this kv head) against a list of 64-token KV tiles.  The tiles'
// descriptors, which carry the physical block ids, are staged in shared
// memory first; then each tile's K and V are copied into a 3-deep shared
// memory ring (cp.async, 16-byte chunks, XOR-swizzled rows) and used by every
// row of the unit.  This is how a block shared by several sequences is read
// from HBM once for all of them.
// Q K^T and P V run on bf16 tensor cores (mma.sync m16n8k16, fp32
// accumulate) with an online softmax in fp32 (base-2 exponent, scale * log2 e
// folded into the scores).  Rows outside a tile's member interval, tokens past
// the tile's end and draft tokens that are not ancestors-or-self of a node
// are masked.  With at most 16 rows the four warps split each tile's tokens
// four ways (with at most 32 rows at head dim 128, two ways) and combine
// their (m, l, o) through shared memory.
//
// 4-bit pages (codes in [-7, 7] and one power-of-two exponent per token row,
// value = code * 2^e) are staged as codes and exponents -- 4.125 bits per
// value at head dim 64 instead of 16.  Units whose warps split the tiles'
// tokens take the codes from shared memory straight into the mma operands
// (exact bf16 code * 2^e, formed in registers); units of more than 16 rows,
// whose warps all read every token, first expand each tile once into a bf16
// tile in shared memory and then run the bf16 path.
//
// A unit writes out (bf16) and lse (fp32, natural log) directly, or -- when
// its rows' keys are split over several units -- normalised partial o and a
// base-2 lse per row, which the merge kernels combine (one warp per query
// head, or per kv head's group of query heads when there are many queries):
//   out = sum_c w_c o_c / sum_c w_c,  w_c = 2^(lse_c - max lse),
//   lse = max lse + log2(sum w)   (converted to natural log).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kv4_codes.cuh"
#include "kvp_internal.h"

namespace kvp {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the kernel before it in the stream still
// runs; griddep_wait() returns once that kernel has completed and its writes
// are visible (at once when launched normally).  griddep_trigger() lets the
// next kernel start launching before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_trigger() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// 2^x on the SFU (hardware instruction); 2^-inf = +0.
__device__ __forceinline__ float exp2_sfu(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t ld_u32(const void *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

// ancestor-or-self bitmask of draft node i of sequence b (bit j = node j)
__device__ uint64_t ancestor_mask(const int32_t *parent, int b, int i, int n, int32_t *err) {
    uint64_t m = 0;
    int j = i;
    for (int step = 0; step < 64 && j >= 0; ++step) {
        m |= 1ull << j;
        const int p = __ldg(parent + (size_t)b * n + j);
        if (p >= j || p < -1) {
            atomicOr(err, 2);
            break;
        }
        j = p;
    }
    return m;
}

// Ancestor-or-self masks of all draft query tokens, once per call, so the
// attention kernels read one word per query row instead of walking the tree.
__global__ void tree_mask_kernel(const int32_t *parent, int32_t nq, int32_t n, uint64_t *mask,
                                 int32_t *err) {
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q < nq) mask[q] = ancestor_mask(parent, q / n, q % n, n, err);
}

// K word (8 dims of one token with exponent e) -> b[0..3] = pairs 0..3
__device__ __forceinline__ void code_pairs_k(uint32_t w, int e, bool fused, uint32_t (&b)[4]) {
    const uint2 sc = exp_pair2(e, e);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = conv_pair(nib_pair(w, i), sc, fused);
}
// V word (4 dims of two tokens) with its exponent pair -> b[0..3]
__device__ __forceinline__ void code_pairs_v(uint32_t w, uint2 sc, bool fused, uint32_t (&b)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = conv_pair(nib_pair(w, i), sc, fused);
}

template <int D>
struct KCfg {
    static constexpr int CH = D / 8;                        // 16-byte chunks per token row
    static constexpr int TILE_BYTES = kTileTokens * D * 2;  // one K (or V) tile
    // three stages and (d 64) four CTAs per SM: more resident warps hide the
    // mma.sync / SFU latencies better than a deeper ring (measured)
    static constexpr int NSTAGE = 3;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int DESC_OFF = NSTAGE * STAGE_BYTES;
    static constexpr int SMEM = DESC_OFF + kMaxItemTiles * (int)sizeof(KvTile);
    static constexpr int MIN_BLOCKS = D == 64 ? 4 : 2;
    static constexpr int NO = D / 8;    // n-tiles of O
    static constexpr int KS = D / 16;   // k-steps of Q K^T
};

// 4-bit pages: a ring of staged codes and exponents, expanded into one bf16
// K/V tile before each tile's math.
template <int D>
struct KCfg4 {
    static constexpr int CH4 = D / 32;                     // 16-byte code chunks per row
    // code rows are 32 (d 64) or 64 (d 128) bytes: chunk c of row tok is
    // stored at chunk c ^ ((tok >> SWS) & (CH4 - 1)), so that the 8 rows an
    // ldmatrix reads fall in different banks
    static constexpr int SWS = CH4 == 2 ? 2 : 1;
    static constexpr int CODE_BYTES = kTileTokens * D / 2; // one K (or V) tile of codes
    static constexpr int NSTAGE = 3;
    static constexpr int STAGE_BYTES = 2 * CODE_BYTES + 2 * kTileTokens;   // codes K, V; exponents K, V
    static constexpr int BF_OFF = NSTAGE * STAGE_BYTES;    // bf16 K then V tile (the mma layout)
    static constexpr int DESC_OFF = BF_OFF + 2 * KCfg<D>::TILE_BYTES;
    static constexpr int SMEM = DESC_OFF + kMaxItemTiles * (int)sizeof(KvTile);
    // the token-split combine overlays the staging ring and bf16 tile
    static_assert(4 * (KCfg<D>::NO * 4 + 4) * 32 * 4 <= DESC_OFF, "combine area");
};

// One work unit with TS warps splitting each tile's tokens.  KV4: the pool
// holds 4-bit codes and row exponents (a.k_pool / a.v_pool are the codes).
template <int D, int TS, bool KV4, bool TREE>
__device__ __forceinline__ void run_unit(const AttnLaunch &a, const WorkItem &it, int l, int kvh,
                                         int ntile, unsigned char *smem, const KvTile *s_tiles, int *s_next) {
    using C = KCfg<D>;
    using C4 = KCfg4<D>;
    constexpr int NSTAGE = KV4 ? C4::NSTAGE : C::NSTAGE;
    constexpr int TOKW = kTileTokens / TS;   // tokens per warp per tile
    constexpr int NT = TOKW / 8;             // score n-tiles per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = warp / TS, sp = warp % TS;
    const int G = a.G;
    const int n_rows = it.n_members * G;
    const int gq = lane >> 2, tq = lane & 3;
    const int row0 = rg * 16 + gq, row1 = row0 + 8;
    const bool has0 = row0 < n_rows, has1 = row1 < n_rows;
    const int mem0 = row0 / G, mem1 = row1 / G;

    const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *kpool = static_cast<const __nv_bfloat16 *>(a.k_pool);
    const __nv_bfloat16 *vpool = static_cast<const __nv_bfloat16 *>(a.v_pool);

    int qt0 = 0, qt1 = 0;
    const __nv_bfloat16 *q0 = nullptr, *q1 = nullptr;
    if (has0) {
        qt0 = __ldg(a.members + it.member_off + mem0);
        q0 = qb + (((size_t)l * a.nq + qt0) * a.Hq + kvh * G + row0 % G) * D;
    }
    if (has1) {
        qt1 = __ldg(a.members + it.member_off + mem1);
        q1 = qb + (((size_t)l * a.nq + qt1) * a.Hq + kvh * G + row1 % G) * D;
    }

    const int bs_log2 = a.bs_log2;
    const int bs_mask = (1 << bs_log2) - 1;
    const size_t head_stride = (size_t)D << bs_log2;            // one (block, head) tile
    const size_t layer_base = (size_t)l * a.NB * a.Hkv * head_stride + (size_t)kvh * head_stride;
    const size_t block_stride = (size_t)a.Hkv * head_stride;

    // 4-bit: codes of row r at row * D/2, exponent at row, row =
    // ((l * NB + block) * Hkv + kvh) * bs + slot
    auto issue4 = [&](int t) {
        const KvTile &kt = s_tiles[t];
        const int ntok = kt.ntok_flags & 0xFFFF;
        const int jb = kt.tok0 >> bs_log2;
        const uint32_t st = smem_addr(smem + (t % NSTAGE) * C4::STAGE_BYTES);
        const uint8_t *kc = static_cast<const uint8_t *>(a.k_pool), *vc = static_cast<const uint8_t *>(a.v_pool);
        const int8_t *ke = static_cast<const int8_t *>(a.k_exp), *ve = static_cast<const int8_t *>(a.v_exp);
        const size_t lrow = (size_t)l * a.NB * a.Hkv;   // + block * Hkv + kvh, times bs
        for (int x = threadIdx.x; x < kTileTokens * C4::CH4; x += kThreads) {
            const int tok = x / C4::CH4, c = x % C4::CH4;
            const uint8_t *sk = kc, *sv = vc;
            int bytes = 0;
            if (tok < ntok) {
                const int pos = kt.tok0 + tok;
                const int blk = kt.blk[(pos >> bs_log2) - jb];
                if ((unsigned)blk < (unsigned)a.NB) {
                    const size_t row = ((lrow + (size_t)blk * a.Hkv + kvh) << bs_log2) + (pos & bs_mask);
                    sk = kc + row * (D / 2) + c * 16;
                    sv = vc + row * (D / 2) + c * 16;
                    bytes = 16;
                } else if (c == 0) {
                    atomicOr(a.err, 1);
                }
            }
            const int cs = (c ^ ((tok >> C4::SWS) & (C4::CH4 - 1))) * 16;
            cp_async16(st + tok * (D / 2) + cs, sk, bytes);
            cp_async16(st + C4::CODE_BYTES + tok * (D / 2) + cs, sv, bytes);
        }
        // exponents: four groups of 16 tokens, each inside one block (tiles
        // start on a block boundary and blocks are a multiple of 16 tokens)
        if (threadIdx.x < 8) {
            const int j = threadIdx.x & 3;
            const bool is_v = threadIdx.x >= 4;
            const int8_t *e = is_v ? ve : ke;
            const int8_t *src = e;
            int bytes = 0;
            if (16 * j < ntok) {
                const int pos = kt.tok0 + 16 * j;
                const int blk = kt.blk[(pos >> bs_log2) - jb];
                if ((unsigned)blk < (unsigned)a.NB) {
                    src = e + ((lrow + (size_t)blk * a.Hkv + kvh) << bs_log2) + (pos & bs_mask);
                    bytes = 16;
                }
            }
            cp_async16(st + 2 * C4::CODE_BYTES + (is_v ? kTileTokens : 0) + 16 * j, src, bytes);
        }
    };
    // expands the staged tile t into the bf16 tile: value = code * 2^e, by a
    // table of each byte's two codes as bf16 pairs and an exact multiply by
    // the power of two
    // expands the staged tile t into the bf16 tile: value = code * 2^e,
    // formed exactly in registers (each thread: one 16-byte chunk of codes,
    // 32 dims of one row, into four 16-byte chunks of the bf16 tile)
    auto expand4 = [&](int t) {
        const unsigned char *stg = smem + (t % NSTAGE) * C4::STAGE_BYTES;
        for (int x = threadIdx.x; x < 2 * kTileTokens * C4::CH4; x += kThreads) {
            const int kv = x / (kTileTokens * C4::CH4);
            const int y = x % (kTileTokens * C4::CH4);
            const int tok = y / C4::CH4, q = y % C4::CH4;   // code chunk q: dims 32 q .. 32 q + 31
            const uint4 cw = *reinterpret_cast<const uint4 *>(
                stg + kv * C4::CODE_BYTES + tok * (D / 2) + ((q ^ ((tok >> C4::SWS) & (C4::CH4 - 1))) << 4));
            const int e = (int)reinterpret_cast<const int8_t *>(stg + 2 * C4::CODE_BYTES + kv * kTileTokens)[tok];
            const bool fused = e >= -126 && e <= 120;
            const uint2 sc = exp_pair2(e, e);
            const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {   // word k: dims 32 q + 8 k .. + 7
                uint4 v;
                expand_word(w[k], sc, fused, *reinterpret_cast<uint32_t(*)[4]>(&v));
                const int c = 4 * q + k;
                *reinterpret_cast<uint4 *>(smem + C4::BF_OFF + kv * C::TILE_BYTES + tok * D * 2 + ((c ^ (tok & 7)) << 4)) = v;
            }
        }
    };

    auto issue = [&](int t) {
        if constexpr (KV4) {
            issue4(t);
            return;
        }
        // a tile may start anywhere in a block (a verify tile's draft tokens
        // start right after the context), so block and slot come from the
        // absolute position
        const KvTile &kt = s_tiles[t];
        const int ntok = kt.ntok_flags & 0xFFFF;
        const int jb = kt.tok0 >> bs_log2;
        const uint32_t dK = smem_addr(smem + (t % C::NSTAGE) * C::STAGE_BYTES);
        const uint32_t dV = dK + C::TILE_BYTES;
        const __nv_bfloat16 *kb = kpool + layer_base, *vb = vpool + layer_base;
        if constexpr (D == 128) {
            // each thread copies chunk c of NI consecutive tokens (a warp's copy
            // instruction covers two whole 256-byte token rows) and finds their
            // block once; the tokens of a group lie in one block unless the tile
            // starts off a block boundary near its end (measured 1.6% faster on
            // MCTS; at head dim 64 the mapping below, whose copy instructions
            // cover 512 contiguous bytes, measured faster)
            constexpr int NI = kTileTokens * C::CH / kThreads;
            const int g0 = (threadIdx.x / C::CH) * NI, c = threadIdx.x % C::CH;
            const int pos0 = kt.tok0 + g0;
            const bool one_block = (pos0 & bs_mask) + NI - 1 <= bs_mask;
            const int blk0 = kt.blk[(pos0 >> bs_log2) - jb];
            const size_t e0 = (size_t)blk0 * block_stride + (size_t)((pos0 & bs_mask) * D + c * 8);
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int tok = g0 + i;
                const uint32_t off = tok * D * 2 + ((c ^ (tok & 7)) << 4);
                const __nv_bfloat16 *sk = kpool, *sv = vpool;
                int bytes = 0;
                if (tok < ntok) {
                    const int pos = pos0 + i;
                    const int blk = one_block ? blk0 : kt.blk[(pos >> bs_log2) - jb];
                    if ((unsigned)blk < (unsigned)a.NB) {
                        const size_t e = one_block ? e0 + (size_t)i * D
                                                   : (size_t)blk * block_stride + (size_t)((pos & bs_mask) * D + c * 8);
                        sk = kb + e;
                        sv = vb + e;
                        bytes = 16;
                    } else if (c == 0) {
                        atomicOr(a.err, 1);
                    }
                }
                cp_async16(dK + off, sk, bytes);
                cp_async16(dV + off, sv, bytes);
            }
        } else {
            const int tok_t = threadIdx.x / C::CH, c = threadIdx.x % C::CH;
#pragma unroll
            for (int i = 0; i < kTileTokens * C::CH / kThreads; ++i) {
                const int tok = tok_t + i * (kThreads / C::CH);
                const uint32_t off = tok * D * 2 + ((c ^ (tok & 7)) << 4);
                const __nv_bfloat16 *sk = kpool, *sv = vpool;
                int bytes = 0;
                if (tok < ntok) {
                    const int pos = kt.tok0 + tok;
                    const int blk = kt.blk[(pos >> bs_log2) - jb];
                    if ((unsigned)blk < (unsigned)a.NB) {
                        const size_t e = (size_t)blk * block_stride + (size_t)((pos & bs_mask) * D + c * 8);
                        sk = kb + e;
                        sv = vb + e;
                        bytes = 16;
                    } else if (c == 0) {
                        atomicOr(a.err, 1);
                    }
                }
                cp_async16(dK + off, sk, bytes);
                cp_async16(dV + off, sv, bytes);
            }
        }
    };

#pragma unroll
    for (int t = 0; t < NSTAGE - 1; ++t) {
        if (t < ntile) issue(t);
        cp_async_commit();
    }

    // REG4: 4-bit codes go from shared memory straight into mma operands.
    // A thread's ldmatrix word of K codes holds 8 dims of one token, 32 c +
    // 8 tq + k for nibble k; nibble pairs (i, i + 4) form its bf16 pairs, so
    // the Q K^T contraction runs over dims in that order and Q's fragments
    // are gathered to match (k-step 2c + h pairs dims 8 tq + 2h + {0, 4} and
    // 8 tq + 2h + {1, 5} of chunk c).
    constexpr bool REG4 = KV4 && TS > 1;
    uint32_t qf[C::KS][4];
    if constexpr (REG4) {
#pragma unroll
        for (int c = 0; c < C4::CH4; ++c) {
            uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
            if (has0) x0 = __ldg(reinterpret_cast<const uint4 *>(q0 + 32 * c + 8 * tq));
            if (has1) x1 = __ldg(reinterpret_cast<const uint4 *>(q1 + 32 * c + 8 * tq));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t lo0 = h ? x0.y : x0.x, hi0 = h ? x0.w : x0.z;
                const uint32_t lo1 = h ? x1.y : x1.x, hi1 = h ? x1.w : x1.z;
                qf[2 * c + h][0] = __byte_perm(lo0, hi0, 0x5410);
                qf[2 * c + h][1] = __byte_perm(lo1, hi1, 0x5410);
                qf[2 * c + h][2] = __byte_perm(lo0, hi0, 0x7632);
                qf[2 * c + h][3] = __byte_perm(lo1, hi1, 0x7632);
            }
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < C::KS; ++kk) {
            const int c = kk * 16 + 2 * tq;
            qf[kk][0] = has0 ? ld_u32(q0 + c) : 0u;
            qf[kk][1] = has1 ? ld_u32(q1 + c) : 0u;
            qf[kk][2] = has0 ? ld_u32(q0 + c + 8) : 0u;
            qf[kk][3] = has1 ? ld_u32(q1 + c + 8) : 0u;
        }
    }
    uint64_t tm0 = ~0ull, tm1 = ~0ull;
    if (TREE) {
        if (has0) tm0 = a.tree_mask[qt0];
        if (has1) tm1 = a.tree_mask[qt1];
    }

    float o[C::NO][4];
#pragma unroll
    for (int n = 0; n < C::NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int t = 0; t < ntile; ++t) {
        cp_async_wait<NSTAGE - 2>();
        __syncthreads();
        // claim the next unit while the last tile computes (every thread
        // read the current one before the first barrier of the loop); by the
        // last warp, which a unit of 33-48 rows leaves without rows
        if (t == ntile - 1 && threadIdx.x == kThreads - 32)
            *s_next = (a.n_tc_units > 0 ? 0 : gridDim.x) + atomicAdd(a.counter, 1);
        if (t + NSTAGE - 1 < ntile) issue(t + NSTAGE - 1);
        cp_async_commit();
        if constexpr (KV4 && !REG4) {
            expand4(t);
            __syncthreads();
        }

        const KvTile &kt = s_tiles[t];
        const int ntok = kt.ntok_flags & 0xFFFF;
        const bool tree = TREE && ((kt.ntok_flags >> 16) & kTileTree);
        const int mlo = kt.members & 0xFFFF, mhi = kt.members >> 16;
        const bool in0 = has0 && mem0 >= mlo && mem0 < mhi;
        const bool in1 = has1 && mem1 >= mlo && mem1 < mhi;
        const int tb = sp * TOKW;
        if (!__any_sync(0xffffffffu, in0 || in1) || tb >= ntok) continue;

        const uint32_t aK = KV4 ? smem_addr(smem + C4::BF_OFF) : smem_addr(smem + (t % C::NSTAGE) * C::STAGE_BYTES);
        const uint32_t aV = aK + C::TILE_BYTES;

        float s[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
        // REG4: codes and exponents of this tile's stage
        const unsigned char *stg4 = REG4 ? smem + (t % NSTAGE) * C4::STAGE_BYTES : smem;
        const uint32_t aK4 = smem_addr(stg4), aV4 = aK4 + C4::CODE_BYTES;
        const int8_t *ek4 = reinterpret_cast<const int8_t *>(stg4 + 2 * C4::CODE_BYTES);
        const int8_t *ev4 = ek4 + kTileTokens;
        // fused conversion code * 2^e = fma(bf16(136 + code), 2^e, -136 * 2^e)
        // needs both factors normal: -126 <= e <= 120 for every token of the
        // warp's share of the tile (else: subtract, then multiply)
        bool fused4 = true;
        if constexpr (REG4) {
#pragma unroll
            for (int j2 = 0; j2 < NT / 2; ++j2) {
                const int t0k = tb + 16 * j2;
                const int e0 = ek4[t0k + gq], e1 = ek4[t0k + 8 + gq];
                const int e2 = ev4[t0k + 2 * tq], e3 = ev4[t0k + 2 * tq + 1];
                const int e4 = ev4[t0k + 8 + 2 * tq], e5 = ev4[t0k + 9 + 2 * tq];
                const int lo = min(min(min(e0, e1), min(e2, e3)), min(e4, e5));
                const int hi = max(max(max(e0, e1), max(e2, e3)), max(e4, e5));
                fused4 = fused4 && lo >= -126 && hi <= 120;
            }
            fused4 = __all_sync(0xffffffffu, fused4);
        }
        if constexpr (REG4) {
#pragma unroll
            for (int j2 = 0; j2 < NT / 2; ++j2) {
                const int t0k = tb + 16 * j2;
#pragma unroll
                for (int cp = 0; cp < C4::CH4 / 2; ++cp) {
                    const int tok = t0k + ((lane >> 4) << 3) + (lane & 7);
                    const int ch = 2 * cp + ((lane >> 3) & 1);
                    uint32_t w[4];
                    ldsm_x4(aK4 + tok * (D / 2) + ((ch ^ ((tok >> C4::SWS) & (C4::CH4 - 1))) << 4), w[0], w[1], w[2],
                            w[3]);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int e = ek4[t0k + ((m >> 1) << 3) + gq];
                        const int c = 2 * cp + (m & 1);
                        uint32_t b[4];
                        code_pairs_k(w[m], e, fused4, b);
                        mma16816(s[2 * j2 + (m >> 1)], qf[2 * c], b[0], b[1]);
                        mma16816(s[2 * j2 + (m >> 1)], qf[2 * c + 1], b[2], b[3]);
                    }
                }
            }
        } else
#pragma unroll
        for (int kk = 0; kk < C::KS; ++kk) {
#pragma unroll
            for (int j2 = 0; j2 < NT / 2; ++j2) {
                const int tok = tb + j2 * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = kk * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(aK + tok * D * 2 + ((ch ^ (tok & 7)) << 4), b0, b1, b2, b3);
                mma16816(s[2 * j2], qf[kk], b0, b1);
                mma16816(s[2 * j2 + 1], qf[kk], b2, b3);
            }
        }
        // raw scores; masked ones -inf.  Padding rows (past the item's rows)
        // are never written, so whole tiles seen by every real row skip masking.
        const bool fast = tb + TOKW <= ntok && !tree && (in0 || !has0) && (in1 || !has1);
        if (!__all_sync(0xffffffffu, fast)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = tb + j * 8 + 2 * tq + (e & 1);
                    const bool hi = e >= 2;
                    bool ok = tok < ntok && (hi ? in1 : in0);
                    if (tree) ok = ok && (((hi ? tm1 : tm0) >> (tok & 63)) & 1ull);
                    if (!ok) s[j][e] = -INFINITY;
                }
            }
        }
        float mx0 = s[0][0], mx1 = s[0][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
            mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // the running max m (base-2, scaled) is raised only when a tile's max
        // exceeds it by more than 8, so p = 2^(s*scale - m) <= 2^8 and O is
        // rarely rescaled
        const float sc = a.scale_log2;
        const float t0 = mx0 * sc, t1 = mx1 * sc;
        const bool up0 = m0 == -INFINITY ? t0 != -INFINITY : t0 > m0 + 8.f;
        const bool up1 = m1 == -INFINITY ? t1 != -INFINITY : t1 > m1 + 8.f;
        if (__any_sync(0xffffffffu, (up0 && m0 != -INFINITY) || (up1 && m1 != -INFINITY))) {
            const float al0 = up0 && m0 != -INFINITY ? exp2_sfu(m0 - t0) : 1.f;
            const float al1 = up1 && m1 != -INFINITY ? exp2_sfu(m1 - t1) : 1.f;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int n = 0; n < C::NO; ++n) {
                o[n][0] *= al0;
                o[n][1] *= al0;
                o[n][2] *= al1;
                o[n][3] *= al1;
            }
        }
        if (up0) m0 = t0;
        if (up1) m1 = t1;
        const float nm0 = m0 == -INFINITY ? 0.f : -m0, nm1 = m1 == -INFINITY ? 0.f : -m1;
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            s[j][0] = exp2_sfu(fmaf(s[j][0], sc, nm0));
            s[j][1] = exp2_sfu(fmaf(s[j][1], sc, nm0));
            s[j][2] = exp2_sfu(fmaf(s[j][2], sc, nm1));
            s[j][3] = exp2_sfu(fmaf(s[j][3], sc, nm1));
            rs0 += s[j][0] + s[j][1];
            rs1 += s[j][2] + s[j][3];
        }
        l0 += rs0;
        l1 += rs1;
#pragma unroll
        for (int k2 = 0; k2 < NT / 2; ++k2) {
            const uint32_t pa[4] = {pack_bf16x2(s[2 * k2][0], s[2 * k2][1]),
                                    pack_bf16x2(s[2 * k2][2], s[2 * k2][3]),
                                    pack_bf16x2(s[2 * k2 + 1][0], s[2 * k2 + 1][1]),
                                    pack_bf16x2(s[2 * k2 + 1][2], s[2 * k2 + 1][3])};
            if constexpr (REG4) {
                // V: .trans ldmatrix words hold 4 dims (32 c + 4 gq + i) of
                // two tokens; n-tile 4 c + i takes nibble i of each
                const int t0k = tb + k2 * 16;
                const uint2 sv0 = exp_pair2(ev4[t0k + 2 * tq], ev4[t0k + 2 * tq + 1]);
                const uint2 sv1 = exp_pair2(ev4[t0k + 8 + 2 * tq], ev4[t0k + 9 + 2 * tq]);
#pragma unroll
                for (int cp = 0; cp < C4::CH4 / 2; ++cp) {
                    const int m = lane >> 3;
                    const int tok = t0k + ((m & 1) << 3) + (lane & 7);
                    const int ch = 2 * cp + (m >> 1);
                    uint32_t w[4];
                    ldsm_x4_t(aV4 + tok * (D / 2) + ((ch ^ ((tok >> C4::SWS) & (C4::CH4 - 1))) << 4), w[0], w[1],
                              w[2], w[3]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t b0[4], b1[4];
                        code_pairs_v(w[2 * h], sv0, fused4, b0);
                        code_pairs_v(w[2 * h + 1], sv1, fused4, b1);
#pragma unroll
                        for (int i = 0; i < 4; ++i) mma16816(o[4 * (2 * cp + h) + i], pa, b0[i], b1[i]);
                    }
                }
                continue;
            }
            const int tok = tb + k2 * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int n2 = 0; n2 < C::NO / 2; ++n2) {
                const int ch = n2 * 2 + (lane >> 4);
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(aV + tok * D * 2 + ((ch ^ (tok & 7)) << 4), v0, v1, v2, v3);
                mma16816(o[2 * n2], pa, v0, v1);
                mma16816(o[2 * n2 + 1], pa, v2, v3);
            }
        }
    }
    cp_async_wait<0>();

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    if constexpr (TS > 1) {
        // combine the token-split warps of each row group through shared memory
        __syncthreads();
        float *red = reinterpret_cast<float *>(smem);
        constexpr int PER_WARP = (C::NO * 4 + 4) * 32;
        float *mine = red + warp * PER_WARP;
#pragma unroll
        for (int n = 0; n < C::NO; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) mine[(n * 4 + e) * 32 + lane] = o[n][e];
        mine[(C::NO * 4 + 0) * 32 + lane] = m0;
        mine[(C::NO * 4 + 1) * 32 + lane] = m1;
        mine[(C::NO * 4 + 2) * 32 + lane] = l0;
        mine[(C::NO * 4 + 3) * 32 + lane] = l1;
        __syncthreads();
        if (sp == 0) {
#pragma unroll
            for (int s2 = 1; s2 < TS; ++s2) {
                const float *oth = red + (warp + s2) * PER_WARP;
                const float om0 = oth[(C::NO * 4 + 0) * 32 + lane];
                const float om1 = oth[(C::NO * 4 + 1) * 32 + lane];
                const float ol0 = oth[(C::NO * 4 + 2) * 32 + lane];
                const float ol1 = oth[(C::NO * 4 + 3) * 32 + lane];
                const float nm0 = fmaxf(m0, om0), nm1 = fmaxf(m1, om1);
                const float c0 = nm0 == -INFINITY ? 0.f : nm0, c1 = nm1 == -INFINITY ? 0.f : nm1;
                const float sa0 = exp2_sfu(m0 - c0), sb0 = exp2_sfu(om0 - c0);
                const float sa1 = exp2_sfu(m1 - c1), sb1 = exp2_sfu(om1 - c1);
#pragma unroll
                for (int n = 0; n < C::NO; ++n) {
                    o[n][0] = o[n][0] * sa0 + oth[(n * 4 + 0) * 32 + lane] * sb0;
                    o[n][1] = o[n][1] * sa0 + oth[(n * 4 + 1) * 32 + lane] * sb0;
                    o[n][2] = o[n][2] * sa1 + oth[(n * 4 + 2) * 32 + lane] * sb1;
                    o[n][3] = o[n][3] * sa1 + oth[(n * 4 + 3) * 32 + lane] * sb1;
                }
                l0 = l0 * sa0 + ol0 * sb0;
                l1 = l1 * sa1 + ol1 * sb1;
                m0 = nm0;
                m1 = nm1;
            }
        }
    }
    if (sp != 0) return;

    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
    const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const float lse2_0 = l0 > 0.f ? m0 + __log2f(l0) : -INFINITY;
    const float lse2_1 = l1 > 0.f ? m1 + __log2f(l1) : -INFINITY;
    if constexpr (REG4) {
        // o[4 c + i][0 / 1] is dim 32 c + 8 tq + i / + 4 + i (rows 0; 2 / 3 for row 1)
        float v0[C::NO * 2], v1[C::NO * 2];
#pragma unroll
        for (int c = 0; c < C4::CH4; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v0[8 * c + i] = o[4 * c + i][0] * inv0;
                v0[8 * c + 4 + i] = o[4 * c + i][1] * inv0;
                v1[8 * c + i] = o[4 * c + i][2] * inv1;
                v1[8 * c + 4 + i] = o[4 * c + i][3] * inv1;
            }
        if (it.out_base < 0) {
            __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(a.out);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (!(r ? has1 : has0)) continue;
                const int qt = r ? qt1 : qt0, row = r ? row1 : row0;
                const float *v = r ? v1 : v0;
                __nv_bfloat16 *dst = ob + (((size_t)l * a.nq + qt) * a.Hq + kvh * G + row % G) * D;
#pragma unroll
                for (int c = 0; c < C4::CH4; ++c)
                    *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * tq) =
                        make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                   pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
                if (a.lse && tq == 0)
                    a.lse[((size_t)l * a.nq + qt) * a.Hq + kvh * G + row % G] =
                        (r ? lse2_1 : lse2_0) * 0.6931471805599453f;
            }
        } else {
            const size_t rb = ((size_t)l * a.Hkv + kvh) * a.P + it.out_base;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (!(r ? has1 : has0)) continue;
                const int row = r ? row1 : row0;
                const float *v = r ? v1 : v0;
                float *dst = a.part_o + (rb + row) * D;
#pragma unroll
                for (int c = 0; c < C4::CH4; ++c) {
                    *reinterpret_cast<float4 *>(dst + 32 * c + 8 * tq) = make_float4(v[8 * c], v[8 * c + 1], v[8 * c + 2], v[8 * c + 3]);
                    *reinterpret_cast<float4 *>(dst + 32 * c + 8 * tq + 4) =
                        make_float4(v[8 * c + 4], v[8 * c + 5], v[8 * c + 6], v[8 * c + 7]);
                }
                if (tq == 0) a.part_lse[rb + row] = r ? lse2_1 : lse2_0;
            }
        }
        return;
    }
    if (it.out_base < 0) {
        __nv_bfloat16 *ob = static_cast<__nv_bfloat16 *>(a.out);
        if (has0) {
            __nv_bfloat16 *dst = ob + (((size_t)l * a.nq + qt0) * a.Hq + kvh * G + row0 % G) * D;
#pragma unroll
            for (int n = 0; n < C::NO; ++n)
                *reinterpret_cast<uint32_t *>(dst + n * 8 + 2 * tq) =
                    pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
            if (a.lse && tq == 0)
                a.lse[((size_t)l * a.nq + qt0) * a.Hq + kvh * G + row0 % G] = lse2_0 * 0.6931471805599453f;
        }
        if (has1) {
            __nv_bfloat16 *dst = ob + (((size_t)l * a.nq + qt1) * a.Hq + kvh * G + row1 % G) * D;
#pragma unroll
            for (int n = 0; n < C::NO; ++n)
                *reinterpret_cast<uint32_t *>(dst + n * 8 + 2 * tq) =
                    pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
            if (a.lse && tq == 0)
                a.lse[((size_t)l * a.nq + qt1) * a.Hq + kvh * G + row1 % G] = lse2_1 * 0.6931471805599453f;
        }
    } else {
        const size_t rb = ((size_t)l * a.Hkv + kvh) * a.P + it.out_base;
        if (has0) {
            float *dst = a.part_o + (rb + row0) * D;
#pragma unroll
            for (int n = 0; n < C::NO; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
            if (tq == 0) a.part_lse[rb + row0] = lse2_0;
        }
        if (has1) {
            float *dst = a.part_o + (rb + row1) * D;
#pragma unroll
            for (int n = 0; n < C::NO; ++n)
                *reinterpret_cast<float2 *>(dst + n * 8 + 2 * tq) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
            if (tq == 0) a.part_lse[rb + row1] = lse2_1;
        }
    }
}

template <int D, bool KV4, bool TREE>
__global__ void __launch_bounds__(kThreads, KCfg<D>::MIN_BLOCKS) attn_item_kernel(const AttnLaunch a) {
    using C = KCfg<D>;
    extern __shared__ __align__(128) unsigned char smem[];
    KvTile *s_tiles = reinterpret_cast<KvTile *>(smem + (KV4 ? KCfg4<D>::DESC_OFF : C::DESC_OFF));
    __shared__ int s_unit;
    // the plan (work items, tile descriptors, counters) was uploaded before
    // the kernel that may still be running; K/V, q and the tree masks are
    // read only after it has completed (with a.wait_first that kernel wrote
    // the plan as well: wait before anything)
    bool waited = false;
    if (a.wait_first) {
        griddep_wait();
        waited = true;
    }
    // units: the first is the block's index, each next one is claimed from
    // the counter during the last tile of the one before.  Beside the
    // tcgen05 kernel, whose CTAs hold SMs when this grid starts, every unit
    // is claimed (a block that starts late must not hold one of the longest
    // units; measured 1% on MCTS)
    if (threadIdx.x == 0) s_unit = a.n_tc_units > 0 ? atomicAdd(a.counter, 1) : (int)blockIdx.x;
    for (;;) {
        __syncthreads();
        const int unit = s_unit;
        if (unit >= a.n_units) {
            griddep_trigger();
            break;
        }
        // item-major order: items are sorted longest first, so the longest
        // units start first (over every layer and kv head) and the shortest
        // fill the tail; row tiles of one item, adjacent in the list, are
        // L * Hkv units apart, well within the units in flight, so they still
        // read their shared blocks from L2
        const int item_idx = unit / (a.L * a.Hkv);
        const int lk = unit % (a.L * a.Hkv);
        const int kvh = lk % a.Hkv, l = lk / a.Hkv;
        const WorkItem it = a.items[item_idx];
        const int ntile = it.tile_end - it.tile_begin;
        const int4 *src = reinterpret_cast<const int4 *>(a.tiles + it.tile_begin);
        int4 *dst = reinterpret_cast<int4 *>(s_tiles);
        for (int i = threadIdx.x; i < ntile * 2; i += kThreads) dst[i] = src[i];
        __syncthreads();
        const int rows = it.n_members * a.G;
        if (!waited) {
            griddep_wait();
            waited = true;
        }
        // The two-way split pays at head dim 128 (two CTAs per SM leave few
        // warps to hide latency); at head dim 64 the extra copy of the tile
        // loop costs more in instruction fetch than the split gains.
        if (rows <= 16) run_unit<D, 4, KV4, TREE>(a, it, l, kvh, ntile, smem, s_tiles, &s_unit);
        else if (D == 128 && rows <= 32) run_unit<D, 2, KV4, TREE>(a, it, l, kvh, ntile, smem, s_tiles, &s_unit);
        else run_unit<D, 1, KV4, TREE>(a, it, l, kvh, ntile, smem, s_tiles, &s_unit);
        __syncthreads();
    }
}

// One warp per (layer, query token, query head).  The first 32 entries are
// read lanes-over-entries (entry id and lse, one load round), so their
// weights sit in registers and the loads of their partial rows are all
// independent; entries past 32 (rare) are taken one by one.
template <int D>
__global__ void __launch_bounds__(kThreads, 8) merge_kernel(const AttnLaunch a) {
    griddep_wait();   // the partial rows come from the attention kernel before
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (kThreads / 32) + warp;
    const int qt = gw / a.Hq, h = gw % a.Hq, l = blockIdx.y;
    if (qt >= a.nq) return;
    const MergeDesc md = a.merge[qt];
    if (md.cnt == 0) return;
    constexpr int V = D / 32;   // values per lane
    const int kvh = h / a.G, g = h % a.G;
    const size_t rb = ((size_t)l * a.Hkv + kvh) * a.P + g;
    const int32_t *ent = a.entries + md.off;
    int e0 = 0;
    float l0 = -INFINITY;
    if (lane < md.cnt) {
        e0 = __ldg(ent + lane);
        l0 = a.part_lse[rb + e0];
    }
    float M = l0;
    for (int c = lane + 32; c < md.cnt; c += 32) M = fmaxf(M, a.part_lse[rb + __ldg(ent + c)]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mb = M == -INFINITY ? 0.f : M;
    const float w0 = lane < md.cnt ? exp2_sfu(l0 - Mb) : 0.f;
    float wsum = w0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    auto add = [&](size_t pr, float w) {
        const float *src = a.part_o + pr * D + lane * V;
        if constexpr (V == 2) {
            const float2 x = *reinterpret_cast<const float2 *>(src);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
        } else {
            const float4 x = *reinterpret_cast<const float4 *>(src);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
            acc[2] += w * x.z;
            acc[3] += w * x.w;
        }
    };
    const int n0 = md.cnt < 32 ? md.cnt : 32;
#pragma unroll 8
    for (int j = 0; j < n0; ++j)
        add(rb + __shfl_sync(0xffffffffu, e0, j), __shfl_sync(0xffffffffu, w0, j));
    for (int c = 32; c < md.cnt; ++c) {
        const size_t pr = rb + __ldg(ent + c);
        const float w = exp2_sfu(a.part_lse[pr] - Mb);
        wsum += w;
        add(pr, w);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                         (((size_t)l * a.nq + qt) * a.Hq + h) * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; v += 2)
        *reinterpret_cast<uint32_t *>(dst + v) = pack_bf16x2(acc[v] * inv, acc[v + 1] * inv);
    if (a.lse && lane == 0)
        a.lse[((size_t)l * a.nq + qt) * a.Hq + h] =
            (wsum > 0.f ? Mb + __log2f(wsum) : -INFINITY) * 0.6931471805599453f;
}

// One warp per (layer, query token, kv head).  The G query heads of a kv
// head share the query's merge entries, and one entry's partial rows for
// those heads are G * D contiguous floats, so the warp loads the entry list
// once and reads each entry as one coalesced block.  Lane p of a chunk of
// 32 / G entries holds the weight of (entry p / G, head p % G).
constexpr int kMergeWarps = 2;
constexpr int kMergeCached = 4;             // entry chunks kept in registers from the max pass
constexpr long long kMergeGroupMin = 2048;   // group warps over all layers

template <int D, int G>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_group_kernel(const AttnLaunch a) {
    griddep_wait();   // the partial rows come from the attention kernel before
    constexpr int NF4 = G * D / 4;        // float4s per entry
    constexpr int K = (NF4 + 31) / 32;    // float4s per lane
    constexpr int E = 32 / G;             // entries per chunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kMergeWarps + warp;
    const int qt = gw / a.Hkv, kvh = gw % a.Hkv, l = blockIdx.y;
    if (qt >= a.nq) return;
    const MergeDesc md = a.merge[qt];
    if (md.cnt == 0) return;
    const size_t rb = ((size_t)l * a.Hkv + kvh) * a.P;
    const int32_t *ent = a.entries + md.off;
    const int g = lane % G, c0 = lane / G;
    int ec[kMergeCached];
    float lc[kMergeCached];
#pragma unroll
    for (int i = 0; i < kMergeCached; ++i) {
        ec[i] = 0;
        if (c0 + i * E < md.cnt) ec[i] = __ldg(ent + c0 + i * E);
    }
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMergeCached; ++i) {
        lc[i] = -INFINITY;
        if (c0 + i * E < md.cnt) lc[i] = a.part_lse[rb + ec[i] + g];
        M = fmaxf(M, lc[i]);
    }
    for (int c = c0 + kMergeCached * E; c < md.cnt; c += E) M = fmaxf(M, a.part_lse[rb + __ldg(ent + c) + g]);
#pragma unroll
    for (int off = 16; off >= G; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mb = M == -INFINITY ? 0.f : M;   // lane's head g

    float4 acc[K];
#pragma unroll
    for (int k = 0; k < K; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    auto chunk = [&](int base, int e, float lv) {
        const float w = exp2_sfu(lv - Mb);   // 0 for pairs past the end
        wsum += w;
        const int n = min(E, md.cnt - base);
#pragma unroll 4
        for (int j = 0; j < n; ++j) {
            const int ej = __shfl_sync(0xffffffffu, e, j * G);
            const float4 *src = reinterpret_cast<const float4 *>(a.part_o + (rb + ej) * D);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const int f = lane + 32 * k;
                const float wj = __shfl_sync(0xffffffffu, w, j * G + f / (D / 4));
                if (NF4 % 32 == 0 || f < NF4) {
                    const float4 x = src[f];
                    acc[k].x += wj * x.x;
                    acc[k].y += wj * x.y;
                    acc[k].z += wj * x.z;
                    acc[k].w += wj * x.w;
                }
            }
        }
    };
#pragma unroll
    for (int i = 0; i < kMergeCached; ++i)
        if (i * E < md.cnt) chunk(i * E, ec[i], lc[i]);
    for (int base = kMergeCached * E; base < md.cnt; base += E) {
        int e = 0;
        float lv = -INFINITY;
        if (base + c0 < md.cnt) {
            e = __ldg(ent + base + c0);
            lv = a.part_lse[rb + e + g];
        }
        chunk(base, e, lv);
    }
#pragma unroll
    for (int off = 16; off >= G; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);

    const size_t ob = ((size_t)l * a.nq + qt) * a.Hq + (size_t)kvh * G;   // first output row
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + ob * D;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int f = lane + 32 * k;
        const float ws = __shfl_sync(0xffffffffu, wsum, f / (D / 4));
        const float inv = ws > 0.f ? 1.f / ws : 0.f;
        if (NF4 % 32 == 0 || f < NF4) {
            uint2 v;
            v.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
            v.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
            *reinterpret_cast<uint2 *>(dst + 4 * f) = v;
        }
    }
    if (a.lse && lane < G)
        a.lse[ob + lane] = (wsum > 0.f ? Mb + __log2f(wsum) : -INFINITY) * 0.6931471805599453f;
}

// KVP_MERGE=group / =head in the environment forces one merge kernel (tests,
// ablations); by default the grouped kernel runs when there are many groups.
int merge_mode() {
    static int mode = [] {
        const char *e = std::getenv("KVP_MERGE");
        if (e && std::strcmp(e, "group") == 0) return 1;
        if (e && std::strcmp(e, "head") == 0) return 2;
        return 0;
    }();
    return mode;
}

// Launches `kernel` with programmatic stream serialisation: it may begin
// while the previous kernel in the stream finishes (it waits with
// griddep_wait() before reading that kernel's results).
template <typename Kernel>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const AttnLaunch &a) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int D>
void launch_merge(const AttnLaunch &a, cudaStream_t stream) {
    const long long groups = (long long)a.nq * a.Hkv;
    dim3 grid((unsigned)((groups + kMergeWarps - 1) / kMergeWarps), a.L);
    // with few groups, one warp per head keeps more loads in flight
    const int mode = merge_mode();
    const bool grouped = mode == 1 || (mode == 0 && groups * a.L >= kMergeGroupMin);
    switch (grouped ? a.G : 0) {
        case 1: launch_pdl(merge_group_kernel<D, 1>, grid, dim3(32 * kMergeWarps), 0, stream, a); return;
        case 2: launch_pdl(merge_group_kernel<D, 2>, grid, dim3(32 * kMergeWarps), 0, stream, a); return;
        case 4: launch_pdl(merge_group_kernel<D, 4>, grid, dim3(32 * kMergeWarps), 0, stream, a); return;
        case 8: launch_pdl(merge_group_kernel<D, 8>, grid, dim3(32 * kMergeWarps), 0, stream, a); return;
        case 16: launch_pdl(merge_group_kernel<D, 16>, grid, dim3(32 * kMergeWarps), 0, stream, a); return;
        default: break;
    }
    const long long warps = (long long)a.nq * a.Hq;
    dim3 g1((unsigned)((warps + kThreads / 32 - 1) / (kThreads / 32)), a.L);
    launch_pdl(merge_kernel<D>, g1, dim3(kThreads), 0, stream, a);
}

struct Occupancy {
    int sms = 0, per_sm = 0;
    bool ok = false;
};

// Per device: the kernel's shared-memory attribute is set and its
// occupancy queried once for each device that runs it.
template <int D, bool KV4 = false, bool TREE = false>
Occupancy &occupancy() {
    static Occupancy occ[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    // no usable device (host-only planning): the configured occupancy
    static Occupancy none{152, KCfg<D>::MIN_BLOCKS, false};
    const int dev = current_device();
    if (dev < 0) return none;
    std::call_once(once[dev], [dev] {
        using C = KCfg<D>;
        Occupancy &o = occ[dev];
        o.per_sm = C::MIN_BLOCKS;
        o.sms = device_sm_count();
        const int smem_bytes = KV4 ? KCfg4<D>::SMEM : C::SMEM;
        if (cudaFuncSetAttribute(attn_item_kernel<D, KV4, TREE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes) != cudaSuccess)
            return;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_item_kernel<D, KV4, TREE>, kThreads, smem_bytes) ==
                cudaSuccess && n > 0)
            o.per_sm = n;
        o.ok = true;
    });
    return occ[dev];
}

// A second stream per (thread, device) so that the tcgen05 and mma.sync
// kernels of one call can share the GPU: the caller's stream forks to it and
// joins back.  Created on first use, with that device current.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    int state = 0;   // 0: not tried, 1: ready, -1: creation failed
    bool ensure() {
        if (state == 0)
            state = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess &&
                            cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess &&
                            cudaEventCreateWithFlags(&join, cudaEventDisableTiming) == cudaSuccess
                        ? 1
                        : -1;
        return state == 1;
    }
};

template <int D>
cudaError_t launch_d(const AttnLaunch &a, cudaStream_t stream, cudaEvent_t before, cudaEvent_t after) {
    using C = KCfg<D>;
    Occupancy &occ = occupancy<D>();
    if (!occ.ok) return cudaErrorInvalidDevice;
    if (before && cudaEventRecord(before, stream) != cudaSuccess) return cudaErrorInvalidResourceHandle;
    if (a.tree_mask && a.nq > 0) {
        tree_mask_kernel<<<(a.nq + 255) / 256, 256, 0, stream>>>(a.tree_parent, a.nq, a.n_draft, a.tree_mask,
                                                                 a.err);
        count_launch();
        cudaError_t e0 = cudaGetLastError();
        if (e0 != cudaSuccess) return e0;
    }
    const bool both = a.n_tc_units > 0 && a.n_units > 0;
    thread_local SideStream sides[kMaxDevices];
    SideStream &side = sides[current_device()];   // occ.ok implies a valid device id
    const bool fork = both && side.ensure();
    cudaStream_t mma_stream = stream;
    if (fork) {
        // fork: the mma.sync kernel runs beside the tcgen05 kernel, which then
        // takes one CTA per SM to leave room for it
        if (cudaEventRecord(side.fork, stream) != cudaSuccess ||
            cudaStreamWaitEvent(side.s, side.fork, 0) != cudaSuccess)
            return cudaErrorUnknown;
        mma_stream = side.s;
    }
    cudaError_t e = launch_attention_tc(a, stream, fork ? 1 : 0);
    if (e != cudaSuccess) return e;
    if (a.n_units > 0 && a.kv4) {
        Occupancy &o4 = occupancy<D, true>();
        if (!o4.ok) return cudaErrorInvalidDevice;
        const int grid = a.n_units < o4.sms * o4.per_sm ? a.n_units : o4.sms * o4.per_sm;
        e = launch_pdl(attn_item_kernel<D, true, false>, dim3(grid), dim3(kThreads), KCfg4<D>::SMEM, mma_stream, a);
        count_launch();
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else if (a.n_units > 0 && a.tree_mask) {
        Occupancy &ot = occupancy<D, false, true>();
        if (!ot.ok) return cudaErrorInvalidDevice;
        const int grid = a.n_units < ot.sms * ot.per_sm ? a.n_units : ot.sms * ot.per_sm;
        e = launch_pdl(attn_item_kernel<D, false, true>, dim3(grid), dim3(kThreads), C::SMEM, mma_stream, a);
        count_launch();
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else if (a.n_units > 0) {
        const int grid = a.n_units < occ.sms * occ.per_sm ? a.n_units : occ.sms * occ.per_sm;
        e = launch_pdl(attn_item_kernel<D, false, false>, dim3(grid), dim3(kThreads), C::SMEM, mma_stream, a);
        count_launch();
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (mma_stream != stream) {
        if (cudaEventRecord(side.join, mma_stream) != cudaSuccess ||
            cudaStreamWaitEvent(stream, side.join, 0) != cudaSuccess)
            return cudaErrorUnknown;
    }
    if (after && cudaEventRecord(after, stream) != cudaSuccess) return cudaErrorInvalidResourceHandle;
    if (a.P == 0) return cudaSuccess;
    launch_merge<D>(a, stream);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

int attention_ctas_per_sm(int D) {
    return D == 64 ? occupancy<64>().per_sm : occupancy<128>().per_sm;
}

cudaError_t launch_attention(const AttnLaunch &a, cudaStream_t stream, cudaEvent_t before,
                             cudaEvent_t after) {
    if (a.D == 64) return launch_d<64>(a, stream, before, after);
    if (a.D == 128) return launch_d<128>(a, stream, before, after);
    return cudaErrorInvalidValue;
}

}  // namespace kvp
