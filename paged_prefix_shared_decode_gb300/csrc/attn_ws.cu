// Paged attention on the 5th-generation tensor cores (tcgen05 + TMA,
// sm_103a) for work items with more than 32 query rows: shared-prefix
// segments read by many sequences, MCTS tree levels and draft-tree
// verification.
//
// Warp-specialised persistent CTA (13 warps), one per SM:
//   warps 0-3   producers: warp 0 claims work units from an atomic counter and
//               stages their 64-token tile descriptors (physical block ids) in
//               shared memory; all four fill a ring of K/V stages -- with
//               TMA (cp.async.bulk.tensor, one box per block and 64-column
//               slab, 128-byte swizzle) for whole tiles when d = 128 or blocks
//               hold 32+ tokens, otherwise (and for ragged tiles) with
//               cp.async (16-byte chunks, same swizzle, zero fill);
//   warp 4      MMA issuer (one thread): S = Q K^T (M=128, N=64, K=d) into a
//               double-buffered TMEM S, then O += P V (M=128, N=d, K=64) into
//               TMEM O; completion is signalled with tcgen05.commit;
//   warps 5-12  softmax: two threads per query row, 32 score columns each;
//               load S from TMEM, mask (tile end, member interval, draft-tree
//               ancestors), exchange the row max, form P = 2^(s - m) in bf16
//               (shared memory, double-buffered), and at the end scale O by
//               1/l and write out / lse or a partial row.  The running max m is
//               only raised when a tile's max exceeds it by more than 8
//               (factor 256); the row of O in TMEM is then rescaled in place.
// Roles hand off through mbarriers: unit slots (2), K/V stages, S buffers,
// P buffers, Q and O.  Every wait is bounded; on a timeout the CTA sets bit 4
// of the workspace error word, every role leaves its loop, and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kvp_internal.h"

namespace kvp {
namespace {

constexpr int kProdWarps = 4;        // warps 0-3: K/V producers
constexpr int kMmaWarp = 4;          // warp 4: MMA issuer
constexpr int kSoftWarp0 = 5;        // warps 5-12: softmax
constexpr int kWsThreads = 416;      // 13 warps
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kSoftThreads = 256;
constexpr int kTmemCols = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}
__device__ __forceinline__ float exp2_sfu(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---- fences and barriers
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Named barrier (ids 1-4) over the two softmax warps that serve the same 32
// query rows, with an OR reduction so both take the same branch.  The id is
// an immediate so the kernel reserves only barriers 0-4.
template <int ID>
__device__ __forceinline__ bool bar_or_id(bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred p, %2, 64, q;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(ID)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool pair_bar_or(int quarter, bool v) {
    switch (quarter) {
        case 0: return bar_or_id<1>(v);
        case 1: return bar_or_id<2>(v);
        case 2: return bar_or_id<3>(v);
        default: return bar_or_id<4>(v);
    }
}

// ---- tcgen05
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}
// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, A K-major,
// B K-major (or MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
        : "memory");
}

#define KVP_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                  "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define KVP_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                  "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : KVP_R8(0), KVP_R8(8), KVP_R8(16), KVP_R8(24)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        KVP_W8(0), KVP_W8(8), KVP_W8(16), KVP_W8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

template <int D>
struct WsCfg {
    static constexpr int CH = D / 8;
    static constexpr int Q_BYTES = 128 * D * 2;
    static constexpr int TILE_BYTES = kTileTokens * D * 2;
    static constexpr int NSTAGE = D == 64 ? 6 : 4;
    static constexpr int MIN_BLOCKS = 1;
    static constexpr int P_BYTES = 128 * kTileTokens * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int STAGE_OFF = Q_OFF + Q_BYTES;
    static constexpr int P_OFF = STAGE_OFF + NSTAGE * 2 * TILE_BYTES;
    static constexpr int DESC_OFF = P_OFF + 2 * P_BYTES;                      // [2][kMaxItemTiles]
    static constexpr int XCH_OFF = DESC_OFF + 2 * kMaxItemTiles * (int)sizeof(KvTile);  // [2][2][128]
    static constexpr int LX_OFF = XCH_OFF + 2 * 2 * 128 * 4;                 // [2][128]
    static constexpr int UNIT_OFF = LX_OFF + 2 * 128 * 4;                    // [2] ints
    static constexpr int BAR_OFF = UNIT_OFF + 16;
    // barrier indices
    static constexpr int B_UNIT_FULL = 0, B_UNIT_EMPTY = 2, B_KV_FULL = 4, B_KV_EMPTY = 4 + NSTAGE,
                         B_S_FULL = 4 + 2 * NSTAGE, B_S_EMPTY = B_S_FULL + 2, B_P_FULL = B_S_EMPTY + 2,
                         B_P_EMPTY = B_P_FULL + 2, B_Q_FULL = B_P_EMPTY + 2, B_Q_EMPTY = B_Q_FULL + 1,
                         B_O_FULL = B_Q_EMPTY + 1, B_O_EMPTY = B_O_FULL + 1, N_BARS = B_O_EMPTY + 1;
    static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;                    // tmem addr, abort
    static constexpr int SMEM = MISC_OFF + 16 + 1024;   // + slack to align the base to 1024
    static constexpr int S_COL = 0, O_COL = 128, HALF_D = D / 2;
};

template <int ROWS_IN_TILE>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((c >> 3) * ROWS_IN_TILE * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct WsParams {
    int32_t box_rows;   // TMA box height: min(block size, 64)
};

template <int D>
__global__ void __launch_bounds__(kWsThreads, WsCfg<D>::MIN_BLOCKS)
    attn_ws_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const AttnLaunch a, const WsParams wp) {
    using C = WsCfg<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    KvTile *s_desc = reinterpret_cast<KvTile *>(smem + C::DESC_OFF);
    float *s_xch = reinterpret_cast<float *>(smem + C::XCH_OFF);
    float *s_lx = reinterpret_cast<float *>(smem + C::LX_OFF);
    volatile int *s_unit = reinterpret_cast<volatile int *>(smem + C::UNIT_OFF);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    const uint32_t bar0 = saddr(smem + C::BAR_OFF);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(bar(C::B_UNIT_FULL), 1);
        mbar_init(bar(C::B_UNIT_FULL + 1), 1);
        // unit slot free: MMA thread + softmax threads + producer warps 1-3
        mbar_init(bar(C::B_UNIT_EMPTY), 1 + kSoftThreads + (kProdWarps - 1));
        mbar_init(bar(C::B_UNIT_EMPTY + 1), 1 + kSoftThreads + (kProdWarps - 1));
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(bar(C::B_KV_FULL + s), kProdThreads);
            mbar_init(bar(C::B_KV_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_S_FULL + s), 1);
            mbar_init(bar(C::B_S_EMPTY + s), kSoftThreads);
            mbar_init(bar(C::B_P_FULL + s), kSoftThreads);
            mbar_init(bar(C::B_P_EMPTY + s), 1);
        }
        mbar_init(bar(C::B_Q_FULL), kSoftThreads);
        mbar_init(bar(C::B_Q_EMPTY), 1);
        mbar_init(bar(C::B_O_FULL), 1);
        mbar_init(bar(C::B_O_EMPTY), kSoftThreads);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         saddr(s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *s_tmem;

    // bounded wait; on a timeout the whole CTA aborts
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        for (uint32_t i = 0; i < kWaitLimit; ++i) {
            if (mbar_try_wait(b, parity)) return true;
            if ((i & 1023) == 1023 && *s_abort) return false;
        }
        *s_abort = 1;
        atomicOr(a.err, 4);
        return false;
    };

    const int n_items = a.n_tc_units / (a.L * a.Hkv);
    const uint32_t q_smem = saddr(smem + C::Q_OFF);
    const uint32_t stage_smem = saddr(smem + C::STAGE_OFF);
    const uint32_t p_smem = saddr(smem + C::P_OFF);
    const int bs_log2 = a.bs_log2, bs = 1 << bs_log2;
    const size_t head_stride = (size_t)D << bs_log2;
    const size_t block_stride = (size_t)a.Hkv * head_stride;

    if (warp < kProdWarps) {
        // ------------------------------------------------------------ producers
        const __nv_bfloat16 *kpool = static_cast<const __nv_bfloat16 *>(a.k_pool);
        const __nv_bfloat16 *vpool = static_cast<const __nv_bfloat16 *>(a.v_pool);
        // TMA for whole tiles when a box is at least 4 KB (d = 128, or blocks
        // of 32+ tokens); for 2 KB boxes the per-box cost of the TMA unit
        // dominates and the 128 producer threads copy 16-byte chunks with
        // cp.async instead (measured on both workloads); each thread's copies
        // arrive on the stage's barrier when they land
        // (cp.async.mbarrier.arrive.noinc), and the MMA thread fences the async
        // proxy after acquiring the stage.  Warp 0 claims units and stages
        // their descriptors; warps 1-3 follow through the unit slots.
        const bool use_tma = wp.box_rows >= 32 || D == 128;
        const int pt = warp * 32 + lane;   // producer thread 0..127
        if (lane == 0 && use_tma) {
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
        }
        // lane 0 waits (acquire) and the warp follows it (__syncwarp orders memory)
        auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
            int ok = 1;
            if (lane == 0) ok = wait(b, parity) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            return ok != 0;
        };
        uint32_t g = 0;        // tiles issued
        for (int uc = 0;; ++uc) {
            const int slot = uc & 1;
            int unit = -1;
            if (warp == 0) {
                bool ok = wait_warp(bar(C::B_UNIT_EMPTY + slot), ((uc >> 1) & 1) ^ 1);
                if (lane == 0) unit = atomicAdd(a.tc_counter, 1);
                unit = __shfl_sync(0xffffffffu, unit, 0);
                const bool done = !ok || unit >= a.n_tc_units || __shfl_sync(0xffffffffu, *s_abort, 0);
                if (!done) {
                    const WorkItem it = a.tc_items[unit % n_items];
                    const int ntile = it.tile_end - it.tile_begin;
                    const int4 *src = reinterpret_cast<const int4 *>(a.tiles + it.tile_begin);
                    int4 *dst = reinterpret_cast<int4 *>(s_desc + slot * kMaxItemTiles);
                    for (int i = lane; i < ntile * 2; i += 32) dst[i] = src[i];
                }
                if (lane == 0) s_unit[slot] = done ? -1 : unit;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_UNIT_FULL + slot));
                if (done) break;
            } else {
                const bool ok = wait_warp(bar(C::B_UNIT_FULL + slot), (uc >> 1) & 1);
                unit = ok ? s_unit[slot] : -1;
                if (unit < 0) break;
            }
            const int item_idx = unit % n_items;
            const int lk = unit / n_items;
            const int kvh = lk % a.Hkv, l = lk / a.Hkv;
            const WorkItem it = a.tc_items[item_idx];
            const int ntile = it.tile_end - it.tile_begin;
            const size_t layer_base = (size_t)l * a.NB * block_stride + (size_t)kvh * head_stride;
            const int row_base_lh = (l * a.NB) * a.Hkv + kvh;   // row of block b = (row_base_lh + b*Hkv) * bs
            const KvTile *tiles = s_desc + slot * kMaxItemTiles;
            for (int t = 0; t < ntile; ++t, ++g) {
                const int stage = g % C::NSTAGE;
                if (!wait_warp(bar(C::B_KV_EMPTY + stage), ((g / C::NSTAGE) & 1) ^ 1)) break;
                const KvTile &kt = tiles[t];
                const int ntok = kt.ntok_flags & 0xFFFF;
                const uint32_t dK = stage_smem + stage * 2 * C::TILE_BYTES;
                const uint32_t dV = dK + C::TILE_BYTES;
                const uint32_t fb = bar(C::B_KV_FULL + stage);
                if (use_tma && ntok == kTileTokens && (kt.tok0 & (wp.box_rows - 1)) == 0) {
                    // the tile's (block, 64-column slab) boxes are spread over
                    // lane 0 of the four producer warps: one issuing thread
                    // cannot keep enough small boxes in flight
                    constexpr int NSLAB = D / 64;
                    const int npair = (kTileTokens / wp.box_rows) * NSLAB;
                    if (lane == 0) {
                        const int mine = (npair - warp + kProdWarps - 1) / kProdWarps;
                        mbar_expect_tx(fb, (uint32_t)(mine * 2 * wp.box_rows * 128));
                        const int yoff = bs > kTileTokens ? (kt.tok0 & (bs - 1)) : 0;
                        for (int pr = warp; pr < npair; pr += kProdWarps) {
                            const int k = pr / NSLAB, cb = pr % NSLAB;
                            const int y = (row_base_lh + kt.blk[k] * a.Hkv) * bs + yoff;
                            const uint32_t off = cb * (kTileTokens * 128) + k * wp.box_rows * 128;
                            tma_load_2d(dK + off, &kmap, cb * 64, y, fb);
                            tma_load_2d(dV + off, &vmap, cb * 64, y, fb);
                        }
                    } else {
                        mbar_arrive(fb);
                    }
                    continue;
                }
                const int jb = kt.tok0 >> bs_log2;
#pragma unroll
                for (int i = 0; i < kTileTokens * C::CH / kProdThreads; ++i) {
                    const int x = pt + i * kProdThreads;
                    const int tok = x / C::CH, c = x % C::CH;
                    const uint32_t off = swz<kTileTokens>(tok, c);
                    const __nv_bfloat16 *sk = kpool, *sv = vpool;
                    int bytes = 0;
                    if (tok < ntok) {
                        const int pos = kt.tok0 + tok;
                        const int blk = kt.blk[(pos >> bs_log2) - jb];
                        if ((unsigned)blk < (unsigned)a.NB) {
                            const size_t e = layer_base + (size_t)blk * block_stride +
                                             (size_t)(pos & (bs - 1)) * D + c * 8;
                            sk = kpool + e;
                            sv = vpool + e;
                            bytes = 16;
                        } else if (c == 0) {
                            atomicOr(a.err, 1);
                        }
                    }
                    cp_async16(dK + off, sk, bytes);
                    cp_async16(dV + off, sv, bytes);
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(fb) : "memory");
            }
            if (warp != 0 && lane == 0) mbar_arrive(bar(C::B_UNIT_EMPTY + slot));
            if (__shfl_sync(0xffffffffu, *s_abort, 0)) {
                // let the consumers see the end
                if (warp == 0 && lane == 0) {
                    const int s2 = (uc + 1) & 1;
                    s_unit[s2] = -1;
                    mbar_arrive(bar(C::B_UNIT_FULL + s2));
                }
                break;
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, kTileTokens, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
            uint32_t g = 0, ns = 0, np = 0;
            for (int uc = 0;; ++uc) {
                const int slot = uc & 1;
                if (!wait(bar(C::B_UNIT_FULL + slot), (uc >> 1) & 1)) break;
                const int unit = s_unit[slot];
                if (unit < 0) break;
                const WorkItem it = a.tc_items[unit % n_items];
                const int ntile = it.tile_end - it.tile_begin;
                if (!wait(bar(C::B_Q_FULL), uc & 1)) break;
                tc_after();
                const uint32_t g0 = g;
                auto do_pv = [&](int tt) -> bool {
                    const uint32_t pb = np & 1;
                    if (!wait(bar(C::B_P_FULL + pb), (np >> 1) & 1)) return false;
                    if (tt == 0 && !wait(bar(C::B_O_EMPTY), (uc & 1) ^ 1)) return false;
                    tc_after();
                    const int stage = (g0 + tt) % C::NSTAGE;
                    const uint32_t vst = stage_smem + stage * 2 * C::TILE_BYTES + C::TILE_BYTES;
                    const uint32_t pbuf = p_smem + pb * C::P_BYTES;
#pragma unroll
                    for (int k = 0; k < kTileTokens / 16; ++k) {
                        const uint64_t da = sdesc(pbuf + k * 32, 16, 1024);
                        const uint64_t db = sdesc(vst + k * (16 * 128), kTileTokens * 128, 1024);
                        umma(tmem + C::O_COL, da, db, IDESC_PV, (tt == 0 && k == 0) ? 0u : 1u);
                    }
                    umma_commit(bar(C::B_P_EMPTY + pb));
                    umma_commit(bar(C::B_KV_EMPTY + stage));
                    np += 1;
                    return true;
                };
                bool ok = true;
                for (int t = 0; t < ntile && ok; ++t, ++g) {
                    const int stage = g % C::NSTAGE;
                    if (!wait(bar(C::B_KV_FULL + stage), (g / C::NSTAGE) & 1)) { ok = false; break; }
                    // stages filled by cp.async were written through the generic proxy
                    fence_async_smem();
                    const uint32_t sb = ns & 1;
                    if (!wait(bar(C::B_S_EMPTY + sb), ((ns >> 1) & 1) ^ 1)) { ok = false; break; }
                    tc_after();
                    const uint32_t kst = stage_smem + stage * 2 * C::TILE_BYTES;
                    const uint32_t d_tm = tmem + C::S_COL + sb * kTileTokens;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t koff = (uint32_t)(k & 3) * 32;
                        const uint64_t da = sdesc(q_smem + (k >> 2) * (128 * 128) + koff, 16, 1024);
                        const uint64_t db = sdesc(kst + (k >> 2) * (kTileTokens * 128) + koff, 16, 1024);
                        umma(d_tm, da, db, IDESC_S, k > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(C::B_S_FULL + sb));
                    ns += 1;
                    if (t == ntile - 1) umma_commit(bar(C::B_Q_EMPTY));
                    if (t > 0 && !do_pv(t - 1)) { ok = false; break; }
                }
                if (!ok) break;
                if (ntile == 0) umma_commit(bar(C::B_Q_EMPTY));
                if (ntile > 0 && !do_pv(ntile - 1)) break;
                umma_commit(bar(C::B_O_FULL));
                mbar_arrive(bar(C::B_UNIT_EMPTY + slot));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3, half = (warp - kSoftWarp0) >> 2;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(a.q);
        uint32_t ns = 0, np = 0;
        for (int uc = 0;; ++uc) {
            const int slot = uc & 1;
            bool ok = wait(bar(C::B_UNIT_FULL + slot), (uc >> 1) & 1);
            const int unit = ok ? s_unit[slot] : -1;
            if (pair_bar_or(quarter, !ok || unit < 0 || *s_abort)) break;
            const int item_idx = unit % n_items;
            const int lk = unit / n_items;
            const int kvh = lk % a.Hkv, l = lk / a.Hkv;
            const WorkItem it = a.tc_items[item_idx];
            const int ntile = it.tile_end - it.tile_begin;
            const KvTile *tiles = s_desc + slot * kMaxItemTiles;
            const int G = a.G;
            const int rows = it.n_members * G;
            const bool has = r < rows;
            const int mem = r / G;
            int qt = 0;
            if (has) qt = __ldg(a.members + it.member_off + mem);
            uint64_t tmask = ~0ull;
            if (has && a.tree_mask) tmask = a.tree_mask[qt];
            tmask >>= 32 * half;

            // Q: half a row per thread (zero for padding rows), once the previous
            // unit's S MMAs are done with the buffer
            ok = wait(bar(C::B_Q_EMPTY), (uc & 1) ^ 1);
            {
                const __nv_bfloat16 *qrow =
                    has ? qb + (((size_t)l * a.nq + qt) * a.Hq + kvh * G + r % G) * D : qb;
#pragma unroll
                for (int c = half * (C::CH / 2); c < (half + 1) * (C::CH / 2); ++c)
                    cp_async16(q_smem + swz<128>(r, c), qrow + c * 8, has ? 16 : 0);
                cp_async_wait_all();
                fence_async_smem();
                mbar_arrive(bar(C::B_Q_FULL));
            }

            float m_used = -INFINITY, lsum = 0.f;
            bool aborted = false;
            for (int t = 0; t < ntile; ++t) {
                const KvTile &kt = tiles[t];
                const int ntok = kt.ntok_flags & 0xFFFF;
                const bool tree = (kt.ntok_flags >> 16) & kTileTree;
                const int mlo = kt.members & 0xFFFF, mhi = kt.members >> 16;
                const bool in = has && mem >= mlo && mem < mhi;
                const int nvalid = in ? ntok - 32 * half : 0;
                const uint32_t sb = ns & 1;
                ok = wait(bar(C::B_S_FULL + sb), (ns >> 1) & 1) && ok;
                tc_after();
                // raw scores of this thread's 32 columns; masked ones are -inf
                float s[32];
                {
                    uint32_t rr[32];
                    tmem_ld32(tmem + lane_base + C::S_COL + sb * kTileTokens + 32 * half, rr);
                    tmem_wait_ld();
                    tc_before();
                    mbar_arrive(bar(C::B_S_EMPTY + sb));
                    if (nvalid >= 32 && !tree) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(rr[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            bool v = j < nvalid;
                            if (tree) v = v && ((tmask >> j) & 1ull);
                            s[j] = v ? __uint_as_float(rr[j]) : -INFINITY;
                        }
                    }
                }
                ns += 1;
                float mq[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
                for (int j = 4; j < 32; j += 4) {
                    mq[0] = fmaxf(mq[0], s[j]);
                    mq[1] = fmaxf(mq[1], s[j + 1]);
                    mq[2] = fmaxf(mq[2], s[j + 2]);
                    mq[3] = fmaxf(mq[3], s[j + 3]);
                }
                // scale > 0: max of scaled scores = scale * max of raw scores
                float *xb = s_xch + (t & 1) * 256;
                xb[half * 128 + r] = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.scale_log2;
                if (pair_bar_or(quarter, !ok || *s_abort)) { aborted = true; break; }
                const float mx = fmaxf(xb[r], xb[128 + r]);
                const float m_new = fmaxf(m_used, mx);
                const bool resc = m_used != -INFINITY && m_new > m_used + 8.f;
                if (__any_sync(0xffffffffu, resc)) {
                    // O must be complete (P V of tile t-1 done) before it is rescaled
                    if (t > 0) ok = wait(bar(C::B_P_EMPTY + ((np - 1) & 1)), ((np - 1) >> 1) & 1) && ok;
                    tc_after();
                    const float f = resc ? exp2_sfu(m_used - m_new) : 1.f;
#pragma unroll
                    for (int c0 = 0; c0 < C::HALF_D; c0 += 32) {
                        uint32_t rr[32];
                        const uint32_t oa = tmem + lane_base + C::O_COL + half * C::HALF_D + c0;
                        tmem_ld32(oa, rr);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * f);
                        tmem_st32(oa, rr);
                    }
                    tmem_wait_st();
                    lsum *= f;
                    if (resc) m_used = m_new;
                }
                if (m_used == -INFINITY) m_used = m_new;
                uint32_t pk[16];
                float rq[4] = {0.f, 0.f, 0.f, 0.f};
                if (m_used == -INFINITY || nvalid <= 0) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) pk[j] = 0u;
                } else {
                    // p = 2^(s * scale - m): one FFMA and one SFU op per score
                    const float sc = a.scale_log2, nm = -m_used;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float e0 = exp2_sfu(fmaf(s[j], sc, nm));
                        const float e1 = exp2_sfu(fmaf(s[j + 1], sc, nm));
                        rq[(j >> 1) & 3] += e0 + e1;
                        pk[j / 2] = pack_bf16x2(e0, e1);
                    }
                }
                lsum += (rq[0] + rq[1]) + (rq[2] + rq[3]);
                // P buffer np & 1 was last read by the P V two tiles back
                const uint32_t pb = np & 1;
                ok = wait(bar(C::B_P_EMPTY + pb), ((np >> 1) & 1) ^ 1) && ok;
                {
                    unsigned char *prow = smem + C::P_OFF + pb * C::P_BYTES;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                        *reinterpret_cast<uint4 *>(prow + swz<128>(r, 4 * half + c)) = v;
                    }
                }
                fence_async_smem();
                tc_before();
                mbar_arrive(bar(C::B_P_FULL + pb));
                np += 1;
            }
            if (aborted) break;
            // epilogue: wait for the last P V, combine the row sums, write
            ok = wait(bar(C::B_O_FULL), uc & 1) && ok;
            tc_after();
            s_lx[half * 128 + r] = lsum;
            if (pair_bar_or(quarter, !ok || *s_abort)) break;
            const float ltot = s_lx[r] + s_lx[128 + r];
            const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
            const float lse2 = ltot > 0.f ? m_used + __log2f(ltot) : -INFINITY;
#pragma unroll
            for (int c0 = 0; c0 < C::HALF_D; c0 += 32) {
                uint32_t rr[32];
                const int col = half * C::HALF_D + c0;
                tmem_ld32(tmem + lane_base + C::O_COL + col, rr);
                tmem_wait_ld();
                if (!has || ntile == 0) continue;
                if (it.out_base < 0) {
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                         (((size_t)l * a.nq + qt) * a.Hq + kvh * G + r % G) * D + col;
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(rr[j + 4]) * inv, __uint_as_float(rr[j + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(rr[j + 6]) * inv, __uint_as_float(rr[j + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + j) = v;
                    }
                } else {
                    float *dst = a.part_o + (((size_t)l * a.Hkv + kvh) * a.P + it.out_base + r) * D + col;
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(dst + j) =
                            make_float4(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv,
                                        __uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
                }
            }
            if (has && ntile > 0 && half == 0) {
                if (it.out_base < 0) {
                    if (a.lse) a.lse[((size_t)l * a.nq + qt) * a.Hq + kvh * G + r % G] = lse2 * 0.6931471805599453f;
                } else {
                    a.part_lse[((size_t)l * a.Hkv + kvh) * a.P + it.out_base + r] = lse2;
                }
            }
            tc_before();
            mbar_arrive(bar(C::B_O_EMPTY));
            mbar_arrive(bar(C::B_UNIT_EMPTY + slot));
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of a pool: rows = L*NB*Hkv*bs token rows of d bf16; box = 64
// columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *pool, int D, long long rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct WsOcc {
    int sms = 0;
    bool ok = false;
};

template <int D>
WsOcc &ws_occ() {
    static WsOcc occ;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return;
        if (cudaFuncSetAttribute(attn_ws_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 WsCfg<D>::SMEM) != cudaSuccess)
            return;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
        occ.sms = sms;
        occ.ok = true;
    });
    return occ;
}

template <int D>
cudaError_t launch_ws_d(const AttnLaunch &a, cudaStream_t stream, int ctas_per_sm) {
    WsOcc &occ = ws_occ<D>();
    if (!occ.ok) return cudaErrorInvalidDevice;
    const int bs = 1 << a.bs_log2;
    const int box_rows = bs < kTileTokens ? bs : kTileTokens;
    const long long rows = (long long)a.L * a.NB * a.Hkv * bs;
    alignas(64) CUtensorMap km, vm;
    if (!make_map(&km, a.k_pool, D, rows, box_rows) || !make_map(&vm, a.v_pool, D, rows, box_rows))
        return cudaErrorInvalidValue;
    WsParams wp{box_rows};
    const int per_sm = ctas_per_sm > 0 && ctas_per_sm < WsCfg<D>::MIN_BLOCKS ? ctas_per_sm
                                                                           : WsCfg<D>::MIN_BLOCKS;
    const int slots = occ.sms * per_sm;
    const int grid = a.n_tc_units < slots ? a.n_tc_units : slots;
    attn_ws_kernel<D><<<grid, kWsThreads, WsCfg<D>::SMEM, stream>>>(km, vm, a, wp);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

bool tc_path_supported(int L, int NB, int Hkv, int bs) {
    // TMA row coordinates are 32-bit
    return (long long)L * NB * Hkv * bs < (1LL << 31);
}

cudaError_t launch_attention_tc(const AttnLaunch &a, cudaStream_t stream, int ctas_per_sm) {
    if (a.n_tc_units <= 0) return cudaSuccess;
    if (a.D == 64) return launch_ws_d<64>(a, stream, ctas_per_sm);
    if (a.D == 128) return launch_ws_d<128>(a, stream, ctas_per_sm);
    return cudaErrorInvalidValue;
}

}  // namespace kvp
