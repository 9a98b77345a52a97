// Paged attention on the 5th-generation tensor cores (tcgen05, sm_103a) for
// work items with more than 32 query rows: shared-prefix segments read by
// many sequences, MCTS tree levels and draft-tree verification.
//
// One CTA of 128 threads per SM pulls work units from an atomic counter.  A
// unit is up to 128 query rows (one thread per row) against a list of
// 64-token KV tiles whose descriptors (with physical block ids) are staged in
// shared memory.  Per tile:
//   S = Q K^T   tcgen05.mma M=128, N=64, K=d; A = Q, B = K tile, both K-major
//               in 128-byte-swizzled shared memory; S lands in TMEM
//               (double-buffered: the MMA for tile t+1 is issued with P V of
//               tile t)
//   softmax     each thread loads its row of S from TMEM (tcgen05.ld), masks
//               (tile end, member interval, draft-tree ancestors), and turns
//               it into P = 2^(s*scale*log2e - m) in bf16, written to shared
//               memory (double-buffered); the running max m is only raised
//               when a tile's max exceeds it by more than 8 (a factor 256),
//               and then the row of O in TMEM is rescaled (ld, scale, st)
//   O += P V    tcgen05.mma M=128, N=d, K=64; A = P (K-major), B = V tile
//               (d contiguous: MN-major); O accumulates in TMEM
// K and V arrive by cp.async into a 4-6 deep ring with the same swizzle; an
// mbarrier per MMA kind (two phases each) tracks completion through
// tcgen05.commit.  Every wait is bounded: on a timeout the kernel sets bit 4
// of the workspace error word, drains and frees its TMEM, and exits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kvp_internal.h"

namespace kvp {
namespace {

constexpr int kTcThreads = 128;
constexpr int kTmemCols = 256;
constexpr uint32_t kWaitLimit = 1u << 22;   // try_wait polls before giving up

__device__ __forceinline__ uint32_t saddr(const void *p) {
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
// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---- fences
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_sync() {
    tc_before_sync();
    __syncthreads();
    tc_after_sync();
}

// ---- tcgen05
// Shared-memory matrix descriptor: 128-byte swizzle, start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 (bits 46-47).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1), A and B
// bf16 (bits 7-9, 10-12 = 1), A K-major, B K-major or MN-major (bit 16),
// N >> 3 (bits 17-22), M >> 4 (bits 24-28).
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

// 32 consecutive TMEM columns of this thread's lane -> r[0..31]
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
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ancestor-or-self bitmask of draft node i of sequence b (bit j = node j)
__device__ uint64_t tc_ancestor_mask(const int32_t *parent, int b, int i, int n, int32_t *err) {
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

template <int D>
struct TcCfg {
    static constexpr int ROWS = 128;
    static constexpr int CH = D / 8;                    // 16-byte chunks per row
    static constexpr int Q_BYTES = ROWS * D * 2;
    static constexpr int TILE_BYTES = kTileTokens * D * 2;
    static constexpr int NSTAGE = D == 64 ? 6 : 4;
    static constexpr int P_BYTES = ROWS * kTileTokens * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int STAGE_OFF = Q_OFF + Q_BYTES;
    static constexpr int P_OFF = STAGE_OFF + NSTAGE * 2 * TILE_BYTES;
    static constexpr int DESC_OFF = P_OFF + 2 * P_BYTES;
    static constexpr int BAR_OFF = DESC_OFF + kMaxItemTiles * (int)sizeof(KvTile);
    static constexpr int SMEM = BAR_OFF + 64 + 1024;   // + slack to align the base to 1024
    static constexpr int S_COL = 0;                     // S buffers at columns 0 and 64
    static constexpr int O_COL = 128;                   // O at columns 128 .. 128+D
};

// byte offset of 16-byte chunk c of row r in a [QB][rows][128 B] swizzled tile
template <int ROWS_IN_TILE>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((c >> 3) * ROWS_IN_TILE * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const AttnLaunch a) {
    using C = TcCfg<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    KvTile *s_tiles = reinterpret_cast<KvTile *>(smem + C::DESC_OFF);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);   // s0, s1, o0, o1
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + 32);
    int *s_unit = reinterpret_cast<int *>(smem + C::BAR_OFF + 40);
    int *s_abort = reinterpret_cast<int *>(smem + C::BAR_OFF + 44);

    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t bar_s0 = saddr(&bars[0]), bar_o0 = saddr(&bars[2]);

    if (tid == 0) {
        mbar_init(bar_s0, 1);
        mbar_init(bar_s0 + 8, 1);
        mbar_init(bar_o0, 1);
        mbar_init(bar_o0 + 8, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         saddr(s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_sync();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;   // this warp's TMEM lanes

    const uint32_t q_smem = saddr(smem + C::Q_OFF);
    const uint32_t stage_smem = saddr(smem + C::STAGE_OFF);
    const uint32_t p_smem = saddr(smem + C::P_OFF);
    const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *kpool = static_cast<const __nv_bfloat16 *>(a.k_pool);
    const __nv_bfloat16 *vpool = static_cast<const __nv_bfloat16 *>(a.v_pool);
    const int bs_log2 = a.bs_log2, bs_mask = (1 << bs_log2) - 1;
    const size_t head_stride = (size_t)D << bs_log2;
    const size_t block_stride = (size_t)a.Hkv * head_stride;
    constexpr uint32_t IDESC_S = idesc_bf16(128, kTileTokens, false);
    constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);

    uint32_t n_s = 0, n_pv = 0;   // S / PV MMAs committed by this CTA so far
    bool ok = true;
    const int lh = a.L * a.Hkv;

    for (;;) {
        if (tid == 0) *s_unit = atomicAdd(a.tc_counter, 1);
        __syncthreads();
        const int unit = *s_unit;
        if (unit >= a.n_tc_units || *s_abort) break;
        const int item_idx = unit / lh;
        const int rem = unit - item_idx * lh;
        const int kvh = rem % a.Hkv, l = rem / a.Hkv;
        const WorkItem it = a.tc_items[item_idx];
        const int ntile = it.tile_end - it.tile_begin;
        {
            const int4 *src = reinterpret_cast<const int4 *>(a.tiles + it.tile_begin);
            int4 *dst = reinterpret_cast<int4 *>(s_tiles);
            for (int i = tid; i < ntile * 2; i += kTcThreads) dst[i] = src[i];
        }
        const int G = a.G;
        const int rows = it.n_members * G;
        const int r = tid;
        const bool has = r < rows;
        const int mem = r / G;
        int qt = 0;
        if (has) qt = __ldg(a.members + it.member_off + mem);
        uint64_t tmask = ~0ull;
        if (has && a.tree_parent)
            tmask = tc_ancestor_mask(a.tree_parent, qt / a.n_draft, qt % a.n_draft, a.n_draft, a.err);
        const size_t layer_base = (size_t)l * a.NB * block_stride + (size_t)kvh * head_stride;

        // Q rows (zero for padding rows), one row per thread
        {
            const __nv_bfloat16 *qrow =
                has ? qb + (((size_t)l * a.nq + qt) * a.Hq + kvh * G + r % G) * D : qb;
#pragma unroll
            for (int c = 0; c < C::CH; ++c)
                cp_async16(q_smem + swz<128>(r, c), qrow + c * 8, has ? 16 : 0);
            cp_async_commit();
        }
        __syncthreads();   // descriptors staged

        auto issue = [&](int t) {
            const KvTile &kt = s_tiles[t];
            const int ntok = kt.ntok_flags & 0xFFFF;
            const int jb = kt.tok0 >> bs_log2;
            const uint32_t dK = stage_smem + (t % C::NSTAGE) * 2 * C::TILE_BYTES;
            const uint32_t dV = dK + C::TILE_BYTES;
#pragma unroll
            for (int i = 0; i < kTileTokens * C::CH / kTcThreads; ++i) {
                const int x = tid + i * kTcThreads;
                const int tok = x / C::CH, c = x % C::CH;
                const uint32_t off = swz<kTileTokens>(tok, c);
                const __nv_bfloat16 *sk = kpool, *sv = vpool;
                int bytes = 0;
                if (tok < ntok) {
                    const int pos = kt.tok0 + tok;
                    const int blk = kt.blk[(pos >> bs_log2) - jb];
                    if ((unsigned)blk < (unsigned)a.NB) {
                        const size_t e = layer_base + (size_t)blk * block_stride +
                                         (size_t)(pos & bs_mask) * D + c * 8;
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
        };
        auto issue_s = [&](int t) {   // S_t = Q K_t^T into S buffer n_s & 1
            const uint32_t kst = stage_smem + (t % C::NSTAGE) * 2 * C::TILE_BYTES;
            const uint32_t d_tm = tmem + C::S_COL + (n_s & 1) * kTileTokens;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t koff = (uint32_t)(k & 3) * 32;
                const uint64_t da = sdesc(q_smem + (k >> 2) * (128 * 128) + koff, 16, 1024);
                const uint64_t db = sdesc(kst + (k >> 2) * (kTileTokens * 128) + koff, 16, 1024);
                umma(d_tm, da, db, IDESC_S, k > 0 ? 1u : 0u);
            }
            umma_commit(bar_s0 + (n_s & 1) * 8);
        };
        auto issue_pv = [&](int t, bool first) {   // O += P_t V_t
            const uint32_t vst = stage_smem + (t % C::NSTAGE) * 2 * C::TILE_BYTES + C::TILE_BYTES;
            const uint32_t pbuf = p_smem + (n_pv & 1) * C::P_BYTES;
#pragma unroll
            for (int k = 0; k < kTileTokens / 16; ++k) {
                const uint64_t da = sdesc(pbuf + k * 32, 16, 1024);
                const uint64_t db = sdesc(vst + k * (16 * 128), kTileTokens * 128, 1024);
                umma(tmem + C::O_COL, da, db, IDESC_PV, (first && k == 0) ? 0u : 1u);
            }
            umma_commit(bar_o0 + (n_pv & 1) * 8);
        };
        auto wait_s = [&](uint32_t idx) {
            if (!mbar_wait(bar_s0 + (idx & 1) * 8, (idx >> 1) & 1)) {
                ok = false;
                atomicOr(a.err, 4);
            }
        };
        auto wait_pv = [&](uint32_t idx) {
            if (!mbar_wait(bar_o0 + (idx & 1) * 8, (idx >> 1) & 1)) {
                ok = false;
                atomicOr(a.err, 4);
            }
        };

#pragma unroll
        for (int t = 0; t < C::NSTAGE - 1; ++t) {
            if (t < ntile) issue(t);
            cp_async_commit();
        }
        // Q and tile 0 resident
        cp_async_wait<C::NSTAGE - 2>();
        fence_async_smem();
        tc_sync();
        const uint32_t s0 = n_s, p0 = n_pv;
        if (tid == 0 && ntile > 0) issue_s(0);
        n_s += ntile > 0 ? 1 : 0;

        float m_used = -INFINITY, lsum = 0.f;
        for (int t = 0; t < ntile; ++t) {
            const KvTile &kt = s_tiles[t];
            const int ntok = kt.ntok_flags & 0xFFFF;
            const bool tree = (kt.ntok_flags >> 16) & kTileTree;
            const int mlo = kt.members & 0xFFFF, mhi = kt.members >> 16;
            const bool in = has && mem >= mlo && mem < mhi;

            wait_s(s0 + t);
            tc_after_sync();
            float s[kTileTokens];
            {
                uint32_t rr[32];
                const uint32_t sa = tmem + lane_base + C::S_COL + ((s0 + t) & 1) * kTileTokens;
                tmem_ld32(sa, rr);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(rr[j]);
                tmem_ld32(sa + 32, rr);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(rr[j]);
            }
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < kTileTokens; ++j) {
                bool v = in && j < ntok;
                if (tree) v = v && ((tmask >> j) & 1ull);
                s[j] = v ? s[j] * a.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[j]);
            }
            const float m_new = fmaxf(m_used, mx);
            const bool resc = m_used != -INFINITY && m_new > m_used + 8.f;
            if (__any_sync(0xffffffffu, resc)) {
                // O must be complete before it is rescaled in place
                if (t > 0) wait_pv(p0 + t - 1);
                tc_after_sync();
                const float f = resc ? exp2_sfu(m_used - m_new) : 1.f;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t rr[32];
                    const uint32_t oa = tmem + lane_base + C::O_COL + c0;
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
            uint32_t pk[kTileTokens / 2];
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < kTileTokens; j += 2) {
                const float e0 = m_used == -INFINITY ? 0.f : exp2_sfu(s[j] - m_used);
                const float e1 = m_used == -INFINITY ? 0.f : exp2_sfu(s[j + 1] - m_used);
                rs += e0 + e1;
                pk[j / 2] = pack_bf16x2(e0, e1);
            }
            lsum += rs;
            // P buffer (p0 + t) & 1 was last read by P V of tile t-2
            if (t >= 2) wait_pv(p0 + t - 2);
            {
                unsigned char *prow = smem + C::P_OFF + ((p0 + t) & 1) * C::P_BYTES;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    *reinterpret_cast<uint4 *>(prow + swz<128>(r, c)) = v;
                }
            }
            fence_async_smem();
            // tile t+1 resident for its S MMA
            cp_async_wait<C::NSTAGE - 3>();
            fence_async_smem();
            if (!ok) *s_abort = 1;
            tc_sync();
            if (*s_abort) break;
            if (tid == 0) {
                issue_pv(t, t == 0);
                if (t + 1 < ntile) issue_s(t + 1);
            }
            n_pv += 1;
            n_s += (t + 1 < ntile) ? 1 : 0;
            // refill the stage of tile t-1 (its P V has finished) with tile t+NSTAGE-1
            if (t >= 1) wait_pv(p0 + t - 1);
            if (t + C::NSTAGE - 1 < ntile) issue(t + C::NSTAGE - 1);
            cp_async_commit();
        }
        cp_async_wait<0>();
        if (ntile > 0) wait_pv(p0 + ntile - 1);
        tc_after_sync();

        // epilogue: O / l (or the partial row) from TMEM
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const float lse2 = lsum > 0.f ? m_used + __log2f(lsum) : -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tmem + lane_base + C::O_COL + c0, rr);
            tmem_wait_ld();
            if (!has || ntile == 0) continue;
            if (it.out_base < 0) {
                __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                     (((size_t)l * a.nq + qt) * a.Hq + kvh * G + r % G) * D + c0;
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
                float *dst = a.part_o + (((size_t)l * a.Hkv + kvh) * a.P + it.out_base + r) * D + c0;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + j) =
                        make_float4(__uint_as_float(rr[j]) * inv, __uint_as_float(rr[j + 1]) * inv,
                                    __uint_as_float(rr[j + 2]) * inv, __uint_as_float(rr[j + 3]) * inv);
            }
        }
        if (has && ntile > 0) {
            if (it.out_base < 0) {
                if (a.lse) a.lse[((size_t)l * a.nq + qt) * a.Hq + kvh * G + r % G] = lse2 * 0.6931471805599453f;
            } else {
                a.part_lse[((size_t)l * a.Hkv + kvh) * a.P + it.out_base + r] = lse2;
            }
        }
        if (!ok) *s_abort = 1;
        tc_sync();   // TMEM O and S buffers free for the next unit
    }
    tc_sync();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

struct TcOcc {
    int sms = 0;
    bool ok = false;
};

template <int D>
TcOcc &tc_occ() {
    static TcOcc occ;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return;
        if (cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcCfg<D>::SMEM) != cudaSuccess)
            return;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
        occ.sms = sms;
        occ.ok = true;
    });
    return occ;
}

template <int D>
cudaError_t launch_tc_d(const AttnLaunch &a, cudaStream_t stream) {
    TcOcc &occ = tc_occ<D>();
    if (!occ.ok) return cudaErrorInvalidDevice;
    const int grid = a.n_tc_units < occ.sms ? a.n_tc_units : occ.sms;
    attn_tc_kernel<D><<<grid, kTcThreads, TcCfg<D>::SMEM, stream>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_tc(const AttnLaunch &a, cudaStream_t stream) {
    if (a.n_tc_units <= 0) return cudaSuccess;
    if (a.D == 64) return launch_tc_d<64>(a, stream);
    if (a.D == 128) return launch_tc_d<128>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace kvp
