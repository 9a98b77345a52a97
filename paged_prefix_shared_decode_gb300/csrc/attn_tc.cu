// Paged attention on the 5th-generation tensor cores (tcgen05 + TMA,
// sm_103a) for work items with more than 32 query rows: shared-prefix
// segments read by many sequences, MCTS tree levels and draft-tree
// verification.
//
// One persistent CTA of 12 warps per SM.  A work unit is (item, layer, kv
// head): up to 128 query rows (the item's members x the GQA group of the kv
// head), or a pair unit of up to 256 rows as two 128-row tiles over one K/V
// stream, against the item's 64-token KV tiles, taken two at a time as
// 128-token steps.
//   warp 0      K producer, warp 1 V producer.  Each fills its own ring, since
//               K is released as soon as S = Q K^T is computed and V only once
//               P V is.  Whole tiles whose blocks start on a box boundary are
//               copied by TMA (cp.async.bulk.tensor, one box per block and
//               64-column slab, 128-byte swizzle, one lane per box); ragged
//               tiles by cp.async (16-byte chunks, same swizzle, zero fill).
//   warp 2      MMA issuer (one thread): S_g = Q K^T (M=128, N=128, K=d) into
//               TMEM buffer g = step parity, and O_g += P_g V (M=128, N=d,
//               K=128) with P_g read from TMEM.
//   warp 3      claims units from an atomic counter, stages their tile
//               descriptors in shared memory (two slots), and loads each
//               unit's Q as soon as the previous unit's last S is done: by
//               TMA boxes of whole rows (the G heads of consecutive query
//               tokens) when the unit's members are consecutive tokens, else
//               by a cp.async gather.
//   warps 4-7   softmax group 0 (even steps), warps 8-11 group 1 (odd
//               steps), one thread per query row.  Each group keeps its own
//               running max m_g, sum l_g and accumulator O_g, so while one
//               group turns step t's scores into P the tensor cores run the
//               other group's P V and next S.  The two groups' (m, l, O) are
//               merged when the unit ends.  In a pair unit group g takes
//               every step for the rows of tile g and writes them alone.
// P (bf16 pairs) overwrites the S columns it came from, so it never passes
// through shared memory.  The running max is raised only when a step's P
// would sum to more than 2^32, so every p <= 2^32; O_g is then rescaled in
// TMEM.
// Every wait is bounded; on a timeout the CTA sets bit 4 of the workspace
// error word and all roles leave their loops; before the CTA frees its TMEM
// and ends, the producers let the copies they issued land and the MMA thread
// lets its MMAs complete (bounded waits too).  Softmax warps none of whose
// rows is in the unit (a half-filled tile) keep only the barriers.
//
// TMEM columns: S_0 [0, 128), S_1 [128, 256), O_0 [256, 256 + d),
// O_1 [256 + d, 256 + 2d).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/kvp.h"
#include "kv4_codes.cuh"
#include "kvp_internal.h"

namespace kvp {
namespace {

constexpr int kProdWarps = 2;        // warp 0: K, warp 1: V
constexpr int kVWarp = 1;
constexpr int kMmaWarp = 2;
constexpr int kUnitWarp = 3;         // claims units, stages descriptors and Q
constexpr int kSoftWarp0 = 4;        // warps 4-7: group 0, 8-11: group 1
constexpr int kTcThreads = 384;      // 12 warps: 3 per SM sub-partition
constexpr int kSoftThreads = 256;
constexpr int kGroupThreads = 128;
constexpr int kStepTokens = 2 * kTileTokens;
constexpr int kTmemCols = 512;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kSlackSum = 4294967296.f;   // 2^32: bound on a step's sum of p

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// arrives on the barrier once every earlier cp.async of this thread has landed
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
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
// adds expected transaction bytes without arriving
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// non-blocking test of a phase
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
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
// Named barrier 1 over the 256 softmax threads with an OR reduction, so that
// all of them take the same branch.
__device__ __forceinline__ bool soft_bar_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\nbar.red.or.pred p, 1, 256, q;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// ---- tcgen05
// (The start address is the low 14 bits, in 16-byte units; shared memory
// addresses stay below 2^18, so a descriptor plus (bytes >> 4) describes the
// operand that many bytes further on.  The MMA thread builds one descriptor
// per operand and step and offsets it per instruction.)
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
// D (TMEM) (+)= A (shared memory) * B (shared memory)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// D (TMEM) (+)= A (TMEM) * B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4}], [%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

template <int D>
struct TcCfg {
    static constexpr int NSLAB = D / 64;               // 64-column slabs (128-byte rows)
    static constexpr int CH = D / 8;                   // 16-byte chunks per row
    static constexpr int SLAB = kStepTokens * 128;     // one slab of a 128-row operand
    static constexpr int OPER = NSLAB * SLAB;          // Q, or K (V) of one step
    static constexpr int NK = D == 64 ? 5 : 2;         // K ring depth (steps)
    static constexpr int NV = D == 64 ? 5 : 2;         // V ring depth (steps)
    static constexpr int Q_OFF = 0;                    // two 128-row Q tiles
    static constexpr int K_OFF = Q_OFF + 2 * OPER;
    static constexpr int V_OFF = K_OFF + NK * OPER;
    // 4-bit pages: each producer stages one 64-token tile of codes and row
    // exponents per buffer, two buffers, and expands it into its ring
    static constexpr int CODE4 = kTileTokens * D / 2;   // codes of one tile
    static constexpr int STG4_BUF = CODE4 + kTileTokens;
    static constexpr int STG4_OFF = V_OFF + NV * OPER;
    static constexpr int DESC_OFF = STG4_OFF + 2 * 2 * STG4_BUF;                      // [2][kMaxItemTiles]
    static constexpr int ML_OFF = DESC_OFF + 2 * kMaxItemTiles * (int)sizeof(KvTile);  // [2][128] float2
    static constexpr int UNIT_OFF = ML_OFF + 2 * 128 * 8;                           // [2] ints
    static constexpr int BAR_OFF = UNIT_OFF + 16;
    static constexpr int B_UNIT_FULL = 0, B_UNIT_EMPTY = 2, B_K_FULL = 4, B_K_EMPTY = B_K_FULL + NK,
                         B_V_FULL = B_K_EMPTY + NK, B_V_EMPTY = B_V_FULL + NV, B_S_FULL = B_V_EMPTY + NV,
                         B_P_FULL = B_S_FULL + 2, B_Q_FULL = B_P_FULL + 2, B_Q_EMPTY = B_Q_FULL + 1,
                         B_O_FULL = B_Q_EMPTY + 1, B_O_EMPTY = B_O_FULL + 1, B_DRAIN = B_O_EMPTY + 1,
                         N_BARS = B_DRAIN + 1;
    static constexpr int MISC_OFF = BAR_OFF + N_BARS * 8;   // tmem address, abort flag
    static constexpr int SMEM = MISC_OFF + 16 + 1024;       // + slack to align the base to 1024
    static constexpr int S_COL = 0, O_COL = 2 * kStepTokens;
};
static_assert(TcCfg<64>::SMEM <= 227 * 1024 && TcCfg<128>::SMEM <= 227 * 1024, "shared memory");

// byte offset of 16-byte chunk c of row `row` in a 128-row operand
// ([slab][row][128 B], 128-byte swizzle)
__device__ __forceinline__ uint32_t swz(int row, int c) {
    return (uint32_t)((c >> 3) * (kStepTokens * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}

// Valid columns j0 .. j0+31 of a 64-token tile for one row, as bits: those
// before the row's valid count nv (0 outside the tile's member interval)
// and, in a draft-tree tile, ancestors-or-self only.
__device__ __forceinline__ uint32_t valid_bits(int nv, bool tree, uint64_t tmask, int j0) {
    uint32_t vm = nv >= j0 + 32 ? 0xffffffffu : (nv <= j0 ? 0u : (1u << (nv - j0)) - 1u);
    if (tree) vm &= (uint32_t)(tmask >> j0);
    return vm;
}
// Max of the valid scores among 32 (-inf if none).  Masking uses selects, not
// per-element branches, and is skipped when the whole warp is unmasked.
__device__ __forceinline__ float max32(const uint32_t (&x)[32], uint32_t vm) {
    float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
    if (__all_sync(0xffffffffu, vm == 0xffffffffu)) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            a0 = fmaxf(a0, __uint_as_float(x[j]));
            a1 = fmaxf(a1, __uint_as_float(x[j + 1]));
            a2 = fmaxf(a2, __uint_as_float(x[j + 2]));
            a3 = fmaxf(a3, __uint_as_float(x[j + 3]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            a0 = fmaxf(a0, (vm >> j) & 1u ? __uint_as_float(x[j]) : -INFINITY);
            a1 = fmaxf(a1, (vm >> (j + 1)) & 1u ? __uint_as_float(x[j + 1]) : -INFINITY);
            a2 = fmaxf(a2, (vm >> (j + 2)) & 1u ? __uint_as_float(x[j + 2]) : -INFINITY);
            a3 = fmaxf(a3, (vm >> (j + 3)) & 1u ? __uint_as_float(x[j + 3]) : -INFINITY);
        }
    }
    return fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
}
// (d0, d1) = (a0, a1) * b + c in one packed instruction
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b, float c) {
    asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %4};\nmov.b64 rc, {%5, %5};\n"
        "fma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}\n"
        : "=f"(d0), "=f"(d1) : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (s0, s1) += (a0, a1) in one packed instruction
__device__ __forceinline__ void fadd2(float &s0, float &s1, float a0, float a1) {
    asm("{\n.reg .b64 ra, rs;\nmov.b64 ra, {%2, %3};\nmov.b64 rs, {%0, %1};\nadd.f32x2 rs, rs, ra;\n"
        "mov.b64 {%0, %1}, rs;\n}\n"
        : "+f"(s0), "+f"(s1) : "f"(a0), "f"(a1));
}
// p = 2^(s * sc + nm) for scores j0 .. j0+15, packed as 8 bf16 pairs; with
// MASKED the invalid ones (bits of vm) give 0.  Adds the sum of p to sum.
template <bool MASKED>
__device__ __forceinline__ void exp_pack16(const uint32_t (&x)[32], int j0, float sc, float nm,
                                           uint32_t vm, uint32_t *p, float &sum) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        float y0, y1;
        ffma2(y0, y1, __uint_as_float(x[j0 + j]), __uint_as_float(x[j0 + j + 1]), sc, nm);
        if (MASKED) {
            y0 = (vm >> (j0 + j)) & 1u ? y0 : -INFINITY;
            y1 = (vm >> (j0 + j + 1)) & 1u ? y1 : -INFINITY;
        }
        const float e0 = exp2_sfu(y0), e1 = exp2_sfu(y1);
        fadd2(s0, s1, e0, e1);
        p[j / 2] = pack_bf16x2(e0, e1);
    }
    sum += s0 + s1;
}

// P = 2^(s * sc + nm) of one step, packed into pk (word i holds scores 2i,
// 2i + 1); adds the sum of P to ls.  S is only read.
__device__ __forceinline__ void p_pass(uint32_t s_tm, float nm, float sc, int nv0, bool tr0, int nv1, bool tr1,
                                       uint64_t tmask, uint32_t (&pk)[64], float &ls) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t x[32], y[32];
        tmem_ld32(s_tm + 64 * hh, x);
        tmem_ld32(s_tm + 64 * hh + 32, y);
        tmem_wait_ld();
        const uint32_t vx = valid_bits(hh ? nv1 : nv0, hh ? tr1 : tr0, tmask, 0);
        const uint32_t vy = valid_bits(hh ? nv1 : nv0, hh ? tr1 : tr0, tmask, 32);
        uint32_t *q = pk + 32 * hh;
        if (__all_sync(0xffffffffu, (vx & vy) == 0xffffffffu)) {
            exp_pack16<false>(x, 0, sc, nm, vx, q, ls);
            exp_pack16<false>(x, 16, sc, nm, vx, q + 8, ls);
            exp_pack16<false>(y, 0, sc, nm, vy, q + 16, ls);
            exp_pack16<false>(y, 16, sc, nm, vy, q + 24, ls);
        } else {
            exp_pack16<true>(x, 0, sc, nm, vx, q, ls);
            exp_pack16<true>(x, 16, sc, nm, vx, q + 8, ls);
            exp_pack16<true>(y, 0, sc, nm, vy, q + 16, ls);
            exp_pack16<true>(y, 16, sc, nm, vy, q + 24, ls);
        }
    }
}
// P overwrites the first 64 S columns (all scores are read by then)
__device__ __forceinline__ void p_store(uint32_t s_tm, const uint32_t (&pk)[64]) {
    tmem_st32(s_tm, *reinterpret_cast<const uint32_t(*)[32]>(pk));
    tmem_st32(s_tm + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
}
// Row max of one step's valid raw scores (-inf if none).
__device__ __forceinline__ float step_max(uint32_t s_tm, int nv0, bool tr0, int nv1, bool tr1, uint64_t tmask) {
    uint32_t x[32], y[32];
    tmem_ld32(s_tm, x);
    tmem_ld32(s_tm + 32, y);
    tmem_wait_ld();
    float mx = fmaxf(max32(x, valid_bits(nv0, tr0, tmask, 0)), max32(y, valid_bits(nv0, tr0, tmask, 32)));
    tmem_ld32(s_tm + 64, x);
    tmem_ld32(s_tm + 96, y);
    tmem_wait_ld();
    return fmaxf(mx, fmaxf(max32(x, valid_bits(nv1, tr1, tmask, 0)), max32(y, valid_bits(nv1, tr1, tmask, 32))));
}
// The slow path, kept out of line so that its registers do not add to the
// common path's: the step's max, the new running max (raised for the rows
// marked bad), P again, stored.  Returns (new m, sum of P).
__device__ __noinline__ float2 recompute_step(uint32_t s_tm, float m, float sc, int nv0, bool tr0, int nv1, bool tr1,
                                              uint64_t tmask, bool bad) {
    const float tmx = step_max(s_tm, nv0, tr0, nv1, tr1, tmask) * sc;
    const float m_new = bad ? fmaxf(m, tmx) : m;
    float ls = 0.f;
    uint32_t pk[64];
    p_pass(s_tm, m_new == -INFINITY ? 0.f : -m_new, sc, nv0, tr0, nv1, tr1, tmask, pk, ls);
    p_store(s_tm, pk);
    return make_float2(m_new, ls);
}

template <int D, bool KV4>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap, const AttnLaunch a, const int box_rows,
                   const int q_tma, const int out32) {
    using C = TcCfg<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    KvTile *s_desc = reinterpret_cast<KvTile *>(smem + C::DESC_OFF);
    float2 *s_ml = reinterpret_cast<float2 *>(smem + C::ML_OFF);
    volatile int *s_unit = reinterpret_cast<volatile int *>(smem + C::UNIT_OFF);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    const uint32_t bar0 = saddr(smem + C::BAR_OFF);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(C::B_UNIT_FULL + s), 1);
            // unit slot free: MMA thread + softmax threads + K and V warps
            mbar_init(bar(C::B_UNIT_EMPTY + s), 1 + kSoftThreads + kProdWarps);
            mbar_init(bar(C::B_S_FULL + s), 1);
            mbar_init(bar(C::B_P_FULL + s), kGroupThreads);
        }
        for (int s = 0; s < C::NK; ++s) {
            mbar_init(bar(C::B_K_FULL + s), 32);
            mbar_init(bar(C::B_K_EMPTY + s), 1);
        }
        for (int s = 0; s < C::NV; ++s) {
            mbar_init(bar(C::B_V_FULL + s), 32);
            mbar_init(bar(C::B_V_EMPTY + s), 1);
        }
        mbar_init(bar(C::B_Q_FULL), 32);
        mbar_init(bar(C::B_Q_EMPTY), 1);
        mbar_init(bar(C::B_O_FULL), 1);
        mbar_init(bar(C::B_O_EMPTY), kSoftThreads);
        mbar_init(bar(C::B_DRAIN), 1);
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

    // bounded wait; on a timeout the whole CTA aborts.  A phase that is
    // already complete is seen by the non-blocking test first, which measured
    // about half the latency of try_wait on the MMA thread's critical path.
    auto wait = [&](uint32_t b, uint32_t parity) -> bool {
        if (mbar_test_wait(b, parity)) return true;
        for (uint32_t i = 0; i < kWaitLimit; ++i) {
            if (mbar_try_wait(b, parity)) return true;
            if ((i & 1023) == 1023 && *s_abort) return false;
        }
        *s_abort = 1;
        atomicOr(a.err, KVP_DEVERR_WAIT_TIMEOUT);
        return false;
    };
    // bounded wait that records nothing: lets copies and MMAs already in
    // flight land before the CTA frees its shared memory and TMEM (after a
    // normal run they have all landed and it returns at once)
    auto settle = [&](uint32_t b, uint32_t parity) {
        for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(b, parity); ++i) {
        }
    };

    const int n_items = a.n_tc_units / (a.L * a.Hkv);
    const int G = a.G;
    const uint32_t q_smem = saddr(smem + C::Q_OFF);
    const uint32_t k_smem = saddr(smem + C::K_OFF);
    const uint32_t v_smem = saddr(smem + C::V_OFF);
    const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(a.q);

    if (warp < kProdWarps) {
        // ------------------------------------------------------------ producers
        const bool is_v = warp == kVWarp;
        const __nv_bfloat16 *pool = static_cast<const __nv_bfloat16 *>(is_v ? a.v_pool : a.k_pool);
        const CUtensorMap *map = is_v ? &vmap : &kmap;
        const int nring = is_v ? C::NV : C::NK;
        const int b_full = is_v ? C::B_V_FULL : C::B_K_FULL;
        const int b_empty = is_v ? C::B_V_EMPTY : C::B_K_EMPTY;
        const uint32_t ring = is_v ? v_smem : k_smem;
        const int bs_log2 = a.bs_log2, bs = 1 << bs_log2;
        const size_t head_stride = (size_t)D << bs_log2;
        const size_t block_stride = (size_t)a.Hkv * head_stride;
        // (block, 64-column slab) boxes of one 64-token tile
        const int nbox = (kTileTokens / box_rows) * C::NSLAB;
        if (!KV4 && lane == 0)
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
        // lane 0 waits (acquire) and the warp follows it (__syncwarp orders memory)
        auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
            int ok = 1;
            if (lane == 0) ok = wait(b, parity) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            return ok != 0;
        };
        uint32_t g = 0;   // steps filled
        for (int uc = 0;; ++uc) {
            const int slot = uc & 1;
            const bool okw = wait_warp(bar(C::B_UNIT_FULL + slot), (uc >> 1) & 1);
            const int unit = okw ? s_unit[slot] : -1;
            if (unit < 0) break;
            const int item_idx = unit % n_items;
            const int lk = unit / n_items;
            const int kvh = lk % a.Hkv, l = lk / a.Hkv;
            const WorkItem it = a.tc_items[item_idx];
            const int ntile = it.tile_end - it.tile_begin;
            const int nsteps = (ntile + 1) >> 1;
            const size_t layer_base = (size_t)l * a.NB * block_stride + (size_t)kvh * head_stride;
            const int row_base_lh = (l * a.NB) * a.Hkv + kvh;   // row of block b = (row_base_lh + b*Hkv) * bs
            const KvTile *tiles = s_desc + slot * kMaxItemTiles;
            // 4-bit pages: tile j's codes and row exponents go to staging
            // buffer j mod 2 by cp.async (the next tile's while this one is
            // expanded); the expansion writes bf16 rows into the ring stage in
            // the layout the MMAs read (64-column slabs, 128-byte swizzle)
            const uint32_t stg4 = saddr(smem + C::STG4_OFF + (is_v ? 2 : 0) * C::STG4_BUF);
            auto load4 = [&](int j) {
                const KvTile &kt = tiles[j];
                const int ntok = kt.ntok_flags & 0xFFFF;
                const int jb = kt.tok0 >> bs_log2;
                const uint8_t *codes = static_cast<const uint8_t *>(is_v ? a.v_pool : a.k_pool);
                const int8_t *exps = static_cast<const int8_t *>(is_v ? a.v_exp : a.k_exp);
                const size_t lrow = (size_t)l * a.NB * a.Hkv;   // + block * Hkv + kvh, times bs
                const uint32_t sb = stg4 + (j & 1) * C::STG4_BUF;
                for (int x = lane; x < kTileTokens * (D / 32); x += 32) {
                    const int tok = x / (D / 32), c = x % (D / 32);
                    const uint8_t *src = codes;
                    int bytes = 0;
                    if (tok < ntok) {
                        const int pos = kt.tok0 + tok;
                        const int blk = kt.blk[(pos >> bs_log2) - jb];
                        if ((unsigned)blk < (unsigned)a.NB) {
                            const size_t row = ((lrow + (size_t)blk * a.Hkv + kvh) << bs_log2) + (pos & (bs - 1));
                            src = codes + row * (D / 2) + c * 16;
                            bytes = 16;
                        } else if (c == 0) {
                            atomicOr(a.err, 1);
                        }
                    }
                    cp_async16(sb + tok * (D / 2) + c * 16, src, bytes);
                }
                // exponents: four groups of 16 tokens, each inside one block
                // (decode tiles start on block boundaries, blocks hold a
                // multiple of 16 tokens)
                if (lane < 4) {
                    const int8_t *src = exps;
                    int bytes = 0;
                    if (16 * lane < ntok) {
                        const int pos = kt.tok0 + 16 * lane;
                        const int blk = kt.blk[(pos >> bs_log2) - jb];
                        if ((unsigned)blk < (unsigned)a.NB) {
                            src = exps + ((lrow + (size_t)blk * a.Hkv + kvh) << bs_log2) + (pos & (bs - 1));
                            bytes = 16;
                        }
                    }
                    cp_async16(sb + C::CODE4 + 16 * lane, src, bytes);
                }
                cp_async_commit();
            };
            // tile in buffer sb to rows 64 h .. 64 h + 63 of the stage at dst:
            // each lane turns 16-byte chunks of codes (32 dims of one row)
            // into four 16-byte chunks of bf16 (exact: code * 2^e)
            const unsigned char *stg4p = smem + C::STG4_OFF + (is_v ? 2 : 0) * C::STG4_BUF;
            auto expand4 = [&](const unsigned char *sb, uint32_t dst, int h) {
                constexpr int CH4 = D / 32;
                for (int x = lane; x < kTileTokens * CH4; x += 32) {
                    const int tok = x / CH4, q = x % CH4;
                    const uint4 cw = *reinterpret_cast<const uint4 *>(sb + tok * (D / 2) + q * 16);
                    const int e = (int)reinterpret_cast<const int8_t *>(sb + C::CODE4)[tok];
                    const bool fused = e >= -126 && e <= 120;
                    const uint2 sc = exp_pair2(e, e);
                    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {   // word k: dims 32 q + 8 k .. + 7, chunk 4 q + k
                        uint32_t v[4];
                        expand_word(w[k], sc, fused, v);
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                                         dst + swz(h * kTileTokens + tok, 4 * q + k)),
                                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                                     : "memory");
                    }
                }
            };
            if constexpr (KV4)
                if (ntile > 0) load4(0);
            bool alive = true;
            for (int t = 0; alive && t < nsteps; ++t, ++g) {
                const int st = g % nring;
                if (!wait_warp(bar(b_empty + st), ((g / nring) & 1) ^ 1)) { alive = false; break; }
                const uint32_t dst = ring + st * C::OPER;
                const uint32_t fb = bar(b_full + st);
                if constexpr (KV4) {
                    for (int h = 0; h < 2 && 2 * t + h < ntile; ++h) {
                        const int j = 2 * t + h;
                        if (j + 1 < ntile) {
                            load4(j + 1);
                            cp_async_wait<1>();
                        } else {
                            cp_async_wait<0>();
                        }
                        __syncwarp();
                        expand4(stg4p + (j & 1) * C::STG4_BUF, dst, h);
                        __syncwarp();
                    }
                    // the bf16 rows were written through the generic proxy
                    fence_async_smem();
                    mbar_arrive(fb);
                    continue;
                }
                // whole tiles by TMA, one box per lane; ragged ones by cp.async
                // with zero fill past the tile's end
                bool tma[2] = {false, false};
                for (int h = 0; h < 2 && 2 * t + h < ntile; ++h) {
                    const KvTile &kt = tiles[2 * t + h];
                    tma[h] = (kt.ntok_flags & 0xFFFF) == kTileTokens && (kt.tok0 & (box_rows - 1)) == 0;
                }
                if (lane == 0 && (tma[0] || tma[1]))
                    mbar_expect_tx(fb, (uint32_t)(((tma[0] ? 1 : 0) + (tma[1] ? 1 : 0)) * nbox * box_rows * 128));
                __syncwarp();
                for (int h = 0; h < 2 && 2 * t + h < ntile; ++h) {
                    const KvTile &kt = tiles[2 * t + h];
                    const int ntok = kt.ntok_flags & 0xFFFF;
                    if (tma[h]) {
                        if (lane < nbox) {
                            const int k = lane / C::NSLAB, cb = lane % C::NSLAB;
                            const int yoff = bs > kTileTokens ? (kt.tok0 & (bs - 1)) : 0;
                            const int y = (row_base_lh + kt.blk[k] * a.Hkv) * bs + yoff;
                            tma_load_2d(dst + cb * C::SLAB + (h * kTileTokens + k * box_rows) * 128, map, cb * 64,
                                        y, fb);
                        }
                        continue;
                    }
                    const int jb = kt.tok0 >> bs_log2;
#pragma unroll 4
                    for (int x = lane; x < kTileTokens * C::CH; x += 32) {
                        const int tok = x / C::CH, c = x % C::CH;
                        const __nv_bfloat16 *src = pool;
                        int bytes = 0;
                        if (tok < ntok) {
                            const int pos = kt.tok0 + tok;
                            const int blk = kt.blk[(pos >> bs_log2) - jb];
                            if ((unsigned)blk < (unsigned)a.NB) {
                                src = pool + layer_base + (size_t)blk * block_stride +
                                      (size_t)(pos & (bs - 1)) * D + c * 8;
                                bytes = 16;
                            } else if (c == 0) {
                                atomicOr(a.err, 1);
                            }
                        }
                        cp_async16(dst + swz(h * kTileTokens + tok, c), src, bytes);
                    }
                }
                cp_async_arrive(fb);
            }
            if (lane == 0) mbar_arrive(bar(C::B_UNIT_EMPTY + slot));
            if (!alive || __shfl_sync(0xffffffffu, *s_abort, 0)) break;
        }
        // this warp's copies land before the CTA ends: its own cp.async, and
        // the transaction bytes of the last stages it armed
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        if (lane == 0)
            for (uint32_t k = g > (uint32_t)nring ? g - (uint32_t)nring : 0u; k < g; ++k)
                settle(bar(b_full + k % nring), (k / nring) & 1);
        __syncwarp();
    } else if (warp == kUnitWarp) {
        // ------------------------------------------------------------ units and Q
        if (q_tma && lane == 0)
            asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
        int last_q = -1;   // last unit whose Q load was issued
        auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
            int ok = 1;
            if (lane == 0) ok = wait(b, parity) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            __syncwarp();
            return ok != 0;
        };
        for (int uc = 0;; ++uc) {
            const int slot = uc & 1;
            bool ok = wait_warp(bar(C::B_UNIT_EMPTY + slot), ((uc >> 1) & 1) ^ 1);
            int unit = -1;
            if (lane == 0) unit = atomicAdd(a.tc_counter, 1);
            unit = __shfl_sync(0xffffffffu, unit, 0);
            const bool done = !ok || unit >= a.n_tc_units || __shfl_sync(0xffffffffu, *s_abort, 0);
            WorkItem it{};
            if (!done) {
                it = a.tc_items[unit % n_items];
                const int ntile = it.tile_end - it.tile_begin;
                const int4 *src = reinterpret_cast<const int4 *>(a.tiles + it.tile_begin);
                int4 *dst = reinterpret_cast<int4 *>(s_desc + slot * kMaxItemTiles);
                for (int i = lane; i < ntile * 2; i += 32) dst[i] = src[i];
            }
            if (lane == 0) s_unit[slot] = done ? -1 : unit;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_UNIT_FULL + slot));
            if (done) break;
            // Q of this unit, once the previous unit's S MMAs are done with it
            ok = wait_warp(bar(C::B_Q_EMPTY), (uc & 1) ^ 1);
            if (!ok) break;
            const int lk = unit / n_items;
            const int kvh = lk % a.Hkv, l = lk / a.Hkv;
            // (one 128-row tile, or two for a pair unit)
            const int rows = it.n_members * G;
            const int ntq = rows > 128 ? 2 : 1;
            last_q = uc;
            // By TMA when every box's members are consecutive query tokens: a
            // box is the kv head's G query heads of max(1, 8 / G) consecutive
            // tokens, i.e. max(8, G) whole rows of one 64-column slab, so each
            // lands on a 1024-byte boundary of the 128-byte swizzle; boxes
            // past the unit's members are read out of range (zero fill).
            // Otherwise lane j gathers rows j + 32 i by cp.async.
            if (q_tma) {
                const int tpb = G < 8 ? 8 / G : 1;       // tokens per box
                const int nbox = ntq * (128 / (tpb * G)) * C::NSLAB;
                const int z_oob = a.L * a.nq;
                bool consec = true;
                int zc[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int b = lane + 32 * j;
                    const int m0 = (b / C::NSLAB) * tpb;   // first member of the box
                    zc[j] = z_oob;
                    if (b < nbox && m0 < it.n_members) {
                        const int q0 = __ldg(a.members + it.member_off + m0);
                        for (int k = 1; k < tpb && m0 + k < it.n_members; ++k)
                            consec = consec && __ldg(a.members + it.member_off + m0 + k) == q0 + k;
                        zc[j] = l * a.nq + q0;
                    }
                }
                if (__all_sync(0xffffffffu, consec) && nbox <= 64) {
                    if (lane == 0) mbar_expect_tx(bar(C::B_Q_FULL), (uint32_t)(ntq * C::OPER));
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int b = lane + 32 * j;
                        if (b < nbox) {
                            const int cb = b % C::NSLAB, row = (b / C::NSLAB) * tpb * G;   // unit row
                            tma_load_3d(q_smem + (row >> 7) * C::OPER + cb * C::SLAB + (row & 127) * 128, &qmap,
                                        cb * 64, kvh * G, zc[j], bar(C::B_Q_FULL));
                        }
                    }
                    cp_async_arrive(bar(C::B_Q_FULL));
                    continue;
                }
            }
            for (int tq = 0; tq < ntq; ++tq) {
                int qt[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 128 * tq + lane + 32 * i;
                    qt[i] = r < rows ? __ldg(a.members + it.member_off + r / G) : 0;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 128 * tq + lane + 32 * i;
                    const __nv_bfloat16 *qrow = qb + (((size_t)l * a.nq + qt[i]) * a.Hq + kvh * G + r % G) * D;
#pragma unroll
                    for (int c = 0; c < C::CH; ++c)
                        cp_async16(q_smem + tq * C::OPER + swz(r & 127, c), r < rows ? qrow + c * 8 : qb,
                                   r < rows ? 16 : 0);
                }
            }
            cp_async_arrive(bar(C::B_Q_FULL));
        }
        // the last Q load lands before the CTA ends (at once after a normal run)
        if (lane == 0 && last_q >= 0) settle(bar(C::B_Q_FULL), last_q & 1);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, kStepTokens, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, D, true);
            uint32_t gk = 0, gv = 0;        // steps taken from the K / V rings
            uint32_t np0 = 0, np1 = 0;      // P_FULL phases consumed per group
            for (int uc = 0;; ++uc) {
                const int slot = uc & 1;
                if (!wait(bar(C::B_UNIT_FULL + slot), (uc >> 1) & 1)) break;
                const int unit = s_unit[slot];
                if (unit < 0) break;
                const WorkItem it = a.tc_items[unit % n_items];
                const int ntile = it.tile_end - it.tile_begin;
                const int nsteps = (ntile + 1) >> 1;
                const bool pair = it.n_members * G > 128;
                bool ok = wait(bar(C::B_Q_FULL), uc & 1);
                // Q was written through the generic proxy (cp.async)
                fence_async_smem();
                tc_after();
                auto issue_s = [&](int t) -> bool {
                    const uint32_t g = gk + t, st = g % C::NK;
                    if (!wait(bar(C::B_K_FULL + st), (g / C::NK) & 1)) return false;
                    fence_async_smem();
                    tc_after();
                    const uint32_t kst = k_smem + st * C::OPER;
                    const uint32_t d_tm = tmem + C::S_COL + (t & 1) * kStepTokens;
                    const uint64_t qd = sdesc(q_smem, 16, 1024), kd = sdesc(kst, 16, 1024);
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t o = ((uint32_t)(k >> 2) * C::SLAB + (uint32_t)(k & 3) * 32) >> 4;
                        umma_ss(d_tm, qd + o, kd + o, IDESC_S, k > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(C::B_S_FULL + (t & 1)));
                    umma_commit(bar(C::B_K_EMPTY + st));
                    return true;
                };
                if (pair) {
                    // Two 128-row tiles over the same K/V: each step serves both,
                    // S_g and O_g belong to tile g, and group g takes every step.
                    auto wait_k = [&](int t) -> bool {
                        const uint32_t g = gk + t, st = g % C::NK;
                        if (!wait(bar(C::B_K_FULL + st), (g / C::NK) & 1)) return false;
                        fence_async_smem();
                        tc_after();
                        return true;
                    };
                    auto issue_sp = [&](int t, int tq) {
                        const uint32_t st = (gk + t) % C::NK;
                        const uint32_t kst = k_smem + st * C::OPER, qs = q_smem + tq * C::OPER;
                        const uint32_t d_tm = tmem + C::S_COL + tq * kStepTokens;
                        const uint64_t qd = sdesc(qs, 16, 1024), kd = sdesc(kst, 16, 1024);
#pragma unroll
                        for (int k = 0; k < D / 16; ++k) {
                            const uint32_t o = ((uint32_t)(k >> 2) * C::SLAB + (uint32_t)(k & 3) * 32) >> 4;
                            umma_ss(d_tm, qd + o, kd + o, IDESC_S, k > 0 ? 1u : 0u);
                        }
                        umma_commit(bar(C::B_S_FULL + tq));
                        if (tq == 1) umma_commit(bar(C::B_K_EMPTY + st));
                    };
                    if (ok && nsteps > 0) {
                        ok = wait_k(0);
                        if (ok) {
                            issue_sp(0, 0);
                            issue_sp(0, 1);
                        }
                    }
                    if (ok) ok = wait(bar(C::B_O_EMPTY), (uc & 1) ^ 1);
                    tc_after();
                    for (int t = 0; ok && t < nsteps; ++t) {
                        const uint32_t g = gv + t, st = g % C::NV;
                        const uint32_t vst = v_smem + st * C::OPER;
                        const int ksteps = 2 * t + 1 < ntile ? kStepTokens / 16 : kTileTokens / 16;
                        for (int tq = 0; ok && tq < 2; ++tq) {
                            if (!wait(bar(C::B_P_FULL + tq), (tq ? np1 : np0) & 1)) { ok = false; break; }
                            if (tq) ++np1; else ++np0;
                            if (tq == 0 && !wait(bar(C::B_V_FULL + st), (g / C::NV) & 1)) { ok = false; break; }
                            if (tq == 0) fence_async_smem();
                            tc_after();
                            const uint64_t vd = sdesc(vst, C::SLAB, 1024);
                            const uint32_t o_tm = tmem + C::O_COL + tq * D, p_tm = tmem + C::S_COL + tq * kStepTokens;
#pragma unroll
                            for (int k = 0; k < kStepTokens / 16; ++k)
                                if (k < ksteps)
                                    umma_ts(o_tm, p_tm + k * 8, vd + k * (2048 >> 4), IDESC_PV,
                                            (t > 0 || k > 0) ? 1u : 0u);
                            if (tq == 1) umma_commit(bar(C::B_V_EMPTY + st));
                            if (t + 1 < nsteps) {
                                if (tq == 0 && !wait_k(t + 1)) { ok = false; break; }
                                issue_sp(t + 1, tq);
                            }
                        }
                    }
                } else {
                if (ok && nsteps > 0) ok = issue_s(0);
                if (ok && nsteps > 1) ok = issue_s(1);
                // the previous unit's epilogue has read O_0 and O_1
                if (ok) ok = wait(bar(C::B_O_EMPTY), (uc & 1) ^ 1);
                tc_after();
                for (int t = 0; ok && t < nsteps; ++t) {
                    const int grp = t & 1;
                    if (!wait(bar(C::B_P_FULL + grp), (grp ? np1 : np0) & 1)) { ok = false; break; }
                    if (grp) ++np1; else ++np0;
                    const uint32_t g = gv + t, st = g % C::NV;
                    if (!wait(bar(C::B_V_FULL + st), (g / C::NV) & 1)) { ok = false; break; }
                    fence_async_smem();
                    tc_after();
                    const uint32_t vst = v_smem + st * C::OPER;
                    // an odd last tile leaves rows 64..127 of V unwritten: skip them
                    const int ksteps = 2 * t + 1 < ntile ? kStepTokens / 16 : kTileTokens / 16;
                    const uint64_t vd = sdesc(vst, C::SLAB, 1024);
                    const uint32_t o_tm = tmem + C::O_COL + grp * D, p_tm = tmem + C::S_COL + grp * kStepTokens;
#pragma unroll
                    for (int k = 0; k < kStepTokens / 16; ++k)
                        if (k < ksteps)
                            umma_ts(o_tm, p_tm + k * 8, vd + k * (2048 >> 4), IDESC_PV, (t >= 2 || k > 0) ? 1u : 0u);
                    umma_commit(bar(C::B_V_EMPTY + st));
                    if (t + 2 < nsteps && !issue_s(t + 2)) { ok = false; break; }
                }
                }
                if (!ok) break;
                // (with steps, the softmax thread that sees the unit's last S
                // releases Q)
                if (nsteps == 0) umma_commit(bar(C::B_Q_EMPTY));
                gk += nsteps;
                gv += nsteps;
                umma_commit(bar(C::B_O_FULL));
                mbar_arrive(bar(C::B_UNIT_EMPTY + slot));
            }
            // every MMA this thread issued completes before TMEM is freed
            umma_commit(bar(C::B_DRAIN));
            settle(bar(C::B_DRAIN), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int grp = (warp - kSoftWarp0) >> 2;
        const int quarter = warp & 3;             // TMEM lanes this warp may access
        const int r = quarter * 32 + lane;        // query row in the unit
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_tm = tmem + lane_base + C::S_COL + grp * kStepTokens;
        const uint32_t o_tm = tmem + lane_base + C::O_COL;
        const float sc = a.scale_log2;
        uint32_t ns = 0;   // S_FULL phases consumed by this group
        for (int uc = 0;; ++uc) {
            const int slot = uc & 1;
            bool ok = wait(bar(C::B_UNIT_FULL + slot), (uc >> 1) & 1);
            const int unit = ok ? s_unit[slot] : -1;
            if (soft_bar_or(!ok || unit < 0 || *s_abort)) break;
            const int item_idx = unit % n_items;
            const int lk = unit / n_items;
            const int kvh = lk % a.Hkv, l = lk / a.Hkv;
            const WorkItem it = a.tc_items[item_idx];
            const int ntile = it.tile_end - it.tile_begin;
            const int nsteps = (ntile + 1) >> 1;
            const KvTile *tiles = s_desc + slot * kMaxItemTiles;
            const int rows = it.n_members * G;
            // one tile: the groups split the steps over the same rows; a pair
            // unit: group g takes every step for the rows of tile g
            const bool pair = rows > 128;
            const int rr = pair ? 128 * grp + r : r;
            const bool has = rr < rows;
            const int mem = rr / G;
            int qt = 0;
            if (has) qt = __ldg(a.members + it.member_off + mem);
            const uint64_t tmask = has && a.tree_mask ? a.tree_mask[qt] : ~0ull;
            // a warp none of whose 32 rows is in the unit (a half-filled
            // 128-row tile) only keeps the group's barriers: the rows of P it
            // would write are never read back into an output row, since every
            // row of O depends on its own row of P alone
            const bool idle = !__any_sync(0xffffffffu, has);

            float m = -INFINITY, lsum = 0.f;
            for (int t = pair ? 0 : grp; t < nsteps; t += pair ? 1 : 2) {
                ok = wait(bar(C::B_S_FULL + grp), ns & 1) && ok;
                ns += 1;
                // the unit's last S is done with Q: one thread of the group
                // that takes it releases Q for the next unit's load, as soon
                // as that S is seen (measured slightly faster than releasing
                // it with an MMA commit)
                if (t == nsteps - 1 && grp == (pair ? 1 : (t & 1)) && quarter == 0 && lane == 0)
                    mbar_arrive(bar(C::B_Q_EMPTY));
                tc_after();
                if (idle) {
                    tc_before();
                    mbar_arrive(bar(C::B_P_FULL + grp));
                    continue;
                }
                int nv0 = 0, nv1 = 0;
                bool tr0 = false, tr1 = false;
                {
                    const KvTile &k0 = tiles[2 * t];
                    const int mlo = k0.members & 0xFFFF, mhi = k0.members >> 16;
                    nv0 = has && mem >= mlo && mem < mhi ? (k0.ntok_flags & 0xFFFF) : 0;
                    tr0 = (k0.ntok_flags >> 16) & kTileTree;
                }
                if (2 * t + 1 < ntile) {
                    const KvTile &k1 = tiles[2 * t + 1];
                    const int mlo = k1.members & 0xFFFF, mhi = k1.members >> 16;
                    nv1 = has && mem >= mlo && mem < mhi ? (k1.ntok_flags & 0xFFFF) : 0;
                    tr1 = (k1.ntok_flags >> 16) & kTileTree;
                }
                // A row's running max m is raised only when the step's P would
                // sum to more than 2^32, so every p <= 2^32, well inside bf16
                // and the fp32 sums.  A step therefore reads S once and forms P
                // with the current m, in registers; only a row whose sum breaks
                // the bound, or that has valid scores but no m yet, takes the
                // slow path (the step's max, O_g and l rescaled, P again)
                // before P overwrites S.
                if (__all_sync(0xffffffffu, m == -INFINITY)) {
                    // this group's first step of the unit: find m first
                    // (scale > 0: max of scaled scores = scale * max of raw scores)
                    m = step_max(s_tm, nv0, tr0, nv1, tr1, tmask) * sc;
                }
                float ls = 0.f;
                uint32_t pk[64];
                p_pass(s_tm, m == -INFINITY ? 0.f : -m, sc, nv0, tr0, nv1, tr1, tmask, pk, ls);
                const bool bad = m == -INFINITY ? (nv0 > 0 || nv1 > 0) : !(ls <= kSlackSum);
                if (!__any_sync(0xffffffffu, bad)) {
                    p_store(s_tm, pk);
                } else {
                    const float2 r2 = recompute_step(s_tm, m, sc, nv0, tr0, nv1, tr1, tmask, bad);
                    const bool resc = r2.x != m && m != -INFINITY;
                    if (__any_sync(0xffffffffu, resc)) {
                        // O_g holds P V up to step t-2, complete since S(t) is
                        const float f = resc ? exp2_sfu(m - r2.x) : 1.f;
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t x[32];
                            tmem_ld32(o_tm + grp * D + c0, x);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(__uint_as_float(x[j]) * f);
                            tmem_st32(o_tm + grp * D + c0, x);
                        }
                        lsum *= f;
                    }
                    m = r2.x;
                    ls = r2.y;
                }
                lsum += ls;
                tmem_wait_st();
                tc_before();
                mbar_arrive(bar(C::B_P_FULL + grp));
            }
            // epilogue: one tile merges the two groups' (m, l, O) and each
            // group writes half of the columns; in a pair unit each group
            // writes its own tile's rows from its own O
            ok = wait(bar(C::B_O_FULL), uc & 1) && ok;
            tc_after();
            s_ml[grp * 128 + r] = make_float2(m, lsum);
            if (soft_bar_or(!ok || *s_abort)) break;
            float w0, w1, lse2;
            int ca, cb;
            if (!pair) {
                const float2 a0 = s_ml[r], a1 = s_ml[128 + r];
                const float c = fmaxf(a0.x, a1.x);
                const float f0 = a0.x == -INFINITY ? 0.f : exp2_sfu(a0.x - c);
                const float f1 = a1.x == -INFINITY ? 0.f : exp2_sfu(a1.x - c);
                const float ltot = a0.y * f0 + a1.y * f1;
                const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
                lse2 = ltot > 0.f ? c + __log2f(ltot) : -INFINITY;
                w0 = f0 * inv;
                w1 = f1 * inv;
                ca = grp * (D / 2);
                cb = ca + D / 2;
            } else {
                const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                lse2 = lsum > 0.f ? m + __log2f(lsum) : -INFINITY;
                w0 = grp == 0 ? inv : 0.f;
                w1 = grp == 1 ? inv : 0.f;
                ca = 0;
                cb = D;
            }
            const bool write = has && nsteps > 0;
            for (int c0 = ca; !idle && c0 < cb; c0 += 32) {
                uint32_t x[32];
                if (pair) {   // this group's own tile: its O alone
                    tmem_ld32(o_tm + grp * D + c0, x);
                    tmem_wait_ld();
                    if (!write) continue;
                    const float w = grp ? w1 : w0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        x[j] = __float_as_uint(w != 0.f ? __uint_as_float(x[j]) * w : 0.f);
                } else {
                    uint32_t y[32];
                    tmem_ld32(o_tm + c0, x);
                    tmem_ld32(o_tm + D + c0, y);
                    tmem_wait_ld();
                    if (!write) continue;
                    // an O with weight 0 may never have been written (a group
                    // with no steps or no valid key): select, do not multiply
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float v0 = w0 != 0.f ? __uint_as_float(x[j]) * w0 : 0.f;
                        const float v1 = w1 != 0.f ? __uint_as_float(y[j]) * w1 : 0.f;
                        x[j] = __float_as_uint(v0 + v1);
                    }
                }
                if (it.out_base < 0 && !out32) {
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                         (((size_t)l * a.nq + qt) * a.Hq + kvh * G + rr % G) * D + c0;
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(x[j]), __uint_as_float(x[j + 1]));
                        v.y = pack_bf16x2(__uint_as_float(x[j + 2]), __uint_as_float(x[j + 3]));
                        v.z = pack_bf16x2(__uint_as_float(x[j + 4]), __uint_as_float(x[j + 5]));
                        v.w = pack_bf16x2(__uint_as_float(x[j + 6]), __uint_as_float(x[j + 7]));
                        *reinterpret_cast<uint4 *>(dst + j) = v;
                    }
                } else if (it.out_base < 0) {
                    // 32-byte stores when the output is 32-byte aligned (a row
                    // of D bf16 is a multiple of 128 bytes and c0 of 32
                    // columns): half the store instructions of 16-byte ones
                    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                         (((size_t)l * a.nq + qt) * a.Hq + kvh * G + rr % G) * D + c0;
#pragma unroll
                    for (int j = 0; j < 32; j += 16)
                        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"l"(dst + j),
                                     "r"(pack_bf16x2(__uint_as_float(x[j]), __uint_as_float(x[j + 1]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 2]), __uint_as_float(x[j + 3]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 4]), __uint_as_float(x[j + 5]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 6]), __uint_as_float(x[j + 7]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 8]), __uint_as_float(x[j + 9]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 10]), __uint_as_float(x[j + 11]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 12]), __uint_as_float(x[j + 13]))),
                                     "r"(pack_bf16x2(__uint_as_float(x[j + 14]), __uint_as_float(x[j + 15])))
                                     : "memory");
                } else {
                    // the workspace is 256-byte aligned: 32-byte stores
                    float *dst = a.part_o + (((size_t)l * a.Hkv + kvh) * a.P + it.out_base + rr) * D + c0;
#pragma unroll
                    for (int j = 0; j < 32; j += 8)
                        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"l"(dst + j),
                                     "r"(x[j]), "r"(x[j + 1]), "r"(x[j + 2]), "r"(x[j + 3]), "r"(x[j + 4]),
                                     "r"(x[j + 5]), "r"(x[j + 6]), "r"(x[j + 7])
                                     : "memory");
                }
            }
            if (write && (pair || grp == 0)) {
                if (it.out_base < 0) {
                    if (a.lse) a.lse[((size_t)l * a.nq + qt) * a.Hq + kvh * G + rr % G] = lse2 * 0.6931471805599453f;
                } else {
                    a.part_lse[((size_t)l * a.Hkv + kvh) * a.P + it.out_base + rr] = lse2;
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

struct TcOcc {
    int sms = 0;
    bool ok = false;
};

// Per device: the shared-memory attribute is set once for each device.
template <int D, bool KV4>
TcOcc &tc_occ() {
    static TcOcc occ[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    static TcOcc none;
    const int dev = current_device();
    if (dev < 0) return none;
    std::call_once(once[dev], [dev] {
        if (cudaFuncSetAttribute(attn_tc_kernel<D, KV4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcCfg<D>::SMEM) != cudaSuccess)
            return;
        occ[dev].sms = device_sm_count();
        occ[dev].ok = true;
    });
    return occ[dev];
}

template <int D, bool KV4>
cudaError_t launch_tc_d(const AttnLaunch &a, cudaStream_t stream) {
    TcOcc &occ = tc_occ<D, KV4>();
    if (!occ.ok) return cudaErrorInvalidDevice;
    const int bs = 1 << a.bs_log2;
    const int box_rows = bs < kTileTokens ? bs : kTileTokens;
    const long long rows = (long long)a.L * a.NB * a.Hkv * bs;
    alignas(64) CUtensorMap km, vm, qm;
    std::memset(&km, 0, sizeof km);
    std::memset(&vm, 0, sizeof vm);
    // (4-bit pages: the producers copy codes by cp.async, no pool maps)
    if (!KV4 && (!make_pool_map(&km, a.k_pool, D, rows, box_rows) || !make_pool_map(&vm, a.v_pool, D, rows, box_rows)))
        return cudaErrorInvalidValue;
    // Q boxes of max(8, G) rows must tile the 128-row operand
    const int G = a.G;
    const bool q_tma = (G <= 8 ? 8 % G == 0 : (G <= 128 && 128 % G == 0)) && make_q_map(&qm, a.q, D, a.Hq, (long long)a.L * a.nq, G);
    if (!q_tma) std::memset(&qm, 0, sizeof qm);
    // one CTA per SM (its shared memory and TMEM allow no more)
    const int grid = a.n_tc_units < occ.sms ? a.n_tc_units : occ.sms;
    const int out32 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0 ? 1 : 0;
    attn_tc_kernel<D, KV4><<<grid, kTcThreads, TcCfg<D>::SMEM, stream>>>(km, vm, qm, a, box_rows, q_tma ? 1 : 0, out32);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

namespace {

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

struct MapKey {
    const void *pool;
    long long rows;
    int D, box_rows;
};

}  // namespace

// 2-D view of a pool: rows = L*NB*Hkv*bs token rows of d bf16; box = 64
// columns x box_rows rows, 128-byte swizzle.  The last few maps built on
// this thread are kept, since every call on the same pool needs the same two.
bool make_pool_map(CUtensorMap *m, const void *pool, int D, long long rows, int box_rows) {
    constexpr int kCache = 4;
    thread_local MapKey keys[kCache] = {};
    thread_local CUtensorMap maps[kCache];
    thread_local int next = 0;
    for (int i = 0; i < kCache; ++i)
        if (keys[i].pool == pool && keys[i].rows == rows && keys[i].D == D && keys[i].box_rows == box_rows) {
            *m = maps[i];
            return true;
        }
    auto fn = encode_fn();
    if (!fn || !pool) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keys[next] = MapKey{pool, rows, D, box_rows};
    maps[next] = *m;
    next = (next + 1) % kCache;
    return true;
}

// 3-D view of the queries [L * nq tokens][Hq heads][D]; box = 64 columns x
// G heads x max(1, 8 / G) tokens, 128-byte swizzle.  Cached like the pool
// maps (the query buffer is usually the same from call to call).
bool make_q_map(CUtensorMap *m, const void *q, int D, int Hq, long long ntok, int G) {
    struct QKey {
        const void *q;
        long long ntok;
        int D, Hq, G;
    };
    constexpr int kCache = 4;
    thread_local QKey keys[kCache] = {};
    thread_local CUtensorMap maps[kCache];
    thread_local int next = 0;
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15) != 0 || ntok >= (1LL << 31) || G > Hq) return false;
    for (int i = 0; i < kCache; ++i)
        if (keys[i].q == q && keys[i].ntok == ntok && keys[i].D == D && keys[i].Hq == Hq && keys[i].G == G) {
            *m = maps[i];
            return true;
        }
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)ntok};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(G < 8 ? 8 / G : 1)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    keys[next] = QKey{q, ntok, D, Hq, G};
    maps[next] = *m;
    next = (next + 1) % kCache;
    return true;
}

bool tc_path_supported(int L, int NB, int Hkv, int bs) {
    // TMA row coordinates are 32-bit
    return (long long)L * NB * Hkv * bs < (1LL << 31);
}

cudaError_t launch_attention_tc(const AttnLaunch &a, cudaStream_t stream, int ctas_per_sm) {
    (void)ctas_per_sm;
    if (a.n_tc_units <= 0) return cudaSuccess;
    if (a.D == 64) return a.kv4 ? launch_tc_d<64, true>(a, stream) : launch_tc_d<64, false>(a, stream);
    if (a.D == 128) return a.kv4 ? launch_tc_d<128, true>(a, stream) : launch_tc_d<128, false>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace kvp
