// K/V write kernel (sm_103a): copy-on-write block copies and the scatter of
// appended tokens into their (block, slot), in one launch.
//
// Copy-on-write ("Dendrite" page, section details: blocks are shared until a
// branch writes and are copied only then): for each (source, copy, used)
// triple, the first `used` slots of every (layer, kv head) tile of the source
// block are copied into the copy block, K and V.  Because a tile is stored
// [bs][d], those slots are one contiguous run of used*d elements.
// The scatter writes token i of the append, [L][ntok][Hkv][d], to slot
// slots[i] = block*bs + slot.  The copies touch slots < used of the copy
// block and the scatter slots >= used, so both run in the same grid.
// Every thread moves 16-byte chunks (d is a multiple of 8).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "kvp_internal.h"

namespace kvp {
namespace {

constexpr int kMaxSlots = 4096;   // tokens per launch (16 KB of parameters)
constexpr int kMaxCow = 256;      // copy-on-write triples per launch
// Decode appends are a few tokens: a small parameter block for those, since
// every launch passes the whole block.
constexpr int kSmallSlots = 64, kSmallCow = 16;
constexpr int kMaxMoves = kMaxDraft;   // kept draft tokens per accept
constexpr int kMaxMoveCow = kMaxDraft; // blocks copied before the moves (bs 1: one per token)
constexpr int kMaxSegs = 4;            // buffers of one copy launch

template <int NS, int NC>
struct KvWriteArgs {
    uint4 *k_pool;
    uint4 *v_pool;
    const uint4 *k;
    const uint4 *v;
    int32_t L, NB, Hkv, bs, CH;       // CH = 16-byte chunks per head row (d / 8)
    int32_t ntok_total;               // tokens in k / v (row stride of the source)
    int32_t tok_begin, ntok;          // this launch's tokens
    int32_t ncow;
    int64_t cow_chunks;               // sum over triples of L*Hkv*used*CH
    int32_t cow[3 * NC];
    int32_t slots[NS];
};

// Chunk x of an append: x < 2 * cow_chunks copies a used slot of a
// copy-on-write block, the rest scatter the new tokens (even x: K, odd: V).
template <int NS, int NC>
__device__ __forceinline__ void kv_write_chunk(const KvWriteArgs<NS, NC> &a, int64_t x) {
    const int64_t tile = (int64_t)a.bs * a.CH;     // chunks per (block, head) tile
    const bool is_v = x & 1;
    int64_t y = x >> 1;
    uint4 *pool = is_v ? a.v_pool : a.k_pool;
    if (y < a.cow_chunks) {
        // find the triple (few per launch)
        int i = 0;
        int64_t per = 0;
        for (; i < a.ncow; ++i) {
            per = (int64_t)a.L * a.Hkv * a.cow[3 * i + 2] * a.CH;
            if (y < per) break;
            y -= per;
        }
        const int64_t run = (int64_t)a.cow[3 * i + 2] * a.CH;   // chunks per (layer, head)
        const int64_t lh = y / run, c = y % run;
        const int64_t l = lh / a.Hkv, h = lh % a.Hkv;
        const int64_t src = ((l * a.NB + a.cow[3 * i]) * a.Hkv + h) * tile + c;
        const int64_t dst = ((l * a.NB + a.cow[3 * i + 1]) * a.Hkv + h) * tile + c;
        pool[dst] = pool[src];
    } else {
        y -= a.cow_chunks;
        const int64_t c = y % a.CH;
        int64_t r = y / a.CH;
        const int64_t h = r % a.Hkv;
        r /= a.Hkv;
        const int64_t t = r % a.ntok;
        const int64_t l = r / a.ntok;
        const int32_t slot = a.slots[t];
        const int64_t blk = slot / a.bs, sl = slot % a.bs;
        const uint4 *srcp = is_v ? a.v : a.k;
        const int64_t src = ((l * a.ntok_total + a.tok_begin + t) * a.Hkv + h) * a.CH + c;
        const int64_t dst = ((l * a.NB + blk) * a.Hkv + h) * tile + sl * a.CH + c;
        pool[dst] = srcp[src];
    }
}

template <int NS, int NC>
__global__ void __launch_bounds__(256) kv_write_kernel(const __grid_constant__ KvWriteArgs<NS, NC> a) {
    const int64_t tok_chunks = (int64_t)a.L * a.ntok * a.Hkv * a.CH;
    const int64_t total = 2 * (a.cow_chunks + tok_chunks);
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x)
        kv_write_chunk(a, x);
}

// A decode step's inputs in one launch: the append (copy-on-write copies and
// the new tokens' K/V, read straight from page-locked host memory or from
// the device), q to its device buffer, and the attention plan, carried in
// the kernel's parameters, into the workspace.  The attention kernels that
// follow wait for this grid before they read anything, so it lets them
// launch at once.
template <int PB>
struct StepWriteArgs {
    KvWriteArgs<kSmallSlots, kSmallCow> w;
    const uint4 *q_src;
    uint4 *q_dst;
    int64_t q_chunks;
    uint4 *plan_dst;
    int32_t plan_chunks;
    uint4 plan[PB / 16];
};

template <int PB>
__global__ void __launch_bounds__(256) step_write_kernel(const __grid_constant__ StepWriteArgs<PB> s) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const KvWriteArgs<kSmallSlots, kSmallCow> &a = s.w;
    const int64_t kv_total = 2 * (a.cow_chunks + (int64_t)a.L * a.ntok * a.Hkv * a.CH);
    const int64_t q_end = kv_total + s.q_chunks, total = q_end + s.plan_chunks;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        if (x < kv_total)
            kv_write_chunk(a, x);
        else if (x < q_end)
            s.q_dst[x - kv_total] = s.q_src[x - kv_total];
        else
            s.plan_dst[x - q_end] = s.plan[x - q_end];
    }
}


// Speculative accept: move the kept draft tokens down to the positions right
// after the context.  One thread per (layer, kv head, 16-byte chunk of a
// token row), K and V.  It first copies its chunk of every copy-on-write
// block (all bs slots), then moves its chunk of each kept token in order.
// The i-th kept draft node has index >= i, so a token's source slot is never
// a slot that an earlier move of the same thread wrote: doing the moves in
// order needs no synchronisation, and threads touch disjoint memory.
struct KvMoveArgs {
    uint4 *k_pool;
    uint4 *v_pool;
    int32_t L, NB, Hkv, bs, CH;
    int32_t ncow, nmove;
    int32_t cow[2 * kMaxMoveCow];   // (source block, copy block)
    int32_t src[kMaxMoves];         // slots: block * bs + slot
    int32_t dst[kMaxMoves];
};

__global__ void __launch_bounds__(256) kv_move_kernel(const __grid_constant__ KvMoveArgs a) {
    const int64_t n = 2LL * a.L * a.Hkv * a.CH;
    const int64_t tile = (int64_t)a.bs * a.CH;     // chunks per (block, head) tile
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (int64_t)gridDim.x * blockDim.x) {
        uint4 *pool = (x & 1) ? a.v_pool : a.k_pool;
        const int64_t y = x >> 1;
        const int64_t c = y % a.CH, lh = y / a.CH;
        const int64_t h = lh % a.Hkv, l = lh / a.Hkv;
        const int64_t head = (l * a.NB * a.Hkv + h) * tile + c;    // + block * Hkv * tile + slot * CH
        const int64_t blk_stride = (int64_t)a.Hkv * tile;
        for (int i = 0; i < a.ncow; ++i)
            for (int sl = 0; sl < a.bs; ++sl)
                pool[head + a.cow[2 * i + 1] * blk_stride + sl * a.CH] =
                    pool[head + a.cow[2 * i] * blk_stride + sl * a.CH];
        for (int i = 0; i < a.nmove; ++i) {
            const int32_t s = a.src[i], d = a.dst[i];
            pool[head + (int64_t)(d / a.bs) * blk_stride + (d % a.bs) * a.CH] =
                pool[head + (int64_t)(s / a.bs) * blk_stride + (s % a.bs) * a.CH];
        }
    }
}

// One launch over tokens [tok_done, tok_done + ntok) and triples
// [cow_done, cow_done + ncow) with a parameter block of NS slots / NC triples.
template <int NS, int NC>
cudaError_t launch_part(const KvWrite &w, int cow_done, int ncow, int tok_done, int ntok, cudaStream_t stream) {
    // on the stack: kernel parameters are copied at launch, so calls on
    // different pools (or threads) never share this block
    KvWriteArgs<NS, NC> a;
    a.k_pool = static_cast<uint4 *>(w.k_pool);
    a.v_pool = static_cast<uint4 *>(w.v_pool);
    a.k = static_cast<const uint4 *>(w.k);
    a.v = static_cast<const uint4 *>(w.v);
    a.L = w.L; a.NB = w.NB; a.Hkv = w.Hkv; a.bs = w.bs; a.CH = w.d / 8;
    a.ntok_total = w.ntok;
    a.ncow = ncow;
    a.cow_chunks = 0;
    for (int i = 0; i < ncow; ++i) {
        a.cow[3 * i] = w.cow[3 * (cow_done + i)];
        a.cow[3 * i + 1] = w.cow[3 * (cow_done + i) + 1];
        a.cow[3 * i + 2] = w.cow[3 * (cow_done + i) + 2];
        a.cow_chunks += (int64_t)w.L * w.Hkv * a.cow[3 * i + 2] * a.CH;
    }
    a.tok_begin = tok_done;
    a.ntok = ntok;
    for (int i = 0; i < ntok; ++i) a.slots[i] = w.slots[tok_done + i];
    const int64_t total = 2 * (a.cow_chunks + (int64_t)w.L * ntok * w.Hkv * a.CH);
    const int64_t want = (total + 255) / 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)device_sm_count() * 16));
    kv_write_kernel<NS, NC><<<blocks, 256, 0, stream>>>(a);
    count_launch();
    return cudaGetLastError();
}

// Copies up to kMaxSegs buffers in one launch, through the SMs: a decode
// step's inputs from page-locked host memory.  Every segment is 16-byte
// aligned; whole 16-byte chunks first, then the last bytes (a multiple of 4)
// one word at a time.
struct CopySegs {
    const void *src[kMaxSegs];
    void *dst[kMaxSegs];
    int64_t bytes[kMaxSegs];
    int32_t n;
};

__global__ void __launch_bounds__(256) copy_segs_kernel(const __grid_constant__ CopySegs c) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int s = 0; s < c.n; ++s) {
        const int64_t n16 = c.bytes[s] >> 4;
        const uint4 *src = static_cast<const uint4 *>(c.src[s]);
        uint4 *dst = static_cast<uint4 *>(c.dst[s]);
        for (int64_t i = t0; i < n16; i += stride) dst[i] = src[i];
        const int64_t w0 = n16 * 4, nw = c.bytes[s] >> 2;
        const uint32_t *sw = static_cast<const uint32_t *>(c.src[s]);
        uint32_t *dw = static_cast<uint32_t *>(c.dst[s]);
        for (int64_t i = w0 + t0; i < nw; i += stride) dw[i] = sw[i];
    }
}

}  // namespace

cudaError_t launch_copy_segments(const void *const *src, void *const *dst, const int64_t *bytes, int n,
                                 cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    if (n > kMaxSegs) return cudaErrorInvalidValue;
    CopySegs c{};
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        c.src[i] = src[i];
        c.dst[i] = dst[i];
        c.bytes[i] = bytes[i];
        total += bytes[i];
    }
    c.n = n;
    // about one 16-byte chunk per thread, at most two CTAs per SM
    const int64_t want = (total / 16 + 255) / 256;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, 2LL * device_sm_count()));
    copy_segs_kernel<<<grid, 256, 0, stream>>>(c);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_kv_move(const KvMove &m, cudaStream_t stream) {
    if (m.ncow == 0 && m.nmove == 0) return cudaSuccess;
    if (m.ncow > kMaxMoveCow || m.nmove > kMaxMoves || m.d % 8 != 0) return cudaErrorInvalidValue;
    KvMoveArgs a{};
    a.k_pool = static_cast<uint4 *>(m.k_pool);
    a.v_pool = static_cast<uint4 *>(m.v_pool);
    a.L = m.L; a.NB = m.NB; a.Hkv = m.Hkv; a.bs = m.bs; a.CH = m.d / 8;
    a.ncow = m.ncow;
    a.nmove = m.nmove;
    for (int i = 0; i < 2 * m.ncow; ++i) a.cow[i] = m.cow[i];
    for (int i = 0; i < m.nmove; ++i) {
        a.src[i] = m.src[i];
        a.dst[i] = m.dst[i];
    }
    const int64_t n = 2LL * m.L * m.Hkv * a.CH;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)device_sm_count() * 16));
    kv_move_kernel<<<blocks, 256, 0, stream>>>(a);
    count_launch();
    return cudaGetLastError();
}

template <int PB>
cudaError_t launch_step_write_pb(const KvWrite &w, const void *q_src, void *q_dst, size_t q_bytes,
                                 const void *plan, void *plan_dst, size_t plan_bytes, cudaStream_t stream) {
    // on the stack: parameters are copied at launch
    StepWriteArgs<PB> s;
    KvWriteArgs<kSmallSlots, kSmallCow> &a = s.w;
    a.k_pool = static_cast<uint4 *>(w.k_pool);
    a.v_pool = static_cast<uint4 *>(w.v_pool);
    a.k = static_cast<const uint4 *>(w.k);
    a.v = static_cast<const uint4 *>(w.v);
    a.L = w.L; a.NB = w.NB; a.Hkv = w.Hkv; a.bs = w.bs; a.CH = w.d / 8;
    a.ntok_total = w.ntok;
    a.ncow = w.ncow;
    a.cow_chunks = 0;
    for (int i = 0; i < w.ncow; ++i) {
        a.cow[3 * i] = w.cow[3 * i];
        a.cow[3 * i + 1] = w.cow[3 * i + 1];
        a.cow[3 * i + 2] = w.cow[3 * i + 2];
        a.cow_chunks += (int64_t)w.L * w.Hkv * a.cow[3 * i + 2] * a.CH;
    }
    a.tok_begin = 0;
    a.ntok = w.ntok;
    for (int i = 0; i < w.ntok; ++i) a.slots[i] = w.slots[i];
    s.q_src = static_cast<const uint4 *>(q_src);
    s.q_dst = static_cast<uint4 *>(q_dst);
    s.q_chunks = q_src ? (int64_t)(q_bytes / 16) : 0;
    s.plan_dst = static_cast<uint4 *>(plan_dst);
    s.plan_chunks = (int32_t)(plan_bytes / 16);
    std::memcpy(s.plan, plan, plan_bytes);
    const int64_t total = 2 * (a.cow_chunks + (int64_t)w.L * w.ntok * w.Hkv * a.CH) + s.q_chunks + s.plan_chunks;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)device_sm_count() * 4));
    step_write_kernel<PB><<<blocks, 256, 0, stream>>>(s);
    count_launch();
    return cudaGetLastError();
}

bool step_write_fits(const KvWrite &w, size_t plan_bytes) {
    return w.ntok <= kSmallSlots && w.ncow <= kSmallCow && plan_bytes <= kStepPlanMax && plan_bytes % 16 == 0 &&
           w.d % 8 == 0;
}

cudaError_t launch_step_write(const KvWrite &w, const void *q_src, void *q_dst, size_t q_bytes, const void *plan,
                              void *plan_dst, size_t plan_bytes, cudaStream_t stream) {
    if (!step_write_fits(w, plan_bytes) || q_bytes % 16 != 0) return cudaErrorInvalidValue;
    if (plan_bytes <= 8192)
        return launch_step_write_pb<8192>(w, q_src, q_dst, q_bytes, plan, plan_dst, plan_bytes, stream);
    return launch_step_write_pb<kStepPlanMax>(w, q_src, q_dst, q_bytes, plan, plan_dst, plan_bytes, stream);
}

cudaError_t launch_kv_write(const KvWrite &w, cudaStream_t stream) {
    if (w.ncow == 0 && w.ntok == 0) return cudaSuccess;
    if (w.ntok <= kSmallSlots && w.ncow <= kSmallCow)
        return launch_part<kSmallSlots, kSmallCow>(w, 0, w.ncow, 0, w.ntok, stream);
    int cow_done = 0, tok_done = 0;
    while (cow_done < w.ncow || tok_done < w.ntok) {
        const int ncow = std::min(kMaxCow, w.ncow - cow_done), ntok = std::min(kMaxSlots, w.ntok - tok_done);
        cudaError_t e = launch_part<kMaxSlots, kMaxCow>(w, cow_done, ncow, tok_done, ntok, stream);
        if (e != cudaSuccess) return e;
        cow_done += ncow;
        tok_done += ntok;
    }
    return cudaSuccess;
}

}  // namespace kvp
