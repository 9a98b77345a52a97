// 4-bit K/V pages (sm_103a): quantise-on-append with copy-on-write, in one
// launch.
//
// Format ("Dendrite" page, section on FlashInfer kernels and TurboQuant
// integration: 4-bit KV that cuts KV memory 3.88x at head dim 64 and is
// computed on directly; the pages leave the quantiser open).  Each (token,
// kv head) row of d values is stored as d signed 4-bit codes in [-7, 7] and
// one power-of-two scale 2^e, e an int8 in [-127, 127]:
//   e      = the smallest integer with max|x| <= 7 * 2^e (-127 for a zero row)
//   code   = round-half-even(x / 2^e)
//   x'     = code * 2^e
// That is 4 + 8 / d bits per value: 4.125 at d = 64 (16 / 4.125 = 3.88x).
// Layout: codes [L][NB][Hkv][bs][d/2] bytes, element 2i in the low nibble of
// byte i, element 2i+1 in the high nibble (two's complement); exponents
// [L][NB][Hkv][bs] int8.  One (block, kv head) tile is bs * d/2 code bytes
// and bs exponent bytes, each contiguous.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kvp_internal.h"

namespace kvp {
namespace {

constexpr int kMaxSlots4 = 4096;   // tokens per launch
constexpr int kMaxCow4 = 256;      // copy-on-write triples per launch

template <int NS, int NC>
struct Kv4WriteArgs {
    uint8_t *k_codes, *v_codes;
    int8_t *k_exp, *v_exp;
    const uint16_t *k, *v;          // appended bf16 [L][ntok_total][Hkv][d]
    int32_t L, NB, Hkv, bs, d;
    int32_t ntok_total, tok_begin, ntok;
    int32_t ncow;
    int32_t cow[3 * NC];            // (source block, copy block, used slots)
    int32_t slots[NS];              // block * bs + slot per token
};

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// e = smallest integer with m <= 7 * 2^e for m > 0, clamped to [-127, 127]:
// m in [2^E, 2^(E+1)) needs e = E - 2 when m <= 1.75 * 2^E, else E - 1 (both
// sides exact in fp32).
__device__ __forceinline__ int row_exponent(float m) {
    if (!(m > 0.f)) return -127;
    int E;
    const float f = frexpf(m, &E);   // m = f * 2^E, f in [0.5, 1)
    E -= 1;                          // m in [2^E, 2^(E+1))
    const int e = (f * 2.f <= 1.75f) ? E - 2 : E - 1;
    return max(-127, min(127, e));
}

// One warp per (layer, head, unit): a copy-on-write triple's rows, or one
// appended token's row (quantised).
template <int NS, int NC>
__global__ void __launch_bounds__(256) kv4_write_kernel(const __grid_constant__ Kv4WriteArgs<NS, NC> a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t lh = (int64_t)a.L * a.Hkv;
    const int64_t cow_units = lh * a.ncow;
    const int64_t tok_units = lh * a.ntok;
    const int rowb = a.d / 2;          // code bytes per row
    const int64_t tile_rows = a.bs;    // rows per (block, head) tile
    for (int64_t u = warp; u < 2 * (cow_units + tok_units); u += nwarps) {
        const bool is_v = u & 1;
        const int64_t y = u >> 1;
        uint8_t *codes = is_v ? a.v_codes : a.k_codes;
        int8_t *exps = is_v ? a.v_exp : a.k_exp;
        if (y < cow_units) {
            const int i = (int)(y / lh);
            const int64_t r = y % lh;
            const int64_t l = r / a.Hkv, h = r % a.Hkv;
            const int src = a.cow[3 * i], dst = a.cow[3 * i + 1], used = a.cow[3 * i + 2];
            const int64_t so = ((l * a.NB + src) * a.Hkv + h) * tile_rows;
            const int64_t dO = ((l * a.NB + dst) * a.Hkv + h) * tile_rows;
            for (int x = lane; x < used * rowb; x += 32) codes[dO * rowb + x] = codes[so * rowb + x];
            for (int x = lane; x < used; x += 32) exps[dO + x] = exps[so + x];
            continue;
        }
        const int64_t z = y - cow_units;
        const int64_t h = z % a.Hkv, lt = z / a.Hkv;
        const int64_t t = lt % a.ntok, l = lt / a.ntok;
        const uint16_t *src = (is_v ? a.v : a.k) + ((l * a.ntok_total + a.tok_begin + t) * a.Hkv + h) * a.d;
        const int slot = a.slots[t];
        const int64_t blk = slot / a.bs, sl = slot % a.bs;
        const int64_t row = ((l * a.NB + blk) * a.Hkv + h) * tile_rows + sl;
        // lane owns values 2*lane, 2*lane+1 (d 64) or 4*lane .. 4*lane+3 (d 128)
        const int vpl = a.d / 32;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t amax = 0;
        for (int j = 0; j < vpl; ++j) {
            x[j] = bf16_bits_to_float(src[lane * vpl + j]);
            amax = max(amax, __float_as_uint(fabsf(x[j])));
        }
        amax = __reduce_max_sync(0xffffffffu, amax);   // |x| bit patterns order like the values
        const int e = row_exponent(__uint_as_float(amax));
        uint32_t packed = 0;
        for (int j = 0; j < vpl; ++j) {
            const float c = fminf(7.f, fmaxf(-7.f, rintf(ldexpf(x[j], -e))));
            packed |= ((uint32_t)(int)c & 0xFu) << (4 * j);
        }
        if (vpl == 2) {
            codes[row * rowb + lane] = (uint8_t)packed;
        } else {
            reinterpret_cast<uint16_t *>(codes + row * rowb)[lane] = (uint16_t)packed;
        }
        if (lane == 0) exps[row] = (int8_t)e;
    }
}

// Speculative accept on a 4-bit pool: copy-on-write copies of whole blocks,
// then the kept draft rows moved down in order.  One warp per (layer, kv
// head), K and V: the warp does every copy and move of its tile in order, so
// a source row is never one that an earlier move of the same warp wrote.
struct Kv4MoveArgs {
    uint8_t *k_codes, *v_codes;
    int8_t *k_exp, *v_exp;
    int32_t L, NB, Hkv, bs, d;
    int32_t ncow, nmove;
    int32_t cow[2 * kMaxDraft];
    int32_t src[kMaxDraft];
    int32_t dst[kMaxDraft];
};

__global__ void __launch_bounds__(256) kv4_move_kernel(const __grid_constant__ Kv4MoveArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t lh = (int64_t)a.L * a.Hkv;
    if (warp >= 2 * lh) return;
    const bool is_v = warp & 1;
    const int64_t r = warp >> 1;
    const int64_t l = r / a.Hkv, h = r % a.Hkv;
    uint8_t *codes = is_v ? a.v_codes : a.k_codes;
    int8_t *exps = is_v ? a.v_exp : a.k_exp;
    const int rowb = a.d / 2;
    auto row_of = [&](int blk, int sl) { return ((l * a.NB + blk) * a.Hkv + h) * (int64_t)a.bs + sl; };
    for (int i = 0; i < a.ncow; ++i) {
        const int64_t s0 = row_of(a.cow[2 * i], 0), d0 = row_of(a.cow[2 * i + 1], 0);
        for (int x = lane; x < a.bs * rowb; x += 32) codes[d0 * rowb + x] = codes[s0 * rowb + x];
        for (int x = lane; x < a.bs; x += 32) exps[d0 + x] = exps[s0 + x];
        __syncwarp();
    }
    for (int i = 0; i < a.nmove; ++i) {
        const int64_t s = row_of(a.src[i] / a.bs, a.src[i] % a.bs), d = row_of(a.dst[i] / a.bs, a.dst[i] % a.bs);
        for (int x = lane; x < rowb; x += 32) codes[d * rowb + x] = codes[s * rowb + x];
        if (lane == 0) exps[d] = exps[s];
        __syncwarp();
    }
}

template <int NS, int NC>
cudaError_t launch_part4(const Kv4Write &w, int cow_done, int ncow, int tok_done, int ntok, cudaStream_t stream) {
    Kv4WriteArgs<NS, NC> a;   // on the stack: parameters are copied at launch
    a.k_codes = static_cast<uint8_t *>(w.k_codes);
    a.v_codes = static_cast<uint8_t *>(w.v_codes);
    a.k_exp = static_cast<int8_t *>(w.k_exp);
    a.v_exp = static_cast<int8_t *>(w.v_exp);
    a.k = static_cast<const uint16_t *>(w.k);
    a.v = static_cast<const uint16_t *>(w.v);
    a.L = w.L; a.NB = w.NB; a.Hkv = w.Hkv; a.bs = w.bs; a.d = w.d;
    a.ntok_total = w.ntok;
    a.tok_begin = tok_done;
    a.ntok = ntok;
    a.ncow = ncow;
    for (int i = 0; i < 3 * ncow; ++i) a.cow[i] = w.cow[3 * cow_done + i];
    for (int i = 0; i < ntok; ++i) a.slots[i] = w.slots[tok_done + i];
    const int64_t warps = 2LL * w.L * w.Hkv * (ncow + ntok);
    const int64_t want = (warps * 32 + 255) / 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)device_sm_count() * 16));
    kv4_write_kernel<NS, NC><<<blocks, 256, 0, stream>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv4_write(const Kv4Write &w, cudaStream_t stream) {
    if (w.ncow == 0 && w.ntok == 0) return cudaSuccess;
    if (w.d != 64 && w.d != 128) return cudaErrorInvalidValue;
    if (w.ntok <= 64 && w.ncow <= 16) return launch_part4<64, 16>(w, 0, w.ncow, 0, w.ntok, stream);
    int cow_done = 0, tok_done = 0;
    while (cow_done < w.ncow || tok_done < w.ntok) {
        const int ncow = std::min(kMaxCow4, w.ncow - cow_done), ntok = std::min(kMaxSlots4, w.ntok - tok_done);
        cudaError_t e = launch_part4<kMaxSlots4, kMaxCow4>(w, cow_done, ncow, tok_done, ntok, stream);
        if (e != cudaSuccess) return e;
        cow_done += ncow;
        tok_done += ntok;
    }
    return cudaSuccess;
}

cudaError_t launch_kv4_move(const Kv4Move &m, cudaStream_t stream) {
    if (m.ncow == 0 && m.nmove == 0) return cudaSuccess;
    if (m.ncow > kMaxDraft || m.nmove > kMaxDraft || (m.d != 64 && m.d != 128)) return cudaErrorInvalidValue;
    Kv4MoveArgs a{};
    a.k_codes = static_cast<uint8_t *>(m.k_codes);
    a.v_codes = static_cast<uint8_t *>(m.v_codes);
    a.k_exp = static_cast<int8_t *>(m.k_exp);
    a.v_exp = static_cast<int8_t *>(m.v_exp);
    a.L = m.L; a.NB = m.NB; a.Hkv = m.Hkv; a.bs = m.bs; a.d = m.d;
    a.ncow = m.ncow;
    a.nmove = m.nmove;
    for (int i = 0; i < 2 * m.ncow; ++i) a.cow[i] = m.cow[i];
    for (int i = 0; i < m.nmove; ++i) {
        a.src[i] = m.src[i];
        a.dst[i] = m.dst[i];
    }
    const int64_t warps = 2LL * m.L * m.Hkv;
    kv4_move_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(a);
    count_launch();
    return cudaGetLastError();
}

}  // namespace kvp
