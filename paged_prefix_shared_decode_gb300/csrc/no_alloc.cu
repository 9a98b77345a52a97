// paged_decode_attention_noalloc: decode attention whose workspace lives in
// the library itself instead of in memory the caller allocates.
//
// Who needs this: callers that cannot allocate device memory when they
// attend.  A serving process whose memory manager has already handed
// (nearly) all device memory to its own pools has nothing left to give a
// workspace; a plug-in running inside a host program cannot reach that
// program's allocator and must not go around it with cudaMalloc.  Such a
// caller passes inputs and outputs only; the scratch space (the uploaded
// work plan, the two work counters, the error word and the partial rows of
// split key ranges) is a fixed array that is part of the library image.
//
// Costs and limits:
//   - the array is KVP_STATIC_WORKSPACE_BYTES (32 MiB) on every GPU that loads
//     the library, held until the process exits;
//   - a batch whose plan needs more than that is rejected (KVP_ERR_INVALID)
//     before anything is enqueued; kvp_decode_workspace_size() tells the
//     size a batch needs;
//   - every call on a device uses the same array, so calls that overlap on the
//     GPU (two streams, two threads) race and corrupt each other; serialise
//     them.  The array keeps the previous call's contents: the parts that must
//     start at zero (the error word and the work counters) are rewritten by
//     each call's plan upload before its kernels run, and partial rows are
//     written before they are read;
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture.
// Nothing here calls cudaMalloc, cudaFree or any other allocating routine;
// planning uses ordinary host memory, as the other entry points do.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/kvp.h"
#include "kvp_internal.h"

namespace {

constexpr size_t kScratchBytes = KVP_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The workspace.  Device code could name it directly; host code must use the
// address that cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return KVP_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return KVP_OK;
}

}  // namespace

extern "C" int paged_decode_attention_noalloc(const void *q, const void *k_pool, const void *v_pool,
                                              const int32_t *block_tables, const int32_t *seq_lens,
                                              int32_t num_seqs, int32_t max_blocks,
                                              const kvp_attn_desc *desc, void *out, float *lse,
                                              void *stream) {
    // paged_decode_attention plans once and rejects a plan larger than the
    // workspace it is given (KVP_ERR_INVALID) before it enqueues anything
    void *ws = nullptr;
    int rc = scratch_address(&ws);
    if (rc != KVP_OK) return rc;
    return paged_decode_attention(q, k_pool, v_pool, block_tables, seq_lens, num_seqs, max_blocks,
                                  desc, out, lse, ws, kScratchBytes, stream);
}
