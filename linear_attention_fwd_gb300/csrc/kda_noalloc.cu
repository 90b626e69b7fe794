// kda_chunk_fwd_noalloc: the two-pass prefill (kda_chunk_fwd_ws) over a scratch area that is
// part of this library's device image, so that the call itself allocates no memory.
//
// Who needs it: a caller that cannot hand the library device memory when it calls.  A host
// that reserved its whole device budget at start-up and may not grow it inside its serving
// loop; a plain C host with no device allocator of its own; a latency-bound loop that cannot
// take the device-wide synchronisation cudaMalloc and cudaFree bring with them.  None of these
// can allocate a workspace per call, and a caching allocator is not something each of them has.
//
// The scratch area is one file-scope __device__ array of KDA_NOALLOC_SCRATCH_BYTES bytes; each
// device that loads this module holds its own copy.  Its address on a device is looked up once,
// the first time the call runs with that device current, and kept; later calls on that device
// only read the kept address.  Nothing in the area has to start at zero: each call's first
// kernel writes the chunk offsets at its head, the chunk-parallel pass then writes every
// per-chunk slot the state pass reads, and nothing is carried from one call to the next.
// Because there is one area per device, calls that overlap in time on a device (two streams,
// two host threads) race on it: the caller keeps them apart.
#include "kda_internal.h"

#include <mutex>

// 256-byte alignment covers the 16 bytes the TMA copies of the two passes need.
static __device__ __align__(256) unsigned char g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices];   // the area's address per device ordinal; null until looked up

// The scratch area's address on the current device: looked up (cudaGetSymbolAddress, which also
// loads this module on the device when that has not happened yet) on the first call with this
// device current, and kept.
cudaError_t scratch_of_current_device(void **ptr) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_kda_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status_t kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                              const void *g, const void *beta,
                                              const float *initial_state, const int32_t *cu_seqlens,
                                              void *out, float *final_state, const kda_dims_t *d,
                                              cudaStream_t stream) {
    // the size check comes first, so that a call that does not fit is rejected before any
    // device state (the address lookup included) is touched
    if (d == nullptr) return KDA_ERR_NULL;
    const size_t need = kda_chunk_fwd_workspace_bytes(d);
    if (need > KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (scratch_of_current_device(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    return kda_chunk_fwd_ws(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                            scratch, KDA_NOALLOC_SCRATCH_BYTES, d, stream);
}
