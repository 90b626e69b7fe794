// Debug-build input checks.
//
// Every kernel here relies on two preconditions that the host cannot check, because the data
// lives in device memory:
//   - the log decay is bounded, g in [-5, 0] ("はじめての自然言語処理 -- Kimi K3", section 3.1:
//     g = -5 sigmoid(x); the tensor-core kernels keep a 16-token cumulative decay within e^-80
//     on the strength of it);
//   - packed offsets satisfy 0 = cu[0] <= cu[1] <= ... <= cu[N] = seqlen.
// A library built with KDA_DEBUG_CHECKS (build.build(debug=True) -> libkda_debug.so) checks both
// on the device before a call's kernels run and records a failure as a bit in a device-wide
// error word; kda_device_status reports it as KDA_ERR_INPUT.  Nothing traps and the call still
// runs (its results are then unspecified, as for any input outside the preconditions).  The
// release library compiles the error word and its reader but launches no check.
#include <cuda_bf16.h>

#include "kda_internal.h"

__device__ unsigned int g_kda_input_errors = 0;

namespace kda {
namespace {

#ifdef KDA_DEBUG_CHECKS
constexpr unsigned int kErrDecay = 1u, kErrOffsets = 2u;   // bits of the error word
constexpr int kCheckThreads = 256;

// Flags any g outside [-5, 0] (NaN included) among n elements.
__global__ void __launch_bounds__(kCheckThreads) check_decay_kernel(const void *g, int64_t n, int is_bf16) {
    bool bad = false;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float x = is_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(g)[i])
                                : static_cast<const float *>(g)[i];
        bad |= !(x >= -5.f && x <= 0.f);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(&g_kda_input_errors, kErrDecay);
}

// Flags offsets that do not start at 0, decrease, leave [0, seqlen] or do not end at seqlen.
__global__ void __launch_bounds__(kCheckThreads) check_offsets_kernel(const int32_t *cu, int n, int64_t seqlen) {
    bool bad = false;
    for (int i = threadIdx.x; i <= n; i += blockDim.x) {
        const int64_t c = cu[i];
        bad |= c < 0 || c > seqlen || (i > 0 && cu[i - 1] > c) || (i == 0 && c != 0) ||
               (i == n && c != seqlen);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(&g_kda_input_errors, kErrOffsets);
}
#endif

}  // namespace

cudaError_t debug_check_inputs(const void *g, int64_t g_elems, kda_dtype_t dt, const int32_t *cu,
                               int num_seqs, int64_t seqlen, cudaStream_t st) {
#ifdef KDA_DEBUG_CHECKS
    if (g != nullptr && g_elems > 0) {
        const int64_t blocks = (g_elems + 4 * kCheckThreads - 1) / (4 * kCheckThreads);
        check_decay_kernel<<<(unsigned)(blocks < 1024 ? blocks : 1024), kCheckThreads, 0, st>>>(
            g, g_elems, dt == KDA_BF16);
    }
    if (cu != nullptr) check_offsets_kernel<<<1, kCheckThreads, 0, st>>>(cu, num_seqs, seqlen);
    return cudaGetLastError();
#else
    (void)g, (void)g_elems, (void)dt, (void)cu, (void)num_seqs, (void)seqlen, (void)st;
    return cudaSuccess;
#endif
}

int debug_checks_built() {
#ifdef KDA_DEBUG_CHECKS
    return (int)(kErrDecay | kErrOffsets);
#else
    return 0;
#endif
}

cudaError_t take_input_errors(cudaStream_t st, unsigned int *bits) {
    static const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(bits, g_kda_input_errors, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_kda_input_errors, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

}  // namespace kda
