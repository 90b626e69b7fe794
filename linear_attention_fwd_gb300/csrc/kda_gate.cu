// The KDA output gate as a separate pass over a chunk call's stored outputs (the path the
// tensor-core kernel does not cover; that kernel applies the gate while staging its output).
//
// "はじめての自然言語処理 -- Kimi K3", the paragraph after the decay bound: the read-out is
// normalised by RMSNorm over its value channels (so that the magnitude of what is read from S
// is evened out), then multiplied channel by channel by a gate in (0, 1) made from the token's
// input:  y = o / sqrt(mean_j o_j^2 + eps) * w * sigmoid(z).
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

// One warp per (token, head) row; dv / 32 channels per lane.
template <typename T, int DV>
__global__ void __launch_bounds__(256) kda_gate_pass_kernel(T *out, const T *gate, const float *w,
                                                             float eps, int64_t rows) {
    constexpr int PER = DV / 32;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    T *o = out + row * DV;
    const T *z = gate + row * DV;
    float x[PER], ss = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        x[e] = to_f(o[lane + 32 * e]);
        ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
    const float rstd = rsqrtf(ss / DV + eps);
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int j = lane + 32 * e;
        const float gz = __fdividef(1.f, 1.f + __expf(-to_f(z[j])));
        o[j] = from_f<T>(x[e] * rstd * (w ? w[j] : 1.f) * gz);
    }
}

template <typename T, int DV>
cudaError_t launch_t(const ChunkArgs &a, int64_t rows, cudaStream_t st) {
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    kda_gate_pass_kernel<T, DV><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<T *>(a.out), static_cast<const T *>(a.gate), a.norm_w, a.norm_eps, rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_pass(const ChunkArgs &a, int64_t tokens, int dv, kda_dtype_t dt,
                             cudaStream_t st) {
    const int64_t rows = tokens * a.heads;
    if (rows == 0) return cudaSuccess;
    if (dt == KDA_F32) return dv == 128 ? launch_t<float, 128>(a, rows, st) : launch_t<float, 64>(a, rows, st);
    return dv == 128 ? launch_t<__nv_bfloat16, 128>(a, rows, st) : launch_t<__nv_bfloat16, 64>(a, rows, st);
}

}  // namespace kda
