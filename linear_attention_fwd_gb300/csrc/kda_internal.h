// Internal declarations shared by libkda's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/kda.h"

namespace kda {

// Chunk length and sub-tile length of the chunkwise form.  A 16-token sub-tile
// keeps every decay factor the kernels form inside [e^-80, e^80] under g >= -5.
constexpr int kChunk = 64;
constexpr int kSub = 16;

struct ChunkArgs {
    const void *q, *k, *v, *g, *beta;
    const float *s0;          // [N, H, dk, dv] or nullptr
    const int32_t *cu;        // [N + 1] or nullptr (dense)
    void *out;
    float *sT;                // [N, H, dk, dv] or nullptr
    int64_t seqlen;           // tokens per dense row, or total packed tokens
    int32_t num_seqs;         // N
    int32_t heads;            // H
    const void *gate;         // [tokens, H, dv] gate logits (io dtype), or nullptr: no output gate
    const float *norm_w;      // [dv] RMSNorm weight, or nullptr (ones)
    float norm_eps;           // RMSNorm epsilon
    float *ckpt;              // [slots, H, dk, dv] state checkpoints, or nullptr
    const int32_t *ckpt_off;  // [N + 1]: sequence n's checkpoints occupy slots [off[n], off[n+1])
    int32_t ckpt_interval;    // tokens between checkpoints (a multiple of the chunk)
    uint32_t wait_polls;      // bound on each device wait of the tensor-core kernel (polls)
    int32_t segments;         // tensor-core kernel: CTAs per (sequence, head), 0 = chosen by the launcher
    int32_t sched_ctas = 0;   // tensor-core kernel: CTAs of the balanced schedule (set by the launcher), or 0
    int32_t dk = 128, dv = 128;   // head sizes in memory (the tensor-core kernel computes at 128 and
                                  // reads the missing channels of a 64-wide head as zeros)
    float qk_eps = -1.f;          // >= 0: q and k rows are L2-normalised first, x / sqrt(|x|^2 + eps)
                                  // in fp32 (a row with |x|^2 + eps = 0 stays zero)
};

// Checkpoint slot for the state after `pos` tokens of sequence n (pos > 0 a multiple of the
// chunk), or -1 when none is due there.
__device__ __forceinline__ int64_t ckpt_slot(const ChunkArgs &a, int n, int64_t pos) {
    if (a.ckpt == nullptr || pos <= 0 || pos % a.ckpt_interval != 0) return -1;
    const int64_t kth = pos / a.ckpt_interval - 1;
    const int64_t b = a.ckpt_off[n], e = a.ckpt_off[n + 1];
    return kth < e - b ? b + kth : -1;
}

struct DecodeArgs {
    const void *q, *k, *v, *g, *beta;
    float *state;
    const int32_t *idx;       // [N] or nullptr
    void *out;                // or nullptr (no outputs)
    int32_t rows;             // N
    int32_t slots;            // pool size
    int32_t heads;
    int32_t ntok;             // tokens per row in the input layout [N, ntok, H, d]
    const int32_t *ntok_row;  // [N] tokens to run per row (clamped to [0, ntok]) or nullptr
    int32_t update;           // write the state back
    float qk_eps = -1.f;      // >= 0: q and k L2-normalised first, as in ChunkArgs
};

// Token range [bos, eos) of sequence n, read on the device and clamped so that
// a malformed offsets array can never index outside the packed tensors.
__device__ __forceinline__ void seq_range(const ChunkArgs &a, int n, int64_t &bos, int64_t &eos) {
    if (a.cu == nullptr) {
        bos = (int64_t)n * a.seqlen;
        eos = bos + a.seqlen;
    } else {
        int64_t b = __ldg(a.cu + n), e = __ldg(a.cu + n + 1);
        b = b < 0 ? 0 : (b > a.seqlen ? a.seqlen : b);
        e = e < b ? b : (e > a.seqlen ? a.seqlen : e);
        bos = b;
        eos = e;
    }
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Two-pass form of the bf16 d = 128 chunk forward: pass 1 (kda_chunk_prep.cu) writes, per
// (64-token chunk, head), T = (I + A)^-1, M and M - fp16(M) as three 64 x 64 fp16 tiles into
// a caller-owned workspace; pass 2 (kda_chunk_state.cu) runs the state chain from them.  The
// workspace starts with int32 chunk_base[N + 1] (the count of chunks before each sequence),
// padded to 1 KB, followed by the slots; slot (chunk_base[n] + c) * H + h.
constexpr size_t kSlotBytes = 3 * 64 * 64 * 2;
inline size_t ws_header_bytes(int64_t num_seqs) { return ((size_t)(num_seqs + 1) * 4 + 1023) / 1024 * 1024; }
int64_t two_pass_slots(int64_t tokens, int64_t num_seqs, int heads);
size_t two_pass_workspace_bytes(int64_t tokens, int64_t num_seqs, int heads);
cudaError_t launch_chunk_prep(const ChunkArgs &a, void *workspace, cudaStream_t s);
cudaError_t launch_chunk_state(const ChunkArgs &a, const void *workspace, cudaStream_t s);
// Wait for `st`, then read and clear the pass's count of expired bounded waits.
cudaError_t take_prep_expiries(cudaStream_t st, unsigned int *count);
cudaError_t take_state_expiries(cudaStream_t st, unsigned int *count);

// Launchers (host).  Each returns cudaSuccess or the launch error.
cudaError_t launch_chunk_simt(const ChunkArgs &a, int dk, int dv, kda_dtype_t dt, cudaStream_t s);
cudaError_t launch_chunk_tc(const ChunkArgs &a, int dk, int dv, kda_dtype_t dt, cudaStream_t s);
bool chunk_tc_supported(int dk, int dv, kda_dtype_t dt);   // any of the head sizes, bf16
bool chunk_tc_full(int dk, int dv, kda_dtype_t dt);        // dk = dv = 128 (gate, checkpoints, two-pass)
// Waits for `st`, then reads and clears this device's count of expired bounded waits.
cudaError_t take_wait_expiries(cudaStream_t st, unsigned int *count);
// Segments per (sequence, head) the tensor-core launcher picks for a plain call on a GPU with
// `sms` SMs: floor(sms / units), at most 8, lowered until segments average >= 16 chunks.
int segments_for(int64_t units, int64_t tokens, int64_t num_seqs, int sms);
int balanced_ctas(int64_t units, int64_t nc, int sms);
int packed_ctas(int64_t units, int64_t tokens, int64_t num_seqs, int sms);
// Debug-build checks of the device-resident preconditions (g in [-5, 0], packed offsets): launched
// on `st` before a call's kernels when the library is built with KDA_DEBUG_CHECKS, no-ops
// otherwise; failures set bits of a device error word that take_input_errors reads and clears.
cudaError_t debug_check_inputs(const void *g, int64_t g_elems, kda_dtype_t dt, const int32_t *cu,
                               int num_seqs, int64_t seqlen, cudaStream_t st);
int debug_checks_built();
cudaError_t take_input_errors(cudaStream_t st, unsigned int *bits);
cudaError_t launch_decode(const DecodeArgs &a, int dk, int dv, kda_dtype_t dt, cudaStream_t s);
// out <- RMSNorm(out) * w * sigmoid(gate) over dv, in place, for every token row of a chunk call
cudaError_t launch_gate_pass(const ChunkArgs &a, int64_t tokens, int dv, kda_dtype_t dt,
                             cudaStream_t s);
cudaError_t launch_state_copy(const ChunkArgs &a, int dk, int dv, cudaStream_t s);

}  // namespace kda
