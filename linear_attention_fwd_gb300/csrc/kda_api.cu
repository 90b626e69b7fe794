// libkda C ABI: argument validation and kernel dispatch.  No allocation; no host
// synchronisation except in kda_device_status; no global mutable state besides per-function
// attribute caches inside the launchers and the device's count of expired bounded waits.
#include <cstdint>
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool head_size_ok(int d) { return d == 64 || d == 128; }

kda_status_t check_chunk(kda_impl_t impl, const void *q, const void *k, const void *v,
                         const void *g, const void *beta, const float *s0, const int32_t *cu,
                         const void *out, const float *sT, const kda_dims_t *d) {
    if (d == nullptr) return KDA_ERR_NULL;
    if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_size_ok(d->dk) || !head_size_ok(d->dv)) return KDA_ERR_UNSUPPORTED;
    if (d->heads <= 0 || d->batch <= 0 || d->seqlen < 0 || d->num_seqs <= 0) return KDA_ERR_SHAPE;
    if (cu == nullptr) {
        if (d->num_seqs != d->batch) return KDA_ERR_SHAPE;
    } else if (d->batch != 1) {
        return KDA_ERR_SHAPE;
    }
    const int64_t tokens = (int64_t)d->batch * d->seqlen;
    if (tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    const uintptr_t es = d->dtype == KDA_F32 ? 4 : 2;
    const void *ptrs[] = {q, k, v, g, out, s0, sT};
    for (const void *p : ptrs)
        if (p && !aligned(p, 16)) return KDA_ERR_ALIGN;
    if (beta && !aligned(beta, es)) return KDA_ERR_ALIGN;
    if (cu && !aligned(cu, 4)) return KDA_ERR_ALIGN;
    if (s0 && sT && s0 != sT) {
        const char *a = reinterpret_cast<const char *>(s0), *b = reinterpret_cast<const char *>(sT);
        const int64_t bytes = (int64_t)d->num_seqs * d->heads * d->dk * d->dv * 4;
        if (a < b + bytes && b < a + bytes) return KDA_ERR_SHAPE;  // partial overlap
    }
    if (impl == KDA_IMPL_TC && !kda::chunk_tc_supported(d->dk, d->dv, d->dtype))
        return KDA_ERR_UNSUPPORTED;
    if (impl != KDA_IMPL_AUTO && impl != KDA_IMPL_SIMT && impl != KDA_IMPL_TC)
        return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

}  // namespace

extern "C" const char *kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_SHAPE: return "inconsistent or non-positive dimensions";
        case KDA_ERR_UNSUPPORTED: return "unsupported head size, dtype or kernel choice";
        case KDA_ERR_ALIGN: return "pointer not aligned as required";
        case KDA_ERR_WORKSPACE: return "workspace too small";
        case KDA_ERR_CUDA: return "CUDA launch or runtime error";
        case KDA_ERR_TIMEOUT: return "a bounded device wait gave up";
        case KDA_ERR_INPUT: return "an input failed a debug-build precondition check";
    }
    return "unknown status";
}

extern "C" kda_status_t kda_device_status(cudaStream_t stream) {
    unsigned int n1 = 0, n2 = 0, n3 = 0, bad = 0;
    if (kda::take_wait_expiries(stream, &n1) != cudaSuccess || kda::take_prep_expiries(stream, &n2) != cudaSuccess ||
        kda::take_state_expiries(stream, &n3) != cudaSuccess || kda::take_input_errors(stream, &bad) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (bad) return KDA_ERR_INPUT;
    return (n1 || n2 || n3) ? KDA_ERR_TIMEOUT : KDA_OK;
}

extern "C" int kda_debug_checks(void) { return kda::debug_checks_built(); }

extern "C" size_t kda_chunk_fwd_workspace_bytes(const kda_dims_t *d) {
    if (d == nullptr || d->heads <= 0 || d->num_seqs <= 0 || d->batch <= 0 || d->seqlen < 0) return 0;
    if (!kda::chunk_tc_full(d->dk, d->dv, d->dtype)) return 0;
    const int64_t tokens = (int64_t)d->batch * d->seqlen;
    if (tokens == 0) return 0;
    return kda::two_pass_workspace_bytes(tokens, d->num_seqs, d->heads);
}

extern "C" kda_status_t kda_chunk_fwd_ws(const void *q, const void *k, const void *v, const void *g,
                                         const void *beta, const float *initial_state,
                                         const int32_t *cu_seqlens, void *out, float *final_state,
                                         void *workspace, size_t workspace_bytes, const kda_dims_t *d,
                                         cudaStream_t stream) {
    kda_status_t st = check_chunk(KDA_IMPL_AUTO, q, k, v, g, beta, initial_state, cu_seqlens, out,
                                  final_state, d);
    if (st != KDA_OK) return st;
    const size_t need = kda_chunk_fwd_workspace_bytes(d);
    if (need == 0)   // no tokens, or a shape the two-pass kernels do not take: the one-pass path
        return kda_chunk_fwd(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, d, stream);
    if (workspace == nullptr) return KDA_ERR_NULL;
    if (workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return KDA_ERR_ALIGN;
    kda::ChunkArgs a{q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                     (int64_t)d->seqlen, d->num_seqs, d->heads, nullptr, nullptr, 0.f,
                     nullptr, nullptr, 0, 1u << 20, 1};
    cudaError_t e = kda::debug_check_inputs(g, (int64_t)d->batch * d->seqlen * d->heads * d->dk, d->dtype,
                                            cu_seqlens, d->num_seqs, d->seqlen, stream);
    if (e == cudaSuccess) e = kda::launch_chunk_prep(a, workspace, stream);
    if (e == cudaSuccess) e = kda::launch_chunk_state(a, workspace, stream);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" int kda_chunk_fwd_selected_impl(const kda_dims_t *d) {
    if (d == nullptr || !head_size_ok(d->dk) || !head_size_ok(d->dv)) return -1;
    if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return -1;
    return kda::chunk_tc_supported(d->dk, d->dv, d->dtype) ? KDA_IMPL_TC : KDA_IMPL_SIMT;
}

extern "C" int kda_chunk_fwd_auto_ctas(const kda_dims_t *d, int packed, int sms) {
    if (d == nullptr || d->heads <= 0 || d->num_seqs <= 0 || d->batch <= 0 || d->seqlen <= 0 || sms <= 0)
        return 0;
    if (!kda::chunk_tc_supported(d->dk, d->dv, d->dtype)) return 0;
    const int64_t tokens = (int64_t)d->batch * d->seqlen, units = (int64_t)d->num_seqs * d->heads;
    if (!packed) return kda::balanced_ctas(units, (d->seqlen + 63) / 64, sms);
    return units < 2 * (int64_t)sms ? kda::packed_ctas(units, tokens, d->num_seqs, sms)
                                    : (int)(units > 0x7fffffffLL ? 0x7fffffff : units);
}

// Validated launch of one chunked forward (optionally writing state checkpoints).
static kda_status_t chunk_run(kda_impl_t impl, const void *q, const void *k, const void *v, const void *g,
                       const void *beta, const float *initial_state, const int32_t *cu_seqlens,
                       void *out, float *final_state, float *ckpt, const int32_t *ckpt_off,
                       int32_t ckpt_interval, const void *gate, const float *norm_w, float norm_eps,
                       const kda_dims_t *d, cudaStream_t stream, uint32_t wait_polls = 1u << 20,
                       int32_t segments = 0, float qk_eps = -1.f) {
    kda_status_t st = check_chunk(impl, q, k, v, g, beta, initial_state, cu_seqlens, out,
                                  final_state, d);
    if (st != KDA_OK) return st;
    kda::ChunkArgs a{q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                     (int64_t)d->seqlen, d->num_seqs, d->heads, gate, norm_w, norm_eps,
                     ckpt, ckpt_off, ckpt_interval, wait_polls, segments};
    a.qk_eps = qk_eps;
    cudaError_t e = kda::debug_check_inputs(g, (int64_t)d->batch * d->seqlen * d->heads * d->dk, d->dtype,
                                            cu_seqlens, d->num_seqs, d->seqlen, stream);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if ((int64_t)d->batch * d->seqlen == 0) {
        if (final_state == nullptr || final_state == initial_state) return KDA_OK;
        e = kda::launch_state_copy(a, d->dk, d->dv, stream);
    } else {
        // the output gate and checkpoints run on the tensor-core kernel at dk = dv = 128 only
        const bool tc_ok = kda::chunk_tc_supported(d->dk, d->dv, d->dtype) &&
                           (kda::chunk_tc_full(d->dk, d->dv, d->dtype) || (!gate && !ckpt));
        if (impl == KDA_IMPL_AUTO) impl = tc_ok ? KDA_IMPL_TC : KDA_IMPL_SIMT;
        else if (impl == KDA_IMPL_TC && !tc_ok) return KDA_ERR_UNSUPPORTED;
        if (impl == KDA_IMPL_TC) {
            e = kda::launch_chunk_tc(a, d->dk, d->dv, d->dtype, stream);   // gate fused
        } else {
            e = kda::launch_chunk_simt(a, d->dk, d->dv, d->dtype, stream);
            if (e == cudaSuccess && gate)
                e = kda::launch_gate_pass(a, (int64_t)d->batch * d->seqlen, d->dv, d->dtype, stream);
        }
    }
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_chunk_fwd_with(kda_impl_t impl, const void *q, const void *k,
                                           const void *v, const void *g, const void *beta,
                                           const float *initial_state, const int32_t *cu_seqlens,
                                           void *out, float *final_state, const kda_dims_t *d,
                                           cudaStream_t stream) {
    return chunk_run(impl, q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, nullptr,
                     nullptr, 0, nullptr, nullptr, 0.f, d, stream);
}

extern "C" kda_status_t kda_chunk_fwd_checkpointed(const void *q, const void *k, const void *v,
                                                   const void *g, const void *beta,
                                                   const float *initial_state,
                                                   const int32_t *cu_seqlens, void *out,
                                                   float *final_state, float *checkpoints,
                                                   const int32_t *checkpoint_offsets,
                                                   int32_t checkpoint_interval,
                                                   const kda_dims_t *d, cudaStream_t stream) {
    if (checkpoints == nullptr || checkpoint_offsets == nullptr) return KDA_ERR_NULL;
    if (checkpoint_interval <= 0 || checkpoint_interval % kda::kChunk != 0) return KDA_ERR_SHAPE;
    if (!aligned(checkpoints, 16) || !aligned(checkpoint_offsets, 4)) return KDA_ERR_ALIGN;
    return chunk_run(KDA_IMPL_AUTO, q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                     checkpoints, checkpoint_offsets, checkpoint_interval, nullptr, nullptr, 0.f, d,
                     stream);
}

extern "C" kda_status_t kda_chunk_fwd_gated(const void *q, const void *k, const void *v,
                                            const void *g, const void *beta, const void *gate,
                                            const float *norm_weight, float norm_eps,
                                            const float *initial_state, const int32_t *cu_seqlens,
                                            void *out, float *final_state, const kda_dims_t *d,
                                            cudaStream_t stream) {
    if (d != nullptr && (int64_t)d->batch * d->seqlen > 0 && gate == nullptr) return KDA_ERR_NULL;
    if (!(norm_eps >= 0.f) || norm_eps > 1e30f) return KDA_ERR_SHAPE;   // also rejects NaN
    if ((gate && !aligned(gate, 16)) || (norm_weight && !aligned(norm_weight, 4))) return KDA_ERR_ALIGN;
    return chunk_run(KDA_IMPL_AUTO, q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                     nullptr, nullptr, 0, gate, norm_weight, norm_eps, d, stream);
}

extern "C" kda_status_t kda_chunk_fwd_bounded(kda_impl_t impl, const void *q, const void *k,
                                              const void *v, const void *g, const void *beta,
                                              const float *initial_state, const int32_t *cu_seqlens,
                                              void *out, float *final_state, uint32_t wait_polls,
                                              const kda_dims_t *d, cudaStream_t stream) {
    return chunk_run(impl, q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, nullptr,
                     nullptr, 0, nullptr, nullptr, 0.f, d, stream, wait_polls);
}

extern "C" kda_status_t kda_chunk_fwd_segmented(kda_impl_t impl, const void *q, const void *k,
                                                const void *v, const void *g, const void *beta,
                                                const float *initial_state,
                                                const int32_t *cu_seqlens, void *out,
                                                float *final_state, int32_t segments,
                                                const kda_dims_t *d, cudaStream_t stream) {
    if (segments < 0 || segments > 64) return KDA_ERR_SHAPE;
    if (segments > 1 && initial_state && initial_state == final_state) return KDA_ERR_UNSUPPORTED;
    return chunk_run(impl, q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, nullptr,
                     nullptr, 0, nullptr, nullptr, 0.f, d, stream, 1u << 20, segments);
}

extern "C" kda_status_t kda_chunk_fwd(const void *q, const void *k, const void *v, const void *g,
                                      const void *beta, const float *initial_state,
                                      const int32_t *cu_seqlens, void *out, float *final_state,
                                      const kda_dims_t *dims, cudaStream_t stream) {
    return kda_chunk_fwd_with(KDA_IMPL_AUTO, q, k, v, g, beta, initial_state, cu_seqlens, out,
                              final_state, dims, stream);
}

extern "C" kda_status_t kda_chunk_fwd_qknorm(const void *q, const void *k, const void *v, const void *g,
                                             const void *beta, float qk_eps, const float *initial_state,
                                             const int32_t *cu_seqlens, void *out, float *final_state,
                                             const kda_dims_t *dims, cudaStream_t stream) {
    if (!(qk_eps >= 0.f) || qk_eps > 1e30f) return KDA_ERR_SHAPE;   // also rejects NaN
    return chunk_run(KDA_IMPL_AUTO, q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                     nullptr, nullptr, 0, nullptr, nullptr, 0.f, dims, stream, 1u << 20, 0, qk_eps);
}

// Validated launch of one or more decode tokens per row.
static kda_status_t decode_run(const void *q, const void *k, const void *v, const void *g,
                               const void *beta, float *state, const int32_t *state_indices,
                               void *out, const kda_dims_t *d, float qk_eps, cudaStream_t stream) {
    if (d == nullptr) return KDA_ERR_NULL;
    if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_size_ok(d->dk) || !head_size_ok(d->dv)) return KDA_ERR_UNSUPPORTED;
    if (d->seqlen != 1 || d->batch < 0 || d->heads <= 0 || d->num_seqs <= 0) return KDA_ERR_SHAPE;
    if (state_indices == nullptr && d->num_seqs < d->batch) return KDA_ERR_SHAPE;
    if (d->batch == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return KDA_ERR_NULL;
    const uintptr_t es = d->dtype == KDA_F32 ? 4 : 2;
    const void *ptrs[] = {q, k, v, g, out, state};
    for (const void *p : ptrs)
        if (!aligned(p, 16)) return KDA_ERR_ALIGN;
    if (!aligned(beta, es)) return KDA_ERR_ALIGN;
    if (state_indices && !aligned(state_indices, 4)) return KDA_ERR_ALIGN;
    kda::DecodeArgs a{q, k, v, g, beta, state, state_indices, out, d->batch, d->num_seqs, d->heads,
                      1, nullptr, 1};
    a.qk_eps = qk_eps;
    cudaError_t e = kda::debug_check_inputs(g, (int64_t)d->batch * d->heads * d->dk, d->dtype, nullptr, 0, 0, stream);
    if (e == cudaSuccess) e = kda::launch_decode(a, d->dk, d->dv, d->dtype, stream);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_recurrent_step(const void *q, const void *k, const void *v,
                                           const void *g, const void *beta, float *state,
                                           const int32_t *state_indices, void *out,
                                           const kda_dims_t *d, cudaStream_t stream) {
    return decode_run(q, k, v, g, beta, state, state_indices, out, d, -1.f, stream);
}

extern "C" kda_status_t kda_recurrent_step_qknorm(const void *q, const void *k, const void *v,
                                                  const void *g, const void *beta, float qk_eps,
                                                  float *state, const int32_t *state_indices,
                                                  void *out, const kda_dims_t *d, cudaStream_t stream) {
    if (!(qk_eps >= 0.f) || qk_eps > 1e30f) return KDA_ERR_SHAPE;   // also rejects NaN
    return decode_run(q, k, v, g, beta, state, state_indices, out, d, qk_eps, stream);
}

// Validated launch of several decode tokens per row.
static kda_status_t steps_run(const void *q, const void *k, const void *v, const void *g,
                              const void *beta, float *state, const int32_t *state_indices,
                              const int32_t *num_tokens, void *out, int update_state,
                              const kda_dims_t *d, float qk_eps, cudaStream_t stream) {
    if (d == nullptr) return KDA_ERR_NULL;
    if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_size_ok(d->dk) || !head_size_ok(d->dv)) return KDA_ERR_UNSUPPORTED;
    if (d->seqlen < 1 || d->batch < 0 || d->heads <= 0 || d->num_seqs <= 0) return KDA_ERR_SHAPE;
    if (state_indices == nullptr && d->num_seqs < d->batch) return KDA_ERR_SHAPE;
    if ((int64_t)d->batch * d->seqlen * d->heads > 0x7fffffffLL) return KDA_ERR_SHAPE;
    if (d->batch == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !state) return KDA_ERR_NULL;
    if (out == nullptr && !update_state) return KDA_OK;   // nothing to write
    const uintptr_t es = d->dtype == KDA_F32 ? 4 : 2;
    const void *ptrs[] = {q, k, v, g, state};
    for (const void *p : ptrs)
        if (!aligned(p, 16)) return KDA_ERR_ALIGN;
    if (out && !aligned(out, 16)) return KDA_ERR_ALIGN;
    if (!aligned(beta, es)) return KDA_ERR_ALIGN;
    if (state_indices && !aligned(state_indices, 4)) return KDA_ERR_ALIGN;
    if (num_tokens && !aligned(num_tokens, 4)) return KDA_ERR_ALIGN;
    kda::DecodeArgs a{q, k, v, g, beta, state, state_indices, out, d->batch, d->num_seqs, d->heads,
                      d->seqlen, num_tokens, update_state ? 1 : 0};
    a.qk_eps = qk_eps;
    cudaError_t e = kda::debug_check_inputs(g, (int64_t)d->batch * d->seqlen * d->heads * d->dk, d->dtype,
                                            nullptr, 0, 0, stream);
    if (e == cudaSuccess) e = kda::launch_decode(a, d->dk, d->dv, d->dtype, stream);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_recurrent_steps(const void *q, const void *k, const void *v,
                                            const void *g, const void *beta, float *state,
                                            const int32_t *state_indices, const int32_t *num_tokens,
                                            void *out, int update_state, const kda_dims_t *d,
                                            cudaStream_t stream) {
    return steps_run(q, k, v, g, beta, state, state_indices, num_tokens, out, update_state, d, -1.f,
                     stream);
}

extern "C" kda_status_t kda_recurrent_steps_qknorm(const void *q, const void *k, const void *v,
                                                   const void *g, const void *beta, float qk_eps,
                                                   float *state, const int32_t *state_indices,
                                                   const int32_t *num_tokens, void *out,
                                                   int update_state, const kda_dims_t *d,
                                                   cudaStream_t stream) {
    if (!(qk_eps >= 0.f) || qk_eps > 1e30f) return KDA_ERR_SHAPE;   // also rejects NaN
    return steps_run(q, k, v, g, beta, state, state_indices, num_tokens, out, update_state, d, qk_eps,
                     stream);
}
