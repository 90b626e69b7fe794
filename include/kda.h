/*
 * kda.h -- C ABI of libkda: Kimi Delta Attention (KDA) forward on one GPU.
 *
 * KDA is the gated delta rule with a per-channel decay described in
 * "はじめての自然言語処理 -- Kimi K3" (ogis-ri.co.jp), section 3.1 "KDA":
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,
 *
 * with S_t a d_k x d_v state per (sequence, head), q_t, k_t, g_t d_k-vectors,
 * v_t a d_v-vector, beta_t a scalar (the shapes list and the four-step
 * delta-rule paragraph; the one-line form is the report's equation (1)).
 * kda_chunk_fwd evaluates it chunkwise (the chunkwise-form and chunk-decay
 * paragraphs of the same section); kda_recurrent_step is the
 * per-token sequential update used for decode (the serving paragraph of
 * "Kimi K3 architecture", orkas.ai: the state update is sequential).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless stated; tensors are dense, row-major,
 *     contiguous, and must be 16-byte aligned (cu_seqlens / state_indices:
 *     4-byte aligned).  The caller allocates and owns all memory; the library
 *     allocates nothing and keeps no state between calls besides device-wide
 *     counts of expired device waits and of failed debug-build input checks
 *     (kda_device_status reads and clears them) and kda_chunk_fwd_noalloc's
 *     fixed scratch area.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and do not
 *     synchronise the host (kda_device_status excepted).  Argument errors are detected on the host, before
 *     anything is launched; on error nothing is written.  Launch failures map
 *     to KDA_ERR_CUDA.  Faults of a launched kernel surface at the caller's next
 *     synchronisation, as for any CUDA call.
 *   - q, k, v, g, beta and out share `dims->dtype` (fp32 or bf16); recurrent
 *     states are always fp32.  Supported head sizes: dk, dv in {64, 128}.
 *   - No scale is applied to q (o = S^T q exactly); callers fold any 1/sqrt(dk)
 *     into q.  q and k are used as given (their L2 normalisation is the
 *     caller's).  g is the log decay; the kernels rely on the lower bound
 *     g >= -5 of the "lower-bound" paragraph (so that a 16-token tile's
 *     cumulative log decay stays >= -80 and e^80 fits bf16/fp32): g in [-5, 0]
 *     is a precondition; outside it results are unspecified.  The release library
 *     does not check it; a library built with debug checks (kda_debug_checks) checks
 *     it, and the packed offsets, on the device before each call and reports a
 *     failure through kda_device_status (KDA_ERR_INPUT).
 *   - v and the initial state may take any magnitude their formats hold: the
 *     operation is linear in them, and the tensor-core kernel keeps its 16-bit
 *     copies of the state and of the per-chunk corrections at a power-of-two
 *     scale per value channel, chosen each 64-token chunk from that channel's
 *     largest entry, so its accuracy relative to the results does not depend on
 *     their scale (a value channel whose values jump by more than 2^126 from one
 *     chunk to the next may lose the smaller part; parts below 2^-112 of a
 *     channel's largest value may be flushed).  The SIMT and decode kernels
 *     compute in fp32 throughout.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,        /* a required pointer is NULL                       */
    KDA_ERR_SHAPE = 2,       /* inconsistent or non-positive dimensions           */
    KDA_ERR_UNSUPPORTED = 3, /* valid but not implemented (head size, dtype, impl) */
    KDA_ERR_ALIGN = 4,       /* a pointer is not aligned as required              */
    KDA_ERR_WORKSPACE = 5,   /* the workspace is smaller than needed              */
    KDA_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed              */
    KDA_ERR_TIMEOUT = 7,     /* a bounded device wait gave up (kda_device_status) */
    KDA_ERR_INPUT = 8        /* an input failed a debug-build check (kda_device_status) */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Which chunk-forward kernel to run.  AUTO picks the tensor-core kernel where
 * it applies (bf16; a head size of 64 runs there at 128 with the missing channels
 * read as zeros, except with the output gate or checkpoints, which need
 * dk = dv = 128) and the SIMT fp32 kernel otherwise. */
typedef enum { KDA_IMPL_AUTO = 0, KDA_IMPL_SIMT = 1, KDA_IMPL_TC = 2 } kda_impl_t;

/* Problem dimensions.
 *   dense : batch = B, seqlen = T, num_seqs = B, tensors [B, T, H, d].
 *   packed: batch = 1, seqlen = total tokens, num_seqs = N, tensors
 *           [1, total, H, d], cu_seqlens int32[N+1] on the device with
 *           cu[0] = 0 <= cu[1] <= ... <= cu[N] = seqlen (each sequence is
 *           chunked from its own start; empty sequences are allowed).
 *   decode: batch = rows N, seqlen = 1, num_seqs = slots in the state pool. */
typedef struct {
    int32_t batch;
    int32_t seqlen;
    int32_t num_seqs;
    int32_t heads;
    int32_t dk;
    int32_t dv;
    kda_dtype_t dtype;
} kda_dims_t;

/* kda_chunk_fwd -- chunkwise-parallel KDA prefill, and prefix-cache resume.
 *
 * Operation: for every sequence n and head h, starting from
 * initial_state[n,h] (zeros when NULL), run the recurrence above over the
 * sequence's tokens, writing o_t to `out` and the state after the last token
 * to final_state[n,h] (skipped when NULL).  Resume from a cached state at a
 * sequence boundary is the same call with initial_state = the saved state
 * ("Kimi K3 architecture", orkas.ai, the serving section's paragraph on prefix
 * reuse; "Kimi K3 アーキテクチャ", poyo.ai, "KDAとプレフィックスキャッシュ").
 *   q, k, g   : [batch, seqlen, H, dk]  dtype
 *   v, out    : [batch, seqlen, H, dv]  dtype (out is written)
 *   beta      : [batch, seqlen, H]      dtype
 *   initial_state, final_state : fp32 [num_seqs, H, dk, dv]; they may be the
 *               same pointer (in-place resume); partial overlap is not allowed.
 *   cu_seqlens: int32 [num_seqs + 1] device, or NULL for dense batches.
 *               Offsets are clamped to [0, seqlen] on the device.
 * Returns KDA_OK or an error listed above; seqlen = 0 is valid (only the
 * final state is written: a copy of the initial state, or zeros).
 * On the tensor-core kernel (kda_chunk_fwd_segmented with segments = 0 says how,
 * kda_chunk_fwd_auto_ctas how many CTAs) a dense batch runs the balanced schedule:
 * one CTA per SM, each taking an equal share of all (sequence, head, chunk)
 * items, so that a sequence may be split between two CTAs; packed sequences
 * do the same when there are fewer units than twice the SMs.
 * The history a split skips contributes less than 2^-160 of the norm of the
 * state it replaces, else the later part starts at the sequence start (a key
 * channel that barely decays makes every later part do so, up to about one
 * sequence more per CTA; kda_chunk_fwd_segmented with segments = 1 runs one CTA
 * per sequence and head instead). */
kda_status_t kda_chunk_fwd(const void *q, const void *k, const void *v,
                           const void *g, const void *beta,
                           const float *initial_state, const int32_t *cu_seqlens,
                           void *out, float *final_state,
                           const kda_dims_t *dims, cudaStream_t stream);

/* kda_chunk_fwd_qknorm -- kda_chunk_fwd with the L2 normalisation of q and k fused in.
 *
 * The method reads q and k after L2 normalisation, so that q . k is a cosine
 * ("はじめての自然言語処理 -- Kimi K3", section 3.1, the associative-memory read-out
 * paragraph); kda_chunk_fwd leaves that to the caller.  Here every token row of q and of k
 * (per head, over dk) is first replaced by x / sqrt(|x|^2 + qk_eps), computed and kept in
 * fp32 (not rounded back to the io dtype, so the products the kernels form from it are as
 * accurate as from the raw inputs); a row with |x|^2 + qk_eps = 0 stays zero.  The inputs in
 * memory are not modified.  The rest is kda_chunk_fwd, on the kernel kda_chunk_fwd would
 * choose.  The tensor-core kernel computes the row norms (mma.sync) on eight warps while they
 * wait for the previous chunk's tensor-core groups, and scales the rows as it forms its
 * operands.
 *   qk_eps : >= 0 and finite (1e-6 is usual), else KDA_ERR_SHAPE.
 * Other arguments, errors and schedules as kda_chunk_fwd. */
kda_status_t kda_chunk_fwd_qknorm(const void *q, const void *k, const void *v,
                                  const void *g, const void *beta, float qk_eps,
                                  const float *initial_state, const int32_t *cu_seqlens,
                                  void *out, float *final_state,
                                  const kda_dims_t *dims, cudaStream_t stream);

/* As kda_chunk_fwd, with an explicit kernel choice (tests and benchmarks).
 * Returns KDA_ERR_UNSUPPORTED when the chosen kernel cannot run the shape. */
kda_status_t kda_chunk_fwd_with(kda_impl_t impl,
                                const void *q, const void *k, const void *v,
                                const void *g, const void *beta,
                                const float *initial_state, const int32_t *cu_seqlens,
                                void *out, float *final_state,
                                const kda_dims_t *dims, cudaStream_t stream);

/* As kda_chunk_fwd_with, with an explicit bound on every device-side wait of the tensor-core
 * kernel (copy and tensor-core completions): `wait_polls` polls of at most about a microsecond
 * each (kda_chunk_fwd uses 2^20).  When a wait gives up, the CTA stops, lets its copies and
 * tensor-core work in flight land (bounded separately, a few milliseconds), writes NaN to its
 * (sequence, head) final state and leaves the context usable; outputs of that unit are then
 * unspecified.  wait_polls = 0 makes every wait give up at once: a test of that path.  The SIMT
 * kernel has no such waits and ignores the bound. */
kda_status_t kda_chunk_fwd_bounded(kda_impl_t impl,
                                   const void *q, const void *k, const void *v,
                                   const void *g, const void *beta,
                                   const float *initial_state, const int32_t *cu_seqlens,
                                   void *out, float *final_state, uint32_t wait_polls,
                                   const kda_dims_t *dims, cudaStream_t stream);

/* kda_chunk_fwd_segmented -- kda_chunk_fwd_with and an explicit number of CTAs per
 * (sequence, head) for the tensor-core kernel (segment parallelism within a sequence on one
 * GPU).  The pages split a sequence over devices by giving each segment a zero-start state
 * and a cumulative transition, composed by a prefix scan ("請求書はサービング側に回ってくる",
 * orkas.ai, the paragraph on splitting a sequence over devices; "学習基盤", xitter.cf/solis).
 * Here the transition is never formed: segment p of P stores the outputs of chunks
 * [p*nc/P, (p+1)*nc/P) (nc = the sequence's 64-token chunks) and starts from a zero state at
 * the latest chunk boundary, at most 16 chunks earlier, past which the product of the per-token
 * bounds max_i exp(g_t,i) * max(1, |1 - beta_t |k_t|^2|) on the transitions' 2-norm is at most
 * 2^-160 (the state it drops contributes less than 2^-160 of its own norm), or else from the
 * start of the sequence with its initial state.  The last segment writes the final state.
 *   segments : 0 = the library's choice (what kda_chunk_fwd does).  A dense batch runs the
 *              balanced schedule: the W = units x chunks items in sequence-major order are
 *              shared out, contiguously, among G = min(SMs, W, 256) CTAs; the shares are drawn
 *              on the host to make the largest cost small (items, plus 4 for a share that
 *              starts inside a sequence -- its warm-up -- plus 0.5 per further sequence it
 *              touches; a share does not end fewer than 8 chunks into a sequence it entered).
 *              Each part that starts inside a sequence warms up as a segment does, and the
 *              part holding the last chunk writes the final state.  Packed sequences with
 *              fewer units than twice the SMs run the same schedule with shares found on the
 *              device (uniform in items, one item per chunk and at least one per unit; a
 *              boundary within 4 chunks of a unit's start or end moved there); with more
 *              units, one CTA per unit, longest first.  1 per unit with checkpoints (each
 *              then equals the final state of a call on its prefix bit for bit) and with an
 *              in-place state.
 *              1..64 = that many uniform segments.
 * Errors: KDA_ERR_SHAPE for segments outside [0, 64]; KDA_ERR_UNSUPPORTED for segments > 1
 * with initial_state == final_state (a later segment would overwrite the state an earlier one
 * may still read).  The SIMT kernel always runs one CTA per unit.  When a bounded wait gives up
 * in a segment other than the last, that segment's outputs are set to NaN. */
kda_status_t kda_chunk_fwd_segmented(kda_impl_t impl,
                                     const void *q, const void *k, const void *v,
                                     const void *g, const void *beta,
                                     const float *initial_state, const int32_t *cu_seqlens,
                                     void *out, float *final_state, int32_t segments,
                                     const kda_dims_t *dims, cudaStream_t stream);

/* kda_chunk_fwd_ws -- kda_chunk_fwd in two passes over a caller-owned device workspace.
 *
 * For bf16 with dk = dv = 128 the chunk work splits in two: the part that does not depend on
 * the recurrent state (the decay-scaled products A and M of each 64-token chunk and
 * T = (I + A)^-1, "はじめての自然言語処理 -- Kimi K3", section 3.1, the chunkwise form)
 * runs first for every chunk of every sequence at once and is written to `workspace`; the
 * state chain then runs per (sequence, head) from it.  Results equal kda_chunk_fwd's up to
 * rounding.  Other shapes (and seqlen = 0) run kda_chunk_fwd and ignore the workspace.
 *   workspace       : device memory of at least kda_chunk_fwd_workspace_bytes(dims) bytes,
 *                     16-byte aligned, owned by the caller; its contents on entry do not
 *                     matter and are overwritten.  Calls that overlap in time on the device
 *                     need workspaces of their own.
 *   workspace_bytes : its size.
 * Errors: as kda_chunk_fwd, plus KDA_ERR_NULL for a NULL workspace, KDA_ERR_WORKSPACE when it
 * is smaller than needed, KDA_ERR_ALIGN when it is not 16-byte aligned. */
kda_status_t kda_chunk_fwd_ws(const void *q, const void *k, const void *v,
                              const void *g, const void *beta,
                              const float *initial_state, const int32_t *cu_seqlens,
                              void *out, float *final_state,
                              void *workspace, size_t workspace_bytes,
                              const kda_dims_t *dims, cudaStream_t stream);

/* Bytes of workspace kda_chunk_fwd_ws needs for `dims`: 24 KB per (64-token chunk, head)
 * counted as heads * (ceil(batch * seqlen / 64) + num_seqs), plus (num_seqs + 1) * 4 bytes
 * rounded up to 1 KB; 0 when it runs the one-pass path (host arithmetic only). */
size_t kda_chunk_fwd_workspace_bytes(const kda_dims_t *dims);

/* kda_chunk_fwd_noalloc -- kda_chunk_fwd_ws over a fixed scratch area compiled into this
 * library, for callers that cannot supply device memory when they call (a host whose device
 * budget is fixed at start-up, a C host with no device allocator, a loop that cannot afford the
 * device-wide synchronisation of cudaMalloc / cudaFree).  The pages have no counterpart: this
 * is an interface for such callers, not part of the method.  The call allocates nothing.
 *   Scratch: one area of KDA_NOALLOC_SCRATCH_BYTES bytes per device.  Calls with
 *            kda_chunk_fwd_workspace_bytes(dims) above that are rejected with
 *            KDA_ERR_WORKSPACE before anything runs.  Nothing in the area has to start at
 *            zero, and nothing is carried from one call to the next.
 *   Set-up:  the first call with a device current looks up the area's address on that device
 *            (and loads the library's device code there if that has not happened); make that
 *            first call before any stream capture.  Later calls only read the kept address.
 *   Overlap: calls that overlap in time on the same device (several streams or host threads)
 *            share the area and race; the caller serialises them.
 * Arguments, layouts, results and the other errors are kda_chunk_fwd_ws's (shapes the
 * two-pass kernels do not take, and seqlen = 0, run kda_chunk_fwd); KDA_ERR_CUDA also when the
 * address lookup fails. */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
kda_status_t kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                   const void *g, const void *beta,
                                   const float *initial_state, const int32_t *cu_seqlens,
                                   void *out, float *final_state,
                                   const kda_dims_t *dims, cudaStream_t stream);

/* kda_chunk_fwd_checkpointed -- kda_chunk_fwd that also writes the recurrent state at every
 * multiple of `checkpoint_interval` tokens strictly inside each sequence, for prefix caching.
 * The pages' account: the cache hashes prompts in 512-token units and keeps recurrent-state
 * checkpoints only at a sparse subset of those endpoints, so that a prefix hit can resume from
 * a stored state ("はじめての自然言語処理 -- Kimi K3", the infrastructure paragraph on
 * prefix reuse; resuming is kda_chunk_fwd with initial_state).
 *   checkpoints       : fp32 [slots, H, dk, dv]; the state after the first (k+1)*interval
 *                       tokens of sequence n goes to slot checkpoint_offsets[n] + k, for
 *                       k < checkpoint_offsets[n+1] - checkpoint_offsets[n] and
 *                       (k+1)*interval < len_n (the state at the end is final_state).
 *                       Slots the kernel does not reach are left untouched.
 *   checkpoint_offsets: int32 [num_seqs + 1] device, nondecreasing, offsets[num_seqs] <= slots.
 *   checkpoint_interval: a positive multiple of 64 (the chunk), else KDA_ERR_SHAPE.
 * Each checkpoint equals, up to rounding, the final state of the same call on the prefix
 * (bit for bit for the same kernel, whose chunks do not depend on later tokens).
 * Everything else as kda_chunk_fwd; NULL checkpoints or offsets give KDA_ERR_NULL. */
kda_status_t kda_chunk_fwd_checkpointed(const void *q, const void *k, const void *v,
                                        const void *g, const void *beta,
                                        const float *initial_state, const int32_t *cu_seqlens,
                                        void *out, float *final_state, float *checkpoints,
                                        const int32_t *checkpoint_offsets,
                                        int32_t checkpoint_interval,
                                        const kda_dims_t *dims, cudaStream_t stream);

/* kda_chunk_fwd_gated -- kda_chunk_fwd followed by the KDA output gate, fused into the output
 * store.  The page's account ("はじめての自然言語処理 -- Kimi K3", the paragraph after the decay
 * bound): the read-out o_t is put through RMSNorm over its value channels (evening out the
 * magnitude of what is read from S) and then multiplied channel by channel by a gate in (0, 1)
 * made from the token's input.  Here, per token and head,
 *   out = o / sqrt(mean_j o_j^2 + norm_eps) * w * sigmoid(z),
 * with z the gate logits (the projection that makes them from the token's input is the
 * caller's) and w the RMSNorm weight.
 *   gate       : [B, T, H, dv] dtype (z), required when there are tokens.
 *   norm_weight: fp32 [dv] or NULL (ones).   norm_eps: >= 0 and finite, else KDA_ERR_SHAPE.
 * The bf16 d = 128 kernel applies the gate while staging its output (no extra traffic beyond
 * reading z); other shapes apply it in a second pass over the stored output.  Everything else
 * as kda_chunk_fwd. */
kda_status_t kda_chunk_fwd_gated(const void *q, const void *k, const void *v,
                                 const void *g, const void *beta, const void *gate,
                                 const float *norm_weight, float norm_eps,
                                 const float *initial_state, const int32_t *cu_seqlens,
                                 void *out, float *final_state,
                                 const kda_dims_t *dims, cudaStream_t stream);

/* The kernel kda_chunk_fwd would run for `dims` (KDA_IMPL_SIMT or
 * KDA_IMPL_TC), or -1 when the dims are invalid.  A library query (host only). */
int kda_chunk_fwd_selected_impl(const kda_dims_t *dims);

/* The number of CTAs kda_chunk_fwd launches for the tensor-core kernel for `dims` on a GPU
 * with `sms` SMs (host arithmetic only, no device call).  packed = 0 (dense batch): the
 * balanced schedule's min(sms, units * ceil(seqlen / 64)), units = num_seqs * heads.
 * packed != 0 (cu_seqlens given): with units < 2 * sms, the balanced schedule's
 * min(sms, 256, heads * (ceil(seqlen / 64) + num_seqs)) (a bound on its items; CTAs past the
 * last item exit at once), else one per unit.  0 for shapes the tensor-core kernel does not run,
 * seqlen = 0 and invalid dims or SM counts.  A call with checkpoints or initial_state ==
 * final_state runs one CTA per unit instead. */
int kda_chunk_fwd_auto_ctas(const kda_dims_t *dims, int packed, int sms);

/* kda_recurrent_step -- one decode token per row, state updated in place.
 *
 * Operation per row n and head h, on the state S = state[slot][h] with
 * slot = state_indices ? state_indices[n] : n, in the order of the four-step
 * delta-rule paragraph (forget, read with the current key, delta, write):
 *   vhat = (Diag(exp g) S)^T k,  e = v - vhat,
 *   S <- Diag(exp g) S + beta k e^T,  o = S^T q.
 *   q, k, g : [N, H, dk] dtype;  v, out : [N, H, dv] dtype;  beta : [N, H]
 *   state   : fp32 [num_seqs, H, dk, dv], read and written in place.
 *   state_indices: int32 [N] device or NULL (identity; then num_seqs >= N).
 *               Rows whose slot is outside [0, num_seqs) are skipped: neither
 *               their state nor their output is written.  Two rows must not
 *               name the same slot.
 * dims: batch = N rows, seqlen = 1, num_seqs = pool slots.
 * Returns KDA_OK, or an error found on the host before any launch (null required
 * pointers, non-positive or inconsistent dims, unsupported head size or dtype,
 * misalignment), in which case nothing is written. */
kda_status_t kda_recurrent_step(const void *q, const void *k, const void *v,
                                const void *g, const void *beta, float *state,
                                const int32_t *state_indices, void *out,
                                const kda_dims_t *dims, cudaStream_t stream);

/* kda_recurrent_step_qknorm -- kda_recurrent_step with q and k L2-normalised first, as in
 * kda_chunk_fwd_qknorm (x / sqrt(|x|^2 + qk_eps) per row, in fp32; a zero row stays
 * zero).  qk_eps >= 0 and finite, else KDA_ERR_SHAPE; the rest as
 * kda_recurrent_step. */
kda_status_t kda_recurrent_step_qknorm(const void *q, const void *k, const void *v,
                                       const void *g, const void *beta, float qk_eps,
                                       float *state, const int32_t *state_indices, void *out,
                                       const kda_dims_t *dims, cudaStream_t stream);

/* kda_recurrent_steps -- up to T decode tokens per row from the row's state, for speculative
 * decoding.  The pages' account of it: the state is updated in place, so a rejected draft
 * cannot be rolled back; the draft tokens' projected inputs (far smaller than the state) are
 * kept instead and the accepted ones are rebuilt on chip ("はじめての自然言語処理 -- Kimi K3",
 * the infrastructure paragraph on speculative decoding).  So a draft is verified with
 * update_state = 0 (outputs only, the state untouched) and the accepted prefix is then replayed
 * into the state with update_state = 1.
 *
 * Row n runs tokens 0 .. m_n - 1, m_n = num_tokens ? clamp(num_tokens[n], 0, T) : T, each as in
 * kda_recurrent_step, starting from S = state[slot][h] (slot as in kda_recurrent_step); the
 * state stays on chip between tokens (one read and at most one write per row and head).
 *   q, k, g : [N, T, H, dk] dtype;  v, out : [N, T, H, dv] dtype;  beta : [N, T, H]
 *   state   : fp32 [num_seqs, H, dk, dv]; written (the state after the row's m_n tokens) only
 *             when update_state != 0 and m_n > 0.
 *   state_indices: as in kda_recurrent_step (rows with a slot outside the pool are skipped).
 *   num_tokens: int32 [N] device or NULL (every row runs all T tokens).
 *   out     : may be NULL (no outputs); outputs of tokens m_n .. T-1 are not written.
 * dims: batch = N rows, seqlen = T, num_seqs = pool slots.  Two rows must not name the same
 * slot when update_state != 0.  Errors as in kda_recurrent_step; out == NULL with
 * update_state == 0 returns KDA_OK without launching. */
kda_status_t kda_recurrent_steps(const void *q, const void *k, const void *v,
                                 const void *g, const void *beta, float *state,
                                 const int32_t *state_indices, const int32_t *num_tokens,
                                 void *out, int update_state,
                                 const kda_dims_t *dims, cudaStream_t stream);

/* kda_recurrent_steps_qknorm -- kda_recurrent_steps with q and k L2-normalised first, as in
 * kda_chunk_fwd_qknorm (x / sqrt(|x|^2 + qk_eps) per token row, in fp32; a zero row stays
 * zero).  qk_eps >= 0 and finite, else KDA_ERR_SHAPE; the rest as kda_recurrent_steps. */
kda_status_t kda_recurrent_steps_qknorm(const void *q, const void *k, const void *v,
                                        const void *g, const void *beta, float qk_eps,
                                        float *state, const int32_t *state_indices,
                                        const int32_t *num_tokens, void *out, int update_state,
                                        const kda_dims_t *dims, cudaStream_t stream);

/* kda_device_status -- waits for the work queued on `stream` to finish, then reads and
 * clears the current device's count of device-side waits of the tensor-core chunk kernels
 * that gave up (see kda_chunk_fwd_bounded; the two passes of kda_chunk_fwd_ws count theirs
 * too) and its word of failed debug-build input checks.  Returns KDA_ERR_INPUT when a check
 * failed since the previous call on this device (only a library built with debug checks
 * makes any), else KDA_ERR_TIMEOUT when at least one wait gave up, KDA_OK when neither
 * happened, and KDA_ERR_CUDA when the stream or the copies fail.  Both are device-global:
 * calls that run concurrently on other streams of the device report into the same word and
 * count.  This is the only call of the library that synchronises the host; it does not
 * depend on final_state being requested. */
kda_status_t kda_device_status(cudaStream_t stream);

/* kda_debug_checks -- which device-side input checks this build of the library runs before
 * each chunk forward and decode call: a bit mask, 1 = g in [-5, 0] (NaN fails), 2 = packed
 * offsets 0 = cu[0] <= ... <= cu[N] = seqlen; 0 for the release build, which runs none (the
 * precondition is "はじめての自然言語処理 -- Kimi K3", section 3.1: g = -5 sigmoid(x)).  A failed
 * check launches nothing extra and traps nothing: the call still runs, its results are
 * unspecified, and kda_device_status returns KDA_ERR_INPUT.  A host query. */
int kda_debug_checks(void);

/* A static, human-readable name for a status code (never NULL). */
const char *kda_status_string(kda_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
