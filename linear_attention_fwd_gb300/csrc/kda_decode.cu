// KDA recurrent decode: one or more tokens per (row, head), fp32 state in place.
//
// Per state column j (columns of S are independent, since v_j only touches
// column j), in the order of the four-step delta rule of "はじめての自然言語処理
// -- Kimi K3" section 3.1 (forget, read with the current key, delta, write):
//   vhat_j = sum_i alpha_i k_i S_ij,   p_j = sum_i alpha_i q_i S_ij,
//   e_j = v_j - vhat_j,   S_ij <- alpha_i S_ij + beta k_i e_j,
//   o_j = sum_i q_i S'_ij = p_j + beta (k.q) e_j.
// The state is streamed through registers exactly once (one HBM read and one
// HBM write of d_k*d_v*4 bytes per (row, head)); that traffic is the roofline.
// Several tokens of a row (speculative decoding: a draft verified without
// touching the state, or the accepted prefix replayed into it) keep the state
// in registers between tokens, so their state traffic is paid once.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;

// MULTI = false: one token per row, outputs and state always written (the plain decode
// step, compiled without the per-token loop and its branches).
template <typename Tin, int DK, int DV, bool MULTI>
__global__ void __launch_bounds__(kDecodeThreads)
kda_recurrent_step_kernel(DecodeArgs a) {
    constexpr int CG = DV / 4;                 // float4 column groups
    constexpr int RG = kDecodeThreads / CG;    // row groups
    constexpr int RPT = DK / RG;               // rows per thread
    static_assert(RPT >= 1 && RG * RPT == DK, "tile split");

    constexpr int TM = MULTI ? 8 : 1;          // tokens whose vectors are staged at once

    const int unit = blockIdx.x;
    const int n = unit / a.heads, h = unit - n * a.heads;
    const int slot = a.idx ? __ldg(a.idx + n) : n;
    if (slot < 0 || slot >= a.slots) return;   // uniform across the block

    // 16-byte aligned: red_v, red_p and se are accessed as float4
    __shared__ __align__(16) float sq[TM][DK];
    __shared__ __align__(16) float sk[TM][DK];
    __shared__ __align__(16) float sa[TM][DK];
    __shared__ __align__(16) float sv[TM][DV];
    __shared__ __align__(16) float se[DV];
    __shared__ __align__(16) float red_v[RG][DV];
    __shared__ __align__(16) float red_p[RG][DV];
    __shared__ float s_beta[TM], s_qk[TM];

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int cg = t % CG, rg = t / CG;
    float *S = a.state + ((int64_t)slot * a.heads + h) * (DK * DV);
    int ntok = MULTI ? a.ntok : 1;
    if (MULTI && a.ntok_row) {
        const int m = __ldg(a.ntok_row + n);
        ntok = m < 0 ? 0 : (m < ntok ? m : ntok);
    }
    if (ntok == 0) return;   // uniform across the block

    // Issue the state loads first: they are the only traffic that matters.
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4 *>(S + (rg * RPT + m) * DV) + cg);

#pragma unroll 1
    for (int p0 = 0; p0 < ntok; p0 += TM) {
        const int nt = ntok - p0 < TM ? ntok - p0 : TM;
        if (p0 > 0) __syncthreads();   // the previous group's vectors are consumed
        // this group's token vectors (alpha = e^g), loaded before any of its tokens runs
        for (int x = t; x < nt * DK; x += kDecodeThreads) {
            const int tk = x / DK, i = x - tk * DK;
            const int64_t row = ((int64_t)n * a.ntok + p0 + tk) * a.heads + h;
            sq[tk][i] = to_f(static_cast<const Tin *>(a.q)[row * DK + i]);
            sk[tk][i] = to_f(static_cast<const Tin *>(a.k)[row * DK + i]);
            sa[tk][i] = expf(to_f(static_cast<const Tin *>(a.g)[row * DK + i]));
        }
        for (int x = t; x < nt * DV; x += kDecodeThreads) {
            const int tk = x / DV, j = x - tk * DV;
            const int64_t row = ((int64_t)n * a.ntok + p0 + tk) * a.heads + h;
            sv[tk][j] = to_f(static_cast<const Tin *>(a.v)[row * DV + j]);
        }
        if (t < nt) {
            const int64_t row = ((int64_t)n * a.ntok + p0 + t) * a.heads + h;
            s_beta[t] = to_f(static_cast<const Tin *>(a.beta)[row]);
        }
        __syncthreads();
        if (a.qk_eps >= 0.f) {   // uniform across the block
            // q and k L2-normalised ("はじめての自然言語処理 -- Kimi K3", section 3.1, the
            // read-out paragraph): x / sqrt(|x|^2 + eps) in fp32; a row with |x|^2 + eps = 0
            // stays zero.  Item u (warps in turn) is token u's q, or for u >= TM
            // token (u - TM)'s k.
            for (int u = warp; u < 2 * TM; u += kDecodeThreads / 32) {
                const int tk = u % TM;
                if (tk >= nt) continue;
                float *x = u < TM ? sq[tk] : sk[tk];
                float ss = 0.f;
                for (int i = lane; i < DK; i += 32) ss = fmaf(x[i], x[i], ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float den = ss + a.qk_eps;
                const float sc = den > 0.f ? rsqrtf(den) : 0.f;
                for (int i = lane; i < DK; i += 32) x[i] *= sc;
            }
            __syncthreads();
        }
        if (warp < nt) {   // k . q of token `warp`
            float d = 0.f;
            for (int i = lane; i < DK; i += 32) d += sk[warp][i] * sq[warp][i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) s_qk[warp] = d;
        }

#pragma unroll 1
        for (int tk = 0; tk < nt; ++tk) {
            const int64_t row = ((int64_t)n * a.ntok + p0 + tk) * a.heads + h;
            // column pairs in packed fp32x2 arithmetic (one instruction per two columns)
            float2 pv0 = make_float2(0.f, 0.f), pv1 = pv0, pp0 = pv0, pp1 = pv0;
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                const int i = rg * RPT + m;
                const float ak = sa[tk][i] * sk[tk][i], aq = sa[tk][i] * sq[tk][i];
                const float2 ak2 = make_float2(ak, ak), aq2 = make_float2(aq, aq);
                const float2 s0 = make_float2(s[m].x, s[m].y), s1 = make_float2(s[m].z, s[m].w);
                pv0 = __ffma2_rn(ak2, s0, pv0);
                pv1 = __ffma2_rn(ak2, s1, pv1);
                pp0 = __ffma2_rn(aq2, s0, pp0);
                pp1 = __ffma2_rn(aq2, s1, pp1);
            }
            *reinterpret_cast<float4 *>(&red_v[rg][4 * cg]) = make_float4(pv0.x, pv0.y, pv1.x, pv1.y);
            *reinterpret_cast<float4 *>(&red_p[rg][4 * cg]) = make_float4(pp0.x, pp0.y, pp1.x, pp1.y);
            __syncthreads();

            const float beta = s_beta[tk];
            Tin *out = (!MULTI || a.out) ? static_cast<Tin *>(a.out) + row * DV : nullptr;
            for (int j = t; j < DV; j += kDecodeThreads) {
                float vh = 0.f, p = 0.f;
#pragma unroll
                for (int r = 0; r < RG; ++r) { vh += red_v[r][j]; p += red_p[r][j]; }
                const float e = sv[tk][j] - vh;
                se[j] = e;
                if (!MULTI || out) out[j] = from_f<Tin>(p + beta * s_qk[tk] * e);
            }
            __syncthreads();

            // the next token's partial sums are written only after its barrier, which every
            // thread reaches after finishing this update
            const float4 e4 = *reinterpret_cast<const float4 *>(&se[4 * cg]);
            const float2 e0 = make_float2(e4.x, e4.y), e1 = make_float2(e4.z, e4.w);
            const bool last = !MULTI || p0 + tk + 1 == ntok;
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                const int i = rg * RPT + m;
                const float al = sa[tk][i], bk = beta * sk[tk][i];
                const float2 al2 = make_float2(al, al), bk2 = make_float2(bk, bk);
                const float2 n0 = __ffma2_rn(al2, make_float2(s[m].x, s[m].y), __fmul2_rn(bk2, e0));
                const float2 n1 = __ffma2_rn(al2, make_float2(s[m].z, s[m].w), __fmul2_rn(bk2, e1));
                s[m] = make_float4(n0.x, n0.y, n1.x, n1.y);
                if (last && (!MULTI || a.update)) __stcs(reinterpret_cast<float4 *>(S + i * DV) + cg, s[m]);
            }
        }
    }
}

template <typename Tin, int DK, int DV>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t st) {
    const int64_t units = (int64_t)a.rows * a.heads;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (a.ntok == 1 && a.ntok_row == nullptr && a.update && a.out)
        kda_recurrent_step_kernel<Tin, DK, DV, false><<<(unsigned)units, kDecodeThreads, 0, st>>>(a);
    else
        kda_recurrent_step_kernel<Tin, DK, DV, true><<<(unsigned)units, kDecodeThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_decode_d(const DecodeArgs &a, int dk, int dv, cudaStream_t st) {
    if (dk == 128 && dv == 128) return launch_decode_t<Tin, 128, 128>(a, st);
    if (dk == 128 && dv == 64) return launch_decode_t<Tin, 128, 64>(a, st);
    if (dk == 64 && dv == 128) return launch_decode_t<Tin, 64, 128>(a, st);
    if (dk == 64 && dv == 64) return launch_decode_t<Tin, 64, 64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int dk, int dv, kda_dtype_t dt, cudaStream_t st) {
    return dt == KDA_F32 ? launch_decode_d<float>(a, dk, dv, st)
                         : launch_decode_d<__nv_bfloat16>(a, dk, dv, st);
}

}  // namespace kda
