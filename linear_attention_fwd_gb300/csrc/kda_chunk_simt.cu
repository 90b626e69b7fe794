// KDA chunkwise forward, SIMT fp32 kernel.
//
// The fp32-mode path (fp32 inputs need fp32 arithmetic throughout, which the
// bf16 tensor-core path cannot give) and the general fallback for head sizes
// the tensor-core kernel does not take.  It evaluates the same chunk algebra
// as the tensor-core kernel.
//
// Chunk form ("はじめての自然言語処理 -- Kimi K3" section 3.1, chunkwise paragraphs
// and "chunk 内の減衰と、その数値範囲"): per chunk of C = 64 tokens, with
// gamma_r = sum_{s<=r} g_s and S the state entering the chunk,
//   A_rs = beta_r sum_c k_rc k_sc e^{gamma_rc - gamma_sc}   (s <  r)
//   M_rs =        sum_c q_rc k_sc e^{gamma_rc - gamma_sc}   (s <= r, the Tril mask)
//   (I + A) U = diag(beta) (V - Kbar S)          (delta-rule correction, WY form)
//   O = Qbar S + M U                              (inter-chunk + intra-chunk terms)
//   S <- Diag(e^{gamma_last}) S + Kp^T U
// where Qbar = Q e^{gamma}, Kbar = K e^{gamma}, Kp = K e^{gamma_last - gamma}.
// The decay between positions is folded into the operands (q times Gamma, k
// divided by Gamma: the report's equation (4)), split at 16-token sub-tiles:
// relative to b_I = gamma just before sub-tile I starts, x = e^{gamma - b_I} is
// in [e^-80, 1] and 1/x in [1, e^80] because g >= -5 (the lower-bound
// paragraph), so the diagonal sub-tiles are ordinary dot products with no
// per-position-pair exponentials.
//
// One CTA of 512 threads per (sequence, head, 64-column slice of d_v).
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 512;
constexpr int kRows = kThreads / 64;   // row phases: a thread takes rows rq, rq + kRows, ...
constexpr int kRpt = kChunk / kRows;   // rows per thread in the 64-row loops
constexpr int kDvs = 64;               // d_v columns per CTA
constexpr int kNb = kChunk / kSub;     // sub-tiles per chunk (4)
constexpr int kLdu = kDvs + 8;         // row stride of the V/Y/U tile (conflict-free solve)

template <int DK>
struct SimtSmem {
    static constexpr int LDQ = DK;       // Q~ / Qbar tile
    static constexpr int LDK = DK;       // K~ / Kbar tile
    static constexpr int LDH = DK + 1;   // gamma, then K^ / Kp tile (odd: column reads)
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kChunk * LDQ;
    static constexpr int kH = kK + kChunk * LDK;
    static constexpr int kU = kH + kChunk * LDH;
    static constexpr int kS = kU + kChunk * kLdu;
    static constexpr int kA = kS + DK * kDvs;
    static constexpr int kM = kA + kChunk * kChunk;
    static constexpr int kB = kM + kChunk * kChunk;
    static constexpr int kRef = kB + kChunk;        // b_I            [4][DK]
    static constexpr int kEB = kRef + kNb * DK;     // e^{b_I}        [4][DK]
    static constexpr int kEL = kEB + kNb * DK;      // e^{gl - b_I}   [4][DK]
    static constexpr int kW = kEL + kNb * DK;       // e^{b_I - b_J}  [6][DK]
    static constexpr int kDec = kW + 6 * DK;        // e^{gl}         [DK]
    static constexpr int kFloats = kDec + DK;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
    static_assert(kK % 4 == 0 && kQ % 4 == 0 && kM % 4 == 0 && kW % 4 == 0 && kU % 4 == 0 && kS % 4 == 0 &&
                      LDQ % 4 == 0 && LDK % 4 == 0 && kLdu % 4 == 0 && kDvs % 4 == 0,
                  "16-byte row loads");
};

__device__ __forceinline__ int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

template <typename Tin, int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
kda_chunk_simt_kernel(ChunkArgs a) {
    using L = SimtSmem<DK>;
    constexpr int C = kChunk;
    constexpr int NSL = DV / kDvs;
    extern __shared__ float sm[];
    float *Qs = sm + L::kQ, *Ks = sm + L::kK, *Hs = sm + L::kH, *Us = sm + L::kU;
    float *Ss = sm + L::kS, *As = sm + L::kA, *Ms = sm + L::kM, *Bs = sm + L::kB;
    float *Ref = sm + L::kRef, *EB = sm + L::kEB, *EL = sm + L::kEL, *Wv = sm + L::kW;
    float *Dec = sm + L::kDec;

    const int t = threadIdx.x;
    const int slice = blockIdx.x % NSL;
    const int uh = blockIdx.x / NSL;
    const int h = uh % a.heads, n = uh / a.heads;
    const int H = a.heads;
    int64_t bos, eos;
    seq_range(a, n, bos, eos);
    const int64_t len = eos - bos;
    const int col0 = slice * kDvs;

    const Tin *q = static_cast<const Tin *>(a.q);
    const Tin *k = static_cast<const Tin *>(a.k);
    const Tin *v = static_cast<const Tin *>(a.v);
    const Tin *g = static_cast<const Tin *>(a.g);
    const Tin *beta = static_cast<const Tin *>(a.beta);
    Tin *out = static_cast<Tin *>(a.out);

    // state slice [DK][64]
    const int64_t soff = ((int64_t)n * H + h) * DK * DV + col0;
    for (int x = t; x < DK * kDvs; x += kThreads) {
        const int c = x / kDvs, j = x % kDvs;
        Ss[x] = a.s0 ? a.s0[soff + (int64_t)c * DV + j] : 0.f;
    }

    const int j = t & (kDvs - 1);   // column owned in the GEMM-like phases
    const int rq = t >> 6;          // row phase (0..kRows-1)

    for (int64_t c0 = 0; c0 < len; c0 += C) {
        const int nr = (int)(len - c0 < C ? len - c0 : C);
        __syncthreads();   // previous chunk fully consumed
        const int64_t cs = ckpt_slot(a, n, c0);   // the state after c0 tokens, if due
        if (cs >= 0) {
            float *dst = a.ckpt + (cs * H + h) * DK * DV + col0;
            for (int x = t; x < DK * kDvs; x += kThreads) {
                const int c = x / kDvs, jj = x % kDvs;
                dst[(int64_t)c * DV + jj] = Ss[x];
            }
        }
        // ---- load the chunk (rows past the sequence end are zero: k = 0, beta = 0, g = 0)
        for (int x = t; x < C * DK; x += kThreads) {
            const int r = x / DK, c = x % DK;
            float qv = 0.f, kv = 0.f, gv = 0.f;
            if (r < nr) {
                const int64_t off = ((bos + c0 + r) * H + h) * DK + c;
                qv = to_f(q[off]); kv = to_f(k[off]); gv = to_f(g[off]);
            }
            Qs[r * L::LDQ + c] = qv; Ks[r * L::LDK + c] = kv; Hs[r * L::LDH + c] = gv;
        }
        for (int x = t; x < C * kDvs; x += kThreads) {
            const int r = x / kDvs, c = x % kDvs;
            Us[r * kLdu + c] = r < nr ? to_f(v[((bos + c0 + r) * H + h) * DV + col0 + c]) : 0.f;
        }
        if (t < C) Bs[t] = t < nr ? to_f(beta[(bos + c0 + t) * H + h]) : 0.f;
        __syncthreads();
        if (a.qk_eps >= 0.f) {
            // q and k rows L2-normalised ("はじめての自然言語処理 -- Kimi K3", section 3.1, the
            // read-out paragraph): x / sqrt(|x|^2 + eps) in fp32; a row with |x|^2 + eps = 0
            // stays zero.  One warp per row; rows past the sequence end are zero and stay so.
            const int warp = t >> 5, lane = t & 31;
            for (int row = warp; row < 2 * C; row += kThreads / 32) {
                float *x = row < C ? Qs + row * L::LDQ : Ks + (row - C) * L::LDK;
                float ss = 0.f;
                for (int c = lane; c < DK; c += 32) ss = fmaf(x[c], x[c], ss);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float den = ss + a.qk_eps;
                const float sc = den > 0.f ? rsqrtf(den) : 0.f;
                for (int c = lane; c < DK; c += 32) x[c] *= sc;
            }
            __syncthreads();
        }

        // ---- cumulative log decay per channel and the per-sub-tile reference vectors
        if (t < DK) {
            const int c = t;
            float run = 0.f, ref[kNb];
            ref[0] = 0.f;
            for (int r = 0; r < C; ++r) {
                if (r > 0 && (r % kSub) == 0) ref[r / kSub] = run;
                run += Hs[r * L::LDH + c];
                Hs[r * L::LDH + c] = run;
            }
            const float gl = run;
            for (int I = 0; I < kNb; ++I) {
                Ref[I * DK + c] = ref[I];
                EB[I * DK + c] = expf(ref[I]);
                EL[I * DK + c] = expf(gl - ref[I]);
                for (int J = 0; J < I; ++J) Wv[pair_index(I, J) * DK + c] = expf(ref[I] - ref[J]);
            }
            Dec[c] = expf(gl);
        }
        __syncthreads();
        // x = e^{gamma - b_I} in [e^-80, 1];  Q~ = Q x,  K~ = K x,  K^ = K / x
        for (int x = t; x < C * DK; x += kThreads) {
            const int r = x / DK, c = x % DK;
            const float d = Hs[r * L::LDH + c] - Ref[(r / kSub) * DK + c];
            const float kv = Ks[r * L::LDK + c];
            Qs[r * L::LDQ + c] *= expf(d);
            Ks[r * L::LDK + c] = kv * expf(d);
            Hs[r * L::LDH + c] = kv * expf(-d);
        }
        __syncthreads();

        // ---- A and M: dense dot products per 16x16 sub-tile pair (I >= J)
        {
            const int s = t & (C - 1);
            const int Js = s / kSub;
            float accA[kRpt], accM[kRpt];
#pragma unroll
            for (int m = 0; m < kRpt; ++m) { accA[m] = 0.f; accM[m] = 0.f; }
            for (int c = 0; c < DK; c += 4) {   // four channels a step: 16-byte row loads
                const float4 kh = make_float4(Hs[s * L::LDH + c], Hs[s * L::LDH + c + 1],
                                              Hs[s * L::LDH + c + 2], Hs[s * L::LDH + c + 3]);
                float4 khI[kNb];
#pragma unroll
                for (int I = 0; I < kNb; ++I) {
                    if (I > Js) {
                        const float4 w = *reinterpret_cast<const float4 *>(Wv + pair_index(I, Js) * DK + c);
                        khI[I] = make_float4(kh.x * w.x, kh.y * w.y, kh.z * w.z, kh.w * w.w);
                    } else {
                        khI[I] = kh;
                    }
                }
#pragma unroll
                for (int m = 0; m < kRpt; ++m) {
                    const int r = rq + kRows * m;   // in sub-tile (kRows m) / kSub: rq < kRows
                    const float4 f = khI[kRows * m / kSub];
                    const float4 k4 = *reinterpret_cast<const float4 *>(Ks + r * L::LDK + c);
                    const float4 q4 = *reinterpret_cast<const float4 *>(Qs + r * L::LDQ + c);
                    accA[m] = fmaf(k4.w, f.w, fmaf(k4.z, f.z, fmaf(k4.y, f.y, fmaf(k4.x, f.x, accA[m]))));
                    accM[m] = fmaf(q4.w, f.w, fmaf(q4.z, f.z, fmaf(q4.y, f.y, fmaf(q4.x, f.x, accM[m]))));
                }
            }
#pragma unroll
            for (int m = 0; m < kRpt; ++m) {
                const int r = rq + kRows * m;
                As[r * C + s] = s < r ? Bs[r] * accA[m] : 0.f;
                Ms[r * C + s] = s <= r ? accM[m] : 0.f;
            }
        }
        __syncthreads();
        // Qbar = Q~ e^{b_I}, Kbar = K~ e^{b_I}, Kp = K^ e^{gl - b_I}
        for (int x = t; x < C * DK; x += kThreads) {
            const int r = x / DK, c = x % DK, I = r / kSub;
            Qs[r * L::LDQ + c] *= EB[I * DK + c];
            Ks[r * L::LDK + c] *= EB[I * DK + c];
            Hs[r * L::LDH + c] *= EL[I * DK + c];
        }
        __syncthreads();

        // ---- Y = diag(beta) (V - Kbar S), in place over V
        {
            float acc[kRpt];
#pragma unroll
            for (int m = 0; m < kRpt; ++m) acc[m] = 0.f;
            for (int c = 0; c < DK; c += 4) {
                const float s0 = Ss[c * kDvs + j], s1 = Ss[(c + 1) * kDvs + j];
                const float s2 = Ss[(c + 2) * kDvs + j], s3 = Ss[(c + 3) * kDvs + j];
#pragma unroll
                for (int m = 0; m < kRpt; ++m) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(Ks + (rq + kRows * m) * L::LDK + c);
                    acc[m] = fmaf(k4.w, s3, fmaf(k4.z, s2, fmaf(k4.y, s1, fmaf(k4.x, s0, acc[m]))));
                }
            }
#pragma unroll
            for (int m = 0; m < kRpt; ++m) {
                const int r = rq + kRows * m;
                Us[r * kLdu + j] = Bs[r] * (Us[r * kLdu + j] - acc[m]);
            }
        }
        __syncthreads();
        // ---- (I + A) U = Y by forward substitution (row r uses rows s < r).  Columns are
        // independent: column jj belongs to eight lanes of one warp, which sync among themselves.
        {
            const int jj = t >> 3, part = t & 7;
            for (int r = 1; r < C; ++r) {
                float acc = 0.f;
                for (int s = part; s < r; s += 8) acc += As[r * C + s] * Us[s * kLdu + jj];
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                if (part == 0) Us[r * kLdu + jj] -= acc;
                __syncwarp();
            }
        }
        __syncthreads();
        // ---- O = Qbar S + M U
        {
            float acc[kRpt];
#pragma unroll
            for (int m = 0; m < kRpt; ++m) acc[m] = 0.f;
            for (int c = 0; c < DK; c += 4) {
                const float s0 = Ss[c * kDvs + j], s1 = Ss[(c + 1) * kDvs + j];
                const float s2 = Ss[(c + 2) * kDvs + j], s3 = Ss[(c + 3) * kDvs + j];
#pragma unroll
                for (int m = 0; m < kRpt; ++m) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(Qs + (rq + kRows * m) * L::LDQ + c);
                    acc[m] = fmaf(q4.w, s3, fmaf(q4.z, s2, fmaf(q4.y, s1, fmaf(q4.x, s0, acc[m]))));
                }
            }
            for (int s = 0; s < C; s += 4) {
                const float u0 = Us[s * kLdu + j], u1 = Us[(s + 1) * kLdu + j];
                const float u2 = Us[(s + 2) * kLdu + j], u3 = Us[(s + 3) * kLdu + j];
#pragma unroll
                for (int m = 0; m < kRpt; ++m) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(Ms + (rq + kRows * m) * C + s);
                    acc[m] = fmaf(m4.w, u3, fmaf(m4.z, u2, fmaf(m4.y, u1, fmaf(m4.x, u0, acc[m]))));
                }
            }
#pragma unroll
            for (int m = 0; m < kRpt; ++m) {
                const int r = rq + kRows * m;
                if (r < nr) out[((bos + c0 + r) * H + h) * DV + col0 + j] = from_f<Tin>(acc[m]);
            }
        }
        __syncthreads();
        // ---- S <- Diag(e^{gl}) S + Kp^T U: a 4 x 4 tile of (key channel, value column) per
        // thread, so each step over r reads four Kp values and one 16-byte row of U
        {
            constexpr int JB = kDvs / 4, CB = DK / 4;
            static_assert(CB * JB <= kThreads, "one tile per thread");
            if (t < CB * JB) {
                const int jb = t % JB, cb = t / JB;
                float4 acc[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int r = 0; r < C; ++r) {
                    const float4 u = *reinterpret_cast<const float4 *>(Us + r * kLdu + 4 * jb);
                    const float *hr = Hs + r * L::LDH + 4 * cb;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float hv = hr[e];
                        acc[e].x = fmaf(hv, u.x, acc[e].x);
                        acc[e].y = fmaf(hv, u.y, acc[e].y);
                        acc[e].z = fmaf(hv, u.z, acc[e].z);
                        acc[e].w = fmaf(hv, u.w, acc[e].w);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 4 * cb + e;
                    float4 *sp = reinterpret_cast<float4 *>(Ss + c * kDvs + 4 * jb);
                    const float4 o = *sp;
                    const float d = Dec[c];
                    *sp = make_float4(fmaf(d, o.x, acc[e].x), fmaf(d, o.y, acc[e].y), fmaf(d, o.z, acc[e].z),
                                      fmaf(d, o.w, acc[e].w));
                }
            }
        }
    }
    __syncthreads();
    if (a.sT) {
        for (int x = t; x < DK * kDvs; x += kThreads) {
            const int c = x / kDvs, jj = x % kDvs;
            a.sT[soff + (int64_t)c * DV + jj] = Ss[x];
        }
    }
}

__global__ void kda_state_copy_kernel(const float *src, float *dst, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : 0.f;
}

template <typename Tin, int DK, int DV>
cudaError_t launch_simt_t(const ChunkArgs &a, cudaStream_t st) {
    constexpr size_t smem = SimtSmem<DK>::kBytes;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_simt_kernel<Tin, DK, DV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.num_seqs * a.heads * (DV / kDvs);
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    kda_chunk_simt_kernel<Tin, DK, DV><<<(unsigned)units, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_simt_d(const ChunkArgs &a, int dk, int dv, cudaStream_t st) {
    if (dk == 128 && dv == 128) return launch_simt_t<Tin, 128, 128>(a, st);
    if (dk == 128 && dv == 64) return launch_simt_t<Tin, 128, 64>(a, st);
    if (dk == 64 && dv == 128) return launch_simt_t<Tin, 64, 128>(a, st);
    if (dk == 64 && dv == 64) return launch_simt_t<Tin, 64, 64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs &a, int dk, int dv, kda_dtype_t dt, cudaStream_t st) {
    return dt == KDA_F32 ? launch_simt_d<float>(a, dk, dv, st)
                         : launch_simt_d<__nv_bfloat16>(a, dk, dv, st);
}

cudaError_t launch_state_copy(const ChunkArgs &a, int dk, int dv, cudaStream_t st) {
    const int64_t n = (int64_t)a.num_seqs * a.heads * dk * dv;
    const int64_t blocks = (n + 255) / 256;
    kda_state_copy_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(a.s0, a.sT, n);
    return cudaGetLastError();
}

}  // namespace kda
