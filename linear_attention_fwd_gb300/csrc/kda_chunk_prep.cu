// KDA chunkwise forward, two-pass form, pass 1: the state-independent part of every chunk.
//
// bf16 inputs, d_k = 128, chunk C = 64, 16-token sub-tiles.  One CTA of 8 warps per
// (64-token chunk, head) of every sequence, all chunks at once (nothing here depends on the
// recurrent state), two CTAs per SM.  Per chunk it forms, as the report's chunkwise form
// does ("はじめての自然言語処理 -- Kimi K3", section 3.1: the Tril intra-chunk term, the
// decay folded into q times Gamma and k over Gamma as in the report's equation (4), and the
// 16-token tiles made dense by the g >= -5 bound):
//   per sub-tile I with reference b_I = gamma before its start, x = e^{gamma - b_I} in
//   [e^-80, 1],  Q~ = Q x (bf16 hi + lo),  K~ = K x,  K^ = K / x (bf16: the range e^+-80);
//   A_rs = beta_r (K~ K^^T)_rs (e^{b_I - b_J} per channel for J < I),  s <  r
//   M_rs =        (Q~ K^^T)_rs (same),                                 s <= r, diagonal exact
//   T = (I + A)^-1  (16x16 diagonal inverses by forward substitution, then the blocks below
//                    the diagonal level by level)
// and writes T (fp16), M (fp16) and M - fp16(M) (fp16) -- three 64 x 64 tiles, 24 KB -- to the
// caller's workspace by TMA store, in the layout pass 2 loads them into (128-byte swizzle).
// Pass 2 (kda_chunk_state.cu) runs the state chain per (sequence, head) from them.
//
// Workspace: [int32 chunk_base[N + 1], padded to 1 KB] then one 24 KB slot per (chunk, head):
// slot (chunk_base[n] + c) * H + h for chunk c of sequence n (chunk_base: the running count
// of 64-token chunks over the sequences before n, written by kda_chunk_base_kernel).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc_ptx.cuh"

namespace kda {

// Count of bounded device waits of this pass that gave up, since the host last read it.
__device__ unsigned int g_kda_prep_timeouts = 0;

namespace {

using namespace ptx;

constexpr int C = 64;          // chunk
constexpr int D = 128;         // d_k
constexpr int NT = 256;        // threads (8 warps)
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {   // 2^x, results below 2^-126 flushed
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 2^x kept down to 2^-190 (for the factors that multiply K^, whose entries reach e^80)
__device__ __forceinline__ float ex2_sub(float x) { return ex2(x + 64.f) * 0x1p-64f; }

// shared memory map, byte offsets from a 1024-aligned base
constexpr uint32_t OFF_Q = 0;          // Q -> Q~hi (bf16)          [64 r][128 i], 64-column halves 8 KB apart
constexpr uint32_t OFF_K = 16384;      // K -> K~   (bf16)
constexpr uint32_t OFF_G = 32768;      // G -> K^   (bf16)
constexpr uint32_t OFF_QLO = 49152;    // Q~ - bf16(Q~) (bf16)
constexpr uint32_t OFF_T = 65536;      // T fp16 [64 r][64 s]        } written out together:
constexpr uint32_t OFF_MT = 73728;     // M fp16                     } three consecutive 8 KB
constexpr uint32_t OFF_MLO = 81920;    // M - fp16(M), fp16          } tiles
constexpr uint32_t OFF_AT = 90112;     // A_IJ (I > J) fp16 [64 r][64 s]
constexpr uint32_t OFF_PART = 98304;   // sub-tile sums of log2 decay [4][128] fp32; A_II (fp32,
constexpr int LDA = 20;                //   [4][16][LDA]) once the factors are made
constexpr uint32_t OFF_W6 = OFF_PART + 4 * 16 * LDA * 4;   // e^{b_I - b_J} [6][128] bf16
constexpr uint32_t OFF_BETA = OFF_W6 + 6 * 128 * 2;        // beta [64] fp32
constexpr uint32_t OFF_MRR = OFF_BETA + 64 * 4;            // q_r . k_r [64] fp32
constexpr uint32_t OFF_BAR = OFF_MRR + 64 * 4;             // one mbarrier
constexpr uint32_t SMEM_BYTES = OFF_BAR + 16 + 1024;       // + alignment slack
static_assert(4 * 128 * 4 <= 4 * 16 * LDA * 4, "sums fit under A_II");
static_assert(OFF_MT == OFF_T + 8192 && OFF_MLO == OFF_MT + 8192, "output tiles are consecutive");
static_assert(2 * SMEM_BYTES <= 228 * 1024, "two CTAs per SM");

__device__ __forceinline__ uint32_t sw(int row, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                      ((col & 7) << 1));
}

__device__ __forceinline__ int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

__global__ void __launch_bounds__(NT, 2)
kda_chunk_prep_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmg, const __grid_constant__ CUtensorMap tmw,
                      const ChunkArgs a, const int32_t *__restrict__ chunk_base, const uint32_t wait_limit) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.heads;

    // ---- which chunk: slot = (chunk_base[n] + c) * H + h
    const int64_t slot = blockIdx.x;
    const int h = (int)(slot % H);
    const int64_t cg = slot / H;   // global chunk index
    int lo = 0, hi = a.num_seqs;   // the last n with chunk_base[n] <= cg (skipping empty sequences)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(chunk_base + mid) <= cg) lo = mid; else hi = mid;
    }
    const int n = lo;
    const int64_t c = cg - __ldg(chunk_base + n);
    int64_t bos, eos;
    seq_range(a, n, bos, eos);
    const int64_t t0 = bos + c * C;
    const int nr = (int)(eos - t0 < C ? eos - t0 : C);
    if (nr <= 0) return;   // a slot past the last chunk (the grid is sized from the chunk count)

    const uint32_t bar = sb + OFF_BAR;
    float *PART = reinterpret_cast<float *>(sm + OFF_PART);
    float *AF = PART;
    __nv_bfloat16 *W6 = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_W6);
    float *BETA = reinterpret_cast<float *>(sm + OFF_BETA);
    float *MRR = reinterpret_cast<float *>(sm + OFF_MRR);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, 3 * 16384);
        tma_load_3d(sb + OFF_Q, &tmq, bar, 0, h, (int)t0);
        tma_load_3d(sb + OFF_Q + 8192, &tmq, bar, 64, h, (int)t0);
        tma_load_3d(sb + OFF_K, &tmk, bar, 0, h, (int)t0);
        tma_load_3d(sb + OFF_K + 8192, &tmk, bar, 64, h, (int)t0);
        tma_load_3d(sb + OFF_G, &tmg, bar, 0, h, (int)t0);
        tma_load_3d(sb + OFF_G + 8192, &tmg, bar, 64, h, (int)t0);
    }
    if (tid < C) BETA[tid] = tid < nr ? __bfloat162float(beta[(t0 + tid) * H + h]) : 0.f;
    // the blocks above the diagonal blocks of T and M are zero
    for (int x = tid; x < 64 * 32; x += NT) {
        const int r = x >> 5, s2 = 2 * (x & 31);
        if ((s2 >> 4) > (r >> 4)) {
            *reinterpret_cast<uint32_t *>(sm + OFF_T + sw(r, s2, 64)) = 0u;
            *reinterpret_cast<uint32_t *>(sm + OFF_MT + sw(r, s2, 64)) = 0u;
            *reinterpret_cast<uint32_t *>(sm + OFF_MLO + sw(r, s2, 64)) = 0u;
        }
    }
    __syncthreads();
    bool got = mbar_wait(bar, 0, wait_limit);
    if (__syncthreads_or(!got)) {   // a bounded wait gave up: let the copies land, count it for
        if (tid == 0) {             // kda_device_status and leave the slot unwritten
            mbar_wait(bar, 0, 1u << 12);
            atomicAdd(&g_kda_prep_timeouts, 1u);
        }
        __syncthreads();
        return;
    }

    const int cp = tid & 63, sub = tid >> 6;   // channel pair, sub-tile (16 rows)
    const int t4 = lane & 3, g = lane >> 2;    // mma.sync fragment coordinates

    // ---- (1) per-channel sums of log2 decay over each 16-token sub-tile (rows >= nr count 0)
    {
        const int c2 = 2 * cp;
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const int r = 16 * sub + rr;
            const float2 g2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_G + sw(r, c2, 64)));
            if (r < nr) { l0 = fmaf(g2.x, LOG2E, l0); l1 = fmaf(g2.y, LOG2E, l1); }
        }
        PART[sub * 128 + c2] = l0;
        PART[sub * 128 + c2 + 1] = l1;
    }
    __syncthreads();
    // ---- (2) warps 0-3: the per-pair factors e^{b_I - b_J}; warps 4-7: q_r . k_r of sub-tile
    // I = warp - 4 from the raw bf16 tiles (exact products, fp32 sums): the diagonal of M
    if (warp < 4) {
        const int ch = tid;   // 128 channels
        const float t0s = PART[ch], t1s = PART[128 + ch], t2s = PART[256 + ch];
        const float bI[4] = {0.f, t0s, t0s + t1s, t0s + t1s + t2s};
#pragma unroll
        for (int I = 1; I < 4; ++I)
#pragma unroll
            for (int J = 0; J < I; ++J)
                W6[pair_index(I, J) * 128 + ch] = __float2bfloat16_rn(ex2_sub(bI[I] - bI[J]));
    } else {
        const int I = warp - 4;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(sb + OFF_Q + sw(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3), 64), a0, a1, a2, a3);
            ldsm_x4(sb + OFF_K + sw(16 * I + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3), 64),
                    b0, b1, b2, b3);
            mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
            mma_16816(acc[1], a0, a1, a2, a3, b2, b3);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (2 * t4 + e == g) MRR[16 * I + g + 8 * hh] = acc[hh][2 * hh + e];
    }
    __syncthreads();

    // ---- (3) operands, each rounded once from the exact inputs (bf16, the range e^+-80 the
    // decay bound admits): Q~ = Q x as hi + lo, K~ = K x, K^ = K / x, in place of Q, K, G.
    // Thread: channel pair cp, the 16 rows of sub-tile `sub`; x restarts at each sub-tile.
    // Rows past the end of the sequence hold finite data (the next sequence, or TMA zero
    // fill): their decay is not accumulated, their beta is 0, and the entries of A and M they
    // would feed lie above the diagonal or in rows the state pass never stores.
    {
        const int c2 = 2 * cp;
        float2 l = make_float2(0.f, 0.f);
        const float2 minus1 = make_float2(-1.f, -1.f);
#pragma unroll 4
        for (int rr = 0; rr < 16; ++rr) {
            const int r = 16 * sub + rr;
            const uint32_t off = sw(r, c2, 64);
            const float2 q2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_Q + off));
            const float2 k2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_K + off));
            const float2 g2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_G + off));
            const float w2 = r < nr ? LOG2E : 0.f;
            l = __ffma2_rn(g2, make_float2(w2, w2), l);
            const float2 x = make_float2(ex2(l.x), ex2(l.y));
            const float2 y = make_float2(ex2(-l.x), ex2(-l.y));
            const float2 qt = __fmul2_rn(q2, x), kt = __fmul2_rn(k2, x), kh = __fmul2_rn(k2, y);
            const uint32_t qh = pack_bf16(qt.x, qt.y);
            const float2 ql = __ffma2_rn(unpack_bf16(qh), minus1, qt);
            *reinterpret_cast<uint32_t *>(sm + OFF_Q + off) = qh;
            *reinterpret_cast<uint32_t *>(sm + OFF_QLO + off) = pack_bf16(ql.x, ql.y);
            *reinterpret_cast<uint32_t *>(sm + OFF_K + off) = pack_bf16(kt.x, kt.y);
            *reinterpret_cast<uint32_t *>(sm + OFF_G + off) = pack_bf16(kh.x, kh.y);
        }
    }
    __syncthreads();

    // ---- (4) A = beta K~ K^^T and M = Q~ K^^T on the 10 sub-tile pairs (I >= J), bf16 products
    // with fp32 accumulation.  Warps 0-3: A_II, I = warp, then (I + A_II)^-1 by forward
    // substitution.  Warps 4-7: M_II, I = warp - 4, as (Q~hi + Q~lo) K^^T below the diagonal and
    // the exact q_r . k_r on it; then the 6 off-diagonal pairs, single bf16 products with the
    // factor e^{b_I - b_J} applied to the right operand: A_IJ (times beta_r) into AT, M_IJ (hi,
    // lo) into M.
    if (warp < 4) {
        const int I = warp;
        float accA[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 4
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t ao = sw(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3), 64);
            const uint32_t bo = sw(16 * I + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3), 64);
            uint32_t ka[4], bh[4];
            ldsm_x4(sb + OFF_K + ao, ka[0], ka[1], ka[2], ka[3]);
            ldsm_x4(sb + OFF_G + bo, bh[0], bh[1], bh[2], bh[3]);
            mma_16816(accA[0], ka[0], ka[1], ka[2], ka[3], bh[0], bh[1]);
            mma_16816(accA[1], ka[0], ka[1], ka[2], ka[3], bh[2], bh[3]);
        }
        // A_II goes to AF (fp32); PART (under it) was last read in (2)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = 16 * I + g + 8 * hh;
                const int s0 = 16 * I + 8 * nt + 2 * t4;
                const float br = BETA[r];
                AF[r * LDA + (s0 & 15)] = s0 < r ? br * accA[nt][2 * hh] : 0.f;
                AF[r * LDA + (s0 & 15) + 1] = s0 + 1 < r ? br * accA[nt][2 * hh + 1] : 0.f;
            }
        __syncwarp();
        if (lane < 16) {
            // column jj of T_II: t_jj = 1, t_r = -sum_{s<r} A_rs t_s (rows above jj are 0)
            const int jj = lane;
            const float *Ab = AF + (16 * I) * LDA;
            float tcol[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float arow[16];
#pragma unroll
                for (int q4 = 0; q4 < (r + 3) / 4; ++q4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Ab + r * LDA + 4 * q4);
                    arow[4 * q4] = a4.x; arow[4 * q4 + 1] = a4.y; arow[4 * q4 + 2] = a4.z; arow[4 * q4 + 3] = a4.w;
                }
                float acc = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < r; ++s2) acc = fmaf(arow[s2], tcol[s2], acc);
                tcol[r] = r == jj ? 1.f : (r < jj ? 0.f : -acc);
            }
            __half *tt = reinterpret_cast<__half *>(sm + OFF_T);
#pragma unroll
            for (int r = 0; r < 16; ++r) tt[sw(16 * I + r, 16 * I + jj, 64) >> 1] = __float2half_rn(tcol[r]);
        }
    } else {
        {
            const int I = warp - 4;
            float accM[2][2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) { accM[0][nt][e] = 0.f; accM[1][nt][e] = 0.f; }
#pragma unroll 2
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ao = sw(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3), 64);
                const uint32_t bo = sw(16 * I + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3), 64);
                uint32_t qh[4], ql[4], bh[4];
                ldsm_x4(sb + OFF_Q + ao, qh[0], qh[1], qh[2], qh[3]);
                ldsm_x4(sb + OFF_QLO + ao, ql[0], ql[1], ql[2], ql[3]);
                ldsm_x4(sb + OFF_G + bo, bh[0], bh[1], bh[2], bh[3]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma_16816(accM[0][nt], qh[0], qh[1], qh[2], qh[3], bh[2 * nt], bh[2 * nt + 1]);
                    mma_16816(accM[1][nt], ql[0], ql[1], ql[2], ql[3], bh[2 * nt], bh[2 * nt + 1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = 16 * I + g + 8 * hh;
                    const int s0 = 16 * I + 8 * nt + 2 * t4;
                    const float mv0 = accM[0][nt][2 * hh] + accM[1][nt][2 * hh];
                    const float mv1 = accM[0][nt][2 * hh + 1] + accM[1][nt][2 * hh + 1];
                    const float m0 = s0 < r ? mv0 : (s0 == r ? MRR[r] : 0.f);
                    const float m1 = s0 + 1 < r ? mv1 : (s0 + 1 == r ? MRR[r] : 0.f);
                    const uint32_t mh = pack_f16(m0, m1);
                    const float2 mhf = unpack_f16(mh);
                    *reinterpret_cast<uint32_t *>(sm + OFF_MT + sw(r, s0, 64)) = mh;
                    *reinterpret_cast<uint32_t *>(sm + OFF_MLO + sw(r, s0, 64)) = pack_f16(m0 - mhf.x, m1 - mhf.y);
                }
        }
        // off-diagonal pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2): warp 4 -> 0, 1; 5 -> 2, 3;
        // 6 -> 4; 7 -> 5
        const int w4 = warp - 4;
        const int p_begin = w4 < 2 ? 2 * w4 : w4 + 2, p_end = w4 < 2 ? 2 * w4 + 2 : w4 + 3;
#pragma unroll 1
        for (int po = p_begin; po < p_end; ++po) {
            const int I = po < 1 ? 1 : (po < 3 ? 2 : 3);
            const int J = po < 1 ? 0 : (po < 3 ? po - 1 : po - 3);
            float accA[2][4], accM[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) { accA[nt][e] = 0.f; accM[nt][e] = 0.f; }
            const __nv_bfloat16 *w = W6 + pair_index(I, J) * 128 + 2 * t4;
#pragma unroll 4
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ao = sw(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3), 64);
                const uint32_t bo = sw(16 * J + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3), 64);
                uint32_t ka[4], qh[4], bh[4];
                ldsm_x4(sb + OFF_K + ao, ka[0], ka[1], ka[2], ka[3]);
                ldsm_x4(sb + OFF_Q + ao, qh[0], qh[1], qh[2], qh[3]);
                ldsm_x4(sb + OFF_G + bo, bh[0], bh[1], bh[2], bh[3]);
                const uint32_t wlo = *reinterpret_cast<const uint32_t *>(w + 16 * kk);
                const uint32_t whi = *reinterpret_cast<const uint32_t *>(w + 16 * kk + 8);
                bh[0] = mul_bf16x2(bh[0], wlo); bh[1] = mul_bf16x2(bh[1], whi);
                bh[2] = mul_bf16x2(bh[2], wlo); bh[3] = mul_bf16x2(bh[3], whi);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma_16816(accA[nt], ka[0], ka[1], ka[2], ka[3], bh[2 * nt], bh[2 * nt + 1]);
                    mma_16816(accM[nt], qh[0], qh[1], qh[2], qh[3], bh[2 * nt], bh[2 * nt + 1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = 16 * I + g + 8 * hh;
                    const int s0 = 16 * J + 8 * nt + 2 * t4;
                    const float br = BETA[r];
                    *reinterpret_cast<uint32_t *>(sm + OFF_AT + sw(r, s0, 64)) =
                        pack_f16(br * accA[nt][2 * hh], br * accA[nt][2 * hh + 1]);
                    const float m0 = accM[nt][2 * hh], m1 = accM[nt][2 * hh + 1];
                    const uint32_t mh = pack_f16(m0, m1);
                    const float2 mhf = unpack_f16(mh);
                    *reinterpret_cast<uint32_t *>(sm + OFF_MT + sw(r, s0, 64)) = mh;
                    *reinterpret_cast<uint32_t *>(sm + OFF_MLO + sw(r, s0, 64)) = pack_f16(m0 - mhf.x, m1 - mhf.y);
                }
        }
    }
    __syncthreads();

    // ---- (5) warps 0-2: the blocks of T below the diagonal, level by level,
    // T_IJ = -(sum_{K=J+1..I} T_IK A_KJ) T_JJ (T_IK with K > J is ready before T_IJ)
    if (warp < 3) {
        auto t_block = [&](int I, int J) {
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int K = J + 1; K <= I; ++K) {
                uint32_t a4[4], b4[4];
                ldsm_x4(sb + OFF_T + sw(16 * I + (lane & 15), 16 * K + ((lane >> 4) << 3), 64), a4[0], a4[1], a4[2], a4[3]);
                ldsm_x4_t(sb + OFF_AT + sw(16 * K + (lane & 7) + (((lane >> 3) & 1) << 3), 16 * J + ((lane >> 4) << 3), 64),
                          b4[0], b4[1], b4[2], b4[3]);
                mma_16816_f16(acc[0], a4[0], a4[1], a4[2], a4[3], b4[0], b4[1]);
                mma_16816_f16(acc[1], a4[0], a4[1], a4[2], a4[3], b4[2], b4[3]);
            }
            // the accumulator fragments of Y are the A fragments of Y T_JJ
            const uint32_t y0 = neg_f16x2(pack_f16(acc[0][0], acc[0][1])), y1 = neg_f16x2(pack_f16(acc[0][2], acc[0][3]));
            const uint32_t y2 = neg_f16x2(pack_f16(acc[1][0], acc[1][1])), y3 = neg_f16x2(pack_f16(acc[1][2], acc[1][3]));
            uint32_t b4[4];
            ldsm_x4_t(sb + OFF_T + sw(16 * J + (lane & 7) + (((lane >> 3) & 1) << 3), 16 * J + ((lane >> 4) << 3), 64),
                      b4[0], b4[1], b4[2], b4[3]);
            float x[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            mma_16816_f16(x[0], y0, y1, y2, y3, b4[0], b4[1]);
            mma_16816_f16(x[1], y0, y1, y2, y3, b4[2], b4[3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    *reinterpret_cast<uint32_t *>(sm + OFF_T + sw(16 * I + (lane >> 2) + 8 * hh, 16 * J + 8 * nt + 2 * (lane & 3), 64)) =
                        pack_f16(x[nt][2 * hh], x[nt][2 * hh + 1]);
        };
        t_block(warp + 1, warp);                 // (1,0) (2,1) (3,2)
        named_bar(1, 96);
        if (warp < 2) t_block(warp + 2, warp);   // (2,0) (3,1)
        named_bar(1, 96);
        if (warp == 0) t_block(3, 0);
    }
    // ---- (6) T, M, M_lo -> the slot, by TMA store (the async proxy reads what the threads wrote)
    fence_async_smem();
    __syncthreads();
    if (tid == 0) {
        tma_store_3d(&tmw, sb + OFF_T, 0, 0, (int)slot);
        tma_store_3d(&tmw, sb + OFF_MT, 0, 64, (int)slot);
        tma_store_3d(&tmw, sb + OFF_MLO, 0, 128, (int)slot);
        bulk_commit();
        bulk_wait0();
    }
}

// chunk_base[n] = number of 64-token chunks of the sequences before n, for n = 0..N (one CTA).
__global__ void kda_chunk_base_kernel(const ChunkArgs a, int32_t *__restrict__ chunk_base) {
    __shared__ int32_t carry, warp_sum[32];
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int N = a.num_seqs;
    for (int base = 0; base <= N; base += blockDim.x) {
        const int n = base + (int)threadIdx.x;
        int32_t v = 0;
        if (n < N) {
            int64_t b, e;
            seq_range(a, n, b, e);
            v = (int32_t)((e - b + C - 1) / C);
        }
        // inclusive scan within the block
        int32_t x = v;
        const int ln = threadIdx.x & 31, wp = threadIdx.x >> 5;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (ln >= o) x += y;
        }
        if (ln == 31) warp_sum[wp] = x;
        __syncthreads();
        if (wp == 0) {
            int32_t s = ln < (int)(blockDim.x >> 5) ? warp_sum[ln] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
                if (ln >= o) s += y;
            }
            warp_sum[ln] = s;
        }
        __syncthreads();
        const int32_t incl = x + (wp > 0 ? warp_sum[wp - 1] : 0) + carry;
        if (n <= N) chunk_base[n] = incl - v;   // exclusive
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = incl;
        __syncthreads();
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

// [tokens][H][128] bf16 as a 3-D tensor (128, H, tokens); 64 x 1 x 64 boxes, 128-byte swizzle.
bool make_map_qkg(CUtensorMap *m, const void *ptr, int64_t tokens, int H) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [tokens][H][128] bf16 as a 3-D tensor with 128 x 1 x 64 boxes and no swizzle: a box is a
// plain row-major [64 tokens][128 channels] tile (the output staging layout).
bool make_map_out_rows(CUtensorMap *m, void *ptr, int64_t tokens, int H) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The workspace's slots as a 3-D fp16 tensor (64 columns, 192 rows, slots): T, M, M_lo of a
// slot are rows 0-63, 64-127, 128-191; 64 x 64 x 1 boxes, 128-byte swizzle.
bool make_map_slots(CUtensorMap *m, void *slots, int64_t nslots) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {64, 192, (cuuint64_t)nslots};
    cuuint64_t strides[2] = {64 * 2, 192 * 64 * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, slots, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t take_prep_expiries(cudaStream_t st, unsigned int *count) {
    static const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(count, g_kda_prep_timeouts, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_kda_prep_timeouts, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

int64_t two_pass_slots(int64_t tokens, int64_t num_seqs, int heads) {
    return ((tokens + C - 1) / C + num_seqs) * heads;
}

size_t two_pass_workspace_bytes(int64_t tokens, int64_t num_seqs, int heads) {
    return ws_header_bytes(num_seqs) + (size_t)two_pass_slots(tokens, num_seqs, heads) * kSlotBytes;
}

cudaError_t launch_chunk_prep(const ChunkArgs &a, void *workspace, cudaStream_t st) {
    const int64_t tokens = a.cu ? a.seqlen : (int64_t)a.num_seqs * a.seqlen;
    if (tokens >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    int32_t *chunk_base = static_cast<int32_t *>(workspace);
    uint8_t *slots = static_cast<uint8_t *>(workspace) + ws_header_bytes(a.num_seqs);
    const int64_t nslots = two_pass_slots(tokens, a.num_seqs, a.heads);
    if (nslots > 0x7fffffffLL) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mg, mw;
    if (!make_map_qkg(&mq, a.q, tokens, a.heads) || !make_map_qkg(&mk, a.k, tokens, a.heads) ||
        !make_map_qkg(&mg, a.g, tokens, a.heads) || !make_map_slots(&mw, slots, nslots))
        return cudaErrorInvalidValue;
    kda_chunk_base_kernel<<<1, 1024, 0, st>>>(a, chunk_base);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kda_chunk_prep_kernel<<<(unsigned)nslots, NT, SMEM_BYTES, st>>>(mq, mk, mg, mw, a, chunk_base, a.wait_polls);
    return cudaGetLastError();
}

}  // namespace kda
