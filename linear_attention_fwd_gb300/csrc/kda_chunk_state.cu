// KDA chunkwise forward, two-pass form, pass 2: the state chain.
//
// bf16 inputs/outputs, d_k = d_v = 128, chunk C = 64, fp32 recurrent state.  One CTA
// (16 warps) per (sequence, head).  Pass 1 (kda_chunk_prep.cu) has already written each
// chunk's T = (I + A)^-1, M and M - fp16(M) to the workspace; per chunk this pass computes
// (the report's chunkwise form, "はじめての自然言語処理 -- Kimi K3", section 3.1)
//   Qbar = Q Gamma, Kbar = K Gamma, Kp = K Gamma_C / Gamma   (Gamma = e^gamma, gamma the
//                                                              cumulative log decay in the chunk)
//   U = T diag(beta) (V - Kbar S),  O = Qbar S + M U,  S <- Diag(Gamma_C) S + Kp^T U
// with the fp32 state resident in tensor memory for the whole sequence (transposed: TMEM lane
// j = value channel, column i = key channel) and its fp16 copies, and those of the per-chunk
// corrections, carried at a per-lane power-of-two scale (as in kda_chunk_tc.cu: S16 = S 2^-a_j
// with its largest entry in [2^14, 2^15), Z16 = Z 2^-z_j in [1, 2), state held at 2^-z_j).
//
// Warps 0-7 run the chain of chunk n; warps 8-15 meanwhile make chunk n + 1's Qbar, Kbar, Kp
// and decay (in shared memory buffers of their own), so the elementwise work overlaps the
// chain's tensor-core waits.  Per chunk, between CTA barriers:
//   A  warps 0-7: the previous chunk's output, 2^a O_I + 2^z (M U + low-order terms), through
//      a staging tile and one TMA store;  warps 8-15: chunk n + 1's decay sums, then S -> S16
//      (scale a_j) once the previous update landed;  T, M of chunk n + 1 requested
//   B  tcgen05: [O_I^T | P^T] = S16^T [Qbar; Kbar]^T, V^T = V^T I (V read MN-major);
//      warps 0-7: Z^T = diag(beta) (V^T - 2^a P^T) -> fp16 hi + lo at z_j;
//      warps 8-15: the first half of chunk n + 1's operand rows
// Copies run one to three chunks ahead (two buffers each for Q/K, G, T/M and Kp), since a
// copy takes a few microseconds to land when every SM streams.
//   C  tcgen05: U^T = Z^T T^T;  warps 0-7: S^T <- S^T Diag(Gamma_C) 2^(s - z), then U -> fp16
//      hi + lo;  warps 8-15: the second half of chunk n + 1's rows
//   D  tcgen05: S^T += U^T Kp (Kp read MN-major), (M U)^T = U^T M^T, low-order terms
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc_ptx.cuh"

namespace kda {

// Count of bounded device waits of this pass that gave up, since the host last read it.
__device__ unsigned int g_kda_state_timeouts = 0;

namespace {

using namespace ptx;

constexpr int C = 64;
constexpr int D = 128;
constexpr int NT = 512;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {   // 2^x, results below 2^-126 flushed
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 2^e as a float for an integer e in [-126, 127] (exact).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }
// 2^e for any integer e <= 127: exact down to 2^-149 (subnormal), 0 below.
__device__ __forceinline__ float pow2f(int e) {
    return e >= -126 ? pow2i(e) : (e >= -149 ? __int_as_float(1 << (e + 149)) : 0.f);
}
// floor(log2 m) for m > 0 finite (subnormals give -127); -1000 for m = 0.
__device__ __forceinline__ int exp2_floor(float m) {
    return m > 0.f ? (int)((__float_as_uint(m) >> 23) & 0xffu) - 127 : -1000;
}
__device__ __forceinline__ int clamp_i(int e, int lo, int hi) { return e < lo ? lo : (e > hi ? hi : e); }
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// max_i |x_i| as a tree of three-input maxima (eight independent chains)
template <int N>
__device__ __forceinline__ float absmax(const float (&x)[N]) {
    static_assert(N % 16 == 0, "multiple of 16");
    float m[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1]));
#pragma unroll
    for (int c = 16; c < N; c += 16)
#pragma unroll
        for (int e = 0; e < 8; ++e) m[e] = max3(m[e], fabsf(x[c + 2 * e]), fabsf(x[c + 2 * e + 1]));
    return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// shared memory map, byte offsets from a 1024-aligned base
constexpr uint32_t OFF_QK = 0;         // 2 x [Q -> Qbar; K -> Kbar] (fp16 over bf16): [64 r][128 i]
                                       // each, interleaved per 64-column half (Q at +0 / +16 KB, K at
                                       // +8 KB / +24 KB), so [Qbar; Kbar] is one 128-row operand
constexpr uint32_t QK_BYTES = 32768;
constexpr uint32_t OFF_G = 65536;      // 2 x G (bf16) [64 r][128 i], halves 8 KB apart
constexpr uint32_t G_BYTES = 16384;
constexpr uint32_t OFF_V = 98304;      // V (bf16) [64 r][128 j]
constexpr uint32_t OFF_KP = 114688;    // 2 x Kp (fp16) [64 r][128 i]: the MN-major B operand; once a
constexpr uint32_t KP_BYTES = 16384;   //   chunk's update has read it, that chunk's output staging
                                       //   tile [64 r][128 j] bf16 (stored by TMA)
constexpr uint32_t OFF_TM = 147456;    // 2 x {T (+0), M (+8 KB), M - fp16(M) (+16 KB)}, fp16 [64][64]
constexpr uint32_t TM_BYTES = 24576;
constexpr uint32_t OFF_NI = 196608;    // I (bf16, constant) [64 s][64 r]: V^T = V^T I
constexpr uint32_t OFF_SC = 204800;    // a_j, z_j ([2][128] int each), E_S [128], [2][128] fp32 maxima
constexpr uint32_t OFF_PART = OFF_SC + 3584;   // sub-tile sums of log2 decay [4][128] fp32
constexpr uint32_t OFF_DEC = OFF_PART + 2048;  // 2 x Gamma_C [128] fp32
constexpr uint32_t OFF_BETA = OFF_DEC + 1024;  // 2 x beta [64] fp32
constexpr uint32_t OFF_BAR = OFF_BETA + 512;   // mbarriers, TMEM address
constexpr uint32_t SMEM_USED = OFF_BAR + 96;
static_assert(OFF_SC >= OFF_NI + 8192, "map");
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_DEC % 16 == 0 && OFF_BETA % 16 == 0 && OFF_BAR % 8 == 0, "alignment");

// tensor memory columns (128 lanes = value channel j), as in the one-pass kernel
constexpr uint32_t TM_S = 0, TM_MU = 128, TM_OI = 192, TM_P = 256, TM_U = 320, TM_S16 = 384;
constexpr uint32_t TM_Z = 448, TM_ZL = 480, TM_UH = TM_Z, TM_UL = TM_ZL, TM_COLS = 512;
static_assert(TM_P == TM_OI + 64, "[O_I | P] is one N = 128 group");

constexpr uint32_t IDESC_N64 = idesc_f16_f32(128, 64);
constexpr uint32_t IDESC_N128 = idesc_f16_f32(128, 128);
constexpr uint32_t IDESC_N128_BMN = idesc_f16_f32(128, 128) | (1u << 16);   // B (Kp) MN-major
constexpr uint32_t IDESC_VT = idesc_bf16_f32(128, 64) | (1u << 15);         // A (V) MN-major

__device__ __forceinline__ uint32_t sw(int row, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                      ((col & 7) << 1));
}
__device__ __forceinline__ uint32_t swqk(int row, int col) {   // the interleaved Q / K tiles
    return (uint32_t)((col >> 6) * 16384 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}

// Longest packed sequences first (the hardware dispatches low block indices first); dense
// batches and large sequence counts keep their natural order.
__device__ __forceinline__ void select_unit(const ChunkArgs &a, int b, int &n, int &h) {
    __shared__ int s_pick;
    const int H = a.heads;
    h = b % H;
    const int r = b / H;
    n = r;
    if (a.cu == nullptr || a.num_seqs > NT) return;
    if (threadIdx.x == 0) s_pick = r;
    __syncthreads();
    const int t = threadIdx.x;
    if (t < a.num_seqs) {
        int64_t b0, e0;
        seq_range(a, t, b0, e0);
        const int64_t lt = e0 - b0;
        int rank = 0;
        for (int s = 0; s < a.num_seqs; ++s) {
            int64_t bs, es;
            seq_range(a, s, bs, es);
            const int64_t ls = es - bs;
            rank += (ls > lt) || (ls == lt && s < t);
        }
        if (rank == r) s_pick = t;
    }
    __syncthreads();
    n = s_pick;
}

__device__ __forceinline__ void tma_tile(const CUtensorMap *map, uint32_t dst, uint32_t bar, int h, int64_t tok,
                                         uint32_t half_stride) {
    tma_load_3d(dst, map, bar, 0, h, (int)tok);
    tma_load_3d(dst + half_stride, map, bar, 64, h, (int)tok);
}

__global__ void __launch_bounds__(NT, 1)
kda_chunk_state_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmg,
                       const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmo,
                       const ChunkArgs a,
                       const int32_t *__restrict__ chunk_base, const uint32_t wait_limit) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.heads;

    int n, h;
    select_unit(a, (int)blockIdx.x, n, h);
    int64_t bos, eos;
    seq_range(a, n, bos, eos);
    const int64_t len = eos - bos;
    const int nchunks = (int)((len + C - 1) / C);
    const int64_t slot0 = (int64_t)__ldg(chunk_base + n) * H + h;   // chunk c: slot0 + c * H

    // mbarriers: Q and K tiles of buffer 0 / 1 landed, G of buffer 0 / 1 landed, V landed, T
    // and M of buffer 0 / 1 landed; [O_I | P] and V^T done; U done; state and (M U_hi) update
    // done; low-order terms done
    const uint32_t bar_qk0 = sb + OFF_BAR, bar_g0 = sb + OFF_BAR + 16, bar_v = sb + OFF_BAR + 32;
    const uint32_t bar_tm0 = sb + OFF_BAR + 40, bar_p = sb + OFF_BAR + 56, bar_u = sb + OFF_BAR + 64;
    const uint32_t bar_s = sb + OFF_BAR + 72, bar_o = sb + OFF_BAR + 80;
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(sm + OFF_BAR + 88);
    int *ASC = reinterpret_cast<int *>(sm + OFF_SC);   // [2][128]
    int *ZSC = ASC + 256;                              // [2][128]
    int *ESC = ZSC + 256;                              // [128]
    float *XCH = reinterpret_cast<float *>(ESC + 128); // [2][128]
    float *PART = reinterpret_cast<float *>(sm + OFF_PART);
    float *DEC = reinterpret_cast<float *>(sm + OFF_DEC);
    float *BETA = reinterpret_cast<float *>(sm + OFF_BETA);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);

    if (tid == 0) {
        mbar_init(bar_qk0, 1);
        mbar_init(bar_qk0 + 8, 1);
        mbar_init(bar_g0, 1);
        mbar_init(bar_g0 + 8, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_tm0, 1);
        mbar_init(bar_tm0 + 8, 1);
        mbar_init(bar_p, 1);
        mbar_init(bar_u, 2);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmg);
        prefetch_tmap(&tmw);
        prefetch_tmap(&tmo);
    }
    if (warp == 0) {
        tmem_alloc(sb + OFF_BAR + 88, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);   // this warp's TMEM lanes
    const int jl = 32 * (warp & 3) + lane;   // this thread's TMEM lane (value channel j)
    const uint64_t dsm = sdesc_sw128(sb);

    // ---- initial state -> TMEM (scale exponent 0)
    const int64_t sbase = ((int64_t)n * H + h) * D * D;
    {
        const int quarter = warp >> 2;
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = a.s0 ? a.s0[sbase + (int64_t)(32 * quarter + c) * D + jl] : 0.f;
        tmem_st32(trow + TM_S + 32 * quarter, v);
        tmem_wait_st();
    }
    if (tid < 256) ZSC[tid] = 0;
    for (int x = tid; x < 64 * 32; x += NT) {   // I: copies V^T into tensor memory inside an MMA
        const int r = x >> 5, s2 = 2 * (x & 31);
        *reinterpret_cast<uint32_t *>(sm + OFF_NI + sw(r, s2, 64)) =
            (s2 == r ? 0x3F80u : 0u) | (s2 + 1 == r ? 0x3F800000u : 0u);
    }
    if (tid == 0 && nchunks > 0) {
        mbar_arrive_expect_tx(bar_qk0, 2 * 16384);
        tma_tile(&tmq, sb + OFF_QK, bar_qk0, h, bos, 16384);
        tma_tile(&tmk, sb + OFF_QK + 8192, bar_qk0, h, bos, 16384);
        mbar_arrive_expect_tx(bar_g0, 16384);
        tma_tile(&tmg, sb + OFF_G, bar_g0, h, bos, 8192);
        mbar_arrive_expect_tx(bar_v, 16384);
        tma_tile(&tmv, sb + OFF_V, bar_v, h, bos, 8192);
        mbar_arrive_expect_tx(bar_tm0, 3 * 8192);
        for (int m = 0; m < 3; ++m) tma_load_3d(sb + OFF_TM + 8192 * m, &tmw, bar_tm0, 0, 64 * m, (int)slot0);
        if (nchunks > 1) {
            mbar_arrive_expect_tx(bar_g0 + 8, 16384);
            tma_tile(&tmg, sb + OFF_G + G_BYTES, bar_g0 + 8, h, bos + C, 8192);
            mbar_arrive_expect_tx(bar_tm0 + 8, 3 * 8192);
            for (int m = 0; m < 3; ++m)
                tma_load_3d(sb + OFF_TM + TM_BYTES + 8192 * m, &tmw, bar_tm0 + 8, 0, 64 * m, (int)(slot0 + H));
            mbar_arrive_expect_tx(bar_qk0 + 8, 2 * 16384);
            tma_tile(&tmq, sb + OFF_QK + QK_BYTES, bar_qk0 + 8, h, bos + C, 16384);
            tma_tile(&tmk, sb + OFF_QK + QK_BYTES + 8192, bar_qk0 + 8, h, bos + C, 16384);
        }
    }
    if (tid < C) BETA[tid] = tid < len ? __bfloat162float(beta[(bos + tid) * H + h]) : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t ph_qk[2] = {0, 0}, ph_g[2] = {0, 0}, ph_v = 0, ph_tm[2] = {0, 0}, ph_p = 0, ph_u = 0, ph_s = 0, ph_o = 0;
    bool ok = true;

    // ---- warps 8-15: chunk m's decay and operands, in two halves of its rows (rows 0-7, then
    // 8-15, of each 16-row group).  Thread: channel pair cp, 16-row group grp.  gamma runs from
    // the chunk start: Gamma = e^gamma in (0, 1], Gamma_C / Gamma = e^{gamma_C - gamma} in
    // (0, 1] -- both within fp16's range, with no inverse decay (the sub-tile references that
    // keep e^{-gamma} within e^80 belong to A and M, made by pass 1).
    const int pt = tid - 256, cp = pt & 63, grp = pt >> 6;
    float2 lrun = make_float2(0.f, 0.f), lC = make_float2(0.f, 0.f);
    auto prep_sums = [&](int m) -> bool {   // returns false when a wait gave up
        bool got = mbar_wait(bar_qk0 + 8 * (m & 1), ph_qk[m & 1], wait_limit);
        got = mbar_wait(bar_g0 + 8 * (m & 1), ph_g[m & 1], wait_limit) && got;
        const uint32_t gt = OFF_G + G_BYTES * (m & 1);
        const int nrm = (int)(len - (int64_t)m * C < C ? len - (int64_t)m * C : C);
        const int c2 = 2 * cp;
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const int r = 16 * grp + rr;
            const float2 g2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + gt + sw(r, c2, 64)));
            if (r < nrm) { l0 = fmaf(g2.x, LOG2E, l0); l1 = fmaf(g2.y, LOG2E, l1); }
        }
        PART[grp * 128 + c2] = l0;
        PART[grp * 128 + c2 + 1] = l1;
        named_bar(5, 256);   // warps 8-15
        float2 base = make_float2(0.f, 0.f), tot = make_float2(0.f, 0.f);
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
            const float2 p2 = *reinterpret_cast<const float2 *>(PART + gg * 128 + c2);
            if (gg < grp) base = make_float2(base.x + p2.x, base.y + p2.y);
            tot = make_float2(tot.x + p2.x, tot.y + p2.y);
        }
        lrun = base;
        lC = tot;
        if (grp == 0) {
            *reinterpret_cast<float2 *>(DEC + 128 * (m & 1) + c2) = make_float2(ex2(tot.x), ex2(tot.y));
        }
        return got;
    };
    auto prep_rows = [&](int m, int half) {
        const int nrm = (int)(len - (int64_t)m * C < C ? len - (int64_t)m * C : C);
        const int c2 = 2 * cp;
        const uint32_t qk = OFF_QK + QK_BYTES * (m & 1), kp = OFF_KP + KP_BYTES * (m & 1), gt = OFF_G + G_BYTES * (m & 1);
#pragma unroll 4
        for (int rr = 0; rr < 8; ++rr) {
            const int r = 16 * grp + 8 * half + rr;
            const uint32_t off = sw(r, c2, 64), oqk = swqk(r, c2);
            const float2 q2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + qk + oqk));
            const float2 k2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + qk + 8192 + oqk));
            const float2 g2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + gt + off));
            const float w2 = r < nrm ? LOG2E : 0.f;   // decay past the sequence end is not summed
            lrun = __ffma2_rn(g2, make_float2(w2, w2), lrun);
            const float2 gm = make_float2(ex2(lrun.x), ex2(lrun.y));
            const float2 gp = make_float2(ex2(lC.x - lrun.x), ex2(lC.y - lrun.y));
            const float2 qb = __fmul2_rn(q2, gm), kb = __fmul2_rn(k2, gm), kpp = __fmul2_rn(k2, gp);
            *reinterpret_cast<uint32_t *>(sm + qk + oqk) = pack_f16(qb.x, qb.y);
            *reinterpret_cast<uint32_t *>(sm + qk + 8192 + oqk) = pack_f16(kb.x, kb.y);
            *reinterpret_cast<uint32_t *>(sm + kp + off) = pack_f16(kpp.x, kpp.y);
        }
    };

    // chunk 0's operands
    if (nchunks > 0 && warp >= 8) {
        const bool got = prep_sums(0);
        prep_rows(0, 0);
        prep_rows(0, 1);
        if (!got) ok = false;
    }
    ph_qk[0] ^= 1;
    ph_g[0] ^= 1;
    fence_async_smem();
    if (__syncthreads_or(!ok)) ok = false;
    if (ok && tid == 256 && nchunks > 2) {   // G buffer 0 is consumed: chunk 2's
        mbar_arrive_expect_tx(bar_g0, 16384);
        tma_tile(&tmg, sb + OFF_G, bar_g0, h, bos + 2 * C, 8192);
    }

    int spar = 1;   // the scale row holding z_j of the TMEM state (row 1 = 0 at start)
    // O^T = 2^a_j O_I^T + 2^z_j ((M U_hi)^T + low-order terms) of the chunk whose scales are in
    // row `par`: a whole chunk goes through the staging tile and one TMA store (issued by thread 0
    // once warps 0-7 have written it); the last, partial chunk of a sequence is stored from
    // registers (a warp writes 64 contiguous bytes per row), so that nothing lands past the
    // sequence.  Warps 0-7; warp w: lanes 32(w%4).., rows 32(w/4)..+31.
    auto stage_store = [&](int par, int64_t t0o, int nro) {
        const int r0 = 32 * (warp >> 2);
        float v[32], w[32];
        tmem_ld32x2(trow + TM_MU + r0, trow + TM_U + r0, v, w);
        const float fz = pow2i(ZSC[par * 128 + jl]), fa = pow2f(ASC[par * 128 + jl]);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = (v[c] + w[c]) * fz;
        tmem_ld32(trow + TM_OI + r0, w);
        if (nro == C) {   // the tile: this chunk's Kp buffer, which its update has read
            __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_KP + KP_BYTES * par);
#pragma unroll
            for (int c = 0; c < 32; ++c) os[(r0 + c) * D + jl] = __float2bfloat16_rn(fmaf(w[c], fa, v[c]));
            fence_async_smem();
            named_bar(6, 256);   // warps 0-7: the tile is written
            if (tid == 0) {   // read out before the next chunk's Kp is written there
                tma_store_3d(&tmo, sb + OFF_KP + KP_BYTES * par, 0, h, (int)t0o);
                bulk_commit();
                bulk_wait_read0();
            }
        } else {
            __nv_bfloat16 *o = out + ((t0o + r0) * H + h) * D + jl;
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (r0 + c < nro) o[(int64_t)c * H * D] = __float2bfloat16_rn(fmaf(w[c], fa, v[c]));
        }
    };

    bool out_pending = false;
    int64_t t0_out = 0;
    int nr_out = 0;
    const uint64_t vdesc = sdesc_sw128_mn(sb + OFF_V, 64 * 128, 1024);
#pragma unroll 1
    for (int ci = 0; ok && ci < nchunks; ++ci) {
        const int64_t t0 = bos + (int64_t)ci * C;
        const int nr = (int)(len - (int64_t)ci * C < C ? len - (int64_t)ci * C : C);
        const bool more = ci + 1 < nchunks;
        const int buf = ci & 1, cpar = ci & 1;
        const uint64_t qkd = dsm + ((OFF_QK + QK_BYTES * buf) >> 4), tmd = dsm + ((OFF_TM + TM_BYTES * buf) >> 4);
        const uint64_t kpd = sdesc_sw128_mn(sb + OFF_KP + KP_BYTES * buf, 64 * 128, 1024);
        bool got = true;

        // ---- A: the previous chunk's output (warps 0-7); the next chunk's sums, then S -> S16
        // once the previous update has landed (warps 8-15); the next chunk's T and M requested
        if (warp < 8) {
            if (out_pending) {
                got = mbar_wait(bar_s, ph_s, wait_limit) && mbar_wait(bar_o, ph_o, wait_limit);
                __syncwarp();
                tc_fence_after();
                if (tid == 0 && got && more) {   // the next chunk's T and M (the previous update read M)
                    const uint32_t bt = bar_tm0 + 8 * (buf ^ 1), dt = sb + OFF_TM + TM_BYTES * (buf ^ 1);
                    mbar_arrive_expect_tx(bt, 3 * 8192);
                    for (int m = 0; m < 3; ++m)
                        tma_load_3d(dt + 8192 * m, &tmw, bt, 0, 64 * m, (int)(slot0 + (int64_t)(ci + 1) * H));
                }
                __syncwarp();
                stage_store(spar, t0_out, nr_out);
            }
        } else {
            if (more) got = prep_sums(ci + 1);   // while the previous update runs
            if (out_pending) got = mbar_wait(bar_s, ph_s, wait_limit) && got;
            __syncwarp();
            tc_fence_after();
            const int i0 = 64 * ((warp - 8) >> 2);
            float v[32], w[32];
            tmem_ld32x2(trow + TM_S + i0, trow + TM_S + i0 + 32, v, w);
            const int sz = ZSC[spar * 128 + jl];   // S = (TMEM state) 2^sz
            XCH[((warp - 8) >> 2) * 128 + jl] = fmaxf(absmax(v), absmax(w));
            named_bar(3, 256);   // warps 8-15 (w and w + 4 share their lanes)
            const int es = exp2_floor(fmaxf(XCH[jl], XCH[128 + jl]));
            const int d = 14 - es < 126 ? 14 - es : 126;   // largest |S16| in [2^14, 2^15)
            if (warp < 12) {
                ASC[cpar * 128 + jl] = sz - d;
                ESC[jl] = es > -1000 ? es + sz : -1000;
            }
            const float2 f1 = make_float2(pow2i(d), pow2i(d));
            uint32_t hv[16], hw[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float2 x = __fmul2_rn(make_float2(v[2 * c], v[2 * c + 1]), f1);
                const float2 y = __fmul2_rn(make_float2(w[2 * c], w[2 * c + 1]), f1);
                hv[c] = pack_f16(x.x, x.y);
                hw[c] = pack_f16(y.x, y.y);
            }
            tmem_st16u(trow + TM_S16 + i0 / 2, hv);
            tmem_st16u(trow + TM_S16 + i0 / 2 + 16, hw);
            tmem_wait_st();
        }
        if (out_pending) {
            ph_s ^= 1;
            ph_o ^= 1;
        }
        if (more) {
            ph_qk[(ci + 1) & 1] ^= 1;
            ph_g[(ci + 1) & 1] ^= 1;
        }
        out_pending = false;
        tc_fence_before();
        if (__syncthreads_or(!got)) { ok = false; break; }
        tc_fence_after();

        // ---- B: [O_I^T | P^T] = S16^T [Qbar; Kbar]^T and V^T = V^T I [commit: P] (thread 0);
        // warps 0-7: Z; warps 8-15: the next chunk's first rows and beta
        bool gv = true;
        if (tid == 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mma_f16_ts(tmem + TM_OI, tmem + TM_S16 + 8 * k, qkd + (((k >> 2) * 16384 + (k & 3) * 32) >> 4),
                           IDESC_N128, k > 0);
            gv = mbar_wait(bar_v, ph_v, wait_limit);
            if (gv) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16_ss(tmem + TM_U, vdesc + ((2048 * k) >> 4), dsm + ((OFF_NI + 32 * k) >> 4), IDESC_VT, k > 0);
            }
            mma_commit(bar_p);
        }
        ph_v ^= 1;
        got = gv;
        if (warp < 8) {
            got = mbar_wait(bar_p, ph_p, wait_limit) && got;
            __syncwarp();   // lane 0 of warp 0 issued above: the warp rejoins before the collective loads
            tc_fence_after();
            const int s0 = 32 * (warp >> 2);
            float pv[32], vv[32];
            tmem_ld32x2(trow + TM_P + s0, trow + TM_U + s0, pv, vv);   // (Kbar S)^T 2^-a_j, V^T
            const float fa = -pow2f(ASC[cpar * 128 + jl]);
            const float2 fa2 = make_float2(fa, fa);
            const float *bt = BETA + 64 * buf + s0;
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 b4 = *reinterpret_cast<const float4 *>(bt + c);
                const float2 t0v = __ffma2_rn(make_float2(pv[c], pv[c + 1]), fa2, make_float2(vv[c], vv[c + 1]));
                const float2 t1v = __ffma2_rn(make_float2(pv[c + 2], pv[c + 3]), fa2, make_float2(vv[c + 2], vv[c + 3]));
                const float2 z0 = __fmul2_rn(t0v, make_float2(b4.x, b4.y)), z1 = __fmul2_rn(t1v, make_float2(b4.z, b4.w));
                pv[c] = z0.x; pv[c + 1] = z0.y; pv[c + 2] = z1.x; pv[c + 3] = z1.y;
            }
            XCH[(warp >> 2) * 128 + jl] = absmax(pv);
            named_bar(4, 256);   // warps 0-7
            // z_j: the lane's largest |Z| maps into [1, 2); at least E_S - 86 so that the state
            // stays below 2^87; within 126 of the state's exponent (one float factor to move it)
            const int eZ = exp2_floor(fmaxf(XCH[jl], XCH[128 + jl]));
            const int eS = ESC[jl], sz = ZSC[spar * 128 + jl];
            const int zj = clamp_i(clamp_i(eZ > eS - 86 ? eZ : eS - 86, sz - 126, sz + 126), -126, 126);
            if (warp < 4) ZSC[cpar * 128 + jl] = zj;
            const float2 fz = make_float2(pow2i(-zj), pow2i(-zj));
            uint32_t zv[16], zl[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float2 z = __fmul2_rn(make_float2(pv[2 * c], pv[2 * c + 1]), fz);
                zv[c] = pack_f16(z.x, z.y);
                const float2 zlo = __ffma2_rn(unpack_f16(zv[c]), make_float2(-1.f, -1.f), z);
                zl[c] = pack_f16(zlo.x, zlo.y);
            }
            tmem_st16u(trow + TM_Z + s0 / 2, zv);
            tmem_st16u(trow + TM_ZL + s0 / 2, zl);
            tmem_wait_st();
        } else if (more) {
            // beta of the next chunk: loads issued first, stored after the rows (their latency
            // hides behind them)
            float bnext[2] = {0.f, 0.f};
            const int64_t nn = len - (int64_t)(ci + 1) * C;
            if (warp == 15)
                for (int e = 0; e < 2; ++e)
                    if (lane + 32 * e < nn) bnext[e] = __bfloat162float(beta[(t0 + C + lane + 32 * e) * H + h]);
            prep_rows(ci + 1, 0);
            if (warp == 15) {
                BETA[64 * (buf ^ 1) + lane] = bnext[0];
                BETA[64 * (buf ^ 1) + lane + 32] = bnext[1];
            }
        }
        ph_p ^= 1;
        tc_fence_before();
        if (__syncthreads_or(!got)) { ok = false; break; }
        // [O_I | P] and V^T have read Qbar, Kbar and V: the Q, K tiles two chunks ahead, and V
        // of the next chunk
        if (tid == 0) {
            if (ci + 2 < nchunks) {
                mbar_arrive_expect_tx(bar_qk0 + 8 * buf, 2 * 16384);
                tma_tile(&tmq, sb + OFF_QK + QK_BYTES * buf, bar_qk0 + 8 * buf, h, t0 + 2 * C, 16384);
                tma_tile(&tmk, sb + OFF_QK + QK_BYTES * buf + 8192, bar_qk0 + 8 * buf, h, t0 + 2 * C, 16384);
            }
            if (more) {
                mbar_arrive_expect_tx(bar_v, 16384);
                tma_tile(&tmv, sb + OFF_V, bar_v, h, t0 + C, 8192);
            }
        }

        // ---- C: U^T = Z^T_hi T^T + Z^T_lo T^T (threads 0 and 32) [commit: U, two arrivals];
        // warps 0-7: the state's decay and rescale, then U -> fp16 hi + lo; warps 8-15: the
        // next chunk's second rows
        bool gt = true;
        if (tid == 0 || tid == 32) {
            gt = mbar_wait(bar_tm0 + 8 * buf, ph_tm[buf], wait_limit);
            tc_fence_after();
            const uint32_t za = tid == 0 ? TM_Z : TM_ZL, ud = tid == 0 ? TM_U : TM_P;
            if (gt) {
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_f16_ts(tmem + ud, tmem + za + 8 * k, tmd + ((k * 32) >> 4), IDESC_N64, k > 0);
            }
            mma_commit(bar_u);
        }
        ph_tm[buf] ^= 1;
        got = gt;
        if (warp < 8) {
            __syncwarp();
            {   // S^T <- S^T Diag(Gamma_C) 2^{s_j - z_j} in place; warp w: 64 columns from 64(w/4)
                const int i0 = 64 * (warp >> 2);
                const float f = pow2i(ZSC[spar * 128 + jl] - ZSC[cpar * 128 + jl]);   // |step| <= 126
                const float2 f1 = make_float2(f, f);
                const float *dec = DEC + 128 * buf + i0;
                float v[32], w[32];
                tmem_ld32x2(trow + TM_S + i0, trow + TM_S + i0 + 32, v, w);
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dec + c);
                    const float4 e4 = *reinterpret_cast<const float4 *>(dec + 32 + c);
                    const float2 a2 = __fmul2_rn(__fmul2_rn(make_float2(v[c], v[c + 1]), f1), make_float2(d4.x, d4.y));
                    const float2 b2 = __fmul2_rn(__fmul2_rn(make_float2(v[c + 2], v[c + 3]), f1), make_float2(d4.z, d4.w));
                    const float2 c2 = __fmul2_rn(__fmul2_rn(make_float2(w[c], w[c + 1]), f1), make_float2(e4.x, e4.y));
                    const float2 e2 = __fmul2_rn(__fmul2_rn(make_float2(w[c + 2], w[c + 3]), f1), make_float2(e4.z, e4.w));
                    v[c] = a2.x; v[c + 1] = a2.y; v[c + 2] = b2.x; v[c + 3] = b2.y;
                    w[c] = c2.x; w[c + 1] = c2.y; w[c + 2] = e2.x; w[c + 3] = e2.y;
                }
                tmem_st32(trow + TM_S + i0, v);
                tmem_st32(trow + TM_S + i0 + 32, w);
                tmem_wait_st();
            }
            got = mbar_wait(bar_u, ph_u, wait_limit) && got;
            __syncwarp();
            tc_fence_after();
            {   // U^T -> fp16 hi + lo; warp w: columns 32(w/4)..
                const int r0 = 32 * (warp >> 2);
                float uv[32], u2[32];
                tmem_ld32x2(trow + TM_U + r0, trow + TM_P + r0, uv, u2);
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 u = __fadd2_rn(make_float2(uv[2 * e], uv[2 * e + 1]), make_float2(u2[2 * e], u2[2 * e + 1]));
                    hi[e] = pack_f16(u.x, u.y);
                    const float2 lo2 = __ffma2_rn(unpack_f16(hi[e]), make_float2(-1.f, -1.f), u);
                    lo[e] = pack_f16(lo2.x, lo2.y);
                }
                tmem_st16u(trow + TM_UH + r0 / 2, hi);
                tmem_st16u(trow + TM_UL + r0 / 2, lo);
                tmem_wait_st();
            }
        } else if (more) {
            prep_rows(ci + 1, 1);
        }
        ph_u ^= 1;
        fence_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!got)) { ok = false; break; }
        tc_fence_after();
        if (tid == 256 && ci + 3 < nchunks) {   // G of the next chunk is consumed: the same buffer
            const uint32_t bg = bar_g0 + 8 * ((ci + 1) & 1);   // for the chunk three ahead
            mbar_arrive_expect_tx(bg, 16384);
            tma_tile(&tmg, sb + OFF_G + G_BYTES * ((ci + 1) & 1), bg, h, t0 + 3 * C, 8192);
        }

        // ---- D: S^T += U^T_hi Kp and (M U)^T = U^T_hi M^T [commit: S] (thread 0);
        // U^T_lo M^T + U^T_hi Mlo^T into the U^T columns (consumed) [commit: O] (thread 32)
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16_ts(tmem + TM_S, tmem + TM_UH + 8 * ks, kpd + ((2048 * ks) >> 4), IDESC_N128_BMN, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16_ts(tmem + TM_MU, tmem + TM_UH + 8 * ks, tmd + ((8192 + ks * 32) >> 4), IDESC_N64, ks > 0);
            mma_commit(bar_s);
        } else if (tid == 32) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16_ts(tmem + TM_U, tmem + TM_UL + 8 * ks, tmd + ((8192 + ks * 32) >> 4), IDESC_N64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_f16_ts(tmem + TM_U, tmem + TM_UH + 8 * ks, tmd + ((16384 + ks * 32) >> 4), IDESC_N64, 1);
            mma_commit(bar_o);
        }
        out_pending = true;
        t0_out = t0;
        nr_out = nr;
        spar = cpar;
    }

    if (ok && out_pending) {   // the last chunk's update and output
        bool got = true;
        if (warp < 8) {
            got = mbar_wait(bar_s, ph_s, wait_limit) && mbar_wait(bar_o, ph_o, wait_limit);
            __syncwarp();
            tc_fence_after();
            if (__all_sync(0xffffffffu, got)) stage_store(spar, t0_out, nr_out);
            if (tid == 0) bulk_wait0();
        }
        ph_s ^= 1;
        ph_o ^= 1;
        if (__syncthreads_or(!got)) ok = false;
    }
    if (!ok) {
        // A bounded wait expired: let copies and MMAs in flight land (at most one phase of each
        // barrier, the one its parity names or the one before), count it and mark the state.
        if (tid == 0) {
            constexpr uint32_t drain = 1u << 12;
            const uint32_t bars[11] = {bar_qk0, bar_qk0 + 8, bar_g0, bar_g0 + 8, bar_v, bar_tm0, bar_tm0 + 8,
                                       bar_p, bar_u, bar_s, bar_o};
            const uint32_t phs[11] = {ph_qk[0], ph_qk[1], ph_g[0], ph_g[1], ph_v, ph_tm[0], ph_tm[1],
                                      ph_p, ph_u, ph_s, ph_o};
            bulk_wait0();
#pragma unroll
            for (int b = 0; b < 11; ++b) {
                mbar_wait(bars[b], phs[b], drain);
                mbar_wait(bars[b], phs[b] ^ 1u, drain);
            }
            atomicAdd(&g_kda_state_timeouts, 1u);
        }
        __syncthreads();
    }
    tc_fence_after();
    if (a.sT) {   // S = (TMEM state) 2^z_j
        const int quarter = warp >> 2;
        float v[32];
        tmem_ld32(trow + TM_S + 32 * quarter, v);
        const float fs = pow2i(ZSC[spar * 128 + jl]);
#pragma unroll
        for (int c = 0; c < 32; ++c)
            a.sT[sbase + (int64_t)(32 * quarter + c) * D + jl] = ok ? v[c] * fs : __int_as_float(0x7fc00000);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

bool make_map_qkg(CUtensorMap *m, const void *ptr, int64_t tokens, int H);
bool make_map_slots(CUtensorMap *m, void *slots, int64_t nslots);
bool make_map_out_rows(CUtensorMap *m, void *ptr, int64_t tokens, int H);

cudaError_t take_state_expiries(cudaStream_t st, unsigned int *count) {
    static const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(count, g_kda_state_timeouts, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_kda_state_timeouts, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

cudaError_t launch_chunk_state(const ChunkArgs &a, const void *workspace, cudaStream_t st) {
    const int64_t tokens = a.cu ? a.seqlen : (int64_t)a.num_seqs * a.seqlen;
    if (tokens >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    const int32_t *chunk_base = static_cast<const int32_t *>(workspace);
    void *slots = static_cast<uint8_t *>(const_cast<void *>(workspace)) + ws_header_bytes(a.num_seqs);
    const int64_t nslots = two_pass_slots(tokens, a.num_seqs, a.heads);
    CUtensorMap mq, mk, mv, mg, mw, mo;
    if (!make_map_qkg(&mq, a.q, tokens, a.heads) || !make_map_qkg(&mk, a.k, tokens, a.heads) ||
        !make_map_qkg(&mv, a.v, tokens, a.heads) || !make_map_qkg(&mg, a.g, tokens, a.heads) ||
        !make_map_slots(&mw, slots, nslots) || !make_map_out_rows(&mo, a.out, tokens, a.heads))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.num_seqs * a.heads;
    if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
    kda_chunk_state_kernel<<<(unsigned)units, NT, SMEM_BYTES, st>>>(mq, mk, mv, mg, mw, mo, a, chunk_base,
                                                                     a.wait_polls);
    return cudaGetLastError();
}

}  // namespace kda
