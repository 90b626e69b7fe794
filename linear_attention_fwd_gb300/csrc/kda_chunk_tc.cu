// KDA chunkwise forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// bf16 inputs/outputs, computed at d_k = d_v = 128 (a 64-wide head reads its missing channels
// as zeros), chunk C = 64, fp32 recurrent state.  CTAs of 16 warps run pieces of (sequence,
// head) units: for a dense batch the balanced schedule (one CTA per SM, each an equal-cost
// share of all chunks, so that a unit may be split between two CTAs), otherwise one CTA per
// unit or uniform segments of one; a piece that starts inside a sequence warms up from a zero
// state (see warm_start).  The fp32 state lives in tensor memory for the whole piece
// (transposed: TMEM lane j = value channel, column i = key channel), so the only HBM traffic is
// the q/k/v/g/beta tiles, the output, and the initial / final states (plus the warm-up chunks'
// tiles).  With the L2 option (kQk) each q and k row is first scaled by 1 / sqrt(|x|^2 + eps),
// the norms taken on mma.sync in step (1).
//
// Chunk algebra ("はじめての自然言語処理 -- Kimi K3" section 3.1: chunkwise form,
// Tril intra-chunk term, decay folded into q times Gamma and k over Gamma as in
// the report's equation (4), 16-token tiles made dense by the g >= -5 bound):
//   per 16-token sub-tile I with reference b_I = gamma before its start,
//     x = e^{gamma - b_I} in [e^-80, 1],  Q~ = Q x,  K~ = K x,  K^ = K / x;
//   A_rs = beta_r (K~ K^^T)_rs * (e^{b_I - b_J} per channel, J < I),  s <  r
//   M_rs =        (Q~ K^^T)_rs * (same), s <= r
//   T = (I + A)^-1 (16x16 diagonal inverses, then the off-diagonal blocks level by level)
//   U = T diag(beta) (V - Kbar S),  O = Qbar S + M U,  S <- Diag(e^{gamma_last}) S + Kp^T U.
//
// Operand precision: the sub-tile-scaled operands of A and M span
// [e^-80, e^80] and are bf16 (the range the decay bound was chosen for; Q~ as hi + lo
// for the diagonal blocks of M, whose diagonal itself is the exact q_r . k_r); every
// other tensor-core operand (S, Z = diag(beta)(V - Kbar S), T, U, Qbar, Kbar, Kp, M)
// is rounded to fp16 for 3 more mantissa bits, Z, U and M as hi + lo pairs where one
// rounding would show in the outputs; accumulation is fp32 throughout.
//
// Range of the fp16 copies.  T, M, Qbar, Kbar and Kp are bounded by the inputs'
// normalisation and the decay, but S, Z and U scale with v and the initial state, which
// the method leaves unbounded: (V, S0) -> (O, S) is linear.  Each value channel j (a TMEM
// lane) evolves on its own -- S[:, j], v_j and o_j are untouched by the other channels --
// so every copy carries a power-of-two scale per lane, chosen each chunk from the lane's
// own maximum: S16 = S 2^-a_j (largest entry in [2^14, 2^15)), Z16 = Z 2^-z_j (largest in
// [1, 2)), and the fp32 state in TMEM is held as S 2^-z_j so that U16 (in Z's scale)
// updates it directly.  Scaling by a power of two is exact; the outputs are
// 2^a_j (Qbar S16) + 2^z_j (M U16), each factor applied per lane in fp32.  Each exponent
// step is one float factor: z_j moves at most 126 from one chunk to the next (a lane whose
// values jump by more than 2^126 within a chunk may lose its smaller part), keeps the state
// below 2^87, and a state below 2^-112 of its scale is carried as fp16 subnormals or zero.
//
// Per chunk (the fp16 copies of S, beta (V - Kbar S) and U are tensor-memory
// operands, so the state path never goes through shared memory):
//   TMA       Q, K, V, G tiles (64 x 128 bf16, 128-byte swizzle) -> smem
//   SIMT      sub-tile cumulative decay, x and 1/x, scaled operands; S -> fp16 (scale a_j)
//   tcgen05   P^T = S16^T Kbar^T,  O_I^T = S16^T Qbar^T           (overlapping the next two steps)
//   mma.sync  A and M as 16x16 sub-tile products (the per-pair decay factor is
//             applied to the B fragments in registers); diagonal inverses by
//             forward substitution; off-diagonal blocks of T
//   SIMT      Z^T = diag(beta) (V^T - 2^a_j P^T) -> fp16 hi + lo (scale z_j, tensor memory only)
//   tcgen05   U^T = Z^T T^T;  then  S^T <- S^T Diag(dec) + U^T Kp,  (MU)^T = U^T M^T
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <type_traits>
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc_ptx.cuh"

namespace kda {

// Count of bounded device waits that gave up, on this device, since the host last read it
// (take_wait_expiries).  Device-global status, not working memory.
__device__ unsigned int g_kda_tc_timeouts = 0;

namespace {

using namespace ptx;

constexpr int C = 64;         // chunk
constexpr int D = 128;        // the head size the kernel computes at (d_k = d_v; 64-wide heads are padded)
constexpr int NT = 512;       // threads (16 warps)
constexpr float LOG2E = 1.4426950408889634f;

// 2^x on the special-function unit, results below 2^-126 flushed to zero.  Used where
// every factor it multiplies is at most O(1), so a flushed result only drops a term
// below 2^-126 of the operands' scale.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 2^x for the decay factors that multiply K^ = K e^{b_I - gamma}, whose entries reach
// e^80 ~ 2^115: a factor flushed at 2^-126 could drop a product as large as 2^-11, so results
// are kept down to 2^-190 (2^(x + 64) on the unit, then an exact scaling by 2^-64 that may
// give a subnormal); what is lost stays below 2^-75.
__device__ __forceinline__ float ex2_sub(float x) { return ex2(x + 64.f) * 0x1p-64f; }

// 2^e as a float for an integer e in [-126, 127] (exact).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// 2^e for any integer e <= 127: exact down to 2^-149 (subnormal), 0 below.
__device__ __forceinline__ float pow2f(int e) {
    return e >= -126 ? pow2i(e) : (e >= -149 ? __int_as_float(1 << (e + 149)) : 0.f);
}

// floor(log2 m) for m > 0 finite (subnormals give -127, which only lowers the scale chosen
// from it); -1000 for m = 0.
__device__ __forceinline__ int exp2_floor(float m) {
    return m > 0.f ? (int)((__float_as_uint(m) >> 23) & 0xffu) - 127 : -1000;
}

__device__ __forceinline__ int clamp_i(int e, int lo, int hi) { return e < lo ? lo : (e > hi ? hi : e); }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// max_i |x_i| over N values as a tree of three-input maxima (eight independent chains),
// so that its latency is a few dependent steps rather than N.
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
constexpr uint32_t OFF_Q = 0;          // Q -> Qbar (fp16)         [64 r][128 i]  swizzled, and
constexpr uint32_t OFF_K = 8192;       // K -> Kbar (fp16): the two tiles interleave per 64-column
                                       // half, so [Qbar; Kbar] is one 128-row MMA operand
constexpr uint32_t OFF_V = 32768;      // V (bf16)                 [64 r][128 j]
constexpr uint32_t OFF_G = 49152;      // G (bf16)                 [64 r][128 i]
constexpr uint32_t OFF_SST = 65536;    // Q~hi, K~ (bf16)          2 x [64 r][128 i]
constexpr uint32_t OFF_UST = 98304;    // Q~lo (bf16)              [64 r][128 i]
constexpr uint32_t OFF_NI = 114688;   // I (bf16, constant)       [64 s][64 r]: V^T = V^T I
constexpr uint32_t OFF_RED = 122880;   // gated output: row sums of squares [4][64] fp32
constexpr uint32_t OFF_SC = OFF_RED + 1024;   // per-lane scales and the maxima exchanged for them:
                                       //   a_j, z_j (int, [2 chunk parities][128]), E_S [128],
                                       //   two [2][128] fp32 exchange rows (3.5 KB; 131071 is the end)
constexpr uint32_t OFF_KPT = 131072;   // Kp^T fp16                [128 i][64 r]
constexpr uint32_t OFF_MT = 147456;    // M fp16                   [64 r][64 s]
constexpr uint32_t OFF_TT = 155648;    // A_IJ (I > J) fp16        [64 r][64 s]
constexpr uint32_t OFF_T = 163840;     // T fp16 [64 r][64 s]; with AT, the output staging tile
constexpr uint32_t OFF_STG = OFF_TT;   //   [64 r][128 j] bf16 at the start of a chunk
constexpr uint32_t OFF_KH = 172032;    // K^hi (bf16)              [64 r][128 i]
constexpr uint32_t OFF_PART = 188416;  // sub-tile half sums [8][128] fp32; A_II (fp32, [4][16][LDA])
constexpr int LDA = 20;                //   once the decay vectors are consumed
constexpr uint32_t OFF_EB = OFF_PART + 8 * 128 * 4;     // e^{b_I}          [4][128]
constexpr uint32_t OFF_EL = OFF_EB + 4 * 128 * 4;       // e^{gl - b_I}     [4][128]
constexpr uint32_t OFF_W6 = OFF_EL + 4 * 128 * 4;       // e^{b_I - b_J}    [6][128] bf16
constexpr uint32_t OFF_DEC = OFF_W6 + 6 * 128 * 2;      // e^{gl}           [128]
constexpr uint32_t OFF_BETA = OFF_DEC + 128 * 4;        // beta             [64]
constexpr uint32_t OFF_MRR = OFF_BETA + 64 * 4;         // q_r . k_r        [64]
constexpr uint32_t OFF_BNEXT = OFF_MRR + 64 * 4;        // the next chunk's beta [64]
constexpr uint32_t OFF_MLO = (OFF_BNEXT + 64 * 4 + 1023) / 1024 * 1024;  // M - fp16(M), fp16 [64 r][64 s]
constexpr uint32_t OFF_BAR = OFF_MLO + 8192;            // 7 mbarriers, TMEM address
constexpr uint32_t OFF_NQK = OFF_BAR + 64;              // q and k row factors 1/|x| (L2 option) [2][64]
constexpr uint32_t SMEM_USED = OFF_NQK + 2 * 64 * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;       // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_KH % 1024 == 0 && OFF_PART % 16 == 0 && OFF_T % 1024 == 0 && OFF_MLO % 1024 == 0 &&
                  OFF_BAR % 8 == 0 && OFF_KH == OFF_T + 8192 && OFF_PART == OFF_KH + 16384,
              "alignment");
static_assert(OFF_T == OFF_TT + 8192, "the output staging tile spans AT and T");
static_assert(4 * 16 * LDA * 4 <= OFF_W6 - OFF_PART, "A_II fits over the sums and vectors");

// tensor memory columns (128 lanes = value channel j)
constexpr uint32_t TM_S = 0;      // S^T 2^-z_j fp32                  128 columns
constexpr uint32_t TM_MU = 128;   // (M U_hi)^T 2^-z_j fp32 (follows S^T: one N = 192 group)    64
constexpr uint32_t TM_OI = 192;   // (Qbar S16)^T fp32                                          64
constexpr uint32_t TM_P = 256;    // (Kbar S16)^T fp32 (follows O_I^T: one N = 128 group)       64
constexpr uint32_t TM_U = 320;    // V^T, then U^T fp32, then the low-order terms of (M U)^T    64
constexpr uint32_t TM_S16 = 384;  // S^T 2^-a_j as fp16 pairs (MMA operand)                     64
constexpr uint32_t TM_Z = 448;    // Z^T fp16 pairs, hi; then U^T hi    32
constexpr uint32_t TM_ZL = 480;   // Z^T - hi, fp16 pairs; then U^T lo  32
constexpr uint32_t TM_UH = TM_Z;  // U^T is made after the U groups have read Z^T
constexpr uint32_t TM_UL = TM_ZL;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t IDESC_N64 = idesc_f16_f32(128, 64);
constexpr uint32_t IDESC_N128 = idesc_f16_f32(128, 128);
constexpr uint32_t IDESC_N192 = idesc_f16_f32(128, 192);
constexpr uint32_t IDESC_VT = idesc_bf16_f32(128, 64) | (1u << 15);   // A (V) MN-major
static_assert(OFF_MT == OFF_KPT + 16384 && TM_MU == TM_S + 128 && TM_P == TM_OI + 64, "adjacent operands");
static_assert(OFF_SC + 3584 <= OFF_KPT, "scale arrays fit");

// Byte offset of element (row, col) in a 128-byte-swizzled K-major tile of
// `rows` rows whose columns are split into 64-element halves.
__device__ __forceinline__ uint32_t sw(int row, int col, int rows) {
    return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                      ((col & 7) << 1));
}

// The same for the interleaved Q / K tiles (64-column halves 16 KB apart).
__device__ __forceinline__ uint32_t swqk(int row, int col) {
    return (uint32_t)((col >> 6) * 16384 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}

__device__ __forceinline__ int pair_index(int I, int J) { return I * (I - 1) / 2 + J; }

// Longest packed sequences first (the hardware dispatches low block indices
// first); dense batches and large sequence counts keep their natural order.
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

// Segments of one sequence on several CTAs.  The state a zero state reaches from chunk
// boundary c_run differs from the true state at a later boundary c_lo by the true state at
// c_run carried through the transitions in between, whose product has a 2-norm of at most
// prod_t max_i e^{g_t,i} * max(1, |1 - beta_t |k_t|^2|)  (||Diag(e^g)|| = max_i e^{g_i}, and
// I - beta k k^T has the eigenvalues 1 and 1 - beta |k|^2).  A CTA that stores the outputs of
// chunks [c_lo, c_hi) therefore starts from a zero state at the latest boundary at most
// kMaxWarmChunks chunks before c_lo where that bound has fallen to 2^-kHorizonLog2 (far below
// fp32 resolution), or else at the start of the sequence with its initial state (exact).
constexpr float kHorizonLog2 = 160.f;
constexpr int kMaxWarmChunks = 16;

// The chunk boundary c_run <= c_lo described above (block-wide; every thread returns the
// same value).  Chunks before c_lo are whole chunks of the sequence.
__device__ int warm_start(const ChunkArgs &a, int64_t bos, int h, int c_lo) {
    __shared__ float s_part[NT / 32];
    const int H = a.heads;
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(a.g);
    const __nv_bfloat16 *kq = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *bq = static_cast<const __nv_bfloat16 *>(a.beta);
    const int tid = threadIdx.x, r = tid >> 3, part = tid & 7;   // 8 threads per token row
    const int c_min = c_lo > kMaxWarmChunks ? c_lo - kMaxWarmChunks : 0;
    float acc = 0.f;   // log2 of the norm bound from chunk c to c_lo
    for (int c = c_lo - 1; c >= c_min; --c) {
        const int64_t tok = bos + (int64_t)c * C + r;
        const uint4 *gp = reinterpret_cast<const uint4 *>(gq + (tok * H + h) * a.dk + 16 * part);
        const uint4 *kp = reinterpret_cast<const uint4 *>(kq + (tok * H + h) * a.dk + 16 * part);
        float gm = -3.0e38f, ks = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (16 * part >= a.dk) break;   // a 64-wide head: parts 4-7 hold nothing
            const uint4 gv = __ldg(gp + u), kv = __ldg(kp + u);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 g2 = unpack_bf16(gw[e]), k2 = unpack_bf16(kw[e]);
                gm = fmaxf(gm, fmaxf(g2.x, g2.y));
                ks = fmaf(k2.x, k2.x, fmaf(k2.y, k2.y, ks));
            }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
            ks += __shfl_xor_sync(0xffffffffu, ks, o);
        }
        // with q and k normalised first, |k|^2 <= |k|^2 / (|k|^2 + eps) times 1 + 2^-7 (the bf16
        // rounding of the normalised entries)
        const float kn = a.qk_eps < 0.f ? ks : (ks + a.qk_eps > 0.f ? ks / (ks + a.qk_eps) * 1.0078125f : 0.f);
        const float amp = fabsf(1.f - __bfloat162float(bq[tok * H + h]) * kn);
        float lam = gm * LOG2E + (amp > 1.f ? __log2f(amp) : 0.f);   // this token's bound, log2
        lam += __shfl_xor_sync(0xffffffffu, lam, 8);    // the warp's 4 rows
        lam += __shfl_xor_sync(0xffffffffu, lam, 16);
        if ((tid & 31) == 0) s_part[tid >> 5] = lam;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) tot += s_part[w];
        __syncthreads();
        acc += tot;
        if (acc <= -kHorizonLog2) return c;
    }
    return 0;
}

// Balanced schedule, packed sequences: the host does not see the lengths, so each CTA finds its
// share on the device.  Items: max(chunks, 1) per (sequence, head) unit, sequence-major (an empty
// sequence's item writes its final state).  CTA b of G takes [snap(b W / G), snap((b+1) W / G)),
// where snap moves a boundary to its unit's start or end when either is at most kSnapChunks
// items away -- a pure function of the boundary, so neighbouring CTAs agree on it.
constexpr int kSnapChunks = 4;
__device__ __forceinline__ int64_t seq_items(const ChunkArgs &a, int n) {
    int64_t b, e;
    seq_range(a, n, b, e);
    const int64_t nc = (e - b + C - 1) / C;
    return nc > 0 ? nc : 1;
}
// Block-wide: W, the raw end (b + 1) W / G, and where the share starts: sequence n, head h,
// chunk c within that unit and the unit's first item us (c is the snapped start; it may equal the
// unit's item count, i.e. the start is the next unit's first item).
__device__ void packed_share(const ChunkArgs &a, int G, int b, int &n, int &h, int &c, int64_t &us,
                             int64_t &raw1) {
    __shared__ long long s_part[NT / 32];
    __shared__ long long s_w, s_start;
    __shared__ int s_seq;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int H = a.heads, N = a.num_seqs;
    long long mine = 0;
    for (int s = t; s < N; s += NT) mine += seq_items(a, s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0) s_part[warp] = mine;
    __syncthreads();
    if (t == 0) {
        long long w = 0;
        for (int i = 0; i < NT / 32; ++i) w += s_part[i];
        s_w = w * H;
        s_seq = 0;
        s_start = 0;
    }
    __syncthreads();
    const long long W = s_w;
    const long long raw0 = (long long)b * W / G;
    raw1 = (long long)(b + 1) * W / G;
    long long run = 0;   // items before this pass's first sequence (the same in every thread)
    for (int base = 0; base < N; base += NT) {
        __syncthreads();   // s_part is reused
        const int s = base + t;
        const long long w = s < N ? (long long)H * seq_items(a, s) : 0;
        long long v = w;   // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (lane == 31) s_part[warp] = v;
        __syncthreads();
        long long off = 0, tot = 0;
        for (int i = 0; i < NT / 32; ++i) {
            const long long u = s_part[i];
            off += i < warp ? u : 0;
            tot += u;
        }
        const long long excl = run + off + v - w;
        if (s < N && excl <= raw0 && raw0 < excl + w) {
            s_seq = s;
            s_start = excl;
        }
        run += tot;
    }
    __syncthreads();
    n = s_seq;
    const long long items = seq_items(a, n);
    h = (int)((raw0 - s_start) / items);
    us = s_start + (long long)h * items;
    const long long cc = raw0 - us;
    c = (int)(cc <= kSnapChunks ? 0 : (items - cc <= kSnapChunks ? items : cc));
    __syncthreads();   // the shared words are read before any later reuse
}

// Balanced schedule: the boundaries x_0 = 0 <= x_1 <= ... <= x_G = W of the CTAs' shares of the
// W items (units of nc chunks each, sequence-major), drawn on the host (draw_schedule).
constexpr int kMaxSchedCtas = 256;
struct SchedBounds {
    int64_t x[kMaxSchedCtas + 1];
};

__device__ __forceinline__ void tma_tile(const CUtensorMap *map, uint32_t dst, uint32_t bar, int h,
                                         int64_t tok, uint32_t half_stride = 8192) {
    tma_load_3d(dst, map, bar, 0, h, (int)tok);
    tma_load_3d(dst + half_stride, map, bar, 64, h, (int)tok);
}

// kMode: 0 = one CTA per unit, 1 = uniform segments (a.segments > 1), 2 = the balanced schedule
// (a.sched_ctas > 0), 3 = the balanced schedule with the output gate (which modes 1 and 2 never
// carry; checkpoints run in mode 0 only).  Each mode is its own instantiation, so that the
// others' logic folds away.  kQk: q and k L2-normalised first (modes 0-2, without the gate or
// checkpoints).
template <int kMode, bool kQk = false>
__global__ void __launch_bounds__(NT, 1)
kda_chunk_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmg,
                    const __grid_constant__ CUtensorMap tmz,
                    const ChunkArgs a, const uint32_t wait_limit, const __grid_constant__ SchedBounds sched) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.heads;

    // The CTA's work: pieces -- (sequence n, head h) and chunks [c_lo, c_hi) -- each run from
    // chunk c_run (see warm_start), storing the outputs of [c_lo, c_hi); the piece that holds a
    // unit's last chunk writes its final state.
    //  - balanced schedule (kMode 2, dense batches): the units' chunks in sequence-major order
    //    are W = units x chunks items; CTA b takes items [sched.x[b], sched.x[b + 1]), one piece
    //    per unit that range touches
    //  - uniform segments (kSeg, P = a.segments > 1): blockIdx.x = p * units + unit, chunks
    //    [p nc / P, (p + 1) nc / P) of that unit
    //  - otherwise blockIdx.x = unit (the longest packed sequences first), the whole unit
    const int64_t units = (int64_t)a.num_seqs * H;
    constexpr bool kSeg = kMode != 0;
    constexpr bool balanced = kMode >= 2;
    constexpr bool kGate = kMode == 0 || kMode == 3;   // the output gate
    constexpr bool kCkpt = kMode == 0;                 // checkpoints
    const int P = kSeg && !balanced && a.segments > 1 ? a.segments : 1;
    const int p = kSeg && !balanced ? (int)(blockIdx.x / units) : 0;
    const int ncd = (int)((a.seqlen + C - 1) / C);   // chunks per unit of a dense batch
    const bool packed = balanced && a.cu != nullptr;   // the share is found on the device
    int n = 0, h = 0, c_start = 0;
    // packed: the current unit's first item, the share's raw end, whether the share ends inside
    // the current unit -- in shared memory (read at piece boundaries only, written by thread 0
    // between barriers), not in registers that the chunk loop needs
    __shared__ long long s_pk[3];
    if (balanced) {
        if (packed) {
            int64_t us0, raw1;
            packed_share(a, a.sched_ctas, (int)blockIdx.x, n, h, c_start, us0, raw1);
            if (threadIdx.x == 0) {
                s_pk[0] = us0;
                s_pk[1] = raw1;
                s_pk[2] = 0;
            }
            __syncthreads();
        } else if (sched.x[blockIdx.x] >= sched.x[blockIdx.x + 1]) {
            return;   // no items (whole CTA, before any setup)
        }
    } else {
        select_unit(a, kSeg ? (int)(blockIdx.x % units) : (int)blockIdx.x, n, h);
    }
    int64_t bos = 0, len = 0;
    int nchunks = 0, c_lo = 0, c_hi = 0, c_run = 0;
    bool last_seg = true;
    // Moves to the CTA's next piece; false when it has none left.  (The balanced schedule's
    // position is recomputed from the current piece rather than kept: registers are scarce.)
    auto next_piece = [&](bool first) -> bool {
        if (packed) {
            int64_t us = s_pk[0], items = seq_items(a, n);
            const int64_t raw1 = s_pk[1];
            bool found = true, ends = false;
            if (first) {
                c_lo = c_start;
            } else if (s_pk[2]) {
                found = false;   // the share ended with the previous piece
            } else {
                c_lo = (int)items;   // the previous piece ended with its unit
            }
            if (found && c_lo >= items) {   // the next unit
                us += items;
                if (++h == H) {
                    h = 0;
                    ++n;
                }
                c_lo = 0;
                found = n < a.num_seqs;
                if (found) items = seq_items(a, n);
            }
            int64_t e = items;   // the piece's end item within the unit
            if (found) {
                ends = raw1 < us + items;
                if (ends) {
                    const int64_t ce = raw1 - us;
                    e = ce <= kSnapChunks ? 0 : (items - ce <= kSnapChunks ? items : ce);
                }
                found = c_lo < e;
            }
            __syncthreads();   // every thread has read s_pk
            if (threadIdx.x == 0) {
                s_pk[0] = us;
                s_pk[2] = ends;
            }
            if (!found) return false;
            int64_t eos;
            seq_range(a, n, bos, eos);
            len = eos - bos;
            nchunks = (int)((len + C - 1) / C);
            c_hi = e < nchunks ? (int)e : nchunks;
            last_seg = e == items;
            return true;
        }
        if (balanced) {
            const int64_t x = first ? sched.x[blockIdx.x] : ((int64_t)n * H + h) * ncd + c_hi;
            const int64_t x_end = sched.x[blockIdx.x + 1];
            if (x >= x_end) return false;
            const int64_t u = x / ncd;
            n = (int)(u / H);
            h = (int)(u % H);
            c_lo = (int)(x - u * ncd);
            c_hi = x_end - u * ncd < ncd ? (int)(x_end - u * ncd) : ncd;
        } else if (!first) {
            return false;
        }
        int64_t eos;
        seq_range(a, n, bos, eos);
        len = eos - bos;
        nchunks = (int)((len + C - 1) / C);
        if (!balanced) {
            c_lo = kSeg ? (int)((int64_t)p * nchunks / P) : 0;
            c_hi = kSeg ? (int)((int64_t)(p + 1) * nchunks / P) : nchunks;
        }
        last_seg = balanced ? c_hi == nchunks : (!kSeg || p == P - 1);
        return true;
    };
    if (!next_piece(true)) return;   // an empty packed share (whole CTA, before any setup)
    if (kSeg && !balanced && c_lo == c_hi && !last_seg) return;   // an empty segment (whole CTA, before any setup)

    // mbarriers: Q, K, G tiles landed; [O_I^T | P^T] done; V tile landed; U^T done; state (and
    // (M U_hi)^T) update done; low-order terms of (M U)^T done
    const uint32_t bar_tma = sb + OFF_BAR, bar_p = sb + OFF_BAR + 8, bar_v = sb + OFF_BAR + 16;
    const uint32_t bar_u = sb + OFF_BAR + 24, bar_s = sb + OFF_BAR + 32, bar_o = sb + OFF_BAR + 40;
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(sm + OFF_BAR + 48);
    const uint32_t bar_z = sb + OFF_BAR + 56;   // a chunk's gate logits landed in the staging tile
    float *AF = reinterpret_cast<float *>(sm + OFF_PART);   // A_II blocks, [4][16][LDA]
    float *PART = reinterpret_cast<float *>(sm + OFF_PART);
    float *MRR = reinterpret_cast<float *>(sm + OFF_MRR);
    float *EB = reinterpret_cast<float *>(sm + OFF_EB);
    float *EL = reinterpret_cast<float *>(sm + OFF_EL);
    __nv_bfloat16 *W6 = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_W6);
    // per-lane scale exponents (value channel j): a_j of S16 and z_j of Z16 / U16 / the
    // TMEM state, one row per chunk parity (a chunk's values are still read while the next
    // chunk's are made); E_S: exponent of the lane's largest |S| entering the chunk
    int *ASC = reinterpret_cast<int *>(sm + OFF_SC);            // [2][128]
    int *ZSC = ASC + 256;                                       // [2][128]
    int *ESC = ZSC + 256;                                       // [128]
    float *XCH = reinterpret_cast<float *>(ESC + 128);          // [2 halves][128] lane maxima
    float *DEC = reinterpret_cast<float *>(sm + OFF_DEC);
    float *BETA = reinterpret_cast<float *>(sm + OFF_BETA);
    const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out);

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_p, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_u, 2);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_z, 1);
        fence_mbar_init();
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmg);
    }
    if (warp == 0) {
        tmem_alloc(sb + OFF_BAR + 48, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);   // this warp's TMEM lanes
    const int jl = 32 * (warp & 3) + lane;   // this thread's TMEM lane (value channel j)
    const int quarter = warp >> 2;           // which column group this warp handles (0..3)
    // shared-memory operand descriptors are this base plus (byte offset >> 4): computed once,
    // outside the single-thread issue branches, so that issuing an MMA costs no address math
    const uint64_t dsm = sdesc_sw128(sb);

    for (int x = tid; x < 64 * 32; x += NT) {   // I: copies V^T into tensor memory inside an MMA
        const int r = x >> 5, s2 = 2 * (x & 31);
        *reinterpret_cast<uint32_t *>(sm + OFF_NI + sw(r, s2, 64)) =
            (s2 == r ? 0x3F80u : 0u) | (s2 + 1 == r ? 0x3F800000u : 0u);
    }
    // the blocks of M above the diagonal blocks stay zero for the whole sequence
    for (int x = tid; x < 64 * 32; x += NT) {
        const int r = x >> 5, s2 = 2 * (x & 31);
        if ((s2 >> 4) > (r >> 4)) {
            *reinterpret_cast<uint32_t *>(sm + OFF_MT + sw(r, s2, 64)) = 0u;
            *reinterpret_cast<uint32_t *>(sm + OFF_MLO + sw(r, s2, 64)) = 0u;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t ph_tma = 0, ph_p = 0, ph_v = 0, ph_u = 0, ph_s = 0, ph_o = 0, ph_z = 0;
    bool out_pending = false;   // the previous chunk's state update and O^T group are in flight
    int64_t t0_out = 0;
    int nr_out = 0;
    int spar = 1;               // the scale row holding z_j of the TMEM state (row 1 = 0 at start)
    // O^T = 2^a_j O_I^T + 2^z_j ((M U_hi)^T + low-order terms), from TMEM, of the chunk whose
    // scales are in row `par` -> bf16 staging tile [64 r][128 j] over the AT and T tiles, by
    // warps 0-7; warp w: lanes 32(w%4).., rows 32(w/4)..+31.  (M U)^T is then cleared for the
    // next chunk's update group, which accumulates into it together with the state.
    // With an output gate (the paragraph after the decay bound on the same page): each row is
    // normalised to unit RMS over its 128 value channels, scaled by the norm weight and
    // multiplied channel-wise by sigmoid(gate logit) before it is rounded to bf16; the chunk's
    // logits were loaded by TMA into the staging tile itself (same row-major layout).
    const bool gate_on = kGate && a.gate != nullptr;
    const float norm_wj = (gate_on && a.norm_w) ? a.norm_w[jl] : 1.f;   // this thread's channel
    auto stage_output = [&](int par) {
        if (warp >= 8) return;
        __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_STG);
        const int r0 = 32 * (warp >> 2);
        float v[32], w[32];
        tmem_ld32x2(trow + TM_MU + r0, trow + TM_U + r0, v, w);
        const float fz = pow2i(ZSC[par * 128 + jl]), fa = pow2f(ASC[par * 128 + jl]);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = (v[c] + w[c]) * fz;
        {
            uint32_t zero[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) zero[c] = 0u;
            tmem_st16u(trow + TM_MU + r0, zero);
            tmem_st16u(trow + TM_MU + r0 + 16, zero);
        }
        tmem_ld32(trow + TM_OI + r0, w);
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = fmaf(w[c], fa, v[c]);
        tmem_wait_st();
        if (gate_on) {
            // sums of squares of rows r0.. over this warp's 32 channels, transposed so that
            // lane L ends with row r0 + L (5 rounds, 31 shuffles)
#pragma unroll
            for (int c = 0; c < 32; ++c) w[c] = v[c] * v[c];
#pragma unroll
            for (int sft = 16; sft > 0; sft >>= 1) {
                const bool up = (lane & sft) != 0;
#pragma unroll
                for (int i = 0; i < sft; ++i) {
                    const float send = up ? w[i] : w[i + sft];
                    const float keep = up ? w[i + sft] : w[i];
                    w[i] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
                }
            }
            float *red = reinterpret_cast<float *>(sm + OFF_RED);   // [4 channel quarters][64 rows]
            red[(warp & 3) * 64 + r0 + lane] = w[0];
            named_bar(5 + (warp >> 2), 128);   // the four quarters of these 32 rows
            const float ms = ((red[r0 + lane] + red[64 + r0 + lane]) + (red[128 + r0 + lane] + red[192 + r0 + lane])) *
                             (1.f / D);
            const float rstd = rsqrtf(ms + a.norm_eps);
#pragma unroll
            for (int c = 0; c < 32; ++c) {   // the logit sits where this thread writes its output
                const float rs = __shfl_sync(0xffffffffu, rstd, c);
                const float z = __bfloat162float(os[(r0 + c) * D + jl]);
                v[c] *= rs * norm_wj * __fdividef(1.f, 1.f + __expf(-z));
            }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) os[(r0 + c) * D + jl] = __float2bfloat16_rn(v[c]);
    };
    // staging tile -> out, 16-byte coalesced stores of the rows inside the sequence
    auto store_output = [&]() {
        const uint4 *os = reinterpret_cast<const uint4 *>(sm + OFF_STG);
#pragma unroll
        for (int e = 0; e < 1024 / NT; ++e) {
            const int idx = tid + NT * e;          // 64 rows x 16 uint4 (the first dv / 8 of a row stored)
            const int r = idx >> 4, c16 = idx & 15;
            if (r < nr_out && c16 < (a.dv >> 3))
                reinterpret_cast<uint4 *>(out + ((t0_out + r) * H + h) * a.dv)[c16] = os[idx];
        }
    };
    // T_IJ = -(sum_{K=J+1..I} T_IK A_KJ) T_JJ for one 16x16 block below the diagonal (one warp)
    auto t_block = [&](int I, int J) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int K = J + 1; K <= I; ++K) {
            uint32_t a4[4], b4[4];
            ldsm_x4(sb + OFF_T + sw(16 * I + (lane & 15), 16 * K + ((lane >> 4) << 3), 64), a4[0], a4[1], a4[2], a4[3]);
            ldsm_x4_t(sb + OFF_TT + sw(16 * K + (lane & 7) + (((lane >> 3) & 1) << 3), 16 * J + ((lane >> 4) << 3), 64),
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
    bool ok = true;
    const int cp = tid & 63, sub = tid >> 6;   // elementwise ownership: channel pair, 8-row group
    const int blk = sub >> 1, hb = sub & 1;    // sub-tile and which half of it
    const int t4 = lane & 3, g = lane >> 2;    // mma.sync fragment coordinates
    // q and k L2-normalised first ("はじめての自然言語処理 -- Kimi K3", section 3.1, the read-out
    // paragraph: q and k enter after L2 normalisation, so q . k is a cosine): each row's factor
    // 1 / sqrt(|x|^2 + eps) comes from a pass of warps 0-7 in step (1) and multiplies the row
    // in fp32 before any operand is rounded from it
    constexpr bool qkn = kQk;

    // (1) of a chunk whose G tile has landed (nr rows inside the sequence), warps 0-7:
    // log2-decay sums over the two 8-row halves of sub-tile warp/2 (cumulative sums restart at
    // each sub-tile)
    // Warps 0-7: the sums of log2 decays over 16-row quarters of the chunk (rows >= nr count as 0).
    auto prephase = [&](int nr) {
        const int c = 2 * cp, q = tid >> 6;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float l0 = 0.f, l1 = 0.f;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = 16 * q + 8 * half + rr;
                const float2 g2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_G + sw(r, c, 64)));
                if (r < nr) { l0 = fmaf(g2.x, LOG2E, l0); l1 = fmaf(g2.y, LOG2E, l1); }
            }
            PART[(2 * q + half) * 128 + c] = l0;
            PART[(2 * q + half) * 128 + c + 1] = l1;
        }
    };
    // Warps 8-11: q_r . k_r for the 16 rows of sub-tile I = warp - 8, from the raw bf16 tiles
    // (exact products, fp32 sums): the diagonal of M, whose entries carry no decay.
    auto diag_qk = [&]() {
        const int I = warp - 8;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(sb + OFF_Q + swqk(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3)), a0, a1, a2, a3);
            ldsm_x4(sb + OFF_K + swqk(16 * I + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3)),
                    b0, b1, b2, b3);
            mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
            mma_16816(acc[1], a0, a1, a2, a3, b2, b3);
        }
        // element (row g + 8hh, col 8nt + 2t4 + e) is diagonal when nt == hh and 2t4 + e == g
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (2 * t4 + e == g) MRR[16 * I + g + 8 * hh] = acc[hh][2 * hh + e];
    };
    // With the L2 option, warps 0-7 after the decay sums (while the previous chunk's groups
    // land): |x_r|^2 for the 16 rows of sub-tile I = warp % 4 of Q (warps 0-3) or K (warps 4-7),
    // the diagonal of X_I X_I^T (exact products, fp32 sums), and from it the row factor
    // 1 / sqrt(|x_r|^2 + eps), 0 where that is 0.  The operands of step (2) take the factors on,
    // and the diagonal of M in step (3).
    auto row_norms = [&]() {
        const int I = warp & 3, which = warp >> 2;
        const uint32_t tile = which ? OFF_K : OFF_Q;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(sb + tile + swqk(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3)), a0, a1, a2, a3);
            ldsm_x4(sb + tile + swqk(16 * I + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3)),
                    b0, b1, b2, b3);
            mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
            mma_16816(acc[1], a0, a1, a2, a3, b2, b3);
        }
        float *nqk = reinterpret_cast<float *>(sm + OFF_NQK) + 64 * which;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (2 * t4 + e == g) {   // element (row g + 8hh, col 8hh + 2t4 + e) is diagonal
                    const float d = acc[hh][2 * hh + e] + a.qk_eps;
                    nqk[16 * I + g + 8 * hh] = d > 0.f ? rsqrtf(d) : 0.f;
                }
    };
    // per-channel decay vectors of that chunk (log2 units), by warps 12-15: thread = channel
    auto vectors = [&]() {
        const int c = tid & 127;
        float t[4];
#pragma unroll
        for (int J = 0; J < 4; ++J) t[J] = PART[(2 * J) * 128 + c] + PART[(2 * J + 1) * 128 + c];
        const float bI[4] = {0.f, t[0], t[0] + t[1], t[0] + t[1] + t[2]};
        const float gl = bI[3] + t[3];
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            EB[I * 128 + c] = ex2(bI[I]);
            EL[I * 128 + c] = ex2_sub(gl - bI[I]);   // multiplies K^ (up to e^80)
#pragma unroll
            for (int J = 0; J < I; ++J)   // likewise; bf16 keeps subnormals down to 2^-133
                W6[pair_index(I, J) * 128 + c] = __float2bfloat16_rn(ex2_sub(bI[I] - bI[J]));
        }
        DEC[c] = ex2(gl);
    };
    bool drained = false;   // a failed wait's in-flight copies and MMAs have been waited for
    for (bool have = true; have; have = next_piece(false)) {
        c_run = ok && kSeg && c_lo > 0 ? warm_start(a, bos, h, c_lo) : 0;
        out_pending = false;
        t0_out = 0;
        nr_out = 0;
        spar = 1;
        if (ok) {
            const int64_t t_run = bos + (int64_t)c_run * C;
            // ---- initial state -> TMEM (S^T: lane j, column i; scale exponent 0)
            {
                const int64_t sbase = ((int64_t)n * H + h) * a.dk * a.dv;
                float v[32];
#pragma unroll
                for (int c = 0; c < 32; ++c)   // S[i][j], zero outside a 64-wide head's channels
                    v[c] = (a.s0 && c_run == 0 && 32 * quarter + c < a.dk && jl < a.dv)
                               ? a.s0[sbase + (int64_t)(32 * quarter + c) * a.dv + jl] : 0.f;
                tmem_st32(trow + TM_S + 32 * quarter, v);
                uint32_t zero[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) zero[c] = 0u;
                tmem_st16u(trow + TM_MU + 16 * quarter, zero);   // (M U)^T = 0 before the first update
                tmem_wait_st();
            }
            if (tid < 256) ZSC[tid] = 0;
            if (tid == 0 && c_run < c_hi) {
                mbar_arrive_expect_tx(bar_tma, 3 * 16384);
                tma_tile(&tmq, sb + OFF_Q, bar_tma, h, t_run, 16384);
                tma_tile(&tmk, sb + OFF_K, bar_tma, h, t_run, 16384);
                tma_tile(&tmg, sb + OFF_G, bar_tma, h, t_run);
                mbar_arrive_expect_tx(bar_v, 16384);
                tma_tile(&tmv, sb + OFF_V, bar_v, h, t_run);
            }
            if (tid < C) BETA[tid] = tid < len - (int64_t)c_run * C ? __bfloat162float(beta[(t_run + tid) * H + h]) : 0.f;
            tc_fence_before();
            __syncthreads();
            tc_fence_after();

#pragma unroll 1
            for (int ci = c_run; ci < c_hi; ++ci) {
                const int64_t t0 = bos + (int64_t)ci * C;
                const int nr = (int)(len - (int64_t)ci * C < C ? len - (int64_t)ci * C : C);
                const bool more = ci + 1 < c_hi;
                const int cpar = (ci - c_run) & 1;   // this chunk's row of scales; the TMEM state's is spar

                if (ci > c_run && tid < C) BETA[tid] = BETA[tid + (OFF_BNEXT - OFF_BETA) / 4];   // loaded during the previous chunk
                bool got = mbar_wait(bar_tma, ph_tma, wait_limit);   // checked at the next barrier
                ph_tma ^= 1;
                // ---- (1) warps 0-7: decay sums, then the previous chunk's output staged; warps 8-11:
                // q_r . k_r; warps 8-15: once the previous state update has landed, S^T -> fp16 pairs
                // (the MMA operand of this chunk), 64 key channels per warp; then warps 12-15: the
                // decay vectors from the sums
                if (warp < 8) {
                    prephase(nr);
                    named_bar_arrive(2, 384);   // the sums are in place for warps 12-15
                    if constexpr (qkn) row_norms();
                    if (out_pending) {   // the previous chunk's output, once its groups landed
                        got = mbar_wait(bar_s, ph_s, wait_limit) && mbar_wait(bar_o, ph_o, wait_limit) && got;
                        if (gate_on) got = mbar_wait(bar_z, ph_z, wait_limit) && got;
                        tc_fence_after();
                        stage_output(spar);
                    }
                } else {
                    if (warp < 12) diag_qk();
                    if (out_pending) got = mbar_wait(bar_s, ph_s, wait_limit) && got;
                    tc_fence_after();
                    const int64_t cs = kCkpt && ci >= c_lo ? ckpt_slot(a, n, (int64_t)ci * C) : -1;   // the state after ci chunks
                    float *ck = cs >= 0 ? a.ckpt + (cs * H + h) * D * D + jl : nullptr;
                    {
                        const int i0 = 64 * ((warp - 8) >> 2);
                        float v[32], w[32];
                        tmem_ld32x2(trow + TM_S + i0, trow + TM_S + i0 + 32, v, w);
                        // the lane's largest |S| over both halves (warps w and w + 4 share the lanes)
                        const int sz = ZSC[spar * 128 + jl];   // S = (TMEM state) 2^sz
                        XCH[((warp - 8) >> 2) * 128 + jl] = fmaxf(absmax(v), absmax(w));
                        named_bar(3, 256);   // warps 8-15 (w and w + 4 share their lanes)
                        const int es = exp2_floor(fmaxf(XCH[jl], XCH[128 + jl]));
                        const int d = 14 - es < 126 ? 14 - es : 126;   // largest |S16| in [2^14, 2^15)
                        if (warp < 12) {
                            ASC[cpar * 128 + jl] = sz - d;              // S16 = S 2^-(sz - d)
                            ESC[jl] = es > -1000 ? es + sz : -1000;     // exponent of the lane's largest |S|
                        }
                        if (ck) {   // S[i][j] = S^T[j][i]: a warp writes 128 contiguous bytes per i
                            const float fs = pow2i(sz);
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                __stcs(ck + (int64_t)(i0 + c) * D, v[c] * fs);
                                __stcs(ck + (int64_t)(i0 + 32 + c) * D, w[c] * fs);
                            }
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
                    if (warp >= 12) {
                        named_bar(2, 384);
                        vectors();
                    }
                }
                if (out_pending) ph_s ^= 1;
                tc_fence_before();
                if (__syncthreads_or(!got)) { ok = false; break; }
                tc_fence_after();
                if (out_pending) {
                    ph_o ^= 1;
                    if (gate_on) ph_z ^= 1;
                    store_output();
                    out_pending = false;
                }

                // ---- (2) operands, each rounded from the exact inputs:
                //   bf16 (range e^+-80): Q~ = Q x as hi + lo, K~ = K x, K^ = K / x;
                //   fp16: Qbar = Q x e^{b_I} (over Q), Kbar (over K), Kp = K / x e^{gl - b_I} (transposed).
                // Rows past the end of the sequence hold finite data (the next sequence, or TMA zero
                // fill) and need no masking: their beta is 0, their decay is not accumulated, and the
                // entries of A and M they would feed lie above the diagonal or in rows never stored.
                // With the L2 option each q and k row is first multiplied by its factor in fp32.
                auto operands = [&](auto qkn_c) {
                    constexpr bool kQkn = decltype(qkn_c)::value;
                    const int c = 2 * cp;
                    const float2 eb = *reinterpret_cast<const float2 *>(EB + blk * 128 + c);
                    const float2 el = *reinterpret_cast<const float2 *>(EL + blk * 128 + c);
                    float2 l = hb ? *reinterpret_cast<const float2 *>(PART + (2 * blk) * 128 + c) : make_float2(0.f, 0.f);
                    const float2 minus1 = make_float2(-1.f, -1.f);
                    uint32_t p0[4], p1[4];
#pragma unroll
                    for (int rr = 0; rr < 8; rr += 2) {
                        float kp[2][2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int r = 16 * blk + 8 * hb + rr + e;
                            const uint32_t off = sw(r, c, 64), oqk = swqk(r, c);
                            float2 q2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_Q + oqk));
                            float2 k2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_K + oqk));
                            if constexpr (kQkn) {
                                const float *nqk = reinterpret_cast<const float *>(sm + OFF_NQK);
                                const float nq = nqk[r], nk = nqk[64 + r];
                                q2 = __fmul2_rn(q2, make_float2(nq, nq));
                                k2 = __fmul2_rn(k2, make_float2(nk, nk));
                            }
                            const float2 g2 = unpack_bf16(*reinterpret_cast<uint32_t *>(sm + OFF_G + off));
                            const float w2 = r < nr ? LOG2E : 0.f;   // decay past the sequence end is not summed
                            l = __ffma2_rn(g2, make_float2(w2, w2), l);
                            const float2 x = make_float2(ex2(l.x), ex2(l.y));
                            const float2 y = make_float2(ex2(-l.x), ex2(-l.y));
                            const float2 qt = __fmul2_rn(q2, x), kt = __fmul2_rn(k2, x), kh = __fmul2_rn(k2, y);
                            const uint32_t qh = pack_bf16(qt.x, qt.y);
                            const float2 ql = __ffma2_rn(unpack_bf16(qh), minus1, qt);
                            *reinterpret_cast<uint32_t *>(sm + OFF_SST + off) = qh;
                            *reinterpret_cast<uint32_t *>(sm + OFF_UST + off) = pack_bf16(ql.x, ql.y);
                            *reinterpret_cast<uint32_t *>(sm + OFF_SST + 16384 + off) = pack_bf16(kt.x, kt.y);
                            *reinterpret_cast<uint32_t *>(sm + OFF_KH + off) = pack_bf16(kh.x, kh.y);
                            const float2 qb = __fmul2_rn(qt, eb), kb = __fmul2_rn(kt, eb), kp2 = __fmul2_rn(kh, el);
                            *reinterpret_cast<uint32_t *>(sm + OFF_Q + oqk) = pack_f16(qb.x, qb.y);
                            *reinterpret_cast<uint32_t *>(sm + OFF_K + oqk) = pack_f16(kb.x, kb.y);
                            kp[e][0] = kp2.x;
                            kp[e][1] = kp2.y;
                        }
                        p0[rr / 2] = pack_f16(kp[0][0], kp[1][0]);
                        p1[rr / 2] = pack_f16(kp[0][1], kp[1][1]);
                    }
                    const int rc = 16 * blk + 8 * hb;
                    *reinterpret_cast<uint4 *>(sm + OFF_KPT + sw(c, rc, 128)) = make_uint4(p0[0], p0[1], p0[2], p0[3]);
                    *reinterpret_cast<uint4 *>(sm + OFF_KPT + sw(c + 1, rc, 128)) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
                };
                operands(std::integral_constant<bool, qkn>());

                fence_async_smem();
                tc_fence_before();
                __syncthreads();
                // [O_I^T | P^T] = S16^T [Qbar; Kbar]^T and V^T = V^T I into the U columns (V read
                // MN-major; free since the previous output was staged) [commit: P], issued by a warp
                // that (3) leaves idle; the same thread loads the next chunk's G (consumed) and, once
                // the group has read Qbar, Kbar and V, its Q, K and V
                bool gtma = true;
                if (warp == 15 && lane == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_f16_ts(tmem + TM_OI, tmem + TM_S16 + 8 * k, dsm + ((OFF_Q + (k >> 2) * 16384 + (k & 3) * 32) >> 4),
                                   IDESC_N128, k > 0);
                    gtma = mbar_wait(bar_v, ph_v, wait_limit);   // this chunk's V
                    if (gtma) {
                        tc_fence_after();
                        const uint64_t vdesc = sdesc_sw128_mn(sb + OFF_V, 64 * 128, 1024);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_f16_ss(tmem + TM_U, vdesc + ((2048 * k) >> 4), dsm + ((OFF_NI + 32 * k) >> 4), IDESC_VT, k > 0);
                    }
                    mma_commit(bar_p);
                    if (more) {
                        mbar_arrive_expect_tx(bar_tma, 3 * 16384);
                        tma_tile(&tmg, sb + OFF_G, bar_tma, h, t0 + C);
                        gtma = mbar_wait(bar_p, ph_p, wait_limit) && gtma;
                        if (gtma) {
                            tma_tile(&tmq, sb + OFF_Q, bar_tma, h, t0 + C, 16384);
                            tma_tile(&tmk, sb + OFF_K, bar_tma, h, t0 + C, 16384);
                            mbar_arrive_expect_tx(bar_v, 16384);
                            tma_tile(&tmv, sb + OFF_V, bar_v, h, t0 + C);
                        }
                    }
                }

                // ---- (3) A = beta K~ K^T and M = Q~ K^T on the 10 sub-tile pairs (I >= J), bf16
                // products with fp32 accumulation.  Warps 0-3: A_II, I = warp, both 8-column halves; the
                // warp then inverts (I + A_II) by forward substitution (one SM sub-partition per block).
                // Warps 4-7: M_II, I = warp - 4, as (Q~hi + Q~lo) K^^T below the diagonal (the largest
                // entries of M, where the bf16 rounding of Q~ shows in the outputs) and the exact
                // q_r . k_r on it.
                // Warps 8-13: the 6 off-diagonal pairs, single bf16 products with the per-channel factor
                // e^{b_I - b_J} (bf16, subnormals kept) applied to the right operand.  Off-diagonal A blocks go to the fp16
                // tile AT; T_II = (I + A_II)^-1 goes to the diagonal blocks of the fp16 tile T.
                if (warp < 4) {
                    const int I = warp;
                    float accA[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 4
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ao = sw(16 * I + (lane & 15), 16 * kk + ((lane >> 4) << 3), 64);
                        const uint32_t bo = sw(16 * I + (lane & 7) + ((lane >> 4) << 3), 16 * kk + (((lane >> 3) & 1) << 3), 64);
                        uint32_t ka[4], bh[4];
                        ldsm_x4(sb + OFF_SST + 16384 + ao, ka[0], ka[1], ka[2], ka[3]);
                        ldsm_x4(sb + OFF_KH + bo, bh[0], bh[1], bh[2], bh[3]);
                        mma_16816(accA[0], ka[0], ka[1], ka[2], ka[3], bh[0], bh[1]);
                        mma_16816(accA[1], ka[0], ka[1], ka[2], ka[3], bh[2], bh[3]);
                    }
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
                    __syncwarp();   // the whole of A_II is in place
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
                        __half *at = reinterpret_cast<__half *>(sm + OFF_T);
#pragma unroll
                        for (int r = 0; r < 16; ++r)
                            at[sw(16 * I + r, 16 * I + jj, 64) >> 1] = __float2half_rn(tcol[r]);
                    }
                } else if (warp < 8) {
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
                        ldsm_x4(sb + OFF_SST + ao, qh[0], qh[1], qh[2], qh[3]);
                        ldsm_x4(sb + OFF_UST + ao, ql[0], ql[1], ql[2], ql[3]);
                        ldsm_x4(sb + OFF_KH + bo, bh[0], bh[1], bh[2], bh[3]);
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
                            float mrr = MRR[r];
                            if constexpr (qkn) {   // q_r . k_r of the normalised rows
                                const float *nqk = reinterpret_cast<const float *>(sm + OFF_NQK);
                                mrr *= nqk[r] * nqk[64 + r];
                            }
                            const float m0 = s0 < r ? mv0 : (s0 == r ? mrr : 0.f);
                            const float m1 = s0 + 1 < r ? mv1 : (s0 + 1 == r ? mrr : 0.f);
                            const uint32_t mh = pack_f16(m0, m1);
                            const float2 mhf = unpack_f16(mh);
                            *reinterpret_cast<uint32_t *>(sm + OFF_MT + sw(r, s0, 64)) = mh;
                            *reinterpret_cast<uint32_t *>(sm + OFF_MLO + sw(r, s0, 64)) = pack_f16(m0 - mhf.x, m1 - mhf.y);
                        }
                } else if (warp == 14) {   // the blocks of T above the diagonal (staging used them), then
                                           // the next chunk's beta
                    for (int x = lane; x < 192; x += 32) {
                        const int b = x >> 5, rr = (x >> 1) & 15, hf = x & 1;   // (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
                        const int I = b < 3 ? 0 : (b < 5 ? 1 : 2);
                        const int J = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
                        *reinterpret_cast<uint4 *>(sm + OFF_T + sw(16 * I + rr, 16 * J + 8 * hf, 64)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    if (more) {   // the next chunk's beta (the load latency is hidden in this step)
                        const int64_t nn = len - (int64_t)(ci + 1) * C;
                        for (int r = lane; r < C; r += 32)
                            BETA[r + (OFF_BNEXT - OFF_BETA) / 4] = r < nn ? __bfloat162float(beta[(t0 + C + r) * H + h]) : 0.f;
                    }
                } else if (warp >= 8 && warp < 14) {
                    const int po = warp - 8;   // (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
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
                        ldsm_x4(sb + OFF_SST + 16384 + ao, ka[0], ka[1], ka[2], ka[3]);
                        ldsm_x4(sb + OFF_SST + ao, qh[0], qh[1], qh[2], qh[3]);
                        ldsm_x4(sb + OFF_KH + bo, bh[0], bh[1], bh[2], bh[3]);
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
                            *reinterpret_cast<uint32_t *>(sm + OFF_TT + sw(r, s0, 64)) =
                                pack_f16(br * accA[nt][2 * hh], br * accA[nt][2 * hh + 1]);
                            const float m0 = accM[nt][2 * hh], m1 = accM[nt][2 * hh + 1];
                            const uint32_t mh = pack_f16(m0, m1);
                            const float2 mhf = unpack_f16(mh);
                            *reinterpret_cast<uint32_t *>(sm + OFF_MT + sw(r, s0, 64)) = mh;
                            *reinterpret_cast<uint32_t *>(sm + OFF_MLO + sw(r, s0, 64)) = pack_f16(m0 - mhf.x, m1 - mhf.y);
                        }
                }
                __syncthreads();

                bool got4 = gtma;
                // ---- (4) warps 0-2: the off-diagonal blocks of T, level by level (T_IK with K > J is
                // ready before T_IJ);  warps 4-11: Z^T = (V^T - 2^a_j P^T) diag(beta) -> fp16 pairs
                // (TMEM) at the lane's scale z_j (warps w and w + 4 share the lanes)
                if (warp < 3) {
                    t_block(warp + 1, warp);                 // (1,0) (2,1) (3,2)
                    named_bar(1, 96);
                    if (warp < 2) t_block(warp + 2, warp);   // (2,0) (3,1)
                    named_bar(1, 96);
                    if (warp == 0) t_block(3, 0);
                } else if (warp >= 4 && warp < 12) {
                    got4 = mbar_wait(bar_p, ph_p, wait_limit) && got4;
                    tc_fence_after();
                    const int s0 = 32 * ((warp - 4) >> 2);
                    float pv[32], vv[32];
                    tmem_ld32x2(trow + TM_P + s0, trow + TM_U + s0, pv, vv);   // (Kbar S)^T 2^-a_j, V^T
                    const float fa = -pow2f(ASC[cpar * 128 + jl]);
                    const float2 fa2 = make_float2(fa, fa);
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(BETA + s0 + c);
                        const float2 t0 = __ffma2_rn(make_float2(pv[c], pv[c + 1]), fa2, make_float2(vv[c], vv[c + 1]));
                        const float2 t1 = __ffma2_rn(make_float2(pv[c + 2], pv[c + 3]), fa2, make_float2(vv[c + 2], vv[c + 3]));
                        const float2 z0 = __fmul2_rn(t0, make_float2(b4.x, b4.y)), z1 = __fmul2_rn(t1, make_float2(b4.z, b4.w));
                        pv[c] = z0.x; pv[c + 1] = z0.y; pv[c + 2] = z1.x; pv[c + 3] = z1.y;
                    }
                    XCH[((warp - 4) >> 2) * 128 + jl] = absmax(pv);
                    named_bar(4, 256);   // warps 4-11 (w and w + 4 share their lanes)
                    // z_j: the lane's largest |Z| maps into [1, 2); at least E_S - 86 so that the state,
                    // held as S 2^-z_j from here on, stays below 2^87; within 126 of the state's
                    // current exponent so that the state moves to it by one float factor
                    const int eZ = exp2_floor(fmaxf(XCH[jl], XCH[128 + jl]));
                    const int eS = ESC[jl], sz = ZSC[spar * 128 + jl];
                    const int zj = clamp_i(clamp_i(eZ > eS - 86 ? eZ : eS - 86, sz - 126, sz + 126), -126, 126);
                    if (warp < 8) ZSC[cpar * 128 + jl] = zj;
                    const float2 fz = make_float2(pow2i(-zj), pow2i(-zj));
                    uint32_t zv[16], zl[16];   // hi and lo: one fp16 rounding of U alone costs 2^-12
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
                }
                ph_p ^= 1;
                ph_v ^= 1;
                fence_async_smem();
                tc_fence_before();
                if (__syncthreads_or(!got4)) { ok = false; break; }
                // U^T = Z^T_hi T^T (U columns) + Z^T_lo T^T (the consumed P columns), issued by two
                // threads [commit: U, two arrivals]
                if (tid == 32) {
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ts(tmem + TM_P, tmem + TM_ZL + 8 * k, dsm + ((OFF_T + k * 32) >> 4), IDESC_N64, k > 0);
                    mma_commit(bar_u);
                }
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16_ts(tmem + TM_U, tmem + TM_Z + 8 * k, dsm + ((OFF_T + k * 32) >> 4), IDESC_N64, k > 0);
                    mma_commit(bar_u);
                }
                {   // while the U^T groups run: S^T <- S^T Diag(dec) in place (S^T was read as fp16 in
                    // (1)), moved from the lane's old scale to z_j (U^T is at z_j); warp w: lanes
                    // 32(w%4).., 32 columns from 32(w/4)
                    const int i0 = 32 * quarter;
                    float v[32];
                    tmem_ld32(trow + TM_S + i0, v);
                    const float f = pow2i(ZSC[spar * 128 + jl] - ZSC[cpar * 128 + jl]);   // |step| <= 126
                    const float2 f1 = make_float2(f, f);
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        const float4 d4 = *reinterpret_cast<const float4 *>(DEC + i0 + c);
                        const float2 a2 = __fmul2_rn(__fmul2_rn(make_float2(v[c], v[c + 1]), f1), make_float2(d4.x, d4.y));
                        const float2 b2 = __fmul2_rn(__fmul2_rn(make_float2(v[c + 2], v[c + 3]), f1), make_float2(d4.z, d4.w));
                        v[c] = a2.x; v[c + 1] = a2.y; v[c + 2] = b2.x; v[c + 3] = b2.y;
                    }
                    tmem_st32(trow + TM_S + i0, v);
                    tmem_wait_st();
                }
                {
                    const bool got = mbar_wait(bar_u, ph_u, wait_limit);
                    ph_u ^= 1;
                    if (__syncthreads_or(!got)) { ok = false; break; }
                }
                if (gate_on && tid == 0) {   // AT and T are consumed: this chunk's gate logits -> staging tile
                    fence_async_smem();
                    mbar_arrive_expect_tx(bar_z, 64 * D * 2);
                    tma_load_3d(sb + OFF_STG, &tmz, bar_z, 0, h, (int)t0);
                }
                tc_fence_after();
                // ---- (5) U^T -> fp16 hi + lo pairs (TMEM); warp w: lanes 32(w%4).., columns 16(w/4)..
                {
                    const int r0 = 16 * quarter;
                    float uv[16], u2[16];
                    tmem_ld16x2(trow + TM_U + r0, trow + TM_P + r0, uv, u2);
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        const float2 a2 = __fadd2_rn(make_float2(uv[e], uv[e + 1]), make_float2(u2[e], u2[e + 1]));
                        uv[e] = a2.x; uv[e + 1] = a2.y;
                    }
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        hi[e] = pack_f16(uv[2 * e], uv[2 * e + 1]);
                        const float2 lo2 = __ffma2_rn(unpack_f16(hi[e]), make_float2(-1.f, -1.f), make_float2(uv[2 * e], uv[2 * e + 1]));
                        lo[e] = pack_f16(lo2.x, lo2.y);
                    }
                    tmem_st8u(trow + TM_UH + r0 / 2, hi);
                    tmem_st8u(trow + TM_UL + r0 / 2, lo);
                    tmem_wait_st();
                }
                tc_fence_before();
                __syncthreads();
                // [S^T | (M U)^T] += U^T_hi [Kp^T; M]^T [commit: S];  low-order terms of (M U)^T,
                // U^T_lo M^T + U^T_hi Mlo^T, into the U^T columns (consumed) [commit: O], issued by a
                // warp with the least work in the next step (1); all at the lanes' scales z_j
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts(tmem + TM_S, tmem + TM_UH + 8 * ks, dsm + ((OFF_KPT + ks * 32) >> 4), IDESC_N192, 1);
                    mma_commit(bar_s);
                } else if (tid == 480) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts(tmem + TM_U, tmem + TM_UL + 8 * ks, dsm + ((OFF_MT + ks * 32) >> 4), IDESC_N64, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts(tmem + TM_U, tmem + TM_UH + 8 * ks, dsm + ((OFF_MLO + ks * 32) >> 4), IDESC_N64, 1);
                    mma_commit(bar_o);
                }
                out_pending = true;
                t0_out = t0;
                nr_out = ci >= c_lo ? nr : 0;   // the warm-up chunks before c_lo store nothing
                spar = cpar;
            }

            if (ok && out_pending) {   // the last chunk's state update and output
                const bool gs = mbar_wait(bar_s, ph_s, wait_limit);
                const bool go = mbar_wait(bar_o, ph_o, wait_limit);
                const bool gg = gate_on ? mbar_wait(bar_z, ph_z, wait_limit) : true;
                ph_s ^= 1;
                ph_o ^= 1;
                if (gate_on) ph_z ^= 1;
                if (__syncthreads_or(!(gs && go && gg))) {
                    ok = false;
                } else {
                    tc_fence_after();
                    stage_output(spar);
                    __syncthreads();
                    store_output();
                }
            }
        }
        if (!ok) {
            // A bounded wait expired: let copies and MMAs in flight land, flag the failure and mark
            // this unit's final state invalid.  At most one phase of each barrier can be in flight
            // (nothing is issued again on a barrier before its last phase was waited for), and it
            // is either the phase the parity names or the one before it: wait for both, with a
            // bound of its own (a few milliseconds) that does not depend on the expired one.
            if (tid == 0 && !drained) {
                constexpr uint32_t drain = 1u << 12;
                const uint32_t bars[7] = {bar_tma, bar_p, bar_v, bar_u, bar_s, bar_o, bar_z};
                const uint32_t phs[7] = {ph_tma, ph_p, ph_v, ph_u, ph_s, ph_o, ph_z};
#pragma unroll
                for (int b = 0; b < 7; ++b) {
                    mbar_wait(bars[b], phs[b], drain);
                    mbar_wait(bars[b], phs[b] ^ 1u, drain);
                }
                atomicAdd(&g_kda_tc_timeouts, 1u);
            }
            drained = true;
            if (kSeg && (P > 1 || balanced)) {   // only the last piece writes the state: mark this piece's outputs
                const int64_t r0 = (int64_t)c_lo * C, r1 = (int64_t)c_hi * C < len ? (int64_t)c_hi * C : len;
                for (int64_t x = tid; x < (r1 - r0) * a.dv; x += NT)
                    out[((bos + r0 + x / a.dv) * H + h) * a.dv + x % a.dv] = __ushort_as_bfloat16((unsigned short)0x7fc0);
            }
            __syncthreads();
        }
        tc_fence_after();
        if (a.sT && last_seg) {   // S = (TMEM state) 2^z_j
            const int64_t sbase = ((int64_t)n * H + h) * a.dk * a.dv;
            float v[32];
            tmem_ld32(trow + TM_S + 32 * quarter, v);
            const float fs = pow2i(ZSC[spar * 128 + jl]);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (32 * quarter + c < a.dk && jl < a.dv)
                    a.sT[sbase + (int64_t)(32 * quarter + c) * a.dv + jl] = ok ? v[c] * fs : __int_as_float(0x7fc00000);
        }
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
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

// [tokens][H][d] bf16 as a 3-D tensor (d, H, tokens); 64 x 1 x 64 boxes, 128-byte swizzle (the
// layout the MMA operand descriptors expect).  With d = 64 the kernel's second 64-channel box lies
// wholly past the tensor's first dimension and lands as zeros.
bool make_map(CUtensorMap *m, const void *ptr, int64_t tokens, int H, int d) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same tensor with 128 x 1 x 64 boxes and no swizzle: a box lands as a plain row-major
// [64 tokens][128 channels] tile (the output staging layout).
bool make_map_rows(CUtensorMap *m, const void *ptr, int64_t tokens, int H) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int segments_for(int64_t units, int64_t tokens, int64_t num_seqs, int sms) {
    constexpr int kMaxSegments = 8, kMinSegChunks = 16;
    if (units <= 0 || num_seqs <= 0 || sms <= 0) return 1;
    int64_t P = sms / units;
    if (P > kMaxSegments) P = kMaxSegments;
    const int64_t avg_chunks = tokens / (num_seqs * C);
    while (P > 1 && avg_chunks < (int64_t)kMinSegChunks * P) --P;
    return P < 1 ? 1 : (int)P;
}

// CTAs of the balanced schedule for a dense batch of `units` units of `nc` chunks on `sms` SMs:
// one per SM (at most kMaxSchedCtas), fewer when there are fewer chunks.
int balanced_ctas(int64_t units, int64_t nc, int sms) {
    const int64_t W = units * nc;
    const int64_t g = sms < kMaxSchedCtas ? sms : kMaxSchedCtas;
    return W <= 0 || g <= 0 ? 0 : (int)(W < g ? W : g);
}

// The CTAs' shares, drawn so that the largest cost is as small as bisection on it finds: a CTA
// costs its items, plus kWarmCost when it starts inside a unit (the warm-up of its first piece,
// which warm_start sets from the data -- one chunk at the decay bound, five with the standard
// decay distribution; the estimate only weighs the split), plus kPieceCost for each further
// piece (its set-up and pipeline refill).  Greedy: each CTA takes whole units while they fit its
// budget and ends inside the next one -- unless that would leave it fewer than kMinTail chunks of
// it, which would cost the next CTA a warm-up for little.
constexpr double kWarmCost = 4.0, kPieceCost = 0.5;
constexpr int64_t kMinTail = 8;
static int64_t fill(int64_t W, int64_t nc, int G, double T, SchedBounds *out) {
    int64_t x = 0;
    for (int b = 0; b < G; ++b) {
        if (out) out->x[b] = x;
        double cost = x % nc ? kWarmCost : 0.0;
        const int64_t start = x;
        while (x < W) {
            const int64_t r = nc - x % nc;
            const double extra = x != start ? kPieceCost : 0.0;
            if (cost + extra + (double)r <= T) {
                x += r;
                cost += extra + (double)r;
                continue;
            }
            const int64_t take = (int64_t)(T - cost - extra);
            if (take > 0 && (x == start || take >= kMinTail)) x += take;
            break;
        }
    }
    if (out) out->x[G] = W;
    return x;
}
static void draw_schedule(int64_t units, int64_t nc, int G, SchedBounds *sb) {
    const int64_t W = units * nc;
    double lo = (double)W / G, hi = lo + (double)nc + kWarmCost + kPieceCost + 1.0;   // hi covers W
    for (int it = 0; it < 30; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (fill(W, nc, G, mid, nullptr) >= W) hi = mid;
        else lo = mid;
    }
    fill(W, nc, G, hi, sb);   // the last CTA ends at W (fill covers W at hi)
}

// CTAs of the balanced schedule for packed sequences: one per SM, fewer when there are fewer
// items than that (W >= units; W <= heads * (ceil(tokens / 64) + sequences) bounds it).
int packed_ctas(int64_t units, int64_t tokens, int64_t num_seqs, int sms) {
    const int64_t w_max = units / (num_seqs > 0 ? num_seqs : 1) * ((tokens + C - 1) / C + num_seqs);
    const int64_t g = sms < kMaxSchedCtas ? sms : kMaxSchedCtas;
    return w_max <= 0 || g <= 0 ? 0 : (int)(w_max < g ? w_max : g);
}

// The library's choice when the caller leaves it open (a.segments == 0): the balanced schedule
// over one CTA per SM, with the output gate too -- shares drawn on the host for a dense batch,
// found on the device for packed sequences.  Packed sequences with at least twice as many units
// as SMs run one CTA per unit instead, longest first: the hardware hands each unit to the first
// SM that frees up, which evens out the spread in per-chunk speed between units that a static
// share cannot see (measured on 16 sequences x 32 heads: 23.95 ms against 24.35 ms balanced).
// One CTA per unit for every launch that writes
// checkpoints (each checkpoint then equals, bit for bit, the final state of a call on its
// prefix: a part of a sequence that warms up from a zero state reaches the same state only to
// within 2^-160 of its norm) or that reads and writes the state in place (a later piece of a
// unit would write the state while an earlier one may still read it).
static void library_schedule(ChunkArgs &a, int64_t units, int64_t tokens) {
    a.segments = 1;
    if (a.ckpt || (a.s0 && a.s0 == a.sT)) return;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return;
    if (a.cu == nullptr) a.sched_ctas = balanced_ctas(units, (a.seqlen + C - 1) / C, sms);
    else if (units < 2 * (int64_t)sms) a.sched_ctas = packed_ctas(units, tokens, a.num_seqs, sms);
}

cudaError_t take_wait_expiries(cudaStream_t st, unsigned int *count) {
    static const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(count, g_kda_tc_timeouts, sizeof(unsigned int), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_kda_tc_timeouts, &zero, sizeof(unsigned int), 0,
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

bool chunk_tc_supported(int dk, int dv, kda_dtype_t dt) {
    return dt == KDA_BF16 && (dk == 64 || dk == D) && (dv == 64 || dv == D);
}

bool chunk_tc_full(int dk, int dv, kda_dtype_t dt) { return dt == KDA_BF16 && dk == D && dv == D; }

cudaError_t launch_chunk_tc(const ChunkArgs &args, int dk, int dv, kda_dtype_t dt, cudaStream_t st) {
    if (!chunk_tc_supported(dk, dv, dt)) return cudaErrorNotSupported;
    ChunkArgs a = args;
    const int64_t tokens = a.cu ? a.seqlen : (int64_t)a.num_seqs * a.seqlen;
    const int64_t units = (int64_t)a.num_seqs * a.heads;
    a.sched_ctas = 0;
    if (a.segments <= 0) library_schedule(a, units, tokens);
    if (tokens >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mg, mz;
    a.dk = dk;
    a.dv = dv;
    if ((a.gate || a.ckpt) && !chunk_tc_full(dk, dv, dt)) return cudaErrorNotSupported;
    const bool qk = a.qk_eps >= 0.f;
    if (qk && (a.gate || a.ckpt)) return cudaErrorNotSupported;
    if (!make_map(&mq, a.q, tokens, a.heads, dk) || !make_map(&mk, a.k, tokens, a.heads, dk) ||
        !make_map(&mv, a.v, tokens, a.heads, dv) || !make_map(&mg, a.g, tokens, a.heads, dk) ||
        !make_map_rows(&mz, a.gate ? a.gate : a.v, tokens, a.heads))   // unused without a gate
        return cudaErrorInvalidValue;
    const int P = a.segments > 1 ? a.segments : 1;
    auto kernel = a.sched_ctas > 0 ? (a.gate ? kda_chunk_tc_kernel<3> : qk ? kda_chunk_tc_kernel<2, true> : kda_chunk_tc_kernel<2>)
                                   : P > 1 ? (qk ? kda_chunk_tc_kernel<1, true> : kda_chunk_tc_kernel<1>)
                                           : (qk ? kda_chunk_tc_kernel<0, true> : kda_chunk_tc_kernel<0>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t grid = a.sched_ctas > 0 ? a.sched_ctas : units * P;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    // the schedule is a kernel parameter (copied at the launch); the last one drawn on this host
    // thread is kept, so that repeated launches of one shape do not redraw it
    static thread_local SchedBounds sb{};
    static thread_local int64_t drawn[3] = {-1, -1, -1};
    if (a.sched_ctas > 0 && a.cu == nullptr) {
        const int64_t nc = (a.seqlen + C - 1) / C;
        if (drawn[0] != units || drawn[1] != nc || drawn[2] != a.sched_ctas) {
            draw_schedule(units, nc, a.sched_ctas, &sb);
            drawn[0] = units;
            drawn[1] = nc;
            drawn[2] = a.sched_ctas;
        }
    }
    kernel<<<(unsigned)grid, NT, SMEM_BYTES, st>>>(mq, mk, mv, mg, mz, a, a.wait_polls, sb);
    return cudaGetLastError();
}

}  // namespace kda
