"""fp64 numpy statement of the chunkwise KDA algebra that the CUDA kernels use.

Test-side only: it checks the *mathematics* the GPU implements against the
token-by-token oracle, independently of any GPU code.

Chunk form ("はじめての自然言語処理 -- Kimi K3" section 3.1, the chunkwise
paragraphs and "chunk 内の減衰と、その数値範囲"): a chunk's outputs are an
inter-chunk term read from the state entering the chunk plus an intra-chunk
causal term (Tril, i <= j); decay between positions i < j is Gamma_j / Gamma_i,
folded into the operands by multiplying q by Gamma and dividing k by Gamma
(the report's equation (4)).  With the per-step bound g >= -5, a 16-token
sub-tile's cumulative log decay stays in [-80, 0], so each factor is at most
e^80 and the diagonal sub-tiles are plain dense products.

Per chunk of C tokens (positions r in [0, C)), gamma_r = sum_{s<=r} g_s:
  * sub-tile reference b_I = gamma just before sub-tile I starts (b_0 = 0);
    x_r = exp(gamma_r - b_I(r)) in [e^-80, 1], y_r = 1 / x_r;
  * A_rs = beta_r sum_c k_rc x_rc k_sc y_sc exp(b_I(r) - b_I(s))   (s <  r)
    M_rs =        sum_c q_rc x_rc k_sc y_sc exp(b_I(r) - b_I(s))   (s <= r)
  * T = (I + A)^-1 (the delta-rule correction inside the chunk, in WY form);
  * Kbar = K * Gamma, Qbar = Q * Gamma, Kp = K * exp(gamma_last - gamma);
  * U = T diag(beta) (V - Kbar S);  O = Qbar S + M U;
    S <- Diag(exp gamma_last) S + Kp^T U.
"""
import numpy as np


def chunk_forward_fp64(q, k, v, g, beta, S0, C=64, sub=16):
    """One (sequence, head): q, k, g [L, dk]; v [L, dv]; beta [L]; S0 [dk, dv]."""
    L, dk = q.shape
    dv = v.shape[1]
    S = S0.copy()
    out = np.zeros((L, dv))
    for c0 in range(0, L, C):
        n = min(C, L - c0)
        Q = np.zeros((C, dk)); K = np.zeros((C, dk)); V = np.zeros((C, dv))
        G = np.zeros((C, dk)); Bt = np.zeros(C)
        Q[:n], K[:n], V[:n], G[:n], Bt[:n] = (q[c0:c0 + n], k[c0:c0 + n], v[c0:c0 + n],
                                               g[c0:c0 + n], beta[c0:c0 + n])
        gam = np.cumsum(G, axis=0)
        blk = np.arange(C) // sub
        ref = np.zeros((C // sub, dk))
        ref[1:] = gam[sub - 1:C - 1:sub]
        x = np.exp(gam - ref[blk])
        y = 1.0 / x
        A = np.zeros((C, C)); M = np.zeros((C, C))
        for I in range(C // sub):
            rI = slice(I * sub, (I + 1) * sub)
            for J in range(I + 1):
                sJ = slice(J * sub, (J + 1) * sub)
                w = np.exp(ref[I] - ref[J])               # <= 1 (== 1 on the diagonal)
                R = K[sJ] * y[sJ] * w                     # right operand of tile (I, J)
                A[rI, sJ] = (K[rI] * x[rI]) @ R.T
                M[rI, sJ] = (Q[rI] * x[rI]) @ R.T
        A = np.tril(A, -1) * Bt[:, None]
        M = np.tril(M, 0)
        T = np.linalg.inv(np.eye(C) + A)
        Gam = np.exp(gam)
        Kbar, Qbar = K * Gam, Q * Gam
        Kp = K * np.exp(gam[-1] - gam)
        U = T @ (Bt[:, None] * (V - Kbar @ S))
        O = Qbar @ S + M @ U
        S = np.exp(gam[-1])[:, None] * S + Kp.T @ U
        out[c0:c0 + n] = O[:n]
    return out, S
