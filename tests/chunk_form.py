"""FP64 numpy statement of the 64-token chunk form of the gated delta rule.

A second, independent algorithm for the same result as the token-by-token
oracle: the CUDA prefill computes this chunk form, so the oracle test that the
two agree (to rounding) checks the algebra the kernels rely on, and a slip in
either (a sign, a transposed operand, an off-by-one in the cumulative decay)
shows up as a mismatch.

Derivation (per chunk of L tokens starting from state S0, K x V):
  Gam_t = sum_{s<=t} g_s (per key channel), X_t = Diag(exp g_t) S_{t-1},
  S_t = X_t + k_t u_t^T with u_t = beta_t (v_t - X_t^T k_t).
  Unrolling, S_r = Diag(e^{Gam_r}) S0 + sum_{i<=r} Diag(e^{Gam_r - Gam_i}) k_i u_i^T, so
  (I + A) U = Diag(beta) (V - Ktil S0) with
     A[t,i]  = beta_t sum_c k_t[c] k_i[c] e^{Gam_t[c]-Gam_i[c]}   (i < t)
     Ktil_t  = k_t * e^{Gam_t}
  hence U = Util - W S0 with W = (I+A)^-1 Diag(beta) Ktil, Util = (I+A)^-1 Diag(beta) V,
     O    = scale (Qtil S0 + P U),  Qtil_t = q_t * e^{Gam_t},
            P[t,i] = sum_c q_t[c] k_i[c] e^{Gam_t[c]-Gam_i[c]}   (i <= t)
     S_L  = Diag(e^{Gam_L}) S0 + Khat^T U,  Khat_i = k_i * e^{Gam_L - Gam_i}.
"""
import numpy as np


def chunk_prefill(q, k, v, g, beta, S0, scale, chunk=64):
    """q,k [T,K] (already normalised), v [T,V], g [T,K] log-decay, beta [T],
    S0 [K,V].  Returns (o [T,V], S_T [K,V], chunk-start states)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T = q.shape[0]
    S = np.array(S0, dtype=np.float64)
    o = np.zeros((T, v.shape[1]))
    starts = []
    for s in range(0, T, chunk):
        starts.append(S.copy())
        e = min(s + chunk, T)
        L = e - s
        gam = np.cumsum(g[s:e], axis=0)
        kk, qq, vv, bb = k[s:e], q[s:e], v[s:e], beta[s:e]
        diff = gam[:, None, :] - gam[None, :, :]
        lower = np.tril(np.ones((L, L), dtype=bool))
        dec = np.where(lower[:, :, None], np.exp(np.minimum(diff, 0.0)), 0.0)
        A = bb[:, None] * np.einsum("tc,ic,tic->ti", kk, kk, dec) * np.tril(np.ones((L, L)), -1)
        P = np.einsum("tc,ic,tic->ti", qq, kk, dec)
        Tinv = np.linalg.inv(np.eye(L) + A)
        W = Tinv @ (bb[:, None] * kk * np.exp(gam))
        Util = Tinv @ (bb[:, None] * vv)
        U = Util - W @ S
        o[s:e] = scale * ((qq * np.exp(gam)) @ S + P @ U)
        khat = kk * np.exp(gam[-1] - gam)
        S = np.exp(gam[-1])[:, None] * S + khat.T @ U
    return o, S, starts
