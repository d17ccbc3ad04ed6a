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


# --- chunk-parallel state passing -------------------------------------------
# The end state of a chunk is affine in its start state:
#   S_L = Diag(e^{Gam_L}) S0 + Khat^T (Util - W S0) = M S0 + B,
#   M = Diag(e^{Gam_L}) - Khat^T W  (K x K),   B = Khat^T Util  (K x V).
# Every chunk-start state is therefore a prefix composition of these maps,
# (M2, B2) o (M1, B1) = (M2 M1, M2 B1 + B2), which a scan finds in log2(n)
# levels instead of n sequential steps.


def chunk_maps(q, k, v, g, beta, chunk=64, dtype=np.float64):
    """The per-chunk maps (M_c, B_c) of a sequence, in `dtype`."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    maps = []
    for s in range(0, q.shape[0], chunk):
        e = min(s + chunk, q.shape[0])
        L = e - s
        gam = np.cumsum(g[s:e], axis=0)
        kk, vv, bb = k[s:e], v[s:e], beta[s:e]
        diff = gam[:, None, :] - gam[None, :, :]
        lower = np.tril(np.ones((L, L), dtype=bool))
        dec = np.where(lower[:, :, None], np.exp(np.minimum(diff, 0.0)), 0.0)
        A = bb[:, None] * np.einsum("tc,ic,tic->ti", kk, kk, dec) * np.tril(np.ones((L, L)), -1)
        Tinv = np.linalg.inv(np.eye(L) + A)
        W = Tinv @ (bb[:, None] * kk * np.exp(gam))
        Util = Tinv @ (bb[:, None] * vv)
        khat = kk * np.exp(gam[-1] - gam)
        maps.append(((np.diag(np.exp(gam[-1])) - khat.T @ W).astype(dtype),
                     (khat.T @ Util).astype(dtype)))
    return maps


def scan_chunk_states(maps, S0):
    """Chunk-start states and the final state from an inclusive
    Hillis-Steele scan of the maps (level d composes each prefix with the one
    d chunks before it), in the maps' precision."""
    Mp = [m for m, _ in maps]
    Bp = [b for _, b in maps]
    n, d = len(maps), 1
    while d < n:
        Mn, Bn = list(Mp), list(Bp)
        for c in range(d, n):
            Mn[c] = Mp[c] @ Mp[c - d]
            Bn[c] = Mp[c] @ Bp[c - d] + Bp[c]
        Mp, Bp, d = Mn, Bn, 2 * d
    S0 = np.asarray(S0, dtype=Mp[0].dtype)
    starts = [S0] + [Mp[c] @ S0 + Bp[c] for c in range(n - 1)]
    return starts, Mp[-1] @ S0 + Bp[-1]


def grouped_prefill(q, k, v, g, beta, S0, scale, group=4, chunk=64):
    """The chunk form with the chain over chunks cut into groups of `group`
    chunks, in three stages and without storing anything per chunk:
      1. every group, independently, runs the chunk recurrence from a zero
         state with the identity carried beside it ([S | P], P <- M_c P), and
         keeps only its end: (S_end, P_end), so that true end = S_end + P_end C;
      2. the true group-start states C_g follow in one short chain:
         C_{g+1} = S_end_g + P_end_g C_g, C_0 = S0;
      3. every group reruns the chunk form from its C_g.
    Returns what chunk_prefill returns (o, final state, chunk-start states)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T, K = q.shape
    bounds = [(s, min(s + chunk, T)) for s in range(0, T, chunk)]
    groups = [bounds[i:i + group] for i in range(0, len(bounds), group)]

    def run(grp, S, P=None):
        """The chunk form over the group's chunks from S (and P when given)."""
        o_parts, starts = [], []
        for s, e in grp:
            L = e - s
            gam = np.cumsum(g[s:e], axis=0)
            kk, qq, vv, bb = k[s:e], q[s:e], v[s:e], beta[s:e]
            diff = gam[:, None, :] - gam[None, :, :]
            lower = np.tril(np.ones((L, L), dtype=bool))
            dec = np.where(lower[:, :, None], np.exp(np.minimum(diff, 0.0)), 0.0)
            A = bb[:, None] * np.einsum("tc,ic,tic->ti", kk, kk, dec) * np.tril(np.ones((L, L)), -1)
            Pm = np.einsum("tc,ic,tic->ti", qq, kk, dec)
            Tinv = np.linalg.inv(np.eye(L) + A)
            W = Tinv @ (bb[:, None] * kk * np.exp(gam))
            U = Tinv @ (bb[:, None] * vv) - W @ S
            starts.append(S.copy())
            o_parts.append(scale * ((qq * np.exp(gam)) @ S + Pm @ U))
            khat = kk * np.exp(gam[-1] - gam)
            S = np.exp(gam[-1])[:, None] * S + khat.T @ U
            if P is not None:
                P = np.exp(gam[-1])[:, None] * P - khat.T @ (W @ P)
        return o_parts, starts, S, P

    ends = [run(grp, np.zeros((K, v.shape[1])), np.eye(K))[2:] for grp in groups]   # stage 1
    C = [np.array(S0, dtype=np.float64)]                                             # stage 2
    for S_end, P_end in ends[:-1]:
        C.append(S_end + P_end @ C[-1])
    o, starts, S = [], [], None                                                      # stage 3
    for grp, Cg in zip(groups, C):
        o_parts, st, S, _ = run(grp, Cg)
        o += o_parts
        starts += st
    return np.concatenate(o), S, starts
