"""Independent fp64 chunked (WY) formulation of the gated delta rule forward.

Used only as a pin for the per-token oracle: it reaches the same result by a
different algorithm, following the step names of the FlashQLA blog post
("FlashQLA: Qwen's Linear Attention Kernel Revolution for Edge AI",
section 2, Hardware-Friendly Algebraic Reformulation): compute the A matrix,
extract W and U, apply the V correction, then produce O.

Per chunk of C tokens with entry state S (gate cumsum restarted per chunk):

    gam_r   = sum_{j <= r} g_j,        D_ri = exp(gam_r - gam_i) for i <= r
    L       = strict_lower(diag(beta) (D o K K^T))
    A       = (I + L)^{-1}
    W       = A diag(beta exp(gam)) K,  U = A diag(beta) V
    U'      = U - W S                                   (V correction)
    O       = scale (diag(exp(gam)) Q S + (D o Q K^T) U')
    S_next  = exp(gam_last) S + K^T diag(exp(gam_last - gam)) U'

Nothing here is shared with the oracle or with the CUDA library.
"""
import numpy as np
import scipy.linalg


def chunked_fwd(q, k, v, g, beta, scale, h0=None, chunk=64):
    """Single sequence, single head: q,k [T,K], v [T,V], g,beta [T]."""
    T, K = k.shape
    V = v.shape[1]
    S = np.zeros((K, V)) if h0 is None else np.array(h0, dtype=np.float64)
    o = np.zeros((T, V))
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        n = e - s
        Q, Kc, Vc, gc, bc = q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e]
        gam = np.cumsum(gc)
        D = np.tril(np.exp(gam[:, None] - gam[None, :]))
        L = np.tril(bc[:, None] * D * (Kc @ Kc.T), -1)
        A = scipy.linalg.solve_triangular(np.eye(n) + L, np.eye(n), lower=True, unit_diagonal=True)
        W = A @ ((bc * np.exp(gam))[:, None] * Kc)
        U = A @ (bc[:, None] * Vc)
        Up = U - W @ S
        o[s:e] = scale * (np.exp(gam)[:, None] * (Q @ S) + (D * (Q @ Kc.T)) @ Up)
        S = np.exp(gam[-1]) * S + Kc.T @ (np.exp(gam[-1] - gam)[:, None] * Up)
    return o, S


def chunked_fwd_all(q, k, v, g, beta, scale, h0=None, chunk=64):
    """Batched wrapper: q,k [B,T,Hq,K], v [B,T,Hv,V] (no varlen)."""
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    G = Hv // Hq
    o = np.zeros((B, T, Hv, V))
    ht = np.zeros((B, Hv, K, V))
    for b in range(B):
        for h in range(Hv):
            oo, S = chunked_fwd(q[b, :, h // G], k[b, :, h // G], v[b, :, h], g[b, :, h],
                                beta[b, :, h], scale, None if h0 is None else h0[b, h], chunk)
            o[b, :, h] = oo
            ht[b, h] = S
    return o, ht
