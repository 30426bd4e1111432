"""Pins for oracle_chunk_aux (the returned gate cumsum and A matrix)."""
import numpy as np

import oracle
from oracle_pins import rand_problem


def test_gcum_is_chunk_local_cumsum():
    # chunk boundaries restart the sum; a constant gate gives (r + 1) * g
    g = np.full((1, 150, 1), -0.25)
    k = np.ones((1, 150, 1, 2)) / np.sqrt(2)
    gc, _ = oracle.oracle_chunk_aux(k, g, np.full((1, 150, 1), 0.5))
    r = np.arange(150) % 64
    assert np.allclose(gc[0, :, 0], -0.25 * (r + 1), atol=1e-14)


def test_A_reproduces_token_recurrence():
    """From a zero state one chunk gives final state K^T diag(E) A diag(beta) V
    (E_i = exp(g_cum_last - g_cum_i)); with V = identity columns and
    orthonormal keys this determines A diag(beta) exactly, so the oracle's A is
    checked against the per-token recurrence, not against its own formula."""
    n, K = 12, 16
    q, _, _, g, beta, _ = rand_problem(21, T=n, K=K, V=n, h0=False)
    Qm, _ = np.linalg.qr(np.random.default_rng(21).standard_normal((K, K)))
    # nearly-orthonormal keys still have nonzero overlaps: mix in a shared component
    k = Qm[:n] + 0.3 * Qm[n:n + 1]
    k = (k / np.linalg.norm(k, axis=1, keepdims=True))[None, :, None, :]
    v = np.eye(n)[None, :, None, :]
    _, ht = oracle.oracle_fwd(q, k, v, g, beta, 1.0, None)
    gc, A = oracle.oracle_chunk_aux(k, g, beta)
    E = np.exp(gc[0, -1, 0] - gc[0, :, 0])
    kk = k[0, :, 0]
    # ht = kk^T diag(E) A diag(beta) I  ->  A diag(beta) = pinv(kk^T diag(E)) ht
    Ab = np.linalg.lstsq(kk.T * E[None, :], ht[0, 0], rcond=None)[0]
    assert np.allclose(Ab, A[0, :, 0, :n] * beta[0, :, 0][None, :], atol=1e-10)


def test_A_unit_lower_triangular_and_ragged():
    q, k, v, g, beta, _ = rand_problem(22, B=1, T=70, K=8, V=4, h0=False)
    _, A = oracle.oracle_chunk_aux(k, g, beta)
    blk = A[0, 64:70, 0, :6]
    assert np.allclose(np.diag(blk), 1.0) and np.allclose(np.triu(blk, 1), 0.0)
    assert np.allclose(A[0, 64:70, 0, 6:], 0.0)
