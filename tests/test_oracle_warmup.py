"""Pins for oracle_fwd_warmup (the sequence-splitting forward with warmup)."""
import numpy as np

import oracle
from oracle_pins import rand_problem


def test_windows_reaching_the_start_are_exact():
    """With h0 = 0 and windows long enough to reach the sequence start, every
    segment's warmup state is the exact state: the result equals the unsplit run."""
    q, k, v, g, beta, _ = rand_problem(31, B=1, T=300, Hq=1, Hv=2, K=6, V=4, h0=False)
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.5, None)
    ow, hw = oracle.oracle_fwd_warmup(q, k, v, g, beta, 0.5, None, seg_len=1, warm=8, chunk=32,
                                      log_eps=1e9)
    assert np.allclose(ow, o, atol=1e-12) and np.allclose(hw, ht, atol=1e-12)


def test_error_bound_of_the_pages():
    """|o_hat_t - o_t| <= scale |q_t| exp(sum_{t0 < tau <= t} g_tau) |S_t0|_F, t0 the window start:
    the state error only shrinks, because |I - beta k k^T| <= 1 for beta |k|^2 in [0, 2]."""
    q, k, v, g, beta, h0 = rand_problem(32, B=1, T=256, Hq=1, Hv=1, K=6, V=4)
    g *= 0.05  # weak decay: the bound is not trivially tiny
    sc = 0.7
    o, _ = oracle.oracle_fwd(q, k, v, g, beta, sc, h0)
    seg, warm, C = 2, 1, 32
    ow, _ = oracle.oracle_fwd_warmup(q, k, v, g, beta, sc, h0, seg_len=seg, warm=warm, chunk=C, log_eps=1e9)
    worst = 0.0
    for p in range(1, 256 // (seg * C)):
        t0 = (p * seg - warm) * C            # window start token
        _, S0 = oracle.oracle_fwd(q[:, :t0], k[:, :t0], v[:, :t0], g[:, :t0], beta[:, :t0], sc, h0)
        nrm = np.linalg.norm(S0[0, 0])
        for t in range(p * seg * C, min(256, (p + 1) * seg * C)):
            bound = sc * np.linalg.norm(q[0, t, 0]) * np.exp(g[0, t0:t + 1, 0].sum()) * nrm
            err = np.abs(ow[0, t, 0] - o[0, t, 0]).max()
            assert err <= bound * (1 + 1e-9) + 1e-14, (p, t, err, bound)
            worst = max(worst, err / bound if bound > 0 else 0)
    assert worst > 1e-3  # the bound is not vacuous for these gates


def test_strong_decay_makes_warmup_exact():
    q, k, v, g, beta, h0 = rand_problem(33, B=1, T=192, Hq=1, Hv=1, K=5, V=3)
    g[0, 64 - 1, 0] = -1e4  # the state is wiped inside the window of segment 1
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.5, h0)
    ow, hw = oracle.oracle_fwd_warmup(q, k, v, g, beta, 0.5, h0, seg_len=2, warm=1, chunk=32, log_eps=1e9)
    assert np.allclose(ow, o, atol=1e-10) and np.allclose(hw, ht, atol=1e-10)


def test_non_decaying_head_runs_unsplit():
    q, k, v, g, beta, h0 = rand_problem(34, B=1, T=192, Hq=1, Hv=2, K=5, V=3)
    g[..., 1] = 0.0
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.5, h0)
    ow, hw = oracle.oracle_fwd_warmup(q, k, v, g, beta, 0.5, h0, seg_len=2, warm=1, chunk=32)
    assert np.allclose(ow[:, :, 1], o[:, :, 1], atol=1e-12) and np.allclose(hw[:, 1], ht[:, 1], atol=1e-12)


def test_segment_transition_identity():
    """The exact split rests on linearity in (v, S): a run from X equals M X + h, with h the run from a
    zero state and M the run with v = 0 from the identity (K = V)."""
    q, k, v, g, beta, h0 = rand_problem(35, B=1, T=90, Hq=1, Hv=1, K=6, V=6)
    _, hx = oracle.oracle_fwd(q, k, v, g, beta, 0.4, h0)
    _, h = oracle.oracle_fwd(q, k, v, g, beta, 0.4, None)
    _, M = oracle.oracle_fwd(q, k, np.zeros_like(v), g, beta, 0.4, np.eye(6)[None, None])
    assert np.allclose(hx[0, 0], M[0, 0] @ h0[0, 0] + h[0, 0], atol=1e-12)
    # and a two-segment scan reproduces the end state of one run
    _, h1 = oracle.oracle_fwd(q[:, :40], k[:, :40], v[:, :40], g[:, :40], beta[:, :40], 0.4, None)
    _, M1 = oracle.oracle_fwd(q[:, :40], k[:, :40], np.zeros_like(v[:, :40]), g[:, :40], beta[:, :40], 0.4,
                              np.eye(6)[None, None])
    _, h2 = oracle.oracle_fwd(q[:, 40:], k[:, 40:], v[:, 40:], g[:, 40:], beta[:, 40:], 0.4, None)
    _, M2 = oracle.oracle_fwd(q[:, 40:], k[:, 40:], np.zeros_like(v[:, 40:]), g[:, 40:], beta[:, 40:], 0.4,
                              np.eye(6)[None, None])
    s1 = M1[0, 0] @ h0[0, 0] + h1[0, 0]
    assert np.allclose(M2[0, 0] @ s1 + h2[0, 0], hx[0, 0], atol=1e-12)
