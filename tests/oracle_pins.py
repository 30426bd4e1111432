"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each ``pin_*`` takes an oracle library handle (so the same checks can run on
deliberately broken builds of the oracle) and raises AssertionError when the
oracle disagrees with the fact it checks.  None of them re-types the oracle's
loop: they use closed forms of special cases, a library filter routine, an
independent chunked algorithm, invariances, central finite differences and
reverse-mode autodiff of an independent formulation.
"""
import numpy as np
import scipy.signal
import torch

import oracle
from chunked_form import chunked_fwd, chunked_fwd_all

TOL = 1e-10


def _rng(seed):
    return np.random.default_rng(seed)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(seed, B=1, T=40, Hq=1, Hv=1, K=8, V=6, h0=True, g_shift=0.0):
    r = _rng(seed)
    q = _unit_rows(r.standard_normal((B, T, Hq, K)))
    k = _unit_rows(r.standard_normal((B, T, Hq, K)))
    v = r.standard_normal((B, T, Hv, V))
    g = -np.log1p(np.exp(r.standard_normal((B, T, Hv)) + g_shift))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, Hv))))
    s0 = 0.1 * r.standard_normal((B, Hv, K, V)) if h0 else None
    return q, k, v, g, beta, s0


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a); b = np.asarray(b)
    err = np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b)))
    assert err <= tol, f"{what}: rel err {err:.3e} > {tol:.1e}"


# ----------------------------------------------------------------- forward pins
def pin_beta0_pure_decay(lib):
    """beta = 0 removes the write: S_t = exp(G_t) h0, o_t = scale exp(G_t) h0^T q_t."""
    q, k, v, g, beta, h0 = rand_problem(1, T=33, K=6, V=5)
    beta[:] = 0.0
    sc = 0.37
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, sc, h0, lib=lib)
    G = np.cumsum(g[0, :, 0])
    ref = sc * np.exp(G)[:, None] * (q[0, :, 0] @ h0[0, 0])
    _close(o[0, :, 0], ref, what="o")
    _close(ht[0, 0], np.exp(G[-1]) * h0[0, 0], what="ht")


def pin_g0_beta0_readout(lib):
    """g = 0, beta = 0: the state never changes, o_t = scale h0^T q_t."""
    q, k, v, g, beta, h0 = rand_problem(2, T=21, K=5, V=7)
    g[:] = 0.0
    beta[:] = 0.0
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.5, h0, lib=lib)
    _close(o[0, :, 0], 0.5 * q[0, :, 0] @ h0[0, 0], what="o")
    _close(ht, h0, what="ht")


def _orthonormal_keys(seed, T, K):
    r = _rng(seed)
    Qm, _ = np.linalg.qr(r.standard_normal((K, K)))
    return Qm[:T]  # T orthonormal rows (T <= K)


def pin_orthogonal_keys_gla(lib):
    """Orthonormal keys, h0 = 0: the erase term vanishes and the rule is gated
    linear attention, o_t = scale sum_{i<=t} exp(G_t - G_i) beta_i (q_t.k_i) v_i."""
    T, K, V = 10, 12, 4
    q, _, v, g, beta, _ = rand_problem(3, T=T, K=K, V=V, h0=False)
    k = _orthonormal_keys(3, T, K)[None, :, None, :]
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.8, None, lib=lib)
    G = np.cumsum(g[0, :, 0])
    qk = q[0, :, 0] @ k[0, :, 0].T
    M = np.tril(np.exp(G[:, None] - G[None, :])) * qk * beta[0, :, 0][None, :]
    _close(o[0, :, 0], 0.8 * M @ v[0, :, 0], what="o")


def pin_orthogonal_keys_linear_attention(lib):
    """Orthonormal keys, g = 0, beta = 1, h0 = 0: causal linear attention."""
    T, K, V = 9, 9, 3
    q, _, v, g, beta, _ = rand_problem(4, T=T, K=K, V=V, h0=False)
    g[:] = 0.0
    beta[:] = 1.0
    k = _orthonormal_keys(4, T, K)[None, :, None, :]
    o, _ = oracle.oracle_fwd(q, k, v, g, beta, 1.0, None, lib=lib)
    ref = np.tril(q[0, :, 0] @ k[0, :, 0].T) @ v[0, :, 0]
    _close(o[0, :, 0], ref, what="o")


def pin_single_token(lib):
    """T = 1 from a nonzero state, written with matrix algebra."""
    q, k, v, g, beta, h0 = rand_problem(5, T=1, K=7, V=3)
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.3, h0, lib=lib)
    a = np.exp(g[0, 0, 0]); b = beta[0, 0, 0]
    kk, vv, qq, S0 = k[0, 0, 0], v[0, 0, 0], q[0, 0, 0], h0[0, 0]
    S1 = a * (np.eye(7) - b * np.outer(kk, kk)) @ S0 + b * np.outer(kk, vv)
    _close(ht[0, 0], S1, what="ht")
    _close(o[0, 0, 0], 0.3 * S1.T @ qq, what="o")


def pin_strong_decay_memoryless(lib):
    """exp(g) = 0 forgets everything: S_t = beta_t k_t v_t^T."""
    q, k, v, g, beta, h0 = rand_problem(6, T=12, K=5, V=4)
    g[:] = -1e4
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 1.3, h0, lib=lib)
    qk = np.sum(q[0, :, 0] * k[0, :, 0], axis=-1)
    _close(o[0, :, 0], 1.3 * (beta[0, :, 0] * qk)[:, None] * v[0, :, 0], what="o")
    _close(ht[0, 0], beta[0, -1, 0] * np.outer(k[0, -1, 0], v[0, -1, 0]), what="ht")


def pin_unit_beta_retrieval(lib):
    """beta = 1 and |k| = 1: the new state maps k_t exactly onto v_t (any gates)."""
    q, k, v, g, beta, h0 = rand_problem(7, T=25, K=6, V=5)
    beta[:] = 1.0
    o, _ = oracle.oracle_fwd(k, k, v, g, beta, 1.0, h0, lib=lib)   # q := k, scale 1
    _close(o, v, what="S_t^T k_t")


def pin_ema_lfilter(lib):
    """One key direction (K = 1, k = 1), constant gate and beta: the rule is the
    exponential moving average S_t = (1 - beta) e^g S_{t-1} + beta v_t, i.e. a
    first-order IIR filter; compared with scipy.signal.lfilter."""
    r = _rng(8)
    T, V = 50, 3
    gv, bv = -0.3, 0.45
    q = r.standard_normal((1, T, 1, 1)); k = np.ones((1, T, 1, 1))
    v = r.standard_normal((1, T, 1, V))
    g = np.full((1, T, 1), gv); beta = np.full((1, T, 1), bv)
    h0 = r.standard_normal((1, 1, 1, V))
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.7, h0, lib=lib)
    c = (1 - bv) * np.exp(gv)
    S = np.empty((T, V))
    for j in range(V):
        zi = scipy.signal.lfiltic([bv], [1.0, -c], y=[h0[0, 0, 0, j]])
        S[:, j], _ = scipy.signal.lfilter([bv], [1.0, -c], v[0, :, 0, j], zi=zi)
    _close(o[0, :, 0], 0.7 * q[0, :, 0, 0][:, None] * S, what="o")
    _close(ht[0, 0, 0], S[-1], what="ht")


def pin_repeated_key_rows(lib):
    """All keys equal to e_0 (K > 1): row 0 of S is the EMA above, the other
    rows only decay, S_t[i] = exp(G_t) h0[i] for i > 0."""
    r = _rng(9)
    T, K, V = 30, 4, 2
    gv, bv = -0.2, 0.6
    k = np.zeros((1, T, 1, K)); k[..., 0] = 1.0
    q = r.standard_normal((1, T, 1, K))
    v = r.standard_normal((1, T, 1, V))
    g = np.full((1, T, 1), gv); beta = np.full((1, T, 1), bv)
    h0 = r.standard_normal((1, 1, K, V))
    _, ht = oracle.oracle_fwd(q, k, v, g, beta, 1.0, h0, lib=lib)
    c = (1 - bv) * np.exp(gv)
    row0 = [scipy.signal.lfilter([bv], [1.0, -c], v[0, :, 0, j],
                                 zi=scipy.signal.lfiltic([bv], [1.0, -c], y=[h0[0, 0, 0, j]]))[0][-1]
            for j in range(V)]
    _close(ht[0, 0, 0], row0, what="row 0")
    _close(ht[0, 0, 1:], np.exp(gv * T) * h0[0, 0, 1:], what="rows > 0")


def pin_chunked_form(lib, chunks=(16, 50, 64)):
    """The independent chunked (WY) algorithm gives the same o and final state,
    for several chunk sizes and a ragged last chunk."""
    q, k, v, g, beta, h0 = rand_problem(10, B=2, T=133, Hq=1, Hv=2, K=8, V=5)
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.35, h0, lib=lib)
    for c in chunks:
        oc, hc = chunked_fwd_all(q, k, v, g, beta, 0.35, h0, chunk=c)
        _close(o, oc, 1e-9, what=f"o chunk={c}")
        _close(ht, hc, 1e-9, what=f"ht chunk={c}")


def pin_split_run(lib):
    """Running T tokens equals running T1 then T - T1 from the final state."""
    q, k, v, g, beta, h0 = rand_problem(11, B=1, T=77, Hq=2, Hv=4, K=6, V=3)
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.5, h0, lib=lib)
    t1 = 30
    o1, h1 = oracle.oracle_fwd(q[:, :t1], k[:, :t1], v[:, :t1], g[:, :t1], beta[:, :t1], 0.5, h0, lib=lib)
    o2, h2 = oracle.oracle_fwd(q[:, t1:], k[:, t1:], v[:, t1:], g[:, t1:], beta[:, t1:], 0.5, h1, lib=lib)
    _close(np.concatenate([o1, o2], 1), o, what="o")
    _close(h2, ht, what="ht")


def pin_varlen_separate(lib):
    """Packed sequences (cu_seqlens, B = 1) equal separate runs."""
    lens = [5, 70, 1, 33]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_problem(12, B=1, T=T, Hq=1, Hv=2, K=5, V=4)
    h0 = 0.1 * _rng(12).standard_normal((len(lens), 2, 5, 4))
    cu = np.concatenate([[0], np.cumsum(lens)])
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.4, h0, cu_seqlens=cu, lib=lib)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        os_, hs = oracle.oracle_fwd(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], 0.4,
                                    h0[s:s + 1], lib=lib)
        _close(o[:, a:b], os_, what=f"o seq {s}")
        _close(ht[s], hs[0], what=f"ht seq {s}")


def pin_gva_repeat(lib):
    """Grouped value heads equal explicit repetition of each q/k head over its
    group of Hv / Hq consecutive value heads."""
    q, k, v, g, beta, h0 = rand_problem(13, B=2, T=20, Hq=2, Hv=6, K=4, V=3)
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, 0.6, h0, lib=lib)
    qr = np.repeat(q, 3, axis=2); kr = np.repeat(k, 3, axis=2)
    o2, h2 = oracle.oracle_fwd(qr, kr, v, g, beta, 0.6, h0, lib=lib)
    _close(o, o2, what="o"); _close(ht, h2, what="ht")
    # and each value head equals a single-head run with its own q/k head
    for h in range(6):
        o3, _ = oracle.oracle_fwd(q[:, :, h // 3:h // 3 + 1], k[:, :, h // 3:h // 3 + 1],
                                  v[:, :, h:h + 1], g[:, :, h:h + 1], beta[:, :, h:h + 1], 0.6,
                                  h0[:, h:h + 1], lib=lib)
        _close(o[:, :, h:h + 1], o3, what=f"head {h}")


# ---------------------------------------------------------------- backward pins
def _loss_fwd(lib, q, k, v, g, beta, sc, h0, do, dht, cu=None):
    o, ht = oracle.oracle_fwd(q, k, v, g, beta, sc, h0, cu_seqlens=cu, lib=lib)
    return float(np.sum(o * do) + np.sum(ht * dht))


def pin_bwd_finite_differences(lib, eps=1e-6, tol=1e-7):
    """Every gradient equals the central finite difference of
    <do, o> + <dht, ht> (fp64, tiny sizes, GVA group of 2)."""
    q, k, v, g, beta, h0 = rand_problem(14, B=1, T=7, Hq=1, Hv=2, K=3, V=2)
    r = _rng(15)
    do = r.standard_normal((1, 7, 2, 2)); dht = r.standard_normal((1, 2, 3, 2))
    sc = 0.45
    dq, dk, dv, db, dg, dh0 = oracle.oracle_bwd(q, k, v, g, beta, do, sc, h0, dht, lib=lib)
    grads = [dq, dk, dv, dg, db, dh0]          # reordered to match ``inputs``
    inputs = [q, k, v, g, beta, h0]
    for idx, (x, gx) in enumerate(zip(inputs, grads)):
        fd = np.zeros_like(x)
        for j in np.ndindex(x.shape):
            old = x[j]
            x[j] = old + eps; lp = _loss_fwd(lib, *inputs[:5], sc, inputs[5], do, dht)
            x[j] = old - eps; lm = _loss_fwd(lib, *inputs[:5], sc, inputs[5], do, dht)
            x[j] = old
            fd[j] = (lp - lm) / (2 * eps)
        err = np.max(np.abs(fd - gx))
        assert err <= tol, f"grad {['q', 'k', 'v', 'g', 'beta', 'h0'][idx]}: |fd - oracle| {err:.2e}"


def _torch_token_loss(q, k, v, g, beta, h0, sc, do, dht, cu):
    """Independent differentiable formulation (matrix form of one step:
    S_t = e^{g_t} (I - beta_t k k^T) S_{t-1} + beta_t k v^T), fp64 autograd."""
    B, T, Hq, K = q.shape
    Hv = v.shape[2]
    G = Hv // Hq
    loss = q.new_zeros(())
    seqs = [(0, int(cu[i]), int(cu[i + 1]), i) for i in range(len(cu) - 1)] if cu is not None \
        else [(b, 0, T, b) for b in range(B)]
    for (b, t0, t1, n) in seqs:
        for h in range(Hv):
            S = h0[n, h]
            for t in range(t0, t1):
                kt = k[b, t, h // G]
                P = torch.eye(K, dtype=q.dtype) - beta[b, t, h] * torch.outer(kt, kt)
                S = torch.exp(g[b, t, h]) * (P @ S) + beta[b, t, h] * torch.outer(kt, v[b, t, h])
                loss = loss + sc * (S.T @ q[b, t, h // G]) @ do[b, t, h]
            loss = loss + (S * dht[n, h]).sum()
    return loss


def pin_bwd_autograd(lib, tol=1e-10):
    """Gradients equal fp64 reverse-mode autodiff of an independent matrix-form
    recurrence; spans more than one 64-token checkpoint block, GVA and varlen."""
    lens = [70, 3, 66]
    T = sum(lens)
    q, k, v, g, beta, _ = rand_problem(16, B=1, T=T, Hq=2, Hv=4, K=4, V=3)
    r = _rng(17)
    h0 = 0.1 * r.standard_normal((3, 4, 4, 3))
    do = r.standard_normal((1, T, 4, 3)); dht = r.standard_normal((3, 4, 4, 3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    sc = 0.5
    dq, dk, dv, db, dg, dh0 = oracle.oracle_bwd(q, k, v, g, beta, do, sc, h0, dht, cu_seqlens=cu,
                                                lib=lib)
    grads = [dq, dk, dv, dg, db, dh0]          # reordered to match the inputs below
    ts = [torch.tensor(x, requires_grad=True) for x in (q, k, v, g, beta, h0)]
    loss = _torch_token_loss(*ts[:5], ts[5], sc, torch.tensor(do), torch.tensor(dht), cu)
    loss.backward()
    for name, t, gx in zip(["q", "k", "v", "g", "beta", "h0"], ts, grads):
        _close(gx, t.grad.numpy(), tol, what=f"d{name}")


FWD_PINS = [pin_beta0_pure_decay, pin_g0_beta0_readout, pin_orthogonal_keys_gla,
            pin_orthogonal_keys_linear_attention, pin_single_token, pin_strong_decay_memoryless,
            pin_unit_beta_retrieval, pin_ema_lfilter, pin_repeated_key_rows, pin_chunked_form,
            pin_split_run, pin_varlen_separate, pin_gva_repeat]
BWD_PINS = [pin_bwd_finite_differences, pin_bwd_autograd]
ALL_PINS = FWD_PINS + BWD_PINS
