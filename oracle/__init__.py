"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it shares no code with the CUDA path.

``oracle_fwd`` / ``oracle_bwd`` run the plain per-token recurrence of
``gdn_oracle.c`` (fp64, OpenMP over independent units).  Inputs are converted
to fp64 exactly (bf16 and fp32 values are representable in fp64).

Parity status: the forward and backward are pinned by closed forms,
invariants, an independent chunked formulation, finite differences and
reverse-mode autodiff (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(extra_flags=(), out_path=None, force=False) -> str:
    """Compile gdn_oracle.c with gcc (-O2 -fopenmp); returns the .so path."""
    out = out_path or _LIB_PATH
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC) and not extra_flags):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", *extra_flags, _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path=None):
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _declare(ctypes.CDLL(path))
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _declare(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.gdn_oracle_fwd.argtypes = [I64] * 7 + [P] * 6 + [ctypes.c_double, P, P, P, ctypes.c_int]
    lib.gdn_oracle_fwd.restype = ctypes.c_int
    lib.gdn_oracle_bwd.argtypes = ([I64] * 7 + [P] * 6 + [ctypes.c_double, P, P, P]
                                   + [P] * 6 + [ctypes.c_int])
    lib.gdn_oracle_bwd.restype = ctypes.c_int
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    return lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact upcast on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(q, v, cu):
    B, T, Hq, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    if cu is not None:
        cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
        n = len(cu) - 1
    else:
        n = B
    return B, T, Hq, Hv, K, V, n, cu


def max_threads(lib=None) -> int:
    return int((lib or load()).gdn_oracle_max_threads())


def oracle_fwd(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
               output_final_state=True, n_threads=0, lib=None):
    """Returns (o [B,T,Hv,V], final_state [N,Hv,K,V] or None) in fp64."""
    lib = lib or load()
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, initial_state))
    B, T, Hq, Hv, K, V, n, cu = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = K ** -0.5
    o = np.zeros((B, T, Hv, V))
    ht = np.zeros((n, Hv, K, V)) if output_final_state else None
    rc = lib.gdn_oracle_fwd(B, T, Hq, Hv, K, V, n, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), float(scale), _ptr(h0), _ptr(o), _ptr(ht), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_fwd: bad arguments (code {rc})")
    return o, ht


def oracle_bwd(q, k, v, g, beta, do, scale=None, initial_state=None, dht=None,
               cu_seqlens=None, n_threads=0, lib=None):
    """Returns (dq, dk, dv, dbeta, dg, dh0 or None) in fp64; dg is w.r.t. the raw g."""
    lib = lib or load()
    q, k, v, g, beta, h0, do, dht = map(_f64, (q, k, v, g, beta, initial_state, do, dht))
    B, T, Hq, Hv, K, V, n, cu = _dims(q, v, cu_seqlens)
    if scale is None:
        scale = K ** -0.5
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    db = np.zeros_like(beta); dg = np.zeros_like(g)
    dh0 = np.zeros((n, Hv, K, V)) if h0 is not None else None
    rc = lib.gdn_oracle_bwd(B, T, Hq, Hv, K, V, n, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                            _ptr(beta), float(scale), _ptr(h0), _ptr(do), _ptr(dht), _ptr(dq),
                            _ptr(dk), _ptr(dv), _ptr(db), _ptr(dg), _ptr(dh0), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_bwd: bad arguments (code {rc})")
    return dq, dk, dv, db, dg, dh0


def oracle_chunk_aux(k, g, beta, cu_seqlens=None, chunk=64):
    """The forward's auxiliary outputs, from their definitions (fp64, numpy).

    For every chunk of ``chunk`` tokens of every sequence (chunks restart at
    each sequence start, the last one may be shorter) and every value head:

      g_cum_r = sum_{j <= r, j in chunk} g_j                (chunk-local cumsum)
      L_ri    = beta_r exp(g_cum_r - g_cum_i) (k_r . k_i)    for i < r, else 0
      A       = (I + L)^{-1}  (unit lower triangular), row r stored at token r,
                columns beyond the chunk length are 0.

    k: [B,T,Hq,K]; g, beta: [B,T,Hv].  Returns (g_cum [B,T,Hv], A [B,T,Hv,chunk]).
    Pinned in tests/test_oracle_aux.py against the per-token oracle.
    """
    import scipy.linalg
    k, g, beta = _f64(k), _f64(g), _f64(beta)
    B, T, Hq, K = k.shape
    Hv = g.shape[2]
    G = Hv // Hq
    if cu_seqlens is not None:
        cu = [int(x) for x in np.asarray(cu_seqlens)]
        spans = [(0, cu[i], cu[i + 1]) for i in range(len(cu) - 1)]
    else:
        spans = [(b, 0, T) for b in range(B)]
    g_cum = np.zeros_like(g)
    A = np.zeros((B, T, Hv, chunk))
    for (b, t0, t1) in spans:
        for s in range(t0, t1, chunk):
            e = min(t1, s + chunk)
            n = e - s
            for h in range(Hv):
                gam = np.cumsum(g[b, s:e, h])
                g_cum[b, s:e, h] = gam
                kc = k[b, s:e, h // G]
                L = np.tril(beta[b, s:e, h][:, None] * np.exp(gam[:, None] - gam[None, :]) * (kc @ kc.T), -1)
                A[b, s:e, h, :n] = scipy.linalg.solve_triangular(np.eye(n) + L, np.eye(n), lower=True,
                                                                unit_diagonal=True)
    return g_cum, A


def oracle_fwd_warmup(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None, seg_len=8,
                      warm=6, log_eps=float(np.log(1e-4)), chunk=64, lib=None):
    """The sequence-splitting forward with warmup, built only from oracle_fwd.

    FlashQLA news page ("Technical Principles": sliding window warmup) and blog
    post (section 1): each sequence of N chunks is cut into segments of
    ``seg_len`` chunks; segment p > 0 starts from the state obtained by running
    the ``warm`` chunks before it from a zero state (no cross-segment
    correction); segment 0 starts from the initial state.  A value head whose
    warmup windows do not all decay (sum of g over a window > log_eps) runs
    unsplit, i.e. exactly.  Returns (o, final_state) in fp64.
    """
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, initial_state))
    B, T, Hq, Kd = q.shape
    Hv, Vd = v.shape[2], v.shape[3]
    G = Hv // Hq
    if scale is None:
        scale = Kd ** -0.5
    spans = ([(0, int(a), int(b)) for a, b in zip(cu_seqlens[:-1], cu_seqlens[1:])]
             if cu_seqlens is not None else [(b, 0, T) for b in range(B)])
    o = np.zeros((B, T, Hv, Vd))
    ht = np.zeros((len(spans), Hv, Kd, Vd))
    for si, (b, t0, t1) in enumerate(spans):
        n_ck = (t1 - t0 + chunk - 1) // chunk
        n_seg = (n_ck + seg_len - 1) // seg_len
        for h in range(Hv):
            sl = lambda x, a0, a1, hh: x[b:b + 1, a0:a1, hh:hh + 1]
            hq = h // G
            s0 = None if h0 is None else h0[si:si + 1, h:h + 1]
            windows = [(max(0, p * seg_len - warm) * chunk + t0, min(t1, p * seg_len * chunk + t0))
                       for p in range(1, n_seg)]
            serial = any(g[b, a0:a1, h].sum() > log_eps for a0, a1 in windows)
            if serial or n_seg <= 1:
                oo, hh_ = oracle_fwd(sl(q, t0, t1, hq), sl(k, t0, t1, hq), sl(v, t0, t1, h), sl(g, t0, t1, h),
                                     sl(beta, t0, t1, h), scale, s0, lib=lib)
                o[b, t0:t1, h] = oo[0, :, 0]
                ht[si, h] = hh_[0, 0]
                continue
            for p in range(n_seg):
                a0, a1 = t0 + p * seg_len * chunk, min(t1, t0 + (p + 1) * seg_len * chunk)
                if p == 0:
                    start = s0
                else:
                    w0, w1 = windows[p - 1]
                    _, start = oracle_fwd(sl(q, w0, w1, hq), sl(k, w0, w1, hq), sl(v, w0, w1, h),
                                          sl(g, w0, w1, h), sl(beta, w0, w1, h), scale, None, lib=lib)
                oo, hh_ = oracle_fwd(sl(q, a0, a1, hq), sl(k, a0, a1, hq), sl(v, a0, a1, h), sl(g, a0, a1, h),
                                     sl(beta, a0, a1, h), scale, start, lib=lib)
                o[b, a0:a1, h] = oo[0, :, 0]
                if p == n_seg - 1:
                    ht[si, h] = hh_[0, 0]
    return o, ht
