"""Shared driver for the GPU parity tests: run the CUDA path through the C ABI
(Python binding) and the fp64 oracle on the same seeded inputs, then compare
with the tolerances of ``parity.py``."""
import numpy as np
import torch

import gated_delta_rule_50_gb300 as gdn
import oracle
from parity import check


def recovered_gate(g_cum, cu_seqlens=None, chunk=64):
    """The raw gate implied by an fp32 chunk-local cumsum, exactly in fp64:
    g_t = g_cum_t - g_cum_{t-1} inside a chunk, g_cum_t at a chunk start."""
    gc = g_cum.detach().cpu().double().numpy()
    B, T, H = gc.shape
    starts = np.zeros(T, dtype=bool)
    if cu_seqlens is None:
        starts[::chunk] = True
    else:
        cu = [int(x) for x in cu_seqlens]
        for a, b in zip(cu[:-1], cu[1:]):
            starts[a:b:chunk] = True
    g = gc.copy()
    g[:, 1:] = gc[:, 1:] - gc[:, :-1]
    g[:, starts] = gc[:, starts]
    return g


def host_gcum(g, cu_seqlens=None, chunk=64):
    """The chunk-local inclusive cumsum of the raw gate, in fp32 on the CPU (the backward's ``g``
    argument), computed independently of the CUDA forward."""
    g32 = g.detach().cpu().float()
    B, T, H = g32.shape
    out = torch.empty_like(g32)
    bounds = ([(a, b) for a, b in zip([int(c) for c in cu_seqlens[:-1]], [int(c) for c in cu_seqlens[1:]])]
              if cu_seqlens is not None else [(0, T)])
    for a, b in bounds:
        for c0 in range(a, b, chunk):
            c1 = min(b, c0 + chunk)
            acc = torch.zeros(B, H, dtype=torch.float32)
            for t in range(c0, c1):   # sequential fp32 sums
                acc = acc + g32[:, t]
                out[:, t] = acc
    return out


def to_dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def select_groups(x, groups, G, n_seqs):
    """Restrict CPU inputs to some q/k head groups (each with its G value heads)."""
    hv = [h for hq in groups for h in range(hq * G, (hq + 1) * G)]
    out = dict(x)
    out["q"] = x["q"][:, :, groups]
    out["k"] = x["k"][:, :, groups]
    for key in ("v", "g", "beta", "do"):
        out[key] = x[key][:, :, hv]
    for key in ("h0", "dht"):
        if x[key] is not None:
            out[key] = x[key][:, hv]
    return out, hv


def run_fwd_case(x, cp_mode="auto", warmup_chunks=8, groups=None, check_aux=True, output_h=False, out_f32=False):
    """Forward parity.  ``groups`` restricts the oracle to some head groups.  ``out_f32`` runs the
    checking mode (o and A stored as fp32 by the same kernels) and holds them to the plain bound."""
    io = x["q"].dtype
    d = to_dev(x)
    G = x["v"].shape[2] // x["q"].shape[2]
    g_cum, A, o, h, ht = gdn.chunk_gated_delta_rule_fwd(
        d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["h0"],
        cu_seqlens=d["cu_seqlens"], output_final_state=True, output_h=output_h, cp_mode=cp_mode,
        warmup_chunks=warmup_chunks, out_f32=out_f32)
    st = torch.float32 if out_f32 else io
    torch.cuda.synchronize()
    n_seqs = ht.shape[0]
    xs, hv = (x, None) if groups is None else select_groups(x, groups, G, n_seqs)
    o_ref, ht_ref = oracle.oracle_fwd(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], x["scale"],
                                      xs["h0"], cu_seqlens=x["cu_seqlens"])
    sel = (lambda t, ax: t) if hv is None else (lambda t, ax: t.index_select(ax, torch.tensor(hv, device=t.device)))
    assert o.dtype == st
    infos = [check("o", sel(o, 2), o_ref, io, st), check("final_state", sel(ht, 1), ht_ref, io, torch.float32)]
    if check_aux:
        gc_ref, A_ref = oracle.oracle_chunk_aux(xs["k"], xs["g"], xs["beta"], cu_seqlens=x["cu_seqlens"])
        gtol = 2.4e-7 if io == torch.float32 else 1e-5
        err = np.abs(sel(g_cum, 2).cpu().double().numpy() - gc_ref)
        assert (err <= gtol * (1 + np.abs(gc_ref))).all(), f"g_cum err {err.max():.3e}"
        infos.append(check("A", sel(A, 2), A_ref, io, st))
    return dict(g_cum=g_cum, A=A, o=o, ht=ht, h=h, infos=infos)


def run_bwd_case(x, groups=None, saved=False, out_f32=False):
    """Backward parity.  The backward's ``g`` argument is the chunk-local fp32 cumsum computed on the
    host (``host_gcum``); the oracle gets the raw gate it implies (exact fp64 differences), so the
    comparison uses no value produced by the CUDA path.  With ``saved`` the save-for-backward pair
    (the training step's launch configuration) also runs, from the CUDA forward, and must equal the
    recomputing backward given that forward's g_cum bit for bit.  ``out_f32`` runs the checking mode
    (dq, dk, dv stored as fp32) and holds them to the plain bound."""
    io = x["q"].dtype
    d = to_dev(x)
    G = x["v"].shape[2] // x["q"].shape[2]
    g_cum = host_gcum(x["g"], x["cu_seqlens"]).cuda()
    if saved:
        g_gpu, A_gpu, _, _, sv = gdn.chunk_gated_delta_rule_fwd_saved(
            d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["h0"],
            cu_seqlens=d["cu_seqlens"])
        grads = gdn.chunk_gated_delta_rule_bwd_saved(
            d["q"], d["k"], d["v"], g_gpu, d["beta"], A_gpu, d["do"], sv, dht=d["dht"], scale=x["scale"],
            initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], out_f32=out_f32)
        del sv
        rec = gdn.chunk_gated_delta_rule_bwd(
            d["q"], d["k"], d["v"], g_gpu, d["beta"], A_gpu, d["do"], dht=d["dht"], scale=x["scale"],
            initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], out_f32=out_f32)
        torch.cuda.synchronize()
        for a, b in zip(grads, rec):
            assert (a is None) == (b is None) and (a is None or torch.equal(a, b))
        del grads, rec
    ref = gdn.chunk_gated_delta_rule_bwd(
        d["q"], d["k"], d["v"], g_cum, d["beta"], None, d["do"], dht=d["dht"], scale=x["scale"],
        initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], out_f32=out_f32)
    torch.cuda.synchronize()
    dq, dk, dv, db, dg, dh0 = ref
    st = torch.float32 if out_f32 else io
    assert dq.dtype == dk.dtype == dv.dtype == st
    g_rec = recovered_gate(g_cum, x["cu_seqlens"])
    xs = dict(x, g=torch.from_numpy(g_rec))
    hv = None
    if groups is not None:
        xs, hv = select_groups(xs, groups, G, None)
    r = oracle.oracle_bwd(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], xs["do"], x["scale"], xs["h0"],
                          xs["dht"], cu_seqlens=x["cu_seqlens"])
    if hv is None:
        selv = selq = (lambda t, ax: t)
    else:
        selv = lambda t, ax: t.index_select(ax, torch.tensor(hv, device=t.device))
        selq = lambda t, ax: t.index_select(ax, torch.tensor(list(groups), device=t.device))
    infos = [check("dq", selq(dq, 2), r[0], io, st), check("dk", selq(dk, 2), r[1], io, st),
             check("dv", selv(dv, 2), r[2], io, st), check("dbeta", selv(db, 2), r[3], io, torch.float32),
             check("dg", selv(dg, 2), r[4], io, torch.float32)]
    if dh0 is not None:
        infos.append(check("dh0", selv(dh0, 1), r[5], io, torch.float32))
    return infos
