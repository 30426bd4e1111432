#!/usr/bin/env python3
"""Benchmark of the gated delta rule chunked prefill, forward + backward, on GB300.

One step = one forward pass (gdn_fwd: gate cumsum, A, state scan, o, final
state, keeping the chunk-entry states) plus one backward pass (gdn_bwd_saved:
dS scan and per-chunk gradients from what the forward kept) over the
training-shaped workload B=2, T=8192, Hq=16, Hv=64, K=V=128, bf16 io with fp32
gates and states, all inputs resident in HBM.  Prints ONE JSON line (rank 0)
with the step's tokens/s and beside it: the recomputing backward (gdn_bwd),
the dominant kernel's roofline, the end-to-end step from pinned host memory,
the split modes of the small-head long-sequence workload, 64-wide heads and
the CPU oracle baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference available; it
is a plain per-token recurrence, not a competitor) on a bounded sample of the
same workload.  Under torchrun (N > 1) every rank runs its own replica of the
workload (weak scaling, no collective on the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from synth import make_inputs, workload  # noqa: E402

WORKLOAD = "train_b2_t8192_h64"
METRIC = "GDN chunked-prefill fwd/bwd tokens/s on 1 GB300; % of tensor/HBM roofline"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_config(w, world):
    """The ``config`` object of both arms' JSON lines (the same workload string in each)."""
    return {"workload": f"{w.name}: B={w.B} T={w.T} Hq={w.Hq} Hv={w.Hv} K={w.K} V={w.V} chunk=64, "
                        "fwd+bwd per step",
            "global_batch": w.B * world, "seq_len": w.T,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "512 MB buffer written between timed steps (outside the per-step events)"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS, sm_max_mhz=2070.0), "fallback"


# ---------------------------------------------------------------- algorithmic work
def algorithmic(w, C=64):
    """Algorithmic flops / bytes of one forward and one backward pass.

    Per token and value head (d = K = V, e = io element bytes, G = Hv / Hq):
      fwd flops = 2C(3K + 2V) + 3 * 2KV            (KK^T, QK^T, W, U, P U'; W S, state update, Q S)
      bwd flops = 16 d^2 + 28 C d + 4 C^2          (recompute + reverse scan + intra-chunk backward)
      fwd bytes = 2Ke/G + 2Ve + 8 + 4 + Ce         (q, k; v, o; g, beta; g_cum; A)
      bwd bytes = 4Ke/G + 3Ve + 16 + Ce            (q, k, dq, dk; v, do, dv; g_cum, beta, dbeta, dg; A)
    plus 4KV bytes per state tensor per (sequence, value head): h0, ht (fwd);
    h0, dht, dh0 (bwd).
    """
    K, V, G = w.K, w.V, w.Hv // w.Hq
    e = 2 if w.io_dtype == torch.bfloat16 else 4
    th = w.tokens * w.Hv
    units = w.n_seqs * w.Hv
    st = 4 * K * V
    nst_f = (1 if w.has_h0 else 0) + 1
    nst_b = (1 if w.has_h0 else 0) * 2 + (1 if w.has_dht else 0)
    d = K
    fwd_f = th * (2 * C * (3 * K + 2 * V) + 6 * K * V)
    bwd_f = th * (16 * d * d + 28 * C * d + 4 * C * C)
    fwd_b = th * (2 * K * e / G + 2 * V * e + 12 + C * e) + units * st * nst_f
    bwd_b = th * (4 * K * e / G + 3 * V * e + 16 + C * e) + units * st * nst_b
    return dict(fwd_flops=fwd_f, bwd_flops=bwd_f, fwd_bytes=fwd_b, bwd_bytes=bwd_b)


def kernel_work(name, w, C=64):
    """(algorithmic flops, algorithmic bytes) of one launch of a kernel over
    workload ``w``: the share of its pass's algorithmic work that the kernel
    performs (per token and value head; d = K = V, e = io bytes, G = Hv / Hq):

      fwd_prep_tc   K K^T, Q K^T                            4CK flops;
                    reads g, beta; writes g_cum, A          12 + Ce bytes
      fwd_tc        the rest of the forward                 fwd - prep
      bwd_prep_tc   K K^T, Q K^T                            4CK flops; reads g_cum, beta: 8 bytes
      bwd_state_tc  W, U, W S, state update                 2C(K + V) + 4KV flops;
                    reads k, v                              Ke/G + Ve bytes
      bwd_dscan_tc  K dS, P^T dO, A^T dDl, state update      6KV + 4CV flops;
                    reads q, k, do, g_cum, beta             2Ke/G + Ve + 8 bytes
      bwd_intra_tc  the rest of the backward's flops;       bwd - prep - state - dscan;
                    reads q, k, v, do, g_cum, beta; writes dq, dk, dv, dbeta, dg
                                                            4Ke/G + 3Ve + 16 bytes
    Workspace traffic (operand images, chunk states) is not algorithmic and is
    not counted.  CUDA-core kernels (fp32 io or other head sizes) use the same
    shares.
    """
    K, V, G = w.K, w.V, w.Hv // w.Hq
    e = 2 if w.io_dtype == torch.bfloat16 else 4
    th = w.tokens * w.Hv
    alg = algorithmic(w, C)
    pr_f = th * 4 * C * K
    st_f = th * (2 * C * (K + V) + 4 * K * V)
    ds_f = th * (6 * K * V + 4 * C * V)
    table = {
        "fwd_prep_tc": (pr_f, th * (12 + C * e)),
        "fwd_tc": (alg["fwd_flops"] - pr_f, alg["fwd_bytes"] - th * (12 + C * e)),
        "bwd_prep_tc": (pr_f, th * 8),
        "bwd_state_tc": (st_f, th * (K * e / G + V * e)),
        "bwd_dscan_tc": (ds_f, th * (2 * K * e / G + V * e + 8)),
        "bwd_intra_tc": (alg["bwd_flops"] - pr_f - st_f - ds_f, th * (4 * K * e / G + 3 * V * e + 16)),
    }
    table["fwd_scan"] = (alg["fwd_flops"], alg["fwd_bytes"])
    table["bwd_state"] = table["bwd_state_tc"]
    table["bwd_dscan"] = table["bwd_dscan_tc"]
    table["bwd_intra"] = table["bwd_intra_tc"]
    return table.get(name)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sms:
            return None
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------- our arm
def kernel_profile(lib):
    import ctypes
    n = 32
    names = ctypes.create_string_buffer(64 * n)
    counts = (ctypes.c_int * n)()
    ms = (ctypes.c_double * n)()
    k = lib.gdn_profile_read(names, 64, counts, ms, n)
    if k < 0:
        raise RuntimeError("gdn_profile_read failed")
    out = {}
    for i in range(k):
        nm = names.raw[64 * i:64 * (i + 1)].split(b"\0")[0].decode()
        out[nm] = (counts[i], ms[i])
    return out


def max_over_ranks(values, world, device):
    """Each timing's maximum over the ranks (the slowest replica sets the job's time); the values
    themselves at world size 1."""
    if world == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed per second of the max-over-ranks time."""
    return world * units_per_rank / (ms / 1e3)


def run_ours(args, rank, world, local_rank):
    import ctypes
    import gated_delta_rule_50_gb300 as gdn
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    lib = gdn.load_library()
    lib.gdn_profile_enable.argtypes = [ctypes.c_int]
    lib.gdn_profile_read.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int]
    w = workload(args.workload)
    x = make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu_cpu = x["cu_seqlens"]
    ws_f = torch.empty(gdn.workspace_bytes("fwd", d["q"], d["v"], d["cu_seqlens"], cu_cpu), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(gdn.workspace_bytes("bwd", d["q"], d["v"], d["cu_seqlens"], cu_cpu), dtype=torch.uint8,
                       device=dev)
    ws_bs = torch.empty(gdn.workspace_bytes("bwd_saved", d["q"], d["v"], d["cu_seqlens"], cu_cpu),
                        dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # The training step: the forward keeps its operand images and chunk-entry states for the backward
    # (the save-for-backward pair, as the autograd function uses it).
    def fwd():
        return gdn.chunk_gated_delta_rule_fwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                                                    initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                                                    cu_seqlens_cpu=cu_cpu, output_final_state=True,
                                                    workspace=ws_f)

    def bwd(f):
        g_cum, A, saved = f[0], f[1], f[4]
        return gdn.chunk_gated_delta_rule_bwd_saved(d["q"], d["k"], d["v"], g_cum, d["beta"], A, d["do"], saved,
                                                    dht=d["dht"], scale=d["scale"], initial_state=d["h0"],
                                                    cu_seqlens=d["cu_seqlens"], cu_seqlens_cpu=cu_cpu,
                                                    workspace=ws_bs)

    def bwd_recompute(f):  # the pages' backward interface: recomputes A, P and the chunk states
        g_cum, A = f[0], f[1]
        return gdn.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], g_cum, d["beta"], A, d["do"],
                                              dht=d["dht"], scale=d["scale"], initial_state=d["h0"],
                                              cu_seqlens=d["cu_seqlens"], cu_seqlens_cpu=cu_cpu,
                                              workspace=ws_b)

    for _ in range(args.warmup):
        bwd(fwd())
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    lib.gdn_profile_enable(1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)           # write > L2 between timed steps
        evs[i][0].record(stream)
        f = fwd()
        evs[i][1].record(stream)
        bwd(f)
        evs[i][2].record(stream)
        f = None                        # a training step frees its saved tensors before the next forward
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    lib.gdn_profile_enable(0)
    kprof = kernel_profile(lib)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    fwd_ms = sum(a.elapsed_time(b) for a, b, _ in evs) / args.steps
    bwd_ms = sum(b.elapsed_time(c) for _, b, c in evs) / args.steps
    # the recomputing backward, timed alone on the same forward output (reported beside the step)
    f_last = fwd()
    rec_ms = 0.0
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        bwd_recompute(f_last)
        e1.record(stream)
        torch.cuda.synchronize()
        rec_ms += e0.elapsed_time(e1) / args.steps
    step_ms = fwd_ms + bwd_ms
    step_ms, fwd_ms, bwd_ms = max_over_ranks([step_ms, fwd_ms, bwd_ms], world, dev)

    peaks, peak_src = load_peaks()
    alg = algorithmic(w)
    tokens = w.tokens
    # dominant kernel
    launches = sum(c for c, _ in kprof.values())
    dom = max(kprof.items(), key=lambda kv: kv[1][1]) if kprof else None
    roof = None
    if dom:
        name, (cnt, tot) = dom
        kw = kernel_work(name, w)
        avg_s = tot / cnt / 1e3
        if kw:
            fl, by = kw
            t_tc = fl / (peaks["bf16_tflops"] * 1e12)
            t_hbm = by / (peaks["hbm_gbs"] * 1e9)
            if t_hbm >= t_tc:
                peak = peaks["hbm_gbs"]
                ach = by / avg_s / 1e9
                roof = {"bound": "hbm", "kernel": name, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(ach / peak, 4), "peak_source": f"hbm_gbs, {peak_src} (burst copy)"}
            else:
                peak = peaks["bf16_tflops"]
                ach = fl / avg_s / 1e12
                roof = {"bound": "tensor", "kernel": name, "achieved": round(ach, 2), "peak": peak,
                        "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                        "peak_source": f"bf16_tflops, {peak_src} (burst cuBLAS)"}
            roof["avg_launch_us"] = round(avg_s * 1e6, 2)
            roof["algorithmic_flops"] = fl
            roof["algorithmic_bytes"] = by
            roof["traffic"] = traffic_bytes(name)
    # whole-pass roofline (both passes, measured peaks)
    bw = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    t_roof_f = max(alg["fwd_flops"] / tc, alg["fwd_bytes"] / bw)
    t_roof_b = max(alg["bwd_flops"] / tc, alg["bwd_bytes"] / bw)
    res = {
        "metric": METRIC,
        "value": round(job_rate(tokens, world, step_ms), 1),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.io_dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded; q,k unit-norm N(0,1), v N(0,1), g=-softplus(N(0,1)) with 10% "
                "of heads g=0, beta=sigmoid(N(0,1)), h0/dht 0.1 N(0,1))",
        "config": workload_config(w, world),
        "fwd": {"ms": round(fwd_ms, 4), "tokens_per_s": round(world * tokens / (fwd_ms / 1e3), 1),
                "roofline_frac": round(t_roof_f / (fwd_ms / 1e3), 4)},
        "bwd": {"ms": round(bwd_ms, 4), "tokens_per_s": round(world * tokens / (bwd_ms / 1e3), 1),
                "roofline_frac": round(t_roof_b / (bwd_ms / 1e3), 4),
                "reuses": "the forward's A / P operand images and chunk-entry states (save for backward)"},
        "bwd_recompute": {"ms": round(rec_ms, 4), "tokens_per_s": round(world * tokens / (rec_ms / 1e3), 1),
                          "note": "backward with the pages' interface (recomputes A, P and the chunk states)"},
        "step_roofline_frac": round((t_roof_f + t_roof_b) / (step_ms / 1e3), 4),
        "roofline": roof,
        "kernels": {k: {"launches": c, "ms_total": round(t, 4)} for k, (c, t) in sorted(kprof.items())},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"]},
    }
    # the pages' forward (no chunk-entry states kept) on this workload and on the prefill workload
    res["fwd_only"] = run_fwd_only(dev, gdn, w, d, cu_cpu, flush, peaks)
    if not args.no_prefill:
        pw = workload("prefill_b4_t4096")
        px = make_inputs(pw)
        pd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in px.items()}
        res["prefill_b4_t4096"] = run_fwd_only(dev, gdn, pw, pd, None, flush, peaks)
        del pd, px
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, w, x, dev, gdn, world)
    if not args.no_autocp and rank == 0:
        res["autocp"] = run_autocp(dev, gdn)
    if not args.no_head64 and rank == 0:
        res["head_dim_64"] = run_head64(dev, gdn)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        res["cpu_baseline"] = cpu_baseline(w, x, budget_s=args.cpu_budget)
    return res


def run_fwd_only(dev, gdn, w, d, cu_cpu, flush, peaks, steps=20, warmup=5):
    """The forward as the pages' interface runs it (o and the final state; no chunk-entry states kept),
    inputs resident in HBM, L2 flushed before every timed call, per-call CUDA events."""
    ws = torch.empty(gdn.workspace_bytes("fwd", d["q"], d["v"], d["cu_seqlens"], cu_cpu), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    def f():
        return gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                                              initial_state=d["h0"], cu_seqlens=d["cu_seqlens"],
                                              cu_seqlens_cpu=cu_cpu, output_final_state=True, workspace=ws)
    for _ in range(warmup):
        f()
    torch.cuda.synchronize(dev)
    tot = 0.0
    for i in range(steps):
        flush.fill_(i & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        f()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tot += e0.elapsed_time(e1)
    ms = tot / steps
    alg = algorithmic(w)
    t_roof = max(alg["fwd_flops"] / (peaks["bf16_tflops"] * 1e12), alg["fwd_bytes"] / (peaks["hbm_gbs"] * 1e9))
    return {"workload": f"{w.name}: B={w.B} T={w.T} Hq={w.Hq} Hv={w.Hv} K={w.K} V={w.V}, forward "
                        f"({'with' if w.has_h0 else 'no'} initial state, final state out, no h)",
            "ms": round(ms, 4), "tokens_per_s": round(w.tokens / (ms / 1e3), 1),
            "roofline_frac": round(t_roof / (ms / 1e3), 4), "roofline_us": round(t_roof * 1e6, 1)}


def run_autocp(dev, gdn, steps=10, warmup=3):
    """The small-head long-sequence workload (B x Hv = 8 meets the AutoCP trigger): forward
    unsplit, exact split and warmup split (8 chunks); backward unsplit and exact split.
    Inputs resident in HBM, CUDA events on the current stream; larger than L2."""
    aw = workload("longseq_b1_t32k_h8")
    ax = make_inputs(aw)
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in ax.items()}
    out = {"workload": f"{aw.name}: B={aw.B} T={aw.T} Hq={aw.Hq} Hv={aw.Hv} K={aw.K} V={aw.V}, forward"}
    plan = gdn.cp_plan(d["q"], d["v"], cp_mode="auto")
    out["segments"] = {"seg_len_chunks": plan[0], "n_seg": plan[1]} if plan else None
    for mode in ("off", "auto", "warmup"):
        def f():
            return gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=ax["scale"],
                                                  initial_state=d["h0"], output_final_state=True, cp_mode=mode,
                                                  warmup_chunks=8)
        for _ in range(warmup):
            f()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            f()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        key = {"off": "unsplit", "auto": "exact_split", "warmup": "warmup_split_8"}[mode]
        out[key] = {"ms": round(ms, 4), "tokens_per_s": round(aw.tokens / (ms / 1e3), 1)}
    # backward: unsplit vs exact split of both chains (warmup does not apply to the backward)
    g_cum, A, _, _, _ = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                       scale=ax["scale"], initial_state=d["h0"])
    for mode in ("off", "auto"):
        def b():
            return gdn.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], g_cum, d["beta"], A, d["do"],
                                                  dht=d["dht"], scale=ax["scale"], initial_state=d["h0"],
                                                  cp_mode=mode)
        for _ in range(warmup):
            b()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(max(3, steps // 2)):
            b()
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / max(3, steps // 2)
        key = {"off": "bwd_unsplit", "auto": "bwd_exact_split"}[mode]
        out[key] = {"ms": round(ms, 4), "tokens_per_s": round(aw.tokens / (ms / 1e3), 1)}
    return out


def run_head64(dev, gdn, steps=10, warmup=3):
    """The training-shaped workload with 64-wide heads (K = V = 64): the 128-wide tensor-core kernels
    on zero-padded copies (the library pads and slices), forward and the save-for-backward training
    step's backward.  Inputs resident in HBM, CUDA events on the current stream."""
    hw = workload("train_b2_t8192_h64").scaled(name="train_b2_t8192_h64_d64", K=64, V=64)
    hx = make_inputs(hw)
    d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in hx.items()}
    out = {"workload": f"{hw.name}: B={hw.B} T={hw.T} Hq={hw.Hq} Hv={hw.Hv} K={hw.K} V={hw.V}",
           "path": "128-wide tensor-core kernels on zero-padded operands"}
    fwd = lambda: gdn.chunk_gated_delta_rule_fwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=hx["scale"],
                                                       initial_state=d["h0"], output_final_state=True)
    f = fwd()
    bwd = lambda: gdn.chunk_gated_delta_rule_bwd_saved(d["q"], d["k"], d["v"], f[0], d["beta"], f[1], d["do"], f[4],
                                                       dht=d["dht"], scale=hx["scale"], initial_state=d["h0"])
    for key, fn in (("fwd", fwd), ("bwd", bwd)):
        ms = time_cuda(fn, dev, steps, warmup)
        out[key] = {"ms": round(ms, 4), "tokens_per_s": round(hw.tokens / (ms / 1e3), 1)}
    return out


def _cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if part:
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def bind_near_gpu(dev):
    """Best effort: restricts this process to the CPUs local to the GPU (its PCI device's local_cpulist in
    sysfs), so that pinned host buffers allocated now sit in the GPU's nearest host memory.  Returns the
    previous affinity (to restore, or None) and what was found: "bound" (restricted now), "local" (every
    allowed CPU is already local to the GPU), "none local" (no allowed CPU is) or "unknown" (no locality
    information)."""
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={dev.index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip()
        dom, rest = bus.split(":", 1)
        with open(f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest.lower()}/local_cpulist") as fh:
            near = _cpulist(fh.read())
        old = os.sched_getaffinity(0)
    except Exception:
        return None, "unknown"
    if not near & old:
        return None, "none local"
    if near & old == old:
        return None, "local"
    os.sched_setaffinity(0, near & old)
    return old, "bound"


def copy_rates(host, dev):
    """Isolated host->device and device->host copy rates (GB/s) of the given pinned tensors."""
    devs = [torch.empty_like(t, device=dev) for t in host]
    nbytes = sum(t.numel() * t.element_size() for t in host)
    rates = []
    for direction in ("h2d", "d2h"):
        for _ in range(2):
            for a, b in zip(host, devs):
                (b.copy_(a, non_blocking=True) if direction == "h2d" else a.copy_(b, non_blocking=True))
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for a, b in zip(host, devs):
            (b.copy_(a, non_blocking=True) if direction == "h2d" else a.copy_(b, non_blocking=True))
        e1.record()
        torch.cuda.synchronize(dev)
        rates.append(round(nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9, 1))
    return rates


def run_e2e(args, w, x, dev, gdn, world):
    """Same step through the public API with host (pinned) buffers: every step copies its inputs
    host->device and all its outputs device->host inside the timed region.  The steps are pipelined
    the way a training loop overlaps data movement with compute: step k+1's inputs are copied (one
    stream) and step k-1's outputs read back (another stream) while step k computes, with two device
    input buffers."""
    names_in = ["q", "k", "v", "g", "beta", "h0", "do", "dht"]
    old_affinity, locality = bind_near_gpu(dev)  # restored once every pinned buffer exists (after the warm-up)
    host = {k: x[k].pin_memory() for k in names_in if x[k] is not None}
    cu_cpu = x["cu_seqlens"]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [{k: torch.empty_like(t, device=dev) for k, t in host.items()} for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer b copied
    ev_free = [torch.cuda.Event() for _ in range(2)]   # compute done with buffer b
    outs_host = [None, None]
    ev_read = [None, None]                             # read-back into host set b done
    d2h = 0
    # workspaces allocated once, as a training loop keeps them (steps run in order on one stream)
    ws_f = torch.empty(gdn.workspace_bytes("fwd", bufs[0]["q"], bufs[0]["v"], None, cu_cpu), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(gdn.workspace_bytes("bwd_saved", bufs[0]["q"], bufs[0]["v"], None, cu_cpu),
                       dtype=torch.uint8, device=dev)

    def copy_in(k):
        b = k & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_free[b])
            for name, t in host.items():
                bufs[b][name].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)

    def compute(k):
        nonlocal d2h
        b = k & 1
        d = bufs[b]
        comp.wait_event(ev_in[b])
        g_cum, A, o, ht, saved = gdn.chunk_gated_delta_rule_fwd_saved(
            d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d.get("h0"),
            output_final_state=True, cu_seqlens_cpu=cu_cpu, workspace=ws_f)
        grads = gdn.chunk_gated_delta_rule_bwd_saved(d["q"], d["k"], d["v"], g_cum, d["beta"], A, d["do"], saved,
                                                     dht=d.get("dht"), scale=x["scale"],
                                                     initial_state=d.get("h0"), cu_seqlens_cpu=cu_cpu,
                                                     workspace=ws_b)
        ev_free[b].record(comp)
        outs = [o, ht] + [t for t in grads if t is not None]
        d2h = sum(t.numel() * t.element_size() for t in outs)
        if outs_host[b] is None:
            outs_host[b] = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_free[b])
            for hb, t in zip(outs_host[b], outs):
                t.record_stream(s_out)
                hb.copy_(t, non_blocking=True)
            ev_read[b] = torch.cuda.Event()
            ev_read[b].record(s_out)

    def run(n):
        copy_in(0)
        for k in range(n):
            if k + 1 < n:
                copy_in(k + 1)
            if ev_read[k & 1] is not None:
                ev_read[k & 1].synchronize()  # host set k & 1 is free again
            compute(k)

    run(max(6, args.warmup))  # long enough for the allocator to settle on two steps in flight
    torch.cuda.synchronize()
    if old_affinity is not None:
        os.sched_setaffinity(0, old_affinity)
    h2d_gbs, d2h_gbs = copy_rates(list(host.values()), dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    run(args.steps)
    comp.wait_stream(s_out)
    comp.wait_stream(s_in)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks([e0.elapsed_time(e1) / args.steps], world, dev)[0]
    return {"value": round(job_rate(w.tokens, world, ms), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copy_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs, "host_cpus": locality},
            "pipelined": "each step's host-to-device inputs and device-to-host outputs are copied on their own "
                         "streams, overlapping the neighbouring steps' compute (two device input buffers)"}


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(w, x, n_groups):
    """A bounded sample of the workload for the oracle: the first n_groups
    q/k head groups (each with its G value heads), all sequences, all tokens."""
    G = w.Hv // w.Hq
    hv = list(range(n_groups * G))
    s = dict(x)
    s["q"], s["k"] = x["q"][:, :, :n_groups], x["k"][:, :, :n_groups]
    for key in ("v", "g", "beta", "do"):
        s[key] = x[key][:, :, hv]
    for key in ("h0", "dht"):
        if x[key] is not None:
            s[key] = x[key][:, hv]
    return s, len(hv)


def time_oracle_step(w, s):
    import oracle
    t0 = time.perf_counter()
    oracle.oracle_fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], s["scale"], s["h0"],
                      cu_seqlens=s["cu_seqlens"])
    oracle.oracle_bwd(s["q"], s["k"], s["v"], s["g"], s["beta"], s["do"], s["scale"], s["h0"], s["dht"],
                      cu_seqlens=s["cu_seqlens"])
    return time.perf_counter() - t0


def cpu_baseline(w, x, budget_s=20.0):
    import oracle
    lib = oracle.load()
    cores = oracle.max_threads(lib)
    G = w.Hv // w.Hq
    s, nh = oracle_sample(w, x, 1)
    dt = time_oracle_step(w, s)
    n_groups = max(1, min(w.Hq, int(budget_s / max(dt, 1e-3))))
    if n_groups > 1:
        s, nh = oracle_sample(w, x, n_groups)
        dt = time_oracle_step(w, s)
    # tokens/s of the whole workload = tokens processed for the sampled heads,
    # scaled by the fraction of value heads sampled
    value = w.tokens * (nh / w.Hv) / dt
    return {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 per-token oracle fwd+bwd on {n_groups} of {w.Hq} q/k head groups "
                      f"({nh} of {w.Hv} value heads), all {w.tokens} tokens; {dt:.1f} s; value scaled "
                      f"to the full workload by the head fraction"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = workload(args.workload)
    x = make_inputs(w)
    import oracle
    lib = oracle.load()
    cores = oracle.max_threads(lib)
    s, nh = oracle_sample(w, x, 1)
    for _ in range(args.warmup):   # untimed warm-up steps on the same sample
        time_oracle_step(w, s)
    times = [time_oracle_step(w, s) for _ in range(args.steps)]
    dt = sum(times) / len(times)
    value = w.tokens * (nh / w.Hv) / dt
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, world),
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"fwd+bwd of 1 of {w.Hq} q/k head groups ({nh} value heads), "
                                       "all tokens, per step; scaled by the head fraction"},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# kernel -> (DRAM bytes read + written per launch at the benchmark workload, from one ncu capture of
# that kernel; sha256 prefix of the kernel's source file when the counters were taken).  A capture on
# the half-size training shape is scaled by the 4x units of the full one (per-unit reads and writes do
# not depend on the unit count).  The figure is reported only while the source is unchanged.
TRAFFIC = {
    # one ncu capture on the half-size training shape: (843.70 + 97.48) MB, scaled by its 4x units
    "bwd_intra_tc": (4 * (843.697408e6 + 97.482496e6), "a40ebf69ffce6835"),
}
KERNEL_SOURCES = {"fwd_prep_tc": "tc_prep.cu", "bwd_prep_tc": "tc_prep.cu", "fwd_tc": "tc_fwd.cu",
                  "bwd_state_tc": "tc_fwd.cu", "bwd_dscan_tc": "tc_bwd.cu", "bwd_intra_tc": "tc_bwd_intra.cu"}


def source_sha16(kernel):
    import hashlib
    f = KERNEL_SOURCES.get(kernel)
    if f is None:
        return None
    with open(os.path.join(ROOT, "gated_delta_rule_50_gb300", "csrc", f), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def traffic_bytes(kernel):
    entry = TRAFFIC.get(kernel)
    if entry is None or entry[1] != source_sha16(kernel):
        return None
    return entry[0]


def time_cuda(fn, dev, steps, warmup):
    """Mean milliseconds of fn() over `steps` calls after `warmup`, CUDA events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


def run_sweep(args):
    """The pages' benchmark shapes on synthetic data (FlashQLA README, "Benchmark"): value-head counts
    {64, 48, 32, 24, 16, 8} (tensor parallelism 1 to 8; q/k heads = value heads / 4 as in the
    training-shaped workload), forward latency over batch lengths at 32768 tokens per batch, and backward
    latency over the total token count.  One JSON line per shape; inputs resident in HBM."""
    import gated_delta_rule_50_gb300 as gdn
    from synth import Workload
    dev = torch.device("cuda", 0)
    rows = []
    heads = (64, 48, 32, 24, 16, 8)
    for hv in heads:
        for T in (2048, 8192, 32768):
            B = 32768 // T
            w = Workload(f"sweep_fwd_h{hv}_t{T}", B=B, T=T, Hq=hv // 4, Hv=hv, K=128, V=128,
                         io_dtype=torch.bfloat16, seed=7, has_h0=True, has_dht=False, bwd=False)
            x = make_inputs(w)
            d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
            ms = time_cuda(lambda: gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                                   initial_state=d["h0"], output_final_state=True),
                           dev, args.steps, args.warmup)
            plan = gdn.cp_plan(d["q"], d["v"], cp_mode="auto")
            rows.append({"sweep": "fwd", "Hv": hv, "Hq": hv // 4, "B": B, "T": T, "ms": round(ms, 4),
                         "tokens_per_s": round(B * T / (ms / 1e3), 1),
                         "split": {"seg_len": plan[0], "n_seg": plan[1]} if plan else None})
            del d, x
    for hv in (64, 16, 8):
        for tokens in (8192, 32768, 65536):
            T = min(tokens, 32768)
            B = tokens // T
            w = Workload(f"sweep_bwd_h{hv}_n{tokens}", B=B, T=T, Hq=hv // 4, Hv=hv, K=128, V=128,
                         io_dtype=torch.bfloat16, seed=8, has_h0=True, has_dht=True, bwd=True)
            x = make_inputs(w)
            d = {k: (t.to(dev) if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
            g_cum, A, _, _, _ = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                               initial_state=d["h0"])
            ms = time_cuda(lambda: gdn.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], g_cum, d["beta"], A,
                                                                   d["do"], dht=d["dht"], initial_state=d["h0"]),
                           dev, max(3, args.steps // 2), args.warmup)
            g_cum, A, _, _, saved = gdn.chunk_gated_delta_rule_fwd_saved(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                                         initial_state=d["h0"])
            ms_saved = time_cuda(lambda: gdn.chunk_gated_delta_rule_bwd_saved(
                d["q"], d["k"], d["v"], g_cum, d["beta"], A, d["do"], saved, dht=d["dht"], initial_state=d["h0"]),
                dev, max(3, args.steps // 2), args.warmup)
            rows.append({"sweep": "bwd", "Hv": hv, "Hq": hv // 4, "B": B, "T": T, "tokens": tokens,
                         "ms": round(ms, 4), "tokens_per_s": round(tokens / (ms / 1e3), 1),
                         "saved_ms": round(ms_saved, 4), "saved_tokens_per_s": round(tokens / (ms_saved / 1e3), 1)})
            del saved
            del d, x
    for r in rows:
        print(json.dumps(r), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-autocp", action="store_true", help="skip the split-mode forward timings")
    ap.add_argument("--no-head64", action="store_true", help="skip the 64-wide-head timings")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill workload's forward")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--sweep", action="store_true",
                    help="the pages' head-count / batch-length / token-count sweep (one JSON line per shape)")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.gpus != world:
        # N ranks come from the launcher (torchrun sets WORLD_SIZE); a bare --gpus N would time one rank
        print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE={world}: launch N > 1 ranks with "
                                   f"torch.distributed.run --nproc-per-node {args.gpus}"}), flush=True)
        sys.exit(2)
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo",
                                             device_id=torch.device("cuda", local_rank)
                                             if torch.cuda.is_available() else None)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
