"""Sequence splitting with warmup (the FlashQLA pages' "AutoCP"; news page,
"FlashQLA's core advantages"): the CUDA path against oracle_fwd_warmup, the
oracle's composition of exact runs over the same segments and windows."""
import numpy as np
import pytest
import torch

import gated_delta_rule_50_gb300 as gdn
import oracle
from gpu_cases import select_groups, to_dev
from parity import BF16_TOL, check
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu


def run(x, warm, groups=None, out_f32=False):
    d = to_dev(x)
    plan = gdn.cp_plan(d["q"], d["v"], cu_seqlens=d["cu_seqlens"], cp_mode="warmup", warmup_chunks=warm)
    assert plan is not None
    _, _, o, _, ht = gdn.chunk_gated_delta_rule_fwd(
        d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["h0"],
        cu_seqlens=d["cu_seqlens"], output_final_state=True, cp_mode="warmup", warmup_chunks=warm,
        out_f32=out_f32)
    torch.cuda.synchronize()
    xs, hv = (x, None) if groups is None else select_groups(x, groups, x["v"].shape[2] // x["q"].shape[2], None)
    o_ref, ht_ref = oracle.oracle_fwd_warmup(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], x["scale"], xs["h0"],
                                             cu_seqlens=x["cu_seqlens"], seg_len=plan[0], warm=warm)
    if hv is not None:
        idx = torch.tensor(hv, device=o.device)
        o, ht = o.index_select(2, idx), ht.index_select(1, idx)
    return plan, o, ht, o_ref, ht_ref, xs


def test_warmup_differs_from_exact_and_matches_its_oracle():
    """Head 0 decays by e^-10.5 per chunk (split, warmup of one chunk) and carries a
    huge state into the first window, so the warmup result is far from the exact
    one; head 1 has g = 0 and must run unsplit (exact)."""
    x = make_inputs(workload("longseq_b1_t32k_h8").scaled(B=1, T=17 * 64 - 27, Hq=1, Hv=2, seed=40))
    x["g"][..., 0] = -10.5 / 64
    x["g"][..., 1] = 0.0
    x["v"][:, 128:192, 0] *= 32768.0
    plan, o, ht, o_ref, ht_ref, _ = run(x, warm=1)
    assert plan == (4, 5)
    L = plan[0] * 64
    o_ex, ht_ex = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    rms1 = np.sqrt(np.mean(o_ex[:, L:, 0] ** 2))
    assert np.abs(o_ref[:, L:, 0] - o_ex[:, L:, 0]).max() > 20 * BF16_TOL * rms1
    check("o seg0 h0", o[:, :L, 0], o_ref[:, :L, 0], torch.bfloat16, torch.bfloat16)
    check("o seg1+ h0", o[:, L:, 0], o_ref[:, L:, 0], torch.bfloat16, torch.bfloat16)
    check("o h1 (unsplit)", o[:, :, 1], o_ex[:, :, 1], torch.bfloat16, torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)
    assert np.allclose(ht_ref[:, 1], ht_ex[:, 1])


def test_warmup_longseq_shape_small():
    x = make_inputs(workload("longseq_b1_t32k_h8").scaled(T=8192 + 100, Hq=2, Hv=4, seed=41))
    plan, o, ht, o_ref, ht_ref, _ = run(x, warm=6)
    assert plan == (11, 12)
    check("o", o, o_ref, torch.bfloat16, torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)


def test_warmup_head64_padded():
    """64-wide heads (zero-padded to the 128-wide kernels) through the warmup split."""
    x = make_inputs(workload("longseq_b1_t32k_h8").scaled(T=4096 + 100, Hq=2, Hv=4, K=64, V=64, seed=43))
    plan, o, ht, o_ref, ht_ref, _ = run(x, warm=6)
    assert plan == (8, 9)
    check("o", o, o_ref, torch.bfloat16, torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)


def test_warmup_varlen():
    x = make_inputs(workload("varlen_8seq_32k").scaled(T=2500, Hq=1, Hv=2, seed=42, n_varlen=3))
    x["cu_seqlens"] = torch.tensor([0, 700, 2200, 2500], dtype=torch.int32)
    x["g"][..., 1] *= 0.02   # weak decay: that head's windows do not decay enough -> unsplit
    plan, o, ht, o_ref, ht_ref, _ = run(x, warm=2)
    assert plan == (5, 5)
    check("o", o, o_ref, torch.bfloat16, torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)


@pytest.mark.parametrize("out_f32", [False, True])
def test_warmup_full_size_sampled(out_f32):
    x = make_inputs(workload("longseq_b1_t32k_h8"))
    _, o, ht, o_ref, ht_ref, _ = run(x, warm=8, groups=[1], out_f32=out_f32)
    check("o", o, o_ref, torch.bfloat16, torch.float32 if out_f32 else torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)


# ------------------------------------------------------------------ exact split (default mode)
def run_exact(x, out_f32=False):
    d = to_dev(x)
    plan = gdn.cp_plan(d["q"], d["v"], cu_seqlens=d["cu_seqlens"], cp_mode="auto")
    assert plan is not None
    _, _, o, _, ht = gdn.chunk_gated_delta_rule_fwd(
        d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"], initial_state=d["h0"],
        cu_seqlens=d["cu_seqlens"], output_final_state=True, cp_mode="auto", out_f32=out_f32)
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"],
                                      cu_seqlens=x["cu_seqlens"])
    return plan, o, ht, o_ref, ht_ref


@pytest.mark.parametrize("out_f32", [False, True])
def test_exact_split_matches_unsplit_with_non_decaying_heads(out_f32):
    """Default mode on a shape the trigger splits: exact even for g = 0 heads, where warmup is invalid."""
    x = make_inputs(workload("longseq_b1_t32k_h8").scaled(T=8192 + 100, Hq=2, Hv=4, seed=43))
    x["g"][..., 1] = 0.0
    x["g"][..., 2] *= 0.02
    plan, o, ht, o_ref, ht_ref = run_exact(x, out_f32=out_f32)
    assert plan == (11, 12)
    check("o", o, o_ref, torch.bfloat16, torch.float32 if out_f32 else torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)


def test_exact_split_varlen_no_h0():
    x = make_inputs(workload("varlen_8seq_32k").scaled(T=2500, Hq=1, Hv=2, seed=44, n_varlen=3))
    x["cu_seqlens"] = torch.tensor([0, 700, 2200, 2500], dtype=torch.int32)
    x["h0"] = None
    plan, o, ht, o_ref, ht_ref = run_exact(x)
    assert plan == (5, 5)
    check("o", o, o_ref, torch.bfloat16, torch.bfloat16)
    check("final_state", ht, ht_ref, torch.bfloat16, torch.float32)


@pytest.mark.parametrize("out_f32", [False, True])
def test_exact_split_backward(out_f32):
    """Both backward chains split through segment transitions (default mode, trigger on)."""
    from gpu_cases import run_bwd_case
    x = make_inputs(workload("longseq_b1_t32k_h8").scaled(T=4096 + 100, Hq=2, Hv=4, seed=45))
    x["g"][..., 1] = 0.0
    d = to_dev(x)
    assert gdn.cp_plan(d["q"], d["v"], cp_mode="auto") == (8, 9)
    run_bwd_case(x, out_f32=out_f32)
