"""CUDA path vs the fp64 oracle, element by element (needs a GB300).

Small cases span several 64-token chunks and a ragged tail and cover the
edge cases (T = 1, exact chunk multiples, empty and 1-token sequences, no
initial state, strong decay, beta = 0, grouped heads G = 1..4, head size 64).
The ``full_*`` cases run each benchmark workload at its full size in the
benchmark's launch configuration and compare sampled head groups, which the
oracle can compute independently of the others.
"""
import pytest
import torch

from gpu_cases import run_bwd_case, run_fwd_case
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return make_inputs(workload(name).scaled(**kw))


CASES = {
    "tiny_fp32": lambda: make_inputs(workload("tiny_fp32")),
    "fp32_ragged_gva": lambda: small("tiny_fp32", T=150, Hq=1, Hv=3, seed=10),
    "bf16_ragged": lambda: small("train_b2_t8192_h64", B=2, T=300, Hq=2, Hv=4, seed=11),
    "bf16_gva4_d64": lambda: small("train_b2_t8192_h64", B=1, T=200, Hq=1, Hv=4, K=64, V=64, seed=12),
    "bf16_t1": lambda: small("train_b2_t8192_h64", B=3, T=1, Hq=2, Hv=2, seed=13),
    "bf16_t64": lambda: small("prefill_b4_t4096", B=1, T=64, Hq=2, Hv=4, seed=14),
    "bf16_no_h0": lambda: small("prefill_b4_t4096", B=2, T=129, Hq=2, Hv=4, seed=15),
    "bf16_strong_decay": lambda: small("longseq_b1_t32k_h8", T=260, Hq=1, Hv=2, g_shift=4.0, seed=16),
    "bf16_dk64_v128": lambda: small("prefill_b4_t4096", B=1, T=100, Hq=1, Hv=2, K=64, V=128, seed=17),
    # a GVA group of 12 value heads: the prep kernel prepares the gates in two groups (8 + 4)
    "bf16_gva12": lambda: small("train_b2_t8192_h64", B=1, T=130, Hq=1, Hv=12, seed=28),
}


def varlen_case():
    x = small("varlen_8seq_32k", T=341, Hq=2, Hv=2, seed=18, n_varlen=6, varlen_min=1, varlen_max=200)
    lens = [1, 64, 65, 0, 130, 81]
    x["cu_seqlens"] = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    return x


CASES["bf16_varlen_edge"] = varlen_case


def beta0_case():
    x = small("train_b2_t8192_h64", B=1, T=140, Hq=1, Hv=2, seed=19)
    x["beta"][..., 0] = 0.0
    x["g"][..., 1] = 0.0
    return x


CASES["bf16_beta0_g0"] = beta0_case
CASES["bf16_dk128_v64"] = lambda: small("train_b2_t8192_h64", B=2, T=150, Hq=1, Hv=2, K=128, V=64, seed=22)


def varlen_d64_case():
    x = small("varlen_8seq_32k", T=341, Hq=2, Hv=2, K=64, V=64, seed=23, n_varlen=6, varlen_min=1, varlen_max=200)
    lens = [1, 64, 65, 0, 130, 81]
    x["cu_seqlens"] = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    return x


CASES["bf16_d64_varlen_edge"] = varlen_d64_case


def split_d64_case():  # 64-wide heads through the exact sequence split; one value head does not decay
    x = small("longseq_b1_t32k_h8", T=4096 + 100, Hq=2, Hv=4, K=64, V=64, seed=24)
    x["g"][..., 1] = 0.0
    return x


CASES["bf16_d64_split"] = split_d64_case


def _store_modes(name):
    """bf16 io runs twice: bf16 outputs (bound + half an ulp of bf16) and the fp32-store checking mode
    (the plain bound); fp32 io has only fp32 outputs."""
    return [False, True] if not name.endswith("fp32") and "fp32_" not in name else [False]


SMALL = [(n, f) for n in CASES for f in _store_modes(n)]


@pytest.mark.parametrize("name,out_f32", SMALL)
def test_fwd_small(name, out_f32):
    x = CASES[name]()
    run_fwd_case(x, out_f32=out_f32)


@pytest.mark.parametrize("name,out_f32", SMALL)
def test_bwd_small(name, out_f32):
    x = CASES[name]()
    if x["do"] is None:
        pytest.skip("no upstream gradient")
    run_bwd_case(x, out_f32=out_f32)


@pytest.mark.parametrize("varlen", [False, True])
def test_fwd_h_output_vs_oracle_and_state_continuation(varlen):
    """The returned chunk-entry states h equal the oracle's final states of the prefix runs (fp32
    output: 2e-3 * RMS), and running two halves with state passing equals one run."""
    import gated_delta_rule_50_gb300 as gdn
    import oracle
    from parity import check
    x = small("train_b2_t8192_h64", B=1, T=300, Hq=1, Hv=2, seed=20)
    cu = torch.tensor([0, 130, 300], dtype=torch.int32) if varlen else None
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    h0 = d["h0"] if not varlen else d["h0"].repeat(2, 1, 1, 1) * torch.tensor([1.0, -0.5], device="cuda").view(2, 1, 1, 1)
    _, _, o, h, ht = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                                    initial_state=h0, output_h=True,
                                                    cu_seqlens=cu.cuda() if varlen else None)
    torch.cuda.synchronize()
    h = h.reshape(-1, 2, 128, 128)  # [chunks over all sequences][Hv][K][V]
    seqs = [(0, 130), (130, 300)] if varlen else [(0, 300)]
    ci = 0
    h0c = h0.cpu()
    for si, (a, b) in enumerate(seqs):
        for c0 in range(a, b, 64):
            if c0 == a:
                ref = h0c[si].double().numpy()
            else:
                sl = slice(a, c0)
                _, ref = oracle.oracle_fwd(x["q"][:, sl], x["k"][:, sl], x["v"][:, sl], x["g"][:, sl],
                                           x["beta"][:, sl], x["scale"], h0c[si:si + 1])
                ref = ref[0]
            check(f"h[{ci}]", h[ci], ref, x["q"].dtype, torch.float32)
            ci += 1
    assert ci == h.shape[0]
    if varlen:
        return
    _, _, o1, _, h1 = gdn.chunk_gated_delta_rule_fwd(d["q"][:, :128], d["k"][:, :128], d["v"][:, :128],
                                                     d["g"][:, :128], d["beta"][:, :128], scale=x["scale"],
                                                     initial_state=d["h0"], out_f32=True)
    _, _, o2, _, h2 = gdn.chunk_gated_delta_rule_fwd(d["q"][:, 128:], d["k"][:, 128:], d["v"][:, 128:],
                                                     d["g"][:, 128:], d["beta"][:, 128:], scale=x["scale"],
                                                     initial_state=h1, out_f32=True)
    _, _, of, _, _ = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                                    initial_state=d["h0"], out_f32=True)
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    check("o (two halves)", torch.cat([o1, o2], 1), o_ref, x["q"].dtype, torch.float32)
    check("o (one run)", of, o_ref, x["q"].dtype, torch.float32)
    check("final_state (two halves)", h2, ht_ref, x["q"].dtype, torch.float32)


def test_autograd_matches_low_level():
    import gated_delta_rule_50_gb300 as gdn
    x = small("train_b2_t8192_h64", B=1, T=130, Hq=1, Hv=2, seed=21)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    leaves = [d[k].clone().requires_grad_(True) for k in ("q", "k", "v", "g", "beta", "h0")]
    o, ht = gdn.chunk_gated_delta_rule(*leaves[:5], initial_state=leaves[5], output_final_state=True)
    torch.autograd.backward([o, ht], [d["do"], d["dht"]])
    g_cum, A, _, _, _ = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                       initial_state=d["h0"])
    ref = gdn.chunk_gated_delta_rule_bwd(d["q"], d["k"], d["v"], g_cum, d["beta"], A, d["do"], dht=d["dht"],
                                         initial_state=d["h0"])
    for leaf, r in zip(leaves, [ref[0], ref[1], ref[2], ref[4], ref[3], ref[5]]):
        assert torch.equal(leaf.grad, r)


# ------------------------------------------------------------- full-size workloads
FULL_FWD = [("prefill_b4_t4096", [0, 9]), ("train_b2_t8192_h64", [3]), ("varlen_8seq_32k", [5]),
            ("longseq_b1_t32k_h8", [2])]
FULL_BWD = [("train_b2_t8192_h64", [7]), ("varlen_8seq_32k", [11]), ("longseq_b1_t32k_h8", [1])]


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("name,groups", FULL_FWD)
def test_fwd_full_size_sampled(name, groups, out_f32):
    x = make_inputs(workload(name))
    run_fwd_case(x, groups=groups, check_aux=(name != "train_b2_t8192_h64"), out_f32=out_f32)


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("name,groups", FULL_BWD)
def test_bwd_full_size_sampled(name, groups, out_f32):
    x = make_inputs(workload(name))
    run_bwd_case(x, groups=groups, out_f32=out_f32)


def test_tiny_fp32_full_config():
    """The tiny fp32 configuration (B=1, T=256, H=2, K=V=64) forward and backward at 1e-5 * RMS."""
    x = make_inputs(workload("tiny_fp32"))
    run_fwd_case(x)
    run_bwd_case(x)


@pytest.mark.parametrize("out_f32", [False, True])
def test_training_step_full_size_sampled(out_f32):
    """The benchmark's training step (save-for-backward pair) at full size: all gradients bit-equal to
    the recomputing backward; sampled head group vs the oracle."""
    x = make_inputs(workload("train_b2_t8192_h64"))
    run_bwd_case(x, groups=[12], saved=True, out_f32=out_f32)
