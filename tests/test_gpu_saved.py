"""The save-for-backward pair (chunk_gated_delta_rule_fwd_saved / _bwd_saved, C entry gdn_bwd_saved)
against the fp64 oracle and against the recomputing backward."""
import pytest
import torch

from gpu_cases import run_bwd_case
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu


def small(name, **kw):
    return make_inputs(workload(name).scaled(**kw))


def varlen_edge():
    x = small("varlen_8seq_32k", T=341, Hq=2, Hv=2, seed=18, n_varlen=6, varlen_min=1, varlen_max=200)
    lens = [1, 64, 65, 0, 130, 81]
    x["cu_seqlens"] = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    return x


def split_case():  # the trigger splits both chains; one value head does not decay
    x = small("longseq_b1_t32k_h8", T=4096 + 100, Hq=2, Hv=4, seed=46)
    x["g"][..., 1] = 0.0
    return x


def split_d64_case():  # 64-wide heads, both chains split exactly; one value head does not decay
    x = small("longseq_b1_t32k_h8", T=4096 + 100, Hq=2, Hv=4, K=64, V=64, seed=27)
    x["g"][..., 1] = 0.0
    return x


CASES = {
    "bf16_ragged": lambda: small("train_b2_t8192_h64", B=2, T=300, Hq=2, Hv=4, seed=11),
    "bf16_d64": lambda: small("train_b2_t8192_h64", B=2, T=200, Hq=2, Hv=4, K=64, V=64, seed=25),
    "bf16_k128_v64": lambda: small("train_b2_t8192_h64", B=1, T=190, Hq=1, Hv=2, K=128, V=64, seed=26),
    "bf16_varlen_edge": varlen_edge,
    "bf16_split": split_case,
    "bf16_d64_split": split_d64_case,
}


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_bwd_saved_matches_oracle_and_recompute(name, out_f32):
    """The saved pair equals the recomputing backward bit for bit (both from the CUDA forward's g_cum);
    the recomputing backward, given a host-computed g_cum, matches the oracle."""
    run_bwd_case(CASES[name](), saved=True, out_f32=out_f32)
