"""Seeded synthetic inputs for the gated delta rule chunked-prefill operator.

This module is shared by the oracle tests, the CUDA parity tests, ``smoke()``
and ``bench.py``.  It holds input *distributions* only and none of the
operator's arithmetic: no recurrence, no chunking, no gate cumsum.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
in a fixed order (q, k, v, g, beta, h0, do, dht, then per-workload extras), so
the GPU path and the oracle receive bit-identical values.  The recipes follow
the five workloads of the operator's test plan (the FlashQLA project page,
"Usage / High-level API" lists the tensor shapes):

* q, k  ~ N(0, 1), L2-normalised per head vector in fp32, then cast to the io
  dtype.
* v     ~ N(0, 1).
* g     = -softplus(N(shift, 1)) (log-decay <= 0); shift = 1 for the
  small-head long-sequence workload, 0 otherwise.
* beta  = sigmoid(N(0, 1)).
* h0    = 0.1 * N(0, 1) (fp32), one state per sequence.
* do    ~ N(0, 1) (io dtype), dht = 0.1 * N(0, 1) (fp32).
* varlen: 8 sequence lengths uniform in [512, 8192], rescaled to sum to
  exactly 32768 tokens, packed as B = 1.
* training-shaped workload: 10 % of the v-heads (the first round(0.1 * H_v)
  entries of a seeded permutation) get g = 0 exactly (no decay).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "varlen_lengths"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int            # tokens per sequence (total tokens when varlen)
    Hq: int
    Hv: int
    K: int
    V: int
    io_dtype: torch.dtype
    seed: int
    has_h0: bool
    has_dht: bool
    bwd: bool
    g_shift: float = 0.0
    zero_g_frac: float = 0.0
    n_varlen: int = 0          # > 0: packed varlen with this many sequences (B == 1)
    varlen_min: int = 512
    varlen_max: int = 8192

    @property
    def n_seqs(self) -> int:
        return self.n_varlen if self.n_varlen else self.B

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (used for small parity cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny fp32 fwd+bwd, parity at 1e-5
    "tiny_fp32": Workload("tiny_fp32", B=1, T=256, Hq=2, Hv=2, K=64, V=64,
                          io_dtype=torch.float32, seed=0, has_h0=True, has_dht=True, bwd=True),
    # forward prefill, bf16, G = 2, no initial state
    "prefill_b4_t4096": Workload("prefill_b4_t4096", B=4, T=4096, Hq=16, Hv=32, K=128, V=128,
                                 io_dtype=torch.bfloat16, seed=1, has_h0=False, has_dht=False,
                                 bwd=False),
    # packed varlen fwd+bwd, 8 sequences, 32768 tokens, G = 1
    "varlen_8seq_32k": Workload("varlen_8seq_32k", B=1, T=32768, Hq=16, Hv=16, K=128, V=128,
                                io_dtype=torch.bfloat16, seed=2, has_h0=True, has_dht=True,
                                bwd=True, n_varlen=8),
    # small head count, long sequence (sequence-parallel trigger applies), strong decay
    "longseq_b1_t32k_h8": Workload("longseq_b1_t32k_h8", B=1, T=32768, Hq=4, Hv=8, K=128, V=128,
                                   io_dtype=torch.bfloat16, seed=3, has_h0=True, has_dht=True,
                                   bwd=True, g_shift=1.0),
    # training-shaped fwd+bwd, G = 4, 10 % of heads without decay
    "train_b2_t8192_h64": Workload("train_b2_t8192_h64", B=2, T=8192, Hq=16, Hv=64, K=128, V=128,
                                   io_dtype=torch.bfloat16, seed=4, has_h0=True, has_dht=True,
                                   bwd=True, zero_g_frac=0.1),
    # half of the training shape (same heads and distributions) for hardware-counter captures: its
    # inputs still exceed the 129 MB L2 while the device footprint stays near 1 GB
    "train_b1_t4096_h64": Workload("train_b1_t4096_h64", B=1, T=4096, Hq=16, Hv=64, K=128, V=128,
                                   io_dtype=torch.bfloat16, seed=5, has_h0=True, has_dht=True,
                                   bwd=True, zero_g_frac=0.1),
}
# positional order matches the workload list of the operator's test plan
WORKLOAD_ORDER = ["tiny_fp32", "prefill_b4_t4096", "varlen_8seq_32k",
                  "longseq_b1_t32k_h8", "train_b2_t8192_h64"]


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[WORKLOAD_ORDER[name_or_index]]
    return WORKLOADS[name_or_index]


def varlen_lengths(n: int, total: int, lo: int, hi: int, seed: int) -> list[int]:
    """n lengths drawn uniformly in [lo, hi], rescaled to sum to ``total``.

    The rounding remainder goes to the last sequence; if any length leaves
    [lo, hi] the draw is repeated with seed + 100.
    """
    s = seed
    for _ in range(64):
        gen = torch.Generator().manual_seed(s)
        raw = torch.randint(lo, hi + 1, (n,), generator=gen).double()
        lens = [int(math.floor(x)) for x in (raw * (total / raw.sum())).tolist()]
        lens[-1] += total - sum(lens)
        if all(lo <= x <= hi for x in lens):
            return lens
        s += 100
    raise RuntimeError("could not draw varlen lengths")


def _l2norm(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_inputs(w: Workload, *, scale: Optional[float] = None) -> dict:
    """Draw all CPU tensors of workload ``w`` (see the module docstring).

    Returns a dict with q, k, v (io dtype), g, beta (fp32), h0 (fp32 or None),
    do (io dtype), dht (fp32 or None), cu_seqlens (int32 or None), scale.
    """
    gen = torch.Generator().manual_seed(w.seed)
    B, T, Hq, Hv, K, V = w.B, w.T, w.Hq, w.Hv, w.K, w.V
    q = _l2norm(torch.randn(B, T, Hq, K, generator=gen)).to(w.io_dtype)
    k = _l2norm(torch.randn(B, T, Hq, K, generator=gen)).to(w.io_dtype)
    v = torch.randn(B, T, Hv, V, generator=gen).to(w.io_dtype)
    g = -torch.nn.functional.softplus(torch.randn(B, T, Hv, generator=gen) + w.g_shift)
    beta = torch.sigmoid(torch.randn(B, T, Hv, generator=gen))
    h0 = 0.1 * torch.randn(w.n_seqs, Hv, K, V, generator=gen)
    do = torch.randn(B, T, Hv, V, generator=gen).to(w.io_dtype)
    dht = 0.1 * torch.randn(w.n_seqs, Hv, K, V, generator=gen)
    if w.zero_g_frac > 0:
        n0 = int(round(w.zero_g_frac * Hv))
        heads = torch.randperm(Hv, generator=gen)[:n0]
        g[:, :, heads] = 0.0
    cu = None
    if w.n_varlen:
        assert B == 1
        lens = varlen_lengths(w.n_varlen, T, w.varlen_min, w.varlen_max, w.seed)
        cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(), g=g.contiguous().float(),
                beta=beta.contiguous().float(),
                h0=h0.contiguous() if w.has_h0 else None,
                do=do.contiguous(),
                dht=dht.contiguous() if w.has_dht else None,
                cu_seqlens=cu,
                scale=(K ** -0.5) if scale is None else scale)
