"""gdn_fwd_noalloc: the forward for callers that cannot allocate device memory
(runtimes that own all device allocations, frozen graph memory pools, C hosts
without an allocator).  Called through the C ABI; it runs the same kernels as
gdn_fwd on the same inputs, so its outputs must equal gdn_fwd's bit for bit,
call after call: a larger call of another shape (64-wide heads, more heads and
chunks) runs first, so that a scratch byte the forward read without writing it
would carry that call's values into the next.  Kept in its own file so that it
is collected last."""
import ctypes

import pytest
import torch

import gated_delta_rule_50_gb300 as gdn
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _ptr(t):
    return None if t is None else P(t.data_ptr())


def _outputs(d, nc):
    B, T, Hq, K = d["q"].shape
    Hv, V = d["v"].shape[2], d["v"].shape[3]
    return (torch.empty(B, T, Hv, dtype=torch.float32, device="cuda"),
            torch.empty(B, T, Hv, 64, dtype=d["q"].dtype, device="cuda"),
            torch.empty(B, T, Hv, V, dtype=d["q"].dtype, device="cuda"),
            torch.empty(nc, Hv, K, V, dtype=torch.float32, device="cuda"),
            torch.empty(B, Hv, K, V, dtype=torch.float32, device="cuda"))


def _noalloc_fwd(lib, x, d):
    B, T = d["q"].shape[:2]
    pr = gdn._problem(d["q"], d["v"], x["scale"], None, None, "auto", 8)
    nc = B * ((T + 63) // 64)
    g_cum, A, o, h, ht = _outputs(d, nc)
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.gdn_fwd_noalloc(ctypes.byref(pr), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g"]),
                             _ptr(d["beta"]), _ptr(d["h0"]), _ptr(o), _ptr(g_cum), _ptr(A), _ptr(h), _ptr(ht),
                             P(st))
    return rc, (g_cum, A, o, h.view(B, nc // B, *h.shape[1:]), ht)


@pytest.fixture(scope="module")
def lib():
    return gdn.load_library()


def test_noalloc_matches_gdn_fwd_call_after_call(lib):
    cases = [dict(B=1, T=900, Hq=2, Hv=8, K=64, V=64, seed=30),    # larger, other shape, padded path
             dict(B=2, T=300, Hq=2, Hv=4, seed=31),                  # then the small problem, twice
             dict(B=2, T=300, Hq=2, Hv=4, seed=32)]
    for kw in cases:
        x = make_inputs(workload("train_b2_t8192_h64").scaled(**kw))
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        assert lib.gdn_fwd_workspace_bytes(ctypes.byref(gdn._problem(d["q"], d["v"], x["scale"], None, None,
                                                                     "auto", 8))) <= (32 << 20)
        rc, got = _noalloc_fwd(lib, x, d)
        assert rc == 0, lib.gdn_status_str(rc)
        ref = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                             initial_state=d["h0"], output_h=True)
        torch.cuda.synchronize()
        for name, a, b in zip(["g_cum", "A", "o", "h", "final_state"], got, ref):
            assert torch.equal(a, b), (kw, name)
        assert lib.gdn_fwd_noalloc_error(P(torch.cuda.current_stream().cuda_stream)) == 0


def test_noalloc_rejects_oversize_problem(lib):
    pr = gdn._Problem()
    pr.B, pr.T, pr.Hq, pr.Hv, pr.K, pr.V, pr.n_seqs = 4, 8192, 16, 64, 128, 128, 4
    pr.io_dtype, pr.scale, pr.cp_mode, pr.warmup_chunks = 1, 0.088, 0, 8
    assert lib.gdn_fwd_workspace_bytes(ctypes.byref(pr)) > (32 << 20)
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")   # real (small) device buffers
    a = _ptr(buf)
    rc = lib.gdn_fwd_noalloc(ctypes.byref(pr), a, a, a, a, a, None, a, None, None, None, None,
                             P(torch.cuda.current_stream().cuda_stream))
    assert rc == 6 and b"no-alloc" in lib.gdn_status_str(6)
