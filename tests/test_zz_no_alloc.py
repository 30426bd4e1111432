"""gdn_fwd_noalloc: the forward for callers that cannot allocate device memory
(runtimes that own all device allocations, frozen graph memory pools, C hosts
without an allocator).  Called through the C ABI; its results must match
gdn_fwd's on the same inputs, on two calls in a row (the shared static scratch
must not carry anything from one call into the next).  Kept in its own file
so that it is collected last."""
import ctypes

import pytest
import torch

import gated_delta_rule_50_gb300 as gdn
from parity import check
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _ptr(t):
    return None if t is None else P(t.data_ptr())


def _noalloc_fwd(lib, x, d):
    B, T, Hq, K = d["q"].shape
    Hv, V = d["v"].shape[2], d["v"].shape[3]
    pr = gdn._problem(d["q"], d["v"], x["scale"], None, None, "auto", 8)
    nc = B * ((T + 63) // 64)
    o = torch.empty(B, T, Hv, V, dtype=d["q"].dtype, device="cuda")
    g_cum = torch.empty(B, T, Hv, dtype=torch.float32, device="cuda")
    A = torch.empty(B, T, Hv, 64, dtype=d["q"].dtype, device="cuda")
    h = torch.empty(nc, Hv, K, V, dtype=torch.float32, device="cuda")
    ht = torch.empty(B, Hv, K, V, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.gdn_fwd_noalloc(ctypes.byref(pr), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g"]),
                             _ptr(d["beta"]), _ptr(d["h0"]), _ptr(o), _ptr(g_cum), _ptr(A), _ptr(h), _ptr(ht),
                             P(st))
    return rc, (g_cum, A, o, h.view(B, nc // B, Hv, K, V), ht)


@pytest.fixture(scope="module")
def lib():
    lib = gdn.load_library()
    lib.gdn_fwd_noalloc.argtypes = [ctypes.POINTER(gdn._Problem)] + [P] * 11 + [P]
    lib.gdn_fwd_noalloc.restype = ctypes.c_int
    return lib


def test_noalloc_matches_gdn_fwd_twice(lib):
    for seed in (31, 32):   # two calls in a row on different inputs
        x = make_inputs(workload("train_b2_t8192_h64").scaled(B=2, T=300, Hq=2, Hv=4, seed=seed))
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
        rc, got = _noalloc_fwd(lib, x, d)
        assert rc == 0, lib.gdn_status_str(rc)
        ref = gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                             initial_state=d["h0"], output_h=True)
        torch.cuda.synchronize()
        io = x["q"].dtype
        for name, a, b, st in zip(["g_cum", "A", "o", "h", "final_state"], got, ref,
                                  [torch.float32, io, io, torch.float32, torch.float32]):
            check(name, a, b, io, st)


def test_noalloc_rejects_oversize_problem(lib):
    x = make_inputs(workload("train_b2_t8192_h64").scaled(B=1, T=64, Hq=1, Hv=1, seed=33))
    pr = gdn._Problem()
    pr.B, pr.T, pr.Hq, pr.Hv, pr.K, pr.V, pr.n_seqs = 4, 8192, 16, 64, 128, 128, 4
    # fp32 io runs the CUDA-core path, whose forward scratch (fp32 A, P per chunk) is large
    pr.io_dtype, pr.scale, pr.cp_mode, pr.warmup_chunks = 0, 0.088, 0, 8
    assert lib.gdn_fwd_workspace_bytes(ctypes.byref(pr)) > (32 << 20)
    dummy = P(256)
    rc = lib.gdn_fwd_noalloc(ctypes.byref(pr), *([dummy] * 5), None, dummy, None, None, None, None, None)
    assert rc == 6 and b"no-alloc" in lib.gdn_status_str(6)
