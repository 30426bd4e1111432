"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import gated_delta_rule_50_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return gdn.load_library()


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert "gdn_fwd" in syms and "gdn_bwd" in syms
    for s in syms:
        assert hasattr(lib, s), f"missing export {s}"


def test_status_strings_and_version(lib):
    assert lib.gdn_status_str(0) == b"ok"
    assert b"timed out" in lib.gdn_status_str(5)
    assert lib.gdn_version().startswith(b"gdn-gb300")


def _prob(**kw):
    p = gdn._Problem()
    p.B, p.T, p.Hq, p.Hv, p.K, p.V, p.n_seqs = 1, 128, 2, 4, 128, 128, 1
    p.io_dtype, p.scale, p.cp_mode, p.warmup_chunks = 1, 0.1, 0, 8
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,ok", [
    ({}, True), ({"Hv": 3}, False), ({"K": 96}, False), ({"io_dtype": 7}, False),
    ({"n_seqs": 2}, False), ({"cp_mode": 9}, False), ({"cp_mode": 2, "warmup_chunks": 0}, False),
    ({"T": 0}, True), ({"B": 0}, False)])
def test_workspace_bytes_validation(lib, kw, ok):
    n = lib.gdn_fwd_workspace_bytes(ctypes.byref(_prob(**kw)))
    assert (n > 0) == ok


# Argument checks that hand the library placeholder addresses run in a child process that sees no GPU
# (CUDA_VISIBLE_DEVICES=""): the statuses asserted come from host validation, and even a regression in the
# validation order could not launch a kernel on a fabricated address.
_NO_GPU_CHECKS = r"""
import ctypes, sys
sys.path.insert(0, ROOT)
import gated_delta_rule_50_gb300 as gdn
lib = gdn.load_library()
P = ctypes.c_void_p
def prob(**kw):
    p = gdn._Problem()
    p.B, p.T, p.Hq, p.Hv, p.K, p.V, p.n_seqs = 1, 128, 2, 4, 128, 128, 1
    p.io_dtype, p.scale, p.cp_mode, p.warmup_chunks = 1, 0.1, 0, 8
    for k, v in kw.items():
        setattr(p, k, v)
    return p
out = {}
# varlen: the host copy of the offsets is validated (the device pointer is never read on this path)
cu = (ctypes.c_int32 * 3)(0, 100, 128)
bad = (ctypes.c_int32 * 3)(0, 100, 120)
p = prob(n_seqs=2, cu_seqlens=P(256), cu_seqlens_host=ctypes.cast(cu, P))
out["varlen_ok"] = lib.gdn_fwd_workspace_bytes(ctypes.byref(p)) > 0
p.cu_seqlens_host = ctypes.cast(bad, P)
out["varlen_bad_end"] = lib.gdn_fwd_workspace_bytes(ctypes.byref(p))
p.cu_seqlens_host = None
out["varlen_no_host"] = lib.gdn_fwd_workspace_bytes(ctypes.byref(p))
p = prob()
out["null_q"] = lib.gdn_fwd(ctypes.byref(p), None, P(256), P(256), P(256), P(256), None, P(256), None, None,
                            None, None, P(256), 1 << 40, None)
out["misaligned"] = lib.gdn_fwd(ctypes.byref(p), P(257), P(256), P(256), P(256), P(256), None, P(256), None,
                                None, None, None, P(256), 1 << 40, None)
out["small_ws"] = lib.gdn_fwd(ctypes.byref(p), P(256), P(256), P(256), P(256), P(256), None, P(256), None, None,
                              None, None, P(256), 16, None)
out["bwd_h0_dh0"] = lib.gdn_bwd(ctypes.byref(p), *([P(256)] * 5), None, P(256), None, P(256), *([P(256)] * 5),
                                None, P(256), 1 << 40, None)
out["out_f32_bad"] = lib.gdn_fwd_workspace_bytes(ctypes.byref(prob(out_f32=2)))
# the no-alloc forward answers an invalid or unsupported problem with gdn_fwd's own status
for name, kw in (("k96", {"K": 96}), ("hv3", {"Hv": 3})):
    q = prob(**kw)
    out["noalloc_" + name] = lib.gdn_fwd_noalloc(ctypes.byref(q), *([None] * 11), None)
    out["fwd_" + name] = lib.gdn_fwd(ctypes.byref(q), *([None] * 11), None, 0, None)
print(repr(out))
"""


def _no_gpu_results():
    import ast
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + _NO_GPU_CHECKS], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return ast.literal_eval(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def no_gpu():
    return _no_gpu_results()


def test_varlen_host_offsets_validated(no_gpu):
    assert no_gpu["varlen_ok"]
    assert no_gpu["varlen_bad_end"] == 0      # does not end at T
    assert no_gpu["varlen_no_host"] == 0      # the host copy is required


def test_bad_pointers_rejected_without_launch(no_gpu):
    assert no_gpu["null_q"] == 1              # null q: rejected on the host
    assert no_gpu["misaligned"] == 1          # misaligned pointer
    assert no_gpu["small_ws"] == 3            # workspace too small
    assert no_gpu["bwd_h0_dh0"] == 1          # dh0 must be given iff h0 is
    assert no_gpu["out_f32_bad"] == 0         # out_f32 is 0 or 1


def test_noalloc_status_matches_gdn_fwd(no_gpu):
    assert no_gpu["noalloc_k96"] == no_gpu["fwd_k96"] == 2
    assert no_gpu["noalloc_hv3"] == no_gpu["fwd_hv3"] == 1


def test_python_api_names_match_pages():
    import json
    c = json.load(open(os.path.join(ROOT, "tests", "golden", "api_contract.json")))
    import inspect
    for key in ("high_level", "low_level_fwd", "low_level_bwd"):
        fn = getattr(gdn, c[key]["name"])
        params = list(inspect.signature(fn).parameters)
        assert params[:len(c[key]["args"])] == c[key]["args"], (key, params)


def test_no_cpu_path():
    import torch
    x = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ValueError):
        gdn.chunk_gated_delta_rule_fwd(x, x, x, torch.zeros(1, 64, 1), torch.zeros(1, 64, 1))


def test_cp_trigger_matches_pages_rule(lib):
    import json
    rule = json.load(open(os.path.join(ROOT, "tests", "golden", "autocp_rule.json")))
    lib.gdn_cp_trigger.argtypes = [ctypes.c_int64] * 3
    lib.gdn_cp_trigger.restype = ctypes.c_int
    for c in rule["cases"]:
        assert lib.gdn_cp_trigger(1, c["bh"], c["seq_len"]) == int(c["on"]), c
        assert lib.gdn_cp_trigger(c["bh"], 1, c["seq_len"]) == int(c["on"]), c


def test_cp_plan_geometry(lib):
    lib.gdn_cp_plan.argtypes = [ctypes.POINTER(gdn._Problem), ctypes.POINTER(ctypes.c_int),
                                ctypes.POINTER(ctypes.c_int)]
    lib.gdn_cp_plan.restype = ctypes.c_int
    L, n = ctypes.c_int(), ctypes.c_int()
    # small-head long sequence: 512 chunks -> L = round(sqrt(512)) = 23, 23 segments
    p = _prob(B=1, T=32768, Hq=4, Hv=8, n_seqs=1, cp_mode=2, warmup_chunks=6)
    assert lib.gdn_cp_plan(ctypes.byref(p), ctypes.byref(L), ctypes.byref(n)) == 1
    assert (L.value, n.value) == (23, 23)
    assert lib.gdn_fwd_workspace_bytes(ctypes.byref(p)) > 8 * 23 * 128 * 128 * 4
    # the default (exact) mode splits through segment transitions
    p.cp_mode = 0
    assert lib.gdn_cp_plan(ctypes.byref(p), ctypes.byref(L), ctypes.byref(n)) == 1
    assert (L.value, n.value) == (23, 23)
    # no splitting when turned off, or with a batch x heads product above the rule
    p.cp_mode = 1
    assert lib.gdn_cp_plan(ctypes.byref(p), ctypes.byref(L), ctypes.byref(n)) == 0
    p = _prob(B=2, T=8192, Hq=16, Hv=64, n_seqs=2, cp_mode=2)
    assert lib.gdn_cp_plan(ctypes.byref(p), ctypes.byref(L), ctypes.byref(n)) == 0


def test_head64_padded_planning(lib):
    """64-wide bf16 heads plan onto the 128-wide tensor-core path: the same sequence split as a 128-wide
    problem, a workspace that holds the padded copies on top of the 128-wide one, and a saved backward
    that reads the forward's states; fp32 problems recompute instead."""
    lib.gdn_cp_plan.argtypes = [ctypes.POINTER(gdn._Problem), ctypes.POINTER(ctypes.c_int),
                                ctypes.POINTER(ctypes.c_int)]
    lib.gdn_cp_plan.restype = ctypes.c_int
    lib.gdn_bwd_saved_uses_saved.argtypes = [ctypes.POINTER(gdn._Problem)]
    lib.gdn_bwd_saved_uses_saved.restype = ctypes.c_int
    L, n = ctypes.c_int(), ctypes.c_int()
    p64 = _prob(B=1, T=32768, Hq=4, Hv=8, n_seqs=1, K=64, V=64)
    p128 = _prob(B=1, T=32768, Hq=4, Hv=8, n_seqs=1)
    assert lib.gdn_cp_plan(ctypes.byref(p64), ctypes.byref(L), ctypes.byref(n)) == 1
    assert (L.value, n.value) == (23, 23)
    tokens, state = 32768, 128 * 128 * 4
    for fn in (lib.gdn_fwd_workspace_bytes, lib.gdn_bwd_workspace_bytes, lib.gdn_bwd_saved_workspace_bytes):
        w64, w128 = fn(ctypes.byref(p64)), fn(ctypes.byref(p128))
        assert w64 > w128 + tokens * 4 * 128 * 2  # at least the padded q (or the padded dq)
    # forward: padded q, k, v, o, h0, ht and per-chunk states beside the 128-wide workspace
    extra = lib.gdn_fwd_workspace_bytes(ctypes.byref(p64)) - lib.gdn_fwd_workspace_bytes(ctypes.byref(p128))
    assert extra >= tokens * (2 * 4 + 2 * 8) * 128 * 2 + (2 * 8 + 512 * 8) * state
    assert lib.gdn_bwd_saved_uses_saved(ctypes.byref(p64)) == 1
    assert lib.gdn_bwd_saved_uses_saved(ctypes.byref(p128)) == 1
    assert lib.gdn_bwd_saved_uses_saved(ctypes.byref(_prob(io_dtype=0, K=64, V=64))) == 0
    assert lib.gdn_bwd_saved_uses_saved(ctypes.byref(_prob(T=0))) == 0
    assert lib.gdn_bwd_saved_uses_saved(ctypes.byref(_prob(Hv=3))) == -1
    # fp32 with 64-wide heads stays on the CUDA-core path: no padded copies in its workspace
    f64 = _prob(B=1, T=32768, Hq=4, Hv=8, n_seqs=1, K=64, V=64, io_dtype=0)
    assert lib.gdn_fwd_workspace_bytes(ctypes.byref(f64)) < lib.gdn_fwd_workspace_bytes(ctypes.byref(p64))
