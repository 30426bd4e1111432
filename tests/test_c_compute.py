"""The compute entry points from plain C: tests/c/run_fwd_bwd.c (C99, -Wall -Werror) allocates device
buffers with the CUDA runtime, runs gdn_fwd and gdn_bwd through include/gdn.h on a tiny bf16 problem and
writes its outputs back; they are checked here against the fp64 oracle at the parity tolerances."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import gated_delta_rule_50_gb300 as gdn
import oracle
from gpu_cases import host_gcum, recovered_gate
from parity import check
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _raw(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().tobytes()
    return t.float().numpy().tobytes()


def _read(path, shape, dtype):
    data = np.fromfile(path, dtype=np.int16 if dtype == torch.bfloat16 else np.float32)
    t = torch.from_numpy(data.copy())
    if dtype == torch.bfloat16:
        t = t.view(torch.bfloat16)
    return t.reshape(shape)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c99_program_runs_fwd_and_bwd(tmp_path):
    gdn.load_library()
    libdir = os.path.dirname(gdn.library_path())
    exe = tmp_path / "run_fwd_bwd"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "run_fwd_bwd.c"),
                        "-o", str(exe), "-L", libdir, "-lgdn", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                        "-lm", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    B, T, Hq, Hv, K, V = 2, 200, 2, 4, 128, 128
    x = make_inputs(workload("train_b2_t8192_h64").scaled(B=B, T=T, Hq=Hq, Hv=Hv, seed=61))
    g_cum = host_gcum(x["g"])
    for name in ("q", "k", "v", "g", "beta", "h0", "do", "dht"):
        (tmp_path / f"{name}.bin").write_bytes(_raw(x[name]))
    (tmp_path / "g_cum.bin").write_bytes(_raw(g_cum))
    r = subprocess.run([str(exe), str(tmp_path), *map(str, (B, T, Hq, Hv, K, V))], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
    io = torch.bfloat16
    o = _read(tmp_path / "o.bin", (B, T, Hv, V), io)
    ht = _read(tmp_path / "ht.bin", (B, Hv, K, V), torch.float32)
    o_ref, ht_ref = oracle.oracle_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"])
    check("o", o, o_ref, io, io)
    check("final_state", ht, ht_ref, io, torch.float32)
    grads = [_read(tmp_path / f"{n}.bin", s, dt) for n, s, dt in
             (("dq", (B, T, Hq, K), io), ("dk", (B, T, Hq, K), io), ("dv", (B, T, Hv, V), io),
              ("dbeta", (B, T, Hv), torch.float32), ("dg", (B, T, Hv), torch.float32),
              ("dh0", (B, Hv, K, V), torch.float32))]
    g_rec = torch.from_numpy(recovered_gate(g_cum))
    ref = oracle.oracle_bwd(x["q"], x["k"], x["v"], g_rec, x["beta"], x["do"], x["scale"], x["h0"], x["dht"])
    for name, got, want, st in zip(["dq", "dk", "dv", "dbeta", "dg", "dh0"], grads, ref,
                                   [io, io, io, torch.float32, torch.float32, torch.float32]):
        check(name, got, want, io, st)
