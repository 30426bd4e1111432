"""The boundary from plain C: tests/c/abi_check.c includes include/gdn.h under -std=c99 -Wall -Werror,
links libgdn.so and calls the host-only entry points; its answers must equal the Python binding's."""
import ctypes
import os
import shutil
import subprocess

import pytest

import gated_delta_rule_50_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem(K, V):
    p = gdn._Problem()
    p.B, p.T, p.Hq, p.Hv, p.K, p.V, p.n_seqs = 2, 8192, 16, 64, K, V, 2
    p.io_dtype, p.scale, p.cp_mode, p.warmup_chunks = 1, 128 ** -0.5, 0, 8
    return p


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c99_program_uses_the_abi(tmp_path):
    lib = gdn.load_library()
    libdir = os.path.dirname(gdn.library_path())
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_check.c"), "-o", str(exe), "-L", libdir, "-lgdn",
                    f"-Wl,-rpath,{libdir}"], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {line.split(" ", 1)[0]: line.split(" ", 1)[1] for line in out.strip().splitlines()}
    lib.gdn_version.restype = ctypes.c_char_p
    assert got["version"] == lib.gdn_version().decode()
    p, p64 = _problem(128, 128), _problem(64, 64)
    assert int(got["fwd_ws"]) == lib.gdn_fwd_workspace_bytes(ctypes.byref(p)) > 0
    assert int(got["bwd_ws"]) == lib.gdn_bwd_workspace_bytes(ctypes.byref(p)) > 0
    assert int(got["bwd_saved_ws"]) == lib.gdn_bwd_saved_workspace_bytes(ctypes.byref(p)) > 0
    assert int(got["fwd_ws_64"]) == lib.gdn_fwd_workspace_bytes(ctypes.byref(p64)) > 0
    assert int(got["bad_ws"]) == 0
    assert got["uses_saved"] == "1"
    assert (got["trigger_8"], got["trigger_128"]) == ("1", "0")
    assert got["plan"] == "1 23 23"
    assert got["status_ok"] == "ok"
