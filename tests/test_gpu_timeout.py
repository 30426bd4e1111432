"""Bounded device-side waits, exercised on the GPU in the permitted form: a short wait limit and a load
that the forward chain's producer skips (gdn_debug_set_wait), so that one wait can never complete.  The
kernel must give up, record GDN_ERR_TIMEOUT in the workspace error word, leave nothing in flight and
return; the next normal call on the same stream must then pass parity."""
import ctypes

import pytest
import torch

import gated_delta_rule_50_gb300 as gdn
from gpu_cases import run_fwd_case, to_dev
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu

GDN_ERR_TIMEOUT = 5


def test_expired_wait_reports_timeout_then_next_call_is_exact():
    lib = gdn.load_library()
    x = make_inputs(workload("train_b2_t8192_h64").scaled(B=2, T=300, Hq=2, Hv=4, seed=71))
    d = to_dev(x)
    ws = torch.empty(gdn.workspace_bytes("fwd", d["q"], d["v"]), dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    try:
        lib.gdn_debug_set_wait(5_000_000, 1)    # 5 ms limit; chunk 1's k / q load is never issued
        gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                       initial_state=d["h0"], workspace=ws)
        status = lib.gdn_workspace_error(ctypes.c_void_p(ws.data_ptr()), st)
    finally:
        lib.gdn_debug_set_wait(0, -1)
    assert status == GDN_ERR_TIMEOUT
    torch.cuda.synchronize()                    # the context is intact
    gdn.chunk_gated_delta_rule_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=x["scale"],
                                   initial_state=d["h0"], workspace=ws)
    assert lib.gdn_workspace_error(ctypes.c_void_p(ws.data_ptr()), st) == 0
    run_fwd_case(x)                             # and a normal call matches the oracle
