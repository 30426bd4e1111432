"""Host-side parts of the benchmark that need no GPU: the sysfs CPU-list parser, the placement of
the end-to-end leg's pinned buffers near the GPU (its four outcomes, with nvidia-smi, sysfs and the
affinity calls replaced by fakes), and the roofline accounting: the algorithmic work per token and value
head, the kernels' shares of it, and the DRAM traffic figure tied to the kernel source it was taken on."""
import io
import types

import pytest

import bench


def test_cpulist_ranges_and_singles():
    assert bench._cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("") == set()


class _Fakes:
    def __init__(self, monkeypatch, local, allowed, bus="00000009:01:00.0", fail=False):
        self.set_calls = []
        self.paths = []

        def run(cmd, **kw):
            if fail:
                raise FileNotFoundError("nvidia-smi")
            return types.SimpleNamespace(stdout=bus + "\n")

        def fake_open(path, *a, **kw):
            self.paths.append(path)
            return io.StringIO(local)

        monkeypatch.setattr(bench.subprocess, "run", run)
        monkeypatch.setattr(bench, "open", fake_open, raising=False)
        monkeypatch.setattr(bench.os, "sched_getaffinity", lambda pid: set(allowed))
        monkeypatch.setattr(bench.os, "sched_setaffinity", lambda pid, cpus: self.set_calls.append(set(cpus)))


DEV = types.SimpleNamespace(index=0)


def test_bind_restricts_to_local_cpus(monkeypatch):
    f = _Fakes(monkeypatch, local="0-3", allowed=range(8))
    old, where = bench.bind_near_gpu(DEV)
    assert where == "bound" and old == set(range(8)) and f.set_calls == [{0, 1, 2, 3}]
    assert f.paths == ["/sys/bus/pci/devices/0009:01:00.0/local_cpulist"]


def test_bind_reports_already_local(monkeypatch):
    f = _Fakes(monkeypatch, local="0-15", allowed=range(16))
    assert bench.bind_near_gpu(DEV) == (None, "local") and f.set_calls == []


def test_bind_reports_no_local_cpu(monkeypatch):
    f = _Fakes(monkeypatch, local="16-31", allowed=range(16))
    assert bench.bind_near_gpu(DEV) == (None, "none local") and f.set_calls == []


@pytest.mark.parametrize("fail", [True, False])
def test_bind_unknown_without_locality(monkeypatch, fail):
    # nvidia-smi missing, or a bus id that does not parse
    f = _Fakes(monkeypatch, local="0-3", allowed=range(8), bus="garbage", fail=fail)
    assert bench.bind_near_gpu(DEV) == (None, "unknown") and f.set_calls == []


# ---------------------------------------------------------------- roofline accounting
def _train_workload():
    from synth import workload
    return workload("train_b2_t8192_h64")


def test_algorithmic_per_token_head_figures():
    """K = V = 128, C = 64, bf16, G = 4: forward 180,224 flops and 652 + 512 / G bytes, backward 507,904
    flops and 912 + 1024 / G bytes per token and value head, plus the fp32 states per (sequence, head)."""
    w = _train_workload()
    assert (w.K, w.V, w.Hv // w.Hq) == (128, 128, 4)
    alg = bench.algorithmic(w)
    th = w.tokens * w.Hv
    units, st = w.n_seqs * w.Hv, 4 * 128 * 128
    assert alg["fwd_flops"] == th * 180224
    assert alg["bwd_flops"] == th * 507904
    assert alg["fwd_bytes"] == th * (652 + 512 / 4) + units * st * 2              # h0 in, final state out
    assert alg["bwd_bytes"] == th * (912 + 1024 / 4) + units * st * 3             # h0, dht in, dh0 out


def test_kernel_shares_add_up_to_the_passes():
    w = _train_workload()
    alg = bench.algorithmic(w)
    kw = {n: bench.kernel_work(n, w) for n in ("fwd_prep_tc", "fwd_tc", "bwd_prep_tc", "bwd_state_tc",
                                               "bwd_dscan_tc", "bwd_intra_tc")}
    assert kw["fwd_prep_tc"][0] + kw["fwd_tc"][0] == alg["fwd_flops"]
    assert kw["fwd_prep_tc"][1] + kw["fwd_tc"][1] == alg["fwd_bytes"]
    assert sum(kw[n][0] for n in ("bwd_prep_tc", "bwd_state_tc", "bwd_dscan_tc", "bwd_intra_tc")) \
        == alg["bwd_flops"]
    # the gradient kernel's bytes: q, k, dq, dk once per group, v, do, dv, four fp32 vectors
    th = w.tokens * w.Hv
    assert kw["bwd_intra_tc"][1] == th * (4 * 128 * 2 / 4 + 3 * 128 * 2 + 16) == 1090519040
    assert bench.kernel_work("no_such_kernel", w) is None


def test_traffic_tied_to_the_kernel_source(monkeypatch):
    name = "bwd_intra_tc"
    value, sha = bench.TRAFFIC[name]
    assert len(bench.source_sha16(name)) == 16
    monkeypatch.setattr(bench, "source_sha16", lambda k: sha)      # the source the counters were taken on
    assert bench.traffic_bytes(name) == value
    monkeypatch.setattr(bench, "source_sha16", lambda k: "0" * 16)  # any other version: not reported
    assert bench.traffic_bytes(name) is None
    assert bench.traffic_bytes("fwd_tc") is None
