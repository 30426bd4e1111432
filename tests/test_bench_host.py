"""Host-side helpers of the benchmark that need no GPU: the sysfs CPU-list parser and the placement of
the end-to-end leg's pinned buffers near the GPU (its four outcomes, with nvidia-smi, sysfs and the
affinity calls replaced by fakes)."""
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
