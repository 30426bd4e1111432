"""The pins are strong enough: plausible mistakes planted in copies of the
oracle's C source (a dropped factor, a flipped sign, a wrong index, a wrong
head grouping, an off-by-one sequence end) must each fail at least one pin.

The mutants are compiled to a temporary directory on the CPU; the committed
oracle is never modified.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")

MUTANTS = [
    ("fwd: prediction not decayed",
     "        p[j] = a * acc;\n        d[j] = beta * (v[j] - p[j]);",
     "        p[j] = acc;\n        d[j] = beta * (v[j] - p[j]);"),
    ("fwd: delta sign",
     "d[j] = beta * (v[j] - p[j]);", "d[j] = beta * (v[j] + p[j]);"),
    ("fwd: state not decayed",
     "S[i * V + j] = a * S[i * V + j] + k[i] * d[j];", "S[i * V + j] = S[i * V + j] + k[i] * d[j];"),
    ("fwd: scale dropped", "ot[j] = scale * acc;", "ot[j] = acc;"),
    ("fwd: interleaved head grouping",
     "int64_t seq = u / Hv, hv = u % Hv, hq = hv / G, b, t0, t1;",
     "int64_t seq = u / Hv, hv = u % Hv, hq = hv % Hq, b, t0, t1;"),
    ("varlen: sequence end off by one",
     "*t1 = s->cu[seq + 1]; }", "*t1 = s->cu[seq + 1] - 1; }"),
    ("bwd: decay missing in dk erase term", "dkt[i] += a * acc;", "dkt[i] += acc;"),
    ("bwd: dg missing factor a", "dg[ix_g(&s, b, t, hv)] = a * da;", "dg[ix_g(&s, b, t, hv)] = da;"),
    ("bwd: dS not decayed",
     "for (int64_t e = 0; e < K * V; ++e) dS[e] *= a;", "/* dS not decayed */"),
    ("bwd: dbeta sign", "dbeta[ix_g(&s, b, t, hv)] = db;", "dbeta[ix_g(&s, b, t, hv)] = -db;"),
    ("bwd: dq from the previous state",
     "acc += Scur[i * V + j] * dot[j];", "acc += Sprev[i * V + j] * dot[j];"),
    ("bwd: erase term dropped from dS",
     "for (int64_t j = 0; j < V; ++j) dS[i * V + j] += kt[i] * dp[j];", "/* dropped */"),
    ("bwd: dv missing beta", "dvt[j] = bt * dd[j];", "dvt[j] = dd[j];"),
    ("bwd: interleaved head grouping",
     "int64_t hv = hq * G + gi;", "int64_t hv = gi * Hq + hq;"),
    ("bwd: recomputed prediction not decayed",
     "                        p[j] = a * acc;\n                        d[j] = bt * (vt[j] - p[j]);",
     "                        p[j] = acc;\n                        d[j] = bt * (vt[j] - p[j]);"),
]


def _fails_a_pin(lib):
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            return pin.__name__
    return None


@pytest.mark.parametrize("name,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, orig, mut, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation site not unique/present: {orig!r}"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(orig, mut))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", str(msrc), "-o",
                    str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    caught = _fails_a_pin(lib)
    assert caught is not None, f"mutant '{name}' passed every pin"
