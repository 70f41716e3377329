"""The oracle reproduces its committed regression fixture (tests/golden/oracle_tiny.txt)."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def _read(path):
    out = {}
    with open(path) as fh:
        lines = [ln.strip() for ln in fh if ln.strip() and not ln.startswith("#")]
    i = 0
    while i < len(lines):
        name, *shape = lines[i].split()
        shape = tuple(int(s) for s in shape)
        n = int(np.prod(shape))
        out[name] = np.array([float(v) for v in lines[i + 1:i + 1 + n]]).reshape(shape)
        i += 1 + n
    return out


def test_oracle_matches_golden():
    ref = _read(os.path.join(HERE, "golden", "oracle_tiny.txt"))
    y, f = make_golden.compute()
    assert np.allclose(y, ref["y"], rtol=1e-13, atol=1e-15)
    assert np.allclose(f, ref["final_state"], rtol=1e-13, atol=1e-15)
