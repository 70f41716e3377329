"""Write tests/golden/oracle_tiny.txt: oracle outputs for one tiny seeded case.

Calls only the oracle (oracle/) and the seeded input generator.  The fixture is
a regression guard: a later change to the oracle's arithmetic must reproduce it
(tests/test_golden.py) or regenerate it with a commit message that names the
passage of the pages justifying the change.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from mamba_ssd_chunked_02_gb300.workloads import Workload, make_inputs  # noqa: E402

CASE = Workload("golden tiny b1 T20 H2 P4 N3 G1 L8 f32 init", 1, 20, 2, 4, 3, 1, 8,
                dtype="f32", dt_lo=1e-2, dt_hi=0.5, init_std=0.1, seed=4242)


def compute():
    inp = make_inputs(CASE)
    y, f = oracle.ssd_recurrent(**inp, ngroups=CASE.ngroups)
    return y, f


def main():
    y, f = compute()
    path = os.path.join(HERE, "oracle_tiny.txt")
    with open(path, "w") as fh:
        fh.write(f"# {CASE.name}, seed {CASE.seed}; written by tests/golden/make_golden.py\n")
        fh.write("# recurrence of the Mamba-2 SSD forward, fp64 oracle (oracle/ssd_oracle.c)\n")
        fh.write("y " + " ".join(str(v) for v in y.shape) + "\n")
        fh.write("\n".join(repr(float(v)) for v in y.ravel()) + "\n")
        fh.write("final_state " + " ".join(str(v) for v in f.shape) + "\n")
        fh.write("\n".join(repr(float(v)) for v in f.ravel()) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
