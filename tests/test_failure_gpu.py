"""Failure detection without a GPU fault: the library's bounded waits give up,
report through the device error word, and leave the context usable.

The self-test kernel waits on an mbarrier that nothing arrives at and on a
global flag word that nothing sets -- the two kinds of wait the tensor-core
kernels use between their roles and between CTAs -- for a short limit.
"""
import time

import numpy as np
import pytest
import torch

import mamba_ssd_chunked_02_gb300 as m2
import oracle
from mamba_ssd_chunked_02_gb300 import workloads as W
from parity import assert_close, run_fwd, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_02_gb300 import build
    build.build()
    m2.load()
    m2.device_error(clear=True)


def test_waits_run_out_report_and_leave_the_context_usable():
    t0 = time.time()
    m2.selftest_wait_timeout(limit_us=2000)
    code = m2.device_error(clear=True)
    elapsed = time.time() - t0
    assert code & m2.DEVERR_SELFTEST, code
    assert elapsed < 5.0
    assert m2.device_error(clear=True) == 0          # cleared
    # The same process keeps computing correct results afterwards.
    w = W.Workload("t b1 T768 H2 P64 N128 G1 L256 bf16", 1, 768, 2, 64, 128, 1, 256, seed=41)
    inp = W.make_inputs(w)
    y, f = run_fwd(inp, w)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=1)
    assert_close(to_np(y), yr, "bf16", "y after the self-test")
    assert_close(to_np(f), fr, "bf16", "final_state after the self-test")
