"""The single-token decode step (mamba2_ssd_decode) against the oracle's
recurrence (T = 1 from a given state), and as the continuation of a prefix
computed by the chunked whole-path call."""
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


def wl(b, H, P, N, G, dtype="bf16", seed=1, T=1):
    return W.Workload(f"d b{b} T{T} H{H} P{P} N{N} G{G} {dtype}", b, T, H, P, N, G, 64,
                      dtype=dtype, init_std=0.1, seed=seed)


DECODE = [
    wl(2, 8, 64, 128, 1, seed=51),
    wl(3, 6, 32, 256, 3, seed=52),
    wl(1, 4, 128, 16, 2, seed=53),
    wl(2, 4, 16, 64, 4, dtype="f32", seed=54),
    wl(8, 80, 64, 128, 1, seed=55),            # the 2.7B layer's heads
    wl(1, 3, 16, 128, 1, seed=57),             # staged: one CTA per head, 4 rows a warp
    wl(2, 4, 128, 256, 2, dtype="f32", seed=58),   # staged: eight CTAs per head
    wl(2, 2, 128, 128, 1, dtype="f32", seed=59),   # staged: four CTAs per head
]


@pytest.mark.parametrize("w", DECODE, ids=[w.name[2:] for w in DECODE])
def test_decode_step_matches_oracle(w):
    inp = W.make_inputs(w)                     # T = 1, initial state ~ N(0, 0.1)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    state = dev["initial_state"].clone()
    y = m2.ssd_decode(state, dev["x"][:, 0], dev["dt"][:, 0], dev["A"], dev["B"][:, 0],
                      dev["C"][:, 0], dev["D"])
    torch.cuda.synchronize()
    assert m2.device_error() == 0
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    assert_close(to_np(y), yr[:, 0], w.dtype, "decode y")
    rel, mx = assert_close(to_np(state), fr, "f32", "decode state")   # fp32 state


def test_decode_continues_a_chunked_prefix():
    """fwd over the first T0 tokens, then one decode step per remaining token:
    the same outputs as fwd over all T tokens (both within the oracle's bounds;
    compared with each other at twice the bound)."""
    w = W.Workload("c b2 T600 H4 P64 N128 G1 L256 bf16", 2, 600, 4, 64, 128, 1, 256, seed=56)
    inp = W.make_inputs(w)
    T0 = 584
    y_all, f_all = run_fwd(inp, w)
    pre = {k: (v[:, :T0].contiguous() if (v is not None and v.dim() >= 3 and k != "initial_state")
               else v) for k, v in inp.items()}
    w0 = w.scaled(seqlen=T0)
    y_pre, f_pre = run_fwd(pre, w0)
    state = f_pre.clone()
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ys = []
    for t in range(T0, w.seqlen):
        ys.append(m2.ssd_decode(state, dev["x"][:, t].contiguous(), dev["dt"][:, t].contiguous(),
                                dev["A"], dev["B"][:, t].contiguous(), dev["C"][:, t].contiguous(),
                                dev["D"]))
    torch.cuda.synchronize()
    y_dec = torch.stack(ys, dim=1)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=1)
    assert_close(to_np(y_dec), yr[:, T0:], "bf16", "decoded tail")
    assert_close(to_np(state), fr, "bf16", "decoded final state")
    d = to_np(y_dec) - to_np(y_all[:, T0:])
    rms = np.sqrt(np.mean(yr[:, T0:] ** 2))
    assert np.abs(d).max() <= 2 * 5e-2 * rms
    assert m2.device_error() == 0
