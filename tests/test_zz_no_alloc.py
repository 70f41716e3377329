"""The allocation-free entry point mamba2_ssd_fwd_noalloc.

It serves callers that cannot allocate device memory (a host framework that
owns all allocations, a plug-in that may not call the CUDA allocator): the
workspace is a fixed 64 MiB device array inside the library.  Through the
C ABI, two calls in a row (with different inputs, so that stale contents of
the shared scratch would show) must match the ordinary entry point
mamba2_ssd_fwd within the parity tolerance; an oversize shape is rejected.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import mamba_ssd_chunked_02_gb300 as m2
from mamba_ssd_chunked_02_gb300 import workloads as W
from parity import assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_02_gb300 import build
    build.build()
    m2.load()
    m2.device_error(clear=True)


def _call_noalloc(lib, sh, dev, y, f):
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.mamba2_ssd_fwd_noalloc(ctypes.byref(sh), p(dev["x"]), p(dev["dt"]), p(dev["A"]),
                                      p(dev["B"]), p(dev["C"]), p(dev["D"]),
                                      p(dev["initial_state"]), p(y), p(f), stream)


@pytest.mark.parametrize("w", [
    W.Workload("noalloc bf16", 1, 1024, 16, 64, 128, 1, 256, seed=501),
    W.Workload("noalloc bf16 ragged grouped init", 2, 700, 8, 64, 64, 2, 128, init_std=0.1,
               seed=502),
    W.Workload("noalloc fp32", 1, 256, 2, 16, 16, 1, 64, dtype="f32", seed=503),
], ids=lambda w: w.name)
def test_noalloc_matches_fwd_on_two_calls(w):
    lib = m2.load()
    sh = None
    for call in range(2):
        inp = W.make_inputs(w.scaled(seed=w.seed + 1000 * call))
        dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
        assert m2.workspace_size(sh) <= m2.NOALLOC_SCRATCH_BYTES
        y_ref, f_ref = m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                                  dev["initial_state"], chunk_size=w.chunk_size,
                                  ngroups=w.ngroups)
        y = torch.full_like(y_ref, float("nan"))
        f = torch.full_like(f_ref, float("nan"))
        assert _call_noalloc(lib, sh, dev, y, f) == m2.OK
        torch.cuda.synchronize()
        assert m2.device_error() == 0
        assert_close(to_np(y), to_np(y_ref), w.dtype, f"y, call {call}")
        assert_close(to_np(f), to_np(f_ref), w.dtype, f"final_state, call {call}")


def test_noalloc_fused_state_path_on_two_calls():
    """The fused stage 2+3 path keeps a ticket counter and per-chunk flag words in
    the shared array; stage 1 must clear them on every call, so a second call
    over the first one's leftovers still matches the ordinary entry point.  Both
    calls go through the Python wrapper ssd_fwd_noalloc."""
    w = W.Workload("noalloc bf16 fused", 1, 1024, 8, 64, 128, 1, 256, seed=504)
    for call in range(2):
        inp = W.make_inputs(w.scaled(seed=w.seed + 1000 * call))
        dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups, m2.FLAG_FUSED_STATE)
        assert sh.nchunks >= 3 and m2.path(sh) == m2.PATH_TCGEN05
        assert m2.workspace_size(sh) <= m2.NOALLOC_SCRATCH_BYTES
        y_ref, f_ref = m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                                  dev["initial_state"], chunk_size=w.chunk_size,
                                  ngroups=w.ngroups, flags=m2.FLAG_FUSED_STATE)
        y = torch.full_like(y_ref, float("nan"))
        f = torch.full_like(f_ref, float("nan"))
        m2.ssd_fwd_noalloc(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                           dev["initial_state"], chunk_size=w.chunk_size, ngroups=w.ngroups,
                           y=y, final_state=f, flags=m2.FLAG_FUSED_STATE)
        torch.cuda.synchronize()
        assert m2.device_error() == 0
        assert_close(to_np(y), to_np(y_ref), w.dtype, f"fused y, call {call}")
        assert_close(to_np(f), to_np(f_ref), w.dtype, f"fused final_state, call {call}")


def test_noalloc_rejects_shapes_beyond_the_scratch():
    lib = m2.load()
    sh = m2.make_shape(8, 4096, 80, 64, 128, 1, 256, m2.BF16)   # needs ~524 MB of workspace
    assert m2.workspace_size(sh) > m2.NOALLOC_SCRATCH_BYTES
    # Null data pointers: the size check returns first; were it ever to come
    # later, the pointer checks would reject the call on the host, so nothing
    # is launched either way.
    rc = lib.mamba2_ssd_fwd_noalloc(ctypes.byref(sh), *([None] * 9), None)
    assert rc == m2.ERR_WORKSPACE
