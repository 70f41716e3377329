"""Host-side tests of the C ABI: no GPU needed, no kernel launched.

The library must load on a machine without a GPU, export every entry point
include/mamba2_ssd.h declares, and reject bad arguments on the host before any
CUDA call.
"""
import ctypes
import os
import re

import pytest

import mamba_ssd_chunked_02_gb300 as m2
from mamba_ssd_chunked_02_gb300 import build as m2build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    m2build.build()
    return m2.load()


def declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MAMBA2_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"
    assert set(m2.SYMBOLS) <= set(names)


def test_noalloc_scratch_size_matches_the_header():
    """The binding's NOALLOC_SCRATCH_BYTES is the header's MAMBA2_NOALLOC_SCRATCH_BYTES."""
    src = open(os.path.join(ROOT, "include", "mamba2_ssd.h")).read()
    m = re.search(r"#define\s+MAMBA2_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", src)
    assert m, "MAMBA2_NOALLOC_SCRATCH_BYTES not found in the header"
    assert m2.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_version_and_status_strings(lib):
    assert re.match(r"\d+\.\d+\.\d+", m2.version())
    for code in range(6):
        assert m2.status_string(code) and "unknown" not in m2.status_string(code)
    assert "unknown" in m2.status_string(99)


def shp(**kw):
    base = dict(batch=2, seqlen=512, nheads=8, headdim=64, dstate=128, ngroups=1,
                chunk_size=256, dtype=m2.BF16, flags=0)
    base.update(kw)
    return m2.make_shape(**base)


def test_check_shape(lib):
    assert m2.check_shape(shp()) == m2.OK
    assert m2.check_shape(shp(seqlen=300)) == m2.OK          # ragged last chunk
    assert m2.check_shape(shp(seqlen=0)) == m2.OK
    assert m2.check_shape(shp(batch=0)) == m2.OK
    assert m2.check_shape(shp(nheads=6, ngroups=4)) == m2.ERR_INVALID_ARG
    assert m2.check_shape(shp(batch=-1)) == m2.ERR_INVALID_ARG
    assert m2.check_shape(shp(headdim=0)) == m2.ERR_INVALID_ARG
    assert m2.check_shape(shp(dtype=7)) == m2.ERR_INVALID_ARG
    assert m2.check_shape(shp(flags=16)) == m2.ERR_INVALID_ARG
    assert m2.check_shape(shp(flags=m2.FLAG_FUSED_STATE | m2.FLAG_FORCE_SIMT)) == m2.OK
    assert m2.check_shape(shp(flags=m2.FLAG_SERIAL | m2.FLAG_DS_BF16)) == m2.OK
    assert m2.check_shape(shp(headdim=48)) == m2.ERR_UNSUPPORTED
    assert m2.check_shape(shp(dstate=96)) == m2.ERR_UNSUPPORTED
    assert m2.check_shape(shp(chunk_size=32)) == m2.ERR_UNSUPPORTED
    assert lib.mamba2_ssd_check_shape(None) == m2.ERR_INVALID_ARG


def test_workspace_size(lib):
    def a256(v):
        return (v + 255) // 256 * 256
    for kw in (dict(), dict(seqlen=300), dict(dtype=m2.F32, headdim=16, dstate=16, chunk_size=64)):
        s = shp(**kw)
        b, T, H, P, N, L = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.chunk_size
        nc = -(-T // L)
        es = 2 if s.dtype == m2.BF16 else 4
        want = 2 * a256(4 * b * H * T) + a256(4 * b * nc * H * P * N) + \
            a256(es * b * nc * H * P * N) + a256(32 * b * nc * H)
        assert m2.workspace_size(s) == want
    assert m2.workspace_size(shp(headdim=48)) == 0
    # The 2.7B-layer workload: cum2 + dtT (2 x 10.5 MB), dS (335.5 MB fp32), Sprev (167.8 MB bf16),
    # max |x| words (160 KB).
    s = shp(batch=8, seqlen=4096, nheads=80)
    assert m2.workspace_size(s) == 2 * 10_485_760 + 335_544_320 + 167_772_160 + 327_680


def test_path_selection(lib):
    assert m2.path(shp(headdim=48)) == -1
    assert m2.path(shp()) == m2.PATH_TCGEN05                  # the 2.7B layer shape
    assert m2.path(shp(chunk_size=128, dstate=64)) == m2.PATH_TCGEN05
    assert m2.path(shp(dstate=256, seqlen=300)) == m2.PATH_TCGEN05
    assert m2.path(shp(headdim=128)) == m2.PATH_TCGEN05       # as twice the heads of P = 64
    assert m2.path(shp(dtype=m2.F32)) == m2.PATH_SIMT
    assert m2.path(shp(chunk_size=64)) == m2.PATH_TCGEN05     # the whole path: 128-token chunks
    assert m2.path(shp(chunk_size=64, dtype=m2.F32)) == m2.PATH_SIMT
    assert m2.path(shp(headdim=32)) == m2.PATH_TCGEN05        # 64-column tiles, 32 kept
    assert m2.path(shp(headdim=16)) == m2.PATH_SIMT
    assert m2.path(shp(flags=m2.FLAG_FORCE_SIMT)) == m2.PATH_SIMT


def test_fwd_rejects_bad_pointers_without_launching(lib):
    s = shp()
    vp = ctypes.c_void_p
    good = vp(1 << 20)       # aligned, never dereferenced: validation fails first
    bad = vp((1 << 20) + 8)  # misaligned
    args = [good] * 9
    # null x
    rc = lib.mamba2_ssd_fwd(ctypes.byref(s), None, *args[1:], good, ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_INVALID_ARG
    # misaligned B
    a = list(args)
    a[3] = bad
    rc = lib.mamba2_ssd_fwd(ctypes.byref(s), *a, good, ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_INVALID_ARG
    # misaligned optional D
    a = list(args)
    a[5] = bad
    rc = lib.mamba2_ssd_fwd(ctypes.byref(s), *a, good, ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_INVALID_ARG
    # invalid shape
    s2 = shp(nheads=6, ngroups=4)
    rc = lib.mamba2_ssd_fwd(ctypes.byref(s2), *args, good, ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_INVALID_ARG
    # unsupported shape
    s3 = shp(dstate=96)
    rc = lib.mamba2_ssd_fwd(ctypes.byref(s3), *args, good, ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_UNSUPPORTED


def test_stage_entry_points_validate(lib):
    s = shp()
    vp = ctypes.c_void_p
    g = vp(1 << 20)
    assert lib.mamba2_ssd_chunk_cumsum(ctypes.byref(s), None, g, g, g, None) == m2.ERR_INVALID_ARG
    assert lib.mamba2_ssd_chunk_state(ctypes.byref(s), g, g, g, g, None, None) == m2.ERR_INVALID_ARG
    assert lib.mamba2_ssd_state_pass(ctypes.byref(s), g, g, vp((1 << 20) + 4), g, g,
                                     None) == m2.ERR_INVALID_ARG
    assert lib.mamba2_ssd_chunk_out(ctypes.byref(s), g, g, g, g, g, g, None, None,
                                    None) == m2.ERR_INVALID_ARG


def test_fused_stage_workspace_and_validation(lib):
    def a256(v):
        return (v + 255) // 256 * 256
    s = shp(batch=8, seqlen=4096, nheads=80)                  # the 2.7B layer: one n-tile
    want = a256(2 * 4 * 8 * 80 * 64 * 128) + a256(4 * (8 * 80 * 1 * 16 + 1))
    assert m2.chunk_state_pass_workspace_size(s) == want
    s2 = shp(dstate=256, seqlen=300)                           # two n-tiles, ragged
    assert m2.chunk_state_pass_workspace_size(s2) == \
        a256(2 * 4 * 2 * 8 * 64 * 256) + a256(4 * (2 * 8 * 2 * 2 + 1))
    assert m2.chunk_state_pass_workspace_size(shp(dtype=m2.F32)) == 0   # no tensor-core path
    vp = ctypes.c_void_p
    g = vp(1 << 20)
    rc = lib.mamba2_ssd_chunk_state_pass(ctypes.byref(shp(dtype=m2.F32)), *([g] * 7), g,
                                         ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_UNSUPPORTED
    rc = lib.mamba2_ssd_chunk_state_pass(ctypes.byref(shp()), None, *([g] * 6), g,
                                         ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_INVALID_ARG
    rc = lib.mamba2_ssd_chunk_state_pass(ctypes.byref(shp()), *([g] * 7), vp((1 << 20) + 64),
                                         ctypes.c_size_t(1 << 40), None)
    assert rc == m2.ERR_WORKSPACE                               # misaligned workspace
    rc = lib.mamba2_ssd_chunk_state_pass(ctypes.byref(shp()), *([g] * 7), g, ctypes.c_size_t(64),
                                         None)
    assert rc == m2.ERR_WORKSPACE                               # too small


def test_selftest_limit_is_validated_on_the_host(lib):
    assert lib.mamba2_ssd_selftest_wait_timeout(0, None) == m2.ERR_INVALID_ARG
    assert lib.mamba2_ssd_selftest_wait_timeout(100001, None) == m2.ERR_INVALID_ARG


def test_decode_validates_without_launching(lib):
    vp = ctypes.c_void_p
    g = vp(1 << 20)
    s = shp(seqlen=1)
    assert lib.mamba2_ssd_decode(ctypes.byref(shp(seqlen=2)), *([g] * 9)) == m2.ERR_INVALID_ARG
    assert lib.mamba2_ssd_decode(ctypes.byref(s), None, *([g] * 7), None) == m2.ERR_INVALID_ARG
    assert lib.mamba2_ssd_decode(ctypes.byref(shp(seqlen=1, dstate=96)), *([g] * 8), None) == \
        m2.ERR_UNSUPPORTED
    s0 = shp(seqlen=1, batch=0)
    assert lib.mamba2_ssd_decode(ctypes.byref(s0), *([None] * 8), None) == m2.OK


def test_empty_problem_is_a_noop(lib):
    # batch 0: nothing to do, no pointer needed, no CUDA call.
    s = shp(batch=0)
    assert m2.workspace_size(s) == 0
    rc = lib.mamba2_ssd_fwd(ctypes.byref(s), *([None] * 9), None, ctypes.c_size_t(0), None)
    assert rc == m2.OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 64, 2, 16)
    with pytest.raises(ValueError, match="CUDA"):
        m2.ssd_fwd(x, torch.zeros(1, 64, 2), torch.zeros(2), torch.zeros(1, 64, 1, 16),
                   torch.zeros(1, 64, 1, 16), chunk_size=64)


def test_fwd_strided_validates_strides_without_launching(lib):
    s = shp()
    b, T, H, P, N, G = s.batch, s.seqlen, s.nheads, s.headdim, s.dstate, s.ngroups
    vp = ctypes.c_void_p
    good = vp(1 << 20)       # aligned, never dereferenced: validation fails first
    args = [good] * 9 + [good, ctypes.c_size_t(1 << 40), None]

    def strides(**over):
        st = m2.Strides()
        st.x[:] = st.y[:] = (T * H * P, H * P)
        st.B[:] = st.C[:] = (T * G * N, G * N)
        st.dt[:] = (T * H, H)
        for k, v in over.items():
            getattr(st, k)[:] = v
        return st

    def call(st):
        return lib.mamba2_ssd_fwd_strided(ctypes.byref(s), ctypes.byref(st) if st is not None else None,
                                          *args)

    assert call(None) == m2.ERR_INVALID_ARG
    assert call(strides(x=(T * H * P, H * P - 1))) == m2.ERR_INVALID_ARG      # token overlap
    assert call(strides(y=(T * H * P - 1, H * P))) == m2.ERR_INVALID_ARG      # batch overlap
    assert call(strides(B=(T * G * N, 0))) == m2.ERR_INVALID_ARG
    assert call(strides(dt=(T * H, -H))) == m2.ERR_INVALID_ARG
    assert call(strides(C=(1 << 41, G * N))) == m2.ERR_INVALID_ARG           # beyond 2^40 elements
    # valid strides, then a bad pointer: the pointer check still fails first
    st = strides(x=(T * (H * P + 2 * G * N), H * P + 2 * G * N))
    rc = lib.mamba2_ssd_fwd_strided(ctypes.byref(s), ctypes.byref(st), None, *args[1:])
    assert rc == m2.ERR_INVALID_ARG


def test_bwd_workspace_size_formula(lib):
    """Backward workspace: cum2 and dtT, dS (then the chunk adjoints; bf16 on the
    tensor-core path, fp32 on the CUDA cores), Sprev in the I/O type, the final
    state and an I/O-type copy of Gn, each rounded up to 256 bytes.  On the
    tensor-core path the y and y' runs leave three per-token dots (two partials
    per token and head each: dy . y, x . y', dy . x; the y' run writes dx itself
    and runs anti-causal on dy, B, C as they are), stage 2 hands them max |x| and
    max |dy| per (b, chunk, head) for their fp16 range check, and dC and dB come
    from their own kernel, which reads x, dy, B, C and the states directly.  On
    the CUDA cores (here: forced) the runs instead need the reversed inputs of
    the y' run (dy, B, C reversed; cum2' and dt' = 1 rows), fp32 y and y', x
    reversed, per-head copies of B and reversed C, cum2 / dt rows per run head
    (Q = N/64 of them per head), the dC and dB runs' per-head outputs and
    Sprev^T, Gn^T."""
    a256 = lambda v: (v + 255) // 256 * 256
    b, T, H, P, N, G, L, E = 2, 512, 8, 64, 128, 1, 256, 2
    nc, Q = T // L, N // 64
    st = b * nc * H * P * N
    cum = a256(4 * b * H * T)
    base = 2 * cum + 3 * a256(E * st) + a256(4 * b * H * P * N)
    dots = a256(4 * 2 * b * H * T)           # per-token dots of the tensor-core y and y' runs
    y_no_skip = a256(4 * b * T * H * P)      # the CUDA-core y run's fp32 y
    y_rev = a256(4 * b * T * H * P)          # the CUDA-core y' run's fp32 y'
    xr = a256(E * b * T * H * P)             # x reversed, read by the dB run
    rev_in = a256(E * b * T * H * P) + 2 * a256(E * b * T * G * N) + 2 * cum   # dy, B, C; cum2', 1
    copies = 4 * a256(E * b * T * H * N) + 4 * a256(4 * Q * b * H * T) + 2 * a256(E * st)
    xabs = a256(32 * b * nc * H)             # max |x|, max |dy| per (b, chunk, head) from stage 2
    assert m2.bwd_workspace_size(shp()) == base + 3 * dots + 2 * xabs
    fp32_states = a256(4 * st) - a256(E * st)   # dS / chunk adjoints in fp32 on the CUDA cores
    assert m2.bwd_workspace_size(shp(flags=m2.FLAG_FORCE_SIMT)) == \
        base + rev_in + y_rev + xr + y_no_skip + copies + fp32_states
    assert m2.bwd_workspace_size(shp(headdim=3)) == 0          # invalid shape


def test_bwd_validates_arguments_without_launching(lib):
    s = shp()
    vp = ctypes.c_void_p
    good = vp(1 << 20)       # aligned, never dereferenced: validation fails first
    ws = m2.bwd_workspace_size(s)

    def call(shape=s, D=good, dD=good, x=good, workspace=good, nbytes=ws):
        return lib.mamba2_ssd_bwd(ctypes.byref(shape), x, good, good, good, good, D, None, good,
                                  None, good, good, good, good, good, dD, None, workspace,
                                  ctypes.c_size_t(nbytes), None)

    assert call(shape=shp(flags=m2.FLAG_FUSED_STATE)) == m2.ERR_INVALID_ARG
    assert call(shape=shp(flags=m2.FLAG_SERIAL)) == m2.ERR_INVALID_ARG
    assert call(dD=None) == m2.ERR_INVALID_ARG                     # D given, dD missing
    assert call(x=vp((1 << 20) + 4)) == m2.ERR_INVALID_ARG         # misaligned
    assert call(x=None) == m2.ERR_INVALID_ARG
    assert call(workspace=None) == m2.ERR_WORKSPACE
    assert call(nbytes=ws - 1) == m2.ERR_WORKSPACE
    assert call(workspace=vp((1 << 20) + 16)) == m2.ERR_WORKSPACE  # not 256-byte aligned
    assert call(shape=shp(headdim=3)) == m2.ERR_UNSUPPORTED


def test_backward_and_decode_bindings_refuse_cpu_tensors(lib):
    import torch
    x = torch.zeros(1, 64, 2, 16)
    args = (x, torch.zeros(1, 64, 2), torch.zeros(2), torch.zeros(1, 64, 1, 16),
            torch.zeros(1, 64, 1, 16))
    with pytest.raises(ValueError, match="CUDA"):
        m2.ssd_bwd(*args, dy=torch.zeros_like(x), chunk_size=64)
    with pytest.raises(ValueError, match="CUDA"):
        m2.ssd_decode(torch.zeros(1, 2, 16, 16), torch.zeros(1, 2, 16), torch.zeros(1, 2),
                      torch.zeros(2), torch.zeros(1, 1, 16), torch.zeros(1, 1, 16))
