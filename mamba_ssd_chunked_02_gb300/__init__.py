"""Mamba-2 SSD chunked forward pass on GB300 (sm_103a).

Thin ctypes binding of the C ABI in include/mamba2_ssd.h (library
``_lib/libmamba2_ssd.so``, built by ``python -m mamba_ssd_chunked_02_gb300.build``).
The binding only marshals arguments: every step of the computation runs in
the library's CUDA kernels.  torch supplies device memory and streams.  There
is no CPU path: calling any entry point without the built library or without a
CUDA device raises.

Entry points (same names as the C ABI, minus the ``mamba2_ssd_`` prefix):
  ssd_fwd, ssd_fwd_noalloc, chunk_cumsum, chunk_state, state_pass,
  chunk_state_pass, chunk_out, ssd_bwd, ssd_decode, workspace_size,
  bwd_workspace_size, chunk_state_pass_workspace_size, path, check_shape,
  tile_choice, tile_override, device_error, selftest_wait_timeout, version.

Pages: "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
"Mamba-2 아키텍처의 핵심 연산" (y_t = c_t^T h_t + D x_t) and "세 가지 핵심 커널
구현" (chunk_cumsum / fwd_pass_state / compute_out); "Accelerating Mamba-2 with
High-Performance Forward Pass Kernels in NVIDIA CUDA Tile" (brifing.si),
sections 4-9.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmamba2_ssd.so")

F32, BF16 = 0, 1
FLAG_FORCE_SIMT = 1
FLAG_FUSED_STATE = 2
FLAG_DS_BF16 = 4
FLAG_SERIAL = 8
PATH_SIMT, PATH_TCGEN05 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_DEVICE = range(6)

# Symbols the library exports (checked by the CPU test suite).
SYMBOLS = ("mamba2_ssd_check_shape", "mamba2_ssd_path", "mamba2_ssd_workspace_size",
           "mamba2_ssd_fwd", "mamba2_ssd_chunk_cumsum", "mamba2_ssd_chunk_state",
           "mamba2_ssd_state_pass", "mamba2_ssd_chunk_out", "mamba2_ssd_device_error",
           "mamba2_status_string", "mamba2_ssd_version", "mamba2_ssd_fwd_noalloc",
           "mamba2_ssd_chunk_state_pass", "mamba2_ssd_chunk_state_pass_workspace_size",
           "mamba2_ssd_selftest_wait_timeout", "mamba2_ssd_decode", "mamba2_ssd_fwd_timed",
           "mamba2_ssd_fwd_strided", "mamba2_ssd_bwd", "mamba2_ssd_bwd_workspace_size",
           "mamba2_ssd_tile_choice", "mamba2_ssd_tile_override")


class Shape(ctypes.Structure):
    """mirror of struct mamba2_ssd_shape"""
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]

    @property
    def nchunks(self) -> int:
        return (self.seqlen + self.chunk_size - 1) // self.chunk_size


class Strides(ctypes.Structure):
    """mirror of struct mamba2_ssd_strides: {batch, token} element strides"""
    _fields_ = [(n, ctypes.c_int64 * 2) for n in ("x", "dt", "B", "C", "y")]


class Mamba2Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def load():
    """Load the C-ABI library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m mamba_ssd_chunked_02_gb300.build`"
                " (there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, sp, i32 = ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_int32
        lib.mamba2_ssd_check_shape.argtypes = [sp]
        lib.mamba2_ssd_check_shape.restype = ctypes.c_int
        lib.mamba2_ssd_path.argtypes = [sp]
        lib.mamba2_ssd_path.restype = i32
        lib.mamba2_ssd_workspace_size.argtypes = [sp]
        lib.mamba2_ssd_workspace_size.restype = ctypes.c_size_t
        lib.mamba2_ssd_fwd.argtypes = [sp] + [vp] * 9 + [vp, ctypes.c_size_t, vp]
        lib.mamba2_ssd_fwd.restype = ctypes.c_int
        lib.mamba2_ssd_fwd_strided.argtypes = [sp, ctypes.POINTER(Strides)] + [vp] * 9 + \
            [vp, ctypes.c_size_t, vp]
        lib.mamba2_ssd_fwd_strided.restype = ctypes.c_int
        lib.mamba2_ssd_chunk_cumsum.argtypes = [sp, vp, vp, vp, vp, vp]
        lib.mamba2_ssd_chunk_cumsum.restype = ctypes.c_int
        lib.mamba2_ssd_chunk_state.argtypes = [sp, vp, vp, vp, vp, vp, vp]
        lib.mamba2_ssd_chunk_state.restype = ctypes.c_int
        lib.mamba2_ssd_state_pass.argtypes = [sp, vp, vp, vp, vp, vp, vp]
        lib.mamba2_ssd_state_pass.restype = ctypes.c_int
        lib.mamba2_ssd_chunk_out.argtypes = [sp] + [vp] * 8 + [vp]
        lib.mamba2_ssd_chunk_out.restype = ctypes.c_int
        lib.mamba2_ssd_device_error.argtypes = [ctypes.POINTER(i32), i32]
        lib.mamba2_ssd_device_error.restype = ctypes.c_int
        lib.mamba2_status_string.argtypes = [ctypes.c_int]
        lib.mamba2_status_string.restype = ctypes.c_char_p
        lib.mamba2_ssd_version.argtypes = []
        lib.mamba2_ssd_version.restype = ctypes.c_char_p
        lib.mamba2_ssd_fwd_noalloc.argtypes = [sp] + [vp] * 9 + [vp]
        lib.mamba2_ssd_fwd_noalloc.restype = ctypes.c_int
        lib.mamba2_ssd_chunk_state_pass_workspace_size.argtypes = [sp]
        lib.mamba2_ssd_chunk_state_pass_workspace_size.restype = ctypes.c_size_t
        lib.mamba2_ssd_chunk_state_pass.argtypes = [sp] + [vp] * 7 + [vp, ctypes.c_size_t, vp]
        lib.mamba2_ssd_chunk_state_pass.restype = ctypes.c_int
        lib.mamba2_ssd_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        lib.mamba2_ssd_selftest_wait_timeout.restype = ctypes.c_int
        lib.mamba2_ssd_decode.argtypes = [sp] + [vp] * 9
        lib.mamba2_ssd_decode.restype = ctypes.c_int
        lib.mamba2_ssd_fwd_timed.argtypes = [sp] + [vp] * 9 + [vp, ctypes.c_size_t, vp,
                                                                ctypes.POINTER(vp)]
        lib.mamba2_ssd_fwd_timed.restype = ctypes.c_int
        lib.mamba2_ssd_bwd_workspace_size.argtypes = [sp]
        lib.mamba2_ssd_bwd_workspace_size.restype = ctypes.c_size_t
        lib.mamba2_ssd_bwd.argtypes = [sp] + [vp] * 16 + [vp, ctypes.c_size_t, vp]
        lib.mamba2_ssd_bwd.restype = ctypes.c_int
        lib.mamba2_ssd_tile_choice.argtypes = [sp, ctypes.POINTER(i32)]
        lib.mamba2_ssd_tile_choice.restype = ctypes.c_int
        lib.mamba2_ssd_tile_override.argtypes = [i32] * 4
        lib.mamba2_ssd_tile_override.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().mamba2_status_string(int(status)).decode()


def version() -> str:
    return load().mamba2_ssd_version().decode()


def make_shape(batch, seqlen, nheads, headdim, dstate, ngroups=1, chunk_size=256,
               dtype=BF16, flags=0) -> Shape:
    return Shape(int(batch), int(seqlen), int(nheads), int(headdim), int(dstate),
                 int(ngroups), int(chunk_size), int(dtype), int(flags))


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return BF16
    if t == torch.float32:
        return F32
    raise TypeError(f"unsupported element type {t}: x, B, C must be bfloat16 or float32")


def shape_of(x, B, chunk_size=256, ngroups=None, flags=0) -> Shape:
    b, T, H, P = x.shape
    G = B.shape[2] if ngroups is None else ngroups
    return make_shape(b, T, H, P, B.shape[3], G, chunk_size, _dtype_code(x.dtype), flags)


def check_shape(shape: Shape) -> int:
    return int(load().mamba2_ssd_check_shape(ctypes.byref(shape)))


def path(shape: Shape) -> int:
    """PATH_TCGEN05 or PATH_SIMT for a valid shape, -1 otherwise."""
    return int(load().mamba2_ssd_path(ctypes.byref(shape)))


def workspace_size(shape: Shape) -> int:
    return int(load().mamba2_ssd_workspace_size(ctypes.byref(shape)))


def _ptr(t, name, dtype=None, shape=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def _token_strided(t, inner):
    """True when t is a view whose last `inner` dims are contiguous (a token's
    data in one piece) but whose batch/token strides are not the contiguous
    ones: the layout mamba2_ssd_fwd_strided takes."""
    if t is None or t.is_contiguous():
        return False
    st, sz = t.stride(), t.shape
    want = 1
    for k in range(t.dim() - 1, t.dim() - 1 - inner, -1):
        if sz[k] != 1 and st[k] != want:
            return False
        want *= sz[k]
    return True


def _strided_ptr(t, name, dtype, shape, inner):
    """Pointer of a token-strided tensor and its {batch, token} element strides."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not (t.is_contiguous() or _token_strided(t, inner)):
        raise ValueError(f"{name}: each token's data must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0), (t.stride(0), t.stride(1))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _io_dtype(shape):
    return torch.bfloat16 if shape.dtype == BF16 else torch.float32


def _check(fn, rc):
    if rc != OK:
        raise Mamba2Error(fn, rc)


def ssd_fwd(x, dt, A, B, C, D=None, initial_state=None, chunk_size=256, ngroups=None, *,
            y=None, final_state=None, workspace=None, stream=None, flags=0, events=None):
    """Forward pass (mamba2_ssd_fwd).  Returns (y, final_state).

    x [b,T,H,P] bf16|f32, dt [b,T,H] f32, A [H] f32, B/C [b,T,G,N] (x's dtype),
    D [H] f32 or None, initial_state [b,H,P,N] f32 or None.  y, final_state and
    workspace are allocated with torch when not given.  x, dt, B, C and y may be
    views with any batch and token strides as long as each token's data is
    contiguous (e.g. column slices of one projection output): they go through
    mamba2_ssd_fwd_strided.  `events`: five torch.cuda.Event (or None entries)
    recorded before stage 1, after each stage and after stage 4
    (mamba2_ssd_fwd_timed; contiguous tensors only).
    """
    lib = load()
    sh = shape_of(x, B, chunk_size, ngroups, flags)
    b, T, H, P, N, G = sh.batch, sh.seqlen, sh.nheads, sh.headdim, sh.dstate, sh.ngroups
    io = _io_dtype(sh)
    if y is None:
        y = torch.empty((b, T, H, P), dtype=io, device=x.device)
    if final_state is None:
        final_state = torch.empty((b, H, P, N), dtype=torch.float32, device=x.device)
    need = workspace_size(sh)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    if any(_token_strided(t, k) for t, k in ((x, 2), (dt, 1), (B, 2), (C, 2), (y, 2))):
        if events is not None:
            raise ValueError("events: contiguous tensors only")
        st = Strides()
        px, st.x[:] = _strided_ptr(x, "x", io, (b, T, H, P), 2)
        pd, st.dt[:] = _strided_ptr(dt, "dt", torch.float32, (b, T, H), 1)
        pb, st.B[:] = _strided_ptr(B, "B", io, (b, T, G, N), 2)
        pc, st.C[:] = _strided_ptr(C, "C", io, (b, T, G, N), 2)
        py, st.y[:] = _strided_ptr(y, "y", io, (b, T, H, P), 2)
        _check("mamba2_ssd_fwd_strided", lib.mamba2_ssd_fwd_strided(
            ctypes.byref(sh), ctypes.byref(st), px, pd, _ptr(A, "A", torch.float32, (H,)), pb, pc,
            _ptr(D, "D", torch.float32, (H,), optional=True),
            _ptr(initial_state, "initial_state", torch.float32, (b, H, P, N), optional=True),
            py, _ptr(final_state, "final_state", torch.float32, (b, H, P, N)),
            _ptr(workspace, "workspace", optional=True),
            ctypes.c_size_t(workspace.numel() * workspace.element_size() if workspace is not None else 0),
            _stream(stream)))
        return y, final_state
    args = [
        _ptr(x, "x", io, (b, T, H, P)), _ptr(dt, "dt", torch.float32, (b, T, H)),
        _ptr(A, "A", torch.float32, (H,)), _ptr(B, "B", io, (b, T, G, N)),
        _ptr(C, "C", io, (b, T, G, N)), _ptr(D, "D", torch.float32, (H,), optional=True),
        _ptr(initial_state, "initial_state", torch.float32, (b, H, P, N), optional=True),
        _ptr(y, "y", io, (b, T, H, P)), _ptr(final_state, "final_state", torch.float32, (b, H, P, N)),
        _ptr(workspace, "workspace", optional=True),
        ctypes.c_size_t(workspace.numel() * workspace.element_size() if workspace is not None else 0),
        _stream(stream)]
    if events is None:
        _check("mamba2_ssd_fwd", lib.mamba2_ssd_fwd(ctypes.byref(sh), *args))
    else:
        evs = (ctypes.c_void_p * 5)()
        for k, ev in enumerate(list(events)[:5]):
            if ev is not None:
                if not ev.cuda_event:       # torch creates the CUDA event on first use
                    ev.record()
                evs[k] = ctypes.c_void_p(ev.cuda_event)
        _check("mamba2_ssd_fwd_timed", lib.mamba2_ssd_fwd_timed(ctypes.byref(sh), *args, evs))
    return y, final_state


def chunk_cumsum(shape, dt, A, cum2, dtT, stream=None):
    """Stage 1 (mamba2_ssd_chunk_cumsum): cum2, dtT [b,H,T] f32 outputs."""
    b, T, H = shape.batch, shape.seqlen, shape.nheads
    _check("mamba2_ssd_chunk_cumsum", load().mamba2_ssd_chunk_cumsum(
        ctypes.byref(shape), _ptr(dt, "dt", torch.float32, (b, T, H)),
        _ptr(A, "A", torch.float32, (H,)), _ptr(cum2, "cum2", torch.float32, (b, H, T)),
        _ptr(dtT, "dtT", torch.float32, (b, H, T)), _stream(stream)))


def _with_ds_dtype(shape, dS):
    """A copy of `shape` whose MAMBA2_FLAG_DS_BF16 bit matches dS's dtype."""
    sh = Shape(*[getattr(shape, f) for f, _ in Shape._fields_])
    if dS is not None and dS.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"dS must be torch.float32 or torch.bfloat16, got {dS.dtype}")
    if dS is not None and dS.dtype == torch.bfloat16:
        sh.flags |= FLAG_DS_BF16
    else:
        sh.flags &= ~FLAG_DS_BF16
    return sh


def chunk_state(shape, x, B, cum2, dtT, dS, stream=None):
    """Stage 2 (mamba2_ssd_chunk_state): dS [b,nc,H,P,N] output, f32 or bf16
    (bf16: the hand-off the whole-path call uses on the tensor-core path)."""
    b, T, H, P, N, G = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                        shape.ngroups)
    io = _io_dtype(shape)
    sh = _with_ds_dtype(shape, dS)
    _check("mamba2_ssd_chunk_state", load().mamba2_ssd_chunk_state(
        ctypes.byref(sh), _ptr(x, "x", io, (b, T, H, P)), _ptr(B, "B", io, (b, T, G, N)),
        _ptr(cum2, "cum2", torch.float32, (b, H, T)), _ptr(dtT, "dtT", torch.float32, (b, H, T)),
        _ptr(dS, "dS", dS.dtype if dS is not None else torch.float32, (b, shape.nchunks, H, P, N)),
        _stream(stream)))


def state_pass(shape, dS, cum2, initial_state, Sprev, final_state, stream=None):
    """Stage 3 (mamba2_ssd_state_pass): Sprev [b,nc,H,P,N] (I/O dtype), final_state f32;
    dS f32 or bf16."""
    b, T, H, P, N = shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate
    nc = shape.nchunks
    sh = _with_ds_dtype(shape, dS)
    _check("mamba2_ssd_state_pass", load().mamba2_ssd_state_pass(
        ctypes.byref(sh), _ptr(dS, "dS", dS.dtype if dS is not None else torch.float32,
                               (b, nc, H, P, N)),
        _ptr(cum2, "cum2", torch.float32, (b, H, T)),
        _ptr(initial_state, "initial_state", torch.float32, (b, H, P, N), optional=True),
        _ptr(Sprev, "Sprev", _io_dtype(shape), (b, nc, H, P, N)),
        _ptr(final_state, "final_state", torch.float32, (b, H, P, N)), _stream(stream)))


DEVERR_SELFTEST = 16
DEVERR_TIMEOUT_DECODE = 32


def ssd_decode(state, x, dt, A, B, C, D=None, *, y=None, stream=None):
    """One decode step (mamba2_ssd_decode): updates `state` [b,H,P,N] f32 in place
    and returns y [b,H,P].  x [b,H,P], dt [b,H] f32, A [H] f32, B/C [b,G,N]
    (x's dtype), D [H] f32 or None."""
    b, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    io = x.dtype
    sh = make_shape(b, 1, H, P, N, G, 64, _dtype_code(io), 0)
    if y is None:
        y = torch.empty((b, H, P), dtype=io, device=x.device)
    _check("mamba2_ssd_decode", load().mamba2_ssd_decode(
        ctypes.byref(sh), _ptr(state, "state", torch.float32, (b, H, P, N)),
        _ptr(x, "x", io, (b, H, P)), _ptr(dt, "dt", torch.float32, (b, H)),
        _ptr(A, "A", torch.float32, (H,)), _ptr(B, "B", io, (b, G, N)),
        _ptr(C, "C", io, (b, G, N)), _ptr(D, "D", torch.float32, (H,), optional=True),
        _ptr(y, "y", io, (b, H, P)), _stream(stream)))
    return y


def selftest_wait_timeout(limit_us=1000, stream=None):
    """Queue the wait self-test: bounded waits that nothing releases run out after
    `limit_us` and set DEVERR_SELFTEST in the device error word."""
    _check("mamba2_ssd_selftest_wait_timeout",
           load().mamba2_ssd_selftest_wait_timeout(int(limit_us), _stream(stream)))


def chunk_state_pass_workspace_size(shape: Shape) -> int:
    return int(load().mamba2_ssd_chunk_state_pass_workspace_size(ctypes.byref(shape)))


def chunk_state_pass(shape, x, B, cum2, dtT, initial_state, Sprev, final_state, workspace,
                     stream=None):
    """Stages 2+3 fused (mamba2_ssd_chunk_state_pass, tensor-core shapes only):
    Sprev [b,nc,H,P,N] and final_state [b,H,P,N] without dS.  `workspace` is a
    uint8 device tensor of chunk_state_pass_workspace_size(shape) bytes."""
    b, T, H, P, N, G = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                        shape.ngroups)
    io = _io_dtype(shape)
    nc = shape.nchunks
    _check("mamba2_ssd_chunk_state_pass", load().mamba2_ssd_chunk_state_pass(
        ctypes.byref(shape), _ptr(x, "x", io, (b, T, H, P)), _ptr(B, "B", io, (b, T, G, N)),
        _ptr(cum2, "cum2", torch.float32, (b, H, T)), _ptr(dtT, "dtT", torch.float32, (b, H, T)),
        _ptr(initial_state, "initial_state", torch.float32, (b, H, P, N), optional=True),
        _ptr(Sprev, "Sprev", io, (b, nc, H, P, N)),
        _ptr(final_state, "final_state", torch.float32, (b, H, P, N)),
        _ptr(workspace, "workspace", optional=True),
        ctypes.c_size_t(workspace.numel() * workspace.element_size() if workspace is not None else 0),
        _stream(stream)))


def chunk_out(shape, x, B, C, cum2, dtT, Sprev, D, y, stream=None):
    """Stage 4 (mamba2_ssd_chunk_out): y [b,T,H,P] output."""
    b, T, H, P, N, G = (shape.batch, shape.seqlen, shape.nheads, shape.headdim, shape.dstate,
                        shape.ngroups)
    io = _io_dtype(shape)
    _check("mamba2_ssd_chunk_out", load().mamba2_ssd_chunk_out(
        ctypes.byref(shape), _ptr(x, "x", io, (b, T, H, P)), _ptr(B, "B", io, (b, T, G, N)),
        _ptr(C, "C", io, (b, T, G, N)), _ptr(cum2, "cum2", torch.float32, (b, H, T)),
        _ptr(dtT, "dtT", torch.float32, (b, H, T)),
        _ptr(Sprev, "Sprev", io, (b, shape.nchunks, H, P, N)),
        _ptr(D, "D", torch.float32, (H,), optional=True), _ptr(y, "y", io, (b, T, H, P)),
        _stream(stream)))


def bwd_workspace_size(shape: Shape) -> int:
    return int(load().mamba2_ssd_bwd_workspace_size(ctypes.byref(shape)))


def ssd_bwd(x, dt, A, B, C, D=None, initial_state=None, dy=None, dfinal=None, chunk_size=256,
            ngroups=None, *, grads=None, workspace=None, stream=None, flags=0):
    """Backward pass (mamba2_ssd_bwd): gradients of a loss with dL/dy = dy and
    dL/dfinal_state = dfinal (None = 0), for the inputs of ssd_fwd.  Returns a
    dict of fp32 tensors dx [b,T,H,P], ddt [b,T,H], dA [H], dB, dC [b,T,G,N],
    dD [H] (None when D is None) and dinit [b,H,P,N] (None when initial_state
    is None).  `grads`: an optional dict of preallocated outputs (same keys)."""
    lib = load()
    sh = shape_of(x, B, chunk_size, ngroups, flags)
    b, T, H, P, N, G = sh.batch, sh.seqlen, sh.nheads, sh.headdim, sh.dstate, sh.ngroups
    io = _io_dtype(sh)
    dev = x.device
    f32 = torch.float32
    shapes = dict(dx=(b, T, H, P), ddt=(b, T, H), dA=(H,), dB=(b, T, G, N), dC=(b, T, G, N),
                  dD=(H,), dinit=(b, H, P, N))
    g = dict(grads or {})
    for k, shp in shapes.items():
        if k == "dD" and D is None:
            g.setdefault(k, None)
        elif k == "dinit" and initial_state is None:
            g.setdefault(k, None)
        elif g.get(k) is None:
            g[k] = torch.empty(shp, dtype=f32, device=dev)
    need = bwd_workspace_size(sh)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check("mamba2_ssd_bwd", lib.mamba2_ssd_bwd(
        ctypes.byref(sh), _ptr(x, "x", io, (b, T, H, P)), _ptr(dt, "dt", f32, (b, T, H)),
        _ptr(A, "A", f32, (H,)), _ptr(B, "B", io, (b, T, G, N)), _ptr(C, "C", io, (b, T, G, N)),
        _ptr(D, "D", f32, (H,), optional=True),
        _ptr(initial_state, "initial_state", f32, (b, H, P, N), optional=True),
        _ptr(dy, "dy", io, (b, T, H, P)),
        _ptr(dfinal, "dfinal", f32, (b, H, P, N), optional=True),
        *[_ptr(g[k], k, f32, shapes[k], optional=k in ("dD", "dinit")) for k in shapes],
        _ptr(workspace, "workspace", optional=True),
        ctypes.c_size_t(workspace.numel() * workspace.element_size() if workspace is not None else 0),
        _stream(stream)))
    return g


# Size of the library's fixed scratch array (MAMBA2_NOALLOC_SCRATCH_BYTES in
# include/mamba2_ssd.h; a CPU test checks that the two agree).
NOALLOC_SCRATCH_BYTES = 64 << 20


def ssd_fwd_noalloc(x, dt, A, B, C, D=None, initial_state=None, chunk_size=256, ngroups=None,
                    *, y, final_state, stream=None, flags=0):
    """Forward pass through mamba2_ssd_fwd_noalloc, for callers that cannot
    allocate device memory: the workspace is the library's own fixed 64 MiB
    device array, so the caller passes preallocated outputs `y` and
    `final_state` and nothing is allocated here.  Calls on one device share
    that array and must not overlap on the GPU."""
    sh = shape_of(x, B, chunk_size, ngroups, flags)
    b, T, H, P, N, G = sh.batch, sh.seqlen, sh.nheads, sh.headdim, sh.dstate, sh.ngroups
    io = _io_dtype(sh)
    args = [
        _ptr(x, "x", io, (b, T, H, P)), _ptr(dt, "dt", torch.float32, (b, T, H)),
        _ptr(A, "A", torch.float32, (H,)), _ptr(B, "B", io, (b, T, G, N)),
        _ptr(C, "C", io, (b, T, G, N)), _ptr(D, "D", torch.float32, (H,), optional=True),
        _ptr(initial_state, "initial_state", torch.float32, (b, H, P, N), optional=True),
        _ptr(y, "y", io, (b, T, H, P)), _ptr(final_state, "final_state", torch.float32, (b, H, P, N)),
        _stream(stream)]
    _check("mamba2_ssd_fwd_noalloc", load().mamba2_ssd_fwd_noalloc(ctypes.byref(sh), *args))
    return y, final_state


SOURCE_MODEL, SOURCE_TABLE, SOURCE_OVERRIDE = 0, 1, 2


def tile_choice(shape: Shape) -> dict:
    """Launch choices of the tensor-core kernels for `shape` (mamba2_ssd_tile_choice)."""
    out = (ctypes.c_int32 * 6)()
    _check("mamba2_ssd_tile_choice", load().mamba2_ssd_tile_choice(ctypes.byref(shape), out))
    return {"stage2_units": out[0], "stage2_source": out[1], "stage4_v1": out[2],
            "stage4_v2": out[3], "stage4_pairs1": out[4], "stage4_source": out[5]}


MODEL_ONLY, EVEN_SPLIT = -1, -2


def tile_override(stage2_units=0, stage4_v1=0, stage4_v2=0, stage4_waves1=0):
    """Force launch choices for later calls (mamba2_ssd_tile_override); zeros clear.
    MODEL_ONLY (-1) bypasses the table; EVEN_SPLIT (-2, stage 2) forces one wave of
    even unit ranges."""
    _check("mamba2_ssd_tile_override",
           load().mamba2_ssd_tile_override(stage2_units, stage4_v1, stage4_v2, stage4_waves1))


def device_error(clear=True) -> int:
    """Synchronise and return the library's device-side error word (0 = none)."""
    code = ctypes.c_int32(0)
    rc = load().mamba2_ssd_device_error(ctypes.byref(code), int(bool(clear)))
    if rc not in (OK, ERR_DEVICE):
        raise Mamba2Error("mamba2_ssd_device_error", rc)
    return int(code.value)
