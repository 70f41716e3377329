"""fp64 CPU oracle for the Mamba-2 SSD forward and backward passes (ctypes wrapper
of ssd_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package.  The CUDA
product path never imports, links or calls it, and it shares no code with it.

Pages cited (by title and section):
  [P2] "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
       "Mamba-2 아키텍처의 핵심 연산" (read-out y_t = c_t^T h_t + D x_t; log-space
       cumulative sum of a_t) and "세 가지 핵심 커널 구현" (the three kernels).
  [P3] "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
       NVIDIA CUDA Tile" (brifing.si), sections 4 (jump formula), 5 (log-space
       decay), 7 (chunk_cumsum), 8 (fwd_pass_state), 9 (compute_out),
       11 (causal masking).

Every function takes numpy arrays (any float dtype; they are widened to float32
first, which is exact for the bf16 / fp32 values the GPU path sees), plus an
optional ``lib`` handle from ``load_variant``, and returns float64 results.  Layouts: x [b,T,H,P], dt [b,T,H], A [H], B and C [b,T,G,N],
D [H] or None, initial_state [b,H,P,N] or None; y [b,T,H,P],
final_state [b,H,P,N]; cum2 [b,H,T]; dS and Sprev [b,nc,H,P,N].

Parity pins (tests/test_oracle.py): brute force (quadratic form), chunk-size
independence including L = 1 and L = T, the A = 0 causal-linear-attention
closed form, the impulse response, dt = 0, the scalar geometric-series closed
form, linearity, group mapping and split-and-resume.  The backward pass
(``ssd_backward``) is pinned by finite differences of the forward oracle and
by the homogeneity identities of the loss (tests/test_oracle_bwd.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libssd_oracle.so")
_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle C source with gcc (OpenMP, -O2, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path):
    lib = ctypes.CDLL(path)
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_ssd_recurrent.argtypes = [i64] * 6 + [vp] * 7 + [vp, i64, vp, vp, ctypes.c_int]
    lib.oracle_ssd_recurrent.restype = ctypes.c_int
    lib.oracle_ssd_chunked.argtypes = [i64] * 7 + [vp] * 7 + [vp] * 5 + [ctypes.c_int]
    lib.oracle_ssd_chunked.restype = ctypes.c_int
    lib.oracle_ssd_quadratic.argtypes = [i64] * 6 + [vp] * 7 + [vp, vp]
    lib.oracle_ssd_quadratic.restype = ctypes.c_int
    lib.oracle_ssd_backward.argtypes = [i64] * 6 + [vp] * 9 + [vp, i64] + [vp] * 7 + [ctypes.c_int]
    lib.oracle_ssd_backward.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = _bind(build())
    return _default


def load_variant(src: str, out: str):
    """Compile and bind another copy of the oracle source (used by the tests that
    plant a mistake in a copy of the oracle and check that a pin catches it).
    Pass the returned handle as ``lib=`` to the functions below."""
    return _bind(build(force=True, src=src, out=out))


def _f32(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor on the CPU
        a = a.detach().float().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(x, B, ngroups):
    b, T, H, P = x.shape
    assert B.shape[0] == b and B.shape[1] == T and B.shape[2] == ngroups, (B.shape, ngroups)
    N = B.shape[3]
    return b, T, H, P, N


def max_threads() -> int:
    """OpenMP threads the oracle uses by default on this host."""
    return int(_load().oracle_max_threads())


def ssd_recurrent(x, dt, A, B, C, D=None, initial_state=None, ngroups=1, pairs=None,
                  nthreads=0, lib=None):
    """Token-by-token recurrence (the definition).  Returns (y, final_state) in float64.

    ``pairs``: optional iterable of (b, h) to compute; other entries of y and
    final_state are left as NaN.
    """
    lib = lib or _load()
    x, dt, A, B, C, D, S0 = map(_f32, (x, dt, A, B, C, D, initial_state))
    b, T, H, P, N = _dims(x, B, ngroups)
    y = np.full((b, T, H, P), np.nan)
    fin = np.full((b, H, P, N), np.nan)
    pr = None
    npairs = 0
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(list(pairs), dtype=np.int64).reshape(-1, 2))
        npairs = pr.shape[0]
    rc = lib.oracle_ssd_recurrent(b, T, H, P, N, ngroups, _ptr(x), _ptr(dt), _ptr(A),
                                  _ptr(B), _ptr(C), _ptr(D), _ptr(S0), _ptr(pr), npairs,
                                  _ptr(y), _ptr(fin), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_ssd_recurrent: invalid arguments")
    return y, fin


def ssd_chunked(x, dt, A, B, C, D=None, initial_state=None, ngroups=1, chunk_size=64,
                nthreads=0, lib=None):
    """The pages' four chunked steps in fp64.

    Returns a dict with y, final_state, cum2 [b,H,T] (log2-scaled chunk-local
    cumsum), dS [b,nc,H,P,N] (chunk states) and Sprev [b,nc,H,P,N] (state
    entering each chunk).
    """
    lib = lib or _load()
    x, dt, A, B, C, D, S0 = map(_f32, (x, dt, A, B, C, D, initial_state))
    b, T, H, P, N = _dims(x, B, ngroups)
    L = int(chunk_size)
    if L <= 0:
        raise ValueError("oracle_ssd_chunked: chunk_size must be positive")
    nc = (T + L - 1) // L
    out = dict(y=np.empty((b, T, H, P)), final_state=np.empty((b, H, P, N)),
               cum2=np.empty((b, H, T)), dS=np.empty((b, nc, H, P, N)),
               Sprev=np.empty((b, nc, H, P, N)))
    rc = lib.oracle_ssd_chunked(b, T, H, P, N, ngroups, L, _ptr(x), _ptr(dt), _ptr(A),
                                _ptr(B), _ptr(C), _ptr(D), _ptr(S0), _ptr(out["cum2"]),
                                _ptr(out["dS"]), _ptr(out["Sprev"]), _ptr(out["y"]),
                                _ptr(out["final_state"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_ssd_chunked: invalid arguments")
    return out


def ssd_quadratic(x, dt, A, B, C, D=None, initial_state=None, ngroups=1, lib=None):
    """Brute-force quadratic form (tiny inputs only).  Returns (y, final_state)."""
    lib = lib or _load()
    x, dt, A, B, C, D, S0 = map(_f32, (x, dt, A, B, C, D, initial_state))
    b, T, H, P, N = _dims(x, B, ngroups)
    y = np.empty((b, T, H, P))
    fin = np.empty((b, H, P, N))
    rc = lib.oracle_ssd_quadratic(b, T, H, P, N, ngroups, _ptr(x), _ptr(dt), _ptr(A),
                                  _ptr(B), _ptr(C), _ptr(D), _ptr(S0), _ptr(y), _ptr(fin))
    if rc != 0:
        raise ValueError("oracle_ssd_quadratic: invalid arguments")
    return y, fin


def ssd_backward(x, dt, A, B, C, D=None, initial_state=None, dy=None, dfinal=None, ngroups=1,
                 pairs=None, nthreads=0, lib=None):
    """Gradients of L = sum(dy * y) + sum(dfinal * final_state) by reverse-mode
    differentiation of the recurrence (the chain rule on the definition; the
    pages give no backward method).  Returns a dict of float64 arrays:
    dx [b,T,H,P], ddt [b,T,H], dA [H], dB and dC [b,T,G,N], dD [H],
    dinit [b,H,P,N].  ``pairs``: optional (b, h) pairs; dx, ddt and dinit of
    other pairs are NaN and dA, dD, dB, dC sum the listed pairs only.
    """
    lib = lib or _load()
    x, dt, A, B, C, D, S0, dy, dfinal = map(_f32, (x, dt, A, B, C, D, initial_state, dy, dfinal))
    b, T, H, P, N = _dims(x, B, ngroups)
    if dy is None or dy.shape != x.shape:
        raise ValueError("ssd_backward: dy must have x's shape")
    out = dict(dx=np.full((b, T, H, P), np.nan), ddt=np.full((b, T, H), np.nan),
               dA=np.empty(H), dB=np.empty((b, T, ngroups, N)), dC=np.empty((b, T, ngroups, N)),
               dD=np.empty(H), dinit=np.full((b, H, P, N), np.nan))
    pr = None
    npairs = 0
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(list(pairs), dtype=np.int64).reshape(-1, 2))
        npairs = pr.shape[0]
    rc = lib.oracle_ssd_backward(b, T, H, P, N, ngroups, _ptr(x), _ptr(dt), _ptr(A), _ptr(B),
                                 _ptr(C), _ptr(D), _ptr(S0), _ptr(dy), _ptr(dfinal), _ptr(pr),
                                 npairs, _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]),
                                 _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
                                 _ptr(out["dinit"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_ssd_backward: invalid arguments")
    return out
