"""Seeded synthetic inputs for the SSD forward pass.

This module only draws random numbers: it holds none of the method's
arithmetic, so that the CUDA path's tests and the fp64 oracle can be fed the
same inputs without sharing any computation.

Distributions (the Mamba-2 layer workloads measured here): x, B, C ~ N(0, 1)
drawn in float32 and rounded to the run dtype; dt = exp(U(ln lo, ln hi)) per
(b, t, h); A_h = -exp(U(ln 1, ln 16)); D_h ~ N(0, 1); initial_state, when the
workload carries one, ~ N(0, 0.1^2) in float32.  A torch CPU generator is
seeded per workload and the tensors are drawn in the fixed order
x, B, C, dt, A, D, initial_state.

For the backward pass, ``make_grads`` draws the incoming gradients from a
second generator (seed + 500 000, so that the forward inputs stay the same):
dy ~ N(0, 1) in the run dtype and, when asked for, dfinal ~ N(0, 1) in float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    chunk_size: int
    dtype: str = "bf16"          # "bf16" or "f32": dtype of x, B, C and y
    dt_lo: float = 1e-3
    dt_hi: float = 1e-1
    init_std: float = 0.0         # 0 => no initial state (zero)
    seed: int = 0

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# Measured workloads.
TINY_F32 = Workload("tiny-fp32 b1 T256 H2 P16 N16 G1 L64", 1, 256, 2, 16, 16, 1, 64,
                    dtype="f32", seed=1001)
MAMBA2_2P7B = Workload("mamba2-2.7b-layer b8 T4096 H80 P64 N128 G1 L256 bf16",
                       8, 4096, 80, 64, 128, 1, 256, seed=1002)
GROUPED_INIT = Workload("grouped-init b2 T8192 H64 P64 N128 G8 L128 bf16",
                        2, 8192, 64, 64, 128, 8, 128, init_std=0.1, seed=1004)
LONG_PREFILL = Workload("long-prefill b1 T131072 H48 P64 N128 G1 L256 bf16",
                        1, 131072, 48, 64, 128, 1, 256, dt_lo=1e-4, seed=1005)


def sweep_workloads():
    """State-size x sequence-length sweep: N in {64,128,256} x T in {1024,4096,16384}."""
    out = []
    for iN, N in enumerate((64, 128, 256)):
        for iT, T in enumerate((1024, 4096, 16384)):
            out.append(Workload(f"sweep b4 T{T} H32 P64 N{N} G1 L256 bf16", 4, T, 32, 64, N,
                                1, 256, seed=1300 + 10 * iN + iT))
    return out


# Layer shapes for the other tensor-core views: head dimension 128 (the same
# inner width as the 2.7B layer, 40 heads of 128), 64-token chunks and head
# dimension 32.
HEADDIM128 = Workload("headdim128-layer b4 T4096 H40 P128 N128 G1 L256 bf16",
                      4, 4096, 40, 128, 128, 1, 256, seed=1006)
CHUNK64 = Workload("chunk64-layer b4 T4096 H32 P64 N128 G1 L64 bf16",
                   4, 4096, 32, 64, 128, 1, 64, seed=1007)
# Head dimension 32 (64 heads of 32: half the inner width of the 2.7B layer).
HEADDIM32 = Workload("headdim32-layer b4 T4096 H64 P32 N128 G1 L256 bf16",
                     4, 4096, 64, 32, 128, 1, 256, seed=1008)


ALL = ([TINY_F32, MAMBA2_2P7B] + sweep_workloads() + [GROUPED_INIT, LONG_PREFILL]
       + [HEADDIM128, CHUNK64, HEADDIM32])


def make_inputs(w: Workload, device="cpu"):
    """Draw the inputs of workload ``w`` (CPU generator), then move them to ``device``.

    Returns a dict x, dt, A, B, C, D, initial_state (None when init_std == 0).
    x, B, C have dtype w.torch_dtype; dt, A, D, initial_state are float32.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    b, T, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    x = torch.randn((b, T, H, P), generator=g, dtype=torch.float32).to(w.torch_dtype)
    B = torch.randn((b, T, G, N), generator=g, dtype=torch.float32).to(w.torch_dtype)
    C = torch.randn((b, T, G, N), generator=g, dtype=torch.float32).to(w.torch_dtype)
    dt = torch.empty((b, T, H), dtype=torch.float32).uniform_(
        math.log(w.dt_lo), math.log(w.dt_hi), generator=g).exp_()
    A = -torch.empty((H,), dtype=torch.float32).uniform_(
        0.0, math.log(16.0), generator=g).exp_()
    D = torch.randn((H,), generator=g, dtype=torch.float32)
    init = None
    if w.init_std > 0:
        init = torch.randn((b, H, P, N), generator=g, dtype=torch.float32) * w.init_std
    out = dict(x=x, dt=dt, A=A, B=B, C=C, D=D, initial_state=init)
    if device != "cpu":
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out


def make_grads(w: Workload, with_dfinal: bool = True, device="cpu"):
    """Incoming gradients for the backward pass of workload ``w``: a dict with
    dy [b,T,H,P] (dtype w.torch_dtype) and dfinal [b,H,P,N] float32 (or None)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed) + 500_000)
    b, T, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    dy = torch.randn((b, T, H, P), generator=g, dtype=torch.float32).to(w.torch_dtype)
    dfinal = torch.randn((b, H, P, N), generator=g, dtype=torch.float32) if with_dfinal else None
    out = dict(dy=dy, dfinal=dfinal)
    if device != "cpu":
        out = {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    return out
