"""The identities the backward kernels are built on, checked in fp64 against the
oracle's reverse sweep of the recurrence (CPU, small shapes, ragged chunks).

The CUDA backward computes every gradient with the forward's chunked output
step ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
CUDA Tile" (brifing.si), section 9) on reordered inputs:

* dx = dt * y' + D dy and ddt = x . y' + A * suffix-sum(dcum), where y' is the
  output step run backwards in time (each chunk's tokens reversed, B and C
  swapped, dt' = 1, cum2' = c2_last - c2, the chunk-leaving adjoint Gn as the
  carried state) and dcum_i = dy_i . (y_i - D x_i) - dt_i x_i . y'_i, plus
  <Gn, S_after> at each chunk's last token; dA = sum dt * suffix-sum(dcum);
* dC = sum_h of the output step with x'' = B, B'' = x, C'' = dy and carried
  state Sprev^T; dB = sum_h dt * (the reversed step with x'' = C, B'' = dy,
  C'' = x and carried state Gn^T).

Here the output step is written out in numpy from its definition (a plain
double loop), so these tests pin the decomposition itself, independently of the
kernels and of the oracle's own backward code.
"""
import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_02_gb300.workloads import Workload, make_grads, make_inputs


def output_step(x, B, C, c2, dtv, Sp, L):
    """y_t = sum_{s<=t, same chunk} (C_t.B_s) 2^(c2_t - c2_s) dt_s x_s + 2^(c2_t) Sp[c] C_t.
    x [T,P], B, C [T,N], c2, dtv [T], Sp [nc,P,N]."""
    T = x.shape[0]
    y = np.zeros_like(x)
    for c in range((T + L - 1) // L):
        t0, t1 = c * L, min(T, (c + 1) * L)
        for t in range(t0, t1):
            acc = 2.0 ** c2[t] * (Sp[c] @ C[t])
            for s in range(t0, t + 1):
                acc = acc + (C[t] @ B[s]) * 2.0 ** (c2[t] - c2[s]) * dtv[s] * x[s]
            y[t] = acc
    return y


def reversal(T, L):
    """Token t of chunk c (Lc tokens) <-> position c L + Lc - 1 - (t - c L)."""
    rev = np.zeros(T, dtype=int)
    for c in range((T + L - 1) // L):
        t0, t1 = c * L, min(T, (c + 1) * L)
        for k in range(t1 - t0):
            rev[t0 + k] = t1 - 1 - k
    return rev


def decomposed_backward(inp, gr, G, L):
    x, dt, A, Bm, Cm, D = inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"]
    dy, dfin = gr["dy"], gr["dfinal"]
    b, T, H, P = x.shape
    nc = (T + L - 1) // L
    hpg = H // G
    ch = oracle.ssd_chunked(**inp, ngroups=G, chunk_size=L)      # cum2, Sprev, final_state
    rev = reversal(T, L)
    out = dict(dx=np.zeros_like(x), ddt=np.zeros_like(dt), dA=np.zeros(H),
               dB=np.zeros_like(Bm), dC=np.zeros_like(Cm))
    for bb in range(b):
        for h in range(H):
            g = h // hpg
            c2, Sp = ch["cum2"][bb, h], ch["Sprev"][bb, :, h]
            last = [min(T, (c + 1) * L) - 1 for c in range(nc)]
            # adjoint of the state leaving each chunk (reverse pass over chunks)
            gv = dfin[bb, h].copy()
            Gn = [None] * nc
            for c in reversed(range(nc)):
                t0, t1 = c * L, last[c] + 1
                Gn[c] = gv.copy()
                gv = (2.0 ** c2[t0:t1, None] * dy[bb, t0:t1, h]).T @ Cm[bb, t0:t1, g] + \
                    2.0 ** c2[t1 - 1] * gv
            c2r = np.array([c2[last[t // L]] - c2[rev[t]] for t in range(T)])
            # y without the skip term, and y' (reversed run, natural order)
            yno = output_step(x[bb, :, h], Bm[bb, :, g], Cm[bb, :, g], c2, dt[bb, :, h], Sp, L)
            yr = output_step(dy[bb, rev, h], Cm[bb, rev, g], Bm[bb, rev, g], c2r, np.ones(T), Gn, L)
            yp = np.empty_like(yr)
            yp[rev] = yr
            out["dx"][bb, :, h] = dt[bb, :, h, None] * yp + D[h] * dy[bb, :, h]
            xy = np.sum(x[bb, :, h] * yp, 1)
            dcum = np.sum(dy[bb, :, h] * yno, 1) - dt[bb, :, h] * xy
            for c in range(nc):
                S_after = Sp[c + 1] if c + 1 < nc else ch["final_state"][bb, h]
                dcum[last[c]] += np.sum(Gn[c] * S_after)
                t0, t1 = c * L, last[c] + 1
                rcs = np.cumsum(dcum[t0:t1][::-1])[::-1]
                out["ddt"][bb, t0:t1, h] = xy[t0:t1] + A[h] * rcs
                out["dA"][h] += np.sum(dt[bb, t0:t1, h] * rcs)
            # the transposed-state runs
            out["dC"][bb, :, g] += output_step(Bm[bb, :, g], x[bb, :, h], dy[bb, :, h], c2,
                                               dt[bb, :, h], np.transpose(Sp, (0, 2, 1)), L)
            z = output_step(Cm[bb, rev, g], dy[bb, rev, h], x[bb, rev, h], c2r, np.ones(T),
                            [gn.T for gn in Gn], L)
            zz = np.empty_like(z)
            zz[rev] = z
            out["dB"][bb, :, g] += dt[bb, :, h, None] * zz
    return out


@pytest.mark.parametrize("shape", [(2, 37, 4, 3, 5, 2, 8, 0.3), (1, 40, 2, 4, 3, 1, 16, 0.0)],
                         ids=["groups-init-ragged", "one-group-no-init"])
def test_backward_decomposition_equals_the_gradient(shape):
    b, T, H, P, N, G, L, init = shape
    w = Workload("ident", b, T, H, P, N, G, L, dtype="f32", init_std=init, seed=9)
    inp = {k: (v.numpy().astype(np.float64) if v is not None else None)
           for k, v in make_inputs(w).items()}
    gr = {k: v.numpy().astype(np.float64) for k, v in make_grads(w).items()}
    ref = oracle.ssd_backward(**inp, **gr, ngroups=G)
    got = decomposed_backward(inp, gr, G, L)
    for k in got:
        rel = np.linalg.norm(got[k] - ref[k]) / np.linalg.norm(ref[k])
        assert rel < 1e-12, (k, rel)
