"""Pins for the oracle's backward pass, checked against things other than itself.

The pages give no backward method; they only note that end-to-end training
speed also depends on one ("NVIDIA、cuTileでMamba-2フォワードパスを高速化"
(ai.newsbites.today), "開発現場への影響と未確認事項"; "NVIDIA CUDA Tile로 Mamba-2
순방향 전달 커널 가속화" (devin.kr), "성능 벤치마크 결과 및 활용").  The oracle's
backward is the chain rule on the recurrence; what pins it here is:

* finite differences of the FORWARD oracle (a five-point stencil in fp64 on
  inputs chosen so that every perturbed value is exact in float32) for every
  element of every input of a small problem with groups and an initial state;
* the homogeneity of the loss L = sum(dy*y) + sum(dfinal*final_state): it is
  linear in (x, initial_state) jointly, y - D x is linear in C, and with a zero
  initial state y - D x and final_state are linear in B -- Euler's identity
  gives sum(grad * input) for each;
* dD = sum over (b, t) of dy . x (the skip term's closed form);
* sampled (b, h) pairs reproduce the full run.

``test_planted_backward_mistakes_are_caught`` compiles copies of the oracle with
one plausible slip each in the backward and checks that a pin rejects it.
"""
import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_02_gb300.workloads import Workload, make_grads, make_inputs

Q = 2.0 ** -12      # grid of x, B, C, A, D, init values
QDT = 2.0 ** -16    # grid of dt values
STEP = {"x": 2.0 ** -10, "B": 2.0 ** -10, "C": 2.0 ** -10, "initial_state": 2.0 ** -10,
        "D": 2.0 ** -10, "A": 2.0 ** -10, "dt": 2.0 ** -14}
GRAD = {"x": "dx", "B": "dB", "C": "dC", "initial_state": "dinit", "D": "dD", "A": "dA",
        "dt": "ddt"}


def problem(b=2, T=10, H=4, P=3, N=4, G=2, init=0.5, seed=11):
    """Inputs on a grid such that v +- 2*STEP is exact in float32 (values are
    small multiples of the grid), dt bounded away from 0."""
    w = Workload("bwdpin", b, T, H, P, N, G, 4, dtype="f32", dt_lo=2e-2, dt_hi=0.4,
                 init_std=init, seed=seed)
    inp = {k: (v.numpy().astype(np.float64) if v is not None else None)
           for k, v in make_inputs(w).items()}
    for k in ("x", "B", "C", "A", "D", "initial_state"):
        if inp[k] is not None:
            inp[k] = np.round(inp[k] / Q) * Q
    inp["dt"] = np.round(inp["dt"] / QDT) * QDT
    gr = {k: v.numpy().astype(np.float64) for k, v in make_grads(w).items()}
    return inp, gr, G


def loss(inp, gr, G, lib=None):
    y, fin = oracle.ssd_recurrent(**inp, ngroups=G, lib=lib)
    return float(np.sum(gr["dy"] * y) + np.sum(gr["dfinal"] * fin))


def fd_grad(inp, gr, G, name, idx, lib=None):
    h = STEP[name]
    vals = []
    for k in (2, 1, -1, -2):
        q = {kk: (v.copy() if v is not None else None) for kk, v in inp.items()}
        q[name][idx] += k * h
        assert np.float32(q[name][idx]) == q[name][idx]      # the perturbation is exact
        vals.append(loss(q, gr, G, lib))
    return (-vals[0] + 8 * vals[1] - 8 * vals[2] + vals[3]) / (12 * h)


def pin_finite_differences(lib=None):
    """Every element of every gradient against a five-point finite difference
    of the forward oracle."""
    inp, gr, G = problem()
    g = oracle.ssd_backward(**inp, **gr, ngroups=G, lib=lib)
    for name in ("x", "B", "C", "initial_state", "D", "A", "dt"):
        ref = g[GRAD[name]]
        scale = max(np.abs(ref).max(), 1.0)
        for idx in np.ndindex(*inp[name].shape):
            if abs(fd_grad(inp, gr, G, name, idx, lib) - ref[idx]) > 1e-8 * scale:
                return False
    return True


def pin_homogeneity(lib=None):
    ok = True
    for init in (0.5, 0.0):
        inp, gr, G = problem(init=init, seed=12)
        y, fin = oracle.ssd_recurrent(**inp, ngroups=G, lib=lib)
        g = oracle.ssd_backward(**inp, **gr, ngroups=G, lib=lib)
        L = np.sum(gr["dy"] * y) + np.sum(gr["dfinal"] * fin)
        dxD = np.sum(gr["dy"] * inp["x"] * inp["D"][None, None, :, None])
        tol = 1e-11 * (abs(L) + 1)
        s0 = inp["initial_state"] if inp["initial_state"] is not None else 0.0
        ok &= abs(np.sum(g["dx"] * inp["x"]) + np.sum(g["dinit"] * s0) - L) < tol
        ok &= abs(np.sum(g["dC"] * inp["C"]) - np.sum(gr["dy"] * y) + dxD) < tol
        if init == 0.0:
            ok &= abs(np.sum(g["dB"] * inp["B"]) - (L - dxD)) < tol
    return bool(ok)


def pin_skip_closed_form(lib=None):
    inp, gr, G = problem(seed=13)
    g = oracle.ssd_backward(**inp, **gr, ngroups=G, lib=lib)
    dD = np.einsum("bthp,bthp->h", gr["dy"], inp["x"])
    return bool(np.abs(g["dD"] - dD).max() < 1e-12 * (np.abs(dD).max() + 1))


def pin_quadratic_closed_forms(lib=None):
    """Brute force from the quadratic view of the recurrence (every decay the
    explicit sum of a_r = dt_r A between the two tokens):
        dinit = sum_t e^{a_0 + .. + a_t} dy_t C_t^T + e^{a_0 + .. + a_{T-1}} dfinal
        dx_s  = dt_s [sum_{t>=s} e^{a_{s+1} + .. + a_t} (C_t . B_s) dy_t
                      + e^{a_{s+1} + .. + a_{T-1}} dfinal B_s] + D dy_s"""
    inp, gr, G = problem(b=1, T=9, H=2, P=2, N=3, G=2, seed=17)
    g = oracle.ssd_backward(**inp, **gr, ngroups=G, lib=lib)
    x, dt, A, B, C, D = inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"]
    dy, dfin = gr["dy"], gr["dfinal"]
    T, H = x.shape[1], x.shape[2]
    ok = True
    for h in range(H):
        gg = h // (H // G)
        a = dt[0, :, h] * A[h]
        dinit = np.exp(a.sum()) * dfin[0, h]
        for t in range(T):
            dinit = dinit + np.exp(a[:t + 1].sum()) * np.outer(dy[0, t, h], C[0, t, gg])
        ok &= np.abs(g["dinit"][0, h] - dinit).max() < 1e-12 * (np.abs(dinit).max() + 1)
        for s_ in range(T):
            acc = np.exp(a[s_ + 1:].sum()) * (dfin[0, h] @ B[0, s_, gg])
            for t in range(s_, T):
                acc = acc + np.exp(a[s_ + 1:t + 1].sum()) * (C[0, t, gg] @ B[0, s_, gg]) * dy[0, t, h]
            dx = dt[0, s_, h] * acc + D[h] * dy[0, s_, h]
            ok &= np.abs(g["dx"][0, s_, h] - dx).max() < 1e-12 * (np.abs(dx).max() + 1)
    return bool(ok)


PINS = {"finite_differences": pin_finite_differences, "homogeneity": pin_homogeneity,
        "skip_closed_form": pin_skip_closed_form, "quadratic_closed_forms": pin_quadratic_closed_forms}


@pytest.mark.parametrize("name", sorted(PINS))
def test_backward_pin(name):
    assert PINS[name]()


def test_backward_without_dfinal_or_init():
    inp, gr, G = problem(init=0.0, seed=14)
    g0 = oracle.ssd_backward(**inp, dy=gr["dy"], dfinal=None, ngroups=G)
    g1 = oracle.ssd_backward(**inp, dy=gr["dy"], dfinal=np.zeros_like(gr["dfinal"]), ngroups=G)
    for k in g0:
        assert np.array_equal(g0[k], g1[k]), k


def test_backward_sampled_pairs_match_full():
    inp, gr, G = problem(seed=15)
    g = oracle.ssd_backward(**inp, **gr, ngroups=G)
    gs = oracle.ssd_backward(**inp, **gr, ngroups=G, pairs=[(1, 3), (0, 0)])
    assert np.array_equal(gs["dx"][1, :, 3], g["dx"][1, :, 3])
    assert np.array_equal(gs["ddt"][0, :, 0], g["ddt"][0, :, 0])
    assert np.array_equal(gs["dinit"][1, 3], g["dinit"][1, 3])
    assert np.isnan(gs["dx"][0, :, 1]).all()


def test_backward_long_sequence_segments():
    """T large enough for several checkpoint segments, against finite differences
    of a few dt and x entries (the segment recomputation must give the sweep's
    states)."""
    inp, gr, G = problem(b=1, T=70, H=2, P=2, N=3, G=1, seed=16)
    g = oracle.ssd_backward(**inp, **gr, ngroups=G)
    for name, idx in (("dt", (0, 3, 1)), ("dt", (0, 40, 0)), ("x", (0, 65, 1, 1)),
                      ("x", (0, 8, 0, 0)), ("B", (0, 33, 0, 2))):
        ref = g[GRAD[name]][idx]
        assert abs(fd_grad(inp, gr, G, name, idx) - ref) < 1e-8 * max(abs(ref), 1.0), (name, idx)


MUTANTS = {
    "bwd_ddt_drop_decay_term": ("ddt[(b * T + t) * H + h] = xgb + Ah * e * gs;",
                                "ddt[(b * T + t) * H + h] = xgb;"),
    "bwd_dB_drop_dt": ("qB[t * N + n] += dtv * ab;", "qB[t * N + n] += ab;"),
    "bwd_dC_previous_state": ("ac += Scur[p * N + n] * (double)dyt[p];",
                              "ac += Sprev[p * N + n] * (double)dyt[p];"),
    "bwd_adjoint_no_decay": ("for (int64_t k = 0; k < PN; ++k) Gs[k] *= e;",
                             "for (int64_t k = 0; k < PN; ++k) Gs[k] *= 1.0;"),
    "bwd_dx_drop_skip": ("dx[((b * T + t) * H + h) * P + p] = dtv * gb + Dh * (double)dyt[p];",
                         "dx[((b * T + t) * H + h) * P + p] = dtv * gb;"),
    "bwd_dA_drop_decay": ("sA += dtv * e * gs;", "sA += dtv * gs;"),
    "bwd_readout_after_decay": (
        "Gs[p * N + n] += (double)dyt[p] * (double)Ct[n];",
        "Gs[p * N + n] += e * (double)dyt[p] * (double)Ct[n];"),
    "bwd_group_interleaved": ("const int64_t g = h / hpg;\n            dA[h]",
                              "const int64_t g = h % G;\n            dA[h]"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_backward_mistakes_are_caught(name, tmp_path):
    find, repl = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(find) == 1, f"mutation anchor not unique/absent: {name}"
    mut = tmp_path / "ssd_oracle_mut.c"
    mut.write_text(src.replace(find, repl))
    lib = oracle.load_variant(str(mut), str(tmp_path / f"libmut_{name}.so"))
    failed = []
    for p, fn in PINS.items():
        try:
            with np.errstate(all="ignore"):
                if not fn(lib):
                    failed.append(p)
        except Exception:
            failed.append(p)
    assert failed, f"no pin caught mutation {name}"
