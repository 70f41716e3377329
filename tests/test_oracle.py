"""Pins for the fp64 oracle, checked against things other than itself.

Pages cited: [P2] "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr),
"Mamba-2 아키텍처의 핵심 연산" (y_t = c_t^T h_t + D x_t; decays as a log-space
cumulative sum of a_t; causal masking); [P3] "Accelerating Mamba-2 with
High-Performance Forward Pass Kernels in NVIDIA CUDA Tile" (brifing.si),
section 2 (chunkwise computation with a fixed-size state), section 4 (jump
formula), section 5 (log-space decay), section 11 (causal masking).

Each pin is a closed form, a special case that reduces to a textbook
computation, an invariant of the recurrence, or brute force on tiny inputs.
``test_planted_mistakes_are_caught`` compiles copies of the oracle with one
plausible mistake each and checks that the pins below reject every one.
"""
import math

import numpy as np
import pytest

import oracle
from mamba_ssd_chunked_02_gb300.workloads import Workload, make_inputs

RTOL = 1e-12


def _np(d):
    return {k: (v.numpy().astype(np.float64) if v is not None else None) for k, v in d.items()}


def small(b=2, T=24, H=4, P=3, N=5, G=2, L=8, init=0.1, seed=7, dt_lo=1e-2, dt_hi=0.5):
    w = Workload("pin", b, T, H, P, N, G, L, dtype="f32", dt_lo=dt_lo, dt_hi=dt_hi,
                 init_std=init, seed=seed)
    return _np(make_inputs(w))


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------- pins ---------------
# Each pin takes an optional oracle handle so that the planted-mistake test can
# re-run it against a mutated copy.  Each returns True when the pin holds.

def pin_bruteforce(lib=None):
    """Quadratic (every decay summed explicitly) == recurrence, tiny inputs."""
    ok = True
    for shp in [dict(b=2, T=17, H=4, P=3, N=5, G=2), dict(b=1, T=9, H=2, P=4, N=2, G=1),
                dict(b=1, T=12, H=3, P=2, N=3, G=3)]:
        inp = small(**shp)
        G = shp["G"]
        y1, f1 = oracle.ssd_recurrent(**inp, ngroups=G, lib=lib)
        y2, f2 = oracle.ssd_quadratic(**inp, ngroups=G, lib=lib)
        ok &= rel(y1, y2) < RTOL and rel(f1, f2) < RTOL
    return ok


def pin_chunk_independence(lib=None):
    """The chunked form equals the recurrence for every chunk length, including
    L = 1 (the recurrence itself), L = T (the quadratic view) and ragged tails."""
    inp = small(b=2, T=17, H=4, P=3, N=5, G=2)
    y, f = oracle.ssd_recurrent(**inp, ngroups=2, lib=lib)
    ok = True
    for L in (1, 2, 3, 4, 5, 8, 16, 17, 32):
        o = oracle.ssd_chunked(**inp, ngroups=2, chunk_size=L, lib=lib)
        ok &= rel(o["y"], y) < RTOL and rel(o["final_state"], f) < RTOL
    return ok


def pin_linear_attention(lib=None, form="recurrent"):
    """A = 0: no decay, so y_t = (S0 + sum_{s<=t} dt_s x_s B_s^T) C_t + D x_t,
    causal linear attention computed here by prefix sums (np.cumsum)."""
    inp = small(b=1, T=20, H=2, P=3, N=4, G=1)
    inp["A"] = np.zeros_like(inp["A"])
    x, dt, B, C, D, S0 = (inp[k] for k in ("x", "dt", "B", "C", "D", "initial_state"))
    kv = np.einsum("bth,bthp,btn->bthpn", dt, x, B[:, :, 0])      # dt_s x_s B_s^T
    S = np.cumsum(kv, axis=1) + S0[:, None]                      # prefix sums over t
    y_ref = np.einsum("bthpn,btn->bthp", S, C[:, :, 0]) + D[None, None, :, None] * x
    if form == "recurrent":
        y, f = oracle.ssd_recurrent(**inp, ngroups=1, lib=lib)
    else:
        o = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=6, lib=lib)
        y, f = o["y"], o["final_state"]
    return rel(y, y_ref) < RTOL and rel(f, S[:, -1]) < RTOL


def pin_impulse(lib=None, form="recurrent"):
    """x nonzero only at t0, no initial state: y_t = 0 for t < t0 and
    y_t = exp(sum_{r=t0+1}^{t} dt_r A) dt_t0 (C_t . B_t0) x_t0 + [t==t0] D x_t0."""
    inp = small(b=1, T=16, H=2, P=3, N=4, G=1, init=0.0)
    t0 = 5
    x = np.zeros_like(inp["x"])
    x[:, t0] = inp["x"][:, t0]
    inp["x"] = x
    dt, A, B, C, D = (inp[k] for k in ("dt", "A", "B", "C", "D"))
    T, H = x.shape[1], x.shape[2]
    y_ref = np.zeros_like(x)
    for h in range(H):
        for t in range(t0, T):
            decay = math.exp(sum(dt[0, r, h] * A[h] for r in range(t0 + 1, t + 1)))
            y_ref[0, t, h] = decay * dt[0, t0, h] * float(C[0, t, 0] @ B[0, t0, 0]) * x[0, t0, h]
        y_ref[0, t0, h] += D[h] * x[0, t0, h]
    if form == "recurrent":
        y, _ = oracle.ssd_recurrent(**inp, ngroups=1, lib=lib)
    else:
        y = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=4, lib=lib)["y"]
    return rel(y, y_ref) < RTOL


def pin_dt_zero(lib=None):
    """dt = 0: no input and decay 1, so the state stays S0: y_t = S0 C_t + D x_t."""
    inp = small(b=1, T=10, H=2, P=3, N=4, G=1)
    inp["dt"] = np.zeros_like(inp["dt"])
    S0, C, D, x = inp["initial_state"], inp["C"], inp["D"], inp["x"]
    y_ref = np.einsum("bhpn,btn->bthp", S0, C[:, :, 0]) + D[None, None, :, None] * x
    ok = True
    for fn in ("r", "c"):
        if fn == "r":
            y, f = oracle.ssd_recurrent(**inp, ngroups=1, lib=lib)
        else:
            o = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=4, lib=lib)
            y, f = o["y"], o["final_state"]
        ok &= rel(y, y_ref) < RTOL and rel(f, S0) < RTOL
    return ok


def pin_geometric(lib=None, form="recurrent"):
    """P = N = 1, constant dt, A, x = B = C = 1: the state is a geometric series,
    S_t = dt (1 - e^{a(t+1)}) / (1 - e^a) with a = dt*A, and y_t = S_t + D."""
    T = 13
    dtv, Av, Dv = 0.3, -1.7, 0.25
    a = dtv * Av
    ones = np.ones((1, T, 1, 1))
    inp = dict(x=ones, dt=np.full((1, T, 1), dtv), A=np.array([Av]), B=ones, C=ones,
               D=np.array([Dv]), initial_state=None)
    t = np.arange(T)
    S_ref = dtv * (1 - np.exp(a * (t + 1))) / (1 - np.exp(a))
    if form == "recurrent":
        y, f = oracle.ssd_recurrent(**inp, ngroups=1, lib=lib)
    else:
        o = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=5, lib=lib)
        y, f = o["y"], o["final_state"]
    # float32 widening of dt, A: compare against the same rounded constants.
    dt32, A32 = float(np.float32(dtv)), float(np.float32(Av))
    a32 = dt32 * A32
    S_ref = dt32 * (1 - np.exp(a32 * (t + 1))) / (1 - np.exp(a32))
    return (rel(y[0, :, 0, 0], S_ref + float(np.float32(Dv))) < 1e-12
            and abs(f[0, 0, 0, 0] - S_ref[-1]) < 1e-12)


def pin_carried_state(lib=None, form="chunked"):
    """x = 0: only the initial state, decayed: y_t = exp(sum_{r<=t} dt_r A) S0 C_t."""
    inp = small(b=1, T=18, H=2, P=3, N=4, G=1)
    inp["x"] = np.zeros_like(inp["x"])
    dt, A, C, S0 = inp["dt"], inp["A"], inp["C"], inp["initial_state"]
    dec = np.exp(np.cumsum(dt[0] * A[None, :], axis=0))              # [T, H]
    y_ref = np.einsum("th,hpn,tn->thp", dec, S0[0], C[0, :, 0])[None]
    if form == "recurrent":
        y, f = oracle.ssd_recurrent(**inp, ngroups=1, lib=lib)
    else:
        o = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=7, lib=lib)
        y, f = o["y"], o["final_state"]
    return rel(y, y_ref) < RTOL and rel(f[0], dec[-1][:, None, None] * S0[0]) < RTOL


def pin_group_mapping(lib=None):
    """Head h reads group h // (H/G): G = 2 equals G = H with B, C repeated in
    contiguous head blocks, and differs from an interleaved assignment."""
    inp = small(b=1, T=9, H=4, P=2, N=3, G=2)
    y, _ = oracle.ssd_recurrent(**inp, ngroups=2, lib=lib)
    rep = dict(inp)
    rep["B"] = np.repeat(inp["B"], 2, axis=2)
    rep["C"] = np.repeat(inp["C"], 2, axis=2)
    y_rep, _ = oracle.ssd_recurrent(**rep, ngroups=4, lib=lib)
    inter = dict(inp)
    inter["B"] = np.tile(inp["B"], (1, 1, 2, 1))
    inter["C"] = np.tile(inp["C"], (1, 1, 2, 1))
    y_int, _ = oracle.ssd_recurrent(**inter, ngroups=4, lib=lib)
    yc = oracle.ssd_chunked(**inp, ngroups=2, chunk_size=4, lib=lib)["y"]
    return rel(y, y_rep) < RTOL and rel(y, y_int) > 1e-3 and rel(yc, y_rep) < RTOL


def pin_split_resume(lib=None, form="chunked"):
    """Running [0, T/2) then [T/2, T) from the mid state equals one run.
    The mid state passes through float32 (the oracle's input type), hence 1e-6."""
    inp = small(b=2, T=24, H=2, P=3, N=4, G=1)
    fn = (lambda d: oracle.ssd_recurrent(**d, ngroups=1, lib=lib)) if form == "recurrent" else \
        (lambda d: (lambda o: (o["y"], o["final_state"]))(
            oracle.ssd_chunked(**d, ngroups=1, chunk_size=5, lib=lib)))
    y, f = fn(inp)
    first = {k: v for k, v in inp.items()}
    second = {k: v for k, v in inp.items()}
    for k in ("x", "dt", "B", "C"):
        first[k] = inp[k][:, :12]
        second[k] = inp[k][:, 12:]
    y1, f1 = fn(first)
    second["initial_state"] = f1
    y2, f2 = fn(second)
    return rel(np.concatenate([y1, y2], axis=1), y) < 1e-6 and rel(f2, f) < 1e-6


def pin_stage_intermediates(lib=None):
    """Chunked intermediates against the definition: exp2(cum2 at a chunk's last
    token) is the product of the per-token decays exp(dt_r A) over that chunk
    (the log-space identity); dS_c is the recurrence run over chunk c alone from
    a zero state; Sprev_c is the recurrence's state after the first c chunks."""
    inp = small(b=1, T=20, H=2, P=3, N=4, G=1)
    L = 8
    o = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=L, lib=lib)
    dt, A = inp["dt"][0], inp["A"]
    ok = True
    for c in range(3):
        t0, t1 = c * L, min((c + 1) * L, 20)
        prod = np.prod(np.exp(dt[t0:t1] * A[None, :]), axis=0)          # [H]
        ok &= rel(np.exp2(o["cum2"][0, :, t1 - 1]), prod) < RTOL
        part = {k: v for k, v in inp.items()}
        for k in ("x", "dt", "B", "C"):
            part[k] = inp[k][:, t0:t1]
        part["initial_state"] = None
        _, f_chunk = oracle.ssd_recurrent(**part, ngroups=1, lib=lib)
        ok &= rel(o["dS"][:, c], f_chunk) < RTOL
        if c > 0:
            pre = {k: v for k, v in inp.items()}
            for k in ("x", "dt", "B", "C"):
                pre[k] = inp[k][:, :t0]
            _, f_pre = oracle.ssd_recurrent(**pre, ngroups=1, lib=lib)
            ok &= rel(o["Sprev"][:, c], f_pre) < RTOL
        else:
            ok &= rel(o["Sprev"][:, 0], inp["initial_state"]) < RTOL
    return ok


def pin_causality(lib=None):
    """y_t does not depend on inputs after t (the causal mask)."""
    inp = small(b=1, T=16, H=2, P=3, N=4, G=1)
    o1 = oracle.ssd_chunked(**inp, ngroups=1, chunk_size=8, lib=lib)["y"]
    pert = {k: (v.copy() if v is not None else None) for k, v in inp.items()}
    t1 = 11
    for k in ("x", "B", "C"):
        pert[k][:, t1:] += 1.0
    pert["dt"][:, t1:] *= 2.0
    o2 = oracle.ssd_chunked(**pert, ngroups=1, chunk_size=8, lib=lib)["y"]
    return np.array_equal(o1[:, :t1], o2[:, :t1]) and not np.allclose(o1[:, t1:], o2[:, t1:])


def pin_linearity(lib=None):
    """y is linear in (x, initial_state): scaling by 2^k scales y and final_state
    by 2^k, and inputs with disjoint supports add.  Both are exact in float32."""
    i1 = small(b=1, T=12, H=2, P=3, N=4, G=1, seed=11)
    odd = (np.arange(12) % 2 == 1)[None, :, None, None]
    xa = np.where(odd, i1["x"], 0.0)
    xb = np.where(odd, 0.0, i1["x"])
    ok = True
    for form in ("r", "c"):
        def run(x, s0):
            d = dict(i1, x=x, initial_state=s0)
            if form == "r":
                return oracle.ssd_recurrent(**d, ngroups=1, lib=lib)
            o = oracle.ssd_chunked(**d, ngroups=1, chunk_size=5, lib=lib)
            return o["y"], o["final_state"]
        y, f = run(i1["x"], i1["initial_state"])
        y4, f4 = run(4.0 * i1["x"], 4.0 * i1["initial_state"])
        ya, fa = run(xa, i1["initial_state"])
        yb, fb = run(xb, None)
        ok &= rel(y4, 4.0 * y) < RTOL and rel(f4, 4.0 * f) < RTOL
        ok &= rel(ya + yb, y) < RTOL and rel(fa + fb, f) < RTOL
    return ok


PINS = {
    "bruteforce": pin_bruteforce,
    "chunk_independence": pin_chunk_independence,
    "linear_attention_recurrent": lambda lib=None: pin_linear_attention(lib, "recurrent"),
    "linear_attention_chunked": lambda lib=None: pin_linear_attention(lib, "chunked"),
    "impulse_recurrent": lambda lib=None: pin_impulse(lib, "recurrent"),
    "impulse_chunked": lambda lib=None: pin_impulse(lib, "chunked"),
    "dt_zero": pin_dt_zero,
    "geometric_recurrent": lambda lib=None: pin_geometric(lib, "recurrent"),
    "geometric_chunked": lambda lib=None: pin_geometric(lib, "chunked"),
    "carried_state_recurrent": lambda lib=None: pin_carried_state(lib, "recurrent"),
    "carried_state_chunked": lambda lib=None: pin_carried_state(lib, "chunked"),
    "group_mapping": pin_group_mapping,
    "split_resume_recurrent": lambda lib=None: pin_split_resume(lib, "recurrent"),
    "split_resume_chunked": lambda lib=None: pin_split_resume(lib, "chunked"),
    "stage_intermediates": pin_stage_intermediates,
    "causality": pin_causality,
    "linearity": pin_linearity,
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    assert PINS[name](), name


def test_oracle_rejects_bad_shapes():
    inp = small(b=1, T=4, H=3, P=2, N=2, G=1)
    with pytest.raises(ValueError):
        oracle.ssd_chunked(**inp, ngroups=1, chunk_size=0)
    bad = dict(inp)
    bad["B"] = np.zeros((1, 4, 2, 2))
    bad["C"] = np.zeros((1, 4, 2, 2))
    with pytest.raises(ValueError):
        oracle.ssd_recurrent(**bad, ngroups=2)      # 3 heads, 2 groups


def test_sampled_pairs_match_full():
    inp = small(b=2, T=10, H=4, P=3, N=4, G=2)
    y, f = oracle.ssd_recurrent(**inp, ngroups=2)
    ys, fs = oracle.ssd_recurrent(**inp, ngroups=2, pairs=[(1, 3), (0, 1)])
    assert np.array_equal(ys[1, :, 3], y[1, :, 3]) and np.array_equal(fs[0, 1], f[0, 1])
    assert np.isnan(ys[0, :, 0]).all()


# ------------------------------------------------ planted mistakes -------------------
# Each mutation is a (find, replace) on the oracle source, a plausible slip: a
# dropped term, a wrong sign, an off-by-one index, a transposed operand, a wrong
# scale.  The pins must reject every one.
MUTANTS = {
    "recurrent_decay_sign": ("const double decay = exp(dtv * Ah);",
                             "const double decay = exp(-dtv * Ah);"),
    "recurrent_drop_dt_input": ("const double u = dtv * (double)xt[p];",
                                "const double u = (double)xt[p];"),
    "recurrent_drop_skip": ("yt[p] = acc + Dh * (double)xt[p];", "yt[p] = acc;"),
    "recurrent_readout_before_update": (
        "Sp[n] = decay * Sp[n] + u * (double)Bt_[n];\n                    acc += Sp[n] * (double)Ct[n];",
        "acc += Sp[n] * (double)Ct[n];\n                    Sp[n] = decay * Sp[n] + u * (double)Bt_[n];"),
    "recurrent_group_interleaved": ("const int64_t g = h / hpg;\n        double* S",
                                    "const int64_t g = h % G;\n        double* S"),
    "chunk_cumsum_no_reset": ("double run = 0.0;\n            for (int64_t t = c * L;",
                              "static double run = 0.0;\n            for (int64_t t = c * L;"),
    "chunk_cumsum_no_log2e": ("cum2[t] = LOG2E_D * run;", "cum2[t] = run;"),
    "chunk_state_wrong_last": ("const double last = cum2[t1 - 1];",
                               "const double last = cum2[t0];"),
    "chunk_state_drop_dt": ("const double w = exp2(last - cum2[s]) * (double)dt[(b * T + s) * H + h];",
                            "const double w = exp2(last - cum2[s]);"),
    "state_pass_no_decay": ("S[k] = chunk_decay * S[k] + dS[c * PN + k];",
                            "S[k] = S[k] + dS[c * PN + k];"),
    "state_pass_sprev_after": (
        "memcpy(Sp + c * PN, S, (size_t)PN * sizeof(double));\n            for (int64_t k = 0; k < PN; ++k) S[k] = chunk_decay * S[k] + dS[c * PN + k];",
        "for (int64_t k = 0; k < PN; ++k) S[k] = chunk_decay * S[k] + dS[c * PN + k];\n            memcpy(Sp + c * PN, S, (size_t)PN * sizeof(double));"),
    "out_carry_no_decay": ("const double carry = exp2(cum2[t]);", "const double carry = 1.0;"),
    "out_mask_strict": ("for (int64_t s = t0; s <= t; ++s) {", "for (int64_t s = t0; s < t; ++s) {"),
    "out_decay_reversed": ("cb * exp2(cum2[t] - cum2[s])", "cb * exp2(cum2[s] - cum2[t])"),
    "out_dt_of_t": ("exp2(cum2[t] - cum2[s]) * (double)dt[(b * T + s) * H + h];",
                    "exp2(cum2[t] - cum2[s]) * (double)dt[(b * T + t) * H + h];"),
    "out_state_transposed": ("acc += Sc[p * N + n] * (double)Ct[n];",
                             "acc += Sc[(n % P) * N + (p % N)] * (double)Ct[n];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    find, repl = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(find) == 1, f"mutation anchor not unique/absent: {name}"
    mut = tmp_path / "ssd_oracle_mut.c"
    mut.write_text(src.replace(find, repl))
    lib = oracle.load_variant(str(mut), str(tmp_path / f"libmut_{name}.so"))
    failed = [p for p, fn in PINS.items() if not _safe(fn, lib)]
    assert failed, f"no pin caught mutation {name}"


def _safe(fn, lib):
    try:
        with np.errstate(all="ignore"):
            return bool(fn(lib))
    except Exception:
        return False
