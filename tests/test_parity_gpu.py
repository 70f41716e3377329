"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Element-by-element comparisons at sizes the oracle finishes in seconds (several
tiles, ragged tails, grouped heads, an initial state), stage by stage and end
to end; full-size workloads in the benchmark's launch configuration on sampled
(batch, head) pairs recomputed by the recurrent oracle; edge cases.
"""
import numpy as np
import pytest
import torch

import mamba_ssd_chunked_02_gb300 as m2
import oracle
from mamba_ssd_chunked_02_gb300 import workloads as W
from parity import (TOL, assert_close, assert_close_sampled, metrics, run_fwd, sample_pairs,
                    sample_pairs_with_row, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_02_gb300 import build
    build.build()
    m2.load()
    m2.device_error(clear=True)


def wl(b, T, H, P, N, G, L, dtype="bf16", init=0.0, seed=1, dt_lo=1e-3, dt_hi=1e-1):
    return W.Workload(f"t b{b} T{T} H{H} P{P} N{N} G{G} L{L} {dtype}", b, T, H, P, N, G, L,
                      dtype=dtype, dt_lo=dt_lo, dt_hi=dt_hi, init_std=init, seed=seed)


SMALL = [
    wl(1, 256, 2, 16, 16, 1, 64, dtype="f32", seed=1001),              # the tiny fp32 workload
    wl(2, 512, 4, 64, 128, 1, 256, seed=11),                            # 2.7B head/state shape
    wl(1, 700, 3, 64, 128, 1, 256, seed=12),                            # ragged tail, odd heads
    wl(2, 384, 16, 64, 128, 8, 128, init=0.1, seed=13),                 # groups + initial state
    wl(1, 1024, 2, 64, 64, 1, 256, seed=14),                            # N = 64
    wl(1, 512, 2, 64, 256, 1, 256, seed=15),                            # N = 256
    wl(1, 640, 2, 64, 128, 1, 256, seed=16, dt_lo=1e-4),                # wide decay range
    wl(1, 300, 4, 128, 64, 2, 128, init=0.1, seed=17),                  # P = 128, ragged
    wl(2, 600, 4, 128, 128, 2, 256, init=0.1, seed=22),                 # P = 128, L = 256, groups
    wl(2, 500, 4, 64, 128, 2, 64, init=0.1, seed=23),                   # L = 64 (whole path: 128)
    # P = 32 on 64-column tiles that also hold the next head's columns: groups
    # (the next head in another group), a ragged tail and the last head (its
    # neighbour columns past the tensor); L = 128 with N = 64; L = 64 (whole path)
    wl(2, 600, 6, 32, 128, 2, 256, init=0.1, seed=24),
    wl(1, 384, 4, 32, 64, 1, 128, seed=25),
    wl(1, 500, 2, 32, 128, 1, 64, init=0.1, seed=26),
    wl(1, 200, 4, 32, 32, 2, 64, seed=18),                              # small P/N, bf16 SIMT
    wl(2, 192, 3, 16, 16, 3, 64, dtype="f32", init=0.1, seed=19),       # fp32, G = H
    wl(1, 100, 2, 64, 128, 1, 256, seed=20),                            # T < L
    wl(1, 1, 2, 64, 128, 1, 128, seed=21),                              # a single token
]


def _ids(ws):
    return [w.name[2:] for w in ws]


@pytest.mark.parametrize("w", SMALL, ids=_ids(SMALL))
def test_fwd_matches_oracle(w):
    inp = W.make_inputs(w)
    y, f = run_fwd(inp, w)
    ref = oracle.ssd_chunked(**inp, ngroups=w.ngroups, chunk_size=w.chunk_size)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    assert np.abs(ref["y"] - yr).max() <= 1e-9 * max(1.0, np.abs(yr).max())
    assert_close(to_np(y), yr, w.dtype, f"y {w.name}")
    assert_close(to_np(f), fr, w.dtype, f"final_state {w.name}")


TC_SMALL = SMALL[1:13]  # bf16 shapes on the tensor-core path (P = 128 as 2H heads of 64)


@pytest.mark.parametrize("w", TC_SMALL, ids=_ids(TC_SMALL))
def test_stages_match_oracle(w):
    """Each stage against the oracle's chunked intermediates."""
    inp = W.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    b, T, H, P, N, nc = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, sh.nchunks
    ref = oracle.ssd_chunked(**inp, ngroups=w.ngroups, chunk_size=w.chunk_size)
    f32 = dict(dtype=torch.float32, device="cuda")

    cum2 = torch.empty((b, H, T), **f32)
    dtT = torch.empty((b, H, T), **f32)
    m2.chunk_cumsum(sh, dev["dt"], dev["A"], cum2, dtT)
    torch.cuda.synchronize()
    rel, _ = metrics(to_np(cum2), ref["cum2"])
    assert rel <= 1e-5, f"cum2 relL2 {rel:.3e}"
    assert torch.equal(dtT.cpu(), inp["dt"].permute(0, 2, 1).contiguous())

    dS = torch.empty((b, nc, H, P, N), **f32)
    m2.chunk_state(sh, dev["x"], dev["B"], cum2, dtT, dS)
    torch.cuda.synchronize()
    assert_close(to_np(dS), ref["dS"], w.dtype, "dS")

    # Stage 3 from the oracle's dS (rounded to fp32), so it is checked on its own.
    dS_ref = torch.from_numpy(ref["dS"]).float().cuda()
    Sprev = torch.empty((b, nc, H, P, N), dtype=w.torch_dtype, device="cuda")
    fin = torch.empty((b, H, P, N), **f32)
    m2.state_pass(sh, dS_ref, cum2, dev["initial_state"], Sprev, fin)
    torch.cuda.synchronize()
    assert_close(to_np(Sprev), ref["Sprev"], w.dtype, "Sprev")
    assert_close(to_np(fin), ref["final_state"], w.dtype, "final_state")

    # Stage 4 from the oracle's Sprev (rounded to the I/O dtype).
    Sp_ref = torch.from_numpy(ref["Sprev"]).to(w.torch_dtype).cuda()
    y = torch.empty((b, T, H, P), dtype=w.torch_dtype, device="cuda")
    m2.chunk_out(sh, dev["x"], dev["B"], dev["C"], cum2, dtT, Sp_ref, dev["D"], y)
    torch.cuda.synchronize()
    assert_close(to_np(y), ref["y"], w.dtype, "y")
    assert m2.device_error() == 0


@pytest.mark.parametrize("w", TC_SMALL, ids=_ids(TC_SMALL))
def test_tensor_core_path_matches_cuda_core_path(w):
    """Both paths are within the tolerance of the oracle (checked above); by the
    triangle inequality they are within twice that tolerance of each other (two
    bf16-rounded outputs may differ by a whole ulp where |y| is large)."""
    inp = W.make_inputs(w)
    y0, f0 = run_fwd(inp, w, flags=m2.FLAG_FORCE_SIMT)
    y1, f1 = run_fwd(inp, w)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    for got, ref in ((y0, yr), (y1, yr), (f0, fr), (f1, fr)):
        assert_close(to_np(got), ref, w.dtype, "vs oracle")
    rel_tol, max_tol = TOL[w.dtype]
    for a, b_, ref in ((y1, y0, yr), (f1, f0, fr)):
        d = to_np(a) - to_np(b_)
        rms = np.sqrt(np.mean(ref ** 2))
        assert np.linalg.norm(d) <= 2 * rel_tol * np.linalg.norm(ref)
        assert np.abs(d).max() <= 2 * max_tol * rms


FUSED = [
    wl(2, 1024, 8, 64, 128, 1, 256, seed=31),                           # 4 chunks
    wl(1, 768, 2, 64, 256, 1, 256, seed=32),                            # N = 256: two n-tiles
    wl(2, 640, 16, 64, 128, 4, 128, init=0.1, seed=33),                 # L = 128, ragged, groups, init
    wl(1, 2048, 4, 64, 64, 1, 256, seed=34),                            # N = 64, 8 chunks
    wl(1, 1024, 4, 128, 128, 2, 256, seed=35),                          # P = 128: 8 heads of 64
]


def run_stages(inp, w):
    """The four stage entry points in a row (dS in fp32 between stages 2 and 3)."""
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    b, T, H, P, N, nc = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, sh.nchunks
    f32 = dict(dtype=torch.float32, device="cuda")
    cum2, dtT = torch.empty((b, H, T), **f32), torch.empty((b, H, T), **f32)
    dS = torch.empty((b, nc, H, P, N), **f32)
    Sp = torch.empty((b, nc, H, P, N), dtype=w.torch_dtype, device="cuda")
    f = torch.empty((b, H, P, N), **f32)
    y = torch.empty((b, T, H, P), dtype=w.torch_dtype, device="cuda")
    m2.chunk_cumsum(sh, dev["dt"], dev["A"], cum2, dtT)
    m2.chunk_state(sh, dev["x"], dev["B"], cum2, dtT, dS)
    m2.state_pass(sh, dS, cum2, dev["initial_state"], Sp, f)
    m2.chunk_out(sh, dev["x"], dev["B"], dev["C"], cum2, dtT, Sp, dev["D"], y)
    torch.cuda.synchronize()
    assert m2.device_error() == 0
    return y, f


@pytest.mark.parametrize("w", FUSED, ids=_ids(FUSED))
def test_fused_state_pass_matches_separate_kernels(w):
    """Stages 2+3 fused (carried state handed from chunk to chunk between CTAs)
    against the stage entry points with dS in fp32: the same fp32 operations in
    the same order (S = fma(decay, S, dS), Sprev rounded to bf16), so the outputs
    are equal bit for bit; the fused call is also checked against the oracle."""
    assert m2.path(m2.make_shape(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                                 w.chunk_size)) == m2.PATH_TCGEN05
    inp = W.make_inputs(w)
    y0, f0 = run_stages(inp, w)
    y1, f1 = run_fwd(inp, w, flags=m2.FLAG_FUSED_STATE)
    assert torch.equal(y0, y1)
    assert torch.equal(f0, f1)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    assert_close(to_np(y1), yr, w.dtype, f"y {w.name}")
    assert_close(to_np(f1), fr, w.dtype, f"final_state {w.name}")


@pytest.mark.parametrize("w", FUSED, ids=_ids(FUSED))
def test_bf16_dS_hand_off_stays_within_its_rounding(w):
    """The whole-path call moves dS from stage 2 to stage 3 in bf16 on the
    tensor-core path.  Each chunk's dS then carries a relative rounding error of
    at most 2^-9, and every carried state is a decayed sum of those, so the final
    state differs from the fp32 hand-off by well under 2^-8 relative (bound used:
    4e-3 in relative L2), and y (whose carried-state term reads Sprev) by less."""
    inp = W.make_inputs(w)
    y0, f0 = run_stages(inp, w)
    y1, f1 = run_fwd(inp, w)
    rel_f, _ = metrics(to_np(f1), to_np(f0))
    rel_y, _ = metrics(to_np(y1), to_np(y0))
    assert rel_f <= 4e-3, rel_f
    assert rel_y <= 4e-3, rel_y
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    assert_close(to_np(y1), yr, w.dtype, f"y {w.name}")
    assert_close(to_np(f1), fr, w.dtype, f"final_state {w.name}")


@pytest.mark.parametrize("w", FUSED[:3], ids=_ids(FUSED[:3]))
def test_fused_stage_entry_point_matches_stages(w):
    """mamba2_ssd_chunk_state_pass against mamba2_ssd_chunk_state followed by
    mamba2_ssd_state_pass: Sprev and final_state equal bit for bit."""
    inp = W.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    b, T, H, P, N, nc = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, sh.nchunks
    f32 = dict(dtype=torch.float32, device="cuda")
    cum2, dtT = torch.empty((b, H, T), **f32), torch.empty((b, H, T), **f32)
    m2.chunk_cumsum(sh, dev["dt"], dev["A"], cum2, dtT)
    dS = torch.empty((b, nc, H, P, N), **f32)
    sp0 = torch.empty((b, nc, H, P, N), dtype=torch.bfloat16, device="cuda")
    f0 = torch.empty((b, H, P, N), **f32)
    m2.chunk_state(sh, dev["x"], dev["B"], cum2, dtT, dS)
    m2.state_pass(sh, dS, cum2, dev["initial_state"], sp0, f0)
    sp1, f1 = torch.full_like(sp0, float("nan")), torch.full_like(f0, float("nan"))
    ws = torch.empty(m2.chunk_state_pass_workspace_size(sh), dtype=torch.uint8, device="cuda")
    m2.chunk_state_pass(sh, dev["x"], dev["B"], cum2, dtT, dev["initial_state"], sp1, f1, ws)
    torch.cuda.synchronize()
    assert m2.device_error() == 0
    assert torch.equal(sp0, sp1)
    assert torch.equal(f0, f1)


def test_fused_path_repeats_exactly():
    """The fused kernel's CTAs take work items from a ticket counter and wait for
    each other through flag words that stage 1 clears: running the same call
    again (same workspace, flags left set by the first run) gives the same bits."""
    w = FUSED[0]
    inp = W.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    ws = torch.empty(m2.workspace_size(sh), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        outs.append(m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                               dev["initial_state"], chunk_size=w.chunk_size, ngroups=w.ngroups,
                               workspace=ws, flags=m2.FLAG_FUSED_STATE))
    torch.cuda.synchronize()
    assert m2.device_error() == 0
    for y, f in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(f, outs[0][1])


@pytest.mark.parametrize("w", TC_SMALL, ids=_ids(TC_SMALL))
def test_overlapped_launches_match_serial(w):
    """Stages 2-4 start early by programmatic dependent launch and read their
    predecessor's outputs only after it completed: the outputs equal those of
    strictly serial launches bit for bit, on every repetition."""
    inp = W.make_inputs(w)
    y0, f0 = run_fwd(inp, w, flags=m2.FLAG_SERIAL)
    for _ in range(3):
        y1, f1 = run_fwd(inp, w)
        assert torch.equal(y0, y1) and torch.equal(f0, f1)


STRIDED = [
    wl(2, 640, 4, 64, 128, 1, 256, seed=51),                            # tensor-core shape
    wl(1, 520, 2, 128, 64, 1, 128, seed=53),                            # tensor cores, P = 128
    wl(1, 300, 4, 32, 32, 2, 64, dtype="f32", init=0.1, seed=52),       # CUDA-core shape
]


@pytest.mark.parametrize("pad", [0, 1], ids=["pitch16", "odd-pitch"])
@pytest.mark.parametrize("w", STRIDED, ids=_ids(STRIDED))
def test_strided_inputs_and_output(w, pad):
    """x, B and C as column slices of one projection output [b, T, H*P + 2*G*N
    (+1)], dt a slice of [b, T, H + 3] and y written into a wider buffer, through
    mamba2_ssd_fwd_strided.  With row pitches that are multiples of 16 bytes the
    same kernels run as for contiguous tensors and the outputs are equal bit for
    bit; an odd pitch takes the CUDA-core kernels (the tensor-core kernels' copies
    need 16-byte strides) and is checked against the oracle.  The padding of the
    output buffer is left untouched."""
    inp = W.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    b, T, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    HP, GN = H * P, G * N
    xbc = torch.zeros((b, T, HP + 2 * GN + pad), dtype=w.torch_dtype, device="cuda")
    xbc[..., :HP] = dev["x"].reshape(b, T, HP)
    xbc[..., HP:HP + GN] = dev["B"].reshape(b, T, GN)
    xbc[..., HP + GN:HP + 2 * GN] = dev["C"].reshape(b, T, GN)
    x = xbc[..., :HP].view(b, T, H, P)
    Bv = xbc[..., HP:HP + GN].view(b, T, G, N)
    Cv = xbc[..., HP + GN:HP + 2 * GN].view(b, T, G, N)
    dtb = torch.zeros((b, T, H + 3), dtype=torch.float32, device="cuda")
    dtb[..., :H] = dev["dt"]
    ypitch = HP + (1 if pad else 8)
    yb = torch.full((b, T, ypitch), float("nan"), dtype=w.torch_dtype, device="cuda")
    y = yb[..., :HP].view(b, T, H, P)
    _, f1 = m2.ssd_fwd(x, dtb[..., :H], dev["A"], Bv, Cv, dev["D"], dev["initial_state"],
                       chunk_size=w.chunk_size, ngroups=G, y=y)
    torch.cuda.synchronize()
    assert m2.device_error() == 0
    assert torch.isnan(yb[..., HP:].float()).all()
    y0, f0 = run_fwd(inp, w)
    simt = m2.path(m2.make_shape(b, T, H, P, N, G, w.chunk_size, m2.BF16 if w.dtype == "bf16"
                                 else m2.F32)) == m2.PATH_SIMT
    if pad == 0 or simt:
        assert torch.equal(y, y0) and torch.equal(f1, f0)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=G)
    assert_close(to_np(y), yr, w.dtype, "strided y")
    assert_close(to_np(f1), fr, w.dtype, "strided final_state")


def test_chunk_size_64_runs_as_128():
    """A bf16 whole-path call with chunk_size 64 on a tensor-core shape runs as
    128-token chunks: the same bits as the call with chunk_size 128."""
    w64 = wl(2, 700, 4, 64, 128, 2, 64, init=0.1, seed=24)
    assert m2.path(m2.make_shape(2, 700, 4, 64, 128, 2, 64, dtype=m2.BF16)) == m2.PATH_TCGEN05
    inp = W.make_inputs(w64)
    y64, f64 = run_fwd(inp, w64)
    y128, f128 = run_fwd(inp, w64.scaled(chunk_size=128))
    assert torch.equal(y64, y128) and torch.equal(f64, f128)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w64.ngroups)
    assert_close(to_np(y64), yr, w64.dtype, "y")
    assert_close(to_np(f64), fr, w64.dtype, "final_state")


def test_chunk_size_independence():
    """The chunking is an evaluation order: L in {64, 128, 256} give the same result."""
    w = wl(1, 1024, 4, 64, 128, 1, 256, seed=31)
    inp = W.make_inputs(w)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=1)
    for L in (64, 128, 256):
        y, f = run_fwd(inp, w, chunk_size=L)
        assert_close(to_np(y), yr, "bf16", f"y L={L}")
        assert_close(to_np(f), fr, "bf16", f"final L={L}")


def test_linear_attention_limit_on_gpu():
    """A -> 0 (decay 1): the GPU matches causal linear attention (oracle, A = 0)."""
    w = wl(1, 512, 2, 64, 128, 1, 128, seed=32)
    inp = W.make_inputs(w)
    inp["A"] = torch.zeros_like(inp["A"])
    y, f = run_fwd(inp, w)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=1)
    assert_close(to_np(y), yr, "bf16", "y A=0")
    assert_close(to_np(f), fr, "bf16", "final A=0")


def test_split_and_resume_on_gpu():
    """Two halves, the second started from the first's final_state, equal one run."""
    w = wl(2, 1024, 16, 64, 128, 8, 128, init=0.1, seed=33)
    inp = W.make_inputs(w)
    y, f = run_fwd(inp, w)
    h1 = dict(inp)
    h2 = dict(inp)
    for k in ("x", "dt", "B", "C"):
        h1[k] = inp[k][:, :512].contiguous()
        h2[k] = inp[k][:, 512:].contiguous()
    w2 = w.scaled(seqlen=512)
    y1, f1 = run_fwd(h1, w2)
    h2["initial_state"] = f1.cpu()
    y2, f2 = run_fwd(h2, w2)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    ys = to_np(torch.cat([y1, y2], dim=1))
    assert_close(ys, yr, "bf16", "split y vs oracle")
    assert_close(to_np(f2), fr, "bf16", "split final vs oracle")
    assert_close(to_np(y), yr, "bf16", "single y vs oracle")
    # GPU vs GPU: each within the tolerance of the oracle, so within twice it of each other.
    rel_tol, max_tol = TOL["bf16"]
    for a, b_, ref in ((ys, to_np(y), yr), (to_np(f2), to_np(f), fr)):
        assert np.linalg.norm(a - b_) <= 2 * rel_tol * np.linalg.norm(ref)
        assert np.abs(a - b_).max() <= 2 * max_tol * np.sqrt(np.mean(ref ** 2))


def test_edge_cases():
    # seqlen 0: final_state is the initial state (or zero), nothing else written.
    w = wl(2, 0, 4, 64, 128, 1, 256, init=0.1, seed=34)
    inp = W.make_inputs(w)
    y, f = run_fwd(inp, w)
    assert y.numel() == 0 and torch.equal(f.cpu(), inp["initial_state"])
    w0 = wl(2, 0, 4, 64, 128, 1, 256, seed=34)
    y, f = run_fwd(W.make_inputs(w0), w0)
    assert torch.count_nonzero(f) == 0
    # batch 0: a no-op.
    wb = wl(0, 64, 4, 64, 128, 1, 64, seed=35)
    y, f = run_fwd(W.make_inputs(wb), wb)
    assert y.numel() == 0 and f.numel() == 0
    # dt = 0 everywhere: y = S0 C + D x exactly up to rounding.
    wd = wl(1, 300, 2, 64, 128, 1, 128, init=0.1, seed=36)
    inp = W.make_inputs(wd)
    inp["dt"] = torch.zeros_like(inp["dt"])
    y, f = run_fwd(inp, wd)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=1)
    assert_close(to_np(y), yr, "bf16", "dt=0")
    assert torch.allclose(f.cpu(), inp["initial_state"], rtol=0, atol=0)


# Input magnitudes far from the unit scale of the standard workloads: the
# tensor-core path picks its 16-bit operand types and scales from the data's
# range (per CTA for C.B^T, per head for x, dt and D), so each of these must
# stay within the same tolerance of the fp64 oracle.
MAGNITUDES = [
    ("x*1e5", dict(x=1e5), 0.0),            # |x| above the fp16 range
    ("x*1e-6", dict(x=1e-6), 0.0),          # |x| below the fp16 normal range
    ("dt*1e-4,D=0", dict(dt=1e-4, D=0.0), 0.0),   # small decay-weighted products
    ("B,C*0.01", dict(B=0.01, C=0.01), 0.0),      # |C.B| below the fp16 normal range
    ("B,C*100", dict(B=100.0, C=100.0), 0.0),     # |C.B| above the fp16 range
    ("D*1e4", dict(D=1e4), 0.0),            # skip term dominates
    # fast decay: dt up to 1, so a token's state decays by up to e^-16 per step; the
    # decay factors and the carried-state term underflow, and the diagonal blocks'
    # cum2 ranges rule out their packed fp16 path
    ("dt*10,init", dict(dt=10.0), 0.1),
]


@pytest.mark.parametrize("name,scale,init", MAGNITUDES, ids=[m[0] for m in MAGNITUDES])
def test_input_magnitudes(name, scale, init):
    w = wl(2, 640, 4, 64, 128, 1, 256, init=init, seed=41)
    inp = W.make_inputs(w)
    for k, s in scale.items():
        inp[k] = (inp[k].double() * s).to(inp[k].dtype)
    y, f = run_fwd(inp, w)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups)
    assert_close(to_np(y), yr, w.dtype, name + ": y")
    if "dt" in scale and scale["dt"] > 1:
        # Under fast decay the final state is nearly one token's dt x B^T (the last
        # token carries about half of its energy here, its largest entries ~13 rms):
        # nothing averages the two bf16 roundings each entry takes on its way (stage
        # 2's decay-weighted operand and the bf16 dS hand-off, 2^-9 relative each),
        # so the bound is relative to the entry sizes: relL2 as everywhere, and
        # max|err| <= 2^-7 max|ref|.
        got = to_np(f)
        rel, _ = metrics(got, fr)
        mxe = np.abs(got - fr).max() / np.abs(fr).max()
        assert np.isfinite(got).all() and rel <= 1e-2 and mxe <= 2.0 ** -7, \
            f"{name}: final state relL2 {rel:.3e}, max|err|/max|ref| {mxe:.3e}"
    else:
        assert_close(to_np(f), fr, w.dtype, name + ": final state")


def test_outputs_do_not_depend_on_workspace_contents():
    w = wl(1, 512, 4, 64, 128, 1, 256, seed=37)
    inp = W.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sh = m2.shape_of(dev["x"], dev["B"], w.chunk_size, w.ngroups)
    outs = []
    for fill in (0, 255):
        ws = torch.full((m2.workspace_size(sh),), fill, dtype=torch.uint8, device="cuda")
        y, f = m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], None,
                          chunk_size=w.chunk_size, workspace=ws)
        outs.append((y.clone(), f.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_workspace_too_small_is_rejected():
    w = wl(1, 256, 2, 64, 128, 1, 256, seed=38)
    inp = W.make_inputs(w)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    sh = m2.shape_of(dev["x"], dev["B"], 256, 1)
    ws = torch.empty(m2.workspace_size(sh) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m2.Mamba2Error) as e:
        m2.ssd_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], workspace=ws,
                   chunk_size=256)
    assert e.value.status == m2.ERR_WORKSPACE


# --------------------------------------------------------------- full size -----------
FULL = ([W.MAMBA2_2P7B, W.GROUPED_INIT, W.LONG_PREFILL] + W.sweep_workloads()
        + [W.HEADDIM128, W.CHUNK64, W.HEADDIM32])


@pytest.mark.parametrize("w", FULL, ids=[w.name.split()[0] + "-" + "-".join(w.name.split()[1:3])
                                         + f"-N{w.dstate}" for w in FULL])
def test_full_size_sampled(w):
    """Full-size workload in the benchmark's launch configuration, on the
    tensor-core path; every head of the last batch row (so every head block of
    the output kernel, both block sizes, and the grid's last work items) plus
    32 random (batch, head) pairs recomputed by the recurrent oracle (4 random
    pairs and one full row for the 131 k-token prefill)."""
    inp = W.make_inputs(w)
    assert w.dtype == "bf16"
    assert m2.path(m2.shape_of(inp["x"], inp["B"], w.chunk_size, w.ngroups)) == m2.PATH_TCGEN05
    y, f = run_fwd(inp, w)
    k = 4 if w.seqlen >= 65536 else 32
    pairs = sample_pairs_with_row(w.batch, w.nheads, k, seed=w.seed)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups, pairs=pairs)
    yg, fg = to_np(y), to_np(f)
    assert_close_sampled([yg[b, :, h] for b, h in pairs], [yr[b, :, h] for b, h in pairs],
                         pairs, w.dtype, f"y {w.name}")
    assert_close_sampled([fg[b, h] for b, h in pairs], [fr[b, h] for b, h in pairs],
                         pairs, w.dtype, f"final {w.name}")
    assert np.isfinite(yg).all() and np.isfinite(fg).all()


def test_split_and_resume_at_grouped_init_size():
    """The grouped workload with a carried initial state (b2 T8192 H64 G8 L128,
    initial state ~ N(0, 0.1)) run as two halves of 4096 tokens, the second
    started from the first's final state, against one run of all 8192 tokens:
    sampled pairs of the concatenated halves against the oracle, and the two GPU
    results against each other over every element (each within the bound of the
    oracle, so within twice it of each other)."""
    w = W.GROUPED_INIT
    assert (w.batch, w.seqlen, w.nheads, w.ngroups, w.chunk_size) == (2, 8192, 64, 8, 128)
    inp = W.make_inputs(w)
    y, f = run_fwd(inp, w)
    half = w.seqlen // 2
    h1, h2 = dict(inp), dict(inp)
    for k_ in ("x", "dt", "B", "C"):
        h1[k_] = inp[k_][:, :half].contiguous()
        h2[k_] = inp[k_][:, half:].contiguous()
    w2 = w.scaled(seqlen=half)
    y1, f1 = run_fwd(h1, w2)
    h2["initial_state"] = f1.cpu()
    y2, f2 = run_fwd(h2, w2)
    ys = to_np(torch.cat([y1, y2], dim=1))
    del y1, y2
    pairs = sample_pairs_with_row(w.batch, w.nheads, 32, seed=w.seed + 7)
    yr, fr = oracle.ssd_recurrent(**inp, ngroups=w.ngroups, pairs=pairs)
    yg, fg, f2g = to_np(y), to_np(f), to_np(f2)
    sl = lambda a: [a[b, :, h] for b, h in pairs]  # noqa: E731
    assert_close_sampled(sl(ys), sl(yr), pairs, w.dtype, "split y")
    assert_close_sampled(sl(yg), sl(yr), pairs, w.dtype, "single y")
    assert_close_sampled([f2g[b, h] for b, h in pairs], [fr[b, h] for b, h in pairs], pairs,
                         w.dtype, "split final")
    rel_tol, max_tol = TOL["bf16"]
    for a, b_ in ((ys, yg), (f2g, fg)):
        ref_rms = np.sqrt(np.mean(b_ ** 2))
        assert np.linalg.norm(a - b_) <= 2 * rel_tol * np.linalg.norm(b_)
        assert np.abs(a - b_).max() <= 2 * max_tol * ref_rms
