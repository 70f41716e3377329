"""The benchmark's fixed roofline models (host arithmetic, no GPU).

The forward's graded byte model and contraction FLOPs were fixed in advance of
any measurement for every measured workload (one table of figures, MB and
GFLOP); bench.model() must reproduce them.  The backward's byte model
(bench.bwd_bytes) is checked against a count written out term by term."""
import pytest

import bench
from mamba_ssd_chunked_02_gb300 import workloads as W

# workload -> (graded MB, GFLOP), as fixed before measuring
FIXED = {
    "mamba2-2.7b-layer b8 T4096 H80 P64 N128 G1 L256 bf16": (2468, 130.1),
    "sweep b4 T1024 H32 P64 N64 G1 L256 bf16": (91, 4.4),
    "sweep b4 T4096 H32 P64 N64 G1 L256 bf16": (359, 17.5),
    "sweep b4 T16384 H32 P64 N64 G1 L256 bf16": (1428, 69.9),
    "sweep b4 T1024 H32 P64 N128 G1 L256 bf16": (129, 6.6),
    "sweep b4 T4096 H32 P64 N128 G1 L256 bf16": (501, 26.3),
    "sweep b4 T16384 H32 P64 N128 G1 L256 bf16": (1992, 105.4),
    "sweep b4 T1024 H32 P64 N256 G1 L256 bf16": (203, 11.0),
    "sweep b4 T4096 H32 P64 N256 G1 L256 bf16": (786, 44.1),
    "sweep b4 T16384 H32 P64 N256 G1 L256 bf16": (3121, 176.2),
    "grouped-init b2 T8192 H64 P64 N128 G8 L128 bf16": (1615, 45.2),
    "long-prefill b1 T131072 H48 P64 N128 G1 L256 bf16": (5916, 314.0),
}


@pytest.mark.parametrize("name", sorted(FIXED))
def test_forward_model_matches_the_fixed_table(name):
    w = {x.name: x for x in W.ALL}[name]
    _, graded, flops = bench.model(w)
    mb, gf = FIXED[name]
    assert abs(graded / 1e6 - mb) <= 0.51 + 1e-3 * mb
    assert abs(flops / 1e9 - gf) <= 0.051 + 1e-3 * gf


def test_backward_byte_model_term_by_term():
    w = W.MAMBA2_2P7B          # b8 T4096 H80 P64 N128 G1 L256 bf16, no initial state
    th, tg = 8 * 4096 * 80, 8 * 4096 * 1
    want = (th * 2 * 64 * 2          # read x, dy (bf16)
            + th * 64 * 4            # write dx (fp32)
            + th * 4 + th * 4        # read dt, write ddt
            + th * 2 * 16 * 64 * 128 // 256   # chunk states at fp32, twice
            + tg * 2 * 128 * 2       # read B, C
            + tg * 2 * 128 * 4       # write dB, dC (fp32)
            + 8 * 80 * 64 * 128 * 4)  # read dfinal
    assert bench.bwd_bytes(w) == want
    wi = W.GROUPED_INIT              # with an initial state: + read it, + write dinit
    b, T, H, P, N, G, L = 2, 8192, 64, 64, 128, 8, 128
    want_i = b * T * (H * (2 * P * 2 + 4 * P + 8 + 2 * 16 * P * N / L) + G * (2 * N * 2 + 8 * N)) + \
        3 * 4 * b * H * P * N
    assert bench.bwd_bytes(wi) == want_i


def test_profile_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    """bench.traffic_from_profile returns the committed ncu traffic of a kernel
    while its source hash matches the summary, and None once the source differs
    (counters taken on another kernel say nothing about this one)."""
    import hashlib
    import json
    w = W.MAMBA2_2P7B
    for k in ("chunk_out", "chunk_state", "state_pass", "chunk_cumsum"):
        meta = json.load(open(bench.os.path.join(bench.ROOT, "profiles", f"{k}_mamba2-2.7b-layer.json")))
        src = open(bench.os.path.join(bench.ROOT, meta["source"]), "rb").read()
        current = hashlib.sha256(src).hexdigest()[:16] == meta["source_sha256_16"]
        t = bench.traffic_from_profile(k, w)
        assert (t is not None and t > 0) if current else t is None, k
    # the same summary against a copy of the repository whose stage-4 source differs
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    src = "mamba_ssd_chunked_02_gb300/csrc/k4_chunk_out_tc.cu"
    (root / src).parent.mkdir(parents=True)
    summary = (bench.os.path.join(bench.ROOT, "profiles", "chunk_out_mamba2-2.7b-layer.json"))
    (root / "profiles" / "chunk_out_mamba2-2.7b-layer.json").write_text(open(summary).read())
    meta = json.load(open(summary))
    (root / src).write_text(open(bench.os.path.join(bench.ROOT, src)).read() + "\n// edited\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.traffic_from_profile("chunk_out", w) is None
    # the same summary against a source whose hash matches it is used
    (root / "profiles" / "chunk_out_mamba2-2.7b-layer.json").write_text(json.dumps(
        dict(meta, source_sha256_16=hashlib.sha256((root / src).read_bytes()).hexdigest()[:16])))
    assert bench.traffic_from_profile("chunk_out", w) == meta["traffic_bytes_per_launch"]
    assert bench.traffic_from_profile("chunk_state", w) is None       # no summary there


def test_io_floor_and_moved_bytes_at_the_2p7b_layer():
    """The I/O floor (x, dt, B, C read once, y written once, final state) and the
    bytes the path's four kernels move with the bf16 hand-off, at the 2.7B layer."""
    w = W.MAMBA2_2P7B
    th, tg = 8 * 4096 * 80, 8 * 4096
    assert bench.io_floor(w) == th * (2 * 64 * 2 + 4) + tg * 2 * 128 * 2 + 8 * 80 * 64 * 128 * 4
    k, _, _ = bench.model(w, 2)
    moved = sum(k[n]["bytes"] for n in bench.KERNELS_SPLIT)
    assert abs(moved / 1e6 - 1797) < 1.0
    assert abs(bench.io_floor(w) / 1e6 - 719) < 1.0

