"""The per-shape launch-choice table and the tuning override (host only: no
kernel runs, the choices are computed on the host).

The table (csrc/tile_table.inc, written by mamba_ssd_chunked_02_gb300/tune.py)
must hold only choices the kernels accept -- block sizes dividing H/G -- in
non-overlapping b*nc buckets, and the library must report, for a shape in an
entry's bucket, exactly that entry.  Without a device the SM count is the
library's fallback (a GB300's 152).
"""
import os
import re

import pytest

import mamba_ssd_chunked_02_gb300 as m2
from mamba_ssd_chunked_02_gb300 import build as m2build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "mamba_ssd_chunked_02_gb300", "csrc", "tile_table.inc")
SMS = 152


@pytest.fixture(scope="module")
def lib():
    m2build.build()
    lib = m2.load()
    yield lib
    m2.tile_override()


@pytest.fixture(autouse=True)
def _clear_override(lib):
    yield
    m2.tile_override()


def entries():
    out = []
    for line in open(TABLE):
        m = re.match(r"\s*\{([-\d,\s]+)\}", line)
        if m:
            out.append(tuple(int(v) for v in m.group(1).split(",")))
    return out


def shape_for(N, P, L, hpg, bnc, G=1):
    # b * nc = bnc with T a whole number of chunks
    return m2.make_shape(1, bnc * L, hpg * G, P, N, G, L, dtype=m2.BF16)


def test_table_entries_are_valid_and_disjoint():
    es = entries()
    seen = {}
    for (N, P, L, hpg, lo, hi, k2, v1, v2, k) in es:
        assert N in (64, 128, 256) and P == 64 and L in (128, 256)
        assert 1 <= lo <= hi
        assert lo & (lo - 1) == 0 and hi == 2 * lo - 1, "power-of-two buckets"
        assert k2 >= 0 and hpg % v1 == 0
        assert k >= 0 and (k == 0 or (v2 > 0 and hpg % v2 == 0))
        for (a, b) in seen.get((N, P, L, hpg), []):
            assert hi < a or lo > b, "overlapping buckets"
        seen.setdefault((N, P, L, hpg), []).append((lo, hi))


def test_tabled_shapes_report_their_entry(lib):
    for (N, P, L, hpg, lo, hi, k2, v1, v2, k) in entries():
        for bnc in sorted({lo, hi, (lo + hi) // 2}):
            c = m2.tile_choice(shape_for(N, P, L, hpg, bnc))
            assert c["stage2_source"] == m2.SOURCE_TABLE and c["stage4_source"] == m2.SOURCE_TABLE
            units = bnc * (N // 128 if N > 128 else 1) * hpg
            assert c["stage2_units"] == (min(k2, units) if k2 else -(-units // SMS))
            assert c["stage4_v1"] == v1
            nq, H = L // 128, hpg
            pairs = bnc if k == 0 else min(bnc, k * SMS // (nq * (H // v1)))
            assert c["stage4_pairs1"] == pairs
            assert c["stage4_v2"] == (v1 if pairs == bnc else v2)


def test_model_choice_outside_the_table(lib):
    # H/G = 6 is in no entry: the cost models decide, and their choices divide H/G
    sh = m2.make_shape(3, 4096, 12, 64, 128, 2, 256, dtype=m2.BF16)
    c = m2.tile_choice(sh)
    assert c["stage2_source"] == m2.SOURCE_MODEL and c["stage4_source"] == m2.SOURCE_MODEL
    # stage 2: blocks of heads of one group, or one wave of even ranges
    units = 3 * 16 * 12
    assert 6 % c["stage2_units"] == 0 or c["stage2_units"] == -(-units // SMS)
    assert 6 % c["stage4_v1"] == 0 and 6 % c["stage4_v2"] == 0
    assert 0 <= c["stage4_pairs1"] <= 3 * 16


def test_override_forces_and_bypasses(lib):
    sh = m2.make_shape(8, 4096, 80, 64, 128, 1, 256, dtype=m2.BF16)
    m2.tile_override(20, 40, 16, 1)
    c = m2.tile_choice(sh)
    assert (c["stage2_units"], c["stage2_source"]) == (20, m2.SOURCE_OVERRIDE)
    # one wave of 152 SMs at 2 query tiles x 2 head blocks per (b, c) pair: 38 pairs
    assert (c["stage4_v1"], c["stage4_v2"], c["stage4_pairs1"], c["stage4_source"]) == \
        (40, 16, 38, m2.SOURCE_OVERRIDE)
    # stage 2 takes any range length; a stage-4 block size that does not divide
    # H/G = 80 is ignored for the shape
    m2.tile_override(3, 3)
    c = m2.tile_choice(sh)
    assert (c["stage2_units"], c["stage2_source"]) == (3, m2.SOURCE_OVERRIDE)
    assert c["stage4_source"] != m2.SOURCE_OVERRIDE
    # one wave of even ranges: 8 * 16 chunks * 80 heads over 152 SMs
    m2.tile_override(m2.EVEN_SPLIT)
    c = m2.tile_choice(sh)
    assert (c["stage2_units"], c["stage2_source"]) == (-(-10240 // SMS), m2.SOURCE_OVERRIDE)
    # -1: the cost model, whatever the table says
    m2.tile_override(-1, -1)
    c = m2.tile_choice(sh)
    assert c["stage2_source"] == m2.SOURCE_MODEL and c["stage4_source"] == m2.SOURCE_MODEL
    # waves 0: v1 for every pair
    m2.tile_override(0, 10, 0, 0)
    c = m2.tile_choice(sh)
    assert (c["stage4_v1"], c["stage4_v2"], c["stage4_pairs1"]) == (10, 10, 8 * 16)


def test_override_validation(lib):
    for args in ((-3, 0, 0, 0), (0, -2, 0, 0), (0, 8, -1, 0), (0, 8, 4, -1), (0, 0, 4, 0),
                 (0, 0, 0, 1), (0, -1, 4, 0), (0, -1, 0, 2)):
        with pytest.raises(m2.Mamba2Error) as e:
            m2.tile_override(*args)
        assert e.value.status == m2.ERR_INVALID_ARG, args
    m2.tile_override()


def test_tile_choice_off_the_tensor_core_path(lib):
    for sh in (m2.make_shape(2, 512, 8, 64, 128, 1, 256, dtype=m2.F32),
               m2.make_shape(2, 512, 8, 64, 128, 1, 256, dtype=m2.BF16, flags=m2.FLAG_FORCE_SIMT),
               m2.make_shape(2, 512, 8, 16, 128, 1, 256, dtype=m2.BF16)):
        with pytest.raises(m2.Mamba2Error) as e:
            m2.tile_choice(sh)
        assert e.value.status == m2.ERR_UNSUPPORTED
    with pytest.raises(m2.Mamba2Error) as e:
        m2.tile_choice(m2.make_shape(2, 512, 8, 64, 100, 1, 256, dtype=m2.BF16))
    assert e.value.status == m2.ERR_UNSUPPORTED


def test_tile_choice_of_empty_shapes(lib):
    """No heads, no batch or no tokens: nothing to launch, and no division by zero."""
    m2.tile_override(0, 8, 4, 1)
    for sh in (m2.make_shape(2, 512, 0, 64, 128, 1, 256, dtype=m2.BF16),
               m2.make_shape(0, 512, 8, 64, 128, 1, 256, dtype=m2.BF16),
               m2.make_shape(2, 0, 8, 64, 128, 1, 256, dtype=m2.BF16)):
        m2.tile_choice(sh)
    m2.tile_override()
    m2.tile_choice(m2.make_shape(2, 512, 0, 64, 128, 1, 256, dtype=m2.BF16))


def test_choices_follow_the_tensor_core_view(lib):
    """P = 128 runs as twice the heads of P = 64, and a whole-path chunk length of
    64 as 128-token chunks: their launch choices are those of that view."""
    a = m2.tile_choice(m2.make_shape(4, 4096, 40, 128, 128, 1, 256, dtype=m2.BF16))
    b = m2.tile_choice(m2.make_shape(4, 4096, 80, 64, 128, 1, 256, dtype=m2.BF16))
    assert a == b
    c = m2.tile_choice(m2.make_shape(2, 4096, 32, 64, 128, 2, 64, dtype=m2.BF16))
    d = m2.tile_choice(m2.make_shape(2, 4096, 32, 64, 128, 2, 128, dtype=m2.BF16))
    assert c == d
    assert m2.path(m2.make_shape(2, 4096, 32, 64, 128, 2, 64, dtype=m2.BF16)) == m2.PATH_TCGEN05
