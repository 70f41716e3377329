"""Launch choices regroup independent work only: every stage-2 range of units
per CTA (blocks of heads, ranges that cross group segments) and every stage-4
head-block split must give the same bits as the library's own choice (table
or cost model)."""
import pytest
import torch

import mamba_ssd_chunked_02_gb300 as m2
from mamba_ssd_chunked_02_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_chunked_02_gb300 import build
    build.build()
    m2.load()
    m2.device_error(clear=True)
    yield
    m2.tile_override()


@pytest.mark.parametrize("w", [
    W.Workload("tiles b2 T2048 H16 P64 N128 G2 L256", 2, 2048, 16, 64, 128, 2, 256, seed=601),
    W.Workload("tiles b3 T1000 H8 P64 N64 G1 L128", 3, 1000, 8, 64, 64, 1, 128, init_std=0.1,
               seed=602),
    W.Workload("tiles b1 T500 H4 P64 N256 G1 L256", 1, 500, 4, 64, 256, 1, 256, seed=603),
], ids=lambda w: w.name)
def test_forced_choices_give_identical_bits(w):
    inp = W.make_inputs(w, device="cuda")
    sh = m2.shape_of(inp["x"], inp["B"], w.chunk_size, w.ngroups)
    assert m2.path(sh) == m2.PATH_TCGEN05

    def run():
        y, fin = m2.ssd_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["initial_state"], chunk_size=w.chunk_size, ngroups=w.ngroups)
        torch.cuda.synchronize()
        assert m2.device_error() == 0
        return y, fin

    m2.tile_override()
    y0, f0 = run()
    hpg = w.nheads // w.ngroups
    divs = [v for v in range(1, hpg + 1) if hpg % v == 0]
    # stage 2: blocks of v heads, ranges crossing segments (3 and 5 units, one
    # wave of even ranges); stage 4: single block sizes
    forced = [(v, v, 0, 0) for v in divs] + [(3, divs[0], 0, 0), (5, divs[-1], 0, 0),
                                             (m2.EVEN_SPLIT, divs[-1], 0, 0)]
    # a two-region split whose first region ends inside the grid: v1 = 1 (the
    # most CTAs per pair) for one wave, v2 = 2 after it
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bc = w.batch * sh.nchunks
    if 0 < sms // ((w.chunk_size // 128) * w.nheads) < bc:
        forced.append((divs[-1], 1, 2, 1))
    for args in forced:
        m2.tile_override(*args)
        c = m2.tile_choice(sh)
        assert c["stage2_source"] == c["stage4_source"] == m2.SOURCE_OVERRIDE
        if args[3]:
            assert 0 < c["stage4_pairs1"] < bc and c["stage4_v2"] == 2
        y, fin = run()
        assert torch.equal(y, y0), args
        assert torch.equal(fin, f0), args
    m2.tile_override()
