"""The small-table counts x table forward (tcgen05 tensor cores) against the oracle and against
the gather path on the same inputs."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bwd_tbe_fwd_gb300 import TBEOptions
from synth import get_config
from synth.configs import IdSpec, LengthSpec, TableSpec
from tbe_harness import Case, check_forward, weights_to_oracle

pytestmark = pytest.mark.gpu


def hist_config(E, D, lengths, B, companion=True, bad=0.0, itype="i64", name="hist"):
    tables = [TableSpec(E, D, lengths, IdSpec("uniform"), histogram=True)]
    if companion:
        tables.append(TableSpec(5000, 64, LengthSpec("poisson", 6.0), IdSpec("uniform")))
    base = get_config("c4")
    return dataclasses.replace(base, name=name, B=B, tables=tuple(tables), bad_id_frac=bad, itype=itype)


CASES = {
    "c4_like": hist_config(64, 128, LengthSpec("fixed", 256), 2048),
    "ragged_tile_E37_D96": hist_config(37, 96, LengthSpec("poisson", 200.0), 333),
    "tail_past_256_D64": hist_config(64, 64, LengthSpec("poisson", 300.0), 200),
    "short_bags_and_empty": hist_config(50, 128, LengthSpec("poisson", 40.0, empty_frac=0.1), 130),
    "int32_ids": hist_config(64, 128, LengthSpec("fixed", 100), 256, itype="i32"),
    "alone": hist_config(64, 112, LengthSpec("fixed", 64), 1000, companion=False),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_histogram_forward_matches_oracle_and_gather(name):
    cfg = CASES[name]
    c = Case(cfg)
    out_hist = c.forward()  # default options: the histogram path serves table 0
    out_gather = c.forward(options=TBEOptions(histogram=0))
    # both within tolerance of the oracle (checked inside forward); and close to each other
    assert torch.allclose(out_hist, out_gather, rtol=1e-5, atol=1e-6)


def test_histogram_skips_out_of_range_ids():
    cfg = hist_config(64, 128, LengthSpec("fixed", 256), 512, bad=0.002, name="hist_bad")
    c = Case(cfg, bounds_check=False)
    w = c.w0.cuda()
    c.tbe.forward(w, c.idx_d, c.off_d, stats=c.stats)
    torch.cuda.synchronize()
    assert c.stats[2].item() == len(c.batch.bad_positions)
    # after repair, the histogram path equals the oracle
    c.run_bounds()
    c.forward()
