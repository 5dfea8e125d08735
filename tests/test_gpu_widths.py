"""Row widths across every short-run bucket (next_pow2(D) from 4 to 1024), including widths that
are not powers of two (lanes past the row's end), for each weight type, unweighted and weighted:
forward and backward against the oracle.  Each problem pairs two widths, so one launch per
bucket serves tables of different widths side by side, and its Zipf ids with a lowered
threshold give both short runs and chunked long runs."""
import pytest

from synth.configs import IdSpec, LengthSpec, TableSpec, TBEConfig
from tbe_harness import Case

pytestmark = pytest.mark.gpu

WIDTHS = [4, 8, 12, 16, 20, 36, 100, 128, 260, 512, 1024]


def width_config(D, D2, wdtype, weighted):
    lengths = LengthSpec("poisson", 10.0, empty_frac=0.05)
    ids = IdSpec("zipf", s=1.2, q=0.0)
    return TBEConfig(
        name=f"widths_{D}_{D2}_{wdtype}_{'w' if weighted else 'u'}",
        description=f"two tables of widths {D} and {D2}, Poisson(10) bags, Zipf(1.2) ids",
        B=96, tables=(TableSpec(700, D, lengths, ids), TableSpec(300, D2, lengths, ids)),
        wdtype=wdtype, itype="i64", weighted=weighted, optimizer="adagrad", lr=0.01, eps=1e-8,
        w_scale=0.05, bad_id_frac=0.0, seed=11 + D)


@pytest.mark.parametrize("weighted", [False, True], ids=["unweighted", "weighted"])
@pytest.mark.parametrize("wdtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", WIDTHS)
def test_width_forward_and_backward(D, wdtype, weighted):
    D2 = WIDTHS[(WIDTHS.index(D) + 4) % len(WIDTHS)]
    c = Case(width_config(D, D2, wdtype, weighted), threshold=24, chunk=16)
    c.forward()
    c.backward()
