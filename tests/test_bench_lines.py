"""Host arithmetic of the bench's per-workload lines, on CPU: the input logit bytes of one round
and the HBM fraction each filter, PyramidSD, tree and config line reports."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import workloads as W  # noqa: E402


@pytest.mark.parametrize("base", [W.PLAIN, W.SAMPLED_TOPP, W.SAMPLED_TOPK, W.SAGUARO, W.MIRROR, W.PYRAMID_QT,
                                  W.PYRAMID_DQ, W.scaled(W.MIRROR, K=56, draft_rows_extra=1)],
                         ids=lambda w: w.name.split()[0] + f"-K{w.K}")
def test_round_logit_bytes_is_the_size_of_the_round_inputs(base):
    """The bytes a line divides by its time are those of the logit tensors the round takes."""
    w = W.scaled(base, B=2, V=96)
    tgt, drf = W.logits(w, 0)
    assert bench.round_logit_bytes(w) == tgt.numel() * tgt.element_size() + drf.numel() * drf.element_size()


def test_pyramid_rows_agree_with_round_bytes():
    for w in (W.PYRAMID_QT, W.PYRAMID_DQ):
        assert bench.round_logit_bytes(w) == w.B * (2 * w.K + 1) * w.V * 2


def test_add_hbm_on_both_time_keys():
    line = {"filters": {"f": {"ms_per_round": 0.5, "logit_bytes_per_round": 4_000_000_000}},
            "pyramid": {},
            "tree": {"t": {"ms_per_round": 2.0, "logit_bytes_per_round": 1_000_000_000}},
            "configs": {"c": {"us_per_round": 250.0, "logit_bytes_per_round": 1_000_000_000}}}
    bench.add_hbm(line, 8000.0)
    f, t, c = line["filters"]["f"]["hbm"], line["tree"]["t"]["hbm"], line["configs"]["c"]["hbm"]
    assert f["achieved_gbs"] == pytest.approx(8000.0) and f["frac"] == pytest.approx(1.0)
    assert t["achieved_gbs"] == pytest.approx(500.0) and t["frac"] == pytest.approx(0.0625)
    assert c["achieved_gbs"] == pytest.approx(4000.0) and c["frac"] == pytest.approx(0.5)
    assert c["peak_gbs"] == 8000.0


def test_whole_call_roofline_divides_the_bytes_read_by_the_call_time():
    r = bench.whole_call_roofline(1_116_340_224, 0.25, 6693.8, "measured")
    assert r["achieved_gbs"] == pytest.approx(1_116_340_224 / 0.25e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved_gbs"] / 6693.8)
    assert r["of_8tbs"] == pytest.approx(r["achieved_gbs"] / 8000.0)


def test_oracle_round_seconds_times_whole_rounds_on_the_pool():
    """The CPU baseline's timing: whole rounds through spawned workers, one time per timed run."""
    w = W.scaled(W.LARGE_BATCH, B=6, V=300)
    t = bench.oracle_round_seconds(w, [0, 1], 2, "cpu", repeats=2)
    assert len(t) == 4 and all(x > 0 for x in t)
