"""The timeline summaries (timeline.py) on hand-made records (no GPU): the
GEMM units' phase durations, span, pair-tile / swap-unit split and bound,
the dispatch blocks' phase ends, and where each region's recording stops."""
import numpy as np
import pytest

from mixture_experts_layer_capacity_b300 import timeline as TL


def _record(t0, wait_acc, wait_stage, issue, epi_start, epi_wait, drain, swap):
    r = np.zeros(8, dtype=np.int64)
    r[TL.MMA_START] = t0
    r[TL.MMA_HAS_ACC] = t0 + wait_acc
    r[TL.FIRST_STAGE_FULL] = t0 + wait_acc + wait_stage
    r[TL.LAST_MMA_ISSUED] = t0 + wait_acc + wait_stage + issue
    r[TL.EPI_START] = epi_start
    r[TL.EPI_ACC_FULL] = epi_start + epi_wait
    r[TL.EPI_DONE] = epi_start + epi_wait + drain
    r[TL.IS_SWAP] = swap
    return r


def _words(recs, region):
    w = np.zeros(TL.MAX_UNITS * TL.WORDS_PER_UNIT * len(TL.REGIONS), dtype=np.uint64)
    base = region * TL.MAX_UNITS * TL.WORDS_PER_UNIT
    for i, r in enumerate(recs):
        w[base + 8 * i: base + 8 * i + 8] = r
    return w


def test_units_stop_at_the_first_unfinished_record():
    recs = [_record(1000 + 100 * i, 1, 2, 50, 1000 + 100 * i, 55, 30, 0) for i in range(5)]
    recs[3][TL.EPI_DONE] = 0           # the epilogue side never wrote this one
    w = _words(recs, 1)
    assert len(TL.units(w, 0)) == 0
    got = TL.units(w, 1)
    assert got.shape == (3, 8) and (got == np.stack(recs[:3])).all()


def test_summary_of_an_epilogue_bound_region():
    # three pair tiles (issue 40, drain 60) then one swap unit (issue 20, drain 10)
    recs = [_record(1000 + 100 * i, 2, 4, 40, 1000 + 100 * i, 46, 60, 0) for i in range(3)]
    recs.append(_record(1300, 6, 2, 20, 1300, 28, 10, 1))
    s = TL.summarize(np.stack(recs))
    assert s["units"] == 4 and s["swap_units"] == 1
    assert s["span_ns"] == (1300 + 28 + 10) - 1000
    ph = s["phases"]
    assert ph["mma_issue"]["total_ns"] == 3 * 40 + 20
    assert ph["mma_issue"]["tile_mean_ns"] == 40 and ph["mma_issue"]["swap_mean_ns"] == 20
    assert ph["mma_waits_accumulator"]["mean_ns"] == pytest.approx((3 * 2 + 6) / 4)
    assert ph["mma_waits_first_stage"]["total_ns"] == 3 * 4 + 2
    assert ph["epilogue_waits_accumulator"]["total_ns"] == 3 * 46 + 28
    assert ph["epilogue_drain"]["mean_ns"] == pytest.approx((3 * 60 + 10) / 4)
    assert s["bound"] == "epilogue"
    assert s["mma_issue_frac"] == pytest.approx(140 / 338)
    assert s["epilogue_drain_frac"] == pytest.approx(190 / 338)
    assert s["tiles_before_swaps"]
    text = TL.format_summary("x", {"gemm1": s, "gemm2": {"units": 0}})
    assert "epilogue-bound" in text and "gemm2: no routed CTA-pair launch" in text


def test_summary_flags_a_swap_unit_ahead_of_a_tile():
    recs = [_record(0 + 100 * i, 1, 1, 80, 100 * i, 82, 10, sw) for i, sw in
            enumerate([0, 1, 0])]
    s = TL.summarize(np.stack(recs))
    assert s["bound"] == "mma" and not s["tiles_before_swaps"]
    assert s["phases"]["epilogue_drain"]["swap_mean_ns"] == 10
    assert TL.summarize(np.zeros((0, 8), dtype=np.int64)) == {"units": 0}


def test_dispatch_summary_and_layout():
    w = np.zeros(TL.DISPATCH_BASE + TL.MAX_UNITS * TL.WORDS_PER_UNIT, dtype=np.uint64)
    assert TL.DISPATCH_BASE + TL.MAX_UNITS * TL.WORDS_PER_UNIT == 98304
    blocks = []
    for b in range(3):
        t0 = 1000 + 10 * b
        r = np.array([t0, t0 + 5, t0 + 7, t0 + 9, t0 + 20, 2000, 2100 + b, 2500 + 100 * b],
                     dtype=np.int64)
        blocks.append(r)
        w[TL.DISPATCH_BASE + 8 * b: TL.DISPATCH_BASE + 8 * b + 8] = r
    rec = TL.dispatch_blocks(w)
    assert rec.shape == (3, 8) and (rec == np.stack(blocks)).all()
    s = TL.summarize_dispatch(rec)
    assert s["blocks"] == 3 and s["span_ns"] == 2700 - 1000
    assert s["phases"]["rows_staged"] == {"median_ns": 15.0, "max_ns": 25}
    assert s["phases"]["grid_barrier"] == {"median_ns": 1000.0, "max_ns": 1000}
    assert s["phases"]["row_copies"]["median_ns"] == 1600.0
    assert TL.summarize_dispatch(np.zeros((0, 8))) == {"blocks": 0}
    text = TL.format_summary("x", {"dispatch": s, "gemm1": {"units": 0}, "gemm2": {"units": 0}})
    assert "dispatch: 3 blocks, span 1.7 us" in text
