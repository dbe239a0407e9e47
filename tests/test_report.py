"""Reporting helpers against the numbers the pages print."""

import os

import pytest

from verify_spec_draft_gb300 import report

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dspine_cycle_cost.txt")


def _rows():
    ex, rows = None, []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("example "):
                ex = dict(kv.split("=") for kv in line.split()[1:])
            elif line.startswith("row "):
                name, *vals = line[4:].strip().split("|")
                rows.append((name, [float(v) for v in vals]))
    return ex, rows


def test_cycle_cost_worked_example():
    ex, _ = _rows()
    c = report.cycle_cost(float(ex["L"]), float(ex["tput"]), float(ex["tput_ar"]))
    assert round(c, 2) == float(ex["c"])


def test_dspine_table_gains():
    """The page's acceptance-gain column is L_DSpine / L_DFlash2 - 1, rounded to 0.1%."""
    _, rows = _rows()
    assert len(rows) == 10
    for name, (l0, l1, lgain, tgain, c0, c1) in rows:
        assert abs(report.gain_pct(l1, l0) - lgain) <= 0.051, name
    mean_l = sum(r[1][2] for r in rows) / 10
    mean_t = sum(r[1][3] for r in rows) / 10
    assert round(mean_l, 1) == 22.8 and round(mean_t, 1) == 14.0   # the page's summary


def test_dspine_table_cycle_cost_consistent():
    """c_DSpine / c_DFlash2 = (L1/L0) / (S1/S0): the implied cost ratio follows from the
    two gain columns (within the page's two-decimal rounding of c)."""
    _, rows = _rows()
    for name, (l0, l1, lgain, tgain, c0, c1) in rows:
        ratio = (1 + lgain / 100) / (1 + tgain / 100)
        assert abs(c1 / c0 - ratio) < 0.02, name


def test_headline_speedups():
    # "Solar Open2 DSpark", section 5: 130 -> 472.8 tok/s is about 3.64x
    assert round(report.speedup(472.8, 130.0), 2) == 3.64
    # DSpine FAQ: 805.53 vs 210.03 tok/s is up to 3.84x
    assert round(report.speedup(805.53, 210.03), 2) == 3.84
    # SpecOPD: 4.95x updates times 3.25x tokens per update is 16.09x supervision
    assert round(4.95 * 3.25, 2) == 16.09


def test_acceptance_length_counts_bonus_and_skips_invalid():
    assert report.acceptance_length([0, 3, 7]) == pytest.approx(13 / 3)
    assert report.acceptance_length([2, -1]) == 3.0
