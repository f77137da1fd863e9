"""Spike protocol decisions (host logic only) and checkpoint file naming.  CPU only."""
import math

import pytest

from bitwise_reproducible_step_gb300 import policy as P
from bitwise_reproducible_step_gb300 import repstep as rs


def decisions(norms, **kw):
    p = P.SpikeSkip(**kw)
    return [p.apply(x) for x in norms]


def test_spike_skips_five_steps_including_itself():
    d = decisions([1, 2, 6, 1, 1, 1, 1, 1, 1])
    assert d == [True, True, False, False, False, False, False, True, True]


def test_spike_inside_the_window_restarts_it():
    d = decisions([1, 7, 1, 9, 1, 1, 1, 1, 1, 1])
    assert d == [True, False, False, False, False, False, False, False, True, True]


def test_threshold_is_strict_and_nonfinite_counts_as_spike():
    assert decisions([5.0, 5.0000005]) == [True, False]
    assert decisions([math.nan, 1, 1, 1, 1, 1]) == [False] * 5 + [True]
    assert decisions([math.inf]) == [False]


def test_span_one_skips_only_the_spike():
    assert decisions([1, 8, 1], span=1) == [True, False, True]
    with pytest.raises(ValueError):
        P.SpikeSkip(span=0)


def test_checkpoint_names():
    assert rs.checkpoint_name(0) == "step_000000.bin"
    assert rs.checkpoint_name(112700) == "step_112700.bin"
    assert rs.checkpoint_name(1234567) == "step_1234567.bin"
    with pytest.raises(ValueError):
        rs.checkpoint_name(-1)


def test_step_log_appends_one_line_per_record(tmp_path):
    p = tmp_path / "run.jsonl"
    log = P.StepLog(p)
    assert log.records() == []
    log.write({"train_step": 1, "norm": 0.5, "root": P.root_hex(-2)})
    P.StepLog(p).write({"train_step": 2, "norm": math.nan})      # reopened: appends
    lines = p.read_text().splitlines()
    assert len(lines) == 2
    recs = log.records()
    assert recs[0] == {"norm": 0.5, "root": "fffffffffffffffe", "train_step": 1}
    assert recs[1]["train_step"] == 2 and math.isnan(recs[1]["norm"])


def test_step_log_bit_formats():
    assert P.f32_bits(1.0) == "3f800000"
    assert P.f32_bits(-0.0) == "80000000"
    assert P.f32_bits(2.0 ** -149) == "00000001"
    assert P.root_hex(0) == "0" * 16
    assert P.root_hex(2**63) == "8000000000000000"
    assert P.root_hex(-1) == "f" * 16
