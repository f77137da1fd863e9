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
