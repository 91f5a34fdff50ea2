"""The oracle reproduces its frozen config-0 sample (a regression fixture
written by tests/golden/make_golden.py from the oracle alone)."""
import os

import pytest

from tests.golden import make_golden


def _read():
    vals = {}
    with open(make_golden.OUT) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            vals[tuple(parts[:-1])] = float(parts[-1])
    return vals


def test_oracle_matches_frozen_sample():
    stored = _read()
    os_, ss, on, sn = make_golden.sample()
    for i, v in os_:
        assert v == pytest.approx(stored[("o",) + tuple(map(str, i))], rel=1e-12, abs=1e-15)
    for i, v in ss:
        assert v == pytest.approx(stored[("s",) + tuple(map(str, i))], rel=1e-12, abs=1e-15)
    assert on == pytest.approx(stored[("o_fro",)], rel=1e-12)
    assert sn == pytest.approx(stored[("s_fro",)], rel=1e-12)
