"""Host side of the per-role clock trace: the period and the median chunk life that
`trace.report` derives from a stamp array, and the time order `trace.report_raw`
prints, checked on synthetic stamps whose answer is known (no GPU)."""
import io

import numpy as np

from gated_deltanet_linear_prefill_gb300 import trace


def _stamps(n_chunks=40, period_cyc=8000, start=100000):
    """Every event of EVENTS stamped at the reference point of its chunk plus a fixed
    per-event offset (the offset of event k is 150 (k - 10) cycles)."""
    T = np.zeros((16, 256, 8), np.int64)
    offs = {}
    for k, (wp, pt) in enumerate(trace.EVENTS):
        offs[(wp, pt)] = 150 * (k - 10)
    offs[trace.REF] = 0
    for c in range(n_chunks):
        ref = start + period_cyc * c
        for (wp, pt), o in offs.items():
            T[wp, c, pt] = ref + o
    return T, offs


def test_report_gives_the_period_and_each_events_offset():
    ghz = 2.0
    T, offs = _stamps()
    period, rows = trace.report(T, ghz, 0, 123.0, file=io.StringIO())
    assert abs(period - 8000 / ghz / 1e3) < 1e-9
    got = {name: t for t, name in rows}
    assert len(got) == len(trace.EVENTS)
    for key, name in trace.EVENTS.items():
        assert abs(got[name] - offs[key] / ghz / 1e3) < 1e-9, name
    # rows come sorted by time
    assert [t for t, _ in rows] == sorted(t for t, _ in rows)


def test_report_ignores_unstamped_points_and_uses_the_median():
    ghz = 1.5
    T, offs = _stamps(n_chunks=30)
    wp, pt = 2, 2  # warp 2's U' issue: drop it on a few chunks, disturb one chunk
    T[wp, 7, pt] = 0
    T[wp, 9, pt] = 0
    T[wp, 12, pt] += 10 ** 6  # one outlier does not move the median
    _, rows = trace.report(T, ghz, 3, 1.0, file=io.StringIO())
    got = {name: t for t, name in rows}
    assert abs(got[trace.EVENTS[(wp, pt)]] - offs[(wp, pt)] / ghz / 1e3) < 1e-9


def test_report_raw_lists_stamps_in_time_order():
    T, _ = _stamps(n_chunks=3)
    buf = io.StringIO()
    evs = trace.report_raw(T, 100000 - 5000, 2.0, 0, 9.9, file=buf)
    times = [t for t, _ in evs]
    assert len(evs) == 3 * len(trace.EVENTS)
    assert min(times) > 0
    lines = buf.getvalue().splitlines()[1:]
    printed = [float(line.split()[0]) for line in lines]
    assert printed == sorted(printed)
