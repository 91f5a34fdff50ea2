"""The bench's reference arm (the fp64 oracle on host cores) prints one JSON line
with the contract's keys, on the same workload as the GPU arm (CPU)."""
import contextlib
import io
import json

import bench


def test_reference_arm_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["config"]["workload"] == "cfg2_varlen_74seq" and line["config"]["total_tokens"] == 62875
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
