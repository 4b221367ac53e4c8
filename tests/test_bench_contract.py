"""The bench's command-line defaults and the reference arm's JSON line (CPU).

The reference arm times the float64 oracle on the host cores; on the small
c1 workload its sample takes milliseconds, so its output line can be checked
here against the keys the bench contract names.  The GPU arm needs a GPU and
is exercised by the full test run.
"""
from __future__ import annotations

import json

import bench


def test_defaults_name_the_largest_workload_and_a_short_run():
    a = bench.parse_args([])
    assert a.workload == "c3"            # 4096 x 32768, the largest configuration
    assert a.gpus == 1 and a.impl == "ours"
    assert a.warmup >= 3 and a.steps >= 1


def test_reference_arm_line(tmp_path, capsys):
    out = tmp_path / "ref.json"
    bench.main(["--impl", "reference", "--workload", "c1", "--steps", "2", "--warmup", "0",
                "--json-out", str(out)])
    printed = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(printed) == 1
    line = json.loads(printed[0])
    assert json.loads(out.read_text()) == line
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "rows/s" and line["value"] > 0
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] >= 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["vs_baseline"] is None and line["data"] == "synthetic"
    assert line["config"]["workload"].startswith("c1:") and line["config"]["M"] == 128
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["ms_per_step"] > 0
