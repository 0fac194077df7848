"""The reference arm of bench.py prints the one-line JSON contract: the base
keys, a cpu_baseline describing the run, and an e2e block with no host-device
traffic.  The oracle processes are stubbed there so the test checks the line,
not the oracle's speed (a real run takes about a minute of CPU time); a
separate test runs the real multi-process oracle on two workers briefly."""

import contextlib
import io
import json
import types

import bench


def _stub_farm(calls):
    class Farm:
        def __init__(self, workers=None):
            self.workers, self.cpu_count = 3, 3

        def run(self, seconds):
            calls.append(seconds)
            return 2.0e9, 0.5, 4

        def close(self):
            calls.append("closed")

        def describe(self, passes, seconds):
            return f"stub: {passes} passes in {seconds} s"
    return Farm


def test_reference_line_keys_and_values(monkeypatch):
    calls = []
    monkeypatch.setattr(bench, "OracleFarm", _stub_farm(calls))
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3"]) == 0
    lines = [ln for ln in out.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    # 4 timed samples of 2 GB in 0.5 s each: 4 GB/s, 500 ms per step
    assert abs(d["value"] - 4.0) < 1e-12 and abs(d["ms_per_step"] - 500.0) < 1e-9
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] == 3 and cb["cpu_count"] == 3 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # 3 warm-up samples then 4 timed ones, each bounded so the whole run stays near a minute
    assert calls[-1] == "closed" and len(calls) == 8 and all(0 < s <= 60.0 for s in calls[:-1])


def test_reference_other_ranks_print_nothing(monkeypatch):
    calls = []
    monkeypatch.setattr(bench, "OracleFarm", _stub_farm(calls))
    args = types.SimpleNamespace(steps=2, warmup=3, gpus=2, cpu_workers=None)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args, 2, 1) == 0
    assert out.getvalue() == "" and calls == []


def test_measured_peaks_file_and_fallback(tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6492.7, "bf16_tflops": 1810.1}))
    assert bench.measured_peaks(str(tmp_path))["hbm_gbs"] == 6492.7
    empty = tmp_path / "none"
    empty.mkdir()
    assert bench.measured_peaks(str(empty)) == {}
    # the fallback figures are the ones the roofline uses without the file
    assert bench.FALLBACK_HBM_GBS == 6400.0 and bench.FALLBACK_BF16_TFLOPS_SUSTAINED == 1400.0


def test_oracle_farm_runs_worker_processes():
    """The CPU baseline's oracle processes: two spawned workers, each over its
    own sequences, run together and report their bytes and passes."""
    farm = bench.OracleFarm(workers=2, seqs_per_worker=1)
    try:
        b, t, passes = farm.run(0.05)
    finally:
        farm.close()
    assert farm.workers == 2 and passes >= 2 and t > 0
    # one pass over a history of at least 4096 tokens reads at least 4 x 4096 x 4 KiB of KV
    assert b >= passes * 4 * 4096 * 4096
    assert "2 single-threaded oracle processes" in farm.describe(passes, t)
