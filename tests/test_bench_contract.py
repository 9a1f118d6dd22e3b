"""The reference arm of bench.py (the CPU oracle timed on the host cores) prints one
JSON line with the keys the benchmark contract requires; checked on CPU with a
reduced sequence so that it runs in seconds."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    real = bench.oracle_rows_rate  # the real oracle timing, on a half-second budget
    monkeypatch.setattr(bench, "oracle_rows_rate", lambda w, budget_s, x=None: real(w, 0.5, x))
    args = type("A", (), {"workload": 5, "seq": 1024, "steps": 1, "warmup": 0})()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(args)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert "workload" in d["config"]
