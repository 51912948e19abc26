"""bench.py's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the keys the measurement contract names.  CPU only: a short
run with a few seconds of oracle work per step."""
import contextlib
import io
import json

import bench


def test_reference_arm_line(monkeypatch):
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-seconds", "4"])
    lines = [x for x in out.getvalue().splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 1, 3)
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "f64"
    assert d["config"]["workload"].startswith("large jagged") and d["config"]["batch"] == 64
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # a step's time is its measured sample (at least 1 s of oracle work), not an
    # extrapolation to the whole workload
    assert 900.0 < d["ms_per_step"] < 20000.0
    # the same config dict the CUDA arm prints: the workload's description only
    w = bench.rank_workload(0, 128)
    cfg = d["config"]
    assert cfg == bench.workload_config(w, cfg["allowed_pairs"], 1)
    assert 1.0e9 < cfg["allowed_pairs"] < 1.1e9


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    """Under torchrun only rank 0 runs the oracle and prints; rank 1 returns at
    once, without output (and without loading the oracle)."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    called = []
    monkeypatch.setattr(bench, "cpu_baseline", lambda *a, **k: called.append(1))
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-seconds", "4"])
    assert out.getvalue() == "" and called == []
