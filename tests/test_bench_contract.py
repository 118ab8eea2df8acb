"""bench.py's JSON contract on the CPU: the reference arm's line, and the
traffic figure it takes from the committed decode profile record.

The reference arm times the fp64 oracle on the host cores, so it runs here
on the smallest workload; the GPU arm prints the same keys plus the
measurement objects and is exercised on a GPU.
"""

from __future__ import annotations

import json

import bench

REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def test_reference_line(capsys, monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
                "--oracle-segments", "2"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1, "exactly one JSON line"
    d = json.loads(lines[0])
    assert REQUIRED <= set(d)
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "steps/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    from adaptive_sparse_paged_gb300 import synth
    assert d["config"]["workload"] == bench.workload_name(synth.CONFIGS["tiny"], 0.99)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert "2 of" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0
    ex = d["extrapolation"]
    assert ex["segments_timed_per_step"] == 2 and ex["segments_per_full_step"] == 2
    # steps x ms_per_step is the time the oracle actually ran; value scales it
    full_ms = d["ms_per_step"] * ex["factor"]
    assert abs(full_ms - 1e3 / d["value"]) < 1e-6 * full_ms
    assert abs(ex["ms_per_full_step"] - full_ms) < 1e-6 * full_ms
    assert set(d["config"]) == {"workload", "gamma", "budget", "l2"}


def test_traffic_follows_the_profiled_source(tmp_path, monkeypatch):
    """The committed figure is used only while the hashed sources are the profiled ones."""
    rec_path = bench.os.path.join(bench.ROOT, bench.TRAFFIC_RECORD)
    rec = json.load(open(rec_path))
    got = bench.decode_traffic_per_page("long128k")
    if rec["sources_sha256_16"] == bench.source_digest(*rec["sources"]):
        assert got == rec["dram_bytes_per_selected_page_head"]
    else:  # profiled on other sources: no traffic figure
        assert got is None
    fake = tmp_path / "adaptive_sparse_paged_gb300" / "csrc"
    fake.mkdir(parents=True)
    for n in rec["sources"]:
        (fake / n).write_text("// another kernel\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / bench.TRAFFIC_RECORD).write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.decode_traffic_per_page("long128k") is None


def test_reference_line_budget_mode(capsys, monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
                "--oracle-segments", "2", "--budget", "5"])
    d = json.loads([l for l in capsys.readouterr().out.splitlines() if l.startswith("{")][0])
    assert d["config"]["budget"] == 5 and d["config"]["workload"].endswith("budget5")
    assert d["value"] > 0
