"""bench.py's JSON contract on the CPU: the reference arm's line, and the
traffic figure it takes from the committed decode profile.

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
    assert abs(d["ms_per_step"] - 1e3 / d["value"]) < 1e-6 * d["ms_per_step"]


def test_traffic_follows_the_profiled_source(tmp_path, monkeypatch):
    """The committed figure is used only while decode.cu is the profiled source."""
    assert bench.decode_traffic_per_page("long128k") is not None
    fake = tmp_path / "adaptive_sparse_paged_gb300" / "csrc"
    fake.mkdir(parents=True)
    (fake / "decode.cu").write_text("// another kernel\n")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "decode_kernel_ncu.md").write_text(
        open(bench.os.path.join(bench.ROOT, "profiles", "decode_kernel_ncu.md")).read())
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
