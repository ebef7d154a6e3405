"""bench.py's command line and the JSON line of its reference arm (the fp64
oracle on the host cores), checked on the CPU: the keys the line must carry,
their types, and that the arm reports what it ran."""
import contextlib
import io
import json

import pytest

import bench


def _run(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(argv)
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert rc == 0 and len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_line(monkeypatch):
    monkeypatch.setattr(bench, "WORKLOAD_ID", bench.WORKLOAD_ID)  # main() sets it; restored afterwards
    d = _run(["--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "1"])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny_f32_n64_E32_H4"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused(monkeypatch):
    monkeypatch.setattr(bench, "WORKLOAD_ID", bench.WORKLOAD_ID)
    with pytest.raises(SystemExit):
        with contextlib.redirect_stderr(io.StringIO()):
            bench.main(["--impl", "reference", "--steps", "1", "--warmup", "2"])


def test_traffic_is_tied_to_the_kernel_source_and_workload(monkeypatch, tmp_path):
    # DRAM bytes from an ncu summary count only for the kernel source they were
    # captured on and for their workload: a stale or foreign entry gives null.
    digest = bench.source_digest(bench.KERNEL_SOURCES["edge_attn"])
    entry = {"dram_bytes_per_launch": 123456789.0, "source_digest": digest,
             "workload": "skewed_n20000_E128_H8, B=16"}
    (tmp_path / "ncu_traffic.json").write_text(json.dumps({"edge_attn": entry}))
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    assert bench.ncu_traffic("edge_attn", "skewed_n20000_E128_H8") == 123456789.0
    assert bench.ncu_traffic("edge_attn", "grn_n2000_E128_H8") is None
    assert bench.ncu_traffic("out_proj", "skewed_n20000_E128_H8") is None
    monkeypatch.setattr(bench, "source_digest", lambda paths: "0" * 16)
    assert bench.ncu_traffic("edge_attn", "skewed_n20000_E128_H8") is None


def test_algorithmic_bytes_of_the_edge_kernel():
    # q, k|v and the mixed rows once, plus col and row_ptr (int32), at n=20k
    w = bench.synth.workload(3)
    got = bench.algorithmic_bytes("edge_attn", w, 16, 400_000)
    E, n, B = 128, 20_000, 16
    assert got == B * n * E * 2 + B * n * 2 * E * 2 + B * n * E * 2 + 400_000 * 4 + (n + 1) * 4


def test_algorithmic_bytes_of_the_fused_edge_kernel():
    # with out_proj inside: q, k|v in, the output rows out, Wo and bo once
    w = bench.synth.workload(3)
    got = bench.algorithmic_bytes("edge_attn_out", w, 16, 400_000)
    E, n, B = 128, 20_000, 16
    assert got == B * n * E * 2 + B * n * 2 * E * 2 + E * E * 2 + E * 2 + B * n * E * 2 + 400_000 * 4 + (n + 1) * 4
