"""Host-side checks of bench.py that need no GPU: the reference arm's JSON
line (the oracle timed on the host cores) carries the keys a reader of the
benchmark relies on, and the dominant launch's DRAM traffic is reported only
while the kernel sources match the ones the ncu capture was taken on."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["value"] > 0
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] == line["value"]
    assert cpu["cpu_model"] and cpu["host_cpus"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == bench.WORKLOAD


def test_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    sha = bench.kernel_source_sha()
    assert len(sha) == 16 and sha == bench.kernel_source_sha()   # stable
    prof = tmp_path / "profiles"
    prof.mkdir()
    entry = {"k": {"kernel_src_sha": sha, "dram_bytes_per_launch": 123}}
    (prof / "roofline_traffic.json").write_text(json.dumps(entry))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: sha)
    assert bench.profiled_traffic("k") == 123
    assert bench.profiled_traffic("other") is None
    entry["k"]["kernel_src_sha"] = "0" * 16   # captured on other sources
    (prof / "roofline_traffic.json").write_text(json.dumps(entry))
    assert bench.profiled_traffic("k") is None


def test_source_hash_covers_code_not_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "quant_weight_gemv_dequant_b300" / "csrc"
    csrc.mkdir(parents=True)
    code = "int f(int a) {\n  return a + 1;   // one more\n}\n/* block\n comment */\n"
    (csrc / "k.cu").write_text(code)
    (csrc / "notes.txt").write_text("not a kernel source")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_source_sha()
    # comments, blank lines and spacing do not count
    (csrc / "k.cu").write_text("// header\n\nint f(int a) {\n    return a + 1;\n}\n")
    assert bench.kernel_source_sha() == base
    (csrc / "notes.txt").write_text("edited")
    assert bench.kernel_source_sha() == base
    # code does
    (csrc / "k.cu").write_text("int f(int a) {\n  return a + 2;\n}\n")
    assert bench.kernel_source_sha() != base
    (csrc / "k.cu").write_text(code)
    (csrc / "k2.cuh").write_text("#define X 1\n")
    assert bench.kernel_source_sha() != base


def test_committed_traffic_entry_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "roofline_traffic.json")) as fh:
        d = json.load(fh)
    e = d["gemv_q4k_gate_up"]
    assert e["dram_bytes_per_launch"] == e["dram_read"] + e["dram_write"]
    assert os.path.exists(os.path.join(ROOT, e["summary"]))
    # reads cover the weights once (188,743,680 B) within 1%
    assert abs(e["dram_read"] - 188_743_680) < 0.01 * 188_743_680


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.measured_peaks()
    assert kind == "fallback" and peaks["hbm_gbs"] == 6400.0
