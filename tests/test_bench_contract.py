"""Host logic of the benchmark, on CPU: the reference arm's JSON line (the
oracle timed on the host cores), its silence on ranks other than 0, the
roofline and clock summaries, and the rule that a committed DRAM-traffic
figure is reported only while its kernel sources are unchanged."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run_reference(extra_env=None):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="2")
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "block_fp32_d64", "--steps", "2", "--warmup", "1"],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run_reference()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["ms_per_step"] > 0 and d["dtype"] == "f64" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "block_fp32_d64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == d["value"]
    assert cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_on_other_ranks():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_end_to_end_roofline_sums_each_kernels_bound():
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 1000.0}
    prof = {"gemm": {"flops": 2e12, "bytes": 1e9},    # 2 ms of flops, 1 ms of bytes: 2 ms
            "ln": {"flops": 0.0, "bytes": 3e9}}       # 3 ms of bytes
    got = bench.e2e_roofline(prof, peaks, steps=5, ms_step=2.0)
    assert got["sum_t_roof_ms"] == pytest.approx((2.0 + 3.0) / 5)
    assert got["frac"] == pytest.approx(0.5)


def test_clock_summary_takes_loaded_samples_and_active_reasons():
    c = bench.ClockSampler(0)
    c.out = "\n".join([
        "0, 300, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2055, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    s = c.summary()
    assert s["sm_mhz"] == 2055 and s["sm_max_mhz"] == 2070 and s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"]
    c.out = ""
    assert c.summary() is None


def test_traffic_figure_needs_the_sources_it_was_taken_from(tmp_path, monkeypatch):
    for rel in {f for files in bench.KERNEL_SOURCES.values() for f in files}:
        p = tmp_path / rel
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text("// " + rel + "\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    dg = bench.source_digest(bench.KERNEL_SOURCES["gemm"])
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# kind workload bytes digest\n"
        f"gemm_c_fc block_bf16_d768 123456 {dg}\n"
        "gemm_c_proj block_bf16_d768 777 000000000000\n")
    assert bench.ncu_traffic("gemm_c_fc", "block_bf16_d768") == 123456.0
    assert bench.ncu_traffic("gemm_c_fc", "forward_bf16_gpt2_small") is None
    assert bench.ncu_traffic("gemm_c_proj", "block_bf16_d768") is None  # stale digest
    (tmp_path / bench.KERNEL_SOURCES["gemm"][0]).write_text("// changed\n")
    assert bench.ncu_traffic("gemm_c_fc", "block_bf16_d768") is None


def test_prefill_and_decode_attention_are_keyed_by_their_own_sources(tmp_path, monkeypatch):
    """A change to the prefill attention's source voids only the prefill
    figure: the decode attention (and its combine) are keyed by theirs."""
    assert bench.kernel_family("attention_prefill") == "attention_prefill"
    assert bench.kernel_family("attention_decode") == "attention_decode"
    assert bench.kernel_family("attention_decode_combine") == "attention_decode"
    for rel in {f for files in bench.KERNEL_SOURCES.values() for f in files}:
        p = tmp_path / rel
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text("// " + rel + "\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    dp = bench.source_digest(bench.KERNEL_SOURCES["attention_prefill"])
    dd = bench.source_digest(bench.KERNEL_SOURCES["attention_decode"])
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        f"attention_prefill block_bf16_d768 100 {dp}\n"
        f"attention_decode decode_bf16_gpt2_medium 200 {dd}\n")
    (tmp_path / "gpt_pre_norm_gb300/csrc/attn_tc.cu").write_text("// changed\n")
    assert bench.ncu_traffic("attention_prefill", "block_bf16_d768") is None
    assert bench.ncu_traffic("attention_decode", "decode_bf16_gpt2_medium") == 200.0
