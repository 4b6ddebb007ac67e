"""bench.py's output line: the keys and units the measurement contract fixes.

The reference arm (the CPU oracle on a bounded sample) runs without a GPU; the
timed arm of the CUDA path needs one."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return r, (json.loads(lines[-1]) if lines else None)


def check_common(d, steps, warmup):
    assert d["metric"] == "SSU decode tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == warmup
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["data"].startswith("synthetic")
    assert d["config"]["workload"] == "mamba2-2.7b-decode-b256"


def test_reference_arm_line():
    r, d = run_bench("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    check_common(d, 3, 3)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == "tokens/s" and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_traffic_records_keyed_to_kernel_code(tmp_path, monkeypatch):
    """The ncu traffic record of a workload holds while the kernel code is the
    code it was captured on: a comment or whitespace edit keeps the key, a code
    edit (or a new source file) changes it, and the SSD and SSU keys are
    independent of each other's sources."""
    sys.path.insert(0, ROOT)
    import bench

    src = os.path.join(ROOT, "mamba2_ssm_decode_gb300", "csrc")
    dst = tmp_path / "mamba2_ssm_decode_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in os.listdir(src):
        if f.endswith((".cu", ".cuh")):
            (dst / f).write_text(open(os.path.join(src, f), encoding="utf-8").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    ssd, ssu = "ssd-prefill-2.7b", "mamba2-2.7b-decode"
    base = {w: bench.kernel_source_hash(w) for w in (ssd, ssu)}
    assert base[ssd] != base[ssu]
    scan = dst / "ssd.cu"
    text = scan.read_text()
    scan.write_text("// a new comment line\n/* and a block\n comment */\n" + text.replace(";\n", ";  \n", 3))
    assert {w: bench.kernel_source_hash(w) for w in (ssd, ssu)} == base
    scan.write_text(text.replace("kSL = 32;", "kSL = 16;", 1))
    assert bench.kernel_source_hash(ssd) != base[ssd] and bench.kernel_source_hash(ssu) == base[ssu]
    scan.write_text(text)
    (dst / "ssu_extra.cuh").write_text("int x;\n")
    assert bench.kernel_source_hash(ssu) != base[ssu] and bench.kernel_source_hash(ssd) == base[ssd]


def test_too_few_warmup_steps_rejected():
    r, d = run_bench("--steps", "3", "--warmup", "2", timeout=120)
    assert r.returncode != 0 and d is None
    assert "--warmup must be >= 3" in r.stderr


@pytest.mark.gpu
def test_cuda_arm_line():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssm_decode_gb300 import build
    build.build()
    r, d = run_bench("--steps", "20", "--warmup", "3", "--no-extras", "--cpu-seconds", "0.5")
    assert r.returncode == 0, r.stderr[-2000:]
    check_common(d, 20, 3)
    assert d["dtype"] == "f32"
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None or rf["traffic"] > 0
    e = d["e2e"]
    assert e["unit"] == "tokens/s" and 0 < e["value"] <= d["value"] * 1.05
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 20          # one SSU launch per timed step
    ck = d["clocks"]
    assert ck["sm_max_mhz"] > 0 and isinstance(ck["reasons"], list)
    assert ck["samples_in_timed_region"] > 0     # the clock record covers the timed steps
    assert d["device_error"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    assert cb["single_core_value"] > 0
    # the GPU step checked against the oracle on the sample, inside the tolerances
    assert cb["parity"]["ok"] and cb["parity"]["sequences"] > 0


@pytest.mark.gpu
def test_ssd_prefill_line():
    """The packed SSD prefill measured alone: per-call byte and flop rooflines,
    the end-to-end rate with its copies, and the GPU call checked against the
    fp64 oracle on a sample of sequences."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssm_decode_gb300 import build
    build.build()
    r, d = run_bench("--workload", "ssd-prefill-2.7b", "--steps", "5", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    assert d["metric"] == "packed SSD prefill tokens/s (1 GPU)" and d["steps"] == 5
    assert d["config"]["workload"] == "ssd-prefill-2.7b" and d["config"]["chunk_size"] == 256
    assert d["value"] > 0 and d["ms_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor") and rf["unit"] == "GB/s"
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["algorithmic_flops_per_call"] > 0 and 0 < rf["tensor_frac"] < 1.2
    assert d["gpu_launches"] == 3 * 5 and d["device_error"] == 0
    e = d["e2e"]
    assert 0 < e["value"] and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["parity"]["ok"], cb["parity"]
