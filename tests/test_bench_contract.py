"""bench.py's host-side contract, without a GPU: the reference arm's JSON
line carries every key the benchmark contract names, with the units and
types it asks for; the roofline arithmetic picks the slower of the byte and
FLOP bounds and reports achieved / peak; the argument rules hold.  The oracle
step itself is replaced by a fake timer here (its arithmetic is pinned by the
oracle tests); only the bookkeeping around it is under test."""

import json

import numpy as np
import pytest

import bench
from lm_head_exact_gb300 import synthetic

PEAKS = {"hbm_gbs": 6781.1, "bf16_tflops": 1946.0, "bf16_tflops_sustained": 1699.3, "source": "measured"}


def test_reference_arm_json_line(monkeypatch, capsys):
    V = synthetic.SHAPES["llama3_8b"]["V"]
    calls = []

    def fake_step(h, W, temp, seed, step, rows):
        calls.append((h.shape, rows, step))
        return 1e-3 * rows / V                       # 1 ms for the whole vocabulary

    monkeypatch.setattr(bench, "_oracle_step", fake_step)
    monkeypatch.setattr(synthetic, "weights", lambda kind, *a, **k: np.zeros((1, 1), np.uint16))
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3", "--batch", "16"])
    line = capsys.readouterr().out.strip().splitlines()[-1]
    r = json.loads(line)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e",
                "gpu_launches"):
        assert key in r, key
    assert r["impl"] == "reference" and r["unit"] == "us/step" and r["higher_is_better"] is False
    assert r["steps"] == 4 and r["warmup"] == 3 and r["n_gpus"] == 1 and r["gpu_launches"] == 0
    assert r["value"] == pytest.approx(1000.0, rel=1e-6)            # 1 ms per full-vocabulary step
    assert r["ms_per_step"] == pytest.approx(r["value"] / 1e3, rel=1e-3)
    assert r["config"]["global_batch"] == 16 and "llama3_8b" in r["config"]["workload"]
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == r["value"] and cb["cores"] >= 1 and cb["sample"]
    assert r["e2e"] == {"value": r["value"], "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # 3 warm-up and 4 timed steps on B = 16 rows, after sizing the vocabulary slice
    timed = [c for c in calls if c[1] == V]
    assert len(timed) >= 7 and all(c[0] == (16, 4096) for c in calls)


def test_reference_arm_is_silent_off_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_roofline_bounds():
    d, V = 4096, 128256
    small = bench.roofline(16, d, V, 155.0, PEAKS)
    assert small["bound"] == "hbm" and small["unit"] == "GB/s" and small["peak"] == PEAKS["hbm_gbs"]
    nbytes = bench.algorithmic_bytes(16, d, V)
    assert nbytes == 2 * V * d + 2 * 16 * d + 16 * 16
    assert small["achieved"] == pytest.approx(nbytes / 155e-6 / 1e9, abs=0.1)
    assert small["frac"] == pytest.approx(small["achieved"] / PEAKS["hbm_gbs"], abs=1e-4)
    big = bench.roofline(1024, d, V, 600.0, PEAKS)
    assert big["bound"] == "tensor" and big["unit"] == "TFLOP/s"
    assert big["achieved"] == pytest.approx(2 * 1024 * d * V / 600e-6 / 1e12, abs=0.1)
    # the crossover: bytes / HBM = FLOPs / tensor peak near B = 300 on this head
    b_star = next(B for B in range(1, 2048)
                  if bench.roofline(B, d, V, 1.0, PEAKS)["bound"] == "tensor")
    assert 250 < b_star < 350
    bias = bench.roofline(8, 8192, V, 300.0, PEAKS, bias=True)
    assert bias["algorithmic_bytes"] == bench.algorithmic_bytes(8, 8192, V) + 4 * 8 * V


def test_argument_rules():
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])                       # the contract asks for W >= 3
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.warmup >= 3 and a.steps >= 1
