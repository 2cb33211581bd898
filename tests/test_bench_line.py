"""The benchmark's JSON line (the contract the runs are read by), built by
bench.report() from a synthetic set of measurements, no GPU: every required
key is present, and the derived figures follow from the inputs -- value =
tokens / time, the dominant kernel's roofline = its algorithmic bytes per
launch / mean launch time / the measured peak, the DRAM traffic scaled by
the captured ratio, the prefill tensor fraction = FLOPs / time / peak."""
import argparse

import pytest

import bench
import synthetic


def _line():
    s = synthetic.SHAPES["4b"]
    args = argparse.Namespace(steps=256, warmup=3, prompt=2048, sessions=32, gpus=1, impl="ours")
    res = {
        "shape": s, "decode_ms": 576.0, "decode_ctx": (2048, 2304),
        "decode_profile": {"decode_step": (588.0, 256), "gemv": (0.0, 0)},
        "decode_profile_ctx": (2304, 2560),
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 6},
        "launches": 256, "per_op_ms": 780.0, "per_op_ctx": (2560, 2816),
        "prefill_ms": 16.3, "prefill_profile": {"gemm": (12.9, 144), "attention": (2.7, 36)},
        "b32_ms": 1024.0, "b32_ctx": [1000.0] * 32, "b32_profile": {"gemm": (100.0, 4640)},
        "b32_profile_steps": 32, "e2e_s": 0.61, "e2e_bytes": (4, 607748),
        "b32_clocks": {"sm_mhz": 1995.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 5},
    }
    pk = {"hbm_gbs": 6767.7, "bf16_tflops": 1929.6, "bf16_tflops_sustained": 1702.9}
    return s, args, res, pk, bench.report(args, res, 1, False, pk, "measured")


def test_required_keys():
    _, _, _, _, line = _line()
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches",
              "e2e"):
        assert k in line, k
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in line["roofline"], k
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in line["e2e"], k
    assert "workload" in line["config"] and "model" not in line["config"]
    # the batch-32 leg carries the clocks sampled during its own timed loop
    assert line["decode_b32"]["clocks"]["reasons"] == ["sw_power_cap"]
    assert line["higher_is_better"] is True and line["n_gpus"] == 1


def test_derived_figures():
    s, args, res, pk, line = _line()
    assert line["value"] == pytest.approx(256 / 0.576, rel=1e-3)
    kb = bench.decode_bytes(s, (2304 + 2560) / 2)
    ach = kb / (588.0 / 256 / 1e3) / 1e9
    r = line["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6767.7
    assert r["achieved"] == pytest.approx(ach, rel=1e-3)
    assert r["frac"] == pytest.approx(ach / 6767.7, rel=1e-3)
    assert r["traffic"] == pytest.approx(bench.DECODE_STEP_TRAFFIC_RATIO * kb, rel=1e-6)
    assert 1.0 <= bench.DECODE_STEP_TRAFFIC_RATIO < 1.01          # no re-reads
    pre = line["prefill"]
    assert pre["value"] == pytest.approx(2048 / 0.0163, rel=1e-3)
    assert pre["tc_roofline"]["frac"] == pytest.approx(bench.prefill_flops(s, 2048) / 0.0163 / 1e12 / 1929.6,
                                                         rel=1e-3)
    assert line["decode_b32"]["value"] == pytest.approx(32 * 256 / 1.024, rel=1e-3)
    assert line["e2e"]["value"] == pytest.approx(256 / 0.61, rel=1e-3)
