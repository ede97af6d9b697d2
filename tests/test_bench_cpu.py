"""bench.py's roofline arithmetic, on the host: the grouped GEMM's tensor fraction, and its
DRAM rate from the recorded ncu traffic next to the weight-stream bound."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


class Ctx:
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    peak_kind = "test"


def test_tensor_fraction_and_dram_rate_of_the_deepseek_shape():
    w = synth.WORKLOADS["dsv3_bf16"]
    alg = bench.algorithmic(w)
    # the expert weights: 256 experts x 3 matrices of 2048 x 7168, one shared expert, bf16
    assert alg["weight_bytes"] == (256 * 3 + 3) * 2048 * 7168 * 2
    r = bench.gemm_roofline(Ctx(), w, 5.0, alg)
    achieved = alg["gemm_flops"] / 5.0e-3 / 1e12
    assert r["bound"] == "tensor" and r["achieved"] == pytest.approx(achieved, rel=1e-3)
    assert r["frac"] == pytest.approx(achieved / 2000.0, abs=1e-3)
    assert r["frac_of_sustained"] == pytest.approx(achieved / 1600.0, abs=1e-3)
    # DRAM: the recorded traffic over the same 5 ms, against the copy rate
    assert r["dram_gbs"] == pytest.approx(r["traffic"] / 5.0e-3 / 1e9, rel=1e-3)
    assert r["dram_frac"] == pytest.approx(r["dram_gbs"] / 6000.0, abs=1e-3)
    assert r["weight_bound_ms"] == pytest.approx(alg["weight_bytes"] / 6000e9 * 1e3, abs=1e-3)


def test_no_dram_rate_without_recorded_traffic():
    w = synth.scaled(synth.WORKLOADS["dsv3_mxfp8"], T=4096)  # no ncu traffic on record for it
    r = bench.gemm_roofline(Ctx(), w, 10.0, bench.algorithmic(w))
    assert r["traffic"] is None and "dram_gbs" not in r


def test_fp32_layer_is_reported_against_the_alu_peak(monkeypatch):
    import torch

    class Props:
        multi_processor_count = 152

    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda dev: Props())
    w = synth.WORKLOADS["tiny_fp32"]
    r = bench.gemm_roofline(Ctx(), w, 0.02, bench.algorithmic(w))
    # 152 SMs x 128 fp32 FMA lanes x 2 flops x 2070 MHz
    assert r["bound"] == "alu" and r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], abs=1e-3)
