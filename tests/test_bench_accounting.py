"""The benchmark's roofline accounting (bench.py), on CPU.

The algorithmic work of a step counts the block's own tensors only: the
touched experts' weights, the router weights, x read once, out, the logits and
the top-k; the intermediates x_perm, h and Y count for nothing.  These tests
write the expected figures out by hand for small layers and check the
dominant-kernel and whole-block roofline objects built from them.
"""
import numpy as np
import pytest

import bench
import moe_inputs as mi

PEAKS = {"bf16_tflops": 1000.0, "bf16_tflops_sustained": 800.0, "hbm_gbs": 5000.0,
         "source": "test"}


def cfg(T, H, E, K, I):
    return mi.MoEConfig(f"acct_{T}_{H}_{E}_{K}_{I}", T, H, E, K, I, True)


def test_weight_bytes():
    assert bench.WEIGHT_BYTES["bf16"] == 2.0
    # 4-bit codes and a bf16 scale and bias per 128 weights: 4.25 bits a weight
    assert bench.WEIGHT_BYTES["q4"] * 8 == pytest.approx(4.25)


def test_stage_work_by_hand():
    c = cfg(T=4, H=256, E=8, K=2, I=128)
    counts = np.array([3, 0, 2, 0, 1, 2, 0, 0])  # 4 experts touched, 8 pairs
    w, touched = bench.stage_work(c, counts)
    assert touched == 4
    # gate/up: two [I,H] matrices of each touched expert, x once; 2 flops per MAC, 2 GEMMs
    assert w["gate_up"]["bytes"] == 4 * 2 * 128 * 256 * 2 + 4 * 256 * 2
    assert w["gate_up"]["flops"] == 2 * 2 * (4 * 2) * 256 * 128
    # down: one [H,I] matrix per touched expert; no activations count
    assert w["down"]["bytes"] == 4 * 256 * 128 * 2
    assert w["down"]["flops"] == 2 * (4 * 2) * 128 * 256
    # router: x, W_router, logits, top-k indices and weights
    assert w["router"]["bytes"] == 4 * 256 * 2 + 8 * 256 * 2 + 4 * 8 * 4 + 4 * 2 * 8
    assert w["router"]["flops"] == 2 * 4 * 256 * 8
    # the gather and the combine only move intermediates: out is all they own
    assert w["combine"]["bytes"] == 4 * 256 * 2 and w["combine"]["flops"] == 0
    # the fused decode kernel carries gate/up, down and the combine
    wf, _ = bench.stage_work(c, counts, fused=True)
    for k in ("bytes", "flops"):
        assert wf["gate_up"][k] == w["gate_up"][k] + w["down"][k] + w["combine"][k]
    # 4-bit weights scale only the weight bytes
    wq, _ = bench.stage_work(c, counts, wb=bench.WEIGHT_BYTES["q4"])
    assert wq["down"]["bytes"] == pytest.approx(4 * 256 * 128 * 0.53125)
    assert wq["gate_up"]["bytes"] == pytest.approx(4 * 2 * 128 * 256 * 0.53125 + 4 * 256 * 2)


def test_block_work_by_hand():
    c = cfg(T=16, H=512, E=4, K=2, I=256)
    counts = np.array([10, 0, 12, 10])
    flops, byts = bench.block_work(c, counts)
    assert flops == 6 * 16 * 2 * 512 * 256 + 2 * 16 * 512 * 4
    assert byts == 3 * 3 * 512 * 256 * 2 + 4 * 512 * 2 + 2 * 16 * 512 * 2 + 16 * 4 * 4 + 16 * 2 * 8 + 4


def test_roofline_picks_the_dominant_kernel_and_its_bound():
    c = cfg(T=4096, H=2048, E=128, K=8, I=768)
    counts = np.full(128, 256)
    w, _ = bench.stage_work(c, counts)
    stage_ms = {"router": 0.01, "dispatch": 0.02, "gate_up": 0.40, "down": 0.20, "combine": 0.02}
    r = bench.roofline_of(w, stage_ms, "tcgen05", PEAKS, c)
    assert r["kernel"] == "gate_up" and r["kernel_ms"] == 0.40
    fl, by = w["gate_up"]["flops"], w["gate_up"]["bytes"]
    # this stage is tensor-bound at these peaks: flops / peak > bytes / bandwidth
    assert fl / 1e15 > by / 5e12
    assert r["bound"] == "tensor"
    assert r["achieved"] == pytest.approx(fl / 0.40e-3 / 1e12)
    assert r["frac"] == pytest.approx(fl / 0.40e-3 / 1e15)
    assert r["frac_sustained"] == pytest.approx(fl / 0.40e-3 / 0.8e15)


def test_roofline_hbm_bound_decode():
    c = cfg(T=1, H=4096, E=128, K=8, I=1536)
    counts = np.zeros(128, dtype=int)
    counts[:8] = 1
    w, touched = bench.stage_work(c, counts, fused=True)
    assert touched == 8
    r = bench.roofline_of(w, {"router": 0.005, "gate_up": 0.07}, "tcgen05_decode", PEAKS, c)
    assert r["bound"] == "hbm" and r["kernel"] == "experts_fused"
    weights = 8 * 3 * 4096 * 1536 * 2
    assert w["gate_up"]["bytes"] == weights + 4096 * 2 + 4096 * 2
    assert r["frac"] == pytest.approx(w["gate_up"]["bytes"] / 0.07e-3 / 5e12)


def test_block_roofline_fraction():
    c = cfg(T=1, H=4096, E=128, K=8, I=1536)
    counts = np.zeros(128, dtype=int)
    counts[:8] = 1
    b = bench.block_roofline_of(c, counts, 2.0, 0.080, PEAKS)
    flops, byts = bench.block_work(c, counts)
    t_roof = max(flops / 1e15, byts / 5e12)
    assert b["bound"] == "hbm"
    assert b["frac"] == pytest.approx(t_roof / 0.080e-3)
    assert b["t_roof_us"] == pytest.approx(t_roof * 1e6)
    assert b["touched_experts"] == 8
