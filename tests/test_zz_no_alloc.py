"""moe_forward_noalloc: the forward for callers that may not allocate device
memory on the call path (fixed memory budgets, hosts that must not take the
allocator's locks, device memory owned by another runtime).  It runs the same
kernels as moe_forward with its scratch in a 32 MiB array inside the library.

Called here through the C ABI (ctypes), twice in a row -- the second call finds
the first call's leftovers in the shared scratch -- and checked against
moe_forward with the tolerance the parity tests use.  This file is collected
last on purpose, and passes both alone and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_inputs as mi
from parity import OUT_REL, W_ATOL, bf16_to_f64, half_ulp_bf16

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def moe(cuda_ok):
    from mixture_experts_layer_98_b300 import build
    build.build()
    import mixture_experts_layer_98_b300 as m
    m.lib()
    return m


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(moe, inp, cfg):
    T, H, E, K, I = cfg.T, cfg.H, cfg.E, cfg.K, cfg.I
    d = inp["x"].device
    out = torch.empty((T, H), dtype=torch.bfloat16, device=d)
    logits = torch.empty((T, E), dtype=torch.float32, device=d)
    idx = torch.empty((T, K), dtype=torch.int32, device=d)
    w = torch.empty((T, K), dtype=torch.float32, device=d)
    aux = torch.empty((1,), dtype=torch.float32, device=d)
    rc = moe.lib().moe_forward_noalloc(
        _p(inp["x"]), T, H, _p(inp["W_router"]), _p(inp["W_gate"]), _p(inp["W_up"]),
        _p(inp["W_down"]), E, K, I, int(cfg.norm), _p(out), _p(logits), _p(idx), _p(w), _p(aux),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, moe.lib().moe_strerror(rc)
    return out, logits, idx, w, aux


def _check_close(got, ref):
    out_g, lg_g, idx_g, w_g, aux_g = [t.cpu() for t in got]
    out_r, lg_r, idx_r, w_r, aux_r = [t.cpu() for t in ref]
    assert torch.equal(idx_g, idx_r)
    assert (w_g - w_r).abs().max().item() <= W_ATOL
    assert (lg_g - lg_r).abs().max().item() <= 1e-5 * (1 + lg_r.abs().max().item())
    assert abs(aux_g.item() - aux_r.item()) <= 1e-5
    a = out_g.double().numpy()
    r = out_r.double().numpy()
    rms = float(np.sqrt((r ** 2).mean()))
    assert (np.abs(a - r) <= OUT_REL * rms + half_ulp_bf16(r)).all()


@pytest.mark.parametrize("name", ["decode_t16", "tiny"])
def test_noalloc_matches_forward_on_two_calls(moe, name):
    cfg = mi.CONFIGS[name]
    assert moe.moe_workspace_bytes(cfg.T, cfg.H, cfg.E, cfg.K, cfg.I) <= SCRATCH_BYTES
    inp = mi.make_inputs(cfg, "cuda")
    ref = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                              inp["W_up"], inp["W_down"], cfg.K, cfg.norm)]
    first = _noalloc(moe, inp, cfg)
    second = _noalloc(moe, inp, cfg)
    torch.cuda.synchronize()
    _check_close(first, ref)
    _check_close(second, ref)


def test_noalloc_two_different_calls_in_a_row(moe):
    # a larger batch leaves more scratch behind; a smaller one must not see it
    big = mi.MoEConfig("big", 200, 4096, 128, 8, 1536, True, seed=4)
    small = mi.CONFIGS["decode_t4"]
    for cfg in (big, small):
        inp = mi.make_inputs(cfg, "cuda")
        ref = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                                  inp["W_up"], inp["W_down"], cfg.K, cfg.norm)]
        got = _noalloc(moe, inp, cfg)
        torch.cuda.synchronize()
        _check_close(got, ref)
        assert np.isfinite(bf16_to_f64(got[0].cpu().view(torch.int16).numpy().view(np.uint16))).all()


def test_noalloc_rejects_sizes_beyond_its_scratch(moe):
    cfg = mi.CONFIGS["prefill_h2048"]
    assert moe.moe_workspace_bytes(cfg.T, cfg.H, cfg.E, cfg.K, cfg.I) > SCRATCH_BYTES
    inp = mi.make_inputs(mi.MoEConfig("w", 1, cfg.H, cfg.E, cfg.K, cfg.I, True), "cuda")
    x = torch.zeros((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(x)
    z = ctypes.c_void_p(0)
    rc = moe.lib().moe_forward_noalloc(
        _p(x), cfg.T, cfg.H, _p(inp["W_router"]), _p(inp["W_gate"]), _p(inp["W_up"]),
        _p(inp["W_down"]), cfg.E, cfg.K, cfg.I, 1, _p(out), z, z, z, z,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 4  # MOE_ERR_WORKSPACE
