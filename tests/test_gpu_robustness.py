"""Failure paths and memory safety of the CUDA library, on the GPU.

- The bounded-wait machinery: a wait on an mbarrier that nothing arrives on
  gives up after its limit, records MOE_ERR_TIMEOUT and leaves the context
  usable (no fault, no hang).
- Guard bands: forwards write nothing past the end of the caller's workspace
  or outside their output tensors (buffers surrounded by sentinel bytes that
  must survive), on the one-CTA dispatch, chunked dispatch, split-K, and
  capacity paths.
- Bad options are refused before any work.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from parity import compare, gpu_forward, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    from mixture_experts_layer_98_b300 import build
    build.build()
    import mixture_experts_layer_98_b300 as m
    m.lib()
    return m


def test_bounded_wait_gives_up_and_the_context_survives(moe):
    assert moe.moe_dbg_wait_timeout(2_000_000) == 6  # MOE_ERR_TIMEOUT after ~2 ms
    cfg = mi.CONFIGS["tiny"]
    inp = mi.make_inputs(cfg, "cuda")
    compare(host_bits(inp), gpu_forward(inp, cfg.K, cfg.norm), cfg.K, cfg.norm)
    assert moe.moe_device_status() == 0


def test_bounded_wait_rejects_bad_limits(moe):
    with pytest.raises(moe.MoEError):
        moe.moe_dbg_wait_timeout(0)
    with pytest.raises(moe.MoEError):
        moe.moe_dbg_wait_timeout(10 ** 10)


# (workload, capacity factor, expert path: 0 AUTO, 4 CTA pairs, 5 fused decode)
CASES = [("tiny", 0.0, 0), ("decode_t1", 0.0, 0), ("decode_t64", 0.0, 0),
         ("prefill_h2048", 0.0, 0), ("prefill_h2048", 1.0, 0), ("decode_t16", 1.0, 0),
         ("prefill_h2048", 0.0, 4), ("prefill_h2048", 1.0, 4), ("decode_t64", 1.0, 5)]


@pytest.fixture
def on_path(moe, request):
    prev = moe.moe_set_expert_path(request.param)
    yield request.param
    moe.moe_set_expert_path(prev)


def _cases():
    return [pytest.param(n, cf, p, id=f"{n}-{cf}-path{p}") for n, cf, p in CASES]


@pytest.mark.parametrize("name,cf,on_path", _cases(), indirect=["on_path"])
def test_nothing_is_written_past_the_workspace(moe, name, cf, on_path):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    need = moe.moe_workspace_bytes(cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)
    guard = 2 << 20
    buf = torch.full((need + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                         cfg.K, cfg.norm, workspace=buf[:need], capacity_factor=cf)
    torch.cuda.synchronize()
    assert bool((buf[need:] == 0xA5).all())
    assert moe.moe_device_status(buf[:need], (cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)) == 0


def _guarded(shape, dtype, fill):
    """A tensor of `shape` inside a buffer with g >= 16 sentinel elements on
    each side (so the view stays 16-byte aligned); returns (buffer, view, g)."""
    rows, cols = shape
    g = max(cols, 16)
    buf = torch.full((rows * cols + 2 * g,), fill, dtype=dtype, device="cuda")
    return buf, buf[g:g + rows * cols].view(rows, cols), g


@pytest.mark.parametrize("name,cf,on_path", _cases(), indirect=["on_path"])
def test_nothing_is_written_outside_the_outputs(moe, name, cf, on_path):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    T, H, E, K = cfg.T, cfg.H, cfg.E, cfg.K
    ob, out, og = _guarded((T, H), torch.bfloat16, -7.0)
    lb, lg, lgg = _guarded((T, E), torch.float32, -7.0)
    ib, idx, ig = _guarded((T, K), torch.int32, -7)
    wb, w, wg = _guarded((T, K), torch.float32, -7.0)
    ab, aux, ag = _guarded((1, 1), torch.float32, -7.0)
    moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                         K, cfg.norm, out=out, router_logits=lg, topk_idx=idx, topk_w=w,
                         aux=aux.view(1), capacity_factor=cf)
    torch.cuda.synchronize()
    for buf, g in ((ob, og), (lb, lgg), (ib, ig), (wb, wg), (ab, ag)):
        assert bool((buf[:g] == -7).all()) and bool((buf[-g:] == -7).all())
    assert bool((idx >= 0).all()) and bool((idx < E).all())


def test_bad_options_are_refused(moe):
    cfg = mi.CONFIGS["tiny"]
    inp = mi.make_inputs(cfg, "cuda")
    args = (inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"], cfg.K,
            cfg.norm)
    with pytest.raises(moe.MoEError):
        moe.moe_forward_opts(*args, capacity_factor=-1.0)
    with pytest.raises(moe.MoEError):
        moe.moe_forward_opts(*args, capacity_factor=float("nan"))
    bias = torch.zeros(cfg.E + 1, device="cuda")[1:]  # 4-byte but not 16-byte aligned
    with pytest.raises(moe.MoEError):
        moe.moe_forward_opts(*args, expert_bias=bias)


def test_stage_calls_leave_the_forward_queries_intact(moe):
    # moe_last_expert_counts / moe_device_status read what the last forward on
    # the stream left in its workspace; a stage entry point called afterwards
    # on the same stream (with more tokens, so its scratch is larger) uses
    # scratch of its own and must not overwrite it
    cfg = mi.CONFIGS["decode_t16"]
    inp = mi.make_inputs(cfg, "cuda")
    g = gpu_forward(inp, cfg.K, cfg.norm)
    rng = np.random.default_rng(3)
    T = 5000
    idx = np.array([rng.permutation(cfg.E)[:cfg.K] for _ in range(T)], np.int32)
    moe.moe_dbg_permute(torch.from_numpy(idx).cuda(), cfg.E)
    torch.cuda.synchronize()
    counts = moe.moe_last_expert_counts(cfg.E).numpy()
    assert np.array_equal(counts, g["counts"])
    assert np.array_equal(counts, np.bincount(g["idx"].ravel(), minlength=cfg.E))
    assert moe.moe_device_status() == 0
