"""The packed expert-weight layout and the forward that streams it.

moe_pack_experts is checked element by element against the layout the header
documents (a numpy transcription of its formula, independent of the CUDA
code).  The packed forward runs the same MMAs in the same order as the
row-major forward, so its outputs must be bitwise identical to moe_forward's;
it is also compared with the oracle like every other path.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from parity import compare, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    from mixture_experts_layer_98_b300 import build
    build.build()
    import mixture_experts_layer_98_b300 as m
    m.lib()
    yield m
    m.moe_set_expert_path(m.MOE_PATH_AUTO)


def layout_reference(W, rows_per_expert, cols):
    """Packed bytes of one row-major [E*R, C] bf16 matrix, from the documented
    formula: blocks (expert, 128-row block, 64-column block) of 16 KB, element
    (r, k) of a block at byte r*128 + (((k/8) ^ (r%8))*16) + (k%8)*2."""
    w = W.reshape(-1, cols)                       # uint16 bit patterns
    n_rb, n_kb = w.shape[0] // 128, cols // 64
    out = np.zeros(n_rb * n_kb * 8192, np.uint16)  # 16 KB = 8192 bf16
    r = np.arange(128)[:, None]
    k = np.arange(64)[None, :]
    pos = r * 64 + ((k // 8) ^ (r % 8)) * 8 + (k % 8)  # in bf16 elements
    for rb in range(n_rb):
        for kb in range(n_kb):
            blk = w[rb * 128:(rb + 1) * 128, kb * 64:(kb + 1) * 64]
            base = (rb * n_kb + kb) * 8192
            out[base + pos.ravel()] = blk.ravel()
    return out


def bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_pack_layout_matches_the_documented_formula(moe):
    cfg = mi.MoEConfig("pack", 1, 512, 3, 1, 256, True, seed=21)
    inp = mi.make_inputs(cfg, "cuda")
    pk = moe.moe_pack_experts(inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    got = pk.data.cpu().numpy().view(np.uint16)
    E, I, H = 3, 256, 512
    mat = E * I * H
    assert got.size == 3 * mat
    assert np.array_equal(got[:mat], layout_reference(bits(inp["W_gate"]), I, H))
    assert np.array_equal(got[mat:2 * mat], layout_reference(bits(inp["W_up"]), I, H))
    assert np.array_equal(got[2 * mat:], layout_reference(bits(inp["W_down"]), H, I))


def _both(moe, cfg, path=0):
    inp = mi.make_inputs(cfg, "cuda")
    prev = moe.moe_set_expert_path(path)
    try:
        ref = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                                  inp["W_up"], inp["W_down"], cfg.K, cfg.norm)]
        pk = moe.moe_pack_experts(inp["W_gate"], inp["W_up"], inp["W_down"])
        got = moe.moe_forward_packed(inp["x"], inp["W_router"], pk, cfg.K, cfg.norm)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_expert_path(prev)
    return inp, ref, got, pk


@pytest.mark.parametrize("name", ["decode_t1", "decode_t4", "decode_t16", "decode_t64",
                                  "prefill_h2048"])
def test_packed_forward_is_bitwise_the_row_major_forward(moe, name):
    cfg = mi.CONFIGS[name]
    _, ref, got, _ = _both(moe, cfg)
    for u, v in zip(ref, got):
        assert torch.equal(u, v)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("path", [2, 3, 4], ids=["tokens_as_m", "weights_as_m", "pair"])
@pytest.mark.parametrize("T,H,E,K,I,norm", [
    (1, 256, 1, 1, 128, False), (77, 512, 64, 6, 384, False), (300, 256, 4, 2, 128, True),
    (2, 1024, 16, 2, 512, True), (513, 512, 32, 2, 256, True)])
def test_packed_against_oracle(moe, path, T, H, E, K, I, norm):
    cfg = mi.MoEConfig("packed", T, H, E, K, I, norm, seed=T + H + E + 1)
    inp, ref, got, _ = _both(moe, cfg, path)
    for u, v in zip(ref, got):
        assert torch.equal(u, v)
    g = {"out": mi.bits(got[0]), "logits": got[1].cpu().numpy(), "idx": got[2].cpu().numpy(),
         "w": got[3].cpu().numpy(), "aux": float(got[4].cpu()[0]),
         "counts": moe.moe_last_expert_counts(E).numpy()}
    compare(host_bits(inp), g, K, norm)


def test_packed_host_call_and_caller_workspace(moe):
    cfg = mi.CONFIGS["decode_t16"]
    inp, ref, got, pk = _both(moe, cfg)
    x_h = inp["x"].cpu().pin_memory()
    out_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    moe.moe_forward_host_packed(x_h, inp["W_router"], pk, cfg.K, cfg.norm, out_h, aux_host=aux_h)
    assert torch.equal(out_h, ref[0].cpu())
    assert torch.equal(aux_h, ref[4].cpu())
    nbytes = moe.moe_workspace_bytes(cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)
    ws = torch.full((nbytes,), 255, dtype=torch.uint8, device="cuda")
    got2 = moe.moe_forward_packed(inp["x"], inp["W_router"], pk, cfg.K, cfg.norm, workspace=ws)
    torch.cuda.synchronize()
    for u, v in zip(ref, got2):
        assert torch.equal(u, v)
    assert moe.moe_device_status(ws, (cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)) == 0


def test_packed_with_selection_bias_matches_row_major(moe):
    cfg = mi.CONFIGS["decode_t64"]
    inp = mi.make_inputs(cfg, "cuda")
    bias = torch.from_numpy((np.random.default_rng(3).standard_normal(cfg.E) * 0.5)
                            .astype(np.float32)).cuda()
    ref = [t.clone() for t in moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"],
                                                   inp["W_up"], inp["W_down"], cfg.K, cfg.norm,
                                                   expert_bias=bias)]
    pk = moe.moe_pack_experts(inp["W_gate"], inp["W_up"], inp["W_down"])
    got = moe.moe_forward_opts(inp["x"], inp["W_router"], None, None, None, cfg.K, cfg.norm,
                               expert_bias=bias, packed=pk)
    torch.cuda.synchronize()
    for u, v in zip(ref, got):
        assert torch.equal(u, v)

