"""4-bit group-quantised experts on the GPU (csdn page, section
"参数量化与存储优化"; the reading is in moe_b300.h and the oracle).

- The quantiser's codes, scales and biases are bitwise the oracle's, read back
  from the buffer through the layout the header documents (a numpy
  transcription of its formula, independent of the CUDA code).
- The dequantiser gives bitwise the oracle's w' = bf16(q·s + b).
- The 4-bit forward computes the bf16 forward on the dequantised weights
  (tokens on the MMA's M side instead of the weights, so only the fp32
  summation order differs): routing outputs bitwise equal, the block output
  within two bf16 ulps, at decode sizes, with K splits, at a prefill size,
  with a capacity and a selection bias; and it is compared with the
  oracle's 4-bit forward (on its own codes) at small and full decode sizes.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
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


def read_q4(buf, E, H, I):
    """(codes, s, b) per matrix from the documented layout: for each of W_gate,
    W_up, W_down a code section (4 KB blocks of 128 rows x 64 columns ordered
    (expert, row block, column block); row r = 8 words from byte r*32; word c
    holds columns 8c+2j in bits 4j.. and 8c+2j+1 in bits 16+4j..) and a scale
    section (512-byte blocks per (expert, row block, 128-column group); word r
    = bf16 s | bf16 b << 16)."""
    data = buf.cpu().numpy()
    out = []
    off = 0
    for R, C in ((I, H), (I, H), (H, I)):
        n_code = E * R * C // 2
        words = data[off:off + n_code].view(np.uint32).reshape(E, R // 128, C // 64, 128, 8)
        off += n_code
        codes = np.zeros((E, R, C), np.uint8)
        for j in range(4):
            lo = (words >> (4 * j)) & 0xF
            hi = (words >> (16 + 4 * j)) & 0xF
            # [E, rb, kb, r, c] -> columns kb*64 + 8c + 2j (+1)
            for half, v in ((0, lo), (1, hi)):
                col = (np.arange(C // 64)[:, None] * 64 + np.arange(8)[None, :] * 8
                       + 2 * j + half)  # [kb, c]
                codes.reshape(E, R // 128, 128, C)[:, :, :, col] = v.transpose(0, 1, 3, 2, 4)
        n_sc = E * R * (C // 128) * 4
        sw = data[off:off + n_sc].view(np.uint32).reshape(E, R // 128, C // 128, 128)
        off += n_sc
        sw = sw.transpose(0, 1, 3, 2).reshape(E, R, C // 128)
        out.append((codes, (sw & 0xFFFF).astype(np.uint16), (sw >> 16).astype(np.uint16)))
    assert off == data.size
    return out


SHAPES = [(8, 1024, 512), (4, 256, 384), (2, 512, 128)]


@pytest.mark.parametrize("E,H,I", SHAPES)
def test_quantiser_and_dequantiser_are_the_oracles(moe, E, H, I):
    cfg = mi.MoEConfig("q4", 4, H, E, 2, I, True, seed=E + H + I)
    inp = mi.make_inputs(cfg, "cuda")
    q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
    deq = moe.moe_dequantize_experts_q4(q4)
    torch.cuda.synchronize()
    assert q4.data.numel() == moe.moe_q4_experts_bytes(H, E, I)
    got = read_q4(q4.data, E, H, I)
    for name, (codes, s, b), dq in zip(("W_gate", "W_up", "W_down"), got, deq):
        rq, rs, rb = oracle.quantize_q4(mi.bits(inp[name]))
        assert np.array_equal(codes, rq), name
        assert np.array_equal(s, rs) and np.array_equal(b, rb), name
        assert np.array_equal(mi.bits(dq), oracle.dequantize_q4(rq, rs, rb)), name


def _bf16_forward_on(moe, cfg, inp, Wd3, **kw):
    prev = moe.moe_set_expert_path(moe.MOE_PATH_TCGEN05_WT)
    try:
        return [t.clone() for t in moe.moe_forward_opts(inp["x"], inp["W_router"], *Wd3, cfg.K,
                                                        cfg.norm, **kw)]
    finally:
        moe.moe_set_expert_path(prev)


def _same_forward(ref, got):
    """Routing outputs bitwise.  The block outputs differ only through the
    order of fp32 sums, after which h, Y and out are rounded to bf16: a
    different order can flip one of those roundings by one ulp, and a flipped
    Y term moves out by up to one ulp of that term, which exceeds a relative
    bound where the K terms of an output cancel.  So: every element within
    2^-6 of itself plus 2^-5 of the RMS (one ulp of any Y term below 4 RMS),
    and at most 1 % of the elements beyond 2^-6 of itself plus 1e-3 of the
    RMS.  A wrong token, feature or expert tile moves every output of a
    (token, expert) pair by about the size of its Y term: thousands of
    elements, by far more than either bound."""
    for i in (1, 2, 3, 4):  # logits, idx, w, aux
        assert torch.equal(ref[i], got[i])
    a, b = ref[0].float(), got[0].float()
    rms = a.pow(2).mean().sqrt()
    d = (a - b).abs()
    loose = d <= 2.0 ** -6 * a.abs() + 2.0 ** -5 * rms
    tight = d <= 2.0 ** -6 * a.abs() + 1e-3 * rms
    n_bad = int((~tight).sum())
    msg = (f"{n_bad} of {a.numel()} beyond the tight bound, max |diff| {float(d.max()):.3g}, "
           f"rms {float(rms):.3g}")
    assert bool(loose.all()), msg
    assert n_bad <= 0.01 * a.numel(), msg


def _q4_forward(moe, path, *args, **kw):
    prev = moe.moe_set_expert_path(path)
    try:
        return [t.clone() for t in moe.moe_forward_q4(*args, **kw)]
    finally:
        moe.moe_set_expert_path(prev)


# both 4-bit kernels: warp-level MMAs on registers (AUTO up to 64 tokens) and
# tcgen05 with the tokens on the M side (AUTO above)
KERNELS = {"warp_mma": 6, "tcgen05": 2}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name", ["decode_t1", "decode_t4", "decode_t16", "decode_t64",
                                  "mixtral_decode_t1", "split_a", "ragged_t24", "prefill_small"])
def test_q4_forward_is_the_bf16_forward_on_dequantised_weights(moe, name, kernel):
    extra = {"split_a": mi.MoEConfig("split_a", 2, 1024, 16, 2, 512, True, seed=7),
             "ragged_t24": mi.MoEConfig("ragged_t24", 24, 768, 4, 3, 384, True, seed=9),
             "prefill_small": mi.MoEConfig("prefill_small", 1024, 512, 16, 4, 256, True, seed=5)}
    cfg = extra.get(name) or mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
    deq = moe.moe_dequantize_experts_q4(q4)
    ref = _bf16_forward_on(moe, cfg, inp, deq)
    got = _q4_forward(moe, KERNELS[kernel], inp["x"], inp["W_router"], q4, cfg.K, cfg.norm)
    torch.cuda.synchronize()
    _same_forward(ref, got)
    assert moe.moe_device_status() == 0


# decode_t4 on the warp-MMA kernels: the gate/up kernel routes the batch itself
# (capacity drops and the selection bias inside the expert kernel)
@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("name", ["decode_t16", "decode_t4"])
def test_q4_options_capacity_and_bias(moe, kernel, name):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
    deq = moe.moe_dequantize_experts_q4(q4)
    bias = (torch.arange(cfg.E, device="cuda", dtype=torch.float32) % 7) * 0.01
    kw = dict(capacity_factor=1.0, expert_bias=bias)
    ref = _bf16_forward_on(moe, cfg, inp, deq, **kw)
    prev = moe.moe_set_expert_path(KERNELS[kernel])
    try:
        got = moe.moe_forward_opts(inp["x"], inp["W_router"], None, None, None, cfg.K, cfg.norm,
                                   q4=q4, **kw)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_expert_path(prev)
    _same_forward(ref, got)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("T,H,E,K,I,norm", [(17, 256, 8, 2, 256, True), (1, 512, 4, 2, 384, False),
                                            (40, 256, 16, 4, 128, True)])
def test_q4_forward_against_the_oracle(moe, T, H, E, K, I, norm, kernel):
    cfg = mi.MoEConfig("q4o", T, H, E, K, I, norm, seed=T + H)
    inp = mi.make_inputs(cfg, "cuda")
    q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
    out, lg, idx, w, aux = _q4_forward(moe, KERNELS[kernel], inp["x"], inp["W_router"], q4, K,
                                       norm)
    torch.cuda.synchronize()
    b = host_bits(inp)
    # the oracle's own quantiser, and its forward on the codes
    q4o = oracle.quantize_experts_q4(b["W_gate"], b["W_up"], b["W_down"])
    g = dict(out=mi.bits(out), logits=lg.cpu().numpy(), idx=idx.cpu().numpy(),
             w=w.cpu().numpy(), aux=float(aux.cpu()[0]), counts=None)
    compare(b, g, K, norm, q4=q4o)


@pytest.mark.parametrize("name,kernel", [("decode_t1", "warp_mma"), ("decode_t1", "tcgen05"),
                                         ("decode_t4", "warp_mma"), ("decode_t16", "warp_mma"),
                                         ("decode_t64", "warp_mma"),
                                         ("mixtral_decode_t1", "warp_mma")])
def test_q4_full_size_against_the_oracle(moe, name, kernel):
    # a full decode layer: the oracle quantises, with its own quantiser, the
    # experts the GPU selected (a selection the oracle does not share fails the
    # index check; the other experts' codes stay zero and are never read) and
    # runs the whole block on the codes
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
    out, lg, idx, w, aux = _q4_forward(moe, KERNELS[kernel], inp["x"], inp["W_router"], q4,
                                       cfg.K, cfg.norm)
    torch.cuda.synchronize()
    b = host_bits(inp)
    chosen = sorted(set(idx.cpu().numpy().ravel().tolist()))
    q4o = {}
    for m, name_q in (("W_gate", "gate"), ("W_up", "up"), ("W_down", "down")):
        E, R, C = b[m].shape
        q = np.zeros((E, R, C), np.uint8)
        sc = np.zeros((E, R, C // 128), np.uint16)
        bi = np.zeros((E, R, C // 128), np.uint16)
        for e in chosen:
            q[e], sc[e], bi[e] = oracle.quantize_q4(b[m][e])
        q4o[name_q] = (q, sc, bi)
    g = dict(out=mi.bits(out), logits=lg.cpu().numpy(), idx=idx.cpu().numpy(),
             w=w.cpu().numpy(), aux=float(aux.cpu()[0]), counts=None)
    compare(b, g, cfg.K, cfg.norm, q4=q4o)


@pytest.mark.parametrize("name", ["decode_t4", "prefill_small"])
def test_q4_host_entry_is_the_device_entry(moe, name):
    # moe_forward_host_q4 copies x in, runs the same kernels, copies the
    # results out: bitwise the device-buffer call's results
    cfg = (mi.MoEConfig("prefill_small", 1024, 512, 16, 4, 256, True, seed=5)
           if name == "prefill_small" else mi.CONFIGS[name])
    inp = mi.make_inputs(cfg, "cuda")
    q4 = moe.moe_quantize_experts_q4(inp["W_gate"], inp["W_up"], inp["W_down"])
    out, lg, idx, w, aux = [t.clone() for t in
                            moe.moe_forward_q4(inp["x"], inp["W_router"], q4, cfg.K, cfg.norm)]
    torch.cuda.synchronize()
    x_h = inp["x"].cpu().pin_memory()
    out_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    lg_h = torch.empty((cfg.T, cfg.E), dtype=torch.float32).pin_memory()
    idx_h = torch.empty((cfg.T, cfg.K), dtype=torch.int32).pin_memory()
    w_h = torch.empty((cfg.T, cfg.K), dtype=torch.float32).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    moe.moe_forward_host_q4(x_h, inp["W_router"], q4, cfg.K, cfg.norm, out_h,
                            router_logits_host=lg_h, topk_idx_host=idx_h, topk_w_host=w_h,
                            aux_host=aux_h)
    for dev, host in ((out, out_h), (lg, lg_h), (idx, idx_h), (w, w_h), (aux, aux_h)):
        assert torch.equal(dev.cpu(), host)


def test_q4_rejects_unsupported_shapes(moe):
    assert moe.moe_q4_experts_bytes(4096, 128, 1536) > 0
    assert moe.moe_q4_experts_bytes(128, 8, 256) == 0   # H % 256 != 0
    assert moe.moe_q4_experts_bytes(256, 8, 192) == 0   # I % 128 != 0
    W = torch.zeros((2, 192, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        moe.moe_quantize_experts_q4(W, W, torch.zeros((2, 256, 192), dtype=torch.bfloat16,
                                                      device="cuda"))
