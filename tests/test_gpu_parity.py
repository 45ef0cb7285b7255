"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Stage tests feed identical inputs to one stage (routing from given logits,
dispatch from given selections, combine from given expert outputs) and require
bit-exact integer results.  End-to-end tests run the whole block on every
configuration of the workload set -- fully where the oracle is quick, on a
seeded sample of token rows at the full prefill sizes -- through both expert
paths (tcgen05 grouped GEMMs and weight streaming).
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity import compare, gpu_forward, host_bits, tile_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_ok):
    import mixture_experts_layer_98_b300 as m
    from mixture_experts_layer_98_b300 import build
    build.build()
    m.lib()
    yield m
    m.moe_set_expert_path(m.MOE_PATH_AUTO)


@pytest.fixture
def path(moe, request):
    prev = moe.moe_set_expert_path(request.param)
    yield request.param
    moe.moe_set_expert_path(prev)


PATHS = [pytest.param(2, id="tcgen05"), pytest.param(1, id="streaming"),
         pytest.param(3, id="tcgen05_wt"), pytest.param(4, id="tcgen05_pair"),
         pytest.param(5, id="tcgen05_decode")]


# ---- stage parity -----------------------------------------------------------------

@pytest.mark.parametrize("E,K", [(8, 2), (16, 4), (128, 8), (256, 16), (1, 1), (33, 7),
                                 (64, 16)])
@pytest.mark.parametrize("norm", [False, True])
def test_route_from_logits_bit_exact(moe, E, K, norm):
    rng = np.random.default_rng(E * 100 + K)
    T = 300
    l = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    l[:40] = np.round(l[:40] * 2) / 2  # exact ties
    l[40:45] = 0.0                     # all equal
    idx, w = moe.moe_dbg_route_from_logits(torch.from_numpy(l).cuda(), K, norm)
    ridx, rw = oracle.route_from_logits(l, K, norm)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.abs(w.cpu().numpy() - rw).max() <= 1e-5


@pytest.mark.parametrize("E,K", [(8, 2), (128, 8), (256, 16), (33, 7)])
@pytest.mark.parametrize("norm", [False, True])
def test_route_with_selection_bias_bit_exact(moe, E, K, norm):
    # keys logit + bias on multiples of 1/4: exact ties between keys
    rng = np.random.default_rng(E * 10 + K)
    T = 200
    l = (rng.integers(-12, 13, (T, E)) / 4).astype(np.float32)
    l[100:] = (rng.standard_normal((T - 100, E)) * 1.5).astype(np.float32)
    b = (rng.integers(-6, 7, E) / 4).astype(np.float32)
    idx, w = moe.moe_dbg_route_from_logits(torch.from_numpy(l).cuda(), K, norm,
                                           expert_bias=torch.from_numpy(b).cuda())
    ridx, rw = oracle.route_from_logits(l, K, norm, bias=b)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert np.abs(w.cpu().numpy() - rw).max() <= 1e-5


@pytest.mark.parametrize("T,E,K", [(1, 8, 2), (255, 8, 2), (256, 16, 4), (257, 128, 8),
                                   (4096, 128, 8), (1000, 256, 16), (37, 1, 1), (0, 8, 2)])
def test_permute_bit_exact(moe, T, E, K):
    rng = np.random.default_rng(T + E)
    idx = np.array([rng.permutation(E)[:K] for _ in range(T)], np.int32).reshape(T, K)
    d = moe.moe_dbg_permute(torch.from_numpy(idx).cuda(), E)
    r = oracle.dispatch(idx, E)
    assert np.array_equal(d["counts"].cpu().numpy(), r["counts"])
    assert np.array_equal(d["offsets"].cpu().numpy(), r["offsets"])
    if T:
        assert np.array_equal(d["perm_tok"].cpu().numpy(), r["perm_tok"])
        assert np.array_equal(d["perm_slot"].cpu().numpy(), r["perm_slot"])
        assert np.array_equal(d["inv"].cpu().numpy(), r["inv"])


@pytest.mark.parametrize("T,E,K,C", [(200, 16, 4, 30), (200, 16, 4, 1), (1000, 128, 8, 40),
                                     (3000, 16, 2, 300), (257, 8, 2, 64)])
def test_permute_with_capacity_bit_exact(moe, T, E, K, C):
    # one-CTA dispatch (T <= 256) and chunked dispatch; capacities that drop
    # most pairs, some pairs, and (C = 300 at ~375 per expert) a few
    rng = np.random.default_rng(T + C)
    idx = np.array([rng.permutation(E)[:K] for _ in range(T)], np.int32).reshape(T, K)
    d = moe.moe_dbg_permute(torch.from_numpy(idx).cuda(), E, capacity=C)
    r = oracle.dispatch(idx, E, capacity=C)
    n = int(r["offsets"][E])
    assert np.array_equal(d["counts"].cpu().numpy(), r["counts"])
    assert np.array_equal(d["offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(d["inv"].cpu().numpy(), r["inv"])
    assert np.array_equal(d["perm_tok"].cpu().numpy()[:n], r["perm_tok"])
    assert np.array_equal(d["perm_slot"].cpu().numpy()[:n], r["perm_slot"])


def test_permute_skewed_all_to_one_expert(moe):
    T, E, K = 3000, 16, 2
    idx = np.zeros((T, K), np.int32)
    idx[:, 1] = 5
    d = moe.moe_dbg_permute(torch.from_numpy(idx).cuda(), E)
    r = oracle.dispatch(idx, E)
    for k in ("counts", "offsets", "perm_tok", "perm_slot"):
        assert np.array_equal(d[k].cpu().numpy(), r[k]), k
    assert np.array_equal(d["inv"].cpu().numpy(), r["inv"])


@pytest.mark.parametrize("T,K,H", [(1, 1, 64), (77, 8, 2048), (300, 2, 128)])
def test_combine(moe, T, K, H):
    g = torch.Generator().manual_seed(T)
    Y = torch.randn((T * K, H), generator=g).to(torch.bfloat16)
    inv = torch.randperm(T * K, generator=g).to(torch.int32).view(T, K)
    out = moe.moe_dbg_combine(Y.cuda(), inv.cuda()).cpu()
    ref = torch.zeros((T, H), dtype=torch.float64)
    for k in range(K):  # sum in k order, fp32 like the kernel's contract
        ref += Y[inv[:, k].long()].to(torch.float64)
    ref32 = torch.zeros((T, H), dtype=torch.float32)
    for k in range(K):
        ref32 += Y[inv[:, k].long()].to(torch.float32)
    assert torch.equal(out, ref32.to(torch.bfloat16))
    assert (out.to(torch.float64) - ref).abs().max() <= 2 ** -7 * ref.abs().max() + 1e-30


# ---- end to end -------------------------------------------------------------------

def run_case(cfg, rows=None):
    inp = mi.make_inputs(cfg, "cuda")
    g = gpu_forward(inp, cfg.K, cfg.norm)
    b = host_bits(inp)
    return compare(b, g, cfg.K, cfg.norm, rows=rows)


@pytest.mark.parametrize("path", PATHS, indirect=True)
def test_tiny(moe, path):
    rep = run_case(mi.CONFIGS["tiny"])
    assert rep["out_excess"] <= 0


@pytest.mark.parametrize("path", PATHS, indirect=True)
@pytest.mark.parametrize("T,H,E,K,I,norm", [
    (1, 64, 1, 1, 64, False), (3, 128, 2, 1, 128, True), (17, 128, 8, 3, 192, True),
    (129, 256, 16, 4, 128, False), (129, 128, 128, 8, 64, True), (300, 192, 8, 8, 320, True),
    (513, 512, 32, 2, 256, True), (64, 128, 4, 4, 256, True),
    # shapes the weights-as-M kernels tile (I % 128 == 0, H % 256 == 0): one row,
    # ragged 16-row boxes, several 64-row tiles per expert, an expert with no rows
    (1, 256, 1, 1, 128, False), (17, 256, 8, 3, 256, True), (300, 256, 4, 2, 128, True),
    (77, 512, 64, 6, 384, False),
    # few items: gate/up K split into 2 slices; 5 slices of 9,9,9,9,8 k-blocks;
    # down split into 2 slices
    (2, 1024, 16, 2, 512, True), (1, 2816, 4, 2, 128, False), (3, 1280, 8, 2, 640, True),
    (1, 512, 4, 2, 1024, True),
    # CTA-pair tiles: experts of ~750 rows (three 256-row tiles and a ragged
    # one), of ~233 rows (one M=256 tile with a ragged second half), and an
    # expert with exactly 256 rows (E = 1)
    (1500, 512, 4, 2, 256, True), (700, 256, 3, 1, 384, False), (256, 256, 1, 1, 128, True)])
def test_shape_fuzz(moe, path, T, H, E, K, I, norm):
    cfg = mi.MoEConfig("fuzz", T, H, E, K, I, norm, seed=T + H + E)
    run_case(cfg)


@pytest.mark.parametrize("path", [pytest.param(0, id="auto"), pytest.param(1, id="streaming")],
                         indirect=True)
@pytest.mark.parametrize("name", ["decode_t1", "decode_t4", "decode_t16", "decode_t64",
                                  "mixtral_decode_t1"])
def test_decode_sweep(moe, path, name):
    cfg = mi.CONFIGS[name]
    if path == 1 and cfg.I * 8 * 2 > 200 * 1024:
        # the streaming kernels stage 8 rows of I in shared memory: refused up front
        inp = mi.make_inputs(cfg, "cuda")
        with pytest.raises(moe.MoEError):
            moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"],
                            inp["W_down"], cfg.K, cfg.norm)
        return
    run_case(cfg)


@pytest.mark.parametrize("path", PATHS[:1], indirect=True)
def test_prefill_h2048_sampled(moe, path):
    cfg = mi.CONFIGS["prefill_h2048"]
    inp = mi.make_inputs(cfg, "cuda")
    g = gpu_forward(inp, cfg.K, cfg.norm)
    compare(host_bits(inp), g, cfg.K, cfg.norm, rows=tile_rows(g["idx"], cfg.E, n_random=96))


# Output rows at the full prefill sizes: every expert's first and last row and
# the first row of its last 64/128/256-row tile (the ragged tails and the M=64
# tail MMAs), every 8th tile of the hot experts' long runs, and 48 random
# tokens (routing is compared on every token).
@pytest.mark.parametrize("name", ["prefill_h4096", "skew", "mixtral_prefill"])
def test_large_sampled(moe, name):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    g = gpu_forward(inp, cfg.K, cfg.norm)
    rows = tile_rows(g["idx"], cfg.E)
    rep = compare(host_bits(inp), g, cfg.K, cfg.norm, rows=rows)
    assert rep["out_excess"] <= 0


# The CTA-pair grouped GEMMs at full size (AUTO runs them for few, large
# experts only): 256-row tiles with ragged M=256 and M=128 tails, skewed
# expert loads, and an expert capacity (dropped pairs leave holes in Y).
@pytest.mark.parametrize("name,cf", [("prefill_h2048", 0.0), ("skew", 0.0),
                                     ("prefill_h2048", 1.0)])
def test_pair_path_large_sampled(moe, name, cf):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    prev = moe.moe_set_expert_path(moe.MOE_PATH_TCGEN05_PAIR)
    try:
        out, lg, idx, w, aux = moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"],
                                                    inp["W_up"], inp["W_down"], cfg.K, cfg.norm,
                                                    capacity_factor=cf)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_expert_path(prev)
    g = dict(out=mi.bits(out), logits=lg.cpu().numpy(), idx=idx.cpu().numpy(),
             w=w.cpu().numpy(), aux=float(aux.cpu()[0]), counts=None)
    C = oracle.capacity_of(cf, cfg.T, cfg.K, cfg.E) if cf > 0 else 0
    rows = tile_rows(g["idx"], cfg.E, capacity=C)
    rep = compare(host_bits(inp), g, cfg.K, cfg.norm, rows=rows, capacity=C)
    assert rep["out_excess"] <= 0
    assert moe.moe_device_status() == 0


# The fused decode kernel (gate/up, down and the combine in one launch) runs
# the same units with the same arithmetic as the three separate kernels: the
# results must agree bit for bit -- one token with a 3-way K split of gate/up,
# a few tokens, 64 tokens (one 64-row tile per expert), two experts of 14336
# rows, split shapes from the fuzz list, and a capacity that drops pairs.  Up
# to six tokens the fused kernel also routes the batch itself (the separate
# path runs the one-CTA routing kernel): logits, top-k, aux and the expert
# counts must agree bit for bit too, with and without a capacity, at the
# largest batch routed in the kernel (6) and the smallest that is not (7).
@pytest.mark.parametrize("name,cf", [("decode_t1", 0.0), ("decode_t4", 0.0), ("decode_t16", 0.0),
                                     ("decode_t64", 0.0), ("mixtral_decode_t1", 0.0),
                                     ("decode_t16", 1.0), ("decode_t64", 1.0),
                                     ("decode_t4", 1.0), ("split_b", 1.0),
                                     ("edge_t6", 0.0), ("edge_t6", 1.25), ("edge_t7", 0.0),
                                     ("split_a", 0.0), ("split_b", 0.0)])
def test_decode_fused_is_bitwise_the_three_kernels(moe, name, cf):
    extra = {"split_a": mi.MoEConfig("split_a", 2, 1024, 16, 2, 512, True, seed=7),
             "split_b": mi.MoEConfig("split_b", 3, 1280, 8, 2, 640, True, seed=8),
             "edge_t6": mi.MoEConfig("edge_t6", 6, 1024, 32, 4, 512, True, seed=9),
             "edge_t7": mi.MoEConfig("edge_t7", 7, 1024, 32, 4, 512, True, seed=10)}
    cfg = extra.get(name) or mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    res, counts = {}, {}
    for p in (moe.MOE_PATH_TCGEN05_WT, moe.MOE_PATH_TCGEN05_DECODE):
        prev = moe.moe_set_expert_path(p)
        try:
            res[p] = [t.clone() for t in moe.moe_forward_opts(
                inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"], cfg.K,
                cfg.norm, capacity_factor=cf)]
            torch.cuda.synchronize()
            counts[p] = moe.moe_last_expert_counts(cfg.E).clone()
        finally:
            moe.moe_set_expert_path(prev)
    for u, v in zip(res[moe.MOE_PATH_TCGEN05_WT], res[moe.MOE_PATH_TCGEN05_DECODE]):
        assert torch.equal(u, v)
    assert torch.equal(counts[moe.MOE_PATH_TCGEN05_WT], counts[moe.MOE_PATH_TCGEN05_DECODE])
    idx = res[moe.MOE_PATH_TCGEN05_DECODE][2].cpu().numpy()
    assert np.array_equal(counts[moe.MOE_PATH_TCGEN05_DECODE].numpy(),
                          np.bincount(idx.ravel(), minlength=cfg.E))
    assert moe.moe_device_status() == 0


def test_zero_tokens(moe):
    cfg = mi.MoEConfig("zero", 0, 128, 8, 2, 256, True)
    inp = mi.make_inputs(cfg, "cuda")
    out, logits, idx, w, aux = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                               inp["W_up"], inp["W_down"], 2, True)
    torch.cuda.synchronize()
    assert out.shape == (0, 128) and float(aux.cpu()[0]) == 0.0


def test_all_tokens_one_expert(moe):
    # x[:,0] = 1 with a large router bias column steers every token to experts 3, 6.
    cfg = mi.MoEConfig("hot", 700, 256, 16, 2, 256, True, seed=3)
    inp = mi.make_inputs(cfg, "cuda")
    inp["x"][:, 0] = 1.0
    inp["W_router"][:, 0] = 0.0
    inp["W_router"][3, 0] = 30.0
    inp["W_router"][6, 0] = 20.0
    g = gpu_forward(inp, 2, True)
    assert (g["idx"][:, 0] == 3).all() and (g["idx"][:, 1] == 6).all()
    compare(host_bits(inp), g, 2, True)


def test_deterministic(moe):
    cfg = mi.CONFIGS["prefill_h2048"]
    inp = mi.make_inputs(cfg, "cuda")
    a = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                        cfg.K, cfg.norm)
    a = [t.clone() for t in a]
    b = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                        cfg.K, cfg.norm)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert moe.moe_device_status() == 0


def test_decode_repeatable_with_dirty_workspace(moe):
    # One decode token splits the expert GEMMs along K (arrival counters in the
    # workspace); a caller workspace full of 0xFF bytes and repeated calls must
    # give the same bits as a fresh forward.
    cfg = mi.CONFIGS["decode_t1"]
    inp = mi.make_inputs(cfg, "cuda")
    ref = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                              inp["W_up"], inp["W_down"], cfg.K, cfg.norm)]
    nbytes = moe.moe_workspace_bytes(cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)
    ws = torch.full((nbytes,), 255, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        got = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"],
                              inp["W_down"], cfg.K, cfg.norm, workspace=ws)
        torch.cuda.synchronize()
        for u, v in zip(ref, got):
            assert torch.equal(u, v)
    assert moe.moe_device_status(ws, (cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)) == 0


def _bias_for(cfg, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(cfg.E) * 0.5).astype(np.float32)


@pytest.mark.parametrize("name,T", [("decode_t4", None), ("decode_t64", None),
                                    ("tiny", None), ("prefill_h2048", 512)])
def test_forward_with_selection_bias(moe, name, T):
    # T <= 32: routing in the one-CTA dispatch; 64: routing kernel after the
    # CUDA-core router; 512: after the tensor-core router
    cfg = mi.CONFIGS[name]
    if T is not None:
        cfg = mi.MoEConfig(name + "_t", T, cfg.H, cfg.E, cfg.K, cfg.I, cfg.norm, seed=cfg.seed)
    inp = mi.make_inputs(cfg, "cuda")
    bias = _bias_for(cfg, 5)
    out, lg, idx, w, aux = moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"],
                                                inp["W_up"], inp["W_down"], cfg.K, cfg.norm,
                                                expert_bias=torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    g = dict(out=mi.bits(out), logits=lg.cpu().numpy(), idx=idx.cpu().numpy(),
             w=w.cpu().numpy(), aux=float(aux.cpu()[0]), counts=None)
    rep = compare(host_bits(inp), g, cfg.K, cfg.norm, bias=bias)
    # the bias moved selections (it is large next to the logit spread at these sizes)
    plain = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"],
                            inp["W_down"], cfg.K, cfg.norm)
    torch.cuda.synchronize()
    assert not torch.equal(plain[2], idx), rep


# The capacity range of the csdn page (section "容量因子设计": factor 1.0-1.25):
# at skew the two hot experts keep 8-10 % of their ~16k pairs, so most tokens
# lose pairs; under a capacity the weighted expert outputs stay fp32 until the
# combine.  Small configs run every row; the large ones the tile-boundary rows
# of the kept pairs (every expert's first, last and last-tile rows, the hot
# experts' runs) and 48 random tokens.
@pytest.mark.parametrize("name,cf", [("tiny", 1.0), ("decode_t4", 1.0), ("decode_t64", 1.0),
                                     ("decode_t64", 1.25), ("prefill_h2048", 1.0),
                                     ("prefill_h4096", 1.0), ("skew", 1.0), ("skew", 1.25)])
def test_forward_with_capacity(moe, name, cf):
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg, "cuda")
    C = oracle.capacity_of(cf, cfg.T, cfg.K, cfg.E)
    out, lg, idx, w, aux = moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"],
                                                inp["W_up"], inp["W_down"], cfg.K, cfg.norm,
                                                capacity_factor=cf)
    torch.cuda.synchronize()
    g = dict(out=mi.bits(out), logits=lg.cpu().numpy(), idx=idx.cpu().numpy(),
             w=w.cpu().numpy(), aux=float(aux.cpu()[0]), counts=None)
    keep = oracle.keep_mask(g["idx"], cfg.E, C)
    assert not keep.all()  # the capacity drops pairs at this size
    rows = None if cfg.T <= 64 else tile_rows(g["idx"], cfg.E, capacity=C)
    rep = compare(host_bits(inp), g, cfg.K, cfg.norm, rows=rows, capacity=C)
    print(f"[capacity] {name} cf={cf}: C={C}, kept {keep.mean():.3f} of the pairs, "
          f"max|err|/RMS = {rep['out_rel']:.2e}")
    assert moe.moe_device_status() == 0


def test_capacity_nobody_reaches_is_the_plain_forward(moe):
    # a capacity at or above every expert's load drops nothing: the routing
    # outputs are bitwise those of the plain forward, and the output is the
    # oracle's (it differs from the plain forward's only in keeping the
    # weighted expert outputs in fp32 until the combine)
    cfg = mi.CONFIGS["decode_t16"]
    inp = mi.make_inputs(cfg, "cuda")
    ref = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                              inp["W_up"], inp["W_down"], cfg.K, cfg.norm)]
    got = moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"],
                               inp["W_down"], cfg.K, cfg.norm,
                               capacity_factor=float(cfg.E))  # C = T·K >= any expert's load
    torch.cuda.synchronize()
    for u, v in zip(ref[1:], got[1:]):
        assert torch.equal(u, v)
    g = dict(out=mi.bits(got[0]), logits=got[1].cpu().numpy(), idx=got[2].cpu().numpy(),
             w=got[3].cpu().numpy(), aux=float(got[4].cpu()[0]), counts=None)
    C = oracle.capacity_of(float(cfg.E), cfg.T, cfg.K, cfg.E)
    compare(host_bits(inp), g, cfg.K, cfg.norm, capacity=C)


def test_zero_selection_bias_is_the_plain_forward(moe):
    cfg = mi.CONFIGS["decode_t16"]
    inp = mi.make_inputs(cfg, "cuda")
    ref = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                          cfg.K, cfg.norm)
    ref = [t.clone() for t in ref]
    got = moe.moe_forward_opts(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"],
                               inp["W_down"], cfg.K, cfg.norm,
                               expert_bias=torch.zeros(cfg.E, device="cuda"))
    torch.cuda.synchronize()
    for u, v in zip(ref, got):
        assert torch.equal(u, v)


def test_prefill_repeatable_over_many_forwards(moe):
    # The gate/up kernel's gathered A tiles reach the tensor cores through
    # cp.async and a proxy fence; a missing ordering would show up as rare
    # differences between otherwise identical forwards.
    cfg = mi.CONFIGS["prefill_h2048"]
    inp = mi.make_inputs(cfg, "cuda")
    ref = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                              inp["W_up"], inp["W_down"], cfg.K, cfg.norm)]
    out = torch.empty_like(ref[0])
    for _ in range(12):
        moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                        cfg.K, cfg.norm, out=out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref[0])
    assert moe.moe_device_status() == 0


def test_forward_ws_and_host_agree(moe):
    cfg = mi.MoEConfig("ws", 300, 256, 16, 4, 256, True, seed=5)
    inp = mi.make_inputs(cfg, "cuda")
    ref = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                          cfg.K, cfg.norm)
    nbytes = moe.moe_workspace_bytes(cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    got = moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                          cfg.K, cfg.norm, workspace=ws)
    torch.cuda.synchronize()
    for u, v in zip(ref, got):
        assert torch.equal(u, v)
    assert moe.moe_device_status(ws, (cfg.T, cfg.H, cfg.E, cfg.K, cfg.I)) == 0
    x_h = inp["x"].cpu().pin_memory()
    out_h = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    lg_h = torch.empty((cfg.T, cfg.E), dtype=torch.float32).pin_memory()
    aux_h = torch.empty(1, dtype=torch.float32).pin_memory()
    moe.moe_forward_host(x_h, inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"], cfg.K,
                         cfg.norm, out_h, router_logits_host=lg_h, aux_host=aux_h)
    assert torch.equal(out_h, ref[0].cpu())
    assert torch.equal(lg_h, ref[1].cpu())
    assert torch.equal(aux_h, ref[4].cpu())
    # too-small workspace is refused before any work
    with pytest.raises(moe.MoEError):
        moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"], inp["W_up"], inp["W_down"],
                        cfg.K, cfg.norm, workspace=ws[: nbytes // 2])


def test_paths_agree(moe):
    cfg = mi.MoEConfig("paths", 1000, 512, 32, 4, 384, True, seed=9)
    inp = mi.make_inputs(cfg, "cuda")
    res = {}
    for p in (1, 2, 3, 4):
        prev = moe.moe_set_expert_path(p)
        try:
            res[p] = [t.clone() for t in moe.moe_forward(inp["x"], inp["W_router"], inp["W_gate"],
                                                         inp["W_up"], inp["W_down"], cfg.K,
                                                         cfg.norm)]
        finally:
            moe.moe_set_expert_path(prev)
    torch.cuda.synchronize()
    b = res[2][0].float()
    rms = b.pow(2).mean().sqrt()
    for p in (1, 3, 4):
        assert torch.equal(res[p][2], res[2][2])  # same routing
        assert (res[p][0].float() - b).abs().max() <= 2e-2 * rms


@pytest.mark.parametrize("T", [64, 300])  # SIMT router below 128 tokens, tcgen05 router above
@pytest.mark.parametrize("norm", [False, True])
def test_router_exact_ties_zero_weights(moe, T, norm):
    # W_router = 0: every logit is exactly 0 on both sides -> experts 0..K-1,
    # weights 1/E (or 1/K renormalised), aux = 1
    cfg = mi.MoEConfig("zeros", T, 256, 16, 4, 128, norm, seed=11)
    inp = mi.make_inputs(cfg, "cuda")
    inp["W_router"].zero_()
    g = gpu_forward(inp, cfg.K, norm)
    assert (g["idx"] == np.arange(cfg.K)).all()
    assert np.abs(g["w"] - (1.0 / cfg.K if norm else 1.0 / cfg.E)).max() < 1e-6
    assert abs(g["aux"] - 1.0) < 1e-5
    compare(host_bits(inp), g, cfg.K, norm, max_near_ties=T)  # every token ties


@pytest.mark.parametrize("T", [100, 700])
def test_router_exact_ties_duplicate_rows(moe, T):
    # experts 2j and 2j+1 share a router row, so their logits tie exactly:
    # whenever 2j+1 is selected, 2j must be selected right before it
    cfg = mi.MoEConfig("dups", T, 512, 32, 6, 128, True, seed=12)
    inp = mi.make_inputs(cfg, "cuda")
    inp["W_router"][1::2] = inp["W_router"][0::2]
    g = gpu_forward(inp, cfg.K, cfg.norm)
    for t in range(T):
        row = g["idx"][t].tolist()
        for k, e in enumerate(row):
            if e % 2 == 1:
                assert k > 0 and row[k - 1] == e - 1, (t, row)
    compare(host_bits(inp), g, cfg.K, cfg.norm, max_near_ties=T)  # exact ties by construction
