"""Comparison of the CUDA path with the CPU oracle on the same seeded inputs.

Acceptance (per output):
  router_logits  |Δ| <= 1e-5·(1 + |l|)
  topk_idx       identical, except tokens whose K-th and (K+1)-th (or adjacent
                 kept) probabilities differ by < 1e-6: more than one selection
                 is correct there; they are counted, their weights are not
                 compared, and their output rows are checked against the
                 oracle evaluated on the GPU's own selection
  topk_w         |Δ| <= 1e-5
  counts         bit-exact against the histogram of the GPU's own selection
  out            |out_gpu - out_exact| <= 2e-2 · RMS(out_exact) + ½ ulp_bf16(out_exact)
                 per element, out_exact being the oracle's block output before
                 its final rounding: the bound is the arithmetic budget plus
                 the half-ulp any bf16 result of that value must carry
  aux            |Δ| <= 1e-5 · max(1, aux)
"""
import numpy as np
import torch

import moe_inputs as mi
import oracle

LOGIT_RTOL = 1e-5
W_ATOL = 1e-5
OUT_REL = 2e-2
TIE_GAP = 1e-6


def half_ulp_bf16(v):
    """Half the spacing of bf16 numbers at |v| (normal range; subnormal floor)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def out_error(got_f64, ref_exact):
    """(max excess over the bound, max|err|/RMS) for the output check."""
    rms = float(np.sqrt(np.mean(ref_exact ** 2))) if ref_exact.size else 0.0
    err = np.abs(got_f64 - ref_exact)
    bound = OUT_REL * rms + half_ulp_bf16(ref_exact)
    return float((err - bound).max()) if err.size else -1.0, (float(err.max()) / rms
                                                               if rms > 0 else 0.0), rms


def bf16_to_f64(b):
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def host_bits(inputs):
    return {k: mi.bits(v) for k, v in inputs.items()}


def gpu_forward(inputs, K, norm):
    import mixture_experts_layer_98_b300 as moe
    out, logits, idx, w, aux = moe.moe_forward(inputs["x"], inputs["W_router"], inputs["W_gate"],
                                               inputs["W_up"], inputs["W_down"], K, norm)
    torch.cuda.synchronize()
    E = inputs["W_router"].shape[0]
    counts = moe.moe_last_expert_counts(E).numpy() if inputs["x"].shape[0] > 0 else None
    return dict(out=mi.bits(out), logits=logits.cpu().numpy(), idx=idx.cpu().numpy(),
                w=w.cpu().numpy(), aux=float(aux.cpu()[0]), counts=counts)


def tile_rows(idx, E, capacity=0, n_random=48, seed=0, tiles=(64, 128, 256)):
    """Token rows whose outputs exercise every expert's tile boundaries: for
    each expert, in dispatch order (token order within the expert, kept pairs
    only under a capacity), the token of its first and last row and of the
    first row of its last tile for each tile height the expert kernels use
    (64-row tails, 128-row tiles, 256-row CTA-pair tiles); for experts of
    >= 1024 rows also the first row of every 8th 128-row tile (the hot
    experts' long tile runs); plus a seeded random sample of n_random tokens."""
    idx = np.asarray(idx)
    T = idx.shape[0]
    keep = oracle.keep_mask(idx, E, capacity) if capacity else np.ones(idx.shape, bool)
    rows = set(mi.sample_rows(T, n_random, seed).tolist()) if T else set()
    tok = np.repeat(np.arange(T), idx.shape[1])
    ex = idx.ravel()
    kp = keep.ravel()
    order = np.lexsort((tok, ex))
    order = order[kp[order]]
    ex_sorted = ex[order]
    tok_sorted = tok[order]
    starts = np.searchsorted(ex_sorted, np.arange(E + 1))
    for e in range(E):
        toks = tok_sorted[starts[e]:starts[e + 1]]
        n = toks.size
        if n == 0:
            continue
        picks = {0, n - 1}
        for h in tiles:
            picks.add((n - 1) // h * h)
        if n >= 1024:
            picks.update(range(0, n, 8 * 128))
        rows.update(int(toks[i]) for i in picks)
    return np.array(sorted(rows), dtype=np.int32)


def near_tie_keys(logits, bias, K, rel):
    """Tokens where the ranking keys l + b (fp32) of two neighbours at the
    K/K+1 boundary, or of two adjacent kept experts, differ by less than the
    two logits' own error bounds rel·(1 + |l|) added: the logits' error can
    reorder such keys, so more than one selection is correct."""
    logits = np.asarray(logits, np.float64)
    keys = (logits + np.asarray(bias, np.float32)[None, :]).astype(np.float32).astype(np.float64)
    m = min(K + 1, keys.shape[1])
    order = np.argsort(-keys, axis=1, kind="stable")[:, :m]
    k = np.take_along_axis(keys, order, axis=1)
    err = rel * (1 + np.abs(np.take_along_axis(logits, order, axis=1)))
    d = k[:, :-1] - k[:, 1:]
    return np.where((d < err[:, :-1] + err[:, 1:]).any(axis=1))[0]


def compare(b, g, K, norm, rows=None, bias=None, capacity=0, max_near_ties=None, q4=None):
    """b: host bits of the inputs; g: GPU results; bias: the selection-only
    expert bias (float32 [E]) when the forward had one; capacity: the pairs
    each expert kept (0: no capacity); max_near_ties: the most near-tie
    tokens allowed (default max(4, T/100); tests that build exact ties on
    purpose pass T); q4: 4-bit experts (oracle.quantize_experts_q4) -- the
    oracle then computes with their exact weights q·s + b and ignores b's
    expert matrices.  Returns a report dict and raises AssertionError on any
    failed check."""
    T, H = b["x"].shape
    E = b["W_router"].shape[0]
    if q4 is None:
        o = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], K,
                               norm, rows=rows, bias=bias, capacity=capacity)

        def token_output(t, idx_row, w_row):
            return oracle.token_output(b["x"][t], idx_row, w_row, b["W_gate"], b["W_up"],
                                       b["W_down"], unrounded=True)[1]
    else:
        o = oracle.moe_forward_q4(b["x"], b["W_router"], q4, K, norm, rows=rows, bias=bias,
                                  capacity=capacity)

        def token_output(t, idx_row, w_row):
            return oracle.token_output_q4(b["x"][t], idx_row, w_row, q4, unrounded=True)[1]
    rep = {}
    # logits
    dl = np.abs(g["logits"].astype(np.float64) - o["logits"])
    rep["logit_err"] = float((dl / (1 + np.abs(o["logits"]))).max()) if T else 0.0
    assert rep["logit_err"] <= LOGIT_RTOL, rep
    # selection
    probs = oracle.softmax(o["logits"])
    if bias is None:
        ties = set(oracle.near_tie_tokens(probs, K, TIE_GAP).tolist())
    else:
        # with a selection bias the experts are ranked by the keys l + b: two
        # keys can trade places only if they differ by less than the two
        # logits' errors added, each at most the largest logit error measured
        # in this very comparison (not the looser test bound)
        ties = set(near_tie_keys(o["logits"], bias, K, max(rep["logit_err"], 1e-7)).tolist())
    mism = np.where((g["idx"] != o["idx"]).any(axis=1))[0]
    bad = [t for t in mism.tolist() if t not in ties]
    rep["near_ties"] = len(ties)
    rep["idx_mismatch"] = len(mism)
    print(f"[parity] T={T} near-tie tokens {len(ties)}, selection differs on {len(mism)}")
    assert not bad, f"top-k differs on non-tie tokens {bad[:10]}"
    # near ties are rare events of the logit distribution (a gap below 1e-6
    # between neighbouring probabilities): a large count would mean the
    # exclusion hides real selection errors
    assert len(ties) <= (max(4, T // 100) if max_near_ties is None else max_near_ties), rep
    keep = np.array([t for t in range(T) if t not in ties], dtype=np.int64)
    if keep.size:
        rep["w_err"] = float(np.abs(g["w"][keep] - o["w"][keep]).max())
        assert rep["w_err"] <= W_ATOL, rep
    if norm and T:
        assert np.abs(g["w"].astype(np.float64).sum(1) - 1).max() < 1e-5
    # counts of the GPU's own selection
    if g.get("counts") is not None:
        assert np.array_equal(g["counts"], np.bincount(g["idx"].ravel(), minlength=E))
    # aux
    rep["aux_err"] = abs(g["aux"] - o["aux"])
    if not mism.size:
        assert rep["aux_err"] <= 1e-5 * max(1.0, abs(o["aux"])), rep
    # output rows
    rows_arr = np.arange(T) if rows is None else np.asarray(rows)
    if rows_arr.size:
        ref = o["out_f64"].copy()
        if capacity and mism.size:
            # a different selection (at a near-tie) shifts which later pairs an
            # expert keeps: evaluate every checked row on the GPU's own selection
            keep = oracle.keep_mask(g["idx"], E, capacity)
            for j, t in enumerate(rows_arr.tolist()):
                ref[j] = token_output(t, g["idx"][t][keep[t]], g["w"][t][keep[t]])
        for j, t in enumerate(rows_arr.tolist()):
            if t in mism and not capacity:
                ref[j] = token_output(t, g["idx"][t], g["w"][t])
        got = bf16_to_f64(g["out"][rows_arr])
        assert np.isfinite(got).all()
        excess, rel, rms = out_error(got, ref)
        rep["out_rms"] = rms
        rep["out_rel"] = rel
        rep["out_excess"] = excess
        # the plain figure beside the bound's verdict: max|err| / RMS(oracle)
        print(f"[parity] {rows_arr.size} rows: max|err|/RMS = {rel:.3e}, "
              f"excess over 2e-2·RMS + half-ulp = {excess:.2e}")
        assert excess <= 0.0, rep
    return rep
