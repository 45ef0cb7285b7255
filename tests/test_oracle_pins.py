"""Pins that tie the CPU oracle to something other than itself.

Each pin checks the oracle against what the pages print (worked examples under
tests/golden/), a closed form, an invariant, a special case that reduces to a
library routine, or brute force on tiny inputs.  test_pins_catch_planted_mistakes
rebuilds the oracle with one plausible mistake planted at a time and checks
that at least one pin fails for each.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import scipy.special
import torch

import moe_inputs as mi
import oracle
from conftest import GOLDEN

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ---- independent helpers (not the oracle's code) ---------------------------

def bf16_bits_to_f64(b):
    """bf16 bits -> float64 via torch (a library conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def f64_rne_bf16_value(v):
    """Round float64 values to the nearest bf16 value, ties to even, by integer
    arithmetic on the float64 bits (normal range only).  Returns float64."""
    v = np.asarray(v, np.float64)
    u = v.view(np.uint64)
    shift = np.uint64(45)  # float64 keeps 52 fraction bits, bf16 keeps 7
    lsb = (u >> shift) & np.uint64(1)
    u2 = ((u + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb) >> shift) << shift
    return u2.view(np.float64)


def np_swiglu(x, Wg, Wu, Wd, round_a=True):
    """float64 numpy expert MLP: down(silu(gate x) * up x); rows of x are tokens."""
    g = x @ Wg.T
    u = x @ Wu.T
    a = g * scipy.special.expit(g) * u
    if round_a:
        a = f64_rne_bf16_value(a)
    return a @ Wd.T


def rand_case(T, H, E, K, I, seed, norm=True):
    cfg = mi.MoEConfig("pin", T, H, E, K, I, norm, seed=seed)
    inp = mi.make_inputs(cfg, "cpu")
    return cfg, {k: mi.bits(v) for k, v in inp.items()}


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---- pins --------------------------------------------------------------------

def pin_bf16_rounding():
    # Against torch's fp32 -> bf16 conversion (round to nearest even) on values
    # that are exact in fp32 (so torch rounds once), incl. ties and subnormals.
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-39).astype(np.float32),  # subnormal range
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e38, -3.4e38, 0.0,
                  -0.0, 2 ** -133, 2 ** -134, 3 * 2 ** -135], np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16(v.astype(np.float64))
    assert np.array_equal(got, ref), np.nonzero(got != ref)
    back = oracle.bf16_to_f64(ref)
    assert np.array_equal(back.view(np.uint64), bf16_bits_to_f64(ref).view(np.uint64))


def pin_worked_example():
    g = dict(line.split(None, 1) for line in read_golden("router_top2_worked_example.txt"))
    logits = np.array([[float(v) for v in g["logits"].split()]], np.float32)
    K = int(g["K"])
    idx, w = oracle.route_from_logits(logits, K, norm=False)
    assert idx[0].tolist() == [int(v) for v in g["topk_idx"].split()]
    idx, w = oracle.route_from_logits(logits, K, norm=True)
    assert idx[0].tolist() == [int(v) for v in g["topk_idx"].split()]


def pin_topk_bruteforce():
    # Full sort with the key (logit descending, index ascending), on logits
    # quantised to create many exact ties.
    rng = np.random.default_rng(2)
    for E, K in [(8, 2), (16, 5), (128, 8), (7, 7), (1, 1)]:
        l = np.round(rng.standard_normal((50, E)) * 4).astype(np.float32) / 4
        idx, _ = oracle.route_from_logits(l, K, norm=False)
        for t in range(l.shape[0]):
            order = np.lexsort((np.arange(E), -l[t].astype(np.float64)))
            assert idx[t].tolist() == order[:K].tolist(), (E, K, t)


def pin_all_equal_logits():
    for E, K in [(8, 2), (128, 8), (5, 5)]:
        idx, w = oracle.route_from_logits(np.zeros((3, E), np.float32), K, norm=False)
        assert (idx == np.arange(K)).all()
        assert np.allclose(w, 1.0 / E, rtol=0, atol=1e-7)


def pin_weights_closed_form():
    # norm=True: softmax over the kept logits only (top-k then softmax) equals
    # softmax, top-k, renormalise.  norm=False: the full softmax (scipy).
    rng = np.random.default_rng(3)
    for E, K in [(8, 2), (128, 8), (16, 16)]:
        l = (rng.standard_normal((40, E)) * 2).astype(np.float32)
        idx, w = oracle.route_from_logits(l, K, norm=True)
        kept = np.take_along_axis(l.astype(np.float64), idx, axis=1)
        ref = scipy.special.softmax(kept, axis=1)
        assert np.abs(w - ref).max() < 1e-6
        assert np.abs(w.astype(np.float64).sum(1) - 1).max() < 1e-6
        idx2, w2 = oracle.route_from_logits(l, K, norm=False)
        assert np.array_equal(idx, idx2)
        full = scipy.special.softmax(l.astype(np.float64), axis=1)
        ref2 = np.take_along_axis(full, idx2, axis=1).astype(np.float32)
        assert np.abs(w2 - ref2).max() <= 1e-7


def pin_router_logits():
    # x·W_routerᵀ in float64 by numpy matmul, rounded to fp32.
    _, b = rand_case(9, 40, 6, 2, 16, seed=4)
    l = oracle.router_logits(b["x"], b["W_router"])
    ref = (bf16_bits_to_f64(b["x"]) @ bf16_bits_to_f64(b["W_router"]).T).astype(np.float32)
    assert np.abs(l.astype(np.float64) - ref).max() <= 1e-6 * np.abs(ref).max()


def pin_dispatch_bruteforce():
    rng = np.random.default_rng(5)
    for T, E, K in [(1, 4, 2), (37, 8, 3), (200, 16, 4), (64, 2, 2)]:
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        d = oracle.dispatch(idx, E)
        tok = np.repeat(np.arange(T), K)
        slot = np.tile(np.arange(K), T)
        key = idx.ravel().astype(np.int64) * T + tok
        order = np.argsort(key, kind="stable")
        assert np.array_equal(d["perm_tok"], tok[order])
        assert np.array_equal(d["perm_slot"], slot[order])
        assert np.array_equal(d["counts"], np.bincount(idx.ravel(), minlength=E))
        assert d["offsets"][0] == 0 and d["offsets"][-1] == T * K
        assert np.array_equal(np.diff(d["offsets"]), d["counts"])
        inv = d["inv"].ravel()
        assert np.array_equal(inv[order], np.arange(T * K))  # inv ∘ perm = id


def pin_single_expert_is_swiglu():
    # E = K = 1: the block is one SwiGLU MLP with weight 1.
    for norm in (False, True):
        _, b = rand_case(11, 64, 1, 1, 48, seed=6, norm=norm)
        r = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 1, norm)
        assert (r["idx"] == 0).all() and (r["w"] == 1.0).all()
        x = bf16_bits_to_f64(b["x"])
        y = np_swiglu(x, bf16_bits_to_f64(b["W_gate"][0]), bf16_bits_to_f64(b["W_up"][0]),
                      bf16_bits_to_f64(b["W_down"][0]))
        assert np.abs(r["out_f64"] - y).max() <= 1e-6 * np.abs(y).max()
        ref = f64_rne_bf16_value(y)
        got = bf16_bits_to_f64(r["out"])
        ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
        assert (np.abs(got - ref) <= ulp).all()
        assert np.mean(got == ref) > 0.99
        # the delivered bf16 output is the round-to-nearest-even of the unrounded sum
        assert np.array_equal(got, f64_rne_bf16_value(r["out_f64"]))


def _dense_reference(b, idx, w, E, round_a=True):
    x = bf16_bits_to_f64(b["x"])
    T = x.shape[0]
    G = np.zeros((T, E))
    for t in range(T):
        for k in range(idx.shape[1]):
            G[t, idx[t, k]] += float(w[t, k])
    acc = np.zeros_like(x)
    for e in range(E):
        y = np_swiglu(x, bf16_bits_to_f64(b["W_gate"][e]), bf16_bits_to_f64(b["W_up"][e]),
                      bf16_bits_to_f64(b["W_down"][e]), round_a)
        acc += G[:, [e]] * y
    return acc


def pin_dense_equivalence():
    # out[t] = Σ_e G[t,e]·MLP_e(x_t) with the dense routing matrix G
    # (k non-zeros per row): every expert on every token, no dispatch.
    for (T, H, E, K, I, norm) in [(13, 32, 6, 3, 24, True), (20, 64, 8, 2, 32, False)]:
        _, b = rand_case(T, H, E, K, I, seed=7 + T, norm=norm)
        r = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], K,
                               norm, flags=oracle.FP64_INTERMEDIATE)
        ref = _dense_reference(b, r["idx"], r["w"], E, round_a=False)
        assert np.abs(r["out_f64"] - ref).max() <= 1e-12 * np.abs(ref).max()
        got = bf16_bits_to_f64(r["out"])
        assert (np.abs(got - f64_rne_bf16_value(ref)) <= np.abs(ref) * 2.0 ** -7 + 1e-30).all()
        # with the default bf16 rounding of the SwiGLU intermediate
        r2 = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], K,
                                norm)
        ref2 = _dense_reference(b, r2["idx"], r2["w"], E, round_a=True)
        assert np.abs(r2["out_f64"] - ref2).max() <= 1e-6 * np.abs(ref2).max()


def pin_soft_router():
    # K = E with norm: the soft (dense) mixture Σ_e softmax(l)_e·MLP_e(x).
    _, b = rand_case(10, 32, 4, 4, 16, seed=8)
    r = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 4, True,
                           flags=oracle.FP64_INTERMEDIATE)
    x = bf16_bits_to_f64(b["x"])
    l = (x @ bf16_bits_to_f64(b["W_router"]).T).astype(np.float32).astype(np.float64)
    p = scipy.special.softmax(l, axis=1)
    acc = np.zeros_like(x)
    for e in range(4):
        acc += p[:, [e]] * np_swiglu(x, bf16_bits_to_f64(b["W_gate"][e]),
                                     bf16_bits_to_f64(b["W_up"][e]),
                                     bf16_bits_to_f64(b["W_down"][e]), round_a=False)
    assert np.abs(r["out_f64"] - acc).max() <= 1e-6 * np.abs(acc).max()
    got = bf16_bits_to_f64(r["out"])
    ref = f64_rne_bf16_value(acc)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -6 + 1e-30).all()


def pin_token_permutation_equivariance():
    _, b = rand_case(24, 32, 8, 2, 16, seed=9)
    r = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 2, True)
    perm = np.random.default_rng(9).permutation(24)
    r2 = oracle.moe_forward(b["x"][perm], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 2,
                            True)
    assert np.array_equal(r2["out"], r["out"][perm])
    assert np.array_equal(r2["idx"], r["idx"][perm])
    assert np.array_equal(r2["counts"], r["counts"])
    assert abs(r2["aux"] - r["aux"]) < 1e-6


def pin_aux():
    L = np.log(3.0)
    for line in read_golden("aux_hand_examples.txt"):
        head, vals, want = [s.strip() for s in line.split("|")]
        _, E, K, T = head.split()
        E, K, T = int(E), int(K), int(T)
        l = np.array([L if v == "L" else float(v) for v in vals.split()], np.float32).reshape(T, E)
        idx, _ = oracle.route_from_logits(l, K, norm=True)
        counts = np.bincount(idx.ravel(), minlength=E).astype(np.int32)
        a = oracle.aux(oracle.softmax(l), counts, K)
        assert abs(a - float(want)) < 1e-6, (line, a)
    # W_router = 0: uniform probabilities -> aux = 1 whatever the assignment.
    _, b = rand_case(33, 32, 8, 3, 16, seed=10)
    r = oracle.moe_forward(b["x"], np.zeros_like(b["W_router"]), b["W_gate"], b["W_up"],
                           b["W_down"], 3, True, want_out=False)
    assert abs(r["aux"] - 1.0) < 1e-6
    # Balanced assignment (each expert gets T·K/E pairs) -> aux = 1 whatever p is.
    rng = np.random.default_rng(11)
    E, K, T = 8, 2, 16
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)], np.int32)
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int32)
    assert (counts == T * K // E).all()
    p = scipy.special.softmax(rng.standard_normal((T, E)), axis=1)
    assert abs(oracle.aux(p, counts, K) - 1.0) < 1e-12
    # Bounds 0 <= aux <= E on random cases.
    for s in range(3):
        _, b = rand_case(40, 32, 8, 2, 16, seed=20 + s)
        r = oracle.moe_forward(b["x"], b["W_router"] * 1, b["W_gate"], b["W_up"], b["W_down"], 2,
                               True, want_out=False)
        assert 0.0 <= r["aux"] <= 8.0


def pin_param_counts():
    g = dict(line.split() for line in read_golden("qwen3_param_counts.txt"))
    H, E, K, I = (int(g[k]) for k in "HEKI")
    cfg = mi.MoEConfig("q", 1, H, E, K, I, True)
    # layouts: W_router [E,H], W_gate/W_up [E,I,H], W_down [E,H,I]
    assert E * H == int(g["router"])
    assert I * H == int(g["gate_proj"]) == int(g["up_proj"]) == int(g["down_proj"])
    assert (cfg.E, cfg.I, cfg.H) == (E, I, H)


# ---- selection-only expert bias (auxiliary-loss-free balancing) --------------

def pin_bias_zero_is_unbiased():
    # a zero bias leaves every selection and weight unchanged
    rng = np.random.default_rng(21)
    l = (rng.standard_normal((50, 16)) * 2).astype(np.float32)
    for norm in (False, True):
        i0, w0 = oracle.route_from_logits(l, 4, norm)
        i1, w1 = oracle.route_from_logits(l, 4, norm, bias=np.zeros(16, np.float32))
        assert np.array_equal(i0, i1) and np.array_equal(w0, w1)


def pin_biased_topk_bruteforce():
    # ranking by the fp32 key logit + bias, ties to the lower index: a full
    # stable sort of the keys (multiples of 1/4, so the sums are exact and tie)
    rng = np.random.default_rng(22)
    T, E, K = 60, 12, 5
    l = (rng.integers(-8, 9, (T, E)) / 4).astype(np.float32)
    b = (rng.integers(-4, 5, E) / 4).astype(np.float32)
    idx, _ = oracle.route_from_logits(l, K, True, bias=b)
    key = (l + b[None, :]).astype(np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(key[t, e]), e))
        assert list(idx[t]) == order[:K], t


def pin_biased_weights_are_unbiased_probs():
    # the bias moves the selection only: weights are the softmax of the
    # unbiased logits at the selected experts (renormalised over them if norm)
    rng = np.random.default_rng(23)
    T, E, K = 40, 16, 4
    l = (rng.standard_normal((T, E)) * 1.5).astype(np.float32)
    b = (rng.standard_normal(E) * 3).astype(np.float32)
    p = scipy.special.softmax(l.astype(np.float64), axis=1)
    for norm in (False, True):
        idx, w = oracle.route_from_logits(l, K, norm, bias=b)
        want = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        if norm:
            want = want / want.sum(axis=1, keepdims=True)
        assert np.abs(w - want).max() <= 1e-7 * max(1.0, np.abs(want).max())


def pin_bias_forces_selection_and_aux():
    # a large bias on two experts makes every token pick them (in key order);
    # aux then counts only those two, with P from the unbiased softmax
    cfg, b = rand_case(40, 64, 8, 2, 64, seed=24, norm=False)
    bias = np.zeros(8, np.float32)
    bias[5], bias[2] = 1000.0, 999.0
    r = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 2, False,
                           bias=bias)
    assert (r["idx"] == np.array([5, 2])).all()
    p = scipy.special.softmax(r["logits"].astype(np.float64), axis=1)
    want = 8 * (0.5 * p[:, 5].mean() + 0.5 * p[:, 2].mean())
    assert abs(r["aux"] - want) <= 1e-6 * max(1.0, want)
    assert np.allclose(r["w"][:, 0], p[:, 5], rtol=1e-6) and np.allclose(r["w"][:, 1], p[:, 2],
                                                                           rtol=1e-6)


# ---- expert capacity (first C pairs of each expert in token order) -----------

def _kept_by_hand(idx, E, C):
    """Brute force: walk the tokens in order, count per expert, keep the first C."""
    seen = [0] * E
    keep = np.zeros(idx.shape, bool)
    for t in range(idx.shape[0]):
        for k in range(idx.shape[1]):
            e = int(idx[t, k])
            keep[t, k] = seen[e] < C
            seen[e] += 1
    return keep


def pin_capacity_bruteforce():
    # out[t] = Σ over the token's kept pairs of w·SwiGLU, in float64 numpy
    cfg, b = rand_case(24, 64, 4, 2, 64, seed=31, norm=True)
    C = 5
    r = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 2, True,
                           capacity=C)
    keep = _kept_by_hand(r["idx"], 4, C)
    assert keep.sum() < keep.size  # some pairs are dropped at this capacity
    x = bf16_bits_to_f64(b["x"])
    Wg, Wu, Wd = (bf16_bits_to_f64(b[k]) for k in ("W_gate", "W_up", "W_down"))
    for t in range(24):
        want = np.zeros(64)
        for k in range(2):
            if keep[t, k]:
                e = int(r["idx"][t, k])
                want += float(r["w"][t, k]) * np_swiglu(x[t:t + 1], Wg[e], Wu[e], Wd[e])[0]
        assert np.abs(r["out_f64"][t] - want).max() <= 1e-9 * (1 + np.abs(want).max()), t
    # aux is the router's statistic: unchanged by the capacity
    r0 = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 2, True)
    assert r["aux"] == r0["aux"] and np.array_equal(r["counts"], r0["counts"])


def pin_capacity_dispatch():
    # kept rows: the first C tokens of each expert, in order; inv = -1 elsewhere
    rng = np.random.default_rng(32)
    T, E, K, C = 50, 6, 3, 7
    idx = np.array([rng.permutation(E)[:K] for _ in range(T)], np.int32)
    d = oracle.dispatch(idx, E, capacity=C)
    keep = _kept_by_hand(idx, E, C)
    assert np.array_equal(d["counts"], np.bincount(idx.ravel(), minlength=E))
    kept_counts = np.minimum(d["counts"], C)
    assert np.array_equal(d["offsets"], np.concatenate([[0], np.cumsum(kept_counts)]))
    for t in range(T):
        for k in range(K):
            r = d["inv"][t, k]
            if keep[t, k]:
                assert 0 <= r < d["perm_tok"].size
                assert d["perm_tok"][r] == t and d["perm_slot"][r] == k
            else:
                assert r == -1
    for e in range(E):
        rows = d["perm_tok"][d["offsets"][e]:d["offsets"][e + 1]]
        assert list(rows) == sorted(np.where((idx == e).any(axis=1))[0].tolist())[:C]
    big = oracle.dispatch(idx, E, capacity=T)  # no expert reaches T pairs: nothing dropped
    plain = oracle.dispatch(idx, E)
    for key in plain:
        assert np.array_equal(big[key], plain[key])


# ---- 4-bit group quantisation (csdn page, section "参数量化与存储优化") --------

def _bf16_of(v):
    """bf16 bits of values that are exactly representable (checked)."""
    v = np.asarray(v, np.float32)
    bits = (v.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), v)
    return bits


def pin_q4_exact_grid():
    # Groups whose entries lie on lo + k·s with s a power of two: the codes are k,
    # scale and bias are s and lo, and dequantisation gives the weights back.
    # Every group (128 entries of a row) has its own lo and s, so groups taken
    # along the wrong axis or indexed wrongly change the codes.
    rng = np.random.default_rng(40)
    rows, cols = 3, 384
    k = rng.integers(0, 16, size=(rows, cols))
    lo = np.empty((rows, cols // 128))
    st = np.empty_like(lo)
    vals = np.empty((rows, cols))
    for r in range(rows):
        for g in range(cols // 128):
            kk = k[r, g * 128:(g + 1) * 128]
            kk[0], kk[1] = 0, 15  # the group's min and max are on the grid's ends
            lo[r, g] = -0.25 * (1 + r + 2 * g)
            st[r, g] = 2.0 ** -(3 + (r + g) % 3)
            vals[r, g * 128:(g + 1) * 128] = lo[r, g] + kk * st[r, g]
    W = _bf16_of(vals)
    q, s, b = oracle.quantize_q4(W)
    assert np.array_equal(q, k)
    assert np.array_equal(s, _bf16_of(st)) and np.array_equal(b, _bf16_of(lo))
    assert np.array_equal(oracle.dequantize_q4(q, s, b), W)


def pin_q4_round_half_even_and_constant_group():
    # lo = 0, hi = 15 -> s = 1: entries at k + 0.5 get the even neighbour
    g = np.zeros(128, np.float32)
    g[1] = 15.0
    g[2:8] = [0.5, 1.5, 2.5, 3.5, 13.5, 14.5]
    # a second group that is constant: scale 0, every code 0, weights unchanged
    W = _bf16_of(np.concatenate([g, np.full(128, -0.375, np.float32)])[None, :])
    q, s, b = oracle.quantize_q4(W)
    assert q[0, 2:8].tolist() == [0, 2, 2, 4, 14, 14]
    assert q[0, 1] == 15 and q[0, 0] == 0
    assert oracle.bf16_to_f64(s)[0].tolist() == [1.0, 0.0]
    assert (q[0, 128:] == 0).all()
    assert np.array_equal(oracle.dequantize_q4(q, s, b)[0, 128:], W[0, 128:])


def pin_q4_error_bound():
    # random weights: codes span 0..15 with the min at 0 and the max at 15, and
    # |w' - w| <= s/2 + half a bf16 ulp of w' (rounding to the grid, then to bf16)
    rng = np.random.default_rng(41)
    W = _bf16_of((rng.standard_normal((16, 512)) * 0.02).astype(np.float32).view(np.uint32)
                 .__and__(np.uint32(0xFFFF0000)).view(np.float32))
    q, s, b = oracle.quantize_q4(W)
    w = oracle.bf16_to_f64(W)
    wd = oracle.bf16_to_f64(oracle.dequantize_q4(q, s, b))
    sv = np.repeat(oracle.bf16_to_f64(s), 128, axis=1)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(wd) + 1e-300)) - 7)
    assert (np.abs(wd - w) <= sv / 2 + ulp / 2 + 1e-12).all()
    for r in range(16):
        for gi in range(4):
            grp = w[r, gi * 128:(gi + 1) * 128]
            qq = q[r, gi * 128:(gi + 1) * 128]
            assert qq[np.argmin(grp)] == 0 and qq[np.argmax(grp)] == 15


def pin_q4_exact_weights():
    # The exact values q·s + b: on a grid they are the original weights; for
    # random weights they lie within s/2 of them (no bf16 term), and the
    # dequantised weights are their nearest bf16.
    rng = np.random.default_rng(42)
    rows, cols = 4, 256
    k = rng.integers(0, 16, size=(rows, cols))
    vals = np.empty((rows, cols))
    for r in range(rows):
        for g in range(cols // 128):
            kk = k[r, g * 128:(g + 1) * 128]
            kk[0], kk[1] = 0, 15
            vals[r, g * 128:(g + 1) * 128] = -0.5 * (1 + r + g) + kk * 2.0 ** -(2 + (r + 2 * g) % 4)
    W = _bf16_of(vals)
    q, s, b = oracle.quantize_q4(W)
    assert np.array_equal(oracle.dequantize_q4_f64(q, s, b), bf16_bits_to_f64(W))
    W = _bf16_of((rng.standard_normal((8, 384)) * 0.02).astype(np.float32).view(np.uint32)
                 .__and__(np.uint32(0xFFFF0000)).view(np.float32))
    q, s, b = oracle.quantize_q4(W)
    we = oracle.dequantize_q4_f64(q, s, b)
    sv = np.repeat(bf16_bits_to_f64(s), 128, axis=1)
    bv = np.repeat(bf16_bits_to_f64(b), 128, axis=1)
    assert np.array_equal(we, q.astype(np.float64) * sv + bv)
    assert (np.abs(we - bf16_bits_to_f64(W)) <= sv / 2 + 1e-12).all()
    assert np.array_equal(bf16_bits_to_f64(oracle.dequantize_q4(q, s, b)), f64_rne_bf16_value(we))


def pin_q4_forward_single_expert_is_swiglu():
    # E = K = 1 on 4-bit weights: one SwiGLU MLP (numpy float64) with the weights
    # bf16(q·s + b), every 128-column group with its own scale and bias.
    _, b = rand_case(9, 256, 1, 1, 256, seed=43, norm=True)
    q4 = oracle.quantize_experts_q4(b["W_gate"], b["W_up"], b["W_down"])
    r = oracle.moe_forward_q4(b["x"], b["W_router"], q4, 1, True)
    Wg, Wu, Wd = (f64_rne_bf16_value(
        q4[n][0].astype(np.float64) * np.repeat(bf16_bits_to_f64(q4[n][1]), 128, -1)
        + np.repeat(bf16_bits_to_f64(q4[n][2]), 128, -1)) for n in ("gate", "up", "down"))
    y = np_swiglu(bf16_bits_to_f64(b["x"]), Wg[0], Wu[0], Wd[0])
    assert np.abs(r["out_f64"] - y).max() <= 1e-9 * np.abs(y).max()
    # and not the bf16 forward on the original weights (the quantisation shows)
    r0 = oracle.moe_forward(b["x"], b["W_router"], b["W_gate"], b["W_up"], b["W_down"], 1, True)
    assert np.abs(r0["out_f64"] - y).max() > 1e-3 * np.abs(y).max()


def pin_q4_forward_on_grid_is_the_bf16_forward():
    # Weights already on each group's 4-bit grid (so q·s + b is the bf16 weight
    # itself): the 4-bit forward is the bf16 forward, to the last bit, routing,
    # selection, combine and all.
    rng = np.random.default_rng(44)
    T, H, E, K, I = 6, 256, 4, 2, 128
    _, b = rand_case(T, H, E, K, I, seed=45, norm=True)

    def on_grid(shape):
        # each group: lo + k·st with its minimum at k = 0 and its maximum at
        # k = 15 (so the quantiser finds lo and st again); all values bf16
        k = rng.integers(0, 16, size=shape)
        k[..., 0::128] = 0
        k[..., 1::128] = 15
        lo = -2.0 ** -5 * (1 + rng.integers(0, 4, size=shape[:-1] + (shape[-1] // 128,)))
        st = 2.0 ** -rng.integers(7, 10, size=lo.shape).astype(np.float64)
        return _bf16_of(np.repeat(lo, 128, -1) + k * np.repeat(st, 128, -1))

    Wg, Wu, Wd = on_grid((E, I, H)), on_grid((E, I, H)), on_grid((E, H, I))
    q4 = oracle.quantize_experts_q4(Wg, Wu, Wd)
    r4 = oracle.moe_forward_q4(b["x"], b["W_router"], q4, K, True)
    r = oracle.moe_forward(b["x"], b["W_router"], Wg, Wu, Wd, K, True)
    assert np.array_equal(r4["out_f64"], r["out_f64"]) and np.array_equal(r4["out"], r["out"])
    assert np.array_equal(r4["idx"], r["idx"]) and r4["aux"] == r["aux"]


PINS = [pin_bf16_rounding, pin_worked_example, pin_topk_bruteforce, pin_all_equal_logits,
        pin_weights_closed_form, pin_router_logits, pin_dispatch_bruteforce,
        pin_single_expert_is_swiglu, pin_dense_equivalence, pin_soft_router,
        pin_token_permutation_equivariance, pin_aux, pin_param_counts,
        pin_bias_zero_is_unbiased, pin_biased_topk_bruteforce,
        pin_biased_weights_are_unbiased_probs, pin_bias_forces_selection_and_aux,
        pin_capacity_bruteforce, pin_capacity_dispatch, pin_q4_exact_grid,
        pin_q4_round_half_even_and_constant_group, pin_q4_error_bound, pin_q4_exact_weights,
        pin_q4_forward_single_expert_is_swiglu, pin_q4_forward_on_grid_is_the_bf16_forward]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_zero_tokens():
    z = np.zeros((0, 16), np.uint16)
    Wr = np.zeros((4, 16), np.uint16)
    W = np.zeros((4, 8, 16), np.uint16)
    Wd = np.zeros((4, 16, 8), np.uint16)
    r = oracle.moe_forward(z, Wr, W, W, Wd, 2, True)
    assert r["out"].shape == (0, 16) and r["aux"] == 0.0 and (r["counts"] == 0).all()


def test_near_tie_detector():
    p = np.array([[0.5, 0.3, 0.3 - 5e-7, 0.1 + 5e-7 - 0.0], [0.4, 0.3, 0.2, 0.1]])
    assert oracle.near_tie_tokens(p, 2).tolist() == [0]
    assert oracle.near_tie_tokens(p, 1).tolist() == []


# ---- planted mistakes: each must break at least one pin -----------------------

MUTATIONS = {
    "silu_sign": ("g / (1.0 + exp(-g))", "g / (1.0 + exp(g))"),
    "norm_dropped": ("if (norm) w = w / sum;", "if (0) w = w / sum;"),
    "tie_break_reversed": ("    return a < b;", "    return a > b;"),
    "gate_up_swapped": ("g += xv * oracle_bf16_to_f64(Wg[", "g += xv * oracle_bf16_to_f64(Wu["),
    "router_transposed": ("oracle_bf16_to_f64(Wr[(size_t)e * H + h])",
                          "oracle_bf16_to_f64(Wr[(size_t)h * E + e])"),
    "softmax_no_shift": ("probs[(size_t)t * E + e] = exp((double)l[e] - m) / z;",
                         "probs[(size_t)t * E + e] = exp((double)l[e]) / z;"),
    "combine_unweighted": ("acc[h] += (double)w_row[k] * y[h];", "acc[h] += y[h];"),
    "aux_per_token_share": ("((double)T * (double)K)", "((double)T)"),
    "dispatch_token_major": ("for (int e = 0; e < E; ++e)\n        for (int t = 0; t < T; ++t)",
                             "for (int t = 0; t < T; ++t)\n        for (int e = 0; e < E; ++e)"),
    "bf16_truncates": ("r = ldexp(nearbyint(q), ulp_exp);", "r = ldexp(floor(q), ulp_exp);"),
    "down_uses_unrounded_gate": ("double ai = silu(g) * u;", "double ai = silu(u) * u;"),
    "topk_by_smallest": ("    if (l[a] > l[b]) return 1;\n    if (l[a] < l[b]) return 0;",
                         "    if (l[a] < l[b]) return 1;\n    if (l[a] > l[b]) return 0;"),
    "bias_ignored": ("keys[i] = bias ? (float)(logits[i] + bias[i % (size_t)E]) : logits[i];",
                     "keys[i] = logits[i];"),
    "capacity_off_by_one": ("(uint8_t)(capacity <= 0 || seen[e] < capacity)",
                            "(uint8_t)(capacity <= 0 || seen[e] <= capacity)"),
    "dropped_pairs_contribute": ("                if (keep[(size_t)t * K + k]) {\n                    ik[nk]",
                                 "                if (1) {\n                    ik[nk]"),
    "q4_bias_dropped": ("(double)code * oracle_bf16_to_f64(s[gi]) + oracle_bf16_to_f64(b[gi]);",
                        "(double)code * oracle_bf16_to_f64(s[gi]);"),
    "q4_sixteen_levels": ("(double)(span / 15.0f)", "(double)(span / 16.0f)"),
    "q4_codes_truncate": ("rintf((q4_f32(w[j]) - bf) / sf)", "truncf((q4_f32(w[j]) - bf) / sf)"),
    "q4_wrong_group": ("const long long gi = r * groups + c / 128;",
                       "const long long gi = r * groups + c % groups;"),
    "q4_forward_bias_dropped": ("const double v = (double)q[row * (size_t)cols + c] * oracle_bf16_to_f64(s[g]) +\n                         oracle_bf16_to_f64(b[g]);",
                                "const double v = (double)q[row * (size_t)cols + c] * oracle_bf16_to_f64(s[g]);"),
    "q4_forward_wrong_group": ("const size_t g = row * (size_t)groups + (size_t)(c / 128);",
                               "const size_t g = row * (size_t)groups + (size_t)(c % groups);"),
    "q4_forward_gate_up_swapped": ("q4_row(W->qg, W->sg, W->bg, row, H, wg);",
                                   "q4_row(W->qu, W->su, W->bu, row, H, wg);"),
    "q4_forward_unrounded_weights": ("out[c] = oracle_bf16_to_f64(oracle_f64_to_bf16(v));",
                                     "out[c] = v;"),
    "weights_from_biased_keys": (
        "logits[i];\n    oracle_softmax(logits, T, E, probs);",
        "logits[i];\n    oracle_softmax(keys, T, E, probs);"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    mut = src.replace(old, new)
    c = os.path.join(mutant_dir, f"{name}.c")
    so = os.path.join(mutant_dir, f"{name}.so")
    open(c, "w").write(mut)
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
                           "-o", so, c, "-lm"])
    failed = []
    with oracle.use_library(so):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
