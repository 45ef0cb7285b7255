"""ctypes wrapper around the C oracle (moe_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  Inputs are numpy arrays; bf16 tensors
travel as their uint16 bit patterns.

Each function follows one step of the block forward printed on the cnblogs page
"大模型-qwen3 MoE 详细解读" (Qwen3MoeSparseMoeBlock.forward); the docstrings in
moe_oracle.c give the exact definitions and the readings taken.
"""
import ctypes
import os

import numpy as np

from .build import build

BF16_LOGITS = 1
FP64_INTERMEDIATE = 2

class _Lib:
    """The loaded C oracle (a copy built from another source can be loaded too,
    which the tests use to show that each pin catches a planted mistake)."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_router_logits.argtypes = [P, i, i, P, i, i, P]
        lib.oracle_softmax.argtypes = [P, i, i, P]
        lib.oracle_route_from_logits.argtypes = [P, i, i, i, i, P, P]
        lib.oracle_route_biased.argtypes = [P, P, i, i, i, i, P, P]
        lib.oracle_dispatch.argtypes = [P, i, i, i, P, P, P, P, P]
        lib.oracle_dispatch_cap.argtypes = [P, i, i, i, i, P, P, P, P, P]
        lib.oracle_keep_mask.argtypes = [P, i, i, i, i, P]
        lib.oracle_quantize_q4.argtypes = [P, i, i, P, P, P]
        lib.oracle_dequantize_q4.argtypes = [P, P, P, i, i, P]
        lib.oracle_dequantize_q4_f64.argtypes = [P, P, P, i, i, P]
        lib.oracle_moe_forward_q4.argtypes = [P, i, i, P, P, i, P, P, P, P, P, P, P, P, P, i, i,
                                              i, i, i, P, i, P, P, P, P, P, P, P]
        lib.oracle_token_output_q4.argtypes = [P, i, P, P, i, P, P, P, P, P, P, P, P, P, i, i, i,
                                               P, P]
        lib.oracle_expert_mlp.argtypes = [P, i, P, P, P, i, i, P]
        lib.oracle_token_output.argtypes = [P, i, P, P, i, P, P, P, i, i, i, P]
        lib.oracle_token_output_ex.argtypes = [P, i, P, P, i, P, P, P, i, i, i, P, P]
        lib.oracle_aux.argtypes = [P, P, i, i, i]
        lib.oracle_aux.restype = ctypes.c_double
        lib.oracle_moe_forward.argtypes = [P, i, i, P, P, P, P, i, i, i, i, i, P, i, P, P, P,
                                           P, P, P, P]
        lib.oracle_moe_forward_b.argtypes = [P, i, i, P, P, i, P, P, P, i, i, i, i, i, P, i, P,
                                             P, P, P, P, P, P]
        self.c = lib


_default = None
_current = None


def _L():
    global _default
    if _current is not None:
        return _current.c
    if _default is None:
        _default = _Lib(build())
    return _default.c


class use_library:
    """Context manager: route every call in this module to another build of
    the oracle (a shared object at `path`)."""

    def __init__(self, path):
        self.lib = _Lib(path)

    def __enter__(self):
        global _current
        self.prev = _current
        _current = self.lib
        return self

    def __exit__(self, *exc):
        global _current
        _current = self.prev
        return False


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def threads():
    """Threads the oracle's OpenMP loops may use (OMP_NUM_THREADS, else affinity)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env:
        return int(env)
    return len(os.sched_getaffinity(0))


def bf16_to_f64(bits):
    """Exact value of each bf16 bit pattern (uint16 array) as float64."""
    L = _L()
    b = _c(bits, np.uint16)
    return np.array([L.oracle_bf16_to_f64(int(v)) for v in b.ravel()]).reshape(b.shape)


def f64_to_bf16(vals):
    """Round float64 values to bf16 bit patterns (nearest, ties to even)."""
    L = _L()
    v = _c(vals, np.float64)
    return np.array([L.oracle_f64_to_bf16(float(z)) for z in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


def router_logits(x, Wr, flags=0):
    """logits[t,e] = x[t]·W_router[e] in double, rounded to fp32 -> float32 [T,E]."""
    x = _c(x, np.uint16)
    Wr = _c(Wr, np.uint16)
    T, H = x.shape
    E = Wr.shape[0]
    out = np.empty((T, E), np.float32)
    _check(_L().oracle_router_logits(_p(x), T, H, _p(Wr), E, flags, _p(out)), "router")
    return out


def softmax(logits):
    """Full softmax over experts in double -> float64 [T,E]."""
    l = _c(logits, np.float32)
    T, E = l.shape
    out = np.empty((T, E), np.float64)
    _check(_L().oracle_softmax(_p(l), T, E, _p(out)), "softmax")
    return out


def route_from_logits(logits, K, norm, bias=None):
    """Top-k (logit desc, index asc) and weights -> (idx int32 [T,K], w float32 [T,K]).
    With bias (float32 [E]): ranked by the fp32 key logit + bias, weighted by the
    unbiased probabilities."""
    l = _c(logits, np.float32)
    T, E = l.shape
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    if bias is None:
        _check(_L().oracle_route_from_logits(_p(l), T, E, K, int(bool(norm)), _p(idx), _p(w)),
               "route")
    else:
        b = _c(bias, np.float32)
        assert b.shape == (E,)
        _check(_L().oracle_route_biased(_p(l), _p(b), T, E, K, int(bool(norm)), _p(idx), _p(w)),
               "route")
    return idx, w


def dispatch(idx, E, capacity=0):
    """Group pairs by (expert, token) -> dict(counts, offsets, perm_tok, perm_slot, inv).
    With capacity > 0 each expert keeps its first `capacity` pairs in token order:
    rows hold the kept pairs, offsets count them, inv = -1 for the dropped ones and
    counts stay the routed pairs; perm_tok / perm_slot have offsets[E] entries."""
    idx = _c(idx, np.int32)
    T, K = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm_tok = np.empty(T * K, np.int32)
    perm_slot = np.empty(T * K, np.int32)
    inv = np.empty(T * K, np.int32)
    _check(_L().oracle_dispatch_cap(_p(idx), T, E, K, int(capacity), _p(counts), _p(offsets),
                                    _p(perm_tok), _p(perm_slot), _p(inv)), "dispatch")
    n = int(offsets[E])
    return dict(counts=counts, offsets=offsets, perm_tok=perm_tok[:n], perm_slot=perm_slot[:n],
                inv=inv.reshape(T, K))


def keep_mask(idx, E, capacity):
    """bool [T,K]: the pairs each expert keeps under the capacity (first in token order)."""
    idx = _c(idx, np.int32)
    T, K = idx.shape
    keep = np.empty((T, K), np.uint8)
    _check(_L().oracle_keep_mask(_p(idx), T, E, K, int(capacity), _p(keep)), "keep_mask")
    return keep.astype(bool)


def expert_mlp(x_row, Wg_e, Wu_e, Wd_e, flags=0):
    """One expert's SwiGLU MLP on one token -> float64 [H]."""
    x_row = _c(x_row, np.uint16)
    Wg_e, Wu_e, Wd_e = (_c(a, np.uint16) for a in (Wg_e, Wu_e, Wd_e))
    I, H = Wg_e.shape
    y = np.empty(H, np.float64)
    _check(_L().oracle_expert_mlp(_p(x_row), H, _p(Wg_e), _p(Wu_e), _p(Wd_e), I, flags, _p(y)),
           "expert_mlp")
    return y


def token_output(x_row, idx_row, w_row, Wg, Wu, Wd, flags=0, unrounded=False):
    """bf16(Σ_k w_k·MLP_{idx_k}(x_row)) -> uint16 [H] for an explicit selection;
    with unrounded=True also the float64 sum before rounding: (bits, f64)."""
    x_row = _c(x_row, np.uint16)
    idx_row = _c(idx_row, np.int32)
    w_row = _c(w_row, np.float32)
    Wg, Wu, Wd = (_c(a, np.uint16) for a in (Wg, Wu, Wd))
    E, I, H = Wg.shape
    out = np.empty(H, np.uint16)
    f64 = np.empty(H, np.float64) if unrounded else None
    _check(_L().oracle_token_output_ex(_p(x_row), H, _p(idx_row), _p(w_row), idx_row.shape[0],
                                       _p(Wg), _p(Wu), _p(Wd), E, I, flags, _p(out), _p(f64)),
           "token_output")
    return (out, f64) if unrounded else out


def aux(probs, counts, K):
    """E·Σ_e (counts_e/(T·K))·mean_t p[t,e] (float64)."""
    p = _c(probs, np.float64)
    c = _c(counts, np.int32)
    T, E = p.shape
    return float(_L().oracle_aux(_p(p), _p(c), T, E, K))


def moe_forward(x, Wr, Wg, Wu, Wd, K, norm, rows=None, flags=0, want_out=True, bias=None,
                capacity=0):
    """The whole block (with bias: the selection-only expert bias of
    route_from_logits; with capacity > 0: each expert keeps its first `capacity`
    pairs in token order and the dropped pairs add nothing to out).  Returns
    dict(out, out_f64, logits, idx, w, aux, counts); counts are the routed pairs.

    out is bf16 bits [n_rows, H] for the listed token rows (all tokens when
    rows is None) and out_f64 the same values before the final bf16 rounding;
    routing, dispatch counts and aux always cover every token.
    """
    x = _c(x, np.uint16)
    Wr, Wg, Wu, Wd = (_c(a, np.uint16) for a in (Wr, Wg, Wu, Wd))
    T, H = x.shape
    E, I, _ = Wg.shape
    assert Wr.shape == (E, H) and Wu.shape == (E, I, H) and Wd.shape == (E, H, I)
    if rows is not None:
        rows = _c(rows, np.int32)
        n = rows.shape[0]
    else:
        n = T
    out = np.empty((n, H), np.uint16) if want_out else None
    out_f64 = np.empty((n, H), np.float64) if want_out else None
    logits = np.empty((T, E), np.float32)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    counts = np.empty(E, np.int32)
    a = np.zeros(1, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    _check(_L().oracle_moe_forward_b(_p(x), T, H, _p(Wr), _p(b), int(capacity), _p(Wg), _p(Wu),
                                     _p(Wd), E, K, I, int(bool(norm)), flags, _p(rows), n,
                                     _p(out),
                                     _p(out_f64), _p(logits), _p(idx), _p(w), _p(a),
                                     _p(counts)), "forward")
    return dict(out=out, out_f64=out_f64, logits=logits, idx=idx, w=w, aux=float(a[0]),
                counts=counts)


def near_tie_tokens(probs, K, gap=1e-6):
    """Tokens whose K-th and (K+1)-th largest probabilities differ by < gap,
    or whose kept experts have adjacent probabilities closer than gap (an
    in-top-K order swap).  Either makes more than one selection correct."""
    p = np.asarray(probs, np.float64)
    T, E = p.shape
    if K >= E:
        s = -np.sort(-p, axis=1)
        d = s[:, :-1] - s[:, 1:]
        return np.where((d < gap).any(axis=1))[0] if E > 1 else np.array([], np.int64)
    s = -np.sort(-p, axis=1)[:, :K + 1]
    d = s[:, :-1] - s[:, 1:]
    return np.where((d < gap).any(axis=1))[0]


def capacity_of(cf, T, K, E):
    """Pairs each expert keeps for capacity factor cf: ceil(cf·T·K/E), at least 1
    (0: no limit).  cf is taken as the fp32 value a caller passes."""
    cf = float(np.float32(cf))
    if cf <= 0:
        return 0
    import math
    return max(1, int(math.ceil(cf * T * K / E)))



def quantize_q4(W):
    """4-bit group quantisation of weight rows (csdn page, section
    "参数量化与存储优化"; the reading is in moe_oracle.c): W [..., cols] bf16 bits
    (cols % 128 == 0) -> (q uint8 codes [..., cols], s, b bf16 bits [..., cols/128])."""
    W = _c(W, np.uint16)
    cols = W.shape[-1]
    rows = W.size // cols
    q = np.empty(W.shape, dtype=np.uint8)
    s = np.empty(W.shape[:-1] + (cols // 128,), dtype=np.uint16)
    b = np.empty_like(s)
    _check(_L().oracle_quantize_q4(_p(W), rows, cols, _p(q), _p(s), _p(b)), "quantize_q4")
    return q, s, b


def dequantize_q4(q, s, b):
    """W' = bf16(q·s + b) per element, rounded once (bf16 bits, the shape of q)."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    b = _c(b, np.uint16)
    cols = q.shape[-1]
    W = np.empty(q.shape, dtype=np.uint16)
    _check(_L().oracle_dequantize_q4(_p(q), _p(s), _p(b), q.size // cols, cols, _p(W)),
           "dequantize_q4")
    return W


def dequantize_q4_f64(q, s, b):
    """The exact values q·s + b (float64, the shape of q), before the one
    rounding to bf16 that gives the dequantised weights."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    b = _c(b, np.uint16)
    cols = q.shape[-1]
    W = np.empty(q.shape, dtype=np.float64)
    _check(_L().oracle_dequantize_q4_f64(_p(q), _p(s), _p(b), q.size // cols, cols, _p(W)),
           "dequantize_q4_f64")
    return W


def quantize_experts_q4(Wg, Wu, Wd):
    """quantize_q4 of the three expert matrices: {"gate": (q, s, b), "up": ..., "down": ...}."""
    return {"gate": quantize_q4(Wg), "up": quantize_q4(Wu), "down": quantize_q4(Wd)}


def _q4_args(q4):
    out = []
    for name in ("gate", "up", "down"):
        q, s, b = q4[name]
        out += [_c(q, np.uint8), _c(s, np.uint16), _c(b, np.uint16)]
    return out


def moe_forward_q4(x, Wr, q4, K, norm, rows=None, flags=0, bias=None, capacity=0):
    """moe_forward on 4-bit experts (q4 from quantize_experts_q4): the expert
    weights are w' = bf16(q·s + b).  Same results dict as moe_forward."""
    x = _c(x, np.uint16)
    Wr = _c(Wr, np.uint16)
    a9 = _q4_args(q4)
    T, H = x.shape
    E, I, _ = a9[0].shape
    assert Wr.shape == (E, H) and a9[3].shape == (E, I, H) and a9[6].shape == (E, H, I)
    if rows is not None:
        rows = _c(rows, np.int32)
        n = rows.shape[0]
    else:
        n = T
    out = np.empty((n, H), np.uint16)
    out_f64 = np.empty((n, H), np.float64)
    logits = np.empty((T, E), np.float32)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    counts = np.empty(E, np.int32)
    a = np.zeros(1, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    _check(_L().oracle_moe_forward_q4(_p(x), T, H, _p(Wr), _p(b), int(capacity),
                                      *[_p(v) for v in a9], E, K, I, int(bool(norm)), flags,
                                      _p(rows), n, _p(out), _p(out_f64), _p(logits), _p(idx),
                                      _p(w), _p(a), _p(counts)), "forward_q4")
    return dict(out=out, out_f64=out_f64, logits=logits, idx=idx, w=w, aux=float(a[0]),
                counts=counts)


def token_output_q4(x_row, idx_row, w_row, q4, flags=0, unrounded=False):
    """token_output on 4-bit experts (weights w' = bf16(q·s + b))."""
    x_row = _c(x_row, np.uint16)
    idx_row = _c(idx_row, np.int32)
    w_row = _c(w_row, np.float32)
    a9 = _q4_args(q4)
    E, I, H = a9[0].shape
    out = np.empty(H, np.uint16)
    f64 = np.empty(H, np.float64) if unrounded else None
    _check(_L().oracle_token_output_q4(_p(x_row), H, _p(idx_row), _p(w_row), idx_row.shape[0],
                                       *[_p(v) for v in a9], E, I, flags, _p(out), _p(f64)),
           "token_output_q4")
    return (out, f64) if unrounded else out
