"""ctypes binding of libmoe_b300.so: same names as the C ABI (include/moe_b300.h),
torch tensors in, data pointers and the current CUDA stream out.  Argument
marshalling only -- every step of the forward runs in the library's kernels.
There is no fallback: without the built library every call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_ALIGNMENT = 2
MOE_ERR_UNSUPPORTED_DEVICE = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_PATH_AUTO = 0
MOE_PATH_STREAMING = 1
MOE_PATH_TCGEN05 = 2
MOE_PATH_TCGEN05_WT = 3
MOE_PATH_TCGEN05_PAIR = 4
MOE_PATH_TCGEN05_DECODE = 5
MOE_PATH_WARP_MMA = 6

EXPORTS = ["moe_forward", "moe_forward_noalloc", "moe_workspace_bytes", "moe_forward_ws", "moe_forward_host",
           "moe_packed_experts_bytes", "moe_pack_experts", "moe_forward_packed",
           "moe_forward_host_packed", "moe_forward_opts", "moe_q4_experts_bytes",
           "moe_quantize_experts_q4", "moe_dequantize_experts_q4", "moe_forward_q4",
           "moe_forward_host_q4",
           "moe_last_expert_counts", "moe_device_status", "moe_strerror", "moe_last_cuda_error",
           "moe_set_expert_path", "moe_set_stage_timing", "moe_set_next_stage_events",
           "moe_stage_times",
           "moe_kernel_launch_count", "moe_dbg_route_from_logits", "moe_dbg_permute",
           "moe_dbg_combine", "moe_dbg_wait_timeout"]
MOE_NUM_STAGES = 5
STAGE_NAMES = ["router", "dispatch", "gate_up", "down", "combine"]


class _Options(ctypes.Structure):
    """struct moe_forward_options."""
    _fields_ = [("expert_bias", ctypes.c_void_p), ("packed_experts", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("capacity_factor", ctypes.c_float), ("q4_experts", ctypes.c_void_p)]


class MoEError(RuntimeError):
    def __init__(self, status, what):
        msg = lib().moe_strerror(status).decode()
        if status == MOE_ERR_CUDA:
            msg += f" (cudaError {lib().moe_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [status {status}]")
        self.status = status


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run python -m mixture_experts_layer_98_b300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        fwd = [P, i, i, P, P, P, P, i, i, i, i, P, P, P, P, P]
        L.moe_forward.argtypes = fwd + [P]
        L.moe_forward_ws.argtypes = fwd + [P, sz, P]
        L.moe_forward_host.argtypes = fwd + [P]
        L.moe_forward_noalloc.argtypes = fwd + [P]
        L.moe_packed_experts_bytes.argtypes = [i, i, i]
        L.moe_packed_experts_bytes.restype = sz
        L.moe_pack_experts.argtypes = [P, P, P, i, i, i, P, P]
        pfwd = [P, i, i, P, P, i, i, i, i, P, P, P, P, P]
        L.moe_forward_packed.argtypes = pfwd + [P, sz, P]
        L.moe_forward_host_packed.argtypes = pfwd + [P]
        L.moe_forward_opts.argtypes = fwd + [ctypes.POINTER(_Options), P]
        L.moe_q4_experts_bytes.argtypes = [i, i, i]
        L.moe_q4_experts_bytes.restype = sz
        L.moe_quantize_experts_q4.argtypes = [P, P, P, i, i, i, P, P]
        L.moe_dequantize_experts_q4.argtypes = [P, i, i, i, P, P, P, P]
        L.moe_forward_q4.argtypes = pfwd + [P, sz, P]
        L.moe_forward_host_q4.argtypes = pfwd + [P]
        L.moe_workspace_bytes.argtypes = [i, i, i, i, i]
        L.moe_workspace_bytes.restype = sz
        L.moe_last_expert_counts.argtypes = [P, i, P]
        L.moe_device_status.argtypes = [P, i, i, i, i, i, P]
        L.moe_strerror.argtypes = [i]
        L.moe_strerror.restype = ctypes.c_char_p
        L.moe_last_cuda_error.argtypes = []
        L.moe_set_expert_path.argtypes = [i]
        L.moe_set_stage_timing.argtypes = [i]
        L.moe_stage_times.argtypes = [P, i]
        L.moe_set_next_stage_events.argtypes = [P]
        L.moe_kernel_launch_count.argtypes = []
        L.moe_kernel_launch_count.restype = ctypes.c_longlong
        L.moe_dbg_route_from_logits.argtypes = [P, i, i, i, i, P, P, P, P]
        L.moe_dbg_permute.argtypes = [P, i, i, i, i, P, P, P, P, P, P]
        L.moe_dbg_combine.argtypes = [P, P, i, i, i, P, P]
        L.moe_dbg_wait_timeout.argtypes = [ctypes.c_longlong, P, P]
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, dtype, name, shape=None):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _call(rc, what):
    if rc != MOE_OK:
        raise MoEError(rc, what)


def _shapes(x, W_router, W_gate, W_up, W_down):
    T, H = x.shape
    E, I, H2 = W_gate.shape
    if H2 != H:
        raise ValueError("W_gate must be [E, I, H]")
    _dev(x, torch.bfloat16, "x")
    _dev(W_router, torch.bfloat16, "W_router", (E, H))
    _dev(W_gate, torch.bfloat16, "W_gate", (E, I, H))
    _dev(W_up, torch.bfloat16, "W_up", (E, I, H))
    _dev(W_down, torch.bfloat16, "W_down", (E, H, I))
    return T, H, E, I


def moe_forward(x, W_router, W_gate, W_up, W_down, K, norm_topk_prob, out=None,
                router_logits=None, topk_idx=None, topk_w=None, aux=None, stream=None,
                workspace=None):
    """Block forward (moe_forward, or moe_forward_ws when `workspace` is a uint8
    CUDA tensor).  Output tensors not given are allocated (router_logits,
    topk_idx, topk_w and aux always are, unless passed as False to skip them).
    Returns (out, router_logits, topk_idx, topk_w, aux)."""
    T, H, E, I = _shapes(x, W_router, W_gate, W_up, W_down)
    out, router_logits, topk_idx, topk_w, aux = _outputs(T, H, E, K, x.device, out, router_logits,
                                                         topk_idx, topk_w, aux)
    args = [_ptr(x), T, H, _ptr(W_router), _ptr(W_gate), _ptr(W_up), _ptr(W_down), E, K, I,
            int(bool(norm_topk_prob)), _ptr(out), _ptr(router_logits), _ptr(topk_idx),
            _ptr(topk_w), _ptr(aux)]
    if workspace is None:
        _call(lib().moe_forward(*args, _stream(stream)), "moe_forward")
    else:
        _dev(workspace, torch.uint8, "workspace")
        _call(lib().moe_forward_ws(*args, _ptr(workspace), workspace.numel(), _stream(stream)),
              "moe_forward_ws")
    return out, router_logits, topk_idx, topk_w, aux


def _outputs(T, H, E, K, dev, out, router_logits, topk_idx, topk_w, aux):
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if router_logits is None:
        router_logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if topk_idx is None:
        topk_idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, K), dtype=torch.float32, device=dev)
    if aux is None:
        aux = torch.empty((1,), dtype=torch.float32, device=dev)
    router_logits = None if router_logits is False else router_logits
    topk_idx = None if topk_idx is False else topk_idx
    topk_w = None if topk_w is False else topk_w
    aux = None if aux is False else aux
    _dev(out, torch.bfloat16, "out", (T, H))
    _dev(router_logits, torch.float32, "router_logits", (T, E))
    _dev(topk_idx, torch.int32, "topk_idx", (T, K))
    _dev(topk_w, torch.float32, "topk_w", (T, K))
    _dev(aux, torch.float32, "aux", (1,))
    return out, router_logits, topk_idx, topk_w, aux


class PackedExperts:
    """Expert weights in the packed tile-major layout of moe_pack_experts:
    `data` is the uint8 CUDA buffer, E, H, I the layer's sizes."""

    def __init__(self, data, E, H, I):
        self.data, self.E, self.H, self.I = data, E, H, I


def moe_packed_experts_bytes(H, E, I):
    return int(lib().moe_packed_experts_bytes(H, E, I))


def moe_pack_experts(W_gate, W_up, W_down, stream=None):
    """Packs the row-major expert weights once (a model-load step); returns a
    PackedExperts for moe_forward_packed / moe_forward_host_packed."""
    E, I, H = W_gate.shape
    _dev(W_gate, torch.bfloat16, "W_gate", (E, I, H))
    _dev(W_up, torch.bfloat16, "W_up", (E, I, H))
    _dev(W_down, torch.bfloat16, "W_down", (E, H, I))
    n = moe_packed_experts_bytes(H, E, I)
    if n == 0:
        raise ValueError(f"expert weights with H={H}, I={I} cannot be packed "
                         "(needs I % 128 == 0 and H % 256 == 0)")
    data = torch.empty(n, dtype=torch.uint8, device=W_gate.device)
    _call(lib().moe_pack_experts(_ptr(W_gate), _ptr(W_up), _ptr(W_down), H, E, I, _ptr(data),
                                 _stream(stream)), "moe_pack_experts")
    return PackedExperts(data, E, H, I)


def moe_forward_packed(x, W_router, packed, K, norm_topk_prob, out=None, router_logits=None,
                       topk_idx=None, topk_w=None, aux=None, stream=None, workspace=None):
    """moe_forward with PackedExperts weights; `workspace` as for moe_forward."""
    T, H = x.shape
    E, I = packed.E, packed.I
    if packed.H != H:
        raise ValueError("x and the packed weights disagree on H")
    _dev(x, torch.bfloat16, "x")
    _dev(W_router, torch.bfloat16, "W_router", (E, H))
    out, router_logits, topk_idx, topk_w, aux = _outputs(T, H, E, K, x.device, out, router_logits,
                                                         topk_idx, topk_w, aux)
    if workspace is not None:
        _dev(workspace, torch.uint8, "workspace")
    _call(lib().moe_forward_packed(_ptr(x), T, H, _ptr(W_router), _ptr(packed.data), E, K, I,
                                   int(bool(norm_topk_prob)), _ptr(out), _ptr(router_logits),
                                   _ptr(topk_idx), _ptr(topk_w), _ptr(aux), _ptr(workspace),
                                   0 if workspace is None else workspace.numel(),
                                   _stream(stream)), "moe_forward_packed")
    return out, router_logits, topk_idx, topk_w, aux


def moe_forward_host_packed(x_host, W_router, packed, K, norm_topk_prob, out_host,
                            router_logits_host=None, topk_idx_host=None, topk_w_host=None,
                            aux_host=None, stream=None):
    """moe_forward_host with PackedExperts weights."""
    T, H = x_host.shape
    _dev(W_router, torch.bfloat16, "W_router", (packed.E, H))
    for n, t in (("x_host", x_host), ("out_host", out_host), ("router_logits_host",
                                                            router_logits_host),
                 ("topk_idx_host", topk_idx_host), ("topk_w_host", topk_w_host),
                 ("aux_host", aux_host)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous host tensor")
    _call(lib().moe_forward_host_packed(_ptr(x_host), T, H, _ptr(W_router), _ptr(packed.data),
                                        packed.E, K, packed.I, int(bool(norm_topk_prob)),
                                        _ptr(out_host), _ptr(router_logits_host),
                                        _ptr(topk_idx_host), _ptr(topk_w_host), _ptr(aux_host),
                                        _stream(stream)), "moe_forward_host_packed")
    return out_host


class Q4Experts:
    """4-bit group-quantised expert weights (moe_quantize_experts_q4): `data` is
    the uint8 CUDA buffer, E, H, I the layer's sizes."""

    def __init__(self, data, E, H, I):
        self.data, self.E, self.H, self.I = data, E, H, I


def moe_q4_experts_bytes(H, E, I):
    return int(lib().moe_q4_experts_bytes(H, E, I))


def moe_quantize_experts_q4(W_gate, W_up, W_down, stream=None):
    """Quantises the row-major expert weights once (a model-load step); returns a
    Q4Experts for moe_forward_q4 / moe_forward_opts(q4=...)."""
    E, I, H = W_gate.shape
    _dev(W_gate, torch.bfloat16, "W_gate", (E, I, H))
    _dev(W_up, torch.bfloat16, "W_up", (E, I, H))
    _dev(W_down, torch.bfloat16, "W_down", (E, H, I))
    n = moe_q4_experts_bytes(H, E, I)
    if n == 0:
        raise ValueError(f"expert weights with H={H}, I={I} cannot be quantised here "
                         "(needs I % 128 == 0 and H % 256 == 0)")
    data = torch.empty(n, dtype=torch.uint8, device=W_gate.device)
    _call(lib().moe_quantize_experts_q4(_ptr(W_gate), _ptr(W_up), _ptr(W_down), H, E, I,
                                        _ptr(data), _stream(stream)), "moe_quantize_experts_q4")
    return Q4Experts(data, E, H, I)


def moe_dequantize_experts_q4(q4, stream=None):
    """The dequantised bf16 weights (W_gate, W_up, W_down) of a Q4Experts."""
    E, H, I = q4.E, q4.H, q4.I
    dev = q4.data.device
    Wg = torch.empty((E, I, H), dtype=torch.bfloat16, device=dev)
    Wu = torch.empty((E, I, H), dtype=torch.bfloat16, device=dev)
    Wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev)
    _call(lib().moe_dequantize_experts_q4(_ptr(q4.data), H, E, I, _ptr(Wg), _ptr(Wu), _ptr(Wd),
                                          _stream(stream)), "moe_dequantize_experts_q4")
    return Wg, Wu, Wd


def moe_forward_q4(x, W_router, q4, K, norm_topk_prob, out=None, router_logits=None,
                   topk_idx=None, topk_w=None, aux=None, stream=None, workspace=None):
    """moe_forward with Q4Experts weights; `workspace` as for moe_forward."""
    T, H = x.shape
    E, I = q4.E, q4.I
    if q4.H != H:
        raise ValueError("x and the 4-bit weights disagree on H")
    _dev(x, torch.bfloat16, "x")
    _dev(W_router, torch.bfloat16, "W_router", (E, H))
    out, router_logits, topk_idx, topk_w, aux = _outputs(T, H, E, K, x.device, out, router_logits,
                                                         topk_idx, topk_w, aux)
    if workspace is not None:
        _dev(workspace, torch.uint8, "workspace")
    _call(lib().moe_forward_q4(_ptr(x), T, H, _ptr(W_router), _ptr(q4.data), E, K, I,
                               int(bool(norm_topk_prob)), _ptr(out), _ptr(router_logits),
                               _ptr(topk_idx), _ptr(topk_w), _ptr(aux), _ptr(workspace),
                               0 if workspace is None else workspace.numel(),
                               _stream(stream)), "moe_forward_q4")
    return out, router_logits, topk_idx, topk_w, aux


def moe_forward_host_q4(x_host, W_router, q4, K, norm_topk_prob, out_host,
                        router_logits_host=None, topk_idx_host=None, topk_w_host=None,
                        aux_host=None, stream=None):
    """moe_forward_host with Q4Experts weights."""
    T, H = x_host.shape
    if q4.H != H:
        raise ValueError("x_host and the 4-bit weights disagree on H")
    _dev(W_router, torch.bfloat16, "W_router", (q4.E, H))
    for n, t in (("x_host", x_host), ("out_host", out_host), ("router_logits_host",
                                                            router_logits_host),
                 ("topk_idx_host", topk_idx_host), ("topk_w_host", topk_w_host),
                 ("aux_host", aux_host)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous host tensor")
    _call(lib().moe_forward_host_q4(_ptr(x_host), T, H, _ptr(W_router), _ptr(q4.data), q4.E, K,
                                    q4.I, int(bool(norm_topk_prob)), _ptr(out_host),
                                    _ptr(router_logits_host), _ptr(topk_idx_host),
                                    _ptr(topk_w_host), _ptr(aux_host), _stream(stream)),
          "moe_forward_host_q4")
    return out_host


def moe_forward_opts(x, W_router, W_gate, W_up, W_down, K, norm_topk_prob, expert_bias=None,
                     packed=None, out=None, router_logits=None, topk_idx=None, topk_w=None,
                     aux=None, stream=None, workspace=None, capacity_factor=0.0, q4=None):
    """moe_forward_opts: expert_bias (fp32 [E] CUDA tensor) is the selection-only
    expert bias; packed a PackedExperts or q4 a Q4Experts (then W_gate / W_up /
    W_down may be None); workspace as for moe_forward; capacity_factor > 0 keeps
    the first ceil(cf·T·K/E) pairs of each expert in token order."""
    T, H = x.shape
    if packed is None and q4 is not None:
        packed_like = q4
    else:
        packed_like = packed
    if packed_like is not None:
        E, I = packed_like.E, packed_like.I
        _dev(x, torch.bfloat16, "x")
        _dev(W_router, torch.bfloat16, "W_router", (E, H))
    else:
        T, H, E, I = _shapes(x, W_router, W_gate, W_up, W_down)
    _dev(expert_bias, torch.float32, "expert_bias", (E,))
    if workspace is not None:
        _dev(workspace, torch.uint8, "workspace")
    out, router_logits, topk_idx, topk_w, aux = _outputs(T, H, E, K, x.device, out, router_logits,
                                                         topk_idx, topk_w, aux)
    opts = _Options(_ptr(expert_bias), None if packed is None else packed.data.data_ptr(),
                    _ptr(workspace), 0 if workspace is None else workspace.numel(),
                    float(capacity_factor), None if q4 is None else q4.data.data_ptr())
    _call(lib().moe_forward_opts(_ptr(x), T, H, _ptr(W_router), _ptr(W_gate), _ptr(W_up),
                                 _ptr(W_down), E, K, I, int(bool(norm_topk_prob)), _ptr(out),
                                 _ptr(router_logits), _ptr(topk_idx), _ptr(topk_w), _ptr(aux),
                                 ctypes.byref(opts), _stream(stream)), "moe_forward_opts")
    return out, router_logits, topk_idx, topk_w, aux


def moe_workspace_bytes(T, H, E, K, I):
    return int(lib().moe_workspace_bytes(T, H, E, K, I))


def moe_forward_host(x_host, W_router, W_gate, W_up, W_down, K, norm_topk_prob, out_host,
                     router_logits_host=None, topk_idx_host=None, topk_w_host=None,
                     aux_host=None, stream=None):
    """End-to-end call: host (ideally pinned) x_host [T,H] bf16 in, host outputs
    filled on return.  Weights are CUDA tensors."""
    T, H = x_host.shape
    E, I, _ = W_gate.shape
    for n, t in (("W_router", W_router), ("W_gate", W_gate), ("W_up", W_up), ("W_down", W_down)):
        _dev(t, torch.bfloat16, n)
    for n, t in (("x_host", x_host), ("out_host", out_host), ("router_logits_host",
                                                            router_logits_host),
                 ("topk_idx_host", topk_idx_host), ("topk_w_host", topk_w_host),
                 ("aux_host", aux_host)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous host tensor")
    _call(lib().moe_forward_host(_ptr(x_host), T, H, _ptr(W_router), _ptr(W_gate), _ptr(W_up),
                                 _ptr(W_down), E, K, I, int(bool(norm_topk_prob)),
                                 _ptr(out_host), _ptr(router_logits_host), _ptr(topk_idx_host),
                                 _ptr(topk_w_host), _ptr(aux_host), _stream(stream)),
          "moe_forward_host")
    return out_host


def moe_last_expert_counts(E, stream=None):
    c = torch.empty(E, dtype=torch.int32)
    _call(lib().moe_last_expert_counts(_ptr(c), E, _stream(stream)), "moe_last_expert_counts")
    return c


def moe_device_status(workspace=None, sizes=(0, 64, 1, 1, 64), stream=None):
    T, H, E, K, I = sizes
    return int(lib().moe_device_status(_ptr(workspace), T, H, E, K, I, _stream(stream)))


def moe_set_expert_path(path):
    prev = lib().moe_set_expert_path(int(path))
    if prev < 0:
        raise ValueError(f"unknown expert path {path}")
    return prev


def moe_set_stage_timing(enable):
    _call(lib().moe_set_stage_timing(int(bool(enable))), "moe_set_stage_timing")


def moe_set_next_stage_events(events):
    """events: MOE_NUM_STAGES + 1 torch.cuda.Event objects (already recorded once,
    so their CUDA events exist) for the next forward's stage boundaries."""
    arr = (ctypes.c_void_p * (MOE_NUM_STAGES + 1))(*[e.cuda_event for e in events])
    _call(lib().moe_set_next_stage_events(arr), "moe_set_next_stage_events")


def moe_stage_times():
    """Per-stage device milliseconds of the last forward timed with stage timing."""
    ms = (ctypes.c_float * MOE_NUM_STAGES)()
    _call(lib().moe_stage_times(ms, MOE_NUM_STAGES), "moe_stage_times")
    return dict(zip(STAGE_NAMES, [float(v) for v in ms]))


def moe_kernel_launch_count():
    return int(lib().moe_kernel_launch_count())


def moe_dbg_route_from_logits(logits, K, norm_topk_prob, stream=None, expert_bias=None):
    T, E = logits.shape
    _dev(logits, torch.float32, "logits")
    _dev(expert_bias, torch.float32, "expert_bias", (E,))
    idx = torch.empty((T, K), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    _call(lib().moe_dbg_route_from_logits(_ptr(logits), T, E, K, int(bool(norm_topk_prob)),
                                          _ptr(expert_bias), _ptr(idx), _ptr(w), _stream(stream)),
          "moe_dbg_route_from_logits")
    return idx, w


def moe_dbg_permute(topk_idx, E, stream=None, capacity=0):
    T, K = topk_idx.shape
    _dev(topk_idx, torch.int32, "topk_idx")
    d = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=d)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=d)
    perm_tok = torch.empty(max(T * K, 1), dtype=torch.int32, device=d)
    perm_slot = torch.empty(max(T * K, 1), dtype=torch.int32, device=d)
    inv = torch.empty(max(T * K, 1), dtype=torch.int32, device=d)
    _call(lib().moe_dbg_permute(_ptr(topk_idx), T, E, K, int(capacity), _ptr(counts),
                                _ptr(offsets),
                                _ptr(perm_tok), _ptr(perm_slot), _ptr(inv), _stream(stream)),
          "moe_dbg_permute")
    n = T * K
    return dict(counts=counts, offsets=offsets, perm_tok=perm_tok[:n], perm_slot=perm_slot[:n],
                inv=inv[:n].view(T, K))


def moe_dbg_combine(Y, inv, stream=None):
    T, K = inv.shape
    H = Y.shape[1]
    _dev(Y, torch.bfloat16, "Y")
    _dev(inv, torch.int32, "inv")
    out = torch.empty((T, H), dtype=torch.bfloat16, device=Y.device)
    _call(lib().moe_dbg_combine(_ptr(Y), _ptr(inv), T, K, H, _ptr(out), _stream(stream)),
          "moe_dbg_combine")
    return out


def moe_dbg_wait_timeout(timeout_ns, stream=None):
    """Runs the bounded-wait self-test; returns the device status word it wrote."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _call(lib().moe_dbg_wait_timeout(int(timeout_ns), _ptr(st), _stream(stream)),
          "moe_dbg_wait_timeout")
    return int(st.cpu()[0])

