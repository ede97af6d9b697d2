"""GB300-native single-GPU Mixture-of-Experts layer forward.

Thin ctypes binding over the C ABI in ``include/moe.h`` (``libmoe_gb300.so``): every
function below has the name of the C entry point it calls and does argument marshalling
only (torch tensors -> device pointers, the current CUDA stream). Every step of the layer
runs in the library's CUDA kernels; there is no other implementation behind these names,
and a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
from ctypes import c_float, c_int32, c_int64, c_size_t, c_void_p, POINTER, byref

from ._build import build as _build_lib, LIB as _LIB_PATH

F32, BF16, E4M3, MXE4M3 = 0, 1, 2, 3
SOFTMAX, SIGMOID = 0, 1
GROUP_TOP2_SUM, GROUP_MAX = 0, 1

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_DEVICE_BAD_INPUT, MOE_ERR_TIMEOUT = 4, 5


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {moe_status_string(code)} (status {code})")


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", c_int32), ("H", c_int32), ("E", c_int32), ("k", c_int32), ("F", c_int32),
                ("n_shared", c_int32), ("F_shared", c_int32), ("score_fn", c_int32),
                ("renorm", c_int32), ("n_groups", c_int32), ("topk_groups", c_int32),
                ("group_score", c_int32), ("routed_scale", c_float), ("act_dtype", c_int32),
                ("xfer_dtype", c_int32)]

    @classmethod
    def make(cls, **kw) -> "MoEConfig":
        c = cls()
        defaults = dict(n_shared=0, F_shared=0, score_fn=SOFTMAX, renorm=0, n_groups=1,
                        topk_groups=1, group_score=GROUP_TOP2_SUM, routed_scale=1.0,
                        act_dtype=BF16)
        defaults.update(kw)
        defaults.setdefault("xfer_dtype", defaults["act_dtype"])
        for name, _ in cls._fields_:
            setattr(c, name, defaults[name])
        return c

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class MoEWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("w_router", "router_bias", "w_gate", "w_up", "w_down",
                                          "s_gate", "s_up", "s_down", "ws_gate", "ws_up",
                                          "ws_down", "ss_gate", "ss_up", "ss_down")]

    @classmethod
    def from_tensors(cls, d: dict) -> "MoEWeights":
        w = cls()
        for name, _ in cls._fields_:
            setattr(w, name, _ptr(d.get(name)))
        return w


class MoEWeightGrads(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("dw_gate", "dw_up", "dw_down", "dws_gate", "dws_up", "dws_down",
                                        "dw_router", "d_router_bias", "dlogits")] + [("aux_loss_coeff", ctypes.c_float)]

    @classmethod
    def from_tensors(cls, d: dict) -> "MoEWeightGrads":
        """Tensors by field name (absent: NULL); ``aux_loss_coeff`` a number (absent: 0)."""
        g = cls()
        for name, _ in cls._fields_[:-1]:
            setattr(g, name, _ptr(d.get(name)))
        g.aux_loss_coeff = float(d.get("aux_loss_coeff", 0.0))
        return g


_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a in-tree (no-op when up to date)."""
    return _build_lib(force=force)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        try:
            L = ctypes.CDLL(_LIB_PATH)
        except OSError as e:
            raise RuntimeError(f"CUDA library not available ({_LIB_PATH}): {e}; run build()") from e
        P, S = c_void_p, ctypes.c_int
        cfg = POINTER(MoEConfig)
        wts = POINTER(MoEWeights)
        sig = {
            "moe_workspace_size": [cfg, POINTER(c_size_t)],
            "moe_forward_workspace_size": [cfg, POINTER(c_size_t)],
            "moe_workspace_init": [P, P],
            "moe_router_logits": [cfg, P, P, P, P, P, P],
            "moe_route": [cfg, P, P, P, P, P, P, P, P, P],
            "moe_route_from_map": [cfg, P, P, P, P, P, P, P],
            "moe_route_launch_count": [cfg, POINTER(c_int32)],
            "moe_aux_loss": [cfg, P, P, ctypes.c_float, P, P, P],
            "moe_dispatch": [cfg, P, P, P, P, P],
            "moe_dispatch_mx": [cfg, P, P, P, P, P, P, P],
            "moe_mx_scale_bytes": [cfg, c_int32, POINTER(c_size_t)],
            "moe_quantize_mx": [P, c_int64, c_int64, P, P, P],
            "moe_backward_workspace_size": [cfg, POINTER(c_size_t)],
            "moe_combine_backward": [cfg, P, P, P, P, P, P, P],
            "moe_grouped_mlp_backward": [cfg, P, P, P, wts, P, P, POINTER(MoEWeightGrads), P, P],
            "moe_dispatch_backward": [cfg, P, P, P, P],
            "moe_backward": [cfg, P, wts, P, P, P, P, POINTER(MoEWeightGrads), P, P],
            "moe_forward_train": [cfg, P, wts, P, P, P, ctypes.c_float, P, P],
            "moe_backward_kept": [cfg, P, wts, P, P, P, P, P, POINTER(MoEWeightGrads), P, P],
            "moe_router_backward_workspace_size": [cfg, POINTER(c_size_t)],
            "moe_router_backward": [cfg, P, P, P, P, ctypes.c_float, P, P, P, P, P, P],
            "moe_dispatch_router_backward": [cfg, P, P, P, P, P, P, P],
            "moe_grouped_mlp": [cfg, P, P, P, P, wts, P, P, P, P, P],
            "moe_grouped_mlp_gather": [cfg, P, P, P, P, P, wts, P, P, P, P],
            "moe_combine": [cfg, P, P, P, P, P],
            "moe_forward": [cfg, P, wts, P, P, P, P, P, P],
            "moe_forward_host": [cfg, P, wts, P, P, P, P, P],
            "moe_quantize_e4m3": [P, c_int64, c_int64, c_int32, c_int32, P, P, P],
            "moe_read_status": [P, P, POINTER(c_int32)],
            "moe_route_static_scratch": [cfg, P, P, P, P, P, P, P, P, P],
            "moe_selftest_bounded_wait": [c_int64, P, P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = S
        L.moe_status_string.argtypes = [S]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def exported_symbols() -> list:
    return ["moe_workspace_size", "moe_forward_workspace_size", "moe_workspace_init",
            "moe_router_logits", "moe_route", "moe_route_launch_count", "moe_route_from_map", "moe_aux_loss",
            "moe_dispatch",
            "moe_grouped_mlp", "moe_grouped_mlp_gather", "moe_combine", "moe_forward", "moe_forward_host",
            "moe_quantize_e4m3",
            "moe_dispatch_mx", "moe_mx_scale_bytes", "moe_quantize_mx",
            "moe_backward_workspace_size", "moe_combine_backward", "moe_grouped_mlp_backward",
            "moe_dispatch_backward", "moe_backward", "moe_forward_train", "moe_backward_kept",
            "moe_router_backward_workspace_size",
            "moe_router_backward", "moe_dispatch_router_backward",
            "moe_read_status", "moe_status_string", "moe_route_static_scratch",
            "moe_selftest_bounded_wait"]


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _host_ptr(t):
    if t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoEError(code, where)


def moe_status_string(code: int) -> str:
    try:
        return lib().moe_status_string(code).decode()
    except RuntimeError:
        return f"status {code}"


def moe_workspace_size(cfg: MoEConfig) -> int:
    n = c_size_t()
    _check(lib().moe_workspace_size(byref(cfg), byref(n)), "moe_workspace_size")
    return n.value


def moe_route_launch_count(cfg: MoEConfig) -> int:
    n = c_int32()
    _check(lib().moe_route_launch_count(byref(cfg), byref(n)), "moe_route_launch_count")
    return n.value


def moe_forward_workspace_size(cfg: MoEConfig) -> int:
    n = c_size_t()
    _check(lib().moe_forward_workspace_size(byref(cfg), byref(n)), "moe_forward_workspace_size")
    return n.value


def moe_workspace_init(ws, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), _stream(stream)), "moe_workspace_init")


def moe_router_logits(cfg, x, w_router, router_bias, logits, ws, stream=None):
    _check(lib().moe_router_logits(byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias),
                                   _ptr(logits), _ptr(ws), _stream(stream)), "moe_router_logits")


def moe_route(cfg, logits, topk_idx, topk_w, counts, offsets, row_token, tok_row, ws, stream=None):
    _check(lib().moe_route(byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
                           _ptr(offsets), _ptr(row_token), _ptr(tok_row), _ptr(ws),
                           _stream(stream)), "moe_route")


def moe_route_from_map(cfg, topk_idx, counts, offsets, row_token, tok_row, ws, stream=None):
    _check(lib().moe_route_from_map(byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                                    _ptr(row_token), _ptr(tok_row), _ptr(ws), _stream(stream)),
           "moe_route_from_map")


def moe_aux_loss(cfg, logits, counts, alpha: float, loss, ws, stream=None):
    _check(lib().moe_aux_loss(byref(cfg), _ptr(logits), _ptr(counts), float(alpha), _ptr(loss), _ptr(ws),
                              _stream(stream)), "moe_aux_loss")


def moe_dispatch(cfg, x, tok_row, xd, xd_scale=None, stream=None):
    _check(lib().moe_dispatch(byref(cfg), _ptr(x), _ptr(tok_row), _ptr(xd), _ptr(xd_scale),
                              _stream(stream)), "moe_dispatch")


def moe_dispatch_mx(cfg, x, topk_idx, tok_row, offsets, xd, xd_sf, stream=None):
    _check(lib().moe_dispatch_mx(byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(tok_row), _ptr(offsets), _ptr(xd),
                                 _ptr(xd_sf), _stream(stream)), "moe_dispatch_mx")


def moe_mx_scale_bytes(cfg: MoEConfig, K: int) -> int:
    n = c_size_t()
    _check(lib().moe_mx_scale_bytes(byref(cfg), int(K), byref(n)), "moe_mx_scale_bytes")
    return n.value


def moe_grouped_mlp(cfg, xd, xd_scale, x, offsets, weights: dict, h, h_scale, yd, ws, stream=None):
    w = MoEWeights.from_tensors(weights)
    _check(lib().moe_grouped_mlp(byref(cfg), _ptr(xd), _ptr(xd_scale), _ptr(x), _ptr(offsets),
                                 byref(w), _ptr(h), _ptr(h_scale), _ptr(yd), _ptr(ws),
                                 _stream(stream)), "moe_grouped_mlp")


def moe_grouped_mlp_gather(cfg, x, row_token, offsets, weights: dict, h, yd, ws, stream=None,
                           tok_row=None, topk_w=None):
    """tok_row and topk_w (both or neither): the routing weights applied in GEMM2's epilogue."""
    w = MoEWeights.from_tensors(weights)
    _check(lib().moe_grouped_mlp_gather(byref(cfg), _ptr(x), _ptr(row_token), _ptr(offsets), _ptr(tok_row),
                                        _ptr(topk_w), byref(w), _ptr(h), _ptr(yd), _ptr(ws), _stream(stream)),
           "moe_grouped_mlp_gather")


def moe_combine(cfg, yd, tok_row, topk_w, y, stream=None):
    _check(lib().moe_combine(byref(cfg), _ptr(yd), _ptr(tok_row), _ptr(topk_w), _ptr(y),
                             _stream(stream)), "moe_combine")


def moe_forward(cfg, x, weights: dict, y, ws, topk_idx_out=None, topk_w_out=None,
                counts_out=None, stream=None):
    w = MoEWeights.from_tensors(weights)
    _check(lib().moe_forward(byref(cfg), _ptr(x), byref(w), _ptr(y), _ptr(ws), _ptr(topk_idx_out),
                             _ptr(topk_w_out), _ptr(counts_out), _stream(stream)), "moe_forward")


def moe_forward_host(cfg, x_host, weights: dict, y_host, x_dev, y_dev, ws, stream=None):
    """The layer on host tokens: x_host -> x_dev, moe_forward, y_dev -> y_host, stream-ordered
    (pin the host tensors to keep the copies asynchronous)."""
    w = MoEWeights.from_tensors(weights)
    _check(lib().moe_forward_host(byref(cfg), _host_ptr(x_host), byref(w), _host_ptr(y_host), _ptr(x_dev),
                                  _ptr(y_dev), _ptr(ws), _stream(stream)), "moe_forward_host")


def moe_quantize_e4m3(src, br: int, bc: int, q, scale, stream=None):
    rows, cols = src.shape
    _check(lib().moe_quantize_e4m3(_ptr(src), rows, cols, br, bc, _ptr(q), _ptr(scale),
                                   _stream(stream)), "moe_quantize_e4m3")


def moe_backward_workspace_size(cfg: MoEConfig) -> int:
    n = c_size_t()
    _check(lib().moe_backward_workspace_size(byref(cfg), byref(n)), "moe_backward_workspace_size")
    return n.value


def moe_combine_backward(cfg, dy, yd, tok_row, topk_w, dyd, dtopk_w, stream=None):
    _check(lib().moe_combine_backward(byref(cfg), _ptr(dy), _ptr(yd), _ptr(tok_row), _ptr(topk_w), _ptr(dyd),
                                      _ptr(dtopk_w), _stream(stream)), "moe_combine_backward")


def moe_grouped_mlp_backward(cfg, xd, x, offsets, weights: dict, dyd, dxd, grads: dict, ws, stream=None):
    w = MoEWeights.from_tensors(weights)
    g = MoEWeightGrads.from_tensors(grads)
    _check(lib().moe_grouped_mlp_backward(byref(cfg), _ptr(xd), _ptr(x), _ptr(offsets), byref(w), _ptr(dyd),
                                          _ptr(dxd), byref(g), _ptr(ws), _stream(stream)), "moe_grouped_mlp_backward")


def moe_dispatch_backward(cfg, dxd, tok_row, dx, stream=None):
    _check(lib().moe_dispatch_backward(byref(cfg), _ptr(dxd), _ptr(tok_row), _ptr(dx), _stream(stream)),
           "moe_dispatch_backward")


def moe_backward(cfg, x, weights: dict, dy, fwd_ws, dx, dtopk_w, grads: dict, bwd_ws, stream=None):
    w = MoEWeights.from_tensors(weights)
    g = MoEWeightGrads.from_tensors(grads)
    _check(lib().moe_backward(byref(cfg), _ptr(x), byref(w), _ptr(dy), _ptr(fwd_ws), _ptr(dx), _ptr(dtopk_w),
                              byref(g), _ptr(bwd_ws), _stream(stream)), "moe_backward")


def moe_forward_train(cfg, x, weights: dict, y, ws, gu, aux_alpha=0.0, aux_loss=None, stream=None):
    """moe_forward that also keeps the gate/up pre-activations in gu [R(+T), 2F] bf16, and
    (aux_loss: a 1-element fp32 CUDA tensor) computes the auxiliary load-balancing loss."""
    w = MoEWeights.from_tensors(weights)
    _check(lib().moe_forward_train(byref(cfg), _ptr(x), byref(w), _ptr(y), _ptr(ws), _ptr(gu), float(aux_alpha),
                                   _ptr(aux_loss), _stream(stream)), "moe_forward_train")


def moe_backward_kept(cfg, x, weights: dict, dy, fwd_ws, gu, dx, dtopk_w, grads: dict, bwd_ws, stream=None):
    """moe_backward reading the gate/up pre-activations kept by moe_forward_train."""
    w = MoEWeights.from_tensors(weights)
    g = MoEWeightGrads.from_tensors(grads)
    _check(lib().moe_backward_kept(byref(cfg), _ptr(x), byref(w), _ptr(dy), _ptr(fwd_ws), _ptr(gu), _ptr(dx),
                                   _ptr(dtopk_w), byref(g), _ptr(bwd_ws), _stream(stream)), "moe_backward_kept")


def moe_router_backward_workspace_size(cfg: MoEConfig) -> int:
    n = c_size_t()
    _check(lib().moe_router_backward_workspace_size(byref(cfg), byref(n)), "moe_router_backward_workspace_size")
    return n.value


def moe_router_backward(cfg, logits, topk_idx, dtopk_w, x, dlogits, dw_router, ws, d_router_bias=None,
                        counts=None, aux_alpha=0.0, stream=None):
    """dlogits (and, given dw_router, the router weight and bias gradients) from the
    routing-weight gradient dtopk_w; counts + aux_alpha add the auxiliary loss's gradient."""
    _check(lib().moe_router_backward(byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(dtopk_w), _ptr(counts),
                                     float(aux_alpha), _ptr(x), _ptr(dlogits), _ptr(dw_router), _ptr(d_router_bias),
                                     _ptr(ws), _stream(stream)), "moe_router_backward")


def moe_dispatch_router_backward(cfg, dxd, tok_row, dlogits, w_router, dx, ws, stream=None):
    """dx = dlogits W_router + the dispatch backward's sum of dxd rows (dxd None: the
    router's share alone). ws: moe_router_backward_workspace_size bytes."""
    _check(lib().moe_dispatch_router_backward(byref(cfg), _ptr(dxd), _ptr(tok_row), _ptr(dlogits), _ptr(w_router),
                                              _ptr(dx), _ptr(ws), _stream(stream)), "moe_dispatch_router_backward")


def moe_quantize_mx(src, q, sf, stream=None):
    rows, cols = src.shape
    _check(lib().moe_quantize_mx(_ptr(src), rows, cols, _ptr(q), _ptr(sf), _stream(stream)), "moe_quantize_mx")


def moe_route_static_scratch(cfg, logits, topk_idx, topk_w, counts, offsets, row_token, tok_row,
                             device_status=None, stream=None):
    """moe_route without a workspace, for callers that cannot allocate device memory: the
    scan's scratch is a fixed 1 MiB array inside the library, shared by every call on a
    device (overlapping calls race; the first call on a device must precede any capture).
    ``device_status``: optional int32 CUDA tensor of 2 elements for device-side faults."""
    _check(lib().moe_route_static_scratch(byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                                          _ptr(counts), _ptr(offsets), _ptr(row_token),
                                          _ptr(tok_row), _ptr(device_status), _stream(stream)),
           "moe_route_static_scratch")


def moe_selftest_bounded_wait(timeout_ns: int, device_status, stream=None):
    _check(lib().moe_selftest_bounded_wait(int(timeout_ns), _ptr(device_status), _stream(stream)),
           "moe_selftest_bounded_wait")


def moe_read_status(ws, stream=None) -> int:
    st = c_int32()
    _check(lib().moe_read_status(_ptr(ws), _stream(stream), byref(st)), "moe_read_status")
    return st.value
