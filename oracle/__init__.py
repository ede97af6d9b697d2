"""CPU oracle for the single-GPU MoE layer forward: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import
this package; the library (``token_routing_expert_router_gb300``) never does, and the two
share no code. The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, OpenMP over rows),
compiled on first use with gcc; this module only marshals numpy arrays into it and chains
the steps of the layer in the order the method states them:

  router logits -> top-k routing (optionally group-limited) -> per-expert counts, offsets
  and the stable permutation -> dispatch -> each expert's SwiGLU MLP -> combine,

plus the independent dense per-token loop that skips the permutation altogether.

Readings where the pages are silent (each one is a config field, so the oracle and the
library expose the same choices): the stable ascending-token order inside each expert,
the lowest-index tie-break, the group score (sum of the two largest sigmoid scores), the
softmax and sigmoid weight formulas, the routed scale, the FP8 block-scale rule
(scale = amax / 448, non-power-of-two fp32) and, for the MXFP8 variant, the OCP MX v1.0
conversion (1x32 blocks, UE8M0 scale 2^(floor(log2 amax) - 8), saturating e4m3). Parity
of these readings against the pages is unpinned (the pages print no formula or worked
example); the tests pin the code to brute force, closed forms, library routines and
invariants instead.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lib = None

F32, BF16, E4M3, MXE4M3 = 0, 1, 2, 3
SOFTMAX, SIGMOID = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -ffp-contract=off, no fast-math) into oracle/_build/."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        sig = {
            "oc_num_threads": (i32, []),
            "oc_det_expf": (f32, [f32]),
            "oc_det_sigmoidf": (f32, [f32]),
            "oc_det_expf_array": (None, [P, P, i64]),
            "oc_router_logits": (None, [P, P, P, i32, i32, i32, P]),
            "oc_route": (i32, [P, i32, i32, i32, i32, i32, i32, i32, i32, f64, P, P]),
            "oc_group_scores": (i32, [P, i32, i32, i32, P]),
            "oc_permute": (i32, [P, i32, i32, i32, P, P, P, P]),
            "oc_dispatch": (None, [P, i32, P, i64, P]),
            "oc_e4m3_decode": (f64, [ctypes.c_uint8]),
            "oc_e4m3_encode": (ctypes.c_uint8, [f32]),
            "oc_e4m3_encode_array": (None, [P, P, i64]),
            "oc_quant_blocks": (None, [P, i64, i64, i32, i32, P, P]),
            "oc_dequant_blocks": (None, [P, P, i64, i64, i32, i32, P]),
            "oc_mx_quant": (None, [P, i64, i64, P, P]),
            "oc_mx_dequant": (None, [P, P, i64, i64, P]),
            "oc_expert_mlp": (None, [P, i64, i32, i32, P, P, P, i32, P]),
            "oc_combine": (None, [P, P, P, P, i32, i32, i32, P]),
            "oc_aux_loss": (f64, [P, P, i32, i32, i32, i32, f64, P]),
            "oc_combine_backward": (None, [P, P, P, P, i32, i32, i32, i32, P, P]),
            "oc_expert_mlp_backward": (None, [P, i64, i32, i32, P, P, P, P, P, P, P, P]),
            "oc_dispatch_backward": (None, [P, P, i32, i32, i32, i32, P]),
            "oc_router_backward": (None, [P, i32, i32, i32, P, i32, i32, f64, P, P]),
            "oc_aux_loss_backward": (None, [P, P, i32, i32, i32, i32, f64, P]),
            "oc_dense_forward": (i32, [P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                       f64, P, P, P, i32, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def num_threads() -> int:
    return int(_L().oc_num_threads())


# ---------------------------------------------------------------- scalar helpers
def det_expf(a) -> np.ndarray:
    a = _c(np.atleast_1d(a), np.float32)
    out = np.empty_like(a)
    _L().oc_det_expf_array(_p(a), _p(out), a.size)
    return out


def det_sigmoidf(l: float) -> float:
    return float(_L().oc_det_sigmoidf(float(l)))


def e4m3_decode_all() -> np.ndarray:
    """Values of all 256 e4m3 codes (fp64; NaN for the two NaN codes)."""
    L = _L()
    return np.array([L.oc_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v) -> np.ndarray:
    v = _c(np.atleast_1d(v), np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _L().oc_e4m3_encode_array(_p(v), _p(out), v.size)
    return out


# ---------------------------------------------------------------- steps of the layer
def router_logits(x, w_router, bias=None) -> np.ndarray:
    x = _c(x, np.float32)
    wr = _c(w_router, np.float32)
    b = _c(bias, np.float32)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), dtype=np.float32)
    _L().oc_router_logits(_p(x), _p(wr), _p(b), T, H, E, _p(out))
    return out


def route(logits, cfg: dict):
    """(topk_idx int32 [T,k], topk_w fp64 [T,k]) from fp32 logits [T,E]."""
    l = _c(logits, np.float32)
    T, E = l.shape
    k = cfg["k"]
    G, g = cfg["n_groups"], cfg["topk_groups"]
    if k > E or E % G or not 1 <= g <= G or (G > 1 and g < G and g * (E // G) < k):
        raise ValueError("oracle route: k larger than the experts the groups allow")
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    rc = _L().oc_route(_p(l), T, E, k, cfg["score_fn"], cfg["renorm"], cfg["n_groups"],
                       cfg["topk_groups"], cfg["group_score"], float(cfg["routed_scale"]),
                       _p(idx), _p(w))
    if rc != 0:
        raise ValueError("oracle route: non-finite logit")
    return idx, w


def group_scores(logits_row, n_groups: int, group_score: int = 0) -> np.ndarray:
    l = _c(logits_row, np.float32)
    out = np.empty(n_groups, dtype=np.float32)
    _L().oc_group_scores(_p(l), l.size, n_groups, group_score, _p(out))
    return out


def permute(topk_idx, E: int):
    """(counts [E], offsets [E+1], row_token [T*k], tok_row [T,k]) — all int32."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    row_token = np.empty(T * k, dtype=np.int32)
    tok_row = np.empty((T, k), dtype=np.int32)
    rc = _L().oc_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(row_token), _p(tok_row))
    if rc != 0:
        raise ValueError("oracle permute: expert id out of range")
    return counts, offsets, row_token, tok_row


def dispatch(x, row_token) -> np.ndarray:
    x = _c(x, np.float32)
    rt = _c(row_token, np.int32)
    out = np.empty((rt.size, x.shape[1]), dtype=np.float32)
    _L().oc_dispatch(_p(x), x.shape[1], _p(rt), rt.size, _p(out))
    return out


def quant_blocks(v, br: int, bc: int):
    """e4m3 codes [rows, cols] and fp32 scales [ceil(rows/br), ceil(cols/bc)]."""
    v = _c(v, np.float32)
    rows, cols = v.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty(((rows + br - 1) // br, (cols + bc - 1) // bc), dtype=np.float32)
    _L().oc_quant_blocks(_p(v), rows, cols, br, bc, _p(q), _p(sc))
    return q, sc


def dequant_blocks(q, scale, br: int, bc: int) -> np.ndarray:
    q = _c(q, np.uint8)
    sc = _c(scale, np.float32)
    rows, cols = q.shape
    out = np.empty((rows, cols), dtype=np.float64)
    _L().oc_dequant_blocks(_p(q), _p(sc), rows, cols, br, bc, _p(out))
    return out


def mx_quant(v):
    """MX (OCP MXFP8 E4M3) quantisation along rows: e4m3 codes [rows, cols] and UE8M0
    scale codes [rows, cols/32] (value = decode(q) * 2^(code - 127))."""
    v = _c(v, np.float32)
    rows, cols = v.shape
    if cols % 32:
        raise ValueError("MX blocks need cols % 32 == 0")
    q = np.empty((rows, cols), dtype=np.uint8)
    sc = np.empty((rows, cols // 32), dtype=np.uint8)
    _L().oc_mx_quant(_p(v), rows, cols, _p(q), _p(sc))
    return q, sc


def mx_dequant(q, sc) -> np.ndarray:
    q = _c(q, np.uint8)
    sc = _c(sc, np.uint8)
    rows, cols = q.shape
    out = np.empty((rows, cols), dtype=np.float64)
    _L().oc_mx_dequant(_p(q), _p(sc), rows, cols, _p(out))
    return out


def expert_mlp(a, wg, wu, wd, quant_h=0) -> np.ndarray:
    """One expert's SwiGLU MLP on rows a [n,H] (fp64 values) -> [n,H] fp64. quant_h: 0 none,
    1 (or True) 1x128 fp32-scale requantisation of h, 2 MX (1x32 UE8M0) requantisation."""
    a = _c(a, np.float64)
    wg, wu, wd = _c(wg, np.float64), _c(wu, np.float64), _c(wd, np.float64)
    n, H = a.shape
    F = wg.shape[0]
    y = np.empty((n, H), dtype=np.float64)
    if n:
        _L().oc_expert_mlp(_p(a), n, H, F, _p(wg), _p(wu), _p(wd), int(quant_h), _p(y))
    return y


def combine(yd, tok_row, topk_w, ys=None) -> np.ndarray:
    yd = _c(yd, np.float64)
    tr = _c(tok_row, np.int32)
    w = _c(topk_w, np.float64)
    ys = _c(ys, np.float64)
    T, k = tr.shape
    H = yd.shape[1]
    y = np.empty((T, H), dtype=np.float64)
    _L().oc_combine(_p(yd), _p(tr), _p(w), _p(ys), T, k, H, _p(y))
    return y


def aux_loss(logits, counts, k: int, score_fn: int, alpha: float = 0.01):
    """(loss, Pbar[E]) of the switch-style load-balancing loss (fp64)."""
    l = _c(logits, np.float32)
    c = _c(counts, np.int32)
    T, E = l.shape
    pbar = np.empty(E, dtype=np.float64)
    loss = _L().oc_aux_loss(_p(l), _p(c), T, E, k, score_fn, float(alpha), _p(pbar))
    return float(loss), pbar


# ---------------------------------------------------------------- whole layer
def _expert_values(cfg: dict, W: np.ndarray, blocks):
    """The values an expert weight stands for: the stored values; for the FP8 variant
    decode(q) * scale of its 128x128-block quantisation; for the MXFP8 variant its 1x32 MX
    quantisation along the reduction dimension (each done here, by the oracle)."""
    if not blocks:
        return W.astype(np.float64)
    if blocks == MXE4M3:
        return mx_dequant(*mx_quant(W))
    q, s = quant_blocks(W, 128, 128)
    return dequant_blocks(q, s, 128, 128)


def forward(cfg: dict, inp: dict, logits=None) -> dict:
    """The layer, step by step, as the method orders it. ``inp`` holds fp32 arrays of exact
    values: x [T,H], w_router [E,H], router_bias [E] or None, w_gate/w_up [E,F,H],
    w_down [E,H,F] and, with a shared expert, ws_gate/ws_up [Fs,H], ws_down [H,Fs].
    Returns every intermediate (fp64 where the layer computes in floating point)."""
    T, H, E, k, F = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["F"]
    xfer = cfg["xfer_dtype"]
    fp8 = xfer if xfer in (E4M3, MXE4M3) else 0  # which quantisation, 0 = none
    quant_h = {0: 0, E4M3: 1, MXE4M3: 2}[fp8]
    out = {}
    out["logits"] = router_logits(inp["x"], inp["w_router"], inp.get("router_bias")) if logits is None else logits
    idx, w = route(out["logits"], cfg)
    counts, offsets, row_token, tok_row = permute(idx, E)
    out.update(topk_idx=idx, topk_w=w, counts=counts, offsets=offsets, row_token=row_token,
               tok_row=tok_row)
    if fp8 == MXE4M3:
        qx, sx = mx_quant(inp["x"])
        out["x_q"], out["x_scale"] = qx, sx
        a_tok = mx_dequant(qx, sx)
    elif fp8:
        qx, sx = quant_blocks(inp["x"], 1, 128)
        out["x_q"], out["x_scale"] = qx, sx
        a_tok = dequant_blocks(qx, sx, 1, 128)
    else:
        a_tok = inp["x"].astype(np.float64)
    xd = a_tok[row_token]
    yd = np.zeros((T * k, H), dtype=np.float64)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            yd[r0:r1] = expert_mlp(xd[r0:r1], _expert_values(cfg, inp["w_gate"][e], fp8),
                                   _expert_values(cfg, inp["w_up"][e], fp8),
                                   _expert_values(cfg, inp["w_down"][e], fp8), quant_h=quant_h)
    out["yd"] = yd
    ys = None
    if cfg["n_shared"]:
        ys = expert_mlp(a_tok, _expert_values(cfg, inp["ws_gate"], fp8),
                        _expert_values(cfg, inp["ws_up"], fp8),
                        _expert_values(cfg, inp["ws_down"], fp8), quant_h=quant_h)
    out["ys"] = ys
    out["y"] = combine(yd, tok_row, w, ys)
    return out


def dense_forward(cfg: dict, inp: dict, logits=None) -> np.ndarray:
    """The independent dense per-token loop (no counts, no permutation, no dispatch)."""
    T, H, E, k, F = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["F"]
    fp8 = cfg["xfer_dtype"] in (E4M3, MXE4M3)
    if logits is None:
        logits = router_logits(inp["x"], inp["w_router"], inp.get("router_bias"))
    l = _c(logits, np.float32)
    if fp8:
        raise NotImplementedError("the dense loop covers the unquantised layers")
    x = _c(inp["x"], np.float64)
    wg = _c(inp["w_gate"], np.float64)
    wu = _c(inp["w_up"], np.float64)
    wd = _c(inp["w_down"], np.float64)
    Fs = cfg["F_shared"] if cfg["n_shared"] else 0
    sg = _c(inp.get("ws_gate"), np.float64) if Fs else None
    su = _c(inp.get("ws_up"), np.float64) if Fs else None
    sd = _c(inp.get("ws_down"), np.float64) if Fs else None
    y = np.empty((T, H), dtype=np.float64)
    rc = _L().oc_dense_forward(_p(x), _p(l), T, H, E, k, F, cfg["score_fn"], cfg["renorm"],
                               cfg["n_groups"], cfg["topk_groups"], cfg["group_score"],
                               float(cfg["routed_scale"]), _p(wg), _p(wu), _p(wd), Fs, _p(sg),
                               _p(su), _p(sd), _p(y))
    if rc != 0:
        raise ValueError("oracle dense loop: non-finite logit")
    return y


# ---------------------------------------------------------------- backward (training step)
def combine_backward(dy, yd, tok_row, topk_w, shared: bool):
    """(dyd [R(+T), H], dtopk_w [T, k]) from dy [T, H] and the forward's yd (fp64)."""
    dy = _c(dy, np.float64)
    yd = _c(yd, np.float64)
    tr = _c(tok_row, np.int32)
    w = _c(topk_w, np.float64)
    T, k = tr.shape
    H = dy.shape[1]
    dyd = np.zeros((T * k + (T if shared else 0), H), dtype=np.float64)
    dw = np.empty((T, k), dtype=np.float64)
    _L().oc_combine_backward(_p(dy), _p(yd), _p(tr), _p(w), T, k, H, int(shared), _p(dyd), _p(dw))
    return dyd, dw


def expert_mlp_backward(a, wg, wu, wd, dyd):
    """(dxd [n,H], dWg [F,H], dWu [F,H], dWd [H,F]) of one expert's SwiGLU MLP (fp64,
    activations recomputed from a)."""
    a = _c(a, np.float64)
    wg, wu, wd = _c(wg, np.float64), _c(wu, np.float64), _c(wd, np.float64)
    dyd = _c(dyd, np.float64)
    n, H = a.shape
    F = wg.shape[0]
    dxd = np.zeros((n, H), dtype=np.float64)
    dwg = np.zeros((F, H), dtype=np.float64)
    dwu = np.zeros((F, H), dtype=np.float64)
    dwd = np.zeros((H, F), dtype=np.float64)
    if n:
        _L().oc_expert_mlp_backward(_p(a), n, H, F, _p(wg), _p(wu), _p(wd), _p(dyd), _p(dxd), _p(dwg), _p(dwu),
                                    _p(dwd))
    return dxd, dwg, dwu, dwd


def dispatch_backward(dxd, tok_row, shared: bool) -> np.ndarray:
    dxd = _c(dxd, np.float64)
    tr = _c(tok_row, np.int32)
    T, k = tr.shape
    H = dxd.shape[1]
    dx = np.empty((T, H), dtype=np.float64)
    _L().oc_dispatch_backward(_p(dxd), _p(tr), T, k, H, int(shared), _p(dx))
    return dx


def router_backward(cfg: dict, logits, topk_idx, dtopk_w) -> np.ndarray:
    """dL/dlogits [T, E] (fp64) from dL/dtopk_w [T, k], the chosen experts held fixed: the
    chain rule through the weight step of the routing (softmax over all experts or over the
    chosen k, or sigmoid with or without normalisation, times the routed scale)."""
    l = _c(logits, np.float32)
    idx = _c(topk_idx, np.int32)
    dw = _c(dtopk_w, np.float64)
    T, E = l.shape
    k = idx.shape[1]
    dl = np.empty((T, E), dtype=np.float64)
    _L().oc_router_backward(_p(l), T, E, k, _p(idx), cfg["score_fn"], cfg["renorm"], float(cfg["routed_scale"]),
                            _p(dw), _p(dl))
    return dl


def aux_loss_backward(logits, counts, k: int, score_fn: int, alpha: float = 0.01) -> np.ndarray:
    """dL_aux/dlogits [T, E] (fp64) of aux_loss, the routed counts held fixed."""
    l = _c(logits, np.float32)
    cn = _c(counts, np.int32)
    T, E = l.shape
    dl = np.zeros((T, E), dtype=np.float64)
    _L().oc_aux_loss_backward(_p(l), _p(cn), T, E, k, score_fn, float(alpha), _p(dl))
    return dl


def router_linear_backward(x, w_router, dlogits):
    """(dW_router [E, H], dx through the router [T, H]) of logits = x W_router^T: the two
    products of the linear map's gradient, in fp64."""
    dl = np.asarray(dlogits, dtype=np.float64)
    return dl.T @ np.asarray(x, dtype=np.float64), dl @ np.asarray(w_router, dtype=np.float64)


def backward(cfg: dict, inp: dict, fwd: dict, dy) -> dict:
    """The layer's backward with the routing of ``fwd`` (an oracle.forward result) held fixed:
    combine backward -> each expert's MLP backward -> dispatch backward. Unquantised layers.
    Returns dyd, dtopk_w, dxd, dx (the gradient reaching x through the experts), the
    expert weight gradients dw_gate/dw_up [E,F,H], dw_down [E,H,F] and, with a shared
    expert, dws_gate/dws_up [F,H], dws_down [H,F]."""
    if cfg["xfer_dtype"] in (E4M3, MXE4M3):
        raise NotImplementedError("the backward covers the unquantised layers")
    T, H, E, k, F = cfg["T"], cfg["H"], cfg["E"], cfg["k"], cfg["F"]
    shared = bool(cfg["n_shared"])
    R = T * k
    yd = fwd["yd"] if not shared else np.concatenate([fwd["yd"], fwd["ys"]])
    dyd, dw = combine_backward(dy, yd, fwd["tok_row"], fwd["topk_w"], shared)
    x = inp["x"].astype(np.float64)
    xd = x[fwd["row_token"]]
    offsets = fwd["offsets"]
    dxd = np.zeros((R + (T if shared else 0), H))
    out = {"dyd": dyd, "dtopk_w": dw,
           "dw_gate": np.zeros((E, F, H)), "dw_up": np.zeros((E, F, H)), "dw_down": np.zeros((E, H, F))}
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            dxd[r0:r1], out["dw_gate"][e], out["dw_up"][e], out["dw_down"][e] = expert_mlp_backward(
                xd[r0:r1], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e], dyd[r0:r1])
    if shared:
        dxd[R:], out["dws_gate"], out["dws_up"], out["dws_down"] = expert_mlp_backward(
            x, inp["ws_gate"], inp["ws_up"], inp["ws_down"], dyd[R:])
    out["dxd"] = dxd
    out["dx"] = dispatch_backward(dxd, fwd["tok_row"], shared)
    return out


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (d if d > 0 else 1.0))
