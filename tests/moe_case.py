"""Helpers shared by the GPU tests: build device inputs from the seeded generator, allocate
the layer's buffers, and run the library through its Python binding. Oracle inputs always
come from the host generator (never from a GPU result)."""
from __future__ import annotations

import numpy as np
import torch

import synth
import token_routing_expert_router_gb300 as moe


def cfg_of(w: dict) -> moe.MoEConfig:
    return moe.MoEConfig.make(**{k: w[k] for k in (
        "T", "H", "E", "k", "F", "n_shared", "F_shared", "score_fn", "renorm", "n_groups",
        "topk_groups", "group_score", "routed_scale", "act_dtype", "xfer_dtype")})


def tdtype(w: dict):
    return torch.bfloat16 if w["act_dtype"] == synth.BF16 else torch.float32


def up(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)  # fp32 -> bf16 is exact for bf16-valued arrays
    return t.cuda()


def quantize_dev(src: torch.Tensor, br: int, bc: int):
    rows, cols = src.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    s = torch.empty(((rows + br - 1) // br, (cols + bc - 1) // bc), dtype=torch.float32, device="cuda")
    moe.moe_quantize_e4m3(src, br, bc, q, s)
    return q, s


def quantize_mx_dev(src: torch.Tensor):
    """MX quantisation on the GPU: e4m3 codes and the scale atoms of the rows."""
    rows, cols = src.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows // 128) * (cols // 128) * 512, dtype=torch.uint8, device="cuda")
    moe.moe_quantize_mx(src, q, sf)
    return q, sf


def is_quant(w: dict) -> bool:
    return w["xfer_dtype"] in (synth.E4M3, synth.MXE4M3)


def _attach_fp8(w: dict, d: dict) -> dict:
    """Replace expert weights by their e4m3 quantisation (on the GPU): 128x128 blocks with
    fp32 scales, or 1x32 MX blocks with scale atoms."""
    if not is_quant(w):
        return d
    names = [("w_gate", "s_gate"), ("w_up", "s_up"), ("w_down", "s_down")]
    if w["n_shared"]:
        names += [("ws_gate", "ss_gate"), ("ws_up", "ss_up"), ("ws_down", "ss_down")]
    for wn, sn in names:
        src = d[wn]
        if w["xfer_dtype"] == synth.MXE4M3:
            q, s = quantize_mx_dev(src.reshape(-1, src.shape[-1]))
        else:
            q, s = quantize_dev(src.reshape(-1, src.shape[-1]), 128, 128)
        d[wn + "_bf16"] = src
        d[wn] = q.reshape(src.shape)
        d[sn] = s
    return d


# ---------------------------------------------------------------- MX scale-atom layout
# The byte of (row, 1x32 block) in a scale-atom buffer, as the C header documents it:
# atom (a, ks) at (a * K/128 + ks) * 512, row i of the atom's 128 and block kb of the
# stage's four at (i % 32) * 16 + (i // 32) * 4 + kb.
def mx_atom_offsets(atom_row: np.ndarray, row_in_tile: np.ndarray, K: int) -> np.ndarray:
    b = np.arange(K // 32)
    ks, kb = b // 4, b % 4
    a = atom_row.astype(np.int64)[:, None]
    i = row_in_tile.astype(np.int64)[:, None]
    return ((a * (K // 128) + ks[None, :]) << 9) + (i % 32) * 16 + (i // 32) * 4 + kb[None, :]


def mx_weight_rows(rows: int):
    r = np.arange(rows)
    return r // 128, r % 128


def mx_grouped_rows(offsets: np.ndarray, T: int, k: int, E: int, shared: bool):
    """(atom row, row in tile) of every dispatched row: expert e's rows start a fresh tile
    at ceil((offsets[e] + 127 e) / 128); the shared expert is e = E with offset T*k."""
    R = T * k
    r = np.arange(R, dtype=np.int64)
    off = offsets.astype(np.int64)
    g = np.searchsorted(off, r, side="right") - 1
    gofs = off[g]
    if shared:
        g = np.concatenate([g, np.full(T, E)])
        gofs = np.concatenate([gofs, np.full(T, R)])
        r = np.concatenate([r, R + np.arange(T)])
    base = (gofs + 127 * g + 127) // 128
    local = r - gofs
    return base + local // 128, local % 128


def device_weights_from_host(w: dict, inp: dict) -> dict:
    dt = tdtype(w)
    d = {"x": up(inp["x"], dt), "w_router": up(inp["w_router"], dt),
         "router_bias": None if inp.get("router_bias") is None else up(inp["router_bias"])}
    for key in ("w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"):
        if key in inp:
            d[key] = up(inp[key], dt)
    return _attach_fp8(w, d)


def device_weights_generated(w: dict, seed: int = 0) -> dict:
    """The same tensors as synth.host_inputs, drawn by the device twin of the generator."""
    dt = tdtype(w)
    T, H, E, F = w["T"], w["H"], w["E"], w["F"]
    s = w["w_std"]

    def gen(shape, tid, std):
        t = torch.empty(shape, dtype=dt, device="cuda")
        return synth.device_normal(t, seed, tid, std)

    d = {"x": gen((T, H), synth.X, 1.0), "w_router": gen((E, H), synth.W_ROUTER, s),
         "w_gate": gen((E, F, H), synth.W_GATE, s), "w_up": gen((E, F, H), synth.W_UP, s),
         "w_down": gen((E, H, F), synth.W_DOWN, s)}
    d["router_bias"] = up(synth.zipf_bias(seed, E)) if w["zipf"] else None
    if w["n_shared"]:
        Fs = w["F_shared"]
        d["ws_gate"] = gen((Fs, H), synth.WS_GATE, s)
        d["ws_up"] = gen((Fs, H), synth.WS_UP, s)
        d["ws_down"] = gen((H, Fs), synth.WS_DOWN, s)
    return _attach_fp8(w, d)


def weights_arg(d: dict) -> dict:
    return {k: d.get(k) for k in ("w_router", "router_bias", "w_gate", "w_up", "w_down", "s_gate",
                                  "s_up", "s_down", "ws_gate", "ws_up", "ws_down", "ss_gate",
                                  "ss_up", "ss_down")}


def alloc(w: dict) -> dict:
    """Buffers of the staged calls."""
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    R = T * k
    rows = R + (T if w["n_shared"] else 0)
    dt = tdtype(w)
    fp8 = w["xfer_dtype"] == synth.E4M3
    mx = w["xfer_dtype"] == synth.MXE4M3
    xdt = torch.uint8 if (fp8 or mx) else dt
    cfg = cfg_of(w)

    def mx_sf(K):  # filled with 0xFF (NaN scales): a read of an unwritten slot shows
        return torch.full((moe.moe_mx_scale_bytes(cfg, K),), 0xFF, dtype=torch.uint8, device="cuda")

    b = {
        "cfg": cfg,
        "ws": torch.zeros(max(moe.moe_workspace_size(cfg), 256) // 4 + 64, dtype=torch.int32, device="cuda"),
        "logits": torch.empty((T, E), dtype=torch.float32, device="cuda"),
        "topk_idx": torch.empty((T, k), dtype=torch.int32, device="cuda"),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
        "counts": torch.empty(E, dtype=torch.int32, device="cuda"),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device="cuda"),
        "row_token": torch.empty(R, dtype=torch.int32, device="cuda"),
        "tok_row": torch.empty((T, k), dtype=torch.int32, device="cuda"),
        "xd": torch.empty((rows, H), dtype=xdt, device="cuda"),
        "xd_scale": torch.empty((H // 128, rows), dtype=torch.float32, device="cuda") if fp8 else (
            mx_sf(H) if mx else None),
        "h": torch.empty((rows, F), dtype=xdt, device="cuda"),
        "h_scale": torch.empty((F // 128, rows), dtype=torch.float32, device="cuda") if fp8 else (
            mx_sf(F) if mx else None),
        "yd": torch.empty((rows, H), dtype=dt, device="cuda"),
        "y": torch.empty((T, H), dtype=dt, device="cuda"),
    }
    moe.moe_workspace_init(b["ws"])
    return b


def run_staged(w: dict, d: dict, b: dict, logits: torch.Tensor | None = None):
    """S0..S7 through the staged entry points. With ``logits`` given, S0 is skipped and the
    routing uses those scores."""
    cfg = b["cfg"]
    if logits is None:
        moe.moe_router_logits(cfg, d["x"], d["w_router"], d["router_bias"], b["logits"], b["ws"])
        logits = b["logits"]
    moe.moe_route(cfg, logits, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    if w["xfer_dtype"] == synth.MXE4M3:
        moe.moe_dispatch_mx(cfg, d["x"], b["topk_idx"], b["tok_row"], b["offsets"], b["xd"], b["xd_scale"])
    else:
        moe.moe_dispatch(cfg, d["x"], b["tok_row"], b["xd"], b["xd_scale"])
    moe.moe_grouped_mlp(cfg, b["xd"], b["xd_scale"], d["x"], b["offsets"], weights_arg(d),
                        b["h"], b["h_scale"], b["yd"], b["ws"])
    moe.moe_combine(cfg, b["yd"], b["tok_row"], b["topk_w"], b["y"])
    return b


def run_forward(w: dict, d: dict):
    cfg = cfg_of(w)
    ws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(ws)
    T, k, E = w["T"], w["k"], w["E"]
    y = torch.empty((T, w["H"]), dtype=tdtype(w), device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    moe.moe_forward(cfg, d["x"], weights_arg(d), y, ws, idx, wt, cnt)
    return y, idx, wt, cnt, ws


def np_of(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


# ---------------------------------------------------------------- exact router inputs
# The router GEMM sums H products in an order each kernel chooses. With x on a 1/16 grid
# and the router weight on a 2^-10 grid, every product is a multiple of 2^-14; if in
# addition sum_h |x_h| |w_eh| <= 2^10 for a token and expert, every partial sum, in any
# order or grouping, is a multiple of 2^-14 below 2^10 in magnitude, which fp32's 24-bit
# significand holds exactly. The logit is then exact before the bias, the bias is added
# once with one rounding on both sides, and the GPU's fp32 logits equal the oracle's
# (fp64, rounded once) bit for bit: the routing of both sides is decided by identical
# scores, and no GPU result is handed to the oracle.
X_GRID, W_GRID, SUM_BOUND = 16.0, 1024.0, 1024.0


def grid_x(x: np.ndarray) -> np.ndarray:
    return (np.round(np.asarray(x, dtype=np.float32) * np.float32(X_GRID)) / np.float32(X_GRID)).astype(np.float32)


def grid_w_router(wr: np.ndarray) -> np.ndarray:
    return (np.round(np.asarray(wr, dtype=np.float32) * np.float32(W_GRID)) / np.float32(W_GRID)).astype(np.float32)


def assert_exact_router_sums(x: np.ndarray, wr: np.ndarray) -> None:
    """The precondition above, on the host, for the given tokens."""
    b = np.abs(np.asarray(x, dtype=np.float64)) @ np.abs(np.asarray(wr, dtype=np.float64)).T
    assert b.max() <= SUM_BOUND, b.max()


def exact_router_inputs(inp: dict) -> dict:
    """A copy of a layer's host inputs with x and the router weight on the grids above (x
    keeps its N(0,1) shape, rounded to multiples of 1/16; the weight its N(0, 0.02^2) shape,
    rounded to multiples of 2^-10; both stay exact in bf16)."""
    out = dict(inp)
    out["x"] = grid_x(inp["x"])
    out["w_router"] = grid_w_router(inp["w_router"])
    assert_exact_router_sums(out["x"], out["w_router"])
    return out


def grid_device_(t: torch.Tensor, grid: float) -> torch.Tensor:
    """The same rounding on a device tensor, in place (scaling by a power of two is exact,
    and both numpy and torch round half to even)."""
    return t.mul_(grid).round_().div_(grid)

