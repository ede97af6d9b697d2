"""Seeded synthetic inputs for the MoE layer forward (test and benchmark infrastructure).

This module holds the random-number recipe and the workload shapes, and none of the
layer's arithmetic. Both sides draw their inputs from here: the CPU oracle (through the
host generator below) and the CUDA path (through the same generator, or its device twin
in ``synth/gen.cu`` for tensors too large to build on the host).

Generator, written from the published definitions:
  * splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
    OOPSLA 2014; the constants are the ones of Vigna's public-domain splitmix64): element i
    of tensor ``tid`` under ``seed`` draws the 64-bit word
        key  = mix64((seed << 32) | tid)
        bits = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)          (mod 2^64)
  * Box-Muller (Box and Muller, 1958) in fp64 on the two 32-bit halves of ``bits``:
        u1 = (hi + 0.5) * 2^-32,  u2 = lo * 2^-32,
        z  = sqrt(-2 ln u1) * cos(2*pi*u2)
  * the value is ``z * std`` in fp64, rounded to nearest-even to fp32 and, for bf16
    tensors, rounded to nearest-even again to bf16.

Workload recipe (x ~ N(0,1), router and expert weights ~ N(0, 0.02^2), a Zipf(1.2) logit
bias for the imbalanced workload) follows the five synthetic layer shapes the method is
measured on: a tiny fp32 layer, a Mixtral-8x7B-shaped layer, a DeepSeek-V3-shaped layer, an
imbalanced-routing layer and an FP8-dispatch variant of the DeepSeek-V3 shapes.
"""
from __future__ import annotations

import math
import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
TWO_PI = 6.283185307179586  # fp64 nearest to 2*pi; the device twin uses the same literal

# Tensor ids: one independent stream per named tensor.
X, W_ROUTER, W_GATE, W_UP, W_DOWN, WS_GATE, WS_UP, WS_DOWN = 1, 2, 3, 4, 5, 6, 7, 8
LOGITS, ZIPF, TOPK_W, YD, ROUTER_BIAS = 9, 10, 11, 12, 13
DY = 14  # output gradient of the backward

_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = _mix64(np.array([((seed & 0xFFFFFFFF) << 32) | (tid & 0xFFFFFFFF)], dtype=np.uint64))
    return k[0]


def bits_at(seed: int, tid: int, idx: np.ndarray) -> np.ndarray:
    """64-bit words for flat element indices ``idx`` (uint64 array)."""
    key = stream_key(seed, tid)
    with np.errstate(over="ignore"):
        z = key + (idx.astype(np.uint64) + np.uint64(1)) * GOLDEN
        return _mix64(z)


def _normal_from_bits(b: np.ndarray) -> np.ndarray:
    hi = (b >> np.uint64(32)).astype(np.float64)
    lo = (b & np.uint64(0xFFFFFFFF)).astype(np.float64)
    u1 = (hi + 0.5) * (2.0 ** -32)
    u2 = lo * (2.0 ** -32)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even); returns the 16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(f32_to_bf16_bits(a))


_HOST = None


def _host_lib():
    """The C host generator (synth/gen_host.c), compiled on first use."""
    global _HOST
    if _HOST is None:
        import ctypes
        import os
        import subprocess
        here = os.path.dirname(os.path.abspath(__file__))
        src = os.path.join(here, "gen_host.c")
        out = os.path.join(here, "_build", "libsynth_host.so")
        os.makedirs(os.path.dirname(out), exist_ok=True)
        if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
            tmp = out + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
                                   "-fPIC", "-shared", "-o", tmp, src, "-lm"])
            os.replace(tmp, out)
        L = ctypes.CDLL(out)
        P = ctypes.c_void_p
        L.synth_normal_host.argtypes = [P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_uint32, ctypes.c_uint32, ctypes.c_double]
        L.synth_normal_host.restype = None
        _HOST = L
    return _HOST


def normal_at_numpy(seed: int, tid: int, idx: np.ndarray, std: float = 1.0, dtype: str = "f32") -> np.ndarray:
    """The recipe written out in numpy (slow; the definition the C generator is pinned to)."""
    idx = np.asarray(idx, dtype=np.uint64).ravel()
    out = np.empty(idx.size, dtype=np.float32)
    for s in range(0, idx.size, _CHUNK):
        z = _normal_from_bits(bits_at(seed, tid, idx[s:s + _CHUNK]))
        v = (z * std).astype(np.float32)
        out[s:s + _CHUNK] = round_bf16(v) if dtype == "bf16" else v
    return out


def normal_at(seed: int, tid: int, idx: np.ndarray, std: float = 1.0, dtype: str = "f32") -> np.ndarray:
    """Values of elements ``idx`` (flat, row-major) of tensor ``tid``; fp32 array holding
    exact fp32 (or exact bf16) values."""
    import ctypes
    idx = np.ascontiguousarray(np.asarray(idx).ravel(), dtype=np.int64)
    out = np.empty(idx.size, dtype=np.float32)
    _host_lib().synth_normal_host(out.ctypes.data_as(ctypes.c_void_p), idx.size,
                                  idx.ctypes.data_as(ctypes.c_void_p), 0, int(dtype == "bf16"),
                                  seed & 0xFFFFFFFF, tid & 0xFFFFFFFF, float(std))
    return out


def normal(seed: int, tid: int, shape, std: float = 1.0, dtype: str = "f32", offset: int = 0) -> np.ndarray:
    """Whole tensor of ``shape`` (flat index = row-major position + ``offset``)."""
    import ctypes
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _host_lib().synth_normal_host(out.ctypes.data_as(ctypes.c_void_p), n, None, offset,
                                  int(dtype == "bf16"), seed & 0xFFFFFFFF, tid & 0xFFFFFFFF, float(std))
    return out.reshape(shape)


def rows(seed: int, tid: int, row_ids, ncols: int, std: float = 1.0, dtype: str = "f32", base: int = 0) -> np.ndarray:
    """Selected rows of a row-major 2-D view with ``ncols`` columns starting at flat ``base``."""
    r = np.asarray(row_ids, dtype=np.uint64).reshape(-1, 1)
    idx = np.uint64(base) + r * np.uint64(ncols) + np.arange(ncols, dtype=np.uint64).reshape(1, -1)
    return normal_at(seed, tid, idx, std, dtype).reshape(len(row_ids), ncols)


def uniform_at(seed: int, tid: int, idx: np.ndarray) -> np.ndarray:
    """U[0,1) with 53-bit resolution from the same words (used for synthetic weights)."""
    b = bits_at(seed, tid, np.asarray(idx, dtype=np.uint64))
    return (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def zipf_bias(seed: int, E: int, alpha: float = 1.2) -> np.ndarray:
    """Per-expert additive logit bias b_e = -alpha * ln(r_e), r a seeded permutation of 1..E.

    ln of an unnormalised Zipf(alpha) weight r^-alpha; the normalising constant would cancel
    in both the softmax and the top-k, so it is left out. fp64, rounded once to fp32."""
    order = np.argsort(bits_at(seed, ZIPF, np.arange(E, dtype=np.uint64)), kind="stable")
    r = np.empty(E, dtype=np.float64)
    r[order] = np.arange(1, E + 1, dtype=np.float64)
    return (-alpha * np.log(r)).astype(np.float32)


# ----------------------------------------------------------------------------------------
# Workloads. Field names follow the layer's notation: T tokens, H hidden, E routed experts,
# k experts per token, F expert FFN width, optional shared expert of width F_shared,
# score function, renormalisation, G groups with g kept (group-limited routing).
# ----------------------------------------------------------------------------------------
F32, BF16, E4M3, MXE4M3 = 0, 1, 2, 3
SOFTMAX, SIGMOID = 0, 1


def workload(name, T, H, E, k, F, *, n_shared=0, F_shared=0, score_fn=SOFTMAX, renorm=0,
             n_groups=1, topk_groups=1, group_score=0, routed_scale=1.0, act=BF16, xfer=None,
             zipf=False, w_std=0.02):
    return dict(name=name, T=T, H=H, E=E, k=k, F=F, n_shared=n_shared, F_shared=F_shared,
                score_fn=score_fn, renorm=renorm, n_groups=n_groups, topk_groups=topk_groups,
                group_score=group_score, routed_scale=routed_scale, act_dtype=act,
                xfer_dtype=act if xfer is None else xfer, zipf=zipf, w_std=w_std)


WORKLOADS = {
    "tiny_fp32": workload("tiny_fp32", 256, 128, 8, 2, 256, act=F32),
    "mixtral_bf16": workload("mixtral_bf16", 4096, 4096, 8, 2, 14336, renorm=1),
    "dsv3_bf16": workload("dsv3_bf16", 8192, 7168, 256, 8, 2048, n_shared=1, F_shared=2048,
                          score_fn=SIGMOID, renorm=1, n_groups=8, topk_groups=4),
    "imbalanced_bf16": workload("imbalanced_bf16", 16384, 2048, 128, 8, 768, zipf=True),
    "dsv3_fp8": workload("dsv3_fp8", 32768, 7168, 256, 8, 2048, n_shared=1, F_shared=2048,
                         score_fn=SIGMOID, renorm=1, n_groups=8, topk_groups=4, xfer=E4M3),
    "dsv3_mxfp8": workload("dsv3_mxfp8", 32768, 7168, 256, 8, 2048, n_shared=1, F_shared=2048,
                           score_fn=SIGMOID, renorm=1, n_groups=8, topk_groups=4, xfer=MXE4M3),
}


def scaled(w: dict, **kw) -> dict:
    """A copy of workload ``w`` with some fields replaced (smaller parity cases)."""
    d = dict(w)
    d.update(kw)
    d["name"] = kw.get("name", w["name"] + "_small")
    return d


def act_name(w: dict) -> str:
    return "f32" if w["act_dtype"] == F32 else "bf16"


def host_inputs(w: dict, seed: int = 0, with_weights: bool = True) -> dict:
    """All layer inputs on the host as fp32 arrays of exact values (bf16-exact for bf16
    workloads). Weights are the unquantised N(0, w_std^2) draws."""
    dt = act_name(w)
    T, H, E, F = w["T"], w["H"], w["E"], w["F"]
    d = {"x": normal(seed, X, (T, H), 1.0, dt),
         "w_router": normal(seed, W_ROUTER, (E, H), w["w_std"], dt)}
    d["router_bias"] = zipf_bias(seed, E) if w["zipf"] else None
    if with_weights:
        d["w_gate"] = normal(seed, W_GATE, (E, F, H), w["w_std"], dt)
        d["w_up"] = normal(seed, W_UP, (E, F, H), w["w_std"], dt)
        d["w_down"] = normal(seed, W_DOWN, (E, H, F), w["w_std"], dt)
        if w["n_shared"]:
            Fs = w["F_shared"]
            d["ws_gate"] = normal(seed, WS_GATE, (Fs, H), w["w_std"], dt)
            d["ws_up"] = normal(seed, WS_UP, (Fs, H), w["w_std"], dt)
            d["ws_down"] = normal(seed, WS_DOWN, (H, Fs), w["w_std"], dt)
    return d


def expert_weights(w: dict, seed: int, e: int) -> tuple:
    """Host copy of one routed expert's (gate, up, down) weights, e in [0, E)."""
    dt = act_name(w)
    H, F = w["H"], w["F"]
    g = normal(seed, W_GATE, (F, H), w["w_std"], dt, offset=e * F * H)
    u = normal(seed, W_UP, (F, H), w["w_std"], dt, offset=e * F * H)
    d = normal(seed, W_DOWN, (H, F), w["w_std"], dt, offset=e * H * F)
    return g, u, d


def synthetic_logits(seed: int, T: int, E: int, std: float = 1.0, tie_levels: int = 0) -> np.ndarray:
    """fp32 router scores for routing-only tests. With ``tie_levels`` > 0 the values are
    snapped to that many distinct levels so equal keys (ties) are frequent."""
    l = normal(seed, LOGITS, (T, E), std, "f32")
    if tie_levels:
        l = (np.round(l * tie_levels / 4.0) * (4.0 / tie_levels)).astype(np.float32)
    return l


def gemm_flops(w: dict) -> float:
    """Algorithmic flops of the two expert GEMMs (routed + shared)."""
    T, H, k, F = w["T"], w["H"], w["k"], w["F"]
    f = 2.0 * T * k * H * (3 * F)
    if w["n_shared"]:
        f += 2.0 * T * H * (3 * w["F_shared"])
    return f


def describe(w: dict) -> str:
    return ", ".join(f"{k}={w[k]}" for k in ("T", "H", "E", "k", "F", "n_shared", "score_fn",
                                              "renorm", "n_groups", "topk_groups"))


# ----------------------------------------------------------------------------------------
# Device twin (synth/gen.cu) for tensors too large to draw on the host.
# ----------------------------------------------------------------------------------------
_DEV = None


def build_device(force: bool = False) -> str:
    import os
    import subprocess
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "gen.cu")
    out = os.path.join(here, "_build", "libsynth.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".{os.getpid()}.tmp"
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                               "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, src])
        os.replace(tmp, out)
    return out


def device_normal(t, seed: int, tid: int, std: float = 1.0, offset: int = 0):
    """Fill CUDA tensor ``t`` (float32 or bfloat16, contiguous) with the generator's values
    for flat indices offset .. offset + t.numel() - 1."""
    global _DEV
    import ctypes
    import torch
    if _DEV is None:
        L = ctypes.CDLL(build_device())
        L.synth_normal.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                                   ctypes.c_uint32, ctypes.c_double, ctypes.c_int64, ctypes.c_void_p]
        L.synth_normal.restype = ctypes.c_int
        _DEV = L
    assert t.is_cuda and t.is_contiguous() and t.dtype in (torch.float32, torch.bfloat16)
    rc = _DEV.synth_normal(t.data_ptr(), t.numel(), int(t.dtype == torch.bfloat16), seed, tid,
                           float(std), offset, torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_normal failed: CUDA error {rc}")
    return t
