"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every entry
point that include/moe.h declares, and rejects invalid arguments on the host before any
CUDA call."""
import os
import re

import pytest

import token_routing_expert_router_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:moe_status_t|const char\*)\s+(moe_\w+)\(", text, re.M)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def test_header_declares_the_boundary():
    names = declared()
    for n in ("moe_route", "moe_route_from_map", "moe_dispatch", "moe_grouped_mlp", "moe_combine",
              "moe_forward", "moe_router_logits", "moe_read_status", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared():
        assert hasattr(L, n), n
    assert sorted(moe.exported_symbols()) == declared()


def test_no_symbol_outside_header(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", moe._build.LIB], capture_output=True, text=True).stdout
    exported = sorted({m for m in re.findall(r"\bT (moe_\w+)", out)})
    assert exported == declared()


def cfg(**kw):
    d = dict(T=64, H=128, E=8, k=2, F=256, act_dtype=moe.BF16)
    d.update(kw)
    return moe.MoEConfig.make(**d)


def test_workspace_sizes(L):
    c = cfg()
    assert moe.moe_workspace_size(c) >= 256
    assert moe.moe_forward_workspace_size(c) > moe.moe_workspace_size(c)


@pytest.mark.parametrize("kw,code", [
    (dict(k=9), moe.MOE_ERR_INVALID_ARG),
    (dict(E=6, n_groups=4, topk_groups=2, score_fn=moe.SIGMOID), moe.MOE_ERR_INVALID_ARG),
    (dict(n_groups=4, topk_groups=5), moe.MOE_ERR_INVALID_ARG),
    (dict(n_groups=4, topk_groups=2), moe.MOE_ERR_UNSUPPORTED),  # group limit needs sigmoid
    (dict(E=8, k=4, n_groups=4, topk_groups=1, score_fn=moe.SIGMOID), moe.MOE_ERR_INVALID_ARG),
    (dict(xfer_dtype=moe.E4M3, act_dtype=moe.F32), moe.MOE_ERR_UNSUPPORTED),
    (dict(xfer_dtype=moe.E4M3, H=200), moe.MOE_ERR_UNSUPPORTED),
    (dict(n_shared=1, F_shared=128), moe.MOE_ERR_UNSUPPORTED),
    (dict(H=100), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), moe.MOE_ERR_INVALID_ARG),
    (dict(k=33, E=64), moe.MOE_ERR_UNSUPPORTED),
])
def test_invalid_configs_rejected_on_host(L, kw, code):
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_workspace_size(cfg(**kw))
    assert ei.value.code == code


def test_null_and_misaligned_pointers_rejected_on_host(L):
    import ctypes
    c = cfg()
    P = ctypes.c_void_p
    assert L.moe_route(ctypes.byref(c), None, None, None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_dispatch(ctypes.byref(c), P(4096 + 8), P(4096), P(4096), None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(c), P(4096), None, P(4096), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(c), P(4096), P(4096), P(4096 + 4), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    # host-buffer forward: host pointers must be given, device staging 16-byte aligned
    assert L.moe_forward_host(ctypes.byref(c), None, None, P(4096), P(4096), P(4096), P(4096),
                              None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_host(ctypes.byref(c), P(4096), None, P(4096), P(4096 + 8), P(4096), P(4096),
                              None) == moe.MOE_ERR_INVALID_ARG
    # the routing-weight epilogue takes tok_row and topk_w together or not at all
    assert L.moe_grouped_mlp_gather(ctypes.byref(c), P(4096), P(4096), P(4096), P(4096), None, None, P(4096),
                                    P(4096), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, None, None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_read_status(None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_status_string(moe.MOE_ERR_TIMEOUT).startswith("device")


def test_variant_mismatches_rejected_on_host(L):
    """Calls for a variant the config does not describe, or shapes a kernel does not take,
    return their error before any launch."""
    import ctypes
    P = ctypes.c_void_p
    mx = cfg(H=256, xfer_dtype=moe.MXE4M3)
    bf = cfg(H=256)
    # MXFP8 dispatch has its own entry point, and it refuses other transfer types
    assert L.moe_dispatch(ctypes.byref(mx), P(4096), P(4096), P(4096), P(4096), None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_dispatch_mx(ctypes.byref(bf), P(4096), P(4096), P(4096), P(4096), P(4096), P(4096),
                             None) == moe.MOE_ERR_INVALID_ARG
    # the backward takes bf16 layers with H and F multiples of 256
    assert L.moe_combine_backward(ctypes.byref(cfg(act_dtype=moe.F32)), P(4096), P(4096), P(4096), P(4096),
                                  P(4096), P(4096), None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_mlp_backward(ctypes.byref(cfg(H=256, F=384)), P(4096), P(4096), P(4096), None, P(4096),
                                      P(4096), None, P(4096), None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_backward(ctypes.byref(cfg(H=256, xfer_dtype=moe.E4M3)), P(4096), None, P(4096), P(4096), P(4096),
                          P(4096), None, P(4096), None) == moe.MOE_ERR_UNSUPPORTED
    # quantisers: the MX one wants multiples of 128, the fp32-scale one 1 or 128 blocks
    assert L.moe_quantize_mx(P(4096), 100, 128, P(4096), P(4096), None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_quantize_mx(P(4096), -1, 128, P(4096), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_e4m3(P(4096), 128, 128, 64, 128, P(4096), P(4096), None) == moe.MOE_ERR_UNSUPPORTED


def test_router_backward_rejected_on_host(L):
    """The router backward's argument rules: the bias gradient only with the weight's, H a
    multiple of 8, 16-byte aligned buffers, a finite loss coefficient; the fused input
    gradient only for bf16 layers."""
    import ctypes
    P = ctypes.c_void_p
    c = cfg()
    rb = lambda cc, **kw: L.moe_router_backward(
        ctypes.byref(cc), kw.get("logits", P(4096)), P(4096), P(4096), kw.get("counts"),
        ctypes.c_float(kw.get("alpha", 0.0)), kw.get("x", P(4096)), kw.get("dl", P(4096)), kw.get("dw", P(4096)),
        kw.get("db"), P(4096), None)
    assert rb(c, dw=None, db=P(4096)) == moe.MOE_ERR_INVALID_ARG
    assert rb(c, x=None) == moe.MOE_ERR_INVALID_ARG
    assert rb(c, logits=P(4096 + 4)) == moe.MOE_ERR_INVALID_ARG
    assert rb(c, counts=P(4096 + 8)) == moe.MOE_ERR_INVALID_ARG
    assert rb(c, alpha=float("nan")) == moe.MOE_ERR_INVALID_ARG
    assert rb(c, dl=None) == moe.MOE_ERR_INVALID_ARG
    assert rb(cfg(H=100)) == moe.MOE_ERR_UNSUPPORTED
    ir = lambda cc, **kw: L.moe_dispatch_router_backward(ctypes.byref(cc), kw.get("dxd", P(4096)),
                                                         kw.get("tok_row", P(4096)), P(4096), P(4096), P(4096),
                                                         kw.get("ws", P(4096)), None)
    assert ir(cfg(act_dtype=moe.F32)) == moe.MOE_ERR_UNSUPPORTED
    assert ir(cfg(H=100)) == moe.MOE_ERR_UNSUPPORTED
    assert ir(c, tok_row=None) == moe.MOE_ERR_INVALID_ARG
    assert ir(c, dxd=P(4096 + 2)) == moe.MOE_ERR_INVALID_ARG
    assert ir(c, ws=None) == moe.MOE_ERR_INVALID_ARG
    # moe_backward: the router fields follow the same rules
    bf = cfg(H=256)
    g = moe.MoEWeightGrads.from_tensors({"dw_gate": 4096, "dw_up": 4096, "dw_down": 4096, "d_router_bias": 4096})
    w = moe.MoEWeights.from_tensors({"w_router": 4096, "w_gate": 4096, "w_up": 4096, "w_down": 4096})
    assert L.moe_backward(ctypes.byref(bf), P(4096), ctypes.byref(w), P(4096), P(4096), P(4096), P(4096),
                          ctypes.byref(g), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    # the training forward keeps g and u only for layers the backward takes, into an aligned buffer
    f0 = ctypes.c_float(0.0)
    assert L.moe_forward_train(ctypes.byref(cfg(act_dtype=moe.F32)), P(4096), ctypes.byref(w), P(4096), P(4096),
                               P(4096), f0, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_forward_train(ctypes.byref(bf), P(4096), ctypes.byref(w), P(4096), P(4096), P(4096 + 8), f0, None,
                               None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_train(ctypes.byref(bf), P(4096), ctypes.byref(w), P(4096), P(4096), P(4096),
                               ctypes.c_float(float("nan")), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    # no tokens: nothing to keep, no buffer is touched
    assert L.moe_forward_train(ctypes.byref(cfg(T=0, H=256)), None, ctypes.byref(w), None, None, None, f0, None,
                               None) == moe.MOE_OK
    g0 = moe.MoEWeightGrads.from_tensors({"dw_gate": 4096, "dw_up": 4096, "dw_down": 4096})
    assert L.moe_backward_kept(ctypes.byref(bf), P(4096), ctypes.byref(w), P(4096), P(4096), None, P(4096),
                               P(4096), ctypes.byref(g0), P(4096), None) == moe.MOE_ERR_INVALID_ARG
    # the router backward's workspace: the status head and S slices of [E, H] + [E] partials
    n = moe.moe_router_backward_workspace_size(c)
    assert n % 256 == 0 and n >= 256 + c.E * c.H * 4 + c.E * 4
    # many experts (tensor-core path): dl in bf16, the router's share of dx, and the K
    # split's per-slice partial sums (at most 255 slices of [E, H])
    big = cfg(T=1000, H=512, E=256, k=8)
    n = moe.moe_router_backward_workspace_size(big)
    base = 256 + 1000 * 256 * 2 + 1000 * 512 * 2
    assert base <= n < base + 255 * 256 * 512 * 4 + 64 * 1024
    assert moe.moe_backward_workspace_size(bf) > moe.moe_router_backward_workspace_size(bf)


@pytest.mark.parametrize("T,k,E,shared", [(64, 2, 8, 0), (300, 8, 16, 1), (1, 1, 4, 0), (0, 2, 8, 1)])
def test_mx_scale_bytes_follow_the_atom_layout(L, T, k, E, shared):
    """Each expert's rows start a fresh 128-row atom row (at ceil((offsets[e] + 127 e) / 128)),
    the shared expert's rows follow, and two spare atom rows close the buffer; every atom row
    holds one 512-byte atom per 128 columns."""
    c = cfg(T=T, k=k, E=E, H=256, xfer_dtype=moe.MXE4M3, n_shared=shared, F_shared=256 if shared else 0)
    rows = -(-(T * k + 127 * E) // 128) + (-(-T // 128) if shared else 0) + 2
    for K in (128, 256, 2048):
        assert moe.moe_mx_scale_bytes(c, K) == rows * (K // 128) * 512
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_mx_scale_bytes(c, 100)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED
