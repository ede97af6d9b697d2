"""The whole layer (moe_forward, S0..S7) on the GPU against the oracle's layer, which
computes its own router logits in fp64.

The layer's x and router weight are put on grids where the router GEMM is exact in fp32
whatever its summation order (see moe_case.exact_router_inputs), so the GPU's fp32 logits
equal the oracle's bit for bit. On identical scores the routing is unique: every token's
top-k must be the oracle's exactly, and the output is compared over all tokens, none
excluded. The router GEMM on unrounded inputs is checked in the router-logit tests."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import alloc, cfg_of, device_weights_from_host, exact_router_inputs, np_of, run_forward, run_staged

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = [
    synth.scaled(W["tiny_fp32"], name="tiny_fp32_full"),
    synth.scaled(W["mixtral_bf16"], T=512, H=512, F=512, name="mixtral_small"),
    synth.scaled(W["dsv3_bf16"], T=200, H=512, E=64, F=256, F_shared=256, name="dsv3_small"),
    synth.scaled(W["imbalanced_bf16"], T=1024, H=256, E=32, F=256, name="imbalanced_small"),
    synth.scaled(W["dsv3_fp8"], T=256, H=512, E=32, F=256, F_shared=256, name="fp8_small"),
    # >= 512 rows per expert on average: the 256-row CTA-pair tiles of the bf16 GEMMs
    synth.scaled(W["mixtral_bf16"], T=1100, H=512, E=4, F=384, name="pair_mixtral"),
    synth.scaled(W["imbalanced_bf16"], T=2100, H=256, E=8, k=2, F=256, name="pair_imbalanced"),
    synth.scaled(W["dsv3_bf16"], T=1200, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2,
                 topk_groups=1, name="pair_shared"),
    synth.scaled(W["dsv3_fp8"], T=1100, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2,
                 topk_groups=1, name="pair_fp8"),
    # single-CTA tiles with two or three m tiles per expert (192..511 rows per expert)
    synth.scaled(W["dsv3_bf16"], T=520, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2,
                 name="mid_dsv3"),
    synth.scaled(W["dsv3_mxfp8"], T=256, H=512, E=32, F=256, F_shared=256, name="mxfp8_small"),
    synth.scaled(W["dsv3_mxfp8"], T=900, H=1024, E=8, k=2, F=384, F_shared=384, n_groups=2,
                 topk_groups=1, name="mxfp8_deep_k"),
    synth.scaled(W["dsv3_mxfp8"], T=1300, H=768, E=4, k=2, F=640, F_shared=640, n_groups=2,
                 topk_groups=1, name="mxfp8_pair"),
    # degenerate layers: one token (a one-row tile per chosen expert), every expert chosen
    # by every token with H = 384 (down-projection tiles of 128 columns, 6 K blocks), and
    # the FP8 variants on one and three tokens
    synth.scaled(W["mixtral_bf16"], T=1, H=512, E=8, F=256, name="one_token"),
    synth.scaled(W["mixtral_bf16"], T=100, H=384, E=4, k=4, F=128, name="k_eq_e_h384"),
    synth.scaled(W["dsv3_fp8"], T=1, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2,
                 name="fp8_one_token"),
    synth.scaled(W["dsv3_mxfp8"], T=3, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2,
                 name="mxfp8_three_tokens"),
]


def tol(w):
    if w["xfer_dtype"] in (synth.E4M3, synth.MXE4M3):
        return 3e-2
    return 1e-5 if w["act_dtype"] == synth.F32 else 1e-2


def check_layer(w, inp, y, idx_gpu, logits_gpu):
    """S0 bit for bit, the routing of every token bit for bit, then the output of all tokens."""
    ref = oracle.forward(w, inp)
    assert np.array_equal(logits_gpu, ref["logits"])
    assert np.array_equal(idx_gpu, ref["topk_idx"]), np.nonzero(np.any(idx_gpu != ref["topk_idx"], 1))[0][:10]
    err = oracle.rel_l2(np_of(y).astype(np.float64), ref["y"])
    assert err < tol(w), err
    return err


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_forward_against_oracle(w):
    inp = exact_router_inputs(synth.host_inputs(w, seed=11))
    d = device_weights_from_host(w, inp)
    y, idx, wt, cnt, ws = run_forward(w, d)
    assert moe.moe_read_status(ws) == moe.MOE_OK
    b = alloc(w)
    moe.moe_router_logits(b["cfg"], d["x"], d["w_router"], d["router_bias"], b["logits"], b["ws"])
    check_layer(w, inp, y, np_of(idx), np_of(b["logits"]))
    c = np_of(cnt)
    assert c.sum() == w["T"] * w["k"]


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_staged_equals_forward(w):
    """The staged entry points and moe_forward run the same kernels: identical bits."""
    inp = synth.host_inputs(w, seed=12)
    d = device_weights_from_host(w, inp)
    y, idx, wt, cnt, _ = run_forward(w, d)
    b = run_staged(w, d, alloc(w))
    assert torch.equal(b["topk_idx"], idx)
    assert torch.equal(b["y"], y)


def test_forward_graph_capture():
    """moe_forward does no host sync, so the whole layer captures into one CUDA graph."""
    w = CASES[2]
    inp = synth.host_inputs(w, seed=13)
    d = device_weights_from_host(w, inp)
    y_ref, *_ = run_forward(w, d)
    cfg = cfg_of(w)
    ws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(ws)
    y = torch.empty_like(y_ref)
    from moe_case import weights_arg
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe.moe_forward(cfg, d["x"], weights_arg(d), y, ws)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_forward(cfg, d["x"], weights_arg(d), y, ws)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("w", [c for c in CASES if c["name"] in ("mixtral_small", "fp8_small", "mxfp8_small")],
                         ids=["mixtral_small", "fp8_small", "mxfp8_small"])
def test_forward_host_equals_forward(w):
    """moe_forward_host (host tokens in, host output back) gives the bits of moe_forward, also
    with two calls in flight on two streams, each with its own workspace and staging."""
    inp = synth.host_inputs(w, seed=14)
    d = device_weights_from_host(w, inp)
    y_ref, *_ = run_forward(w, d)
    from moe_case import weights_arg
    cfg = cfg_of(w)
    T, H = w["T"], w["H"]
    xh = d["x"].cpu().pin_memory()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for s in streams:
        ws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
        moe.moe_workspace_init(ws)
        yh = torch.full((T, H), 7, dtype=y_ref.dtype).pin_memory()
        outs.append((ws, torch.empty_like(d["x"]), torch.empty_like(y_ref), yh, s))
    torch.cuda.synchronize()
    for ws, xdev, ydev, yh, s in outs:
        moe.moe_forward_host(cfg, xh, weights_arg(d), yh, xdev, ydev, ws, stream=s)
    torch.cuda.synchronize()
    for ws, xdev, ydev, yh, s in outs:
        assert torch.equal(yh, y_ref.cpu())
        assert moe.moe_read_status(ws) == moe.MOE_OK
