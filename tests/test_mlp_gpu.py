"""S4-S6 (the grouped expert MLP) and S0 (router logits) on the GPU against the oracle, on
sizes the oracle finishes in seconds that still span several tiles, ragged segment tails,
empty and hot experts, and the shared expert."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import (alloc, assert_exact_router_sums, device_weights_from_host, grid_w_router, grid_x, np_of, tdtype, up,
                      weights_arg)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = [
    synth.scaled(W["tiny_fp32"], name="tiny_fp32"),
    # fp32 layers through the SIMT GEMMs: with a shared expert, and with F = 600 (a ragged last
    # N tile of the gate/up GEMM and a ragged last K step of the down projection)
    synth.scaled(W["tiny_fp32"], T=130, H=64, E=4, F=128, n_shared=1, F_shared=128, name="tiny_fp32_shared"),
    synth.scaled(W["tiny_fp32"], T=200, H=128, F=600, name="tiny_fp32_ragged_f"),
    # the narrowest rows the layer takes (H = 8: K = 8 in GEMM1, 8 output columns in GEMM2)
    synth.scaled(W["tiny_fp32"], T=70, H=8, E=4, F=24, name="tiny_fp32_narrow"),
    synth.scaled(W["mixtral_bf16"], T=600, H=512, F=384, name="mixtral_small"),
    synth.scaled(W["dsv3_bf16"], T=260, H=512, E=32, F=256, F_shared=256, name="dsv3_small"),
    synth.scaled(W["imbalanced_bf16"], T=700, H=256, E=32, k=4, F=384, name="imbalanced_small"),
    synth.scaled(W["dsv3_fp8"], T=300, H=512, E=16, F=256, F_shared=256, n_groups=4,
                 topk_groups=2, name="fp8_small"),
    # >= 512 rows per expert on average: the 256-row CTA-pair tiles of the bf16 GEMMs
    synth.scaled(W["mixtral_bf16"], T=1100, H=512, E=4, F=384, name="pair_mixtral"),
    synth.scaled(W["imbalanced_bf16"], T=2100, H=256, E=8, k=2, F=256, name="pair_imbalanced"),
    synth.scaled(W["dsv3_bf16"], T=1200, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2,
                 topk_groups=1, name="pair_shared"),
    synth.scaled(W["dsv3_fp8"], T=1100, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2,
                 topk_groups=1, name="pair_fp8"),
    # 192..511 rows per expert on average: single-CTA tiles, two or three m tiles per expert
    # (full 128-row tiles, M = 64 tails), hot and empty experts
    synth.scaled(W["dsv3_bf16"], T=520, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2,
                 name="mid_dsv3"),
    synth.scaled(W["mixtral_bf16"], T=1060, H=512, E=8, F=384, name="mid_mixtral"),
    synth.scaled(W["imbalanced_bf16"], T=800, H=256, E=16, k=4, F=256, name="mid_imbalanced"),
]


def tol(w):
    return {synth.F32: 1e-5, synth.BF16: 1e-2}[w["act_dtype"]] if w["xfer_dtype"] != synth.E4M3 else 3e-2


def logits_for(w, seed):
    l = synth.synthetic_logits(seed, w["T"], w["E"])
    if w["zipf"]:
        l = (l + 4.0 * synth.zipf_bias(seed, w["E"])).astype(np.float32)  # hot + empty experts
    return l


def routing(w, seed):
    idx, wt = oracle.route(logits_for(w, seed), w)
    return idx, wt, oracle.permute(idx, w["E"])


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_grouped_mlp_against_oracle(w):
    seed = 4
    inp = synth.host_inputs(w, seed=seed)
    idx, wt, (counts, offsets, row_token, tok_row) = routing(w, seed)
    if w["zipf"]:
        assert (counts == 0).any() and counts.max() > 3 * counts.mean()
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    fp8 = w["xfer_dtype"] == synth.E4M3
    T, H, k = w["T"], w["H"], w["k"]
    R = T * k
    if fp8:
        q, s = oracle.quant_blocks(inp["x"], 1, 128)
        rows = np.concatenate([row_token, np.arange(T)]) if w["n_shared"] else row_token
        b["xd"].copy_(up(q[rows]))
        b["xd_scale"].copy_(up(np.ascontiguousarray(s[rows].T)))
    else:
        xd = oracle.dispatch(inp["x"], row_token)
        b["xd"][:R].copy_(up(xd, tdtype(w)))
    moe.moe_grouped_mlp(b["cfg"], b["xd"], b["xd_scale"], d["x"], up(offsets), weights_arg(d),
                        b["h"], b["h_scale"], b["yd"], b["ws"])
    ref = oracle.forward(w, inp, logits=logits_for(w, seed))
    assert np.array_equal(ref["offsets"], offsets)
    got = np_of(b["yd"]).astype(np.float64)
    assert oracle.rel_l2(got[:R], ref["yd"]) < tol(w)
    for e in range(w["E"]):  # every expert segment on its own (ragged tails included)
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            assert oracle.rel_l2(got[r0:r1], ref["yd"][r0:r1]) < tol(w), e
    if w["n_shared"]:
        assert oracle.rel_l2(got[R:], ref["ys"]) < tol(w)
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK


# CTA-pair shapes (at least 512 rows per expert on average) with explicit segment sizes:
# tails of 1-64 rows (run with their tokens on the MMA's N axis), a whole expert of 64 rows,
# an empty expert, tails of 76 and more rows (ordinary tiles), and a shared expert whose
# 1060 rows end in a 36-row tail
TAIL_CASES = [
    (synth.scaled(W["dsv3_bf16"], T=1060, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2, topk_groups=1,
                  name="tails_shared"), [64, 300, 1035, 721]),
    (synth.scaled(W["mixtral_bf16"], T=1100, H=512, E=4, F=384, name="tails_empty_expert"), [0, 34, 1100, 1066]),
    (synth.scaled(W["mixtral_bf16"], T=1100, H=512, E=4, F=384, name="tails_tiny"), [1, 2, 17, 2180]),
]


@pytest.mark.parametrize("w,counts", TAIL_CASES, ids=[c[0]["name"] for c in TAIL_CASES])
def test_pair_segment_tails_against_oracle(w, counts):
    """Every expert segment, and separately the rows of its last (partial) 256-row tile,
    against the oracle's per-expert MLP, for segment sizes chosen to hit each tail form."""
    T, H, E, k = w["T"], w["H"], w["E"], w["k"]
    R = T * k
    assert sum(counts) == R and R >= 512 * E
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    seed = 12
    inp = synth.host_inputs(w, seed=seed)
    xd = synth.normal(seed + 1, synth.X, (R, H), 1.0, synth.act_name(w))
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    b["xd"][:R].copy_(up(xd, tdtype(w)))
    moe.moe_grouped_mlp(b["cfg"], b["xd"], None, d["x"], up(offsets), weights_arg(d), b["h"], None, b["yd"],
                        b["ws"])
    torch.cuda.synchronize()
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
    got = np_of(b["yd"]).astype(np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        ref = oracle.expert_mlp(xd[r0:r1], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e])
        assert oracle.rel_l2(got[r0:r1], ref) < 1e-2, e
        tail = (r1 - r0) % 256 or 256
        assert oracle.rel_l2(got[r1 - tail:r1], ref[-tail:]) < 1e-2, (e, tail)
    if w["n_shared"]:
        ref = oracle.expert_mlp(inp["x"], inp["ws_gate"], inp["ws_up"], inp["ws_down"])
        assert oracle.rel_l2(got[R:], ref) < 1e-2
        tail = T % 256
        assert oracle.rel_l2(got[R + T - tail:], ref[-tail:]) < 1e-2


ROUTER_CASES = [c for c in CASES if c["name"] in ("tiny_fp32", "mixtral_small", "dsv3_small", "imbalanced_small")]


@pytest.mark.parametrize("w", ROUTER_CASES, ids=[c["name"] for c in ROUTER_CASES])
def test_router_logits_against_oracle(w):
    inp = synth.host_inputs(w, seed=6, with_weights=False)
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    moe.moe_router_logits(b["cfg"], d["x"], d["w_router"], d["router_bias"], b["logits"], b["ws"])
    ref = oracle.router_logits(inp["x"], inp["w_router"], inp["router_bias"])
    assert oracle.rel_l2(np_of(b["logits"]), ref) < (1e-5 if w["act_dtype"] == synth.F32 else 1e-4)


@pytest.mark.parametrize("name,T,H,E", [("dsv3_router", 1000, 7168, 256), ("imb_router", 2000, 2048, 128),
                                        ("mixtral_router", 700, 4096, 8),
                                        # >= one 128-token tile per SM: 256-wide N tiles, ragged last tile
                                        ("dsv3_router_wide", 20000, 2048, 256)])
def test_router_logits_real_widths(name, T, H, E):
    w = synth.workload(name, T, H, E, 2, 128)
    inp = synth.host_inputs(w, seed=7, with_weights=False)
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    moe.moe_router_logits(b["cfg"], d["x"], d["w_router"], None, b["logits"], b["ws"])
    ref = oracle.router_logits(inp["x"], inp["w_router"], None)
    assert oracle.rel_l2(np_of(b["logits"]), ref) < 1e-4


@pytest.mark.parametrize("T,H,E", [(701, 2048, 5), (4096, 4096, 8), (333, 2048, 12), (130, 2048, 16),
                                   (1, 4096, 8), (3, 2048, 16), (257, 768, 24), (64, 1280, 32),
                                   (100, 7168, 8), (50, 768, 8), (333, 1280, 6), (2100, 512, 7)])
def test_router_logits_small_e_tensor_core_shapes(T, H, E):
    """The small-expert router on the tensor cores (bf16, E <= 32, H a multiple of 256):
    ragged last 16-token tiles, E below each 8-expert tile's width (1 to 4 tiles), a bias,
    and H whose 32-wide K steps split evenly over the warps (512 to 7168) or not (768, 1280:
    some warps get none). On the exact-sum grids every logit equals the oracle's bit for bit,
    whatever the summation order."""
    w = synth.workload("tc_router", T, H, E, 2, 128)
    inp = synth.host_inputs(w, seed=9, with_weights=False)
    x, wr = grid_x(inp["x"]), grid_w_router(inp["w_router"])
    assert_exact_router_sums(x, wr)
    bias = synth.zipf_bias(9, E)
    b = alloc(w)
    moe.moe_router_logits(b["cfg"], up(x, torch.bfloat16), up(wr, torch.bfloat16), up(bias), b["logits"], b["ws"])
    assert np.array_equal(np_of(b["logits"]), oracle.router_logits(x, wr, bias))


@pytest.mark.parametrize("T,H,E", [(100, 128, 48), (37, 8, 40), (300, 256, 64), (200, 248, 33), (90, 264, 48)])
def test_router_logits_fp32_simt_exact(T, H, E):
    """The fp32 router for more than 32 experts (SIMT): the small-problem form, which holds
    a tile's whole K in shared memory (K a multiple of 4 up to 256; here 8, 128, 248 and 256),
    and the 64 x 64 form (K = 264); ragged token tiles and expert columns, a bias. On the
    exact-sum grids every logit equals the oracle's bit for bit."""
    w = synth.workload("simt_router", T, H, E, 2, 128, act=synth.F32)
    inp = synth.host_inputs(w, seed=10, with_weights=False)
    x, wr = grid_x(inp["x"]), grid_w_router(inp["w_router"])
    assert_exact_router_sums(x, wr)
    bias = synth.zipf_bias(10, E)
    b = alloc(w)
    moe.moe_router_logits(b["cfg"], up(x), up(wr), up(bias), b["logits"], b["ws"])
    assert np.array_equal(np_of(b["logits"]), oracle.router_logits(x, wr, bias))


BF16_CASES = [c for c in CASES if c["act_dtype"] == synth.BF16 and c["xfer_dtype"] == synth.BF16]


@pytest.mark.parametrize("w", BF16_CASES, ids=[c["name"] for c in BF16_CASES])
def test_gathered_rows_equal_dispatched_rows(w):
    """The fused permutation: GEMM1 gathering its rows from x by token gives bit-identical h
    and yd to dispatch + grouped MLP on the dispatched copy."""
    seed = 5
    inp = synth.host_inputs(w, seed=seed)
    idx, wt, (counts, offsets, row_token, tok_row) = routing(w, seed)
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    moe.moe_dispatch(b["cfg"], d["x"], up(tok_row), b["xd"], None)
    moe.moe_grouped_mlp(b["cfg"], b["xd"], None, d["x"], up(offsets), weights_arg(d), b["h"], None,
                        b["yd"], b["ws"])
    h2, yd2 = torch.empty_like(b["h"]), torch.empty_like(b["yd"])
    moe.moe_grouped_mlp_gather(b["cfg"], d["x"], up(row_token), up(offsets), weights_arg(d), h2, yd2,
                               b["ws"])
    assert torch.equal(h2, b["h"])
    assert torch.equal(yd2, b["yd"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK


@pytest.mark.parametrize("w", BF16_CASES, ids=[c["name"] for c in BF16_CASES])
def test_routing_weight_in_down_projection_epilogue(w):
    """The other half of the fused permutation: GEMM2's epilogue scales each routed row by
    its routing weight before rounding, so that the combine is a plain sum. Each weighted
    routed row is within two bf16 roundings of the weight times the unweighted row, shared
    rows are untouched, and the unit-weight combine gives the layer output of the oracle."""
    seed = 6
    T, H, k = w["T"], w["H"], w["k"]
    R = T * k
    inp = synth.host_inputs(w, seed=seed)
    logits = logits_for(w, seed)
    idx, wt, (counts, offsets, row_token, tok_row) = routing(w, seed)
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    h1, yd1 = torch.empty_like(b["h"]), torch.empty_like(b["yd"])
    moe.moe_grouped_mlp_gather(b["cfg"], d["x"], up(row_token), up(offsets), weights_arg(d), h1, yd1, b["ws"])
    wt32 = wt.astype(np.float32)
    h2, yd2 = torch.empty_like(b["h"]), torch.empty_like(b["yd"])
    moe.moe_grouped_mlp_gather(b["cfg"], d["x"], up(row_token), up(offsets), weights_arg(d), h2, yd2, b["ws"],
                               tok_row=up(tok_row), topk_w=up(wt32))
    assert torch.equal(h2, h1)
    w_row = np.empty(R, dtype=np.float32)
    w_row[tok_row.ravel()] = wt32.ravel()
    u = np_of(yd1).astype(np.float64)
    g = np_of(yd2).astype(np.float64)
    expect = w_row[:, None].astype(np.float64) * u[:R]
    assert np.all(np.abs(g[:R] - expect) <= 2.0 ** -7 * 1.01 * np.abs(expect) + 1e-30)
    assert np.array_equal(g[R:], u[R:])
    y = torch.empty((T, H), dtype=tdtype(w), device="cuda")
    moe.moe_combine(b["cfg"], yd2, up(tok_row), None, y)
    ref = oracle.forward(w, inp, logits=logits)
    assert oracle.rel_l2(np_of(y).astype(np.float64), ref["y"]) < tol(w)
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
