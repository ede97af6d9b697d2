"""S3 dispatch and S7 combine on the GPU against the oracle (bit-exact dispatch payloads and
FP8 scales; combine within fp32 accumulation / one output rounding), the identity-expert
round trip k*x, and the offline e4m3 block quantiser."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import alloc, cfg_of, np_of, up

pytestmark = pytest.mark.gpu


def routed(w, seed=0):
    l = synth.synthetic_logits(seed, w["T"], w["E"])
    idx, wt = oracle.route(l, w)
    return (idx, wt) + oracle.permute(idx, w["E"])


CASES = [
    synth.scaled(synth.WORKLOADS["tiny_fp32"], name="tiny"),
    synth.scaled(synth.WORKLOADS["mixtral_bf16"], T=1000, name="mixtral_h4096"),
    synth.scaled(synth.WORKLOADS["dsv3_bf16"], T=700, name="dsv3_h7168_shared"),
    synth.scaled(synth.WORKLOADS["imbalanced_bf16"], T=2048, name="imbalanced_h2048"),
]


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_dispatch_bit_exact(w):
    idx, _, counts, offsets, row_token, tok_row = routed(w)
    x = synth.normal(0, synth.X, (w["T"], w["H"]), 1.0, synth.act_name(w))
    b = alloc(w)
    dt = torch.bfloat16 if w["act_dtype"] == synth.BF16 else torch.float32
    moe.moe_dispatch(b["cfg"], up(x, dt), up(tok_row), b["xd"], None)
    R = w["T"] * w["k"]
    got = np_of(b["xd"][:R])
    assert np.array_equal(got, oracle.dispatch(x, row_token))


@pytest.mark.parametrize("T,shared", [(300, 1), (513, 0), (4096, 1)])
def test_dispatch_e4m3_bit_exact(T, shared):
    w = synth.scaled(synth.WORKLOADS["dsv3_fp8"], T=T, n_shared=shared)
    idx, _, counts, offsets, row_token, tok_row = routed(w)
    x = synth.normal(0, synth.X, (T, w["H"]), 1.0, "bf16")
    x[5, :128] = 0.0  # an all-zero block: scale 1, codes 0
    x[6, 200] = 8192.0  # a large value: it becomes its block's 448, the rest shrink
    b = alloc(w)
    moe.moe_dispatch(b["cfg"], up(x, torch.bfloat16), up(tok_row), b["xd"], b["xd_scale"])
    q, s = oracle.quant_blocks(x, 1, 128)
    R = T * w["k"]
    xd = np_of(b["xd"])
    sc = np_of(b["xd_scale"])  # [H/128, rows]
    assert np.array_equal(xd[:R], q[row_token])
    assert np.array_equal(sc[:, :R].T, s[row_token])
    if shared:
        assert np.array_equal(xd[R:], q)
        assert np.array_equal(sc[:, R:].T, s)


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_dispatch_combine_identity_experts_give_kx(w):
    idx, _, counts, offsets, row_token, tok_row = routed(w, seed=2)
    x = synth.normal(2, synth.X, (w["T"], w["H"]), 1.0, synth.act_name(w))
    dt = torch.bfloat16 if w["act_dtype"] == synth.BF16 else torch.float32
    b = alloc(w)
    moe.moe_dispatch(b["cfg"], up(x, dt), up(tok_row), b["xd"], None)
    R = w["T"] * w["k"]
    yd = b["yd"]
    yd[:R].copy_(b["xd"][:R])
    if w["n_shared"]:
        yd[R:].zero_()
    ones = torch.ones((w["T"], w["k"]), dtype=torch.float32, device="cuda")
    moe.moe_combine(b["cfg"], yd, up(tok_row), ones, b["y"])
    # sums of k <= 8 copies of a bf16 value are exact in fp32, and k is a power of two
    assert np.array_equal(np_of(b["y"]), (w["k"] * x).astype(np.float32))


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_combine_against_oracle(w):
    idx, wt, counts, offsets, row_token, tok_row = routed(w, seed=3)
    T, H, k = w["T"], w["H"], w["k"]
    rows = T * k + (T if w["n_shared"] else 0)
    yd = synth.normal(3, synth.YD, (rows, H), 1.0, synth.act_name(w))
    wts = (synth.uniform_at(3, synth.TOPK_W, np.arange(T * k)).reshape(T, k)).astype(np.float32)
    dt = torch.bfloat16 if w["act_dtype"] == synth.BF16 else torch.float32
    b = alloc(w)
    moe.moe_combine(b["cfg"], up(yd, dt), up(tok_row), up(wts), b["y"])
    ref = oracle.combine(yd[:T * k], tok_row, wts.astype(np.float64),
                         yd[T * k:] if w["n_shared"] else None)
    got = np_of(b["y"]).astype(np.float64)
    if w["act_dtype"] == synth.F32:
        assert oracle.rel_l2(got, ref) < 1e-6
    else:
        # fp32 accumulation, then one bf16 rounding (relative 2^-9)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


@pytest.mark.parametrize("shape,br,bc", [((512, 384), 128, 128), ((300, 1024), 1, 128),
                                         ((2048, 7168), 128, 128), ((130, 200), 128, 128)])
def test_quantize_e4m3_bit_exact(shape, br, bc):
    v = synth.normal(5, 77, shape, 0.02, "bf16")
    v[:2, :] = 0.0
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(((shape[0] + br - 1) // br, (shape[1] + bc - 1) // bc), dtype=torch.float32, device="cuda")
    moe.moe_quantize_e4m3(up(v, torch.bfloat16), br, bc, q, s)
    qo, so = oracle.quant_blocks(v, br, bc)
    assert np.array_equal(np_of(q), qo)
    assert np.array_equal(np_of(s), so)
