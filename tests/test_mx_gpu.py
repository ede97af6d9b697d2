"""The MXFP8 variant on the GPU against the oracle: the offline weight quantiser and the
MX dispatch bit for bit (e4m3 payload and UE8M0 scale codes, read back from the scale
atoms through the layout the C header documents), the grouped MLP on the block-scaled
tensor-core MMA within the FP8 tolerance, on sizes that span several tiles, K-stage ring
wraps, ragged segment tails, empty and hot experts and the shared expert."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import (alloc, device_weights_from_host, mx_atom_offsets, mx_grouped_rows, mx_weight_rows, np_of,
                      quantize_mx_dev, up, weights_arg)

pytestmark = pytest.mark.gpu

MX = synth.WORKLOADS["dsv3_mxfp8"]
TOL = 3e-2  # the FP8 variants' rel-L2 bound against the quantisation-mirroring oracle

CASES = [
    # ragged tails, shared expert, group-limited routing
    synth.scaled(MX, T=300, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2, name="mx_small"),
    # 8 K stages in GEMM1 and 5 in GEMM2 (the 4-stage ring wraps), several M tiles per expert
    synth.scaled(MX, T=700, H=1024, E=8, k=2, F=640, F_shared=640, n_groups=2, topk_groups=1, name="mx_deep_k"),
    # hot and empty experts (Zipf-biased logits), no shared expert
    synth.scaled(MX, T=600, H=256, E=32, k=4, F=128, n_shared=0, F_shared=0, n_groups=1, topk_groups=1,
                 score_fn=synth.SOFTMAX, renorm=0, zipf=True, name="mx_imbalanced"),
    # >= 512 rows per expert on average: 256-row CTA-pair tiles, ragged pair tails, shared expert
    synth.scaled(MX, T=1100, H=512, E=4, k=2, F=384, F_shared=384, n_groups=2, topk_groups=1, name="mx_pair"),
]


def logits_for(w, seed):
    l = synth.synthetic_logits(seed, w["T"], w["E"])
    if w["zipf"]:
        l = (l + 4.0 * synth.zipf_bias(seed, w["E"])).astype(np.float32)
    return l


def routing(w, seed):
    idx, wt = oracle.route(logits_for(w, seed), w)
    return idx, wt, oracle.permute(idx, w["E"])


def act_rows(w, offsets):
    return mx_grouped_rows(offsets, w["T"], w["k"], w["E"], bool(w["n_shared"]))


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (384, 1024), (2048, 7168)])
def test_quantize_mx_bit_exact(shape):
    v = synth.normal(5, 78, shape, 0.02, "bf16")
    v[0, :64] = 0.0                        # all-zero blocks: code 0, payload 0
    v[1, :32] *= np.float32(2.0 ** 60)     # far from the centre of the scale range
    v[2, 32:64] *= np.float32(2.0 ** -60)
    q, sf = quantize_mx_dev(up(v, torch.bfloat16))
    qo, so = oracle.mx_quant(v)
    assert np.array_equal(np_of(q), qo)
    a, i = mx_weight_rows(shape[0])
    assert np.array_equal(np_of(sf)[mx_atom_offsets(a, i, shape[1])], so)


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_dispatch_mx_bit_exact(w):
    T, H, k = w["T"], w["H"], w["k"]
    idx, _, (counts, offsets, row_token, tok_row) = routing(w, 3)
    if w["zipf"]:
        assert (counts == 0).any()
    x = synth.normal(0, synth.X, (T, H), 1.0, "bf16")
    x[5, :64] = 0.0
    x[6, 100] = 8192.0
    b = alloc(w)
    moe.moe_dispatch_mx(b["cfg"], up(x, torch.bfloat16), up(idx), up(tok_row), up(offsets), b["xd"],
                        b["xd_scale"])
    q, s = oracle.mx_quant(x)
    R = T * k
    rows = np.concatenate([row_token, np.arange(T)]) if w["n_shared"] else row_token
    assert np.array_equal(np_of(b["xd"])[:len(rows)], q[rows])
    sf = np_of(b["xd_scale"])
    pos = mx_atom_offsets(*act_rows(w, offsets), H)
    assert np.array_equal(sf[pos], s[rows])
    # nothing else in the atom buffer was written (it was filled with 0xFF)
    untouched = np.ones(sf.size, dtype=bool)
    untouched[pos.ravel()] = False
    assert np.all(sf[untouched] == 0xFF)
    assert pos.size == R * (H // 32) + (T * H // 32 if w["n_shared"] else 0)


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_grouped_mlp_mx_against_oracle(w):
    seed = 4
    T, H, k = w["T"], w["H"], w["k"]
    R = T * k
    inp = synth.host_inputs(w, seed=seed)
    idx, wt, (counts, offsets, row_token, tok_row) = routing(w, seed)
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    # A operand and its scale atoms from the oracle's quantisation of x
    q, s = oracle.mx_quant(inp["x"])
    rows = np.concatenate([row_token, np.arange(T)]) if w["n_shared"] else row_token
    b["xd"].copy_(up(q[rows]))
    sf = np_of(b["xd_scale"]).copy()
    sf[mx_atom_offsets(*act_rows(w, offsets), H)] = s[rows]
    b["xd_scale"].copy_(up(sf))
    moe.moe_grouped_mlp(b["cfg"], b["xd"], b["xd_scale"], d["x"], up(offsets), weights_arg(d), b["h"],
                        b["h_scale"], b["yd"], b["ws"])
    ref = oracle.forward(w, inp, logits=logits_for(w, seed))
    assert np.array_equal(ref["offsets"], offsets)
    got = np_of(b["yd"]).astype(np.float64)
    assert np.all(np.isfinite(got))
    assert oracle.rel_l2(got[:R], ref["yd"]) < TOL
    for e in range(w["E"]):  # every expert segment on its own (ragged tails included)
        r0, r1 = offsets[e], offsets[e + 1]
        if r1 > r0:
            assert oracle.rel_l2(got[r0:r1], ref["yd"][r0:r1]) < TOL, e
    if w["n_shared"]:
        assert oracle.rel_l2(got[R:], ref["ys"]) < TOL
    # h's scale atoms: every live row's codes written, the rest untouched
    hs = np_of(b["h_scale"])
    pos = mx_atom_offsets(*act_rows(w, offsets), w["F"])
    untouched = np.ones(hs.size, dtype=bool)
    untouched[pos.ravel()] = False
    assert np.all(hs[untouched] == 0xFF)
    assert np.all(hs[pos] != 0xFF)
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
