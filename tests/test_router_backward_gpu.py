"""The router's backward on the GPU against the oracle: the logit gradient through every
weight rule (softmax over all experts or over the chosen, sigmoid with or without
normalisation, group-limited choice, a routed scale), the auxiliary loss's gradient, the
router weight and bias gradients (token slices with a ragged last slice, ragged column
tiles, expert counts from one warp lane to sixteen), and the input gradient (the router's
share plus the dispatch backward's rows, shared expert included). Layers with E a
multiple of 128 and H of 256 take the tensor-core path (dl rounded to bf16 for the two products, a
ragged last 64-token K stage and 128- or 256-row dgrad tiles); the others the fp32 one.
Every input is seeded on the host; the oracle never sees a GPU result."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import np_of, up

pytestmark = pytest.mark.gpu


def rcfg(T, H, E, k, score_fn=0, renorm=0, n_groups=1, topk_groups=1, group_score=0, rho=1.0, act=synth.BF16,
         shared=0):
    return dict(T=T, H=H, E=E, k=k, F=256, n_shared=shared, F_shared=256 if shared else 0, score_fn=score_fn,
                renorm=renorm, n_groups=n_groups, topk_groups=topk_groups, group_score=group_score,
                routed_scale=rho, act_dtype=act, xfer_dtype=act)


def mcfg(c):
    return moe.MoEConfig.make(**c)


def tc_path(c):
    """The library's rule for the router's products on the tensor cores."""
    return (c["act_dtype"] == synth.BF16 and c["E"] % 128 == 0 and c["H"] % 256 == 0
            and c["k"] + c["n_shared"] + 1 <= 10)


def rws_of(cfg):
    ws = torch.zeros(moe.moe_router_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(ws)
    return ws


CASES = {
    # E = 8: one lane per expert row slot, slices of the weight gradient, 8-expert tiles
    "softmax_all_e8": rcfg(1000, 264, 8, 2),
    "softmax_topk_e16": rcfg(777, 512, 16, 4, renorm=1, rho=2.5),
    "sigmoid_e40": rcfg(513, 384, 40, 3, score_fn=1, rho=1.5),
    "sigmoid_groups_e256": rcfg(300, 1032, 256, 8, score_fn=1, renorm=1, n_groups=8, topk_groups=4, rho=2.5),
    "softmax_all_e512_fp32": rcfg(70, 136, 512, 6, act=synth.F32),
    "softmax_k_eq_e": rcfg(129, 128, 4, 4, renorm=1),
    # tensor-core path: 700 tokens = 10 K stages of 64 + 60; E = 512 two M tiles
    "tc_sigmoid_groups_e256": rcfg(700, 512, 256, 8, score_fn=1, renorm=1, n_groups=8, topk_groups=4, rho=2.5),
    "tc_softmax_all_e512": rcfg(300, 256, 512, 4),
    # 128 experts: the weight gradient as single-CTA 128-row tiles
    "tc_softmax_topk_e128": rcfg(450, 512, 128, 8, renorm=1),
}


def inputs(c, seed):
    T, H, E, k = c["T"], c["H"], c["E"], c["k"]
    logits = synth.synthetic_logits(seed, T, E)
    idx, _ = oracle.route(logits, c)
    dw = synth.normal(seed, 1, (T, k), 1.0, "f32")
    x = synth.normal(seed, 2, (T, H), 1.0, "bf16" if c["act_dtype"] == synth.BF16 else "f32")
    return logits, idx, dw, x


def run_router_backward(c, logits, idx, dw, x, counts=None, alpha=0.0, weight=True):
    T, H, E = c["T"], c["H"], c["E"]
    cfg = mcfg(c)
    xt = up(x, torch.bfloat16 if c["act_dtype"] == synth.BF16 else torch.float32)
    ws = rws_of(cfg)
    dl = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    dwr = torch.full((E, H), float("nan"), dtype=torch.float32, device="cuda") if weight else None
    db = torch.full((E,), float("nan"), dtype=torch.float32, device="cuda") if weight else None
    moe.moe_router_backward(cfg, up(logits), up(idx), up(dw), xt, dl, dwr, ws, d_router_bias=db,
                            counts=None if counts is None else up(counts.astype(np.int32)), aux_alpha=alpha)
    assert moe.moe_read_status(ws) == moe.MOE_OK
    return np_of(dl).astype(np.float64), (None if dwr is None else np_of(dwr).astype(np.float64)), (
        None if db is None else np_of(db).astype(np.float64))


@pytest.mark.parametrize("name", list(CASES))
def test_router_backward_against_oracle(name):
    c = CASES[name]
    logits, idx, dw, x = inputs(c, 40)
    dl, dwr, db = run_router_backward(c, logits, idx, dw, x)
    ref = oracle.router_backward(c, logits, idx, dw.astype(np.float64))
    assert oracle.rel_l2(dl, ref) < 1e-5
    assert np.abs(dl - ref).max() <= 1e-5 * np.abs(ref).max()
    if not (c["score_fn"] == 0 and c["renorm"] == 0):
        chosen = np.zeros(ref.shape, bool)
        np.put_along_axis(chosen, idx.astype(np.int64), True, axis=1)
        assert np.all(dl[~chosen] == 0.0)  # experts no weight depends on: exactly zero
    wref, _ = oracle.router_linear_backward(x, np.zeros((c["E"], c["H"])), ref)
    if tc_path(c):  # dl rounded to bf16 (relative 2^-8 per element), fp32 accumulation
        assert oracle.rel_l2(dwr, wref) < 8e-3
    else:
        assert oracle.rel_l2(dwr, wref) < 1e-5
        assert np.abs(dwr - wref).max() <= 1e-5 * np.abs(wref).max()
    assert np.allclose(db, ref.sum(axis=0), rtol=1e-4, atol=1e-5 * np.abs(ref.sum(axis=0)).max())


@pytest.mark.parametrize("score_fn", [0, 1])
def test_aux_loss_gradient_against_oracle(score_fn):
    """With a zero routing-weight gradient the logit gradient is the auxiliary loss's alone;
    with both, the two add."""
    c = rcfg(900, 256, 64, 6, score_fn=score_fn, renorm=1)
    logits, idx, dw, x = inputs(c, 41)
    counts = oracle.permute(idx, c["E"])[0]
    alpha = 0.01
    dl0, _, _ = run_router_backward(c, logits, idx, np.zeros_like(dw), x, counts=counts, alpha=alpha, weight=False)
    aux = oracle.aux_loss_backward(logits, counts, c["k"], score_fn, alpha)
    assert oracle.rel_l2(dl0, aux) < 1e-5
    dl, dwr, _ = run_router_backward(c, logits, idx, dw, x, counts=counts, alpha=alpha)
    ref = oracle.router_backward(c, logits, idx, dw.astype(np.float64)) + aux
    assert oracle.rel_l2(dl, ref) < 1e-5
    assert oracle.rel_l2(dwr, ref.T @ x.astype(np.float64)) < (8e-3 if tc_path(c) else 1e-5)


def test_router_backward_rejects_an_expert_id_out_of_range():
    c = CASES["softmax_topk_e16"]
    logits, idx, dw, x = inputs(c, 42)
    bad = idx.copy()
    bad[5, 1] = c["E"]
    cfg = mcfg(c)
    ws = rws_of(cfg)
    dl = torch.zeros((c["T"], c["E"]), dtype=torch.float32, device="cuda")
    moe.moe_router_backward(cfg, up(logits), up(bad), up(dw), None, dl, None, ws)
    assert moe.moe_read_status(ws) == moe.MOE_ERR_DEVICE_BAD_INPUT


IG_CASES = {
    "e8_k2": rcfg(200, 264, 8, 2),
    "e40_k3_shared": rcfg(333, 384, 40, 3, shared=1),
    "e256_k8_shared": rcfg(130, 1032, 256, 8, score_fn=1, renorm=1, shared=1),
    "one_token": rcfg(1, 128, 16, 2),
    # tensor-core path: 600 tokens as CTA-pair tiles (256 rows, ragged last), 130 as single
    # CTA tiles (128 rows + 2)
    "tc_e256_k8_shared": rcfg(600, 512, 256, 8, shared=1),
    "tc_e256_k2_few_tokens": rcfg(130, 256, 256, 2),
    "tc_e128_k8": rcfg(700, 512, 128, 8),
}


@pytest.mark.parametrize("name", list(IG_CASES))
@pytest.mark.parametrize("with_rows", [True, False], ids=["rows", "router_only"])
def test_dispatch_router_backward_against_oracle(name, with_rows):
    """dx = dl W_router (+ the rows' sum), one bf16 rounding of the fp32 sum: every element
    within the rounding (relative 2^-8) of the fp64 value plus a bound on the fp32 sum's
    own error; on the tensor-core path also two bf16 roundings of the router's share (dl,
    and dl W_router before the rows are added)."""
    c = IG_CASES[name]
    T, H, E, k = c["T"], c["H"], c["E"], c["k"]
    logits = synth.synthetic_logits(43, T, E)
    idx, _ = oracle.route(logits, c)
    _, _, _, tok_row = oracle.permute(idx, E)
    rows = T * k + (T if c["n_shared"] else 0)
    dl = synth.normal(43, 3, (T, E), 0.05, "f32")
    wr = synth.normal(43, 4, (E, H), 0.02, "bf16")
    dxd = synth.normal(43, 5, (rows, H), 1.0, "bf16")
    dx = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    cfg = mcfg(c)
    ws = rws_of(cfg)
    moe.moe_dispatch_router_backward(cfg, up(dxd, torch.bfloat16) if with_rows else None, up(tok_row), up(dl),
                                     up(wr, torch.bfloat16), dx, ws)
    assert moe.moe_read_status(ws) == moe.MOE_OK
    got = np_of(dx.float()).astype(np.float64)
    ref = dl.astype(np.float64) @ wr.astype(np.float64)
    mag = np.abs(dl.astype(np.float64)) @ np.abs(wr.astype(np.float64))
    mag_r = mag.copy()
    if with_rows:
        ref = ref + oracle.dispatch_backward(dxd, tok_row, bool(c["n_shared"]))
        mag = mag + oracle.dispatch_backward(np.abs(dxd), tok_row, bool(c["n_shared"]))
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * (E + k + 1) * mag + 1e-30
    if tc_path(c):
        bound += 2.0 ** -6 * mag_r
    assert np.all(np.abs(got - ref) <= bound), np.max(np.abs(got - ref) / bound)
