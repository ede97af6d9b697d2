"""The backward (training step) on the GPU against the oracle's chain rule: combine
backward (row gradients and routing-weight gradients), the experts' grouped dgrad/wgrad
with the SwiGLU activation recomputed, and dispatch backward, on bf16 layers that span
several tiles, ragged segments, K tails of the weight-gradient reductions, empty and hot
experts, the shared expert and the CTA-pair form of the recomputed gate/up GEMM. The
routing is the oracle's (uploaded); the GPU runs its own forward on it."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import alloc, cfg_of, device_weights_from_host, np_of, up, weights_arg

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = [
    synth.scaled(W["mixtral_bf16"], T=600, H=512, E=4, F=512, name="mixtral_small"),
    synth.scaled(W["dsv3_bf16"], T=260, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2,
                 name="dsv3_small"),
    synth.scaled(W["imbalanced_bf16"], T=700, H=256, E=32, k=4, F=256, name="imbalanced_small"),
    # >= 512 rows per expert: the recomputed gate/up GEMM runs as CTA pairs
    synth.scaled(W["dsv3_bf16"], T=1200, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2, topk_groups=1,
                 name="pair_shared"),
    # 192..511 rows per expert: the recomputed gate/up GEMM on two or three m tiles per expert
    synth.scaled(W["dsv3_bf16"], T=520, H=512, E=16, F=256, F_shared=256, n_groups=4, topk_groups=2,
                 name="mid_shared"),
    # 256 experts: the router's products on the tensor cores (most experts get a few rows)
    synth.scaled(W["dsv3_bf16"], T=600, H=512, E=256, k=8, F=256, F_shared=256, n_groups=8, topk_groups=4,
                 name="e256_shared"),
    # CTA pairs whose segments (~530 rows) and shared expert (1060 rows) end in tails of at
    # most 64 rows: the forward's tokens-on-N tail tiles, with g and u kept for the backward
    synth.scaled(W["dsv3_bf16"], T=1060, H=512, E=4, k=2, F=256, F_shared=256, n_groups=2, topk_groups=1,
                 name="pair_tails"),
]
TOL = 1e-2  # bf16 layers


def logits_for(w, seed):
    l = synth.synthetic_logits(seed, w["T"], w["E"])
    if w["zipf"]:
        l = (l + 4.0 * synth.zipf_bias(seed, w["E"])).astype(np.float32)
    return l


def grads_alloc(w):
    E, H, F = w["E"], w["H"], w["F"]
    g = {"dw_gate": torch.empty((E, F, H), dtype=torch.float32, device="cuda"),
         "dw_up": torch.empty((E, F, H), dtype=torch.float32, device="cuda"),
         "dw_down": torch.empty((E, H, F), dtype=torch.float32, device="cuda")}
    if w["n_shared"]:
        g["dws_gate"] = torch.empty((F, H), dtype=torch.float32, device="cuda")
        g["dws_up"] = torch.empty((F, H), dtype=torch.float32, device="cuda")
        g["dws_down"] = torch.empty((H, F), dtype=torch.float32, device="cuda")
    return g


def run_staged_backward(w, d, b, dy):
    """GPU forward on the routing already in b, then the three staged backward calls."""
    cfg = b["cfg"]
    T, H, k = w["T"], w["H"], w["k"]
    rows = T * k + (T if w["n_shared"] else 0)
    moe.moe_dispatch(cfg, d["x"], b["tok_row"], b["xd"], None)
    moe.moe_grouped_mlp(cfg, b["xd"], None, d["x"], b["offsets"], weights_arg(d), b["h"], None, b["yd"], b["ws"])
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(bws)
    out = {"dyd": torch.empty((rows, H), dtype=torch.bfloat16, device="cuda"),
           "dtopk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
           "dxd": torch.empty((rows, H), dtype=torch.bfloat16, device="cuda"),
           "dx": torch.empty((T, H), dtype=torch.bfloat16, device="cuda")}
    g = grads_alloc(w)
    moe.moe_combine_backward(cfg, dy, b["yd"], b["tok_row"], b["topk_w"], out["dyd"], out["dtopk_w"])
    moe.moe_grouped_mlp_backward(cfg, b["xd"], d["x"], b["offsets"], weights_arg(d), out["dyd"], out["dxd"], g, bws)
    moe.moe_dispatch_backward(cfg, out["dxd"], b["tok_row"], out["dx"])
    out.update(g)
    assert moe.moe_read_status(bws) == moe.MOE_OK
    return out


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_backward_against_oracle(w):
    seed = 31
    T, H, E, k = w["T"], w["H"], w["E"], w["k"]
    R = T * k
    inp = synth.host_inputs(w, seed=seed)
    logits = logits_for(w, seed)
    ref_fwd = oracle.forward(w, inp, logits=logits)
    dy_h = synth.normal(seed, 50, (T, H), 1.0, "bf16")
    ref = oracle.backward(w, inp, ref_fwd, dy_h.astype(np.float64))
    counts = ref_fwd["counts"]
    if w["zipf"]:
        assert (counts == 0).any()
    d = device_weights_from_host(w, inp)
    b = alloc(w)
    b["topk_w"].copy_(up(ref_fwd["topk_w"].astype(np.float32)))
    b["offsets"].copy_(up(ref_fwd["offsets"]))
    b["tok_row"].copy_(up(ref_fwd["tok_row"]))
    got = run_staged_backward(w, d, b, up(dy_h, torch.bfloat16))
    # the router's backward on the same routing: dlogits, dW_router, and dx with both shares
    cfg = b["cfg"]
    rws = torch.zeros(moe.moe_router_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(rws)
    dl = torch.empty((T, E), dtype=torch.float32, device="cuda")
    dwr = torch.empty((E, H), dtype=torch.float32, device="cuda")
    moe.moe_router_backward(cfg, up(logits), up(ref_fwd["topk_idx"]), got["dtopk_w"], d["x"], dl, dwr, rws)
    dx_all = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch_router_backward(cfg, got["dxd"], b["tok_row"], dl, d["w_router"], dx_all, rws)
    assert moe.moe_read_status(rws) == moe.MOE_OK
    dl_ref = oracle.router_backward(w, logits, ref_fwd["topk_idx"], ref["dtopk_w"])
    dwr_ref, dxr_ref = oracle.router_linear_backward(inp["x"], inp["w_router"], dl_ref)
    assert oracle.rel_l2(np_of(dl).astype(np.float64), dl_ref) < TOL
    assert oracle.rel_l2(np_of(dwr).astype(np.float64), dwr_ref) < TOL
    assert oracle.rel_l2(np_of(dx_all.float()).astype(np.float64), ref["dx"] + dxr_ref) < TOL
    g = {key: np_of(v).astype(np.float64) for key, v in got.items()}
    assert oracle.rel_l2(g["dyd"], ref["dyd"]) < TOL
    assert oracle.rel_l2(g["dtopk_w"], ref["dtopk_w"]) < TOL
    assert oracle.rel_l2(g["dxd"], ref["dxd"]) < TOL
    assert oracle.rel_l2(g["dx"], ref["dx"]) < TOL
    off = ref_fwd["offsets"]
    for e in range(E):  # each expert's rows and weight gradients on their own
        if counts[e] == 0:
            for key in ("dw_gate", "dw_up", "dw_down"):
                assert not g[key][e].any(), (key, e)
            continue
        assert oracle.rel_l2(g["dxd"][off[e]:off[e + 1]], ref["dxd"][off[e]:off[e + 1]]) < TOL, e
        for key in ("dw_gate", "dw_up", "dw_down"):
            assert oracle.rel_l2(g[key][e], ref[key][e]) < TOL, (key, e)
    if w["n_shared"]:
        for key in ("dws_gate", "dws_up", "dws_down"):
            assert oracle.rel_l2(g[key], ref[key]) < TOL, key
        assert oracle.rel_l2(g["dxd"][R:], ref["dxd"][R:]) < TOL


@pytest.mark.parametrize("w", [CASES[1], CASES[3], CASES[4], CASES[5]],
                         ids=["dsv3_small", "pair_shared", "mid_shared", "e256_shared"])
def test_backward_after_forward_equals_staged(w):
    """moe_backward reads the routing, xd and yd from moe_forward's workspace and runs the
    same kernels as the staged calls: identical bits."""
    seed = 32
    T, H, E, k = w["T"], w["H"], w["E"], w["k"]
    inp = synth.host_inputs(w, seed=seed)
    d = device_weights_from_host(w, inp)
    cfg = cfg_of(w)
    fws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(fws)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_forward(cfg, d["x"], weights_arg(d), y, fws, idx, wt)
    dy = up(synth.normal(seed, 50, (T, H), 1.0, "bf16"), torch.bfloat16)
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(bws)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dtw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    g1 = grads_alloc(w)
    moe.moe_backward(cfg, d["x"], weights_arg(d), dy, fws, dx, dtw, g1, bws)
    assert moe.moe_read_status(bws) == moe.MOE_OK
    # with the router (and the auxiliary loss's gradient): dx gains the router's share
    dx_r = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    g2 = grads_alloc(w)
    g2.update(dw_router=torch.empty((E, H), dtype=torch.float32, device="cuda"),
              d_router_bias=torch.empty((E,), dtype=torch.float32, device="cuda"),
              dlogits=torch.empty((T, E), dtype=torch.float32, device="cuda"))
    moe.moe_backward(cfg, d["x"], weights_arg(d), dy, fws, dx_r, dtw, dict(g2, aux_loss_coeff=0.01), bws)
    assert moe.moe_read_status(bws) == moe.MOE_OK
    # staged, on the same routing (the permutation rebuilt from the forward's map)
    b = alloc(w)
    moe.moe_route_from_map(b["cfg"], idx, b["counts"], b["offsets"], b["row_token"], b["tok_row"], b["ws"])
    b["topk_w"].copy_(wt)
    got = run_staged_backward(w, d, b, dy)
    assert torch.equal(got["dx"], dx)
    assert torch.equal(got["dtopk_w"], dtw)
    for key in g1:
        assert torch.equal(got[key], g1[key]), key
        assert torch.equal(got[key], g2[key]), key
    # the router's staged calls on the forward's logits (moe_router_logits recomputes them)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(cfg, d["x"], d["w_router"], d.get("router_bias"), logits, b["ws"])
    rws = torch.zeros(moe.moe_router_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(rws)
    dl = torch.empty((T, E), dtype=torch.float32, device="cuda")
    dwr = torch.empty((E, H), dtype=torch.float32, device="cuda")
    db = torch.empty((E,), dtype=torch.float32, device="cuda")
    moe.moe_router_backward(cfg, logits, idx, got["dtopk_w"], d["x"], dl, dwr, rws, d_router_bias=db,
                            counts=b["counts"], aux_alpha=0.01)
    dx2 = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch_router_backward(cfg, got["dxd"], b["tok_row"], dl, d["w_router"], dx2, rws)
    assert moe.moe_read_status(rws) == moe.MOE_OK
    assert torch.equal(dl, g2["dlogits"])
    assert torch.equal(dwr, g2["dw_router"])
    assert torch.equal(db, g2["d_router_bias"])
    assert torch.equal(dx2, dx_r)
    assert not torch.equal(dx_r, dx)


@pytest.mark.parametrize("w", [CASES[0], CASES[2], CASES[3], CASES[5], CASES[6]],
                         ids=["mixtral_small", "imbalanced_small", "pair_shared", "e256_shared", "pair_tails"])
def test_forward_train_keeps_what_the_backward_recomputes(w):
    """moe_forward_train gives moe_forward's y and keeps g and u; moe_backward_kept on them
    gives moe_backward's every output bit for bit (the recomputed gate/up GEMM is the same
    GEMM), router and auxiliary loss included. g and u match the plain products xd Wg^T,
    xd Wu^T."""
    seed = 34
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    rows = T * k + (T if w["n_shared"] else 0)
    inp = synth.host_inputs(w, seed=seed)
    d = device_weights_from_host(w, inp)
    cfg = cfg_of(w)
    fws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(fws)
    y0 = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, d["x"], weights_arg(d), y0, fws)
    y1 = torch.empty_like(y0)
    gu = torch.full((rows, 2 * F), float("nan"), dtype=torch.bfloat16, device="cuda")
    aux = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_forward_train(cfg, d["x"], weights_arg(d), y1, fws, gu, aux_alpha=0.01, aux_loss=aux)
    assert moe.moe_read_status(fws) == moe.MOE_OK
    assert torch.equal(y0, y1)
    dy = up(synth.normal(seed, 50, (T, H), 1.0, "bf16"), torch.bfloat16)
    outs = []
    for kept in (False, True):
        bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
        moe.moe_workspace_init(bws)
        dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        dtw = torch.empty((T, k), dtype=torch.float32, device="cuda")
        g = grads_alloc(w)
        g.update(dw_router=torch.empty((E, H), dtype=torch.float32, device="cuda"),
                 dlogits=torch.empty((T, E), dtype=torch.float32, device="cuda"), aux_loss_coeff=0.01)
        if kept:
            moe.moe_backward_kept(cfg, d["x"], weights_arg(d), dy, fws, gu, dx, dtw, g, bws)
        else:
            moe.moe_backward(cfg, d["x"], weights_arg(d), dy, fws, dx, dtw, g, bws)
        assert moe.moe_read_status(bws) == moe.MOE_OK
        outs.append(dict(g, dx=dx, dtopk_w=dtw))
    for key, v in outs[0].items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(v, outs[1][key]), key
    # g and u of a few rows against the plain products (the routing read back from the forward)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    b = alloc(w)
    moe.moe_forward(cfg, d["x"], weights_arg(d), y0, fws, idx)
    moe.moe_route_from_map(b["cfg"], idx, b["counts"], b["offsets"], b["row_token"], b["tok_row"], b["ws"])
    # the auxiliary loss it returned is moe_aux_loss on the same logits and counts
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(cfg, d["x"], d["w_router"], d.get("router_bias"), logits, b["ws"])
    aux2 = torch.empty((1,), dtype=torch.float32, device="cuda")
    moe.moe_aux_loss(cfg, logits, b["counts"], 0.01, aux2, b["ws"])
    assert torch.equal(aux, aux2) and bool(torch.isfinite(aux).all())
    row_token = np_of(b["row_token"])
    offsets = np_of(b["offsets"])
    x64 = inp["x"].astype(np.float64)
    got = np_of(gu.float()).astype(np.float64)
    for r in np.linspace(0, rows - 1, 12).astype(int):
        if r < T * k:
            e = int(np.searchsorted(offsets, r, side="right") - 1)
            a, wg, wu = x64[row_token[r]], inp["w_gate"][e], inp["w_up"][e]
        else:
            a, wg, wu = x64[r - T * k], inp["ws_gate"], inp["ws_up"]
        gref, uref = wg.astype(np.float64) @ a, wu.astype(np.float64) @ a
        blocks = got[r].reshape(F // 128, 2, 128)
        assert oracle.rel_l2(blocks[:, 0].ravel(), gref) < 1e-2, r
        assert oracle.rel_l2(blocks[:, 1].ravel(), uref) < 1e-2, r


def test_training_step_replays_from_a_cuda_graph():
    """moe_forward_train + moe_backward_kept (router and auxiliary loss included) issue no
    host sync, so the whole training step captures into one CUDA graph; a replay gives the
    eager call's bits."""
    w = CASES[4]
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    rows = T * k + (T if w["n_shared"] else 0)
    inp = synth.host_inputs(w, seed=35)
    d = device_weights_from_host(w, inp)
    cfg = cfg_of(w)
    fws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(fws)
    moe.moe_workspace_init(bws)
    dy = up(synth.normal(35, 50, (T, H), 1.0, "bf16"), torch.bfloat16)

    def buffers():
        g = grads_alloc(w)
        g.update(dw_router=torch.empty((E, H), dtype=torch.float32, device="cuda"),
                 dlogits=torch.empty((T, E), dtype=torch.float32, device="cuda"), aux_loss_coeff=0.01)
        return dict(g, y=torch.empty((T, H), dtype=torch.bfloat16, device="cuda"),
                    gu=torch.empty((rows, 2 * F), dtype=torch.bfloat16, device="cuda"),
                    dx=torch.empty((T, H), dtype=torch.bfloat16, device="cuda"),
                    dtw=torch.empty((T, k), dtype=torch.float32, device="cuda"),
                    aux=torch.empty((1,), dtype=torch.float32, device="cuda"))

    def step(b):
        moe.moe_forward_train(cfg, d["x"], weights_arg(d), b["y"], fws, b["gu"], aux_alpha=0.01, aux_loss=b["aux"])
        moe.moe_backward_kept(cfg, d["x"], weights_arg(d), dy, fws, b["gu"], b["dx"], b["dtw"], b, bws)

    eager = buffers()
    step(eager)
    torch.cuda.synchronize()
    replayed = buffers()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(replayed)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    for v in replayed.values():
        if isinstance(v, torch.Tensor):
            v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(replayed)
    graph.replay()
    torch.cuda.synchronize()
    assert moe.moe_read_status(fws) == moe.MOE_OK and moe.moe_read_status(bws) == moe.MOE_OK
    for key, v in eager.items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(v, replayed[key]), key


def test_backward_no_tokens_gives_zero_weight_gradients():
    w = synth.scaled(CASES[1], T=0)
    cfg = cfg_of(w)
    inp = synth.host_inputs(synth.scaled(CASES[1], T=4), seed=33)
    d = device_weights_from_host(synth.scaled(CASES[1], T=4), inp)
    g = grads_alloc(w)
    g.update(dw_router=torch.empty((w["E"], w["H"]), dtype=torch.float32, device="cuda"),
             d_router_bias=torch.empty((w["E"],), dtype=torch.float32, device="cuda"))
    for v in g.values():
        v.fill_(7.0)
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_backward(cfg, None, weights_arg(d), None, None, None, None, g, bws)
    torch.cuda.synchronize()
    for key, v in g.items():
        assert not v.any(), key
    for v in g.values():
        v.fill_(7.0)
    moe.moe_backward_kept(cfg, None, weights_arg(d), None, None, None, None, None, g, bws)
    torch.cuda.synchronize()
    for key, v in g.items():
        assert not v.any(), key


@pytest.mark.parametrize("w", [
    synth.scaled(W["dsv3_bf16"], T=8192, H=256, E=256, F=256, F_shared=256, name="e256_t8192"),
    synth.scaled(W["imbalanced_bf16"], T=16384, H=256, E=128, F=256, name="imbalanced_t16384"),
], ids=["e256_t8192", "imbalanced_t16384"])
def test_forward_train_aux_loss_with_two_level_counts(w):
    """At these sizes the single routing launch has more than 8192 per-block counts, so it
    sums them in two levels (a scan down each expert's column, then a second grid barrier),
    and adds up the auxiliary loss's per-block sums in the same pass. The training forward's
    loss equals moe_aux_loss on the same logits and counts bit for bit, and its routing and
    output equal moe_forward's."""
    T, H, E, k = w["T"], w["H"], w["E"], w["k"]
    inp = synth.host_inputs(w, seed=41)
    d = device_weights_from_host(w, inp)
    cfg = cfg_of(w)
    assert moe.moe_route_launch_count(cfg) == 1
    fws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(fws)
    y0 = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    idx0 = torch.empty((T, k), dtype=torch.int32, device="cuda")
    moe.moe_forward(cfg, d["x"], weights_arg(d), y0, fws, idx0)
    y1 = torch.empty_like(y0)
    gu = torch.empty((T * k + (T if w["n_shared"] else 0), 2 * w["F"]), dtype=torch.bfloat16, device="cuda")
    aux = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_forward_train(cfg, d["x"], weights_arg(d), y1, fws, gu, aux_alpha=0.01, aux_loss=aux)
    assert moe.moe_read_status(fws) == moe.MOE_OK
    assert torch.equal(y0, y1)
    b = alloc(w)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    moe.moe_router_logits(cfg, d["x"], d["w_router"], d.get("router_bias"), logits, b["ws"])
    moe.moe_route(cfg, logits, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["row_token"],
                  b["tok_row"], b["ws"])
    assert torch.equal(b["topk_idx"], idx0)
    aux2 = torch.empty((1,), dtype=torch.float32, device="cuda")
    moe.moe_aux_loss(cfg, logits, b["counts"], 0.01, aux2, b["ws"])
    assert torch.equal(aux, aux2) and bool(torch.isfinite(aux).all())
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
