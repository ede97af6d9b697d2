"""Parity at the workloads' full sizes, in the launch configuration the benchmark times
(moe_forward captured once in a CUDA graph and replayed), on outputs the oracle computes
one by one: sampled router-logit rows, sampled dispatched rows, sampled rows of sampled
experts' MLP outputs, sampled combined tokens, and the whole-layer output of sampled
tokens. Large weights are drawn on the GPU by the device twin of the generator; every
oracle input is redrawn on the host from the same counters (never read back from a GPU
result). x and the router weight are rounded, on both sides, to grids on which the router
GEMM is exact in fp32 (moe_case.exact_router_inputs), so the GPU's logits equal the
oracle's bit for bit, the routing is unique, and every sampled token is compared."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import (W_GRID, X_GRID, assert_exact_router_sums, cfg_of, device_weights_generated, grid_device_,
                      grid_w_router, grid_x, mx_atom_offsets, mx_grouped_rows, np_of, up, weights_arg)

pytestmark = pytest.mark.gpu

NAMES = ["mixtral_bf16", "dsv3_bf16", "imbalanced_bf16", "dsv3_fp8", "dsv3_mxfp8"]
SAMPLE_TOKENS = {"mixtral_bf16": 6, "dsv3_bf16": 4, "imbalanced_bf16": 8, "dsv3_fp8": 3, "dsv3_mxfp8": 3}


def qmode(w):
    """0 unquantised, 1 FP8 with fp32 block scales, 2 MXFP8 (the oracle's quant_h codes)."""
    return {synth.E4M3: 1, synth.MXE4M3: 2}.get(w["xfer_dtype"], 0)


def quant_act(a, mode):
    """The values the dispatched rows stand for, quantised by the oracle."""
    if mode == 1:
        return oracle.dequant_blocks(*oracle.quant_blocks(a, 1, 128), 1, 128)
    if mode == 2:
        return oracle.mx_dequant(*oracle.mx_quant(a))
    return a.astype(np.float64)


def quant_weight(m, mode):
    if mode == 1:
        return oracle.dequant_blocks(*oracle.quant_blocks(m, 128, 128), 128, 128)
    if mode == 2:
        return oracle.mx_dequant(*oracle.mx_quant(m))
    return m.astype(np.float64)


class Layer:
    """One full-size layer on the GPU: generated weights, one forward by graph replay."""

    def __init__(self, name):
        w = synth.WORKLOADS[name]
        self.w = w
        self.d = device_weights_generated(w, seed=0)
        for key in list(self.d):
            if key.endswith("_bf16"):
                del self.d[key]  # keep only what the layer reads
        grid_device_(self.d["x"], X_GRID)  # the exact-router grids, also applied by x_rows
        grid_device_(self.d["w_router"], W_GRID)
        cfg = cfg_of(w)
        self.cfg = cfg
        T, k, E, H = w["T"], w["k"], w["E"], w["H"]
        ws = torch.zeros(moe.moe_forward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
        moe.moe_workspace_init(ws)
        dt = torch.bfloat16 if w["act_dtype"] == synth.BF16 else torch.float32
        self.y = torch.empty((T, H), dtype=dt, device="cuda")
        self.idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        self.wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
        self.cnt = torch.empty(E, dtype=torch.int32, device="cuda")
        args = (cfg, self.d["x"], weights_arg(self.d), self.y, ws, self.idx, self.wt, self.cnt)
        moe.moe_forward(*args)  # warm-up outside the capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            moe.moe_forward(*args)
        self.y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_read_status(ws) == moe.MOE_OK
        self.logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        moe.moe_router_logits(cfg, self.d["x"], self.d["w_router"], self.d["router_bias"],
                              self.logits, ws)
        torch.cuda.synchronize()
        self.ws = ws


_CACHE = {}


def layer(name):
    if name not in _CACHE:
        _CACHE.clear()
        torch.cuda.empty_cache()
        _CACHE[name] = Layer(name)
    return _CACHE[name]


def sample_tokens(w, n, seed=5):
    T = w["T"]
    rng = synth.bits_at(seed, 90, np.arange(n, dtype=np.uint64)) % np.uint64(T)
    return np.unique(np.concatenate([[0, T - 1], rng.astype(np.int64)]))


def x_rows(w, toks, dt=None):
    """Host rows of the layer's x: the generator's rows on the exact-router grid."""
    return grid_x(synth.rows(0, synth.X, toks, w["H"], 1.0, dt or synth.act_name(w)))


def w_router_host(w):
    return grid_w_router(synth.normal(0, synth.W_ROUTER, (w["E"], w["H"]), w["w_std"], synth.act_name(w)))


def host_expert(w, e, mode):
    return tuple(quant_weight(m, mode) for m in synth.expert_weights(w, 0, e))


def host_shared(w, mode):
    H, Fs, s, dt = w["H"], w["F_shared"], w["w_std"], synth.act_name(w)
    mats = (synth.normal(0, synth.WS_GATE, (Fs, H), s, dt), synth.normal(0, synth.WS_UP, (Fs, H), s, dt),
            synth.normal(0, synth.WS_DOWN, (H, Fs), s, dt))
    return tuple(quant_weight(m, mode) for m in mats)


@pytest.mark.parametrize("name", NAMES)
def test_fullsize_generator_twin_and_router_logits(name):
    L = layer(name)
    w = L.w
    toks = sample_tokens(w, 16)
    xs = x_rows(w, toks)
    assert np.array_equal(np_of(L.d["x"][torch.from_numpy(toks).cuda()]), xs)  # device twin == host
    wr = w_router_host(w)
    assert np.array_equal(np_of(L.d["w_router"]), wr)
    assert_exact_router_sums(xs, wr)
    bias = synth.zipf_bias(0, w["E"]) if w["zipf"] else None
    ref = oracle.router_logits(xs, wr, bias)
    got = np_of(L.logits[torch.from_numpy(toks).cuda()])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("name", NAMES)
def test_fullsize_layer_sampled_tokens(name):
    L = layer(name)
    w = L.w
    mode = qmode(w)
    T, H, E, k = w["T"], w["H"], w["E"], w["k"]
    toks = sample_tokens(w, SAMPLE_TOKENS[name])
    counts = np_of(L.cnt)
    assert counts.sum() == T * k
    xs = x_rows(w, toks)
    wr = w_router_host(w)
    assert_exact_router_sums(xs, wr)
    bias = synth.zipf_bias(0, E) if w["zipf"] else None
    l_ref = oracle.router_logits(xs, wr, bias)
    idx_ref, wt_ref = oracle.route(l_ref, dict(w, T=len(toks)))
    assert np.array_equal(np_of(L.logits[torch.from_numpy(toks).cuda()]), l_ref)
    assert np.array_equal(np_of(L.idx)[toks], idx_ref)
    a = quant_act(xs, mode)
    y_ref = np.zeros((len(toks), H))
    for e in sorted(set(idx_ref.ravel().tolist())):
        mats = host_expert(w, e, mode)
        for i in range(len(toks)):
            for j in range(k):
                if idx_ref[i, j] == e:
                    y_ref[i] += wt_ref[i, j] * oracle.expert_mlp(a[i:i + 1], *mats, quant_h=mode)[0]
    if w["n_shared"]:
        y_ref += oracle.expert_mlp(a, *host_shared(w, mode), quant_h=mode)
    got = np_of(L.y)[toks].astype(np.float64)
    tol = 3e-2 if mode else 1e-2
    err = oracle.rel_l2(got, y_ref)
    assert err < tol, err


@pytest.mark.parametrize("name", ["dsv3_bf16", "dsv3_fp8", "dsv3_mxfp8"])
def test_fullsize_dispatch_and_expert_rows(name):
    """Dispatch of the full batch with the oracle's own routing of generator scores, then the
    grouped MLP on it; sampled rows of three experts and of the shared expert."""
    L = layer(name)
    w = L.w
    mode = qmode(w)
    fp8, mx = mode == 1, mode == 2
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    R = T * k
    rows = R + T
    l = synth.synthetic_logits(7, T, E)
    idx, wt = oracle.route(l, w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    xdt = torch.uint8 if mode else torch.bfloat16
    xd = torch.empty((rows, H), dtype=xdt, device="cuda")
    if mx:
        xs = torch.empty(moe.moe_mx_scale_bytes(L.cfg, H), dtype=torch.uint8, device="cuda")
        hs = torch.empty(moe.moe_mx_scale_bytes(L.cfg, F), dtype=torch.uint8, device="cuda")
        moe.moe_dispatch_mx(L.cfg, L.d["x"], up(idx), up(tok_row), up(offsets), xd, xs)
    else:
        xs = torch.empty((H // 128, rows), dtype=torch.float32, device="cuda") if fp8 else None
        hs = torch.empty((F // 128, rows), dtype=torch.float32, device="cuda") if fp8 else None
        moe.moe_dispatch(L.cfg, L.d["x"], up(tok_row), xd, xs)
    h = torch.empty((rows, F), dtype=xdt, device="cuda")
    yd = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_mlp(L.cfg, xd, xs, L.d["x"], up(offsets), weights_arg(L.d), h, hs, yd, L.ws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(L.ws) == moe.MOE_OK
    # sampled dispatched rows are bit-exact copies (or quantisations) of host-drawn tokens
    pick = np.unique(np.concatenate([[0, R - 1], (synth.bits_at(8, 91, np.arange(24, dtype=np.uint64)) % np.uint64(R)).astype(np.int64)]))
    xt = x_rows(w, row_token[pick], "bf16")
    if fp8:
        q, s = oracle.quant_blocks(xt, 1, 128)
        assert np.array_equal(np_of(xd[torch.from_numpy(pick).cuda()]), q)
        assert np.array_equal(np_of(xs[:, torch.from_numpy(pick).cuda()]).T, s)
    elif mx:
        q, s = oracle.mx_quant(xt)
        assert np.array_equal(np_of(xd[torch.from_numpy(pick).cuda()]), q)
        arow, irow = mx_grouped_rows(offsets, T, k, E, True)
        pos = mx_atom_offsets(arow[pick], irow[pick], H)
        assert np.array_equal(np_of(xs[torch.from_numpy(pos.ravel()).cuda()]).reshape(pos.shape), s)
    else:
        assert np.array_equal(np_of(xd[torch.from_numpy(pick).cuda()]), xt)
    # sampled rows of three experts (first, largest, last non-empty) and of the shared expert
    nz = np.nonzero(counts)[0]
    experts = sorted({int(nz[0]), int(np.argmax(counts)), int(nz[-1])})
    got_all = []
    ref_all = []
    for e in experts:
        r0, r1 = offsets[e], offsets[e + 1]
        rr = np.unique(np.array([r0, (r0 + r1) // 2, r1 - 1]))
        xa = quant_act(x_rows(w, row_token[rr], "bf16"), mode)
        ref_all.append(oracle.expert_mlp(xa, *host_expert(w, e, mode), quant_h=mode))
        got_all.append(np_of(yd[torch.from_numpy(rr).cuda()]))
    ts = np.array([0, T // 2, T - 1])
    xa = quant_act(x_rows(w, ts, "bf16"), mode)
    ref_all.append(oracle.expert_mlp(xa, *host_shared(w, mode), quant_h=mode))
    got_all.append(np_of(yd[torch.from_numpy(R + ts).cuda()]))
    got = np.concatenate(got_all).astype(np.float64)
    ref = np.concatenate(ref_all)
    assert oracle.rel_l2(got, ref) < (3e-2 if mode else 1e-2)


@pytest.mark.parametrize("name", ["mixtral_bf16", "dsv3_bf16"])
def test_fullsize_gathered_rows_equal_dispatched_rows(name):
    """The fused permutation at full size (CTA-pair TMA row gathers on the Mixtral shape,
    single-CTA cp.async gathers with routed/shared tile switches on the DeepSeek-V3 shape):
    GEMM1 gathering its rows from x by token gives h and yd bit-identical to dispatch +
    grouped MLP on the dispatched copy."""
    L = layer(name)
    w = L.w
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    R = T * k
    rows = R + (T if w["n_shared"] else 0)
    idx, _ = oracle.route(synth.synthetic_logits(11, T, E), w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    xd = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(L.cfg, L.d["x"], up(tok_row), xd, None)
    h1 = torch.empty((rows, F), dtype=torch.bfloat16, device="cuda")
    yd1 = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_mlp(L.cfg, xd, None, L.d["x"], up(offsets), weights_arg(L.d), h1, None, yd1, L.ws)
    del xd
    h2, yd2 = torch.empty_like(h1), torch.empty_like(yd1)
    moe.moe_grouped_mlp_gather(L.cfg, L.d["x"], up(row_token), up(offsets), weights_arg(L.d), h2, yd2, L.ws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(L.ws) == moe.MOE_OK
    assert torch.equal(h2, h1)
    assert torch.equal(yd2, yd1)


@pytest.mark.parametrize("name", ["dsv3_bf16", "imbalanced_bf16"])
def test_fullsize_combine_sampled(name):
    L = layer(name)
    w = L.w
    T, H, E, k = w["T"], w["H"], w["E"], w["k"]
    R = T * k
    rows = R + (T if w["n_shared"] else 0)
    idx, _ = oracle.route(synth.synthetic_logits(9, T, E), w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    yd = torch.empty((rows, H), dtype=torch.bfloat16, device="cuda")
    synth.device_normal(yd, 9, synth.YD, 1.0)
    wts = synth.uniform_at(9, synth.TOPK_W, np.arange(T * k)).reshape(T, k).astype(np.float32)
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    moe.moe_combine(L.cfg, yd, up(tok_row), up(wts), y)
    toks = sample_tokens(w, 12, seed=9)
    ref = np.zeros((len(toks), H))
    for i, t in enumerate(toks):
        r = tok_row[t]
        ydr = synth.rows(9, synth.YD, r, H, 1.0, "bf16").astype(np.float64)
        ref[i] = wts[t].astype(np.float64) @ ydr
        if w["n_shared"]:
            ref[i] += synth.rows(9, synth.YD, [R + t], H, 1.0, "bf16")[0]
    got = np_of(y[torch.from_numpy(toks).cuda()]).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


@pytest.mark.parametrize("name", ["mixtral_bf16", "dsv3_bf16"])
def test_fullsize_training_step_sampled_tokens(name):
    """The training step at full size, in the calls the benchmark times (moe_forward_train,
    then moe_backward_kept with the router's backward): for sampled tokens, routed by the
    oracle from the layer's own fp32 scores, dx (through the experts and through the router)
    and dlogits against the oracle's chain rule, token by token; and dW_router against its defining identity
    dl^T x on sampled experts (a property of the outputs at any size). dy is drawn on the
    GPU by the generator's device twin and redrawn on the host from the same counters."""
    L = layer(name)
    w, cfg, d = L.w, L.cfg, L.d
    T, H, E, k, F = w["T"], w["H"], w["E"], w["k"], w["F"]
    shared = bool(w["n_shared"])
    rows = T * k + (T if shared else 0)
    bf, f32 = dict(dtype=torch.bfloat16, device="cuda"), dict(dtype=torch.float32, device="cuda")
    gu = torch.empty((rows, 2 * F), **bf)
    y = torch.empty((T, H), **bf)
    moe.moe_forward_train(cfg, d["x"], weights_arg(d), y, L.ws, gu)
    dy = synth.device_normal(torch.empty((T, H), **bf), 0, synth.DY, 1.0)
    bws = torch.zeros(moe.moe_backward_workspace_size(cfg) // 4 + 64, dtype=torch.int32, device="cuda")
    moe.moe_workspace_init(bws)
    g = {"dw_gate": torch.empty((E, F, H), **f32), "dw_up": torch.empty((E, F, H), **f32),
         "dw_down": torch.empty((E, H, F), **f32), "dw_router": torch.empty((E, H), **f32),
         "dlogits": torch.empty((T, E), **f32)}
    if shared:
        Fs = w["F_shared"]
        g.update(dws_gate=torch.empty((Fs, H), **f32), dws_up=torch.empty((Fs, H), **f32),
                 dws_down=torch.empty((H, Fs), **f32))
    dx = torch.empty((T, H), **bf)
    dtw = torch.empty((T, k), **f32)
    moe.moe_backward_kept(cfg, d["x"], weights_arg(d), dy, L.ws, gu, dx, dtw, g, bws)
    torch.cuda.synchronize()
    assert moe.moe_read_status(bws) == moe.MOE_OK
    # sampled tokens, routed by the oracle from its own logits (equal to the layer's)
    toks = sample_tokens(w, 3)
    xs = x_rows(w, toks, "bf16")
    dys = synth.rows(0, synth.DY, toks, H, 1.0, "bf16")
    assert np.array_equal(np_of(dy[torch.from_numpy(toks).cuda()].float()), dys)  # device twin == host
    wr = w_router_host(w)
    assert_exact_router_sums(xs, wr)
    bias = synth.zipf_bias(0, E) if w["zipf"] else None
    l_ref = oracle.router_logits(xs, wr, bias)
    assert np.array_equal(np_of(L.logits[torch.from_numpy(toks).cuda()]), l_ref)
    idx_ref, wt_ref = oracle.route(l_ref, dict(w, T=len(toks)))
    assert np.array_equal(np_of(L.idx)[toks], idx_ref)
    experts = {}
    dx_gpu = np_of(dx.float()).astype(np.float64)[toks]
    dl_gpu = np_of(g["dlogits"]).astype(np.float64)[toks]
    for i in range(len(toks)):
        a = xs[i:i + 1].astype(np.float64)
        dyt = dys[i].astype(np.float64)
        dx_ref = np.zeros(H)
        dtw_ref = np.zeros(k)
        for j in range(k):
            e = int(idx_ref[i, j])
            if e not in experts:
                experts[e] = host_expert(w, e, 0)
            wg, wu, wd = experts[e]
            dtw_ref[j] = dyt @ oracle.expert_mlp(a, wg, wu, wd)[0]
            dx_ref += oracle.expert_mlp_backward(a, wg, wu, wd, (wt_ref[i, j] * dyt)[None])[0][0]
        if shared:
            dx_ref += oracle.expert_mlp_backward(a, *host_shared(w, 0), dyt[None])[0][0]
        dl_ref = oracle.router_backward(w, l_ref[i:i + 1], idx_ref[i:i + 1], dtw_ref[None])[0]
        dx_ref += dl_ref @ wr.astype(np.float64)
        assert oracle.rel_l2(dx_gpu[i], dx_ref) < 2e-2, (i, oracle.rel_l2(dx_gpu[i], dx_ref))
        # dlogits is a difference of the routing-weight gradients (softmax: q_j (g_j - <g, q>)),
        # each a dot product over H taken from bf16 expert outputs, so it is bounded against
        # their scale, rho * max |dtopk_w|, not its own (which can be a small difference)
        scale = float(w["routed_scale"]) * np.abs(dtw_ref).max()
        assert np.abs(dl_gpu[i] - dl_ref).max() <= 2e-2 * scale, (i, dl_gpu[i], dl_ref, scale)
    # dW_router = dl^T x on sampled experts (x redrawn on the host)
    x_all = grid_x(synth.normal(0, synth.X, (T, H), 1.0, "bf16")).astype(np.float64)
    dl_all = np_of(g["dlogits"]).astype(np.float64)
    dwr = np_of(g["dw_router"]).astype(np.float64)
    tc_path = E % 128 == 0 and H % 256 == 0
    for e in (0, E // 2, E - 1):
        ident = dl_all[:, e] @ x_all
        assert oracle.rel_l2(dwr[e], ident) < (8e-3 if tc_path else 1e-5), e
