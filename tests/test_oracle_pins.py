"""Pins of the CPU oracle to things other than itself (no GPU).

Each test checks one oracle function against what the mathematics or a library routine
fixes: brute force on tiny inputs, closed forms, special cases that reduce to a textbook
routine, invariants, and the fixed points of the e4m3 format. A plausible mistake in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a wrong tie-break)
fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cfg(E, k, score_fn=0, renorm=0, n_groups=1, topk_groups=1, group_score=0, rho=1.0, **kw):
    d = dict(T=0, H=0, E=E, k=k, F=0, n_shared=0, F_shared=0, score_fn=score_fn, renorm=renorm,
             n_groups=n_groups, topk_groups=topk_groups, group_score=group_score,
             routed_scale=rho, act_dtype=0, xfer_dtype=0)
    d.update(kw)
    return d


# ------------------------------------------------------------------ input generator
def test_splitmix64_published_sequence():
    # splitmix64 from state 0 (Steele, Lea, Flood 2014; Vigna's reference code): the first
    # two outputs are 0xE220A8397B1DCDAF and 0x6E789E6AA1B965F4.
    with np.errstate(over="ignore"):
        z = synth._mix64(np.array([synth.GOLDEN, synth.GOLDEN * np.uint64(2)], dtype=np.uint64))
    assert int(z[0]) == 0xE220A8397B1DCDAF
    assert int(z[1]) == 0x6E789E6AA1B965F4


def test_generator_moments_and_counter_access():
    a = synth.normal(3, synth.X, (512, 256), 1.0, "f32")
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    r = synth.rows(3, synth.X, [7, 300], 256, 1.0, "f32")
    assert np.array_equal(r, a[[7, 300]])
    b = synth.normal(3, synth.X, (512, 256), 0.02, "bf16")
    assert np.array_equal(b, synth.round_bf16(b))
    assert np.array_equal(torch.from_numpy(b).to(torch.bfloat16).float().numpy(), b)


def test_bf16_rounding_matches_torch():
    v = synth.normal(1, 99, (4096,), 3.0, "f32")
    ours = synth.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ours, ref)


def test_zipf_bias_recipe():
    b = synth.zipf_bias(0, 128)
    r = np.rint(np.exp(-b.astype(np.float64) / 1.2)).astype(int)
    assert sorted(r.tolist()) == list(range(1, 129))
    assert b.max() == 0.0 and abs(b.min() + 1.2 * math.log(128)) < 1e-5


# ------------------------------------------------------------------ deterministic exp
def test_det_expf_accuracy_against_fp64():
    a = np.concatenate([np.linspace(-103.0, 88.7, 200001, dtype=np.float32),
                        synth.normal(5, 98, (100000,), 4.0, "f32")])
    ours = oracle.det_expf(a).astype(np.float64)
    ref = np.exp(a.astype(np.float64))
    normal = ref > 1.2e-38
    ulp = np.spacing(ref[normal].astype(np.float32)).astype(np.float64)
    err = np.abs(ours[normal] - ref[normal]) / ulp
    assert err.max() <= 2.0, err.max()
    tiny = ~normal
    assert np.all(np.abs(ours[tiny] - ref[tiny]) <= 2.0 ** -149 * 2)


def test_det_expf_special_values():
    v = oracle.det_expf(np.array([0.0, -0.0, 89.0, -104.0, np.inf, -np.inf], np.float32))
    assert v[0] == 1.0 and v[1] == 1.0 and np.isinf(v[2]) and v[3] == 0.0
    assert np.isinf(v[4]) and v[5] == 0.0
    assert oracle.det_sigmoidf(0.0) == 0.5


def test_det_sigmoid_close_to_fp64():
    l = synth.normal(2, 97, (20000,), 3.0, "f32")
    ours = np.array([oracle.det_sigmoidf(float(x)) for x in l[:2000]])
    ref = 1.0 / (1.0 + np.exp(-l[:2000].astype(np.float64)))
    assert np.max(np.abs(ours - ref) / ref) < 4 * 2.0 ** -24


# ------------------------------------------------------------------ e4m3 codec
def test_e4m3_decode_all_codes_match_torch():
    ours = oracle.e4m3_decode_all()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_spec_points_golden():
    vals = oracle.e4m3_decode_all()
    with open(os.path.join(GOLDEN, "e4m3_ocp_points.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code, v = line.split()
            c = int(code, 16)
            if v == "nan":
                assert np.isnan(vals[c])
            else:
                assert vals[c] == float(v) and math.copysign(1, vals[c]) == math.copysign(1, float(v))
                assert oracle.e4m3_encode(np.float32(float(v)))[0] == c


def test_e4m3_encode_roundtrip_midpoints_and_saturation():
    vals = oracle.e4m3_decode_all()
    fin = [c for c in range(256) if not np.isnan(vals[c])]
    # every finite code round-trips
    assert all(oracle.e4m3_encode(np.float32(vals[c]))[0] == c for c in fin)
    # midpoints between neighbours go to the even (lower mantissa bit 0) code
    pos = sorted((vals[c], c) for c in range(128) if not np.isnan(vals[c]))
    for (v0, c0), (v1, c1) in zip(pos, pos[1:]):
        mid = np.float32((v0 + v1) / 2)
        assert float(mid) == (v0 + v1) / 2  # representable in fp32
        got = oracle.e4m3_encode(mid)[0]
        assert got == (c0 if c0 % 2 == 0 else c1), (v0, v1)
        # just off the midpoint goes to the nearer one
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(0)))[0] == c0
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(1e9)))[0] == c1
    # satfinite
    big = np.array([448.0, 460.0, 464.0, 1e6, np.inf, -1e30], np.float32)
    assert list(oracle.e4m3_encode(big)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e4m3_encode_in_range_matches_torch_cast():
    v = synth.normal(4, 96, (200000,), 60.0, "f32")
    v = v[np.abs(v) < 448]
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------ block quantisation
def test_quant_blocks_rule_and_error_bound():
    v = synth.normal(6, 95, (64, 384), 1.0, "bf16")
    v[3, 128:256] = 0.0  # an all-zero block
    q, s = oracle.quant_blocks(v, 1, 128)
    assert s.shape == (64, 3)
    assert s[3, 1] == 1.0 and not q[3, 128:256].any()
    amax = np.abs(v.reshape(64, 3, 128)).max(-1)
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    # the largest element of each block lands on +-448 exactly
    arg = np.abs(v.reshape(64, 3, 128)).argmax(-1)
    codes = np.take_along_axis(q.reshape(64, 3, 128), arg[..., None], -1)[..., 0]
    assert np.all((codes[nz] & 0x7F) == 0x7E)
    dq = oracle.dequant_blocks(q, s, 1, 128)
    # e4m3 has 3 mantissa bits: relative error <= 2^-4 for normals, abs <= 2^-10*scale below
    sc = np.repeat(s, 128, axis=1).astype(np.float64)
    bound = np.maximum(np.abs(v) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(dq - v) <= bound)
    # q matches the rule written with numpy + torch's cast
    with np.errstate(divide="ignore", invalid="ignore"):
        rs = (np.float32(448.0) / np.repeat(amax.astype(np.float32), 128, 1)).astype(np.float32)
        prod = (v * rs).astype(np.float32)
    ref = torch.from_numpy(np.clip(prod, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    m = np.repeat(nz, 128, axis=1)
    assert np.array_equal(q[m], ref[m])


def test_quant_blocks_128x128():
    w = synth.normal(7, 94, (256, 384), 0.02, "bf16")
    q, s = oracle.quant_blocks(w, 128, 128)
    assert s.shape == (2, 3)
    for bi in range(2):
        for bj in range(3):
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            assert s[bi, bj] == np.float32(np.abs(blk).max()) / np.float32(448)
    dq = oracle.dequant_blocks(q, s, 128, 128)
    assert oracle.rel_l2(dq, w) < 0.05


# ------------------------------------------------------------------ MX (MXFP8) quantisation
def test_mx_quant_worked_points():
    """Hand-derived points of the OCP MX v1.0 conversion to MXFP8 E4M3 (1x32 blocks)."""
    v = np.zeros((4, 32), dtype=np.float32)
    # amax 1.0: s = floor(log2 1) - 8 = -8 (code 119); 1.0 * 2^8 = 256 = 2^8 -> e4m3 0x78;
    # 0.3 * 2^8 = 76.8 = 9.6 * 2^3 -> mantissa rounds to 10 -> 80 = 1.25 * 2^6 -> 0x6A,
    # standing for 80 / 256 = 0.3125; -0.5 * 2^8 = -128 -> 0xF0
    v[0, 0], v[0, 5], v[0, 31] = 1.0, 0.3, -0.5
    # amax 1.9: s = -8; 1.9 * 256 = 486.4 > 448 saturates to 0x7E (stands for 1.75)
    v[1, 7], v[1, 8] = 1.9, np.float32(2.0 ** -9)
    # all-zero block: s = -127 (code 0), every element 0
    # amax 3 * 2^-140 (an fp32 subnormal): floor(log2) = -139, s = -147 clamps to -127;
    # 3 * 2^-140 * 2^127 = 3 * 2^-13 is below half the smallest e4m3 subnormal (2^-9) -> 0
    v[3, 2] = np.float32(3.0) * np.float32(2.0 ** -70) * np.float32(2.0 ** -70)
    q, sc = oracle.mx_quant(v)
    assert list(sc[:, 0]) == [119, 119, 0, 0]
    assert (q[0, 0], q[0, 5], q[0, 31]) == (0x78, 0x6A, 0xF0)
    assert q[1, 7] == 0x7E
    # 2^-9 * 2^8 = 0.5 = 2^-1 -> exponent field 6, mantissa 0 -> 0x30
    assert q[1, 8] == 0x30
    assert not q[2].any() and not q[3].any()
    dq = oracle.mx_dequant(q, sc)
    assert dq[0, 5] == 0.3125 and dq[1, 7] == 1.75 and dq[0, 31] == -0.5


def test_mx_quant_scale_invariant_and_error_bound():
    v = synth.normal(12, 93, (48, 256), 1.0, "bf16")
    v[5, 64:96] = 0.0
    v[9, 0:32] *= np.float32(2.0 ** 40)   # scale codes far from the centre of the range
    v[10, 32:64] *= np.float32(2.0 ** -40)
    q, sc = oracle.mx_quant(v)
    assert sc.shape == (48, 8) and sc.dtype == np.uint8
    blk = np.abs(v.reshape(48, 8, 32)).astype(np.float64)
    amax = blk.max(-1)
    s = sc.astype(np.int64) - 127
    nz = amax > 0
    # the defining property of s = floor(log2(amax)) - 8: amax * 2^-s in [256, 512)
    scaled = amax[nz] * np.exp2(-s[nz].astype(np.float64))
    assert np.all((scaled >= 256) & (scaled < 512))
    assert np.all(sc[~nz] == 0)
    dq = oracle.mx_dequant(q, sc)
    X = np.repeat(np.exp2(s.astype(np.float64)), 32, axis=1)
    a = np.abs(v).astype(np.float64)
    sat = a / X > 448
    # unsaturated: 3 mantissa bits -> relative error <= 2^-4, absolute <= 2^-10 * X below
    # the smallest normal; saturated elements (in (448, 512) * X) stand for 448 * X
    bound = np.maximum(a * 2.0 ** -4, X * 2.0 ** -10) * (1 + 1e-9)
    assert np.all(np.abs(dq - v)[~sat] <= bound[~sat])
    assert np.array_equal(np.abs(dq[sat]), 448 * X[sat])
    # in-range codes agree with torch's float8_e4m3fn cast of v * 2^-s (a library routine)
    prod = (v.astype(np.float64) / X).astype(np.float32)
    ref = torch.from_numpy(np.clip(prod, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q[~sat], ref[~sat])


def test_mx_quant_lossless_on_representable_blocks():
    """A block whose values are e4m3 values times one power of two, with its largest
    magnitude in [256, 448] * 2^j, is reproduced exactly: the scale comes out as 2^j."""
    vals = oracle.e4m3_decode_all()
    codes = np.arange(256)
    fin = codes[np.isfinite(vals)]
    rng = np.random.default_rng(5)
    rows = []
    for j in (-20, -8, 0, 3, 30):
        c = rng.choice(fin, size=32)
        c[rng.integers(32)] = rng.choice([0x78, 0x7A, 0x7E, 0xFE])  # 256, 320, 448, -448
        rows.append(vals[c] * 2.0 ** j)
    v = np.array(rows, dtype=np.float32)
    q, sc = oracle.mx_quant(v)
    assert list(sc[:, 0].astype(int) - 127) == [-20, -8, 0, 3, 30]
    assert np.array_equal(oracle.mx_dequant(q, sc), v.astype(np.float64))


# ------------------------------------------------------------------ router logits
def test_router_logits_fp64_then_round():
    x = synth.normal(0, 1, (64, 96), 1.0, "bf16")
    wr = synth.normal(0, 2, (16, 96), 0.02, "bf16")
    b = synth.zipf_bias(0, 16)
    l = oracle.router_logits(x, wr, b)
    exact = x.astype(np.float64) @ wr.astype(np.float64).T + b.astype(np.float64)
    assert np.max(np.abs(l - exact.astype(np.float32))) <= np.max(np.spacing(np.abs(l))) + 0
    assert np.mean(l == exact.astype(np.float32)) > 0.99


# ------------------------------------------------------------------ routing
def brute_topk(row, k, allowed=None):
    items = [(-float(row[e]), e) for e in range(len(row)) if allowed is None or allowed[e]]
    items.sort()
    return [e for _, e in items[:k]]


@pytest.mark.parametrize("E,k", [(4, 1), (8, 2), (8, 8), (16, 3), (16, 16), (12, 5)])
def test_topk_brute_force_with_ties(E, k):
    for seed, levels in [(0, 0), (1, 3), (2, 6)]:
        l = synth.synthetic_logits(seed, 200, E, 1.0, tie_levels=levels)
        l[0, :] = 0.0
        l[1, :] = -0.0
        l[2, ::2] = 0.0
        l[2, 1::2] = -0.0
        idx, w = oracle.route(l, cfg(E, k))
        for t in range(l.shape[0]):
            assert list(idx[t]) == brute_topk(l[t], k), (t, l[t])


def test_softmax_weights_closed_forms():
    l = synth.synthetic_logits(3, 100, 8)
    # k = E: every expert selected; weights = full softmax (no renorm) in selection order
    idx, w = oracle.route(l, cfg(8, 8))
    p = np.exp(l.astype(np.float64) - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.allclose(w, np.take_along_axis(p, idx, 1), rtol=1e-14, atol=0)
    # renormalised top-2 sums to 1 and equals softmax over the two logits
    idx, w = oracle.route(l, cfg(8, 2, renorm=1, rho=1.0))
    assert np.allclose(w.sum(1), 1.0, rtol=1e-14)
    l2 = np.take_along_axis(l.astype(np.float64), idx, 1)
    ref = 1.0 / (1.0 + np.exp(l2[:, 1] - l2[:, 0]))
    assert np.allclose(w[:, 0], ref, rtol=1e-13)
    # no renorm: weights are the softmax probabilities of the chosen experts
    idx, w = oracle.route(l, cfg(8, 2, renorm=0, rho=2.5))
    assert np.allclose(w, 2.5 * np.take_along_axis(p, idx, 1), rtol=1e-13)


def test_sigmoid_weights_closed_form():
    l = synth.synthetic_logits(4, 100, 16)
    idx, w = oracle.route(l, cfg(16, 4, score_fn=1, renorm=1))
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(l.astype(np.float64), idx, 1)))
    assert np.allclose(w, s / s.sum(1, keepdims=True), rtol=1e-13)
    idx, w = oracle.route(l, cfg(16, 4, score_fn=1, renorm=0, rho=0.5))
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(l.astype(np.float64), idx, 1)))
    assert np.allclose(w, 0.5 * s, rtol=1e-13)


def test_group_limited_special_cases_reduce_to_plain_topk():
    l = synth.synthetic_logits(5, 300, 32, tie_levels=8)
    plain, _ = oracle.route(l, cfg(32, 4, score_fn=1))
    g1, _ = oracle.route(l, cfg(32, 4, score_fn=1, n_groups=1, topk_groups=1))
    gG, _ = oracle.route(l, cfg(32, 4, score_fn=1, n_groups=4, topk_groups=4))
    assert np.array_equal(plain, g1) and np.array_equal(plain, gG)


@pytest.mark.parametrize("group_score", [0, 1])
def test_group_limited_brute_force(group_score):
    E, G, g, k = 16, 4, 2, 3
    l = synth.synthetic_logits(6, 400, E, 2.0, tie_levels=12)
    idx, _ = oracle.route(l, cfg(E, k, score_fn=1, n_groups=G, topk_groups=g, group_score=group_score))
    gs = E // G
    for t in range(l.shape[0]):
        s = [oracle.det_sigmoidf(float(v)) for v in l[t]]
        # group score written from the definition with Python's sort
        scores = []
        for q in range(G):
            top = sorted(s[q * gs:(q + 1) * gs], reverse=True)
            scores.append(np.float32(np.float32(top[0]) + np.float32(top[1])) if group_score == 0 else np.float32(top[0]))
        assert np.array_equal(oracle.group_scores(l[t], G, group_score), np.array(scores, np.float32))
        # enumerate all subsets of g groups; the kept set is the lexicographically first
        # subset among those whose sorted score vector is largest
        best = max(itertools.combinations(range(G), g),
                   key=lambda c: (sorted([scores[q] for q in c], reverse=True), [-q for q in c]))
        allowed = [(e // gs) in best for e in range(E)]
        assert list(idx[t]) == brute_topk(l[t], k, allowed), t


def test_group_score_uses_sigmoid_not_logit():
    # two groups: A has one huge and one tiny logit, B two moderate ones; the sum of
    # sigmoids prefers B although A's top logit is far larger
    l = np.array([[8.0, -8.0, 1.0, 1.0]], np.float32)
    idx, _ = oracle.route(l, cfg(4, 1, score_fn=1, n_groups=2, topk_groups=1))
    assert idx[0, 0] == 2
    idx, _ = oracle.route(l, cfg(4, 1, score_fn=1, n_groups=2, topk_groups=1, group_score=1))
    assert idx[0, 0] == 0


def test_route_rejects_non_finite():
    l = np.zeros((2, 8), np.float32)
    l[1, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.route(l, cfg(8, 2))


# ------------------------------------------------------------------ counts / permutation
@pytest.mark.parametrize("E,k,T", [(8, 2, 256), (128, 8, 1000), (16, 16, 33), (4, 1, 1)])
def test_permutation_invariants(E, k, T):
    l = synth.synthetic_logits(7, T, E, 1.0)
    l[:, : min(E, 3)] += 3.0  # hot experts
    idx, _ = oracle.route(l, cfg(E, k))
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[E] == T * k
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(tok_row.ravel()), np.arange(T * k))
    for e in range(E):
        seg = row_token[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.array_equal(seg, np.nonzero((idx == e).any(1))[0])
    for t in range(T):
        for j in range(k):
            r = tok_row[t, j]
            assert row_token[r] == t and offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]


def test_permute_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 8]], np.int32), 8)


# ------------------------------------------------------------------ dispatch + combine
@pytest.mark.parametrize("k", [2, 8])
def test_dispatch_combine_identity_experts_give_kx(k):
    T, H, E = 300, 64, 16
    x = synth.normal(8, 1, (T, H), 1.0, "bf16")
    idx, _ = oracle.route(synth.synthetic_logits(8, T, E), cfg(E, k))
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    xd = oracle.dispatch(x, row_token)
    assert np.array_equal(xd, x[row_token])
    y = oracle.combine(xd, tok_row, np.ones((T, k)))
    assert np.array_equal(y, k * x.astype(np.float64))


def test_combine_definition_with_shared_rows():
    T, H, k = 50, 32, 3
    yd = synth.normal(9, 12, (T * k, H), 1.0, "f32").astype(np.float64)
    ys = synth.normal(9, 13, (T, H), 1.0, "f32").astype(np.float64)
    perm = np.argsort(synth.bits_at(9, 14, np.arange(T * k, dtype=np.uint64)), kind="stable")
    tok_row = perm.reshape(T, k).astype(np.int32)
    w = synth.uniform_at(9, 15, np.arange(T * k)).reshape(T, k)
    y = oracle.combine(yd, tok_row, w, ys)
    ref = np.einsum("tj,tjh->th", w, yd[tok_row]) + ys
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-14)


# ------------------------------------------------------------------ expert MLP
def test_expert_mlp_matches_torch_swiglu():
    n, H, F = 37, 64, 96
    a = synth.normal(10, 1, (n, H), 1.0, "f32").astype(np.float64)
    wg = synth.normal(10, 3, (F, H), 0.1, "f32").astype(np.float64)
    wu = synth.normal(10, 4, (F, H), 0.1, "f32").astype(np.float64)
    wd = synth.normal(10, 5, (H, F), 0.1, "f32").astype(np.float64)
    y = oracle.expert_mlp(a, wg, wu, wd)
    A, G, U, D = (torch.from_numpy(v) for v in (a, wg, wu, wd))
    ref = (torch.nn.functional.silu(A @ G.T) * (A @ U.T)) @ D.T
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_expert_mlp_quantised_h():
    n, H, F = 9, 128, 256
    a = synth.normal(11, 1, (n, H), 1.0, "f32").astype(np.float64)
    wg = synth.normal(11, 3, (F, H), 0.1, "f32").astype(np.float64)
    wu = synth.normal(11, 4, (F, H), 0.1, "f32").astype(np.float64)
    wd = synth.normal(11, 5, (H, F), 0.1, "f32").astype(np.float64)
    A, G, U = (torch.from_numpy(v) for v in (a, wg, wu))
    h = (torch.nn.functional.silu(A @ G.T) * (A @ U.T)).numpy().astype(np.float32)
    q, s = oracle.quant_blocks(h, 1, 128)
    ref = oracle.dequant_blocks(q, s, 1, 128) @ wd.T
    y = oracle.expert_mlp(a, wg, wu, wd, quant_h=True)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    assert oracle.rel_l2(y, oracle.expert_mlp(a, wg, wu, wd)) < 0.05


def test_expert_mlp_mx_quantised_h():
    n, H, F = 9, 128, 256
    a = synth.normal(11, 1, (n, H), 1.0, "f32").astype(np.float64)
    wg = synth.normal(11, 3, (F, H), 0.1, "f32").astype(np.float64)
    wu = synth.normal(11, 4, (F, H), 0.1, "f32").astype(np.float64)
    wd = synth.normal(11, 5, (H, F), 0.1, "f32").astype(np.float64)
    A, G, U = (torch.from_numpy(v) for v in (a, wg, wu))
    h = (torch.nn.functional.silu(A @ G.T) * (A @ U.T)).numpy().astype(np.float32)
    ref = oracle.mx_dequant(*oracle.mx_quant(h)) @ wd.T
    y = oracle.expert_mlp(a, wg, wu, wd, quant_h=2)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    assert oracle.rel_l2(y, oracle.expert_mlp(a, wg, wu, wd)) < 0.05


# ------------------------------------------------------------------ whole layer
def small(name, **kw):
    return synth.scaled(synth.WORKLOADS[name], **kw)


SMALL = {
    "tiny": small("tiny_fp32", T=64),
    "mixtral": small("mixtral_bf16", T=96, H=128, F=256),
    "dsv3": small("dsv3_bf16", T=64, H=128, E=32, F=128, F_shared=128),
    "imbalanced": small("imbalanced_bf16", T=128, H=128, E=16, F=128),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_permuted_oracle_equals_dense_loop(name):
    w = SMALL[name]
    inp = synth.host_inputs(w, seed=1)
    a = oracle.forward(w, inp)
    b = oracle.dense_forward(w, inp)
    assert oracle.rel_l2(a["y"], b) < 1e-12


def test_identical_experts_with_renorm_equal_dense_mlp():
    w = small("mixtral_bf16", T=40, H=64, E=8, F=96, renorm=1)
    inp = synth.host_inputs(w, seed=2)
    for key in ("w_gate", "w_up", "w_down"):
        inp[key] = np.repeat(inp[key][:1], w["E"], axis=0)
    y = oracle.forward(w, inp)["y"]
    X = torch.from_numpy(inp["x"].astype(np.float64))
    G, U, D = (torch.from_numpy(inp[k][0].astype(np.float64)) for k in ("w_gate", "w_up", "w_down"))
    ref = ((torch.nn.functional.silu(X @ G.T) * (X @ U.T)) @ D.T).numpy()
    assert oracle.rel_l2(y, ref) < 1e-12


def test_single_expert_layer_is_dense_mlp_with_shared():
    w = small("dsv3_bf16", T=16, H=64, E=1, k=1, F=64, F_shared=32, n_groups=1, topk_groups=1)
    inp = synth.host_inputs(w, seed=3)
    y = oracle.forward(w, inp)["y"]
    X = torch.from_numpy(inp["x"].astype(np.float64))

    def mlp(g, u, d):
        g, u, d = (torch.from_numpy(v.astype(np.float64)) for v in (g, u, d))
        return (torch.nn.functional.silu(X @ g.T) * (X @ u.T)) @ d.T

    ref = mlp(inp["w_gate"][0], inp["w_up"][0], inp["w_down"][0]) + mlp(inp["ws_gate"], inp["ws_up"], inp["ws_down"])
    assert oracle.rel_l2(y, ref.numpy()) < 1e-12


def test_fp8_layer_close_to_unquantised():
    w = small("dsv3_fp8", T=32, H=256, E=16, F=128, F_shared=128, n_groups=4, topk_groups=2)
    inp = synth.host_inputs(w, seed=4)
    q = oracle.forward(w, inp)
    ref = oracle.forward(dict(w, xfer_dtype=synth.BF16), inp)
    assert np.array_equal(q["topk_idx"], ref["topk_idx"])
    # three e4m3 rounding points (x, weights, h), each up to 2^-4 relative
    assert 1e-3 < oracle.rel_l2(q["y"], ref["y"]) < 0.1


def test_mxfp8_layer_close_to_unquantised():
    w = small("dsv3_mxfp8", T=32, H=256, E=16, F=128, F_shared=128, n_groups=4, topk_groups=2)
    inp = synth.host_inputs(w, seed=4)
    q = oracle.forward(w, inp)
    ref = oracle.forward(dict(w, xfer_dtype=synth.BF16), inp)
    assert np.array_equal(q["topk_idx"], ref["topk_idx"])
    assert q["x_scale"].shape == (32, 256 // 32)
    # three e4m3 rounding points (x, weights, h) with power-of-two block scales
    assert 1e-3 < oracle.rel_l2(q["y"], ref["y"]) < 0.1


def test_mxfp8_layer_with_representable_inputs_is_exact_before_h():
    """With x and every weight already MX-representable, the MXFP8 layer differs from the
    unquantised one only through the requantisation of h (checked step by step)."""
    w = small("dsv3_mxfp8", T=16, H=128, E=4, k=2, F=64, n_shared=0, F_shared=0, n_groups=1,
              topk_groups=1)
    inp = synth.host_inputs(w, seed=6)
    for key in ("x", "w_gate", "w_up", "w_down"):
        a = inp[key]
        flat = a.reshape(-1, a.shape[-1])
        inp[key] = oracle.mx_dequant(*oracle.mx_quant(flat)).astype(np.float32).reshape(a.shape)
    q = oracle.forward(w, inp)
    assert np.array_equal(oracle.mx_dequant(q["x_q"], q["x_scale"]), inp["x"].astype(np.float64))
    y = np.zeros_like(q["yd"])
    for e in range(w["E"]):
        r0, r1 = q["offsets"][e], q["offsets"][e + 1]
        a = inp["x"][q["row_token"][r0:r1]].astype(np.float64)
        y[r0:r1] = oracle.expert_mlp(a, inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e], quant_h=2)
    assert np.array_equal(y, q["yd"])


def _e4m3_blocks(rng, rows, cols, br, bc, exps):
    """Values that are e4m3 values times one power of two 2^j per br x bc block, each block
    holding +-448 * 2^j exactly once and no other magnitude of 448, so a block quantiser of
    that shape reproduces them exactly (scale = amax / 448 = 2^j). Returns (values, codes,
    per-block j)."""
    vals = oracle.e4m3_decode_all()
    fin = np.array([c for c in range(256) if np.isfinite(vals[c]) and abs(vals[c]) < 448])
    codes = rng.choice(fin, size=(rows, cols)).astype(np.uint8)
    nbr, nbc = -(-rows // br), -(-cols // bc)
    j = rng.choice(exps, size=(nbr, nbc))
    for bi in range(nbr):
        for bj in range(nbc):
            r = bi * br + rng.integers(min(br, rows - bi * br))
            c = bj * bc + rng.integers(min(bc, cols - bj * bc))
            codes[r, c] = rng.choice([0x7E, 0xFE])  # +448, -448
    scale = np.exp2(np.repeat(np.repeat(j, br, 0), bc, 1)[:rows, :cols].astype(np.float64))
    return (vals[codes] * scale).astype(np.float32), codes, j


def test_fp8_layer_with_representable_inputs_is_exact_before_h():
    """The FP8 layer's composition step by step: x quantised per 1x128 block of a token's
    row, each expert weight per 128x128 block, and h requantised per 1x128 block before the
    down projection. With x and the weights built from e4m3 codes times a power-of-two scale
    per block of those shapes, the first two quantisations are exact, so the layer must equal
    the per-expert MLP with the 1x128 h requantisation alone, on those values, bit for bit.
    Blocks of any other shape (x in 128x1 columns, weights in 1x128 rows) are lossy on the
    same values, which the last asserts show."""
    w = small("dsv3_fp8", T=16, H=256, E=4, k=2, F=128, F_shared=128, n_groups=1, topk_groups=1)
    T, H, E, F = w["T"], w["H"], w["E"], w["F"]
    rng = np.random.default_rng(31)
    inp = synth.host_inputs(w, seed=7)
    x, x_codes, x_j = _e4m3_blocks(rng, T, H, 1, 128, np.arange(-9, -3))
    inp["x"] = x
    wexp = np.arange(-14, -8)
    for key, shape in (("w_gate", (E, F, H)), ("w_up", (E, F, H)), ("w_down", (E, H, F))):
        inp[key] = np.stack([_e4m3_blocks(rng, shape[1], shape[2], 128, 128, wexp)[0] for _ in range(E)])
    for key, shape in (("ws_gate", (F, H)), ("ws_up", (F, H)), ("ws_down", (H, F))):
        inp[key] = _e4m3_blocks(rng, shape[0], shape[1], 128, 128, wexp)[0]
    q = oracle.forward(w, inp)
    # x: one fp32 scale per (token, 128 columns), equal to the block's 2^j; codes unchanged
    assert q["x_scale"].shape == (T, H // 128)
    assert np.array_equal(q["x_scale"], np.exp2(x_j).astype(np.float32))
    assert np.array_equal(q["x_q"], x_codes)
    # the experts, the shared expert and combine on the exact values
    x64 = x.astype(np.float64)
    yd = np.zeros_like(q["yd"])
    for e in range(E):
        r0, r1 = q["offsets"][e], q["offsets"][e + 1]
        yd[r0:r1] = oracle.expert_mlp(x64[q["row_token"][r0:r1]], inp["w_gate"][e], inp["w_up"][e],
                                      inp["w_down"][e], quant_h=1)
    assert np.array_equal(yd, q["yd"])
    ys = oracle.expert_mlp(x64, inp["ws_gate"], inp["ws_up"], inp["ws_down"], quant_h=1)
    assert np.array_equal(ys, q["ys"])
    assert np.array_equal(oracle.combine(yd, q["tok_row"], q["topk_w"], ys), q["y"])
    # the same values through blocks of the other orientation are not reproduced
    assert not np.array_equal(oracle.dequant_blocks(*oracle.quant_blocks(x, 128, 1), 128, 1), x64)
    wg0 = inp["w_gate"][0]
    assert not np.array_equal(oracle.dequant_blocks(*oracle.quant_blocks(wg0, 1, 128), 1, 128),
                              wg0.astype(np.float64))


# ------------------------------------------------------------------ backward
def test_expert_mlp_backward_matches_torch_autograd():
    n, H, F = 13, 48, 40
    a = synth.normal(20, 1, (n, H), 1.0, "f32").astype(np.float64)
    wg = synth.normal(20, 3, (F, H), 0.2, "f32").astype(np.float64)
    wu = synth.normal(20, 4, (F, H), 0.2, "f32").astype(np.float64)
    wd = synth.normal(20, 5, (H, F), 0.2, "f32").astype(np.float64)
    dyd = synth.normal(20, 6, (n, H), 1.0, "f32").astype(np.float64)
    dxd, dwg, dwu, dwd = oracle.expert_mlp_backward(a, wg, wu, wd, dyd)
    A, G, U, D = (torch.tensor(v, requires_grad=True) for v in (a, wg, wu, wd))
    y = (torch.nn.functional.silu(A @ G.T) * (A @ U.T)) @ D.T
    y.backward(torch.from_numpy(dyd))
    for ours, ref in ((dxd, A), (dwg, G), (dwu, U), (dwd, D)):
        assert np.allclose(ours, ref.grad.numpy(), rtol=1e-11, atol=1e-13)


def test_combine_and_dispatch_backward_are_adjoints():
    """<combine(yd), dy> = <yd, combine_bwd(dy)>, <dispatch(x), z> = <x, dispatch_bwd(z)>,
    and the weight gradient is <dy[t], yd[r_tj]>: the backward steps are the transposes of
    the forward permutations."""
    T, k, E, H = 40, 3, 6, 24
    idx, w = oracle.route(synth.synthetic_logits(21, T, E), cfg(E, k, renorm=1))
    counts, offsets, row_token, tok_row = oracle.permute(idx, E)
    R = T * k
    for shared in (False, True):
        rows = R + (T if shared else 0)
        yd = synth.normal(21, 7, (rows, H), 1.0, "f32").astype(np.float64)
        dy = synth.normal(21, 8, (T, H), 1.0, "f32").astype(np.float64)
        y = oracle.combine(yd[:R], tok_row, w, yd[R:] if shared else None)
        dyd, dw = oracle.combine_backward(dy, yd, tok_row, w, shared)
        assert np.isclose(np.sum(y * dy), np.sum(yd * dyd), rtol=1e-12)
        assert np.allclose(dw, np.einsum("th,tjh->tj", dy, yd[tok_row]), rtol=1e-12)
        x = synth.normal(21, 9, (T, H), 1.0, "f32").astype(np.float64)
        z = synth.normal(21, 10, (rows, H), 1.0, "f32").astype(np.float64)
        xd = x[row_token] if not shared else np.concatenate([x[row_token], x])
        dx = oracle.dispatch_backward(z, tok_row, shared)
        assert np.isclose(np.sum(xd * z), np.sum(x * dx), rtol=1e-12)


@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_layer_backward_matches_finite_differences(name):
    """L = <dy, y>; with the routing held fixed, the central difference of L along a random
    direction of x or of each weight equals <grad, direction> (error O(eps^2))."""
    w = {"mixtral": small("mixtral_bf16", T=10, H=32, E=4, F=24, renorm=1),
         "dsv3": small("dsv3_bf16", T=8, H=32, E=8, k=2, F=16, F_shared=16, n_groups=2, topk_groups=1)}[name]
    inp = {kk: (v.astype(np.float64) if isinstance(v, np.ndarray) else v)
           for kk, v in synth.host_inputs(w, seed=22).items()}
    logits = synth.synthetic_logits(22, w["T"], w["E"])
    fwd = oracle.forward(w, inp, logits=logits)
    dy = synth.normal(22, 11, (w["T"], w["H"]), 1.0, "f32").astype(np.float64)
    g = oracle.backward(w, inp, fwd, dy)
    pairs = [("x", "dx"), ("w_gate", "dw_gate"), ("w_up", "dw_up"), ("w_down", "dw_down")]
    if w["n_shared"]:
        pairs += [("ws_gate", "dws_gate"), ("ws_up", "dws_up"), ("ws_down", "dws_down")]
    for tid, (key, gkey) in enumerate(pairs):
        v = synth.normal(23, 40 + tid, inp[key].shape, 1.0, "f32").astype(np.float64)
        eps = 1e-5 * np.abs(inp[key]).max()

        def L(delta):
            p = dict(inp)
            p[key] = inp[key] + delta * v
            return float(np.sum(oracle.forward(w, p, logits=logits)["y"] * dy))

        fd = (L(eps) - L(-eps)) / (2 * eps)
        an = float(np.sum(g[gkey] * v))
        assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (key, fd, an)


ROUTER_BWD = {
    "softmax_all": cfg(8, 2, score_fn=0, renorm=0),
    "softmax_topk": cfg(8, 2, score_fn=0, renorm=1, rho=2.5),
    "sigmoid": cfg(16, 3, score_fn=1, renorm=0, rho=1.5),
    "sigmoid_renorm_groups": cfg(16, 4, score_fn=1, renorm=1, n_groups=4, topk_groups=2, group_score=1, rho=2.5),
    "softmax_k_eq_e": cfg(4, 4, score_fn=0, renorm=1),
}


FD_EPS = 2.0 ** -16


def _grid_logits(seed, T, E):
    """Logits on the grid 2^-16 with |l| < 2^7, so that l +- 2^-16 * v for small integer v
    is an exact fp32 value and the finite difference sees exactly the step it divides by."""
    l = synth.synthetic_logits(seed, T, E).astype(np.float64)
    assert np.abs(l).max() < 100.0
    return (np.round(l / FD_EPS) * FD_EPS).astype(np.float32)


@pytest.mark.parametrize("name", list(ROUTER_BWD))
def test_router_backward_matches_finite_differences_of_the_weights(name):
    """With the chosen experts fixed, <g, w(l + eps v) - w(l - eps v)> / (2 eps) equals
    <dl, v> for dl = router_backward(g), up to O(eps^2)."""
    c = ROUTER_BWD[name]
    T, E, k = 24, c["E"], c["k"]
    l = _grid_logits(30, T, E)
    idx, _ = oracle.route(l, c)
    g = synth.normal(30, 1, (T, k), 1.0, "f32").astype(np.float64)
    dl = oracle.router_backward(c, l, idx, g)
    eps = FD_EPS
    v = np.round(synth.normal(30, 2, (T, E), 2.0, "f32").astype(np.float64))
    lp, lm = (l.astype(np.float64) + eps * v).astype(np.float32), (l.astype(np.float64) - eps * v).astype(np.float32)
    assert np.array_equal(lp.astype(np.float64) - l, eps * v) and np.array_equal(l - lm.astype(np.float64), eps * v)
    ip, wp = oracle.route(lp, c)
    im, wm = oracle.route(lm, c)
    assert np.array_equal(ip, idx) and np.array_equal(im, idx), "a step this small changed a choice"
    fd = np.sum(g * (wp - wm), axis=1) / (2 * eps)
    an = np.sum(dl * v, axis=1)
    assert np.allclose(fd, an, rtol=1e-6, atol=1e-8 * np.abs(an).max())
    # experts no weight depends on get no gradient
    chosen = np.zeros((T, E), bool)
    np.put_along_axis(chosen, idx.astype(np.int64), True, axis=1)
    if not (c["score_fn"] == 0 and c["renorm"] == 0):
        assert np.all(dl[~chosen] == 0.0)


@pytest.mark.parametrize("renorm", [0, 1])
def test_router_backward_softmax_is_shift_invariant(renorm):
    """Softmax weights do not change when every logit of a token moves by the same amount,
    so each token's logit gradient sums to zero; with k = E and renorm the weight step is
    the plain softmax, whose Jacobian-vector product is p * (g - <g, p>)."""
    c = cfg(8, 3, score_fn=0, renorm=renorm, rho=1.7)
    T = 40
    l = synth.synthetic_logits(31, T, 8)
    idx, _ = oracle.route(l, c)
    g = synth.normal(31, 1, (T, 3), 1.0, "f32").astype(np.float64)
    dl = oracle.router_backward(c, l, idx, g)
    assert np.allclose(dl.sum(axis=1), 0.0, atol=1e-14 * np.abs(dl).max())
    ce = cfg(6, 6, score_fn=0, renorm=1)
    le = synth.synthetic_logits(32, T, 6)
    ie, _ = oracle.route(le, ce)
    ge = synth.normal(32, 1, (T, 6), 1.0, "f32").astype(np.float64)
    p = np.exp(le.astype(np.float64) - le.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    gp = np.zeros((T, 6))
    np.put_along_axis(gp, ie.astype(np.int64), ge, axis=1)  # g in expert order
    want = p * (gp - np.sum(gp * p, axis=1, keepdims=True))
    assert np.allclose(oracle.router_backward(ce, le, ie, ge), want, rtol=1e-12, atol=1e-15)


def test_router_backward_sigmoid_without_renorm_is_the_logistic_derivative():
    """Without normalisation each weight is rho * sigma(l_i) alone: dl_i = rho g_i s_i (1 - s_i)."""
    c = cfg(8, 2, score_fn=1, renorm=0, rho=3.0)
    l = synth.synthetic_logits(33, 16, 8)
    idx, _ = oracle.route(l, c)
    g = synth.normal(33, 1, (16, 2), 1.0, "f32").astype(np.float64)
    dl = oracle.router_backward(c, l, idx, g)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(l.astype(np.float64), idx.astype(np.int64), axis=1)))
    assert np.allclose(np.take_along_axis(dl, idx.astype(np.int64), axis=1), 3.0 * g * s * (1 - s), rtol=1e-13)


@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_layer_backward_through_the_router_matches_finite_differences(name):
    """L = <dy, y> as a function of the logits (selection fixed): the combine backward's
    dtopk_w fed through router_backward gives dL/dlogits; the linear router's products give
    dL/dW_router = dl^T x and x's share dl W_router, checked on the linear map's definition."""
    w = {"mixtral": small("mixtral_bf16", T=10, H=32, E=4, F=24, renorm=1),
         "dsv3": small("dsv3_bf16", T=8, H=32, E=8, k=2, F=16, F_shared=16, n_groups=2, topk_groups=1)}[name]
    inp = {kk: (v.astype(np.float64) if isinstance(v, np.ndarray) else v)
           for kk, v in synth.host_inputs(w, seed=24).items()}
    l = _grid_logits(24, w["T"], w["E"])
    fwd = oracle.forward(w, inp, logits=l)
    dy = synth.normal(24, 11, (w["T"], w["H"]), 1.0, "f32").astype(np.float64)
    g = oracle.backward(w, inp, fwd, dy)
    dl = oracle.router_backward(w, l, fwd["topk_idx"], g["dtopk_w"])
    eps = FD_EPS
    v = np.round(synth.normal(24, 12, l.shape, 2.0, "f32").astype(np.float64))

    def L(sign):
        lx = (l.astype(np.float64) + sign * eps * v).astype(np.float32)
        o = oracle.forward(w, inp, logits=lx)
        assert np.array_equal(o["topk_idx"], fwd["topk_idx"])
        return float(np.sum(o["y"] * dy))

    fd = (L(1) - L(-1)) / (2 * eps)
    an = float(np.sum(dl * v))
    assert abs(fd - an) <= 1e-6 * max(abs(an), 1e-3), (fd, an)
    # the linear router: logits = x W^T, so <dl, dlogits> = <dW, dWdir> + <dx_r, dxdir>
    dwr, dxr = oracle.router_linear_backward(inp["x"], inp["w_router"], dl)
    vx = synth.normal(24, 13, inp["x"].shape, 1.0, "f32").astype(np.float64)
    vw = synth.normal(24, 14, inp["w_router"].shape, 1.0, "f32").astype(np.float64)
    x64, w64 = inp["x"].astype(np.float64), inp["w_router"].astype(np.float64)
    dlog = vx @ w64.T + x64 @ vw.T  # the exact first-order change of the logits
    assert np.isclose(np.sum(dl * dlog), np.sum(dwr * vw) + np.sum(dxr * vx), rtol=1e-12)


# ------------------------------------------------------------------ aux load-balancing loss
@pytest.mark.parametrize("score_fn", [0, 1])
def test_aux_loss_backward_matches_finite_differences(score_fn):
    """With the counts fixed, (L(l + eps v) - L(l - eps v)) / (2 eps) = <dL/dl, v>; and for
    softmax each token's gradient sums to zero (the loss does not see a shift of a row)."""
    T, E, k = 32, 8, 2
    l = _grid_logits(34, T, E)
    counts = oracle.permute(oracle.route(l, cfg(E, k))[0], E)[0]
    dl = oracle.aux_loss_backward(l, counts, k, score_fn, 0.01)
    v = np.round(synth.normal(34, 2, (T, E), 2.0, "f32").astype(np.float64))
    lp = (l.astype(np.float64) + FD_EPS * v).astype(np.float32)
    lm = (l.astype(np.float64) - FD_EPS * v).astype(np.float32)
    fd = (oracle.aux_loss(lp, counts, k, score_fn, 0.01)[0] - oracle.aux_loss(lm, counts, k, score_fn, 0.01)[0]) / (
        2 * FD_EPS)
    an = float(np.sum(dl * v))
    assert abs(fd - an) <= 1e-6 * abs(an), (fd, an)
    if score_fn == 0:
        assert np.allclose(dl.sum(axis=1), 0.0, atol=1e-14 * np.abs(dl).max())
    # uniform counts make the loss alpha * E / (T k) * (T k / E) * sum_e Pbar_e = alpha for
    # softmax, whatever the logits: its gradient vanishes
    flat = np.full(E, T * k // E, np.int32)
    if score_fn == 0:
        assert np.abs(oracle.aux_loss_backward(l, flat, k, 0, 0.01)).max() < 1e-18


def test_aux_loss_closed_forms():
    T, E, k = 64, 8, 2
    c8 = cfg(E, k)
    # uniform probabilities: Pbar = 1/E, loss = alpha whatever the counts
    l = np.zeros((T, E), np.float32)
    idx, _ = oracle.route(l, c8)
    counts = oracle.permute(idx, E)[0]
    loss, pbar = oracle.aux_loss(l, counts, k, 0, 0.01)
    assert np.allclose(pbar, 1.0 / E, rtol=1e-15) and loss == pytest.approx(0.01, rel=1e-14)
    # all tokens on experts 0 and 1 with equal, dominant logits: Pbar_0 = Pbar_1 -> 1/2,
    # loss -> alpha * E / k
    l = np.zeros((T, E), np.float32)
    l[:, :2] = 40.0
    idx, _ = oracle.route(l, c8)
    counts = oracle.permute(idx, E)[0]
    loss, _ = oracle.aux_loss(l, counts, k, 0, 0.01)
    assert loss == pytest.approx(0.01 * E / k, rel=1e-12)


def test_aux_loss_matches_numpy_definition():
    T, E, k = 200, 16, 3
    l = synth.synthetic_logits(12, T, E, 2.0)
    for score_fn in (0, 1):
        idx, _ = oracle.route(l, cfg(E, k, score_fn=score_fn))
        counts = oracle.permute(idx, E)[0]
        loss, pbar = oracle.aux_loss(l, counts, k, score_fn, 0.01)
        L = l.astype(np.float64)
        p = np.exp(L - L.max(1, keepdims=True)) if score_fn == 0 else 1.0 / (1.0 + np.exp(-L))
        p /= p.sum(1, keepdims=True)
        ref_pbar = p.mean(0)
        assert np.allclose(pbar, ref_pbar, rtol=1e-12)
        assert loss == pytest.approx(0.01 * E / (T * k) * float(np.dot(np.bincount(idx.ravel(), minlength=E), ref_pbar)), rel=1e-12)
