"""S1 + S2 on the GPU against the oracle: routing maps, counts, offsets and permutation
indices bit-exact when both sides get identical fp32 router scores; weights within fp32
rounding; deterministic across runs; device-side input faults reported in the status word."""
import numpy as np
import pytest
import torch

import oracle
import synth
import token_routing_expert_router_gb300 as moe
from moe_case import alloc, cfg_of, np_of, up

pytestmark = pytest.mark.gpu

S, G = synth.SOFTMAX, synth.SIGMOID


def rcase(name, T, E, k, score_fn=S, renorm=0, n_groups=1, topk_groups=1, group_score=0,
          ties=0, zipf=False, rho=1.0):
    w = synth.workload(name, T, 128, E, k, 128, score_fn=score_fn, renorm=renorm,
                       n_groups=n_groups, topk_groups=topk_groups, group_score=group_score,
                       routed_scale=rho, zipf=zipf)
    w["ties"] = ties
    return w


CASES = [
    rcase("tiny", 256, 8, 2),
    rcase("mixtral", 4096, 8, 2, renorm=1),
    rcase("dsv3", 8192, 256, 8, G, 1, 8, 4),
    rcase("imbalanced", 16384, 128, 8, zipf=True),
    rcase("dsv3_fp8_tokens", 32768, 256, 8, G, 1, 8, 4),
    rcase("ties_e16", 1000, 16, 3, ties=6),
    rcase("ties_groups", 2000, 64, 6, G, 1, 8, 3, ties=10),
    rcase("group_max", 1500, 64, 4, G, 0, 8, 2, group_score=1, rho=2.5),
    rcase("k_eq_e", 300, 4, 4),
    rcase("e512_k32", 700, 512, 32, G, 1, 16, 12),
    rcase("e33_ragged", 333, 33, 5),
    rcase("one_token", 1, 64, 8, G, 1, 8, 4),
    rcase("e512_long", 20000, 512, 8, G, 1, 16, 8),
    # more than 8192 per-block counts with E not a multiple of 4: the two-level count scan
    rcase("e33_long", 30000, 33, 5),
]


def logits_of(w, seed=0):
    l = synth.synthetic_logits(seed, w["T"], w["E"], 1.0, tie_levels=w.get("ties", 0))
    if w.get("ties"):
        l[0, :] = 0.0
        if w["T"] > 1:
            l[1, ::2] = -0.0
    if w["zipf"]:
        l = (l + synth.zipf_bias(seed, w["E"])).astype(np.float32)
    return l


def gpu_route(w, l):
    b = alloc(w)
    moe.moe_route(b["cfg"], up(l), b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    return b


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_route_bit_exact(w):
    l = logits_of(w)
    idx, wt = oracle.route(l, w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, w["E"])
    b = gpu_route(w, l)
    assert np.array_equal(np_of(b["topk_idx"]), idx)
    assert np.array_equal(np_of(b["counts"]), counts)
    assert np.array_equal(np_of(b["offsets"]), offsets)
    assert np.array_equal(np_of(b["row_token"]), row_token)
    assert np.array_equal(np_of(b["tok_row"]), tok_row)
    g = np_of(b["topk_w"]).astype(np.float64)
    assert np.allclose(g, wt, rtol=4e-6, atol=1e-7), np.abs(g - wt).max()
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK


@pytest.mark.parametrize("w", [CASES[2], CASES[3]], ids=["dsv3", "imbalanced"])
def test_route_deterministic(w):
    l = logits_of(w, seed=1)
    a = gpu_route(w, l)
    b = gpu_route(w, l)
    for key in ("topk_idx", "topk_w", "counts", "offsets", "row_token", "tok_row"):
        assert torch.equal(a[key], b[key]), key


def test_route_empty_and_hot_experts():
    w = rcase("hot", 3000, 32, 4)
    l = logits_of(w)
    l[:, :3] += 20.0       # every token picks experts 0..2
    l[:, 10:20] -= 50.0    # experts 10..19 are never picked
    idx, _ = oracle.route(l, w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, w["E"])
    assert counts[0] == 3000 and counts[10:20].sum() == 0
    b = gpu_route(w, l)
    assert np.array_equal(np_of(b["offsets"]), offsets)
    assert np.array_equal(np_of(b["row_token"]), row_token)


def test_router_replay_from_map():
    w = rcase("replay", 5000, 128, 8)
    idx, _ = oracle.route(logits_of(w, seed=3), w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, w["E"])
    b = alloc(w)
    moe.moe_route_from_map(b["cfg"], up(idx), b["counts"], b["offsets"], b["row_token"],
                           b["tok_row"], b["ws"])
    assert np.array_equal(np_of(b["counts"]), counts)
    assert np.array_equal(np_of(b["row_token"]), row_token)
    assert np.array_equal(np_of(b["tok_row"]), tok_row)
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK


def test_device_status_bad_inputs():
    w = rcase("bad", 200, 16, 2)
    b = alloc(w)
    idx = np.tile(np.array([[1, 2]], np.int32), (200, 1))
    idx[7, 1] = 16  # out of range
    moe.moe_route_from_map(b["cfg"], up(idx), b["counts"], b["offsets"], b["row_token"],
                           b["tok_row"], b["ws"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_ERR_DEVICE_BAD_INPUT
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK  # reading clears it
    tr = np_of(b["tok_row"])
    assert tr.min() >= 0 and tr.max() < 400  # outputs stay in bounds
    idx[7] = [2, 2]  # repeated id in one row
    moe.moe_route_from_map(b["cfg"], up(idx), b["counts"], b["offsets"], b["row_token"],
                           b["tok_row"], b["ws"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_ERR_DEVICE_BAD_INPUT
    l = logits_of(w)
    l[5, 3] = np.nan
    moe.moe_route(b["cfg"], up(l), b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_ERR_DEVICE_BAD_INPUT
    ti = np_of(b["topk_idx"])
    assert ti.min() >= 0 and ti.max() < 16


def test_zero_tokens():
    w = rcase("empty", 0, 8, 2)
    cfg = cfg_of(w)
    counts = torch.full((8,), 7, dtype=torch.int32, device="cuda")
    offsets = torch.full((9,), 7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(1024, dtype=torch.int32, device="cuda")
    e = torch.empty(0, device="cuda")
    moe.moe_route(cfg, e, e, e, counts, offsets, e, e, ws)
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0


@pytest.mark.parametrize("w", [CASES[0], CASES[2], CASES[3], CASES[4], CASES[10]],
                         ids=["tiny", "dsv3", "imbalanced", "dsv3_fp8_tokens", "e33_ragged"])
def test_aux_loss_against_oracle(w):
    l = logits_of(w, seed=4)
    idx, _ = oracle.route(l, w)
    counts = oracle.permute(idx, w["E"])[0]
    ref, _ = oracle.aux_loss(l, counts, w["k"], w["score_fn"], 0.01)
    b = alloc(w)
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_aux_loss(b["cfg"], up(l), up(counts), 0.01, loss, b["ws"])
    got = float(loss.item())
    assert got == pytest.approx(ref, rel=2e-5)
    loss2 = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_aux_loss(b["cfg"], up(l), up(counts), 0.01, loss2, b["ws"])
    assert torch.equal(loss, loss2)  # deterministic


@pytest.mark.parametrize("score_fn", [synth.SOFTMAX, synth.SIGMOID], ids=["softmax", "sigmoid"])
@pytest.mark.parametrize("T,E,k", [(700, 4, 2), (300, 256, 8), (5000, 8, 2)])
def test_aux_loss_of_equal_scores_is_alpha(T, E, k, score_fn):
    """Equal logits: each probability is 1/E (softmax, or sigmoid scores of 1/2 over their
    sum; exact, E a power of two), so Pbar_e = 1/E and the loss is
    alpha * E / (T k) * sum_e counts[e] / E = alpha for any counts summing to T k. The
    fixed-point sums are exact, so the result is alpha to the last bit."""
    w = rcase("equal", T, E, k, score_fn=score_fn)
    b = alloc(w)
    counts = np.full(E, T * k // E, dtype=np.int32)
    counts[: T * k % E] += 1
    assert counts.sum() == T * k
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    moe.moe_aux_loss(b["cfg"], torch.zeros((T, E), dtype=torch.float32, device="cuda"), up(counts), 0.01, loss,
                     b["ws"])
    assert float(loss.item()) == np.float32(0.01)


def test_both_routing_paths_are_exercised():
    """moe_route takes one cooperative launch where a block's token chunk times ceil(E / 32)
    stays within 1024, else the top-k launch and the scan passes. The bit-exact cases above
    cover both: every workload-sized routing takes the single launch, the 20000-token one
    over 512 grouped experts the top-k launch and the three scan passes."""
    n = {w["name"]: moe.moe_route_launch_count(cfg_of(w)) for w in CASES}
    assert n["mixtral"] == 1 and n["tiny"] == 1 and n["dsv3"] == 1 and n["imbalanced"] == 1
    assert n["dsv3_fp8_tokens"] == 1
    assert n["e512_long"] == 4
    assert set(n.values()) <= {1, 2, 4}
    assert moe.moe_route_launch_count(cfg_of(synth.scaled(CASES[0], T=0))) == 0
