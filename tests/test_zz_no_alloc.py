"""moe_route_static_scratch: routing for callers that cannot allocate device memory (a
plugin handed only its input and output buffers, a runtime with a fixed memory budget
reserved up front). It must give exactly what moe_route gives (same kernels, same bits)
while its scan scratch lives in the library's fixed array, call after call. This file is
collected last so that a failure here comes after every other test has run."""
import numpy as np
import pytest
import torch

import synth
import token_routing_expert_router_gb300 as moe
from moe_case import alloc, cfg_of, up

pytestmark = pytest.mark.gpu

CASES = [
    synth.workload("dsv3_route", 8192, 128, 256, 8, 128, score_fn=synth.SIGMOID, renorm=1,
                   n_groups=8, topk_groups=4),
    synth.workload("imbalanced_route", 16384, 128, 128, 8, 128, zipf=True),
    synth.workload("tiny_route", 256, 128, 8, 2, 128),
]

KEYS = ("topk_idx", "topk_w", "counts", "offsets", "row_token", "tok_row")


def fresh(w):
    T, E, k = w["T"], w["E"], w["k"]
    o = {"topk_idx": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
         "topk_w": torch.full((T, k), -7.0, dtype=torch.float32, device="cuda"),
         "counts": torch.full((E,), -7, dtype=torch.int32, device="cuda"),
         "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
         "row_token": torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
         "tok_row": torch.full((T, k), -7, dtype=torch.int32, device="cuda")}
    return o


@pytest.mark.parametrize("w", CASES, ids=[c["name"] for c in CASES])
def test_static_scratch_matches_moe_route(w):
    l = synth.synthetic_logits(2, w["T"], w["E"])
    if w["zipf"]:
        l = (l + synth.zipf_bias(2, w["E"])).astype(np.float32)
    lg = up(l)
    b = alloc(w)
    moe.moe_route(b["cfg"], lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    for call in range(2):  # the shared array keeps the previous call's contents
        o = fresh(w)
        moe.moe_route_static_scratch(b["cfg"], lg, o["topk_idx"], o["topk_w"], o["counts"],
                                     o["offsets"], o["row_token"], o["tok_row"], status)
        torch.cuda.synchronize()
        for key in KEYS:  # same kernels on the same scores: every output bit for bit
            assert torch.equal(o[key], b[key]), (call, key)
        assert int(status[0]) == 0


def test_static_scratch_reports_bad_scores_and_rejects_oversize():
    w = CASES[2]
    l = synth.synthetic_logits(3, w["T"], w["E"])
    l[9, 1] = np.inf
    o = fresh(w)
    status = torch.zeros(2, dtype=torch.int32, device="cuda")
    moe.moe_route_static_scratch(cfg_of(w), up(l), o["topk_idx"], o["topk_w"], o["counts"],
                                 o["offsets"], o["row_token"], o["tok_row"], status)
    torch.cuda.synchronize()
    assert int(status[0]) == moe.MOE_ERR_DEVICE_BAD_INPUT
    big = cfg_of(synth.workload("too_big", 1 << 20, 128, 256, 8, 128))
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route_static_scratch(big, o["topk_idx"], o["topk_idx"], o["topk_w"], o["counts"],
                                     o["offsets"], o["row_token"], o["tok_row"], None)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED
