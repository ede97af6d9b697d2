"""Failure detection without a GPU fault: a bounded wait that runs out (a barrier nothing
arrives on) reports MOE_ERR_TIMEOUT through the status word and returns, and the context
stays usable; faults found on the device are reported, never trapped."""
import time

import numpy as np
import torch
import pytest

import synth
import token_routing_expert_router_gb300 as moe
from moe_case import alloc, np_of, up

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_context_survives():
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    moe.moe_selftest_bounded_wait(2_000_000, st)  # 2 ms limit
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st[0]) == moe.MOE_ERR_TIMEOUT
    assert dt < 5.0
    # the context still runs the library's kernels correctly
    w = synth.workload("after", 512, 128, 16, 2, 128)
    b = alloc(w)
    l = synth.synthetic_logits(0, 512, 16)
    moe.moe_route(b["cfg"], up(l), b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
    assert int(np_of(b["counts"]).sum()) == 1024


def test_bounded_wait_rejects_bad_limits():
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    for bad in (0, -1, 11_000_000_000):
        with pytest.raises(moe.MoEError):
            moe.moe_selftest_bounded_wait(bad, st)


def test_routing_barrier_wait_gives_up_with_a_safe_map():
    """The single-launch routing's grid barrier lives in the workspace head (its counter at
    byte 128, word 32; its flag 128 bytes later). A counter left at a value no arrival can
    complete (here 7, for a grid of one block) makes the barrier's wait run out after its
    2 s limit: the call reports
    MOE_ERR_TIMEOUT and leaves a map every later launch can read in bounds (no routed rows,
    tok_row all 0). A fresh moe_workspace_init clears the head and routing works again."""
    import oracle
    w = synth.workload("barrier", 16, 128, 8, 2, 128)
    b = alloc(w)
    assert moe.moe_route_launch_count(b["cfg"]) == 1
    l = synth.synthetic_logits(3, 16, 8)
    moe.moe_workspace_init(b["ws"])
    b["ws"][32] = 7
    b["counts"].fill_(-1)
    b["offsets"].fill_(-1)
    b["tok_row"].fill_(-1)
    t0 = time.perf_counter()
    moe.moe_route(b["cfg"], up(l), b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert moe.moe_read_status(b["ws"]) == moe.MOE_ERR_TIMEOUT
    assert not np_of(b["counts"]).any() and not np_of(b["offsets"]).any()
    assert not np_of(b["tok_row"]).any()
    # the head cleared, the same call routes as the oracle does
    moe.moe_workspace_init(b["ws"])
    moe.moe_route(b["cfg"], up(l), b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                  b["row_token"], b["tok_row"], b["ws"])
    assert moe.moe_read_status(b["ws"]) == moe.MOE_OK
    idx, _ = oracle.route(l, w)
    counts, offsets, row_token, tok_row = oracle.permute(idx, w["E"])
    assert np.array_equal(np_of(b["topk_idx"]), idx)
    assert np.array_equal(np_of(b["row_token"]), row_token)
    assert np.array_equal(np_of(b["tok_row"]), tok_row)
