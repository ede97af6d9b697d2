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
