"""The multi-GPU form of the path, on CPU: token-sharded replicas with no data-path
collective. Two gloo ranks exercise the host logic bench.py uses under torchrun (per-rank
token shard, max-over-ranks time, whole-job throughput, rank-0-only reference arm), and the
oracle shows why replicas are exact: the layer routes and transforms every token on its own,
so two shards give the same outputs as one batch of both."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w_, r_, l_ = bench.rank_env()
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
    m = bench.max_over_ranks(local_ms, dist, "cpu")
    val = bench.job_tokens_per_s(w_, 4096, 3, m)
    x = synth.normal(bench.shard_seed(rank), synth.X, (4, 8), 1.0, "f32")
    xs = [torch.zeros(4, 8) for _ in range(world)]
    dist.all_gather(xs, torch.from_numpy(x))
    dist.destroy_process_group()
    out.put((rank, w_, r_, m, val, torch.stack(xs).numpy()))


def test_two_gloo_ranks_time_and_shards():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, world, r, m, val, shards in res:
        assert world == 2 and r == rank
        assert m == 15.0  # the slowest rank's time
        assert val == pytest.approx(2 * 4096 * 3 / 0.015)
        assert not np.array_equal(shards[0], shards[1])  # distinct token shards


def test_reference_arm_only_on_rank0(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"steps": 1, "warmup": 3, "cpu_tokens": 1})()
    assert bench.run_reference(args, synth.WORKLOADS["tiny_fp32"]) is None


def test_shards_equal_one_batch():
    """Replicas are exact: the layer on two token shards == the layer on their union."""
    w = synth.scaled(synth.WORKLOADS["dsv3_bf16"], T=48, H=128, E=16, F=128, F_shared=128,
                     n_groups=4, topk_groups=2)
    inp = synth.host_inputs(w, seed=0)
    full = oracle.forward(w, inp)["y"]
    parts = []
    for lo, hi in [(0, 20), (20, 48)]:
        sub = dict(inp, x=inp["x"][lo:hi])
        parts.append(oracle.forward(dict(w, T=hi - lo), sub)["y"])
    assert np.array_equal(np.concatenate(parts), full)
