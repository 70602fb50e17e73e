"""Host logic of the data-parallel layout: head shards and the cross-rank
timing reduction, run as two gloo ranks on the CPU; plus, on a GPU, a call on
one head shard (offset pointers) against the whole call."""
import os
import socket

import pytest
import torch

from exact_attention_18_gb300.sharding import job_throughput, max_over_ranks, shard_heads


@pytest.mark.parametrize("bh", [0, 1, 2, 7, 64, 1001])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shards_are_contiguous_disjoint_and_cover(bh, world):
    spans = [shard_heads(bh, r, world) for r in range(world)]
    pos = 0
    for start, count in spans:
        assert start == pos and count >= 0
        pos += count
    assert pos == bh
    counts = [c for _, c in spans]
    assert max(counts) - min(counts) <= 1


def test_shard_arguments_are_checked():
    with pytest.raises(ValueError):
        shard_heads(4, 2, 2)
    with pytest.raises(ValueError):
        shard_heads(4, 0, 0)
    with pytest.raises(ValueError):
        shard_heads(-1, 0, 1)


def test_single_process_reduction_and_rate():
    assert max_over_ranks(3.5) == 3.5
    # 2 ranks x 1e12 units per step x 10 steps in 5 ms -> 4e15 units/s
    assert job_throughput(1e12, 10, 2, 5.0) == pytest.approx(4e15)
    with pytest.raises(ValueError):
        job_throughput(1.0, 1, 1, 0.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bh = 7
        start, count = shard_heads(bh, rank, world)
        got = [None] * world
        dist.all_gather_object(got, (start, count))
        # The ranks' times differ; every rank must see the slowest.
        t_max = max_over_ranks(1.0 + rank, dist)
        rate = job_throughput(2.0, 3, world, t_max)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr((got, t_max, rate)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    results = [eval((tmp_path / f"rank{r}.txt").read_text()) for r in range(world)]
    for got, t_max, rate in results:
        assert got == [(0, 4), (4, 3)]
        assert t_max == 2.0
        assert rate == pytest.approx(world * 2.0 * 3 / 2e-3)


@pytest.mark.gpu
def test_head_shard_call_matches_whole_call():
    import exact_attention_18_gb300 as fa
    from seeded_inputs import Workload, make_inputs
    w = Workload("shard", 2, 3, 200, 64, "fp16", True, backward=True, seed=3)
    inp = make_inputs(w)
    dev = torch.device("cuda:0")
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    flat = lambda x: x.reshape(w.B * w.H, *x.shape[2:])
    for rank in range(2):
        start, count = shard_heads(w.B * w.H, rank, 2)
        sl = lambda x: flat(x)[start:start + count].unsqueeze(0)  # [1, count, S, D] view, offset pointer
        o_s, l_s = fa.forward(sl(q), sl(k), sl(v), causal=True, scale=w.scale)
        g_s = fa.backward(sl(q), sl(k), sl(v), o_s, sl(do), l_s, causal=True, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(o_s, sl(o)) and torch.equal(l_s, flat(lse)[start:start + count].unsqueeze(0))
        for a, b in zip(g_s, (dq, dk, dv)):
            assert torch.equal(a, sl(b))
