"""Host logic of the data-parallel layout: head shards and the cross-rank
timing reduction, run as two gloo ranks on the CPU; plus, on a GPU, a call on
one head shard (offset pointers) against the whole call."""
import os
import socket

import pytest
import torch

from exact_attention_18_gb300.sharding import job_throughput, max_over_ranks, shard_heads, shard_keys


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


@pytest.mark.parametrize("S", [0, 1, 127, 128, 1000, 4096])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_key_shards_cover_in_aligned_ranges(S, world):
    spans = [shard_keys(S, r, world) for r in range(world)]
    pos = 0
    for k0, k1 in spans:
        assert k0 == pos or k0 == k1 == S
        assert k0 % 128 == 0 or k0 == S
        pos = max(pos, k1)
    assert pos == S
    with pytest.raises(ValueError):
        shard_keys(10, 3, 3)


def _context_rank(rank, world, port, out_dir):
    """Context-parallel forward on the CPU: each rank attends every query to its key shard
    (the fp64 oracle stands in for the kernels), the partials are all-gathered, and the
    logsumexp merge must give the unsplit result."""
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = torch.Generator().manual_seed(5)
        q, k, v = (torch.randn(2, 300, 16, generator=g, dtype=torch.float64) for _ in range(3))
        k0, k1 = shard_keys(300, rank, world)
        o_s, l_s = oracle.forward_shards(q, k, v, True, 0.25, [(k0, k1)])
        o_all = [torch.empty_like(o_s) for _ in range(world)]
        l_all = [torch.empty_like(l_s) for _ in range(world)]
        dist.all_gather(o_all, o_s)
        dist.all_gather(l_all, l_s)
        o, lse = oracle.merge_lse(torch.cat(o_all), torch.cat(l_all))
        ref_o, ref_l = oracle.forward(q, k, v, True, 0.25)
        err = max(float((o - ref_o).abs().max()), float((lse - ref_l).abs().max()))
        with open(os.path.join(out_dir, f"ctx{rank}.txt"), "w") as f:
            f.write(repr((k0, k1, err)))
    finally:
        dist.destroy_process_group()


def test_context_parallel_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_context_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    results = [eval((tmp_path / f"ctx{r}.txt").read_text()) for r in range(world)]
    assert [(a, b) for a, b, _ in results] == [(0, 256), (256, 300)]
    for _, _, err in results:
        assert err < 1e-12


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
