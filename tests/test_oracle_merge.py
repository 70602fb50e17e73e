"""Pins for the split-KV / logsumexp-merge oracle, without a GPU.

``oracle.merge_lse`` combines per-shard (O_s, L_s); ``oracle.forward_shards``
gives the partials of key ranges.  Pins: merging the shards of any split
reproduces the unsplit oracle (the identity the merge exists for); a closed
form for two one-key shards in scalar math; one shard is the identity; shard
order does not matter; empty shards carry no weight; rows with no key at all.
Planted mistakes in the merge must each fail a pin.
"""
import math

import pytest
import torch

from oracle import attention as A
from oracle import merge as M

F64 = torch.float64


def rnd(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * std


def pin_split_equals_whole(merge):
    q, k, v = rnd((2, 3, 13, 4), 1, 2.0), rnd((2, 3, 13, 4), 2, 2.0), rnd((2, 3, 13, 4), 3)
    for causal in (False, True):
        ref_o, ref_l = A.forward(q, k, v, causal, 0.6)
        for bounds in (M.split_bounds(13, 4), M.split_bounds(13, 1), [(0, 7), (7, 13)], [(0, 13)]):
            o_p, l_p = M.forward_shards(q, k, v, causal, 0.6, bounds)
            o, lse = merge(o_p, l_p)
            assert torch.allclose(o, ref_o, rtol=0, atol=1e-12), (causal, bounds)
            assert torch.allclose(lse, ref_l, rtol=0, atol=1e-12), (causal, bounds)


def pin_two_single_key_shards(merge):
    """Shards {key 0}, {key 1} of one row: L_s = s_j, O_s = v_j; the merge must be softmax of two."""
    s0, s1 = 0.7, -1.9
    v0, v1 = [1.0, -2.0], [3.5, 0.25]
    o_p = torch.tensor([[v0], [v1]], dtype=F64)      # [P=2, rows=1, D=2]
    l_p = torch.tensor([[s0], [s1]], dtype=F64)
    o, lse = merge(o_p, l_p)
    z = math.exp(s0) + math.exp(s1)
    for d in range(2):
        assert abs(float(o[0, d]) - (math.exp(s0) * v0[d] + math.exp(s1) * v1[d]) / z) < 1e-15
    assert abs(float(lse[0]) - math.log(z)) < 1e-15


def pin_identity_and_order(merge):
    o_p, l_p = rnd((4, 6, 5), 10), rnd((4, 6), 11, 3.0)
    o1, l1 = merge(o_p[:1], l_p[:1])
    assert torch.allclose(o1, o_p[0], rtol=0, atol=1e-15) and torch.allclose(l1, l_p[0], rtol=0, atol=1e-15)
    perm = torch.tensor([2, 0, 3, 1])
    o2, l2 = merge(o_p, l_p)
    o3, l3 = merge(o_p[perm], l_p[perm])
    assert torch.allclose(o2, o3, rtol=0, atol=1e-14) and torch.allclose(l2, l3, rtol=0, atol=1e-14)


def pin_empty_shards(merge):
    """A shard with L = -inf (and O = 0) changes nothing; rows with every shard empty give O = 0, L = -inf."""
    o_p, l_p = rnd((3, 4, 5), 20), rnd((3, 4), 21)
    o_ref, l_ref = merge(o_p[:2], l_p[:2])
    o_e = torch.cat([o_p[:2], torch.zeros(1, 4, 5, dtype=F64)])
    l_e = torch.cat([l_p[:2], torch.full((1, 4), float("-inf"), dtype=F64)])
    o, lse = merge(o_e, l_e)
    assert torch.allclose(o, o_ref, rtol=0, atol=1e-15) and torch.allclose(lse, l_ref, rtol=0, atol=1e-15)
    o, lse = merge(torch.zeros(2, 3, 5, dtype=F64), torch.full((2, 3), float("-inf"), dtype=F64))
    assert torch.equal(o, torch.zeros(3, 5, dtype=F64)) and bool(torch.all(torch.isneginf(lse)))


PINS = [pin_split_equals_whole, pin_two_single_key_shards, pin_identity_and_order, pin_empty_shards]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_merge_pin(pin):
    pin(M.merge_lse)


def test_split_bounds_cover_the_keys():
    assert M.split_bounds(10, 4) == [(0, 4), (4, 8), (8, 10)]
    assert M.split_bounds(8, 8) == [(0, 8)]


def _mut(kind):
    def f(o_p, l_p):
        o_p, l_p = A.as_f64(o_p), A.as_f64(l_p)
        m = l_p.amax(0)
        if kind == "linear_weights":
            w = l_p - m + 1.0
        else:
            w = torch.exp(l_p - m)
        total = w.sum(0)
        if kind == "lse_is_max":
            lse = m
        else:
            lse = m + torch.log(total)
        if kind == "unnormalised":
            o = (w.unsqueeze(-1) * o_p).sum(0)
        else:
            o = ((w / total).unsqueeze(-1) * o_p).sum(0)
        return o, lse
    return f


@pytest.mark.parametrize("kind", ["linear_weights", "lse_is_max", "unnormalised"])
def test_planted_merge_mistake_is_caught(kind):
    f = _mut(kind)
    caught = []
    for pin in PINS[:3]:  # the -inf pin needs the guarded form; the first three pin the arithmetic
        try:
            pin(f)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"planted merge mistake {kind!r} passed every pin"
