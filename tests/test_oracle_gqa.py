"""Pins for the grouped-query (GQA / MQA) oracle, checked without a GPU.

Each pin ties ``oracle.forward_gqa`` / ``oracle.backward_gqa`` to something
other than their own formula: exact values for inputs built so the answer is
known in closed form (constant V rows, zero keys), the K/V-head sums that the
softmax fixes, brute-force loops, and fp64 central differences.  Planted
mistakes (the other head map, one head of a group, a mean instead of a sum)
must each fail at least one pin.
"""
import math

import pytest
import torch

from oracle import attention as A
from oracle import grouped as G

F64 = torch.float64


def rnd(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * std


# ----------------------------------------------------------------------------------
# Pins, parameterised by the implementation.
# ----------------------------------------------------------------------------------

def pin_constant_values_name_the_kv_head(fwd):
    """Rows of V_g all equal to c_g make O_h = c_{h // G} exactly (softmax weights sum to 1)."""
    B, H, Hkv, S, D = 2, 6, 2, 5, 3
    q, k = rnd((B, H, S, D), 1), rnd((B, Hkv, S, D), 2)
    c = torch.tensor([[[100.0 * b + 10.0 * (g + 1) + d for d in range(D)] for g in range(Hkv)]
                      for b in range(B)], dtype=F64)
    v = c.view(B, Hkv, 1, D).expand(B, Hkv, S, D).contiguous()
    for causal in (False, True):
        o, _ = fwd(q, k, v, causal, 0.7)
        for b in range(B):
            for h in range(H):
                want = c[b, h // (H // Hkv)].view(1, D).expand(S, D)
                assert torch.allclose(o[b, h], want, rtol=0, atol=1e-12), (b, h, causal)


def pin_zero_keys_give_log_count(fwd):
    """K_0 = 0 makes every score of group 0 zero: L_i = ln(visible keys), O_i = mean of visible V rows."""
    B, H, Hkv, S, D = 1, 4, 2, 6, 2
    q, v = rnd((B, H, S, D), 3), rnd((B, Hkv, S, D), 4)
    k = rnd((B, Hkv, S, D), 5)
    k[:, 0] = 0
    grp = H // Hkv
    for causal in (False, True):
        o, lse = fwd(q, k, v, causal, 1.3)
        for i in range(S):
            n = i + 1 if causal else S
            for h in range(grp):  # group 0
                assert abs(float(lse[0, h, i]) - math.log(n)) < 1e-12, (h, i, causal)
                assert torch.allclose(o[0, h, i], v[0, 0, :n].mean(0), rtol=0, atol=1e-12)
            for h in range(grp, H):  # group 1 has random keys
                if n > 1:
                    assert abs(float(lse[0, h, i]) - math.log(n)) > 1e-6, (h, i, causal)


def pin_bruteforce(fwd):
    """Scalar loops over (b, h, i) with K/V head h // G, on tiny inputs, incl. MQA."""
    for B, H, Hkv, S, D in [(1, 4, 2, 4, 3), (2, 3, 1, 3, 2), (1, 2, 2, 3, 2)]:
        q, k, v = rnd((B, H, S, D), 6 + H), rnd((B, Hkv, S, D), 7 + H), rnd((B, Hkv, S, D), 8 + H)
        grp = H // Hkv
        for causal in (False, True):
            o, lse = fwd(q, k, v, causal, 0.6)
            for b in range(B):
                for h in range(H):
                    g = h // grp
                    for i in range(S):
                        keys = range(i + 1) if causal else range(S)
                        s = [0.6 * sum(float(q[b, h, i, d]) * float(k[b, g, j, d]) for d in range(D)) for j in keys]
                        m = max(s)
                        e = [math.exp(x - m) for x in s]
                        z = sum(e)
                        for d in range(D):
                            ref = sum(e[t] * float(v[b, g, j, d]) for t, j in enumerate(keys)) / z
                            assert abs(float(o[b, h, i, d]) - ref) < 1e-12
                        assert abs(float(lse[b, h, i]) - (m + math.log(z))) < 1e-12


def pin_grad_central_differences(fwd, bwd):
    """dQ, dK, dV of loss = <O, dO> against fp64 central differences (GQA and MQA)."""
    h = 1e-6
    for causal in (False, True):
        for B, H, Hkv, S, D in [(1, 4, 2, 4, 2), (1, 3, 1, 3, 2)]:
            q, k, v = rnd((B, H, S, D), 20 + H), rnd((B, Hkv, S, D), 21 + H), rnd((B, Hkv, S, D), 22 + H)
            do = rnd((B, H, S, D), 23 + H)
            grads = bwd(q, k, v, do, causal, 0.8)
            for which, x in enumerate((q, k, v)):
                assert grads[which].shape == x.shape, (which, tuple(grads[which].shape))
                num = torch.zeros_like(x)
                flat = x.view(-1)
                for idx in range(flat.numel()):
                    old = float(flat[idx])
                    flat[idx] = old + h
                    lp = float((fwd(q, k, v, causal, 0.8)[0] * do).sum())
                    flat[idx] = old - h
                    lm = float((fwd(q, k, v, causal, 0.8)[0] * do).sum())
                    flat[idx] = old
                    num.view(-1)[idx] = (lp - lm) / (2 * h)
                err = (grads[which] - num).abs().max() / max(1.0, float(num.abs().max()))
                assert err <= 1e-7, (causal, H, Hkv, which, float(err))


def pin_group_sums(bwd):
    """Per K/V head: sum_j dK_g[j] = 0 and sum_j dV_g[j] = sum of dO over the group's query heads."""
    B, H, Hkv, S, D = 2, 6, 3, 7, 4
    q, do = rnd((B, H, S, D), 30), rnd((B, H, S, D), 31)
    k, v = rnd((B, Hkv, S, D), 32), rnd((B, Hkv, S, D), 33)
    grp = H // Hkv
    for causal in (False, True):
        dq, dk, dv = bwd(q, k, v, do, causal, 0.5)
        assert torch.allclose(dk.sum(-2), torch.zeros(B, Hkv, D, dtype=F64), atol=1e-12)
        want = do.sum(-2).view(B, Hkv, grp, D).sum(2)
        assert torch.allclose(dv.sum(-2), want, atol=1e-12)


def pin_single_group_member_is_mha(fwd, bwd):
    """H_kv = H (one query head per K/V head) is the multi-head oracle, unchanged."""
    q, k, v, do = (rnd((2, 3, 5, 4), s) for s in (40, 41, 42, 43))
    for causal in (False, True):
        o1, l1 = fwd(q, k, v, causal, 0.5)
        o2, l2 = A.forward(q, k, v, causal, 0.5)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        for x, y in zip(bwd(q, k, v, do, causal, 0.5), A.backward(q, k, v, do, causal, 0.5)):
            assert torch.equal(x, y)


FWD_PINS = [pin_constant_values_name_the_kv_head, pin_zero_keys_give_log_count, pin_bruteforce]
BWD_PINS = [pin_group_sums]
PAIR_PINS = [pin_grad_central_differences, pin_single_group_member_is_mha]


@pytest.mark.parametrize("pin", FWD_PINS, ids=lambda f: f.__name__)
def test_forward_pin(pin):
    pin(G.forward_gqa)


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(G.backward_gqa)


@pytest.mark.parametrize("pin", PAIR_PINS, ids=lambda f: f.__name__)
def test_pair_pin(pin):
    pin(G.forward_gqa, G.backward_gqa)


def test_group_size_checks():
    assert G.group_size(32, 4) == 8  # the page's example: 32 query heads on 4 K/V heads
    for h, hk in [(6, 4), (4, 0), (3, 6)]:
        with pytest.raises(ValueError):
            G.group_size(h, hk)


# ----------------------------------------------------------------------------------
# Planted mistakes: each must fail at least one pin.
# ----------------------------------------------------------------------------------

def _expand(x, h_q, kind):
    hk = x.shape[-3]
    grp = h_q // hk
    if kind == "kv_modulo":  # query head h reads K/V head h % H_kv
        idx = torch.arange(h_q) % hk
    elif kind == "kv_first_only":
        idx = torch.zeros(h_q, dtype=torch.long)
    else:
        idx = torch.arange(h_q) // grp
    return A.as_f64(x).index_select(-3, idx)


def _fwd_mut(kind):
    def f(q, k, v, causal, scale):
        h_q = q.shape[-3]
        return A.forward(q, _expand(k, h_q, kind), _expand(v, h_q, kind), causal, scale)
    return f


def _bwd_mut(kind):
    def g(q, k, v, do, causal, scale):
        h_q, hk = q.shape[-3], k.shape[-3]
        grp = h_q // hk
        dq, dk_h, dv_h = A.backward(q, _expand(k, h_q, "none"), _expand(v, h_q, "none"), do, causal, scale)
        lead, s, d = dk_h.shape[:-3], dk_h.shape[-2], dk_h.shape[-1]
        if kind == "dkv_first_of_group":
            dk = dk_h.reshape(*lead, hk, grp, s, d)[..., 0, :, :]
            dv = dv_h.reshape(*lead, hk, grp, s, d)[..., 0, :, :]
        elif kind == "dkv_mean":
            dk = dk_h.reshape(*lead, hk, grp, s, d).mean(-3)
            dv = dv_h.reshape(*lead, hk, grp, s, d).mean(-3)
        elif kind == "dkv_sum_by_modulo":  # sums heads h with h % H_kv = g
            dk = dk_h.reshape(*lead, grp, hk, s, d).sum(-4)
            dv = dv_h.reshape(*lead, grp, hk, s, d).sum(-4)
        else:
            dk = dk_h.reshape(*lead, hk, grp, s, d).sum(-3)
            dv = dv_h.reshape(*lead, hk, grp, s, d).sum(-3)
        return dq, dk, dv
    return g


def _fails(fn):
    try:
        fn()
    except (AssertionError, RuntimeError):
        return True
    return False


@pytest.mark.parametrize("kind", ["kv_modulo", "kv_first_only"])
def test_planted_forward_mistake_is_caught(kind):
    f = _fwd_mut(kind)
    caught = [p.__name__ for p in FWD_PINS if _fails(lambda p=p: p(f))]
    assert caught, f"planted forward mistake {kind!r} passed every pin"


@pytest.mark.parametrize("kind", ["dkv_first_of_group", "dkv_mean", "dkv_sum_by_modulo"])
def test_planted_backward_mistake_is_caught(kind):
    g = _bwd_mut(kind)
    caught = [p.__name__ for p in BWD_PINS if _fails(lambda p=p: p(g))]
    caught += [p.__name__ for p in PAIR_PINS if _fails(lambda p=p: p(G.forward_gqa, g))]
    assert caught, f"planted backward mistake {kind!r} passed every pin"


def test_unmutated_copies_pass():
    f, g = _fwd_mut("none"), _bwd_mut("none")
    for p in FWD_PINS:
        p(f)
    for p in BWD_PINS:
        p(g)
    for p in PAIR_PINS:
        p(f, g)
