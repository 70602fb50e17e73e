"""Pins for the oracle's window band (sliding-window attention), without a GPU.

``oracle.forward(..., window=(left, right))`` hides key j from query i unless
i - left <= j <= i + right (negative = unlimited).  The pins below tie it to
scalar brute force, to the unwindowed and causal oracles it must reduce to,
to the exact (0, 0) band, to the locality of the band (keys outside a row's
band cannot change it), and to fp64 central differences; planted mistakes
(an off-by-one edge, swapped sides, a dropped side) must each fail a pin.
"""
import math

import pytest
import torch

from oracle import attention as A

F64 = torch.float64


def rnd(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * std


def visible(i, j, causal, left, right):
    if causal and j > i:
        return False
    if left >= 0 and j < i - left:
        return False
    if right >= 0 and j > i + right:
        return False
    return True


BANDS = [(0, 0), (1, 0), (2, 3), (-1, 1), (3, -1), (0, 4)]


def pin_bruteforce(fwd):
    S, D = 7, 3
    q, k, v = rnd((1, 2, S, D), 1), rnd((1, 2, S, D), 2), rnd((1, 2, S, D), 3)
    for causal in (False, True):
        for left, right in BANDS:
            o, lse = fwd(q, k, v, causal, 0.8, (left, right))
            for h in range(2):
                for i in range(S):
                    keys = [j for j in range(S) if visible(i, j, causal, left, right)]
                    s = [0.8 * sum(float(q[0, h, i, d]) * float(k[0, h, j, d]) for d in range(D)) for j in keys]
                    m = max(s)
                    e = [math.exp(x - m) for x in s]
                    z = sum(e)
                    for d in range(D):
                        ref = sum(e[t] * float(v[0, h, j, d]) for t, j in enumerate(keys)) / z
                        assert abs(float(o[0, h, i, d]) - ref) < 1e-12, (causal, left, right, i, d)
                    assert abs(float(lse[0, h, i]) - (m + math.log(z))) < 1e-12


def pin_reductions(fwd):
    """Unlimited or wide bands are the plain oracle; (-1, 0) is the causal oracle (bitwise)."""
    q, k, v = rnd((2, 2, 9, 4), 10), rnd((2, 2, 9, 4), 11), rnd((2, 2, 9, 4), 12)
    for causal in (False, True):
        ref = A.forward(q, k, v, causal, 0.5)
        for band in ((-1, -1), (9, 9), (100, -1)):
            o, lse = fwd(q, k, v, causal, 0.5, band)
            assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1]), (causal, band)
    o, lse = fwd(q, k, v, False, 0.5, (-1, 0))
    ref = A.forward(q, k, v, True, 0.5)
    assert torch.equal(o, ref[0]) and torch.equal(lse, ref[1])


def pin_diagonal_band(fwd):
    """(0, 0): every row sees only its own key, so O_i = v_i and L_i = scale q_i . k_i."""
    q, k, v = rnd((1, 3, 6, 5), 20), rnd((1, 3, 6, 5), 21), rnd((1, 3, 6, 5), 22)
    for causal in (False, True):
        o, lse = fwd(q, k, v, causal, 0.7, (0, 0))
        assert torch.allclose(o, v, rtol=0, atol=1e-15)
        assert torch.allclose(lse, 0.7 * (q * k).sum(-1), rtol=0, atol=1e-13)


def pin_band_locality(fwd):
    """Row i depends only on keys i-left .. i+right: changing others leaves it bitwise unchanged."""
    S, D, left, right = 12, 3, 2, 1
    q, k, v = rnd((1, 1, S, D), 30), rnd((1, 1, S, D), 31), rnd((1, 1, S, D), 32)
    o1, l1 = fwd(q, k, v, False, 1.0, (left, right))
    i = 6
    k2, v2 = k.clone(), v.clone()
    outside = [j for j in range(S) if not (i - left <= j <= i + right)]
    k2[0, 0, outside] += 5.0
    v2[0, 0, outside] -= 3.0
    o2, l2 = fwd(q, k2, v2, False, 1.0, (left, right))
    assert torch.equal(o1[0, 0, i], o2[0, 0, i]) and torch.equal(l1[0, 0, i], l2[0, 0, i])
    k3 = k.clone()
    k3[0, 0, i - left] += 1.0  # the band's lower edge is inside
    _, l3 = fwd(q, k3, v, False, 1.0, (left, right))
    assert not torch.equal(l1[0, 0, i], l3[0, 0, i])
    k4 = k.clone()
    k4[0, 0, i + right] += 1.0  # and so is its upper edge
    _, l4 = fwd(q, k4, v, False, 1.0, (left, right))
    assert not torch.equal(l1[0, 0, i], l4[0, 0, i])


def pin_grad_central_differences(fwd, bwd):
    h = 1e-6
    for causal, band in ((False, (1, 2)), (True, (2, -1)), (False, (0, 1))):
        q, k, v, do = (rnd((1, 1, 6, 2), s) for s in (40, 41, 42, 43))
        grads = bwd(q, k, v, do, causal, 0.9, band)
        for which, x in enumerate((q, k, v)):
            num = torch.zeros_like(x)
            flat = x.view(-1)
            for idx in range(flat.numel()):
                old = float(flat[idx])
                flat[idx] = old + h
                lp = float((fwd(q, k, v, causal, 0.9, band)[0] * do).sum())
                flat[idx] = old - h
                lm = float((fwd(q, k, v, causal, 0.9, band)[0] * do).sum())
                flat[idx] = old
                num.view(-1)[idx] = (lp - lm) / (2 * h)
            err = (grads[which] - num).abs().max() / max(1.0, float(num.abs().max()))
            assert err <= 1e-7, (causal, band, which, float(err))


def pin_gradient_sums(bwd):
    q, k, v, do = (rnd((2, 2, 11, 4), s) for s in (50, 51, 52, 53))
    for causal, band in ((False, (3, 2)), (True, (4, -1))):
        dq, dk, dv = bwd(q, k, v, do, causal, 0.6, band)
        assert torch.allclose(dk.sum(-2), torch.zeros(2, 2, 4, dtype=F64), atol=1e-12)
        assert torch.allclose(dv.sum(-2), do.sum(-2), atol=1e-12)


def fwd_oracle(q, k, v, causal, scale, band):
    return A.forward(q, k, v, causal, scale, window=band)


def bwd_oracle(q, k, v, do, causal, scale, band):
    return A.backward(q, k, v, do, causal, scale, window=band)


FWD_PINS = [pin_bruteforce, pin_reductions, pin_diagonal_band, pin_band_locality]


@pytest.mark.parametrize("pin", FWD_PINS, ids=lambda f: f.__name__)
def test_forward_pin(pin):
    pin(fwd_oracle)


def test_central_differences_pin():
    pin_grad_central_differences(fwd_oracle, bwd_oracle)


def test_gradient_sums_pin():
    pin_gradient_sums(bwd_oracle)


# ----------------------------------------------------------------------------------
# Planted mistakes in the band.
# ----------------------------------------------------------------------------------

def _mut(kind):
    def f(q, k, v, causal, scale, band):
        left, right = band
        if kind == "swapped_sides":
            left, right = right, left
        elif kind == "right_side_dropped":
            right = -1
        q, k, v = (A.as_f64(x) for x in (q, k, v))
        s = scale * torch.matmul(q, k.transpose(-1, -2))
        n = s.shape[-1]
        qi = torch.arange(n).view(n, 1)
        kj = torch.arange(n).view(1, n)
        if causal:
            s = s.masked_fill(kj > qi, float("-inf"))
        off = 1 if kind == "edge_off_by_one" else 0
        if left >= 0:
            s = s.masked_fill(kj < qi - left + off, float("-inf"))
        if right >= 0:
            s = s.masked_fill(kj > qi + right, float("-inf"))
        p, lse = A.softmax_rows(s)
        return torch.matmul(p, v), lse
    return f


@pytest.mark.parametrize("kind", ["edge_off_by_one", "swapped_sides", "right_side_dropped"])
def test_planted_band_mistake_is_caught(kind):
    f = _mut(kind)
    caught = []
    for pin in FWD_PINS:
        try:
            pin(f)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"planted band mistake {kind!r} passed every pin"


def test_unmutated_copy_passes():
    f = _mut("none")
    for pin in FWD_PINS:
        pin(f)
