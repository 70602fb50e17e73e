"""Pins for the packed variable-length (varlen) oracle, checked without a GPU.

The pins tie ``oracle.forward_varlen`` / ``oracle.backward_varlen`` to
independent facts: a scalar brute force that walks the packed [T, H, D]
tensors token by token, the batched oracle on equal-length samples, the
isolation of samples (changing one sample changes no other sample's result),
and fp64 central differences.  Planted mistakes must each fail a pin.
"""
import math

import pytest
import torch

from oracle import attention as A
from oracle import grouped as G
from oracle import varlen as V

F64 = torch.float64


def rnd(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * std


CASES = [  # (cu_seqlens, H, H_kv, D)
    ([0, 3, 7], 2, 2, 3),
    ([0, 1, 1, 5, 6], 2, 1, 2),  # an empty sample and single-token samples; MQA
    ([0, 4], 4, 2, 2),
]


def pin_bruteforce(fwd):
    """Scalar loops over packed tokens: token t of sample [a, b) sees keys a..b-1 (a..t if causal)."""
    for cu, H, Hkv, D in CASES:
        T = cu[-1]
        q, k, v = rnd((T, H, D), 1 + T), rnd((T, Hkv, D), 2 + T), rnd((T, Hkv, D), 3 + T)
        grp = H // Hkv
        for causal in (False, True):
            o, lse = fwd(q, k, v, torch.tensor(cu), causal, 0.7)
            assert tuple(o.shape) == (T, H, D) and tuple(lse.shape) == (H, T)
            for a, b in zip(cu[:-1], cu[1:]):
                for t in range(a, b):
                    keys = range(a, t + 1) if causal else range(a, b)
                    for h in range(H):
                        g = h // grp
                        s = [0.7 * sum(float(q[t, h, d]) * float(k[j, g, d]) for d in range(D)) for j in keys]
                        m = max(s)
                        e = [math.exp(x - m) for x in s]
                        z = sum(e)
                        for d in range(D):
                            ref = sum(e[i] * float(v[j, g, d]) for i, j in enumerate(keys)) / z
                            assert abs(float(o[t, h, d]) - ref) < 1e-12, (cu, t, h, d)
                        assert abs(float(lse[h, t]) - (m + math.log(z))) < 1e-12, (cu, t, h)


def pin_equal_lengths_are_the_batched_problem(fwd, bwd):
    """B samples of length S packed back to back equal the [B, H, S, D] oracle, rearranged."""
    B, H, Hkv, S, D = 3, 4, 2, 5, 3
    qb, kb, vb, dob = rnd((B, H, S, D), 10), rnd((B, Hkv, S, D), 11), rnd((B, Hkv, S, D), 12), rnd((B, H, S, D), 13)
    pack = lambda x: x.permute(0, 2, 1, 3).reshape(B * S, x.shape[1], D)  # noqa: E731
    cu = torch.arange(0, B * S + 1, S)
    for causal in (False, True):
        o_ref, l_ref = G.forward_gqa(qb, kb, vb, causal, 0.5)
        o, lse = fwd(pack(qb), pack(kb), pack(vb), cu, causal, 0.5)
        assert torch.allclose(o, pack(o_ref), rtol=0, atol=1e-13)
        assert torch.allclose(lse, l_ref.permute(1, 0, 2).reshape(H, B * S), rtol=0, atol=1e-13)
        g_ref = G.backward_gqa(qb, kb, vb, dob, causal, 0.5)
        g = bwd(pack(qb), pack(kb), pack(vb), pack(dob), cu, causal, 0.5)
        for x, r in zip(g, g_ref):
            assert torch.allclose(x, pack(r), rtol=0, atol=1e-13)


def pin_samples_are_isolated(fwd, bwd):
    """Changing every input of one sample leaves the other samples' O, L and gradients bitwise unchanged."""
    cu = torch.tensor([0, 4, 9, 12])
    T, H, D = 12, 2, 3
    q, k, v, do = rnd((T, H, D), 20), rnd((T, H, D), 21), rnd((T, H, D), 22), rnd((T, H, D), 23)
    q2, k2, v2, do2 = (x.clone() for x in (q, k, v, do))
    for x, s in zip((q2, k2, v2, do2), (24, 25, 26, 27)):
        x[4:9] = rnd((5, H, D), s)
    keep = torch.tensor([t for t in range(T) if not 4 <= t < 9])
    for causal in (False, True):
        o1, l1 = fwd(q, k, v, cu, causal, 0.9)
        o2, l2 = fwd(q2, k2, v2, cu, causal, 0.9)
        assert torch.equal(o1[keep], o2[keep]) and torch.equal(l1[:, keep], l2[:, keep])
        assert not torch.allclose(o1[4:9], o2[4:9])
        g1 = bwd(q, k, v, do, cu, causal, 0.9)
        g2 = bwd(q2, k2, v2, do2, cu, causal, 0.9)
        for a, b in zip(g1, g2):
            assert torch.equal(a[keep], b[keep])


def pin_grad_central_differences(fwd, bwd):
    """dQ, dK, dV of loss = <O, dO> against fp64 central differences on a packed batch."""
    h = 1e-6
    cu = torch.tensor([0, 2, 2, 5])
    T, H, Hkv, D = 5, 2, 1, 2
    q, k, v, do = rnd((T, H, D), 30), rnd((T, Hkv, D), 31), rnd((T, Hkv, D), 32), rnd((T, H, D), 33)
    for causal in (False, True):
        grads = bwd(q, k, v, do, cu, causal, 0.8)
        for which, x in enumerate((q, k, v)):
            num = torch.zeros_like(x)
            flat = x.view(-1)
            for idx in range(flat.numel()):
                old = float(flat[idx])
                flat[idx] = old + h
                lp = float((fwd(q, k, v, cu, causal, 0.8)[0] * do).sum())
                flat[idx] = old - h
                lm = float((fwd(q, k, v, cu, causal, 0.8)[0] * do).sum())
                flat[idx] = old
                num.view(-1)[idx] = (lp - lm) / (2 * h)
            err = (grads[which] - num).abs().max() / max(1.0, float(num.abs().max()))
            assert err <= 1e-7, (causal, which, float(err))


FWD_PINS = [pin_bruteforce]
PAIR_PINS = [pin_equal_lengths_are_the_batched_problem, pin_samples_are_isolated, pin_grad_central_differences]


@pytest.mark.parametrize("pin", FWD_PINS, ids=lambda f: f.__name__)
def test_forward_pin(pin):
    pin(V.forward_varlen)


@pytest.mark.parametrize("pin", PAIR_PINS, ids=lambda f: f.__name__)
def test_pair_pin(pin):
    pin(V.forward_varlen, V.backward_varlen)


def test_bad_cu_seqlens():
    q = torch.zeros(4, 1, 2, dtype=F64)
    for cu in ([1, 4], [0, 3, 2, 4], []):
        with pytest.raises(ValueError):
            V.forward_varlen(q, q, q, torch.tensor(cu, dtype=torch.long), False, 1.0)


# ----------------------------------------------------------------------------------
# Planted mistakes.
# ----------------------------------------------------------------------------------

def _fwd_mut(kind):
    def f(q, k, v, cu, causal, scale):
        q, k, v = (A.as_f64(x) for x in (q, k, v))
        T, H, D = q.shape
        grp = H // k.shape[1]
        cu = [int(x) for x in cu.tolist()]
        o = torch.zeros(T, H, D, dtype=F64)
        lse = torch.zeros(H, T, dtype=F64)
        spans = [(0, T)] if kind == "no_sample_boundary" else list(zip(cu[:-1], cu[1:]))
        for a, b in spans:
            if a == b:
                continue
            for h in range(H):
                g = h // grp
                qa = q[a:b, h]
                ka = k[a:b, g] if kind != "keys_shifted" else k[min(a + 1, T - (b - a)):min(a + 1, T - (b - a)) + b - a, g]
                va = v[a:b, g]
                ob, lb = A.forward(qa, ka, va, causal, scale)
                o[a:b, h] = ob
                if kind == "lse_token_major":
                    lse.view(T, H)[a:b, h] = lb
                else:
                    lse[h, a:b] = lb
        return o, lse
    return f


def _bwd_mut(kind):
    def g(q, k, v, do, cu, causal, scale):
        q, k, v, do = (A.as_f64(x) for x in (q, k, v, do))
        dq, dk, dv = (torch.zeros(x.shape, dtype=F64) for x in (q, k, v))
        cu = [int(x) for x in cu.tolist()]
        # Samples in reverse order, as independent blocks of a parallel kernel
        # may finish: a write past a sample's end then clobbers its successor.
        for a, b in reversed(list(zip(cu[:-1], cu[1:]))):
            if a == b:
                continue
            r = G.backward_gqa(q[a:b].transpose(0, 1), k[a:b].transpose(0, 1), v[a:b].transpose(0, 1),
                               do[a:b].transpose(0, 1), causal, scale)
            dq[a:b] = r[0].transpose(0, 1)
            if kind == "dkv_overwrite_next":  # writes one row past the sample end too
                e = min(b + 1, q.shape[0])
                dk[a:e] = torch.cat([r[1].transpose(0, 1), torch.zeros(e - b, *dk.shape[1:], dtype=F64)])
                dv[a:e] = torch.cat([r[2].transpose(0, 1), torch.zeros(e - b, *dv.shape[1:], dtype=F64)])
            else:
                dk[a:b] = r[1].transpose(0, 1)
                dv[a:b] = r[2].transpose(0, 1)
        return dq, dk, dv
    return g


def _fails(fn):
    try:
        fn()
    except (AssertionError, RuntimeError):
        return True
    return False


@pytest.mark.parametrize("kind", ["no_sample_boundary", "keys_shifted", "lse_token_major"])
def test_planted_forward_mistake_is_caught(kind):
    f = _fwd_mut(kind)
    caught = [p.__name__ for p in FWD_PINS if _fails(lambda p=p: p(f))]
    caught += [p.__name__ for p in PAIR_PINS if _fails(lambda p=p: p(f, V.backward_varlen))]
    assert caught, f"planted forward mistake {kind!r} passed every pin"


@pytest.mark.parametrize("kind", ["dkv_overwrite_next"])
def test_planted_backward_mistake_is_caught(kind):
    g = _bwd_mut(kind)
    caught = [p.__name__ for p in PAIR_PINS if _fails(lambda p=p: p(V.forward_varlen, g))]
    assert caught, f"planted backward mistake {kind!r} passed every pin"


def test_unmutated_copies_pass():
    f, g = _fwd_mut("none"), _bwd_mut("none")
    for p in FWD_PINS:
        p(f)
    for p in PAIR_PINS:
        p(f, g)
