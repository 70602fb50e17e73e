"""Pins for the CPU fp64 oracle: values, closed forms and invariants fixed by the pages
and by the mathematics, not by the oracle itself.

Each pin is a function of the implementation under test, so the same pins are
also run against copies of the oracle with a planted mistake (a dropped term, a
wrong sign, a transposed operand, a wrong mask or loop bound); every planted
mistake must fail at least one pin.
"""
import json
import math
import os
import random

import pytest
import torch

import oracle
from oracle import attention as A
from oracle import online_softmax as OS

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "t5_worked_example.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def rnd(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=F64) * std


# ----------------------------------------------------------------------------------
# Closed forms computed here with scalar math, independent of the oracle's tensors.
# ----------------------------------------------------------------------------------

def closed_form_row(s, v):
    """Softmax weights, output and natural-log LSE of one score row (scalar math)."""
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    p = [x / z for x in e]
    o = sum(pi * vi for pi, vi in zip(p, v))
    return p, o, m + math.log(z)


def brute_force(q, k, v, causal, scale):
    """Pure-Python loops over every (b, h, i): O and L from the definition."""
    B, H, S, D = q.shape
    Sk = k.shape[2]
    o = torch.zeros(B, H, S, D, dtype=F64)
    lse = torch.zeros(B, H, S, dtype=F64)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                keys = range(Sk) if not causal else range(min(i + 1, Sk))
                s = [scale * sum(float(q[b, h, i, d]) * float(k[b, h, j, d]) for d in range(D))
                     for j in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                for d in range(D):
                    o[b, h, i, d] = sum(e[t] * float(v[b, h, j, d]) for t, j in enumerate(keys)) / z
                lse[b, h, i] = m + math.log(z)
    return o, lse


# ----------------------------------------------------------------------------------
# Pins, parameterised by the implementation (fwd, bwd, blockwise).
# Each returns normally on success and raises AssertionError on failure.
# ----------------------------------------------------------------------------------

def pin_worked_example(fwd, bwd):
    g = golden()["worked_example"]
    q = torch.tensor([[[[1.0]]]], dtype=F64)
    k = torch.tensor(g["scores"], dtype=F64).view(1, 1, 4, 1)
    v = torch.tensor(g["v"], dtype=F64).view(1, 1, 4, 1)
    p, o_ref, l_ref = closed_form_row(g["scores"], g["v"])
    o, lse = fwd(q, k, v, False, 1.0)
    assert abs(float(o[0, 0, 0, 0]) - o_ref) < 1e-12, (float(o), o_ref)
    assert abs(float(lse[0, 0, 0]) - l_ref) < 1e-12
    # dO = 1: dP_j = v_j, rowsum(P o dP) = O, so dS_j = P_j (v_j - O); dV_j = P_j.
    do = torch.ones(1, 1, 1, 1, dtype=F64)
    dq, dk, dv = bwd(q, k, v, do, False, 1.0)
    ds = [pj * (vj - o_ref) for pj, vj in zip(p, g["v"])]
    assert abs(float(dq[0, 0, 0, 0]) - sum(d * kj for d, kj in zip(ds, g["scores"]))) < 1e-11
    for j in range(4):
        assert abs(float(dv[0, 0, j, 0]) - p[j]) < 1e-12
        assert abs(float(dk[0, 0, j, 0]) - ds[j] * 1.0) < 1e-11


def pin_bruteforce(fwd):
    for causal in (False, True):
        for seed, (S, D) in enumerate([(5, 3), (7, 2), (4, 4)]):
            q, k, v = rnd((1, 2, S, D), 10 + seed), rnd((1, 2, S, D), 20 + seed), rnd((1, 2, S, D), 30 + seed)
            scale = 0.7
            o_ref, l_ref = brute_force(q, k, v, causal, scale)
            o, lse = fwd(q, k, v, causal, scale)
            assert torch.allclose(o, o_ref, atol=1e-12, rtol=0), (causal, S, D)
            assert torch.allclose(lse, l_ref, atol=1e-12, rtol=0), (causal, S, D)


def pin_uniform_scores(fwd):
    S, D = 9, 3
    q = torch.zeros(1, 1, S, D, dtype=F64)
    k, v = rnd((1, 1, S, D), 1), rnd((1, 1, S, D), 2)
    o, lse = fwd(q, k, v, False, 0.5)
    assert torch.allclose(o[0, 0], v[0, 0].mean(0).expand(S, D), atol=1e-13)
    assert torch.allclose(lse, torch.full((1, 1, S), math.log(S), dtype=F64), atol=1e-13)
    o, lse = fwd(q, k, v, True, 0.5)
    for i in range(S):
        assert torch.allclose(o[0, 0, i], v[0, 0, : i + 1].mean(0), atol=1e-13), i
        assert abs(float(lse[0, 0, i]) - math.log(i + 1)) < 1e-13


def pin_causal_first_row(fwd):
    q, k, v = rnd((2, 2, 6, 4), 3), rnd((2, 2, 6, 4), 4), rnd((2, 2, 6, 4), 5)
    o, lse = fwd(q, k, v, True, 0.5)
    assert torch.equal(o[:, :, 0], v[:, :, 0]) or torch.allclose(o[:, :, 0], v[:, :, 0], atol=1e-15)
    s00 = 0.5 * (q[:, :, 0] * k[:, :, 0]).sum(-1)
    assert torch.allclose(lse[:, :, 0], s00, atol=1e-14)


def pin_rows_sum_to_one(fwd):
    for causal in (False, True):
        q, k = rnd((1, 3, 11, 5), 6, 2.0), rnd((1, 3, 11, 5), 7, 2.0)
        v = torch.ones(1, 3, 11, 5, dtype=F64)
        o, _ = fwd(q, k, v, causal, 0.9)
        assert torch.allclose(o, torch.ones_like(o), atol=1e-13)


def pin_key_shift(fwd):
    """Adding one vector c to every key shifts row i's scores by scale*q_i.c: same O, L + that."""
    q, k, v = rnd((1, 2, 8, 4), 8), rnd((1, 2, 8, 4), 9), rnd((1, 2, 8, 4), 10)
    c = rnd((4,), 11)
    for causal in (False, True):
        o1, l1 = fwd(q, k, v, causal, 0.6)
        o2, l2 = fwd(q, k + c, v, causal, 0.6)
        assert torch.allclose(o1, o2, atol=1e-12)
        assert torch.allclose(l2, l1 + 0.6 * (q * c).sum(-1), atol=1e-12)


def pin_key_permutation(fwd):
    q, k, v = rnd((1, 2, 7, 3), 12), rnd((1, 2, 7, 3), 13), rnd((1, 2, 7, 3), 14)
    perm = torch.tensor([3, 0, 6, 1, 5, 2, 4])
    o1, l1 = fwd(q, k, v, False, 0.8)
    o2, l2 = fwd(q, k[:, :, perm], v[:, :, perm], False, 0.8)
    assert torch.allclose(o1, o2, atol=1e-12) and torch.allclose(l1, l2, atol=1e-12)


def pin_causal_independence(fwd):
    """Row i never sees keys j > i: changing K, V rows after i leaves O_i, L_i unchanged."""
    q, k, v = rnd((1, 1, 8, 3), 15), rnd((1, 1, 8, 3), 16), rnd((1, 1, 8, 3), 17)
    o1, l1 = fwd(q, k, v, True, 1.0)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 5:] += 3.0
    v2[:, :, 5:] -= 2.0
    o2, l2 = fwd(q, k2, v2, True, 1.0)
    assert torch.equal(o1[:, :, :5], o2[:, :, :5]) and torch.equal(l1[:, :, :5], l2[:, :, :5])
    assert not torch.allclose(o1[:, :, 5:], o2[:, :, 5:])


def pin_grad_central_differences(fwd, bwd):
    """dQ, dK, dV of loss = <O, dO> against fp64 central differences, h = 1e-6."""
    h = 1e-6
    for causal in (False, True):
        for S, D in [(1, 2), (3, 1), (5, 4), (8, 2)]:
            q, k, v = rnd((1, 2, S, D), 40 + S), rnd((1, 2, S, D), 50 + S), rnd((1, 2, S, D), 60 + S)
            do = rnd((1, 2, S, D), 70 + S)
            scale = 0.9
            grads = bwd(q, k, v, do, causal, scale)
            for which, x in enumerate((q, k, v)):
                num = torch.zeros_like(x)
                flat = x.view(-1)
                for idx in range(flat.numel()):
                    old = float(flat[idx])
                    flat[idx] = old + h
                    lp = float((fwd(q, k, v, causal, scale)[0] * do).sum())
                    flat[idx] = old - h
                    lm = float((fwd(q, k, v, causal, scale)[0] * do).sum())
                    flat[idx] = old
                    num.view(-1)[idx] = (lp - lm) / (2 * h)
                err = (grads[which] - num).abs().max() / max(1.0, float(num.abs().max()))
                assert err <= 1e-7, (causal, S, D, which, float(err))


def pin_gradient_sums(bwd):
    """sum_j dS_ij = 0 gives sum_j dK_j = 0; rows of P sum to 1 give sum_j dV_j = sum_i dO_i."""
    for causal in (False, True):
        q, k, v, do = (rnd((2, 2, 13, 6), s) for s in (80, 81, 82, 83))
        dq, dk, dv = bwd(q, k, v, do, causal, 0.4)
        assert torch.allclose(dk.sum(-2), torch.zeros(2, 2, 6, dtype=F64), atol=1e-12)
        assert torch.allclose(dv.sum(-2), do.sum(-2), atol=1e-12)


def pin_dv_causal_tail(bwd):
    """If dO rows >= t are zero, dK and dV rows >= t are exactly zero under the causal mask."""
    q, k, v, do = (rnd((1, 1, 9, 3), s) for s in (90, 91, 92, 93))
    do[:, :, 6:] = 0
    dq, dk, dv = bwd(q, k, v, do, True, 1.0)
    assert torch.count_nonzero(dk[:, :, 6:]) == 0 and torch.count_nonzero(dv[:, :, 6:]) == 0
    assert torch.count_nonzero(dv[:, :, :6]) > 0


def pin_blockwise_trace(blockwise):
    """The worked example's block-by-block state, derived by hand from the recurrence."""
    g = golden()["worked_example"]
    q = torch.tensor([[[[1.0]]]], dtype=F64)
    k = torch.tensor(g["scores"], dtype=F64).view(1, 1, 4, 1)
    v = torch.tensor(g["v"], dtype=F64).view(1, 1, 4, 1)
    tr = []
    o, lse = blockwise(q, k, v, False, 1.0, 1, g["block_n"], tr)
    assert len(tr) == 2
    e = math.exp
    # block 0: scores [1, 2] -> m = 2, alpha = exp(-inf) = 0 (the page's statement)
    assert float(tr[0]["alpha"]) == g["first_block_alpha"]
    assert float(tr[0]["m"]) == 2.0
    assert abs(float(tr[0]["l"]) - (e(-1) + 1.0)) < 1e-14
    assert abs(float(tr[0]["acc"]) - (10 * e(-1) + 20)) < 1e-13
    # block 1: scores [3, 0] -> m = 3, alpha = e^-1
    assert float(tr[1]["m"]) == 3.0
    assert abs(float(tr[1]["alpha"]) - e(-1)) < 1e-15
    l1 = e(-1) * (e(-1) + 1.0) + 1.0 + e(-3)
    acc1 = e(-1) * (10 * e(-1) + 20) + 30 + 40 * e(-3)
    assert abs(float(tr[1]["l"]) - l1) < 1e-14
    assert abs(float(tr[1]["acc"]) - acc1) < 1e-12
    _, o_ref, l_ref = closed_form_row(g["scores"], g["v"])
    assert abs(float(o) - o_ref) < 1e-12 and abs(float(lse) - l_ref) < 1e-12


def pin_blockwise_matches_definition(blockwise):
    rng = random.Random(5)
    for trial in range(12):
        S = rng.choice([1, 5, 16, 37, 64])
        D = rng.choice([1, 3, 8])
        bm, bn = rng.choice([1, 2, 5, 16, 32]), rng.choice([1, 3, 4, 16, 64])
        causal = bool(trial % 2)
        q, k, v = (rnd((1, 2, S, D), 100 + trial * 3 + t, 1.5) for t in range(3))
        o_ref, l_ref = brute_force(q, k, v, causal, 0.7) if S <= 16 else A.forward(q, k, v, causal, 0.7)
        o, lse = blockwise(q, k, v, causal, 0.7, bm, bn)
        assert torch.allclose(o, o_ref, atol=1e-12), (S, D, bm, bn, causal)
        assert torch.allclose(lse, l_ref, atol=1e-12), (S, D, bm, bn, causal)


FWD_PINS = [pin_bruteforce, pin_uniform_scores, pin_causal_first_row, pin_rows_sum_to_one,
            pin_key_shift, pin_key_permutation, pin_causal_independence]
BWD_PINS = [pin_worked_example, pin_grad_central_differences]
GRAD_PINS = [pin_gradient_sums, pin_dv_causal_tail]


# ----------------------------------------------------------------------------------
# The oracle passes every pin.
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("pin", FWD_PINS, ids=lambda f: f.__name__)
def test_forward_pin(pin):
    pin(A.forward)


@pytest.mark.parametrize("pin", BWD_PINS, ids=lambda f: f.__name__)
def test_forward_backward_pin(pin):
    pin(A.forward, A.backward)


@pytest.mark.parametrize("pin", GRAD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(A.backward)


def test_blockwise_trace_pin():
    pin_blockwise_trace(OS.forward_blockwise)


def test_blockwise_matches_definition_pin():
    pin_blockwise_matches_definition(OS.forward_blockwise)


def test_delta_identity():
    """rowsum(dO o O) equals the Jacobian row term rowsum(P o dP)."""
    for causal in (False, True):
        q, k, v, do = (rnd((2, 3, 17, 8), s) for s in (120, 121, 122, 123))
        o, _ = A.forward(q, k, v, causal, 0.35)
        p, _ = A.softmax_rows(A.scores(q, k, 0.35, causal))
        dp = torch.matmul(do, v.transpose(-1, -2))
        assert torch.allclose(A.delta(o, do), (p * dp).sum(-1), atol=1e-12)


def test_library_special_case_sdpa():
    """torch's own scaled_dot_product_attention and autograd in float64 agree with the oracle."""
    import torch.nn.functional as Fn
    for causal in (False, True):
        q, k, v, do = (rnd((2, 3, 33, 16), s) for s in (130, 131, 132, 133))
        q.requires_grad_(True), k.requires_grad_(True), v.requires_grad_(True)
        o_t = Fn.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=0.25)
        o_t.backward(do)
        s = 0.25 * q.detach() @ k.detach().transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), float("-inf"))
        l_t = torch.logsumexp(s, dim=-1)
        o, lse = A.forward(q, k, v, causal, 0.25)
        dq, dk, dv = A.backward(q, k, v, do, causal, 0.25)
        assert torch.allclose(o, o_t.detach(), atol=1e-12)
        assert torch.allclose(lse, l_t, atol=1e-12)
        assert torch.allclose(dq, q.grad, atol=1e-11)
        assert torch.allclose(dk, k.grad, atol=1e-11)
        assert torch.allclose(dv, v.grad, atol=1e-11)


def test_row_blocking_and_sampled_rows_are_the_same_definition():
    q, k, v, do = (rnd((1, 2, 50, 8), s) for s in (140, 141, 142, 143))
    for causal in (False, True):
        o, lse = A.forward(q, k, v, causal, 0.3)
        o2, l2 = A.forward(q, k, v, causal, 0.3, row_block=7)
        assert torch.allclose(o, o2, atol=1e-14) and torch.allclose(lse, l2, atol=1e-14)
        g = A.backward(q, k, v, do, causal, 0.3)
        g2 = A.backward(q, k, v, do, causal, 0.3, row_block=9)
        for a, b in zip(g, g2):
            assert torch.allclose(a, b, atol=1e-12)
        rows = [0, 3, 17, 49]
        o3, l3 = A.forward_rows(q, k, v, causal, 0.3, rows)
        assert torch.allclose(o3, o[:, :, rows], atol=1e-14)
        assert torch.allclose(l3, lse[:, :, rows], atol=1e-14)


def test_causal_block_count_and_program_count():
    g = golden()
    c = g["causal_block_count"]
    assert OS.causal_blocks_visited(c["seq_len"], c["block_m"], c["block_n"]) == c["blocks_computed"]
    assert (c["seq_len"] // c["block_m"]) * (c["seq_len"] // c["block_n"]) == c["blocks_total"]
    p = g["program_count"]
    assert math.ceil(p["S"] / p["block_m"]) * p["B"] * p["H"] == p["programs"]


def test_fully_masked_row_reading():
    """Reading for an all-masked row (never reached with equal lengths): O = 0, L = -inf."""
    s = torch.tensor([[float("-inf"), float("-inf")], [0.0, 1.0]], dtype=F64)
    p, lse = A.softmax_rows(s)
    assert torch.equal(p[0], torch.zeros(2, dtype=F64)) and lse[0] == float("-inf")
    assert abs(float(p[1].sum()) - 1.0) < 1e-15


# ----------------------------------------------------------------------------------
# Planted mistakes: copies of the oracle with one plausible error each.  Every one
# must fail at least one pin, which shows the pins constrain each term.
# ----------------------------------------------------------------------------------

def _fwd_mut(kind):
    def f(q, k, v, causal, scale):
        q, k, v = A.as_f64(q), A.as_f64(k), A.as_f64(v)
        sc = 1.0 if kind == "drop_scale" else scale
        if kind == "transpose_qk":
            s = sc * torch.matmul(k, q.transpose(-1, -2))
        else:
            s = sc * torch.matmul(q, k.transpose(-1, -2))
        if causal:
            n = s.shape[-1]
            diag = 0 if kind == "mask_diagonal_too" else 1
            if kind == "mask_lower":
                s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).tril(-1), float("-inf"))
            else:
                s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(diag), float("-inf"))
        m = s.amax(-1, keepdim=True)
        e = torch.exp(s - m)
        l = e.sum(-1, keepdim=True)
        p = e if kind == "no_normalise" else e / l
        if kind == "pv_transposed":
            o = torch.matmul(p.transpose(-1, -2), v)
        else:
            o = torch.matmul(p, v)
        if kind == "lse_log2":
            lse = m + torch.log2(l)
        elif kind == "lse_no_max":
            lse = torch.log(l)
        else:
            lse = m + torch.log(l)
        return o, lse.squeeze(-1)
    return f


def _bwd_mut(kind):
    def g(q, k, v, do, causal, scale):
        q, k, v, do = (A.as_f64(x) for x in (q, k, v, do))
        p, _ = A.softmax_rows(A.scores(q, k, scale, causal))
        dv = torch.matmul(p, do) if kind == "dv_not_transposed" else torch.matmul(p.transpose(-1, -2), do)
        dp = torch.matmul(do, v.transpose(-1, -2))
        row = (p * dp).sum(-1, keepdim=True)
        if kind == "drop_row_term":
            ds = p * dp
        elif kind == "row_term_sign":
            ds = p * (dp + row)
        else:
            ds = p * (dp - row)
        dq = torch.matmul(ds, k) if kind == "dq_no_scale" else scale * torch.matmul(ds, k)
        if kind == "dk_transposed":
            dk = scale * torch.matmul(ds, q)
        else:
            dk = scale * torch.matmul(ds.transpose(-1, -2), q)
        return dq, dk, dv
    return g


def _blockwise_mut(kind):
    def h(q, k, v, causal, scale, block_m, block_n, trace=None):
        q, k, v = (A.as_f64(x) for x in (q, k, v))
        n, n_k = q.shape[-2], k.shape[-2]
        o = torch.empty(q.shape, dtype=F64)
        lse = torch.empty(q.shape[:-1], dtype=F64)
        for i0 in range(0, n, block_m):
            i1 = min(n, i0 + block_m)
            rows = i1 - i0
            m = torch.full(q.shape[:-2] + (rows,), float("-inf"), dtype=F64)
            l = torch.zeros(q.shape[:-2] + (rows,), dtype=F64)
            acc = torch.zeros(q.shape[:-2] + (rows, q.shape[-1]), dtype=F64)
            if causal and kind == "causal_hi_block_n":
                hi = min(n_k, (i0 // block_m + 1) * block_n)
            else:
                hi = min(n_k, i1) if causal else n_k
            for j0 in range(0, hi, block_n):
                j1 = min(n_k, j0 + block_n)
                s = scale * torch.matmul(q[..., i0:i1, :], k[..., j0:j1, :].transpose(-1, -2))
                if causal:
                    s = s.masked_fill(torch.arange(j0, j1).view(1, -1) > torch.arange(i0, i1).view(-1, 1),
                                      float("-inf"))
                m_new = torch.maximum(m, s.amax(-1))
                alpha = torch.exp(m - m_new)
                base = m if (kind == "p_uses_m_old" and j0 > 0) else m_new
                p = torch.exp(s - base.unsqueeze(-1))
                l = alpha * l + p.sum(-1)
                if kind == "acc_without_alpha":
                    acc = acc + torch.matmul(p, v[..., j0:j1, :])
                else:
                    acc = alpha.unsqueeze(-1) * acc + torch.matmul(p, v[..., j0:j1, :])
                m = m_new
                if trace is not None:
                    trace.append({"m": m.clone(), "alpha": alpha.clone(), "l": l.clone(), "acc": acc.clone()})
            o[..., i0:i1, :] = acc / l.unsqueeze(-1)
            lse[..., i0:i1] = m + torch.log(l)
        return o, lse
    return h


def _fails(fn):
    """True when a pin rejects the implementation (a wrong value or a shape error)."""
    try:
        fn()
    except (AssertionError, RuntimeError):
        return True
    return False


FWD_MUTANTS = ["transpose_qk", "drop_scale", "mask_diagonal_too", "mask_lower", "no_normalise",
               "pv_transposed", "lse_log2", "lse_no_max"]
BWD_MUTANTS = ["dv_not_transposed", "drop_row_term", "row_term_sign", "dq_no_scale", "dk_transposed"]
BLOCKWISE_MUTANTS = ["acc_without_alpha", "p_uses_m_old", "causal_hi_block_n"]


@pytest.mark.parametrize("kind", FWD_MUTANTS)
def test_planted_forward_mistake_is_caught(kind):
    f = _fwd_mut(kind)
    caught = [p.__name__ for p in FWD_PINS if _fails(lambda p=p: p(f))]
    caught += [p.__name__ for p in BWD_PINS if _fails(lambda p=p: p(f, A.backward))]
    assert caught, f"planted forward mistake {kind!r} passed every pin"


@pytest.mark.parametrize("kind", BWD_MUTANTS)
def test_planted_backward_mistake_is_caught(kind):
    g = _bwd_mut(kind)
    caught = [p.__name__ for p in BWD_PINS if _fails(lambda p=p: p(A.forward, g))]
    caught += [p.__name__ for p in GRAD_PINS if _fails(lambda p=p: p(g))]
    assert caught, f"planted backward mistake {kind!r} passed every pin"


@pytest.mark.parametrize("kind", BLOCKWISE_MUTANTS)
def test_planted_blockwise_mistake_is_caught(kind):
    h = _blockwise_mut(kind)
    caught = _fails(lambda: pin_blockwise_trace(h)) or _fails(lambda: pin_blockwise_matches_definition(h))
    assert caught, f"planted recurrence mistake {kind!r} passed every pin"


def test_unmutated_copies_pass():
    """The mutation harness itself is faithful: the unmutated copies pass every pin."""
    f, g, h = _fwd_mut("none"), _bwd_mut("none"), _blockwise_mut("none")
    for p in FWD_PINS:
        p(f)
    pin_worked_example(f, g)
    for p in GRAD_PINS:
        p(g)
    pin_blockwise_trace(h)
    pin_blockwise_matches_definition(h)
