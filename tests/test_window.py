"""Sliding-window attention on the GPU (through the C ABI) against the fp64
oracle with the same band, on the library's own forward outputs.

Bars as for the grouped-head tests (cases beyond the configured workloads):
``assert_close_stored``, with sqrt(G) for dK and dV of grouped heads.
"""
import math

import pytest
import torch

import oracle
from seeded_inputs import CONFIGS, Workload, make_inputs
from tests.parity import assert_close_stored, assert_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


def run(fa, w, inp, window):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale, window=window)
    grads = fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, window=window)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    return o, lse, grads


def check(inp, w, o, lse, grads, window, heads=None, row_block=None):
    grp = w.H // w.kv_heads
    groups = [(b, g) for b in range(w.B) for g in range(w.kv_heads)] if heads is None else heads
    for b, g in groups:
        hs = slice(g * grp, (g + 1) * grp)
        q, k, v, do = inp["q"][b, hs], inp["k"][b, g:g + 1], inp["v"][b, g:g + 1], inp["do"][b, hs]
        o_ref, l_ref = oracle.forward_gqa(q, k, v, w.causal, w.scale, row_block=row_block, window=window)
        assert_close_stored(f"O[{b},{hs}]", o[b, hs], o_ref)
        assert_lse(lse[b, hs], l_ref)
        r = oracle.backward_gqa(q, k, v, do, w.causal, w.scale, row_block=row_block, window=window)
        assert_close_stored(f"dQ[{b},{hs}]", grads[0][b, hs], r[0])
        assert_close_stored(f"dK[{b},{g}]", grads[1][b, g:g + 1], r[1], spread=math.sqrt(grp))
        assert_close_stored(f"dV[{b},{g}]", grads[2][b, g:g + 1], r[2], spread=math.sqrt(grp))


BANDS = [(0, 0), (1, 0), (37, 5), (100, -1), (-1, 130), (200, 64)]


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("band", BANDS, ids=lambda b: f"{b[0]}_{b[1]}")
def test_bands(fa, D, dtype, causal, band):
    """Whole tensors, S = 700 (several tiles and a ragged tail), two query heads per K/V head."""
    w = Workload("win", 1, 4, 700, D, dtype, causal, backward=True, seed=400 + D + band[0], H_kv=2)
    inp = make_inputs(w)
    o, lse, grads = run(fa, w, inp, band)
    check(inp, w, o, lse, grads, band)


@pytest.mark.parametrize("S", [1, 17, 130])
def test_short_sequences(fa, S):
    w = Workload("win_short", 2, 2, S, 64, "bf16", True, backward=True, seed=500 + S)
    inp = make_inputs(w)
    o, lse, grads = run(fa, w, inp, (5, 0))
    check(inp, w, o, lse, grads, (5, 0))


@pytest.mark.parametrize("causal", [False, True])
def test_window_covering_the_sequence_is_the_plain_call(fa, causal):
    """A band wider than the sequence runs the ordinary kernels: results bit for bit the same."""
    w = Workload("wide", 2, 4, 600, 64, "fp16", causal, backward=True, seed=14)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o1, l1 = fa.forward(q, k, v, causal=causal)
    o2, l2 = fa.forward(q, k, v, causal=causal, window=(600, 600))
    g1 = fa.backward(q, k, v, o1, do, l1, causal=causal)
    g2 = fa.backward(q, k, v, o2, do, l2, causal=causal, window=(-1, -1))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_band_locality(fa):
    """Rows whose band misses a changed key block stay bitwise unchanged."""
    w = Workload("loc", 1, 2, 1024, 64, "fp16", True, backward=False, seed=15)
    inp = make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True, window=(100, 0))
    k2 = k.clone()
    k2[:, :, 300:320] = -k2[:, :, 300:320]
    o2, l2 = fa.forward(q, k2, v, causal=True, window=(100, 0))
    torch.cuda.synchronize()
    assert torch.equal(o1[:, :, :300], o2[:, :, :300]) and torch.equal(o1[:, :, 420:], o2[:, :, 420:])
    assert not torch.equal(o1[:, :, 300:420], o2[:, :, 300:420])


def test_full_size_window_workload(fa):
    """B4 H16 S4096 D64 causal fp16 with a 1024-key window: two heads, every row."""
    w = CONFIGS["window"]
    inp = make_inputs(w)
    o, lse, grads = run(fa, w, inp, w.window)
    check(inp, w, o, lse, grads, w.window, heads=[(0, 0), (3, 15)], row_block=1024)
