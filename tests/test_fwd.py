"""Forward parity: the CUDA forward (through the C ABI) against the fp64 oracle."""
import math

import pytest
import torch

import oracle
from seeded_inputs import CONFIGS, Workload, make_inputs, randn
from tests.parity import (TOL_LSE, assert_close, assert_lse, check_forward_heads, errors, run_forward)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 17, 128, 130, 257, 512])
def test_small_shapes(fa, D, dtype, causal, S):
    w = Workload("small", 2, 3, S, D, dtype, causal, seed=S + D)
    inp = make_inputs(w)
    q, k, v, o, lse = run_forward(fa, inp, causal, w.scale)
    o_ref, l_ref = oracle.forward(inp["q"], inp["k"], inp["v"], causal, w.scale)
    assert_close("O", o, o_ref)
    assert_lse(lse, l_ref)


@pytest.mark.parametrize("D", [32, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [6144, 6208])
def test_both_d64_forward_kernels_at_their_switch(fa, D, causal, S):
    """At D <= 64 fixed-length calls of up to 6144 rows run the persistent two-pipeline kernel,
    longer ones the four-tile kernel: both sides of the switch, every row of two heads (one with
    a ragged last item or tile)."""
    w = Workload("switch", 1, 2, S, D, "bf16", causal, seed=S + D + causal)
    inp = make_inputs(w)
    q, k, v, o, lse = run_forward(fa, inp, causal, w.scale)
    check_forward_heads(inp, o, lse, causal, w.scale, [(0, 0), (0, 1)], row_block=2048)


def test_many_items_per_pipeline(fa):
    """More 256-row items than pipelines several times over (B16 H16 S1024: 1024 items), so every
    pipeline runs several items and carries its barrier phases across them."""
    w = Workload("items", 16, 16, 1024, 64, "fp16", True, seed=5)
    inp = make_inputs(w)
    q, k, v, o, lse = run_forward(fa, inp, True, w.scale)
    check_forward_heads(inp, o, lse, True, w.scale, [(0, 0), (7, 3), (15, 15)])


def test_config_c1_full(fa):
    w = CONFIGS["c1"]
    inp = make_inputs(w)
    q, k, v, o, lse = run_forward(fa, inp, w.causal, w.scale)
    assert o.shape == (1, 1, 256, 64) and lse.shape == (1, 1, 256) and lse.dtype == torch.float32
    o_ref, l_ref = oracle.forward(inp["q"], inp["k"], inp["v"], w.causal, w.scale)
    assert_close("O", o, o_ref)
    assert_lse(lse, l_ref)


def test_config_c2_sampled_heads(fa):
    w = CONFIGS["c2"]
    inp = make_inputs(w)
    q, k, v, o, lse = run_forward(fa, inp, w.causal, w.scale)
    check_forward_heads(inp, o, lse, w.causal, w.scale, [(0, 0), (2, 9), (3, 15)])


def test_config_c5_sampled_rows_and_no_score_matrix(fa):
    """S = 32768: sampled rows of two heads; the [S, S] matrix (2 GiB per head) is never allocated."""
    w = CONFIGS["c5"]
    inp = make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)  # first call: module load
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    fa.forward(q, k, v, causal=True, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_before - free_after < 64 << 20, "the forward allocated device memory"
    assert fa.fa_check_device_errors(None) == 0
    g = torch.Generator().manual_seed(7)
    rows = sorted(set([0, 1, 2, 127, 128, 129, 4095, 4096, 16383, 16384, 32766, 32767] +
                      torch.randint(0, w.S, (20,), generator=g).tolist()))
    for h in (0, 7):
        o_ref, l_ref = oracle.forward_rows(inp["q"][0, h], inp["k"][0, h], inp["v"][0, h], True, w.scale, rows)
        assert_close(f"O[0,{h}] rows", o[0, h, rows], o_ref)
        assert_lse(lse[0, h, rows], l_ref)


def test_causal_mask_is_exact(fa):
    """Changing K and V rows after t leaves O and L of rows <= t bitwise unchanged."""
    w = Workload("mask", 1, 2, 300, 64, "fp16", True, seed=3)
    inp = make_inputs(w)
    _, _, _, o1, l1 = run_forward(fa, inp, True, w.scale)
    t = 150
    inp2 = dict(inp)
    inp2["k"] = inp["k"].clone()
    inp2["v"] = inp["v"].clone()
    inp2["k"][:, :, t + 1:] = randn(inp["k"][:, :, t + 1:].shape, 99, torch.float16, 3.0)
    inp2["v"][:, :, t + 1:] = randn(inp["v"][:, :, t + 1:].shape, 98, torch.float16)
    _, _, _, o2, l2 = run_forward(fa, inp2, True, w.scale)
    assert torch.equal(o1[:, :, : t + 1], o2[:, :, : t + 1])
    assert torch.equal(l1[:, :, : t + 1], l2[:, :, : t + 1])
    assert not torch.equal(o1[:, :, t + 1:], o2[:, :, t + 1:])


def test_causal_first_row_is_v0(fa):
    for dtype in ("fp16", "bf16"):
        w = Workload("row0", 2, 2, 200, 128, dtype, True, seed=5)
        inp = make_inputs(w)
        q, k, v, o, lse = run_forward(fa, inp, True, w.scale)
        assert torch.equal(o[:, :, 0].cpu(), inp["v"][:, :, 0])
        s00 = w.scale * (inp["q"][:, :, 0].double() * inp["k"][:, :, 0].double()).sum(-1)
        assert float((lse[:, :, 0].cpu().double() - s00).abs().max()) <= TOL_LSE


def test_uniform_scores(fa):
    """Q = 0: O is the mean of the visible V rows and L = ln(#visible keys)."""
    S, D = 333, 64
    q = torch.zeros(1, 2, S, D, dtype=torch.float16)
    k = randn((1, 2, S, D), 1, torch.float16)
    v = randn((1, 2, S, D), 2, torch.float16)
    for causal in (False, True):
        _, _, _, o, lse = run_forward(fa, {"q": q, "k": k, "v": v}, causal, 0.125)
        vv = v.double()
        if causal:
            ref = vv.cumsum(2) / torch.arange(1, S + 1, dtype=torch.float64).view(1, 1, S, 1)
            lref = torch.log(torch.arange(1, S + 1, dtype=torch.float64)).expand(1, 2, S)
        else:
            ref = vv.mean(2, keepdim=True).expand_as(vv)
            lref = torch.full((1, 2, S), math.log(S), dtype=torch.float64)
        assert_close("O", o, ref)
        assert_lse(lse, lref)


@pytest.mark.parametrize("scale", [0.0, -0.3, 0.9])
def test_unusual_scales(fa, scale):
    w = Workload("scale", 1, 2, 190, 32, "bf16", True, seed=11)
    inp = make_inputs(w)
    _, _, _, o, lse = run_forward(fa, inp, True, scale)
    o_ref, l_ref = oracle.forward(inp["q"], inp["k"], inp["v"], True, scale)
    assert_close("O", o, o_ref)
    assert_lse(lse, l_ref)


def test_large_scores_stress_rescaling(fa):
    """Q, K ~ N(0, 2) and N(0, 4): large score spread forces many running-max updates."""
    for std in (math.sqrt(2.0), 2.0):
        w = Workload("stress", 1, 4, 1000, 128, "bf16", False, qk_std=std, seed=21)
        inp = make_inputs(w)
        _, _, _, o, lse = run_forward(fa, inp, False, w.scale)
        o_ref, l_ref = oracle.forward(inp["q"], inp["k"], inp["v"], False, w.scale)
        assert_close("O", o, o_ref)
        assert_lse(lse, l_ref)


def test_empty_inputs(fa):
    for shape in ((0, 2, 16, 64), (2, 0, 16, 64), (1, 1, 0, 64)):
        q = torch.empty(shape, dtype=torch.float16, device="cuda")
        o, lse = fa.forward(q, q, q, causal=True)
        assert o.shape == shape and lse.shape == shape[:3]


def test_three_dim_inputs_without_head_axis(fa):
    w = Workload("nohead", 3, 1, 140, 64, "bf16", True, seed=4)
    inp = make_inputs(w)
    q, k, v = (inp[n][:, 0].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=True)
    assert o.shape == (3, 140, 64) and lse.shape == (3, 140)
    o_ref, l_ref = oracle.forward(inp["q"][:, 0], inp["k"][:, 0], inp["v"][:, 0], True, w.scale)
    assert_close("O", o, o_ref)
    assert_lse(lse, l_ref)


def test_bad_head_dim_raises(fa):
    q = torch.zeros(1, 1, 16, 48, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FAError, match="FA_ERR_UNSUPPORTED"):
        fa.forward(q, q, q)
