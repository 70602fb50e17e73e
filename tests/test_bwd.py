"""Backward parity: the CUDA recompute backward (through the C ABI) against the
fp64 oracle's closed-form gradients, on the library's own forward outputs."""
import dataclasses
import math

import pytest
import torch

import oracle
from seeded_inputs import C3_D, C3_S, CONFIGS, Workload, make_inputs
from tests.parity import (assert_close, assert_close_stored, assert_lse, assert_within_bound,
                          backward_rounding_bounds, check_backward_heads, check_forward_heads, run_backward,
                          run_forward)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


def fwd_bwd(fa, w, inp):
    q, k, v, o, lse = run_forward(fa, inp, w.causal, w.scale)
    grads = run_backward(fa, q, k, v, o, lse, inp["do"], w.causal, w.scale)
    return o, lse, grads


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 17, 130, 257, 512])
def test_small_shapes(fa, D, dtype, causal, S):
    w = Workload("small", 2, 2, S, D, dtype, causal, backward=True, seed=100 + S + D)
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = fwd_bwd(fa, w, inp)
    r = oracle.backward(inp["q"], inp["k"], inp["v"], inp["do"], causal, w.scale)
    assert_close("dQ", dq, r[0])
    assert_close("dK", dk, r[1])
    assert_close("dV", dv, r[2])


@pytest.mark.parametrize("D", C3_D)
@pytest.mark.parametrize("S", C3_S)
def test_config_c3(fa, D, S):
    """Causal fwd+bwd, batch 8 without a head axis, bf16: every (D, S) point."""
    w = CONFIGS[f"c3_d{D}_s{S}"]
    inp = make_inputs(w)
    o, lse, grads = fwd_bwd(fa, w, inp)
    heads = [(b, 0) for b in range(8)] if S <= 1024 else ([(0, 0), (7, 0)] if S <= 4096 else [(7, 0)])
    rb = None if S <= 4096 else 2048
    check_forward_heads(inp, o, lse, True, w.scale, heads, row_block=rb)
    check_backward_heads(inp, grads, True, w.scale, heads, row_block=rb)


def test_config_c4_sampled_heads(fa):
    """Non-causal B2 H32 S8192 D128 bf16 with Q, K ~ N(0, 2)."""
    w = CONFIGS["c4"]
    inp = make_inputs(w)
    o, lse, grads = fwd_bwd(fa, w, inp)
    heads = [(0, 0), (0, 17), (1, 5), (1, 31)]
    check_forward_heads(inp, o, lse, False, w.scale, heads, row_block=2048)
    check_backward_heads(inp, grads, False, w.scale, heads, row_block=2048)


def test_std2_variant(fa):
    """The other reading of "N(0, 2)": standard deviation 2, an extra stress case.

    The configured workload reads N(0, 2) as variance 2 and meets the absolute
    bars.  With standard deviation 2 the forward still does (checked here),
    but the exact gradients reach |6.6|, where one bf16 rounding of the
    stored result alone costs up to 0.015: no backward that rounds P, dS and
    its outputs to bf16 can meet 2e-2 max-abs there.  The backward is held,
    element by element, to the first-order bound of its bf16 roundings
    (tests.parity.backward_rounding_bounds, u = 2^-8), computed from the fp64
    oracle's own P, dS and gradients, and to the stated 2e-3 mean bar.
    """
    w = Workload("c4_std2", 1, 2, 2048, 128, "bf16", False, qk_std=2.0, backward=True, seed=0)
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = fwd_bwd(fa, w, inp)
    check_forward_heads(inp, o, lse, False, w.scale, [(0, 0), (0, 1)])
    for h in (0, 1):
        args = [inp[n][0, h] for n in ("q", "k", "v", "do")]
        ref = oracle.backward(*args, False, w.scale)
        bounds = backward_rounding_bounds(*args, False, w.scale, u=2.0 ** -8)
        for name, got, r, bnd in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref, bounds):
            assert_within_bound(f"{name}[0,{h}]", got[0, h], r, bnd)


def test_config_c2_backward_sampled_heads(fa):
    """The benchmark's own backward: causal B4 H16 S4096 D64 fp16, first, middle and last heads,
    every row, at the stated bars."""
    w = dataclasses.replace(CONFIGS["c2"], backward=True)
    inp = make_inputs(w)
    o, lse, grads = fwd_bwd(fa, w, inp)
    heads = [(0, 0), (1, 7), (2, 12), (3, 15)]
    check_forward_heads(inp, o, lse, True, w.scale, heads, row_block=1024)
    check_backward_heads(inp, grads, True, w.scale, heads, row_block=1024)


@pytest.mark.parametrize("S,causal", [(4160, True), (4224, True), (2048, False), (2112, False)])
def test_both_dkdv_kernels_at_their_switch(fa, S, causal):
    """At D <= 64 the dK/dV pass runs its persistent kernel while a work item averages at most 32
    partner blocks (64-row query blocks, halved under the causal mask) and the per-tile kernel
    beyond: both sides of that switch, every row of two heads (the last tile ragged)."""
    w = Workload("dkdv_switch", 1, 2, S, 64, "fp16", causal, backward=True, seed=S + causal)
    inp = make_inputs(w)
    o, lse, grads = fwd_bwd(fa, w, inp)
    check_backward_heads(inp, grads, causal, w.scale, [(0, 0), (0, 1)], row_block=2048)


def test_grouped_heads_in_persistent_dkdv_items(fa):
    """Grouped K/V heads with short rows keep the persistent dK/dV pass (two query heads per
    work item, and CTAs splitting a group when there are few K/V heads): every row of every K/V
    head against the grouped oracle."""
    for B, H, Hkv, S in ((2, 8, 4, 1024), (1, 8, 1, 512)):
        w = Workload("gqa_persistent", B, H, S, 64, "bf16", True, backward=True, seed=S + Hkv, H_kv=Hkv)
        inp = make_inputs(w)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
        dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
        torch.cuda.synchronize()
        assert fa.fa_check_device_errors(None) == 0
        r = oracle.backward_gqa(inp["q"], inp["k"], inp["v"], inp["do"], True, w.scale)
        g = H // Hkv
        assert_close_stored("dQ", dq, r[0])
        assert_close_stored("dK", dk, r[1], spread=math.sqrt(g))
        assert_close_stored("dV", dv, r[2], spread=math.sqrt(g))


def test_leaderboard_workload_sampled_heads(fa):
    """Causal B1 H16 S16384 D64 bf16 ("CS336 Assignment 2" §6 leaderboard shape): first,
    a middle and the last head, every row, forward and backward, at the stated bars."""
    w = CONFIGS["leaderboard"]
    inp = make_inputs(w)
    o, lse, grads = fwd_bwd(fa, w, inp)
    heads = [(0, 0), (0, 9), (0, 15)]
    check_forward_heads(inp, o, lse, True, w.scale, heads, row_block=2048)
    check_backward_heads(inp, grads, True, w.scale, heads, row_block=2048)


def test_zero_dout_rows_give_exact_zero_dk_dv(fa):
    """Causal: if dO rows >= t are zero, dK and dV rows >= t are exactly zero."""
    w = Workload("tailzero", 1, 2, 400, 64, "fp16", True, backward=True, seed=8)
    inp = make_inputs(w)
    t = 250
    inp["do"][:, :, t:] = 0
    o, lse, (dq, dk, dv) = fwd_bwd(fa, w, inp)
    assert torch.count_nonzero(dk[:, :, t:]) == 0
    assert torch.count_nonzero(dv[:, :, t:]) == 0
    assert torch.count_nonzero(dv[:, :, :t]) > 0


def test_gradient_sum_identities(fa):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, up to rounding of the outputs."""
    w = Workload("sums", 1, 2, 640, 64, "fp16", False, backward=True, seed=9)
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = fwd_bwd(fa, w, inp)
    assert float(dk.double().sum(2).abs().max()) < 0.05
    assert float((dv.double().sum(2).cpu() - inp["do"].double().sum(2)).abs().max()) < 0.05


def test_bwd_workspace_checks(fa):
    w = Workload("ws", 1, 1, 64, 64, "fp16", False, backward=True)
    inp = make_inputs(w)
    q, k, v, o, lse = run_forward(fa, inp, False, w.scale)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError, match="FA_ERR_WORKSPACE"):
        fa.backward(q, k, v, o, inp["do"].cuda(), lse, workspace=small)


@pytest.mark.parametrize("D,dtype,causal,S,gqa", [(64, "fp16", True, 1000, False), (32, "bf16", False, 300, False),
                                                  (16, "fp16", True, 129, False), (64, "bf16", True, 777, True),
                                                  (128, "fp16", True, 300, False)])
def test_delta_left_in_the_workspace(fa, D, dtype, causal, S, gqa):
    """The backward leaves D_i = rowsum(dO o O) of every query row at the start of its
    workspace: computed by the dQ pass (D <= 64, which then runs before the dK/dV pass) or
    by the Delta kernel (D = 128).  O and L are the oracle's forward, rounded to the
    input dtype; a ragged last tile leaves rows past S in the last work item."""
    H_kv = 2 if gqa else None
    w = Workload("delta_ws", 2, 4, S, D, dtype, causal, backward=True, seed=91, H_kv=H_kv)
    inp = make_inputs(w)
    kx = oracle.expand_kv(inp["k"], w.H) if gqa else inp["k"]
    vx = oracle.expand_kv(inp["v"], w.H) if gqa else inp["v"]
    o_ref, l_ref = oracle.forward(inp["q"], kx, vx, causal, w.scale)
    o_in = o_ref.to(inp["q"].dtype)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = o_in.cuda(), l_ref.float().cuda()
    ws_bytes = fa.fa_bwd_gqa_workspace_size(w.B, w.H, k.shape[1], S, D)
    ws = torch.full((ws_bytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    fa.backward(q, k, v, o, do, lse, causal=causal, scale=w.scale, workspace=ws)
    assert fa.fa_check_device_errors(None) == 0, fa.fa_last_error_detail()
    got = ws[: w.B * w.H * S].view(w.B, w.H, S).cpu().double()
    ref = oracle.delta(o_in, inp["do"])
    # Products of two 16-bit values are exact in fp32; D fp32 additions in any order stay
    # within D * 2^-24 * sum |terms| of the exact sum.
    bound = D * 2.0 ** -24 * (o_in.double() * inp["do"].double()).abs().sum(-1) * 1.01 + 1e-30
    err = (got - ref).abs()
    assert bool((err <= bound).all()), f"max |Delta - oracle| {float(err.max()):.3e}"
