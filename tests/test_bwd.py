"""Backward parity: the CUDA recompute backward (through the C ABI) against the
fp64 oracle's closed-form gradients, on the library's own forward outputs."""
import math

import pytest
import torch

import oracle
from seeded_inputs import C3_D, C3_S, CONFIGS, Workload, make_inputs
from tests.parity import (assert_close, assert_lse, check_backward_heads, check_forward_heads, run_backward,
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
    heads = [(0, 0), (1, 31)]
    check_forward_heads(inp, o, lse, False, w.scale, heads, row_block=2048)
    check_backward_heads(inp, grads, False, w.scale, heads, row_block=2048)


def test_std2_variant(fa):
    """The other reading of "N(0, 2)": standard deviation 2, an extra stress case.

    The configured workload reads N(0, 2) as variance 2 and meets the absolute
    bars.  With standard deviation 2 the forward still does (checked here), but
    the backward's max-abs error is set by bf16 itself: the gradients reach
    |6.6|, where one bf16 rounding alone costs up to 0.015, and an emulation of
    the 16-bit pipeline on exact inputs (P and dS rounded to bf16 as MMA
    operands, Delta taken from the bf16 output O) reaches 0.040 in dQ.  So the
    backward is held to the stated mean-abs bar (2e-3) and to a norm-wise
    relative error ||got - ref|| / ||ref|| <= 1e-2 (about 2.5 bf16 unit
    roundoffs; the emulation gives 0.0037), both against the fp64 oracle.
    """
    w = Workload("c4_std2", 1, 2, 2048, 128, "bf16", False, qk_std=2.0, backward=True, seed=0)
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = fwd_bwd(fa, w, inp)
    check_forward_heads(inp, o, lse, False, w.scale, [(0, 0), (0, 1)])
    for h in (0, 1):
        ref = oracle.backward(inp["q"][0, h], inp["k"][0, h], inp["v"][0, h], inp["do"][0, h], False, w.scale)
        for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            d = got[0, h].double().cpu() - r
            rel = float(d.norm() / r.norm())
            mean = float(d.abs().mean())
            assert rel <= 1e-2 and mean <= 2e-3, \
                f"{name}[0,{h}]: relative error {rel:.2e}, mean abs {mean:.2e}, max abs {float(d.abs().max()):.2e}"


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
