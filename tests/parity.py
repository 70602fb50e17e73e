"""Helpers for the GPU parity tests: run the library through its C ABI on seeded
inputs and compare with the CPU fp64 oracle on the same inputs.

Tolerances (fp16/bf16 inputs against the fp64 oracle): O, dQ, dK, dV max abs
error <= 2e-2 and mean abs error <= 2e-3; L max abs error <= 1e-3.
"""
from __future__ import annotations

import torch

import oracle
from seeded_inputs import Workload, make_inputs

TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE = 1e-3


def errors(got: torch.Tensor, ref: torch.Tensor):
    d = (got.detach().to("cpu", torch.float64) - ref).abs()
    return float(d.max()) if d.numel() else 0.0, float(d.mean()) if d.numel() else 0.0


def assert_close(name, got, ref, tol_max=TOL_MAX, tol_mean=TOL_MEAN):
    mx, mean = errors(got, ref)
    assert mx <= tol_max and mean <= tol_mean, f"{name}: max abs err {mx:.3e}, mean abs err {mean:.3e}"
    return mx, mean


# Unit roundoff of the 16-bit output types.
UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def assert_close_stored(name, got, ref, spread=1.0):
    """The bars above for results beyond the configured workloads, plus the
    rounding of the stored 16-bit result itself: elementwise
    |got - ref| <= spread * 2e-2 + u * |ref| (u = 2^-8 bf16, 2^-11 fp16), and
    mean abs error <= spread * 2e-3.  At bf16 a result of magnitude 4..8 is
    stored with up to 2^-6 of rounding, most of the 2e-2 bar by itself, so
    cases with larger gradients (other seeds, sums over grouped heads) carry
    that term; ``spread`` widens the bars for sums of several per-head terms.
    """
    u = UNIT_ROUNDOFF[got.dtype]
    r = ref.to(torch.float64)
    d = (got.detach().to("cpu", torch.float64) - r).abs()
    if d.numel() == 0:
        return 0.0, 0.0
    allowed = spread * TOL_MAX + u * r.abs()
    over = float((d - allowed).max())
    mean = float(d.mean())
    assert over <= 0 and mean <= spread * TOL_MEAN, \
        f"{name}: max abs err {float(d.max()):.3e} (worst excess over the bar {over:.3e}), mean abs err {mean:.3e}"
    return float(d.max()), mean


def assert_lse(got, ref):
    mx, _ = errors(got, ref)
    assert mx <= TOL_LSE, f"lse: max abs err {mx:.3e}"
    return mx


def run_forward(fa, inp, causal, scale, device="cuda"):
    q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    return q, k, v, o, lse


def run_backward(fa, q, k, v, o, lse, do_cpu, causal, scale, device="cuda"):
    do = do_cpu.to(device)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    return dq, dk, dv


def check_forward_heads(inp, o, lse, causal, scale, heads, row_block=None):
    """Compare every row of the listed (b, h) heads with the oracle."""
    for b, h in heads:
        o_ref, l_ref = oracle.forward(inp["q"][b, h], inp["k"][b, h], inp["v"][b, h], causal, scale,
                                      row_block=row_block)
        assert_close(f"O[{b},{h}]", o[b, h], o_ref)
        assert_lse(lse[b, h], l_ref)


def check_backward_heads(inp, grads, causal, scale, heads, row_block=None):
    dq, dk, dv = grads
    for b, h in heads:
        r = oracle.backward(inp["q"][b, h], inp["k"][b, h], inp["v"][b, h], inp["do"][b, h], causal, scale,
                            row_block=row_block)
        assert_close(f"dQ[{b},{h}]", dq[b, h], r[0])
        assert_close(f"dK[{b},{h}]", dk[b, h], r[1])
        assert_close(f"dV[{b},{h}]", dv[b, h], r[2])


def workload_inputs(w: Workload, with_dout=None):
    return make_inputs(w, with_dout=with_dout)
