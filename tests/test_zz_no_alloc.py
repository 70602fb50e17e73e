"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code inside a custom allocator, a fully carved-up memory pool, a
framework that forbids cudaMalloc on its hot path) cannot provide fa_bwd's
workspace, so this entry point keeps its scratch in a fixed array inside the
library.  These tests call it through the C ABI, compare it bit for bit with
fa_bwd (the same kernels, so the same bits) and with the fp64 oracle, on
calls in a row: the larger call first, so that when the second, shorter one
runs, rows past its end in the shared array still hold the first call's
values.  The file is named to be collected last.
"""
import pytest
import torch

import exact_attention_18_gb300 as fa
import oracle
from seeded_inputs import Workload, make_inputs
from tests.parity import assert_close

MAX_ROWS = 1 << 21  # the fixed array's capacity in B*H*S rows


def _ptrs(*ts):
    return [t.data_ptr() for t in ts]


def _noalloc(w, q, k, v, o, do, lse):
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    stream = torch.cuda.current_stream().cuda_stream
    dt = fa.FA_FP16 if w.dtype == "fp16" else fa.FA_BF16
    st = fa.fa_bwd_noalloc(*_ptrs(q, k, v, o, do, lse, dq, dk, dv), w.B, w.H, w.S, w.D, w.causal, w.scale,
                           dt, stream)
    assert st == 0, fa.fa_last_error_detail()
    assert fa.fa_check_device_errors(stream) == 0
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_backward_matches_fa_bwd_and_oracle_on_calls_in_a_row():
    fa.load_library()
    cases = [Workload("noalloc_a", 1, 4, 1024, 128, "bf16", False, backward=True, seed=42),
             Workload("noalloc_b", 2, 3, 300, 64, "fp16", True, backward=True, seed=41)]
    for w in cases:
        inp = make_inputs(w)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
        ref = fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
        got = _noalloc(w, q, k, v, o, do, lse)
        exact = oracle.backward(inp["q"], inp["k"], inp["v"], inp["do"], w.causal, w.scale)
        for name, g, r, e in zip(("dQ", "dK", "dV"), got, ref, exact):
            assert torch.equal(g, r), f"{w.name} {name}: differs from fa_bwd"
            assert_close(f"{w.name} {name}", g, e)


@pytest.mark.gpu
def test_noalloc_at_exactly_its_capacity():
    """B*H*S = 2^21 rows fill the whole array; first, middle and last heads match fa_bwd
    bit for bit, and the last head matches the oracle."""
    fa.load_library()
    w = Workload("noalloc_full", 1, 512, 4096, 16, "fp16", True, backward=True, seed=43)
    assert w.B * w.H * w.S == MAX_ROWS
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    ref = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    got = _noalloc(w, q, k, v, o, do, lse)
    for h in (0, 255, 511):
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(g[0, h], r[0, h]), f"head {h} {name}: differs from fa_bwd"
    exact = oracle.backward(inp["q"][0, 511], inp["k"][0, 511], inp["v"][0, 511], inp["do"][0, 511], True,
                            w.scale, row_block=1024)
    for name, g, e in zip(("dQ", "dK", "dV"), got, exact):
        assert_close(f"head 511 {name}", g[0, 511], e)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """2^21 rows fit; one head more does not.  Rejected before any CUDA call."""
    fa.load_library()
    p = 0x10000
    st = fa.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 513, 4096, 64, 1, 0.125, fa.FA_FP16, None)
    assert st == 2  # FA_ERR_UNSUPPORTED
    assert "scratch" in fa.fa_last_error_detail()
