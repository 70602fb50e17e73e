"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code inside a custom allocator, a fully carved-up memory pool, a
framework that forbids cudaMalloc on its hot path) cannot provide fa_bwd's
workspace, so this entry point keeps its scratch in a fixed array inside the
library.  These tests call it through the C ABI and compare it with fa_bwd on
two calls in a row, which also shows that the shared array's leftover contents
from one call do not leak into the next.  The file is named to be collected
last.
"""
import pytest
import torch

import exact_attention_18_gb300 as fa
from seeded_inputs import Workload, make_inputs
from tests.parity import assert_close


def _ptrs(*ts):
    return [t.data_ptr() for t in ts]


@pytest.mark.gpu
def test_noalloc_backward_matches_fa_bwd_on_two_calls_in_a_row():
    fa.load_library()
    cases = [Workload("noalloc_a", 2, 3, 300, 64, "fp16", True, backward=True, seed=41),
             Workload("noalloc_b", 1, 4, 1024, 128, "bf16", False, backward=True, seed=42)]
    for w in cases:
        inp = make_inputs(w)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
        ref = fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        stream = torch.cuda.current_stream().cuda_stream
        dt = fa.FA_FP16 if w.dtype == "fp16" else fa.FA_BF16
        st = fa.fa_bwd_noalloc(*_ptrs(q, k, v, o, do, lse, dq, dk, dv), w.B, w.H, w.S, w.D, w.causal, w.scale,
                               dt, stream)
        assert st == 0, fa.fa_last_error_detail()
        assert fa.fa_check_device_errors(stream) == 0
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            assert_close(f"{w.name} {name}", got, want.double().cpu())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """2^21 rows fit; one head more does not.  Rejected before any CUDA call."""
    fa.load_library()
    p = 0x10000
    st = fa.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 513, 4096, 64, 1, 0.125, fa.FA_FP16, None)
    assert st == 2  # FA_ERR_UNSUPPORTED
    assert "scratch" in fa.fa_last_error_detail()
