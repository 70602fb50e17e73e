"""The kernels' bounded pipeline waits, made to run out on purpose.

Every wait on a barrier that another warp of the same CTA completes gives up
after a time limit (2 s by default).  A CTA whose wait gives up drains its own
copies and MMAs, frees its tensor memory and exits; the call then reports
FA_ERR_TIMEOUT through fa_check_device_errors, and the context stays usable.
These tests launch ordinary, correct calls with a limit of a few nanoseconds,
so that waits that are not satisfied at once give up, and check the status
and that the next call with the default limit is correct again.  Nothing here
skips an arrival or touches memory out of bounds: the early exits are the
kernels' own abort path.
"""
import pytest
import torch

import oracle
from seeded_inputs import Workload, make_inputs
from tests.parity import assert_close, assert_lse

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_TIMEOUT = 0, 6


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


@pytest.fixture
def short_limit(fa):
    """Run the test body's launches with a 1 ns wait limit; always restore the default."""
    assert fa.fa_check_device_errors(None) == FA_OK
    prev = fa.fa_set_wait_limit_ns(1)
    try:
        yield
    finally:
        fa.fa_set_wait_limit_ns(0)
        fa.fa_check_device_errors(None)  # clear whatever the body left
    assert prev == 2_000_000_000


def _recovers(fa, D, dtype):
    """A normal call after the aborted one matches the oracle and reports no error."""
    w = Workload("after", 1, 2, 300, D, dtype, True, backward=True, seed=7)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    assert fa.fa_check_device_errors(None) == FA_OK
    o_ref, l_ref = oracle.forward(inp["q"], inp["k"], inp["v"], True, w.scale)
    g_ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["do"], True, w.scale)
    assert_close("O", o, o_ref)
    assert_lse(lse, l_ref)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), g_ref):
        assert_close(name, got, ref)


@pytest.mark.parametrize("D", [64, 128])
def test_forward_wait_runs_out(fa, short_limit, D):
    w = Workload("abort", 2, 8, 2048, D, "fp16", True, seed=1)
    inp = make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    fa.forward(q, k, v, causal=True, scale=w.scale)
    assert fa.fa_check_device_errors(None) == FA_ERR_TIMEOUT
    assert "timed out" in fa.fa_last_error_detail()


@pytest.mark.parametrize("D", [64, 128])
def test_backward_wait_runs_out(fa, D):
    w = Workload("abort", 2, 8, 2048, D, "bf16", True, backward=True, seed=2)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)  # default limit: a valid O and L
    assert fa.fa_check_device_errors(None) == FA_OK
    prev = fa.fa_set_wait_limit_ns(1)
    try:
        fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
        st = fa.fa_check_device_errors(None)
    finally:
        fa.fa_set_wait_limit_ns(0)
    assert prev == 2_000_000_000
    assert st == FA_ERR_TIMEOUT


@pytest.mark.parametrize("D", [64, 128])
def test_next_call_is_correct(fa, D):
    """After an aborted call on this context, default-limit calls give oracle results."""
    prev = fa.fa_set_wait_limit_ns(1)
    try:
        w = Workload("abort", 1, 4, 1024, D, "fp16", True, seed=3)
        inp = make_inputs(w)
        q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
        fa.forward(q, k, v, causal=True, scale=w.scale)
        fa.fa_check_device_errors(None)
    finally:
        fa.fa_set_wait_limit_ns(prev)
    for dtype in ("fp16", "bf16"):
        _recovers(fa, D, dtype)

