"""Repeated calls give the same bits.

Every kernel of the library sums in a fixed order (no atomics, no split
reductions whose order depends on timing), so calling the forward and the
backward again on the same inputs must reproduce their outputs bit for bit.
A race between the warps of a CTA (a barrier phase completing before all the
data it guards is written, say) shows up here as a call whose results differ
from the first call's, or as a device error; timing varies from call to call,
so each case runs many times.  The first call is also checked against the
fp64 oracle on sampled heads, so the repeated result is the right one.
"""
import pytest
import torch

import oracle
from seeded_inputs import PACKED_CONFIGS, Workload, make_inputs, make_packed_inputs
from tests.parity import assert_close, assert_lse

pytestmark = pytest.mark.gpu

REPEATS = 30


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


def _call(fa, w, q, k, v, do):
    o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
    st = fa.fa_check_device_errors(None)
    assert st == 0, fa.fa_last_error_detail()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("D,dtype,causal", [(64, "fp16", True), (64, "bf16", False), (32, "fp16", True),
                                            (128, "bf16", True)])
def test_repeated_calls_are_bitwise_equal(fa, D, dtype, causal):
    w = Workload("repeat", 4, 16, 2048, D, dtype, causal, backward=True, seed=77)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    first = _call(fa, w, q, k, v, do)
    names = ("O", "L", "dQ", "dK", "dV")
    for rep in range(REPEATS):
        again = _call(fa, w, q, k, v, do)
        for name, a, b in zip(names, first, again):
            assert torch.equal(a, b), f"call {rep + 1}: {name} differs from the first call"
    o, lse, dq, dk, dv = first
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        args = [inp[n][b, h] for n in ("q", "k", "v", "do")]
        o_ref, l_ref = oracle.forward(*args[:3], causal, w.scale)
        assert_close(f"O[{b},{h}]", o[b, h], o_ref)
        assert_lse(lse[b, h], l_ref)
        g_ref = oracle.backward(*args, causal, w.scale)
        for name, got, ref in zip(("dQ", "dK", "dV"), (dq[b, h], dk[b, h], dv[b, h]), g_ref):
            assert_close(f"{name}[{b},{h}]", got, ref)


def _same(first, again, names, rep):
    for name, a, b in zip(names, first, again):
        assert torch.equal(a, b), f"call {rep + 1}: {name} differs from the first call"


@pytest.mark.parametrize("path", ["gqa", "window", "varlen"])
def test_repeated_calls_of_the_other_paths(fa, path):
    """The grouped-query, window and packed-batch entry points (their own tests cover parity)."""
    names = ("O", "L", "dQ", "dK", "dV")
    if path == "varlen":
        w = PACKED_CONFIGS["varlen"]
        inp = make_packed_inputs(w)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
        cu = inp["cu_seqlens"].cuda()

        def call():
            o, lse = fa.forward_varlen(q, k, v, cu, w.max_seqlen, causal=w.causal, scale=w.scale)
            g = fa.backward_varlen(q, k, v, o, do, lse, cu, w.max_seqlen, causal=w.causal, scale=w.scale)
            st = fa.fa_check_device_errors(None)
            assert st == 0, fa.fa_last_error_detail()
            return (o, lse, *g)
    else:
        if path == "gqa":
            w = Workload("repeat_gqa", 2, 16, 2048, 64, "bf16", True, backward=True, seed=78, H_kv=4)
            window = None
        else:
            w = Workload("repeat_window", 2, 8, 2048, 64, "fp16", True, backward=True, seed=79, window=(512, 0))
            window = w.window
        inp = make_inputs(w)
        q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))

        def call():
            o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale, window=window)
            g = fa.backward(q, k, v, o, do, lse, causal=w.causal, scale=w.scale, window=window)
            st = fa.fa_check_device_errors(None)
            assert st == 0, fa.fa_last_error_detail()
            return (o, lse, *g)
    first = call()
    for rep in range(REPEATS):
        _same(first, call(), names, rep)


@pytest.mark.parametrize("D,dtype,path", [(64, "fp16", "fixed"), (32, "bf16", "gqa"), (128, "bf16", "fixed"),
                                          (64, "fp16", "window")])
def test_stale_workspace_never_reaches_the_gradients(fa, D, dtype, path):
    """The backward's kernels overlap: each starts its CTAs while the one before it finishes,
    and waits for it only before reading Delta, which the Delta kernel (or, at D <= 64 with
    fixed lengths, the dQ pass) writes into the workspace during the same call.  With the
    workspace filled with NaN before every call, a read of Delta before it is written would
    show up as NaN in dQ, dK or dV; every call must also reproduce the first one's bits."""
    H_kv = 4 if path == "gqa" else None
    window = (512, 0) if path == "window" else None
    w = Workload("stale_ws", 2, 16, 2048, D, dtype, True, backward=True, seed=93, H_kv=H_kv, window=window)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale, window=window)
    ws_bytes = fa.fa_bwd_gqa_workspace_size(w.B, w.H, k.shape[1], w.S, D)
    ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
    first = None
    for rep in range(REPEATS):
        ws.fill_(float("nan"))
        g = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale, window=window, workspace=ws)
        assert fa.fa_check_device_errors(None) == 0, fa.fa_last_error_detail()
        for name, t in zip(("dQ", "dK", "dV"), g):
            assert bool(torch.isfinite(t).all()), f"call {rep + 1}: {name} has non-finite values"
        if first is None:
            first = g
        else:
            _same(first, g, ("dQ", "dK", "dV"), rep)


@pytest.mark.parametrize("D,dtype", [(64, "fp16"), (128, "bf16")])
def test_marked_backward_gives_the_same_bits(fa, D, dtype):
    """fa_bwd_marked runs the same kernels as fa_bwd, with events recorded between them (at
    D = 64 the dQ pass, which computes Delta, first; at D = 128 the Delta kernel first): the
    results are bit-identical, the four events complete in order, and at D = 64 no kernel runs
    between the last two."""
    w = Workload("marked", 2, 8, 1024, D, dtype, True, backward=True, seed=95)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True, scale=w.scale)
    ref = fa.backward(q, k, v, o, do, lse, causal=True, scale=w.scale)
    ws_bytes = fa.fa_bwd_workspace_size(w.B, w.H, w.S, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:  # create the events before the library records them
        e.record(stream)
    dt = fa.FA_FP16 if dtype == "fp16" else fa.FA_BF16
    st = fa.fa_bwd_marked(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                          got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(), w.B, w.H, w.S, D, True, w.scale,
                          dt, ws.data_ptr(), ws_bytes, stream.cuda_stream, [e.cuda_event for e in ev])
    assert st == 0, fa.fa_last_error_detail()
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0, fa.fa_last_error_detail()
    _same(ref, got, ("dQ", "dK", "dV"), 0)
    gaps = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(g >= 0 for g in gaps), gaps
    assert gaps[0] > 0 and gaps[1] > 0, gaps
    if D == 64:
        assert gaps[2] < 0.5 * min(gaps[0], gaps[1]), gaps
