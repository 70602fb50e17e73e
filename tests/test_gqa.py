"""Grouped-query and multi-query attention on the GPU (through the C ABI) against
the fp64 GQA oracle, on the library's own forward outputs.

Tolerances: O, L and dQ are per-query-head results and keep the multi-head
bars (max abs <= 2e-2, mean abs <= 2e-3, L max abs <= 1e-3), plus the rounding
of the stored 16-bit value (``assert_close_stored``: these are cases beyond
the configured workloads, with other seeds and larger gradients).  dK and dV
of a K/V head are sums of G = H / H_kv per-head gradients, each of which meets
the multi-head bar, and grow with G; with independent per-head errors adding
in quadrature they are held to sqrt(G) times the bars.
"""
import math

import pytest
import torch

import oracle
from seeded_inputs import CONFIGS, Workload, make_inputs
from tests.parity import assert_close_stored, assert_lse

pytestmark = pytest.mark.gpu


def assert_group_sum_close(name, got, ref, group):
    return assert_close_stored(name, got, ref, spread=math.sqrt(group))


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


def run(fa, w, inp, backward=True):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    grads = None
    if backward:
        grads = fa.backward(q, k, v, o, inp["do"].cuda(), lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    return o, lse, grads


def check_group(inp, w, o, lse, grads, b, g, row_block=None):
    """Every row of K/V head (b, g) and of the query heads that read it."""
    grp = w.H // w.kv_heads
    hs = slice(g * grp, (g + 1) * grp)
    q, k, v = inp["q"][b, hs], inp["k"][b, g:g + 1], inp["v"][b, g:g + 1]
    o_ref, l_ref = oracle.forward_gqa(q, k, v, w.causal, w.scale, row_block=row_block)
    assert_close_stored(f"O[{b},{hs}]", o[b, hs], o_ref)
    assert_lse(lse[b, hs], l_ref)
    if grads is not None:
        r = oracle.backward_gqa(q, k, v, inp["do"][b, hs], w.causal, w.scale, row_block=row_block)
        assert_close_stored(f"dQ[{b},{hs}]", grads[0][b, hs], r[0])
        assert_group_sum_close(f"dK[{b},{g}]", grads[1][b, g:g + 1], r[1], grp)
        assert_group_sum_close(f"dV[{b},{g}]", grads[2][b, g:g + 1], r[2], grp)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (8, 8)])
@pytest.mark.parametrize("S", [17, 300])
def test_small_shapes(fa, D, dtype, causal, H, Hkv, S):
    """Whole tensors against the oracle: GQA (G = 2), MQA (G = 6) and G = 1, ragged S."""
    w = Workload("gqa_small", 2, H, S, D, dtype, causal, backward=True, seed=200 + S + D + H, H_kv=Hkv)
    inp = make_inputs(w)
    o, lse, (dq, dk, dv) = run(fa, w, inp)
    assert dk.shape == (2, Hkv, S, D) and dv.shape == (2, Hkv, S, D)
    o_ref, l_ref = oracle.forward_gqa(inp["q"], inp["k"], inp["v"], causal, w.scale)
    assert_close_stored("O", o, o_ref)
    assert_lse(lse, l_ref)
    r = oracle.backward_gqa(inp["q"], inp["k"], inp["v"], inp["do"], causal, w.scale)
    assert_close_stored("dQ", dq, r[0])
    assert_group_sum_close("dK", dk, r[1], H // Hkv)
    assert_group_sum_close("dV", dv, r[2], H // Hkv)


@pytest.mark.parametrize("causal", [False, True])
def test_group_of_one_matches_multihead_call_bitwise(fa, causal):
    """fa_fwd_gqa / fa_bwd_gqa with H_kv = H run the same kernels as fa_fwd / fa_bwd."""
    w = Workload("g1", 1, 4, 520, 64, "bf16", causal, backward=True, seed=5)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    B, H, S, D = q.shape
    o1, l1 = fa.forward(q, k, v, causal=causal)
    o2, l2 = torch.empty_like(q), torch.empty_like(l1)
    assert fa.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(), B, H, H, S, D,
                         causal, w.scale, fa.FA_BF16, torch.cuda.current_stream().cuda_stream) == 0
    g1 = fa.backward(q, k, v, o1, do, l1, causal=causal)
    g2 = [torch.empty_like(q) for _ in range(3)]
    ws = torch.empty(fa.fa_bwd_gqa_workspace_size(B, H, H, S, D), dtype=torch.uint8, device="cuda")
    assert fa.fa_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), do.data_ptr(), l1.data_ptr(),
                         g2[0].data_ptr(), g2[1].data_ptr(), g2[2].data_ptr(), B, H, H, S, D, causal, w.scale,
                         fa.FA_BF16, ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_shared_kv_equals_replicated_kv(fa):
    """A grouped call equals the multi-head call on K, V copied out to H heads:
    outputs and dQ bitwise; dK, dV equal the per-group sums of the copies'
    gradients up to the rounding of those sums (the grouped kernel sums in fp32
    before rounding once)."""
    w = Workload("rep", 2, 8, 777, 64, "fp16", True, backward=True, seed=6, H_kv=2)
    inp = make_inputs(w)
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True)
    kr, vr = (x.repeat_interleave(4, dim=1).contiguous() for x in (k, v))
    o2, lse2 = fa.forward(q, kr, vr, causal=True)
    dq2, dk2, dv2 = fa.backward(q, kr, vr, o2, do, lse2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(dq, dq2)
    for got, per_head in ((dk, dk2), (dv, dv2)):
        summed = per_head.float().view(2, 2, 4, 777, 64).sum(2)
        assert float((got.float() - summed).abs().max()) < 2e-2


def test_group_streamed_by_one_cta(fa):
    """Enough (K/V head, key tile) pairs to fill the GPU: each dK/dV CTA streams its whole group
    (no partial sums); causal bf16, two query heads per K/V head."""
    w = Workload("gqa_nosplit", 4, 8, 2432, 64, "bf16", True, backward=True, seed=7, H_kv=4)
    B, H, S, D = w.B, w.H, w.S, w.D
    assert fa.fa_bwd_gqa_workspace_size(B, H, w.kv_heads, S, D) == fa.fa_bwd_workspace_size(B, H, S, D)
    inp = make_inputs(w)
    o, lse, grads = run(fa, w, inp)
    for b, g in ((0, 0), (3, 3), (2, 1)):
        check_group(inp, w, o, lse, grads, b, g)


@pytest.mark.parametrize("name", ["gqa", "mqa"])
def test_full_size_sampled_groups(fa, name):
    """B4 H16 S4096 D64 causal fp16 with H_kv = 2 and 1: first and last K/V head, every row."""
    w = CONFIGS[name]
    inp = make_inputs(w)
    o, lse, grads = run(fa, w, inp)
    last = (w.B - 1, w.kv_heads - 1)
    for b, g in {(0, 0), last}:
        check_group(inp, w, o, lse, grads, b, g, row_block=1024)


def test_kv_head_argument_checks(fa):
    q = torch.zeros(1, 6, 64, 64, dtype=torch.float16, device="cuda")
    kv = torch.zeros(1, 4, 64, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        fa.forward(q, kv, kv)
    o, l = torch.empty_like(q), torch.empty(1, 6, 64, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for hk in (4, 0, 7, -1):
        st = fa.fa_fwd_gqa(q.data_ptr(), kv.data_ptr(), kv.data_ptr(), o.data_ptr(), l.data_ptr(), 1, 6, hk, 64, 64,
                           0, 0.125, fa.FA_FP16, s)
        assert fa.STATUS[st] == "FA_ERR_INVALID_ARG", hk
