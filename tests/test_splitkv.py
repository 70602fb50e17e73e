"""Split-KV forward and the logsumexp merge on the GPU (through the C ABI)
against the fp64 oracle.  Bars: ``assert_close_stored`` (cases beyond the
configured workloads); L max abs <= 1e-3."""
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


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_splitkv_forward(fa, D, dtype, causal, splits):
    """Whole tensors, S = 1000 (ragged last shard and tile), two query heads per K/V head."""
    w = Workload("skv", 1, 4, 1000, D, dtype, causal, seed=600 + D + splits, H_kv=2)
    inp = make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward_splitkv(q, k, v, causal=causal, scale=w.scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    o_ref, l_ref = oracle.forward_gqa(inp["q"], inp["k"], inp["v"], causal, w.scale)
    assert_close_stored("O", o, o_ref)
    assert_lse(lse, l_ref)


def test_splitkv_matches_unsplit_call(fa):
    """Shards merged by L against the one-pass forward: equal up to fp32 rounding of the merge."""
    w = Workload("skv2", 2, 4, 2048, 64, "bf16", True, seed=21)
    inp = make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward_splitkv(q, k, v, causal=True, num_splits=4)
    torch.cuda.synchronize()
    assert float((l1 - l2).abs().max()) < 1e-4
    assert float((o1.float() - o2.float()).abs().max()) < 2e-2


def test_merge_kernel(fa):
    """fa_merge_lse on random partials, some shards empty (L = -inf) and some rows empty in every shard."""
    P, rows, D = 5, 777, 64
    g = torch.Generator().manual_seed(3)
    o_p = torch.randn(P, rows, D, generator=g, dtype=torch.float32)
    l_p = torch.randn(P, rows, generator=g, dtype=torch.float32) * 3
    l_p[1, ::3] = float("-inf")
    o_p[1, ::3] = 0
    l_p[:, 10] = float("-inf")
    o_p[:, 10] = 0
    o, lse = fa.merge_lse(o_p.cuda(), l_p.cuda(), torch.float16)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.merge_lse(o_p, l_p)
    assert_close_stored("O", o, o_ref)
    fin = torch.isfinite(l_ref)
    assert bool(torch.isneginf(lse.cpu()[~fin]).all())
    assert_lse(lse.cpu()[fin], l_ref[fin])
    assert torch.count_nonzero(o[10]) == 0


def test_full_size_splitkv(fa):
    """One long causal head (B1 H1 S16384 D64 fp16), auto split count: sampled rows across shards."""
    w = CONFIGS["splitkv"]
    inp = make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    n = fa.fa_splitkv_num_splits(w.B, w.H, w.S, w.D)
    assert n > 1
    o, lse = fa.forward_splitkv(q, k, v, causal=True, num_splits=n)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    rows = [0, 1, 127, 128, 1663, 1664, 5000, 8191, 8192, 12345, 16383]
    o_ref, l_ref = oracle.forward_rows(inp["q"][0, 0], inp["k"][0, 0], inp["v"][0, 0], True, w.scale, rows)
    assert_close_stored("O", o[0, 0, rows], o_ref)
    assert_lse(lse[0, 0, rows], l_ref)


def test_splitkv_argument_checks(fa):
    q = torch.zeros(1, 2, 256, 64, dtype=torch.float16, device="cuda")
    o, l = torch.empty_like(q), torch.empty(1, 2, 256, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_size(1, 2, 256, 64, 2), dtype=torch.uint8, device="cuda")
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), l.data_ptr(), 1, 2, 2, 256, 64, 1)
    assert fa.STATUS[fa.fa_fwd_splitkv(*args, 0, 0.125, fa.FA_FP16, ws.data_ptr(), ws.numel(), s)] == \
        "FA_ERR_INVALID_ARG"
    assert fa.STATUS[fa.fa_fwd_splitkv(*args, 2, 0.125, fa.FA_FP16, ws.data_ptr(), 64, s)] == "FA_ERR_WORKSPACE"
    assert fa.fa_fwd_splitkv(*args, 2, 0.125, fa.FA_FP16, ws.data_ptr(), ws.numel(), s) == 0
    torch.cuda.synchronize()
