"""Packed variable-length batches on the GPU (through the C ABI) against the
fp64 varlen oracle, on the library's own forward outputs.

Bars as for the grouped-head tests (cases beyond the configured workloads):
``assert_close_stored`` with sqrt(G) for dK and dV of grouped heads.
"""
import math

import pytest
import torch

import oracle
from seeded_inputs import PACKED_CONFIGS, PackedWorkload, make_packed_inputs
from tests.parity import assert_close_stored, assert_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_18_gb300 as m
    m.load_library()
    return m


def run(fa, w, inp, backward=True, max_seqlen=None):
    q, k, v, do = (inp[n].cuda() for n in ("q", "k", "v", "do"))
    cu = inp["cu_seqlens"].cuda()
    ms = w.max_seqlen if max_seqlen is None else max_seqlen
    o, lse = fa.forward_varlen(q, k, v, cu, ms, causal=w.causal, scale=w.scale)
    grads = fa.backward_varlen(q, k, v, o, do, lse, cu, ms, causal=w.causal, scale=w.scale) if backward else None
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    return o, lse, grads


def check(inp, w, o, lse, grads, tokens=None):
    """Every row against the oracle (or only the samples covering ``tokens``)."""
    grp = w.H // w.kv_heads
    cu = inp["cu_seqlens"].tolist()
    spans = list(zip(cu[:-1], cu[1:]))
    if tokens is not None:
        spans = [(a, b) for a, b in spans if any(a <= t < b for t in tokens)]
    for a, b in spans:
        if a == b:
            continue
        sub = {n: inp[n][a:b] for n in ("q", "k", "v", "do")}
        cu1 = torch.tensor([0, b - a])
        o_ref, l_ref = oracle.forward_varlen(sub["q"], sub["k"], sub["v"], cu1, w.causal, w.scale)
        assert_close_stored(f"O[{a}:{b}]", o[a:b], o_ref)
        assert_lse(lse[:, a:b], l_ref)
        if grads is not None:
            r = oracle.backward_varlen(sub["q"], sub["k"], sub["v"], sub["do"], cu1, w.causal, w.scale)
            assert_close_stored(f"dQ[{a}:{b}]", grads[0][a:b], r[0])
            assert_close_stored(f"dK[{a}:{b}]", grads[1][a:b], r[1], spread=math.sqrt(grp))
            assert_close_stored(f"dV[{a}:{b}]", grads[2][a:b], r[2], spread=math.sqrt(grp))


MIXES = {
    "ragged": (17, 300, 1, 0, 130, 257),        # ragged tails, an empty and a one-token sample
    "tiles": (128, 512, 256),                   # whole tiles
    "one": (389,),                              # a single sample
}


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mix", sorted(MIXES))
def test_packed_batches(fa, D, dtype, causal, mix):
    w = PackedWorkload("packed", MIXES[mix], 4, D, dtype, causal, seed=300 + D + len(mix), H_kv=2)
    inp = make_packed_inputs(w)
    o, lse, grads = run(fa, w, inp)
    check(inp, w, o, lse, grads)


@pytest.mark.parametrize("Hkv", [1, 3])
def test_packed_grouped_heads(fa, Hkv):
    """MQA and G = 1 (H = 3) inside a packed batch."""
    w = PackedWorkload("packed_g", (200, 77, 640), 3, 64, "bf16", True, seed=9, H_kv=Hkv)
    inp = make_packed_inputs(w)
    o, lse, grads = run(fa, w, inp)
    check(inp, w, o, lse, grads)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_the_batched_call_bitwise(fa, causal):
    """B samples of length S packed equal fa_fwd / fa_bwd on [B, H, S, D], rearranged, bit for bit."""
    B, H, S, D = 3, 4, 384, 64
    w = PackedWorkload("eq", (S,) * B, H, D, "fp16", causal, seed=11)
    inp = make_packed_inputs(w)
    o, lse, (dq, dk, dv) = run(fa, w, inp)
    unpack = lambda x: x.view(B, S, x.shape[1], D).permute(0, 2, 1, 3).contiguous()  # noqa: E731
    q, k, v, do = (unpack(inp[n]).cuda() for n in ("q", "k", "v", "do"))
    o2, lse2 = fa.forward(q, k, v, causal=causal)
    dq2, dk2, dv2 = fa.backward(q, k, v, o2, do, lse2, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(unpack(o), o2)
    assert torch.equal(lse.view(H, B, S).permute(1, 0, 2), lse2)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(unpack(a), b)


def test_samples_do_not_see_each_other(fa):
    """Changing one sample's tokens leaves every other sample's outputs bitwise unchanged."""
    w = PackedWorkload("iso", (300, 200, 333), 4, 64, "fp16", True, seed=12)
    inp = make_packed_inputs(w)
    o1, l1, g1 = run(fa, w, inp)
    inp2 = {n: t.clone() for n, t in inp.items()}
    for n in ("q", "k", "v", "do"):
        inp2[n][300:500] = -inp2[n][300:500]
    o2, l2, g2 = run(fa, w, inp2)
    keep = torch.cat([torch.arange(0, 300), torch.arange(500, 833)]).cuda()
    assert torch.equal(o1[keep], o2[keep]) and torch.equal(l1[:, keep], l2[:, keep])
    for a, b in zip(g1, g2):
        assert torch.equal(a[keep], b[keep])


def test_full_size_packed_workload(fa):
    """The packed benchmark workload (16384 tokens in ten samples, causal H16 D64 fp16):
    the shortest, a middle and the longest sample, every row."""
    w = PACKED_CONFIGS["varlen"]
    inp = make_packed_inputs(w)
    o, lse, grads = run(fa, w, inp)
    cu = inp["cu_seqlens"].tolist()
    longest = max(range(w.batch), key=lambda b: w.lengths[b])
    shortest = min(range(w.batch), key=lambda b: w.lengths[b])
    check(inp, w, o, lse, grads, tokens=[cu[longest], cu[shortest], cu[4]])


def test_sample_longer_than_max_seqlen_is_reported(fa):
    """cu_seqlens that contradict max_seqlen are caught by the kernels' own check before any
    access; fa_check_device_errors reports FA_ERR_INVALID_ARG and the context stays usable."""
    w = PackedWorkload("bad", (100, 300), 2, 64, "fp16", True, seed=13)
    inp = make_packed_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"].cuda()
    fa.forward_varlen(q, k, v, cu, 200, causal=True)
    assert fa.STATUS[fa.fa_check_device_errors(None)] == "FA_ERR_INVALID_ARG"
    o, lse = fa.forward_varlen(q, k, v, cu, 300, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_check_device_errors(None) == 0
    assert torch.isfinite(o.float()).all()


def test_varlen_argument_checks(fa):
    q = torch.zeros(64, 4, 64, dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    o, l = torch.empty_like(q), torch.empty(4, 64, dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_varlen(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), l.data_ptr(), 0, 1, 64, 64, 4, 4,
                          64, 1, 0.125, fa.FA_FP16, s)
    assert fa.STATUS[st] == "FA_ERR_INVALID_ARG"
    st = fa.fa_fwd_varlen(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), l.data_ptr(), cu.data_ptr() + 2, 1,
                          64, 64, 4, 4, 64, 1, 0.125, fa.FA_FP16, s)
    assert fa.STATUS[st] == "FA_ERR_ALIGNMENT"
    st = fa.fa_fwd_varlen(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), l.data_ptr(), cu.data_ptr(), 1,
                          64, 64, 4, 3, 64, 1, 0.125, fa.FA_FP16, s)
    assert fa.STATUS[st] == "FA_ERR_INVALID_ARG"
    with pytest.raises(ValueError):
        fa.forward_varlen(q, q, q, cu.long(), 64)
