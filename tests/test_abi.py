"""The C-ABI library loads, exports every entry point fa.h declares, and rejects
bad arguments before any CUDA call (these tests need no GPU)."""
import ctypes
import os
import re

import pytest

import exact_attention_18_gb300 as fa
from exact_attention_18_gb300 import build as fab

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fab.build_library()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
                     "fa_last_error_detail", "fa_check_device_errors"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in fa.STATUS.items():
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


def test_wait_limit_setter_round_trip(lib):
    """0 restores the 2 s default; the setter returns the limit it replaces (no launch involved)."""
    old = fa.fa_set_wait_limit_ns(12345)
    try:
        assert fa.fa_set_wait_limit_ns(0) == 12345
        assert fa.fa_set_wait_limit_ns(0) == 2_000_000_000
    finally:
        fa.fa_set_wait_limit_ns(old)


def test_workspace_size(lib):
    assert fa.fa_bwd_workspace_size(2, 32, 8192, 128) == 2 * 32 * 8192 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 3, 64) == 256  # rounded up to 256 bytes
    assert fa.fa_bwd_workspace_size(0, 4, 16, 64) == 0


def test_gqa_workspace_size(lib):
    """Delta for every query row, plus fp32 partial dK/dV rows when the dK/dV pass splits a group."""
    delta = 4 * 16 * 4096 * 4
    assert fa.fa_bwd_gqa_workspace_size(1, 4, 4, 128, 64) == fa.fa_bwd_workspace_size(1, 4, 128, 64)
    # 8 K/V heads x 32 key tiles = 256 CTAs < 304: two CTAs share each (K/V head, key tile)
    assert fa.fa_bwd_gqa_workspace_size(4, 16, 2, 4096, 64) == delta + 2 * 8 * 4096 * 128 * 4
    # 4 x 32 = 128 CTAs: four per (K/V head, key tile), four query heads each
    assert fa.fa_bwd_gqa_workspace_size(4, 16, 1, 4096, 64) == delta + 4 * 4 * 4096 * 128 * 4
    # enough CTAs from the K/V heads alone: no partial sums
    assert fa.fa_bwd_gqa_workspace_size(4, 8, 4, 2432, 64) == 4 * 8 * 2432 * 4
    # too few CTAs even with one head per CTA: split over the whole group
    assert fa.fa_bwd_gqa_workspace_size(1, 8, 2, 256, 64) == 1 * 8 * 256 * 4 + 4 * 2 * 256 * 128 * 4
    assert fa.fa_bwd_gqa_workspace_size(1, 6, 4, 128, 64) == 0
    assert fa.fa_bwd_gqa_workspace_size(0, 6, 3, 128, 64) == 0


P = 0x10000  # a fake, 16-byte aligned address: never dereferenced by these calls


def fwd(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=1, S=128, D=64, causal=0, scale=0.125, dtype=0, stream=None)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["S"], a["D"], a["causal"],
                     a["scale"], a["dtype"], a["stream"])


def bwd(**kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, B=1, H=1, S=128, D=64, causal=0, scale=0.125,
             dtype=0, ws=P * 16, wsb=1 << 20, stream=None)
    a.update(kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"], a["H"],
                     a["S"], a["D"], a["causal"], a["scale"], a["dtype"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=48), 2), (dict(D=256), 2), (dict(D=8), 2),
    (dict(q=0), 1), (dict(lse=0), 1), (dict(o=0), 1),
    (dict(k=P + 8), 3), (dict(v=P + 2), 3), (dict(lse=P + 4), 3),
    (dict(S=-1), 1), (dict(B=-2), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(dtype=7), 1),
    (dict(S=65536 * 128), 2),
])
def test_fwd_rejects_bad_arguments(lib, kw, status):
    assert fwd(**kw) == status
    assert fa.fa_last_error_detail() != ""


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=0), dict(S=0), dict(S=0, q=0, k=0, v=0, o=0, lse=0)])
def test_fwd_empty_is_a_no_op(lib, kw):
    assert fwd(**kw) == 0


def test_empty_call_still_validates_shape_arguments(lib):
    assert fwd(S=0, D=48) == 2
    assert fwd(B=0, scale=float("nan")) == 1


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), 2), (dict(do=0), 1), (dict(dq=P + 8), 3), (dict(ws=0), 4), (dict(wsb=100), 4),
    (dict(ws=P * 16 + 16), 3), (dict(scale=float("-inf")), 1),
])
def test_bwd_rejects_bad_arguments(lib, kw, status):
    assert bwd(**kw) == status
    assert fa.fa_last_error_detail() != ""


def test_bwd_empty_is_a_no_op(lib):
    assert bwd(S=0) == 0
    assert bwd(B=0, ws=0, wsb=0) == 0
    assert bwd(S=0, q=0, dq=0, ws=0, wsb=0) == 0


def fwd_gqa(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H=4, H_kv=2, S=128, D=64, causal=0, scale=0.125, dtype=0, stream=None)
    a.update(kw)
    return fa.fa_fwd_gqa(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["H_kv"], a["S"], a["D"],
                         a["causal"], a["scale"], a["dtype"], a["stream"])


def bwd_gqa(**kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, B=1, H=4, H_kv=2, S=128, D=64, causal=0,
             scale=0.125, dtype=0, ws=P * 16, wsb=1 << 20, stream=None)
    a.update(kw)
    return fa.fa_bwd_gqa(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"],
                         a["H"], a["H_kv"], a["S"], a["D"], a["causal"], a["scale"], a["dtype"], a["ws"], a["wsb"],
                         a["stream"])


GQA_BAD = [
    (dict(H=6, H_kv=4), 1), (dict(H_kv=0), 1), (dict(H_kv=8), 1), (dict(H_kv=-1), 1), (dict(H=0, H_kv=1), 1),
    (dict(H=0, H_kv=0, D=48), 2), (dict(D=48), 2), (dict(k=P + 8), 3), (dict(q=0), 1),
]


@pytest.mark.parametrize("kw,status", GQA_BAD)
def test_fwd_gqa_rejects_bad_arguments(lib, kw, status):
    assert fwd_gqa(**kw) == status
    assert fa.fa_last_error_detail() != ""


@pytest.mark.parametrize("kw,status", GQA_BAD + [(dict(ws=0), 4), (dict(dk=P + 4), 3)])
def test_bwd_gqa_rejects_bad_arguments(lib, kw, status):
    assert bwd_gqa(**kw) == status
    assert fa.fa_last_error_detail() != ""


@pytest.mark.parametrize("kw", [dict(H=0, H_kv=0), dict(B=0), dict(S=0, q=0, k=0, v=0, o=0, lse=0)])
def test_gqa_empty_is_a_no_op(lib, kw):
    assert fwd_gqa(**kw) == 0
    assert bwd_gqa(**kw) == 0


def fwd_varlen(**kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, cu=P, batch=2, max_seqlen=128, total=200, H=4, H_kv=2, D=64, causal=1,
             scale=0.125, dtype=0, stream=None)
    a.update(kw)
    return fa.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["batch"], a["max_seqlen"],
                            a["total"], a["H"], a["H_kv"], a["D"], a["causal"], a["scale"], a["dtype"], a["stream"])


def bwd_varlen(**kw):
    a = dict(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, cu=P, batch=2, max_seqlen=128, total=200, H=4,
             H_kv=2, D=64, causal=1, scale=0.125, dtype=0, ws=P * 16, wsb=1 << 24, stream=None)
    a.update(kw)
    return fa.fa_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"], a["dv"], a["cu"],
                            a["batch"], a["max_seqlen"], a["total"], a["H"], a["H_kv"], a["D"], a["causal"],
                            a["scale"], a["dtype"], a["ws"], a["wsb"], a["stream"])


VARLEN_BAD = [
    (dict(cu=0), 1), (dict(cu=P + 2), 3), (dict(total=-1), 1), (dict(max_seqlen=-5), 1), (dict(batch=-1), 1),
    (dict(H_kv=3), 1), (dict(D=80), 2), (dict(q=P + 8), 3), (dict(total=1 << 31), 2),
    (dict(max_seqlen=65536 * 128), 2),
]


@pytest.mark.parametrize("kw,status", VARLEN_BAD)
def test_fwd_varlen_rejects_bad_arguments(lib, kw, status):
    assert fwd_varlen(**kw) == status
    assert fa.fa_last_error_detail() != ""


@pytest.mark.parametrize("kw,status", VARLEN_BAD + [(dict(ws=0), 4), (dict(wsb=64), 4), (dict(dv=P + 4), 3)])
def test_bwd_varlen_rejects_bad_arguments(lib, kw, status):
    assert bwd_varlen(**kw) == status
    assert fa.fa_last_error_detail() != ""


@pytest.mark.parametrize("kw", [dict(batch=0), dict(total=0), dict(max_seqlen=0), dict(H=0, H_kv=0),
                                dict(total=0, cu=0, q=0, k=0, v=0, o=0, lse=0)])
def test_varlen_empty_is_a_no_op(lib, kw):
    assert fwd_varlen(**kw) == 0
    assert bwd_varlen(**kw) == 0


def test_varlen_workspace_size(lib):
    # Delta: 4 heads x 700 tokens; 3 samples x 2 K/V heads x 3 tiles = 18 CTAs -> the group (2) is split
    assert fa.fa_bwd_varlen_workspace_size(3, 300, 700, 4, 2, 64) == 11264 + 2 * 700 * 2 * 128 * 4
    assert fa.fa_bwd_varlen_workspace_size(3, 300, 700, 4, 4, 64) == 11264
    assert fa.fa_bwd_varlen_workspace_size(3, 300, 700, 4, 3, 64) == 0


def test_splitkv_sizes_and_checks(lib):
    # S = 16384 in ten shards of 1664 keys (1639 rounded up to 128): 10 * 16384 * (64 + 1) floats
    assert fa.fa_splitkv_num_splits(1, 1, 16384, 64) == 10
    assert fa.fa_splitkv_num_splits(4, 16, 4096, 64) == 1
    assert fa.fa_splitkv_num_splits(1, 1, 100, 64) == 1
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 16384, 64, 10) == 10 * 16384 * 65 * 4
    assert fa.fa_fwd_splitkv_workspace_size(1, 1, 16384, 64, 0) == 0
    args = (P, P, P, P, P, 1, 2, 2, 256, 64, 1)
    assert fa.fa_fwd_splitkv(*args, 0, 0.125, 0, P * 16, 1 << 20, None) == 1
    assert fa.fa_fwd_splitkv(*args, 2, 0.125, 0, 0, 1 << 20, None) == 4
    assert fa.fa_fwd_splitkv(*args, 2, 0.125, 0, P * 16, 16, None) == 4
    assert fa.fa_fwd_splitkv(*args, 2, 0.125, 0, P * 16 + 8, 1 << 20, None) == 3
    assert fa.fa_fwd_splitkv(P, P, P, P, P, 1, 2, 2, 256, 48, 1, 2, 0.125, 0, P * 16, 1 << 20, None) == 2


def test_merge_checks(lib):
    assert fa.fa_merge_lse(P, P, P, P, 0, 10, 64, 0, None) == 1
    assert fa.fa_merge_lse(P, P, P, P, 2, 10, 80, 0, None) == 2
    assert fa.fa_merge_lse(P, P, P, P, 2, 10, 64, 5, None) == 1
    assert fa.fa_merge_lse(P + 4, P, P, P, 2, 10, 64, 0, None) == 3
    assert fa.fa_merge_lse(0, 0, 0, 0, 2, 0, 64, 0, None) == 0  # no rows: nothing to do


def test_binding_has_no_fallback(monkeypatch):
    """Without the compiled library the binding raises instead of computing anything."""
    import importlib
    mod = importlib.import_module("exact_attention_18_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    monkeypatch.setattr(mod, "LIB_PATH", "/nonexistent/libfa_gb300.so")
    with pytest.raises(RuntimeError, match="not built"):
        mod.fa_status_string(0)
