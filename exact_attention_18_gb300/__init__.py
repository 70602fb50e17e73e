"""Python binding of the exact-attention C-ABI library (fa.h) for GB300.

Argument marshalling only: every step of the attention computation runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.

The raw entry points keep the C names and signatures (pointers as ints):
``fa_fwd``, ``fa_fwd_gqa``, ``fa_bwd``, ``fa_bwd_marked``, ``fa_bwd_gqa``,
``fa_bwd_gqa_marked``, ``fa_bwd_noalloc``, ``fa_bwd_workspace_size``, ``fa_bwd_gqa_workspace_size``,
``fa_fwd_window``, ``fa_bwd_window``, ``fa_bwd_window_marked``, ``fa_fwd_splitkv``,
``fa_fwd_splitkv_workspace_size``, ``fa_splitkv_num_splits``, ``fa_merge_lse``,
``fa_fwd_varlen``, ``fa_bwd_varlen``, ``fa_bwd_varlen_marked``,
``fa_bwd_varlen_workspace_size``, ``fa_status_string``, ``fa_last_error_detail``,
``fa_check_device_errors``, ``fa_set_wait_limit_ns``.  ``forward`` and ``backward`` wrap them for
contiguous [B, H, S, D] CUDA tensors; K and V (and dK, dV) may have fewer heads
H_kv dividing H (grouped-query and multi-query attention), in which case they
call the ``_gqa`` entry points; ``window=(left, right)`` selects the
sliding-window entry points.  ``forward_varlen`` and ``backward_varlen`` do
the same for packed batches: [T, H, D] tensors and int32 ``cu_seqlens``.

The first call loads the compiled library and raises if it has not been built
(``python -m exact_attention_18_gb300.build``); there is no fallback
implementation.
"""
from __future__ import annotations

import ctypes
import math
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libfa_gb300.so")

__all__ = ["fa_fwd", "fa_fwd_gqa", "fa_bwd", "fa_bwd_marked", "fa_bwd_gqa", "fa_bwd_gqa_marked", "fa_bwd_noalloc",
           "fa_bwd_workspace_size", "fa_bwd_gqa_workspace_size", "fa_fwd_varlen", "fa_bwd_varlen",
           "fa_bwd_varlen_marked", "fa_bwd_varlen_workspace_size", "forward_varlen", "backward_varlen",
           "fa_fwd_window", "fa_bwd_window", "fa_bwd_window_marked", "fa_fwd_splitkv",
           "fa_fwd_splitkv_workspace_size", "fa_splitkv_num_splits", "fa_merge_lse", "forward_splitkv", "merge_lse", "fa_status_string", "fa_last_error_detail",
           "fa_check_device_errors", "fa_set_wait_limit_ns", "forward", "backward", "FAError", "FA_FP16", "FA_BF16", "STATUS",
           "library_path", "load_library"]

FA_FP16, FA_BF16 = 0, 1
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ALIGNMENT",
          4: "FA_ERR_WORKSPACE", 5: "FA_ERR_CUDA", 6: "FA_ERR_TIMEOUT"}

_lib = None


def _load():
    """Load the compiled library once; raise if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"the CUDA library {LIB_PATH} is not built; run "
                           "`python -m exact_attention_18_gb300.build` (nvcc, sm_103a) first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.restype = i32
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, i32, vp]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd_workspace_size.argtypes = [i64, i64, i64, i64]
    lib.fa_bwd.restype = i32
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, i32, vp, sz, vp]
    lib.fa_bwd_marked.restype = i32
    lib.fa_bwd_marked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, i32, vp, sz,
                                  vp, ctypes.POINTER(vp)]
    lib.fa_fwd_gqa.restype = i32
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp]
    lib.fa_bwd_gqa.restype = i32
    lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp, sz,
                               vp]
    lib.fa_bwd_gqa_marked.restype = i32
    lib.fa_bwd_gqa_marked.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32, f32, i32, vp,
                                      sz, vp, ctypes.POINTER(vp)]
    lib.fa_bwd_gqa_workspace_size.restype = sz
    lib.fa_bwd_gqa_workspace_size.argtypes = [i64, i64, i64, i64, i64]
    lib.fa_fwd_varlen.restype = i32
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, f32, i32, vp]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_bwd_varlen_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64]
    lib.fa_bwd_varlen.restype = i32
    lib.fa_bwd_varlen.argtypes = [vp] * 10 + [i64] * 6 + [i32, f32, i32, vp, sz, vp]
    lib.fa_bwd_varlen_marked.restype = i32
    lib.fa_bwd_varlen_marked.argtypes = [vp] * 10 + [i64] * 6 + [i32, f32, i32, vp, sz, vp, ctypes.POINTER(vp)]
    lib.fa_fwd_window.restype = i32
    lib.fa_fwd_window.argtypes = [vp] * 5 + [i64] * 5 + [i32, i64, i64, f32, i32, vp]
    lib.fa_bwd_window.restype = i32
    lib.fa_bwd_window.argtypes = [vp] * 9 + [i64] * 5 + [i32, i64, i64, f32, i32, vp, sz, vp]
    lib.fa_bwd_window_marked.restype = i32
    lib.fa_bwd_window_marked.argtypes = [vp] * 9 + [i64] * 5 + [i32, i64, i64, f32, i32, vp, sz, vp,
                                                                ctypes.POINTER(vp)]
    lib.fa_fwd_splitkv.restype = i32
    lib.fa_fwd_splitkv.argtypes = [vp] * 5 + [i64] * 5 + [i32, i64, f32, i32, vp, sz, vp]
    lib.fa_fwd_splitkv_workspace_size.restype = sz
    lib.fa_fwd_splitkv_workspace_size.argtypes = [i64] * 5
    lib.fa_splitkv_num_splits.restype = i64
    lib.fa_splitkv_num_splits.argtypes = [i64] * 4
    lib.fa_merge_lse.restype = i32
    lib.fa_merge_lse.argtypes = [vp] * 4 + [i64] * 3 + [i32, vp]
    lib.fa_bwd_noalloc.restype = i32
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, i32, vp]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [i32]
    lib.fa_last_error_detail.restype = ctypes.c_char_p
    lib.fa_last_error_detail.argtypes = []
    lib.fa_check_device_errors.restype = i32
    lib.fa_check_device_errors.argtypes = [vp]
    lib.fa_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    _lib = lib
    return lib


def library_path() -> str:
    return LIB_PATH


def load_library():
    """The ctypes handle of the compiled library (loading it if needed)."""
    return _load()


# ----------------------------------------------------------------------- raw C ABI
def fa_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, stream) -> int:
    return _load().fa_fwd(q, k, v, o, lse, B, H, S, D, int(causal), float(scale), int(dtype), stream)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, dtype, workspace, workspace_bytes,
           stream) -> int:
    return _load().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, int(causal), float(scale), int(dtype),
                       workspace, workspace_bytes, stream)


def fa_bwd_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, dtype, workspace,
                  workspace_bytes, stream, marks) -> int:
    arr = None
    if marks is not None:
        arr = (ctypes.c_void_p * 4)(*[m if m else None for m in marks])
    return _load().fa_bwd_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, int(causal), float(scale),
                                 int(dtype), workspace, workspace_bytes, stream, arr)


def fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, S, D, causal, scale, dtype, stream) -> int:
    return _load().fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, S, D, int(causal), float(scale), int(dtype), stream)


def fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, scale, dtype, workspace,
               workspace_bytes, stream) -> int:
    return _load().fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, int(causal), float(scale),
                              int(dtype), workspace, workspace_bytes, stream)


def fa_bwd_gqa_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, scale, dtype, workspace,
                      workspace_bytes, stream, marks) -> int:
    arr = None
    if marks is not None:
        arr = (ctypes.c_void_p * 4)(*[m if m else None for m in marks])
    return _load().fa_bwd_gqa_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, int(causal),
                                     float(scale), int(dtype), workspace, workspace_bytes, stream, arr)


def fa_fwd_window(q, k, v, o, lse, B, H, H_kv, S, D, causal, window_left, window_right, scale, dtype,
                  stream) -> int:
    return _load().fa_fwd_window(q, k, v, o, lse, B, H, H_kv, S, D, int(causal), int(window_left),
                                 int(window_right), float(scale), int(dtype), stream)


def fa_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, window_left, window_right, scale,
                  dtype, workspace, workspace_bytes, stream) -> int:
    return _load().fa_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, int(causal), int(window_left),
                                 int(window_right), float(scale), int(dtype), workspace, workspace_bytes, stream)


def fa_bwd_window_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, window_left, window_right,
                         scale, dtype, workspace, workspace_bytes, stream, marks) -> int:
    arr = None
    if marks is not None:
        arr = (ctypes.c_void_p * 4)(*[m if m else None for m in marks])
    return _load().fa_bwd_window_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, int(causal),
                                        int(window_left), int(window_right), float(scale), int(dtype), workspace,
                                        workspace_bytes, stream, arr)


def fa_fwd_splitkv(q, k, v, o, lse, B, H, H_kv, S, D, causal, num_splits, scale, dtype, workspace, workspace_bytes,
                   stream) -> int:
    return _load().fa_fwd_splitkv(q, k, v, o, lse, B, H, H_kv, S, D, int(causal), int(num_splits), float(scale),
                                  int(dtype), workspace, workspace_bytes, stream)


def fa_fwd_splitkv_workspace_size(B, H, S, D, num_splits) -> int:
    return _load().fa_fwd_splitkv_workspace_size(B, H, S, D, num_splits)


def fa_splitkv_num_splits(B, H, S, D) -> int:
    return _load().fa_splitkv_num_splits(B, H, S, D)


def fa_merge_lse(o_part, lse_part, o, lse, shards, rows, D, dtype, stream) -> int:
    return _load().fa_merge_lse(o_part, lse_part, o, lse, shards, rows, D, int(dtype), stream)


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, batch, max_seqlen, total, H, H_kv, D, causal, scale, dtype,
                  stream) -> int:
    return _load().fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, batch, max_seqlen, total, H, H_kv, D, int(causal),
                                 float(scale), int(dtype), stream)


def fa_bwd_varlen_workspace_size(batch, max_seqlen, total, H, H_kv, D) -> int:
    return _load().fa_bwd_varlen_workspace_size(batch, max_seqlen, total, H, H_kv, D)


def fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, max_seqlen, total, H, H_kv, D, causal, scale,
                  dtype, workspace, workspace_bytes, stream) -> int:
    return _load().fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, max_seqlen, total, H, H_kv,
                                 D, int(causal), float(scale), int(dtype), workspace, workspace_bytes, stream)


def fa_bwd_varlen_marked(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, max_seqlen, total, H, H_kv, D,
                         causal, scale, dtype, workspace, workspace_bytes, stream, marks) -> int:
    arr = None
    if marks is not None:
        arr = (ctypes.c_void_p * 4)(*[m if m else None for m in marks])
    return _load().fa_bwd_varlen_marked(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, max_seqlen, total, H,
                                        H_kv, D, int(causal), float(scale), int(dtype), workspace, workspace_bytes,
                                        stream, arr)


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, dtype, stream) -> int:
    """fa_bwd for callers that cannot allocate: its scratch is a fixed array inside the library."""
    return _load().fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, int(causal), float(scale),
                                  int(dtype), stream)


def fa_bwd_workspace_size(B, H, S, D) -> int:
    return _load().fa_bwd_workspace_size(B, H, S, D)


def fa_bwd_gqa_workspace_size(B, H, H_kv, S, D) -> int:
    return _load().fa_bwd_gqa_workspace_size(B, H, H_kv, S, D)


def fa_status_string(status: int) -> str:
    return _load().fa_status_string(status).decode()


def fa_last_error_detail() -> str:
    return _load().fa_last_error_detail().decode()


def fa_check_device_errors(stream=None) -> int:
    return _load().fa_check_device_errors(stream)


def fa_set_wait_limit_ns(ns: int) -> int:
    """Limit of each kernel pipeline wait from now on (0 = the 2 s default); returns the previous one."""
    return _load().fa_set_wait_limit_ns(ns)


# ----------------------------------------------------------------------- tensor wrappers
class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}: {fa_last_error_detail()}")
        self.status = status


def _check(status: int, what: str):
    if status != 0:
        raise FAError(status, what)


def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float16 or bfloat16")


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _bhsd(x, name):
    if x.dim() == 3:  # [B, S, D] with no head dimension
        x = x.unsqueeze(1)
    if x.dim() != 4 or not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor [B, H, S, D] (or [B, S, D])")
    return x


def _kv_heads(q, k, v):
    """H_kv of K, V [B, H_kv, S, D] against Q [B, H, S, D]; H must be a multiple of H_kv."""
    B, H, S, D = q.shape
    hk = k.shape[1]
    grouped = hk == H == 0 or (hk >= 1 and H % hk == 0)
    if k.shape != (B, hk, S, D) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype or not grouped:
        raise ValueError("k and v must be [B, H_kv, S, D] with H_kv dividing H, in q's dtype")
    return hk


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None,
            window=None):
    """O and fp32 natural-log LSE of exact attention; tensors [B, H, S, D] (or [B, S, D]).

    K and V may have H_kv heads with H a multiple of H_kv (grouped-query
    attention; query head h reads K/V head h // (H // H_kv)).  ``window =
    (left, right)`` restricts query i to keys i - left .. i + right (negative =
    unlimited).
    """
    import torch
    squeeze = q.dim() == 3
    q, k, v = _bhsd(q, "q"), _bhsd(k, "k"), _bhsd(v, "v")
    B, H, S, D = q.shape
    hk = _kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q) if out is None else out.view(q.shape)
    l = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if lse is None else lse.view(B, H, S)
    if window is not None:
        _check(fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, hk, S, D,
                             causal, window[0], window[1], scale, _dtype_code(q), _stream_ptr(stream)),
               "fa_fwd_window")
    elif hk == H:
        _check(fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, S, D, causal,
                      scale, _dtype_code(q), _stream_ptr(stream)), "fa_fwd")
    else:
        _check(fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, hk, S, D,
                          causal, scale, _dtype_code(q), _stream_ptr(stream)), "fa_fwd_gqa")
    if squeeze:
        return o.squeeze(1), l.squeeze(1)
    return o, l


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
             workspace=None, stream=None, window=None):
    """dQ, dK, dV of exact attention from the forward's O and LSE (recompute backward).

    With K, V of H_kv < H heads, dK and dV have H_kv heads and sum over each
    K/V head's group of query heads.
    """
    import torch
    squeeze = q.dim() == 3
    q, k, v, o, do = (_bhsd(x, n) for x, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")))
    B, H, S, D = q.shape
    hk = _kv_heads(q, k, v)
    if o.shape != q.shape or do.shape != q.shape:
        raise ValueError("o and do must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lse = lse.reshape(B, H, S)
    dq = torch.empty_like(q) if dq is None else dq.view(q.shape)
    dk = torch.empty_like(k) if dk is None else dk.view(k.shape)
    dv = torch.empty_like(k) if dv is None else dv.view(k.shape)
    need = fa_bwd_gqa_workspace_size(B, H, hk, S, D) if hk else 0
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if window is not None:
        _check(fa_bwd_window(*args, B, H, hk, S, D, causal, window[0], window[1], scale, _dtype_code(q), *ws),
               "fa_bwd_window")
    elif hk == H:
        _check(fa_bwd(*args, B, H, S, D, causal, scale, _dtype_code(q), *ws), "fa_bwd")
    else:
        _check(fa_bwd_gqa(*args, B, H, hk, S, D, causal, scale, _dtype_code(q), *ws), "fa_bwd_gqa")
    if squeeze:
        return dq.squeeze(1), dk.squeeze(1), dv.squeeze(1)
    return dq, dk, dv


def _packed(x, name, heads=None):
    if x.dim() != 3 or not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor [T, H, D]")
    if heads is not None and x.shape[1] != heads:
        raise ValueError(f"{name} must have {heads} heads")
    return x


def _cu(cu_seqlens, T):
    import torch
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_cuda \
            or not cu_seqlens.is_contiguous() or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 CUDA tensor [batch + 1]")
    return cu_seqlens.numel() - 1


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale: float | None = None,
                   out=None, lse=None, stream=None):
    """O [T, H, D] and L [H, T] of a packed batch (samples cu_seqlens[b] .. cu_seqlens[b+1]-1).

    ``max_seqlen`` must bound every sample length (a host integer, so no device
    read is needed); a violation is detected on the device and reported by
    ``fa_check_device_errors``.
    """
    import torch
    q = _packed(q, "q")
    T, H, D = q.shape
    k, v = _packed(k, "k"), _packed(v, "v")
    hk = k.shape[1]
    if k.shape[0] != T or k.shape[2] != D or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype \
            or hk < 1 or H % hk != 0:
        raise ValueError("k and v must be [T, H_kv, D] with H_kv dividing H, in q's dtype")
    batch = _cu(cu_seqlens, T)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), cu_seqlens.data_ptr(),
                         batch, int(max_seqlen), T, H, hk, D, causal, scale, _dtype_code(q), _stream_ptr(stream)),
           "fa_fwd_varlen")
    return o, l


def backward_varlen(q, k, v, o, do, lse, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: float | None = None, workspace=None, stream=None):
    """dQ [T, H, D], dK, dV [T, H_kv, D] of a packed batch from the forward's O and L."""
    import torch
    q, o, do = _packed(q, "q"), _packed(o, "o"), _packed(do, "do")
    T, H, D = q.shape
    k, v = _packed(k, "k"), _packed(v, "v")
    hk = k.shape[1]
    if o.shape != q.shape or do.shape != q.shape or v.shape != k.shape or hk < 1 or H % hk != 0:
        raise ValueError("o, do must match q; k, v must be [T, H_kv, D] with H_kv dividing H")
    batch = _cu(cu_seqlens, T)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    need = fa_bwd_varlen_workspace_size(batch, int(max_seqlen), T, H, hk, D)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens.data_ptr(), batch, int(max_seqlen),
                         T, H, hk, D, causal, scale, _dtype_code(q), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), _stream_ptr(stream)), "fa_bwd_varlen")
    return dq, dk, dv


def forward_splitkv(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int | None = None,
                    workspace=None, stream=None):
    """O and L of exact attention computed as key shards merged by logsumexp ([B, H, S, D] tensors)."""
    import torch
    q, k, v = _bhsd(q, "q"), _bhsd(k, "k"), _bhsd(v, "v")
    B, H, S, D = q.shape
    hk = _kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n = fa_splitkv_num_splits(B, H, S, D) if num_splits is None else int(num_splits)
    o = torch.empty_like(q)
    l = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    need = fa_fwd_splitkv_workspace_size(B, H, S, D, n)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), B, H, hk, S, D, causal,
                          n, scale, _dtype_code(q), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                          _stream_ptr(stream)), "fa_fwd_splitkv")
    return o, l


def merge_lse(o_part, lse_part, dtype, stream=None):
    """Merge fp32 partials o_part [P, rows, D], lse_part [P, rows] into (O [rows, D] of `dtype`, L [rows])."""
    import torch
    if o_part.dtype != torch.float32 or lse_part.dtype != torch.float32 or o_part.dim() != 3 \
            or lse_part.shape != o_part.shape[:2] or not o_part.is_contiguous() or not lse_part.is_contiguous():
        raise ValueError("o_part must be contiguous fp32 [P, rows, D] and lse_part fp32 [P, rows]")
    P, rows, D = o_part.shape
    o = torch.empty((rows, D), dtype=dtype, device=o_part.device)
    l = torch.empty((rows,), dtype=torch.float32, device=o_part.device)
    code = FA_FP16 if dtype == torch.float16 else FA_BF16
    _check(fa_merge_lse(o_part.data_ptr(), lse_part.data_ptr(), o.data_ptr(), l.data_ptr(), P, rows, D, code,
                        _stream_ptr(stream)), "fa_merge_lse")
    return o, l
