"""CPU fp64 oracle for packed variable-length batches (varlen).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

"Inside FlashAttention" §6.1 (variable-length packing): samples of different
lengths are concatenated into one long sequence with no padding; a prefix-sum
array cu_seqlens of batch + 1 entries marks where each sample starts, and no
token attends to a token of another sample.  The page's tensors are
[total_tokens, heads, d].

Layout and readings (where the page is silent):
  q, o, dq      [T, H, D]       T = cu_seqlens[-1] tokens, token-major;
  k, v, dk, dv  [T, H_kv, D]    (grouped K/V heads as in ``oracle.grouped``);
  lse           [H, T]          natural-log logsumexp, one row per head;
  cu_seqlens    [batch + 1]     cu[0] = 0, non-decreasing; sample b is tokens
                                cu[b] .. cu[b+1]-1, and may be empty;
  the same cu_seqlens serves queries and keys (each sample attends to
  itself), and the causal mask is top-left within each sample: its i-th
  token sees its tokens 0..i.

The method is then the per-sample definition, written out as such: each
sample is cut out, attended on its own by the grouped-head oracle, and put
back in place; gradients likewise (a sample's K/V rows get gradient only from
its own queries).
"""
from __future__ import annotations

import torch

from .attention import F64, as_f64
from .grouped import backward_gqa, forward_gqa


def _bounds(cu_seqlens):
    cu = [int(x) for x in torch.as_tensor(cu_seqlens).tolist()]
    if not cu or cu[0] != 0 or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError(f"cu_seqlens must start at 0 and not decrease: {cu}")
    return list(zip(cu[:-1], cu[1:]))


def _heads_first(x):
    """[n, heads, D] -> [heads, n, D]."""
    return x.transpose(0, 1)


def forward_varlen(q, k, v, cu_seqlens, causal: bool, scale: float):
    """O [T, H, D] and L [H, T] of a packed batch."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    T, H, _ = q.shape
    o = torch.zeros(q.shape, dtype=F64)
    lse = torch.zeros(H, T, dtype=F64)
    for a, b in _bounds(cu_seqlens):
        if b == a:
            continue
        ob, lb = forward_gqa(_heads_first(q[a:b]), _heads_first(k[a:b]), _heads_first(v[a:b]), causal, scale)
        o[a:b] = _heads_first(ob)
        lse[:, a:b] = lb
    return o, lse


def backward_varlen(q, k, v, do, cu_seqlens, causal: bool, scale: float):
    """(dQ [T, H, D], dK [T, H_kv, D], dV [T, H_kv, D]) of loss = <O, dO> for a packed batch."""
    q, k, v, do = as_f64(q), as_f64(k), as_f64(v), as_f64(do)
    dq = torch.zeros(q.shape, dtype=F64)
    dk = torch.zeros(k.shape, dtype=F64)
    dv = torch.zeros(v.shape, dtype=F64)
    for a, b in _bounds(cu_seqlens):
        if b == a:
            continue
        g = backward_gqa(_heads_first(q[a:b]), _heads_first(k[a:b]), _heads_first(v[a:b]), _heads_first(do[a:b]),
                         causal, scale)
        dq[a:b], dk[a:b], dv[a:b] = (_heads_first(x) for x in g)
    return dq, dk, dv
