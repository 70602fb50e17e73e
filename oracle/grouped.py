"""CPU fp64 oracle for grouped-query and multi-query attention (GQA / MQA).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

"Inside FlashAttention" §6.1 (the MQA / GQA interface): several query heads
share one K/V head; K and V are passed with fewer heads H_kv and are not
copied out to H heads.  Its example has 32 query heads on 4 K/V heads, so 8
query heads per K/V head.

Reading where the page is silent: the page does not say WHICH query heads
share a K/V head.  Here query head h reads K/V head h // G with G = H / H_kv,
i.e. each K/V head serves a run of G consecutive query heads (the grouping
that keeps a group's query heads adjacent in memory).

With that map the method is ordinary attention per query head:

  O_h = softmax(scale * Q_h K_{h//G}^T (+ causal mask)) V_{h//G},

and, since K/V head g enters the loss through every query head of its group,
its gradients are the sums over the group:

  dK_g = sum_{h : h//G = g} dK_h,    dV_g = sum_{h : h//G = g} dV_h,

where dK_h, dV_h are the per-head gradients of the multi-head backward.
Both are written below exactly so: K and V repeated out to H heads (the copy
the page says the fused kernel avoids; here it is only the definition), the
multi-head oracle, and a sum over each group.
"""
from __future__ import annotations

import torch

from .attention import as_f64, backward, forward


def group_size(h_q: int, h_kv: int) -> int:
    """G = H / H_kv query heads per K/V head; H must be a positive multiple of H_kv."""
    if h_kv < 1 or h_q % h_kv != 0:
        raise ValueError(f"H={h_q} is not a positive multiple of H_kv={h_kv}")
    return h_q // h_kv


def expand_kv(x: torch.Tensor, h_q: int) -> torch.Tensor:
    """[..., H_kv, S, D] -> [..., H, S, D]: query head h gets K/V head h // G."""
    g = group_size(h_q, x.shape[-3])
    return torch.repeat_interleave(as_f64(x), g, dim=-3)


def forward_gqa(q, k, v, causal: bool, scale: float, row_block: int | None = None, window=None):
    """O [..., H, S, D] and L [..., H, S] with K, V of H_kv heads (window as in ``oracle.forward``)."""
    h_q = q.shape[-3]
    return forward(q, expand_kv(k, h_q), expand_kv(v, h_q), causal, scale, row_block=row_block, window=window)


def backward_gqa(q, k, v, do, causal: bool, scale: float, row_block: int | None = None, window=None):
    """(dQ [..., H, S, D], dK [..., H_kv, S, D], dV [..., H_kv, S, D]) of loss = <O, dO>."""
    h_q, h_kv = q.shape[-3], k.shape[-3]
    g = group_size(h_q, h_kv)
    dq, dk_h, dv_h = backward(q, expand_kv(k, h_q), expand_kv(v, h_q), do, causal, scale, row_block=row_block,
                              window=window)
    lead = dk_h.shape[:-3]
    s, d = dk_h.shape[-2], dk_h.shape[-1]
    dk = dk_h.reshape(*lead, h_kv, g, s, d).sum(dim=-3)
    dv = dv_h.reshape(*lead, h_kv, g, s, d).sum(dim=-3)
    return dq, dk, dv
