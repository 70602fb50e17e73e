"""Blockwise online-softmax forward in fp64: a CPU trace of the recurrence.

TEST INFRASTRUCTURE ONLY (same rule as ``oracle.attention``).

This restates the FlashAttention-2 forward recurrence step by step so that the
tests can check it against the naive definition and against the hand-worked
example of "T5 讲解：FlashAttention forward" §④ (one query, four keys,
BLOCK_N = 2, D = 1).  Notation follows "从零训练语言模型（第二部分）" §安全 / 在线
softmax and §FlashAttention 简述:

  for each K/V block:
      m_new = max(m_old, rowmax(S_blk))
      alpha = exp(m_old - m_new)
      P~    = exp(S_blk - m_new)
      l     = alpha * l + rowsum(P~)
      acc   = alpha * acc + P~ V_blk
      m_old = m_new
  O = acc / l,  L = m + ln l

The initial state is m = -inf, l = 0, acc = 0; on the first block alpha is
exp(-inf) = 0 (T5 §④).  Causal blocks wholly above the diagonal are skipped,
with the loop bound at the end of the query block (T5 §⑤).
"""
from __future__ import annotations

import math

import torch

from .attention import as_f64, F64


def forward_blockwise(q, k, v, causal: bool, scale: float, block_m: int, block_n: int,
                      trace: list | None = None):
    """O, L via the online-softmax recurrence; appends per-block state to ``trace``."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    n_q, n_k = q.shape[-2], k.shape[-2]
    o = torch.empty(q.shape, dtype=F64)
    lse = torch.empty(q.shape[:-1], dtype=F64)
    for i0 in range(0, n_q, block_m):
        i1 = min(n_q, i0 + block_m)
        qi = q[..., i0:i1, :]
        rows = i1 - i0
        m = torch.full(q.shape[:-2] + (rows,), float("-inf"), dtype=F64)
        l = torch.zeros(q.shape[:-2] + (rows,), dtype=F64)
        acc = torch.zeros(q.shape[:-2] + (rows, q.shape[-1]), dtype=F64)
        hi = min(n_k, i1) if causal else n_k
        for j0 in range(0, hi, block_n):
            j1 = min(n_k, j0 + block_n)
            s = scale * torch.matmul(qi, k[..., j0:j1, :].transpose(-1, -2))
            if causal:
                qpos = torch.arange(i0, i1).view(-1, 1)
                kpos = torch.arange(j0, j1).view(1, -1)
                s = s.masked_fill(kpos > qpos, float("-inf"))
            m_new = torch.maximum(m, s.amax(dim=-1))
            alpha = torch.exp(m - m_new)
            p = torch.exp(s - m_new.unsqueeze(-1))
            l = alpha * l + p.sum(dim=-1)
            acc = alpha.unsqueeze(-1) * acc + torch.matmul(p, v[..., j0:j1, :])
            m = m_new
            if trace is not None:
                trace.append({"i0": i0, "j0": j0, "m": m.clone(), "alpha": alpha.clone(),
                              "l": l.clone(), "acc": acc.clone()})
        o[..., i0:i1, :] = acc / l.unsqueeze(-1)
        lse[..., i0:i1] = m + torch.log(l)
    return o, lse


def causal_blocks_visited(n: int, block_m: int, block_n: int) -> int:
    """Number of (Q-block, K-block) pairs the causal loop computes (T5 §⑤)."""
    total = 0
    for i0 in range(0, n, block_m):
        hi = min(n, i0 + block_m)
        total += math.ceil(hi / block_n)
    return total
