"""CPU fp64 oracle for split-KV attention and the logsumexp merge of shards.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may use it.

"T5 讲解" §⑥: storing L = m + log l (the row's logsumexp) is what allows the
results of shards to be merged.  Split the keys into shards s; per shard the
row has a normalised partial output O_s (softmax over the shard's keys only)
and its logsumexp L_s.  Since exp(L_s) is the shard's total softmax mass,

  L = ln sum_s exp(L_s),      O = sum_s exp(L_s - L) O_s

is the attention over all keys.  A shard in which a row sees no key has
L_s = -inf and O_s = 0 (weight 0); a row with no key at all gets O = 0,
L = -inf.  ``merge_lse`` writes that formula out; ``forward_shards`` gives the
per-shard partials straight from the definition (the other keys masked).
"""
from __future__ import annotations

import torch

from .attention import F64, as_f64, scores, softmax_rows


def forward_shards(q, k, v, causal: bool, scale: float, bounds):
    """Per-shard (O_s, L_s) for key ranges bounds = [(k0, k1), ...]: O [P, ..., S, D], L [P, ..., S]."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    outs, lses = [], []
    nk = k.shape[-2]
    for k0, k1 in bounds:
        s = scores(q, k, scale, causal)
        kj = torch.arange(nk).view(1, nk)
        s = s.masked_fill((kj < k0) | (kj >= k1), float("-inf"))
        p, lse = softmax_rows(s)
        outs.append(torch.matmul(p, v))
        lses.append(lse)
    return torch.stack(outs), torch.stack(lses)


def merge_lse(o_parts, lse_parts):
    """Merge shards: o_parts [P, ..., D], lse_parts [P, ...] -> (O [..., D], L [...])."""
    o_parts, lse_parts = as_f64(o_parts), as_f64(lse_parts)
    m = lse_parts.amax(dim=0)
    empty = torch.isinf(m) & (m < 0)
    m_safe = torch.where(empty, torch.zeros_like(m), m)
    w = torch.exp(lse_parts - m_safe)                 # exp(L_s - m), 0 for L_s = -inf
    total = w.sum(dim=0)
    lse = torch.where(empty, torch.full_like(m, float("-inf")), m_safe + torch.log(total))
    wn = torch.where(empty, torch.zeros_like(w), w / torch.where(empty, torch.ones_like(total), total))
    o = (wn.unsqueeze(-1) * o_parts).sum(dim=0)       # sum_s exp(L_s - L) O_s
    return o, lse


def split_bounds(S: int, chunk: int):
    """Key ranges [k0, k0 + chunk) covering 0 .. S-1."""
    return [(k0, min(S, k0 + chunk)) for k0 in range(0, S, chunk)]


__all__ = ["forward_shards", "merge_lse", "split_bounds", "F64"]
