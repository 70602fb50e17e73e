"""CPU fp64 oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA library and never calls it.

Everything here is the plain, materialised definition, in float64 on the CPU:

  S = scale * Q K^T                          (causal: S_ij = -inf for key j > query i)
  m_i = max_j S_ij
  P_ij = exp(S_ij - m_i) / sum_t exp(S_it - m_i)
  O = P V
  L_i = m_i + ln sum_t exp(S_it - m_i)       (natural-log logsumexp of the scaled scores)

following "从零训练语言模型（第二部分：FlashAttention 与设备内存）" §安全 / 在线 softmax and
§使用 LSE 连接正向和反向传播, "Inside FlashAttention" §1.1, and the naive
attention listing of the leightonwang "fa-triton" post (§性能测试).

Backward, with loss gradient dO given (same pages, §反向传播):

  dV = P^T dO
  dP = dO V^T
  dS = P o (dP - rowsum(P o dP))    (closed-form softmax Jacobian, row by row)
  dQ = scale * dS K
  dK = scale * dS^T Q

The row term is computed as rowsum(P o dP) straight from the Jacobian
diag(P_i) - P_i P_i^T; the pages' shortcut rowsum(dO o O) equals it, and the
tests check that identity separately.

Readings where the pages are silent: the exported L uses the natural log; a
query row whose keys are all masked (unreachable with equal query and key
lengths and a top-left causal mask) gets O_i = 0 and L_i = -inf.

``row_block`` only bounds memory: each block of query rows is computed from its
complete score rows, exactly as above; dK and dV then sum the per-block terms.

Window band ("Inside FlashAttention" §6.1, sliding window: only keys inside a
window around the query count, ``window_size=(left, right)``): with
``window=(left, right)`` key j is visible to query i only if
i - left <= j <= i + right, a negative side meaning unlimited; ``causal``
additionally hides j > i (so causal with (left, 0) is the page's example).
The band is applied as one more -inf mask on S, nothing else changes.
"""
from __future__ import annotations

import torch

F64 = torch.float64


def as_f64(x: torch.Tensor) -> torch.Tensor:
    """Exact upcast of the caller's (fp16/bf16/fp32) values to CPU float64."""
    return x.detach().to(device="cpu", dtype=F64)


def scores(q: torch.Tensor, k: torch.Tensor, scale: float, causal: bool,
           row_start: int = 0, window=None) -> torch.Tensor:
    """S = scale * q k^T for query rows row_start.. of q; -inf above the diagonal if
    causal, and outside the band i - left <= j <= i + right if a window is given."""
    s = scale * torch.matmul(q, k.transpose(-1, -2))
    nq, nk = s.shape[-2], s.shape[-1]
    qi = torch.arange(row_start, row_start + nq).view(nq, 1)
    kj = torch.arange(nk).view(1, nk)
    if causal:
        s = s.masked_fill(kj > qi, float("-inf"))
    if window is not None:
        left, right = window
        if left is not None and left >= 0:
            s = s.masked_fill(kj < qi - left, float("-inf"))
        if right is not None and right >= 0:
            s = s.masked_fill(kj > qi + right, float("-inf"))
    return s


def softmax_rows(s: torch.Tensor):
    """Row softmax P and logsumexp L of the score rows s (max-subtracted form)."""
    m = s.amax(dim=-1, keepdim=True)
    m_safe = torch.where(torch.isinf(m) & (m < 0), torch.zeros_like(m), m)
    e = torch.exp(s - m_safe)
    l = e.sum(dim=-1, keepdim=True)
    empty = l == 0
    p = torch.where(empty, torch.zeros_like(e), e / torch.where(empty, torch.ones_like(l), l))
    lse = torch.where(empty, torch.full_like(l, float("-inf")), m_safe + torch.log(l))
    return p, lse.squeeze(-1)


def forward(q, k, v, causal: bool, scale: float, row_block: int | None = None, window=None):
    """Exact attention output O [..., S, D] and logsumexp L [..., S] in fp64."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    n = q.shape[-2]
    rb = n if row_block is None else max(1, int(row_block))
    o = torch.empty(q.shape, dtype=F64)
    lse = torch.empty(q.shape[:-1], dtype=F64)
    for r0 in range(0, n, rb):
        r1 = min(n, r0 + rb)
        p, l_blk = softmax_rows(scores(q[..., r0:r1, :], k, scale, causal, r0, window))
        o[..., r0:r1, :] = torch.matmul(p, v)
        lse[..., r0:r1] = l_blk
    return o, lse


def backward(q, k, v, do, causal: bool, scale: float, row_block: int | None = None, window=None):
    """Gradients (dQ, dK, dV) of loss = <O, dO> from the closed-form softmax Jacobian."""
    q, k, v, do = as_f64(q), as_f64(k), as_f64(v), as_f64(do)
    n = q.shape[-2]
    rb = n if row_block is None else max(1, int(row_block))
    dq = torch.empty(q.shape, dtype=F64)
    dk = torch.zeros(k.shape, dtype=F64)
    dv = torch.zeros(v.shape, dtype=F64)
    for r0 in range(0, n, rb):
        r1 = min(n, r0 + rb)
        p, _ = softmax_rows(scores(q[..., r0:r1, :], k, scale, causal, r0, window))
        do_b = do[..., r0:r1, :]
        dv += torch.matmul(p.transpose(-1, -2), do_b)
        dp = torch.matmul(do_b, v.transpose(-1, -2))
        ds = p * (dp - (p * dp).sum(dim=-1, keepdim=True))
        dq[..., r0:r1, :] = scale * torch.matmul(ds, k)
        dk += scale * torch.matmul(ds.transpose(-1, -2), q[..., r0:r1, :])
    return dq, dk, dv


def delta(o, do) -> torch.Tensor:
    """Per-row term D_i = rowsum(dO o O) that the recompute backward precomputes."""
    return (as_f64(do) * as_f64(o)).sum(dim=-1)


def forward_rows(q, k, v, causal: bool, scale: float, rows) -> tuple:
    """O and L for the listed query rows only (every row from its full score row).

    Used at sizes where the whole [S, S] matrix does not fit: each sampled row
    is still exactly the definition above.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    rows = torch.as_tensor(rows, dtype=torch.long)
    s = scale * torch.matmul(q[..., rows, :], k.transpose(-1, -2))
    if causal:
        kj = torch.arange(k.shape[-2]).view(1, -1)
        s = s.masked_fill(kj > rows.view(-1, 1), float("-inf"))
    p, lse = softmax_rows(s)
    return torch.matmul(p, v), lse
