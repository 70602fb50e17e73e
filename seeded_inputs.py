"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws random numbers and casts them; it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle may use it.

Recipe: every tensor is drawn on the CPU as float32 from its own
``torch.Generator`` (Q from ``seed``, K from ``seed + 1``, V from ``seed + 2``,
dO from ``seed + 3``), multiplied by its standard deviation, then rounded to
the compute dtype.  The oracle upcasts exactly these rounded values to fp64,
so both sides see bit-identical inputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def randn(shape, seed: int, dtype: torch.dtype, std: float = 1.0) -> torch.Tensor:
    """i.i.d. N(0, std^2) on the CPU, drawn in fp32 and rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes [B, H, S, D], dtype, mask and input law."""

    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str = "fp16"
    causal: bool = False
    qk_std: float = 1.0
    backward: bool = False
    seed: int = 0
    H_kv: int | None = None  # K/V heads (grouped-query attention); None = H
    window: tuple | None = None  # (left, right) band; negative side = unlimited; None = no band

    @property
    def kv_heads(self) -> int:
        return self.H if self.H_kv is None else self.H_kv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def describe(self) -> str:
        mask = "causal" if self.causal else "non-causal"
        kv = "" if self.kv_heads == self.H else f" H_kv{self.kv_heads}"
        win = "" if self.window is None else f" window{tuple(self.window)}"
        return f"B{self.B} H{self.H}{kv} S{self.S} D{self.D} {self.dtype} {mask}{win}"


def make_inputs(w: Workload, with_dout: bool | None = None) -> dict:
    """CPU tensors q, k, v (and do) for workload ``w`` per the module recipe.

    K and V have ``w.kv_heads`` heads; Q and dO have ``w.H``.
    """
    shape = (w.B, w.H, w.S, w.D)
    kv_shape = (w.B, w.kv_heads, w.S, w.D)
    dt = w.torch_dtype
    out = {
        "q": randn(shape, w.seed, dt, w.qk_std),
        "k": randn(kv_shape, w.seed + 1, dt, w.qk_std),
        "v": randn(kv_shape, w.seed + 2, dt),
    }
    if with_dout if with_dout is not None else w.backward:
        out["do"] = randn(shape, w.seed + 3, dt)
    return out


# The five workloads the library is measured and checked on.
CONFIGS = {
    "c1": Workload("c1_noncausal_fwd_B1H1S256D64_fp16", 1, 1, 256, 64, "fp16", False),
    "c2": Workload("c2_causal_fwd_B4H16S4096D64_fp16", 4, 16, 4096, 64, "fp16", True),
    "c4": Workload("c4_noncausal_fwdbwd_B2H32S8192D128_bf16", 2, 32, 8192, 128, "bf16", False,
                   qk_std=math.sqrt(2.0), backward=True),
    "c5": Workload("c5_causal_fwd_B1H8S32768D128_fp16", 1, 8, 32768, 128, "fp16", True),
}
# Config 3: causal fwd+bwd, batch 8 with no head dimension (H = 1), bf16.
C3_D = (16, 32, 64, 128)
C3_S = (256, 1024, 4096, 8192, 16384)
for _d in C3_D:
    for _s in C3_S:
        CONFIGS[f"c3_d{_d}_s{_s}"] = Workload(
            f"c3_causal_fwdbwd_B8H1S{_s}D{_d}_bf16", 8, 1, _s, _d, "bf16", True, backward=True)

# The leaderboard shape of "CS336 Assignment 2" §6 (causal forward + backward
# at 16 heads, head dimension 64, sequence length 16384, bf16), batch 1.
CONFIGS["leaderboard"] = Workload("leaderboard_causal_fwdbwd_B1H16S16384D64_bf16", 1, 16, 16384, 64, "bf16", True,
                                  backward=True)

# Grouped-query attention: the forward+backward of the causal B4 H16 S4096 D64
# fp16 shape with 8 query heads per K/V head (H_kv = 2), and multi-query
# attention (H_kv = 1) on the same shape.
CONFIGS["gqa"] = Workload("gqa_causal_fwdbwd_B4H16Hkv2S4096D64_fp16", 4, 16, 4096, 64, "fp16", True,
                          backward=True, H_kv=2)
CONFIGS["mqa"] = Workload("mqa_causal_fwdbwd_B4H16Hkv1S4096D64_fp16", 4, 16, 4096, 64, "fp16", True,
                          backward=True, H_kv=1)


@dataclass(frozen=True)
class PackedWorkload:
    """A packed variable-length batch: samples of the given lengths back to back,
    tensors [T, H, D] (K, V: [T, H_kv, D]), int32 cu_seqlens [batch + 1]."""

    name: str
    lengths: tuple
    H: int
    D: int
    dtype: str = "fp16"
    causal: bool = True
    seed: int = 0
    H_kv: int | None = None

    @property
    def kv_heads(self) -> int:
        return self.H if self.H_kv is None else self.H_kv

    @property
    def total(self) -> int:
        return sum(self.lengths)

    @property
    def batch(self) -> int:
        return len(self.lengths)

    @property
    def max_seqlen(self) -> int:
        return max(self.lengths) if self.lengths else 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def cu_seqlens(self) -> torch.Tensor:
        cu = [0]
        for n in self.lengths:
            cu.append(cu[-1] + int(n))
        return torch.tensor(cu, dtype=torch.int32)

    def describe(self) -> str:
        mask = "causal" if self.causal else "non-causal"
        kv = "" if self.kv_heads == self.H else f" H_kv{self.kv_heads}"
        return (f"packed {self.batch} samples ({self.total} tokens, max {self.max_seqlen}) H{self.H}{kv} "
                f"D{self.D} {self.dtype} {mask}")


def make_packed_inputs(w: PackedWorkload) -> dict:
    """CPU tensors q, k, v, do [T, heads, D] and cu_seqlens for ``w`` (same recipe as make_inputs)."""
    dt = w.torch_dtype
    T = w.total
    return {
        "q": randn((T, w.H, w.D), w.seed, dt),
        "k": randn((T, w.kv_heads, w.D), w.seed + 1, dt),
        "v": randn((T, w.kv_heads, w.D), w.seed + 2, dt),
        "do": randn((T, w.H, w.D), w.seed + 3, dt),
        "cu_seqlens": w.cu_seqlens(),
    }


# A packed batch with the token count of the causal B4 H16 S4096 D64 workload
# (16384 tokens) split into ten samples of mixed, mostly ragged lengths.
VARLEN_LENGTHS = (4000, 3100, 2048, 1999, 1536, 1100, 1024, 700, 577, 300)
PACKED_CONFIGS = {
    "varlen": PackedWorkload("varlen_causal_fwdbwd_T16384_10seq_H16D64_fp16", VARLEN_LENGTHS, 16, 64, "fp16", True),
}

# Sliding window: c2's shape and mask with a local band of 1024 keys to the
# left of each query (the page's window_size=(left, 0) example form).
CONFIGS["window"] = Workload("window_causal_fwdbwd_B4H16S4096D64_fp16_left1024", 4, 16, 4096, 64, "fp16", True,
                             backward=True, window=(1024, 0))

# Split-KV: one long causal head, where the query tiles alone (32 CTAs of 512
# rows) cannot fill the GPU.
CONFIGS["splitkv"] = Workload("splitkv_causal_fwdbwd_B1H1S16384D64_fp16", 1, 1, 16384, 64, "fp16", True,
                              backward=True)
