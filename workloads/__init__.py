"""Seeded synthetic GEMM inputs, shared by the tests, the smoke check and the
benchmark.  This module draws random numbers and casts them; it holds none of
the product's arithmetic and imports neither the oracle nor the CUDA library.

Recipe (the same for every workload): one CPU ``torch.Generator`` seeded with
the workload's seed; A is drawn first, then B, in float32; uniform[-1, 1) is
``2 * rand - 1``; N(0, s) is ``s * randn``; the 8192^3 workload scales both
operands by 1/sqrt(K) in float32; the values are then rounded to fp16/bf16
with round-to-nearest-even (``Tensor.to``).  Padding beyond the logical
columns of a padded leading dimension is filled with NaN so that a kernel that
reads it poisons its output.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    dtype: str          # "f16" or "bf16"
    dist_a: str         # "uniform", "normal"
    dist_b: str
    scale_a: float
    scale_b: float
    seed: int
    note: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes_alg(self) -> int:
        """One read of A and B (2 B/elem) and one write of C (4 B/elem)."""
        return 2 * (self.M * self.K + self.K * self.N) + 4 * self.M * self.N


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("gemm256_f16", 256, 256, 256, "f16", "uniform", "uniform", 1.0, 1.0, 0,
                 "256^3 fp16, uniform[-1,1)"),
        Workload("ragged1023x1000x1029_f16", 1023, 1000, 1029, "f16", "uniform", "uniform", 1.0,
                 1.0, 1, "ragged M=1023 K=1000 N=1029 fp16, uniform[-1,1)"),
        Workload("square4096_bf16", 4096, 4096, 4096, "bf16", "normal", "normal", 1.0, 1.0, 2,
                 "4096^3 bf16, N(0,1)"),
        Workload("square8192_bf16", 8192, 8192, 8192, "bf16", "normal", "normal",
                 1.0 / math.sqrt(8192), 1.0 / math.sqrt(8192), 3, "8192^3 bf16, N(0,1)/sqrt(K)"),
        Workload("skinny16x4096x14336_bf16", 16, 4096, 14336, "bf16", "normal", "normal", 1.0,
                 0.02, 4, "M=16 K=4096 N=14336 bf16, A N(0,1), B N(0,0.02)"),
    ]
}


def _draw(g: torch.Generator, rows: int, cols: int, dist: str, scale: float) -> torch.Tensor:
    if dist == "uniform":
        x = torch.rand(rows, cols, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    elif dist == "int4":   # integers in [-4, 4]: products and partial sums stay exact in fp32
        x = torch.randint(-4, 5, (rows, cols), generator=g).to(torch.float32)
    else:
        raise ValueError(dist)
    if scale != 1.0:
        x = x * torch.tensor(scale, dtype=torch.float32)
    return x


def _place(x: torch.Tensor, ld: int | None, dtype: torch.dtype) -> torch.Tensor:
    rows, cols = x.shape
    if ld is None or ld == cols:
        return x.to(dtype).contiguous()
    if ld < cols:
        raise ValueError(f"leading dimension {ld} < {cols}")
    out = torch.full((rows, ld), float("nan"), dtype=dtype)
    out[:, :cols] = x.to(dtype)
    return out


def make_inputs(w: Workload | str, *, lda: int | None = None, ldb: int | None = None
                ) -> tuple[torch.Tensor, torch.Tensor]:
    """CPU tensors (A stored as (M, lda), B stored as (K, ldb)) of the workload's dtype."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator().manual_seed(w.seed)
    a = _draw(g, w.M, w.K, w.dist_a, w.scale_a)
    b = _draw(g, w.K, w.N, w.dist_b, w.scale_b)
    return _place(a, lda, w.torch_dtype), _place(b, ldb, w.torch_dtype)


def custom(M: int, K: int, N: int, dtype: str, seed: int, dist: str = "uniform",
           scale: float = 1.0, lda: int | None = None, ldb: int | None = None
           ) -> tuple[torch.Tensor, torch.Tensor]:
    """Ad-hoc shape with the same recipe (used by the ragged sweeps and edge cases)."""
    w = Workload(f"custom{M}x{K}x{N}", M, K, N, dtype, dist, dist, scale, scale, seed)
    return make_inputs(w, lda=lda, ldb=ldb)


# ---------------------------------------------------------------- row-wise softmax
#
# Recipe: one CPU ``torch.Generator`` seeded with the workload's seed draws the
# M x N float32 matrix with ``torch.randn`` (the distribution of the softmax
# chapter's demo input, whose scores stand in for QK^T / sqrt(d) rows), times
# ``scale``.  A padded leading dimension is filled with NaN beyond column N.

@dataclasses.dataclass(frozen=True)
class RowsWorkload:
    name: str
    M: int
    N: int
    scale: float
    seed: int
    note: str = ""

    @property
    def bytes_alg(self) -> int:
        """One read of X and one write of Y, 4 B per element each."""
        return 8 * self.M * self.N


SOFTMAX_WORKLOADS: dict[str, RowsWorkload] = {
    w.name: w
    for w in [
        RowsWorkload("softmax128x1000_f32", 128, 1000, 1.0, 20,
                     "the softmax chapter's demo shape: 128 rows of 1000, N(0,1)"),
        RowsWorkload("softmax65536x1000_f32", 65536, 1000, 1.0, 21,
                     "65536 rows of the demo's length: 262 MB in, 262 MB out (> L2)"),
        RowsWorkload("softmax4096x32768_f32", 4096, 32768, 1.0, 22,
                     "long rows (tens of thousands of elements): 537 MB in, 537 MB out"),
    ]
}


def make_rows(w: RowsWorkload | str, *, ld: int | None = None) -> torch.Tensor:
    """CPU float32 tensor stored as (M, ld) with the workload's values in the first N columns."""
    if isinstance(w, str):
        w = SOFTMAX_WORKLOADS[w]
    g = torch.Generator().manual_seed(w.seed)
    x = torch.randn(w.M, w.N, generator=g, dtype=torch.float32)
    if w.scale != 1.0:
        x = x * torch.tensor(w.scale, dtype=torch.float32)
    return _place(x, ld, torch.float32)


def custom_rows(M: int, N: int, seed: int, scale: float = 1.0, ld: int | None = None) -> torch.Tensor:
    """Ad-hoc softmax input with the same recipe."""
    return make_rows(RowsWorkload(f"rows{M}x{N}", M, N, scale, seed), ld=ld)


# ---------------------------------------------------------------- attention forward
#
# Recipe: one CPU ``torch.Generator`` per workload draws Q, then K, then V, each
# [BH, seq, d] float32 ``torch.randn`` (unit-variance rows, so Q K^T / sqrt(d)
# has unit-variance scores), rounded to fp16/bf16 to nearest-even.  BH
# independent heads (e.g. batch 2 x 8 heads for BH = 16) share the layout
# [BH, seq, d], row-major, d contiguous.

@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    name: str
    BH: int
    seq: int
    d: int
    dtype: str
    causal: bool
    seed: int
    note: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    @property
    def flops(self) -> int:
        """2 flops per multiply-add of Q K^T and of P V, over the (query, key)
        pairs the mask keeps: seq^2 pairs, or seq (seq + 1) / 2 when causal."""
        pairs = self.seq * (self.seq + 1) // 2 if self.causal else self.seq * self.seq
        return 4 * self.BH * pairs * self.d


ATTN_WORKLOADS: dict[str, AttnWorkload] = {
    w.name: w
    for w in [
        AttnWorkload("attn_bh2_s256_d64_f16_causal", 2, 256, 64, "f16", True, 30,
                     "small causal case: 2 heads of 256 x 64"),
        AttnWorkload("attn_bh2_s1000_d64_bf16", 2, 1000, 64, "bf16", False, 31,
                     "ragged sequence (1000 = 7 x 128 + 104), no mask"),
        AttnWorkload("attn_bh16_s8192_d64_bf16_causal", 16, 8192, 64, "bf16", True, 32,
                     "the section's sequence length 8192 and head dimension 64, causal, 16 heads"),
        AttnWorkload("attn_bh16_s8192_d64_bf16", 16, 8192, 64, "bf16", False, 33,
                     "the same without the mask"),
        AttnWorkload("attn_bh16_s8192_d128_bf16_causal", 16, 8192, 128, "bf16", True, 34,
                     "head dimension 128, causal, 16 heads"),
    ]
}


def make_qkv(w: AttnWorkload | str) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """CPU tensors Q, K, V of shape [BH, seq, d] in the workload's dtype."""
    if isinstance(w, str):
        w = ATTN_WORKLOADS[w]
    g = torch.Generator().manual_seed(w.seed)
    out = []
    for _ in range(3):
        out.append(torch.randn(w.BH, w.seq, w.d, generator=g, dtype=torch.float32).to(w.torch_dtype))
    return out[0], out[1], out[2]


def custom_qkv(BH: int, seq: int, d: int, dtype: str, seed: int, causal: bool = False):
    """Ad-hoc attention input with the same recipe."""
    return make_qkv(AttnWorkload(f"attn{BH}x{seq}x{d}", BH, seq, d, dtype, causal, seed))
