"""Seeded synthetic workloads for the bf16 GEMM D = alpha*A*B + beta*C.

This module only makes inputs: shapes, seeds, value distributions, row
strides. It holds none of the GEMM's arithmetic, so the CUDA path and the CPU
oracle can both be fed from it without sharing any computation.

The shapes stand in for the transformer layers whose GEMMs "TorchInductor ganha
suporte a GEMMs de alta performance com CuteDSL" says dominate a forward pass
(attention projections, fully-connected layers) and for the decode shapes with
M between 8 and 64 that the same page's BF16 results paragraph singles out. No
dataset or trained weight is used: activations are N(0,1), weights N(0,0.02),
the tiny case U[-1,1], and the integer variant draws from {-4..4}.

Generation recipe (fixed, so a seed reproduces the bytes): a CPU
``torch.Generator`` seeded with the config's seed draws A, then B, then C, in
fp32, each then rounded to bf16 by PyTorch's round-to-nearest-even cast. A C
that is not bf16 (the fp32-output variants) is drawn in fp32 and kept.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class GemmConfig:
    name: str
    M: int
    N: int
    K: int
    seed: int
    a_dist: tuple  # ("uniform", lo, hi) | ("normal", std) | ("int", lo, hi)
    b_dist: tuple
    c_dist: tuple | None
    alpha: float
    beta: float
    out_dtype: str  # "bf16" | "f32"
    description: str

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


CONFIGS = {
    "tiny": GemmConfig("tiny", 256, 256, 256, 0, ("uniform", -1.0, 1.0), ("uniform", -1.0, 1.0),
                       None, 1.0, 0.0, "f32", "tiny GEMM 256x256x256, U[-1,1], fp32 output"),
    "square": GemmConfig("square", 4096, 4096, 4096, 1, ("normal", 1.0), ("normal", 1.0), None,
                         1.0, 0.0, "bf16", "square GEMM 4096x4096x4096, N(0,1), bf16 output"),
    "qkv": GemmConfig("qkv", 8192, 6144, 4096, 2, ("normal", 1.0), ("normal", 0.02), None, 1.0,
                      0.0, "bf16", "GQA QKV projection, 8192 tokens, N=4096+2*1024, K=4096"),
    "mlp_down": GemmConfig("mlp_down", 8192, 4096, 14336, 3, ("normal", 1.0), ("normal", 0.02),
                           ("normal", 1.0), 1.0, 1.0, "bf16",
                           "MLP down-projection 8192x4096x14336 with residual C, beta=1"),
    "decode": GemmConfig("decode", 16, 28672, 4096, 4, ("normal", 1.0), ("normal", 0.02), None,
                         1.0, 0.0, "bf16",
                         "decode-shape fused gate+up projection, M=16 tokens, N=28672, K=4096"),
}

ORDER = ["tiny", "square", "qkv", "mlp_down", "decode"]


def _draw(shape, dist, gen, ld=None, pad_value=float("nan")):
    """Draw a [rows, cols] fp32 matrix; with ld > cols the row stride is ld and
    the padding columns hold pad_value (a sentinel no reader may use)."""
    rows, cols = shape
    kind = dist[0]
    if kind == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * (dist[2] - dist[1]) + dist[1]
    elif kind == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * dist[1]
    elif kind == "int":
        x = torch.randint(dist[1], dist[2] + 1, shape, generator=gen).to(torch.float32)
    else:
        raise ValueError(kind)
    if ld is None or ld == cols:
        return x
    full = torch.full((rows, ld), pad_value, dtype=torch.float32)
    full[:, :cols] = x
    return full[:, :cols]


def make_inputs(cfg: GemmConfig, integer: bool = False, M: int | None = None,
                N: int | None = None, K: int | None = None, lda=None, ldb=None, ldc=None,
                seed: int | None = None, c_for_beta: bool | None = None):
    """Seeded CPU inputs (A, B, C) for `cfg`, optionally with other sizes/strides.

    integer=True replaces every distribution with integers in {-4..4} (the
    bit-exact variant). C is drawn when cfg has a C distribution or
    c_for_beta is True, in the output dtype. Returns bf16 views that may have
    padded row strides (padding filled with NaN).
    """
    M = cfg.M if M is None else M
    N = cfg.N if N is None else N
    K = cfg.K if K is None else K
    gen = torch.Generator(device="cpu")
    gen.manual_seed(cfg.seed if seed is None else seed)
    ad = ("int", -4, 4) if integer else cfg.a_dist
    bd = ("int", -4, 4) if integer else cfg.b_dist
    A = _draw((M, K), ad, gen, lda)
    B = _draw((K, N), bd, gen, ldb)
    want_c = cfg.c_dist is not None if c_for_beta is None else c_for_beta
    C = None
    if want_c:
        cd = ("int", -4, 4) if integer else (cfg.c_dist or ("normal", 1.0))
        C = _draw((M, N), cd, gen, ldc)
    A = _to_bf16_keep_stride(A)
    B = _to_bf16_keep_stride(B)
    if C is not None and cfg.out_dtype == "bf16":
        C = _to_bf16_keep_stride(C)
    return A, B, C


def _to_bf16_keep_stride(x: torch.Tensor) -> torch.Tensor:
    """Round to bf16 (PyTorch's RNE cast) keeping the row stride of the base."""
    if x.stride(0) == x.shape[1] or x.numel() == 0:
        return x.contiguous().to(torch.bfloat16)
    rows, cols = x.shape
    ld = x.stride(0)
    base = torch.as_strided(x, (rows, ld), (ld, 1))
    return base.to(torch.bfloat16)[:, :cols]


def sample_rows(M: int, count: int, tile: int = 128, seed: int = 1234):
    """Deterministic row sample for full-size parity: the first and last rows of
    the first, second and last row tiles, plus seeded random rows."""
    if M <= count:
        return list(range(M))
    fixed = {0, 1, tile - 1, tile, 2 * tile - 1, M - 1, M - 2, (M - 1) // tile * tile}
    fixed = {r for r in fixed if 0 <= r < M}
    g = torch.Generator().manual_seed(seed)
    extra = torch.randperm(M, generator=g)[: max(0, count - len(fixed))].tolist()
    return sorted(fixed | set(extra))[:count] if len(fixed | set(extra)) > count else sorted(fixed | set(extra))
