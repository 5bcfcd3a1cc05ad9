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


# ------------------------------------------------------------------ block-scaled (MXFP8) inputs
#
# The MXFP8 workloads of the block-scaled GEMM (scaled_mm): the shapes of the
# QKV projection and of the decode projection above, plus a medium square one,
# the shape classes whose MXFP8 results "TorchInductor ganha suporte a GEMMs de
# alta performance com CuteDSL" reports. Elements are drawn as N(0,1) (A) and
# N(0,1) (B), cast to E4M3 by PyTorch's round-to-nearest-even conversion
# (clamped to the format's largest finite value first); the E8M0 block scales
# are drawn uniformly from 2^-3..2^3 for A and 2^-10..2^-6 for B (weights near
# N(0, 0.02)). The integer variant draws elements from {-4..4} and scales from
# {2^-1, 2^0, 2^1}, so that every partial sum is exact in fp32.

@dataclasses.dataclass(frozen=True)
class MxConfig:
    name: str
    M: int
    N: int
    K: int
    seed: int
    description: str

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


MX_CONFIGS = {
    "mx_qkv": MxConfig("mx_qkv", 8192, 6144, 4096, 12, "MXFP8 QKV projection 8192x6144x4096, E4M3, bf16 output"),
    "mx_medium": MxConfig("mx_medium", 2048, 4096, 4096, 13, "MXFP8 medium GEMM 2048x4096x4096, E4M3, bf16 output"),
    "mx_decode": MxConfig("mx_decode", 16, 28672, 4096, 14,
                          "MXFP8 decode projection 16x28672x4096, E4M3, bf16 output"),
}

_FP8_DTYPES = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}
_FP8_MAX = {0: 448.0, 1: 57344.0}


def _fp8_codes(x: torch.Tensor, fmt: int) -> torch.Tensor:
    x = x.clamp(-_FP8_MAX[fmt], _FP8_MAX[fmt])
    return x.to(_FP8_DTYPES[fmt]).view(torch.uint8)


def make_mx_inputs(M: int, N: int, K: int, seed: int, integer: bool = False, fmt_a: int = 0, fmt_b: int = 0,
                   lda: int | None = None, ldb: int | None = None):
    """Seeded MXFP8 inputs as uint8 CPU tensors: A [M, K] and Bt [N, K] element
    codes (B transposed), SA [M, K/32] and SB [N, K/32] E8M0 scale codes, all
    row-major; lda / ldb > K give padded rows whose padding holds 0xFF."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if integer:
        a = torch.randint(-4, 5, (M, K), generator=gen).to(torch.float32)
        b = torch.randint(-4, 5, (N, K), generator=gen).to(torch.float32)
        sa = torch.randint(126, 129, (M, K // 32), generator=gen).to(torch.uint8)
        sb = torch.randint(126, 129, (N, K // 32), generator=gen).to(torch.uint8)
    else:
        a = torch.randn((M, K), generator=gen)
        b = torch.randn((N, K), generator=gen)
        sa = torch.randint(124, 131, (M, K // 32), generator=gen).to(torch.uint8)
        sb = torch.randint(117, 122, (N, K // 32), generator=gen).to(torch.uint8)
    A = _fp8_codes(a, fmt_a)
    Bt = _fp8_codes(b, fmt_b)

    def padded(x, ld):
        if ld is None or ld == x.shape[1]:
            return x
        base = torch.full((x.shape[0], ld), 0xFF, dtype=torch.uint8)
        base[:, :x.shape[1]] = x
        return base[:, :x.shape[1]]

    return padded(A, lda), sa, padded(Bt, ldb), sb


def mx_blocked_scales(S, pad: int = 127) -> "np.ndarray":
    """Scale codes [R, K/block] (row-major) rearranged into the blocked layout
    gemm_run_mx and gemm_run_fp4 take: 512-byte chunks of 128 rows x 4 scale
    columns in (row block, column block) order, the scale of row r, column c of
    a chunk at byte (r % 32) * 16 + (r / 32) * 4 + c. Padding rows and columns
    hold `pad` (127, a scale of 1 in E8M0; 0x38 is 1 in E4M3). A permutation of
    bytes, nothing else."""
    import numpy as np
    S = np.asarray(S, dtype=np.uint8)
    R, nb = S.shape
    rbs, kc = -(-R // 128), -(-nb // 4)
    P = np.full((rbs * 128, kc * 4), pad, dtype=np.uint8)
    P[:R, :nb] = S
    return np.ascontiguousarray(P.reshape(rbs, 4, 32, kc, 4).transpose(0, 3, 2, 1, 4).reshape(-1))


# ---------------------------------------------------------------- FP4 (NVFP4, MXFP4)

FP4_NV, FP4_MX = 0, 1  # the library's TPGEMM_NVFP4 and TPGEMM_MXFP4
FP4_BLOCK = {FP4_NV: 16, FP4_MX: 32}
E4M3_ONE = 0x38  # 1.0 as an E4M3 scale code (padding of NVFP4 scale layouts)


@dataclasses.dataclass(frozen=True)
class Fp4Config:
    name: str
    fmt: int
    M: int
    N: int
    K: int
    seed: int
    description: str

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


FP4_CONFIGS = {
    "nvfp4_decode": Fp4Config("nvfp4_decode", FP4_NV, 16, 28672, 4096, 15,
                              "NVFP4 decode projection 16x28672x4096, E4M3 scales per 16, bf16 output"),
    "nvfp4_m256": Fp4Config("nvfp4_m256", FP4_NV, 256, 28672, 4096, 16,
                            "NVFP4 GEMM with 256 rows 256x28672x4096, E4M3 scales per 16, bf16 output"),
    "nvfp4_qkv": Fp4Config("nvfp4_qkv", FP4_NV, 8192, 6144, 4096, 17,
                           "NVFP4 QKV projection 8192x6144x4096, E4M3 scales per 16, bf16 output"),
    "mxfp4_qkv": Fp4Config("mxfp4_qkv", FP4_MX, 8192, 6144, 4096, 18,
                           "MXFP4 QKV projection 8192x6144x4096, E8M0 scales per 32, bf16 output"),
}

# magnitudes of the eight E2M1 codes 0..7 (the sign is bit 3)
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_codes(x: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code of each value (magnitudes clamped to 6; ties go to the
    smaller magnitude), as uint8 codes 0..15."""
    grid = torch.tensor(_E2M1_MAG, dtype=torch.float32)
    mids = (grid[1:] + grid[:-1]) / 2
    mag = torch.bucketize(x.abs().clamp(max=6.0), mids, right=False).to(torch.uint8)
    sign = ((x < 0) & (mag != 0)).to(torch.uint8) << 3
    return mag | sign


def _pack_fp4(codes: torch.Tensor) -> torch.Tensor:
    """[R, K] codes 0..15 -> [R, K/2] bytes, the even element in the low nibble."""
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()


def make_fp4_inputs(M: int, N: int, K: int, seed: int, fmt: int = FP4_NV, integer: bool = False,
                    lda: int | None = None, ldb: int | None = None):
    """Seeded FP4 inputs as uint8 CPU tensors: A [M, K/2] and Bt [N, K/2]
    packed E2M1 codes (B transposed; the even element in the low nibble), SA
    [M, K/block] and SB [N, K/block] scale codes (E4M3 for NVFP4, E8M0 for
    MXFP4), row-major; lda / ldb (bytes) > K/2 give padded rows whose padding
    holds 0xFF.

    integer=True: uniformly random codes (all sixteen, -0 included) with scales
    of 1/2, 1 and 2, so every partial sum of the product is exact in fp32 (for
    K up to 7281). Otherwise N(0,1) data quantised the usual way: per block,
    the scale is the block's largest magnitude over 6 (NVFP4: rounded to
    E4M3; MXFP4: the power of two at or above it) and each element the nearest
    E2M1 value of data / scale."""
    block = FP4_BLOCK[fmt]
    if K % block:
        raise ValueError(f"K must be a multiple of {block}")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)

    def one(rows):
        if integer:
            codes = torch.randint(0, 16, (rows, K), generator=gen).to(torch.uint8)
            if fmt == FP4_NV:
                s = torch.tensor([0x30, 0x38, 0x40], dtype=torch.uint8)[
                    torch.randint(0, 3, (rows, K // block), generator=gen)]
            else:
                s = torch.randint(126, 129, (rows, K // block), generator=gen).to(torch.uint8)
            return _pack_fp4(codes), s
        x = torch.randn((rows, K), generator=gen)
        amax = x.view(rows, K // block, block).abs().amax(dim=2).clamp(min=1e-30)
        if fmt == FP4_NV:
            sc = (amax / 6.0).clamp(min=2.0 ** -9).to(torch.float8_e4m3fn)  # never a zero scale
            s = sc.view(torch.uint8).clone()
            scale = sc.to(torch.float32)
        else:
            e = torch.ceil(torch.log2(amax / 6.0)).clamp(-127, 127)
            s = (e + 127).to(torch.uint8)
            scale = torch.exp2(e)
        q = x / scale.repeat_interleave(block, dim=1)
        return _pack_fp4(_e2m1_codes(q)), s

    A, SA = one(M)
    Bt, SB = one(N)

    def padded(x, ld):
        if ld is None or ld == x.shape[1]:
            return x
        base = torch.full((x.shape[0], ld), 0xFF, dtype=torch.uint8)
        base[:, :x.shape[1]] = x
        return base[:, :x.shape[1]]

    return padded(A, lda), SA, padded(Bt, ldb), SB
