"""CPU oracle for D = alpha*A*B + beta*C (fp64 accumulation, one final rounding).

TEST INFRASTRUCTURE ONLY. The test suite, the package smoke check and the
benchmark's CPU-baseline leg may load this module; the product path never does.
It shares no code with the CUDA library: the arithmetic lives in ``oracle.c``
(plain C, fp64), and this file only marshals arguments through ctypes.

The definition it follows, and every reading of the pages it rests on, is in
the header comment of ``oracle.c``. Parity of each function here is pinned by
``tests/test_oracle_pins.py`` against closed forms, brute force and the IEEE-754
rounding definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

OUT_BF16 = 0
OUT_F32 = 1
ACT_NONE = 0
ACT_RELU = 1
ACT_SIGMOID = 2
ACT_TANH = 3
FP8_E4M3 = 0
FP8_E5M2 = 1
SCALE_E8M0 = 2
FP4_E2M1 = 3
SCALE_E4M3 = 0
MX_BLOCK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "oracle_mx.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, no contraction, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or any(os.path.getmtime(_LIB) < os.path.getmtime(f) for f in _SRCS)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                   "-pthread", "-std=c11", "-Wall", "-o", tmp, *_SRCS, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_rows.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, dbl, dbl,
                                         ctypes.c_int, vp, i64, vp, i64, vp, i64, ctypes.c_int]
        lib.oracle_gemm_rows_epilogue.restype = ctypes.c_int
        lib.oracle_gemm_rows_epilogue.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, dbl, dbl,
                                                  ctypes.c_int, vp, i64, vp, i64, vp, i64, ctypes.c_int,
                                                  vp, ctypes.c_int, ctypes.c_int, vp, i64]
        lib.oracle_act.restype = dbl
        lib.oracle_act.argtypes = [ctypes.c_int, dbl]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [dbl]
        lib.oracle_round_f32.restype = ctypes.c_float
        lib.oracle_round_f32.argtypes = [dbl]
        lib.oracle_round_bf16_from_f32_bits.restype = None
        lib.oracle_round_bf16_from_f32_bits.argtypes = [vp, vp, i64]
        lib.oracle_round_bf16_array.restype = None
        lib.oracle_round_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_mx_gemm_rows.restype = ctypes.c_int
        lib.oracle_mx_gemm_rows.argtypes = [i64, i64, i64, vp, i64, ctypes.c_int, vp, i64, vp, i64, ctypes.c_int,
                                            vp, i64, vp, i64, dbl, dbl, ctypes.c_int, vp, i64, vp, i64, vp, i64,
                                            ctypes.c_int]
        lib.oracle_bs_gemm_rows.restype = ctypes.c_int
        lib.oracle_bs_gemm_rows.argtypes = [i64, i64, i64, vp, i64, ctypes.c_int, vp, i64, vp, i64, ctypes.c_int,
                                            vp, i64, ctypes.c_int, ctypes.c_int, vp, i64, dbl, dbl, ctypes.c_int, vp,
                                            i64, vp, i64, vp, i64, ctypes.c_int]
        lib.oracle_decode_mx_array.restype = None
        lib.oracle_decode_mx_array.argtypes = [ctypes.c_int, vp, vp, i64]
        _lib = lib
    return _lib


def library_path() -> str:
    _load()
    return _LIB


def _bits_view(t: torch.Tensor, name: str):
    """(pointer, row stride in elements) of a 2-D CPU tensor with unit column stride."""
    if t.device.type != "cpu" or t.dim() != 2:
        raise ValueError(f"{name}: need a 2-D CPU tensor")
    if t.numel() and t.stride(1) != 1:
        raise ValueError(f"{name}: need unit column stride")
    return t.data_ptr(), (t.stride(0) if t.numel() else max(t.shape[1], 1))


def gemm_rows(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None, alpha: float,
              beta: float, out_dtype: int, rows=None, want_pre: bool = False,
              nthreads: int | None = None):
    """Rows `rows` (default: all) of D = alpha*A*B + beta*C, computed on the CPU.

    A [M,K] and B [K,N] are bf16 CPU tensors (row-major, any row stride); C is
    [M,N] of the output dtype or None when beta == 0. alpha and beta are taken
    as fp32 values (the boundary's parameter type) and widened to fp64.
    Returns (D, pre): D is numpy uint16 (bf16 bits) or float32, shape
    [len(rows), N]; pre is the fp64 value before rounding (or None).
    """
    lib = _load()
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    alpha = float(np.float32(alpha))
    beta = float(np.float32(beta))
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    a_ptr, lda = _bits_view(A, "A")
    b_ptr, ldb = _bits_view(B, "B")
    c_ptr, ldc = 0, max(N, 1)
    if beta != 0.0:
        want = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
        if C is None or C.dtype != want or tuple(C.shape) != (M, N):
            raise ValueError("C must be [M,N] of the output dtype when beta != 0")
        c_ptr, ldc = _bits_view(C, "C")
    out_np = np.uint16 if out_dtype == OUT_BF16 else np.float32
    D = np.zeros((len(rows), N), dtype=out_np)
    pre = np.zeros((len(rows), N), dtype=np.float64) if want_pre else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_gemm_rows(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, alpha, beta,
                              out_dtype, rows.ctypes.data, len(rows), D.ctypes.data, max(N, 1),
                              pre.ctypes.data if pre is not None else None, max(N, 1),
                              int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_gemm_rows rejected its arguments")
    return D, pre


def gemm_rows_epilogue(A, B, C, alpha, beta, out_dtype, bias=None, act=ACT_NONE, aux=None, rows=None,
                       want_pre=False, nthreads=None):
    """gemm_rows followed by the fused epilogue: v = alpha*acc + beta*C + bias[n];
    v = act(v); v = v * aux[m, n]; one rounding. bias is a 1-D bf16/fp32 CPU
    tensor of N values; aux an [M, N] CPU tensor of the output dtype."""
    lib = _load()
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bf16")
    M, K = A.shape
    N = B.shape[1]
    alpha = float(np.float32(alpha))
    beta = float(np.float32(beta))
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    a_ptr, lda = _bits_view(A, "A")
    b_ptr, ldb = _bits_view(B, "B")
    c_ptr, ldc = 0, max(N, 1)
    if beta != 0.0:
        c_ptr, ldc = _bits_view(C, "C")
    bias_ptr, bias_dt = None, OUT_F32
    if bias is not None:
        bias = bias.contiguous()
        if bias.numel() != N:
            raise ValueError("bias must have N elements")
        bias_ptr = bias.data_ptr()
        bias_dt = OUT_BF16 if bias.dtype == torch.bfloat16 else OUT_F32
    aux_ptr, ldaux = None, max(N, 1)
    if aux is not None:
        aux_ptr, ldaux = _bits_view(aux, "aux")
    out_np = np.uint16 if out_dtype == OUT_BF16 else np.float32
    D = np.zeros((len(rows), N), dtype=out_np)
    pre = np.zeros((len(rows), N), dtype=np.float64) if want_pre else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_gemm_rows_epilogue(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, alpha, beta,
                                       out_dtype, rows.ctypes.data, len(rows), D.ctypes.data, max(N, 1),
                                       pre.ctypes.data if pre is not None else None, max(N, 1),
                                       int(nthreads), bias_ptr, bias_dt, int(act), aux_ptr, ldaux)
    if rc != 0:
        raise RuntimeError("oracle_gemm_rows_epilogue rejected its arguments")
    return D, pre


def activation(act: int, x: float) -> float:
    return float(_load().oracle_act(int(act), float(x)))


def round_bf16(x: float) -> int:
    """fp64 -> bf16 bits, round to nearest even, one rounding."""
    return int(_load().oracle_round_bf16(float(x)))


def round_bf16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def round_bf16_from_f32_bits(u: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u, dtype=np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    _load().oracle_round_bf16_from_f32_bits(u.ctypes.data, out.ctypes.data, u.size)
    return out


def round_f32(x: float) -> float:
    return float(_load().oracle_round_f32(float(x)))


# ------------------------------------------------------------------ block-scaled (MX) GEMM

def decode_mx(codes, fmt: int) -> np.ndarray:
    """Values of 8-bit codes: fmt FP8_E4M3, FP8_E5M2 or SCALE_E8M0 (see oracle_mx.c)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_mx_array(int(fmt), c.ctypes.data, out.ctypes.data, c.size)
    return out


def _u8_view(t, name):
    a = t.numpy() if isinstance(t, torch.Tensor) else t
    if a.dtype != np.uint8 or a.ndim != 2:
        raise ValueError(f"{name}: need a 2-D uint8 array")
    if a.size and a.strides[1] != 1:
        raise ValueError(f"{name}: need unit column stride")
    return a, a.ctypes.data, (a.strides[0] if a.size else max(a.shape[1], 1))


def mx_gemm_rows(A, SA, Bt, SB, C, alpha: float, beta: float, out_dtype: int, fmt_a: int = FP8_E4M3,
                 fmt_b: int = FP8_E4M3, rows=None, want_pre: bool = False, nthreads: int | None = None):
    """Rows `rows` (default: all) of the block-scaled GEMM
        D = alpha * sum_b SA[:, b] SB[:, b]^T * (A_b Bt_b^T) + beta * C
    on the CPU. A [M, K] and Bt [N, K] hold FP8 codes (uint8, row-major, any
    row stride), SA [M, K/32] and SB [N, K/32] E8M0 scale codes; C is [M, N] of
    the output dtype or None when beta == 0. Returns (D, pre) like gemm_rows."""
    lib = _load()
    A, a_ptr, lda = _u8_view(A, "A")
    SA, sa_ptr, ldsa = _u8_view(SA, "SA")
    Bt, b_ptr, ldb = _u8_view(Bt, "Bt")
    SB, sb_ptr, ldsb = _u8_view(SB, "SB")
    M, K = A.shape
    N = Bt.shape[0]
    if Bt.shape[1] != K or K % MX_BLOCK or SA.shape != (M, K // MX_BLOCK) or SB.shape != (N, K // MX_BLOCK):
        raise ValueError("shapes of A, SA, Bt, SB do not agree")
    alpha = float(np.float32(alpha))
    beta = float(np.float32(beta))
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c_ptr, ldc = 0, max(N, 1)
    if beta != 0.0:
        want = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
        if C is None or C.dtype != want or tuple(C.shape) != (M, N):
            raise ValueError("C must be [M,N] of the output dtype when beta != 0")
        c_ptr, ldc = _bits_view(C, "C")
    out_np = np.uint16 if out_dtype == OUT_BF16 else np.float32
    D = np.zeros((len(rows), N), dtype=out_np)
    pre = np.zeros((len(rows), N), dtype=np.float64) if want_pre else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_mx_gemm_rows(M, N, K, a_ptr, lda, int(fmt_a), sa_ptr, ldsa, b_ptr, ldb, int(fmt_b), sb_ptr,
                                 ldsb, c_ptr, ldc, alpha, beta, out_dtype, rows.ctypes.data, len(rows),
                                 D.ctypes.data, max(N, 1), pre.ctypes.data if pre is not None else None,
                                 max(N, 1), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_mx_gemm_rows rejected its arguments")
    return D, pre


def bs_gemm_rows(A, SA, Bt, SB, C, alpha: float, beta: float, out_dtype: int, fmt_a: int, fmt_b: int,
                 scale_fmt: int, block: int, rows=None, want_pre: bool = False, nthreads: int | None = None):
    """The block-scaled GEMM in general form (see oracle_mx.c): element formats
    FP8_E4M3, FP8_E5M2 or FP4_E2M1 (two per byte, the even element in the low
    four bits, so a row of K elements is K/2 bytes), scale format SCALE_E8M0 or
    SCALE_E4M3, `block` (16 or 32) elements per scale. A [M, K or K/2] and Bt
    [N, K or K/2] are uint8 codes, SA [M, K/block] and SB [N, K/block] scale
    codes. Returns (D, pre) like gemm_rows."""
    lib = _load()
    A, a_ptr, lda = _u8_view(A, "A")
    SA, sa_ptr, ldsa = _u8_view(SA, "SA")
    Bt, b_ptr, ldb = _u8_view(Bt, "Bt")
    SB, sb_ptr, ldsb = _u8_view(SB, "SB")
    M = A.shape[0]
    N = Bt.shape[0]
    K = A.shape[1] * (2 if fmt_a == FP4_E2M1 else 1)
    kb_ = Bt.shape[1] * (2 if fmt_b == FP4_E2M1 else 1)
    if kb_ != K or K % block or SA.shape != (M, K // block) or SB.shape != (N, K // block):
        raise ValueError("shapes of A, SA, Bt, SB do not agree")
    alpha = float(np.float32(alpha))
    beta = float(np.float32(beta))
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c_ptr, ldc = 0, max(N, 1)
    if beta != 0.0:
        want = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
        if C is None or C.dtype != want or tuple(C.shape) != (M, N):
            raise ValueError("C must be [M,N] of the output dtype when beta != 0")
        c_ptr, ldc = _bits_view(C, "C")
    out_np = np.uint16 if out_dtype == OUT_BF16 else np.float32
    D = np.zeros((len(rows), N), dtype=out_np)
    pre = np.zeros((len(rows), N), dtype=np.float64) if want_pre else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_bs_gemm_rows(M, N, K, a_ptr, lda, int(fmt_a), sa_ptr, ldsa, b_ptr, ldb, int(fmt_b), sb_ptr,
                                 ldsb, int(scale_fmt), int(block), c_ptr, ldc, alpha, beta, out_dtype,
                                 rows.ctypes.data, len(rows), D.ctypes.data, max(N, 1),
                                 pre.ctypes.data if pre is not None else None, max(N, 1), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_bs_gemm_rows rejected its arguments")
    return D, pre
