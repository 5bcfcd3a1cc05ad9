"""Helpers for the GPU tests: move seeded CPU inputs to the device (keeping
their row strides), call gemm_run through the C ABI, and compare with the CPU
oracle under the stated tolerances.

Tolerances (the GEMM's own accuracy contract, written here once):
  integer inputs in {-4..4}: bit-exact (every partial sum is an integer below
  2^24, so fp32 accumulation is exact in any order and a single rounding of the
  exact value is unique);
  fp32 output: max|D-O| / max|O| <= 1e-5, and the same ratio of the matrix
  infinity norms (largest absolute row sum) <= 1e-5;
  bf16 output: |D-O| <= 2^-7 |O| + 1e-5 max|O| for every element.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from workloads import mx_blocked_scales as mx_blocked  # noqa: F401 (re-exported for the tests)

BF16_NAN = 0x7FC0
DEV = torch.device("cuda:0")


def round8(x: int) -> int:
    return (x + 7) // 8 * 8


def to_device(t: torch.Tensor | None):
    """Copy a 2-D CPU view to the GPU keeping its row stride (and padding)."""
    if t is None:
        return None
    rows, cols = t.shape
    ld = t.stride(0)
    if rows <= 1 or cols == 0 or ld == cols:
        return t.contiguous().to(DEV)
    base = torch.as_strided(t, (rows, ld), (ld, 1))
    return base.to(DEV)[:, :cols]


def alloc_out(M: int, N: int, dtype: torch.dtype, ldd: int | None = None, guard_rows: int = 2):
    """D view [M, N] inside a NaN-filled base [M + guard_rows, ldd]."""
    ldd = round8(N) if ldd is None else ldd
    base = torch.empty((M + guard_rows, ldd), dtype=dtype, device=DEV)
    if dtype == torch.bfloat16:
        base.view(torch.int16).fill_(BF16_NAN)
    else:
        base.fill_(float("nan"))
    return base[:M, :N], base


def out_code(dtype: torch.dtype) -> int:
    return tpd.OUT_F32 if dtype == torch.float32 else tpd.OUT_BF16


def ld_of(t: torch.Tensor | None, cols: int) -> int:
    if t is None:
        return max(round8(cols), 8)
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), round8(cols))


def run(h, A, B, C, alpha, beta, out_dtype, ldd=None, stream=None, D=None):
    """gemm_run through the C ABI on device copies of A, B, C. Returns (D, base)."""
    M, K = A.shape
    N = B.shape[1]
    Ad, Bd, Cd = A, B, C
    if A.device.type == "cpu":
        Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    base = None
    if D is None:
        D, base = alloc_out(M, N, out_dtype, ldd)
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run(h, M, N, K, Ad.data_ptr() if K else None, ld_of(Ad, K),
                      Bd.data_ptr() if K else None, ld_of(Bd, N),
                      Cd.data_ptr() if Cd is not None else None, ld_of(Cd, N), D.data_ptr(),
                      ld_of(D, N), float(alpha), float(beta), out_code(out_dtype), s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    st = tpd.gemm_sync_status(h, s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    return D, base


def bits(t: torch.Tensor) -> np.ndarray:
    """Exact bit patterns of a CPU/GPU tensor as numpy (uint16 for bf16)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()


def oracle_out(A, B, C, alpha, beta, out_dtype, rows=None):
    D, _ = oracle.gemm_rows(A, B, C, alpha, beta, out_code(out_dtype), rows=rows)
    return D


def as_f64(x: np.ndarray, out_dtype: torch.dtype) -> np.ndarray:
    if out_dtype == torch.bfloat16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def assert_bit_exact(got: np.ndarray, want: np.ndarray, what: str = ""):
    # +0 and -0 compare equal: the oracle's sum starts from +0, while a sum of
    # only -0 products (K = 1, a zero times a negative) is -0 under IEEE rules.
    if got.dtype == np.float32:
        eq = (got.view(np.uint32) == want.view(np.uint32)) | ((got == 0) & (want == 0))
    else:
        eq = (got == want) | (((got & 0x7FFF) == 0) & ((want & 0x7FFF) == 0))
    if not eq.all():
        idx = np.argwhere(~eq)[:5]
        raise AssertionError(f"{what}: {int((~eq).sum())} of {eq.size} elements differ; first at "
                             f"{idx.tolist()}: got {[got[tuple(i)] for i in idx]} want "
                             f"{[want[tuple(i)] for i in idx]}")


def assert_within_tolerance(got: np.ndarray, want: np.ndarray, out_dtype: torch.dtype, what: str = ""):
    g = as_f64(got, out_dtype)
    o = as_f64(want, out_dtype)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    omax = float(np.abs(o).max()) if o.size else 0.0
    err = np.abs(g - o)
    if out_dtype == torch.float32:
        rel = float(err.max()) / omax if omax > 0 else float(err.max())
        assert rel <= 1e-5, f"{what}: max|D-O|/max|O| = {rel:.3e} > 1e-5"
        rown_o = float(np.abs(o).sum(axis=1).max()) if o.size else 0.0
        rown_e = float(err.sum(axis=1).max()) if o.size else 0.0
        assert rown_e <= 1e-5 * max(rown_o, 1e-30), f"{what}: inf-norm ratio {rown_e / max(rown_o, 1e-30):.3e}"
    else:
        bound = 2.0 ** -7 * np.abs(o) + 1e-5 * omax
        bad = err > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements outside 2^-7|O| + 1e-5 max|O|; "
                               f"worst excess {float((err - bound).max()):.3e}")

