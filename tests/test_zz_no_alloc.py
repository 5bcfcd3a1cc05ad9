"""The allocation-free entry point, gemm_run_noalloc, against gemm_run.

gemm_run_noalloc exists for callers that cannot call cudaMalloc (code whose
device memory must all come from a pool owned by an outer framework, serving
loops that forbid allocation after warm-up): it needs no handle, and its
kernel's scratch status word lives in a static device array instead of memory
from gemm_create. This file is collected last so that a run stopping at the
first failure has already run every other test; it passes both alone in a
fresh process and after the other tests.
"""
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import alloc_out, assert_bit_exact, assert_within_tolerance, bits, to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc(A, B, C, D, alpha, beta, out_code, check):
    M, K = A.shape
    N = B.shape[1]
    s = torch.cuda.current_stream().cuda_stream
    return tpd.gemm_run_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                C.data_ptr() if C is not None else None, C.stride(0) if C is not None else N,
                                D.data_ptr(), D.stride(0), alpha, beta, out_code, s, check)


def _reference(h, A, B, C, D, alpha, beta, out_code):
    M, K = A.shape
    N = B.shape[1]
    s = torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run(h, M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                      C.data_ptr() if C is not None else None, C.stride(0) if C is not None else N,
                      D.data_ptr(), D.stride(0), alpha, beta, out_code, s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_noalloc_matches_gemm_run_twice(out_dtype):
    out_code = tpd.OUT_F32 if out_dtype == torch.float32 else tpd.OUT_BF16
    M, N, K = 520, 780, 1000  # several tiles, ragged in M, N (incl. a partial 16-byte cell for bf16) and K
    cfg = CONFIGS["mlp_down"]
    A, B, C = make_inputs(cfg, M=M, N=N, K=K, lda=1008, ldb=784, ldc=784, seed=21)
    if out_dtype == torch.float32:
        C = C.to(torch.float32)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    h = tpd.gemm_create(0)
    try:
        want, _ = alloc_out(M, N, out_dtype, ldd=792)
        _reference(h, Ad, Bd, Cd, want, 0.75, -1.5, out_code)
    finally:
        tpd.gemm_destroy(h)
    ref = bits(want)
    for call in range(2):  # two calls in a row: the shared scratch must not carry state over
        got, _ = alloc_out(M, N, out_dtype, ldd=792)
        st = _noalloc(Ad, Bd, Cd, got, 0.75, -1.5, out_code, check=call)
        assert st == tpd.OK, tpd.gemm_status_string(st)
        torch.cuda.synchronize()
        assert_within_tolerance(bits(got), ref, out_dtype, f"noalloc call {call}")
        assert_bit_exact(bits(got), ref, f"noalloc call {call} (same kernel, same bits)")


def test_noalloc_integer_and_errors():
    cfg = CONFIGS["tiny"]
    A, B, _ = make_inputs(cfg, integer=True, M=300, N=264, K=72)
    Ad, Bd = to_device(A), to_device(B)
    h = tpd.gemm_create(0)
    try:
        want = torch.empty((300, 264), dtype=torch.float32, device="cuda")
        _reference(h, Ad, Bd, None, want, 1.0, 0.0, tpd.OUT_F32)
    finally:
        tpd.gemm_destroy(h)
    for call in range(2):
        got = torch.full((300, 264), float("nan"), device="cuda")
        assert _noalloc(Ad, Bd, None, got, 1.0, 0.0, tpd.OUT_F32, check=1) == tpd.OK
        assert_bit_exact(bits(got), bits(want), f"integer call {call}")
    # argument errors are reported before anything runs
    s = torch.cuda.current_stream().cuda_stream
    assert tpd.gemm_run_noalloc(2 ** 31, 8, 8, Ad.data_ptr(), 72, Bd.data_ptr(), 264, None, 264,
                                want.data_ptr(), 264, 1.0, 0.0, tpd.OUT_F32, s, 0) == tpd.ERR_TOO_LARGE
    assert tpd.gemm_run_noalloc(300, 264, 72, Ad.data_ptr(), 72, Bd.data_ptr(), 264, None, 264,
                                Ad.data_ptr(), 264, 1.0, 0.0, tpd.OUT_F32, s, 0) == tpd.ERR_OVERLAP
