"""The allocation-free entry point, gemm_run_noalloc, against the oracle and
against gemm_run.

gemm_run_noalloc exists for callers that cannot call cudaMalloc (code whose
device memory must all come from a pool owned by an outer framework, serving
loops that forbid allocation after warm-up): it needs no handle, and its
kernel's scratch status word lives in a static device array instead of memory
from gemm_create. Every case makes two calls in a row, so a status word or
any other state left by one call that leaked into the next would show.

The cases cover both branches of its launch plan:
  - few tiles, where the CTAs of a cluster share a tile's K range (K split of
    2 or 4);
  - more tiles than co-resident clusters, or a single K block, where the
    persistent 1-CTA schedule runs with no K split (its last round cut into
    column pieces), including M well above 128 rows.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes both alone in a fresh process and
after the other tests.
"""
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import alloc_out, assert_bit_exact, assert_within_tolerance, bits, oracle_out, to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc(A, B, C, D, alpha, beta, out_code, check):
    M, K = A.shape
    N = B.shape[1]
    s = torch.cuda.current_stream().cuda_stream
    return tpd.gemm_run_noalloc(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                                C.data_ptr() if C is not None else None, C.stride(0) if C is not None else N,
                                D.data_ptr(), D.stride(0), alpha, beta, out_code, s, check)


def _gemm_run(h, A, B, C, D, alpha, beta, out_code):
    M, K = A.shape
    N = B.shape[1]
    s = torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run(h, M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
                      C.data_ptr() if C is not None else None, C.stride(0) if C is not None else N,
                      D.data_ptr(), D.stride(0), alpha, beta, out_code, s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK


def _all_nan(x, out_dtype):
    if out_dtype == torch.bfloat16:
        return bool(((x & 0x7F80) == 0x7F80).all() and ((x & 0x007F) != 0).all())
    return bool((x != x).all())


def _ksplit_of_plan(M, N, K, out_code):
    """The K split gemm_run (automatic plan) and gemm_run_noalloc share for
    this shape: the cluster size of a 1-CTA plan, else 1."""
    h = tpd.gemm_create(0)
    try:
        p = tpd.gemm_query_plan(h, M, N, K, out_code)
    finally:
        tpd.gemm_destroy(h)
    return p["cluster"] if p["variant"] == tpd.VARIANT_TILED else 1


def _with_forced_tiled(fn):
    h = tpd.gemm_create(0)
    try:
        assert tpd.gemm_force_variant(h, tpd.VARIANT_TILED) == tpd.OK
        return fn(h)
    finally:
        tpd.gemm_destroy(h)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_noalloc_random_ksplit_branch_twice(out_dtype):
    out_code = tpd.OUT_F32 if out_dtype == torch.float32 else tpd.OUT_BF16
    M, N, K = 520, 780, 1000  # several tiles, ragged in M, N (incl. a partial 16-byte cell for bf16) and K
    assert _ksplit_of_plan(M, N, K, out_code) > 1
    cfg = CONFIGS["mlp_down"]
    A, B, C = make_inputs(cfg, M=M, N=N, K=K, lda=1008, ldb=784, ldc=784, seed=21)
    if out_dtype == torch.float32:
        C = C.to(torch.float32)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    want = oracle_out(A, B, C, 0.75, -1.5, out_dtype)
    h = tpd.gemm_create(0)
    try:
        ref, _ = alloc_out(M, N, out_dtype, ldd=792)
        _gemm_run(h, Ad, Bd, Cd, ref, 0.75, -1.5, out_code)
    finally:
        tpd.gemm_destroy(h)
    for call in range(2):  # two calls in a row: the shared scratch must not carry state over
        got, _ = alloc_out(M, N, out_dtype, ldd=792)
        st = _noalloc(Ad, Bd, Cd, got, 0.75, -1.5, out_code, check=call)
        assert st == tpd.OK, tpd.gemm_status_string(st)
        torch.cuda.synchronize()
        assert_within_tolerance(bits(got), want, out_dtype, f"noalloc call {call} against the oracle")
        assert_bit_exact(bits(got), bits(ref), f"noalloc call {call} against gemm_run (same plan, same bits)")


# (M, N, K): 1100 x 2600 has 9 x 11 = 99 tiles of 128 x 256 and 640 x 4100
# has 5 x 17 = 85, more than the co-resident clusters of two; K = 64 is one K
# block, nothing to share.
NO_SPLIT = [(1100, 2600, 200), (300, 520, 64), (640, 4100, 96)]


@pytest.mark.parametrize("shape", NO_SPLIT, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_noalloc_integer_persistent_branch_twice(shape, out_dtype):
    M, N, K = shape
    out_code = tpd.OUT_F32 if out_dtype == torch.float32 else tpd.OUT_BF16
    assert _ksplit_of_plan(M, N, K, out_code) == 1, "the shape must take the branch without a K split"
    A, B, C = make_inputs(CONFIGS["mlp_down"], integer=True, M=M, N=N, K=K, lda=K + 8, ldb=N + 8 - N % 8,
                          ldc=N + 8 - N % 8, seed=M + N + K)
    C = C.to(out_dtype)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    want = oracle_out(A, B, C, 2.0, -1.0, out_dtype)

    def forced(h):
        D, _ = alloc_out(M, N, out_dtype)
        _gemm_run(h, Ad, Bd, Cd, D, 2.0, -1.0, out_code)
        return bits(D)

    ref = _with_forced_tiled(forced)
    assert_bit_exact(ref, want, "gemm_run with 1-CTA tiles against the oracle")
    for call in range(2):
        got, base = alloc_out(M, N, out_dtype)
        assert _noalloc(Ad, Bd, Cd, got, 2.0, -1.0, out_code, check=1) == tpd.OK
        assert_bit_exact(bits(got), want, f"noalloc call {call} against the oracle")
        assert_bit_exact(bits(got), ref, f"noalloc call {call} against gemm_run")
        assert _all_nan(bits(base)[M:], out_dtype), "rows below D were written"


def test_noalloc_integer_f32_no_c_and_errors():
    cfg = CONFIGS["tiny"]
    A, B, _ = make_inputs(cfg, integer=True, M=300, N=264, K=72)
    Ad, Bd = to_device(A), to_device(B)
    want = oracle_out(A, B, None, 1.0, 0.0, torch.float32)
    for call in range(2):
        got = torch.full((300, 264), float("nan"), device="cuda")
        assert _noalloc(Ad, Bd, None, got, 1.0, 0.0, tpd.OUT_F32, check=1) == tpd.OK
        assert_bit_exact(bits(got), want, f"integer call {call}")
    # argument errors are reported before anything runs
    s = torch.cuda.current_stream().cuda_stream
    assert tpd.gemm_run_noalloc(2 ** 31, 8, 8, Ad.data_ptr(), 72, Bd.data_ptr(), 264, None, 264,
                                got.data_ptr(), 264, 1.0, 0.0, tpd.OUT_F32, s, 0) == tpd.ERR_TOO_LARGE
    assert tpd.gemm_run_noalloc(300, 264, 72, Ad.data_ptr(), 72, Bd.data_ptr(), 264, None, 264,
                                Ad.data_ptr(), 264, 1.0, 0.0, tpd.OUT_F32, s, 0) == tpd.ERR_OVERLAP
