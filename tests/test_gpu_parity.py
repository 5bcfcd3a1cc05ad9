"""GPU parity against the CPU oracle on shapes the oracle finishes in seconds:
several tiles, ragged tails in M, N and K, padded row strides, both output
dtypes, alpha/beta, both kernel variants. Every call goes through the C ABI
(gemm_run). Integer inputs are compared bit for bit, random inputs within the
stated tolerances (tests/_gpu.py)."""
import numpy as np
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import (alloc_out, assert_bit_exact, assert_within_tolerance, bits, oracle_out, round8, run,
                  to_device)
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

# (M, N, K): single elements, every ragged combination of the edge sizes the
# tiles (128 x 256 x 64, and 128-wide panels for M <= 64) meet, and multi-tile cases.
EDGE_SHAPES = [
    (1, 8, 8), (1, 1, 1), (7, 15, 1), (15, 64, 7), (16, 128, 64), (64, 127, 15), (64, 264, 1000),
    (65, 256, 64), (127, 129, 64), (129, 255, 127), (255, 257, 129), (257, 1000, 255),
    (1000, 1, 257), (1, 1000, 1000), (128, 256, 64), (384, 768, 320), (520, 600, 2048),
]


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


def _inputs(M, N, K, seed, integer, with_c, c_dtype, pad=0):
    cfg = CONFIGS["tiny"]
    A, B, C = make_inputs(cfg, integer=integer, M=M, N=N, K=K, lda=round8(K) + pad,
                          ldb=round8(N) + pad, ldc=round8(N) + pad, seed=seed, c_for_beta=with_c)
    if C is not None and C.dtype != c_dtype:
        C = _cast_keep_stride(C, c_dtype)
    return A, B, C


def _cast_keep_stride(t, dtype):
    """Cast a padded row-major view without losing its row stride."""
    rows, cols = t.shape
    if rows <= 1 or t.stride(0) == cols:
        return t.to(dtype)
    base = torch.as_strided(t, (rows, t.stride(0)), (t.stride(0), 1))
    return base.to(dtype)[:, :cols]


def _variant(h, v):
    assert tpd.gemm_force_variant(h, v) == tpd.OK


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("ab", [(1.0, 0.0), (0.5, -2.0), (2.0, 1.0)], ids=["a1b0", "a.5b-2", "a2b1"])
def test_integer_bit_exact(h, shape, out_dtype, ab):
    M, N, K = shape
    alpha, beta = ab
    A, B, C = _inputs(M, N, K, seed=M * 7 + N * 3 + K, integer=True, with_c=beta != 0, c_dtype=out_dtype,
                      pad=8 if (M + N) % 2 else 0)
    _variant(h, tpd.VARIANT_AUTO)
    D, base = run(h, A, B, C, alpha, beta, out_dtype, ldd=round8(N) + 8)
    want = oracle_out(A, B, C, alpha, beta, out_dtype)
    assert_bit_exact(bits(D), want, f"{shape} {out_dtype} {ab}")
    # nothing outside the M x N view was written: padding columns and guard rows keep the sentinel
    sentinel = alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]
    b = bits(base).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(sentinel).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]), "row-stride padding of D was written"
    assert np.array_equal(b[M:], s[M:]), "rows below D were written"


@pytest.mark.parametrize("shape", [s for s in EDGE_SHAPES if s[0] <= 64], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant", [tpd.VARIANT_TILED, tpd.VARIANT_STREAM], ids=["tiled", "stream"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_small_m_both_variants(h, shape, variant, out_dtype):
    M, N, K = shape
    A, B, C = _inputs(M, N, K, seed=11, integer=True, with_c=True, c_dtype=out_dtype)
    _variant(h, variant)
    try:
        D, _ = run(h, A, B, C, 1.0, -1.0, out_dtype)
    finally:
        _variant(h, tpd.VARIANT_AUTO)
    assert_bit_exact(bits(D), oracle_out(A, B, C, 1.0, -1.0, out_dtype), f"{shape} variant {variant}")


@pytest.mark.parametrize("shape", [(256, 256, 256), (300, 520, 1000), (129, 264, 4096), (48, 4096, 4096),
                                   (16, 2048, 14336), (640, 512, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_random_within_tolerance(h, shape, out_dtype):
    M, N, K = shape
    cfg = CONFIGS["mlp_down"]  # A N(0,1), B N(0,0.02), C N(0,1)
    A, B, C = make_inputs(cfg, M=M, N=N, K=K, seed=M + N + K)
    if out_dtype == torch.float32:
        C = C.to(torch.float32)
    D, _ = run(h, A, B, C, 1.0, 1.0, out_dtype)
    assert_within_tolerance(bits(D), oracle_out(A, B, C, 1.0, 1.0, out_dtype), out_dtype, str(shape))


def test_uniform_tiny_config_fp32(h):
    cfg = CONFIGS["tiny"]
    A, B, _ = make_inputs(cfg)
    D, _ = run(h, A, B, None, cfg.alpha, cfg.beta, torch.float32)
    assert_within_tolerance(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.float32), torch.float32, "tiny")


def test_k_zero_gives_beta_c(h):
    M, N = 130, 264
    C = torch.randint(-4, 5, (M, N)).to(torch.float32)
    A = torch.zeros((M, 0), dtype=torch.bfloat16)
    B = torch.zeros((0, N), dtype=torch.bfloat16)
    for out_dtype in (torch.float32, torch.bfloat16):
        Cx = C.to(out_dtype)
        D, _ = run(h, A, B, Cx, 1.0, -2.0, out_dtype)
        want = (-2.0 * Cx.to(torch.float32)).to(out_dtype)  # small integers: exact in both dtypes
        assert_bit_exact(bits(D), bits(want), "K=0")
        D, _ = run(h, A, B, None, 1.0, 0.0, out_dtype)
        assert np.all(bits(D).astype(np.float64) == 0)


def test_beta_zero_never_reads_c(h):
    M, N, K = 200, 264, 128
    A, B, _ = _inputs(M, N, K, seed=3, integer=True, with_c=False, c_dtype=torch.float32)
    Cnan = torch.full((M, N), float("nan"), device="cuda")
    Ad, Bd = to_device(A), to_device(B)
    D, _ = alloc_out(M, N, torch.float32)
    st = tpd.gemm_run(h, M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), Cnan.data_ptr(), N,
                      D.data_ptr(), D.stride(0), 1.0, 0.0, tpd.OUT_F32, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.float32), "beta=0")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("M", [40, 300])
def test_in_place_d_equals_c(h, out_dtype, M):
    N, K = 520, 256
    A, B, C = _inputs(M, N, K, seed=5, integer=True, with_c=True, c_dtype=out_dtype)
    want = oracle_out(A, B, C, 1.0, 1.0, out_dtype)
    Cd = to_device(C)
    D, _ = run(h, A, B, Cd, 1.0, 1.0, out_dtype, D=Cd)
    assert_bit_exact(bits(Cd), want, "in place")


@pytest.mark.parametrize("shape", [(2560, 2048, 64), (2560, 1800, 72), (300, 520, 256)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant", [tpd.VARIANT_TILED, tpd.VARIANT_TILED_PAIR], ids=["tiled", "pair"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_tiled_modes_with_tail_split(h, shape, variant, out_dtype):
    """Both tiled modes on shapes whose last round is cut into column pieces
    (2560 x 2048: 160 tiles on 152 CTAs leave 8, cut into 64-column quarters;
    80 pair tiles on 76 pairs leave 4, cut into halves); with N = 1800 some
    pieces lie entirely right of N; 300 x 520 has fewer tiles than CTAs, so
    every tile is cut."""
    M, N, K = shape
    A, B, C = _inputs(M, N, K, seed=M + N, integer=True, with_c=True, c_dtype=out_dtype)
    _variant(h, variant)
    try:
        D, base = run(h, A, B, C, 1.0, 1.0, out_dtype, ldd=round8(N) + 8)
    finally:
        _variant(h, tpd.VARIANT_AUTO)
    assert_bit_exact(bits(D), oracle_out(A, B, C, 1.0, 1.0, out_dtype), f"{shape} variant {variant}")
    b = bits(base).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]) and np.array_equal(b[M:], s[M:])
