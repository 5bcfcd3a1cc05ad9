"""GPU parity of the block-scaled FP4 GEMM, gemm_run_fp4, against the
block-scaled oracle: the NVFP4 and MXF4 GEMMs of "TorchInductor ganha suporte
a GEMMs de alta performance com CuteDSL" (enablement and results paragraphs),
read as E2M1 elements two to a byte with E4M3 scales per 16 elements (NVFP4)
or E8M0 scales per 32 (MXFP4).

Integer-valued inputs (all sixteen E2M1 codes, scales of 1/2, 1 and 2) make
every partial sum exact in fp32, so the result is unique and compared bit for
bit; N(0,1) data quantised per block is compared within the GEMM's
tolerances. The shapes cover 256 x 256 pair tiles and 128 x 128 single-CTA
tiles, the 32- and 64-row A boxes of small M, ragged M, N and K (K not a
multiple of the 256-element stage, partial scale chunks), padded row strides,
beta*C, both output dtypes and both formats.
"""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import DEV, alloc_out, assert_bit_exact, assert_within_tolerance, bits, mx_blocked, out_code, round8
from workloads import E4M3_ONE, FP4_BLOCK, FP4_CONFIGS, FP4_MX, FP4_NV, make_fp4_inputs

pytestmark = pytest.mark.gpu

FORMATS = [FP4_NV, FP4_MX]
FMT_IDS = ["nvfp4", "mxfp4"]


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


def _u8_to_device(t: torch.Tensor) -> torch.Tensor:
    rows, cols = t.shape
    ld = t.stride(0)
    if rows <= 1 or ld == cols:
        return t.contiguous().to(DEV)
    return torch.as_strided(t, (rows, ld), (ld, 1)).to(DEV)[:, :cols]


def _strided_to_device(t: torch.Tensor) -> torch.Tensor:
    rows, cols = t.shape
    ld = t.stride(0)
    return torch.as_strided(t, (rows, ld), (ld, 1)).to(DEV)[:, :cols]


def _blocked(fmt, S):
    return torch.from_numpy(mx_blocked(S.numpy(), pad=E4M3_ONE if fmt == FP4_NV else 127)).to(DEV)


def _run_fp4(h, fmt, A, SA, Bt, SB, C, alpha, beta, out_dtype, ldd=None, D=None):
    M, K = A.shape[0], 2 * A.shape[1]
    N = Bt.shape[0]
    Ad, Bd = _u8_to_device(A), _u8_to_device(Bt)
    sad, sbd = _blocked(fmt, SA), _blocked(fmt, SB)
    assert sad.numel() == tpd.gemm_fp4_scale_bytes(fmt, M, K) and sbd.numel() == tpd.gemm_fp4_scale_bytes(fmt, N, K)
    Cd = None
    if C is not None:
        Cd = C.to(DEV) if C.device.type == "cpu" else C
    base = None
    if D is None:
        D, base = alloc_out(M, N, out_dtype, ldd)
    s = torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run_fp4(h, M, N, K, fmt, Ad.data_ptr(), Ad.stride(0) if M > 1 else K // 2, sad.data_ptr(),
                          Bd.data_ptr(), Bd.stride(0) if N > 1 else K // 2, sbd.data_ptr(),
                          Cd.data_ptr() if Cd is not None else None, Cd.stride(0) if Cd is not None else N,
                          D.data_ptr(), D.stride(0), float(alpha), float(beta), out_code(out_dtype), s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    return D, base


def _want(fmt, A, SA, Bt, SB, C, alpha, beta, out_dtype, rows=None):
    sf = oracle.SCALE_E4M3 if fmt == FP4_NV else oracle.SCALE_E8M0
    D, _ = oracle.bs_gemm_rows(A, SA, Bt, SB, C, alpha, beta, out_code(out_dtype), oracle.FP4_E2M1,
                               oracle.FP4_E2M1, sf, FP4_BLOCK[fmt], rows=rows)
    return D


# (M, N, K, lda, ldb), strides in bytes: 256 x 192 pair tiles with a ragged
# last one; ragged everything with K = 96 (part of one stage, a partial scale
# chunk) and N = 200 on 256 x 256 pairs whose second CTA owns rows past M;
# single CTAs with 128 x 128 tiles (N <= 128, two row tiles); many 256 x 256
# pair tiles, N ragged; 256 x 192 pairs whose second CTA has one row, N odd
# (the column tail goes around the tensor map, and the last tile starts 64
# rows into a scale row block); M <= 32 and M <= 64 on 128 x 192 tiles with
# 32- and 64-row A boxes; 128-row boxes for M in (64, 128]; one 128 x 128 tile
# with a long K; degenerate outputs: one element with K of a single NVFP4
# block (16) or MXFP4 block (32), and a few rows and columns with K = 64.
SHAPES = [(256, 512, 512, None, None), (300, 200, 96, 64, 48), (200, 100, 320, 176, 160),
          (640, 1000, 1024, None, 528), (129, 577, 160, 96, 80), (16, 1000, 512, None, None),
          (33, 600, 192, None, None), (64, 577, 160, 96, 80), (100, 300, 256, None, None),
          (128, 128, 4096, None, None), (1, 1, 32, None, None), (3, 5, 64, None, None)]


def _ids(s):
    return "x".join(map(str, s[:3]))


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
def test_fp4_integer_bit_exact(h, fmt, shape, out_dtype):
    M, N, K, lda, ldb = shape
    A, SA, Bt, SB = make_fp4_inputs(M, N, K, seed=M + N + K + fmt, fmt=fmt, integer=True, lda=lda, ldb=ldb)
    g = torch.Generator().manual_seed(K)
    C = torch.zeros((M, round8(N)), dtype=out_dtype)[:, :N]  # row stride a multiple of 16 bytes
    C.copy_(torch.randint(-4, 5, (M, N), generator=g))
    D, base = _run_fp4(h, fmt, A, SA, Bt, SB, _strided_to_device(C), 2.0, -1.0, out_dtype, ldd=round8(N) + 8)
    assert_bit_exact(bits(D), _want(fmt, A, SA, Bt, SB, C, 2.0, -1.0, out_dtype), f"{shape} {out_dtype}")
    sentinel = alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]
    b = bits(base).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(sentinel).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]), "row-stride padding of D was written"
    assert np.array_equal(b[M:], s[M:]), "rows below D were written"


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
def test_fp4_random_within_tolerance_and_deterministic(h, fmt, out_dtype):
    M, N, K = 1000, 1000, 2048
    A, SA, Bt, SB = make_fp4_inputs(M, N, K, seed=7 + fmt, fmt=fmt)
    C = torch.randn(M, N, generator=torch.Generator().manual_seed(8)).to(out_dtype)
    D, _ = _run_fp4(h, fmt, A, SA, Bt, SB, C, 0.5, 1.0, out_dtype)
    got = bits(D)
    assert_within_tolerance(got, _want(fmt, A, SA, Bt, SB, C, 0.5, 1.0, out_dtype), out_dtype, "fp4 random")
    D2, _ = _run_fp4(h, fmt, A, SA, Bt, SB, C, 0.5, 1.0, out_dtype)
    assert np.array_equal(got.view(np.uint8), bits(D2).view(np.uint8)), "run-to-run difference"


def test_fp4_nibble_order(h):
    """One nonzero element pair: the low nibble is the even element along K.
    A row holds 1.0 at element 2 only (byte 1, low nibble); B's column 0 holds
    6.0 at element 2 and 0.5 at element 3, column 1 the reverse. D[0, 0] =
    6 and D[0, 1] = 0.5 only if the kernel pairs nibbles as the oracle does."""
    M, N, K = 1, 2, 64
    A = torch.zeros((M, K // 2), dtype=torch.uint8)
    A[0, 1] = 0x02  # element 2 = 1.0, element 3 = 0
    Bt = torch.zeros((N, K // 2), dtype=torch.uint8)
    Bt[0, 1] = 0x17  # element 2 = 6.0, element 3 = 0.5
    Bt[1, 1] = 0x71  # element 2 = 0.5, element 3 = 6.0
    SA = torch.full((M, K // 16), E4M3_ONE, dtype=torch.uint8)
    SB = torch.full((N, K // 16), E4M3_ONE, dtype=torch.uint8)
    D, _ = _run_fp4(h, FP4_NV, A, SA, Bt, SB, None, 1.0, 0.0, torch.float32)
    want = _want(FP4_NV, A, SA, Bt, SB, None, 1.0, 0.0, torch.float32)
    assert_bit_exact(bits(D), want, "nibble order")
    assert want.view(np.float32)[0, 0] == 6.0 and want.view(np.float32)[0, 1] == 0.5


@pytest.mark.parametrize("name", list(FP4_CONFIGS))
def test_fp4_workloads_every_element(h, name):
    """The benchmarked FP4 shapes at full size, every element: integer inputs
    bit for bit, quantised random inputs within the bf16 tolerance."""
    cfg = FP4_CONFIGS[name]
    A, SA, Bt, SB = make_fp4_inputs(cfg.M, cfg.N, cfg.K, seed=cfg.seed, fmt=cfg.fmt, integer=True)
    D, _ = _run_fp4(h, cfg.fmt, A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16)
    assert_bit_exact(bits(D), _want(cfg.fmt, A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16), f"{name} integer")
    del D
    A, SA, Bt, SB = make_fp4_inputs(cfg.M, cfg.N, cfg.K, seed=cfg.seed, fmt=cfg.fmt)
    D, _ = _run_fp4(h, cfg.fmt, A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16)
    assert_within_tolerance(bits(D), _want(cfg.fmt, A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16),
                            torch.bfloat16, f"{name} random")


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
def test_fp4_in_place_and_k_zero(h, fmt):
    M, N, K = 300, 400, 256
    A, SA, Bt, SB = make_fp4_inputs(M, N, K, seed=3, fmt=fmt, integer=True)
    C = torch.randint(-4, 5, (M, N), generator=torch.Generator().manual_seed(3)).to(torch.float32)
    want = _want(fmt, A, SA, Bt, SB, C, 1.0, 1.0, torch.float32)
    Cd = C.to(DEV)
    _run_fp4(h, fmt, A, SA, Bt, SB, Cd, 1.0, 1.0, torch.float32, D=Cd)
    assert_bit_exact(bits(Cd), want, "in place")
    D = torch.full((M, N), float("nan"), device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    Cd = C.to(DEV)
    assert tpd.gemm_run_fp4(h, M, N, 0, fmt, None, 0, None, None, 0, None, Cd.data_ptr(), N, D.data_ptr(), N, 1.0,
                            -2.0, tpd.OUT_F32, s) == tpd.OK
    torch.cuda.synchronize()
    assert torch.equal(D.cpu(), -2.0 * C)


def test_fp4_argument_errors(h):
    s = torch.cuda.current_stream().cuda_stream
    A = torch.zeros((128, 128), dtype=torch.uint8, device=DEV)
    B = torch.zeros((128, 128), dtype=torch.uint8, device=DEV)
    S = torch.zeros(tpd.gemm_fp4_scale_bytes(tpd.NVFP4, 128, 256), dtype=torch.uint8, device=DEV)
    D = torch.zeros((128, 128), dtype=torch.float32, device=DEV)
    args = dict(M=128, N=128, K=256, fmt=tpd.NVFP4)

    def run(**kw):
        a = dict(A=A.data_ptr(), lda=128, SA=S.data_ptr(), B=B.data_ptr(), ldb=128, SB=S.data_ptr(),
                 D=D.data_ptr(), ldd=128, **args)
        a.update(kw)
        return tpd.gemm_run_fp4(h, a["M"], a["N"], a["K"], a["fmt"], a["A"], a["lda"], a["SA"], a["B"], a["ldb"],
                                a["SB"], None, a["N"], a["D"], a["ldd"], 1.0, 0.0, tpd.OUT_F32, s)

    assert run() == tpd.OK
    assert run(K=120) == tpd.ERR_INVALID_ARG           # K not a multiple of 16
    assert run(K=240, fmt=tpd.MXFP4) == tpd.ERR_INVALID_ARG  # nor of 32 for MXFP4
    assert run(fmt=2) == tpd.ERR_INVALID_ARG           # unknown format
    assert run(lda=100) == tpd.ERR_INVALID_ARG         # lda < K/2 bytes
    assert run(K=224, lda=120) == tpd.ERR_ALIGNMENT    # row stride not a multiple of 16 bytes
    assert run(SA=S.data_ptr() + 8) == tpd.ERR_ALIGNMENT
    assert run(D=S.data_ptr()) == tpd.ERR_OVERLAP      # D on top of the scales
    torch.cuda.synchronize()
    assert tpd.gemm_sync_status(h, s) == tpd.OK


def test_fp4_plan(h):
    sms = tpd.gemm_num_sms(h)
    for fmt in FORMATS:
        p = tpd.gemm_fp4_query_plan(h, fmt, 8192, 6144, 4096)
        assert p["tile_m"] == 256 and p["tile_n"] == 256 and p["num_tiles"] == 32 * 24 and p["cluster"] == 2
        assert p["grid"] % 2 == 0 and sms - 8 <= p["grid"] <= sms
        p = tpd.gemm_fp4_query_plan(h, fmt, 256, 28672, 4096)  # up to 256 rows: 256 x 192 pairs, 150 tiles
        assert p["tile_m"] == 256 and p["tile_n"] == 192 and p["cluster"] == 2 and p["num_tiles"] == 150
        p = tpd.gemm_fp4_query_plan(h, fmt, 16, 28672, 4096)  # 128 rows or fewer: single CTAs, one wave
        assert p["tile_m"] == 128 and p["tile_n"] == 192 and p["cluster"] == 1 and p["num_tiles"] == 150
        sizes = {p["smem_bytes"]}
        for m in (64, 100):  # 64-row A boxes, then 128-row ones: each its own ring
            p = tpd.gemm_fp4_query_plan(h, fmt, m, 28672, 4096)
            assert p["tile_n"] == 192 and p["smem_bytes"] not in sizes
            sizes.add(p["smem_bytes"])
        p = tpd.gemm_fp4_query_plan(h, fmt, 100, 128, 4096)  # N <= 128: 128 x 128 tiles
        assert p["tile_n"] == 128 and p["num_tiles"] == 1
        assert max(sizes) <= 232448


def test_fp4_single_nvfp4_block(h):
    """M = N = 1, K = 16: one NVFP4 block, a fraction of a stage, a chunk and a
    TMA box; integer codes, so the one output is exact."""
    A, SA, Bt, SB = make_fp4_inputs(1, 1, 16, seed=5, fmt=FP4_NV, integer=True)
    D, _ = _run_fp4(h, FP4_NV, A, SA, Bt, SB, None, 1.0, 0.0, torch.float32)
    assert_bit_exact(bits(D), _want(FP4_NV, A, SA, Bt, SB, None, 1.0, 0.0, torch.float32), "1x1x16")
