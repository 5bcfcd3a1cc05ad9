"""Addressing at the extremes: row strides and slice strides that put element
offsets past 2^32, and an output of more than 2^31 elements. Integer inputs,
compared with the oracle bit for bit on every written element (or on sampled
rows where the output is large); the untouched rest of each buffer must stay
NaN. The buffers are sparse in use but large in extent (up to ~20 GB)."""
import numpy as np
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import BF16_NAN, assert_bit_exact, bits, oracle_out, out_code

pytestmark = pytest.mark.gpu


def far_ld(M: int) -> int:
    """A row stride (a multiple of 64 elements) that puts the last row's first
    element past 2^32."""
    return ((2 ** 32) // (M - 1) // 64 + 1) * 64


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)
    torch.cuda.empty_cache()


def _ints(shape, g):
    return torch.randint(-4, 5, shape, generator=g).to(torch.bfloat16)


def _nan_buffer(elems, dtype):
    t = torch.empty(elems, dtype=dtype, device="cuda")
    if dtype == torch.bfloat16:
        t.view(torch.int16).fill_(BF16_NAN)
    else:
        t.fill_(float("nan"))
    return t


def _strided(buf, rows, cols, ld):
    return torch.as_strided(buf, (rows, cols), (ld, 1))


def _written_count(buf, chunk=2 ** 28):
    """Elements that are not NaN, counted on the GPU a slice at a time."""
    n = 0
    for i in range(0, buf.numel(), chunk):
        n += int((~torch.isnan(buf[i:i + chunk])).sum().item())
    return n


def _run_strided(h, M, N, K, out_dtype, beta, g):
    ld = far_ld(M)
    assert (M - 1) * ld > 2 ** 32
    A, B = _ints((M, K), g), _ints((K, N), g)
    Ad, Bd = A.cuda(), B.cuda()
    Cv, Cbuf = None, None
    if beta != 0.0:
        Cv = _ints((M, N), g).to(out_dtype)
        Cbuf = _nan_buffer((M - 1) * ld + N, out_dtype)
        _strided(Cbuf, M, N, ld).copy_(Cv.cuda())
    Dbuf = _nan_buffer((M - 1) * ld + N + 64, out_dtype)
    st = tpd.gemm_run(h, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, Cbuf.data_ptr() if Cbuf is not None else None,
                      ld, Dbuf.data_ptr(), ld, 1.0, beta, out_code(out_dtype), torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    D = _strided(Dbuf, M, N, ld).cpu()
    want = oracle_out(A, B, Cv, 1.0, beta, out_dtype)
    assert_bit_exact(bits(D), want, f"M={M} N={N} ld={ld}")
    # every written element is inside D (integer results are never NaN)
    assert _written_count(Dbuf) == M * N
    del Cbuf, Dbuf
    torch.cuda.empty_cache()


@pytest.mark.parametrize("out_dtype,beta", [(torch.bfloat16, 1.0), (torch.float32, 0.0)], ids=["bf16", "f32"])
@pytest.mark.parametrize("shape", [(16, 4096, 128), (300, 520, 128), (100, 1000, 72)],
                         ids=["stream", "pair", "cta"])
def test_row_strides_past_2_32(h, shape, out_dtype, beta):
    """D (and C) rows far apart: the epilogue's and the TMA maps' row offsets
    must be 64-bit. Decode-sized M runs the streaming kernel, M = 300 the CTA
    pairs and M = 100 the 1-CTA tiles (ragged N and K in both)."""
    M, N, K = shape
    g = torch.Generator().manual_seed(M + N)
    _run_strided(h, M, N, K, out_dtype, beta, g)


def test_batched_slice_stride_past_2_32(h):
    """Two slices of D 2^32 + 64 elements apart (CTA-pair tiles, ragged M and N)."""
    batch, M, N, K = 2, 300, 264, 64
    sD = 2 ** 32 + 64
    g = torch.Generator().manual_seed(7)
    A, B = _ints((batch, M, K), g), _ints((batch, K, N), g)
    Ad, Bd = A.cuda(), B.cuda()
    Dbuf = _nan_buffer(sD + M * N + 64, torch.bfloat16)
    st = tpd.gemm_run_batched(h, batch, M, N, K, Ad.data_ptr(), K, M * K, Bd.data_ptr(), N, K * N, None, N, 0,
                              Dbuf.data_ptr(), N, sD, 1.0, 0.0, tpd.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    for b in range(batch):
        D = Dbuf[b * sD: b * sD + M * N].view(M, N).cpu()
        assert_bit_exact(bits(D), oracle_out(A[b], B[b], None, 1.0, 0.0, torch.bfloat16), f"slice {b}")
    assert _written_count(Dbuf) == batch * M * N
    del Dbuf
    torch.cuda.empty_cache()


def test_output_of_more_than_2_31_elements(h):
    """131072 x 16896 = 2.2e9 outputs (4.4 GB of bf16) on the CTA pairs; sampled
    rows, including the last ones, against the oracle."""
    M, N, K = 131072, 16896, 64
    assert M * N > 2 ** 31
    g = torch.Generator().manual_seed(11)
    A, B = _ints((M, K), g), _ints((K, N), g)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    D.view(torch.int16).fill_(BF16_NAN)
    st = tpd.gemm_run(h, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 0.0,
                      tpd.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    rows = np.array(sorted({0, 1, 255, 256, 65535, 65536, 100000, M - 257, M - 2, M - 1}), dtype=np.int64)
    got = D[torch.from_numpy(rows).cuda()].cpu()
    assert_bit_exact(bits(got), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16, rows=rows), "sampled rows")
    assert _written_count(D.view(-1)) == M * N
    del D
    torch.cuda.empty_cache()
