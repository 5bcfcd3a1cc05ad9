"""Batched (bmm) and grouped (grouped_mm, mixture-of-experts) GEMM against the
oracle, slice by slice and group by group ("TorchInductor ganha suporte a
GEMMs de alta performance com CuteDSL", enablement paragraph: NVGEMM covers
mm, bmm, scaled_mm and grouped_mm). Integer inputs are compared bit for bit,
random inputs within the stated tolerances; sentinels check that nothing
outside the output slices or rows is written."""
import numpy as np
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import BF16_NAN, assert_bit_exact, assert_within_tolerance, bits, oracle_out, out_code, round8
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


def _stack(mats, ld, gap_rows=0, dtype=None):
    """Slices stacked with row stride ld and gap_rows NaN rows between them.
    Returns (base tensor on the GPU, slice stride in elements)."""
    rows, cols = mats[0].shape
    dtype = dtype or mats[0].dtype
    stride = (rows + gap_rows) * ld
    base = torch.full((len(mats) * (rows + gap_rows), ld), float("nan"), dtype=torch.float32).to(dtype)
    for b, m in enumerate(mats):
        base[b * (rows + gap_rows): b * (rows + gap_rows) + rows, :cols] = m.to(dtype)
    return base.cuda(), stride


def _nan_base(shape, dtype):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    if dtype == torch.bfloat16:
        t.view(torch.int16).fill_(BF16_NAN)
    else:
        t.fill_(float("nan"))
    return t


@pytest.mark.parametrize("shape", [(300, 520, 136), (64, 264, 72), (256, 200, 64)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("share", ["none", "B", "C"])
def test_batched_integer_bit_exact(h, shape, out_dtype, share):
    M, N, K = shape
    batch = 3
    g = torch.Generator().manual_seed(M + N)
    As = [torch.randint(-4, 5, (M, K), generator=g).to(torch.bfloat16) for _ in range(batch)]
    Bs = [torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16) for _ in range(batch)]
    Cs = [torch.randint(-4, 5, (M, N), generator=g).to(out_dtype) for _ in range(batch)]
    if share == "B":
        Bs = [Bs[0]] * batch
    if share == "C":
        Cs = [Cs[0]] * batch
    lda, ldb, ldc, ldd = round8(K) + 8, round8(N), round8(N) + 8, round8(N) + 8
    Ab, sA = _stack(As, lda, gap_rows=1)
    Bb, sB = _stack(Bs if share != "B" else Bs[:1], ldb)
    Cb, sC = _stack(Cs if share != "C" else Cs[:1], ldc)
    gap = 2
    D = _nan_base((batch * (M + gap), ldd), out_dtype)
    sD = (M + gap) * ldd
    s = torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run_batched(h, batch, M, N, K, Ab.data_ptr(), lda, sA, Bb.data_ptr(), ldb,
                              0 if share == "B" else sB, Cb.data_ptr(), ldc, 0 if share == "C" else sC, D.data_ptr(),
                              ldd, sD, 1.0, -2.0, out_code(out_dtype), s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    d = bits(D)
    sentinel = bits(_nan_base((1, ldd), out_dtype))[0]
    for b in range(batch):
        rows = slice(b * (M + gap), b * (M + gap) + M)
        want = oracle_out(As[b], Bs[b], Cs[b], 1.0, -2.0, out_dtype)
        assert_bit_exact(d[rows, :N], want, f"batch {b}")
        view = np.uint16 if out_dtype == torch.bfloat16 else np.uint32
        assert np.all(d[rows, N:].view(view) == sentinel[N:].view(view)), "padding written"
        gap_rows = d[b * (M + gap) + M: (b + 1) * (M + gap)]
        assert np.all(gap_rows.view(view) == sentinel.view(view)), "rows between slices written"


def test_batched_random_within_tolerance(h):
    batch, M, N, K = 4, 512, 768, 1024
    cfg = CONFIGS["qkv"]
    As, Bs = [], []
    for b in range(batch):
        A, B, _ = make_inputs(cfg, M=M, N=N, K=K, seed=10 + b)
        As.append(A)
        Bs.append(B)
    Ab = torch.stack(As).cuda()
    Bb = torch.stack(Bs).cuda()
    D = torch.empty((batch, M, N), dtype=torch.bfloat16, device="cuda")
    st = tpd.gemm_run_batched(h, batch, M, N, K, Ab.data_ptr(), K, M * K, Bb.data_ptr(), N, K * N, None, N, 0,
                              D.data_ptr(), N, M * N, 1.0, 0.0, tpd.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK and tpd.gemm_sync_status(h, None) == tpd.OK
    for b in range(batch):
        assert_within_tolerance(bits(D[b]), oracle_out(As[b], Bs[b], None, 1.0, 0.0, torch.bfloat16),
                                torch.bfloat16, f"batch {b}")


def test_batched_matches_single_calls_bitwise(h):
    """A batched launch and batch separate gemm_run calls give the same bits
    on integer inputs. (A single call this size shares each tile's K range
    between the CTAs of a cluster, so on random inputs its fp32 sums are
    rounded in another order than the batched kernel's.)"""
    batch, M, N, K = 3, 384, 512, 256
    g = torch.Generator().manual_seed(13)
    A = torch.randint(-4, 5, (batch, M, K), generator=g).bfloat16().cuda()
    B = torch.randint(-4, 5, (batch, K, N), generator=g).bfloat16().cuda()
    D1 = torch.empty(batch, M, N, device="cuda", dtype=torch.bfloat16)
    D2 = torch.empty_like(D1)
    s = torch.cuda.current_stream().cuda_stream
    assert tpd.gemm_run_batched(h, batch, M, N, K, A.data_ptr(), K, M * K, B.data_ptr(), N, K * N, None, N, 0,
                                D1.data_ptr(), N, M * N, 1.0, 0.0, tpd.OUT_BF16, s) == tpd.OK
    for b in range(batch):
        assert tpd.gemm_run(h, M, N, K, A[b].data_ptr(), K, B[b].data_ptr(), N, None, N, D2[b].data_ptr(), N, 1.0,
                            0.0, tpd.OUT_BF16, s) == tpd.OK
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))


GROUPS = {
    "ragged": [0, 37, 300, 129, 0, 256, 1, 64],      # empty groups, tiles crossing group ends
    "large": [512, 300, 700, 256],                    # CTA pairs (average > 128 rows)
    "one": [333],
    "many_small": [17] * 40,
}


@pytest.mark.parametrize("name", list(GROUPS))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_grouped_integer_bit_exact(h, name, out_dtype):
    rows = GROUPS[name]
    G, total = len(rows), sum(rows)
    N, K = 520, 136
    g = torch.Generator().manual_seed(G)
    A = torch.randint(-4, 5, (total, K), generator=g).to(torch.bfloat16)
    Bs = [torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16) for _ in range(G)]
    C = torch.randint(-4, 5, (total, N), generator=g).to(out_dtype)
    ldb = round8(N)
    Bb, sB = _stack(Bs, ldb)
    ldd = round8(N) + 8
    D = _nan_base((total + 4, ldd), out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    Ad, Cd = A.cuda(), C.cuda()
    st = tpd.gemm_run_grouped(h, rows, N, K, Ad.data_ptr(), K, Bb.data_ptr(), ldb, sB, Cd.data_ptr(), N,
                              D.data_ptr(), ldd, 2.0, 1.0, out_code(out_dtype), s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    d = bits(D)
    view = np.uint16 if out_dtype == torch.bfloat16 else np.uint32
    sentinel = bits(_nan_base((1, ldd), out_dtype))[0].view(view)
    r0 = 0
    for gi, r in enumerate(rows):
        if r:
            want = oracle_out(A[r0:r0 + r], Bs[gi], C[r0:r0 + r], 2.0, 1.0, out_dtype)
            assert_bit_exact(d[r0:r0 + r, :N], want, f"group {gi}")
        r0 += r
    assert np.all(d[:total, N:].view(view) == sentinel[N:]), "padding written"
    assert np.all(d[total:].view(view) == sentinel), "rows after the last group written"


def test_grouped_random_within_tolerance(h):
    rows = [1000, 24, 512, 300]
    N, K = 1024, 2048
    cfg = CONFIGS["mlp_down"]
    A, _, _ = make_inputs(cfg, M=sum(rows), N=8, K=K, seed=5)
    Bs = [make_inputs(cfg, M=8, N=N, K=K, seed=20 + i)[1] for i in range(len(rows))]
    Bb = torch.stack(Bs).cuda()
    D = torch.empty((sum(rows), N), dtype=torch.bfloat16, device="cuda")
    st = tpd.gemm_run_grouped(h, rows, N, K, A.cuda().data_ptr(), K, Bb.data_ptr(), N, K * N, None, N,
                              D.data_ptr(), N, 1.0, 0.0, tpd.OUT_BF16, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK and tpd.gemm_sync_status(h, None) == tpd.OK
    r0 = 0
    for gi, r in enumerate(rows):
        want = oracle_out(A[r0:r0 + r], Bs[gi], None, 1.0, 0.0, torch.bfloat16)
        assert_within_tolerance(bits(D[r0:r0 + r]), want, torch.bfloat16, f"group {gi}")
        r0 += r


def test_batched_and_grouped_argument_errors(h):
    A = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((256, 64), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # D slices overlapping each other
    assert tpd.gemm_run_batched(h, 2, 128, 64, 64, A.data_ptr(), 64, 128 * 64, B.data_ptr(), 64, 0, None, 64, 0,
                                D.data_ptr(), 64, 64 * 64, 1.0, 0.0, tpd.OUT_F32, s) == tpd.ERR_OVERLAP
    # misaligned batch stride
    assert tpd.gemm_run_batched(h, 2, 64, 64, 64, A.data_ptr(), 64, 64 * 64 + 4, B.data_ptr(), 64, 0, None, 64, 0,
                                D.data_ptr(), 64, 128 * 64, 1.0, 0.0, tpd.OUT_F32, s) == tpd.ERR_ALIGNMENT
    assert tpd.gemm_run_batched(h, -1, 64, 64, 64, A.data_ptr(), 64, 0, B.data_ptr(), 64, 0, None, 64, 0,
                                D.data_ptr(), 64, 0, 1.0, 0.0, tpd.OUT_F32, s) == tpd.ERR_INVALID_ARG
    # grouped: too many groups, negative rows
    assert tpd.gemm_run_grouped(h, [1] * 257, 64, 64, A.data_ptr(), 64, B.data_ptr(), 64, 0, None, 64, D.data_ptr(),
                                64, 1.0, 0.0, tpd.OUT_F32, s) == tpd.ERR_TOO_LARGE
    assert tpd.gemm_run_grouped(h, [4, -1], 64, 64, A.data_ptr(), 64, B.data_ptr(), 64, 0, None, 64, D.data_ptr(),
                                64, 1.0, 0.0, tpd.OUT_F32, s) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_sync_status(h, None) == tpd.OK


def test_batched_and_grouped_k_zero(h):
    C = torch.randint(-4, 5, (2, 70, 264)).float().cuda()
    D = torch.empty_like(C)
    s = torch.cuda.current_stream().cuda_stream
    assert tpd.gemm_run_batched(h, 2, 70, 264, 0, None, 0, 0, None, 264, 0, C.data_ptr(), 264, 70 * 264,
                                D.data_ptr(), 264, 70 * 264, 1.0, 3.0, tpd.OUT_F32, s) == tpd.OK
    torch.cuda.synchronize()
    assert torch.equal(D, 3.0 * C)
    D2 = torch.empty(140, 264, device="cuda")
    assert tpd.gemm_run_grouped(h, [100, 40], 264, 0, None, 0, None, 264, 0, C.view(140, 264).data_ptr(), 264,
                                D2.data_ptr(), 264, 1.0, -1.0, tpd.OUT_F32, s) == tpd.OK
    torch.cuda.synchronize()
    assert torch.equal(D2, -C.view(140, 264))
