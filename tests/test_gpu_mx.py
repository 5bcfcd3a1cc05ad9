"""GPU parity of the block-scaled (MXFP8) GEMM, gemm_run_mx, against the MX
oracle: the scaled_mm of "TorchInductor ganha suporte a GEMMs de alta
performance com CuteDSL" (enablement and MXFP8 results paragraphs) with the
OCP Microscaling formats (32-element blocks along K, E8M0 scales, E4M3 or
E5M2 elements).

Integer-valued elements in {-4..4} with scales in {2^-1, 2^0, 2^1} make every
partial sum exact in fp32, so the result is unique and compared bit for bit;
random N(0,1) elements with spread scales are compared within the GEMM's
tolerances. The shapes cover 192- and 128-column tiles, tiles that start 64
rows into a scale chunk of B, ragged M, N and K (K not a multiple of 128),
padded row strides, beta*C, both output dtypes and both element formats.
"""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import DEV, alloc_out, assert_bit_exact, assert_within_tolerance, bits, mx_blocked, out_code, round8
from workloads import MX_CONFIGS, make_mx_inputs

pytestmark = pytest.mark.gpu


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


def _run_mx(h, A, SA, Bt, SB, C, alpha, beta, out_dtype, fmt_a=0, fmt_b=0, ldd=None, D=None):
    M, K = A.shape
    N = Bt.shape[0]
    Ad, Bd = _u8_to_device(A), _u8_to_device(Bt)
    sad = torch.from_numpy(mx_blocked(SA.numpy())).to(DEV)
    sbd = torch.from_numpy(mx_blocked(SB.numpy())).to(DEV)
    assert sad.numel() == tpd.gemm_mx_scale_bytes(M, K) and sbd.numel() == tpd.gemm_mx_scale_bytes(N, K)
    Cd = None
    if C is not None:
        Cd = C.to(DEV) if C.device.type == "cpu" else C
    base = None
    if D is None:
        D, base = alloc_out(M, N, out_dtype, ldd)
    s = torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run_mx(h, M, N, K, Ad.data_ptr(), Ad.stride(0) if M > 1 else K, fmt_a, sad.data_ptr(),
                         Bd.data_ptr(), Bd.stride(0) if N > 1 else K, fmt_b, sbd.data_ptr(),
                         Cd.data_ptr() if Cd is not None else None, Cd.stride(0) if Cd is not None else N,
                         D.data_ptr(), D.stride(0), float(alpha), float(beta), out_code(out_dtype), s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    return D, base


def _want(A, SA, Bt, SB, C, alpha, beta, out_dtype, fmt_a=0, fmt_b=0, rows=None):
    D, _ = oracle.mx_gemm_rows(A, SA, Bt, SB, C, alpha, beta, out_code(out_dtype), fmt_a, fmt_b, rows=rows)
    return D


# (M, N, K, lda, ldb): one 256 x 256 pair tile and a second one whose second
# scale chunk does not exist (N = 384); ragged everything with K = 96 (a
# partial K block and a partial scale chunk) and N = 200, on pairs whose second
# CTA owns rows past M; 128-column
# tiles on single CTAs (N <= 128); single CTAs with 192-wide tiles (M <= 128);
# several pair tiles in both directions with many K blocks; a pair whose
# second CTA has one row; M <= 32 on 32-row A boxes, M <= 64 on 64-row ones, and
# M <= 64 with N <= 128 on the 128-wide tiles that keep 128-row boxes.
SHAPES = [(256, 384, 256, None, None), (300, 200, 96, 112, 96), (200, 100, 320, 336, 352),
          (128, 577, 160, 176, 160), (640, 1000, 1024, None, 1040), (129, 577, 160, 176, 160),
          (16, 1000, 512, None, None), (33, 600, 192, None, None), (64, 577, 160, 176, 160),
          (40, 100, 256, None, None)]


def _ids(s):
    return "x".join(map(str, s[:3]))


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_mx_integer_bit_exact(h, shape, out_dtype):
    M, N, K, lda, ldb = shape
    A, SA, Bt, SB = make_mx_inputs(M, N, K, seed=M + N + K, integer=True, lda=lda, ldb=ldb)
    g = torch.Generator().manual_seed(K)
    C = torch.zeros((M, round8(N)), dtype=out_dtype)[:, :N]  # row stride a multiple of 16 bytes
    C.copy_(torch.randint(-4, 5, (M, N), generator=g))
    D, base = _run_mx(h, A, SA, Bt, SB, _strided_to_device(C), 2.0, -1.0, out_dtype, ldd=round8(N) + 8)
    assert_bit_exact(bits(D), _want(A, SA, Bt, SB, C, 2.0, -1.0, out_dtype), f"{shape} {out_dtype}")
    sentinel = alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]
    b = bits(base).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(sentinel).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]), "row-stride padding of D was written"
    assert np.array_equal(b[M:], s[M:]), "rows below D were written"


@pytest.mark.parametrize("fmts", [(1, 1), (0, 1), (1, 0)], ids=["e5m2", "e4m3xe5m2", "e5m2xe4m3"])
def test_mx_formats_integer_bit_exact(h, fmts):
    M, N, K = 256, 448, 512
    A, SA, Bt, SB = make_mx_inputs(M, N, K, seed=40 + fmts[0] * 2 + fmts[1], integer=True, fmt_a=fmts[0],
                                   fmt_b=fmts[1])
    D, _ = _run_mx(h, A, SA, Bt, SB, None, 1.0, 0.0, torch.float32, *fmts)
    assert_bit_exact(bits(D), _want(A, SA, Bt, SB, None, 1.0, 0.0, torch.float32, *fmts), f"formats {fmts}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_mx_random_within_tolerance_and_deterministic(h, out_dtype):
    M, N, K = 1000, 1000, 2048
    A, SA, Bt, SB = make_mx_inputs(M, N, K, seed=7)
    C = torch.randn(M, N, generator=torch.Generator().manual_seed(8)).to(out_dtype)
    D, _ = _run_mx(h, A, SA, Bt, SB, C, 0.5, 1.0, out_dtype)
    got = bits(D)
    assert_within_tolerance(got, _want(A, SA, Bt, SB, C, 0.5, 1.0, out_dtype), out_dtype, "mx random")
    D2, _ = _run_mx(h, A, SA, Bt, SB, C, 0.5, 1.0, out_dtype)
    assert np.array_equal(got.view(np.uint8), bits(D2).view(np.uint8)), "run-to-run difference"


@pytest.mark.parametrize("name", list(MX_CONFIGS))
def test_mx_workloads_every_element(h, name):
    """The benchmarked MXFP8 shapes at full size, every element: integer
    inputs bit for bit, random inputs within the bf16 tolerance."""
    cfg = MX_CONFIGS[name]
    A, SA, Bt, SB = make_mx_inputs(cfg.M, cfg.N, cfg.K, seed=cfg.seed, integer=True)
    D, _ = _run_mx(h, A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16)
    assert_bit_exact(bits(D), _want(A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16), f"{name} integer")
    del D
    A, SA, Bt, SB = make_mx_inputs(cfg.M, cfg.N, cfg.K, seed=cfg.seed)
    D, _ = _run_mx(h, A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16)
    assert_within_tolerance(bits(D), _want(A, SA, Bt, SB, None, 1.0, 0.0, torch.bfloat16), torch.bfloat16,
                            f"{name} random")


def test_mx_in_place_and_k_zero(h):
    M, N, K = 300, 400, 256
    A, SA, Bt, SB = make_mx_inputs(M, N, K, seed=3, integer=True)
    C = torch.randint(-4, 5, (M, N), generator=torch.Generator().manual_seed(3)).to(torch.float32)
    want = _want(A, SA, Bt, SB, C, 1.0, 1.0, torch.float32)
    Cd = C.to(DEV)
    _run_mx(h, A, SA, Bt, SB, Cd, 1.0, 1.0, torch.float32, D=Cd)
    assert_bit_exact(bits(Cd), want, "in place")
    # K == 0: D = beta * C
    D = torch.full((M, N), float("nan"), device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    Cd = C.to(DEV)
    assert tpd.gemm_run_mx(h, M, N, 0, None, 0, 0, None, None, 0, 0, None, Cd.data_ptr(), N, D.data_ptr(), N, 1.0,
                           -2.0, tpd.OUT_F32, s) == tpd.OK
    torch.cuda.synchronize()
    assert torch.equal(D.cpu(), -2.0 * C)


def test_mx_argument_errors(h):
    s = torch.cuda.current_stream().cuda_stream
    A = torch.zeros((128, 256), dtype=torch.uint8, device=DEV)
    B = torch.zeros((128, 256), dtype=torch.uint8, device=DEV)
    S = torch.zeros(tpd.gemm_mx_scale_bytes(128, 256), dtype=torch.uint8, device=DEV)
    D = torch.zeros((128, 128), dtype=torch.float32, device=DEV)
    args = dict(M=128, N=128, K=256)

    def run(**kw):
        a = dict(A=A.data_ptr(), lda=256, fa=0, SA=S.data_ptr(), B=B.data_ptr(), ldb=256, fb=0, SB=S.data_ptr(),
                 D=D.data_ptr(), ldd=128, **args)
        a.update(kw)
        return tpd.gemm_run_mx(h, a["M"], a["N"], a["K"], a["A"], a["lda"], a["fa"], a["SA"], a["B"], a["ldb"],
                               a["fb"], a["SB"], None, a["N"], a["D"], a["ldd"], 1.0, 0.0, tpd.OUT_F32, s)

    assert run() == tpd.OK
    assert run(K=100) == tpd.ERR_INVALID_ARG          # K not a multiple of 32
    assert run(fa=2) == tpd.ERR_INVALID_ARG           # unknown element format
    assert run(lda=200) == tpd.ERR_INVALID_ARG        # lda < K
    assert run(lda=264) == tpd.ERR_ALIGNMENT          # row stride not a multiple of 16 bytes
    assert run(SA=S.data_ptr() + 8) == tpd.ERR_ALIGNMENT
    assert run(D=S.data_ptr()) == tpd.ERR_OVERLAP     # D on top of the scales
    torch.cuda.synchronize()
    assert tpd.gemm_sync_status(h, s) == tpd.OK


def test_mx_plan(h):
    sms = tpd.gemm_num_sms(h)
    p = tpd.gemm_mx_query_plan(h, 8192, 6144, 4096)
    assert p["tile_m"] == 256 and p["tile_n"] == 256 and p["num_tiles"] == 32 * 24 and p["cluster"] == 2
    assert p["grid"] % 2 == 0 and sms - 8 <= p["grid"] <= sms
    p = tpd.gemm_mx_query_plan(h, 16, 28672, 4096)  # 128 rows or fewer: single CTAs
    assert p["tile_m"] == 128 and p["tile_n"] == 192 and p["cluster"] == 1 and p["num_tiles"] == 150
    sizes = {p["smem_bytes"]}
    for m in (64, 100):  # 64-row A boxes, then 128-row ones: each its own ring
        p = tpd.gemm_mx_query_plan(h, m, 28672, 4096)
        assert p["tile_m"] == 128 and p["cluster"] == 1 and p["smem_bytes"] not in sizes
        sizes.add(p["smem_bytes"])
    p = tpd.gemm_mx_query_plan(h, 256, 128, 4096)
    assert p["tile_m"] == 128 and p["tile_n"] == 128 and p["num_tiles"] == 2 and p["grid"] == 2


def test_mx_graph_replay_and_two_streams(h):
    """gemm_run_mx allocates nothing and keeps no per-call state in the
    handle: a captured call replays with new inputs, and calls on two streams
    may run at the same time."""
    M, N, K = 384, 640, 512
    Ad = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    Bd = torch.empty((N, K), dtype=torch.uint8, device=DEV)
    SAd = torch.empty(tpd.gemm_mx_scale_bytes(M, K), dtype=torch.uint8, device=DEV)
    SBd = torch.empty(tpd.gemm_mx_scale_bytes(N, K), dtype=torch.uint8, device=DEV)
    D = torch.empty((M, N), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            st = tpd.gemm_run_mx(h, M, N, K, Ad.data_ptr(), K, 0, SAd.data_ptr(), Bd.data_ptr(), K, 0, SBd.data_ptr(),
                                 None, N, D.data_ptr(), N, 1.0, 0.0, tpd.OUT_F32,
                                 torch.cuda.current_stream().cuda_stream)
            assert st == tpd.OK
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for rep in range(3):
        A, SA, Bt, SB = make_mx_inputs(M, N, K, seed=300 + rep, integer=True)
        Ad.copy_(A)
        Bd.copy_(Bt)
        SAd.copy_(torch.from_numpy(mx_blocked(SA.numpy())))
        SBd.copy_(torch.from_numpy(mx_blocked(SB.numpy())))
        graph.replay()
        torch.cuda.synchronize()
        assert tpd.gemm_sync_status(h, None) == tpd.OK
        assert_bit_exact(bits(D), _want(A, SA, Bt, SB, None, 1.0, 0.0, torch.float32), f"replay {rep}")
    del graph
    # two streams at once, each with its own inputs and output
    jobs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for i, s in enumerate(streams):
        A, SA, Bt, SB = make_mx_inputs(M, N, K, seed=400 + i, integer=True)
        ins = [A.to(DEV), Bt.to(DEV), torch.from_numpy(mx_blocked(SA.numpy())).to(DEV),
               torch.from_numpy(mx_blocked(SB.numpy())).to(DEV)]
        out = torch.empty((M, N), dtype=torch.float32, device=DEV)
        jobs.append((A, SA, Bt, SB, ins, out, s))
    torch.cuda.synchronize()
    for A, SA, Bt, SB, ins, out, s in jobs:
        st = tpd.gemm_run_mx(h, M, N, K, ins[0].data_ptr(), K, 0, ins[2].data_ptr(), ins[1].data_ptr(), K, 0,
                             ins[3].data_ptr(), None, N, out.data_ptr(), N, 1.0, 0.0, tpd.OUT_F32, s.cuda_stream)
        assert st == tpd.OK
    torch.cuda.synchronize()
    for A, SA, Bt, SB, ins, out, s in jobs:
        assert_bit_exact(bits(out), _want(A, SA, Bt, SB, None, 1.0, 0.0, torch.float32), "two streams")
