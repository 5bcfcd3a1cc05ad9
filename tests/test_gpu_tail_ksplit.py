"""The K split of the CTA-pair kernel's last partial round (gemm_set_workspace).

The tiles left over after the whole rounds are cut into two pieces. With a
workspace attached and K of at least 32 blocks, piece p accumulates K blocks
[p*kb/2, (p+1)*kb/2) over the tile's full width and owns column half p; the
two pairs of a tile trade their fp32 partial sums of each other's half
through the workspace, and each adds the other's part before its epilogue
(the sum of two fp32 parts does not depend on their order). Every output element keeps one writer ("cuTile Rust explained",
"Ownership crosses the launch boundary"). Integer inputs are compared with
the oracle bit for bit, random inputs within the stated tolerances, and the
flags are checked across back-to-back calls and replays of a captured graph
whose inputs change between replays.
"""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import (DEV, alloc_out, assert_bit_exact, assert_within_tolerance, bits, oracle_out, out_code, round8, run,
                  to_device)
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ws():
    h = tpd.gemm_create(0)
    nbytes = tpd.gemm_workspace_size(h)
    assert nbytes > 0
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=DEV)
    ptr = (buf.data_ptr() + 255) // 256 * 256
    s = torch.cuda.current_stream().cuda_stream
    assert tpd.gemm_set_workspace(h, ptr, nbytes, s) == tpd.OK
    yield h, buf, ptr, nbytes
    tpd.gemm_set_workspace(h, None, 0, None)
    torch.cuda.synchronize()
    tpd.gemm_destroy(h)


@pytest.fixture(scope="module")
def plain():
    h = tpd.gemm_create(0)
    yield h
    tpd.gemm_destroy(h)


def _full_size_gpu(h):
    return tpd.gemm_num_sms(h) >= 148


# (M, N, K) in CTA-pair mode with a tail on a 152-SM GB300 (76 pairs):
#  - 80 pair tiles leave 4;
#  - the same with ragged M, N and K: N = 1800 ends 8 columns into the last
#    tile column, so the second piece of those tiles owns no stored column,
#    and 33 K blocks make parts of 16 and 17;
#  - 65 K blocks (32 and 33);
#  - 176 tiles leave 24, and the same with 33 K blocks and ragged N;
#  - the square 4096^3 workload (28 left over).
SHAPES = [(2560, 2048, 2048, 1), (2500, 1800, 2100, 1), (2560, 2048, 4160, 1), (2816, 4096, 2048, 1),
          (2800, 4000, 2112, 1), (4096, 4096, 4096, 1)]


def _ids(s):
    return "x".join(map(str, s[:3]))


def _int_inputs(M, N, K, out_dtype, seed):
    A, B, C = make_inputs(CONFIGS["mlp_down"], integer=True, M=M, N=N, K=K, lda=round8(K), ldb=round8(N),
                          ldc=round8(N), c_for_beta=True, seed=seed)
    Cp = torch.empty((M, round8(N)), dtype=out_dtype)[:, :N]
    Cp.copy_(C)
    return A, B, Cp


def test_plan_uses_the_tail_split_only_with_a_workspace(ws, plain):
    h = ws[0]
    if not _full_size_gpu(h):
        pytest.skip("tile counts assume a full GB300")
    for M, N, K, pieces in SHAPES:
        assert tpd.gemm_plan_tail_ksplit(h, M, N, K, tpd.OUT_BF16) == pieces, (M, N, K)
        assert tpd.gemm_plan_tail_ksplit(plain, M, N, K, tpd.OUT_BF16) == 0, (M, N, K)
    # qkv: 768 tiles leave 8; mlp_down: 512 leave 56, too many to cut
    assert tpd.gemm_plan_tail_ksplit(h, 8192, 6144, 4096, tpd.OUT_BF16) == 1
    assert tpd.gemm_plan_tail_ksplit(h, 8192, 4096, 14336, tpd.OUT_BF16) == 0
    # fewer than 32 K blocks: the exchange would cost more than it saves
    assert tpd.gemm_plan_tail_ksplit(h, 2560, 2048, 1984, tpd.OUT_BF16) == 0
    assert tpd.gemm_plan_tail_ksplit(h, 2560, 2048, 64, tpd.OUT_BF16) == 0
    # small M goes to other kernels
    assert tpd.gemm_plan_tail_ksplit(h, 16, 28672, 4096, tpd.OUT_BF16) == 0


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_tail_ksplit_integer_bit_exact(ws, shape, out_dtype):
    h = ws[0]
    M, N, K, _ = shape
    if (M, N, K) == (4096, 4096, 4096) and out_dtype == torch.float32:
        pytest.skip("the bf16 case covers the full-size shape")
    A, B, C = _int_inputs(M, N, K, out_dtype, seed=M + 5 * N + 3 * K)
    D, base = run(h, A, B, C, 2.0, -1.0, out_dtype, ldd=round8(N) + 8)
    assert_bit_exact(bits(D), oracle_out(A, B, C, 2.0, -1.0, out_dtype), f"{shape} {out_dtype}")
    sentinel = alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]
    b = bits(base).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(sentinel).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]), "row-stride padding of D was written"
    assert np.array_equal(b[M:], s[M:]), "rows below D were written"


@pytest.mark.parametrize("shape", [(2560, 2048, 2048), (2816, 4096, 2048)], ids=lambda s: "x".join(map(str, s)))
def test_tail_ksplit_matches_column_halves_on_integers(ws, plain, shape):
    M, N, K = shape
    A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, seed=77)
    Ad, Bd = to_device(A), to_device(B)
    split = bits(run(ws[0], Ad, Bd, None, 1.0, 0.0, torch.bfloat16)[0])
    halves = bits(run(plain, Ad, Bd, None, 1.0, 0.0, torch.bfloat16)[0])
    assert np.array_equal(split, halves)


@pytest.mark.parametrize("shape", [(2500, 1800, 2100), (2800, 4000, 2112)], ids=lambda s: "x".join(map(str, s)))
def test_tail_ksplit_in_place(ws, shape):
    M, N, K = shape
    out_dtype = torch.float32
    A, B, C = _int_inputs(M, N, K, out_dtype, seed=9)
    want = oracle_out(A, B, C, 1.0, 1.0, out_dtype)
    Cd = to_device(C)
    run(ws[0], A, B, Cd, 1.0, 1.0, out_dtype, D=Cd)
    assert_bit_exact(bits(Cd), want, "in place")


@pytest.mark.parametrize("shape", [(2560, 2048, 2048), (4096, 4096, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_tail_ksplit_random_deterministic(ws, shape):
    """Two parts add to the same fp32 value in either order, so the result is
    the same on every run."""
    M, N, K = shape
    A, B, C = make_inputs(CONFIGS["square"], M=M, N=N, K=K, seed=13, c_for_beta=True)
    C = C.to(torch.float32)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    outs = [bits(run(ws[0], Ad, Bd, Cd, 1.0, 0.5, torch.float32)[0]) for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32)), "run-to-run difference"
    rows = np.arange(M) if M <= 2560 else np.concatenate([np.arange(0, M, 7), np.arange(M - 300, M)])
    rows = np.unique(rows)
    want = oracle_out(A, B, C, 1.0, 0.5, torch.float32, rows=rows)
    assert_within_tolerance(outs[0][rows], want, torch.float32, str(shape))


@pytest.mark.parametrize("act", [tpd.ACT_RELU, tpd.ACT_TANH], ids=["relu", "tanh"])
def test_tail_ksplit_fused_epilogue(ws, act):
    h = ws[0]
    M, N, K = 2560, 2048, 2048
    assert tpd.gemm_plan_tail_ksplit(h, M, N, K, tpd.OUT_F32) == int(_full_size_gpu(h))
    g = torch.Generator().manual_seed(31)
    A = torch.randint(-4, 5, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16)
    bias = torch.randint(-64, 65, (N,), generator=g).to(torch.float32)
    aux = torch.randint(-2, 3, (M, N), generator=g).to(torch.float32)
    Ad, Bd, bd, Xd = to_device(A), to_device(B), bias.cuda(), to_device(aux)
    D, _ = alloc_out(M, N, torch.float32)
    epi = tpd.Epilogue(bd.data_ptr(), tpd.OUT_F32, act, Xd.data_ptr(), Xd.stride(0))
    s = torch.cuda.current_stream().cuda_stream
    st = tpd.gemm_run_epilogue(h, M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), None, N,
                               D.data_ptr(), D.stride(0), 1.0, 0.0, tpd.OUT_F32, epi, s)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    want, _ = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_F32, bias=bias, act=act, aux=aux)
    if act == tpd.ACT_RELU:
        assert_bit_exact(bits(D), want, "tail K split + bias + relu + aux")
    else:
        assert_within_tolerance(bits(D), want, torch.float32, "tail K split + bias + tanh + aux")


def test_back_to_back_calls_share_the_workspace(ws):
    """Calls of different shapes in a row on one stream, with no host
    synchronisation between them, each read only their own partial sums."""
    h = ws[0]
    shapes = [(2560, 2048, 2048), (2800, 4000, 2112), (2500, 1800, 2100), (2560, 2048, 2048)]
    s = torch.cuda.current_stream().cuda_stream
    jobs = []
    for i, (M, N, K) in enumerate(shapes):
        A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, lda=round8(K), ldb=round8(N),
                              seed=100 + i)
        Ad, Bd = to_device(A), to_device(B)
        D, _ = alloc_out(M, N, torch.bfloat16)
        st = tpd.gemm_run(h, M, N, K, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(), Bd.stride(0), None, N,
                          D.data_ptr(), D.stride(0), 1.0, 0.0, tpd.OUT_BF16, s)
        assert st == tpd.OK
        jobs.append((A, B, Ad, Bd, D))
    assert tpd.gemm_sync_status(h, s) == tpd.OK
    for A, B, _, _, D in jobs:
        assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16), "back to back")


def test_graph_replays_with_new_inputs(ws):
    """A captured call replayed three times, its inputs overwritten between
    replays: a flag left set by one replay would let the next read stale
    partial sums, and the output would no longer match its inputs."""
    h = ws[0]
    M, N, K = 2560, 2048, 2048
    Ad = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    Bd = torch.empty((K, N), dtype=torch.bfloat16, device=DEV)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            st = tpd.gemm_run(h, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 0.0,
                              tpd.OUT_BF16, torch.cuda.current_stream().cuda_stream)
            assert st == tpd.OK
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for rep in range(3):
        A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, seed=200 + rep)
        Ad.copy_(A)
        Bd.copy_(B)
        graph.replay()
        torch.cuda.synchronize()
        assert tpd.gemm_sync_status(h, None) == tpd.OK
        assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16), f"replay {rep}")
    del graph


def test_workspace_argument_errors(ws):
    h, buf, ptr, nbytes = ws
    assert tpd.gemm_set_workspace(h, ptr + 16, nbytes - 256, None) == tpd.ERR_ALIGNMENT
    assert tpd.gemm_set_workspace(h, ptr, 1024, None) == tpd.ERR_INVALID_ARG
    # the rejected calls left the attached workspace in place
    assert tpd.gemm_plan_tail_ksplit(h, 2560, 2048, 2048, tpd.OUT_BF16) == int(_full_size_gpu(h))


def test_operand_overlapping_the_workspace_is_rejected():
    """D placed on the workspace: the call is refused before anything runs
    (the buffer holds both, so even a launch would stay in bounds)."""
    h = tpd.gemm_create(0)
    try:
        if not _full_size_gpu(h):
            pytest.skip("tile counts assume a full GB300")
        M, N, K = 2560, 2048, 2048
        big = torch.zeros(M * N * 2 + tpd.gemm_workspace_size(h) + 256, dtype=torch.uint8, device=DEV)
        ptr = (big.data_ptr() + 255) // 256 * 256
        assert tpd.gemm_set_workspace(h, ptr, tpd.gemm_workspace_size(h), None) == tpd.OK
        assert tpd.gemm_plan_tail_ksplit(h, M, N, K, tpd.OUT_BF16) == 1
        Ad = torch.zeros((M, K), dtype=torch.bfloat16, device=DEV)
        Bd = torch.zeros((K, N), dtype=torch.bfloat16, device=DEV)
        st = tpd.gemm_run(h, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, ptr, N, 1.0, 0.0,
                          tpd.OUT_BF16, torch.cuda.current_stream().cuda_stream)
        assert st == tpd.ERR_OVERLAP
        assert tpd.gemm_set_workspace(h, None, 0, None) == tpd.OK
        torch.cuda.synchronize()
    finally:
        tpd.gemm_destroy(h)


def test_small_workspace_falls_back():
    """A workspace too small for a shape's tail leaves that shape on column
    halves (still exact); shapes whose tail fits use it."""
    h = tpd.gemm_create(0)
    try:
        small = 4096 + 4 * 4 * 128 * 128 * 4  # flags + four tail tiles
        buf = torch.empty(small + 256, dtype=torch.uint8, device=DEV)
        ptr = (buf.data_ptr() + 255) // 256 * 256
        assert tpd.gemm_set_workspace(h, ptr, small, None) == tpd.OK
        if _full_size_gpu(h):
            assert tpd.gemm_plan_tail_ksplit(h, 2560, 2048, 2048, tpd.OUT_BF16) == 1  # 4 tail tiles
            assert tpd.gemm_plan_tail_ksplit(h, 4096, 4096, 2048, tpd.OUT_BF16) == 0  # 28
        M, N, K = 2560, 2048, 2048
        A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, seed=4)
        D, _ = run(h, A, B, None, 1.0, 0.0, torch.bfloat16)
        assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16), "tail split")
        M, N, K = 4096, 4096, 2048
        A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, seed=3)
        D, _ = run(h, A, B, None, 1.0, 0.0, torch.bfloat16)
        assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16), "fallback")
        assert tpd.gemm_set_workspace(h, None, 0, None) == tpd.OK
        assert tpd.gemm_plan_tail_ksplit(h, 2560, 2048, 2048, tpd.OUT_BF16) == 0
        torch.cuda.synchronize()
    finally:
        tpd.gemm_destroy(h)


def test_gemm_object_with_a_workspace():
    """The torch convenience class attaches its own workspace when asked, uses
    the K split tail, and detaches it on close."""
    g = tpd.Gemm(0, workspace=True)
    try:
        M, N, K = 2560, 2048, 2048
        if _full_size_gpu(g.handle):
            assert tpd.gemm_plan_tail_ksplit(g.handle, M, N, K, tpd.OUT_BF16) == 1
        A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, seed=61)
        D = g(to_device(A), to_device(B), out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert tpd.gemm_sync_status(g.handle, None) == tpd.OK
        assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16), "Gemm(workspace=True)")
    finally:
        g.close()
    assert g.handle is None
