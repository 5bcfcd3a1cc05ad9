"""The weight-streaming (decode) variant with its K range split over 1 to 4
CTAs of a cluster ("TorchInductor ganha suporte a GEMMs de alta performance com
CuteDSL", BF16 results paragraph: decode shapes with M from 8 to 64). The
CTAs after the first hand their fp32 partials to the first through
distributed shared memory and it adds them in a fixed order, so every panel
has one writer and the result is the same on every run. Integer inputs are
compared with the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import assert_bit_exact, bits, oracle_out, out_code, round8, run, to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


# (M, N, K): on a 152-SM GB300 these plan K splits of 4 (32 panels), 2 (48
# panels: 46 clusters of 3 would leave two panels for a second round; 224
# panels) and 1 (a single K block); a ragged K (65 blocks); 48 and 64 token
# rows, whose reduction slots leave room for smaller splits (64 x 512 x 8192
# plans a split of 3).
SHAPES = [(16, 4096, 14336), (16, 6144, 4096), (16, 28672, 4096), (32, 1024, 64), (5, 2048, 4100),
          (33, 640, 1000), (64, 512, 8192), (1, 4096, 2048)]


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_stream_splits_bit_exact(h, out_dtype):
    seen = set()
    for (M, N, K) in SHAPES:
        plan = tpd.gemm_query_plan(h, M, N, K, out_code(out_dtype))
        assert plan["variant"] == tpd.VARIANT_STREAM, (M, N, K, plan)
        split = plan["cluster"]
        assert 1 <= split <= 4 and plan["grid"] % split == 0
        assert split <= (K + 63) // 64
        seen.add(split)
        A, B, C = make_inputs(CONFIGS["decode"], integer=True, M=M, N=N, K=K, lda=round8(K), ldb=round8(N),
                              ldc=round8(N), c_for_beta=True, seed=M * 7 + N)
        C = C.to(out_dtype)
        D, _ = run(h, A, B, C, 1.0, 1.0, out_dtype, ldd=round8(N) + 8)
        assert_bit_exact(bits(D), oracle_out(A, B, C, 1.0, 1.0, out_dtype), f"{(M, N, K)} split {split}")
    if tpd.gemm_num_sms(h) >= 148:
        assert seen == {1, 2, 3, 4}, seen


@pytest.mark.parametrize("shape", [(16, 4096, 14336), (16, 6144, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_stream_split_random_deterministic(h, shape):
    M, N, K = shape
    A, B, _ = make_inputs(CONFIGS["decode"], M=M, N=N, K=K, seed=3)
    Ad, Bd = to_device(A), to_device(B)
    outs = [bits(run(h, Ad, Bd, None, 1.0, 0.0, torch.float32)[0]) for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32)), "run-to-run difference"
    want = oracle_out(A, B, None, 1.0, 0.0, torch.float32)
    err = np.abs(outs[0].astype(np.float64) - want.astype(np.float64)).max() / np.abs(want).max()
    assert err <= 1e-5, err


def test_stream_split4_fused_epilogue(h):
    M, N, K = 16, 4096, 14336
    assert tpd.gemm_query_plan(h, M, N, K, tpd.OUT_F32)["variant"] == tpd.VARIANT_STREAM
    g = torch.Generator().manual_seed(17)
    A = torch.randint(-4, 5, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16)
    bias = torch.randint(-64, 65, (N,), generator=g).to(torch.float32)
    aux = torch.randint(-2, 3, (M, N), generator=g).to(torch.float32)
    Ad, Bd, biasd, auxd = A.cuda(), B.cuda(), bias.cuda(), aux.cuda()
    D = torch.full((M, N), float("nan"), device="cuda")
    epi = tpd.Epilogue(biasd.data_ptr(), tpd.OUT_F32, tpd.ACT_RELU, auxd.data_ptr(), N)
    st = tpd.gemm_run_epilogue(h, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 0.0,
                               tpd.OUT_F32, epi, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    want, _ = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_F32, bias=bias, act=oracle.ACT_RELU, aux=aux)
    assert_bit_exact(bits(D), want, "split-4 stream + fused epilogue")


def test_b_written_by_the_previous_gemm(h):
    """The streaming kernel prefetches the first B blocks of its first panel
    into L2 before it waits for the previous grid in the stream. Here B is the
    output of the GEMM launched just before it, and the two overlap through
    programmatic dependent launch, three times over with new values each time:
    every second GEMM must read what the first one wrote. Integer inputs keep
    both products exact (|B| <= 256 is exact in bf16; the sums stay below
    2^24), so the comparison with the oracle is bit for bit."""
    K1, M2, N2, K2 = 16, 16, 28672, 4096
    plan = tpd.gemm_query_plan(h, M2, N2, K2, tpd.OUT_F32)
    assert plan["variant"] == tpd.VARIANT_STREAM
    # more panels than clusters: the prefetching case
    assert plan["num_tiles"] > plan["grid"] // plan["cluster"], plan
    g = torch.Generator().manual_seed(23)
    ints = lambda *shape: torch.randint(-4, 5, shape, generator=g).to(torch.bfloat16)
    B1, A2 = ints(K1, N2), ints(M2, K2)
    A1s = [ints(K2, K1) for _ in range(3)]
    B1d, A2d = B1.cuda(), A2.cuda()
    A1ds = [a.cuda() for a in A1s]
    B2 = torch.empty((K2, N2), dtype=torch.bfloat16, device="cuda")
    outs = [torch.full((M2, N2), float("nan"), device="cuda") for _ in range(3)]
    s = torch.cuda.current_stream().cuda_stream
    for i in range(3):
        st = tpd.gemm_run(h, K2, N2, K1, A1ds[i].data_ptr(), K1, B1d.data_ptr(), N2, None, N2, B2.data_ptr(), N2,
                          1.0, 0.0, tpd.OUT_BF16, s)
        assert st == tpd.OK
        st = tpd.gemm_run(h, M2, N2, K2, A2d.data_ptr(), K2, B2.data_ptr(), N2, None, N2, outs[i].data_ptr(), N2,
                          1.0, 0.0, tpd.OUT_F32, s)
        assert st == tpd.OK
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    for i in range(3):
        b2 = torch.from_numpy(oracle_out(A1s[i], B1, None, 1.0, 0.0, torch.bfloat16).view(np.int16)).view(
            torch.bfloat16)
        want = oracle_out(A2, b2, None, 1.0, 0.0, torch.float32)
        assert_bit_exact(bits(outs[i]), want, f"chain {i}")
