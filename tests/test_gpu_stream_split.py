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


# (M, N, K): on a 152-SM GB300 these plan K splits of 4 (32 panels), 3 (48
# panels), 2 (224 panels) and 1 (a single K block); a ragged K (65 blocks);
# 48 and 64 token rows, whose reduction slots leave room for smaller splits.
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
