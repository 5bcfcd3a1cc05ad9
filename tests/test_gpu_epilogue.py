"""GPU parity of the fused epilogue (bias, ReLU/sigmoid/tanh, aux multiply)
against the oracle, in every kernel that runs it: the tiled kernel in 1-CTA
and CTA-pair mode, the streaming kernel (M <= 64) and the K == 0 kernel.
The epilogue is the EFC list of the epilogue-fusion roadmap paragraph of
"TorchInductor ganha suporte a GEMMs de alta performance com CuteDSL"."""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import alloc_out, assert_bit_exact, assert_within_tolerance, bits, out_code, round8, to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu

ACTS = [tpd.ACT_NONE, tpd.ACT_RELU, tpd.ACT_SIGMOID, tpd.ACT_TANH]
ACT_IDS = ["none", "relu", "sigmoid", "tanh"]


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


def _run(h, A, B, C, alpha, beta, out_dtype, bias, act, aux, variant=tpd.VARIANT_AUTO, ldd=None):
    M, K = A.shape
    N = B.shape[1]
    Ad, Bd, Cd, Xd = to_device(A), to_device(B), to_device(C), to_device(aux)
    bd = bias.to("cuda") if bias is not None else None
    D, base = alloc_out(M, N, out_dtype, ldd)
    epi = tpd.Epilogue(bd.data_ptr() if bd is not None else None,
                       tpd.OUT_F32 if (bd is not None and bd.dtype == torch.float32) else tpd.OUT_BF16,
                       act, Xd.data_ptr() if Xd is not None else None,
                       Xd.stride(0) if Xd is not None else round8(N))
    assert tpd.gemm_force_variant(h, variant) == tpd.OK
    try:
        s = torch.cuda.current_stream().cuda_stream
        st = tpd.gemm_run_epilogue(h, M, N, K, Ad.data_ptr() if K else None, Ad.stride(0) if K else K,
                                   Bd.data_ptr() if K else None, Bd.stride(0) if K else round8(N),
                                   Cd.data_ptr() if Cd is not None else None, Cd.stride(0) if Cd is not None else N,
                                   D.data_ptr(), D.stride(0), alpha, beta, out_code(out_dtype), epi, s)
        assert st == tpd.OK, tpd.gemm_status_string(st)
        assert tpd.gemm_sync_status(h, s) == tpd.OK
    finally:
        tpd.gemm_force_variant(h, tpd.VARIANT_AUTO)
    return D, base


def _want(A, B, C, alpha, beta, out_dtype, bias, act, aux):
    D, _ = oracle.gemm_rows_epilogue(A, B, C, alpha, beta, out_code(out_dtype), bias=bias, act=act, aux=aux)
    return D


SHAPES = [(300, 520, 1000, tpd.VARIANT_AUTO), (100, 264, 512, tpd.VARIANT_AUTO), (16, 1000, 2048, tpd.VARIANT_AUTO),
          (40, 776, 320, tpd.VARIANT_TILED), (257, 300, 64, tpd.VARIANT_TILED_PAIR)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:3])) + f"-v{s[3]}")
@pytest.mark.parametrize("act", ACTS, ids=ACT_IDS)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_random_within_tolerance(h, shape, act, out_dtype):
    M, N, K, variant = shape
    A, B, C = make_inputs(CONFIGS["mlp_down"], M=M, N=N, K=K, lda=round8(K), ldb=round8(N), ldc=round8(N),
                          seed=M + K + act)
    g = torch.Generator().manual_seed(N + act)
    bias = torch.randn(N, generator=g) * 0.5
    bias = bias.to(torch.bfloat16) if act % 2 else bias  # both bias dtypes
    aux_base = torch.full((M, round8(N)), float("nan"))
    aux_base[:, :N] = torch.rand(M, N, generator=g) * 2 - 0.5
    aux = _cast_keep_stride(aux_base[:, :N], out_dtype)
    if out_dtype == torch.float32:
        C = C.to(torch.float32)
    D, _ = _run(h, A, B, C, 1.0, 0.5, out_dtype, bias, act, aux, variant)
    assert_within_tolerance(bits(D), _want(A, B, C, 1.0, 0.5, out_dtype, bias, act, aux), out_dtype,
                            f"{shape} act {act}")


@pytest.mark.parametrize("shape", [(300, 523, 200, tpd.VARIANT_AUTO), (130, 517, 72, tpd.VARIANT_TILED),
                                   (48, 301, 128, tpd.VARIANT_AUTO), (260, 7, 64, tpd.VARIANT_TILED_PAIR)],
                         ids=lambda s: "x".join(map(str, s[:3])) + f"-v{s[3]}")
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("bias_dtype", [torch.bfloat16, torch.float32], ids=["bbf16", "bf32"])
def test_integer_relu_bias_aux_bit_exact(h, shape, out_dtype, bias_dtype):
    """Integer inputs, bias and aux: relu(acc + C + bias) * aux is an exact
    integer, so the result is unique, including the ragged last columns."""
    M, N, K, variant = shape
    A, B, C = make_inputs(CONFIGS["tiny"], integer=True, M=M, N=N, K=K, lda=round8(K), ldb=round8(N) + 8,
                          ldc=round8(N), c_for_beta=True, seed=N)
    C = _cast_keep_stride(C, out_dtype)
    g = torch.Generator().manual_seed(M)
    bias = torch.randint(-6, 7, (N,), generator=g).to(bias_dtype)
    base = torch.full((M, round8(N) + 16), float("nan"))
    aux = base[:, :N]
    aux[:] = torch.randint(-2, 3, (M, N), generator=g).to(torch.float32)
    aux = _cast_keep_stride(aux, out_dtype)
    D, dbase = _run(h, A, B, C, 1.0, -1.0, out_dtype, bias, tpd.ACT_RELU, aux, variant, ldd=round8(N) + 8)
    assert_bit_exact(bits(D), _want(A, B, C, 1.0, -1.0, out_dtype, bias, tpd.ACT_RELU, aux), f"{shape}")
    b = bits(dbase).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]) and np.array_equal(b[M:], s[M:])


def _cast_keep_stride(t, dtype):
    rows, cols = t.shape
    if rows <= 1 or t.stride(0) == cols:
        return t.to(dtype)
    base = torch.as_strided(t, (rows, t.stride(0)), (t.stride(0), 1))
    return base.to(dtype)[:, :cols]


def test_k_zero_with_epilogue(h):
    M, N = 70, 264
    C = torch.randint(-4, 5, (M, N)).to(torch.float32)
    bias = torch.randint(-3, 4, (N,)).to(torch.float32)
    aux = torch.randint(-2, 3, (M, N)).to(torch.float32)
    A = torch.zeros((M, 0), dtype=torch.bfloat16)
    B = torch.zeros((0, N), dtype=torch.bfloat16)
    D, _ = _run(h, A, B, C, 1.0, 2.0, torch.float32, bias, tpd.ACT_RELU, aux)
    want = (torch.clamp(2.0 * C + bias[None, :], min=0) * aux).numpy()
    assert_bit_exact(bits(D), want.astype(np.float32), "K=0 epilogue")


def test_in_place_aux_equals_d(h):
    M, N, K = 256, 512, 128
    A, B, _ = make_inputs(CONFIGS["tiny"], integer=True, M=M, N=N, K=K)
    Ad, Bd = to_device(A), to_device(B)
    D = torch.randint(-2, 3, (M, N)).to(torch.float32).cuda()
    aux_cpu = D.cpu().clone()
    epi = tpd.Epilogue(None, tpd.OUT_F32, tpd.ACT_NONE, D.data_ptr(), N)
    st = tpd.gemm_run_epilogue(h, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 0.0,
                               tpd.OUT_F32, epi, torch.cuda.current_stream().cuda_stream)
    assert st == tpd.OK and tpd.gemm_sync_status(h, None) == tpd.OK
    want = _want(A, B, None, 1.0, 0.0, torch.float32, None, tpd.ACT_NONE, aux_cpu)
    assert_bit_exact(bits(D), want, "aux == D")


def test_epilogue_argument_errors(h):
    M = N = K = 64
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((M, N), device="cuda")
    bias = torch.zeros(N + 8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def run(epi):
        return tpd.gemm_run_epilogue(h, M, N, K, A.data_ptr(), K, B.data_ptr(), N, None, N, D.data_ptr(), N, 1.0,
                                     0.0, tpd.OUT_F32, epi, s)
    assert run(tpd.Epilogue(None, 0, 7, None, N)) == tpd.ERR_INVALID_ARG
    assert run(tpd.Epilogue(bias.data_ptr(), 5, 0, None, N)) == tpd.ERR_INVALID_ARG
    assert run(tpd.Epilogue(bias.data_ptr() + 4, tpd.OUT_F32, 0, None, N)) == tpd.ERR_ALIGNMENT
    assert run(tpd.Epilogue(D.data_ptr() + 64, tpd.OUT_F32, 0, None, N)) == tpd.ERR_OVERLAP
    assert run(tpd.Epilogue(None, 0, 0, D.data_ptr() + 16, N)) == tpd.ERR_OVERLAP
    assert run(tpd.Epilogue(None, 0, 0, bias.data_ptr(), N - 8)) == tpd.ERR_INVALID_ARG
    assert run(tpd.Epilogue(bias.data_ptr(), tpd.OUT_F32, tpd.ACT_TANH, None, N)) == tpd.OK
    assert run(None) == tpd.OK
    assert tpd.gemm_sync_status(h, None) == tpd.OK


def test_torch_convenience_matmul_with_epilogue():
    A, B, _ = make_inputs(CONFIGS["tiny"], M=192, N=256, K=128)
    bias = torch.linspace(-1, 1, 256)
    D = tpd.matmul(A.cuda(), B.cuda(), bias=bias.cuda(), activation=tpd.ACT_SIGMOID, out_dtype=torch.float32)
    torch.cuda.synchronize()
    want = _want(A, B, None, 1.0, 0.0, torch.float32, bias, tpd.ACT_SIGMOID, None)
    assert_within_tolerance(bits(D), want, torch.float32, "matmul(bias, sigmoid)")
