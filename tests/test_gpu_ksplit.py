"""The tiled kernel's K split: when an output has few 128 x 256 tiles (a short M
with a narrow N), the 2 or 4 CTAs of a cluster share each tile's K range. Each
CTA owns a quarter (or half) of the tile's columns: the others hand it their
fp32 partial sums of those columns through distributed shared memory, and it
adds them in rank order (part 0 + part 1 + ...) before the epilogue, so every
output element has one writer and the result is the same on every run
("cuTile Rust explained", "Ownership crosses the launch boundary"). Integer
inputs are compared with the oracle bit for bit; random inputs within the
stated tolerances."""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import alloc_out, assert_bit_exact, assert_within_tolerance, bits, oracle_out, out_code, round8, run, \
    to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


# (M, N, K, K split on a 152-SM GB300): 4, with ragged M, N and K and with 5 K
# blocks in 4 unequal parts; a single-column output (three of four CTAs own no
# stored column); 2 for 64 tiles, and for 3 K blocks; 4 for a prefill-sized
# 256 x 4096 x 4096.
SHAPES = [(257, 1000, 255, 4), (384, 768, 320, 4), (1000, 1, 257, 4), (129, 264, 4096, 4), (520, 600, 2048, 4),
          (512, 4096, 256, 2), (256, 4096, 4096, 4), (65, 2000, 130, 2)]


def _ids(s):
    return "x".join(map(str, s[:3]))


def _plan(h, M, N, K, out_dtype):
    p = tpd.gemm_query_plan(h, M, N, K, out_code(out_dtype))
    assert p["variant"] == tpd.VARIANT_TILED, p
    return p


@pytest.mark.parametrize("shape", SHAPES, ids=_ids)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_ksplit_integer_bit_exact(h, shape, out_dtype):
    M, N, K, ks = shape
    p = _plan(h, M, N, K, out_dtype)
    if tpd.gemm_num_sms(h) >= 148:
        assert p["cluster"] == ks, p
    A, B, C = make_inputs(CONFIGS["mlp_down"], integer=True, M=M, N=N, K=K, lda=round8(K), ldb=round8(N),
                          ldc=round8(N), c_for_beta=True, seed=M + 3 * N + 7 * K)
    # keep C's padded row stride through the dtype change
    Cp = torch.empty((M, round8(N)), dtype=out_dtype)[:, :N]
    Cp.copy_(C)
    C = Cp
    D, base = run(h, A, B, C, 2.0, -1.0, out_dtype, ldd=round8(N) + 8)
    assert_bit_exact(bits(D), oracle_out(A, B, C, 2.0, -1.0, out_dtype), f"{shape} {out_dtype}")
    # nothing outside the M x N view was written
    sentinel = alloc_out(M, N, out_dtype, ldd=round8(N) + 8)[1]
    b = bits(base).view(np.uint16 if out_dtype == torch.bfloat16 else np.uint32)
    s = bits(sentinel).view(b.dtype)
    assert np.array_equal(b[:M, N:], s[:M, N:]), "row-stride padding of D was written"
    assert np.array_equal(b[M:], s[M:]), "rows below D were written"


@pytest.mark.parametrize("shape", [(256, 4096, 4096), (512, 4096, 1024), (300, 520, 1000)], ids=lambda s: "x".join(map(str, s)))
def test_ksplit_random_deterministic(h, shape):
    M, N, K = shape
    assert _plan(h, M, N, K, torch.float32)["cluster"] > 1
    A, B, C = make_inputs(CONFIGS["mlp_down"], M=M, N=N, K=K, seed=5)
    C = C.to(torch.float32)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    outs = [bits(run(h, Ad, Bd, Cd, 1.0, 1.0, torch.float32)[0]) for _ in range(3)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32)), "run-to-run difference"
    assert_within_tolerance(outs[0], oracle_out(A, B, C, 1.0, 1.0, torch.float32), torch.float32, str(shape))


@pytest.mark.parametrize("act", [tpd.ACT_RELU, tpd.ACT_SIGMOID], ids=["relu", "sigmoid"])
def test_ksplit_fused_epilogue(h, act):
    """bias + activation + aux multiply on the owning CTA's columns after the
    partial sums are added."""
    M, N, K = 200, 1000, 1000
    assert _plan(h, M, N, K, torch.float32)["cluster"] > 1
    g = torch.Generator().manual_seed(29)
    A = torch.randint(-4, 5, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16)
    bias = torch.randint(-64, 65, (N,), generator=g).to(torch.float32)
    aux = torch.randint(-2, 3, (M, round8(N)), generator=g).to(torch.float32)[:, :N]
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
        assert_bit_exact(bits(D), want, "K split + bias + relu + aux")
    else:
        assert_within_tolerance(bits(D), want, torch.float32, "K split + bias + sigmoid + aux")


def test_ksplit_matches_unsplit_on_integers(h):
    """The same integer GEMM through the K split and through the forced
    unsplit 1-CTA path gives the same bits."""
    M, N, K = 256, 2048, 2048
    assert _plan(h, M, N, K, torch.bfloat16)["cluster"] > 1
    A, B, _ = make_inputs(CONFIGS["square"], integer=True, M=M, N=N, K=K, seed=41)
    Ad, Bd = to_device(A), to_device(B)
    split = bits(run(h, Ad, Bd, None, 1.0, 0.0, torch.bfloat16)[0])
    assert tpd.gemm_force_variant(h, tpd.VARIANT_TILED) == tpd.OK
    try:
        assert tpd.gemm_query_plan(h, M, N, K, tpd.OUT_BF16)["cluster"] == 1
        plain = bits(run(h, Ad, Bd, None, 1.0, 0.0, torch.bfloat16)[0])
    finally:
        tpd.gemm_force_variant(h, tpd.VARIANT_AUTO)
    assert np.array_equal(split, plain)
