"""Parity at the workloads' full sizes, on every element: tiny 256^3 (fp32
out), square 4096^3, GQA QKV projection 8192x6144x4096, MLP down-projection
8192x4096x14336 with residual C, and the decode shape 16x28672x4096.

Each workload runs under two plans and both are compared with the oracle on
all M x N outputs:
  - "plain": a handle without a workspace;
  - "bench": a handle with gemm_workspace_size bytes attached, as the
    benchmark runs it, so the CTA-pair kernel splits the last partial round
    over K where its rule says so (the QKV shape: 768 pair tiles on 76 pairs
    leave 8, cut into K halves).
Integer inputs in {-4..4} are compared bit for bit, in bf16 and in fp32 output;
the seeded random inputs within the stated tolerances ("the GPU result must be
bit-exact against the oracle on small-integer inputs", normwise 1e-5 for fp32
and 2^-7|O| + 1e-5 max|O| per element for bf16). The oracle runs once per
input set; both plans are compared with that one result.

The fused-epilogue shape the benchmark times (QKV, D = sigmoid(A*B + bias) *
aux) is checked the same way against the oracle's epilogue.
"""
import numpy as np
import pytest
import torch

import oracle
import tile_partitioned_dense_gb300 as tpd
from _gpu import DEV, assert_bit_exact, assert_within_tolerance, bits, oracle_out, run, to_device
from workloads import CONFIGS, ORDER, make_inputs

pytestmark = pytest.mark.gpu

PLANS = ["plain", "bench"]


@pytest.fixture(scope="module")
def handles():
    plain = tpd.gemm_create(0)
    bench = tpd.gemm_create(0)
    nbytes = tpd.gemm_workspace_size(bench)
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=DEV)
    ptr = (buf.data_ptr() + 255) // 256 * 256
    assert tpd.gemm_set_workspace(bench, ptr, nbytes, torch.cuda.current_stream().cuda_stream) == tpd.OK
    torch.cuda.synchronize()
    yield {"plain": plain, "bench": bench}
    torch.cuda.synchronize()
    tpd.gemm_set_workspace(bench, None, 0, None)
    tpd.gemm_destroy(bench)
    tpd.gemm_destroy(plain)
    del buf


def _dt(cfg):
    return torch.float32 if cfg.out_dtype == "f32" else torch.bfloat16


def _on_device(A, B, C):
    return to_device(A), to_device(B), to_device(C)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("name", ORDER)
def test_config_integer_every_element_bit_exact(handles, name, out_dtype):
    cfg = CONFIGS[name]
    A, B, C = make_inputs(cfg, integer=True)
    if C is not None:
        C = C.to(out_dtype)
    Ad, Bd, Cd = _on_device(A, B, C)
    want = oracle_out(A, B, C, cfg.alpha, cfg.beta, out_dtype)
    for plan in PLANS:
        D, _ = run(handles[plan], Ad, Bd, Cd, cfg.alpha, cfg.beta, out_dtype)
        assert_bit_exact(bits(D), want, f"{name} {plan}")
        del D


@pytest.mark.parametrize("name", ORDER)
def test_config_random_every_element_within_tolerance(handles, name):
    cfg = CONFIGS[name]
    A, B, C = make_inputs(cfg)
    out = _dt(cfg)
    Ad, Bd, Cd = _on_device(A, B, C)
    want = oracle_out(A, B, C, cfg.alpha, cfg.beta, out)
    for plan in PLANS:
        D, _ = run(handles[plan], Ad, Bd, Cd, cfg.alpha, cfg.beta, out)
        got = bits(D)
        assert_within_tolerance(got, want, out, f"{name} {plan}")
        # determinism: the same inputs give the same bits (fixed k order per tile, no atomics)
        D2, _ = run(handles[plan], Ad, Bd, Cd, cfg.alpha, cfg.beta, out)
        assert np.array_equal(got.view(np.uint8), bits(D2).view(np.uint8)), f"{name} {plan}: run-to-run difference"
        del D, D2


def test_bench_plans(handles):
    """The plans the benchmark times on a full GB300: CTA pairs for the large
    shapes, with the K split tail on QKV only when a workspace is attached."""
    h = handles["bench"]
    if tpd.gemm_num_sms(h) < 148:
        pytest.skip("tile counts assume a full GB300")
    want_tail = {"square": 1, "qkv": 1, "mlp_down": 0, "tiny": 0, "decode": 0}
    for name in ORDER:
        cfg = CONFIGS[name]
        oc = tpd.OUT_F32 if cfg.out_dtype == "f32" else tpd.OUT_BF16
        assert tpd.gemm_plan_tail_ksplit(h, cfg.M, cfg.N, cfg.K, oc) == want_tail[name], name
        assert tpd.gemm_plan_tail_ksplit(handles["plain"], cfg.M, cfg.N, cfg.K, oc) == 0, name


def test_qkv_fused_bias_sigmoid_aux_every_element(handles):
    """The benchmark's fused shape: QKV with D = sigmoid(A*B + bias) * aux in
    bf16, bias and aux drawn as the benchmark draws them, every element within
    the bf16 tolerance of the oracle's epilogue."""
    cfg = CONFIGS["qkv"]
    A, B, _ = make_inputs(cfg)
    g = torch.Generator().manual_seed(cfg.seed + 100)
    bias = (torch.randn(cfg.N, generator=g) * 0.1).to(torch.bfloat16)
    aux = torch.rand(cfg.M, cfg.N, generator=g).to(torch.bfloat16)
    want, _ = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_BF16, bias=bias,
                                        act=oracle.ACT_SIGMOID, aux=aux)
    Ad, Bd, Xd, bd = to_device(A), to_device(B), to_device(aux), bias.to(DEV)
    for plan in PLANS:
        h = handles[plan]
        D = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=DEV)
        epi = tpd.Epilogue(bd.data_ptr(), tpd.OUT_BF16, tpd.ACT_SIGMOID, Xd.data_ptr(), Xd.stride(0))
        s = torch.cuda.current_stream().cuda_stream
        st = tpd.gemm_run_epilogue(h, cfg.M, cfg.N, cfg.K, Ad.data_ptr(), cfg.K, Bd.data_ptr(), cfg.N, None, cfg.N,
                                   D.data_ptr(), cfg.N, 1.0, 0.0, tpd.OUT_BF16, epi, s)
        assert st == tpd.OK, tpd.gemm_status_string(st)
        assert tpd.gemm_sync_status(h, s) == tpd.OK
        assert_within_tolerance(bits(D), want, torch.bfloat16, f"qkv fused {plan}")
        del D


def test_plans_match_the_design(handles):
    h = handles["plain"]
    sms = tpd.gemm_num_sms(h)
    p = tpd.gemm_query_plan(h, 4096, 4096, 4096, tpd.OUT_BF16)
    assert p["variant"] == tpd.VARIANT_TILED_PAIR and p["tile_m"] == 256 and p["tile_n"] == 256
    assert p["num_tiles"] == 16 * 16 and p["cluster"] == 2 and p["launches"] == 1
    assert p["grid"] % 2 == 0 and sms - 8 <= p["grid"] <= sms
    p = tpd.gemm_query_plan(h, 16, 28672, 4096, tpd.OUT_BF16)
    assert p["variant"] == tpd.VARIANT_STREAM and p["num_tiles"] == 224 and p["cluster"] == 2
    assert p["grid"] % 2 == 0 and p["grid"] <= sms
    # few tiles: 1-CTA tiles whose K range is shared by the 4 (or 2) CTAs of a cluster
    p = tpd.gemm_query_plan(h, 256, 256, 256, tpd.OUT_F32)
    assert p["variant"] == tpd.VARIANT_TILED and p["num_tiles"] == 2 and p["cluster"] == 4 and p["grid"] == 8
    p = tpd.gemm_query_plan(h, 100, 256, 256, tpd.OUT_F32)
    assert p["variant"] == tpd.VARIANT_TILED and p["cluster"] == 4 and p["grid"] == 4
    p = tpd.gemm_query_plan(h, 128, 8192, 4096, tpd.OUT_BF16)  # 32 tiles
    assert p["variant"] == tpd.VARIANT_TILED and p["cluster"] == 4 and p["grid"] == 128
    p = tpd.gemm_query_plan(h, 512, 4096, 4096, tpd.OUT_BF16)  # 64 tiles: pairs of CTAs
    assert p["variant"] == tpd.VARIANT_TILED and p["cluster"] == 2 and p["grid"] == 128
    p = tpd.gemm_query_plan(h, 512, 4096, 64, tpd.OUT_BF16)  # one K block: nothing to share
    assert p["variant"] == tpd.VARIANT_TILED_PAIR and p["cluster"] == 2
    p = tpd.gemm_query_plan(h, 1024, 4096, 4096, tpd.OUT_BF16)  # 128 tiles: more than 76 pairs
    assert p["variant"] == tpd.VARIANT_TILED_PAIR
    # forced 1-CTA tiles keep the column pieces: one tile cut into four quarters on four CTAs
    assert tpd.gemm_force_variant(h, tpd.VARIANT_TILED) == tpd.OK
    try:
        p = tpd.gemm_query_plan(h, 100, 256, 256, tpd.OUT_F32)
        assert p["variant"] == tpd.VARIANT_TILED and p["cluster"] == 1 and p["grid"] == 4
        p = tpd.gemm_query_plan(h, 128, 8192, 4096, tpd.OUT_BF16)  # 32 tiles -> 128 quarter tiles
        assert p["cluster"] == 1 and p["grid"] == min(128, sms)
    finally:
        tpd.gemm_force_variant(h, tpd.VARIANT_AUTO)
    p = tpd.gemm_query_plan(h, 5, 5, 0, tpd.OUT_F32)
    assert p["variant"] == tpd.VARIANT_EPILOGUE_ONLY
