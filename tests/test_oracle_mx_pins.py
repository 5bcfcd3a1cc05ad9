"""Pins of the block-scaled (MX) oracle to things other than itself (CPU only).

The oracle (oracle/oracle_mx.c) computes the scaled_mm that "TorchInductor
ganha suporte a GEMMs de alta performance com CuteDSL" lists among its GEMMs
(the enablement paragraph) with the MXFP8 formats of its results paragraph,
read from the OCP Microscaling (MX) v1.0 specification: blocks of 32 elements
along K, one E8M0 scale per block, E4M3 or E5M2 elements. Each test ties it to
an independent decoder, a value the specification fixes, a hand computation,
exact rational brute force, or an invariant, so that a plausible slip (a wrong
exponent bias, a dropped subnormal, a scale applied to the wrong block, row or
operand, a transposed operand) fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CODES = np.arange(256, dtype=np.uint8)


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(both_nan | eq))


# ---------------------------------------------------------------- element and scale decoding

def test_e4m3_all_codes_match_torch_float8_e4m3fn():
    want = torch.from_numpy(CODES.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same(oracle.decode_mx(CODES, oracle.FP8_E4M3), want)


def test_e5m2_all_codes_are_the_top_byte_of_binary16():
    # E5M2 is binary16 with the low 8 significand bits dropped: numpy's IEEE
    # half-precision decoder of (code << 8) is an independent reference.
    want = (CODES.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    assert _same(oracle.decode_mx(CODES, oracle.FP8_E5M2), want)


def test_e8m0_all_codes_match_torch_float8_e8m0fnu():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no float8_e8m0fnu")
    want = torch.from_numpy(CODES.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert _same(oracle.decode_mx(CODES, oracle.SCALE_E8M0), want)


def test_values_the_specification_fixes():
    e4 = oracle.decode_mx(CODES, oracle.FP8_E4M3)
    assert e4[0x7E] == 448.0 and e4[0xFE] == -448.0          # largest finite
    assert e4[0x08] == 2.0 ** -6                              # smallest normal
    assert e4[0x07] == 0.875 * 2.0 ** -6                      # largest subnormal
    assert e4[0x01] == 2.0 ** -9                              # smallest subnormal
    assert np.isnan(e4[0x7F]) and np.isnan(e4[0xFF])          # the only NaNs, no infinities
    assert int(np.isnan(e4).sum()) == 2 and not np.isinf(e4).any()
    assert e4[0x38] == 1.0 and e4[0x80] == 0.0 and math.copysign(1, e4[0x80]) < 0
    e5 = oracle.decode_mx(CODES, oracle.FP8_E5M2)
    assert e5[0x7B] == 57344.0 and e5[0x04] == 2.0 ** -14 and e5[0x01] == 2.0 ** -16
    assert e5[0x7C] == math.inf and e5[0xFC] == -math.inf
    assert int(np.isnan(e5).sum()) == 6 and e5[0x3C] == 1.0
    s = oracle.decode_mx(CODES, oracle.SCALE_E8M0)
    assert s[127] == 1.0 and s[0] == 2.0 ** -127 and s[254] == 2.0 ** 127 and np.isnan(s[255])
    assert np.all(s[1:255] / s[:254] == 2.0)                  # consecutive codes double


# ---------------------------------------------------------------- hand case

def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "mx_hand_1x2x64.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *rest = line.split()
                vals[key] = rest
    return vals


def _row(spec, K=64):
    r = np.zeros((1, K), dtype=np.uint8)
    for item in spec:
        k, code = item.split(":")
        r[0, int(k)] = int(code, 16)
    return r


def _hex(spec):
    return np.array([[int(x, 16) for x in spec]], dtype=np.uint8)


@pytest.mark.parametrize("out_dtype", [oracle.OUT_F32, oracle.OUT_BF16])
def test_hand_computed_1x2x64(out_dtype):
    g = _golden()
    A, SA = _row(g["A_codes"]), _hex(g["SA"])
    got = []
    for bt, sb, fmt in [("Bt0_e4m3", "SB0", oracle.FP8_E4M3), ("Bt1_e5m2", "SB1", oracle.FP8_E5M2)]:
        D, _ = oracle.mx_gemm_rows(A, SA, _row(g[bt]), _hex(g[sb]), None, 1.0, 0.0, out_dtype, fmt_b=fmt)
        got.append(D[0, 0])
    if out_dtype == oracle.OUT_F32:
        assert got == [float(x) for x in g["D_f32"]]
    else:
        assert [int(x) for x in got] == [int(x, 16) for x in g["D_bf16"]]


# ---------------------------------------------------------------- brute force and invariants

def _random_mx(rng, M, N, K, fmt_a=oracle.FP8_E4M3, fmt_b=oracle.FP8_E4M3, scale_lo=120, scale_hi=134):
    """Random finite codes: FP8 elements with NaN/inf codes replaced, scales in a range."""
    def finite(shape, fmt):
        c = rng.integers(0, 256, size=shape, dtype=np.uint8)
        bad = ~np.isfinite(oracle.decode_mx(c, fmt))
        c[bad] = 0x30
        return c
    A = finite((M, K), fmt_a)
    Bt = finite((N, K), fmt_b)
    SA = rng.integers(scale_lo, scale_hi + 1, size=(M, K // 32), dtype=np.uint8)
    SB = rng.integers(scale_lo, scale_hi + 1, size=(N, K // 32), dtype=np.uint8)
    return A, SA, Bt, SB


def _exact(A, SA, Bt, SB, fmt_a, fmt_b):
    """Exact rational result with Python loops, from torch's (independent) decoders."""
    def dec(c, fmt):
        t = torch.from_numpy(np.ascontiguousarray(c))
        dt = torch.float8_e4m3fn if fmt == oracle.FP8_E4M3 else torch.float8_e5m2
        return t.view(dt).to(torch.float64).numpy()
    a, b = dec(A, fmt_a), dec(Bt, fmt_b)
    M, K = A.shape
    N = Bt.shape[0]
    out = np.zeros((M, N))
    for i in range(M):
        for n in range(N):
            total = Fraction(0)
            for k in range(K):
                sa = Fraction(2) ** (int(SA[i, k // 32]) - 127)
                sb = Fraction(2) ** (int(SB[n, k // 32]) - 127)
                total += sa * sb * Fraction(a[i, k]) * Fraction(b[n, k])
            out[i, n] = float(total)
    return out


@pytest.mark.parametrize("fmts", [(0, 0), (1, 1), (0, 1)], ids=["e4m3", "e5m2", "e4m3xe5m2"])
def test_brute_force_exact_rationals(fmts):
    rng = np.random.default_rng(5 + fmts[0] + 2 * fmts[1])
    M, N, K = 3, 4, 96
    A, SA, Bt, SB = _random_mx(rng, M, N, K, *fmts)
    _, pre = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, *fmts, want_pre=True)
    want = _exact(A, SA, Bt, SB, *fmts)
    # fp64 sums of up to 96 terms: within 96 ulps of the largest partial magnitude
    bound = 96 * 2.0 ** -52 * np.abs(want).max()
    assert np.all(np.abs(pre - want) <= bound)


def test_unit_scales_reduce_to_a_plain_integer_gemm():
    rng = np.random.default_rng(1)
    M, N, K = 7, 9, 160
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0, 3.0, -3.0, 4.0, -4.0])
    codes = np.array([0x00, 0x38, 0xB8, 0x40, 0xC0, 0x44, 0xC4, 0x48, 0xC8], dtype=np.uint8)
    ia = rng.integers(0, 9, size=(M, K))
    ib = rng.integers(0, 9, size=(N, K))
    A, Bt = codes[ia], codes[ib]
    SA = np.full((M, K // 32), 127, dtype=np.uint8)
    SB = np.full((N, K // 32), 127, dtype=np.uint8)
    D, _ = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32)
    want = vals[ia].astype(np.int64) @ vals[ib].astype(np.int64).T
    np.testing.assert_array_equal(D, want.astype(np.float32))


def test_scale_of_one_block_of_one_row_acts_only_there():
    rng = np.random.default_rng(2)
    M, N, K = 4, 5, 128
    A, SA, Bt, SB = _random_mx(rng, M, N, K)
    _, p0 = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    # A's block 2 of row 1 made zero: row 1 loses exactly that block's contribution,
    # after which its scale is irrelevant
    A2 = A.copy()
    A2[1, 64:96] = 0
    SA2 = SA.copy()
    SA2[1, 2] = 200
    _, p1 = oracle.mx_gemm_rows(A2, SA2, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    np.testing.assert_array_equal(p1[[0, 2, 3]], p0[[0, 2, 3]])
    only = A.copy()
    only[:, :64] = 0
    only[:, 96:] = 0
    _, pb = oracle.mx_gemm_rows(only[1:2], SA[1:2], Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    np.testing.assert_allclose(p1[1] + pb[0], p0[1], rtol=0, atol=1e-12 * np.abs(p0[1]).max())
    # one scale step up on a row doubles that row exactly, whatever its blocks hold
    SA3 = SA.copy()
    SA3[3, :] += 1
    _, p3 = oracle.mx_gemm_rows(A, SA3, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    np.testing.assert_array_equal(p3[3], 2 * p0[3])
    np.testing.assert_array_equal(p3[:3], p0[:3])
    # and a step on B's scales of column 4 doubles that column
    SB3 = SB.copy()
    SB3[4, :] += 1
    _, p4 = oracle.mx_gemm_rows(A, SA, Bt, SB3, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    np.testing.assert_array_equal(p4[:, 4], 2 * p0[:, 4])
    np.testing.assert_array_equal(p4[:, :4], p0[:, :4])


def test_transposed_problem_gives_the_transposed_result():
    rng = np.random.default_rng(3)
    A, SA, Bt, SB = _random_mx(rng, 6, 5, 96, oracle.FP8_E4M3, oracle.FP8_E5M2)
    _, p = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, oracle.FP8_E4M3, oracle.FP8_E5M2,
                               want_pre=True)
    _, pt = oracle.mx_gemm_rows(Bt, SB, A, SA, None, 1.0, 0.0, oracle.OUT_F32, oracle.FP8_E5M2, oracle.FP8_E4M3,
                                want_pre=True)
    np.testing.assert_array_equal(p, pt.T)


def test_strided_rows_and_row_subsets():
    rng = np.random.default_rng(4)
    A, SA, Bt, SB = _random_mx(rng, 9, 7, 64)
    D, _ = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_BF16)
    pad = lambda x, extra: np.pad(x, ((0, 0), (0, extra)), constant_values=0xFF)[:, :x.shape[1]]
    Ds, _ = oracle.mx_gemm_rows(pad(A, 16), pad(SA, 14), pad(Bt, 32), pad(SB, 6), None, 1.0, 0.0,
                                oracle.OUT_BF16, rows=[8, 0, 5])
    np.testing.assert_array_equal(Ds, D[[8, 0, 5]])


def test_alpha_beta_and_the_single_rounding():
    rng = np.random.default_rng(6)
    M, N, K = 5, 6, 64
    A, SA, Bt, SB = _random_mx(rng, M, N, K)
    C = torch.randn(M, N, generator=torch.Generator().manual_seed(6), dtype=torch.float32)
    _, p1 = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    _, pab = oracle.mx_gemm_rows(A, SA, Bt, SB, C, 0.5, -2.0, oracle.OUT_F32, want_pre=True)
    np.testing.assert_array_equal(pab, 0.5 * p1 + (-2.0) * C.double().numpy())
    D, _ = oracle.mx_gemm_rows(A, SA, Bt, SB, C, 0.0, 1.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D, C.numpy())
    Db, pb = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_BF16, want_pre=True)
    np.testing.assert_array_equal(Db, oracle.round_bf16_array(pb))


def test_nan_scale_poisons_only_its_row():
    rng = np.random.default_rng(7)
    A, SA, Bt, SB = _random_mx(rng, 3, 4, 64)
    A[1, :] = 0x38  # no zero element in row 1
    SA[1, 1] = 255
    D, _ = oracle.mx_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32)
    assert np.isnan(D[1]).all() and np.isfinite(D[[0, 2]]).all()


def test_bad_arguments_are_rejected():
    z = np.zeros((2, 64), dtype=np.uint8)
    s = np.zeros((2, 2), dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.mx_gemm_rows(np.zeros((2, 48), dtype=np.uint8), s[:, :1], z[:, :48], s[:, :1], None, 1.0, 0.0,
                            oracle.OUT_F32)
    with pytest.raises(RuntimeError):
        oracle.mx_gemm_rows(z, s, z, s, None, 1.0, 0.0, oracle.OUT_F32, fmt_a=3)


def test_blocked_scale_layout_helper_matches_its_definition():
    """The test harness's rearrangement of row-major scales into the kernel's
    blocked layout, checked byte by byte against the layout's definition."""
    from _gpu import mx_blocked
    rng = np.random.default_rng(9)
    for R, nb in [(128, 4), (130, 5), (300, 3), (1, 1)]:
        S = rng.integers(0, 255, size=(R, nb), dtype=np.uint8)
        got = mx_blocked(S)
        kc = -(-nb // 4)
        assert got.size == -(-R // 128) * kc * 512
        for r in range(R):
            for c in range(nb):
                off = ((r // 128) * kc + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
                assert got[off] == S[r, c]
