"""Pins of the block-scaled oracle's FP4 forms (CPU only): NVFP4 (E2M1
elements, blocks of 16 with E4M3 scales) and MXFP4 (E2M1, blocks of 32 with
E8M0 scales), the FP4 GEMMs "TorchInductor ganha suporte a GEMMs de alta
performance com CuteDSL" names. Each test ties oracle_bs_gemm_rows to the
values the OCP specification's E2M1 table fixes, a hand computation, exact
rational brute force or an invariant, so that a slip in the nibble order, the
block length, the scale format or an index fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
# E2M1 values of codes 0..7 (the OCP MX specification's table); 8..15 are their negatives
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
NV = dict(scale_fmt=oracle.SCALE_E4M3, block=16)
MX4 = dict(scale_fmt=oracle.SCALE_E8M0, block=32)


def test_e2m1_codes_match_the_specification_table():
    got = oracle.decode_mx(np.arange(16, dtype=np.uint8), oracle.FP4_E2M1)
    want = np.array(E2M1 + [-v for v in E2M1])
    assert np.array_equal(got, want) and np.signbit(got[8])
    # only the low four bits of a byte are one element
    assert np.array_equal(oracle.decode_mx(np.arange(16, dtype=np.uint8) | 0xA0, oracle.FP4_E2M1), want)


def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "fp4_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *rest = line.split()
                vals[key] = rest
    return vals


def _bytes(spec, n):
    r = np.zeros((1, n), dtype=np.uint8)
    for item in spec:
        k, code = item.split(":")
        r[0, int(k)] = int(code, 16)
    return r


def _hex(spec):
    return np.array([[int(x, 16) for x in spec]], dtype=np.uint8)


@pytest.mark.parametrize("out_dtype", [oracle.OUT_F32, oracle.OUT_BF16])
@pytest.mark.parametrize("kind", ["nv", "mx"])
def test_hand_computed(kind, out_dtype):
    g = _golden()
    K = 32 if kind == "nv" else 64
    kw = NV if kind == "nv" else MX4
    D, _ = oracle.bs_gemm_rows(_bytes(g[f"{kind}_A"], K // 2), _hex(g[f"{kind}_SA"]), _bytes(g[f"{kind}_Bt"], K // 2),
                               _hex(g[f"{kind}_SB"]), None, 1.0, 0.0, out_dtype, oracle.FP4_E2M1, oracle.FP4_E2M1,
                               **kw)
    if out_dtype == oracle.OUT_F32:
        assert float(D[0, 0]) == float(g[f"{kind}_D_f32"][0])
    else:
        assert int(D[0, 0]) == int(g[f"{kind}_D_bf16"][0], 16)


def _fp4(rng, rows, K):
    return rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)


def _unpack(codes):
    """FP4 bytes [R, K/2] -> values [R, K] from the specification's table."""
    tab = np.array(E2M1 + [-v for v in E2M1])
    lo = tab[codes & 0xF]
    hi = tab[codes >> 4]
    out = np.empty((codes.shape[0], codes.shape[1] * 2))
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def _scale_values(S, scale_fmt):
    t = torch.from_numpy(np.ascontiguousarray(S))
    if scale_fmt == oracle.SCALE_E4M3:
        return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.ldexp(1.0, S.astype(np.int64) - 127)


@pytest.mark.parametrize("kind", ["nv", "mx"])
def test_brute_force_exact_rationals(kind):
    kw = NV if kind == "nv" else MX4
    block = kw["block"]
    rng = np.random.default_rng(11 if kind == "nv" else 12)
    M, N, K = 3, 5, 4 * block
    A, Bt = _fp4(rng, M, K), _fp4(rng, N, K)
    if kind == "nv":  # positive finite E4M3 scales
        SA = rng.integers(0x20, 0x50, size=(M, K // block), dtype=np.uint8)
        SB = rng.integers(0x20, 0x50, size=(N, K // block), dtype=np.uint8)
    else:
        SA = rng.integers(120, 135, size=(M, K // block), dtype=np.uint8)
        SB = rng.integers(120, 135, size=(N, K // block), dtype=np.uint8)
    _, pre = oracle.bs_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, oracle.FP4_E2M1, oracle.FP4_E2M1,
                                 want_pre=True, **kw)
    a, b = _unpack(A), _unpack(Bt)
    sa, sb = _scale_values(SA, kw["scale_fmt"]), _scale_values(SB, kw["scale_fmt"])
    for i in range(M):
        for n in range(N):
            total = Fraction(0)
            for k in range(K):
                total += Fraction(sa[i, k // block]) * Fraction(sb[n, k // block]) * Fraction(a[i, k]) * Fraction(b[n, k])
            assert pre[i, n] == float(total)  # every term and partial sum is exact in fp64 here


def test_unit_scales_reduce_to_an_integer_gemm():
    rng = np.random.default_rng(3)
    M, N, K = 6, 7, 96
    ints = {0x0: 0, 0x2: 1, 0x4: 2, 0x5: 3, 0x6: 4, 0x7: 6, 0xA: -1, 0xC: -2, 0xD: -3, 0xE: -4, 0xF: -6}
    codes = np.array(list(ints), dtype=np.uint8)
    vals = np.array([ints[c] for c in codes], dtype=np.int64)
    ia, ib = rng.integers(0, len(codes), size=(M, K)), rng.integers(0, len(codes), size=(N, K))
    pack = lambda idx: (codes[idx[:, 0::2]] | (codes[idx[:, 1::2]] << 4)).astype(np.uint8)
    for kw, one in [(NV, 0x38), (MX4, 127)]:
        SA = np.full((M, K // kw["block"]), one, dtype=np.uint8)
        SB = np.full((N, K // kw["block"]), one, dtype=np.uint8)
        D, _ = oracle.bs_gemm_rows(pack(ia), SA, pack(ib), SB, None, 1.0, 0.0, oracle.OUT_F32, oracle.FP4_E2M1,
                                   oracle.FP4_E2M1, **kw)
        np.testing.assert_array_equal(D, (vals[ia] @ vals[ib].T).astype(np.float32))


def test_sixteen_element_blocks_and_nibble_pairing():
    """NVFP4: the scale of block b covers elements 16b .. 16b+15 only; and
    A's nibbles pair with B's in place (low with low, high with high). Which
    of the two is element 2i cannot change D (both operands use the same
    order, and a block holds whole bytes), so no test of D can pin it: it is
    the layout the interface states, and the inputs are packed that way."""
    rng = np.random.default_rng(5)
    M, N, K = 2, 3, 64
    A, Bt = _fp4(rng, M, K), _fp4(rng, N, K)
    SA = rng.integers(0x30, 0x48, size=(M, 4), dtype=np.uint8)
    SB = rng.integers(0x30, 0x48, size=(N, 4), dtype=np.uint8)
    args = (oracle.OUT_F32, oracle.FP4_E2M1, oracle.FP4_E2M1)
    _, p0 = oracle.bs_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, *args, want_pre=True, **NV)
    # zero elements 16..31 of row 0 (bytes 8..15): then block 1's scale of row 0 has no effect
    A1 = A.copy()
    A1[0, 8:16] = 0
    SA1 = SA.copy()
    SA1[0, 1] = 0x70
    _, p1 = oracle.bs_gemm_rows(A1, SA1, Bt, SB, None, 1.0, 0.0, *args, want_pre=True, **NV)
    SA2 = SA.copy()
    SA2[0, 1] = 0x70
    _, p2 = oracle.bs_gemm_rows(A1, SA, Bt, SB, None, 1.0, 0.0, *args, want_pre=True, **NV)
    np.testing.assert_array_equal(p1, p2)
    np.testing.assert_array_equal(p1[1], p0[1])
    # pairing: with B's low nibble nonzero and its high nibble zero, only A's low nibble counts
    B2 = np.zeros_like(Bt)
    B2[:, 0] = 0x02  # element 0 = 1.0, element 1 = 0
    A2 = np.zeros_like(A)
    A2[:, 0] = 0x70  # element 0 = 0, element 1 = 6
    _, p3 = oracle.bs_gemm_rows(A2, SA, B2, SB, None, 1.0, 0.0, *args, want_pre=True, **NV)
    assert np.all(p3 == 0.0)
    A2[:, 0] = 0x07  # element 0 = 6
    _, p4 = oracle.bs_gemm_rows(A2, SA, B2, SB, None, 1.0, 0.0, *args, want_pre=True, **NV)
    sa = _scale_values(SA[:, :1], oracle.SCALE_E4M3)
    sb = _scale_values(SB[:, :1], oracle.SCALE_E4M3)
    np.testing.assert_array_equal(p4, 6.0 * sa * sb.T)


def test_alpha_carries_the_per_tensor_scale_and_transpose_identity():
    rng = np.random.default_rng(7)
    M, N, K = 4, 6, 48
    A, Bt = _fp4(rng, M, K), _fp4(rng, N, K)
    SA = rng.integers(0x30, 0x48, size=(M, 3), dtype=np.uint8)
    SB = rng.integers(0x30, 0x48, size=(N, 3), dtype=np.uint8)
    f = (oracle.FP4_E2M1, oracle.FP4_E2M1)
    _, p1 = oracle.bs_gemm_rows(A, SA, Bt, SB, None, 1.0, 0.0, oracle.OUT_F32, *f, want_pre=True, **NV)
    _, p8 = oracle.bs_gemm_rows(A, SA, Bt, SB, None, 0.125, 0.0, oracle.OUT_F32, *f, want_pre=True, **NV)
    np.testing.assert_array_equal(p8, 0.125 * p1)
    _, pt = oracle.bs_gemm_rows(Bt, SB, A, SA, None, 1.0, 0.0, oracle.OUT_F32, *f, want_pre=True, **NV)
    np.testing.assert_array_equal(p1, pt.T)


def test_fp4_arguments_are_checked():
    z = np.zeros((2, 16), dtype=np.uint8)
    with pytest.raises(RuntimeError):  # block of 8 is not a format
        oracle.bs_gemm_rows(z, np.zeros((2, 4), np.uint8), z, np.zeros((2, 4), np.uint8), None, 1.0, 0.0,
                            oracle.OUT_F32, oracle.FP4_E2M1, oracle.FP4_E2M1, oracle.SCALE_E4M3, 8)
    with pytest.raises(ValueError):  # scales for the wrong block length
        oracle.bs_gemm_rows(z, np.zeros((2, 1), np.uint8), z, np.zeros((2, 1), np.uint8), None, 1.0, 0.0,
                            oracle.OUT_F32, oracle.FP4_E2M1, oracle.FP4_E2M1, **NV)
