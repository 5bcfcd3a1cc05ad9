"""Pins of the CPU oracle to things other than itself (CPU only, no GPU).

Each test ties the oracle to a closed form, a hand computation, brute force, or
the IEEE-754 rounding definition, chosen so that a plausible slip in the oracle
(a dropped term, a wrong sign, a swapped index or stride, a transposed operand,
double rounding) fails at least one of them. The oracle follows the definition
D = alpha*A*B + beta*C of the GEMM that "TorchInductor ganha suporte a GEMMs de
alta performance com CuteDSL" puts at the centre of transformer cost; its
readings of the pages are listed in the header of oracle/oracle.c.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from workloads import CONFIGS, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _dec(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float64 values (PyTorch's exact widening)."""
    return t.to(torch.float64).numpy()


def _bf16(values, shape) -> torch.Tensor:
    return torch.tensor(values, dtype=torch.float64).reshape(shape).to(torch.bfloat16)


def _padded(t: torch.Tensor, ld: int) -> torch.Tensor:
    """Same values with a larger row stride; padding holds NaN sentinels."""
    rows, cols = t.shape
    base = torch.full((rows, ld), float("nan"), dtype=t.dtype)
    base[:, :cols] = t
    return base[:, :cols]


# ---------------------------------------------------------------- hand cases

def _read_golden_gemm(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    return vals


@pytest.mark.parametrize("out_dtype", [oracle.OUT_F32, oracle.OUT_BF16])
def test_hand_computed_2x3x2(out_dtype):
    g = _read_golden_gemm("gemm_hand_2x3x2.txt")
    M, N, K = int(g["M"][0]), int(g["N"][0]), int(g["K"][0])
    A = _bf16(g["A"], (M, K))
    B = _bf16(g["B"], (K, N))
    Cf = torch.tensor(g["C"], dtype=torch.float32).reshape(M, N)
    C = Cf if out_dtype == oracle.OUT_F32 else Cf.to(torch.bfloat16)
    D, pre = oracle.gemm_rows(A, B, C, g["alpha"][0], g["beta"][0], out_dtype, want_pre=True)
    np.testing.assert_array_equal(pre, np.array(g["D"]).reshape(M, N))
    _, ab = oracle.gemm_rows(A, B, None, 1.0, 0.0, out_dtype, want_pre=True)
    np.testing.assert_array_equal(ab, np.array(g["AB"]).reshape(M, N))
    if out_dtype == oracle.OUT_F32:
        np.testing.assert_array_equal(D, np.array(g["D"], dtype=np.float32).reshape(M, N))


def test_2x2x2_integers():
    # [[1,2],[3,4]] @ [[5,6],[7,8]] = [[19,22],[43,50]]
    A = _bf16([1, 2, 3, 4], (2, 2))
    B = _bf16([5, 6, 7, 8], (2, 2))
    D, _ = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D, np.array([[19, 22], [43, 50]], dtype=np.float32))
    # negative entries: [[-1,2],[3,-4]] @ [[5,-6],[7,8]] = [[9,22],[-13,-50]]
    A = _bf16([-1, 2, 3, -4], (2, 2))
    B = _bf16([5, -6, 7, 8], (2, 2))
    D, _ = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D, np.array([[9, 22], [-13, -50]], dtype=np.float32))


# ---------------------------------------------------------------- closed forms

def test_identity_returns_B_bit_exact():
    K, N = 37, 53
    g = torch.Generator().manual_seed(7)
    B = (torch.rand(K, N, generator=g) * 2 - 1).to(torch.bfloat16)
    A = torch.eye(K, dtype=torch.bfloat16)
    A_p, B_p = _padded(A, 40), _padded(B, 56)
    D32, _ = oracle.gemm_rows(A_p, B_p, None, 1.0, 0.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D32, B.to(torch.float32).numpy())
    D16, _ = oracle.gemm_rows(A_p, B_p, None, 1.0, 0.0, oracle.OUT_BF16)
    np.testing.assert_array_equal(D16, B.view(torch.int16).numpy().view(np.uint16))


def test_all_ones_A_gives_column_sums_of_B():
    M, K, N = 5, 33, 19
    g = torch.Generator().manual_seed(11)
    B = torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16)
    A = torch.ones(M, K, dtype=torch.bfloat16)
    _, pre = oracle.gemm_rows(A, _padded(B, 24), None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    colsum = np.zeros(N, dtype=np.int64)
    Bi = B.to(torch.int64).numpy()
    for k in range(K):  # a separate loop over integer values
        colsum += Bi[k]
    for i in range(M):
        np.testing.assert_array_equal(pre[i], colsum.astype(np.float64))
    # random B: every row equals the exactly rounded column sum within the
    # sequential-summation bound K * 2^-53 * sum|b|
    Br = (torch.rand(K, N, generator=g) * 2 - 1).to(torch.bfloat16)
    _, pre = oracle.gemm_rows(A, Br, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    b = _dec(Br)
    for j in range(N):
        exact = math.fsum(b[:, j])
        bound = K * 2.0 ** -53 * float(np.abs(b[:, j]).sum())
        assert np.all(np.abs(pre[:, j] - exact) <= bound)


def test_transpose_identity_bitwise():
    # (A*B)^T = B^T * A^T; the products and the k order are the same, so the
    # fp64 values before rounding agree bit for bit.
    M, N, K = 23, 41, 67
    g = torch.Generator().manual_seed(3)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    _, pre = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    _, preT = oracle.gemm_rows(B.t().contiguous(), A.t().contiguous(), None, 1.0, 0.0,
                               oracle.OUT_F32, want_pre=True)
    assert np.array_equal(pre.T.view(np.uint64), preT.view(np.uint64))


@pytest.mark.parametrize("K", [1, 2, 17, 1000])
def test_brute_force_1x1xK(K):
    g = torch.Generator().manual_seed(K)
    A = torch.randn(1, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, 1, generator=g).to(torch.bfloat16)
    _, pre = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    p = _dec(A)[0] * _dec(B)[:, 0]  # each product exact in fp64
    exact = math.fsum(p)
    assert abs(pre[0, 0] - exact) <= K * 2.0 ** -53 * float(np.abs(p).sum())


def test_brute_force_small_with_strides_and_epilogue():
    """Every element against a pure-Python loop, with padded strides on A, B,
    C, a subset of rows in a permuted order, alpha and beta both non-trivial."""
    M, N, K = 9, 13, 21
    g = torch.Generator().manual_seed(5)
    A = _padded(torch.randn(M, K, generator=g).to(torch.bfloat16), 24)
    B = _padded(torch.randn(K, N, generator=g).to(torch.bfloat16), 16)
    C32 = _padded(torch.randn(M, N, generator=g), 20)
    alpha, beta = 0.75, -1.25
    rows = [8, 0, 3, 7]
    D, pre = oracle.gemm_rows(A, B, C32, alpha, beta, oracle.OUT_F32, rows=rows, want_pre=True)
    a, b, c = _dec(A), _dec(B), C32.to(torch.float64).numpy()
    for r, i in enumerate(rows):
        for j in range(N):
            p = [a[i, k] * b[k, j] for k in range(K)]
            s = math.fsum(p)
            bound = K * 2.0 ** -53 * sum(abs(x) for x in p)
            expect = alpha * s + beta * c[i, j]
            assert abs(pre[r, j] - expect) <= abs(alpha) * bound + 2.0 ** -52 * abs(expect)
            assert D[r, j] == np.float32(pre[r, j])
    # the same rows with a bf16 C and bf16 output
    C16 = _padded(torch.randn(M, N, generator=g).to(torch.bfloat16), 24)
    D16, pre16 = oracle.gemm_rows(A, B, C16, alpha, beta, oracle.OUT_BF16, rows=rows, want_pre=True)
    c16 = _dec(C16)
    for r, i in enumerate(rows):
        for j in range(N):
            s = math.fsum(a[i, k] * b[k, j] for k in range(K))
            expect = alpha * s + beta * c16[i, j]
            assert abs(pre16[r, j] - expect) <= 1e-12 * (abs(expect) + 1)
    assert np.array_equal(D16, oracle.round_bf16_array(pre16))


def test_integer_inputs_give_exact_integers():
    cfg = CONFIGS["tiny"]
    A, B, _ = make_inputs(cfg, integer=True, M=64, N=48, K=256)
    _, pre = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    assert np.all(pre == np.round(pre))
    exact = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy()
    np.testing.assert_array_equal(pre, exact.astype(np.float64))


# ---------------------------------------------------------------- epilogue

def test_linearity_in_alpha_beta():
    M, N, K = 16, 24, 40
    g = torch.Generator().manual_seed(9)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    C = torch.randn(M, N, generator=g)
    _, p10 = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32, want_pre=True)
    for alpha, beta in [(2.0, 0.0), (0.5, 3.0), (-1.5, -0.25), (0.0, 1.0)]:
        _, p = oracle.gemm_rows(A, B, C, alpha, beta, oracle.OUT_F32, want_pre=True)
        expect = alpha * p10 + beta * C.to(torch.float64).numpy()
        ulp = np.spacing(np.maximum(np.abs(expect), np.abs(p)))
        assert np.all(np.abs(p - expect) <= 2 * ulp)


@pytest.mark.parametrize("out_dtype", [oracle.OUT_F32, oracle.OUT_BF16])
def test_alpha0_beta1_returns_C(out_dtype):
    M, N, K = 7, 9, 5
    g = torch.Generator().manual_seed(1)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, generator=g).to(torch.bfloat16)
    C = torch.randn(M, N, generator=g)
    if out_dtype == oracle.OUT_BF16:
        C = C.to(torch.bfloat16)
    D, _ = oracle.gemm_rows(A, B, C, 0.0, 1.0, out_dtype)
    want = C.numpy() if out_dtype == oracle.OUT_F32 else C.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(D, want)


def test_beta0_does_not_read_C():
    M, N, K = 4, 6, 8
    A = torch.ones(M, K, dtype=torch.bfloat16)
    B = torch.ones(K, N, dtype=torch.bfloat16)
    Cnan = torch.full((M, N), float("nan"))
    D, _ = oracle.gemm_rows(A, B, Cnan, 1.0, 0.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D, np.full((M, N), K, dtype=np.float32))
    D, _ = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D, np.full((M, N), K, dtype=np.float32))


def test_K0_gives_beta_C():
    M, N = 3, 5
    A = torch.zeros(M, 0, dtype=torch.bfloat16)
    B = torch.zeros(0, N, dtype=torch.bfloat16)
    C = torch.arange(M * N, dtype=torch.float32).reshape(M, N)
    D, _ = oracle.gemm_rows(A, B, C, 1.0, -2.0, oracle.OUT_F32)
    np.testing.assert_array_equal(D, (-2.0 * C).numpy())


# ---------------------------------------------------------------- rounding

def _rne_cases():
    out = []
    with open(os.path.join(GOLDEN, "rne_cases.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                x, bits, *_ = line.split()
                out.append((float.fromhex(x), int(bits, 16), line.strip()))
    return out


@pytest.mark.parametrize("x,bits,line", _rne_cases())
def test_round_bf16_hand_cases(x, bits, line):
    assert oracle.round_bf16(x) == bits, line


def test_round_bf16_nan_inf():
    assert oracle.round_bf16(float("nan")) == 0x7FC0
    assert oracle.round_bf16(float("inf")) == 0x7F80
    assert oracle.round_bf16(float("-inf")) == 0xFF80


def test_round_f32_hand_cases():
    # binary32 quantum at [1,2) is 2^-23
    assert oracle.round_f32(1 + 2.0 ** -24) == 1.0  # tie -> even (1.0)
    assert oracle.round_f32(1 + 3 * 2.0 ** -24) == 1 + 2.0 ** -22  # tie -> even
    assert oracle.round_f32(1 + 2.0 ** -24 + 2.0 ** -40) == 1 + 2.0 ** -23  # above tie
    assert oracle.round_f32(float.fromhex("0x1.fffffefffffffp127")) == float.fromhex("0x1.fffffep127")
    assert math.isinf(oracle.round_f32(float.fromhex("0x1.ffffffp127")))


def test_round_bf16_exhaustive_against_integer_rne(tmp_path):
    """All 2^32 binary32 patterns through the oracle's fp64 -> bf16 rounding
    against an independent integer round-to-nearest-even (tests/c/rne_exhaustive.c)."""
    lib = oracle.library_path()
    exe = tmp_path / "rne"
    src = os.path.join(os.path.dirname(__file__), "c", "rne_exhaustive.c")
    subprocess.run(["gcc", "-O2", "-pthread", "-o", str(exe), src, lib,
                    f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True)
    nt = max(1, len(os.sched_getaffinity(0)))
    r = subprocess.run([str(exe), str(nt)], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout


def test_round_bf16_batch_matches_scalar():
    g = np.random.default_rng(0)
    u = g.integers(0, 2 ** 32, size=4096, dtype=np.uint64).astype(np.uint32)
    batch = oracle.round_bf16_from_f32_bits(u)
    for k in range(0, 4096, 97):
        assert batch[k] == oracle.round_bf16(float(u[k:k + 1].view(np.float32)[0]))


# ---------------------------------------------------------------- argument checks

def test_oracle_rejects_bad_rows():
    A = torch.ones(2, 2, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError):
        oracle.gemm_rows(A, A, None, 1.0, 0.0, oracle.OUT_F32, rows=[2])


def test_row_subset_equals_full_rows():
    cfg = CONFIGS["tiny"]
    A, B, _ = make_inputs(cfg, M=40, N=24, K=32)
    Dfull, pfull = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_BF16, want_pre=True, nthreads=3)
    rows = [39, 2, 17]
    Dsub, psub = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_BF16, rows=rows, want_pre=True,
                                  nthreads=1)
    np.testing.assert_array_equal(Dsub, Dfull[rows])
    np.testing.assert_array_equal(psub, pfull[rows])


def test_gemm_bf16_output_rounds_once():
    """A*B = 1 + 2^-8 + 2^-40 exactly. One rounding to bf16 gives 1 + 2^-7
    (0x3F81, the value is above the halfway point); a detour through fp32 would
    land on the tie 1 + 2^-8 and then round to even, 1.0 (0x3F80)."""
    A = _bf16([1.0, 2.0 ** -8, 2.0 ** -40], (1, 3))
    B = _bf16([1.0, 1.0, 1.0], (3, 1))
    D, pre = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_BF16, want_pre=True)
    assert pre[0, 0] == 1 + 2.0 ** -8 + 2.0 ** -40
    assert int(D[0, 0]) == 0x3F81
    # the same trap through the epilogue: alpha*acc + beta*C with C = 2^-40
    A = _bf16([1.0, 2.0 ** -8], (1, 2))
    B = _bf16([1.0, 1.0], (2, 1))
    C = _bf16([2.0 ** -40], (1, 1))
    D, _ = oracle.gemm_rows(A, B, C, 1.0, 1.0, oracle.OUT_BF16)
    assert int(D[0, 0]) == 0x3F81
