"""Pins of the oracle's fused epilogue (CPU only).

The epilogue follows the EFC capabilities named in the epilogue-fusion roadmap
paragraph of "TorchInductor ganha suporte a GEMMs de alta performance com
CuteDSL" (auxiliary tensor loads, element-wise add and mul, ReLU, sigmoid,
tanh). Reading taken for the order:
    v = alpha*acc + beta*C;  v += bias[n];  v = act(v);  v *= aux[m, n]
The pins tie it to invariants of the activations, to cases where any other
order of the steps gives a different value, and to brute force.
"""
import math

import numpy as np
import pytest
import torch

import oracle

S, R, T, NONE = oracle.ACT_SIGMOID, oracle.ACT_RELU, oracle.ACT_TANH, oracle.ACT_NONE


def _bf16(values, shape):
    return torch.tensor(values, dtype=torch.float64).reshape(shape).to(torch.bfloat16)


# ---------------------------------------------------------------- activations

def test_relu_closed_form():
    for x in [-3.5, -1e-300, -0.0, 0.0, 1e-300, 2.25, 1e30]:
        assert oracle.activation(R, x) == (x if x > 0 else 0.0)


def test_sigmoid_invariants():
    assert oracle.activation(S, 0.0) == 0.5
    for x in [1e-8, 0.25, 1.0, 3.0, 10.0, 30.0]:
        s, t = oracle.activation(S, x), oracle.activation(S, -x)
        assert 0.5 < s < 1.0 and 0.0 < t < 0.5
        assert abs(s + t - 1.0) <= 4 * 2.0 ** -53
    xs = np.linspace(-8, 8, 321)
    ys = [oracle.activation(S, float(x)) for x in xs]
    assert all(b > a for a, b in zip(ys, ys[1:]))  # strictly increasing
    assert oracle.activation(S, 800.0) == 1.0 and oracle.activation(S, -800.0) == 0.0


def test_tanh_invariants():
    assert oracle.activation(T, 0.0) == 0.0
    for x in [1e-8, 0.3, 1.0, 2.5, 9.0]:
        assert oracle.activation(T, -x) == -oracle.activation(T, x)  # odd
        # tanh(x) = 2*sigmoid(2x) - 1 ties the two independently computed paths
        assert abs(oracle.activation(T, x) - (2.0 * oracle.activation(S, 2.0 * x) - 1.0)) <= 8 * 2.0 ** -53
    assert oracle.activation(T, 25.0) == 1.0 and oracle.activation(T, -25.0) == -1.0


def test_identity_activation():
    for x in [-2.0, 0.0, 3.75]:
        assert oracle.activation(NONE, x) == x


# ---------------------------------------------------------------- composition

def _one_element(acc, c=0.0, bias=None, act=NONE, aux=None, alpha=1.0, beta=0.0, out=oracle.OUT_F32):
    """1x1x1 GEMM with A = acc, B = 1, so that alpha*acc is exact."""
    A = _bf16([acc], (1, 1))
    B = _bf16([1.0], (1, 1))
    dt = torch.float32 if out == oracle.OUT_F32 else torch.bfloat16
    C = torch.tensor([[c]], dtype=dt)
    b = None if bias is None else torch.tensor([bias], dtype=torch.float32)
    x = None if aux is None else torch.tensor([[aux]], dtype=dt)
    _, pre = oracle.gemm_rows_epilogue(A, B, C, alpha, beta, out, bias=b, act=act, aux=x, want_pre=True)
    return pre[0, 0]


def test_step_order():
    # bias before the activation: relu(1 + (-3)) = 0; the other order gives -2
    assert _one_element(1.0, bias=-3.0, act=R) == 0.0
    # aux after the activation: relu(-2) * (-1) = 0; multiplying first gives 2
    assert _one_element(-2.0, act=R, aux=-1.0) == 0.0
    # beta*C before bias and activation: relu(2*1 + 1*(-4) + 1) = 0
    assert _one_element(1.0, c=-4.0, bias=1.0, act=R, alpha=2.0, beta=1.0) == 0.0
    assert _one_element(1.0, c=4.0, bias=1.0, act=R, alpha=2.0, beta=1.0) == 7.0
    # sigmoid of an exactly zero pre-activation (acc + bias = 0) is 0.5, times aux 4 = 2
    assert _one_element(2.0, bias=-2.0, act=S, aux=4.0) == 2.0
    # tanh(0) * anything = 0; without the bias it would be tanh(3) * 5
    assert _one_element(3.0, bias=-3.0, act=T, aux=5.0) == 0.0


def test_bias_indexed_by_column_aux_by_row_and_column():
    M, N, K = 3, 5, 4
    A = torch.ones(M, K, dtype=torch.bfloat16)
    B = torch.zeros(K, N, dtype=torch.bfloat16)  # acc = 0 everywhere
    bias = torch.tensor([1.0, -2.0, 3.0, -4.0, 5.0])
    base = torch.full((M, 8), float("nan"))        # padded aux, NaN in the padding
    aux = base[:, :N]
    aux[:] = torch.arange(M * N, dtype=torch.float32).reshape(M, N)
    D, _ = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_F32, bias=bias, act=R, aux=aux)
    want = np.maximum(bias.numpy(), 0)[None, :] * np.arange(M * N, dtype=np.float32).reshape(M, N)
    np.testing.assert_array_equal(D, want.astype(np.float32))


def test_bf16_bias_and_output():
    M, N, K = 2, 3, 2
    A = _bf16([1, 2, 3, 4], (M, K))
    B = _bf16([1, 0, -1, 0, 1, 2], (K, N))   # A*B = [[1,2,3],[3,4,5]]
    bias = torch.tensor([0.5, -10.0, 0.25]).to(torch.bfloat16)
    aux = torch.tensor([[2, 2, 2], [-1, -1, -1]], dtype=torch.float32).to(torch.bfloat16)
    D, pre = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_BF16, bias=bias, act=R, aux=aux,
                                       want_pre=True)
    np.testing.assert_array_equal(pre, np.array([[3.0, 0.0, 6.5], [-3.5, 0.0, -5.25]]))


@pytest.mark.parametrize("act", [NONE, R, S, T])
@pytest.mark.parametrize("out", [oracle.OUT_F32, oracle.OUT_BF16])
def test_brute_force_small(act, out):
    """Every element against a pure-Python loop (fsum of exact products,
    then the steps in order) with padded strides on A, B, C and aux."""
    M, N, K = 6, 9, 13
    g = torch.Generator().manual_seed(act * 7 + out)
    dt = torch.float32 if out == oracle.OUT_F32 else torch.bfloat16
    pad = lambda t, ld: torch.cat([t, torch.full((t.shape[0], ld - t.shape[1]), float("nan"), dtype=t.dtype)], 1)[:, :t.shape[1]]
    A = pad(torch.randn(M, K, generator=g).to(torch.bfloat16), 16)
    B = pad(torch.randn(K, N, generator=g).to(torch.bfloat16), 16)
    C = pad(torch.randn(M, N, generator=g).to(dt), 16)
    aux = pad((torch.rand(M, N, generator=g) * 2).to(dt), 12)
    bias = torch.randn(N, generator=g).to(torch.bfloat16)
    alpha, beta = 0.5, -0.75
    _, pre = oracle.gemm_rows_epilogue(A, B, C, alpha, beta, out, bias=bias, act=act, aux=aux, want_pre=True)
    a, b = A.double().numpy(), B.double().numpy()
    c, x, bb = C.double().numpy(), aux.double().numpy(), bias.double().numpy()
    f = {NONE: lambda v: v, R: lambda v: max(v, 0.0), S: lambda v: 1.0 / (1.0 + math.exp(-v)), T: math.tanh}[act]
    for i in range(M):
        for j in range(N):
            s = math.fsum(a[i, k] * b[k, j] for k in range(K))
            v = f(alpha * s + beta * c[i, j] + bb[j]) * x[i, j]
            assert abs(pre[i, j] - v) <= 1e-12 * (abs(v) + 1.0)


def test_integer_inputs_stay_exact_through_relu_bias_aux():
    M, N, K = 8, 16, 32
    g = torch.Generator().manual_seed(2)
    A = torch.randint(-4, 5, (M, K), generator=g).to(torch.bfloat16)
    B = torch.randint(-4, 5, (K, N), generator=g).to(torch.bfloat16)
    bias = torch.randint(-8, 9, (N,), generator=g).to(torch.float32)
    aux = torch.randint(-2, 3, (M, N), generator=g).to(torch.float32)
    _, pre = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_F32, bias=bias, act=R, aux=aux,
                                       want_pre=True)
    exact = np.maximum(A.to(torch.int64).numpy() @ B.to(torch.int64).numpy() + bias.numpy().astype(np.int64), 0)
    np.testing.assert_array_equal(pre, (exact * aux.numpy().astype(np.int64)).astype(np.float64))


def test_plain_entry_equals_epilogue_entry_without_extras():
    g = torch.Generator().manual_seed(4)
    A = torch.randn(5, 7, generator=g).to(torch.bfloat16)
    B = torch.randn(7, 6, generator=g).to(torch.bfloat16)
    D0, p0 = oracle.gemm_rows(A, B, None, 1.0, 0.0, oracle.OUT_BF16, want_pre=True)
    D1, p1 = oracle.gemm_rows_epilogue(A, B, None, 1.0, 0.0, oracle.OUT_BF16, want_pre=True)
    np.testing.assert_array_equal(D0, D1)
    np.testing.assert_array_equal(p0, p1)


def test_epilogue_rejects_bad_activation():
    A = torch.ones(1, 1, dtype=torch.bfloat16)
    with pytest.raises(RuntimeError):
        oracle.gemm_rows_epilogue(A, A, None, 1.0, 0.0, oracle.OUT_F32, act=9)
