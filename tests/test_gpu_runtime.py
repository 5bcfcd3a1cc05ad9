"""Runtime behaviour on the GPU: the bounded-wait watchdog, stream and graph
use of gemm_run, concurrent calls, and the multi-GPU shardings simulated on one
GPU (the shards run one after another; the host concatenates or sums them in a
fixed order)."""
import numpy as np
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import alloc_out, assert_bit_exact, assert_within_tolerance, bits, oracle_out, run, to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


def test_watchdog_times_out_and_context_survives(h):
    # A wait that nothing will ever satisfy must give up after its limit with
    # an error status, not hang ("Real-world Failure Modes").
    st = tpd.gemm_watchdog_selftest(h, 2_000_000, None)  # 2 ms
    assert st == tpd.ERR_TIMEOUT
    assert tpd.gemm_sync_status(h, None) == tpd.OK  # the self-test leaves the word clear
    # the context still works
    A, B, _ = make_inputs(CONFIGS["tiny"], integer=True, M=130, N=264, K=72)
    D, _ = run(h, A, B, None, 1.0, 0.0, torch.float32)
    assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.float32), "after watchdog")


def test_watchdog_rejects_out_of_range_limits(h):
    assert tpd.gemm_watchdog_selftest(h, 10, None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_watchdog_selftest(h, 10 ** 10, None) == tpd.ERR_INVALID_ARG


def test_argument_errors_launch_nothing(h):
    M = N = K = 64
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    D = torch.full((M, N), 7.0, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert tpd.gemm_run(h, M, N, K, A.data_ptr() + 2, K, B.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 0.0,
                        tpd.OUT_F32, s) == tpd.ERR_ALIGNMENT
    assert tpd.gemm_run(h, M, N, K, A.data_ptr(), K, B.data_ptr(), N, None, N, A.data_ptr(), N, 1.0, 0.0,
                        tpd.OUT_F32, s) == tpd.ERR_OVERLAP
    assert tpd.gemm_run(h, M, N, K, A.data_ptr(), K, B.data_ptr(), N, None, N, D.data_ptr(), N, 1.0, 1.0,
                        tpd.OUT_F32, s) == tpd.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(D == 7.0)  # untouched


def test_graph_capture_and_replay(h):
    # gemm_run allocates nothing and never synchronises, so it can be captured
    # ("cuTile Rust explained", "Why scoped graph capture helps borrowing").
    A, B, C = make_inputs(CONFIGS["tiny"], integer=True, M=384, N=512, K=256, c_for_beta=True)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    D = torch.empty((384, 512), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            st = tpd.gemm_run(h, 384, 512, 256, Ad.data_ptr(), 256, Bd.data_ptr(), 512, Cd.data_ptr(), 512,
                              D.data_ptr(), 512, 1.0, 1.0, tpd.OUT_F32, side.cuda_stream)
    assert st == tpd.OK
    D.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    assert_bit_exact(bits(D), oracle_out(A, B, C, 1.0, 1.0, torch.float32), "graph replay")


def test_two_streams_concurrently(h):
    cfg = CONFIGS["tiny"]
    A1, B1, _ = make_inputs(cfg, integer=True, M=1024, N=1024, K=512, seed=1)
    A2, B2, _ = make_inputs(cfg, integer=True, M=16, N=4096, K=1024, seed=2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    D1, _ = alloc_out(1024, 1024, torch.float32)
    D2, _ = alloc_out(16, 4096, torch.float32)
    A1d, B1d, A2d, B2d = to_device(A1), to_device(B1), to_device(A2), to_device(B2)
    torch.cuda.synchronize()
    for _ in range(3):
        assert tpd.gemm_run(h, 1024, 1024, 512, A1d.data_ptr(), 512, B1d.data_ptr(), 1024, None, 1024,
                            D1.data_ptr(), D1.stride(0), 1.0, 0.0, tpd.OUT_F32, s1.cuda_stream) == tpd.OK
        assert tpd.gemm_run(h, 16, 4096, 1024, A2d.data_ptr(), 1024, B2d.data_ptr(), 4096, None, 4096,
                            D2.data_ptr(), D2.stride(0), 1.0, 0.0, tpd.OUT_F32, s2.cuda_stream) == tpd.OK
    torch.cuda.synchronize()
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    assert_bit_exact(bits(D1), oracle_out(A1, B1, None, 1.0, 0.0, torch.float32), "stream 1")
    assert_bit_exact(bits(D2), oracle_out(A2, B2, None, 1.0, 0.0, torch.float32), "stream 2")


@pytest.mark.parametrize("shards", [2, 4])
def test_column_parallel_shards(h, shards):
    """Column-parallel split (QKV / gate-up): each shard owns B[:, cols] and
    D[:, cols]; concatenating the shards' D is the full D, bit for bit."""
    M, N, K = 256, 2048, 512
    A, B, _ = make_inputs(CONFIGS["qkv"], integer=True, M=M, N=N, K=K)
    Ad, Bd = to_device(A), to_device(B)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    w = N // shards
    s = torch.cuda.current_stream().cuda_stream
    for r in range(shards):  # pointer/stride offsets into the same buffers
        st = tpd.gemm_run(h, M, w, K, Ad.data_ptr(), K, Bd[:, r * w:].data_ptr(), N, None, N,
                          D[:, r * w:].data_ptr(), N, 1.0, 0.0, tpd.OUT_BF16, s)
        assert st == tpd.OK
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    assert_bit_exact(bits(D), oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16), "column shards")


@pytest.mark.parametrize("integer", [True, False])
def test_row_parallel_shards(h, integer):
    """Row-parallel split (down-projection): shard r owns A[:, k_r] and
    B[k_r, :] and computes an fp32 partial; the partials are summed in rank
    order on the host (the all-reduce) and beta*C is added once."""
    M, N, K, P = 256, 512, 2048, 4
    A, B, C = make_inputs(CONFIGS["mlp_down"], integer=integer, M=M, N=N, K=K)
    Ad, Bd = to_device(A), to_device(B)
    kr = K // P
    s = torch.cuda.current_stream().cuda_stream
    parts = []
    for r in range(P):
        Dp = torch.empty((M, N), dtype=torch.float32, device="cuda")
        st = tpd.gemm_run(h, M, N, kr, Ad[:, r * kr:].data_ptr(), K, Bd[r * kr:, :].data_ptr(), N, None, N,
                          Dp.data_ptr(), N, 1.0, 0.0, tpd.OUT_F32, s)
        assert st == tpd.OK
        parts.append(Dp)
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    total = parts[0].double().cpu()
    for p in parts[1:]:
        total = total + p.double().cpu()
    total = total + C.double()  # beta = 1, added once
    got = total.to(torch.bfloat16)
    want = oracle_out(A, B, C, 1.0, 1.0, torch.bfloat16)
    if integer:
        assert_bit_exact(bits(got), want, "row shards")
    else:
        assert_within_tolerance(bits(got), want, torch.bfloat16, "row shards")


def test_concurrent_host_threads_on_one_fresh_handle():
    """Four host threads make their first calls on a new handle at once (its
    occupancy caches start empty), each on its own stream with its own shape
    and kernel variant; every result is bit-exact."""
    import threading
    h2 = tpd.gemm_create(0)
    shapes = [(300, 520, 256), (16, 4096, 1024), (64, 2048, 512), (1000, 264, 128)]
    inputs, outs, errors = [], [], []
    for i, (M, N, K) in enumerate(shapes):
        A, B, _ = make_inputs(CONFIGS["tiny"], integer=True, M=M, N=N, K=K, seed=40 + i)
        inputs.append((A, B, to_device(A), to_device(B)))
        outs.append(torch.full((M, N), float("nan"), device="cuda"))
    streams = [torch.cuda.Stream() for _ in shapes]
    torch.cuda.synchronize()
    barrier = threading.Barrier(len(shapes))

    def work(i):
        M, N, K = shapes[i]
        _, _, Ad, Bd = inputs[i]
        barrier.wait()
        for _ in range(3):
            st = tpd.gemm_run(h2, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, outs[i].data_ptr(), N,
                              1.0, 0.0, tpd.OUT_F32, streams[i].cuda_stream)
            if st != tpd.OK:
                errors.append((i, st))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    try:
        assert not errors, errors
        assert tpd.gemm_sync_status(h2, None) == tpd.OK
        for i, (A, B, _, _) in enumerate(inputs):
            assert_bit_exact(bits(outs[i]), oracle_out(A, B, None, 1.0, 0.0, torch.float32), f"thread {i}")
    finally:
        tpd.gemm_destroy(h2)
