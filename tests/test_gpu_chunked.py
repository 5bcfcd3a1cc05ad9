"""M-chunked GEMM and its stream/event contract ("Implementing Tensor
Parallelism Communication Overlays ...", "Pipelining GEMM and Collectives: The
Core Overlay Loop"): chunk i's GEMM on the compute stream, then event i; a
communication stream waits on event i and works on chunk i's rows while
chunk i+1 computes. Here the communication step is a device copy of the
chunk's rows (the collective itself needs several GPUs)."""
import numpy as np
import pytest
import torch

import tile_partitioned_dense_gb300 as tpd
from _gpu import assert_bit_exact, bits, oracle_out, round8, to_device
from workloads import CONFIGS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    handle = tpd.gemm_create(0)
    yield handle
    tpd.gemm_destroy(handle)


def _events(n, timing=True):
    evs = [torch.cuda.Event(enable_timing=timing) for _ in range(n)]
    for e in evs:
        e.record()  # creates the underlying cudaEvent_t
    torch.cuda.synchronize()
    return evs


def _bounds(M, chunks):
    b = [0] + [((i + 1) * M // chunks) // 128 * 128 for i in range(chunks - 1)] + [M]
    return [max(b[i], max(b[:i + 1])) for i in range(len(b))]


@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("shape", [(1000, 520, 136), (300, 264, 64), (2048, 1024, 512)],
                         ids=lambda s: "x".join(map(str, s)))
def test_chunked_equals_oracle_and_events_complete_in_order(h, chunks, shape):
    M, N, K = shape
    A, B, C = make_inputs(CONFIGS["tiny"], integer=True, M=M, N=N, K=K, c_for_beta=True, seed=chunks)
    Ad, Bd, Cd = to_device(A), to_device(B), to_device(C)
    D = torch.full((M, N), float("nan"), device="cuda")
    evs = _events(chunks)
    s = torch.cuda.current_stream()
    start = torch.cuda.Event(enable_timing=True)
    start.record(s)
    st = tpd.gemm_run_chunked(h, chunks, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, Cd.data_ptr(), N, D.data_ptr(),
                              N, 1.0, 1.0, tpd.OUT_F32, [e.cuda_event for e in evs], s.cuda_stream)
    assert st == tpd.OK, tpd.gemm_status_string(st)
    torch.cuda.synchronize()
    assert tpd.gemm_sync_status(h, None) == tpd.OK
    assert_bit_exact(bits(D), oracle_out(A, B, C, 1.0, 1.0, torch.float32), f"{shape} chunks {chunks}")
    assert all(e.query() for e in evs)
    t = [start.elapsed_time(e) for e in evs]
    assert all(b >= a for a, b in zip(t, t[1:])), t


@pytest.mark.parametrize("chunks", [2, 4])
def test_overlay_comm_stream_sees_finished_chunks(h, chunks):
    """The communication stream starts on chunk i as soon as event i fires;
    what it copies must be chunk i's final values."""
    M, N, K = 2048, 2048, 1024
    A, B, _ = make_inputs(CONFIGS["qkv"], integer=True, M=M, N=N, K=K)
    Ad, Bd = to_device(A), to_device(B)
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    sent = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    evs = _events(chunks, timing=False)
    compute = torch.cuda.Stream()
    comm = torch.cuda.Stream()
    compute.wait_stream(torch.cuda.current_stream())
    st = tpd.gemm_run_chunked(h, chunks, M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, None, N, D.data_ptr(), N, 1.0,
                              0.0, tpd.OUT_BF16, [e.cuda_event for e in evs], compute.cuda_stream)
    assert st == tpd.OK
    b = _bounds(M, chunks)
    with torch.cuda.stream(comm):
        for i, e in enumerate(evs):
            comm.wait_event(e)
            sent[b[i]:b[i + 1]].copy_(D[b[i]:b[i + 1]])
    torch.cuda.synchronize()
    want = oracle_out(A, B, None, 1.0, 0.0, torch.bfloat16)
    assert_bit_exact(bits(sent), want, "rows received by the communication stream")


def test_chunked_argument_errors(h):
    A = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((256, 64), device="cuda")
    evs = _events(2)
    s = torch.cuda.current_stream().cuda_stream
    args = (256, 64, 64, A.data_ptr(), 64, B.data_ptr(), 64, None, 64, D.data_ptr(), 64, 1.0, 0.0, tpd.OUT_F32)
    assert tpd.gemm_run_chunked(h, 0, *args, [], s) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_run_chunked(h, 65, *args, [evs[0].cuda_event] * 65, s) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_run_chunked(h, 2, *args, [evs[0].cuda_event, 0], s) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_run_chunked(h, 2, *args, [e.cuda_event for e in evs], s) == tpd.OK
    assert tpd.gemm_sync_status(h, None) == tpd.OK
