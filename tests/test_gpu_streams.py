"""GPU: the library on several streams, inside CUDA graphs and from several
host threads.  Every call enqueues on the stream it is given and touches only
the caller's buffers, so concurrent products with separate workspaces, graph
replays and calls from other threads must give the bits of plain serial
calls (the run-to-run determinism of the Tencent AI-infra article's "背景"
carried to concurrent use)."""
import threading

import pytest
import torch

import deterministic_invariant_gemm_gb300 as dig
import workloads
from gemm_check import bits_equal

pytestmark = pytest.mark.gpu

# (M, N, K, split_k): decode-like, ragged, folded-size and unsplit products, and
# a small long-K product on narrow (64-column) tiles
CASES = [(16, 4096, 4096, 8), (300, 600, 1000, 3), (1024, 4096, 2048, 4), (256, 512, 1536, 1),
         (64, 256, 16384, 8)]


@pytest.fixture(scope="module", autouse=True)
def _device(cuda_device):
    dig.load()
    yield
    assert dig.bigemm_device_status(reset=True) == 0


def inputs():
    out = []
    for i, (M, N, K, S) in enumerate(CASES):
        A, B = workloads.pair(M, N, K, 900 + i)
        out.append((A.cuda(), B.cuda(), S))
    return out


def serial(data):
    res = [dig.matmul(A, B, split_k=S) for A, B, S in data]
    torch.cuda.synchronize()
    return res


def test_concurrent_streams_match_serial_calls():
    data = inputs()
    want = serial(data)
    streams = [torch.cuda.Stream() for _ in data]
    outs = [torch.empty_like(w) for w in want]
    wss = [torch.empty(max(dig.bigemm_workspace_bytes(A.shape[0], B.shape[1], A.shape[1], S), 16),
                       dtype=torch.uint8, device="cuda") for A, B, S in data]
    torch.cuda.synchronize()
    for rep in range(3):
        for (A, B, S), C, ws, st in zip(data, outs, wss, streams):
            with torch.cuda.stream(st):
                dig.matmul(A, B, split_k=S, out=C, workspace=ws, stream=st)
        torch.cuda.synchronize()
        for C, w in zip(outs, want):
            assert bits_equal(C, w), rep


def test_graph_replays_match_eager_calls():
    data = inputs()
    want = serial(data)
    outs = [torch.empty_like(w) for w in want]
    wss = [torch.empty(max(dig.bigemm_workspace_bytes(A.shape[0], B.shape[1], A.shape[1], S), 16),
                       dtype=torch.uint8, device="cuda") for A, B, S in data]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (A, B, S), C, ws in zip(data, outs, wss):
            dig.matmul(A, B, split_k=S, out=C, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(5):
        for C in outs:
            C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for C, w in zip(outs, want):
            assert bits_equal(C, w), rep


def test_calls_from_two_host_threads():
    data = inputs()
    want = serial(data)
    errors = []

    def worker(idx):
        try:
            st = torch.cuda.Stream()
            for _ in range(4):
                with torch.cuda.stream(st):
                    got = [dig.matmul(A, B, split_k=S, stream=st) for A, B, S in data]
                st.synchronize()
                for g, w in zip(got, want):
                    if not bits_equal(g, w):
                        errors.append("thread %d: bits differ" % idx)
        except Exception as e:  # reported below
            errors.append("thread %d: %r" % (idx, e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_default_stream_is_torchs_current_stream():
    """stream=None means torch's current stream, read through its raw
    accessor: the same handle as torch.cuda.current_stream(), inside and
    outside a stream context."""
    assert dig._current_raw_stream() == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert dig._current_raw_stream() == s.cuda_stream
    assert dig._current_raw_stream() == torch.cuda.current_stream().cuda_stream
