"""The library's calls recorded into a CUDA graph (after a first eager call
on the same stream, which builds the descriptors and any workspace) replay
with the same results as eager calls: dense two-consumer, small-M (whole
tiles and cluster split) and grouped launches, all in one graph."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_tensor_core_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from blackwell_tensor_core_gb300 import build
    build.build()


def test_calls_replay_from_a_cuda_graph():
    from blackwell_tensor_core_gb300 import ops
    dev = torch.device("cuda")
    g = wl.generator(9500)
    shapes = [(1024, 2048, 512), (72, 16384, 256), (72, 4096, 1024)]
    mats = [(wl.randint_matrix(M, K, -2, 2, g).to(dev), wl.randint_matrix(K, N, -2, 2, g).to(dev))
            for (M, N, K) in shapes]
    counts = [300, 0, 700]
    off = torch.from_numpy(wl.offsets_from_counts(counts)).to(dev)
    Ag = wl.randint_matrix(1000, 256, -2, 2, g).to(dev)
    Bg = [wl.randint_matrix(256, 512, -2, 2, g).to(dev) for _ in counts]
    s = torch.cuda.Stream()
    outs = [torch.empty((M, N), dtype=torch.float32, device=dev) for (M, N, K) in shapes]
    Dg = torch.empty((1000, 512), dtype=torch.bfloat16, device=dev)

    def work():
        for (A, B), D in zip(mats, outs):
            ops.gemm(A, B, out=D, stream=torch.cuda.current_stream())
        ops.grouped_gemm(Ag, Bg, off, out=Dg, stream=torch.cuda.current_stream())

    with torch.cuda.stream(s):
        work()  # eager first: descriptors, device state
    torch.cuda.synchronize()
    eager = [D.clone() for D in outs] + [Dg.clone()]
    for D in outs:
        D.zero_()
    Dg.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        work()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        st, word = ops.last_device_error()
        assert st == 0, hex(word)
        for D, E in zip(outs + [Dg], eager):
            assert torch.equal(D, E)
    for (A, B), D in zip(mats, outs):
        ref, _ = oracle.gemm(wl.bits(A.cpu()), wl.bits(B.cpu()))
        assert np.array_equal(D.cpu().double().numpy(), ref)
