"""The library's launches captured into CUDA graphs and replayed.

A gemm_run launch enqueues only kernels on the caller's stream, so it can be captured once
the first call on that device has set its kernel attributes.  Each test captures GEMMs
with torch.cuda.graph, changes the inputs in place, replays, and compares with the oracle
bit for bit (integer inputs).
"""
import numpy as np
import pytest
import torch

from dense_tiled_gemm_04_gb300 import native
from dense_tiled_gemm_04_gb300.workloads import make_inputs

import oracle
from test_gpu_parity import assert_exact, codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_tiled_gemm_04_gb300 import build

    build.build()
    oracle.build()
    h = native.Gemm(0)
    yield h
    h.close()


@pytest.mark.parametrize("config", [native.CONFIG_AUTO, native.CONFIG_128x128, native.CONFIG_128x64,
                                    native.CONFIG_256x256])
def test_gemm_run_captured_and_replayed(g, config):
    M, N, K = 1100, 1000, 1800  # several tiles, a part-empty last wave: stream-K in the graph too
    A, B = make_inputs(M, N, K, "TN", "bf16", "int", seed=301)
    A2, _ = make_inputs(M, N, K, "TN", "bf16", "int", seed=302)
    dA, dB = A.cuda(), B.cuda()
    C = native.empty_output(M, N, torch.bfloat16, "cuda")
    g.set_option(native.OPT_CONFIG, config)
    try:
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            g.run(dA, dB, C, layout="TN")          # first call: kernel attributes, tensor maps
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.run(dA, dB, C, layout="TN")          # enqueued on the capture stream
        dA.copy_(A2.cuda())
        C.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert g.sync_status() == native.OK
        assert_exact(codes(C), oracle.gemm(A2, B, "TN", "bf16"), f"replay cfg{config}")
        dA.copy_(A.cuda())
        graph.replay()
        torch.cuda.synchronize()
        assert_exact(codes(C), oracle.gemm(A, B, "TN", "bf16"), f"second replay cfg{config}")
    finally:
        g.set_option(native.OPT_CONFIG, native.CONFIG_AUTO)


def test_chain_of_gemms_in_one_graph(g):
    # C1 = A·B, C2 = C1·B2 in one graph: the second reads what the first wrote.
    M, N, K, N2 = 640, 512, 384, 256
    A, B = make_inputs(M, N, K, "NN", "f16", "int", seed=303)
    _, B2 = make_inputs(M, N2, N, "NN", "f16", "int", seed=304)
    dA, dB, dB2 = A.cuda(), B.cuda(), B2.cuda()
    C1 = native.empty_output(M, N, torch.float16, "cuda")
    C2 = native.empty_output(M, N2, torch.float16, "cuda")
    g.run(dA, dB, C1, layout="NN")
    g.run(C1, dB2, C2, layout="NN")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.run(dA, dB, C1, layout="NN")
        g.run(C1, dB2, C2, layout="NN")
    dA.neg_()
    graph.replay()
    torch.cuda.synchronize()
    ref1 = oracle.gemm((-A.float()).to(torch.float16), B, "NN", "f16")
    assert_exact(codes(C1), ref1, "C1")
    c1 = torch.from_numpy(ref1.view(np.int16)).view(torch.float16)
    assert_exact(codes(C2), oracle.gemm(c1, B2, "NN", "f16"), "C2")
