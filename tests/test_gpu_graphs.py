"""The library's launches captured into CUDA graphs and replayed.

A launch enqueues only kernels (and, for the no-allocation entry point, one memset) on the
caller's stream, so it can be captured once the first call on that device has set its
kernel attributes.  Each test captures GEMMs with torch.cuda.graph, changes the inputs in
place, replays, and compares with the oracle bit for bit (integer inputs).
"""
import ctypes

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


@pytest.mark.parametrize("config", [native.CONFIG_AUTO, native.CONFIG_128x128, native.CONFIG_256x256,
                                    native.CONFIG_512x256])
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


def test_noalloc_entry_point_captured_and_replayed(g):
    lib = native.load()
    M, N, K = 512, 768, 640
    A, B = make_inputs(M, N, K, "TN", "f16", "int", seed=305)
    A2, _ = make_inputs(M, N, K, "TN", "f16", "int", seed=306)
    dA, dB = A.cuda(), B.cuda()
    C = native.empty_output(M, N, torch.float16, "cuda")

    def call():
        s = torch.cuda.current_stream().cuda_stream
        return lib.gemm_run_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, dA.stride(0),
                                    dB.stride(0), C.stride(0), native.LAYOUT_TN, native.DTYPE_F16, s or None, None)

    assert call() == native.OK                    # first call on this device: before any capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert call() == native.OK
    dA.copy_(A2.cuda())
    graph.replay()
    torch.cuda.synchronize()
    assert_exact(codes(C), oracle.gemm(A2, B, "TN", "f16"), "no-alloc replay")
    info = (ctypes.c_int32 * 4)()
    assert lib.gemm_run_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, dA.stride(0), dB.stride(0),
                                C.stride(0), native.LAYOUT_TN, native.DTYPE_F16, None, info) == native.OK
