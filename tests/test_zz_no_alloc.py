"""The allocation-free GEMM entry point (qoq_w4a8_gemm_noalloc).

It serves callers that cannot allocate device memory (a plugin handed only
its input and output buffers, or a path that must not call cudaMalloc
because it can synchronize the device): its scratch is a fixed array inside
the library.  This file runs last so that a failure here leaves every other
test already run; it passes alone in a fresh process or after the others.
"""
import ctypes

import numpy as np
import pytest

import oracle
import w4a8_quantized_serving_qoq_gb300 as qoq
from w4a8_quantized_serving_qoq_gb300 import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def _case(M, N, K, seed):
    W = synthetic.weights(N, K, seed, 0.02, 2)
    X = synthetic.activations(M, K, seed, 4)
    wq = oracle.quantize_weights_group(W, 128)
    Qx, sx, tx = oracle.quant_act(X)
    packed = qoq.qoq_pack_weights(_t(wq["q4"]), _t(wq["s_g"]), _t(wq["z"]), 128)
    return _t(Qx), _t(sx), packed, _t(wq["s_w"])


@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (64, 4096, 4096), (1, 1024, 14336)])
def test_noalloc_matches_workspace_entry_point_twice(M, N, K):
    lib = qoq.load()
    Qx, sx, packed, sw = _case(M, N, K, 500 + M)
    ref = qoq.qoq_w4a8_gemm(Qx, sx, None, packed, sw, N, K, 128)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # the shared scratch must be usable again right after a call
        O = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        st = lib.qoq_w4a8_gemm_noalloc(
            ctypes.c_void_p(Qx.data_ptr()), ctypes.c_void_p(sx.data_ptr()), None,
            ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sw.data_ptr()), M, N, K, 128,
            ctypes.c_void_p(O.data_ptr()), stream)
        assert st == 0, qoq.qoq_status_string(st)
        torch.cuda.synchronize()
        ok = oracle.o_within_tolerance(O.cpu().numpy().astype(np.float64),
                                       ref.cpu().numpy().astype(np.float64))
        assert ok.all()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = qoq.load()
    # many weight tiles keep 128-token tiles, whose partial slots need more than 8 MiB of scratch
    M, N, K = 256, 16384, 4096
    assert qoq.qoq_gemm_workspace_bytes(M, N, K, 128) > (8 << 20)
    # any valid packed weights and activations: the call must be refused before running
    q4, sg, z = synthetic.random_codes(N, K, 7)
    packed = qoq.qoq_pack_weights(_t(q4), _t(sg), _t(z), 128)
    Qx = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.ones((M,), dtype=torch.float16, device="cuda")
    sw = torch.ones((N,), dtype=torch.float16, device="cuda")
    O = torch.empty((M, N), dtype=torch.float16, device="cuda")
    st = lib.qoq_w4a8_gemm_noalloc(
        ctypes.c_void_p(Qx.data_ptr()), ctypes.c_void_p(sx.data_ptr()), None,
        ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sw.data_ptr()), M, N, K, 128,
        ctypes.c_void_p(O.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4  # QOQ_ERR_WORKSPACE
