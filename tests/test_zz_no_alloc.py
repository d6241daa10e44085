"""The allocation-free GEMM entry point (qoq_w4a8_gemm_noalloc).

It serves callers that cannot allocate device memory (a plugin handed only
its input and output buffers, or a path that must not call cudaMalloc
because it can synchronize the device): its scratch is a fixed array inside
the library.  Each call's output is checked against the oracle's fp64
epilogue and against the workspace entry point (qoq_w4a8_gemm), and the
array's device status word is read back after each call.  This file runs
last so that a failure here leaves every other test already run; it passes
alone in a fresh process or after the others.
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
    Qx, sx, _ = oracle.quant_act(X)
    packed = qoq.qoq_pack_weights(_t(wq["q4"]), _t(wq["s_g"]), _t(wq["z"]), 128)
    O_ref = oracle.epilogue_f64(oracle.gemm_i32_group(Qx, wq["q4"], wq["s_g"], wq["z"]), sx, wq["s_w"])
    return _t(Qx), _t(sx), packed, _t(wq["s_w"]), O_ref


def _call(lib, Qx, sx, packed, sw, M, N, K, O):
    return lib.qoq_w4a8_gemm_noalloc(
        ctypes.c_void_p(Qx.data_ptr()), ctypes.c_void_p(sx.data_ptr()), None,
        ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(sw.data_ptr()), M, N, K, 128,
        ctypes.c_void_p(O.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (64, 4096, 4096), (1, 1024, 14336)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(M, N, K):
    lib = qoq.load()
    Qx, sx, packed, sw, O_ref = _case(M, N, K, 500 + M)
    ref = qoq.qoq_w4a8_gemm(Qx, sx, None, packed, sw, N, K, 128)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy().astype(np.float64)
    for _ in range(2):  # the shared scratch must be usable again right after a call
        O = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        st = _call(lib, Qx, sx, packed, sw, M, N, K, O)
        assert st == 0, qoq.qoq_status_string(st)
        st, bits = qoq.qoq_noalloc_status()  # synchronizes the stream
        assert (st, bits) == (0, 0)
        got = O.cpu().numpy().astype(np.float64)
        assert oracle.o_within_tolerance(got, O_ref).all()
        assert oracle.o_within_tolerance(got, ref).all()


def test_noalloc_reports_bad_packed_weights_through_its_status():
    lib = qoq.load()
    M, N, K = 16, 256, 512
    Qx, sx, packed, sw, _ = _case(M, N, K, 77)
    # packed holds N = 256 rows; a call with N = 128 (every buffer sized for
    # that call) must be refused on the device: no output, status bit 2
    O = torch.zeros((M, N - 128), dtype=torch.float16, device="cuda")
    assert _call(lib, Qx, sx, packed, sw, M, N - 128, K, O) == 0
    st, bits = qoq.qoq_noalloc_status()
    assert st == 7 and bits & 2  # QOQ_ERR_DEVICE
    assert float(O.abs().max()) == 0.0
    assert qoq.qoq_noalloc_status() == (0, 0)  # the read cleared the word
    O = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert _call(lib, Qx, sx, packed, sw, M, N, K, O) == 0
    assert qoq.qoq_noalloc_status() == (0, 0)


@pytest.mark.parametrize("M,N,K", [(256, 16384, 4096), (64, 8192, 29568)])
def test_noalloc_rejects_shapes_beyond_its_scratch(M, N, K):
    lib = qoq.load()
    # the need depends on the shape: 128-token tiles over many weight tiles, or
    # a long K with 64-token tiles (Qwen1.5-72B down at M = 64)
    assert qoq.qoq_gemm_workspace_bytes(M, N, K, 128) > (8 << 20)
    # buffers of the right sizes; the call must be refused before running
    packed = torch.zeros((qoq.qoq_packed_weight_bytes(N, K, 128),), dtype=torch.uint8, device="cuda")
    Qx = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.ones((M,), dtype=torch.float16, device="cuda")
    sw = torch.ones((N,), dtype=torch.float16, device="cuda")
    O = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert _call(lib, Qx, sx, packed, sw, M, N, K, O) == 4  # QOQ_ERR_WORKSPACE
