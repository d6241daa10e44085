"""GPU parity of the fused norm / activation + quantization kernels.

qoq_rmsnorm_quant_act and qoq_silu_mul_quant_act compute an fp16 row (RMS
norm of X, or SiLU(G) * U) in fp32 and quantize it per token.  Checked
against the oracle in two parts:
  * the fp16 rows the quantizer saw (the test-mode output Y) are within one
    fp16 ulp of the oracle's fp64 norm / activation, element by element (the
    bound of a row rounded to fp16 from an fp32 computation, whose relative
    error is far below the 2^-11 of the rounding itself);
  * Qx, s_x and t_x equal the oracle's quantizer applied to those fp16 rows,
    bit for bit, and the activation operand equals what qoq_quant_act_ex
    writes for them (that operand is checked against its format text in the
    parity tests).
"""
import numpy as np
import pytest

import oracle
import w4a8_quantized_serving_qoq_gb300 as qoq
from w4a8_quantized_serving_qoq_gb300 import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _np(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def _check_quantized(Y16, Qx, sx, tx, act, kind):
    Qx_r, sx_r, tx_r = oracle.quant_act(Y16)
    assert np.array_equal(_np(Qx), Qx_r)
    assert np.array_equal(_np(sx).view(np.uint16), sx_r.view(np.uint16))
    assert np.array_equal(_np(tx), tx_r)
    if act is not None:
        _, _, _, act_ref = qoq.qoq_quant_act_ex(_t(Y16), kind=kind)
        assert torch.equal(act, act_ref)


def _gamma(K, seed):
    return (1.0 + 0.2 * np.random.default_rng(seed).standard_normal(K)).astype(np.float16)


@pytest.mark.parametrize("M,K", [(1, 4096), (5, 1024), (16, 4096), (129, 256), (300, 14336), (3, 8), (2, 29568),
                                 (2003, 384), (600, 4096), (297, 29568)])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_rmsnorm_quant_matches_oracle(M, K, kind):
    if kind and K % 128:
        pytest.skip("an activation operand needs K % 128 == 0")
    X = synthetic.activations(M, K, 600 + M, 4)
    if M > 2:
        X[1] = 0                      # an all-zero row
    gamma = _gamma(K, 601 + K)
    eps = 1e-5
    Qx, sx, tx, act, Y = qoq.qoq_rmsnorm_quant_act(_t(X), _t(gamma), eps, kind=max(kind, 1), with_act=kind > 0,
                                                   with_y=True)
    Y16 = _np(Y)
    ref = oracle.rmsnorm_f64(X, gamma, eps)
    assert oracle.fp16_within_one_ulp(Y16.astype(np.float64), ref).all()
    _check_quantized(Y16, Qx, sx, tx, act, kind)
    # the same call without the test-mode output gives the same codes
    Qx2, sx2, tx2, _, _ = qoq.qoq_rmsnorm_quant_act(_t(X), _t(gamma), eps, with_act=False)
    assert torch.equal(Qx, Qx2) and torch.equal(sx, sx2) and torch.equal(tx, tx2)


def test_rmsnorm_quant_zero_row_without_eps_and_constant_rows():
    K = 512
    X = np.zeros((3, K), np.float16)
    X[1] = 0.5                        # constant row: normalizes to 1 * gamma
    X[2, 3] = -2.0                    # lone value: -sqrt(K) * gamma
    gamma = np.ones(K, np.float16)
    Qx, sx, tx, _, Y = qoq.qoq_rmsnorm_quant_act(_t(X), _t(gamma), 0.0, with_act=False, with_y=True)
    Y16 = _np(Y).astype(np.float64)
    assert not Y16[0].any() and (_np(Qx)[0] == 0).all() and float(_np(sx)[0]) == 0.0
    assert (Y16[1] == 1.0).all()
    assert Y16[2, 3] == np.float16(-np.sqrt(K)) and np.count_nonzero(Y16[2]) == 1
    _check_quantized(_np(Y), Qx, sx, tx, None, 0)


def _gate_up(M, F, seed):
    rng = np.random.default_rng(seed)
    G = (rng.standard_normal((M, F)) * 3.0).astype(np.float16)
    U = rng.standard_normal((M, F)).astype(np.float16)
    G[0, :6] = [0.0, 30.0, -30.0, -90.0, 11.0, -0.25]   # zero, both tails, e^-g overflow
    U[0, :6] = [1.0, 1.0, 2.0, 3.0, -4.0, 0.5]
    return np.concatenate([G, U], axis=1)


@pytest.mark.parametrize("M,F", [(1, 14336), (7, 1024), (32, 128), (256, 14336), (300, 2048), (2, 8),
                                 (1999, 1024), (320, 14336), (300, 29568)])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_silu_mul_quant_matches_oracle(M, F, kind):
    if kind and F % 128:
        pytest.skip("an activation operand needs F % 128 == 0")
    H = _gate_up(M, F, 700 + M + F)
    Qx, sx, tx, act, Y = qoq.qoq_silu_mul_quant_act(_t(H), kind=max(kind, 1), with_act=kind > 0, with_y=True)
    Y16 = _np(Y)
    ref = oracle.silu_mul_f64(H)
    assert oracle.fp16_within_one_ulp(Y16.astype(np.float64), ref).all()
    _check_quantized(Y16, Qx, sx, tx, act, kind)
    Qx2, sx2, tx2, _, _ = qoq.qoq_silu_mul_quant_act(_t(H), with_act=False)
    assert torch.equal(Qx, Qx2) and torch.equal(sx, sx2) and torch.equal(tx, tx2)


@pytest.mark.parametrize("M", [1, 32, 128])
def test_fused_quant_feeds_the_gemm(M):
    """norm + quant -> gate_up GEMM -> SiLU-mul + quant -> down GEMM, chained
    with launch overlap, equals the oracle on the fp16 rows each quantizer
    saw (the FFN of one Llama-style block, scaled down)."""
    K, F = 512, 384
    X = synthetic.activations(M, K, 800 + M, 4)
    gamma = _gamma(K, 801)
    Wg = synthetic.weights(2 * F, K, 802, 0.02, 2)
    Wd = synthetic.weights(K, F, 803, 0.02, 2)
    wg = oracle.quantize_weights_group(Wg, 128)
    wd = oracle.quantize_weights_group(Wd, 128)
    pg = qoq.qoq_pack_weights(_t(wg["q4"]), _t(wg["s_g"]), _t(wg["z"]), 128)
    pd = qoq.qoq_pack_weights(_t(wd["q4"]), _t(wd["s_g"]), _t(wd["z"]), 128)
    flags = qoq.QOQ_LAUNCH_OVERLAP
    kg = qoq.qoq_gemm_path(M, 2 * F, K, 128)
    Qx, sx, _, act, Y = qoq.qoq_rmsnorm_quant_act(_t(X), _t(gamma), 1e-5, kind=kg, with_t=False, with_y=True,
                                                  flags=flags)
    H = qoq.qoq_w4a8_gemm_ex(Qx, sx, None, pg, _t(wg["s_w"]), 2 * F, K, 128,
                             options=qoq.gemm_options(act_operand=act, flags=flags))
    kd = qoq.qoq_gemm_path(M, K, F, 128)
    Qa, sa, _, act2, A = qoq.qoq_silu_mul_quant_act(H, kind=kd, with_t=False, with_y=True, flags=flags)
    O = qoq.qoq_w4a8_gemm_ex(Qa, sa, None, pd, _t(wd["s_w"]), K, F, 128,
                             options=qoq.gemm_options(act_operand=act2, flags=flags))
    # first GEMM against the oracle on the normalized rows
    Qx_r, sx_r, _ = oracle.quant_act(_np(Y))
    H_ref = oracle.epilogue_f64(oracle.gemm_i32_group(Qx_r, wg["q4"], wg["s_g"], wg["z"]), sx_r, wg["s_w"])
    H16 = _np(H)
    assert oracle.o_within_tolerance(H16.astype(np.float64), H_ref).all()
    # the activation kernel on the GEMM's own fp16 output, then the second GEMM
    assert oracle.fp16_within_one_ulp(_np(A).astype(np.float64), oracle.silu_mul_f64(H16)).all()
    Qa_r, sa_r, _ = oracle.quant_act(_np(A))
    assert np.array_equal(_np(Qa), Qa_r)
    O_ref = oracle.epilogue_f64(oracle.gemm_i32_group(Qa_r, wd["q4"], wd["s_g"], wd["z"]), sa_r, wd["s_w"])
    assert oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref).all()


def test_fused_quant_argument_errors():
    X = torch.zeros((4, 256), dtype=torch.float16, device=DEV)
    g = torch.ones((256,), dtype=torch.float16, device=DEV)
    with pytest.raises(qoq.QoqError) as e:
        qoq.qoq_rmsnorm_quant_act(X, g, -1.0)
    assert e.value.status == 1
    with pytest.raises(qoq.QoqError) as e:
        qoq.qoq_rmsnorm_quant_act(X, g, float("nan"))
    assert e.value.status == 1
    with pytest.raises(qoq.QoqError) as e:   # activation operand needs K % 128 == 0
        qoq.qoq_silu_mul_quant_act(torch.zeros((4, 2 * 72), dtype=torch.float16, device=DEV), kind=2)
    assert e.value.status == 2
