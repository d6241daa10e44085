"""Parity at the full workload sizes, in the launch configuration the
benchmark uses (automatic tile size and persistent-CTA count).

The oracle quantizes the full weight matrix and the activations (so the
device GEMM is checked on oracle-made codes), then computes the int32
accumulators at sampled (m, n) positions and whole rows; the device must
match them bit for bit, and its fp16 output must meet the row tolerance on
the whole rows.  The device quantizers are checked bit-exact against the
oracle's codes for the full matrices.
"""
import functools

import numpy as np
import pytest

import oracle
import w4a8_quantized_serving_qoq_gb300 as qoq
from w4a8_quantized_serving_qoq_gb300 import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"

LLAMA = {l.name: l for l in synthetic.LLAMA3_8B}
QWEN = {l.name: l for l in synthetic.QWEN_72B}


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@functools.lru_cache(maxsize=2)
def _weights(workload: int, name: str, group: int):
    layers = QWEN if workload == 3 else LLAMA
    layer = layers[name]
    _, _, _, sigma, wo, _, _ = synthetic.WORKLOADS[workload]
    W = synthetic.weights(layer.N, layer.K, synthetic.layer_seed(workload, layer), sigma, wo)
    wq = oracle.quantize_weights_group(W, 128) if group else oracle.quantize_weights_channel(W)
    return layer, W, wq


def _check_point(workload, name, M, group=128, check_quantizer=False):
    layer, W, wq = _weights(workload, name, group)
    _, _, _, _, _, xo, _ = synthetic.WORKLOADS[workload]
    X = synthetic.activations(M, layer.K, synthetic.layer_seed(workload, layer), xo)
    Qx, sx, tx = oracle.quant_act(X)
    N, K = layer.N, layer.K
    packed = qoq.qoq_pack_weights(_t(wq["q4"]), _t(wq["s_g"]) if group else None, _t(wq["z"]), group)
    sw = _t(wq["s_w"])
    # device activation quantizer (with the fp8-path activation operand, as
    # the benchmark calls it), bit-exact at full size
    Qx_d, sx_d, tx_d, act_d = qoq.qoq_quant_act_ex(_t(X), kind=qoq.qoq_gemm_path(M, N, K, group))
    torch.cuda.synchronize()
    assert np.array_equal(Qx_d.cpu().numpy(), Qx)
    assert np.array_equal(sx_d.cpu().numpy().view(np.uint16), sx.view(np.uint16))
    assert np.array_equal(tx_d.cpu().numpy(), tx)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    qoq.qoq_w4a8_gemm_ex(Qx_d, None, tx_d, packed, None, N, K, group,
                         options=qoq.gemm_options(acc_out=acc, act_operand=act_d))
    O = qoq.qoq_w4a8_gemm_ex(Qx_d, sx_d, tx_d, packed, sw, N, K, group,
                             options=qoq.gemm_options(act_operand=act_d))
    O_plain = qoq.qoq_w4a8_gemm(Qx_d, sx_d, tx_d, packed, sw, N, K, group)
    torch.cuda.synchronize()
    assert torch.equal(O, O_plain)  # operand from the quantizer == operand built by the GEMM
    acc = acc.cpu().numpy()
    O = O.cpu().numpy().astype(np.float64)

    rng = np.random.default_rng(M * 7919 + N)
    ms = np.concatenate([rng.integers(0, M, 200), [0, M - 1, M - 1, 0]]).astype(np.int32)
    ns = np.concatenate([rng.integers(0, N, 200), [0, N - 1, 0, N - 1]]).astype(np.int32)
    if group:
        ref = oracle.gemm_i32_group_at(Qx, wq["q4"], wq["s_g"], wq["z"], ms, ns)
    else:
        ref = oracle.gemm_i32_channel_at(Qx, tx, wq["q4"], wq["z"], ms, ns)
    assert np.array_equal(acc[ms, ns], ref)

    # whole rows for the fp16 tolerance (row maximum needs the full row)
    for m in sorted({0, M - 1}):
        mm = np.full(N, m, np.int32)
        nn = np.arange(N, dtype=np.int32)
        if group:
            row = oracle.gemm_i32_group_at(Qx, wq["q4"], wq["s_g"], wq["z"], mm, nn)
        else:
            row = oracle.gemm_i32_channel_at(Qx, tx, wq["q4"], wq["z"], mm, nn)
        assert np.array_equal(acc[m], row)
        O_ref = oracle.epilogue_f64(row[None, :], sx[m:m + 1], wq["s_w"])
        assert oracle.o_within_tolerance(O[m:m + 1], O_ref).all()

    if check_quantizer:
        d = qoq.qoq_quantize_weights(_t(W), group)
        torch.cuda.synchronize()
        assert np.array_equal(d["q4"].cpu().numpy(), wq["q4"])
        assert np.array_equal(d["z"].cpu().numpy(), wq["z"])
        assert np.array_equal(d["s_w"].cpu().numpy().view(np.uint16), wq["s_w"].view(np.uint16))
        if group:
            assert np.array_equal(d["s_g"].cpu().numpy(), wq["s_g"])


# Every configuration point of the four full-size workloads.  Points are
# ordered layer by layer so that each layer's oracle-quantized weights are
# made once (the cache above holds the last two).
DECODE_POINTS = [(name, M) for name in ("qkv", "o", "gate_up", "down") for M in synthetic.DECODE_MS]
QWEN_POINTS = [(name, M) for name in ("gate_up", "down") for M in synthetic.QWEN_MS]


@pytest.mark.parametrize("name,M", DECODE_POINTS)
def test_llama_decode_full_size(name, M):
    _check_point(1, name, M, check_quantizer=(M == synthetic.DECODE_MS[0]))


@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
def test_llama_prefill_full_size(name):
    _check_point(2, name, synthetic.PREFILL_M)


@pytest.mark.parametrize("name,M", QWEN_POINTS)
def test_qwen_full_size(name, M):
    _check_point(3, name, M, check_quantizer=(M == synthetic.QWEN_MS[0]))


@pytest.mark.parametrize("M", synthetic.CHANNEL_MS)
def test_per_channel_gate_up_full_size(M):
    _check_point(4, "gate_up", M, group=0, check_quantizer=(M == synthetic.CHANNEL_MS[0]))
