"""Guard bands: no kernel writes outside the buffers it is given.

Every output buffer -- the activation quantizer's Qx, s_x, t_x and
activation operand, the GEMM's fp16 O or int32 accumulators, and its
workspace beyond the bytes the planner asked for -- is placed inside a larger
allocation whose bytes before and after it hold a sentinel pattern.  After
tile-size and stream-K variants of both tensor-core paths, and after
full-size Llama-3-8B and Qwen1.5-72B GEMMs in the benchmark's launch
configuration, every guard byte must still hold the sentinel, and the
results must equal the same calls on unguarded buffers.
"""
import numpy as np
import pytest

import w4a8_quantized_serving_qoq_gb300 as qoq
from w4a8_quantized_serving_qoq_gb300 import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096          # bytes on each side; keeps the inner buffer 256-byte aligned
SENTINEL = 0xA5


class Guarded:
    """`nbytes` of device memory between two sentinel bands."""

    def __init__(self, nbytes):
        self.nbytes = int(nbytes)
        inner = (self.nbytes + 255) // 256 * 256
        self.buf = torch.full((GUARD + inner + GUARD,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.raw = self.buf[GUARD:GUARD + self.nbytes]

    def view(self, dtype, shape):
        return self.raw.view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        lo = self.buf[:GUARD]
        hi = self.buf[GUARD + self.nbytes:]
        return bool((lo == SENTINEL).all()) and bool((hi == SENTINEL).all())


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _weights(N, K, seed):
    """Packed g128 weights made on the device (the device quantizer is checked
    bit-exact against the oracle elsewhere); only the guards matter here."""
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    W = (torch.randn((N, K), generator=gen, device=DEV) * 0.02).to(torch.float16)
    wq = qoq.qoq_quantize_weights(W, 128)
    return qoq.qoq_pack_weights(wq["q4"], wq["s_g"], wq["z"], 128), wq["s_w"]


def _run(X, packed, sw, N, opt_kw, guarded):
    """Quantizer (with the activation operand of the GEMM's path) then GEMM,
    into guarded or plain buffers; returns (O, acc, guards)."""
    M, K = X.shape
    opt0 = qoq.gemm_options(**opt_kw)
    kind = qoq.qoq_gemm_path(M, N, K, 128, opt0)
    sizes = dict(Qx=M * K, sx=2 * M, tx=4 * M, act=qoq.qoq_act_operand_bytes(M, K, kind),
                 O=2 * M * N, acc=4 * M * N, ws=qoq.qoq_gemm_workspace_bytes(M, N, K, 128, opt0))
    if guarded:
        g = {k: Guarded(v) for k, v in sizes.items()}
        bufs = dict(Qx=g["Qx"].view(torch.int8, (M, K)), sx=g["sx"].view(torch.float16, (M,)),
                    tx=g["tx"].view(torch.int32, (M,)), act=g["act"].raw,
                    O=g["O"].view(torch.float16, (M, N)), acc=g["acc"].view(torch.int32, (M, N)),
                    ws=g["ws"].raw)
    else:
        g = {}
        bufs = dict(Qx=torch.empty((M, K), dtype=torch.int8, device=DEV),
                    sx=torch.empty((M,), dtype=torch.float16, device=DEV),
                    tx=torch.empty((M,), dtype=torch.int32, device=DEV),
                    act=torch.empty((sizes["act"],), dtype=torch.uint8, device=DEV),
                    O=torch.empty((M, N), dtype=torch.float16, device=DEV),
                    acc=torch.empty((M, N), dtype=torch.int32, device=DEV),
                    ws=torch.empty((sizes["ws"],), dtype=torch.uint8, device=DEV))
    qoq.qoq_workspace_init(bufs["ws"])
    qoq.qoq_quant_act_ex(X, bufs["Qx"], bufs["sx"], bufs["tx"], bufs["act"], kind=kind)
    qoq.qoq_w4a8_gemm_ex(bufs["Qx"], bufs["sx"], None, packed, sw, N, K, 128, O=bufs["O"],
                         workspace=bufs["ws"], options=qoq.gemm_options(act_operand=bufs["act"], **opt_kw))
    qoq.qoq_w4a8_gemm_ex(bufs["Qx"], None, None, packed, None, N, K, 128, workspace=bufs["ws"],
                         options=qoq.gemm_options(acc_out=bufs["acc"], act_operand=bufs["act"], **opt_kw))
    torch.cuda.synchronize()
    assert qoq.qoq_workspace_status(bufs["ws"])[0] == qoq.QOQ_OK
    return bufs, g


def _compare(X, packed, sw, N, opt_kw):
    got, g = _run(X, packed, sw, N, opt_kw, guarded=True)
    bad = [k for k, v in g.items() if not v.intact()]
    assert not bad, f"guard bands overwritten around {bad}"
    ref, _ = _run(X, packed, sw, N, opt_kw, guarded=False)
    for k in ("Qx", "sx", "tx", "act", "acc"):
        assert torch.equal(got[k], ref[k]), k
    assert torch.equal(got["O"].view(torch.int16), ref["O"].view(torch.int16))


@pytest.mark.parametrize("kernel,bt", [(1, 16), (1, 32), (1, 64), (1, 128), (2, 16), (2, 32)])
@pytest.mark.parametrize("ctas", [0, 3, 13])
@pytest.mark.parametrize("publish", [0, 2])
def test_guard_bands_tile_and_stream_k_variants(kernel, bt, ctas, publish):
    M, N, K = 37, 384, 1152   # ragged token tail, 9 groups, split tiles at 3 and 13 CTAs
    X = _t(synthetic.activations(M, K, 88, 4))
    packed, sw = _weights(N, K, 89)
    _compare(X, packed, sw, N, dict(kernel=kernel, tokens_per_tile=bt, num_ctas=ctas, debug_flags=publish))


@pytest.mark.parametrize("M", [1, 5, 17, 64, 130, 256])
def test_guard_bands_automatic_plan(M):
    N, K = 1024, 2048
    X = _t(synthetic.activations(M, K, 90 + M, 4))
    packed, sw = _weights(N, K, 91)
    _compare(X, packed, sw, N, {})


@pytest.mark.parametrize("workload,name,M", [(1, "o", 1), (1, "qkv", 64), (1, "gate_up", 256),
                                             (1, "down", 32), (2, "o", 4096), (3, "down", 64)])
def test_guard_bands_full_size(workload, name, M):
    layers = {l.name: l for l in synthetic.WORKLOADS[workload][1]}
    layer = layers[name]
    _, _, _, _, _, xo, _ = synthetic.WORKLOADS[workload]
    X = _t(synthetic.activations(M, layer.K, synthetic.layer_seed(workload, layer), xo))
    packed, sw = _weights(layer.N, layer.K, 92)
    _compare(X, packed, sw, layer.N, {})
