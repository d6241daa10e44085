"""GPU parity: every step of the CUDA path against the CPU oracle.

Integers (codes, scales, zeros, packed bytes, int32 accumulators) must match
bit for bit; fp16 outputs must satisfy, per row m,
    |O_gpu - O_ref| <= 2e-3 * max_n |O_ref[m, :]| + ulp16(|O_ref[m, n]|)
against the oracle's fp64 epilogue.
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


def _pack_spec(q4, s_g, z, group):
    """Independent numpy packer written from the packed-format description in
    include/qoq.h (no code shared with the CUDA packer)."""
    N, K = q4.shape
    G = K // 128
    blk = 8192 + (512 if group else 0)
    body = np.zeros((N // 128, G, blk), np.uint8)
    q = q4.reshape(N // 128, 128, G, 4, 4, 8)  # tile, r, group, p, word j, k-in-word
    lo = q[..., :4].astype(np.uint8)
    hi = q[..., 4:].astype(np.uint8)
    byte = (lo & 15) | ((hi & 15) << 4)             # [..., p, j, b]
    # chunk (p*128 + r), 16 bytes = words j (4 bytes b each)
    codes = byte.transpose(0, 2, 3, 1, 4, 5).reshape(N // 128, G, 512 * 16)
    body[:, :, :8192] = codes
    if group:
        csum = q4.reshape(N, G, 128).astype(np.int64).sum(axis=2)          # [N][G]
        meta = np.stack([s_g.reshape(N // 128, 128, G), z.reshape(N // 128, 128, G),
                         (csum & 0xFF).reshape(N // 128, 128, G), (csum >> 8).reshape(N // 128, 128, G)],
                        axis=-1).astype(np.uint8)
        body[:, :, 8192:] = meta.transpose(0, 2, 1, 3).reshape(N // 128, G, 512)
    out = body.reshape(-1)
    if not group:
        zpad = np.zeros((N + 15) // 16 * 16, np.uint8)
        zpad[:N] = z
        out = np.concatenate([out, zpad])
    return out


# ------------------------------------------------------------ quantizers --
@pytest.mark.parametrize("M,K", [(16, 512), (1, 4096), (5, 1024), (129, 256), (300, 14336), (2500, 256),
                                 (1000, 4096)])
def test_quant_act_bit_exact(M, K):
    X = synthetic.activations(M, K, 100 + M, 4)
    X[0, : min(K, 8)] = 0
    if M > 2:
        X[2] = 0  # all-zero row
    Qx_r, sx_r, tx_r = oracle.quant_act(X)
    Qx, sx, tx = qoq.qoq_quant_act(_t(X))
    assert np.array_equal(_np(Qx), Qx_r)
    assert np.array_equal(_np(sx).view(np.uint16), sx_r.view(np.uint16))
    assert np.array_equal(_np(tx), tx_r)


def _act_operand_spec(Qx):
    """The fp8-path activation operand written out from its description in
    include/qoq.h: u = Qx + 128 split into high/low nibble planes, then the
    per-128-k-group sums of Qx as [K/128][Mp] int32 (Mp = M rounded up to 4)."""
    M, K = Qx.shape
    u = Qx.astype(np.int64) + 128
    hi = (u // 16).astype(np.uint8)
    lo = (u % 16).astype(np.uint8)
    Mp = (M + 3) // 4 * 4
    tg = np.zeros((K // 128, Mp), np.int32)
    tg[:, :M] = Qx.astype(np.int64).reshape(M, K // 128, 128).sum(axis=2).T
    return hi, lo, tg


@pytest.mark.parametrize("M,K", [(1, 128), (3, 512), (16, 4096), (17, 1152), (300, 14336), (2501, 256),
                                 (777, 4096)])
@pytest.mark.parametrize("kind", [1, 2])
def test_quant_act_ex_act_operand_bit_exact(M, K, kind):
    X = synthetic.activations(M, K, 300 + M, 4)
    if M > 2:
        X[1] = 0
    Qx_r, sx_r, tx_r = oracle.quant_act(X)
    nbytes = qoq.qoq_act_operand_bytes(M, K, kind)
    Mp = (M + 3) // 4 * 4
    assert nbytes == (2 * M * K if kind == 1 else 2 * M * K + (K // 128) * Mp * 4)
    Qx, sx, tx, act = qoq.qoq_quant_act_ex(_t(X), kind=kind)
    assert np.array_equal(_np(Qx), Qx_r)
    assert np.array_equal(_np(sx).view(np.uint16), sx_r.view(np.uint16))
    assert np.array_equal(_np(tx), tx_r)
    a = _np(act)
    if kind == 1:  # the same integers as fp16
        assert np.array_equal(a.view(np.float16).reshape(M, K).astype(np.float64), Qx_r.astype(np.float64))
        return
    hi, lo, tg = _act_operand_spec(Qx_r)
    assert np.array_equal(a[: M * K].reshape(M, K), hi)
    assert np.array_equal(a[M * K: 2 * M * K].reshape(M, K), lo)
    got_tg = a[2 * M * K:].view(np.int32).reshape(K // 128, Mp)
    assert np.array_equal(got_tg[:, :M], tg[:, :M])
    assert not got_tg[:, M:].any()  # padding columns zero-filled by the last row


@pytest.mark.parametrize("M,K", [(7, 1024), (400, 1024), (310, 14336)])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_quant_act_row_scales_from_subnormal_to_large(M, K, kind):
    """Rows scaled from 1e-7 to 1e3: the fp16 scale s_x runs from zero and
    subnormal values (where the clamp to +-127 acts: max|x| / s_x can exceed
    127 when s_x is a rounded subnormal) to normal ones, and the codes of every
    row (both quantizer kernels, M < 296 and M >= 296; both branches of the
    row-streaming kernel) equal the oracle's bit for bit."""
    rng = np.random.default_rng(4000 + M + K + kind)
    X = rng.standard_normal((M, K))
    scales = 10.0 ** rng.uniform(-7, 3, M)
    scales[:4] = [1e-7, 3e-7, 1.2e-6, 6e-6]     # s_x zero, smallest subnormals
    X = (X * scales[:, None]).astype(np.float16)
    Qx_r, sx_r, tx_r = oracle.quant_act(X)
    assert (sx_r.view(np.uint16)[:M] < 0x0400).any() and (sx_r.view(np.uint16) >= 0x0400).any()
    if kind == 0:
        Qx, sx, tx = qoq.qoq_quant_act(_t(X))
    else:
        Qx, sx, tx, act = qoq.qoq_quant_act_ex(_t(X), kind=kind)
        if kind == 1:
            assert np.array_equal(_np(act).view(np.float16).reshape(M, K).astype(np.float64),
                                  Qx_r.astype(np.float64))
    assert np.array_equal(_np(Qx), Qx_r)
    assert np.array_equal(_np(sx).view(np.uint16), sx_r.view(np.uint16))
    assert np.array_equal(_np(tx), tx_r)


def test_quant_act_ties_half_even():
    row = np.zeros(128, np.float32)
    row[0] = 127 * 0.125
    row[1:7] = np.array([2.5, 3.5, -2.5, -0.5, 1.5, 0.5]) * 0.125
    X = np.stack([row, -row]).astype(np.float16)
    Qx, sx, tx = qoq.qoq_quant_act(_t(X))
    q = _np(Qx)
    assert list(q[0, :7]) == [127, 2, 4, -2, 0, 2, 0]
    assert list(q[1, :7]) == [-127, -2, -4, 2, 0, -2, 0]


@pytest.mark.parametrize("N,K", [(256, 512), (384, 4096), (128, 128)])
def test_quantize_weights_group_bit_exact(N, K):
    W = synthetic.weights(N, K, 7 + N, 0.02, 2)
    W[3] = 0
    ref = oracle.quantize_weights_group(W, 128)
    assert ref["n_overflow"] == 0
    out = qoq.qoq_quantize_weights(_t(W), 128)
    assert np.array_equal(_np(out["q4"]), ref["q4"])
    assert np.array_equal(_np(out["s_g"]), ref["s_g"])
    assert np.array_equal(_np(out["z"]), ref["z"])
    assert np.array_equal(_np(out["s_w"]).view(np.uint16), ref["s_w"].view(np.uint16))


def test_quantize_weights_channel_bit_exact():
    W = synthetic.weights(256, 1024, 31, 0.02, 2)
    W[5] = 0
    ref = oracle.quantize_weights_channel(W)
    out = qoq.qoq_quantize_weights(_t(W), 0)
    assert np.array_equal(_np(out["q4"]), ref["q4"])
    assert np.array_equal(_np(out["z"]), ref["z"])
    assert np.array_equal(_np(out["s_w"]).view(np.uint16), ref["s_w"].view(np.uint16))


# ------------------------------------------------------------------ pack --
@pytest.mark.parametrize("group", [128, 0])
def test_pack_matches_spec_and_round_trips(group):
    N, K = 256, 512
    q4, s_g, z = synthetic.random_codes(N, K, 5)
    if not group:
        z = z[:, 0].copy()
    packed = qoq.qoq_pack_weights(_t(q4), _t(s_g) if group else None, _t(z), group)
    p = _np(packed)
    hdr = p[:256].view(np.uint32)
    assert hdr[0] == 0x57514F51 and hdr[1] == 2
    assert hdr[2] == N and hdr[3] == K and hdr[4] == group and hdr[6] == 0
    assert np.array_equal(p[256:], _pack_spec(q4, s_g, z, group))
    q4b, sgb, zb = qoq.qoq_unpack_weights(packed, N, K, group)
    assert np.array_equal(_np(q4b), q4)
    assert np.array_equal(_np(zb), z)
    if group:
        assert np.array_equal(_np(sgb), s_g)


def test_pack_counts_illegal_codes():
    N, K = 128, 256
    q4, s_g, z = synthetic.random_codes(N, K, 6)
    q4[0, 0] = 15
    s_g[0, 0] = 16
    z[0, 0] = 0  # (15 - 0) * 16 = 240 > 127: illegal
    q4[1, 1] = 16  # not a 4-bit code
    packed = qoq.qoq_pack_weights(_t(q4), _t(s_g), _t(z), 128)
    assert _np(packed)[:256].view(np.uint32)[6] >= 2


# ------------------------------------------------------------------ GEMM --
def _gemm_case(M, N, K, seed, group=128):
    W = synthetic.weights(N, K, seed, 0.02, 2)
    X = synthetic.activations(M, K, seed, 4)
    if group:
        wq = oracle.quantize_weights_group(W, 128)
    else:
        wq = oracle.quantize_weights_channel(W)
    Qx, sx, tx = oracle.quant_act(X)
    return wq, Qx, sx, tx


def _device_weights(wq, group):
    packed = qoq.qoq_pack_weights(_t(wq["q4"]), _t(wq["s_g"]) if group else None, _t(wq["z"]), group)
    return packed, _t(wq["s_w"])


def _ref_acc(wq, Qx, tx, group):
    if group:
        return oracle.gemm_i32_group(Qx, wq["q4"], wq["s_g"], wq["z"])
    return oracle.gemm_i32_channel(Qx, tx, wq["q4"], wq["z"])


CASES = [(16, 256, 512), (1, 256, 512), (2, 128, 128), (3, 384, 1024), (5, 256, 256),
         (7, 128, 2048), (33, 256, 640), (64, 128, 384), (127, 256, 512), (129, 128, 256),
         (200, 256, 1152)]


@pytest.mark.parametrize("M,N,K", CASES)
@pytest.mark.parametrize("group", [128, 0])
def test_gemm_i32_bit_exact(M, N, K, group):
    wq, Qx, sx, tx = _gemm_case(M, N, K, 1000 + M + N + K, group)
    packed, sw = _device_weights(wq, group)
    acc = qoq.qoq_w4a8_gemm_i32(_t(Qx), _t(tx), packed, N, K, group)
    assert np.array_equal(_np(acc), _ref_acc(wq, Qx, tx, group))


@pytest.mark.parametrize("bt", [16, 32, 64, 128])
@pytest.mark.parametrize("ctas", [1, 2, 5, 13, 0])
@pytest.mark.parametrize("publish", [0, 2])
def test_gemm_tiles_and_stream_k_splits(bt, ctas, publish):
    """Every tile size, and persistent-CTA counts that cut output tiles at
    different k-stages (exact int32 reduction of split tiles), with the last
    contributor finishing a tile directly or (debug bit 1) every contributor
    publishing its partial for a fix-up by the last arriver."""
    M, N, K = 37, 256, 1152  # ragged token tail; 9 groups (one chunk boundary)
    wq, Qx, sx, tx = _gemm_case(M, N, K, 77)
    packed, sw = _device_weights(wq, 128)
    ref = _ref_acc(wq, Qx, tx, 128)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    opt = qoq.gemm_options(tokens_per_tile=bt, num_ctas=ctas, acc_out=acc, debug_flags=publish)
    ws = qoq.new_workspace(qoq.qoq_gemm_workspace_bytes(M, N, K, 128, opt))
    for _ in range(2):  # the workspace must come back zeroed
        acc.fill_(0)
        qoq.qoq_w4a8_gemm_ex(_t(Qx), None, None, packed, None, N, K, 128, workspace=ws, options=opt)
        assert np.array_equal(_np(acc), ref)
    O_ref = oracle.epilogue_f64(ref, sx, wq["s_w"])
    for _ in range(2):
        O = qoq.qoq_w4a8_gemm_ex(_t(Qx), _t(sx), None, packed, sw, N, K, 128, workspace=ws,
                                 options=qoq.gemm_options(tokens_per_tile=bt, num_ctas=ctas, debug_flags=publish))
        assert oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref).all()
    assert qoq.qoq_workspace_status(ws)[0] == qoq.QOQ_OK


@pytest.mark.parametrize("schedule", [1, 2, 3, 4])
@pytest.mark.parametrize("bt,ctas", [(32, 7), (64, 3), (128, 5), (16, 13), (32, 0)])
@pytest.mark.parametrize("publish", [0, 2])
def test_gemm_schedules_bit_exact(schedule, bt, ctas, publish):
    """Stream-K only, data-parallel waves then stream-K, the banded tile
    order and the weight-tile-fastest order, over enough tiles for two or
    more waves: int32 bit-exact, the
    workspace left zeroed, both split-tile completion routes."""
    M, N, K = 300, 512, 1152
    wq, Qx, sx, tx = _gemm_case(M, N, K, 78)
    packed, sw = _device_weights(wq, 128)
    ref = _ref_acc(wq, Qx, tx, 128)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    opt = qoq.gemm_options(kernel=1, tokens_per_tile=bt, num_ctas=ctas, acc_out=acc, debug_flags=publish,
                           schedule=schedule)
    ws = qoq.new_workspace(qoq.qoq_gemm_workspace_bytes(M, N, K, 128, opt))
    for _ in range(2):
        acc.fill_(0)
        qoq.qoq_w4a8_gemm_ex(_t(Qx), None, None, packed, None, N, K, 128, workspace=ws, options=opt)
        assert np.array_equal(_np(acc), ref)
    assert qoq.qoq_workspace_status(ws)[0] == qoq.QOQ_OK


FP8_CASES = [(1, 256, 512), (3, 128, 384), (8, 384, 1024), (16, 256, 896), (17, 128, 640), (31, 256, 256),
             (32, 128, 1152),
             # several 32-token tiles (the planner's choice for M <= 64 when a
             # launch has few k-stages per CTA), ragged last tile
             (48, 256, 512), (64, 128, 384), (100, 128, 640)]


@pytest.mark.parametrize("M,N,K", FP8_CASES)
@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("ctas", [0, 3])
@pytest.mark.parametrize("publish", [0, 2])
def test_both_tensor_core_paths_bit_exact(M, N, K, kernel, ctas, publish):
    """The fp16-operand path and the fp8-operand path (exact e4m3 codes, per-
    group drain) give the same int32 accumulators at decode sizes, including
    odd group counts (a last stage with one group) and split tiles, finished
    directly or (debug bit 1) through published partials."""
    wq, Qx, sx, tx = _gemm_case(M, N, K, 4242 + M + K)
    packed, sw = _device_weights(wq, 128)
    ref = _ref_acc(wq, Qx, tx, 128)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    opt = qoq.gemm_options(num_ctas=ctas, acc_out=acc, kernel=kernel, debug_flags=publish)
    ws = qoq.new_workspace(qoq.qoq_gemm_workspace_bytes(M, N, K, 128, opt))
    for _ in range(2):
        acc.fill_(0)
        qoq.qoq_w4a8_gemm_ex(_t(Qx), None, None, packed, None, N, K, 128, workspace=ws, options=opt)
        assert np.array_equal(_np(acc), ref)
    O_ref = oracle.epilogue_f64(ref, sx, wq["s_w"])
    for _ in range(2):
        O = qoq.qoq_w4a8_gemm_ex(_t(Qx), _t(sx), None, packed, sw, N, K, 128, workspace=ws,
                                 options=qoq.gemm_options(num_ctas=ctas, kernel=kernel, debug_flags=publish))
        assert oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref).all()
    assert qoq.qoq_workspace_status(ws)[0] == qoq.QOQ_OK


@pytest.mark.parametrize("M,N,K", FP8_CASES)
def test_fp8_path_with_quantizer_act_operand(M, N, K):
    """The activation operand written by qoq_quant_act_ex, handed to the GEMM,
    gives the oracle's accumulators and the same fp16 output as the GEMM
    building the operand itself."""
    W = synthetic.weights(N, K, 5150 + M, 0.02, 2)
    X = synthetic.activations(M, K, 5151 + M, 4)
    wq = oracle.quantize_weights_group(W, 128)
    Qx_r, sx_r, _ = oracle.quant_act(X)
    packed, sw = _device_weights(wq, 128)
    ref = _ref_acc(wq, Qx_r, None, 128)
    Qx, sx, _, act = qoq.qoq_quant_act_ex(_t(X), kind=2, with_t=False)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    for ctas in (0, 3):
        acc.fill_(0)
        qoq.qoq_w4a8_gemm_ex(Qx, None, None, packed, None, N, K, 128,
                             options=qoq.gemm_options(num_ctas=ctas, acc_out=acc, kernel=2, act_operand=act))
        assert np.array_equal(_np(acc), ref)
    O = qoq.qoq_w4a8_gemm_ex(Qx, sx, None, packed, sw, N, K, 128,
                             options=qoq.gemm_options(kernel=2, act_operand=act))
    O_self = qoq.qoq_w4a8_gemm_ex(Qx, sx, None, packed, sw, N, K, 128, options=qoq.gemm_options(kernel=2))
    assert torch.equal(O, O_self)
    O_ref = oracle.epilogue_f64(ref, sx_r, wq["s_w"])
    assert oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref).all()


@pytest.mark.parametrize("M,N,K", [(33, 256, 640), (64, 128, 1152), (129, 256, 384), (200, 128, 2304)])
@pytest.mark.parametrize("group", [128, 0])
def test_fp16_path_with_quantizer_act_operand(M, N, K, group):
    """The fp16 activation operand written by qoq_quant_act_ex, handed to the
    fp16-operand GEMM, gives the oracle's accumulators and the same output as
    the GEMM building the operand itself (every tile size)."""
    W = synthetic.weights(N, K, 6150 + M, 0.02, 2)
    X = synthetic.activations(M, K, 6151 + M, 4)
    wq = oracle.quantize_weights_group(W, 128) if group else oracle.quantize_weights_channel(W)
    Qx_r, sx_r, tx_r = oracle.quant_act(X)
    packed, sw = _device_weights(wq, group)
    ref = _ref_acc(wq, Qx_r, tx_r, group)
    Qx, sx, tx, act = qoq.qoq_quant_act_ex(_t(X), kind=1)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    for bt in (16, 32, 64, 128):
        acc.fill_(0)
        qoq.qoq_w4a8_gemm_ex(Qx, None, tx, packed, None, N, K, group,
                             options=qoq.gemm_options(tokens_per_tile=bt, acc_out=acc, kernel=1, act_operand=act))
        assert np.array_equal(_np(acc), ref)
    O = qoq.qoq_w4a8_gemm_ex(Qx, sx, tx, packed, sw, N, K, group, options=qoq.gemm_options(kernel=1, act_operand=act))
    O_self = qoq.qoq_w4a8_gemm_ex(Qx, sx, tx, packed, sw, N, K, group, options=qoq.gemm_options(kernel=1))
    assert torch.equal(O, O_self)
    O_ref = oracle.epilogue_f64(ref, sx_r, wq["s_w"])
    assert oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref).all()


GEMV_CASES = [(1, 256, 512), (2, 384, 1024), (3, 128, 384), (5, 256, 1152), (8, 128, 128), (7, 256, 2304),
              (4, 128, 29568)]


@pytest.mark.parametrize("M,N,K", GEMV_CASES)
@pytest.mark.parametrize("group", [128, 0])
@pytest.mark.parametrize("csize", [1, 2, 4, 8])
def test_cuda_core_path_bit_exact(M, N, K, group, csize):
    """The dp4a path (M <= 8): every K split over a thread-block cluster
    (1, 2, 4, 8 CTAs, including splits that leave a CTA or a warp group
    without a block), group and per-channel weights, int32 bit-exact and the
    fp16 output within tolerance."""
    wq, Qx, sx, tx = _gemm_case(M, N, K, 6000 + M + K, group)
    packed, sw = _device_weights(wq, group)
    ref = _ref_acc(wq, Qx, tx, group)
    assert qoq.qoq_gemm_path(M, N, K, group, qoq.gemm_options(kernel=3, num_ctas=csize)) == 3
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    opt = qoq.gemm_options(kernel=3, num_ctas=csize, acc_out=acc)
    ws = qoq.new_workspace(qoq.qoq_gemm_workspace_bytes(M, N, K, group, opt))
    for _ in range(2):
        acc.fill_(0)
        qoq.qoq_w4a8_gemm_ex(_t(Qx), None, _t(tx), packed, None, N, K, group, workspace=ws, options=opt)
        assert np.array_equal(_np(acc), ref)
    O = qoq.qoq_w4a8_gemm_ex(_t(Qx), _t(sx), _t(tx), packed, sw, N, K, group, workspace=ws,
                             options=qoq.gemm_options(kernel=3, num_ctas=csize))
    O_ref = oracle.epilogue_f64(ref, sx, wq["s_w"])
    assert oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref).all()
    assert qoq.qoq_workspace_status(ws)[0] == qoq.QOQ_OK


def test_cuda_core_path_refuses_mismatched_weights():
    M, N, K = 4, 256, 512
    wq, Qx, sx, tx = _gemm_case(M, N, K, 5)
    packed, sw = _device_weights(wq, 128)
    ws = qoq.new_workspace(256)
    O = torch.zeros((M, N - 128), dtype=torch.float16, device=DEV)
    qoq.qoq_w4a8_gemm_ex(_t(Qx), _t(sx), None, packed, sw, N - 128, K, 128, O=O, workspace=ws,
                         options=qoq.gemm_options(kernel=3))
    st, bits = qoq.qoq_workspace_status(ws)
    assert st == 7 and bits & 2
    assert float(O.abs().max()) == 0.0


def test_gemm_exact_at_chunk_extremes():
    """Largest-magnitude products over whole 1024-k chunks: the fp32
    accumulation per chunk must still be exact (sums up to 127*128*1024)."""
    M, N, K = 4, 128, 3072
    q4 = np.zeros((N, K), np.uint8)
    s_g = np.full((N, K // 128), 8, np.uint8)
    z = np.full((N, K // 128), 0, np.uint8)
    q4[:64] = 15                 # +120
    s_g[64:] = 16
    z[64:] = 8
    q4[64:] = 0                  # (0 - 8) * 16 = -128
    q4[100, ::3] = 15            # mixed row: (15 - 8) * 16 = 112
    Qx = np.full((M, K), 127, np.int8)
    Qx[1] = -127
    Qx[2, ::2] = -127
    Qx[3] = np.random.default_rng(1).integers(-127, 128, K).astype(np.int8)
    packed = qoq.qoq_pack_weights(_t(q4), _t(s_g), _t(z), 128)
    ref = oracle.gemm_i32_group(Qx, q4, s_g, z)
    assert abs(int(ref[0, 0])) == 127 * 120 * K
    for ctas in (1, 7, 0):
        for kernel in (1, 2, 3):
            acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
            qoq.qoq_w4a8_gemm_ex(_t(Qx), None, None, packed, None, N, K, 128,
                                 options=qoq.gemm_options(num_ctas=ctas, acc_out=acc, kernel=kernel))
            assert np.array_equal(_np(acc), ref)


@pytest.mark.parametrize("M,N,K", [(16, 256, 512), (1, 512, 4096), (77, 256, 1024)])
@pytest.mark.parametrize("group", [128, 0])
def test_gemm_fp16_within_tolerance(M, N, K, group):
    wq, Qx, sx, tx = _gemm_case(M, N, K, 31 + M, group)
    packed, sw = _device_weights(wq, group)
    O = qoq.qoq_w4a8_gemm(_t(Qx), _t(sx), _t(tx), packed, sw, N, K, group)
    O_ref = oracle.epilogue_f64(_ref_acc(wq, Qx, tx, group), sx, wq["s_w"])
    ok = oracle.o_within_tolerance(_np(O).astype(np.float64), O_ref)
    assert ok.all(), np.argwhere(~ok)[:5]


def test_end_to_end_tiny_workload():
    """The tiny 16x256x512 workload through every device step (weights
    quantized on the device, activations quantized on the device)."""
    (layer,) = synthetic.WORKLOADS[0][1]
    W, X = synthetic.workload_layer_inputs(0, layer, 16)
    ref = oracle.reference_forward_group(W, X, 128)
    wq = qoq.qoq_quantize_weights(_t(W), 128)
    packed = qoq.qoq_pack_weights(wq["q4"], wq["s_g"], wq["z"], 128)
    Qx, sx, tx = qoq.qoq_quant_act(_t(X))
    acc = qoq.qoq_w4a8_gemm_i32(Qx, tx, packed, layer.N, layer.K, 128)
    O = qoq.qoq_w4a8_gemm(Qx, sx, tx, packed, wq["s_w"], layer.N, layer.K, 128)
    assert np.array_equal(_np(acc), ref["acc"])
    assert oracle.o_within_tolerance(_np(O).astype(np.float64), ref["O"]).all()


# ----------------------------------------------------------- error paths --
def test_workspace_too_small_rejected():
    M, N, K = 16, 256, 4096   # a tensor-core path (M <= 8 needs only the status area)
    need = qoq.qoq_gemm_workspace_bytes(M, N, K, 128)
    assert need > 256  # status area plus counters and partial-tile slots
    ws = qoq.new_workspace(256)
    wq, Qx, sx, tx = _gemm_case(M, N, K, 3)
    packed, sw = _device_weights(wq, 128)
    with pytest.raises(qoq.QoqError) as e:
        qoq.qoq_w4a8_gemm(_t(Qx), _t(sx), None, packed, sw, N, K, 128, workspace=ws)
    assert e.value.status == 4


def test_mismatched_packed_weights_reported_on_device():
    M, N, K = 8, 256, 512
    wq, Qx, sx, tx = _gemm_case(M, N, K, 4)
    packed, sw = _device_weights(wq, 128)
    ws = qoq.new_workspace(qoq.qoq_gemm_workspace_bytes(M, N - 128, K, 128))
    O = torch.zeros((M, N - 128), dtype=torch.float16, device=DEV)
    # packed holds N = 256 rows; calling with N = 128 must be refused on the device
    qoq.qoq_w4a8_gemm(_t(Qx), _t(sx), None, packed, sw, N - 128, K, 128, O=O, workspace=ws)
    st, bits = qoq.qoq_workspace_status(ws)
    assert st == 7 and bits & 2
    assert float(O.abs().max()) == 0.0  # nothing written
    st, bits = qoq.qoq_workspace_status(ws)
    assert st == 0 and bits == 0  # cleared by the read


def _overlap_chain(points, bufs, ws, use_flags):
    flags = qoq.QOQ_LAUNCH_OVERLAP if use_flags else 0
    for pt in points:
        M, N, K = pt["M"], pt["N"], pt["K"]
        Qx = bufs["Qx"][: M * K].view(M, K)
        sx = bufs["sx"][:M]
        kind = qoq.qoq_gemm_path(M, N, K, 128)
        act = bufs["act"][: qoq.qoq_act_operand_bytes(M, K, kind)]
        qoq.qoq_quant_act_ex(pt["X"], Qx, sx, None, act, kind=kind, with_t=False, flags=flags)
        qoq.qoq_w4a8_gemm_ex(Qx, sx, None, pt["packed"], pt["sw"], N, K, 128, O=pt["O"], workspace=ws,
                             options=qoq.gemm_options(act_operand=act, flags=flags))


@pytest.mark.parametrize("graph", [False, True])
def test_overlapped_launch_chain_with_shared_buffers(graph):
    """Programmatic dependent launch: quantizer and GEMM of consecutive
    (M, layer) points share the activation, operand, scale and workspace
    buffers, so a kernel that touched them before its predecessor finished
    would corrupt an earlier point; every point must still equal the oracle,
    launched eagerly and replayed from a CUDA graph."""
    shapes = [(8, 256, 512), (48, 384, 1024), (1, 128, 640), (40, 256, 512), (16, 384, 1024), (130, 128, 384)]
    points = []
    for i, (M, N, K) in enumerate(shapes):
        W = synthetic.weights(N, K, 7100 + i, 0.02, 2)
        X = synthetic.activations(M, K, 7200 + i, 4)
        wq = oracle.quantize_weights_group(W, 128)
        Qx_r, sx_r, _ = oracle.quant_act(X)
        ref = oracle.epilogue_f64(_ref_acc(wq, Qx_r, None, 128), sx_r, wq["s_w"])
        packed, sw = _device_weights(wq, 128)
        points.append(dict(M=M, N=N, K=K, X=_t(X), packed=packed, sw=sw, ref=ref,
                           O=torch.full((M, N), float("nan"), dtype=torch.float16, device=DEV)))
    maxMK = max(M * K for M, _, K in shapes)
    bufs = dict(Qx=torch.empty(maxMK, dtype=torch.int8, device=DEV),
                sx=torch.empty(max(M for M, _, _ in shapes), dtype=torch.float16, device=DEV),
                act=torch.empty(max(qoq.qoq_act_operand_bytes(M, K, k) for M, _, K in shapes for k in (1, 2)),
                                dtype=torch.uint8, device=DEV))
    ws = qoq.new_workspace(max(qoq.qoq_gemm_workspace_bytes(M, N, K, 128) for M, N, K in shapes))
    _overlap_chain(points, bufs, ws, True)  # eager first (sets kernel attributes before any capture)
    torch.cuda.synchronize()
    if graph:
        for pt in points:
            pt["O"].fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            _overlap_chain(points, bufs, ws, True)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
    for pt in points:
        assert oracle.o_within_tolerance(_np(pt["O"]).astype(np.float64), pt["ref"]).all()
    assert qoq.qoq_workspace_status(ws)[0] == qoq.QOQ_OK


@pytest.mark.parametrize("kernel", [1, 2])
def test_bounded_wait_timeout_reports_status_and_context_survives(kernel):
    """The copy warp withholds one stage (debug flag), so the consumers'
    bounded waits expire: the kernel must return, report QOQ_ERR_TIMEOUT
    through the status word, free its resources, and leave the context
    usable for a correct GEMM right after."""
    M, N, K = 16, 256, 1024
    wq, Qx, sx, tx = _gemm_case(M, N, K, 9)
    packed, sw = _device_weights(wq, 128)
    opt = qoq.gemm_options(num_ctas=1, debug_flags=1, timeout_ns=50_000_000, kernel=kernel)
    ws = qoq.new_workspace(qoq.qoq_gemm_workspace_bytes(M, N, K, 128, opt))
    O = torch.zeros((M, N), dtype=torch.float16, device=DEV)
    qoq.qoq_w4a8_gemm_ex(_t(Qx), _t(sx), None, packed, sw, N, K, 128, O=O, workspace=ws, options=opt)
    st, bits = qoq.qoq_workspace_status(ws)
    assert st == 6 and bits & 1
    qoq.qoq_workspace_init(ws)
    acc = qoq.qoq_w4a8_gemm_i32(_t(Qx), None, packed, N, K, 128)
    assert np.array_equal(_np(acc), _ref_acc(wq, Qx, tx, 128))
