"""Pins of the CPU oracle against what the QServe pages and mathematics fix.

No test here re-types an oracle formula: each checks the oracle against a
value printed on the pages, an exhaustive sweep of a bound the pages derive,
a closed form, a brute force, a library routine (numpy / Python fractions),
or an invariant that any correct implementation must satisfy.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from w4a8_quantized_serving_qoq_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = int(v)
    return vals


# ---------------------------------------------------------------- fp16 ----
def test_half_to_float_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_rn_vs_numpy():
    rng = np.random.default_rng(7)
    parts = [
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 6, 20000).astype(np.float32),
        # exact midpoints between adjacent fp16 values (ties) in normal and subnormal range
        ((np.arange(0, 2048, dtype=np.float64) + 0.5) * 2.0 ** -24).astype(np.float32),
        ((np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0 ** -3).astype(np.float32),
        np.array([65504, 65519.99, 65520, 65535, 1e9, 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26,
                  6.1e-5, 5.96e-8, 0.0, -0.0, 1.0, -1.0, np.inf, -np.inf], np.float32),
        rng.uniform(-70000, 70000, 5000).astype(np.float32),
    ]
    x = np.concatenate(parts)
    x = np.concatenate([x, -x])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half_rn(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------- rounding ----
def test_rne_f32_vs_numpy_rint():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.uniform(-300, 300, 20000).astype(np.float32),
        np.arange(-300, 300, dtype=np.float32) + np.float32(0.5),
        np.array([2.0 ** 23 + 1, -(2.0 ** 23) - 1, 1e9, -0.5, 0.5, 1.5, 2.5], np.float32),
    ])
    got = np.array([oracle.rne_f32(float(v)) for v in x])
    assert np.array_equal(got, np.rint(x.astype(np.float64)).astype(np.int64))


def test_rne_div_vs_fraction_round():
    # Python's round() of a Fraction is exact round-half-even.
    for b in range(1, 18):
        for a in range(-300, 301):
            assert oracle.rne_div(a, b) == round(Fraction(a, b)), (a, b)


# ------------------------------------------------ progressive quantization --
def test_worked_group_from_pages():
    """Unprotected [-113, 120] group: scale 16, zero 7, 120 -> code 15 -> 128."""
    gv = _golden("protective_range_worked_group.txt")
    group = np.array([gv["group_min"], 0, 5, -40, gv["value"], gv["group_max"]], np.int32)
    q4, s, z, bad = oracle.group_step(group)
    assert s == gv["scale"]
    assert z == gv["zero"]
    i = list(group).index(gv["value"])
    assert q4[i] == gv["code"]
    assert (int(q4[i]) - z) * s == gv["reconstruction"]
    assert bad >= 1  # 128 leaves the INT8 range


def test_scale_bound_from_pages():
    """s_u8 <= (127 - (-128)) / (15 - 0) = 17 on the full INT8 range, and the
    protective range keeps every group scale at or below 16."""
    gv = _golden("protective_range_worked_group.txt")
    _, s, _, _ = oracle.group_step(np.array([-128, 127], np.int32))
    assert s == gv["scale_bound"]
    _, s, _, _ = oracle.group_step(np.array([-119, 119], np.int32))
    assert s <= 16


def test_rounding_bound_from_pages():
    """⌊q/s⌉·s <= q + s/2 for every INT8 q and scale s <= 17, hence
    reconstructions of q <= 119 stay <= 119.5 + ... <= 127 (2x to stay integral)."""
    gv = _golden("protective_range_worked_group.txt")
    for s in range(1, gv["scale_bound"] + 1):
        for q in range(-128, 128):
            r = oracle.rne_div(q, s) * s
            assert 2 * r <= 2 * q + s
            assert 2 * r >= 2 * q - s
    # q <= 119.5 is the page's bound for the first level: 2*119 < 239 <= 2*127 - 15
    assert 2 * 119 < gv["first_level_bound_x2"]


def _sweep(lo_min, hi_max, step=1):
    overflow = 0
    max_abs = 0
    max_s = 0
    for lo in range(lo_min, 1):
        for hi in range(0, hi_max + 1):
            group = np.arange(lo, hi + 1, step, dtype=np.int32)
            group = np.unique(np.concatenate([group, [lo, hi]]).astype(np.int32))
            q4, s, z, bad = oracle.group_step(group)
            w = (q4.astype(np.int64) - z) * s
            overflow += int(((w < -128) | (w > 127)).sum())
            assert bad == int(((w < -128) | (w > 127)).sum())
            max_abs = max(max_abs, int(np.abs(w).max()))
            max_s = max(max_s, s)
            assert 0 <= z <= 15 and q4.max() <= 15
    return overflow, max_abs, max_s


def test_protective_range_exhaustive_no_overflow():
    """Every group inside [-119, 119] reconstructs inside INT8 (all values)."""
    overflow, max_abs, max_s = _sweep(-119, 119)
    assert overflow == 0
    assert max_abs <= 127
    assert max_s <= 16


def test_full_range_overflows_exist():
    """Without the protective range some groups overflow (the pages' point)."""
    overflow, max_abs, max_s = _sweep(-128, 127, step=3)
    assert overflow > 0
    assert max_abs > 127
    assert max_s == 17


def _rand_weights(N, K, seed=11):
    return synthetic.weights(N, K, seed, 0.02, 2)


def test_step1_invariants():
    W = _rand_weights(48, 512)
    r = oracle.quantize_weights_group(W, 128)
    Wf = W.astype(np.float64)
    sw = r["s_w"].astype(np.float64)
    q8 = r["q8"].astype(np.int64)
    assert np.abs(q8).max() <= 119
    # the largest-magnitude weight of each row maps to +-119
    arg = np.argmax(np.abs(Wf), axis=1)
    assert np.array_equal(np.abs(q8[np.arange(48), arg]), np.full(48, 119))
    # round-to-nearest: |W/s_w - q8| <= 1/2 (up to one fp32 rounding of the quotient)
    err = np.abs(Wf / sw[:, None] - q8)
    assert err.max() <= 0.5 + 1e-5
    # fp16 channel scale is the correctly rounded max/119 (checked via numpy's converter)
    amax = np.abs(W.astype(np.float32)).max(axis=1)
    assert np.array_equal(r["s_w"].view(np.uint16), (amax / np.float32(119)).astype(np.float16).view(np.uint16))


def test_step2_invariants():
    W = _rand_weights(40, 1024, seed=5)
    r = oracle.quantize_weights_group(W, 128)
    assert r["n_overflow"] == 0
    q8 = r["q8"].astype(np.int64).reshape(40, 8, 128)
    q4 = r["q4"].astype(np.int64).reshape(40, 8, 128)
    s = r["s_g"].astype(np.int64)[:, :, None]
    z = r["z"].astype(np.int64)[:, :, None]
    lo = np.minimum(0, q8.min(axis=2, keepdims=True))
    hi = np.maximum(0, q8.max(axis=2, keepdims=True))
    assert (z >= 0).all() and (z <= 15).all() and (q4 <= 15).all()
    # the 16 levels cover the group range, with the smallest such integer scale
    assert (15 * s >= hi - lo).all()
    assert ((s == 1) | (15 * (s - 1) < hi - lo)).all()
    # nearest-level reconstruction with no clipping
    w8 = (q4 - z) * s
    assert (2 * np.abs(w8 - q8) <= s).all()
    assert np.abs(w8).max() <= 127
    # byte-lane legality: q4*s_g and z*s_g fit in a byte
    assert (q4 * s <= 255).all() and (z * s <= 255).all()


def test_degenerate_weight_rows():
    W = np.zeros((3, 256), np.float16)
    W[1, 7] = np.float16(-0.5)
    W[2, :128] = np.float16(0.25)  # a whole positive group
    r = oracle.quantize_weights_group(W, 128)
    assert r["s_w"].view(np.uint16)[0] == 0x3C00  # all-zero row: s_w = 1
    assert (r["q8"][0] == 0).all() and (r["s_g"][0] == 1).all() and (r["z"][0] == 0).all()
    assert r["q8"][1, 7] == -119
    assert r["q8"][2, 0] == 119 and r["z"][2, 0] == 0 and r["s_g"][2, 0] == 8
    assert r["n_overflow"] == 0


def test_channel_quantizer_invariants():
    W = _rand_weights(32, 512, seed=9)
    r = oracle.quantize_weights_channel(W)
    Wf = W.astype(np.float64)
    s = r["s_w"].astype(np.float64)[:, None]
    z = r["z"].astype(np.int64)[:, None]
    q4 = r["q4"].astype(np.int64)
    assert q4.max() <= 15 and z.max() <= 15
    lo = np.minimum(0, Wf.min(axis=1, keepdims=True))
    hi = np.maximum(0, Wf.max(axis=1, keepdims=True))
    # zero point places 0 within half a level; codes within half a level (+clip slack)
    assert (np.abs(z - (-lo / s)) <= 0.5 + 1e-4).all()
    rec = (q4 - z) * s
    inside = (Wf >= lo) & (Wf <= hi)
    assert (np.abs(rec - Wf)[inside] <= (0.5 + 1e-3) * np.broadcast_to(s, Wf.shape)[inside] + 1e-3 * s.max()).all()


def _channel_rows_with_edge_cases(N, K, seed):
    W = _rand_weights(N, K, seed=seed)
    W[0] = 0                                   # all-zero row: the scale guard
    W[1] = np.abs(W[1])                        # non-negative row: lo = 0, z = 0
    W[2] = -np.abs(W[2])                       # non-positive row: hi = 0
    W[3, :] = 0
    W[3, 5] = np.float16(2.0 ** -20)           # a lone subnormal weight
    return W


def test_channel_scale_bits_vs_numpy_converter():
    """s_W = fp16_rn(fp32(hi - lo) / 15), bit for bit, with numpy's IEEE fp32
    arithmetic and its own binary16 converter (a library routine) -- the
    per-channel counterpart of the step-1 scale check.  A truncated scale, an
    fp16 (instead of fp32) difference or a missing zero guard fails here."""
    W = _channel_rows_with_edge_cases(64, 768, seed=19)
    r = oracle.quantize_weights_channel(W)
    Wf = W.astype(np.float32)
    lo = np.minimum(np.float32(0), Wf.min(axis=1))
    hi = np.maximum(np.float32(0), Wf.max(axis=1))
    s = ((hi - lo) / np.float32(15)).astype(np.float16)
    s[s == 0] = np.float16(1.0)
    assert np.array_equal(r["s_w"].view(np.uint16), s.view(np.uint16))
    # zero and codes: IEEE fp32 quotients by the stored fp16 scale, numpy.rint (half-even)
    sf = s.astype(np.float32)
    z = np.clip(np.rint(-lo / sf), 0, 15).astype(np.int64)
    q4 = np.clip(np.rint(Wf / sf[:, None]) + z[:, None], 0, 15)
    assert np.array_equal(r["z"].astype(np.int64), z)
    assert np.array_equal(r["q4"].astype(np.int64), q4.astype(np.int64))
    assert r["s_w"].view(np.uint16)[0] == 0x3C00 and r["z"][0] == 0 and (r["q4"][0] == 0).all()
    assert r["z"][1] == 0 and r["z"][2] == 15


def test_channel_scale_difference_taken_in_fp32():
    """A row whose fp16 difference hi - lo rounds to a different scale than the
    fp32 difference: the oracle must follow the fp32 reading."""
    found = None
    cand = np.arange(0x3C00, 0x3C00 + 64, dtype=np.uint16).view(np.float16)      # hi in [1, 1.0625)
    lows = -np.arange(0x0400, 0x1C00, 7, dtype=np.uint16).view(np.float16)      # lo in (-2^-6, -2^-14]
    for hi in cand:
        d16 = (np.float16(hi) - lows).astype(np.float16)                        # fp16 difference (RN)
        d32 = np.float32(hi) - lows.astype(np.float32)                          # fp32 difference (RN)
        s16 = (d16.astype(np.float32) / np.float32(15)).astype(np.float16)
        s32 = (d32 / np.float32(15)).astype(np.float16)
        diff = np.nonzero(s16.view(np.uint16) != s32.view(np.uint16))[0]
        if diff.size:
            found = (hi, lows[diff[0]], s32[diff[0]], s16[diff[0]])
            break
    assert found is not None
    hi, lo, s32, s16 = found
    W = np.zeros((1, 128), np.float16)
    W[0, 0], W[0, 1] = hi, lo
    r = oracle.quantize_weights_channel(W)
    assert r["s_w"].view(np.uint16)[0] == s32.view(np.uint16)
    assert r["s_w"].view(np.uint16)[0] != s16.view(np.uint16)


def test_channel_constructed_ties_half_even():
    """Exact ties of rne(-lo / s_W) and rne(W / s_W), with every value exact
    in fp16 and s_W = 0.125 exactly ((hi - lo) / 15 = 1.875 / 15)."""
    s = 0.125
    r0 = np.zeros(128); r0[0], r0[1] = -2.5 * s, 1.875 - 2.5 * s     # z = rne(2.5) = 2 (half-away: 3)
    r1 = np.zeros(128); r1[0], r1[1] = -3.5 * s, 1.875 - 3.5 * s     # z = rne(3.5) = 4
    vals = np.array([0.5, 1.5, -0.5, -1.5, 2.5, 3.5, 4.5]) * s        # code ties
    r0[2:9] = vals
    r1[2:9] = vals
    W = np.stack([r0, r1]).astype(np.float16)
    assert np.array_equal(W.astype(np.float64), np.stack([r0, r1]))  # all exact in fp16
    r = oracle.quantize_weights_channel(W)
    assert list(r["s_w"].astype(np.float64)) == [s, s]
    assert list(r["z"]) == [2, 4]
    # rne: 0.5 -> 0, 1.5 -> 2, -0.5 -> 0, -1.5 -> -2, 2.5 -> 2, 3.5 -> 4, 4.5 -> 4; plus z
    assert list(r["q4"][0, 2:9]) == [2, 4, 2, 0, 4, 6, 6]
    assert list(r["q4"][1, 2:9]) == [4, 6, 4, 2, 6, 8, 8]
    # the range ends: lo -> rne(-2.5) + 2 = 0, hi = 12.5 s -> 12 + 2 = 14
    assert r["q4"][0, 0] == 0 and r["q4"][0, 1] == 14
    # row 1: hi = 11.5 s -> rne 12, + z = 4 gives 16, clipped to 15
    assert round(Fraction(23, 2)) == 12
    assert r["q4"][1, 0] == 0 and r["q4"][1, 1] == 15


# --------------------------------------------------------------- activations
def test_quant_act_invariants():
    X = synthetic.activations(24, 768, 4, 4)
    Qx, sx, tx = oracle.quant_act(X)
    Xf = X.astype(np.float64)
    s = sx.astype(np.float64)[:, None]
    assert np.abs(Qx.astype(np.int64)).max() <= 127
    arg = np.argmax(np.abs(Xf), axis=1)
    assert np.array_equal(np.abs(Qx[np.arange(24), arg].astype(np.int64)), np.full(24, 127))
    assert np.abs(Xf / s - Qx).max() <= 0.5 + 1e-5
    assert np.array_equal(tx, Qx.astype(np.int64).sum(axis=1))
    amax = np.abs(X.astype(np.float32)).max(axis=1)
    assert np.array_equal(sx.view(np.uint16), (amax / np.float32(127)).astype(np.float16).view(np.uint16))


def test_quant_act_ties_half_even_and_zero_row():
    s = np.float32(0.125)  # exact in fp16
    row = np.zeros(64, np.float32)
    row[0] = 127 * s       # defines s_x = 0.125 exactly
    row[1] = 2.5 * s       # tie -> 2
    row[2] = 3.5 * s       # tie -> 4
    row[3] = -2.5 * s      # tie -> -2
    row[4] = -0.5 * s      # tie -> 0
    row[5] = 1.5 * s       # tie -> 2
    X = np.stack([row, np.zeros(64, np.float32)]).astype(np.float16)
    Qx, sx, tx = oracle.quant_act(X)
    assert float(sx[0]) == 0.125
    assert list(Qx[0, :6]) == [127, 2, 4, -2, 0, 2]
    assert float(sx[1]) == 0.0 and (Qx[1] == 0).all() and tx[1] == 0


def test_quant_act_vs_torch_cpu_restatement():
    torch = pytest.importorskip("torch")
    X = synthetic.activations(8, 1024, 21, 4)
    Qx, sx, tx = oracle.quant_act(X)
    Xt = torch.from_numpy(X.astype(np.float32))
    s = (Xt.abs().amax(dim=1) / 127.0).to(torch.float16).to(torch.float32)
    q = torch.clamp(torch.round(Xt / s[:, None]), -127, 127).to(torch.int8)
    assert np.array_equal(Qx, q.numpy())
    assert np.array_equal(sx.astype(np.float32), s.numpy())


# -------------------------------------------------------------------- GEMM --
def test_gemm_group_vs_numpy_int64():
    M, N, K = 7, 40, 512
    q4, sg, z = synthetic.random_codes(N, K, 1)
    rng = np.random.default_rng(2)
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    w8 = (q4.astype(np.int64) - np.repeat(z, 128, axis=1)) * np.repeat(sg, 128, axis=1)
    ref = Qx.astype(np.int64) @ w8.T
    got = oracle.gemm_i32_group(Qx, q4, sg, z)
    assert np.array_equal(got.astype(np.int64), ref)
    ms = np.array([0, 6, 3, 3]); ns = np.array([0, 39, 17, 18])
    assert np.array_equal(oracle.gemm_i32_group_at(Qx, q4, sg, z, ms, ns), ref[ms, ns])


def test_gemm_group_brute_force_python():
    M, N, K, g = 2, 3, 256, 128
    q4, sg, z = synthetic.random_codes(N, K, 3)
    Qx = np.random.default_rng(4).integers(-127, 128, size=(M, K)).astype(np.int8)
    got = oracle.gemm_i32_group(Qx, q4, sg, z)
    for m in range(M):
        for n in range(N):
            tot = 0
            for k in range(K):
                tot += int(Qx[m, k]) * (int(q4[n, k]) - int(z[n, k // g])) * int(sg[n, k // g])
            assert got[m, n] == tot


def test_gemm_extremes_fit_int32():
    # |acc| <= K * 127 * 127 for the largest K of the workloads
    assert 29568 * 127 * 127 < 2 ** 31
    K = 1024
    q4 = np.full((2, K), 15, np.uint8)
    sg = np.full((2, K // 128), 8, np.uint8)
    z = np.zeros((2, K // 128), np.uint8)
    Qx = np.full((2, K), 127, np.int8)
    Qx[1] = -127
    got = oracle.gemm_i32_group(Qx, q4, sg, z)
    assert got[0, 0] == K * 127 * 120 and got[1, 1] == -K * 127 * 120


def test_channel_folded_equals_direct():
    """Pages' eq. 13 fold: sum Qx*q4 - z*t_x == sum Qx*(q4 - z), exactly."""
    M, N, K = 5, 33, 384
    rng = np.random.default_rng(8)
    Qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    tx = Qx.astype(np.int64).sum(axis=1).astype(np.int32)
    q4 = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    z = rng.integers(0, 16, size=N).astype(np.uint8)
    direct = Qx.astype(np.int64) @ (q4.astype(np.int64) - z.astype(np.int64)[:, None]).T
    got = oracle.gemm_i32_channel(Qx, tx, q4, z)
    assert np.array_equal(got.astype(np.int64), direct)
    ms = np.array([4, 0]); ns = np.array([32, 1])
    assert np.array_equal(oracle.gemm_i32_channel_at(Qx, tx, q4, z, ms, ns), direct[ms, ns])


def test_channel_closed_form_fp64():
    """O = (QxQw) ⊙ (s_W × s_X) − (Qx ⊙ S_X) Z S_W, re-derived with matrices."""
    M, N, K = 6, 20, 256
    W = _rand_weights(N, K, seed=13)
    X = synthetic.activations(M, K, 14, 4)
    wq = oracle.quantize_weights_channel(W)
    Qx, sx, tx = oracle.quant_act(X)
    acc = oracle.gemm_i32_channel(Qx, tx, wq["q4"], wq["z"])
    O = oracle.epilogue_f64(acc, sx, wq["s_w"])
    Qxf = Qx.astype(np.float64)
    Qw = wq["q4"].astype(np.float64)
    sW = wq["s_w"].astype(np.float64)
    sX = sx.astype(np.float64)
    Z = np.tile(wq["z"].astype(np.float64)[None, :], (K, 1))   # K x N zero matrix
    first = (Qxf @ Qw.T) * np.outer(sX, sW)
    second = ((Qxf * sX[:, None]) @ Z) * sW[None, :]
    ref = first - second
    assert np.allclose(O, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_group_closed_form_fp64():
    """Per group g: Qw := q4*s_g, Z := z*s_g; O = s_x s_w sum_g (Qx_g Qw_g^T - (Qx_g 1) Z_g^T)."""
    M, N, K, g = 4, 24, 512, 128
    W = _rand_weights(N, K, seed=15)
    X = synthetic.activations(M, K, 16, 4)
    ref_all = oracle.reference_forward_group(W, X, g)
    wq = ref_all["wq"]
    Qxf = ref_all["Qx"].astype(np.float64)
    tot = np.zeros((M, N))
    for gi in range(K // g):
        sl = slice(gi * g, (gi + 1) * g)
        Qw = wq["q4"][:, sl].astype(np.float64) * wq["s_g"][:, gi].astype(np.float64)[:, None]
        Zg = wq["z"][:, gi].astype(np.float64) * wq["s_g"][:, gi].astype(np.float64)
        tot += Qxf[:, sl] @ Qw.T - np.outer(Qxf[:, sl].sum(axis=1), Zg)
    ref = tot * np.outer(ref_all["s_x"].astype(np.float64), wq["s_w"].astype(np.float64))
    assert np.allclose(ref_all["O"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_tolerance_helper():
    O_ref = np.array([[1.0, -2.0, 1000.0]])
    # bound = 2e-3 * 1000 + ulp16(|O_ref|): 2 + 2^-10 at 1.0, 2 + 0.5 at 1000
    ok = oracle.o_within_tolerance(O_ref + np.array([[2.0, 0.0, -2.6]]), O_ref)
    assert ok.tolist() == [[True, True, False]]
    assert oracle.fp16_ulp(np.array([1.0]))[0] == 2.0 ** -10
    assert oracle.fp16_ulp(np.array([0.0]))[0] == 2.0 ** -24


# ------------------------------------------- norm and activation in front of a GEMM --
def test_rmsnorm_closed_forms():
    K = 256
    one = np.ones(K, np.float16)
    # a constant row with eps = 0 normalizes to sign(c) everywhere
    X = np.stack([np.full(K, 0.75), np.full(K, -3.0)]).astype(np.float16)
    Y = oracle.rmsnorm_f64(X, one, 0.0)
    assert np.allclose(Y[0], 1.0, rtol=0, atol=1e-15) and np.allclose(Y[1], -1.0, rtol=0, atol=1e-15)
    # a lone nonzero a: a / sqrt(a^2 / K) = sign(a) sqrt(K); the zeros stay zero
    X = np.zeros((1, K), np.float16)
    X[0, 7] = -0.5
    Y = oracle.rmsnorm_f64(X, one, 0.0)
    assert Y[0, 7] == pytest.approx(-np.sqrt(K), rel=1e-15) and np.count_nonzero(Y) == 1
    # eps enters under the root: c / sqrt(c^2 + eps); gamma scales each channel
    g = (np.arange(K) % 5 + 1).astype(np.float16)
    X = np.full((1, K), 0.5, np.float16)
    Y = oracle.rmsnorm_f64(X, g, 1e-2)
    assert np.allclose(Y[0], g.astype(np.float64) * 0.5 / np.sqrt(0.25 + 1e-2), rtol=1e-14, atol=0)
    # an all-zero row stays zero (0 / sqrt(eps), and 0 / 0 read as 0 when eps = 0)
    Z = np.zeros((2, K), np.float16)
    assert not oracle.rmsnorm_f64(Z, one, 1e-6).any() and not oracle.rmsnorm_f64(Z, one, 0.0).any()


def test_rmsnorm_vs_torch_cpu():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    if not hasattr(F, "rms_norm"):
        pytest.skip("torch without rms_norm")
    X = synthetic.activations(6, 4096, 31, 4)
    gamma = (1.0 + 0.1 * np.random.default_rng(3).standard_normal(4096)).astype(np.float16)
    Y = oracle.rmsnorm_f64(X, gamma, 1e-5)
    ref = F.rms_norm(torch.from_numpy(X.astype(np.float64)), (4096,),
                     weight=torch.from_numpy(gamma.astype(np.float64)), eps=1e-5).numpy()
    assert np.allclose(Y, ref, rtol=1e-13, atol=1e-13)


def test_silu_mul_closed_forms_and_library():
    special = pytest.importorskip("scipy.special")
    F = 512
    rng = np.random.default_rng(12)
    G = (rng.standard_normal((3, F)) * 4).astype(np.float16)
    U = rng.standard_normal((3, F)).astype(np.float16)
    G[0, :4] = [0.0, 30.0, -30.0, 1.0]
    U[0, :4] = [5.0, 1.0, 1.0, 2.0]
    A = oracle.silu_mul_f64(np.concatenate([G, U], axis=1))
    g, u = G.astype(np.float64), U.astype(np.float64)
    # the logistic function from scipy (a library routine): SiLU(g) = g * expit(g)
    assert np.allclose(A, g * special.expit(g) * u, rtol=1e-14, atol=1e-300)
    assert A[0, 0] == 0.0                                   # SiLU(0) = 0
    assert A[0, 1] == pytest.approx(30.0, rel=1e-12)        # SiLU(g) -> g for large g
    assert abs(A[0, 2]) < 1e-11                             # SiLU(g) -> 0 for very negative g
    assert A[0, 3] == pytest.approx(2.0 / (1.0 + np.exp(-1.0)) * 1.0 * 1.0, rel=1e-15)
    # SiLU(g) - SiLU(-g) = g exactly in real arithmetic (odd part of g * sigmoid(g))
    ones = np.ones_like(G)
    Ap = oracle.silu_mul_f64(np.concatenate([G, ones], axis=1))
    Am = oracle.silu_mul_f64(np.concatenate([-G, ones], axis=1))
    assert np.allclose(Ap - Am, g, rtol=1e-13, atol=1e-13)


def test_fp16_one_ulp_helper():
    ref = np.array([1.0, 1.0, 1.0, 0.0, 3e-8])
    got = np.array([1.0 + 2 ** -10, 1.0 + 2 ** -9, 1.0 - 2 ** -11, 2 ** -24, 0.0])
    assert oracle.fp16_within_one_ulp(got, ref).tolist() == [True, False, True, True, True]


# ------------------------------------------------------------------ KV4 cache --
def _kv(n, d, seed, outliers=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d)).astype(np.float32)
    if outliers:
        x[:, rng.choice(d, outliers, replace=False)] *= 10.0   # fixed outlier channels of a key head
    return x.astype(np.float16)


def test_kv4_quantize_vs_numpy_fp32():
    """Scale, zero and codes bit for bit against numpy's IEEE fp32 arithmetic,
    its binary16 converter and numpy.rint (half-even); includes a constant
    vector (scale guard) and all-positive / all-negative vectors."""
    x = _kv(40, 128, 5, outliers=3)
    x[0] = np.float16(0.75)
    x[1] = np.abs(x[1]) + np.float16(1.0)
    x[2] = -np.abs(x[2]) - np.float16(2.0)
    q, s, z = oracle.kv4_quantize(x)
    xf = x.astype(np.float32)
    lo, hi = xf.min(axis=1), xf.max(axis=1)
    s_ref = ((hi - lo) / np.float32(15)).astype(np.float16)
    s_ref[s_ref == 0] = np.float16(1.0)
    sf = s_ref.astype(np.float32)
    z_ref = np.rint(-lo / sf).astype(np.float16)
    q_ref = np.clip(np.rint(xf / sf[:, None]) + z_ref.astype(np.float32)[:, None], 0, 15)
    assert np.array_equal(s.view(np.uint16), s_ref.view(np.uint16))
    assert np.array_equal(z.view(np.uint16), z_ref.view(np.uint16))
    assert np.array_equal(q, q_ref.astype(np.uint8))
    # all-positive vector: negative zero point; all-negative: zero point above 15
    assert float(z[1]) < 0 and float(z[2]) > 15
    # reconstruction error: half a level, or one level where the top code clips
    rec = (q.astype(np.float64) - z.astype(np.float64)[:, None]) * s.astype(np.float64)[:, None]
    assert (np.abs(rec - x.astype(np.float64)) <= 1.001 * s.astype(np.float64)[:, None]).all()
    assert rec[0, 0] == 1.0 and (q[0] == 0).all()      # constant 0.75: s = 1, z = -1


def test_kv4_quantize_constructed_ties():
    """s = 1.875 / 15 = 0.125 exactly; rne(2.5) = 2 for the zero point and
    half-even code ties (every value exact in fp16)."""
    s = 0.125
    v = np.zeros(128)
    v[0], v[1] = -2.5 * s, 1.875 - 2.5 * s
    v[2:8] = np.array([0.5, 1.5, -0.5, -1.5, 2.5, 3.5]) * s
    v[8:] = 0.5 * s
    x = v[None, :].astype(np.float16)
    assert np.array_equal(x.astype(np.float64)[0], v)
    q, sc, z = oracle.kv4_quantize(x)
    assert float(sc[0]) == s and float(z[0]) == 2.0
    assert list(q[0, :8]) == [0, 14, 2, 4, 2, 0, 4, 6]


def _deq(q, s, z):
    return (q.astype(np.float64) - z.astype(np.float64)[:, None]) * s.astype(np.float64)[:, None]


def test_kv4_attention_closed_forms():
    d = 128
    Q = _kv(4, d, 6)
    Kq, Ks, Kz = oracle.kv4_quantize(_kv(9, d, 7, outliers=2))
    Vq, Vs, Vz = oracle.kv4_quantize(_kv(9, d, 8))
    # one cached token: the output is that token's value for every head
    O = oracle.kv4_attention_f64(Q, Kq[:1], Ks[:1], Kz[:1], Vq[:1], Vs[:1], Vz[:1], 0.088)
    assert np.allclose(O, np.broadcast_to(_deq(Vq[:1], Vs[:1], Vz[:1]), (4, d)), rtol=0, atol=1e-15)
    # identical keys: uniform attention, the mean of the values
    Kr = np.repeat(Kq[:1], 9, axis=0)
    O = oracle.kv4_attention_f64(Q, Kr, np.repeat(Ks[:1], 9), np.repeat(Kz[:1], 9), Vq, Vs, Vz, 0.088)
    assert np.allclose(O, np.broadcast_to(_deq(Vq, Vs, Vz).mean(axis=0), (4, d)), rtol=1e-13, atol=1e-13)
    # a key far ahead of the others takes all the weight
    Q1 = np.zeros((1, d), np.float16)
    Q1[0, :] = 1.0
    Kq2 = np.zeros((3, d), np.uint8)
    Kq2[1] = 15
    one = np.ones(3, np.float16)
    zero = np.zeros(3, np.float16)
    O = oracle.kv4_attention_f64(Q1, Kq2, one, zero, Vq[:3], Vs[:3], Vz[:3], 1.0)
    assert np.allclose(O[0], _deq(Vq[1:2], Vs[1:2], Vz[1:2])[0], rtol=0, atol=1e-12)


def test_kv4_attention_vs_scipy_softmax():
    special = pytest.importorskip("scipy.special")
    d, L, G = 128, 77, 4
    Q = _kv(G, d, 9)
    Kq, Ks, Kz = oracle.kv4_quantize(_kv(L, d, 10, outliers=2))
    Vq, Vs, Vz = oracle.kv4_quantize(_kv(L, d, 11))
    scale = 1.0 / np.sqrt(d)
    O = oracle.kv4_attention_f64(Q, Kq, Ks, Kz, Vq, Vs, Vz, scale)
    P = special.softmax(scale * Q.astype(np.float64) @ _deq(Kq, Ks, Kz).T, axis=1)
    assert np.allclose(O, P @ _deq(Vq, Vs, Vz), rtol=1e-12, atol=1e-12)
