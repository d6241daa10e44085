"""QoQ W4A8 oracle -- test infrastructure, not product code.

A numpy front end over the plain single-threaded C restatement in
``qoq_oracle.c`` (built with gcc, no fast-math, no FP contraction).  Only the
test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it and
it never imports the CUDA library.

Every function cites the passage of the QServe pages it restates; see the
header of ``qoq_oracle.c`` for the page list.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qoq_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libqoq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_lib/libqoq_oracle.so``."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-fvisibility=hidden", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            sig = {
                "oracle_half_to_float": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_float_to_half_rn": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_rne_f32": (i64, [ctypes.c_float]),
                "oracle_rne_div": (i64, [i64, i64]),
                "oracle_group_step": (ctypes.c_int, [P, ctypes.c_int, P, P, P]),
                "oracle_quantize_weights_group": (i64, [P, i32, i32, i32, P, P, P, P, P]),
                "oracle_quantize_weights_channel": (None, [P, i32, i32, P, P, P]),
                "oracle_quant_act": (None, [P, i32, i32, P, P, P]),
                "oracle_gemm_i32_group": (None, [P, P, P, P, i32, i32, i32, i32, P]),
                "oracle_gemm_i32_group_at": (None, [P, P, P, P, i32, i32, i32, i32, P, P, i32, P]),
                "oracle_gemm_i32_channel": (None, [P, P, P, P, i32, i32, i32, P]),
                "oracle_gemm_i32_channel_at": (None, [P, P, P, P, i32, i32, i32, P, P, i32, P]),
                "oracle_epilogue_f64": (None, [P, P, P, i32, i32, P]),
                "oracle_rmsnorm_f64": (None, [P, P, ctypes.c_double, i32, i32, P]),
                "oracle_silu_mul_f64": (None, [P, i32, i32, P]),
                "oracle_kv4_quantize": (None, [P, i32, i32, P, P, P]),
                "oracle_kv4_attention_f64": (None, [P, i32, i32, i32, P, P, P, P, P, P, ctypes.c_double, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_half_bits(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    assert x.dtype == np.uint16
    return np.ascontiguousarray(x)


# --------------------------------------------------------------------------
# Scalars: IEEE binary16 conversion and round-half-even
# --------------------------------------------------------------------------
def half_to_float(bits: int) -> float:
    return float(_load().oracle_half_to_float(int(bits)))


def float_to_half_rn(x: float) -> int:
    return int(_load().oracle_float_to_half_rn(float(x)))


def rne_f32(x: float) -> int:
    return int(_load().oracle_rne_f32(float(x)))


def rne_div(a: int, b: int) -> int:
    return int(_load().oracle_rne_div(int(a), int(b)))


# --------------------------------------------------------------------------
# Progressive group quantization (QServe summary, "渐进式组量化" eq. 4/5,
# "保护性量化范围"; QServe review 3.1)
# --------------------------------------------------------------------------
def group_step(q8) -> tuple[np.ndarray, int, int, int]:
    """Step 2 on one group of INT8 intermediate codes.

    Returns (q4, s_g, z, n_overflow) where n_overflow counts reconstructions
    (q4 - z) * s_g outside [-128, 127].
    """
    q8 = np.ascontiguousarray(np.asarray(q8, dtype=np.int32))
    q4 = np.zeros(q8.shape[0], np.uint8)
    sg = np.zeros(1, np.uint8)
    z = np.zeros(1, np.uint8)
    bad = _load().oracle_group_step(_p(q8), q8.shape[0], _p(q4), _p(sg), _p(z))
    return q4, int(sg[0]), int(z[0]), int(bad)


def quantize_weights_group(W, g: int = 128):
    """W fp16 [N][K] -> dict(q4 [N][K] u8, s_g [N][K/g] u8, z [N][K/g] u8,
    s_w [N] fp16, q8 [N][K] i8, n_overflow)."""
    W = _as_half_bits(W)
    N, K = W.shape
    assert K % g == 0
    G = K // g
    q4 = np.zeros((N, K), np.uint8)
    sg = np.zeros((N, G), np.uint8)
    z = np.zeros((N, G), np.uint8)
    sw = np.zeros(N, np.uint16)
    q8 = np.zeros((N, K), np.int8)
    bad = _load().oracle_quantize_weights_group(_p(W), N, K, g, _p(q4), _p(sg), _p(z), _p(sw), _p(q8))
    return dict(q4=q4, s_g=sg, z=z, s_w=sw.view(np.float16), q8=q8, n_overflow=int(bad))


def quantize_weights_channel(W):
    """Per-channel asymmetric UINT4: W fp16 [N][K] -> dict(q4, z [N], s_w [N] fp16)."""
    W = _as_half_bits(W)
    N, K = W.shape
    q4 = np.zeros((N, K), np.uint8)
    z = np.zeros(N, np.uint8)
    sw = np.zeros(N, np.uint16)
    _load().oracle_quantize_weights_channel(_p(W), N, K, _p(q4), _p(z), _p(sw))
    return dict(q4=q4, z=z, s_w=sw.view(np.float16))


def quant_act(X):
    """Per-token symmetric INT8: X fp16 [M][K] -> (Qx i8 [M][K], s_x fp16 [M], t_x i32 [M])."""
    X = _as_half_bits(X)
    M, K = X.shape
    Qx = np.zeros((M, K), np.int8)
    sx = np.zeros(M, np.uint16)
    tx = np.zeros(M, np.int32)
    _load().oracle_quant_act(_p(X), M, K, _p(Qx), _p(sx), _p(tx))
    return Qx, sx.view(np.float16), tx


# --------------------------------------------------------------------------
# Integer GEMMs and the fp64 epilogue
# --------------------------------------------------------------------------
def gemm_i32_group(Qx, q4, s_g, z, g: int = 128) -> np.ndarray:
    Qx = np.ascontiguousarray(Qx, dtype=np.int8)
    q4 = np.ascontiguousarray(q4, dtype=np.uint8)
    s_g = np.ascontiguousarray(s_g, dtype=np.uint8)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    M, K = Qx.shape
    N = q4.shape[0]
    acc = np.zeros((M, N), np.int32)
    _load().oracle_gemm_i32_group(_p(Qx), _p(q4), _p(s_g), _p(z), M, N, K, g, _p(acc))
    return acc


def gemm_i32_group_at(Qx, q4, s_g, z, ms, ns, g: int = 128) -> np.ndarray:
    Qx = np.ascontiguousarray(Qx, dtype=np.int8)
    q4 = np.ascontiguousarray(q4, dtype=np.uint8)
    s_g = np.ascontiguousarray(s_g, dtype=np.uint8)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    ms = np.ascontiguousarray(ms, dtype=np.int32)
    ns = np.ascontiguousarray(ns, dtype=np.int32)
    M, K = Qx.shape
    N = q4.shape[0]
    out = np.zeros(ms.shape[0], np.int32)
    _load().oracle_gemm_i32_group_at(_p(Qx), _p(q4), _p(s_g), _p(z), M, N, K, g,
                                     _p(ms), _p(ns), ms.shape[0], _p(out))
    return out


def gemm_i32_channel(Qx, t_x, q4, z) -> np.ndarray:
    Qx = np.ascontiguousarray(Qx, dtype=np.int8)
    t_x = np.ascontiguousarray(t_x, dtype=np.int32)
    q4 = np.ascontiguousarray(q4, dtype=np.uint8)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    M, K = Qx.shape
    N = q4.shape[0]
    acc = np.zeros((M, N), np.int32)
    _load().oracle_gemm_i32_channel(_p(Qx), _p(t_x), _p(q4), _p(z), M, N, K, _p(acc))
    return acc


def gemm_i32_channel_at(Qx, t_x, q4, z, ms, ns) -> np.ndarray:
    Qx = np.ascontiguousarray(Qx, dtype=np.int8)
    t_x = np.ascontiguousarray(t_x, dtype=np.int32)
    q4 = np.ascontiguousarray(q4, dtype=np.uint8)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    ms = np.ascontiguousarray(ms, dtype=np.int32)
    ns = np.ascontiguousarray(ns, dtype=np.int32)
    M, K = Qx.shape
    N = q4.shape[0]
    out = np.zeros(ms.shape[0], np.int32)
    _load().oracle_gemm_i32_channel_at(_p(Qx), _p(t_x), _p(q4), _p(z), M, N, K,
                                       _p(ms), _p(ns), ms.shape[0], _p(out))
    return out


def epilogue_f64(acc, s_x, s_w) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    M, N = acc.shape
    sx = _as_half_bits(s_x)
    sw = _as_half_bits(s_w)
    O = np.zeros((M, N), np.float64)
    _load().oracle_epilogue_f64(_p(acc), _p(sx), _p(sw), M, N, _p(O))
    return O


# --------------------------------------------------------------------------
# The fp16 kernels in front of the GEMMs, into which the activation
# quantization is fused (QServe summary, "QServe系统运行时"; QServe review
# section 4, step 2)
# --------------------------------------------------------------------------
def rmsnorm_f64(X, gamma, eps: float) -> np.ndarray:
    """Y = gamma * X / sqrt(mean(X^2) + eps) per row, in fp64 (X [M][K],
    gamma [K] fp16)."""
    X = _as_half_bits(X)
    gamma = _as_half_bits(gamma)
    M, K = X.shape
    assert gamma.shape == (K,)
    Y = np.zeros((M, K), np.float64)
    _load().oracle_rmsnorm_f64(_p(X), _p(gamma), float(eps), M, K, _p(Y))
    return Y


def silu_mul_f64(H) -> np.ndarray:
    """A = SiLU(G) * U, in fp64, for H = [G | U] of shape [M][2F] (fp16)."""
    H = _as_half_bits(H)
    M, F2 = H.shape
    assert F2 % 2 == 0
    A = np.zeros((M, F2 // 2), np.float64)
    _load().oracle_silu_mul_f64(_p(H), M, F2 // 2, _p(A))
    return A


# --------------------------------------------------------------------------
# KV4 cache quantization and decode attention (QServe summary, KV cache
# management in "QServe系统运行时" and "QServe中的KV4注意力"; QServe review 3.2)
# --------------------------------------------------------------------------
def kv4_quantize(x):
    """Per-vector asymmetric UINT4 with fp16 scale and zero: x fp16 [n][d] ->
    (codes u8 [n][d], s fp16 [n], z fp16 [n]); x ~ (codes - z) * s."""
    x = _as_half_bits(x)
    n, d = x.shape
    q = np.zeros((n, d), np.uint8)
    s = np.zeros(n, np.uint16)
    z = np.zeros(n, np.uint16)
    _load().oracle_kv4_quantize(_p(x), n, d, _p(q), _p(s), _p(z))
    return q, s.view(np.float16), z.view(np.float16)


def kv4_attention_f64(Q, Kq, Ks, Kz, Vq, Vs, Vz, scale: float) -> np.ndarray:
    """softmax(scale * Q Khat^T) Vhat for the G query heads of one KV head
    and one sequence, in fp64: Q fp16 [G][d]; K/V codes [L][d], scales and
    zeros fp16 [L] -> O [G][d]."""
    Q = _as_half_bits(Q)
    G, d = Q.shape
    Kq = np.ascontiguousarray(Kq, dtype=np.uint8)
    Vq = np.ascontiguousarray(Vq, dtype=np.uint8)
    L = Kq.shape[0]
    assert L >= 1 and Kq.shape == (L, d) and Vq.shape == (L, d)
    Ks, Kz, Vs, Vz = (_as_half_bits(a) for a in (Ks, Kz, Vs, Vz))
    O = np.zeros((G, d), np.float64)
    _load().oracle_kv4_attention_f64(_p(Q), G, d, L, _p(Kq), _p(Ks), _p(Kz), _p(Vq), _p(Vs), _p(Vz),
                                     float(scale), _p(O))
    return O


def fp16_within_one_ulp(Y16, Y_ref) -> np.ndarray:
    """Per element: |Y16 - Y_ref| <= ulp16(|Y_ref|), the bound of an fp16
    result rounded from an fp32 computation of Y_ref (relative error far below
    2^-11) -- half an ulp for the final rounding plus the fp32 error."""
    Y16 = np.asarray(Y16, dtype=np.float64)
    Y_ref = np.asarray(Y_ref, dtype=np.float64)
    return np.abs(Y16 - Y_ref) <= fp16_ulp(Y_ref)


def fp16_ulp(x) -> np.ndarray:
    """Spacing of binary16 values at |x| (2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def o_within_tolerance(O_gpu, O_ref) -> np.ndarray:
    """Per-element check of the fp16 output bound, row by row:
    |O_gpu - O_ref| <= 2e-3 * max_n |O_ref[m, :]| + ulp16(|O_ref[m, n]|)."""
    O_gpu = np.asarray(O_gpu, dtype=np.float64)
    O_ref = np.asarray(O_ref, dtype=np.float64)
    rowmax = np.max(np.abs(O_ref), axis=1, keepdims=True) if O_ref.shape[1] else 0.0
    bound = 2e-3 * rowmax + fp16_ulp(O_ref)
    return np.abs(O_gpu - O_ref) <= bound


def reference_forward_group(W, X, g: int = 128):
    """Whole path on the CPU: quantize W and X, integer GEMM, fp64 epilogue."""
    wq = quantize_weights_group(W, g)
    Qx, sx, tx = quant_act(X)
    acc = gemm_i32_group(Qx, wq["q4"], wq["s_g"], wq["z"], g)
    O = epilogue_f64(acc, sx, wq["s_w"])
    return dict(wq=wq, Qx=Qx, s_x=sx, t_x=tx, acc=acc, O=O)
