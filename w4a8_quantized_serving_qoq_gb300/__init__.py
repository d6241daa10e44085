"""GB300-native W4A8 GEMM: the hot path of the QoQ / QServe method.

A thin ctypes binding over ``libqoq.so`` (C ABI declared in
``include/qoq.h``).  Each function has the name of the C entry point and does
argument marshalling only: torch tensors provide device memory and the
current CUDA stream; every step of the computation runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing or fails
to load, every call raises.  With QOQ_DEBUG=1 in the environment at the first
call, the bounds-check build ``libqoq_debug.so`` is loaded instead (see
qoq_bounds_checked in ``include/qoq.h``).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build

_lock = threading.Lock()
_lib = None

QOQ_OK = 0
QOQ_LAUNCH_OVERLAP = 1  # programmatic dependent launch (include/qoq.h)
QOQ_PLAN_RULES = 2      # plan by the rules alone, not the measured dispatch table
STATUS_NAMES = {
    0: "QOQ_OK", 1: "QOQ_ERR_INVALID_ARG", 2: "QOQ_ERR_UNSUPPORTED", 3: "QOQ_ERR_MISALIGNED",
    4: "QOQ_ERR_WORKSPACE", 5: "QOQ_ERR_CUDA", 6: "QOQ_ERR_TIMEOUT", 7: "QOQ_ERR_DEVICE",
}


class QoqError(RuntimeError):
    def __init__(self, func: str, status: int):
        super().__init__(f"{func} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


class qoq_gemm_options(ctypes.Structure):
    _fields_ = [
        ("tokens_per_tile", ctypes.c_int),
        ("num_ctas", ctypes.c_int),
        ("timeout_ns", ctypes.c_uint64),
        ("debug_flags", ctypes.c_uint32),
        ("acc_out", ctypes.c_void_p),
        ("kernel", ctypes.c_int),
        ("act_operand", ctypes.c_void_p),
        ("flags", ctypes.c_uint32),
        ("schedule", ctypes.c_int),
    ]


def debug_build_requested() -> bool:
    """True when QOQ_DEBUG=1 asks for the bounds-check library."""
    return os.environ.get("QOQ_DEBUG", "") == "1"


def library_path() -> str:
    return _build.library(debug_build_requested())


def build(force: bool = False) -> str:
    """Compile libqoq.so and libqoq_debug.so for sm_103a (in-tree)."""
    return _build.build(force=force)


def header_functions() -> list[str]:
    """Names of the functions declared in include/qoq.h."""
    path = os.path.join(_build.ROOT, "include", "qoq.h")
    text = open(path).read()
    return sorted(set(re.findall(r"\b(qoq_[a-z0-9_]+)\s*\(", text)) - {"qoq_gemm_options"})


class qoq_gemm_plan_info(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int),
        ("tokens_per_tile", ctypes.c_int),
        ("num_ctas", ctypes.c_int),
        ("tiles", ctypes.c_longlong),
        ("k_stages", ctypes.c_longlong),
        ("workspace_bytes", ctypes.c_size_t),
    ]


def load():
    """Load libqoq.so (building it first if it is missing or stale)."""
    global _lib
    lib = _lib
    if lib is not None:  # fast path: every entry point calls this
        return lib
    with _lock:
        if _lib is None:
            dbg = debug_build_requested()
            if not _build.up_to_date(dbg):
                _build.build(debug=dbg)
            lib = ctypes.CDLL(_build.library(dbg))
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            sigs = {
                "qoq_status_string": (ctypes.c_char_p, [I]),
                "qoq_version": (I, []),
                "qoq_bounds_checked": (I, []),
                "qoq_quantize_weights": (I, [P, I, I, I, P, P, P, P, P]),
                "qoq_packed_weight_bytes": (S, [I, I, I]),
                "qoq_pack_weights": (I, [P, P, P, I, I, I, P, P]),
                "qoq_unpack_weights": (I, [P, I, I, I, P, P, P, P]),
                "qoq_quant_act": (I, [P, I, I, P, P, P, P]),
                "qoq_act_operand_bytes": (S, [I, I, I]),
                "qoq_quant_act_ex": (I, [P, I, I, P, P, P, I, P, ctypes.c_uint32, P]),
                "qoq_rmsnorm_quant_act": (I, [P, P, ctypes.c_float, I, I, P, P, P, I, P, P, ctypes.c_uint32, P]),
                "qoq_silu_mul_quant_act": (I, [P, I, I, P, P, P, I, P, P, ctypes.c_uint32, P]),
                "qoq_kv4_page_bytes": (S, [I]),
                "qoq_kv4_append": (I, [P, P, I, I, P, P, P, I, I, P, I, P, P]),
                "qoq_kv4_attention_workspace_bytes": (S, [I, I, I, I]),
                "qoq_kv4_decode_attention": (I, [P, P, I, P, P, I, I, I, I, ctypes.c_float, P, P, S, P]),
                "qoq_gemm_workspace_bytes": (S, [I, I, I, I]),
                "qoq_gemm_workspace_bytes_ex": (S, [I, I, I, I, ctypes.POINTER(qoq_gemm_options)]),
                "qoq_gemm_path": (I, [I, I, I, I, ctypes.POINTER(qoq_gemm_options)]),
                "qoq_gemm_plan": (I, [I, I, I, I, I, ctypes.POINTER(qoq_gemm_options),
                                      ctypes.POINTER(qoq_gemm_plan_info)]),
                "qoq_workspace_init": (I, [P, S, P]),
                "qoq_w4a8_gemm": (I, [P, P, P, P, P, I, I, I, I, P, P, S, P]),
                "qoq_w4a8_gemm_i32": (I, [P, P, P, I, I, I, I, P, P, S, P]),
                "qoq_w4a8_gemm_ex": (I, [P, P, P, P, P, I, I, I, I, P, P, S,
                                         ctypes.POINTER(qoq_gemm_options), P]),
                "qoq_workspace_status": (I, [P, ctypes.POINTER(ctypes.c_uint32), P]),
                "qoq_w4a8_gemm_noalloc": (I, [P, P, P, P, P, I, I, I, I, P, P]),
                "qoq_noalloc_status": (I, [ctypes.POINTER(ctypes.c_uint32), P]),
            }
            for name, (res, args) in sigs.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


# ---------------------------------------------------------------- helpers --
_torch_mod = None
_raw_stream = None


def _torch():
    global _torch_mod
    if _torch_mod is None:
        import torch
        _torch_mod = torch
    return _torch_mod


def _stream(stream, device=None):
    """cudaStream_t of `stream`, else of the current stream of `device` (a
    torch.device or index; None: the current device)."""
    global _raw_stream
    if stream is not None:
        return stream.cuda_stream
    torch = _torch()
    if _raw_stream is None:
        # The raw handle of the current stream, as torch's own generated code
        # reads it; the public call builds a Stream object each time.
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _raw_stream:
        if device is None:
            index = torch.cuda.current_device()
        else:
            index = device.index if isinstance(device, torch.device) else int(device)
            if index is None:
                index = torch.cuda.current_device()
        return _raw_stream(index)
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    """Device address of a tensor as an int (the prototypes declare c_void_p)."""
    return None if t is None else t.data_ptr()


def _dev(t, dtype, name):
    torch = _torch()
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    _ = torch


def _check(func: str, status: int):
    if status != QOQ_OK:
        raise QoqError(func, status)


# ------------------------------------------------------------ entry points --
def qoq_status_string(status: int) -> str:
    return load().qoq_status_string(int(status)).decode()


def qoq_version() -> int:
    return int(load().qoq_version())


def qoq_bounds_checked() -> bool:
    """True when the loaded library is the bounds-check build."""
    return bool(load().qoq_bounds_checked())


def qoq_quantize_weights(W, group: int = 128, stream=None):
    """fp16 W [N][K] -> dict(q4 [N][K] u8, s_g [N][K/128] u8 or None, z, s_w fp16 [N])."""
    torch = _torch()
    _dev(W, torch.float16, "W")
    N, K = W.shape
    q4 = torch.empty((N, K), dtype=torch.uint8, device=W.device)
    s_g = torch.empty((N, K // 128), dtype=torch.uint8, device=W.device) if group else None
    z = torch.empty((N, K // 128) if group else (N,), dtype=torch.uint8, device=W.device)
    s_w = torch.empty((N,), dtype=torch.float16, device=W.device)
    _check("qoq_quantize_weights", load().qoq_quantize_weights(
        _ptr(W), N, K, group, _ptr(q4), _ptr(s_g), _ptr(z), _ptr(s_w), _stream(stream)))
    return dict(q4=q4, s_g=s_g, z=z, s_w=s_w)


def qoq_packed_weight_bytes(N: int, K: int, group: int = 128) -> int:
    return int(load().qoq_packed_weight_bytes(N, K, group))


def qoq_pack_weights(q4, s_g, z, group: int = 128, packed=None, stream=None):
    torch = _torch()
    _dev(q4, torch.uint8, "q4")
    _dev(s_g, torch.uint8, "s_g")
    _dev(z, torch.uint8, "z")
    N, K = q4.shape
    nbytes = qoq_packed_weight_bytes(N, K, group)
    if nbytes == 0:
        raise QoqError("qoq_pack_weights", 2)
    if packed is None:
        packed = torch.empty((nbytes,), dtype=torch.uint8, device=q4.device)
    _dev(packed, torch.uint8, "packed")
    _check("qoq_pack_weights", load().qoq_pack_weights(
        _ptr(q4), _ptr(s_g), _ptr(z), N, K, group, _ptr(packed), _stream(stream)))
    return packed


def qoq_unpack_weights(packed, N: int, K: int, group: int = 128, stream=None):
    torch = _torch()
    _dev(packed, torch.uint8, "packed")
    q4 = torch.empty((N, K), dtype=torch.uint8, device=packed.device)
    s_g = torch.empty((N, K // 128), dtype=torch.uint8, device=packed.device) if group else None
    z = torch.empty((N, K // 128) if group else (N,), dtype=torch.uint8, device=packed.device)
    _check("qoq_unpack_weights", load().qoq_unpack_weights(
        _ptr(packed), N, K, group, _ptr(q4), _ptr(s_g), _ptr(z), _stream(stream)))
    return q4, s_g, z


def qoq_quant_act(X, Qx=None, s_x=None, t_x=None, with_t: bool = True, stream=None):
    """fp16 X [M][K] -> (Qx int8 [M][K], s_x fp16 [M], t_x int32 [M] or None)."""
    torch = _torch()
    _dev(X, torch.float16, "X")
    M, K = X.shape
    if Qx is None:
        Qx = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float16, device=X.device)
    if t_x is None and with_t:
        t_x = torch.empty((M,), dtype=torch.int32, device=X.device)
    _dev(Qx, torch.int8, "Qx")
    _dev(s_x, torch.float16, "s_x")
    _dev(t_x, torch.int32, "t_x")
    _check("qoq_quant_act", load().qoq_quant_act(
        _ptr(X), M, K, _ptr(Qx), _ptr(s_x), _ptr(t_x), _stream(stream)))
    return Qx, s_x, t_x


def qoq_act_operand_bytes(M: int, K: int, kind: int) -> int:
    return int(load().qoq_act_operand_bytes(M, K, kind))


def qoq_quant_act_ex(X, Qx=None, s_x=None, t_x=None, act=None, kind: int = 2, with_t: bool = True,
                     with_act: bool = True, flags: int = 0, stream=None):
    """qoq_quant_act plus the activation operand of `kind` (1: fp16 copy of
    Qx for the fp16-operand path, 2: fp8-path planes and group sums), a uint8
    tensor of qoq_act_operand_bytes(M, K, kind) bytes -> (Qx, s_x, t_x, act)."""
    torch = _torch()
    _dev(X, torch.float16, "X")
    M, K = X.shape
    if Qx is None:
        Qx = torch.empty((M, K), dtype=torch.int8, device=X.device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float16, device=X.device)
    if t_x is None and with_t:
        t_x = torch.empty((M,), dtype=torch.int32, device=X.device)
    if act is None and with_act and kind != 3:  # kind 3: the CUDA-core GEMM reads Qx, no operand
        nbytes = qoq_act_operand_bytes(M, K, kind)
        if nbytes == 0:
            raise QoqError("qoq_quant_act_ex", 2)
        act = torch.empty((nbytes,), dtype=torch.uint8, device=X.device)
    _dev(Qx, torch.int8, "Qx")
    _dev(s_x, torch.float16, "s_x")
    _dev(t_x, torch.int32, "t_x")
    _dev(act, torch.uint8, "act")
    _check("qoq_quant_act_ex", load().qoq_quant_act_ex(
        _ptr(X), M, K, _ptr(Qx), _ptr(s_x), _ptr(t_x), int(kind), _ptr(act), int(flags), _stream(stream)))
    return Qx, s_x, t_x, act


def _quant_outputs(M, K, device, Qx, s_x, t_x, act, kind, with_t, with_act, Y, with_y):
    torch = _torch()
    if Qx is None:
        Qx = torch.empty((M, K), dtype=torch.int8, device=device)
    if s_x is None:
        s_x = torch.empty((M,), dtype=torch.float16, device=device)
    if t_x is None and with_t:
        t_x = torch.empty((M,), dtype=torch.int32, device=device)
    if act is None and with_act and kind != 3:
        nbytes = qoq_act_operand_bytes(M, K, kind)
        if nbytes == 0:
            raise QoqError("qoq_act_operand_bytes", 2)
        act = torch.empty((nbytes,), dtype=torch.uint8, device=device)
    if Y is None and with_y:
        Y = torch.empty((M, K), dtype=torch.float16, device=device)
    _dev(Qx, torch.int8, "Qx")
    _dev(s_x, torch.float16, "s_x")
    _dev(t_x, torch.int32, "t_x")
    _dev(act, torch.uint8, "act")
    _dev(Y, torch.float16, "Y")
    return Qx, s_x, t_x, act, Y


def qoq_rmsnorm_quant_act(X, gamma, eps: float = 1e-5, Qx=None, s_x=None, t_x=None, act=None, kind: int = 2,
                          with_t: bool = True, with_act: bool = True, Y=None, with_y: bool = False,
                          flags: int = 0, stream=None):
    """RMS norm of X [M][K] (gamma [K]) fused with the per-token INT8
    quantization -> (Qx, s_x, t_x, act, Y); Y is the fp16 normalized rows
    (only with with_y or a given Y)."""
    torch = _torch()
    _dev(X, torch.float16, "X")
    _dev(gamma, torch.float16, "gamma")
    M, K = X.shape
    Qx, s_x, t_x, act, Y = _quant_outputs(M, K, X.device, Qx, s_x, t_x, act, kind, with_t, with_act, Y, with_y)
    _check("qoq_rmsnorm_quant_act", load().qoq_rmsnorm_quant_act(
        _ptr(X), _ptr(gamma), float(eps), M, K, _ptr(Qx), _ptr(s_x), _ptr(t_x), int(kind), _ptr(act), _ptr(Y),
        int(flags), _stream(stream)))
    return Qx, s_x, t_x, act, Y


def qoq_silu_mul_quant_act(H, Qx=None, s_x=None, t_x=None, act=None, kind: int = 2, with_t: bool = True,
                           with_act: bool = True, Y=None, with_y: bool = False, flags: int = 0, stream=None):
    """SiLU(G) * U of H = [G | U] [M][2F] fused with the per-token INT8
    quantization -> (Qx, s_x, t_x, act, Y) over F columns."""
    torch = _torch()
    _dev(H, torch.float16, "H")
    M, F2 = H.shape
    F = F2 // 2
    Qx, s_x, t_x, act, Y = _quant_outputs(M, F, H.device, Qx, s_x, t_x, act, kind, with_t, with_act, Y, with_y)
    _check("qoq_silu_mul_quant_act", load().qoq_silu_mul_quant_act(
        _ptr(H), M, F, _ptr(Qx), _ptr(s_x), _ptr(t_x), int(kind), _ptr(act), _ptr(Y), int(flags),
        _stream(stream)))
    return Qx, s_x, t_x, act, Y


def qoq_gemm_workspace_bytes(M: int, N: int, K: int, group: int = 128, options=None) -> int:
    if options is None:
        return int(load().qoq_gemm_workspace_bytes(M, N, K, group))
    return int(load().qoq_gemm_workspace_bytes_ex(M, N, K, group, ctypes.byref(options)))


def qoq_gemm_path(M: int, N: int, K: int, group: int = 128, options=None) -> int:
    """1 = fp16-operand path, 2 = fp8-operand path (each reads the activation
    operand of its kind), 3 = CUDA-core path for M <= 8 (reads Qx itself)."""
    st = int(load().qoq_gemm_path(M, N, K, group, None if options is None else ctypes.byref(options)))
    if st < 0:
        raise QoqError("qoq_gemm_path", -st)
    return st


def qoq_gemm_plan(M: int, N: int, K: int, group: int = 128, num_sms: int = 152, options=None) -> dict:
    """The launch plan on a GPU with num_sms SMs (host only, no GPU needed)."""
    info = qoq_gemm_plan_info()
    _check("qoq_gemm_plan", load().qoq_gemm_plan(M, N, K, group, num_sms,
                                                 None if options is None else ctypes.byref(options),
                                                 ctypes.byref(info)))
    return {f: getattr(info, f) for f, _ in qoq_gemm_plan_info._fields_}


def qoq_workspace_init(workspace, stream=None):
    _check("qoq_workspace_init", load().qoq_workspace_init(
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def new_workspace(nbytes: int, device="cuda", stream=None):
    """A zero-filled workspace tensor of at least nbytes (16-byte aligned)."""
    torch = _torch()
    ws = torch.empty((max(256, (nbytes + 255) // 256 * 256),), dtype=torch.uint8, device=device)
    qoq_workspace_init(ws, stream)
    return ws


def qoq_w4a8_gemm(Qx, s_x, t_x, packed, s_w, N: int, K: int, group: int = 128, O=None,
                  workspace=None, stream=None):
    torch = _torch()
    _dev(Qx, torch.int8, "Qx")
    M = Qx.shape[0]
    if O is None:
        O = torch.empty((M, N), dtype=torch.float16, device=Qx.device)
    if workspace is None:
        workspace = new_workspace(qoq_gemm_workspace_bytes(M, N, K, group), Qx.device, stream)
    _check("qoq_w4a8_gemm", load().qoq_w4a8_gemm(
        _ptr(Qx), _ptr(s_x), _ptr(t_x), _ptr(packed), _ptr(s_w), M, N, K, group, _ptr(O),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return O


def qoq_w4a8_gemm_i32(Qx, t_x, packed, N: int, K: int, group: int = 128, acc=None,
                      workspace=None, stream=None):
    torch = _torch()
    _dev(Qx, torch.int8, "Qx")
    M = Qx.shape[0]
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=Qx.device)
    if workspace is None:
        workspace = new_workspace(qoq_gemm_workspace_bytes(M, N, K, group), Qx.device, stream)
    _check("qoq_w4a8_gemm_i32", load().qoq_w4a8_gemm_i32(
        _ptr(Qx), _ptr(t_x), _ptr(packed), M, N, K, group, _ptr(acc), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return acc


def gemm_options(tokens_per_tile=0, num_ctas=0, timeout_ns=0, debug_flags=0, acc_out=None, kernel=0,
                 act_operand=None, flags=0, schedule=0):
    return qoq_gemm_options(tokens_per_tile, num_ctas, timeout_ns, debug_flags,
                            None if acc_out is None else acc_out.data_ptr(), kernel,
                            None if act_operand is None else act_operand.data_ptr(), flags, schedule)


def qoq_w4a8_gemm_ex(Qx, s_x, t_x, packed, s_w, N: int, K: int, group: int = 128, O=None,
                     workspace=None, options=None, stream=None, check: bool = True):
    torch = _torch()
    _dev(Qx, torch.int8, "Qx")
    M = Qx.shape[0]
    if options is None:
        options = qoq_gemm_options()
    if O is None and not options.acc_out:
        O = torch.empty((M, N), dtype=torch.float16, device=Qx.device)
    if workspace is None:
        workspace = new_workspace(qoq_gemm_workspace_bytes(M, N, K, group, options), Qx.device, stream)
    st = load().qoq_w4a8_gemm_ex(
        _ptr(Qx), _ptr(s_x), _ptr(t_x), _ptr(packed), _ptr(s_w), M, N, K, group, _ptr(O),
        _ptr(workspace), workspace.numel(), ctypes.byref(options), _stream(stream))
    if check:
        _check("qoq_w4a8_gemm_ex", st)
        return O
    return st


def qoq_w4a8_gemm_noalloc(Qx, s_x, t_x, packed, s_w, N: int, K: int, group: int = 128, O=None,
                          stream=None):
    """The GEMM for callers that cannot allocate device memory: the scratch
    comes from a fixed array inside the library (see include/qoq.h for its
    size limit and the rule that overlapping calls race)."""
    torch = _torch()
    _dev(Qx, torch.int8, "Qx")
    M = Qx.shape[0]
    if O is None:
        O = torch.empty((M, N), dtype=torch.float16, device=Qx.device)
    _check("qoq_w4a8_gemm_noalloc", load().qoq_w4a8_gemm_noalloc(
        _ptr(Qx), _ptr(s_x), _ptr(t_x), _ptr(packed), _ptr(s_w), M, N, K, group, _ptr(O),
        _stream(stream)))
    return O


# ------------------------------------------------------------------- KV4 --
QOQ_KV4_PAGE_TOKENS = 64
QOQ_KV4_HEAD_DIM = 128


def qoq_kv4_page_bytes(num_kv_heads: int) -> int:
    return int(load().qoq_kv4_page_bytes(num_kv_heads))


def qoq_kv4_append(K, V, token_seq, token_pos, page_table, pages, status=None, stream=None):
    """Quantize K, V fp16 [T][H_kv][128] into their slots of the uint8 page
    pool `pages` ([num_pages][page bytes]); token t -> (token_seq[t],
    token_pos[t]) through page_table int32 [num_seqs][max_pages]."""
    torch = _torch()
    _dev(K, torch.float16, "K")
    _dev(V, torch.float16, "V")
    _dev(token_seq, torch.int32, "token_seq")
    _dev(token_pos, torch.int32, "token_pos")
    _dev(page_table, torch.int32, "page_table")
    _dev(pages, torch.uint8, "pages")
    _dev(status, torch.int32, "status")
    T, H = K.shape[0], K.shape[1]
    num_seqs, max_pages = page_table.shape
    num_pages = pages.shape[0]
    _check("qoq_kv4_append", load().qoq_kv4_append(
        _ptr(K), _ptr(V), T, H, _ptr(token_seq), _ptr(token_pos), _ptr(page_table), num_seqs, max_pages,
        _ptr(pages), num_pages, _ptr(status), _stream(stream)))


def qoq_kv4_attention_workspace_bytes(B: int, num_q_heads: int, num_kv_heads: int, max_pages: int) -> int:
    return int(load().qoq_kv4_attention_workspace_bytes(B, num_q_heads, num_kv_heads, max_pages))


def qoq_kv4_decode_attention(Q, pages, page_table, seq_lens, num_kv_heads: int, softmax_scale: float, O=None,
                             workspace=None, stream=None):
    """Decode attention over the KV4 page pool: Q fp16 [B][H_q][128] -> O."""
    torch = _torch()
    _dev(Q, torch.float16, "Q")
    _dev(pages, torch.uint8, "pages")
    _dev(page_table, torch.int32, "page_table")
    _dev(seq_lens, torch.int32, "seq_lens")
    B, Hq = Q.shape[0], Q.shape[1]
    max_pages = page_table.shape[1]
    if O is None:
        O = torch.empty_like(Q)
    _dev(O, torch.float16, "O")
    if workspace is None:
        workspace = new_workspace(qoq_kv4_attention_workspace_bytes(B, Hq, num_kv_heads, max_pages), Q.device, stream)
    _check("qoq_kv4_decode_attention", load().qoq_kv4_decode_attention(
        _ptr(Q), _ptr(pages), pages.shape[0], _ptr(page_table), _ptr(seq_lens), B, Hq, num_kv_heads, max_pages,
        float(softmax_scale), _ptr(O), _ptr(workspace), workspace.numel(), _stream(stream)))
    return O


def qoq_noalloc_status(stream=None):
    """(status code, raw status bits) of the allocation-free GEMM's internal
    array on the current device; synchronizes the stream and clears the word."""
    bits = ctypes.c_uint32(0)
    st = load().qoq_noalloc_status(ctypes.byref(bits), _stream(stream))
    return int(st), int(bits.value)


def qoq_workspace_status(workspace, stream=None):
    """(status code, raw status bits); synchronizes the stream."""
    bits = ctypes.c_uint32(0)
    st = load().qoq_workspace_status(_ptr(workspace), ctypes.byref(bits), _stream(stream))
    return int(st), int(bits.value)


__all__ = [n for n in dir() if n.startswith("qoq_")] + [
    "QoqError", "build", "load", "library_path", "debug_build_requested", "header_functions", "new_workspace",
    "gemm_options",
    "QOQ_LAUNCH_OVERLAP", "QOQ_PLAN_RULES",
]
