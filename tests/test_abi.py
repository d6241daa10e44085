"""Host-only checks of the C ABI: the library loads, exports every function
include/qoq.h declares, and rejects bad arguments before any launch."""
import ctypes

import pytest

import w4a8_quantized_serving_qoq_gb300 as qoq


@pytest.fixture(scope="module")
def lib():
    return qoq.load()


def test_exports_every_header_function(lib):
    names = qoq.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n


def test_loaded_library_matches_request(lib):
    """QOQ_DEBUG=1 loads the bounds-check build; otherwise the release one."""
    assert qoq.qoq_bounds_checked() == qoq.debug_build_requested()
    assert qoq.library_path().endswith("libqoq_debug.so" if qoq.debug_build_requested() else "libqoq.so")


def test_bounds_check_build_exports_every_header_function():
    """The bounds-check library is built beside the release one, exports the
    same C ABI and says which build it is."""
    from w4a8_quantized_serving_qoq_gb300 import _build
    _build.build(debug=True)
    dbg = ctypes.CDLL(_build.LIB_DEBUG)
    for n in qoq.header_functions():
        assert hasattr(dbg, n), n
    dbg.qoq_bounds_checked.restype = ctypes.c_int
    assert dbg.qoq_bounds_checked() == 1
    rel = ctypes.CDLL(_build.LIB)
    rel.qoq_bounds_checked.restype = ctypes.c_int
    assert rel.qoq_bounds_checked() == 0


def test_status_strings(lib):
    for code, name in qoq.STATUS_NAMES.items():
        assert qoq.qoq_status_string(code) == name
    assert qoq.qoq_status_string(99) == "QOQ_ERR_UNKNOWN"
    assert qoq.qoq_version() == 2


def test_packed_bytes_host_only(lib):
    # header + N*K/2 codes + (group) 4 bytes per row per group of 128
    assert qoq.qoq_packed_weight_bytes(256, 512, 128) == 256 + 256 * 512 // 2 + 256 * 4 * 4
    assert qoq.qoq_packed_weight_bytes(6144, 4096, 128) == 256 + 6144 * 2048 + 6144 * 32 * 4
    assert qoq.qoq_packed_weight_bytes(128, 128, 0) == 256 + 8192 + 128
    assert qoq.qoq_packed_weight_bytes(130, 128, 128) == 0
    assert qoq.qoq_packed_weight_bytes(128, 100, 128) == 0
    assert qoq.qoq_packed_weight_bytes(128, 128, 64) == 0


A = ctypes.c_void_p(0x10000)       # 16-byte aligned fake device address (never dereferenced)
B = ctypes.c_void_p(0x20008)       # 8-byte aligned, not 16
NUL = None
S = ctypes.c_void_p(0)


def test_gemm_validation_before_launch(lib):
    f = lib.qoq_w4a8_gemm
    ok = (A, A, A, A, A, 16, 256, 512, 128, A, A, 1 << 20, S)
    # null pointers
    assert f(NUL, *ok[1:]) == 1
    assert f(*ok[:3], NUL, *ok[4:]) == 1
    assert f(*ok[:10], NUL, *ok[11:]) == 1
    # non-positive sizes
    assert f(*ok[:5], 0, *ok[6:]) == 1
    assert f(*ok[:5], 16, -128, *ok[7:]) == 1
    # unsupported shapes / group
    assert f(*ok[:5], 16, 200, 512, 128, *ok[9:]) == 2
    assert f(*ok[:5], 16, 256, 500, 128, *ok[9:]) == 2
    assert f(*ok[:5], 16, 256, 512, 64, *ok[9:]) == 2
    # per-channel needs t_x
    assert f(A, A, NUL, A, A, 16, 256, 512, 0, A, A, 1 << 20, S) == 1
    # misaligned activations / packed / workspace
    assert f(B, *ok[1:]) == 3
    assert f(*ok[:3], B, *ok[4:]) == 3
    assert f(*ok[:10], B, *ok[11:]) == 3
    assert f(A, ctypes.c_void_p(0x10001), *ok[2:]) == 3
    # the fp16 output is written by tensor bulk copies: 16-byte aligned
    assert f(*ok[:9], ctypes.c_void_p(0x10008), *ok[10:]) == 3
    assert lib.qoq_w4a8_gemm_noalloc(A, A, NUL, A, A, 16, 256, 512, 128, ctypes.c_void_p(0x10008), S) == 3


def test_gemm_options_validation(lib):
    opt = qoq.qoq_gemm_options(48, 0, 0, 0, None)
    assert lib.qoq_w4a8_gemm_ex(A, A, A, A, A, 16, 256, 512, 128, A, A, 1 << 20,
                                ctypes.byref(opt), S) == 2
    opt = qoq.qoq_gemm_options(0, -1, 0, 0, None)
    assert lib.qoq_w4a8_gemm_ex(A, A, A, A, A, 16, 256, 512, 128, A, A, 1 << 20,
                                ctypes.byref(opt), S) == 2


def test_act_operand_entry_points_validation(lib):
    # sizes of both operand kinds; invalid shapes / kinds give 0
    assert lib.qoq_act_operand_bytes(5, 256, 1) == 2 * 5 * 256
    assert lib.qoq_act_operand_bytes(5, 256, 2) == 2 * 5 * 256 + 2 * 8 * 4
    assert lib.qoq_act_operand_bytes(5, 200, 1) == 0
    assert lib.qoq_act_operand_bytes(5, 256, 3) == 0
    assert lib.qoq_act_operand_bytes(0, 256, 1) == 0
    # quant_act_ex: bad kind with an operand, K not a multiple of 128, misaligned operand
    assert lib.qoq_quant_act_ex(A, 4, 512, A, A, A, 0, A, 0, S) == 1
    assert lib.qoq_quant_act_ex(A, 4, 520, A, A, A, 1, A, 0, S) == 2
    assert lib.qoq_quant_act_ex(A, 4, 512, A, A, A, 2, B, 0, S) == 3
    # unknown launch flags
    assert lib.qoq_quant_act_ex(A, 4, 512, A, A, A, 2, A, 2, S) == 2
    opt = qoq.qoq_gemm_options()
    opt.flags = 4
    assert lib.qoq_w4a8_gemm_ex(A, A, A, A, A, 16, 256, 512, 128, A, A, 1 << 20, ctypes.byref(opt), S) == 2
    # the path query validates like the GEMM
    assert lib.qoq_gemm_path(16, 200, 512, 128, None) == -2
    assert lib.qoq_gemm_path(0, 256, 512, 128, None) == -1


def test_other_entry_points_validation(lib):
    assert lib.qoq_quant_act(NUL, 4, 512, A, A, A, S) == 1
    assert lib.qoq_quant_act(A, 4, 500, A, A, A, S) == 2
    assert lib.qoq_quant_act(B, 4, 512, A, A, A, S) == 3
    assert lib.qoq_quant_act(A, 0, 512, A, A, A, S) == 1
    assert lib.qoq_pack_weights(A, A, A, 256, 512, 128, NUL, S) == 1
    assert lib.qoq_pack_weights(A, A, A, 250, 512, 128, A, S) == 2
    assert lib.qoq_pack_weights(B, A, A, 256, 512, 128, A, S) == 3
    assert lib.qoq_pack_weights(A, NUL, A, 256, 512, 128, A, S) == 1
    assert lib.qoq_unpack_weights(A, 256, 512, 7, A, A, A, S) == 2
    assert lib.qoq_quantize_weights(A, 256, 500, 128, A, A, A, A, S) == 2
    assert lib.qoq_quantize_weights(A, 256, 512, 128, A, NUL, A, A, S) == 1
    assert lib.qoq_workspace_init(NUL, 256, S) == 1
    st = ctypes.c_uint32(0)
    assert lib.qoq_workspace_status(NUL, ctypes.byref(st), S) == 1
    assert lib.qoq_workspace_status(B, ctypes.byref(st), S) == 3
