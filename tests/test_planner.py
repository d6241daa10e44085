"""The GEMM launch planner (qoq_gemm_plan, host only): which tensor-core path,
tile size and CTA count each Llama-3-8B decode shape gets on a 152-SM GB300,
the option overrides, the workspace layout and argument errors."""
import os
import re

import pytest

import w4a8_quantized_serving_qoq_gb300 as qoq

SMS = 152
QKV, O, GATE_UP, DOWN = (6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336)


def _plan(M, NK, group=128, **opt):
    """The planner's rules (the measured dispatch table is pinned separately)."""
    N, K = NK
    opt["flags"] = opt.get("flags", 0) | qoq.QOQ_PLAN_RULES
    return qoq.qoq_gemm_plan(M, N, K, group, SMS, qoq.gemm_options(**opt))


@pytest.mark.parametrize("M", [16, 32])
@pytest.mark.parametrize("NK", [QKV, O, GATE_UP, DOWN])
def test_decode_sizes_take_the_fp8_path_and_leave_8_sms(M, NK):
    p = _plan(M, NK)
    assert p["path"] == 2
    assert p["tokens_per_tile"] == (16 if M <= 16 else 32)
    assert p["num_ctas"] == SMS - 8
    assert p["tiles"] == (NK[0] // 128)
    assert p["k_stages"] == p["tiles"] * (NK[1] // 128)


@pytest.mark.parametrize("M,MT", [(1, 1), (2, 2), (3, 4), (4, 4)])
@pytest.mark.parametrize("NK,csize", [(QKV, 8), (O, 8), (GATE_UP, 4), (DOWN, 8), ((59136, 8192), 1),
                                      ((8192, 29568), 8)])
def test_up_to_4_tokens_take_the_cuda_core_path(M, MT, NK, csize):
    """M <= 4: the dp4a path, tokens rounded up to 1, 2 or 4; the K split
    (cluster size) is the largest of 8, 4, 2, 1 that keeps at most six CTAs
    per SM with a block per K half; only the status word in the workspace."""
    p = _plan(M, NK)
    assert (p["path"], p["tokens_per_tile"]) == (3, MT)
    assert p["num_ctas"] == (NK[0] // 128) * csize
    assert p["workspace_bytes"] == 256
    for group in (0, 128):
        assert _plan(M, NK, group=group)["path"] == 3


@pytest.mark.parametrize("M", [5, 8])
@pytest.mark.parametrize("NK", [QKV, GATE_UP, (59136, 8192)])
def test_5_to_8_tokens_take_the_tensor_cores_unless_forced(M, NK):
    """From 5 tokens the rules leave the dp4a path (its work per weight grows
    with the tokens): fp8 for g128, fp16 for per-channel weights; forcing the
    path still gives it, with 8-token tiles."""
    assert _plan(M, NK)["path"] == 2
    assert _plan(M, NK, group=0)["path"] == 1
    p = _plan(M, NK, kernel=3)
    assert (p["path"], p["tokens_per_tile"]) == (3, 8)


def test_cuda_core_path_options():
    assert _plan(1, O, kernel=3, num_ctas=2)["num_ctas"] == 32 * 2     # forced cluster size
    assert _plan(1, O, kernel=2)["path"] == 2                          # forced tensor-core path
    assert _plan(8, O, tokens_per_tile=16)["path"] == 2                # a token tile forces the tensor cores
    lib = qoq.load()
    info = qoq.qoq_gemm_plan_info()
    opt = qoq.gemm_options(kernel=3)
    # more than 8 tokens cannot take the CUDA-core path
    assert lib.qoq_gemm_plan(9, 4096, 4096, 128, SMS, qoq.ctypes.byref(opt), qoq.ctypes.byref(info)) == 2


def test_per_channel_weights_take_the_fp16_path_above_8_tokens():
    for M in (9, 32, 64, 256):
        assert _plan(M, GATE_UP, group=0)["path"] == 1


def test_half_width_tiles_when_a_launch_has_few_stages():
    # qkv at M = 64: 48 x 32 = 1536 stages at 64 tokens <= 16 x 152 -> 32-token fp8 tiles,
    # and 2 x 48 = 96 tiles fill 60 % of a wave -> one whole tile per CTA
    p = _plan(64, QKV)
    assert (p["path"], p["tokens_per_tile"], p["tiles"], p["num_ctas"]) == (2, 32, 96, 96)
    # o at M = 128: 32 x 32 = 1024 stages at 128 tokens -> 64-token fp16 tiles, stream-K over every SM
    p = _plan(128, O)
    assert (p["path"], p["tokens_per_tile"], p["tiles"], p["num_ctas"]) == (1, 64, 64, SMS)


def test_natural_tiles_for_long_launches():
    p = _plan(64, GATE_UP)  # 224 x 32 stages: no halving
    assert (p["path"], p["tokens_per_tile"], p["num_ctas"]) == (1, 64, SMS)
    p = _plan(256, GATE_UP)
    assert (p["path"], p["tokens_per_tile"], p["tiles"], p["k_stages"]) == (1, 128, 448, 448 * 32)
    p = _plan(256, QKV)  # 96 tiles of 128 tokens: one whole tile per CTA
    assert (p["tokens_per_tile"], p["tiles"], p["num_ctas"]) == (128, 96, 96)


def test_options_override_the_plan():
    assert _plan(256, GATE_UP, tokens_per_tile=64)["tokens_per_tile"] == 64
    p = _plan(256, GATE_UP, kernel=2)
    assert (p["path"], p["tokens_per_tile"]) == (2, 32)
    assert _plan(256, GATE_UP, num_ctas=7)["num_ctas"] == 7
    assert _plan(1, O, num_ctas=5000, kernel=2)["num_ctas"] == 32 * 32  # clamped to the k-stages


def _aligned(x, a=256):
    return (x + a - 1) // a * a


@pytest.mark.parametrize("M,NK", [(16, QKV), (64, QKV), (128, O), (256, GATE_UP), (32, DOWN)])
def test_workspace_layout(M, NK):
    """[256-byte status][CTA counters][CTAs x tile x 128 int32 slots][activation operand]."""
    N, K = NK
    p = _plan(M, NK)
    slots = 256 + _aligned(p["num_ctas"] * 4)
    act = 2 * M * K if p["path"] == 1 else 2 * M * K + (K // 128) * ((M + 3) // 4 * 4) * 4
    expect = _aligned(slots + p["num_ctas"] * p["tokens_per_tile"] * 128 * 4) + act
    assert p["workspace_bytes"] == expect


def test_argument_errors():
    lib = qoq.load()
    info = qoq.qoq_gemm_plan_info()
    byref = qoq.ctypes.byref
    assert lib.qoq_gemm_plan(16, 256, 512, 128, 0, None, byref(info)) == 1      # no SMs
    assert lib.qoq_gemm_plan(16, 256, 512, 128, SMS, None, None) == 1           # no output
    assert lib.qoq_gemm_plan(0, 256, 512, 128, SMS, None, byref(info)) == 1     # M = 0
    assert lib.qoq_gemm_plan(16, 200, 512, 128, SMS, None, byref(info)) == 2    # N % 128
    assert lib.qoq_gemm_plan(16, 256, 512, 64, SMS, None, byref(info)) == 2     # group
    opt = qoq.gemm_options(tokens_per_tile=48)
    assert lib.qoq_gemm_plan(16, 256, 512, 128, SMS, byref(opt), byref(info)) == 2


def test_allocation_free_limit_depends_on_the_shape():
    """The allocation-free entry point admits a shape when its scratch need
    (the planned workspace) is at most 8 MiB: every Llama-3-8B layer up to
    M = 64 (qkv and o also at 128), not Qwen1.5-72B down at M = 64."""
    limit = 8 << 20
    for M in (1, 8, 16, 32, 64):
        for NK in (QKV, O, GATE_UP, DOWN):
            assert _plan(M, NK)["workspace_bytes"] <= limit
    assert _plan(128, QKV)["workspace_bytes"] <= limit
    assert _plan(128, O)["workspace_bytes"] <= limit
    assert _plan(128, GATE_UP)["workspace_bytes"] > limit
    assert _plan(64, (8192, 29568))["workspace_bytes"] > limit


# ---------------------------------------------------------- dispatch table --
TABLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                     "w4a8_quantized_serving_qoq_gb300", "csrc", "qoq_dispatch_table.inc")


def _table():
    rows = []
    for line in open(TABLE):
        m = re.match(r"\{([-\d, ]+)\},", line.strip())
        if m:
            rows.append(tuple(int(v) for v in m.group(1).split(",")))
    return rows


def test_table_entries_are_what_an_automatic_plan_gets():
    """Every measured entry {N, K, group, M, num_sms, path, tokens, ctas} is
    the plan of that shape on a GPU with that SM count (cluster size for the
    CUDA-core path), and of every M down to the next smaller tuned M."""
    rows = _table()
    for N, K, group, M, sms, path, bt, ctas, sched in rows:
        p = qoq.qoq_gemm_plan(M, N, K, group, sms)
        assert p["path"] == path
        if path == 3:
            assert p["num_ctas"] == (N // 128) * ctas
        else:
            assert (p["tokens_per_tile"], p["num_ctas"]) == (bt, min(ctas, p["k_stages"]))
        below = [r[3] for r in rows if r[:3] == (N, K, group) and r[4] == sms and r[3] < M]
        lo = max(below) + 1 if below else 1
        assert qoq.qoq_gemm_plan(lo, N, K, group, sms)["path"] == (path if lo <= 8 or path != 3 else p["path"])


def test_table_applies_only_to_its_gpu_and_shapes():
    rows = _table()
    for N, K, group, M, sms, path, bt, ctas, sched in rows[:5]:
        other = qoq.qoq_gemm_plan(M, N, K, group, sms + 4)
        rules = qoq.qoq_gemm_plan(M, N, K, group, sms + 4, qoq.gemm_options(flags=qoq.QOQ_PLAN_RULES))
        assert other == rules
    # a shape nobody tuned plans by the rules
    p = qoq.qoq_gemm_plan(8, 1024, 1024, 128, 152)
    assert p == qoq.qoq_gemm_plan(8, 1024, 1024, 128, 152, qoq.gemm_options(flags=qoq.QOQ_PLAN_RULES))
    # beyond the largest tuned M of a shape: the rules
    big = max((r for r in rows if r[:3] == (4096, 4096, 128)), key=lambda r: r[3])
    p = qoq.qoq_gemm_plan(big[3] * 2, 4096, 4096, 128, big[4])
    assert p == qoq.qoq_gemm_plan(big[3] * 2, 4096, 4096, 128, big[4], qoq.gemm_options(flags=qoq.QOQ_PLAN_RULES))
