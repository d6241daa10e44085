"""Roofline arithmetic for the W4A8 GEMM (host-side helpers for the benchmark).

Algorithmic traffic of one GEMM (4-bit weights plus 8-bit activations):
    B = N*K/2 + M*K bytes,
and its work is 2*M*N*K operations.  The roofline time is the slower of the
memory bound and the compute bound:
    T = max(B / BW, 2*M*N*K / P).
The QServe pages motivate W4A8 with the A100 roofline (FP16 / INT8 tensor
peaks of 312 / 624 TOPS and 2 TB/s): for m << n, k the GEMM intensity is
about m MACs per weight element, W4A16 wins below m = 78 and W8A8 above it
("QServe：把 W4A8KV4 的理论收益做成实测吞吐的量化—系统协同设计", section 2
"roofline 解释"; "QServe: W4A8KV4 Quantization and System Co-design for
Efficient LLM Serving", section "为什么选择W4A8KV4").
"""
from __future__ import annotations


def w4a8_bytes(M: int, N: int, K: int) -> int:
    """4-bit weight plus 8-bit activation bytes."""
    return N * K // 2 + M * K


def w4a8_bytes_full(M: int, N: int, K: int, group: int = 128) -> int:
    """The stricter traffic: B plus the group metadata (the UINT8 scale and
    the zero, one byte each, per 128 weights; per-channel: one zero byte per
    row), s_w, s_x and the fp16 output."""
    meta = (N * (K // group) * 2) if group else N
    return w4a8_bytes(M, N, K) + meta + 2 * N + 2 * M + 2 * M * N


def gemm_ops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def roof_time(M: int, N: int, K: int, bw_bytes_per_s: float, peak_ops_per_s: float) -> float:
    return max(w4a8_bytes(M, N, K) / bw_bytes_per_s, gemm_ops(M, N, K) / peak_ops_per_s)


def bound(M: int, N: int, K: int, bw_bytes_per_s: float, peak_ops_per_s: float) -> str:
    t_mem = w4a8_bytes(M, N, K) / bw_bytes_per_s
    t_cmp = gemm_ops(M, N, K) / peak_ops_per_s
    return "hbm" if t_mem >= t_cmp else "tensor"


def attainable_macs(m: float, weight_bytes: float, bw: float, peak_macs: float) -> float:
    """MAC/s of an m-token GEMM whose traffic is dominated by weights of
    `weight_bytes` per element, capped by the tensor peak (in MAC/s)."""
    return min(m * bw / weight_bytes, peak_macs)


def w4a16_w8a8_crossover(bw: float, fp16_tops: float, int8_tops: float) -> float:
    """Smallest m at which W8A8 (1 B/weight, INT8 peak) is at least as fast as
    W4A16 (0.5 B/weight, FP16 peak); found by bisection on the two rooflines."""
    def w4a16(m):
        return attainable_macs(m, 0.5, bw, fp16_tops / 2)

    def w8a8(m):
        return attainable_macs(m, 1.0, bw, int8_tops / 2)

    lo, hi = 1.0, 1e6
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if w8a8(mid) >= w4a16(mid):
            hi = mid
        else:
            lo = mid
    return hi


def ridge_m(bw: float, peak_ops: float) -> float:
    """Token count where the W4A8 GEMM turns compute-bound: 2MNK / (NK/2) = 4M ops/byte."""
    return peak_ops / (4.0 * bw)
