"""Seeded synthetic inputs for the W4A8 GEMM workloads.

This module only draws random fp16 weights and activations with the shapes
and value distributions of the workloads; it holds none of the quantization
or GEMM arithmetic.  Both the CUDA path and the CPU oracle consume its output.

Distributions (stand-ins for Llama-3-8B / Qwen1.5-72B linear layers; no
dataset or trained weights are used):
  * W [N][K] fp16 ~ N(0, sigma_w^2) i.i.d. (sigma_w = 0.02 for the Llama
    shapes, 0.01 for the Qwen shapes); then ``w_outliers`` input-channel
    columns (2, or 8 for Qwen) drawn from the same stream are multiplied by 10.
  * X [M][K] fp16 ~ N(0, 1) i.i.d.; ``x_outliers`` input channels (4, or 16
    for Qwen) are multiplied by 20.
  * Generator: numpy PCG64 (``numpy.random.default_rng``).  Weights use seed
    ``2*s``, activations ``2*s + 1``, where ``s`` is the layer seed
    (0 for the tiny case, ``1000*workload_id + layer_index`` otherwise).
    The outlier columns are drawn before the values, and values fill rows in
    order, so the activations for M rows are the first M rows of any larger
    draw with the same seed.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Layer:
    name: str
    N: int
    K: int
    layer_index: int


# Llama-3-8B linear layers (d_model 4096, d_ff 14336, GQA 32/8 heads of 128).
LLAMA3_8B = (
    Layer("qkv", 6144, 4096, 0),
    Layer("o", 4096, 4096, 1),
    Layer("gate_up", 28672, 4096, 2),
    Layer("down", 4096, 14336, 3),
)
# Qwen1.5-72B-shaped FFN layers (d_model 8192, d_ff 29568).
QWEN_72B = (
    Layer("gate_up", 59136, 8192, 0),
    Layer("down", 8192, 29568, 1),
)

DECODE_MS = (1, 8, 32, 64, 128, 256)
PREFILL_M = 4096
QWEN_MS = (64, 1024)
CHANNEL_MS = tuple(2 ** i for i in range(13))

# workload id -> (description, layers, Ms, sigma_w, w_outliers, x_outliers, group)
WORKLOADS = {
    0: ("tiny 16x256x512 g128", (Layer("tiny", 256, 512, 0),), (16,), 0.02, 2, 4, 128),
    1: ("Llama-3-8B decode GEMMs g128", LLAMA3_8B, DECODE_MS, 0.02, 2, 4, 128),
    2: ("Llama-3-8B prefill GEMMs g128", LLAMA3_8B, (PREFILL_M,), 0.02, 2, 4, 128),
    3: ("Qwen1.5-72B-shaped FFN GEMMs g128", QWEN_72B, QWEN_MS, 0.01, 8, 16, 128),
    4: ("Llama-3-8B gate_up per-channel", (LLAMA3_8B[2],), CHANNEL_MS, 0.02, 2, 4, 0),
}


def layer_seed(workload_id: int, layer: Layer) -> int:
    return 0 if workload_id == 0 else 1000 * workload_id + layer.layer_index


def weights(N: int, K: int, seed: int, sigma: float = 0.02, outliers: int = 2,
            rows: int | None = None) -> np.ndarray:
    """fp16 [N][K] weights, seed stream 2*seed; with `rows`, only the first
    `rows` rows of that matrix (the values fill rows in order)."""
    rng = np.random.default_rng(2 * seed)
    cols = rng.choice(K, size=min(outliers, K), replace=False)
    W = rng.standard_normal((N if rows is None else min(rows, N), K), dtype=np.float32)
    W *= np.float32(sigma)
    W[:, cols] *= np.float32(10.0)
    return W.astype(np.float16)


def activations(M: int, K: int, seed: int, outliers: int = 4) -> np.ndarray:
    """fp16 [M][K] activations, seed stream 2*seed + 1."""
    rng = np.random.default_rng(2 * seed + 1)
    cols = rng.choice(K, size=min(outliers, K), replace=False)
    X = rng.standard_normal((M, K), dtype=np.float32)
    X[:, cols] *= np.float32(20.0)
    return X.astype(np.float16)


def workload_layer_inputs(workload_id: int, layer: Layer, M: int):
    """(W, X) for one layer of a workload at M tokens."""
    _, _, _, sigma, wo, xo, _ = WORKLOADS[workload_id]
    s = layer_seed(workload_id, layer)
    return weights(layer.N, layer.K, s, sigma, wo), activations(M, layer.K, s, xo)


def random_codes(N: int, K: int, seed: int, g: int = 128):
    """Uniformly random legal group codes (q4, s_g, z) for GEMM-only tests.

    Draws s_g in [1, 16] and z in [0, 15] per group, then each q4 uniformly
    among the codes within floor(127 / s_g) of z (so every reconstructed
    weight lies in [-127, 127]).  No quantizer arithmetic is involved.
    """
    rng = np.random.default_rng(seed)
    G = K // g
    s_g = rng.integers(1, 17, size=(N, G), dtype=np.int64)
    z = rng.integers(0, 16, size=(N, G), dtype=np.int64)
    reach = 127 // s_g
    lo = np.repeat(np.maximum(0, z - reach), g, axis=1)
    hi = np.repeat(np.minimum(15, z + reach), g, axis=1)
    q4 = lo + np.floor(rng.random((N, K)) * (hi - lo + 1)).astype(np.int64)
    return q4.astype(np.uint8), s_g.astype(np.uint8), z.astype(np.uint8)
