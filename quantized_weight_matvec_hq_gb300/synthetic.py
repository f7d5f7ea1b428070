"""Seeded synthetic inputs for the quantized-weight matvec.

This module only draws random numbers: it holds none of the method's
arithmetic (no quantization, no dequantization, no dot products), so that the
CPU oracle and the CUDA path can both be fed from it without sharing any step
of the computation.  It imports neither the oracle nor the CUDA library.

The recipe follows the workloads on the pages:

* weights W ~ N(0, 0.02) fp32, quantized afterwards by each side's own
  quantizer;
* activations x ~ N(0, 1) fp32, ``n_vec`` vectors of one length (n_vec 1..8:
  batch-1 decode up to the speculative-verify widths q in [1, 8] of
  "DeepSeek-V4 on Hanzo Engine", section "A Fused Attention Kernel for
  512-Wide Latent Heads");
* MoE routing: every token picks ``n_active`` distinct experts uniformly at
  random (a draw without replacement), slot order as drawn.

Generator: NumPy ``Generator(PCG64(seed))``.  The default seed of workload i is
``SEED_BASE + i``.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202

# Decode shapes (rows = output features, cols = input features).
QWEN3_0_6B_LAYER = (
    ("q", 2048, 1024), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 1024, 2048),
    ("gate", 3072, 1024), ("up", 3072, 1024), ("down", 1024, 3072),
)
QWEN3_0_6B_LAYERS = 28
QWEN3_0_6B_LM_HEAD = ("lm_head", 151936, 1024)

DENSE_8B_LAYER = (
    ("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
    ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336),
)
DENSE_8B_LAYERS = 32
DENSE_8B_LM_HEAD = ("lm_head", 128256, 4096)

MOE_N_EXPERTS = 128
MOE_N_ACTIVE = 8
MOE_HIDDEN = 2048
MOE_FFN = 768

INT8_SHAPES = ((1024, 3072), (3072, 1024))


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def weights(g: np.random.Generator, rows: int, cols: int, std: float = 0.02) -> np.ndarray:
    """fp32 [rows][cols] ~ N(0, std)."""
    return g.standard_normal((rows, cols), dtype=np.float32) * np.float32(std)


def activations(g: np.random.Generator, n_vec: int, cols: int) -> np.ndarray:
    """fp32 [n_vec][cols] ~ N(0, 1)."""
    return g.standard_normal((n_vec, cols), dtype=np.float32)


def sparse_outlier_weights(g: np.random.Generator, rows: int, cols: int, magnitude: float = 1.0):
    """fp32 [rows][cols] whose every 32-element block holds one element of
    +-magnitude (random sign per row) and 31 zeros, the non-zero element at
    the same position of the block in every row (a pruned input-channel
    pattern).  Returns (W, outlier_cols): the column of each block's
    non-zero element."""
    nb = cols // 32
    outlier_cols = np.arange(nb) * 32 + g.integers(0, 32, size=nb)
    W = np.zeros((rows, cols), dtype=np.float32)
    W[:, outlier_cols] = np.where(g.integers(0, 2, size=(rows, nb)) == 0, -1.0, 1.0).astype(np.float32) \
        * np.float32(magnitude)
    return W, outlier_cols


def expert_ids(g: np.random.Generator, n_vec: int, n_active: int, n_experts: int) -> np.ndarray:
    """int32 [n_vec][n_active]: distinct experts per token, uniformly at random."""
    out = np.empty((n_vec, n_active), dtype=np.int32)
    for t in range(n_vec):
        out[t] = g.permutation(n_experts)[:n_active]
    return out


def router_weights(g: np.random.Generator, n_vec: int, n_active: int) -> np.ndarray:
    """fp32 [n_vec][n_active]: positive weights summing to 1 per token, as a
    router hands its chosen experts (exponential draws, normalised)."""
    w = g.exponential(1.0, size=(n_vec, n_active))
    return (w / w.sum(axis=1, keepdims=True)).astype(np.float32)


def fuse_same_input(layer):
    """Row-concatenate the projections that read the same activation vector:
    q|k|v (the attention input) and gate|up (the MLP input).  The weight bytes
    are unchanged; a decode step then makes 4 matvec calls per layer, not 7."""
    by = dict((n, (r, c)) for n, r, c in layer)
    qkv = ("qkv", by["q"][0] + by["k"][0] + by["v"][0], by["q"][1])
    gate_up = ("gate_up", by["gate"][0] + by["up"][0], by["gate"][1])
    return (qkv, ("o",) + by["o"], gate_up, ("down",) + by["down"])


def decode_token_shapes(model: str, fused: bool = False):
    """The (name, rows, cols) list of one decode token's matvecs, lm_head last;
    with fused=True, q|k|v and gate|up are single row-concatenated matvecs."""
    if model == "qwen3-0.6b":
        layer, n, head = QWEN3_0_6B_LAYER, QWEN3_0_6B_LAYERS, QWEN3_0_6B_LM_HEAD
    elif model == "8b-dense":
        layer, n, head = DENSE_8B_LAYER, DENSE_8B_LAYERS, DENSE_8B_LM_HEAD
    else:
        raise ValueError(model)
    if fused:
        layer = fuse_same_input(layer)
    return [s for _ in range(n) for s in layer] + [head]
