"""Independent NumPy / big-integer restatements used to pin the C oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Nothing here calls the
C oracle: block decoding goes through NumPy's own float16 type, the matvec is
``dequant(bytes) @ x`` in f64, and the gemmlowp rounding rules are restated as
exact rational arithmetic on Python integers.

Sources: "One Native Stack for Private, Continuously-Learning AI", section
"The Unified Quant Core" (Q8_0 34 B / 32, Q4_0 18 B / 32, ggml layouts), and
"Blue -- porting zen-nano (Qwen3-0.6B) to deterministic on-chain inference",
section "Quantization recipe (validated)" (per-channel int8, SRDHM then
RoundingDivideByPOT).
"""
from __future__ import annotations

import numpy as np

QK = 32


def _scales(blocks: np.ndarray, rows: int, nb: int, bpb: int) -> np.ndarray:
    b = blocks.reshape(rows, nb, bpb)
    return b[:, :, 0:2].copy().view(np.float16).reshape(rows, nb).astype(np.float64)


def dequant_q8_0(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    nb = cols // QK
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(rows, nb, 34)
    d = _scales(b, rows, nb, 34)
    q = b[:, :, 2:].view(np.int8).astype(np.float64)          # [rows][nb][32]
    return (q * d[:, :, None]).reshape(rows, cols)


def dequant_q4_0(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    nb = cols // QK
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(rows, nb, 18)
    d = _scales(b, rows, nb, 18)
    qs = b[:, :, 2:]
    lo = (qs & 0x0F).astype(np.float64) - 8.0                  # elements 0..15
    hi = (qs >> 4).astype(np.float64) - 8.0                    # elements 16..31
    q = np.concatenate([lo, hi], axis=2)
    return (q * d[:, :, None]).reshape(rows, cols)


def matvec(fmt: str, blocks: np.ndarray, x: np.ndarray, rows: int, cols: int):
    """Brute force: (dequant(bytes) @ x^T)^T in f64, and T = |W| @ |x|."""
    Wd = dequant_q8_0(blocks, rows, cols) if fmt == "q8_0" else dequant_q4_0(blocks, rows, cols)
    X = np.asarray(x, dtype=np.float32).reshape(-1, cols).astype(np.float64)
    y = X @ Wd.T
    T = np.abs(X) @ np.abs(Wd).T
    return y, T


def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns decoded from the IEEE fields (sign, 8-bit exponent with
    bias 127, 7-bit fraction), not by reinterpreting bits."""
    h = np.asarray(h, dtype=np.int64)
    s = np.where((h >> 15) & 1, -1.0, 1.0)
    e = (h >> 7) & 0xFF
    m = (h & 0x7F).astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        normal = s * np.ldexp(1.0 + m / 128.0, (e - 127).astype(np.int64))
        sub = s * np.ldexp(m / 128.0, -126)
        special = np.where(m == 0, s * np.inf, np.nan)
    return np.where(e == 0, sub, np.where(e == 255, special, normal))


def lora_delta(A: np.ndarray, B: np.ndarray, x: np.ndarray, scale: float):
    """scale * B (A x) and its magnitude, f64 matrix products of the decoded factors."""
    Af, Bf = bf16_to_f64(A), bf16_to_f64(B)
    X = np.asarray(x, dtype=np.float32).reshape(-1, Af.shape[1]).astype(np.float64)
    delta = scale * (X @ Af.T) @ Bf.T
    T = abs(scale) * (np.abs(X) @ np.abs(Af).T) @ np.abs(Bf).T
    return delta, T


# ----------------------------------------------------------- MoE epilogues

def silu_tanh(z):
    """silu through the identity sigmoid(z) = (1 + tanh(z/2)) / 2, a route that
    shares no step with the C oracle's z / (1 + e^-z)."""
    z = np.asarray(z, dtype=np.float64)
    return z * 0.5 * (1.0 + np.tanh(0.5 * z))


def moe_swiglu_q8_0(bank: np.ndarray, ids: np.ndarray, x: np.ndarray, n_experts: int,
                    rows: int, cols: int) -> np.ndarray:
    """SwiGLU of an interleaved gate/up bank by brute force: dequantize each
    chosen expert, split its rows into even (gate) and odd (up), multiply, gate.
    x: fp32 [n_vec][cols] shared by a token's slots.  Returns f64 [n_vec][n_active][rows/2]."""
    ids = np.asarray(ids)
    n_vec, n_active = ids.shape
    mat = rows * (cols // QK) * 34
    bank = np.ascontiguousarray(bank, dtype=np.uint8).reshape(-1)
    h = np.empty((n_vec, n_active, rows // 2))
    for t in range(n_vec):
        for k in range(n_active):
            e = int(ids[t, k])
            Wd = dequant_q8_0(bank[e * mat:(e + 1) * mat], rows, cols)
            xv = x[t].astype(np.float64)
            gate, up = Wd[0::2] @ xv, Wd[1::2] @ xv
            h[t, k] = silu_tanh(gate) * up
    return h


def moe_combine(y: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[t][i] = sum_k w[t][k] y[t][k][i] as one einsum."""
    return np.einsum("tk,tki->ti", np.asarray(w, dtype=np.float64), np.asarray(y, dtype=np.float64))


# ----------------------------------------------------------- independent quantizers
# A second, vectorised statement of the same readings (fp32 arithmetic), used
# to cross-check the C quantizers byte for byte.

def quantize_q8_0(W: np.ndarray) -> np.ndarray:
    W = np.asarray(W, dtype=np.float32)
    rows, cols = W.shape
    nb = cols // QK
    w = W.reshape(rows, nb, QK)
    amax = np.abs(w).max(axis=2)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(d[:, :, None] != 0, w / d[:, :, None], np.float32(0)).astype(np.float32)
    # round half away from zero
    q = np.sign(t) * np.floor(np.abs(t) + np.float32(0.5))
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty((rows, nb, 34), dtype=np.uint8)
    out[:, :, 0:2] = d.astype(np.float16).view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = q.view(np.uint8)
    return out.reshape(rows, nb * 34)


def quantize_q4_0(W: np.ndarray) -> np.ndarray:
    W = np.asarray(W, dtype=np.float32)
    rows, cols = W.shape
    nb = cols // QK
    w = W.reshape(rows, nb, QK)
    idx = np.abs(w).argmax(axis=2)                              # first index on ties
    m = np.take_along_axis(w, idx[:, :, None], axis=2)[:, :, 0]
    d = (m / np.float32(-8.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (w / d[:, :, None]).astype(np.float32) + np.float32(8.5)
    n = np.where(d[:, :, None] != 0, np.clip(np.floor(t), 0, 15), 8).astype(np.uint8)
    out = np.empty((rows, nb, 18), dtype=np.uint8)
    out[:, :, 0:2] = d.astype(np.float16).view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = n[:, :, :16] | (n[:, :, 16:] << 4)
    return out.reshape(rows, nb * 18)


# ----------------------------------------------------------- exact integer rules

INT32_MIN = -(2 ** 31)
INT32_MAX = 2 ** 31 - 1


def srdhm_exact(a: int, b: int) -> int:
    """floor(a*b / 2^31 + 1/2): the high word of 2ab rounded to nearest, ties up;
    the product INT32_MIN * INT32_MIN (the only one that overflows) saturates."""
    if a == INT32_MIN and b == INT32_MIN:
        return INT32_MAX
    return (a * b + 2 ** 30) // 2 ** 31


def rdivbypot_exact(x: int, e: int) -> int:
    """x / 2^e rounded to nearest, ties away from zero."""
    q, r = divmod(abs(x), 2 ** e)
    if 2 * r >= 2 ** e and e > 0:
        q += 1
    return q if x >= 0 else -q


def requant_exact(acc: int, mult: int, shift: int) -> int:
    v = rdivbypot_exact(srdhm_exact(acc, mult), shift)
    return max(-128, min(127, v))
