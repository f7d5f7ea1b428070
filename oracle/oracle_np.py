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


QK_K = 256


def q4_k_fields(blocks: np.ndarray, rows: int, cols: int):
    """(d, dmin, sc, m, q) of every Q4_K super-block, read with NumPy: d, dmin
    f64 [rows][nsb]; sc, m int [rows][nsb][8]; q int [rows][nsb][256].  The
    six-bit fields are gathered from their bit positions: sub-block j < 4 has
    sc = bits 0-5 of byte 4+j and m = bits 0-5 of byte 8+j; j >= 4 has the low
    four bits of sc / m in the low / high nibble of byte 8+j and the top two
    bits in bits 6-7 of byte j (sc) / byte 4+j (m), counting from byte 4."""
    nsb = cols // QK_K
    b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(rows, nsb, 144).astype(np.int64)
    d = b[:, :, 0:2].astype(np.uint8).copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[:, :, 2:4].astype(np.uint8).copy().view(np.float16)[..., 0].astype(np.float64)
    s12 = b[:, :, 4:16]
    sc = np.empty((rows, nsb, 8), np.int64)
    m = np.empty((rows, nsb, 8), np.int64)
    sc[..., :4] = s12[..., 0:4] % 64
    m[..., :4] = s12[..., 4:8] % 64
    sc[..., 4:] = (s12[..., 8:12] % 16) + 16 * (s12[..., 0:4] // 64)
    m[..., 4:] = (s12[..., 8:12] // 16) + 16 * (s12[..., 4:8] // 64)
    qs = b[:, :, 16:].reshape(rows, nsb, 4, 32)                 # 4 groups of 32 bytes
    lo, hi = qs % 16, qs // 16                                  # sub-blocks 2g and 2g+1
    q = np.stack([lo, hi], axis=3).reshape(rows, nsb, 256)      # [g][lo|hi][32] = element order
    return d, dmin, sc, m, q


def dequant_q4_k(blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    d, dmin, sc, m, q = q4_k_fields(blocks, rows, cols)
    nsb = cols // QK_K
    sub = np.repeat(np.arange(8), 32)                           # sub-block of each element
    a = d[:, :, None] * sc[:, :, sub]
    c = dmin[:, :, None] * m[:, :, sub]
    return (a * q - c).reshape(rows, nsb * QK_K)


def dequant(fmt: str, blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    return {"q8_0": dequant_q8_0, "q4_0": dequant_q4_0, "q4_k": dequant_q4_k}[fmt](blocks, rows, cols)


def matvec(fmt: str, blocks: np.ndarray, x: np.ndarray, rows: int, cols: int):
    """Brute force: (dequant(bytes) @ x^T)^T in f64, and T = |W| @ |x|."""
    Wd = dequant(fmt, blocks, rows, cols)
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


def quantize_q4_k(W: np.ndarray) -> np.ndarray:
    """The Q4_K min/max encoder restated with NumPy fp32 arrays: per sub-block
    scale = (max - min(0, min)) / 15 and min = -min(0, min); d, dmin = the
    largest of each / 63 stored fp16; 6-bit sc, m by rounding against the
    largest; q = round((w + dmin m) / (d sc)) clamped to [0, 15]."""
    W = np.asarray(W, dtype=np.float32)
    rows, cols = W.shape
    nsb = cols // QK_K
    w = W.reshape(rows, nsb, 8, 32)
    mn = np.minimum(w.min(axis=3), np.float32(0))
    mx = w.max(axis=3)
    scale = ((mx - mn) / np.float32(15)).astype(np.float32)
    minv = (-mn).astype(np.float32)
    ms = scale.max(axis=2)
    mm = minv.max(axis=2)
    # the largest scale and min, taken from +0 upwards (an all-zero super-block
    # has min -0: its stored dmin is +0, as the running maximum from 0 gives)
    ms = np.where(ms > 0, ms, np.float32(0)).astype(np.float32)
    mm = np.where(mm > 0, mm, np.float32(0)).astype(np.float32)
    dh = (ms / np.float32(63)).astype(np.float32).astype(np.float16)
    mh = (mm / np.float32(63)).astype(np.float32).astype(np.float16)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv_s = np.where(ms > 0, np.float32(63) / ms, np.float32(0)).astype(np.float32)
        inv_m = np.where(mm > 0, np.float32(63) / mm, np.float32(0)).astype(np.float32)

    def rnd(t):                                              # half away from zero
        return np.sign(t) * np.floor(np.abs(t) + np.float32(0.5))
    sc = np.clip(rnd((scale * inv_s[:, :, None]).astype(np.float32)), 0, 63).astype(np.int64)
    m = np.clip(rnd((minv * inv_m[:, :, None]).astype(np.float32)), 0, 63).astype(np.int64)
    a = (dh.astype(np.float32)[:, :, None] * sc.astype(np.float32)).astype(np.float32)
    b = (mh.astype(np.float32)[:, :, None] * m.astype(np.float32)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((w + b[..., None]).astype(np.float32) / a[..., None]).astype(np.float32)
    q = np.where(a[..., None] > 0, np.clip(rnd(t), 0, 15), 0).astype(np.int64)   # [rows][nsb][8][32]
    out = np.zeros((rows, nsb, 144), dtype=np.uint8)
    out[:, :, 0:2] = dh.view(np.uint8).reshape(rows, nsb, 2)
    out[:, :, 2:4] = mh.view(np.uint8).reshape(rows, nsb, 2)
    out[:, :, 4:8] = sc[..., :4] + 64 * (sc[..., 4:] // 16)
    out[:, :, 8:12] = m[..., :4] + 64 * (m[..., 4:] // 16)
    out[:, :, 12:16] = (sc[..., 4:] % 16) + 16 * (m[..., 4:] % 16)
    qg = q.reshape(rows, nsb, 4, 2, 32)
    out[:, :, 16:] = (qg[:, :, :, 0, :] + 16 * qg[:, :, :, 1, :]).reshape(rows, nsb, 128)
    return out.reshape(rows, nsb * 144)


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
