"""The CPU oracle for the quantized-weight matvec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library
(``quantized_weight_matvec_hq_gb300``) never imports, links or runs it, and
this package imports nothing from the product.

Two independent implementations live here:

* ``hq_oracle.c`` (loaded below through ctypes): the plain scalar C oracle,
  f64 accumulation, one function per step of the method.
* ``oracle_np.py``: a NumPy f64 brute force over ``dequant(bytes) @ x`` and
  big-integer restatements of the gemmlowp rounding rules, used to pin the C
  oracle on small inputs.

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against hand-worked blocks, closed forms, round-trip bounds, brute force and
exact rational arithmetic; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_p = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """Build (if stale) and load liboracle.so."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.hqo_half_to_float.argtypes = [ctypes.c_uint16]
        L.hqo_half_to_float.restype = ctypes.c_float
        L.hqo_float_to_half_rne.argtypes = [ctypes.c_float]
        L.hqo_float_to_half_rne.restype = ctypes.c_uint16
        for name in ("hqo_quantize_q8_0", "hqo_quantize_q4_0", "hqo_quantize_q4_k"):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = None
        L.hqo_quantize_i8_rows.argtypes = [_p, _i64, _i64, _p, _p]
        L.hqo_quantize_i8_rows.restype = None
        for name in ("hqo_dequant_q8_0", "hqo_dequant_q4_0", "hqo_dequant_q4_k"):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = None
        for name in ("hqo_matvec_q8_0", "hqo_matvec_q4_0", "hqo_matvec_q4_k"):
            getattr(L, name).argtypes = [_p, _p, _i64, _i64, _int, _p, _p]
            getattr(L, name).restype = None
        L.hqo_matvec_rows.argtypes = [_int, _p, _p, _i64, _i64, _i64, _i64, _int, _p, _p]
        L.hqo_matvec_rows.restype = None
        L.hqo_moe_matvec_q8_0.argtypes = [_p, _p, _p, _int, _i64, _int, _i64, _i64, _int, _p, _p]
        L.hqo_moe_matvec_q8_0.restype = _int
        L.hqo_srdhm.argtypes = [ctypes.c_int32, ctypes.c_int32]
        L.hqo_srdhm.restype = ctypes.c_int32
        L.hqo_rdivbypot.argtypes = [ctypes.c_int32, _int]
        L.hqo_rdivbypot.restype = ctypes.c_int32
        L.hqo_requant.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
        L.hqo_requant.restype = ctypes.c_int8
        L.hqo_matvec_i8_requant.argtypes = [_p, _p, _p, _p, _i64, _i64, _int, _p, _p]
        L.hqo_matvec_i8_requant.restype = _int
        L.hqo_requant_array.argtypes = [_p, _p, _p, _i64, _i64, _p]
        L.hqo_requant_array.restype = None
        L.hqo_requant_params.argtypes = [_p, _i64, _p, _p]
        L.hqo_requant_params.restype = _int
        L.hqo_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.hqo_bf16_to_float.restype = ctypes.c_float
        L.hqo_lora_delta.argtypes = [_p, _p, _p, ctypes.c_double, _i64, _i64, _i64, _i64, _p, _p]
        L.hqo_silu.argtypes = [ctypes.c_double]
        L.hqo_silu.restype = ctypes.c_double
        L.hqo_swiglu_pairs.argtypes = [_p, _i64, _p]
        L.hqo_moe_combine.argtypes = [_p, _p, _p, _int, _int, _i64, _p, _p]
        L.hqo_lora_delta.restype = ctypes.c_int
        L.hqo_version.restype = _int
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- half floats

def half_to_float(h: int) -> float:
    return float(lib().hqo_half_to_float(int(h) & 0xFFFF))


def float_to_half(f: float) -> int:
    return int(lib().hqo_float_to_half_rne(float(np.float32(f))))


# ---------------------------------------------------------------- quantizers

Q8_0_BYTES = 34
Q4_0_BYTES = 18
Q4_K_BYTES = 144
QK = 32
QK_K = 256
# format name -> (weights per block, bytes per block, code of the C matvec_rows)
FORMATS = {"q8_0": (QK, Q8_0_BYTES, 8), "q4_0": (QK, Q4_0_BYTES, 4), "q4_k": (QK_K, Q4_K_BYTES, ord("K"))}


def row_bytes(fmt: str, cols: int) -> int:
    qk, bb, _ = FORMATS[fmt]
    return cols // qk * bb


def quantize_q8_0(W: np.ndarray) -> np.ndarray:
    """fp32 [rows][cols] -> uint8 [rows][cols/32*34] (ggml Q8_0 blocks)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    assert cols % QK == 0
    out = np.empty((rows, cols // QK * Q8_0_BYTES), dtype=np.uint8)
    lib().hqo_quantize_q8_0(_ptr(W), rows, cols, _ptr(out))
    return out


def quantize_q4_0(W: np.ndarray) -> np.ndarray:
    """fp32 [rows][cols] -> uint8 [rows][cols/32*18] (ggml Q4_0 blocks)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    assert cols % QK == 0
    out = np.empty((rows, cols // QK * Q4_0_BYTES), dtype=np.uint8)
    lib().hqo_quantize_q4_0(_ptr(W), rows, cols, _ptr(out))
    return out


def quantize_q4_k(W: np.ndarray) -> np.ndarray:
    """fp32 [rows][cols] -> uint8 [rows][cols/256*144] (ggml Q4_K super-blocks,
    encoded by the oracle's min/max reading; cols % 256 == 0)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    assert cols % QK_K == 0
    out = np.empty((rows, cols // QK_K * Q4_K_BYTES), dtype=np.uint8)
    lib().hqo_quantize_q4_k(_ptr(W), rows, cols, _ptr(out))
    return out


def quantize(fmt: str, W: np.ndarray) -> np.ndarray:
    return {"q8_0": quantize_q8_0, "q4_0": quantize_q4_0, "q4_k": quantize_q4_k}[fmt](W)


def quantize_i8_rows(W: np.ndarray):
    """fp32 [rows][cols] -> (int8 [rows][cols], fp32 scale [rows])."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    q = np.empty((rows, cols), dtype=np.int8)
    s = np.empty(rows, dtype=np.float32)
    lib().hqo_quantize_i8_rows(_ptr(W), rows, cols, _ptr(q), _ptr(s))
    return q, s


def dequant(fmt: str, blocks: np.ndarray, rows: int, cols: int) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty((rows, cols), dtype=np.float64)
    fn = {"q8_0": lib().hqo_dequant_q8_0, "q4_0": lib().hqo_dequant_q4_0, "q4_k": lib().hqo_dequant_q4_k}[fmt]
    fn(_ptr(blocks), rows, cols, _ptr(out))
    return out


# ---------------------------------------------------------------- matvecs

def matvec(fmt: str, blocks: np.ndarray, x: np.ndarray, rows: int, cols: int):
    """Return (y, T), both f64 [n_vec][rows]; x is fp32 [n_vec][cols]."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
    n_vec = x.shape[0]
    y = np.empty((n_vec, rows), dtype=np.float64)
    T = np.empty((n_vec, rows), dtype=np.float64)
    fn = {"q8_0": lib().hqo_matvec_q8_0, "q4_0": lib().hqo_matvec_q4_0, "q4_k": lib().hqo_matvec_q4_k}[fmt]
    fn(_ptr(blocks), _ptr(x), rows, cols, n_vec, _ptr(y), _ptr(T))
    return y, T


def matvec_rows(fmt: str, blocks: np.ndarray, x: np.ndarray, rows: int, cols: int,
                row_lo: int, row_hi: int):
    """Rows [row_lo, row_hi) of (y, T) only -- for sampled checks at full size."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
    n_vec = x.shape[0]
    y = np.zeros((n_vec, rows), dtype=np.float64)
    T = np.zeros((n_vec, rows), dtype=np.float64)
    lib().hqo_matvec_rows(FORMATS[fmt][2], _ptr(blocks), _ptr(x), row_lo,
                          row_hi, rows, cols, n_vec, _ptr(y), _ptr(T))
    return y[:, row_lo:row_hi], T[:, row_lo:row_hi]


def moe_matvec_q8_0(bank: np.ndarray, ids: np.ndarray, x: np.ndarray, x_per_slot: bool,
                    n_experts: int, n_active: int, rows: int, cols: int, n_vec: int):
    """Return (y, T), f64 [n_vec][n_active][rows]."""
    bank = np.ascontiguousarray(bank, dtype=np.uint8)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty((n_vec, n_active, rows), dtype=np.float64)
    T = np.empty((n_vec, n_active, rows), dtype=np.float64)
    rc = lib().hqo_moe_matvec_q8_0(_ptr(bank), _ptr(ids), _ptr(x), int(bool(x_per_slot)),
                                   n_experts, n_active, rows, cols, n_vec, _ptr(y), _ptr(T))
    if rc != 0:
        raise ValueError("expert id out of range")
    return y, T


# ---------------------------------------------------------------- integer path

def srdhm(a: int, b: int) -> int:
    return int(lib().hqo_srdhm(int(a), int(b)))


def rdivbypot(x: int, e: int) -> int:
    return int(lib().hqo_rdivbypot(int(x), int(e)))


def requant(acc: int, mult: int, shift: int) -> int:
    return int(lib().hqo_requant(int(acc), int(mult), int(shift)))


def requant_array(acc: np.ndarray, mult: np.ndarray, shift: np.ndarray) -> np.ndarray:
    """Element i uses (mult, shift)[i % len(mult)]."""
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    mult = np.ascontiguousarray(mult, dtype=np.int32)
    shift = np.ascontiguousarray(shift, dtype=np.int32)
    y = np.empty(acc.shape, dtype=np.int8)
    lib().hqo_requant_array(_ptr(acc), _ptr(mult), _ptr(shift), acc.size, mult.size, _ptr(y))
    return y


def matvec_i8_requant(Wq: np.ndarray, xq: np.ndarray, mult: np.ndarray, shift: np.ndarray):
    """Return (y int8 [n_vec][rows], acc int32 [n_vec][rows])."""
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    rows, cols = Wq.shape
    xq = np.ascontiguousarray(xq, dtype=np.int8).reshape(-1, cols)
    n_vec = xq.shape[0]
    mult = np.ascontiguousarray(mult, dtype=np.int32)
    shift = np.ascontiguousarray(shift, dtype=np.int32)
    y = np.empty((n_vec, rows), dtype=np.int8)
    acc = np.empty((n_vec, rows), dtype=np.int32)
    rc = lib().hqo_matvec_i8_requant(_ptr(Wq), _ptr(xq), _ptr(mult), _ptr(shift), rows, cols,
                                     n_vec, _ptr(y), _ptr(acc))
    if rc != 0:
        raise OverflowError("int32 accumulator overflow")
    return y, acc


def requant_params(M: np.ndarray):
    """Real multipliers in (0,1) -> (mult int32, shift int32)."""
    M = np.ascontiguousarray(M, dtype=np.float64)
    mult = np.empty(M.shape, dtype=np.int32)
    shift = np.empty(M.shape, dtype=np.int32)
    if lib().hqo_requant_params(_ptr(M), M.size, _ptr(mult), _ptr(shift)) != 0:
        raise ValueError("multiplier outside (0,1) or shift beyond 31")
    return mult, shift


def int8_workload(W: np.ndarray, x: np.ndarray, out_quantile: float = 0.99):
    """The int8 input recipe, computed by the oracle: per-row int8 weights,
    per-tensor int8 activations, and per-row (mult, shift) from
    M[o] = s_w[o] * s_x / s_out with s_out = quantile(|y_float|)/127, so that
    about 1 % of outputs saturate.  Returns (Wq, xq, mult, shift)."""
    Wq, s_w = quantize_i8_rows(W)
    x = np.ascontiguousarray(x, dtype=np.float32)
    xq_rows, s_x_rows = quantize_i8_rows(x.reshape(1, -1))
    s_x = float(s_x_rows[0])
    xq = xq_rows.reshape(x.shape)
    acc = xq.astype(np.int64) @ Wq.astype(np.int64).T            # [n_vec][rows]
    y_float = acc.astype(np.float64) * s_w.astype(np.float64)[None, :] * s_x
    s_out = float(np.quantile(np.abs(y_float), out_quantile)) / 127.0
    M = s_w.astype(np.float64) * s_x / s_out
    mult, shift = requant_params(M)
    return Wq, xq, mult, shift


# ---------------------------------------------------------------- QLoRA adapter term

def bf16_to_float(h: int) -> float:
    return float(lib().hqo_bf16_to_float(int(h)))


def lora_delta(A: np.ndarray, B: np.ndarray, x: np.ndarray, scale: float):
    """The QLoRA adapter term scale * B (A x) in f64 and its magnitude T.
    A: bf16 bits uint16 [rank][cols]; B: bf16 bits uint16 [rows][rank];
    x: fp32 [n_vec][cols].  Returns (delta, T), f64 [n_vec][rows]."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    rank, cols = A.shape
    rows = B.shape[0]
    assert B.shape[1] == rank
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, cols)
    n_vec = x.shape[0]
    delta = np.empty((n_vec, rows), dtype=np.float64)
    T = np.empty((n_vec, rows), dtype=np.float64)
    rc = lib().hqo_lora_delta(_ptr(A), _ptr(B), _ptr(x), float(scale), rank, rows, cols, n_vec, _ptr(delta),
                              _ptr(T))
    if rc != 0:
        raise ValueError(f"hqo_lora_delta failed (rank {rank})")
    return delta, T


# ---------------------------------------------------------------- MoE epilogues

def silu(z: float) -> float:
    return float(lib().hqo_silu(float(z)))


def swiglu_pairs(y: np.ndarray) -> np.ndarray:
    """h[..., i] = silu(y[..., 2i]) * y[..., 2i+1] in f64 (interleaved gate/up rows)."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    assert y.shape[-1] % 2 == 0
    h = np.empty(y.shape[:-1] + (y.shape[-1] // 2,), dtype=np.float64)
    lib().hqo_swiglu_pairs(_ptr(y), h.size, _ptr(h))
    return h


def moe_combine(y: np.ndarray, T, w: np.ndarray):
    """Router-weighted sum over the slots: y, T f64 [n_vec][n_active][rows],
    w fp32 [n_vec][n_active].  Returns (out, Tout), f64 [n_vec][rows]."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    n_vec, n_active, rows = y.shape
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(n_vec, n_active)
    Tp = None
    if T is not None:
        T = np.ascontiguousarray(T, dtype=np.float64)
        Tp = _ptr(T)
    out = np.empty((n_vec, rows), dtype=np.float64)
    Tout = np.empty((n_vec, rows), dtype=np.float64)
    lib().hqo_moe_combine(_ptr(y), Tp, _ptr(w), n_vec, n_active, rows, _ptr(out), _ptr(Tout))
    return out, Tout


def version() -> int:
    return int(lib().hqo_version())
