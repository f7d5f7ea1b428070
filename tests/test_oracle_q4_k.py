"""Pins of the oracle's Q4_K format ("One Native Stack ...", section "Ported
Versus Novel": every format is ggml's, verbatim; Q4_K is the 256-weight
super-block of 144 bytes with six-bit sub-block scales and mins).

What fixes each part: two hand-worked super-blocks (tests/golden), an
independent NumPy decode of the bit fields, a NumPy restatement of the encoder
(byte for byte), a round-trip bound derived from the encoder's arithmetic,
brute-force matvecs, and closed forms."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_k_blocks.json")


def _golden():
    with open(GOLDEN) as f:
        return {b["name"]: b for b in json.load(f)["blocks"]}


def _block_bytes(g):
    head = bytes.fromhex(g["header_hex"])
    rule = eval("lambda l: " + g["quant_byte_rule"])          # a fixed expression from the golden file
    qs = bytes(rule(l) for l in range(32)) * 4
    return np.frombuffer(head + qs, dtype=np.uint8).copy()


def test_hand_worked_decode():
    g = _golden()["q4_k_decode"]
    blk = _block_bytes(g)
    assert len(blk) == 144
    assert oracle.half_to_float(int(blk[0]) | (int(blk[1]) << 8)) == g["d"]
    assert oracle.half_to_float(int(blk[2]) | (int(blk[3]) << 8)) == g["dmin"]
    w = oracle.dequant("q4_k", blk, 1, 256)[0]
    for e, v in g["values"].items():
        assert w[int(e)] == v, e
    # every element by the rule the derivation states
    for e in range(256):
        j, l = divmod(e, 32)
        q = l % 16 if j % 2 == 0 else 15 - l % 16
        assert w[e] == g["d"] * g["sc"][j] * q - g["dmin"] * g["m"][j]
    y, T = oracle.matvec("q4_k", blk, np.ones((1, 256), np.float32), 1, 256)
    assert y[0, 0] == g["ones_dot"]
    assert T[0, 0] == np.abs(w).sum()
    # the NumPy field decode agrees on the same bytes
    d, dmin, sc, m, q = oracle_np.q4_k_fields(blk, 1, 256)
    assert list(sc[0, 0]) == g["sc"] and list(m[0, 0]) == g["m"]
    assert np.array_equal(oracle_np.dequant_q4_k(blk, 1, 256)[0], w)


def test_hand_worked_encode():
    g = _golden()["q4_k_encode_ramp"]
    W = np.tile(np.array([(l % 16) - 7.5 for l in range(32)], np.float32), 8).reshape(1, 256)
    got = oracle.quantize_q4_k(W)
    assert got.tobytes() == _block_bytes(g).tobytes()
    w = oracle.dequant("q4_k", got, 1, 256)[0]
    k = np.tile(np.arange(32) % 16, 8).astype(np.float64)
    assert np.array_equal(w, g["a"] * k - g["b"])


def _special_weights(rows, cols, seed):
    g = synthetic.rng(seed)
    W = synthetic.weights(g, rows, cols)
    W[::5] *= np.float32(40.0)                       # super-blocks of very different scales
    W[1::7, :32] = np.abs(W[1::7, :32]) + 0.01       # a sub-block without negative values (min -> 0)
    W[2::7, 32:64] = -np.abs(W[2::7, 32:64]) - 0.01  # all negative
    W[3::7, 64:96] = 0                               # all zero
    W[4::7, :] = 0                                   # whole super-block zero
    W[5::7, 100] = 3.0                               # one outlier: other sub-blocks get small 6-bit scales
    return W


def test_encoder_matches_numpy_restatement():
    for seed, (rows, cols) in enumerate([(64, 256), (40, 1024), (9, 4096)]):
        W = _special_weights(rows, cols, 300 + seed)
        assert np.array_equal(oracle.quantize_q4_k(W), oracle_np.quantize_q4_k(W))


def test_decode_matches_numpy_fields():
    for seed, (rows, cols) in enumerate([(64, 256), (40, 1024)]):
        W = _special_weights(rows, cols, 400 + seed)
        blk = oracle.quantize_q4_k(W)
        assert np.array_equal(oracle.dequant("q4_k", blk, rows, cols), oracle_np.dequant_q4_k(blk, rows, cols))
    # random bytes (any d, dmin, six-bit fields, nibbles) decode alike, except
    # where a random fp16 is not finite
    g = np.random.Generator(np.random.PCG64(7))
    raw = g.integers(0, 256, size=(50, 144 * 2), dtype=np.uint8)
    for h in (0, 2, 144, 146):
        raw[:, h + 1] &= 0x3B                             # keep the fp16 exponents finite
    assert np.array_equal(oracle.dequant("q4_k", raw, 50, 512), oracle_np.dequant_q4_k(raw, 50, 512))


def test_round_trip_bound():
    """For sub-block j with min mn = min(0, min w), s = (max w - mn)/15 (f64),
    and the stored a = d sc_j, b = dmin m_j: writing x = mn + t s (t in
    [0, 15]) and x' = (x + b)/a, the error is a |x' - q| <= a/2 when x' is in
    [-0.5, 15.5]; clamped at 15 it is at most 15 |s - a| + |b + mn|; clamped at
    0 at most |b + mn|.  So |w - w_deq| <= a/2 + 15 |s - a| + |b + mn| (plus a
    few fp32 ulps of the division, 1e-6 a)."""
    rows, cols = 2000, 512
    W = _special_weights(rows, cols, 500)
    blk = oracle.quantize_q4_k(W)
    Wd = oracle.dequant("q4_k", blk, rows, cols)
    d, dmin, sc, m, _ = oracle_np.q4_k_fields(blk, rows, cols)
    w = W.astype(np.float64).reshape(rows, cols // 256, 8, 32)
    mn = np.minimum(w.min(axis=3), 0.0)
    s = (w.max(axis=3) - mn) / 15.0
    a = d[..., None] * sc
    b = dmin[..., None] * m
    bound = a / 2 + 15 * np.abs(s - a) + np.abs(b + mn) + 1e-6 * a + 1e-12
    err = np.abs(w - Wd.reshape(w.shape)).max(axis=3)
    assert np.all(err <= bound)
    # and on ordinary N(0, 0.02) weights the 6-bit scales cost little: within 0.6 of a step
    W2 = synthetic.weights(synthetic.rng(501), 500, 1024)
    blk2 = oracle.quantize_q4_k(W2)
    d2, _, sc2, _, _ = oracle_np.q4_k_fields(blk2, 500, 1024)
    err2 = np.abs(W2.astype(np.float64) - oracle.dequant("q4_k", blk2, 500, 1024)).reshape(500, 4, 8, 32).max(axis=3)
    s2 = (W2.reshape(500, 4, 8, 32).max(axis=3) - np.minimum(W2.reshape(500, 4, 8, 32).min(axis=3), 0)) / 15.0
    assert np.all(err2 <= 0.6 * s2 + 1e-9)


@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 512), (5, 768)])
def test_brute_force_matvec(rows, cols):
    g = synthetic.rng(600 + rows)
    blk = oracle.quantize_q4_k(_special_weights(rows, cols, 600 + cols))
    for n_vec in range(1, 9):
        x = synthetic.activations(g, n_vec, cols)
        y, T = oracle.matvec("q4_k", blk, x, rows, cols)
        y2, T2 = oracle_np.matvec("q4_k", blk, x, rows, cols)
        assert np.allclose(y, y2, rtol=1e-12, atol=1e-12)
        assert np.allclose(T, T2, rtol=1e-12, atol=1e-12)
        lo, hi = (1, rows) if rows > 1 else (0, 1)
        yr, Tr = oracle.matvec_rows("q4_k", blk, x, rows, cols, lo, hi)
        assert np.array_equal(yr, y[:, lo:hi]) and np.array_equal(Tr, T[:, lo:hi])


def test_closed_forms():
    rows, cols = 6, 512
    blk = oracle.quantize_q4_k(_special_weights(rows, cols, 700))
    Wd = oracle.dequant("q4_k", blk, rows, cols)
    y, _ = oracle.matvec("q4_k", blk, np.ones((1, cols), np.float32), rows, cols)
    assert np.allclose(y[0], Wd.sum(axis=1), rtol=1e-13, atol=0)
    for j in (0, 31, 32, 255, 256, 300, 511):
        x = np.zeros((1, cols), np.float32)
        x[0, j] = 1.0
        assert np.array_equal(oracle.matvec("q4_k", blk, x, rows, cols)[0][0], Wd[:, j])
    z = oracle.quantize_q4_k(np.zeros((2, 256), np.float32))
    assert np.all(z == 0)
    assert np.all(oracle.matvec("q4_k", z, np.ones((3, 256), np.float32), 2, 256)[0] == 0)
