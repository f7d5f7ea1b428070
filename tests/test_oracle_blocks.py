"""Pins of the oracle's half-float conversion and block quantizers.

Each pin checks the C oracle against something other than itself: NumPy's
own float16 conversion, hand-worked blocks (tests/golden/blocks.json),
round-trip error bounds that follow from the block definitions, and an
independently written vectorised quantizer.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic


def test_half_to_float_matches_numpy_for_all_65536_patterns():
    L = oracle.lib()
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([L.hqo_half_to_float(int(b)) for b in bits], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_float_to_half_rne_matches_numpy():
    L = oracle.lib()
    g = np.random.Generator(np.random.PCG64(1))
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(0.02),
        (g.standard_normal(5000) * 1e4).astype(np.float32),
        (g.standard_normal(5000) * 1e-5).astype(np.float32),          # subnormal halves
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24,
                  2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11),
                  5.9604645e-08, 6.1035156e-05, 0.1, 0.01, 1.0 / 3.0], dtype=np.float32),
    ])
    # every halfway point between consecutive finite halves (exercises ties-to-even)
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    mids = mids[mids.astype(np.float64) == (lo + hi) / 2]               # exact in fp32
    vals = np.concatenate([vals, mids, -mids])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([L.hqo_float_to_half_rne(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "blocks.json")) as f:
        return {b["name"]: b for b in json.load(f)["blocks"]}


def _weights(name):
    w = np.zeros(32, dtype=np.float32)
    if name == "q8_0_ramp":
        w[0] = np.float32(-1.27)
        for j in range(1, 32):
            w[j] = np.float32((j - 16) * 0.01)
    elif name == "q4_0_negative_absmax":
        w[0] = np.float32(-0.8)
        for j in range(1, 32):
            w[j] = np.float32(((j % 15) - 7) * 0.1)
    elif name == "q4_0_opposite_sign_clamp":
        w[0] = np.float32(0.8)
        w[5] = np.float32(-0.8)
    elif name == "q8_0_rounding":
        w[:6] = np.array([1.27, 0.026, -0.026, 0.024, -0.024, 0.0149], dtype=np.float32)
    elif name == "q4_0_rounding":
        w[:5] = np.array([-0.8, 0.26, -0.26, 0.24, -0.24], dtype=np.float32)
    return w.reshape(1, 32)


@pytest.mark.parametrize("name", ["q8_0_ramp", "q4_0_negative_absmax", "q4_0_opposite_sign_clamp",
                                  "q8_0_zero", "q4_0_zero", "q8_0_rounding", "q4_0_rounding"])
def test_hand_worked_blocks(golden_dir, name):
    g = _golden(golden_dir)[name]
    w = _weights(name)
    quant = oracle.quantize_q8_0 if g["format"] == "q8_0" else oracle.quantize_q4_0
    got = quant(w).tobytes()
    assert got == bytes.fromhex(g["bytes_hex"])
    # the stored scale decodes to the hand-worked value (sign of zero included)
    d = oracle.half_to_float(got[0] | (got[1] << 8))
    assert d == g["scale"] and np.signbit(d) == np.signbit(g["scale"])
    # dequantization of the hand-worked bytes
    wd = oracle.dequant(g["format"], np.frombuffer(got, dtype=np.uint8), 1, 32)
    if name == "q8_0_ramp":
        q = np.array([-127] + [j - 16 for j in range(1, 32)], dtype=np.float64)
        assert np.array_equal(wd[0], q * g["scale"])
        y, _ = oracle.matvec("q8_0", np.frombuffer(got, dtype=np.uint8), np.ones((1, 32), np.float32), 1, 32)
        assert y[0, 0] == g["ones_dot"]
    if name == "q4_0_opposite_sign_clamp":
        assert wd[0, 5] == g["w_deq_5"]
        assert wd[0, 0] == -8 * g["scale"]
    if name.endswith("zero"):
        assert np.all(wd == 0)


def _rand_blocks(n, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    W = synthetic.weights(g, n, 32)
    # heavier tails and outlier blocks, so clamps and small scales occur
    W[::7] *= np.float32(50.0)
    W[1::11, 3] = np.float32(0.5)
    return W


def test_q8_0_round_trip_bound():
    """|w - w_deq| <= |d|/2 + 127*|d - fp16(d)| (q = round(w/d), |q| <= 127)."""
    W = _rand_blocks(100000 // 32 * 32, 2).reshape(-1, 32)
    blocks = oracle.quantize_q8_0(W)
    wd = oracle.dequant("q8_0", blocks, W.shape[0], 32)
    d = (np.abs(W).max(axis=1) / np.float32(127)).astype(np.float32).astype(np.float64)
    dh = blocks[:, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
    bound = np.abs(d) / 2 * (1 + 1e-6) + 127 * np.abs(d - dh)
    err = np.abs(W.astype(np.float64) - wd).max(axis=1)
    assert np.all(err <= bound)
    # fp16 rounding moves d by at most 2^-11 relative, so the bound is <= (1/2 + 127/2048)|d|
    assert np.all(bound <= (0.5 + 127 / 2048) * np.abs(d) * (1 + 1e-6) + 1e-30)


def test_q4_0_round_trip_bound():
    """Unclamped elements: |w - w_deq| <= |d|/2 + 8|d - fp16(d)|; the one element
    that can clamp (+|m| when d<0 maps to n=16) has error <= |d|(1 + 2^-8)."""
    W = _rand_blocks(100000 // 32 * 32, 3).reshape(-1, 32)
    blocks = oracle.quantize_q4_0(W)
    wd = oracle.dequant("q4_0", blocks, W.shape[0], 32)
    idx = np.abs(W).argmax(axis=1)
    m = W[np.arange(W.shape[0]), idx]
    d = (m / np.float32(-8)).astype(np.float32).astype(np.float64)
    dh = blocks[:, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
    err = np.abs(W.astype(np.float64) - wd)
    t = W.astype(np.float64) / d[:, None] + 8.5
    clamped = t >= 16
    unclamped_bound = np.abs(d)[:, None] / 2 * (1 + 1e-6) + 8 * np.abs(d - dh)[:, None]
    assert np.all(err[~clamped] <= np.broadcast_to(unclamped_bound, err.shape)[~clamped])
    clamp_bound = np.abs(d)[:, None] * (1 + 2.0 ** -8)
    assert np.all(err[clamped] <= np.broadcast_to(clamp_bound, err.shape)[clamped])
    # the absmax element itself is reproduced to within the fp16 rounding of d
    assert np.all(np.abs(wd[np.arange(W.shape[0]), idx] - m) <= 8 * np.abs(d - dh) + 1e-12)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_quantizers_match_independent_numpy(fmt):
    g = synthetic.rng(5)
    W = synthetic.weights(g, 37, 32 * 9)
    W[3, :32] = 0
    W[5, 40] = np.float32(-1.0)
    got = (oracle.quantize_q8_0 if fmt == "q8_0" else oracle.quantize_q4_0)(W)
    ref = (oracle_np.quantize_q8_0 if fmt == "q8_0" else oracle_np.quantize_q4_0)(W)
    assert np.array_equal(got, ref)


def test_int8_row_quantizer():
    g = synthetic.rng(6)
    W = synthetic.weights(g, 40, 96)
    W[7] = 0
    q, s = oracle.quantize_i8_rows(W)
    assert np.all(s[7] == 0) and np.all(q[7] == 0)
    amax = np.abs(W).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(127)).astype(np.float32))
    # the absmax element of every row maps to +-127 and |q| never exceeds 127
    rows = np.arange(40)[amax > 0]
    j = np.abs(W).argmax(axis=1)[rows]
    assert np.all(np.abs(q[rows, j].astype(int)) == 127)
    assert np.abs(q.astype(int)).max() <= 127
    # round-trip: |w - q*s| <= s/2 (+ fp32 slack)
    err = np.abs(W.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-6))
