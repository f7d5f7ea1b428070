"""Pins of the oracle's integer path: gemmlowp SaturatingRoundingDoublingHighMul
and RoundingDivideByPOT, the int8 GEMV and its requant
("Blue -- porting zen-nano (Qwen3-0.6B) to deterministic on-chain inference",
section "Quantization recipe (validated)").

The C scalar rules are checked against hand-worked values
(tests/golden/gemmlowp_worked.json) and against exact rational arithmetic on
Python integers over many random and extreme arguments.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic

I32_MIN, I32_MAX = -(2 ** 31), 2 ** 31 - 1


def _worked(golden_dir):
    with open(os.path.join(golden_dir, "gemmlowp_worked.json")) as f:
        return json.load(f)


def test_worked_values(golden_dir):
    w = _worked(golden_dir)
    for c in w["srdhm"]:
        assert oracle.srdhm(c["a"], c["b"]) == c["out"], c
        assert oracle_np.srdhm_exact(c["a"], c["b"]) == c["out"], c
    for c in w["rdivbypot"]:
        assert oracle.rdivbypot(c["x"], c["e"]) == c["out"], c
        assert oracle_np.rdivbypot_exact(c["x"], c["e"]) == c["out"], c
    for c in w["requant"]:
        assert oracle.requant(c["acc"], c["mult"], c["shift"]) == c["out"], c
    for c in w["requant_params"]:
        m, s = oracle.requant_params(np.array([c["M"]]))
        assert (int(m[0]), int(s[0])) == (c["mult"], c["shift"]), c


def _random_i32(g, n):
    a = g.integers(I32_MIN, I32_MAX, size=n, endpoint=True, dtype=np.int64)
    extremes = np.array([I32_MIN, I32_MIN + 1, -1, 0, 1, I32_MAX - 1, I32_MAX,
                         2 ** 30, -(2 ** 30), 2 ** 30 + 1, -(2 ** 30) - 1], dtype=np.int64)
    a[: extremes.size] = extremes
    small = g.integers(-5000, 5000, size=n // 4, dtype=np.int64)
    return np.concatenate([a, small])


def test_srdhm_and_rdivbypot_equal_exact_rationals():
    g = np.random.Generator(np.random.PCG64(11))
    a = _random_i32(g, 40000)
    b = _random_i32(g, 40000)[: a.size]
    g.shuffle(b)
    e = g.integers(0, 32, size=a.size)
    L = oracle.lib()
    for ai, bi, ei in zip(a.tolist(), b.tolist(), e.tolist()):
        v = L.hqo_srdhm(ai, bi)
        assert v == oracle_np.srdhm_exact(ai, bi)
        assert L.hqo_rdivbypot(ai, ei) == oracle_np.rdivbypot_exact(ai, ei)
    # every pair (a, INT32_MIN), (INT32_MIN, b) edge of the saturating case
    for bi in (I32_MIN, I32_MIN + 1, -1, 1, I32_MAX):
        assert L.hqo_srdhm(I32_MIN, bi) == oracle_np.srdhm_exact(I32_MIN, bi)


def test_requant_array_equals_exact():
    g = np.random.Generator(np.random.PCG64(12))
    acc = _random_i32(g, 20000).astype(np.int32)
    rows = 97
    mult = g.integers(2 ** 30, 2 ** 31 - 1, size=rows, dtype=np.int64).astype(np.int32)
    mult[:3] = [I32_MIN, I32_MAX, 1]
    shift = g.integers(0, 32, size=rows).astype(np.int32)
    y = oracle.requant_array(acc, mult, shift)
    ref = [oracle_np.requant_exact(int(a), int(mult[i % rows]), int(shift[i % rows]))
           for i, a in enumerate(acc.tolist())]
    assert np.array_equal(y, np.array(ref, dtype=np.int8))


@pytest.mark.parametrize("rows,cols", [(7, 12), (33, 100), (64, 3072)])
def test_int8_gemv_accumulator_and_requant(rows, cols):
    g = synthetic.rng(13 + rows)
    W = synthetic.weights(g, rows, cols)
    x = synthetic.activations(g, 3, cols)
    Wq, xq, mult, shift = oracle.int8_workload(W, x)
    y, acc = oracle.matvec_i8_requant(Wq, xq, mult, shift)
    acc_ref = xq.astype(np.int64) @ Wq.astype(np.int64).T
    assert np.array_equal(acc, acc_ref.astype(np.int32))
    ref = np.array([[oracle_np.requant_exact(int(acc_ref[v, o]), int(mult[o]), int(shift[o]))
                     for o in range(rows)] for v in range(3)], dtype=np.int8)
    assert np.array_equal(y, ref)


def test_int8_workload_recipe():
    """(mult, shift) encode M = s_w s_x / s_out to 2^-31 relative, and about 1 %
    of the outputs saturate (s_out is the 99th percentile of |y_float| / 127)."""
    g = synthetic.rng(14)
    rows, cols = 1024, 3072
    W = synthetic.weights(g, rows, cols)
    x = synthetic.activations(g, 1, cols)
    Wq, xq, mult, shift = oracle.int8_workload(W, x)
    assert np.all((mult >= 2 ** 30) & (shift >= 0) & (shift <= 31))
    y, acc = oracle.matvec_i8_requant(Wq, xq, mult, shift)
    sat = np.mean((y == 127) | (y == -128))
    assert 0.003 <= sat <= 0.03
    # the requantized int8 output tracks acc * M to within one unit (+ saturation)
    M = mult.astype(np.float64) * 2.0 ** -31 * 2.0 ** (-shift.astype(np.float64))
    approx = acc[0].astype(np.float64) * M
    ok = np.abs(approx) < 127
    assert np.all(np.abs(y[0][ok].astype(np.float64) - approx[ok]) <= 0.5 + 1e-6 * np.abs(approx[ok]) + 1e-9)


def test_requant_params_relative_accuracy():
    g = np.random.Generator(np.random.PCG64(15))
    M = np.exp(g.uniform(np.log(1e-9), np.log(0.999), size=5000))
    mult, shift = oracle.requant_params(M)
    back = mult.astype(np.float64) * 2.0 ** -31 * 2.0 ** (-shift.astype(np.float64))
    assert np.all(np.abs(back / M - 1) <= 2.0 ** -30)
    with pytest.raises(ValueError):
        oracle.requant_params(np.array([1.5]))
