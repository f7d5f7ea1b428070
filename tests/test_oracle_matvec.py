"""Pins of the oracle's float matvecs and MoE variant.

y = W_deq . x over the stored bytes ("One Native Stack for Private,
Continuously-Learning AI", section "The Central Efficiency Thesis", Lemma on
QLoRA over the unified core: y_i = sum_j What_ij x_j with What = DEQ_cpu(W)).
The C oracle is checked against an independent NumPy f64 brute force on tiny
shapes, against closed forms, and the MoE variant against a loop of
single-expert matvecs.
"""
import numpy as np
import pytest

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic


def _quant(fmt, W):
    return oracle.quantize_q8_0(W) if fmt == "q8_0" else oracle.quantize_q4_0(W)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows", [1, 2, 5])
@pytest.mark.parametrize("cols", [32, 64, 96])
def test_brute_force_tiny(fmt, rows, cols):
    g = synthetic.rng(100 + rows * 7 + cols)
    W = synthetic.weights(g, rows, cols)
    blocks = _quant(fmt, W)
    for n_vec in range(1, 9):
        x = synthetic.activations(g, n_vec, cols)
        y, T = oracle.matvec(fmt, blocks, x, rows, cols)
        y_ref, T_ref = oracle_np.matvec(fmt, blocks, x, rows, cols)
        assert np.allclose(y, y_ref, rtol=1e-12, atol=1e-12 * T_ref.max())
        assert np.allclose(T, T_ref, rtol=1e-12, atol=0)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_closed_forms(fmt):
    rows, cols = 9, 32 * 6
    g = synthetic.rng(7)
    W = synthetic.weights(g, rows, cols)
    W[4] = 0                                    # an all-zero row of blocks
    blocks = _quant(fmt, W)
    Wd = oracle_np.dequant_q8_0(blocks, rows, cols) if fmt == "q8_0" else oracle_np.dequant_q4_0(blocks, rows, cols)
    # all-ones x gives the row sums of the dequantized matrix
    y, _ = oracle.matvec(fmt, blocks, np.ones((1, cols), np.float32), rows, cols)
    assert np.allclose(y[0], Wd.sum(axis=1), rtol=1e-13, atol=1e-15)
    # a one-hot x picks out one column, exactly
    for j in (0, 31, 32, 100, cols - 1):
        e = np.zeros((1, cols), np.float32)
        e[0, j] = 1
        y, T = oracle.matvec(fmt, blocks, e, rows, cols)
        assert np.array_equal(y[0], Wd[:, j])
        assert np.array_equal(T[0], np.abs(Wd[:, j]))
    # all-zero blocks give exactly zero
    x = synthetic.activations(g, 3, cols)
    y, T = oracle.matvec(fmt, blocks, x, rows, cols)
    assert np.all(y[:, 4] == 0) and np.all(T[:, 4] == 0)
    # each of the n_vec columns equals its own n_vec = 1 matvec
    for v in range(3):
        y1, _ = oracle.matvec(fmt, blocks, x[v:v + 1], rows, cols)
        assert np.array_equal(y1[0], y[v])
    # linearity in x: y(2x) = 2 y(x) exactly (scaling by 2 is exact)
    y2, _ = oracle.matvec(fmt, blocks, 2 * x, rows, cols)
    assert np.array_equal(y2, 2 * y)


def test_rows_subset_matches_full():
    g = synthetic.rng(8)
    W = synthetic.weights(g, 40, 128)
    blocks = oracle.quantize_q8_0(W)
    x = synthetic.activations(g, 2, 128)
    y, T = oracle.matvec("q8_0", blocks, x, 40, 128)
    ys, Ts = oracle.matvec_rows("q8_0", blocks, x, 40, 128, 13, 29)
    assert np.array_equal(ys, y[:, 13:29]) and np.array_equal(Ts, T[:, 13:29])


def test_moe_equals_loop_of_single_expert_matvecs():
    n_experts, n_active, rows, cols, n_vec = 6, 3, 10, 64, 4
    g = synthetic.rng(9)
    W = synthetic.weights(g, n_experts * rows, cols)
    bank = oracle.quantize_q8_0(W)                      # experts stacked along rows
    ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
    per = bank.reshape(n_experts, rows, -1)
    for x_per_slot in (False, True):
        x = synthetic.activations(g, n_vec * (n_active if x_per_slot else 1), cols)
        y, T = oracle.moe_matvec_q8_0(bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
        for t in range(n_vec):
            for k in range(n_active):
                xv = x[t * n_active + k] if x_per_slot else x[t]
                y1, T1 = oracle_np.matvec("q8_0", per[ids[t, k]], xv, rows, cols)
                assert np.allclose(y[t, k], y1[0], rtol=1e-12, atol=1e-12 * T1.max())
                assert np.allclose(T[t, k], T1[0], rtol=1e-12)


def test_moe_all_same_expert_is_copies():
    n_experts, n_active, rows, cols, n_vec = 4, 2, 8, 96, 3
    g = synthetic.rng(10)
    bank = oracle.quantize_q8_0(synthetic.weights(g, n_experts * rows, cols))
    ids = np.full((n_vec, n_active), 2, dtype=np.int32)
    x = synthetic.activations(g, n_vec, cols)
    y, _ = oracle.moe_matvec_q8_0(bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
    y1, _ = oracle.matvec("q8_0", bank.reshape(n_experts, rows, -1)[2], x, rows, cols)
    for k in range(n_active):
        assert np.array_equal(y[:, k], y1)


def test_moe_rejects_out_of_range_ids():
    bank = np.zeros((2 * 4, 34), np.uint8)
    ids = np.array([[0, 2]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.moe_matvec_q8_0(bank, ids, np.zeros((1, 32), np.float32), False, 2, 2, 4, 32, 1)
