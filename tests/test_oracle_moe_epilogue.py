"""Pins of the oracle's MoE epilogues: SwiGLU over an interleaved gate/up
matvec output ("Blue -- porting zen-nano (Qwen3-0.6B) ...", section
"Architecture": the feed-forward is SwiGLU(gate, up, down)) and the
router-weighted sum over a token's slots ("Economical Serving and the
hanzo.ai Platform", paragraph "MoE is the cheapest-per-quality tier": a
sparsely gated mixture).

silu is pinned by special values the mathematics fixes (sigmoid(ln k) =
k / (k + 1) exactly), its odd-part identity, its limits and an independent
tanh route; the pairing and the combine by hand-made cases and a NumPy brute
force over dequantized banks."""
import math

import numpy as np

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    # sigmoid(ln k) = k / (k + 1): silu(ln k) = ln k * k / (k + 1), silu(-ln k) = -ln k / (k + 1)
    for k in (2.0, 3.0, 7.0, 0.25):
        z = math.log(k)
        assert math.isclose(oracle.silu(z), z * k / (k + 1.0), rel_tol=4e-16)
        assert math.isclose(oracle.silu(-z), -z / (k + 1.0), rel_tol=4e-16)


def test_silu_identities_and_limits():
    z = np.concatenate([np.linspace(-30, 30, 241), [1e-300, -1e-300, 1e-8, 700.0]])
    s = np.array([oracle.silu(v) for v in z])
    sn = np.array([oracle.silu(-v) for v in z])
    # z sigmoid(z) + z sigmoid(-z) = z
    assert np.allclose(s - sn, z, rtol=1e-14, atol=1e-300)
    # the independent tanh route (it cancels in the far negative tail: absolute there)
    assert np.allclose(s, oracle_np.silu_tanh(z), rtol=1e-13, atol=1e-14)
    # silu(z) ~ z for large z, ~ z e^z for very negative z, ~ z/2 near 0
    assert oracle.silu(40.0) == 40.0
    assert math.isclose(oracle.silu(-40.0) / -40.0, 4.248354255291589e-18, rel_tol=1e-12)
    assert math.isclose(oracle.silu(1e-8), 0.5e-8, rel_tol=1e-8)
    assert oracle.silu(-1000.0) == 0.0 and oracle.silu(1000.0) == 1000.0


def test_swiglu_pairs_order():
    ln3 = math.log(3.0)
    y = np.array([[ln3, 2.0, -ln3, 4.0, 0.0, 9.0]])
    h = oracle.swiglu_pairs(y)
    # row 2i is the gate, row 2i+1 the up value
    assert np.allclose(h, [[0.75 * ln3 * 2.0, -0.25 * ln3 * 4.0, 0.0]], rtol=1e-15, atol=0)


def test_swiglu_bank_brute_force():
    for seed, (n_experts, n_active, inter, cols, n_vec) in enumerate([(6, 3, 4, 64, 2), (4, 4, 8, 96, 1)]):
        g = synthetic.rng(300 + seed)
        rows = 2 * inter
        bank = oracle.quantize_q8_0(synthetic.weights(g, n_experts * rows, cols))
        ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
        x = synthetic.activations(g, n_vec, cols) * 20.0          # gates well into both tails
        y, _ = oracle.moe_matvec_q8_0(bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
        h = oracle.swiglu_pairs(y)
        h_ref = oracle_np.moe_swiglu_q8_0(bank, ids, x, n_experts, rows, cols)
        assert np.allclose(h, h_ref, rtol=1e-12, atol=1e-15)


def test_combine_closed_forms():
    g = synthetic.rng(320)
    n_vec, n_active, rows = 3, 4, 5
    y = g.standard_normal((n_vec, n_active, rows))
    T = np.abs(y) * 3.0
    # one-hot weights pick a slot exactly
    for k in range(n_active):
        w = np.zeros((n_vec, n_active), np.float32)
        w[:, k] = 1.0
        out, Tout = oracle.moe_combine(y, T, w)
        assert np.array_equal(out, y[:, k]) and np.array_equal(Tout, T[:, k])
    # equal unit weights give the plain sum over slots, in slot order
    out, _ = oracle.moe_combine(y, T, np.ones((n_vec, n_active), np.float32))
    assert np.array_equal(out, ((y[:, 0] + y[:, 1]) + y[:, 2]) + y[:, 3])
    # a token's weights touch only its own outputs, and the sum is linear in them
    w = g.standard_normal((n_vec, n_active)).astype(np.float32)
    out, Tout = oracle.moe_combine(y, T, w)
    w2 = w.copy()
    w2[1] *= 2.0
    out2, _ = oracle.moe_combine(y, T, w2)
    assert np.array_equal(out2[[0, 2]], out[[0, 2]]) and np.allclose(out2[1], 2.0 * out[1], rtol=1e-15)
    assert np.allclose(Tout, np.einsum("tk,tki->ti", np.abs(w.astype(np.float64)), T), rtol=1e-14)
    assert np.allclose(out, oracle_np.moe_combine(y, w), rtol=1e-13, atol=1e-15)
