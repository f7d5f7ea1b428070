"""Pins of the oracle's QLoRA adapter term ("One Native Stack ...", section
"The Central Efficiency Thesis", Lemma "QLoRA over the unified core is
exact": y_i = sum_j What_ij x_j + (alpha/r) (B_A (A x))_i, A and B_A in bf16).

The C oracle returns the adapter term alone; it is checked here against the
IEEE bf16 definition, a NumPy f64 statement built from the decoded fields,
and closed forms that fix each index and the scale."""
import numpy as np

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic


def _bf16_bits(a):
    """fp32 values -> bf16 bit patterns, rounded to nearest even (test data only)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def test_bf16_known_values():
    # values fixed by the IEEE bf16 layout (1 sign, 8 exponent bits, 7 fraction bits)
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0x3E80: 0.25, 0x4049: 3.140625,
             0x0000: 0.0, 0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
             0xC2F6: -123.0, 0x3DCD: 0.10009765625}
    for h, v in cases.items():
        assert oracle.bf16_to_float(h) == v, hex(h)
    assert np.copysign(1.0, oracle.bf16_to_float(0x8000)) == -1.0
    assert oracle.bf16_to_float(0x7F80) == float("inf")


def test_bf16_all_finite_patterns_match_field_decode():
    h = np.arange(0, 1 << 16, dtype=np.uint16)
    fin = ((h >> 7) & 0xFF) != 0xFF
    got = np.array([oracle.bf16_to_float(int(v)) for v in h[fin][::13]])
    ref = oracle_np.bf16_to_f64(h[fin][::13])
    assert np.array_equal(got, ref)


def _case(seed, rank, rows, cols, n_vec):
    g = synthetic.rng(seed)
    A = _bf16_bits(g.standard_normal((rank, cols)) * 0.05)
    B = _bf16_bits(g.standard_normal((rows, rank)) * 0.05)
    x = synthetic.activations(g, n_vec, cols)
    return A, B, x


def test_brute_force_against_numpy():
    for seed, (rank, rows, cols, n_vec) in enumerate([(1, 3, 32, 1), (4, 7, 96, 3), (16, 33, 256, 8), (8, 5, 40, 2)]):
        A, B, x = _case(100 + seed, rank, rows, cols, n_vec)
        for scale in (2.0, -0.37, 1.0 / 16):
            d, T = oracle.lora_delta(A, B, x, scale)
            d_ref, T_ref = oracle_np.lora_delta(A, B, x, scale)
            assert np.allclose(d, d_ref, rtol=1e-12, atol=1e-14)
            assert np.allclose(T, T_ref, rtol=1e-12, atol=1e-14)


def test_ranks_beyond_the_kernel_limit():
    # the oracle has no rank limit of its own: ranks 65 and 100 (above the
    # kernels' 64) still equal the NumPy statement term for term, and a rank
    # below 1 is refused rather than answered
    for seed, rank in ((11, 65), (12, 100)):
        A, B, x = _case(seed, rank, 9, 64, 2)
        d, T = oracle.lora_delta(A, B, x, 0.75)
        d_ref, T_ref = oracle_np.lora_delta(A, B, x, 0.75)
        assert np.allclose(d, d_ref, rtol=1e-12, atol=1e-14)
        assert np.allclose(T, T_ref, rtol=1e-12, atol=1e-14)
        # the last adapter row matters: dropping it changes the answer
        d_cut, _ = oracle_np.lora_delta(A[:64], B[:, :64], x, 0.75)
        assert not np.allclose(d, d_cut, rtol=1e-9, atol=0)
    try:
        oracle.lora_delta(np.zeros((0, 32), np.uint16), np.zeros((3, 0), np.uint16),
                          np.zeros((1, 32), np.float32), 1.0)
    except ValueError:
        pass
    else:
        raise AssertionError("rank 0 was accepted")


def test_closed_forms():
    rank, rows, cols = 3, 4, 8
    x = np.arange(1, 2 * cols + 1, dtype=np.float32).reshape(2, cols)
    one = 0x3F80
    # A picks columns 5, 0, 7; B sends adapter k to row (k+1) % rows and row 0 also gets adapter 2 twice
    A = np.zeros((rank, cols), np.uint16)
    A[0, 5] = A[1, 0] = A[2, 7] = one
    B = np.zeros((rows, rank), np.uint16)
    B[1, 0] = B[2, 1] = B[3, 2] = one
    B[0, 2] = 0x4000                                  # 2.0
    d, T = oracle.lora_delta(A, B, x, 0.5)
    for v in range(2):
        u = [x[v, 5], x[v, 0], x[v, 7]]
        assert list(d[v]) == [0.5 * 2 * u[2], 0.5 * u[0], 0.5 * u[1], 0.5 * u[2]]
    assert np.array_equal(T, np.abs(d))
    # B = 0 gives no term; the term is linear in the scale and per column independent
    A, B, x = _case(7, 5, 6, 64, 3)
    assert np.all(oracle.lora_delta(A, np.zeros_like(B), x, 3.0)[0] == 0)
    d1, _ = oracle.lora_delta(A, B, x, 1.0)
    d3, _ = oracle.lora_delta(A, B, x, -3.0)
    assert np.allclose(d3, -3.0 * d1, rtol=1e-15, atol=0)
    for v in range(3):
        assert np.array_equal(oracle.lora_delta(A, B, x[v:v + 1], 1.0)[0][0], d1[v])
