"""The exact folded decode of the wide-vector kernels, checked in plain
arithmetic on the CPU (no GPU, no kernel code): for every finite fp16 scale d
and every quant value, one fused multiply-add of the 2^23-biased quant with
the scaled d gives the dequantized weight exactly.

Q8_0: the byte u = q + 128 at bits 8..15 of 2^23 is f = 2^23 + 256 u; with
d' = d / 256 and c = -(2^23 + 2^15) d', fma(f, d', c) = q d.
Q4_0: the nibble n at bit p of 2^23 is f = 2^23 + n 2^p; with d_p = d 2^-p and
c_p = -(2^23 + 8 2^p) d_p, fma(f, d_p, c_p) = (n - 8) d for p = 8, 12, 16.

Each step the kernels take in fp32 is checked to be exact: the scaling of d,
the constant c (an fp32 product), and the fma, whose exact value is formed in
float64 (every operand and product here has at most 35 significant bits) and
must survive rounding to fp32 unchanged.
"""
import numpy as np


def finite_fp16_scales():
    bits = np.arange(1 << 16, dtype=np.uint16)
    d = bits.view(np.float16)
    return d[np.isfinite(d)].astype(np.float32)


def exact_in_f32(x64):
    return np.all(x64.astype(np.float32).astype(np.float64) == x64)


def test_q8_0_fold_is_exact():
    d = finite_fp16_scales()                                        # 63,488 values incl. subnormals and 0
    dq = d * np.float32(1.0 / 256.0)
    assert np.array_equal(dq.astype(np.float64), d.astype(np.float64) / 256.0)    # exact scaling
    c = np.float32(-8421376.0) * dq                                  # fp32 product, as on the GPU
    assert np.array_equal(c.astype(np.float64), -8421376.0 * dq.astype(np.float64))
    for q in range(-128, 128):
        f = np.float64(8388608.0 + 256.0 * (q + 128))
        fma = f * dq.astype(np.float64) + c.astype(np.float64)        # the fma's exact value
        assert exact_in_f32(fma), q
        assert np.array_equal(fma, q * d.astype(np.float64)), q


def test_q4_0_fold_is_exact_at_bits_8_12_16():
    d = finite_fp16_scales()
    for p in (8, 12, 16):
        dp = d * np.float32(2.0 ** -p)
        assert np.array_equal(dp.astype(np.float64), d.astype(np.float64) * 2.0 ** -p)
        k = np.float32(-(2.0 ** 23 + 8 * 2.0 ** p))
        c = k * dp
        assert np.array_equal(c.astype(np.float64), np.float64(k) * dp.astype(np.float64)), p
        for n in range(16):
            f = np.float64(2.0 ** 23 + n * 2.0 ** p)
            fma = f * dp.astype(np.float64) + c.astype(np.float64)
            assert exact_in_f32(fma), (p, n)
            assert np.array_equal(fma, (n - 8) * d.astype(np.float64)), (p, n)


def test_q4_0_fold_fails_at_low_bits():
    """The reason the wide Q4_0 decode moves every nibble to bit 8 or above: at
    bit 0 the constant (2^23 + 8) d is not an fp32 value for some d, and the
    folded weight would be rounded."""
    d = finite_fp16_scales()
    k = np.float64(2.0 ** 23 + 8)
    c32 = (np.float32(k) * d).astype(np.float64)
    assert not np.array_equal(c32, k * d.astype(np.float64))
