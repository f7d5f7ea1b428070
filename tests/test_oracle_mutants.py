"""Planted mistakes: each test copies the C oracle to a temporary directory,
plants one plausible bug by a textual edit (a dropped term, a wrong sign or
index, a swapped nibble, a transposed operand, a wrong rounding rule), builds
it with gcc and runs the same pins the real oracle passes.  At least one pin
must catch every mutant.  Nothing here touches the GPU or the product.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import oracle_np
from quantized_weight_matvec_hq_gb300 import synthetic

SRC = os.path.join(os.path.dirname(oracle.__file__), "hq_oracle.c")

MUTANTS = {
    "nibble_order_swapped": ("int lo = blk[2 + j] & 0x0f;\n                int hi = blk[2 + j] >> 4;",
                             "int hi = blk[2 + j] & 0x0f;\n                int lo = blk[2 + j] >> 4;"),
    "matvec_nibble_order_swapped": ("(j < 16 ? (blk[2 + j] & 0x0f) : (blk[2 + j - 16] >> 4))",
                                    "(j < 16 ? (blk[2 + j] >> 4) : (blk[2 + j - 16] & 0x0f))"),
    "q8_unsigned_quants": ("if (fmt == 8) q = (int8_t)blk[2 + j];", "if (fmt == 8) q = (uint8_t)blk[2 + j];"),
    "dropped_last_element": ("for (int j = 0; j < HQO_QK; ++j) {\n                    int q;",
                             "for (int j = 0; j < HQO_QK - 1; ++j) {\n                    int q;"),
    "q4_offset_7": ("- 8;\n                    double w = d * (double)q;", "- 7;\n                    double w = d * (double)q;"),
    "transposed_x": ("x[(int64_t)v * cols + b * HQO_QK + j]", "x[(b * HQO_QK + j) * n_vec + v]"),
    "scale_wrong_byte_order": ("static uint16_t load_u16le(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }",
                               "static uint16_t load_u16le(const uint8_t *p) { return (uint16_t)(p[1] | (p[0] << 8)); }"),
    "srdhm_nudge_sign": ("int64_t nudge = ab >= 0 ? ((int64_t)1 << 30) : (1 - ((int64_t)1 << 30));",
                         "int64_t nudge = ((int64_t)1 << 30);"),
    "rdivbypot_no_negative_adjust": ("int64_t thr = (mask >> 1) + (x < 0 ? 1 : 0);", "int64_t thr = (mask >> 1);"),
    "requant_order_swapped": ("int32_t r = hqo_rdivbypot(hqo_srdhm(acc, mult), shift);",
                              "int32_t r = hqo_srdhm(hqo_rdivbypot(acc, shift), mult);"),
    "half_ties_away": ("if (rem > 0.5 || (rem == 0.5 && (ki & 1u))) ki += 1;", "if (rem >= 0.5) ki += 1;"),
    "q8_scale_254": ("float d = amax / 127.0f;\n            uint16_t dh", "float d = amax / 254.0f;\n            uint16_t dh"),
    "q4_scale_positive": ("float d = m / -8.0f;", "float d = m / 8.0f;"),
    "q4_round_down": ("float t = w[j] / d + 8.5f;", "float t = w[j] / d + 8.0f;"),
    "lora_A_transposed": ("hqo_bf16_to_float(A[k * cols + j])", "hqo_bf16_to_float(A[j * rank + k])"),
    "lora_B_transposed": ("hqo_bf16_to_float(B[i * rank + k])", "hqo_bf16_to_float(B[k * rows + i])"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "swiglu_gate_up_swapped": ("double gate = y[2 * i], up = y[2 * i + 1];",
                               "double gate = y[2 * i + 1], up = y[2 * i];"),
    "combine_weights_transposed": ("double wk = (double)w[t * n_active + k];",
                                   "double wk = (double)w[k * n_vec + t];"),
    "lora_scale_dropped": ("delta[v * rows + i] = scale * acc;", "delta[v * rows + i] = acc;"),
    "bf16_shift_15": ("uint32_t u = (uint32_t)h << 16;", "uint32_t u = (uint32_t)h << 15;"),
    "q4k_sub_block_nibbles_swapped": ("return (j & 1) ? (b >> 4) : (b & 0x0f);",
                                      "return (j & 1) ? (b & 0x0f) : (b >> 4);"),
    "q4k_interleaved_nibbles": ("uint8_t b = blk[16 + 32 * (j / 2) + l];\n    return (j & 1) ? (b >> 4) : (b & 0x0f);",
                                "uint8_t b = blk[16 + e / 2];\n    (void)j; (void)l;\n    return (e & 1) ? (b >> 4) : (b & 0x0f);"),
    "q4k_min_term_sign": ("return d * (double)sc * (double)q4k_quant(blk, e) - dmin * (double)m;",
                          "return d * (double)sc * (double)q4k_quant(blk, e) + dmin * (double)m;"),
    "q4k_scale_high_bits_wrong_byte": ("*sc = (s12[j + 4] & 0x0f) | ((s12[j - 4] >> 6) << 4);",
                                       "*sc = (s12[j + 4] & 0x0f) | ((s12[j] >> 6) << 4);"),
    "q4k_d_dmin_swapped": ("double d = (double)hqo_half_to_float(load_u16le(blk));\n    double dmin = (double)hqo_half_to_float(load_u16le(blk + 2));",
                           "double d = (double)hqo_half_to_float(load_u16le(blk + 2));\n    double dmin = (double)hqo_half_to_float(load_u16le(blk));"),
    "q4k_encoder_min_not_clamped": ("if (mn > 0.0f) mn = 0.0f;\n", "\n"),
    "q4k_encoder_scale_over_16": ("scale[j] = (mx - mn) / 15.0f;", "scale[j] = (mx - mn) / 16.0f;"),
}


def _build_mutant(tmp_path, name):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    p = tmp_path / f"{name}.c"
    p.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(p), "-lm"], check=True)
    L = ctypes.CDLL(str(so))
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    for fn in ("hqo_quantize_q8_0", "hqo_quantize_q4_0", "hqo_quantize_q4_k"):
        getattr(L, fn).argtypes = [vp, i64, i64, vp]
    for fn in ("hqo_dequant_q8_0", "hqo_dequant_q4_0", "hqo_dequant_q4_k"):
        getattr(L, fn).argtypes = [vp, i64, i64, vp]
    for fn in ("hqo_matvec_q8_0", "hqo_matvec_q4_0", "hqo_matvec_q4_k"):
        getattr(L, fn).argtypes = [vp, vp, i64, i64, ci, vp, vp]
    L.hqo_srdhm.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.hqo_srdhm.restype = ctypes.c_int32
    L.hqo_rdivbypot.argtypes = [ctypes.c_int32, ci]
    L.hqo_rdivbypot.restype = ctypes.c_int32
    L.hqo_requant.argtypes = [ctypes.c_int32] * 3
    L.hqo_requant.restype = ctypes.c_int8
    L.hqo_float_to_half_rne.argtypes = [ctypes.c_float]
    L.hqo_float_to_half_rne.restype = ctypes.c_uint16
    L.hqo_bf16_to_float.argtypes = [ctypes.c_uint16]
    L.hqo_bf16_to_float.restype = ctypes.c_float
    L.hqo_lora_delta.argtypes = [vp, vp, vp, ctypes.c_double, i64, i64, i64, i64, vp, vp]
    L.hqo_silu.argtypes = [ctypes.c_double]
    L.hqo_silu.restype = ctypes.c_double
    L.hqo_swiglu_pairs.argtypes = [vp, i64, vp]
    L.hqo_moe_combine.argtypes = [vp, vp, vp, ci, ci, i64, vp, vp]
    return L


def _pins_fail(L, golden_dir):
    """Run the oracle's pins against library L; return the names of those that fail."""
    failed = []
    ptr = lambda a: a.ctypes.data
    # golden blocks
    gold = json.load(open(os.path.join(golden_dir, "blocks.json")))["blocks"]
    from test_oracle_blocks import _weights
    for b in gold:
        w = _weights(b["name"])
        out = np.empty(34 if b["format"] == "q8_0" else 18, np.uint8)
        fn = L.hqo_quantize_q8_0 if b["format"] == "q8_0" else L.hqo_quantize_q4_0
        fn(ptr(w), 1, 32, ptr(out))
        if out.tobytes() != bytes.fromhex(b["bytes_hex"]):
            failed.append("golden:" + b["name"])
    # the independent vectorised quantizers, byte for byte
    g = synthetic.rng(78)
    W = synthetic.weights(g, 16, 128)
    for fmt, bpb in (("q8_0", 34), ("q4_0", 18)):
        out = np.empty((16, 4 * bpb), np.uint8)
        (L.hqo_quantize_q8_0 if fmt == "q8_0" else L.hqo_quantize_q4_0)(ptr(W), 16, 128, ptr(out))
        ref = oracle_np.quantize_q8_0(W) if fmt == "q8_0" else oracle_np.quantize_q4_0(W)
        if not np.array_equal(out, ref):
            failed.append("quantizer:" + fmt)
    # brute force matvec and dequant on tiny shapes
    for fmt in ("q8_0", "q4_0"):
        g = synthetic.rng(77)
        rows, cols, n_vec = 5, 96, 3
        W = synthetic.weights(g, rows, cols)
        blocks = oracle.quantize_q8_0(W) if fmt == "q8_0" else oracle.quantize_q4_0(W)
        x = synthetic.activations(g, n_vec, cols)
        y = np.empty((n_vec, rows)); T = np.empty((n_vec, rows))
        (L.hqo_matvec_q8_0 if fmt == "q8_0" else L.hqo_matvec_q4_0)(
            ptr(blocks), ptr(x), rows, cols, n_vec, ptr(y), ptr(T))
        y_ref, _ = oracle_np.matvec(fmt, blocks, x, rows, cols)
        if not np.allclose(y, y_ref, rtol=1e-12, atol=1e-12):
            failed.append("brute:" + fmt)
        Wd = np.empty((rows, cols))
        (L.hqo_dequant_q8_0 if fmt == "q8_0" else L.hqo_dequant_q4_0)(ptr(blocks), rows, cols, ptr(Wd))
        ref = oracle_np.dequant_q8_0(blocks, rows, cols) if fmt == "q8_0" else oracle_np.dequant_q4_0(blocks, rows, cols)
        if not np.array_equal(Wd, ref):
            failed.append("dequant:" + fmt)
    # Q4_K: the hand-worked super-blocks, the NumPy encoder and decoder, brute force
    from test_oracle_q4_k import _golden as q4k_golden, _block_bytes as q4k_bytes, _special_weights
    gk = q4k_golden()
    blk = q4k_bytes(gk["q4_k_decode"])
    wd = np.empty(256)
    L.hqo_dequant_q4_k(ptr(blk), 1, 256, ptr(wd))
    for e in range(256):
        j, l = divmod(e, 32)
        q = l % 16 if j % 2 == 0 else 15 - l % 16
        if wd[e] != gk["q4_k_decode"]["d"] * gk["q4_k_decode"]["sc"][j] * q - gk["q4_k_decode"]["dmin"] * gk["q4_k_decode"]["m"][j]:
            failed.append("golden:q4_k_decode")
            break
    ramp = np.tile(np.array([(l % 16) - 7.5 for l in range(32)], np.float32), 8).reshape(1, 256)
    out = np.empty(144, np.uint8)
    L.hqo_quantize_q4_k(ptr(ramp), 1, 256, ptr(out))
    if out.tobytes() != q4k_bytes(gk["q4_k_encode_ramp"]).tobytes():
        failed.append("golden:q4_k_encode_ramp")
    Wk = _special_weights(21, 512, 79)
    out = np.empty((21, 288), np.uint8)
    L.hqo_quantize_q4_k(ptr(Wk), 21, 512, ptr(out))
    if not np.array_equal(out, oracle_np.quantize_q4_k(Wk)):
        failed.append("quantizer:q4_k")
    blocks = oracle.quantize_q4_k(Wk)
    Wd = np.empty((21, 512))
    L.hqo_dequant_q4_k(ptr(blocks), 21, 512, ptr(Wd))
    if not np.array_equal(Wd, oracle_np.dequant_q4_k(blocks, 21, 512)):
        failed.append("dequant:q4_k")
    xk = synthetic.activations(synthetic.rng(80), 3, 512)
    y = np.empty((3, 21)); T = np.empty((3, 21))
    L.hqo_matvec_q4_k(ptr(blocks), ptr(xk), 21, 512, 3, ptr(y), ptr(T))
    if not np.allclose(y, oracle_np.matvec("q4_k", blocks, xk, 21, 512)[0], rtol=1e-12, atol=1e-12):
        failed.append("brute:q4_k")
    # integer rules
    w = json.load(open(os.path.join(golden_dir, "gemmlowp_worked.json")))
    if any(L.hqo_srdhm(c["a"], c["b"]) != c["out"] for c in w["srdhm"]):
        failed.append("srdhm")
    if any(L.hqo_rdivbypot(c["x"], c["e"]) != c["out"] for c in w["rdivbypot"]):
        failed.append("rdivbypot")
    if any(L.hqo_requant(c["acc"], c["mult"], c["shift"]) != c["out"] for c in w["requant"]):
        failed.append("requant")
    # half conversion ties
    h = np.arange(0, 0x7BFF, dtype=np.uint16)
    mids = ((h.view(np.float16).astype(np.float64) + (h + 1).view(np.float16).astype(np.float64)) / 2)
    mids = mids[mids == mids.astype(np.float32).astype(np.float64)].astype(np.float32)[::37]
    ref = mids.astype(np.float16).view(np.uint16)
    if any(L.hqo_float_to_half_rne(float(v)) != r for v, r in zip(mids, ref)):
        failed.append("half")
    # QLoRA adapter term: bf16 values and a non-square brute force
    if L.hqo_bf16_to_float(0x3F80) != 1.0 or L.hqo_bf16_to_float(0xC2F6) != -123.0:
        failed.append("bf16")
    from test_oracle_lora import _case
    rank, rows, cols, n_vec = 3, 7, 40, 2
    A, B, x = _case(11, rank, rows, cols, n_vec)
    d = np.empty((n_vec, rows)); T = np.empty((n_vec, rows))
    L.hqo_lora_delta(ptr(A), ptr(B), ptr(x), 0.75, rank, rows, cols, n_vec, ptr(d), ptr(T))
    d_ref, _ = oracle_np.lora_delta(A, B, x, 0.75)
    if not np.allclose(d, d_ref, rtol=1e-12, atol=1e-14):
        failed.append("lora")
    # MoE epilogues: sigmoid(ln 3) = 3/4, the gate/up pairing, a brute-force combine
    ln3 = np.log(3.0)
    if abs(L.hqo_silu(ln3) - 0.75 * ln3) > 1e-15 or abs(L.hqo_silu(-ln3) + 0.25 * ln3) > 1e-15:
        failed.append("silu")
    yp = np.array([ln3, 2.0, 0.5, -1.0]); hp = np.empty(2)
    L.hqo_swiglu_pairs(ptr(yp), 2, ptr(hp))
    if abs(hp[0] - 1.5 * ln3) > 1e-15:
        failed.append("swiglu")
    g = synthetic.rng(321)
    yc = g.standard_normal((2, 3, 4)); wc = g.standard_normal((2, 3)).astype(np.float32)
    oc = np.empty((2, 4)); Tc = np.empty((2, 4))
    L.hqo_moe_combine(ptr(yc), ptr(np.abs(yc)), ptr(wc), 2, 3, 4, ptr(oc), ptr(Tc))
    if not np.allclose(oc, oracle_np.moe_combine(yc, wc), rtol=1e-13):
        failed.append("combine")
    return failed


def test_unmutated_oracle_passes_all_pins(tmp_path, golden_dir):
    MUTANTS["identity"] = ("int hqo_version(void) { return 1; }", "int hqo_version(void) { return 1; }")
    try:
        assert _pins_fail(_build_mutant(tmp_path, "identity"), golden_dir) == []
    finally:
        del MUTANTS["identity"]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, golden_dir, name):
    assert _pins_fail(_build_mutant(tmp_path, name), golden_dir), f"mutant {name} passed every pin"
