"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/hq.h declares, validates arguments on the host before any launch, and
its host-only function (hq_requant_params) matches the oracle bit for bit.
No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from quantized_weight_matvec_hq_gb300 import build as hq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hq():
    hq_build.build()
    import quantized_weight_matvec_hq_gb300 as hq
    hq.lib()
    return hq


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "hq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(hq):
    names = _declared_functions()
    assert len(names) >= 12
    L = ctypes.CDLL(hq.lib_path())
    for n in names:
        assert hasattr(L, n), n
    # and the binding wraps each one under the same name
    for n in names:
        assert callable(getattr(hq, n)), n


def test_version_and_error_string(hq):
    assert hq.hq_version() == 10000
    assert isinstance(hq.hq_last_error(), str)


def test_host_validation_before_any_launch(hq):
    L = hq.lib()
    # null pointers
    assert L.hq_matvec_q8_0(0, 0, 0, 4, 64, 1, 0) == hq.HQ_ERR_NULL
    assert "non-null" in hq.hq_last_error()
    fake = 1 << 40                              # 16-byte aligned, never dereferenced
    # n_vec out of range
    assert L.hq_matvec_q8_0(fake, fake, fake, 4, 64, 0, 0) == hq.HQ_ERR_NVEC
    assert L.hq_matvec_q4_0(fake, fake, fake, 4, 64, 9, 0) == hq.HQ_ERR_NVEC
    # shapes
    assert L.hq_matvec_q8_0(fake, fake, fake, 0, 64, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_matvec_q8_0(fake, fake, fake, 4, 48, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_matvec_q8_0(fake, fake, fake, 4, 16, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_matvec_i8_requant(fake, fake, fake, fake, fake, 4, 6, 1, 0) == hq.HQ_ERR_SHAPE
    # alignment
    assert L.hq_matvec_q8_0(fake + 2, fake, fake, 4, 64, 1, 0) == hq.HQ_ERR_ALIGN
    assert L.hq_matvec_q4_0(fake, fake + 4, fake, 4, 64, 1, 0) == hq.HQ_ERR_ALIGN
    # MoE
    assert L.hq_moe_matvec_q8_0(fake, fake, fake, 0, fake, 4, 5, 8, 256, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_moe_matvec_q8_0(fake, fake, fake, 2, fake, 4, 2, 8, 256, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_moe_matvec_q8_0(fake, fake, fake, 0, fake, 64, 64, 8, 256, 8, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_moe_matvec_q8_0(fake, fake, fake, 0, fake, 4, 2, 8, 288, 1, 0) == hq.HQ_ERR_SHAPE
    # SwiGLU pairs rows: an odd row count is refused; the combine needs its weights and workspaces
    assert L.hq_moe_matvec_q8_0_swiglu(fake, fake, fake, 0, fake, 4, 2, 9, 256, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_moe_matvec_q8_0_swiglu(fake, fake, 0, 0, fake, 4, 2, 8, 256, 1, 0) == hq.HQ_ERR_NULL
    assert L.hq_moe_matvec_q8_0_combine(fake, fake, fake, 1, 0, fake, 4, 2, 8, 256, 1, 0) == hq.HQ_ERR_NULL
    assert L.hq_moe_matvec_q8_0_combine(fake, fake, fake, 1, fake + 2, fake, 4, 2, 8, 256, 1, 0) == hq.HQ_ERR_ALIGN
    assert L.hq_moe_matvec_q8_0_combine(fake, fake, fake, 1, fake, fake, 4, 5, 8, 256, 1, 0) == hq.HQ_ERR_SHAPE
    # MoE with flags: unknown epilogues and flags are refused, the combine needs its weights
    Le = L.hq_moe_matvec_q8_0_ex
    assert Le(fake, fake, fake, 0, 0, fake, 4, 2, 8, 256, 1, 3, 0, 0) == hq.HQ_ERR_UNSUPPORTED
    assert Le(fake, fake, fake, 0, 0, fake, 4, 2, 8, 256, 1, 0, 2, 0) == hq.HQ_ERR_UNSUPPORTED
    assert Le(fake, fake, fake, 1, 0, fake, 4, 2, 8, 256, 1, 2, 1, 0) == hq.HQ_ERR_NULL
    assert Le(fake, fake, fake, 0, 0, fake, 4, 2, 9, 256, 1, 1, 1, 0) == hq.HQ_ERR_SHAPE
    assert Le(fake, fake, fake, 0, 0, fake, 4, 5, 8, 256, 1, 0, 1, 0) == hq.HQ_ERR_SHAPE
    # Q4_K: super-blocks of 256 columns, W and x 16-byte aligned
    assert L.hq_matvec_q4_k(fake, fake, fake, 4, 288, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_matvec_q4_k(fake, fake, fake, 4, 224, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_matvec_q4_k(fake + 8, fake, fake, 4, 256, 1, 0) == hq.HQ_ERR_ALIGN
    assert L.hq_matvec_q4_k(fake, fake, fake, 4, 256, 0, 0) == hq.HQ_ERR_NVEC
    assert L.hq_quantize_q4_k(fake, fake, 4, 288, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_quantize_q4_k(fake, fake + 8, 4, 256, 0) == hq.HQ_ERR_ALIGN
    # quantizers
    assert L.hq_quantize_q8_0(fake, fake, 4, 40, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_quantize_q4_0(0, fake, 4, 64, 0) == hq.HQ_ERR_NULL
    # QLoRA entry points
    Lq = L.hq_matvec_q8_0_lora
    assert Lq(fake, fake, 0, fake, 1.0, 16, fake, fake, 4, 64, 1, 0) == hq.HQ_ERR_NULL
    assert Lq(fake, fake, fake, fake, 1.0, 0, fake, fake, 4, 64, 1, 0) == hq.HQ_ERR_SHAPE
    assert Lq(fake, fake, fake, fake, 1.0, 65, fake, fake, 4, 64, 1, 0) == hq.HQ_ERR_SHAPE
    assert Lq(fake, fake, fake, fake, float("inf"), 16, fake, fake, 4, 64, 1, 0) == hq.HQ_ERR_SHAPE
    assert Lq(fake, fake, fake + 2, fake, 1.0, 16, fake, fake, 4, 64, 1, 0) == hq.HQ_ERR_ALIGN
    assert L.hq_matvec_q4_0_lora(fake, fake, fake, fake, 1.0, 16, fake, fake, 4, 64, 9, 0) == hq.HQ_ERR_NVEC
    assert L.hq_matvec_q8_0_lora_noalloc(fake, fake, fake, fake, 1.0, 65, fake, 4, 64, 1, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_matvec_q8_0_lora_noalloc(fake, fake, 0, fake, 1.0, 16, fake, 4, 64, 1, 0) == hq.HQ_ERR_NULL
    # the wait-timeout self-test bounds its limit before touching a device
    assert L.hq_selftest_wait_timeout(0, 0) == hq.HQ_ERR_SHAPE
    assert L.hq_selftest_wait_timeout(5_000_000_000, 0) == hq.HQ_ERR_SHAPE
    with pytest.raises(hq.HQError):
        hq.hq_matvec_q8_0(0, 0, 0, 4, 64, 1, stream=0)


def test_requant_params_match_oracle(hq):
    g = np.random.Generator(np.random.PCG64(21))
    M = np.exp(g.uniform(np.log(1e-9), np.log(0.9999), size=20000))
    M[:4] = [0.5, 0.75, 2.0 ** -10, 0.3]
    mult = np.empty(M.size, np.int32)
    shift = np.empty(M.size, np.int32)
    hq.hq_requant_params(M, M.size, mult, shift)
    om, osh = oracle.requant_params(M)
    assert np.array_equal(mult, om) and np.array_equal(shift, osh)
    with pytest.raises(hq.HQError):
        hq.hq_requant_params(np.array([1.5]), 1, np.empty(1, np.int32), np.empty(1, np.int32))


def test_header_cites_each_entry_point():
    text = open(os.path.join(ROOT, "include", "hq.h")).read()
    for name in ("hq_matvec_q8_0", "hq_matvec_q4_0", "hq_matvec_q4_k", "hq_matvec_i8_requant",
                 "hq_moe_matvec_q8_0", "hq_quantize_q8_0", "hq_quantize_q4_k", "hq_requant_params",
                 "hq_requant_i32_debug"):
        block = text[text.index(" * " + name) if (" * " + name) in text else text.index(name):]
        assert "Source:" in block.split(");")[0] or "Source:" in block[:2500], name
