"""GB300 (sm_103a) quantized-weight matvec library: Python binding.

The compute lives in ``libhq.so`` (hand-written CUDA, C ABI in
``include/hq.h``); this package only marshals arguments to it.  Every entry
point has the C name and the C argument order; tensors may be passed as torch
tensors (their ``data_ptr()`` is used) or as raw integer device addresses.
``stream`` defaults to torch's current CUDA stream.

There is no CPU fallback: if the library is missing or no sm_103a GPU is
present, the calls raise ``HQError``.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    HQError,
    HQ_OK, HQ_ERR_NULL, HQ_ERR_SHAPE, HQ_ERR_ALIGN, HQ_ERR_NVEC, HQ_ERR_LAUNCH,
    HQ_ERR_UNSUPPORTED, HQ_ERR_DEVICE, HQ_FAULT_WAIT_TIMEOUT, HQ_FAULT_EXPERT_ID,
    lib, lib_path, hq_version, hq_last_error,
    hq_matvec_q8_0, hq_matvec_q4_0, hq_matvec_i8_requant, hq_moe_matvec_q8_0,
    hq_matvec_q4_k, hq_quantize_q4_k, FMT_CODES, QK_K, Q4_K_BLOCK_BYTES,
    hq_moe_matvec_q8_0_swiglu, hq_moe_matvec_q8_0_combine, hq_moe_matvec_q8_0_ex,
    HQ_MOE_EPI_NONE, HQ_MOE_EPI_SWIGLU, HQ_MOE_EPI_COMBINE, HQ_MOE_IDS_READY,
    hq_matvec_q8_0_lora, hq_matvec_q4_0_lora, hq_matvec_q8_0_lora_noalloc,
    hq_quantize_q8_0, hq_quantize_q4_0, hq_quantize_i8_rows, hq_requant_params,
    hq_requant_i32_debug, hq_device_fault, hq_selftest_wait_timeout, hq_launch_count, hq_debug_plan,
    Q8_0_BLOCK_BYTES, Q4_0_BLOCK_BYTES, QK, row_bytes,
)
