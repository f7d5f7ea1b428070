"""ctypes binding for libhq.so: argument marshalling only, same names as include/hq.h."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(HERE, "libhq.so")

HQ_OK = 0
HQ_ERR_NULL = -1
HQ_ERR_SHAPE = -2
HQ_ERR_ALIGN = -3
HQ_ERR_NVEC = -4
HQ_ERR_LAUNCH = -5
HQ_ERR_UNSUPPORTED = -6
HQ_ERR_DEVICE = -7
HQ_FAULT_WAIT_TIMEOUT = 1
HQ_FAULT_EXPERT_ID = 2

QK = 32
Q8_0_BLOCK_BYTES = 34
Q4_0_BLOCK_BYTES = 18
QK_K = 256
Q4_K_BLOCK_BYTES = 144
# format codes of hq_debug_plan
FMT_CODES = {"q8_0": 8, "q4_0": 4, "q4_k": 75, "i8": 1}

_NAMES = {HQ_ERR_NULL: "HQ_ERR_NULL", HQ_ERR_SHAPE: "HQ_ERR_SHAPE", HQ_ERR_ALIGN: "HQ_ERR_ALIGN",
          HQ_ERR_NVEC: "HQ_ERR_NVEC", HQ_ERR_LAUNCH: "HQ_ERR_LAUNCH",
          HQ_ERR_UNSUPPORTED: "HQ_ERR_UNSUPPORTED", HQ_ERR_DEVICE: "HQ_ERR_DEVICE"}


class HQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int

_SIGS = {
    "hq_version": ([], _int),
    "hq_last_error": ([], ctypes.c_char_p),
    "hq_matvec_q8_0": ([_vp, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "hq_matvec_q4_0": ([_vp, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "hq_matvec_q4_k": ([_vp, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "hq_quantize_q4_k": ([_vp, _vp, _i64, _i64, _vp], _int),
    "hq_matvec_i8_requant": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "hq_matvec_q8_0_lora": ([_vp, _vp, _vp, _vp, ctypes.c_float, _int, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "hq_matvec_q4_0_lora": ([_vp, _vp, _vp, _vp, ctypes.c_float, _int, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "hq_matvec_q8_0_lora_noalloc": ([_vp, _vp, _vp, _vp, ctypes.c_float, _int, _vp, _i64, _i64, _int, _vp], _int),
    "hq_moe_matvec_q8_0": ([_vp, _vp, _vp, _int, _vp, _i64, _int, _i64, _i64, _int, _vp], _int),
    "hq_moe_matvec_q8_0_swiglu": ([_vp, _vp, _vp, _int, _vp, _i64, _int, _i64, _i64, _int, _vp], _int),
    "hq_moe_matvec_q8_0_combine": ([_vp, _vp, _vp, _int, _vp, _vp, _i64, _int, _i64, _i64, _int, _vp], _int),
    "hq_moe_matvec_q8_0_ex": ([_vp, _vp, _vp, _int, _vp, _vp, _i64, _int, _i64, _i64, _int, _int, _int, _vp], _int),
    "hq_quantize_q8_0": ([_vp, _vp, _i64, _i64, _vp], _int),
    "hq_quantize_q4_0": ([_vp, _vp, _i64, _i64, _vp], _int),
    "hq_quantize_i8_rows": ([_vp, _vp, _vp, _i64, _i64, _vp], _int),
    "hq_requant_params": ([_vp, _i64, _vp, _vp], _int),
    "hq_requant_i32_debug": ([_vp, _vp, _vp, _vp, _i64, _i64, _vp], _int),
    "hq_device_fault": ([_vp], _int),
    "hq_selftest_wait_timeout": ([_i64, _vp], _int),
    "hq_launch_count": ([], ctypes.c_uint64),
    "hq_debug_plan": ([_int, _int, _i64, _i64, _int, _int, _int, ctypes.POINTER(ctypes.c_int64), _int], _int),
}


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libhq.so (built by ``build.py``); raise HQError if it is missing."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(_LIB_PATH):
                    raise HQError(HQ_ERR_UNSUPPORTED,
                                  f"{_LIB_PATH} is missing: run quantized_weight_matvec_hq_gb300/build.py")
                L = ctypes.CDLL(_LIB_PATH)
                for name, (args, res) in _SIGS.items():
                    fn = getattr(L, name)
                    fn.argtypes = args
                    fn.restype = res
                _lib = L
    return _lib


def _addr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return int(t.data_ptr())
    if hasattr(t, "ctypes"):                      # numpy array (host functions)
        return int(t.ctypes.data)
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(s) -> int:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(status: int) -> int:
    if status != HQ_OK:
        raise HQError(status, lib().hq_last_error().decode())
    return status


def row_bytes(fmt: str, cols: int) -> int:
    """Bytes of one quantized row: cols/32 blocks of 34 (Q8_0) or 18 (Q4_0)
    bytes, or cols/256 super-blocks of 144 (Q4_K) bytes."""
    if fmt == "q4_k":
        return cols // QK_K * Q4_K_BLOCK_BYTES
    return cols // QK * (Q8_0_BLOCK_BYTES if fmt == "q8_0" else Q4_0_BLOCK_BYTES)


def hq_version() -> int:
    return int(lib().hq_version())


def hq_last_error() -> str:
    return lib().hq_last_error().decode()


def hq_matvec_q8_0(W, x, y, rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_q8_0(_addr(W), _addr(x), _addr(y), rows, cols, n_vec, _stream(stream)))


def hq_matvec_q4_0(W, x, y, rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_q4_0(_addr(W), _addr(x), _addr(y), rows, cols, n_vec, _stream(stream)))


def hq_matvec_q4_k(W, x, y, rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_q4_k(_addr(W), _addr(x), _addr(y), rows, cols, n_vec, _stream(stream)))


def hq_quantize_q4_k(W, out, rows: int, cols: int, stream=None) -> int:
    return _check(lib().hq_quantize_q4_k(_addr(W), _addr(out), rows, cols, _stream(stream)))


def hq_matvec_q8_0_lora(W, x, lora_A, lora_B, scale: float, rank: int, workspace, y, rows: int, cols: int,
                        n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_q8_0_lora(_addr(W), _addr(x), _addr(lora_A), _addr(lora_B), float(scale),
                                            int(rank), _addr(workspace), _addr(y), rows, cols, n_vec,
                                            _stream(stream)))


def hq_matvec_q4_0_lora(W, x, lora_A, lora_B, scale: float, rank: int, workspace, y, rows: int, cols: int,
                        n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_q4_0_lora(_addr(W), _addr(x), _addr(lora_A), _addr(lora_B), float(scale),
                                            int(rank), _addr(workspace), _addr(y), rows, cols, n_vec,
                                            _stream(stream)))


def hq_matvec_q8_0_lora_noalloc(W, x, lora_A, lora_B, scale: float, rank: int, y, rows: int, cols: int,
                                n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_q8_0_lora_noalloc(_addr(W), _addr(x), _addr(lora_A), _addr(lora_B),
                                                    float(scale), int(rank), _addr(y), rows, cols, n_vec,
                                                    _stream(stream)))


def hq_matvec_i8_requant(W, x, mult, shift, y, rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_matvec_i8_requant(_addr(W), _addr(x), _addr(mult), _addr(shift), _addr(y),
                                             rows, cols, n_vec, _stream(stream)))


def hq_moe_matvec_q8_0(W_bank, expert_ids, x, x_per_slot: int, y, n_experts: int, n_active: int,
                       rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_moe_matvec_q8_0(_addr(W_bank), _addr(expert_ids), _addr(x), int(x_per_slot),
                                           _addr(y), n_experts, n_active, rows, cols, n_vec,
                                           _stream(stream)))


def hq_moe_matvec_q8_0_swiglu(W_bank, expert_ids, x, x_per_slot: int, h, n_experts: int, n_active: int,
                              rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_moe_matvec_q8_0_swiglu(_addr(W_bank), _addr(expert_ids), _addr(x), int(x_per_slot),
                                                  _addr(h), n_experts, n_active, rows, cols, n_vec,
                                                  _stream(stream)))


def hq_moe_matvec_q8_0_combine(W_bank, expert_ids, x, x_per_slot: int, router_w, y, n_experts: int,
                               n_active: int, rows: int, cols: int, n_vec: int, stream=None) -> int:
    return _check(lib().hq_moe_matvec_q8_0_combine(_addr(W_bank), _addr(expert_ids), _addr(x), int(x_per_slot),
                                                   _addr(router_w), _addr(y), n_experts, n_active, rows, cols,
                                                   n_vec, _stream(stream)))


HQ_MOE_EPI_NONE, HQ_MOE_EPI_SWIGLU, HQ_MOE_EPI_COMBINE = 0, 1, 2
HQ_MOE_IDS_READY = 1


def hq_moe_matvec_q8_0_ex(W_bank, expert_ids, x, x_per_slot: int, router_w, y, n_experts: int, n_active: int,
                          rows: int, cols: int, n_vec: int, epilogue: int, flags: int, stream=None) -> int:
    return _check(lib().hq_moe_matvec_q8_0_ex(_addr(W_bank), _addr(expert_ids), _addr(x), int(x_per_slot),
                                              _addr(router_w), _addr(y), n_experts, n_active, rows, cols, n_vec,
                                              int(epilogue), int(flags), _stream(stream)))


def hq_quantize_q8_0(W, out, rows: int, cols: int, stream=None) -> int:
    return _check(lib().hq_quantize_q8_0(_addr(W), _addr(out), rows, cols, _stream(stream)))


def hq_quantize_q4_0(W, out, rows: int, cols: int, stream=None) -> int:
    return _check(lib().hq_quantize_q4_0(_addr(W), _addr(out), rows, cols, _stream(stream)))


def hq_quantize_i8_rows(W, Wq, scale, rows: int, cols: int, stream=None) -> int:
    return _check(lib().hq_quantize_i8_rows(_addr(W), _addr(Wq), _addr(scale), rows, cols, _stream(stream)))


def hq_requant_params(M, n: int, mult, shift) -> int:
    """HOST function: M float64, mult/shift int32 host arrays (numpy) of n elements."""
    return _check(lib().hq_requant_params(_addr(M), n, _addr(mult), _addr(shift)))


def hq_requant_i32_debug(acc, mult, shift, y, n: int, rows: int, stream=None) -> int:
    return _check(lib().hq_requant_i32_debug(_addr(acc), _addr(mult), _addr(shift), _addr(y), n, rows,
                                             _stream(stream)))


def hq_selftest_wait_timeout(cycles: int, stream=None) -> int:
    """Test-only: a bounded wait that nothing completes; sets the fault word."""
    return _check(lib().hq_selftest_wait_timeout(int(cycles), _stream(stream)))


def hq_device_fault() -> int:
    """Synchronize the device, then return and clear its fault word (0 = no fault)."""
    v = ctypes.c_uint32(0)
    st = lib().hq_device_fault(ctypes.byref(v))
    if st != HQ_OK and st != HQ_ERR_DEVICE:
        _check(st)
    return int(v.value)


PLAN_FIELDS = ("policy", "cons_warps", "tile_rows", "grid", "ksplit", "stages", "smem", "ctas_per_sm",
               "slots", "tiles")


def hq_debug_plan(fmt: int, n_vec: int, rows: int, cols: int, num_sms: int, smem_optin: int, regs: int) -> dict:
    """HOST function (test-only): the launch geometry the library would choose, as a dict."""
    out = (ctypes.c_int64 * len(PLAN_FIELDS))()
    _check(lib().hq_debug_plan(int(fmt), int(n_vec), int(rows), int(cols), int(num_sms), int(smem_optin),
                               int(regs), out, len(PLAN_FIELDS)))
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


def hq_launch_count() -> int:
    """Kernels the library has launched or captured so far in this process."""
    return int(lib().hq_launch_count())
