"""ctypes loader for ``libfp4codec.so`` (the C ABI in include/fp4codec.h).

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``python -m block_scaled_fp4_e2m1_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp4codec.so")

P = ctypes.c_void_p
I64 = ctypes.c_int64
U64 = ctypes.c_uint64
I32 = ctypes.c_int32
INT = ctypes.c_int
F32 = ctypes.c_float

# name -> (restype, argtypes), in the order of include/fp4codec.h
SIGNATURES = {
    "fp4_status_string": (ctypes.c_char_p, [INT]),
    "fp4_abi_version": (INT, []),
    "fp4_kernel_launches": (U64, []),
    "fp4_wait_timeouts": (U64, []),
    "fp4_test_encode_wait_timeout": (INT, [P, I64, I64, P, P, P, P]),
    "nvfp4_amax": (INT, [P, INT, I64, P, P, P]),
    "nvfp4_quantize": (INT, [P, INT, I64, P, INT, U64, U64, INT, P, P, P, P, P]),
    "nvfp4_dequantize": (INT, [P, P, P, I64, P, INT, P]),
    "nvfp4_qdq_amax": (INT, [P, P, F32, P, I64, P, P]),
    "nvfp4_qdq": (INT, [P, P, F32, I64, P, INT, U64, U64, INT, P, P, P, P, P]),
    "nvfp4_quantize_noalloc": (INT, [P, INT, I64, P, INT, U64, U64, P, P, P, P]),
    "fp4_blocked_scales_size": (I64, [I64, I64]),
    "fp4_scales_to_blocked": (INT, [P, I64, I64, P, P]),
    "fp4_scales_from_blocked": (INT, [P, I64, I64, P, P]),
    "nvfp4_quantize_blocked": (INT, [P, INT, I64, I64, P, INT, U64, U64, INT, P, P, P, P, P]),
    "fp4_batch_plan": (INT, [P, I32, P]),
    "nvfp4_amax_batched": (INT, [P, I32, I64, INT, P, P]),
    "nvfp4_quantize_batched": (INT, [P, I32, I64, INT, INT, U64, U64, INT, P, P, P]),
    "nvfp4_quantize_batched_blocked": (INT, [P, P, I32, I64, INT, INT, U64, U64, INT, P, P, P]),
    "fp4_batch_plan_blocked": (INT, [P, P, I32, P]),
    "nvfp4_dequantize_batched": (INT, [P, I32, I64, P, INT, P]),
    "mxfp4_quantize": (INT, [P, INT, I64, I64, P, P, P]),
    "fp4_to_fp8_row": (INT, [P, P, I64, I64, P, P, P]),
    "fp8_to_fp4_row": (INT, [P, P, I64, I64, P, P, P]),
    "mxfp4_dequantize": (INT, [P, P, I64, I64, P, INT, P]),
    "fp4_scaled_quantize": (INT, [P, INT, I64, ctypes.c_float, P, P]),
    "fp4_scaled_dequantize": (INT, [P, I64, ctypes.c_float, P, INT, P]),
    "fp4_scaled_quantize_amax": (INT, [P, INT, I64, P, P, P, P]),
    "fp4_scaled_dequantize_dev": (INT, [P, I64, P, P, INT, P]),
    "fp4_to_fp8_col": (INT, [P, P, I64, P, P, I32, I64, I64, P, P, P]),
    "fp4_to_fp8_col_runs": (INT, [P, P, I64, P, P, I32, I64, I64, I32, P, P, P]),
    "fp4_seg_scale_offsets": (INT, [P, I32, P]),
    "fp4quant_encode": (INT, [P, INT, I64, I64, INT, P, P, P, P]),
    "fp4quant_decode": (INT, [P, P, P, I64, I64, INT, P, INT, P]),
}

# status codes (fp4_status)
OK, ERR_NULL, ERR_ALIGN, ERR_SHAPE, ERR_DTYPE, ERR_ARG, ERR_CUDA, ERR_INTERNAL = range(8)
F32_DTYPE, BF16_DTYPE = 0, 1
RTN, SR = 0, 1
TSCALE_GIVEN, TSCALE_COMPUTE, TSCALE_FROM_AMAX = 0, 1, 2

_lock = threading.Lock()
_lib = None


class Fp4Error(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {message} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -m block_scaled_fp4_e2m1_gb300.build` "
                    "(nvcc for sm_103a)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(fn: str, status: int) -> None:
    if status != OK:
        msg = lib().fp4_status_string(status).decode()
        raise Fp4Error(fn, status, msg)


def call(fn: str, *args) -> None:
    check(fn, getattr(lib(), fn)(*args))
