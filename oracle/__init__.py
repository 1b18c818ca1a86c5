"""CPU oracle for block-scaled FP4 (E2M1) quantization -- test infrastructure.

A plain, slow, single-threaded C implementation (``*.c`` beside this file),
compiled with ``-ffp-contract=off`` and no fast-math so that every fp32
operation is one correctly rounded IEEE operation.  Only the tests, the smoke
check and the CPU-baseline leg of ``bench.py`` may import this package; the
CUDA library never does, and the two share no code.

This module only marshals numpy arrays into the C functions; every step of
the arithmetic is in the C sources, each function citing the page it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_SOURCES = ["formats.c", "philox.c", "nvfp4.c", "mxfp4.c", "fp4quant.c", "layout.c", "arrays.c"]
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]

RTN, SR = 0, 1
TSCALE_GIVEN, TSCALE_COMPUTE = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, C11)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    deps = srcs + [os.path.join(_HERE, "fp4_oracle.h")]
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(d) for d in deps)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, *srcs, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_I32 = ctypes.c_int32
_F = ctypes.c_float

_SIGS = {
    "ora_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
    "ora_e2m1_rn": (ctypes.c_uint8, [_F]),
    "ora_e2m1_sr": (ctypes.c_uint8, [_F, ctypes.c_uint32]),
    "ora_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
    "ora_e4m3_rn_d": (ctypes.c_uint8, [ctypes.c_double]),
    "ora_ue8m0_value": (ctypes.c_double, [ctypes.c_uint8]),
    "ora_bf16_rn": (ctypes.c_uint16, [_F]),
    "ora_philox4x32_10": (None, [_P, _P, _P]),
    "ora_rng_word": (ctypes.c_uint32, [_U64, _U64, _U64]),
    "ora_nvfp4_amax": (_F, [_P, _P, _I64]),
    "ora_nvfp4_tensor_scale": (_F, [_F]),
    "ora_nvfp4_sanitize_scale": (_F, [_F]),
    "ora_nvfp4_quantize": (ctypes.c_int, [_P, _I64, _P, ctypes.c_int, _U64, _U64,
                                          ctypes.c_int, _P, _P, _P]),
    "ora_nvfp4_dequantize": (ctypes.c_int, [_P, _P, _F, _I64, _P]),
    "ora_nvfp4_qdq": (ctypes.c_int, [_P, _P, _F, _I64, _P, ctypes.c_int, _U64, _U64,
                                     ctypes.c_int, _P, _P, _P]),
    "ora_nvfp4_qdq_amax": (_F, [_P, _P, _F, _P, _I64]),
    "ora_nvfp4_blocks": (None, [_P, _I64, _I64, _F, ctypes.c_int, _U64, _U64, _P, _P, _P]),
    "ora_mxfp4_quantize": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "ora_fp4_to_fp8_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "ora_fp8_to_fp4_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _P, _P]),
    "ora_mxfp4_dequantize": (ctypes.c_int, [_P, _P, _I64, _I64, _P]),
    "ora_fp4_scaled_quantize": (ctypes.c_int, [_P, _I64, ctypes.c_float, _P]),
    "ora_fp4_scaled_dequantize": (ctypes.c_int, [_P, _I64, ctypes.c_float, _P]),
    "ora_fp4_to_fp8_col": (ctypes.c_int, [_P, _P, _I64, _P, _I32, _P, _P]),
    "ora_fp4_to_fp8_col_segment": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P, _P]),
    "ora_blocked_scales_size": (_I64, [_I64, _I64]),
    "ora_scales_to_blocked": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "ora_scales_from_blocked": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "ora_wht_norm": (_F, [ctypes.c_int]),
    "ora_wht": (None, [_P, ctypes.c_int]),
    "ora_fp4quant_encode": (ctypes.c_int, [_P, _I64, _I64, ctypes.c_int, _P, _P, _P]),
    "ora_fp4quant_decode": (ctypes.c_int, [_P, _P, _P, _I64, _I64, ctypes.c_int, _P]),
    "ora_e2m1_rn_array": (None, [_P, _I64, _P]),
    "ora_e2m1_sr_array": (None, [_P, _P, _I64, _P]),
    "ora_e4m3_rn_array": (None, [_P, _I64, _P]),
    "ora_bf16_rn_array": (None, [_P, _I64, _P]),
    "ora_rng_word_array": (None, [_U64, _U64, _P, _I64, _P]),
}


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            handle = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: bad argument")


# ------------------------------------------------------------------ formats

def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def e2m1_value(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    table = np.array([L.ora_e2m1_value(i) for i in range(16)], dtype=np.float64)
    return table[c & 0xF]


def e2m1_rn(a) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint8)
    lib().ora_e2m1_rn_array(_ptr(a), a.size, _ptr(out))
    return out


def e2m1_sr(a, words) -> np.ndarray:
    a = _c(a, np.float32)
    w = _c(np.broadcast_to(words, a.shape), np.uint32)
    out = np.empty(a.shape, np.uint8)
    lib().ora_e2m1_sr_array(_ptr(a), _ptr(w), a.size, _ptr(out))
    return out


def e4m3_value(b) -> np.ndarray:
    L = lib()
    table = np.array([L.ora_e4m3_value(i) for i in range(256)], dtype=np.float64)
    return table[np.asarray(b, dtype=np.uint8)]


def e4m3_rn(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    lib().ora_e4m3_rn_array(_ptr(x), x.size, _ptr(out))
    return out


def ue8m0_value(b) -> np.ndarray:
    L = lib()
    table = np.array([L.ora_ue8m0_value(i) for i in range(256)], dtype=np.float64)
    return table[np.asarray(b, dtype=np.uint8)]


def bf16_rn(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().ora_bf16_rn_array(_ptr(x), x.size, _ptr(out))
    return out


# ------------------------------------------------------------------- Philox

def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.empty(4, np.uint32)
    lib().ora_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def rng_words(seed: int, step: int, g) -> np.ndarray:
    g = _c(g, np.uint64)
    out = np.empty(g.shape, np.uint32)
    lib().ora_rng_word_array(seed, step, _ptr(g), g.size, _ptr(out))
    return out


# -------------------------------------------------------------------- NVFP4

def nvfp4_amax(x, residual=None) -> float:
    x = _c(x, np.float32).ravel()
    r = None if residual is None else _c(residual, np.float32).ravel()
    return float(lib().ora_nvfp4_amax(_ptr(x), _ptr(r), x.size))


def nvfp4_tensor_scale(amax: float) -> float:
    return float(lib().ora_nvfp4_tensor_scale(amax))


def nvfp4_sanitize_scale(s: float) -> float:
    return float(lib().ora_nvfp4_sanitize_scale(s))


def nvfp4_quantize(x, residual=None, rounding=RTN, seed=0, step=0,
                   tscale_mode=TSCALE_COMPUTE, tensor_scale=1.0):
    """Returns (packed uint8[n/2], scales uint8[n/16], tensor_scale float).

    ``residual`` (float32, contiguous, writable) is updated in place."""
    x = _c(x, np.float32).ravel()
    n = x.size
    if residual is not None:
        assert residual.dtype == np.float32 and residual.flags.c_contiguous
    packed = np.empty(n // 2, np.uint8)
    scales = np.empty(n // 16, np.uint8)
    ts = np.array([tensor_scale], np.float32)
    rc = lib().ora_nvfp4_quantize(_ptr(x), n, _ptr(residual), rounding, seed, step,
                                  tscale_mode, _ptr(ts), _ptr(packed), _ptr(scales))
    _check(rc, "nvfp4_quantize")
    return packed, scales, float(ts[0])


def nvfp4_blocks(v, b0: int, s_t: float, rounding=RTN, seed=0, step=0):
    """Quantize consecutive blocks starting at block index b0 with tensor scale
    s_t; ``v`` already includes any residual.  Returns (packed, scales, q)."""
    v = _c(v, np.float32).ravel()
    nb = v.size // 16
    packed = np.empty(nb * 8, np.uint8)
    scales = np.empty(nb, np.uint8)
    q = np.empty(nb * 16, np.float32)
    lib().ora_nvfp4_blocks(_ptr(v), b0, nb, s_t, rounding, seed, step, _ptr(packed),
                           _ptr(scales), _ptr(q))
    return packed, scales, q


def nvfp4_dequantize(packed, scales, tensor_scale: float, n: int) -> np.ndarray:
    p = _c(packed, np.uint8)
    s = _c(scales, np.uint8)
    y = np.empty(n, np.float32)
    _check(lib().ora_nvfp4_dequantize(_ptr(p), _ptr(s), tensor_scale, n, _ptr(y)),
           "nvfp4_dequantize")
    return y


def nvfp4_qdq(w_bits, g=None, lr=0.0, residual=None, rounding=RTN, seed=0, step=0,
              tscale_mode=TSCALE_COMPUTE, tensor_scale=1.0):
    """One fused step on a bf16 weight.  ``w_bits`` (uint16) and ``residual``
    (float32) are updated in place.  Returns (packed, scales, tensor_scale)."""
    assert w_bits.dtype == np.uint16 and w_bits.flags.c_contiguous
    n = w_bits.size
    gg = None if g is None else _c(g, np.float32).ravel()
    if residual is not None:
        assert residual.dtype == np.float32 and residual.flags.c_contiguous
    packed = np.empty(n // 2, np.uint8)
    scales = np.empty(n // 16, np.uint8)
    ts = np.array([tensor_scale], np.float32)
    rc = lib().ora_nvfp4_qdq(_ptr(w_bits), _ptr(gg), lr, n, _ptr(residual), rounding,
                             seed, step, tscale_mode, _ptr(ts), _ptr(packed),
                             _ptr(scales))
    _check(rc, "nvfp4_qdq")
    return packed, scales, float(ts[0])


def nvfp4_qdq_amax(w_bits, g=None, lr=0.0, residual=None) -> float:
    w = _c(w_bits, np.uint16).ravel()
    gg = None if g is None else _c(g, np.float32).ravel()
    r = None if residual is None else _c(residual, np.float32).ravel()
    return float(lib().ora_nvfp4_qdq_amax(_ptr(w), _ptr(gg), lr, _ptr(r), w.size))


# -------------------------------------------------------------------- MXFP4

def mxfp4_quantize(x):
    x = _c(x, np.float32)
    rows, cols = x.shape
    packed = np.empty((rows, cols // 2), np.uint8)
    scales = np.empty((rows, cols // 32), np.uint8)
    _check(lib().ora_mxfp4_quantize(_ptr(x), rows, cols, _ptr(packed), _ptr(scales)),
           "mxfp4_quantize")
    return packed, scales


def fp4_to_fp8_row(packed, scales):
    p = _c(packed, np.uint8)
    s = _c(scales, np.uint8)
    rows, half = p.shape
    cols = half * 2
    fp8 = np.empty((rows, cols), np.uint8)
    fsc = np.empty((rows, cols // 128), np.float32)
    _check(lib().ora_fp4_to_fp8_rows(_ptr(p), _ptr(s), rows, cols, _ptr(fp8), _ptr(fsc)),
           "fp4_to_fp8_row")
    return fp8, fsc


def fp8_to_fp4_row(fp8, fp8_scales):
    """Backward-path FP4: E4M3 [rows, cols] with fp32 scales [rows, cols/128]
    -> MXFP4 (packed [rows, cols/2], UE8M0 [rows, cols/32])."""
    f = _c(fp8, np.uint8)
    s = _c(fp8_scales, np.float32)
    rows, cols = f.shape
    packed = np.empty((rows, cols // 2), np.uint8)
    scales = np.empty((rows, cols // 32), np.uint8)
    _check(lib().ora_fp8_to_fp4_rows(_ptr(f), _ptr(s), rows, cols, _ptr(packed), _ptr(scales)),
           "fp8_to_fp4_row")
    return packed, scales


def mxfp4_dequantize(packed, scales):
    """MXFP4 -> fp32 [rows, cols]."""
    p = _c(packed, np.uint8)
    s = _c(scales, np.uint8)
    rows, half = p.shape
    y = np.empty((rows, 2 * half), np.float32)
    _check(lib().ora_mxfp4_dequantize(_ptr(p), _ptr(s), rows, 2 * half, _ptr(y)),
           "mxfp4_dequantize")
    return y


def fp4_scaled_quantize(x, scale: float):
    """One fp32 scale for the whole (flat) tensor: packed codes RN_e2m1(RN(x/s))."""
    x = _c(np.asarray(x, np.float32).reshape(-1), np.float32)
    packed = np.empty(x.size // 2, np.uint8)
    _check(lib().ora_fp4_scaled_quantize(_ptr(x), x.size, float(np.float32(scale)), _ptr(packed)),
           "fp4_scaled_quantize")
    return packed


def fp4_scaled_dequantize(packed, n: int, scale: float):
    p = _c(np.asarray(packed, np.uint8).reshape(-1), np.uint8)
    y = np.empty(n, np.float32)
    _check(lib().ora_fp4_scaled_dequantize(_ptr(p), n, float(np.float32(scale)), _ptr(y)),
           "fp4_scaled_dequantize")
    return y


def blocked_scales_size(rows: int, cols: int) -> int:
    return int(lib().ora_blocked_scales_size(rows, cols))


def scales_to_blocked(scales, rows: int, cols: int) -> np.ndarray:
    """[rows, cols] uint8 scales -> the blocked (swizzled) uint8 buffer."""
    s = _c(scales, np.uint8).reshape(-1)
    assert s.size == rows * cols
    out = np.full(blocked_scales_size(rows, cols), 0xA5, dtype=np.uint8)
    _check(lib().ora_scales_to_blocked(_ptr(s), rows, cols, _ptr(out)), "scales_to_blocked")
    return out


def scales_from_blocked(blocked, rows: int, cols: int) -> np.ndarray:
    """The inverse of scales_to_blocked: [rows, cols] uint8."""
    b = _c(blocked, np.uint8).reshape(-1)
    assert b.size == blocked_scales_size(rows, cols)
    out = np.empty(rows * cols, dtype=np.uint8)
    _check(lib().ora_scales_from_blocked(_ptr(b), rows, cols, _ptr(out)), "scales_from_blocked")
    return out.reshape(rows, cols)


def seg_scale_offsets(row_off) -> np.ndarray:
    row_off = np.asarray(row_off, dtype=np.int64)
    nb = (np.diff(row_off) + 127) // 128
    return np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)


def fp4_to_fp8_col(packed, scales, row_off):
    """Returns (fp8_t flat uint8[cols * R], scales flat float32[cols * nb_total])."""
    p = _c(packed, np.uint8)
    s = _c(scales, np.uint8)
    off = _c(row_off, np.int64)
    cols = p.shape[1] * 2
    total = int(off[-1])
    so = seg_scale_offsets(off)
    out = np.empty(cols * total, np.uint8)
    osc = np.empty(cols * int(so[-1]), np.float32)
    _check(lib().ora_fp4_to_fp8_col(_ptr(p), _ptr(s), cols, _ptr(off), off.size - 1,
                                    _ptr(out), _ptr(osc)), "fp4_to_fp8_col")
    return out, osc


def fp4_to_fp8_col_segment(packed, scales, row0: int, n_e: int):
    p = _c(packed, np.uint8)
    s = _c(scales, np.uint8)
    cols = p.shape[1] * 2
    nb = (n_e + 127) // 128
    out = np.empty((cols, n_e), np.uint8)
    osc = np.empty((cols, nb), np.float32)
    _check(lib().ora_fp4_to_fp8_col_segment(_ptr(p), _ptr(s), cols, row0, n_e, _ptr(out),
                                            _ptr(osc)), "fp4_to_fp8_col_segment")
    return out, osc


# ----------------------------------------------------------------- FP4Quant

def wht_norm(group: int) -> float:
    return float(lib().ora_wht_norm(group))


def wht(y, group: int) -> np.ndarray:
    y = np.array(y, dtype=np.float32).ravel()
    assert y.size == group
    lib().ora_wht(_ptr(y), group)
    return y


def fp4quant_encode(x, group: int):
    x = _c(x, np.float32)
    rows, cols = x.shape
    packed = np.empty((rows, cols // 2), np.uint8)
    s1 = np.empty((rows, cols // group), np.float32)
    s2 = np.empty((rows, cols // group), np.float32)
    _check(lib().ora_fp4quant_encode(_ptr(x), rows, cols, group, _ptr(packed), _ptr(s1),
                                     _ptr(s2)), "fp4quant_encode")
    return packed, s1, s2


def fp4quant_decode(packed, s1, s2, group: int) -> np.ndarray:
    p = _c(packed, np.uint8)
    a = _c(s1, np.float32)
    b = _c(s2, np.float32)
    rows = p.shape[0]
    cols = p.shape[1] * 2
    x = np.empty((rows, cols), np.float32)
    _check(lib().ora_fp4quant_decode(_ptr(p), _ptr(a), _ptr(b), rows, cols, group,
                                     _ptr(x)), "fp4quant_decode")
    return x
