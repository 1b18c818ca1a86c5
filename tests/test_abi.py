"""The C-ABI library loads and exports every function include/fp4codec.h
declares; argument checks return their status before anything is enqueued
(CPU only: every call here fails validation, so no CUDA call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4codec.h")


@pytest.fixture(scope="module")
def L():
    from block_scaled_fp4_e2m1_gb300 import build as b
    b.build()
    from block_scaled_fp4_e2m1_gb300 import _lib
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s*([a-z_0-9]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["nvfp4_amax", "nvfp4_quantize", "nvfp4_dequantize", "nvfp4_qdq_amax",
                 "nvfp4_qdq", "mxfp4_quantize", "fp4_to_fp8_row", "fp4_to_fp8_col",
                 "fp4_to_fp8_col_runs",
                 "fp4_seg_scale_offsets", "fp4quant_encode", "fp4quant_decode",
                 "fp4_status_string", "fp4_abi_version", "fp4_kernel_launches",
                 "fp4_wait_timeouts", "fp4_test_encode_wait_timeout",
                 "fp4_blocked_scales_size", "fp4_scales_to_blocked", "fp4_scales_from_blocked",
                 "nvfp4_quantize_blocked"]:
        assert want in names, want


def test_library_exports_every_declared_symbol(L):
    from block_scaled_fp4_e2m1_gb300 import _lib
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in _lib.SIGNATURES, name


def test_version_and_status_strings(L):
    assert L.fp4_abi_version() == 1
    for s in range(8):
        assert L.fp4_status_string(s)
    assert L.fp4_status_string(0) == b"ok"
    assert L.fp4_status_string(99) == b"unknown status"


def test_seg_scale_offsets_host_helper(L):
    import numpy as np
    off = np.array([0, 0, 1, 128, 129, 400, 400], np.int64)
    out = np.zeros(7, np.int64)
    assert L.fp4_seg_scale_offsets(off.ctypes.data, 6, out.ctypes.data) == 0
    assert list(out) == [0, 0, 1, 2, 3, 6, 6]
    bad = np.array([0, 5, 3], np.int64)
    out2 = np.full(3, -7, np.int64)
    assert L.fp4_seg_scale_offsets(bad.ctypes.data, 2, out2.ctypes.data) == 3
    assert L.fp4_seg_scale_offsets(None, 2, out2.ctypes.data) == 1


# Fake device addresses: never dereferenced, because every call below fails
# a host-side check first.
A = 0x100000          # 1 MiB: aligned to everything
MIS = A + 8           # 8-byte aligned only


def test_nvfp4_argument_checks(L):
    q = L.nvfp4_quantize
    ok = dict(x=A, dtype=1, n=64, res=None, rnd=0, seed=0, step=0, mode=0, ts=A, ws=A, pk=A, sc=A)

    def call(**kw):
        a = dict(ok, **kw)
        return q(a["x"], a["dtype"], a["n"], a["res"], a["rnd"], a["seed"], a["step"], a["mode"],
                 a["ts"], a["ws"], a["pk"], a["sc"], None)

    assert call(n=15) == 3            # FP4_ERR_SHAPE: n % 16
    assert call(n=-16) == 3
    assert call(dtype=7) == 4         # FP4_ERR_DTYPE
    assert call(rnd=2) == 5           # FP4_ERR_ARG
    assert call(mode=3) == 5
    assert call(ts=None) == 1         # FP4_ERR_NULL
    assert call(mode=1, ws=None) == 1
    assert call(x=None) == 1
    assert call(x=MIS) == 2           # FP4_ERR_ALIGN: x needs 32 B
    assert call(res=MIS) == 2
    assert call(pk=A + 4) == 2
    d = L.nvfp4_dequantize
    assert d(A, A, None, 17, A, 0, None) == 3
    assert d(A, A, None, 16, A, 5, None) == 4
    assert d(A, A, None, 16, MIS, 0, None) == 2
    assert d(None, A, None, 16, A, 0, None) == 1
    assert L.nvfp4_amax(A, 1, 16, None, None, None) == 1
    assert L.nvfp4_amax(A, 1, 8, None, A, None) == 3
    qd = L.nvfp4_qdq
    assert qd(A, None, 0.0, 32, None, 0, 0, 0, 0, A, A, A, None, None) == 1   # packed w/o scales
    assert qd(A, None, 0.0, 31, None, 0, 0, 0, 0, A, A, None, None, None) == 3
    assert qd(MIS, None, 0.0, 32, None, 0, 0, 0, 0, A, A, None, None, None) == 2
    assert L.nvfp4_qdq_amax(A, A, 0.0, None, 32, None, None) == 1


def test_mx_fp8_fp4quant_argument_checks(L):
    assert L.mxfp4_quantize(A, 1, 4, 48, A, A, None) == 3        # cols % 32
    assert L.mxfp4_quantize(A, 2, 4, 64, A, A, None) == 4
    assert L.mxfp4_quantize(MIS, 1, 4, 64, A, A, None) == 2
    assert L.fp4_to_fp8_row(A, A, 4, 96, A, A, None) == 3        # cols % 128
    assert L.fp4_to_fp8_row(A, A + 1, 4, 128, A, A, None) == 2
    assert L.fp4_to_fp8_row(None, A, 4, 128, A, A, None) == 1
    assert L.fp8_to_fp4_row(A, A, 4, 96, A, A, None) == 3       # cols % 128
    assert L.fp8_to_fp4_row(MIS, A, 4, 128, A, A, None) == 2     # fp8 needs 32 B
    assert L.fp8_to_fp4_row(A, None, 4, 128, A, A, None) == 1
    assert L.mxfp4_dequantize(A, A, 4, 48, A, 1, None) == 3      # cols % 32
    assert L.mxfp4_dequantize(A, A, 4, 64, A, 7, None) == 4
    assert L.mxfp4_dequantize(A, A, 4, 64, MIS, 1, None) == 2
    assert L.mxfp4_dequantize(A, A, 4, 64, None, 1, None) == 1
    assert L.fp4_scaled_quantize(A, 1, 24, 1.0, A, None) == 3      # n % 16
    assert L.fp4_scaled_quantize(A, 1, 32, 0.0, A, None) == 5      # scale > 0
    assert L.fp4_scaled_quantize(A, 1, 32, float("inf"), A, None) == 5
    assert L.fp4_scaled_quantize(MIS, 1, 32, 1.0, A, None) == 2
    assert L.fp4_scaled_dequantize(A, 32, 1.0, None, 1, None) == 1
    assert L.fp4_scaled_dequantize(A, 32, 1.0, A, 9, None) == 4
    col = L.fp4_to_fp8_col
    assert col(A, A, 96, A, A, 2, 10, 2, A, A, None) == 3
    assert col(A, A, 128, None, A, 2, 10, 2, A, A, None) == 1
    assert col(A, A, 128, A, A, 2, 10, 5, A, A, None) == 3       # too many blocks
    assert col(A, A, 128, A, A, 2, 1 << 40, 1 << 31, A, A, None) == 3  # 2^31 blocks
    assert col(A, A, 128, A + 4, A, 2, 10, 2, A, A, None) == 2
    hook = L.fp4_test_encode_wait_timeout
    assert hook(A, 2, 192, A, A, A, None) == 3                   # cols % 128
    assert hook(A, 1 << 20, 128, A, A, A, None) == 3             # above 2^24 elements
    assert hook(A, 2, 256, None, A, A, None) == 1
    assert hook(MIS, 2, 256, A, A, A, None) == 2
    runs = L.fp4_to_fp8_col_runs
    assert runs(A, A, 128, A, A, 2, 10, 2, -1, A, A, None) == 3      # run_blocks < 0
    assert runs(A, A, 128, A, A, 2, 10, 2, (1 << 20) + 1, A, A, None) == 3
    assert runs(A, A, 96, A, A, 2, 10, 2, 8, A, A, None) == 3
    assert runs(A, A, 128, A + 4, A, 2, 10, 2, 8, A, A, None) == 2
    enc = L.fp4quant_encode
    assert enc(A, 1, 2, 128, 32, A, A, A, None) == 5             # group
    assert enc(A, 1, 2, 96, 64, A, A, A, None) == 3              # cols % group
    assert enc(A, 1, 2, 128, 64, A, None, A, None) == 1
    assert enc(MIS, 1, 2, 128, 64, A, A, A, None) == 2
    assert enc(A, 1, 1 << 34, 1 << 7, 64, A, A, A, None) == 3    # above 2^40 elements
    dec = L.fp4quant_decode
    assert dec(A, A, A, 2, 128, 512, A, 1, None) == 5
    assert dec(A, A, A, 2, 128, 64, A, 9, None) == 4
    assert dec(A, A, A, 1 << 34, 1 << 7, 64, A, 1, None) == 3    # above 2^40 elements


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from block_scaled_fp4_e2m1_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_batch_plan_host_helper(L):
    import numpy as np
    desc = np.dtype([("x", "<u8"), ("packed", "<u8"), ("scales", "<u8"), ("y", "<u8"),
                     ("n", "<i8"), ("chunk_start", "<i8")])
    assert desc.itemsize == 48
    h = np.zeros(4, desc)
    h["x"] = A
    h["packed"] = A
    h["scales"] = A
    h["n"] = [16 * 256 * 3 + 16, 0, 16, 16 * 256]
    total = ctypes.c_int64(-1)
    assert L.fp4_batch_plan(h.ctypes.data, 4, ctypes.addressof(total)) == 0
    assert list(h["chunk_start"]) == [0, 4, 4, 5] and total.value == 6
    h["n"][2] = 8
    assert L.fp4_batch_plan(h.ctypes.data, 4, ctypes.addressof(total)) == 3
    h["n"][2] = 16
    h["scales"][1] = A + 1
    assert L.fp4_batch_plan(h.ctypes.data, 4, ctypes.addressof(total)) == 2
    assert L.fp4_batch_plan(None, 4, ctypes.addressof(total)) == 1
    # batched entry points: checks before anything is enqueued
    assert L.nvfp4_amax_batched(A, 2, 3, 7, A, None) == 4
    assert L.nvfp4_amax_batched(A, 2, 3, 1, None, None) == 1
    assert L.nvfp4_amax_batched(A + 4, 2, 3, 1, A, None) == 2
    assert L.nvfp4_amax_batched(A, -1, 3, 1, A, None) == 3
    assert L.nvfp4_quantize_batched(A, 2, 3, 1, 5, 0, 0, 1, A, A, None) == 5
    assert L.nvfp4_quantize_batched(A, 2, 3, 1, 0, 0, 0, 1, A, None, None) == 1
    assert L.nvfp4_quantize_batched(A, 2, 3, 1, 0, 0, 0, 0, None, None, None) == 1
    assert L.nvfp4_dequantize_batched(A, 2, 3, A + 2, 0, None) == 2
    assert L.nvfp4_dequantize_batched(A, 2, 3, None, 3, None) == 4


def test_blocked_scale_layout_host_checks(L):
    size = L.fp4_blocked_scales_size
    assert size(0, 0) == 0
    assert size(1, 1) == 512
    assert size(129, 5) == 256 * 8
    assert size(4096, 256) == 4096 * 256
    assert size(-1, 4) == -1 and size(4, -1) == -1
    assert size(1 << 40, 1) == -1
    assert size(1 << 30, 1 << 20) == -1                        # > 2^44 padded scales
    to, frm = L.fp4_scales_to_blocked, L.fp4_scales_from_blocked
    assert to(A, -1, 4, A, None) == 3
    assert to(None, 4, 4, A, None) == 1
    assert to(A, 4, 4, A + 4, None) == 2                         # blocked needs 16 B
    assert frm(A, 4, 4, None, None) == 1
    assert frm(MIS, 4, 4, A, None) == 2
    assert to(None, 0, 7, None, None) == 0                       # empty: nothing to do
    qb = L.nvfp4_quantize_blocked
    ok = dict(x=A, dtype=1, rows=4, k=64, res=None, rnd=0, seed=0, step=0, mode=0, ts=A, ws=A,
              pk=A, sc=A)

    def call(**kw):
        a = dict(ok, **kw)
        return qb(a["x"], a["dtype"], a["rows"], a["k"], a["res"], a["rnd"], a["seed"], a["step"],
                  a["mode"], a["ts"], a["ws"], a["pk"], a["sc"], None)

    assert call(k=24) == 3            # k % 16
    assert call(rows=-1) == 3
    assert call(rows=1 << 30, k=1 << 16) == 3
    assert call(dtype=3) == 4
    assert call(rnd=9) == 5
    assert call(sc=None) == 1
    assert call(mode=2, ws=None) == 1
    assert call(x=MIS) == 2
    assert call(pk=A + 8) == 2


def test_batch_plan_blocked_host_helper(L):
    import numpy as np
    desc = np.dtype([("x", "<u8"), ("packed", "<u8"), ("scales", "<u8"), ("y", "<u8"),
                     ("n", "<i8"), ("chunk_start", "<i8")])
    d = np.zeros(3, desc)
    d["n"] = [64, 4096 * 16, 0]
    total = ctypes.c_int64(-1)
    ok = np.array([32, 4096, 16], np.int64)
    assert L.fp4_batch_plan_blocked(d.ctypes.data, ok.ctypes.data, 3, ctypes.addressof(total)) == 0
    assert total.value == 1 + 16 + 0   # chunks of 256 blocks
    for bad in ([48, 4096, 16], [24, 4096, 16], [32, 4096, 0], [32, 4096 * 3, 16]):
        b = np.array(bad, np.int64)
        assert L.fp4_batch_plan_blocked(d.ctypes.data, b.ctypes.data, 3,
                                        ctypes.addressof(total)) == 3, bad
    assert L.fp4_batch_plan_blocked(d.ctypes.data, None, 3, ctypes.addressof(total)) == 1
    assert L.nvfp4_quantize_batched_blocked(A, None, 3, 2, 1, 0, 0, 0, 1, A, A, None) == 1
    assert L.nvfp4_quantize_batched_blocked(A, A + 4, 3, 2, 1, 0, 0, 0, 1, A, A, None) == 2
