"""The Python binding checks every caller-supplied tensor before it hands a
raw pointer to the library: a buffer that is too short, of the wrong dtype,
on another device or not contiguous raises ValueError and nothing is
launched.  CPU only: the device test is replaced by a stand-in that accepts
CPU tensors, and the library call by a recorder, so no kernel can run."""
import pytest
import torch

from block_scaled_fp4_e2m1_gb300 import codec
from block_scaled_fp4_e2m1_gb300.error_feedback import ErrorFeedback

F32, BF16, U8 = torch.float32, torch.bfloat16, torch.uint8


# host-only helpers of the library (no device work): these still run
HOST_ONLY = ("fp4_seg_scale_offsets", "fp4_batch_plan", "fp4_batch_plan_blocked")


@pytest.fixture
def calls(monkeypatch):
    from block_scaled_fp4_e2m1_gb300 import build
    build.build()
    seen = []
    real = codec.call

    def record(fn, *a):
        if fn in HOST_ONLY:
            return real(fn, *a)
        seen.append(fn)

    monkeypatch.setattr(codec, "_is_device_tensor", lambda t: True)
    monkeypatch.setattr(codec, "_stream", lambda dev: 0)
    monkeypatch.setattr(codec, "call", record)
    return seen


def z(n, dt):
    return torch.zeros(n, dtype=dt)


N = 256


def _raises(calls, fn, *a, **kw):
    with pytest.raises(ValueError):
        fn(*a, **kw)
    assert calls == [], "a call was made after a failed check"


def test_well_formed_calls_reach_the_library(calls):
    x = z(N, BF16)
    codec.nvfp4_amax(x, residual=z(N, F32), amax_ws=z(1, F32))
    codec.nvfp4_quantize(x, residual=z(N, F32), packed=z(N // 2, U8), scales=z(N // 16, U8))
    codec.nvfp4_dequantize(z(N // 2, U8), z(N // 16, U8), z(1, F32), (N,), BF16, out=z(N, BF16))
    codec.nvfp4_qdq(x, z(N, F32), 1e-3, z(N, F32))
    codec.nvfp4_quantize_noalloc(x)
    codec.mxfp4_quantize(z(N, BF16).view(2, 128))
    codec.fp4quant_encode(z(N, BF16).view(1, 256), 128)
    assert calls == ["nvfp4_amax", "nvfp4_quantize", "nvfp4_dequantize", "nvfp4_qdq",
                     "nvfp4_quantize_noalloc", "mxfp4_quantize", "fp4quant_encode"]


@pytest.mark.parametrize("kw", [
    dict(residual=z(N - 16, F32)),            # too short
    dict(residual=z(N, BF16)),                # wrong dtype
    dict(residual=z(2 * N, F32)[::2]),        # not contiguous
    dict(packed=z(N // 2 - 1, U8)),
    dict(packed=z(N // 2, torch.int8)),
    dict(scales=z(N // 16 - 1, U8)),
    dict(tensor_scale=z(2, F32)),
    dict(amax_ws=z(1, torch.float64)),
    dict(rounding="nearest"),
    dict(tscale="auto"),
])
def test_nvfp4_quantize_rejects(calls, kw):
    _raises(calls, codec.nvfp4_quantize, z(N, BF16), **kw)


def test_buffer_on_another_device_is_rejected(calls):
    meta = torch.empty(N, dtype=F32, device="meta")
    _raises(calls, codec.nvfp4_quantize, z(N, BF16), residual=meta)
    _raises(calls, codec.nvfp4_amax, z(N, F32), residual=meta)


@pytest.mark.parametrize("kw", [
    dict(residual=z(N // 2, F32)), dict(amax_ws=z(4, F32)), dict(amax_ws=z(1, BF16))])
def test_nvfp4_amax_rejects(calls, kw):
    _raises(calls, codec.nvfp4_amax, z(N, F32), **kw)


@pytest.mark.parametrize("args,kw", [
    ((z(N // 2 - 8, U8), z(N // 16, U8), None, (N,)), {}),             # short codes
    ((z(N // 2, U8), z(N // 16 - 1, U8), None, (N,)), {}),             # short scales
    ((z(N // 2, U8), z(N // 16, U8), z(1, BF16), (N,)), {}),           # bf16 tensor scale
    ((z(N // 2, U8), z(N // 16, U8), None, (N,)), dict(out=z(N - 1, F32))),
    ((z(N // 2, U8), z(N // 16, U8), None, (N,)), dict(out=z(N, BF16))),  # out dtype mismatch
    ((z(N // 2, U8), z(N // 16, U8), None, (N,)), dict(out_dtype=torch.float16)),
])
def test_nvfp4_dequantize_rejects(calls, args, kw):
    _raises(calls, codec.nvfp4_dequantize, *args, **kw)


@pytest.mark.parametrize("g,r,w", [
    (z(N - 16, F32), None, z(N, BF16)),        # short gradient
    (z(N, BF16), None, z(N, BF16)),            # bf16 gradient
    (None, z(N - 16, F32), z(N, BF16)),        # short residual
    (None, z(N, BF16), z(N, BF16)),            # bf16 residual
    (None, None, z(N, F32)),                   # the weight must be bf16
])
def test_nvfp4_qdq_rejects(calls, g, r, w):
    _raises(calls, codec.nvfp4_qdq, w, g, 1e-3, r)
    _raises(calls, codec.nvfp4_qdq_amax, w, g, 1e-3, r)


def test_qdq_packed_outputs_are_checked(calls):
    _raises(calls, codec.nvfp4_qdq, z(N, BF16), packed=z(N // 2 - 1, U8))
    _raises(calls, codec.nvfp4_qdq, z(N, BF16), packed=z(N // 2, U8), scales=z(N // 16, U8),
            want_packed=False)


def test_noalloc_rejects(calls):
    _raises(calls, codec.nvfp4_quantize_noalloc, z(N, BF16), residual=z(N, BF16))
    _raises(calls, codec.nvfp4_quantize_noalloc, z(N, BF16), tensor_scale=z(0, F32))
    _raises(calls, codec.nvfp4_quantize_noalloc, z(N, BF16), scales=z(N // 8, U8))


def test_mx_and_fp8_rejects(calls):
    x = z(4 * 256, BF16).view(4, 256)
    _raises(calls, codec.mxfp4_quantize, x, packed=z(4 * 64, U8))
    _raises(calls, codec.mxfp4_quantize, x, scales=z(4 * 8, torch.int16))
    pk, sc = z(4 * 128, U8).view(4, 128), z(4 * 8, U8)
    _raises(calls, codec.fp4_to_fp8_row, pk, z(4 * 7, U8))
    _raises(calls, codec.fp4_to_fp8_row, pk, sc, fp8=z(4 * 255, U8))
    _raises(calls, codec.fp4_to_fp8_row, pk, sc, fp8_scales=z(4 * 2, BF16))
    _raises(calls, codec.mxfp4_dequantize, pk, sc, out=z(4 * 256, F32))  # default out is bf16
    _raises(calls, codec.fp8_to_fp4_row, z(4 * 256, U8).view(4, 256), z(4, F32))
    _raises(calls, codec.fp8_to_fp4_row, z(4 * 256, U8).view(4, 256), z(8, F32),
            packed=z(4 * 127, U8))


def test_column_conversion_rejects(calls):
    pk, sc = z(300 * 64, U8).view(300, 64), z(300 * 4, U8)
    segs = codec.Segments(torch.tensor([0, 100, 299]), "cpu")    # covers 299 of 300 rows
    _raises(calls, codec.fp4_to_fp8_col, pk, sc, segs)
    segs = codec.Segments(torch.tensor([0, 100, 300]), "cpu")
    _raises(calls, codec.fp4_to_fp8_col, pk, sc, segs, fp8_t=z(128 * 300 - 1, U8))
    _raises(calls, codec.fp4_to_fp8_col, pk, sc, segs,
            fp8_t_scales=z(128 * segs.total_blocks, BF16))
    _raises(calls, codec.fp4_to_fp8_col, pk, sc, segs, run_blocks=-1)
    _raises(calls, codec.fp4_to_fp8_col, pk, sc, segs, run_blocks=(1 << 20) + 1)


def test_column_conversion_run_length_picks_the_entry_point(calls):
    pk, sc = z(300 * 64, U8).view(300, 64), z(300 * 4, U8)
    segs = codec.Segments(torch.tensor([0, 100, 300]), "cpu")
    codec.fp4_to_fp8_col(pk, sc, segs)
    codec.fp4_to_fp8_col(pk, sc, segs, run_blocks=7)
    assert calls == ["fp4_to_fp8_col", "fp4_to_fp8_col_runs"]


def test_fp4quant_rejects(calls):
    x = z(2 * 512, BF16).view(2, 512)
    _raises(calls, codec.fp4quant_encode, x, 96)
    _raises(calls, codec.fp4quant_encode, x, 128, s1=z(7, F32))
    _raises(calls, codec.fp4quant_encode, x, 128, packed=z(511, U8))
    pk = z(2 * 256, U8).view(2, 256)
    _raises(calls, codec.fp4quant_decode, pk, z(8, F32), z(7, F32), 128)
    _raises(calls, codec.fp4quant_decode, pk, z(8, F32), z(8, F32), 128, out=z(1023, BF16))


def test_scaled_and_blocked_rejects(calls):
    _raises(calls, codec.fp4_scaled_quantize, z(N, F32), 1.0, packed=z(N // 4, U8))
    _raises(calls, codec.fp4_scaled_dequantize, z(N // 2, U8), N + 2, 1.0)
    _raises(calls, codec.fp4_scales_from_blocked, z(511, U8), 128, 4)


def test_batch_checks_every_tensor(calls):
    xs = [z(256, BF16), z(512, BF16)]
    pks = [z(128, U8), z(256, U8)]
    scs = [z(16, U8), z(32, U8)]
    with pytest.raises(ValueError):
        codec.Batch(xs=xs, packed=[pks[0], z(255, U8)], scales=scs)
    with pytest.raises(ValueError):
        codec.Batch(xs=xs, packed=pks, scales=[scs[0], z(31, U8)])
    with pytest.raises(ValueError):
        codec.Batch(xs=[xs[0], z(512, F32)], packed=pks, scales=scs)   # mixed dtypes
    with pytest.raises(ValueError):
        codec.Batch(xs=xs, packed=pks[:1], scales=scs)                 # ragged lists
    with pytest.raises(ValueError):
        codec.Batch(packed=pks, scales=scs, ys=[z(256, BF16), z(511, BF16)],
                    sizes=[256, 512])
    assert calls == []


def test_error_feedback_rejects_mismatched_gradients(calls):
    ef = ErrorFeedback()
    w = z(N, BF16)
    with pytest.raises(ValueError):
        ef.step("w", w, z(N - 16, F32), 1e-3)
    with pytest.raises(ValueError):
        ef.step("w", w, torch.empty(N, device="meta"), 1e-3)
    with pytest.raises(ValueError):
        ef.qdq("w", z(N, torch.float64))
    assert calls == []


def test_error_feedback_state_is_stored_contiguous():
    ef = ErrorFeedback()
    base = torch.arange(64, dtype=F32).view(8, 8)
    ef.load_state_dict({"k": base.t()})
    r = ef.state_dict()["k"]
    assert r.is_contiguous() and torch.equal(r, base.t())
    with pytest.raises(ValueError):
        ef.load_state_dict({"k": base.to(BF16)})
