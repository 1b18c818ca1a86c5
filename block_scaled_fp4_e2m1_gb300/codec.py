"""Python binding of the C ABI (include/fp4codec.h), one function per entry
point with the same name.  Argument marshalling only: output tensors are
allocated with PyTorch on the input's device, pointers and the current CUDA
stream are passed to the library, and a non-OK status raises.  Every step of
the computation runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence, Tuple

import torch

from . import _lib
from ._lib import call

_DT = {torch.float32: _lib.F32_DTYPE, torch.bfloat16: _lib.BF16_DTYPE}
_ROUND = {"rtn": _lib.RTN, "sr": _lib.SR}
_TSCALE = {"given": _lib.TSCALE_GIVEN, "compute": _lib.TSCALE_COMPUTE,
           "from_amax": _lib.TSCALE_FROM_AMAX}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _cuda(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dtype(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"{name} must be float32 or bfloat16, got {t.dtype}")
    return _DT[t.dtype]


def _scalar(device, value=None) -> torch.Tensor:
    if value is None:
        return torch.empty(1, dtype=torch.float32, device=device)
    return torch.full((1,), float(value), dtype=torch.float32, device=device)


# ------------------------------------------------------------------ NVFP4

def nvfp4_amax(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
               amax_ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(x, "x")
    amax_ws = _scalar(x.device) if amax_ws is None else amax_ws
    call("nvfp4_amax", _ptr(x), _dtype(x, "x"), x.numel(), _ptr(residual), _ptr(amax_ws),
         _stream(x.device))
    return amax_ws


def nvfp4_quantize(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
                   rounding: str = "rtn", seed: int = 0, step: int = 0,
                   tscale: str = "compute", tensor_scale: Optional[torch.Tensor] = None,
                   amax_ws: Optional[torch.Tensor] = None,
                   packed: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None
                   ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Returns (packed uint8[n/2], scales uint8[n/16] e4m3, tensor_scale fp32[1])."""
    _cuda(x, "x")
    n = x.numel()
    dev = x.device
    if tensor_scale is None:
        tensor_scale = _scalar(dev, 1.0)
    if amax_ws is None and tscale != "given":
        amax_ws = _scalar(dev)
    packed = torch.empty(n // 2, dtype=torch.uint8, device=dev) if packed is None else packed
    scales = torch.empty(n // 16, dtype=torch.uint8, device=dev) if scales is None else scales
    call("nvfp4_quantize", _ptr(x), _dtype(x, "x"), n, _ptr(residual), _ROUND[rounding],
         seed, step, _TSCALE[tscale], _ptr(tensor_scale), _ptr(amax_ws), _ptr(packed),
         _ptr(scales), _stream(dev))
    return packed, scales, tensor_scale


def fp4_blocked_scales_size(rows: int, cols: int) -> int:
    """Bytes of the blocked (swizzled) form of a [rows, cols] scale matrix."""
    size = int(_lib.lib().fp4_blocked_scales_size(rows, cols))
    if size < 0:
        raise ValueError(f"scale matrix [{rows}, {cols}] out of range")
    return size


def fp4_scales_to_blocked(scales: torch.Tensor, out: Optional[torch.Tensor] = None
                          ) -> torch.Tensor:
    """[rows, cols] uint8 scales -> the blocked layout block-scaled matmuls
    read (uint8, fp4_blocked_scales_size(rows, cols) bytes)."""
    _cuda(scales, "scales")
    if scales.dim() != 2 or scales.dtype != torch.uint8:
        raise ValueError("scales must be a 2-D uint8 tensor")
    rows, cols = scales.shape
    dev = scales.device
    if out is None:
        out = torch.empty(fp4_blocked_scales_size(rows, cols), dtype=torch.uint8, device=dev)
    call("fp4_scales_to_blocked", _ptr(scales), rows, cols, _ptr(out), _stream(dev))
    return out


def fp4_scales_from_blocked(blocked: torch.Tensor, rows: int, cols: int,
                            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The inverse of fp4_scales_to_blocked: uint8 [rows, cols]."""
    _cuda(blocked, "blocked")
    if blocked.numel() != fp4_blocked_scales_size(rows, cols):
        raise ValueError("blocked has the wrong size for this scale matrix")
    dev = blocked.device
    out = torch.empty((rows, cols), dtype=torch.uint8, device=dev) if out is None else out
    call("fp4_scales_from_blocked", _ptr(blocked), rows, cols, _ptr(out), _stream(dev))
    return out


def nvfp4_quantize_blocked(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
                           rounding: str = "rtn", seed: int = 0, step: int = 0,
                           tscale: str = "compute",
                           tensor_scale: Optional[torch.Tensor] = None,
                           amax_ws: Optional[torch.Tensor] = None,
                           packed: Optional[torch.Tensor] = None,
                           blocked_scales: Optional[torch.Tensor] = None
                           ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """nvfp4_quantize of the [rows, k] matrix x with its block scales written
    in the blocked layout.  Returns (packed uint8[rows, k/2], blocked uint8
    [fp4_blocked_scales_size(rows, k/16)], tensor_scale fp32[1])."""
    _cuda(x, "x")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, k]")
    rows, k = x.shape
    dev = x.device
    if tensor_scale is None:
        tensor_scale = _scalar(dev, 1.0)
    if amax_ws is None and tscale != "given":
        amax_ws = _scalar(dev)
    if packed is None:
        packed = torch.empty((rows, k // 2), dtype=torch.uint8, device=dev)
    if blocked_scales is None:
        blocked_scales = torch.empty(fp4_blocked_scales_size(rows, k // 16),
                                     dtype=torch.uint8, device=dev)
    call("nvfp4_quantize_blocked", _ptr(x), _dtype(x, "x"), rows, k, _ptr(residual),
         _ROUND[rounding], seed, step, _TSCALE[tscale], _ptr(tensor_scale), _ptr(amax_ws),
         _ptr(packed), _ptr(blocked_scales), _stream(dev))
    return packed, blocked_scales, tensor_scale


def nvfp4_dequantize(packed: torch.Tensor, scales: torch.Tensor,
                     tensor_scale: Optional[torch.Tensor], shape: Sequence[int],
                     out_dtype: torch.dtype = torch.float32,
                     out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(packed, "packed")
    dev = packed.device
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(tuple(shape), dtype=out_dtype, device=dev) if out is None else out
    call("nvfp4_dequantize", _ptr(packed), _ptr(scales), _ptr(tensor_scale), n, _ptr(out),
         _DT[out_dtype], _stream(dev))
    return out


def nvfp4_qdq_amax(w: torch.Tensor, g: Optional[torch.Tensor], lr: float,
                   residual: Optional[torch.Tensor],
                   amax_ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(w, "w")
    amax_ws = _scalar(w.device) if amax_ws is None else amax_ws
    call("nvfp4_qdq_amax", _ptr(w), _ptr(g), lr, _ptr(residual), w.numel(), _ptr(amax_ws),
         _stream(w.device))
    return amax_ws


def nvfp4_qdq(w: torch.Tensor, g: Optional[torch.Tensor] = None, lr: float = 0.0,
              residual: Optional[torch.Tensor] = None, rounding: str = "rtn", seed: int = 0,
              step: int = 0, tscale: str = "compute",
              tensor_scale: Optional[torch.Tensor] = None,
              amax_ws: Optional[torch.Tensor] = None, packed: Optional[torch.Tensor] = None,
              scales: Optional[torch.Tensor] = None, want_packed: bool = True):
    """One step W <- qdq((W - lr*G) + r) on a bf16 weight, in place; the
    residual (fp32) is updated in place.  Returns (w, packed, scales,
    tensor_scale); packed/scales are None when want_packed is False."""
    _cuda(w, "w")
    if w.dtype != torch.bfloat16:
        raise ValueError("w must be bfloat16")
    n = w.numel()
    dev = w.device
    if tensor_scale is None:
        tensor_scale = _scalar(dev, 1.0)
    if amax_ws is None and tscale != "given":
        amax_ws = _scalar(dev)
    if want_packed:
        packed = torch.empty(n // 2, dtype=torch.uint8, device=dev) if packed is None else packed
        scales = torch.empty(n // 16, dtype=torch.uint8, device=dev) if scales is None else scales
    else:
        packed = scales = None
    call("nvfp4_qdq", _ptr(w), _ptr(g), lr, n, _ptr(residual), _ROUND[rounding], seed, step,
         _TSCALE[tscale], _ptr(tensor_scale), _ptr(amax_ws), _ptr(packed), _ptr(scales),
         _stream(dev))
    return w, packed, scales, tensor_scale


def nvfp4_quantize_noalloc(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
                           rounding: str = "rtn", seed: int = 0, step: int = 0,
                           tensor_scale: Optional[torch.Tensor] = None,
                           packed: Optional[torch.Tensor] = None,
                           scales: Optional[torch.Tensor] = None):
    """nvfp4_quantize with a computed tensor scale whose amax workspace is
    the library's own device array (for callers that cannot allocate device
    memory).  Calls that overlap on the GPU must be serialized."""
    _cuda(x, "x")
    n = x.numel()
    dev = x.device
    tensor_scale = _scalar(dev) if tensor_scale is None else tensor_scale
    packed = torch.empty(n // 2, dtype=torch.uint8, device=dev) if packed is None else packed
    scales = torch.empty(n // 16, dtype=torch.uint8, device=dev) if scales is None else scales
    call("nvfp4_quantize_noalloc", _ptr(x), _dtype(x, "x"), n, _ptr(residual), _ROUND[rounding],
         seed, step, _ptr(tensor_scale), _ptr(packed), _ptr(scales), _stream(dev))
    return packed, scales, tensor_scale


# --------------------------------------------------------- NVFP4, batched

class Batch:
    """A list of independent tensors for the batched NVFP4 calls: the
    descriptor table of include/fp4codec.h (fp4_tensor_desc), checked and
    numbered on the host by fp4_batch_plan and uploaded once to the device.
    Holds references to the tensors it points at."""

    DESC = None  # numpy dtype of fp4_tensor_desc, built on first use

    def __init__(self, xs=None, packed=None, scales=None, ys=None, sizes=None, device=None,
                 ks=None):
        import numpy as np
        if Batch.DESC is None:
            Batch.DESC = np.dtype([("x", "<u8"), ("packed", "<u8"), ("scales", "<u8"),
                                   ("y", "<u8"), ("n", "<i8"), ("chunk_start", "<i8")])
        lists = [lst for lst in (xs, packed, scales, ys) if lst is not None]
        count = len(lists[0]) if lists else len(sizes)
        if sizes is None:
            src = xs if xs is not None else ys
            sizes = [t.numel() for t in src]
        self.count = count
        self.sizes = [int(s) for s in sizes]
        self._keep = [xs, packed, scales, ys]
        host = np.zeros(count, Batch.DESC)
        for name, lst in (("x", xs), ("packed", packed), ("scales", scales), ("y", ys)):
            if lst is not None:
                for i, t in enumerate(lst):
                    _cuda(t, name)
                    host[name][i] = t.data_ptr()
        host["n"] = self.sizes
        total = ctypes.c_int64(0)
        if ks is None:
            call("fp4_batch_plan", host.ctypes.data, count, ctypes.addressof(total))
        else:
            # row lengths for the blocked scale layout (nvfp4_quantize_batched_blocked)
            kh = np.ascontiguousarray(np.asarray(ks, dtype=np.int64))
            if kh.size != count:
                raise ValueError("ks needs one row length per tensor")
            call("fp4_batch_plan_blocked", host.ctypes.data, kh.ctypes.data, count,
                 ctypes.addressof(total))
        self.total_chunks = int(total.value)
        self.host = host
        dev = device if device is not None else (lists[0][0].device if lists and count else "cuda")
        self.desc = torch.from_numpy(host.view(np.uint8).copy()).to(dev)
        self.device = self.desc.device
        self.kdev = None if ks is None else torch.from_numpy(kh).to(self.device)


def nvfp4_amax_batched(batch: Batch, dtype: torch.dtype,
                       amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    amax = torch.empty(batch.count, dtype=torch.float32, device=batch.device) if amax is None else amax
    call("nvfp4_amax_batched", _ptr(batch.desc), batch.count, batch.total_chunks, _DT[dtype],
         _ptr(amax), _stream(batch.device))
    return amax


def nvfp4_quantize_batched(batch: Batch, dtype: torch.dtype, rounding: str = "rtn",
                           seed: int = 0, step: int = 0, tscale: str = "compute",
                           tensor_scale: Optional[torch.Tensor] = None,
                           amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quantizes every tensor of the batch into its packed/scales buffers;
    returns the per-tensor scales (fp32 [count])."""
    dev = batch.device
    if tensor_scale is None:
        tensor_scale = torch.ones(batch.count, dtype=torch.float32, device=dev)
    if amax is None and tscale != "given":
        amax = torch.empty(batch.count, dtype=torch.float32, device=dev)
    call("nvfp4_quantize_batched", _ptr(batch.desc), batch.count, batch.total_chunks, _DT[dtype],
         _ROUND[rounding], seed, step, _TSCALE[tscale], _ptr(tensor_scale), _ptr(amax),
         _stream(dev))
    return tensor_scale


def nvfp4_quantize_batched_blocked(batch: Batch, dtype: torch.dtype, rounding: str = "rtn",
                                   seed: int = 0, step: int = 0, tscale: str = "compute",
                                   tensor_scale: Optional[torch.Tensor] = None,
                                   amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    """nvfp4_quantize_batched with every tensor's scales in the blocked layout
    of its [n / k, k] matrix; the batch is built with ks (row lengths) and its
    scales buffers hold fp4_blocked_scales_size(n / k, k / 16) bytes each."""
    if batch.kdev is None:
        raise ValueError("the batch was built without ks")
    dev = batch.device
    if tensor_scale is None:
        tensor_scale = torch.ones(batch.count, dtype=torch.float32, device=dev)
    if amax is None and tscale != "given":
        amax = torch.empty(batch.count, dtype=torch.float32, device=dev)
    call("nvfp4_quantize_batched_blocked", _ptr(batch.desc), _ptr(batch.kdev), batch.count,
         batch.total_chunks, _DT[dtype], _ROUND[rounding], seed, step, _TSCALE[tscale],
         _ptr(tensor_scale), _ptr(amax), _stream(dev))
    return tensor_scale


def nvfp4_dequantize_batched(batch: Batch, tensor_scale: Optional[torch.Tensor],
                             out_dtype: torch.dtype = torch.bfloat16) -> None:
    call("nvfp4_dequantize_batched", _ptr(batch.desc), batch.count, batch.total_chunks,
         _ptr(tensor_scale), _DT[out_dtype], _stream(batch.device))


# ------------------------------------------------------------------ MXFP4

def mxfp4_quantize(x: torch.Tensor, packed: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None):
    """x [rows, cols] -> (packed uint8[rows, cols/2], scales uint8[rows, cols/32])."""
    _cuda(x, "x")
    rows, cols = x.shape
    dev = x.device
    packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev) if packed is None else packed
    scales = torch.empty(rows, cols // 32, dtype=torch.uint8, device=dev) if scales is None else scales
    call("mxfp4_quantize", _ptr(x), _dtype(x, "x"), rows, cols, _ptr(packed), _ptr(scales),
         _stream(dev))
    return packed, scales


def fp4_scaled_quantize(x: torch.Tensor, scale: float,
                        packed: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One fp32 scale for the whole tensor: codes RN_e2m1(RN(x / scale)),
    packed two per byte (n/2 bytes)."""
    _cuda(x, "x")
    n = x.numel()
    packed = torch.empty(n // 2, dtype=torch.uint8, device=x.device) if packed is None else packed
    call("fp4_scaled_quantize", _ptr(x), _dtype(x, "x"), n, float(scale), _ptr(packed),
         _stream(x.device))
    return packed


def fp4_scaled_dequantize(packed: torch.Tensor, n: int, scale: float,
                          out_dtype: torch.dtype = torch.float32,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """value(code) * scale for the n codes of packed."""
    _cuda(packed, "packed")
    out = torch.empty(n, dtype=out_dtype, device=packed.device) if out is None else out
    call("fp4_scaled_dequantize", _ptr(packed), n, float(scale), _ptr(out), _dtype(out, "out"),
         _stream(packed.device))
    return out


def fp8_to_fp4_row(fp8: torch.Tensor, fp8_scales: torch.Tensor,
                   packed: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None):
    """(E4M3 bytes uint8[rows, cols], fp32 scales [rows, cols/128]) ->
    (packed uint8[rows, cols/2], UE8M0 scales uint8[rows, cols/32])."""
    _cuda(fp8, "fp8")
    rows, cols = fp8.shape
    dev = fp8.device
    packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev) if packed is None else packed
    scales = torch.empty(rows, cols // 32, dtype=torch.uint8, device=dev) if scales is None else scales
    call("fp8_to_fp4_row", _ptr(fp8), _ptr(fp8_scales), rows, cols, _ptr(packed), _ptr(scales),
         _stream(dev))
    return packed, scales


def mxfp4_dequantize(packed: torch.Tensor, scales: torch.Tensor,
                     out_dtype: torch.dtype = torch.bfloat16,
                     out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """(packed [rows, cols/2], UE8M0 scales [rows, cols/32]) -> [rows, cols]
    fp32 or bf16."""
    _cuda(packed, "packed")
    rows, half = packed.shape
    cols = 2 * half
    dev = packed.device
    out = torch.empty(rows, cols, dtype=out_dtype, device=dev) if out is None else out
    call("mxfp4_dequantize", _ptr(packed), _ptr(scales), rows, cols, _ptr(out),
         _dtype(out, "out"), _stream(dev))
    return out


def fp4_to_fp8_row(packed: torch.Tensor, scales: torch.Tensor,
                   fp8: Optional[torch.Tensor] = None,
                   fp8_scales: Optional[torch.Tensor] = None):
    """(packed [rows, cols/2], UE8M0 scales [rows, cols/32]) -> (E4M3 bytes
    uint8[rows, cols], fp32 scales [rows, cols/128])."""
    _cuda(packed, "packed")
    rows, half = packed.shape
    cols = 2 * half
    dev = packed.device
    fp8 = torch.empty(rows, cols, dtype=torch.uint8, device=dev) if fp8 is None else fp8
    fp8_scales = (torch.empty(rows, cols // 128, dtype=torch.float32, device=dev)
                  if fp8_scales is None else fp8_scales)
    call("fp4_to_fp8_row", _ptr(packed), _ptr(scales), rows, cols, _ptr(fp8), _ptr(fp8_scales),
         _stream(dev))
    return fp8, fp8_scales


def fp4_seg_scale_offsets(row_off: torch.Tensor) -> torch.Tensor:
    """Host helper: running sum of ceil(n_e / 128) (CPU int64 in and out)."""
    ro = row_off.to(device="cpu", dtype=torch.int64).contiguous()
    out = torch.empty_like(ro)
    call("fp4_seg_scale_offsets", ro.data_ptr(), ro.numel() - 1, out.data_ptr())
    return out


class Segments:
    """Ragged expert segments: row offsets (host int64 [E+1]) with their
    scale-block offsets, both uploaded once to the device."""

    def __init__(self, row_off: torch.Tensor, device):
        self.row_off_host = row_off.to(device="cpu", dtype=torch.int64).contiguous()
        self.scale_off_host = fp4_seg_scale_offsets(self.row_off_host)
        self.row_off = self.row_off_host.to(device)
        self.scale_off = self.scale_off_host.to(device)
        self.num_segments = self.row_off_host.numel() - 1
        self.total_rows = int(self.row_off_host[-1])
        self.total_blocks = int(self.scale_off_host[-1])


def fp4_to_fp8_col(packed: torch.Tensor, scales: torch.Tensor, segments: Segments,
                   fp8_t: Optional[torch.Tensor] = None,
                   fp8_t_scales: Optional[torch.Tensor] = None):
    """Per segment e: [cols, n_e] E4M3 at fp8_t[cols*row_off[e]:] and
    [cols, ceil(n_e/128)] fp32 scales at fp8_t_scales[cols*scale_off[e]:]
    (flat outputs)."""
    _cuda(packed, "packed")
    rows, half = packed.shape
    cols = 2 * half
    dev = packed.device
    fp8_t = (torch.empty(cols * segments.total_rows, dtype=torch.uint8, device=dev)
             if fp8_t is None else fp8_t)
    fp8_t_scales = (torch.empty(cols * segments.total_blocks, dtype=torch.float32, device=dev)
                    if fp8_t_scales is None else fp8_t_scales)
    call("fp4_to_fp8_col", _ptr(packed), _ptr(scales), cols, _ptr(segments.row_off),
         _ptr(segments.scale_off), segments.num_segments, segments.total_rows,
         segments.total_blocks, _ptr(fp8_t), _ptr(fp8_t_scales), _stream(dev))
    return fp8_t, fp8_t_scales


# --------------------------------------------------------------- FP4Quant

def fp4quant_encode(x: torch.Tensor, group: int, packed: Optional[torch.Tensor] = None,
                    s1: Optional[torch.Tensor] = None, s2: Optional[torch.Tensor] = None):
    """x [rows, cols] -> (packed uint8[rows, cols/2], s1, s2 fp32[rows, cols/group])."""
    _cuda(x, "x")
    rows, cols = x.shape
    dev = x.device
    packed = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev) if packed is None else packed
    s1 = torch.empty(rows, cols // group, dtype=torch.float32, device=dev) if s1 is None else s1
    s2 = torch.empty(rows, cols // group, dtype=torch.float32, device=dev) if s2 is None else s2
    call("fp4quant_encode", _ptr(x), _dtype(x, "x"), rows, cols, group, _ptr(packed), _ptr(s1),
         _ptr(s2), _stream(dev))
    return packed, s1, s2


def fp4quant_decode(packed: torch.Tensor, s1: torch.Tensor, s2: torch.Tensor, group: int,
                    out_dtype: torch.dtype = torch.bfloat16,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(packed, "packed")
    rows, half = packed.shape
    cols = 2 * half
    dev = packed.device
    out = torch.empty(rows, cols, dtype=out_dtype, device=dev) if out is None else out
    call("fp4quant_decode", _ptr(packed), _ptr(s1), _ptr(s2), rows, cols, group, _ptr(out),
         _DT[out_dtype], _stream(dev))
    return out


def kernel_launches() -> int:
    return int(_lib.lib().fp4_kernel_launches())
