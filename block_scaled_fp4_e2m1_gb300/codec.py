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


def _is_device_tensor(t: torch.Tensor) -> bool:
    return t.is_cuda


def _cuda(t: torch.Tensor, name: str) -> None:
    """The main input of a call: a contiguous CUDA tensor."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not _is_device_tensor(t):
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _expect(t: Optional[torch.Tensor], name: str, device: torch.device, numel: Optional[int],
            dtypes) -> None:
    """A caller-supplied tensor the kernels read or write through a raw
    pointer: it must be contiguous, on the call's device, of one of `dtypes`
    and hold exactly `numel` elements, or the kernel would run past its end.
    None is accepted (optional arguments)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call runs on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not isinstance(dtypes, tuple):
        dtypes = (dtypes,)
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")


def _dtype(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"{name} must be float32 or bfloat16, got {t.dtype}")
    return _DT[t.dtype]


def _out_dtype(dt: torch.dtype) -> int:
    if dt not in _DT:
        raise ValueError(f"out_dtype must be float32 or bfloat16, got {dt}")
    return _DT[dt]


def _choice(table, value, name):
    if value not in table:
        raise ValueError(f"{name} must be one of {sorted(table)}, got {value!r}")
    return table[value]


def _scalar(device, value=None) -> torch.Tensor:
    if value is None:
        return torch.empty(1, dtype=torch.float32, device=device)
    return torch.full((1,), float(value), dtype=torch.float32, device=device)


def _numel(shape: Sequence[int]) -> int:
    n = 1
    for s in shape:
        n *= int(s)
    return n


# ------------------------------------------------------------------ NVFP4

_F32, _BF16, _U8 = torch.float32, torch.bfloat16, torch.uint8


def _nvfp4_buffers(dev, n, residual, tensor_scale, amax_ws, tscale):
    """Check the optional fp32 buffers of an NVFP4 quantize of n elements
    and allocate the scalars that were not given."""
    _choice(_TSCALE, tscale, "tscale")
    _expect(residual, "residual", dev, n, _F32)
    _expect(tensor_scale, "tensor_scale", dev, 1, _F32)
    _expect(amax_ws, "amax_ws", dev, 1, _F32)
    if tensor_scale is None:
        tensor_scale = _scalar(dev, 1.0)
    if amax_ws is None and tscale != "given":
        amax_ws = _scalar(dev)
    return tensor_scale, amax_ws


def _codes_out(dev, n, packed, scales):
    """Check or allocate the packed codes (n/2 bytes) and linear e4m3 block
    scales (n/16 bytes) of n elements."""
    _expect(packed, "packed", dev, n // 2, _U8)
    _expect(scales, "scales", dev, n // 16, _U8)
    packed = torch.empty(n // 2, dtype=_U8, device=dev) if packed is None else packed
    scales = torch.empty(n // 16, dtype=_U8, device=dev) if scales is None else scales
    return packed, scales


def nvfp4_amax(x: torch.Tensor, residual: Optional[torch.Tensor] = None,
               amax_ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(x, "x")
    dt = _dtype(x, "x")
    _expect(residual, "residual", x.device, x.numel(), _F32)
    _expect(amax_ws, "amax_ws", x.device, 1, _F32)
    amax_ws = _scalar(x.device) if amax_ws is None else amax_ws
    call("nvfp4_amax", _ptr(x), dt, x.numel(), _ptr(residual), _ptr(amax_ws),
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
    dt = _dtype(x, "x")
    rnd = _choice(_ROUND, rounding, "rounding")
    n = x.numel()
    dev = x.device
    tensor_scale, amax_ws = _nvfp4_buffers(dev, n, residual, tensor_scale, amax_ws, tscale)
    packed, scales = _codes_out(dev, n, packed, scales)
    call("nvfp4_quantize", _ptr(x), dt, n, _ptr(residual), rnd, seed, step, _TSCALE[tscale],
         _ptr(tensor_scale), _ptr(amax_ws), _ptr(packed), _ptr(scales), _stream(dev))
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
    if scales.dim() != 2 or scales.dtype != _U8:
        raise ValueError("scales must be a 2-D uint8 tensor")
    rows, cols = scales.shape
    dev = scales.device
    size = fp4_blocked_scales_size(rows, cols)
    _expect(out, "out", dev, size, _U8)
    if out is None:
        out = torch.empty(size, dtype=_U8, device=dev)
    call("fp4_scales_to_blocked", _ptr(scales), rows, cols, _ptr(out), _stream(dev))
    return out


def fp4_scales_from_blocked(blocked: torch.Tensor, rows: int, cols: int,
                            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The inverse of fp4_scales_to_blocked: uint8 [rows, cols]."""
    _cuda(blocked, "blocked")
    dev = blocked.device
    _expect(blocked, "blocked", dev, fp4_blocked_scales_size(rows, cols), _U8)
    _expect(out, "out", dev, rows * cols, _U8)
    out = torch.empty((rows, cols), dtype=_U8, device=dev) if out is None else out
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
    dt = _dtype(x, "x")
    rnd = _choice(_ROUND, rounding, "rounding")
    rows, k = x.shape
    dev = x.device
    size = fp4_blocked_scales_size(rows, k // 16)
    _expect(blocked_scales, "blocked_scales", dev, size, _U8)
    _expect(packed, "packed", dev, rows * (k // 2), _U8)
    tensor_scale, amax_ws = _nvfp4_buffers(dev, rows * k, residual, tensor_scale, amax_ws,
                                           tscale)
    if packed is None:
        packed = torch.empty((rows, k // 2), dtype=_U8, device=dev)
    if blocked_scales is None:
        blocked_scales = torch.empty(size, dtype=_U8, device=dev)
    call("nvfp4_quantize_blocked", _ptr(x), dt, rows, k, _ptr(residual), rnd, seed, step,
         _TSCALE[tscale], _ptr(tensor_scale), _ptr(amax_ws), _ptr(packed),
         _ptr(blocked_scales), _stream(dev))
    return packed, blocked_scales, tensor_scale


def nvfp4_dequantize(packed: torch.Tensor, scales: torch.Tensor,
                     tensor_scale: Optional[torch.Tensor], shape: Sequence[int],
                     out_dtype: torch.dtype = torch.float32,
                     out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(packed, "packed")
    dev = packed.device
    n = _numel(shape)
    odt = _out_dtype(out_dtype)
    _expect(packed, "packed", dev, n // 2, _U8)
    _expect(scales, "scales", dev, n // 16, _U8)
    if scales is None:
        raise ValueError("scales are required")
    _expect(tensor_scale, "tensor_scale", dev, 1, _F32)
    _expect(out, "out", dev, n, out_dtype)
    out = torch.empty(tuple(shape), dtype=out_dtype, device=dev) if out is None else out
    call("nvfp4_dequantize", _ptr(packed), _ptr(scales), _ptr(tensor_scale), n, _ptr(out),
         odt, _stream(dev))
    return out


def _qdq_inputs(w, g, residual):
    _cuda(w, "w")
    if w.dtype != _BF16:
        raise ValueError("w must be bfloat16")
    _expect(g, "g", w.device, w.numel(), _F32)
    _expect(residual, "residual", w.device, w.numel(), _F32)


def nvfp4_qdq_amax(w: torch.Tensor, g: Optional[torch.Tensor], lr: float,
                   residual: Optional[torch.Tensor],
                   amax_ws: Optional[torch.Tensor] = None) -> torch.Tensor:
    _qdq_inputs(w, g, residual)
    _expect(amax_ws, "amax_ws", w.device, 1, _F32)
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
    _qdq_inputs(w, g, residual)
    rnd = _choice(_ROUND, rounding, "rounding")
    n = w.numel()
    dev = w.device
    tensor_scale, amax_ws = _nvfp4_buffers(dev, n, None, tensor_scale, amax_ws, tscale)
    if want_packed:
        packed, scales = _codes_out(dev, n, packed, scales)
    elif packed is not None or scales is not None:
        raise ValueError("packed/scales given with want_packed=False")
    call("nvfp4_qdq", _ptr(w), _ptr(g), lr, n, _ptr(residual), rnd, seed, step,
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
    dt = _dtype(x, "x")
    rnd = _choice(_ROUND, rounding, "rounding")
    n = x.numel()
    dev = x.device
    _expect(residual, "residual", dev, n, _F32)
    _expect(tensor_scale, "tensor_scale", dev, 1, _F32)
    tensor_scale = _scalar(dev) if tensor_scale is None else tensor_scale
    packed, scales = _codes_out(dev, n, packed, scales)
    call("nvfp4_quantize_noalloc", _ptr(x), dt, n, _ptr(residual), rnd, seed, step,
         _ptr(tensor_scale), _ptr(packed), _ptr(scales), _stream(dev))
    return packed, scales, tensor_scale


# --------------------------------------------------------- NVFP4, batched

class Batch:
    """A list of independent tensors for the batched NVFP4 calls: the
    descriptor table of include/fp4codec.h (fp4_tensor_desc), checked and
    numbered on the host by fp4_batch_plan and uploaded once to the device.
    Holds references to the tensors it points at.

    Every tensor must be contiguous and on one device: xs (float32 or
    bfloat16, all of one dtype) and ys (float32 or bfloat16) hold n_t
    elements, packed n_t / 2 bytes, scales n_t / 16 bytes (or, with ks, the
    blocked size of the [n_t / k_t, k_t / 16] scale matrix)."""

    DESC = None  # numpy dtype of fp4_tensor_desc, built on first use

    def __init__(self, xs=None, packed=None, scales=None, ys=None, sizes=None, device=None,
                 ks=None):
        import numpy as np
        if Batch.DESC is None:
            Batch.DESC = np.dtype([("x", "<u8"), ("packed", "<u8"), ("scales", "<u8"),
                                   ("y", "<u8"), ("n", "<i8"), ("chunk_start", "<i8")])
        lists = [lst for lst in (xs, packed, scales, ys) if lst is not None]
        count = len(lists[0]) if lists else len(sizes)
        if any(len(lst) != count for lst in lists) or (sizes is not None and len(sizes) != count):
            raise ValueError("every list of a batch needs one entry per tensor")
        if sizes is None:
            src = xs if xs is not None else ys
            if src is None:
                raise ValueError("sizes are needed when neither xs nor ys is given")
            sizes = [t.numel() for t in src]
        self.count = count
        self.sizes = [int(s) for s in sizes]
        kh = None
        if ks is not None:
            kh = np.ascontiguousarray(np.asarray(ks, dtype=np.int64))
            if kh.size != count:
                raise ValueError("ks needs one row length per tensor")
        first = next((lst[0] for lst in lists if len(lst)), None)
        dev = torch.device(device) if device is not None else (
            first.device if first is not None else torch.device("cuda"))
        self.x_dtype = None
        self.y_dtype = None
        for i, n in enumerate(self.sizes):
            if xs is not None:
                _cuda(xs[i], f"xs[{i}]")
                _expect(xs[i], f"xs[{i}]", dev, n, (_F32, _BF16))
                if self.x_dtype is None:
                    self.x_dtype = xs[i].dtype
                elif xs[i].dtype != self.x_dtype:
                    raise ValueError("every x of a batch must have one dtype")
            if packed is not None:
                _cuda(packed[i], f"packed[{i}]")
                _expect(packed[i], f"packed[{i}]", dev, n // 2, _U8)
            if scales is not None:
                _cuda(scales[i], f"scales[{i}]")
                want = n // 16
                if kh is not None:
                    k = int(kh[i])
                    want = (fp4_blocked_scales_size(n // k, k // 16)
                            if k > 0 and k % 16 == 0 and n % k == 0 else None)
                _expect(scales[i], f"scales[{i}]", dev, want, _U8)
            if ys is not None:
                _cuda(ys[i], f"ys[{i}]")
                _expect(ys[i], f"ys[{i}]", dev, n, (_F32, _BF16))
                if self.y_dtype is None:
                    self.y_dtype = ys[i].dtype
                elif ys[i].dtype != self.y_dtype:
                    raise ValueError("every y of a batch must have one dtype")
        self._keep = [xs, packed, scales, ys]
        host = np.zeros(count, Batch.DESC)
        for name, lst in (("x", xs), ("packed", packed), ("scales", scales), ("y", ys)):
            if lst is not None:
                for i, t in enumerate(lst):
                    host[name][i] = t.data_ptr()
        host["n"] = self.sizes
        total = ctypes.c_int64(0)
        if kh is None:
            call("fp4_batch_plan", host.ctypes.data, count, ctypes.addressof(total))
        else:
            # row lengths for the blocked scale layout (nvfp4_quantize_batched_blocked)
            call("fp4_batch_plan_blocked", host.ctypes.data, kh.ctypes.data, count,
                 ctypes.addressof(total))
        self.total_chunks = int(total.value)
        self.host = host
        self.has = {"x": xs is not None, "packed": packed is not None,
                    "scales": scales is not None, "y": ys is not None}
        self.desc = torch.from_numpy(host.view(np.uint8).copy()).to(dev)
        self.device = self.desc.device
        self.kdev = None if kh is None else torch.from_numpy(kh).to(self.device)

    def _needs(self, *names):
        for nm in names:
            if self.count and not self.has[nm]:
                raise ValueError(f"this batch was built without {nm}")


def nvfp4_amax_batched(batch: Batch, dtype: torch.dtype,
                       amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    batch._needs("x")
    if batch.x_dtype is not None and dtype != batch.x_dtype:
        raise ValueError(f"the batch's inputs are {batch.x_dtype}, not {dtype}")
    _expect(amax, "amax", batch.device, batch.count, _F32)
    amax = torch.empty(batch.count, dtype=_F32, device=batch.device) if amax is None else amax
    call("nvfp4_amax_batched", _ptr(batch.desc), batch.count, batch.total_chunks,
         _out_dtype(dtype), _ptr(amax), _stream(batch.device))
    return amax


def _batched_scales(batch, dtype, rounding, tscale, tensor_scale, amax):
    batch._needs("x", "packed", "scales")
    if batch.x_dtype is not None and dtype != batch.x_dtype:
        raise ValueError(f"the batch's inputs are {batch.x_dtype}, not {dtype}")
    _choice(_ROUND, rounding, "rounding")
    _choice(_TSCALE, tscale, "tscale")
    dev = batch.device
    _expect(tensor_scale, "tensor_scale", dev, batch.count, _F32)
    _expect(amax, "amax", dev, batch.count, _F32)
    if tensor_scale is None:
        tensor_scale = torch.ones(batch.count, dtype=_F32, device=dev)
    if amax is None and tscale != "given":
        amax = torch.empty(batch.count, dtype=_F32, device=dev)
    return tensor_scale, amax


def nvfp4_quantize_batched(batch: Batch, dtype: torch.dtype, rounding: str = "rtn",
                           seed: int = 0, step: int = 0, tscale: str = "compute",
                           tensor_scale: Optional[torch.Tensor] = None,
                           amax: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quantizes every tensor of the batch into its packed/scales buffers;
    returns the per-tensor scales (fp32 [count])."""
    if batch.kdev is not None:
        raise ValueError("the batch was built with ks: use nvfp4_quantize_batched_blocked")
    tensor_scale, amax = _batched_scales(batch, dtype, rounding, tscale, tensor_scale, amax)
    call("nvfp4_quantize_batched", _ptr(batch.desc), batch.count, batch.total_chunks,
         _out_dtype(dtype), _ROUND[rounding], seed, step, _TSCALE[tscale], _ptr(tensor_scale),
         _ptr(amax), _stream(batch.device))
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
    tensor_scale, amax = _batched_scales(batch, dtype, rounding, tscale, tensor_scale, amax)
    call("nvfp4_quantize_batched_blocked", _ptr(batch.desc), _ptr(batch.kdev), batch.count,
         batch.total_chunks, _out_dtype(dtype), _ROUND[rounding], seed, step, _TSCALE[tscale],
         _ptr(tensor_scale), _ptr(amax), _stream(batch.device))
    return tensor_scale


def nvfp4_dequantize_batched(batch: Batch, tensor_scale: Optional[torch.Tensor],
                             out_dtype: torch.dtype = torch.bfloat16) -> None:
    batch._needs("packed", "scales", "y")
    if batch.kdev is not None:
        raise ValueError("the batch's scales are blocked; dequantize reads linear scales")
    if batch.y_dtype is not None and out_dtype != batch.y_dtype:
        raise ValueError(f"the batch's outputs are {batch.y_dtype}, not {out_dtype}")
    _expect(tensor_scale, "tensor_scale", batch.device, batch.count, _F32)
    call("nvfp4_dequantize_batched", _ptr(batch.desc), batch.count, batch.total_chunks,
         _ptr(tensor_scale), _out_dtype(out_dtype), _stream(batch.device))


# ------------------------------------------------------------------ MXFP4

def _matrix(t: torch.Tensor, name: str):
    _cuda(t, name)
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    return t.shape


def mxfp4_quantize(x: torch.Tensor, packed: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None):
    """x [rows, cols] -> (packed uint8[rows, cols/2], scales uint8[rows, cols/32])."""
    rows, cols = _matrix(x, "x")
    dt = _dtype(x, "x")
    dev = x.device
    _expect(packed, "packed", dev, rows * (cols // 2), _U8)
    _expect(scales, "scales", dev, rows * (cols // 32), _U8)
    packed = torch.empty(rows, cols // 2, dtype=_U8, device=dev) if packed is None else packed
    scales = torch.empty(rows, cols // 32, dtype=_U8, device=dev) if scales is None else scales
    call("mxfp4_quantize", _ptr(x), dt, rows, cols, _ptr(packed), _ptr(scales), _stream(dev))
    return packed, scales


def fp4_scaled_quantize(x: torch.Tensor, scale: float,
                        packed: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One fp32 scale for the whole tensor: codes RN_e2m1(RN(x / scale)),
    packed two per byte (n/2 bytes)."""
    _cuda(x, "x")
    dt = _dtype(x, "x")
    n = x.numel()
    _expect(packed, "packed", x.device, n // 2, _U8)
    packed = torch.empty(n // 2, dtype=_U8, device=x.device) if packed is None else packed
    call("fp4_scaled_quantize", _ptr(x), dt, n, float(scale), _ptr(packed), _stream(x.device))
    return packed


def fp4_scaled_dequantize(packed: torch.Tensor, n: int, scale: float,
                          out_dtype: torch.dtype = torch.float32,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """value(code) * scale for the n codes of packed."""
    _cuda(packed, "packed")
    dev = packed.device
    odt = _out_dtype(out_dtype)
    _expect(packed, "packed", dev, n // 2, _U8)
    _expect(out, "out", dev, n, out_dtype)
    out = torch.empty(n, dtype=out_dtype, device=dev) if out is None else out
    call("fp4_scaled_dequantize", _ptr(packed), n, float(scale), _ptr(out), odt, _stream(dev))
    return out


def fp4_scaled_quantize_amax(x: torch.Tensor, amax: torch.Tensor,
                             scale_out: Optional[torch.Tensor] = None,
                             packed: Optional[torch.Tensor] = None):
    """One scale per tensor chosen on the device from its amax (fp32[1], e.g.
    nvfp4_amax(x)): scale = RN(amax / 6), 1 if that is not finite and > 0.
    Returns (packed uint8[n/2], scale fp32[1])."""
    _cuda(x, "x")
    dt = _dtype(x, "x")
    n = x.numel()
    dev = x.device
    if amax is None:
        raise ValueError("amax is required")
    _expect(amax, "amax", dev, 1, _F32)
    _expect(scale_out, "scale_out", dev, 1, _F32)
    _expect(packed, "packed", dev, n // 2, _U8)
    scale_out = _scalar(dev) if scale_out is None else scale_out
    packed = torch.empty(n // 2, dtype=_U8, device=dev) if packed is None else packed
    call("fp4_scaled_quantize_amax", _ptr(x), dt, n, _ptr(amax), _ptr(scale_out), _ptr(packed),
         _stream(dev))
    return packed, scale_out


def fp4_scaled_dequantize_dev(packed: torch.Tensor, n: int, scale: torch.Tensor,
                              out_dtype: torch.dtype = torch.float32,
                              out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """value(code) * scale for the n codes of packed, scale an fp32[1] on the
    device."""
    _cuda(packed, "packed")
    dev = packed.device
    odt = _out_dtype(out_dtype)
    _expect(packed, "packed", dev, n // 2, _U8)
    if scale is None:
        raise ValueError("scale is required")
    _expect(scale, "scale", dev, 1, _F32)
    _expect(out, "out", dev, n, out_dtype)
    out = torch.empty(n, dtype=out_dtype, device=dev) if out is None else out
    call("fp4_scaled_dequantize_dev", _ptr(packed), n, _ptr(scale), _ptr(out), odt, _stream(dev))
    return out


def fp8_to_fp4_row(fp8: torch.Tensor, fp8_scales: torch.Tensor,
                   packed: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None):
    """(E4M3 bytes uint8[rows, cols], fp32 scales [rows, cols/128]) ->
    (packed uint8[rows, cols/2], UE8M0 scales uint8[rows, cols/32])."""
    rows, cols = _matrix(fp8, "fp8")
    dev = fp8.device
    _expect(fp8, "fp8", dev, rows * cols, _U8)
    if fp8_scales is None:
        raise ValueError("fp8_scales are required")
    _expect(fp8_scales, "fp8_scales", dev, rows * (cols // 128), _F32)
    _expect(packed, "packed", dev, rows * (cols // 2), _U8)
    _expect(scales, "scales", dev, rows * (cols // 32), _U8)
    packed = torch.empty(rows, cols // 2, dtype=_U8, device=dev) if packed is None else packed
    scales = torch.empty(rows, cols // 32, dtype=_U8, device=dev) if scales is None else scales
    call("fp8_to_fp4_row", _ptr(fp8), _ptr(fp8_scales), rows, cols, _ptr(packed), _ptr(scales),
         _stream(dev))
    return packed, scales


def _mx_source(packed, scales):
    rows, half = _matrix(packed, "packed")
    cols = 2 * half
    dev = packed.device
    _expect(packed, "packed", dev, rows * half, _U8)
    if scales is None:
        raise ValueError("scales are required")
    _expect(scales, "scales", dev, rows * (cols // 32), _U8)
    return rows, cols, dev


def mxfp4_dequantize(packed: torch.Tensor, scales: torch.Tensor,
                     out_dtype: torch.dtype = torch.bfloat16,
                     out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """(packed [rows, cols/2], UE8M0 scales [rows, cols/32]) -> [rows, cols]
    fp32 or bf16."""
    rows, cols, dev = _mx_source(packed, scales)
    odt = _out_dtype(out_dtype)
    _expect(out, "out", dev, rows * cols, out_dtype)
    out = torch.empty(rows, cols, dtype=out_dtype, device=dev) if out is None else out
    call("mxfp4_dequantize", _ptr(packed), _ptr(scales), rows, cols, _ptr(out), odt,
         _stream(dev))
    return out


def fp4_to_fp8_row(packed: torch.Tensor, scales: torch.Tensor,
                   fp8: Optional[torch.Tensor] = None,
                   fp8_scales: Optional[torch.Tensor] = None):
    """(packed [rows, cols/2], UE8M0 scales [rows, cols/32]) -> (E4M3 bytes
    uint8[rows, cols], fp32 scales [rows, cols/128])."""
    rows, cols, dev = _mx_source(packed, scales)
    _expect(fp8, "fp8", dev, rows * cols, _U8)
    _expect(fp8_scales, "fp8_scales", dev, rows * (cols // 128), _F32)
    fp8 = torch.empty(rows, cols, dtype=_U8, device=dev) if fp8 is None else fp8
    fp8_scales = (torch.empty(rows, cols // 128, dtype=_F32, device=dev)
                  if fp8_scales is None else fp8_scales)
    call("fp4_to_fp8_row", _ptr(packed), _ptr(scales), rows, cols, _ptr(fp8), _ptr(fp8_scales),
         _stream(dev))
    return fp8, fp8_scales


def fp4_seg_scale_offsets(row_off: torch.Tensor) -> torch.Tensor:
    """Host helper: running sum of ceil(n_e / 128) (CPU int64 in and out)."""
    ro = row_off.to(device="cpu", dtype=torch.int64).contiguous()
    if ro.dim() != 1 or ro.numel() < 1:
        raise ValueError("row_off must be a 1-D list of E + 1 offsets")
    out = torch.empty_like(ro)
    call("fp4_seg_scale_offsets", ro.data_ptr(), ro.numel() - 1, out.data_ptr())
    return out


class Segments:
    """Ragged expert segments: row offsets (host int64 [E+1]) with their
    scale-block offsets, both uploaded once to the device."""

    def __init__(self, row_off: torch.Tensor, device):
        self.row_off_host = row_off.to(device="cpu", dtype=torch.int64).contiguous()
        self.scale_off_host = fp4_seg_scale_offsets(self.row_off_host)
        if int(self.row_off_host[0]) != 0:
            raise ValueError("row_off[0] must be 0")
        self.row_off = self.row_off_host.to(device)
        self.scale_off = self.scale_off_host.to(device)
        self.num_segments = self.row_off_host.numel() - 1
        self.total_rows = int(self.row_off_host[-1])
        self.total_blocks = int(self.scale_off_host[-1])
        self.device = self.row_off.device


def fp4_to_fp8_col(packed: torch.Tensor, scales: torch.Tensor, segments: Segments,
                   fp8_t: Optional[torch.Tensor] = None,
                   fp8_t_scales: Optional[torch.Tensor] = None, run_blocks: int = 0):
    """Per segment e: [cols, n_e] E4M3 at fp8_t[cols*row_off[e]:] and
    [cols, ceil(n_e/128)] fp32 scales at fp8_t_scales[cols*scale_off[e]:]
    (flat outputs).  The segments must cover exactly the rows of packed.
    run_blocks fixes the token blocks per CTA work unit (0: the library's
    choice); the output does not depend on it."""
    if not 0 <= int(run_blocks) <= 1 << 20:
        raise ValueError(f"run_blocks must be in [0, 2^20], got {run_blocks}")
    rows, cols, dev = _mx_source(packed, scales)
    if segments.total_rows != rows:
        raise ValueError(f"the segments cover {segments.total_rows} rows, packed has {rows}")
    if segments.device != dev:
        raise ValueError(f"the segments are on {segments.device}, packed on {dev}")
    _expect(fp8_t, "fp8_t", dev, cols * segments.total_rows, _U8)
    _expect(fp8_t_scales, "fp8_t_scales", dev, cols * segments.total_blocks, _F32)
    fp8_t = (torch.empty(cols * segments.total_rows, dtype=_U8, device=dev)
             if fp8_t is None else fp8_t)
    fp8_t_scales = (torch.empty(cols * segments.total_blocks, dtype=_F32, device=dev)
                    if fp8_t_scales is None else fp8_t_scales)
    if run_blocks:
        call("fp4_to_fp8_col_runs", _ptr(packed), _ptr(scales), cols, _ptr(segments.row_off),
             _ptr(segments.scale_off), segments.num_segments, segments.total_rows,
             segments.total_blocks, int(run_blocks), _ptr(fp8_t), _ptr(fp8_t_scales),
             _stream(dev))
    else:
        call("fp4_to_fp8_col", _ptr(packed), _ptr(scales), cols, _ptr(segments.row_off),
             _ptr(segments.scale_off), segments.num_segments, segments.total_rows,
             segments.total_blocks, _ptr(fp8_t), _ptr(fp8_t_scales), _stream(dev))
    return fp8_t, fp8_t_scales


# --------------------------------------------------------------- FP4Quant

def _group_ok(group: int, cols: int) -> None:
    if group not in (64, 128, 256):
        raise ValueError(f"group must be 64, 128 or 256, got {group}")
    if cols % group != 0:
        raise ValueError(f"cols ({cols}) must be a multiple of the group ({group})")


def fp4quant_encode(x: torch.Tensor, group: int, packed: Optional[torch.Tensor] = None,
                    s1: Optional[torch.Tensor] = None, s2: Optional[torch.Tensor] = None):
    """x [rows, cols] -> (packed uint8[rows, cols/2], s1, s2 fp32[rows, cols/group])."""
    rows, cols = _matrix(x, "x")
    dt = _dtype(x, "x")
    _group_ok(group, cols)
    dev = x.device
    _expect(packed, "packed", dev, rows * (cols // 2), _U8)
    _expect(s1, "s1", dev, rows * (cols // group), _F32)
    _expect(s2, "s2", dev, rows * (cols // group), _F32)
    packed = torch.empty(rows, cols // 2, dtype=_U8, device=dev) if packed is None else packed
    s1 = torch.empty(rows, cols // group, dtype=_F32, device=dev) if s1 is None else s1
    s2 = torch.empty(rows, cols // group, dtype=_F32, device=dev) if s2 is None else s2
    call("fp4quant_encode", _ptr(x), dt, rows, cols, group, _ptr(packed), _ptr(s1), _ptr(s2),
         _stream(dev))
    return packed, s1, s2


def fp4quant_decode(packed: torch.Tensor, s1: torch.Tensor, s2: torch.Tensor, group: int,
                    out_dtype: torch.dtype = torch.bfloat16,
                    out: Optional[torch.Tensor] = None) -> torch.Tensor:
    rows, half = _matrix(packed, "packed")
    cols = 2 * half
    _group_ok(group, cols)
    dev = packed.device
    odt = _out_dtype(out_dtype)
    _expect(packed, "packed", dev, rows * half, _U8)
    if s1 is None or s2 is None:
        raise ValueError("s1 and s2 are required")
    _expect(s1, "s1", dev, rows * (cols // group), _F32)
    _expect(s2, "s2", dev, rows * (cols // group), _F32)
    _expect(out, "out", dev, rows * cols, out_dtype)
    out = torch.empty(rows, cols, dtype=out_dtype, device=dev) if out is None else out
    call("fp4quant_decode", _ptr(packed), _ptr(s1), _ptr(s2), rows, cols, group, _ptr(out),
         odt, _stream(dev))
    return out


def kernel_launches() -> int:
    return int(_lib.lib().fp4_kernel_launches())


def wait_timeouts() -> int:
    """Bounded waits in the library's kernels that gave up (0 in a healthy
    run; see fp4_wait_timeouts in the C header)."""
    return int(_lib.lib().fp4_wait_timeouts())
