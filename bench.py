"""Benchmark of the block-scaled FP4 codec on one GB300 (or N independent
replicas under torchrun).

One step runs every kernel of the codec once on its workload:
  nvfp4_roundtrip   fp32 [1024, 1024]: amax, quantize (RTN), dequantize -> fp32
  fp4quant_acts     bf16 [16384, 4096], G = 64, 128, 256: encode, decode -> bf16
  nvfp4_train       bf16 W [6144, 2048] + fp32 G_t + fp32 residual: amax pass,
                    fused qdq step (stochastic rounding + error feedback); step
                    k of the bench is training step t = k mod 100 of the
                    100-step schedule, with its own gradient G_t (seed + 1 + t,
                    all 100 drawn once, before timing, and resident in HBM)
  moe_tokens        bf16 [32768, 7168] -> MXFP4; the top-8 dispatch of 262144
                    rows (gathered once, outside the timed region) -> FP8 E4M3
                    row form and ragged column form
  qwen3_8b_weights  252 bf16 matrices (6.95 G weights): amax, quantize (RTN),
                    dequantize -> bf16
The step's order keeps every consumer away from its producer: the FP4Quant
decodes and the qdq pass run after the MoE kernels (about 2.5 GB of other
traffic), so no kernel reads another's output, or its own input, from the
129 MB L2.  Inputs are resident in HBM and the step touches ~58 GB.

Timing: the step loop is bracketed by CUDA events (value, ms_per_step).  The
per-kernel figures (`kernels`, `roofline`) come from a second pass in which
L2 is flushed before every kernel group: a 512 MB buffer (four times L2) is
written and then read back, outside the group's events, so the group starts
with no line of its inputs in L2 and no dirty line of earlier work left to
write back.  Beside each group's figure, `copy_same_bytes` is a plain device
copy of the same number of bytes per launch, timed the same way: the
ceiling of a memory-bound kernel at that size (launches up to 4 GB).

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantize/dequantize GB/s per kernel and % of GB300 HBM peak, 1 GPU"
WORKLOAD = "fp4_codec_suite"
HBM_FALLBACK_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--small", action="store_true",
                   help="reduced shapes (a quick check, not a bench value)")
    p.add_argument("--kernel", metavar="NAME",
                   help="time one kernel alone on a tensor of --size-mb input (a kernel "
                        "study for profiling; prints its own JSON line)")
    p.add_argument("--size-mb", type=float, default=1024.0)
    p.add_argument("--sweep", action="store_true",
                   help="NVFP4 amax / quantize / dequantize over the 1 MiB - 4 GiB size sweep "
                        "of the weight-set workload, one JSON line per kernel and size")
    p.add_argument("--quality", action="store_true",
                   help="print the FP4 quality table (zero share, average error) of the four "
                        "methods on layer-18-shaped synthetic weights, one JSON line per matrix")
    p.add_argument("--train-report", action="store_true",
                   help="run the training workload's 100 steps under SR+EF, RTN+EF and RTN and "
                        "print the share of weights changed per step and the drift of mean(W) "
                        "against the fp32 reference, one JSON line per mode")
    p.add_argument("--source-hash", metavar="GROUP",
                   help="print the source hash a traffic figure of GROUP must carry")
    p.add_argument("--summarize-launches", metavar="CSV",
                   help="print a per-kernel table of an ncu gpu__time_duration.sum launch list "
                        "(this library's kernels, last --steps steps) and exit")
    return p.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


# --------------------------------------------------------------- workload

class Group:
    """One kernel (entry point) on one workload: `launches` calls per step,
    `bytes_per_launch` algorithmic bytes each."""

    def __init__(self, kernel, workload, bytes_per_launch, calls):
        self.kernel = kernel
        self.workload = workload
        self.bytes_per_launch = bytes_per_launch
        self.calls = calls          # list of zero-arg callables
        self.times_ms = []
        self.copy_ms = None         # size-matched copy (copy_at_sizes), when timed

    @property
    def name(self):
        return f"{self.kernel}@{self.workload}"

    @property
    def bytes_per_step(self):
        return self.bytes_per_launch * len(self.calls)


TRAIN_STEPS = 100  # the training workload's schedule: 100 steps, G_t from seed + 1 + t


def build_suite(device, rank=0, small=False, host_inputs=False):
    """Allocate inputs and outputs on `device` and return (groups, state).
    The groups are in step order (see the module docstring)."""
    import torch
    import block_scaled_fp4_e2m1_gb300 as m
    from block_scaled_fp4_e2m1_gb300 import workloads as W

    seed = 1000 * rank
    by = {}
    st = {}
    f32, bf16, u8 = torch.float32, torch.bfloat16, torch.uint8

    def zeros(shape, dt):
        return torch.empty(shape, dtype=dt, device=device)

    def add(g):
        by[g.name] = g
        return g

    # nvfp4_roundtrip: fp32 [1024, 1024]
    x1 = W.nvfp4_roundtrip(seed=seed, device=device).view(-1)
    n1 = x1.numel()
    a1, t1 = zeros(1, f32), zeros(1, f32)
    p1, s1, y1 = zeros(n1 // 2, u8), zeros(n1 // 16, u8), zeros(n1, f32)
    add(Group("nvfp4_amax", "nvfp4_roundtrip", 4 * n1, [lambda: m.nvfp4_amax(x1, amax_ws=a1)]))
    add(Group("nvfp4_quantize", "nvfp4_roundtrip", n1 * (4 + 0.5 + 1 / 16),
              [lambda: m.nvfp4_quantize(x1, tscale="from_amax", amax_ws=a1, tensor_scale=t1,
                                        packed=p1, scales=s1)]))
    add(Group("nvfp4_dequantize", "nvfp4_roundtrip", n1 * (0.5 + 1 / 16 + 4),
              [lambda: m.nvfp4_dequantize(p1, s1, t1, (n1,), f32, out=y1)]))

    # fp4quant_acts: bf16 [16384, 4096]
    T2, H2 = (1024, 4096) if small else (16384, 4096)
    x2 = W.fp4quant_acts(seed=seed, tokens=T2, hidden=H2, device=device)
    n2 = x2.numel()
    fq_out = []
    for G in (64, 128, 256):
        pk, q1, q2 = zeros((T2, H2 // 2), u8), zeros((T2, H2 // G), f32), zeros((T2, H2 // G), f32)
        yy = zeros((T2, H2), bf16)
        fq_out += [pk, q1, q2, yy]
        b = n2 * (2 + 0.5 + 8 / G)
        add(Group(f"fp4quant_encode_g{G}", "fp4quant_acts", b,
                  [lambda G=G, pk=pk, q1=q1, q2=q2: m.fp4quant_encode(x2, G, pk, q1, q2)]))
        add(Group(f"fp4quant_decode_g{G}", "fp4quant_acts", b,
                  [lambda G=G, pk=pk, q1=q1, q2=q2, yy=yy:
                   m.fp4quant_decode(pk, q1, q2, G, bf16, out=yy)]))

    # nvfp4_train: bf16 W [6144, 2048]; bench step k is training step
    # t = k mod 100 with its own gradient G_t, all drawn before timing
    shp3 = (6144, 2048)
    w3 = W.nvfp4_train_weight(seed=seed, shape=shp3, device=device).view(-1)
    n3 = w3.numel()
    ng = 10 if small else TRAIN_STEPS
    gbank = [W.nvfp4_train_grad(seed, t, shape=shp3, device=device).view(-1) for t in range(ng)]
    r3 = torch.zeros(n3, dtype=f32, device=device)
    a3, t3 = zeros(1, f32), zeros(1, f32)
    p3, s3 = zeros(n3 // 2, u8), zeros(n3 // 16, u8)
    st["train_step"] = [0]
    st["g_override"] = None   # the end-to-end run feeds its uploaded gradient here

    def cur_g():
        if st["g_override"] is not None:
            return st["g_override"]
        return gbank[st["train_step"][0] % ng]

    def qdq_amax():
        m.nvfp4_qdq_amax(w3, cur_g(), 1e-4, r3, amax_ws=a3)

    def qdq():
        k = st["train_step"][0]
        m.nvfp4_qdq(w3, cur_g(), 1e-4, r3, rounding="sr", seed=seed, step=k % ng,
                    tscale="from_amax", amax_ws=a3, tensor_scale=t3, packed=p3, scales=s3)
        st["train_step"][0] = k + 1

    add(Group("nvfp4_qdq_amax", "nvfp4_train", n3 * (2 + 4 + 4), [qdq_amax]))
    add(Group("nvfp4_qdq", "nvfp4_train", n3 * (10 + 2 + 4 + 0.5 + 1 / 16), [qdq]))

    # moe_tokens: bf16 [32768, 7168], top-8 of 256 Zipf experts
    T4, H4, E4 = (2048, 7168, 256) if small else (32768, 7168, 256)
    x4 = W.moe_tokens(seed=seed, tokens=T4, hidden=H4, device=device)
    row_token, row_off = W.moe_routing(seed=seed, tokens=T4, experts=E4)
    mp, ms = m.mxfp4_quantize(x4)
    idx = row_token.to(device)
    dp = mp.index_select(0, idx).contiguous()     # dispatch gather: setup, untimed
    ds = ms.index_select(0, idx).contiguous()
    del idx
    R4 = dp.shape[0]
    segs = m.Segments(row_off, device)
    f8, f8s = zeros((R4, H4), u8), zeros((R4, H4 // 128), f32)
    ft, fts = zeros(H4 * R4, u8), zeros(H4 * segs.total_blocks, f32)
    n4 = x4.numel()
    add(Group("mxfp4_quantize", "moe_tokens", n4 * (2 + 0.5 + 1 / 32),
              [lambda: m.mxfp4_quantize(x4, mp, ms)]))
    nd = R4 * H4
    add(Group("fp4_to_fp8_row", "moe_tokens", nd * (0.5 + 1 / 32 + 1 + 4 / 128),
              [lambda: m.fp4_to_fp8_row(dp, ds, f8, f8s)]))
    add(Group("fp4_to_fp8_col", "moe_tokens", nd * (0.5 + 1 / 32 + 1) + 4 * H4 * segs.total_blocks,
              [lambda: m.fp4_to_fp8_col(dp, ds, segs, ft, fts)]))

    # qwen3_8b_weights: 252 Laplace bf16 matrices, one batched launch per pass
    shapes = W.qwen3_8b_weight_shapes(layers=2 if small else 36)
    mats, pk5, sc5, out5 = [], [], [], []
    for i, (r, c) in enumerate(shapes):
        w = W.laplace_weight(seed + i, (r, c), device=device).view(-1)
        mats.append(w)
        pk5.append(zeros(r * c // 2, u8))
        sc5.append(zeros(r * c // 16, u8))
        out5.append(zeros(r * c, bf16))
    k5 = len(mats)
    amax5, ts5 = zeros(k5, f32), zeros(k5, f32)
    qbatch = m.Batch(xs=mats, packed=pk5, scales=sc5)
    dbatch = m.Batch(packed=pk5, scales=sc5, ys=out5, sizes=[w.numel() for w in mats])
    n5 = sum(w.numel() for w in mats)
    add(Group("nvfp4_amax", "qwen3_8b_weights", 2 * n5,
              [lambda: m.nvfp4_amax_batched(qbatch, bf16, amax=amax5)]))
    add(Group("nvfp4_quantize", "qwen3_8b_weights", n5 * (2 + 0.5 + 1 / 16),
              [lambda: m.nvfp4_quantize_batched(qbatch, bf16, tscale="from_amax",
                                                tensor_scale=ts5, amax=amax5)]))
    add(Group("nvfp4_dequantize", "qwen3_8b_weights", n5 * (0.5 + 1 / 16 + 2),
              [lambda: m.nvfp4_dequantize_batched(dbatch, ts5, bf16)]))
    st["elements"] = {"nvfp4_roundtrip": n1, "fp4quant_acts": n2, "nvfp4_train": n3,
                      "moe_tokens": n4, "moe_dispatched": nd, "qwen3_8b_weights": n5}

    order = (["nvfp4_amax@nvfp4_roundtrip", "nvfp4_quantize@nvfp4_roundtrip",
              "nvfp4_dequantize@nvfp4_roundtrip"] +
             [f"fp4quant_encode_g{G}@fp4quant_acts" for G in (64, 128, 256)] +
             ["nvfp4_qdq_amax@nvfp4_train", "mxfp4_quantize@moe_tokens",
              "fp4_to_fp8_row@moe_tokens", "fp4_to_fp8_col@moe_tokens"] +
             [f"fp4quant_decode_g{G}@fp4quant_acts" for G in (64, 128, 256)] +
             ["nvfp4_qdq@nvfp4_train", "nvfp4_amax@qwen3_8b_weights",
              "nvfp4_quantize@qwen3_8b_weights", "nvfp4_dequantize@qwen3_8b_weights"])
    assert sorted(order) == sorted(by)
    groups = [by[k] for k in order]

    # The same work cut into stages for the end-to-end pipeline: each stage
    # has its inputs, its calls and its outputs.  The weight set goes in
    # chunks of whole layers (each chunk one batched launch per pass), so
    # that one chunk's upload, another's kernels and a third's download can
    # overlap.  The training stage uploads its gradient into g_e2e.
    calls = lambda *names: [by[nm].calls[0] for nm in names]
    g_e2e = zeros(n3, f32)
    st["g_e2e"] = g_e2e
    stages = [([x1], calls("nvfp4_amax@nvfp4_roundtrip", "nvfp4_quantize@nvfp4_roundtrip",
                           "nvfp4_dequantize@nvfp4_roundtrip"), [p1, s1, y1, t1])]
    stages.append(([x2], [c for G in (64, 128, 256)
                          for c in calls(f"fp4quant_encode_g{G}@fp4quant_acts",
                                         f"fp4quant_decode_g{G}@fp4quant_acts")], fq_out))
    stages.append(([w3, g_e2e, r3], [qdq_amax, qdq], [w3, r3, p3, s3, t3]))
    stages.append(([x4, dp, ds], calls("mxfp4_quantize@moe_tokens", "fp4_to_fp8_row@moe_tokens",
                                       "fp4_to_fp8_col@moe_tokens"),
                   [mp, ms, f8, f8s, ft, fts]))
    per_layer = 7
    layers = k5 // per_layer
    chunk_layers = max(1, min(4, layers))
    for l0 in range(0, layers, chunk_layers):
        i0, i1 = l0 * per_layer, min(k5, (l0 + chunk_layers) * per_layer)
        qb = m.Batch(xs=mats[i0:i1], packed=pk5[i0:i1], scales=sc5[i0:i1])
        db = m.Batch(packed=pk5[i0:i1], scales=sc5[i0:i1], ys=out5[i0:i1],
                     sizes=[w.numel() for w in mats[i0:i1]])
        am, ts = amax5[i0:i1], ts5[i0:i1]
        stages.append((mats[i0:i1],
                       [lambda qb=qb, am=am: m.nvfp4_amax_batched(qb, bf16, amax=am),
                        lambda qb=qb, am=am, ts=ts: m.nvfp4_quantize_batched(
                            qb, bf16, tscale="from_amax", tensor_scale=ts, amax=am),
                        lambda db=db, ts=ts: m.nvfp4_dequantize_batched(db, ts, bf16)],
                       pk5[i0:i1] + sc5[i0:i1] + out5[i0:i1] + [ts]))
    st["stages"] = stages
    st["gbank0"] = gbank[0]
    return groups, st


class L2Flush:
    """Leaves L2 holding only clean lines of a 512 MB buffer (four times the
    129 MB L2): the buffer is written, which evicts everything, then read
    back, which writes the dirty lines to HBM.  The next kernel therefore
    finds none of its inputs in L2 and pays for no earlier work's
    write-backs."""

    def __init__(self, device, nbytes=512 << 20):
        import torch
        self.buf = torch.empty(nbytes // 8, dtype=torch.int64, device=device)
        self.sink = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        import torch
        self.buf.zero_()
        torch.sum(self.buf, dim=0, out=self.sink)


COPY_MAX_BYTES = 4 << 30  # size-matched copies only for launches up to this many bytes


def copy_at_sizes(nbytes, device, passes, flush):
    """Median CUDA-event time (ms) of a plain device copy moving each of the
    byte counts in `nbytes` (half read, half written: torch's bf16 copy_,
    the kernel behind the measured copy bandwidth), timed as the kernels
    are: L2 flushed before every launch, events around it.  It is the
    ceiling of a memory-bound kernel at that size: at tens of MB the fixed
    cost of a launch (launch, CTA ramp, the first loads' latency, the tail)
    is a visible share of it.  Returns {nbytes: ms}."""
    import torch
    sizes = sorted({int(b) for b in nbytes if 0 < b <= COPY_MAX_BYTES})
    if not sizes:
        return {}
    elems = {b: max(8, b // 4 // 8 * 8) for b in sizes}  # bf16 elements copied
    top = max(elems.values())
    src = torch.ones(top, dtype=torch.bfloat16, device=device)
    dst = torch.empty_like(src)
    out = {}
    for b in sizes:
        k = elems[b]
        s, d = src[:k], dst[:k]
        d.copy_(s)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(passes)]
        for p in range(passes):
            flush()
            ev[p][0].record()
            d.copy_(s)
            ev[p][1].record()
        torch.cuda.synchronize()
        out[b] = statistics.median(a.elapsed_time(e) for a, e in ev)
    del src, dst
    return out


def run_step(groups, events):
    import torch
    for gi, g in enumerate(groups):
        if events is not None:
            events[gi][0].record()
        for c in g.calls:
            c()
        if events is not None:
            events[gi][1].record()


# ------------------------------------------------------------------ clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- CPU side

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


_ORACLE_INPUTS = {}


def _cached(key, make):
    """Inputs of the CPU baseline, drawn once per process and size."""
    if key not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[key] = make()
    return _ORACLE_INPUTS[key]


def cpu_oracle_rates(big_mb=256.0, small_scale=1.0, parallel=True):
    """Time the CPU oracle (plain single-threaded C) on bounded slices of each
    kernel's workload.  Returns (single, multi, sample, cores): GB/s per
    group on one core, GB/s per group with the slice's rows split over
    `cores` threads (each thread runs the same C oracle on its rows; the
    ctypes calls release the GIL), a description of the slices, and the
    thread count.  The weight-set and MoE slices hold big_mb MB of input;
    the others are scaled by small_scale.  Quantize passes take the tensor
    scale as given (computed before timing), as the bench's quantize
    kernels take it from the preceding amax pass."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import torch
    import oracle as ora
    from block_scaled_fp4_e2m1_gb300 import workloads as W

    ora.build()
    cores = host_cores() if parallel else 1
    pool = ThreadPoolExecutor(max_workers=cores) if cores > 1 else None
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    single, multi = {}, {}

    def parts(n, unit):
        """[a, b) ranges of n rows (multiples of unit) over `cores` threads."""
        k = max(1, min(cores, n // unit))
        cuts = [((n // unit) * i // k) * unit for i in range(k)] + [n]
        return list(zip(cuts, cuts[1:]))

    def timed(name, nbytes, fn, part_fn=None, ranges=None):
        t0 = time.perf_counter()
        reps = 0
        while True:   # tiny slices repeat up to ~0.2 s
            fn()
            reps += 1
            el = time.perf_counter() - t0
            if el >= 0.2 or reps >= 20:
                break
        single[name] = nbytes * reps / el / 1e9
        if pool is not None and part_fn is not None:
            t0 = time.perf_counter()
            list(pool.map(lambda ab: part_fn(*ab), ranges))
            multi[name] = nbytes / (time.perf_counter() - t0) / 1e9

    G_ = ora.TSCALE_GIVEN
    # nvfp4 round-trip: fp32 [1024 * small_scale, 1024]
    r1 = max(16, int(1024 * small_scale))
    x = _cached(("x1", r1), lambda: W.nvfp4_roundtrip(seed=0, shape=(r1, 1024)).numpy().ravel())
    n = x.size
    ts = ora.nvfp4_tensor_scale(ora.nvfp4_amax(x))
    rg = parts(n, 4096)
    timed("nvfp4_amax@nvfp4_roundtrip", 4 * n, lambda: ora.nvfp4_amax(x),
          lambda a, b: ora.nvfp4_amax(x[a:b]), rg)
    pq = ora.nvfp4_quantize(x, tscale_mode=G_, tensor_scale=ts)
    timed("nvfp4_quantize@nvfp4_roundtrip", 4.5625 * n,
          lambda: ora.nvfp4_quantize(x, tscale_mode=G_, tensor_scale=ts),
          lambda a, b: ora.nvfp4_quantize(x[a:b], tscale_mode=G_, tensor_scale=ts), rg)
    timed("nvfp4_dequantize@nvfp4_roundtrip", 4.5625 * n,
          lambda: ora.nvfp4_dequantize(pq[0], pq[1], ts, n),
          lambda a, b: ora.nvfp4_dequantize(pq[0][a // 2:b // 2], pq[1][a // 16:b // 16], ts,
                                            b - a), rg)
    # FP4Quant activations: [1024 * small_scale, 4096] tokens
    t2 = max(16, int(1024 * small_scale))
    a = _cached(("a2", t2),
                lambda: ora.bf16_to_f32(bits(W.fp4quant_acts(seed=0, tokens=t2, hidden=4096))))
    rg = parts(t2, 1)
    for G in (64, 128, 256):
        enc = ora.fp4quant_encode(a, G)
        b_ = a.size * (2.5 + 8 / G)
        timed(f"fp4quant_encode_g{G}@fp4quant_acts", b_, lambda: ora.fp4quant_encode(a, G),
              lambda i, j: ora.fp4quant_encode(a[i:j], G), rg)
        timed(f"fp4quant_decode_g{G}@fp4quant_acts", b_, lambda: ora.fp4quant_decode(*enc, G),
              lambda i, j: ora.fp4quant_decode(enc[0][i:j], enc[1][i:j], enc[2][i:j], G), rg)
    # training step: [512 * small_scale, 2048] of W, G_0, r
    r3 = max(16, int(512 * small_scale))
    w = _cached(("w3", r3), lambda: bits(W.nvfp4_train_weight(seed=0, shape=(r3, 2048)))
                .ravel().copy())
    g = _cached(("g3", r3), lambda: W.nvfp4_train_grad(0, 0, shape=(r3, 2048)).numpy().ravel())
    r = np.zeros(w.size, np.float32)
    ts3 = ora.nvfp4_tensor_scale(ora.nvfp4_qdq_amax(w, g, 1e-4, r))
    rg = parts(w.size, 4096)
    timed("nvfp4_qdq_amax@nvfp4_train", 10 * w.size, lambda: ora.nvfp4_qdq_amax(w, g, 1e-4, r),
          lambda i, j: ora.nvfp4_qdq_amax(w[i:j], g[i:j], 1e-4, r[i:j]), rg)
    timed("nvfp4_qdq@nvfp4_train", 16.5625 * w.size,
          lambda: ora.nvfp4_qdq(w, g, 1e-4, r, rounding=ora.SR, tscale_mode=G_,
                                tensor_scale=ts3),
          lambda i, j: ora.nvfp4_qdq(w[i:j], g[i:j], 1e-4, r[i:j], rounding=ora.SR,
                                     tscale_mode=G_, tensor_scale=ts3), rg)
    # MoE: big_mb MB of bf16 tokens; then big_mb MB of dispatched MXFP4 rows
    # (0.53125 B per element), cut into expert segments of the workload's
    # mean length (1024 rows)
    t4 = max(8, int(big_mb * 1e6 / (2 * 7168)))
    t = _cached(("t4", t4),
                lambda: ora.bf16_to_f32(bits(W.moe_tokens(seed=0, tokens=t4, hidden=7168))))
    timed("mxfp4_quantize@moe_tokens", t.size * 2.53125, lambda: ora.mxfp4_quantize(t),
          lambda i, j: ora.mxfp4_quantize(t[i:j]), parts(t4, 1))
    rd = max(128, int(big_mb * 1e6 / (0.53125 * 7168)))

    def dispatched():
        mp, ms = ora.mxfp4_quantize(t)
        reps = -(-rd // t4)
        return (np.ascontiguousarray(np.tile(mp, (reps, 1))[:rd]),
                np.ascontiguousarray(np.tile(ms, (reps, 1))[:rd]))

    dp, dsc = _cached(("d4", t4, rd), dispatched)
    nd = rd * 7168
    timed("fp4_to_fp8_row@moe_tokens", nd * 1.5625, lambda: ora.fp4_to_fp8_row(dp, dsc),
          lambda i, j: ora.fp4_to_fp8_row(dp[i:j], dsc[i:j]), parts(rd, 1))
    off = np.array(list(range(0, rd, 1024)) + [rd], np.int64)
    segs = list(zip(off[:-1], off[1:]))
    seg_ranges = parts(len(segs), 1)

    def col_part(i, j):
        for a_, b_ in segs[i:j]:
            ora.fp4_to_fp8_col_segment(dp, dsc, int(a_), int(b_ - a_))

    timed("fp4_to_fp8_col@moe_tokens", nd * 1.5625, lambda: ora.fp4_to_fp8_col(dp, dsc, off),
          col_part, seg_ranges)
    # weight set: big_mb MB of one Laplace matrix [., 4096]
    r5 = max(16, int(big_mb * 1e6 / (2 * 4096)))
    wq = _cached(("w5", r5), lambda: ora.bf16_to_f32(bits(W.laplace_weight(0, (r5, 4096)))).ravel())
    nq = wq.size
    ts5 = ora.nvfp4_tensor_scale(ora.nvfp4_amax(wq))
    rg = parts(nq, 4096)
    timed("nvfp4_amax@qwen3_8b_weights", 2 * nq, lambda: ora.nvfp4_amax(wq),
          lambda i, j: ora.nvfp4_amax(wq[i:j]), rg)
    pw = ora.nvfp4_quantize(wq, tscale_mode=G_, tensor_scale=ts5)
    timed("nvfp4_quantize@qwen3_8b_weights", 2.5625 * nq,
          lambda: ora.nvfp4_quantize(wq, tscale_mode=G_, tensor_scale=ts5),
          lambda i, j: ora.nvfp4_quantize(wq[i:j], tscale_mode=G_, tensor_scale=ts5), rg)
    timed("nvfp4_dequantize@qwen3_8b_weights", 2.5625 * nq,
          lambda: ora.nvfp4_dequantize(pw[0], pw[1], ts5, nq),
          lambda i, j: ora.nvfp4_dequantize(pw[0][i // 2:j // 2], pw[1][i // 16:j // 16], ts5,
                                            j - i), rg)
    if pool is not None:
        pool.shutdown()
    mb = lambda v: f"{v / 1e6:.0f} MB"
    sample = (f"the C oracle on slices of each workload: fp32 round-trip [{r1}, 1024], "
              f"activations [{t2}, 4096] per G, training step [{r3}, 2048], MoE tokens "
              f"[{t4}, 7168] ({mb(2 * t4 * 7168)} bf16) and {rd} dispatched MXFP4 rows "
              f"({mb(0.53125 * nd)}, segments of 1024 rows), weights [{r5}, 4096] "
              f"({mb(2 * nq)} bf16); one pass per slice (tiny ones repeated to 0.2 s); "
              f"step GB/s = step bytes / sum over kernels of (kernel bytes / oracle GB/s)")
    return single, multi, sample, cores


def combine_rate(groups, rates):
    total = sum(g.bytes_per_step for g in groups)
    secs = sum(g.bytes_per_step / (rates[g.name] * 1e9) for g in groups)
    return total / secs / 1e9


# ------------------------------------------------------------ reference arm

def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # the step's byte mix (shapes only; nothing allocated)
    groups = suite_shapes()
    steps, warm = max(1, args.steps), max(0, args.warmup)
    # each step: the oracle on slices sized so that the whole run ends in a
    # few minutes (about 150 s of CPU work over all steps)
    # the slices' inputs are drawn once; the oracle then needs about 0.25 s
    # per MB of the large slices on one core
    budget = max(1.0, min(30.0, 120.0 / (steps + warm)))
    big_mb = max(2.0, budget / 0.25)
    small = max(0.02, budget / 60.0)
    vals, walls = [], []
    sample = ""
    for i in range(warm + steps):
        t0 = time.perf_counter()
        rates, _, sample, _ = cpu_oracle_rates(big_mb=big_mb, small_scale=small, parallel=False)
        wall = time.perf_counter() - t0
        if i >= warm:
            vals.append(combine_rate(groups, rates))
            walls.append(wall)
    v = statistics.median(vals)
    full_ms = sum(g.bytes_per_step for g in groups) / (v * 1e9) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": round(statistics.median(walls) * 1e3, 1),
        "ms_per_step_kind": ("measured wall time of one sampled step: the oracle on a slice "
                             "of every kernel's workload (the slices are drawn once, in the "
                             "first warm-up step)"),
        "full_step_ms_extrapolated": round(full_ms, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": WORKLOAD},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "host_cores": host_cores(), "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def suite_shapes():
    """Groups with the byte counts of the full workload, without allocating."""
    from block_scaled_fp4_e2m1_gb300 import workloads as W
    gs = []
    n1 = 1024 * 1024
    gs += [Group("nvfp4_amax", "nvfp4_roundtrip", 4 * n1, [None]),
           Group("nvfp4_quantize", "nvfp4_roundtrip", 4.5625 * n1, [None]),
           Group("nvfp4_dequantize", "nvfp4_roundtrip", 4.5625 * n1, [None])]
    n2 = 16384 * 4096
    for G in (64, 128, 256):
        gs += [Group(f"fp4quant_encode_g{G}", "fp4quant_acts", n2 * (2.5 + 8 / G), [None]),
               Group(f"fp4quant_decode_g{G}", "fp4quant_acts", n2 * (2.5 + 8 / G), [None])]
    n3 = 6144 * 2048
    gs += [Group("nvfp4_qdq_amax", "nvfp4_train", 10 * n3, [None]),
           Group("nvfp4_qdq", "nvfp4_train", 16.5625 * n3, [None])]
    n4 = 32768 * 7168
    nd = 8 * n4
    gs += [Group("mxfp4_quantize", "moe_tokens", 2.53125 * n4, [None]),
           Group("fp4_to_fp8_row", "moe_tokens", 1.5625 * nd, [None]),
           Group("fp4_to_fp8_col", "moe_tokens", 1.5625 * nd, [None])]
    n5 = sum(r * c for r, c in W.qwen3_8b_weight_shapes())
    gs += [Group("nvfp4_amax", "qwen3_8b_weights", 2 * n5, [None]),
           Group("nvfp4_quantize", "qwen3_8b_weights", 2.5625 * n5, [None]),
           Group("nvfp4_dequantize", "qwen3_8b_weights", 2.5625 * n5, [None])]
    return gs


# --------------------------------------------------------------------- ours

def host_mem_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except Exception:
        pass
    return 0


def e2e_measure(groups, st, steps, warmup, device):
    """Whole step through the public API with host buffers: every step copies
    all inputs host -> device from pinned memory, runs the kernels and copies
    all outputs back.  The step is a three-stream pipeline over its stages
    (build_suite): uploads on one copy stream, the kernels on the compute
    stream, downloads on a second copy stream.  Events order each stage's
    upload -> kernels -> download, so the two copy directions and the
    kernels of different stages overlap.  The timed region ends when every
    download has landed in host memory."""
    import torch
    stages = st["stages"]
    seen = set()
    uniq = lambda ts: [t for t in ts if not (t.data_ptr() in seen or seen.add(t.data_ptr()))]
    ins = [uniq(s_in) for s_in, _, _ in stages]
    seen = set()
    outs = [uniq(s_out) for _, _, s_out in stages]
    h2d = sum(t.numel() * t.element_size() for ts in ins for t in ts)
    d2h = sum(t.numel() * t.element_size() for ts in outs for t in ts)
    if host_mem_available() < 1.5 * (h2d + d2h):
        return None, h2d, d2h
    st["g_e2e"].copy_(st["gbank0"])
    st["g_override"] = st["g_e2e"]
    h_in = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ts] for ts in ins]
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ts] for ts in outs]
    for hs, ts in zip(h_in, ins):
        for h, t in zip(hs, ts):
            h.copy_(t)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    comp = torch.cuda.current_stream(device)
    torch.cuda.synchronize()
    times = []
    for i in range(warmup + steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ready = []
        with torch.cuda.stream(up):
            for hs, ts in zip(h_in, ins):
                for h, t in zip(hs, ts):
                    t.copy_(h, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(up)
                ready.append(ev)
        for k, (_, calls, _) in enumerate(stages):
            comp.wait_event(ready[k])
            for c in calls:
                c()
            done = torch.cuda.Event()
            done.record(comp)
            down.wait_event(done)
            with torch.cuda.stream(down):
                for h, t in zip(h_out[k], outs[k]):
                    h.copy_(t, non_blocking=True)
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    # the downloads waited for their kernels: the host copies of the small
    # stages and of the last chunk's tensor scales equal the device tensors
    for k in list(range(min(4, len(stages)))) + [len(stages) - 1]:
        for h, t in zip(h_out[k], outs[k]):
            if t.numel() * t.element_size() <= (256 << 20) and not torch.equal(h.to(device), t):
                raise RuntimeError(f"e2e stage {k}: a downloaded output differs from the device")
    del h_in, h_out
    st["g_override"] = None
    return statistics.median(times), h2d, d2h


def kernel_pass_steps(steps):
    """Steps of the L2-flushed per-kernel pass that follows the timed steps."""
    return max(5, min(steps, 30))


def summarize_launches(path, steps, warmup):
    """Per-kernel launches, total device time and share, from an ncu CSV
    launch list (one gpu__time_duration.sum row per launch), restricted to
    this library's kernels in the last `steps` bench steps."""
    import csv
    import re
    rows = []
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        name = r["Kernel Name"]
        if "fp4::" not in name:
            continue
        m = re.search(r"fp4::(?:<unnamed>|\(anonymous namespace\))::([A-Za-z0-9_]+(?:<[^()]*>)?)", name)
        short = m.group(1) if m else name[:80]
        unit = r.get("Metric Unit", "ns")
        v = float(r["Metric Value"].replace(",", ""))
        ns = v * {"ns": 1.0, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}.get(unit, 1.0)
        rows.append((short, ns, r["Grid Size"], r["Block Size"]))
    # the run is: one setup launch (the MXFP4 quantize feeding the dispatch
    # gather), max(3, warmup) warm-up steps, the timed steps, then the
    # L2-flushed per-kernel pass of kernel_pass_steps(steps) steps
    total = len(rows)
    warm = max(3, warmup)
    nsteps = warm + steps + kernel_pass_steps(steps)
    per_step = (total - 1) // nsteps
    if per_step * nsteps + 1 != total:
        raise ValueError(f"{total} launches do not split into {nsteps} steps + 1")
    sel = rows[1 + warm * per_step:1 + (warm + steps) * per_step]
    agg = {}
    for short, ns, grid, block in sel:
        a = agg.setdefault(short, [0, 0.0, grid, block])
        a[0] += 1
        a[1] += ns
    tot = sum(a[1] for a in agg.values())
    out = ["| kernel | launches | total ms | share | grid | block |", "|---|---|---|---|---|---|"]
    for k, (n, ns, grid, block) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        out.append(f"| `{k}` | {n} | {ns / 1e6:.3f} | {ns / tot:.1%} | {grid} | {block} |")
    out.append(f"| total | {sum(a[0] for a in agg.values())} | {tot / 1e6:.3f} | 100% | | |")
    return "\n".join(out)


KERNEL_STUDIES = ["nvfp4_amax", "nvfp4_quantize", "nvfp4_quantize_sr", "nvfp4_dequantize",
                  "nvfp4_qdq", "mxfp4_quantize", "fp4_to_fp8_row", "fp4_to_fp8_col",
                  "fp4quant_encode_g64", "fp4quant_encode_g128", "fp4quant_encode_g256",
                  "fp4quant_decode_g64", "fp4quant_decode_g128", "fp4quant_decode_g256",
                  "nvfp4_amax_batched", "nvfp4_quantize_batched", "nvfp4_dequantize_batched",
                  "fp8_to_fp4_row", "mxfp4_dequantize", "nvfp4_quantize_blocked",
                  "fp4_scales_to_blocked", "fp4_scales_from_blocked",
                  "nvfp4_quantize_batched_blocked"]


def kernel_study(name, size_mb, steps, warmup, device):
    """One kernel on a bf16 input of ~size_mb MB (the shapes of its bench
    workload, rows scaled), timed per launch with CUDA events, L2 flushed
    (L2Flush) before every launch.  Returns (group, per-launch ms list)."""
    import torch
    import block_scaled_fp4_e2m1_gb300 as m
    from block_scaled_fp4_e2m1_gb300 import workloads as W
    f32, bf16, u8 = torch.float32, torch.bfloat16, torch.uint8
    n = int(size_mb * 1e6 / 2) // 4096 * 4096
    def z(shape, dt):
        return torch.empty(shape, dtype=dt, device=device)
    if name in ("nvfp4_amax", "nvfp4_quantize", "nvfp4_quantize_sr", "nvfp4_dequantize"):
        w = W.laplace_weight(7, (n // 4096, 4096), device=device).view(-1)
        a, t = z(1, f32), z(1, f32)
        pk, sc, y = z(n // 2, u8), z(n // 16, u8), z(n, bf16)
        m.nvfp4_amax(w, amax_ws=a)
        m.nvfp4_quantize(w, tscale="from_amax", amax_ws=a, tensor_scale=t, packed=pk, scales=sc)
        if name == "nvfp4_amax":
            g = Group(name, "study", 2 * n, [lambda: m.nvfp4_amax(w, amax_ws=a)])
        elif name == "nvfp4_dequantize":
            g = Group(name, "study", 2.5625 * n,
                      [lambda: m.nvfp4_dequantize(pk, sc, t, (n,), bf16, out=y)])
        else:
            rnd = "sr" if name.endswith("_sr") else "rtn"
            g = Group(name, "study", 2.5625 * n,
                      [lambda: m.nvfp4_quantize(w, rounding=rnd, tscale="from_amax", amax_ws=a,
                                                tensor_scale=t, packed=pk, scales=sc)])
    elif name == "nvfp4_qdq":
        n3 = n // 4
        w = W.nvfp4_train_weight(seed=0, shape=(n3 // 2048, 2048), device=device).view(-1)
        gr = W.nvfp4_train_grad(0, 0, shape=(n3,), device=device)
        r = torch.zeros(n3, dtype=f32, device=device)
        a, t = z(1, f32), z(1, f32)
        pk, sc = z(n3 // 2, u8), z(n3 // 16, u8)
        m.nvfp4_qdq_amax(w, gr, 1e-4, r, amax_ws=a)
        g = Group(name, "study", 16.5625 * n3,
                  [lambda: m.nvfp4_qdq(w, gr, 1e-4, r, rounding="sr", tscale="from_amax",
                                       amax_ws=a, tensor_scale=t, packed=pk, scales=sc)])
    elif name == "mxfp4_quantize":
        x = W.moe_tokens(seed=0, tokens=n // 7168, hidden=7168, device=device)
        pk, sc = m.mxfp4_quantize(x)
        g = Group(name, "study", 2.53125 * x.numel(), [lambda: m.mxfp4_quantize(x, pk, sc)])
    elif name in ("fp4_to_fp8_row", "fp4_to_fp8_col"):
        T = max(8, n // 7168 // 8)
        x = W.moe_tokens(seed=0, tokens=T, hidden=7168, device=device)
        row_token, row_off = W.moe_routing(seed=0, tokens=T, experts=256)
        mp, ms = m.mxfp4_quantize(x)
        idx = row_token.to(device)
        dp, ds = mp.index_select(0, idx).contiguous(), ms.index_select(0, idx).contiguous()
        del x, mp, ms
        nd = dp.shape[0] * 7168
        if name == "fp4_to_fp8_row":
            f8, fs = m.fp4_to_fp8_row(dp, ds)
            g = Group(name, "study", 1.5625 * nd, [lambda: m.fp4_to_fp8_row(dp, ds, f8, fs)])
        else:
            segs = m.Segments(row_off, device)
            ft, fts = m.fp4_to_fp8_col(dp, ds, segs)
            g = Group(name, "study", nd * (0.5 + 1 / 32 + 1) + 4 * 7168 * segs.total_blocks,
                      [lambda: m.fp4_to_fp8_col(dp, ds, segs, ft, fts)])
    elif name.startswith("fp4quant_"):
        G = int(name.rsplit("_g", 1)[1])
        x = W.fp4quant_acts(seed=0, tokens=n // 4096, hidden=4096, device=device)
        pk, s1, s2 = m.fp4quant_encode(x, G)
        y = torch.empty_like(x)
        b = x.numel() * (2.5 + 8 / G)
        if "encode" in name:
            g = Group(name, "study", b, [lambda: m.fp4quant_encode(x, G, pk, s1, s2)])
        else:
            g = Group(name, "study", b, [lambda: m.fp4quant_decode(pk, s1, s2, G, bf16, out=y)])
    elif name in ("fp8_to_fp4_row", "mxfp4_dequantize"):
        # the backward-path exchange on MoE-shaped gradients: FP8 -> MXFP4 -> bf16
        x = W.moe_tokens(seed=1, tokens=max(8, n // 7168), hidden=7168, device=device)
        pk, sc = m.mxfp4_quantize(x)
        f8, fs = m.fp4_to_fp8_row(pk, sc)
        nd = x.numel()
        if name == "fp8_to_fp4_row":
            g = Group(name, "study", nd * (1 + 4 / 128 + 0.5 + 1 / 32),
                      [lambda: m.fp8_to_fp4_row(f8, fs, pk, sc)])
        else:
            y = torch.empty_like(x)
            g = Group(name, "study", nd * (0.5 + 1 / 32 + 2),
                      [lambda: m.mxfp4_dequantize(pk, sc, bf16, out=y)])
    elif name == "nvfp4_quantize_blocked":
        # a [rows, 4096] bf16 weight matrix, block scales straight into the
        # blocked layout of block-scaled matmuls
        w = W.laplace_weight(7, (n // 4096, 4096), device=device)
        a, t = z(1, f32), z(1, f32)
        pk = z((n // 4096, 2048), u8)
        blk = z(m.fp4_blocked_scales_size(n // 4096, 256), u8)
        m.nvfp4_amax(w.view(-1), amax_ws=a)
        g = Group(name, "study", 2.5 * n + blk.numel(),
                  [lambda: m.nvfp4_quantize_blocked(w, tscale="from_amax", amax_ws=a,
                                                    tensor_scale=t, packed=pk,
                                                    blocked_scales=blk)])
    elif name in ("fp4_scales_to_blocked", "fp4_scales_from_blocked"):
        # the e4m3 scales of a [rows, 4096] weight: [rows, 256] bytes of size_mb MB
        rows = max(128, int(size_mb * 1e6 / 256) // 128 * 128)
        sc = torch.randint(0, 127, (rows, 256), dtype=u8, device=device)
        blk = m.fp4_scales_to_blocked(sc)
        if name == "fp4_scales_to_blocked":
            g = Group(name, "study", sc.numel() + blk.numel(),
                      [lambda: m.fp4_scales_to_blocked(sc, out=blk)])
        else:
            g = Group(name, "study", sc.numel() + blk.numel(),
                      [lambda: m.fp4_scales_from_blocked(blk, rows, 256, out=sc)])
    elif name == "nvfp4_quantize_batched_blocked":
        # whole layers of the weight set, scales straight into the blocked
        # layout of block-scaled matmuls (a GEMM-ready copy of the model)
        layers = max(1, int(round(size_mb / 386.0)))
        shapes = W.qwen3_8b_weight_shapes(layers=layers)
        mats = [W.laplace_weight(100 + i, s, device=device).view(-1) for i, s in enumerate(shapes)]
        nq = sum(w.numel() for w in mats)
        pks = [z(w.numel() // 2, u8) for w in mats]
        blks = [z(m.fp4_blocked_scales_size(r, c // 16), u8) for r, c in shapes]
        qb = m.Batch(xs=mats, packed=pks, scales=blks, ks=[c for _, c in shapes])
        am, ts = z(len(mats), f32), z(len(mats), f32)
        m.nvfp4_amax_batched(qb, bf16, amax=am)
        g = Group(name, "study", 2.5 * nq + sum(b.numel() for b in blks),
                  [lambda: m.nvfp4_quantize_batched_blocked(qb, bf16, tscale="from_amax",
                                                            tensor_scale=ts, amax=am)])
    elif name.endswith("_batched"):
        # whole layers of the Qwen3-8B-shaped set (~386 MB of bf16 per layer)
        layers = max(1, int(round(size_mb / 386.0)))
        mats = [W.laplace_weight(100 + i, s, device=device).view(-1)
                for i, s in enumerate(W.qwen3_8b_weight_shapes(layers=layers))]
        nq = sum(w.numel() for w in mats)
        pks = [z(w.numel() // 2, u8) for w in mats]
        scs = [z(w.numel() // 16, u8) for w in mats]
        ys = [z(w.numel(), bf16) for w in mats]
        qb = m.Batch(xs=mats, packed=pks, scales=scs)
        db = m.Batch(packed=pks, scales=scs, ys=ys, sizes=[w.numel() for w in mats])
        am, ts = z(len(mats), f32), z(len(mats), f32)
        m.nvfp4_amax_batched(qb, bf16, amax=am)
        m.nvfp4_quantize_batched(qb, bf16, tscale="from_amax", tensor_scale=ts, amax=am)
        if name.startswith("nvfp4_amax"):
            g = Group(name, "study", 2 * nq, [lambda: m.nvfp4_amax_batched(qb, bf16, amax=am)])
        elif name.startswith("nvfp4_quantize"):
            g = Group(name, "study", 2.5625 * nq,
                      [lambda: m.nvfp4_quantize_batched(qb, bf16, tscale="from_amax",
                                                        tensor_scale=ts, amax=am)])
        else:
            g = Group(name, "study", 2.5625 * nq, [lambda: m.nvfp4_dequantize_batched(db, ts, bf16)])
    else:
        raise SystemExit(f"unknown kernel {name}; one of {KERNEL_STUDIES}")
    torch.cuda.synchronize()
    for _ in range(max(1, warmup)):
        g.calls[0]()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    flush = L2Flush(device)
    torch.cuda.synchronize()
    for s in range(steps):
        flush()
        ev[s][0].record()
        g.calls[0]()
        ev[s][1].record()
    torch.cuda.synchronize()
    g.copy_ms = copy_at_sizes([int(g.bytes_per_launch)], device, steps, flush).get(
        int(g.bytes_per_launch))
    return g, [a.elapsed_time(b) for a, b in ev]


def size_sweep(device, steps):
    """NVFP4 amax, RTN quantize (scale from that amax) and dequantize to bf16
    of one bf16 Laplace matrix [n / 4096, 4096] per size of the 1 MiB - 4 GiB
    sweep.  L2 is flushed (L2Flush: 512 MB written, then read back) before
    every timed launch, so the small sizes are measured from HBM too and no
    write-back of the flush lands in the kernel's time; the events bracket
    the kernel alone."""
    import torch
    import block_scaled_fp4_e2m1_gb300 as m
    from block_scaled_fp4_e2m1_gb300 import workloads as W
    peak, kind = measured_peak()
    flush = L2Flush(device)
    for nbytes in W.size_sweep_bytes():
        n = nbytes // 2
        w = W.laplace_weight(11, (n // 4096, 4096), device=device).view(-1)
        a, t = torch.empty(1, device=device), torch.empty(1, device=device)
        pk = torch.empty(n // 2, dtype=torch.uint8, device=device)
        sc = torch.empty(n // 16, dtype=torch.uint8, device=device)
        y = torch.empty(n, dtype=torch.bfloat16, device=device)
        calls = {
            "nvfp4_amax": (2.0 * n, lambda: m.nvfp4_amax(w, amax_ws=a)),
            "nvfp4_quantize": (2.5625 * n, lambda: m.nvfp4_quantize(
                w, tscale="from_amax", amax_ws=a, tensor_scale=t, packed=pk, scales=sc)),
            "nvfp4_dequantize": (2.5625 * n, lambda: m.nvfp4_dequantize(
                pk, sc, t, (n,), torch.bfloat16, out=y)),
        }
        for name, (byt, f) in calls.items():
            for _ in range(3):
                f()
            times = []
            for _ in range(steps):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                f()
                e1.record()
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.median(times)
            gbs = byt / (ms * 1e-3) / 1e9
            print(json.dumps({"kernel": name, "bytes": nbytes, "ms_median": round(ms, 4),
                              "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                              "peak_kind": kind, "l2": "flushed before each launch"}),
                  flush=True)
        del w, pk, sc, y
        torch.cuda.empty_cache()


def train_report(device, steps=TRAIN_STEPS, check_elems=65536):
    """The training workload run for its full schedule: W <- qdq(W - lr G_t)
    on the bf16 [6144, 2048] weight, lr 1e-4, G_t ~ N(0, 1) from seed 1 + t,
    under SR + error feedback, RTN + error feedback and plain RTN ([fp4-train]
    "Correctness": RTN stalls on updates below one quantization step, EF and
    SR do not), each with the tensor scale computed from every step's amax
    and with it held at its step-0 value.  Per step: the share of weights
    whose stored bf16 value changed and mean(W) minus the mean of the
    unquantized fp32 reference W_ref <- W_ref - lr G_t; at the end, the share
    of the reference's total update that W followed,
    <W_T - W_0, R_T - W_0> / |R_T - W_0|^2.  The first check_elems weights
    and residuals are compared with the CPU oracle at every step, with the
    tensor scale the GPU used.  One JSON line per run."""
    import numpy as np
    import torch
    import block_scaled_fp4_e2m1_gb300 as m
    import oracle as ora
    from block_scaled_fp4_e2m1_gb300 import workloads as W

    ora.build()
    shp = (6144, 2048)
    lr = 1e-4
    w0 = W.nvfp4_train_weight(seed=0, shape=shp, device=device).view(-1)
    n = w0.numel()
    grads = [W.nvfp4_train_grad(0, t, shape=shp, device=device).view(-1) for t in range(steps)]
    ref = w0.float()
    ref_mean = [float(ref.double().mean())]
    for t in range(steps):
        ref = ref - lr * grads[t]
        ref_mean.append(float(ref.double().mean()))
    ref_upd = ref.double() - w0.double()
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    for tsmode in ("computed", "fixed"):
        for mode, rnd, ef in (("sr+ef", "sr", True), ("rtn+ef", "rtn", True),
                              ("rtn", "rtn", False)):
            w = w0.clone()
            r = torch.zeros(n, dtype=torch.float32, device=device) if ef else None
            amax, ts = torch.empty(1, device=device), torch.empty(1, device=device)
            m.nvfp4_qdq_amax(w, grads[0], lr, r, amax_ws=amax)
            ts_fixed = torch.tensor([ora.nvfp4_tensor_scale(float(amax.item()))],
                                    dtype=torch.float32, device=device)
            ow = bits(w0)[:check_elems].copy()
            orr = np.zeros(check_elems, np.float32) if ef else None
            changed, drift, mismatch = [], [], 0
            for t in range(steps):
                prev = w.clone()
                if tsmode == "computed":
                    m.nvfp4_qdq_amax(w, grads[t], lr, r, amax_ws=amax)
                    m.nvfp4_qdq(w, grads[t], lr, r, rounding=rnd, seed=0, step=t,
                                tscale="from_amax", amax_ws=amax, tensor_scale=ts,
                                want_packed=False)
                else:
                    ts.copy_(ts_fixed)
                    m.nvfp4_qdq(w, grads[t], lr, r, rounding=rnd, seed=0, step=t,
                                tscale="given", tensor_scale=ts, want_packed=False)
                changed.append(float((w.view(torch.int16) != prev.view(torch.int16))
                                     .double().mean()))
                drift.append(float(w.double().mean()) - ref_mean[t + 1])
                ora.nvfp4_qdq(ow, grads[t][:check_elems].cpu().numpy(), lr, orr,
                              rounding=ora.SR if rnd == "sr" else ora.RTN, seed=0, step=t,
                              tscale_mode=ora.TSCALE_GIVEN, tensor_scale=float(ts.item()))
                same = np.array_equal(bits(w)[:check_elems], ow)
                if ef:
                    same = same and np.array_equal(
                        r[:check_elems].cpu().numpy().view(np.uint32), orr.view(np.uint32))
                mismatch += 0 if same else 1
            upd = w.double() - w0.double()
            print(json.dumps({
                "train_report": mode, "tensor_scale": tsmode, "steps": steps, "lr": lr,
                "shape": list(shp),
                "changed_mean": round(statistics.mean(changed), 6),
                "changed_first5": [round(c, 6) for c in changed[:5]],
                "changed_last5": [round(c, 6) for c in changed[-5:]],
                "update_followed": float((upd * ref_upd).sum() / (ref_upd * ref_upd).sum()),
                "mean_w_minus_ref_final": drift[-1],
                "mean_abs_w_minus_ref_final": float((w.double() - ref.double()).abs().mean()),
                "drift_every20": [drift[i] for i in range(19, steps, 20)],
                "oracle_slice": check_elems, "oracle_steps_mismatched": mismatch,
            }), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.kernel:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        dev = torch.device("cuda", 0)
        names = KERNEL_STUDIES if args.kernel == "all" else args.kernel.split(",")
        peak, kind = measured_peak()
        for nm in names:
            g, ts = kernel_study(nm, args.size_mb, args.steps, args.warmup, dev)
            t = statistics.median(ts)
            gbs = g.bytes_per_launch / (t * 1e-3) / 1e9
            rec = {"kernel": nm, "size_mb": args.size_mb,
                   "bytes_per_launch": int(g.bytes_per_launch),
                   "ms_median": round(t, 4), "ms_min": round(min(ts), 4),
                   "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "peak_kind": kind}
            if g.copy_ms is not None:
                cgbs = g.bytes_per_launch / (g.copy_ms * 1e-3) / 1e9
                rec["copy_same_bytes"] = {"ms": round(g.copy_ms, 4),
                                          "frac": round(cgbs / peak, 4),
                                          "kernel_over_copy": round(gbs / cgbs, 4)}
            print(json.dumps(rec), flush=True)
            torch.cuda.empty_cache()
        return 0
    if args.sweep:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        size_sweep(torch.device("cuda", 0), args.steps if args.steps != 60 else 10)
        return 0
    if args.train_report:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        train_report(torch.device("cuda", 0))
        return 0
    if args.quality:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        import block_scaled_fp4_e2m1_gb300 as m
        from block_scaled_fp4_e2m1_gb300 import workloads as W
        names = ["q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj"]
        for i, (nm, shp) in enumerate(zip(names, W.qwen3_8b_weight_shapes(layers=1))):
            w = W.laplace_weight(1800 + i, shp, device=torch.device("cuda", 0))
            print(json.dumps({"matrix": nm, "shape": list(shp), "quality": m.fp4_quality(w)}),
                  flush=True)
        return 0
    if args.source_hash:
        print(kernel_source_hash(args.source_hash))
        return 0
    if args.summarize_launches:
        print(summarize_launches(args.summarize_launches, args.steps, args.warmup))
        return 0
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_fp4_e2m1_gb300 as m

    groups, st = build_suite(device, rank=rank, small=args.small)
    torch.cuda.synchronize()

    # warm-up
    for _ in range(max(3, args.warmup)):
        run_step(groups, None)
    torch.cuda.synchronize()

    steps = args.steps
    events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in groups] for _ in range(steps)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_id = vis.split(",")[local].strip() if vis else str(local)
    sampler = ClockSampler(smi_id)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = m.kernel_launches()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for s in range(steps):
        run_step(groups, events[s])
    t_end.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = m.kernel_launches() - launches0
    clocks = sampler.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), device if world > 1 else None)
    ms_per_step = total_ms / steps

    for gi, g in enumerate(groups):
        g.step_times_ms = [events[s][gi][0].elapsed_time(events[s][gi][1]) for s in range(steps)]
    bytes_step = sum(g.bytes_per_step for g in groups)
    value = job_gbs(bytes_step, world, ms_per_step)
    peak, peak_kind = measured_peak()

    # per-kernel pass: L2 flushed (clean) before every group, outside its events
    flush = L2Flush(device)
    kpass = kernel_pass_steps(steps)
    kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in groups] for _ in range(kpass)]
    for s_ in range(kpass):
        for gi, g in enumerate(groups):
            flush()
            kev[s_][gi][0].record()
            for c in g.calls:
                c()
            kev[s_][gi][1].record()
    torch.cuda.synchronize()
    for gi, g in enumerate(groups):
        g.times_ms = [kev[s_][gi][0].elapsed_time(kev[s_][gi][1]) for s_ in range(kpass)]
    copy_ms = copy_at_sizes([int(g.bytes_per_launch) for g in groups], device, kpass, flush)
    del flush

    kernels = {}
    for g in groups:
        t = statistics.median(g.times_ms)
        gbs = g.bytes_per_step / (t * 1e-3) / 1e9
        t_step = statistics.median(g.step_times_ms)
        kernels[g.name] = {"gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                           "ms": round(t, 4), "launches": len(g.calls),
                           "bytes_per_launch": int(g.bytes_per_launch),
                           "ms_in_step": round(t_step, 4),
                           "frac_in_step": round(g.bytes_per_step / (t_step * 1e-3) / 1e9 / peak, 4)}
        tc = copy_ms.get(int(g.bytes_per_launch))
        if tc is not None:
            cgbs = g.bytes_per_launch / (tc * 1e-3) / 1e9
            kernels[g.name]["copy_same_bytes"] = {"ms": round(tc, 4),
                                                  "frac": round(cgbs / peak, 4),
                                                  "kernel_over_copy": round(gbs / cgbs, 4)}
    dom = max(groups, key=lambda g: statistics.mean(g.times_ms))
    dom_launch_ms = statistics.mean(dom.times_ms) / len(dom.calls)
    achieved = dom.bytes_per_launch / (dom_launch_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom.name, "achieved": round(achieved, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": None}
    traffic = load_traffic(dom.name)
    if traffic is not None:
        roofline["traffic"] = traffic

    e2e = None
    if not args.no_e2e:
        try:
            t_e2e, h2d, d2h = e2e_measure(groups, st, args.e2e_steps, 1, device)
            if t_e2e is not None:
                e2e = {"value": round(bytes_step * world / t_e2e / 1e9, 2), "unit": "GB/s",
                       "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                       "ms_per_step": round(t_e2e * 1e3, 2)}
            else:
                e2e = {"value": None, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                       "d2h_bytes_per_step": int(d2h), "skipped": "host memory too small"}
        except Exception as ex:  # report, do not hide
            e2e = {"value": None, "unit": "GB/s", "error": repr(ex)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rates, mrates, sample, cores = cpu_oracle_rates()
        cpu = {"value": round(combine_rate(groups, rates), 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "host_cores": host_cores(), "sample": sample,
               "per_kernel_gbs": {k: round(v, 4) for k, v in rates.items()}}
        if mrates:
            cpu["all_cores"] = {"value": round(combine_rate(groups, mrates), 4), "unit": "GB/s",
                                "cores": cores,
                                "how": "the same C oracle on each slice, rows split over "
                                       "threads",
                                "per_kernel_gbs": {k: round(v, 4) for k, v in mrates.items()}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD + ("_small" if args.small else ""),
                       "elements": st["elements"], "bytes_per_step": int(bytes_step),
                       "l2": ("step: inputs larger than L2 (~58 GB per step, L2 129 MB; every "
                              "consumer separated from its producer by >= 2.5 GB of other "
                              "traffic); kernels and roofline: L2 flushed before every group "
                              "(512 MB written then read back)"),
                       "train": (f"bench step k = training step k mod {TRAIN_STEPS} of one SR+EF "
                                 "qdq (amax pass + qdq pass), gradient G_t resident"),
                       "parallelism": f"replicas{world}"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clocks, "kernels": kernels,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def max_over_ranks(ms, device=None):
    """The slowest rank's time (every rank gets it); no-op without a process
    group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step, world, ms_per_step):
    """Whole-job GB/s: every rank processes its own copy of the workload
    (weak scaling), timed by the slowest rank."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


# Sources whose build a traffic figure belongs to, per bench kernel group.
TRAFFIC_SOURCES = {
    "nvfp4_amax@qwen3_8b_weights": ["nvfp4_batched.cu", "nvfp4_device.cuh", "common.cuh"],
    "nvfp4_quantize@qwen3_8b_weights": ["nvfp4_batched.cu", "nvfp4_device.cuh", "common.cuh"],
    "nvfp4_dequantize@qwen3_8b_weights": ["nvfp4_batched.cu", "nvfp4_device.cuh", "common.cuh"],
    "fp4_to_fp8_col@moe_tokens": ["fp8_convert.cu", "common.cuh"],
}


def kernel_source_hash(kernel_name):
    """sha256 (first 16 hex digits) of the CUDA sources a kernel group is built
    from, or None if the group is not listed."""
    import hashlib
    files = TRAFFIC_SOURCES.get(kernel_name)
    if not files:
        return None
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_scaled_fp4_e2m1_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel_name):
    """DRAM bytes (read + write) per launch of `kernel_name` from
    profiles/traffic.json, or None when there is no figure or the kernel's
    sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f).get(kernel_name)
        if not d or d.get("source_hash") != kernel_source_hash(kernel_name):
            return None
        return d.get("bytes_per_launch")
    except Exception:
        return None


if __name__ == "__main__":
    sys.exit(main())
