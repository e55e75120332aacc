"""Benchmark of the MX hot path on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mx|reference]
                    [--workload all|sweep|gemm|fp4|fused|pipeline256]

A step is one pass of the whole hot path over its synthetic inputs:
  sweep  QuantizeMX on [8192, 8192] for {bf16, f16} x {e4m3fn, e5m2} x
         {plain, interleaved} scales, 8x4 blocks along dim=-2 (8 launches,
         repeated 8 times in one timed span);
  gemm   for e4m3fn -> bf16 and e5m2 -> f32: QuantizeMX of A and Bt
         ([8192, 8192] bf16, 1x32 blocks along K), repack of both scale
         tensors to the tensor-core layout, ScaledMatmul 8192^3;
  fp4    QuantizeMX [16384, 16384] bf16 -> e2m1, 8x4, packed, interleaved;
  dequant  MX dequantize of [8192, 8192] e4m3fn codes with 8x4 scales to bf16;
  fused  activation quantize + ScaledMatmul in one launch, X [16384, 8192]
         bf16 times a pre-quantized e4m3fn weight W [8192, 28672] -> bf16,
         next to the same product as two launches;
  gemm_fp4  MXFP4 ScaledMatmul 8192^3 (e2m1 operands quantized along K in
         the tensor-core nibble order, repacked scales) -> bf16;
  dot    batched block-scaled dot, 16 problems of 2048^3 e4m3fn -> bf16:
         rhs stored [B, N, K] (read in place) and [B, K, N] (through the
         transposing copy), one call each.
The headline `value` is QuantizeMX GB/s over the sweep (algorithmic bytes:
2 read + 1 written + 1/32 scale written per element); `scaled_matmul`,
`fp4_quantize` and `fused` carry the other workloads with their own rooflines.
Inputs are larger than L2 and rotated so no launch re-reads the previous
launch's input from L2.  Kernel times come from CUDA events on the launching
stream; the whole step is bracketed by a barrier and a synchronize.

--impl reference times the CPU oracle (plain C, as it stands) on the sweep
workload, one worker process per host core, with the same metric and unit;
the main arm's cpu_baseline is the same measurement.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mx_synth as syn  # noqa: E402

METRIC = "QuantizeMX GB/s & ScaledMatmul TFLOP/s on 1 GB300, % of HBM/MXFP8 peak"
SWEEP = (8192, 8192)
SWEEP_VARIANTS = [(i, f) for i in ("bf16", "f16") for f in ("e4m3fn", "e5m2")]
SWEEP_BYTES = 2 * 8192 * 8192 + 8192 * 8192 + 1024 * 2048          # 203,423,744 per launch
FP4_SHAPE = (16384, 16384)
FP4_BYTES = 2 * 16384 * 16384 + 16384 * 16384 // 2 + 2048 * 4096  # 679,477,248
GEMM_N = 8192
GEMM_FLOP = 2 * GEMM_N ** 3
FUSED = (16384, 28672, 8192)
FUSED_FLOP = 2 * FUSED[0] * FUSED[1] * FUSED[2]
DOT = (16, 2048, 2048, 2048)  # batch, M, N, K
SMALL_M = (16, 64, 128)       # M of M x 8192 x 8192 ScaledMatmuls (HBM-bound: one pass over B)
SMALL_M_COPIES = 4            # B copies rotated so every call reads B from HBM (4 x 64 MiB > L2)
DOT_FLOP = 2 * DOT[0] * DOT[1] * DOT[2] * DOT[3]
# nominal dense MXFP8 : bf16 and FP4 : bf16 tensor ratios (4.5 and 13.5 : 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0
FP4_OVER_BF16 = 6.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sust": p.get("bf16_tflops_sustained"),
                "src": "of measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sust": 1700.0, "src": "of fallback"}


def code_text(src):
    """Source text without C/C++ comments and with whitespace runs collapsed:
    what the compiler sees, so that editing a comment keeps the hash."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "mx_fp8_microscaling_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(code_text(f.read()).encode())
    return h.hexdigest()[:16]


def _src_hashes():
    """Hashes of each kernel family's sources (its .cu file and the headers
    it is built from) that traffic.json entries are keyed on."""
    return (source_hash("quantize.cu", "quant_math.cuh", "mx_device.cuh", "pdl.cuh"),
            source_hash("gemm.cu", "tcgen05.cuh", "quant_math.cuh", "mx_device.cuh", "pdl.cuh"),
            source_hash("dequantize.cu", "mx_device.cuh", "pdl.cuh"))


def profiled_traffic(kernel_key, src_hash):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        entry = json.load(open(path)).get(kernel_key)
    except (ValueError, OSError):
        return None
    if not entry or entry.get("source_hash") != src_hash:
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [[c.strip() for c in line.split(",")] for line in out.strip().splitlines() if line.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx_ = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            if len(r) < 9:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        load = [s for s in sm if mx_ and s >= 0.5 * max(mx_)] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx_) if mx_ else None, "reasons": sorted(reasons),
                "samples": len(rows)}


# ---------------------------------------------------------------- workloads

class Timer:
    """CUDA-event durations per label on the current stream.  Event pairs are
    created up front so recording a span costs two cudaEventRecord calls."""

    def __init__(self, torch, capacity=4096):
        self.torch = torch
        self.events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(capacity)]
        self.used = []
        self.totals = {}
        self.counts = {}

    def run(self, label, fn):
        a, b = self.events[len(self.used)]
        a.record()
        fn()
        b.record()
        self.used.append((label, a, b))

    def collect(self):
        for label, a, b in self.used:
            ms = a.elapsed_time(b)
            self.totals[label] = self.totals.get(label, 0.0) + ms
            self.counts[label] = self.counts.get(label, 0) + 1
        self.used = []

    def avg_ms(self, label):
        return self.totals[label] / self.counts[label]

    def reset(self):
        self.used, self.totals, self.counts = [], {}, {}


class Api:
    """Direct C-ABI calls with arguments marshalled once (the binding's
    per-call conveniences cost more host time than a 35 us kernel)."""

    def __init__(self, torch, mx):
        import ctypes
        self.torch, self.mx, self.lib, self.ct = torch, mx, mx.raw_library(), ctypes

    def stream(self):
        return self.ct.c_void_p(self.torch.cuda.current_stream().cuda_stream)

    def quantize(self, x, fmt, geometry, dim, layout, data, scale, **cfg_kw):
        mx, ct = self.mx, self.ct
        rows, cols, ld = mx._view2d(x, dim)
        cfg = mx.make_cfg(geometry, dim, layout, **cfg_kw)
        args = (ct.c_void_p(x.data_ptr()), mx.DTYPES[mx._in_dtype(x)], rows, cols, ld, mx.DTYPES[fmt],
                ct.byref(cfg), ct.c_void_p(data.data_ptr()), ct.c_void_p(scale.data_ptr()), self.stream())
        fn = self.lib.mx_quantize

        def call():
            st = fn(*args)
            if st:
                raise mx.MxError(st, "mx_quantize")
        call.cfg = cfg  # keep the struct alive
        return call

    def repack(self, plain, k, sf):
        mx, ct = self.mx, self.ct
        args = (ct.c_void_p(plain.data_ptr()), plain.shape[0], k, plain.stride(0), ct.c_void_p(sf.data_ptr()),
                self.stream())
        fn = self.lib.mx_repack_scales

        def call():
            st = fn(*args)
            if st:
                raise mx.MxError(st, "mx_repack_scales")
        return call

    def matmul_sf(self, a, bt, sfa, sfb, fmt, out_dtype, c, K):
        mx, ct = self.mx, self.ct
        args = (ct.c_void_p(a.data_ptr()), ct.c_void_p(bt.data_ptr()), ct.c_void_p(sfa.data_ptr()),
                ct.c_void_p(sfb.data_ptr()), 1, mx.DTYPES[fmt], a.shape[0], bt.shape[0], K, mx.DTYPES[out_dtype],
                ct.c_void_p(c.data_ptr()), c.stride(0), None, 0, self.stream())
        fn = self.lib.mx_scaled_matmul

        def call():
            st = fn(*args)
            if st:
                raise mx.MxError(st, "mx_scaled_matmul")
        return call

    def dot(self, lhs, rhs, ls, rs, dims, fmt, out_dtype, out, work):
        mx, ct = self.mx, self.ct
        lshape, rshape = mx._dims_array(lhs.shape), mx._dims_array(rhs.shape)
        args = (ct.c_void_p(lhs.data_ptr()), lshape, lhs.dim(), ct.c_void_p(ls.data_ptr()),
                ct.c_void_p(rhs.data_ptr()), rshape, rhs.dim(), ct.c_void_p(rs.data_ptr()), ct.byref(dims),
                mx.DTYPES[fmt], mx.DTYPES[out_dtype], ct.c_void_p(out.data_ptr()), ct.c_void_p(work.data_ptr()),
                work.numel(), self.stream())
        fn = self.lib.mx_block_scaled_dot

        def call():
            st = fn(*args)
            if st:
                raise mx.MxError(st, "mx_block_scaled_dot")
        call.keep = (dims, lshape, rshape)
        return call

    def fused(self, x, wt, wsf, fmt, out_dtype, c, work):
        mx, ct = self.mx, self.ct
        M, K = x.shape
        args = (ct.c_void_p(x.data_ptr()), mx.DTYPES[mx._in_dtype(x)], x.stride(0), ct.c_void_p(wt.data_ptr()),
                ct.c_void_p(wsf.data_ptr()), mx.DTYPES[fmt], M, wt.shape[0], K, mx.DTYPES[out_dtype],
                ct.c_void_p(c.data_ptr()), c.stride(0), ct.c_void_p(work.data_ptr()), work.numel(), self.stream())
        fn = self.lib.mx_fused_quantize_matmul

        def call():
            st = fn(*args)
            if st:
                raise mx.MxError(st, "mx_fused_quantize_matmul")
        return call


def dev_bits(torch, bits, in_dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16 if in_dtype == "bf16" else torch.float16).cuda()


class Sweep:
    def __init__(self, torch, mx, api):
        self.mx, self.torch = mx, torch
        self.host, self.x, self.out = {}, {}, {}
        for in_dtype, fmt in SWEEP_VARIANTS:
            bits = syn.sweep_input(*SWEEP, in_dtype, fmt, seed=0)
            self.host[(in_dtype, fmt)] = bits
            self.x[(in_dtype, fmt)] = dev_bits(torch, bits, in_dtype)
        self.ops = []
        # layouts outermost: consecutive launches read different 128 MiB inputs
        for layout in ("plain", "interleave"):
            for in_dtype, fmt in SWEEP_VARIANTS:
                cfg = mx.make_cfg("8x4", -2, layout)
                _, sr, sc = mx.mx_quantize_sizes(*SWEEP, in_dtype, fmt, cfg)
                d = torch.empty(SWEEP[0] * SWEEP[1], dtype=torch.uint8, device="cuda")
                s = torch.empty(sr * sc, dtype=torch.uint8, device="cuda")
                self.out[(layout, in_dtype, fmt)] = (d, s)
                self.ops.append(("sweep", api.quantize(self.x[(in_dtype, fmt)], fmt, "8x4", -2, layout, d, s)))
        self.launches = self.REPEATS * len(self.ops)

    # One event pair around REPEATS x 8 back-to-back launches (per-launch
    # event records would add their own gaps to 33 us kernels).  A span ends
    # with its last launch's writes partly still in L2 (about 58 of 69 MB);
    # over 64 launches that is under 0.5 % of the span's bytes.
    REPEATS = 8

    def step(self, timer):
        def all_launches():
            for _ in range(self.REPEATS):
                for _, fn in self.ops:
                    fn()
        timer.run("sweep", all_launches)


class Gemm:
    CASES = [("e4m3fn", "bf16"), ("e5m2", "f32")]

    def __init__(self, torch, mx, api):
        a_bits, b_bits = syn.gemm_operands(GEMM_N, GEMM_N, GEMM_N, seed=0)
        a = dev_bits(torch, a_bits, "bf16")
        b = dev_bits(torch, b_bits, "bf16")
        n = GEMM_N
        qa = torch.empty((n, n), dtype=torch.uint8, device="cuda")
        qb = torch.empty((n, n), dtype=torch.uint8, device="cuda")
        sa = torch.empty((n, n // 32), dtype=torch.uint8, device="cuda")
        sb = torch.empty((n, n // 32), dtype=torch.uint8, device="cuda")
        sfb = mx.mx_sf_layout_bytes(n, n)
        sfa_t = torch.empty(sfb, dtype=torch.uint8, device="cuda")
        sfb_t = torch.empty(sfb, dtype=torch.uint8, device="cuda")
        self.keep = (a, b, qa, qb, sa, sb, sfa_t, sfb_t)
        self.c = {"bf16": torch.empty((n, n), dtype=torch.bfloat16, device="cuda"),
                  "f32": torch.empty((n, n), dtype=torch.float32, device="cuda")}
        self.ops = []
        for fmt, out in self.CASES:
            self.ops.append(("gemm_quantize", api.quantize(a, fmt, "1x32", -1, "plain", qa, sa)))
            self.ops.append(("gemm_quantize", api.quantize(b, fmt, "1x32", -1, "plain", qb, sb)))
            self.ops.append(("gemm_repack", api.repack(sa, n, sfa_t)))
            self.ops.append(("gemm_repack", api.repack(sb, n, sfb_t)))
            self.ops.append((f"gemm_{fmt}_{out}", api.matmul_sf(qa, qb, sfa_t, sfb_t, fmt, out, self.c[out], n)))
        self.launches = 2 * (2 + 2 + 1)

    def step(self, timer):
        for label, fn in self.ops:
            timer.run(label, fn)


class Fp4:
    """QuantizeMX [16384, 16384] bf16 -> e2m1, 8x4 blocks, interleaved
    scales: 16 back-to-back launches a step alternating over two inputs
    (seeds 0 and 1, 512 MiB each), timed as one span like the sweep."""
    LAUNCHES = 16

    def __init__(self, torch, mx, api):
        cfg = mx.make_cfg("8x4", -2, "interleave")
        db, sr, sc = mx.mx_quantize_sizes(*FP4_SHAPE, "bf16", "e2m1", cfg)
        self.keep = []
        calls = []
        for seed in range(2):
            x = dev_bits(torch, syn.fp4_input(*FP4_SHAPE, seed=seed), "bf16")
            d = torch.empty(db, dtype=torch.uint8, device="cuda")
            s = torch.empty(sr * sc, dtype=torch.uint8, device="cuda")
            self.keep.append((x, d, s))
            calls.append(api.quantize(x, "e2m1", "8x4", -2, "interleave", d, s))
        self.ops = [calls[i % 2] for i in range(self.LAUNCHES)]
        self.launches = self.LAUNCHES

    def step(self, timer):
        def all_launches():
            for fn in self.ops:
                fn()
        timer.run("fp4", all_launches)


class Dequant:
    """[8192, 8192] e4m3fn codes + plain 8x4 scales -> bf16 (1 + 1/32 B read,
    2 B written per element): 32 back-to-back launches a step alternating
    over two code / output sets (388 MiB, larger than L2), timed as one span
    like the sweep."""
    LAUNCHES = 32

    def __init__(self, torch, mx, api):
        import ctypes
        self.cfg = mx.make_cfg("8x4", -2, "plain")
        lib = mx.raw_library()
        self.keep = []
        calls = []
        for seed in range(2):
            bits = syn.sweep_input(*SWEEP, "bf16", "e4m3fn", seed=seed)
            x = dev_bits(torch, bits, "bf16")
            d, s = mx.mx_quantize(x, "e4m3fn", geometry="8x4", dim=-2)
            del x
            out = torch.empty(SWEEP, dtype=torch.bfloat16, device="cuda")
            self.keep.append((d, s, out))
            args = (ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(s.data_ptr()), mx.DTYPES["e4m3fn"], SWEEP[0],
                    SWEEP[1], ctypes.byref(self.cfg), mx.DTYPES["bf16"], ctypes.c_void_p(out.data_ptr()), SWEEP[1],
                    api.stream())

            def call(args=args):
                st = lib.mx_dequantize(*args)
                if st:
                    raise mx.MxError(st, "mx_dequantize")
            calls.append(call)
        self.ops = [calls[i % 2] for i in range(self.LAUNCHES)]
        self.launches = self.LAUNCHES

    def step(self, timer):
        def all_launches():
            for fn in self.ops:
                fn()
        timer.run("dequant", all_launches)


class Fused:
    SHAPE = FUSED  # --fused-shape M,N,K (profiling runs a smaller case)

    def __init__(self, torch, mx, api):
        M, N, K = self.SHAPE
        x_bits, w_bits = syn.fused_operands(M, N, K, seed=0)
        self.x = dev_bits(torch, x_bits, "bf16")
        wt = dev_bits(torch, w_bits, "bf16")
        del w_bits
        # offline weight preparation (not timed): QuantizeMX of W along K,
        # stored K-contiguous with tensor-core layout scales
        self.wq, self.ws = mx.mx_quantize(wt, "e4m3fn", geometry="1x32", dim=-1, scale_layout="sf")
        del wt
        self.c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        self.work = torch.empty(mx.mx_fused_quantize_matmul_workspace(M, N, K), dtype=torch.uint8, device="cuda")
        self.op = api.fused(self.x, self.wq, self.ws, "e4m3fn", "bf16", self.c, self.work)
        # the same product unfused: QuantizeMX of X into SF-layout scales,
        # then ScaledMatmul, as two calls (reported as the fused call's split)
        self.xq = torch.empty((M, K), dtype=torch.uint8, device="cuda")
        self.xs = torch.empty(mx.mx_sf_layout_bytes(M, K), dtype=torch.uint8, device="cuda")
        self.unfused = [("fused_split_quantize", api.quantize(self.x, "e4m3fn", "1x32", -1, "sf", self.xq, self.xs)),
                        ("fused_split_gemm", api.matmul_sf(self.xq, self.wq, self.xs, self.ws, "e4m3fn", "bf16",
                                                           self.c, K))]
        self.op()
        torch.cuda.synchronize()
        # 3: the pair kernel with the fused quantize, the whole call one launch
        self.launches_per_call = 1 if mx.mx_debug_last_gemm_launch()[0] == 3 else 2
        self.launches = self.launches_per_call + 2

    def step(self, timer):
        timer.run("fused", self.op)
        for label, fn in self.unfused:
            timer.run(label, fn)


class GemmFp4:
    """MXFP4 ScaledMatmul 8192^3 -> bf16: quantize A and Bt to e2m1 (1x32
    along K, element 2i in the low nibble), repack both scale tensors, GEMM."""

    def __init__(self, torch, mx, api):
        n = GEMM_N
        a_bits, b_bits = syn.gemm_operands(n, n, n, seed=0)
        self.a = dev_bits(torch, a_bits, "bf16")
        self.b = dev_bits(torch, b_bits, "bf16")
        del a_bits, b_bits
        self.qa = torch.empty(n * n // 2, dtype=torch.uint8, device="cuda")
        self.qb = torch.empty(n * n // 2, dtype=torch.uint8, device="cuda")
        self.sa = torch.empty(n * n // 32, dtype=torch.uint8, device="cuda")
        self.sb = torch.empty(n * n // 32, dtype=torch.uint8, device="cuda")
        sfb = mx.mx_sf_layout_bytes(n, n)
        self.sfa = torch.empty(sfb, dtype=torch.uint8, device="cuda")
        self.sfb = torch.empty(sfb, dtype=torch.uint8, device="cuda")
        self.c = torch.empty((n, n), dtype=torch.bfloat16, device="cuda")
        self.ops = [("fp4_quantize_operands", api.quantize(self.a, "e2m1", "1x32", -1, "plain", self.qa, self.sa,
                                                          fp4_lane_stride=1, fp4_nibble_parity=1)),
                    ("fp4_quantize_operands", api.quantize(self.b, "e2m1", "1x32", -1, "plain", self.qb, self.sb,
                                                          fp4_lane_stride=1, fp4_nibble_parity=1)),
                    ("fp4_repack", api.repack(self.sa.view(n, n // 32), n, self.sfa)),
                    ("fp4_repack", api.repack(self.sb.view(n, n // 32), n, self.sfb)),
                    ("gemm_fp4", api.matmul_sf(self.qa.view(n, n // 2), self.qb.view(n, n // 2), self.sfa, self.sfb,
                                               "e2m1", "bf16", self.c, n))]
        self.launches = 5

    def step(self, timer):
        for label, fn in self.ops:
            timer.run(label, fn)


class Dot:
    """Batched block-scaled dot, 16 x (2048 x 2048 x 2048), e4m3fn -> bf16.
    Operands: bf16 N(0,1) * 2^U(-8,8) per row, quantized along K (1x32,
    plain scales) before timing; the [B, K, N] copy of rhs is made once by
    a device transpose, also before timing; the call reads it in place as
    MN-major tiles."""
    CASES = ("rhs_bnk", "rhs_bkn")

    def __init__(self, torch, mx, api):
        B, M, N, K = DOT
        a_bits, b_bits = syn.gemm_operands(B * M, B * N, K, seed=0)
        a = dev_bits(torch, a_bits, "bf16")
        b = dev_bits(torch, b_bits, "bf16")
        del a_bits, b_bits
        qa, sa = mx.mx_quantize(a, "e4m3fn", geometry="1x32", dim=-1)
        qb, sb = mx.mx_quantize(b, "e4m3fn", geometry="1x32", dim=-1)
        del a, b
        lhs, ls = qa.view(B, M, K), sa.view(B, M, K // 32)
        rhs, rs = qb.view(B, N, K), sb.view(B, N, K // 32)
        rhs_kn = rhs.transpose(1, 2).contiguous()
        rs_kn = rs.transpose(1, 2).contiguous()
        self.out = torch.empty((B, M, N), dtype=torch.bfloat16, device="cuda")
        d_nk = mx.make_dot_dims((0,), (0,), (2,), (2,))
        d_kn = mx.make_dot_dims((0,), (0,), (2,), (1,))
        w = max(mx.mx_block_scaled_dot_workspace(lhs.shape, rhs.shape, d_nk),
                mx.mx_block_scaled_dot_workspace(lhs.shape, rhs_kn.shape, d_kn))
        self.work = torch.empty(w, dtype=torch.uint8, device="cuda")
        self.keep = (lhs, ls, rhs, rs, rhs_kn, rs_kn)
        self.ops = [("dot_rhs_bnk", api.dot(lhs, rhs, ls, rs, d_nk, "e4m3fn", "bf16", self.out, self.work)),
                    ("dot_rhs_bkn", api.dot(lhs, rhs_kn, ls, rs_kn, d_kn, "e4m3fn", "bf16", self.out, self.work))]
        self.launches = 3 + 3  # repack x2 + GEMM, both cases ([B, K, N] rhs read in place, MN-major)

    def step(self, timer):
        for label, fn in self.ops:
            timer.run(label, fn)


class Pipeline256:
    """The MX-FP8 pipeline at M = N = K = 256, seed 0: QuantizeMX of A and
    Bt (bf16, N(0,1) x 2^U(-20,20) per 32-block) along K to e4m3fn with
    plain scales, repack of both scale tensors, ScaledMatmul to f32.  Five
    launches, a few microseconds each: latency-bound, reported in us."""

    def __init__(self, torch, mx, api):
        self.torch = torch
        a_bits, b_bits = syn.pipeline_operands(256, 256, 256, seed=0)
        self.a, self.b = dev_bits(torch, a_bits, "bf16"), dev_bits(torch, b_bits, "bf16")
        self.qa = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        self.qb = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        self.sa = torch.empty((256, 8), dtype=torch.uint8, device="cuda")
        self.sb = torch.empty((256, 8), dtype=torch.uint8, device="cuda")
        self.sfa = torch.empty(mx.mx_sf_layout_bytes(256, 256), dtype=torch.uint8, device="cuda")
        self.sfb = torch.empty(mx.mx_sf_layout_bytes(256, 256), dtype=torch.uint8, device="cuda")
        self.c = torch.empty((256, 256), dtype=torch.float32, device="cuda")
        self.ops = [api.quantize(self.a, "e4m3fn", "1x32", -1, "plain", self.qa, self.sa),
                    api.quantize(self.b, "e4m3fn", "1x32", -1, "plain", self.qb, self.sb),
                    api.repack(self.sa, 256, self.sfa), api.repack(self.sb, 256, self.sfb),
                    api.matmul_sf(self.qa, self.qb, self.sfa, self.sfb, "e4m3fn", "f32", self.c, 256)]
        self.launches = 5
        # the same five calls captured once as a CUDA graph (bound to the
        # capturing stream), timed after the main loop: the device time
        # without host dispatch
        self.side = torch.cuda.Stream()
        with torch.cuda.stream(self.side):
            ops = [api.quantize(self.a, "e4m3fn", "1x32", -1, "plain", self.qa, self.sa),
                   api.quantize(self.b, "e4m3fn", "1x32", -1, "plain", self.qb, self.sb),
                   api.repack(self.sa, 256, self.sfa), api.repack(self.sb, 256, self.sfb),
                   api.matmul_sf(self.qa, self.qb, self.sfa, self.sfb, "e4m3fn", "f32", self.c, 256)]
            for fn in ops:
                fn()
        self.side.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.side):
            for fn in ops:
                fn()
        torch.cuda.synchronize()

    def graph_us(self, reps=200):
        torch = self.torch
        for _ in range(10):
            self.graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            self.graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def run_all(self):
        for fn in self.ops:
            fn()

    def step(self, timer):
        timer.run("pipeline_256", self.run_all)


class GemmSmallM:
    """ScaledMatmul with few rows: M in SMALL_M, N = K = 8192, e4m3fn ->
    bf16 with SF-layout scales.  The kernel streams B once, so HBM bounds
    it.  B rotates over SMALL_M_COPIES copies (256 MiB, larger than L2); each
    shape's 4 calls (one per copy) run as one CUDA graph, since host launch
    cost is comparable to these ~17-20 us kernels.  A holds the first M rows
    of one quantized [128, 8192] operand."""

    def __init__(self, torch, mx, api):
        n = GEMM_N
        a_bits, b_bits = syn.gemm_operands(max(SMALL_M), n, n, seed=0)
        a = dev_bits(torch, a_bits, "bf16")
        b = dev_bits(torch, b_bits, "bf16")
        del a_bits, b_bits
        qa, sa = mx.mx_quantize(a, "e4m3fn", geometry="1x32", dim=-1)
        qb, sfb = mx.mx_quantize(b, "e4m3fn", geometry="1x32", dim=-1, scale_layout="sf")
        del a, b
        self.qb = [qb] + [qb.clone() for _ in range(SMALL_M_COPIES - 1)]
        self.sfb = sfb
        self.a = {}
        for m in SMALL_M:
            sfa = torch.empty(mx.mx_sf_layout_bytes(m, n), dtype=torch.uint8, device="cuda")
            mx.mx_repack_scales(sa.view(max(SMALL_M), n // 32)[:m], n, out=sfa)
            self.a[m] = (qa.view(max(SMALL_M), n)[:m], sfa, torch.empty((m, n), dtype=torch.bfloat16,
                                                                         device="cuda"))
        torch.cuda.synchronize()
        self.split = {}
        self.graphs = {}
        for m in SMALL_M:
            qa_m, sfa, c = self.a[m]

            def calls(qa_m=qa_m, sfa=sfa, c=c):
                for qb_i in self.qb:
                    mx.mx_scaled_matmul(qa_m, qb_i, sfa, self.sfb, "e4m3fn", "bf16", scales_are_sf_layout=True,
                                        out=c)
            self.graphs[m] = capture_graph(torch, calls)
            self.split[m] = mx.mx_debug_last_gemm_launch()[1]
        self.launches = SMALL_M_COPIES * len(SMALL_M)

    def bytes_per_call(self, m):
        n = GEMM_N
        return n * n + m * n + sf_layout_bytes(n, n) + sf_layout_bytes(m, n) + 2 * m * n

    def step(self, timer):
        for m in SMALL_M:
            timer.run(f"small_m_{m}", self.graphs[m].replay)


def sf_layout_bytes(rows, k):
    """Bytes of an SF-layout scale tensor: 512-byte tiles of 128 rows x 4
    scale columns (four 32-element blocks)."""
    return -(-rows // 128) * -(-(k // 32) // 4) * 512


def capture_graph(torch, fn):
    """fn() once on a side stream (warm-up: attributes, cached queries), then
    captured into a CUDA graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    return graph


def vendor_small_m_reference(torch, g, steps):
    """cuBLASLt's block-scaled FP8 GEMM (torch._scaled_mm) on the same
    operands, scales and B rotation, also as one CUDA graph per shape, timed
    after the main loop: a comparison point, not part of the timed step."""
    try:
        out = {}
        for m in SMALL_M:
            qa_m, sfa, _ = g.a[m]
            a8 = qa_m.view(torch.float8_e4m3fn)
            sa8 = sfa.view(torch.float8_e8m0fnu)
            sb8 = g.sfb.view(torch.float8_e8m0fnu)

            def calls(a8=a8, sa8=sa8):
                for qb_i in g.qb:
                    torch._scaled_mm(a8, qb_i.view(torch.float8_e4m3fn).t(), sa8, sb8, out_dtype=torch.bfloat16)
            graph = capture_graph(torch, calls)
            ts = {"ours": [], "cublaslt": []}
            for it in range(3 + steps):
                for which, gr in (("ours", g.graphs[m]), ("cublaslt", graph)):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    gr.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    if it >= 3:
                        ts[which].append(e0.elapsed_time(e1) * 1e3 / SMALL_M_COPIES)
            out[str(m)] = {k: round(statistics.median(v), 2) for k, v in ts.items()}
        return {"us_per_call": out, "what": "cuBLASLt via torch._scaled_mm, same operands and graphs"}
    except Exception as e:
        return {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}


def vendor_gemm_reference(torch, g, steps):
    """cuBLASLt's block-scaled FP8 GEMM (torch._scaled_mm with E8M0 scales in
    the same tensor-core layout) on the same e4m3fn operands and scales as
    this library's 8192^3 GEMM, timed after the main loop in the same
    pattern (operand quantize + repack, then the GEMM): a comparison point,
    not part of this library's path or of the timed step."""
    try:
        qa, qb, sfa, sfb = g.keep[2], g.keep[3], g.keep[6], g.keep[7]
        a8 = qa.view(torch.float8_e4m3fn)
        b8 = qb.view(torch.float8_e4m3fn)
        sa8 = sfa.view(torch.float8_e8m0fnu)
        sb8 = sfb.view(torch.float8_e8m0fnu)
        quant = [fn for label, fn in g.ops[:4]]            # e4m3fn case: quantize A, B, repack A, B
        ours = g.ops[4][1]
        times = {"ours": [], "cublaslt": []}
        for it in range(3 + steps):
            for which in ("ours", "cublaslt"):
                for fn in quant:
                    fn()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                if which == "ours":
                    ours()
                else:
                    torch._scaled_mm(a8, b8.t(), sa8, sb8, out_dtype=torch.bfloat16)
                e1.record()
                torch.cuda.synchronize()
                if it >= 3:
                    times[which].append(e0.elapsed_time(e1))
        out = {k: round(GEMM_FLOP / (statistics.median(v) * 1e-3) / 1e12, 1) for k, v in times.items()}
        return {"tflops": out, "what": "8192^3 e4m3fn -> bf16, same operands and scales; cuBLASLt via "
                                      "torch._scaled_mm"}
    except Exception as e:  # a torch build without block-scaled _scaled_mm
        return {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}


def vendor_fp4_reference(torch, g, steps):
    """cuBLASLt's FP4 GEMM at the same size for context.  torch._scaled_mm
    offers block-scaled FP4 only as NVFP4 (16-element blocks, e4m3 scales),
    so this times that format on the same packed e2m1 operands with unit
    scales, alternating with this library's MXFP4 GEMM: a comparison of the
    FP4 tensor-core rate, not of the same arithmetic."""
    try:
        n = GEMM_N
        a4 = g.qa.view(n, n // 2).view(torch.float4_e2m1fn_x2)
        b4 = g.qb.view(n, n // 2).view(torch.float4_e2m1fn_x2)
        s4 = torch.full((n * n // 16,), 0x38, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
        ours = g.ops[4][1]
        times = {"ours_mxfp4": [], "cublaslt_nvfp4": []}
        for it in range(3 + steps):
            for which in times:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                if which == "ours_mxfp4":
                    ours()
                else:
                    torch._scaled_mm(a4, b4.t(), s4, s4, out_dtype=torch.bfloat16)
                e1.record()
                torch.cuda.synchronize()
                if it >= 3:
                    times[which].append(e0.elapsed_time(e1))
        out = {k: round(GEMM_FLOP / (statistics.median(v) * 1e-3) / 1e12, 1) for k, v in times.items()}
        return {"tflops": out, "what": "same packed e2m1 codes; cuBLASLt runs NVFP4 (1x16, e4m3 scales)"}
    except Exception as e:
        return {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}


# ------------------------------------------------------------- CPU oracle

# The oracle runs as it stands (plain C, one call per slice) in a pool of
# worker processes, one per host core, started with "spawn" (a pool forked
# after CUDA initialisation can hang).  Each worker makes its inputs, waits
# on a barrier with the others, and times its own calls; the throughput is
# all workers' bytes over the span from the first start to the last end.

_POOL_BARRIER = None


def _pool_init(barrier):
    global _POOL_BARRIER
    _POOL_BARRIER = barrier


def _oracle_sweep_task(task):
    rows, part = task
    import oracle as orc
    samples = [(i, f, syn.sweep_input(rows, 8192, i, f, seed=1000 + part)) for i, f in SWEEP_VARIANTS]
    _POOL_BARRIER.wait()
    t0 = time.perf_counter()
    nbytes = 0
    for layout in ("plain", "interleave"):
        for in_dtype, fmt, bits in samples:
            orc.quantize(bits, in_dtype, fmt, geometry="8x4", dim=-2, scale_layout=layout)
            nbytes += 3 * bits.size + bits.size // 32
    return nbytes, t0, time.perf_counter()


def _oracle_gemm_task(part):
    import oracle as orc
    rng = np.random.default_rng(part)
    K = GEMM_N
    a = rng.integers(0, 0x7E, size=(1, K)).astype(np.uint8)
    bt = rng.integers(0, 0x7E, size=(GEMM_N, K)).astype(np.uint8)
    sa = np.full((1, K // 32), 127, np.uint8)
    sb = np.full((GEMM_N, K // 32), 127, np.uint8)
    ms, ns = np.zeros(GEMM_N, np.int64), np.arange(GEMM_N, dtype=np.int64)
    _POOL_BARRIER.wait()
    t0 = time.perf_counter()
    orc.scaled_matmul_entries(a, bt, sa, sb, "e4m3fn", "e4m3fn", ms, ns)
    return 2.0 * GEMM_N * K, t0, time.perf_counter()


def _run_pool(fn, tasks):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(tasks))
    with ctx.Pool(len(tasks), initializer=_pool_init, initargs=(barrier,)) as pool:
        res = pool.map(fn, tasks, chunksize=1)
    work = sum(r[0] for r in res)
    span = max(r[2] for r in res) - min(r[1] for r in res)
    return work, span


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sweep_parallel(cores=None, rows=None):
    """The oracle on the whole sweep workload: every core quantizes a
    [rows, 8192] slice (rows = 8192 / cores, rounded down to whole
    interleave groups, unless given) of each of the 4 inputs, both scale
    layouts.  Returns (GB/s over algorithmic bytes, seconds, cores,
    description)."""
    cores = cores or host_cores()
    rows = rows or max(32, 8192 // cores // 32 * 32)
    nbytes, dt = _run_pool(_oracle_sweep_task, [(rows, i) for i in range(cores)])
    return nbytes / dt / 1e9, dt, cores, \
        f"the sweep's 8 variants over [{rows * cores}, 8192] rows ([{rows}, 8192] a core, own seeds), " \
        f"plain C oracle, {cores} worker processes"


def oracle_gemm_parallel(cores=None):
    """The oracle's binary64 scaled dot, one full output row of the 8192^3
    ScaledMatmul per core (k-ordered sums in C).  Returns (TFLOP/s, seconds,
    cores)."""
    cores = cores or host_cores()
    flop, dt = _run_pool(_oracle_gemm_task, list(range(cores)))
    return flop / dt / 1e12, dt, cores


def oracle_pipeline_256(repeats=5):
    """The oracle's 256^3 MX-FP8 pipeline (quantize both operands along K,
    then the binary64 ScaledMatmul); median microseconds over `repeats`."""
    import oracle as orc
    a_bits, b_bits = syn.pipeline_operands(256, 256, 256, seed=0)
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        qa, sa = orc.quantize(a_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
        qb, sb = orc.quantize(b_bits, "bf16", "e4m3fn", geometry="1x32", dim=-1)
        orc.scaled_matmul(qa, qb, sa, sb, "e4m3fn")
        times.append(time.perf_counter() - t0)
    return statistics.median(times) * 1e6


# ------------------------------------------------------------------- main

def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _all_reduce(ws, value, op_name):
    """Reduce a host scalar over ranks (timing bookkeeping only; the data
    path has no collective)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=getattr(dist.ReduceOp, op_name))
    return float(t.item())


def max_over_ranks(ws, value):
    return _all_reduce(ws, value, "MAX")


def sum_over_ranks(ws, value):
    return _all_reduce(ws, value, "SUM")


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # each step: the oracle over the whole sweep workload on every host core
    # (the same sample as the main arm's cpu_baseline)
    cores = host_cores()
    vals, spans = [], []
    for _ in range(args.warmup):
        oracle_sweep_parallel(cores, args.reference_rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, dt, _, desc = oracle_sweep_parallel(cores, args.reference_rows)
        vals.append(v)
        spans.append(dt)
    total = time.perf_counter() - t0
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8/f32",
        "data": "synthetic",
        "config": {"workload": "QuantizeMX sweep [8192,8192] {bf16,f16}x{e4m3fn,e5m2}x{plain,interleave}, 8x4 "
                               "blocks, dim=-2", "sample": desc},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc, "seconds_median": round(statistics.median(spans), 3)},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mx", choices=["mx", "reference"])
    ap.add_argument("--workload", default="all",
                    choices=["all", "sweep", "gemm", "fp4", "fused", "dequant", "dot", "gemm_fp4", "gemm_small_m",
                             "pipeline_256"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-rows", type=int, default=None,
                    help="rows of the [rows, 8192] slice each core quantizes in the reference arm (default: the "
                         "whole sweep workload over all cores; smaller for quick checks)")
    ap.add_argument("--fused-shape", default=None,
                    help="M,N,K of the fused workload (default 16384,28672,8192; smaller cases for profiling)")
    ap.add_argument("--fused-one-launch", action="store_true",
                    help="with --workload fused: run the fused call as one launch at any size (profiling small "
                         "cases; by default shorter products run as two launches)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
        return

    if args.fused_shape:
        Fused.SHAPE = tuple(int(v) for v in args.fused_shape.split(","))
    import torch
    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    import mx_fp8_microscaling_gb300 as mx

    peaks = load_peaks()
    global QUANT_SRC, GEMM_SRC, DEQUANT_SRC
    QUANT_SRC, GEMM_SRC, DEQUANT_SRC = _src_hashes()
    parts = {}
    want = (["sweep", "gemm", "fp4", "dequant", "fused", "dot", "gemm_fp4", "gemm_small_m", "pipeline_256"]
            if args.workload == "all"
            else [args.workload])
    builders = {"sweep": Sweep, "gemm": Gemm, "fp4": Fp4, "dequant": Dequant, "fused": Fused, "dot": Dot,
                "gemm_fp4": GemmFp4, "gemm_small_m": GemmSmallM, "pipeline_256": Pipeline256}
    api = Api(torch, mx)
    if args.fused_one_launch:
        if want != ["fused"]:
            raise SystemExit("--fused-one-launch needs --workload fused")
        mx.mx_debug_set_gemm_variant(2)
    for name in want:
        parts[name] = builders[name](torch, mx, api)
    torch.cuda.synchronize()
    launches_per_step = sum(p.launches for p in parts.values())

    timer = Timer(torch, capacity=max(args.steps, args.warmup) * sum(
        len(getattr(p, "ops", [None])) for p in parts.values()) + 64)
    for _ in range(args.warmup):
        for p in parts.values():
            p.step(timer)
    torch.cuda.synchronize()
    timer.collect()
    timer.reset()
    assert mx.mx_get_device_status() == 0

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.4)
    barrier(ws)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for _ in range(args.steps):
        for p in parts.values():
            p.step(timer)
    t_end.record()
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    timer.collect()
    status = mx.mx_get_device_status()
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")
    total_ms = max_over_ranks(ws, t_start.elapsed_time(t_end))

    line = {"metric": METRIC, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "mxfp8/f32",
            "data": "synthetic (seeded; distributions of the workload descriptions)",
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks}
    peak_fp8 = peaks["bf16"] * FP8_OVER_BF16
    fp8_src = f"{peaks['src']} bf16 burst x {FP8_OVER_BF16} (nominal MXFP8/bf16)"

    if "sweep" in parts:
        per_span = parts["sweep"].launches
        sweep_ms = max_over_ranks(ws, timer.totals["sweep"])
        n_launch = timer.counts["sweep"] * per_span
        value = sum_over_ranks(ws, SWEEP_BYTES * n_launch) / (sweep_ms * 1e-3) / 1e9
        # average launch duration = each step's span / its launches (gaps included)
        achieved = SWEEP_BYTES / (timer.avg_ms("sweep") / per_span * 1e-3) / 1e9
        line.update({"value": round(value, 2), "unit": "GB/s",
                     "config": {"workload": "QuantizeMX sweep [8192,8192] {bf16,f16}x{e4m3fn,e5m2}x"
                                            "{plain,interleave}, 8x4 blocks, dim=-2",
                                "bytes_per_launch": SWEEP_BYTES, "launches_per_step": per_span,
                                "l2": "inputs (128 MiB each, 4 distinct) larger than L2 and rotated",
                                "parallelism": f"replicas x{ws}"},
                     "roofline": {"bound": "hbm", "kernel": "quant_g84", "achieved": round(achieved, 1),
                                  "peak": peaks["hbm"], "unit": "GB/s",
                                  "frac": round(achieved / peaks["hbm"], 4), "peak_source": peaks["src"],
                                  "traffic": profiled_traffic("quant_g84", QUANT_SRC)}})
    else:
        line.update({"value": None, "unit": None, "config": {"workload": args.workload}})

    if "gemm" in parts:
        g = {}
        for fmt, out in Gemm.CASES:
            ms = timer.avg_ms(f"gemm_{fmt}_{out}")
            tf = GEMM_FLOP / (ms * 1e-3) / 1e12
            g[f"{fmt}_{out}"] = {"tflops": round(tf, 1), "ms": round(ms, 4), "frac": round(tf / peak_fp8, 4)}
        avg = statistics.mean(v["tflops"] for v in g.values())
        pipe_ms = (timer.totals["gemm_quantize"] + timer.totals["gemm_repack"]
                   + sum(timer.totals[f"gemm_{f}_{o}"] for f, o in Gemm.CASES)) / args.steps / 2
        line["scaled_matmul_vendor"] = vendor_gemm_reference(torch, parts["gemm"], args.steps)
        line["scaled_matmul"] = {
            "value": round(avg, 1), "unit": "TFLOP/s", "config": "M=N=K=8192, E8M0 per 32 along K",
            "pipeline_tflops_incl_quantize_repack": round(GEMM_FLOP / (pipe_ms * 1e-3) / 1e12, 1),
            "cases": g,
            "roofline": {"bound": "tensor", "kernel": "mx_gemm_2sm_kernel", "achieved": round(avg, 1),
                         "peak": round(peak_fp8, 1), "unit": "TFLOP/s", "frac": round(avg / peak_fp8, 4),
                         "peak_source": fp8_src,
                         "traffic": profiled_traffic("mx_gemm_2sm_kernel", GEMM_SRC)}}
    if "fp4" in parts:
        ms = timer.avg_ms("fp4") / Fp4.LAUNCHES   # per launch, from the span of back-to-back launches
        gbs = FP4_BYTES / (ms * 1e-3) / 1e9
        line["fp4_quantize"] = {"value": round(gbs, 1), "unit": "GB/s", "ms": round(ms, 4),
                                "config": f"[16384,16384] bf16 -> e2m1, 8x4, interleaved; {Fp4.LAUNCHES} launches "
                                          "a span",
                                "roofline": {"bound": "hbm", "kernel": "quant_g84<e2m1>", "achieved": round(gbs, 1),
                                             "peak": peaks["hbm"], "unit": "GB/s",
                                             "frac": round(gbs / peaks["hbm"], 4), "peak_source": peaks["src"],
                                             "traffic": profiled_traffic("quant_g84_fp4",
                                                                         QUANT_SRC)}}
    if "dequant" in parts:
        ms = timer.avg_ms("dequant") / Dequant.LAUNCHES   # per launch, from the span
        gbs = SWEEP_BYTES / (ms * 1e-3) / 1e9
        line["dequantize"] = {"value": round(gbs, 1), "unit": "GB/s", "ms": round(ms, 4),
                              "config": f"[8192,8192] e4m3fn + 8x4 scales -> bf16; {Dequant.LAUNCHES} launches a span",
                              "roofline": {"bound": "hbm", "kernel": "dequant_kernel", "achieved": round(gbs, 1),
                                           "peak": peaks["hbm"], "unit": "GB/s",
                                           "frac": round(gbs / peaks["hbm"], 4), "peak_source": peaks["src"],
                                           "traffic": profiled_traffic("dequant_kernel",
                                                                       DEQUANT_SRC)}}
    if "fused" in parts:
        fu = parts["fused"]
        ms = timer.avg_ms("fused")
        fused_flop = 2 * Fused.SHAPE[0] * Fused.SHAPE[1] * Fused.SHAPE[2]
        tf = fused_flop / (ms * 1e-3) / 1e12
        q_ms, g_ms = timer.avg_ms("fused_split_quantize"), timer.avg_ms("fused_split_gemm")
        line["fused"] = {"value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 4),
                         "launches_per_call": fu.launches_per_call,
                         "two_launches": {"quantize_x_ms": round(q_ms, 4), "gemm_ms": round(g_ms, 4),
                                          "total_ms": round(q_ms + g_ms, 4),
                                          "tflops": round(fused_flop / ((q_ms + g_ms) * 1e-3) / 1e12, 1)},
                         "config": "X[{0},{2}] bf16 quantized along K to e4m3fn in the GEMM launch, "
                                   "x W[{2},{1}] e4m3fn -> bf16".format(*Fused.SHAPE),
                         "roofline": {"bound": "tensor", "kernel": "mx_gemm_2sm_kernel<fused e4m3fn>",
                                      "achieved": round(tf, 1), "peak": round(peak_fp8, 1), "unit": "TFLOP/s",
                                      "frac": round(tf / peak_fp8, 4), "peak_source": fp8_src,
                                      "traffic": profiled_traffic("mx_gemm_2sm_kernel_fused",
                                                                  GEMM_SRC)}}

    if "gemm_fp4" in parts:
        ms = timer.avg_ms("gemm_fp4")
        tf = GEMM_FLOP / (ms * 1e-3) / 1e12
        peak_fp4 = peaks["bf16"] * FP4_OVER_BF16
        pipe_ms = (timer.totals["fp4_quantize_operands"] + timer.totals["fp4_repack"]
                   + timer.totals["gemm_fp4"]) / timer.counts["gemm_fp4"]
        line["scaled_matmul_fp4"] = {
            "value": round(tf, 1), "unit": "TFLOP/s", "ms": round(ms, 4),
            "config": "M=N=K=8192 e2m1 x e2m1 (kind::mxf4), E8M0 per 32 along K -> bf16",
            "pipeline_tflops_incl_quantize_repack": round(GEMM_FLOP / (pipe_ms * 1e-3) / 1e12, 1),
            "roofline": {"bound": "tensor", "kernel": "mx_gemm_2sm_kernel<true>", "achieved": round(tf, 1),
                         "peak": round(peak_fp4, 1), "unit": "TFLOP/s", "frac": round(tf / peak_fp4, 4),
                         "peak_source": f"{peaks['src']} bf16 burst x {FP4_OVER_BF16} (nominal FP4/bf16)",
                         "traffic": profiled_traffic("mx_gemm_2sm_kernel_fp4", GEMM_SRC)}}
        line["scaled_matmul_fp4"]["vendor_reference"] = vendor_fp4_reference(torch, parts["gemm_fp4"], args.steps)
    if "pipeline_256" in parts:
        us = timer.avg_ms("pipeline_256") * 1e3
        line["pipeline_256"] = {"us": round(us, 2), "tflops": round(2 * 256 ** 3 / (us * 1e-6) / 1e12, 3),
                                "us_cuda_graph": round(parts["pipeline_256"].graph_us(), 2),
                                "config": "M=N=K=256: quantize A, Bt (1x32 along K, e4m3fn), repack x2, "
                                          "ScaledMatmul -> f32; 5 launches, latency-bound"}
    if "gemm_small_m" in parts:
        sm = parts["gemm_small_m"]
        cases = {}
        for m in SMALL_M:
            us = timer.avg_ms(f"small_m_{m}") * 1e3 / SMALL_M_COPIES
            gbs = sm.bytes_per_call(m) / (us * 1e-6) / 1e9
            cases[str(m)] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm"], 4),
                             "split_k": sm.split[m]}
        top = cases[str(max(SMALL_M))]
        line["scaled_matmul_small_m"] = {
            "unit": "GB/s", "config": f"M x 8192 x 8192, M in {list(SMALL_M)}, e4m3fn -> bf16, SF-layout scales; "
                                      f"B rotated over {SMALL_M_COPIES} copies (256 MiB > L2); CUDA graphs",
            "cases": cases,
            "roofline": {"bound": "hbm", "kernel": "mx_gemm_kernel (split-K)", "achieved": top["gbs"],
                         "peak": peaks["hbm"], "unit": "GB/s", "frac": top["frac"], "peak_source": peaks["src"],
                         "traffic": profiled_traffic("mx_gemm_kernel_small_m", GEMM_SRC),
                         "note": f"M = {max(SMALL_M)}; bytes = B + A + both scale tensors + C"}}
        line["scaled_matmul_small_m"]["vendor_reference"] = vendor_small_m_reference(torch, sm, args.steps)
    if "dot" in parts:
        cases = {}
        for c in Dot.CASES:
            ms = timer.avg_ms(f"dot_{c}")
            cases[c] = {"tflops": round(DOT_FLOP / (ms * 1e-3) / 1e12, 1), "ms": round(ms, 4)}
        best = cases["rhs_bnk"]["tflops"]
        line["block_scaled_dot"] = {
            "value": best, "unit": "TFLOP/s",
            "config": "16 x 2048^3 e4m3fn -> bf16, batch dim 0, K innermost on lhs; rhs [B,N,K] or [B,K,N]; "
                      "whole call",
            "cases": cases,
            "roofline": {"bound": "tensor", "kernel": "mx_gemm_2sm_kernel", "achieved": best,
                         "peak": round(peak_fp8, 1), "unit": "TFLOP/s", "frac": round(best / peak_fp8, 4),
                         "peak_source": fp8_src, "note": "whole call, repack launches included"}}

    # end to end through the public API with host buffers: one
    # mx_quantize_host_batch call per step takes the 8 pinned host inputs and
    # writes pinned host outputs, copying chunks in and out on its own copy
    # streams while the previous chunk is quantized
    if "sweep" in parts:
        sw = parts["sweep"]
        host_in = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16 if k[0] == "bf16" else torch.float16)
                   .pin_memory() for k, v in sw.host.items()}
        host_out = {k: (torch.empty(d.numel(), dtype=torch.uint8).pin_memory(),
                        torch.empty(s.numel(), dtype=torch.uint8).pin_memory()) for k, (d, s) in sw.out.items()}
        specs = []
        for layout in ("plain", "interleave"):
            for in_dtype, fmt in SWEEP_VARIANTS:
                hd, hs = host_out[(layout, in_dtype, fmt)]
                specs.append(dict(x=host_in[(in_dtype, fmt)], out_dtype=fmt, out_data=hd, out_scale=hs,
                                  geometry="8x4", dim=-2, scale_layout=layout))
        jobs = mx.make_host_jobs(specs)
        work = torch.empty(mx.mx_quantize_host_batch_workspace(jobs, len(specs)), dtype=torch.uint8, device="cuda")
        batch_fn = mx.raw_library().mx_quantize_host_batch
        import ctypes
        stream_ptr = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        step_h2d = sum(sp["x"].numel() * 2 for sp in specs)
        # interleaved scales: only the live rows (4 of every 32) travel
        step_d2h = sum(sp["out_data"].numel() + (sp["out_scale"].numel() // 8 if sp["scale_layout"] == "interleave"
                                                 else sp["out_scale"].numel()) for sp in specs)
        h2d = d2h = 0

        def e2e_step():
            nonlocal h2d, d2h
            st = batch_fn(jobs, len(specs), 0, ctypes.c_void_p(work.data_ptr()), work.numel(), stream_ptr)
            if st:
                raise mx.MxError(st, "mx_quantize_host_batch")
            h2d += step_h2d
            d2h += step_d2h

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        h2d = d2h = 0
        barrier(ws)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize()
        dt = max_over_ranks(ws, time.perf_counter() - t0)
        e2e_value = sum_over_ranks(ws, SWEEP_BYTES * 8 * args.steps) / dt / 1e9
        line["e2e"] = {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d // args.steps,
                       "d2h_bytes_per_step": d2h // args.steps,
                       "note": "mx_quantize_host_batch: the 8 sweep tensors from pinned host memory, chunked "
                               "copies in, QuantizeMX, copies out to pinned host, overlapped; one call per step"}

    if rank == 0 and not args.no_cpu_baseline:
        v, dt, cores, desc = oracle_sweep_parallel()
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": round(dt, 2)}
        if "gemm" in parts:
            tf, dtg, gcores = oracle_gemm_parallel()
            line["cpu_baseline"]["scaled_matmul"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": gcores,
                                                     "sample": f"{gcores} full output rows of the 8192^3 product, "
                                                               "binary64 k-ordered sums, one row a core",
                                                     "seconds": round(dtg, 2)}
        if "pipeline_256" in parts:
            us = oracle_pipeline_256()
            line["cpu_baseline"]["pipeline_256"] = {"us": round(us, 1), "cores": 1,
                                                    "sample": "the whole 256^3 pipeline on one core"}
    # secondary results first, the headline ones last (readers that keep
    # only the end of the line still see them)
    order = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
             "vs_baseline", "dtype", "data", "gpu_launches", "config", "roofline", "clocks", "e2e", "cpu_baseline",
             "scaled_matmul_small_m", "block_scaled_dot", "pipeline_256", "scaled_matmul_fp4", "scaled_matmul_vendor",
             "dequantize", "fp4_quantize", "fused", "scaled_matmul"]
    line = {k: line[k] for k in order if k in line} | {k: v for k, v in line.items() if k not in order}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
