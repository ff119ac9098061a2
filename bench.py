"""Benchmark of the block-scaled quantization + GEMM hot path on GB300.

One step = one pass over every row of the hot path, each on its own seeded synthetic workload
(all inputs resident in HBM before the timed region):
  q2   MXFP8 quantize of 16384x4096 bf16 activations (4 outlier channels): E4M3 and E5M2,
       row-wise + column-wise, all four copies from one read (mx_quantize_dual)
  lin  MXFP8 linear layer M=8192 K=4096 N=14336: quantize X, W (E4M3) and G (E5M2) row- and
       column-wise, then fprop Y = X W^T, dgrad dX = G W, wgrad dW = G^T X (bf16 out)
  nv   NVFP4 8192^3: two-pass quantize of A and B, block-scaled FP4 GEMM (FP32 out)
  ds   DeepSeek FP8 M=4096 K=7168 N=2048: 1x128 / 128x128 quantize, GEMM with FP32 promotion
       every 128 of K (bf16 out)
An extra group, not part of the default step, is measured with --only mx4:
  mx4  MXFP4 8192^3: quantize A and B to E2M1 with E8M0 scales per 32 (row-wise), FP4 GEMM
       with the block scales in the MMA (FP32 out)
  fuse fprop 8192x4096x14336 with the MX (E4M3) quantization of Y fused into the GEMM epilogue
       (row-wise, then row- and column-wise), against the unfused pair (bf16 fprop, then
       row-wise MX quantize of Y)
  moe  grouped GEMM: 8 experts (K=4096 -> N=14336 each), 16384 routed rows split unevenly
       in multiples of 128, one launch (bf16 out), MXFP8 and NVFP4 (one global scale per expert);
       and the grouped NVFP4 quantization of the 8 experts' weights (one global scale each); the
       same experts as DeepSeek FP8 (1x128 token tiles, 128x128 weight blocks, promotion per 128)
  nvt  NVFP4 training options on one 8192x8192 tensor: the 16-point random Hadamard transform,
       stochastic rounding (random bytes read from HBM), both, and 16x16 2-D blocks written in
       both orientations
  blk  Float8BlockScaling through the MX GEMM at the DeepSeek shape (M=4096 K=7168 N=2048):
       power-of-two 1x128 / 128x128 quantize, scale conversion to E8M0, MXFP8 GEMM (bf16 out);
       and 2-D 32x32 MX quantize of the 14336x4096 weight (row- and column-wise)
value = sum of GEMM FLOPs in the step / step time (TFLOP/s); per-row times, GB/s, TFLOP/s and
roofline fractions are reported under "rows".  Every input exceeds or, within one step, is
separated from its next use by far more than the 129 MB L2, so no explicit flush is needed.

--impl reference times the CPU oracle (the plain C reference) on a bounded sample of the same
step and prints the same metric.  Multi-GPU runs (torchrun) are independent replicas: the path
has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MXFP8 GEMM TFLOP/s & quantize GB/s on 1 GB300 (fraction of roofline)"
WORKLOAD = "mxfp8_q16384x4096+mxfp8_linear_8192x4096x14336+nvfp4_8192^3+deepseek_fp8_4096x7168x2048"

# algorithmic work per call
F_LIN = 2 * 8192 * 4096 * 14336            # each of fprop / dgrad / wgrad
F_NV = 2 * 8192 ** 3
F_DS = 2 * 4096 * 7168 * 2048
F_MX4 = 2 * 8192 ** 3
MOE_SIZES = (3328, 1536, 2432, 1024, 2816, 1920, 2176, 1152)    # rows per expert, sum 16384
F_MOE = 2 * sum(MOE_SIZES) * 14336 * 4096
GEMM_FLOPS_STEP = 3 * F_LIN + F_NV + F_DS


def mx_q_bytes(rows, cols, copies=2):
    # read bf16 once + write codes (1 B) + E8M0 scales (1/32 B) for each copy
    return rows * cols * (2 + copies * (1 + 1 / 32))


def nv_q_bytes(rows, cols):
    # two reads of bf16 (amax pass, quantize pass) + packed codes (1/2 B) + UE4M3 scales (1/16 B)
    return rows * cols * (2 + 2 + 0.5 + 1 / 16)


def ds_q_bytes(rows, cols, tile_rows):
    return rows * cols * (2 + 1) + 4 * (rows // tile_rows) * (cols // 128)


Q2_BYTES = mx_q_bytes(16384, 4096, copies=4)
LINQ_BYTES = mx_q_bytes(8192, 4096) + mx_q_bytes(14336, 4096) + mx_q_bytes(8192, 14336)
NVQ_BYTES = 2 * nv_q_bytes(8192, 8192)
DSQ_BYTES = ds_q_bytes(4096, 7168, 1) + ds_q_bytes(2048, 7168, 128)
# MXFP4 row-wise: read bf16 + packed codes (1/2 B) + E8M0 scales (1/32 B), A and B
MX4Q_BYTES = 2 * 8192 * 8192 * (2 + 0.5 + 1 / 32)
# scale conversion: read the FP32 block scales, write one E8M0 byte per 32 elements
BLKCONV_BYTES = 4 * 4096 * 56 + 4 * 16 * 56 + (4096 + 2048) * 7168 // 32
W2DQ_BYTES = mx_q_bytes(14336, 4096)
NVT_RHT_BYTES = nv_q_bytes(8192, 8192)
NVT_SR_BYTES = nv_q_bytes(8192, 8192) + 8192 * 8192          # + one random byte per element
NVT_2D_BYTES = 8192 * 8192 * (2 + 2 + 2 * (0.5 + 1 / 16))       # both orientations
MOE4Q_BYTES = nv_q_bytes(len(MOE_SIZES) * 14336, 4096)           # every expert's weights, by groups


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# Dense tensor-core peaks.  "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 8, gives the
# dense rates as FP4 : FP8 : BF16 = 9 : 4.5 : 2.25 PFLOP/s, i.e. FP8 = 2x and FP4 = 4x BF16.  The
# FP8 and FP4 peaks are derived from the measured BF16 rate by that ratio; the BF16 figure is the
# burst one (a cuBLAS GEMM timed alone), because every timed GEMM here is one launch of a few
# hundred microseconds inside a sub-second region, not a seconds-long loop under the power cap
# (that loop ran at a median 1462 MHz; the bench's GEMMs run near 2000 MHz).
NOMINAL_TFLOPS = {"fp8": 4500.0, "fp4": 9000.0}
FP4_ROWS = ("nvgemm", "mx4gemm", "moe4gemm")


def tensor_peaks(peaks):
    """Derived dense peaks (TFLOP/s) for FP8 and FP4 from the measured BF16 burst rate."""
    b = peaks["bf16_tflops"]
    return {"fp8": 2.0 * b, "fp4": 4.0 * b,
            "source": f"{peaks['source']} bf16 burst {b:g} TFLOP/s x 2 (FP8) / x 4 (FP4): dense ratio "
                      "FP4:FP8:BF16 = 9:4.5:2.25 ('NVFP4: high accuracy with 4 bits' sec 8); nominal "
                      "FP8 4500 / FP4 9000 TFLOP/s beside it"}


# ------------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1] or [s for (_, s) in self.samples]
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz)}


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the driver's libnvidia-ml, by ctypes)
    every couple of milliseconds, so that a timed region of a few tens of milliseconds still gets
    dozens of samples.  Reads only; falls back to ClockSampler (nvidia-smi) where NVML cannot be
    loaded."""
    NVML_CLOCK_SM = 1
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid, index, period_s=0.002):
        self.uuid, self.index, self.period = uuid, index, period_s
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        self.thread = None

    def start(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = 1
            if self.uuid:
                rc = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h))
            if rc != 0:
                rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(self.index)), ctypes.byref(h))
            if rc != 0:
                return
            mx = ctypes.c_uint(0)
            lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx))
            self.max_mhz = float(mx.value)
            reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError, ValueError):
            return
        self.ok = True

        def run():
            mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
            while not self._stop.is_set():
                if lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) == 0 and \
                        reasons_fn(h, ctypes.byref(rs)) == 0:
                    self.samples.append((time.time(), float(mhz.value), int(rs.value)))
                time.sleep(self.period)

        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [r for r in self.samples if t0 <= r[0] <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": getattr(self, "max_mhz", None), "reasons": [], "samples": 0,
                    "source": "nvml"}
        reasons = sorted({name for (_, _, bits) in rows for b, name in self.REASONS.items() if bits & b})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(rows), "sm_mhz_min": min(r[1] for r in rows), "source": "nvml"}


def clock_sampler(dev_index):
    """An NVML sampler for the GPU torch calls `dev_index`, else nvidia-smi's."""
    import torch
    phys = os.environ.get("CUDA_VISIBLE_DEVICES", str(dev_index)).split(",")[dev_index] if os.environ.get(
        "CUDA_VISIBLE_DEVICES") else str(dev_index)
    uuid = None
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        uuid = u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        uuid = phys if phys.startswith("GPU-") else None
    s = NvmlSampler(uuid, phys if phys.isdigit() else dev_index)
    s.start()
    if s.ok:
        return s
    s = ClockSampler(phys)
    s.start()
    return s


# ------------------------------------------------------------------------------------ workload
def make_host_inputs(groups):
    """The seeded bf16 inputs of the given row groups, on the host (CPU tensors)."""
    from block_scaled_precision_mx_gb300 import synthetic
    host = {}
    if "q2" in groups:
        host["x2"] = synthetic.mxfp8_quantize()
    if "lin" in groups:
        host["X"], host["W"], host["G"] = synthetic.mxfp8_linear()
    if "nv" in groups:
        host["A4"], host["B4"] = synthetic.nvfp4_pair()
    if "ds" in groups:
        host["A5"], host["B5"] = synthetic.deepseek_pair()
    if "mx4" in groups:
        host["A6"], host["B6"] = synthetic.mxfp4_pair()
    if "nvt" in groups:
        host["A8"] = synthetic.nvfp4_pair()[0]
    if "fuse" in groups:
        host["X10"], host["W10"], _ = synthetic.mxfp8_linear()
    if "moe" in groups:
        host["A9"] = synthetic.normal(sum(MOE_SIZES), 4096, 1.0, 9000)
        host["B9"] = synthetic.normal(len(MOE_SIZES) * 14336, 4096, 0.02, 9001)
    if "blk" in groups:
        host["A7"], host["B7"] = synthetic.deepseek_pair()
        host["W7"] = synthetic.mxfp8_linear()[1]
    return host


class Workload:
    """All inputs and outputs of one step, resident on the device."""

    GROUPS = ("q2", "lin", "nv", "ds")   # the default step; "mx4" only with --only

    def __init__(self, dev, groups=GROUPS, host=None):
        """host: host inputs to reuse (from make_host_inputs, or another Workload's for the second
        buffer set of the pipelined end-to-end run) instead of drawing them again."""
        import torch
        import block_scaled_precision_mx_gb300 as mx
        self.mx = mx
        self.torch = torch
        self.dev = dev
        self.groups = tuple(groups)
        t = lambda x: x.to(dev)
        self.host = make_host_inputs(groups) if host is None else dict(host)
        self.d = {k: t(v) for k, v in self.host.items()}
        groups = self.groups
        u8 = lambda *s: torch.empty(*s, dtype=torch.uint8, device=dev)
        f32 = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)
        bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=dev)
        sb = mx.mx_scale_bytes
        self.launches_per_step = 0
        self._outs = []
        if "q2" in groups:   # E4M3 and E5M2 outputs
            self.q2 = {e: (u8(16384, 4096), u8(sb(16384, 4096)), u8(4096, 16384), u8(sb(4096, 16384))) for e in (0, 1)}
            self.launches_per_step += 1
            self._outs += [self.q2[0][0], self.q2[0][2], self.q2[1][0], self.q2[1][2]]
        if "lin" in groups:
            self.Xq = (u8(8192, 4096), u8(sb(8192, 4096)), u8(4096, 8192), u8(sb(4096, 8192)))
            self.Wq = (u8(14336, 4096), u8(sb(14336, 4096)), u8(4096, 14336), u8(sb(4096, 14336)))
            self.Gq = (u8(8192, 14336), u8(sb(8192, 14336)), u8(14336, 8192), u8(sb(14336, 8192)))
            self.Y, self.dX, self.dW = bf(8192, 14336), bf(8192, 4096), bf(14336, 4096)
            self.launches_per_step += 6
            self._outs += [self.Y, self.dX, self.dW]
        if "nv" in groups:
            self.A4q = (u8(8192, 4096), u8(sb(8192, 8192, 16, 1, mx.SCALE_UE4M3)), f32(1), u8(16))
            self.B4q = (u8(8192, 4096), u8(sb(8192, 8192, 16, 1, mx.SCALE_UE4M3)), f32(1), u8(16))
            self.Y4 = f32(8192, 8192)
            self.launches_per_step += 7
            self._outs += [self.Y4]
        if "ds" in groups:
            self.A5q = (u8(4096, 7168), f32(56, 4096))
            self.B5q = (u8(2048, 7168), f32(16, 56))
            self.Y5 = bf(4096, 2048)
            self.launches_per_step += 3
            self._outs += [self.Y5]
        if "fuse" in groups:
            self.X10q = (u8(8192, 4096), u8(sb(8192, 4096)))
            self.W10q = (u8(14336, 4096), u8(sb(14336, 4096)))
            self.Y10q = (u8(8192, 14336), u8(sb(8192, 14336)))
            self.Y10qT = (u8(14336, 8192), u8(sb(14336, 8192)))
            self.Y10 = bf(8192, 14336)
            self.launches_per_step += 4
            self._outs += [self.Y10q[0]]
        if "moe" in groups:
            m9, n9 = sum(MOE_SIZES), len(MOE_SIZES) * 14336
            self.A9q = (u8(m9, 4096), u8(sb(m9, 4096)))
            self.B9q = (u8(n9, 4096), u8(sb(n9, 4096)))
            self.off9 = torch.tensor([0] + list(__import__("itertools").accumulate(MOE_SIZES)), dtype=torch.int64,
                                     device=dev)
            self.Y9 = bf(m9, 14336)
            # NVFP4 experts: the tokens as one tensor (one global scale), each expert's weights as
            # their own tensor (one global scale each)
            self.A9n = (u8(m9, 2048), u8(sb(m9, 4096, 16, 1, mx.SCALE_UE4M3)), f32(1), u8(16))
            self.B9n = (u8(n9, 2048), u8(sb(n9, 4096, 16, 1, mx.SCALE_UE4M3)), f32(len(MOE_SIZES)),
                        u8(16 * len(MOE_SIZES)))
            self.woff9 = torch.arange(0, n9 + 1, 14336, dtype=torch.int64, device=dev)
            # DeepSeek FP8 experts: tokens in 1x128 tiles, the stacked weights in 128x128 blocks
            self.A9d = (u8(m9, 4096), f32(4096 // 128, m9))
            self.B9d = (u8(n9, 4096), f32(n9 // 128, 4096 // 128))
            self.launches_per_step += 6
            self._outs += [self.Y9]
        if "nvt" in groups:
            g8 = torch.Generator(device="cpu").manual_seed(8100)
            self.R8 = torch.randint(0, 256, (8192, 8192), dtype=torch.uint8, generator=g8).to(dev)
            nsb = sb(8192, 8192, 16, 1, mx.SCALE_UE4M3)
            self.A8q = (u8(8192, 4096), u8(nsb), f32(1), u8(16))
            self.A8t = (u8(8192, 4096), u8(nsb), u8(4096, 8192), u8(nsb))
            self.launches_per_step += 12
            self._outs += [self.A8q[0], self.A8t[0], self.A8t[2]]
        if "blk" in groups:
            self.A7q = (u8(4096, 7168), f32(56, 4096), u8(4096 * 7168 // 32))
            self.B7q = (u8(2048, 7168), f32(16, 56), u8(2048 * 7168 // 32))
            self.W7q = (u8(14336, 4096), u8(sb(14336, 4096)), u8(4096, 14336), u8(sb(4096, 14336)))
            self.Y7 = bf(4096, 2048)
            self.launches_per_step += 6
            self._outs += [self.Y7]
        if "mx4" in groups:
            self.A6q = (u8(8192, 4096), u8(sb(8192, 8192)))
            self.B6q = (u8(8192, 4096), u8(sb(8192, 8192)))
            self.Y6 = f32(8192, 8192)
            self.launches_per_step += 3
            self._outs += [self.Y6]

    def outputs(self):
        return list(self._outs)

    def step(self, ev=None):
        """One pass of the hot path.  `ev(name)` records a CUDA event at row boundaries."""
        mx = self.mx
        d = self.d
        mark = ev or (lambda name: None)
        g = self.groups
        if "q2" in g:
            mark("q2")
            mx.mx_quantize_dual(d["x2"], layout=mx.BOTH, e4m3=self.q2[0], e5m2=self.q2[1])
        if "lin" in g:
            mark("linq")
            for src, dst, e in ((d["X"], self.Xq, 0), (d["W"], self.Wq, 0), (d["G"], self.Gq, 1)):
                mx.mx_quantize(src, elem=e, layout=mx.BOTH, q_row=dst[0], s_row=dst[1], q_col=dst[2], s_col=dst[3])
            mark("fprop")
            mx.mx_gemm(self.Xq[0], self.Xq[1], 0, self.Wq[0], self.Wq[1], 0, 8192, 14336, 4096, mx.OUT_BF16, out=self.Y)
            mark("dgrad")
            mx.mx_gemm(self.Gq[0], self.Gq[1], 1, self.Wq[2], self.Wq[3], 0, 8192, 4096, 14336, mx.OUT_BF16,
                       out=self.dX)
            mark("wgrad")
            mx.mx_gemm(self.Gq[2], self.Gq[3], 1, self.Xq[2], self.Xq[3], 0, 14336, 4096, 8192, mx.OUT_BF16,
                       out=self.dW)
        if "nv" in g:
            mark("nvq")
            for src, dst in ((d["A4"], self.A4q), (d["B4"], self.B4q)):
                mx.nvfp4_quantize(src, q_packed=dst[0], s_ue4m3=dst[1], gscale=dst[2], workspace=dst[3])
            mark("nvgemm")
            mx.nvfp4_gemm(self.A4q[0], self.A4q[1], self.A4q[2], self.B4q[0], self.B4q[1], self.B4q[2], 8192, 8192,
                          8192, mx.OUT_F32, out=self.Y4)
        if "ds" in g:
            mark("dsq")
            mx.mx_quantize(d["A5"], block=128, block_rows=1, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE,
                           q_row=self.A5q[0], s_row=self.A5q[1])
            mx.mx_quantize(d["B5"], block=128, block_rows=128, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE,
                           q_row=self.B5q[0], s_row=self.B5q[1])
            mark("dsgemm")
            mx.fp8_blockwise_gemm(self.A5q[0], self.A5q[1], self.B5q[0], self.B5q[1], 4096, 2048, 7168, mx.OUT_BF16,
                                  out=self.Y5)
        if "fuse" in g:
            if not getattr(self, "_fuse_quantized", False):     # operands quantized once, outside the rows
                mx.mx_quantize(d["X10"], layout=mx.ROWWISE, q_row=self.X10q[0], s_row=self.X10q[1])
                mx.mx_quantize(d["W10"], layout=mx.ROWWISE, q_row=self.W10q[0], s_row=self.W10q[1])
                self._fuse_quantized = True
            mark("fusedgemm")
            mx.mx_gemm_mxout(self.X10q[0], self.X10q[1], mx.E4M3, self.W10q[0], self.W10q[1], mx.E4M3, 8192, 14336,
                             4096, q_out=self.Y10q[0], s_out=self.Y10q[1])
            mark("fusedboth")
            mx.mx_gemm_mxout_ex(self.X10q[0], self.X10q[1], mx.E4M3, self.W10q[0], self.W10q[1], mx.E4M3, 8192,
                                14336, 4096, layout=mx.BOTH, q_row=self.Y10q[0], s_row=self.Y10q[1],
                                q_col=self.Y10qT[0], s_col=self.Y10qT[1])
            mark("unfused")
            mx.mx_gemm(self.X10q[0], self.X10q[1], mx.E4M3, self.W10q[0], self.W10q[1], mx.E4M3, 8192, 14336, 4096,
                       mx.OUT_BF16, out=self.Y10)
            mx.mx_quantize(self.Y10, layout=mx.ROWWISE, q_row=self.Y10q[0], s_row=self.Y10q[1])
        if "moe" in g:
            if not getattr(self, "_moe_quantized", False):      # operands quantized once, outside the rows
                mx.mx_quantize(d["A9"], layout=mx.ROWWISE, q_row=self.A9q[0], s_row=self.A9q[1])
                mx.mx_quantize(d["B9"], layout=mx.ROWWISE, q_row=self.B9q[0], s_row=self.B9q[1])
                self._moe_quantized = True
                a = self.A9n
                mx.nvfp4_quantize(d["A9"], q_packed=a[0], s_ue4m3=a[1], gscale=a[2], workspace=a[3])
                mx.mx_quantize(d["A9"], block=128, block_rows=1, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE,
                               q_row=self.A9d[0], s_row=self.A9d[1])
                mx.mx_quantize(d["B9"], block=128, block_rows=128, sfmt=mx.SCALE_FP32, layout=mx.ROWWISE,
                               q_row=self.B9d[0], s_row=self.B9d[1])
            mark("moe4q")
            b = self.B9n                                          # each expert's weights: own global scale
            mx.nvfp4_quantize_grouped(d["B9"], self.woff9, q_packed=b[0], s_ue4m3=b[1], gscale=b[2], workspace=b[3])
            mark("moegemm")
            mx.mx_gemm_grouped(self.A9q[0], self.A9q[1], mx.E4M3, self.B9q[0], self.B9q[1], mx.E4M3, self.off9,
                               sum(MOE_SIZES), 14336, 4096, mx.OUT_BF16, out=self.Y9)
            mark("moe4gemm")
            mx.nvfp4_gemm_grouped(self.A9n[0], self.A9n[1], self.A9n[2], self.B9n[0], self.B9n[1], self.B9n[2],
                                  self.off9, sum(MOE_SIZES), 14336, 4096, mx.OUT_BF16, out=self.Y9)
            mark("moedsgemm")
            mx.fp8_blockwise_gemm_grouped(self.A9d[0], self.A9d[1], self.B9d[0], self.B9d[1], self.off9,
                                          sum(MOE_SIZES), 14336, 4096, mx.OUT_BF16, out=self.Y9)
        if "nvt" in g:
            q = self.A8q
            mark("nvq_rht")
            mx.nvfp4_quantize_ex(d["A8"], rht=True, signs=0xB4D2, q_packed=q[0], s_ue4m3=q[1], gscale=q[2],
                                 workspace=q[3])
            mark("nvq_sr")
            mx.nvfp4_quantize_ex(d["A8"], rbits=self.R8, q_packed=q[0], s_ue4m3=q[1], gscale=q[2], workspace=q[3])
            mark("nvq_rht_sr")
            mx.nvfp4_quantize_ex(d["A8"], rht=True, signs=0xB4D2, rbits=self.R8, q_packed=q[0], s_ue4m3=q[1],
                                 gscale=q[2], workspace=q[3])
            mark("nvq_2d")
            mx.nvfp4_quantize_2d(d["A8"], out=self.A8t, gscale=q[2], workspace=q[3])
        if "blk" in g:
            mark("blkq")
            mx.mx_quantize(d["A7"], block=128, block_rows=1, sfmt=mx.SCALE_FP32_POW2, layout=mx.ROWWISE,
                           q_row=self.A7q[0], s_row=self.A7q[1])
            mx.mx_quantize(d["B7"], block=128, block_rows=128, sfmt=mx.SCALE_FP32_POW2, layout=mx.ROWWISE,
                           q_row=self.B7q[0], s_row=self.B7q[1])
            mark("blkconv")
            mx.mx_scales_from_fp32_blocks(self.A7q[1], 4096, 7168, 1, out=self.A7q[2])
            mx.mx_scales_from_fp32_blocks(self.B7q[1], 2048, 7168, 128, out=self.B7q[2])
            mark("blkgemm")
            mx.mx_gemm(self.A7q[0], self.A7q[2], mx.E4M3, self.B7q[0], self.B7q[2], mx.E4M3, 4096, 2048, 7168,
                       mx.OUT_BF16, out=self.Y7)
            mark("w2dq")
            mx.mx_quantize(d["W7"], block=32, block_rows=32, layout=mx.BOTH, q_row=self.W7q[0], s_row=self.W7q[1],
                           q_col=self.W7q[2], s_col=self.W7q[3])
        if "mx4" in g:
            mark("mx4q")
            for src, dst in ((d["A6"], self.A6q), (d["B6"], self.B6q)):
                mx.mx_quantize(src, elem=mx.E2M1, layout=mx.ROWWISE, q_row=dst[0], s_row=dst[1])
            mark("mx4gemm")
            mx.mx_gemm(self.A6q[0], self.A6q[1], mx.E2M1, self.B6q[0], self.B6q[1], mx.E2M1, 8192, 8192, 8192,
                       mx.OUT_F32, out=self.Y6)
        mark("end")


ROW_ORDER = ["q2", "linq", "fprop", "dgrad", "wgrad", "nvq", "nvgemm", "dsq", "dsgemm", "blkq", "blkconv", "blkgemm",
             "w2dq", "mx4q", "mx4gemm", "nvq_rht", "nvq_sr", "nvq_rht_sr", "nvq_2d", "moe4q", "moegemm", "moe4gemm",
             "moedsgemm", "fusedgemm", "fusedboth", "unfused"]


def row_report(name, ms, peaks):
    """Per-row throughput and roofline fraction from its average time per step (ms)."""
    s = ms / 1e3
    hbm_rows = {"q2": Q2_BYTES, "linq": LINQ_BYTES, "nvq": NVQ_BYTES, "dsq": DSQ_BYTES, "mx4q": MX4Q_BYTES,
                "blkq": DSQ_BYTES, "blkconv": BLKCONV_BYTES, "w2dq": W2DQ_BYTES, "nvq_rht": NVT_RHT_BYTES,
                "nvq_sr": NVT_SR_BYTES, "nvq_rht_sr": NVT_SR_BYTES, "nvq_2d": NVT_2D_BYTES, "moe4q": MOE4Q_BYTES}
    if name in hbm_rows:
        b = hbm_rows[name]
        gbs = b / s / 1e9
        return {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                "bound": "hbm", "bytes": int(b)}
    f = ROW_FLOPS[name]
    tf = f / s / 1e12
    kind = "fp4" if name in FP4_ROWS else "fp8"
    peak = tensor_peaks(peaks)[kind]
    return {"ms": round(ms, 4), "TFLOP/s": round(tf, 1), "frac": round(tf / peak, 4),
            "frac_nominal": round(tf / NOMINAL_TFLOPS[kind], 4), "bound": "tensor", "peak": kind, "flops": int(f)}


ROW_FLOPS = {"fprop": F_LIN, "dgrad": F_LIN, "wgrad": F_LIN, "nvgemm": F_NV, "dsgemm": F_DS, "mx4gemm": F_MX4,
             "blkgemm": F_DS, "moegemm": F_MOE, "moe4gemm": F_MOE, "moedsgemm": F_MOE, "fusedgemm": F_LIN,
             "fusedboth": F_LIN, "unfused": F_LIN}


# ------------------------------------------------------------------------------------ CPU oracle
ORACLE_GEMMS = ("fprop", "dgrad", "wgrad", "nvgemm", "dsgemm")
ORACLE_QUANT_BYTES = {"q2": Q2_BYTES, "linq": LINQ_BYTES, "nvq": NVQ_BYTES, "dsq": DSQ_BYTES}


def oracle_quantize_all(host):
    """Every quantizer of the default step on its full tensor, by the CPU oracle.  Returns the
    oracle's codes and scales the sampled products read, and the seconds each row took."""
    import oracle as orc
    t, out = {}, {}

    def timed(name, fn):
        t0 = time.perf_counter()
        r = fn()
        t[name] = time.perf_counter() - t0
        return r

    timed("q2", lambda: [(orc.mx_quantize_rowwise(host["x2"], f), orc.mx_quantize_colwise(host["x2"], f))
                         for f in (orc.E4M3, orc.E5M2)])

    def linq():
        for name, f in (("X", orc.E4M3), ("W", orc.E4M3), ("G", orc.E5M2)):
            out[name] = (orc.mx_quantize_rowwise(host[name], f), orc.mx_quantize_colwise(host[name], f))
    timed("linq", linq)
    out["A4"], out["B4"] = timed("nvq", lambda: (orc.nv_quantize(host["A4"]), orc.nv_quantize(host["B4"])))
    out["A5"], out["B5"] = timed("dsq", lambda: (orc.ds_quantize_1x128(host["A5"]), orc.ds_quantize_128x128(host["B5"])))
    return out, t


def oracle_gemm_sample(q, rows_per_gemm, which=ORACLE_GEMMS):
    """The products `which` of the default step, each on `rows_per_gemm` evenly spaced output rows
    (all N columns, full K), from the oracle's own codes; returns {row: (seconds, flops,
    full-size flops)}."""
    import numpy as np
    import oracle as orc
    (xr, xc), (wr, wc), (gr, gc) = q["X"], q["W"], q["G"]
    prods = {  # name: (fn(rows), M, N, K)
        "fprop": (lambda r: orc.mx_gemm(xr[0], xr[1], orc.E4M3, wr[0], wr[1], orc.E4M3, rows=r), 8192, 14336, 4096),
        "dgrad": (lambda r: orc.mx_gemm(gr[0], gr[1], orc.E5M2, wc[0], wc[1], orc.E4M3, rows=r), 8192, 4096, 14336),
        "wgrad": (lambda r: orc.mx_gemm(gc[0], gc[1], orc.E5M2, xc[0], xc[1], orc.E4M3, rows=r), 14336, 4096, 8192),
        "nvgemm": (lambda r: orc.nv_gemm(*q["A4"], *q["B4"], rows=r), 8192, 8192, 8192),
        "dsgemm": (lambda r: orc.ds_gemm(q["A5"][0], q["A5"][1], q["B5"][0], q["B5"][1], rows=r), 4096, 2048, 7168),
    }
    res = {}
    for name in which:
        fn, M, N, K = prods[name]
        rows = np.linspace(0, M - 1, rows_per_gemm).astype(np.int64)
        t0 = time.perf_counter()
        fn(rows)
        res[name] = (time.perf_counter() - t0, 2.0 * len(rows) * N * K, 2.0 * M * N * K)
    return res


def oracle_step(host, quant_runs, rows_per_gemm, which=ORACLE_GEMMS):
    """The CPU oracle on one bounded sample of the step: every quantizer on its full tensor
    (the median of `quant_runs` runs), the products `which` on `rows_per_gemm` output rows each.
    `value` is the GEMM FLOPs the sample computed over the seconds it took (quantizers included),
    the metric the GPU step reports; the linear projection of the products to all their rows is
    reported beside it (only when every product was sampled)."""
    import oracle as orc
    runs = []
    q = None
    for _ in range(quant_runs):
        q, t = oracle_quantize_all(host)
        runs.append(t)
    tq = {k: statistics.median(r[k] for r in runs) for k in runs[0]}
    g = oracle_gemm_sample(q, rows_per_gemm, which)
    t_q = sum(tq.values())
    t_g = sum(v[0] for v in g.values())
    f_g = sum(v[1] for v in g.values())
    t_proj = t_q + sum(v[0] * v[2] / v[1] for v in g.values())
    return {
        "value": f_g / (t_q + t_g) / 1e12, "unit": "TFLOP/s", "cores": orc.num_threads(), "kind": "oracle",
        "seconds": t_q + t_g,
        "sample": (f"every quantizer on its full tensor (median of {quant_runs}); {', '.join(which)} "
                   f"on {rows_per_gemm} evenly spaced output rows each (all columns, full K); "
                   "value = the sample's GEMM FLOPs / its seconds"),
        "quantize_GB/s": round(sum(ORACLE_QUANT_BYTES.values()) / t_q / 1e9, 3),
        "quantize_s": {k: round(v, 3) for k, v in tq.items()},
        "gemm_GFLOP/s": round(f_g / t_g / 1e9, 3),
        "projected_full_step_s": round(t_proj, 1) if len(which) == len(ORACLE_GEMMS) else None,
        "projected_full_step_TFLOP/s": GEMM_FLOPS_STEP / t_proj / 1e12 if len(which) == len(ORACLE_GEMMS) else None,
    }


# ------------------------------------------------------------------------------------ main
def max_over_ranks(ms, dist=None, device=None):
    """Slowest rank's time (ms): the whole job finishes when the last replica does."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job throughput: units every rank processed / the slowest rank's time (per second)."""
    return world * units_per_rank / (ms_max / 1e3)


def run_library_reference(args):
    """Context only: cuBLASLt through torch._scaled_mm (and bf16 matmul) on the bench's GEMM
    shapes, with random operands of the same types.  Prints one JSON line; never part of the
    bench value and never on the product path."""
    import torch
    dev = torch.device("cuda")

    def timeit(fn, reps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    out = {"kind": "library_reference", "library": f"cuBLASLt via torch {torch.__version__}",
           "device": torch.cuda.get_device_name(), "TFLOP/s": {}}
    for (M, N, K) in [(8192, 14336, 4096), (8192, 4096, 14336), (14336, 4096, 8192), (8192, 8192, 8192),
                      (4096, 2048, 7168)]:
        fl = 2 * M * N * K
        key = f"{M}x{N}x{K}"
        res = {}
        a = torch.randn(M, K, device=dev, dtype=torch.bfloat16)
        b = torch.randn(N, K, device=dev, dtype=torch.bfloat16)
        res["bf16"] = round(fl / timeit(lambda: a @ b.t()) / 1e9, 1)
        a8, b8 = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev)
        try:
            res["fp8_per_tensor"] = round(fl / timeit(lambda: torch._scaled_mm(
                a8, b8.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)) / 1e9, 1)
        except Exception as e:  # noqa: BLE001 -- report, do not fail
            res["fp8_per_tensor"] = f"unavailable: {str(e)[:80]}"
        try:
            sa = torch.full((M * K // 32,), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
            sb = torch.full((N * K // 32,), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
            res["mxfp8"] = round(fl / timeit(lambda: torch._scaled_mm(
                a8, b8.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)) / 1e9, 1)
        except Exception as e:  # noqa: BLE001
            res["mxfp8"] = f"unavailable: {str(e)[:80]}"
        try:
            a4 = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
            b4 = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
            sa4 = torch.full((M * K // 16,), 0x38, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
            sb4 = torch.full((N * K // 16,), 0x38, dtype=torch.uint8, device=dev).view(torch.float8_e4m3fn)
            res["nvfp4"] = round(fl / timeit(lambda: torch._scaled_mm(
                a4, b4.t(), scale_a=sa4, scale_b=sb4, out_dtype=torch.bfloat16)) / 1e9, 1)
        except Exception as e:  # noqa: BLE001
            res["nvfp4"] = f"unavailable: {str(e)[:80]}"
        out["TFLOP/s"][key] = res
    print(json.dumps(out))
    return 0


def headline(rows, rows_ms, present, peaks):
    """The metric's two figures as top-level keys -- the MXFP8 linear-layer GEMMs' TFLOP/s and the
    quantizers' GB/s -- and which rows meet the targets (quantizers >= 0.80 of HBM, block-scaled
    GEMMs >= 0.70 of the dense peak), each against the derived and the nominal peak."""
    out = {}
    tpk = tensor_peaks(peaks)
    lin = [n for n in ("fprop", "dgrad", "wgrad") if n in present]
    if lin:
        tf = len(lin) * F_LIN / (sum(rows_ms[n] for n in lin) / 1e3) / 1e12
        out["mxfp8_gemm_tflops"] = round(tf, 1)
        out["mxfp8_gemm_frac"] = round(tf / tpk["fp8"], 4)
        out["mxfp8_gemm_frac_nominal"] = round(tf / NOMINAL_TFLOPS["fp8"], 4)
    qrows = [n for n in present if "bytes" in rows[n]]
    if qrows:
        gbs = sum(rows[n]["bytes"] for n in qrows) / (sum(rows_ms[n] for n in qrows) / 1e3) / 1e9
        out["quantize_gbs"] = round(gbs, 1)
        out["quantize_frac"] = round(gbs / peaks["hbm_gbs"], 4)
    tq = {n: rows[n]["frac"] for n in qrows}
    tg = {n: (rows[n]["frac"], rows[n]["frac_nominal"]) for n in present if rows[n].get("bound") == "tensor"}
    out["targets"] = {
        "quantizers_hbm_0.80": {"met": sorted(n for n, f in tq.items() if f >= 0.80),
                                "missed": {n: f for n, f in tq.items() if f < 0.80}},
        "gemms_peak_0.70": {"met": sorted(n for n, (f, fn) in tg.items() if f >= 0.70),
                            "missed": {n: f for n, (f, fn) in tg.items() if f < 0.70},
                            "met_nominal": sorted(n for n, (f, fn) in tg.items() if fn >= 0.70),
                            "missed_nominal": {n: fn for n, (f, fn) in tg.items() if fn < 0.70}},
    }
    return out


def measure_mx512(dev, peaks, reps=200):
    """MXFP8 512x512x512 (E4M3, FP32 out) from its seeded bf16 operands: the quantization of both
    operands and the product, each timed per call with CUDA events on the launching stream
    (median of `reps`).  A latency-bound case: its operands stay in L2 between calls."""
    import torch
    import block_scaled_precision_mx_gb300 as mx
    from block_scaled_precision_mx_gb300 import synthetic
    a, b = (t.to(dev) for t in synthetic.mxfp8_gemm_512())
    sb = mx.mx_scale_bytes(512, 512)
    qa, sa, qb, sb_ = (torch.empty(n, dtype=torch.uint8, device=dev) for n in (512 * 512, sb, 512 * 512, sb))
    y = torch.empty(512, 512, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def quant():
        mx.mx_quantize(a, layout=mx.ROWWISE, q_row=qa, s_row=sa)
        mx.mx_quantize(b, layout=mx.ROWWISE, q_row=qb, s_row=sb_)

    def gemm():
        mx.mx_gemm(qa, sa, mx.E4M3, qb, sb_, mx.E4M3, 512, 512, 512, mx.OUT_F32, out=y)

    def median_us(fn):
        for _ in range(10):
            fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ts) * 1e3

    def graph_us(fn, n=50):
        """Device time per call from a CUDA graph of n back-to-back calls (no per-call host work)."""
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                fn()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    for _ in range(n):
                        fn()
            stream.wait_stream(side)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / n
        except Exception:  # noqa: BLE001 -- capture unsupported here: report the per-call time only
            torch.cuda.synchronize()
            return None

    tq, tg = median_us(quant), median_us(gemm)
    gq, gg = graph_us(quant), graph_us(gemm)
    flops = 2 * 512 ** 3
    tf = flops / (tg / 1e6) / 1e12
    qbytes = 2 * mx_q_bytes(512, 512, copies=1)
    return {"mx512": {"config": "MXFP8 E4M3 GEMM 512x512x512, FP32 out, operands quantized row-wise (E8M0 per 32)",
                      "gemm_us": round(tg, 2), "TFLOP/s": round(tf, 1),
                      "frac": round(tf / tensor_peaks(peaks)["fp8"], 5),
                      "frac_nominal": round(tf / NOMINAL_TFLOPS["fp8"], 5),
                      "quantize_us": round(tq, 2), "quantize_GB/s": round(qbytes / (tq / 1e6) / 1e9, 1),
                      "gemm_us_graph": None if gg is None else round(gg, 2),
                      "quantize_us_graph": None if gq is None else round(gq, 2),
                      "reps": reps,
                      "timing": "*_us: CUDA events around each call (the binding's argument marshalling, the "
                                "library's tensor-map lookup and the launch included); *_us_graph: per call inside "
                                "a CUDA graph of 50 back-to-back calls",
                      "bound": "latency (2 launches / 1 launch of a few microseconds; L2-resident)"}}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


BASE_CONFIG = {"workload": WORKLOAD,
               "l2": "inputs larger than L2 (129 MB) between reuses; no explicit flush",
               "rows": "per-row times and roofline from a second timed pass of the same K steps with an "
                       "event at every row boundary; value from K steps with none"}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample of the step per
    timed step (rank 0 only; other ranks exit without work)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as orc
    orc.build()
    host = make_host_inputs(Workload.GROUPS)
    # each step: every quantizer on its full tensor and one product (in turn) on one output row
    # per host thread, so that K + W steps take a few minutes
    rows = orc.num_threads()
    samples = []
    t0 = time.perf_counter()
    for i in range(args.warmup + args.steps):
        r = oracle_step(host, 1, rows, (ORACLE_GEMMS[i % len(ORACLE_GEMMS)],))
        if i >= args.warmup:
            samples.append(r)
    wall = time.perf_counter() - t0
    sec = sum(r["seconds"] for r in samples)
    flops = sum(r["value"] * 1e12 * r["seconds"] for r in samples)
    value = flops / sec / 1e12
    cpu = dict(samples[-1])
    cpu["value"] = value
    cpu["sample"] = ("per step: every quantizer on its full tensor; one of " + ", ".join(ORACLE_GEMMS) +
                     f" in turn on {rows} evenly spaced output rows (all columns, full K); value = the steps' "
                     "GEMM FLOPs / their seconds")
    for k in ("seconds", "projected_full_step_s", "projected_full_step_TFLOP/s", "quantize_s", "gemm_GFLOP/s"):
        cpu.pop(k, None)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec / len(samples) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": dict(BASE_CONFIG, parallelism=f"replicas x{world}"),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--library-reference", action="store_true",
                    help="print cuBLASLt reference throughputs for the GEMM shapes (context only)")
    ap.add_argument("--only", default=None,
                    help="comma-separated subset of row groups (q2, lin, nv, ds; mx4, blk, nvt, moe and fuse are measured only here) for profiling runs; "
                         "a line printed with --only is not a bench value")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.library_reference:
        return run_library_reference(args)
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_env()
    groups = tuple(args.only.split(",")) if args.only else Workload.GROUPS
    host = make_host_inputs(groups)
    # the oracle runs (and its OpenMP pool is created) before the first GPU call
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only:
        import oracle as orc
        orc.build()
        cpu = oracle_step(host, 3, orc.num_threads())

    import torch
    import block_scaled_precision_mx_gb300 as mx
    from block_scaled_precision_mx_gb300 import build as mxbuild
    mxbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    peaks = load_peaks()

    wl = Workload(dev, groups, host=host)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        wl.step()
    assert mx.mx_check() == mx.MX_OK

    # per-row events over the timed steps
    evs = []

    def mark_factory(lst):
        def mark(name):
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            lst.append((name, e))
        return mark

    sampler = clock_sampler(local)
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        wl.step()            # no events between the rows: events there cost ~1.5% of the step
    stop.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if pg:
        pg.barrier()
    # per-row times and the roofline: a second timed pass of K steps with an event at every row
    # boundary (the clock samples cover both passes)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        lst = []
        wl.step(mark_factory(lst))
        evs.append(lst)
    torch.cuda.synchronize()
    t_wall2 = time.time()
    if pg:
        pg.barrier()
    sampler.stop()
    status = mx.mx_check()
    if status != mx.MX_OK:
        raise RuntimeError(f"device status after timed region: {mx.status_string(status)}")
    ms_total = max_over_ranks(start.elapsed_time(stop), pg, dev)
    ms_step = ms_total / args.steps

    rows_ms = {n: 0.0 for n in ROW_ORDER}
    for lst in evs:
        for (n, e0), (_, e1) in zip(lst[:-1], lst[1:]):
            rows_ms[n] += e0.elapsed_time(e1)
    rows_ms = {n: v / len(evs) for n, v in rows_ms.items()}
    present = [n for n in ROW_ORDER if rows_ms[n] > 0]
    rows = {n: row_report(n, rows_ms[n], peaks) for n in present}
    # the unfused comparison repeats the fused rows' product: its FLOPs are not counted again
    step_flops = sum(ROW_FLOPS.get(n, 0) for n in present if n != "unfused")

    # dominant kernel: the kernel (all its launches in the step) with the largest share
    kernels = {"mx_gemm": ["fprop", "dgrad", "wgrad"], "nvfp4_gemm": ["nvgemm"], "fp8_blockwise_gemm": ["dsgemm"],
               "mx_quantize": ["q2", "linq"], "nvfp4_quantize": ["nvq"], "ds_quantize": ["dsq"],
               "mxfp4_gemm": ["mx4gemm"], "mxfp4_quantize": ["mx4q"], "mx_gemm_blocks": ["blkgemm"],
               "pow2_block_quantize": ["blkq"], "mx_scales_from_fp32_blocks": ["blkconv"],
               "mx_quantize_2d32": ["w2dq"], "nvfp4_quantize_ex": ["nvq_rht", "nvq_sr", "nvq_rht_sr"],
               "nvfp4_quantize_2d": ["nvq_2d"], "nvfp4_quantize_grouped": ["moe4q"], "mx_gemm_grouped": ["moegemm"],
               "nvfp4_gemm_grouped": ["moe4gemm"], "fp8_blockwise_gemm_grouped": ["moedsgemm"],
               "mx_gemm_mxout": ["fusedgemm", "fusedboth"],
               "mx_gemm_then_quantize": ["unfused"]}
    kernels = {k: [r for r in v if r in present] for k, v in kernels.items()}
    kernels = {k: v for k, v in kernels.items() if v}
    launches = {"mx_gemm": len(kernels.get("mx_gemm", [])), "nvfp4_gemm": 1, "fp8_blockwise_gemm": 1,
                "mx_quantize": 1 * ("q2" in present) + 3 * ("linq" in present), "nvfp4_quantize": 6,
                "ds_quantize": 2, "mxfp4_gemm": 1, "mxfp4_quantize": 2, "mx_gemm_blocks": 1,
                "pow2_block_quantize": 2, "mx_scales_from_fp32_blocks": 2, "mx_quantize_2d32": 1,
                "nvfp4_quantize_ex": 9, "nvfp4_quantize_2d": 3, "nvfp4_quantize_grouped": 3, "mx_gemm_grouped": 1,
                "nvfp4_gemm_grouped": 1, "fp8_blockwise_gemm_grouped": 1, "mx_gemm_mxout": 2,
                "mx_gemm_then_quantize": 2}
    dom = max(kernels, key=lambda k: sum(rows_ms[r] for r in kernels[k]))
    dom_ms = sum(rows_ms[r] for r in kernels[dom])
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            traffic = json.load(f).get(dom)
    tpk = tensor_peaks(peaks)
    gemm_flops = {"mx_gemm": len(kernels.get("mx_gemm", [])) * F_LIN, "nvfp4_gemm": F_NV, "fp8_blockwise_gemm": F_DS,
                  "mxfp4_gemm": F_MX4, "mx_gemm_blocks": F_DS, "mx_gemm_grouped": F_MOE, "nvfp4_gemm_grouped": F_MOE,
                  "fp8_blockwise_gemm_grouped": F_MOE, "mx_gemm_mxout": len(kernels.get("mx_gemm_mxout", [])) * F_LIN,
                  "mx_gemm_then_quantize": F_LIN}
    if dom in gemm_flops:
        flops = gemm_flops[dom]
        kind = "fp4" if dom in ("nvfp4_gemm", "mxfp4_gemm", "nvfp4_gemm_grouped") else "fp8"
        peak = tpk[kind]
        ach = flops / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 1), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / peak, 4), "traffic": traffic,
                "frac_nominal": round(ach / NOMINAL_TFLOPS[kind], 4), "peak_nominal": NOMINAL_TFLOPS[kind],
                "per_launch": {"flops": flops // launches[dom], "avg_ms": round(dom_ms / launches[dom], 4)},
                "peak_source": f"derived ({kind.upper()}): " + tpk["source"]}
        if ach > peak:
            roof["note"] = "achieved above the derived peak: the peak understates this GPU's rate at the clock seen"
    else:
        b = sum(rows[r]["bytes"] for r in kernels[dom])
        ach = b / (dom_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic,
                "per_launch": {"bytes": int(b // launches[dom]), "avg_ms": round(dom_ms / launches[dom], 4)},
                "peak_source": f"{peaks['source']} copy bandwidth"}
    roof["launches_per_step"] = launches[dom]

    # configuration of the 512^3 product: timed on its own (a latency-bound case, not in the step)
    latency = measure_mx512(dev, peaks) if not args.only else None

    # end to end through the public API with host buffers
    e2e = None
    h2d = sum(v.numel() * v.element_size() for v in wl.host.values())
    outs = wl.outputs()
    d2h = sum(o.numel() * o.element_size() for o in outs)
    if args.e2e_steps > 0:
        # Every step copies its inputs in from pinned host memory and its results out to pinned
        # host memory.  Two buffer sets and three streams let step i's results go out while step
        # i+1's inputs come in and step i+1 computes (the host link runs both directions at once).
        pinned_in = {k: v.pin_memory() for k, v in wl.host.items()}
        slots = [wl, Workload(dev, groups, host=wl.host)]
        for _ in range(2):
            slots[1].step()
        pinned_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in w.outputs()] for w in slots]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        started = [False, False]

        def e2e_step(i):
            k = i % 2
            w = slots[k]
            with torch.cuda.stream(s_in):
                if started[k]:
                    s_in.wait_event(comp_done[k])        # the slot's previous step has read its inputs
                for name, v in pinned_in.items():
                    w.d[name].copy_(v, non_blocking=True)
                in_done[k].record(s_in)
            stream.wait_event(in_done[k])
            if started[k]:
                stream.wait_event(out_done[k])           # the slot's previous results have left
            w.step()
            comp_done[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[k])
                for o, p in zip(w.outputs(), pinned_out[k]):
                    p.copy_(o, non_blocking=True)
                out_done[k].record(s_out)
            started[k] = True

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.e2e_steps):
            e2e_step(i)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, pg, dev)
        e2e = {"value": round(job_throughput(step_flops, world, e_ms) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e_ms, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "overlap": "inputs in, compute and results out on three streams over two buffer sets"}

    clocks = sampler.summary(t_wall0, t_wall2)
    value = job_throughput(step_flops, world, ms_step) / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8/fp4 inputs, f32 accumulate", "data": "synthetic",
        "config": dict(BASE_CONFIG, parallelism=f"replicas x{world}"),
    }
    line.update(headline(rows, rows_ms, present, peaks))
    line.update({"rows": rows, "roofline": roof, "gpu_launches": wl.launches_per_step * args.steps,
                 "clocks": clocks, "e2e": e2e})
    if latency is not None:
        line["latency"] = latency
    if cpu is not None:
        cpu.pop("seconds", None)
        line["cpu_baseline"] = cpu
    if args.only:
        line["config"]["only"] = args.only
        line["note"] = "profiling subset (--only): not a bench value"
    if rank == 0:
        print(json.dumps(line))
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
