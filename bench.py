#!/usr/bin/env python
"""Benchmark of the dynamic quantized int8 GEMM and QuantizeLinear on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl i8q|reference]

One step is one Forward of the dynamic quantized inner product on the large
workload (A bf16 8192 x 4096 quantized per row to uint8, constant int8 B
4096 x 14336 with per-column scales, exact int32 product, dequantization,
bias, GELU, bf16 C): the row quantization kernel and the GEMM kernel with
its fused epilogue.  `value` is algorithmic TOPS (2*M*N*K per step) over
all ranks.  The same run also times QuantizeLinear and DequantizeLinear on
the [32,1024,4096] fp32 round-trip workload (HBM GB/s).

Multi-GPU: one process per GPU (torchrun); every rank runs its own
replica (weak scaling, no data-path collective); the time is the max over
ranks.  --impl reference times the CPU oracle on a bounded sample of the
same workload on this host's cores (rank 0 only).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M, K, N = 8192, 4096, 14336
QDQ_SHAPE = (32, 1024, 4096)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD = ("dynamic quantized GEMM M=8192 K=4096 N=14336: bf16 A quantized per row to uint8, constant int8 B with "
            "per-column scales, int32 product, dequant + bias + GELU, bf16 C")


# DRAM bytes (read + written) per launch of the GEMM kernels, from one ncu
# capture of the headline step (dram__bytes_read.sum + dram__bytes_write.sum,
# a single-pass capture of the full-size launch).  Keyed by the SHA-256 of the
# kernel's sources: the figure is reported only while they are unchanged.
NCU_TRAFFIC = {
    "gemm_tc_pair": {"sources": ["int8_quantized_gb300/csrc/gemm_tc.cu", "int8_quantized_gb300/csrc/tcgen05.cuh",
                                 "int8_quantized_gb300/csrc/common.cuh"],
                     "sha256": "dfd3d191094acca86cbfde8c8c0d64895d9ba5f8879ad2f5720a3f09355167cf",
                     "bytes": (365.95 + 220.94) * 1e6,
                     "profile": "profiles/gemm_tc_pair_large_gemm.md"},
}


def ncu_traffic(kernel):
    """Bytes per launch from the committed capture, or None when the kernel
    has no capture or its sources changed since."""
    import hashlib
    e = NCU_TRAFFIC.get(kernel)
    if e is None:
        return None
    h = hashlib.sha256()
    try:
        for f in e["sources"]:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    return e["bytes"] if h.hexdigest() == e["sha256"] else None


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="i8q", choices=["i8q", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=2048, help="rows of the CPU-baseline sample")
    p.add_argument("--no-rows", action="store_true", help="skip the other hot-path workloads")
    p.add_argument("--rows", default=None,
                   help="comma-separated names of the hot-path workloads to time (default: all of them)")
    p.add_argument("--m", type=int, default=M,
                   help="rows of A in the GEMM step (default: the full workload; smaller for profiler captures)")
    p.add_argument("--detail", default=None,
                   help="also write the per-kernel split of every workload to this JSON file")
    return p.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value, world):
    """Max of a float over all ranks (the initialized process group)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def weak_scaling_value(ops_per_rank_step, steps, world, max_seconds):
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return ops_per_rank_step * steps * world / max_seconds


def pci_bus_id(dev):
    """'dddddddd:bb:dd.0' of a torch CUDA device, or None."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return "%08x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except AttributeError:
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs:
    NVML (read-only queries through ctypes) every 10 ms, else nvidia-smi
    every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of the NVML API
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, index, pci_bus_id=None):
        self.index = index
        self.pci = pci_bus_id
        self.proc = None
        self.file = None
        self.thread = None
        self.samples = []
        self.smax = None

    def _nvml_handle(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.pci:
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        try:
            reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def start(self):
        import ctypes
        import threading
        try:
            lib, h, reasons = self._nvml_handle()
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.smax = float(mx.value)
            self.stop_flag = threading.Event()

            def poll():
                clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self.stop_flag.is_set():
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                            reasons(h, ctypes.byref(rs)) == 0:
                        self.samples.append((float(clk.value), int(rs.value)))
                    self.stop_flag.wait(0.01)

            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            self.thread = None
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.pci or str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            if not self.samples:
                return None
            reasons = sorted(n for n, b in self.REASON_BITS.items() if any(r & b for _, r in self.samples))
            return {"sm_mhz": statistics.median(s for s, _ in self.samples),
                    "sm_max_mhz": self.smax or max(s for s, _ in self.samples), "reasons": reasons,
                    "samples": len(self.samples), "source": "nvml, 10 ms"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 200 ms"}


def time_loop(fn, steps, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3  # seconds


def cpu_baseline(rows, seed=2):
    """The oracle, as it stands, on `rows` rows of the large workload:
    row quantization, integer product and epilogue.  Returns (TOPS, threads,
    seconds, sample text)."""
    import numpy as np

    import oracle
    from int8_quantized_gb300 import workloads
    w = workloads.large_gemm(seed=seed, M=rows)
    oracle.lib()
    t0 = time.perf_counter()
    oracle.dynamic_quantized_inner_product(w["A_bf16"], iB=w["iB"], scaleB=w["scaleB"], bias=w["bias"],
                                           act=oracle.ACT_GELU, typeC="bf16")
    dt = time.perf_counter() - t0
    del np
    return (2.0 * rows * N * K / dt / 1e12, oracle.num_threads(), dt,
            f"{rows} of {M} rows of the large GEMM (row quantization, int32 product, dequant, bias, GELU, bf16); "
            f"TOPS = 2*rows*N*K / time")


def oracle_row_baselines(d=None):
    """The oracle, as it stands, on bounded samples of the other workloads
    (QuantizeLinear / DequantizeLinear, dense and depthwise QLinearConv, the
    LSTM, the small inner product whole): {row: {value, unit, sample,
    seconds}}, each a few seconds of host work at most."""
    import numpy as np

    import oracle
    from int8_quantized_gb300 import workloads
    out = {}

    def timed(f):
        t0 = time.perf_counter()
        r = f()
        return r, time.perf_counter() - t0

    d = workloads.qdq(seed=1) if d is None else d   # the round-trip workload, when the caller has it
    x = np.ascontiguousarray(d["x"][:8])
    y, dt = timed(lambda: oracle.quantize_linear(x, d["scale"], d["zero_point"], axis=2, ytype="u8"))
    out["quantize_linear"] = {"value": 5.0 * x.size / dt / 1e9, "unit": "GB/s", "seconds": round(dt, 3),
                              "sample": "8 of 32 rows of x [32,1024,4096], per-axis -> uint8"}
    _, dt = timed(lambda: oracle.dequantize_linear(y, d["scale"], d["zero_point"], axis=2))
    out["dequantize_linear"] = {"value": 5.0 * x.size / dt / 1e9, "unit": "GB/s", "seconds": round(dt, 3),
                                "sample": "8 of 32 rows, per-axis uint8 -> fp32"}
    del d, x, y
    for dw in (False, True):
        c = workloads.qlinearconv(seed=3, depthwise=dw)
        n = 1 if not dw else 32
        xs = np.ascontiguousarray(c["x"][:n])
        _, dt = timed(lambda: oracle.qlinearconv(xs, c["x_scale"], c["x_zero_point"], c["w"], c["w_scale"],
                                                 c["w_zero_point"], c["y_scale"], c["y_zero_point"], c["B"],
                                                 pads=c["pads"], group=c["group"]))
        ops = 2.0 * n * 256 * 56 * 56 * (c["w"].shape[1] * 9)
        out["qlinearconv_depthwise" if dw else "qlinearconv_dense"] = {
            "value": ops / dt / 1e12, "unit": "TOPS", "seconds": round(dt, 3),
            "sample": f"{n} of 32 images"}
    w = workloads.lstm(seed=4, T=2)
    _, dt = timed(lambda: oracle.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"],
                                                       direction="bidirectional"))
    ops = 2 * (2.0 * 2 * 64 * 1024 * 4096) * 2
    out["dq_lstm_bidirectional"] = {"value": ops / dt / 1e12, "unit": "TOPS", "seconds": round(dt, 3),
                                    "sample": "2 of 512 steps (projection and recurrence), both directions"}
    w = workloads.inner_product(seed=0)
    _, dt = timed(lambda: oracle.dynamic_quantized_inner_product(w["A"], w["B"], bias=w["bias"]))
    out["inner_product_64x128x256"] = {"value": dt * 1e6, "unit": "us", "seconds": round(dt, 4),
                                       "sample": "the whole 64x128x256 product (one Forward)"}
    return out


def _timed(fn, steps, warmup, stream):
    """Per-call seconds over `steps` calls after `warmup` (kernel timing off,
    so the timed calls run as they would in use), then one more call with
    the library's per-kernel event timing: {name: (launches, ms) per call}."""
    import torch

    import int8_quantized_gb300 as q
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    secs = time_loop(fn, steps, stream)
    q.profile_enable(True)
    fn()
    prof = q.profile_collect()
    q.profile_enable(False)
    q.sync_status()
    return secs / steps, {k: (v[0], v[1]) for k, v in prof.items()}


def measure_rows(args, dev, stream, world):
    """The other workloads of the hot path, each timed on its own (per
    call, device-resident inputs): algorithmic rate and per-kernel times."""
    import numpy as np
    import torch

    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads
    steps, warm = max(3, args.steps // 2), max(2, args.warmup)
    out = {}
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    sel = set(args.rows.split(",")) if getattr(args, "rows", None) else None
    want = lambda *keys: sel is None or any(k in sel for k in keys)  # noqa: E731
    if want("large_gemm_avoid_overflow"):
        _row_avoid_overflow(out, dev, stream, steps, warm, t)
    if want("inner_product_64x128x256"):
        _row_inner_product(out, dev, stream, steps, warm, t)
    for dw in (False, True):
        if want("qlinearconv_depthwise" if dw else "qlinearconv_dense"):
            _row_qlinearconv(out, dev, stream, steps, warm, t, dw)
    if want("qgemm_u8s8_to_u8", "matmul_integer_to_float", "dynamic_quantize_matmul"):
        _row_qgemm_family(out, dev, stream, steps, warm, t)
    if want("qlinear_add", "qlinear_leaky_relu"):
        _row_qlinear_ew(out, dev, stream, steps, warm)
    if want("dq_lstm_bidirectional"):
        _row_lstm(out, dev, stream, t)
    return out


def _row_avoid_overflow(out, dev, stream, steps, warm, t):
    import numpy as np
    import torch

    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads
    # large GEMM with avoidOverflow: non-constant fp32 B quantized in every Forward
    w = workloads.large_gemm(seed=2, avoid_overflow=True)
    ctx = q.QGemmDyn(M, N, K, q.BF16, q.F32, q.BF16, constB=False, bias=True, activation=q.ACT_GELU,
                     avoidOverflow=True)
    ctx.set_params(None, None, t(w["bias"]))
    A = t(w["A_bf16"].view(np.int16)).view(torch.bfloat16)
    B = t(w["B"])
    C = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    buf = torch.empty(ctx.external_buffer_size(), dtype=torch.uint8, device=dev)
    sec, prof = _timed(lambda: ctx.forward(A, C, B=B, buf=buf), steps, warm, stream)
    out["large_gemm_avoid_overflow"] = {"ms": sec * 1e3, "TOPS": 2.0 * M * N * K / sec / 1e12, "kernels": prof,
                                        "workload": "as the headline step, B fp32 [4096,14336] quantized to "
                                                    "[-64,63] inside each Forward"}
    ctx.clear()
    del A, B, C, buf


def _row_inner_product(out, dev, stream, steps, warm, t):
    import torch

    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads
    # small inner product (latency)
    w = workloads.inner_product(seed=0)
    ctx = q.QGemmDyn(64, 128, 256, q.F32, q.F32, q.F32, constB=True, bias=True)
    ctx.set_params(t(w["B"]), None, t(w["bias"]))
    A = t(w["A"])
    C = torch.empty(64, 128, device=dev)
    sec, prof = _timed(lambda: ctx.forward(A, C), steps * 10, warm, stream)
    out["inner_product_64x128x256"] = {"us": sec * 1e6, "kernels": prof}
    ctx.clear()


def _row_qlinearconv(out, dev, stream, steps, warm, t, dw):
    import torch

    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads
    # QLinearConv dense or depthwise
    c = workloads.qlinearconv(seed=3, depthwise=dw)
    x, wt = t(c["x"]), t(c["w"])
    ws, wz, bias = t(c["w_scale"]), t(c["w_zero_point"]), t(c["B"])
    y = torch.empty(32, 256, 56, 56, dtype=torch.uint8, device=dev)
    wsb = q.qlinearconv_workspace_size(c["x"].shape, c["w"].shape, c["pads"], (1, 1), (1, 1), c["group"])
    wsp = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    fn = lambda: q.qlinearconv(x, float(c["x_scale"]), c["x_zero_point"], wt, ws, wz,  # noqa: E731
                               float(c["y_scale"]), c["y_zero_point"], y, B=bias, pads=c["pads"],
                               group=c["group"], workspace=wsp if wsb else None)
    sec, prof = _timed(fn, steps, warm, stream)
    ops = 2.0 * 32 * 256 * 56 * 56 * (c["w"].shape[1] * 9)
    moved = c["x"].nbytes + c["w"].nbytes + y.numel()
    key = "qlinearconv_depthwise" if dw else "qlinearconv_dense"
    out[key] = {"ms": sec * 1e3, "TOPS": ops / sec / 1e12, "GB/s": moved / sec / 1e9, "kernels": prof,
                "workload": "x u8 [32,256,56,56], w [256,%d,3,3], pad 1, per-channel w" % c["w"].shape[1]}
    del x, wt, y, wsp


def _row_qgemm_family(out, dev, stream, steps, warm, t):
    import numpy as np
    import torch

    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads
    # QGemm at the large GEMM's shape: u8 A x s8 B with per-column
    # parameters, int32 C of shape (1, N), alpha, u8 output
    w = workloads.qgemm(seed=5)
    A, B = t(w["A"]), t(w["B"])
    bs, bz, Cb = t(w["b_scale"]), t(w["b_zero_point"]), t(w["C"])
    Y = torch.empty(M, N, dtype=torch.uint8, device=dev)
    wsp = torch.empty(q.qgemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    fn = lambda: q.qgemm(A, float(w["a_scale"]), w["a_zero_point"], B, bs, Y, b_zero_point=bz, C=Cb,  # noqa: E731
                         alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), y_zero_point=w["y_zero_point"],
                         workspace=wsp)
    sec, prof = _timed(fn, steps, warm, stream)
    out["qgemm_u8s8_to_u8"] = {"ms": sec * 1e3, "TOPS": 2.0 * M * N * K / sec / 1e12, "kernels": prof,
                               "workload": "QGemm M=8192 K=4096 N=14336, u8 A, s8 B per-column scale and zero point, "
                                           "C (1,N), alpha 1.5, u8 Y; both operands centred every call"}
    del Y, wsp

    # MatMulIntegerToFloat and DynamicQuantizeMatMul at the same shape, fp32 Y
    Yf = torch.empty(M, N, dtype=torch.float32, device=dev)
    wsp = torch.empty(q.matmul_integer_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    a_s = torch.tensor([float(w["a_scale"])], device=dev)
    a_z = torch.tensor([w["a_zero_point"]], dtype=torch.uint8, device=dev)
    bias = torch.from_numpy(workloads.large_gemm(seed=2, M=1, K=1, N=N)["bias"]).to(dev)
    fn = lambda: q.matmul_integer_to_float(A, B, a_s, bs, Yf, a_zero_point=a_z, b_zero_point=bz,  # noqa: E731
                                           bias=bias, workspace=wsp)
    sec, prof = _timed(fn, steps, warm, stream)
    out["matmul_integer_to_float"] = {"ms": sec * 1e3, "TOPS": 2.0 * M * N * K / sec / 1e12, "kernels": prof,
                                      "workload": "M=8192 K=4096 N=14336, u8 A per tensor, s8 B per column, bias, "
                                                  "fp32 Y"}
    del A
    Af = t((workloads.large_gemm(seed=2, M=M, K=K, N=1)["A_bf16"].astype(np.uint32) << 16).view(np.float32))
    fn = lambda: q.dynamic_quantize_matmul(Af, B, bs, Yf, b_zero_point=bz, bias=bias, workspace=wsp)  # noqa: E731
    sec, prof = _timed(fn, steps, warm, stream)
    out["dynamic_quantize_matmul"] = {"ms": sec * 1e3, "TOPS": 2.0 * M * N * K / sec / 1e12, "kernels": prof,
                                      "workload": "M=8192 K=4096 N=14336, fp32 A quantized per tensor, s8 B per "
                                                  "column, bias, fp32 Y"}
    del Af, B, Yf, wsp


def _row_qlinear_ew(out, dev, stream, steps, warm):
    import torch

    import int8_quantized_gb300 as q
    # QLinear elementwise on the [32,1024,4096] uint8 tensors: QLinearAdd of
    # two same-shape tensors (3 B per element), QLinearLeakyRelu (2 B)
    g = torch.Generator(device="cpu").manual_seed(6)
    Xa = torch.randint(0, 256, QDQ_SHAPE, generator=g, dtype=torch.uint8).to(dev)
    Xb = torch.randint(0, 256, QDQ_SHAPE, generator=g, dtype=torch.uint8).to(dev)
    Yq = torch.empty(QDQ_SHAPE, dtype=torch.uint8, device=dev)
    nel = Xa.numel()
    fn = lambda: q.qlinear_binary("add", Xa, 0.02, 128, Xb, 0.03, 120, 0.04, 125, Yq)  # noqa: E731
    sec, prof = _timed(fn, steps, warm, stream)
    hbm = load_peaks()[0].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out["qlinear_add"] = {"ms": sec * 1e3, "GB/s": 3.0 * nel / sec / 1e9, "frac_hbm": 3.0 * nel / sec / 1e9 / hbm,
                          "kernels": prof, "workload": "QLinearAdd u8 [32,1024,4096] + same shape, 3 B per element"}
    fn = lambda: q.qlinear_unary("leaky_relu", Xa, 0.02, 128, 0.015, 100, Yq, alpha=0.1)  # noqa: E731
    sec, prof = _timed(fn, steps, warm, stream)
    out["qlinear_leaky_relu"] = {"ms": sec * 1e3, "GB/s": 2.0 * nel / sec / 1e9,
                                 "frac_hbm": 2.0 * nel / sec / 1e9 / hbm, "kernels": prof,
                                 "workload": "QLinearLeakyRelu u8 [32,1024,4096], 2 B per element"}
    del Xa, Xb, Yq


def _row_lstm(out, dev, stream, t):
    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads
    import torch
    # DynamicQuantizeLSTM, bidirectional T=512 batch=64 I=H=1024
    w = workloads.lstm(seed=4)
    T_, b_, I_, H_ = 512, 64, 1024, 1024
    X, Wd, Rd = t(w["X"]), t(w["W"]), t(w["R"])
    Ws, Rs, Bb = t(w["W_scale"]), t(w["R_scale"]), t(w["B"])
    wsp = torch.empty(q.dq_lstm_workspace_size(T_, b_, I_, H_, q.LSTM_BIDIRECTIONAL), dtype=torch.uint8, device=dev)
    Y = torch.empty(T_, 2, b_, H_, device=dev)
    Yh = torch.empty(2, b_, H_, device=dev)
    Yc = torch.empty(2, b_, H_, device=dev)
    fn = lambda: q.dq_lstm_forward(X, Wd, Rd, Ws, Rs, wsp, direction=q.LSTM_BIDIRECTIONAL,  # noqa: E731
                                   B=Bb, Y=Y, Y_h=Yh, Y_c=Yc)
    sec, prof = _timed(fn, 2, 1, stream)
    ops = 2 * (2.0 * T_ * b_ * I_ * 4 * H_) + 2 * (2.0 * T_ * b_ * H_ * 4 * H_)
    out["dq_lstm_bidirectional"] = {"ms": sec * 1e3, "TOPS": ops / sec / 1e12, "kernels": prof,
                                    "workload": "T=512 batch=64 I=H=1024, projection + 512 steps per direction"}
    del X, Wd, Rd, wsp, Y


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    rows = max(8, min(args.cpu_rows // 4, 64))
    for _ in range(args.warmup):
        cpu_baseline(rows)
    times = []
    info = None
    for _ in range(args.steps):
        tops, threads, dt, sample = cpu_baseline(rows)
        times.append(dt)
        info = (threads, sample)
    total = sum(times)
    value = 2.0 * rows * N * K * args.steps / total / 1e12
    line = {"impl": "reference", "metric": "dyn-quant int8 GEMM TOPS & % INT8 tensor peak; QuantizeLinear HBM GB/s",
            "value": value, "unit": "TOPS", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8*s8->s32", "data": "synthetic",
            "config": {"workload": WORKLOAD + f"; sampled {rows} rows per step on the host CPU"},
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": info[0], "kind": "oracle", "sample": info[1]},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_i8q(args):
    import numpy as np
    import torch

    import int8_quantized_gb300 as q
    from int8_quantized_gb300 import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()

    # ---- large dynamic quantized GEMM -------------------------------------
    Mr = args.m
    w = workloads.large_gemm(seed=2 + rank, M=Mr)
    ctx = q.QGemmDyn(Mr, N, K, q.BF16, q.S8, q.BF16, constB=True, bias=True, activation=q.ACT_GELU)
    ctx.set_params(torch.from_numpy(w["iB"]).to(dev), torch.from_numpy(w["scaleB"]).to(dev),
                   torch.from_numpy(w["bias"]).to(dev))
    A = torch.from_numpy(w["A_bf16"].view(np.int16)).to(dev).view(torch.bfloat16)
    C = torch.empty(Mr, N, dtype=torch.bfloat16, device=dev)
    buf = torch.empty(ctx.external_buffer_size(), dtype=torch.uint8, device=dev)
    step = lambda: ctx.forward(A, C, buf=buf)  # noqa: E731
    for _ in range(args.warmup):
        step()
    q.sync_status()
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local, pci_bus_id(dev))
    clocks.start()
    q.profile_enable(True)
    secs = time_loop(step, args.steps, stream)
    prof = q.profile_collect()
    q.profile_enable(False)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    q.sync_status()
    max_secs = reduce_max(secs, world)
    ops = 2.0 * Mr * N * K
    value = weak_scaling_value(ops, args.steps, world, max_secs) / 1e12
    launches = sum(v[0] for v in prof.values())
    gemm_name = max((k for k in prof if k.startswith("gemm")), key=lambda k: prof[k][1])
    gemm_ms = prof[gemm_name][1] / prof[gemm_name][0]
    gemm_tops = ops / (gemm_ms * 1e-3) / 1e12
    int8_peak = q.measure_int8_mma_peak()
    if gemm_name == "gemm_imma":
        peak, peak_note = int8_peak, "int8 mma.sync peak measured in this run"
    else:
        # the kernel is timed alone in a loop of tens of milliseconds, not
        # seconds under the power cap: the burst bf16 rate is its peak
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        peak_note = f"bf16 dense burst ({peak_src})"

    # ---- end to end through the host-buffer entry point -------------------
    A_h = torch.from_numpy(w["A_bf16"].view(np.int16)).view(torch.bfloat16).pin_memory()
    C_h = torch.empty(Mr, N, dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        ctx.forward_host(A_h, C_h)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ctx.forward_host(A_h, C_h)
    e2e_secs = reduce_max(time.perf_counter() - t0, world)
    e2e = {"value": weak_scaling_value(ops, args.steps, world, e2e_secs) / 1e12, "unit": "TOPS",
           "h2d_bytes_per_step": A_h.numel() * 2, "d2h_bytes_per_step": C_h.numel() * 2}
    del A_h, C_h, buf, C, A
    ctx.clear()

    # ---- QuantizeLinear / DequantizeLinear round trip ---------------------
    d = workloads.qdq(seed=1)
    x = torch.from_numpy(d["x"]).to(dev)
    s = torch.from_numpy(d["scale"]).to(dev)
    z = torch.from_numpy(d["zero_point"]).to(dev)
    y = torch.empty(QDQ_SHAPE, dtype=torch.uint8, device=dev)
    xr = torch.empty(QDQ_SHAPE, dtype=torch.float32, device=dev)
    nel = x.numel()
    qstep = lambda: q.quantize_linear(x, s, z, y, axis=2)  # noqa: E731
    dstep = lambda: q.dequantize_linear(y, s, z, xr, axis=2)  # noqa: E731
    for _ in range(args.warmup):
        qstep()
        dstep()
    torch.cuda.synchronize()
    barrier(world)
    q_secs = reduce_max(time_loop(qstep, args.steps, stream), world)
    dq_secs = reduce_max(time_loop(dstep, args.steps, stream), world)
    # the per-tensor variant: int8 codes, scale 0.02, zero point 0
    s1 = torch.tensor([float(d["s8_scale"])], dtype=torch.float32, device=dev)
    z1 = torch.tensor([int(d["s8_zero_point"])], dtype=torch.int8, device=dev)
    y8 = torch.empty(QDQ_SHAPE, dtype=torch.int8, device=dev)
    q8step = lambda: q.quantize_linear(x, s1, z1, y8)  # noqa: E731
    d8step = lambda: q.dequantize_linear(y8, s1, z1, xr)  # noqa: E731
    for _ in range(args.warmup):
        q8step()
        d8step()
    torch.cuda.synchronize()
    barrier(world)
    q8_secs = reduce_max(time_loop(q8step, args.steps, stream), world)
    dq8_secs = reduce_max(time_loop(d8step, args.steps, stream), world)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    q_gbs = weak_scaling_value(5.0 * nel, args.steps, world, q_secs) / 1e9
    dq_gbs = weak_scaling_value(5.0 * nel, args.steps, world, dq_secs) / 1e9
    q8_gbs = weak_scaling_value(5.0 * nel, args.steps, world, q8_secs) / 1e9
    dq8_gbs = weak_scaling_value(5.0 * nel, args.steps, world, dq8_secs) / 1e9
    del x, y, xr, y8

    rows = {} if args.no_rows else measure_rows(args, dev, stream, world)

    cpu = None
    row_cpu = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tops, threads, dt, sample = cpu_baseline(args.cpu_rows)
        cpu = {"value": tops, "unit": "TOPS", "cores": threads, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2)}
        row_cpu = oracle_row_baselines(d)

    if rank == 0:
        def qdq_entry(gbs, secs, what):
            return {"value": round(gbs, 1), "unit": "GB/s", "ms": round(secs / args.steps * 1e3, 4),
                    "frac_hbm": round(gbs / world / hbm, 4), "frac_8tbs": round(gbs / world / 8000.0, 4),
                    "workload": what}

        def compact(r):
            e = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()
                 if k in ("ms", "us", "TOPS", "GB/s", "frac_hbm")}
            return e

        qdq = {"quantize_linear": qdq_entry(q_gbs, q_secs, "x fp32 [32,1024,4096] per-axis(2) -> uint8"),
               "dequantize_linear": qdq_entry(dq_gbs, dq_secs, "uint8 per-axis(2) -> fp32"),
               "quantize_linear_s8_per_tensor": qdq_entry(q8_gbs, q8_secs, "fp32 per-tensor 0.02 -> int8"),
               "dequantize_linear_s8_per_tensor": qdq_entry(dq8_gbs, dq8_secs, "int8 per-tensor -> fp32")}
        for k, v in row_cpu.items():
            if k in qdq:
                qdq[k]["oracle"] = {"value": round(v["value"], 3), "unit": v["unit"]}
        rows_c = {k: compact(v) for k, v in rows.items()}
        for k, v in row_cpu.items():
            if k in rows_c:
                rows_c[k]["oracle"] = {"value": round(v["value"], 5), "unit": v["unit"]}
        line = {
            "metric": "dyn-quant int8 GEMM TOPS & % INT8 tensor peak; QuantizeLinear HBM GB/s",
            "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": max_secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8*s8->s32", "data": "synthetic",
            "config": {"workload": WORKLOAD if Mr == M else WORKLOAD.replace("M=8192", f"M={Mr}"),
                       "M": Mr, "K": K, "N": N, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (A 67 MB + B 59 MB + C 235 MB per step)",
                       "kernel": gemm_name},
            "roofline": {"bound": "tensor", "achieved": gemm_tops, "peak": peak, "unit": "TFLOP/s",
                         "frac": gemm_tops / peak, "traffic": ncu_traffic(gemm_name), "peak_source": peak_note,
                         "kernel": gemm_name, "kernel_ms": gemm_ms},
            "int8_tensor_peak_tops": int8_peak,
            "pct_int8_tensor_peak": 100.0 * value / world / int8_peak,
            "pct_bf16_dense_peak": 100.0 * value / world / peaks.get("bf16_tflops", 1900.0),
            "rows": rows_c,
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk,
            "peaks_source": peak_src,
            # last, so that the end of the line carries the second half of the metric
            **qdq,
        }
        print(json.dumps(line), flush=True)
        if args.detail:
            with open(args.detail, "w") as f:
                json.dump({"kernels": {k: {"launches": v[0], "ms": v[1] / max(v[0], 1)} for k, v in prof.items()},
                           "rows": rows, "oracle_rows": row_cpu}, f, indent=1)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_i8q(args)


if __name__ == "__main__":
    sys.exit(main())
