#!/usr/bin/env python
"""Benchmark of the fused SwiGLU projection on GB300.

One step = the whole hot path over the Qwen-2.5-72B MLP workload
(K=8192, N=29568, M in {2048, 8192, 16384}), each M in both weight forms
(separate W1/W2 and interleaved W_fused): six fused-kernel launches.
Metric: TFLOP/s = sum(4*M*N*K) / time.  ``--workload`` selects the other
configurations (Qwen-2.5-0.5B and 7B, FP8, weight formats, the MLP block).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is device time of K back-to-back
replays of a CUDA graph of the step, inputs resident in HBM; each call reads
its own copy of the weights and its own A and writes its own Y, so every
step touches ~9.9 GB at 72B (~390 MB at 0.5B, 3x the 129 MB L2) and no call
finds its inputs in L2.
``e2e`` repeats the step through the public Python API with A copied in
from pinned host memory and Y copied back every step.  ``--impl reference``
times the CPU oracle (the deliberately slow reference arm) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "Fused SwiGLU-GEMM TFLOP/s (4·M·N·K/t) and % of GB300 BF16 roofline"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024

WORKLOADS = {
    # name: (K, N, Ms, seed)
    "qwen2.5-0.5b": (896, 4864, (128, 512, 2048, 8192), 1),
    "qwen2.5-0.5b-m64": (896, 4864, (64,), 0),
    "qwen2.5-7b": (3584, 18944, (256, 1024, 2048, 4096), 2),
    "qwen2.5-72b": (8192, 29568, (2048, 8192, 16384), 3),
    "qwen2.5-7b-fp8": (3584, 18944, (512, 4096), 4),
    # the FP8 projection fed by its producer (RMSNorm of the hidden state X and
    # per-tensor E4M3 quantisation of A), timed together
    "qwen2.5-7b-fp8-rmsnorm": (3584, 18944, (512, 4096), 4),
    # INT4 weights (group 128), BF16 A and Y
    "qwen2.5-0.5b-w4": (896, 4864, (64, 128, 512, 2048), 1),
    "qwen2.5-7b-w4": (3584, 18944, (128, 256, 1024), 2),
    # MXFP8 / NVFP4 weights (decoded to BF16 in the kernel), BF16 A and Y
    "qwen2.5-0.5b-mxfp8": (896, 4864, (64, 128, 512), 1),
    "qwen2.5-7b-mxfp8": (3584, 18944, (128, 256), 2),
    "qwen2.5-0.5b-nvfp4": (896, 4864, (64, 128, 512), 1),
    "qwen2.5-7b-nvfp4": (3584, 18944, (128, 256), 2),
    # the SwiGLU MLP block: (H, F, Ms, seed)
    "qwen2.5-0.5b-mlp": (896, 4864, (128, 512, 2048, 8192), 1),
    "qwen2.5-7b-mlp": (3584, 18944, (256, 1024, 4096), 2),
}
DEFAULT_WORKLOAD = "qwen2.5-72b"
RMS_EPS = 1e-6   # RMSNorm epsilon of the producer workload (Qwen-2.5's value)
W4_GROUP = 128   # K rows per INT4 scale group
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "swiglu_gemm_transformer_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ----------------------------------------------------------------------------- helpers

def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(files=None) -> str:
    """Hash of the kernel sources a capture was taken on: the named files of
    the CUDA source folder, or all of them."""
    h = hashlib.sha256()
    for f in sorted(files or os.listdir(CSRC)):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel_key: str):
    """Per-launch DRAM bytes from the committed ncu summary, or None when it is
    absent or was taken on different kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get(kernel_key)
    if not ent or ent.get("source_digest") != source_digest(ent.get("sources")):
        return None
    return ent.get("dram_bytes_per_launch")


# Kernel sources a traffic record depends on, by kernel family.
TRAFFIC_SOURCES = {
    "pair": ["sm103_ptx.cuh", "tc_common.cuh", "swiglu_tc2_kernel.cuh", "swiglu_tc_kernel.cuh",
             "launch_tc.cuh", "launch.h", "k_bf16_separate.cu", "k_bf16_interleaved.cu",
             "swiglu_api.cu"],
    "sk": ["k_bf16_sk.cu", "launch.h", "sm103_ptx.cuh", "swiglu_api.cu", "swiglu_sk_kernel.cuh",
           "tc_common.cuh", "weight_decode.cuh"],
}


def record_traffic(csv_path: str, kernel_key: str, family: str, capture: str):
    """Write one traffic record from an ncu CSV of dram__bytes_read.sum and
    dram__bytes_write.sum (one captured launch), stamped with the digest of
    the current kernel sources.  Run right after the capture, on the sources
    it was taken on."""
    import csv
    vals = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f)]
    hdr = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    for r in rows[hdr + 1:]:
        d = dict(zip(rows[hdr], r))
        if d.get("Metric Name") in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[d["Metric Unit"]]
            vals[d["Metric Name"]] = int(round(float(d["Metric Value"].replace(",", "")) * scale))
    rd, wr = vals["dram__bytes_read.sum"], vals["dram__bytes_write.sum"]
    try:
        with open(TRAFFIC_FILE) as f:
            table = json.load(f)
    except FileNotFoundError:
        table = {}
    srcs = TRAFFIC_SOURCES[family]
    table[kernel_key] = {"dram_bytes_per_launch": rd + wr, "dram_read_bytes": rd,
                         "dram_write_bytes": wr, "sources": srcs,
                         "source_digest": source_digest(srcs), "capture": capture}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(table, f, indent=2)
        f.write("\n")
    return table[kernel_key]


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception as e:  # no nvidia-smi: report what we have
            log(f"clock sampling unavailable: {e}")
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        smax = max(r[1] for r in rows)
        pmax = max(r[2] for r in rows)
        # samples "under load": power above half the run's maximum
        loaded = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": pmax}


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The timed region's duration as the job sees it: the slowest rank's."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step_per_rank: float, steps: int, ms_max: float, ws: int) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return ws * flops_per_step_per_rank * steps / (ms_max * 1e-3) / 1e12


def roofline_entry(flops: float, nbytes: float, us: float, peak_tflops: float, peak_gbs: float) -> dict:
    """Bound (tensor or HBM) of one launch and the fraction of it achieved."""
    t_tc = flops / (peak_tflops * 1e12)
    t_hbm = nbytes / (peak_gbs * 1e9)
    bound = "tensor" if t_tc >= t_hbm else "hbm"
    return {"bound": bound,
            "tflops": flops / (us * 1e-6) / 1e12,
            "gbs": nbytes / (us * 1e-6) / 1e9,
            "frac_of_roofline": max(t_tc, t_hbm) / (us * 1e-6)}


def describe_workload(name: str) -> str:
    """The config.workload text of a workload, the same for both arms."""
    K, N, Ms, seed = WORKLOADS[name]
    if name.endswith("-mlp"):
        return (f"{name} SwiGLU MLP block H={K} F={N} M={list(Ms)} "
                f"(fused gate/up projection + down projection), seed {seed}")
    if name.endswith("-fp8-rmsnorm"):
        return (f"{name} FP8 projection K={K} N={N} M={list(Ms)} fed by its producer (RMSNorm "
                f"of X, eps {RMS_EPS}, per-tensor E4M3 quantisation), separate and interleaved "
                f"weights, seed {seed}")
    if name.endswith("-w4"):
        return (f"{name} MLP projection K={K} N={N} M={list(Ms)} with INT4 weights (group "
                f"{W4_GROUP}, BF16 scales) as [K, N/2] codes and K-major, BF16 A and Y, seed {seed}")
    if name.endswith(("-mxfp8", "-nvfp4")):
        fmt = name.rsplit("-", 1)[1]
        codes = "[K, N]" if fmt == "mxfp8" else "[K, N/2]"
        return (f"{name} MLP projection K={K} N={N} M={list(Ms)} with {fmt.upper()} weights as "
                f"{codes} codes and K-major, BF16 A and Y, seed {seed}")
    return (f"{name} MLP projection K={K} N={N} M={list(Ms)}, separate and interleaved weights, "
            f"seed {seed}")


# ----------------------------------------------------------------------------- our arm

class Workload:
    """Device-resident inputs and the list of calls of one step.

    kinds: "bf16" (fused projection, separate and interleaved weights),
    "fp8" (the same with E4M3 operands), "mlp" (the SwiGLU MLP block, fused
    projection followed by the down projection)."""

    def __init__(self, name, dev, variant=0, only=None):
        import torch
        import swiglu_gemm_transformer_gb300 as sg
        import swiglu_inputs as si
        self.sg = sg
        self.lib = sg.lib()
        self.name = name
        K, N, Ms, seed = WORKLOADS[name]
        self.K, self.N, self.Ms, self.seed = K, N, Ms, seed
        self.dev = dev
        self.producer = name.endswith("-fp8-rmsnorm")
        self.kind = ("fp8" if name.endswith("-fp8") or self.producer else
                     "mlp" if name.endswith("-mlp") else "w4" if name.endswith("-w4") else
                     "mx" if name.endswith(("-mxfp8", "-nvfp4")) else "bf16")
        self.mxfmt = name.rsplit("-", 1)[1] if self.kind == "mx" else None
        self.fp8 = self.kind == "fp8"
        self.eb = 1 if self.fp8 else 2
        # INT4, MXFP8 and NVFP4: the codes as [K, N], and K-major, decoded into
        # tensor memory (packed once at set-up, like a model load)
        forms = (("mlp",) if self.kind == "mlp" else ("separate", "kmajor") if self.kind in ("w4", "mx")
                 else ("separate", "interleaved"))
        self.host = {}
        for M in Ms:
            if self.producer:   # X and gamma in BF16; the FP8 weights of the same recipe
                q, sc = si.make_e4m3(1, N, K, seed)
                X, gamma = si.make_producer_inputs(M, K, seed)
                self.host[M] = (X, q[1].t().contiguous(), q[2].t().contiguous(), sc, gamma)
            elif self.fp8:
                q, sc = si.make_e4m3(M, N, K, seed)
                self.host[M] = (q[0], q[1].t().contiguous(), q[2].t().contiguous(), sc)
            elif self.kind == "w4":
                A, (W1q, S1), (W2q, S2) = si.make_w4(M, N, K, seed, W4_GROUP)
                self.host[M] = (A, W1q, S1, W2q, S2)
            elif self.kind == "mx":
                A, w1, w2 = si.make_mx(M, N, K, seed, self.mxfmt)
                if self.mxfmt == "mxfp8":
                    self.host[M] = (A, w1[0], w1[1], w2[0], w2[1])
                else:
                    f32 = lambda v: torch.tensor([v], dtype=torch.float32)
                    self.host[M] = (A, w1[0], w1[1], f32(w1[2]), w2[0], w2[1], f32(w2[2]))
            elif self.kind == "mlp":   # K = H (hidden), N = F (intermediate)
                A, W1, W2 = si.make_bf16(M, N, K, seed)
                self.host[M] = (A, W1, W2, si.make_bf16(1, K, N, seed + 100)[1])
            else:
                self.host[M] = si.make_bf16(M, N, K, seed)
        self.calls, self.buffers, self.fns = [], [], []
        self.bytes_touched = 0
        self.flops = 0
        for form in forms:
            for M in Ms:
                if only is not None and (form, M) not in only:
                    continue
                v = variant or (self.lib.swiglu_select_variant(M, N, K, int(form == "interleaved"))
                                if self.kind == "bf16" else -1)
                bufs = self._device_buffers(form, M)
                self.calls.append((form, M, v))
                self.buffers.append(bufs)
                self.fns.append(self.launcher(form, M, v, bufs))
                self.bytes_touched += self.algorithmic_bytes(M)
                self.flops += self.flops_of(M)
        torch.cuda.synchronize(dev)

    # -- per-call quantities
    def flops_of(self, M):
        return (6 if self.kind == "mlp" else 4) * M * self.N * self.K

    def algorithmic_bytes(self, M):
        """Inputs read once and the output written once (the MLP's Y is internal;
        with the producer, A's codes are written once and read once more)."""
        if self.kind == "mlp":
            return 2 * (M * self.K + 3 * self.K * self.N + M * self.K)
        if self.kind == "w4":   # A, two code matrices, two scale matrices, Y
            return (2 * M * self.K + 2 * (self.K * self.N // 2)
                    + 2 * (self.K // W4_GROUP) * self.N * 2 + 2 * M * self.N)
        if self.kind == "mx":
            if self.mxfmt == "mxfp8":   # one byte per code, one per 32 codes of a column
                w = 2 * (self.K * self.N + (self.K // 32) * self.N)
            else:                       # half a byte per code, one per 16, two tensor scales
                w = 2 * (self.K * self.N // 2 + (self.K // 16) * self.N) + 8
            return 2 * M * self.K + w + 2 * M * self.N
        b = self.eb * (M * self.K + 2 * self.K * self.N) + M * self.N * 2
        if self.producer:
            b += self.producer_bytes(M)
        return b

    def producer_bytes(self, M):
        """RMSNorm + quantisation: X read (BF16), gamma read, codes written."""
        return 2 * M * self.K + 2 * self.K + M * self.K

    def out_shape(self, M):
        return (M, self.K) if self.kind == "mlp" else (M, self.N)

    # -- buffers and launches
    def _device_buffers(self, form, M):
        import torch
        dev, sg = self.dev, self.sg
        h = self.host[M]
        out = torch.empty(self.out_shape(M), dtype=torch.bfloat16, device=dev)
        if self.kind == "w4" and form == "kmajor":   # (A, W1k, S1, W2k, S2, Y)
            return (h[0].to(dev), sg.swiglu_pack_w4_kmajor(h[1].to(dev)), h[2].to(dev),
                    sg.swiglu_pack_w4_kmajor(h[3].to(dev)), h[4].to(dev), out)
        if self.mxfmt == "mxfp8" and form == "kmajor":   # (A, C1k, S1, C2k, S2, Y)
            return (h[0].to(dev), h[1].t().contiguous().to(dev), h[2].to(dev),
                    h[3].t().contiguous().to(dev), h[4].to(dev), out)
        if self.kind == "mx" and form == "kmajor":   # (A, C1k, S1, g1, C2k, S2, g2, Y)
            return (h[0].to(dev), sg.swiglu_pack_w4_kmajor(h[1].to(dev)), h[2].to(dev), h[3].to(dev),
                    sg.swiglu_pack_w4_kmajor(h[4].to(dev)), h[5].to(dev), h[6].to(dev), out)
        if self.kind in ("w4", "mx"):
            return tuple(t.to(dev) for t in h) + (out,)
        if self.kind == "mlp":
            ws = torch.empty(int(self.lib.swiglu_mlp_workspace_size(M, self.K, self.N)),
                             dtype=torch.uint8, device=dev)
            return (h[0].to(dev), h[1].to(dev), h[2].to(dev), h[3].to(dev), out, ws)
        if self.fp8:
            s = torch.tensor(list(h[3]), dtype=torch.float32, device=dev)
            extra = ()
            if self.producer:   # (X, gamma, Aq): the producer writes Aq and s[0]
                extra = (h[4].to(dev), torch.empty(M, self.K, dtype=torch.float8_e4m3fn, device=dev))
            if form == "separate":
                return (h[0].to(dev), h[1].to(dev), h[2].to(dev), out, s) + extra
            return (h[0].to(dev), sg.swiglu_pack_interleaved_fp8(h[1].to(dev), h[2].to(dev)), out,
                    s) + extra
        if form == "separate":
            return (h[0].to(dev), h[1].to(dev), h[2].to(dev), out)
        return (h[0].to(dev), sg.swiglu_pack_interleaved(h[1].to(dev), h[2].to(dev)), out)

    def _stream(self):
        import torch
        return torch.cuda.current_stream().cuda_stream

    def launcher(self, form, M, v, bufs, with_producer=True):
        """A closure launching this call through the C ABI on the current stream."""
        lib, N, K, sg = self.lib, self.N, self.K, self.sg
        d = [b.data_ptr() for b in bufs]

        def check(name, rc):
            if rc:
                raise sg.SwigluError(name, rc)
        if self.kind == "w4" and form == "kmajor":
            return lambda: check("swiglu_fused_w4_kmajor", lib.swiglu_fused_w4_kmajor(
                d[0], d[1], d[2], d[3], d[4], d[5], M, N, K, W4_GROUP, self._stream()))
        if self.kind == "w4":
            return lambda: check("swiglu_fused_w4", lib.swiglu_fused_w4(
                d[0], d[1], d[2], d[3], d[4], d[5], M, N, K, W4_GROUP, self._stream()))
        if self.mxfmt == "mxfp8" and form == "kmajor":
            return lambda: check("swiglu_fused_mxfp8_kmajor", lib.swiglu_fused_mxfp8_kmajor(
                d[0], d[1], d[2], d[3], d[4], d[5], M, N, K, self._stream()))
        if self.kind == "mx" and self.mxfmt == "mxfp8":
            return lambda: check("swiglu_fused_mxfp8", lib.swiglu_fused_mxfp8(
                d[0], d[1], d[2], d[3], d[4], d[5], M, N, K, self._stream()))
        if self.kind == "mx" and form == "kmajor":
            return lambda: check("swiglu_fused_nvfp4_kmajor", lib.swiglu_fused_nvfp4_kmajor(
                d[0], d[1], d[2], d[3], d[4], d[5], d[6], d[7], M, N, K, self._stream()))
        if self.kind == "mx":
            return lambda: check("swiglu_fused_nvfp4", lib.swiglu_fused_nvfp4(
                d[0], d[1], d[2], d[3], d[4], d[5], d[6], d[7], M, N, K, self._stream()))
        if self.kind == "mlp":
            nbytes = bufs[5].numel()
            return lambda: check("swiglu_mlp", lib.swiglu_mlp(d[0], d[1], d[2], d[3], None, d[4],
                                                               M, K, N, d[5], nbytes, self._stream()))
        if self.fp8:
            ns = 4 if form == "separate" else 3        # index of the scales
            sp = (d[ns], d[ns] + 4, d[ns] + 8)
            a = d[0]
            prod = None
            if self.producer:
                a = d[ns + 2]                          # the codes the producer writes
                if with_producer:
                    prod = self.producer_launcher(form, M, v, bufs)
            if form == "separate":
                f = lambda: check("swiglu_fused_fp8", lib.swiglu_fused_fp8(
                    a, d[1], d[2], sp[0], sp[1], sp[2], d[3], M, N, K, self._stream()))
            else:
                f = lambda: check("swiglu_fused_interleaved_fp8", lib.swiglu_fused_interleaved_fp8(
                    a, d[1], sp[0], sp[1], sp[2], d[2], M, N, K, self._stream()))
            if prod is None:
                return f
            return lambda: (prod(), f())
        if form == "separate":
            return lambda: check("swiglu_fused_ex", lib.swiglu_fused_ex(
                d[0], d[1], d[2], d[3], M, N, K, v, self._stream()))
        return lambda: check("swiglu_fused_interleaved_ex", lib.swiglu_fused_interleaved_ex(
            d[0], d[1], d[2], M, N, K, v, self._stream()))

    def gemm_launcher(self, form, M, v, bufs):
        """The FP8 projection alone, on the codes the producer left in the buffers."""
        return self.launcher(form, M, v, bufs, with_producer=False)

    def producer_launcher(self, form, M, v, bufs):
        """The producer alone: RMSNorm of X and E4M3 quantisation into Aq, s[0]."""
        lib, K, sg = self.lib, self.K, self.sg
        ns = 4 if form == "separate" else 3
        X, s, gamma, Aq = bufs[0], bufs[ns], bufs[ns + 1], bufs[ns + 2]
        px, pg, pq, ps = X.data_ptr(), gamma.data_ptr(), Aq.data_ptr(), s.data_ptr()

        def run():
            rc = lib.swiglu_rmsnorm_quant_fp8(px, pg, RMS_EPS, pq, ps, M, K, self._stream())
            if rc:
                raise sg.SwigluError("swiglu_rmsnorm_quant_fp8", rc)
        return run

    def api_call(self, form, M, v, bufs):
        """The same call through the public Python API; returns the output tensor."""
        sg = self.sg
        if self.kind == "w4" and form == "kmajor":
            return sg.swiglu_fused_w4_kmajor(*bufs[:5], bufs[5], group=W4_GROUP)
        if self.kind == "w4":
            return sg.swiglu_fused_w4(*bufs[:5], bufs[5], group=W4_GROUP)
        if self.mxfmt == "mxfp8" and form == "kmajor":
            return sg.swiglu_fused_mxfp8_kmajor(*bufs[:5], bufs[5])
        if self.kind == "mx" and self.mxfmt == "mxfp8":
            return sg.swiglu_fused_mxfp8(*bufs[:5], bufs[5])
        if self.kind == "mx" and form == "kmajor":
            return sg.swiglu_fused_nvfp4_kmajor(*bufs[:7], bufs[7])
        if self.kind == "mx":
            return sg.swiglu_fused_nvfp4(*bufs[:7], bufs[7])
        if self.kind == "mlp":
            return sg.swiglu_mlp(bufs[0], bufs[1], bufs[2], bufs[3], None, bufs[4], workspace=bufs[5])
        if self.fp8:
            ns = 4 if form == "separate" else 3
            sc = bufs[ns]
            s3 = (sc[0:1], sc[1:2], sc[2:3])
            a = bufs[0]
            if self.producer:
                a, _ = sg.swiglu_rmsnorm_quant_fp8(bufs[0], bufs[ns + 1], RMS_EPS, bufs[ns + 2], s3[0])
            if form == "separate":
                return sg.swiglu_fused_fp8(a, bufs[1], bufs[2], *s3, bufs[3])
            return sg.swiglu_fused_interleaved_fp8(a, bufs[1], *s3, bufs[2])
        if form == "separate":
            return sg.swiglu_fused(bufs[0], bufs[1], bufs[2], bufs[3], variant=v)
        return sg.swiglu_fused_interleaved(bufs[0], bufs[1], bufs[2], variant=v)

    def launches_per_call(self, M):
        """Kernels one call enqueues (the MLP: fused projection, down projection,
        and the split-K reduction when the down projection splits K)."""
        if self.producer:
            return 3   # amax pass, quantise pass, FP8 projection
        if self.kind != "mlp":
            return 1
        return 2 + (1 if self.lib.swiglu_linear_workspace_size(M, self.K, self.N) > 0 else 0)

    def variant_label(self, v, M, form="separate"):
        if self.kind == "mlp":
            return "mlp"
        if self.producer:
            return "rmsnorm_quant+2sm_fp8"
        if form == "kmajor":
            return ("w4" if self.kind == "w4" else self.mxfmt) + "_kmajor_tmem"
        if self.kind in ("w4", "mx"):   # the library's choice of kernel
            fmt = "w4" if self.kind == "w4" else self.mxfmt
            return f"{fmt}_{self.sg.WEIGHT_KERNELS[self.sg.swiglu_select_weight_kernel(M, self.N)]}"
        return "2sm_fp8" if self.fp8 else self.sg.variant_name(v)

    def step(self):
        for fn in self.fns:
            fn()


def measure_calls(wl, stream, launches, factory=None, pairs=None):
    """Average duration (us) of each call of the step, launched alone and back
    to back inside a CUDA graph, rotating over copies of its inputs so that
    the copies together exceed 2.5x the L2 size.  ``factory(form, M, v, bufs)``
    builds the launch closure (default: the fused call through the C ABI);
    ``pairs`` ((form, M, v), bufs) defaults to every call of the step."""
    import torch
    factory = factory or wl.launcher
    out = []
    for (form, M, v), bufs in (pairs or list(zip(wl.calls, wl.buffers))):
        per = wl.algorithmic_bytes(M)
        ncopy = max(2, min(24, math.ceil(2.5 * L2_BYTES / per)))
        copies = [bufs] + [tuple(t.clone() for t in bufs) for _ in range(ncopy - 1)]
        fns = [factory(form, M, v, cb) for cb in copies]
        reps = max(1, math.ceil(launches / ncopy))

        def body():
            for _ in range(reps):
                for f in fns:
                    f()
        with torch.cuda.stream(stream):
            for f in fns:       # first calls outside the capture (module loads, compilation)
                f()
            g = capture(body, stream)
            g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
        e1.synchronize()
        out.append(1e3 * e0.elapsed_time(e1) / (reps * ncopy))
        del g, copies, fns
    torch.cuda.empty_cache()
    return out


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist
    import swiglu_gemm_transformer_gb300 as sg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sg.lib()
    only = None
    if args.only:
        only = {(f, int(m)) for f, m in (x.split(":") for x in args.only.split(","))}
    wl = Workload(args.workload, dev, variant=sg.VARIANTS[args.variant], only=only)
    if not wl.calls:
        raise SystemExit(f"no calls selected from workload {args.workload}")
    stream = torch.cuda.Stream(device=dev)
    n_calls = len(wl.calls)

    with torch.cuda.stream(stream):
        for _ in range(2):          # load modules, set function attributes, before capture
            wl.step()
        stream.synchronize()
        rc, detail = sg.swiglu_device_status(stream)
        if rc != sg.OK:
            raise RuntimeError(f"device status after warm-up: {sg.status_string(rc)} ({detail})")
        g_step = capture(wl.step, stream)
        for _ in range(args.warmup):
            g_step.replay()
        stream.synchronize()

    sampler = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)  # let the sampler take a baseline sample
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record()
        for _ in range(args.steps):
            g_step.replay()
        t_end.record()
    t_end.synchronize()
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    clocks = sampler.stop()
    rc, detail = sg.swiglu_device_status(stream)
    if rc != sg.OK:
        raise RuntimeError(f"device status after timing: {sg.status_string(rc)} ({detail})")

    # The end-to-end figure next, under the same conditions as the timed
    # region (before the per-call measurements below heat the GPU further).
    e2e = None if args.no_e2e else run_e2e(args, wl, stream, ws)

    # Per-call launch durations: each call alone, launched back to back on
    # rotating copies of its inputs (enough copies to exceed 2.5x L2), in a graph.
    per_call_us = measure_calls(wl, stream, args.call_launches)

    t_max = max_over_ranks(ms_total, ws, dev)
    ms_per_step = t_max / args.steps
    value = job_tflops(wl.flops, args.steps, t_max, ws)

    peaks, peak_src = load_peaks()
    sustained = t_max > 1000.0
    peak_tf = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    if wl.fp8:
        peak_tf *= 2.0  # dense FP8 = 2x dense BF16 (nominal 4.5 vs 2.25 PFLOP/s)
    kernels = []
    chain = None
    if wl.producer:
        # the two kernels of each call timed alone: the FP8 projection (on the
        # codes the producer wrote during warm-up) and the producer
        gemm_us = measure_calls(wl, stream, args.call_launches, wl.gemm_launcher)
        prod_us = measure_calls(wl, stream, args.call_launches, wl.producer_launcher)
        chain = [{"form": f, "M": M, "us": round(per_call_us[c], 3),
                  "tflops": round(wl.flops_of(M) / (per_call_us[c] * 1e-6) / 1e12, 1)}
                 for c, (f, M, v) in enumerate(wl.calls)]
    for c, (form, M, v) in enumerate(wl.calls):
        us = gemm_us[c] if wl.producer else per_call_us[c]
        flops = wl.flops_of(M)
        abytes = wl.algorithmic_bytes(M) - (wl.producer_bytes(M) if wl.producer else 0)
        r = roofline_entry(flops, abytes, us, peak_tf, peaks["hbm_gbs"])
        bound, achieved_tf, achieved_gbs = r["bound"], r["tflops"], r["gbs"]
        kernels.append({
            "form": form, "M": M, "variant": "2sm_fp8" if wl.producer else wl.variant_label(v, M, form),
            "us": round(us, 3),
            "tflops": round(achieved_tf, 1), "gbs": round(achieved_gbs, 1), "bound": bound,
            "frac_of_roofline": round(r["frac_of_roofline"], 4),
            "share": 0.0,
        })
        if wl.producer:
            pb = wl.producer_bytes(M)
            gbs = pb / (prod_us[c] * 1e-6) / 1e9
            kernels.append({
                "form": form, "M": M, "variant": "rmsnorm_quant", "us": round(prod_us[c], 3),
                "tflops": 0.0, "gbs": round(gbs, 1), "bound": "hbm",
                "frac_of_roofline": round(gbs / peaks["hbm_gbs"], 4), "share": 0.0,
            })
    tot_us = sum(k["us"] for k in kernels)
    for k in kernels:
        k["share"] = round(k["us"] / tot_us, 4)
    dom = max(range(len(kernels)), key=lambda i: kernels[i]["us"])
    dk = kernels[dom]
    form, M = dk["form"], dk["M"]
    kernel_key = f"{wl.name}:{form}:M{M}:{dk['variant']}"
    if dk["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dk["tflops"], "peak": peak_tf, "unit": "TFLOP/s",
                "frac": round(dk["tflops"] / peak_tf, 4)}
    else:
        roof = {"bound": "hbm", "achieved": dk["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(dk["gbs"] / peaks["hbm_gbs"], 4)}
    roof["traffic"] = load_traffic(kernel_key)
    roof["traffic_note"] = ("dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu "
                            "capture of this kernel on the current sources (null otherwise); "
                            "output bytes still dirty in L2 when the kernel ends are not yet "
                            "written to DRAM and are not counted, so traffic can fall below the "
                            "algorithmic bytes")
    roof["kernel"] = kernel_key
    roof["algorithmic_per_launch"] = (wl.flops_of(M) if dk["bound"] == "tensor"
                                      else wl.producer_bytes(M) if dk["variant"] == "rmsnorm_quant"
                                      else wl.algorithmic_bytes(M))
    roof["peak_source"] = (f"{peak_src} ({'sustained' if sustained and dk['bound'] == 'tensor' else 'burst'})"
                           + (", x2 for FP8" if wl.fp8 and dk["bound"] == "tensor" else ""))

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8e4m3" if wl.fp8 else "bf16",
        "data": "synthetic",
        "impl": "ours",
        "config": {
            "workload": describe_workload(wl.name),
            "calls_per_step": n_calls,
            "l2": f"inputs larger than L2: each call has its own A, weights and Y; "
                  f"{wl.bytes_touched / 2**20:.0f} MiB per step vs {L2_BYTES / 2**20:.0f} MiB L2",
            "timing": "CUDA graph of one step replayed back to back, CUDA events around the "
                      "timed region, max over ranks; per-call durations from graphs of "
                      "back-to-back launches of that call on rotating input copies",
            "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
        },
        "gpu_launches": sum(wl.launches_per_call(M) for (_, M, _) in wl.calls) * args.steps,
        "roofline": roof,
        "clocks": clocks,
        "kernels": kernels,
        "timing_check": {"sum_of_call_ms": round(sum(per_call_us) / 1e3, 5)},
        "e2e": e2e,
        "calls": chain,
    }
    return out, wl, stream


def run_e2e(args, wl, stream, ws):
    """Same step through the public API: A in from pinned host memory, Y out to it.

    The copies and the kernels are pipelined over three streams (host-to-device,
    compute, device-to-host) ordered by events, as a serving loop would: call i's
    input copy overlaps call i-1's kernel, and its output copy overlaps call i+1's."""
    import torch
    import swiglu_gemm_transformer_gb300 as sg
    dev = wl.dev
    host_a, host_y = [], []
    h2d = d2h = 0
    for (form, M, v), bufs in zip(wl.calls, wl.buffers):
        A_host = wl.host[M][0].pin_memory()
        Y_host = torch.empty(wl.out_shape(M), dtype=torch.bfloat16).pin_memory()
        host_a.append(A_host)
        host_y.append(Y_host)
        h2d += A_host.numel() * A_host.element_size()
        d2h += Y_host.numel() * 2
    n = len(wl.calls)
    s_in, s_cmp, s_out = torch.cuda.Stream(device=dev), stream, torch.cuda.Stream(device=dev)
    a_ready = [torch.cuda.Event() for _ in range(n)]
    a_free = [torch.cuda.Event() for _ in range(n)]
    y_ready = [torch.cuda.Event() for _ in range(n)]
    y_free = [torch.cuda.Event() for _ in range(n)]

    def step():
        for i, ((form, M, v), bufs) in enumerate(zip(wl.calls, wl.buffers)):
            Ad = bufs[0]
            with torch.cuda.stream(s_in):
                s_in.wait_event(a_free[i])          # the previous step's kernel has read A
                Ad.copy_(host_a[i], non_blocking=True)
                a_ready[i].record()
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(a_ready[i])
                s_cmp.wait_event(y_free[i])         # the previous step's Y has been copied out
                Y = wl.api_call(form, M, v, bufs)
                a_free[i].record()
                y_ready[i].record()
            with torch.cuda.stream(s_out):
                s_out.wait_event(y_ready[i])
                host_y[i].copy_(Y, non_blocking=True)
                y_free[i].record()

    steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(steps):
        step()
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    e1.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    val = job_tflops(wl.flops, steps, ms, ws)
    return {"value": round(val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "weights resident in HBM; each step copies every call's A in and Y out "
                    "(pinned host memory), copies and kernels pipelined over three streams"}


def unfused_fn(wl):
    """The unfused computation of one call in plain torch: the gate and up
    products as two cuBLAS GEMMs on the separate weights, then SiLU and the
    product as separate kernels.  It is the common baseline of both fused
    forms (one GEMM on W_fused followed by strided SiLU and product slices is
    slower than the two GEMMs, so it would flatter the interleaved form)."""
    import torch.nn.functional as F
    if wl.kind == "mlp":
        return lambda A, W1, W2, W3: (F.silu(A @ W1) * (A @ W2)) @ W3
    return lambda A, W1, W2: F.silu(A @ W1) * (A @ W2)


def unfused_factory(wl, compiled=False):
    """Launch-closure factory for measure_calls running the unfused path
    (eager, or the torch.compile'd version of the same function) on the
    separate-form buffers of a call.  The result goes to a tensor the graph's
    memory pool provides, as in a model."""
    import torch
    f = unfused_fn(wl)
    if compiled:
        f = torch.compile(f, dynamic=False, fullgraph=True)

    def factory(form, M, v, bufs):
        ins = bufs[:4] if wl.kind == "mlp" else bufs[:3]
        return lambda: f(*ins)
    return factory


def unfused_pairs(wl):
    """One ((form, M, v), bufs) per distinct M, on separate-form (or MLP)
    buffers: the unfused baseline is timed once per M and serves both forms."""
    seen = {}
    for (form, M, v), bufs in zip(wl.calls, wl.buffers):
        if form in ("separate", "mlp") and M not in seen:
            seen[M] = ((form, M, v), bufs)
    return seen


def fusion_report(wl, fused_us, eager_us, hbm_gbs):
    """Fusion efficiency per call: the time fusion actually saved against the
    eager unfused path, over the time the eliminated intermediate traffic
    would take at the measured HBM bandwidth.  The eliminated traffic is the
    gate and up tensors written and read once each (8·M·N bytes in BF16; for
    the interleaved form the [M, 2N] product, the same bytes).  Also the
    arithmetic-intensity increase: unfused bytes over fused bytes, minus one."""
    rows = []
    for (form, M, v), tf, te in zip(wl.calls, fused_us, eager_us):
        saved_bytes = 8 * M * wl.N
        t_theory = saved_bytes / (hbm_gbs * 1e9) * 1e6
        fb = wl.algorithmic_bytes(M)
        rows.append({"form": form, "M": M, "fused_us": round(tf, 3), "eager_us": round(te, 3),
                     "speedup": round(te / tf, 3),
                     "bytes_eliminated": saved_bytes, "t_eliminated_theory_us": round(t_theory, 3),
                     "fusion_efficiency": round((te - tf) / t_theory, 3),
                     "ai_increase": round((fb + saved_bytes) / fb - 1.0, 3)})
    return rows


def run_context(args, wl, stream, fused_us, hbm_gbs):
    """Context only: the unfused eager path (cuBLAS GEMMs, SiLU, multiply) on
    the same inputs, per call and as one step; fusion efficiency per call;
    optionally the same function under torch.compile."""
    import torch
    if wl.fp8 or wl.kind in ("w4", "mx"):
        return None
    factory = unfused_factory(wl)
    base = unfused_pairs(wl)
    if any(M not in base for (_, M, _) in wl.calls):
        return None   # a step restricted to interleaved calls has no baseline buffers
    by_m = dict(zip(base, measure_calls(wl, stream, args.call_launches, factory,
                                        list(base.values()))))
    eager_us = [by_m[M] for (_, M, _) in wl.calls]

    # the eager step: every call of the fused step replaced by the two-GEMM path
    fns = [factory(*base[M][0], base[M][1]) for (_, M, _) in wl.calls]

    def step():
        for f in fns:
            f()
    steps = min(args.steps, 200)
    with torch.cuda.stream(stream):
        step()
        g = capture(step, stream)
        for _ in range(3):
            g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    what = ("torch eager: (silu(A@W1) * (A@W2)) @ W3 (cuBLAS)" if wl.kind == "mlp" else
            "torch eager: A@W1, A@W2 (two cuBLAS GEMMs on the separate weights), silu, mul; "
            "the common baseline of both fused forms")
    out = {"eager": {"what": what, "ms_per_step": round(ms, 5),
                     "tflops": round(wl.flops / (ms * 1e-3) / 1e12, 2),
                     "per_call_us": [round(u, 3) for u in eager_us]},
           "fusion": fusion_report(wl, fused_us, eager_us, hbm_gbs)}
    one = one_gemm_context(args, wl, stream)
    if one is not None:
        out["one_gemm_same_weight_bytes"] = one
    if not args.no_compile_context:
        out["compile"] = run_compile_context(args, wl, stream, fused_us)
    return out


def one_gemm_context(args, wl, stream):
    """A library floor for reading the same bytes: one cuBLAS GEMM A @ W_fused
    ([K, 2N], the gate and up weights side by side) per call, timed like the
    fused calls.  It reads the weights the fused call reads, once, and writes
    the [M, 2N] product unfused (twice Y's bytes); for small M, where the
    weights dominate, it is what a tuned library takes to stream them."""
    import torch
    if wl.kind != "bf16":
        return None
    pairs = {}
    for (form, M, v), bufs in zip(wl.calls, wl.buffers):
        if form == "interleaved" and M not in pairs:
            pairs[M] = ((form, M, v), bufs)
    if any(M not in pairs for (_, M, _) in wl.calls):
        return None

    def factory(form, M, v, bufs):
        A, Wf = bufs[0], bufs[1]
        return lambda: torch.matmul(A, Wf)
    by_m = dict(zip(pairs, measure_calls(wl, stream, args.call_launches, factory,
                                         list(pairs.values()))))
    return {"what": "cuBLAS A @ W_fused (one GEMM over the same weight bytes, [M, 2N] output)",
            "per_call_us": [round(by_m[M], 3) for (_, M, _) in wl.calls]}


def run_compile_context(args, wl, stream, fused_us):
    """The same unfused function under torch.compile (default mode, static
    shapes), timed per call like the fused calls."""
    import torch
    if "TRITON_PTXAS_PATH" not in os.environ and os.path.exists("/usr/local/cuda/bin/ptxas"):
        os.environ["TRITON_PTXAS_PATH"] = "/usr/local/cuda/bin/ptxas"
    t0 = time.time()
    base = unfused_pairs(wl)
    try:
        by_m = dict(zip(base, measure_calls(wl, stream, args.call_launches,
                                            unfused_factory(wl, compiled=True),
                                            list(base.values()))))
    except Exception as e:  # report, do not fail the benchmark line
        return {"error": f"{type(e).__name__}: {str(e).splitlines()[0][:200]}"}
    comp_us = [by_m[M] for (_, M, _) in wl.calls]
    return {"what": f"torch.compile(fullgraph=True, dynamic=False) of the eager function, "
                    f"torch {torch.__version__}",
            "compile_and_time_s": round(time.time() - t0, 1),
            "per_call_us": [round(u, 3) for u in comp_us],
            "fused_speedup_vs_compile": [round(c / f, 3) for c, f in zip(comp_us, fused_us)]}


# ----------------------------------------------------------------------------- oracle (CPU) arm

class OracleSampler:
    """The CPU oracle on bounded samples of a workload: for every call of the
    step, the same number of seeded rows.  Inputs are made and the oracle's
    rate calibrated once; each sample() then times one row sample."""

    def __init__(self, workload: str):
        import numpy as np
        import oracle
        import swiglu_inputs as si
        self.workload = workload
        K, N, Ms, seed = WORKLOADS[workload]
        self.K, self.N, self.Ms = K, N, Ms
        oracle.build()
        self.threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
        self.rng = np.random.default_rng(seed)
        mlp = workload.endswith("-mlp")
        fp8 = workload.endswith("-fp8")
        prod = workload.endswith("-fp8-rmsnorm")
        w4 = workload.endswith("-w4")
        mxf = workload.rsplit("-", 1)[1] if workload.endswith(("-mxfp8", "-nvfp4")) else None
        if mxf:
            Amx, m1, m2 = si.make_mx(max(Ms), N, K, seed, mxf)
            amx = si.bits_u16(Amx)
            cv = lambda w: tuple(x.numpy() if hasattr(x, "numpy") else x for x in w)
            mxargs = (mxf, cv(m1), cv(m2))
        if w4:
            A4, (W1q, S1), (W2q, S2) = si.make_w4(max(Ms), N, K, seed, W4_GROUP)
            a4 = si.bits_u16(A4)
            w4args = (W1q.numpy(), si.bits_u16(S1), W2q.numpy(), si.bits_u16(S2), W4_GROUP)
        if prod:   # the producer's inputs per M, the FP8 weights of the same recipe
            (_, W1q, W2q), sc = si.make_e4m3(1, N, K, seed)
            w18, w28 = si.bits_u8(W1q), si.bits_u8(W2q)
            xg = {M: tuple(si.bits_u16(t) for t in si.make_producer_inputs(M, K, seed)) for M in Ms}
        elif fp8:
            (Aq, W1q, W2q), sc = si.make_e4m3(max(Ms), N, K, seed)
            a8, w18, w28 = si.bits_u8(Aq), si.bits_u8(W1q), si.bits_u8(W2q)
        else:
            A, W1, W2 = si.make_bf16(max(Ms), N, K, seed)
            a, w1, w2 = si.bits_u16(A), si.bits_u16(W1), si.bits_u16(W2)
            wf = oracle.pack_interleaved(w1, w2)
            w3 = si.bits_u16(si.make_bf16(1, K, N, seed + 100)[1]) if mlp else None
        self.forms = (("mlp",) if mlp else ("separate", "kmajor") if w4 or mxf
                      else ("separate", "interleaved"))
        self.per_row = (6 if mlp else 4) * N * K

        def call(form, M, rows):
            if mxf:
                oracle.swiglu_mx(amx[:M], *mxargs, rows=rows)
            elif w4:
                oracle.swiglu_w4(a4[:M], *w4args, rows=rows)
            elif prod:   # RMSNorm and quantisation of all of A (the scale needs every row)
                sA, aq = oracle.rmsnorm_quant_e4m3(xg[M][0], xg[M][1], RMS_EPS)
                oracle.swiglu_e4m3(aq, w18, w28, sA, sc[1], sc[2], rows=rows)
            elif mlp:
                oracle.mlp_bf16(a[:M], w1, w2, w3, rows=rows)
            elif fp8:
                oracle.swiglu_e4m3(a8[:M], w18, w28, *sc, rows=rows)
            elif form == "separate":
                oracle.swiglu_bf16(a[:M], w1, w2, rows=rows)
            else:
                oracle.swiglu_interleaved_bf16(a[:M], wf, rows=rows)

        self._call = call
        self.calls = [(form, M) for form in self.forms for M in self.Ms]
        f0, s0 = self._one(max(1, self.threads))   # calibration
        self.rate = f0 / s0
        self._min_all_s = None
        self._next = 0

    @property
    def min_all_s(self):
        """The least a sample of every call costs: one row each (the oracle
        decodes the weights on every call, whatever the row count)."""
        if self._min_all_s is None:
            self._min_all_s = self._one(1)[1]
        return self._min_all_s

    def _one(self, rows_per_call, calls=None):
        import numpy as np
        t0 = time.perf_counter()
        flops = 0
        for form, M in calls or self.calls:
            rows = np.sort(self.rng.integers(0, M, size=rows_per_call))
            self._call(form, M, rows)
            flops += self.per_row * rows_per_call
        return flops, time.perf_counter() - t0

    def sample(self, target_s: float):
        """Time one sample of about target_s seconds (at least one row per
        call).  Returns (TFLOP/s, seconds, description)."""
        ncalls = len(self.calls)
        rows = max(1, int(target_s * self.rate / (self.per_row * ncalls)))
        flops, secs = self._one(rows)
        desc = (f"{rows} seeded rows of each of the {ncalls} calls (M in {list(self.Ms)}, "
                f"{'/'.join(self.forms)}), all output columns, K={self.K}: "
                f"{flops / 1e9:.1f} GFLOP in {secs:.2f} s")
        return flops / secs / 1e12, secs, desc

    def sample_one_call(self, target_s: float):
        """A smaller step: one call's seeded rows (the calls in turn).
        Returns (flops, seconds)."""
        form, M = self.calls[self._next % len(self.calls)]
        self._next += 1
        rows = max(1, int(target_s * self.rate / self.per_row))
        return self._one(rows, [(form, M)])


def oracle_sample(workload: str, target_s: float):
    """One bounded sample of about target_s seconds (the cpu_baseline).
    Returns (TFLOP/s, threads, description, seconds)."""
    sampler = OracleSampler(workload)
    v, secs, desc = sampler.sample(target_s)
    return v, sampler.threads, desc, secs


def run_reference(args, ws, rank):
    """The oracle as it stands, on the host cores: inputs made and the rate
    calibrated once, then every warm-up and timed step one row sample, sized
    so that all steps together take about --cpu-seconds (at least one row of
    each call per step, at most 6 s per step)."""
    if rank != 0:
        return None
    sampler = OracleSampler(args.workload)
    target = min(args.cpu_seconds / max(1, args.steps + args.warmup), 6.0)
    vals = []
    desc = ""
    threads = sampler.threads
    if target >= sampler.min_all_s:   # every step samples every call
        for i in range(args.warmup + args.steps):
            v, secs, desc = sampler.sample(target)
            if i >= args.warmup:
                vals.append((v, secs))
    else:   # many steps: each step samples one call, the calls in turn
        flops_t = 0
        for i in range(args.warmup + args.steps):
            f, secs = sampler.sample_one_call(target)
            if i >= args.warmup:
                vals.append((f / secs / 1e12, secs))
                flops_t += f
        desc = (f"{args.steps} steps of one call each (the {len(sampler.calls)} calls in turn, "
                f"M in {list(sampler.Ms)}, {'/'.join(sampler.forms)}), seeded rows, all output "
                f"columns, K={sampler.K}: {flops_t / 1e9:.1f} GFLOP")
    tot_flops = sum(v * s for v, s in vals)
    tot_s = sum(s for _, s in vals)
    value = tot_flops / tot_s
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / max(1, len(vals)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": describe_workload(args.workload),
                   "sample": "each step is a bounded row sample; see cpu_baseline"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ----------------------------------------------------------------------------- variant sweep

SWEEP_BF16 = ("qwen2.5-0.5b-m64", "qwen2.5-0.5b", "qwen2.5-7b", "qwen2.5-72b")
SWEEP_WEIGHTS = ("qwen2.5-0.5b-w4", "qwen2.5-7b-w4", "qwen2.5-0.5b-mxfp8", "qwen2.5-7b-mxfp8",
                 "qwen2.5-0.5b-nvfp4", "qwen2.5-7b-nvfp4")
SWEEP_VARIANTS = ("1sm_n128", "1sm_n64", "1sm_n32", "2sm_n128", "1sm_n64_sk2", "2sm_swap")
SWEEP_MAX_M = {"2sm_swap": 128}   # variants that take a bounded number of rows


def run_sweep(args):
    """Every BF16 variant for every (M, N, K) and weight form of the BF16
    configurations, and every weight-format kernel for the INT4/MXFP8/NVFP4
    configurations, each timed alone like the per-call durations of the main
    run (back-to-back launches in a CUDA graph on rotating input copies).
    Writes the table the variant choice is checked against."""
    import torch
    import swiglu_gemm_transformer_gb300 as sg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    lib = sg.lib()
    stream = torch.cuda.Stream(device=dev)
    entries = []
    sampler = ClockSampler(0)
    sampler.start()
    t0 = time.time()
    names = [w for w in args.sweep_workloads.split(",") if w] or list(SWEEP_BF16 + SWEEP_WEIGHTS)
    for name in names:
        wl = Workload(name, dev)
        for (form, M, v), bufs in zip(wl.calls, wl.buffers):
            if form == "kmajor":   # a separate entry point, not a choice among kernels
                continue
            us = {}
            if wl.kind == "bf16":
                for vn in SWEEP_VARIANTS:
                    if M > SWEEP_MAX_M.get(vn, M):
                        continue
                    us[vn] = round(measure_calls(wl, stream, args.call_launches, None,
                                                 [((form, M, sg.VARIANTS[vn]), bufs)])[0], 3)
                auto = sg.variant_name(v)
            else:
                auto = sg.WEIGHT_KERNELS[sg.swiglu_select_weight_kernel(M, wl.N)]
                for k, kn in enumerate(sg.WEIGHT_KERNELS):
                    sg.swiglu_set_weight_kernel(k)
                    try:
                        us[kn] = round(measure_calls(wl, stream, args.call_launches, None,
                                                     [((form, M, v), bufs)])[0], 3)
                    finally:
                        sg.swiglu_set_weight_kernel(-1)
            rc, detail = sg.swiglu_device_status(stream)
            if rc != sg.OK:
                raise RuntimeError(f"device status in the sweep: {sg.status_string(rc)} ({detail})")
            entries.append({"workload": name, "kind": wl.kind, "form": form, "M": M, "N": wl.N,
                            "K": wl.K, "us": us, "auto": auto})
            log(f"sweep {name} {form} M={M}: auto {auto}, {us}")
        del wl
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    props = torch.cuda.get_device_properties(dev)
    return {"_note": "Per-call device time (us) of every BF16 variant and every weight-format "
                     "kernel, each timed alone: back-to-back launches in a CUDA graph over "
                     "rotating input copies (> 2.5x L2). Written by bench.py --sweep; the "
                     "variant choice is tested against it.",
            "gpu": props.name, "sm_count": props.multi_processor_count,
            "torch": torch.__version__, "clocks": clocks,
            "seconds": round(time.time() - t0, 1), "entries": entries}


def run_small_m_floor(args):
    """The floor under the 0.5B small- and mid-M calls: time, on this GPU and in the same
    way as the per-call durations (back-to-back launches in a CUDA graph over
    rotating input copies larger than L2), a read-only reduction over the
    same weight bytes (one kernel reading W1 and W2 once), cuBLAS on the same
    bytes (one GEMM A x [W1 W2], no activation), and the fused call."""
    import torch
    import swiglu_gemm_transformer_gb300 as sg
    import swiglu_inputs as si
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sg.lib()
    stream = torch.cuda.Stream(device=dev)
    K, N, _, seed = WORKLOADS["qwen2.5-0.5b"]
    peaks, src = load_peaks()
    rows = []
    for M in (64, 128, 512):
        A, W1, W2 = si.make_bf16(M, N, K, seed)
        wbytes = 2 * K * N * 2
        ncopy = max(2, min(32, math.ceil(2.5 * L2_BYTES / wbytes)))
        sets = []
        for _ in range(ncopy):
            Wc = torch.cat([W1, W2], dim=1).to(dev)            # [K, 2N]: the same bytes
            sets.append((A.to(dev), Wc, Wc[:, :N].contiguous(), Wc[:, N:].contiguous(),
                         torch.empty(M, N, dtype=torch.bfloat16, device=dev)))

        def timed(make):
            fns = [make(*c) for c in sets]
            reps = max(1, math.ceil(args.call_launches / ncopy))

            def body():
                for _ in range(reps):
                    for f in fns:
                        f()
            with torch.cuda.stream(stream):
                for f in fns:
                    f()
                g = capture(body, stream)
                g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
            e1.synchronize()
            return 1e3 * e0.elapsed_time(e1) / (reps * ncopy)
        read_us = timed(lambda a, wc, w1, w2, y: (lambda: torch.sum(wc, dtype=torch.float32)))
        gemm_us = timed(lambda a, wc, w1, w2, y: (lambda: torch.matmul(a, wc)))
        fused_us = timed(lambda a, wc, w1, w2, y: (lambda: sg.swiglu_fused(a, w1, w2, y)))
        rc, detail = sg.swiglu_device_status(stream)
        if rc != sg.OK:
            raise RuntimeError(f"device status: {sg.status_string(rc)} ({detail})")
        abytes = 2 * M * K + wbytes + 2 * M * N
        tflop = 4 * M * N * K / 1e12
        rows.append({"M": M, "N": N, "K": K, "weight_bytes": wbytes, "algorithmic_bytes": abytes,
                     "fused_frac_of_tensor": round(tflop / (fused_us * 1e-6) / peaks["bf16_tflops"], 4),
                     "cublas_frac_of_tensor": round(tflop / (gemm_us * 1e-6) / peaks["bf16_tflops"], 4),
                     "read_reduction_us": round(read_us, 3), "cublas_gemm_us": round(gemm_us, 3),
                     "fused_us": round(fused_us, 3),
                     "fused_frac_of_hbm": round(abytes / (fused_us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                     "read_reduction_frac_of_hbm": round(wbytes / (read_us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                     "variant": sg.variant_name(sg.lib().swiglu_select_variant(M, N, K, 0))})
        log(f"small-M floor M={M}: {rows[-1]}")
    props = torch.cuda.get_device_properties(dev)
    return {"what": "floor under the 0.5B small- and mid-M calls (K=896, N=4864)", "gpu": props.name,
            "hbm_gbs_peak": peaks["hbm_gbs"], "peak_source": src, "torch": torch.__version__,
            "rows": rows}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--variant", default="auto",
                    choices=("auto", "1sm_n128", "1sm_n64", "2sm_n128", "1sm_n32", "1sm_n64_sk2",
                             "2sm_swap"))
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--call-launches", type=int, default=96,
                    help="launches per call when timing calls one by one")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="bounded CPU-oracle sample size for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-compile-context", action="store_true",
                    help="skip timing the unfused function under torch.compile (context)")
    ap.add_argument("--sweep", default="",
                    help="time every variant of every configuration and write the table to this file")
    ap.add_argument("--sweep-workloads", default="",
                    help="comma-separated workloads for --sweep (default: all BF16 and weight formats)")
    ap.add_argument("--record-traffic", nargs=4, metavar=("CSV", "KERNEL_KEY", "FAMILY", "CAPTURE"),
                    help="write a traffic record from an ncu CSV (no GPU work)")
    ap.add_argument("--only", default="",
                    help="restrict the step to calls FORM:M[,FORM:M...] (profiling a single kernel)")
    ap.add_argument("--small-m-floor", action="store_true",
                    help="time the floor under the 0.5B small-M calls (read-only reduction and "
                         "cuBLAS on the same weight bytes, and the fused call) and print it")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    ws, rank, local = dist_env()

    if args.record_traffic:
        print(json.dumps(record_traffic(*args.record_traffic)))
        return

    if args.small_m_floor:
        print(json.dumps(run_small_m_floor(args)), flush=True)
        return

    if args.sweep:
        table = run_sweep(args)
        with open(args.sweep, "w") as f:
            json.dump(table, f, indent=1)
        log(f"wrote {args.sweep}")
        return

    if args.impl == "reference":
        out = run_reference(args, ws, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    import torch
    import torch.distributed as dist
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        out, wl, stream = run_ours(args, ws, rank, local)
        if not args.no_context:
            peaks, _ = load_peaks()
            out["context"] = run_context(args, wl, stream, [k["us"] for k in out["kernels"]],
                                         peaks["hbm_gbs"])
        if rank == 0:
            if args.no_cpu_baseline or ws > 1:
                out["cpu_baseline"] = None
            else:
                v, threads, desc, _ = oracle_sample(args.workload, args.cpu_seconds)
                out["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": threads,
                                       "kind": "oracle", "sample": desc}
            print(json.dumps(out), flush=True)
    finally:
        if ws > 1:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
