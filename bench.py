#!/usr/bin/env python3
"""Benchmark of the dense GEMM hot path on GB300.

One "step" is one call of the library's public C ABI on one batch of synthetic input
(resident in HBM).  The default workload is the FP32 SGEMM M = N = K = 4096,
alpha = 1, beta = 0.5; --workload picks another of the path's configurations
(ffn_bf16, ffn_gate_up, bf16_4096, decode_m1 / decode_m4 / decode_m16,
decode_chain_m1 / decode_chain_m16, qk_batched,
attn_batched, attn_causal_8k, fp8_ffn, fp8_quant_gemm, sgemm_ragged, sgemm_256).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the launching stream; rotating
copies of the inputs make the working set larger than L2 between successive steps.
Rank 0 prints one JSON line.  Under torchrun each rank runs an independent replica of
the workload (the path is one problem; ranks exchange nothing) and `value` is the sum
of the ranks' work divided by the slowest rank's time.

--impl reference times the CPU oracle (the repository's FP64 reference) on a bounded
sample of the same workload, on the host cores, and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS (2MNK/s) and % of GB300 BF16/FP32 roofline; GB/s at M=1..16"
L2_BYTES = 126.5 * 2 ** 20
FP32_LANES_PER_SM = 128          # FP32 FMA units per SM (4 partitions x 32)
SM_MAX_MHZ_NOMINAL = 2070.0      # only if MEASURED_PEAKS.json gives no maximum SM clock

# ncu DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum, one capture of
# the workload's kernel), keyed by workload; an entry is used only while the hash of the
# kernel's sources (kernel file, planner, headers) matches the one it was taken with.
COMMON_SOURCES = ["api.cu", "dg_internal.h", "ptx.cuh", "tile_sched.h"]
MEASURED_TRAFFIC = {
    "sgemm_4096": {"bytes_per_launch": 388_868_608, "source_hash": "e90c5c171ec77a81"},
    "sgemm_ragged": {"bytes_per_launch": 24_665_344, "source_hash": "e90c5c171ec77a81"},
    "sgemm_256": {"bytes_per_launch": 554_240, "source_hash": "e90c5c171ec77a81"},
    "ffn_bf16": {"bytes_per_launch": 150_730_752, "source_hash": "b49d157f5b547065"},
    "ffn_gate_up": {"bytes_per_launch": 232_507_904, "source_hash": "b49d157f5b547065"},
    "bf16_4096": {"bytes_per_launch": 131_843_328, "source_hash": "b49d157f5b547065"},
    "qk_batched": {"bytes_per_launch": 1_078_787_584, "source_hash": "b49d157f5b547065"},
    "decode_m1": {"bytes_per_launch": 104_879_616, "source_hash": "fcbaba222da94a3d"},
    "decode_m4": {"bytes_per_launch": 105_319_424, "source_hash": "fcbaba222da94a3d"},
    "decode_m16": {"bytes_per_launch": 105_675_520, "source_hash": "fcbaba222da94a3d"},
    "decode_chain_m1": {"bytes_per_launch": 408_517_376, "source_hash": "2e8a06e855c12dd8"},
    "attn_batched": {"bytes_per_launch": 116_075_008, "source_hash": "5c5fab7452fd54ff"},
    "attn_causal_8k": {"bytes_per_launch": 6_360_064, "source_hash": "5c5fab7452fd54ff"},
    "fp8_ffn": {"bytes_per_launch": 57_798_912, "source_hash": "2d2f1dc164bf18bc"},
    "fp8_quant_gemm": {"bytes_per_launch": 23_177_472, "source_hash": "2d2f1dc164bf18bc", "quantiser_bytes_per_launch": 12_605_696},
}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    sm_max_mhz=d.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL), source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sustained=1700.0, sm_max_mhz=SM_MAX_MHZ_NOMINAL,
                source="fallback")


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "dense_gemm_sm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- workloads

class Workload:
    """Device buffers (rotating copies) + one step = one library call."""

    def __init__(self, name, torch, dg, inputs):
        self.name = name
        self.torch = torch
        self.dg = dg
        spec = self.spec(name, inputs)
        self.__dict__.update(spec)

    # ---- description of each configuration
    @staticmethod
    def spec(name, inputs):
        if name in ("sgemm_4096", "sgemm_ragged", "sgemm_256"):
            w = {"sgemm_4096": inputs.sgemm_4096, "sgemm_ragged": inputs.sgemm_ragged,
                 "sgemm_256": inputs.sgemm_256}[name]()
            M, N, K = w["M"], w["N"], w["K"]
            return dict(kind="f32", w=w, batch=1, flops=2.0 * M * N * K,
                        algo_bytes=4.0 * (M * K + K * N + (2 if w["beta"] != 0 else 1) * M * N),
                        bound="alu", unit="TFLOPS",
                        kernel="sgemm_small_kernel" if name == "sgemm_256" else "sgemm_tma_kernel",
                        sources=["sgemm_simt.cu"] + COMMON_SOURCES,
                        desc=f"FP32 SGEMM M={M} N={N} K={K} lda={w['lda']} ldb={w['ldb']} "
                             f"ldc={w['ldc']} alpha={float(w['alpha'])} beta={float(w['beta'])}")
        if name == "ffn_bf16":
            w = inputs.ffn_bf16()
            M, N, K = w["M"], w["N"], w["K"]
            return dict(kind="bf16", w=w, batch=1, flops=2.0 * M * N * K,
                        algo_bytes=2.0 * (M * K + K * N + M * N), bound="tensor", unit="TFLOPS",
                        kernel="gemm_tc_kernel", sources=["gemm_tc.cu"] + COMMON_SOURCES,
                        desc=f"BF16 FFN projection C=XW M={M} N={N} K={K}, FP32 accumulate, BF16 out")
        if name == "ffn_gate_up":
            w = inputs.ffn_gate_up()
            M, N, K = w["M"], w["N"], w["K"]
            w = dict(w, A=w["X"], B=w["Wg"], B2=w["Wu"], lda=K, ldb=N, ldc=N, C0=None,
                     alpha=1.0, beta=0.0)
            return dict(kind="gate_up", w=w, batch=1, flops=4.0 * M * N * K,
                        algo_bytes=2.0 * (M * K + 2 * K * N + M * N), bound="tensor",
                        unit="TFLOPS", kernel="gemm_tc_kernel",
                        sources=["gemm_tc.cu"] + COMMON_SOURCES,
                        desc=f"BF16 FFN gate/up Z=SiLU(XW_g)*(XW_u) M={M} N={N} K={K}, "
                             f"FP32 accumulate, BF16 out")
        if name in ("attn_batched", "attn_causal_8k"):
            causal = name == "attn_causal_8k"
            w = inputs.attention(1, 8192, causal=True) if causal else inputs.attention()
            b, L, Lkv, d = w["batch"], w["Lq"], w["Lkv"], w["d"]
            pairs = b * (L * (L + 1) // 2 if causal else L * Lkv)   # (query, visible key) pairs
            w = dict(w, A=w["Q"], B=w["K"], B2=w["V"])
            return dict(kind="attn", w=w, batch=b, flops=4.0 * d * pairs,
                        algo_bytes=2.0 * b * d * (2 * L + 2 * Lkv), bound="tensor", unit="TFLOPS",
                        kernel="attn_fwd_kernel", sources=["attention.cu"] + COMMON_SOURCES,
                        desc=f"fused attention O=softmax(QK^T/sqrt(d))V heads={b} L={L} d={d} "
                             f"{'causal' if causal else 'non-causal'}, BF16 in/out, FP32 accumulate")
        if name in ("fp8_ffn", "fp8_quant_gemm"):
            # fp8_ffn: the FFN shape on resident E4M3 codes; fp8_quant_gemm: the pages' FP8
            # example (A BF16 [4096, 4096] quantised per row each step, then the GEMM with
            # resident E4M3 weights [1536, 4096]); both BF16 out.
            w = inputs.fp8_gemm() if name == "fp8_ffn" else inputs.fp8_gemm(4096, 1536, 4096)
            M, N, K = w["M"], w["N"], w["K"]
            quant = name == "fp8_quant_gemm"
            return dict(kind="fp8", w=dict(w, quant=quant), batch=1, flops=2.0 * M * N * K,
                        algo_bytes=(M * K + K * N + 2.0 * M * N + (3.0 * M * K if quant else 0.0)),
                        bound="tensor8", unit="TFLOPS", kernel="gemm_tc_kernel",
                        sources=["gemm_tc.cu", "quant.cu"] + COMMON_SOURCES,
                        desc=(f"FP8 E4M3 GEMM C=diag(sa)(A B^T)diag(sb) M={M} N={N} K={K}, "
                              f"FP32 accumulate, BF16 out"
                              + (", per-row quantisation of BF16 A inside each step" if quant else "")))
        if name.startswith("decode_chain_m"):
            m = int(name[len("decode_chain_m"):])
            w = inputs.decode_chain(m)
            dims = w["dims"]
            L = len(dims) - 1
            byts = sum(2.0 * (m * dims[l] + dims[l] * dims[l + 1] + m * dims[l + 1]) for l in range(L))
            fl = sum(2.0 * m * dims[l] * dims[l + 1] for l in range(L))
            return dict(kind="chain", w=w, batch=1, flops=fl, algo_bytes=byts, bound="hbm",
                        unit="GB/s", kernel="gemm_chain_kernel",
                        sources=["gemm_chain.cu"] + COMMON_SOURCES,
                        desc=f"persistent decode chain of {L} BF16 GEMMs, M={m}, widths "
                             f"{'-'.join(str(d) for d in dims)}, one launch, BF16 out")
        if name == "bf16_4096":
            w = inputs.bf16_square(4096)
            M, N, K = w["M"], w["N"], w["K"]
            return dict(kind="bf16", w=w, batch=1, flops=2.0 * M * N * K,
                        algo_bytes=2.0 * (M * K + K * N + M * N), bound="tensor", unit="TFLOPS",
                        kernel="gemm_tc_kernel", sources=["gemm_tc.cu"] + COMMON_SOURCES,
                        desc=f"BF16 GEMM M=N=K={M}, FP32 accumulate, BF16 out")
        if name.startswith("decode_m"):
            m = int(name[len("decode_m"):])
            w = inputs.decode_bf16(m)
            M, N, K = w["M"], w["N"], w["K"]
            return dict(kind="bf16", w=w, batch=1, flops=2.0 * M * N * K,
                        algo_bytes=2.0 * (M * K + K * N + M * N), bound="hbm", unit="GB/s",
                        kernel="gemm_thin_kernel", sources=["gemm_thin.cu"] + COMMON_SOURCES,
                        desc=f"BF16 decode GEMM M={M} N={N} K={K}, BF16 out")
        if name == "qk_batched":
            w = inputs.qk_batched()
            b, S, D = w["batch"], w["M"], w["K"]
            return dict(kind="bf16b", w=w, batch=b, flops=2.0 * b * S * S * D,
                        algo_bytes=2.0 * b * (2 * S * D) + 4.0 * b * S * S, bound="hbm",
                        unit="TFLOPS", kernel="gemm_tc_kernel", sources=["gemm_tc.cu"] + COMMON_SOURCES,
                        desc=f"strided-batched BF16 S=QK^T*alpha batch={b} S={S} d={D}, FP32 out")
        raise ValueError(f"unknown workload {name}")

    def setup(self, copies=None):
        torch = self.torch
        w = self.w
        per_copy = self.algo_bytes
        if copies is None:
            # Enough rotating copies that the inputs of the steps between two uses of a copy
            # exceed twice the L2 (small workloads get many small copies).
            copies = max(2, int(np.ceil(2.0 * L2_BYTES / per_copy)) + 1)
            copies = min(copies, 512)
        self.copies = copies
        self.bufs = []
        if self.kind == "chain":
            dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()
            dims = w["dims"]
            for i in range(copies):
                X = dev(w["X"])
                Ws = [dev(W) for W in w["Ws"]]
                Ys = [torch.empty(w["M"] * dims[l + 1], dtype=torch.bfloat16, device="cuda")
                      for l in range(len(Ws))]
                self.bufs.append((X, Ws, Ys))
            torch.cuda.synchronize()
            self.stream = torch.cuda.current_stream().cuda_stream
            return
        if self.kind == "fp8":
            # Resident codes and scales, made by the library's own quantiser (setup, untimed).
            M, N, K = w["M"], w["N"], w["K"]
            dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()
            for i in range(copies):
                X, Wt = dev(w["X"]), dev(w["W"])
                A = torch.empty((M, K), dtype=torch.uint8, device="cuda")
                SA = torch.empty((M,), dtype=torch.float32, device="cuda")
                B = torch.empty((N, K), dtype=torch.uint8, device="cuda")
                SB = torch.empty((N,), dtype=torch.float32, device="cuda")
                self.dg.quantize_rows_e4m3(M, K, X, K, A, K, SA)
                self.dg.quantize_rows_e4m3(N, K, Wt, K, B, K, SB)
                del Wt
                C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
                self.bufs.append(((A, SA, X), (B, SB), C))
            torch.cuda.synchronize()
            self.stream = torch.cuda.current_stream().cuda_stream
            return
        if self.kind == "f32":
            for i in range(copies):
                A = torch.from_numpy(w["A"]).cuda()
                B = torch.from_numpy(w["B"]).cuda()
                C = torch.from_numpy(w["C0"]).cuda() if w["C0"] is not None else \
                    torch.zeros((w["M"], w["ldc"]), dtype=torch.float32, device="cuda")
                self.bufs.append((A, B, C))
        else:
            def bf(bits):
                return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()
            for i in range(copies):
                A, B = bf(w["A"]), bf(w["B"])
                if self.kind in ("gate_up", "attn"):
                    B = torch.cat([B.reshape(-1), bf(w["B2"]).reshape(-1)])  # [W_g | W_u], [K | V]
                if self.kind == "attn":
                    C = torch.empty((w["batch"], w["Lq"], w["d"]), dtype=torch.bfloat16, device="cuda")
                    self.bufs.append((A, B, C))
                    continue
                if self.kind == "bf16b":
                    C = torch.empty((w["batch"], w["M"], w["N"]), dtype=torch.float32, device="cuda")
                else:
                    C = torch.empty((w["M"], w["N"]), dtype=torch.bfloat16, device="cuda")
                self.bufs.append((A, B, C))
        torch.cuda.synchronize()
        self.stream = torch.cuda.current_stream().cuda_stream

    def step(self, i, bufs=None):
        A, B, C = bufs if bufs is not None else self.bufs[i % self.copies]
        w, dg, s = self.w, self.dg, self.stream
        if self.kind == "f32":
            dg.gemm_f32(w["M"], w["N"], w["K"], float(w["alpha"]), A, w["lda"], B, w["ldb"],
                        float(w["beta"]), C, w["ldc"], stream=s)
        elif self.kind == "gate_up":
            kn = w["K"] * w["N"]
            dg.gemm_bf16_gate_up_silu(w["M"], w["N"], w["K"], A, w["lda"], B, w["ldb"],
                                      B.data_ptr() + 2 * kn, w["ldb"], C, w["ldc"], stream=s)
        elif self.kind == "chain":
            dims = w["dims"]
            dg.gemm_bf16_decode_chain(w["M"], dims, A, dims[0], B, dims[1:], C, stream=s)
        elif self.kind == "fp8":
            (qa, sa, X), (qb, sb) = A, B
            M, N, K = w["M"], w["N"], w["K"]
            if w["quant"]:
                dg.quantize_rows_e4m3(M, K, X, K, qa, K, sa, stream=s)
            dg.gemm_fp8_e4m3(M, N, K, qa, K, sa, qb, K, sb, C, N, dg.DG_OUT_BF16, stream=s)
        elif self.kind == "attn":
            kv = w["batch"] * w["Lkv"] * w["d"]
            dg.attention_bf16(w["batch"], w["Lq"], w["Lkv"], w["d"], float(w["scale"]), w["causal"],
                              A, w["ldq"], w["sQ"], B, w["ldk"], w["sK"], B.data_ptr() + 2 * kv,
                              w["ldv"], w["sV"], C, w["ldo"], w["sO"], stream=s)
        elif self.kind == "bf16":
            dg.gemm_bf16(w["M"], w["N"], w["K"], float(w["alpha"]), A, w["lda"], B, w["ldb"],
                         float(w["beta"]), C, w["ldc"], dg.DG_OUT_BF16, stream=s)
        else:
            dg.gemm_bf16_strided_batched(w["M"], w["N"], w["K"], float(w["alpha"]), A, w["lda"],
                                         w["strideA"], B, w["ldb"], w["strideB"], w["op_b"],
                                         float(w["beta"]), C, w["ldc"], w["strideC"], w["batch"],
                                         dg.DG_OUT_F32, stream=s)

    def metric_value(self, seconds_per_step):
        if self.unit == "GB/s":
            return self.algo_bytes / seconds_per_step / 1e9
        return self.flops / seconds_per_step / 1e12

    def roofline(self, sec_per_launch, peaks, sm_mhz):
        """Roofline object of the workload's kernel.  Every kernel here is timed in
        isolation (back-to-back calls over a region of milliseconds, not inside a
        seconds-long step), so the tensor peaks are the burst figures of the measured
        peaks; the FP32 CUDA-core peak comes from this device's SM count and the maximum
        SM clock."""
        if self.bound == "alu":
            sms = self.torch.cuda.get_device_properties(self.torch.cuda.current_device()).multi_processor_count
            peak = sms * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
            achieved = self.flops / sec_per_launch / 1e12
            unit = "TFLOP/s"
            note = (f"FP32 CUDA-core peak = {sms} SMs (this device) x {FP32_LANES_PER_SM} FMA/clk x 2 "
                    f"x {peaks['sm_max_mhz']:.0f} MHz (maximum SM clock)")
        elif self.bound == "tensor8":
            peak = 2.0 * peaks["bf16"]
            achieved = self.flops / sec_per_launch / 1e12
            unit = "TFLOP/s"
            note = (f"fp8 dense = 2 x the bf16 burst cuBLAS figure of {peaks['source']} peaks "
                    f"(nominal fp8 / bf16 ratio 4.5 / 2.25); kernel timed in isolation")
        elif self.bound == "tensor":
            peak = peaks["bf16"]
            achieved = self.flops / sec_per_launch / 1e12
            unit = "TFLOP/s"
            note = f"bf16 dense, burst cuBLAS figure of {peaks['source']} peaks; kernel timed in isolation"
        else:
            peak = peaks["hbm_gbs"]
            achieved = self.algo_bytes / sec_per_launch / 1e9
            unit = "GB/s"
            note = f"HBM copy bandwidth of {peaks['source']} peaks"
        traffic = None
        other = None
        t = MEASURED_TRAFFIC.get(self.name)
        if t and t["source_hash"] == kernel_source_hash(self.sources):
            traffic = t["bytes_per_launch"]
            if "quantiser_bytes_per_launch" in t:
                # the step's other kernel (the per-row quantiser before the FP8 GEMM)
                other = {"kernel": "quantize_rows_kernel", "traffic": t["quantiser_bytes_per_launch"]}
        out = {"bound": "tensor" if self.bound == "tensor8" else self.bound,
               "achieved": round(achieved, 3), "peak": round(peak, 1),
               "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
               "kernel": self.kernel, "algorithmic": {"flops": self.flops, "bytes": self.algo_bytes},
               "peak_note": note}
        if other is not None:
            out["other_kernel"] = other
        return out


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        use = inside if inside else sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for k, name in enumerate(names):
                if r[3][5 + k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(inside)}


# --------------------------------------------------------------------------- runs

def time_steps(torch, wl, steps, warmup, barrier):
    """Warm-up, then exactly `steps` back-to-back steps between one pair of CUDA events on
    the launching stream (events between the launches would add their own gaps).  Each
    step is one kernel launch, so total / steps is the kernel's average launch duration
    over the timed region."""
    for i in range(warmup):
        wl.step(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        wl.step(warmup + i)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t1 = time.time()
    total_ms = start.elapsed_time(end)
    return total_ms, [total_ms / steps], t0, t1


def time_graph(torch, wl, steps, warmup):
    """The same back-to-back steps captured once in a CUDA graph and replayed: one submission
    launches all `steps` kernels, so the host's per-call cost drops out of the time.  The
    capture stream gets its own library workspace, set up by warm-up calls on that stream
    before the capture.  Returns milliseconds per step."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    saved = wl.stream
    wl.stream = side.cuda_stream
    try:
        with torch.cuda.stream(side):
            for i in range(warmup):
                wl.step(i)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(steps):
                wl.step(warmup + i)
        graph.replay()  # once, untimed
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(cur)
        graph.replay()
        end.record(cur)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps
    finally:
        wl.stream = saved


# Short kernels also timed as a CUDA-graph replay (launch and submission cost removed).
GRAPH_WORKLOADS = ("sgemm_256", "ffn_bf16", "ffn_gate_up", "decode_m1", "decode_m4", "decode_m16",
                   "decode_chain_m1")


def aggregate_ranks(ms_local, metric_of_seconds, world, dist, device):
    """Whole-job figure of N independent replicas: the slowest rank's time per step (max
    over ranks) and the work of all ranks divided by that time."""
    ms = ms_local
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, metric_of_seconds(ms / 1e3) * world


def aggregate_e2e(e2e, metric_of_seconds, world, dist, device):
    """The e2e object for the whole job, like `value`: the slowest rank's step time, and the
    work and the copies of all ranks (e2e["_ms"] is this rank's unrounded step time)."""
    if e2e is None:
        return None
    ms, value = aggregate_ranks(e2e.pop("_ms"), metric_of_seconds, world, dist, device)
    e2e.update(value=round(value, 3), ms_per_step=round(ms, 4),
               h2d_bytes_per_step=e2e["h2d_bytes_per_step"] * world,
               d2h_bytes_per_step=e2e["d2h_bytes_per_step"] * world)
    return e2e


def time_e2e(torch, wl, steps, warmup):
    """Same workload through the public API with host inputs.  Every step copies that step's
    inputs from pinned host memory, calls the library and reads the result back into pinned
    host memory.  The copies run on two copy streams (host to device, device to host) into
    two sets of device buffers, so that one step's copies overlap its neighbours' kernels, as
    a server streams independent problems; events keep each buffer set's copy-in, kernel and
    read-back in order.  The timed region holds every copy of every timed step.  The last
    two results are compared bit for bit with a serial call (copy in, call, copy out)."""
    w = wl.w
    if wl.kind in ("fp8", "chain"):
        return None  # suite entries on device-resident inputs only
    A0, B0, C0 = wl.bufs[0]
    hA = A0.cpu().pin_memory()
    hB = B0.cpu().pin_memory()
    hC = C0.cpu().pin_memory()
    nbuf = 2
    outs = [torch.empty_like(hC).pin_memory() for _ in range(nbuf)]
    h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
    reads_c = wl.kind == "f32" and w.get("beta", 0) != 0
    if reads_c:
        h2d += hC.numel() * hC.element_size()
    d2h = outs[0].numel() * outs[0].element_size()
    dev = [(torch.empty_like(A0), torch.empty_like(B0), torch.empty_like(C0)) for _ in range(nbuf)]
    comp = torch.cuda.current_stream()
    if comp.cuda_stream != wl.stream:
        raise RuntimeError("the workload's stream is not the current stream")
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]

    # Serial reference result.
    ref = torch.empty_like(hC).pin_memory()
    dA, dB, dC = dev[0]
    dA.copy_(hA)
    dB.copy_(hB)
    dC.copy_(hC)
    wl.step(0, bufs=(dA, dB, dC))
    ref.copy_(dC)
    torch.cuda.synchronize()

    def one(i):
        k = i % nbuf
        dA, dB, dC = dev[k]
        # Buffer set k is free once the kernel of step i - nbuf has finished and its result
        # has been read back (events never recorded are no-ops).
        cin.wait_event(ev_done[k])
        cin.wait_event(ev_out[k])
        with torch.cuda.stream(cin):
            dA.copy_(hA, non_blocking=True)
            dB.copy_(hB, non_blocking=True)
            if reads_c:
                dC.copy_(hC, non_blocking=True)
        ev_in[k].record(cin)
        comp.wait_event(ev_in[k])
        wl.step(0, bufs=(dA, dB, dC))
        ev_done[k].record(comp)
        cout.wait_event(ev_done[k])
        with torch.cuda.stream(cout):
            outs[k].copy_(dC, non_blocking=True)
        ev_out[k].record(cout)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(comp)
    cin.wait_stream(comp)
    cout.wait_stream(comp)
    for i in range(steps):
        one(i)
    comp.wait_stream(cin)
    comp.wait_stream(cout)
    end.record(comp)
    torch.cuda.synchronize()
    sec = start.elapsed_time(end) / 1e3 / steps
    same = all(torch.equal(outs[(steps - 1 - j) % nbuf], ref) for j in range(min(nbuf, steps)))
    return {"value": round(wl.metric_value(sec), 3), "unit": wl.unit, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(sec * 1e3, 4), "_ms": sec * 1e3,
            "overlap": f"copies on two copy streams, {nbuf} device buffer sets",
            "result_equals_serial_call": bool(same)}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, budget_s=15.0, nthreads=None):
    """The oracle, as it stands, on a bounded sample (the first R rows of C) of the workload.
    `nthreads` is the number of host threads the oracle's loops use (all cores by default);
    the returned `cores` is the number it actually used."""
    import oracle
    w = wl.w
    nthreads = nthreads or os.cpu_count() or 1
    if wl.kind == "attn":
        return attn_cpu_baseline(wl, budget_s, nthreads)
    if wl.kind == "chain":
        # The whole chain: four layers of M x 4096 x 12288 are a few seconds of FP64 work at
        # M <= 16, inside any budget used here.
        t = time.perf_counter()
        oracle.decode_chain(w["M"], w["dims"], w["X"], w["dims"][0], w["Ws"], w["dims"][1:],
                            nthreads=nthreads)
        dt = time.perf_counter() - t
        return {"value": round(wl.algo_bytes / dt / 1e9, 6), "unit": wl.unit, "cores": nthreads,
                "kind": "oracle", "sample": f"the whole chain ({len(w['Ws'])} layers), FP64, {dt:.2f} s"}
    if wl.kind == "fp8":
        M, N, K = w["M"], w["N"], w["K"]
        rows = min(M, 64)
        t = time.perf_counter()
        qa, sa = oracle.quantize_rows_e4m3(rows, K, w["X"], K)
        qb, sb = oracle.quantize_rows_e4m3(N, K, w["W"], K)
        oracle.gemm_fp8(rows, N, K, qa, K, sa, qb, K, sb, nthreads=nthreads)
        dt = time.perf_counter() - t
        return {"value": round(2.0 * rows * N * K / dt / 1e12, 6), "unit": wl.unit, "cores": nthreads,
                "kind": "oracle", "sample": f"rows 0..{rows - 1} of C ({rows}/{M}), quantisation of "
                                            f"those rows and of all of B, FP64 GEMM, {dt:.2f} s"}
    M, N, K = w["M"], w["N"], w["K"]
    batch = w.get("batch", 1)
    op_b = w.get("op_b", 0)

    def run(rows):
        A = w["A"].reshape(-1)[: rows * w["lda"]] if batch == 1 else w["A"].reshape(-1)
        C0 = w["C0"]
        if C0 is not None:
            C0 = C0.reshape(-1)[: rows * w["ldc"]]
        t = time.perf_counter()
        if wl.kind == "gate_up":
            oracle.gate_up_silu(rows, N, K, A, w["lda"], w["B"].reshape(-1), w["ldb"],
                                w["B2"].reshape(-1), w["ldb"], nthreads=nthreads)
            return time.perf_counter() - t
        oracle.gemm(rows, N, K, w["alpha"], A, w["lda"], w["B"].reshape(-1), w["ldb"], w["beta"],
                    C0, w["ldc"], op_b=op_b, nthreads=nthreads)
        return time.perf_counter() - t

    rows = min(M, max(nthreads, 16))
    dt = run(rows)
    target = int(rows * budget_s / max(dt, 1e-6) * 0.8)
    rows2 = max(rows, min(M, target))
    if rows2 > rows:
        rows, dt = rows2, run(rows2)
    flops = wl.flops * rows / M / batch
    byts = wl.algo_bytes * rows / M / batch
    value = byts / dt / 1e9 if wl.unit == "GB/s" else flops / dt / 1e12
    return {"value": round(value, 6), "unit": wl.unit, "cores": nthreads, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of C ({rows}/{M} rows{' of batch 0' if batch > 1 else ''}), "
                      f"FP64 triple loop, {dt:.2f} s"}


def attn_cpu_baseline(wl, budget_s, nthreads=None):
    """The attention oracle on the first R query rows of head 0 (numpy float64 matmuls).
    Its matmul steps run on numpy's BLAS threads; a single-thread run limits them with
    threadpoolctl, and returns None where that package is missing (the thread count of a
    BLAS already loaded cannot be changed otherwise)."""
    import oracle
    w = wl.w
    limit = None
    cores = _blas_threads()
    if nthreads is not None and nthreads < cores:
        try:
            from threadpoolctl import threadpool_limits
        except ImportError:
            return None
        limit = threadpool_limits(limits=nthreads, user_api="blas")
        cores = nthreads

    def run(rows):
        t = time.perf_counter()
        oracle.attention(1, w["Lq"], w["Lkv"], w["d"], float(w["scale"]), w["causal"], w["Q"],
                         w["ldq"], w["sQ"], w["K"], w["ldk"], w["sK"], w["V"], w["ldv"], w["sV"],
                         rows=np.arange(rows))
        return time.perf_counter() - t

    try:
        rows = 64
        dt = run(rows)
        target = int(rows * budget_s / max(dt, 1e-6) * 0.8)
        rows2 = max(rows, min(w["Lq"], target))
        if rows2 > rows:
            rows, dt = rows2, run(rows2)
    finally:
        if limit is not None:
            limit.restore_original_limits()
    pairs = rows * (rows + 1) // 2 if w["causal"] else rows * w["Lkv"]
    value = 4.0 * w["d"] * pairs / dt / 1e12
    return {"value": round(value, 6), "unit": wl.unit, "cores": cores, "kind": "oracle",
            "sample": f"query rows 0..{rows - 1} of head 0 ({rows}/{w['Lq']} rows of 1/{w['batch']} "
                      f"heads), float64 softmax(QK^T)V, {dt:.2f} s"}


def _blas_threads():
    """Threads numpy's BLAS may use (the oracle's matmul steps): the CPU count unless limited."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def reference_arm(args):
    """--impl reference: the oracle timed as the reference on this workload's metric."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from dense_gemm_sm_gb300 import inputs
    spec = Workload.spec(args.workload, inputs)

    class W:  # minimal stand-in with the fields cpu_baseline needs
        pass

    wl = W()
    wl.__dict__.update(spec)
    # About 150 s of oracle work for the whole run (steps + warm-up), at least 0.5 s a step.
    per_step = max(0.5, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(wl, budget_s=per_step)
    vals = [cpu_baseline(wl, budget_s=per_step) for _ in range(args.steps)]
    value = float(np.median([v["value"] for v in vals]))
    cb = dict(vals[-1])
    cb["value"] = round(value, 6)
    cb["cpu_model"] = cpu_model()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": wl.unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64)", "config": {"workload": args.workload, "desc": wl.desc},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 6), "unit": wl.unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="sgemm_4096")
    ap.add_argument("--no-suite", action="store_true", help="skip the other workloads' summary")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import dense_gemm_sm_gb300 as dg
    from dense_gemm_sm_gb300 import inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()

    dg.load()
    peaks = read_peaks()
    wl = Workload(args.workload, torch, dg, inputs)
    wl.setup()

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    total_ms, per_launch, t0, t1 = time_steps(torch, wl, args.steps, args.warmup, barrier)
    if sampler:
        time.sleep(0.2)
        sampler.stop()
    st = dg.dg_device_status()
    if st != dg.DG_OK:
        raise SystemExit(f"device status after the timed region: {dg.status_string(st)}")

    ms, value = aggregate_ranks(total_ms / args.steps, wl.metric_value, world, dist,
                                torch.device("cuda"))
    launch_ms = float(np.mean(per_launch))

    e2e = None if args.no_e2e else time_e2e(torch, wl, max(3, min(args.steps, 20)), 2)
    e2e = aggregate_e2e(e2e, wl.metric_value, world, dist, torch.device("cuda"))

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    clocks = sampler.summary(t0, t1) if sampler else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": wl.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"f32": "f32", "fp8": "e4m3"}.get(wl.kind, "bf16"),
        "data": "synthetic (seeded PCG64; shapes and distributions of the pages' workloads)",
        "config": {"workload": args.workload, "desc": wl.desc,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"{wl.copies} rotating input copies "
                         f"({wl.copies * wl.algo_bytes / 2 ** 20:.0f} MiB) > L2 between steps"},
        "roofline": wl.roofline(launch_ms / 1e3, peaks, clocks and clocks["sm_mhz"]),
        "clocks": clocks,
        # One library kernel a step; the FP8 workload that quantises inside each step adds the
        # quantiser's.
        "gpu_launches": args.steps * (2 if wl.kind == "fp8" and wl.w.get("quant") else 1),
        "e2e": e2e,
    }
    if not args.no_suite:
        suite = {}
        for name in ("ffn_bf16", "ffn_gate_up", "bf16_4096", "decode_m1", "decode_m4",
                     "decode_m16", "decode_chain_m1", "decode_chain_m16", "qk_batched",
                     "attn_batched", "attn_causal_8k", "fp8_ffn", "fp8_quant_gemm", "sgemm_ragged",
                     "sgemm_256"):
            if name == args.workload:
                continue
            other = Workload(name, torch, dg, inputs)
            other.setup()
            # 20 steps, or enough for the timed region to span 2 ms: the first launch of a
            # region overlaps no predecessor, which 20 calls of 20 us would not amortise.
            n = 20
            tot, per, _, _ = time_steps(torch, other, n, 3, barrier)
            if tot < 2.0:
                n = int(math.ceil(n * 2.0 / max(tot, 1e-3)))
                tot, per, _, _ = time_steps(torch, other, n, 3, barrier)
            s = tot / n / 1e3
            rf = other.roofline(float(np.mean(per)) / 1e3, peaks, None)
            suite[name] = {"value": round(other.metric_value(s), 3), "unit": other.unit,
                           "ms_per_step": round(s * 1e3, 4), "steps": n, "roofline_frac": rf["frac"],
                           "bound": rf["bound"], "traffic": rf["traffic"]}
            if name in GRAPH_WORKLOADS:
                gms = time_graph(torch, other, n, 3)
                suite[name]["graph"] = {"value": round(other.metric_value(gms / 1e3), 3),
                                        "ms_per_step": round(gms, 4)}
            del other
            torch.cuda.empty_cache()
        st = dg.dg_device_status()
        if st != dg.DG_OK:
            raise SystemExit(f"device status after the suite: {dg.status_string(st)}")
        line["suite"] = suite
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl)
        line["cpu_baseline"]["cpu_model"] = cpu_model()
        # The same oracle on one host thread, beside the all-cores figure (left out where the
        # oracle's threads cannot be limited to one).
        one = cpu_baseline(wl, budget_s=5.0, nthreads=1)
        if one is not None:
            line["cpu_baseline"]["single_thread"] = {"value": one["value"], "cores": one["cores"],
                                                     "sample": one["sample"]}
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
