#!/usr/bin/env python3
"""Benchmark of the online-softmax attention / softmax hot path on GB300.

One JSON line on stdout (rank 0).  Default workload: the batched GQA causal prefill
(B=2, Hq=32, Hkv=8, Sq=Sk=4096, D=128, bf16), whose bf16 tensor-core throughput is the headline
attention metric; the other workloads (single-head fp32/bf16 4096x4096 d=64, the M=64 N=100
d=32 single head, split-K decode, row softmax, 1-D softmax, and the "next" rows) are measured
before it in the same run (so the headline is timed on a GPU already under load) and reported
under "suite", the last key of the line, each as a short
object (value, unit, ms per step, roofline bound / peak / fraction / ncu DRAM bytes, and for the
problem statement's configurations the oracle's throughput on all host cores and on one core).
The full suite entries go to stderr, one JSON object per line.

cpu_baseline: the fp64 oracle on a bounded sample of the headline workload, on all host cores,
and under "one_core" in a child process pinned to one core with one BLAS thread (its
"full_workload_s" extrapolates the sample's rate to the whole workload).

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA events on the
launching stream; between timed steps, outside the events, L2 is flushed by writing a 512 MiB
buffer and then reading a second 256 MiB one (so no dirty lines are left behind to be written back
during the next step).
Barrier + synchronize on both sides of the timed loop; the max over ranks is reported.
With torchrun (N > 1) every rank runs its own replica of the workload (weak scaling: the
path shards over (batch, kv head) with no exchange).

--impl reference times the fp64 CPU oracle (the reference arm) on a bounded
sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
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

import numpy as np  # noqa: E402

METRIC = "attention fwd TFLOP/s & % bf16 TC peak; softmax/decode HBM GB/s & % of 8 TB/s"

WORKLOADS = {
    "gqa_causal_prefill": dict(kind="attn", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128, causal=True,
                               dtype="bf16",
                               desc="batched GQA causal prefill B=2 Hq=32 Hkv=8 Sq=Sk=4096 D=128 bf16 [B,H,S,D]"),
    "gqa_causal_prefill_bshd": dict(kind="attn", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128, causal=True,
                                    dtype="bf16", layout="bshd",
                                    desc="batched GQA causal prefill B=2 Hq=32 Hkv=8 Sq=Sk=4096 D=128 bf16 "
                                         "stored [B,S,H,D], read through strides"),
    "gqa_chunked_prefill": dict(kind="attn", B=2, Hq=32, Hkv=8, Sq=1024, Sk=4096, D=128, causal=True,
                                mask="bottom_right", dtype="bf16",
                                desc="GQA chunked prefill: 1024 new rows after a 3072-key cache (Sk=4096), "
                                     "bottom-right causal, B=2 Hq=32 Hkv=8 D=128 bf16"),
    "gqa_causal_backward": dict(kind="attn_bwd", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128, causal=True,
                                dtype="bf16",
                                desc="backward (dQ, dK, dV) of the GQA causal prefill B=2 Hq=32 Hkv=8 S=4096 D=128 "
                                     "bf16, from O, lse and dO"),
    "single_head_4096_bf16": dict(kind="attn", B=1, Hq=1, Hkv=1, Sq=4096, Sk=4096, D=64, causal=False,
                                  dtype="bf16", desc="single-head attention M=N=4096 d=64 bf16"),
    "single_head_4096_f32": dict(kind="attn", B=1, Hq=1, Hkv=1, Sq=4096, Sk=4096, D=64, causal=False,
                                 dtype="f32", desc="single-head attention M=N=4096 d=64 fp32"),
    "single_head_m64_n100": dict(kind="solve", M=64, N=100, d=32, dtype="f32",
                                 desc="single-head attention solve M=64 N=100 d=32 fp32"),
    "gqa_decode": dict(kind="attn", B=8, Hq=32, Hkv=8, Sq=1, Sk=32768, D=128, causal=False, dtype="bf16",
                       desc="GQA decode B=8 Hq=32 Hkv=8 Sq=1 Sk=32768 D=128 bf16, split-K + LSE combine"),
    "gqa_speculative_decode": dict(kind="attn", B=8, Hq=32, Hkv=8, Sq=4, Sk=32768, D=128, causal=True,
                                   mask="bottom_right", dtype="bf16",
                                   desc="GQA speculative decode: 4 draft rows per head against a 32768-key cache, "
                                        "bottom-right causal, B=8 Hq=32 Hkv=8 D=128 bf16"),
    "softmax_rows": dict(kind="softmax", rows=4096, T=32768,
                         desc="row softmax fp32 [4096, 32768], 8*N(0,1) + one +30 spike per row"),
    "softmax_1d": dict(kind="softmax", rows=1, T=1 << 26,
                       desc="1-D softmax fp32 N=2^26, 8*N(0,1) + one +30 spike"),
    "softmax_rows_bf16": dict(kind="softmax", rows=4096, T=32768, dtype="bf16",
                              desc="row softmax bf16 in, bf16 out [4096, 32768], 8*N(0,1) + one +30 spike per row"),
    "softmax_causal_bf16": dict(kind="softmax", rows=8 * 4096, T=4096, dtype="bf16", period=4096,
                                scale=128 ** -0.5,
                                desc="causal scaled softmax of attention weights, 8 heads x [4096, 4096] bf16, "
                                     "scale 128^-0.5 (columns above the diagonal not read)"),
}
DEFAULT = "gqa_causal_prefill"

# Fallback peaks (one earlier GB300 measurement) when the measured-peaks file is absent.
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}
# FP32 FMA peak for the CUDA-core paths: 152 SMs x 128 FMA lanes x 2 flop x max SM clock.
SM_COUNT_GB300 = 152

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum per launch, from one ncu capture) of
# each workload's dominant kernel, keyed by the sha256 of the CUDA source it was taken on; a
# source that changed since the capture reports null.
TRAFFIC = {
    "gqa_causal_prefill": {"source": "online_softmax_flash_gb300/csrc/attn_tc.cu", "sha": "33729601088ac731",
                           "bytes": 136.62e6, "scope": "attn_tc_kernel<128>, one launch"},
    "gqa_causal_prefill_bshd": {"source": "online_softmax_flash_gb300/csrc/attn_tc.cu", "sha": "33729601088ac731",
                                "bytes": 133.67e6, "scope": "attn_tc_kernel<128> on [B, S, H, D] views, one launch"},
    "gqa_chunked_prefill": {"source": "online_softmax_flash_gb300/csrc/attn_tc.cu", "sha": "33729601088ac731",
                            "bytes": 52.13e6, "scope": "attn_tc_kernel<128>, bottom-right mask, one launch"},
    "gqa_decode": {"source": "online_softmax_flash_gb300/csrc/decode.cu", "sha": "08ba6f0fc6b184f5",
                   "bytes": 1079.13e6, "scope": "decode_kernel<128>, one launch"},
    "gqa_speculative_decode": {"source": "online_softmax_flash_gb300/csrc/decode.cu", "sha": "08ba6f0fc6b184f5",
                               "bytes": 1085.72e6, "scope": "decode_kernel<128>, 16 rows per kv head, one launch"},
    "softmax_rows": {"source": "online_softmax_flash_gb300/csrc/softmax.cu", "sha": "aa0692536436b66b",
                     "bytes": 1013.79e6, "scope": "softmax_rows_resident_kernel<8>, one launch"},
    "softmax_1d": {"source": "online_softmax_flash_gb300/csrc/softmax.cu", "sha": "aa0692536436b66b",
                   "bytes": 753.31e6, "scope": "step: chunk state + chunk normalise kernels"},
    "softmax_rows_bf16": {"source": "online_softmax_flash_gb300/csrc/softmax_ex.cu", "sha": "d07ea9a9b6620ae0",
                          "bytes": 475.47e6, "scope": "softmax_ex_split_kernel<bf16, bf16, 256, 8>, one launch"},
    "softmax_causal_bf16": {"source": "online_softmax_flash_gb300/csrc/softmax_ex.cu", "sha": "d07ea9a9b6620ae0",
                            "bytes": 343.07e6, "scope": "softmax_ex_pair_kernel<bf16, bf16, 64>, one launch"},
    "gqa_causal_backward": {"source": "online_softmax_flash_gb300/csrc/attn_bwd_tc.cu", "sha": "6b2edd0b274b2cfa",
                            "bytes": 1441.99e6,
                            "scope": "bwd_tc_kernel<128> (dK/dV CTAs, writing 1.07 GB of dS^T), one launch"},
    "single_head_4096_f32": {"source": "online_softmax_flash_gb300/csrc/attn_tc.cu", "sha": "33729601088ac731",
                             "bytes": 4.34e6, "scope": "attn_tc_kernel<64, x3>, one launch"},
    "single_head_4096_bf16": {"source": "online_softmax_flash_gb300/csrc/attn_tc.cu", "sha": "33729601088ac731",
                              "bytes": 1.63e6, "scope": "attn_tc_kernel<64>, one launch (8 key splits)"},
}


def peaks():
    p = dict(FALLBACK)
    src = "fallback"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained", "sm_max_mhz"):
            if k in m:
                p[k] = float(m[k])
        src = "measured"
    except (OSError, ValueError):
        pass
    return p, src


def work_units(w):
    """(algorithmic amount per step, unit, roofline bound)."""
    if w["kind"] == "solve":
        return 4.0 * w["M"] * w["N"] * w["d"] / 1e12, "TFLOP/s", "alu"
    if w["kind"] == "attn_bwd":
        # five [Sq, Sk] x D products (S, dP, dV, dK, dQ) against the forward's two
        f = 2.5 * 4.0 * w["B"] * w["Hq"] * w["Sq"] * w["Sk"] * w["D"] / (2 if w["causal"] else 1)
        return f / 1e12, "TFLOP/s", "tensor"
    if w["kind"] == "attn":
        if w["Sq"] * w["Hq"] // w["Hkv"] <= 16:  # decode: every K/V byte read once, plus Q and O
            es = 2 if w["dtype"] == "bf16" else 4
            b = es * (2 * w["B"] * w["Hkv"] * w["Sk"] * w["D"] + 2 * w["B"] * w["Hq"] * w["Sq"] * w["D"])
            return b / 1e9, "GB/s", "hbm"
        f = 4.0 * w["B"] * w["Hq"] * w["Sq"] * w["Sk"] * w["D"]
        if w.get("mask") == "bottom_right":
            # exactly the visible (row, key) pairs: row i sees min(Sk, i + Sk - Sq + 1) keys
            off = w["Sk"] - w["Sq"]
            pairs = sum(max(0, min(w["Sk"], i + off + 1)) for i in range(w["Sq"]))
            f = 4.0 * w["B"] * w["Hq"] * pairs * w["D"]
        elif w["causal"]:
            f /= 2   # the "halved for causal" convention of the headline workload
        if w["dtype"] == "bf16":
            return f / 1e12, "TFLOP/s", "tensor"
        # float32 with D = 64 runs on the bf16 tensor cores as sums of bf16 part products
        return f / 1e12, "TFLOP/s", ("tensor_split" if w["D"] == 64 and w["Sq"] > 1 else "alu")
    # softmax: on-chip rows read once and write once; longer rows read twice
    if w.get("dtype") == "bf16":   # bf16 in and out; a causal row reads only its kept columns
        P, T = w.get("period", 0), w["T"]
        read = w["rows"] * T if not P else (w["rows"] // P) * sum(min(T, r + 1) for r in range(P))
        return 2 * (read + w["rows"] * T) / 1e9, "GB/s", "hbm"
    per = 8 if w["T"] <= 32768 else 12
    return per * w["rows"] * w["T"] / 1e9, "GB/s", "hbm"


def arith_dtype(w):
    """The arithmetic a workload runs in (inputs of float32 attention with D = 64 are split into
    bf16 parts for the tensor cores, with float32 accumulation)."""
    if w["kind"] == "attn" and w.get("dtype") == "f32" and work_units(w)[2] == "tensor_split":
        return "f32 (bf16 parts, f32 accumulate)"
    return w.get("dtype", "f32")


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ----------------------------------------------------------------------------- inputs
def make_inputs(name, w, seed=0):
    import seeded_inputs as si
    if w["kind"] == "solve":
        return si.qkv((w["M"], w["d"]), (w["N"], w["d"]), seed)
    if w["kind"] in ("attn", "attn_bwd"):
        q, k, v = si.qkv((w["B"], w["Hq"], w["Sq"], w["D"]), (w["B"], w["Hkv"], w["Sk"], w["D"]), seed,
                         dtype=w["dtype"])
        if w["kind"] == "attn":
            return q, k, v
        dout = si.qkv((w["B"], w["Hq"], w["Sq"], w["D"]), (1, 1, 1, w["D"]), seed + 1000, dtype=w["dtype"])[0]
        return q, k, v, dout
    if w.get("dtype") == "bf16":
        return (si.f32_to_bf16_bits(si.softmax_rows_input(w["rows"], w["T"], seed)),)
    return (si.softmax_rows_input(w["rows"], w["T"], seed),)


def host_tensors(w, arrays, pin):
    import torch
    out = []
    for a in arrays:
        if a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(a)
        out.append(t.pin_memory() if pin else t)
    return out


class Runner:
    """Device buffers and one call of the hot path for a workload."""

    def __init__(self, name, w, dev, osf, host):
        import torch
        self.w, self.osf, self.dev = w, osf, dev
        self.host = host
        self.bshd = w.get("layout") == "bshd"
        if self.bshd:   # store [B, S, H, D]; the call reads transposed views through strides
            self.host = [h.permute(0, 2, 1, 3).contiguous().pin_memory() for h in host]
        self.d_in = [h.to(dev) for h in self.host]
        if w["kind"] == "solve":
            self.out = torch.empty(w["M"], w["d"], device=dev)
            self.ws = None
        elif w["kind"] == "attn_bwd":
            q, k, v, dout = self.d_in
            dt = osf.OSF_BF16 if w["dtype"] == "bf16" else osf.OSF_F32
            self.lse = torch.empty(w["B"], w["Hq"], w["Sq"], device=dev)
            n = osf.osf_attn_workspace_bytes(dt, w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Sk"], w["D"])
            fws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
            # the forward pass (outside the timed steps) provides O and lse
            self.o = osf.osf_attn_fwd_gqa(q, k, v, causal=w["causal"], lse=self.lse, workspace=fws)
            self.grads = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
            self.out = self.grads[0]
            n = osf.osf_attn_bwd_workspace_bytes(dt, w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Sk"], w["D"])
            self.ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        elif w["kind"] == "attn":
            self.out = torch.empty_like(self.d_in[0])
            self.views = [t.transpose(1, 2) for t in self.d_in + [self.out]] if self.bshd else None
            dt = osf.OSF_BF16 if w["dtype"] == "bf16" else osf.OSF_F32
            n = osf.osf_attn_workspace_bytes(dt, w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Sk"], w["D"])
            self.ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        else:
            self.out = torch.empty_like(self.d_in[0])
            n = osf.osf_softmax_ex_workspace_bytes(w["rows"], w["T"])
            self.ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        self.out_host = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        # attention on contiguous [B, H, S, D] host arrays: the library's host-buffer entry point
        # (copies in, attention and copy out in overlapping chunks)
        self.host_api = w["kind"] == "attn" and not self.bshd and "mask" not in w
        if self.host_api:
            n = osf.osf_attn_host_buffer_bytes(dt, w["B"], w["Hq"], w["Hkv"], w["Sq"], w["Sk"], w["D"], w["causal"])
            self.hbuf = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        if w["kind"] == "attn_bwd":
            self.grads_host = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in self.grads]

    def call(self):
        w, osf = self.w, self.osf
        if w["kind"] == "solve":
            q, k, v = self.d_in
            osf.osf_attn_fwd(q, k, v, self.out, w["M"], w["N"], w["d"])
        elif w["kind"] == "attn_bwd":
            q, k, v, dout = self.d_in
            osf.osf_attn_bwd_gqa(q, k, v, self.o, dout, self.lse, *self.grads,
                                 mask="top_left" if w["causal"] else "none", workspace=self.ws)
        elif w["kind"] == "attn" and (self.bshd or "mask" in w):
            q, k, v, o = self.views if self.bshd else self.d_in + [self.out]
            osf.osf_attn_fwd_gqa_ex(q, k, v, out=o, workspace=self.ws,
                                    mask=w.get("mask", "top_left" if w["causal"] else "none"))
        elif w["kind"] == "attn":
            q, k, v = self.d_in
            osf.osf_attn_fwd_gqa(q, k, v, out=self.out, causal=w["causal"], workspace=self.ws)
        else:
            if w.get("dtype") == "bf16":
                osf.osf_softmax_rows_ex(self.d_in[0], self.out, scale=w.get("scale", 1.0),
                                        causal_period=w.get("period", 0), workspace=self.ws)
            else:
                osf.osf_softmax_rows(self.d_in[0], self.out, workspace=self.ws)

    def call_e2e(self):
        """Host buffers in, host buffer out: H2D copies, the call, D2H copy of the result."""
        if self.host_api:
            q, k, v = self.host
            self.osf.osf_attn_fwd_gqa_host(q, k, v, out=self.out_host, causal=self.w["causal"],
                                           device_buffer=self.hbuf)
            return
        for d, h in zip(self.d_in, self.host):
            d.copy_(h, non_blocking=True)
        self.call()
        if self.w["kind"] == "attn_bwd":
            for g, h in zip(self.grads, self.grads_host):
                h.copy_(g, non_blocking=True)
        else:
            self.out_host.copy_(self.out, non_blocking=True)

    def h2d_bytes(self):
        return sum(h.numel() * h.element_size() for h in self.host)

    def d2h_bytes(self):
        if self.w["kind"] == "attn_bwd":
            return sum(g.numel() * g.element_size() for g in self.grads)
        return self.out.numel() * self.out.element_size()


# ------------------------------------------------------------------------------ clocks
def _physical_index(index):
    """nvidia-smi / NVML number of the GPU that is CUDA ordinal `index` in this process."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").strip()
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if index < len(ids) and ids[index].isdigit():
            return int(ids[index])
    return index


# clock event reason bits of NVML (nvmlClocksEventReason*)
_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


# Child process that reads NVML every millisecond and prints "monotonic_time sm_mhz max_mhz reasons
# mem_mhz" lines (read-only queries); a separate process, so the sampling does not wait on this
# process's interpreter lock while it launches work.
_NVML_CHILD = r"""
import ctypes, sys, time
lib = ctypes.CDLL("libnvidia-ml.so.1")
assert lib.nvmlInit_v2() == 0
h = ctypes.c_void_p()
assert lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(sys.argv[1])), ctypes.byref(h)) == 0
rf = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
sm, mx, rs, mem = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
print("ready", flush=True)
i = 0
while True:
    lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm))
    rf(h, ctypes.byref(rs))
    if i % 8 == 0:   # the maximum and the memory clock change rarely: every eighth sample
        lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
        lib.nvmlDeviceGetClockInfo(h, 2, ctypes.byref(mem))
    print(time.monotonic(), sm.value, mx.value, rs.value, mem.value, flush=True)
    i += 1
    time.sleep(0.0005)
"""


class NvmlSampler:
    """SM clock, its maximum, the clock event reasons and the memory clock, read through NVML about
    every millisecond by a child process; only samples taken inside the window (first warm-up
    step to last timed step, on the system's monotonic clock) count."""

    def __init__(self, index):
        ctypes = __import__("ctypes")
        ctypes.CDLL("libnvidia-ml.so.1")   # raises OSError where NVML is absent
        self.index = _physical_index(index)
        self.rows = []
        self.windows = []
        self.proc = None

    def start(self):
        self.proc = subprocess.Popen([sys.executable, "-c", _NVML_CHILD, str(self.index)], stdout=subprocess.PIPE,
                                     stderr=subprocess.DEVNULL, text=True)
        if self.proc.stdout.readline().strip() != "ready":
            raise OSError("NVML sampler did not start")
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            f = line.split()
            if len(f) == 5:
                self.rows.append((float(f[0]), float(f[1]), float(f[2]), int(f[3]), float(f[4])))

    def window_open(self):
        self.windows.append([time.monotonic(), None])

    def window_close(self):
        self.windows[-1][1] = time.monotonic()

    def stop(self):
        time.sleep(0.01)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        smp = [r[1:] for r in self.rows if any(a <= r[0] <= (b or a) for a, b in self.windows)]
        if not smp:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvml"}
        reasons = sorted(n for n, b in _REASON_BITS.items() if any(s[2] & b for s in smp))
        return {"sm_mhz": statistics.median(s[0] for s in smp), "sm_max_mhz": max(s[1] for s in smp),
                "reasons": reasons, "samples": len(smp), "window": "warm-up + timed steps",
                "mem_mhz": [min(s[3] for s in smp), statistics.median(s[3] for s in smp)],
                "source": "nvml, ~1 ms, child process"}


class ClockSampler:
    """nvidia-smi samples (every 50 ms) kept while the measured loop (warm-up + timed steps) runs;
    the fallback when NVML cannot be loaded."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = _physical_index(index)
        self.samples = []
        self.open = False
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            if self.open:
                self.samples.append([c.strip() for c in line.split(",")])

    def window_open(self):
        self.open = True

    def window_close(self):
        self.open = False

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": "nvidia-smi"}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples), "window": "warm-up + timed steps",
                "source": "nvidia-smi, 50 ms"}


class _Samplers:
    """The NVML sampler, else the nvidia-smi one when NVML cannot be loaded or started."""

    def __init__(self, index):
        self.index = index
        try:
            self.s = NvmlSampler(index)
        except (OSError, AttributeError):
            self.s = ClockSampler(index)

    def start(self):
        try:
            self.s.start()
        except OSError:
            self.s.stop()
            self.s = ClockSampler(self.index)
            self.s.start()

    def __getattr__(self, name):
        return getattr(self.s, name)


def make_sampler(index):
    return _Samplers(index)


# ----------------------------------------------------------------------------- timing
def make_flush(dev):
    import torch
    return (torch.empty(128 << 20, dtype=torch.float32, device=dev),   # 512 MiB, written
            torch.ones(64 << 20, dtype=torch.float32, device=dev),     # 256 MiB, read
            torch.empty(1, dtype=torch.float32, device=dev))


def flush_l2(flush):
    """Evict L2 (129 MB on GB300): write a buffer larger than L2, then read another one."""
    import torch
    w, r, sink = flush
    w.fill_(1.0)
    torch.sum(r, dim=0, out=sink[0])


def time_steps(fn, steps, warmup, flush, stream, barrier=None, sampler=None):
    """Per-step CUDA-event times (ms) of ``fn`` on ``stream``, L2 flushed between steps."""
    import torch
    if sampler:
        sampler.window_open()
    for _ in range(warmup):
        fn()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        if flush is not None:
            flush_l2(flush)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if sampler:
        sampler.window_close()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], wall


def measure(name, w, osf, dev, steps, warmup, flush, barrier=None, sampler=None, e2e=True):
    import torch
    arrays = make_inputs(name, w)
    host = host_tensors(w, arrays, pin=True)
    r = Runner(name, w, dev, osf, host)
    stream = torch.cuda.current_stream(dev)
    amount, unit, bound = work_units(w)
    n0 = osf.osf_launch_count()
    r.call()
    torch.cuda.synchronize()
    launches_per_call = osf.osf_launch_count() - n0
    n1 = osf.osf_launch_count()
    ms, wall = time_steps(r.call, steps, warmup, flush, stream, barrier, sampler)
    launches = osf.osf_launch_count() - n1 - warmup * launches_per_call
    status = osf.osf_device_status()
    res = {"name": name, "amount": amount, "unit": unit, "bound": bound, "ms": ms, "wall_s": wall,
           "launches": int(launches), "launches_per_call": int(launches_per_call), "status": status}
    if e2e:
        ems, _ = time_steps(r.call_e2e, max(3, steps // 4), 2, flush, stream, barrier)
        res["e2e_ms"] = ems
        res["e2e_call"] = ("osf_attn_fwd_gqa_host (C ABI on pinned host buffers; chunked copies overlap "
                           "the attention)" if r.host_api else
                           "H2D copies of the inputs, the C-ABI call on device buffers, D2H copy of the result")
        res["h2d"] = r.h2d_bytes()
        res["d2h"] = r.d2h_bytes()
    del r
    torch.cuda.empty_cache()
    return res


def roofline(res, pk, w):
    mean_ms = statistics.mean(res["ms"])
    achieved = res["amount"] / (mean_ms / 1e3)
    note = None
    if res["bound"] == "tensor":
        peak, unit = pk["bf16_tflops"], "TFLOP/s"
    elif res["bound"] == "tensor_split":
        # six bf16 products per score product (three-part Q, K) and three per PV product
        # (two-part P, V): the attainable rate is the bf16 peak / 4.5
        peak, unit = pk["bf16_tflops"] / 4.5, "TFLOP/s"
        note = "bf16 tensor peak / 4.5 (float32 as bf16 parts: 6 products per score product, 3 per PV product)"
    elif res["bound"] == "hbm":
        peak, unit = pk["hbm_gbs"], "GB/s"
    else:  # FP32 FMA pipe
        peak, unit = SM_COUNT_GB300 * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12, "TFLOP/s"
    t = TRAFFIC.get(res["name"])
    traffic = scope = None
    if t and source_hash(os.path.join(ROOT, t["source"])) == t["sha"]:
        traffic, scope = t["bytes"], t["scope"]
    out = {"bound": "tensor" if res["bound"] == "tensor_split" else res["bound"], "achieved": round(achieved, 3),
           "peak": round(peak, 1), "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
           "traffic_scope": scope, "algorithmic": round(res["amount"] * (1e12 if unit == "TFLOP/s" else 1e9)),
           "per": "flop" if unit == "TFLOP/s" else "byte"}
    if note:
        out["peak_note"] = note
    return out


# ------------------------------------------------------------------------------ oracle arm
def host_cores():
    """Host cores this process may run on (numpy's BLAS starts one thread per core)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_timed(name, w, budget_s):
    """Oracle throughput on a bounded sample of a workload: `budget_s` seconds of oracle time,
    input generation outside the clock (and the whole loop capped at four times the budget)."""
    import oracle
    import seeded_inputs as si
    amount, unit, _ = work_units(w)
    cores = host_cores()
    elapsed, done, n = 0.0, 0.0, 0
    wall0 = time.perf_counter()
    budget_left = lambda: elapsed < budget_s and time.perf_counter() - wall0 < 4 * budget_s
    if w["kind"] == "solve":
        Q, K, V = make_inputs(name, w)
        while elapsed < min(budget_s, 2.0):
            t = time.perf_counter()
            oracle.attention(Q, K, V)
            elapsed += time.perf_counter() - t
            n += 1
            done += amount
        return done / elapsed, unit, f"{n} full solves", cores
    if w["kind"] == "attn_bwd":
        B, Hq, S, D = w["B"], w["Hq"], w["Sq"], w["D"]
        per_head = amount / (B * Hq)
        while n < B * Hq and budget_left():
            q, kk, vv, g = (si.normal_f32((S, D), n, st) for st in (si.STREAM_Q, si.STREAM_K, si.STREAM_V, si.STREAM_X))
            q, kk, vv, g = (si.bf16_bits_to_f32(si.f32_to_bf16_bits(a)) for a in (q, kk, vv, g))
            t = time.perf_counter()
            oracle.attention_bwd(q, kk, vv, g, q_index=np.arange(S) if w["causal"] else None)
            elapsed += time.perf_counter() - t
            n += 1
            done += per_head
        return done / elapsed, unit, f"{n} of {B * Hq} (b, q-head) problems, full {S}x{w['Sk']} gradients each", cores
    if w["kind"] == "attn" and w["Sq"] > 1:
        B, Hq, S, D = w["B"], w["Hq"], w["Sq"], w["D"]
        per_head = amount / (B * Hq)
        while n < B * Hq and budget_left():
            q = si.normal_f32((S, D), n, si.STREAM_Q)
            kk = si.normal_f32((w["Sk"], D), n, si.STREAM_K)
            vv = si.normal_f32((w["Sk"], D), n, si.STREAM_V)
            if w["dtype"] == "bf16":
                q, kk, vv = (si.bf16_bits_to_f32(si.f32_to_bf16_bits(a)) for a in (q, kk, vv))
            qi = None
            if w.get("mask") == "bottom_right":
                qi = np.arange(S) + (w["Sk"] - S)
            t = time.perf_counter()
            oracle.attention(q, kk, vv, causal=w["causal"], q_index=qi)
            elapsed += time.perf_counter() - t
            n += 1
            done += per_head
        return done / elapsed, unit, f"{n} of {B * Hq} (b, q-head) problems, full {S}x{w['Sk']} scores each", cores
    if w["kind"] == "attn":
        B, Hq, Hkv, Sk, D = w["B"], w["Hq"], w["Hkv"], w["Sk"], w["D"]
        G = Hq // Hkv
        per = amount / (B * Hkv)
        while n < B * Hkv and budget_left():
            q = si.normal_f32((1, G, 1, D), n, si.STREAM_Q)
            kk = si.normal_f32((1, 1, Sk, D), n, si.STREAM_K)
            vv = si.normal_f32((1, 1, Sk, D), n, si.STREAM_V)
            t = time.perf_counter()
            oracle.attention_gqa(q, kk, vv)
            elapsed += time.perf_counter() - t
            n += 1
            done += per
        return done / elapsed, unit, f"{n} of {B * Hkv} (b, kv-head) groups", cores
    rows, T = w["rows"], w["T"]
    P = w.get("period", 0)
    step = P if P else (64 if rows > 1 else 1)   # whole score matrices keep the causal row numbers
    while n < rows and budget_left():
        x = si.softmax_rows_input(step, T, n)
        if w.get("dtype") == "bf16":
            x = si.bf16_bits_to_f32(si.f32_to_bf16_bits(x))
        t = time.perf_counter()
        if w.get("dtype") == "bf16" or P:
            oracle.softmax_masked(x, w.get("scale", 1.0), P)
        else:
            oracle.softmax(x)
        elapsed += time.perf_counter() - t
        n += step
        done += amount * step / rows
    return done / elapsed, unit, f"{n} of {rows} rows of {T}", cores


# Thread-count variables of the BLAS libraries numpy may be built on.
ONE_THREAD_ENV = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                                  "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")}


def oracle_probe(name, budget_s):
    """Child-process side of `oracle_one_core`: pin this process to one core, time the oracle and
    print one JSON object.  The BLAS thread variables were set before numpy was imported."""
    try:
        cpu = min(os.sched_getaffinity(0))
        os.sched_setaffinity(0, {cpu})
    except (AttributeError, OSError):
        pass
    v, unit, sample, _ = oracle_timed(name, WORKLOADS[name], budget_s)
    print(json.dumps({"value": v, "unit": unit, "sample": sample, "cores": host_cores()}), flush=True)
    return 0


def oracle_one_core(name, budget_s):
    """The oracle timed on ONE host core: a child process with one BLAS thread, pinned to one
    core (`oracle_probe`).  None when the child fails."""
    env = dict(os.environ, **ONE_THREAD_ENV)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-probe", name, "--cpu-budget", str(budget_s)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=30 + 6 * budget_s)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except (subprocess.SubprocessError, OSError, ValueError, IndexError):
        return None


# The configurations the metric is quoted on (one per problem statement item); the others are the
# "next" rows.  Their oracle is timed on all host cores and on one core beside the GPU number.
BASELINE_CONFIGS = ("single_head_m64_n100", "single_head_4096_f32", "single_head_4096_bf16", "gqa_causal_prefill",
                    "gqa_decode", "softmax_rows", "softmax_1d")


def compact(entry, oracle=None):
    """A suite entry as a short object: value, unit, ms per step (4 significant digits), and the
    roofline: its bound, peak and the achieved fraction of it, and the DRAM megabytes per launch
    from ncu (null when not captured for the current source); `oracle`: the oracle's throughput
    in the same unit, [on all host cores, on one core]."""
    rl = entry["roofline"]
    g4 = lambda x: None if x is None else float(f"{x:.4g}")
    out = {"v": g4(entry["value"]), "u": entry["unit"], "ms": g4(entry["ms_per_step"]), "bound": rl["bound"],
           "peak": rl["peak"], "frac": rl["frac"], "dram_mb": None if rl["traffic"] is None else g4(rl["traffic"] / 1e6)}
    if oracle:
        out["oracle"] = oracle
    return out


# Order of the suite in the result line: the configurations the metric is quoted on, and the
# backward, come last, where a reader of only the end of the output still finds them.
TAIL_FIRST = ("gqa_causal_backward",)


def suite_order(names):
    late = [n for n in TAIL_FIRST if n in names] + [n for n in BASELINE_CONFIGS if n in names]
    return [n for n in names if n not in late] + late


def headline_oracle(cpu):
    """[all host cores, one core] oracle throughput of the headline workload, or None."""
    if not cpu:
        return None
    one = cpu.get("one_core")
    return [float(f"{cpu['value']:.4g}"), float(f"{one['value']:.4g}") if one else None]


# ------------------------------------------------------------------------------ main
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(vals, world, device):
    """Element-wise maximum of per-rank values over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return [float(v) for v in vals]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(world, amount_per_rank, total_ms, steps):
    """Whole-job throughput: every rank processes `amount_per_rank` units per step (weak
    scaling), and a step lasts as long as the slowest rank's (already reduced) time."""
    mean_ms = total_ms / steps
    return world * amount_per_rank / (mean_ms / 1e3), mean_ms


def reference_arm(args, world, rank):
    w = WORKLOADS[args.workload]
    if rank != 0:
        return 0
    vals = []
    sample = cores = unit = None
    for _ in range(args.warmup):
        oracle_timed(args.workload, w, args.ref_budget / 4)
    for _ in range(args.steps):
        v, unit, sample, cores = oracle_timed(args.workload, w, args.ref_budget)
        vals.append(v)
    value = statistics.median(vals)
    amount, _, _ = work_units(w)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": amount / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w["desc"], "oracle": "fp64 numpy three-pass"},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": unit, "cores": cores,
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="osf", choices=["osf", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--no-suite", action="store_true", help="skip the other workloads")
    ap.add_argument("--suite-steps", type=int, default=50)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time (cpu_baseline)")
    ap.add_argument("--ref-budget", type=float, default=8.0, help="seconds per reference-arm step")
    ap.add_argument("--rows", type=int, default=0,
                    help="row count of a softmax workload instead of its own (a smaller case to profile)")
    ap.add_argument("--suite-oracle-budget", type=float, default=2.5,
                    help="seconds of oracle time per suite configuration (all cores, then one core)")
    ap.add_argument("--oracle-probe", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_probe:
        return oracle_probe(args.oracle_probe, args.cpu_budget)
    if args.rows:
        w0 = WORKLOADS[args.workload]
        if w0["kind"] != "softmax" or args.rows < 1:
            ap.error("--rows takes a positive count and applies to the softmax workloads only")
        WORKLOADS[args.workload] = dict(w0, rows=args.rows, desc=f"{w0['desc']} (rows set to {args.rows})")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    import online_softmax_flash_gb300 as osf
    from online_softmax_flash_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        dist.barrier()
        if rank != 0:
            _build.build()
        barrier = dist.barrier
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    osf.lib()
    pk, pk_src = peaks()
    flush = make_flush(dev)

    w = WORKLOADS[args.workload]
    # Before anything is timed the GPU runs the L2-flush kernels for ~0.3 s (the first workload
    # timed straight after the idle build and input generation read 3-8 % slow), and the suite
    # runs before the headline workload.
    t_warm = time.perf_counter()
    while time.perf_counter() - t_warm < 0.3:
        for _ in range(20):
            flush_l2(flush)
        torch.cuda.synchronize()
    suite = {}
    if not args.no_suite:
        for name, ww in WORKLOADS.items():
            if name == args.workload:
                continue
            r2 = measure(name, ww, osf, dev, args.suite_steps, 3, flush, barrier, None, e2e=False)
            m2 = statistics.mean(r2["ms"])
            suite[name] = {"workload": ww["desc"], "value": round(r2["amount"] / (m2 / 1e3), 3),
                           "unit": r2["unit"], "ms_per_step": round(m2, 5), "dtype": arith_dtype(ww),
                           "roofline": roofline(r2, pk, ww), "launches_per_call": r2["launches_per_call"],
                           "device_status": r2["status"]}

    sampler = make_sampler(local)
    sampler.start()
    res = measure(args.workload, w, osf, dev, args.steps, args.warmup, flush, barrier, sampler)
    sampler.stop()
    total_ms, e2e_ms = max_over_ranks([sum(res["ms"]), statistics.mean(res["e2e_ms"])], world, dev)
    value, mean_ms = job_rate(world, res["amount"], total_ms, args.steps)
    rl = roofline(res, pk, w)
    rl["peak_source"] = pk_src + (" burst" if rl["bound"] == "tensor" else "")

    cpu = None
    suite_oracle = {}
    if rank == 0:
        v, unit, sample, cores = oracle_timed(args.workload, w, args.cpu_budget)
        cpu = {"value": v, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}
        one = oracle_one_core(args.workload, args.cpu_budget)
        if one:
            one["full_workload_s"] = round(res["amount"] / one["value"], 1)   # one core, extrapolated
            cpu["one_core"] = one
        if not args.no_suite:
            for name in BASELINE_CONFIGS:
                if name not in suite:
                    continue
                a = oracle_timed(name, WORKLOADS[name], args.suite_oracle_budget)
                o = oracle_one_core(name, args.suite_oracle_budget)
                # [all host cores (cpu_baseline.cores of them), one core]
                suite_oracle[name] = [float(f"{a[0]:.4g}"), float(f"{o['value']:.4g}") if o else None]
        # the full suite entries, one line each, on stderr (stdout carries the one result line)
        for name, e in suite.items():
            print(json.dumps({"suite_entry": name, **e, "oracle": suite_oracle.get(name)}), file=sys.stderr,
                  flush=True)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": res["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": arith_dtype(w), "data": "synthetic",
            "config": {"workload": w["desc"], "l2": "flushed between timed steps (512 MiB write, then 256 MiB read)",
                       "gpu_warmup": "0.3 s of L2-flush kernels, then the suite, before the headline's warm-up steps",
                       "inputs": "seeded i.i.d. N(0,1) (SplitMix64 + Box-Muller), resident in HBM",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "roofline": rl, "cpu_baseline": cpu,
            "e2e": {"value": round(job_rate(world, res["amount"], e2e_ms, 1)[0], 3), "unit": res["unit"],
                    "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                    "ms_per_step": round(e2e_ms, 5), "call": res["e2e_call"]},
            "gpu_launches": res["launches"], "launches_per_step": res["launches_per_call"],
            "device_status": res["status"], "clocks": sampler.summary(),
            # last, and short, so that the end of the line holds every workload's number
            "suite": {n: compact(suite[n], suite_oracle.get(n)) for n in suite_order(list(suite))},
            # the headline again in the suite's short form, at the very end
            "headline": {args.workload: compact({"value": value, "unit": res["unit"], "ms_per_step": mean_ms,
                                                 "roofline": rl}, headline_oracle(cpu))},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
