"""Benchmark of the KDA forward prefill on GB300.

Workload: B=8, T=4096, H=32, K=V=128, bf16 q/k/v/g/beta, fp32 state (zero initial
state passed explicitly, final state written), lower_bound=-5, scale=1/sqrt(128),
seeded synthetic inputs (see kimi_delta_attention_08_gb300/synth.py).  One step is
one kda_fwd over the whole batch.

Reported (one JSON line on rank 0):
  value        tokens/s with inputs resident in HBM (CUDA events, max over ranks)
  e2e          same metric through the public API with host (pinned) buffers:
               H2D of the step's inputs + kda_fwd + D2H of the output, every step,
               pipelined across steps with two device buffer sets
  roofline     algorithmic bytes per launch / measured launch time vs the measured
               HBM copy bandwidth
  cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload
  clocks       nvidia-smi samples taken during the timed region
Multi-GPU: --gpus N runs N ranks, one per GPU (started here through
torch.distributed.run unless the launcher already set WORLD_SIZE); every rank
runs its own batch (independent (sequence, head) units, no collective): weak
scaling.

--impl reference times the CPU oracle as the reference arm (rank 0 only).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, T, H, KD = 8, 4096, 32, 128
BYTES_PER_TOKEN_HEAD = 4 * KD * 2 + 2 + KD * 2  # q,k,v,g + beta + out = 1282
METRIC = "KDA fwd prefill tokens/s & % roofline (bf16 TC/HBM), B=8 T=4096 H=32"
FLOP_PER_TOKEN_HEAD = 6 * KD * KD + 4 * 16 * KD + 2 * 16 * KD + 16 * 16 // 3  # stated count, C=16


def algorithmic_bytes(b=None, t=None, h=None, init=True, final=True, state_bytes=4):
    b, t, h = (B if b is None else b), (T if t is None else t), (H if h is None else h)
    n = b * t * h * BYTES_PER_TOKEN_HEAD
    n += b * h * KD * KD * state_bytes * (int(init) + int(final))
    n += h * 4 + h * KD * 4
    return n


KERNEL_SRC = os.path.join(ROOT, "kimi_delta_attention_08_gb300", "csrc", "kda_chunk_fwd.cu")
# the forward kernel's sources, hashed in order for its ncu records
FWD_SRCS = (KERNEL_SRC, os.path.join(ROOT, "kimi_delta_attention_08_gb300", "csrc", "kda_inverse.cuh"))
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "kda_chunk_fwd_B8_T1024_H32.json")
TRAFFIC_PROFILE_GVA = os.path.join(ROOT, "profiles", "kda_chunk_fwd_g32_B8_T1024_H16_HV32.json")
BWD_SRCS = tuple(os.path.join(ROOT, "kimi_delta_attention_08_gb300", "csrc", f)
                 for f in ("kda_bwd.cu", "kda_internal.h"))
TRAFFIC_PROFILE_BWD = os.path.join(ROOT, "profiles", "kda_bwd_B8_T1024_H32.json")
BWD_CHUNK_SRCS = tuple(os.path.join(ROOT, "kimi_delta_attention_08_gb300", "csrc", f)
                       for f in ("kda_bwd_chunk.cu", "kda_inverse.cuh", "kda_internal.h", "kda_ptx.cuh"))
TRAFFIC_PROFILE_BWD_CHUNK = os.path.join(ROOT, "profiles", "kda_bwd_chunk_B8_T1024_H32.json")


def source_sha256(srcs):
    import hashlib
    h = hashlib.sha256()
    for src in srcs:
        with open(src, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(abytes_full, profile=TRAFFIC_PROFILE, srcs=FWD_SRCS):
    """DRAM bytes (read + write) per launch of a kernel from the JSON record beside
    its committed ncu summary, scaled from the profiled case to this workload by
    algorithmic bytes; None when the kernel's sources (srcs, hashed in order)
    changed since the capture."""
    if not os.path.exists(profile):
        return None, "no ncu record"
    with open(profile) as f:
        fields = json.load(f)
    if fields.get("kernel_source_sha256") != source_sha256(srcs):
        return None, "kernel changed since the ncu capture"
    try:
        dram = float(fields["dram_bytes_per_launch"])
        small = float(fields["algorithmic_bytes_per_launch"])
    except (KeyError, ValueError, TypeError):
        return None, "ncu record incomplete"
    return dram * abytes_full / small, (f"ncu dram read+write {dram:.4g} B per launch at "
                                        f"{fields.get('workload', '?')}, scaled by algorithmic "
                                        f"bytes x{abytes_full / small:.3f}")


# fp32 FLOP of the backward per (token, head): per state element (128 x 128), one
# recomputed forward step (alpha S: 1, d = S'^T k: 2, S' + k u^T: 2) and the reverse
# step (alpha S_{t-1}: 1; d: 2; S_t: 2; S_t do: 2; dS += q do^T: 2; dS^T k: 2; dS u: 2;
# S' dd: 2; dS' = dS + k dd^T: 2; dS' o S_{t-1}: 2; alpha dS': 1).
BWD_FLOPS_PER_TOKEN_HEAD = (5 + 20) * KD * KD
# bf16 tensor-core FLOP the chunked backward issues per 64-token chunk of one head
# (M x N x K of each tcgen05.mma, x 2): the forward sweep's Gram, R, U and state
# update (3,670,016 MAC) and the reverse sweep's Gram pair, R, U, dU, U dS'^T,
# T^T dU, [dR~; dO] U^T, S [dO; -dR]^T, the dS update and the two pair products
# (15,204,352 MAC).  Issued, not minimal: some stacks compute unused halves.
BWD_CHUNK_FLOPS_PER_TOKEN_HEAD = 2 * (3_670_016 + 15_204_352) // 64
SMS, FP32_LANES_PER_SM = 152, 128


def fp32_peak_tflops():
    """Plain fp32 FMA peak: SMs x fp32 lanes per SM x 2 FLOP x the maximum SM clock
    (the measured record's, else the GB300's nominal 2070 MHz)."""
    mhz, src = 2070.0, "nominal 2070 MHz"
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "sm_max_mhz" in d:
            mhz, src = float(d["sm_max_mhz"]), f"measured sm_max_mhz {d['sm_max_mhz']:g}"
    return SMS * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, \
        f"{SMS} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2 FLOP x {src}"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class NvmlClocks:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM clock,
    its maximum, and the active clock-event reasons of one GPU."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.h)):
            raise OSError("no NVML handle")
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def sm_mhz(self):
        v = self.ct.c_uint(0)
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(v)) == 0 else None

    def sm_max_mhz(self):
        v = self.ct.c_uint(0)
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(v)) == 0 \
            else None

    def reasons(self):
        v = self.ct.c_ulonglong(0)
        if self.reason_fn(self.h, self.ct.byref(v)) != 0:
            return set()
        return {nm for bit, nm in self.REASONS.items() if v.value & bit}

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event reasons sampled while the with-block runs: NVML
    polled every 2 ms from a thread, else nvidia-smi every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.nvml = None

    def __enter__(self):
        import threading
        self.nvml = None
        try:
            self.nvml = NvmlClocks(self.gpu)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.samples, self.reasons, self.stop = [], set(), threading.Event()

            def poll():
                while not self.stop.is_set():
                    c = self.nvml.sm_mhz()
                    if c is not None:
                        self.samples.append(float(c))
                    self.reasons |= self.nvml.reasons()
                    time.sleep(0.002)

            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            return self
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join()
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.nvml is not None:
            smax = self.nvml.sm_max_mhz()
            self.nvml.close()
            return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                    "sm_max_mhz": float(smax) if smax else None, "samples": len(self.samples),
                    "source": "NVML every 2 ms during the timed loop",
                    "reasons": sorted(self.reasons)}
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


def timed_calls(fn, steps, warmup, gpu_index=0):
    """At least 3 untimed calls, then `steps` calls between CUDA events on the
    current stream, with the SM clock and its event reasons sampled while they
    run.  Returns (milliseconds per call, clock record)."""
    import torch
    for _ in range(max(warmup, 3)):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, clk.summary()


def cpu_baseline(target_s=12.0):
    """fp64 oracle on a bounded sample: whole (sequence, head) units of the
    workload (T tokens each), repeated until about target_s seconds of wall time."""
    import oracle
    from kimi_delta_attention_08_gb300 import synth
    cores = os.cpu_count() or 1
    units = 4 * cores  # heads of one T-token sequence per oracle call
    w = synth.make("cpu_sample", 1, T, units, init="zero", seed=2)
    Tn = w.tensors

    def once():
        return oracle.fwd(Tn["q"], Tn["k"], Tn["v"], Tn["g"], Tn["beta"], Tn["A_log"],
                          Tn["dt_bias"], -5.0, 1 / math.sqrt(128), Tn["initial_state"],
                          nthreads=cores)[2]

    dt, reps, used = 0.0, 0, cores
    while dt < target_s and reps < 1000:
        t0 = time.perf_counter()
        used = once()
        dt += time.perf_counter() - t0
        reps += 1
    token_heads = reps * T * units
    tokens_per_s = token_heads / H / dt  # workload tokens carry H heads each
    return {"value": tokens_per_s, "unit": "tokens/s", "cores": int(used), "kind": "oracle",
            "sample": f"{reps} x ({units} heads x {T} tokens) = {token_heads} token-heads, "
                      f"{dt:.1f} s wall, fp64 token recurrence; tokens/s = token-heads/s / {H}"}


def cpu_baseline_bwd(Tt, Hh, target_s=10.0):
    """fp64 oracle backward on a bounded sample: whole (sequence, head) units of Tt
    tokens (2 x cores heads per oracle call), repeated until about target_s seconds
    of wall time; tokens/s counts Hh heads per token like the GPU line."""
    import oracle
    from kimi_delta_attention_08_gb300 import synth
    cores = os.cpu_count() or 1
    units = 2 * cores
    w = synth.make("cpu_sample_bwd", 1, Tt, units, init="randn", seed=3)
    Tn = w.tensors
    dout = synth.normal_bf16((1, Tt, units, KD), 3, 9)
    dfin = synth.normal_f32((1, units, KD, KD), 3, 10)
    dt, reps = 0.0, 0
    while dt < target_s and reps < 1000:
        t0 = time.perf_counter()
        oracle.bwd(Tn["q"], Tn["k"], Tn["v"], Tn["g"], Tn["beta"], Tn["A_log"], Tn["dt_bias"],
                   -5.0, 1 / math.sqrt(128), dout, Tn["initial_state"], dfin, nthreads=cores)
        dt += time.perf_counter() - t0
        reps += 1
    token_heads = reps * Tt * units
    return {"value": token_heads / Hh / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x ({units} heads x {Tt} tokens) = {token_heads} token-heads, "
                      f"{dt:.1f} s wall, fp64 reverse mode of the token recurrence; "
                      f"tokens/s = token-heads/s / {Hh}"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    steps_val = []
    info = None
    for _ in range(args.warmup):
        cpu_baseline(target_s=1.0)
    for _ in range(args.steps):
        info = cpu_baseline(target_s=6.0)
        steps_val.append(info["value"])
    v = statistics.median(steps_val)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            # each step times a bounded sample; this is the whole workload at that rate
            "ms_per_step": B * T / v * 1e3, "ms_per_step_note": "extrapolated from the sample",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(),
            "cpu_baseline": {"kind": "oracle", "cores": info["cores"], "sample": info["sample"],
                             "value": v, "unit": "tokens/s"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def host_overhead_us(dev, calls=200):
    """Host time per kda_fwd call, measured on the small B=1 T=64 H=2 problem so the GPU
    keeps up and the launch queue never blocks: through the Python binding (argument
    checks included) and through the C entry point with pre-built ctypes arguments."""
    import ctypes
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import _lib, synth
    w = synth.tiny_ref()
    Tn = w.tensors
    bf = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    d = {nm: bf(Tn[nm]) for nm in ("q", "k", "v", "g", "beta")}
    A_log = torch.from_numpy(Tn["A_log"]).to(dev)
    dt_bias = torch.from_numpy(Tn["dt_bias"]).to(dev)
    out = torch.empty_like(d["q"])
    fin = torch.empty((1, w.H, KD, KD), dtype=torch.float32, device=dev)
    ws = kda.make_workspace(w.B * w.T, w.H, dev)
    py = lambda: kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, A_log,
                             dt_bias, w.lower_bound, None, fin, None, ws)
    lib = _lib.load()
    opts = _lib.kda_options()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    sh = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    cargs = (P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), w.scale, P(out),
             P(A_log), P(dt_bias), w.lower_bound, None, P(fin), None, w.B, w.T, w.H, w.B, 0,
             P(ws), ws.numel(), ctypes.byref(opts), sh)
    c = lambda: lib.kda_fwd(*cargs)
    res = {}
    for name, f in (("c_abi_via_ctypes", c), ("python_binding", py)):
        for _ in range(20):
            f()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            f()
        res[name] = (time.perf_counter() - t0) / calls * 1e6
        torch.cuda.synchronize()
    res["workload"] = "B=1 T=64 H=2, wall clock per call, no synchronisation inside"
    return res


def workload_config():
    return {"workload": f"kda_prefill_B{B}_T{T}_H{H}", "B": B, "T": T, "H": H, "K": KD,
            "V": KD, "inputs": "bf16", "state": "fp32 zero initial state, final written",
            "lower_bound": -5.0, "scale": "1/sqrt(128)",
            "l2": "inputs (1.07 GB per step) larger than the 129 MB L2; no flush"}


def run_decode(args):
    """Decode steps on the token-by-token path: B sequences x T tokens (defaults
    256 x 1), H = 32, fp32 state read and written.  Bytes per (sequence, head):
    the state in and out (64 KB each) plus 1,282 B per token."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import build, synth
    build.build()
    Bd = args.B if args.B != B else 256
    Td = args.T if args.T != T else 1
    Hd = H
    dev = torch.device("cuda", 0)
    w = synth.make(f"decode_B{Bd}_T{Td}_H{Hd}", Bd, Td, Hd, init="randn", seed=5)
    Tn = w.tensors
    bf = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    d = {nm: bf(Tn[nm]) for nm in ("q", "k", "v", "g", "beta")}
    A_log = torch.from_numpy(Tn["A_log"]).to(dev)
    dt_bias = torch.from_numpy(Tn["dt_bias"]).to(dev)
    init = torch.from_numpy(Tn["initial_state"]).to(dev)
    fin = torch.empty_like(init)
    out = torch.empty_like(d["q"])
    ws = kda.make_workspace(Bd * Td, Hd, dev)

    def timed(path):
        f = lambda: kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, A_log,
                                dt_bias, w.lower_bound, init, fin, None, ws, path=path)
        return timed_calls(f, args.steps, args.warmup)

    ms, clocks = timed("recurrent")
    ms_chunked, _ = timed("chunked")
    st = kda.kda_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status: {kda.status_string(st)}")
    hbm, _, src = load_peaks()
    abytes = algorithmic_bytes(Bd, Td, Hd)
    achieved = abytes / (ms * 1e-3) / 1e9
    line = {"metric": f"KDA fwd decode tokens/s, B={Bd} T={Td} H={Hd}", "value": Bd * Td / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"kda_decode_B{Bd}_T{Td}_H{Hd}", "B": Bd, "T": Td, "H": Hd,
                       "state": "fp32 initial state read, final written", "path": "recurrent",
                       "l2": f"{abytes / 1e9:.2f} GB per step vs the 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None,
                         "kernel": "kda_recurrent_kernel",
                         "note": f"algorithmic bytes {abytes} per launch; peak = {src} HBM copy "
                                 f"bandwidth"},
            "clocks": clocks, "gpu_launches": args.steps,
            "chunked_path_ms_per_step": ms_chunked}
    print(json.dumps(line), flush=True)
    return 0


def gva_bytes(b, t, h, hv, g_bytes=4, state_bytes=4):
    """Algorithmic bytes of one grouped-head launch: q, k over the h key heads;
    v, g (g_bytes per element), beta and out over the hv value heads; the fp32
    state read and written per (sequence, value head); A_log and dt_bias."""
    per_tok = 2 * h * KD * 2 + hv * (KD * 2 + KD * g_bytes + 2 + KD * 2)
    return b * t * per_tok + 2 * b * hv * KD * KD * state_bytes + hv * 4 + hv * KD * 4


def run_gva(args):
    """Grouped value heads with an fp32 gate on the chunked path: B x T tokens
    (defaults 8 x 4096), H = 16 q/k heads, HV = 32 value heads."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import build, synth
    build.build()
    Bg, Tg, Hk, HV = args.B, args.T, 16, 32
    dev = torch.device("cuda", 0)
    w = synth.make(f"gva_B{Bg}_T{Tg}_H{Hk}_HV{HV}", Bg, Tg, Hk, HV=HV, g_dtype="fp32",
                   init="zero", seed=6)
    Tn = w.tensors
    bf = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    d = {nm: bf(Tn[nm]) for nm in ("q", "k", "v", "beta")}
    g = torch.from_numpy(Tn["g"]).to(dev)
    A_log = torch.from_numpy(Tn["A_log"]).to(dev)
    dt_bias = torch.from_numpy(Tn["dt_bias"]).to(dev)
    init = torch.from_numpy(Tn["initial_state"]).to(dev)
    fin = torch.empty_like(init)
    out = torch.empty_like(d["v"])
    ws = kda.make_workspace(Bg * Tg, HV, dev)
    f = lambda: kda.kda_fwd(d["q"], d["k"], d["v"], g, d["beta"], w.scale, out, A_log, dt_bias,
                            w.lower_bound, init, fin, None, ws)
    ms, clocks = timed_calls(f, args.steps, args.warmup)
    st = kda.kda_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status: {kda.status_string(st)}")
    hbm, _, src = load_peaks()
    abytes = gva_bytes(Bg, Tg, Hk, HV)
    achieved = abytes / (ms * 1e-3) / 1e9
    traffic, traffic_note = measured_traffic(abytes, TRAFFIC_PROFILE_GVA)
    line = {"metric": f"KDA fwd prefill tokens/s, grouped value heads H={Hk} HV={HV}, fp32 gate",
            "value": Bg * Tg / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"kda_prefill_gva_B{Bg}_T{Tg}_H{Hk}_HV{HV}_g32", "B": Bg,
                       "T": Tg, "H": Hk, "HV": HV, "gate": "fp32",
                       "state": "fp32 zero initial state, final written", "path": "chunked",
                       "l2": f"{abytes / 1e9:.2f} GB per step vs the 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": traffic,
                         "traffic_note": traffic_note,
                         "kernel": "kda_chunk_fwd_kernel<fp32 gate>",
                         "note": f"algorithmic bytes {abytes} per launch; peak = {src} HBM copy "
                                 f"bandwidth"},
            "clocks": clocks, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)
    return 0


def run_bwd(args):
    """The backward pass (kda_bwd) on the prefill workload, B=8 T=4096 H=32, fp32
    states (initial state read, final-state gradient read, initial-state gradient
    written).  Algorithmic bytes per token-head: q, k, v, g, beta and dout read
    (1,282 B) and the fp32 gradients of q, k, v, g and beta written (2,052 B); per
    unit three fp32 states.  Checkpoint and scratch traffic is not counted.
    Default path: the chunked tensor-core kernel, reported against the HBM roofline
    (its tensor-core share is in the note); --bwd-path recurrent times the
    token-by-token fp32 kernel against the fp32 FMA peak."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import build, synth
    build.build()
    dev = torch.device("cuda", 0)
    w = synth.prefill(B=args.B, T=args.T)
    Tn = w.tensors
    bf = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    d = {nm: bf(Tn[nm]) for nm in ("q", "k", "v", "g", "beta")}
    A_log = torch.from_numpy(Tn["A_log"]).to(dev)
    dt_bias = torch.from_numpy(Tn["dt_bias"]).to(dev)
    init = torch.from_numpy(Tn["initial_state"]).to(dev)
    dout = bf(synth.normal_bf16(tuple(d["v"].shape), 7, 9))
    dfin = torch.from_numpy(synth.normal_f32(tuple(init.shape), 7, 10)).to(dev)
    ws = kda.make_bwd_workspace(w.B * w.T, w.N, w.H, 0, dev)
    path = args.bwd_path
    f = lambda: kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, A_log, dt_bias,
                            w.lower_bound, dout, init, dfin, None, ws, path=path)
    ms, clocks = timed_calls(f, args.steps, args.warmup)
    st = kda.kda_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status: {kda.status_string(st)}")
    th = w.B * w.T * w.H
    abytes = th * (BYTES_PER_TOKEN_HEAD + 4 * KD * 4 + 4) + 3 * w.B * w.H * KD * KD * 4 \
        + 2 * (w.H * 4 + w.H * KD * 4)
    hbm, tc_peak, src = load_peaks()
    hbm_achieved = abytes / (ms * 1e-3) / 1e9
    chunked = path != "recurrent"
    line = {"metric": f"KDA bwd tokens/s, B={w.B} T={w.T} H={w.H}",
            "value": w.B * w.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16" if chunked else "f32",
            "data": "synthetic",
            "config": {"workload": f"kda_bwd_B{w.B}_T{w.T}_H{w.H}", "B": w.B, "T": w.T,
                       "H": w.H, "gradients": "fp32", "state": "fp32",
                       "path": "chunked, tensor cores (bf16 operands, fp32 accumulation)"
                               if chunked else "token by token, fp32",
                       "l2": f"{abytes / 1e9:.2f} GB per step vs the 129 MB L2; no flush"},
            "clocks": clocks, "gpu_launches": 2 * args.steps}
    if chunked:
        traffic, traffic_note = measured_traffic(abytes, TRAFFIC_PROFILE_BWD_CHUNK, BWD_CHUNK_SRCS)
        tflops = th * BWD_CHUNK_FLOPS_PER_TOKEN_HEAD / (ms * 1e-3) / 1e12
        line["roofline"] = {
            "bound": "hbm", "achieved": hbm_achieved, "peak": hbm, "unit": "GB/s",
            "frac": hbm_achieved / hbm, "traffic": traffic, "kernel": "kda_bwd_chunk_kernel",
            "note": f"algorithmic bytes {abytes} per step ({src} copy bandwidth); tensor: "
                    f"{BWD_CHUNK_FLOPS_PER_TOKEN_HEAD} issued bf16 FLOP per token-head, "
                    f"{tflops:.1f} TFLOP/s = {tflops / tc_peak:.4f} of the {src} bf16 peak; "
                    f"traffic: {traffic_note}"}
    else:
        traffic, traffic_note = measured_traffic(abytes, TRAFFIC_PROFILE_BWD, BWD_SRCS)
        flops = th * BWD_FLOPS_PER_TOKEN_HEAD
        alu_peak, alu_src = fp32_peak_tflops()
        achieved = flops / (ms * 1e-3) / 1e12
        line["roofline"] = {
            "bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s",
            "frac": achieved / alu_peak, "traffic": traffic, "kernel": "kda_bwd_kernel",
            "note": f"fp32 FLOP per step {flops:.4g} (one recomputed forward step and one "
                    f"reverse step per state element per token-head); peak = {alu_src}; "
                    f"HBM: algorithmic bytes {abytes} per step, {hbm_achieved:.1f} GB/s = "
                    f"{hbm_achieved / hbm:.4f} of the {src} copy bandwidth; traffic: {traffic_note}"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(w.T, w.H)
    print(json.dumps(line), flush=True)
    return 0


def run_train(args):
    """One training step's KDA work on the prefill workload (B=8 T=4096 H=32, fp32
    states): kda_fwd writes out, the final state and every chunk's start state
    (kda_options.chunk_states); kda_bwd then reads those states instead of running
    its own state-checkpoint forward.  The same step with the backward's own pass is
    timed beside it.  Algorithmic bytes: the forward's (inputs, out, two states)
    plus the backward's (inputs, dout, fp32 gradients, three states)."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import build, synth
    build.build()
    dev = torch.device("cuda", 0)
    w = synth.prefill(B=args.B, T=args.T)
    Tn = w.tensors
    bf = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    d = {nm: bf(Tn[nm]) for nm in ("q", "k", "v", "g", "beta")}
    A_log = torch.from_numpy(Tn["A_log"]).to(dev)
    dt_bias = torch.from_numpy(Tn["dt_bias"]).to(dev)
    init = torch.from_numpy(Tn["initial_state"]).to(dev)
    fin = torch.empty_like(init)
    out = torch.empty_like(d["v"])
    dout = bf(synth.normal_bf16(tuple(d["v"].shape), 7, 9))
    dfin = torch.from_numpy(synth.normal_f32(tuple(init.shape), 7, 10)).to(dev)
    fws = kda.make_workspace(w.B * w.T, w.H, dev)
    bws = kda.make_bwd_workspace(w.B * w.T, w.N, w.H, 0, dev)
    cs = kda.make_chunk_states(w.B * w.T, w.N, w.H, dev)

    def step(reuse):
        kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, A_log, dt_bias,
                    w.lower_bound, init, fin, None, fws, chunk_states=cs if reuse else None)
        kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, A_log, dt_bias,
                    w.lower_bound, dout, init, dfin, None, bws, chunk_states=cs if reuse else None)

    ms, clocks = timed_calls(lambda: step(True), args.steps, args.warmup)
    ms_own, _ = timed_calls(lambda: step(False), args.steps, args.warmup)
    for ws in (fws, bws):
        st = kda.kda_get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status: {kda.status_string(st)}")
    th = w.B * w.T * w.H
    states = w.B * w.H * KD * KD * 4
    abytes = (th * BYTES_PER_TOKEN_HEAD + 2 * states) + \
        (th * (BYTES_PER_TOKEN_HEAD + 4 * KD * 4 + 4) + 3 * states) + 4 * (w.H * 4 + w.H * KD * 4)
    hbm, _, src = load_peaks()
    achieved = abytes / (ms * 1e-3) / 1e9
    line = {"metric": f"KDA fwd+bwd tokens/s, B={w.B} T={w.T} H={w.H}",
            "value": w.B * w.T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"kda_train_step_B{w.B}_T{w.T}_H{w.H}", "B": w.B, "T": w.T,
                       "H": w.H, "gradients": "fp32", "state": "fp32",
                       "step": "kda_fwd writing chunk states, then kda_bwd reading them",
                       "l2": f"{abytes / 1e9:.2f} GB per step vs the 129 MB L2; no flush"},
            "ms_per_step_backward_own_states": ms_own,
            "clocks": clocks, "gpu_launches": 3 * args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None,
                         "kernel": "kda_bwd_chunk_kernel",
                         "note": f"algorithmic bytes {abytes} per step over the whole step "
                                 f"({src} copy bandwidth); the kernels' own ncu figures are "
                                 "in the prefill and bwd lines"}}
    print(json.dumps(line), flush=True)
    return 0


def run_varlen(args, which):
    """The varlen schedule and the segment scan on their two workloads, chunked path:
    irregular varlen (H = 16, eight sequences of 1 .. 65,537 tokens, bf16 states) and
    one long sequence (H = 8, 65,536 + 5 x 1,024 tokens, fp32 states).  Times the
    default plan (segment scan AUTO) and, beside it, the plan without splits (OFF)."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import build, synth
    build.build()
    dev = torch.device("cuda", 0)
    w = synth.irregular_varlen() if which == "varlen" else synth.long_sequence()
    Tn = w.tensors
    bf = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    d = {nm: bf(Tn[nm]) for nm in ("q", "k", "v", "g", "beta")}
    A_log = torch.from_numpy(Tn["A_log"]).to(dev)
    dt_bias = torch.from_numpy(Tn["dt_bias"]).to(dev)
    init = Tn["initial_state"]
    init = (bf(init) if w.state_dtype == "bf16" else torch.from_numpy(init).to(dev))
    fin = torch.empty_like(init)
    out = torch.empty_like(d["q"])
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    ws = kda.make_workspace(w.total_tokens, w.H, dev)

    def timed(cp_mode):
        f = lambda: kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, A_log,
                                dt_bias, w.lower_bound, init, fin, cu, ws, cp_mode=cp_mode)
        r = timed_calls(f, args.steps, args.warmup)
        st = kda.kda_get_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status: {kda.status_string(st)}")
        return r

    ms, clocks = timed("auto")
    ms_off, _ = timed("off")
    sb = 2 if w.state_dtype == "bf16" else 4
    abytes = (w.total_tokens * w.H * BYTES_PER_TOKEN_HEAD + 2 * w.N * w.H * KD * KD * sb
              + w.H * 4 + w.H * KD * 4)
    hbm, _, src = load_peaks()
    achieved = abytes / (ms * 1e-3) / 1e9
    name = ("irregular_varlen_H16_N8" if which == "varlen" else "long_sequence_H8")
    line = {"metric": f"KDA fwd varlen tokens/s, {name}", "value": w.total_tokens / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": name, "H": w.H, "lengths": w.lengths,
                       "state": f"{w.state_dtype} initial state read, final written",
                       "path": "chunked", "cp_mode": "auto",
                       "l2": f"{abytes / 1e9:.2f} GB per step vs the 129 MB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None,
                         "kernel": "kda_plan_kernel + kda_chunk_fwd_kernel (+ merge)",
                         "note": f"algorithmic bytes {abytes} per step; peak = {src} HBM copy "
                                 f"bandwidth"},
            "clocks": clocks, "cp_off_ms_per_step": ms_off}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-host-overhead", action="store_true",
                    help="skip the host-time-per-call measurement (for profiler launch lists)")
    ap.add_argument("--B", type=int, default=B, help="batch override (profiling runs only)")
    ap.add_argument("--T", type=int, default=T, help="sequence length override (profiling)")
    ap.add_argument("--workload", default="prefill",
                    choices=["prefill", "decode", "gva", "varlen", "longseq", "bwd", "train"],
                    help="decode: the token-by-token path's line instead; gva: grouped "
                         "value heads (H=16, HV=32) with an fp32 gate; varlen / longseq: the "
                         "varlen schedule and segment scan workloads; bwd: the backward pass; "
                         "train: forward writing chunk states, then the backward reading them")
    ap.add_argument("--bwd-path", default="auto", choices=["auto", "chunked", "recurrent"],
                    help="backward workload: the chunked tensor-core kernel (auto) or the "
                         "token-by-token fp32 kernel")
    args = ap.parse_args()
    if args.workload == "decode":
        return run_decode(args)
    if args.workload == "gva":
        return run_gva(args)
    if args.workload in ("varlen", "longseq"):
        return run_varlen(args, args.workload)
    if args.workload == "bwd":
        return run_bwd(args)
    if args.workload == "train":
        return run_train(args)
    globals()["B"], globals()["T"] = args.B, args.T
    if args.impl == "reference":
        return run_reference(args)

    from kimi_delta_attention_08_gb300 import ranks
    rank, world, local = ranks.world_info()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not launched per rank: start one process per GPU and wait for them
        return ranks.spawn_world(args.gpus, [os.path.abspath(__file__)] + sys.argv[1:])
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {world}", file=sys.stderr)
        return 2

    import numpy as np
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import kimi_delta_attention_08_gb300 as kda
    from kimi_delta_attention_08_gb300 import build, synth
    build.build()

    def to_torch_f32(x, device):
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)

    w = synth.prefill(B=B, T=T, H=H, seed=ranks.rank_seed(2, rank))  # own batch per rank
    Tn = w.tensors
    # pinned host copies (for e2e) and device-resident copies (for value)
    host = {nm: torch.from_numpy(Tn[nm].view(np.int16)).view(torch.bfloat16).pin_memory()
            for nm in ("q", "k", "v", "g", "beta")}
    d = {nm: host[nm].to(dev) for nm in host}
    A_log = to_torch_f32(Tn["A_log"], dev)
    dt_bias = to_torch_f32(Tn["dt_bias"], dev)
    init_h = torch.from_numpy(Tn["initial_state"]).pin_memory()
    init = init_h.to(dev)
    out = torch.empty_like(d["q"])
    fin = torch.empty_like(init)
    ws = kda.make_workspace(B * T, H, dev)
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(128.0)

    def step(dd, o, ini, fi):
        kda.kda_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], scale, o, A_log, dt_bias,
                    -5.0, ini, fi, None, ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step(d, out, init, fin)
    torch.cuda.synchronize(dev)
    st = kda.kda_get_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {kda.status_string(st)}")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing, per-launch events on the launching stream
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            evs[i][0].record(stream)
            step(d, out, init, fin)
            evs[i][1].record(stream)
        t_all1.record(stream)
        barrier()
    clocks = clk.summary()
    total_ms = t_all0.elapsed_time(t_all1)
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    ms = ranks.max_over_ranks(total_ms / args.steps, dist, dev)
    value = ranks.aggregate_tokens_per_s(B * T, world, ms)

    # ---- end to end through the API with host buffers
    e2e = None
    if not args.no_e2e:
        # Two device buffer sets: step i+1's host->device copies (one copy stream)
        # overlap step i's kernel and its device->host read (another copy stream);
        # every step's copies are inside the timed region.
        out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        fin_h = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(2)]
        sets = [({nm: torch.empty_like(d[nm]) for nm in d}, torch.empty_like(init),
                 torch.empty_like(out), torch.empty_like(fin)) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]   # inputs of set j are on the device
        ev_k = [torch.cuda.Event() for _ in range(2)]    # the kernel on set j has finished
        ev_out = [torch.cuda.Event() for _ in range(2)]  # set j's output has been read back
        h2d = sum(host[nm].numel() * host[nm].element_size() for nm in host) + \
            init_h.numel() * init_h.element_size()
        d2h = out.numel() * out.element_size() + fin.numel() * fin.element_size()

        def e2e_step(i):
            j = i & 1
            dd, ini2, o2, f2 = sets[j]
            s_in.wait_event(ev_k[j])
            with torch.cuda.stream(s_in):
                for nm in dd:
                    dd[nm].copy_(host[nm], non_blocking=True)
                ini2.copy_(init_h, non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])
            step(dd, o2, ini2, f2)
            ev_k[j].record(stream)
            s_out.wait_event(ev_k[j])
            with torch.cuda.stream(s_out):
                out_h[j].copy_(o2, non_blocking=True)
                fin_h[j].copy_(f2, non_blocking=True)
            ev_out[j].record(s_out)

        for i in range(2):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        e1.record(s_out)
        barrier()
        ems = ranks.max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, dev)
        e2e = {"value": ranks.aggregate_tokens_per_s(B * T, world, ems), "unit": "tokens/s",
               "ms_per_step": ems, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "pinned host buffers; every step copies its inputs and initial state "
                       "in and its output and final state out; H2D of step i+1 overlaps kernel "
                       "+ D2H of step i (two device buffer sets, each with its own output and "
                       "final state)"}

    hbm, tc, src = load_peaks()
    launch_avg = statistics.mean(launch_ms)
    abytes = algorithmic_bytes()
    achieved = abytes / (launch_avg * 1e-3) / 1e9
    flops = B * T * H * FLOP_PER_TOKEN_HEAD
    traffic, traffic_note = measured_traffic(abytes)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "traffic_note": traffic_note,
                "kernel": "kda_chunk_fwd_kernel",
                "note": f"algorithmic bytes {abytes} per launch (1282 B per token-head + fp32 "
                        f"state in/out) over the CUDA-event launch time {launch_avg*1e3:.1f} us; "
                        f"peak = {src} HBM copy bandwidth; tensor side: "
                        f"{flops/(launch_avg*1e-3)/1e12:.1f} TFLOP/s of {tc:.0f} ({src}) at "
                        f"{FLOP_PER_TOKEN_HEAD} FLOP per token-head"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    host_us = host_overhead_us(dev) if rank == 0 and not args.no_host_overhead else None
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic", "config": workload_config(),
                "e2e": e2e, "gpu_launches": args.steps * 1, "roofline": roofline,
                "cpu_baseline": cpu, "clocks": clocks, "host_us_per_call": host_us,
                "launch_us": {"mean": launch_avg * 1e3, "min": min(launch_ms) * 1e3,
                              "max": max(launch_ms) * 1e3}}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
