"""Benchmark of the block-scaled fp8 GEMM path on one GB300.

Headline workload: the weight-only fp8 decode GEMM, M=16, N=K=4096 (bf16
activations ~N(0,1) used unquantised, e4m3 weights from N(0,0.02) with one fp32
scale per 128x128 block, fp32 accumulate, bf16 out, seed 1).  One step = one
call of r9q_gemm_fp8w_bf16a.  value = achieved HBM GB/s (algorithmic bytes per
call / time per call); ms_per_step gives the us/call.

Timing: every step reads its own copy of weights and activations, rotating
over enough copies (> 3x the 129 MB L2) that each call streams from HBM; K
calls are captured in CUDA graphs and replayed; CUDA events on the replay
stream bracket exactly K steps, with a device synchronise on both sides.  SM
clocks and throttle reasons are sampled through NVML (read-only) during the
timed region.  A sweep over the other configurations follows the headline.

--impl reference times the CPU oracle (test infrastructure, plain C, single
thread) on whole calls of the same workload and prints the same JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
SPIN_CYCLES = 400_000          # ~0.2 ms at 2 GHz
FALLBACK_HBM = 6800.0
FALLBACK_BF16 = 1900.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", FALLBACK_HBM), d.get("bf16_tflops", FALLBACK_BF16), "measured"
    return FALLBACK_HBM, FALLBACK_BF16, "fallback"


def gemm_bytes(M, N, K):
    """Algorithmic bytes per call: e4m3 W + fp32 block scales + bf16 A in + bf16 Y out."""
    return N * K + 4 * (N // 128) * (K // 128) + 2 * M * K + 2 * M * N


def mlp_bytes(M, H, I, Ho):
    return gemm_bytes(M, 2 * I, H) - 2 * M * 2 * I + 2 * M * I + gemm_bytes(M, Ho, I) - 2 * M * I + 2 * M * I


# ------------------------------------------------ captured DRAM traffic --

# The sources each timed kernel is built from; a capture under profiles/ only
# describes the kernel while these files are unchanged.
KERNEL_SOURCES = {
    "stream_sync_kernel": ["r9q_api.cu", "r9q_device.cuh", "r9q_kernels.h", "r9q_stream_common.cuh",
                           "r9q_stream_sync.cuh", "r9q_stream_launch.cuh", "r9q_stream_bf16.cu"],
    "stream_gemm_kernel": ["r9q_api.cu", "r9q_device.cuh", "r9q_kernels.h", "r9q_stream_common.cuh",
                           "r9q_stream.cuh", "r9q_stream_launch.cuh", "r9q_stream_quant.cu"],
    "tc_gemm_kernel": ["r9q_api.cu", "r9q_device.cuh", "r9q_kernels.h", "r9q_tc.cu"],
}


def sources_hash(kernel):
    import hashlib
    d = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        rel = "block_scaled_fp8_x128_gb300/csrc/" + f
        d.update(rel.encode())
        with open(os.path.join(ROOT, rel), "rb") as fh:
            d.update(fh.read())
    return d.hexdigest()[:16]


def captured_traffic(profile, kernel):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch from the ncu
    summary profiles/<profile>, or None when the summary is missing or the
    kernel's sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- `") and "`: " in line:
                k, v = line[3:].split("`: ", 1)
                kv[k.strip()] = v.strip().strip("`")
    if kv.get("sources_sha256") != sources_hash(kernel):
        return None
    try:
        return int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------- NVML clocks --

class ClockSampler:
    """Samples SM clock and clock-event reasons with NVML through ctypes (reads only)."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index=0, period_s=0.002):
        self.ok = False
        self.samples = []
        self.reasons = 0
        self.period = period_s
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(mx))   # NVML_CLOCK_SM
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _one(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, ctypes.c_int(1), ctypes.byref(c))
        self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(r))
        return c.value, r.value

    def start(self):
        self.samples, self.reasons, self._stop = [], 0, False
        if not self.ok:
            return

        def run():
            while not self._stop:
                c, r = self._one()
                self.samples.append(c)
                self.reasons |= r
                time.sleep(self.period)
        self._t = threading.Thread(target=run, daemon=True)
        self._t.start()

    def stop(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        self._stop = True
        self._t.join()
        if not self.samples:
            self.samples.append(self._one()[0])
        names = [n for b, n in self.REASONS.items() if self.reasons & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(self.samples)}


# --------------------------------------------------------------- GPU arm --

def _make_inputs(torch, r9q, kind, M, N, K, seed, p, factor, copies, dev):
    import synth
    xb = synth.to_bf16_bits(synth.activations(seed, M, K, p, factor))
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    wq, ws = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(seed, N, K)).to(dev))
    W = [wq] + [wq.clone() for _ in range(copies - 1)]
    S = [ws] + [ws.clone() for _ in range(copies - 1)]
    X = [x] + [x.clone() for _ in range(copies - 1)]
    Y = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    return X, W, S, Y


def _copies_for(bytes_per_call):
    return max(2, math.ceil(3 * L2_BYTES / bytes_per_call))


def _graph(torch, fn, n_calls, copies, stream, begin=None, end=None):
    """One CUDA graph of n_calls steps; begin/end run inside the capture
    (fork side streams off the capture stream, join them back)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        if begin:
            begin()
        for i in range(n_calls):
            fn(i % copies)
        if end:
            end()
    return g


# Set by main() under torchrun: a barrier across ranks on both sides of every
# timed region.
_BARRIER = None


def _time_steps(torch, fn, K, copies, stream, sampler=None, begin=None, end=None):
    """Replay graphs covering exactly K calls; returns (ms_total)."""
    G = copies * max(1, 64 // copies)
    reps, rem = divmod(K, G)
    g_full = _graph(torch, fn, G, copies, stream, begin, end) if reps else None
    g_rem = _graph(torch, fn, rem, copies, stream, begin, end) if rem else None
    for g in (g_full, g_rem):      # upload and run once: the timed replays are warm
        if g:
            g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        torch.cuda.synchronize()
        if _BARRIER:
            _BARRIER()
        # a short device-side spin ahead of the start event keeps the stream
        # busy while the host submits the graph launches, so the timed region
        # holds the K steps' device work and not the host's submission latency
        torch.cuda._sleep(SPIN_CYCLES)
        e0.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_rem:
            g_rem.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if _BARRIER:
            _BARRIER()
    clocks = sampler.stop() if sampler else None
    return e0.elapsed_time(e1), clocks


def measure_fp8_peak(torch, stream, sampler=None):
    """Dense fp8 (e4m3) tensor throughput of the library-free reference point:
    torch._scaled_mm (cuBLASLt) at 8192^3, bf16 out, unit scales; ten timed
    batches of ten back-to-back GEMMs, best batch, clocks sampled meanwhile."""
    n = 8192
    try:
        gen = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn((n, n), device="cuda", generator=gen).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device="cuda", generator=gen).to(torch.float8_e4m3fn)
        one = torch.ones((), device="cuda", dtype=torch.float32)
        bt = b.t()                                  # column-major operand

        def mm():
            return torch._scaled_mm(a, bt, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        with torch.cuda.stream(stream):
            for _ in range(3):
                mm()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        best = float("inf")
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                torch.cuda._sleep(SPIN_CYCLES)
                e0.record(stream)
                for _ in range(10):
                    mm()
                e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 10)
        clocks = sampler.stop() if sampler else None
        del a, b, bt
        torch.cuda.empty_cache()
        return {"tflops": round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1), "ms_per_gemm": round(best, 4),
                "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3, best of 10 batches of 10", "clocks": clocks}
    except Exception as e:                     # no fp8 GEMM in this torch build
        return {"tflops": None, "error": f"{type(e).__name__}: {e}"[:200]}


def run_gpu(args):
    import torch
    import block_scaled_fp8_x128_gb300 as r9q
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm, bf16, src = peaks()
    fp8_nominal = 2.0 * bf16        # nominal fp8:bf16 dense ratio of 2 on the measured bf16 peak
    stream = torch.cuda.Stream()
    fp8_meas = measure_fp8_peak(torch, stream, ClockSampler(local)) if not args.no_sweep else None

    # ---- headline: weight-only decode GEMM, M=16, N=K=4096, seed 1 ----
    M, N, K_ = 16, 4096, 4096
    bpc = gemm_bytes(M, N, K_)
    copies = _copies_for(bpc)
    X, W, S, Y = _make_inputs(torch, r9q, "w8bf16", M, N, K_, 1, 0.0, 1.0, copies, dev)
    torch.cuda.synchronize()
    # decode-step launch mode: weights are constant, so each GEMM may start
    # streaming them while the previous call finishes (include/r9q.h, r9q_set_pdl)
    r9q.r9q_set_pdl(not args.no_pdl)

    def step(i):
        r9q.r9q_gemm_fp8w_bf16a(X[i], W[i], S[i], y=Y[i])

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i % copies)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    ms, clocks = _time_steps(torch, step, args.steps, copies, stream, sampler)
    us_call = ms * 1e3 / args.steps
    gbs = bpc / (us_call * 1e-6) / 1e9

    # ---- e2e: host (pinned) activations in, bf16 result out, through the same call ----
    h2d = M * K_ * 2
    d2h = M * N * 2
    us_e2e = float("nan")
    if not args.no_e2e:
        hx = [X[0].cpu().pin_memory() for _ in range(copies)]
        hy = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(copies)]
        # Copies run on their own streams, so a step's host-to-device copy
        # overlaps the previous step's GEMM and its result copy the next one's;
        # a buffer slot is rewritten only after its previous GEMM read it and
        # its previous result left it.  Every step's two copies are inside the
        # timed region.
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(copies)]
        ev_mm = [torch.cuda.Event() for _ in range(copies)]
        ev_out = [torch.cuda.Event() for _ in range(copies)]
        used = set()

        def e2e_begin():
            used.clear()
            cur = torch.cuda.current_stream()
            s_in.wait_stream(cur)
            s_out.wait_stream(cur)

        def e2e_end():
            cur = torch.cuda.current_stream()
            cur.wait_stream(s_in)
            cur.wait_stream(s_out)

        def e2e_step(i):
            cur = torch.cuda.current_stream()
            if i in used:
                s_in.wait_event(ev_mm[i])
                cur.wait_event(ev_out[i])
            used.add(i)
            with torch.cuda.stream(s_in):
                X[i].copy_(hx[i], non_blocking=True)
                ev_in[i].record(s_in)
            cur.wait_event(ev_in[i])
            r9q.r9q_gemm_fp8w_bf16a(X[i], W[i], S[i], y=Y[i])
            ev_mm[i].record(cur)
            s_out.wait_event(ev_mm[i])
            with torch.cuda.stream(s_out):
                hy[i].copy_(Y[i], non_blocking=True)
                ev_out[i].record(s_out)

        with torch.cuda.stream(stream):
            e2e_begin()
            for i in range(args.warmup):
                e2e_step(i % copies)
            e2e_end()
        torch.cuda.synchronize()
        ms_e2e, _ = _time_steps(torch, e2e_step, args.steps, copies, stream, begin=e2e_begin, end=e2e_end)
        us_e2e = ms_e2e * 1e3 / args.steps

    out = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": us_call / 1e3,
        "us_per_call": round(us_call, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 weights x bf16 activations, fp32 accumulate",
        "data": "synthetic (seeded splitmix64/Box-Muller: x~N(0,1) bf16, W~N(0,0.02) fp32 -> e4m3 + 128x128 fp32 scales)",
        "config": dict(HEADLINE),
        "timing": {"l2": f"inputs larger than L2: rotating {copies} weight/activation copies "
                         f"({copies * bpc / 1e6:.0f} MB > 129 MB L2)",
                   "how": "CUDA-graph replay of exactly K calls (graphs uploaded and run once before), "
                          "CUDA events on the replay stream behind a device-side spin",
                   "pdl": not args.no_pdl},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4),
                     "traffic": captured_traffic("stream_gemm_w8bf16_M16_N4096_K4096.md", "stream_sync_kernel"),
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback"},
        "e2e": {"value": None if args.no_e2e else round(bpc / (us_e2e * 1e-6) / 1e9, 1), "unit": "GB/s",
                "us_per_call": None if args.no_e2e else round(us_e2e, 3),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "per step: pinned-host activations -> device, r9q_gemm_fp8w_bf16a, bf16 result -> pinned host; "
                        "weights resident; the copies run on their own streams and overlap neighbouring steps' GEMMs"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    del X, W, S, Y
    torch.cuda.empty_cache()

    if not args.no_sweep:
        out["fp8_peak_measured"] = fp8_meas
        out["sweep"] = sweep(torch, r9q, stream, hbm, fp8_nominal, (fp8_meas or {}).get("tflops"), src)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    return out


def sweep(torch, r9q, stream, hbm, fp8_nominal, fp8_measured, src):
    res = []
    dev = torch.device("cuda", torch.cuda.current_device())

    def timeit(fn, copies, calls):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i % copies)
        torch.cuda.synchronize()
        ms, _ = _time_steps(torch, fn, calls, copies, stream)
        return ms * 1e3 / calls

    cases = [("c0", "w8a8", 1, 512, 1024, 0.01, 20.0, 0)]
    cases += [("c2", "w8a8", m, 12288, 4096, 0.005, 50.0, 2) for m in (1, 2, 4, 8, 16)]
    cases += [("c4", "w8a8", m, 4096, 4096, 0.0, 1.0, 4) for m in (32, 64, 128, 255, 8192)]
    for name, kind, M, N, K, p, fac, seed in cases:
        bpc = gemm_bytes(M, N, K)
        copies = min(_copies_for(bpc), 64)
        X, W, S, Y = _make_inputs(torch, r9q, kind, M, N, K, seed, p, fac, copies, dev)
        torch.cuda.synchronize()

        # one scratch for the case's calls (they run in stream order); zeroed once
        wsp = torch.zeros(max(r9q.r9q_workspace_bytes(r9q.R9Q_OP_GEMM_W8A8, M, N, K), 256), dtype=torch.uint8,
                          device=dev)

        def fn(i, wsp=wsp):
            r9q.r9q_gemm_fp8_block_qa(X[i], W[i], S[i], y=Y[i], workspace=wsp)
        calls = 2000 if M <= 255 else 20
        us = timeit(fn, copies, calls)
        flops = 2.0 * M * N * K
        row = {"config": name, "mode": "W8A8 fused quant", "M": M, "N": N, "K": K, "us_per_call": round(us, 3),
               "GBps": round(bpc / us / 1e3, 1), "frac_hbm": round(bpc / us / 1e3 / hbm, 4),
               "TFLOPS": round(flops / us / 1e6, 2),
               "frac_fp8_2x_bf16": round(flops / us / 1e6 / fp8_nominal, 4)}
        if fp8_measured:
            row["frac_fp8_measured"] = round(flops / us / 1e6 / fp8_measured, 4)
        res.append(row)
        del X, W, S, Y, wsp
        torch.cuda.empty_cache()

    # c3: fused expert MLP M=8, H=4096, I=1536, H_out=4096
    import synth
    M, H, I, Ho = 8, 4096, 1536, 4096
    bpc = mlp_bytes(M, H, I, Ho)
    copies = _copies_for(bpc)
    xb = synth.to_bf16_bits(synth.activations(3, M, H))
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    wgu, sgu = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(3, 2 * I, H, tensor=1)).to(dev))
    wdn, sdn = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(3, Ho, I, tensor=2)).to(dev))
    WG = [wgu.clone() for _ in range(copies)]
    WD = [wdn.clone() for _ in range(copies)]
    HB = [torch.empty((M, I), dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    YB = [torch.empty((M, Ho), dtype=torch.bfloat16, device=dev) for _ in range(copies)]
    torch.cuda.synchronize()
    for flags, label in ((0, "fused"), (r9q.R9Q_MLP_UNFUSED, "separate launches")):
        ws_b = r9q.r9q_workspace_bytes(r9q.R9Q_OP_GATE_UP_SWIGLU_DOWN, M, I, H, Ho, flags)
        wsp = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=dev)

        def fn(i, flags=flags, wsp=wsp):
            r9q.r9q_gate_up_swiglu_down(x, WG[i], sgu, WD[i], sdn, y=YB[i], h=HB[i], flags=flags, workspace=wsp)
        us = timeit(fn, copies, 2000)
        res.append({"config": "c3", "mode": f"expert MLP W8A8 ({label})", "M": M, "H": H, "I": I, "H_out": Ho,
                    "us_per_call": round(us, 3), "GBps": round(bpc / us / 1e3, 1),
                    "frac_hbm": round(bpc / us / 1e3 / hbm, 4)})
    del WG, WD, HB, YB
    torch.cuda.empty_cache()

    # A decode layer's GEMM sequence at M=8 (attention between them is out of
    # scope): QKV projection N=12288, output projection 4096x4096, then the
    # fused expert MLP on the projection's output; every layer reads its own
    # copy of all weights (copies > 3x L2).  Chained: programmatic dependent
    # launch on; serialised: off.  Both replay CUDA graphs of whole layers.
    Ml = 8
    xl = torch.from_numpy(synth.to_bf16_bits(synth.activations(50, Ml, H, 0.01, 20.0)).view(np.int16)).view(
        torch.bfloat16).to(dev)
    wq_, sq_ = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(51, 3 * H, H)).to(dev))
    wo_, so_ = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(52, H, H)).to(dev))
    bpl = gemm_bytes(Ml, 3 * H, H) + gemm_bytes(Ml, H, H) + mlp_bytes(Ml, H, I, H)
    copies_l = _copies_for(bpl)
    LW = [(wq_.clone(), wo_.clone(), wgu.clone(), wdn.clone()) for _ in range(copies_l)]
    qkv_b = torch.empty((Ml, 3 * H), dtype=torch.bfloat16, device=dev)
    o_b = torch.empty((Ml, H), dtype=torch.bfloat16, device=dev)
    y_b = torch.empty((Ml, H), dtype=torch.bfloat16, device=dev)
    mlp_ws = torch.empty(max(r9q.r9q_workspace_bytes(r9q.R9Q_OP_GATE_UP_SWIGLU_DOWN, Ml, I, H, H), 256),
                         dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def layer(i):
        a, b, c, d = LW[i]
        r9q.r9q_gemm_fp8_block_qa(xl, a, sq_, y=qkv_b)
        r9q.r9q_gemm_fp8_block_qa(xl, b, so_, y=o_b)
        r9q.r9q_gate_up_swiglu_down(o_b, c, sgu, d, sdn, y=y_b, workspace=mlp_ws)
    prev = r9q.r9q_set_pdl(True)
    us_chained = timeit(layer, copies_l, 500)
    r9q.r9q_set_pdl(False)
    us_serial = timeit(layer, copies_l, 500)
    r9q.r9q_set_pdl(prev)
    res.append({"config": "layer", "mode": "decode layer GEMMs at M=8 (QKV N=12288, O 4096x4096, expert MLP "
                "I=1536), 4 launches, W8A8 fused quant, CUDA graph", "M": Ml,
                "us_per_layer_chained_pdl": round(us_chained, 3), "us_per_layer_serialised": round(us_serial, 3),
                "GBps_chained": round(bpl / us_chained / 1e3, 1), "frac_hbm_chained": round(bpl / us_chained / 1e3 / hbm, 4),
                "bytes_per_layer": bpl})
    del LW
    torch.cuda.empty_cache()

    # MoE decode layer: E experts with T tokens each (the c3 expert shape), grouped
    # gate_up (SwiGLU epilogue) + grouped down (fused quant of h): two launches,
    # against E separate fused expert-MLP calls.  Every expert has its own weight
    # copy (same values), rotated over copies > 3x L2.
    E, T = 8, 8
    bpc_e = E * bpc
    copies_e = _copies_for(bpc_e)
    xe = torch.from_numpy(synth.to_bf16_bits(synth.activations(3, E * T, H)).view(np.int16)).view(torch.bfloat16).to(dev)
    GU = [torch.stack([wgu] * E).clone() for _ in range(copies_e)]
    DN = [torch.stack([wdn] * E).clone() for _ in range(copies_e)]
    SGU, SDN = torch.stack([sgu] * E), torch.stack([sdn] * E)
    he = torch.empty((E * T, I), dtype=torch.bfloat16, device=dev)
    ye = torch.empty((E * T, Ho), dtype=torch.bfloat16, device=dev)
    off = [T * e for e in range(E + 1)]
    torch.cuda.synchronize()

    def grouped(i):
        r9q.r9q_grouped_gemm_fp8(xe, off, GU[i], SGU, y=he, flags=r9q.R9Q_GROUPED_SWIGLU)
        r9q.r9q_grouped_gemm_fp8(he, off, DN[i], SDN, y=ye)

    def per_expert(i):
        for e in range(E):
            r9q.r9q_gate_up_swiglu_down(xe[T * e:T * (e + 1)], GU[i][e], sgu, DN[i][e], sdn,
                                        y=ye[T * e:T * (e + 1)], h=he[T * e:T * (e + 1)])
    for fn, label in ((grouped, "grouped, 2 launches"), (per_expert, f"{E} fused expert-MLP calls")):
        us = timeit(fn, copies_e, 500)
        res.append({"config": "moe", "mode": f"MoE decode layer W8A8, {E} experts x {T} tokens ({label})",
                    "E": E, "T": T, "H": H, "I": I, "H_out": Ho, "us_per_call": round(us, 3),
                    "GBps": round(bpc_e / us / 1e3, 1), "frac_hbm": round(bpc_e / us / 1e3 / hbm, 4)})
    return res


# ---------------------------------------------------------- CPU baseline --

HEADLINE = {"workload": "weight-only fp8 decode GEMM M=16 N=4096 K=4096 (seed 1)",
            "M": 16, "N": 4096, "K": 4096, "bytes_per_call": gemm_bytes(16, 4096, 4096)}
METRIC = "block-fp8 GEMM us/call & achieved HBM GB/s (M=1..16), fp8 TFLOPS (M=8192)"


def _oracle_call(oracle, synth, case, rows):
    """Build the inputs of one configuration and return a function that runs
    the oracle on the token rows `rows` of it (W8A8: quant + GEMM)."""
    name, kind, M, N, K, seed, p, fac = case
    xb = synth.to_bf16_bits(synth.activations(seed, M, K, p, fac))
    if kind == "mlp":
        I, Ho = N, K
        H = 4096
        xb = synth.to_bf16_bits(synth.activations(seed, M, H))
        wgu, sgu = oracle.quant_block128(synth.weights(seed, 2 * I, H, tensor=1))
        wdn, sdn = oracle.quant_block128(synth.weights(seed, Ho, I, tensor=2))
        return lambda: oracle.gate_up_swiglu_down(xb[rows], wgu, sgu, wdn, sdn)
    wq, ws = oracle.quant_block128(synth.weights(seed, N, K))
    if kind == "w8bf16":
        return lambda: oracle.gemm_w8bf16(xb, wq, ws, rows=rows)

    def w8a8():
        q, sc = oracle.quant_group(xb[rows])
        return oracle.gemm_w8a8(q, sc, wq, ws)
    return w8a8


# (name, kind, M, N, K, seed, outlier p, factor); the MLP row reads N = I, K = H_out
CPU_CASES = [("c0 W8A8 M=1 N=512 K=1024", "w8a8", 1, 512, 1024, 0, 0.01, 20.0),
             ("c1 weight-only M=16 N=4096 K=4096", "w8bf16", 16, 4096, 4096, 1, 0.0, 1.0),
             ("c2 W8A8 M=16 N=12288 K=4096", "w8a8", 16, 12288, 4096, 2, 0.005, 50.0),
             ("c3 expert MLP M=8 H=4096 I=1536 H_out=4096", "mlp", 8, 1536, 4096, 3, 0.0, 1.0),
             ("c4 W8A8 M=8192 N=4096 K=4096", "w8a8", 8192, 4096, 4096, 4, 0.0, 1.0)]


def _time_oracle(fn, budget_s, min_calls=1):
    calls, t0 = 0, time.perf_counter()
    while True:
        fn()
        calls += 1
        el = time.perf_counter() - t0
        if calls >= min_calls and el >= budget_s:
            return el / calls, calls


def cpu_baseline(budget_s=10.0):
    """The oracle (plain C, -O2) timed on the host cores.  Headline value: the
    single-threaded oracle as it stands on whole calls of the headline
    workload.  `configs`: every configuration, on a bounded sample of its
    token rows (scaled to a whole call by M / rows), single-threaded and with
    the OpenMP build of the same source on all cores."""
    import oracle
    import synth
    case = CPU_CASES[1]
    run = _oracle_call(oracle, synth, case, np.arange(16))
    per, calls = _time_oracle(run, budget_s)
    us = per * 1e6
    res = {"value": round(HEADLINE["bytes_per_call"] / us / 1e3, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "us_per_call": round(us, 1),
           "sample": f"{calls} whole M=16 N=4096 K=4096 weight-only calls of the C oracle, 1 thread"}
    table = []
    try:
        nthreads = oracle.use_all_cores(True)
        oracle.use_all_cores(False)
    except Exception as e:                  # no OpenMP on this host compiler
        nthreads = 0
        table.append({"error": f"OpenMP build unavailable: {e}"[:200]})
    for case in CPU_CASES:
        name, kind, M, N, K = case[:5]
        rows = np.arange(min(M, 16)) if M <= 16 else np.linspace(0, M - 1, 8).astype(np.int64)
        scale = M / len(rows)
        entry = {"config": name, "sample_rows": int(len(rows)), "scaled_to_M": M}
        for label, threads in (("1t", 1), ("all", nthreads)):
            if threads == 0:
                continue
            oracle.use_all_cores(threads > 1)
            fn = _oracle_call(oracle, synth, case, rows)
            per, calls = _time_oracle(fn, budget_s / 8)
            us = per * 1e6 * scale
            entry[f"us_per_call_{label}"] = round(us, 1)
            entry[f"threads_{label}"] = threads
            if kind == "mlp":
                bpc = mlp_bytes(M, 4096, N, K)
            else:
                bpc = gemm_bytes(M, N, K)
            entry[f"GBps_{label}"] = round(bpc / us / 1e3, 4)
            if kind != "mlp":
                entry[f"GFLOPS_{label}"] = round(2.0 * M * N * K / us / 1e3, 3)
        oracle.use_all_cores(False)
        table.append(entry)
    res["configs"] = table
    res["host_cores"] = os.cpu_count()
    return res


def run_reference(args):
    """The oracle as it stands (single-threaded C) on the host cores, on the
    headline workload: each step is one whole M=16 N=4096 K=4096 weight-only
    call, the same configuration as the GPU arm."""
    import oracle
    import synth
    run = _oracle_call(oracle, synth, CPU_CASES[1], np.arange(16))
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    us_call = el * 1e6 / args.steps
    gbs = HEADLINE["bytes_per_call"] / us_call / 1e3
    return {"impl": "reference", "metric": METRIC,
            "value": round(gbs, 4), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 weights x bf16 activations, fp32 accumulate", "data": "synthetic",
            "config": dict(HEADLINE),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} whole calls of the headline workload, plain C oracle, 1 thread"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(case, calls):
    """A few plain calls of one workload, for ncu; prints nothing to time."""
    import torch
    import block_scaled_fp8_x128_gb300 as r9q
    import synth
    dev = torch.device("cuda", 0)
    if case == "quant-8192":
        M, K = 8192, 4096
        X = [torch.from_numpy(synth.to_bf16_bits(synth.activations(4, M, K)).view(np.int16)).view(torch.bfloat16).to(dev)
             for _ in range(4)]
        for i in range(calls):
            r9q.r9q_quant_group128(X[i % 4])
        torch.cuda.synchronize()
        return
    if case == "c3":
        M, H, I, Ho = 8, 4096, 1536, 4096
        x = torch.from_numpy(synth.to_bf16_bits(synth.activations(3, M, H)).view(np.int16)).view(torch.bfloat16).to(dev)
        wgu, sgu = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(3, 2 * I, H, tensor=1)).to(dev))
        wdn, sdn = r9q.r9q_quant_weight_block128(torch.from_numpy(synth.weights(3, Ho, I, tensor=2)).to(dev))
        for _ in range(calls):
            r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn)
    else:
        M, N, K, seed, wonly = {"c1": (16, 4096, 4096, 1, True), "c4-8192": (8192, 4096, 4096, 4, False),
                                "c4-128": (128, 4096, 4096, 4, False), "c2-16": (16, 12288, 4096, 2, False),
                                "c2-1": (1, 12288, 4096, 2, False)}[case]
        copies = max(1, min(8, _copies_for(gemm_bytes(M, N, K))))
        X, W, S, Y = _make_inputs(torch, r9q, "w8a8", M, N, K, seed, 0.0, 1.0, copies, dev)
        for i in range(calls):
            if wonly:
                r9q.r9q_gemm_fp8w_bf16a(X[i % copies], W[i % copies], S[i % copies], y=Y[i % copies])
            else:
                r9q.r9q_gemm_fp8_block_qa(X[i % copies], W[i % copies], S[i % copies], y=Y[i % copies])
    torch.cuda.synchronize()


def aggregate_over_ranks(out, world, all_reduce_max):
    """Whole-job figures from one rank's result line.  Every rank runs the same
    single-GPU step on its own GPU (replicas); all_reduce_max(x) returns the
    maximum of x over the ranks.  value = the bytes all ranks moved per step
    divided by the slowest rank's time per step."""
    out = json.loads(json.dumps(out))
    bpc = out["config"]["bytes_per_call"]
    ms = all_reduce_max(out["ms_per_step"])
    gbs_one = bpc / (ms * 1e-3) / 1e9
    out["ms_per_step"] = ms
    out["us_per_call"] = round(ms * 1e3, 3)
    out["n_gpus"] = world
    out["value"] = round(world * gbs_one, 1)
    # the roofline stays per GPU: the dominant kernel at the slowest rank's pace
    out["roofline"]["achieved"] = round(gbs_one, 1)
    out["roofline"]["frac"] = round(gbs_one / out["roofline"]["peak"], 4)
    e2e = out.get("e2e") or {}
    us = e2e.get("us_per_call")
    us = all_reduce_max(us if us is not None else -1.0)
    if us > 0:
        e2e["us_per_call"] = round(us, 3)
        e2e["value"] = round(world * bpc / (us * 1e-6) / 1e9, 1)
    out["gpu_launches"] = world * out["gpu_launches"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default 20000; 20 for --impl reference)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="r9q", choices=["r9q", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-pdl", action="store_true", help="launch every GEMM fully serialised")
    ap.add_argument("--profile-case", choices=["c1", "c4-8192", "c4-128", "c2-1", "c2-16", "c3", "quant-8192"],
                    default=None,
                    help="only run a few calls of one workload (for an external profiler) and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 20000
    if args.profile_case:
        profile_case(args.profile_case, args.steps)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        # replicas only: the path does not shard across GPUs here; every rank
        # runs the same single-GPU step and rank 0 reports the aggregate
        import torch
        import torch.distributed as dist
        global _BARRIER
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
        _BARRIER = dist.barrier
        # the CPU baseline is timed on rank 0 alone
        if rank != 0:
            args.no_cpu_baseline = True
    out = run_gpu(args)
    if world > 1:
        import torch
        import torch.distributed as dist

        def all_reduce_max(v):
            t = torch.tensor([float(v)], dtype=torch.float64, device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return t.item()
        out = aggregate_over_ranks(out, world, all_reduce_max)
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
