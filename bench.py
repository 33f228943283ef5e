"""Benchmark of the selective-scan forward on B300.

One step = one ssm_selective_scan_fwd call over the whole workload (every row of
the hot path: load, step size, discretisation, scan with chunk carries,
readout + gate epilogue, final state).  Default workload: the long-context
bf16 layer (batch 1, L = 131072, D = 2560, N = 16), whose inputs (2.69 GB) are
larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline] [--no-e2e]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload (the scan shards over batch rows and channels with no
exchange), so scaling is weak and `value` is the sum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan tokens*channels/s"
UNIT = "tokens*channels/s"
# Arithmetic roofline of a state update (Abar = ex2(step * A * log2 e), h = Abar h + (step x) B,
# y += C h): one MUFU ex2 and four FP32 FMA-pipe lane operations.  Measured on this B300
# (single-purpose throughput kernels): 32 ex2 and 128 FMA lanes per SM per clock, so
# both units allow 32 updates per SM per clock.
EX2_PER_SM_CLK = 32
FMA_LANES_PER_SM_CLK = 128
FMA_OPS_PER_UPDATE = 4
UPDATES_PER_SM_CLK = min(EX2_PER_SM_CLK, FMA_LANES_PER_SM_CLK / FMA_OPS_PER_UPDATE)

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one whole call (all of
# its kernel launches), from one ncu capture, with the sha256 of the kernel sources it
# was taken on; reported as null once the sources change.  See profiles/.
TRAFFIC = {
    # long_bf16_16k capture (aggregate launch 166.6 MB + output launch 315.6 MB, means
    # of 5), scaled by the units processed (x8) to the 131072-step workload
    "long_bf16": {"bytes_per_call": 3857600000, "kernel_src_sha": "30a783e390386982"},
    "long_bf16_16k": {"bytes_per_call": 482200000, "kernel_src_sha": "30a783e390386982"},
}


def kernel_src_sha() -> str:
    """Hash of the sources of the tiled forward kernels (the kernel the recorded traffic
    belongs to): scan_tile.cuh, kernel_table.cuh and the kernels_*.cu instantiations."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "selective_state_space_112_b300", "csrc")
    files = ([os.path.join(csrc, n) for n in ("scan_tile.cuh", "kernel_table.cuh")]
             + glob.glob(os.path.join(csrc, "kernels_*.cu")))
    h = hashlib.sha256()
    for f in sorted(files):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk.get("sm_max_mhz", 2032.0)), "measured"
    except Exception:
        return 6400.0, 2032.0, "fallback"


class ClockSampler:
    """Samples SM clock and throttle reasons while running: NVML when the Python
    binding is importable, else `nvidia-smi -lms` in a background process."""

    REASONS = {  # NVML clocks-event-reason bits
        0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
    }

    def __init__(self, local_rank: int, period_s: float = 0.005):
        cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [c for c in cvd.split(",") if c.strip()]
        self.index = int(ids[local_rank]) if local_rank < len(ids) and ids[local_rank].strip().isdigit() \
            else local_rank
        self.period = period_s
        self.samples = []       # (mhz, reason bitmask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None

    def __enter__(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
            return self
        except Exception:
            pass
        import subprocess
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._run_smi, daemon=True)
            self._t.start()
            time.sleep(0.3)  # let nvidia-smi start sampling before the timed work
        except Exception:
            self._proc = None
        return self

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                self.samples.append((nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM),
                                     nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)))
            except Exception:
                pass
            time.sleep(self.period)

    def _run_smi(self):
        for line in self._proc.stdout:
            if self._stop.is_set():
                break
            parts = [x.strip() for x in line.split(",")]
            try:
                mhz, mx = float(parts[0]), float(parts[1])
                rs = int(parts[2], 16) if parts[2].startswith("0x") else int(parts[2])
                self.max_mhz = mx
                self.samples.append((mhz, rs))
            except Exception:
                continue

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._t:
            self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"],
                    "samples": 0}
        seen = set()
        for _, rs in self.samples:
            for bit, name in self.REASONS.items():
                if rs & bit:
                    seen.add(name)
        return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(seen),
                "samples": len(self.samples)}


def device_tensors(w, torch, device):
    def dev(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return {k: dev(getattr(w, k)) for k in ("x", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0")}


def oracle_sample(w, k, cv=None):
    """The float64 oracle, as it stands, on channels 0..k-1 of batch row 0 over the
    full sequence length (with the block prologue when ``cv`` is given); returns
    seconds."""
    import oracle
    # the sample's inputs: batch row 0, channels 0..k-1 (sliced outside the timed region)
    sl = lambda a: None if a is None else np.ascontiguousarray(a[:1, :, :k])
    ch = lambda a: None if a is None else np.ascontiguousarray(a[:k])
    x, delta, z = sl(w.x), sl(w.delta), sl(w.z)
    A, D, bias = ch(w.A), ch(w.D), ch(w.delta_bias)
    if w.per_channel_bc:
        B, C = ch(w.B), ch(w.C)
    else:
        B, C = np.ascontiguousarray(w.B[:1]), np.ascontiguousarray(w.C[:1])
    h0 = None if w.h0 is None else np.ascontiguousarray(w.h0[:1, :k])
    t = time.perf_counter()
    if cv is None:
        oracle.selective_scan(x, delta, A, B, C, D=D, z=z, delta_bias=bias, h0=h0,
                              delta_softplus=w.delta_softplus, per_channel_bc=w.per_channel_bc,
                              io_dtype=w.io)
    else:
        oracle.conv_selective_scan(x, ch(cv.w), ch(cv.b), None, delta, A, B, C, D=D, z=z,
                                   delta_bias=bias, h0=h0, delta_softplus=w.delta_softplus,
                                   io_dtype=w.io)
    return time.perf_counter() - t


# One sample rule for the CPU baseline and the reference arm: channels 0..k-1 of
# batch row 0 over the whole sequence, k = min(dim, CPU_SAMPLE_CHANNELS), with the
# sample's inputs sliced before the timed region.  At 512 channels the fixed cost of
# a call (widening B and C of the whole sequence) is a few percent of its time.
CPU_SAMPLE_CHANNELS = 512


def cpu_sample_channels(w) -> int:
    return min(w.dim, CPU_SAMPLE_CHANNELS)


def cpu_baseline(w, cv=None):
    import oracle
    cores = oracle.max_threads()
    k = cpu_sample_channels(w)
    oracle_sample(w, min(k, cores), cv)  # loads the library, starts the thread pool
    t = oracle_sample(w, k, cv)
    units = k * w.seqlen
    what = "block prologue + scan" if cv is not None else "scan"
    return {"value": units / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"channels 0..{k - 1} of batch row 0, all {w.seqlen} steps, N={w.dstate}, {what} "
                      f"({units} tokens*channels, {t:.2f} s, float64 C + OpenMP)"}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over all ranks (the job's time is the slowest rank's)."""
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, steps: int, ms_max: float, world: int) -> float:
    """Whole-job units per second: every rank ran its own replica of the workload."""
    return world * units_per_rank * steps / (ms_max * 1e-3)


def whole_call_traffic(workload: str, conv: bool):
    """DRAM bytes (read + write) of one whole call from the recorded ncu capture, or
    None when none is recorded for the current kernel sources."""
    tr = TRAFFIC.get(workload)
    if tr and not conv and tr["kernel_src_sha"] == kernel_src_sha():
        return tr["bytes_per_call"]
    return None


def roofline(w, ms_call, prof, torch, device, clocks, traffic=None):
    """HBM roofline of one call (all of its kernels) and the arithmetic bound beside it.

    achieved = algorithmic bytes of the call / device time of the call; peak = the
    measured copy bandwidth.  The arithmetic bound counts one MUFU ex2 per state update
    at 32 per SM per clock, at the median SM clock sampled while timing."""
    hbm_peak, sm_max, peak_kind = load_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    alg = w.algorithmic_bytes()
    achieved = alg / (ms_call * 1e-3) / 1e9
    mhz = clocks.get("sm_mhz") or sm_max
    upd_peak = UPDATES_PER_SM_CLK * sms * mhz * 1e6 / 1e9           # Gupdate/s
    upd_achieved = w.element_updates / (ms_call * 1e-3) / 1e9
    total_ms = sum(v[1] for v in prof.values()) or 1.0
    return {"bound": "hbm", "kernel": "whole call (" + ", ".join(sorted(prof)) + ")",
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "peak_source": peak_kind,
            "traffic": traffic, "algorithmic_bytes_per_launch": alg,
            "kernel_ms_avg": round(ms_call, 4),
            "alu": {"achieved": round(upd_achieved, 1), "peak": round(upd_peak, 1),
                    "unit": "Gupdate/s", "frac": round(upd_achieved / upd_peak, 4),
                    "peak_basis": (f"min({EX2_PER_SM_CLK} MUFU ex2, {FMA_LANES_PER_SM_CLK}/"
                                   f"{FMA_OPS_PER_UPDATE} FMA lanes) state updates per SM per clock"
                                   f" (measured on B300) x {sms} SMs x {mhz:.0f} MHz (median sampled)")},
            "kernels": {k: {"launches": v[0], "ms_avg": round(v[1] / v[0], 4),
                            "share": round(v[1] / total_ms, 4)} for k, v in prof.items()}}


def timed_calls(fn, torch, stream, reps, flush=None):
    """Device times (ms) of `reps` calls of fn, each bracketed by CUDA events on the
    launch stream; flush() (an L2-sized write) runs between calls, outside the events.
    A short device-side wait before the first event lets the host enqueue the call
    while the GPU is still busy, so that the host's launch cost stays outside."""
    times = []
    for _ in range(reps):
        if flush is not None:
            flush()
        torch.cuda._sleep(400000)  # about 0.2 ms of device time
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    return times


def other_workloads(torch, ssm, device, names, reps=20):
    """The other scan workloads, timed in the same run: per call the median, min and
    90th percentile of `reps` calls with the L2 flushed between them, the HBM and
    arithmetic fractions, and the per-kernel split.  The recurrent-step workload is
    also timed as 128 chained steps in one CUDA graph (its state stays in L2 across
    steps, as in decoding)."""
    from selective_state_space_112_b300.workloads import config
    stream = torch.cuda.current_stream(device)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    flush = lambda: flush_buf.zero_()
    out = {}
    for name in names:
        w = config(name)
        t = device_tensors(w, torch, device)
        o = torch.empty_like(t["x"])
        state_in = w.h0 is not None
        fs = t["h0"].clone() if state_in else torch.empty((w.batch, w.dim, w.dstate),
                                                           dtype=torch.float32, device=device)

        def call():
            ssm.ssm_selective_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                       t["delta_bias"], out=o, final_state=fs,
                                       delta_softplus=w.delta_softplus, state_in=state_in)
        for _ in range(3):
            call()
        assert ssm.ssm_check_status() == 0
        ssm.ssm_profile_enable(True)
        with ClockSampler(torch.cuda.current_device()) as clk:
            times = timed_calls(call, torch, stream, reps, flush)
        ssm.ssm_profile_enable(False)
        prof = ssm.ssm_profile_read()
        assert ssm.ssm_check_status() == 0
        times.sort()
        med = statistics.median(times)
        latency = w.algorithmic_bytes() < 126e6 and name != "step_bf16"
        rf = roofline(w, med, prof, torch, device, clk.summary())
        rec = {"shape": {"batch": w.batch, "seqlen": w.seqlen, "dim": w.dim, "dstate": w.dstate,
                         "io_dtype": w.io, "gate": w.z is not None, "state_in": state_in},
               "ms_median": round(med, 5), "ms_min": round(times[0], 5),
               "ms_p90": round(times[int(0.9 * (len(times) - 1))], 5),
               "tokens_channels_per_s": w.tokens_channels / (med * 1e-3),
               "reps": reps, "l2": "flushed between calls (256 MB write)",
               "roofline": None if latency else {k: rf[k] for k in ("bound", "achieved", "peak",
                                                                   "unit", "frac", "alu")},
               "kernels": rf["kernels"], "clocks": clk.summary()}
        if latency:
            rec["note"] = "inputs fit in L2: a latency figure, no roofline claim"
        if name == "step_bf16":
            # 128 recurrent steps chained in one CUDA graph, each advancing the state
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for _ in range(3):
                    call()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            with torch.cuda.graph(g):
                for _ in range(128):
                    call()
            g.replay()
            torch.cuda.synchronize()
            gt = timed_calls(g.replay, torch, stream, 10)
            gm = statistics.median(gt) / 128
            rec["graph_chain"] = {"steps": 128, "ms_per_step": round(gm, 5),
                                  "hbm_gbs": round(w.algorithmic_bytes() / (gm * 1e-3) / 1e9, 1),
                                  "l2": "state carried in L2 across the chained steps"}
            del g
        out[name] = rec
        del t, o, fs
        torch.cuda.empty_cache()
    return out


def e2e_scan(args, w, t, out, fs, state_in, conv, torch, ssm, device, stream, world, dist, units):
    """The same call through the public API with host buffers: every step copies its
    inputs from pinned host memory and its results (out, final state) back, inside the
    timed region.  Consecutive steps overlap as a serving loop would run them: two sets
    of device buffers, the inputs of step k+1 copied (on their own stream) while step k
    computes and step k-1's results copy back (on a third stream), so that a step costs
    about its host-to-device copy rather than the sum of both copies and the call."""
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in t.items()}
    extra_h = {}
    if conv is not None:  # the prologue's taps and bias are inputs of every step too
        extra_h = {"cw": conv[0].cpu().pin_memory(), "cb": conv[1].cpu().pin_memory()}
    slots = []
    for _ in range(2):
        slots.append({
            "in": {k: (torch.empty_like(v) if v is not None else None) for k, v in t.items()},
            "ex": {k: torch.empty(v.shape, dtype=v.dtype, device=device) for k, v in extra_h.items()},
            "cs": (torch.empty_like(conv[2]) if conv is not None and conv[2] is not None else None),
            "out": torch.empty_like(out), "fs": torch.empty_like(fs),
            "out_h": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
            "fs_h": torch.empty(fs.shape, dtype=fs.dtype).pin_memory()})
    h2d = (sum(v.numel() * v.element_size() for v in host.values() if v is not None)
           + sum(v.numel() * v.element_size() for v in extra_h.values()))
    d2h = out.numel() * out.element_size() + fs.numel() * fs.element_size()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # the slot's inputs have landed
    ev_call = [torch.cuda.Event() for _ in range(2)]  # the slot's call is done
    ev_back = [torch.cuda.Event() for _ in range(2)]  # the slot's results are on the host

    def e2e_step(k):
        i = k % 2
        sl = slots[i]
        fsd = sl["in"]["h0"] if state_in else sl["fs"]
        # inputs: the slot's buffers are free once its previous call ran and its
        # previous results left (an event not yet recorded is no wait)
        s_in.wait_event(ev_call[i])
        s_in.wait_event(ev_back[i])
        with torch.cuda.stream(s_in):
            for key, v in host.items():
                if v is not None:
                    sl["in"][key].copy_(v, non_blocking=True)
            for key, v in extra_h.items():
                sl["ex"][key].copy_(v, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        stream.wait_event(ev_back[i])
        d = sl["in"]
        if conv is not None:
            ssm.ssm_conv_selective_scan_fwd(d["x"], sl["ex"]["cw"], sl["ex"]["cb"], sl["cs"], d["delta"],
                                            d["A"], d["B"], d["C"], d["D"], d["z"], d["delta_bias"],
                                            out=sl["out"], final_state=fsd,
                                            delta_softplus=w.delta_softplus, state_in=state_in)
        else:
            ssm.ssm_selective_scan_fwd(d["x"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                       d["delta_bias"], out=sl["out"], final_state=fsd,
                                       delta_softplus=w.delta_softplus, state_in=state_in)
        ev_call[i].record(stream)
        s_out.wait_event(ev_call[i])
        with torch.cuda.stream(s_out):
            sl["out_h"].copy_(sl["out"], non_blocking=True)
            sl["fs_h"].copy_(fsd, non_blocking=True)
            ev_back[i].record(s_out)

    for k in range(2):  # warm both slots
        e2e_step(k)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(args.e2e_steps):
        e2e_step(k)
    for i in range(2):
        stream.wait_event(ev_back[i])
    e1.record(stream)
    torch.cuda.synchronize()
    assert ssm.ssm_check_status() == 0
    ems = e0.elapsed_time(e1)
    if world > 1:
        ems = max_over_ranks(ems, dist, device)
    return {"value": job_throughput(units, args.e2e_steps, ems, world), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ems / args.e2e_steps,
            "overlap": "step k+1's inputs copy while step k computes and step k-1's results copy back"}


def ssd_and_backward_configs(torch, ssm, device, main_w=None, main_t=None, reps=10):
    """The Mamba-2 SSD layers and the backward pass of the long-context layer, timed in
    the same run as the headline (median of `reps` calls; inputs larger than L2), so
    that their figures appear in the line: per call the time, the HBM fraction of the
    algorithmic bytes and, for SSD, the tensor fraction of its flops; for the backward
    the split over its kernels and the fraction of its MUFU bound.  The headline's
    tensors are reused when it is the long-context layer (same seed on rank 0)."""
    from selective_state_space_112_b300.workloads import (SSD_CONFIGS, config, f32_to_bf16_bits,
                                                          make_ssd)
    stream = torch.cuda.current_stream(device)
    hbm_peak, sm_max, peak_kind = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tc_peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        tc_peak = 1800.0
    out = {}
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    for name in ("mamba2_2p7b_bf16", "mamba2_n256_bf16"):
        w = make_ssd(name, **SSD_CONFIGS[name])
        t = {k: (None if getattr(w, k) is None else
                 (bf(getattr(w, k)) if getattr(w, k).dtype == np.uint16 else
                  torch.from_numpy(getattr(w, k))).to(device))
             for k in ("x", "dt", "A", "B", "C", "D", "z", "dt_bias")}
        o = torch.empty_like(t["x"])
        fs = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=device)

        def call():
            ssm.ssm_ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["dt_bias"],
                            out=o, final_state=fs)
        for _ in range(3):
            call()
        assert ssm.ssm_check_status() == 0
        with ClockSampler(torch.cuda.current_device()) as clk:
            times = sorted(timed_calls(call, torch, stream, reps))
        assert ssm.ssm_check_status() == 0
        med = statistics.median(times)
        byt, flops = ssd_algorithmic(w)
        out["ssd_" + name] = {
            "layer": "Mamba-2 SSD", "kernel": "ssd_tc_kernel",
            "shape": {"batch": w.batch, "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
                      "dstate": w.dstate, "ngroups": w.ngroups},
            "ms_median": round(med, 5), "ms_min": round(times[0], 5),
            "tokens_channels_per_s": w.tokens_channels / (med * 1e-3),
            "hbm": {"achieved": round(byt / (med * 1e-3) / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(byt / (med * 1e-3) / 1e9 / hbm_peak, 4), "peak_source": peak_kind},
            "tensor": {"achieved": round(flops / (med * 1e-3) / 1e12, 2), "peak": tc_peak,
                       "unit": "TFLOP/s", "frac": round(flops / (med * 1e-3) / 1e12 / tc_peak, 4)},
            "reps": reps, "clocks": clk.summary()}
        del t, o, fs
        torch.cuda.empty_cache()
    # the backward pass of the long-context layer
    if main_w is not None and main_w.name == "long_bf16":
        w, t = main_w, main_t
    else:
        w = config("long_bf16")
        t = device_tensors(w, torch, device)
    rng = np.random.default_rng(w.seed + 4242)
    dout = bf(f32_to_bf16_bits(rng.standard_normal(w.x.shape, dtype=np.float32))).to(device)
    grads = ssm.ssm_selective_scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                       t["delta_bias"], t["h0"], dout, delta_softplus=w.delta_softplus)

    def bwd():
        ssm.ssm_selective_scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                   t["delta_bias"], t["h0"], dout, delta_softplus=w.delta_softplus,
                                   grads=grads)
    for _ in range(3):
        bwd()
    assert ssm.ssm_check_status() == 0
    ssm.ssm_profile_enable(True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        times = sorted(timed_calls(bwd, torch, stream, max(3, reps // 2)))
    ssm.ssm_profile_enable(False)
    prof = ssm.ssm_profile_read()
    assert ssm.ssm_check_status() == 0
    med = statistics.median(times)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    dom = max(prof, key=lambda k: prof[k][1]) if prof else None
    dom_ms = prof[dom][1] / prof[dom][0] if dom else med
    upd_peak = EX2_PER_SM_CLK / BWD_EX2_PER_UPDATE * sms * sm_max * 1e6 / 1e9
    esz = 2
    alg = (w.tokens_channels * esz * 7 + w.batch * w.seqlen * w.dstate * (2 * esz + 8)
           + w.dim * (w.dstate + 2) * 8)
    out["backward_long_bf16"] = {
        "pass": "backward (gradients of every input, states rebuilt from checkpoints)",
        "shape": {"batch": w.batch, "seqlen": w.seqlen, "dim": w.dim, "dstate": w.dstate},
        "ms_median": round(med, 4), "ms_min": round(times[0], 4),
        "hbm": {"achieved": round(alg / (med * 1e-3) / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(alg / (med * 1e-3) / 1e9 / hbm_peak, 4)},
        "alu": {"kernel": dom, "achieved": round(w.element_updates / (dom_ms * 1e-3) / 1e9, 1),
                "peak": round(upd_peak, 1), "unit": "Gupdate/s",
                "frac": round(w.element_updates / (dom_ms * 1e-3) / 1e9 / upd_peak, 4),
                "peak_basis": f"{EX2_PER_SM_CLK} ex2 / SM / clock / {BWD_EX2_PER_UPDATE} ex2 per update"},
        "kernels": {k: {"launches": v[0], "ms_avg": round(v[1] / v[0], 4)} for k, v in prof.items()},
        "clocks": clk.summary()}
    del grads, dout
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_bf16")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads (the line's `configs` object)")
    ap.add_argument("--conv", action="store_true",
                    help="the Mamba-block prologue (causal conv of width 4 + silu) fused in")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (gradients of every input) instead")
    ap.add_argument("--ssd", action="store_true",
                    help="time the Mamba-2 SSD layer (default workload mamba2_2p7b_bf16) instead")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from selective_state_space_112_b300.workloads import CONFIGS, SSD_CONFIGS, make_workload
    if args.ssd:
        if args.workload not in SSD_CONFIGS:
            args.workload = "mamba2_2p7b_bf16"
        if args.impl == "reference":
            return reference_arm(args, world, rank)
        return ssd_bench(args, world, rank, local)
    if args.workload not in CONFIGS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(CONFIGS)}")

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    import torch.distributed as dist
    import selective_state_space_112_b300 as ssm

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    spec = dict(CONFIGS[args.workload])
    spec["seed"] = spec["seed"] + 1000 * rank  # independent replica per rank
    w = make_workload(args.workload, **spec)
    t = device_tensors(w, torch, device)
    if args.backward:
        return backward_bench(args, w, t, world, rank, local, device, dist, torch, ssm)
    out = torch.empty_like(t["x"])
    fs0 = t["h0"]
    fs = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    state_in = w.h0 is not None

    if state_in:
        fs.copy_(fs0)  # recurrent-step workload: each step advances the stored state
    cv = cw = cb = cs = None
    if args.conv:
        from selective_state_space_112_b300.workloads import make_conv
        cv = make_conv(w, hist=state_in)
        cw = torch.from_numpy(cv.w).to(device)
        cb = torch.from_numpy(cv.b).to(device)
        cs = torch.from_numpy(cv.hist).to(device) if state_in else None

    def scan(x, delta, A, B, C, D, z, bias, final_state):
        if args.conv:
            ssm.ssm_conv_selective_scan_fwd(x, cw, cb, cs, delta, A, B, C, D, z, bias, out=out,
                                            final_state=final_state,
                                            delta_softplus=w.delta_softplus, state_in=state_in)
        else:
            ssm.ssm_selective_scan_fwd(x, delta, A, B, C, D, z, bias, out=out,
                                       final_state=final_state,
                                       delta_softplus=w.delta_softplus, state_in=state_in)

    def step():
        scan(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], fs)

    for _ in range(args.warmup):
        step()
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()

    # ---- timed region: K steps, events on the launch stream, barrier + sync both sides
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = ssm.ssm_kernel_launches()
    ssm.ssm_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    ssm.ssm_profile_enable(False)
    prof = ssm.ssm_profile_read()
    launches = ssm.ssm_kernel_launches() - launches0
    assert ssm.ssm_check_status() == 0
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        ms = max_over_ranks(ms, dist, device)
        dist.barrier()
    ms_step = ms / args.steps
    units = w.tokens_channels
    value = job_throughput(units, args.steps, ms, world)

    # ---- roofline: the whole call against HBM (the path's stated roofline: the
    # minimum bytes in and out over the copy bandwidth), with the arithmetic bound
    # beside it at the SM clock sampled during the timed region
    clocks = clk.summary()
    roof = roofline(w, ms_step, prof, torch, device, clocks,
                    traffic=whole_call_traffic(args.workload, args.conv))

    res = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f32", "data": "synthetic",
           "config": {"workload": args.workload, "batch": w.batch, "seqlen": w.seqlen,
                      "dim": w.dim, "dstate": w.dstate, "io_dtype": w.io,
                      "gate": w.z is not None, "state_in": state_in,
                      "prologue": "causal conv width 4 + silu" if args.conv else "none",
                      "parallelism": f"replica x{world}" if world > 1 else "single",
                      "l2": f"inputs {w.algorithmic_bytes() / 1e9:.2f} GB > 126 MB L2; no flush needed"
                            if w.algorithmic_bytes() > 4 * 126e6 else "L2 resident (latency case)"},
           "roofline": roof, "gpu_launches": int(launches), "clocks": clocks}

    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        res["e2e"] = e2e_scan(args, w, t, out, fs, state_in, (cw, cb, cs) if args.conv else None,
                              torch, ssm, device, stream, world, dist, units)

    if rank == 0 and world == 1 and not args.no_configs and not args.conv:
        others = [n for n in ("mamba130m_f32", "mamba1p4b_bf16", "step_bf16", "lti_f32", "tiny_f32")
                  if n != args.workload]
        res["configs"] = other_workloads(torch, ssm, device, others)
        res["configs"].update(ssd_and_backward_configs(torch, ssm, device, w, t))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, cv=cv)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


# The main backward kernel forms Abar three times per state update (the checkpoint
# sweep, the segment rebuild and the adjoint sweep): its MUFU ex2 roofline.
BWD_EX2_PER_UPDATE = 3


def backward_bench(args, w, t, world, rank, local, device, dist, torch, ssm):
    """One step = one ssm_selective_scan_bwd call over the whole workload, with a
    seeded upstream gradient dout ~ N(0, 1) in the io dtype."""
    from selective_state_space_112_b300.workloads import f32_to_bf16_bits
    rng = np.random.default_rng(w.seed + 4242)
    dout = rng.standard_normal(w.x.shape, dtype=np.float32)
    if w.io == "bf16":
        dout = f32_to_bf16_bits(dout)
    t["dout"] = (torch.from_numpy(dout.view(np.int16)).view(torch.bfloat16) if w.io == "bf16"
                 else torch.from_numpy(dout)).to(device)
    stream = torch.cuda.current_stream(device)
    grads = ssm.ssm_selective_scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                       t["delta_bias"], t["h0"], t["dout"],
                                       delta_softplus=w.delta_softplus)

    def bwd(x, delta, A, B, C, D, z, bias, h0, dout_):
        ssm.ssm_selective_scan_bwd(x, delta, A, B, C, D, z, bias, h0, dout_,
                                   delta_softplus=w.delta_softplus, grads=grads)

    def step():
        bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], t["h0"], t["dout"])

    for _ in range(args.warmup):
        step()
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = ssm.ssm_kernel_launches()
    ssm.ssm_profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    ssm.ssm_profile_enable(False)
    prof = ssm.ssm_profile_read()
    launches = ssm.ssm_kernel_launches() - launches0
    assert ssm.ssm_check_status() == 0
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        ms = max_over_ranks(ms, dist, device)
        dist.barrier()
    ms_step = ms / args.steps
    units = w.tokens_channels
    value = job_throughput(units, args.steps, ms, world)

    hbm_peak, sm_max, peak_kind = load_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    esz = 2 if w.io == "bf16" else 4
    bt = w.batch * w.seqlen
    # inputs x, delta, z, dout and outputs dx, ddelta, dz per (b, t, d); B, C in and
    # dB, dC (fp32) out per (b, t, n); A, D, bias and their gradients per channel
    per_tc = 7 if w.z is not None else 5  # (x, delta, [z], dout) in, (dx, ddelta, [dz]) out
    alg = units * esz * per_tc + bt * w.dstate * (2 * esz + 8) + w.dim * (w.dstate + 2) * 8
    dom = max(prof, key=lambda k: prof[k][1]) if prof else None
    dom_ms = prof[dom][1] / prof[dom][0] if dom else ms_step
    total_ms = sum(v[1] for v in prof.values()) or 1.0
    upd_peak = EX2_PER_SM_CLK / BWD_EX2_PER_UPDATE * sms * sm_max * 1e6 / 1e9
    upd_achieved = w.element_updates / (dom_ms * 1e-3) / 1e9
    hbm_achieved = alg / (dom_ms * 1e-3) / 1e9
    roof = {"bound": "alu", "kernel": dom, "achieved": round(upd_achieved, 1), "peak": round(upd_peak, 1),
            "unit": "Gupdate/s", "frac": round(upd_achieved / upd_peak, 4),
            "peak_basis": (f"{EX2_PER_SM_CLK} MUFU ex2 per SM per clock (measured on B300) / "
                           f"{BWD_EX2_PER_UPDATE} ex2 per state update in the main backward kernel x "
                           f"{sms} SMs x {sm_max:.0f} MHz"),
            "traffic": None, "algorithmic_bytes_per_launch": alg, "kernel_ms_avg": round(dom_ms, 4),
            "hbm": {"achieved": round(hbm_achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(hbm_achieved / hbm_peak, 4), "peak_source": peak_kind},
            "kernels": {k: {"launches": v[0], "ms_avg": round(v[1] / v[0], 4),
                            "share": round(v[1] / total_ms, 4)} for k, v in prof.items()}}
    res = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f32", "data": "synthetic",
           "config": {"workload": args.workload, "pass": "backward", "batch": w.batch,
                      "seqlen": w.seqlen, "dim": w.dim, "dstate": w.dstate, "io_dtype": w.io,
                      "gate": w.z is not None, "state_in": w.h0 is not None,
                      "parallelism": f"replica x{world}" if world > 1 else "single",
                      "l2": f"inputs {alg / 1e9:.2f} GB > 126 MB L2; no flush needed"
                            if alg > 4 * 126e6 else "L2 resident (latency case)"},
           "hbm_gbs_step": round(alg / (ms_step * 1e-3) / 1e9, 1),
           "roofline": roof, "gpu_launches": int(launches), "clocks": clk.summary()}

    if not args.no_e2e:
        names = ("x", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0", "dout")
        host = {k: (t[k].cpu().pin_memory() if t[k] is not None else None) for k in names}
        dev_in = {k: (torch.empty_like(v) if v is not None else None) for k, v in t.items() if k in names}
        outs = {k: v for k, v in grads.items() if v is not None}
        outs_h = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = sum(v.numel() * v.element_size() for v in outs_h.values())

        def e2e_step():
            for k, v in host.items():
                if v is not None:
                    dev_in[k].copy_(v, non_blocking=True)
            bwd(*[dev_in[k] for k in names])
            for k, v in outs.items():
                outs_h[k].copy_(v, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = e0.elapsed_time(e1)
        if world > 1:
            ems = max_over_ranks(ems, dist, device)
        res["e2e"] = {"value": job_throughput(units, args.e2e_steps, ems, world), "unit": UNIT,
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": ems / args.e2e_steps}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_bwd(w, dout)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def cpu_baseline_bwd(w, dout, budget_s: float = 15.0):
    """The float64 oracle's backward on channels 0..k-1 of batch row 0, whole sequence."""
    import oracle
    from selective_state_space_112_b300.workloads import bf16_bits_to_f32
    cores = oracle.max_threads()
    g64 = bf16_bits_to_f32(dout).astype(np.float64) if w.io == "bf16" else dout.astype(np.float64)

    def run(k):
        sl = lambda a: None if a is None else np.ascontiguousarray(a[:1, :, :k])
        ch = lambda a: None if a is None else np.ascontiguousarray(a[:k])
        args = (sl(w.x), sl(w.delta), ch(w.A), np.ascontiguousarray(w.B[:1]), np.ascontiguousarray(w.C[:1]),
                ch(w.D), sl(w.z), ch(w.delta_bias),
                None if w.h0 is None else np.ascontiguousarray(w.h0[:1, :k]))
        gs = sl(g64)
        t0 = time.perf_counter()
        oracle.selective_scan_bwd(*args, dout=gs, delta_softplus=w.delta_softplus, io_dtype=w.io)
        return time.perf_counter() - t0

    cap = min(w.dim, 512)
    k = min(cap, max(cores, 8))
    t = run(k)
    k2 = int(min(cap, max(k, k * budget_s / max(t, 1e-3))))
    k2 = max(1, (k2 // cores) * cores) if k2 >= cores else k2
    if k2 > k:
        t, k = run(k2), k2
    units = k * w.seqlen
    return {"value": units / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"backward, channels 0..{k - 1} of batch row 0, all {w.seqlen} steps, N={w.dstate} "
                      f"({units} tokens*channels, {t:.1f} s, float64 C + OpenMP)"}


SSD_Q = 128  # chunk length of the SSD kernel's dual form


def ssd_algorithmic(w):
    """Bytes and multiply-add flops one SSD call must move / do at least.
    Bytes: x, z in and out once (b L H P, bf16), dt (b L H), B and C (b L G N), the
    per-head parameters and the final state (b H P N fp32).  Flops: the dual form per
    128-step chunk and head: the causal half of C B^T (Q(Q+1)/2 N) and of M x
    (Q(Q+1)/2 P), the readout of the carried state C h (Q P N) and its update B^T x
    (N P Q), two flops per multiply-add."""
    tc = w.batch * w.seqlen * w.nheads * w.headdim
    byt = (tc * 2 * (3 if w.z is not None else 2) + w.batch * w.seqlen * w.nheads * 2
           + 2 * w.batch * w.seqlen * w.ngroups * w.dstate * 2 + 3 * w.nheads * 4
           + w.batch * w.nheads * w.headdim * w.dstate * 4)
    Q, P, N = SSD_Q, w.headdim, w.dstate
    nch = (w.seqlen + Q - 1) // Q
    flops = w.batch * w.nheads * nch * 2 * (Q * (Q + 1) // 2 * (N + P) + 2 * Q * P * N)
    return byt, flops


def ssd_bench(args, world, rank, local):
    """One step = one ssm_ssd_fwd call over a Mamba-2-shaped layer (bf16 in and out,
    fp32 state), inputs resident in HBM; e2e adds the host copies."""
    import torch
    import torch.distributed as dist
    import selective_state_space_112_b300 as ssm
    from selective_state_space_112_b300.workloads import SSD_CONFIGS, make_ssd
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    spec = dict(SSD_CONFIGS[args.workload])
    spec["seed"] = spec["seed"] + 1000 * rank
    w = make_ssd(args.workload, **spec)
    names = ("x", "dt", "A", "B", "C", "D", "z", "dt_bias")
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    host = {k: (None if getattr(w, k) is None else
                (bf(getattr(w, k)) if getattr(w, k).dtype == np.uint16 else torch.from_numpy(getattr(w, k))))
            for k in names}
    t = {k: (v.to(device) if v is not None else None) for k, v in host.items()}
    out = torch.empty_like(t["x"])
    fs = torch.empty((w.batch, w.nheads, w.headdim, w.dstate), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def call(d, o, f):
        ssm.ssm_ssd_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                        out=o, final_state=f)

    for _ in range(args.warmup):
        call(t, out, fs)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = ssm.ssm_kernel_launches()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            call(t, out, fs)
        ev1.record(stream)
        torch.cuda.synchronize()
    launches = ssm.ssm_kernel_launches() - launches0
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        ms = max_over_ranks(ms, dist, device)
        dist.barrier()
    ms_step = ms / args.steps
    units = w.tokens_channels
    value = job_throughput(units, args.steps, ms, world)
    byt, flops = ssd_algorithmic(w)
    hbm_peak, _, peak_kind = load_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tc_peak, tc_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tc_peak, tc_kind = 1800.0, "fallback"
    # one kernel launch per step: the step's event time is the kernel's duration
    hbm_ach = byt / (ms_step * 1e-3) / 1e9
    tc_ach = flops / (ms_step * 1e-3) / 1e12
    t_hbm, t_tc = byt / (hbm_peak * 1e9), flops / (tc_peak * 1e12)
    hbm_obj = {"bound": "hbm", "achieved": round(hbm_ach, 1), "peak": hbm_peak, "unit": "GB/s",
               "frac": round(hbm_ach / hbm_peak, 4), "peak_source": peak_kind}
    tc_obj = {"bound": "tensor", "achieved": round(tc_ach, 2), "peak": tc_peak, "unit": "TFLOP/s",
              "frac": round(tc_ach / tc_peak, 4), "peak_source": f"{tc_kind} bf16 burst"}
    main_obj, other = (hbm_obj, tc_obj) if t_hbm >= t_tc else (tc_obj, hbm_obj)
    roof = dict(main_obj, kernel="ssd_tc_kernel", traffic=None, algorithmic_bytes_per_launch=byt,
                algorithmic_flops_per_launch=flops, kernel_ms_avg=round(ms_step, 4),
                roofline_ms={"hbm": round(t_hbm * 1e3, 4), "tensor": round(t_tc * 1e3, 4)},
                other=other)
    res = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic",
           "config": {"workload": args.workload, "layer": "Mamba-2 SSD", "batch": w.batch,
                      "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
                      "ngroups": w.ngroups, "dstate": w.dstate, "gate": w.z is not None,
                      "parallelism": f"replica x{world}" if world > 1 else "single",
                      "l2": f"inputs {byt / 1e9:.2f} GB > 126 MB L2; no flush needed"},
           "roofline": roof, "gpu_launches": int(launches), "clocks": clk.summary()}
    if not args.no_e2e:
        hp = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
        dev_in = {k: (torch.empty_like(v) if v is not None else None) for k, v in t.items()}
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in hp.values() if v is not None)
        d2h = out_h.numel() * out_h.element_size() + fs_h.numel() * fs_h.element_size()

        def e2e_step():
            for k, v in hp.items():
                if v is not None:
                    dev_in[k].copy_(v, non_blocking=True)
            call(dev_in, out, fs)
            out_h.copy_(out, non_blocking=True)
            fs_h.copy_(fs, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = e0.elapsed_time(e1)
        if world > 1:
            ems = max_over_ranks(ems, dist, device)
        res["e2e"] = {"value": job_throughput(units, args.e2e_steps, ems, world), "unit": UNIT,
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": ems / args.e2e_steps}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_ssd(w)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def cpu_baseline_ssd(w, budget_s: float = 15.0):
    """The float64 oracle's SSD recurrence on the first k heads of the first r batch
    rows, whole sequence (k grows first, then r, to about budget_s of host time)."""
    import oracle
    cores = oracle.max_threads()
    hpg = w.nheads // w.ngroups

    def run(r, k):
        g1 = (k - 1) // hpg + 1  # groups the first k heads read
        sl = lambda a: None if a is None else np.ascontiguousarray(a[:r, :, :k])
        t0 = time.perf_counter()
        oracle.ssd(sl(w.x), sl(w.dt), w.A[:k], np.ascontiguousarray(w.B[:r, :, :g1]),
                   np.ascontiguousarray(w.C[:r, :, :g1]), D=None if w.D is None else w.D[:k],
                   z=sl(w.z), dt_bias=None if w.dt_bias is None else w.dt_bias[:k])
        return time.perf_counter() - t0

    r, k = 1, min(w.nheads, max(1, min(cores, 4)))
    t = run(r, k)
    k2 = int(min(w.nheads, max(k, k * budget_s / max(t, 1e-3))))
    if k2 > k:
        t, k = run(r, k2), k2
    if k == w.nheads and t < budget_s / 2 and w.batch > 1:
        r2 = int(min(w.batch, max(1, budget_s / max(t, 1e-3))))
        if r2 > r:
            t, r = run(r2, k), r2
    units = r * k * w.headdim * w.seqlen
    return {"value": units / t, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"SSD, heads 0..{k - 1} of batch rows 0..{r - 1}, all {w.seqlen} steps, "
                      f"P={w.headdim}, N={w.dstate} ({units} tokens*channels, {t:.1f} s, float64 C + OpenMP)"}


def reference_arm(args, world, rank):
    """The oracle as the reference arm: timed on the host cores, each step a
    bounded sample of the same workload.  Under torchrun only rank 0 runs."""
    if rank != 0:
        return
    if getattr(args, "ssd", False):
        return reference_arm_ssd(args, world)
    from selective_state_space_112_b300.workloads import config
    import oracle
    w = config(args.workload)
    cores = oracle.max_threads()
    k = cpu_sample_channels(w)
    oracle_sample(w, min(k, cores))  # loads the library, starts the thread pool
    t1 = oracle_sample(w, k)
    budget = 240.0  # seconds for all warm-up and timed steps
    if (args.steps + args.warmup) * t1 > budget:
        # the same rule on fewer channels, so that the run ends within minutes
        k = max(min(k, cores), int(k * budget / ((args.steps + args.warmup) * t1)))
    for _ in range(max(args.warmup - 1, 0)):
        oracle_sample(w, k)
    el = 0.0
    for _ in range(args.steps):
        el += oracle_sample(w, k)
    units = k * w.seqlen
    value = units * args.steps / el
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "batch": w.batch, "seqlen": w.seqlen,
                      "dim": w.dim, "dstate": w.dstate, "io_dtype": w.io},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": f"channels 0..{k - 1} of batch row 0, all {w.seqlen} steps, "
                                      f"N={w.dstate}, per step (the CPU baseline's sample rule)"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def reference_arm_ssd(args, world):
    """The SSD oracle as the reference arm: each step its bounded head sample."""
    from selective_state_space_112_b300.workloads import SSD_CONFIGS, make_ssd
    w = make_ssd(args.workload, **SSD_CONFIGS[args.workload])
    el = units = 0.0
    sample = None
    for i in range(args.steps):
        cb = cpu_baseline_ssd(w, budget_s=5.0)
        units_i = float(cb["sample"].split("(")[1].split(" ")[0])
        el += units_i / cb["value"]
        units += units_i
        sample, cores = cb["sample"], cb["cores"]
    value = units / el
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": args.workload, "layer": "Mamba-2 SSD", "batch": w.batch,
                      "seqlen": w.seqlen, "nheads": w.nheads, "headdim": w.headdim,
                      "ngroups": w.ngroups, "dstate": w.dstate},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": f"{sample}, per step"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
