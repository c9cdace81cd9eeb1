"""Benchmark of the displaced-patch layer step on GB300.

A step is one patch_layer_step (DPP_STALE with refresh) of the SDXL-1024
mid-level workload: bf16, B=2 (CFG halves), 64x64 map, C=640, P=4 row patches,
GroupNorm 32 groups, 10 heads x 64, conv3x3 640->640 -- GroupNorm with spliced
statistics, halo conv, QKV projection, stale-KV attention, output projection and
the compressed-residual refresh of K, V and the conv halo rows.

Timed region: W warm-up steps, then exactly K steps with a barrier and a device
synchronize on both sides; the L2 is flushed (a 256 MiB write, outside the step
events) before every timed step.  Each step's stage boundaries carry CUDA events
recorded on the launch stream inside the library, which gives the per-kernel
times used for the roofline lines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (test infrastructure) on the host cores on
a bounded sample of the same workload.  Prints one JSON line.
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

METRIC = "patch-layer steps/s; attention TFLOP/s & refresh GB/s as % of GB300 roofline"
# dram__bytes_read.sum + dram__bytes_write.sum per launch (median over the run's stale-step
# launches), from one ncu capture of this bench's own command with the current kernels
# (its summary is under profiles/); None where no capture of the current version
# exists.  Writes that are still in L2 when a kernel ends are not counted by the capture.
TRAFFIC = {
    "attention_sdxl1024_step": 52.55e6,
    "conv_sdxl1024_step": 29.40e6,
    "qkv_proj_sdxl1024_step": 13.02e6,
    "out_proj_sdxl1024_step": 11.33e6,
    "groupnorm_sdxl1024_step": 21.11e6,
    "refresh_sdxl1024_step": 44.16e6,
    "attention_sdxl3840": 983.3e6,
    "conv_vae_1x256x256x512": 93.44e6,
    "conv_sdxl3840_latent_step": 264.9e6,
    "refresh_sweep_200MiB": 684.6e6,
    "refresh_2x256x256x640_step": 1157.3e6,
    "groupnorm_2x240x240x640_step": 531.1e6,
}
WORKLOAD = "sdxl1024_mid_b2_64x64_c640_p4_bf16"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sus=m["bf16_tflops_sustained"],
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    lrank = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, lrank


class NvmlClockSampler:
    """Polls SM clock and clock-event reasons through NVML (read-only queries) every
    millisecond while the timed region runs; falls back to nvidia-smi sampling."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period_s: float = 0.001):
        self.index, self.period = index, period_s
        self.samples, self.reason_bits = [], 0
        self.max_mhz = None
        self.ok = False
        self.fallback = None

    def _setup(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        n = ctypes.c_uint(0)
        lib.nvmlDeviceGetCount_v2(ctypes.byref(n))
        h = ctypes.c_void_p()
        idx = 0 if n.value == 1 else self.index
        if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
            raise OSError("nvml handle")
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        try:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.lib, self.h = lib, h

    def _poll(self):
        import ctypes
        mhz = ctypes.c_uint(0)
        reasons = ctypes.c_ulonglong(0)
        while not self.stop:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if self.reasons_fn(self.h, ctypes.byref(reasons)) == 0:
                self.reason_bits |= reasons.value
            time.sleep(self.period)

    def __enter__(self):
        try:
            self._setup()
            self.stop = False
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            self.ok = True
        except Exception:
            self.fallback = ClockSampler(self.index).__enter__()
        return self

    def __exit__(self, *a):
        if self.ok:
            self.stop = True
            self.t.join(timeout=2)
        elif self.fallback:
            self.fallback.__exit__(*a)

    def summary(self):
        if not self.ok:
            out = self.fallback.summary() if self.fallback else {"reasons": ["unsampled"]}
            out["source"] = "nvidia-smi"
            return out
        reasons = sorted(v for k, v in self.REASONS.items() if self.reason_bits & k)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0, "source": "nvml"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml"}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(x: float, dev) -> float:
    """Max of a per-rank float over all ranks (the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(steps: int, world: int, max_total_ms: float) -> float:
    """Steps per second of the whole job: every rank ran `steps` steps, timed by the slowest."""
    return world * steps / (max_total_ms / 1e3)


def _roof(name, kernel, bound, work, ms, peaks, algorithmic):
    """One roofline row: algorithmic work per launch / the event-timed duration, against
    the measured burst peak (these kernels are timed in short runs), with the sustained
    tensor ratio beside it; traffic = ncu DRAM bytes per launch of the current version."""
    if bound == "hbm":
        ach = work / (ms * 1e-3) / 1e9
        row = {"name": name, "kernel": kernel, "bound": "hbm", "achieved": ach,
               "peak": peaks["hbm"], "unit": "GB/s", "frac": ach / peaks["hbm"],
               "peak_kind": f"HBM copy bandwidth, {peaks['src']}"}
    else:
        ach = work / (ms * 1e-3) / 1e12
        row = {"name": name, "kernel": kernel, "bound": "tensor", "achieved": ach,
               "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": ach / peaks["bf16"],
               "peak_kind": f"bf16 dense burst, {peaks['src']}",
               "frac_of_sustained": ach / peaks["bf16_sus"]}
    row.update({"traffic": TRAFFIC.get(name), "ms": ms, "algorithmic": algorithmic})
    return row


def _layer_setup(dev, fuse_gn=False, seed=0):
    import torch

    import stale_activations_gb300 as dpp
    import synth
    cfg = synth.SDXL1024_MID
    wts = synth.layer_weights(cfg, seed=seed)
    x, x_prev = synth.layer_inputs(cfg, seed=seed)
    prm = dpp.make_params(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G, cfg.heads, dpp.BF16,
                          refresh=True, eps=cfg.eps, fuse_gn=fuse_gn)
    state, ws = dpp.alloc_layer(prm, device=dev)
    wd = {k: v.to(dev) for k, v in wts.items()}
    xd, xpd = x.to(dev), x_prev.to(dev)
    out = torch.empty_like(xd)
    # the stale state of this step is what the synchronous step over x_prev leaves
    dpp.patch_layer_step(prm, wd, state, xpd, out, dpp.SYNC, ws)
    return cfg, prm, wd, state, ws, x, xd, out


def run_gpu(args):
    import torch
    import torch.distributed as tdist

    import stale_activations_gb300 as dpp

    ws_n, rank, lrank = _dist()
    torch.cuda.set_device(lrank)
    dev = torch.device("cuda", lrank)
    if ws_n > 1:
        tdist.init_process_group("nccl", device_id=dev)
    dpp.load()
    peaks = _peaks()
    cfg, prm, wd, state, wsb, x_host, xd, out = _layer_setup(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    nst = dpp.NUM_STAGE_EVENTS

    def step(evs=None):
        dpp.patch_layer_step(prm, wd, state, xd, out, dpp.STALE, wsb, stage_events=evs)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if dpp.read_device_status(wsb) != 0:
        raise RuntimeError("device status set during warm-up")

    K = args.steps
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(K)]
    for row in events:      # create the events (the library re-records them in the step)
        for e in row:
            e.record(stream)

    def barrier():
        if ws_n > 1:
            tdist.barrier()
        torch.cuda.synchronize()

    # The step time comes from one start/end event pair per step: events recorded
    # between the stages would keep each kernel from overlapping its predecessor's
    # tail (the kernels are launched as programmatic dependents).  A second pass
    # with per-stage events gives the breakdown.
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    with NvmlClockSampler(lrank) as clocks:
        barrier()
        t0 = time.perf_counter()
        for i in range(K):
            flush.fill_(1)
            step_ev[i][0].record(stream)
            step()
            step_ev[i][1].record(stream)
        barrier()
        wall = time.perf_counter() - t0
        for i in range(K):
            flush.fill_(1)
            step(events[i])
        barrier()
    st = dpp.read_device_status(wsb)
    if st != 0:
        raise RuntimeError(f"device status {st} in the timed region")
    stage_ms = [[events[i][s].elapsed_time(events[i][s + 1]) for s in range(nst - 1)]
                for i in range(K)]
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    tot_ms = reduce_max(sum(step_ms), dev)
    ms_per_step = tot_ms / K
    value = whole_job_rate(K, ws_n, tot_ms)

    # per-stage averages and the roofline of the dominant kernel (attention)
    avg = {name: sum(r[i] for r in stage_ms) / K for i, name in enumerate(dpp.STAGES)}
    B, L, C, P = cfg.B, cfg.L, cfg.C, cfg.P
    attn_flop = 4.0 * B * cfg.heads * L * L * cfg.head_dim
    conv_flop = 2.0 * B * L * C * 9 * C
    qkv_flop = 2.0 * B * L * C * 3 * C
    o_flop = 2.0 * B * L * C * C
    act = B * L * C
    # x read by the stats and the apply kernel, y written (at this size the stale V's
    # maximum for the attention's V range is taken by the conv, not by the GroupNorm)
    gn_bytes = 3 * act * 2
    halo_elems = B * (P - 1) * 2 * cfg.W * C
    refresh_elems = 2 * act + halo_elems
    refresh_bytes = 7.03125 * refresh_elems
    attn_tfs = attn_flop / (avg["attention"] * 1e-3) / 1e12
    kernels = {
        "groupnorm": {"ms": avg["groupnorm"], "GB/s": gn_bytes / (avg["groupnorm"] * 1e-3) / 1e9},
        "halo_conv": {"ms": avg["halo_conv"], "TFLOP/s": conv_flop / (avg["halo_conv"] * 1e-3) / 1e12},
        "qkv_proj": {"ms": avg["qkv_proj"], "TFLOP/s": qkv_flop / (avg["qkv_proj"] * 1e-3) / 1e12},
        "attention": {"ms": avg["attention"], "TFLOP/s": attn_tfs},
        "out_proj": {"ms": avg["out_proj"], "TFLOP/s": o_flop / (avg["out_proj"] * 1e-3) / 1e12},
        "state_update": {"ms": avg["state_update"],
                         "GB/s": refresh_bytes / (avg["state_update"] * 1e-3) / 1e9},
    }
    for k, v in kernels.items():
        if "GB/s" in v:
            v["frac_hbm"] = v["GB/s"] / peaks["hbm"]
        else:
            v["frac_bf16_sustained"] = v["TFLOP/s"] / peaks["bf16_sus"]
    roofline = _roof("attention_sdxl1024_step", "tc_attn_kernel (stale_kv_attention_split)",
                     "tensor", attn_flop, avg["attention"], peaks,
                     f"4*B*heads*L^2*d = {attn_flop:.4g} FLOP per launch (B=2, L=4096, 10 heads)")
    rows = [dict(roofline),
            _roof("conv_sdxl1024_step", "tc_gemm_kernel<conv> (halo_conv3x3)", "tensor",
                  conv_flop, avg["halo_conv"], peaks,
                  f"2*B*H*W*C*9*C = {conv_flop:.4g} FLOP (2x64x64, 640->640)"),
            _roof("qkv_proj_sdxl1024_step", "tc_gemm_kernel<linear>", "tensor", qkv_flop,
                  avg["qkv_proj"], peaks, f"2*M*3C*C = {qkv_flop:.4g} FLOP"),
            _roof("out_proj_sdxl1024_step", "tc_gemm_kernel<linear>", "tensor", o_flop,
                  avg["out_proj"], peaks, f"2*M*C*C = {o_flop:.4g} FLOP"),
            _roof("groupnorm_sdxl1024_step", "gn_stats_kernel + gn_apply_kernel", "hbm",
                  gn_bytes, avg["groupnorm"], peaks,
                  f"6 B per element x {act} = {gn_bytes:.4g} B: x read twice, y written "
                  "(latency-bound at 31 MB)"),
            _roof("refresh_sdxl1024_step", "refresh_kernel", "hbm", refresh_bytes,
                  avg["state_update"], peaks,
                  f"7.03125 B per element x {refresh_elems} = {refresh_bytes:.4g} B")]

    # End to end through the public API with host buffers (pinned), copies timed.
    # (1) latency: each step alone -- H2D of its input, the step, D2H of its output.
    x_pin = x_host.pin_memory()
    out_pin = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    lat_ms = 0.0
    for i in range(K):
        flush.fill_(1)
        e0.record(stream)
        xd.copy_(x_pin, non_blocking=True)
        step()
        out_pin[0].copy_(out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        lat_ms += e0.elapsed_time(e1)
    # (2) throughput: a serving loop with double-buffered device input/output; the
    # input of step i+1 is copied (copy stream) while step i computes, the output of
    # step i is read back after it.  Steps rotate over NI independent instances of the
    # layer (own weights, state and workspace; ~0.5 GB together, 4x L2), so that a step
    # finds its operands evicted by the steps in between, as in a network of layers,
    # instead of timing an L2 flush that is not part of the work.
    NI = 4
    inst = [(prm, wd, state, wsb)]
    for k in range(1, NI):
        _, prm_k, wd_k, state_k, ws_k, _, _, _ = _layer_setup(dev, seed=k)
        inst.append((prm_k, wd_k, state_k, ws_k))
    for _ in range(NI):  # warm each instance once
        for (pk, wk, sk, wsk) in inst:
            dpp.patch_layer_step(pk, wk, sk, xd, out, dpp.STALE, wsk)
    torch.cuda.synchronize()
    xds = [xd, torch.empty_like(xd)]
    outs = [out, torch.empty_like(out)]
    cstream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]    # input b on the device
    computed = [torch.cuda.Event() for _ in range(2)]  # step done with input b / output b
    drained = [torch.cuda.Event() for _ in range(2)]   # output b read back

    def step_io(i, xin, xout):
        pk, wk, sk, wsk = inst[i % NI]
        dpp.patch_layer_step(pk, wk, sk, xin, xout, dpp.STALE, wsk)

    barrier()
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0e.record(stream)
    cstream.wait_stream(stream)
    with torch.cuda.stream(cstream):
        xds[0].copy_(x_pin, non_blocking=True)
        copied[0].record(cstream)
    for i in range(K):
        b = i % 2
        if i + 1 < K:  # next input, once step i-1 no longer reads its buffer
            with torch.cuda.stream(cstream):
                if i >= 1:
                    cstream.wait_event(computed[1 - b])
                xds[1 - b].copy_(x_pin, non_blocking=True)
                copied[1 - b].record(cstream)
        stream.wait_event(copied[b])
        if i >= 2:  # output buffer b was step i-2's: read back by now
            stream.wait_event(drained[b])
        step_io(i, xds[b], outs[b])
        computed[b].record(stream)
        with torch.cuda.stream(cstream):
            cstream.wait_event(computed[b])
            out_pin[b].copy_(outs[b], non_blocking=True)
            drained[b].record(cstream)
    stream.wait_stream(cstream)
    t1e.record(stream)
    t1e.synchronize()
    if any(dpp.read_device_status(w) != 0 for (_, _, _, w) in inst):
        raise RuntimeError("device status set in the end-to-end loop")
    e2e_ms = reduce_max(t0e.elapsed_time(t1e), dev)
    lat_ms = reduce_max(lat_ms, dev)
    e2e = {"value": whole_job_rate(K, ws_n, e2e_ms), "unit": "steps/s",
           "h2d_bytes_per_step": x_pin.numel() * x_pin.element_size(),
           "d2h_bytes_per_step": out_pin[0].numel() * out_pin[0].element_size(),
           "mode": "serving loop: copies of step i+1 / i-1 overlap step i (copy stream, "
                   "double-buffered device input and output); steps rotate over 4 "
                   "independent instances of the layer (working set ~0.5 GB, 4x L2: "
                   "operands cold, no flush)",
           "latency_ms_per_step": lat_ms / K,
           "latency_note": "one step alone: H2D, step, D2H on one stream, flush outside"}

    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": ws_n, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": cfg.H, "W": cfg.W, "C": C, "P": P,
                   "G": cfg.G, "heads": cfg.heads, "head_dim": cfg.head_dim,
                   "mode": "DPP_STALE+refresh", "parallelism": f"replicas x{ws_n}",
                   "l2": "flushed (256 MiB write) before every timed step"},
        "roofline": roofline, "kernels": kernels, "e2e": e2e,
        "gpu_launches": dpp.layer_kernel_count(prm, dpp.STALE) * K,
        "wall_s_timed_region": wall,
        "ms_per_step_with_stage_events": statistics.mean(
            events[i][0].elapsed_time(events[i][nst - 1]) for i in range(K)),
    }
    line["clocks"] = clocks.summary()
    if not args.no_secondary:
        a3840 = measure_attention_3840(dev, peaks)
        sweep = measure_refresh_sweep(dev, peaks)
        big = measure_large_layer(dev, peaks)
        lat = measure_large_layer(dev, peaks, H=240, W=240)
        vae = measure_vae_conv(dev, peaks)
        line["secondary"] = {"attention_sdxl3840": a3840, "refresh_sweep": sweep,
                             "layer_2x256x256x640_p8": big,
                             "layer_sdxl3840_2x240x240x640_p8": lat,
                             "halo_conv_vae": vae,
                             "tiny_f32_step": measure_tiny_f32(dev),
                             "otil_exchange_2x4x128x128_p4": measure_otil(dev),
                             "layer_fusions": measure_fusions(dev)}
        rows += [
            _roof("attention_sdxl3840", "tc_attn_kernel (stale_kv_attention_split)", "tensor",
                  a3840["flop_per_launch"], a3840["ms_mean"], peaks,
                  "4*B*heads*L^2*d, B=2, L=57600, 10 heads, P=8 (standalone launches)"),
            _roof("conv_vae_1x256x256x512", "tc_gemm_kernel<conv>", "tensor",
                  vae["flop_per_launch"], vae["ms_mean"], peaks,
                  "2*H*W*C*9*C, 1x256x256, 512->512, P=8 (standalone, L2 flushed)"),
            _roof("conv_sdxl3840_latent_step", "tc_gemm_kernel<conv, padded row tiles>",
                  "tensor", lat["conv_flop"], lat["stage_ms"]["halo_conv"], peaks,
                  "2*B*H*W*C*9*C, 2x240x240, 640->640, P=8 (W=240: tiles of 120 pixels of "
                  "one row)"),
            _roof("refresh_sweep_200MiB", "refresh_kernel", "hbm", sweep["bytes_per_launch"],
                  sweep["ms_mean"], peaks,
                  "7.03125 B per element x 104988672 (standalone, L2 flushed)"),
            _roof("refresh_2x256x256x640_step", "refresh_kernel", "hbm", big["refresh_bytes"],
                  big["stage_ms"]["state_update"], peaks,
                  "7.03125 B per element x (K, V, halo rows) of a 2x256x256x640 P=8 step"),
            _roof("groupnorm_2x240x240x640_step", "gn_stats_kernel + gn_apply_kernel", "hbm",
                  lat["groupnorm_bytes"], lat["stage_ms"]["groupnorm"], peaks,
                  "8 B per element x 2x240x240x640 (stats read, apply read + write, stale V "
                  "read for the attention's V range)"),
        ]
    line["roofline"]["kernels"] = rows
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_budget_s)
        if not args.no_oracle_plan:
            line["cpu_baseline"]["plan"] = cpu_oracle_plan()
    if ws_n > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def _randn_bf16(shape, gen, dev):
    import torch
    return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)


def measure_attention_3840(dev, peaks, iters=5):
    """The attention alone at the SDXL-3840 attention level: B=2, L=57600, 10 heads x 64,
    P=8; K/V_stale = fresh + N(0, 0.05^2).  Inputs (0.74 GB) exceed L2.  Timed with the
    split schedule the layer step uses (stale_kv_attention_split, attention + merge) and
    with whole units per CTA (stale_kv_attention)."""
    import torch

    import stale_activations_gb300 as dpp
    B, L, heads, P = 2, 57600, 10, 8
    g = torch.Generator(device=dev).manual_seed(1)
    q, kf, vf = (_randn_bf16((B, L, 640), g, dev) for _ in range(3))
    ks = (kf.float() + 0.05 * torch.randn(kf.shape, generator=g, device=dev)).to(torch.bfloat16)
    vs = (vf.float() + 0.05 * torch.randn(vf.shape, generator=g, device=dev)).to(torch.bfloat16)
    o = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    scratch = {sp: torch.empty(dpp.attention_scratch_size(B, L, heads, P, split=sp),
                               dtype=torch.uint8, device=dev) for sp in (True, False)}
    flop = 4.0 * B * heads * L * L * 64

    def run(split):
        if split:
            dpp.stale_kv_attention_split(q, kf, vf, ks, vs, o, heads, P, scratch=scratch[True],
                                         dev_status=st)
        else:
            dpp.stale_kv_attention(q, kf, vf, ks, vs, o, heads, P, scratch=scratch[False],
                                   dev_status=st)

    res = {}
    for split in (True, False):
        for _ in range(2):
            run(split)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
        torch.cuda.synchronize()
        ev[0].record()
        for i in range(iters):
            run(split)
            ev[i + 1].record()
        torch.cuda.synchronize()
        if st.item() != 0:
            raise RuntimeError("attention device status set")
        ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(iters)]
        res[split] = (statistics.mean(ms), min(ms), flop / (statistics.mean(ms) * 1e-3) / 1e12)
    ms_mean, ms_min, tfs = res[True]
    return {"ms_mean": ms_mean, "ms_min": ms_min, "TFLOP/s": tfs,
            "frac_of_burst_bf16": tfs / peaks["bf16"], "peak_burst": peaks["bf16"],
            "frac_of_sustained_bf16": tfs / peaks["bf16_sus"], "flop_per_launch": flop,
            "launches": iters, "schedule": "split (cut units merged inside the attention kernel)",
            "whole_units": {"ms_mean": res[False][0], "TFLOP/s": res[False][2]},
            "note": "back-to-back launches, inputs > L2"}


def measure_refresh_sweep(dev, peaks, iters=5):
    """refresh_residual alone over 200 MiB of bf16 stale buffers + the 2x4x128x128 noise
    prediction (one flat buffer); stale restored and L2 flushed before each launch."""
    import torch

    import stale_activations_gb300 as dpp
    n = 200 * 1024 * 1024 // 2 + 2 * 4 * 128 * 128
    g = torch.Generator(device=dev).manual_seed(2)
    stale0 = _randn_bf16((n,), g, dev)
    nblk = n // 128
    spike = (torch.rand(nblk, generator=g, device=dev) < 0.1).repeat_interleave(128)
    std = torch.where(spike, 1.0, 0.05)
    fresh = (stale0.float() + std * torch.randn(n, generator=g, device=dev)).to(torch.bfloat16)
    del spike, std
    stale = torch.empty_like(stale0)
    codes = torch.empty(n, dtype=torch.int8, device=dev)
    scales = torch.empty(nblk, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ms = []
    for i in range(iters + 2):
        stale.copy_(stale0)
        flush.fill_(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dpp.refresh_residual(fresh, stale, codes, scales)
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            ms.append(e0.elapsed_time(e1))
    nbytes = 7.03125 * n
    gbs = nbytes / (statistics.mean(ms) * 1e-3) / 1e9
    return {"ms_mean": statistics.mean(ms), "ms_min": min(ms), "GB/s": gbs,
            "frac_hbm": gbs / peaks["hbm"], "peak_hbm": peaks["hbm"], "elements": n,
            "bytes_per_launch": nbytes, "launches": iters}


def measure_vae_conv(dev, peaks, iters=5):
    """halo_conv3x3 alone at the VAE-decoder-like size: 1x256x256x512 -> 512, P=8 row
    bands with stale halo rows (inputs 64 MiB each; L2 flushed before each launch)."""
    import torch

    import stale_activations_gb300 as dpp
    B, H, W, C, P = 1, 256, 256, 512, 8
    g = torch.Generator(device=dev).manual_seed(4)
    y = _randn_bf16((B, H, W, C), g, dev)
    ys = (y.float() + 0.05 * torch.randn(y.shape, generator=g, device=dev)).to(torch.bfloat16)
    w = (0.02 * torch.randn(C, 3, 3, C, generator=g, device=dev)).to(torch.bfloat16)
    out = torch.empty_like(y)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    ms = []
    for i in range(iters + 2):
        flush.fill_(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dpp.halo_conv3x3(y, ys, w, out, P, dev_status=st)
        e1.record()
        torch.cuda.synchronize()
        if i >= 2:
            ms.append(e0.elapsed_time(e1))
    if st.item() != 0:
        raise RuntimeError("conv device status set")
    flop = 2.0 * B * H * W * C * 9 * C
    tfs = flop / (statistics.mean(ms) * 1e-3) / 1e12
    return {"ms_mean": statistics.mean(ms), "ms_min": min(ms), "TFLOP/s": tfs,
            "frac_of_sustained_bf16": tfs / peaks["bf16_sus"], "flop_per_launch": flop,
            "launches": iters}


def measure_tiny_f32(dev, iters=50):
    """The tiny fp32 workload's layer step on the GPU (1x32x32x64, P=2, G=8, one head,
    fp32 SIMT kernels): steps/s of back-to-back STALE steps with refresh."""
    import torch

    import stale_activations_gb300 as dpp
    import synth
    cfg = synth.TINY_F32
    prm = dpp.make_params(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G, cfg.heads, dpp.F32,
                          refresh=True, eps=cfg.eps)
    wts = {k: v.to(dev) for k, v in synth.layer_weights(cfg, seed=0).items()}
    x, x_prev = (t.to(dev) for t in synth.layer_inputs(cfg, seed=0))
    state, ws = dpp.alloc_layer(prm, device=dev)
    out = torch.empty_like(x)
    dpp.patch_layer_step(prm, wts, state, x_prev, out, dpp.SYNC, ws)
    for _ in range(5):
        dpp.patch_layer_step(prm, wts, state, x, out, dpp.STALE, ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(iters):
        dpp.patch_layer_step(prm, wts, state, x, out, dpp.STALE, ws)
    e1.record()
    torch.cuda.synchronize()
    if dpp.read_device_status(ws) != 0:
        raise RuntimeError("device status set in the tiny fp32 steps")
    ms = e0.elapsed_time(e1) / iters
    return {"workload": cfg.name, "ms_per_step": ms, "steps/s": 1e3 / ms,
            "note": "back-to-back steps, launch-bound at this size"}


def measure_otil(dev, iters=20):
    """The OTIL exchange alone at the pages' noise-prediction shape: [2, 4, 128, 128]
    bf16, P = 4 ranks, 8 x 32 sub-blocks (K = 16 per band), k = 4 sent per rank and
    step: one dpp_otil_step (score, select, pack, copy to the other ranks) per launch."""
    import torch

    import stale_activations_gb300 as dpp
    B, C, H, W, P, bh, bw, k = 2, 4, 128, 128, 4, 8, 32, 4
    prm = dpp.otil_params(B, C, H, W, P, bh, bw, k, dpp.BF16)
    g = torch.Generator(device=dev).manual_seed(5)
    xs = [torch.randn(B, C, H, W, generator=g, device=dev).to(torch.bfloat16) for _ in range(4)]
    st = dpp.otil_alloc(prm, xs[0], device=dev)
    for i in range(3):
        dpp.otil_step(prm, xs[i % 4], st)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(iters + 1)]
    torch.cuda.synchronize()
    ev[0].record()
    for i in range(iters):
        dpp.otil_step(prm, xs[i % 4], st)
        ev[i + 1].record()
    torch.cuda.synchronize()
    ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(iters)]
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    dpp.otil_finalize(prm, xs[0], st, reset=True)
    f1.record()
    torch.cuda.synchronize()
    return {"ms_per_step": statistics.median(ms), "finalize_ms": f0.elapsed_time(f1),
            "sent_bytes_per_step": P * k * B * C * bh * bw * 2,
            "note": "back-to-back exchange steps (launch-bound at this size)"}


def measure_fusions(dev, iters=20):
    """The headline layer step in its four arrangements, same workload and L2 flush:
    the default; the GroupNorm apply fused into the conv's operand path (fuse_gn); the
    new state written to a second set (swapped after each step) by the separate refresh
    pass; and that with the K/V refresh in the projection epilogue (fuse_refresh)."""
    import torch

    import stale_activations_gb300 as dpp
    res = {}
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for name, fuse_gn, dbuf, frx in (("separate", False, False, False),
                                     ("fuse_gn", True, False, False),
                                     ("second_state", False, True, False),
                                     ("second_state_fuse_refresh", False, True, True)):
        cfg, prm, wd, state, ws, _, xd, out = _layer_setup(dev, fuse_gn=fuse_gn)
        prm.fuse_refresh = 1 if frx else 0
        if dbuf:
            st2, _ = dpp.alloc_layer(prm, device=dev, double_buffer=True)
            for k in dpp.STATE_KEYS:
                st2[k].copy_(state[k])
            st2["codes"], st2["scales"] = state["codes"], state["scales"]
            state = st2

        def step(evs=None):
            dpp.patch_layer_step(prm, wd, state, xd, out, dpp.STALE, ws, stage_events=evs)
            if dbuf:
                dpp.swap_state(state)

        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(dpp.NUM_STAGE_EVENTS)]
               for _ in range(iters)]
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(iters)]
        for row in evs:
            for e in row:
                e.record()
        for _ in range(3):
            flush.fill_(1)
            step()
        for i in range(iters):
            flush.fill_(1)
            pairs[i][0].record()
            step()
            pairs[i][1].record()
        for i in range(iters):
            flush.fill_(1)
            step(evs[i])
        torch.cuda.synchronize()
        if dpp.read_device_status(ws) != 0:
            raise RuntimeError(f"device status set in the {name} arrangement")
        res[name] = {
            "ms_per_step": statistics.median(a.elapsed_time(b) for a, b in pairs),
            "stage_ms": {n: statistics.median(evs[i][k].elapsed_time(evs[i][k + 1])
                                              for i in range(iters))
                         for k, n in enumerate(dpp.STAGES)}}
        del state, ws
    return res


def measure_large_layer(dev, peaks, iters=3, H=256, W=256):
    """One STALE layer step on a map larger than L2 (B=2, HxW = 256x256 or the SDXL-3840
    latent 240x240, C=640, P=8, 10 heads): the GroupNorm and refresh stages as HBM
    streams, with per-stage CUDA events."""
    import torch

    import stale_activations_gb300 as dpp
    B, C, P, G, heads = 2, 640, 8, 32, 10
    prm = dpp.make_params(B, H, W, C, P, G, heads, dpp.BF16, refresh=True)
    state, ws = dpp.alloc_layer(prm, device=dev)
    g = torch.Generator(device=dev).manual_seed(3)
    wts = {"gamma": torch.ones(C, device=dev), "beta": torch.zeros(C, device=dev),
           "w_conv": (0.02 * torch.randn(C, 3, 3, C, generator=g, device=dev)).to(torch.bfloat16),
           "w_qkv": (0.02 * torch.randn(3 * C, C, generator=g, device=dev)).to(torch.bfloat16),
           "w_o": (0.02 * torch.randn(C, C, generator=g, device=dev)).to(torch.bfloat16)}
    x = _randn_bf16((B, H, W, C), g, dev)
    xp = (x.float() + 0.05 * torch.randn(x.shape, generator=g, device=dev)).to(torch.bfloat16)
    out = torch.empty_like(x)
    dpp.patch_layer_step(prm, wts, state, xp, out, dpp.SYNC, ws)
    dpp.patch_layer_step(prm, wts, state, x, out, dpp.STALE, ws)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(dpp.NUM_STAGE_EVENTS)]
           for _ in range(iters)]
    for row in evs:
        for e in row:
            e.record()
    for i in range(iters):
        dpp.patch_layer_step(prm, wts, state, x, out, dpp.STALE, ws, stage_events=evs[i])
    torch.cuda.synchronize()
    if dpp.read_device_status(ws) != 0:
        raise RuntimeError("device status set in the large layer")
    avg = {n: sum(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(iters)) / iters
           for k, n in enumerate(dpp.STAGES)}
    act = B * H * W * C
    L = H * W
    gn_gbs = 4 * act * 2 / (avg["groupnorm"] * 1e-3) / 1e9
    ref_bytes = 7.03125 * (2 * act + B * (P - 1) * 2 * W * C)
    ref_gbs = ref_bytes / (avg["state_update"] * 1e-3) / 1e9
    attn_tfs = 4.0 * B * heads * L * L * 64 / (avg["attention"] * 1e-3) / 1e12
    conv_tfs = 2.0 * B * L * C * 9 * C / (avg["halo_conv"] * 1e-3) / 1e12
    step_ms = sum(avg.values())
    return {"ms_per_step": step_ms, "stage_ms": avg, "groupnorm_bytes": 4 * act * 2,
            "refresh_bytes": ref_bytes, "conv_flop": 2.0 * B * L * C * 9 * C,
            "groupnorm_GB/s": gn_gbs, "groupnorm_frac_hbm": gn_gbs / peaks["hbm"],
            "refresh_GB/s": ref_gbs, "refresh_frac_hbm": ref_gbs / peaks["hbm"],
            "attention_TFLOP/s": attn_tfs, "conv_TFLOP/s": conv_tfs,
            "note": "GroupNorm algorithmic bytes 8 B/elem (stats read, apply read+write, stale V "
                    "read for the attention's V range)"}


# ------------------------------------------------------------------ CPU oracle (reference arm)
def _oracle_case():
    import numpy as np

    import oracle
    import synth
    cfg = synth.SDXL1024_MID
    wts = synth.layer_weights(cfg, seed=0)
    x, x_prev = synth.layer_inputs(cfg, seed=0)
    wn = {k: v.double().numpy() for k, v in wts.items()}
    st0 = oracle.empty_state(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G)
    _, state, _, _ = oracle.patch_layer_step(x_prev.double().numpy(), st0, wn, cfg.P, cfg.G,
                                             cfg.heads, cfg.eps, "bf16", oracle.SYNC)
    return cfg, wn, np.asarray(x.double().numpy()), state


def _oracle_step(case):
    import oracle
    cfg, wn, x, state = case
    return oracle.patch_layer_step(x, state, wn, cfg.P, cfg.G, cfg.heads, cfg.eps, "bf16",
                                   oracle.STALE, refresh=True)


def cpu_baseline(budget_s: float):
    """The oracle, as it is, on this host: whole STALE layer steps of the same
    workload, as many as fit in the budget (at least one)."""
    case = _oracle_case()
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(case)
        n += 1
        el = time.perf_counter() - t0
        if el > budget_s or n >= 3:
            break
    return {"value": n / el, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} full oracle layer step(s) of {WORKLOAD} (numpy fp64 with its BLAS "
                      f"threads + C refresh), {el:.1f} s"}


def _oracle_plan_child(threads: str):
    """Runs in a fresh process whose BLAS/OpenMP thread counts the parent set: times the
    oracle on each of the five workloads (bounded samples where a full run takes minutes)
    and prints one JSON object."""
    import numpy as np

    import oracle
    import synth
    out = {"threads": threads}

    def np64(t):
        return t.double().numpy()

    # tiny fp32 layer step, in full
    cfg = synth.TINY_F32
    wn = {k: np64(v) for k, v in synth.layer_weights(cfg, seed=0).items()}
    x, xp = synth.layer_inputs(cfg, seed=0)
    st = oracle.empty_state(cfg.B, cfg.H, cfg.W, cfg.C, cfg.P, cfg.G)
    _, st, _, _ = oracle.patch_layer_step(np64(xp), st, wn, cfg.P, cfg.G, cfg.heads, cfg.eps,
                                          "f32", oracle.SYNC)
    n, t0 = 0, time.perf_counter()
    while n < 20 and (n == 0 or time.perf_counter() - t0 < 2.0):
        oracle.patch_layer_step(np64(x), st, wn, cfg.P, cfg.G, cfg.heads, cfg.eps, "f32",
                                oracle.STALE)
        n += 1
    el = time.perf_counter() - t0
    out["tiny_f32_step"] = {"value": n / el, "unit": "steps/s", "s": el,
                            "sample": f"{n} full STALE steps with refresh"}
    # the SDXL-1024 layer step: timed in the parent with all cores; one step here with one
    if threads == "1":
        case = _oracle_case()
        t0 = time.perf_counter()
        _oracle_step(case)
        el = time.perf_counter() - t0
        out["sdxl1024_step"] = {"value": 1 / el, "unit": "steps/s", "s": el,
                                "sample": "one full STALE step with refresh"}
    # SDXL-3840 attention: 256 query rows per (patch, head), keys and values in full, then
    # extrapolated to all 2 x 57600 rows of all 10 heads (rows are independent)
    B, L, heads, P = 2, 57600, 10, 8
    hs = heads if threads != "1" else 1  # one head on one thread (extrapolated over heads)
    Lp = L // P
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([p * Lp + rng.choice(Lp, 256, replace=False)
                                   for p in range(P)]))
    gen = [oracle.to_storage(np64(synth.normal((1, L, hs * 64), 0, t)), "bf16")
           for t in ("q", "k", "v", "k_noise", "v_noise")]
    t0 = time.perf_counter()
    oracle.stale_kv_attention(gen[0], gen[1], gen[2], gen[3], gen[4], hs, P, "bf16", rows=rows)
    el = time.perf_counter() - t0
    scale = (B * L * heads) / (len(rows) * hs)
    flop = 4.0 * B * heads * L * L * 64
    out["sdxl3840_attention"] = {
        "value": flop / (el * scale) / 1e12, "unit": "TFLOP/s", "s": el,
        "s_per_launch_extrapolated": el * scale,
        "sample": f"{len(rows)} query rows (256 per patch) x {hs} head(s) of batch 0 over all "
                  f"57600 keys; extrapolated x{scale:.0f} to the full launch (rows independent)"}
    # VAE-sized halo conv, in full
    yf, ys, w = synth.conv_inputs(1, 256, 256, 512, 512, "bf16", seed=0)
    a, b, c = np64(yf), np64(ys), np64(w)
    t0 = time.perf_counter()
    oracle.halo_conv3x3(a, b, c, 8, "bf16")
    el = time.perf_counter() - t0
    out["vae_conv_1x256x256x512"] = {"value": 2.0 * 65536 * 512 * 9 * 512 / el / 1e12,
                                     "unit": "TFLOP/s", "s": el, "sample": "one full conv"}
    # 200 MiB refresh sweep, in full (exact fp32 C code, OpenMP over blocks)
    f, s_ = synth.refresh_sweep_inputs(seed=0)
    f64, s64 = np64(f), np64(s_)
    del f, s_
    t0 = time.perf_counter()
    oracle.refresh_residual(f64, s64, "bf16")
    el = time.perf_counter() - t0
    out["refresh_sweep_200MiB"] = {"value": 7.03125 * f64.size / el / 1e9, "unit": "GB/s",
                                   "s": el, "sample": "one full sweep (104988672 elements)"}
    print(json.dumps(out))


def cpu_oracle_plan():
    """The oracle on this host's cores for the five workloads, with every core and with
    one thread (BLAS and OpenMP thread counts fixed before numpy loads, in a fresh
    process each)."""
    import subprocess
    res = {"nproc": os.cpu_count()}
    for threads in ("all", "1"):
        env = dict(os.environ)
        if threads == "1":
            env.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-plan-child",
                            threads], env=env, capture_output=True, text=True, timeout=900)
        if r.returncode != 0:
            res[threads] = {"error": r.stderr.strip().splitlines()[-1:]}
            continue
        res["all_cores" if threads == "all" else "single_thread"] = json.loads(
            r.stdout.strip().splitlines()[-1])
    return res


def run_reference(args):
    ws_n, rank, _ = _dist()
    if rank != 0:
        return
    case = _oracle_case()
    for _ in range(args.warmup if args.warmup < 1 else 1):
        _oracle_step(case)
    K = args.steps
    t0 = time.perf_counter()
    for _ in range(K):
        _oracle_step(case)
    el = time.perf_counter() - t0
    v = K / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": ws_n,
            "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * el / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": 2, "H": 64, "W": 64, "C": 640, "P": 4,
                       "G": 32, "heads": 10, "head_dim": 64, "mode": "DPP_STALE+refresh"},
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{K} full oracle layer steps (one warm-up), {el:.1f} s"},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


ONLY = {
    "attention_sdxl3840": lambda dev, peaks: measure_attention_3840(dev, peaks),
    "refresh_sweep": lambda dev, peaks: measure_refresh_sweep(dev, peaks),
    "layer_2x256x256x640": lambda dev, peaks: measure_large_layer(dev, peaks),
    "layer_sdxl3840_2x240x240x640": lambda dev, peaks: measure_large_layer(dev, peaks, H=240,
                                                                           W=240),
    "halo_conv_vae": lambda dev, peaks: measure_vae_conv(dev, peaks),
}


def run_only(name):
    import torch

    import stale_activations_gb300 as dpp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dpp.load()
    res = ONLY[name](dev, _peaks())
    print(json.dumps({"only": name, **res}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the standalone SDXL-3840 attention and refresh-sweep lines")
    ap.add_argument("--no-oracle-plan", action="store_true",
                    help="skip the oracle timings of the five workloads on the host cores")
    ap.add_argument("--oracle-plan-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--only", default=None, choices=sorted(ONLY),
                    help="run one secondary measurement alone and print its line (for "
                         "profiling one workload's kernels; no headline line)")
    args = ap.parse_args()
    if args.only:
        run_only(args.only)
        return
    if args.oracle_plan_child:
        _oracle_plan_child(args.oracle_plan_child)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
