"""Benchmark of the fused GEMM + epilogue path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch of synthetic input:
the large linear-layer pair at fp16 with fp32 accumulation --
  forward  RELU_AUX_BIAS  Y = ReLU(X W + bias), relu_aux    X[65536,16384] W[16384,8192]
  backward DRELU_BGRAD    dZ = (dY W^T) masked, bgrad      dY[65536,8192], mask [65536,16384]
(the fp16 (65536,16384) x (16384,8192) workload of "Fusing Matmul Epilogs
with nvmath-python", section "Suitable evaluation scenarios"). Inputs are
seeded synthetic draws (synth) already resident in HBM; every operand is far
larger than L2, so no flush is needed between steps.

Prints one JSON line: throughput in TFLOP/s (2*M*N*K per GEMM), % of the
dense fp16/bf16 peak, the dominant kernel's roofline, the CPU oracle as a
timed baseline, an end-to-end figure through the C ABI from pinned host
buffers, and the epilogue's overhead against the same kernel with no
epilogue. ``--impl reference`` times the CPU oracle on the same workload.
Several GPUs run independent replicas (the path has no exchange step).
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

M, K, N = 65536, 16384, 8192  # forward X[M,K] . W[K,N]; backward dY[M,N] . W^T -> [M,K]
WORKLOAD = "linear_pair_fp16_fwd_relu_aux_bias_bwd_drelu_bgrad_65536x16384x8192"
METRIC = "fused GEMM+epilogue TFLOP/s and % of GB300 FP16/BF16 dense peak, 1 GPU"
FLOP_PER_GEMM = 2.0 * M * N * K
FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles",
                               "gemm_epilog_pair_kernel_wide_fp16_16384_rows_dram_traffic.md")


def kernel_sources_sha256() -> str:
    """Digest of the kernel sources: a recorded ncu traffic figure is only
    reported while the kernels it was measured on are unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_epilogue_tmem_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic():
    """(fwd, bwd) DRAM bytes per launch from the committed ncu summary, or
    None when it is missing or was taken on other kernel sources."""
    if not os.path.exists(TRAFFIC_PROFILE):
        return None
    vals = {}
    with open(TRAFFIC_PROFILE) as f:
        for line in f:
            line = line.strip().strip("`")
            if ":" in line and line.split(":")[0] in ("sources_sha256", "fwd_bytes_per_launch",
                                                      "bwd_bytes_per_launch"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("sources_sha256") != kernel_sources_sha256():
        return None
    try:
        return float(vals["fwd_bytes_per_launch"]), float(vals["bwd_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def max_over_ranks(value: float, device) -> float:
    """The largest value over the ranks of the default process group (the
    slowest replica's time bounds the job)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines: list[str] = []
        self.times: list[float] = []  # time.monotonic() when each sample arrived

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.times.append(time.monotonic())
            self.lines.append(line.strip())

    def keep_from(self, n: int):
        """Drop the first n samples."""
        self.lines, self.times = self.lines[n:], self.times[n:]

    def stop(self, window=None) -> dict:
        """Median clock, power and the throttle reasons seen, over the samples
        that arrived within window = (t0, t1) of time.monotonic() (all
        samples when None)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln, t in zip(self.lines, self.times):
            if window is not None and not window[0] <= t <= window[1]:
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "power_w_median": statistics.median(power) if power else None,
               "samples": len(sm), "reasons": sorted(reasons)}
        if window is not None:
            out["sampled"] = "only while the timed loop ran"
            if not sm:
                out["note"] = ("the timed region (%.0f ms) is shorter than the 200 ms sampling "
                               "interval; the steady-state comparison has sampled clocks"
                               % (1e3 * (window[1] - window[0])))
        return out


def pick_peak(pk: dict, pk_kind: str, busy_s: float):
    """The dense bf16/fp16 peak a kernel is held against: the burst figure
    when the GPU was busy for under 2 s around the measurement (the clock has
    not settled at the power cap yet), the sustained one for longer runs.
    Returns (peak TFLOP/s, description)."""
    key = "bf16_tflops_sustained" if busy_s >= 2.0 else "bf16_tflops"
    if key not in pk:
        key = "bf16_tflops"
    return float(pk[key]), f"{pk_kind} {key} (GPU busy {busy_s:.1f} s around the measurement)"


def stats_ms(times: list) -> dict:
    return {"median": statistics.median(times), "min": min(times),
            "mean": statistics.mean(times), "n": len(times)}


def sustained_windows(torch, fns: dict, seconds: float, rounds: int, gpu: int,
                      group: int = 4) -> dict:
    """Steady-state time of each function: the functions take turns, `rounds`
    times, each running back to back for `seconds` (launches timed in groups
    of `group` between CUDA events on the current stream) while nvidia-smi
    samples the SM clock. Per function: median and minimum ms per call over
    all groups, and the median SM clock of its windows, so that time x clock
    (cycles) can be compared between functions that ran at different clocks
    under the power cap. Each function runs once untimed first."""
    for fn in fns.values():
        fn()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu)
    sampler.start()
    times = {k: [] for k in fns}
    mhz = {k: [] for k in fns}
    t_busy = time.time()
    for _ in range(rounds):
        for name, fn in fns.items():
            n0 = len(sampler.lines)
            evs = []
            t_end = time.time() + seconds
            while time.time() < t_end:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(group):
                    fn()
                b.record()
                evs.append((a, b))
                if len(evs) % 4 == 0:
                    b.synchronize()
            torch.cuda.synchronize()
            times[name] += [a.elapsed_time(b) / group for a, b in evs]
            for ln in sampler.lines[n0:]:
                parts = [x.strip() for x in ln.split(",")]
                try:
                    mhz[name].append(float(parts[1]))
                except (IndexError, ValueError):
                    pass
    busy = time.time() - t_busy
    clk = sampler.stop()
    out = {}
    for name in fns:
        med = statistics.median(times[name])
        f = statistics.median(mhz[name]) if mhz[name] else None
        out[name] = {"ms_median": med, "ms_min": min(times[name]), "calls": len(times[name]) * group,
                     "sm_mhz": f, "mcycles": med * 1e-3 * f if f else None}
    return {"per_fn": out, "clocks": clk, "busy_s": busy}


# --------------------------------------------------------------- CPU oracle leg
_ORACLE_INPUTS = {}


def _oracle_inputs():
    """Host copies of the step's weight, bias and backward mask (generated once)."""
    if not _ORACLE_INPUTS:
        t0 = time.time()
        _ORACLE_INPUTS["W"] = synth.normal((K, N), synth.F16, 0, synth.TID_B, 1 / 128)
        _ORACLE_INPUTS["bias"] = synth.normal((N,), synth.F16, 0, synth.TID_BIAS, 0.1)
        _ORACLE_INPUTS["words"] = synth.mask_words(M, K, 0)  # backward mask, [M/32, K]
        _ORACLE_INPUTS["rows"] = synth.sample_rows(M, 64, 0)
        _ORACLE_INPUTS["gen_s"] = time.time() - t0
    return _ORACLE_INPUTS


def oracle_sample(rows_fwd: int, rows_bwd: int, nthreads: int, offset: int = 0,
                  outputs: dict | None = None):
    """Run the CPU oracle on sampled rows of both GEMMs of one step (full N,
    full K). Returns (flops done, seconds of oracle work, description); with
    `outputs` given, also leaves there the rows' ids and the oracle's Y, z
    (pre-activation) and dZ."""
    import oracle
    inp = _oracle_inputs()
    rows = inp["rows"]
    rf = np.roll(rows, -offset)[:rows_fwd]
    rb = np.roll(rows, -offset)[:rows_bwd]
    X = synth.normal((M, K), synth.F16, 0, synth.TID_A, 1.0, rows=rf)
    dY = synth.normal((M, N), synth.F16, 0, synth.TID_DY, 1.0, rows=rb)
    t0 = time.time()
    y_o, z_o = oracle.relu_bias(X, inp["W"], inp["bias"], oracle.F16, oracle.B_KN,
                                oracle.BIAS_COL, row_ids=rf, nthreads=nthreads)
    # backward: dY . W^T, W [K, N] being the [n, k] storage of B = W^T
    dz_o, _, _ = oracle.drelu_bgrad(dY, inp["W"], inp["words"], oracle.F16, oracle.B_NK,
                                    row_ids=rb, nthreads=nthreads)
    sec = time.time() - t0
    if outputs is not None:
        outputs.update(rows_fwd=rf, rows_bwd=rb, Y=oracle.decode(y_o, oracle.F16), z=z_o,
                       dZ=oracle.decode(dz_o, oracle.F16))
    flops = 2.0 * len(rf) * N * K + 2.0 * len(rb) * K * N
    desc = (f"{len(rf)} sampled rows of the forward and {len(rb)} of the backward GEMM + epilogue "
            f"(full N, full K) per sample, {nthreads} threads; host input generation "
            f"({inp['gen_s']:.1f}s) not timed")
    return flops, sec, desc


def sampled_parity(dev: dict, ref: dict) -> dict:
    """The device's sampled rows against the oracle's: normalised max error
    max|g - o| / max|o| and relative L2 error of Y and dZ (bounds 2e-2 and
    5e-3), and ReLU-mask bits that differ outside / inside the band
    |z| < 1e-3 max_j |z[i, j]| where accumulation order may flip a sign."""
    def errs(g, o):
        g = np.asarray(g, dtype=np.float64)
        o = np.asarray(o, dtype=np.float64)
        return {"nmax": float(np.abs(g - o).max() / max(np.abs(o).max(), 1e-30)),
                "rel_l2": float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30))}
    rf = ref["rows_fwd"]
    words = dev["aux_rows"].astype(np.uint32)  # word row (r // 32) of each sampled row
    bits = (words >> (rf % 32)[:, None].astype(np.uint32)) & 1
    want = ref["z"] > 0
    band = np.abs(ref["z"]) < 1e-3 * np.abs(ref["z"]).max(axis=1, keepdims=True)
    diff = bits.astype(bool) != want
    y, dz = errs(dev["Y"], ref["Y"]), errs(dev["dZ"], ref["dZ"])
    out_band = int((diff & ~band).sum())
    ok = all(e["nmax"] <= 2e-2 and e["rel_l2"] <= 5e-3 for e in (y, dz)) and out_band == 0
    return {"rows_fwd": len(rf), "rows_bwd": len(ref["rows_bwd"]), "Y": y, "dZ": dz,
            "mask_mismatch_outside_band": out_band, "mask_mismatch_in_band": int((diff & band).sum()),
            "bounds": {"nmax": 2e-2, "rel_l2": 5e-3}, "pass": bool(ok)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    nthreads = os.cpu_count() or 1
    # bounded work per step: about 200 sampled rows per GEMM over the whole run
    per_step_rows = max(1, min(args.ref_step_rows, 200 // max(args.steps, 1)))
    for _ in range(args.warmup):
        oracle_sample(1, 1, nthreads)
    times, flops_tot = [], 0.0
    desc = ""
    for i in range(args.steps):
        fl, sec, desc = oracle_sample(per_step_rows, per_step_rows, nthreads, offset=i)
        times.append(sec)
        flops_tot += fl
    total = sum(times)
    value = flops_tot / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- end to end
def run_e2e(args, gf, torch, fwd, bwd, dev, world, barrier, dev_in0, dev_out0):
    """The step through the C ABI from pinned host memory: every step copies
    its inputs host -> device, runs the fused forward and backward, and copies
    every output device -> host. Copies of later / earlier steps run on their
    own streams under the compute of step i (`--e2e-depth` buffer sets), the
    way a training or serving loop would overlap them."""
    depth = max(2, args.e2e_depth)
    host_in = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in dev_in0.items()}
    for n, t in dev_in0.items():
        host_in[n].copy_(t)
    host_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                 for n, t in dev_out0.items()} for _ in range(depth)]
    dev_in = [dev_in0] + [{n: torch.empty_like(t) for n, t in dev_in0.items()}
                          for _ in range(depth - 1)]
    dev_out = [dev_out0] + [{n: torch.empty_like(t) for n, t in dev_out0.items()}
                            for _ in range(depth - 1)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_comp = torch.cuda.current_stream(dev)
    sc = s_comp.cuda_stream
    h2d_done = [torch.cuda.Event() for _ in range(depth)]
    comp_done = [torch.cuda.Event() for _ in range(depth)]
    d2h_done = [torch.cuda.Event() for _ in range(depth)]

    def run(n):
        for i in range(n):
            b = i % depth
            if i >= depth:  # buffer set b is free once step i - depth is done with it
                s_h2d.wait_event(comp_done[b])
            with torch.cuda.stream(s_h2d):
                for k, t in dev_in[b].items():
                    t.copy_(host_in[k], non_blocking=True)
            h2d_done[b].record(s_h2d)
            s_comp.wait_event(h2d_done[b])
            if i >= depth:
                s_comp.wait_event(d2h_done[b])
            di, do = dev_in[b], dev_out[b]
            gf.gf_matmul_execute(fwd, di["X"], di["W"], bias=di["bias"], out=do["Y"],
                                 aux_out=do["aux"], stream=sc)
            gf.gf_matmul_execute(bwd, di["dY"], di["W"], out=do["dZ"], aux_in=di["mask"],
                                 bgrad=do["bgrad"], stream=sc)
            comp_done[b].record(s_comp)
            s_d2h.wait_event(comp_done[b])
            with torch.cuda.stream(s_d2h):
                for k, t in do.items():
                    host_out[b][k].copy_(t, non_blocking=True)
            d2h_done[b].record(s_d2h)

    run(depth)
    barrier()
    # enough steps that the pipeline's fill (the first step's copy in) and
    # drain (the last step's copy out) are a small share of the timed region
    n = max(3, min(args.steps, 30))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_h2d)
    run(n)
    s_d2h.wait_event(d2h_done[(n - 1) % depth])
    t1.record(s_d2h)
    barrier()
    ms = t0.elapsed_time(t1) / n
    ok = gf.gf_plan_status(fwd, sc) == gf.GF_OK and gf.gf_plan_status(bwd, sc) == gf.GF_OK

    # what bounds it: one step's copies with no kernels running, each
    # direction alone and both at once (median of 3)
    def copies(dirs):
        out = []
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s_h2d)
            s_d2h.wait_stream(s_h2d)
            if "in" in dirs:
                with torch.cuda.stream(s_h2d):
                    for k, t in dev_in[0].items():
                        t.copy_(host_in[k], non_blocking=True)
            if "out" in dirs:
                with torch.cuda.stream(s_d2h):
                    for k, t in dev_out[0].items():
                        host_out[0][k].copy_(t, non_blocking=True)
            s_h2d.wait_stream(s_d2h)
            b.record(s_h2d)
            b.synchronize()
            out.append(a.elapsed_time(b))
        return sorted(out)[1]
    c_in, c_out, c_both = copies(("in",)), copies(("out",)), copies(("in", "out"))
    link = {"h2d_alone_ms": c_in, "d2h_alone_ms": c_out, "both_at_once_ms": c_both,
            "h2d_gbs": h2d / (c_in * 1e-3) / 1e9, "d2h_gbs": d2h / (c_out * 1e-3) / 1e9,
            "note": "one step's copies with no kernels running: the step cannot be shorter "
                    "than both_at_once_ms or than the kernels"}
    del host_in, host_out, dev_in, dev_out
    torch.cuda.empty_cache()
    return {"value": world * 2 * FLOP_PER_GEMM / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": f"{depth} buffer sets: H2D of later steps and D2H of earlier steps on "
                       "their own streams under step i; the timed region includes the first "
                       "step's H2D and the last step's D2H",
            "host_link": link, "status_ok": ok}


# ------------------------------------------------------------------- GPU leg
def run_gpu(args):
    import torch

    import gemm_epilogue_tmem_gb300 as gf

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gf.build()
    synth.build_cuda()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    f16 = torch.float16
    X = torch.empty((M, K), dtype=f16, device=dev)
    W = torch.empty((K, N), dtype=f16, device=dev)
    bias = torch.empty((N,), dtype=f16, device=dev)
    dY = torch.empty((M, N), dtype=f16, device=dev)
    mask = torch.empty((M // 32, K), dtype=torch.int32, device=dev)
    Y = torch.empty((M, N), dtype=f16, device=dev)
    aux = torch.empty((M // 32, N), dtype=torch.int32, device=dev)
    dZ = torch.empty((M, K), dtype=f16, device=dev)
    bgrad = torch.empty((K,), dtype=torch.float32, device=dev)
    seed = 0
    synth.dev_normal(X, synth.F16, seed, synth.TID_A, 1.0, sp)
    synth.dev_normal(W, synth.F16, seed, synth.TID_B, 1 / 128, sp)
    synth.dev_normal(bias, synth.F16, seed, synth.TID_BIAS, 0.1, sp)
    synth.dev_normal(dY, synth.F16, seed, synth.TID_DY, 1.0, sp)
    synth.dev_mask_words(mask, M, K, seed, synth.TID_MASK, sp)
    torch.cuda.synchronize()

    fwd = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL,
                               gf.GF_B_KN)
    bwd = gf.gf_matmul_plan_ex(M, K, N, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                               gf.GF_B_NK)
    fwd_none = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                                    gf.GF_B_KN)
    bwd_none = gf.gf_matmul_plan_ex(M, K, N, gf.GF_F16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                                    gf.GF_B_NK)
    # fused forward, fused backward (+ the bias-gradient finalize), as the
    # plans enqueue them
    # the bare GEMMs without a k split, as the fused plans run
    for pl in (fwd_none, bwd_none):
        gf.gf_plan_set_option(pl, gf.GF_OPT_SPLIT_K, 1)
    if args.kernel:
        for pl in (fwd, bwd, fwd_none, bwd_none):
            gf.gf_plan_set_option(pl, gf.GF_OPT_KERNEL, args.kernel)
    if args.autotune:
        gf.gf_matmul_autotune(fwd, X, W, bias=bias, out=Y, aux_out=aux, stream=sp, reps=2)
        gf.gf_matmul_autotune(bwd, dY, W, out=dZ, aux_in=mask, bgrad=bgrad, stream=sp, reps=2)
    plans = {"fwd": gf.gf_plan_describe(fwd), "bwd": gf.gf_plan_describe(bwd),
             "autotuned": bool(args.autotune)}
    launches_per_step = plans["fwd"]["launches"] + plans["bwd"]["launches"]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        gf.gf_matmul_execute(fwd, X, W, bias=bias, out=Y, aux_out=aux, stream=sp)
        if ev is not None:
            ev[1].record(stream)
        gf.gf_matmul_execute(bwd, dY, W, out=dZ, aux_in=mask, bgrad=bgrad, stream=sp)
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step()
    barrier()
    assert gf.gf_plan_status(fwd, sp) == gf.GF_OK and gf.gf_plan_status(bwd, sp) == gf.GF_OK

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    h0 = time.monotonic()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    clk = clocks.stop(window=(h0, time.monotonic()))
    status_ok = gf.gf_plan_status(fwd, sp) == gf.GF_OK and gf.gf_plan_status(bwd, sp) == gf.GF_OK
    ms_total = t_start.elapsed_time(t_end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)

    # the device's outputs of the sampled rows, for the parity check against the oracle
    rows_t = torch.as_tensor(synth.sample_rows(M, 64, 0), dtype=torch.long, device=dev)
    dev_rows = {"Y": Y.index_select(0, rows_t).float().cpu().numpy(),
                "aux_rows": aux.index_select(0, rows_t // 32).cpu().numpy().view(np.uint32),
                "dZ": dZ.index_select(0, rows_t).float().cpu().numpy()}

    # the same step captured once in a CUDA graph and replayed
    graph = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                cs = torch.cuda.current_stream().cuda_stream
                gf.gf_matmul_execute(fwd, X, W, bias=bias, out=Y, aux_out=aux, stream=cs)
                gf.gf_matmul_execute(bwd, dY, W, out=dZ, aux_in=mask, bgrad=bgrad, stream=cs)
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        reps = max(3, min(args.steps, 20))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        gms = a.elapsed_time(b) / reps
        graph = {"ms_per_step": gms, "value": 2 * FLOP_PER_GEMM / (gms * 1e-3) / 1e12,
                 "unit": "TFLOP/s", "replays": reps,
                 "status_ok": gf.gf_plan_status(fwd, sp) == gf.GF_OK and
                 gf.gf_plan_status(bwd, sp) == gf.GF_OK}
        del g

    # Steady-state comparison at the power cap, the configurations taking
    # turns in windows of back-to-back launches (so that clock and power drift
    # fall on all of them alike): the fused kernels, the same kernels and
    # tiles with no epilogue (the epilogue's overhead), torch.matmul of the
    # same operands (cuBLAS, no epilogue; context), and the same work unfused
    # in torch as the pages' comparison has it -- the GEMM, then the bias add,
    # the ReLU and the mask pack as separate kernels; the GEMM with W^T, then
    # the mask unpacked and applied, then the column sum.
    cmp = None
    if not args.no_compare:
        Wt = W.t()
        shifts = torch.arange(32, dtype=torch.int32, device=dev)
        Z = torch.empty((M, N), dtype=f16, device=dev)
        G = torch.empty((M, K), dtype=f16, device=dev)

        def unfused_fwd():
            torch.matmul(X, W, out=Z)
            Z.add_(bias)
            pos = Z > 0
            torch.clamp(Z, min=0, out=Y)
            bits = pos.view(M // 32, 32, N).to(torch.int32) << shifts.view(1, 32, 1)
            aux.copy_(bits.sum(1, dtype=torch.int32))

        def unfused_bwd():
            torch.matmul(dY, Wt, out=G)
            bits = (mask.view(M // 32, 1, K) >> shifts.view(1, 32, 1)) & 1
            torch.mul(G, bits.view(M, K), out=dZ)
            bgrad.copy_(dZ.sum(0, dtype=torch.float32))

        fns = {
            "fwd_fused": lambda: gf.gf_matmul_execute(fwd, X, W, bias=bias, out=Y, aux_out=aux,
                                                      stream=sp),
            "fwd_none": lambda: gf.gf_matmul_execute(fwd_none, X, W, out=Y, stream=sp),
            "bwd_fused": lambda: gf.gf_matmul_execute(bwd, dY, W, out=dZ, aux_in=mask,
                                                      bgrad=bgrad, stream=sp),
            "bwd_none": lambda: gf.gf_matmul_execute(bwd_none, dY, W, out=dZ, stream=sp),
        }
        if not args.no_cublas:
            fns["fwd_cublas"] = lambda: torch.matmul(X, W, out=Y)
            fns["bwd_cublas"] = lambda: torch.matmul(dY, Wt, out=dZ)
            fns["fwd_torch_unfused"] = unfused_fwd
            fns["bwd_torch_unfused"] = unfused_bwd
        cmp = sustained_windows(torch, fns, args.cmp_seconds, args.cmp_rounds, local)
        del Z, G
        torch.cuda.empty_cache()
        cmp_ok = gf.gf_plan_status(fwd, sp) == gf.GF_OK and gf.gf_plan_status(bwd, sp) == gf.GF_OK

    # end to end through the C ABI from pinned host memory
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, gf, torch, fwd, bwd, dev, world, barrier,
                      {"X": X, "W": W, "bias": bias, "dY": dY, "mask": mask},
                      {"Y": Y, "aux": aux, "dZ": dZ, "bgrad": bgrad})

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        return 0

    pk, pk_kind = peaks()
    ms_step = ms_total / args.steps
    value = world * 2 * FLOP_PER_GEMM / (ms_step * 1e-3) / 1e12
    fwd_st, bwd_st = stats_ms(fwd_ms), stats_ms(bwd_ms)
    rec = recorded_traffic()
    fwd_dom = fwd_st["median"] >= bwd_st["median"]
    traffic = None if rec is None else (rec[0] if fwd_dom else rec[1])
    dom_name, dom = ("fused forward RELU_AUX_BIAS", fwd_st) if fwd_dom else \
        ("fused backward DRELU_BGRAD (+ finalize)", bwd_st)
    # the timed loop ran for ms_total: burst peak for a short loop, sustained for a long one
    peak, peak_src = pick_peak(pk, pk_kind, ms_total * 1e-3)
    achieved = FLOP_PER_GEMM / (dom["median"] * 1e-3) / 1e12

    comparison = None
    if cmp is not None:
        c = cmp["per_fn"]

        def ratio(a, b, key="ms_median"):
            return c[a][key] / c[b][key] if a in c and b in c and c[b][key] else None

        comparison = {
            "protocol": (f"{args.cmp_rounds} rounds; in each, every configuration runs back to back "
                         f"for {args.cmp_seconds:.1f} s (groups of 4 launches between CUDA events); "
                         "median and min ms per launch over all groups; SM MHz = median "
                         "nvidia-smi sample of its windows; Mcycles = median ms x MHz"),
            "per_config": c,
            "busy_s": cmp["busy_s"],
            "status_ok": cmp_ok,
        }
        epi_overhead = {"fwd": ratio("fwd_fused", "fwd_none") - 1,
                        "bwd": ratio("bwd_fused", "bwd_none") - 1,
                        "fwd_cycles": ratio("fwd_fused", "fwd_none", "mcycles") - 1
                        if c["fwd_none"]["mcycles"] else None,
                        "bwd_cycles": ratio("bwd_fused", "bwd_none", "mcycles") - 1
                        if c["bwd_none"]["mcycles"] else None,
                        "method": "steady-state windows (comparison.protocol): fused / same kernel "
                                  "and tiles with EPILOG_NONE - 1, by time and by cycles"}
        cublas = None
        unfused = None
        if "fwd_cublas" in c:
            cublas = {"fwd_ms": c["fwd_cublas"]["ms_median"], "bwd_ms": c["bwd_cublas"]["ms_median"],
                      "fwd_tflops": FLOP_PER_GEMM / (c["fwd_cublas"]["ms_median"] * 1e-3) / 1e12,
                      "bwd_tflops": FLOP_PER_GEMM / (c["bwd_cublas"]["ms_median"] * 1e-3) / 1e12,
                      "fwd_none_vs_cublas": ratio("fwd_none", "fwd_cublas"),
                      "bwd_none_vs_cublas": ratio("bwd_none", "bwd_cublas"),
                      "fwd_fused_vs_cublas": ratio("fwd_fused", "fwd_cublas"),
                      "bwd_fused_vs_cublas": ratio("bwd_fused", "bwd_cublas"),
                      "note": "torch.matmul of the same operands, no epilogue (time ratios: "
                              "ours / cuBLAS); context, not the metric"}
            unfused = {"fwd": ratio("fwd_torch_unfused", "fwd_fused"),
                       "bwd": ratio("bwd_torch_unfused", "bwd_fused"),
                       "fwd_ms": c["fwd_torch_unfused"]["ms_median"],
                       "bwd_ms": c["bwd_torch_unfused"]["ms_median"],
                       "what": "time of the same work unfused in torch / fused time. Forward: "
                               "torch.matmul, then bias add, ReLU and mask pack as separate "
                               "kernels; backward: torch.matmul with W^T, then the mask unpacked "
                               "and applied, then the fp32 column sum",
                       "context": "the pages quote about 30% less time for fused GEMM + bias + "
                                  "ReLU against three separate kernels, on H100 (not this "
                                  "hardware; not a target)"}
    else:
        epi_overhead, cublas, unfused = None, None, None

    cpu = None
    parity = None
    if not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        ref_rows = {}
        fl, sec, desc = oracle_sample(args.ref_rows, args.ref_rows, nthreads, outputs=ref_rows)
        cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
               "sample": desc, "seconds": sec,
               # the whole step at this rate (an extrapolation from the sampled rows)
               "extrapolated_full_step_s": 2 * FLOP_PER_GEMM / (fl / sec)}
        fl1, sec1, _ = oracle_sample(4, 4, 1, offset=1)
        cpu["single_thread"] = {"value": fl1 / sec1 / 1e12, "unit": "TFLOP/s",
                                "sample": "4 sampled rows of each GEMM, 1 thread",
                                "seconds": sec1}
        n_f, n_b = len(ref_rows["rows_fwd"]), len(ref_rows["rows_bwd"])
        parity = sampled_parity({"Y": dev_rows["Y"][:n_f], "aux_rows": dev_rows["aux_rows"][:n_f],
                                 "dZ": dev_rows["dZ"][:n_b]}, ref_rows)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "seed": 0,
                   "l2": "inputs larger than L2 (X 2.1 GB, dY 1.1 GB); no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU", "plans": plans},
        "pct_of_peak": {"value": 100 * value / world / peak, "peak_tflops": peak,
                        "peak_kind": peak_src,
                        "vs_nominal_2250": 100 * value / world / 2250.0},
        "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": peak_src,
                     "achieved_from": "median CUDA-event time of the kernel's launches in the "
                                      "timed loop",
                     "algorithmic_flop_per_launch": FLOP_PER_GEMM,
                     "traffic_note": "DRAM bytes per launch from the committed ncu summary "
                                     "(16384-row case scaled to the full rows), null when the "
                                     "kernel sources changed since"},
        "kernels_ms": {"fwd_relu_aux_bias": fwd_st, "bwd_drelu_bgrad": bwd_st},
        "epilogue_overhead": epi_overhead,
        "cublas_same_shapes": cublas,
        "fused_vs_torch_unfused": unfused,
        "comparison": comparison,
        "parity": parity,
        "gpu": torch.cuda.get_device_name(dev),
        "cuda_graph_replay": graph,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "status_ok": status_ok,
    }
    print(json.dumps(line), flush=True)
    for p in (fwd, bwd, fwd_none, bwd_none):
        p.free()
    return 0


def run_profile_case(args):
    """One fused GEMM + epilogue of the given shape, launched warmup + steps
    times: the small case the ncu captures run (no oracle, no timing)."""
    import torch

    import gemm_epilogue_tmem_gb300 as gf

    m, n, k = (int(x) for x in args.profile_case.split(","))
    if args.epilog in ("swiglu_save", "dswiglu"):
        return run_profile_case_swiglu(args, m, n, k)
    if args.epilog in ("gelu_aux_bias", "dgelu_bgrad"):
        return run_profile_case_gelu(args, m, n, k)
    epi = {"relu_aux_bias": gf.GF_EPILOG_RELU_AUX_BIAS, "drelu_bgrad": gf.GF_EPILOG_DRELU_BGRAD,
           "none": gf.GF_EPILOG_NONE, "relu_bias": gf.GF_EPILOG_RELU_BIAS}[args.epilog]
    layout = gf.GF_B_NK if epi == gf.GF_EPILOG_DRELU_BGRAD else gf.GF_B_KN
    gf.build()
    synth.build_cuda()
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    A = torch.empty((m, k), dtype=torch.float16, device=dev)
    B = torch.empty((k, n) if layout == gf.GF_B_KN else (n, k), dtype=torch.float16, device=dev)
    bias = torch.empty((n,), dtype=torch.float16, device=dev)
    out = torch.empty((m, n), dtype=torch.float16, device=dev)
    aux = torch.empty(((m + 31) // 32, n), dtype=torch.int32, device=dev)
    bgrad = torch.empty((n,), dtype=torch.float32, device=dev)
    synth.dev_normal(A, synth.F16, 0, synth.TID_A, 1.0, sp)
    synth.dev_normal(B, synth.F16, 0, synth.TID_B, 1 / np.sqrt(k), sp)
    synth.dev_normal(bias, synth.F16, 0, synth.TID_BIAS, 0.1, sp)
    synth.dev_mask_words(aux, m, n, 0, synth.TID_MASK, sp)
    plan = gf.gf_matmul_plan_ex(m, n, k, gf.GF_F16, epi, gf.GF_BIAS_COL, layout)
    if args.kernel:
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, args.kernel)
    if args.l2_hints >= 0:
        gf.gf_plan_set_option(plan, gf.GF_OPT_L2_HINTS, args.l2_hints)
    if args.group_m:
        gf.gf_plan_set_option(plan, gf.GF_OPT_GROUP_M, args.group_m)
    if args.split:
        gf.gf_plan_set_option(plan, gf.GF_OPT_SPLIT_K, args.split)
    for _ in range(args.warmup + args.steps):
        if epi == gf.GF_EPILOG_DRELU_BGRAD:
            gf.gf_matmul_execute(plan, A, B, out=out, aux_in=aux, bgrad=bgrad, stream=sp)
        else:
            gf.gf_matmul_execute(plan, A, B, bias=bias, out=out, aux_out=aux, stream=sp)
    torch.cuda.synchronize()
    st = gf.gf_plan_status(plan, sp)
    print(json.dumps({"profile_case": [m, n, k], "epilog": args.epilog, "status": st,
                      "plan": gf.gf_plan_describe(plan)}))
    plan.free()
    return 0 if st == gf.GF_OK else 1


def run_profile_case_gelu(args, m, n, k):
    """--profile-case M,N,K with --epilog gelu_aux_bias (X[M,K] W[K,N], the
    pre-activation saved in bf16) or dgelu_bgrad (dY[M,K] with W given [N,K],
    the saved pre-activation [M,N] read back), bf16."""
    import torch

    import gemm_epilogue_tmem_gb300 as gf
    gf.build()
    synth.build_cuda()
    sp = torch.cuda.current_stream().cuda_stream
    bf = torch.bfloat16
    dev = torch.device("cuda", 0)

    def filled(shape, tid, sigma):
        t = torch.empty(shape, dtype=bf, device=dev)
        synth.dev_normal(t, synth.BF16, 0, tid, sigma, sp)
        return t

    out = torch.empty((m, n), dtype=bf, device=dev)
    fwd = args.epilog == "gelu_aux_bias"
    A = filled((m, k), synth.TID_A if fwd else synth.TID_DY, 1.0)
    B = filled((k, n) if fwd else (n, k), synth.TID_B, 1 / np.sqrt(k))
    if fwd:
        bias, pre = filled((n,), synth.TID_BIAS, 0.1), torch.empty((m, n), dtype=bf, device=dev)
        plan = gf.gf_matmul_plan_ex(m, n, k, gf.GF_BF16, gf.GF_EPILOG_GELU_AUX_BIAS,
                                    gf.GF_BIAS_COL, gf.GF_B_KN)
        fn = lambda: gf.gf_matmul_execute(plan, A, B, bias=bias, out=out, aux_out=pre,  # noqa: E731
                                          stream=sp)
    else:
        pre, bgrad = filled((m, n), synth.TID_PREACT, 1.0), torch.empty((n,), dtype=torch.float32,
                                                                        device=dev)
        plan = gf.gf_matmul_plan_ex(m, n, k, gf.GF_BF16, gf.GF_EPILOG_DGELU_BGRAD,
                                    gf.GF_BIAS_COL, gf.GF_B_NK)
        fn = lambda: gf.gf_matmul_execute(plan, A, B, out=out, aux_in=pre,  # noqa: E731
                                          bgrad=bgrad, stream=sp)
    if args.kernel:
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, args.kernel)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    st = gf.gf_plan_status(plan, sp)
    print(json.dumps({"profile_case": [m, n, k], "epilog": args.epilog, "status": st,
                      "plan": gf.gf_plan_describe(plan)}))
    plan.free()
    return 0 if st == gf.GF_OK else 1


def run_profile_case_swiglu(args, m, n, k):
    """--profile-case M,I,H with --epilog swiglu_save (gate+up forward saving
    g and u) or dswiglu (dh = dout Wd with the dSwiGLU epilogue), bf16."""
    import torch

    import gemm_epilogue_tmem_gb300 as gf
    gf.build()
    synth.build_cuda()
    sp = torch.cuda.current_stream().cuda_stream
    bf = torch.bfloat16
    dev = torch.device("cuda", 0)

    def filled(shape, tid, sigma):
        t = torch.empty(shape, dtype=bf, device=dev)
        synth.dev_normal(t, synth.BF16, 0, tid, sigma, sp)
        return t

    outs = [torch.empty((m, n), dtype=bf, device=dev) for _ in range(3)]
    if args.epilog == "swiglu_save":
        x, wg, wu = filled((m, k), synth.TID_A, 1.0), filled((n, k), synth.TID_WG, 0.02), \
            filled((n, k), synth.TID_WU, 0.02)
        plan = gf.gf_swiglu_plan(m, n, k, gf.GF_BF16, save_gu=True)
        fn = lambda: gf.gf_swiglu_execute(plan, x, wg, wu, *outs, stream=sp)  # noqa: E731
    else:
        dout, wd = filled((m, k), synth.TID_DOUT, 1.0), filled((k, n), synth.TID_WD, 0.02)
        g, u = filled((m, n), synth.TID_G_SAVED, 1.0), filled((m, n), synth.TID_U_SAVED, 1.0)
        plan = gf.gf_dswiglu_plan(m, n, k, gf.GF_BF16)
        fn = lambda: gf.gf_dswiglu_execute(plan, dout, wd, g, u, outs[0], outs[1],  # noqa: E731
                                           stream=sp)
    if args.kernel:
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, args.kernel)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    st = gf.gf_plan_status(plan, sp)
    print(json.dumps({"profile_case": [m, n, k], "epilog": args.epilog, "status": st,
                      "plan": gf.gf_plan_describe(plan)}))
    plan.free()
    return 0 if st == gf.GF_OK else 1


def _interleaved(torch, fns: dict, reps: int, rounds: int = 3) -> dict:
    """Per function: median and minimum ms per call, from `reps` back-to-back
    calls between two events on the current stream, the functions taken in
    turn `rounds` times so that clock and power drift fall on all of them
    alike."""
    for fn in fns.values():
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    times = {k: [] for k in fns}
    s = torch.cuda.current_stream()
    for _ in range(rounds):
        for name, fn in fns.items():
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(reps):
                fn()
            b.record(s)
            torch.cuda.synchronize()
            times[name].append(a.elapsed_time(b) / reps)
    return {k: {"median": statistics.median(v), "min": min(v)} for k, v in times.items()}


def _flushed(torch, fns: dict, reps: int, dev) -> dict:
    """Per function: median and minimum ms of single calls, each timed alone
    between two events right after a 256 MB write (twice the L2) has evicted
    its inputs from L2."""
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.int32, device=dev)
    times = {k: [] for k in fns}
    s = torch.cuda.current_stream()
    for _ in range(reps):
        for name, fn in fns.items():
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            torch.cuda.synchronize()
            times[name].append(a.elapsed_time(b))
    del flush
    return {k: {"median": statistics.median(v), "min": min(v)} for k, v in times.items()}


def _dev_fill(torch, recipe, name, dev, sp, view=None):
    t = recipe.tensors[name]
    tdt = torch.float16 if recipe.dtype == synth.F16 else torch.bfloat16
    x = view if view is not None else torch.empty(t.shape, dtype=tdt, device=dev)
    synth.dev_normal(x, recipe.dtype, 0, t.tensor_id, t.sigma, sp)
    return x


def _host(recipe, name, rows=None):
    t = recipe.tensors[name]
    return synth.normal(t.shape, recipe.dtype, 0, t.tensor_id, t.sigma, rows=rows)


def _errs(g, o) -> dict:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    return {"nmax": float(np.abs(g - o).max() / max(np.abs(o).max(), 1e-30)),
            "rel_l2": float(np.linalg.norm(g - o) / max(np.linalg.norm(o), 1e-30))}


def _parity_block(out: dict, bgrad_keys=(), mask=None) -> dict:
    """Pass/fail of a set of output errors against the parity bounds (outputs
    2e-2 / 5e-3, bias gradients 1e-2 / 1e-2; mask bits outside the band 0)."""
    ok = True
    for k, e in out.items():
        lim = (1e-2, 1e-2) if k in bgrad_keys else (2e-2, 5e-3)
        ok = ok and e["nmax"] <= lim[0] and e["rel_l2"] <= lim[1]
    blk = dict(out)
    if mask is not None:
        blk.update(mask)
        ok = ok and mask["mask_mismatch_outside_band"] == 0
    blk["bounds"] = {"outputs": {"nmax": 2e-2, "rel_l2": 5e-3},
                     "bias_gradients": {"nmax": 1e-2, "rel_l2": 1e-2}}
    blk["pass"] = bool(ok)
    return blk


def _timed_steps(torch, step_fns: dict, steps: int, warmup: int, gpu: int) -> dict:
    """The workload's step (its kernels in order, back to back) run `warmup`
    times untimed, then `steps` times between CUDA events, each kernel
    bracketed by events too, while nvidia-smi samples the clocks."""
    for _ in range(warmup):
        for fn in step_fns.values():
            fn()
    torch.cuda.synchronize()
    names = list(step_fns)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(steps)]
    sampler = ClockSampler(gpu)
    sampler.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    h0 = time.monotonic()
    t0.record(s)
    for i in range(steps):
        for j, fn in enumerate(step_fns.values()):
            evs[i][j].record(s)
            fn()
        evs[i][-1].record(s)
    t1.record(s)
    torch.cuda.synchronize()
    clk = sampler.stop(window=(h0, time.monotonic()))
    per = {n: stats_ms([e[j].elapsed_time(e[j + 1]) for e in evs]) for j, n in enumerate(names)}
    return {"ms_total": t0.elapsed_time(t1), "per_kernel": per, "clocks": clk}


def _roofline(per_kernel: dict, flops: dict, peak: float, peak_src: str) -> dict:
    dom = max(per_kernel, key=lambda k: per_kernel[k]["median"])
    ach = flops[dom] / (per_kernel[dom]["median"] * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "traffic": None, "peak_source": peak_src,
            "achieved_from": "median CUDA-event time of the kernel's launches in the timed loop",
            "algorithmic_flop_per_launch": flops[dom]}


def run_gelu_workload(args, gf, torch, dev, sp, pk, pk_kind):
    """GELU_AUX_BIAS forward X[8192,4096] W[4096,16384] + DGELU_BGRAD backward
    dY[8192,16384] W^T on a seeded pre-activation [8192,4096], bf16."""
    import torch.nn.functional as F
    rc = synth.GELU_BIAS
    Mg, Kg = rc.tensors["X"].shape
    Ng = rc.tensors["W"].shape[1]
    bf = torch.bfloat16
    X, W, bias, dY, pre_b = (_dev_fill(torch, rc, n, dev, sp)
                             for n in ("X", "W", "bias", "dY", "preact"))
    Y = torch.empty((Mg, Ng), dtype=bf, device=dev)
    pre = torch.empty((Mg, Ng), dtype=bf, device=dev)
    dX = torch.empty((Mg, Kg), dtype=bf, device=dev)
    bgrad = torch.empty((Kg,), dtype=torch.float32, device=dev)
    plan = {
        "fwd": gf.gf_matmul_plan_ex(Mg, Ng, Kg, gf.GF_BF16, gf.GF_EPILOG_GELU_AUX_BIAS,
                                    gf.GF_BIAS_COL, gf.GF_B_KN),
        "bwd": gf.gf_matmul_plan_ex(Mg, Kg, Ng, gf.GF_BF16, gf.GF_EPILOG_DGELU_BGRAD,
                                    gf.GF_BIAS_COL, gf.GF_B_NK),
        "fwd_none": gf.gf_matmul_plan_ex(Mg, Ng, Kg, gf.GF_BF16, gf.GF_EPILOG_NONE,
                                         gf.GF_BIAS_COL, gf.GF_B_KN),
        "bwd_none": gf.gf_matmul_plan_ex(Mg, Kg, Ng, gf.GF_BF16, gf.GF_EPILOG_NONE,
                                         gf.GF_BIAS_COL, gf.GF_B_NK),
    }
    # the bare GEMMs run in the fused plans' kernel and tile configuration,
    # without a k split
    for a, b in (("fwd_none", "fwd"), ("bwd_none", "bwd")):
        gf.gf_plan_set_option(plan[a], gf.GF_OPT_SPLIT_K, 1)
        d = gf.gf_plan_describe(plan[b])
        kern = (3 if d["tile_n"] == 512 else 2) if d["tile_m"] == 256 else 1
        gf.gf_plan_set_option(plan[a], gf.GF_OPT_KERNEL, kern)
        if d["tile_m"] != 256:
            gf.gf_plan_set_option(plan[a], gf.GF_OPT_TILE_N, d["tile_n"])
    ex = gf.gf_matmul_execute
    fused = {
        "fwd_gelu_aux_bias": lambda: ex(plan["fwd"], X, W, bias=bias, out=Y, aux_out=pre,
                                        stream=sp),
        "bwd_dgelu_bgrad": lambda: ex(plan["bwd"], dY, W, out=dX, aux_in=pre_b, bgrad=bgrad,
                                      stream=sp),
    }
    flop = 2.0 * Mg * Ng * Kg
    tl = _timed_steps(torch, fused, args.steps, args.warmup, dev.index or 0)
    ok = all(gf.gf_plan_status(plan[k], sp) == gf.GF_OK for k in ("fwd", "bwd"))

    # parity: sampled rows of both kernels, sampled columns of the bias gradient
    rows = synth.sample_rows(Mg, 64, 0)
    cols = synth.sample_cols(Kg, 64, 0)
    ridx = torch.as_tensor(rows, device=dev)
    y_d, pre_d, dx_d = (t.index_select(0, ridx).float().cpu().numpy() for t in (Y, pre, dX))
    bg_d = bgrad.cpu().numpy()

    def unfused_fwd():
        torch.addmm(bias, X, W, out=pre)
        F.gelu(pre, approximate="tanh")

    def unfused_bwd():
        g = torch.matmul(dY, W.t())
        dz = torch.ops.aten.gelu_backward(g, pre_b, approximate="tanh")
        dz.float().sum(0)

    cmp = None
    if not args.no_compare:
        cmp = sustained_windows(torch, {
            **fused,
            "fwd_none": lambda: ex(plan["fwd_none"], X, W, out=Y, stream=sp),
            "bwd_none": lambda: ex(plan["bwd_none"], dY, W, out=dX, stream=sp),
            "torch_unfused_fwd": unfused_fwd,
            "torch_unfused_bwd": unfused_bwd,
        }, args.cmp_seconds, args.cmp_rounds, dev.index or 0)
    ok = ok and all(gf.gf_plan_status(p, sp) == gf.GF_OK for p in plan.values())
    launches = sum(gf.gf_plan_describe(plan[k])["launches"] for k in ("fwd", "bwd"))
    for p in plan.values():
        p.free()
    del X, W, bias, dY, pre_b, Y, pre, dX, bgrad
    torch.cuda.empty_cache()

    nthreads = os.cpu_count() or 1
    import oracle
    W_h, b_h = _host(rc, "W"), _host(rc, "bias")
    Xs, dYs, pres = _host(rc, "X", rows), _host(rc, "dY", rows), _host(rc, "preact", rows)
    t_cpu = time.time()
    y_o, aux_o, _ = oracle.gelu_aux_bias(Xs, W_h, b_h, oracle.BF16, row_ids=rows,
                                         nthreads=nthreads)
    dz_o, _, _ = oracle.dgelu_bgrad(dYs, W_h, pres, oracle.BF16, oracle.B_NK, full_rows=False,
                                    nthreads=nthreads)
    cpu_s = time.time() - t_cpu
    dY_all = _host(rc, "dY")
    pre_all = _host(rc, "preact")
    _, bg_o, _ = oracle.dgelu_bgrad(dY_all, W_h[cols], pre_all[:, cols], oracle.BF16, oracle.B_NK,
                                    nthreads=nthreads)
    dec = lambda a: oracle.decode(a, oracle.BF16)  # noqa: E731
    parity = _parity_block({"Y": _errs(y_d, dec(y_o)), "preact_aux": _errs(pre_d, dec(aux_o)),
                            "dX": _errs(dx_d, dec(dz_o)),
                            "bgrad_sampled_cols": _errs(bg_d[cols], bg_o)},
                           bgrad_keys=("bgrad_sampled_cols",))
    parity.update({"rows": len(rows), "bgrad_cols": len(cols)})
    cpu_flop = 2.0 * len(rows) * Ng * Kg * 2
    step = tl["ms_total"] / args.steps
    peak, peak_src = pick_peak(pk, pk_kind, tl["ms_total"] * 1e-3)
    line = {
        "workload": f"gelu_bf16_fwd_gelu_aux_bias_bwd_dgelu_bgrad_{Mg}x{Ng}x{Kg}",
        "config": {"workload": f"gelu_bf16_fwd_gelu_aux_bias_bwd_dgelu_bgrad_{Mg}x{Ng}x{Kg}",
                   "M": Mg, "N": Ng, "K": Kg, "seed": 0,
                   "l2": "X, W, dY, pre-activation 0.67 GB in all: larger than L2; no flush"},
        "value": 2 * flop / (step * 1e-3) / 1e12, "ms_per_step": step,
        "steps": args.steps, "warmup": args.warmup,
        "pct_of_peak": {"value": 100 * 2 * flop / (step * 1e-3) / 1e12 / peak, "peak_tflops": peak,
                        "peak_kind": peak_src},
        "kernels_ms": tl["per_kernel"],
        "roofline": _roofline(tl["per_kernel"], {k: flop for k in fused}, peak, peak_src),
        "parity": parity,
        "cpu_baseline": {"value": cpu_flop / cpu_s / 1e12, "unit": "TFLOP/s", "cores": nthreads,
                         "kind": "oracle", "seconds": cpu_s,
                         "sample": f"{len(rows)} sampled rows of the forward and of the backward "
                                   f"GEMM + epilogue (full N, full K), {nthreads} threads"},
        "clocks": tl["clocks"], "gpu_launches": launches * args.steps, "status_ok": ok,
    }
    if cmp is not None:
        c = cmp["per_fn"]
        line["comparison"] = {"per_config": c, "busy_s": cmp["busy_s"]}
        line["epilogue_overhead"] = {
            "fwd": c["fwd_gelu_aux_bias"]["ms_median"] / c["fwd_none"]["ms_median"] - 1,
            "bwd": c["bwd_dgelu_bgrad"]["ms_median"] / c["bwd_none"]["ms_median"] - 1}
        line["fused_vs_torch_unfused"] = {
            "fwd": c["torch_unfused_fwd"]["ms_median"] / c["fwd_gelu_aux_bias"]["ms_median"],
            "bwd": c["torch_unfused_bwd"]["ms_median"] / c["bwd_dgelu_bgrad"]["ms_median"]}
    return [line]


def run_swiglu_workload(args, gf, torch, dev, sp, pk, pk_kind, Ms):
    """SwiGLU MLP at H = 5120, I = 17408, bf16: the fused gate+up forward
    (saving g and u), the down GEMM h Wd^T, and dh = dout Wd with the dSwiGLU
    epilogue, for each M; against the same work unfused in torch (cuBLAS GEMMs
    + elementwise ops) and against one bare GEMM x [Wg; Wu]^T of the same
    flops."""
    import oracle
    import torch.nn.functional as F
    out = []
    nthreads = os.cpu_count() or 1
    rc0 = synth.swiglu(Ms[0])
    host_w = {n: _host(rc0, n) for n in ("Wg", "Wu", "Wd")}
    for Mw in Ms:
        rc = synth.swiglu(Mw)
        H = rc.tensors["x"].shape[1]
        I = rc.tensors["Wg"].shape[0]
        bf = torch.bfloat16
        x = _dev_fill(torch, rc, "x", dev, sp)
        Wgu = torch.empty((2 * I, H), dtype=bf, device=dev)
        Wg = _dev_fill(torch, rc, "Wg", dev, sp, view=Wgu[:I])
        Wu = _dev_fill(torch, rc, "Wu", dev, sp, view=Wgu[I:])
        Wd = _dev_fill(torch, rc, "Wd", dev, sp)
        dout = _dev_fill(torch, rc, "dout", dev, sp)
        h, g, u, dgt, dup = (torch.empty((Mw, I), dtype=bf, device=dev) for _ in range(5))
        o = torch.empty((Mw, H), dtype=bf, device=dev)
        gu = torch.empty((Mw, 2 * I), dtype=bf, device=dev)
        fwd = gf.gf_swiglu_plan(Mw, I, H, gf.GF_BF16, save_gu=True)
        down = gf.gf_matmul_plan_ex(Mw, H, I, gf.GF_BF16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                                    gf.GF_B_NK)
        bwd = gf.gf_dswiglu_plan(Mw, I, H, gf.GF_BF16)
        bare = gf.gf_matmul_plan_ex(Mw, 2 * I, H, gf.GF_BF16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                                    gf.GF_B_NK)
        dh_none = gf.gf_matmul_plan_ex(Mw, I, H, gf.GF_BF16, gf.GF_EPILOG_NONE, gf.GF_BIAS_COL,
                                       gf.GF_B_KN)
        # the bare GEMMs run in the fused plans' kernel and tile configuration
        # (the gate+up kernel's tiles are half as wide as the bare GEMM's of
        # [Wg; Wu]: each output column takes a column of both operands),
        # without a k split
        for a, b, wide_n in ((bare, fwd, 256), (dh_none, bwd, 512)):
            gf.gf_plan_set_option(a, gf.GF_OPT_SPLIT_K, 1)
            d = gf.gf_plan_describe(b)
            kern = (3 if d["tile_n"] == wide_n else 2) if d["tile_m"] == 256 else 1
            gf.gf_plan_set_option(a, gf.GF_OPT_KERNEL, kern)
            if d["tile_m"] != 256:
                gf.gf_plan_set_option(a, gf.GF_OPT_TILE_N, d["tile_n"])
        plans = (fwd, down, bwd, bare, dh_none)
        plan_desc = {"gate_up_swiglu": gf.gf_plan_describe(fwd),
                     "down_none": gf.gf_plan_describe(down),
                     "dh_dswiglu": gf.gf_plan_describe(bwd)}

        def t_gateup():
            gt = torch.matmul(x, Wg.t())
            ut = torch.matmul(x, Wu.t())
            return F.silu(gt) * ut

        def t_dswiglu():
            dh = torch.matmul(dout, Wd)
            sg = torch.sigmoid(g)
            return dh * u * sg * (1 + g * (1 - sg)), dh * (g * sg)

        step_fns = {
            "gate_up_swiglu": lambda: gf.gf_swiglu_execute(fwd, x, Wg, Wu, h, g, u, stream=sp),
            "down_none": lambda: gf.gf_matmul_execute(down, h, Wd, out=o, stream=sp),
            "dh_dswiglu": lambda: gf.gf_dswiglu_execute(bwd, dout, Wd, g, u, dgt, dup, stream=sp),
        }
        f_gu, f_mm = 4.0 * Mw * I * H, 2.0 * Mw * I * H
        flops = {"gate_up_swiglu": f_gu, "down_none": f_mm, "dh_dswiglu": f_mm,
                 "gate_up_bare_gemm": f_gu, "dh_bare_gemm": f_mm,
                 "torch_gate_up_silu_mul": f_gu, "torch_dh_dswiglu": f_mm}
        tl = _timed_steps(torch, step_fns, args.steps, args.warmup, dev.index or 0)
        ok = all(gf.gf_plan_status(p, sp) == gf.GF_OK for p in (fwd, down, bwd))
        rows = synth.sample_rows(Mw, 32, 0)
        ridx = torch.as_tensor(rows, device=dev)
        dv = {k: t.index_select(0, ridx).float().cpu().numpy()
              for k, t in (("h", h), ("g", g), ("u", u), ("out", o), ("d_gate", dgt),
                           ("d_up", dup))}
        cmp = None
        if not args.no_compare:
            cmp = sustained_windows(torch, {
                **step_fns,
                "gate_up_bare_gemm": lambda: gf.gf_matmul_execute(bare, x, Wgu, out=gu, stream=sp),
                "dh_bare_gemm": lambda: gf.gf_matmul_execute(dh_none, dout, Wd, out=h, stream=sp),
                "torch_gate_up_silu_mul": t_gateup,
                "torch_dh_dswiglu": t_dswiglu,
            }, args.cmp_seconds, args.cmp_rounds, dev.index or 0)
        ok = ok and all(gf.gf_plan_status(p, sp) == gf.GF_OK for p in plans)
        for p in plans:
            p.free()
        del x, Wgu, Wg, Wu, Wd, dout, h, g, u, dgt, dup, o, gu
        torch.cuda.empty_cache()

        # the oracle on the sampled rows: forward from x, the down projection
        # of the oracle's own h, the backward from the oracle's own saved g, u
        xs, ds = _host(rc, "x", rows), _host(rc, "dout", rows)
        t_cpu = time.time()
        h_o, g_o, u_o, _, _ = oracle.swiglu_forward(xs, host_w["Wg"], host_w["Wu"], oracle.BF16,
                                                    nthreads=nthreads)
        out_o = oracle.epilog_none(h_o, host_w["Wd"], oracle.BF16, oracle.B_NK, nthreads=nthreads)
        dg_o, du_o, _ = oracle.dswiglu_backward(ds, host_w["Wd"], g_o, u_o, oracle.BF16,
                                                nthreads=nthreads)
        cpu_s = time.time() - t_cpu
        dec = lambda a: oracle.decode(a, oracle.BF16)  # noqa: E731
        parity = _parity_block({"h": _errs(dv["h"], dec(h_o)), "g": _errs(dv["g"], dec(g_o)),
                                "u": _errs(dv["u"], dec(u_o)), "out": _errs(dv["out"], dec(out_o)),
                                "d_gate": _errs(dv["d_gate"], dec(dg_o)),
                                "d_up": _errs(dv["d_up"], dec(du_o))})
        parity["rows"] = len(rows)
        step = tl["ms_total"] / args.steps
        v = (f_gu + 2 * f_mm) / (step * 1e-3) / 1e12
        peak, peak_src = pick_peak(pk, pk_kind, tl["ms_total"] * 1e-3)
        wl = f"swiglu_mlp_bf16_M{Mw}_H{H}_I{I}"
        line = {
            "workload": wl,
            "config": {"workload": wl, "M": Mw, "H": H, "I": I, "seed": 0,
                       "l2": "weights 0.53 GB: larger than L2; no flush"},
            "value": v, "ms_per_step": step, "steps": args.steps, "warmup": args.warmup,
            "pct_of_peak": {"value": 100 * v / peak, "peak_tflops": peak, "peak_kind": peak_src},
            "kernels_ms": tl["per_kernel"],
            "plans": plan_desc,
            "roofline": _roofline(tl["per_kernel"], flops, peak, peak_src),
            "parity": parity,
            "cpu_baseline": {"value": len(rows) / Mw * (f_gu + 2 * f_mm) / cpu_s / 1e12,
                             "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "seconds": cpu_s,
                             "sample": f"{len(rows)} sampled rows of gate+up, down and dh + "
                                       f"dSwiGLU (full widths), {nthreads} threads"},
            "clocks": tl["clocks"],
            "gpu_launches": sum(v["launches"] for v in plan_desc.values()) * args.steps,
            "status_ok": ok,
        }
        if cmp is not None:
            c = cmp["per_fn"]
            line["comparison"] = {"per_config": c, "busy_s": cmp["busy_s"]}
            line["epilogue_overhead"] = {
                "gate_up": c["gate_up_swiglu"]["ms_median"] / c["gate_up_bare_gemm"]["ms_median"] - 1,
                "dh": c["dh_dswiglu"]["ms_median"] / c["dh_bare_gemm"]["ms_median"] - 1}
            line["fused_vs_torch_unfused"] = {
                "gate_up": c["torch_gate_up_silu_mul"]["ms_median"] / c["gate_up_swiglu"]["ms_median"],
                "dh": c["torch_dh_dswiglu"]["ms_median"] / c["dh_dswiglu"]["ms_median"],
                "context": "the page quotes 1.05-1.20x for the fused gate+up forward and ~2.3x "
                           "for the dSwiGLU epilogue, on B200 (not this hardware; not a target)"}
        out.append(line)
    return out


def run_small_workloads(args, gf, torch, dev, sp, pk, pk_kind):
    """The pages' two small workloads, latency-bound (reported, not held to a
    peak fraction): the tiny 2-layer ReLU MLP step (layer-1 forward
    RELU_AUX_BIAS 256x384x512 + backward DRELU_BGRAD G = dY W2^T 256x384x128)
    and the row-bias RELU_BIAS GEMM 1024x512x2048, seeds 0-4. Each is timed
    with its inputs in L2 (back-to-back calls, and replays of a CUDA graph)
    and with L2 flushed before every call; parity over the whole output
    against the oracle; the oracle timed on the whole problem."""
    import oracle
    out = []
    nthreads = os.cpu_count() or 1
    f16 = torch.float16
    peak, peak_src = pick_peak(pk, pk_kind, 0.0)
    # ---------------------------------------------------------------- MLP step
    rc = synth.MLP_TINY
    X, W1, b1, W2, dY = (_dev_fill(torch, rc, n, dev, sp) for n in ("X", "W1", "b1", "W2", "dY"))
    Mx, Kx = rc.tensors["X"].shape
    Nh = rc.tensors["W1"].shape[1]
    No = rc.tensors["W2"].shape[1]
    Y = torch.empty((Mx, Nh), dtype=f16, device=dev)
    aux = torch.empty(((Mx + 31) // 32, Nh), dtype=torch.int32, device=dev)
    G = torch.empty((Mx, Nh), dtype=f16, device=dev)
    bg = torch.empty((Nh,), dtype=torch.float32, device=dev)
    fwd = gf.gf_matmul_plan(Mx, Nh, Kx, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL)
    bwd = gf.gf_matmul_plan_ex(Mx, Nh, No, gf.GF_F16, gf.GF_EPILOG_DRELU_BGRAD, gf.GF_BIAS_COL,
                               gf.GF_B_NK)

    def fused_step():
        gf.gf_matmul_execute(fwd, X, W1, bias=b1, out=Y, aux_out=aux, stream=sp)
        gf.gf_matmul_execute(bwd, dY, W2, out=G, aux_in=aux, bgrad=bg, stream=sp)

    def torch_step():
        z = torch.addmm(b1, X, W1)
        y = torch.relu(z)
        m = z > 0
        g = torch.matmul(dY, W2.t()) * m
        return y, g.float().sum(0)

    # the same step captured once in a CUDA graph: launch overhead removed
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            cs = torch.cuda.current_stream().cuda_stream
            gf.gf_matmul_execute(fwd, X, W1, bias=b1, out=Y, aux_out=aux, stream=cs)
            gf.gf_matmul_execute(bwd, dY, W2, out=G, aux_in=aux, bgrad=bg, stream=cs)
    torch.cuda.current_stream(dev).wait_stream(cap)
    warm = _interleaved(torch, {"fused": fused_step, "fused_graph": graph.replay,
                                "torch_unfused": torch_step}, reps=200)
    cold = _flushed(torch, {"fused": fused_step, "torch_unfused": torch_step}, 50, dev)
    ok = gf.gf_plan_status(fwd, sp) == gf.GF_OK and gf.gf_plan_status(bwd, sp) == gf.GF_OK
    y_d, aux_d, g_d, bg_d = (Y.float().cpu().numpy(), aux.cpu().numpy().view(np.uint32),
                             G.float().cpu().numpy(), bg.cpu().numpy())
    del graph
    mlp_launches = gf.gf_plan_describe(fwd)["launches"] + gf.gf_plan_describe(bwd)["launches"]
    fwd.free()
    bwd.free()
    # oracle: the whole step from the generator's inputs (the oracle's own mask
    # feeds its backward)
    Xh, W1h, b1h, W2h, dYh = (_host(rc, n) for n in ("X", "W1", "b1", "W2", "dY"))
    t_cpu = time.time()
    y_o, words_o, z_o = oracle.relu_aux_bias(Xh, W1h, b1h, oracle.F16, nthreads=nthreads)
    dz_o, bg_o, _ = oracle.drelu_bgrad(dYh, W2h, words_o, oracle.F16, oracle.B_NK,
                                       nthreads=nthreads)
    cpu_s = time.time() - t_cpu
    bits_d = np.unpackbits(aux_d.view(np.uint8), bitorder="little").reshape(
        aux_d.shape[0], Nh, 32).transpose(0, 2, 1).reshape(-1, Nh)[:Mx]
    band = np.abs(z_o) < 1e-3 * np.abs(z_o).max(axis=1, keepdims=True)
    diff = bits_d.astype(bool) != (z_o > 0)
    parity = _parity_block({"Y": _errs(y_d, oracle.decode(y_o, oracle.F16)),
                            "G": _errs(g_d, oracle.decode(dz_o, oracle.F16)),
                            "bgrad": _errs(bg_d, bg_o)}, bgrad_keys=("bgrad",),
                           mask={"mask_mismatch_outside_band": int((diff & ~band).sum()),
                                 "mask_mismatch_in_band": int((diff & band).sum())})
    parity["what"] = "every element of Y, relu_aux, G and bgrad"
    flop = 2.0 * Mx * Nh * Kx + 2.0 * Mx * Nh * No
    wl = f"mlp2_relu_fp16_fwd_{Mx}x{Nh}x{Kx}_bwd_{Mx}x{Nh}x{No}"
    ms = warm["fused"]["median"]
    out.append({
        "workload": wl, "config": {"workload": wl, "seed": 0,
                                   "l2": "both: inputs in L2 (warm) and L2 flushed before each call"},
        "value": flop / (ms * 1e-3) / 1e12, "ms_per_step": ms,
        "us_per_step": {"warm_direct": {k: 1e3 * v for k, v in warm["fused"].items()},
                        "warm_graph_replay": {k: 1e3 * v for k, v in warm["fused_graph"].items()},
                        "l2_flushed_direct": {k: 1e3 * v for k, v in cold["fused"].items()}},
        "torch_unfused_us": {"warm": 1e3 * warm["torch_unfused"]["median"],
                             "l2_flushed": 1e3 * cold["torch_unfused"]["median"]},
        "fused_vs_torch_unfused": {"warm": warm["torch_unfused"]["median"] / ms,
                                   "l2_flushed": cold["torch_unfused"]["median"] /
                                   cold["fused"]["median"]},
        "roofline": {"bound": "tensor", "kernel": f"forward + backward (one step, {mlp_launches} "
                                                  "launches)",
                     "achieved": flop / (ms * 1e-3) / 1e12, "peak": peak, "unit": "TFLOP/s",
                     "frac": flop / (ms * 1e-3) / 1e12 / peak, "traffic": None,
                     "peak_source": peak_src,
                     "note": f"latency-bound: 0.13 GFLOP over {mlp_launches} launches; not held "
                             "to a fraction"},
        "parity": parity,
        "cpu_baseline": {"value": flop / cpu_s / 1e12, "unit": "TFLOP/s", "cores": nthreads,
                         "kind": "oracle", "seconds": cpu_s,
                         "sample": f"the whole step (forward, backward, bias gradient), "
                                   f"{nthreads} threads"},
        "launches_per_step": mlp_launches, "status_ok": ok})

    # ------------------------------------------------------------ row-bias GEMM
    rc = synth.RELU_BIAS_ROW
    Mr, Kr = rc.tensors["A"].shape
    Nr = rc.tensors["B"].shape[1]
    plan = gf.gf_matmul_plan(Mr, Nr, Kr, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    nosplit = gf.gf_matmul_plan(Mr, Nr, Kr, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    gf.gf_plan_set_option(nosplit, gf.GF_OPT_SPLIT_K, 1)
    errs = {}
    cpu_s = 0.0
    timing = None
    for seed in rc.seeds:
        A = torch.empty((Mr, Kr), dtype=f16, device=dev)
        B = torch.empty((Kr, Nr), dtype=f16, device=dev)
        bias = torch.empty((Mr,), dtype=f16, device=dev)
        for t, n in ((A, "A"), (B, "B"), (bias, "bias")):
            tt = rc.tensors[n]
            synth.dev_normal(t, rc.dtype, seed, tt.tensor_id, tt.sigma, sp)
        Yr = torch.empty((Mr, Nr), dtype=f16, device=dev)
        if timing is None:  # seed 0: the timing
            graphs = {}
            for name, pl in (("fused_graph", plan), ("fused_graph_no_split", nosplit)):
                g = torch.cuda.CUDAGraph()
                cap.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(cap):
                    with torch.cuda.graph(g, stream=cap):
                        cs = torch.cuda.current_stream().cuda_stream
                        for _ in range(20):
                            gf.gf_matmul_execute(pl, A, B, bias=bias, out=Yr, stream=cs)
                torch.cuda.current_stream(dev).wait_stream(cap)
                graphs[name] = g
            fused = lambda: gf.gf_matmul_execute(plan, A, B, bias=bias, out=Yr, stream=sp)  # noqa
            unf = lambda: torch.relu(torch.addmm(bias[:, None], A, B))  # noqa: E731
            w = _interleaved(torch, {"fused": fused, "fused_graph": graphs["fused_graph"].replay,
                                     "fused_graph_no_split": graphs["fused_graph_no_split"].replay,
                                     "torch_unfused": unf}, reps=200)
            c = _flushed(torch, {"fused": fused, "torch_unfused": unf}, 50, dev)
            timing = (w, c)
            del graphs
        gf.gf_matmul_execute(plan, A, B, bias=bias, out=Yr, stream=sp)
        y_d = Yr.float().cpu().numpy()
        Ah, Bh, bh = (synth.normal(rc.tensors[n].shape, rc.dtype, seed, rc.tensors[n].tensor_id,
                                   rc.tensors[n].sigma) for n in ("A", "B", "bias"))
        t_cpu = time.time()
        y_o, _ = oracle.relu_bias(Ah, Bh, bh, oracle.F16, axis=oracle.BIAS_ROW, nthreads=nthreads)
        cpu_s += time.time() - t_cpu
        errs[f"Y_seed{seed}"] = _errs(y_d, oracle.decode(y_o, oracle.F16))
        del A, B, bias, Yr
    w, c = timing
    ok = gf.gf_plan_status(plan, sp) == gf.GF_OK and gf.gf_plan_status(nosplit, sp) == gf.GF_OK
    desc = gf.gf_plan_describe(plan)
    plan.free()
    nosplit.free()
    parity = _parity_block(errs)
    parity["what"] = f"every element of Y, seeds {list(rc.seeds)}"
    flop = 2.0 * Mr * Nr * Kr
    ms = w["fused"]["median"]
    g_ms = w["fused_graph"]["median"] / 20
    wl = f"relu_bias_rowbias_fp16_{Mr}x{Nr}x{Kr}"
    out.append({
        "workload": wl, "config": {"workload": wl, "seeds": list(rc.seeds),
                                   "l2": "both: inputs in L2 (warm) and L2 flushed before each call"},
        "value": flop / (ms * 1e-3) / 1e12, "ms_per_step": ms,
        "us_per_step": {"warm_direct": {k: 1e3 * v for k, v in w["fused"].items()},
                        "warm_graph_replay": {k: 1e3 * v / 20 for k, v in w["fused_graph"].items()},
                        "warm_graph_replay_no_split": {k: 1e3 * v / 20 for k, v in
                                                       w["fused_graph_no_split"].items()},
                        "l2_flushed_direct": {k: 1e3 * v for k, v in c["fused"].items()}},
        "graph_replay_tflops": flop / (g_ms * 1e-3) / 1e12,
        "torch_unfused_us": {"warm": 1e3 * w["torch_unfused"]["median"],
                             "l2_flushed": 1e3 * c["torch_unfused"]["median"]},
        "fused_vs_torch_unfused": {"warm": w["torch_unfused"]["median"] / ms,
                                   "l2_flushed": c["torch_unfused"]["median"] /
                                   c["fused"]["median"]},
        "roofline": {"bound": "tensor", "kernel": "RELU_BIAS (k split)",
                     "achieved": flop / (ms * 1e-3) / 1e12, "peak": peak, "unit": "TFLOP/s",
                     "frac": flop / (ms * 1e-3) / 1e12 / peak, "traffic": None,
                     "peak_source": peak_src,
                     "note": "latency-bound: 32 output tiles of 128 x 128 on 152 SMs"},
        "parity": parity,
        "cpu_baseline": {"value": flop * len(rc.seeds) / cpu_s / 1e12, "unit": "TFLOP/s",
                         "cores": nthreads, "kind": "oracle", "seconds": cpu_s,
                         "sample": f"the whole GEMM + epilogue for each of {len(rc.seeds)} "
                                   f"seeds, {nthreads} threads"},
        "plan": desc, "launches_per_step": 1, "status_ok": ok})
    return out


def run_workload(args):
    """`--workload gelu|swiglu|small`: the pages' other workloads, one JSON
    line each, with the same blocks as the headline line (throughput, the
    kernels' times, roofline, sampled parity against the oracle, the oracle
    as a timed CPU baseline, clocks) plus the epilogue overhead against a
    bare GEMM and the unfused torch time of the same work."""
    import torch

    import gemm_epilogue_tmem_gb300 as gf
    gf.build()
    synth.build_cuda()
    dev = torch.device("cuda", torch.cuda.current_device())
    sp = torch.cuda.current_stream().cuda_stream
    pk_d, kind = peaks()
    if args.workload == "gelu":
        lines = run_gelu_workload(args, gf, torch, dev, sp, pk_d, kind)
    elif args.workload == "small":
        lines = run_small_workloads(args, gf, torch, dev, sp, pk_d, kind)
    else:
        Ms = [int(v) for v in args.swiglu_m.split(",")]
        lines = run_swiglu_workload(args, gf, torch, dev, sp, pk_d, kind, Ms)
    for ln in lines:
        print(json.dumps({"metric": METRIC, "unit": "TFLOP/s", "n_gpus": 1,
                          "dtype": "f16" if args.workload == "small" else "bf16",
                          "data": "synthetic", "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, **ln}), flush=True)
    return 0 if all(ln["status_ok"] and ln["parity"]["pass"] for ln in lines) else 1


def run_compare_schedules(args):
    """Steady-state comparison of the CTA-pair kernel's tile schedules on the
    full-size fused forward, and torch.matmul (cuBLAS, no epilogue) for
    context: each configuration runs `--seconds` back to back after a
    warm-up while nvidia-smi samples SM clock and power; the list is run
    twice. One JSON line per run."""
    import torch

    import gemm_epilogue_tmem_gb300 as gf

    gf.build()
    synth.build_cuda()
    sp = torch.cuda.current_stream().cuda_stream
    X = torch.empty((M, K), dtype=torch.float16, device="cuda")
    W = torch.empty((K, N), dtype=torch.float16, device="cuda")
    bias = torch.empty((N,), dtype=torch.float16, device="cuda")
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    aux = torch.empty((M // 32, N), dtype=torch.int32, device="cuda")
    synth.dev_normal(X, synth.F16, 0, synth.TID_A, 1.0, sp)
    synth.dev_normal(W, synth.F16, 0, synth.TID_B, 1 / 128, sp)
    synth.dev_normal(bias, synth.F16, 0, synth.TID_BIAS, 0.1, sp)
    torch.cuda.synchronize()
    cfgs = {}
    for name, sched, kern in (("dynamic", 2, 2), ("static", 3, 2), ("one_tile_per_pair", 1, 2),
                              ("wide_256x512_dynamic", 2, 3)):
        plan = gf.gf_matmul_plan_ex(M, N, K, gf.GF_F16, gf.GF_EPILOG_RELU_AUX_BIAS, gf.GF_BIAS_COL,
                                    gf.GF_B_KN)
        gf.gf_plan_set_option(plan, gf.GF_OPT_KERNEL, kern)
        gf.gf_plan_set_option(plan, gf.GF_OPT_SCHEDULE, sched)
        cfgs[name] = (plan, (lambda p: lambda: gf.gf_matmul_execute(
            p, X, W, bias=bias, out=Y, aux_out=aux, stream=sp))(plan))
    cfgs["cublas_matmul_no_epilogue"] = (None, lambda: torch.matmul(X, W, out=Y))

    def run(fn):
        sampler = ClockSampler(0)
        sampler.start()
        t_end = time.time() + 1.5
        while time.time() < t_end:
            fn()
            torch.cuda.synchronize()
        n0 = len(sampler.lines)
        times = []
        t_end = time.time() + args.seconds
        while time.time() < t_end:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        sampler.keep_from(n0)
        clk = sampler.stop()
        ms = statistics.median(times)
        return {"ms": ms, "tflops": FLOP_PER_GEMM / (ms * 1e-3) / 1e12, "sm_mhz": clk["sm_mhz"],
                "power_w": clk.get("power_w_median"), "launches": len(times),
                "gcycles": ms * 1e-3 * clk["sm_mhz"] * 1e6 / 1e9 if clk["sm_mhz"] else None}

    for rnd in range(2):
        for name, (plan, fn) in cfgs.items():
            print(json.dumps({"config": name, "repeat": rnd, "shape": [M, N, K], **run(fn)}),
                  flush=True)
    for plan, _ in cfgs.values():
        if plan is not None:
            plan.free()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--compare-schedules", action="store_true",
                    help="steady-state comparison of the tile schedules (not the bench line)")
    ap.add_argument("--seconds", type=float, default=4.0)
    ap.add_argument("--profile-case", default="",
                    help="M,N,K: run one fused GEMM of this shape (for ncu captures)")
    ap.add_argument("--epilog", default="relu_aux_bias",
                    choices=["relu_aux_bias", "drelu_bgrad", "none", "relu_bias", "swiglu_save",
                             "dswiglu", "gelu_aux_bias", "dgelu_bgrad"])
    ap.add_argument("--kernel", type=int, default=0,
                    help="0 plan's choice, 1 single CTA, 2 pair, 3 pair with 256 x 512 tiles")
    ap.add_argument("--l2-hints", type=int, default=-1,
                    help="--profile-case: GF_OPT_L2_HINTS of the plan (-1: the plan's default)")
    ap.add_argument("--group-m", type=int, default=0,
                    help="--profile-case: GF_OPT_GROUP_M of the plan (0: the plan's default)")
    ap.add_argument("--split", type=int, default=0,
                    help="--profile-case: GF_OPT_SPLIT_K of the plan (0: the plan's choice, "
                         "1: none)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gf", choices=["gf", "reference"])
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="sampled rows per GEMM in the CPU-oracle baseline of the GPU run")
    ap.add_argument("--ref-step-rows", type=int, default=4,
                    help="sampled rows per GEMM in each step of --impl reference")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-depth", type=int, default=2,
                    help="buffer sets of the e2e pipeline (inputs and outputs of that many "
                         "steps in flight)")
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the steady-state comparison (NONE epilogue, cuBLAS, unfused torch)")
    ap.add_argument("--cmp-seconds", type=float, default=1.0,
                    help="seconds per configuration and round in the steady-state comparison")
    ap.add_argument("--cmp-rounds", type=int, default=2)
    ap.add_argument("--autotune", action="store_true",
                    help="let gf_matmul_autotune pick the kernels before the warm-up")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="linear_pair",
                    choices=["linear_pair", "gelu", "swiglu", "small"],
                    help="gelu / swiglu / small: the other workloads, one JSON line each")
    ap.add_argument("--swiglu-m", default="2048,8192,16384")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gf":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_case:
        return run_profile_case(args)
    if args.compare_schedules:
        return run_compare_schedules(args)
    if args.workload != "linear_pair":
        return run_workload(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
