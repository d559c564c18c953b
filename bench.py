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
                               "linear_pair_fp16_65536x16384x8192_dram_traffic.md")


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
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


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
    every output device -> host. Copies of step i+1 / i-1 run on their own
    streams under the compute of step i (two buffer sets), the way a training
    or serving loop would overlap them."""
    host_in = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in dev_in0.items()}
    for n, t in dev_in0.items():
        host_in[n].copy_(t)
    host_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                 for n, t in dev_out0.items()} for _ in range(2)]
    dev_in = [dev_in0, {n: torch.empty_like(t) for n, t in dev_in0.items()}]
    dev_out = [dev_out0, {n: torch.empty_like(t) for n, t in dev_out0.items()}]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_comp = torch.cuda.current_stream(dev)
    sc = s_comp.cuda_stream
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            b = i % 2
            if i >= 2:
                s_h2d.wait_event(comp_done[b])
            with torch.cuda.stream(s_h2d):
                for k, t in dev_in[b].items():
                    t.copy_(host_in[k], non_blocking=True)
            h2d_done[b].record(s_h2d)
            s_comp.wait_event(h2d_done[b])
            if i >= 2:
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

    run(2)
    barrier()
    n = max(3, min(args.steps, 10))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_h2d)
    run(n)
    s_d2h.wait_event(d2h_done[(n - 1) % 2])
    t1.record(s_d2h)
    barrier()
    ms = t0.elapsed_time(t1) / n
    ok = gf.gf_plan_status(fwd, sc) == gf.GF_OK and gf.gf_plan_status(bwd, sc) == gf.GF_OK
    del host_in, host_out, dev_in, dev_out
    torch.cuda.empty_cache()
    return {"value": world * 2 * FLOP_PER_GEMM / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "steps": n, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "H2D of step i+1 and D2H of step i-1 on their own streams under step i",
            "status_ok": ok}


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
    launches_per_step = 3  # fused forward, fused backward, bgrad finalize
    if args.kernel:
        for pl in (fwd, bwd, fwd_none, bwd_none):
            gf.gf_plan_set_option(pl, gf.GF_OPT_KERNEL, args.kernel)
    if args.autotune:
        gf.gf_matmul_autotune(fwd, X, W, bias=bias, out=Y, aux_out=aux, stream=sp, reps=2)
        gf.gf_matmul_autotune(bwd, dY, W, out=dZ, aux_in=mask, bgrad=bgrad, stream=sp, reps=2)
    plans = {"fwd": gf.gf_plan_describe(fwd), "bwd": gf.gf_plan_describe(bwd),
             "autotuned": bool(args.autotune)}

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
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
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

    # epilogue overhead: the same kernels and tiles with no epilogue
    # interleaved, so that clock and power drift hit both variants alike
    def one(fn):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    f_none = lambda: gf.gf_matmul_execute(fwd_none, X, W, out=Y, stream=sp)  # noqa: E731
    f_epi = lambda: gf.gf_matmul_execute(fwd, X, W, bias=bias, out=Y, aux_out=aux,  # noqa: E731
                                         stream=sp)
    b_none = lambda: gf.gf_matmul_execute(bwd_none, dY, W, out=dZ, stream=sp)  # noqa: E731
    b_epi = lambda: gf.gf_matmul_execute(bwd, dY, W, out=dZ, aux_in=mask, bgrad=bgrad,  # noqa: E731
                                         stream=sp)
    samples = {"fn": [], "fe": [], "bn": [], "be": []}
    for _ in range(max(3, min(args.steps, 7))):
        samples["fn"].append(one(f_none))
        samples["fe"].append(one(f_epi))
        samples["bn"].append(one(b_none))
        samples["be"].append(one(b_epi))
    t_fwd_none, t_fwd_epi = statistics.median(samples["fn"]), statistics.median(samples["fe"])
    t_bwd_none, t_bwd_epi = statistics.median(samples["bn"]), statistics.median(samples["be"])

    # context only: the same two products through torch.matmul (cuBLAS), no epilogue
    cublas = None
    if not args.no_cublas:
        Wt = W.t()
        c_f = lambda: torch.matmul(X, W, out=Y)  # noqa: E731
        c_b = lambda: torch.matmul(dY, Wt, out=dZ)  # noqa: E731
        cf, cb = [], []
        for _ in range(max(3, min(args.steps, 5))):
            cf.append(one(c_f))
            cb.append(one(c_b))
        cublas = {"fwd_ms": statistics.median(cf), "bwd_ms": statistics.median(cb),
                  "fwd_tflops": FLOP_PER_GEMM / (statistics.median(cf) * 1e-3) / 1e12,
                  "bwd_tflops": FLOP_PER_GEMM / (statistics.median(cb) * 1e-3) / 1e12,
                  "note": "torch.matmul of the same operands, no epilogue; context, not the metric"}

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
    fwd_avg, bwd_avg = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    rec = recorded_traffic()
    traffic = None if rec is None else (rec[0] if fwd_avg >= bwd_avg else rec[1])
    dom_name, dom_ms = ("fused forward RELU_AUX_BIAS", fwd_avg) if fwd_avg >= bwd_avg else \
        ("fused backward DRELU_BGRAD (+ finalize)", bwd_avg)
    peak_key = "bf16_tflops_sustained" if "bf16_tflops_sustained" in pk else "bf16_tflops"
    peak = float(pk[peak_key])
    achieved = FLOP_PER_GEMM / (dom_ms * 1e-3) / 1e12

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
                        "peak_kind": f"{pk_kind} {peak_key}",
                        "vs_nominal_2250": 100 * value / world / 2250.0},
        "roofline": {"bound": "tensor", "kernel": dom_name, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{pk_kind} {peak_key}",
                     "algorithmic_flop_per_launch": FLOP_PER_GEMM},
        "kernels_ms": {"fwd_relu_aux_bias": fwd_avg, "bwd_drelu_bgrad": bwd_avg,
                       "fwd_none": t_fwd_none, "bwd_none": t_bwd_none,
                       "fwd_epi_isolated": t_fwd_epi, "bwd_epi_isolated": t_bwd_epi},
        "epilogue_overhead": {"fwd": t_fwd_epi / t_fwd_none - 1, "bwd": t_bwd_epi / t_bwd_none - 1},
        "cublas_same_shapes": cublas,
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
    """Median ms per call of each function: `reps` back-to-back calls between
    two events on the current stream, the functions taken in turn `rounds`
    times so that clock and power drift fall on all of them alike."""
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
    return {k: statistics.median(v) for k, v in times.items()}


def _dev_fill(torch, recipe, name, dev, sp, view=None):
    t = recipe.tensors[name]
    tdt = torch.float16 if recipe.dtype == synth.F16 else torch.bfloat16
    x = view if view is not None else torch.empty(t.shape, dtype=tdt, device=dev)
    synth.dev_normal(x, recipe.dtype, 0, t.tensor_id, t.sigma, sp)
    return x


def run_gelu_workload(args, gf, torch, dev, sp, peak, pk):
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
    # the bare GEMMs run in the fused plans' kernel and tile configuration
    for a, b in (("fwd_none", "fwd"), ("bwd_none", "bwd")):
        d = gf.gf_plan_describe(plan[b])
        gf.gf_plan_set_option(plan[a], gf.GF_OPT_KERNEL, 2 if d["tile_m"] == 256 else 1)
        if d["tile_m"] != 256:
            gf.gf_plan_set_option(plan[a], gf.GF_OPT_TILE_N, d["tile_n"])
    ex = gf.gf_matmul_execute

    def unfused_fwd():
        torch.addmm(bias, X, W, out=pre)
        F.gelu(pre, approximate="tanh")

    def unfused_bwd():
        g = torch.matmul(dY, W.t())
        dz = torch.ops.aten.gelu_backward(g, pre_b, approximate="tanh")
        dz.float().sum(0)

    fns = {
        "fwd_gelu_aux_bias": lambda: ex(plan["fwd"], X, W, bias=bias, out=Y, aux_out=pre,
                                        stream=sp),
        "bwd_dgelu_bgrad": lambda: ex(plan["bwd"], dY, W, out=dX, aux_in=pre_b, bgrad=bgrad,
                                      stream=sp),
        "fwd_none": lambda: ex(plan["fwd_none"], X, W, out=Y, stream=sp),
        "bwd_none": lambda: ex(plan["bwd_none"], dY, W, out=dX, stream=sp),
        "torch_unfused_fwd": unfused_fwd,
        "torch_unfused_bwd": unfused_bwd,
    }
    flop = 2.0 * Mg * Ng * Kg
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    ms = _interleaved(torch, fns, reps=max(5, args.steps))
    clk = clocks.stop()
    ok = all(gf.gf_plan_status(p, sp) == gf.GF_OK for p in plan.values())
    for p in plan.values():
        p.free()
    step = ms["fwd_gelu_aux_bias"] + ms["bwd_dgelu_bgrad"]
    return {
        "workload": f"gelu_bf16_fwd_gelu_aux_bias_bwd_dgelu_bgrad_{Mg}x{Ng}x{Kg}",
        "value": 2 * flop / (step * 1e-3) / 1e12, "ms_per_step": step,
        "pct_of_peak": 100 * 2 * flop / (step * 1e-3) / 1e12 / peak, "peak_source": pk,
        "kernels_ms": ms,
        "kernels_tflops": {k: flop / (v * 1e-3) / 1e12 for k, v in ms.items()},
        "epilogue_overhead": {"fwd": ms["fwd_gelu_aux_bias"] / ms["fwd_none"] - 1,
                              "bwd": ms["bwd_dgelu_bgrad"] / ms["bwd_none"] - 1},
        "fused_vs_torch_unfused": {"fwd": ms["torch_unfused_fwd"] / ms["fwd_gelu_aux_bias"],
                                   "bwd": ms["torch_unfused_bwd"] / ms["bwd_dgelu_bgrad"]},
        "clocks": clk, "status_ok": ok,
    }


def run_swiglu_workload(args, gf, torch, dev, sp, peak, pk, Ms):
    """SwiGLU MLP at H = 5120, I = 17408, bf16: the fused gate+up forward
    (saving g and u), the down GEMM h Wd^T, and dh = dout Wd with the dSwiGLU
    epilogue, for each M; against the same work unfused in torch (cuBLAS GEMMs
    + elementwise ops) and against one bare GEMM x [Wg; Wu]^T of the same
    flops."""
    import torch.nn.functional as F
    out = []
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

        def t_gateup():
            gt = torch.matmul(x, Wg.t())
            ut = torch.matmul(x, Wu.t())
            return F.silu(gt) * ut

        def t_dswiglu():
            dh = torch.matmul(dout, Wd)
            sg = torch.sigmoid(g)
            return dh * u * sg * (1 + g * (1 - sg)), dh * (g * sg)

        fns = {
            "gate_up_swiglu": lambda: gf.gf_swiglu_execute(fwd, x, Wg, Wu, h, g, u, stream=sp),
            "down_none": lambda: gf.gf_matmul_execute(down, h, Wd, out=o, stream=sp),
            "dh_dswiglu": lambda: gf.gf_dswiglu_execute(bwd, dout, Wd, g, u, dgt, dup, stream=sp),
            "gate_up_bare_gemm": lambda: gf.gf_matmul_execute(bare, x, Wgu, out=gu, stream=sp),
            "dh_bare_gemm": lambda: gf.gf_matmul_execute(dh_none, dout, Wd, out=h, stream=sp),
            "torch_gate_up_silu_mul": t_gateup,
            "torch_dh_dswiglu": t_dswiglu,
        }
        clocks = ClockSampler(dev.index or 0)
        clocks.start()
        ms = _interleaved(torch, fns, reps=max(5, args.steps))
        clk = clocks.stop()
        ok = all(gf.gf_plan_status(p, sp) == gf.GF_OK for p in (fwd, down, bwd, bare, dh_none))
        for p in (fwd, down, bwd, bare, dh_none):
            p.free()
        f_gu, f_mm = 4.0 * Mw * I * H, 2.0 * Mw * I * H
        flops = {"gate_up_swiglu": f_gu, "down_none": f_mm, "dh_dswiglu": f_mm,
                 "gate_up_bare_gemm": f_gu, "dh_bare_gemm": f_mm,
                 "torch_gate_up_silu_mul": f_gu, "torch_dh_dswiglu": f_mm}
        step = ms["gate_up_swiglu"] + ms["down_none"] + ms["dh_dswiglu"]
        v = (f_gu + 2 * f_mm) / (step * 1e-3) / 1e12
        out.append({
            "workload": f"swiglu_mlp_bf16_M{Mw}_H{H}_I{I}", "M": Mw,
            "value": v, "ms_per_step": step, "pct_of_peak": 100 * v / peak, "peak_source": pk,
            "kernels_ms": ms,
            "kernels_tflops": {k: flops[k] / (t * 1e-3) / 1e12 for k, t in ms.items()},
            "epilogue_overhead": {"gate_up": ms["gate_up_swiglu"] / ms["gate_up_bare_gemm"] - 1,
                                  "dh": ms["dh_dswiglu"] / ms["dh_bare_gemm"] - 1},
            "fused_vs_torch_unfused": {
                "gate_up": ms["torch_gate_up_silu_mul"] / ms["gate_up_swiglu"],
                "dh": ms["torch_dh_dswiglu"] / ms["dh_dswiglu"]},
            "clocks": clk, "status_ok": ok,
        })
        del x, Wgu, Wg, Wu, Wd, dout, h, g, u, dgt, dup, o, gu
        torch.cuda.empty_cache()
    return out


def run_small_workloads(args, gf, torch, dev, sp, peak, pk):
    """The pages' two small workloads, latency-bound (reported, not held to a
    peak fraction): the tiny 2-layer ReLU MLP step (layer-1 forward
    RELU_AUX_BIAS 256x384x512 + backward DRELU_BGRAD G = dY W2^T 256x384x128)
    and the row-bias RELU_BIAS GEMM 1024x512x2048; per launch, L2 warm
    (the inputs fit in L2), against the same work unfused in torch."""
    out = []
    f16 = torch.float16
    # MLP step
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
    ms = _interleaved(torch, {"fused": fused_step, "fused_graph": graph.replay,
                              "torch_unfused": torch_step}, reps=200)
    flop = 2.0 * Mx * Nh * Kx + 2.0 * Mx * Nh * No
    ok = gf.gf_plan_status(fwd, sp) == gf.GF_OK and gf.gf_plan_status(bwd, sp) == gf.GF_OK
    out.append({"workload": f"mlp2_relu_fp16_fwd_{Mx}x{Nh}x{Kx}_bwd_{Mx}x{Nh}x{No}",
                "value": flop / (ms["fused"] * 1e-3) / 1e12, "ms_per_step": ms["fused"],
                "us_per_step": 1e3 * ms["fused"], "graph_replay_us": 1e3 * ms["fused_graph"],
                "torch_unfused_us": 1e3 * ms["torch_unfused"],
                "fused_vs_torch_unfused": ms["torch_unfused"] / ms["fused"], "launches_per_step": 3,
                "l2": "inputs fit in L2 (latency-bound)", "status_ok": ok})
    del graph
    fwd.free()
    bwd.free()
    # row-bias RELU_BIAS
    rc = synth.RELU_BIAS_ROW
    A, B, bias = (_dev_fill(torch, rc, n, dev, sp) for n in ("A", "B", "bias"))
    Mr, Kr = rc.tensors["A"].shape
    Nr = rc.tensors["B"].shape[1]
    Yr = torch.empty((Mr, Nr), dtype=f16, device=dev)
    plan = gf.gf_matmul_plan(Mr, Nr, Kr, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    # 20 launches captured once (launch overhead of the host removed), the
    # same with the k split switched off, and cuBLAS + torch unfused
    nosplit = gf.gf_matmul_plan(Mr, Nr, Kr, gf.GF_F16, gf.GF_EPILOG_RELU_BIAS, gf.GF_BIAS_ROW)
    gf.gf_plan_set_option(nosplit, gf.GF_OPT_SPLIT_K, 1)
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
    ms = _interleaved(torch, {
        "fused": lambda: gf.gf_matmul_execute(plan, A, B, bias=bias, out=Yr, stream=sp),
        "fused_graph": graphs["fused_graph"].replay,
        "fused_graph_no_split": graphs["fused_graph_no_split"].replay,
        "torch_unfused": lambda: torch.relu(torch.addmm(bias[:, None], A, B)),
    }, reps=200)
    g_ms = ms["fused_graph"] / 20
    flop = 2.0 * Mr * Nr * Kr
    out.append({"workload": f"relu_bias_rowbias_fp16_{Mr}x{Nr}x{Kr}",
                "value": flop / (ms["fused"] * 1e-3) / 1e12, "ms_per_step": ms["fused"],
                "us_per_step": 1e3 * ms["fused"], "graph_replay_us": 1e3 * g_ms,
                "graph_replay_tflops": flop / (g_ms * 1e-3) / 1e12,
                "graph_replay_no_split_us": 1e3 * ms["fused_graph_no_split"] / 20,
                "torch_unfused_us": 1e3 * ms["torch_unfused"],
                "fused_vs_torch_unfused": ms["torch_unfused"] / ms["fused"], "launches_per_step": 1,
                "plan": gf.gf_plan_describe(plan), "l2": "inputs fit in L2 (latency-bound)",
                "status_ok": gf.gf_plan_status(plan, sp) == gf.GF_OK and
                gf.gf_plan_status(nosplit, sp) == gf.GF_OK})
    del graphs
    plan.free()
    nosplit.free()
    return out


def run_workload(args):
    """`--workload gelu|swiglu`: the pages' other two workloads, one JSON line
    each, with the fused kernels' throughput, the epilogue overhead against a
    bare GEMM of the same flops and the unfused torch (cuBLAS + elementwise)
    time of the same work."""
    import torch

    import gemm_epilogue_tmem_gb300 as gf
    gf.build()
    synth.build_cuda()
    dev = torch.device("cuda", torch.cuda.current_device())
    sp = torch.cuda.current_stream().cuda_stream
    pk_d, kind = peaks()
    key = "bf16_tflops_sustained"
    peak = float(pk_d.get(key) or FALLBACK[key])
    pk = f"{kind} {key}"
    if args.workload == "gelu":
        lines = [run_gelu_workload(args, gf, torch, dev, sp, peak, pk)]
    elif args.workload == "small":
        lines = run_small_workloads(args, gf, torch, dev, sp, peak, pk)
    else:
        Ms = [int(v) for v in args.swiglu_m.split(",")]
        lines = run_swiglu_workload(args, gf, torch, dev, sp, peak, pk, Ms)
    for ln in lines:
        print(json.dumps({"metric": METRIC, "unit": "TFLOP/s",
                          "dtype": "f16" if args.workload == "small" else "bf16",
                          "data": "synthetic", "higher_is_better": True, **ln}), flush=True)
    return 0 if all(ln["status_ok"] for ln in lines) else 1


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
        sampler.lines = sampler.lines[n0:]
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
                             "dswiglu"])
    ap.add_argument("--kernel", type=int, default=0,
                    help="0 plan's choice, 1 single CTA, 2 pair, 3 pair with 256 x 512 tiles")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gf", choices=["gf", "reference"])
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="sampled rows per GEMM in the CPU-oracle baseline of the GPU run")
    ap.add_argument("--ref-step-rows", type=int, default=4,
                    help="sampled rows per GEMM in each step of --impl reference")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
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
