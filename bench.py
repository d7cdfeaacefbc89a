"""Benchmark of the DISCO hot path on one or more GPUs (replicas).

One step = the whole hot path on one batch of the largest workload
(B=1, C=256 -> 256, 721x1440 -> 361x720, K=9 anisotropic, bf16):
disco_fwd (x -> X), disco_bwd (G -> gx), disco_fused_conv (x, W -> y) and
disco_fused_conv_bwd_input (dy, W -> gx).  The metric is the forward +
transpose contraction throughput in algorithmic HBM GB/s (compulsory bytes:
input + output + psi), with the fused convolution's ms/call alongside.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica (no data-path
collective; the path shards by batch), timing is max over ranks and rank 0
prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "down_fused_bwd_721x1440_to_361x720"
# the oracle arm's warm-up and timed steps together take about this long
REF_TOTAL_S = 150.0
METRIC = "DISCO fwd/bwd contraction HBM GB/s (% of peak); fused conv ms/call"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

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
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
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
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks (the job's time is the
    slowest rank's); the values themselves on a single process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def algorithmic(w, psi_c):
    """Compulsory bytes and useful flops per call (see the design notes)."""
    esz = 2 if w.dtype == "bf16" else 4
    B, C, K = w.B, w.C, w.K
    Hin, Win = w.grid_in[:2]
    Hout, Wout = w.grid_out[:2]
    x = B * C * Hin * Win * esz
    X = B * C * K * Hout * Wout * esz
    psi = psi_c.nruns * 32 + psi_c.nhval * psi_c.K_pad * 4 + (Hout + 1) * 8
    out = {"fwd_bytes": x + X + psi, "bwd_bytes": X + x + psi,
           "csr_flops": 2.0 * B * C * Wout * psi_c.nnz_csr}
    if w.Cout is not None:
        y = B * w.Cout * Hout * Wout * esz
        Wb = w.Cout * C * K * esz
        out["fused_bytes"] = x + Wb + y + psi
        out["fused_bwd_bytes"] = y + Wb + x + psi
        out["einsum_flops"] = 2.0 * B * w.Cout * C * K * Hout * Wout
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    import sparse_spherical_convolution_gb300 as d
    from sparse_spherical_convolution_gb300.workloads import WORKLOADS

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    d.load_library()
    psi = d.Psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    B, C, Co, K = w.B, w.C, w.Cout, w.K
    sh = w.shapes()
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 1000 + rank)
    dt = w.torch_dtype
    x = torch.randn(sh["x"], generator=g, device=dev).to(dt)
    G = torch.randn(sh["X"], generator=g, device=dev).to(dt)
    Wt = (torch.randn(sh["W"], generator=g, device=dev) / math.sqrt(C * K)).to(dt)
    dy = torch.randn(sh["y"], generator=g, device=dev).to(dt)
    X = torch.empty(sh["X"], dtype=dt, device=dev)
    gx = torch.empty(sh["x"], dtype=dt, device=dev)
    y = torch.empty(sh["y"], dtype=dt, device=dev)
    gx2 = torch.empty(sh["x"], dtype=dt, device=dev)
    wsb = max(d.disco_fused_conv_bwd_input_workspace_bytes(psi.c, B, C),
              d.disco_fused_conv_workspace_bytes(psi.c, B, C, Co))
    wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)  # shared: the calls run in sequence
    stream = torch.cuda.current_stream(dev)
    alg = algorithmic(w, psi.c)

    calls = [
        ("fwd", lambda: d.disco_fwd(psi.c, x, X, B, C, stream)),
        ("bwd", lambda: d.disco_bwd(psi.c, G, gx, B, C, stream)),
        ("fused", lambda: d.disco_fused_conv(psi.c, x, Wt, y, B, C, Co, wsp, stream)),
        ("fused_bwd", lambda: d.disco_fused_conv_bwd_input(psi.c, dy, Wt, gx2, B, C, Co, wsp, stream)),
    ]
    launches_per_step = 6  # fwd, bwd, fused (contraction + einsum), fused bwd (dX gemm + transpose)

    def step(ev=None):
        for i, (_, fn) in enumerate(calls):
            if ev is not None:
                ev[i][0].record(stream)
            fn()
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if d.disco_device_status() != 0:
        raise RuntimeError("a bounded wait timed out during warm-up")

    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in calls] for _ in range(args.steps)]
    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0e.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t1e.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    total_ms = t0e.elapsed_time(t1e)
    per = {name: [evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(args.steps)]
           for i, (name, _) in enumerate(calls)}
    contr_ms = sum(per["fwd"]) + sum(per["bwd"])
    total_ms, contr_ms = _max_over_ranks([total_ms, contr_ms], dev)
    if d.disco_device_status() != 0:
        raise RuntimeError("a bounded wait timed out during the timed region")

    # the weight gradient (a scope extension, not part of the step): timed alone
    dw_ms = None
    nwb = d.disco_fused_conv_bwd_weight_workspace_bytes(psi.c, B, C, Co) if Co is not None else 0
    if nwb > 0:
        wsw = torch.empty(nwb, dtype=torch.uint8, device=dev)
        dW = torch.empty(sh["W"], dtype=dt, device=dev)
        for _ in range(2):
            d.disco_fused_conv_bwd_weight(psi.c, x, dy, dW, B, C, Co, wsw, stream)
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        for _ in range(5):
            d.disco_fused_conv_bwd_weight(psi.c, x, dy, dW, B, C, Co, wsw, stream)
        q1.record(stream)
        torch.cuda.synchronize()
        dw_ms = q0.elapsed_time(q1) / 5
        del wsw, dW

    # end to end through the C ABI with host buffers: the host-buffer entry
    # points take pinned inputs and outputs, copy each 128-channel block in,
    # contract it and copy it out, with consecutive blocks overlapped; the
    # forward and the transpose run on two streams, so one's copies also
    # overlap the other's kernels.  Every copy is inside the timed region.
    e2e = None
    if rank == 0 or ws > 1:
        xh = x.cpu().pin_memory()
        Gh = G.cpu().pin_memory()
        Xh = torch.empty(sh["X"], dtype=dt).pin_memory()
        gxh = torch.empty(sh["x"], dtype=dt).pin_memory()
        code = d.DISCO_BF16 if dt == torch.bfloat16 else d.DISCO_F32
        wf = torch.empty(d.disco_host_workspace_bytes(psi.c, B, C, True, code), dtype=torch.uint8, device=dev)
        wb = torch.empty(d.disco_host_workspace_bytes(psi.c, B, C, False, code), dtype=torch.uint8, device=dev)
        s_f, s_b = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_step():
            d.disco_fwd_host(psi.c, xh, Xh, B, C, wf, s_f)
            d.disco_bwd_host(psi.c, Gh, gxh, B, C, wb, s_b)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        ne = max(1, min(args.steps, 5))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        s_f.wait_event(a0)
        s_b.wait_event(a0)
        for _ in range(ne):
            e2e_step()
        stream.wait_stream(s_f)
        stream.wait_stream(s_b)
        a1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a0.elapsed_time(a1) / ne
        e2e_ms = _max_over_ranks([e2e_ms], dev)[0]
        # the host link's own ceiling for these bytes: the same pinned copies
        # alone, both directions at once (no kernels)
        hin = torch.empty(Gh.shape, dtype=dt, pin_memory=True)
        hout = torch.empty(Xh.shape, dtype=dt, pin_memory=True)
        din = torch.empty(hin.shape, dtype=dt, device=dev)
        dout = torch.empty(hout.shape, dtype=dt, device=dev)
        hin2 = torch.empty(xh.shape, dtype=dt, pin_memory=True)
        hout2 = torch.empty(gxh.shape, dtype=dt, pin_memory=True)
        din2 = torch.empty(hin2.shape, dtype=dt, device=dev)
        dout2 = torch.empty(hout2.shape, dtype=dt, device=dev)

        def copies():
            with torch.cuda.stream(s_f):
                din.copy_(hin, non_blocking=True)
                din2.copy_(hin2, non_blocking=True)
            with torch.cuda.stream(s_b):
                hout.copy_(dout, non_blocking=True)
                hout2.copy_(dout2, non_blocking=True)

        copies()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        s_f.wait_event(c0)
        s_b.wait_event(c0)
        for _ in range(3):
            copies()
        stream.wait_stream(s_f)
        stream.wait_stream(s_b)
        c1.record(stream)
        torch.cuda.synchronize()
        copy_ms = c0.elapsed_time(c1) / 3
        del hin, hout, din, dout, hin2, hout2, din2, dout2
        e2e = {"value": round(ws * (alg["fwd_bytes"] + alg["bwd_bytes"]) / (e2e_ms * 1e6), 2),
               "unit": "GB/s",
               "h2d_bytes_per_step": x.numel() * x.element_size() + G.numel() * G.element_size(),
               "d2h_bytes_per_step": X.numel() * X.element_size() + gx.numel() * gx.element_size(),
               "ms_per_step": round(e2e_ms, 3),
               "copies_alone_ms_per_step": round(copy_ms, 3)}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    peaks, peak_src = _peaks()
    value = ws * (alg["fwd_bytes"] + alg["bwd_bytes"]) * args.steps / (contr_ms * 1e6)
    med = {k: statistics.median(v) for k, v in per.items()}
    share = {k: sum(v) for k, v in per.items()}
    clocks = clk.summary()
    # Dominant kernel: the transpose (bwd_tc_kernel) or forward (fwd_tc_kernel)
    # contraction, each launched twice per step (disco_bwd / disco_fwd alone
    # and inside the fused calls); the disco_bwd and disco_fwd calls are one
    # launch each, so their events time the kernel alone.  Bound: HBM, with
    # the algorithmic bytes of one launch (input + output + psi).
    dom = "bwd" if med["bwd"] >= med["fwd"] else "fwd"
    kname = {"bwd": "bwd_tc_kernel", "fwd": "fwd_tcp_kernel"}
    dom_kernel = kname[dom]
    dom_bytes = alg[dom + "_bytes"]
    achieved = dom_bytes / (med[dom] * 1e-3) / 1e9
    traffic = _traffic_from_profiles(dom_kernel, w.name)
    other = "fwd" if dom == "bwd" else "bwd"
    o_ach = alg[other + "_bytes"] / (med[other] * 1e-3) / 1e9

    def hbm_frac(nbytes, ms):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"gbs": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4), "ms": round(ms, 3)}

    # the fused calls against their own compulsory bytes, and the einsum's
    # tensor rate inside the fused call (its flops over the whole call's time:
    # a lower bound on the einsum's own rate) against the sustained bf16 peak
    tc_peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    # useful flops of the contractions (CSR non-zeros only) against what the
    # FP32 CUDA cores could do at most: SMs x 128 FP32 lanes x 2 flop x clock.
    # Above 1 means beyond the bound of a CUDA-core gather (the tensor-core
    # Toeplitz tiles run 5-10x the useful flops).
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    fp32_peak = sms * 128 * 2 * sm_mhz * 1e6 / 1e12
    contraction_flops = {"useful_flops_per_call": alg["csr_flops"],
                         "fp32_alu_peak_tflops": round(fp32_peak, 1),
                         "fp32_alu_peak_derivation": f"{sms} SMs x 128 FP32 lanes x 2 flop x {sm_mhz:.0f} MHz"}
    for nm in ("fwd", "bwd"):
        tf = alg["csr_flops"] / (med[nm] * 1e-3) / 1e12
        contraction_flops[nm + "_tflops"] = round(tf, 1)
        contraction_flops[nm + "_frac_of_fp32_alu"] = round(tf / fp32_peak, 3)
    fused_calls = None
    if "fused_bytes" in alg:
        ein_tf = alg["einsum_flops"] / (med["fused"] * 1e-3) / 1e12
        # the fused call is the forward kernel (X into the workspace) followed by
        # the einsum GEMM, so the GEMM's own time is the call's minus the forward's
        ein_ms = med["fused"] - med["fwd"]
        fused_calls = {
            "einsum_gemm": {"ms_by_subtraction": round(ein_ms, 3),
                            "tflops": round(alg["einsum_flops"] / (ein_ms * 1e-3) / 1e12, 1) if ein_ms > 0 else None,
                            "frac_of_sustained_peak": round(alg["einsum_flops"] / (ein_ms * 1e-3) / 1e12 / tc_peak, 4)
                            if ein_ms > 0 else None},
            "fused_conv": hbm_frac(alg["fused_bytes"], med["fused"]),
            "fused_conv_bwd_input": hbm_frac(alg["fused_bwd_bytes"], med["fused_bwd"]),
            "einsum": {"flops_per_call": alg["einsum_flops"], "tflops_over_fused_call": round(ein_tf, 1),
                       "peak_tflops": tc_peak, "frac_of_sustained_peak": round(ein_tf / tc_peak, 4),
                       "peak_source": f"{peak_src} (cuBLAS bf16, sustained)"},
        }
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) inputs, W ~ N(0, 1/(Cin*K)))",
        "config": {"workload": w.name, "B": w.B, "Cin": w.C, "Cout": w.Cout,
                   "grid_in": list(w.grid_in), "grid_out": list(w.grid_out), "K": w.K,
                   "basis": "anisotropic 3 radial hats x {1, cos, sin}", "cutoff_rad": w.cutoff,
                   "step": "disco_fwd + disco_bwd + disco_fused_conv + disco_fused_conv_bwd_input",
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{ws}"},
        "hbm_frac_of_measured_peak": round(value / ws / peaks["hbm_gbs"], 4),
        "fused_conv_ms_per_call": round(med["fused"], 3),
        "fused_conv_bwd_input_ms_per_call": round(med["fused_bwd"], 3),
        "fused_conv_bwd_weight_ms_per_call": round(dw_ms, 3) if dw_ms is not None else None,
        "kernel_ms": {k: round(v, 3) for k, v in med.items()},
        "roofline": {"bound": "hbm", "kernel": dom_kernel, "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "ms_per_launch": round(med[dom], 3),
                     "peak_source": f"{peak_src} (copy bandwidth)"},
        "roofline_other_contraction": {"bound": "hbm", "kernel": kname[other], "achieved": round(o_ach, 1),
                                       "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": round(o_ach / peaks["hbm_gbs"], 4),
                                       "algorithmic_bytes_per_launch": alg[other + "_bytes"],
                                       "ms_per_launch": round(med[other], 3)},
        "fused_calls": fused_calls,
        "contraction_flops": contraction_flops,
        "hbm_peak_gbs": peaks["hbm_gbs"], "hbm_peak_source": peak_src,
        "clocks": clocks, "gpu_launches": launches_per_step * args.steps, "e2e": e2e,
    }
    if not args.no_cpu_baseline and ws == 1:
        out["cpu_baseline"] = cpu_baseline(w, args.cpu_budget_s)
    print(json.dumps(out), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _traffic_from_profiles(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    record profiles/traffic.json, or None when there is none for this
    workload or the kernel's source changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("workload") != workload:
            return None
        e = t["kernels"][kernel]
        with open(os.path.join(ROOT, e["source"]), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != e["sha1"]:
                return None
        return int(e["dram_read"]) + int(e["dram_write"])
    except Exception:
        return None


def _psi_rows(ref, m: int):
    """The oracle's psi restricted to every m-th output row (all k): a sample
    of the output rows, spread over all latitudes (the polar rows cost more).
    Only the CSR arrays, which the oracle's contractions read, are sliced;
    the oracle computes on them as it stands."""
    import dataclasses
    import numpy as np
    if m <= 1:
        return ref, 1.0
    rows = np.arange(0, ref.Hout, m)
    starts = np.array([ref.csr_row_ptr[k * ref.Hout + h] for k in range(ref.K) for h in rows], np.int64)
    ends = np.array([ref.csr_row_ptr[k * ref.Hout + h + 1] for k in range(ref.K) for h in rows], np.int64)
    ptr = np.concatenate([[0], np.cumsum(ends - starts)]).astype(np.int64)
    sel = np.concatenate([np.arange(a, b) for a, b in zip(starts, ends)]) if len(starts) else np.zeros(0, np.int64)
    sub = dataclasses.replace(ref, grid_out=(len(rows), ref.grid_out[1], ref.grid_out[2]), csr_row_ptr=ptr,
                              csr_col=np.ascontiguousarray(ref.csr_col[sel]),
                              csr_val=np.ascontiguousarray(ref.csr_val[sel]))
    return sub, len(rows) / ref.Hout


def cpu_baseline(w, budget_s: float, ref=None, row_stride: int = 1):
    """The fp64 oracle, as it stands, on a bounded sample of the workload:
    the forward and transpose contractions over the first n channels (n =
    host cores, one OpenMP thread each) and every row_stride-th output row,
    scaled to the same GB/s metric.  `ref` is the oracle's psi for the
    workload (built here when None; the build is init work, outside the
    timed sample)."""
    import numpy as np
    import torch
    import oracle

    cores = os.cpu_count() or 1
    if ref is None:
        ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    sub, rfrac = _psi_rows(ref, row_stride)
    g = torch.Generator().manual_seed(w.seed)
    Hin, Win = w.grid_in[:2]
    Hout, Wout = w.grid_out[:2]
    n = max(1, min(w.C, cores))
    x = torch.randn((1, n, Hin, Win), generator=g).to(torch.bfloat16).double().numpy()
    G = torch.randn((1, n, w.K, sub.Hout, Wout), generator=g).to(torch.bfloat16).double().numpy()
    t0 = time.perf_counter()
    oracle.fwd(sub, x)
    t1 = time.perf_counter()
    oracle.bwd(sub, G)
    t2 = time.perf_counter()
    esz = 2
    frac = n / w.C
    # fwd + bwd, input + output, for the sampled channels; the sampled rows
    # carry that fraction of the work
    byts = (x.size + n * w.K * Hout * Wout) * esz * 2 * rfrac
    del np
    rows = "all output rows" if row_stride <= 1 else f"every {row_stride}th output row ({rfrac:.3f} of them)"
    return {"value": round(byts / (t2 - t0) / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"fp64 oracle fwd + bwd over {n} of {w.C} channels ({frac:.3f} of the "
                      f"workload) and {rows}, {t1 - t0:.2f} s + {t2 - t1:.2f} s"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from sparse_spherical_convolution_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    ref = oracle.build_psi(w.grid_in, w.grid_out, w.kind, w.nrad, w.cutoff)
    # every step samples every m-th output row, m chosen from one full-row
    # step so that the warm-up and timed steps together take about
    # REF_TOTAL_S (or cpu_budget_s per step, whichever is less)
    t0 = time.perf_counter()
    cpu_baseline(w, args.cpu_budget_s, ref)
    full_s = time.perf_counter() - t0
    per_step = min(args.cpu_budget_s, REF_TOTAL_S / max(1, args.steps + args.warmup))
    m = max(1, min(w.grid_out[0], math.ceil(full_s / per_step)))
    vals = []
    cb = None
    for _ in range(args.warmup):
        cpu_baseline(w, args.cpu_budget_s, ref, m)
    for _ in range(args.steps):
        cb = cpu_baseline(w, args.cpu_budget_s, ref, m)
        vals.append(cb["value"])
    v = round(statistics.median(vals), 4)
    out = {"metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": w.name, "step": "fp64 CPU oracle fwd + bwd on a channel sample"},
           "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cb["cores"], "kind": "oracle",
                            "sample": cb["sample"]},
           "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
