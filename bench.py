"""Benchmark: mHC layer forward + backward on GB300, tokens/s and HBM roofline.

One step = one pass of the whole hot path over one seeded synthetic batch:
  mhc_layer_fwd (proj_rms_compute_h -> h_aggregate -> h_post_bda)
  mhc_layer_bwd (post_bda, aggregate/compute_h and residual-gradient passes)
  rmsnorm_fwd + rmsnorm_bwd on a standalone [T, C] bf16 tensor
Default workload: T=16384 tokens, n=4 streams, C=4096 (7B-scale), seed 3.

`python bench.py [--gpus N --steps K --warmup W]` prints one JSON line.
Under torchrun each rank runs its own batch (weak scaling; the layer needs
no exchange between ranks).  `--impl reference` times the fp64 CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mhc_inputs as mi  # noqa: E402

ITERS, EPS_SK, EPS_RMS, EPS_NORM = mi.ITERS, mi.EPS_SK, mi.EPS_RMS, mi.EPS_NORM
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "mHC layer fwd+bwd tokens/sec on 1 GB300; achieved HBM GB/s vs ~8 TB/s peak"


# ---------------------------------------------------------------------------
# byte model
# ---------------------------------------------------------------------------

def model_bytes(T, n, C):
    """Bytes one step must move through HBM (U = one bf16 [T, C] tensor).

    This is the byte model of the mHC layer as three forward and three
    backward streaming passes: it is the yardstick the throughput target is
    quoted in (70% of 8 TB/s on these bytes).
    layer fwd (4n+2)U: projection reads x (nU); aggregate reads x, writes y
    ((n+1)U); post_bda reads x and f, writes out ((2n+1)U).
    layer bwd (6n+4)U: post_bda pass reads dout, x, f, writes df ((2n+2)U);
    aggregate/compute_h pass reads x, dy ((n+1)U); residual-gradient pass
    reads x, dy, dout, writes dx ((3n+1)U).
    RMSNorm: fwd 2U, bwd 3U.  Small terms (W, H, u, r, dW) are left out.
    """
    U = T * C * 2
    return {"layer_fwd": (4 * n + 2) * U, "layer_bwd": (6 * n + 4) * U, "rmsnorm": 5 * U}


def moved_bytes(T, n, C):
    """Bytes this implementation's passes move: as model_bytes, except that
    the backward reads x once for the post_bda and aggregate reductions
    together ((2n+3)U token pass), so the layer backward is (5n+4)U."""
    U = T * C * 2
    return {"layer_fwd": (4 * n + 2) * U, "layer_bwd": (5 * n + 4) * U, "rmsnorm": 5 * U}


def kernel_bytes(name, T, n, C):
    """Algorithmic bytes of one launch of a library kernel in the layer step."""
    U = T * C * 2
    O = n * n + 2 * n
    K = n * C
    small = T * O * 4
    table = {
        "k_w_split": K * O * 4 + (3 * O + 15) // 16 * 16 * K * 2,
        "k_proj_tc": n * U + K * O * 4,
        "k_compute_h_fwd": small,
        "k_agg_fwd": (n + 1) * U,
        "k_post_fwd": (2 * n + 1) * U,
        "k_bwd_tok": (2 * n + 3) * U,
        "k_bwd_tc": (3 * n + 1) * U,
        "k_bwd_finalize": small,
        "k_post_bwd_tok": (2 * n + 2) * U,
        "k_agg_bwd": (n + 1) * U,
        "k_compute_h_bwd": 3 * small,
        "k_rms_fwd": 2 * U,
        "k_rms_bwd": 3 * U,
    }
    return table.get(name)


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def csrc_hash():
    d = os.path.join(ROOT, "layers_proj_rms_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
    except Exception:
        return None
    if d.get("csrc_hash") != csrc_hash():
        return None
    e = d.get("kernels", {}).get(workload, {}).get(kernel)
    return None if e is None else float(e)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class Clocks:
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        self.out = None
        try:
            self.out = open(os.path.join("/tmp", f"mhc_clocks_{os.getpid()}.csv"), "w")
            self.path = self.out.name
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    sm.append(float(f[0]))
                    mx.append(float(f[1]))
                except ValueError:
                    continue
                for nm, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# multi-rank helpers (one process per GPU; tokens sharded, no data-path
# collective: only the timings are reduced)
# ---------------------------------------------------------------------------

def max_over_ranks(v, world, device):
    """The largest value of v over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed, rank):
    """Each rank draws its own batch of the workload (weak scaling)."""
    return seed + 1000 * rank


def job_tokens_per_s(T, world, ms):
    """Whole-job throughput: every rank's T tokens over the slowest rank's time."""
    return T * world / (ms / 1e3)


# ---------------------------------------------------------------------------
# every op of the C ABI on its own, at the workload's sizes
# ---------------------------------------------------------------------------

def bench_ops(M, d, o, T, n, C, dev, reps=5):
    """Per op: `ms` the device time per call (reps calls replayed as one
    CUDA graph), `ms_eager` the event-timed average of reps back-to-back
    calls through the binding (includes the host's per-call overhead, which
    exceeds the kernels of the small ops), its algorithmic HBM bytes (U = one
    bf16 [T, C] tensor) and the GB/s `ms` gives.  Inputs reuse the step's
    tensors; all are larger than L2 except the Sinkhorn batch (32768
    matrices, latency-bound)."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    e = lambda *sh, dt=f32: torch.empty(*sh, dtype=dt, device=dev)  # noqa: E731
    U = T * C * 2
    O = n * n + 2 * n
    K = n * C
    x, f, bias, W = d["x"], d["f"], d["bias"], d["W"]
    alpha, b, dout, dy = d["alpha"], d["b"], d["dout"], d["dy"]
    Hp, Hq, Hr = o["H_pre"], o["H_post"], o["H_res"]
    g = torch.ones(C, device=dev)
    Hs = torch.full((n,), 0.5, device=dev)
    y, dxb, dfb = e(T, C, dt=bf), e(T, n, C, dt=bf), e(T, C, dt=bf)
    outb = e(T, n, C, dt=bf)
    dHp, dHq, dHr = (torch.full((T, n), 0.1, device=dev), torch.full((T, n), 0.1, device=dev),
                     torch.full((T, n, n), 0.1, device=dev))
    y2, dx2 = e(T, C, dt=bf), e(T, C, dt=bf)
    rstd, dg = e(T), e(C)
    u, sq, r = e(T, O), e(T), e(T)
    du, coef, dal, dbb, dW = e(T, O), e(T), e(3), e(O), e(K, O)
    Cs = C // 2
    xs = x[:, :, :Cs].contiguous()
    Ws = torch.cat([W[i * C:i * C + Cs] for i in range(n)]).contiguous()
    dxs, dWs = e(T, n, Cs, dt=bf), e(n * Cs, O)
    Mm = 32768
    lg = torch.randn(Mm, n, n, device=dev)
    dP = torch.randn(Mm, n, n, device=dev)
    P, dl = e(Mm, n, n), e(Mm, n, n)
    W_ = lambda op, c=C: M.workspace(op, T, n, c, dev)  # noqa: E731
    wsf, wsb = W_(M.OP_PROJ_RMS_COMPUTE_H_FWD), W_(M.OP_PROJ_RMS_COMPUTE_H_BWD)
    wspb, wsas = W_(M.OP_H_POST_BDA_BWD), W_(M.OP_H_AGGREGATE_STATIC_BWD)
    wsr, wsan = M.workspace(M.OP_RMSNORM_RESIDUAL_BWD, T, 0, C, dev), W_(M.OP_H_AGGREGATE_RMSNORM_BWD)
    wspf, wspb2 = W_(M.OP_PROJ_RMS_PARTIAL_FWD, Cs), W_(M.OP_PROJ_RMS_PARTIAL_BWD, Cs)
    wsch = W_(M.OP_COMPUTE_H_BWD, 8)
    wspp = W_(M.OP_H_POST_BDA_COMPUTE_H_FWD)
    Hp2, Hq2, Hr2, u2, r2 = e(T, n), e(T, n), e(T, n, n), e(T, O), e(T)
    it, es, er = ITERS, EPS_SK, EPS_RMS
    ops = {
        "mhc_sinkhorn_fwd": (lambda: M.mhc_sinkhorn_fwd(lg, P, it, es), Mm * n * n * 8),
        "mhc_sinkhorn_bwd": (lambda: M.mhc_sinkhorn_bwd(dP, lg, dl, it, es), Mm * n * n * 12),
        "mhc_proj_rms_compute_h_fwd": (lambda: M.mhc_proj_rms_compute_h_fwd(
            x, W, alpha, b, it, es, er, Hp, Hq, Hr, u, r, wsf), n * U),
        "mhc_proj_rms_compute_h_bwd": (lambda: M.mhc_proj_rms_compute_h_bwd(
            dHp, dHq, dHr, x, W, alpha, b, u, r, it, es, er, dxb, dW, dal, dbb, wsb), 2 * n * U),
        "mhc_h_aggregate_fwd": (lambda: M.mhc_h_aggregate_fwd(x, Hp, y), (n + 1) * U),
        "mhc_h_aggregate_bwd": (lambda: M.mhc_h_aggregate_bwd(dy, x, Hp, dxb, dHp),
                                (2 * n + 1) * U),
        "mhc_h_post_bda_fwd": (lambda: M.mhc_h_post_bda_fwd(x, f, bias, Hr, Hq, outb),
                               (2 * n + 1) * U),
        "mhc_h_post_bda_bwd": (lambda: M.mhc_h_post_bda_bwd(dout, x, f, bias, Hr, Hq, dxb, dfb,
                                                            dg, dHr, dHq, wspb), (3 * n + 2) * U),
        # post-mix of this layer + the next layer's proj_rms pass on its output
        # (the separate ops move (2n+1)U + nU)
        "mhc_h_post_bda_compute_h_fwd": (lambda: M.mhc_h_post_bda_compute_h_fwd(
            x, f, bias, Hr, Hq, W, alpha, b, it, es, er, outb, Hp2, Hq2, Hr2, u2, r2, wspp),
            (2 * n + 1) * U),
        "rmsnorm_fwd": (lambda: M.rmsnorm_fwd(y, dfb, rstd, EPS_NORM), 2 * U),
        "rmsnorm_bwd": (lambda: M.rmsnorm_bwd(dy, y, rstd, dfb, EPS_NORM), 3 * U),
        "mhc_h_aggregate_static_fwd": (lambda: M.mhc_h_aggregate_static_fwd(x, Hs, y),
                                       (n + 1) * U),
        "mhc_h_aggregate_static_bwd": (lambda: M.mhc_h_aggregate_static_bwd(
            dy, x, Hs, dxb, dHp[0], wsas), (2 * n + 1) * U),
        "rmsnorm_residual_fwd": (lambda: M.rmsnorm_residual_fwd(
            y, f, g, dfb, y2, rstd, EPS_NORM), 4 * U),
        "rmsnorm_residual_bwd": (lambda: M.rmsnorm_residual_bwd(
            dy, None, y, f, g, rstd, dx2, dg, EPS_NORM, wsr), 4 * U),
        "mhc_h_aggregate_rmsnorm_fwd": (lambda: M.mhc_h_aggregate_rmsnorm_fwd(
            x, Hp, g, y, dfb, rstd, EPS_NORM), (n + 2) * U),
        "mhc_h_aggregate_rmsnorm_bwd": (lambda: M.mhc_h_aggregate_rmsnorm_bwd(
            dy, None, x, Hp, g, rstd, dxb, dHp, dg, EPS_NORM, wsan), (2 * n + 1) * U),
        "mhc_proj_rms_partial_fwd": (lambda: M.mhc_proj_rms_partial_fwd(xs, Ws, u, sq, wspf),
                                     n * U // 2),
        "mhc_compute_h_fwd": (lambda: M.mhc_compute_h_fwd(u, sq, K, alpha, b, it, es, er, Hp, Hq,
                                                          Hr, r), T * (O + 1) * 4),
        "mhc_compute_h_bwd": (lambda: M.mhc_compute_h_bwd(dHp, dHq, dHr, u, sq, K, alpha, b, it,
                                                          es, er, du, coef, dal, dbb, wsch),
                              T * (3 * O + 1) * 4),
        "mhc_proj_rms_partial_bwd": (lambda: M.mhc_proj_rms_partial_bwd(xs, Ws, du, coef, dxs,
                                                                        dWs, wspb2), n * U),
    }
    stream = torch.cuda.current_stream()

    def graph_ms(fn):
        """Device time per call: `reps` calls captured into one CUDA graph,
        replayed (no host call overhead between the launches)."""
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()
        stream.wait_stream(side)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            for _ in range(reps):
                fn()
        cg.replay()
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            cg.replay()
        z.record(stream)
        torch.cuda.synchronize()
        del cg
        return a.elapsed_time(z) / (3 * reps)

    res = {}
    for name, (fn, nbytes) in ops.items():
        fn(); fn()
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        z.record(stream)
        torch.cuda.synchronize()
        eager = a.elapsed_time(z) / reps
        try:
            ms = graph_ms(fn)
        except Exception:  # noqa: BLE001  (capture refused: keep the eager number)
            ms = None
        dev_ms = ms if ms is not None else eager
        res[name] = {"ms": round(dev_ms, 4), "ms_eager": round(eager, 4), "alg_bytes": int(nbytes),
                     "gbs": round(nbytes / (dev_ms / 1e3) / 1e9, 1)}
    return res


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def collect_kernel_times(M):
    """The library profiler's per-kernel totals since it was last collected:
    {name: (launches, total ms)}."""
    import ctypes

    class KT(ctypes.Structure):
        _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                    ("total_ms", ctypes.c_double)]

    buf = (KT * 64)()
    M.lib.mhc_profiler_collect.argtypes = [ctypes.c_void_p, ctypes.c_int]
    nk = M.lib.mhc_profiler_collect(ctypes.cast(buf, ctypes.c_void_p), 64)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(nk)}


def top_kernel_roofline(kernels, T, n, C, peak, workload):
    """Roofline of the kernel with the largest total time: its algorithmic
    bytes per launch over its average event-timed launch duration."""
    if not kernels:
        return None
    name, (nl, tot) = max(kernels.items(), key=lambda kv: kv[1][1])
    avg_ms = tot / nl
    kb = kernel_bytes(name, T, n, C)
    if kb is None:
        return None
    ach = kb / (avg_ms / 1e3) / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
            "unit": "GB/s", "frac": round(ach / peak, 4),
            "traffic": ncu_traffic(name, workload),
            "algorithmic_bytes_per_launch": int(kb), "avg_launch_ms": round(avg_ms, 4)}


def run_wide(M, dev, steps, warmup, peak, barrier, world):
    """The wide-stream workload (T=8192, n=8, C=7168, seed 4): the layer
    forward + backward, timed as the main step is (events on the launching
    stream, inputs larger than L2), then once more under the library's event
    profiler for the per-kernel times and the dominant kernel's roofline."""
    import torch
    wl = "wide_T8192_n8_C7168"
    T, n, C, w_std, seed = mi.LAYER_WORKLOADS[wl]
    O = n * n + 2 * n
    inp = mi.layer_inputs(T, n, C, seed, w_std=w_std)
    bf = torch.bfloat16
    d = {k: (torch.from_numpy(v.view(np.int16)).to(dev).view(bf) if v.dtype == np.uint16
             else torch.from_numpy(v).to(dev)) for k, v in inp.items()}
    del inp
    e = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
    o = {"H_pre": e(T, n), "H_post": e(T, n), "H_res": e(T, n, n), "u": e(T, O), "r": e(T),
         "y": e(T, C, dt=bf), "out": e(T, n, C, dt=bf), "dx": e(T, n, C, dt=bf),
         "df": e(T, C, dt=bf), "dW": e(n * C, O), "dalpha": e(3), "db": e(O), "dbias": e(C)}
    wsf = M.workspace(M.OP_LAYER_FWD, T, n, C, dev)
    wsb = M.workspace(M.OP_LAYER_BWD, T, n, C, dev)

    def step():
        M.mhc_layer_fwd(d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"], ITERS, EPS_SK,
                        EPS_RMS, o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], o["y"],
                        o["out"], wsf)
        M.mhc_layer_bwd(d["dout"], d["dy"], d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"],
                        o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], ITERS, EPS_SK,
                        EPS_RMS, o["dx"], o["df"], o["dW"], o["dalpha"], o["db"], o["dbias"], wsb)

    for _ in range(warmup):
        step()
    barrier()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / steps, world, dev)
    collect_kernel_times(M)  # drop anything recorded before
    M.lib.mhc_profiler_enable(1)
    for _ in range(steps):
        step()
    barrier()
    M.lib.mhc_profiler_enable(0)
    kernels = collect_kernel_times(M)
    assert M.mhc_device_error() == 0, "a kernel reported a device fault"
    mb = model_bytes(T, n, C)
    lb = mb["layer_fwd"] + mb["layer_bwd"]
    gbs = lb / (ms / 1e3) / 1e9
    return {"workload": wl, "step": "mhc_layer_fwd + mhc_layer_bwd", "ms_per_step": round(ms, 4),
            "tokens_per_s": round(job_tokens_per_s(T, world, ms)),
            "model_bytes_per_step": int(lb), "achieved_gbs": round(gbs, 1),
            "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "frac_of_measured": round(gbs / peak, 4),
            "roofline": top_kernel_roofline(kernels, T, n, C, peak, wl),
            "kernels_ms": {k: round(v[1] / v[0], 4) for k, v in
                           sorted(kernels.items(), key=lambda kv: -kv[1][1])}}

def run_ours(args, rank, world):
    import torch

    import layers_proj_rms_gb300 as M

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    T, n, C, w_std, seed = mi.LAYER_WORKLOADS[args.workload]
    O = n * n + 2 * n
    inp = mi.layer_inputs(T, n, C, rank_seed(seed, rank), w_std=w_std, rmsnorm=True)

    def h2d_src(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.pin_memory()

    host_in = {k: h2d_src(v) for k, v in inp.items()}
    bf = torch.bfloat16

    def dev_of(k):
        h = host_in[k]
        t = h.to(dev)
        return t.view(bf) if h.dtype == torch.int16 else t

    d = {k: dev_of(k) for k in host_in}
    e = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
    o = {"H_pre": e(T, n), "H_post": e(T, n), "H_res": e(T, n, n), "u": e(T, O), "r": e(T),
         "y": e(T, C, dt=bf), "out": e(T, n, C, dt=bf), "dx": e(T, n, C, dt=bf),
         "df": e(T, C, dt=bf), "dW": e(n * C, O), "dalpha": e(3), "db": e(O), "dbias": e(C),
         "yn": e(T, C, dt=bf), "rstd": e(T), "dxn": e(T, C, dt=bf)}
    wsf = M.workspace(M.OP_LAYER_FWD, T, n, C, dev)
    wsb = M.workspace(M.OP_LAYER_BWD, T, n, C, dev)

    def step():
        step_on(d)

    def step_on(d):
        M.mhc_layer_fwd(d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"], ITERS, EPS_SK,
                        EPS_RMS, o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], o["y"],
                        o["out"], wsf)
        M.mhc_layer_bwd(d["dout"], d["dy"], d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"],
                        o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], ITERS, EPS_SK,
                        EPS_RMS, o["dx"], o["df"], o["dW"], o["dalpha"], o["db"], o["dbias"], wsb)
        M.rmsnorm_fwd(d["x_norm"], o["yn"], o["rstd"], EPS_NORM)
        M.rmsnorm_bwd(d["dy_norm"], d["x_norm"], o["rstd"], o["dxn"], EPS_NORM)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    clocks = Clocks(dev.index if dev.index is not None else 0)
    # keep the GPU busy ~1 s before the timed region so the clock samples
    # taken around it are under load
    t_end = time.time() + 1.0
    while time.time() < t_end:
        step()
        torch.cuda.synchronize()
    barrier()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # The timed region: K steps as a user runs them.  Every library kernel is
    # launched with programmatic stream serialization, so a kernel's launch
    # overlaps the end of the previous one.
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    # The same K steps again with the library's event profiler on: an event
    # pair around every launch gives each kernel's duration (these events sit
    # between the launches and serialise them, so this step time is longer).
    M.lib.mhc_profiler_enable(1)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    M.lib.mhc_profiler_enable(0)
    clk = clocks.stop()
    ms_prof = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    assert M.mhc_device_error() == 0, "a kernel reported a device fault"

    kernels = collect_kernel_times(M)
    launches = int(sum(v[0] for v in kernels.values()))

    ms = max_over_ranks(ms, world, dev)

    # ---- the layer alone (fwd + bwd, no RMSNorm), for the layer byte model ----
    def layer_step():
        M.mhc_layer_fwd(d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"], ITERS, EPS_SK,
                        EPS_RMS, o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], o["y"],
                        o["out"], wsf)
        M.mhc_layer_bwd(d["dout"], d["dy"], d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"],
                        o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], ITERS, EPS_SK,
                        EPS_RMS, o["dx"], o["df"], o["dW"], o["dalpha"], o["db"], o["dbias"], wsb)

    for _ in range(3):
        layer_step()
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        layer_step()
    ev1.record(stream)
    barrier()
    lms = ev0.elapsed_time(ev1) / args.steps
    lms = max_over_ranks(lms, world, dev)

    # ---- per-step times: the same steps with an event after each ----
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        step()
        evs[i + 1].record(stream)
    barrier()
    per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    per_step = {"median_ms": round(max_over_ranks(per[len(per) // 2], world, dev), 4),
                "min_ms": round(max_over_ranks(per[0], world, dev), 4),
                "max_ms": round(max_over_ranks(per[-1], world, dev), 4),
                "what": "the bench step timed one by one (an event after each), median over the "
                        "K steps"}

    # ---- the layer forward alone ----
    def fwd_step():
        M.mhc_layer_fwd(d["x"], d["W"], d["alpha"], d["b"], d["f"], d["bias"], ITERS, EPS_SK,
                        EPS_RMS, o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], o["y"],
                        o["out"], wsf)

    for _ in range(3):
        fwd_step()
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        fwd_step()
    ev1.record(stream)
    barrier()
    fms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)

    # ---- the same step captured once into a CUDA graph and replayed ----
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg):
            step()
        for _ in range(3):
            cg.replay()
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            cg.replay()
        ev1.record(stream)
        barrier()
        gms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
        graph = {"ms_per_step": round(gms, 4), "tokens_per_s": job_tokens_per_s(T, world, gms),
                 "what": "the bench step captured once into a CUDA graph, replayed (no launch gaps "
                         "between its kernels); same kernels and inputs"}
        del cg

    # ---- every op on its own ----
    ops = None if args.no_ops else bench_ops(M, d, o, T, n, C, dev)

    # ---- end to end: pinned host inputs -> device -> step -> host grads ----
    e2e = None
    if not args.no_e2e:
        out_host = {k: torch.empty(o[k].shape, dtype=o[k].dtype, pin_memory=True)
                    for k in ("dW", "dalpha", "db", "dbias")}
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in out_host.values())

        # Two sets of device inputs: while step i computes on one set, the
        # copies of step i+1's inputs (pinned host -> device, pieces of at
        # most 64 MiB on a copy stream) fill the other; a set is refilled
        # only after the step that used it has finished.
        nstreams = max(1, args.copy_streams)
        cstreams = [torch.cuda.Stream(device=dev) for _ in range(nstreams)]
        sets = [d, {k: torch.empty_like(v) for k, v in d.items()}]

        def pieces_of(dset):
            ps = []
            for k, h in host_in.items():
                dst = (dset[k].view(torch.int16) if dset[k].dtype == bf else dset[k]).reshape(-1)
                src = h.reshape(-1)
                step_el = max(1, (64 << 20) // src.element_size())
                for a0 in range(0, src.numel(), step_el):
                    ps.append((dst[a0:a0 + step_el], src[a0:a0 + step_el]))
            return ps

        set_pieces = [pieces_of(sets[0]), pieces_of(sets[1])]
        copied = [[torch.cuda.Event() for _ in range(nstreams)] for _ in range(2)]
        used = [torch.cuda.Event(), torch.cuda.Event()]
        for ev in used:
            ev.record(stream)

        def issue_copies(j):
            for i, cs in enumerate(cstreams):
                cs.wait_event(used[j])
                with torch.cuda.stream(cs):
                    for dst, src in set_pieces[j][i::nstreams]:
                        dst.copy_(src, non_blocking=True)
                copied[j][i].record(cs)

        state = {"i": 0}
        issue_copies(0)

        def e2e_step():
            j = state["i"] & 1
            issue_copies(j ^ 1)  # the next step's inputs, behind the step that last used them
            for ev in copied[j]:
                stream.wait_event(ev)
            step_on(sets[j])
            used[j].record(stream)
            for k, h in out_host.items():
                h.copy_(o[k], non_blocking=True)
            state["i"] += 1

        for _ in range(2):
            e2e_step()
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        # the copies issued for the step after the last are counted too
        for ev in copied[state["i"] & 1]:
            stream.wait_event(ev)
        ev1.record(stream)
        barrier()
        ems = ev0.elapsed_time(ev1) / args.steps
        ems = max_over_ranks(ems, world, dev)
        e2e = {"value": job_tokens_per_s(T, world, ems), "unit": "tokens/s", "ms_per_step": ems,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "copy_streams": nstreams,
               "api": "pinned host -> cudaMemcpyAsync (pieces of <= 64 MiB on a copy stream, "
                      "step i+1's inputs copied while step i computes; two input sets) -> "
                      "mhc_layer_fwd/bwd + rmsnorm_fwd/bwd -> host dW, dalpha, db, dbias"}

    # ---- the wide-stream workload (n = 8), its own step ----
    wide = None
    if not args.no_wide and args.workload != "wide_T8192_n8_C7168":
        pk, _ = measured_hbm_peak()
        wide = run_wide(M, dev, args.steps, args.warmup, pk, barrier, world)

    if rank != 0:
        return None
    mb = model_bytes(T, n, C)
    total_b = sum(mb.values())
    moved_b = sum(moved_bytes(T, n, C).values())
    peak, peak_kind = measured_hbm_peak()
    # dominant kernel
    roof = top_kernel_roofline(kernels, T, n, C, peak, args.workload)
    if roof:
        roof["peak_source"] = ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                               else "fallback 6.8 TB/s")
        roof["share_of_step"] = round(kernels[roof["kernel"]][1] / (ms_prof * args.steps), 4)
    res = {
        "metric": METRIC,
        "value": job_tokens_per_s(T, world, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "profiled": {"ms_per_step": round(ms_prof, 4),
                     "what": "the same steps with an event pair around every kernel launch "
                             "(source of 'kernels' and 'roofline'); the events serialise the "
                             "launches"},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 residual/grad tensors, random-init W)",
        "config": {"workload": args.workload, "T": T, "n": n, "C": C, "w_std": w_std,
                   "seed": seed, "iters": ITERS, "global_batch_tokens": T * world,
                   "step": "mhc_layer_fwd + mhc_layer_bwd + rmsnorm_fwd + rmsnorm_bwd",
                   "l2": "inputs larger than L2 (x alone is %d MB per step)" % (T * n * C * 2 >> 20),
                   "parallelism": f"replicas x{world} (tokens sharded, no collective)"},
        "hbm": {"model_bytes_per_step": int(total_b),
                "achieved_gbs": round(total_b / (ms / 1e3) / 1e9, 1),
                "frac_of_nominal_8tbs": round(total_b / (ms / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4),
                "frac_of_measured": round(total_b / (ms / 1e3) / 1e9 / peak, 4),
                "moved_bytes_per_step": int(moved_b),
                "moved_gbs": round(moved_b / (ms / 1e3) / 1e9, 1),
                "moved_frac_of_measured": round(moved_b / (ms / 1e3) / 1e9 / peak, 4)},
        "per_step": per_step,
        "roofline": roof,
        "kernels": {k: {"launches": v[0], "avg_ms": round(v[1] / v[0], 4),
                        "share": round(v[1] / (ms_prof * args.steps), 4)} for k, v in
                    sorted(kernels.items(), key=lambda kv: -kv[1][1])},
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
        "graph": graph,
        "ops": ops,
        # last, so that they stay in the tail of the line
        "layer_only": {"step": "mhc_layer_fwd + mhc_layer_bwd", "ms_per_step": round(lms, 4),
                       "tokens_per_s": round(job_tokens_per_s(T, world, lms)),
                       "model_bytes_per_step": int(mb["layer_fwd"] + mb["layer_bwd"]),
                       "achieved_gbs": round((mb["layer_fwd"] + mb["layer_bwd"]) / (lms / 1e3) / 1e9, 1),
                       "frac_of_nominal_8tbs": round((mb["layer_fwd"] + mb["layer_bwd"]) / (lms / 1e3)
                                                     / 1e9 / NOMINAL_HBM_GBS, 4)},
        "forward_only": {"step": "mhc_layer_fwd (the 7B-scale forward's shapes)",
                         "ms_per_step": round(fms, 4),
                         "tokens_per_s": round(job_tokens_per_s(T, world, fms)),
                         "model_bytes_per_step": int(mb["layer_fwd"]),
                         "achieved_gbs": round(mb["layer_fwd"] / (fms / 1e3) / 1e9, 1),
                         "frac_of_nominal_8tbs": round(mb["layer_fwd"] / (fms / 1e3) / 1e9
                                                       / NOMINAL_HBM_GBS, 4)},
        "wide": wide,
    }
    return res


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_step(orc, sub, n):
    f = orc.layer_fwd(sub, n, ITERS, EPS_SK, EPS_RMS)
    orc.layer_bwd(sub, f, n, ITERS, EPS_SK, EPS_RMS)
    _, rstd = orc.rmsnorm_fwd(sub["x_norm"], EPS_NORM)
    orc.rmsnorm_bwd(sub["dy_norm"], sub["x_norm"], EPS_NORM)


def sample_of(inp, tokens):
    sub = dict(inp)
    for k in ("x", "f", "dout", "dy", "x_norm", "dy_norm"):
        sub[k] = inp[k][:tokens]
    return sub


def cpu_baseline(args, tokens):
    import oracle as orc
    orc.build()
    T, n, C, w_std, seed = mi.LAYER_WORKLOADS[args.workload]
    inp = mi.layer_inputs(T, n, C, seed, w_std=w_std, rmsnorm=True)
    sub = sample_of(inp, tokens)
    # repeat the sample until about 10 s of CPU work (at most 20 passes)
    reps, t0 = 0, time.time()
    while True:
        oracle_step(orc, sub, n)
        reps += 1
        dt = time.time() - t0
        if dt >= 10.0 or reps >= 20:
            break
    return {"value": reps * tokens / dt, "unit": "tokens/s", "cores": orc.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"first {tokens} of the {T} tokens of the seeded batch, {reps} passes: full "
                      f"layer fwd+bwd (all outputs) and RMSNorm fwd+bwd on those rows, fp64 C oracle"}


def run_reference(args):
    """The oracle as the reference arm: each step one bounded sample."""
    import oracle as orc
    orc.build()
    T, n, C, w_std, seed = mi.LAYER_WORKLOADS[args.workload]
    tokens = args.ref_tokens
    inp = mi.layer_inputs(T, n, C, seed, w_std=w_std, rmsnorm=True)
    sub = sample_of(inp, tokens)
    for _ in range(args.warmup):
        oracle_step(orc, sub, n)
    t0 = time.time()
    for _ in range(args.steps):
        oracle_step(orc, sub, n)
    dt = (time.time() - t0) / args.steps
    v = tokens / dt
    sample = (f"first {tokens} of the {T} tokens of the seeded batch per step: full layer "
              f"fwd+bwd and RMSNorm fwd+bwd, fp64 C oracle")
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "T": T, "n": n, "C": C,
                                        "sample_tokens": tokens},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b_fwdbwd_T16384_n4_C4096",
                    choices=[k for k in mi.LAYER_WORKLOADS if "fwd_" not in k])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="streams the e2e host-to-device copies are spread over")
    ap.add_argument("--no-ops", action="store_true", help="skip the per-op timings")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--no-wide", action="store_true",
                    help="skip the wide-stream (n = 8) workload's step")
    ap.add_argument("--cpu-tokens", type=int, default=4096)
    ap.add_argument("--ref-tokens", type=int, default=1024)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            cb = cpu_baseline(args, args.cpu_tokens)
        else:
            cb = None
        # the line ends with the layer-only, forward-only and wide numbers
        tail = {k: res.pop(k) for k in ("layer_only", "forward_only", "wide")}
        res["cpu_baseline"] = cb
        res.update(tail)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
