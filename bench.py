"""Throughput of the selective-scan hot path on GB300.

One step = the whole path over one batch of synthetic Mamba-1.4B-shaped input
(B=4, L=2048, d_model=2048, d_inner=4096, N=16, d_conv=4; bf16 activations,
fp32 state and gradients), all inputs resident in HBM:
    ss_scan_fwd -> ss_scan_bwd -> conv1d_causal_bwd ([B, L, 4096]) -> rmsnorm_bwd ([B*L, 2048])
value = B*L*D elements per step / step time, summed over ranks (each rank runs
its own replica: the path has no cross-GPU exchange at this size).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
Prints one JSON line (rank 0).
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scan fwd+bwd (B·L·D)/s and achieved HBM GB/s vs GB300 peak, 1 GPU"
UNIT = "(B*L*D)/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mamba1p4b")
    ap.add_argument("--chunk", type=int, default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip timing the kernels next to the hot path")
    ap.add_argument("--no-others", action="store_true", help="skip timing the scan on the other workloads")
    ap.add_argument("--profile", choices=["scan", "side"], default=None,
                    help="only run the scan (or the conv1d / RMSNorm kernels) a few times on seeded device tensors, "
                         "for a profiler to capture; prints nothing but 'ok'")
    ap.add_argument("--B", type=int, default=None, help="--profile: batch rows (default: the workload's)")
    ap.add_argument("--L", type=int, default=None, help="--profile: sequence length (default: the workload's)")
    ap.add_argument("--iters", type=int, default=4, help="--profile: calls of each kernel")
    return ap.parse_args()


# ---------------------------------------------------------------- accounting

# The method's own checkpoint interval for the byte count: one checkpoint per 256 steps (the long-context
# workload's interval).  A kernel run at a shorter interval moves more checkpoint bytes; those are reported as
# overhead, not as algorithmic work.
ALG_CHUNK = 256


def algorithmic_bytes(wl, chunk=ALG_CHUNK):
    """Bytes each call must move (scratch excluded): reads of its inputs, writes of its outputs; the scan's
    checkpoints are counted after the first (the first is the initial state) at one per `chunk` steps."""
    e = 2 if wl.dtype == "bf16" else 4
    B, L, D, N, K, H = wl.B, wl.L, wl.D, wl.N, wl.d_conv, wl.d_model
    E = B * L * D
    nck = -(-L // chunk)
    ck = B * D * (nck - 1) * N * 4
    small = (D * N + D) * 4
    return {
        "scan_fwd": E * 4 * e + B * L * N * 2 * e + ck + small,
        "scan_bwd": E * (4 * e + 12) + B * L * N * (2 * e + 8) + ck + 3 * small,
        "conv1d_bwd": E * (4 + e + 4) + D * (K + 1) * 4 * 3,
        "rmsnorm_bwd": B * L * H * (2 * e + 4) + B * L * 4 + 3 * H * 4,
    }


def checkpoint_overhead_bytes(wl, chunk):
    """Checkpoint bytes one scan call moves beyond the algorithmic count: the forward writes, and the backward
    reads, all ceil(L/chunk) checkpoints (the first included), where the count allows ceil(L/256) - 1."""
    moved = wl.B * wl.D * (-(-wl.L // chunk)) * wl.N * 4
    counted = wl.B * wl.D * (-(-wl.L // ALG_CHUNK) - 1) * wl.N * 4
    return moved - counted


# FP32 operations per (b, t, d, n) cell on the recurrence (fused multiply-adds and multiplies, one each):
# forward  delta*A, delta*x*B, the state update, the C.h sum                                   -> 4
# backward the rebuild (delta*A, delta*x*B, update), G, a*G, q = aG*h, q*A, G*B, C*h, dA, dB, dC -> 12
FP32_OPS_PER_CELL = {"scan_fwd": 4, "scan_bwd": 12}


# Unit rates per SM per clock on GB300, measured on this machine by throughput probes (independent chains, one CTA
# per SM): ex2.approx.ftz 32 results (1.0 warp instruction), FP32 fused multiply-add 123 lanes (packed f32x2
# issues at 1.93 warp instructions per clock, each two lanes' work).
SFU_PER_CLK_PER_SM = 32
FMA_PER_CLK_PER_SM = 123


def alu_co_bounds(wl, ms_fwd, ms_bwd, sms):
    """The two arithmetic pipes' bounds beside the HBM roofline, from the method's own operation counts: one
    exp(delta*A) per (b, t, d, n) in each direction, and FP32_OPS_PER_CELL multiply-adds per cell."""
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    cells = wl.B * wl.L * wl.D * wl.N
    s = (ms_fwd + ms_bwd) * 1e-3
    exps = 2 * cells
    fma = cells * (FP32_OPS_PER_CELL["scan_fwd"] + FP32_OPS_PER_CELL["scan_bwd"])
    pk_exp = SFU_PER_CLK_PER_SM * sms * mhz * 1e6
    pk_fma = FMA_PER_CLK_PER_SM * sms * mhz * 1e6
    return {
        "mufu_ex2": {"per_step": exps, "achieved": exps / s, "peak": pk_exp, "unit": "exp/s",
                     "frac": round(exps / s / pk_exp, 4), "floor_us": round(exps / pk_exp * 1e6, 1)},
        "fp32_fma": {"per_step": fma, "achieved": fma / s, "peak": pk_fma, "unit": "op/s",
                     "frac": round(fma / s / pk_fma, 4), "floor_us": round(fma / pk_fma * 1e6, 1)},
        "peak_from": f"per clock per SM x {sms} SMs x {mhz:.0f} MHz",
        "measured_pipes": {n: profiled_pipes(n, wl.name) for n in ("scan_fwd", "scan_bwd")},
    }


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(name):
    f = {"scan_bwd": "scan_bwd.cu", "scan_fwd": "scan_fwd.cu", "conv1d_bwd": "conv1d_bwd.cu",
         "rmsnorm_bwd": "rmsnorm_bwd.cu"}[name]
    h = hashlib.sha256()
    for part in (f, "scan_common.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "mamba_selective_ssm_gb300", "csrc", part), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_pipes(name, wl_name):
    """Pipe utilisation of a kernel from a committed ncu summary (profiles/pipes.json), if taken on the current
    source: issue, FMA-pipe and XU (exponent) fractions of peak."""
    p = os.path.join(ROOT, "profiles", "pipes.json")
    try:
        with open(p) as f:
            rec = json.load(f)[f"{name}:{wl_name}"]
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash(name):
        return None
    return {k: rec[k] for k in ("issue_active", "fma_pipe", "xu_pipe", "smem_wavefronts", "warps_per_sm", "how") if k in rec}


def profiled_traffic(name, wl_name):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[f"{name}:{wl_name}"]
    except Exception:
        return None
    return rec["bytes_per_launch"] if rec.get("source_hash") == kernel_source_hash(name) else None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (timestamped) of SM clock and throttle reasons; keeps those inside [t0, t1]."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        if bus_id:
            cmd.insert(1, f"--id={bus_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for (ts, s) in self.samples if t0 - 0.03 <= ts <= t1 + 0.03]
        if not inside:
            inside = [s for (_, s) in self.samples[-3:]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------- distributed

def dist_init(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws, device=None):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle (CPU baseline / reference arm)

def oracle_sample(wl, d_sample, seed=0, b_sample=1):
    """The float64 oracle on b_sample batch rows and the first d_sample channels of the workload."""
    import numpy as np
    from oracle import conv1d_causal_bwd_ref, rmsnorm_bwd_ref, scan_bwd_ref, scan_fwd_ref
    from workloads import make_conv_inputs, make_rmsnorm_inputs, make_scan_inputs
    sw = wl.with_(B=b_sample, D=d_sample, d_model=max(8, d_sample // 2))
    inp = make_scan_inputs(sw, seed)
    cv = make_conv_inputs(sw, seed)
    rm = make_rmsnorm_inputs(sw, seed)
    args = (inp["x"], inp["delta"], inp["A"], inp["Bm"], inp["Cm"], inp["Dv"], inp["z"])

    def run():
        scan_fwd_ref(*args, chunk=wl.chunk)
        scan_bwd_ref(*args, inp["dy"])
        conv1d_causal_bwd_ref(cv["dout"], cv["x"], cv["w"])
        rmsnorm_bwd_ref(rm["dy"], rm["x"], rm["scale"], rm["rms"])

    return run, sw.B * sw.L * sw.D, f"B={b_sample}, L={sw.L}, D={d_sample}, N={sw.N} of the {wl.name} layer (scan fwd+bwd, " \
                                    f"conv1d bwd, RMSNorm bwd [B*L, {sw.d_model}]), float64 NumPy"


def cpu_baseline(wl, d_sample=None, b_sample=None):
    """About 10-15 s of one host core on a slice of the workload (3 of 4 rows x all channels for the 1.4B layer)."""
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    d_sample = d_sample or min(wl.D, 4096)
    b_sample = b_sample or max(1, min(wl.B - 1, (3 * 2048 * 4096) // (wl.L * d_sample)))
    run, elems, desc = oracle_sample(wl, d_sample, b_sample=b_sample)
    t = time.perf_counter()
    run()
    dt = time.perf_counter() - t
    return {"value": elems / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc, "seconds": round(dt, 3)}


def run_reference(args, ws, rank):
    from workloads import get_config
    wl = get_config(args.workload)
    if args.chunk:
        wl = wl.with_(chunk=args.chunk)
    if rank != 0:
        return
    d_sample = 64
    run, elems, desc = oracle_sample(wl, d_sample)
    for _ in range(args.warmup):
        run()
    t = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t
    v = elems * args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "L": wl.L, "D": wl.D, "N": wl.N, "d_conv": wl.d_conv,
                   "d_model": wl.d_model, "chunk": wl.chunk, "sample": desc},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ---------------------------------------------------------------- our arm

def time_scan_workload(wl, dev, peak, iters=10, warmup=3):
    """Scan forward and backward of one workload through the public API, each call bracketed by CUDA events on
    the current stream (inputs resident in HBM, parameter gradients accumulating), with the algorithmic bytes."""
    import numpy as np
    import torch

    import mamba_selective_ssm_gb300 as ss
    from workloads import make_scan_inputs

    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    inp = make_scan_inputs(wl, seed=0)
    X = {k: torch.from_numpy(np.ascontiguousarray(v)).to(tdt if k not in ("A", "Dv") else torch.float32).to(dev)
         for k, v in inp.items() if k in ("x", "delta", "z", "Bm", "Cm", "dy", "A", "Dv")}
    del inp
    st = torch.cuda.current_stream(dev)
    f32 = dict(device=dev, dtype=torch.float32)
    B, L, D, N = wl.B, wl.L, wl.D, wl.N
    out = {"dx": torch.empty((B, L, D), **f32), "ddelta": torch.empty((B, L, D), **f32), "dz": torch.empty((B, L, D), **f32),
           "dB": torch.empty((B, L, N), **f32), "dC": torch.empty((B, L, N), **f32), "dh0": torch.empty((B, D, N), **f32)}
    dA, dD = torch.zeros((D, N), **f32), torch.zeros((D,), **f32)
    wsz = max(ss.scan_bwd_workspace_size(B, L, D, N, wl.chunk, tdt), ss.scan_fwd_workspace_size(B, L, D, N, wl.chunk, tdt), 16)
    W = torch.empty(wsz, device=dev, dtype=torch.uint8)
    tf, tb = [], []
    for i in range(warmup + iters):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(st)
        y, ck, _ = ss.ss_scan_fwd(X["x"], X["delta"], X["A"], X["Bm"], X["Cm"], X["Dv"], X["z"], chunk=wl.chunk,
                                  workspace=W)
        e1.record(st)
        ss.ss_scan_bwd(X["x"], X["delta"], X["A"], X["Bm"], X["Cm"], X["Dv"], X["z"], ck, X["dy"], chunk=wl.chunk,
                       dA=dA, dD=dD, workspace=W, out=out)
        e2.record(st)
        if i >= warmup:
            tf.append((e0, e1))
            tb.append((e1, e2))
    torch.cuda.synchronize(dev)
    ms_f = statistics.median(a.elapsed_time(b) for a, b in tf)
    ms_b = statistics.median(a.elapsed_time(b) for a, b in tb)
    alg = algorithmic_bytes(wl)
    ovh = checkpoint_overhead_bytes(wl, wl.chunk)
    res = {"config": {"B": B, "L": L, "D": D, "N": N, "dtype": wl.dtype, "chunk": wl.chunk}}
    for n, ms in (("scan_fwd", ms_f), ("scan_bwd", ms_b)):
        gbs = alg[n] / (ms * 1e-3) / 1e9
        res[n] = {"ms": round(ms, 5), "alg_bytes": alg[n], "overhead_bytes": ovh, "GB/s": round(gbs, 1),
                  "frac": round(gbs / peak, 4)}
    both = alg["scan_fwd"] + alg["scan_bwd"]
    res["scan_fwd_bwd"] = {"ms": round(ms_f + ms_b, 5), "elems_per_s": B * L * D / ((ms_f + ms_b) * 1e-3),
                           "frac": round(both / ((ms_f + ms_b) * 1e-3) / 1e9 / peak, 4)}
    return res


def time_decode_tokens(wl, dev, stream, p, lib, X, sdt, tdt, T=64, reps=10):
    """One sequence (B = 1) decoded T tokens at a time through this layer's conv step and SSM step: the per-token
    time when every call is launched from the host, and when the T tokens' launches are captured once in a CUDA
    graph and replayed (the library's calls are capturable: no allocation, synchronisation or host read inside).
    Launch-bound at B = 1: the two kernels move ~1 MB per token."""
    import torch

    D, N, K = wl.D, wl.N, wl.d_conv
    g = torch.Generator(device=dev).manual_seed(7)
    xs = torch.randn((T, 1, D), device=dev, generator=g).to(tdt)
    dl = (0.001 + 0.099 * torch.rand((T, 1, D), device=dev, generator=g)).to(tdt)
    zs = torch.randn((T, 1, D), device=dev, generator=g).to(tdt)
    Bs = torch.randn((T, 1, N), device=dev, generator=g).to(tdt)
    Cs = torch.randn((T, 1, N), device=dev, generator=g).to(tdt)
    h = torch.zeros((1, D, N), device=dev, dtype=torch.float32)
    cs = torch.zeros((1, D, K), device=dev, dtype=torch.float32)
    u = torch.empty((T, 1, D), device=dev, dtype=tdt)
    y = torch.empty((T, 1, D), device=dev, dtype=tdt)
    bias = torch.zeros((D,), device=dev, dtype=torch.float32)
    sp = ctypes.c_void_p(stream.cuda_stream)

    def tokens(sp_):
        for t in range(T):
            if lib.conv1d_causal_step(p(xs[t]), p(cs), p(X["c_w"]), p(bias), p(u[t]), 1, D, K, 1, sdt, sp_) != 0:
                raise RuntimeError("conv1d_causal_step failed")
            if lib.ss_scan_step(p(u[t]), p(dl[t]), p(X["A"]), p(Bs[t]), p(Cs[t]), p(X["Dv"]), p(zs[t]), p(h), p(y[t]),
                                1, D, N, sdt, sp_) != 0:
                raise RuntimeError("ss_scan_step failed")

    tokens(sp)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        tokens(sp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us_eager = e0.elapsed_time(e1) * 1e3 / (reps * T)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        tokens(ctypes.c_void_p(cap.cuda_stream))
    stream.wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us_graph = e0.elapsed_time(e1) * 1e3 / (reps * T)
    return {"us_per_token_host_launched": round(us_eager, 2), "us_per_token_cuda_graph": round(us_graph, 2),
            "tokens": T, "B": 1, "launches_per_token": 2}


def profile_run(args):
    """The scan forward + backward (or conv1d fwd/bwd and RMSNorm fwd/bwd) on seeded device tensors of the
    workload's shape (B and L overridable), args.iters times: a fixed, short launch sequence to profile."""
    import torch

    import mamba_selective_ssm_gb300 as ss
    from workloads import get_config

    ss.build()
    wl = get_config(args.workload)
    B, L = args.B or wl.B, args.L or wl.L
    D, N, H, K = wl.D, wl.N, wl.d_model, wl.d_conv
    dev = torch.device("cuda", 0)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    g = torch.Generator(device=dev).manual_seed(0)
    rn = lambda *sh: torch.randn(*sh, device=dev, generator=g)
    if args.profile == "scan":
        x, z, dy = rn(B, L, D).to(tdt), rn(B, L, D).to(tdt), rn(B, L, D).to(tdt)
        delta = (0.001 + 0.099 * torch.rand(B, L, D, device=dev, generator=g)).to(tdt)
        Bm, Cm = rn(B, L, N).to(tdt), rn(B, L, N).to(tdt)
        A = (-(torch.arange(N, device=dev) + 1.0)).repeat(D, 1).contiguous()
        Dv = torch.ones(D, device=dev)
        for _ in range(args.iters):
            y, ck, _ = ss.ss_scan_fwd(x, delta, A, Bm, Cm, Dv, z, chunk=wl.chunk)
            ss.ss_scan_bwd(x, delta, A, Bm, Cm, Dv, z, ck, dy, chunk=wl.chunk)
    else:
        x, dout = rn(B, L, D).to(tdt), rn(B, L, D)
        w, bias = 0.5 * rn(D, K), 0.1 * rn(D)
        rx, rdy = rn(B * L, H).to(tdt), rn(B * L, H).to(tdt)
        sc = 1 + 0.1 * rn(H)
        _, rms = ss.rmsnorm_fwd(rx, sc, 1e-5)
        for _ in range(args.iters):
            ss.rmsnorm_bwd(rdy, rx, sc, rms)
            ss.rmsnorm_fwd(rx, sc, 1e-5)
            ss.conv1d_causal_fwd(x, w, bias, silu=True)
            ss.conv1d_causal_silu_bwd(dout, x, w, bias)
            ss.conv1d_causal_bwd(dout, x, w)
    torch.cuda.synchronize(dev)
    print("ok")


def main():
    args = parse()
    if args.profile:
        profile_run(args)
        return
    if args.impl == "reference":
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    ws, rank, local = dist_init(args)
    import numpy as np
    import torch

    import mamba_selective_ssm_gb300 as ss
    from mamba_selective_ssm_gb300 import _capi
    from workloads import get_config, make_conv_inputs, make_rmsnorm_inputs, make_scan_inputs

    ss.build()
    lib = ss.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = get_config(args.workload)
    if args.chunk:
        wl = wl.with_(chunk=args.chunk)
    chunk = wl.chunk
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    sdt = _capi.SS_BF16 if wl.dtype == "bf16" else _capi.SS_F32
    B, L, D, N, K, H = wl.B, wl.L, wl.D, wl.N, wl.d_conv, wl.d_model

    # ---- inputs (seeded, synthetic; host copies kept pinned for the end-to-end leg)
    inp = make_scan_inputs(wl, seed=rank)
    cv = make_conv_inputs(wl, seed=rank)
    rm = make_rmsnorm_inputs(wl, seed=rank)

    def host_t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dt).pin_memory()

    H_in = {
        "x": host_t(inp["x"], tdt), "delta": host_t(inp["delta"], tdt), "z": host_t(inp["z"], tdt),
        "Bm": host_t(inp["Bm"], tdt), "Cm": host_t(inp["Cm"], tdt), "dy": host_t(inp["dy"], tdt),
        "A": host_t(inp["A"], torch.float32), "Dv": host_t(inp["Dv"], torch.float32),
        "c_dout": host_t(cv["dout"], torch.float32), "c_x": host_t(cv["x"], tdt), "c_w": host_t(cv["w"], torch.float32),
        "r_dy": host_t(rm["dy"], tdt), "r_x": host_t(rm["x"], tdt), "r_scale": host_t(rm["scale"], torch.float32),
        "r_rms": host_t(rm["rms"], torch.float32),
    }
    del inp, cv, rm
    X = {k: v.to(dev) for k, v in H_in.items()}
    f32 = dict(device=dev, dtype=torch.float32)
    nck = lib.ss_scan_num_chunks(L, chunk)
    O = {
        "y": torch.empty((B, L, D), device=dev, dtype=tdt), "ckpt": torch.empty((B, nck, D, N), **f32),
        "h_last": torch.empty((B, D, N), **f32),
        "dx": torch.empty((B, L, D), **f32), "ddelta": torch.empty((B, L, D), **f32), "dz": torch.empty((B, L, D), **f32),
        "dB": torch.empty((B, L, N), **f32), "dC": torch.empty((B, L, N), **f32), "dh0": torch.empty((B, D, N), **f32),
        "dA": torch.zeros((D, N), **f32), "dD": torch.zeros((D,), **f32),
        "c_dx": torch.empty((B, L, D), **f32), "c_dw": torch.zeros((D, K), **f32), "c_db": torch.zeros((D,), **f32),
        "r_dx": torch.empty((B * L, H), **f32), "r_dscale": torch.zeros((H,), **f32),
    }
    ws_scan = max(lib.ss_scan_bwd_workspace_size(B, L, D, N, chunk, sdt), lib.ss_scan_fwd_workspace_size(B, L, D, N, chunk, sdt))
    ws_conv = lib.conv1d_causal_bwd_workspace_size(B, L, D, K)
    ws_rms = lib.rmsnorm_bwd_workspace_size(B * L, H)
    W = torch.empty(max(ws_scan, ws_conv, ws_rms), device=dev, dtype=torch.uint8)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    wsz = W.numel()

    calls = {
        "scan_fwd": lambda: lib.ss_scan_fwd(p(X["x"]), p(X["delta"]), p(X["A"]), p(X["Bm"]), p(X["Cm"]), p(X["Dv"]),
                                            p(X["z"]), None, p(O["y"]), p(O["ckpt"]), p(O["h_last"]),
                                            B, L, D, N, chunk, sdt, None, 0, p(W), wsz, sp),
        "scan_bwd": lambda: lib.ss_scan_bwd(p(X["x"]), p(X["delta"]), p(X["A"]), p(X["Bm"]), p(X["Cm"]), p(X["Dv"]),
                                            p(X["z"]), p(O["ckpt"]), p(X["dy"]), None, p(O["dx"]), p(O["ddelta"]),
                                            p(O["dz"]), p(O["dA"]), p(O["dB"]), p(O["dC"]), p(O["dD"]), p(O["dh0"]),
                                            B, L, D, N, chunk, sdt, None, 0, None, p(W), wsz, sp),
        "conv1d_bwd": lambda: lib.conv1d_causal_bwd(p(X["c_dout"]), p(X["c_x"]), p(X["c_w"]), p(O["c_dx"]),
                                                    p(O["c_dw"]), p(O["c_db"]), B, L, D, K, sdt, p(W), wsz, sp),
        "rmsnorm_bwd": lambda: lib.rmsnorm_bwd(p(X["r_dy"]), p(X["r_x"]), p(X["r_scale"]), p(X["r_rms"]),
                                               p(O["r_dx"]), p(O["r_dscale"]), B * L, H, sdt, p(W), wsz, sp),
    }
    launches_per_step = 1 + 2 + 2 + 2  # fwd; bwd + its reductions (dB/dC and dA/dD in one launch); conv + sum; rms + sum
    names = list(calls)

    def step(ev=None):
        for i, n in enumerate(names):
            if ev is not None:
                ev[i][0].record(stream)
            rc = calls[n]()
            if rc != 0:
                raise RuntimeError(f"{n}: {_capi.strerror(rc)}")
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus) if rank == 0 else None
    time.sleep(0.15)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in names] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(ws)
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, ws, dev)
    per_call = {n: sum(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(args.steps)) / args.steps
                for i, n in enumerate(names)}
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    if _capi.load().ss_device_status(sp) != 0:
        raise RuntimeError("a kernel reported a device-side wait timeout")

    ms_step = ms_total / args.steps
    elems = B * L * D
    value = elems * ws / (ms_step * 1e-3)
    alg = algorithmic_bytes(wl)
    ovh = checkpoint_overhead_bytes(wl, chunk)
    peak, peak_kind = measured_peak()
    kern = {}
    for n in names:
        gbs = alg[n] / (per_call[n] * 1e-3) / 1e9
        kern[n] = {"ms": round(per_call[n], 5), "alg_bytes": alg[n], "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
        if n in ("scan_fwd", "scan_bwd"):
            kern[n]["overhead_bytes"] = ovh
    dom = max(names, key=lambda n: per_call[n])
    traffic = profiled_traffic(dom, wl.name)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kern[dom]["GB/s"], "peak": peak, "unit": "GB/s",
                "frac": kern[dom]["frac"], "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                "alg_bytes_per_launch": alg[dom],
                "alg_bytes_from": f"one checkpoint per {ALG_CHUNK} steps (after the first); the run's chunk-{chunk} "
                                  "checkpoints are overhead_bytes",
                "overhead_bytes": kern[dom].get("overhead_bytes", 0)}
    scan_ms = per_call["scan_fwd"] + per_call["scan_bwd"]
    scan_bytes = alg["scan_fwd"] + alg["scan_bwd"]

    # ---- the producers and fusions next to the hot path, each timed alone on the same tensors (L2 flushed)
    nxt = {}
    if not args.no_next:
        e = 2 if wl.dtype == "bf16" else 4
        c_bias = torch.zeros((D,), **f32)
        N_ = {"conv_out": torch.empty((B, L, D), device=dev, dtype=tdt), "r_y": torch.empty((B * L, H), device=dev, dtype=tdt),
              "r_rms": torch.empty((B * L,), **f32)}
        extra = {
            "conv1d_silu_fwd": (lambda: lib.conv1d_causal_fwd(p(X["c_x"]), p(X["c_w"]), p(c_bias), p(N_["conv_out"]),
                                                              B, L, D, K, 1, sdt, sp), 2 * elems * e),
            "conv1d_silu_bwd": (lambda: lib.conv1d_causal_silu_bwd(p(X["c_dout"]), p(X["c_x"]), p(X["c_w"]), p(c_bias),
                                                                   p(O["c_dx"]), p(O["c_dw"]), p(O["c_db"]), B, L, D, K,
                                                                   sdt, p(W), wsz, sp), elems * (8 + e)),
            "rmsnorm_fwd": (lambda: lib.rmsnorm_fwd(p(X["r_x"]), p(X["r_scale"]), ctypes.c_float(1e-5), p(N_["r_y"]),
                                                    p(N_["r_rms"]), B * L, H, sdt, sp), B * L * (2 * H * e + 4)),
        }
        # the scan with delta = softplus(raw + dt_bias) computed in its prologues (same tensors, delta read as raw)
        dtb = torch.zeros((D,), **f32)
        ddtb = torch.zeros((D,), **f32)
        extra["scan_fwd_fused_softplus"] = (
            lambda: lib.ss_scan_fwd(p(X["x"]), p(X["delta"]), p(X["A"]), p(X["Bm"]), p(X["Cm"]), p(X["Dv"]), p(X["z"]),
                                    None, p(O["y"]), p(O["ckpt"]), p(O["h_last"]), B, L, D, N, chunk, sdt, p(dtb), 1,
                                    p(W), wsz, sp), alg["scan_fwd"] + D * 4)
        extra["scan_bwd_fused_softplus"] = (
            lambda: lib.ss_scan_bwd(p(X["x"]), p(X["delta"]), p(X["A"]), p(X["Bm"]), p(X["Cm"]), p(X["Dv"]), p(X["z"]),
                                    p(O["ckpt"]), p(X["dy"]), None, p(O["dx"]), p(O["ddelta"]), p(O["dz"]), p(O["dA"]),
                                    p(O["dB"]), p(O["dC"]), p(O["dD"]), p(O["dh0"]), B, L, D, N, chunk, sdt, p(dtb), 1,
                                    p(ddtb), p(W), wsz, sp), alg["scan_bwd"] + 2 * D * 4)
        # decode: one token for Bd sequences of this layer; Bd = 1024 puts the state (Bd*D*N fp32) above L2
        Bd = 1024
        g = torch.Generator(device=dev).manual_seed(rank)
        dec = {"x": torch.randn((Bd, D), device=dev, generator=g).to(tdt),
               "delta": (0.001 + 0.099 * torch.rand((Bd, D), device=dev, generator=g)).to(tdt),
               "z": torch.randn((Bd, D), device=dev, generator=g).to(tdt),
               "Bm": torch.randn((Bd, N), device=dev, generator=g).to(tdt),
               "Cm": torch.randn((Bd, N), device=dev, generator=g).to(tdt),
               "h": torch.zeros((Bd, D, N), **f32), "y": torch.empty((Bd, D), device=dev, dtype=tdt),
               "cs": torch.zeros((Bd, D, K), **f32), "co": torch.empty((Bd, D), device=dev, dtype=tdt)}
        extra["scan_step_decode"] = (
            lambda: lib.ss_scan_step(p(dec["x"]), p(dec["delta"]), p(X["A"]), p(dec["Bm"]), p(dec["Cm"]), p(X["Dv"]),
                                     p(dec["z"]), p(dec["h"]), p(dec["y"]), Bd, D, N, sdt, sp),
            2 * Bd * D * N * 4 + 4 * Bd * D * e + 2 * Bd * N * e + D * N * 4 + D * 4)
        extra["conv_step_decode"] = (
            lambda: lib.conv1d_causal_step(p(dec["x"]), p(dec["cs"]), p(X["c_w"]), p(c_bias), p(dec["co"]), Bd, D, K, 1,
                                           sdt, sp),
            2 * Bd * D * K * 4 + 2 * Bd * D * e + D * K * 4 + D * 4)
        # each launch timed alone after a read of 256 MB (> L2): no launch reads what the previous one left in L2,
        # and the L2 holds only clean lines when it starts (a write-based flush would leave ~L2-sized dirty data
        # to be written back inside the timed launch)
        flush = torch.ones((64 << 20,), device=dev, dtype=torch.float32)
        for n, (fn, nbytes) in extra.items():
            for _ in range(3):
                if fn() != 0:
                    raise RuntimeError(f"{n} failed")
            iters = 20
            evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
            for a0, a1 in evp:
                flush.sum()
                a0.record(stream)
                fn()
                a1.record(stream)
            torch.cuda.synchronize(dev)
            ms = sum(a0.elapsed_time(a1) for a0, a1 in evp) / iters
            gbs = nbytes / (ms * 1e-3) / 1e9
            nxt[n] = {"ms": round(ms, 5), "alg_bytes": nbytes, "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
        nxt["decode_tokens_b1"] = time_decode_tokens(wl, dev, stream, p, lib, X, sdt, tdt)

    # ---- the scan on the other workloads of the method (timed the same way, inputs resident in HBM)
    others = {}
    if not args.no_others and ws == 1:
        for oname in ("long", "short", "mamba130m"):
            if oname == wl.name:
                continue
            others[oname] = time_scan_workload(get_config(oname), dev, peak, iters=10)

    # ---- end to end through the public API: pinned host inputs in, results out, every step.
    # Three streams pipeline consecutive steps: step i's host->device copies (into one of two input slots)
    # overlap step i-1's kernels and step i-2's device->host copies; every copy of every step stays inside
    # the timed region.
    e2e = None
    if not args.no_e2e:
        keys_in = list(H_in)
        h2d = sum(H_in[k].numel() * H_in[k].element_size() for k in keys_in)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        slots = [{k: torch.empty_like(H_in[k], device=dev) for k in keys_in} for _ in range(2)]
        host_out = [{}, {}]
        freed = [torch.cuda.Event(), torch.cuda.Event()]  # compute done with an input slot
        for ev in freed:
            ev.record(stream)

        def e2e_step(i):
            sl, ho = slots[i % 2], host_out[i % 2]
            s_in.wait_event(freed[i % 2])
            with torch.cuda.stream(s_in):
                for k in keys_in:
                    sl[k].copy_(H_in[k], non_blocking=True)
            stream.wait_stream(s_in)
            Xd = sl
            y, ck, hl = ss.ss_scan_fwd(Xd["x"], Xd["delta"], Xd["A"], Xd["Bm"], Xd["Cm"], Xd["Dv"], Xd["z"], chunk=chunk)
            g = ss.ss_scan_bwd(Xd["x"], Xd["delta"], Xd["A"], Xd["Bm"], Xd["Cm"], Xd["Dv"], Xd["z"], ck, Xd["dy"],
                               chunk=chunk)
            cdx, cdw, cdb = ss.conv1d_causal_bwd(Xd["c_dout"], Xd["c_x"], Xd["c_w"])
            rdx, rds = ss.rmsnorm_bwd(Xd["r_dy"], Xd["r_x"], Xd["r_scale"], Xd["r_rms"])
            freed[i % 2].record(stream)
            res = {"y": y, "h_last": hl, "cdx": cdx, "cdw": cdw, "cdb": cdb, "rdx": rdx, "rds": rds}
            res.update({k: v for k, v in g.items() if v is not None})
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_out):
                for k, v in res.items():
                    if k not in ho:
                        ho[k] = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                    ho[k].copy_(v, non_blocking=True)
                    v.record_stream(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        s_in.wait_stream(stream)
        for i in range(args.steps):
            e2e_step(i)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        ms_e2e = max_over_ranks(e0.elapsed_time(e1), ws, dev) / args.steps
        e2e = {"value": elems * ws / (ms_e2e * 1e-3), "unit": UNIT, "ms_per_step": round(ms_e2e, 4),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "how": "public Python API; inputs copied from pinned host memory and every result copied back each "
                      "step, on copy streams pipelined with the compute stream"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "L": L, "D": D, "N": N, "d_conv": K, "d_model": H, "chunk": chunk,
                       "activations": wl.dtype, "state_and_grads": "f32", "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2 (no flush): x, delta, z, dy alone are "
                             f"{4 * elems * (2 if wl.dtype == 'bf16' else 4) / 1e6:.0f} MB vs 129 MB L2"},
            "roofline": roofline,
            "scan_fwd_bwd": {"ms": round(scan_ms, 5), "elems_per_s": elems / (scan_ms * 1e-3),
                             "alg_GB/s": round(scan_bytes / (scan_ms * 1e-3) / 1e9, 1),
                             "frac": round(scan_bytes / (scan_ms * 1e-3) / 1e9 / peak, 4),
                             "alg_bytes": scan_bytes, "overhead_bytes": 2 * ovh,
                             "alu_co_bounds": alu_co_bounds(wl, per_call["scan_fwd"], per_call["scan_bwd"],
                                                            torch.cuda.get_device_properties(dev).multi_processor_count)},
            "other_workloads": others or None,
            "kernels": kern, "next_kernels": nxt or None, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": launches_per_step * args.steps,
        }), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
