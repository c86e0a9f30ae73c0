#!/usr/bin/env python
"""Benchmark of the dilution-attention forward (and cached decode) on GB300.

Default workload: bf16 forward, B=4, H=12, T=16384, d=64 (the training
context of the 24-layer decoders), tau = 1, eps = 1e-6, seeded synthetic
inputs with 128 planted retrieval pairs per head.  One step = one call of
dilution_attn_fwd (row statistics, demand sweep, finalize).  The JSON line
reports forward TFLOP/s on the algorithmic count 3 * d * T(T+1) * B * H
(q.k for the normaliser, q.k again in the sweep, share.v; causal pairs only),
plus tokens/s, the dominant kernel's roofline, an end-to-end number through
host buffers, clocks, the cached-decode step at 8 x 131072 tokens, and the
float64 CPU oracle timed on a bounded sample as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(heads are independent; there is no data-path collective): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dilution-attn fwd TFLOP/s & tokens/s at T=16K, % of GB300 BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SWEEP_SOURCES = ["long_context_attention_gb300/csrc/fwd_bf16.cu", "long_context_attention_gb300/csrc/da_ptx.cuh",
                 "long_context_attention_gb300/csrc/da_internal.h"]
SWEEP_PROFILE = os.path.join(ROOT, "profiles", "sweep_kernel_fwd_bf16_t16384.md")
DECODE_SOURCES = ["long_context_attention_gb300/csrc/decode.cu", "long_context_attention_gb300/csrc/da_internal.h",
                  "long_context_attention_gb300/csrc/da_ptx.cuh"]
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_bf16_ctx131072.md")


# --------------------------------------------------------------------------- helpers
def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="fwd_bf16_t16384")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-train", action="store_true", help="skip the forward+backward training-step timing")
    ap.add_argument("--no-d128", action="store_true", help="skip the head-dimension-128 forward timing")
    ap.add_argument("--train-only", action="store_true", help="time only the training step (profiling)")
    ap.add_argument("--train-batch", type=int, default=None, help="training-step batch (default: the workload's)")
    ap.add_argument("--train-t", type=int, default=None, help="training-step sequence length (default: 16384)")
    ap.add_argument("--train-d", type=int, default=None, help="training-step head dimension (default: 64)")
    ap.add_argument("--decode-ctx", type=int, default=None, help="cached tokens per sequence (default: the workload's)")
    ap.add_argument("--decode-steps", type=int, default=None, help="decode steps timed (default: the workload's)")
    ap.add_argument("--decode-only", action="store_true", help="skip the forward measurement")
    ap.add_argument("--cpu-heads", type=int, default=5, help="full T=16384 heads in the oracle's CPU sample")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (smaller cases for profiling; not a bench line)")
    return ap.parse_args(argv)


def fwd_flops(B, H, T, d):
    """Algorithmic forward FLOP: 3 contractions x 2d x causal pairs."""
    return 3 * d * T * (T + 1) * B * H


def sweep_flops(B, H, T, d):
    """The demand sweep's share: q.k again and share.v over the causal pairs."""
    return 2 * d * T * (T + 1) * B * H


# Special-function-unit (MUFU) results the forward issues per causal pair:
# one exponential in the row statistics; one exponential and one reciprocal per
# pair of queries in the sweep.  Peak: 32 MUFU results per SM per clock (an
# isolated ex2 loop reached 29.6 on GB300), times the SM count and clock.
SFU_PER_PAIR = {"rowstats": 1.0, "sweep": 1.5}
SFU_PER_SM_CLK = 32


def sfu_report(B, H, T, kern_ms, n_sm, sm_mhz):
    """Achieved MUFU results/s of the two forward kernels and of the step."""
    pairs = T * (T + 1) // 2 * B * H
    peak = SFU_PER_SM_CLK * n_sm * sm_mhz * 1e6 / 1e12
    out = {"unit": "Tops/s", "peak": peak, "peak_source": f"{SFU_PER_SM_CLK}/SM/clk x {n_sm} SMs x {sm_mhz:.0f} MHz",
           "ops_per_pair": SFU_PER_PAIR}
    tot_ops, tot_ms = 0.0, 0.0
    for k_, per in SFU_PER_PAIR.items():
        ops = per * pairs
        out[k_] = {"achieved": ops / (kern_ms[k_] * 1e-3) / 1e12}
        out[k_]["frac"] = out[k_]["achieved"] / peak
        tot_ops += ops
        tot_ms += kern_ms[k_]
    out["achieved"] = tot_ops / (tot_ms * 1e-3) / 1e12
    out["frac"] = out["achieved"] / peak
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def sources_hash(sources=None):
    h = hashlib.sha256()
    for rel in sources or SWEEP_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile=None, sources=None, workload=None):
    """DRAM bytes per launch (per step for the decode) from a committed ncu
    summary, if it was taken on the current kernel source and on this
    workload (its `profile_workload` line, e.g. "fwd_bf16_t16384 B=4 H=12
    T=16384 d=64"), else None."""
    try:
        text = open(profile or SWEEP_PROFILE).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ")
        if ":" in line:
            key, _, val = line.partition(":")
            vals[key.strip().strip("`")] = val.strip().strip("`")
    if vals.get("kernel_source_hash") != sources_hash(sources):
        return None
    if workload is not None and vals.get("profile_workload") != workload:
        return None
    try:
        return float(vals["traffic_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(x, device=None):
    """The largest value of x over the ranks of the default process group
    (x itself when no group is initialised): every replica's timing is taken
    and the slowest one defines the job's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(seed, rank):
    """Seed of rank `rank`'s independent replica batch."""
    return seed + 1000 * rank


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0, t1):
        """Median SM clock of the samples taken in [t0, t1] (wall clock)."""
        samples = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                samples.append((ts, float(f[2]), float(f[3]), f[5:]))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [s for s in samples if t0 - 1.0 <= s[0] <= t1 + 1.0] or samples
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in inside:
            for n, v in zip(names[1:], s[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


# ------------------------------------------------------------------ CPU oracle sample
def oracle_sample(q, k, v, rows, tau=1.0, eps=1e-6):
    """Time the float64 oracle on the first ``rows`` queries of one head;
    returns (algorithmic FLOP, seconds, the oracle's output rows)."""
    import oracle.dilution as od
    t0 = time.perf_counter()
    r = od.dilution_forward_rowblocked_head(q, k, v, tau, eps, rows=rows)
    dt = time.perf_counter() - t0
    d = q.shape[1]
    flops = 3 * d * rows * (rows + 1)    # causal pairs of the first `rows` queries, 3 x 2d each
    return flops, dt, r["out"]


def cpu_baseline(heads, seed=2, gpu_forward=None):
    """The oracle on `heads` full heads (T = 16384) of the benchmark workload,
    generated on the host with the same recipe (about 10-30 s of CPU work).

    With ``gpu_forward`` (q, k, v host tensors -> out as float64 NumPy, run by
    this library's kernels) the same heads also go through the GPU path and
    the second return value reports the largest |out - oracle| against the
    bf16 bound of 2e-2; else it is None."""
    import numpy as np
    from long_context_attention_gb300 import inputs
    w = inputs.WORKLOADS["fwd_bf16_t16384"]
    q, k, v = inputs.make_qkv(1, heads, w.T, w.d, q_std=w.q_std, pairs=w.pairs, seed=seed, dtype="bf16")
    tot_f, tot_t = 0, 0.0
    ref = []
    for h in range(heads):
        qh, kh, vh = (x[0, h].double().numpy() for x in (q, k, v))
        f, t, o = oracle_sample(qh, kh, vh, w.T)
        tot_f += f
        tot_t += t
        ref.append(o)
    base = {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"float64 NumPy oracle (row-blocked), {heads} full heads of 1 x 12 x 16384 x 64 with the "
                      f"workload's recipe ({tot_f / 1e9:.0f} GFLOP algorithmic, {tot_t:.1f} s)",
            "seconds": tot_t, "cpu_count": os.cpu_count(), "np": np.__version__}
    if gpu_forward is None:
        return base, None
    got = gpu_forward(q, k, v)
    err = max(float(np.abs(got[0, h] - ref[h]).max()) for h in range(heads))
    parity = {"heads": heads, "rows_per_head": w.T, "shape": f"1 x {heads} x {w.T} x {w.d} bf16, the workload's recipe",
              "max_abs_err_out": err, "tolerance": 2e-2, "ok": err <= 2e-2,
              "against": "the float64 oracle's output on the same heads (the cpu_baseline sample)"}
    return base, parity


# ---------------------------------------------------------------------- reference arm
def workload_config(args, w, B, world, ws_bytes):
    """The ``config`` object of both arms: the workload and how the timed steps
    treat the L2 (no flush; the per-step inputs and workspace exceed it)."""
    in_bytes = 3 * B * w.H * w.T * w.d * (2 if w.dtype == "bf16" else 4)
    l2 = (f"no flush; inputs {in_bytes / 1e6:.0f} MB + workspace {ws_bytes / 1e6:.0f} MB per step"
          + (", larger than the 129 MB L2" if in_bytes + ws_bytes > 129e6 else " (fits in L2: small case)"))
    return {"workload": args.workload, "B": B, "H": w.H, "T": w.T, "d": w.d, "tau": 1.0, "eps": w.eps,
            "planted_pairs_per_head": w.pairs, "parallelism": f"replicas{world}", "l2": l2}


def run_reference(args):
    """The oracle as it stands, on the host cores, on this arm's workload.  Each
    timed step is one whole (batch, head) slice of the workload (all T query
    rows of one of its B x H independent heads, taken in turn); its TFLOP/s is
    that head's algorithmic FLOP over the step's time, the same unit as the GPU
    arm's whole-batch figure.  Warm-up steps run the first 1024 rows of a head."""
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    from long_context_attention_gb300 import binding as b
    from long_context_attention_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    B = args.batch or w.B
    q, k, v = inputs.make_qkv(B, w.H, w.T, w.d, q_std=w.q_std, pairs=w.pairs, seed=w.seed, dtype=w.dtype)
    heads = [(bb, hh) for bb in range(B) for hh in range(w.H)]

    def head(j):
        bb, hh = heads[j % len(heads)]
        return (x[bb, hh].double().numpy() for x in (q, k, v))

    for j in range(args.warmup):
        oracle_sample(*head(j), rows=min(1024, w.T))
    tot_f, tot_t = 0, 0.0
    for j in range(args.steps):
        f, t, _ = oracle_sample(*head(j), rows=w.T)
        tot_f += f
        tot_t += t
    val = tot_f / tot_t / 1e12
    sample = (f"float64 NumPy oracle (row-blocked), one whole head of the {args.workload} workload per step "
              f"({args.steps} heads, all {w.T} query rows each, {tot_t:.1f} s)")
    ws_bytes = b.dilution_attn_fwd_workspace_size(B, w.H, w.T, w.d, b.DA_BF16 if w.dtype == "bf16" else b.DA_F32)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args, w, B, world, ws_bytes),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------ our arm
def run_fwd_workload(torch, b, inputs, dev, name, steps, warmup, peaks):
    """Forward of another workload (d = 128): K timed steps with the three
    kernels' events; returns TFLOP/s, per-kernel ms and the sweep's and row
    statistics' fractions of the bf16 peak."""
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_qkv(w.B, w.H, w.T, w.d, q_std=w.q_std, pairs=w.pairs, seed=w.seed, dtype=w.dtype,
                              device=dev)
    out = torch.empty_like(q)
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(w.B, w.H, w.T, w.d, b._dtype_code(q)), dtype=torch.uint8,
                     device=dev)
    for _ in range(warmup):
        b.dilution_attn_fwd(q, k, v, out, workspace=ws)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        b.dilution_attn_fwd_with_events(q, k, v, out, workspace=ws, events=evs[i], check=False)
    t1.record()
    torch.cuda.synchronize()
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    ms = t0.elapsed_time(t1) / steps
    kern = {n_: statistics.mean(e4[j].elapsed_time(e4[j + 1]) for e4 in evs)
            for j, n_ in enumerate(("rowstats", "sweep", "finalize"))}
    fl = fwd_flops(w.B, w.H, w.T, w.d)
    sw = sweep_flops(w.B, w.H, w.T, w.d)
    peak = peaks["bf16_tflops"]
    res = {"workload": name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "steps": steps, "ms_per_step": ms,
           "tflops": fl / (ms * 1e-3) / 1e12, "pct_of_bf16_peak": 100.0 * fl / (ms * 1e-3) / 1e12 / peak,
           "tokens_per_s": w.B * w.T / (ms * 1e-3), "kernels_ms": kern,
           "sweep_frac": sw / (kern["sweep"] * 1e-3) / 1e12 / peak,
           "rowstats_frac": (fl - sw) / (kern["rowstats"] * 1e-3) / 1e12 / peak, "gpu_launches": 4 * steps}
    del q, k, v, out, ws
    torch.cuda.empty_cache()
    return res


def run_decode(torch, b, inputs, dev, warmup, peaks, ctx=None, n_steps=None):
    """8 independent 131072-token caches (built by an untimed prefill), 256 steps."""
    w = inputs.WORKLOADS["decode_bf16_ctx131072"]
    B, H, N, d = w.B, w.H, ctx or w.T, w.d
    steps = n_steps or w.extra["steps"]
    from long_context_attention_gb300 import yarn_tau
    tau = yarn_tau(w.tau_scale)
    T_cap = N + steps
    q, k, v = inputs.make_workload(w, device=dev, T=N)
    kc = torch.empty(B, H, T_cap, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    kc[:, :, :N] = k
    vc[:, :, :N] = v
    dem = torch.zeros(B, H, T_cap, device=dev)
    dem_n = torch.empty(B, H, N, device=dev)
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, N, d, b.DA_BF16), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    # prefill at 131072 tokens (also reported, as the long-context prefill)
    b.dilution_attn_fwd(q, k, v, out, None, None, dem_n, tau=tau, eps=w.eps, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    b.dilution_attn_fwd(q, k, v, out, None, None, dem_n, tau=tau, eps=w.eps, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    pre_ms = e0.elapsed_time(e1)
    pre = {"workload": f"prefill_bf16_t{N}_b{B}", "B": B, "H": H, "T": N, "tau": tau,
           "ms": pre_ms, "tflops": fwd_flops(B, H, N, d) / (pre_ms * 1e-3) / 1e12,
           "tokens_per_s": B * N / (pre_ms * 1e-3)}
    dem[:, :, :N] = dem_n
    del q, out, ws, dem_n
    qs = inputs.make_like((steps, B, H, d), std=w.q_std, seed=w.seed + 100, dtype="bf16", device=dev)
    ks = inputs.make_like((steps, B, H, d), seed=w.seed + 101, dtype="bf16", device=dev)
    vs = inputs.make_like((steps, B, H, d), seed=w.seed + 102, dtype="bf16", device=dev)
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    dws = torch.empty(b.dilution_attn_decode_workspace_size(B, H, T_cap, d), dtype=torch.uint8, device=dev)
    dem0 = dem.clone()
    for i in range(warmup):   # warm-up steps on the real state, then restore it
        b.dilution_attn_decode_step(qs[i], ks[i], vs[i], kc, vc, dem, N, o, tau=tau, eps=w.eps, workspace=dws)
    torch.cuda.synchronize()
    dem.copy_(dem0)
    del dem0
    torch.cuda.synchronize()
    e0.record()
    for i in range(steps):
        b.dilution_attn_decode_step(qs[i], ks[i], vs[i], kc, vc, dem, N + i, o, tau=tau, eps=w.eps, workspace=dws)
    e1.record()
    torch.cuda.synchronize()
    assert b.dilution_attn_get_error(dws) == b.DA_OK
    ms = e0.elapsed_time(e1)
    keys = sum((N + i + 1) for i in range(steps)) * B * H
    algo_bytes = (4 * d + 8) * keys     # K and V rows (bf16) + demand read and write (fp32)
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    return pre, {"workload": f"decode_bf16_ctx{N}", "B": B, "H": H, "n_ctx": N, "steps": steps, "tau": tau,
                 "ms_per_step": ms / steps, "tokens_per_s": B * steps / (ms * 1e-3),
                 "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": gbs / peaks["hbm_gbs"],
                              "traffic": profiled_traffic(DECODE_PROFILE, DECODE_SOURCES,
                                                          f"{w.name} B={B} H={H} n_ctx={N} d={d}"),
                              "bytes_per_step": algo_bytes / steps},
                 "gpu_launches": 3 * steps}


def bwd_flops(B, H, T, d):
    """Algorithmic backward FLOP: the five contractions S = Q K^T, dA = dout V^T,
    dV = A^T dout, dK = ds^T Q, dQ = ds K over the causal pairs."""
    return 5 * d * T * (T + 1) * B * H


def run_train(torch, b, inputs, dev, steps=5, batch=None, T=None, d=None):
    """Forward + backward at the training shape (4 x 12 x 16384 x 64, all N(0,1));
    ``batch`` / ``T`` / ``d`` override it (profiling, head dimension 128)."""
    w = inputs.WORKLOADS["train_bf16_t16384"]
    B, H, d = batch or w.B, w.H, d or w.d
    T = T or w.T
    q, k, v = inputs.make_qkv(B, H, T, d, q_std=w.q_std, pairs=w.pairs, seed=w.seed, dtype=w.dtype, device=dev)
    g = inputs.make_like((B, H, T, d), seed=w.seed + 1, dtype=w.dtype, device=dev)
    out = torch.empty_like(q)
    lse2 = torch.empty(B, H, T, device=dev)
    # one workspace: the forward keeps its demand checkpoints and accumulators
    # there for the backward (DA_FLAG_KEEP_FOR_BACKWARD)
    keep = b.DA_FLAG_KEEP_FOR_BACKWARD
    bws = torch.empty(b.dilution_attn_bwd_workspace_size(B, H, T, d, b.DA_BF16), dtype=torch.uint8, device=dev)
    fws = bws
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]

    def step(e3=None):
        if e3:
            e3[0].record()
        b.dilution_attn_fwd_ex(q, k, v, out, lse2, flags=keep, workspace=bws)
        if e3:
            e3[1].record()
        b.dilution_attn_bwd_ex(q, k, v, g, lse2, dq, dk, dv, flags=keep, workspace=bws)
        if e3:
            e3[2].record()

    step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        step(ev[i])
    e1.record()
    torch.cuda.synchronize()
    assert b.dilution_attn_get_error(fws) == b.DA_OK and b.dilution_attn_get_error(bws) == b.DA_OK
    ms = e0.elapsed_time(e1) / steps
    bwd_ms = statistics.mean(e3[1].elapsed_time(e3[2]) for e3 in ev)
    fwd_f, bwd_f = fwd_flops(B, H, T, d), bwd_flops(B, H, T, d)
    return {"workload": "train_bf16_t16384" if (B, T, d) == (w.B, w.T, w.d) else f"train_bf16_b{B}_t{T}_d{d}",
            "B": B, "H": H, "T": T, "d": d, "steps": steps, "ms_per_step": ms,
            "tokens_per_s": B * T / (ms * 1e-3), "bwd_ms": bwd_ms,
            "tflops": (fwd_f + bwd_f) / (ms * 1e-3) / 1e12, "bwd_tflops": bwd_f / (bwd_ms * 1e-3) / 1e12,
            "backward": "tcgen05: the forward keeps its demand checkpoints; a reverse pass (rho, dV, the u-part of dK), a light pass (the rho-part of dK), a dQ pass",
            "fwd_flop": fwd_f, "bwd_flop": bwd_f}


def run_ours(args):
    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from long_context_attention_gb300 import binding as b
    from long_context_attention_gb300 import inputs
    b.load(build_if_missing=True)
    peaks, peaks_kind = load_peaks()

    if args.train_only:
        res = run_train(torch, b, inputs, dev, steps=max(1, args.steps), batch=args.train_batch, T=args.train_t,
                        d=args.train_d)
        if rank == 0:
            print(json.dumps({"train_step": res}), flush=True)
        return 0
    if args.decode_only:
        pre, dec = run_decode(torch, b, inputs, dev, max(3, args.warmup), peaks, args.decode_ctx, args.decode_steps)
        if rank == 0:
            print(json.dumps({"decode": dec, "prefill": pre}), flush=True)
        return 0
    w = inputs.WORKLOADS[args.workload]
    B, H, T, d = (args.batch or w.B), w.H, w.T, w.d
    # each rank is an independent replica with its own seeded batch
    q, k, v = inputs.make_qkv(B, H, T, d, q_std=w.q_std, pairs=w.pairs, seed=replica_seed(w.seed, rank),
                              dtype=w.dtype, device=dev)
    out = torch.empty_like(q)
    ws = torch.empty(b.dilution_attn_fwd_workspace_size(B, H, T, d, b._dtype_code(q)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e4 in evs:            # materialise the CUDA events before timing
        for e in e4:
            e.record()
    for _ in range(W):
        b.dilution_attn_fwd(q, k, v, out, workspace=ws)
    torch.cuda.synchronize()
    assert b.dilution_attn_get_error(ws) == b.DA_OK

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        t_start.record(stream)
        for i in range(K):
            b.dilution_attn_fwd_with_events(q, k, v, out, workspace=ws, events=evs[i], check=False)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        w1 = time.time()
    assert b.dilution_attn_get_error(ws) == b.DA_OK
    ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    per = {"rowstats": [], "sweep": [], "finalize": []}
    for e4 in evs:
        per["rowstats"].append(e4[0].elapsed_time(e4[1]))
        per["sweep"].append(e4[1].elapsed_time(e4[2]))
        per["finalize"].append(e4[2].elapsed_time(e4[3]))
    kern_ms = {k_: statistics.mean(v_) for k_, v_ in per.items()}
    flops_step = fwd_flops(B, H, T, d)
    ms_step = ms / K
    value = world * flops_step * K / (ms * 1e-3) / 1e12
    timed_s = ms * 1e-3
    peak_t = peaks["bf16_tflops_sustained"] if timed_s > 1.0 else peaks["bf16_tflops"]
    sweep_tf = sweep_flops(B, H, T, d) / (kern_ms["sweep"] * 1e-3) / 1e12
    rs_tf = (flops_step - sweep_flops(B, H, T, d)) / (kern_ms["rowstats"] * 1e-3) / 1e12
    clocks = clk.summary(w0, w1)

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": workload_config(args, w, B, world, ws.numel()),
            "tokens_per_s": world * B * T * K / (ms * 1e-3),
            "pct_of_bf16_peak": 100.0 * value / world / peak_t,
            "kernels_ms": kern_ms,
            "roofline": {"bound": "tensor", "kernel": "sweep_kernel", "achieved": sweep_tf, "peak": peak_t,
                         "unit": "TFLOP/s", "frac": sweep_tf / peak_t,
                         "traffic": profiled_traffic(workload=f"{w.name} B={B} H={H} T={T} d={d}"),
                         "peak_source": f"{peaks_kind} {'sustained' if timed_s > 1.0 else 'burst'} bf16",
                         "rowstats_achieved": rs_tf, "rowstats_frac": rs_tf / peak_t},
            "sfu": sfu_report(B, H, T, kern_ms, torch.cuda.get_device_properties(dev).multi_processor_count,
                              clocks.get("sm_max_mhz") or 2070.0),
            "gpu_launches": 4 * K, "clocks": clocks}

    if not args.no_e2e:
        # Host buffers in, result back, every step.  The batch goes through in
        # chunks on three streams (copy in / compute / copy out), so that the
        # copies of one chunk overlap the compute of another, as a caller
        # streaming requests would do; every byte still crosses inside the
        # timed region.
        Ke = max(1, min(K, 10))
        nch = 2 if B % 2 == 0 else 1
        Bc = B // nch
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        dq, dk, dv = (torch.empty_like(x) for x in (q, k, v))
        wsc = torch.empty(b.dilution_attn_fwd_workspace_size(Bc, H, T, d, b._dtype_code(q)), dtype=torch.uint8,
                          device=dev)
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(nch)] for _ in range(3))
        for e in ev_in + ev_cmp + ev_out:
            e.record()

        def e2e_step():
            for c in range(nch):
                sl = slice(c * Bc, (c + 1) * Bc)
                s_in.wait_event(ev_cmp[c])          # the chunk's inputs are free again
                with torch.cuda.stream(s_in):
                    dq[sl].copy_(hq[sl], non_blocking=True)
                    dk[sl].copy_(hk[sl], non_blocking=True)
                    dv[sl].copy_(hv[sl], non_blocking=True)
                ev_in[c].record(s_in)
                s_cmp.wait_event(ev_in[c])
                s_cmp.wait_event(ev_out[c])         # the chunk's output was read back
                b.dilution_attn_fwd(dq[sl], dk[sl], dv[sl], out[sl], workspace=wsc, stream=s_cmp)
                ev_cmp[c].record(s_cmp)
                s_out.wait_event(ev_cmp[c])
                with torch.cuda.stream(s_out):
                    hout[sl].copy_(out[sl], non_blocking=True)
                ev_out[c].record(s_out)

        e2e_step()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(cur)
        for st in (s_in, s_cmp, s_out):
            st.wait_stream(cur)
        for _ in range(Ke):
            e2e_step()
        for st in (s_in, s_cmp, s_out):
            cur.wait_stream(st)
        e1.record(cur)
        torch.cuda.synchronize()
        assert b.dilution_attn_get_error(wsc) == b.DA_OK
        ems = max_over_ranks(e0.elapsed_time(e1), dev)
        line["e2e"] = {"value": world * flops_step * Ke / (ems * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": 3 * q.numel() * q.element_size(),
                       "d2h_bytes_per_step": out.numel() * out.element_size(), "steps": Ke,
                       "ms_per_step": ems / Ke, "chunks": nch,
                       "overlap": "copy-in, compute and copy-out streams per batch chunk"}
        del wsc
        del hq, hk, hv, hout, dq, dk, dv

    del q, k, v, out, ws
    torch.cuda.empty_cache()
    if not args.no_d128 and args.workload != "fwd_bf16_t16384_d128":
        line["fwd_d128"] = run_fwd_workload(torch, b, inputs, dev, "fwd_bf16_t16384_d128", max(3, min(K, 20)),
                                            max(3, W), peaks)
    if not args.no_train:
        line["train_step"] = run_train(torch, b, inputs, dev, batch=args.train_batch, T=args.train_t)
    if not args.no_decode:
        pre, dec = run_decode(torch, b, inputs, dev, max(3, W), peaks, args.decode_ctx, args.decode_steps)
        line["prefill_131072"] = pre
        line["decode"] = dec

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def gpu_forward(qh, kh, vh):
            o = b.dilution_attn_fwd(*(x.to(dev) for x in (qh, kh, vh)), tau=1.0, eps=w.eps)
            torch.cuda.synchronize()
            return o.double().cpu().numpy()

        line["cpu_baseline"], line["parity"] = cpu_baseline(args.cpu_heads, gpu_forward=gpu_forward)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
