#!/usr/bin/env python
"""Benchmark of the attention-KL hot path on one GB300 (or N independent ranks).

Default workload: B=1, H=32, N_Q=N_K=65536, D=128, causal, bf16 inputs; one
step is the forward (KL, LSE1, LSE2) plus the setting-1 backward (dQ2, dK2).
Counted FLOPs are the MMA FLOPs on unmasked (query, key) pairs: 4D per pair for
the forward and 8D per pair for the backward.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of a launch,
# divided by its algorithmic bytes, from the ncu summaries under profiles/ for
# the current build of each kernel (scaled to a full launch by the units it
# processes); absent until measured, and removed when the kernel changes.
NCU_TRAFFIC_RATIO = {"splitk": 1.0011}  # profiles/splitk_partial_decode_b2h32_nq4_nk131072.md
# For tensor-bound kernels: measured DRAM bytes per unmasked (query, key) pair.
NCU_TRAFFIC_PER_PAIR = {"fwd": 0.0321, "bwd_fused": 0.0744}  # profiles/fwd_tc_b1h4_n65536_causal.md, profiles/bwd_fused_b1h4_n65536_causal.md

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="kl_b1h32_n65536_d128_causal")
    ap.add_argument("--setting", type=int, default=1, choices=[1, 2])
    ap.add_argument("--bwd-mode", default="auto", choices=["auto", "fused", "separate", "mutual"],
                    help="with --mutual: mutual = one recompute for both settings; fused / separate = a pass per "
                         "setting")
    ap.add_argument("--nonsplit", action="store_true", help="decode workloads: time the non-split forward")
    ap.add_argument("--mutual", action="store_true", help="both settings' gradients (Q1, K1, Q2, K2 all train)")
    ap.add_argument("--split-separate", action="store_true",
                    help="separate path: launch the dQ and the dK kernels one after the other (per-kernel times and "
                         "profiles) instead of as one launch")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--full", action="store_true",
                    help="with --impl reference: each step runs the oracle over the whole workload (every head and "
                         "row), not a sample; about a minute at B2 H32 N4096, several for decode, where drawing "
                         "the 256 heads' inputs dominates")
    ap.add_argument("--heads", type=int, default=0, help="override H (smaller cases for profiling)")
    ap.add_argument("--batch", type=int, default=0, help="override B (smaller cases for profiling)")
    ap.add_argument("--nq", type=int, default=0, help="override N_Q")
    ap.add_argument("--nk", type=int, default=0, help="override N_K")
    ap.add_argument("--causal", type=int, default=-1, choices=[-1, 0, 1], help="override the mask (1 causal, 0 none)")
    ap.add_argument("--no-decode", action="store_true",
                    help="training workloads: skip the Split-K decode section of the JSON line")
    ap.add_argument("--decode-steps", type=int, default=10)
    ap.add_argument("--layout", default="bhnd", choices=["bhnd", "bnhd"],
                    help="storage of Q/K: contiguous [B,H,N,D], or [B,N,H,D] read in place through strides")
    return ap.parse_args()


def pick_workload(synth, args):
    w = synth.WORKLOADS[args.workload]
    over = {k: v for k, v in (("B", args.batch), ("H", args.heads), ("NQ", args.nq), ("NK", args.nk)) if v}
    if args.causal >= 0:
        over["causal"] = bool(args.causal)
    if over:
        tag = ",".join(f"{k}={int(v) if isinstance(v, bool) else v}" for k, v in over.items())
        w = w.with_(name=f"{w.name}[{tag}]", **over)
    return w


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank: float, ms_per_step: float, world: int, unit_scale: float) -> float:
    """Aggregate rate: every rank does `work_per_rank` per step in (max-over-ranks) `ms_per_step`."""
    return world * work_per_rank / (ms_per_step / 1e3) / unit_scale


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(self.FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        smax = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        reasons = sorted({n for r in rows for n, v in zip(names, r[3:]) if v.lower().startswith("active")})
        # "under load": samples taken while the GPU draws well above idle
        loaded = [s for s, p in zip(sm, pw) if p is not None and pw and p > 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


def gpu_id_for(dev_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[dev_index]
        return str(dev_index)


# ----------------------------------------------------------------------------- oracle (CPU) sample

def oracle_sample(w, settings, target_s: float):
    """Times the fp64 oracle's forward + the backward of each setting in `settings` on
    the last R query rows of head (0, 0); a decode workload (no settings) runs all of
    its query rows of that head and is counted in bytes of K1 and K2 read.

    Returns (value in TFLOP/s, or GB/s for decode; seconds, rows, description)."""
    from attention_kl_divergence_streamkl_gb300 import synth
    from oracle import oracle as O
    q1, k1, q2, k2 = (synth.bf16_bits_to_f64(synth.head_slice(w, k, 0, 0)) for k in ("q1", "k1", "q2", "k2"))
    g = synth.upstream_grad(w)[0, 0].astype(np.float64)

    def run(rows):
        t0 = time.perf_counter()
        O.rows_forward(q1, k1, q2, k2, w.softmax_scale, w.causal, rows)
        for setting in settings:
            O.head_backward_rows(setting, q1, k1, q2, k2, w.softmax_scale, w.causal, g, rows)
        return time.perf_counter() - t0

    if not settings:
        rows = np.arange(w.NQ)
        reps = max(1, int(min(target_s, 2.0) / max(run(rows), 1e-6)))
        dt = sum(run(rows) for _ in range(reps))
        nbytes = 2 * w.NK * w.D * 2 + 2 * w.NQ * w.D * 2
        desc = (f"fp64 oracle forward on all {w.NQ} query rows of head (0,0) against its {w.NK} keys, {reps} times "
                f"({nbytes} bytes of K1, K2, Q1 and Q2 in bf16 each, the GPU figure's count for one head)")
        return reps * nbytes / dt / 1e9, dt, w.NQ, desc

    def pairs(rows):
        if not w.causal:
            return rows.size * w.NK
        return int(np.minimum(w.NK, rows + (w.NK - w.NQ) + 1).sum())

    probe = np.arange(max(0, w.NQ - 16), w.NQ)
    dt = run(probe)
    R = int(min(w.NQ, max(16, probe.size * target_s / max(dt, 1e-6))))
    rows = np.arange(w.NQ - R, w.NQ)
    dt = run(rows)
    flops = (4 + 8 * len(settings)) * w.D * pairs(rows)
    which = " + ".join(f"setting-{s}" for s in settings)
    desc = (f"fp64 oracle forward + {which} backward on the last {R} query rows of head (0,0) "
            f"({pairs(rows)} unmasked pairs, {flops:.3e} counted FLOP)")
    return flops / dt / 1e12, dt, R, desc


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_threads():
    """Threads of the BLAS behind numpy (None if it cannot be read)."""
    try:
        import threadpoolctl
        info = [x for x in threadpoolctl.threadpool_info() if x.get("user_api") == "blas"]
        if info:
            return int(info[0]["num_threads"])
    except Exception:
        pass
    import ctypes
    import glob
    libdir = os.path.join(os.path.dirname(os.path.dirname(np.__file__)), "numpy.libs")
    for path in sorted(glob.glob(os.path.join(libdir, "*openblas*.so*"))):
        for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
            try:
                return int(getattr(ctypes.CDLL(path), name)())
            except (OSError, AttributeError):
                continue
    env = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(env) if env and env.isdigit() else None


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from attention_kl_divergence_streamkl_gb300 import synth
    from oracle import oracle as O
    w = pick_workload(synth, args)
    decode = w.name.startswith("decode")
    settings = () if decode else ((1, 2) if args.mutual else (args.setting,))
    G = synth.upstream_grad(w).astype(np.float64)

    def head(b, h):
        return tuple(synth.bf16_bits_to_f64(synth.head_slice(w, k, b, h)) for k in ("q1", "k1", "q2", "k2"))

    def run_head(ins, g, rows):
        """The oracle on `rows` of one head; returns its seconds (input generation not timed)."""
        t = time.perf_counter()
        O.rows_forward(*ins, w.softmax_scale, w.causal, rows)
        for setting in settings:
            O.head_backward_rows(setting, *ins, w.softmax_scale, w.causal, g, rows)
        return time.perf_counter() - t

    if args.full:
        # every head and every query row; one head's inputs are generated at a time
        rows = np.arange(w.NQ)
        heads, pairs = w.B * w.H, w.unmasked_pairs()

        def step():
            return sum(run_head(head(b, h), G[b, h], rows) for b in range(w.B) for h in range(w.H))
        sample = f"fp64 oracle on the whole of {w.name} per step: all {heads} heads, all {w.NQ} query rows"
    else:
        ins, g = head(0, 0), G[0, 0]
        # rows per step: sized so that one step is ~ a couple of seconds of CPU work
        R = 64 if not decode else w.NQ
        rows = np.arange(w.NQ - R, w.NQ)
        heads = 1
        pairs = int(np.minimum(w.NK, rows + (w.NK - w.NQ) + 1).sum()) if w.causal else rows.size * w.NK

        def step():
            return run_head(ins, g, rows)
        sample = f"fp64 oracle on the last {R} query rows of head (0,0) of {w.name} per step ({pairs} pairs)"

    for _ in range(args.warmup):
        step()
    dt = sum(step() for _ in range(args.steps))
    # the whole workload's oracle time at this step's rate (an extrapolation unless --full)
    if decode:
        full_s = dt / args.steps * (w.B * w.H) / heads
    else:
        full_s = dt / args.steps * w.unmasked_pairs() / pairs
    if decode:
        nbytes = heads * (2 * w.NK * w.D * 2 + 2 * w.NQ * w.D * 2)  # the GPU figure's byte count per head
        value = args.steps * nbytes / dt / 1e9
        metric, unit = "attn-KL split-K decode fwd GB/s (B8 H32 N_K=131072 D128)", "GB/s"
    else:
        value = args.steps * (4 + 8 * len(settings)) * w.D * pairs / dt / 1e12
        metric, unit = "attn-KL fwd+bwd TFLOP/s & ms (H32 D128 N64K causal), % bf16 TC peak", "TFLOP/s"
        if args.mutual:
            metric = "attn-KL fwd + both settings' bwd TFLOP/s (mutual case; 20D FLOP per unmasked pair)"
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N_Q": w.NQ, "N_K": w.NK, "D": w.D,
                       "causal": w.causal,
                       "setting": None if decode else ("mutual" if args.mutual else args.setting),
                       "path": ("oracle rows_forward" if decode else "oracle rows_forward + head_backward_rows"),
                       "per_gpu_units": "a bounded sample of the workload per step (see cpu_baseline.sample)",
                       "parallelism": "replicas1"},
            "cpu_baseline": {"value": value, "unit": unit, "cores": cpu_cores(), "blas_threads": blas_threads(),
                             "kind": "oracle", "sample": sample,
                             "full_workload_s": full_s,
                             "full_workload_s_is": "measured" if args.full else "extrapolated from the sample's rate"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- decode section

DECODE_NQ = (1, 4, 16)


def time_decode(args, dev, peaks, peak_src):
    """Split-K and non-split forward on the decode workloads (B8 H32 N_K=131072 D128, N_Q = 1, 4, 16).

    The three workloads share their keys (the same seed and per-head streams),
    and the N_Q = 1 and 4 queries are the first rows of the N_Q = 16 ones, so
    one set of inputs is generated.  K1 + K2 (17.2 GB) is far larger than L2.
    Each variant: W warm-up calls, then `decode_steps` calls timed with CUDA
    events on the launching stream; the clock sampler runs over the section.
    """
    import torch
    import attention_kl_divergence_streamkl_gb300 as skl
    from attention_kl_divergence_streamkl_gb300 import synth

    w16 = synth.WORKLOADS["decode_b8h32_nq16_nk131072_d128"]
    inp = synth.make_inputs(w16)
    dev_t = {k: torch.from_numpy(inp[k].view(np.int16)).view(torch.bfloat16).to(dev) for k in ("q1", "k1", "q2", "k2")}
    del inp
    stream = torch.cuda.current_stream(dev)
    scale = w16.softmax_scale
    out = {}
    sampler = ClockSampler(gpu_id_for(dev.index))
    torch.cuda.synchronize(dev)
    sampler.start()
    for nq in DECODE_NQ:
        q1 = dev_t["q1"][:, :, :nq].contiguous()
        q2 = dev_t["q2"][:, :, :nq].contiguous()
        k1, k2 = dev_t["k1"], dev_t["k2"]
        nbytes = 2 * w16.B * w16.H * w16.NK * w16.D * 2 + 2 * w16.B * w16.H * nq * w16.D * 2
        row = {"workload": f"decode_b8h32_nq{nq}_nk131072_d128", "bytes_per_call": nbytes}
        for name, fn in (("splitk", lambda: skl.fwd_splitk(q1, k1, q2, k2, scale, False)),
                         ("nonsplit", lambda: skl.fwd(q1, k1, q2, k2, scale, False))):
            for _ in range(args.warmup):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(stream)
            for _ in range(args.decode_steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / args.decode_steps
            gbs = nbytes / (ms / 1e3) / 1e9
            row[name] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
        out[str(nq)] = row
    clocks = sampler.stop()
    assert skl.check_device_status(dev) == 0, "device-side timeout in the decode section"
    del dev_t
    torch.cuda.empty_cache()
    return {"metric": "attn-KL split-K decode fwd GB/s (B8 H32 N_K=131072 D128)", "unit": "GB/s",
            "peak": peaks["hbm_gbs"], "peak_source": f"{peak_src} hbm_gbs", "steps": args.decode_steps,
            "warmup": args.warmup, "launches_per_call": {"splitk": 2, "nonsplit": 1}, "nq": out, "clocks": clocks,
            "l2": "inputs larger than L2, no flush between calls"}


# ----------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from attention_kl_divergence_streamkl_gb300 import build as B
    B.build()
    import attention_kl_divergence_streamkl_gb300 as skl
    from attention_kl_divergence_streamkl_gb300 import synth

    w = pick_workload(synth, args)
    decode = w.name.startswith("decode")
    mode = {"auto": skl.BWD_AUTO, "fused": skl.BWD_FUSED, "separate": skl.BWD_SEPARATE,
            "mutual": "mutual"}[args.bwd_mode]
    if mode == "mutual" and not args.mutual:
        raise SystemExit("--bwd-mode mutual needs --mutual")
    if args.mutual and not decode and mode == skl.BWD_AUTO:
        props = torch.cuda.get_device_properties(dev)
        pick = skl.bwd_mutual_select(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size, props.multi_processor_count,
                                     w.causal)
        mode = "mutual" if pick == skl.BWD_SEPARATE else skl.BWD_FUSED
    elif not decode and mode == skl.BWD_AUTO:
        props = torch.cuda.get_device_properties(dev)
        mode = skl.bwd_select(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size, props.multi_processor_count,
                              w.causal)
    inp = synth.make_inputs(w)
    host = [torch.from_numpy(inp[k].view(np.int16)).view(torch.bfloat16) for k in ("q1", "k1", "q2", "k2")]
    if args.layout == "bnhd":  # same values stored [B, N, H, D], viewed as [B, H, N, D]
        host = [t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in host]
    host_g = torch.from_numpy(inp["g"])

    def like(t, pinned=False):
        """An empty tensor with t's shape and storage order."""
        perm = (0, 2, 1, 3) if args.layout == "bnhd" else (0, 1, 2, 3)
        shp = tuple(t.shape[i] for i in perm)
        e = torch.empty(shp, dtype=t.dtype, pin_memory=True) if pinned else torch.empty(shp, dtype=t.dtype, device=dev)
        return e.permute(*perm)

    q1, k1, q2, k2 = (like(t).copy_(t) for t in host)
    g = host_g.to(dev)
    scale, causal = w.softmax_scale, w.causal
    pairs = w.unmasked_pairs()
    stream = torch.cuda.current_stream(dev)

    # ---- one step, with an event between kernels so each is timed on its stream
    def step(qs, ev=None, gq=None):
        a, b, c, d = qs
        g_ = g if gq is None else gq
        if decode:
            out = skl.fwd(a, b, c, d, scale, causal) if args.nonsplit else skl.fwd_splitk(a, b, c, d, scale, causal)
            if ev:
                ev[1].record(stream)
            return out
        kl, l1, l2 = skl.fwd(a, b, c, d, scale, causal)
        if ev:
            ev[1].record(stream)
        if args.mutual:
            if mode == "mutual":
                grads = skl.bwd_mutual(a, b, c, d, l1, l2, kl, g_, scale, causal, skl.BWD_SEPARATE)
                if ev:
                    ev[2].record(stream)
            else:
                grads = skl.bwd_s1(a, b, c, d, l1, l2, g_, scale, causal, mode)
                if ev:
                    ev[2].record(stream)
                grads = grads + skl.bwd_s2(a, b, c, d, l1, l2, kl, g_, scale, causal, mode)
            if ev:
                ev[3].record(stream)
            return (kl,) + tuple(grads)
        bwd = skl.bwd_s1 if args.setting == 1 else skl.bwd_s2
        extra = () if args.setting == 1 else (kl,)
        if mode == skl.BWD_SEPARATE and args.split_separate:
            dq = bwd(a, b, c, d, l1, l2, *extra, g_, scale, causal, skl.BWD_DQ_ONLY)[0]
            if ev:
                ev[2].record(stream)
            dk = bwd(a, b, c, d, l1, l2, *extra, g_, scale, causal, skl.BWD_DK_ONLY)[1]
        else:
            dq, dk = bwd(a, b, c, d, l1, l2, *extra, g_, scale, causal, mode)
            if ev:
                ev[2].record(stream)
        if ev:
            ev[3].record(stream)
        return kl, dq, dk

    key_ranges = None
    if decode:
        kernels = ["fwd" if args.nonsplit else "splitk"]
        algo = {kernels[0]: 4 * w.D * pairs}
        launches_per_step = 1 if args.nonsplit else 2
    elif mode == "mutual":
        kernels = ["fwd", "bwd_mutual", "none"]
        algo = {"fwd": 4 * w.D * pairs, "bwd_mutual": 16 * w.D * pairs}
        launches_per_step = 3
    elif args.mutual:
        tag = "fused" if mode == skl.BWD_FUSED else "separate"
        kernels = ["fwd", f"bwd_s1_{tag}", f"bwd_s2_{tag}"]
        algo = {"fwd": 4 * w.D * pairs, kernels[1]: 8 * w.D * pairs, kernels[2]: 8 * w.D * pairs}
        props = torch.cuda.get_device_properties(dev)
        key_ranges = skl.bwd_fused_plan(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size,
                                        props.multi_processor_count, w.causal)[0]
        if mode == skl.BWD_FUSED:
            launches_per_step = 1 + 2 * (2 * key_ranges + (1 if key_ranges > 1 else 0))
        else:
            key_ranges = None
            launches_per_step = 5
    elif mode == skl.BWD_SEPARATE and args.split_separate:
        kernels = ["fwd", "bwd_dq", "bwd_dk"]
        algo = {"fwd": 4 * w.D * pairs, "bwd_dq": 6 * w.D * pairs, "bwd_dk": 6 * w.D * pairs}
        launches_per_step = 3
    elif mode == skl.BWD_SEPARATE:
        kernels = ["fwd", "bwd_separate", "none"]
        algo = {"fwd": 4 * w.D * pairs, "bwd_separate": 12 * w.D * pairs}
        launches_per_step = 2
    else:
        kernels = ["fwd", "bwd_fused", "none"]
        algo = {"fwd": 4 * w.D * pairs, "bwd_fused": 8 * w.D * pairs}
        props = torch.cuda.get_device_properties(dev)
        key_ranges = skl.bwd_fused_plan(w.B, w.H, w.NQ, w.NK, w.D, props.L2_cache_size,
                                        props.multi_processor_count, w.causal)[0]
        # fwd; per key range the fused kernel and the dK conversion; the dQ conversion with several ranges
        launches_per_step = 1 + 2 * key_ranges + (1 if key_ranges > 1 else 0)

    for _ in range(args.warmup):
        step((q1, k1, q2, k2))
    torch.cuda.synchronize(dev)
    assert skl.check_device_status(dev) == 0, "device-side timeout during warm-up"

    # ---- extra HBM of one step (outside the timed region): the allocator's peak during the step minus what was
    # allocated before it (the inputs) and minus the step's outputs (KL, LSE1, LSE2 and the gradients)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    before = torch.cuda.memory_allocated(dev)
    outs = step((q1, k1, q2, k2))
    torch.cuda.synchronize(dev)
    peak = torch.cuda.max_memory_allocated(dev)
    rows = w.B * w.H * w.NQ * 4
    # a decode step returns KL, LSE1, LSE2; a training step KL and the gradients (its LSE1, LSE2 are outputs of
    # the forward too, freed when the step returns)
    out_bytes = sum(t.numel() * t.element_size() for t in outs if t is not None) + (0 if decode else 2 * rows)
    extra_bytes = max(0, peak - before - out_bytes)
    del outs
    p_bytes = 2 * w.unmasked_pairs() * 2 if not decode else 2 * w.B * w.H * w.NQ * w.NK * 2
    extra_hbm = {"bytes": int(extra_bytes), "peak_bytes": int(peak), "inputs_bytes": int(before),
                 "outputs_bytes": int(out_bytes), "materialised_p1_p2_bf16_bytes": int(p_bytes),
                 "materialised_over_extra": (p_bytes / extra_bytes) if extra_bytes else None,
                 "note": "the fused backward's fp32 dK accumulator (and, over key ranges, the fp32 dQ sum) is the "
                         "workspace; a path that materialises P1 and P2 holds at least the bf16 bytes given"}

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for(local))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    t_start.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        step((q1, k1, q2, k2), evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_kernel = {k: 0.0 for k in kernels}
    for e in evs:
        per_kernel[kernels[0]] += e[0].elapsed_time(e[1])
        if len(kernels) > 1:
            per_kernel[kernels[1]] += e[1].elapsed_time(e[2])
            per_kernel[kernels[2]] += e[2].elapsed_time(e[3])
    per_kernel.pop("none", None)
    status = skl.check_device_status(dev)
    assert status == 0, f"device-side timeout in the timed region (status {status})"

    elapsed_ms = max_over_ranks(elapsed_ms, dev)

    peaks, peak_src = load_peaks()
    ms_step = elapsed_ms / args.steps
    if decode:
        bytes_step = 2 * w.B * w.H * w.NK * w.D * 2 + 2 * w.B * w.H * w.NQ * w.D * 2
        value = whole_job_rate(bytes_step, ms_step, world, 1e9)
        metric, unit = "attn-KL split-K decode fwd GB/s (B8 H32 N_K=131072 D128)", "GB/s"
        dom = kernels[0]
        achieved = bytes_step / (per_kernel[dom] / args.steps / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "kernel": dom,
                "traffic": NCU_TRAFFIC_RATIO[dom] * bytes_step if dom in NCU_TRAFFIC_RATIO else None,
                "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": bytes_step}
    else:
        flops_step = (20 if args.mutual else 12) * w.D * pairs
        value = whole_job_rate(flops_step, ms_step, world, 1e12)
        metric, unit = "attn-KL fwd+bwd TFLOP/s & ms (H32 D128 N64K causal), % bf16 TC peak", "TFLOP/s"
        if args.mutual:
            metric = "attn-KL fwd + both settings' bwd TFLOP/s (mutual case; 20D FLOP per unmasked pair)"
        dom = max(per_kernel, key=per_kernel.get)
        avg_ms = per_kernel[dom] / args.steps
        achieved = algo[dom] / (avg_ms / 1e3) / 1e12
        peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": NCU_TRAFFIC_PER_PAIR[dom] * pairs if dom in NCU_TRAFFIC_PER_PAIR else None, "kernel": dom,
                "peak_source": f"{peak_src} bf16_tflops_sustained (kernel timed inside a long step)",
                "algorithmic_flops_per_launch": algo[dom],
                "frac_of_burst_peak_whole_step": value / world / peaks["bf16_tflops"]}

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        pinned = [like(t, pinned=True).copy_(t) for t in host]
        pg = host_g.pin_memory()
        out_host = torch.empty((w.B, w.H, w.NQ), dtype=torch.float32).pin_memory()
        # Inputs stream in as in a training loop: a copy stream fills one of two device
        # input sets while the compute stream works on the other.  Every step's
        # host->device copy and its result's read-back lie inside the timed region.
        copy_stream = torch.cuda.Stream(dev)
        bufs = [[like(t) for t in pinned] for _ in range(2)]
        gbufs = [torch.empty_like(pg, device=dev) for _ in range(2)]
        ready = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]

        def load(k):
            b = k % 2
            if k >= 2:
                copy_stream.wait_event(freed[b])  # step k - 2 is done with this set
            with torch.cuda.stream(copy_stream):
                for dst, src in zip(bufs[b], pinned):
                    dst.copy_(src, non_blocking=True)
                if not decode:
                    gbufs[b].copy_(pg, non_blocking=True)  # the upstream gradient is a host input too
            ready[b].record(copy_stream)

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        copy_stream.wait_event(e0)
        load(0)
        for k in range(args.steps):
            b = k % 2
            if k + 1 < args.steps:
                load(k + 1)
            stream.wait_event(ready[b])
            kl = step(bufs[b], gq=gbufs[b])[0]
            out_host.copy_(kl, non_blocking=True)
            freed[b].record(stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / args.steps
        h2d = sum(t.numel() * t.element_size() for t in pinned) + (0 if decode else pg.numel() * 4)
        d2h = out_host.numel() * 4
        work = (bytes_step if decode else flops_step)
        e2e = {"value": world * work / (e2e_ms / 1e3) / (1e9 if decode else 1e12), "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        settings = () if decode else ((1, 2) if args.mutual else (args.setting,))
        v, dt, R, desc = oracle_sample(w, settings, args.cpu_seconds)
        cpu = {"value": v, "unit": unit, "cores": cpu_cores(), "blas_threads": blas_threads(), "kind": "oracle",
               "sample": desc, "seconds": dt}

    decode_section = None
    if not decode and not args.no_decode and not args.mutual and args.workload == "kl_b1h32_n65536_d128_causal" and not (
            args.heads or args.batch or args.nq or args.nk or args.causal >= 0):
        del q1, k1, q2, k2
        torch.cuda.empty_cache()
        decode_section = time_decode(args, dev, peaks, peak_src)

    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N_Q": w.NQ, "N_K": w.NK, "D": w.D,
                       "causal": w.causal, "setting": args.setting if not decode else None,
                       "layout": args.layout,
                       "bwd_path": None if decode else {1: "fused", 2: "separate", "mutual": "mutual"}[mode],
                       "bwd_key_ranges": key_ranges,
                       "path": ("nonsplit" if args.nonsplit else "splitk") if decode else "fwd+bwd",
                       "per_gpu_units": "the whole workload on every rank (independent heads)",
                       "l2": "inputs larger than L2, no flush between steps",
                       "parallelism": f"replicas{world}"},
            "roofline": roof, "per_kernel_ms": {k: v / args.steps for k, v in per_kernel.items()},
            "extra_hbm": extra_hbm,
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu}
    if decode_section is not None:
        line["decode"] = decode_section
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
