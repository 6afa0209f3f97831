"""Benchmark of the Mamba-2 SSD layer (ssd_fwd + ssd_bwd) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-cpu-baseline]

A step is one pass of the whole layer -- ssd_fwd then ssd_bwd through the C
ABI -- over one batch of the workload, inputs resident in HBM.  L2 is flushed
(a 256 MB write) between steps, outside the timed events; each step is timed
with CUDA events on the launching stream.  Under torchrun every rank runs its
own copy of the workload (independent problems, no collective): weak scaling,
``value`` = tokens of all ranks / max over ranks of the timed region.

``--impl reference`` times the float64 CPU oracle instead (rank 0 only), each
step a bounded prefix of the same workload.

``--op gated_rmsnorm`` measures the Mamba-2 block's gated RMSNorm instead
(forward + backward through the C ABI) on the norm that follows the
workload's scan: rows = tokens, dim = nheads * headdim, group = dim / ngroups.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
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

METRIC = "SSD layer fwd+bwd tokens/s (ms) at b2·L8192 bf16; % of HBM / tensor roofline"
DEFAULT_WORKLOAD = "b2_L8192_bf16"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
CSRC_DIR = os.path.join(ROOT, "mamba_selective_state_gb300", "csrc")
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)


# ----------------------------------------------------------------------------
# algorithmic bytes and flops per launch: the compulsory reads and writes of
# each kernel (per-unit figures times the units of one launch)
# ----------------------------------------------------------------------------
def eval_chunk(cfg, dtype_bytes):
    """Chunk length the library evaluates: the tensor-core path (bf16,
    headdim 64, d_state >= 16, at most 256 heads per group) uses 128-token
    chunks whatever the problem's chunk_size; otherwise chunk_size."""
    tc = (dtype_bytes == 2 and cfg["headdim"] == 64 and cfg["dstate"] >= 16
          and cfg["nheads"] // cfg["ngroups"] <= 256)
    return 128 if tc else cfg["chunk"]


def kernel_model(cfg, dtype_bytes, keep=False):
    b, L, H, P, N, G = (cfg[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate",
                                          "ngroups"))
    Q = eval_chunk(cfg, dtype_bytes)
    nc = -(-L // Q)
    Lp = nc * Q
    s = dtype_bytes
    T = b * L
    tokx = T * H * P * s          # one (b,L,H,P) tensor in dtype
    tokbc = T * G * N * s         # one (b,L,G,N) tensor in dtype
    st32 = b * H * nc * P * N * 4  # chunk states / dHloc (fp32)
    stS = b * H * nc * P * N * s   # carry-in states / dS (dtype)
    per_tok = b * H * Lp * 4      # one fp32 per-token-per-head vector
    units = b * H * nc            # (row, head, chunk) tiles
    gunits = b * G * nc           # (row, group, chunk) tiles
    m = {}
    m["dt_cumsum"] = dict(bytes=T * H * s + 2 * per_tok, flops=0)
    m["chunk_state"] = dict(bytes=tokx + tokbc + 2 * per_tok + st32, flops=2 * units * Q * P * N)
    m["state_passing_fwd"] = dict(bytes=st32 + stS, flops=2 * units * P * N)
    # a forward that keeps its intermediates, or the backward's recompute,
    # also keeps the fp32 carry-in states (in place over the chunk states)
    m["state_passing_fwd_keep"] = dict(bytes=2 * st32 + stS, flops=2 * units * P * N)
    # chunk_scan: per (group, chunk) C B^T (at chunk 128 also C_rev B^T, the
    # copy with its row blocks reversed that balances the mask pass); per head
    # Y1 = A_hat X and Y2 = C H_in^T
    scan_cb = (4 if Q == 128 else 2) * Q * Q * N
    scan_head = 2 * Q * Q * P + 2 * Q * N * P
    m["chunk_scan"] = dict(bytes=2 * tokx + 2 * tokbc + stS + 2 * per_tok,
                           flops=gunits * scan_cb + units * scan_head)
    m["chunk_dstate"] = dict(bytes=tokx + tokbc + per_tok + st32, flops=2 * units * Q * P * N)
    # reads dHloc and the fp32 carry-in states (for dL/da_c), writes dS
    m["state_passing_bwd"] = dict(bytes=2 * st32 + stS, flops=4 * units * P * N)
    # Backward flops are counted from the matrix products each kernel issues
    # (2 flops per multiply-add, dense tiles): the token kernel forms C B^T
    # once per group and, per head, dM = dy x^T, dX_s = B dS^T,
    # Y_c = C H_in^T and dX = M^T dY; the dB/dC kernel, per head, dM again,
    # dC += dy H, dB += x dS; once per group on the heads' summed dCB, S B and S^T C.
    bwd_tok_flops = gunits * 2 * Q * Q * N + units * (4 * Q * Q * P + 4 * Q * P * N)
    bwd_dbc_flops = units * (2 * Q * Q * P + 4 * Q * N * P) + gunits * 4 * Q * Q * N
    # per-head token gradients (dx, ddt_eff, dl): x, dy, B, C, dS, H_in in; dx out
    m["chunk_bwd"] = dict(bytes=3 * tokx + 2 * tokbc + 2 * stS + 4 * per_tok, flops=bwd_tok_flops)
    # group gradients dB, dC: x, dy, B, C, dS, H_in, l, dt_eff in; dB, dC out;
    # and the per-token ddt: dt, dL/dl, ddt_eff in, ddt out
    m["chunk_bwd_dbc"] = dict(bytes=2 * tokx + 4 * tokbc + 2 * stS + 4 * per_tok + 2 * T * H * s,
                              flops=bwd_dbc_flops)
    m["dt_bwd"] = dict(bytes=2 * T * H * s + 4 * per_tok, flops=0)
    # the backward's state chains, one pass each: forward reads x, B, l, dt_eff
    # and writes the bf16 carry-in states; reverse reads dy, C, l and the
    # carry-in states and writes dS (M = 128 rows issued per product)
    m["state_chain_fwd"] = dict(bytes=tokx + tokbc + 2 * per_tok + stS,
                                flops=units * 2 * 128 * P * Q)
    m["state_chain_bwd"] = dict(bytes=tokx + tokbc + per_tok + 2 * stS,
                                flops=units * (2 * 128 * P * Q + 2 * P * N))
    # single-pass forward: reads x, dt, B, C (and the initial states), writes
    # y and the final states; per (row, head, 128-token chunk) it issues C B^T,
    # Y2 = C H_in^T, S^T = B^T (w.X) (M = 128 rows issued) and Y1 = A_hat X
    nq = -(-L // 128)
    fq = 2 * 128 * 128 * N + 2 * 128 * P * N + 2 * 128 * P * 128 + 2 * 128 * 128 * P
    # (keeping its intermediates for the backward it also writes the carry-in
    # states, dt_eff, the chunk cumsums and the per-chunk decays)
    kept = stS + 2 * per_tok + b * H * nc * 4 if keep else 0
    m["ssd_fwd_fused"] = dict(bytes=2 * tokx + T * H * s + 2 * tokbc + 2 * b * H * P * N * 4 + kept,
                              flops=b * H * nq * fq)
    m["param_reduce"] = dict(bytes=b * nc * H * 4 * 4, flops=0)
    m["status_reset"] = dict(bytes=4, flops=0)
    # a kept backward on the separate kernels zeroes the reverse scan's flags
    # (one per (row, head, 512-element block, scan segment))
    nflags = b * H * -(-(P * N) // 512) * max(-(-nc // 16), -(-nc // 8))
    m["kept_scan_reset"] = dict(bytes=4 * nflags + 4, flops=0)
    # compulsory IO of the layer (fwd reads x dt B C, writes y; bwd reads x dt
    # B C dy, writes dx ddt dB dC)
    layer_io = (tokx + T * H * s + 2 * tokbc + tokx) + (2 * tokx + T * H * s + 2 * tokbc
                                                        + tokx + T * H * s + 2 * tokbc)
    return m, layer_io


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of a b2_L8192_bf16 step as the bench runs it (the forward
# keeping its intermediates; the committed launch-list summary of that
# workload), keyed by kernel, with the sha1 of the sources the kernel was built from: the
# figure is reported only while those sources are unchanged and the workload
# is the one captured, else null.
NCU_TRAFFIC_WORKLOAD = "b2_L8192_bf16"
NCU_TRAFFIC = {
    "ssd_fwd_fused": (('k_ssd_fwd_fused.cu', 'tc_common.cuh', 'ssd_internal.cuh'), 4.2920e+08, "e7466ed302e73f4bef870b5dc3def204965de329"),
    "state_chain_bwd": (('k_state_chain.cu', 'tc_common.cuh', 'ssd_internal.cuh'), 4.1255e+08, "22731e6f826befc3796e68e18ad666a48df40a29"),
    "chunk_bwd_tc": (('k_chunk_bwd_tok_tc.cu', 'tc_common.cuh', 'ssd_internal.cuh'), 7.4205e+08, "c2a97b3e80190f9c280635e1ce909908fa87c8b8"),
    "chunk_bwd_dbc_tc": (('k_chunk_bwd_group_tc.cu', 'tc_common.cuh', 'ssd_internal.cuh'), 6.9040e+08, "fa041e274942dd2af296ed376774e190f5ad315a"),
}


def ncu_traffic(kname, workload):
    ent = NCU_TRAFFIC.get(kname)
    if ent is None or workload != NCU_TRAFFIC_WORKLOAD:
        return None
    files, nbytes, sha = ent
    h = hashlib.sha1()
    for fn in files:
        with open(os.path.join(CSRC_DIR, fn), "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest() == sha else None


def base_name(kname):
    for suf in ("_simt", "_tc"):
        if kname.endswith(suf):
            return kname[: -len(suf)]
    return kname


def layer_summary(kernels, model, steps, ms_per_step, layer_io, hbm_peak, tc_peak):
    """The whole layer against both roofs: its compulsory IO bytes per step
    over the step time against HBM, and the matrix-product flops of all its
    launches in a step (the kernel model's flops times launches per step)
    against the dense bf16 tensor peak."""
    flops = sum(model[base_name(k)]["flops"] * v["launches"] / steps
                for k, v in kernels.items() if base_name(k) in model)
    sec = ms_per_step / 1e3
    return {"compulsory_io_bytes": layer_io,
            "achieved_GBps": layer_io / sec / 1e9,
            "frac_of_hbm": layer_io / sec / 1e9 / hbm_peak,
            "flops_per_step": flops,
            "achieved_TFLOPps": flops / sec / 1e12,
            "frac_of_tensor": flops / sec / 1e12 / tc_peak}


def load_peaks():
    try:
        with open(PEAKS_PATH) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle timing (the baseline and the reference arm)
# ----------------------------------------------------------------------------
class OracleSample:
    """Bounded prefix sample of a workload for the oracle, calibrated so that
    one fwd+bwd takes about ``target_s`` seconds."""

    def __init__(self, name, target_s):
        from mamba_selective_state_gb300.inputs import make_workload
        from oracle import ssd_ref
        self.name = name
        self.full = make_workload(name, seed=0, dfinal=False)
        self.f = {n: self.full.f64(n) for n in ["x", "dt", "dt_bias", "A", "B", "C", "D", "dy",
                                                 "initial_states", "seq_idx"]}
        ssd_ref.build_oracle()
        probe = max(16, min(self.full.seqlen, 64))
        t = self.run(probe)[0]
        per_tok = max(t / probe, 1e-7)
        self.Lp = int(max(16, min(self.full.seqlen, target_s / per_tok)))

    def run(self, Lp):
        from oracle import ssd_ref
        cut = lambda a: None if a is None else a[:, :Lp]  # noqa: E731
        a = dict(self.f)
        for n in ("x", "dt", "B", "C", "dy", "seq_idx"):
            a[n] = cut(a[n])
        args = [a[n] for n in ["x", "dt", "dt_bias", "A", "B", "C", "D"]]
        kw = dict(initial_states=a["initial_states"], seq_idx=a["seq_idx"])
        t0 = time.perf_counter()
        ssd_ref.ssd_fwd(*args, **kw)
        th_f = ssd_ref.last_threads()
        ssd_ref.ssd_bwd(*args, a["dy"], **kw)
        th_b = ssd_ref.last_threads()
        return time.perf_counter() - t0, max(th_f, th_b)

    def describe(self):
        return (f"float64 oracle fwd+bwd on the first {self.Lp} of {self.full.seqlen} tokens of "
                f"every row ({self.full.batch} rows, all {self.full.nheads} heads) of {self.name}")


def cpu_baseline(name, target_s=15.0, min_s=10.0, single_core_s=4.0, parity_of=None):
    """The oracle on a bounded sample of the workload: a prefix sized to about
    target_s seconds, repeated (whole workload too small) until at least
    min_s seconds of CPU work have been timed, on every host core; then a
    shorter prefix on one core (``single_core``).  With ``parity_of`` =
    (inputs, device buffers) the same leg also checks the benched step's
    outputs against the oracle (``parity``, see oracle_parity)."""
    from oracle import ssd_ref
    smp = OracleSample(name, target_s)
    secs, threads, reps = 0.0, 1, 0
    while reps == 0 or (secs < min_s and reps < 20):
        t, threads = smp.run(smp.Lp)
        secs += t
        reps += 1
    tok = smp.full.batch * smp.Lp * reps
    sample = smp.describe() + (f", run {reps} times" if reps > 1 else "")
    out = {"value": tok / secs, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": sample, "seconds": secs}
    # one core: a prefix sized from the all-core rate to about single_core_s
    per_tok_1 = secs / tok * threads
    lp1 = int(max(1, min(smp.full.seqlen, single_core_s / max(per_tok_1 * smp.full.batch, 1e-9))))
    ssd_ref.set_threads(1)
    try:
        t1, th1 = smp.run(lp1)
    finally:
        ssd_ref.set_threads(0)
    out["single_core"] = {"value": smp.full.batch * lp1 / t1, "unit": "tokens/s", "cores": th1,
                          "seconds": t1,
                          "sample": f"the first {lp1} tokens of every row, same workload"}
    if parity_of is not None:
        out["parity"] = oracle_parity(*parity_of)
    return out


def run_reference(args, world, rank):
    if rank != 0:
        return
    total_budget = 150.0
    per_step = max(0.2, min(10.0, total_budget / max(1, args.steps + args.warmup)))
    smp = OracleSample(args.workload, per_step)
    for _ in range(args.warmup):
        smp.run(smp.Lp)
    times, threads = [], 1
    for _ in range(args.steps):
        t, threads = smp.run(smp.Lp)
        times.append(t)
    tot = sum(times)
    tok = smp.full.batch * smp.Lp * len(times)
    value = tok / tot
    cfg = workload_config(args.workload)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": smp.describe()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(name):
    from mamba_selective_state_gb300.inputs import WORKLOADS
    cfg = dict(WORKLOADS[name])
    out = {"workload": name}
    out.update({k: v for k, v in cfg.items() if k != "dtype"})
    return out


def step_flags(args):
    """Flags of the benchmarked step: its forward keeps the intermediates the
    backward would recompute, and the backward takes them (the usual
    training step); --recompute benchmarks the stateless backward."""
    from mamba_selective_state_gb300 import _lib
    flags = 0 if args.recompute else _lib.SSD_KEEP_FWD_STATES
    if getattr(args, "scan", "sequential") == "warp_shuffle":
        flags |= _lib.SSD_SCAN_WARP_SHUFFLE
    return flags


# ----------------------------------------------------------------------------
def run_gpu(args, world, rank, local):
    import torch
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.inputs import make_workload
    from mamba_selective_state_gb300.runner import SSDDevice

    inp = make_workload(args.workload, seed=rank, dfinal=False)
    dev = SSDDevice(inp, device=f"cuda:{local}", extra_flags=step_flags(args))
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev.device)

    def step(mid=None):
        dev.fwd(stream=stream)
        if mid is not None:
            mid.record(stream)
        dev.bwd(stream=stream)

    # one checked step first: the backward's first kernel resets the status
    # word, so the forward's own status is read before it runs
    dev.fwd(stream=stream)
    if dev.device_status(stream) != 0:
        raise RuntimeError("device status word reports an error after the forward")
    dev.bwd(stream=stream)
    if dev.device_status(stream) != 0:
        raise RuntimeError("device status word reports an error after the backward")
    w0 = torch.cuda.Event(enable_timing=True)
    w1 = torch.cuda.Event(enable_timing=True)
    for k in range(args.warmup):
        if k == args.warmup - 1:
            flush.fill_(0.0)
            w0.record(stream)
        step()
    w1.record(stream)
    torch.cuda.synchronize()
    if dev.device_status(stream) != 0:
        raise RuntimeError("device status word reports an error after warm-up")
    # the timed region runs at least --steps steps and at least MIN_TIMED_S
    # seconds, so that the clock record under load has enough samples
    est_ms = max(w0.elapsed_time(w1), 1e-3)
    nsteps = max(args.steps, int(args.min_timed_s * 1e3 / est_ms) + 1)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(nsteps)]
    clocks = ClockSampler(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    # the timed region: nothing between the kernels of a step (no per-kernel
    # events, no event between forward and backward)
    t_wall0 = time.perf_counter()
    for i in range(nsteps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier(world)
    clk = clocks.stop() if clocks else None
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    tot_ms = sum(step_ms)
    # per-kernel means and the forward/backward split: a second pass over
    # the same steps with the library's per-kernel events (and an event
    # between forward and backward), after the timed region
    nprof = min(nsteps, PROFILED_STEPS)
    pstarts = [torch.cuda.Event(enable_timing=True) for _ in range(nprof)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(nprof)]
    pends = [torch.cuda.Event(enable_timing=True) for _ in range(nprof)]
    _lib.profile_start()
    for i in range(nprof):
        flush.fill_(float(i))
        pstarts[i].record(stream)
        step(mids[i])
        pends[i].record(stream)
    torch.cuda.synchronize()
    prof = _lib.profile_stop()
    fwd_ms = [s.elapsed_time(m) for s, m in zip(pstarts, mids)]
    pstep_ms = [s.elapsed_time(e) for s, e in zip(pstarts, pends)]
    tot_ms_max = max_over_ranks(world, tot_ms)
    if dev.device_status(stream) != 0:
        raise RuntimeError("device status word reports an error in the timed region")

    tokens = inp.batch * inp.seqlen
    value = world * tokens * nsteps / (tot_ms_max / 1e3)

    # ---- end to end: pinned host inputs -> device, fwd+bwd, results -> host
    e2e = run_e2e(inp, dev, args, stream)

    # ---- roofline of the dominant kernel
    peaks, src = load_peaks()
    cfg = workload_config(args.workload)
    s_bytes = 2 if inp.dtype == "bf16" else 4
    model, layer_io = kernel_model(dict(cfg, batch=inp.batch, seqlen=inp.seqlen), s_bytes,
                                   keep=not args.recompute)
    kernels = {k: {"launches": n, "ms_per_launch": ms / n} for k, (n, ms) in prof.items()
               if not k.startswith("_")}
    # the library's kernels launched in the timed region (per step as counted
    # in the profiled pass, times the timed steps)
    launches = sum(v["launches"] for v in kernels.values()) // nprof * nsteps
    dom = max(kernels, key=lambda k: kernels[k]["launches"] * kernels[k]["ms_per_launch"])
    dm = model[base_name(dom)]
    dur_s = kernels[dom]["ms_per_launch"] / 1e3
    hbm_peak = peaks["hbm_gbs"]
    tc_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    ach_gbs = dm["bytes"] / dur_s / 1e9
    ach_tfs = dm["flops"] / dur_s / 1e12
    if dom.endswith("_simt") and dm["flops"] > 0:
        # FP32 FMA on the CUDA cores: 152 SMs x 128 lanes x 2 flop x max SM clock
        alu_peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": ach_tfs, "peak": alu_peak, "unit": "TFLOP/s",
                "frac": ach_tfs / alu_peak, "traffic": None, "kernel": dom,
                "peak_source": "derived: 152 SM x 128 FP32 lanes x 2 x max SM clock"}
    elif dm["flops"] and dm["flops"] / dm["bytes"] > tc_peak * 1e12 / (hbm_peak * 1e9):
        roof = {"bound": "tensor", "achieved": ach_tfs, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": ach_tfs / tc_peak, "traffic": None, "kernel": dom,
                "peak_source": f"{src} bf16_tflops_sustained"}
    else:
        roof = {"bound": "hbm", "achieved": ach_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": ach_gbs / hbm_peak, "traffic": None, "kernel": dom,
                "peak_source": f"{src} hbm_gbs"}
    roof["traffic"] = ncu_traffic(dom, args.workload)
    roof["algorithmic_bytes"] = dm["bytes"]
    roof["algorithmic_flops"] = dm["flops"]
    roof["ms_per_launch"] = kernels[dom]["ms_per_launch"]
    for k, v in kernels.items():
        mk = model.get(base_name(k))
        if mk:
            d = v["ms_per_launch"] / 1e3
            v["GBps"] = mk["bytes"] / d / 1e9
            v["TFLOPps"] = mk["flops"] / d / 1e12
    ms_per_step = tot_ms_max / nsteps
    layer = layer_summary(kernels, model, nprof, ms_per_step, layer_io, hbm_peak, tc_peak)
    layer.update(fwd_ms_mean=statistics.mean(fwd_ms),
                 bwd_ms_mean=statistics.mean(t - f for t, f in zip(pstep_ms, fwd_ms)),
                 step_ms_median=statistics.median(step_ms),
                 split_and_kernels=f"from a second, profiled pass of {nprof} steps "
                                   f"({statistics.mean(pstep_ms):.4f} ms per step with the "
                                   "per-kernel events)")

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": nsteps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": inp.dtype, "data": "synthetic",
            "config": dict(cfg, l2="flushed between steps (256 MB write, outside the events); "
                                   "inputs larger than L2", parallelism="replicas" if world > 1
                           else "single GPU",
                           fwd_intermediates="recomputed by the backward" if args.recompute else
                           "kept by the forward for the backward (SSD_KEEP_FWD_STATES)",
                           **({"scan": "warp_shuffle (SSD_SCAN_WARP_SHUFFLE)"}
                              if args.scan == "warp_shuffle" else {})),
            "roofline": roof, "layer_roofline": layer, "e2e": e2e,
            "gpu_launches": launches, "kernels": kernels, "clocks": clk,
            "wall_s_timed": t_wall,
            "timed_region": f"{nsteps} steps (at least --steps {args.steps} and at least "
                            f"{args.min_timed_s} s of step time), no events between a step's "
                            "kernels; per-kernel figures from a profiled pass after it"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline(args.workload, parity_of=(inp, dev))
        line["parity"] = base.pop("parity")
        line["cpu_baseline"] = base
    return line


def oracle_parity(inp, dev):
    """Part of the oracle leg, after the timed region: the benched step's
    outputs (the device buffers hold the last step's results) against the
    float64 oracle on one sampled group of the same inputs -- every batch row,
    the group's heads, every token -- as max|diff| / max|ref| per tensor."""
    import numpy as np
    from oracle import ssd_ref
    g = int(np.random.default_rng(0).integers(inp.ngroups))
    hpg = inp.nheads // inp.ngroups
    hs = slice(g * hpg, (g + 1) * hpg)
    f = inp.f64
    t0 = time.perf_counter()
    init = f("initial_states")
    ref = ssd_ref.ssd_group(*[f(n) for n in ["x", "dt", "dt_bias", "A", "B", "C", "D"]],
                            f("dy"), g, inp.ngroups, initial_states=init,
                            seq_idx=f("seq_idx"), dfinal_states=None,
                            want_dinit=init is not None)
    secs = time.perf_counter() - t0
    got = dev.results()
    errs = {}
    for k, r in ref.items():
        v = got[k].numpy()
        if k in ("y", "dx", "ddt"):
            v = v[:, :, hs]
        elif k in ("final_states", "dinitial_states"):
            v = v[:, hs]
        elif k in ("dA", "dD", "ddt_bias"):
            v = v[hs]
        else:
            v = v[:, :, g:g + 1]
        errs[k] = float(np.abs(v - r).max() / max(np.abs(r).max(), 1e-30))
    tol = 2e-2 if inp.dtype == "bf16" else 1e-4
    return {"metric": "max|diff| / max|ref| per tensor", "tolerance": tol,
            "group": g, "heads": [hs.start, hs.stop], "rel_err": errs,
            "pass": all(e <= tol for e in errs.values()), "oracle_seconds": secs,
            "sample": f"group {g} of {inp.ngroups}: every batch row, heads {hs.start}.."
                      f"{hs.stop - 1}, every token"}


E2E_BUFFER_SETS = 3
PROFILED_STEPS = 200  # steps of the per-kernel profiled pass after the timed region
MIN_TIMED_S = 1.2


def run_e2e(inp, dev, args, stream):
    """The same step through the public call with host buffers: every step
    copies its inputs in from pinned host memory, runs fwd+bwd and copies all
    of its outputs and gradients back, inside the timed region.  Three device
    buffer sets rotate so that, as a user streaming batches would, the copy in
    of step k+1 and the copy out of step k-1 run on their own streams at the
    same time as each other and as the compute of step k (with two sets the
    copy in of step k+1 would have to wait for the copy out of step k-1 to
    free its buffers); the time is from the first copy in to the last copy
    out."""
    import torch
    from mamba_selective_state_gb300.runner import SSDDevice
    nb = E2E_BUFFER_SETS
    devs = [dev] + [SSDDevice(inp, device=dev.device, dfinal=False, extra_flags=step_flags(args))
                    for _ in range(nb - 1)]
    names_in = ["x", "dt", "B", "C", "dy", "dt_bias", "A", "D"]
    if dev.init is not None:
        names_in.append("init")
    if dev.seq_idx is not None:
        names_in.append("seq_idx")
    host_in = {n: getattr(dev, n).to("cpu").pin_memory() for n in names_in}
    names_out = ["y", "final", "dx", "ddt", "dB", "dC", "dA", "dD", "ddt_bias"]
    host_out = [{n: torch.empty_like(getattr(dev, n), device="cpu").pin_memory() for n in names_out}
                for _ in range(nb)]
    bi = sum(t.numel() * t.element_size() for t in host_in.values())
    bo = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    steps = max(4, min(args.steps, 12))
    torch.cuda.synchronize()

    def run(nsteps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        free = [None] * nb  # event: buffer set k % nb has been copied out
        e0.record(s_in)
        for k in range(nsteps):
            d = devs[k % nb]
            if free[k % nb] is not None:
                s_in.wait_event(free[k % nb])
            with torch.cuda.stream(s_in):
                for n, t in host_in.items():
                    getattr(d, n).copy_(t, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(s_in)
            stream.wait_event(ready)
            d.fwd(stream=stream)
            d.bwd(stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            s_out.wait_event(done)
            with torch.cuda.stream(s_out):
                for n, t in host_out[k % nb].items():
                    t.copy_(getattr(d, n), non_blocking=True)
            free[k % nb] = torch.cuda.Event()
            free[k % nb].record(s_out)
        e1.record(s_out)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    run(2)  # warm-up
    ms = run(steps) / steps
    tokens = inp.batch * inp.seqlen
    return {"value": tokens / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "overlap": f"{nb} device buffer sets; copies in and out on their own streams "
                       "overlap each other and the neighbouring steps' compute"}


# ----------------------------------------------------------------------------
# gated RMSNorm of the Mamba-2 block (--op gated_rmsnorm)
# ----------------------------------------------------------------------------
NORM_METRIC = "gated RMSNorm fwd+bwd tokens/s (ms); % of HBM"


def norm_model(rows, dim, G, gate, s):
    """Compulsory bytes of each norm kernel: every input read once, every
    output written once (the backward's per-block dweight partials and their
    fold are not counted: they are the reduction's own traffic)."""
    e = rows * dim * s
    nt = 2 if gate else 1
    return {"gated_norm_fwd": dict(bytes=nt * e + e + rows * G * 4 + dim * 4, flops=0),
            "gated_norm_bwd": dict(bytes=(nt + 1) * e + nt * e + 2 * dim * 4, flops=0)}


def norm_oracle_seconds(inp, block_rows=1024):
    """One float64 oracle fwd+bwd over every row of ``inp``, by row blocks."""
    import torch
    from oracle import gated_norm
    w = inp.f64("weight")
    t0 = time.perf_counter()
    for r0 in range(0, inp.rows, block_rows):
        sl = slice(r0, min(inp.rows, r0 + block_rows))
        y = inp.y[sl].to(torch.float64).numpy()
        z = None if inp.z is None else inp.z[sl].to(torch.float64).numpy()
        d = inp.dout[sl].to(torch.float64).numpy()
        gated_norm.gated_rmsnorm_fwd(y, z, w, inp.group_size, inp.eps)
        gated_norm.gated_rmsnorm_bwd(y, z, w, d, inp.group_size, inp.eps)
    return time.perf_counter() - t0


def norm_config(name, inp):
    return {"workload": f"gated_rmsnorm after {name}", "rows": inp.rows, "dim": inp.dim,
            "group_size": inp.group_size, "eps": inp.eps, "gate": inp.z is not None}


def run_norm_reference(args, rank):
    if rank != 0:
        return
    from mamba_selective_state_gb300.inputs import make_norm_workload
    inp = make_norm_workload(args.workload, seed=0)
    for _ in range(min(args.warmup, 1)):
        norm_oracle_seconds(inp)
    times = [norm_oracle_seconds(inp) for _ in range(max(1, min(args.steps, 5)))]
    value = inp.rows * len(times) / sum(times)
    desc = f"float64 numpy oracle fwd+bwd over all {inp.rows} rows, 1024-row blocks, 1 thread"
    line = {"impl": "reference", "op": "gated_rmsnorm", "metric": NORM_METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": norm_config(args.workload, inp),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_norm(args, world, rank, local):
    import torch
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.inputs import make_norm_workload
    from mamba_selective_state_gb300.runner import NormDevice

    inp = make_norm_workload(args.workload, seed=rank)
    dev = NormDevice(inp, device=f"cuda:{local}")
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=f"cuda:{local}")

    def step():
        dev.fwd(stream=stream)
        dev.bwd(stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    _lib.profile_start()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    prof = _lib.profile_stop()
    barrier(world)
    clk = clocks.stop() if clocks else None
    tot_ms = max_over_ranks(world, sum(s.elapsed_time(e) for s, e in zip(starts, ends)))
    ms_per_step = tot_ms / args.steps
    value = world * inp.rows * args.steps / (tot_ms / 1e3)

    # end to end: inputs from pinned host memory, outputs back, copies and
    # compute one after the other on the launching stream
    names_in = ["y", "z", "weight", "dout"] if dev.z is not None else ["y", "weight", "dout"]
    names_out = ["out", "rstd", "dy", "dweight"] + (["dz"] if dev.dz is not None else [])
    host_in = {n: getattr(dev, n).to("cpu").pin_memory() for n in names_in}
    host_out = {n: torch.empty_like(getattr(dev, n), device="cpu").pin_memory() for n in names_out}
    bi = sum(t.numel() * t.element_size() for t in host_in.values())
    bo = sum(t.numel() * t.element_size() for t in host_out.values())

    def e2e_step():
        for n, t in host_in.items():
            getattr(dev, n).copy_(t, non_blocking=True)
        step()
        for n, t in host_out.items():
            t.copy_(getattr(dev, n), non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(3, min(args.steps, 10))
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    e2e = {"value": inp.rows / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
           "overlap": "none: copies in, fwd+bwd and copies out in turn on one stream"}

    peaks, src = load_peaks()
    s_bytes = 2 if inp.dtype == "bf16" else 4
    model = norm_model(inp.rows, inp.dim, inp.dim // inp.group_size, dev.z is not None, s_bytes)
    kernels = {k: {"launches": n, "ms_per_launch": ms / n} for k, (n, ms) in prof.items()
               if not k.startswith("_")}
    for k, v in kernels.items():
        if k in model:
            v["GBps"] = model[k]["bytes"] / (v["ms_per_launch"] / 1e3) / 1e9
    dom = max(kernels, key=lambda k: kernels[k]["launches"] * kernels[k]["ms_per_launch"])
    hbm_peak = peaks["hbm_gbs"]
    ach = kernels[dom].get("GBps", 0.0)
    roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
            "frac": ach / hbm_peak, "traffic": ncu_traffic(dom, args.workload), "kernel": dom,
            "peak_source": f"{src} hbm_gbs", "algorithmic_bytes": model.get(dom, {}).get("bytes"),
            "ms_per_launch": kernels[dom]["ms_per_launch"]}
    io = model["gated_norm_fwd"]["bytes"] + model["gated_norm_bwd"]["bytes"]
    line = {"op": "gated_rmsnorm", "metric": NORM_METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": inp.dtype, "data": "synthetic",
            "config": dict(norm_config(args.workload, inp),
                           l2="flushed between steps (256 MB write, outside the events)",
                           parallelism="replicas" if world > 1 else "single GPU"),
            "roofline": roof,
            "layer_roofline": {"compulsory_io_bytes": io,
                               "achieved_GBps": io / (ms_per_step / 1e3) / 1e9,
                               "frac_of_hbm": io / (ms_per_step / 1e3) / 1e9 / hbm_peak},
            "e2e": e2e, "gpu_launches": sum(v["launches"] for v in kernels.values()),
            "kernels": kernels, "clocks": clk}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the whole workload, repeated until at least 10 s of CPU work
        secs, reps = 0.0, 0
        while reps == 0 or (secs < 10.0 and reps < 20):
            secs += norm_oracle_seconds(inp)
            reps += 1
        line["cpu_baseline"] = {"value": inp.rows * reps / secs, "unit": "tokens/s", "cores": 1,
                                "kind": "oracle", "seconds": secs,
                                "sample": f"float64 numpy oracle fwd+bwd over all {inp.rows} "
                                          f"rows, 1024-row blocks, 1 thread, run {reps} times"}
    return line


# ----------------------------------------------------------------------------
# context parallelism of the layer (--op context_parallel)
# ----------------------------------------------------------------------------
CP_METRIC = ("SSD layer fwd+bwd tokens/s over a sequence split into context-parallel shards "
             "(joined by the shard folds)")


def run_cp(args, world, rank, local):
    """The workload's sequence split into --shards equal shards, run one
    after another on this GPU through the shard driver (every shard twice
    forward and twice backward, with the decay and fold kernels between),
    next to the unsharded layer on the same inputs.  On R GPUs the shard
    passes would run at once; here their sum is timed."""
    import torch
    from mamba_selective_state_gb300 import _lib
    from mamba_selective_state_gb300.context_parallel import (ShardedLayer, StackExchange,
                                                              shard_bounds, shard_inputs)
    from mamba_selective_state_gb300.inputs import make_workload
    from mamba_selective_state_gb300.runner import SSDDevice

    inp = make_workload(args.workload, seed=rank, dfinal=False)
    R = args.shards
    L = inp.seqlen
    sizes = [L // R + (1 if k < L % R else 0) for k in range(R)]
    shards = [shard_inputs(inp, a, e) for a, e in shard_bounds(L, sizes)]
    layer = ShardedLayer(shards, list(range(R)), StackExchange(R), device=f"cuda:{local}")
    dev = SSDDevice(inp, device=f"cuda:{local}")
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=f"cuda:{local}")

    def timed(fn, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i in range(n):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev)

    def sharded():
        layer.run(initial_states=inp.initial_states, stream=stream)

    def plain():
        dev.fwd(stream=stream)
        dev.bwd(stream=stream)

    for _ in range(args.warmup):
        sharded()
        plain()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    barrier(world)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    _lib.profile_start()
    tot = timed(sharded, args.steps)
    prof = _lib.profile_stop()
    clk = clocks.stop() if clocks else None
    tot_plain = timed(plain, args.steps)
    tot = max_over_ranks(world, tot)
    ms = tot / args.steps
    tokens = inp.batch * L
    kernels = {k: {"launches": n, "ms_per_launch": t / n} for k, (n, t) in prof.items()
               if not k.startswith("_")}
    return {"op": "context_parallel", "metric": CP_METRIC, "value": world * tokens / (ms / 1e3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": inp.dtype, "data": "synthetic",
            "config": dict(workload_config(args.workload), shards=R, shard_tokens=sizes,
                           execution="shards one after another on one GPU; the exchange is a "
                                     "stack in one process",
                           l2="flushed between steps (256 MB write, outside the events)"),
            "unsharded_ms_per_step": tot_plain / args.steps,
            "overhead_vs_unsharded": ms / (tot_plain / args.steps),
            "gpu_launches": sum(v["launches"] for v in kernels.values()), "kernels": kernels,
            "clocks": clk}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scan", default="sequential", choices=["sequential", "warp_shuffle"],
                    help="the separate kernels' forward state-passing scan: each thread scans its "
                         "elements over a segment's chunks (default), or the lanes of a warp hold "
                         "the chunks and warp shuffles compose them (comparison)")
    ap.add_argument("--recompute", action="store_true",
                    help="the backward recomputes the forward's intermediates instead of taking "
                         "the ones the step's forward kept")
    ap.add_argument("--min-timed-s", type=float, default=MIN_TIMED_S,
                    help="least step time in the timed region (0: exactly --steps, for profiling)")
    ap.add_argument("--op", default="ssd", choices=["ssd", "gated_rmsnorm", "context_parallel"])
    ap.add_argument("--shards", type=int, default=4, help="--op context_parallel: shards")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":  # host-only: rank 0 runs, the other ranks exit
        rank0 = int(os.environ.get("RANK", "0"))
        if args.op == "gated_rmsnorm":
            run_norm_reference(args, rank0)
        else:
            run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), rank0)
        return
    world, rank, local = dist_setup(args)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    if world > 1 and rank != 0:
        __graft_entry__.build()
    run = {"gated_rmsnorm": run_norm, "context_parallel": run_cp}.get(args.op, run_gpu)
    line = run(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
