#!/usr/bin/env python
"""Throughput of the chunked KDA forward on GB300, one JSON line on rank 0.

Default workload: B=2, H=64, T=8192, K=V=128, bf16 q/k/v, fp32 g and beta,
with the Aqk / Akk_inv / W / U intermediates written (the headline
configuration).  A step is one kda_chunk_fwd call through the C ABI over
inputs resident in HBM; the inputs (1.34 GB) are larger than L2 (129 MB), so
no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--path auto|fused|two_pass] [--cp-chunks N]
  python bench.py --impl reference ...   # the FP64 CPU oracle, timed on the host

A step's work ends with the exact path's check of the per-chain flags (no
chunk of these workloads passes the gate range); `--cp-chunks N` times
intra-card context parallelism (segments of N chunks; fixed-length, K == V).

Multi-GPU (torchrun, one process per GPU): each rank runs an independent
replica of the workload (the path has no exchange step); `value` is the
aggregate tokens/s over all ranks, from the max per-rank time.
"""

from __future__ import annotations

import argparse
import hashlib
import ctypes
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd ms/call & tokens/s, B=2 H=64 T=8192 K=V=128 bf16; % of roofline"
# cuLA PR #131 (Performance table), CuTeDSL on SM100/SM103, K and V not
# stated: the complete public forward at B=2 H=64 T=8192 with FP32 beta
# (0.8564 ms) and T=1024 with BF16 beta (0.1320 ms); the grouped-value forward
# at B=1 Hq=16 Hv=64 T=4096, BF16 (0.2379 ms).
PAGE_MS = {"mha_8k": 0.8564, "mha_1k": 0.1320, "gva_4k": 0.2379}
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def _peaks():
    """HBM GB/s, bf16 TFLOP/s burst and sustained, and where they come from."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ bytes
def _chunk_count(w):
    if w["cu_seqlens"] is None:
        return w["B"] * ((w["T"] + 63) // 64)
    lens = np.diff(w["cu_seqlens"].cpu().numpy())
    return int(np.sum((lens + 63) // 64))


def algorithmic_bytes(w, N):
    """Bytes the method must move once (inputs, initial state, o, final state,
    the requested exports), and per kernel of each path: the method's bytes it
    moves, and the design's own extra traffic (state-pass operands handed from
    one kernel to the next through HBM)."""
    BT = w["B"] * w["T"]
    Hq, Hv, K, V = w["Hq"], w["Hv"], w["K"], w["V"]
    nc = _chunk_count(w)
    bsz = 4 if w["beta"].dtype.itemsize == 4 else 2
    inputs = BT * (2 * Hq * K * 2 + Hv * V * 2 + Hv * K * 4 + Hv * bsz)
    h0 = N * Hv * K * V * 4 if w["initial_state"] is not None else 0
    exports = BT * Hv * (64 * 4 * 2 + K * 2 + V * 2) if w["intermediates"] else 0
    outputs = BT * Hv * V * 2 + N * Hv * K * V * 4
    path = inputs + h0 + outputs + exports
    # two-pass design: Qs, Aqk (bf16), Kl, gamma written by the intra kernel and
    # read by the state kernel, and W, U kept in the workspace when not exported
    state_ops = BT * Hv * (K * 2 + 64 * 2 + K * 2) + nc * Hv * K * 4
    wu_internal = 0 if w["intermediates"] else BT * Hv * (K * 2 + V * 2)
    wu_reads = BT * Hv * (K * 2 + V * 2)
    return {
        "path": path,
        "fused": path,                                   # one kernel moves exactly the method's bytes
        "intra": inputs + exports,                       # the method's bytes the intra kernel moves
        "state": h0 + outputs,                           # and the state kernel
        "intra_design": state_ops + wu_internal,         # design traffic: state-pass operands written
        "state_design": state_ops + wu_reads,            # ... and read back
    }


def algorithmic_flops(w):
    """Tile-dense FLOPs of the path: per 64-token chunk and value head, the
    products Aqk, Akk, W, U (64 x 64 x K or V), W S and Qg S (64 x K x V),
    Aqk Delta (64 x 64 x V) and the state update K^T Delta (K x 64 x V)."""
    K, V = w["K"], w["V"]
    per = 2 * (3 * 64 * 64 * K + 64 * 64 * V + 2 * 64 * K * V + 64 * 64 * V + K * 64 * V)
    return _chunk_count(w) * w["Hv"] * per


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of a
# kernel from one single-pass ncu capture of the named workload, keyed by the
# SHA-1 of the sources the kernel was built from: once those change, the
# number no longer describes the kernel and is not reported.
MEASURED_TRAFFIC = {
    ("mha_8k", "fused"): (1349053696 + 1296978176, "a116875a0421d6677a733db693470474797dc048"),
    ("mha_8k", "intra"): (1378036992 + 1701146624, "aece64d32770adfd8facff429106cf6f43e78a21"),
    ("mha_8k", "state"): (1234033408 + 249490432, "e32552c36dc8c56d650d597a36ce1a2c1bc87bfb"),
}
KERNEL_SOURCES = {"intra": ("kda_intra.cu", "kda_internal.cuh", "kda_ptx.cuh"),
                  "state": ("kda_state.cu", "kda_internal.cuh", "kda_ptx.cuh"),
                  "fused": ("kda_fused.cu", "kda_internal.cuh", "kda_ptx.cuh")}


def measured_traffic(workload, kernel):
    entry = MEASURED_TRAFFIC.get((workload, kernel))
    if entry is None:
        return None
    h = hashlib.sha1()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "chunked_gated_delta_03_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return entry[0] if h.hexdigest() == entry[1] else None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle
def _oracle_head(args):
    q, k, v, g, beta, h0, scale = args
    from oracle import kda_ref as ref
    t = time.perf_counter()
    ref.kda_chunked(q, k, v, g, beta, scale, h0, chunk_size=64)
    return time.perf_counter() - t


def _head_problems(w, count):
    """Single-(sequence, value head) slices of the workload, as FP64 numpy arrays."""
    grp = w["Hv"] // w["Hq"]
    f64 = lambda t: t.double().numpy()
    probs = []
    for j in range(count):
        b = j % w["B"]
        hv = (j * 7) % w["Hv"]
        hq = hv // grp
        h0 = None if w["initial_state"] is None else f64(w["initial_state"][b:b + 1, hv:hv + 1])
        probs.append((f64(w["q"][b:b + 1, :, hq:hq + 1]), f64(w["k"][b:b + 1, :, hq:hq + 1]),
                      f64(w["v"][b:b + 1, :, hv:hv + 1]), f64(w["g"][b:b + 1, :, hv:hv + 1]),
                      f64(w["beta"][b:b + 1, :, hv:hv + 1]), h0, w["scale"]))
    return probs


def oracle_rate(pool, cores, w, rounds):
    """Oracle throughput in the metric's unit (tokens/s of the whole workload):
    `rounds` x `cores` single-head problems of T tokens, run `cores` at a time."""
    probs = _head_problems(w, cores)
    t0 = time.perf_counter()
    done = 0
    for _ in range(rounds):
        pool.map(_oracle_head, probs)
        done += len(probs)
    dt = time.perf_counter() - t0
    token_heads = done * w["T"]
    return token_heads / dt / w["Hv"], dt, done


def make_pool():
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("MKL_NUM_THREADS", "1")
    cores = len(os.sched_getaffinity(0))
    return mp.get_context("spawn").Pool(cores), cores


# ------------------------------------------------------------ ranks
def max_over_ranks(ms, world, device):
    """The slowest rank's time (every rank gets it); the rank's own time at world 1."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(ms, world, tokens_per_rank):
    """Tokens per second of the whole job: every rank runs one replica of the
    workload, and the job takes the slowest rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mha_8k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--path", choices=["auto", "fused", "two_pass"], default="auto")
    ap.add_argument("--cp-chunks", type=int, default=0,
                    help="intra-card context parallelism: segments of this many chunks (0: off)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.warmup < 3:
        args.warmup = 3

    from chunked_gated_delta_03_gb300.workloads import WORKLOADS, make_inputs
    wl = WORKLOADS[args.workload]
    config = {"workload": f"{wl.name}: B={wl.B} H={wl.Hv} (Hq={wl.Hq}) T={wl.T} K={wl.K} V={wl.V}, bf16 q/k/v, "
                          f"fp32 g, {wl.beta_dtype} beta" + (", Aqk/Akk_inv/W/U written" if wl.intermediates else ""),
              "B": wl.B, "T": wl.T, "Hq": wl.Hq, "Hv": wl.Hv, "K": wl.K, "V": wl.V,
              "l2": "inputs larger than L2 (no flush needed)", "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        if rank != 0:
            return
        w = make_inputs(wl)
        w["intermediates"] = wl.intermediates
        pool, cores = make_pool()
        for _ in range(args.warmup):
            oracle_rate(pool, cores, w, 1)
        rates, secs, done = [], 0.0, 0
        for _ in range(args.steps):
            r, dt, n = oracle_rate(pool, cores, w, 1)
            rates.append(r)
            secs += dt
            done += n
        pool.close()
        value = statistics.mean(rates)
        problems = w["N"] * wl.Hv
        frac = (done / args.steps) / problems
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                # a step is the sampled part of the workload: its measured wall time
                "ms_per_step": 1e3 * secs / args.steps, "sampled_fraction": frac,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"per step {cores} single-(sequence, head) problems of T={wl.T}, "
                                           f"one per core ({frac:.4f} of the workload's {problems}); tokens/s of "
                                           f"the whole workload = token-heads/s / Hv"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    # CPU baseline pool before any CUDA work (spawned workers)
    pool = cores = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool, cores = make_pool()

    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import __graft_entry__
    __graft_entry__.build()
    from chunked_gated_delta_03_gb300 import _lib, ops

    host = make_inputs(wl)
    host["intermediates"] = wl.intermediates
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    B, T, Hq, Hv, K, V, N = (host[x] for x in ("B", "T", "Hq", "Hv", "K", "V", "N"))
    a, _ = ops.make_args(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["scale"],
                         dev["initial_state"], dev["cu_seqlens"])
    a.path = ops._PATHS[args.path]
    a.cp_chunks = args.cp_chunks
    fused = args.path == "fused" or (args.path == "auto" and not a.intra_tf32)
    o = torch.empty(B, T, Hv, V, dtype=torch.bfloat16, device="cuda")
    fin = torch.empty(N, Hv, K, V, dtype=torch.float32, device="cuda")
    outs = {"o": o, "final_state": fin}
    a.o, a.final_state = o.data_ptr(), fin.data_ptr()
    if wl.intermediates:
        for name, shape, dt in (("Aqk", (B, T, Hv, 64), torch.float32), ("Akk_inv", (B, T, Hv, 64), torch.float32),
                                ("W", (B, T, Hv, K), torch.bfloat16), ("U", (B, T, Hv, V), torch.bfloat16)):
            outs[name] = torch.empty(shape, dtype=dt, device="cuda")
            setattr(a, name, outs[name].data_ptr())
    ws_bytes = _lib.kda_workspace_size(a)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def step(ev=None):
        a.profile_events = ev
        rc = _lib.kda_chunk_fwd(a, ws.data_ptr(), ws_bytes, sh)
        if rc != 0:
            raise RuntimeError(f"kda_chunk_fwd: {_lib.status_string(rc)}")

    # per-step kernel events: [start, after intra, after state]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for trio in evs:
        for e in trio:
            e.record(stream)
    handles = []
    for trio in evs:
        arr = (ctypes.c_void_p * 3)(*[e.cuda_event for e in trio])
        handles.append(arr)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(ctypes.cast(handles[i], ctypes.c_void_p))
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    st = ops.device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status after the timed region: {_lib.status_string(st)}")
    ms = t_start.elapsed_time(t_end) / args.steps
    intra_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][1]) for i in range(args.steps))
    state_ms = statistics.mean(evs[i][1].elapsed_time(evs[i][2]) for i in range(args.steps))
    ms = max_over_ranks(ms, world, "cuda")
    value = whole_job_rate(ms, world, B * T)

    # ---- end to end through the same C call, from/to pinned host memory.
    # Steps are pipelined the way a serving loop runs them: two device sets of
    # inputs and outputs, one stream each for host->device copies, compute and
    # device->host copies, so step i+1's inputs arrive while step i computes and
    # step i-1's results leave.  Every step's copies are inside the timed region.
    e2e = None
    if rank == 0:
        in_keys = ["q", "k", "v", "g", "beta"] + (["initial_state"] if host["initial_state"] is not None else [])
        pin = {k: host[k].pin_memory() for k in in_keys}
        h2d = sum(t.numel() * t.element_size() for t in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in outs.values())
        sets = []
        for sidx in range(2):
            din = dev if sidx == 0 else {k: torch.empty_like(dev[k]) for k in in_keys}
            dout = outs if sidx == 0 else {k: torch.empty_like(v) for k, v in outs.items()}
            sa, _ = ops.make_args(din["q"], din["k"], din["v"], din["g"], din["beta"], dev["scale"],
                                  din.get("initial_state"), dev["cu_seqlens"])
            sa.path = a.path
            sa.cp_chunks = a.cp_chunks
            sa.o, sa.final_state = dout["o"].data_ptr(), dout["final_state"].data_ptr()
            for name in ("Aqk", "Akk_inv", "W", "U"):
                if name in dout:
                    setattr(sa, name, dout[name].data_ptr())
            back = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in dout.items()}
            sets.append({"in": din, "out": dout, "args": sa, "back": back})
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set s copied in
        ev_done = [torch.cuda.Event() for _ in range(2)]   # compute on set s finished
        ev_out = [torch.cuda.Event() for _ in range(2)]    # results of set s copied out

        def e2e_run(n):
            for i in range(n):
                st = sets[i & 1]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_done[i & 1])
                    for k, t in pin.items():
                        st["in"][k].copy_(t, non_blocking=True)
                    ev_in[i & 1].record(s_in)
                stream.wait_event(ev_in[i & 1])
                if i >= 2:
                    stream.wait_event(ev_out[i & 1])
                rc = _lib.kda_chunk_fwd(st["args"], ws.data_ptr(), ws_bytes, sh)
                if rc != 0:
                    raise RuntimeError(f"kda_chunk_fwd: {_lib.status_string(rc)}")
                ev_done[i & 1].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[i & 1])
                    for k, t in st["back"].items():
                        t.copy_(st["out"][k], non_blocking=True)
                    ev_out[i & 1].record(s_out)

        e2e_run(3)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        e2e_run(args.e2e_steps)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
        e2e = {"value": B * T / (e2e_ms * 1e-3), "unit": "tokens/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "pipelining": "2 device buffer sets; copy-in, compute and copy-out streams overlap across steps"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm, bf16, bf16_sus, src = _peaks()
    by = algorithmic_bytes(host, N)
    flops = algorithmic_flops(host)
    kern = {"fused": intra_ms} if fused else {"intra": intra_ms, "state": state_ms}
    top = max(kern, key=kern.get)
    # the dominant kernel against the slower of its bytes at the HBM peak and
    # the path's FLOPs at the bf16 tensor peak (sustained: the kernel runs
    # inside a long step); achieved counts the method's bytes only
    t_bytes = by[top] / (hbm * 1e9)
    t_flops = (flops / (bf16_sus * 1e12)) if top == "fused" else 0.0
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    if bound == "hbm":
        achieved = by[top] / (kern[top] * 1e-3) / 1e9
        peak, unit = hbm, "GB/s"
    else:
        achieved = flops / (kern[top] * 1e-3) / 1e12
        peak, unit = bf16_sus, "TFLOP/s"
    design = by.get(f"{top}_design", 0)
    roof = {"kernel": f"kda::{top}_kernel", "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": measured_traffic(args.workload, top), "peak_source": src,
            "algorithmic_bytes_per_launch": by[top], "design_bytes_per_launch": design,
            "design_over_method": (by[top] + design) / by[top]}
    path_gbs = by["path"] / (ms * 1e-3) / 1e9
    roof_ms = max(by["path"] / (hbm * 1e9), flops / (bf16_sus * 1e12)) * 1e3
    path = {"bytes_per_step": by["path"], "flops_per_step": flops, "achieved": path_gbs, "peak": hbm,
            "unit": "GB/s", "roofline_ms": roof_ms, "frac": roof_ms / ms,
            "bytes_ms": by["path"] / (hbm * 1e9) * 1e3, "flops_ms": flops / (bf16_sus * 1e12) * 1e3}

    cpu = None
    if pool is not None:
        r, dt, done = oracle_rate(pool, cores, host, 2)
        pool.close()
        cpu = {"value": r, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{done} single-(sequence, head) problems of T={T} ({dt:.1f} s on {cores} cores); "
                         f"tokens/s of the whole workload = token-heads/s / Hv"}

    page = PAGE_MS.get(wl.name)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / (B * T / (page * 1e-3))) if page else None,
            "dtype": "bf16", "data": "synthetic", "config": config,
            "kernels_ms": kern, "roofline": roof, "path_roofline": path, "cpu_baseline": cpu, "e2e": e2e,
            # per step: the fused kernel, or intra + state, then the exact
            # path's check of the chain flags (its CTAs return at once unless a
            # chunk passed the gate range); varlen adds the sequence-order
            # kernel (and, on the two-pass path, the chunk table)
            # (with --cp-chunks: the segment table, three passes of the fused
            # kernel over the segments as packed sequences, each with its
            # sequence order and flag check, the identity start states and
            # the scan)
            "gpu_launches": args.steps * (
                (1 + 3 * 3 + 1 + 1) if (args.cp_chunks and -(-T // 64) > args.cp_chunks) else
                ((1 if fused else 2) + 1 + (0 if host["cu_seqlens"] is None else (1 if fused else 2)))),
            "path": "fused" if fused else "two_pass",
            "clocks": clocks}
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
