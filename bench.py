"""Benchmark: causal GQA attention forward + backward on one GB300 (or N independent replicas).

One step = upipe_attn_fwd + upipe_attn_bwd over the whole workload (all head groups, all
trunks), inputs resident in HBM. Default workload: the Llama3-8B-shaped attention layer at
S = 131072 (B=1, Hq=32, Hkv=8, D=128, head_chunk=8, seq_trunk=131072, causal), the size the
throughput target is quoted on. FLOPs follow the FlashAttention benchmark convention:
fwd = 4*B*Hq*D*S^2/2 (causal), bwd = 2.5 * fwd.

Prints ONE JSON line (rank 0). Under torchrun every rank runs an independent replica on its own
GPU (the path does not shard on one box); value = total FLOPs of all ranks / max rank time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--head-chunk H] [--seq-trunk T] [--impl ours|reference]

--workload llama8b_readout_s128k (or readout_small) measures the sequence-tiled readout +
cross-entropy loss instead (one step = upipe_ce_fwd + upipe_ce_bwd over S tokens, seq_tile
tokens at a time; FLOPs: fwd 2*S*V*Dm, bwd 3x that) and prints its own JSON line;
--workload llama8b_mlp_s128k (or mlp_small) the sequence-tiled SwiGLU MLP (upipe_mlp_fwd +
upipe_mlp_bwd; FLOPs: fwd 6*S*Dm*F, bwd 16*S*Dm*F).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("causal attn fwd+bwd TFLOP/s & % BF16 tensor peak on 1 GB300; peak workspace GB")
UNIT = "TFLOP/s"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama8b_s128k")
    ap.add_argument("--head-chunk", type=int, default=None)
    ap.add_argument("--seq-trunk", type=int, default=None)
    ap.add_argument("--seq-tile", type=int, default=None,
                    help="tokens per tile for the loss workloads (default: the workload's)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-explicit-copies", action="store_true",
                    help="tiled workloads: measure e2e through the library's host staging only "
                         "(skips the user-copy variant and its second set of pinned buffers, "
                         "for sequences whose activations would not fit host memory twice)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override S (small profiling captures only; not a bench line)")
    ap.add_argument("--sweep", default=None, choices=["chunk-trunk", "host-kv"],
                    help="print one JSON line per sweep point instead of the bench line: "
                         "chunk-trunk = head_chunk x seq_trunk grid; host-kv = the same "
                         "workload with K/V on the device and in pinned host memory")
    ap.add_argument("--head-chunks", default=None,
                    help="comma-separated head_chunk values for --sweep (default: per sweep)")
    ap.add_argument("--seq-trunks", default=None,
                    help="comma-separated seq_trunk values for --sweep (default: per sweep)")
    ap.add_argument("--kv-modes", default=None,
                    help="for --sweep host-kv: comma-separated subset of device,host,host+dkdv,all "
                         "(host+dkdv: dK/dV in pinned host memory as well; all: q, o, dout, dq "
                         "too)")
    return ap.parse_args()


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch, from a one-pass ncu
# capture of the first launch of each attention kernel on the default workload (one launch =
# one head group over the whole sequence; ncu printed these two in GB and MB to three
# significant figures). A figure holds only for the kernel source file it was
# taken on (by SHA-256) and for that workload; otherwise the bench reports null.
TRAFFIC = {
    "attn_bwd": {"workload": "llama8b_s128k", "head_chunk": 8, "seq_trunk": 131072,
                 "files": ["context_parallelism_gb300/csrc/attn_bwd_pp.cu"],
                 "sha256": "8c3a428d82d25b4312eb8dbaa3d6875f5f292b8189bd9fce9eee8faf92ff7549",
                 "bytes": 8_090_000_000 + 4_000_000_000},
    "attn_fwd": {"workload": "llama8b_s128k", "head_chunk": 8, "seq_trunk": 131072,
                 "files": ["context_parallelism_gb300/csrc/attn_fwd_pp.cu"],
                 "sha256": "93229bb574184d13c422be91979798dc0c1c9378df0e312d2c854d17e2250521",
                 "bytes": 696_250_000 + 235_360_000},
    # the sequence-tiled GEMMs (one class, one kernel with several epilogues), one entry per
    # workload; the schedule key is (seq_tile, None) and the figure is the mean over one
    # step's launches. Loss, per 8192-token tile: forward logits 2.21 GB, backward recompute
    # 4.28 GB, dh 8.47 GB, dw 8.71 GB. MLP: gate/up 0.76 GB, y 1.00 GB, recompute 1.24 GB,
    # dg|du 1.52 GB, dWd 1.02 GB, dWgu 1.97 GB, dx 1.94 GB.
    "loss_gemm": [
        {"workload": "llama8b_readout_s128k", "head_chunk": 8192, "seq_trunk": None,
         "files": ["context_parallelism_gb300/csrc/gemm_tc.cu",
                   "context_parallelism_gb300/csrc/seqtile_api.cpp"],
         "sha256": "5b0cf150e036e4cdb96d44b4d44b8dadbc20c1104278578e50a0d005ae7919c6",
         "bytes": 5925325980},
        {"workload": "llama8b_mlp_s128k", "head_chunk": 8192, "seq_trunk": None,
         "files": ["context_parallelism_gb300/csrc/gemm_tc.cu",
                   "context_parallelism_gb300/csrc/seqtile_api.cpp"],
         "sha256": "5b0cf150e036e4cdb96d44b4d44b8dadbc20c1104278578e50a0d005ae7919c6",
         "bytes": 1367694834},
    ],
}


def source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_per_launch(kernel, workload, head_chunk, seq_trunk):
    """The captured DRAM bytes per launch of `kernel`, or None when the capture does not
    apply (other workload or schedule, kernel source changed since, or no capture)."""
    entries = TRAFFIC.get(kernel) or []
    if isinstance(entries, dict):
        entries = [entries]
    for t in entries:
        if t["bytes"] is None:
            continue
        if (t["workload"], t["head_chunk"], t["seq_trunk"]) != (workload, head_chunk, seq_trunk):
            continue
        return t["bytes"] if source_hash(t["files"]) == t["sha256"] else None
    return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# ---- clocks sampled during the timed region ------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, _, _, f in rows for n, v in zip(names, f[1:]) if v == "Active"})
        load = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in load),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "samples": len(rows), "reasons": reasons}


# ---- the CPU oracle on a bounded sample ----------------------------------------------------
def oracle_sample(w, S_sample, inputs=None):
    """Times the fp64 oracle's forward + backward on the first S_sample tokens of the workload
    (an exact causal sub-problem). Returns (tflops, seconds, flops, description, cores)."""
    import numpy as np
    import oracle
    from workloads import make_inputs
    if inputs is not None:
        q, k, v, do = (t[:, :S_sample].float().cpu().numpy().astype(np.float64) for t in inputs)
        src = "prefix of the seeded workload tensors"
    else:
        ws = w.with_(S=S_sample)
        q, k, v, do = (t.float().numpy().astype(np.float64) for t in make_inputs(ws, "cpu"))
        src = "same recipe regenerated on the CPU at the sample length"
    flops = 3.5 * w.with_(S=S_sample).flops_fwd()
    t0 = time.perf_counter()
    oracle.attn_bwd_ref(q, k, v, do, causal=w.causal)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"fp64 numpy oracle fwd+bwd on the first {S_sample} of {w.S} tokens, all {w.Hq} "
            f"q-heads ({src}); FLOPs by the same causal convention")
    return flops / dt / 1e12, dt, flops, desc, cores


def job_throughput(local_ms, steps, flops_per_step, world, reduce_max=None):
    """Whole-job TFLOP/s of N independent replicas: every rank ran `steps` steps of
    `flops_per_step`; the job takes as long as its slowest rank. Returns (tflops, max_ms)."""
    t_max = float(local_ms)
    if reduce_max is not None:
        t_max = float(reduce_max(t_max))
    return world * flops_per_step * steps / (t_max / 1e3) / 1e12, t_max


def torch_reduce_max(device):
    """MAX all-reduce of one float over the default process group (NCCL or gloo)."""
    import torch
    import torch.distributed as dist

    def f(x):
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return f


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_reference(a):
    """The reference arm: the fp64 oracle on the host cores, rank 0 only."""
    rank, world, _ = _dist()
    if rank != 0:
        return
    from workloads import WORKLOADS
    w = WORKLOADS[a.workload]
    S_sample = min(w.S, 1024)
    vals = []
    for i in range(a.warmup + a.steps):
        tf, dt, flops, desc, cores = oracle_sample(w, S_sample)
        if i >= a.warmup:
            vals.append((tf, dt))
    value = sum(flops for _ in vals) / sum(dt for _, dt in vals) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": 1000.0 * statistics.mean(dt for _, dt in vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "head_chunk": a.head_chunk or w.head_chunk,
                   "seq_trunk": a.seq_trunk or w.seq_trunk, "causal": w.causal,
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(a):
    import torch
    import torch.distributed as dist

    import context_parallelism_gb300 as up
    from workloads import WORKLOADS, make_inputs

    rank, world, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[a.workload]
    if a.seq_len:
        w = w.with_(S=a.seq_len, seq_trunk=min(w.seq_trunk, a.seq_len),
                    name=f"{w.name}@S={a.seq_len}")
    hc = a.head_chunk or w.head_chunk
    T = a.seq_trunk or w.seq_trunk
    kv_host = w.kv_on_host
    B, S, Hq, Hkv, D = w.B, w.S, w.Hq, w.Hkv, w.D

    q, k, v, do = make_inputs(w, str(dev) if w.gen_device == "cuda" else "cpu")
    q, do = q.to(dev), do.to(dev)
    if kv_host:
        kh = torch.empty(k.shape, dtype=k.dtype, pin_memory=True); kh.copy_(k)
        vh = torch.empty(v.shape, dtype=v.dtype, pin_memory=True); vh.copy_(v)
        k_in, v_in = kh, vh
    else:
        k_in, v_in = k.to(dev), v.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    dq = torch.empty_like(q)
    dk = torch.empty((B, S, Hkv, D), dtype=q.dtype, device=dev)
    dv = torch.empty_like(dk)
    ws_bytes = up.upipe_workspace_bytes(B, S, Hq, Hkv, D, 1, hc, T, up.UPIPE_PASS_BOTH, kv_host)
    ws_full = up.upipe_workspace_bytes(B, S, Hq, Hkv, D, 1, Hq, T, up.UPIPE_PASS_BOTH, kv_host)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        up.upipe_attn_fwd(q, k_in, v_in, o, lse, B, S, Hq, Hkv, D, 1, hc, T, ws, ws_bytes, stream)
        up.upipe_attn_bwd(q, k_in, v_in, o, lse, do, dq, dk, dv, B, S, Hq, Hkv, D, 1, hc, T, ws,
                          ws_bytes, stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(a.warmup):
        step()
    up.upipe_sync_status(stream)

    # ---- timed region: K steps, device events on the launching stream ----
    fwd_ms = bwd_ms = 0.0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    up.upipe_profile_read()  # drop anything recorded before
    up.upipe_profile_enable(True)
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    time.sleep(0.3)
    launches0 = up.upipe_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(a.steps):
        ev[i][0].record(stream)
        up.upipe_attn_fwd(q, k_in, v_in, o, lse, B, S, Hq, Hkv, D, 1, hc, T, ws, ws_bytes, stream)
        ev[i][1].record(stream)
        up.upipe_attn_bwd(q, k_in, v_in, o, lse, do, dq, dk, dv, B, S, Hq, Hkv, D, 1, hc, T, ws,
                          ws_bytes, stream)
        ev[i][2].record(stream)
    t_end.record(stream)
    barrier()
    launches = up.upipe_launch_count() - launches0
    clk = clocks.stop()
    up.upipe_profile_enable(False)
    prof = up.upipe_profile_read()
    up.upipe_sync_status(stream)
    elapsed = t_start.elapsed_time(t_end)
    for e0, e1, e2 in ev:
        fwd_ms += e0.elapsed_time(e1)
        bwd_ms += e1.elapsed_time(e2)
    f_fwd, f_bwd = w.flops_fwd(), w.flops_bwd()
    red = torch_reduce_max(dev) if world > 1 else None
    value, t_max = job_throughput(elapsed, a.steps, f_fwd + f_bwd, world, red)
    ms_per_step = t_max / a.steps
    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])

    # dominant kernel: the class with the most device time; its algorithmic FLOPs are the
    # causal FLOPs of the pass it belongs to (all of them run inside that kernel class)
    algo = {"attn_fwd": f_fwd * a.steps, "attn_bwd": f_bwd * a.steps}
    top = max(prof, key=lambda kname: prof[kname][0])
    tot_ms, n_launch = prof[top]
    if top in algo and tot_ms > 0:
        achieved = algo[top] / (tot_ms / 1e3) / 1e12
        roofline = {"kernel": top, "bound": "tensor", "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": f"{peak_src} bf16_tflops_sustained",
                    "launches": n_launch, "avg_launch_ms": tot_ms / max(n_launch, 1),
                    "traffic": traffic_per_launch(top, w.name, hc, T),
                    "traffic_unit": "bytes per launch"}
    else:
        roofline = {"kernel": top, "bound": "hbm", "achieved": None, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": None, "traffic": None}
    kernels = {kname: {"ms_per_step": t / a.steps, "launches_per_step": n / a.steps}
               for kname, (t, n) in prof.items() if n}
    # HBM-bound kernels against the measured copy bandwidth: algorithmic bytes per step (each
    # element read and written once) over their summed event time.
    elem_q = B * S * Hq * D
    elem_kv = 0 if kv_host else 2 * B * S * Hkv * D
    hbm_bytes = {
        "layout": 2 * 2 * 2 * (elem_q + elem_kv),  # fwd + bwd gathers, bf16 read + write
        "bwd_pre": elem_q * (2 + 2 + 2 + 4),        # read O, dO; write dO gather, zero dQ acc
        "dq_convert": elem_q * (4 + 2),             # read fp32 dQ acc, write bf16 dQ
    }
    for kname, nbytes in hbm_bytes.items():
        if kname in kernels and kernels[kname]["ms_per_step"] > 0:
            gbs = nbytes / (kernels[kname]["ms_per_step"] / 1e3) / 1e9
            kernels[kname].update({"algorithmic_gb_per_step": nbytes / 1e9, "gbs": gbs,
                                   "frac_of_hbm": gbs / float(peaks["hbm_gbs"])})

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,%g) bf16, no weights)" % w.std,
        "config": {"workload": w.name, "B": B, "S": S, "Hq": Hq, "Hkv": Hkv, "D": D,
                   "head_chunk": hc, "seq_trunk": T, "causal": True, "kv_on_host": kv_host,
                   "l2": "inputs larger than L2 (q is %.2f GiB)" % (q.nbytes / 2**30),
                   "parallelism": "replicas" if world > 1 else "single"},
        "fwd_tflops": world * f_fwd * a.steps / (fwd_ms / 1e3) / 1e12,
        "bwd_tflops": world * f_bwd * a.steps / (bwd_ms / 1e3) / 1e12,
        "frac_of_bf16_peak": value / world / peak,
        "peak_tflops": peak, "peak_source": peak_src,
        "workspace_gb": ws_bytes / 1e9, "workspace_unchunked_gb": ws_full / 1e9,
        "workspace_ratio": ws_bytes / ws_full,
        "roofline": roofline, "kernels": kernels,
        "gpu_launches": int(launches), "clocks": clk,
    }

    # ---- end to end: host buffers in, results out, copies inside the timed region ----
    if not a.no_e2e:
        hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True); hq.copy_(q)
        hdo = torch.empty(do.shape, dtype=do.dtype, pin_memory=True); hdo.copy_(do)
        if kv_host:
            hk, hv = k_in, v_in
        else:
            hk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True); hk.copy_(k_in)
            hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True); hv.copy_(v_in)
        outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse, dq, dk, dv)]
        h2d = hq.nbytes + hdo.nbytes + (0 if kv_host else hk.nbytes + hv.nbytes)
        d2h = sum(t.nbytes for t in outs_h)

        # The step a user would write: dO is copied in on a side stream while the forward
        # runs (only the backward reads it), and O and LSE are copied out on that stream while
        # the backward runs; q, k, v in and dQ, dK, dV out sit on the compute stream.
        side = torch.cuda.Stream(dev)
        ev_start = torch.cuda.Event()
        ev_do = torch.cuda.Event()
        ev_fwd = torch.cuda.Event()
        ev_out = torch.cuda.Event()

        def e2e_step_marked(evs=None):
            if evs:
                evs[0].record(stream)
            ev_start.record(stream)
            side.wait_event(ev_start)
            with torch.cuda.stream(side):
                do.copy_(hdo, non_blocking=True)
            ev_do.record(side)
            q.copy_(hq, non_blocking=True)
            if not kv_host:
                k_in.copy_(hk, non_blocking=True)
                v_in.copy_(hv, non_blocking=True)
            if evs:
                evs[1].record(stream)
            up.upipe_attn_fwd(q, k_in, v_in, o, lse, B, S, Hq, Hkv, D, 1, hc, T, ws, ws_bytes, stream)
            ev_fwd.record(stream)
            side.wait_event(ev_fwd)
            with torch.cuda.stream(side):
                outs_h[0].copy_(o, non_blocking=True)
                outs_h[1].copy_(lse, non_blocking=True)
            ev_out.record(side)
            stream.wait_event(ev_do)
            up.upipe_attn_bwd(q, k_in, v_in, o, lse, do, dq, dk, dv, B, S, Hq, Hkv, D, 1, hc, T,
                              ws, ws_bytes, stream)
            if evs:
                evs[2].record(stream)
            for hdst, dsrc in zip(outs_h[2:], (dq, dk, dv)):
                hdst.copy_(dsrc, non_blocking=True)
            # the next step overwrites o/lse: their copy-out must be done (and so must this one)
            stream.wait_event(ev_out)
            if evs:
                evs[3].record(stream)

        e2e_step_marked()
        barrier()
        # per-phase events (host->device, compute, device->host) of the same steps
        ph = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(a.steps)]

        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(a.steps):
            e2e_step_marked(ph[i])
        e1.record(stream)
        barrier()
        breakdown = {k: sum(ev[i].elapsed_time(ev[i + 1]) for ev in ph) / a.steps
                     for i, k in enumerate(("h2d_ms", "compute_ms", "d2h_ms"))}
        e2e_copy_value, _ = job_throughput(e0.elapsed_time(e1), a.steps, f_fwd + f_bwd, world, red)
        explicit = {"value": e2e_copy_value, "per_step_ms": breakdown,
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "method": "user copies around device-buffer calls; dO in during the forward, "
                              "O and LSE out during the backward"}

        # The same step through the library with every tensor in pinned host memory: q, k, v,
        # dout in and o, dq, dk, dv out are staged by the library one head group (and key/value
        # trunk) at a time while the neighbouring group computes; LSE stays on the device and
        # is read back at the end of each step.
        mask = up.UPIPE_HOST_KV | up.UPIPE_HOST_ACT
        ws_h_bytes = up.upipe_workspace_bytes(B, S, Hq, Hkv, D, 1, hc, T, up.UPIPE_PASS_BOTH, mask)
        ws_h = torch.empty(ws_h_bytes, dtype=torch.uint8, device=dev)
        ho, hdq = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(2))
        hdk, hdv = (torch.empty(k.shape, dtype=k.dtype, pin_memory=True) for _ in range(2))
        hlse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

        def e2e_host_step():
            up.upipe_attn_fwd(hq, hk, hv, ho, lse, B, S, Hq, Hkv, D, 1, hc, T, ws_h, ws_h_bytes,
                              stream)
            up.upipe_attn_bwd(hq, hk, hv, ho, lse, hdo, hdq, hdk, hdv, B, S, Hq, Hkv, D, 1, hc, T,
                              ws_h, ws_h_bytes, stream)
            hlse.copy_(lse, non_blocking=True)

        e2e_host_step()
        barrier()
        e0.record(stream)
        for i in range(a.steps):
            e2e_host_step()
        e1.record(stream)
        barrier()
        e2e_value, _ = job_throughput(e0.elapsed_time(e1), a.steps, f_fwd + f_bwd, world, red)
        # bytes the library moves per step: the forward reads q, k, v and writes o; the
        # backward reads q, k, v, o, dout and writes dq, dk, dv; plus the LSE read-back
        h2d = 2 * (hq.nbytes + hk.nbytes + hv.nbytes) + ho.nbytes + hdo.nbytes
        d2h = ho.nbytes + hdq.nbytes + hdk.nbytes + hdv.nbytes + hlse.nbytes
        line["e2e"] = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                       "d2h_bytes_per_step": int(d2h),
                       "method": "upipe_attn_fwd/bwd with q, k, v, dout, o, dq, dk, dv in pinned "
                                 "host memory (library stages them per head group); LSE read back",
                       "workspace_gb": ws_h_bytes / 1e9, "explicit_copies": explicit}
        up.upipe_sync_status(stream)

    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        tf, dt, flops, desc, cores = oracle_sample(w, min(S, 2048), (q, k, v, do))
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_sweep(a):
    """Forward + backward TFLOP/s and workspace over a grid of schedules (one GPU)."""
    import torch

    import context_parallelism_gb300 as up
    from workloads import WORKLOADS, make_inputs

    w = WORKLOADS[a.workload]
    if a.seq_len:
        w = w.with_(S=a.seq_len, seq_trunk=min(w.seq_trunk, a.seq_len))
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in make_inputs(w, "cuda" if w.gen_device == "cuda" else "cpu"))
    def ints(text, default):
        return [int(x) for x in text.split(",")] if text else list(default)

    if a.sweep == "chunk-trunk":
        hcs = ints(a.head_chunks, (4, 8, 16, 32))
        Ts = ints(a.seq_trunks, (16384, 32768, w.S))
        grid = sorted({(hc, T) for hc in hcs if hc % w.G == 0 and w.Hq % hc == 0
                       for T in Ts if T <= w.S})
        kv_modes = ["device"]
    else:
        grid = [(hc, T) for hc in ints(a.head_chunks, [a.head_chunk or w.head_chunk])
                for T in ints(a.seq_trunks, [a.seq_trunk or w.seq_trunk])]
        kv_modes = (a.kv_modes or "device,host").split(",")
    device_ms = {}
    for mode in kv_modes:
        kv_host = mode in ("host", "host+dkdv", "all")
        dkdv_host = mode in ("host+dkdv", "all")
        act_host = mode == "all"  # q, o, dout, dq pinned on the host as well
        if act_host:
            qq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
            qq.copy_(q)
            ddo = torch.empty(do.shape, dtype=do.dtype, pin_memory=True)
            ddo.copy_(do)
        else:
            qq, ddo = q, do
        if kv_host:
            kk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
            kk.copy_(k)
            vv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
            vv.copy_(v)
        else:
            kk, vv = k, v
        for hc, T in grid:
            mask = (up.UPIPE_HOST_KV if kv_host else 0) | (up.UPIPE_HOST_ACT if act_host else 0)
            ws_b = up.upipe_workspace_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, 1, hc, T,
                                            up.UPIPE_PASS_BOTH, mask)
            ws = torch.empty(ws_b, dtype=torch.uint8, device=dev)
            if act_host:
                o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
                dq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
            else:
                o = torch.empty_like(q)
                dq = torch.empty_like(q)
            lse = torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, device=dev)
            if dkdv_host:
                dk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
                dv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
            else:
                dk = torch.empty_like(k)
                dv = torch.empty_like(v)
            args = (w.B, w.S, w.Hq, w.Hkv, w.D, 1, hc, T)

            def fwd():
                up.upipe_attn_fwd(qq, kk, vv, o, lse, *args, ws, ws_b)

            def bwd():
                up.upipe_attn_bwd(qq, kk, vv, o, lse, ddo, dq, dk, dv, *args, ws, ws_b)

            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            for _ in range(max(1, a.warmup)):
                fwd()
                bwd()
            torch.cuda.synchronize()
            lib_alloc = free0 - torch.cuda.mem_get_info()[0]
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            tf = tb = 0.0
            for _ in range(a.steps):
                e[0].record()
                fwd()
                e[1].record()
                bwd()
                e[2].record()
                torch.cuda.synchronize()
                tf += e[0].elapsed_time(e[1])
                tb += e[1].elapsed_time(e[2])
            up.upipe_sync_status()
            ms_step = (tf + tb) / a.steps
            if mode == "device":
                device_ms[(hc, T)] = ms_step
            copies = {}
            if kv_host:
                # one more step with the library's event bracketing on: the copy stream's busy
                # time per staged key/value trunk (and dK/dV trunk) against the kernels' time
                up.upipe_profile_read()
                up.upipe_profile_enable(True)
                e[0].record()
                fwd()
                bwd()
                e[1].record()
                torch.cuda.synchronize()
                up.upipe_profile_enable(False)
                st = up.upipe_profile_read()
                kv_ms, kv_n = st["kv_h2d"]
                kv_bytes = 2 * (k.numel() + v.numel()) * k.element_size()  # fwd and bwd pass
                kern_ms = sum(st[c][0] for c in ("layout", "attn_fwd", "bwd_pre", "attn_bwd",
                                                 "dq_convert"))
                copies = {
                    "profiled_step_ms": e[0].elapsed_time(e[1]),
                    "kernel_ms": kern_ms,
                    "kv_h2d_ms": kv_ms, "kv_h2d_trunks": kv_n,
                    "kv_h2d_gbs": kv_bytes / (kv_ms * 1e-3) / 1e9 if kv_ms else None,
                    "dkdv_d2h_ms": st["dkdv_d2h"][0], "dkdv_d2h_trunks": st["dkdv_d2h"][1],
                    # the compute stream's stalls waiting for staged trunks: copy time not
                    # hidden behind compute, measured directly
                    "kv_wait_ms": st["kv_wait"][0],
                }
                if (hc, T) in device_ms:
                    # the whole difference to the device-resident run: copy stalls plus the
                    # trunk-by-trunk launch structure staging needs
                    copies["vs_device_ms"] = ms_step - device_ms[(hc, T)]
            ff, fb = w.flops_fwd() * a.steps, w.flops_bwd() * a.steps
            print(json.dumps({
                "sweep": a.sweep, "workload": w.name, "S": w.S, "head_chunk": hc,
                "seq_trunk": T, "kv_on_host": kv_host, "dkdv_on_host": dkdv_host,
                "activations_on_host": act_host,
                "fwd_tflops": ff / tf / 1e9,
                "bwd_tflops": fb / tb / 1e9, "fwdbwd_tflops": (ff + fb) / (tf + tb) / 1e9,
                "ms_per_step": ms_step, **copies, "workspace_gb": ws_b / 1e9,
                "workspace_unchunked_gb": up.upipe_workspace_bytes(
                    w.B, w.S, w.Hq, w.Hkv, w.D, 1, w.Hq, T, up.UPIPE_PASS_BOTH, mask) / 1e9,
                "device_bytes_allocated_by_calls": int(lib_alloc)}), flush=True)
            del ws


LOSS_METRIC = "sequence-tiled readout + cross-entropy fwd+bwd TFLOP/s on 1 GB300"
MLP_METRIC = "sequence-tiled SwiGLU MLP fwd+bwd TFLOP/s on 1 GB300"


def loss_oracle_sample(lw, S_sample, inputs):
    """Times the fp64 oracle's loss forward + backward on the first S_sample tokens (the full
    vocabulary and width). Returns (tflops, seconds, description, cores)."""
    import oracle
    h, w, t, g = inputs
    hs, ts, gs = h[:S_sample].cpu(), t[:S_sample].cpu(), g[:S_sample].cpu()
    ws = w.cpu()
    flops = lw.with_(S=S_sample).flops_fwd() + lw.with_(S=S_sample).flops_bwd()
    t0 = time.perf_counter()
    oracle.ce_loss_bwd_ref(hs, ws, ts, gs)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"fp64 numpy oracle loss fwd+bwd on the first {S_sample} of {lw.S} tokens, full "
            f"vocabulary {lw.V} x width {lw.Dm}; FLOPs by the same convention")
    return flops / dt / 1e12, dt, desc, cores


def _loss_spec(a, dev, up):
    from workloads import LOSS_WORKLOADS, make_loss_inputs
    import torch
    lw = LOSS_WORKLOADS[a.workload]
    if a.seq_len:
        lw = lw.with_(S=a.seq_len, name=f"{lw.name}@S={a.seq_len}")
    T = a.seq_tile or lw.seq_tile
    S, Dm, V = lw.S, lw.Dm, lw.V
    h, w, t, g = (x.to(dev) for x in make_loss_inputs(lw, str(dev) if lw.gen_device == "cuda"
                                                      else "cpu"))
    loss = torch.empty(S, dtype=torch.float32, device=dev)
    lse = torch.empty(S, dtype=torch.float32, device=dev)
    dh = torch.empty_like(h)
    dw = torch.empty((V, Dm), dtype=torch.float32, device=dev)
    ws_bytes = up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BOTH)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def host_setup():
        # h in and dh out through the library's tile staging; targets in and the per-token
        # loss out by the caller; w and dw stay on the device (weights and their gradients)
        ha = up.UPIPE_HOST_ACT
        wb = up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_BOTH, ha)
        wsh = torch.empty(wb, dtype=torch.uint8, device=dev)
        hh = torch.empty(h.shape, dtype=h.dtype, pin_memory=True)
        hh.copy_(h)
        dhh = torch.empty(h.shape, dtype=h.dtype, pin_memory=True)
        th = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        th.copy_(t)
        lossh = torch.empty(loss.shape, dtype=loss.dtype, pin_memory=True)

        def step():
            t.copy_(th, non_blocking=True)
            up.upipe_ce_fwd(hh, w, t, loss, lse, S, Dm, V, T, wsh, wb, stream)
            up.upipe_ce_bwd(hh, w, t, lse, g, dhh, dw, S, Dm, V, T, wsh, wb, stream)
            lossh.copy_(loss, non_blocking=True)
        return step, hh.nbytes + th.nbytes, dhh.nbytes + lossh.nbytes, wb, \
            "h in pinned host memory staged tile by tile by the library (dh likewise out); " \
            "targets in and the per-token loss out by the caller; w and dw on the device"

    def fused_measure(steps, warmup):
        # the one-call forward + backward for a dloss known up front: same results, no logits
        # recompute; timed on its own, same inputs
        wbf = up.upipe_ce_workspace_bytes(S, Dm, V, T, up.UPIPE_PASS_FUSED)
        wsf = torch.empty(wbf, dtype=torch.uint8, device=dev)

        def step():
            up.upipe_ce_fwd_bwd(h, w, t, g, loss, lse, dh, dw, S, Dm, V, T, wsf, wbf, stream)
        for _ in range(warmup):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        up.upipe_sync_status(stream)
        ms = e0.elapsed_time(e1) / steps
        executed = 3 * lw.flops_fwd()  # logits, dh and dw GEMMs
        return {"fused": {"ms_per_step": ms, "tokens_per_s": S / (ms / 1e3),
                          "tflops_executed": executed / (ms / 1e3) / 1e12,
                          "workspace_gb": wbf / 1e9,
                          "method": "upipe_ce_fwd_bwd: the forward keeps fp32 logits, dlogits "
                                    "from them (no recompute GEMM); TFLOP/s over the three "
                                    "GEMMs executed"}}

    return {
        "metric": LOSS_METRIC, "name": lw.name, "seq_tile": T, "host_setup": host_setup,
        "extra_measure": fused_measure,
        "fwd": lambda: up.upipe_ce_fwd(h, w, t, loss, lse, S, Dm, V, T, ws, ws_bytes, stream),
        "bwd": lambda: up.upipe_ce_bwd(h, w, t, lse, g, dh, dw, S, Dm, V, T, ws, ws_bytes, stream),
        "f_fwd": lw.flops_fwd(), "f_bwd": lw.flops_bwd(), "ws_bytes": ws_bytes,
        "data": "synthetic (seeded: h N(0,1), w N(0,%g/sqrt(Dm)) bf16, uniform targets, "
                "%.4f ignored)" % (lw.w_std, lw.ignore_frac),
        "config": {"workload": lw.name, "S": S, "Dm": Dm, "V": V, "seq_tile": T,
                   "l2": "inputs larger than L2 (w is %.2f GiB)" % (w.nbytes / 2**30)},
        "extra": {"untiled_logits_gb": S * V * 4 / 1e9},
        "inputs": (h, w, t, g), "outputs": (loss, lse, dh, dw),
        "cpu": lambda: loss_oracle_sample(lw, min(S, 32), (h, w, t, g)),
    }


def _mlp_spec(a, dev, up):
    from workloads import MLP_WORKLOADS, make_mlp_inputs
    import torch
    mw = MLP_WORKLOADS[a.workload]
    if a.seq_len:
        mw = mw.with_(S=a.seq_len, name=f"{mw.name}@S={a.seq_len}")
    T = a.seq_tile or mw.seq_tile
    S, Dm, F = mw.S, mw.Dm, mw.F
    x, w_gu, w_d, dy = (t.to(dev) for t in make_mlp_inputs(mw, str(dev) if mw.gen_device == "cuda"
                                                         else "cpu"))
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    dw_gu = torch.empty((2 * F, Dm), dtype=torch.float32, device=dev)
    dw_d = torch.empty((Dm, F), dtype=torch.float32, device=dev)
    ws_bytes = up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_BOTH)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def host_setup():
        # x and dy in, y and dx out, all through the library's tile staging; the weights and
        # their gradients stay on the device
        ha = up.UPIPE_HOST_ACT
        wb = up.upipe_mlp_workspace_bytes(S, Dm, F, T, up.UPIPE_PASS_BOTH, ha)
        wsh = torch.empty(wb, dtype=torch.uint8, device=dev)
        xh, dyh, yh, dxh = (torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
                            for _ in range(4))
        xh.copy_(x)
        dyh.copy_(dy)

        def step():
            up.upipe_mlp_fwd(xh, w_gu, w_d, yh, S, Dm, F, T, wsh, wb, stream)
            up.upipe_mlp_bwd(xh, w_gu, w_d, dyh, dxh, dw_gu, dw_d, S, Dm, F, T, wsh, wb, stream)
        return step, xh.nbytes + dyh.nbytes, yh.nbytes + dxh.nbytes, wb, \
            "x, dy in and y, dx out in pinned host memory, staged tile by tile by the library; " \
            "weights and their gradients on the device"

    return {
        "metric": MLP_METRIC, "name": mw.name, "seq_tile": T, "host_setup": host_setup,
        "fwd": lambda: up.upipe_mlp_fwd(x, w_gu, w_d, y, S, Dm, F, T, ws, ws_bytes, stream),
        "bwd": lambda: up.upipe_mlp_bwd(x, w_gu, w_d, dy, dx, dw_gu, dw_d, S, Dm, F, T, ws,
                                        ws_bytes, stream),
        "f_fwd": mw.flops_fwd(), "f_bwd": mw.flops_bwd(), "ws_bytes": ws_bytes,
        "data": "synthetic (seeded: x, dy N(0,1), w_gu N(0,1/sqrt(Dm)), w_d N(0,1/sqrt(F)) bf16)",
        "config": {"workload": mw.name, "S": S, "Dm": Dm, "F": F, "seq_tile": T,
                   "l2": "inputs larger than L2 (x is %.2f GiB)" % (x.nbytes / 2**30)},
        "extra": {"untiled_intermediates_gb": 5 * S * F * 2 / 1e9},
        "inputs": (x, w_gu, w_d, dy), "outputs": (y, dx, dw_gu, dw_d),
        "cpu": lambda: mlp_oracle_sample(mw, min(S, 256), (x, w_gu, w_d, dy)),
    }


def run_tiled(a, make_spec):
    """A sequence-tiled workload (loss or MLP) on one GPU (N replicas under torchrun)."""
    import torch
    import torch.distributed as dist

    import context_parallelism_gb300 as up

    rank, world, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sp = make_spec(a, dev, up)
    fwd, bwd = sp["fwd"], sp["bwd"]
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(a.warmup):
        fwd()
        bwd()
    up.upipe_sync_status(stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    up.upipe_profile_read()
    up.upipe_profile_enable(True)
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    time.sleep(0.3)
    launches0 = up.upipe_launch_count()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(a.steps):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    t1.record(stream)
    barrier()
    launches = up.upipe_launch_count() - launches0
    clk = clocks.stop()
    up.upipe_profile_enable(False)
    prof = up.upipe_profile_read()
    up.upipe_sync_status(stream)
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    f_fwd, f_bwd = sp["f_fwd"], sp["f_bwd"]
    red = torch_reduce_max(dev) if world > 1 else None
    value, t_max = job_throughput(t0.elapsed_time(t1), a.steps, f_fwd + f_bwd, world, red)
    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops_sustained") or peaks["bf16_tflops"])
    gemm_ms, gemm_n = prof["loss_gemm"]
    achieved = (f_fwd + f_bwd) * a.steps / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    roofline = {"kernel": "loss_gemm", "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak if achieved else None,
                "peak_source": f"{peak_src} bf16_tflops_sustained", "launches": gemm_n,
                "avg_launch_ms": gemm_ms / max(gemm_n, 1),
                "traffic": traffic_per_launch("loss_gemm", sp["name"], sp["seq_tile"], None),
                "traffic_unit": "bytes per launch"}
    kernels = {k: {"ms_per_step": tm / a.steps, "launches_per_step": n / a.steps}
               for k, (tm, n) in prof.items() if n}
    extra_measured = sp["extra_measure"](a.steps, a.warmup) if "extra_measure" in sp else {}
    if "fused" in extra_measured:
        extra_measured["fused"]["speedup_vs_two_calls"] = \
            (t_max / a.steps) / extra_measured["fused"]["ms_per_step"]
    config = dict(sp["config"])
    config["parallelism"] = "replicas" if world > 1 else "single"
    line = {
        "metric": sp["metric"], "value": value, "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": t_max / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": sp["data"], "config": config,
        "fwd_tflops": world * f_fwd * a.steps / (fwd_ms / 1e3) / 1e12,
        "bwd_tflops": world * f_bwd * a.steps / (bwd_ms / 1e3) / 1e12,
        "frac_of_bf16_peak": value / world / peak, "peak_tflops": peak,
        "workspace_gb": sp["ws_bytes"] / 1e9, **sp["extra"],
        "roofline": roofline, "kernels": kernels, "gpu_launches": int(launches), "clocks": clk,
        **extra_measured,
    }
    if not a.no_e2e and not a.no_explicit_copies:
        # host buffers in (every input), every output out, each step
        ins, outs_d = sp["inputs"], sp["outputs"]
        hh = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in ins]
        for src, dst in zip(ins, hh):
            dst.copy_(src)
        outs = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs_d]

        def e2e_step():
            for dst, src in zip(ins, hh):
                dst.copy_(src, non_blocking=True)
            fwd()
            bwd()
            for dst, src in zip(outs, outs_d):
                dst.copy_(src, non_blocking=True)

        e2e_step()
        barrier()
        t0.record(stream)
        for _ in range(a.steps):
            e2e_step()
        t1.record(stream)
        barrier()
        explicit_value, _ = job_throughput(t0.elapsed_time(t1), a.steps, f_fwd + f_bwd, world,
                                           red)
        explicit = {"value": explicit_value,
                    "h2d_bytes_per_step": int(sum(x.nbytes for x in hh)),
                    "d2h_bytes_per_step": int(sum(x.nbytes for x in outs)),
                    "method": "every input (weights included) copied in from pinned host memory "
                              "and every output copied out, on the compute stream, around "
                              "device-buffer calls"}
        del hh, outs
    else:
        explicit = None
    if not a.no_e2e:
        # the step through the library with the activations in pinned host memory
        host_step, h2d, d2h, wb, method = sp["host_setup"]()
        host_step()
        barrier()
        t0.record(stream)
        for _ in range(a.steps):
            host_step()
        t1.record(stream)
        barrier()
        e2e_value, _ = job_throughput(t0.elapsed_time(t1), a.steps, f_fwd + f_bwd, world, red)
        line["e2e"] = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                       "d2h_bytes_per_step": int(d2h), "method": method,
                       "workspace_gb": wb / 1e9, "explicit_copies": explicit}
        up.upipe_sync_status(stream)
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        tf, dt, desc, cores = sp["cpu"]()
        line["cpu_baseline"] = {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def mlp_oracle_sample(mw, S_sample, inputs):
    """Times the fp64 oracle's MLP forward + backward on the first S_sample tokens."""
    import oracle
    x, w_gu, w_d, dy = inputs
    xs, dys = x[:S_sample].cpu(), dy[:S_sample].cpu()
    flops = mw.with_(S=S_sample).flops_fwd() + mw.with_(S=S_sample).flops_bwd()
    t0 = time.perf_counter()
    oracle.mlp_bwd_ref(xs, w_gu.cpu(), w_d.cpu(), dys)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = (f"fp64 numpy oracle MLP fwd+bwd on the first {S_sample} of {mw.S} tokens, width "
            f"{mw.Dm}, hidden {mw.F}; FLOPs by the same convention")
    return flops / dt / 1e12, dt, desc, cores


def run_mlp_reference(a):
    """Reference arm for the MLP workloads: the fp64 oracle on the host cores, rank 0 only."""
    rank, _, _ = _dist()
    if rank != 0:
        return
    from workloads import MLP_WORKLOADS, make_mlp_inputs
    mw = MLP_WORKLOADS[a.workload]
    S_sample = min(mw.S, 256)
    inputs = make_mlp_inputs(mw.with_(S=S_sample, gen_device="cpu"), "cpu")
    vals = []
    for i in range(a.warmup + a.steps):
        tf, dt, desc, cores = mlp_oracle_sample(mw, S_sample, inputs)
        if i >= a.warmup:
            vals.append(dt)
    flops = mw.with_(S=S_sample).flops_fwd() + mw.with_(S=S_sample).flops_bwd()
    value = flops * len(vals) / sum(vals) / 1e12
    print(json.dumps({
        "impl": "reference", "metric": MLP_METRIC, "value": value, "unit": UNIT,
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": 1000.0 * statistics.mean(vals), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": mw.name, "S": mw.S, "Dm": mw.Dm, "F": mw.F,
                   "seq_tile": a.seq_tile or mw.seq_tile, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + " (recipe regenerated on the CPU at the sample length)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_loss_reference(a):
    """Reference arm for the loss workloads: the fp64 oracle on the host cores, rank 0 only."""
    rank, _, _ = _dist()
    if rank != 0:
        return
    from workloads import LOSS_WORKLOADS, make_loss_inputs
    lw = LOSS_WORKLOADS[a.workload]
    S_sample = min(lw.S, 32)
    inputs = make_loss_inputs(lw.with_(S=S_sample, gen_device="cpu"), "cpu")
    # the sample regenerates the recipe at the sample length: same shapes and distributions
    vals = []
    for i in range(a.warmup + a.steps):
        tf, dt, desc, cores = loss_oracle_sample(lw, S_sample, inputs)
        if i >= a.warmup:
            vals.append(dt)
    flops = lw.with_(S=S_sample).flops_fwd() + lw.with_(S=S_sample).flops_bwd()
    value = flops * len(vals) / sum(vals) / 1e12
    line = {
        "impl": "reference", "metric": LOSS_METRIC, "value": value, "unit": UNIT,
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": 1000.0 * statistics.mean(vals), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": lw.name, "S": lw.S, "Dm": lw.Dm, "V": lw.V,
                   "seq_tile": a.seq_tile or lw.seq_tile, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc + " (recipe regenerated on the CPU at the sample length)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    a = _args()
    from workloads import LOSS_WORKLOADS, MLP_WORKLOADS
    if a.workload in LOSS_WORKLOADS:
        if a.impl == "reference":
            run_loss_reference(a)
        else:
            run_tiled(a, _loss_spec)
        return
    if a.workload in MLP_WORKLOADS:
        if a.impl == "reference":
            run_mlp_reference(a)
        else:
            run_tiled(a, _mlp_spec)
        return
    if a.sweep:
        run_sweep(a)
        return
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
