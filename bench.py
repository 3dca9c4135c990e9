"""Benchmark of the Mesh-Attention hot path on GB300: one step = tile forward over every
(Q partition, tile) item of the plan + LSE merge, on a synthetic workload resident in HBM.

Prints one JSON line (rank 0).  Default workload: the largest single-GPU configuration, the
merge-heavy long-context stress case: bf16 causal, B=1, Hq=16, Hkv=4, S=262144, d=128, K rows
scaled by 4, P=1024 partitions of 256 tokens on a 32x32 mesh with KV Partition Rotation and
greedy order (68 GB of fp32 partials).  The backward pass is measured beside it on the bf16
causal 16K workload.  `--impl reference` times the fp64 CPU oracle on the host cores instead.
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mesh_inputs import WORKLOADS, make_do, make_qkv, sample_rows  # noqa: E402

METRIC = "mesh-tiled attention fwd TFLOP/s & % bf16 tensor peak; merge HBM GB/s (1 GB300)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algorithmic_flops(w) -> float:
    """4 d per visible (query, key) pair: QK^T and PV, 2 flops per multiply-add each."""
    pairs = w.S * (w.S + 1) // 2 if w.causal else w.S * w.S
    return 4.0 * w.d * w.B * w.Hq * pairs


def executed_flops_fwd(m, plan, w) -> float:
    """Flops the bf16 tile kernel's products execute: full 128 x 128 blocks, including the masked
    half of causal diagonal blocks and the padding of a ragged last block (a diagnostic beside
    the algorithmic count).  A unit is a pair of 128-row query tiles of one work item, and it
    visits every 128-key block of the item's KV partitions up to its last tile on the causal
    diagonal partition."""
    items, _, kvs = m.mesh_attn_plan_order(plan)
    nb = -(-w.L // 128)
    per_item = 0
    for (p, _t, _slot), kl in zip(items, kvs):
        for a0 in range(0, nb, 2):
            ntiles = min(2, nb - a0)
            a_max = a0 + ntiles - 1
            blocks = sum(min(nb, a_max + 1) if (w.causal and k == p) else nb for k in kl)
            per_item += blocks * ntiles
    return 4.0 * 128 * 128 * w.d * per_item * w.B * w.Hq


def sample_flops(w, rows: np.ndarray) -> float:
    vis = (rows + 1).sum() if w.causal else rows.size * w.S
    return 4.0 * w.d * float(vis)


def rows_for_budget(w, flops_budget: float) -> int:
    """Seeded rows per head whose oracle work (4 d per visible pair, every head) is about
    flops_budget: a bounded sample of the workload for the CPU timing."""
    avg_vis = (w.S + 1) / 2 if w.causal else w.S
    n = int(flops_budget / (4.0 * w.d * avg_vis * w.Hq * w.B))
    return max(16, min(w.S, 4096, n))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                val = line.split(":", 1)[1].strip()
                if val and not val.isdigit():
                    return val
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def merge_bytes(w, n_slots: int) -> float:
    es = 2 if w.dtype == "bf16" else 4
    read = n_slots * w.L * w.Hq * w.B * (4 * w.d + 4)
    write = w.B * w.Hq * w.S * (es * w.d + 4)
    return float(read + write)


def kernel_sources(w):
    """Source files whose content the tile kernel's DRAM counters describe: the kernel, its
    inline-PTX helpers and the planner (it fixes the launch order of the work items)."""
    return ("tile_fwd_tc.cu", "ptx.cuh", "planner.cpp")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while the timed region runs (the
    sampler's first sample is awaited before the region starts)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 3.0 and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(x: float, device) -> float:
    """Largest value of x over all ranks (the job's time is its slowest rank's)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_throughput(world: int, flops_per_rank: float, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own copy of the workload (weak scaling)."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


_INPUTS = {}


def time_oracle(w, n_rows: int, heads, threads: int, qkv=None):
    """fp64 oracle on n_rows seeded rows of the given heads (batch 0); returns (seconds, algorithmic
    flops, {head: (rows, O, LSE)})."""
    from oracle.attention import attention_rows, default_scale
    torch.set_num_threads(threads)
    if (w.name, n_rows) not in _INPUTS:
        _INPUTS[(w.name, n_rows)] = (qkv if qkv is not None else make_qkv(w), sample_rows(w, n_rows))
    (q, k, v), rows = _INPUTS[(w.name, n_rows)]
    g = w.Hq // w.Hkv
    t0 = time.perf_counter()
    fl = 0.0
    out = {}
    for h in heads:
        pos = torch.as_tensor(rows[0, h])
        o, lse = attention_rows(q[0, h].double()[pos], pos, k[0, h // g], v[0, h // g], default_scale(w.d), w.causal)
        fl += sample_flops(w, rows[0, h])
        out[h] = (rows[0, h], o, lse)
    return time.perf_counter() - t0, fl, out


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    # about 1.5e10 oracle flops (well under a second of host time) per step, at most 256 rows
    avg_vis = (w.S + 1) / 2 if w.causal else w.S
    rows_per_step = max(16, min(256, int(1.5e10 / (4.0 * w.d * avg_vis))))
    for i in range(args.warmup):
        time_oracle(w, rows_per_step, [i % w.Hq], threads)
    secs, fl = 0.0, 0.0
    for i in range(args.steps):
        s, f, _ = time_oracle(w, rows_per_step, [i % w.Hq], threads)
        secs += s
        fl += f
    value = fl / secs / 1e12
    sample = f"{rows_per_step} seeded query rows of one head per step (head cycles), fp64 oracle, full key range"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def counted_volumes(m, w):
    """Per-device receive bytes a real mesh (KVR) and a plain ring would move for this workload,
    counted by the planner (no communication happens on one GPU)."""
    mesh = m.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
    _, byts, ring_kv = m.mesh_attn_plan_volumes(mesh, w.Hq, w.Hkv, w.d,
                                                torch.bfloat16 if w.dtype == "bf16" else torch.float32)
    per_dev = [sum(b) for b in byts]
    mx = max(per_dev) if per_dev else 0
    return {"mesh_max_recv_bytes": mx, "mesh_mean_recv_bytes": sum(per_dev) / max(1, len(per_dev)),
            "ring_recv_bytes": ring_kv, "reduction_vs_ring": (1 - mx / ring_kv) if ring_kv else None}


def run_e2e(m, w, args, q, k, v, dev, flops, world, barrier):
    """End to end through the public call with host buffers.  Every step copies its Q, K and V
    from pinned host memory to the device, runs the whole path (plan, tile forward, merge:
    mesh_attention) and copies O and LSE back to pinned host memory.

    Steps are software-pipelined over three streams with two buffer sets, the way a serving
    loop would run them: the input copy of step i+1 and the output copy of step i-1 overlap
    the compute of step i.  The serial variant (copy in, compute, copy out on one stream) is
    reported beside it."""
    n = max(3, min(args.steps, 20))
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    Oh = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(2)]
    Lh = [torch.empty((w.B, w.Hq, w.S), dtype=torch.float32, pin_memory=True) for _ in range(2)]
    dq = [torch.empty(q.shape, dtype=q.dtype, device=dev) for _ in range(2)]
    dk = [torch.empty(k.shape, dtype=k.dtype, device=dev) for _ in range(2)]
    dv = [torch.empty(v.shape, dtype=v.dtype, device=dev) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def make_plan():
        return (m.mesh_attn_plan_create_ring(w.S, w.P, w.causal) if args.plan == "ring"
                else m.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy))

    def pipelined(steps):
        for i in range(steps):
            b = i % 2
            if i >= 2:
                s_in.wait_event(comp_done[b])  # step i-2 no longer reads input set b
            with torch.cuda.stream(s_in):
                dq[b].copy_(qh, non_blocking=True)
                dk[b].copy_(kh, non_blocking=True)
                dv[b].copy_(vh, non_blocking=True)
                h2d_done[b].record(s_in)
            s_comp.wait_event(h2d_done[b])
            if i >= 2:
                s_comp.wait_event(d2h_done[b])  # host output set b has been written back
            with torch.cuda.stream(s_comp):
                Od, Ld = m.mesh_attention(dq[b], dk[b], dv[b], w.P, w.causal, plan=make_plan(), check_status=False)
                comp_done[b].record(s_comp)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                Oh[b].copy_(Od, non_blocking=True)
                Lh[b].copy_(Ld, non_blocking=True)
                d2h_done[b].record(s_out)
            Od.record_stream(s_out)
            Ld.record_stream(s_out)

    def serial(steps):
        for _ in range(steps):
            a, b_, c = qh.to(dev, non_blocking=True), kh.to(dev, non_blocking=True), vh.to(dev, non_blocking=True)
            Od, Ld = m.mesh_attention(a, b_, c, w.P, w.causal, plan=make_plan(), check_status=False)
            Oh[0].copy_(Od, non_blocking=True)
            Lh[0].copy_(Ld, non_blocking=True)

    def timed(fn, steps):
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        fn(steps)
        torch.cuda.synchronize()
        ms = (time.perf_counter() - t0) * 1e3 / steps
        barrier()
        return max_over_ranks(ms, dev)

    pipelined(max(2, args.warmup))
    serial(1)
    torch.cuda.synchronize()
    p_ms = timed(pipelined, n)
    s_ms = timed(serial, n)
    es = q.element_size()
    return {"value": job_throughput(world, flops, p_ms), "unit": UNIT,
            "h2d_bytes_per_step": int((q.numel() + k.numel() + v.numel()) * es),
            "d2h_bytes_per_step": int(q.numel() * es + w.B * w.Hq * w.S * 4),
            "ms_per_step": p_ms, "steps": n, "timing": "host wall clock around synchronised steps",
            "schedule": "3 streams, 2 buffer sets: copy-in of step i+1 and copy-out of step i-1 overlap step i",
            "serial_value": job_throughput(world, flops, s_ms), "serial_ms_per_step": s_ms}


def run_backward(m, w, dev, args, stream):
    """Time the backward pass (D = dO . O, tile backward, reduce) with CUDA events, inputs resident,
    on workload w (its own inputs; the forward's O and LSE come from one untimed forward call).

    Algorithmic flops of the tile backward: the four gradient products dP = dO V^T, dV = P^T dO,
    dQ = dS K, dK = dS^T Q over the visible pairs = 2x the forward's; the kernels also recompute
    S (dK/dV kernel) and S, dP (dQ kernel): executed = 3.5x the forward's.
    """
    flops = algorithmic_flops(w)
    q, k, v = make_qkv(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    del q, k, v
    plan = m.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
    O, LSE = m.mesh_attention(qd, kd, vd, w.P, w.causal, plan=plan)
    dO = make_do(w).to(dev)
    dq_p, dk_p, dv_p = m.new_bwd_partials(plan, w.B, w.Hq, w.Hkv, w.d, dev)
    wsb = m.new_bwd_workspace(plan, dev)
    st = m.new_status(dev)
    D = torch.empty(w.B, w.Hq, w.S, dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)

    def bstep(ev=None):
        if ev is not None:
            ev[0].record(stream)
        m.mesh_attn_bwd_prep(O, dO, D, st, stream)
        if ev is not None:
            ev[1].record(stream)
        m.mesh_attn_tile_bwd(plan, qd, kd, vd, dO, LSE, D, None, dq_p, dk_p, dv_p, wsb, st, stream)
        if ev is not None:
            ev[2].record(stream)
        m.mesh_attn_bwd_reduce(plan, w.B, w.Hq, w.Hkv, w.d, dq_p, dk_p, dv_p, dQ, dK, dV, wsb, st, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(1, min(args.warmup, 3))):
        bstep()
    steps = max(1, args.steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        bstep(evs[i])
    torch.cuda.synchronize()
    code = m.mesh_attn_read_status(st, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} in the backward pass: {st.tolist()}")
    prep_ms, tile_ms, red_ms = (sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps for j in range(3))
    peaks, _ = load_peaks()
    es = 2 if w.dtype == "bf16" else 4
    alg = 2 * flops
    tflops = alg / (tile_ms * 1e-3) / 1e12
    nq, nkv = m.mesh_attn_bwd_partials_size(plan, w.B, w.Hq, w.Hkv, w.d)
    red_bytes = 4.0 * (nq + 2 * nkv) + es * (w.B * w.Hq * w.S * w.d + 2 * w.B * w.Hkv * w.S * w.d)
    prep_bytes = 2.0 * es * w.B * w.Hq * w.S * w.d + 4.0 * w.B * w.Hq * w.S
    line = {"workload": w.name, "ms_per_step": prep_ms + tile_ms + red_ms, "steps": steps,
            "tile_bwd_ms": tile_ms, "prep_ms": prep_ms, "reduce_ms": red_ms,
            "flops_per_step": alg, "tflops": tflops, "unit": "TFLOP/s",
            "executed_tflops": 3.5 * flops / (tile_ms * 1e-3) / 1e12,
            "reduce_gbs": red_bytes / (red_ms * 1e-3) / 1e9, "prep_gbs": prep_bytes / (prep_ms * 1e-3) / 1e9}
    if w.dtype == "bf16":
        line["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": tflops / peaks["bf16_tflops"], "traffic": None,
                            "kernel": "bwd_dkdv_kernel + bwd_dq_kernel"}
        if peaks.get("bf16_tflops_sustained"):
            line["roofline"]["frac_of_sustained"] = tflops / peaks["bf16_tflops_sustained"]
    return line


def workload_config(w, plan="mesh"):
    return {"workload": w.name, "plan": plan, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "d": w.d, "in_dtype": w.dtype,
            "causal": w.causal, "P": w.P, "mesh": f"{w.R}x{w.R}", "kvr": w.kvr, "greedy": w.greedy,
            "k_scale": w.k_scale, "l2": "inputs and partials larger than L2 (no flush)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="stress_256k", choices=sorted(WORKLOADS))
    ap.add_argument("--backward-workload", default="bf16_causal_16k", choices=sorted(WORKLOADS),
                    help="workload of the backward-pass object of the line")
    ap.add_argument("--in-dtype", default=None, choices=["bf16", "f32"],
                    help="override the workload's input dtype (f32 runs the three-piece tensor-core path)")
    ap.add_argument("--plan", default="mesh", choices=["mesh", "ring"],
                    help="tile assignment: sqrt(P) x sqrt(P) mesh with KVR (default) or Ring-Attention rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward-pass measurement")
    ap.add_argument("--wait-limit-ns", type=int, default=None,
                    help="bound on every device-side wait (default 2e9); raise it for runs under a profiler, "
                         "whose replay passes can slow a kernel by orders of magnitude")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]
    if args.in_dtype is not None and args.in_dtype != w.dtype:
        w = w.with_(dtype=args.in_dtype, name=f"{w.name}_{args.in_dtype}")
    if args.impl == "reference":
        return run_reference(args, w)

    import tiled_distributed_attention_gb300 as m
    m.load_library()
    if args.wait_limit_ns is not None:
        m.mesh_attn_set_wait_limit_ns(args.wait_limit_ns)
    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    q, k, v = make_qkv(w)

    # cpu baseline first (before any GPU work is queued), rank 0 at N=1 only: the fp64 oracle on
    # a bounded sample of seeded rows of every head (about 2.5e11 flops, 10-20 s on the host);
    # its outputs also give the line's parity check of the timed path on those rows
    cpu_base, ref_rows = None, None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        n_rows = rows_for_budget(w, 2.5e11)
        secs, fl, ref_rows = time_oracle(w, n_rows, range(w.Hq), threads, qkv=(q, k, v))
        full = algorithmic_flops(w)
        cpu_base = {"value": fl / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
                    "cpu_model": cpu_model(),
                    "sample": f"{n_rows} seeded query rows x {w.Hq} heads of batch 0 of the workload (forced rows "
                              f"0, S-1 and partition edges), full key range, fp64, {secs:.1f} s",
                    "sample_seconds": secs, "sample_flops": fl,
                    "extrapolated_full_s": secs * full / fl,
                    "extrapolation": "extrapolated: sample time x (visible pairs of the whole workload / visible "
                                     "pairs of the sampled rows)"}

    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if args.plan == "ring":
        plan = m.mesh_attn_plan_create_ring(w.S, w.P, w.causal)
    else:
        plan = m.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy)
    # host time to build the plan (tiles, greedy order, slot lists): reported, not in the step
    t_plan = time.perf_counter()
    (m.mesh_attn_plan_create_ring(w.S, w.P, w.causal) if args.plan == "ring"
     else m.mesh_attn_plan_create(w.S, w.P, w.causal, w.kvr, w.greedy))
    plan_ms = (time.perf_counter() - t_plan) * 1e3
    po, pl = m.new_partials(plan, w.B, w.Hq, w.d, dev)
    wsp = m.new_workspace(plan, dev, qd, kd)
    st = m.new_status(dev)
    O = torch.empty_like(qd)
    LSE = torch.empty(w.B, w.Hq, w.S, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        m.mesh_attn_tile_fwd(plan, qd, kd, vd, None, po, pl, wsp, st, stream)
        if ev is not None:
            ev[1].record(stream)
        m.mesh_attn_merge(plan, w.B, w.Hq, w.d, po, pl, O, LSE, wsp, st, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    code = m.mesh_attn_read_status(st, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} during warm-up: {st.tolist()}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    code = m.mesh_attn_read_status(st, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} in the timed region: {st.tolist()}")
    total_ms = t_start.elapsed_time(t_end)
    tile_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    merge_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / args.steps
    flops = algorithmic_flops(w)
    value = job_throughput(ws, flops, ms_per_step)

    # parity of the timed path's output on the oracle's sampled rows
    parity = None
    if ref_rows is not None:
        to, tl = (2e-2, 1e-3) if w.dtype == "bf16" else (1e-4, 1e-4)
        eo = el = 0.0
        finite = True
        for h, (rows_h, o_ref, l_ref) in ref_rows.items():
            idx = torch.as_tensor(rows_h, device=dev)
            og = O[0, h].index_select(0, idx).double().cpu()
            lg = LSE[0, h].index_select(0, idx).double().cpu()
            finite = finite and bool(torch.isfinite(og).all()) and bool(torch.isfinite(lg).all())
            eo = max(eo, (og - o_ref).abs().max().item())
            el = max(el, (lg - l_ref).abs().max().item())
        parity = {"rows": f"{len(next(iter(ref_rows.values()))[0])} seeded rows x {len(ref_rows)} heads (batch 0), "
                          "the cpu_baseline sample", "max_abs_err_O": eo, "max_abs_err_LSE": el,
                  "tol_O": to, "tol_LSE": tl, "pass": finite and eo <= to and el <= tl}
    del po, pl, O, LSE
    torch.cuda.empty_cache()

    # backward pass on its own workload (a separate object of the line; not part of `value`)
    bwd = None
    if not args.no_backward:
        bwd = run_backward(m, WORKLOADS[args.backward_workload], dev, args, stream)
        torch.cuda.empty_cache()

    # end to end through the public call, host buffers in pinned memory
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(m, w, args, q, k, v, dev, flops, ws, barrier)

    if rank != 0:
        return
    peaks, peak_kind = load_peaks()
    tile_tflops = flops / (tile_ms * 1e-3) / 1e12
    mbytes = merge_bytes(w, plan.n_slots)
    merge_gbs = mbytes / (merge_ms * 1e-3) / 1e9
    traffic, traffic_note = None, None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        import hashlib
        with open(prof) as f:
            rec = json.load(f).get(w.name, {}).get("tile_fwd")
        h = hashlib.sha256()
        for name in kernel_sources(w):  # the kernel, its inline-PTX helpers and the planner's order
            with open(os.path.join(ROOT, "tiled_distributed_attention_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()
        # counters only describe the kernel they were taken on
        if rec and sha.startswith(rec["source_sha256_prefix"]):
            traffic = rec["bytes"]
            traffic_note = rec.get("note")
    # A timed region of a second or more runs the tile kernel back to back under the power cap:
    # its denominator is then the sustained (seconds-long) GEMM rate, else the burst rate.
    sustained = total_ms >= 1000.0 and bool(peaks.get("bf16_tflops_sustained"))
    peak_bf16 = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    if w.dtype == "bf16":
        roof = {"bound": "tensor", "achieved": tile_tflops, "peak": peak_bf16, "unit": "TFLOP/s",
                "frac": tile_tflops / peak_bf16, "traffic": traffic,
                "kernel": "tile_fwd_tc_kernel",
                "peak_kind": f"{peak_kind} bf16 dense {'sustained' if sustained else 'burst'}",
                "frac_of_burst": tile_tflops / peaks["bf16_tflops"]}
        if peaks.get("bf16_tflops_sustained"):
            roof["frac_of_sustained"] = tile_tflops / peaks["bf16_tflops_sustained"]
        if traffic_note:
            roof["traffic_source"] = traffic_note
        exe = executed_flops_fwd(m, plan, w)
        roof["executed_tflops"] = exe / (tile_ms * 1e-3) / 1e12  # full blocks, masked halves included
        roof["executed_over_algorithmic"] = exe / flops
        launches_per_step = 2  # tile, merge
    else:
        # fp32 inputs: every product is six bf16 tensor-core products of the operands' exact
        # three-piece split, so the ceiling for the fp32 rate is the bf16 peak / 6
        peak32 = peak_bf16 / 6
        roof = {"bound": "tensor", "achieved": tile_tflops, "peak": peak32, "unit": "TFLOP/s",
                "frac": tile_tflops / peak32, "traffic": None,
                "kernel": "split_kernel + tile_fwd_tc32_kernel",
                "peak_kind": f"{peak_kind} bf16 dense {'sustained' if sustained else 'burst'} / 6 "
                             "(six bf16 products per fp32 product)"}
        launches_per_step = 3  # split, tile, merge
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": workload_config(w, args.plan),
        "roofline": roof,
        "merge": {"bound": "hbm", "achieved": merge_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                  "frac": merge_gbs / peaks["hbm_gbs"], "bytes_per_launch": mbytes, "ms": merge_ms},
        "tile_fwd_ms": tile_ms, "merge_ms": merge_ms, "plan_ms": plan_ms, "backward": bwd,
        "comm_counted": counted_volumes(m, w),
        "parity": parity, "cpu_baseline": cpu_base, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
