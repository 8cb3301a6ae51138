#!/usr/bin/env python
"""Benchmark of the GB300 exact attention forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

One step is one fused attention forward over the benchmark workload
(default: B=2, H=16, N=8192, d=128, bf16, non-causal), with Q, K, V already
resident in HBM.  The timed region holds exactly K launches, bracketed by a
barrier and a device synchronisation; the inputs plus output (256 MiB) exceed
the 129 MB L2, so steps do not reuse a warm cache.  Rank 0 prints one JSON line.

Also measured in the same run (each in its own timed loop): the FP8 E4M3 path
(attention alone, and preparation + attention) on the 8192-token FP8 workload,
the other bf16 workloads, an end-to-end figure through the same C ABI with
pinned host buffers (host-to-device copies of Q, K, V and device-to-host copies
of O and lse inside the timed region), and the CPU oracle on a bounded sample
of the workload.

With --impl reference the float64 CPU oracle is timed instead (all host
cores), on bounded samples of the same workload; only rank 0 works.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path shards over independent (batch, head) slices with no exchange), value is
the sum over ranks using the slowest rank's time.
"""
from __future__ import annotations

import os

# The CPU oracle runs in a thread pool; keep each BLAS call single-threaded so
# the pool size is the number of cores actually used.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")

import argparse
import concurrent.futures
import json
import math
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16, FP8) and fraction of GB300 tensor peak"
UNIT = "TFLOP/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i] == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def kernel_source_hash() -> str:
    """Hash of the attention kernel sources; an ncu summary records the hash of
    the sources it was taken on, so stale counters are never reported."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_forward_fwd_gb300", "csrc")
    for name in ("attn_kernel.cuh", "ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(name):
    """DRAM bytes per launch from profiles/<name>.md ('dram_bytes_per_launch:' and
    'kernel_source_hash:' lines), or None if absent or taken on other sources."""
    import re
    path = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != kernel_source_hash():
        return None
    return float(m_b.group(1))


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The slowest rank's time: all-reduce MAX (NCCL on CUDA tensors, gloo on CPU)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, ms_max: float, world_size: int) -> float:
    """Replicas: every rank runs the same workload; the job's throughput is the
    units of all ranks over the slowest rank's time."""
    return flops_per_rank * world_size / (ms_max * 1e-3) / 1e12


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws == 1:
        return 0, 1, 0, None
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    return rank, ws, local, dist


def _time_loop(fn, steps, stream):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps   # ms per step


def _flushed_times(fn, steps, stream, flush):
    """ms of fn for each of `steps` launches, each timed alone after a write of
    `flush` (larger than L2) so that no launch finds its inputs in L2."""
    import torch
    out = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def _oracle_run(q, k, v, w, heads, threads):
    """Time the float64 oracle on every query row of the listed (b, h) slices of
    the workload's own inputs (CPU bf16 tensors); returns (seconds, flops)."""
    import numpy as np
    from oracle import attention as oa
    f64 = lambda t: t.float().numpy().astype(np.float64)
    rows = np.arange(w.N)
    chunk = 256
    jobs = [(b, h, rows[i:i + chunk]) for (b, h) in heads for i in range(0, w.N, chunk)]
    vis = (rows + 1) if w.causal else np.full(rows.shape, w.N)
    flops = 4.0 * w.d * float(vis.sum()) * len(heads)
    slices = {(b, h): (f64(q[b, h]), f64(k[b, h]), f64(v[b, h])) for (b, h) in heads}
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda j: oa.three_pass_rows(*slices[(j[0], j[1])], w.scale, w.causal, j[2]),
                    jobs))
    return time.perf_counter() - t0, flops


def _oracle_full(q, k, v, w, threads):
    """The float64 oracle on every row of every head of the workload (CPU bf16
    tensors), threaded over (b, h, 256-row chunks).  Returns (O, lse, seconds)."""
    import numpy as np
    from oracle import attention as oa
    f64 = lambda t: t.float().numpy().astype(np.float64)
    group = w.H // w.kv_heads
    qs = {(b, h): f64(q[b, h]) for b in range(w.B) for h in range(w.H)}
    kvs = {(b, g): (f64(k[b, g]), f64(v[b, g])) for b in range(w.B) for g in range(w.kv_heads)}
    O = np.zeros((w.B, w.H, w.N, w.d))
    L = np.zeros((w.B, w.H, w.N))
    rows = np.arange(w.N)
    jobs = [(b, h, rows[i:i + 256]) for b in range(w.B) for h in range(w.H)
            for i in range(0, w.N, 256)]

    def one(j):
        b, h, r = j
        kk, vv = kvs[(b, h // group)]
        o, l = oa.three_pass_rows(qs[(b, h)], kk, vv, w.scale, w.causal, r, w.window)
        O[b, h, r[0]:r[-1] + 1] = o
        L[b, h, r[0]:r[-1] + 1] = l

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, jobs))
    return O, L, time.perf_counter() - t0


def _errors(o, lse, O_ref, L_ref, fp8=False):
    """Error statistics of a GPU result against the oracle (all rows)."""
    import numpy as np
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - O_ref)
    out = {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
           "rmse": float(np.sqrt((err ** 2).mean())),
           "rel_rmse": float(np.sqrt((err ** 2).mean() / (O_ref ** 2).mean())),
           "lse_max_abs": float(np.abs(lse - L_ref).max()), "rows": "all"}
    if not fp8:
        import torch
        Ob = torch.from_numpy(O_ref).to(torch.bfloat16).double().numpy()
        out["bf16_rounding_floor_mean_abs"] = float(np.abs(Ob - O_ref).mean())
        out["gates"] = "max abs <= 1e-2 beyond bf16 output rounding, mean abs <= 1e-3, lse <= 1e-3"
    else:
        out["gates"] = "rmse <= 3e-2 against the oracle on the unquantised inputs"
    return out


def _ideal_bytes(w):
    """Q, K, V read once, O and lse written once (FP8: 1-byte operands and the
    three tensors' block scales)."""
    q_el = w.B * w.H * w.N * w.d
    kv_el = w.B * w.kv_heads * w.N * w.d
    if w.dtype == "fp8":
        nblk = -(-w.N // 128)
        return q_el + 2 * kv_el + 2 * q_el + 4 * w.B * w.H * w.N + 3 * 4 * w.B * w.H * nblk
    return 2 * (q_el + 2 * kv_el) + 2 * q_el + 4 * w.B * w.H * w.N


def run_reference(args):
    from exact_attention_forward_fwd_gb300 import inputs
    rank, ws, _, dist = _dist()
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    q, k, v = inputs.workload_inputs(w)
    threads = os.cpu_count() or 1
    all_heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    per_step = 2
    times, flops = [], 0.0
    for i in range(args.warmup + args.steps):
        heads = [all_heads[(per_step * i + j) % len(all_heads)] for j in range(per_step)]
        t, f = _oracle_run(q, k, v, w, heads, threads)
        if i >= args.warmup:
            times.append(t)
            flops += f
    total = sum(times)
    value = flops / total / 1e12
    sample = (f"{per_step} (batch, head) slices x all {w.N} query rows of {w.name} per step "
              f"(float64 three-pass oracle)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                                         "d": w.d, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_mine(args):
    import torch
    import exact_attention_forward_fwd_gb300 as ga
    from exact_attention_forward_fwd_gb300 import build, inputs

    rank, ws, local, dist = _dist()
    torch.cuda.set_device(local)
    if dist is not None:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    ga.lib()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks = _peaks()
    w = inputs.WORKLOADS[args.workload]

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    mor = lambda x: max_over_ranks(x, dist, dev)

    # ---------------------------------------------------------------- main
    qh, kh, vh = inputs.workload_inputs(w)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    step = lambda: ga.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
    for _ in range(args.warmup):
        step()
    barrier()
    with ClockSampler(local) as clk:
        ms = _time_loop(step, args.steps, stream)
    barrier()
    if ga.device_status() != 0:
        raise RuntimeError("kernel status word set during the benchmark")
    ms = mor(ms)
    tflops_launch = w.flops / (ms * 1e-3) / 1e12
    value = whole_job_tflops(w.flops, ms, ws)
    # The same launch timed alone after an L2 flush (a 256 MiB write), median
    # of at least 20: the method the scope table states, next to the mean of
    # back-to-back launches above.
    flush0 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ts_main = _flushed_times(step, max(20, args.steps), stream, flush0)
    del flush0
    ms_flushed = mor(statistics.median(ts_main))

    # ---------------------------------------------------------------- e2e
    # End to end through the public API: every step uploads its Q, K, V from
    # pinned host memory, runs attn_fwd and downloads its O and lse.  Steps are
    # pipelined over two device buffer sets and three streams (upload, compute,
    # download): the upload of step i+1 and the download of step i-1 overlap the
    # compute of step i.  The timed interval runs from before the first upload to
    # after the last download.
    qp, kp, vp = (t.pin_memory() for t in (qh, kh, vh))
    qb = [q, torch.empty_like(q)]
    kb = [k, torch.empty_like(k)]
    vb = [v, torch.empty_like(v)]
    ob = [o, torch.empty_like(o)]
    lb = [lse, torch.empty_like(lse)]
    op = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    lp = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
    s_up, s_comp, s_down = (torch.cuda.Stream(dev) for _ in range(3))
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_up):
                if i >= 2:
                    s_up.wait_event(comp_done[b])       # step i-2 no longer reads slot b
                qb[b].copy_(qp, non_blocking=True)
                kb[b].copy_(kp, non_blocking=True)
                vb[b].copy_(vp, non_blocking=True)
                up_done[b].record(s_up)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(up_done[b])
                if i >= 2:
                    s_comp.wait_event(down_done[b])     # step i-2's result was read back
                ga.attn_fwd(qb[b], kb[b], vb[b], causal=w.causal, scale=w.scale, out=ob[b], lse=lb[b])
                comp_done[b].record(s_comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(comp_done[b])
                op[b].copy_(ob[b], non_blocking=True)
                lp[b].copy_(lb[b], non_blocking=True)
                down_done[b].record(s_down)

    e2e_steps(2)
    torch.cuda.synchronize(dev)
    barrier()
    # Enough steps that filling and draining the three-stage pipeline (about one
    # step's latency) is a small part of the timed interval.
    n_e2e = max(20, args.steps)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_up)
    e2e_steps(n_e2e)
    s_up.wait_stream(s_down)
    t1.record(s_up)
    t1.synchronize()
    ms_e2e = mor(t0.elapsed_time(t1) / n_e2e)
    barrier()
    if ga.device_status() != 0:
        raise RuntimeError("kernel status word set during the end-to-end loop")
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * 4
    del qb[1], kb[1], vb[1], ob[1], lb[1]

    # ---------------------------------------------------------------- FP8
    # Prep + attention and prep alone, back to back (the per-config section
    # below times the attention alone with L2 flushed and checks its errors).
    fp8 = None
    if not args.no_extra:
        wf = inputs.WORKLOADS["fp8_n8192_d128"]
        fq, fk, fv = (t.to(dev) for t in inputs.workload_inputs(wf))
        signs = inputs.make_signs(wf.H, wf.d, wf.seed).to(dev)
        q8, sq = ga.fp8_prep(fq, signs)
        k8, sk = ga.fp8_prep(fk, signs)
        v8, sv = ga.fp8_prep(fv, None, transpose=True)
        of = torch.empty_like(fq)
        lf = torch.empty(wf.B, wf.H, wf.N, dtype=torch.float32, device=dev)
        attn8 = lambda: ga.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, causal=wf.causal, scale=wf.scale,
                                        out=of, lse=lf)

        def prep8():
            ga.fp8_prep(fq, signs, out=q8, scales=sq)
            ga.fp8_prep(fk, signs, out=k8, scales=sk)
            ga.fp8_prep(fv, None, transpose=True, out=v8, scales=sv)

        def full8():
            prep8()
            attn8()

        for _ in range(args.warmup):
            full8()
        barrier()
        ms8 = mor(_time_loop(attn8, args.steps, stream))
        ms8p = mor(_time_loop(full8, args.steps, stream))
        msprep = mor(_time_loop(prep8, args.steps, stream))
        barrier()
        prep_bytes = 3 * fq.numel() * 2 + 3 * fq.numel() + 3 * sq.numel() * 4
        t8 = wf.flops / (ms8 * 1e-3) / 1e12
        fp8 = {"workload": wf.name, "attn_tflops": t8 * ws,
               "attn_plus_prep_tflops": wf.flops / (ms8p * 1e-3) / 1e12 * ws,
               "ms_attn": ms8, "ms_prep": msprep,
               "roofline": {"bound": "tensor", "achieved": t8, "peak": 2 * peaks["bf16"],
                            "unit": "TFLOP/s", "frac": t8 / (2 * peaks["bf16"]),
                            "peak_note": "measured bf16 x 2 (nominal fp8/bf16 ratio)"},
               "prep_roofline": {"bound": "hbm", "achieved": prep_bytes / (msprep * 1e-3) / 1e9,
                                 "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": prep_bytes / (msprep * 1e-3) / 1e9 / peaks["hbm_gbs"]}}
        del fq, fk, fv, q8, k8, v8, of

    # ------------------------------------------------------------ backward
    # dQ, dK, dV of the benchmark workload (and its causal form) from the
    # forward's O and lse; FLOPs by the page's convention, 2.5 x the forward
    # (five 128x128 tile products per (query block, key block); the kernels do
    # seven, recomputing S and dP for dQ instead of adding it atomically).
    bwd = None
    if not args.no_extra:
        io_mib = 5 * w.B * w.H * w.N * w.d * 2 / 2 ** 20
        bwd = {"flops_convention": "2.5 x forward FLOPs (5 tile products); the kernels execute 7",
               "l2": f"Q, K, V, O, dO {io_mib:.0f} MiB (L2 129 MB; no flush)"}
        g = torch.Generator().manual_seed(w.seed + 60)
        dO = torch.randn(w.B, w.H, w.N, w.d, generator=g).to(torch.bfloat16).to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        wsb = torch.empty(ga.bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
        for causal in (False, True):
            ga.attn_fwd(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)
            fb = lambda: ga.attn_bwd(q, k, v, o, lse, dO, causal=causal, scale=w.scale, dq=dq, dk=dk,
                                     dv=dv, workspace=wsb)
            for _ in range(args.warmup):
                fb()
            barrier()
            msb = mor(_time_loop(fb, args.steps, stream))
            fl = 2.5 * w.flops / (2 if causal else 1)
            tb = fl / (msb * 1e-3) / 1e12
            bwd["causal" if causal else "non_causal"] = {
                "tflops": tb * ws, "ms": msb,
                "roofline": {"bound": "tensor", "achieved": tb, "peak": peaks["bf16"], "unit": "TFLOP/s",
                             "frac": tb / peaks["bf16"], "executed_frac": 1.4 * tb / peaks["bf16"]}}
        if ga.device_status() != 0:
            raise RuntimeError("kernel status word set during the backward benchmark")
        del dO, dq, dk, dv, wsb

    # ------------------------------------------------------- per workload
    # Every workload of the catalogue: each launch timed alone after a 256 MiB
    # write that flushes L2 (median of the launches), the fraction of the
    # tensor peak, ideal HBM bytes against those ncu measured (where a summary
    # taken on the current kernel source exists), and the errors against the
    # float64 oracle over every row, with the oracle's own wall time.
    others = {}
    if not args.no_extra:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        threads = os.cpu_count() or 1
        for name in ("n256_d64", "n2048_d128", "n2048_d128_causal", "n2048_d128_k8",
                     "n2048_d128_k8_causal", "n8192_d128", "n8192_d128_causal",
                     "n32768_d64_causal", "fp8_n8192_d128", "n8192_d128_gqa4_window4096",
                     "n8192_d128_b1h2", "n8192_d128_b1h2_causal"):
            wo = inputs.WORKLOADS[name]
            qh_, kh_, vh_ = inputs.workload_inputs(wo)
            a, b, c = qh_.to(dev), kh_.to(dev), vh_.to(dev)
            oo = torch.empty_like(a)
            lo = torch.empty(wo.B, wo.H, wo.N, dtype=torch.float32, device=dev)
            is8 = wo.dtype == "fp8"
            if is8:
                sg = inputs.make_signs(wo.H, wo.d, wo.seed).to(dev)
                a8, sa = ga.fp8_prep(a, sg)
                b8, sb = ga.fp8_prep(b, sg)
                c8, sc = ga.fp8_prep(c, None, transpose=True)
                fn = lambda: ga.attn_fwd_fp8(a8, b8, c8, sa, sb, sc, causal=wo.causal,
                                             scale=wo.scale, out=oo, lse=lo)
            elif wo.H_kv or wo.window:
                fn = lambda: ga.attn_fwd_ex(a, b, c, causal=wo.causal, window=wo.window,
                                            scale=wo.scale, out=oo, lse=lo)
            else:
                fn = lambda: ga.attn_fwd(a, b, c, causal=wo.causal, scale=wo.scale, out=oo, lse=lo)
            for _ in range(args.warmup):
                fn()
            barrier()
            ts = _flushed_times(fn, max(20, args.steps), stream, flush)
            msm = mor(statistics.median(ts))
            tfl = wo.flops / (msm * 1e-3) / 1e12
            peak = (2 if is8 else 1) * peaks["bf16"]
            kern = f"attn_fwd_{'fp8' if is8 else 'bf16'}_d{wo.d}_{wo.name}"
            entry = {"tflops": tfl * ws, "ms_median": msm, "ms_mean": mor(statistics.fmean(ts)),
                     "launches": len(ts), "l2": "flushed before each launch",
                     "roofline": {"bound": "tensor", "achieved": tfl, "peak": peak,
                                  "unit": "TFLOP/s", "frac": tfl / peak,
                                  "peak_note": "measured bf16 burst" + (" x 2" if is8 else "")},
                     "hbm": {"ideal_bytes": _ideal_bytes(wo),
                             "dram_bytes_ncu": _profiled_traffic(kern)}}
            if entry["hbm"]["dram_bytes_ncu"]:
                entry["hbm"]["ratio"] = entry["hbm"]["dram_bytes_ncu"] / entry["hbm"]["ideal_bytes"]
            if name.startswith("n8192_d128_b1h2"):
                # Split-KV on the same inputs, with the library's default split count.
                S = ga.splitkv_default_splits(wo.B, wo.H, wo.N, wo.d, wo.causal, sms)
                wsp = torch.empty(ga.splitkv_workspace_bytes(wo.B, wo.H, wo.N, wo.d, S),
                                  dtype=torch.uint8, device=dev)
                fs = lambda: ga.attn_fwd_splitkv(a, b, c, causal=wo.causal, scale=wo.scale,
                                                 num_splits=S, workspace=wsp, out=oo, lse=lo)
                for _ in range(args.warmup):
                    fs()
                barrier()
                mss = mor(statistics.median(_flushed_times(fs, max(20, args.steps), stream, flush)))
                entry["splitkv"] = {"tflops": wo.flops / (mss * 1e-3) / 1e12 * ws,
                                    "ms_median": mss, "splits": S, "launches_per_call": 2}
                del wsp
            if rank == 0 and not args.no_cpu_baseline:
                fn()
                torch.cuda.synchronize(dev)
                O_ref, L_ref, secs = _oracle_full(qh_, kh_, vh_, wo, threads)
                entry["errors"] = _errors(oo, lo, O_ref, L_ref, fp8=is8)
                entry["oracle"] = {"seconds": secs, "cores": threads, "rows": "all",
                                   "tflops": wo.flops / secs / 1e12}
                del O_ref, L_ref
            others[name] = entry
            del a, b, c, oo, lo
            if is8:
                del a8, b8, c8
        del flush
        barrier()
    if ga.device_status() != 0:
        raise RuntimeError("kernel status word set during the benchmark")

    # -------------------------------------------------------------- context
    # torch's scaled_dot_product_attention on the same inputs, timed the same
    # way: a context number only (whatever backend torch dispatches to), never
    # a path of this library.
    context = None
    if not args.no_extra:
        import torch.nn.functional as F
        sdpa = lambda: F.scaled_dot_product_attention(q, k, v, is_causal=w.causal, scale=w.scale)
        try:
            for _ in range(args.warmup):
                sdpa()
            barrier()
            ms_sdpa = mor(_time_loop(sdpa, args.steps, stream))
            context = {"torch_sdpa": {"tflops": w.flops / (ms_sdpa * 1e-3) / 1e12 * ws, "ms": ms_sdpa,
                                      "torch": torch.__version__, "workload": w.name}}
        except RuntimeError as e:   # no backend for this device in this torch build
            context = {"torch_sdpa": {"unavailable": str(e).splitlines()[0][:160]}}
        barrier()

    # ---------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        heads = [(b, h) for b in range(w.B) for h in range(w.H)]
        secs, flops = _oracle_run(qh, kh, vh, w, heads, threads)
        cpu = {"value": flops / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"the whole {w.name} workload, every row of every head (float64 "
                         f"three-pass oracle, {secs:.1f} s)"}

    traffic = _profiled_traffic(f"attn_fwd_bf16_d{w.d}_{w.name}")
    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "parallelism": f"replicas x{ws}",
                       "l2": "inputs + output 256 MiB > 129 MB L2 (no flush)"},
            "roofline": {"bound": "tensor", "achieved": tflops_launch, "peak": peaks["bf16"],
                         "unit": "TFLOP/s", "frac": tflops_launch / peaks["bf16"],
                         "traffic": traffic, "peak_source": peaks["source"] + " bf16 burst"},
            "timing_l2_flushed": {"ms_median": ms_flushed, "launches": len(ts_main),
                                  "tflops": whole_job_tflops(w.flops, ms_flushed, ws)},
            "e2e": {"value": w.flops / (ms_e2e * 1e-3) / 1e12 * ws, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                    "steps": n_e2e, "pipelined": "2 buffer sets, upload/compute/download streams"},
            "gpu_launches": args.steps,
            "clocks": {k2: clocks[k2] for k2 in ("sm_mhz", "sm_max_mhz", "reasons")},
            "cpu_baseline": cpu,
            "fp8": fp8,
            "backward": bwd,
            "workloads": others,
            "context": context,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default="n8192_d128")
    ap.add_argument("--no-extra", action="store_true", help="skip FP8 and other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)      # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_mine(args)


if __name__ == "__main__":
    main()
