#!/usr/bin/env python
"""Benchmark of the packed native-resolution 2D-RoPE varlen attention path.

One step = the whole hot path over one pack: mf_pack (cu_seqlens + (r, c)
tables), the forward (2D RoPE of Q/K + block-diagonal attention, O and LSE) and
the backward (dQ, dK, dV with the RoPE transpose folded in), all through the C
ABI.  The workload is the mixed-resolution training pack to a 50,000-token
budget (latent grids {32x32, 48x64, 64x48, 64x64, 40x96, 96x40}, text U[32, 512],
24 heads x 128, bf16 N(0,1), seeded).  Metric: attention TFLOP/s of the step,
counting 4 * sum(L_i^2) * d * heads forward and 2.5x that backward.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun each rank runs its own pack (seed = rank): replicas, no data-path
collective (weak scaling); the timing is max over ranks.  Prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "packed 2D-RoPE varlen attention TFLOP/s fwd/bwd at 50k tokens; % BF16 peak"
UNIT = "TFLOP/s"
# NVIDIA's dense bf16 tensor figure for one B300: the denominator the targets of
# the problem statement (>= 55 % forward, >= 40 % backward) are stated against.
NOMINAL_BF16_TFLOPS = 2250.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed_50k")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--budget", type=int, default=None,
                    help="token budget of the packed workload (default 50,000)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the timing of the attention's memory-bound neighbours")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--bwd-form", default="stored_ds", choices=["stored_ds", "recompute"],
                    help="the backward's form: dS stored by the dK/dV kernel and read back by "
                         "a streaming dQ GEMM (a larger workspace), or dQ recomputing S and dP")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="streams per copy direction in the end-to-end leg (2 or 3 measured "
                         "no faster: the host link, not a copy engine, is the limit)")
    return ap.parse_args()


def workload_desc(wl) -> str:
    return (f"{wl.name}: seed-{wl.seed} pack of {len(wl.specs)} samples, T={wl.total}, "
            f"max L={wl.max_len}, {wl.heads} heads x {wl.head_dim}, bf16 N(0,1)")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_burst": float(p["bf16_tflops"]), "bf16_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_burst": 1800.0, "bf16_sustained": 1400.0, "hbm_gbs": 6400.0, "source": "fallback"}


# ------------------------------------------------------------ CPU oracle leg
def oracle_sample(wl, q, k, v, do, max_pairs):
    """The first `max_pairs` (sample, head) pairs, smallest samples first, as a
    sub-pack of one-head samples (exact: samples and heads are independent)."""
    import oracle
    cu, pos = oracle.pack3d(wl.specs) if wl.edit else oracle.pack(wl.specs)
    L = np.diff(cu)
    pairs = [(int(i), a) for i in np.argsort(L, kind="stable") for a in range(wl.heads)][:max_pairs]
    f = synth.bf16_bits_to_f64
    sl = lambda x, i, a: x[cu[i]:cu[i + 1], a:a + 1, :]  # noqa: E731
    sub = [np.concatenate([f(sl(x, i, a)) for (i, a) in pairs], 0) for x in (q, k, v, do)]
    lens = [int(L[i]) for (i, _) in pairs]
    cu_s = np.concatenate([[0], np.cumsum(lens)])
    pos_s = np.concatenate([pos[cu[i]:cu[i + 1]] for (i, _) in pairs], 0)
    flops = 3.5 * 4.0 * sum(x * x for x in lens) * wl.head_dim
    return sub, cu_s, pos_s, flops, pairs


def run_oracle_step(sub, cu_s, pos_s):
    import oracle
    q, k, v, do = sub
    if pos_s.shape[1] == 3:  # editing pack: frame-aware 3D positions
        oracle.attn_fwd3d(q, k, v, cu_s, pos_s)
        oracle.attn_bwd3d(q, k, v, do, cu_s, pos_s)
    else:
        oracle.attn_fwd(q, k, v, cu_s, pos_s)
        oracle.attn_bwd(q, k, v, do, cu_s, pos_s)


def cpu_baseline(wl, q, k, v, do, budget_s):
    """The oracle as it stands on this host's cores: forward + backward of
    (sample, head) pairs, smallest samples first, in batches of one pair per core,
    until `budget_s` seconds have passed."""
    cores = len(os.sched_getaffinity(0))
    total_pairs = len(wl.specs) * wl.heads
    done_flops, n_pairs, t0 = 0.0, 0, time.perf_counter()
    while n_pairs < total_pairs and time.perf_counter() - t0 < budget_s:
        take = min(total_pairs, n_pairs + cores)
        sub, cu_s, pos_s, _, pairs = oracle_sample(wl, q, k, v, do, take)
        # only the new pairs of this batch
        sub_new, cu_new, pos_new, fl, _ = _slice_pairs(sub, cu_s, pos_s, n_pairs, take, wl.head_dim)
        run_oracle_step(sub_new, cu_new, pos_new)
        done_flops += fl
        n_pairs = take
    el = time.perf_counter() - t0
    return {"value": done_flops / el / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"FP64 C oracle, forward + backward of {n_pairs} of {total_pairs} (sample, head) "
                      f"pairs of the same pack, smallest samples first, {el:.1f} s wall, "
                      f"OpenMP over query and key rows"}


def _slice_pairs(sub, cu_s, pos_s, a, b, d):
    s, e = int(cu_s[a]), int(cu_s[b])
    lens = np.diff(cu_s[a:b + 1])
    cu_new = np.concatenate([[0], np.cumsum(lens)])
    return [x[s:e] for x in sub], cu_new, pos_s[s:e], 3.5 * 4.0 * float((lens ** 2).sum()) * d, None


def reference_arm(args):
    """The FP64 oracle timed as the reference arm, on this host's cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = synth.workload(args.workload, args.seed, args.budget)
    q, k, v, do = synth.make_inputs(wl, with_do=True)
    cores = len(os.sched_getaffinity(0))
    sub, cu_s, pos_s, flops, pairs = oracle_sample(wl, q, k, v, do, cores)
    for _ in range(args.warmup):
        run_oracle_step(sub, cu_s, pos_s)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run_oracle_step(sub, cu_s, pos_s)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    val = flops / (ms / 1e3) / 1e12
    sample = (f"FP64 C oracle, forward + backward of {len(pairs)} (sample, head) pairs "
              f"(smallest samples first) of the pack per step")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl), "sample": sample},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm
def rank_workload(name: str, seed: int, rank: int, budget=None):
    """The pack a rank processes: its own seeded draw of the workload (seed + rank).
    Ranks share no data, so the path needs no collective (weak scaling)."""
    return synth.workload(name, seed + rank, budget)


def reduce_over_ranks(ms: float, flops: float, world: int):
    """(max over ranks of the step time, sum over ranks of the work): the
    whole-job throughput is the second over the first.  Host-side gloo / NCCL
    all-reduces of two scalars; nothing on the data path."""
    if world <= 1:
        return ms, flops
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, flops], dtype=torch.float64)
    tmax, tsum = t.clone(), t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
    return float(tmax[0]), float(tsum[1])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = bus_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.bus_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        time.sleep(0.15)

    def result(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_local_cpus(bus: str):
    """CPUs of the NUMA node next to the GPU at PCI address `bus` (sysfs
    local_cpulist), limited to those this process may use; empty if unknown."""
    path = f"/sys/bus/pci/devices/{bus.lower()[4:]}/local_cpulist"
    try:
        text = open(path).read().strip()
    except OSError:
        return set()
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus & os.sched_getaffinity(0)


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    import packed_resolution_diffusion_pack_b300 as mf

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    mf.load()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    wl = rank_workload(args.workload, args.seed, rank, args.budget)
    q, k, v, do = synth.make_inputs(wl, with_do=True)
    T, max_len = mf.pack3d_size(wl.specs) if wl.edit else mf.pack_size(wl.specs)
    n, h, d = len(wl.specs), wl.heads, wl.head_dim
    props = torch.cuda.get_device_properties(local)
    bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    # Pinned host buffers are placed on the NUMA node of the allocating CPU: allocate
    # them from the CPUs next to this GPU (as a data loader pinned to that node would),
    # then restore the affinity.
    saved = os.sched_getaffinity(0)
    local_cpus = gpu_local_cpus(bus)
    if local_cpus:
        os.sched_setaffinity(0, local_cpus)
    pin = lambda b: synth.bits_to_torch(b).pin_memory()  # noqa: E731
    hq, hk, hv, hdo = pin(q), pin(k), pin(v), pin(do)
    qd, kd, vd, dod = (x.cuda() for x in (hq, hk, hv, hdo))
    o = torch.empty_like(qd)
    lse = torch.empty((h, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    # one workspace for forward and backward: the backward reuses the forward's
    # rotated fp16 operands (mf_varlen_attn_bwd_after_fwd); sized for the stored-dS
    # form of the backward unless --bwd-form recompute (or the form is unavailable)
    ds_ok = args.bwd_form == "stored_ds" and mf.attn_workspace_bytes_ds(T, n, h, d, max_len) > 0
    ws = mf.workspace(T, n, h, d, True, store_ds_max_len=max_len if ds_ok else None)
    bwd_form = "stored_ds" if ds_ok else "recompute"
    cu = torch.empty(n + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty((T, 3 if wl.edit else 2), dtype=torch.int32, device="cuda")
    packer = mf.pack3d if wl.edit else mf.pack

    def step(qd=qd, kd=kd, vd=vd, dod=dod):
        packer(wl.specs, cu=cu, pos=pos)
        mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len, o=o, lse=lse, ws=ws)
        mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, dq=dq, dk=dk, dv=dv, ws=ws,
                           after_fwd=True)

    for _ in range(max(args.warmup, 3)):
        step()
    mf.get_status(ws)
    barrier()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    mf.timing_enable(True)
    mf.timing_reset()
    with ClockSampler(bus) as clk:
        barrier()
        ev0.record()
        for _ in range(args.steps):
            step()
        ev1.record()
        barrier()
    clocks = clk.result()
    kern = mf.timing_read()
    mf.timing_enable(False)
    mf.get_status(ws)
    ms = ev0.elapsed_time(ev1) / args.steps

    flops_fwd, flops_bwd = wl.flops_fwd(), wl.flops_bwd()
    ms_max, flops_all = reduce_over_ranks(ms, flops_fwd + flops_bwd, world)
    value = flops_all / (ms_max / 1e3) / 1e12

    # ---- end to end through the public API with pinned host buffers.  Every step
    # uploads its q, k, v, dO from pinned host memory and downloads o, lse, dq, dk,
    # dv; separate streams pipeline consecutive steps (upload of step i, compute of
    # step i-1, download of step i-2), as a data loader feeds a training loop.
    # Each direction's tensors are dealt to --copy-streams streams, so that several
    # copy engines work on one direction at once.  Two device buffer sets; events
    # keep a set's inputs until its compute has read them and its outputs until
    # their download has read them.
    pinned = lambda: torch.empty(hq.shape, dtype=hq.dtype, pin_memory=True)  # noqa: E731
    NB = 2
    NC = max(1, args.copy_streams)  # streams per copy direction (copy engines work in parallel)
    ups = [torch.cuda.Stream() for _ in range(NC)]
    downs = [torch.cuda.Stream() for _ in range(NC)]
    s_comp = torch.cuda.Stream()
    dev_in = [[torch.empty_like(qd) for _ in range(4)] for _ in range(NB)]
    dev_out = [{"o": torch.empty_like(qd), "lse": torch.empty((h, T), dtype=torch.float32, device="cuda"),
                "dq": torch.empty_like(qd), "dk": torch.empty_like(qd), "dv": torch.empty_like(qd)}
               for _ in range(NB)]
    host_out = [{"o": pinned(), "lse": torch.empty((h, T), dtype=torch.float32, pin_memory=True),
                 "dq": pinned(), "dk": pinned(), "dv": pinned()} for _ in range(NB)]
    ev_up = [[torch.cuda.Event() for _ in range(NC)] for _ in range(NB)]
    ev_comp = [torch.cuda.Event() for _ in range(NB)]
    ev_down = [[torch.cuda.Event() for _ in range(NC)] for _ in range(NB)]
    os.sched_setaffinity(0, saved)
    for b in range(NB):  # recorded once, so the first waits are satisfied
        ev_comp[b].record(s_comp)
        for c in range(NC):
            ev_down[b][c].record(downs[c])
    e2e_steps = max(3, min(args.steps, 20))
    # tensors dealt to the copy streams in turn (largest first)
    in_names = list(range(4))
    out_names = ["o", "dq", "dk", "dv", "lse"]

    def e2e_step(i):
        b = i % NB
        for c, st in enumerate(ups):
            st.wait_event(ev_comp[b])
            with torch.cuda.stream(st):
                for j in in_names[c::NC]:
                    dev_in[b][j].copy_((hq, hk, hv, hdo)[j], non_blocking=True)
            ev_up[b][c].record(st)
        for c in range(NC):
            s_comp.wait_event(ev_up[b][c])
            s_comp.wait_event(ev_down[b][c])
        qq, kk, vv, dd = dev_in[b]
        out = dev_out[b]
        packer(wl.specs, cu=cu, pos=pos, stream=s_comp)
        mf.varlen_attn_fwd(qq, kk, vv, cu, pos, max_len, o=out["o"], lse=out["lse"], ws=ws,
                           stream=s_comp)
        mf.varlen_attn_bwd(qq, kk, vv, out["o"], out["lse"], dd, cu, pos, max_len, dq=out["dq"],
                           dk=out["dk"], dv=out["dv"], ws=ws, stream=s_comp, after_fwd=True)
        ev_comp[b].record(s_comp)
        for c, st in enumerate(downs):
            st.wait_event(ev_comp[b])
            with torch.cuda.stream(st):
                for name in out_names[c::NC]:
                    host_out[b][name].copy_(out[name], non_blocking=True)
            ev_down[b][c].record(st)

    for i in range(NB):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(ups[0])
    for st in ups[1:]:
        st.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    last = (e2e_steps - 1) % NB
    for c in range(1, NC):
        downs[0].wait_event(ev_down[last][c])
    e1.record(downs[0])
    barrier()
    mf.get_status(ws, s_comp)
    ms_e2e, _ = reduce_over_ranks(e0.elapsed_time(e1) / e2e_steps, 0.0, world)
    elem = T * h * d
    h2d = 4 * elem * 2
    d2h = 4 * elem * 2 + h * T * 4

    pk = peaks()
    per_launch = {}
    for name, (tot, cnt) in kern.items():
        if cnt:
            per_launch[name] = {"ms_per_launch": tot / cnt, "launches": cnt,
                                "share": tot / max(1e-9, sum(x[0] for x in kern.values()))}
    # Denominator: the burst bf16 figure, measured at full clocks, when the SM clock
    # under our load stayed at its maximum (as sampled); else the sustained one.
    full_clock = (clocks.get("sm_mhz") or 0) >= 0.95 * (clocks.get("sm_max_mhz") or 1e9)
    peak_tc = pk["bf16_burst"] if full_clock else pk["bf16_sustained"]
    peak_name = (f"{pk['source']} bf16 " + ("burst (cuBLAS 8192^3, SM clock at max under our "
                 "load)" if full_clock else "sustained (cuBLAS, seconds-long loop)"))
    # algorithmic work per launch: FLOPs for the attention kernels, bytes for the
    # memory-bound ones (rope: the forward's pre-pass reads q, k, v bf16 and writes
    # Q', K', V' fp16; the backward reuses them).  The backward's five GEMMs of
    # 4 sum(L^2) d h FLOP / 2 each: the dK/dV kernel ("attn_bwd") runs four of them
    # (S^T, dP^T, dV, dK: 0.8 of the backward's FLOPs); the dQ kernel
    # ("attn_bwd_q") runs the fifth (dQ: 0.2) and recomputes S and dP (0.4 more,
    # executed but not credited).
    elems = float(T * h * d)
    algo = {"attn_fwd": ("tensor", flops_fwd), "attn_bwd": ("tensor", 0.8 * flops_bwd),
            "attn_bwd_q": ("tensor", 0.2 * flops_bwd),
            # stored-dS form: reads the padded dS^T blocks (a_i = L_i rounded up to
            # 128) and K' once, writes dQ
            "attn_bwd_dq": ("hbm", 2.0 * h * sum((128 * -(-L // 128)) ** 2 for L in wl.lengths)
                            + 4.0 * elems),
            "rope": ("hbm", 12.0 * elems + 8.0 * T),
            "bwd_pre": ("hbm", 6.0 * elems + 12.0 * h * T)}
    for name, (bound, amount) in algo.items():
        if name in per_launch:
            pl = per_launch[name]
            if bound == "tensor":
                ach = amount / (pl["ms_per_launch"] / 1e3) / 1e12
                pl.update(achieved_tflops=ach, frac=ach / peak_tc,
                          frac_of_sustained=ach / pk["bf16_sustained"],
                          frac_of_burst=ach / pk["bf16_burst"],
                          frac_of_nominal=ach / NOMINAL_BF16_TFLOPS)
                if name == "attn_bwd_q":  # S, dP and dQ executed
                    pl["executed_tflops"] = 3.0 * ach
            else:
                ach = amount / (pl["ms_per_launch"] / 1e3) / 1e9
                pl.update(achieved_gbs=ach, frac_of_hbm=ach / pk["hbm_gbs"])
            pl.update(algorithmic=amount, traffic=_recorded_traffic(name))
    dom = max(("attn_fwd", "attn_bwd", "attn_bwd_q"), key=lambda nm: kern[nm][0])
    q_kernel = "attn_bwd_dq" if bwd_form == "stored_ds" else "attn_bwd_q"
    traffic = _recorded_traffic(dom)
    ach = per_launch[dom]["achieved_tflops"]
    roofline = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak_tc,
                "unit": "TFLOP/s", "frac": ach / peak_tc, "traffic": traffic,
                "peak_kind": peak_name, "frac_of_nominal": ach / NOMINAL_BF16_TFLOPS}
    fwd_ms = per_launch["attn_fwd"]["ms_per_launch"]
    # the backward's attention: the dK/dV kernel and the dQ kernel
    bwd_ms = per_launch["attn_bwd"]["ms_per_launch"] + per_launch[q_kernel]["ms_per_launch"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(wl), "global_tokens": T * world,
                   "step": "mf_pack + mf_varlen_attn_fwd (RoPE + attention) + "
                           "mf_varlen_attn_bwd_after_fwd (one shared workspace)",
                   "bwd_form": bwd_form, "workspace_gb": round(ws.numel() / 1e9, 2),
                   "l2": "no flush: Q, K, V, dO alone are %.2f GB, far above the 126 MB L2" % (
                       4 * elem * 2 / 1e9),
                   "parallelism": "replicas: one pack per GPU, no data-path collective"},
        "fwd_tflops": flops_fwd / (fwd_ms / 1e3) / 1e12,
        "bwd_tflops": flops_bwd / (bwd_ms / 1e3) / 1e12,
        "fwd_frac_of_peak": flops_fwd / (fwd_ms / 1e3) / 1e12 / peak_tc,
        "bwd_frac_of_peak": flops_bwd / (bwd_ms / 1e3) / 1e12 / peak_tc,
        "peak_tflops": peak_tc,
        # the targets are stated against the nominal dense bf16 peak
        "fwd_frac_of_nominal": flops_fwd / (fwd_ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
        "bwd_frac_of_nominal": flops_bwd / (bwd_ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
        "nominal_peak_tflops": NOMINAL_BF16_TFLOPS,
        "targets_vs_nominal": {"fwd": 0.55, "bwd": 0.40},
        "roofline": roofline,
        "kernels": per_launch,
        "gpu_launches": int(sum(x[1] for x in kern.values())),
        "e2e": {"value": flops_all / (ms_e2e / 1e3) / 1e12, "unit": UNIT, "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "copy_streams_per_direction": NC,
                "how": "public API, pinned host buffers, upload / compute / download of "
                       "consecutive steps pipelined on separate streams"},
        "clocks": clocks,
    }
    if not args.no_extras:
        line["extras"] = neighbours(mf, wl, pk["hbm_gbs"])
        line["extras"]["forward_only"] = forward_only(mf, wl, qd, kd, vd, cu, pos, max_len, ws,
                                                      peak_tc)
        if d == 128:
            line["extras"]["fp8_forward"] = fp8_forward(mf, wl, qd, kd, vd, cu, pos, max_len, ws,
                                                        peak_tc, pk["hbm_gbs"])
        line["extras"]["backward_forms"] = backward_forms(mf, wl, qd, kd, vd, dod, cu, pos, max_len,
                                                          o, lse, peak_tc)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, q, k, v, do, args.cpu_budget_s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def neighbours(mf, wl, hbm_gbs, reps=20):
    """Device time (per kernel, from the library's timing hook) and HBM throughput of the memory-bound neighbours of the
    attention, outside the timed step: the adaptive LayerNorm modulation and the
    gated residual on this pack's [T, heads x head_dim] activations, and the
    packed-CFG Euler step on 32 2048^2 (cond, uncond) pairs with 64 latent
    channels (every working set is above the 126 MB L2).  Algorithmic bytes: adaLN reads x and writes y (4 T Dm); the gated
    residual reads x, h and writes out (6 T Dm); the CFG step reads both branches'
    bf16 image rows and reads and writes the fp32 latent (12 N C)."""
    import torch
    T, Dm, n = wl.total, wl.heads * wl.head_dim, len(wl.specs)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(wl.lengths)]), dtype=torch.int32, device="cuda")
    x = synth.bits_to_torch(synth.normal_bf16_bits(wl.seed, 32, (T, Dm))).cuda()
    h = synth.bits_to_torch(synth.normal_bf16_bits(wl.seed, 35, (T, Dm))).cuda()
    vec = synth.bits_to_torch(synth.normal_bf16_bits(wl.seed, 33, (n, Dm))).cuda()
    y = torch.empty_like(x)
    specs = [(512, 128, 128), (64, 128, 128)] * 32
    Tc, _ = mf.pack_size(specs)
    C = 64
    v = synth.bits_to_torch(synth.normal_bf16_bits(wl.seed, 30, (Tc, C))).cuda()
    N = 32 * 128 * 128
    z = torch.zeros((N, C), dtype=torch.float32, device="cuda")
    cases = {
        "adaln_modulate": (lambda: mf.adaln_modulate(x, cu, vec, vec, 1e-6, y=y), 4.0 * T * Dm,
                           f"T={T}, Dm={Dm}, bf16"),
        "gated_residual": (lambda: mf.gated_residual(x, h, cu, vec, out=y), 6.0 * T * Dm,
                           f"T={T}, Dm={Dm}, bf16"),
        "cfg_euler_step": (lambda: mf.cfg_euler_step(v, specs, 4.0, 0.05, z), 12.0 * N * C,
                           f"32 pairs of 2048^2 (16384 image tokens each), C={C}"),
    }
    traffic_name = {"adaln_modulate": "adaln", "gated_residual": "gated_residual",
                    "cfg_euler_step": "cfg_euler"}
    out = {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kernel_id = {"adaln_modulate": "adaln", "gated_residual": "gated_residual",
                 "cfg_euler_step": "cfg_euler"}
    for name, (fn, nbytes, shape) in cases.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        mf.timing_enable(True)
        mf.timing_reset()
        ev0.record()
        for _ in range(reps):
            fn()
        ev1.record()
        torch.cuda.synchronize()
        kern = mf.timing_read()
        mf.timing_enable(False)
        # the kernel's device time (the Python call's argument marshalling can take
        # as long as these short kernels, so the call-to-call time is host bound)
        tot, cnt = kern[kernel_id[name]]
        ms = tot / max(1, cnt)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"ms": ms, "achieved_gbs": gbs, "frac_of_hbm": gbs / hbm_gbs, "shape": shape,
                     "bytes": nbytes, "traffic": _recorded_traffic(traffic_name[name]),
                     "call_ms": ev0.elapsed_time(ev1) / reps}
    return out


def forward_only(mf, wl, qd, kd, vd, cu, pos, max_len, ws, peak_bf16, reps=10):
    """The forward alone (a sampling step's attention), outside the timed step, in
    its two forms on the same pack: the two-pass call (mf_varlen_attn_fwd: the fp16
    rotation pre-pass, then attention on the rotated operands) and the
    rotate-on-load call (mf_varlen_attn_fwd_fused_rope: a (cos, sin) table, then
    attention that rotates the bf16 Q and K tiles in shared memory).  Both give the
    same O and LSE bit for bit.  Each call timed with CUDA events over `reps` calls,
    and each kernel's device time."""
    import torch
    T, h = wl.total, wl.heads
    o = torch.empty_like(qd)
    lse = torch.empty((h, T), dtype=torch.float32, device="cuda")
    flops = wl.flops_fwd()
    forms = {
        "two_pass": (lambda: mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len, o=o, lse=lse, ws=ws),
                     ("schedule", "rope", "attn_fwd")),
        "fused_rope": (lambda: mf.varlen_attn_fwd_fused_rope(qd, kd, vd, cu, pos, max_len, o=o,
                                                             lse=lse, ws=ws),
                       ("schedule", "rope_table", "attn_fwd_rot")),
    }
    out = {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, (call, kernels) in forms.items():
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        mf.timing_enable(True)
        mf.timing_reset()
        ev0.record()
        for _ in range(reps):
            call()
        ev1.record()
        torch.cuda.synchronize()
        kern = mf.timing_read()
        mf.timing_enable(False)
        mf.get_status(ws)
        ms = ev0.elapsed_time(ev1) / reps
        per = {k: kern[k][0] / max(1, kern[k][1]) for k in kernels}
        attn_ms = per[kernels[-1]]
        out[name] = {"ms_per_call": ms, "tflops_per_call": flops / (ms / 1e3) / 1e12,
                     "kernel_ms": per, "attn_tflops": flops / (attn_ms / 1e3) / 1e12,
                     "attn_frac": flops / (attn_ms / 1e3) / 1e12 / peak_bf16}
    out["fused_over_two_pass"] = out["two_pass"]["ms_per_call"] / out["fused_rope"]["ms_per_call"]
    return out


def backward_forms(mf, wl, qd, kd, vd, dod, cu, pos, max_len, o, lse, peak_bf16, reps=5):
    """The backward in its two forms on the same pack, outside the timed step, each
    on a workspace of its own after a forward on it: recompute (the dQ kernel
    recomputes S and dP; mf_attn_workspace_bytes) and stored dS (the dK / dV kernel
    stores dS^T, a streaming kernel forms dQ from it; mf_attn_workspace_bytes_ds).
    Per form: CUDA-event time per backward call and each attention kernel's time."""
    import torch
    T, n, h, d = wl.total, len(wl.specs), wl.heads, wl.head_dim
    flops = wl.flops_bwd()
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    out = {}
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for form, ds_len, kq in (("recompute", None, "attn_bwd_q"),
                             ("stored_ds", max_len, "attn_bwd_dq")):
        if ds_len is not None and mf.attn_workspace_bytes_ds(T, n, h, d, ds_len) == 0:
            continue
        ws = mf.workspace(T, n, h, d, True, store_ds_max_len=ds_len)
        mf.varlen_attn_fwd(qd, kd, vd, cu, pos, max_len, o=o, lse=lse, ws=ws)
        call = lambda: mf.varlen_attn_bwd(qd, kd, vd, o, lse, dod, cu, pos, max_len, dq=dq,  # noqa: E731
                                          dk=dk, dv=dv, ws=ws, after_fwd=True)
        for _ in range(2):
            call()
        torch.cuda.synchronize()
        mf.timing_enable(True)
        mf.timing_reset()
        ev0.record()
        for _ in range(reps):
            call()
        ev1.record()
        torch.cuda.synchronize()
        kern = mf.timing_read()
        mf.timing_enable(False)
        mf.get_status(ws)
        ms = ev0.elapsed_time(ev1) / reps
        kv_ms = kern["attn_bwd"][0] / max(1, kern["attn_bwd"][1])
        q_ms = kern[kq][0] / max(1, kern[kq][1])
        out[form] = {"ms_per_call": ms, "workspace_gb": ws.numel() / 1e9, "dkdv_ms": kv_ms,
                     "dq_ms": q_ms, "attn_ms": kv_ms + q_ms,
                     "attn_tflops": flops / ((kv_ms + q_ms) / 1e3) / 1e12,
                     "attn_frac": flops / ((kv_ms + q_ms) / 1e3) / 1e12 / peak_bf16}
        del ws
        torch.cuda.empty_cache()
    return out


def fp8_forward(mf, wl, qd, kd, vd, cu, pos, max_len, ws, peak_bf16, hbm_gbs, reps=10):
    """The 8-bit (E4M3) variant of the forward on the same pack, outside the timed
    step: the whole call (schedule, the two quantisation passes, attention) timed
    with CUDA events, and each kernel's device time.  The tensor-core peak for E4M3
    operands is twice the measured bf16 one (the nominal dense ratio, 4.5 vs
    2.25 PFLOP/s).  Algorithmic bytes: the maxima pass reads k and v (4 T h d); the
    quantiser reads q, k, v (6 T h d) and writes the E4M3 copies (3 T h d) and
    the Q row scales (4 T h)."""
    import torch
    T, h, d = wl.total, wl.heads, wl.head_dim
    o = torch.empty_like(qd)
    lse = torch.empty((h, T), dtype=torch.float32, device="cuda")
    call = lambda: mf.varlen_attn_fwd_fp8(qd, kd, vd, cu, pos, max_len, o=o, lse=lse, ws=ws)  # noqa: E731
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    mf.timing_enable(True)
    mf.timing_reset()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(reps):
        call()
    ev1.record()
    torch.cuda.synchronize()
    kern = mf.timing_read()
    mf.timing_enable(False)
    mf.get_status(ws)
    ms = ev0.elapsed_time(ev1) / reps
    flops = wl.flops_fwd()
    peak8 = 2.0 * peak_bf16
    elems = float(T * h * d)
    per = lambda name: kern[name][0] / max(1, kern[name][1])  # noqa: E731
    attn_ms = per("attn_fwd_f8")
    amax_bytes, quant_bytes = 4.0 * elems, 9.0 * elems + 4.0 * T * h
    return {
        "ms_per_call": ms, "tflops_per_call": flops / (ms / 1e3) / 1e12,
        "attn_ms": attn_ms, "attn_tflops": flops / (attn_ms / 1e3) / 1e12,
        "attn_frac_of_e4m3_peak": flops / (attn_ms / 1e3) / 1e12 / peak8,
        "e4m3_peak_tflops": peak8,
        "amax_ms": per("f8_amax"),
        "amax_frac_of_hbm": amax_bytes / (per("f8_amax") / 1e3) / 1e9 / hbm_gbs,
        "quant_ms": per("f8_quant"),
        "quant_frac_of_hbm": quant_bytes / (per("f8_quant") / 1e3) / 1e9 / hbm_gbs,
        "amax_traffic": _recorded_traffic("f8_amax"), "quant_traffic": _recorded_traffic("f8_quant"),
        "roofline": {"bound": "tensor", "kernel": "attn_fwd_f8",
                     "achieved": flops / (attn_ms / 1e3) / 1e12, "peak": peak8, "unit": "TFLOP/s",
                     "frac": flops / (attn_ms / 1e3) / 1e12 / peak8,
                     "traffic": _recorded_traffic("attn_fwd_f8"),
                     "peak_kind": "2 x the measured bf16 peak (nominal E4M3 / bf16 dense ratio)"},
        "call": "mf_varlen_attn_fwd_fp8 (E4M3 operands and probabilities, fp32 accumulation)",
    }


def _recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed capture records
    (profiles/dram_traffic.json), if the record was taken on the current kernel
    source (the SHA-256 prefix it stores still matches); else None."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            records = json.load(f)["records"]
    except (OSError, KeyError, ValueError):
        return None
    for rec in records:
        if rec.get("kernel") != kernel:
            continue
        src = os.path.join(ROOT, "packed_resolution_diffusion_pack_b300", "csrc", rec["source"])
        try:
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        except OSError:
            return None
        return int(rec["dram_bytes_per_launch"]) if sha == rec["sha16"] else None
    return None


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
