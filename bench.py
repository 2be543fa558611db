"""Benchmark: packed DAG attention forward + backward (useful TFLOP/s) and paged decode
(HBM GB/s) on one GB300, through the C ABI.

One step = one pass of the training hot path over the full episode (16K prefix, 7
branches x 32K owned tokens, 3 rewinds, 6 mounts; 16 q / 4 kv heads, d 128, page 64,
bf16): the GPU plan compile (positions + tile list + CSC), the forward, and the backward.
The decode leg times the decode plan and the paged decode of 256 cursors (32 episodes x 8,
mean context ~26K tokens) the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own episode (a different seed): weak scaling, no
collective on the data path; rank 0 prints the JSON line with the max time over ranks.
--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed DAG attention fwd+bwd useful TFLOP/s & % bf16 peak; decode HBM GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained") or bf
            if hbm and bf:
                return float(hbm), float(bf), float(bfs), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        sms, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


def rank_seed(seed, rank):
    """Each rank runs its own episode: the units (episodes) are independent, so the
    data path has no collective."""
    return seed + rank


def max_over_ranks(value, dist):
    """The job's step time is the slowest rank's."""
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def unique_tokens(entries, num_pages, P):
    seen = np.zeros((num_pages, P), dtype=bool)
    for lo in range(P):
        sel = (entries["kv_lo"] <= lo) & (entries["kv_hi"] > lo)
        seen[entries["kv_page"][sel].astype(np.int64), lo] = True
    return int(seen.sum())


# --------------------------------------------------------------------------------------
L2_BYTES = 129 * 2**20   # GB300 L2


def profiled_traffic(workload, call, profile="dram_traffic_episode.md", profiled_workload="episode"):
    """DRAM bytes per call of `call` from a committed ncu summary of the full-size workload,
    or None when the workload differs or a kernel source's code changed since the counters."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", profile)
    if workload != profiled_workload or not os.path.exists(path):
        return None
    want, got = {}, None
    for line in open(path):
        line = line.strip()
        if " sha256/16: " in line:
            name, h = line.split(" sha256/16: ")
            want[name] = h
        elif line.startswith(call + " bytes per call: "):
            got = int(line.split(": ")[1])
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "packed_tree_attention_gb300", "csrc")
    for name, h in want.items():
        if code_fingerprint(os.path.join(src, name)) != h:
            return None
    return got if want else None


def code_fingerprint(path):
    """sha256/16 of a C++/CUDA source with // comments and blank lines removed: edits to
    comments keep it, any change to the code does not."""
    import hashlib
    lines = []
    for line in open(path, encoding="utf-8"):
        line = line.split("//", 1)[0].rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


WORKLOAD_DESC = {
    "episode": "episode: 16K prefix, 7 branches x 32K owned tokens, 3 rewinds, 6 mounts",
    "tree_fwd": "tree: 4K prefix, 4 x 8K branches, 2 mounts",
    "train_step": "train step: 8 trees of ~140K owned tokens, fan-out 2-6, depth <= 3, mounts",
    "tiny": "tiny: 64-token prefix, 2 x 32 branches, 1 mount",
    "decode": "paged decode: 32 episodes x 8 cursors, shared prefix 2-8K, paths 8-32K, 0-3 sibling mounts of 0.5-8K",
    "decode_small": "paged decode: 4 episodes x 8 cursors, shared prefix 2-8K, paths 8-32K, 0-3 sibling mounts",
}


def workload_desc(name, cfg):
    return "%s; %dq/%dkv heads, d=%d, page %d, q-tile 128, %s fwd+bwd" % (
        WORKLOAD_DESC.get(name, name), cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"], cfg.get("dtype", "bf16"))


# workload construction (device tensors from the counter-based generator)
# --------------------------------------------------------------------------------------
def build_episode(pta, torch, name, seed, dev):
    cfg = synth.CONFIGS[name]
    Hq, Hkv, d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
    ep = synth.make_preset(name, seed=seed)
    npages = sum((L + P - 1) // P for L in ep.length) + 8 + 4 * len(ep.cursors)   # room for decode steps
    kp = torch.empty((npages, Hkv, P, d), dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    pool = pta.Pool(npages, P, Hkv, d, pta.DTYPE_BF16, kp, vp)
    sK, sV = synth.STREAM_K + 16 * seed, synth.STREAM_V + 16 * seed
    t = 0
    chunk = 1 << 16
    for op in ep.ops:
        kind = op[0]
        if kind == "append":
            _, c, n = op
            for a in range(0, n, chunk):
                m = min(chunk, n - a)
                K = synth.hash_fill(sK, (m, Hkv, d), torch.bfloat16, dev, 0.5, row_start=t + a)
                V = synth.hash_fill(sV, (m, Hkv, d), torch.bfloat16, dev, 0.5, row_start=t + a)
                pool.append(c, m, K, V)
            t += n
        elif kind == "root":
            pool.root()
        elif kind == "fork":
            pool.fork(op[1], op[2])
        elif kind == "mount":
            pool.mount(*op[1:])
        elif kind == "rewind":
            pool.rewind(op[1], op[2])
        elif kind == "done":
            pool.done(op[1])
    return ep, pool, kp, vp, cfg


# --------------------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# --------------------------------------------------------------------------------------
def oracle_sample(name, seed, budget_s=15.0, n_rows_max=256):
    """Times the fp64 oracle's forward + backward on a seeded sample of packed rows of the
    workload (all 16 heads of each row; the backward's dK/dV from those rows only).
    Returns (TFLOP/s, threads, description)."""
    import torch
    import oracle
    cfg = synth.CONFIGS[name]
    Hq, Hkv, d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
    ep = synth.make_preset(name, seed=seed)
    T = ep.n_tokens
    npages = sum((L + P - 1) // P for L in ep.length) + 8 + 4 * len(ep.cursors)   # room for decode steps
    orc = oracle.Oracle(P, npages, Hkv, d)
    K = synth.hash_rows(synth.STREAM_K + 16 * seed, np.arange(T), Hkv * d, torch.bfloat16, 0.5).reshape(T, Hkv, d)
    V = synth.hash_rows(synth.STREAM_V + 16 * seed, np.arange(T), Hkv * d, torch.bfloat16, 0.5).reshape(T, Hkv, d)
    orc.replay(ep, K, V)
    del K, V
    opl = orc.pack(ep.roots, 128, tile_stride=1 << 30)
    N = opl.n_rows
    rng = np.random.default_rng(seed)
    threads = os.cpu_count() or 1
    scale = 1.0 / math.sqrt(d)
    done_rows, flops, elapsed = 0, 0.0, 0.0
    batch = 8
    while elapsed < budget_s and done_rows < n_rows_max:
        rows = np.sort(rng.choice(N, size=batch, replace=False)).astype(np.int32)
        Q = np.zeros((N, Hq, d))
        dO = np.zeros((N, Hq, d))
        Q[rows] = synth.hash_rows(synth.STREAM_Q + 16 * seed, rows, Hq * d, torch.bfloat16, 0.5).reshape(-1, Hq, d)
        dO[rows] = synth.hash_rows(synth.STREAM_DO + 16 * seed, rows, Hq * d, torch.bfloat16, 1.0).reshape(-1, Hq, d)
        need = np.zeros(N, dtype=np.uint8)
        need[rows] = 1
        pairs = sum(len(opl.row_context(int(r))[0]) for r in rows)
        t0 = time.perf_counter()
        opl.fwd(Q, scale, rows=rows, nthreads=threads)
        opl.bwd(Q, dO, scale, need_dq=need, need_dkdv=np.zeros(T, dtype=np.uint8), nthreads=threads,
                partial=True)
        elapsed += time.perf_counter() - t0
        flops += 14.0 * d * Hq * pairs
        done_rows += batch
    desc = ("fp64 oracle fwd+bwd of %d sampled rows x %d heads of the %s workload (%.3g of its %d rows); "
            "useful FLOPs 14*d*Hq*pairs of the sample" % (done_rows, Hq, name, done_rows / N, N))
    return flops / elapsed / 1e12, threads, desc, elapsed


# --------------------------------------------------------------------------------------
# GPU legs
# --------------------------------------------------------------------------------------
def timed(torch, stream, fn, steps, warmup, dist=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    times = []
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for _ in range(steps):
        times.append(fn())
    t_all1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    return t_all0.elapsed_time(t_all1), times


def decode_leg(pta, torch, name, seed, dev, stream, steps, warmup, world, dist, hbm, peak_src):
    """Paged decode of the cursors of decode workload `name`: kernel-only GB/s of the
    algorithmic bytes (unique visible K/V tokens + queries, outputs, plan), then plan +
    decode."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    cfg = synth.CONFIGS[name]
    Hq, Hkv, d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
    scale = 1.0 / math.sqrt(d)
    dep, dpool, dkp, dvp, dcfg = build_episode(pta, torch, name, seed, dev)
    curs = dep.cursors
    n = len(curs)
    qd = synth.hash_fill(synth.STREAM_DECODE_Q + 16 * seed, (n, Hq, d), torch.bfloat16, dev, 0.5)
    od = torch.empty_like(qd)
    ld = torch.empty((n, Hq), dtype=torch.float32, device=dev)
    dplan = dpool.decode_plan(curs)
    wsn = dplan.decode_workspace_size(Hq)
    wsd = torch.empty(max(1, wsn), dtype=torch.uint8, device=dev)
    ent = dplan.copy_out()["entries"]
    uniq = unique_tokens(ent, dpool.num_pages, P)
    logical = int((ent["kv_hi"].astype(np.int64) - ent["kv_lo"]).sum())
    tok_bytes = 2 * Hkv * d * 2
    alg_bytes = uniq * tok_bytes + 2 * qd.numel() * 2 + ld.numel() * 4 + len(ent) * 24
    # timed: the decode kernel alone (plan reused), then plan + decode
    dec_times = []

    def dstep():
        a, b = ev(), ev()
        a.record(stream)
        dplan.decode(Hq, qd, od, ld, scale, wsd, wsn, stream=stream)
        b.record(stream)
        dec_times.append((a, b))

    dl0 = pta.launch_count()
    dclk = ClockSampler(dev.index)
    dclk.start()
    dtot, _ = timed(torch, stream, dstep, steps, warmup, dist)
    dclocks = dclk.stop()
    dlaunch = pta.launch_count() - dl0
    kern_ms = statistics.mean([a.elapsed_time(b) for a, b in dec_times[warmup:]])
    plan_ms_list = []

    def pstep():
        a, b = ev(), ev()
        a.record(stream)
        p2 = dpool.decode_plan(curs, stream)
        p2.decode(Hq, qd, od, ld, scale, wsd, wsn, stream=stream)
        b.record(stream)
        plan_ms_list.append((a, b, p2))

    timed(torch, stream, pstep, 3, 1, dist)
    full_ms = statistics.mean([a.elapsed_time(b) for a, b, _ in plan_ms_list[1:]])
    # plan upkeep per decoded token: every cursor one token longer (layout only), then the
    # plan advanced in place vs compiled afresh (both synchronous: wall time)
    upkeep = None
    if all(dpool.append(c, 1, check=False) == pta.OK for c in curs):
        adv_t, fresh_t = [], []
        for it in range(4):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if dplan.advance(stream, check=False) != pta.OK:
                break
            t1 = time.perf_counter()
            p3 = dpool.decode_plan(curs, stream)
            t2 = time.perf_counter()
            adv_t.append(t1 - t0)
            fresh_t.append(t2 - t1)
            del p3
            if it < 3 and not all(dpool.append(c, 1, check=False) == pta.OK for c in curs):
                break
        if adv_t:
            upkeep = {"advance_ms": 1e3 * statistics.median(adv_t),
                      "fresh_plan_ms": 1e3 * statistics.median(fresh_t)}
    world_bytes = world * alg_bytes
    dec = {"metric": "paged decode HBM GB/s", "value": world_bytes / (kern_ms * 1e-3) / 1e9, "unit": "GB/s",
           "workload": WORKLOAD_DESC[name] + "; 16q/4kv heads, d=128, page 64, bf16",
           "ms_per_step": kern_ms, "ms_per_step_with_plan": full_ms, "plan_upkeep": upkeep,
           "cursors": n, "unique_kv_tokens": uniq, "logical_kv_tokens": logical,
           "algorithmic_bytes": alg_bytes, "logical_bytes": logical * tok_bytes,
           "roofline": {"bound": "hbm", "achieved": alg_bytes / (kern_ms * 1e-3) / 1e9, "peak": hbm,
                        "unit": "GB/s", "frac": alg_bytes / (kern_ms * 1e-3) / 1e9 / hbm,
                        "peak_source": peak_src,
                        "traffic": profiled_traffic(name, "octo_decode", "ncu_decode.md", "decode"),
                        "traffic_unit": "bytes per call (ncu dram__bytes_read + write)"},
           "gpu_launches": dlaunch, "clocks": dclocks, "kernel_path": dplan.kernel_path(Hq, 2)}
    del dpool, dkp, dvp
    torch.cuda.empty_cache()
    return dec


def run_ours(args, rank, world, dist):
    import torch
    import packed_tree_attention_gb300 as pta
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pta.load()
    stream = torch.cuda.current_stream()
    hbm, bf16, bf16s, peak_src = peaks()
    seed = rank_seed(args.seed, rank)

    if args.decode_only:
        dec = decode_leg(pta, torch, args.decode_workload, seed, dev, stream, args.decode_steps, args.warmup,
                         world, dist, hbm, peak_src)
        if rank == 0:
            print(json.dumps({"metric": dec["metric"], "value": dec["value"], "unit": dec["unit"], "n_gpus": world,
                              "steps": args.decode_steps, "warmup": args.warmup, "ms_per_step": dec["ms_per_step"],
                              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                              "data": "synthetic (counter-based generator, seed %d + rank)" % args.seed,
                              "config": {"workload": dec["workload"],
                                         "l2": "K/V read larger than L2 (%d MB unique)" % (dec["algorithmic_bytes"] // 10**6)},
                              "decode": dec}))
        return

    # ---------------- training leg: episode fwd + bwd ----------------
    ep, pool, kp, vp, cfg = build_episode(pta, torch, args.workload, seed, dev)
    Hq, Hkv, d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
    scale = 1.0 / math.sqrt(d)
    plan = pool.pack_tree(ep.roots, 128)
    N = plan.info["n_rows"]
    pairs = plan.info["pairs"]
    q = synth.hash_fill(synth.STREAM_Q + 16 * seed, (N, Hq, d), torch.bfloat16, dev, 0.5)
    do = synth.hash_fill(synth.STREAM_DO + 16 * seed, (N, Hq, d), torch.bfloat16, dev, 1.0)
    o = torch.empty_like(q)
    lse = torch.empty((Hq, N), dtype=torch.float32, device=dev)
    dq = torch.empty((N, Hq, d), dtype=torch.float32, device=dev)
    dk = torch.empty((pool.num_pages, Hkv, P, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    ws = torch.empty(max(1, plan.attn_bwd_workspace_size(Hq)), dtype=torch.uint8, device=dev)
    del plan
    q_bytes = q.numel() * q.element_size()
    fwd_flops = 4.0 * d * Hq * pairs
    bwd_flops = 10.0 * d * Hq * pairs
    ev = lambda: torch.cuda.Event(enable_timing=True)
    per = {"pack": [], "fwd": [], "bwd": []}

    def step():
        e0, e1, e2, e3 = ev(), ev(), ev(), ev()
        e0.record(stream)
        pl = pool.pack_tree(ep.roots, 128, stream)
        e1.record(stream)
        pl.attn_fwd(Hq, q, o, lse, scale, stream=stream)
        e2.record(stream)
        pl.attn_bwd(Hq, q, o, lse, do, dq, dk, dv, scale, ws, stream=stream)
        e3.record(stream)
        return (e0, e1, e2, e3, pl)

    launches0 = pta.launch_count()
    clk = ClockSampler(dev.index)
    # warm-up, then the timed steps (inputs > L2: 1 GB of Q alone)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches0 = pta.launch_count()
    clk.start()
    total_ms, recs = timed(torch, stream, step, args.steps, 0, dist)
    clocks = clk.stop()
    launches = pta.launch_count() - launches0
    for e0, e1, e2, e3, pl in recs:
        per["pack"].append(e0.elapsed_time(e1))
        per["fwd"].append(e1.elapsed_time(e2))
        per["bwd"].append(e2.elapsed_time(e3))
    path_fwd = recs[0][4].kernel_path(Hq, 0)
    path_bwd = recs[0][4].kernel_path(Hq, 1)
    del recs
    ms_step = max_over_ranks(total_ms / args.steps, dist)
    value = world * (fwd_flops + bwd_flops) / (ms_step * 1e-3) / 1e12
    fwd_ms = statistics.mean(per["fwd"])
    bwd_ms = statistics.mean(per["bwd"])
    dom = "bwd" if bwd_ms >= fwd_ms else "fwd"
    dom_flops = bwd_flops if dom == "bwd" else fwd_flops
    dom_ms = max(bwd_ms, fwd_ms)
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12

    # ---------------- e2e leg: host buffers through the public API ----------------
    e2e = None
    if not args.no_e2e:
        hq = q.cpu().pin_memory()
        hdo = do.cpu().pin_memory()
        hk = kp.cpu().pin_memory()
        hv = vp.cpu().pin_memory()
        hdq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
        hdk = torch.empty(dk.shape, dtype=dk.dtype).pin_memory()
        hdv = torch.empty(dv.shape, dtype=dv.dtype).pin_memory()
        q2, do2 = torch.empty_like(q), torch.empty_like(do)

        def e2e_step():
            q2.copy_(hq, non_blocking=True)
            do2.copy_(hdo, non_blocking=True)
            kp.copy_(hk, non_blocking=True)
            vp.copy_(hv, non_blocking=True)
            pl = pool.pack_tree(ep.roots, 128, stream)
            pl.attn_fwd(Hq, q2, o, lse, scale, stream=stream)
            pl.attn_bwd(Hq, q2, o, lse, do2, dq, dk, dv, scale, ws, stream=stream)
            hdq.copy_(dq, non_blocking=True)
            hdk.copy_(dk, non_blocking=True)
            hdv.copy_(dv, non_blocking=True)
            return pl

        e2e_steps = max(1, min(args.steps, 3))
        e_ms, _ = timed(torch, stream, e2e_step, e2e_steps, 1, dist)
        e_ms = max_over_ranks(e_ms / e2e_steps, dist)
        h2d = sum(x.numel() * x.element_size() for x in (hq, hdo, hk, hv))
        d2h = sum(x.numel() * x.element_size() for x in (hdq, hdk, hdv))
        e2e = {"value": world * (fwd_flops + bwd_flops) / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}
        del hq, hdo, hk, hv, hdq, hdk, hdv, q2, do2

    # ---------------- rotary embedding leg (rows of the episode plan) ----------------
    rope = None
    if not args.no_rope:
        rplan = pool.pack_tree(ep.roots, 128)
        rt = []

        def rstep():
            a, b, c = ev(), ev(), ev()
            a.record(stream)
            rplan.rope_rows(Hq, q, 10000.0, stream=stream)              # queries, bf16
            b.record(stream)
            rplan.rope_rows(Hq, dq, 10000.0, inverse=True, stream=stream)   # query gradients, fp32
            c.record(stream)
            rt.append((a, b, c))

        timed(torch, stream, rstep, 5, 3, dist)
        q_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in rt[3:])
        g_ms = statistics.mean(b.elapsed_time(c) for _, b, c in rt[3:])
        qb = 2 * q.numel() * q.element_size() + N * 4       # read + write + row positions
        gb = 2 * dq.numel() * dq.element_size() + N * 4
        rope = {"metric": "rotary embedding of packed rows, HBM GB/s",
                "q_bf16": {"value": qb / (q_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": q_ms,
                           "frac": qb / (q_ms * 1e-3) / 1e9 / hbm},
                "dq_f32_inverse": {"value": gb / (g_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": g_ms,
                                   "frac": gb / (g_ms * 1e-3) / 1e9 / hbm},
                "peak": hbm, "peak_source": peak_src}
        del rplan

    # ---------------- per-token log-probability / loss leg (rows of the episode plan) ----
    logprob = None
    if not args.no_logprob:
        lplan = pool.pack_tree(ep.roots, 128)
        V, R = 151936, min(16384, N)
        lx = synth.hash_fill(synth.STREAM_Q + 101 + 16 * seed, (R, V), torch.bfloat16, dev, 3.0, chunk_rows=1024)
        lg = torch.empty_like(lx)
        rng = np.random.default_rng(seed)
        lids = torch.from_numpy(rng.integers(0, V, N).astype(np.int32)).to(dev)
        lw = torch.from_numpy(rng.uniform(0, 1, N).astype(np.float32)).to(dev)
        llogp = torch.empty(N, dtype=torch.float32, device=dev)
        lloss = torch.empty(1, dtype=torch.float32, device=dev)
        lws = torch.empty(lplan.token_logprob_workspace_size(R), dtype=torch.uint8, device=dev)
        lt = []

        def lstep():
            a, b, c = ev(), ev(), ev()
            a.record(stream)
            lplan.token_logprob(0, R, lx, V, lids, lw, llogp, lws, loss=lloss, stream=stream)   # terms only
            b.record(stream)
            lplan.token_logprob(0, R, lx, V, lids, lw, llogp, lws, dlogits=lg, loss=lloss, stream=stream)
            c.record(stream)
            lt.append((a, b, c))

        timed(torch, stream, lstep, 6, 3, dist)
        f_ms = statistics.mean(a.elapsed_time(b) for a, b, _ in lt[3:])
        g_ms = statistics.mean(b.elapsed_time(c) for _, b, c in lt[3:])
        small = 3 * N * 4 + R * 4                       # ids, weights, logp; loss partials
        fb = lx.numel() * 2 + small                      # one read of the logits
        gb = 2 * lx.numel() * 2 + small                  # + one write of the gradient
        logprob = {"metric": "per-token log-prob / loss over packed rows, HBM GB/s",
                   "workload": "%d episode rows x vocabulary %d, bf16 logits (%.1f GB)" % (R, V, lx.numel() * 2 / 1e9),
                   "terms": {"value": fb / (f_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": f_ms,
                             "frac": fb / (f_ms * 1e-3) / 1e9 / hbm},
                   "terms_and_gradient": {"value": gb / (g_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": g_ms,
                                          "frac": gb / (g_ms * 1e-3) / 1e9 / hbm},
                   "peak": hbm, "peak_source": peak_src}
        del lplan, lx, lg, lids, lw, llogp, lloss, lws

    # free the training leg before the decode leg
    del pool, kp, vp, q, do, o, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()

    # ---------------- decode leg ----------------
    dec = None
    if not args.no_decode:
        dec = decode_leg(pta, torch, args.decode_workload, seed, dev, stream, args.decode_steps, args.warmup,
                         world, dist, hbm, peak_src)

    # ---------------- cursor view: the context of one 128K-token cursor ----------------
    view = None
    if not args.no_decode:
        vpool = pta.Pool(2112, 64, Hkv, d, pta.DTYPE_BF16)    # metadata only: no K/V arrays
        r0 = vpool.root()
        vpool.append(r0, 16384)
        kids = vpool.fork(r0, 2)
        vpool.append(kids[0], 8192)
        vpool.append(kids[1], 16384)
        vpool.mount(kids[1], kids[0], 1024, 8192)          # a sibling span read in place
        vpool.append(kids[1], 131072 - 16384 - 16384 - 7168)
        vt = []
        for i in range(8):
            a, b = ev(), ev()
            a.record(stream)
            vp_ = vpool.decode_plan([kids[1]], stream)
            b.record(stream)
            torch.cuda.synchronize()
            vt.append(a.elapsed_time(b))
            ctx = vp_.info["pairs"]
            del vp_
        view = {"metric": "cursor view (context runs of one cursor, via the decode plan)",
                "context_tokens": int(ctx), "ms": statistics.median(vt[2:])}
        del vpool

    # ---------------- CPU baseline (rank 0, N = 1) ----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, thr, desc, el = oracle_sample(args.workload, seed, budget_s=args.cpu_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc, "seconds": el}

    out = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (counter-based generator, seed %d + rank)" % args.seed,
        "config": {"workload": workload_desc(args.workload, cfg),
                   "packed_tokens": N, "visible_pairs": pairs, "useful_tflop_per_step": (fwd_flops + bwd_flops) / 1e12,
                   "step": "plan compile + fwd + bwd",
                   "l2": ("inputs larger than L2 (Q alone %.0f MB)" if q_bytes > L2_BYTES else
                          "inputs fit in L2 (Q %.0f MB): timings include L2 reuse") % (q_bytes / 1e6),
                   "parallelism": "replicas: one episode per GPU, no collective"},
        "breakdown_ms": {k: statistics.mean(v) for k, v in per.items()},
        "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": bwd_flops / (bwd_ms * 1e-3) / 1e12,
        "roofline": {"bound": "tensor", "kernel": "octo_attn_" + dom, "achieved": achieved, "peak": bf16s,
                     "unit": "TFLOP/s", "frac": achieved / bf16s, "peak_source": peak_src + " (sustained bf16)",
                     "traffic": profiled_traffic(args.workload, "octo_attn_" + dom),
                     "traffic_unit": "bytes per call (ncu dram__bytes_read + write)"},
        "kernel_path": {"fwd": path_fwd, "bwd": path_bwd},
        "clocks": clocks,
        "gpu_launches": launches,
        "e2e": e2e,
        "decode": dec,
        "rope": rope,
        "token_logprob": logprob,
        "cursor_view": view,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out))


def run_reference(args, rank, world):
    if rank != 0:
        return
    per = []
    thr = None
    desc = None
    for i in range(args.warmup + args.steps):
        v, thr, desc, el = oracle_sample(args.workload, args.seed, budget_s=args.ref_budget, n_rows_max=64)
        if i >= args.warmup:
            per.append((v, el))
    value = statistics.mean(v for v, _ in per)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(e for _, e in per),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (counter-based generator, seed %d)" % args.seed,
           "config": {"workload": workload_desc(args.workload, synth.CONFIGS[args.workload]) +
                                  "; each step a bounded row sample"},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--decode-steps", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="episode")
    ap.add_argument("--no-rope", action="store_true")
    ap.add_argument("--no-logprob", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--decode-only", action="store_true", help="only the decode leg (profiling runs)")
    ap.add_argument("--decode-workload", default="decode", help="decode or decode_small (32 cursors)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=8.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    run_ours(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
