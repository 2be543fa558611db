"""Benchmark: packed DAG attention forward + backward (useful TFLOP/s) and paged decode
(HBM GB/s) on one GB300, through the C ABI.

One step = one pass of the training hot path over the training-step workload (8 random
trees of 140K owned tokens each, 1.12M packed rows; fork fan-out 2-6, depth <= 3, 0-4
mounted spans per reader; 16 q / 4 kv heads, d 128, page 64, bf16): the GPU plan compile
(positions + tile list + CSC), the forward, and the backward.  The same step over the
episode workload (16K prefix, 7 branches x 32K owned tokens, 3 rewinds, 6 mounts) is a
second object on the line.  The decode leg times the decode plan and the paged decode of
256 cursors (32 episodes x 8, mean context ~26K tokens) the same way.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own workload (a different seed): weak scaling, no
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


# ncu traffic may be taken on a smaller case of the same kernels: one tree of the training
# step, 32 of the 256 decode cursors; bench scales it to the workload by its units of work
TRAFFIC_CASES = {"train_step": ("train_tree", "train_step"), "episode": ("episode",),
                 "decode": ("decode_small", "decode"), "decode_small": ("decode_small",)}


def profiled_traffic(workload, call, units):
    """(DRAM bytes per call, note) of `call` on `workload` from the committed ncu summaries
    under profiles/.  A line 'traffic: <call> <case> <bytes> bytes per call, <units> units'
    gives the bytes measured on <case> with <units> units of work (visible pairs for the
    attention calls, algorithmic bytes for the decode); a case in TRAFFIC_CASES[workload]
    is scaled to `units`.  (None, reason) when no summary has it or when a kernel source
    named by a fingerprint line of that summary has changed since the counters."""
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "packed_tree_attention_gb300", "csrc")
    cases = TRAFFIC_CASES.get(workload, (workload,))
    best = None
    for fname in sorted(os.listdir(os.path.join(here, "profiles"))):
        if not fname.endswith(".md"):
            continue
        want, found = {}, []
        for line in open(os.path.join(here, "profiles", fname)):
            line = line.strip()
            if " sha256/16: " in line:
                name, h = line.split(" sha256/16: ")
                want[name] = h
            elif line.startswith("traffic: "):
                f = line[len("traffic: "):].replace(",", "").split()
                if len(f) >= 7 and f[0] == call and f[1] in cases:
                    found.append((cases.index(f[1]), f[1], int(f[2]), int(f[6])))
        if not found:
            continue
        if any(code_fingerprint(os.path.join(src, n)) != h for n, h in want.items()):
            best = best or (None, "%s: kernel sources changed since the counters" % fname)
            continue
        rank, case, b, u = min(found)
        if best is None or best[0] is None:
            scaled = int(round(b * units / u))
            note = ("profiles/%s, measured on %s" % (fname, case) +
                    ("" if case == workload else ", scaled by units of work %d/%d" % (units, u)))
            best = (scaled, note)
    return best if best else (None, "no ncu summary for this workload")


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
    "train_step": "train step: 8 trees of 140K owned tokens (1.12M), fan-out 2-6, depth <= 3, 0-4 mounts per reader",
    "train_tree": "one tree of the train step: 140K owned tokens, fan-out 2-6, depth <= 3, 0-4 mounts per reader",
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
class OracleSampler:
    """The fp64 oracle's forward + backward on seeded samples of packed rows of a workload
    (all 16 heads of each row; the backward's dK/dV from those rows only).  The oracle
    replays the op log without values and gets K/V rows only for the tokens in the sampled
    rows' contexts, generated on `kv_device` before the timed calls.  The training step's
    trees are independent units of the same statistics, so its rows are sampled from its
    first tree, replayed alone."""

    def __init__(self, name, seed, kv_device="cpu"):
        import oracle
        self.name, self.seed, self.kv_device = name, seed, kv_device
        cfg = synth.CONFIGS[name]
        self.Hq, self.Hkv, self.d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
        self.unit = "train_tree" if name == "train_step" else name
        ep = synth.make_preset(self.unit, seed=seed)
        self.T = ep.n_tokens
        npages = sum((L + P - 1) // P for L in ep.length) + 8 + 4 * len(ep.cursors)
        self.orc = oracle.Oracle(P, npages, self.Hkv, self.d)
        self.orc.replay(ep)
        self.opl = self.orc.pack(ep.roots, 128, tile_stride=1 << 30)
        self.N = self.opl.n_rows
        self.rng = np.random.default_rng(seed)
        self.threads = os.cpu_count() or 1
        self.kv_set = np.zeros(self.T, dtype=bool)
        self.rows_done = 0

    def batch(self, n_rows):
        """One timed batch of n_rows sampled rows: returns (useful FLOPs, seconds)."""
        import torch
        Hq, Hkv, d, seed = self.Hq, self.Hkv, self.d, self.seed
        rows = np.sort(self.rng.choice(self.N, size=n_rows, replace=False)).astype(np.int32)
        ctx = [self.opl.row_context(int(r))[0] for r in rows]
        toks = np.unique(np.concatenate(ctx))
        toks = toks[~self.kv_set[toks]]
        if len(toks):
            K = synth.hash_rows(synth.STREAM_K + 16 * seed, toks, Hkv * d, torch.bfloat16, 0.5, self.kv_device)
            V = synth.hash_rows(synth.STREAM_V + 16 * seed, toks, Hkv * d, torch.bfloat16, 0.5, self.kv_device)
            self.orc.set_kv(toks, K.reshape(-1, Hkv, d), V.reshape(-1, Hkv, d))
            self.kv_set[toks] = True
        Q = np.zeros((self.N, Hq, d))
        dO = np.zeros((self.N, Hq, d))
        Q[rows] = synth.hash_rows(synth.STREAM_Q + 16 * seed, rows, Hq * d, torch.bfloat16, 0.5,
                                  self.kv_device).reshape(-1, Hq, d)
        dO[rows] = synth.hash_rows(synth.STREAM_DO + 16 * seed, rows, Hq * d, torch.bfloat16, 1.0,
                                   self.kv_device).reshape(-1, Hq, d)
        need = np.zeros(self.N, dtype=np.uint8)
        need[rows] = 1
        pairs = sum(len(c) for c in ctx)
        scale = 1.0 / math.sqrt(d)
        t0 = time.perf_counter()
        self.opl.fwd(Q, scale, rows=rows, nthreads=self.threads)
        self.opl.bwd(Q, dO, scale, need_dq=need, need_dkdv=np.zeros(self.T, dtype=np.uint8), nthreads=self.threads,
                     partial=True)
        el = time.perf_counter() - t0
        self.rows_done += n_rows
        return 14.0 * d * Hq * pairs, el

    def describe(self):
        where = ("its first tree (%d of its rows; the 8 trees are independent)" % self.N
                 if self.unit != self.name else "its %d rows" % self.N)
        return ("fp64 oracle fwd+bwd of %d rows x %d heads sampled from %s of the %s workload; useful FLOPs "
                "14*d*Hq*pairs of the sample" % (self.rows_done, self.Hq, where, self.name))


def oracle_sample(name, seed, budget_s=15.0, n_rows_max=256, kv_device="cpu"):
    """(TFLOP/s, threads, description, seconds) of the oracle on row batches of 8 until
    about budget_s seconds of timed oracle work."""
    smp = OracleSampler(name, seed, kv_device)
    flops, elapsed = 0.0, 0.0
    while elapsed < budget_s and smp.rows_done < n_rows_max:
        f, el = smp.batch(8)
        flops += f
        elapsed += el
    return flops / elapsed / 1e12, smp.threads, smp.describe(), elapsed


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
    algorithmic bytes (unique visible K/V tokens + queries, outputs, plan); then a fresh
    plan + decode, and serving steps of one new token per cursor with the plan advanced in
    place + decode."""
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
    wsd = torch.empty(max(1, 2 * wsn), dtype=torch.uint8, device=dev)   # room for runs added by advances
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
    fresh_ms = statistics.mean([a.elapsed_time(b) for a, b, _ in plan_ms_list[1:]])
    # serving steps with plan upkeep: every cursor gets one token (octo_append_step, layout
    # only: the new slots keep their zeroed K/V), the plan is advanced in place and the
    # cursors decoded;
    # CUDA-event time per step over the whole run (host work between launches included
    # where the GPU waits for it), and the advance's wall time on the host
    upkeep = None
    adv_wall = []

    def ustep():
        if dpool.append_step(curs, stream=stream, check=False) != pta.OK:
            raise RuntimeError("decode pool full")
        t0 = time.perf_counter()
        dplan.advance(stream)
        adv_wall.append(time.perf_counter() - t0)
        wsz = dplan.decode_workspace_size(Hq)
        assert wsz <= 2 * wsn
        dplan.decode(Hq, qd, od, ld, scale, wsd, wsz, stream=stream)

    u_steps = 20
    u_ms, _ = timed(torch, stream, ustep, u_steps, 3, dist)
    upkeep = {"ms_per_step_advance_and_decode": u_ms / u_steps, "advance_wall_ms": 1e3 * statistics.median(adv_wall),
              "steps": u_steps, "fresh_plan_and_decode_ms": fresh_ms}
    world_bytes = world * alg_bytes
    dec_traffic, dec_note = profiled_traffic(name, "octo_decode", alg_bytes)
    dec = {"metric": "paged decode HBM GB/s", "value": world_bytes / (kern_ms * 1e-3) / 1e9, "unit": "GB/s",
           "workload": WORKLOAD_DESC[name] + "; 16q/4kv heads, d=128, page 64, bf16",
           "ms_per_step": kern_ms, "plan_upkeep": upkeep,
           "cursors": n, "unique_kv_tokens": uniq, "logical_kv_tokens": logical,
           "algorithmic_bytes": alg_bytes, "logical_bytes": logical * tok_bytes,
           "roofline": {"bound": "hbm", "achieved": alg_bytes / (kern_ms * 1e-3) / 1e9, "peak": hbm,
                        "unit": "GB/s", "frac": alg_bytes / (kern_ms * 1e-3) / 1e9 / hbm,
                        "peak_source": peak_src,
                        "traffic": dec_traffic, "traffic_note": dec_note,
                        "traffic_unit": "bytes per call (ncu dram__bytes_read + write)"},
           "gpu_launches": dlaunch, "clocks": dclocks, "kernel_path": dplan.kernel_path(Hq, 2)}
    del dpool, dkp, dvp
    torch.cuda.empty_cache()
    return dec


def train_leg(pta, torch, name, seed, dev, stream, steps, warmup, world, dist, bf16s, peak_src, with_e2e):
    """One step = plan compile + forward + backward of training workload `name`; useful
    TFLOP/s over the step, per-call times, the backward's roofline and (with_e2e) the same
    step through host buffers.  Returns a dict; its "_state", "_q" and "_dq" entries hand
    the workload on to the legs that reuse it."""
    ep, pool, kp, vp, cfg = build_episode(pta, torch, name, seed, dev)
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

    clk = ClockSampler(dev.index)
    # warm-up, then the timed steps (inputs > L2: Q alone is hundreds of MB)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    launches0 = pta.launch_count()
    clk.start()
    total_ms, recs = timed(torch, stream, step, steps, 0, dist)
    clocks = clk.stop()
    launches = pta.launch_count() - launches0
    for e0, e1, e2, e3, pl in recs:
        per["pack"].append(e0.elapsed_time(e1))
        per["fwd"].append(e1.elapsed_time(e2))
        per["bwd"].append(e2.elapsed_time(e3))
    path_fwd = recs[0][4].kernel_path(Hq, 0)
    path_bwd = recs[0][4].kernel_path(Hq, 1)
    del recs
    ms_step = max_over_ranks(total_ms / steps, dist)
    value = world * (fwd_flops + bwd_flops) / (ms_step * 1e-3) / 1e12
    fwd_ms = statistics.mean(per["fwd"])
    bwd_ms = statistics.mean(per["bwd"])
    dom = "bwd" if bwd_ms >= fwd_ms else "fwd"
    dom_flops = bwd_flops if dom == "bwd" else fwd_flops
    dom_ms = max(bwd_ms, fwd_ms)
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12

    # e2e: host buffers through the public API, copies inside the timed region.  The
    # steps are pipelined the way a training loop prefetches its batches: while step i
    # computes, step i + 1's Q, dO and K/V come in on one copy stream and step i - 1's dQ,
    # dK, dV go out on another.  Q / dO and the gradients are double-buffered; K/V land in
    # a device staging buffer and are copied into the pool's storage at the step's start
    # (the pool owns one K/V store).  Every step's inputs are copied in and its gradients
    # read back inside the timed region.
    e2e = None
    if with_e2e:
        hq = q.cpu().pin_memory()
        hdo = do.cpu().pin_memory()
        hk = kp.cpu().pin_memory()
        hv = vp.cpu().pin_memory()
        hdq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
        hdk = torch.empty(dk.shape, dtype=dk.dtype).pin_memory()
        hdv = torch.empty(dv.shape, dtype=dv.dtype).pin_memory()
        qb = [torch.empty_like(q), torch.empty_like(q)]
        dob = [torch.empty_like(do), torch.empty_like(do)]
        kst, vst = torch.empty_like(kp), torch.empty_like(vp)
        dqb, dkb, dvb = [dq, torch.empty_like(dq)], [dk, torch.empty_like(dk)], [dv, torch.empty_like(dv)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        mk = lambda: torch.cuda.Event()
        in_ready, in_free, out_free, done = [mk(), mk()], [mk(), mk()], [mk(), mk()], [mk(), mk()]
        stage_free = mk()

        def load(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(in_free[b])      # step i - 2 is done with these buffers
                qb[b].copy_(hq, non_blocking=True)
                dob[b].copy_(hdo, non_blocking=True)
                if i >= 1:
                    s_in.wait_event(stage_free)      # step i - 1 has taken its K/V from staging
                kst.copy_(hk, non_blocking=True)
                vst.copy_(hv, non_blocking=True)
                in_ready[b].record(s_in)

        def e2e_run(n):
            load(0)
            for i in range(n):
                b = i & 1
                stream.wait_event(in_ready[b])
                kp.copy_(kst, non_blocking=True)
                vp.copy_(vst, non_blocking=True)
                stage_free.record(stream)
                if i + 1 < n:
                    load(i + 1)
                if i >= 2:
                    stream.wait_event(out_free[b])   # step i - 2's gradients are out
                pl = pool.pack_tree(ep.roots, 128, stream)
                pl.attn_fwd(Hq, qb[b], o, lse, scale, stream=stream)
                pl.attn_bwd(Hq, qb[b], o, lse, dob[b], dqb[b], dkb[b], dvb[b], scale, ws, stream=stream)
                in_free[b].record(stream)
                done[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[b])
                    hdq.copy_(dqb[b], non_blocking=True)
                    hdk.copy_(dkb[b], non_blocking=True)
                    hdv.copy_(dvb[b], non_blocking=True)
                    out_free[b].record(s_out)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)

        dq_ref = dq.cpu()   # the device-only step's dQ: the pipelined steps must reproduce it bit for bit
        e2e_run(2)   # warm-up
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e2e_steps = max(3, steps)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        s_in.wait_stream(stream)
        e2e_run(e2e_steps)
        t1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        e_ms = max_over_ranks(t0.elapsed_time(t1) / e2e_steps, dist)
        if not torch.equal(hdq, dq_ref):
            raise RuntimeError("e2e: the pipelined step's dQ differs from the device-only step's")
        del dq_ref
        h2d = sum(x.numel() * x.element_size() for x in (hq, hdo, hk, hv))
        d2h = sum(x.numel() * x.element_size() for x in (hdq, hdk, hdv))
        e2e = {"value": world * (fwd_flops + bwd_flops) / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": e2e_steps, "overlap": "copies of the neighbouring steps overlap each step's compute",
               "check": "the last step's dQ read back equals the device-only step's bit for bit"}
        del hq, hdo, hk, hv, hdq, hdk, hdv, qb, dob, kst, vst, dqb, dkb, dvb
    traffic, traffic_note = profiled_traffic(name, "octo_attn_" + dom, pairs)
    out = {
        "value": value, "ms_per_step": ms_step,
        "config": {"workload": workload_desc(name, cfg),
                   "packed_tokens": N, "visible_pairs": pairs, "useful_tflop_per_step": (fwd_flops + bwd_flops) / 1e12,
                   "step": "plan compile + fwd + bwd",
                   "l2": ("inputs larger than L2 (Q alone %.0f MB)" if q_bytes > L2_BYTES else
                          "inputs fit in L2 (Q %.0f MB): timings include L2 reuse") % (q_bytes / 1e6),
                   "parallelism": "replicas: one workload per GPU, no collective"},
        "breakdown_ms": {k: statistics.mean(v) for k, v in per.items()},
        "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": bwd_flops / (bwd_ms * 1e-3) / 1e12,
        "roofline": {"bound": "tensor", "kernel": "octo_attn_" + dom, "achieved": achieved, "peak": bf16s,
                     "unit": "TFLOP/s", "frac": achieved / bf16s, "peak_source": peak_src + " (sustained bf16)",
                     "traffic": traffic, "traffic_note": traffic_note,
                     "traffic_unit": "bytes per call (ncu dram__bytes_read + write)"},
        "kernel_path": {"fwd": path_fwd, "bwd": path_bwd},
        "clocks": clocks,
        "gpu_launches": launches,
        "e2e": e2e,
    }
    del o, lse, do, dk, dv, ws
    out["_state"] = (ep, pool, kp, vp, cfg)
    out["_q"], out["_dq"] = q, dq
    return out


# FP32 fused multiply-add peak of GB300 from its unit counts: 152 SMs x 128 FP32 lanes x
# 2 FLOP per FMA x the 2070 MHz maximum SM clock
FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def recurrent_flops(n_chunks, H, D, C=64):
    """Executed FLOPs of the chunked gated delta rule (every chunk computed at full size):
    forward 3 C D^2 + 5 C^2 D + C^3 / 6 multiply-adds per (chunk, head), backward
    9 C D^2 + 14 C^2 D."""
    fwd = 2.0 * (3 * C * D * D + 5 * C * C * D + C ** 3 / 6) * n_chunks * H
    bwd = 2.0 * (9 * C * D * D + 14 * C * C * D) * n_chunks * H
    return fwd, bwd


def recurrent_leg(pta, torch, name, seed, dev, stream, steps, warmup, dist, H=16, D=128):
    """Tree-packed recurrent layer (gated delta rule) over the rows of training workload
    `name`: forward and backward, fp32, H heads of head_dim D."""
    ep = synth.make_preset(name, seed=seed)
    P = synth.CONFIGS[name]["P"]
    pool = pta.Pool(sum((L + P - 1) // P for L in ep.length) + 8, P, 1, 64, pta.DTYPE_F32)   # layout only
    for op in ep.ops:
        kind = op[0]
        if kind == "root":
            pool.root()
        elif kind == "append":
            pool.append(op[1], op[2])
        elif kind == "fork":
            pool.fork(op[1], op[2])
        elif kind == "mount":
            pool.mount(*op[1:])
        elif kind == "rewind":
            pool.rewind(op[1], op[2])
        elif kind == "done":
            pool.done(op[1])
    plan = pool.pack_tree(ep.roots, 128)
    N = plan.info["n_rows"]
    gen = lambda s, shape: synth.hash_fill(s, shape, torch.float32, dev, 1.0)
    q = gen(synth.STREAM_Q + 200 + 16 * seed, (N, H, D))
    k = gen(synth.STREAM_K + 200 + 16 * seed, (N, H, D))
    k /= k.norm(dim=2, keepdim=True)
    v = gen(synth.STREAM_V + 200 + 16 * seed, (N, H, D))
    do = gen(synth.STREAM_DO + 200 + 16 * seed, (N, H, D))
    g = torch.Generator(device=dev).manual_seed(seed)
    a = 0.6 + 0.4 * torch.rand((N, H), generator=g, device=dev)
    b = torch.rand((N, H), generator=g, device=dev)
    o = torch.empty_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    da, db = torch.empty_like(a), torch.empty_like(a)
    ws = torch.empty(plan.recurrent_workspace_size(H, D), dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    rec = []

    def step():
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        plan.recurrent_fwd(H, D, q, k, v, a, b, o, ws, stream=stream)
        e1.record(stream)
        plan.recurrent_bwd(H, D, q, k, v, a, b, do, dq, dk, dv, da, db, ws, stream=stream)
        e2.record(stream)
        rec.append((e0, e1, e2))

    l0 = pta.launch_count()
    timed(torch, stream, step, steps, warmup, dist)
    launches = (pta.launch_count() - l0) // (steps + warmup)
    fwd_ms = statistics.mean(x.elapsed_time(y) for x, y, _ in rec[warmup:])
    bwd_ms = statistics.mean(y.elapsed_time(z) for _, y, z in rec[warmup:])
    fwd_f, bwd_f = recurrent_flops(plan.info["n_rec_chunks"], H, D)
    out = {"metric": "tree-packed recurrent layer (gated delta rule) fwd + bwd, executed TFLOP/s",
           "workload": "%s DAG rows (%d packed rows), %d heads, head_dim %d, fp32, chunks of 64" % (name, N, H, D),
           "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
           "fwd_tflops": fwd_f / (fwd_ms * 1e-3) / 1e12, "bwd_tflops": bwd_f / (bwd_ms * 1e-3) / 1e12,
           "launches_per_step": launches,
           "roofline": {"bound": "alu", "achieved": (fwd_f + bwd_f) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
                        "peak": FFMA_PEAK_TFLOPS, "unit": "TFLOP/s",
                        "frac": (fwd_f + bwd_f) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12 / FFMA_PEAK_TFLOPS,
                        "peak_source": "derived: FP32 FMA lanes x 2 x max SM clock", "traffic": None}}
    del q, k, v, do, a, b, o, dq, dk, dv, da, db, ws, plan, pool
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, dist):
    import torch
    import packed_tree_attention_gb300 as pta
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pta.load()
    stream = torch.cuda.current_stream()
    hbm, bf16, bf16s, peak_src = peaks()
    seed = rank_seed(args.seed, rank)

    if args.recurrent_only:
        rec = recurrent_leg(pta, torch, args.recurrent_workload, seed, dev, stream, args.steps, args.warmup, dist)
        if rank == 0:
            print(json.dumps({"metric": rec["metric"], "value": rec["roofline"]["achieved"], "unit": "TFLOP/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": rec["fwd_ms"] + rec["bwd_ms"], "higher_is_better": True,
                              "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                              "data": "synthetic (counter-based generator, seed %d + rank)" % args.seed,
                              "config": {"workload": rec["workload"]}, "recurrent": rec}))
        return

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

    # ---------------- training leg: fwd + bwd of the headline workload ----------------
    tr = train_leg(pta, torch, args.workload, seed, dev, stream, args.steps, args.warmup, world, dist, bf16s,
                   peak_src, with_e2e=not args.no_e2e)
    ep, pool, kp, vp, cfg = tr.pop("_state")
    Hq, Hkv, d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
    q, dq, N = tr.pop("_q"), tr.pop("_dq"), tr["config"]["packed_tokens"]
    ev = lambda: torch.cuda.Event(enable_timing=True)

    # ---------------- rotary embedding leg (rows of the headline workload's plan) ----------------
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

    # ---------------- per-token log-probability / loss leg (rows of the same plan) ----
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
                   "workload": "%d packed rows of the %s workload x vocabulary %d, bf16 logits (%.1f GB)" % (
                       R, args.workload, V, lx.numel() * 2 / 1e9),
                   "terms": {"value": fb / (f_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": f_ms,
                             "frac": fb / (f_ms * 1e-3) / 1e9 / hbm},
                   "terms_and_gradient": {"value": gb / (g_ms * 1e-3) / 1e9, "unit": "GB/s", "ms": g_ms,
                                          "frac": gb / (g_ms * 1e-3) / 1e9 / hbm},
                   "peak": hbm, "peak_source": peak_src}
        del lplan, lx, lg, lids, lw, llogp, lloss, lws

    # free the headline workload, then the second training workload (same step, fewer steps)
    del pool, kp, vp, q, dq, ep
    torch.cuda.empty_cache()
    second = None
    if args.second_workload and args.second_workload != args.workload:
        second = train_leg(pta, torch, args.second_workload, seed, dev, stream, max(3, min(args.steps, 10)),
                           args.warmup, world, dist, bf16s, peak_src, with_e2e=False)
        for k in ("_state", "_q", "_dq"):
            second.pop(k)
        torch.cuda.empty_cache()

    # ---------------- tree-packed recurrent layer (episode DAG rows) ----------------
    rec = None
    if not args.no_recurrent:
        rec = recurrent_leg(pta, torch, "episode", seed, dev, stream, 3, 2, dist)

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
        v, thr, desc, el = oracle_sample(args.workload, seed, budget_s=args.cpu_budget, kv_device="cuda")
        cpu = {"value": v, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc, "seconds": el}

    out = {
        "metric": METRIC,
        "value": tr["value"],
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tr["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (counter-based generator, seed %d + rank)" % args.seed,
        "config": tr["config"],
        "breakdown_ms": tr["breakdown_ms"],
        "fwd_tflops": tr["fwd_tflops"],
        "bwd_tflops": tr["bwd_tflops"],
        "roofline": tr["roofline"],
        "kernel_path": tr["kernel_path"],
        "clocks": tr["clocks"],
        "gpu_launches": tr["gpu_launches"],
        "e2e": tr["e2e"],
        "second_workload": second,
        "recurrent": rec,
        "decode": dec,
        "rope": rope,
        "token_logprob": logprob,
        "cursor_view": view,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(out))


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle, as it stands, on the host cores; each step one
    batch of sampled rows of the same workload (the oracle state built once, untimed)."""
    if rank != 0:
        return
    smp = OracleSampler(args.workload, args.seed)
    per = []
    for i in range(args.warmup + args.steps):
        f, el = smp.batch(args.ref_rows)
        if i >= args.warmup:
            per.append((f, el))
    flops = sum(f for f, _ in per)
    secs = sum(e for _, e in per)
    value = flops / secs / 1e12
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(per),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (counter-based generator, seed %d)" % args.seed,
           "config": {"workload": workload_desc(args.workload, synth.CONFIGS[args.workload]) +
                                  "; each step a batch of %d sampled rows" % args.ref_rows},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": smp.threads, "kind": "oracle",
                            "sample": smp.describe()},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--decode-steps", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="train_step")
    ap.add_argument("--second-workload", default="episode", help="a second training workload on the same line ('' = none)")
    ap.add_argument("--no-rope", action="store_true")
    ap.add_argument("--no-logprob", action="store_true")
    ap.add_argument("--no-recurrent", action="store_true")
    ap.add_argument("--recurrent-only", action="store_true", help="only the recurrent-layer leg (profiling runs)")
    ap.add_argument("--recurrent-workload", default="episode", help="DAG whose rows the recurrent leg runs over")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--decode-only", action="store_true", help="only the decode leg (profiling runs)")
    ap.add_argument("--decode-workload", default="decode", help="decode or decode_small (32 cursors)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=2, help="sampled rows per step of the reference arm")
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
