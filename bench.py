#!/usr/bin/env python
"""Benchmark of the MALA hot path on GB300.

One step = one pass of the whole path on synthetic planted-peak data:
  MALA forward + backward on the 128K prefill workload (B=1, 8 query / 8 KV
  heads, L=131072, d=128, bf16, 128x128 tiles) and one split-KV decode step on
  the 128K decode workload (batch 8, 32 query / 8 KV heads, 131072-token bf16
  cache, 16 splits), all at tau = 1.
The same steps are then timed at tau = 0 (dense, same kernels) for the speedup,
and the 32K prefill workload's forward and backward are timed at both taus
(reported under "secondary").

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MALA fwd/bwd ms & TFLOP/s at 32K/128K, decode µs/token at 128K; % roofline"
WORKLOADS = {
    "128k": ("prefill_128k", "decode_128k"),
    "32k": ("prefill_32k", "decode_128k"),
}
L2_BYTES = 129 * 1024 * 1024
SMS = 152


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["mala", "reference"], default="mala")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="128k")
    p.add_argument("--tau", type=float, default=1.0)
    p.add_argument("--no-dense", action="store_true", help="skip the tau = 0 comparison loop")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-32k", action="store_true",
                   help="skip the secondary timings (32K prefill, per-head decode)")
    p.add_argument("--sample-seconds", type=float, default=15.0)
    p.add_argument("--e2e-chunks", type=int, default=8,
                   help="head chunks of the end-to-end prefill pipeline (rounded to a divisor of the KV heads)")
    return p.parse_args()


def code_sha1(text):
    """sha1 of a CUDA / C++ source's code: comments (// to the end of a line,
    /* ... */ blocks), trailing blanks and empty lines removed, so that an edit
    of the comments alone leaves it unchanged."""
    import hashlib
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return hashlib.sha1("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def _traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from a recorded ncu
    capture (profiles/traffic.json), or None when there is no record or the
    kernel's code has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel, {}).get(workload)
    if not rec:
        return None
    src = os.path.join(ROOT, "mass_adaptive_sparse_gb300", "csrc", rec["source"])
    if not os.path.exists(src) or code_sha1(open(src).read()) != rec["code_sha1"]:
        return None
    return rec["bytes_per_launch"]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "sm_max_mhz": d.get("sm_max_mhz", 2070.0),
                "sustained_sm_mhz": d.get("clocks_under_load", {}).get("sm_mhz_median"),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "sustained_sm_mhz": None, "source": "fallback"}


def config_of(pc, dc, tau, world):
    """The workload keys of the JSON line (both arms)."""
    return {"workload": f"{pc.name}+{dc.name}", "prefill": f"B={pc.B} H={pc.H}/{pc.Hkv} L={pc.L} d={pc.d} "
            f"tiles {pc.block}x{pc.block}", "decode": f"B={dc.B} H={dc.H}/{dc.Hkv} N={dc.N} d={dc.d} "
            f"block {dc.block} splits {dc.num_splits}", "tau": tau, "grad_dtype": "fp32",
            "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"}


# ---------------------------------------------------------------------------
# Work accounting (tile granularity, as the paper counts executed slots).
# ---------------------------------------------------------------------------

def prefill_units(cfg):
    t = -(-cfg.L // cfg.block)
    legal = cfg.B * cfg.H * t * (t + 1) // 2
    return {"legal_tiles": legal, "tile_flops": 2.0 * cfg.block * cfg.block * cfg.d}


def fwd_flops(cfg, kept):
    u = prefill_units(cfg)
    return u["tile_flops"] * (u["legal_tiles"] + kept)          # QK on every legal tile, PV on kept


def bwd_flops(cfg, kept):
    u = prefill_units(cfg)
    return u["tile_flops"] * (u["legal_tiles"] + 4 * kept)      # QK recompute + dP, dV, dK, dQ on kept


def decode_bytes(cfg, kept_tiles, num_splits=None):
    """Bytes a decode step reads or writes: K of every tile, V of kept tiles,
    q and o, and each split's (m, l, u) record written and read back."""
    splits = cfg.num_splits if num_splits is None else num_splits
    tile = cfg.block * cfg.d * 2
    n_tiles = cfg.B * cfg.Hkv * -(-cfg.N // cfg.block)
    k_bytes = n_tiles * tile
    v_bytes = kept_tiles * tile
    other = cfg.B * cfg.H * cfg.d * 2 * 2 + splits * cfg.B * cfg.H * (cfg.d + 4) * 4 * 2
    return k_bytes + v_bytes + other


# ---------------------------------------------------------------------------
# Clocks during the timed region.
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"mala_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            if self.uuid and self.uuid not in f[1]:
                continue
            try:
                sm.append(float(f[2]))
                smax.append(float(f[3]))
            except ValueError:
                continue
            for n, val in zip(names, f[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        top = max(sm)
        loaded = [x for x in sm if x >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (the cpu_baseline leg and the reference arm).
# ---------------------------------------------------------------------------

def _oracle_unit(task):
    """Runs in a spawned worker with single-threaded BLAS; returns seconds."""
    import numpy as np  # noqa: F401
    import oracle as orc
    from mass_adaptive_sparse_gb300 import synthetic
    import dataclasses
    kind, name, seed, arg = task
    cfg = synthetic.CONFIGS[name]
    if kind == "prefill":
        # one head of the same recipe (the sample's unit of work is a tile)
        cfg = dataclasses.replace(cfg, H=1, Hkv=1, amplitude=cfg.amplitude[:1])
        x = _WORKER_DATA.get((name, seed))
        if x is None:
            x = synthetic.prefill_inputs(cfg, seed=seed)
            x = {n: x[n][0, :, 0].double().numpy() for n in ("q", "k", "v", "do")}
            _WORKER_DATA.clear()
            _WORKER_DATA[(name, seed)] = x
        t0 = time.perf_counter()
        scale = 1 / math.sqrt(cfg.d)
        i = arg
        f = orc.mala_forward(x["q"], x["k"], x["v"], scale, 1.0, cfg.block, cfg.block, query_blocks=[i])
        orc.mala_backward(x["q"], x["k"], x["v"], f.o, x["do"], f.lse, scale, 1.0, cfg.block, cfg.block,
                          tiles=lambda ii, jj: ii == i)
        return time.perf_counter() - t0, i + 1          # seconds, tiles (fwd) == tiles (bwd)
    # one (sequence, KV head) group of the same recipe
    grp = cfg.H // cfg.Hkv
    cfg = dataclasses.replace(cfg, B=1, H=grp, Hkv=1)
    x = _WORKER_DATA.get((name, seed + arg))
    if x is None:
        y = synthetic.decode_inputs(cfg, seed=seed + arg)
        x = {n: y[n][0].double().numpy() for n in ("q", "k", "v")}
        _WORKER_DATA.clear()
        _WORKER_DATA[(name, seed + arg)] = x
    t0 = time.perf_counter()
    orc.mala_decode(x["q"], x["k"][:, 0], x["v"][:, 0], 1 / math.sqrt(cfg.d), 1.0, cfg.block, cfg.num_splits)
    return time.perf_counter() - t0, 1


_WORKER_DATA = {}


def _worker_init():
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"


def oracle_sample(workload, pool, cores, rank_seed=0, rounds=1):
    """Times the oracle on a bounded sample and extrapolates to one full step.
    Sample: forward + the matching backward dQ column for `rounds * cores`
    query blocks of head 0 of the prefill workload (spread over the
    sequence), and up to `rounds * cores` (sequence, KV head) groups of the
    decode workload."""
    from mass_adaptive_sparse_gb300 import synthetic
    pname, dname = WORKLOADS[workload]
    pc, dc = synthetic.CONFIGS[pname], synthetic.CONFIGS[dname]
    tr = pc.L // pc.block
    nblk = min(tr, max(2, cores * rounds))
    blocks = sorted({int(round((tr - 1) * (s + 1) / nblk)) for s in range(nblk)})
    groups = list(range(max(1, min(cores * rounds, dc.B * dc.Hkv))))
    tasks = [("prefill", pname, pc.seed + rank_seed, i) for i in blocks]
    tasks += [("decode", dname, dc.seed + rank_seed, g) for g in groups]
    t0 = time.perf_counter()
    res = pool.map(_oracle_unit, tasks)
    wall = time.perf_counter() - t0
    pre = res[:len(blocks)]
    dec = res[len(blocks):]
    pre_cpu = sum(r[0] for r in pre)
    pre_tiles = sum(r[1] for r in pre)
    dec_cpu = sum(r[0] for r in dec)
    full_tiles = prefill_units(pc)["legal_tiles"]
    full_groups = dc.B * dc.Hkv
    # per-unit CPU seconds x full units, spread over `cores` workers
    step_s = (pre_cpu / pre_tiles * full_tiles + dec_cpu / len(dec) * full_groups) / cores
    shown = blocks if len(blocks) <= 16 else f"{len(blocks)} evenly spaced from {blocks[0]} to {blocks[-1]}"
    sample = (f"fp64 oracle: forward + backward dQ column of query blocks {shown} (head 0, "
              f"{pre_tiles} tiles each way) of {pname} and decode of {len(dec)} (sequence, KV head) "
              f"groups of {dname}; extrapolated by tiles ({full_tiles}) and groups ({full_groups})")
    return step_s * 1e3, wall, sample


def run_reference(args):
    from mass_adaptive_sparse_gb300.replicas import rank_env
    rank, _, _ = rank_env()
    if rank != 0:
        return
    cores = min(16, os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_worker_init) as pool:
        vals = []
        for s in range(args.warmup + args.steps):
            v, _, sample = oracle_sample(args.workload, pool, cores)
            if s >= args.warmup:
                vals.append(v)
    value = statistics.mean(vals)
    from mass_adaptive_sparse_gb300 import synthetic
    pname, dname = WORKLOADS[args.workload]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "ms", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(synthetic.CONFIGS[pname], synthetic.CONFIGS[dname], args.tau, args.gpus),
            "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm.
# ---------------------------------------------------------------------------

def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
        return
    from mass_adaptive_sparse_gb300.replicas import Ranks, rank_env, replica_seed
    rank, world, local = rank_env()
    pool = None
    cores = min(16, os.cpu_count() or 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool = mp.get_context("spawn").Pool(cores, initializer=_worker_init)   # before any GPU work

    import torch
    from mass_adaptive_sparse_gb300 import api, synthetic

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pname, dname = WORKLOADS[args.workload]
    pc, dc = synthetic.CONFIGS[pname], synthetic.CONFIGS[dname]
    tau = args.tau

    # inputs (seeded per rank: each rank runs its own replica of the workload)
    xp = synthetic.prefill_inputs(pc, seed=replica_seed(pc.seed, rank))
    xd = synthetic.decode_inputs(dc, seed=replica_seed(dc.seed, rank))
    host_in = {n: xp[n].pin_memory() for n in ("q", "k", "v", "do")}
    host_in.update({"qd": xd["q"].pin_memory(), "kc": xd["k"].pin_memory(), "vc": xd["v"].pin_memory()})
    d = {n: t.to(dev) for n, t in host_in.items()}
    B, L, H, D = d["q"].shape
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    for n, like in (("dq", "q"), ("dk", "k"), ("dv", "v")):
        d[n] = torch.empty(d[like].shape, dtype=torch.float32, device=dev)
    d["ws_b"] = torch.empty(max(256, api.mala_bwd_workspace_size(d["q"], d["k"], torch.float32)),
                            dtype=torch.uint8, device=dev)
    d["od"] = torch.empty_like(d["qd"])
    d["lsed"] = torch.empty((dc.B, dc.H), dtype=torch.float32, device=dev)
    d["ws_d"] = torch.empty(max(256, api.mala_decode_workspace_size(dc.B, dc.H, dc.d, dc.num_splits)),
                            dtype=torch.uint8, device=dev)
    tr = -(-L // pc.block)
    cf = torch.zeros((B, H, tr), dtype=torch.int32, device=dev)
    cb = torch.zeros((B, H, tr), dtype=torch.int32, device=dev)
    cd = torch.zeros((dc.B, dc.Hkv, dc.num_splits), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def fwd(t):
        api.mala_fwd(d["q"], d["k"], d["v"], d["o"], d["lse"], block=pc.block, tau=t, retained_counts=cf)

    def bwd(t):
        api.mala_bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], d["dq"], d["dk"], d["dv"], d["ws_b"],
                     block=pc.block, tau=t, retained_counts=cb)

    def dec(t):
        api.mala_decode(d["qd"], d["kc"], d["vc"], d["od"], d["lsed"], d["ws_d"], block=dc.block,
                        num_splits=dc.num_splits, tau=t, retained_counts=cd)

    ranks = Ranks(dist, dev, torch.cuda.synchronize)
    barrier = ranks.barrier
    max_over_ranks = ranks.max

    def timed(t, steps):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for s in range(steps):
            ev[s][0].record(stream)
            fwd(t)
            ev[s][1].record(stream)
            bwd(t)
            ev[s][2].record(stream)
            dec(t)
            ev[s][3].record(stream)
        barrier()
        ph = {"fwd": [], "bwd": [], "decode": [], "step": []}
        for e in ev:
            ph["fwd"].append(e[0].elapsed_time(e[1]))
            ph["bwd"].append(e[1].elapsed_time(e[2]))
            ph["decode"].append(e[2].elapsed_time(e[3]))
            ph["step"].append(e[0].elapsed_time(e[3]))
        return {k: statistics.mean(v) for k, v in ph.items()}

    # --- tau = 1 (the measured configuration) ---
    for _ in range(args.warmup):
        fwd(tau); bwd(tau); dec(tau)
    barrier()
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    n0 = api.mala_launch_count()
    t_main = timed(tau, args.steps)
    launches = api.mala_launch_count() - n0
    clocks = sampler.stop()
    kept_f = int(cf.sum().item())
    kept_b = int(cb.sum().item())
    kept_d = int(cd.sum().item())
    step_ms = max_over_ranks(t_main["step"])

    # --- tau = 0: dense through the same kernels ---
    t_dense = None
    if not args.no_dense:
        for _ in range(min(args.warmup, 2)):
            fwd(0.0); bwd(0.0); dec(0.0)
        barrier()
        t_dense = timed(0.0, args.steps)

    # --- end to end through the public API with host buffers ---
    # The prefill runs in head chunks (heads are independent; one KV head per
    # chunk by default), so that later chunks' inputs arrive while earlier ones
    # compute and earlier chunks' gradients leave while later backwards run:
    # only the first chunk's inputs and the last chunk's gradients are exposed.
    # Four streams: copies in (in the order they are needed), compute, the
    # decode (as soon as its cache is in, alongside the prefill), copies out.
    e2e = None
    if not args.no_e2e:
        nchunk = math.gcd(max(1, args.e2e_chunks), pc.Hkv)
        hk_per = pc.Hkv // nchunk
        hq_per = hk_per * (pc.H // pc.Hkv)
        chunks = []
        for c in range(nchunk):
            hq = slice(c * hq_per, (c + 1) * hq_per)
            hkv = slice(c * hk_per, (c + 1) * hk_per)
            hin = {n: host_in[n][:, :, hq if n in ("q", "do") else hkv].contiguous().pin_memory()
                   for n in ("q", "k", "v", "do")}
            dev_c = {n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in hin.items()}
            dev_c["o"] = torch.empty_like(dev_c["q"])
            dev_c["lse"] = torch.empty((B, hq_per, L), dtype=torch.float32, device=dev)
            for n, like in (("dq", "q"), ("dk", "k"), ("dv", "v")):
                dev_c[n] = torch.empty(dev_c[like].shape, dtype=torch.float32, device=dev)
            dev_c["ws"] = torch.empty(max(256, api.mala_bwd_workspace_size(dev_c["q"], dev_c["k"], torch.float32)),
                                      dtype=torch.uint8, device=dev)
            hout = {n: torch.empty(dev_c[n].shape, dtype=dev_c[n].dtype, pin_memory=True)
                    for n in ("o", "lse", "dq", "dk", "dv")}
            chunks.append((hin, dev_c, hout))
        dec_out = {n: torch.empty(d[n].shape, dtype=d[n].dtype, pin_memory=True) for n in ("od", "lsed")}
        h2d = sum(t.numel() * t.element_size() for c in chunks for t in c[0].values()) + \
            sum(host_in[n].numel() * host_in[n].element_size() for n in ("qd", "kc", "vc"))
        d2h = sum(t.numel() * t.element_size() for c in chunks for t in c[2].values()) + \
            sum(t.numel() * t.element_size() for t in dec_out.values())

        def fwd_c(x):
            api.mala_fwd(x["q"], x["k"], x["v"], x["o"], x["lse"], block=pc.block, tau=tau)

        def bwd_c(x):
            api.mala_bwd(x["q"], x["k"], x["v"], x["o"], x["do"], x["lse"], x["dq"], x["dk"], x["dv"], x["ws"],
                         block=pc.block, tau=tau)

        s_in, s_cmp, s_dec, s_out = (torch.cuda.Stream(dev) for _ in range(4))

        def ev(st_, timing=False):
            e_ = torch.cuda.Event(enable_timing=timing)
            e_.record(st_)
            return e_

        def e2e_step(stamps=None):
            start = ev(stream, stamps is not None)
            for st_ in (s_in, s_cmp, s_dec, s_out):
                st_.wait_event(start)
            with torch.cuda.stream(s_in):
                in_qkv, in_do = [], []
                for hin, dev_c, _ in chunks:
                    for n in ("q", "k", "v"):
                        dev_c[n].copy_(hin[n], non_blocking=True)
                    in_qkv.append(ev(s_in))
                for hin, dev_c, _ in chunks:
                    dev_c["do"].copy_(hin["do"], non_blocking=True)
                    in_do.append(ev(s_in))
                for n in ("qd", "kc", "vc"):
                    d[n].copy_(host_in[n], non_blocking=True)
                in_cache = ev(s_in)
            with torch.cuda.stream(s_cmp):
                done_f, done_b = [], []
                for i, (_, dev_c, _) in enumerate(chunks):
                    s_cmp.wait_event(in_qkv[i])
                    fwd_c(dev_c)
                    done_f.append(ev(s_cmp))
                for i, (_, dev_c, _) in enumerate(chunks):
                    s_cmp.wait_event(in_do[i])
                    bwd_c(dev_c)
                    done_b.append(ev(s_cmp))
            with torch.cuda.stream(s_dec):
                s_dec.wait_event(in_cache)
                dec(tau)
                done_d = ev(s_dec)
            with torch.cuda.stream(s_out):
                for i, (_, dev_c, hout) in enumerate(chunks):
                    s_out.wait_event(done_f[i])
                    for n in ("o", "lse"):
                        hout[n].copy_(dev_c[n], non_blocking=True)
                for i, (_, dev_c, hout) in enumerate(chunks):
                    s_out.wait_event(done_b[i])
                    for n in ("dq", "dk", "dv"):
                        hout[n].copy_(dev_c[n], non_blocking=True)
                s_out.wait_event(done_d)
                for n in ("od", "lsed"):
                    dec_out[n].copy_(d[n], non_blocking=True)
            ends = [ev(st_, stamps is not None) for st_ in (s_in, s_cmp, s_dec, s_out)]
            for e_ in ends:
                stream.wait_event(e_)
            if stamps is not None:
                stamps.extend([start] + ends)

        e2e_step()
        barrier()
        n_e2e = max(1, min(args.steps, 10))
        es = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
        es[0].record(stream)
        for i in range(n_e2e):
            e2e_step()
            es[i + 1].record(stream)
        barrier()
        per_step = [es[i].elapsed_time(es[i + 1]) for i in range(n_e2e)]
        e2e_ms = max_over_ranks(statistics.mean(per_step))
        # diagnostics, outside the timed region: when each stream finished its
        # part of one more step, and the plain pinned-copy bandwidth of this machine
        stamps = []
        e2e_step(stamps)
        torch.cuda.synchronize()
        stream_ms = {n: stamps[0].elapsed_time(e_) for n, e_ in zip(("copies_in", "compute", "decode", "copies_out"),
                                                                     stamps[1:])}
        probe = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
        probe_d = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
        bw = {}
        for name, dst, src in (("h2d_gbs", probe_d, probe), ("d2h_gbs", probe, probe_d)):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            dst.copy_(src, non_blocking=True)
            c0.record(stream)
            for _ in range(3):
                dst.copy_(src, non_blocking=True)
            c1.record(stream)
            torch.cuda.synchronize()
            bw[name] = 3 * (1 << 30) / (c0.elapsed_time(c1) * 1e-3) / 1e9
        del probe, probe_d
        e2e = {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e, "step_ms": per_step,
               "pipeline": f"prefill in {nchunk} head chunks; copies in, compute, decode and copies out on "
                           "four streams",
               "stream_end_ms": stream_ms, "pinned_copy": bw}
        del chunks

    if not ranks.reports:
        if dist is not None:
            dist.destroy_process_group()
        return

    peaks = _peaks()
    ff, fb = fwd_flops(pc, kept_f), bwd_flops(pc, kept_b)
    db = decode_bytes(dc, kept_d)
    phases = {
        "fwd": {"ms": t_main["fwd"], "tflops": ff / t_main["fwd"] / 1e9, "algorithmic_flops": ff,
                "kept_tiles": kept_f, "legal_tiles": prefill_units(pc)["legal_tiles"]},
        "bwd": {"ms": t_main["bwd"], "tflops": fb / t_main["bwd"] / 1e9, "algorithmic_flops": fb,
                "kept_tiles": kept_b, "legal_tiles": prefill_units(pc)["legal_tiles"]},
        "decode": {"us_per_token": t_main["decode"] * 1e3, "gbs": db / t_main["decode"] / 1e6,
                   "algorithmic_bytes": db, "kept_tiles": kept_d,
                   "tiles": dc.B * dc.Hkv * -(-dc.N // dc.block)},
    }
    for ph in ("fwd", "bwd"):
        legal = phases[ph]["legal_tiles"]
        # Eq. 11: a kept B_q x B_k tile gives B_k post-score slots to each of its B_q rows
        phases[ph]["slots_per_query"] = phases[ph]["kept_tiles"] * pc.block * pc.block / (pc.B * pc.H * L)
        phases[ph]["kept_fraction"] = phases[ph]["kept_tiles"] / legal
    if t_dense is not None:
        pd = prefill_units(pc)["legal_tiles"]
        phases["dense"] = {
            "fwd_ms": t_dense["fwd"], "bwd_ms": t_dense["bwd"], "decode_us": t_dense["decode"] * 1e3,
            "fwd_tflops": fwd_flops(pc, pd) / t_dense["fwd"] / 1e9,
            "bwd_tflops": bwd_flops(pc, pd) / t_dense["bwd"] / 1e9,
            "speedup_fwd": t_dense["fwd"] / t_main["fwd"], "speedup_bwd": t_dense["bwd"] / t_main["bwd"],
            "speedup_decode": t_dense["decode"] / t_main["decode"], "step_ms": t_dense["step"]}

    # roofline of every phase; the dominant one (longest) is the headline
    roofs = {
        "fwd": {"kernel": "fwd_tc_kernel", "bound": "tensor", "achieved": phases["fwd"]["tflops"],
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"},
        "bwd": {"kernel": "bwd_tc_kernel", "bound": "tensor", "achieved": phases["bwd"]["tflops"],
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s"},
        "decode": {"kernel": "decode_mma_kernel", "bound": "hbm", "achieved": phases["decode"]["gbs"],
                   "peak": peaks["hbm_gbs"], "unit": "GB/s"},
    }
    for ph, rf in roofs.items():
        rf["frac"] = rf["achieved"] / rf["peak"]
        rf["traffic"] = _traffic(rf["kernel"], pname if ph != "decode" else dname)
        if rf["unit"] == "TFLOP/s":
            # the burst peak beside the sustained one (taken under the power cap,
            # at the median SM clock given here)
            rf["peak_burst"] = peaks["bf16_tflops"]
            rf["frac_burst"] = rf["achieved"] / peaks["bf16_tflops"]
            rf["peak_source"] = (f"measured sustained bf16 (cuBLAS, seconds-long loop, median SM clock "
                                 f"{peaks['sustained_sm_mhz']} MHz); frac_burst against the measured burst "
                                 f"({peaks['source']})")
        else:
            rf["peak_source"] = f"measured HBM copy ({peaks['source']})"
    step_phase_ms = {"fwd": t_main["fwd"], "bwd": t_main["bwd"], "decode": t_main["decode"]}
    dom = max(step_phase_ms, key=step_phase_ms.get)
    roofline = dict(roofs[dom])
    decode_roof = roofs["decode"]

    # --- the metric's second length: 32K prefill, fwd + bwd at tau and at 0 ---
    # (its tensors fit in L2, so L2 is flushed before every timed launch)
    secondary = None
    if args.workload == "128k" and not args.no_32k:
        c32 = synthetic.CONFIGS["prefill_32k"]
        x32 = synthetic.prefill_inputs(c32, seed=replica_seed(c32.seed, rank))
        e = {n: x32[n].to(dev) for n in ("q", "k", "v", "do")}
        del x32
        B3, L3, H3, _ = e["q"].shape
        e["o"] = torch.empty_like(e["q"])
        e["lse"] = torch.empty((B3, H3, L3), dtype=torch.float32, device=dev)
        for n, like in (("dq", "q"), ("dk", "k"), ("dv", "v")):
            e[n] = torch.empty(e[like].shape, dtype=torch.float32, device=dev)
        e["ws"] = torch.empty(max(256, api.mala_bwd_workspace_size(e["q"], e["k"], torch.float32)),
                              dtype=torch.uint8, device=dev)
        tr3 = -(-L3 // c32.block)
        cf3 = torch.zeros((B3, H3, tr3), dtype=torch.int32, device=dev)
        cb3 = torch.zeros((B3, H3, tr3), dtype=torch.int32, device=dev)
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

        def f32k(t):
            api.mala_fwd(e["q"], e["k"], e["v"], e["o"], e["lse"], block=c32.block, tau=t, retained_counts=cf3)

        def b32k(t):
            api.mala_bwd(e["q"], e["k"], e["v"], e["o"], e["do"], e["lse"], e["dq"], e["dk"], e["dv"], e["ws"],
                         block=c32.block, tau=t, retained_counts=cb3)

        def time32(t):
            for _ in range(max(3, args.warmup)):
                f32k(t); b32k(t)
            barrier()
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
            for s_ in range(args.steps):
                flush.zero_()
                ev[s_][0].record(stream); f32k(t); ev[s_][1].record(stream)
                flush.zero_()
                ev[s_][2].record(stream); b32k(t); ev[s_][3].record(stream)
            barrier()
            return (max_over_ranks(statistics.mean(x[0].elapsed_time(x[1]) for x in ev)),
                    max_over_ranks(statistics.mean(x[2].elapsed_time(x[3]) for x in ev)))

        f1, b1 = time32(tau)
        kf3, kb3 = int(cf3.sum().item()), int(cb3.sum().item())
        f0, b0 = time32(0.0)
        u3 = prefill_units(c32)
        secondary = {"prefill_32k": {
            "shape": f"B={B3} H={H3}/{e['k'].shape[2]} L={L3} d={c32.d} tiles {c32.block}x{c32.block}",
            "l2": "flushed before every timed launch",
            "fwd": {"ms": f1, "tflops": fwd_flops(c32, kf3) / f1 / 1e9, "kept_fraction": kf3 / u3["legal_tiles"]},
            "bwd": {"ms": b1, "tflops": bwd_flops(c32, kb3) / b1 / 1e9, "kept_fraction": kb3 / u3["legal_tiles"]},
            "dense": {"fwd_ms": f0, "bwd_ms": b0, "speedup_fwd": f0 / f1, "speedup_bwd": b0 / b1}}}
        del e, flush

    # --- the decode workload with each query head deciding alone (same kernels) ---
    if not args.no_32k:
        T_d = -(-dc.N // dc.block)
        cdh = torch.zeros((dc.B, dc.H, dc.num_splits), dtype=torch.int32, device=dev)
        mdh = torch.zeros((dc.B, dc.H, T_d), dtype=torch.uint8, device=dev)

        def dech(t):
            api.mala_decode_per_head(d["qd"], d["kc"], d["vc"], d["od"], d["lsed"], d["ws_d"], block=dc.block,
                                     num_splits=dc.num_splits, tau=t, retained_counts=cdh, tile_mask=mdh)

        for _ in range(max(3, args.warmup)):
            dech(tau)
        barrier()
        evh = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        evh[0].record(stream)
        for s_ in range(args.steps):
            dech(tau)
            evh[s_ + 1].record(stream)
        barrier()
        us_h = max_over_ranks(statistics.mean(evh[i].elapsed_time(evh[i + 1]) for i in range(args.steps))) * 1e3
        grp = dc.H // dc.Hkv
        v_tiles = int(mdh.view(dc.B, dc.Hkv, grp, T_d).amax(dim=2).sum().item())   # V read when any head keeps
        db_h = decode_bytes(dc, v_tiles)
        secondary = secondary or {}
        secondary["decode_per_head"] = {
            "what": "decode_128k with each query head deciding alone (mala_decode_per_head)",
            "us_per_token": us_h, "gbs": db_h / (us_h * 1e-3) / 1e6,
            "kept_fraction_heads": int(cdh.sum().item()) / (dc.B * dc.H * T_d),
            "v_tiles_read": v_tiles, "tiles": dc.B * dc.Hkv * T_d}

    # --- the decode skip path: split counts, and sharper queries over the same cache ---
    # The 128K decode workload keeps every tile (each split's own normaliser is
    # small), so V is read for every tile; the peaked queries (amplitude 12 on
    # the same 4 planted rows) let a split that has met its targets skip the
    # older tiles' V.
    if not args.no_32k:
        cpk = synthetic.CONFIGS["decode_128k_peaked"]
        q_peak = synthetic.decode_query(cpk, host_in["kc"], seed=replica_seed(cpk.seed, rank)).to(dev)
        T_d = -(-dc.N // dc.block)
        n_tiles = dc.B * dc.Hkv * T_d
        sweep = []
        for qname, qq in (("decode_128k", d["qd"]), ("decode_128k_peaked", q_peak)):
            for ns in (2, 4, 16):
                ws_s = torch.empty(max(256, api.mala_decode_workspace_size(dc.B, dc.H, dc.d, ns)), dtype=torch.uint8,
                                   device=dev)
                cnt = torch.zeros((dc.B, dc.Hkv, ns), dtype=torch.int32, device=dev)
                res = {}
                for t in (tau, 0.0):
                    def decs(t=t):
                        api.mala_decode(qq, d["kc"], d["vc"], d["od"], d["lsed"], ws_s, block=dc.block,
                                        num_splits=ns, tau=t, retained_counts=cnt)
                    for _ in range(max(3, args.warmup)):
                        decs()
                    barrier()
                    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
                    evs[0].record(stream)
                    for s_ in range(args.steps):
                        decs()
                        evs[s_ + 1].record(stream)
                    barrier()
                    us = max_over_ranks(statistics.mean(evs[i].elapsed_time(evs[i + 1])
                                                        for i in range(args.steps))) * 1e3
                    res[t] = (us, int(cnt.sum().item()))
                us1, kept1 = res[tau]
                us0, _ = res[0.0]
                byt = decode_bytes(dc, kept1, ns)
                sweep.append({"queries": qname, "num_splits": ns, "us_tau": us1, "us_tau0": us0,
                              "us_saved": us0 - us1, "speedup": us0 / us1, "v_tiles_read": kept1,
                              "k_tiles_read": n_tiles, "bytes_read": byt, "gbs": byt / (us1 * 1e-3) / 1e6})
        skipped_any = {qn: any(r["v_tiles_read"] < r["k_tiles_read"] for r in sweep if r["queries"] == qn)
                       for qn in ("decode_128k", "decode_128k_peaked")}
        secondary = secondary or {}
        secondary["decode_splits"] = {
            "what": "decode at tau and at 0 for 2, 4 and 16 splits; V bytes are read only for kept tiles",
            "queries": {"decode_128k": "the 128K decode workload's queries (amplitude 6)",
                        "decode_128k_peaked": "amplitude 12 on the same 4 planted cache rows, same cache"},
            "note": "; ".join(f"{qn}: " + ("some V tiles skipped" if sk else "no tile skipped at any split count")
                              for qn, sk in skipped_any.items()),
            "runs": sweep}
        del q_peak

    cpu = None
    if pool is not None:
        # a short calibration round, then a sample of about --sample-seconds
        _, wall1, _ = oracle_sample(args.workload, pool, cores)
        rounds = max(1, int(round(args.sample_seconds / max(wall1, 1e-3))))
        val, wall, sample = oracle_sample(args.workload, pool, cores, rounds=rounds)
        cpu = {"value": val, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample,
               "sample_wall_s": wall}
        pool.close()

    line = {
        "metric": METRIC, "value": step_ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(pc, dc, tau, world),
        "clocks": clocks, "e2e": e2e, "gpu_launches": launches, "roofline": roofline,
        "roofline_by_phase": roofs, "phases": phases, "secondary": secondary, "peaks": peaks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
