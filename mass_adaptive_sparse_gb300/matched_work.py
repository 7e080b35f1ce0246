"""Normalized-mass allocation at matched work, on synthetic inputs.

The study of the MALA paper's §3 "Normalized-Mass Allocation at Matched Work"
(Table 1; construction in App. C.2).  It asks how close MALA's online
decisions come to allocating post-score work by the final reference mass.
Every policy executes the same total number of post-score tiles; the policies
differ only in how the tiles are spread over decisions.  A decision is one
(input, head, query block), and its candidate regions are the block's legal
key tiles.

* MALA: the tiles the forward kernel kept, from its own online test.
* Per-instance control: MALA's count for each decision, filled with the
  decision's highest-mass tiles.
* Head/position control: one count per (head, query block), MALA's average
  over the inputs (the paper's layer-head-position control; one layer here).
* Position control: one count per query block, MALA's average over inputs
  and heads.

The averages become integers by a rule that looks only at indices: each of a
cell's n copies gets floor(average), and the e copies x with
(x - cell) mod n < e get one more, e being the cell's remaining units.  So
each cell, and the whole, executes exactly MALA's work.

Every policy's output is computed by the same forced-decision forward (CUDA
cores, fp32 probabilities and output), against the same kernel with every
legal tile kept as the reference.  Reported per decision, then pooled: the
omitted reference mass 1 - exp(lse - lse_ref) (App. C.2) and the relative
output error |o - o_ref| / |o_ref|, each averaged over the decision's rows.

    python -m mass_adaptive_sparse_gb300.matched_work --workload study_8k --inputs 4
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math

import numpy as np
import torch

from . import api, synthetic

SCOPES = ("position", "head_position", "instance")
POLICIES = ("position", "head_position", "instance", "mala")
LABELS = {"position": "Position / final reference mass",
          "head_position": "Head/Position / final reference mass",
          "instance": "Input/Head/Position / final reference mass",
          "mala": "Input/Head/Position / MALA online test"}


def legal_tile_mask(lq: int, lk: int, block: int, causal: bool = True) -> np.ndarray:
    """[Tr, Tc] bool: the tile holds at least one legal (query, key) pair."""
    tr, tc = -(-lq // block), -(-lk // block)
    i = np.arange(tr)[:, None]
    j = np.arange(tc)[None, :]
    if not causal:
        return np.ones((tr, tc), dtype=bool)
    return j * block <= np.minimum((i + 1) * block, lq) - 1


def allocate(counts: np.ndarray, scope: str) -> np.ndarray:
    """Tiles per decision for a control; counts [I, H, Tr] are MALA's."""
    counts = np.asarray(counts, dtype=np.int64)
    n_in, n_h, tr = counts.shape
    if scope == "instance":
        return counts.copy()
    if scope == "head_position":
        n = n_in
        totals = counts.sum(axis=0)                                   # [H, Tr]
        cell = (np.arange(n_h)[:, None] * tr + np.arange(tr)[None, :])[None]
        copy = np.arange(n_in)[:, None, None]
    elif scope == "position":
        n = n_in * n_h
        totals = counts.sum(axis=(0, 1))[None, :]                     # [1, Tr]
        cell = np.arange(tr)[None, None, :]
        copy = (np.arange(n_in)[:, None] * n_h + np.arange(n_h)[None, :])[:, :, None]
    else:
        raise ValueError(f"unknown scope {scope!r}")
    base, extra = totals // n, totals % n
    return base[None] + ((copy - cell) % n < extra[None]).astype(np.int64)


def top_mass_keep(mass: torch.Tensor, n_keep: torch.Tensor, legal: torch.Tensor) -> torch.Tensor:
    """Keep each decision's n_keep highest-mass legal tiles (equal masses:
    the newer tile first).  mass [..., Tr, Tc], n_keep [..., Tr], legal
    [Tr, Tc] -> uint8 [..., Tr, Tc]."""
    tc = mass.shape[-1]
    m = torch.where(legal, mass, torch.full_like(mass, -math.inf)).flip(-1)   # newest tile first
    order = torch.sort(m, dim=-1, descending=True, stable=True).indices
    rank = torch.empty_like(order)
    rank.scatter_(-1, order, torch.arange(tc, device=mass.device).expand_as(order).contiguous())
    keep = (rank < n_keep.unsqueeze(-1)).flip(-1) & legal
    return keep.to(torch.uint8)


@dataclasses.dataclass
class Decisions:
    """Everything one input contributes: MALA's decisions and the reference."""
    inputs: dict
    mala_keep: torch.Tensor     # uint8 [B, H, Tr, Tc]
    counts: torch.Tensor        # int32 [B, H, Tr]
    mass: torch.Tensor          # fp32 [B, H, Tr, Tc]
    o_ref: torch.Tensor
    lse_ref: torch.Tensor
    ms: dict                    # CUDA-event times of the reference forward and the region masses


def _forced(x, keep, block):
    q, k, v = x["q"], x["k"], x["v"]
    B, L, H, _ = q.shape
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    api.mala_fwd_forced(q, k, v, o, lse, keep, block=block)
    return o, lse


def decisions(x: dict, tau: float, block: int) -> Decisions:
    """MALA's online decisions on one input, the dense reference and the
    region masses (all through the library's kernels)."""
    q, k, v = x["q"], x["k"], x["v"]
    B, L, H, _ = q.shape
    tr = -(-L // block)
    dev = q.device
    o = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    counts = torch.zeros((B, H, tr), dtype=torch.int32, device=dev)
    mask = torch.zeros((B, H, tr, tr), dtype=torch.uint8, device=dev)
    api.mala_fwd(q, k, v, o, lse, block=block, tau=tau, retained_counts=counts, tile_mask=mask)
    legal = torch.from_numpy(legal_tile_mask(L, L, block)).to(dev)
    mask &= legal.to(torch.uint8)
    all_legal = legal.to(torch.uint8).expand(B, H, tr, tr).contiguous()
    mass = torch.empty((B, H, tr, tr), dtype=torch.float32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if q.is_cuda else None
    if ev:
        ev[0].record()
    o_ref, lse_ref = _forced(x, all_legal, block)
    if ev:
        ev[1].record()
    api.mala_region_mass(q, k, lse_ref, mass, block=block)
    ms = {}
    if ev:
        ev[2].record()
        torch.cuda.synchronize()
        ms = {"fwd_forced_dense": ev[0].elapsed_time(ev[1]), "region_mass": ev[1].elapsed_time(ev[2])}
    return Decisions(x, mask, counts, mass, o_ref, lse_ref, ms)


def decision_metrics(o, lse, o_ref, lse_ref, block):
    """Per decision [B, H, Tr]: the mean over the block's rows of the omitted
    reference mass and of the relative output error."""
    B, L, H, _ = o.shape
    tr = -(-L // block)
    omitted = (1.0 - torch.exp(lse.double() - lse_ref.double()))                 # [B, H, L]
    err = (torch.linalg.vector_norm((o - o_ref).double(), dim=-1) /
           torch.linalg.vector_norm(o_ref.double(), dim=-1)).permute(0, 2, 1)   # [B, H, L]
    pad = tr * block - L
    def per_block(x):
        x = torch.nn.functional.pad(x, (0, pad))
        rows = torch.full((tr,), float(block), dtype=torch.float64, device=x.device)
        rows[-1] = block - pad
        return x.view(B, H, tr, block).sum(-1) / rows
    return per_block(omitted), per_block(err)


def run(ds: list, block: int) -> dict:
    """The four policies over the inputs' decisions; returns one row per
    policy (and the kernels' times).  The sequences of a batch count as heads
    of one input."""
    dev = ds[0].counts.device
    B, H, tr = ds[0].counts.shape
    L = ds[0].inputs["q"].shape[1]
    legal = torch.from_numpy(legal_tile_mask(L, L, block)).to(dev)
    counts = np.stack([d.counts.cpu().numpy().reshape(B * H, tr) for d in ds])    # [I, B*H, Tr]
    rows_per_block = np.full(tr, block)
    rows_per_block[-1] = L - (tr - 1) * block
    out = {}
    for pol in POLICIES:
        n = counts if pol == "mala" else allocate(counts, pol)
        om, er = [], []
        for i, d in enumerate(ds):
            if pol == "mala":
                keep = d.mala_keep
            else:
                nk = torch.from_numpy(n[i].reshape(B, H, tr)).to(dev)
                keep = top_mass_keep(d.mass, nk, legal)
            o, lse = _forced(d.inputs, keep, block)
            a, b = decision_metrics(o, lse, d.o_ref, d.lse_ref, block)
            om.append(a.flatten())
            er.append(b.flatten())
            if pol != "mala" and not torch.equal(keep.sum(-1, dtype=torch.int64).cpu(),
                                                 torch.from_numpy(n[i].reshape(B, H, tr))):
                raise RuntimeError(f"{pol}: the selection does not run the allocated number of tiles")
        om, er = torch.cat(om).cpu().numpy(), torch.cat(er).cpu().numpy()
        slots = float((n * block * rows_per_block[None, None, :]).sum() / (len(ds) * B * H * L))
        out[pol] = {"policy": LABELS[pol], "tiles": int(n.sum()), "mean_slots": slots,
                    "omitted_mean_pct": 100 * float(om.mean()), "omitted_p95_pct": 100 * float(np.percentile(om, 95)),
                    "error_mean_pct": 100 * float(er.mean()), "error_p95_pct": 100 * float(np.percentile(er, 95)),
                    "per_decision_omitted": om}
    if ds[0].ms:
        legal_tiles = int(legal.sum()) * B * H
        d = ds[0].inputs["q"].shape[-1]
        fl = {"fwd_forced_dense": 4.0 * legal_tiles * block * block * d,      # Q K^T and P V per legal tile
              "region_mass": 2.0 * legal_tiles * block * block * d}          # Q K^T per legal tile
        med = {n: float(np.median([x.ms[n] for x in ds])) for n in fl}     # the first input pays the first launch
        out["kernels"] = {n: {"ms": med[n], "tflops": fl[n] / med[n] / 1e9} for n in fl}
    return out


def study(workload: str = "study_8k", n_inputs: int = 4, tau: float = 1.0, L: int | None = None,
          heads: int | None = None, device: str = "cuda") -> dict:
    """Generate `n_inputs` seeded inputs of a workload and run every policy."""
    cfg = synthetic.CONFIGS[workload]
    if heads is not None:
        cfg = dataclasses.replace(cfg, H=heads, Hkv=max(1, heads * cfg.Hkv // cfg.H))
    ds = []
    for i in range(n_inputs):
        x = synthetic.prefill_inputs(cfg, L=L, seed=cfg.seed + 1000 + i)
        x = {n: x[n].to(device) for n in ("q", "k", "v")}
        ds.append(decisions(x, tau, cfg.block))
    return run(ds, cfg.block)


def main():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--workload", default="study_8k", choices=sorted(synthetic.CONFIGS))
    p.add_argument("--inputs", type=int, default=4)
    p.add_argument("--tau", type=float, default=1.0)
    p.add_argument("--L", type=int, default=None)
    p.add_argument("--heads", type=int, default=None)
    args = p.parse_args()
    res = study(args.workload, args.inputs, args.tau, args.L, args.heads)
    print(f"{'allocation / selection':46s} {'tiles':>8s} {'slots/query':>11s} {'omitted % mean':>15s} "
          f"{'p95':>8s} {'error % mean':>13s} {'p95':>8s}")
    for pol in POLICIES:
        r = res[pol]
        print(f"{r['policy']:46s} {r['tiles']:8d} {r['mean_slots']:11.1f} {r['omitted_mean_pct']:15.5f} "
              f"{r['omitted_p95_pct']:8.5f} {r['error_mean_pct']:13.5f} {r['error_p95_pct']:8.5f}")
    for n, r in res.get("kernels", {}).items():
        print(f"kernel {n}: {r['ms']:.3f} ms, {r['tflops']:.1f} TFLOP/s (CUDA cores, fp32)")
    print(json.dumps({"workload": args.workload, "inputs": args.inputs, "tau": args.tau,
                      "rows": [{k: v for k, v in res[p].items() if k != "per_decision_omitted"} for p in POLICIES],
                      "kernels": res.get("kernels")}))


if __name__ == "__main__":
    main()
