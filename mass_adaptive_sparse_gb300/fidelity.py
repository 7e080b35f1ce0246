"""Operator fidelity across context lengths, on synthetic inputs.

The measurement of the MALA paper's §3 "Operator Fidelity Across Context
Lengths" (Figure 2; protocol in App. C.3).  For prefixes of growing length of
the same sequences, MALA at tau and the same kernels at tau = 0 (screening
disabled) run forward and backward on identical inputs; the output gradient
is a deterministic Rademacher probe, as in App. C.3.  Reported per prefix
length:

* realised work: mean post-score key slots per query, forward and backward
  (a kept B_q x B_k tile gives B_k slots to each of its B_q rows; §2.3);
* omitted reference mass 1 - exp(lse - lse_ref) per query (App. C.2),
  averaged over each (input, head) state's queries;
* relative L2 error of each head's whole O and dQ (query heads) and dK, dV
  (KV heads): |x - x_ref| / |x_ref|, App. C.3's head-level aggregation.

The states are then pooled (mean and P95), as the paper does.  Outputs are taken
in fp32 (the tensor-core forward's fp32-output variant) so that storage
rounding does not hide the screening error; the backward runs on the bf16
output, as in training.

    python -m mass_adaptive_sparse_gb300.fidelity --workload study_8k --lengths 1024,2048,4096,8192,16384,32768
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import api, synthetic


def rel_heads(x: torch.Tensor, ref: torch.Tensor) -> torch.Tensor:
    """Relative L2 (Frobenius) error per head: [B, L, H, D] -> [B, H]."""
    num = torch.linalg.vector_norm((x - ref).double(), dim=(1, 3))
    den = torch.linalg.vector_norm(ref.double(), dim=(1, 3))
    return num / den


def slots_per_query(kept_tiles: torch.Tensor, L: int, block: int) -> torch.Tensor:
    """Mean post-score key slots per query of each (input, head) state from
    per-block kept-tile counts [B, H, T] (forward: per query block, whose
    last may be ragged; backward: per key block, every kept tile counted with
    the rows of its query block, taken as full)."""
    return kept_tiles.double().sum(-1) * block * block / L


def measure(x: dict, tau: float, block: int) -> dict:
    """One prefix of one input: per-(input, head) statistics [B, H]."""
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    L = q.shape[1]
    res = {}
    runs = {}
    for name, t in (("mala", tau), ("ref", 0.0)):
        o32, lse, fi = api.forward(q, k, v, t, block=block, out_dtype=torch.float32, counts=True)
        o16, _, _ = api.forward(q, k, v, t, block=block)
        dq, dk, dv, bi = api.backward(q, k, v, o16, do, lse, t, block=block, counts=True)
        runs[name] = dict(o=o32, lse=lse, dq=dq, dk=dk, dv=dv, fc=fi["counts"], bc=bi["counts"])
    m, r = runs["mala"], runs["ref"]
    last = L - (-(-L // block) - 1) * block
    fwd_rows = torch.full((m["fc"].shape[-1],), float(block), device=q.device, dtype=torch.float64)
    fwd_rows[-1] = last
    res["fwd_slots"] = (m["fc"].double() * block * fwd_rows).sum(-1) / L
    res["bwd_slots"] = slots_per_query(m["bc"], L, block)
    res["omitted"] = (1.0 - torch.exp(m["lse"].double() - r["lse"].double())).mean(-1)
    res["o_err"] = rel_heads(m["o"], r["o"])
    res["dq_err"] = rel_heads(m["dq"], r["dq"])
    res["dk_err"] = rel_heads(m["dk"], r["dk"])
    res["dv_err"] = rel_heads(m["dv"], r["dv"])
    return {n: t.flatten().cpu().numpy() for n, t in res.items()}


def pool(per_state: list) -> dict:
    """Mean and P95 over the (input, head) states of every statistic."""
    out = {}
    for n in per_state[0]:
        v = np.concatenate([s[n] for s in per_state])
        out[n] = {"mean": float(v.mean()), "p95": float(np.percentile(v, 95))}
    return out


def study(workload: str = "study_8k", lengths=(1024, 2048, 4096, 8192), n_inputs: int = 2, tau: float = 1.0,
          device: str = "cuda") -> dict:
    cfg = synthetic.CONFIGS[workload]
    lmax = max(lengths)
    full = []
    for i in range(n_inputs):
        x = synthetic.prefill_inputs(cfg, L=lmax, seed=cfg.seed + 3000 + i, with_do=False)
        x["do"] = synthetic.rademacher(tuple(x["q"].shape), cfg.seed + 4000 + i, x["q"].dtype)
        full.append({n: x[n].to(device) for n in ("q", "k", "v", "do")})
    out = {}
    for L in lengths:
        states = [measure({n: t[:, :L].contiguous() for n, t in x.items()}, tau, cfg.block) for x in full]
        out[L] = pool(states)
    return out


def main():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--workload", default="study_8k", choices=sorted(synthetic.CONFIGS))
    p.add_argument("--lengths", default="1024,2048,4096,8192,16384,32768")
    p.add_argument("--inputs", type=int, default=2)
    p.add_argument("--tau", type=float, default=1.0)
    args = p.parse_args()
    lengths = [int(s) for s in args.lengths.split(",")]
    res = study(args.workload, lengths, args.inputs, args.tau)
    print(f"{'L':>7s} {'fwd slots':>10s} {'bwd slots':>10s} {'omitted %':>10s} {'p95':>8s} {'O err %':>9s} "
          f"{'p95':>8s} {'dQ err %':>9s} {'dK err %':>9s} {'dV err %':>9s}")
    for L in lengths:
        r = res[L]
        print(f"{L:7d} {r['fwd_slots']['mean']:10.1f} {r['bwd_slots']['mean']:10.1f} "
              f"{100 * r['omitted']['mean']:10.5f} {100 * r['omitted']['p95']:8.5f} "
              f"{100 * r['o_err']['mean']:9.5f} {100 * r['o_err']['p95']:8.5f} {100 * r['dq_err']['mean']:9.5f} "
              f"{100 * r['dk_err']['mean']:9.5f} {100 * r['dv_err']['mean']:9.5f}")
    print(json.dumps({"workload": args.workload, "tau": args.tau, "inputs": args.inputs,
                      "by_length": {str(L): res[L] for L in lengths}}))


if __name__ == "__main__":
    main()
