"""Run one MALA operation on a synthetic workload, for profilers.

    python -m mass_adaptive_sparse_gb300.profile_case --op bwd --workload prefill_8k --iters 2

Generates the workload's seeded inputs (optionally with fewer heads, a
shorter sequence or fewer sequences), then calls the operation ``--iters``
times on the current CUDA device and synchronises.  Every call goes through
the C ABI; nothing else is launched between calls.
"""
from __future__ import annotations

import argparse
import dataclasses

import torch

from . import api, synthetic


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--op", choices=["fwd", "bwd", "decode"], required=True)
    p.add_argument("--workload", default="prefill_8k", choices=sorted(synthetic.CONFIGS))
    p.add_argument("--heads", type=int, default=None, help="query heads (KV heads scale with them)")
    p.add_argument("--L", type=int, default=None, help="sequence / cache length")
    p.add_argument("--batch", type=int, default=None)
    p.add_argument("--tau", type=float, default=1.0)
    p.add_argument("--iters", type=int, default=2)
    args = p.parse_args()
    cfg = synthetic.CONFIGS[args.workload]
    dev = torch.device("cuda")
    if args.op == "decode":
        if args.heads is not None:
            cfg = dataclasses.replace(cfg, H=args.heads, Hkv=max(1, args.heads * cfg.Hkv // cfg.H))
        x = synthetic.decode_inputs(cfg, N=args.L, B=args.batch)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        B, Hq, D = q.shape
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        ws = torch.empty(api.mala_decode_workspace_size(B, Hq, D, cfg.num_splits), dtype=torch.uint8, device=dev)
        for _ in range(args.iters):
            api.mala_decode(q, k, v, o, lse, ws, block=cfg.block, num_splits=cfg.num_splits, tau=args.tau)
    else:
        if args.heads is not None:
            cfg = dataclasses.replace(cfg, H=args.heads, Hkv=max(1, args.heads * cfg.Hkv // cfg.H),
                                      amplitude=cfg.amplitude[:1] if len(cfg.amplitude) > 1 else cfg.amplitude)
        x = synthetic.prefill_inputs(cfg, L=args.L)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        B, L, H, D = q.shape
        o = torch.empty_like(q)
        lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        api.mala_fwd(q, k, v, o, lse, block=cfg.block, tau=args.tau)
        if args.op == "fwd":
            for _ in range(args.iters - 1):
                api.mala_fwd(q, k, v, o, lse, block=cfg.block, tau=args.tau)
        else:
            dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
            dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
            dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
            ws = torch.empty(api.mala_bwd_workspace_size(q, k, torch.float32), dtype=torch.uint8, device=dev)
            for _ in range(args.iters):
                api.mala_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, block=cfg.block, tau=args.tau)
    torch.cuda.synchronize()
    status = api.mala_device_status()
    print(f"{args.op} {args.workload} done, device status {status}, launches {api.mala_launch_count()}")
    if status != 0:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
