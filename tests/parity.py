"""Helpers that compare the CUDA library with the fp64 oracle.

Tolerances (written here once and used by every parity test):
  fp32 workloads : output max |err| <= 1e-4; gradients max |err| <= 1e-4 * max(1, |ref|max)
  bf16 workloads : O, dQ, dK, dV max |err| <= 2e-2 and mean relative error
                   sum|gpu - ref| / sum|ref| <= 1e-3, where ref is the oracle
                   rounded to the output dtype (round-to-nearest-even) when the
                   output is bf16;  lse max |err| <= 1e-3.
  tile masks     : identical, except that a tile whose oracle contribution
                   ratio lies within 1e-3 (relative) of tau / L_q may be decided
                   either way.

A borderline forward tile decided the other way changes the online state of
its query block, so later decisions and the block's output may change with
it.  Such a block is replayed: the oracle runs it again, following the GPU's
decision at each tile that is borderline on the replay's own state and
deciding every other tile itself.  Every GPU decision must then equal the
replay's, bit for bit, and the block's outputs are compared with the replay's
element by element.  Decode rows are replayed the same way; backward tiles
are decided independently, and a backward replay follows the GPU at its
borderline tiles only.  No row is left out of the comparison.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as orc

BF16_MAX_ABS = 2e-2
BF16_MEAN_REL = 1e-3
FP32_MAX_ABS = 1e-4
LSE_ABS = 1e-3
ZERO_REF_MEAN = 1e-6      # below this mean |ref| the mean relative error is undefined
MAX_FLIPPED_FRACTION = 0.01

# How often the checks met a borderline disagreement and replayed (reported at
# the end of the run by tests/conftest.py): units compared, units replayed,
# borderline tiles the replay took the other way from the oracle's own test.
REPLAY_STATS = {"fwd_blocks": 0, "fwd_replayed": 0, "decode_rows": 0, "decode_replayed": 0,
                "bwd_tiles": 0, "bwd_replayed_tiles": 0, "overridden_tiles": 0}


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def round_like(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32).to(dtype).to(torch.float64).numpy()


def is_borderline(margin) -> np.ndarray:
    return orc.is_borderline(margin)


FP16_UNIT_ROUNDOFF = 2.0 ** -11


def check_close(name, got, ref, out_dtype, ref_round=True, fp32=False, abs_floor_rel=0.0):
    """Assert the tolerance of the output dtype; returns the metrics.
    ``abs_floor_rel`` > 0 raises the bf16 max-abs bound to
    max(BF16_MAX_ABS, abs_floor_rel * max|ref|)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    if fp32:
        lim = FP32_MAX_ABS * max(1.0, float(np.abs(ref).max())) if name.startswith("d") else FP32_MAX_ABS
        assert err.max() <= lim, f"{name}: max abs err {err.max():.3g} > {lim:.3g}"
        return {"max_abs": float(err.max())}
    rref = round_like(ref, out_dtype) if (ref_round and out_dtype == torch.bfloat16) else ref
    mean_rel = float(np.abs(got - rref).sum() / max(np.abs(rref).sum(), 1e-30))
    lim = max(BF16_MAX_ABS, abs_floor_rel * float(np.abs(ref).max()))
    assert err.max() <= lim, f"{name}: max abs err {err.max():.3g} > {lim:.3g}"
    # A reference that is zero up to rounding (a one-token sequence's dQ: P = 1,
    # so dS = P (dP - D) = 0) has no scale to be relative to; max-abs decides.
    if np.abs(rref).mean() >= ZERO_REF_MEAN:
        assert mean_rel <= BF16_MEAN_REL, f"{name}: mean rel err {mean_rel:.3g} > {BF16_MEAN_REL}"
    return {"max_abs": float(err.max()), "mean_rel": mean_rel}


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def check_close_bf16_rounded(name, got, ref):
    """bf16 outputs whose magnitudes reach past the range where a bf16 step is
    below BF16_MAX_ABS (gradients through the bias coordinate reach ~40):
    compare with the oracle rounded to bf16; each element within
    max(BF16_MAX_ABS, one bf16 step of the rounded value), and the mean
    relative error within BF16_MEAN_REL."""
    got = np.asarray(got, np.float64)
    rref = round_like(np.asarray(ref, np.float64), torch.bfloat16)
    assert got.shape == rref.shape, (name, got.shape, rref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - rref)
    lim = np.maximum(BF16_MAX_ABS, bf16_ulp(rref))
    bad = err > lim
    assert not bad.any(), f"{name}: {int(bad.sum())} elements beyond max(2e-2, 1 bf16 step); worst {err.max():.3g}"
    mean_rel = float(err.sum() / max(np.abs(rref).sum(), 1e-30))
    assert mean_rel <= BF16_MEAN_REL, f"{name}: mean rel err {mean_rel:.3g} > {BF16_MEAN_REL}"
    return {"max_abs": float(err.max()), "mean_rel": mean_rel}


def check_forward(gpu_o, gpu_lse, gpu_mask, ref, q, k, v, scale, tau, block, out_dtype, fp32,
                  heads, causal=True, blocks=None):
    """Compare forward results (numpy: o BSHD, lse [B,H,L], mask [B,H,Tr,Tc])
    with the oracle dict from mala_forward_bshd on the listed query ``heads``;
    ``blocks`` restricts the comparison to those query blocks.

    A query block whose GPU decisions differ from the oracle's anywhere is
    replayed: the oracle runs the block again following the GPU's decision at
    each tile that is borderline on the replay's own (m, l), and deciding every
    other tile itself (``forced``).  Every GPU decision must then equal the
    replay's, and the block's O and lse are compared with the replay's.  So
    every decision and every row is checked; a borderline tile only chooses
    which of the two valid paths the expected values follow.  Returns metrics."""
    B, L, H, D = gpu_o.shape
    grp = H // k.shape[2]
    tr = ref["legal"].shape[2]
    blocks = list(range(tr)) if blocks is None else list(blocks)
    exp_o = np.array(ref["o"], dtype=np.float64, copy=True)
    exp_lse = np.array(ref["lse"], dtype=np.float64, copy=True)
    rows_ok = np.zeros((B, H, L), dtype=bool)
    replayed = overridden = 0
    for b in range(B):
        for h in heads:
            legal = ref["legal"][b, h]
            g = gpu_mask[b, h].astype(bool)
            diff = [i for i in blocks if ((g[i] != ref["retained"][b, h, i]) & legal[i]).any()]
            if diff:
                rep = orc.mala_forward(q[b, :, h], k[b, :, h // grp], v[b, :, h // grp], scale, tau, block, block,
                                       causal, query_blocks=diff, forced=g)
                for i in diff:
                    bad = (g[i] != rep.retained[i]) & rep.legal[i]
                    assert not bad.any(), (
                        f"(b={b}, h={h}) query block {i}: tiles {np.flatnonzero(bad).tolist()} decided differently "
                        f"from the oracle's replay of the GPU's borderline decisions; margins {rep.margin[i, bad]}")
                    r0, r1 = i * block, min(L, (i + 1) * block)
                    exp_o[b, r0:r1, h] = rep.o[r0:r1]
                    exp_lse[b, h, r0:r1] = rep.lse[r0:r1]
                replayed += len(diff)
                overridden += int(rep.overridden.sum())
            for i in blocks:
                rows_ok[b, h, i * block:min(L, (i + 1) * block)] = True
    n_blocks = B * len(heads) * len(blocks)
    REPLAY_STATS["fwd_blocks"] += n_blocks
    REPLAY_STATS["fwd_replayed"] += replayed
    REPLAY_STATS["overridden_tiles"] += overridden
    assert replayed <= max(1, MAX_FLIPPED_FRACTION * n_blocks), f"{replayed} of {n_blocks} blocks replayed"
    sel = np.transpose(rows_ok, (0, 2, 1))               # [B, L, H]
    metrics = check_close("o", gpu_o[sel], exp_o[sel], out_dtype, fp32=fp32)
    lse_err = np.abs(gpu_lse[rows_ok] - exp_lse[rows_ok]).max()
    assert lse_err <= LSE_ABS, f"lse max abs err {lse_err:.3g}"
    legal = ref["legal"][:, heads][:, :, blocks]
    metrics.update(lse_max_abs=float(lse_err), replayed_blocks=replayed, overridden_tiles=overridden,
                   kept=int(ref["retained"][:, heads][:, :, blocks].sum()), legal=int(legal.sum()))
    return metrics


def decode_expected(gpu_mask, ref_o, ref_lse, ref_retained, q, k, v, scale, tau, block, splits):
    """Expected results of one decision row of a decode (a KV head's group of
    query heads, or one query head): ref_o [G, d], ref_lse [G], masks [T];
    q [G, d] and the cache k, v [N, d] it attends to.  If the GPU's tile
    decisions differ from the oracle's, the row is replayed with the GPU's
    decisions at borderline tiles (``mala_decode(..., forced=...)``) and every
    decision must equal the replay's; the replay's O and lse are then the
    expected values.  Returns (o, lse, replayed)."""
    g = np.asarray(gpu_mask, bool)
    REPLAY_STATS["decode_rows"] += 1
    if not (g != np.asarray(ref_retained, bool)).any():
        return ref_o, ref_lse, False
    REPLAY_STATS["decode_replayed"] += 1
    rep = orc.mala_decode(q, k, v, scale, tau, block, splits, forced=g)
    bad = g != rep.retained
    assert not bad.any(), (f"decode tiles {np.flatnonzero(bad).tolist()} decided differently from the oracle's "
                           f"replay of the GPU's borderline decisions; margins {rep.margin[bad]}")
    REPLAY_STATS["overridden_tiles"] += int(rep.overridden.sum())
    return rep.o, rep.lse, True


def check_backward(gpu, ref, block, fp32, dq_rows=None, dk_rows=None, causal=True, grad_dtype=torch.float32,
                   replay=None, legal_tiles=None):
    """gpu / ref: dicts with dq, dk, dv (numpy, BSHD) and mask / retained,
    legal, margin ([B, H, Tr, Tc]).  ``dq_rows`` / ``dk_rows`` restrict the
    comparison to boolean masks [B, L, H] / [B, L, Hkv] (sampled checks).

    Backward decisions read only the fixed lse (Eq. 4), so they are
    independent.  If the GPU decided any tile differently, ``replay()`` must
    return the oracle's backward run again with ``forced`` = the GPU's mask
    (the same dict layout): it follows the GPU exactly at the tiles that are
    borderline for it.  Every GPU decision must then equal the replay's, and
    all gradients are compared with the replay's.

    With grouped query heads, dK and dV sum over the group, so they grow with
    it while their error stays near fp16's unit roundoff relative to the
    largest value (the post-score products take fp16 operands): their max-abs
    bound is max(2e-2, 2^-11 max|ref|).  Without groups the bound is 2e-2."""
    B, Lq, H, D = gpu["dq"].shape
    Lk, Hkv = gpu["dk"].shape[1], gpu["dk"].shape[2]
    grp = H // Hkv
    okq = np.ones((B, Lq, H), bool) if dq_rows is None else dq_rows.copy()
    okk = np.ones((B, Lk, Hkv), bool) if dk_rows is None else dk_rows.copy()
    gmask = gpu["mask"].astype(bool)
    diff = (gmask != ref["retained"]) & ref["legal"]
    metrics = {"replayed_tiles": int(diff.sum())}
    REPLAY_STATS["bwd_tiles"] += int(ref["legal"].sum())
    REPLAY_STATS["bwd_replayed_tiles"] += int(diff.sum())
    if diff.any():
        assert replay is not None, "the GPU decided backward tiles differently and no replay was given"
        # a sanity cap before the replay, over the whole call (``legal_tiles``:
        # the legal tiles of every sequence of a packed call checked in slices)
        n_legal = ref["legal"].sum() if legal_tiles is None else legal_tiles
        assert diff.sum() <= max(1, MAX_FLIPPED_FRACTION * n_legal)
        ref = replay()
        bad = (gmask != ref["retained"]) & ref["legal"]
        if bad.any():
            b, h, i, j = (int(x[0]) for x in np.nonzero(bad))
            raise AssertionError(f"{int(bad.sum())} bwd tiles decided differently from the oracle's replay, e.g. "
                                 f"(b={b}, h={h}, i={i}, j={j}) with margin {ref['margin'][b, h, i, j]:.4g}")
        metrics["overridden_tiles"] = int(ref["overridden"].sum())
        REPLAY_STATS["overridden_tiles"] += metrics["overridden_tiles"]
    for name, ok in (("dq", okq), ("dk", okk), ("dv", okk)):
        if grad_dtype == torch.bfloat16:
            metrics[name] = check_close_bf16_rounded(name, gpu[name][ok], ref[name][ok])
        else:
            floor = FP16_UNIT_ROUNDOFF if (grp > 1 and name != "dq") else 0.0
            metrics[name] = check_close(name, gpu[name][ok], ref[name][ok], torch.float32, ref_round=False,
                                        fp32=fp32, abs_floor_rel=floor)
    return metrics
