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

A flipped borderline forward tile changes the online state of its query block,
so every later decision and the block's output may differ; such blocks are
left out of the element-wise comparison and checked instead for validity: the
GPU output must equal softmax renormalised over the tiles the GPU kept, and
the first disagreement in traversal order must be borderline.  Backward tiles
are decided independently; a flipped borderline tile excludes the rows it
touches.
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


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def round_like(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32).to(dtype).to(torch.float64).numpy()


def is_borderline(margin) -> np.ndarray:
    m = np.asarray(margin, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return np.isfinite(m) & (np.abs(np.expm1(m)) <= orc.BORDERLINE_REL)


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


def fwd_block_agreement(gpu_mask, ref_retained, ref_legal, ref_margin):
    """Per query block: True if every legal decision agrees.  Asserts that any
    block that disagrees does so first (in the diagonal-to-oldest traversal)
    at a borderline tile.  Arrays are [Tr, Tc] for one (b, h)."""
    tr = ref_legal.shape[0]
    agree = np.ones(tr, dtype=bool)
    for i in range(tr):
        legal = ref_legal[i]
        if not legal.any():
            continue
        diff = (gpu_mask[i].astype(bool) != ref_retained[i]) & legal
        if diff.any():
            agree[i] = False
            first = np.nonzero(diff)[0].max()            # traversal runs from high j to low j
            assert is_borderline(ref_margin[i, first]), \
                f"query block {i}: tile {first} decided differently with margin {ref_margin[i, first]:.4g}"
    return agree


def check_forward(gpu_o, gpu_lse, gpu_mask, ref, q, k, v, scale, block, out_dtype, fp32,
                  heads, causal=True, blocks=None):
    """Compare forward results (numpy: o BSHD, lse [B,H,L], mask [B,H,Tr,Tc])
    with the oracle dict from mala_forward_bshd on the listed query ``heads``;
    ``blocks`` restricts the comparison to those query blocks.  Returns metrics."""
    B, L, H, D = gpu_o.shape
    grp = H // k.shape[2]
    tr = ref["legal"].shape[2]
    blocks = list(range(tr)) if blocks is None else list(blocks)
    rows_ok = np.zeros((B, H, L), dtype=bool)
    flipped = 0
    for b in range(B):
        for h in heads:
            agree = fwd_block_agreement(gpu_mask[b, h], ref["retained"][b, h], ref["legal"][b, h],
                                        ref["margin"][b, h])
            for i in blocks:
                r0, r1 = i * block, min(L, (i + 1) * block)
                if agree[i]:
                    rows_ok[b, h, r0:r1] = True
                    continue
                flipped += 1
                keep = gpu_mask[b, h].astype(bool) & ref["legal"][b, h]
                rows = np.arange(r0, r1)
                o_r, lse_r = orc.restricted_attention(q[b, :, h], k[b, :, h // grp], v[b, :, h // grp],
                                                      scale, keep, block, block, causal, rows)
                check_close("o (flipped block)", gpu_o[b, r0:r1, h], o_r, out_dtype, fp32=fp32)
                assert np.abs(gpu_lse[b, h, r0:r1] - lse_r).max() <= LSE_ABS
    n_blocks = B * len(heads) * len(blocks)
    assert flipped <= max(1, MAX_FLIPPED_FRACTION * n_blocks), f"{flipped} of {n_blocks} blocks flipped"
    sel = np.transpose(rows_ok, (0, 2, 1))               # [B, L, H]
    metrics = check_close("o", gpu_o[sel], ref["o"][sel], out_dtype, fp32=fp32)
    lse_err = np.abs(gpu_lse[rows_ok] - ref["lse"][rows_ok]).max()
    assert lse_err <= LSE_ABS, f"lse max abs err {lse_err:.3g}"
    legal = ref["legal"][:, heads][:, :, blocks]
    metrics.update(lse_max_abs=float(lse_err), flipped_blocks=flipped,
                   kept=int(ref["retained"][:, heads][:, :, blocks].sum()), legal=int(legal.sum()))
    return metrics


def check_backward(gpu, ref, block, fp32, dq_rows=None, dk_rows=None, causal=True, grad_dtype=torch.float32):
    """gpu / ref: dicts with dq, dk, dv (numpy, BSHD) and mask / retained,
    legal, margin ([B, H, Tr, Tc]).  ``dq_rows`` / ``dk_rows`` restrict the
    comparison to boolean masks [B, L, H] / [B, L, Hkv] (sampled checks).

    With grouped query heads, dK and dV sum over the group, so they grow with
    it while their error stays near fp16's unit roundoff relative to the
    largest value (the post-score products take fp16 operands): their max-abs
    bound is max(2e-2, 2^-11 max|ref|).  Without groups the bound is 2e-2."""
    B, Lq, H, D = gpu["dq"].shape
    Lk, Hkv = gpu["dk"].shape[1], gpu["dk"].shape[2]
    grp = H // Hkv
    okq = np.ones((B, Lq, H), bool) if dq_rows is None else dq_rows.copy()
    okk = np.ones((B, Lk, Hkv), bool) if dk_rows is None else dk_rows.copy()
    legal = ref["legal"]
    diff = (gpu["mask"].astype(bool) != ref["retained"]) & legal
    if diff.any():
        bs, hs, iis, jjs = np.nonzero(diff)
        for b, h, i, j in zip(bs, hs, iis, jjs):
            assert is_borderline(ref["margin"][b, h, i, j]), \
                f"bwd tile (b={b}, h={h}, i={i}, j={j}) decided differently, margin {ref['margin'][b, h, i, j]:.4g}"
            okq[b, i * block:(i + 1) * block, h] = False
            okk[b, j * block:(j + 1) * block, h // grp] = False
    assert diff.sum() <= max(1, MAX_FLIPPED_FRACTION * legal.sum())
    metrics = {"flipped_tiles": int(diff.sum())}
    for name, ok in (("dq", okq), ("dk", okk), ("dv", okk)):
        if grad_dtype == torch.bfloat16:
            metrics[name] = check_close_bf16_rounded(name, gpu[name][ok], ref[name][ok])
        else:
            floor = FP16_UNIT_ROUNDOFF if (grp > 1 and name != "dq") else 0.0
            metrics[name] = check_close(name, gpu[name][ok], ref[name][ok], torch.float32, ref_round=False,
                                        fp32=fp32, abs_floor_rel=floor)
    return metrics
