"""GPU parity of mala_fwd_varlen / mala_bwd_varlen (packed variable-length
batches) against the oracle, through the C ABI.

Each sequence is drawn by its workload's recipe at its own length and the
sequences are packed along one token axis.  Every sequence's slice is then
checked exactly as a one-sequence mala_fwd / mala_bwd call is (element by
element, borderline tiles replayed the same way).  Equal lengths must give
bit-for-bit what the fixed-length batched call gives, and a sequence whose
bounds break the contract raises the status bit and is left unwritten.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import api, synthetic
from tests import parity

pytestmark = pytest.mark.gpu


def _packed(cfg, lens, seed, heads=None, hkv=None):
    parts = {n: [] for n in ("q", "k", "v", "do")}
    for b, n in enumerate(lens):
        x = synthetic.prefill_inputs(cfg, L=n, seed=seed + b)
        for name in parts:
            t = x[name][0]
            if heads is not None:
                t = t[:, :heads] if name in ("q", "do") else t[:, :hkv]
            parts[name].append(t)
    out = {n: torch.cat(ts, 0).contiguous() for n, ts in parts.items()}
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return out, cu


def _run(cfg, lens, tau, seed, heads=None, hkv=None, grad_dtype=torch.float32, causal=True):
    x, cu = _packed(cfg, lens, seed, heads, hkv)
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    block = cfg.block
    d = q.shape[2]
    scale = 1.0 / math.sqrt(d)
    fp32 = q.dtype == torch.float32
    cu_d = torch.from_numpy(cu).cuda()
    lmax = max(lens)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse, info = api.forward_varlen(qd, kd, vd, cu_d, lmax, tau, causal=causal, block=block,
                                      counts=True, mask=True)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    q64, k64, v64, do64 = (parity.to64(t) for t in (q, k, v, do))
    ref = orc.mala_forward_varlen(q64, k64, v64, cu, scale, tau, block, block, causal)
    go, glse, gmask = parity.to64(o), parity.to64(lse), info["mask"].cpu().numpy()
    counts = info["counts"].cpu().numpy()
    H = q.shape[1]
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = slice(int(cu[b]), int(cu[b + 1]))
        t = -(-n // block)
        rb = {key: ref[key][b:b + 1, :, :t, :t] for key in ("retained", "legal", "margin")}
        rb["o"] = ref["o"][None, sl]
        rb["lse"] = ref["lse"][None, :, sl]
        parity.check_forward(go[None, sl], glse[None, :, sl], gmask[b:b + 1, :, :t, :t], rb, q64[None, sl],
                             k64[None, sl], v64[None, sl], scale, tau, block, o.dtype, fp32, heads=list(range(H)),
                             causal=causal)
        legal = np.tril(np.ones((t, t), bool)) if causal else np.ones((t, t), bool)
        np.testing.assert_array_equal(counts[b, :, :t], (gmask[b, :, :t, :t].astype(bool) & legal).sum(-1))
    # backward on the oracle's O (in the input dtype) and lse
    o_in = torch.from_numpy(ref["o"]).to(q.dtype).cuda()
    lse_in = torch.from_numpy(ref["lse"]).float().cuda()
    dq, dk, dv, binfo = api.backward_varlen(qd, kd, vd, o_in, dod, lse_in, cu_d, lmax, tau, causal=causal,
                                            block=block, grad_dtype=grad_dtype, counts=True, mask=True)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    refb = orc.mala_backward_varlen(q64, k64, v64, parity.to64(o_in), do64, parity.to64(lse_in), cu, scale, tau,
                                    block, block, causal)
    gq, gk, gv, gm = parity.to64(dq), parity.to64(dk), parity.to64(dv), binfo["mask"].cpu().numpy()
    bcounts = binfo["counts"].cpu().numpy()
    for b, n in enumerate(lens):
        if n == 0:
            continue
        sl = slice(int(cu[b]), int(cu[b + 1]))
        t = -(-n // block)
        rb = {key: refb[key][b:b + 1, :, :t, :t] for key in ("retained", "legal", "margin")}
        rb.update(dq=refb["dq"][None, sl], dk=refb["dk"][None, sl], dv=refb["dv"][None, sl])
        gb = {"dq": gq[None, sl], "dk": gk[None, sl], "dv": gv[None, sl], "mask": gm[b:b + 1, :, :t, :t]}

        def replay(sl=sl, b=b, t=t):
            r = orc.mala_backward_bshd(q64[None, sl], k64[None, sl], v64[None, sl], parity.to64(o_in)[None, sl],
                                       do64[None, sl], parity.to64(lse_in)[None, :, sl], scale, tau, block, block,
                                       causal, forced=gm[b:b + 1, :, :t, :t].astype(bool))
            return r

        parity.check_backward(gb, rb, block, fp32, causal=causal, grad_dtype=grad_dtype, replay=replay,
                              legal_tiles=int(refb["legal"].sum()))
        legal = np.tril(np.ones((t, t), bool)) if causal else np.ones((t, t), bool)
        np.testing.assert_array_equal(bcounts[b, :, :t], (gm[b, :, :t, :t].astype(bool) & legal).sum(-2))


@pytest.mark.parametrize("tau", [1.0, 4.0, 0.0])
def test_varlen_bf16_ragged(tau):
    """Tensor-core kernels: one row, a partial tile, exactly one tile, one row
    past a tile, and longer sequences, packed."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run(cfg, [1, 77, 128, 129, 300, 640], tau, 71, heads=2, hkv=2)


def test_varlen_bf16_gqa_and_bf16_grads():
    cfg = synthetic.PrefillConfig("vgqa", 1, 4, 2, 700, 128, 128, torch.bfloat16, 3, (4.0,), 3.0, 0.01)
    _run(cfg, [200, 700, 64], 1.0, 73, grad_dtype=torch.bfloat16)


@pytest.mark.parametrize("lens,heads,hkv,tau", [([4133, 2048, 129, 1, 700], 4, 4, 1.0),
                                                 ([3000, 1500, 257], 8, 2, 4.0)])
def test_varlen_medium_lengths(lens, heads, hkv, tau):
    """Packed sequences of thousands of tokens (many tiles each, ragged tails,
    a one-token sequence), MHA and grouped heads; every sequence compared in
    full with the oracle."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run(cfg, lens, tau, 81, heads=heads, hkv=hkv)


def test_varlen_noncausal():
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run(cfg, [130, 5, 260], 64.0, 75, heads=2, hkv=2, causal=False)


def test_varlen_fp32_d64():
    """The CUDA-core kernels (fp32, head_dim 64, 64-wide tiles)."""
    cfg = synthetic.CONFIGS["tiny_fp32"]
    _run(cfg, [1, 50, 64, 65, 200], 4.0, 77)


def test_varlen_equal_lengths_match_the_batched_call_exactly():
    """Three sequences of 384 rows packed give bit-for-bit the [3, 384, H, D] result."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    lens = [384, 384, 384]
    x, cu = _packed(cfg, lens, 79, heads=2, hkv=2)
    cu_d = torch.from_numpy(cu).cuda()
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o1, lse1, _ = api.forward_varlen(q, k, v, cu_d, 384, 1.0)
    shp = lambda t: t.view(3, 384, t.shape[1], t.shape[2])
    o2, lse2, _ = api.forward(shp(q), shp(k), shp(v), 1.0)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(3, 384, -1, 128), o2)
    assert torch.equal(lse1.view(-1, 3, 384).permute(1, 0, 2), lse2)
    g1 = api.backward_varlen(q, k, v, o1, do, lse1, cu_d, 384, 1.0)
    g2 = api.backward(shp(q), shp(k), shp(v), o2, shp(do), lse2, 1.0)
    torch.cuda.synchronize()
    for a, b in zip(g1[:3], g2[:3]):
        assert torch.equal(a.view(b.shape), b)


def test_varlen_rejects_bad_bounds_per_sequence():
    """A sequence longer than max_seqlen sets status bit 2 and is not computed;
    the others match the oracle."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    lens = [100, 300, 100]
    x, cu = _packed(cfg, lens, 81, heads=2, hkv=2)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
    api.mala_fwd_varlen(q, k, v, o, lse, torch.from_numpy(cu).cuda(), 200, tau=1.0)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 2
    assert api.mala_device_status() == 0
    go, glse = parity.to64(o), parity.to64(lse)
    assert np.isnan(go[100:400]).all() and np.isnan(glse[:, 100:400]).all()
    ref = orc.mala_forward_varlen(parity.to64(x["q"]), parity.to64(x["k"]), parity.to64(x["v"]), cu,
                                  1 / math.sqrt(128), 1.0, 128, 128, seqs=[0, 2])
    for sl in (slice(0, 100), slice(400, 500)):
        parity.check_close("o", go[sl], ref["o"][sl], q.dtype)
        assert np.abs(glse[:, sl] - ref["lse"][:, sl]).max() <= parity.LSE_ABS
