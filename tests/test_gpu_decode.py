"""GPU parity of mala_decode (split-KV decode + exact merge) against the oracle."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import api, synthetic
from tests import parity

pytestmark = pytest.mark.gpu


def _check(cfg, N, B, tau, splits, block, seed, batches=None, dtype=None, d=None, lens=None, per_head=False,
           query_cfg=None):
    """Decode on the GPU and compare with the oracle; `lens` (one cache length
    per sequence, each in [1, N]) selects the variable-length entry point over
    caches padded to N, `per_head` the entry point whose query heads decide
    alone (masks and counts per query head), `query_cfg` another workload's
    query recipe over this workload's cache."""
    x = synthetic.decode_inputs(cfg, N=N, B=B, seed=seed)
    q, k, v = x["q"], x["k"], x["v"]
    if query_cfg is not None:
        q = synthetic.decode_query(query_cfg, k)
    if d is not None:
        q, k, v = q[..., :d].contiguous(), k[..., :d].contiguous(), v[..., :d].contiguous()
    if dtype is not None:
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    D = q.shape[-1]
    scale = 1 / math.sqrt(D)
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse, info = api.decode(q.cuda(), k.cuda(), v.cuda(), tau, block=block, num_splits=splits,
                              counts=True, mask=True, cache_lens=lens_t, per_head=per_head)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    batches = list(range(B)) if batches is None else batches
    q64, k64, v64 = (parity.to64(t) for t in (q, k, v))
    if per_head:
        ref = orc.mala_decode_per_head_bhd(q64, k64, v64, scale, tau, block, splits, batches=batches)
    elif lens is None:
        ref = orc.mala_decode_bhd(q64, k64, v64, scale, tau, block, splits, batches=batches)
    else:
        ref = orc.mala_decode_varlen_bhd(q64, k64, v64, lens, scale, tau, block, splits, batches=batches)
    go, glse, gmask = parity.to64(o), parity.to64(lse), info["mask"].cpu().numpy()
    Hq, Hkv = q.shape[1], k.shape[2]
    grp = Hq // Hkv
    # a decision row is a KV head's group of query heads, or one query head
    rows = [(h, slice(h, h + 1), h // grp) for h in range(Hq)] if per_head else \
        [(hk, slice(hk * grp, (hk + 1) * grp), hk) for hk in range(Hkv)]
    fp32 = q.dtype == torch.float32
    replayed = 0
    counts = info["counts"].cpu().numpy()
    exp_o, exp_lse = ref["o"].copy(), ref["lse"].copy()
    for b in batches:
        n_b = N if lens is None else lens[b]
        T = -(-n_b // block)
        per = -(-T // splits)
        for row, hs, hk in rows:
            for sp in range(splits):
                np.testing.assert_array_equal(counts[b, row, sp], gmask[b, row, sp * per:min(T, (sp + 1) * per)].sum())
            # every decision must equal the oracle's, or its replay of the GPU's borderline decisions
            exp_o[b, hs], exp_lse[b, hs], rep = parity.decode_expected(
                gmask[b, row, :T], ref["o"][b, hs], ref["lse"][b, hs], ref["retained"][b, row, :T], q64[b, hs],
                k64[b, :n_b, hk], v64[b, :n_b, hk], scale, tau, block, splits)
            replayed += rep
    assert replayed <= max(1, parity.MAX_FLIPPED_FRACTION * len(batches) * len(rows))
    m = parity.check_close("o", go[batches], exp_o[batches], q.dtype, fp32=fp32)
    assert np.abs(glse[batches] - exp_lse[batches]).max() <= parity.LSE_ABS
    return m, gmask


@pytest.mark.parametrize("splits", [1, 3, 16])
@pytest.mark.parametrize("tau", [0.0, 1.0, 16.0])
def test_decode_small_bf16(splits, tau):
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 1000, 2, tau, splits, 128, 11)


@pytest.mark.parametrize("block", [64, 128])
def test_decode_small_fp32_d64(block):
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 777, 2, 1.0, 5, block, 12, dtype=torch.float32, d=64)


@pytest.mark.parametrize("H,Hkv", [(16, 2), (8, 4), (4, 4)])
def test_decode_group_sizes(H, Hkv):
    """Query-head groups of 8, 2 and 1 (the tensor-core kernel takes up to 8)."""
    cfg = dataclasses.replace(synthetic.CONFIGS["decode_128k"], H=H, Hkv=Hkv)
    _check(cfg, 1500, 2, 1.0, 4, 128, 41)


def test_decode_single_partial_tile():
    """A cache shorter than one tile: one ragged tile, every other split empty."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 77, 2, 1.0, 16, 128, 53)


def test_decode_tau0_is_dense_for_any_split():
    cfg = synthetic.CONFIGS["decode_128k"]
    _, mask = _check(cfg, 2048, 1, 0.0, 7, 128, 13)
    assert mask.all()


def test_decode_128k_full_size_sampled():
    """Batch 8, 32 query heads over 8 KV heads, 131072-token cache, 16 splits;
    sequences 0 and 5 (tau = 1) and 3 and 7 (tau = 0) are compared with the oracle."""
    cfg = synthetic.CONFIGS["decode_128k"]
    for tau, seqs in ((1.0, [0, 5]), (0.0, [3, 7])):
        _check(cfg, cfg.N, cfg.B, tau, cfg.num_splits, cfg.block, cfg.seed, batches=seqs)


@pytest.mark.parametrize("splits", [2, 16])
def test_decode_128k_peaked_sampled(splits):
    """The sharper queries (amplitude 12 on the same planted rows) over the 128K
    decode cache, where a split that has met its targets skips older V tiles:
    sequences 1 and 6 at tau = 1 compared with the oracle; with 2 splits some
    tiles are skipped."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _, mask = _check(cfg, cfg.N, cfg.B, 1.0, splits, cfg.block, cfg.seed, batches=[1, 6],
                     query_cfg=synthetic.CONFIGS["decode_128k_peaked"])
    if splits == 2:
        assert not mask[[1, 6]].all()


@pytest.mark.parametrize("tau", [1.0, 0.0])
def test_decode_varlen_bf16(tau):
    """Per-sequence cache lengths over a cache padded to 1500 rows: one row,
    a partial tile, exactly one tile, one row past a tile, and the full cache."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 1500, 6, tau, 4, 128, 61, lens=[1, 77, 128, 129, 1000, 1500])


def test_decode_varlen_full_size():
    """Batch 8 over caches padded to 131072 rows, lengths from one row to the
    full cache (ragged tails, a split boundary, one token past a tile), 16
    splits; sequences 1, 4 and 7 compared with the oracle."""
    cfg = synthetic.CONFIGS["decode_128k"]
    lens = [131072, 100003, 65536, 4097, 1, 128, 129, 77777]
    _check(cfg, cfg.N, cfg.B, 1.0, cfg.num_splits, cfg.block, cfg.seed, batches=[1, 4, 7], lens=lens)


def test_decode_varlen_fp32_d64():
    """The CUDA-core split kernel (fp32, head_dim 64, 64-key tiles)."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 700, 4, 1.0, 5, 64, 67, dtype=torch.float32, d=64, lens=[700, 1, 333, 64])


def test_decode_varlen_rejects_bad_lengths_per_sequence():
    """A length of 0 or past the padded cache raises status bit 2 and gives NaN
    for that sequence only; the others match the oracle."""
    cfg = synthetic.CONFIGS["decode_128k"]
    N, B = 600, 4
    lens = [300, 0, 601, 600]
    x = synthetic.decode_inputs(cfg, N=N, B=B, seed=71)
    q, k, v = x["q"], x["k"], x["v"]
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse, _ = api.decode(q.cuda(), k.cuda(), v.cuda(), 1.0, block=128, num_splits=4, cache_lens=lens_t)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 2
    assert api.mala_device_status() == 0          # reading clears the word
    go, glse = parity.to64(o), parity.to64(lse)
    assert np.isnan(go[1]).all() and np.isnan(go[2]).all()
    assert np.isnan(glse[1]).all() and np.isnan(glse[2]).all()
    q64, k64, v64 = (parity.to64(t) for t in (q, k, v))
    ref = orc.mala_decode_varlen_bhd(q64, k64, v64, [300, 1, 1, 600], 1 / math.sqrt(128), 1.0, 128, 4,
                                     batches=[0, 3])
    for b in (0, 3):
        parity.check_close("o", go[b], ref["o"][b], q.dtype)
        assert np.abs(glse[b] - ref["lse"][b]).max() <= parity.LSE_ABS


@pytest.mark.parametrize("splits", [1, 3, 16])
@pytest.mark.parametrize("tau", [0.0, 1.0, 16.0])
def test_decode_per_head_small_bf16(splits, tau):
    """Each query head decides alone (tensor-core split kernel, group of 4)."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 1000, 2, tau, splits, 128, 11, per_head=True)


@pytest.mark.parametrize("H,Hkv", [(16, 2), (8, 4)])
def test_decode_per_head_group_sizes(H, Hkv):
    cfg = dataclasses.replace(synthetic.CONFIGS["decode_128k"], H=H, Hkv=Hkv)
    _check(cfg, 1500, 2, 1.0, 4, 128, 43, per_head=True)


def test_decode_per_head_fp32_d64():
    """The CUDA-core split kernel (fp32, head_dim 64, 64-key tiles)."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, 777, 2, 4.0, 5, 64, 47, dtype=torch.float32, d=64, per_head=True)


def test_decode_per_head_128k_full_size_sampled():
    """Batch 8, 32 query heads over 8 KV heads, 131072-token cache, 16 splits,
    each head deciding alone; sequences 1 and 6 compared with the oracle."""
    cfg = synthetic.CONFIGS["decode_128k"]
    _check(cfg, cfg.N, cfg.B, 1.0, cfg.num_splits, cfg.block, cfg.seed, batches=[1, 6], per_head=True)


@pytest.mark.parametrize("splits,kept", [(1, [0, 2, 5]), (2, [1, 2, 5]), (3, [0, 1, 2, 3, 5]),
                                         (6, [0, 1, 2, 3, 4, 5])])
def test_decode_split_state_closed_form(splits, kept):
    """Six 128-key tiles whose keys repeat one score per tile, tau = 3 over
    N = 768 keys: the closed form of the oracle pin on per-split state, tile
    for tile (every tile's mass is 128 times the one-key case and so is
    tau / N's denominator).  Each split starts from its own empty state, so two
    splits keep tile 1 and skip tile 0 where one pass does the opposite."""
    scores = [math.log(1.56), math.log(1.25), math.log(2.0), -50.0, -50.0, 0.0]
    B, G, N, D, blk = 1, 4, 768, 128, 128
    scale = 1 / math.sqrt(D)
    q = torch.zeros((B, G, D))
    q[..., 0] = 16.0
    k = torch.zeros((B, N, 1, D))
    for j, s in enumerate(scores):
        k[0, j * blk:(j + 1) * blk, 0, 0] = s / (16.0 * scale)
    v = torch.from_numpy(np.random.default_rng(61).standard_normal((B, N, 1, D)))
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    q64, k64, v64 = (parity.to64(t) for t in (q, k, v))
    ref = orc.mala_decode_bhd(q64, k64, v64, scale, 3.0, blk, splits)
    assert np.flatnonzero(ref["retained"][0, 0]).tolist() == kept
    o, lse, info = api.decode(q.cuda(), k.cuda(), v.cuda(), 3.0, block=blk, num_splits=splits,
                              counts=True, mask=True)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    assert np.flatnonzero(info["mask"].cpu().numpy()[0, 0]).tolist() == kept
    parity.check_close("o", parity.to64(o), ref["o"], q.dtype)
    assert np.abs(parity.to64(lse) - ref["lse"]).max() <= parity.LSE_ABS
