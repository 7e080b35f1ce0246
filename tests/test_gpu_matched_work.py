"""GPU parity of the matched-work study's kernels (§3 Table 1, App. C.2)
against the oracle, through the C ABI, and the study's own invariants.

* mala_region_mass: each (query block, key tile) region's reference mass,
  against the oracle's tile_reference_mass given the same (oracle) lse.
* mala_fwd_forced: attention over a given tile set, against the oracle's
  restricted_attention; a block that keeps no tile gives o = 0, lse = -inf.
* the study on a small workload: equal work for every policy, and the
  per-instance control never omits more than MALA on any decision (both run
  the same number of tiles; the control takes the heaviest ones).
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import api, matched_work as mw, synthetic
from tests import parity

pytestmark = pytest.mark.gpu


def _inputs(L, H, Hkv, seed, lk=None):
    n = max(L, lk or L)
    cfg = synthetic.PrefillConfig("mw", 1, H, Hkv, n, 128, 128, torch.bfloat16, 3, (4.0,), 3.0, 0.01)
    x = synthetic.prefill_inputs(cfg, seed=seed)
    q, k, v = x["q"][:, :L].contiguous(), x["k"][:, :lk or L].contiguous(), x["v"][:, :lk or L].contiguous()
    return q, k, v


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("L,lk,causal", [(300, None, True), (640, None, True), (200, 333, False)])
def test_region_mass_matches_oracle(block, L, lk, causal):
    H, Hkv = 4, 2
    q, k, v = _inputs(L, H, Hkv, 71, lk)
    scale = 1 / math.sqrt(128)
    q64, k64, v64 = (parity.to64(t) for t in (q, k, v))
    lse = np.zeros((1, H, L))
    ref = []
    for h in range(H):
        hk = h // (H // Hkv)
        _, lse[0, h] = orc.dense_attention(q64[0, :, h], k64[0, :, hk], v64[0, :, hk], scale, causal=causal)
        ref.append(orc.tile_reference_mass(q64[0, :, h], k64[0, :, hk], scale, block, block, causal=causal))
    ref = np.stack(ref)[None]
    mass = torch.full(ref.shape, float("nan"), dtype=torch.float32, device="cuda")
    api.mala_region_mass(q.cuda(), k.cuda(), torch.from_numpy(lse).float().cuda(), mass, causal=causal, block=block)
    torch.cuda.synchronize()
    got = mass.cpu().double().numpy()
    np.testing.assert_allclose(got, ref, rtol=2e-4, atol=1e-6)
    legal = orc.legal_tiles(L, lk or L, block, block, causal)
    assert (got[..., ~legal] == 0).all()


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_forced_forward_matches_oracle(block, out_dtype):
    L, H, Hkv = 300, 4, 2
    q, k, v = _inputs(L, H, Hkv, 73)
    scale = 1 / math.sqrt(128)
    tr = -(-L // block)
    legal = orc.legal_tiles(L, L, block, block)
    rng = np.random.default_rng(74)
    keep = (rng.random((1, H, tr, tr)) < 0.5) & legal
    keep[0, :, :, 0] |= legal[:, 0]                 # every block keeps its oldest tile ...
    keep[0, 1, 1, :] = False                        # ... but one, which keeps nothing
    o = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    lse = torch.empty((1, H, L), dtype=torch.float32, device="cuda")
    counts = torch.zeros((1, H, tr), dtype=torch.int32, device="cuda")
    api.mala_fwd_forced(q.cuda(), k.cuda(), v.cuda(), o, lse, torch.from_numpy(keep.astype(np.uint8)).cuda(),
                        block=block, retained_counts=counts)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    np.testing.assert_array_equal(counts.cpu().numpy(), keep.sum(-1))
    q64, k64, v64 = (parity.to64(t) for t in (q, k, v))
    go, glse = parity.to64(o), parity.to64(lse)
    for h in range(H):
        hk = h // (H // Hkv)
        rows = np.array([r for r in range(L) if keep[0, h, r // block].any()])
        ro, rl = orc.restricted_attention(q64[0, :, h], k64[0, :, hk], v64[0, :, hk], scale, keep[0, h],
                                          block, block, rows=rows)
        if out_dtype == torch.float32:
            assert np.abs(go[0, rows, h] - ro).max() <= parity.FP32_MAX_ABS
        else:
            parity.check_close("o", go[0, rows, h], ro, out_dtype)
        assert np.abs(glse[0, h, rows] - rl).max() <= 1e-4
    empty = slice(block, min(L, 2 * block))
    assert (go[0, empty, 1] == 0).all() and np.isneginf(glse[0, 1, empty]).all()


def test_study_small_invariants():
    """Two inputs of a 2048-token cut of the study's workload at tau = 1."""
    res = mw.study("study_8k", n_inputs=2, tau=1.0, L=2048)
    tiles = {p: res[p]["tiles"] for p in mw.POLICIES}
    assert len(set(tiles.values())) == 1, tiles
    assert len({round(res[p]["mean_slots"], 9) for p in mw.POLICIES}) == 1
    for p in mw.POLICIES:
        om = res[p]["per_decision_omitted"]
        assert ((om > -1e-6) & (om < 1 + 1e-6)).all()
    # MALA's own decisions obey the forward bound (App. B Eq. 6): at most tau / (1 + tau) per row
    assert (res["mala"]["per_decision_omitted"] <= 0.5 + 1e-6).all()
    assert (res["instance"]["per_decision_omitted"] <= res["mala"]["per_decision_omitted"] + 1e-5).all()
