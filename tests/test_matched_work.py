"""Host logic of the matched-work study (§3 Table 1, App. C.2) against the
oracle's plain-loop statement of the same rules, on the CPU."""
import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import matched_work as mw


@pytest.mark.parametrize("lq,lk,block,causal", [(300, 300, 128, True), (256, 256, 64, True),
                                                (1, 1, 64, True), (300, 700, 128, False)])
def test_legal_tiles(lq, lk, block, causal):
    np.testing.assert_array_equal(mw.legal_tile_mask(lq, lk, block, causal),
                                  orc.legal_tiles(lq, lk, block, block, causal))


@pytest.mark.parametrize("scope", ["instance", "head_position", "position"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_allocation_matches_oracle(scope, seed):
    rng = np.random.default_rng(200 + seed)
    n_in, n_h, tr = rng.integers(1, 6), rng.integers(1, 9), rng.integers(1, 12)
    counts = rng.integers(1, np.arange(1, tr + 1) + 1, size=(n_in, n_h, tr))
    np.testing.assert_array_equal(mw.allocate(counts, scope), orc.matched_work_allocation(counts, scope))


@pytest.mark.parametrize("seed", [0, 1])
def test_top_mass_selection_matches_oracle(seed):
    rng = np.random.default_rng(210 + seed)
    tr = 9
    legal = orc.legal_tiles(tr * 16, tr * 16, 16, 16)
    mass = np.round(rng.random((3, tr, tr)), 1)             # coarse values: many equal masses
    n_keep = rng.integers(1, np.arange(1, tr + 1) + 1, size=(3, tr))
    got = mw.top_mass_keep(torch.from_numpy(mass), torch.from_numpy(n_keep), torch.from_numpy(legal)).numpy()
    for h in range(3):
        np.testing.assert_array_equal(got[h].astype(bool), orc.top_mass_keep(mass[h], n_keep[h], legal))


def test_decision_metrics_closed_form():
    """Half the reference mass omitted (lse lower by log 2) and the output off
    by 10% of its norm, on every row; the last block is ragged."""
    B, L, H, D, block = 1, 100, 2, 4, 64
    o_ref = torch.randn(B, L, H, D, dtype=torch.float64)
    lse_ref = torch.randn(B, H, L, dtype=torch.float64)
    dirs = torch.randn(B, L, H, D, dtype=torch.float64)
    dirs = dirs / torch.linalg.vector_norm(dirs, dim=-1, keepdim=True)
    o = o_ref + 0.1 * torch.linalg.vector_norm(o_ref, dim=-1, keepdim=True) * dirs
    om, er = mw.decision_metrics(o, lse_ref - np.log(2.0), o_ref, lse_ref, block)
    np.testing.assert_allclose(om.numpy(), 0.5, rtol=1e-12)
    np.testing.assert_allclose(er.numpy(), 0.1, rtol=1e-12)
