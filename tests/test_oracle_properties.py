"""Randomised pins of the oracle over shapes the fixed pins do not reach:
ragged lengths, several tile sizes, tolerances and seeds.  Each property is
one that the pages or the mathematics fix (cited beside it); none re-types
the oracle's own formulas.  CPU only; skipped where hypothesis is missing."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import synthetic
from tests.test_oracle_pins import _brute_force_forward

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings

SCALE = 1 / math.sqrt(32)


def _case(L, seed, recency):
    cfg = synthetic.PrefillConfig("prop", 1, 1, 1, L, 32, 16, torch.float32, 3, (4.0,), 3.0, recency)
    x = synthetic.prefill_inputs(cfg, L=L, seed=seed)
    return tuple(x[n][0, :, 0].double().numpy() for n in ("q", "k", "v", "do"))


shapes = dict(L=st.integers(1, 150), b=st.sampled_from([8, 16, 32]), tau=st.sampled_from([0.25, 1.0, 4.0]),
              seed=st.integers(0, 10_000), recency=st.sampled_from([0.0, 0.05, 0.2]))


@settings(max_examples=60, deadline=None, derandomize=True)
@given(**shapes)
def test_forward_is_the_ratio_rule_and_renormalised_softmax(L, b, tau, seed, recency):
    """Algorithm 1 equals the explicit ratio rule (Eq. 1-3) on any shape, and its
    output is softmax renormalised over the kept tiles (§2.2)."""
    q, k, v, _ = _case(L, seed, recency)
    r = orc.mala_forward(q, k, v, SCALE, tau, b, b)
    o, lse, keep = _brute_force_forward(q, k, v, SCALE, tau, b)
    np.testing.assert_array_equal(r.retained, keep)
    np.testing.assert_allclose(r.o, o, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(r.lse, lse, rtol=1e-11, atol=1e-11)
    # every block keeps its diagonal tile, the first it visits (l = 0 retains, §2.2)
    t = -(-L // b)
    assert r.retained[np.arange(t), np.arange(t)].all()


@settings(max_examples=60, deadline=None, derandomize=True)
@given(**shapes)
def test_forward_omitted_mass_within_eq6(L, b, tau, seed, recency):
    """App. B Eq. 6: every query omits at most tau / (1 + tau) of the dense mass."""
    q, k, v, _ = _case(L, seed, recency)
    r = orc.mala_forward(q, k, v, SCALE, tau, b, b)
    _, lse_d = orc.dense_attention(q, k, v, SCALE)
    eps = orc.omitted_mass(r.lse, lse_d)
    assert np.all(eps >= -1e-12) and np.all(eps <= tau / (1 + tau) + 1e-12)


@settings(max_examples=60, deadline=None, derandomize=True)
@given(**shapes)
def test_backward_support_nested_in_forward(L, b, tau, seed, recency):
    """§2.2: tested against the final normaliser, the backward keeps no tile the
    forward skipped (support nesting)."""
    q, k, v, do = _case(L, seed, recency)
    f = orc.mala_forward(q, k, v, SCALE, tau, b, b)
    g = orc.mala_backward(q, k, v, f.o, do, f.lse, SCALE, tau, b, b)
    assert not (g.retained & ~f.retained).any()


@settings(max_examples=60, deadline=None, derandomize=True)
@given(n=st.integers(1, 300), bk=st.sampled_from([8, 16, 32]), splits=st.integers(1, 9),
       tau=st.sampled_from([0.5, 1.0, 8.0]), seed=st.integers(0, 10_000))
def test_decode_is_renormalised_softmax_over_its_kept_tiles(n, bk, splits, tau, seed):
    """App. A.1 split-KV decode: whatever the splits decide, the merged output is
    softmax over the kept keys (the merge identity is exact), the newest tile of
    every non-empty split is kept, and the omitted mass stays within Eq. 6."""
    rng = np.random.default_rng(seed)
    g = 2
    qg = rng.standard_normal((g, 32)) * 2
    kc = rng.standard_normal((n, 32))
    vc = rng.standard_normal((n, 32))
    r = orc.mala_decode(qg, kc, vc, SCALE, tau, bk, splits)
    t = -(-n // bk)
    per = -(-t // splits)
    for sp in range(splits):
        top = min(t, (sp + 1) * per) - 1
        if top >= sp * per:
            assert r.retained[top]
    o_r, lse_r = orc.restricted_attention(qg, kc, vc, SCALE, r.retained[None, :], g, bk, causal=False)
    np.testing.assert_allclose(r.o, o_r, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(r.lse, lse_r, rtol=1e-11, atol=1e-11)
    _, lse_d = orc.dense_attention(qg, kc, vc, SCALE, causal=False)
    assert np.all(orc.omitted_mass(r.lse, lse_d) <= tau / (1 + tau) + 1e-12)
