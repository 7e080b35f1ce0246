"""Pins for the fp64 oracle: each check ties the oracle to something other than
itself -- the worked examples printed on the pages, closed forms, a library
routine for the dense special case, finite differences, the bounds the paper
proves, and a brute-force restatement of the skip rule in its ratio form.

Citations name the page and its section / equation:
  MALA = "MassAlloc Attention: Let Attention Allocate Its Own Compute";
  MERGE = "Why exact attention does not need a quadratic matrix".
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "merge_examples.txt")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _sdpa(q, k, v, scale, causal=True, mask=None):
    """torch's fp64 scaled_dot_product_attention on one head; also returns lse."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64)[None, None] for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=None if mask is None else torch.tensor(mask)[None, None],
        is_causal=causal and mask is None, scale=scale)
    s = scale * (tq @ tk.transpose(-1, -2))
    if mask is not None:
        s = s.masked_fill(~torch.tensor(mask)[None, None], float("-inf"))
    elif causal:
        n = q.shape[0]
        s = s.masked_fill(torch.ones(n, k.shape[0], dtype=torch.bool).triu(1), float("-inf"))
    return o[0, 0].numpy(), torch.logsumexp(s, -1)[0, 0].numpy()


def _sdpa_grads(q, k, v, do, scale, causal=True):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                         is_causal=causal, scale=scale)[0, 0]
    (o * torch.tensor(do)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


PIN_SCALE = 1 / math.sqrt(32)


def _peaked(L=256, seed=7):
    """One head of the planted-peak recipe at d = 32 with a strong recency
    bias (-0.1 (i - j)), so that small cases skip a good share of tiles."""
    cfg = synthetic.PrefillConfig("pin", 1, 1, 1, L, 32, 16, torch.float32, 3, (4.0,), 3.0, 0.1)
    x = synthetic.prefill_inputs(cfg, L=L, seed=seed)
    return (x["q"][0, :, 0].double().numpy(), x["k"][0, :, 0].double().numpy(),
            x["v"][0, :, 0].double().numpy(), x["do"][0, :, 0].double().numpy())


# ---------------------------------------------------------------------------
# MERGE, Example 1 and its variant (golden values printed on the page).
# ---------------------------------------------------------------------------

def _parse(tok):
    out = []
    for t in tok.split(","):
        out.append(math.log(2) if t == "log2" else math.log(4) if t == "log4" else float(t))
    return out


def test_merge_worked_examples():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 2
    for case, a_s, a_v, b_s, b_v, a_sum, b_sum, merged, weights in rows:
        sa = orc.block_summary(_parse(a_s), _parse(a_v))
        sb = orc.block_summary(_parse(b_s), _parse(b_v))
        for got, want in ((sa, _parse(a_sum)), (sb, _parse(b_sum))):
            assert got[0] == pytest.approx(want[0], abs=1e-15)
            assert got[1] == pytest.approx(want[1], abs=1e-15)
            assert got[2][0] == pytest.approx(want[2], abs=1e-15)
        m, l, u = orc.merge_summaries([sa, sb])
        assert u[0] / l == pytest.approx(float(merged), abs=1e-14), case
        # averaging local outputs is right in example 1 only by coincidence
        avg = 0.5 * (sa[2][0] / sa[1] + sb[2][0] / sb[1])
        assert (avg == pytest.approx(float(merged))) == (case == "example1")
        if weights != "-":
            s = np.array(_parse(a_s) + _parse(b_s))
            w = np.exp(s) / np.exp(s).sum()
            np.testing.assert_allclose(w, _parse(weights), atol=1e-15)
        # the merge is order independent and ignores empty blocks
        m2, l2, u2 = orc.merge_summaries([sb, (0.0, 0.0, np.zeros(1)), sa])
        assert u2[0] / l2 == pytest.approx(float(merged), abs=1e-14)


# ---------------------------------------------------------------------------
# Dense attention (the tau = 0 case) against closed forms and torch.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_dense_matches_library(causal):
    q, k, v = _rand((70, 16), 1), _rand((70, 16), 2), _rand((70, 16), 3)
    o, lse = orc.dense_attention(q, k, v, 0.3, causal)
    o_ref, lse_ref = _sdpa(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_dense_closed_forms():
    q, k, v = _rand((40, 8), 4), _rand((40, 8), 5), _rand((40, 8), 6)
    o, lse = orc.dense_attention(q, k, v, 0.5)
    # row 0 sees only key 0
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert lse[0] == pytest.approx(0.5 * q[0] @ k[0], abs=1e-14)
    # a zero query attends uniformly over its prefix
    o0, lse0 = orc.dense_attention(np.zeros_like(q), k, v, 0.5)
    np.testing.assert_allclose(o0, np.cumsum(v, 0) / np.arange(1, 41)[:, None], atol=1e-14)
    np.testing.assert_allclose(lse0, np.log(np.arange(1, 41)), atol=1e-14)


def test_dense_grads_match_library_and_finite_differences():
    q, k, v, do = (_rand((24, 8), s) for s in (7, 8, 9, 10))
    dq, dk, dv = orc.dense_attention_grads(q, k, v, do, 0.4)
    for got, want in zip((dq, dk, dv), _sdpa_grads(q, k, v, do, 0.4)):
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    # central differences of f = <o, dO>
    f = lambda qq, kk, vv: (orc.dense_attention(qq, kk, vv, 0.4)[0] * do).sum()
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0), (5, 3), (23, 7), (11, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if n == name else y for n, y in (("q", q), ("k", k), ("v", v))]
            args_m = [xm if n == name else y for n, y in (("q", q), ("k", k), ("v", v))]
            fd = (f(*args_p) - f(*args_m)) / (2 * eps)
            assert fd == pytest.approx(g[idx], rel=1e-6, abs=1e-9), (name, idx)


# ---------------------------------------------------------------------------
# MALA forward (MALA §2.2 Eq. 2-3, Algorithm 1, App. B).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L,bq", [(128, 32), (200, 64), (97, 16)])
def test_forward_tau0_is_dense(L, bq):
    q, k, v = _rand((L, 16), 11, 2.0), _rand((L, 16), 12), _rand((L, 16), 13)
    r = orc.mala_forward(q, k, v, 0.25, 0.0, bq, bq)
    o_ref, lse_ref = _sdpa(q, k, v, 0.25)
    np.testing.assert_allclose(r.o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r.lse, lse_ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(r.retained, r.legal)
    t = -(-L // bq)
    assert np.array_equal(r.legal, np.tril(np.ones((t, t), dtype=bool)))


def test_forward_huge_tau_keeps_only_diagonal_tiles():
    L, b = 128, 32
    q, k, v = _rand((L, 16), 14), _rand((L, 16), 15), _rand((L, 16), 16)
    r = orc.mala_forward(q, k, v, 0.25, 1e30, b, b)
    assert np.array_equal(r.retained, np.eye(L // b, dtype=bool))
    blk = np.arange(L) // b
    mask = (blk[:, None] == blk[None, :]) & (np.arange(L)[None, :] <= np.arange(L)[:, None])
    o_ref, lse_ref = _sdpa(q, k, v, 0.25, mask=mask)
    np.testing.assert_allclose(r.o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r.lse, lse_ref, rtol=1e-12, atol=1e-12)


def _brute_force_forward(q, k, v, scale, tau, b):
    """Eq. 2 in ratio form with the retained key set kept explicitly: before
    each tile, Z = sum over retained keys of exp(s) (Eq. 1), and the tile is
    skipped iff exp(max legal s) / Z < tau / L_q for every row (Z = 0 retains).
    Output = softmax over the retained keys."""
    L = q.shape[0]
    s_all = scale * q @ k.T
    t = -(-L // b)
    keep = np.zeros((t, t), dtype=bool)
    o = np.zeros_like(q)
    lse = np.zeros(L)
    for i in range(t):
        rows = range(i * b, min(L, (i + 1) * b))
        kept_keys = {r: [] for r in rows}
        for j in range(i, -1, -1):
            skip = True
            for r in rows:
                legal = [c for c in range(j * b, min(L, (j + 1) * b)) if c <= r]
                if not legal:
                    continue
                z = sum(math.exp(s_all[r, c]) for c in kept_keys[r])
                if z == 0 or math.exp(max(s_all[r, c] for c in legal)) / z >= tau / (r + 1):
                    skip = False
            if skip:
                continue
            keep[i, j] = True
            for r in rows:
                kept_keys[r] += [c for c in range(j * b, min(L, (j + 1) * b)) if c <= r]
        for r in rows:
            w = np.array([math.exp(s_all[r, c]) for c in kept_keys[r]])
            o[r] = (w[:, None] * v[kept_keys[r]]).sum(0) / w.sum()
            lse[r] = math.log(w.sum())
    return o, lse, keep


@pytest.mark.parametrize("tau,b,seed", [(1.0, 16, 3), (1.0, 8, 11), (2.0, 16, 5), (0.5, 8, 6)])
def test_forward_matches_brute_force_ratio_rule(tau, b, seed):
    q, k, v, _ = _peaked(L=128, seed=seed)
    r = orc.mala_forward(q, k, v, PIN_SCALE, tau, b, b)
    o, lse, keep = _brute_force_forward(q, k, v, PIN_SCALE, tau, b)
    assert np.array_equal(r.retained, keep)
    assert (~keep & np.tril(np.ones_like(keep))).any(), "case must skip something"
    np.testing.assert_allclose(r.o, o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r.lse, lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("tau,b", [(1.0, 16), (1.0, 64), (0.1, 32), (3.0, 16)])
def test_forward_bounds_of_appendix_b(tau, b):
    q, k, v, _ = _peaked(L=256, seed=11)
    scale = PIN_SCALE
    r = orc.mala_forward(q, k, v, scale, tau, b, b)
    # the output is ordinary softmax renormalised over the retained tiles (§2.2)
    o_r, lse_r = orc.restricted_attention(q, k, v, scale, r.retained, b, b)
    np.testing.assert_allclose(r.o, o_r, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r.lse, lse_r, rtol=1e-12, atol=1e-12)
    o_d, lse_d = orc.dense_attention(q, k, v, scale)
    L = q.shape[0]
    lq = np.arange(1, L + 1)
    s = scale * q @ k.T
    blk = np.arange(L) // b
    omitted = (~r.retained[blk[:, None], blk[None, :]]) & (np.arange(L)[None, :] <= np.arange(L)[:, None])
    assert omitted.any()
    # every omitted key: exp(s_k) / Z_R < tau / L_q  (App. B, Eq. 7 with Z_R >= Z_t)
    rr, cc = np.nonzero(omitted)
    assert np.all(s[rr, cc] - r.lse[rr] < math.log(tau) - np.log(lq[rr]))
    # omitted mass eps_q <= tau / (1 + tau)  (Eq. 6), measured as in App. C.2
    eps = orc.omitted_mass(r.lse, lse_d)
    assert np.all(eps >= -1e-12) and np.all(eps <= tau / (1 + tau))
    # ||p - p~||_1 = 2 eps  (Eq. 9)  and  ||o - o~|| <= 2 tau/(1+tau) V_max  (Eq. 10)
    p = np.exp(np.where(np.tril(np.ones((L, L), bool)), s, -np.inf) - lse_d[:, None])
    pt = np.where(omitted, 0.0, np.exp(np.where(np.tril(np.ones((L, L), bool)), s, -np.inf) - r.lse[:, None]))
    np.testing.assert_allclose(np.abs(p - pt).sum(1), 2 * eps, atol=1e-12)
    vmax = np.linalg.norm(v, axis=1).max()
    assert np.all(np.linalg.norm(o_d - r.o, axis=1) <= 2 * tau / (1 + tau) * vmax + 1e-12)


def test_uniform_scores_closed_form():
    """All scores equal (q = 0) and 1x1 tiles: when row r tests key k it has
    retained n keys, each key's ratio is 1/n, and the key is skipped iff
    1/n < tau/L_r with L_r = r + 1 (Eq. 2).  So row r keeps its newest
    n* = min(r + 1, floor((r + 1)/tau) + 1) keys; lse = log n*; o = their mean.
    Backward then skips every entry, since (r + 1)/n* < tau (Eq. 4)."""
    L, tau = 64, math.pi
    q = np.zeros((L, 4))
    k, v, do = _rand((L, 4), 51), _rand((L, 4), 52), _rand((L, 4), 53)
    r = orc.mala_forward(q, k, v, 1.0, tau, 1, 1)
    for row in range(L):
        n_star = min(row + 1, math.floor((row + 1) / tau) + 1)
        assert r.retained[row].sum() == n_star
        assert r.retained[row, row - n_star + 1: row + 1].all()
        assert r.lse[row] == pytest.approx(math.log(n_star), abs=1e-13)
        np.testing.assert_allclose(r.o[row], v[row - n_star + 1: row + 1].mean(0), atol=1e-13)
    g = orc.mala_backward(q, k, v, r.o, do, r.lse, 1.0, tau, 1, 1)
    assert not g.retained.any()


def test_decode_uniform_scores_closed_form():
    """Decode analogue with L = N: one split keeps the newest floor(N/tau) + 1
    keys; two splits each keep their own newest floor(N/tau) + 1."""
    n, tau = 50, math.pi
    kc, vc = _rand((n, 4), 54), _rand((n, 4), 55)
    r = orc.mala_decode(np.zeros((2, 4)), kc, vc, 1.0, tau, 1, 1)
    n_star = math.floor(n / tau) + 1
    assert r.retained.sum() == n_star and r.retained[n - n_star:].all()
    np.testing.assert_allclose(r.lse, math.log(n_star), atol=1e-13)
    np.testing.assert_allclose(r.o[0], vc[n - n_star:].mean(0), atol=1e-13)
    r2 = orc.mala_decode(np.zeros((2, 4)), kc, vc, 1.0, tau, 1, 2)
    assert r2.retained[:25].sum() == n_star and r2.retained[25 - n_star:25].all()
    assert r2.retained[25:].sum() == n_star and r2.retained[n - n_star:].all()
    keep = np.r_[np.arange(25 - n_star, 25), np.arange(n - n_star, n)]
    np.testing.assert_allclose(r2.o[1], vc[keep].mean(0), atol=1e-13)


def test_forward_first_tile_always_retained_and_rows_nonempty():
    q, k, v, _ = _peaked(L=200, seed=12)
    r = orc.mala_forward(q, k, v, PIN_SCALE, 1.0, 32, 32)
    assert np.all(np.diag(r.retained))
    assert np.all(np.isfinite(r.lse)) and np.all(np.isfinite(r.o))


# ---------------------------------------------------------------------------
# MALA backward (MALA §2.2 Eq. 4, Algorithm 2).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L,b", [(96, 32), (200, 64)])
def test_backward_tau0_is_dense_gradient(L, b):
    q, k, v, do = (_rand((L, 16), s) for s in (21, 22, 23, 24))
    f = orc.mala_forward(q, k, v, 0.25, 0.0, b, b)
    g = orc.mala_backward(q, k, v, f.o, do, f.lse, 0.25, 0.0, b, b)
    for got, want in zip((g.dq, g.dk, g.dv), _sdpa_grads(q, k, v, do, 0.25)):
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-11)


def test_backward_huge_tau_skips_everything():
    q, k, v, do = (_rand((64, 16), s) for s in (25, 26, 27, 28))
    f = orc.mala_forward(q, k, v, 0.25, 1e30, 16, 16)
    g = orc.mala_backward(q, k, v, f.o, do, f.lse, 0.25, 1e30, 16, 16)
    assert not g.retained.any()
    assert not (g.dq.any() or g.dk.any() or g.dv.any())


@pytest.mark.parametrize("tau,b,seed", [(1.0, 16, 31), (1.0, 32, 32), (0.5, 8, 33)])
def test_backward_support_nested_in_forward(tau, b, seed):
    q, k, v, do = _peaked(L=256, seed=seed)
    f = orc.mala_forward(q, k, v, PIN_SCALE, tau, b, b)
    g = orc.mala_backward(q, k, v, f.o, do, f.lse, PIN_SCALE, tau, b, b)
    assert np.array_equal(g.legal, f.legal)
    assert not (g.retained & ~f.retained).any()          # bwd support within fwd support
    assert (f.retained & ~g.retained).any() or True       # may be strictly smaller


def test_backward_brute_force_entry_rule():
    """Eq. 4 as a loop over single entries: tile (j, i) is kept iff some valid
    entry has exp(s - lse_q) >= tau / L_q."""
    q, k, v, do = _peaked(L=128, seed=34)
    b, tau = 16, 1.0
    f = orc.mala_forward(q, k, v, PIN_SCALE, tau, b, b)
    g = orc.mala_backward(q, k, v, f.o, do, f.lse, PIN_SCALE, tau, b, b)
    s = PIN_SCALE * (q @ k.T)
    t = 128 // b
    for i in range(t):
        for j in range(i + 1):
            keep = any(math.exp(s[r, c] - f.lse[r]) >= tau / (r + 1)
                       for r in range(i * b, (i + 1) * b) for c in range(j * b, (j + 1) * b) if c <= r)
            assert g.retained[i, j] == keep


def test_backward_is_gradient_of_forward_when_supports_coincide():
    """Where the backward support equals the forward one and no test is near
    its threshold, MALA forward is smooth and Algorithm 2 is its exact
    gradient (central differences)."""
    q, k, v, do = _peaked(L=128, seed=3)
    scale, tau, b = PIN_SCALE, 1.0, 16
    f = orc.mala_forward(q, k, v, scale, tau, b, b)
    g = orc.mala_backward(q, k, v, f.o, do, f.lse, scale, tau, b, b)
    assert np.array_equal(g.retained, f.retained) and not np.array_equal(f.retained, f.legal)
    assert np.nanmin(np.abs(f.margin[f.legal & np.isfinite(f.margin)])) > 1e-3
    assert np.nanmin(np.abs(g.margin[g.legal])) > 1e-3
    fun = lambda qq, kk, vv: (orc.mala_forward(qq, kk, vv, scale, tau, b, b).o * do).sum()
    eps = 1e-6
    rng = np.random.default_rng(0)
    for name, x, gr in (("q", q, g.dq), ("k", k, g.dk), ("v", v, g.dv)):
        for _ in range(6):
            idx = (rng.integers(0, 128), rng.integers(0, 32))
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap = [xp if n == name else y for n, y in (("q", q), ("k", k), ("v", v))]
            am = [xm if n == name else y for n, y in (("q", q), ("k", k), ("v", v))]
            fd = (fun(*ap) - fun(*am)) / (2 * eps)
            assert fd == pytest.approx(gr[idx], rel=1e-5, abs=1e-8), (name, idx)


# ---------------------------------------------------------------------------
# Split-KV decode (MALA §2.4, App. A.1) and the merge.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,splits", [(512, 1), (512, 4), (500, 3), (100, 8)])
def test_decode_tau0_is_dense(n, splits):
    qg = _rand((4, 16), 41, 2.0)
    kc, vc = _rand((n, 16), 42), _rand((n, 16), 43)
    r = orc.mala_decode(qg, kc, vc, 0.25, 0.0, 32, splits)
    o_ref, lse_ref = _sdpa(qg, kc, vc, 0.25, causal=False)
    np.testing.assert_allclose(r.o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r.lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_decode_single_split_equals_forward_on_the_head_group():
    """With one split, decode is Algorithm 1 on a query block made of the G
    heads of a group, all seeing the full cache (L = N)."""
    cfg = synthetic.CONFIGS["decode_128k"]
    x = synthetic.decode_inputs(cfg, N=1000, B=1, seed=3)
    qg = x["q"][0, 0:4].double().numpy()
    kc, vc = x["k"][0, :, 0].double().numpy(), x["v"][0, :, 0].double().numpy()
    scale = 1 / math.sqrt(128)
    r = orc.mala_decode(qg, kc, vc, scale, 1.0, 128, 1)
    f = orc.mala_forward(qg, kc, vc, scale, 1.0, 4, 128, causal=False)
    np.testing.assert_allclose(r.o, f.o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r.lse, f.lse, rtol=1e-13)
    assert np.array_equal(r.retained, f.retained[0])


def test_decode_split_output_is_renormalised_softmax_and_bounded():
    cfg = synthetic.CONFIGS["decode_128k"]
    x = synthetic.decode_inputs(cfg, N=2048, B=1, seed=4)
    qg = x["q"][0, 4:8].double().numpy()
    kc, vc = x["k"][0, :, 1].double().numpy(), x["v"][0, :, 1].double().numpy()
    scale = 1 / math.sqrt(128)
    for splits in (1, 4, 16):
        r = orc.mala_decode(qg, kc, vc, scale, 1.0, 64, splits)
        keep = np.tile(r.retained[None, :], (4, 1))
        # query "block" index is the head row here: one block of 4 rows
        o_r, lse_r = orc.restricted_attention(qg, kc, vc, scale, r.retained[None, :], 4, 64, causal=False)
        np.testing.assert_allclose(r.o, o_r, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(r.lse, lse_r, rtol=1e-12)
        _, lse_d = orc.dense_attention(qg, kc, vc, scale, causal=False)
        assert np.all(orc.omitted_mass(r.lse, lse_d) <= 0.5)
        assert keep.shape == (4, 32)


def test_decode_varlen_uses_each_sequence_length_uniform_scores():
    """Uniform scores (q = 0) make every decision a closed form.  A 100-token
    sequence in a cache padded to 200 rows, 32-key tiles, one split, tau = 4:
    the newest (4-key) tile is retained (l = 0), the next gives ratio
    -log 4 >= log(4/100) and is retained (l = 36), the older two give
    -log 36 < log(4/100) and are skipped.  With L = 200 instead, tile 1 would
    be retained (-log 36 >= log(4/200)).  The output is the mean of v over
    keys 64..99 (the retained keys).  The full 200-row cache (L = 200, newest
    tile of 8 keys) keeps tiles 6, 5, 4 (-log 40 >= log(4/200) > -log 72)."""
    n_max, n = 200, 100
    q = np.zeros((1, 2, 8))
    k = _rand((1, n_max, 1, 8), 91)
    v = _rand((1, n_max, 1, 8), 92)
    r = orc.mala_decode_varlen_bhd(q, k, v, [n], 0.5, 4.0, 32, 1)
    assert r["retained"][0, 0].tolist() == [False, False, True, True, False, False, False]
    np.testing.assert_allclose(r["o"][0, 0], v[0, 64:100, 0].mean(axis=0), rtol=1e-13)
    np.testing.assert_allclose(r["lse"][0], math.log(36.0), rtol=1e-13)
    full = orc.mala_decode_varlen_bhd(q, k, v, [n_max], 0.5, 4.0, 32, 1)
    assert full["retained"][0, 0].tolist() == [False, False, False, False, True, True, True]
    np.testing.assert_allclose(full["o"][0, 0], v[0, 128:200, 0].mean(axis=0), rtol=1e-13)
    np.testing.assert_allclose(full["lse"][0], math.log(72.0), rtol=1e-13)


@pytest.mark.parametrize("lens,splits", [([40, 200, 1, 129], 3), ([200, 200, 200, 200], 4)])
def test_decode_varlen_tau0_is_dense_over_each_prefix(lens, splits):
    """tau = 0: each sequence's output is plain softmax attention over its own
    first cache_lens[b] keys."""
    q = _rand((4, 2, 16), 93, 2.0)
    k, v = _rand((4, 200, 1, 16), 94), _rand((4, 200, 1, 16), 95)
    r = orc.mala_decode_varlen_bhd(q, k, v, lens, 0.25, 0.0, 32, splits)
    for b, n in enumerate(lens):
        o_ref, lse_ref = _sdpa(q[b], k[b, :n, 0], v[b, :n, 0], 0.25, causal=False)
        np.testing.assert_allclose(r["o"][b], o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["lse"][b], lse_ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Per-head decode: §2.2's rule with each query head as its own one-row block.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("splits", [1, 3])
def test_decode_per_head_tau0_is_dense(splits):
    q = _rand((2, 4, 16), 101, 2.0)
    k, v = _rand((2, 300, 2, 16), 102), _rand((2, 300, 2, 16), 103)
    r = orc.mala_decode_per_head_bhd(q, k, v, 0.25, 0.0, 32, splits)
    for b in range(2):
        for h in range(4):
            o_ref, lse_ref = _sdpa(q[b, h:h + 1], k[b, :, h // 2], v[b, :, h // 2], 0.25, causal=False)
            np.testing.assert_allclose(r["o"][b, h], o_ref[0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(r["lse"][b, h], lse_ref[0], rtol=1e-12)
    assert r["retained"].all()


def test_decode_per_head_single_split_equals_forward_on_one_row():
    """With one split, each head's decode is Algorithm 1 on a one-row query
    block seeing the whole cache (L = N), tiles newest first."""
    cfg = synthetic.CONFIGS["decode_128k"]
    x = synthetic.decode_inputs(cfg, N=1000, B=1, seed=5)
    q = x["q"][:, 0:4].double().numpy()
    kc, vc = x["k"][:, :, 0:1].double().numpy(), x["v"][:, :, 0:1].double().numpy()
    scale = 1 / math.sqrt(128)
    r = orc.mala_decode_per_head_bhd(q, kc, vc, scale, 1.0, 128, 1)
    for h in range(4):
        f = orc.mala_forward(q[0, h:h + 1], kc[0, :, 0], vc[0, :, 0], scale, 1.0, 1, 128, causal=False)
        np.testing.assert_allclose(r["o"][0, h], f.o[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r["lse"][0, h], f.lse[0], rtol=1e-13)
        assert np.array_equal(r["retained"][0, h], f.retained[0])


def test_decode_per_head_differs_from_group_closed_form():
    """Two heads over one 100-token cache, 32-key tiles, one split, tau = 4,
    L = 100.  Head 0 sees uniform scores (q = 0): it keeps the newest tile
    (l = 0), then the next (ratio -log 4 >= log(4/100)), and skips the two
    older ones (-log 36 < log(4/100)): output = mean of v over keys 64..99,
    lse = log 36.  Head 1 sees the same zeros except one score of 9 at key 5:
    it also keeps the oldest tile (9 - log 36 >= log(4/100)), so its output is
    (sum of v over keys 0..31 and 64..99, key 5 weighted e^9) / (67 + e^9 - 1).
    Deciding as a group, head 0 would have taken the oldest tile too."""
    n, d = 100, 8
    k = _rand((1, n, 1, d), 111)
    k[0, :, 0, 0] = 0.0
    k[0, 5, 0, 0] = 9.0
    v = _rand((1, n, 1, d), 112)
    q = np.zeros((1, 2, d))
    q[0, 1, 0] = 1.0
    r = orc.mala_decode_per_head_bhd(q, k, v, 1.0, 4.0, 32, 1)
    assert r["retained"][0, 0].tolist() == [False, False, True, True]
    assert r["retained"][0, 1].tolist() == [True, False, True, True]
    np.testing.assert_allclose(r["o"][0, 0], v[0, 64:100, 0].mean(axis=0), rtol=1e-13)
    np.testing.assert_allclose(r["lse"][0, 0], math.log(36.0), rtol=1e-13)
    w = np.zeros(n)
    w[0:32] = 1.0
    w[64:100] = 1.0
    w[5] = math.exp(9.0)
    np.testing.assert_allclose(r["o"][0, 1], (w[:, None] * v[0, :, 0]).sum(0) / w.sum(), rtol=1e-12)
    np.testing.assert_allclose(r["lse"][0, 1], math.log(w.sum()), rtol=1e-13)
    g = orc.mala_decode_bhd(q, k, v, 1.0, 4.0, 32, 1)
    assert g["retained"][0, 0].tolist() == [True, False, True, True]
    np.testing.assert_allclose(g["o"][0, 0], v[0, list(range(32)) + list(range(64, 100)), 0].mean(axis=0),
                               rtol=1e-12)


def test_decode_per_head_with_single_head_groups_is_the_group_decode():
    q = _rand((2, 3, 16), 121, 2.0)
    k, v = _rand((2, 250, 3, 16), 122), _rand((2, 250, 3, 16), 123)
    a = orc.mala_decode_per_head_bhd(q, k, v, 0.25, 2.0, 32, 3)
    b = orc.mala_decode_bhd(q, k, v, 0.25, 2.0, 32, 3)
    np.testing.assert_array_equal(a["retained"], b["retained"])
    np.testing.assert_allclose(a["o"], b["o"], rtol=0, atol=0)


# ---------------------------------------------------------------------------
# Packed variable-length prefill: each sequence is its own context.
# ---------------------------------------------------------------------------

def test_varlen_tau0_is_dense_causal_per_sequence():
    lens = [1, 5, 40, 17]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v = _rand((63, 2, 8), 131, 2.0), _rand((63, 1, 8), 132), _rand((63, 1, 8), 133)
    r = orc.mala_forward_varlen(q, k, v, cu, 0.3, 0.0, 8, 8)
    for b, n in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        for h in range(2):
            o_ref, lse_ref = _sdpa(q[sl, h], k[sl, 0], v[sl, 0], 0.3, causal=True)
            np.testing.assert_allclose(r["o"][sl, h], o_ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(r["lse"][h, sl], lse_ref, rtol=1e-12, atol=1e-12)
    do = _rand((63, 2, 8), 134)
    g = orc.mala_backward_varlen(q, k, v, r["o"], do, r["lse"], cu, 0.3, 0.0, 8, 8)
    for b, n in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        dk_sum = np.zeros((n, 8))
        dv_sum = np.zeros((n, 8))
        for h in range(2):
            dq_r, dk_r, dv_r = _sdpa_grads(q[sl, h], k[sl, 0], v[sl, 0], do[sl, h], 0.3)
            np.testing.assert_allclose(g["dq"][sl, h], dq_r, rtol=1e-10, atol=1e-12)
            dk_sum += dk_r
            dv_sum += dv_r
        np.testing.assert_allclose(g["dk"][sl, 0], dk_sum, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dv"][sl, 0], dv_sum, rtol=1e-10, atol=1e-12)


def test_varlen_equal_lengths_is_the_batched_layout():
    """Packing B sequences of L rows is the [B, L, H, d] batch laid end to end."""
    q, k, v = _rand((3, 40, 2, 8), 141, 2.0), _rand((3, 40, 2, 8), 142), _rand((3, 40, 2, 8), 143)
    a = orc.mala_forward_varlen(q.reshape(120, 2, 8), k.reshape(120, 2, 8), v.reshape(120, 2, 8),
                                [0, 40, 80, 120], 0.35, 2.0, 8, 8)
    b = orc.mala_forward_bshd(q, k, v, 0.35, 2.0, 8, 8)
    np.testing.assert_array_equal(a["o"], b["o"].reshape(120, 2, 8))
    np.testing.assert_array_equal(a["lse"], b["lse"].transpose(1, 0, 2).reshape(2, 120))
    np.testing.assert_array_equal(a["retained"], b["retained"])


# Scores of six one-key tiles (newest last) whose decisions are a closed form
# with tau / L = 0.5 (tau = 3, L = N = 6), for the split test below.
SPLIT_SCORES = [math.log(1.56), math.log(1.25), math.log(2.0), -50.0, -50.0, 0.0]


def _split_case():
    s = np.array(SPLIT_SCORES)
    q = np.array([[1.0, 0.0]])
    k = np.stack([s, np.zeros(6)], axis=1)
    v = _rand((6, 3), 95)
    return q, k, v


def test_decode_splits_start_from_empty_state_closed_form():
    """Each split starts from an empty (m, l) and walks its own tiles newest
    first (MALA §2.4 and App. A.1, fused decoding execution; Algorithm 1 per
    split), so more splits can keep a tile that one pass skips and also skip
    one that it keeps.  §2.4 calls the split's smaller normalizer more
    conservative; that holds only while the split's normalizer is no larger
    than the one-pass one, and it is larger once the split has kept a tile
    that the one pass skipped (tile 1 below).

    Tile masses w = exp(score): tile 5 = 1, tiles 4, 3 = e^-50, tile 2 = 2,
    tile 1 = 1.25, tile 0 = 1.56; keep iff w_max / Z >= 0.5 (Z = retained
    mass so far in the split, l = 0 keeps).
    One split: 5 kept (Z 1); 4, 3 skipped; 2 kept (2/1, Z 3); 1 skipped
    (1.25/3 = 0.42); 0 kept (1.56/3 = 0.52).
    Two splits {3,4,5}, {0,1,2}: 5 kept, 4 and 3 skipped; 2 kept (first),
    1 kept (1.25/2 = 0.63, Z 3.25), 0 skipped (1.56/3.25 = 0.48).
    Three splits {4,5}, {2,3}, {0,1}: 5 kept, 4 skipped; 3 kept (first), 2 kept;
    1 kept (first), 0 kept (1.56/1.25).
    The merged output is the softmax renormalised over the kept keys."""
    q, k, v = _split_case()
    w = np.exp(np.array(SPLIT_SCORES))
    for splits, kept in ((1, [0, 2, 5]), (2, [1, 2, 5]), (3, [0, 1, 2, 3, 5])):
        r = orc.mala_decode(q, k, v, 1.0, 3.0, 1, splits)
        assert np.flatnonzero(r.retained).tolist() == kept, splits
        z = w[kept].sum()
        np.testing.assert_allclose(r.lse, [math.log(z)], rtol=1e-14)
        np.testing.assert_allclose(r.o[0], (w[kept, None] * v[kept]).sum(0) / z, rtol=1e-13)
    # with 6 splits every tile is its split's first, so every tile is kept: dense
    r6 = orc.mala_decode(q, k, v, 1.0, 3.0, 1, 6)
    assert r6.retained.all()
    np.testing.assert_allclose(r6.lse, [math.log(w.sum())], rtol=1e-14)


# ---------------------------------------------------------------------------
# Matched-work controls (§3 Table 1, App. C.2).
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [True, False])
def test_tile_reference_mass_uniform_scores_closed_form(causal):
    """q = 0 makes every row's softmax uniform over its legal keys, so a
    region's mass is a count: sum over the block's rows r of
    (legal keys of r in the tile) / (legal keys of r)."""
    nq = nk = 10
    bq = bk = 4
    q = np.zeros((nq, 3))
    k = _rand((nk, 3), 101)
    got = orc.tile_reference_mass(q, k, 0.7, bq, bk, causal=causal)
    want = np.zeros((3, 3))
    for r in range(nq):
        visible = r + 1 if causal else nk
        for key in range(visible):
            want[r // bq, key // bk] += 1.0 / visible
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)
    legal = orc.legal_tiles(nq, nk, bq, bk, causal)
    assert (got[~legal] == 0).all() and (got[legal] > 0).all()


def test_tile_reference_mass_blocks_hold_their_rows():
    q, k = _rand((37, 8), 102, 2.0), _rand((37, 8), 103, 2.0)
    mass = orc.tile_reference_mass(q, k, 0.5, 16, 16)
    np.testing.assert_allclose(mass.sum(axis=1), [16, 16, 5], rtol=1e-13)


def test_top_mass_keep_is_the_best_subset_brute_force():
    """For every block and every n, the kept tiles carry the largest mass any
    n legal tiles can (checked against all subsets)."""
    import itertools
    rng = np.random.default_rng(104)
    mass = rng.random((4, 6))
    legal = orc.legal_tiles(4 * 3, 6 * 2, 3, 2)        # a causal pattern of 4 x 6 tiles
    for n in range(1, 7):
        keep = orc.top_mass_keep(mass, [n] * 4, legal)
        for i in range(4):
            cands = np.flatnonzero(legal[i])
            best = max(sum(mass[i, list(c)]) for c in itertools.combinations(cands, min(n, len(cands))))
            assert keep[i].sum() == min(n, len(cands))
            assert not (keep[i] & ~legal[i]).any()
            assert mass[i, keep[i]].sum() == pytest.approx(best, rel=1e-14)


def test_matched_work_allocation_closed_form():
    counts = np.array([[[1, 3], [2, 2]], [[1, 4], [3, 2]]])      # [input, head, query block]
    np.testing.assert_array_equal(orc.matched_work_allocation(counts, "instance"), counts)
    # (head, block) cells 0..3: totals 2, 7, 5, 4 over 2 inputs; cell 1 gives its
    # extra unit to input 1, cell 2 to input 0
    np.testing.assert_array_equal(orc.matched_work_allocation(counts, "head_position"),
                                  [[[1, 3], [3, 2]], [[1, 4], [2, 2]]])
    # block cells 0, 1: totals 7 and 11 over 4 copies (x = 2 i + h): base 1 + extra
    # for x = 0, 1, 2; base 2 + extra for x = 1, 2, 3
    np.testing.assert_array_equal(orc.matched_work_allocation(counts, "position"),
                                  [[[2, 2], [2, 3]], [[2, 3], [1, 3]]])


@pytest.mark.parametrize("scope", ["head_position", "position"])
def test_matched_work_allocation_matches_work_exactly(scope):
    rng = np.random.default_rng(105)
    legal_per_block = np.arange(1, 9)                         # causal: block i has i + 1 legal tiles
    counts = rng.integers(1, legal_per_block + 1, size=(5, 3, 8))
    alloc = orc.matched_work_allocation(counts, scope)
    axes = (0,) if scope == "head_position" else (0, 1)
    np.testing.assert_array_equal(alloc.sum(axis=axes), counts.sum(axis=axes))    # per cell, so in total
    assert (alloc.max(axis=axes) - alloc.min(axis=axes) <= 1).all()              # one allocation per cell
    assert (alloc >= 1).all() and (alloc <= legal_per_block).all()


# ---------------------------------------------------------------------------
# Forced-decision replay (MALA §2.2 Eq. 3 and Algorithm 1: each test reads the
# (m, l) that the earlier decisions produced), used by the parity checks at
# borderline tiles.
# ---------------------------------------------------------------------------

def three_key_case():
    """Causal rows 0-2 with d = 1, scale 1 and one-key tiles, so row 2 visits
    keys 2, 1, 0 (newest first) with scores 0, log 0.5, log 0.6; tau = 1.5, so
    row 2's threshold is tau / L = 0.5 on the ratio exp(s) / Z.  Key 2 is kept
    (l = 0).  Key 1's ratio is 0.5 / 1: exactly the threshold, a borderline
    tile.  Key 0's ratio is 0.6 / 1.5 = 0.4 (skip) if key 1 was kept and
    0.6 / 1 = 0.6 (keep) if it was not: both 20% from the threshold."""
    q = np.ones((3, 1))
    k = np.array([[math.log(0.6)], [math.log(0.5)], [0.0]])
    v = np.array([[1.0], [10.0], [100.0]])
    return q, k, v, 1.5


def test_replay_follows_a_borderline_tile_and_the_later_tests_follow_the_state():
    q, k, v, tau = three_key_case()
    free = orc.mala_forward(q, k, v, 1.0, tau, 1, 1)
    assert orc.is_borderline(free.margin[2, 1])
    # kept key 1: Z = 1.5, key 0 skipped; o = (0.5 * 10 + 100) / 1.5
    r = orc.mala_forward(q, k, v, 1.0, tau, 1, 1, forced=np.tril(np.ones((3, 3), bool)))
    assert r.retained[2].tolist() == [False, True, True]
    assert r.o[2, 0] == pytest.approx(105.0 / 1.5, rel=1e-14)
    assert r.lse[2] == pytest.approx(math.log(1.5), rel=1e-14)
    assert r.margin[2, 0] == pytest.approx(math.log(0.8), rel=1e-12)
    # skipped key 1: Z = 1, key 0 kept; o = (0.6 * 1 + 100) / 1.6
    forced = np.tril(np.ones((3, 3), bool))
    forced[2, 1] = False
    r = orc.mala_forward(q, k, v, 1.0, tau, 1, 1, forced=forced)
    assert r.retained[2].tolist() == [True, False, True]
    assert r.o[2, 0] == pytest.approx(100.6 / 1.6, rel=1e-14)
    assert r.lse[2] == pytest.approx(math.log(1.6), rel=1e-14)
    assert r.margin[2, 0] == pytest.approx(math.log(1.2), rel=1e-12)
    # rows 0 and 1 have no borderline tile and are untouched by the forced mask
    for rr in (0, 1):
        assert r.retained[rr].tolist() == free.retained[rr].tolist()
        assert r.o[rr, 0] == free.o[rr, 0]


def test_replay_ignores_forced_decisions_at_tiles_that_are_not_borderline():
    q, k, v, tau = three_key_case()
    # key 0 of row 2 is 20% from the threshold on either path: never followed
    forced = np.zeros((3, 3), bool)
    forced[2, 2] = True                        # key 1 skipped, and key 0 "skipped" (ignored)
    r = orc.mala_forward(q, k, v, 1.0, tau, 1, 1, forced=forced)
    assert r.retained[2].tolist() == [True, False, True]
    assert r.retained[1].tolist() == [True, True, False]      # row 1 keeps both keys regardless
    forced = np.ones((3, 3), bool)             # key 1 kept, and key 0 "kept" (ignored)
    r = orc.mala_forward(q, k, v, 1.0, tau, 1, 1, forced=forced)
    assert r.retained[2].tolist() == [False, True, True]


def test_replay_with_the_runs_own_decisions_or_their_complement_is_the_run():
    """On inputs with no borderline tile any forced mask leaves every result
    unchanged; with the run's own mask nothing is overridden."""
    q, k, v, _ = _peaked(L=192, seed=21)
    free = orc.mala_forward(q, k, v, PIN_SCALE, 1.0, 16, 16)
    assert not orc.is_borderline(free.margin).any()
    assert (~free.retained & free.legal).any() and free.retained.any()
    for forced in (free.retained, ~free.retained):
        r = orc.mala_forward(q, k, v, PIN_SCALE, 1.0, 16, 16, forced=forced)
        for name in ("o", "lse", "retained", "legal", "margin"):
            np.testing.assert_array_equal(getattr(r, name), getattr(free, name))
        assert not r.overridden.any()


def test_decode_replay_closed_form():
    """The three keys as a one-query cache (N = 3, one split): the same path
    dependence as row 2 of the prefill case."""
    _, k, v, tau = three_key_case()
    qg = np.ones((1, 1))
    free = orc.mala_decode(qg, k, v, 1.0, tau, 1, 1)
    assert orc.is_borderline(free.margin[1])
    r = orc.mala_decode(qg, k, v, 1.0, tau, 1, 1, forced=np.array([False, False, True]))
    assert r.retained.tolist() == [True, False, True]
    assert r.o[0, 0] == pytest.approx(100.6 / 1.6, rel=1e-14)
    r = orc.mala_decode(qg, k, v, 1.0, tau, 1, 1, forced=np.array([True, True, True]))
    assert r.retained.tolist() == [False, True, True]
    assert r.lse[0] == pytest.approx(math.log(1.5), rel=1e-14)


def test_backward_replay_follows_only_borderline_tiles():
    """One query, one key, S = 0, tau = 1, L = 1: the Eq. 4 margin S - lse is
    exactly 0 at lse = 0 (borderline) and 1 at lse = -1 (kept, P = e)."""
    q = k = v = do = o = np.ones((1, 1))
    k = np.zeros((1, 1))
    for forced, dv in ((True, 1.0), (False, 0.0)):
        r = orc.mala_backward(q, k, v, o, do, np.zeros(1), 1.0, 1.0, 1, 1, forced=np.array([[forced]]))
        assert r.retained[0, 0] == forced
        assert r.dv[0, 0] == pytest.approx(dv, abs=1e-15)
    r = orc.mala_backward(q, k, v, o, do, np.array([-1.0]), 1.0, 1.0, 1, 1, forced=np.array([[False]]))
    assert r.retained[0, 0]
    assert r.dv[0, 0] == pytest.approx(math.e, rel=1e-14)
