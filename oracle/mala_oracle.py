"""fp64 CPU oracle for MassAlloc Attention (MALA).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg use it.  It shares no code with the CUDA library.

Everything here is written to be checked by eye against the pages:

* "MassAlloc Attention: Let Attention Allocate Its Own Compute" (arXiv HTML):
  §2.1 (score discovery, visible-key counts L_q, threshold tau/L_q),
  §2.2 Eq. (1)-(4) (online forward test, offline backward test, support
  nesting), Algorithm 1 (forward), Algorithm 2 (backward), App. A.1 (fused
  forward/backward/decoding execution, split-KV), App. B Eq. (5)-(10)
  (omitted-mass bound), App. C.2 (omitted-mass measurement, matched-work
  allocation controls), §3 Table 1 (the matched-work study).
* "Why exact attention does not need a quadratic matrix": Method/Mechanism
  (block summary (m, l, u) and the merge identity), Example 1.

Conventions (one head at a time; the *_bshd wrappers loop over batch/heads):
  q [Nq, d], k/v [Nk, d], all float64.  Scores are s = scale * q k^T with the
  softmax scale applied to the scores (the paper absorbs it into Q, §2.1).
  Natural exp/log throughout (§2.1).  Zero-based positions; causal prefill
  means key k is visible to query q iff k <= q, so L_q = q + 1 (§2.1).

Readings of points the pages leave open:
  * only key blocks with at least one legal entry for the query block are
    visited (Algorithm 1 loops over all j; App. A.1 walks only the legal ones);
  * rows (or entries) that are out of range or fully masked in a tile do not
    constrain the test (§2.2 text after Eq. 3 and after Eq. 4);
  * the skip test is a strict "<"; equality retains;
  * l = 0 is an explicit "+inf ratio, retain" branch (§2.2, first-tile rule);
  * tau = 0 runs no test at all (dense: §2.3 notes that the tau -> 0 limit
    is full attention);
  * decode: the query block is the group of query heads sharing one KV head,
    the split partition is num_splits equal ranges of whole tiles, tiles are
    visited newest to oldest inside a split, and L = N_k (§2.1, App. A.1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "visible_key_counts", "dense_attention", "dense_attention_grads",
    "restricted_attention", "mala_forward", "mala_backward",
    "block_summary", "merge_summaries", "mala_decode",
    "mala_forward_bshd", "mala_backward_bshd", "mala_forward_varlen", "mala_backward_varlen",
    "mala_decode_bhd", "mala_decode_per_head_bhd",
    "mala_decode_varlen_bhd",
    "omitted_mass", "BORDERLINE_REL", "is_borderline",
    "legal_tiles", "tile_reference_mass", "matched_work_allocation", "top_mass_keep",
]

# A tile whose largest contribution ratio lies within this relative distance
# of tau/L_q is "borderline": fp32 and fp64 evaluations may legitimately
# decide it differently.
BORDERLINE_REL = 1e-3


def is_borderline(margin):
    """True where a tile's largest contribution ratio lies within
    BORDERLINE_REL (relative) of the threshold: margin is the log of
    ratio / (tau / L_q), so the band is |exp(margin) - 1| <= BORDERLINE_REL.
    Infinite margins (l = 0, always retained) and NaN (not tested) are not
    borderline."""
    m = np.asarray(margin, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return np.isfinite(m) & (np.abs(np.expm1(m)) <= BORDERLINE_REL)


def _follow(skip, margin, forced):
    """Forced-decision replay: at a borderline tile, where an fp32 and an fp64
    evaluation of the same test may legitimately disagree, take the given
    decision (forced = keep) instead of this run's own; elsewhere keep the
    test's.  Returns (skip, overridden)."""
    if forced is None or not is_borderline(margin):
        return skip, False
    follow_skip = not bool(forced)
    return follow_skip, follow_skip != skip


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def visible_key_counts(n_q: int, n_k: int, causal: bool) -> np.ndarray:
    """L_q = |C_q| (§2.1): q + 1 for zero-based causal rows, else N_k."""
    if causal:
        return np.arange(1, n_q + 1, dtype=np.float64)
    return np.full(n_q, float(n_k))


def _scores(q, k, scale, rows, cols, causal):
    """Score tile S = scale * Q_rows K_cols^T with causal entries set to -inf."""
    s = scale * (q[rows] @ k[cols].T)
    if causal:
        s = np.where(cols[None, :] > rows[:, None], -np.inf, s)
    return s


# ---------------------------------------------------------------------------
# Dense causal softmax attention and its analytic gradients (the tau = 0 case).
# ---------------------------------------------------------------------------

def dense_attention(q, k, v, scale, causal=True, rows=None):
    """Plain softmax attention: o_q = sum_k p_qk v_k, lse_q = log sum_k exp(s_qk).

    Row-independent, so rows may be evaluated in any order or subset.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(k.shape[0])
    o = np.zeros((len(rows), v.shape[1]))
    lse = np.zeros(len(rows))
    for a in range(0, len(rows), 256):
        r = rows[a:a + 256]
        s = _scores(q, k, scale, r, cols, causal)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        z = p.sum(axis=1, keepdims=True)
        o[a:a + 256] = (p @ v) / z
        lse[a:a + 256] = (m + np.log(z))[:, 0]
    return o, lse


def dense_attention_grads(q, k, v, do, scale, causal=True):
    """Analytic softmax-attention gradients w.r.t. the unscaled q, k and v.

    P = softmax(S), dV = P^T dO, dP = dO V^T, D = rowsum(dO o O),
    dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    rows = np.arange(q.shape[0])
    cols = np.arange(k.shape[0])
    s = _scores(q, k, scale, rows, cols, causal)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    p /= p.sum(axis=1, keepdims=True)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    dd = (do * o).sum(axis=1, keepdims=True)
    ds = p * (dp - dd)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def restricted_attention(q, k, v, scale, keep, bq, bk, causal=True, rows=None):
    """Softmax attention renormalised over the kept tiles only (§2.2: MALA's
    output equals plain softmax attention over the retained tiles, normalised
    over them).  keep[i, j] says whether tile (query block i, key block j) is kept.
    Written directly as a masked softmax, with no online update.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, nk = q.shape[0], k.shape[0]
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    cols = np.arange(nk)
    s = _scores(q, k, scale, rows, cols, causal)
    kept = np.asarray(keep, dtype=bool)[(rows // bq)[:, None], (cols // bk)[None, :]]
    s = np.where(kept, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    z = p.sum(axis=1, keepdims=True)
    return (p @ v) / z, (m + np.log(z))[:, 0]


def omitted_mass(lse_screened, lse_reference):
    """App. C.2: 1 - exp(l_screened - l_reference), the dense-softmax mass of
    the positions the screened operator omitted."""
    return 1.0 - np.exp(_f64(lse_screened) - _f64(lse_reference))


# ---------------------------------------------------------------------------
# MALA forward: Algorithm 1 with the online test of §2.2 Eq. (2)-(3).
# ---------------------------------------------------------------------------

@dataclass
class MalaForward:
    o: np.ndarray          # [Nq, d]
    lse: np.ndarray        # [Nq] final log-normaliser m + log l (natural log)
    retained: np.ndarray   # [Tr, Tc] bool: post-score path executed
    legal: np.ndarray      # [Tr, Tc] bool: tile has >= 1 legal entry (visited)
    margin: np.ndarray     # [Tr, Tc] max over rows of (log-ratio - log(tau/L)); skip iff < 0
    overridden: np.ndarray = None  # [Tr, Tc] bool: borderline tiles where a forced decision
                                   # differed from this run's own test (replay only)


def _log_threshold(tau, lq):
    return math.log(tau) - np.log(lq)


def mala_forward(q, k, v, scale, tau, bq, bk, causal=True, query_blocks=None, forced=None):
    """MALA forward for one head (Algorithm 1).

    For each query block, legal key blocks are visited from the diagonal
    toward earlier keys (App. A.1).  For each tile the scores are formed
    first; the tile is skipped iff for every row with a legal entry in it
    rowmax(S) - m - log(l) < log(tau / L_q)  (Eq. 3), where a row with l = 0
    has ratio +inf and therefore retains (§2.2).  A skipped tile leaves
    (m, l, O) untouched; a retained one takes the standard online-softmax
    update.  Finalisation: O /= l and lse = m + log(l).
    ``query_blocks`` restricts the work to a subset of blocks (others stay 0).

    ``forced`` ([Tr, Tc] bool, e.g. another implementation's tile mask) makes
    this a forced-decision replay: at a tile whose margin, measured on this
    run's own (m, l), is borderline (``is_borderline``), the given decision is
    taken instead of the test's; every other tile is decided by Eq. 3 as
    usual.  Because each later test reads the (m, l) that the earlier
    decisions produced (Algorithm 1), the replay is the oracle's result for
    the path on which every borderline tile went the given way.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if tau < 0 or not np.isfinite(tau):
        raise ValueError("tau must be finite and >= 0")
    nq, nk = q.shape[0], k.shape[0]
    tr, tc = -(-nq // bq), -(-nk // bk)
    lvis = visible_key_counts(nq, nk, causal)
    o = np.zeros((nq, v.shape[1]))
    lse = np.full(nq, np.nan)
    retained = np.zeros((tr, tc), dtype=bool)
    legal = np.zeros((tr, tc), dtype=bool)
    margin = np.full((tr, tc), np.nan)
    overridden = np.zeros((tr, tc), dtype=bool)
    blocks = range(tr) if query_blocks is None else query_blocks
    for i in blocks:
        rows = np.arange(i * bq, min(nq, (i + 1) * bq))
        m = np.full(len(rows), -np.inf)
        l = np.zeros(len(rows))
        acc = np.zeros((len(rows), v.shape[1]))
        thr = _log_threshold(tau, lvis[rows]) if tau > 0 else None
        for j in reversed(range(tc)):
            cols = np.arange(j * bk, min(nk, (j + 1) * bk))
            s = _scores(q, k, scale, rows, cols, causal)
            has = np.isfinite(s).any(axis=1)      # rows with a legal entry here
            if not has.any():
                continue                          # fully masked: not a legal tile
            legal[i, j] = True
            mt = np.where(has, s.max(axis=1), -np.inf)
            if tau > 0:
                with np.errstate(divide="ignore"):
                    ratio = np.where(l > 0, mt - m - np.log(np.where(l > 0, l, 1.0)), np.inf)
                gap = (ratio - thr)[has]
                margin[i, j] = gap.max()
                skip, overridden[i, j] = _follow(bool(np.all(gap < 0)), margin[i, j],
                                                 None if forced is None else forced[i, j])
                if skip:
                    continue                      # skip block (i, j)
            retained[i, j] = True
            # online-softmax update; rows without a legal key here keep their state
            m_new = np.where(has, np.maximum(m, mt), m)
            alpha = np.ones(len(rows))            # exp(m - m_new); empty rows have nothing to rescale
            live = l > 0
            alpha[live] = np.exp(m[live] - m_new[live])
            p = np.zeros_like(s)
            p[has] = np.exp(s[has] - m_new[has][:, None])
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ v[cols]
            m = m_new
        o[rows] = acc / l[:, None]
        lse[rows] = m + np.log(l)
    return MalaForward(o, lse, retained, legal, margin, overridden)


# ---------------------------------------------------------------------------
# MALA backward: Algorithm 2 with the offline test of §2.2 Eq. (4).
# ---------------------------------------------------------------------------

@dataclass
class MalaBackward:
    dq: np.ndarray
    dk: np.ndarray
    dv: np.ndarray
    retained: np.ndarray   # [Tr, Tc] bool (indexed [query block, key block])
    legal: np.ndarray
    margin: np.ndarray     # max over valid entries of (S - lse - log(tau/L)); skip iff < 0
    overridden: np.ndarray = None  # borderline tiles where a forced decision differed (replay only)


def mala_backward(q, k, v, o, do, lse, scale, tau, bq, bk, causal=True, tiles=None, forced=None):
    """MALA backward for one head (Algorithm 2), key-major.

    For each key block j, the query blocks i with a legal entry are visited in
    ascending order.  The recomputed tile S_ji is skipped iff
    S_ji - lse_i^T < log(tau / L_i)^T for every valid causal entry (Eq. 4).
    A retained tile executes P = exp(S - lse), dP = V dO^T,
    dS = P o (dP - rowsum(O o dO)), dV += P dO, dK += dS Q, dQ += dS^T K,
    with the softmax scale carried onto dQ and dK (gradients are w.r.t. the
    unscaled q and k).  ``tiles`` (a predicate on (i, j)) restricts the work
    to a subset of tiles, for sampled checks at large sizes.  ``forced``
    ([Tr, Tc] bool) replays given decisions at borderline tiles, as in
    ``mala_forward``; here each test reads only the fixed lse, so a followed
    decision changes no other tile's.
    """
    q, k, v, o, do, lse = (_f64(x) for x in (q, k, v, o, do, lse))
    if tau < 0 or not np.isfinite(tau):
        raise ValueError("tau must be finite and >= 0")
    nq, nk = q.shape[0], k.shape[0]
    tr, tc = -(-nq // bq), -(-nk // bk)
    lvis = visible_key_counts(nq, nk, causal)
    dd = (o * do).sum(axis=1)                     # D = rowsum(O o dO)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    retained = np.zeros((tr, tc), dtype=bool)
    legal = np.zeros((tr, tc), dtype=bool)
    margin = np.full((tr, tc), np.nan)
    overridden = np.zeros((tr, tc), dtype=bool)
    for j in range(tc):
        cols = np.arange(j * bk, min(nk, (j + 1) * bk))
        for i in range(tr):
            if tiles is not None and not tiles(i, j):
                continue
            rows = np.arange(i * bq, min(nq, (i + 1) * bq))
            st = _scores(q, k, scale, rows, cols, causal).T     # S_ji = K_j Q_i^T
            valid = np.isfinite(st)
            if not valid.any():
                continue
            legal[i, j] = True
            if tau > 0:
                thr = _log_threshold(tau, lvis[rows])
                gap = (st - lse[rows][None, :] - thr[None, :])[valid]
                margin[i, j] = gap.max()
                skip, overridden[i, j] = _follow(bool(np.all(gap < 0)), margin[i, j],
                                                 None if forced is None else forced[i, j])
                if skip:
                    continue                                     # skip block (j, i)
            retained[i, j] = True
            p = np.where(valid, np.exp(st - lse[rows][None, :]), 0.0)
            dp = v[cols] @ do[rows].T
            ds = p * (dp - dd[rows][None, :])
            dv[cols] += p @ do[rows]
            dk[cols] += scale * (ds @ q[rows])
            dq[rows] += scale * (ds.T @ k[cols])
    return MalaBackward(dq, dk, dv, retained, legal, margin, overridden)


# ---------------------------------------------------------------------------
# Block summaries and the exact merge ("Why exact attention does not need a
# quadratic matrix", Method/Mechanism).
# ---------------------------------------------------------------------------

def block_summary(scores, values):
    """(m, l, u) of one non-empty block of finite scores for one query:
    m = max s, l = sum exp(s - m), u = sum exp(s - m) v."""
    s = _f64(scores)
    vals = _f64(values)
    m = s.max()
    w = np.exp(s - m)
    return m, w.sum(), (w[:, None] * vals.reshape(len(s), -1)).sum(axis=0)


def merge_summaries(summaries):
    """Merge identity: m = max m_b; rescale each (l_b, u_b) by exp(m_b - m)
    and add.  Empty blocks (l = 0, e.g. fully masked) carry no weight and are
    left out explicitly rather than evaluating -inf - (-inf)."""
    live = [(m, l, u) for (m, l, u) in summaries if l > 0]
    if not live:
        raise ValueError("merge of empty blocks only")
    m = max(mb for mb, _, _ in live)
    l = sum(math.exp(mb - m) * lb for mb, lb, _ in live)
    u = sum(math.exp(mb - m) * np.asarray(ub, dtype=np.float64) for mb, _, ub in live)
    return m, l, u


# ---------------------------------------------------------------------------
# MALA split-KV decode (App. A.1 "Fused decoding execution", §2.4).
# ---------------------------------------------------------------------------

@dataclass
class MalaDecode:
    o: np.ndarray          # [G, d]
    lse: np.ndarray        # [G]
    retained: np.ndarray   # [T] bool per key tile
    margin: np.ndarray     # [T]
    summaries: list        # per split: (m [G], l [G], u [G, d])
    overridden: np.ndarray = None  # [T] borderline tiles where a forced decision differed (replay only)


def mala_decode(qg, kc, vc, scale, tau, bk, num_splits, forced=None):
    """One query position of G query heads sharing one KV head, against an
    N-token cache (the cache already holds the current token, so L = N).

    The T = ceil(N / bk) key tiles are cut into ``num_splits`` contiguous
    ranges of ceil(T / num_splits) whole tiles.  Each split starts from its
    own empty (m, l) and visits its tiles newest to oldest, scoring every
    tile; a tile is skipped iff rowmax - m - log l < log(tau / N) holds for
    all G rows (Eq. 3 with the group of heads as the query block, l = 0 =>
    retain).  The splits' (m, l, u) are merged with the exact identity.
    ``forced`` ([T] bool) replays given decisions at borderline tiles, as in
    ``mala_forward`` (each split's later tests read the state they produce).
    """
    qg, kc, vc = _f64(qg), _f64(kc), _f64(vc)
    if tau < 0 or not np.isfinite(tau):
        raise ValueError("tau must be finite and >= 0")
    g, n = qg.shape[0], kc.shape[0]
    t = -(-n // bk)
    per = -(-t // num_splits)
    thr = math.log(tau) - math.log(n) if tau > 0 else None
    retained = np.zeros(t, dtype=bool)
    margin = np.full(t, np.nan)
    overridden = np.zeros(t, dtype=bool)
    summaries = []
    for sp in range(num_splits):
        m = np.full(g, -np.inf)
        l = np.zeros(g)
        u = np.zeros((g, vc.shape[1]))
        for j in reversed(range(sp * per, min(t, (sp + 1) * per))):
            cols = np.arange(j * bk, min(n, (j + 1) * bk))
            s = scale * (qg @ kc[cols].T)
            mt = s.max(axis=1)
            if tau > 0:
                with np.errstate(divide="ignore"):
                    ratio = np.where(l > 0, mt - m - np.log(np.where(l > 0, l, 1.0)), np.inf)
                gap = ratio - thr
                margin[j] = gap.max()
                skip, overridden[j] = _follow(bool(np.all(gap < 0)), margin[j],
                                              None if forced is None else forced[j])
                if skip:
                    continue
            retained[j] = True
            m_new = np.maximum(m, mt)
            alpha = np.ones(g)                    # exp(m - m_new); an empty state has nothing to rescale
            live = l > 0
            alpha[live] = np.exp(m[live] - m_new[live])
            p = np.exp(s - m_new[:, None])
            l = alpha * l + p.sum(axis=1)
            u = alpha[:, None] * u + p @ vc[cols]
            m = m_new
        summaries.append((m, l, u))
    o = np.zeros((g, vc.shape[1]))
    lse = np.zeros(g)
    for r in range(g):
        mr, lr, ur = merge_summaries([(m[r], l[r], u[r]) for (m, l, u) in summaries])
        o[r] = ur / lr
        lse[r] = mr + math.log(lr)
    return MalaDecode(o, lse, retained, margin, summaries, overridden)


# ---------------------------------------------------------------------------
# Batched wrappers over the library's layouts (BSHD for prefill, GQA mapping
# query head h -> KV head h // (Hq / Hkv)).
# ---------------------------------------------------------------------------

def mala_forward_bshd(q, k, v, scale, tau, bq, bk, causal=True, heads=None,
                      batches=None, query_blocks=None, forced=None):
    """q [B, L, Hq, d], k/v [B, L, Hkv, d] -> dict of o [B, L, Hq, d],
    lse [B, Hq, L], retained/legal/margin/overridden [B, Hq, Tr, Tc].
    ``forced`` [B, Hq, Tr, Tc]: decisions to replay at borderline tiles."""
    bsz, nq, hq, d = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    grp = hq // hkv
    tr, tc = -(-nq // bq), -(-nk // bk)
    out = {
        "o": np.zeros((bsz, nq, hq, v.shape[3])),
        "lse": np.full((bsz, hq, nq), np.nan),
        "retained": np.zeros((bsz, hq, tr, tc), dtype=bool),
        "legal": np.zeros((bsz, hq, tr, tc), dtype=bool),
        "margin": np.full((bsz, hq, tr, tc), np.nan),
        "overridden": np.zeros((bsz, hq, tr, tc), dtype=bool),
    }
    for b in (range(bsz) if batches is None else batches):
        for h in (range(hq) if heads is None else heads):
            r = mala_forward(q[b, :, h], k[b, :, h // grp], v[b, :, h // grp], scale, tau,
                             bq, bk, causal, query_blocks, None if forced is None else forced[b, h])
            out["o"][b, :, h] = r.o
            out["lse"][b, h] = r.lse
            out["retained"][b, h] = r.retained
            out["legal"][b, h] = r.legal
            out["margin"][b, h] = r.margin
            out["overridden"][b, h] = r.overridden
    return out


def mala_backward_bshd(q, k, v, o, do, lse, scale, tau, bq, bk, causal=True, heads=None,
                       batches=None, tiles=None, forced=None):
    """Gradients for BSHD inputs; dk/dv of a KV head sum over its query heads.
    ``forced`` [B, Hq, Tr, Tc]: decisions to replay at borderline tiles."""
    bsz, nq, hq, d = q.shape
    nk, hkv = k.shape[1], k.shape[2]
    grp = hq // hkv
    tr, tc = -(-nq // bq), -(-nk // bk)
    out = {
        "dq": np.zeros(q.shape), "dk": np.zeros(k.shape), "dv": np.zeros(v.shape),
        "retained": np.zeros((bsz, hq, tr, tc), dtype=bool),
        "legal": np.zeros((bsz, hq, tr, tc), dtype=bool),
        "margin": np.full((bsz, hq, tr, tc), np.nan),
        "overridden": np.zeros((bsz, hq, tr, tc), dtype=bool),
    }
    for b in (range(bsz) if batches is None else batches):
        for h in (range(hq) if heads is None else heads):
            r = mala_backward(q[b, :, h], k[b, :, h // grp], v[b, :, h // grp], o[b, :, h],
                              do[b, :, h], lse[b, h], scale, tau, bq, bk, causal, tiles,
                              None if forced is None else forced[b, h])
            out["dq"][b, :, h] = r.dq
            out["dk"][b, :, h // grp] += r.dk
            out["dv"][b, :, h // grp] += r.dv
            out["retained"][b, h] = r.retained
            out["legal"][b, h] = r.legal
            out["margin"][b, h] = r.margin
            out["overridden"][b, h] = r.overridden
    return out


def mala_forward_varlen(q, k, v, cu_seqlens, scale, tau, bq, bk, causal=True, heads=None, seqs=None,
                        forced=None):
    """Packed variable-length forward: sequence b is rows cu_seqlens[b] ..
    cu_seqlens[b + 1] - 1 of q [total, Hq, d], k / v [total, Hkv, d] and is
    its own context (§2.1 counts L_q per row within it), i.e. exactly
    ``mala_forward_bshd`` on that slice.  Returns o [total, Hq, d], lse
    [Hq, total] and retained / legal / margin [B, Hq, Tm, Tm] with
    Tm = ceil(max length / bq) (entries past a sequence's tiles False / NaN).
    ``forced`` [B, Hq, Tm, Tm]: decisions to replay at borderline tiles."""
    total, hq, d = q.shape
    nseq = len(cu_seqlens) - 1
    lens = [int(cu_seqlens[b + 1]) - int(cu_seqlens[b]) for b in range(nseq)]
    tm = -(-max(lens) // bq)
    out = {
        "o": np.zeros((total, hq, v.shape[2])),
        "lse": np.full((hq, total), np.nan),
        "retained": np.zeros((nseq, hq, tm, tm), dtype=bool),
        "legal": np.zeros((nseq, hq, tm, tm), dtype=bool),
        "margin": np.full((nseq, hq, tm, tm), np.nan),
        "overridden": np.zeros((nseq, hq, tm, tm), dtype=bool),
    }
    for b in (range(nseq) if seqs is None else seqs):
        s0, n = int(cu_seqlens[b]), lens[b]
        if n == 0:
            continue
        t = -(-n // bq)
        fb = None if forced is None else np.asarray(forced)[b:b + 1, :, :t, :t]
        r = mala_forward_bshd(q[None, s0:s0 + n], k[None, s0:s0 + n], v[None, s0:s0 + n], scale, tau, bq, bk,
                              causal, heads=heads, forced=fb)
        out["o"][s0:s0 + n] = r["o"][0]
        out["lse"][:, s0:s0 + n] = r["lse"][0]
        for key in ("retained", "legal", "margin", "overridden"):
            out[key][b, :, :t, :t] = r[key][0]
    return out


def mala_backward_varlen(q, k, v, o, do, lse, cu_seqlens, scale, tau, bq, bk, causal=True, heads=None, seqs=None,
                         forced=None):
    """Packed variable-length backward (layouts as ``mala_forward_varlen``):
    ``mala_backward_bshd`` on each sequence's slice."""
    total, hq, d = q.shape
    nseq = len(cu_seqlens) - 1
    lens = [int(cu_seqlens[b + 1]) - int(cu_seqlens[b]) for b in range(nseq)]
    tm = -(-max(lens) // bq)
    out = {"dq": np.zeros(q.shape), "dk": np.zeros(k.shape), "dv": np.zeros(v.shape),
           "retained": np.zeros((nseq, hq, tm, tm), dtype=bool),
           "legal": np.zeros((nseq, hq, tm, tm), dtype=bool),
           "margin": np.full((nseq, hq, tm, tm), np.nan),
           "overridden": np.zeros((nseq, hq, tm, tm), dtype=bool)}
    for b in (range(nseq) if seqs is None else seqs):
        s0, n = int(cu_seqlens[b]), lens[b]
        if n == 0:
            continue
        sl = slice(s0, s0 + n)
        t = -(-n // bq)
        fb = None if forced is None else np.asarray(forced)[b:b + 1, :, :t, :t]
        r = mala_backward_bshd(q[None, sl], k[None, sl], v[None, sl], o[None, sl], do[None, sl],
                               lse[None, :, sl], scale, tau, bq, bk, causal, heads=heads, forced=fb)
        out["dq"][sl] = r["dq"][0]
        out["dk"][sl] = r["dk"][0]
        out["dv"][sl] = r["dv"][0]
        for key in ("retained", "legal", "margin", "overridden"):
            out[key][b, :, :t, :t] = r[key][0]
    return out


def mala_decode_bhd(q, k_cache, v_cache, scale, tau, bk, num_splits, batches=None, forced=None):
    """q [B, Hq, d], caches [B, N, Hkv, d] -> o [B, Hq, d], lse [B, Hq],
    retained/margin/overridden [B, Hkv, T].  ``forced`` [B, Hkv, T]:
    decisions to replay at borderline tiles."""
    bsz, hq, d = q.shape
    n, hkv = k_cache.shape[1], k_cache.shape[2]
    grp = hq // hkv
    t = -(-n // bk)
    o = np.zeros((bsz, hq, v_cache.shape[3]))
    lse = np.full((bsz, hq), np.nan)
    retained = np.zeros((bsz, hkv, t), dtype=bool)
    margin = np.full((bsz, hkv, t), np.nan)
    overridden = np.zeros((bsz, hkv, t), dtype=bool)
    for b in (range(bsz) if batches is None else batches):
        for hk in range(hkv):
            r = mala_decode(q[b, hk * grp:(hk + 1) * grp], k_cache[b, :, hk], v_cache[b, :, hk],
                            scale, tau, bk, num_splits, None if forced is None else forced[b, hk])
            o[b, hk * grp:(hk + 1) * grp] = r.o
            lse[b, hk * grp:(hk + 1) * grp] = r.lse
            retained[b, hk] = r.retained
            margin[b, hk] = r.margin
            overridden[b, hk] = r.overridden
    return {"o": o, "lse": lse, "retained": retained, "margin": margin, "overridden": overridden}


def mala_decode_per_head_bhd(q, k_cache, v_cache, scale, tau, bk, num_splits, batches=None, forced=None):
    """Per-head decode: the skip rule of §2.2 with each query head as its own
    one-row query block, i.e. ``mala_decode`` on each head alone against its
    KV head (same splits, order and merge).  q [B, Hq, d], caches
    [B, N, Hkv, d] -> o [B, Hq, d], lse [B, Hq], retained/margin/overridden
    [B, Hq, T].  ``forced`` [B, Hq, T]: decisions to replay at borderline tiles."""
    bsz, hq, d = q.shape
    n, hkv = k_cache.shape[1], k_cache.shape[2]
    grp = hq // hkv
    t = -(-n // bk)
    o = np.zeros((bsz, hq, v_cache.shape[3]))
    lse = np.full((bsz, hq), np.nan)
    retained = np.zeros((bsz, hq, t), dtype=bool)
    margin = np.full((bsz, hq, t), np.nan)
    overridden = np.zeros((bsz, hq, t), dtype=bool)
    for b in (range(bsz) if batches is None else batches):
        for h in range(hq):
            r = mala_decode(q[b, h:h + 1], k_cache[b, :, h // grp], v_cache[b, :, h // grp],
                            scale, tau, bk, num_splits, None if forced is None else forced[b, h])
            o[b, h] = r.o[0]
            lse[b, h] = r.lse[0]
            retained[b, h] = r.retained
            margin[b, h] = r.margin
            overridden[b, h] = r.overridden
    return {"o": o, "lse": lse, "retained": retained, "margin": margin, "overridden": overridden}


def mala_decode_varlen_bhd(q, k_cache, v_cache, cache_lens, scale, tau, bk, num_splits, batches=None,
                           forced=None):
    """Variable-length decode: sequence b attends to the first cache_lens[b]
    rows of its (padded) cache, which hold its current token, so its L is
    cache_lens[b] (§2.1: L counts the query's own causal context; App. A.1
    for the split-KV decode).  Each sequence is exactly ``mala_decode`` on its
    truncated cache.  retained / margin / overridden are
    [B, Hkv, ceil(N_max / bk)], with tiles past a sequence's own tiles left
    False / NaN.  ``forced`` (same shape): decisions to replay at borderline
    tiles."""
    bsz, hq, d = q.shape
    n_max, hkv = k_cache.shape[1], k_cache.shape[2]
    grp = hq // hkv
    t_max = -(-n_max // bk)
    o = np.zeros((bsz, hq, v_cache.shape[3]))
    lse = np.full((bsz, hq), np.nan)
    retained = np.zeros((bsz, hkv, t_max), dtype=bool)
    margin = np.full((bsz, hkv, t_max), np.nan)
    overridden = np.zeros((bsz, hkv, t_max), dtype=bool)
    for b in (range(bsz) if batches is None else batches):
        n = int(cache_lens[b])
        if not 1 <= n <= n_max:
            raise ValueError(f"cache length {n} of sequence {b} is outside [1, {n_max}]")
        t = -(-n // bk)
        for hk in range(hkv):
            r = mala_decode(q[b, hk * grp:(hk + 1) * grp], k_cache[b, :n, hk], v_cache[b, :n, hk],
                            scale, tau, bk, num_splits, None if forced is None else np.asarray(forced)[b, hk, :t])
            o[b, hk * grp:(hk + 1) * grp] = r.o
            lse[b, hk * grp:(hk + 1) * grp] = r.lse
            retained[b, hk, :t] = r.retained
            margin[b, hk, :t] = r.margin
            overridden[b, hk, :t] = r.overridden
    return {"o": o, "lse": lse, "retained": retained, "margin": margin, "overridden": overridden}


# ---------------------------------------------------------------------------
# Matched-work allocation controls: §3 "Normalized-Mass Allocation at Matched
# Work" (Table 1) and App. C.2.  A decision is one (input, head, query block);
# its candidate regions are the key tiles legal for the block.
# ---------------------------------------------------------------------------

def legal_tiles(n_q, n_k, bq, bk, causal=True):
    """[Tr, Tc] bool: tile (i, j) holds at least one legal (query, key) pair."""
    tr, tc = -(-n_q // bq), -(-n_k // bk)
    legal = np.zeros((tr, tc), dtype=bool)
    for i in range(tr):
        last_row = min(n_q, (i + 1) * bq) - 1
        for j in range(tc):
            legal[i, j] = (not causal) or j * bk <= last_row
    return legal


def tile_reference_mass(q, k, scale, bq, bk, causal=True):
    """Reference mass of every region (App. C.2: the operator with screening
    disabled serves as the reference mass of each candidate region): the
    dense softmax probabilities of tile j's keys summed over the rows of query
    block i.  Returns [Tr, Tc]; illegal tiles have mass 0, and each block's
    masses add up to its number of rows."""
    q, k = _f64(q), _f64(k)
    nq, nk = q.shape[0], k.shape[0]
    s = _scores(q, k, scale, np.arange(nq), np.arange(nk), causal)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    tr, tc = -(-nq // bq), -(-nk // bk)
    mass = np.zeros((tr, tc))
    for i in range(tr):
        for j in range(tc):
            mass[i, j] = p[i * bq:(i + 1) * bq, j * bk:(j + 1) * bk].sum()
    return mass


def matched_work_allocation(counts, scope):
    """Tiles per decision under one of the diagnostic controls of App. C.2.

    counts [I, H, Tr]: the tiles MALA kept for each decision (input i, head h,
    query block).  scope:
      "instance"      - MALA's own count for each decision;
      "head_position" - one allocation per (head, query block), the average
                        over inputs (the paper's layer-head-position control;
                        here there is one layer);
      "position"      - one allocation per query block, the average over
                        inputs and heads.
    A pooled cell's average becomes integers by a rule that looks only at
    indices: every copy of the cell gets floor(average), and the e copies
    x with (x - cell) mod n < e get one more, where n is the number of copies
    and e the cell's remaining units.  So every cell, and the whole, executes
    exactly MALA's total (App. C.2 rounds to integers without looking at the data).
    Copies are numbered input-major: x = i for head_position, i * H + h for
    position; cells are numbered h * Tr + query block, or the query block.
    """
    counts = np.asarray(counts, dtype=np.int64)
    n_in, n_h, tr = counts.shape
    out = np.zeros_like(counts)
    if scope == "instance":
        return counts.copy()
    if scope == "head_position":
        for h in range(n_h):
            for qb in range(tr):
                cell, n = h * tr + qb, n_in
                total = int(sum(counts[i, h, qb] for i in range(n_in)))
                base, extra = total // n, total % n
                for i in range(n_in):
                    out[i, h, qb] = base + (1 if (i - cell) % n < extra else 0)
        return out
    if scope == "position":
        for qb in range(tr):
            cell, n = qb, n_in * n_h
            total = int(sum(counts[i, h, qb] for i in range(n_in) for h in range(n_h)))
            base, extra = total // n, total % n
            for i in range(n_in):
                for h in range(n_h):
                    out[i, h, qb] = base + (1 if (i * n_h + h - cell) % n < extra else 0)
        return out
    raise ValueError(f"unknown scope {scope!r}")


def top_mass_keep(mass, n_keep, legal):
    """The controls' selection (App. C.2: a control keeps the candidate
    regions of largest reference mass): for query block i keep the n_keep[i]
    legal tiles of largest reference mass; equal masses prefer the newer
    (higher) tile.  Returns [Tr, Tc] bool."""
    mass = _f64(mass)
    legal = np.asarray(legal, dtype=bool)
    keep = np.zeros(mass.shape, dtype=bool)
    for i in range(mass.shape[0]):
        cands = sorted((j for j in range(mass.shape[1]) if legal[i, j]), key=lambda j: (-mass[i, j], -j))
        for j in cands[:int(n_keep[i])]:
            keep[i, j] = True
    return keep
