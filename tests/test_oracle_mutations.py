"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch each one.  Every mutant is built from the oracle's source on the CPU;
the real oracle module is never modified."""
import inspect
import sys
import types

import pytest

import oracle.mala_oracle as real
import tests.test_oracle_pins as pins

SRC = inspect.getsource(real)

# (name, text in the oracle, replacement)
MUTATIONS = [
    ("rescale sign", "alpha[live] = np.exp(m[live] - m_new[live])\n            p = np.zeros_like(s)",
     "alpha[live] = np.exp(m_new[live] - m[live])\n            p = np.zeros_like(s)"),
    ("test sign on log l", "mt - m - np.log(np.where(l > 0, l, 1.0)), np.inf)\n                gap = (ratio - thr)[has]",
     "mt - m + np.log(np.where(l > 0, l, 1.0)), np.inf)\n                gap = (ratio - thr)[has]"),
    ("L_q off by one", "return np.arange(1, n_q + 1, dtype=np.float64)",
     "return np.arange(2, n_q + 2, dtype=np.float64)"),
    ("any instead of all", "gap = (ratio - thr)[has]\n                margin[i, j] = gap.max()\n                skip, overridden[i, j] = _follow(bool(np.all(gap < 0))",
     "gap = (ratio - thr)[has]\n                margin[i, j] = gap.max()\n                skip, overridden[i, j] = _follow(bool(np.any(gap < 0))"),
    ("decode L off by one", "thr = math.log(tau) - math.log(n) if tau > 0 else None",
     "thr = math.log(tau) - math.log(n + 1) if tau > 0 else None"),
    ("ascending forward traversal", "for j in reversed(range(tc)):", "for j in range(tc):"),
    ("dS sign of D", "ds = p * (dp - dd[rows][None, :])", "ds = p * (dp + dd[rows][None, :])"),
    ("dQ drops scale", "dq[rows] += scale * (ds.T @ k[cols])", "dq[rows] += ds.T @ k[cols]"),
    ("dK transposed operand", "dk[cols] += scale * (ds @ q[rows])", "dk[cols] += scale * (p @ q[rows])"),
    ("bwd threshold sign", "gap = (st - lse[rows][None, :] - thr[None, :])[valid]",
     "gap = (st - lse[rows][None, :] + thr[None, :])[valid]"),
    ("decode oldest first", "for j in reversed(range(sp * per, min(t, (sp + 1) * per))):",
     "for j in range(sp * per, min(t, (sp + 1) * per)):"),
    ("merge without rescale", "l = sum(math.exp(mb - m) * lb for mb, lb, _ in live)",
     "l = sum(lb for mb, lb, _ in live)"),
    ("causal mask hides diagonal", "s = np.where(cols[None, :] > rows[:, None], -np.inf, s)",
     "s = np.where(cols[None, :] >= rows[:, None], -np.inf, s)"),
    ("dense D dropped", "ds = p * (dp - dd)", "ds = p * dp"),
    ("lse drops max", "lse[rows] = m + np.log(l)", "lse[rows] = np.log(l)"),
    ("split state carried over", "    for sp in range(num_splits):\n        m = np.full(g, -np.inf)\n        l = np.zeros(g)\n        u = np.zeros((g, vc.shape[1]))\n",
     "    m = np.full(g, -np.inf)\n    l = np.zeros(g)\n    u = np.zeros((g, vc.shape[1]))\n    for sp in range(num_splits):\n"),
    ("region mass transposed", "mass[i, j] = p[i * bq:(i + 1) * bq, j * bk:(j + 1) * bk].sum()",
     "mass[i, j] = p[j * bk:(j + 1) * bk, i * bq:(i + 1) * bq].sum()"),
    ("region mass unnormalised", "    p /= p.sum(axis=1, keepdims=True)\n    tr, tc", "    tr, tc"),
    ("selection keeps lowest mass", "key=lambda j: (-mass[i, j], -j))", "key=lambda j: (mass[i, j], -j))"),
    ("rounding extra by value", "out[i, h, qb] = base + (1 if (i - cell) % n < extra else 0)",
     "out[i, h, qb] = base + (1 if counts[i, h, qb] > base else 0)"),
    ("replay follows every tile", "if forced is None or not is_borderline(margin):", "if forced is None:"),
    ("replay ignores the forced mask", "if forced is None or not is_borderline(margin):", "if True:"),
    ("replay band on the log margin", "return np.isfinite(m) & (np.abs(np.expm1(m)) <= BORDERLINE_REL)",
     "return np.isfinite(m) & (np.abs(m) <= 0.25)"),
    ("position pools one head", "total = int(sum(counts[i, h, qb] for i in range(n_in) for h in range(n_h)))",
     "total = int(sum(counts[i, 0, qb] for i in range(n_in) for h in range(n_h)))"),
]

PIN_TESTS = [
    (pins.test_merge_worked_examples, {}),
    (pins.test_dense_matches_library, {"causal": True}),
    (pins.test_dense_closed_forms, {}),
    (pins.test_dense_grads_match_library_and_finite_differences, {}),
    (pins.test_forward_tau0_is_dense, {"L": 200, "bq": 64}),
    (pins.test_forward_matches_brute_force_ratio_rule, {"tau": 1.0, "b": 16, "seed": 3}),
    (pins.test_forward_bounds_of_appendix_b, {"tau": 1.0, "b": 16}),
    (pins.test_backward_tau0_is_dense_gradient, {"L": 96, "b": 32}),
    (pins.test_backward_brute_force_entry_rule, {}),
    (pins.test_backward_is_gradient_of_forward_when_supports_coincide, {}),
    (pins.test_decode_tau0_is_dense, {"n": 500, "splits": 3}),
    (pins.test_decode_single_split_equals_forward_on_the_head_group, {}),
    (pins.test_uniform_scores_closed_form, {}),
    (pins.test_decode_uniform_scores_closed_form, {}),
    (pins.test_decode_splits_start_from_empty_state_closed_form, {}),
    (pins.test_tile_reference_mass_uniform_scores_closed_form, {"causal": True}),
    (pins.test_tile_reference_mass_blocks_hold_their_rows, {}),
    (pins.test_top_mass_keep_is_the_best_subset_brute_force, {}),
    (pins.test_matched_work_allocation_closed_form, {}),
    (pins.test_matched_work_allocation_matches_work_exactly, {"scope": "head_position"}),
    (pins.test_matched_work_allocation_matches_work_exactly, {"scope": "position"}),
    (pins.test_replay_follows_a_borderline_tile_and_the_later_tests_follow_the_state, {}),
    (pins.test_replay_ignores_forced_decisions_at_tiles_that_are_not_borderline, {}),
    (pins.test_replay_with_the_runs_own_decisions_or_their_complement_is_the_run, {}),
    (pins.test_decode_replay_closed_form, {}),
    (pins.test_backward_replay_follows_only_borderline_tiles, {}),
]


def _mutant(old, new):
    assert SRC.count(old) == 1, old
    mod = types.ModuleType("mala_oracle_mutant")
    sys.modules[mod.__name__] = mod          # dataclasses look the module up by name
    exec(compile(SRC.replace(old, new), "mala_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, monkeypatch):
    mod = _mutant(old, new)
    monkeypatch.setattr(pins, "orc", mod)
    caught = []
    for fn, kw in PIN_TESTS:
        try:
            fn(**kw)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            caught.append(fn.__name__)
    assert caught, f"no pin catches the planted mistake: {name}"
