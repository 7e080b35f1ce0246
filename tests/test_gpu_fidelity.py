"""GPU run of the operator-fidelity measurement (§3 Figure 2, App. C.3) on a
short cut of the study's inputs: the tensor-core kernels at tau = 1 against
themselves at tau = 0."""
import numpy as np
import pytest

from mass_adaptive_sparse_gb300 import fidelity as fd

pytestmark = pytest.mark.gpu


def test_fidelity_invariants():
    res = fd.study("study_8k", (1024, 2048), 1, 1.0)
    for L, r in res.items():
        dense = (L + 128) / 2                       # causal slots per query with 128-key tiles
        assert 0 < r["fwd_slots"]["mean"] <= dense + 1e-9
        # backward support nested in the forward's (§2.2), so no more work
        assert r["bwd_slots"]["mean"] <= r["fwd_slots"]["mean"] + 1e-9
        # Eq. 6: omitted mass at most tau / (1 + tau) per query
        assert -1e-6 <= r["omitted"]["mean"] <= 0.5
        for n in ("o_err", "dq_err", "dk_err", "dv_err"):
            assert np.isfinite(r[n]["mean"]) and r[n]["p95"] < 0.05, (L, n, r[n])


def test_fidelity_tau0_is_exact():
    """Screening disabled on both sides: the forward is deterministic, so the
    output and lse agree exactly; the gradients agree up to the order of the
    dQ reduce-adds."""
    res = fd.study("study_8k", (1024,), 1, 0.0)[1024]
    assert res["omitted"]["mean"] == 0.0 and res["o_err"]["mean"] == 0.0
    assert res["fwd_slots"]["mean"] == res["bwd_slots"]["mean"] == (1024 + 128) / 2
    assert res["dk_err"]["mean"] <= 1e-6 and res["dv_err"]["mean"] <= 1e-6 and res["dq_err"]["mean"] <= 1e-6
