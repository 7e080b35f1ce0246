"""Host-side statistics of the operator-fidelity measurement (§3 Figure 2,
App. C.3), on the CPU."""
import numpy as np
import torch

from mass_adaptive_sparse_gb300 import fidelity as fd, synthetic


def test_relative_errors_closed_form():
    """One head's tensor off by a tenth of itself, another's by a vector of 2%
    of its norm in every row (so 2% of the whole)."""
    B, L, H, D = 2, 7, 3, 5
    ref = torch.randn(B, L, H, D, dtype=torch.float64)
    u = torch.randn(B, L, D, dtype=torch.float64)
    u = u / torch.linalg.vector_norm(u, dim=-1, keepdim=True)
    x = ref.clone()
    x[:, :, 2] += 0.02 * torch.linalg.vector_norm(ref[:, :, 2], dim=-1, keepdim=True) * u
    np.testing.assert_allclose(fd.rel_heads(x, ref).numpy()[:, 2], 0.02, rtol=1e-12)
    y = ref.clone()
    y[:, :, 1] *= 1.1
    np.testing.assert_allclose(fd.rel_heads(y, ref).numpy(), [[0, 0.1, 0]] * B, atol=1e-15, rtol=1e-12)


def test_slots_and_pooling():
    # 3 key blocks of 128 with 1, 2, 3 kept tiles over L = 384 queries: 6 * 128 * 128 / 384 = 256 slots
    kept = torch.tensor([[[1, 2, 3]]])
    np.testing.assert_allclose(fd.slots_per_query(kept, 384, 128).numpy(), [[256.0]])
    states = [{"a": np.array([1.0, 2.0])}, {"a": np.array([3.0])}]
    p = fd.pool(states)
    assert p["a"]["mean"] == 2.0
    assert p["a"]["p95"] == np.percentile([1.0, 2.0, 3.0], 95)


def test_rademacher_probe():
    a = synthetic.rademacher((3, 1000), 5)
    assert set(a.float().unique().tolist()) == {-1.0, 1.0}
    assert torch.equal(a, synthetic.rademacher((3, 1000), 5))
    assert not torch.equal(a, synthetic.rademacher((3, 1000), 6))
    assert abs(float(a.float().mean())) < 0.1
