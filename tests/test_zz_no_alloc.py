"""mala_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a serving process whose device memory all comes from a pool
fixed at start-up, or a plugin host that offers no allocator and no way to
pass scratch space).  It keeps its split records in a fixed array inside the
library instead of a caller workspace.

The check: through the C ABI, two calls in a row (with different inputs, so
the second call runs on an array that still holds the first call's records)
give the same results as mala_decode with a workspace, within the parity
tolerances of the other tests.  This file is collected last on purpose; it
also passes when run alone in a fresh process.
"""
import pytest
import torch

from mass_adaptive_sparse_gb300 import api, synthetic
from tests import parity

pytestmark = pytest.mark.gpu


def _case(seed, N, B, splits, tau):
    cfg = synthetic.CONFIGS["decode_128k"]
    x = synthetic.decode_inputs(cfg, N=N, B=B, seed=seed)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o_ref, lse_ref, ref_info = api.decode(q, k, v, tau, block=128, num_splits=splits, mask=True)
    o = torch.empty_like(q)
    lse = torch.empty((B, q.shape[1]), dtype=torch.float32, device="cuda")
    mask = torch.zeros_like(ref_info["mask"])
    api.mala_decode_noalloc(q, k, v, o, lse, block=128, num_splits=splits, tau=tau, tile_mask=mask)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    return o, lse, mask, o_ref, lse_ref, ref_info["mask"]


def test_noalloc_decode_matches_workspace_decode_twice_in_a_row():
    cap = api.lib().mala_decode_noalloc_max_floats()
    assert cap == 1 << 20
    for seed, N, B, splits, tau in ((31, 5000, 3, 16, 1.0), (32, 2100, 2, 7, 16.0)):
        assert splits * B * 32 * (128 + 4) <= cap
        o, lse, mask, o_ref, lse_ref, mask_ref = _case(seed, N, B, splits, tau)
        assert torch.equal(mask, mask_ref)
        parity.check_close("o", parity.to64(o), parity.to64(o_ref), torch.bfloat16, ref_round=False)
        assert (lse - lse_ref).abs().max().item() <= parity.LSE_ABS


def test_noalloc_decode_rejects_shapes_beyond_its_array():
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((64, 128, 8, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((64, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(api.MalaError) as err:      # 16 * 64 * 32 * 132 floats > 1 Mi floats
        api.mala_decode_noalloc(q, kv, kv, o, lse, block=128, num_splits=16)
    assert err.value.code == 3
