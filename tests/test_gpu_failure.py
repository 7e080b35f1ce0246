"""Failure detection on the GPU, without a fault: a forward call in which one
CTA never receives its first K tile has that CTA's bounded waits expire.  The
call returns, the device status word reports the expired wait
(MALA_ERR_TIMEOUT), and the next call on the same context is correct."""
import math
import time

import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import api, synthetic
from tests import parity

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_stays_usable():
    cfg = synthetic.CONFIGS["prefill_8k"]
    x = synthetic.prefill_inputs(cfg, L=1024, seed=91)
    q, k, v = (x[n][:, :, :2].contiguous() for n in ("q", "k", "v"))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert api.mala_device_status() == 0
    api.mala_test_drop_next_load()
    t0 = time.monotonic()
    api.forward(qd, kd, vd, 1.0)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    code = api.mala_device_status()
    assert code & 1, f"status word {code}: the expired wait was not reported"
    assert elapsed < 60
    assert api.mala_device_status() == 0          # reading clears the word
    # the hook is one-shot: the next call runs normally on the same context
    o, lse, info = api.forward(qd, kd, vd, 1.0, mask=True)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    q64, k64, v64 = (parity.to64(t) for t in (q, k, v))
    scale = 1 / math.sqrt(128)
    ref = orc.mala_forward_bshd(q64, k64, v64, scale, 1.0, 128, 128)
    parity.check_forward(parity.to64(o), parity.to64(lse), info["mask"].cpu().numpy(), ref, q64, k64, v64,
                         scale, 1.0, 128, o.dtype, False, heads=[0, 1])
