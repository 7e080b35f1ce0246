"""The parity checks themselves, on the CPU: results made up from the oracle
stand in for a GPU's, and each check must accept a valid result and reject
a plausible wrong one.  The cases use the three-key closed form of the oracle
pins ("MassAlloc Attention", §2.2 Eq. 3 and Algorithm 1), in which a
borderline tile decides whether a later, clearly decided tile is kept."""
import numpy as np
import pytest
import torch

import oracle as orc
from tests import parity
from tests.test_oracle_pins import three_key_case


def _bshd(q, k, v):
    return q[None, :, None], k[None, :, None], v[None, :, None]


def _fake_gpu(q, k, v, tau, mask_row2):
    """O and lse of softmax renormalised over the given tile set (rows 0, 1 as
    the oracle decides them, row 2 as given), and that mask."""
    free = orc.mala_forward(q, k, v, 1.0, tau, 1, 1)
    mask = free.retained.copy()
    mask[2] = mask_row2
    o, lse = orc.restricted_attention(q, k, v, 1.0, mask, 1, 1)
    return o[None, :, None], lse[None, None], mask[None, None].astype(np.uint8)


def _check(o, lse, mask):
    q, k, v, tau = three_key_case()
    ref = orc.mala_forward_bshd(*_bshd(q, k, v), 1.0, tau, 1, 1)
    return parity.check_forward(o, lse, mask, ref, *_bshd(q, k, v), 1.0, tau, 1, torch.float32, True, heads=[0])


def test_forward_check_accepts_the_other_side_of_a_borderline_tile():
    q, k, v, tau = three_key_case()
    m = _check(*_fake_gpu(q, k, v, tau, [True, False, True]))
    assert m["replayed_blocks"] <= 1


def test_forward_check_rejects_a_wrong_decision_after_a_borderline_flip():
    """Key 1 skipped (borderline, allowed), then key 0 skipped too, although
    its ratio is then 0.6, 20% above the threshold.  The output is exactly
    softmax over the tiles kept, so a check that only asked for the first
    disagreement to be borderline and the output to match the kept set would
    pass it."""
    q, k, v, tau = three_key_case()
    o, lse, mask = _fake_gpu(q, k, v, tau, [False, False, True])
    o_r, lse_r = orc.restricted_attention(q, k, v, 1.0, mask[0, 0].astype(bool), 1, 1)
    np.testing.assert_array_equal(o[0, :, 0], o_r)
    with pytest.raises(AssertionError, match="decided differently"):
        _check(o, lse, mask)


def test_forward_check_rejects_a_wrong_decision_at_a_clear_tile():
    q, k, v, tau = three_key_case()
    o, lse, mask = _fake_gpu(q, k, v, tau, [True, False, True])
    mask[0, 0, 1, 0] = 0                        # row 1 skips key 0 (ratio 1.2 against 0.75)
    with pytest.raises(AssertionError, match="decided differently"):
        _check(o, lse, mask)


def test_forward_check_rejects_a_wrong_output_on_the_right_tiles():
    q, k, v, tau = three_key_case()
    o, lse, mask = _fake_gpu(q, k, v, tau, [True, False, True])
    o = o.copy()
    o[0, 2, 0, 0] += 1e-3
    with pytest.raises(AssertionError, match="max abs err"):
        _check(o, lse, mask)


def test_decode_check_replays_and_rejects():
    _, k, v, tau = three_key_case()
    qg = np.ones((1, 1))
    free = orc.mala_decode(qg, k, v, 1.0, tau, 1, 1)
    o, lse, rep = parity.decode_expected([True, False, True], free.o, free.lse, free.retained, qg, k, v, 1.0, tau,
                                         1, 1)
    assert rep and o[0, 0] == pytest.approx(100.6 / 1.6, rel=1e-14)
    with pytest.raises(AssertionError, match="decided differently"):
        parity.decode_expected([False, False, True], free.o, free.lse, free.retained, qg, k, v, 1.0, tau, 1, 1)


def test_backward_check_needs_and_uses_the_replay():
    """One query and one key at the Eq. 4 threshold: a GPU that skipped the
    tile has dV = 0, which only the replay expects."""
    q = v = do = o = np.ones((1, 1, 1, 1))
    k = np.zeros((1, 1, 1, 1))
    lse = np.zeros((1, 1, 1))
    args = (q, k, v, o, do, lse, 1.0, 1.0, 1, 1)
    ref = orc.mala_backward_bshd(*args)
    gpu = {"dq": np.zeros((1, 1, 1, 1)), "dk": np.zeros((1, 1, 1, 1)), "dv": np.zeros((1, 1, 1, 1)),
           "mask": np.zeros((1, 1, 1, 1), np.uint8)}
    if ref["retained"][0, 0, 0, 0]:
        with pytest.raises(AssertionError, match="no replay"):
            parity.check_backward(gpu, ref, 1, True)
    replay = lambda: orc.mala_backward_bshd(*args, forced=gpu["mask"].astype(bool))
    parity.check_backward(gpu, ref, 1, True, replay=replay)
    gpu["dv"] = np.ones((1, 1, 1, 1))           # the kept tile's dV on a skipped tile's mask
    with pytest.raises(AssertionError):
        parity.check_backward(gpu, ref, 1, True, replay=replay)
