"""GPU parity of mala_fwd / mala_bwd against the fp64 oracle, through the C ABI.

Small cases are compared element by element (several tiles, ragged tails,
GQA, batch 2, non-causal with Lq != Lk, bf16 gradients, fp32 output from bf16
inputs, tau in {0, 1, 4, 64, 1e30}); the 8K, 32K and 128K workloads run at full size
in the launch configuration the benchmark times and are compared on sampled
heads and query / key blocks, which the oracle computes exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from mass_adaptive_sparse_gb300 import api, synthetic
from tests import parity

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(cfg, L=None, seed=None, heads=None, hkv=None, lk=None):
    """The recipe's q, k, v, dO; `lk` (non-causal cases) keeps the first L query
    rows and the first lk key rows of a sequence as long as the longer of them."""
    x = synthetic.prefill_inputs(cfg, L=L if lk is None else max(L, lk), seed=seed)
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    if heads is not None:
        q, do = q[:, :, :heads].contiguous(), do[:, :, :heads].contiguous()
        k, v = k[:, :, :hkv].contiguous(), v[:, :, :hkv].contiguous()
    if lk is not None:
        q, do = q[:, :L].contiguous(), do[:, :L].contiguous()
        k, v = k[:, :lk].contiguous(), v[:, :lk].contiguous()
    return q, k, v, do


def _gpu(*ts):
    return [t.to(DEV) for t in ts]


def _oracle_bwd_inputs(ref_fwd, gpu_o, gpu_lse, heads, blocks, block, dtype):
    """Backward inputs: oracle O (rounded to the GPU dtype) and lse (fp32) on
    the sampled (head, query block) rows, the GPU's own forward elsewhere."""
    o_in = gpu_o.clone()
    lse_in = gpu_lse.clone()
    L = gpu_o.shape[1]
    for h in heads:
        for i in blocks:
            r0, r1 = i * block, min(L, (i + 1) * block)
            o_in[:, r0:r1, h] = torch.from_numpy(ref_fwd["o"][:, r0:r1, h]).to(dtype).to(DEV)
            lse_in[:, h, r0:r1] = torch.from_numpy(ref_fwd["lse"][:, h, r0:r1]).float().to(DEV)
    return o_in, lse_in


def _run_case(cfg, L, tau, seed, heads=None, hkv=None, block=None, fp32=None, grad=True,
              q_blocks=None, dq_blocks=None, dk_blocks=None, ref_heads=None, causal=True, lk=None,
              grad_dtype=torch.float32, out_dtype=None):
    block = block or cfg.block
    q, k, v, do = _inputs(cfg, L=L, seed=seed, heads=heads, hkv=hkv, lk=lk)
    fp32 = (q.dtype == torch.float32) if fp32 is None else fp32
    d = q.shape[3]
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dod = _gpu(q, k, v, do)
    o, lse, info = api.forward(qd, kd, vd, tau, causal=causal, block=block, out_dtype=out_dtype,
                               counts=True, mask=True)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    q64, k64, v64, do64 = (parity.to64(t) for t in (q, k, v, do))
    H = q.shape[2]
    ref_heads = list(range(H)) if ref_heads is None else ref_heads
    tr, tc = -(-L // block), -(-k.shape[1] // block)
    fwd_blocks = q_blocks if q_blocks is not None else list(range(tr))
    if dq_blocks is not None:
        fwd_blocks = sorted(set(fwd_blocks) | set(dq_blocks) | {i for i in range(tr) if i >= min(dk_blocks)})
    ref = orc.mala_forward_bshd(q64, k64, v64, scale, tau, block, block, causal=causal, heads=ref_heads,
                                query_blocks=fwd_blocks)
    gpu_o, gpu_lse, gpu_mask = parity.to64(o), parity.to64(lse), info["mask"].cpu().numpy()
    metrics = parity.check_forward(gpu_o, gpu_lse, gpu_mask, ref, q64, k64, v64, scale, tau, block, o.dtype,
                                   fp32, heads=ref_heads, causal=causal, blocks=q_blocks)
    counts = info["counts"].cpu().numpy()
    legal_gpu = np.tril(np.ones((tr, tc), bool)) if causal else np.ones((tr, tc), bool)
    np.testing.assert_array_equal(counts, (gpu_mask.astype(bool) & legal_gpu).sum(-1))
    if not grad:
        return metrics
    if dq_blocks is None:
        o_in, lse_in = _oracle_bwd_inputs(ref, o, lse, ref_heads, range(tr), block, q.dtype)
        tiles = None
    else:
        o_in, lse_in = _oracle_bwd_inputs(ref, o, lse, ref_heads, fwd_blocks, block, q.dtype)
        tiles = lambda i, j: i in dq_blocks or j in dk_blocks
    dq, dk, dv, binfo = api.backward(qd, kd, vd, o_in, dod, lse_in, tau, causal=causal, block=block,
                                     grad_dtype=grad_dtype, counts=True, mask=True)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    o_in64, lse_in64 = parity.to64(o_in), parity.to64(lse_in)
    refb = orc.mala_backward_bshd(q64, k64, v64, o_in64, do64, lse_in64, scale, tau, block, block,
                                  causal=causal, heads=ref_heads, tiles=tiles)
    gpu_b = {"dq": parity.to64(dq), "dk": parity.to64(dk), "dv": parity.to64(dv),
             "mask": binfo["mask"].cpu().numpy()}
    # compare only the sampled heads (and KV heads whose every query head is sampled)
    grp = H // k.shape[2]
    full_kv = [hk for hk in range(k.shape[2]) if all(h in ref_heads for h in range(hk * grp, (hk + 1) * grp))]
    dq_rows = np.zeros(q.shape[:3], bool)
    dk_rows = np.zeros(k.shape[:3], bool)
    for h in ref_heads:
        if dq_blocks is None:
            dq_rows[:, :, h] = True
        else:
            for i in dq_blocks:
                dq_rows[:, i * block:(i + 1) * block, h] = True
    for hk in full_kv:
        if dk_blocks is None:
            dk_rows[:, :, hk] = True
        else:
            for j in dk_blocks:
                dk_rows[:, j * block:(j + 1) * block, hk] = True
    sel_legal = refb["legal"].copy()
    gmask = gpu_b["mask"].copy()
    for h in range(H):
        if h not in ref_heads:
            sel_legal[:, h] = False
    refb_cmp = dict(refb, legal=sel_legal)

    def replay():
        r = orc.mala_backward_bshd(q64, k64, v64, o_in64, do64, lse_in64, scale, tau, block, block,
                                   causal=causal, heads=ref_heads, tiles=tiles, forced=gmask.astype(bool))
        return dict(r, legal=sel_legal)

    bm = parity.check_backward(gpu_b, refb_cmp, block, fp32, dq_rows=dq_rows, dk_rows=dk_rows,
                               grad_dtype=grad_dtype, replay=replay)
    # backward support is nested in the forward support on oracle-fed rows (MALA §2.2)
    assert not (refb["retained"] & ~ref["retained"] & sel_legal).any()
    np.testing.assert_array_equal(binfo["counts"].cpu().numpy(), (gmask.astype(bool) & legal_gpu).sum(-2))
    metrics["bwd"] = bm
    return metrics


def test_tiny_fp32_workload():
    """B=1, H=2, L=256, d=64, 64x64 tiles, tau=1, fp32: the full case."""
    cfg = synthetic.CONFIGS["tiny_fp32"]
    m = _run_case(cfg, cfg.L, 1.0, cfg.seed)
    assert m["max_abs"] <= parity.FP32_MAX_ABS


@pytest.mark.parametrize("tau", [0.0, 4.0, 64.0, 1e30])
@pytest.mark.parametrize("L", [256, 200])
def test_tiny_fp32_tau_and_ragged(tau, L):
    cfg = synthetic.CONFIGS["tiny_fp32"]
    _run_case(cfg, L, tau, cfg.seed + 7)


@pytest.mark.parametrize("block", [64, 128])
@pytest.mark.parametrize("L,tau", [(1000, 1.0), (777, 4.0), (1024, 0.0), (640, 1e30)])
def test_bf16_small_cases(block, L, tau):
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run_case(cfg, L, tau, 17, heads=2, hkv=2, block=block)


def test_bf16_gqa_small():
    cfg = synthetic.PrefillConfig("gqa", 1, 4, 2, 600, 128, 128, torch.bfloat16, 3, (4.0,), 3.0, 0.01)
    _run_case(cfg, 600, 1.0, 23, block=128)


def test_bf16_batch2_gqa():
    """Two sequences, 8 query heads over 2 KV heads (group 4), ragged length."""
    cfg = synthetic.PrefillConfig("b2gqa", 2, 8, 2, 700, 128, 128, torch.bfloat16, 3, (4.0,), 3.0, 0.01)
    _run_case(cfg, 700, 1.0, 43, block=128)


def test_bf16_gqa_group_of_8():
    """16 query heads over 2 KV heads (group 8, the paper's model shares each KV
    head among 8 query heads), ragged length, tau = 1 and 4."""
    cfg = synthetic.PrefillConfig("gqa8", 1, 16, 2, 900, 128, 128, torch.bfloat16, 3, (4.0,), 3.0, 0.01)
    for tau in (1.0, 4.0):
        _run_case(cfg, 900, tau, 53, block=128)


@pytest.mark.parametrize("L,lk", [(300, 700), (640, 256)])
@pytest.mark.parametrize("tau", [1.0, 64.0])
def test_bf16_noncausal(L, lk, tau):
    """causal = 0: every key visible to every query, L_q = Lk, Lq != Lk."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run_case(cfg, L, tau, 37, heads=2, hkv=2, block=128, causal=False, lk=lk)


@pytest.mark.parametrize("tau", [1.0, 0.0])
def test_bf16_gradients_in_bf16(tau):
    """grad dtype bf16: the fp32 dQ accumulator in the workspace, then a
    conversion; compared with the oracle rounded to bf16."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run_case(cfg, 600, tau, 31, heads=2, hkv=2, block=128, grad_dtype=torch.bfloat16)


def test_fp32_output_from_bf16_inputs():
    """out dtype fp32 for bf16 q, k, v (forward only: the backward takes O in the input dtype)."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run_case(cfg, 1000, 1.0, 47, heads=2, hkv=2, block=128, out_dtype=torch.float32, grad=False)


def test_fp32_d128_block64():
    cfg = synthetic.PrefillConfig("f32d128", 1, 2, 2, 300, 128, 64, torch.float32, 3, (4.0,), 3.0, 0.05)
    _run_case(cfg, 300, 1.0, 29, block=64)


def test_prefill_8k_full_size():
    """All 16 heads run; heads 0, 5, 9 and 15 are compared element by element."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    _run_case(cfg, cfg.L, 1.0, cfg.seed, ref_heads=[0, 5, 9, 15])


@pytest.mark.parametrize("tau", [1.0, 0.0])
def test_prefill_32k_sampled(tau):
    """All 8 heads at full size; query blocks at both ends and the middle, dQ
    at both ends, dK / dV of the last two key blocks."""
    cfg = synthetic.CONFIGS["prefill_32k"]
    tr = cfg.L // cfg.block
    _run_case(cfg, cfg.L, tau, cfg.seed, ref_heads=list(range(cfg.H)), q_blocks=[0, 1, tr // 2, tr - 2, tr - 1],
              dq_blocks=[0, 2, tr - 1], dk_blocks=[tr - 2, tr - 1])


def test_prefill_32k_first_key_block_gradients():
    """dK / dV of key block 0 (every query row of the sequence contributes, so
    the oracle runs the whole forward of the head to give the backward its O
    and lse) and dQ of the last query block, on head 0."""
    cfg = synthetic.CONFIGS["prefill_32k"]
    tr = cfg.L // cfg.block
    _run_case(cfg, cfg.L, 1.0, cfg.seed, ref_heads=[0], q_blocks=[tr - 1], dq_blocks=[tr - 1], dk_blocks=[0])


@pytest.mark.parametrize("tau", [1.0, 0.0])
def test_prefill_128k_sampled(tau):
    """All 8 heads at full size, tau = 1 and the dense tau = 0 that the
    benchmark times beside it: query blocks {0, 1, 511, 1022, 1023}; dQ of
    query blocks 1 and 1022; dK / dV of the last two key blocks."""
    cfg = synthetic.CONFIGS["prefill_128k"]
    tr = cfg.L // cfg.block
    _run_case(cfg, cfg.L, tau, cfg.seed, ref_heads=list(range(cfg.H)), q_blocks=[0, 1, tr // 2 - 1, tr - 2, tr - 1],
              dq_blocks=[1, tr - 2], dk_blocks=[tr - 2, tr - 1])


def test_bf16_input_beyond_fp16_range_is_reported():
    """The tensor-core backward takes fp16 operands: a finite bf16 input beyond
    65504 sets bit 4 of the device status word; 65280, the largest bf16 value
    below it, does not."""
    cfg = synthetic.CONFIGS["prefill_8k"]
    q, k, v, do = _gpu(*_inputs(cfg, L=256, seed=5, heads=2, hkv=2))
    o, lse, _ = api.forward(q, k, v, 1.0)
    torch.cuda.synchronize()
    assert api.mala_device_status() == 0
    for name, val, want in (("v", 65280.0, 0), ("v", 70000.0, 4), ("do", -1.0e5, 4), ("q", 3.0e38, 4)):
        args = {"q": q, "k": k, "v": v, "do": do}
        t = args[name].clone()
        t[0, 3, 1, 5] = val
        args[name] = t
        api.backward(args["q"], args["k"], args["v"], o, args["do"], lse, 1.0)
        torch.cuda.synchronize()
        assert api.mala_device_status() == want, (name, val)
    assert api.mala_device_status() == 0
