"""Seeded synthetic inputs for MALA: the planted-peak attention workloads.

This module only draws numbers; it holds none of the attention arithmetic.
Both the CUDA library's callers and the CPU oracle's tests take their inputs
from here.

The generator plants, for each query position i, a few "target" keys drawn
uniformly from its causal prefix [0, i] and sets
    q_i = A * mean(k_targets) + N(0, 1)
so each query row has a few large scores above a Gaussian background.  With
target_rows = G > 1, each group of G consecutive rows shares one draw of
targets (over the group's first row's prefix), which makes the peaks coherent
across a query block.  Per-head amplitudes are drawn from the input's seed, or
from amp_seed when it is set (the same heads for every input).  Two
logit biases are folded into the last head-dim coordinate, because the
operator takes only q, k and v:
    q[..., d-1] = 16,   k[j, d-1] = (sink * [j == 0] + c * j) * sqrt(d) / 16,
which adds  sink * [j == 0] + c * j  to the score of key j under the softmax
scale 1/sqrt(d).  The recency bias -c (i - j) differs from that by the
row-constant -c * i, which changes neither the softmax nor any contribution
test.  Planted terms and noise use coordinates 0 .. d-2.

Large tensors are drawn in fixed-size chunks, each from its own child of the
seed's SeedSequence, on a thread pool; the values do not depend on the number
of threads.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_CHUNK = 1 << 22  # elements per independently seeded chunk


def _normal(seed_seq: np.random.SeedSequence, n: int) -> np.ndarray:
    """n standard normals (float32), drawn chunk-wise in parallel."""
    out = np.empty(n, dtype=np.float32)
    nchunks = -(-n // _CHUNK)
    children = seed_seq.spawn(nchunks)

    def work(c):
        a = c * _CHUNK
        b = min(n, a + _CHUNK)
        np.random.default_rng(children[c]).standard_normal(b - a, dtype=np.float32, out=out[a:b])

    workers = min(32, os.cpu_count() or 1, nchunks)
    if workers <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def rademacher(shape: tuple, seed: int, dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """A deterministic Rademacher probe: independent +-1 entries of `shape`
    from `seed` (exact in every float dtype)."""
    rng = np.random.default_rng(np.random.SeedSequence(seed))
    signs = rng.integers(0, 2, size=int(np.prod(shape)), dtype=np.int8) * 2 - 1
    return torch.from_numpy(signs.astype(np.float32).reshape(shape)).to(dtype)


def _round(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """Round-to-nearest-even into ``dtype`` (torch's conversion)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype)


@dataclass
class PrefillConfig:
    """One prefill (forward + backward) workload."""
    name: str
    B: int
    H: int            # query heads
    Hkv: int          # key/value heads
    L: int
    d: int
    block: int        # B_q = B_k
    dtype: torch.dtype
    n_targets: int
    amplitude: tuple  # one value, or one per head (drawn from this set per head)
    sink: float
    recency: float    # c in the bias -c (i - j)
    taus: tuple = (1.0,)
    seed: int = 0
    target_rows: int = 1          # consecutive query rows that share their target keys
    amp_seed: int | None = None   # draw the per-head amplitudes from this seed (fixed across inputs)


@dataclass
class DecodeConfig:
    """One split-KV decode workload (a single new query per sequence)."""
    name: str
    B: int
    H: int
    Hkv: int
    N: int            # cache length, including the current token
    d: int
    block: int
    num_splits: int
    dtype: torch.dtype
    n_targets: int
    amplitude: float
    taus: tuple = (1.0, 0.0)
    seed: int = 0


# The five workloads: a tiny fp32 case, then 8K, 32K and 128K bf16 prefill,
# then 128K bf16 decode with grouped-query heads (4 query heads per KV head).
CONFIGS = {
    "tiny_fp32": PrefillConfig("tiny_fp32", 1, 2, 2, 256, 64, 64, torch.float32, 3, (4.0,), 3.0, 0.0, (1.0,), 1001),
    "prefill_8k": PrefillConfig("prefill_8k", 1, 16, 16, 8192, 128, 128, torch.bfloat16, 3, (4.0,), 3.0, 0.002, (1.0,), 1002),
    "prefill_32k": PrefillConfig("prefill_32k", 1, 8, 8, 32768, 128, 128, torch.bfloat16, 3, (2.0, 4.0, 8.0), 3.0, 0.002, (1.0, 0.0), 1003),
    "prefill_128k": PrefillConfig("prefill_128k", 1, 8, 8, 131072, 128, 128, torch.bfloat16, 5, (6.0,), 3.0, 1e-4, (1.0, 0.0), 1004),
    # the matched-work study's inputs: 8K tokens, 8 heads of fixed amplitudes 2 / 4 / 8,
    # targets shared by each 128-row query block
    "study_8k": PrefillConfig("study_8k", 1, 8, 8, 8192, 128, 128, torch.bfloat16, 3, (2.0, 4.0, 8.0), 3.0, 0.002,
                              (1.0,), 1006, target_rows=128, amp_seed=1007),
    "decode_128k": DecodeConfig("decode_128k", 8, 32, 8, 131072, 128, 128, 16, torch.bfloat16, 4, 6.0, (1.0, 0.0), 1005),
    # the same cache (same seed) with sharper queries: amplitude 12 on the 4 planted cache rows,
    # used to time the decode's skip path (the 128K decode workload keeps every tile)
    "decode_128k_peaked": DecodeConfig("decode_128k_peaked", 8, 32, 8, 131072, 128, 128, 16, torch.bfloat16, 4,
                                       12.0, (1.0, 0.0), 1005),
}


def _head_amplitudes(rng: np.random.Generator, amplitude: tuple, h: int) -> np.ndarray:
    if len(amplitude) == 1:
        return np.full(h, float(amplitude[0]))
    return rng.choice(np.asarray(amplitude, dtype=np.float64), size=h)


def prefill_inputs(cfg: PrefillConfig, L: int | None = None, seed: int | None = None,
                   with_do: bool = True) -> dict:
    """Planted-peak q, k, v (and dO ~ N(0, 1)) in BSHD layout on the CPU.

    ``L`` overrides the sequence length (same recipe, e.g. for ragged-tail
    cases); ``seed`` overrides the config's seed.
    """
    L = cfg.L if L is None else L
    seed = cfg.seed if seed is None else seed
    B, H, Hkv, d = cfg.B, cfg.H, cfg.Hkv, cfg.d
    ss = np.random.SeedSequence(seed)
    s_k, s_v, s_noise, s_tgt, s_amp, s_do = ss.spawn(6)
    k = _normal(s_k, B * L * Hkv * d).reshape(B, L, Hkv, d)
    v = _normal(s_v, B * L * Hkv * d).reshape(B, L, Hkv, d)
    amp_rng = np.random.default_rng(s_amp if cfg.amp_seed is None else np.random.SeedSequence(cfg.amp_seed))
    amp = _head_amplitudes(amp_rng, cfg.amplitude, H)
    q = _normal(s_noise, B * L * H * d).reshape(B, L, H, d)
    rng_t = np.random.default_rng(s_tgt)
    grp = H // Hkv
    pos = np.arange(L)
    for b in range(B):
        for h in range(H):
            # n_targets keys per query, uniform over the causal prefix [0, i]; a group
            # of target_rows consecutive rows shares one draw over its first row's prefix
            g = cfg.target_rows
            first = pos[::g]
            tgt = np.floor(rng_t.random((len(first), cfg.n_targets)) * (first[:, None] + 1)).astype(np.int64)
            tgt = np.repeat(tgt, g, axis=0)[:L]
            kk = k[b, :, h // grp, : d - 1]
            mean_t = kk[tgt].mean(axis=1)
            q[b, :, h, : d - 1] += (amp[h] * mean_t).astype(np.float32)
    q[..., d - 1] = 16.0
    k[:, :, :, d - 1] = ((cfg.sink * (pos == 0) + cfg.recency * pos) * math.sqrt(d) / 16.0)[None, :, None]
    out = {
        "q": _round(q, cfg.dtype), "k": _round(k, cfg.dtype), "v": _round(v, cfg.dtype),
        "amplitude": amp, "L": L, "seed": seed,
    }
    if with_do:
        out["do"] = _round(_normal(s_do, B * L * H * d).reshape(B, L, H, d), cfg.dtype)
    return out


def decode_inputs(cfg: DecodeConfig, N: int | None = None, B: int | None = None,
                  seed: int | None = None) -> dict:
    """Cache k, v ~ N(0, 1) [B, N, Hkv, d]; each query head
    q = A * mean(4 random cache keys of its KV head) + N(0, 1); q is [B, H, d]."""
    N = cfg.N if N is None else N
    B = cfg.B if B is None else B
    seed = cfg.seed if seed is None else seed
    H, Hkv, d = cfg.H, cfg.Hkv, cfg.d
    ss = np.random.SeedSequence(seed)
    s_k, s_v, s_noise, s_tgt = ss.spawn(4)
    k = _normal(s_k, B * N * Hkv * d).reshape(B, N, Hkv, d)
    v = _normal(s_v, B * N * Hkv * d).reshape(B, N, Hkv, d)
    q = _normal(s_noise, B * H * d).reshape(B, H, d)
    rng_t = np.random.default_rng(s_tgt)
    grp = H // Hkv
    for b in range(B):
        for h in range(H):
            tgt = rng_t.integers(0, N, size=cfg.n_targets)
            q[b, h] += (cfg.amplitude * k[b, tgt, h // grp].mean(axis=0)).astype(np.float32)
    return {"q": _round(q, cfg.dtype), "k": _round(k, cfg.dtype), "v": _round(v, cfg.dtype),
            "N": N, "B": B, "seed": seed}


def decode_query(cfg: DecodeConfig, k: torch.Tensor, seed: int | None = None) -> torch.Tensor:
    """The query recipe of ``decode_inputs`` against a given cache k [B, N, Hkv, d]
    (any float dtype, e.g. one already rounded to bf16): each query head
    q = A * mean(n_targets random cache keys of its KV head) + N(0, 1), with
    the noise and the target rows drawn from the seed exactly as
    ``decode_inputs`` draws them.  Returns q [B, H, d] in cfg.dtype."""
    seed = cfg.seed if seed is None else seed
    B, N, Hkv, d = k.shape
    H = cfg.H
    _, _, s_noise, s_tgt = np.random.SeedSequence(seed).spawn(4)
    q = _normal(s_noise, B * H * d).reshape(B, H, d)
    rng_t = np.random.default_rng(s_tgt)
    grp = H // Hkv
    for b in range(B):
        for h in range(H):
            tgt = rng_t.integers(0, N, size=cfg.n_targets)
            rows = k[b, torch.from_numpy(tgt), h // grp].to(torch.float64).numpy()
            q[b, h] += (cfg.amplitude * rows.mean(axis=0)).astype(np.float32)
    return _round(q, cfg.dtype)
