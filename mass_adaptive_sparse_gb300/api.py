"""ctypes binding of libmala.so (declared in include/mala.h).

The raw entry points keep the C names (``mala_fwd``, ``mala_bwd``,
``mala_decode`` ...) and only marshal arguments: shapes are read from the
torch tensors, pointers and the current CUDA stream are passed through, and a
non-OK status raises :class:`MalaError`.  Every step of the computation runs
in the library's CUDA kernels; there is no other implementation behind these
names.  ``forward`` / ``backward`` / ``decode`` allocate outputs and
workspace with torch and call the raw entry points.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# MALA_LIBRARY=debug selects the bounds-checked build (same kernels compiled
# with -DMALA_DEBUG); anything else, or unset, the release build.
LIB_PATH = os.path.join(_HERE, "libmala_debug.so" if os.environ.get("MALA_LIBRARY") == "debug" else "libmala.so")

MALA_BF16, MALA_FP32 = 0, 1
STATUS = {0: "MALA_OK", 1: "MALA_ERR_INVALID_ARG", 2: "MALA_ERR_UNSUPPORTED", 3: "MALA_ERR_WORKSPACE",
          4: "MALA_ERR_CUDA", 5: "MALA_ERR_TIMEOUT"}
EXPORTS = ("mala_status_string", "mala_fwd", "mala_bwd_workspace_size", "mala_bwd",
           "mala_fwd_varlen", "mala_bwd_varlen_workspace_size", "mala_bwd_varlen",
           "mala_decode_workspace_size", "mala_decode", "mala_decode_per_head", "mala_decode_varlen",
           "mala_decode_noalloc", "mala_decode_noalloc_max_floats", "mala_device_status", "mala_launch_count",
           "mala_test_drop_next_load", "mala_last_cuda_error", "mala_cuda_error_string",
           "mala_fwd_forced", "mala_region_mass")


class MalaError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}" + (f" ({detail})" if detail else ""))
        self.code = code


_lib = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """Load libmala.so (built by ``build.py``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} not built ({LIB_PATH}); run "
                               "`python -m mass_adaptive_sparse_gb300.build` first")
        L = ctypes.CDLL(LIB_PATH)
        L.mala_status_string.restype = ctypes.c_char_p
        L.mala_status_string.argtypes = [_i]
        L.mala_fwd.restype = _i
        L.mala_fwd.argtypes = [_vp] * 5 + [_i] * 6 + [_i, _i, _i, _i, _i, _f, _f, _vp, _vp, _vp]
        L.mala_fwd_forced.restype = _i
        L.mala_fwd_forced.argtypes = [_vp] * 5 + [_i] * 6 + [_i, _i, _i, _i, _i, _f, _vp, _vp, _vp, _vp]
        L.mala_region_mass.restype = _i
        L.mala_region_mass.argtypes = [_vp] * 4 + [_i] * 6 + [_i, _i, _i, _i, _f, _vp]
        L.mala_bwd_workspace_size.restype = _sz
        L.mala_bwd_workspace_size.argtypes = [_i] * 8
        L.mala_bwd.restype = _i
        L.mala_bwd.argtypes = [_vp] * 9 + [_i] * 6 + [_i, _i, _i, _i, _i, _f, _f, _vp, _sz, _vp, _vp, _vp]
        L.mala_fwd_varlen.restype = _i
        L.mala_fwd_varlen.argtypes = [_vp] * 6 + [_i] * 6 + [_i, _i, _i, _i, _i, _f, _f, _vp, _vp, _vp]
        L.mala_bwd_varlen_workspace_size.restype = _sz
        L.mala_bwd_varlen_workspace_size.argtypes = [_i] * 6
        L.mala_bwd_varlen.restype = _i
        L.mala_bwd_varlen.argtypes = [_vp] * 10 + [_i] * 6 + [_i, _i, _i, _i, _i, _f, _f, _vp, _sz, _vp, _vp, _vp]
        L.mala_decode_workspace_size.restype = _sz
        L.mala_decode_workspace_size.argtypes = [_i] * 4
        L.mala_decode.restype = _i
        L.mala_decode.argtypes = [_vp] * 5 + [_i] * 5 + [_i, _i, _i, _i, _f, _f, _vp, _sz, _vp, _vp, _vp]
        L.mala_decode_per_head.restype = _i
        L.mala_decode_per_head.argtypes = [_vp] * 5 + [_i] * 5 + [_i, _i, _i, _i, _f, _f, _vp, _sz, _vp, _vp, _vp]
        L.mala_decode_varlen.restype = _i
        L.mala_decode_varlen.argtypes = [_vp] * 6 + [_i] * 9 + [_f, _f, _vp, _sz, _vp, _vp, _vp]
        L.mala_decode_noalloc.restype = _i
        L.mala_decode_noalloc.argtypes = [_vp] * 5 + [_i] * 5 + [_i, _i, _i, _i, _f, _f, _vp, _vp, _vp]
        L.mala_decode_noalloc_max_floats.restype = _sz
        L.mala_decode_noalloc_max_floats.argtypes = []
        L.mala_device_status.restype = _i
        L.mala_device_status.argtypes = [_vp, ctypes.POINTER(_i)]
        L.mala_launch_count.restype = ctypes.c_uint64
        L.mala_launch_count.argtypes = []
        L.mala_test_drop_next_load.restype = None
        L.mala_test_drop_next_load.argtypes = []
        L.mala_last_cuda_error.restype = _i
        L.mala_last_cuda_error.argtypes = []
        L.mala_cuda_error_string.restype = ctypes.c_char_p
        L.mala_cuda_error_string.argtypes = [_i]
        _lib = L
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MALA_BF16
    if t.dtype == torch.float32:
        return MALA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, code: int):
    if code != 0:
        detail = ""
        if code == 4:
            err = lib().mala_last_cuda_error()
            detail = f"cuda error {err}: {lib().mala_cuda_error_string(err).decode()}"
        raise MalaError(fn, code, detail)


def _scale(d, softmax_scale):
    return 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)


# ---------------------------------------------------------------------------
# Raw entry points (same names as the C ABI).
# ---------------------------------------------------------------------------

def mala_fwd(q, k, v, o, lse, *, causal=True, block=128, tau=1.0, softmax_scale=None,
             retained_counts=None, tile_mask=None, stream=None):
    B, Lq, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _check("mala_fwd", lib().mala_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Lq, Lk, Hq, Hkv, D, _dt(q), _dt(o),
        int(causal), block, block, float(tau), _scale(D, softmax_scale),
        _ptr(retained_counts), _ptr(tile_mask), _stream(stream)))


def mala_fwd_forced(q, k, v, o, lse, tile_keep, *, causal=True, block=128, softmax_scale=None,
                    retained_counts=None, tile_mask=None, stream=None):
    """Forward over the tiles `tile_keep` (uint8 [B, Hq, Tr, Tc]) marks, no test."""
    B, Lq, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    if tile_keep.dtype != torch.uint8 or tile_keep.shape != (B, Hq, -(-Lq // block), -(-Lk // block)):
        raise ValueError("tile_keep must be uint8 [B, Hq, ceil(Lq / block), ceil(Lk / block)]")
    _check("mala_fwd_forced", lib().mala_fwd_forced(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Lq, Lk, Hq, Hkv, D, _dt(q), _dt(o),
        int(causal), block, block, _scale(D, softmax_scale), _ptr(tile_keep),
        _ptr(retained_counts), _ptr(tile_mask), _stream(stream)))


def mala_region_mass(q, k, lse, region_mass, *, causal=True, block=128, softmax_scale=None, stream=None):
    """region_mass (fp32 [B, Hq, Tr, Tc]) = each (query block, key tile) region's
    softmax mass under the row log-normalisers `lse`, summed over the block's rows."""
    B, Lq, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    if region_mass.dtype != torch.float32 or region_mass.shape != (B, Hq, -(-Lq // block), -(-Lk // block)):
        raise ValueError("region_mass must be float32 [B, Hq, ceil(Lq / block), ceil(Lk / block)]")
    _check("mala_region_mass", lib().mala_region_mass(
        _ptr(q), _ptr(k), _ptr(lse), _ptr(region_mass), B, Lq, Lk, Hq, Hkv, D, _dt(q), int(causal),
        block, block, _scale(D, softmax_scale), _stream(stream)))


def mala_bwd_workspace_size(q, k, grad_dtype):
    B, Lq, Hq, D = q.shape
    return lib().mala_bwd_workspace_size(B, Lq, k.shape[1], Hq, k.shape[2], D, _dt(q),
                                         MALA_BF16 if grad_dtype == torch.bfloat16 else MALA_FP32)


def mala_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, *, causal=True, block=128, tau=1.0,
             softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    B, Lq, Hq, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _check("mala_bwd", lib().mala_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        B, Lq, Lk, Hq, Hkv, D, _dt(q), _dt(dq), int(causal), block, block, float(tau),
        _scale(D, softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(retained_counts), _ptr(tile_mask), _stream(stream)))


def _check_cu(cu_seqlens, batch):
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.shape != (batch + 1,) or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be an int32 CUDA tensor of shape [batch + 1]")


def mala_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, *, causal=True, block=128, tau=1.0,
                    softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    """Packed variable-length forward: q, o [total, Hq, D], k, v [total, Hkv, D],
    lse [Hq, total]; sequence b is rows cu_seqlens[b] .. cu_seqlens[b + 1] - 1."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.shape[0] - 1
    _check_cu(cu_seqlens, B)
    _check("mala_fwd_varlen", lib().mala_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), B, T, int(max_seqlen), Hq, Hkv, D,
        _dt(q), _dt(o), int(causal), block, block, float(tau), _scale(D, softmax_scale),
        _ptr(retained_counts), _ptr(tile_mask), _stream(stream)))


def mala_bwd_varlen_workspace_size(q, k, grad_dtype):
    T, Hq, D = q.shape
    return lib().mala_bwd_varlen_workspace_size(T, Hq, k.shape[1], D, _dt(q),
                                                MALA_BF16 if grad_dtype == torch.bfloat16 else MALA_FP32)


def mala_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens, max_seqlen, workspace, *, causal=True,
                    block=128, tau=1.0, softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    """Packed variable-length backward (layouts as mala_fwd_varlen)."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.shape[0] - 1
    _check_cu(cu_seqlens, B)
    _check("mala_bwd_varlen", lib().mala_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens),
        B, T, int(max_seqlen), Hq, Hkv, D, _dt(q), _dt(dq), int(causal), block, block, float(tau),
        _scale(D, softmax_scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(retained_counts), _ptr(tile_mask), _stream(stream)))


def mala_decode_workspace_size(B, Hq, D, num_splits):
    return lib().mala_decode_workspace_size(B, Hq, D, num_splits)


def mala_decode(q, k_cache, v_cache, o, lse, workspace, *, block=128, num_splits=16, tau=1.0,
                softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    B, Hq, D = q.shape
    N, Hkv = k_cache.shape[1], k_cache.shape[2]
    _check("mala_decode", lib().mala_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, N, Hq, Hkv, D, _dt(q), _dt(o),
        block, num_splits, float(tau), _scale(D, softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(retained_counts), _ptr(tile_mask),
        _stream(stream)))


def mala_decode_per_head(q, k_cache, v_cache, o, lse, workspace, *, block=128, num_splits=16, tau=1.0,
                         softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    """mala_decode with each query head deciding alone; counts / mask per query head."""
    B, Hq, D = q.shape
    N, Hkv = k_cache.shape[1], k_cache.shape[2]
    _check("mala_decode_per_head", lib().mala_decode_per_head(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, N, Hq, Hkv, D, _dt(q), _dt(o),
        block, num_splits, float(tau), _scale(D, softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(retained_counts), _ptr(tile_mask),
        _stream(stream)))


def mala_decode_varlen(q, k_cache, v_cache, o, lse, cache_lens, workspace, *, block=128, num_splits=16,
                       tau=1.0, softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    """mala_decode with per-sequence cache lengths (int32 CUDA tensor [B]) over
    caches padded to k_cache.shape[1]."""
    B, Hq, D = q.shape
    N, Hkv = k_cache.shape[1], k_cache.shape[2]
    if cache_lens.dtype != torch.int32 or cache_lens.shape != (B,):
        raise ValueError("cache_lens must be an int32 tensor of shape [B]")
    _check("mala_decode_varlen", lib().mala_decode_varlen(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), _ptr(cache_lens), B, N, Hq, Hkv, D,
        _dt(q), _dt(o), block, num_splits, float(tau), _scale(D, softmax_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(retained_counts), _ptr(tile_mask),
        _stream(stream)))


def mala_decode_noalloc(q, k_cache, v_cache, o, lse, *, block=128, num_splits=16, tau=1.0,
                        softmax_scale=None, retained_counts=None, tile_mask=None, stream=None):
    """mala_decode with the split records in the library's fixed device array
    (for callers that cannot allocate; see include/mala.h)."""
    B, Hq, D = q.shape
    N, Hkv = k_cache.shape[1], k_cache.shape[2]
    _check("mala_decode_noalloc", lib().mala_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, N, Hq, Hkv, D, _dt(q), _dt(o),
        block, num_splits, float(tau), _scale(D, softmax_scale), _ptr(retained_counts), _ptr(tile_mask),
        _stream(stream)))


def mala_device_status(stream=None) -> int:
    code = _i(0)
    rc = lib().mala_device_status(_stream(stream), ctypes.byref(code))
    if rc not in (0, 1, 5):     # OK, a rejected sequence length, an expired wait
        raise MalaError("mala_device_status", rc)
    return code.value


def mala_test_drop_next_load():
    """Failure-detection test hook: the next tensor-core forward call has one
    CTA's bounded waits expire (see include/mala.h)."""
    lib().mala_test_drop_next_load()


def mala_launch_count() -> int:
    return int(lib().mala_launch_count())


# ---------------------------------------------------------------------------
# Allocating conveniences.
# ---------------------------------------------------------------------------

def _ntiles(n, b):
    return -(-n // b)


def forward(q, k, v, tau=1.0, *, causal=True, block=128, softmax_scale=None, out_dtype=None,
            counts=False, mask=False, stream=None):
    """Returns (o, lse, info) with info holding 'counts' / 'mask' when asked."""
    B, Lq, Hq, D = q.shape
    o = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    tr, tc = _ntiles(Lq, block), _ntiles(k.shape[1], block)
    info = {}
    if counts:
        info["counts"] = torch.zeros((B, Hq, tr), dtype=torch.int32, device=q.device)
    if mask:
        info["mask"] = torch.zeros((B, Hq, tr, tc), dtype=torch.uint8, device=q.device)
    mala_fwd(q, k, v, o, lse, causal=causal, block=block, tau=tau, softmax_scale=softmax_scale,
             retained_counts=info.get("counts"), tile_mask=info.get("mask"), stream=stream)
    return o, lse, info


def backward(q, k, v, o, do, lse, tau=1.0, *, causal=True, block=128, softmax_scale=None,
             grad_dtype=torch.float32, counts=False, mask=False, stream=None):
    """Returns (dq, dk, dv, info)."""
    B, Lq, Hq, D = q.shape
    dev = q.device
    dq = torch.empty(q.shape, dtype=grad_dtype, device=dev)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=dev)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=dev)
    ws = torch.empty(max(256, mala_bwd_workspace_size(q, k, grad_dtype)), dtype=torch.uint8, device=dev)
    tr, tc = _ntiles(Lq, block), _ntiles(k.shape[1], block)
    info = {}
    if counts:
        info["counts"] = torch.zeros((B, Hq, tc), dtype=torch.int32, device=dev)
    if mask:
        info["mask"] = torch.zeros((B, Hq, tr, tc), dtype=torch.uint8, device=dev)
    mala_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, causal=causal, block=block, tau=tau,
             softmax_scale=softmax_scale, retained_counts=info.get("counts"),
             tile_mask=info.get("mask"), stream=stream)
    return dq, dk, dv, info


def forward_varlen(q, k, v, cu_seqlens, max_seqlen, tau=1.0, *, causal=True, block=128, softmax_scale=None,
                   out_dtype=None, counts=False, mask=False, stream=None):
    """Packed variable-length forward; returns (o [total, Hq, D], lse [Hq, total], info)."""
    T, Hq, D = q.shape
    B = cu_seqlens.shape[0] - 1
    o = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    t = _ntiles(max_seqlen, block)
    info = {}
    if counts:
        info["counts"] = torch.zeros((B, Hq, t), dtype=torch.int32, device=q.device)
    if mask:
        info["mask"] = torch.zeros((B, Hq, t, t), dtype=torch.uint8, device=q.device)
    mala_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, causal=causal, block=block, tau=tau,
                    softmax_scale=softmax_scale, retained_counts=info.get("counts"), tile_mask=info.get("mask"),
                    stream=stream)
    return o, lse, info


def backward_varlen(q, k, v, o, do, lse, cu_seqlens, max_seqlen, tau=1.0, *, causal=True, block=128,
                    softmax_scale=None, grad_dtype=torch.float32, counts=False, mask=False, stream=None):
    """Packed variable-length backward; returns (dq, dk, dv, info)."""
    T, Hq, D = q.shape
    B = cu_seqlens.shape[0] - 1
    dev = q.device
    dq = torch.empty(q.shape, dtype=grad_dtype, device=dev)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=dev)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=dev)
    ws = torch.empty(max(256, mala_bwd_varlen_workspace_size(q, k, grad_dtype)), dtype=torch.uint8, device=dev)
    t = _ntiles(max_seqlen, block)
    info = {}
    if counts:
        info["counts"] = torch.zeros((B, Hq, t), dtype=torch.int32, device=dev)
    if mask:
        info["mask"] = torch.zeros((B, Hq, t, t), dtype=torch.uint8, device=dev)
    mala_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_seqlens, max_seqlen, ws, causal=causal, block=block,
                    tau=tau, softmax_scale=softmax_scale, retained_counts=info.get("counts"),
                    tile_mask=info.get("mask"), stream=stream)
    return dq, dk, dv, info


def decode(q, k_cache, v_cache, tau=1.0, *, block=128, num_splits=16, softmax_scale=None,
           out_dtype=None, counts=False, mask=False, cache_lens=None, per_head=False, stream=None):
    """Returns (o, lse, info).  `cache_lens` (int32 CUDA tensor [B]) selects
    the variable-length decode over caches padded to k_cache.shape[1];
    `per_head` lets each query head decide alone (counts / mask per query head)."""
    B, Hq, D = q.shape
    N, Hkv = k_cache.shape[1], k_cache.shape[2]
    dev = q.device
    o = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, mala_decode_workspace_size(B, Hq, D, num_splits)), dtype=torch.uint8, device=dev)
    info = {}
    if per_head and cache_lens is not None:
        raise ValueError("per_head and cache_lens are separate entry points")
    rows = Hq if per_head else Hkv
    if counts:
        info["counts"] = torch.zeros((B, rows, num_splits), dtype=torch.int32, device=dev)
    if mask:
        info["mask"] = torch.zeros((B, rows, _ntiles(N, block)), dtype=torch.uint8, device=dev)
    if per_head:
        mala_decode_per_head(q, k_cache, v_cache, o, lse, ws, block=block, num_splits=num_splits, tau=tau,
                             softmax_scale=softmax_scale, retained_counts=info.get("counts"),
                             tile_mask=info.get("mask"), stream=stream)
    elif cache_lens is None:
        mala_decode(q, k_cache, v_cache, o, lse, ws, block=block, num_splits=num_splits, tau=tau,
                    softmax_scale=softmax_scale, retained_counts=info.get("counts"),
                    tile_mask=info.get("mask"), stream=stream)
    else:
        mala_decode_varlen(q, k_cache, v_cache, o, lse, cache_lens, ws, block=block, num_splits=num_splits,
                           tau=tau, softmax_scale=softmax_scale, retained_counts=info.get("counts"),
                           tile_mask=info.get("mask"), stream=stream)
    return o, lse, info
