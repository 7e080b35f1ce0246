"""Host-side checks of libmala.so: it loads, exports every entry point that
include/mala.h declares, and rejects bad arguments before touching the GPU.
No compute call is made (these run without a GPU)."""
import ctypes
import os
import re

import pytest

from mass_adaptive_sparse_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mala.h")


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mala_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(api.LIB_PATH):
        from mass_adaptive_sparse_gb300 import build
        build.build()
    return api.lib()


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert {"mala_fwd", "mala_bwd", "mala_decode"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in mala.h but not exported"
    assert set(names) == set(api.EXPORTS)


def test_bounds_checked_build_exports_the_same_symbols():
    """libmala_debug.so (the -DMALA_DEBUG build) is a drop-in for libmala.so."""
    from mass_adaptive_sparse_gb300 import build
    if not os.path.exists(build.LIB_DEBUG):
        build.build(variants=("debug",))
    dbg = ctypes.CDLL(build.LIB_DEBUG)
    for n in declared_entry_points():
        assert hasattr(dbg, n), f"{n} not exported by libmala_debug.so"


def test_status_strings(lib):
    for code, name in api.STATUS.items():
        assert lib.mala_status_string(code).decode() == name
    assert lib.mala_status_string(99).decode() == "MALA_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    B, L, H, D = 1, 8192, 16, 128
    ws_f32 = lib.mala_bwd_workspace_size(B, L, L, H, H, D, 0, 1)
    ws_bf16 = lib.mala_bwd_workspace_size(B, L, L, H, H, D, 0, 0)
    assert ws_f32 >= B * L * H * 4 and ws_f32 % 256 == 0
    assert ws_bf16 >= ws_f32 + B * L * H * D * 4
    assert lib.mala_bwd_workspace_size(0, L, L, H, H, D, 0, 1) == 0
    dec = lib.mala_decode_workspace_size(8, 32, 128, 16)
    assert dec >= 16 * 8 * 32 * 132 * 4 and dec % 256 == 0
    assert lib.mala_decode_workspace_size(8, 32, 128, 0) == 0


FAKE = ctypes.c_void_p(0x10000)        # aligned, never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def _fwd(lib, q=FAKE, B=1, L=256, Hq=2, Hkv=2, D=64, dt=1, causal=1, bq=64, bk=64, tau=1.0, scale=0.125, Lk=None):
    return lib.mala_fwd(q, FAKE, FAKE, FAKE, FAKE, B, L, L if Lk is None else Lk, Hq, Hkv, D, dt, dt,
                        causal, bq, bk, tau, scale, None, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(q=MISALIGNED), 1), (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1),
    (dict(dt=7), 1), (dict(causal=2), 1), (dict(Lk=300), 1), (dict(tau=-1.0), 1),
    (dict(tau=float("nan")), 1), (dict(tau=float("inf")), 1), (dict(scale=0.0), 1),
    (dict(D=96), 2), (dict(bq=64, bk=128), 2), (dict(bq=32, bk=32), 2),
    # more CTAs (batch x heads x tiles) than 32-bit CTA numbering holds
    (dict(B=65535, Hq=65535, Hkv=65535, L=128, bq=64, bk=64), 2),
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert _fwd(lib, **kw) == code


def test_bwd_rejects_small_workspace(lib):
    args = [FAKE] * 9 + [1, 256, 256, 2, 2, 64, 1, 1, 1, 64, 64, 1.0, 0.125]
    assert lib.mala_bwd(*args, None, 1 << 20, None, None, None) == 3
    assert lib.mala_bwd(*args, FAKE, 16, None, None, None) == 3
    assert lib.mala_bwd(*args, ctypes.c_void_p(0x10010), 1 << 20, None, None, None) == 3
    assert lib.mala_bwd(*([None] + args[1:]), FAKE, 1 << 20, None, None, None) == 1


def _bwd(lib, ptr=None, ptr_at=None, B=1, L=256, Hq=2, Hkv=2, D=64, dt=1, gdt=1, causal=1, blk=64, tau=1.0,
         scale=0.125, ws=FAKE, ws_bytes=1 << 30):
    ptrs = [FAKE] * 9                  # q, k, v, o, dO, lse, dQ, dK, dV
    if ptr_at is not None:
        ptrs[ptr_at] = ptr
    return lib.mala_bwd(*ptrs, B, L, L, Hq, Hkv, D, dt, gdt, causal, blk, blk, tau, scale, ws, ws_bytes,
                        None, None, None)


@pytest.mark.parametrize("kw,code", [
    *[(dict(ptr=None, ptr_at=i), 1) for i in range(9)],
    *[(dict(ptr=MISALIGNED, ptr_at=i), 1) for i in range(9)],
    (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(dt=7), 1), (dict(gdt=7), 1), (dict(causal=2), 1),
    (dict(tau=-1.0), 1), (dict(tau=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(D=96), 2), (dict(blk=32), 2),
])
def test_bwd_rejects_bad_arguments(lib, kw, code):
    """Every pointer (null or misaligned) and the shared shape checks, before
    the workspace is looked at."""
    assert _bwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(splits=0), 1), (dict(splits=300), 1), (dict(Hq=12, Hkv=8), 1), (dict(Hq=48, Hkv=3), 2),
    (dict(D=80), 2), (dict(blk=32), 2), (dict(tau=-0.5), 1), (dict(ws=None), 3), (dict(ws_bytes=64), 3),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    p = dict(B=8, N=1024, Hq=32, Hkv=8, D=128, blk=128, splits=16, tau=1.0, ws=FAKE, ws_bytes=1 << 30)
    p.update(kw)
    rc = lib.mala_decode(FAKE, FAKE, FAKE, FAKE, FAKE, p["B"], p["N"], p["Hq"], p["Hkv"], p["D"], 0, 0,
                         p["blk"], p["splits"], p["tau"], 0.08, p["ws"], p["ws_bytes"], None, None, None)
    assert rc == code


def test_noalloc_decode_rejects_oversize_before_any_launch(lib):
    cap = lib.mala_decode_noalloc_max_floats()
    assert cap == 1 << 20
    # 16 splits * 64 sequences * 32 heads * 132 floats > cap: rejected by shape alone
    rc = lib.mala_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 1024, 32, 8, 128, 0, 0, 128, 16, 1.0, 0.08,
                                 None, None, None)
    assert rc == 3
    rc = lib.mala_decode_noalloc(None, FAKE, FAKE, FAKE, FAKE, 1, 1024, 32, 8, 128, 0, 0, 128, 16, 1.0, 0.08,
                                 None, None, None)
    assert rc == 1


def test_device_status_rejects_null(lib):
    assert lib.mala_device_status(None, None) == 1


@pytest.mark.parametrize("cu,batch,total,lmax", [
    (None, 2, 512, 256), (ctypes.c_void_p(0x10002), 2, 512, 256), (FAKE, 0, 512, 256),
    (FAKE, 2, 0, 256), (FAKE, 2, 512, 0), (FAKE, 2, 512, 513),
])
def test_packed_prefill_rejects_bad_sequence_bounds(lib, cu, batch, total, lmax):
    """cu_seqlens null or misaligned, no sequence, no token, or a longest
    sequence of 0 or past the packed total: both packed entry points refuse
    before any launch."""
    fwd = lib.mala_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, cu, batch, total, lmax, 2, 2, 64, 1, 1, 1, 64, 64,
                              1.0, 0.125, None, None, None)
    bwd = lib.mala_bwd_varlen(*([FAKE] * 9), cu, batch, total, lmax, 2, 2, 64, 1, 1, 1, 64, 64, 1.0, 0.125,
                              FAKE, 1 << 30, None, None, None)
    assert fwd == 1 and bwd == 1


def test_decode_varlen_rejects_missing_or_misaligned_lengths(lib):
    args = [FAKE] * 5
    shape = [8, 1024, 32, 8, 128, 0, 0, 128, 16, 1.0, 0.08, FAKE, 1 << 30, None, None, None]
    assert lib.mala_decode_varlen(*args, None, *shape) == 1
    assert lib.mala_decode_varlen(*args, ctypes.c_void_p(0x10002), *shape) == 1
    # shape checks are those of mala_decode
    bad = list(shape)
    bad[2], bad[3] = 48, 3                      # group of 16
    assert lib.mala_decode_varlen(*args, FAKE, *bad) == 2


def test_forced_forward_rejects_bad_arguments(lib):
    shape = [1, 256, 256, 2, 2, 128, 0, 1, 1, 128, 128, 0.088]
    assert lib.mala_fwd_forced(*[FAKE] * 5, *shape, None, None, None, None) == 1        # no tile set
    assert lib.mala_fwd_forced(None, *[FAKE] * 4, *shape, FAKE, None, None, None) == 1
    bad = list(shape)
    bad[5] = 96                                                                        # head_dim
    assert lib.mala_fwd_forced(*[FAKE] * 5, *bad, FAKE, None, None, None) == 2


def test_region_mass_rejects_bad_arguments(lib):
    shape = [1, 256, 256, 2, 2, 128, 0, 1, 128, 128, 0.088]
    assert lib.mala_region_mass(FAKE, FAKE, None, FAKE, *shape, None) == 1
    assert lib.mala_region_mass(FAKE, FAKE, ctypes.c_void_p(0x10002), FAKE, *shape, None) == 1
    bad = list(shape)
    bad[3], bad[4] = 3, 2                                                              # Hq % Hkv
    assert lib.mala_region_mass(FAKE, FAKE, FAKE, FAKE, *bad, None) == 1
    bad = list(shape)
    bad[8], bad[9] = 64, 128                                                           # block_q != block_k
    assert lib.mala_region_mass(FAKE, FAKE, FAKE, FAKE, *bad, None) == 2
