"""C-ABI checks that need no GPU: the library loads, exports exactly what
include/tri.h declares, and rejects bad arguments on the host before launching
anything (every call below carries at least one argument the host check refuses).
"""
import ctypes
import os
import re

import pytest

from kv_cache_compression_06_b300 import tri as T

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tri.h")
FAKE = 1 << 20          # an aligned non-null address; never dereferenced (host checks reject first)


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"TRI_API\s+[\w\s\*]+?\b(tri_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = T.lib()
    decl = declared_functions()
    assert len(decl) >= 10
    for name in decl:
        assert hasattr(lib, name), name
    assert sorted(T.EXPORTED) == decl


def test_version_and_status_strings():
    assert T.lib().tri_version() == 100
    assert T.status_string(T.TRI_OK) == "ok"
    assert "invalid" in T.status_string(T.TRI_ERR_INVALID)
    assert "unknown" in T.status_string(99)


def _cache(**kw):
    c = T.tri_cache()
    c.k, c.v, c.dtype, c.L, c.S, c.Hkv, c.d, c.cap, c.seq_len = FAKE, FAKE, T.TRI_BF16, 2, 3, 4, 128, 100, FAKE
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _stats(Hq=16):
    s = T.tri_stats()
    s.center, s.R, s.mag, s.Hq = FAKE, FAKE, FAKE, Hq
    return s


def _params(**kw):
    arr = (ctypes.c_int32 * 3)(1, 2, 4)
    p = T.tri_params()
    p.theta, p.pairing, p.t, p.offsets, p.n_offsets, p.budget = 1e6, T.TRI_PAIR_HALF, FAKE, arr, 3, 64
    for k, v in kw.items():
        setattr(p, k, v)
    return p, arr


BAD_CACHES = [
    dict(d=96),                 # unsupported head dim
    dict(d=0),
    dict(L=0),
    dict(S=-1),
    dict(cap=0),
    dict(seq_len=None),
    dict(k=FAKE + 4),           # misaligned
    dict(v=None),
    dict(dtype=7),
    dict(block_table=FAKE, max_blocks=6, block=16, nblocks=10),   # cap != max_blocks*block
]


@pytest.mark.parametrize("bad", BAD_CACHES)
def test_compress_step_rejects_bad_cache(bad):
    c = _cache(**bad)
    s = _stats()
    p, _a = _params()
    st = T.lib().tri_compress_step(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), 0, None, None,
                                   None, 0, None)
    assert st in (T.TRI_ERR_INVALID, T.TRI_ERR_UNSUPPORTED)


@pytest.mark.parametrize("Hq,want", [(6, T.TRI_ERR_INVALID), (48, T.TRI_ERR_UNSUPPORTED), (0, T.TRI_ERR_INVALID)])
def test_score_rejects_bad_group(Hq, want):
    c, s = _cache(), _stats(Hq)
    p, _a = _params()
    assert T.lib().tri_score(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), FAKE, None, None, 0, None) == want


@pytest.mark.parametrize("bad", [dict(theta=0.0), dict(theta=float("nan")), dict(n_offsets=0),
                                 dict(budget=0), dict(t=None), dict(pairing=5)])
def test_score_rejects_bad_params(bad):
    c, s = _cache(), _stats()
    p, _a = _params(**bad)
    assert T.lib().tri_score(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), FAKE, None, None, 0,
                             None) == T.TRI_ERR_INVALID


def test_negative_offset_rejected():
    c, s = _cache(), _stats()
    arr = (ctypes.c_int32 * 2)(1, -2)
    p, _a = _params()
    p.offsets, p.n_offsets = arr, 2
    assert T.lib().tri_score(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), FAKE, None, None, 0,
                             None) == T.TRI_ERR_INVALID


def test_null_outputs_and_aliasing_rejected():
    c, s = _cache(), _stats()
    p, _a = _params()
    L = T.lib()
    assert L.tri_score(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), None, None, None, 0, None) == T.TRI_ERR_INVALID
    assert L.tri_select_topb(ctypes.byref(c), None, 4, FAKE, None, 0, None) == T.TRI_ERR_INVALID
    assert L.tri_select_topb(ctypes.byref(c), FAKE, 0, FAKE, None, 0, None) == T.TRI_ERR_INVALID
    assert L.tri_compact_kv(ctypes.byref(c), None, 4, 0, None, None) == T.TRI_ERR_INVALID
    assert L.tri_compact_kv(ctypes.byref(c), FAKE, 4, 7, None, None) == T.TRI_ERR_UNSUPPORTED   # no such layout
    # new_len aliasing seq_len would race with units still reading N
    assert L.tri_compact_kv(ctypes.byref(c), FAKE, 4, 0, FAKE, None) == T.TRI_ERR_INVALID
    assert L.tri_compress_step(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), 0, None, FAKE, None, 0,
                               None) == T.TRI_ERR_INVALID
    assert L.tri_get_device_status(None, None) == T.TRI_ERR_INVALID


def test_calibrate_rejects_bad_arguments():
    L = T.lib()
    assert L.tri_calibrate_stats(None, 0, 10, 1, 2, 64, 0, FAKE, FAKE, FAKE, None) == T.TRI_ERR_INVALID
    assert L.tri_calibrate_stats(FAKE, 0, 0, 1, 2, 64, 0, FAKE, FAKE, FAKE, None) == T.TRI_ERR_INVALID
    assert L.tri_calibrate_stats(FAKE, 0, 10, 1, 2, 80, 0, FAKE, FAKE, FAKE, None) == T.TRI_ERR_INVALID
    assert L.tri_calibrate_stats(FAKE, 3, 10, 1, 2, 64, 0, FAKE, FAKE, FAKE, None) == T.TRI_ERR_INVALID


def test_workspace_query_is_host_only():
    """Workspace sizing is pure host arithmetic: 0 when a unit's scores fit one
    CTA, raw scores + per-tile moments otherwise."""
    L = T.lib()
    s = _stats(32)
    p, _a = _params()
    n = ctypes.c_size_t(123)
    c = _cache(Hkv=8, cap=2176)
    assert L.tri_workspace_bytes(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), ctypes.byref(n)) == 0
    assert n.value == 0
    c = _cache(Hkv=8, cap=32768)
    assert L.tri_workspace_bytes(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), ctypes.byref(n)) == 0
    units, G, ntiles = 2 * 3 * 8, 4, 16
    assert n.value >= units * G * 32768 * 4 + units * ntiles * G * 8


def test_streamed_calibration_rejects_bad_arguments():
    L = T.lib()
    # reset / merge / finalize: shapes and pointers
    assert L.tri_calib_reset(None, 1, 2, 64, None) == T.TRI_ERR_INVALID
    assert L.tri_calib_reset(FAKE + 4, 1, 2, 64, None) == T.TRI_ERR_INVALID        # not 8-byte aligned
    assert L.tri_calib_reset(FAKE, 0, 2, 64, None) == T.TRI_ERR_INVALID
    assert L.tri_calib_reset(FAKE, 1, 2, 96, None) == T.TRI_ERR_INVALID
    assert L.tri_calib_merge(FAKE, FAKE, 1, 2, 64, None) == T.TRI_ERR_INVALID      # acc aliases other
    assert L.tri_calib_merge(FAKE, None, 1, 2, 64, None) == T.TRI_ERR_INVALID
    assert L.tri_calib_finalize(FAKE, 1, 2, 64, FAKE, None, FAKE, None) == T.TRI_ERR_INVALID
    # accumulate: q alignment, dtype, pairing, strides
    acc = FAKE
    args = dict(q=FAKE, dt=T.TRI_BF16, n=10, L=1, H=2, d=64, pr=0, ss=0, ls=0)

    def call(**kw):
        a = {**args, **kw}
        return L.tri_calib_accumulate(a["q"], a["dt"], a["n"], a["L"], a["H"], a["d"], a["pr"], a["ss"], a["ls"],
                                      acc, None)

    assert call(q=None) == T.TRI_ERR_INVALID
    assert call(q=FAKE + 8) == T.TRI_ERR_INVALID          # q must be 16-byte aligned
    assert call(dt=5) == T.TRI_ERR_INVALID
    assert call(pr=3) == T.TRI_ERR_INVALID
    assert call(n=-1) == T.TRI_ERR_INVALID
    assert call(ss=100) == T.TRI_ERR_INVALID              # < H*d
    assert call(ss=130) == T.TRI_ERR_INVALID              # not a multiple of 4 elements
    assert call(L=2, ls=6) == T.TRI_ERR_INVALID
    assert call(n=0) == T.TRI_OK                          # nothing to add: returns before any launch
    assert call(n=0, q=None) == T.TRI_OK                  # and reads nothing


def test_distance_curves_reject_bad_arguments():
    L = T.lib()

    def call(Hq=4, Hkv=2, d=64, theta=1e4, n=100, nd=50, q=FAKE, k=FAKE, lc=FAKE, corr=FAKE, dt=0, pr=0):
        return L.tri_distance_curves(FAKE, FAKE, q, k, dt, n, 1, Hq, Hkv, d, theta, pr, nd, FAKE, lc, corr, None)

    assert call(Hq=6, Hkv=4) == T.TRI_ERR_INVALID
    assert call(d=48) == T.TRI_ERR_INVALID
    assert call(theta=-1.0) == T.TRI_ERR_INVALID
    assert call(nd=0) == T.TRI_ERR_INVALID
    assert call(nd=101) == T.TRI_ERR_INVALID              # more distances than samples
    assert call(q=None) == T.TRI_ERR_INVALID              # logit curve asked for without samples
    assert call(lc=None) == T.TRI_ERR_INVALID             # corr needs the logit curve
    assert call(dt=9) == T.TRI_ERR_INVALID
    assert call(pr=2) == T.TRI_ERR_INVALID


def test_bounded_wait_check_rejects_bad_limits():
    assert T.lib().tri_check_bounded_wait(0, None) == T.TRI_ERR_INVALID
    assert T.lib().tri_check_bounded_wait(1000001, None) == T.TRI_ERR_INVALID
