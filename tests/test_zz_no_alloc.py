"""tri_compress_step_static_scratch: the compression step for callers that cannot
allocate device memory (for example a serving engine that reserved nearly all of
it for its KV-cache pool and forbids later allocations).  Such callers cannot
pass the workspace that long units need, so the library uses a fixed scratch
array built into it instead.

The GPU test runs two calls in a row (the second one sees the first one's
leftovers in the shared scratch) on long, ragged units that take the
scratch-using path, and checks each against tri_compress_step with a caller
workspace: kept indices, new lengths and compacted K/V must be identical, for
both compaction layouts (ordered and hole-fill).
This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import kv_cache_compression_06_b300 as tk
from kv_cache_compression_06_b300 import tri as T
from synth import Workload, generate

FAKE = 1 << 20   # aligned non-null address; the host check rejects before any use

_GEO16 = tuple(2 ** i for i in range(17))
# Two long-unit workloads (scores of a unit do not fit one CTA's shared memory).
CASES = [
    Workload(name="static_scratch_a", L=1, S=2, Hq=16, Hkv=4, d=128, theta=1e6, dtype="bf16",
             budget=1024, offsets=_GEO16, n_range=(11000, 16000)),
    Workload(name="static_scratch_b", L=2, S=3, Hq=16, Hkv=2, d=128, theta=1e6, dtype="bf16",
             budget=2048, offsets=_GEO16, n_range=(1500, 20000)),
]


def test_rejects_steps_larger_than_the_builtin_scratch():
    """Host-only: a step needing more than TRI_STATIC_SCRATCH_BYTES of scratch is
    refused with TRI_ERR_WORKSPACE before anything is launched."""
    c = T.tri_cache()
    c.k, c.v, c.dtype, c.L, c.S, c.Hkv, c.d, c.cap, c.seq_len = FAKE, FAKE, T.TRI_BF16, 1, 64, 8, 128, 32768, FAKE
    s = T.tri_stats()
    s.center, s.R, s.mag, s.Hq = FAKE, FAKE, FAKE, 32
    arr = (ctypes.c_int32 * 3)(1, 2, 4)
    p = T.tri_params()
    p.theta, p.pairing, p.t, p.offsets, p.n_offsets, p.budget = 1e6, T.TRI_PAIR_HALF, FAKE, arr, 3, 2048
    need = ctypes.c_size_t(0)
    assert T.lib().tri_workspace_bytes(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), ctypes.byref(need)) == 0
    assert need.value > T.TRI_STATIC_SCRATCH_BYTES
    st = T.lib().tri_compress_step_static_scratch(ctypes.byref(c), ctypes.byref(s), ctypes.byref(p), 0, None,
                                                  None, None)
    assert st == T.TRI_ERR_WORKSPACE


def _setup(w, dev):
    data = generate(w, device=dev)
    cache = tk.KVCache(data["k"], data["v"], data["seq_len"], Hkv=w.Hkv)
    stats = tk.tri_calibrate_stats(data["q_pre"])
    params = tk.Params(w.theta, data["t"], w.offsets, w.budget)
    return cache, stats, params


@pytest.mark.gpu
@pytest.mark.parametrize("compact", ["ordered", "holefill"])
def test_static_scratch_matches_workspace_entry_point_twice_in_a_row(compact):
    dev = torch.device("cuda:0")
    for w in CASES:
        cache, stats, params = _setup(w, dev)
        need = tk.tri_workspace_bytes(cache, stats, params)
        assert 0 < need <= T.TRI_STATIC_SCRATCH_BYTES, "case must take the scratch-using path"
        k0, v0 = cache.k.clone(), cache.v.clone()
        shape = (cache.L, cache.S, cache.Hkv, w.budget)

        # existing entry point, caller-provided workspace
        ws = tk.workspace(cache, stats, params)
        idx_ref = torch.full(shape, -7, dtype=torch.int32, device=dev)
        len_ref = torch.full((cache.S,), -7, dtype=torch.int32, device=dev)
        tk.tri_compress_step(cache, stats, params, idx_out=idx_ref, new_len=len_ref, ws=ws, compact=compact)
        torch.cuda.synchronize()
        assert tk.tri_get_device_status() == 0
        k_ref, v_ref = cache.k.clone(), cache.v.clone()

        # the same step through the built-in scratch, from the pristine cache
        cache.k.copy_(k0)
        cache.v.copy_(v0)
        idx = torch.full(shape, -7, dtype=torch.int32, device=dev)
        new_len = torch.full((cache.S,), -7, dtype=torch.int32, device=dev)
        tk.tri_compress_step_static_scratch(cache, stats, params, idx_out=idx, new_len=new_len, compact=compact)
        torch.cuda.synchronize()
        assert tk.tri_get_device_status() == 0

        assert torch.equal(idx, idx_ref)
        assert torch.equal(new_len, len_ref)
        lens = cache.seq_len.tolist()
        for s, n in enumerate(lens):
            m = min(n, w.budget)
            assert torch.equal(cache.k[:, s, :, :m], k_ref[:, s, :, :m])
            assert torch.equal(cache.v[:, s, :, :m], v_ref[:, s, :, :m])
        assert any(n > w.budget for n in lens)
