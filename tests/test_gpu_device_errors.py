"""Device-side argument errors: conditions the host cannot see (a block id out
of range, an idx row that is not strictly increasing, seq_len > cap) make the
kernels skip the affected unit and record a status code, readable with
tri_get_device_status; the other units are processed normally and a cleared
status reads TRI_OK again.  The kernels check these conditions before any
memory access they would govern, so no fault is involved.
"""
import pytest
import torch

import kv_cache_compression_06_b300 as tk
from kv_cache_compression_06_b300 import tri as T
from synth import Workload, generate
from tests import _gpu_check as C

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
GEO16 = tuple(2 ** i for i in range(17))


def _paged(name, n_range, budget):
    return Workload(name=name, L=1, S=3, Hq=8, Hkv=2, d=128, theta=1e6, dtype="bf16", budget=budget,
                    offsets=GEO16, n_range=n_range, paged=True)


def _reference_idx(w, data):
    """idx of a clean run (all sequences valid)."""
    cache, stats, params = C.setup(w, {k: (v.clone() if torch.is_tensor(v) else v) for k, v in data.items()}, DEV)
    idx = torch.full((1, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=DEV)
    tk.tri_compress_step(cache, stats, params, idx_out=idx)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == T.TRI_OK
    return idx


@pytest.mark.parametrize("n_range,budget", [((1200, 2000), 600), ((12000, 16000), 1024)],
                         ids=["fused", "long"])
def test_block_id_out_of_range_skips_that_sequence(n_range, budget):
    w = _paged(f"err_block_{budget}", n_range, budget)
    data = generate(w, device=DEV)
    ref = _reference_idx(w, data)
    bt = data["block_table"].clone()
    bt[1, 3] = int(data["nblocks"]) + 5            # sequence 1 points past the pool
    cache, stats, params = C.setup(w, {**data, "block_table": bt}, DEV)
    k_before = cache.k.clone()
    idx = torch.full((1, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=DEV)
    new_len = torch.full((w.S,), -7, dtype=torch.int32, device=DEV)
    tk.tri_clear_device_status()
    tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == T.TRI_ERR_BOUNDS
    lens = data["seq_len"].tolist()
    assert new_len.tolist() == [min(lens[0], w.budget), lens[1], min(lens[2], w.budget)]
    for s in (0, 2):                                 # untouched sequences: same result as the clean run
        assert torch.equal(idx[0, s], ref[0, s])
    # nothing of sequence 1 was written: its idx rows keep the fill value, its
    # blocks (all but the bad entry) keep their rows
    assert torch.all(idx[0, 1] == -7)
    nb = -(-int(data["seq_len"][1]) // w.block)
    blocks = [int(b) for b in bt[1, :nb].tolist() if b < int(data["nblocks"])]
    assert torch.equal(cache.k[0, blocks], k_before[0, blocks])
    tk.tri_clear_device_status()
    assert tk.tri_get_device_status() == T.TRI_OK


def test_compact_rejects_idx_rows_that_do_not_increase():
    w = Workload(name="err_idx", L=1, S=2, Hq=8, Hkv=2, d=128, theta=1e6, dtype="bf16", budget=500,
                 offsets=GEO16, n_keys=900)
    data = generate(w, device=DEV)
    cache, stats, params = C.setup(w, data, DEV)
    good = torch.arange(400, 900, dtype=torch.int32, device=DEV)
    idx = good.expand(1, 2, 2, 500).contiguous()
    idx[0, 1, 0, 10] = idx[0, 1, 0, 9]                # repeated slot in unit (s=1, g=0)
    k_before = cache.k.clone()
    tk.tri_clear_device_status()
    tk.tri_compact_kv(cache, idx, w.budget)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == T.TRI_ERR_INVALID
    assert torch.equal(cache.k[0, 1, 0], k_before[0, 1, 0])             # bad unit untouched
    assert torch.equal(cache.k[0, 0, 0, :500], k_before[0, 0, 0, 400:900])   # good unit compacted
    tk.tri_clear_device_status()


def test_seq_len_beyond_cap_is_reported():
    w = Workload(name="err_len", L=1, S=2, Hq=8, Hkv=2, d=128, theta=1e6, dtype="bf16", budget=300,
                 offsets=GEO16, n_keys=700)
    data = generate(w, device=DEV)
    data["seq_len"] = torch.tensor([700, 701], dtype=torch.int32, device=DEV)   # cap is 700
    cache, stats, params = C.setup(w, data, DEV)
    k_before = cache.k.clone()
    tk.tri_clear_device_status()
    tk.tri_compress_step(cache, stats, params)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == T.TRI_ERR_BOUNDS
    assert torch.equal(cache.k[0, 1], k_before[0, 1])
    assert not torch.equal(cache.k[0, 0], k_before[0, 0])
    tk.tri_clear_device_status()


@pytest.mark.parametrize("n_keys,budget", [(900, 500), (12000, 1024)], ids=["fused", "long"])
def test_bounded_wait_gives_up_and_later_calls_return_without_work(n_keys, budget):
    """tri_check_bounded_wait waits (1 ms limit) on a barrier nothing arrives at,
    with nothing in flight: the wait gives up and records TRI_ERR_TIMEOUT.  The
    next tri_compress_step then returns without touching the cache, idx or the
    new lengths; once the status is cleared the same call runs normally."""
    w = Workload(name=f"wait_check_{n_keys}", L=1, S=2, Hq=8, Hkv=2, d=128, theta=1e6, dtype="bf16",
                 budget=budget, offsets=GEO16, n_keys=n_keys)
    data = generate(w, device=DEV)
    ref = _reference_idx(w, data)
    cache, stats, params = C.setup(w, data, DEV)
    ws = tk.workspace(cache, stats, params)
    k0, v0 = cache.k.clone(), cache.v.clone()
    idx = torch.full((1, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=DEV)
    new_len = torch.full((w.S,), -7, dtype=torch.int32, device=DEV)
    try:
        tk.tri_clear_device_status()
        T.tri_check_bounded_wait(1000)
        torch.cuda.synchronize()
        assert tk.tri_get_device_status() == T.TRI_ERR_TIMEOUT
        tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len, ws=ws)
        torch.cuda.synchronize()
        assert tk.tri_get_device_status() == T.TRI_ERR_TIMEOUT
        assert torch.equal(cache.k, k0) and torch.equal(cache.v, v0)
        assert torch.all(idx == -7) and torch.all(new_len == -7)
    finally:
        tk.tri_clear_device_status()
    assert tk.tri_get_device_status() == T.TRI_OK
    tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len, ws=ws)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == T.TRI_OK
    assert torch.equal(idx, ref)
    assert new_len.tolist() == [budget] * w.S
