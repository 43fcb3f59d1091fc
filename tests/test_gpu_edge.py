"""GPU edge cases against the fp64 oracle, on small seeded workloads that reach
every kernel variant: the fused short-unit kernel and the split long-unit path
(tensor-core and CUDA-core scoring), dense and paged caches (16- and 32-token
blocks), G = 1, 2, 4, 8, head dim 64 and 128, bf16 and fp32, both band
pairings, ragged lengths with units at N < B, N = B and N = B + 1 in one call,
t != N, and a unit whose keys are all equal (every score ties).
"""
import dataclasses

import numpy as np
import pytest
import torch

from synth import Workload, generate
from tests import _gpu_check as C

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
GEO16 = tuple(2 ** i for i in range(17))
GEO10 = tuple(2 ** i for i in range(11))
# the linear offset set of the offset ablation (results section of the method's
# write-up: geometric sampling beats linear), o = 64 k, k = 1..32
LIN32 = tuple(64 * k for k in range(1, 33))


def W(name, **kw):
    base = dict(L=1, S=3, Hq=8, Hkv=2, d=128, theta=1e6, dtype="bf16", budget=512, offsets=GEO16)
    base.update(kw)
    return Workload(name=name, **base)


CASES = [
    # fused short-unit kernel
    W("edge_fused_g1_bf16", Hq=2, n_range=(300, 900)),
    W("edge_fused_g2_inter_d64", Hq=4, d=64, pairing="interleaved", n_range=(500, 1500)),
    W("edge_fused_g4_f32", Hq=8, dtype="f32", n_range=(600, 1800), budget=700),
    W("edge_fused_g8_bf16", Hq=16, n_range=(1000, 3000), budget=1024),
    W("edge_fused_paged16_g4", Hq=8, n_range=(700, 2500), paged=True),
    W("edge_fused_paged32_g2_d64", Hq=4, d=64, n_range=(700, 2500), paged=True, block=32),
    # split long-unit path (scores larger than one CTA's shared memory)
    W("edge_long_mma_g4", Hq=8, n_range=(9000, 13000), budget=1024),
    W("edge_long_mma_g8_d64", Hq=16, d=64, n_range=(15000, 20000), budget=2048),
    W("edge_long_mma_g1", Hq=2, n_range=(40000, 60000), budget=4096, S=2),
    W("edge_long_mma_g2_paged", Hq=4, n_range=(26000, 30000), budget=1024, paged=True, S=2),
    W("edge_long_mma_g8_paged32", Hq=16, n_range=(12000, 16000), budget=1024, paged=True, block=32),
    W("edge_long_cuda_f32_g2", Hq=4, d=64, dtype="f32", n_range=(30000, 40000), budget=2048, S=2),
    # paged blocks of 128 head-rows (8 heads x 16 rows, 4 x 32): every KV head of
    # a block scored by one CTA from one copy (score_heads_mma_kernel); lengths
    # off the 2048-key CTA boundaries and partial last blocks
    W("edge_long_hg_g8_h8_paged16", Hq=64, Hkv=8, n_range=(2100, 9000), budget=1024, paged=True, S=2),
    W("edge_long_hg_g4_h8_paged16", Hq=32, Hkv=8, n_range=(4000, 14000), budget=2048, paged=True, S=2),
    W("edge_long_hg_g1_h8_paged16", Hq=8, Hkv=8, n_range=(30000, 40000), budget=4096, paged=True, S=2),
    W("edge_long_hg_g2_h4_paged32", Hq=8, Hkv=4, n_range=(30000, 36000), budget=2048, paged=True, block=32, S=2),
    W("edge_long_cuda_inter_g4", Hq=8, pairing="interleaved", n_range=(11000, 14000), budget=1024),
    # linear future offsets instead of geometric ones
    W("edge_linear_offsets_fused_g4", Hq=8, n_range=(600, 1800), budget=700, offsets=LIN32),
    W("edge_linear_offsets_long_g4", Hq=8, n_range=(9000, 13000), budget=1024, offsets=LIN32),
    W("edge_linear_offsets_long_g8_paged", Hq=16, n_range=(12000, 16000), budget=1024, paged=True, offsets=LIN32),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_edge_every_unit(w):
    data = generate(w, device=DEV)
    units = [(0, s, g) for s in range(w.S) for g in range(w.Hkv)]
    C.run_and_check(w, data, units, DEV)


def test_budget_boundaries_and_t_offset():
    """One call with N = B - 1, B, B + 1 and a long unit; t = N + 37."""
    w = W("edge_bounds", Hq=8, S=4, budget=1000, n_keys=1200)
    data = generate(w, device=DEV)
    lens = [999, 1000, 1001, 1200]
    data["seq_len"] = torch.tensor(lens, dtype=torch.int32, device=DEV)
    data["t"] = data["seq_len"] + 37
    w2 = dataclasses.replace(w, n_keys=None, n_range=(999, 1200))
    object.__setattr__(w2, "seq_lengths", lambda: lens)
    units = [(0, s, g) for s in range(4) for g in range(w.Hkv)]
    C.run_and_check(w2, data, units, DEV)


@pytest.mark.parametrize("n_keys,Hq", [(800, 4), (20000, 4), (20000, 2)])
def test_all_zero_keys_tie_everywhere(n_keys, Hq):
    """A unit whose keys are all zero (a cleared or padded region): every score
    is exactly 0 on both sides, the z-score of each head is 0/0 := 0, all keys
    tie, the lowest B slots are kept and nothing moves (fused path at N = 800,
    split path at N = 20000).  On the split path every key is a candidate after
    the first digit: at G = 2 the candidate pairs just fit the unit's dead raw
    scores, at G = 1 they do not and the selection takes its full-pass route."""
    w = W(f"edge_ties_{n_keys}_g{Hq // 2}", Hq=Hq, S=1, Hkv=2, budget=300, n_keys=n_keys)
    data = generate(w, device=DEV)
    data["k"][0, 0, 1].zero_()          # KV head 1
    # the zero unit must keep exactly slots 0..B-1: no difference, even in the tie band
    assert C.run_and_check(w, data, [(0, 0, 1)], DEV) == 0
    C.run_and_check(w, generate(w, device=DEV), [(0, 0, 0)], DEV)


def test_long_unit_top_keys_off_the_sampled_slots():
    """The long-unit selection brackets the threshold with a sample of every
    (N / 1024)-th slot.  A unit's score depends only on the stored (post-RoPE)
    row, not on its slot, so moving the rows of the B highest aggregated scores
    onto slots the sample never reads hides them from it: its range then sits
    below the threshold and the selection must notice and take its full passes.
    Parity with the oracle as for every unit (both KV heads; head 0 moved)."""
    import kv_cache_compression_06_b300 as tk
    N, B = 20000, 300
    w = W("edge_sample_miss_g4", Hq=8, S=1, Hkv=2, budget=B, n_keys=N)
    data = generate(w, device=DEV)
    cache, stats, params = C.setup(w, data, DEV)
    probe = tk.KVCache(cache.k.clone(), cache.v.clone(), cache.seq_len, Hkv=w.Hkv)
    agg = torch.zeros((1, 1, w.Hkv, w.cap), dtype=torch.float32, device=DEV)
    tk.tri_score(probe, stats, params, agg=agg)
    a = agg[0, 0, 0, :N].double().cpu().numpy()
    top = np.argsort(-a, kind="stable")[:B]
    sampled = {(j * N) // 1024 for j in range(1024)}
    free = np.array([i for i in range(N) if i not in sampled])
    rest = np.array([i for i in range(N) if i not in set(top.tolist())])
    order = np.empty(N, dtype=np.int64)          # order[slot] = original row now at slot
    order[free[:B]] = top
    others = np.array([i for i in range(N) if i not in set(free[:B].tolist())])
    order[others] = rest
    perm = torch.as_tensor(order, device=DEV)
    for t in ("k", "v"):
        data[t][0, 0, 0, :N] = data[t][0, 0, 0, :N][perm].clone()
    C.run_and_check(w, data, [(0, 0, 0), (0, 0, 1)], DEV)


HOLEFILL_CASES = [
    W("hf_fused_g4", Hq=8, n_range=(600, 1900), budget=700),
    W("hf_fused_paged_g2_d64", Hq=4, d=64, n_range=(700, 2500), paged=True),
    W("hf_long_mma_g4", Hq=8, n_range=(9000, 13000), budget=1024),
    W("hf_long_mma_g8_paged", Hq=16, n_range=(12000, 16000), budget=1024, paged=True),
    W("hf_long_cuda_f32", Hq=4, d=64, dtype="f32", n_range=(30000, 40000), budget=2048, S=2),
    # B = 8192: the list and holes (64 KB) exceed holefill_apply_kernel's cap, so
    # compact_only_kernel moves the rows itself
    W("hf_long_mma_b8192_in_compaction", Hq=8, n_range=(18000, 26000), budget=8192, S=2),
]


@pytest.mark.parametrize("w", HOLEFILL_CASES, ids=[w.name for w in HOLEFILL_CASES])
def test_holefill_every_unit(w):
    data = generate(w, device=DEV)
    units = [(0, s, g) for s in range(w.S) for g in range(w.Hkv)]
    C.run_and_check_holefill(w, data, units, DEV)


DEFER_CASES = [
    W("hf_defer_fused_g4", Hq=8, n_range=(600, 1900), budget=700),
    W("hf_defer_fused_g8", Hq=16, n_range=(1000, 3000), budget=1024),
    W("hf_defer_fused_paged16_g4", Hq=8, n_range=(700, 2500), paged=True),
    W("hf_defer_fused_f32_inter_g2", Hq=4, d=64, dtype="f32", pairing="interleaved", n_range=(500, 1500)),
]


@pytest.mark.parametrize("w", DEFER_CASES, ids=[w.name for w in DEFER_CASES])
def test_holefill_moves_without_idx_out_match_the_apply_kernel(w):
    """With idx_out the fused kernel leaves the hole-fill moves to
    holefill_apply_kernel; without it the fused kernel moves the rows itself.
    Both give the same cache, bit for bit, and the same lengths."""
    import kv_cache_compression_06_b300 as tk
    data = generate(w, device=DEV)
    out = []
    for with_idx in (True, False):
        cache, stats, params = C.setup(w, data, DEV)
        cache = tk.KVCache(cache.k.clone(), cache.v.clone(), cache.seq_len, Hkv=w.Hkv,
                           block_table=cache.block_table, block=w.block)
        L = cache.k.shape[0]
        idx = torch.full((L, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=DEV) if with_idx else None
        new_len = torch.full((w.S,), -7, dtype=torch.int32, device=DEV)
        tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len, compact="holefill")
        torch.cuda.synchronize()
        assert tk.tri_get_device_status() == 0
        out.append((cache.k, cache.v, new_len))
    assert torch.equal(out[0][2], out[1][2])
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])
