"""GPU parity of the decode loop around the compression step, through the C ABI:
tri_append_kv and tri_decode_attention every token, tri_compress_step every 128
tokens (the pruning paragraph's trigger), on small seeded caches that grow by
two windows.

The host tracks the position of the key in every slot (appends add the token's
position; a compression moves positions as idx_out says), so at every trigger
each unit is checked against the oracle's per-offset route (which un-rotates
keys by their true positions, not their slots): kept sets equal outside the tie
band, compacted K/V bit-exact against the pre-step rows at the GPU's indices.
Appended rows: the key equals the pre-RoPE key rotated in fp64 to within one
bf16 rounding, the value bit-exact.  Attention outputs at sampled steps: within
1e-3 of the largest output of the unit from the oracle's fp64 softmax attention
over the same rows.
"""
import numpy as np
import pytest
import torch

import kv_cache_compression_06_b300 as tk
from oracle import tri_oracle as O
from synth import Workload, generate, sequence_samples, unit_rows
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
GEO16 = tuple(2 ** i for i in range(17))
WINDOW = 128


def grown(w, data, extra):
    """The generated cache with room for `extra` more tokens per sequence
    (dense: a larger cap; paged: more blocks per sequence, new block ids drawn
    from a larger pool in a seeded random order)."""
    lens = data["seq_len"].tolist()
    gen = w.seq_lengths()              # rows (and blocks) the generator allocated
    L = data["k"].shape[0]
    if not w.paged:
        cap = max(lens) + extra
        K = torch.zeros((L, w.S, w.Hkv, cap, w.d), dtype=data["k"].dtype, device=DEV)
        V = torch.zeros_like(K)
        K[:, :, :, : data["k"].shape[3]] = data["k"]
        V[:, :, :, : data["v"].shape[3]] = data["v"]
        return K, V, None, cap
    bt_old = data["block_table"].cpu().numpy()
    nb_old = int(data["nblocks"])
    have = [-(-n // w.block) for n in gen]
    need = [max(h, -(-(n + extra) // w.block)) for h, n in zip(have, lens)]
    add = sum(a - b for a, b in zip(need, have))
    rng = np.random.default_rng(7)
    fresh = iter((nb_old + rng.permutation(add)).tolist())
    bt = np.zeros((w.S, max(need)), dtype=np.int32)
    for s in range(w.S):
        bt[s, : have[s]] = bt_old[s, : have[s]]
        for b in range(have[s], need[s]):
            bt[s, b] = next(fresh)
    K = torch.zeros((L, nb_old + add) + tuple(data["k"].shape[2:]), dtype=data["k"].dtype, device=DEV)
    V = torch.zeros_like(K)
    K[:, :nb_old] = data["k"]
    V[:, :nb_old] = data["v"]
    return K, V, torch.as_tensor(bt, device=DEV), max(need) * w.block


def token_samples(w, L, n):
    """Pre-RoPE q [n][L][S][Hq][d], k, v [n][L][S][Hkv][d] (bf16) of n new tokens."""
    q = torch.empty((n, L, w.S, w.Hq, w.d), dtype=torch.bfloat16, device=DEV)
    k = torch.empty((n, L, w.S, w.Hkv, w.d), dtype=torch.bfloat16, device=DEV)
    v = torch.empty_like(k)
    for l in range(L):
        for s in range(w.S):
            a, b, c = sequence_samples(w, l, n, device=DEV, tag=f"decode_tokens_{s}")
            q[:, l, s], k[:, l, s], v[:, l, s] = a.to(torch.bfloat16), b.to(torch.bfloat16), c.to(torch.bfloat16)
    return q, k, v


def rows_of(w, K, V, bt, l, s, g, n):
    d = {"k": K, "v": V, "seq_len": torch.full((w.S,), n, dtype=torch.int32), "block_table": bt}
    return (unit_rows(w, d, l, s, g, "k").double().cpu().numpy(), unit_rows(w, d, l, s, g, "v").double().cpu().numpy())


CASES = [
    # (name, paged, block, compact, Hq, Hkv, d, pairing)
    ("dense_ordered_g4", False, 16, "ordered", 8, 2, 128, "half"),
    ("paged16_ordered_g4", True, 16, "ordered", 8, 2, 128, "half"),
    ("paged16_holefill_g4", True, 16, "holefill", 8, 2, 128, "half"),
    ("dense_holefill_g8_d64_inter", False, 16, "holefill", 16, 2, 64, "interleaved"),
    ("paged32_ordered_g2", True, 32, "ordered", 4, 2, 128, "half"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_loop_two_windows(case):
    name, paged, block, compact, Hq, Hkv, d, pairing = case
    B = 256
    w = Workload(name=f"decode_loop_{name}", L=2, S=3, Hq=Hq, Hkv=Hkv, d=d, theta=1e6, dtype="bf16", budget=B,
                 offsets=GEO16, n_keys=300, paged=paged, block=block, pairing=pairing)
    data = generate(w, device=DEV)
    lens0 = [100, 256, 300]          # one unit stays at or below B at the first trigger; rows past
    data["seq_len"] = torch.tensor(lens0, dtype=torch.int32, device=DEV)   # lens0 are stale
    L = data["k"].shape[0]
    steps = 2 * WINDOW
    K, V, bt, cap = grown(w, data, max(max(lens0), B) + WINDOW - min(lens0) + 8)
    cache = tk.KVCache(K, V, data["seq_len"].clone(), Hkv=Hkv, block_table=bt, block=block)
    stats = tk.tri_calibrate_stats(data["q_pre"], pairing=pairing)
    ostats = [O.calibrate(data["q_pre"][l].double().cpu().numpy(), pairing) for l in range(L)]
    pos0 = torch.tensor(lens0, dtype=torch.int32, device=DEV)
    loop = tk.DecodeLoop(cache, stats, w.theta, w.offsets, B, pos0, window=WINDOW, compact=compact, pairing=pairing)
    qs, ks, vs = token_samples(w, L, steps)
    # positions of the keys in every slot, per unit
    slot_pos = {(l, s, g): list(range(lens0[s])) for l in range(L) for s in range(w.S) for g in range(Hkv)}
    check_attn = {0, 77, WINDOW - 1, WINDOW, 2 * WINDOW - 1}
    n_band = 0
    for i in range(steps):
        lens = cache.seq_len.tolist()
        pos = loop.pos.tolist()
        loop.append(ks[i], vs[i])
        if i in (0, WINDOW + 3):
            torch.cuda.synchronize()
            for (l, s, g) in slot_pos:
                kr, vr = rows_of(w, cache.k, cache.v, bt, l, s, g, lens[s] + 1)
                want = O.rope(ks[i, l, s, g].double().cpu().numpy(), float(pos[s]), w.theta, pairing)
                assert np.all(np.abs(kr[lens[s]] - want) <= 2.0 ** -8 * np.abs(want) + 1e-6)
                np.testing.assert_array_equal(vr[lens[s]], vs[i, l, s, g].double().cpu().numpy())
        out = loop.attend(qs[i])
        if i in check_attn:
            torch.cuda.synchronize()
            for (l, s, g) in slot_pos:
                n = lens[s] + 1
                kr, vr = rows_of(w, cache.k, cache.v, bt, l, s, g, n)
                qh = qs[i, l, s, g * w.G:(g + 1) * w.G].double().cpu().numpy()
                ref = O.decode_attention(O.rope(qh, float(pos[s]), w.theta, pairing), kr, vr, d ** -0.5)
                got = out[l, s, g * w.G:(g + 1) * w.G].double().cpu().numpy()
                assert np.abs(got - ref).max() <= 1e-3 * np.abs(ref).max(), (i, l, s, g)
        for (l, s, g), sp in slot_pos.items():
            sp.append(pos[s])
        if loop.advance():
            lens = cache.seq_len.tolist()
            t = loop.pos.tolist()
            torch.cuda.synchronize()
            before = {u: rows_of(w, cache.k, cache.v, bt, *u, lens[u[1]]) for u in slot_pos}
            idx = loop.compress()
            torch.cuda.synchronize()
            assert tk.tri_get_device_status() == 0
            new = cache.seq_len.tolist()
            assert new == [min(n, B) for n in lens]
            for (l, s, g), sp in slot_pos.items():
                kr, vr = before[(l, s, g)]
                N = lens[s]
                c, R, m = H.unit_stats(*ostats[l], g, w.G)
                ref = O.compress_unit(c, R, m, kr, vr, np.array(sp, dtype=np.float64), t[s], list(w.offsets),
                                      w.theta, B, pairing)
                gi = idx[l, s, g].cpu().numpy().astype(np.int64)
                ka, va = rows_of(w, cache.k, cache.v, bt, l, s, g, min(N, B))
                if N <= B:
                    H.check_kept(gi, ref["idx"], ref["a"], B)
                    np.testing.assert_array_equal(ka, kr)
                    continue
                kept = np.sort(gi) if compact == "holefill" else gi
                n_band += H.check_kept(kept, ref["idx"], ref["a"], B)
                if compact == "holefill":
                    assert np.array_equal(gi, O.holefill_layout(kept, B))
                np.testing.assert_array_equal(ka, kr[gi])
                np.testing.assert_array_equal(va, vr[gi])
                slot_pos[(l, s, g)] = [sp[j] for j in gi]
    assert loop.tokens == steps
    assert n_band <= 4
