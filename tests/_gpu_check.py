"""GPU-versus-oracle check shared by the GPU test files.

run_and_check() runs, through the C ABI, tri_calibrate_stats, tri_score (raw
and aggregated scores), tri_select_topb, tri_compress_step (fused) and
tri_compact_kv (unfused compaction on a copy of the pristine cache, from the
selected indices) on one workload, then compares the listed units with the fp64
oracle on the same seeded inputs (tolerances: tests/_helpers.py):
  calibration stats      rel 1e-4
  raw per-head scores    1e-3 * max(|s|, std_h)
  aggregated scores      1e-3 * max(|a|, 1)
  kept sets              equal outside the tie band around the B-th score
  fused vs unfused idx   identical
  compacted K/V          bit-exact against the pristine rows at the GPU's idx,
                         and identical between the fused and unfused paths
"""
import numpy as np
import torch

import kv_cache_compression_06_b300 as tk
from oracle import tri_oracle as O
from synth import unit_rows
from tests import _helpers as H


def setup(w, data, dev):
    cache = tk.KVCache(data["k"].to(dev), data["v"].to(dev), data["seq_len"].to(dev), Hkv=w.Hkv,
                       block_table=None if not w.paged else data["block_table"].to(dev), block=w.block)
    stats = tk.tri_calibrate_stats(data["q_pre"].to(dev), pairing=w.pairing)
    params = tk.Params(w.theta, data["t"].to(dev), w.offsets, w.budget, pairing=w.pairing)
    return cache, stats, params


def _check_stats(stats, ref, li):
    c, R, m = ref
    gc = stats.center[li].double().cpu().numpy()
    np.testing.assert_allclose(gc[..., 0], c.real, rtol=1e-4, atol=1e-5 * np.abs(c).max())
    np.testing.assert_allclose(gc[..., 1], c.imag, rtol=1e-4, atol=1e-5 * np.abs(c).max())
    np.testing.assert_allclose(stats.R[li].double().cpu().numpy(), R, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(stats.mag[li].double().cpu().numpy(), m, rtol=1e-4)


def run_and_check(w, data, units, dev, unfused=True, route="offsets"):
    """Runs every entry point on the whole workload and checks `units`
    (list of (layer index, sequence, KV head)).  Returns the number of kept-set
    differences that fell inside the tie band."""
    cache, stats, params = setup(w, data, dev)
    pristine = {}
    for (li, s, g) in units:
        pristine[(li, s, g)] = (unit_rows(w, data, li, s, g, "k").double().cpu().numpy(),
                                unit_rows(w, data, li, s, g, "v").double().cpu().numpy())
    L = data["k"].shape[0]
    agg = torch.zeros((L, w.S, w.Hkv, w.cap), dtype=torch.float32, device=dev)
    raw = torch.zeros((L, w.S, w.Hq, w.cap), dtype=torch.float32, device=dev)
    tk.tri_score(cache, stats, params, agg=agg, raw=raw)
    idx_sel = tk.tri_select_topb(cache, agg, w.budget)
    k_copy = v_copy = None
    if unfused:
        k_copy, v_copy = cache.k.clone(), cache.v.clone()
    idx = torch.full((L, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=dev)
    new_len = torch.zeros(w.S, dtype=torch.int32, device=dev)
    tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len)
    if unfused:
        other = tk.KVCache(k_copy, v_copy, cache.seq_len, Hkv=w.Hkv, block_table=cache.block_table,
                           block=w.block)
        len2 = torch.zeros(w.S, dtype=torch.int32, device=dev)
        tk.tri_compact_kv(other, idx_sel, w.budget, new_len=len2)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == 0
    if unfused:
        assert torch.equal(len2, new_len)
    ostats = {}
    n_band = 0
    for (li, s, g) in units:
        if li not in ostats:
            ostats[li] = O.calibrate(data["q_pre"][li].double().cpu().numpy(), w.pairing)
            _check_stats(stats, ostats[li], li)
        kr, vr = pristine[(li, s, g)]
        N = kr.shape[0]
        t = int(data["t"][s])
        ref = H.oracle_unit(w, ostats[li], kr, vr, g, t, route=route)
        H.check_scores(raw[li, s, g * w.G:(g + 1) * w.G, :N].cpu().numpy(), ref["s"])
        H.check_agg(agg[li, s, g, :N].cpu().numpy(), ref["a"])
        gi = idx[li, s, g].cpu().numpy()
        assert np.array_equal(gi, idx_sel[li, s, g].cpu().numpy()), "fused and unfused idx differ"
        n_band += H.check_kept(gi, ref["idx"], ref["a"], w.budget)
        assert int(new_len[s]) == min(N, w.budget)
        kd = {"k": cache.k, "v": cache.v}
        k_after = unit_rows(w, {**data, **kd}, li, s, g, "k").double().cpu().numpy()
        v_after = unit_rows(w, {**data, **kd}, li, s, g, "v").double().cpu().numpy()
        if N > w.budget:
            H.check_compacted(k_after, kr, gi, w.budget)
            H.check_compacted(v_after, vr, gi, w.budget)
            if np.array_equal(gi, ref["idx"]):
                np.testing.assert_array_equal(k_after[: w.budget], ref["k"])
                np.testing.assert_array_equal(v_after[: w.budget], ref["v"])
            if unfused:
                od = {"k": other.k, "v": other.v}
                np.testing.assert_array_equal(
                    unit_rows(w, {**data, **od}, li, s, g, "k").double().cpu().numpy()[: w.budget],
                    k_after[: w.budget])
                np.testing.assert_array_equal(
                    unit_rows(w, {**data, **od}, li, s, g, "v").double().cpu().numpy()[: w.budget],
                    v_after[: w.budget])
        else:
            # untouched units keep every row
            np.testing.assert_array_equal(k_after, kr)
            np.testing.assert_array_equal(v_after, vr)
    return n_band


def sample_units(w, L, n, seed):
    rng = np.random.default_rng(seed)
    lens = w.seq_lengths()
    units = {(int(rng.integers(L)), int(rng.integers(w.S)), int(rng.integers(w.Hkv))) for _ in range(n)}
    units.add((L - 1, int(np.argmax(lens)), w.Hkv - 1))
    units.add((0, int(np.argmin(lens)), 0))
    return sorted(units)


def run_and_check_holefill(w, data, units, dev):
    """Hole-fill layout through tri_compress_step and tri_compact_kv: the kept
    set matches the oracle (tie band), the layout is the oracle's hole-fill
    layout of the GPU's own kept set, every row is bit-exact, and the fused and
    unfused paths agree."""
    cache, stats, params = setup(w, data, dev)
    pristine = {}
    for (li, s, g) in units:
        pristine[(li, s, g)] = (unit_rows(w, data, li, s, g, "k").double().cpu().numpy(),
                                unit_rows(w, data, li, s, g, "v").double().cpu().numpy())
    L = data["k"].shape[0]
    agg = torch.zeros((L, w.S, w.Hkv, w.cap), dtype=torch.float32, device=dev)
    tk.tri_score(cache, stats, params, agg=agg)
    idx_sel = tk.tri_select_topb(cache, agg, w.budget)
    k_copy, v_copy = cache.k.clone(), cache.v.clone()
    idx = torch.full((L, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=dev)
    new_len = torch.zeros(w.S, dtype=torch.int32, device=dev)
    tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len, compact="holefill")
    other = tk.KVCache(k_copy, v_copy, cache.seq_len, Hkv=w.Hkv, block_table=cache.block_table, block=w.block)
    tk.tri_compact_kv(other, idx_sel, w.budget, compact="holefill")
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == 0
    ostats = {}
    for (li, s, g) in units:
        if li not in ostats:
            ostats[li] = O.calibrate(data["q_pre"][li].double().cpu().numpy(), w.pairing)
        kr, vr = pristine[(li, s, g)]
        N = kr.shape[0]
        ref = H.oracle_unit(w, ostats[li], kr, vr, g, int(data["t"][s]))
        gi = idx[li, s, g].cpu().numpy().astype(np.int64)
        gsel = idx_sel[li, s, g].cpu().numpy().astype(np.int64)
        assert int(new_len[s]) == min(N, w.budget)
        if N <= w.budget:
            H.check_kept(gi, ref["idx"], ref["a"], w.budget)
            continue
        assert np.array_equal(np.sort(gi), gsel), "fused and unfused kept sets differ"
        H.check_kept(gsel, ref["idx"], ref["a"], w.budget)
        assert np.array_equal(gi, O.holefill_layout(gsel, w.budget)), "not the hole-fill layout"
        kd = {"k": cache.k, "v": cache.v}
        k_after = unit_rows(w, {**data, **kd}, li, s, g, "k").double().cpu().numpy()
        v_after = unit_rows(w, {**data, **kd}, li, s, g, "v").double().cpu().numpy()
        np.testing.assert_array_equal(k_after[: w.budget], kr[gi])
        np.testing.assert_array_equal(v_after[: w.budget], vr[gi])
        if np.array_equal(gsel, ref["idx"]):
            assert np.array_equal(gi, ref["hf_src"])
            np.testing.assert_array_equal(k_after[: w.budget], ref["hf_k"])
            np.testing.assert_array_equal(v_after[: w.budget], ref["hf_v"])
        od = {"k": other.k, "v": other.v}
        np.testing.assert_array_equal(unit_rows(w, {**data, **od}, li, s, g, "k").double().cpu().numpy()[: w.budget],
                                      k_after[: w.budget])
        np.testing.assert_array_equal(unit_rows(w, {**data, **od}, li, s, g, "v").double().cpu().numpy()[: w.budget],
                                      v_after[: w.budget])
