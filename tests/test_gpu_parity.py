"""GPU parity: libtri (through the C ABI) against the fp64 oracle on the same
seeded inputs, for the five workloads of the compression step.

Small workloads are generated on the CPU and compared on every unit; the large
ones are generated on the GPU and compared on seeded sampled units (plus the
longest and shortest), whose pristine rows are copied to the host before the
kernels run.  Tolerances: see tests/_helpers.py.
"""
import numpy as np
import pytest
import torch

import kv_cache_compression_06_b300 as tk
from oracle import tri_oracle as O
from synth import WORKLOADS, generate, unit_rows
from tests import _helpers as H

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _setup(w, data):
    cache = tk.KVCache(data["k"].to(DEV), data["v"].to(DEV), data["seq_len"].to(DEV), Hkv=w.Hkv,
                       block_table=None if not w.paged else data["block_table"].to(DEV), block=w.block)
    stats = tk.tri_calibrate_stats(data["q_pre"].to(DEV), pairing=w.pairing)
    params = tk.Params(w.theta, data["t"].to(DEV), w.offsets, w.budget, pairing=w.pairing)
    return cache, stats, params


def _oracle_stats(data, li):
    return O.calibrate(data["q_pre"][li].double().cpu().numpy())


def _check_stats(stats, ref, li):
    c, R, m = ref
    gc = stats.center[li].double().cpu().numpy()
    np.testing.assert_allclose(gc[..., 0], c.real, rtol=1e-4, atol=1e-5 * np.abs(c).max())
    np.testing.assert_allclose(gc[..., 1], c.imag, rtol=1e-4, atol=1e-5 * np.abs(c).max())
    np.testing.assert_allclose(stats.R[li].double().cpu().numpy(), R, rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(stats.mag[li].double().cpu().numpy(), m, rtol=1e-4)


def _run_full(w, data, units):
    """Score (agg + raw), select and fused step on the whole workload; compare the
    listed units (li, s, g) with the oracle.  data lives on any device."""
    cache, stats, params = _setup(w, data)
    pristine = {}
    for (li, s, g) in units:
        pristine[(li, s, g)] = (unit_rows(w, data, li, s, g, "k").double().cpu().numpy(),
                                unit_rows(w, data, li, s, g, "v").double().cpu().numpy())
    L = data["k"].shape[0]
    agg = torch.zeros((L, w.S, w.Hkv, w.cap), dtype=torch.float32, device=DEV)
    raw = torch.zeros((L, w.S, w.Hq, w.cap), dtype=torch.float32, device=DEV)
    tk.tri_score(cache, stats, params, agg=agg, raw=raw)
    idx_sel = tk.tri_select_topb(cache, agg, w.budget)
    idx = torch.full((L, w.S, w.Hkv, w.budget), -7, dtype=torch.int32, device=DEV)
    new_len = torch.zeros(w.S, dtype=torch.int32, device=DEV)
    tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len)
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == 0
    out = {"K": cache.k, "V": cache.v}
    ostats = {}
    n_band = 0
    for (li, s, g) in units:
        if li not in ostats:
            ostats[li] = _oracle_stats(data, li)
            _check_stats(stats, ostats[li], li)
        kr, vr = pristine[(li, s, g)]
        N = kr.shape[0]
        t = int(data["t"][s])
        ref = H.oracle_unit(w, ostats[li], kr, vr, g, t)
        H.check_scores(raw[li, s, g * w.G:(g + 1) * w.G, :N].cpu().numpy(), ref["s"])
        H.check_agg(agg[li, s, g, :N].cpu().numpy(), ref["a"])
        gi = idx[li, s, g].cpu().numpy()
        assert np.array_equal(gi, idx_sel[li, s, g].cpu().numpy()), "fused and unfused idx differ"
        n_band += H.check_kept(gi, ref["idx"], ref["a"], w.budget)
        assert int(new_len[s]) == min(N, w.budget)
        if N > w.budget:
            kd = {"k": out["K"], "v": out["V"]}
            k_after = unit_rows(w, {**data, **kd}, li, s, g, "k").double().cpu().numpy()
            v_after = unit_rows(w, {**data, **kd}, li, s, g, "v").double().cpu().numpy()
            H.check_compacted(k_after, kr, gi, w.budget)
            H.check_compacted(v_after, vr, gi, w.budget)
            if np.array_equal(gi, ref["idx"]):
                np.testing.assert_array_equal(k_after[: w.budget], ref["k"])
                np.testing.assert_array_equal(v_after[: w.budget], ref["v"])
    return n_band


def test_tiny_d64_fp32_every_unit():
    w = WORKLOADS["tiny_d64_gqa2_n1024"]
    data = generate(w, device="cpu")
    _run_full(w, data, [(0, 0, 0)])


def test_qwen3_8b_single_layer_every_unit():
    w = WORKLOADS["qwen3_8b_layer_n2176"]
    data = generate(w, device="cpu")
    _run_full(w, data, [(0, 0, g) for g in range(w.Hkv)])


def _sample_units(w, L, n, seed):
    rng = np.random.default_rng(seed)
    lens = w.seq_lengths()
    units = {(int(rng.integers(L)), int(rng.integers(w.S)), int(rng.integers(w.Hkv))) for _ in range(n)}
    units.add((L - 1, int(np.argmax(lens)), w.Hkv - 1))
    units.add((0, int(np.argmin(lens)), 0))
    return sorted(units)


def test_qwen3_8b_full_step_sampled_units():
    w = WORKLOADS["qwen3_8b_36l_b16_n2176"]
    data = generate(w, device=DEV)
    _run_full(w, data, _sample_units(w, w.L, 64, 3))


def test_qwen3_8b_long_32k_sampled_units():
    w = WORKLOADS["qwen3_8b_36l_b4_n32768"]
    data = generate(w, device=DEV)
    _run_full(w, data, _sample_units(w, w.L, 8, 4))


def test_qwen3_32b_paged_sampled_units_layer_subset():
    """Full per-layer shape (64 sequences, ragged N, 16-token pages, G=8, B=1024);
    K+V for all 64 layers (~293 GB) exceeds HBM, so two of the 64 layers are
    generated (each from its own seed, identical to the full workload's)."""
    w = WORKLOADS["qwen3_32b_64l_b64_paged"]
    data = generate(w, device=DEV, layers=[0, 37])
    _run_full(w, data, _sample_units(w, 2, 6, 5))
