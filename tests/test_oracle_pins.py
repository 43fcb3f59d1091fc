"""Pins for the fp64 oracle: each test checks it against something other than itself
(textbook RoPE, closed forms, invariants, exhaustive search), chosen so that a
plausible slip (wrong sign of a phase, conj on the wrong operand, wrong band
pairing, sum instead of mean, sample instead of population sigma, wrong tie rule)
fails at least one of them.

Sources: the TriAttention write-up "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
(yeyulingfeng.com), section 主要方法; the pages print no worked numeric example,
so no test vector comes from them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import tri_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- textbook RoPE
def rope_textbook(x, pos, theta, pairing):
    """RoPE as the model applies it, written with real 2x2 rotations.

    rotate-half (Qwen3/NeoX): out = x*cos + rotate_half(x)*sin with
    cos/sin = cat(freqs, freqs), rotate_half(x) = cat(-x2, x1).
    interleaved (GPT-J): each pair (x[2f], x[2f+1]) rotated by angle pos*omega_f.
    """
    d = x.shape[-1]
    inv = 1.0 / (theta ** (np.arange(0, d, 2, dtype=np.float64) / d))
    ang = pos * inv
    if pairing == "half":
        cos = np.concatenate([np.cos(ang), np.cos(ang)])
        sin = np.concatenate([np.sin(ang), np.sin(ang)])
        x1, x2 = x[: d // 2], x[d // 2:]
        rot = np.concatenate([-x2, x1])
        return x * cos + rot * sin
    out = np.empty_like(x)
    for f in range(d // 2):
        c, s = math.cos(ang[f]), math.sin(ang[f])
        a, b = x[2 * f], x[2 * f + 1]
        out[2 * f] = a * c - b * s
        out[2 * f + 1] = a * s + b * c
    return out


@pytest.mark.parametrize("pairing", ["half", "interleaved"])
@pytest.mark.parametrize("d,theta", [(64, 1e4), (128, 1e6), (8, 10.0)])
def test_trig_series_equals_exact_rope_logit_when_q_is_center(pairing, d, theta):
    """[W3-TRIG]: with q equal to its center, the trig-series score at offset o is
    exactly the RoPE logit q~(t+o) . k~(p)."""
    rng = np.random.default_rng(0)
    N = 7
    q = rng.normal(size=d)
    keys_pre = rng.normal(size=(N, d))
    pos = rng.integers(0, 5000, size=N).astype(np.float64)
    k_post = np.stack([rope_textbook(keys_pre[i], pos[i], theta, pairing) for i in range(N)])
    center = O.to_bands(q[None, :], pairing)          # the center IS q
    for t, o in [(5000, 1), (5000, 64), (123, 65536), (0, 3)]:
        got = O.trig_score_at_offset(center, k_post, pos, t, o, theta, pairing)[0]
        qr = rope_textbook(q, t + o, theta, pairing)
        want = k_post @ qr
        np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-9 * np.abs(want).max())


@pytest.mark.parametrize("pairing", ["half", "interleaved"])
def test_offset_average_is_mean_of_exact_logits(pairing):
    """[W3-PRUNE]: the score averages over the future offsets; checked against the
    mean of textbook RoPE logits (catches sum-vs-mean and offset-sign slips)."""
    rng = np.random.default_rng(1)
    d, theta, N = 16, 1e4, 5
    q = rng.normal(size=d)
    kp = rng.normal(size=(N, d))
    pos = np.arange(N, dtype=np.float64) * 3
    k_post = np.stack([rope_textbook(kp[i], pos[i], theta, pairing) for i in range(N)])
    offs = [1, 2, 4, 8, 16]
    t = 40
    want = np.mean([k_post @ rope_textbook(q, t + o, theta, pairing) for o in offs], axis=0)
    got = O.trig_score(O.to_bands(q[None], pairing), k_post, pos, t, offs, theta, pairing)[0]
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("pairing", ["half", "interleaved"])
@pytest.mark.parametrize("d,theta,K", [(64, 1e4, 10), (128, 1e6, 16)])
def test_closed_form_matches_bruteforce_offset_loop(pairing, d, theta, K):
    rng = np.random.default_rng(2)
    G, N = 3, 33
    center = rng.normal(size=(G, d // 2)) + 1j * rng.normal(size=(G, d // 2))
    k_post = rng.normal(size=(N, d))
    pos = np.sort(rng.choice(40000, size=N, replace=False)).astype(np.float64)
    offs = [2 ** i for i in range(K + 1)]
    t = 40000
    bf = O.trig_score(center, k_post, pos, t, offs, theta, pairing)
    cf = O.trig_score_closed_form(center, k_post, t, offs, theta, pairing)
    np.testing.assert_allclose(cf, bf, rtol=1e-9, atol=1e-9 * np.abs(bf).max())


def test_golden_single_band_worked_example():
    """d = 2 (one band, omega_0 = 1 for any theta), c = 1, pre-RoPE keys = 1 at
    positions 0..3, t = 4, offsets {1, 2}, R = 1.  Closed form:
    s_p = (cos(5-p) + cos(6-p)) / 2, norm score 0, keep the top 2 of 4."""
    with open(os.path.join(GOLDEN, "single_band_worked_example.json")) as f:
        g = json.load(f)
    pos = np.array(g["positions"], dtype=np.float64)
    k_post = np.stack([np.cos(pos), np.sin(pos)], axis=1)   # e^{ip} in rotate-half layout
    closed = np.array([(math.cos(5 - p) + math.cos(6 - p)) / 2 for p in pos])
    np.testing.assert_allclose(np.array(g["s"]), closed, rtol=0, atol=1e-12)
    res = O.compress_unit(np.array([[1.0 + 0j]]), np.array([[1.0]]), np.array([[1.0]]),
                          k_post, np.eye(4), pos, g["t"], g["offsets"], g["theta"], g["B"])
    np.testing.assert_allclose(res["s"][0], closed, rtol=0, atol=1e-12)
    assert res["idx"].tolist() == g["idx"]
    np.testing.assert_array_equal(res["k"], k_post[g["idx"]])


# ---------------------------------------------------------------- calibration
def test_R_is_one_for_identical_vectors():
    v = np.random.default_rng(3).normal(size=(1, 2, 64))
    q = np.repeat(v, 50, axis=0) * np.linspace(0.5, 2.0, 50)[:, None, None]   # same direction
    c, R, m = O.calibrate(q)
    np.testing.assert_allclose(R, 1.0, rtol=0, atol=1e-14)
    bands = O.to_bands(v[0])
    np.testing.assert_allclose(m, np.abs(bands) * np.mean(np.linspace(0.5, 2.0, 50)), rtol=1e-13)
    np.testing.assert_allclose(c, bands * np.mean(np.linspace(0.5, 2.0, 50)), rtol=1e-13)


@pytest.mark.parametrize("n", [2, 3, 8, 13])
def test_R_is_zero_for_equally_spaced_phases(n):
    ph = 2 * np.pi * np.arange(n) / n + 0.3
    q = np.zeros((n, 1, 2))
    q[:, 0, 0] = 2.5 * np.cos(ph)
    q[:, 0, 1] = 2.5 * np.sin(ph)
    c, R, m = O.calibrate(q)
    assert abs(R[0, 0]) < 1e-14 and abs(c[0, 0]) < 1e-14
    assert abs(m[0, 0] - 2.5) < 1e-14


@pytest.mark.parametrize("kappa", [0.5, 2.0, 4.0, 20.0])
def test_R_matches_von_mises_mean_resultant_length(kappa):
    """For von Mises(kappa) angles the population R is I1(kappa)/I0(kappa);
    the sample R of n draws is within a few 1/sqrt(n) of it.  Angles drawn by
    numpy's own sampler (independent of the synthetic generator)."""
    from scipy.special import i0e, i1e
    rng = np.random.default_rng(4)
    n = 20000
    ang = rng.vonmises(0.7, kappa, size=(n, 1, 4))
    r = rng.lognormal(0, 0.3, size=(n, 1, 4))
    q = np.concatenate([r * np.cos(ang), r * np.sin(ang)], axis=-1)
    _, R, _ = O.calibrate(q)
    assert np.all(np.abs(R - i1e(kappa) / i0e(kappa)) < 4 / math.sqrt(n))


def test_R_depends_on_directions_only():
    """R is the resultant length of unit vectors, not |center|/mean|q|: opposite
    directions with unequal magnitudes give R = 0 while |c|/m = 0.5."""
    q = np.zeros((2, 1, 2))
    q[0, 0] = [1.0, 0.0]
    q[1, 0] = [-3.0, 0.0]
    c, R, m = O.calibrate(q)
    assert abs(R[0, 0]) < 1e-15
    assert abs(abs(c[0, 0]) / m[0, 0] - 0.5) < 1e-15


def test_R_skips_zero_samples_and_uses_bands_not_elements():
    q = np.zeros((4, 1, 4))
    q[0, 0] = [1, 0, 0, 1]     # band0 = 1, band1 = i
    q[1, 0] = [2, 0, 0, 3]
    # samples 2, 3 are zero vectors -> skipped for R, counted for mean magnitude
    c, R, m = O.calibrate(q)
    np.testing.assert_allclose(R[0], [1.0, 1.0])
    np.testing.assert_allclose(m[0], [3 / 4, 4 / 4])
    np.testing.assert_allclose(c[0], [3 / 4, 4j / 4])


# ---------------------------------------------------------------- norm score
def test_norm_score_special_cases_and_rotation_invariance():
    rng = np.random.default_rng(5)
    d, N, G = 32, 11, 2
    k = rng.normal(size=(N, d))
    m = rng.uniform(0.5, 2, size=(G, d // 2))
    # all R = 1: nothing from the norm term
    assert np.all(O.norm_score(np.ones((G, d // 2)), m, k) == 0)
    # all R = 0, m = 1: sum over bands of |k_f| = hypot of the two halves
    want = np.hypot(k[:, : d // 2], k[:, d // 2:]).sum(axis=1)
    np.testing.assert_allclose(O.norm_score(np.zeros((1, d // 2)), np.ones((1, d // 2)), k)[0], want, rtol=1e-13)
    # |k_f| is unchanged by RoPE: holds only if the pairing matches the rotation
    R = rng.uniform(0, 1, size=(G, d // 2))
    for pairing in ["half", "interleaved"]:
        rot = np.stack([rope_textbook(k[i], 977.0 * i, 1e4, pairing) for i in range(N)])
        np.testing.assert_allclose(O.norm_score(R, m, rot, pairing), O.norm_score(R, m, k, pairing), rtol=1e-12)


def test_norm_score_weight_is_linear_in_the_mean_magnitude_of_its_band():
    """With R = 0 the norm score is sum_f m_f |k_f|: a one-hot m of value c at band
    f gives c times the modulus of that band's (re, im) pair, and nothing from the
    other bands.  Fails if m is dropped (the result would not scale with c), squared
    (it would scale with c^2) or applied to the wrong band."""
    rng = np.random.default_rng(15)
    d, N = 16, 7
    F = d // 2
    k = rng.normal(size=(N, d))
    for pairing in ["half", "interleaved"]:
        for f in [0, 3, F - 1]:
            for c in [0.5, 2.0, 3.0]:
                m = np.zeros((1, F))
                m[0, f] = c
                got = O.norm_score(np.zeros((1, F)), m, k, pairing)[0]
                re_i, im_i = (f, f + F) if pairing == "half" else (2 * f, 2 * f + 1)
                want = [c * math.hypot(k[i, re_i], k[i, im_i]) for i in range(N)]
                np.testing.assert_allclose(got, want, rtol=1e-14)


def test_two_sample_calibration_feeds_the_norm_weight_with_R_below_one():
    """End to end through calibrate -> compress_unit with a band that is not
    concentrated.  One band (d = 2, omega_0 = 1 for any theta); two calibration
    queries q_A = 2 and q_B = 4i, so center c = 1 + 2i, m = (2 + 4) / 2 = 3 and
    R = |(1 + i) / 2| = 1/sqrt(2).  A key of modulus 1 stored post-RoPE at position
    p = t + o with pre-RoPE phase 0 has trig score Re[c] = 1 for the single offset
    o, so s = 1 + (1 - 1/sqrt(2)) * 3 * 1 = 1.878680...  A key of modulus 5 at the
    same phase scores 5 + (1 - 1/sqrt(2)) * 3 * 5.  Dropping m gives 1.29 for the
    first key; squaring it gives 3.64."""
    q = np.zeros((2, 1, 2))
    q[0, 0] = [2.0, 0.0]
    q[1, 0] = [0.0, 4.0]
    c, R, m = O.calibrate(q)
    assert abs(c[0, 0] - (1 + 2j)) < 1e-15
    assert abs(m[0, 0] - 3.0) < 1e-15
    assert abs(R[0, 0] - 1 / math.sqrt(2)) < 1e-15
    t, o, theta = 10, 3, 1e4
    p = t + o
    # post-RoPE keys at position p: pre-RoPE (r, 0) rotated by angle p
    k_post = np.array([[math.cos(p), math.sin(p)], [5 * math.cos(p), 5 * math.sin(p)]])
    res = O.compress_unit(c, R, m, k_post, np.eye(2), np.array([p, p], dtype=np.float64), t, [o], theta, 1)
    w = (1 - 1 / math.sqrt(2)) * 3.0
    np.testing.assert_allclose(res["s"][0], [1 + w, 5 * (1 + w)], rtol=1e-12)


def test_norm_score_weight_falls_with_concentration():
    k = np.ones((1, 4))
    m = np.ones((1, 2))
    lo = O.norm_score(np.array([[0.9, 0.9]]), m, k)[0, 0]
    hi = O.norm_score(np.array([[0.2, 0.2]]), m, k)[0, 0]
    assert hi > lo > 0


# ---------------------------------------------------------------- GQA z / max
def test_zscore_population_moments_and_max():
    rng = np.random.default_rng(6)
    s = rng.normal(3.0, 5.0, size=(4, 101))
    a = O.gqa_aggregate(s)
    z = (s - s.mean(1, keepdims=True)) / s.std(1, keepdims=True)     # numpy std is population
    np.testing.assert_allclose(z.mean(1), 0, atol=1e-12)
    np.testing.assert_allclose((z ** 2).mean(1), 1, rtol=1e-12)
    np.testing.assert_allclose(a, z.max(0), rtol=1e-12)


def test_zscore_invariant_to_per_head_affine_and_G1_is_raw_ranking():
    rng = np.random.default_rng(7)
    s = rng.normal(size=(3, 50))
    s2 = s * np.array([[2.0], [0.01], [7.0]]) + np.array([[5.0], [-3.0], [100.0]])
    np.testing.assert_allclose(O.gqa_aggregate(s2), O.gqa_aggregate(s), rtol=1e-9, atol=1e-12)
    one = s[:1]
    assert O.select_topb(O.gqa_aggregate(one), 20).tolist() == sorted(np.argsort(-one[0], kind="stable")[:20].tolist())


def test_zscore_sigma_zero_gives_zero():
    s = np.vstack([np.full(10, 3.0), np.arange(10.0)])
    a = O.gqa_aggregate(s)
    z1 = (np.arange(10.0) - 4.5) / np.arange(10.0).std()
    np.testing.assert_allclose(a, np.maximum(0.0, z1))


def test_zscore_of_a_constant_head_is_exactly_zero():
    """A value whose running sum is inexact (0.1 * 800 is not 80 in binary):
    the z-score of a constant head is 0/0 and is defined as 0, exactly."""
    s = np.full((2, 800), 0.1)
    s[1] *= -7.3
    assert np.all(O.gqa_aggregate(s) == 0.0)
    naive_mu = s.mean(axis=1, keepdims=True)
    assert np.any(s != naive_mu)   # the unshifted mean is off by rounding here


# ---------------------------------------------------------------- top-B
@pytest.mark.parametrize("seed", range(12))
def test_topb_matches_exhaustive_search(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 11))
    B = int(rng.integers(1, 11))
    a = rng.integers(-3, 4, size=N).astype(np.float64)    # many ties
    if seed % 3 == 0:
        a[rng.integers(0, N)] = np.nan
    assert O.select_topb(a, B).tolist() == O.select_topb_bruteforce(a, B).tolist()


def test_topb_ties_keep_lower_slot_and_nan_lowest():
    a = np.array([1.0, 5.0, 1.0, np.nan, 1.0, 0.0])
    assert O.select_topb(a, 3).tolist() == [0, 1, 2]
    assert O.select_topb(a, 5).tolist() == [0, 1, 2, 4, 5]
    assert O.select_topb(a, 10).tolist() == [0, 1, 2, 3, 4, 5]


# ---------------------------------------------------------------- compaction
def test_inplace_ordered_compaction_equals_gather():
    """Copying rows in increasing destination order inside the same array gives
    the out-of-place gather, because strictly increasing idx has idx_j >= j."""
    rng = np.random.default_rng(8)
    for _ in range(20):
        N = int(rng.integers(1, 60))
        B = int(rng.integers(1, N + 1))
        idx = np.sort(rng.choice(N, size=B, replace=False))
        x = rng.normal(size=(N, 3))
        want = O.compact(x, idx)
        y = x.copy()
        for j, i in enumerate(idx):
            assert i >= j
            y[j] = y[i]
        np.testing.assert_array_equal(y[:B], want)


def test_paged_logical_rows_match_dense_scatter():
    rng = np.random.default_rng(9)
    block, Hkv, d, n = 4, 3, 5, 13
    nb = -(-n // block)
    pool = np.zeros((10, block, Hkv, d))
    table = rng.permutation(10)[:nb]
    dense = rng.normal(size=(Hkv, n, d))
    for j in range(n):
        pool[table[j // block], j % block] = dense[:, j]
    for g in range(Hkv):
        np.testing.assert_array_equal(O.paged_logical_rows(pool, table, g, n, block), dense[g])


# ---------------------------------------------------------------- hole-fill layout
def _holefill_brute(kept, B):
    """Move by move: walk the slots below B in order; each evicted one takes
    the next kept slot at or above B."""
    kept = set(int(i) for i in kept)
    movers = iter(sorted(i for i in kept if i >= B))
    out = []
    for j in range(B):
        out.append(j if j in kept else next(movers))
    return out


@pytest.mark.parametrize("seed", range(10))
def test_holefill_layout_matches_move_by_move_and_keeps_the_set(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(2, 60))
    B = int(rng.integers(1, N))
    kept = np.sort(rng.choice(N, size=B, replace=False))
    src = O.holefill_layout(kept, B)
    assert src.tolist() == _holefill_brute(kept, B)
    assert sorted(src.tolist()) == kept.tolist()                 # same kept set as the ordered layout
    inside = kept[kept < B]
    assert np.all(src[inside] == inside)                         # kept slots below B do not move
    assert int(np.sum(src != np.arange(B))) == int(np.sum(kept >= B))   # one move per kept slot >= B


def test_holefill_rows_and_unit_output():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(12, 3))
    kept = np.array([0, 2, 3, 7, 9, 11])
    src = O.holefill_layout(kept, 6)
    assert src.tolist() == [0, 7, 2, 3, 9, 11]
    np.testing.assert_array_equal(O.compact(x, src), x[[0, 7, 2, 3, 9, 11]])
