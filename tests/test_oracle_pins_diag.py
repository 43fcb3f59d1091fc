"""Pins of the oracle's RoPE and distance-preference functions against routes
that do not share their code: the complex band form of RoPE, explicit 2x2
rotation matrices on tiny inputs, a library correlation, and the identity the
trig-series paragraph rests on (with Q/K at their centers the mean RoPE logit at
distance delta is the trigonometric series of the centers).
"""
import math

import numpy as np
import pytest

from oracle import tri_oracle as O
from synth import WORKLOADS, sequence_samples


@pytest.mark.parametrize("pairing", ["half", "interleaved"])
def test_rope_equals_band_phase_multiplication(pairing):
    rng = np.random.default_rng(30)
    d, theta = 16, 1e4
    x = rng.normal(size=(6, d))
    pos = rng.integers(0, 50000, size=6).astype(np.float64)
    om = O.band_frequencies(d, theta)
    want = O.to_bands(x, pairing) * np.exp(1j * om[None, :] * pos[:, None])
    np.testing.assert_allclose(O.to_bands(O.rope(x, pos, theta, pairing), pairing), want, rtol=1e-9, atol=1e-9)


def test_rope_is_a_rotation_group_in_the_position():
    rng = np.random.default_rng(31)
    x = rng.normal(size=(4, 32))
    a, b = 123.0, 4567.0
    np.testing.assert_allclose(O.rope(x, 0.0, 1e6), x, rtol=0, atol=0)
    np.testing.assert_allclose(O.rope(O.rope(x, a, 1e6), b, 1e6), O.rope(x, a + b, 1e6), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(np.linalg.norm(O.rope(x, a, 1e6), axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)


def test_logit_curve_bruteforce_with_rotation_matrices():
    """n = 5 tokens, d = 4 (two bands), every (query, key) pair at distance
    delta rotated by explicit 2x2 matrices built here."""
    rng = np.random.default_rng(32)
    n, d, theta = 5, 4, 100.0
    q, k = rng.normal(size=(n, d)), rng.normal(size=(n, d))
    om = [theta ** (-2.0 * f / d) for f in range(d // 2)]

    def rot(x, p):
        y = np.empty(d)
        for f in range(d // 2):
            c, s = math.cos(om[f] * p), math.sin(om[f] * p)
            M = np.array([[c, -s], [s, c]])
            y[[f, f + d // 2]] = M @ x[[f, f + d // 2]]
        return y

    want = []
    for dl in range(n):
        vals = [float(rot(q[i + dl], i + dl) @ rot(k[i], i)) for i in range(n - dl)]
        want.append(sum(vals) / len(vals))
    np.testing.assert_allclose(O.logit_curve(q, k, theta, n), want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("pairing", ["half", "interleaved"])
def test_center_curve_is_the_logit_curve_of_samples_at_their_centers(pairing):
    """Every query sample equal to cq and every key sample equal to ck: the mean
    RoPE logit at distance delta is exactly the trig series of the centers."""
    rng = np.random.default_rng(33)
    d, n, theta = 32, 300, 1e4
    F = d // 2
    cq = rng.normal(size=F) + 1j * rng.normal(size=F)
    ck = rng.normal(size=F) + 1j * rng.normal(size=F)

    def vec(c):
        return np.concatenate([c.real, c.imag]) if pairing == "half" else np.stack([c.real, c.imag], 1).ravel()

    q = np.tile(vec(cq), (n, 1))
    k = np.tile(vec(ck), (n, 1))
    np.testing.assert_allclose(O.logit_curve(q, k, theta, 200, pairing), O.center_curve(cq, ck, d, theta, 200),
                               rtol=1e-9, atol=1e-9)


def test_logit_curve_at_distance_zero_is_the_pre_rope_dot_product():
    rng = np.random.default_rng(34)
    q, k = rng.normal(size=(40, 16)), rng.normal(size=(40, 16))
    assert abs(O.logit_curve(q, k, 1e4, 1)[0] - np.mean(np.sum(q * k, axis=1))) < 1e-12


def test_pearson_matches_library_correlation():
    rng = np.random.default_rng(35)
    a, b = rng.normal(size=200), rng.normal(size=200)
    assert abs(O.pearson(a, 0.3 * a + b) - np.corrcoef(a, 0.3 * a + b)[0, 1]) < 1e-12
    assert abs(O.pearson(a, 5 * a + 2) - 1.0) < 1e-12
    assert abs(O.pearson(a, -a) + 1.0) < 1e-12
    assert O.pearson(a, np.ones(200)) == 0.0


def test_concentrated_heads_have_a_predictive_center_curve():
    """The trig-series paragraph's claim on the synthetic recipe: with
    concentrated Q/K (kappa = 16) the center curve tracks the sequence's mean
    logit curve (correlation near 1); with uniform phases (kappa = 0) the
    centers shrink toward 0 and the correlation is low."""
    w = WORKLOADS["qwen3_8b_layer_n2176"].with_(Hq=4, Hkv=1)
    n, nd = 2048, 256
    out = {}
    for kappa in (16.0, 0.0):
        q, k, _ = sequence_samples(w, 0, n, kappa_q=kappa, kappa_k=kappa, tag="curve_pin")
        q, k = q.numpy(), k.numpy()
        cq, _, _ = O.calibrate(q)
        ck, _, _ = O.calibrate(k)
        out[kappa] = [O.pearson(O.center_curve(cq[h], ck[0], w.d, w.theta, nd),
                                O.logit_curve(q[:, h], k[:, 0], w.theta, nd)) for h in range(w.Hq)]
    assert min(out[16.0]) > 0.95, out[16.0]
    assert max(out[0.0]) < 0.5, out[0.0]


# ---------------------------------------------------------------- decode attention
def test_decode_attention_special_cases():
    rng = np.random.default_rng(40)
    N, d = 9, 8
    k, v = rng.normal(size=(N, d)), rng.normal(size=(N, d))
    # q = 0: every logit is 0, uniform weights, the mean of the values
    np.testing.assert_allclose(O.decode_attention(np.zeros((2, d)), k, v, 0.3), np.tile(v.mean(0), (2, 1)),
                               rtol=1e-13)
    # one key: its value, whatever the query
    np.testing.assert_allclose(O.decode_attention(rng.normal(size=(3, d)), k[:1], v[:1], 0.3), np.tile(v[0], (3, 1)),
                               rtol=1e-13)
    # two keys whose logits differ by x: weights 1/(1+e^x) and e^x/(1+e^x)
    q = rng.normal(size=(1, d))
    x = 0.3 * float(q[0] @ (k[1] - k[0]))
    want = (v[0] + math.exp(x) * v[1]) / (1 + math.exp(x))
    np.testing.assert_allclose(O.decode_attention(q, k[:2], v[:2], 0.3)[0], want, rtol=1e-12)
    # a key whose logit exceeds the others by ~1e3: its value, with no overflow
    kk = k.copy()
    kk[4] = 1000.0 * q[0] / float(q[0] @ q[0])
    np.testing.assert_allclose(O.decode_attention(q, kk, v, 1.0)[0], v[4], rtol=1e-12, atol=1e-12)


def test_decode_attention_is_invariant_to_the_slot_order():
    """Keys and values permuted together (as hole-fill compaction reorders
    them) give the same output."""
    rng = np.random.default_rng(41)
    q, k, v = rng.normal(size=(4, 16)), rng.normal(size=(50, 16)), rng.normal(size=(50, 16))
    perm = rng.permutation(50)
    np.testing.assert_allclose(O.decode_attention(q, k[perm], v[perm], 0.25), O.decode_attention(q, k, v, 0.25),
                               rtol=1e-12)
