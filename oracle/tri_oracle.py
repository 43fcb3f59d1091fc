"""Plain, slow fp64 CPU oracle of the TriAttention periodic KV-compression step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
shares no code with the CUDA library and reads none of its outputs.

Sources (page titles; "§" = section on that page):
  [W3] "实现单卡4090跑通OpenClaw!英伟达&浙大等提出长上下文推理KV压缩新方法TriAttention"
       (yeyulingfeng.com), § 主要方法 (main method).  Its paragraphs, in order:
       [W3-MRL]   Q/K concentration around fixed centers, measured by the mean
                  resultant length R (R -> 1 means concentrated);
       [W3-TRIG]  the RoPE logit as a sum over frequency bands that depends on the
                  query-key distance; with Q/K near their centers it becomes a
                  trigonometric series in that distance;
       [W3-SCORE] two per-key scores: the trigonometric-series score (calibrated
                  Q center against the key's band representation) and the norm
                  score, whose weight falls where a band is concentrated and rises
                  where it is not; the two are fused (the fusion formula itself
                  was lost from the page);
       [W3-PRUNE] averaging over a geometric set of future offsets; pruning every
                  128 generated tokens when the cache exceeds the budget: score all
                  keys, keep the top B; GQA: z-score inside each query head, then
                  max over the heads sharing a KV head.
  [W2] "TriAttention：用三角级数压缩KV缓存，让长推理模型跑在消费级显卡上"
       (zingnex.cn), § TriAttention的核心机制 (Q/K norms as auxiliary signal).

Notation: d head dim, F = d/2 bands, omega_f = theta^(-2f/d), band f of a vector x
is the complex number x_f = x[f] + i*x[f+F] ("half", rotate-half layout) or
x[2f] + i*x[2f+1] ("interleaved").  RoPE at position p multiplies x_f by
e^{i*omega_f*p}.  Stored keys are post-RoPE.

Where the pages are silent or garbled, the readings taken here are:
  * pairing: rotate-half (the Qwen3 layout); interleaved behind a flag;
  * R: mean resultant length of the unit vectors q_f/|q_f| (zero samples skipped);
    the norm statistic is the mean magnitude m = mean |q_f|;
  * trig score: real part of sum_f c_f * conj(k_f) * e^{i*omega_f*(t+o-p)} with the
    query center c of each query head and the actual (un-rotated) key k, no 1/sqrt(d);
  * offsets are relative to the current position t, averaged (mean);
  * norm score: sum_f (1 - R_f) * m_f * |k_f|;
  * fusion: plain sum of the two scores (parity to the paper's lost formula is
    unpinned: nothing on the pages fixes it);
  * z-score with the population standard deviation over all N keys of the unit,
    sigma = 0 gives z = 0; aggregation = max over the G query heads of a KV head;
  * top-B: order by (score descending, slot ascending), NaN lowest, N <= B keeps all;
  * compaction: stable, kept rows to slots 0..B-1 in ascending original slot;
    the hole-fill alternative (holefill_layout) keeps the same set in place
    below B and fills the evicted slots below B with the kept slots above.
"""
from __future__ import annotations

import itertools
import math
from typing import Sequence

import numpy as np


# ----------------------------------------------------------------------------
# RoPE bands  [W3-TRIG]
# ----------------------------------------------------------------------------
def band_frequencies(d: int, theta: float) -> np.ndarray:
    """omega_f = theta^(-2f/d), f = 0..d/2-1 (fp64)."""
    f = np.arange(d // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * f / d)


def to_bands(x: np.ndarray, pairing: str = "half") -> np.ndarray:
    """[..., d] real -> [..., d/2] complex band representation."""
    x = np.asarray(x, dtype=np.float64)
    F = x.shape[-1] // 2
    if pairing == "half":
        return x[..., :F] + 1j * x[..., F:]
    if pairing == "interleaved":
        return x[..., 0::2] + 1j * x[..., 1::2]
    raise ValueError(pairing)


# ----------------------------------------------------------------------------
# RoPE as the model applies it (real 2x2 rotation of each band pair)  [W3-TRIG]
# ----------------------------------------------------------------------------
def rope(x: np.ndarray, pos, theta: float, pairing: str = "half") -> np.ndarray:
    """Rotates x [..., d] to position pos (a scalar, or an array broadcasting
    against x's leading dimensions): the pair (a, b) of band f becomes
    (a*cos(w) - b*sin(w), a*sin(w) + b*cos(w)), w = omega_f * pos.  Written with
    real rotations, independently of to_bands."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    F = d // 2
    om = band_frequencies(d, theta)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * om            # [..., F]
    c, sn = np.cos(ang), np.sin(ang)
    if pairing == "half":
        ia, ib = np.arange(F), np.arange(F) + F
    elif pairing == "interleaved":
        ia, ib = 2 * np.arange(F), 2 * np.arange(F) + 1
    else:
        raise ValueError(pairing)
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (d,)))
    a, b = x[..., ia], x[..., ib]
    out[..., ia] = a * c - b * sn
    out[..., ib] = a * sn + b * c
    return out


# ----------------------------------------------------------------------------
# Offline calibration  [W3-MRL], [W3-PRUNE] ("离线统计 Q/K 中心、范数与集中度")
# ----------------------------------------------------------------------------
def calibrate(q_pre: np.ndarray, pairing: str = "half"):
    """q_pre [n][H][d] pre-RoPE queries -> (center [H][F] complex, R [H][F], m [H][F]).

    center = mean of q_f; m = mean of |q_f|; R = |mean of q_f/|q_f|| over the
    samples with |q_f| > 0 (0 when there are none).
    """
    qb = to_bands(q_pre, pairing)                       # [n][H][F]
    center = qb.mean(axis=0)
    mag = np.abs(qb)
    m = mag.mean(axis=0)
    nz = mag > 0
    unit = np.where(nz, qb / np.where(nz, mag, 1.0), 0.0)
    cnt = nz.sum(axis=0)
    R = np.where(cnt > 0, np.abs(unit.sum(axis=0)) / np.maximum(cnt, 1), 0.0)
    return center, R, m


# ----------------------------------------------------------------------------
# Scores  [W3-TRIG], [W3-SCORE], [W3-PRUNE]
# ----------------------------------------------------------------------------
def trig_score_at_offset(center, k_post, pos, t, o, theta, pairing="half"):
    """T_{h,i}(o) = sum_f Re[c_{h,f} * conj(k_{i,f}) * e^{i*omega_f*(t+o-p_i)}].

    center [G][F] complex; k_post [N][d] stored (post-RoPE) keys; pos [N] their
    positions.  The stored key is first un-rotated to its pre-RoPE band value
    k_{i,f} = k~_{i,f} * e^{-i*omega_f*p_i}.
    """
    d = k_post.shape[-1]
    om = band_frequencies(d, theta)
    pos = np.asarray(pos, dtype=np.float64)
    k_pre = to_bands(k_post, pairing) * np.exp(-1j * om[None, :] * pos[:, None])     # [N][F]
    dist = (float(t) + float(o)) - pos                                                  # [N]
    rot = np.exp(1j * om[None, :] * dist[:, None])                                     # [N][F]
    terms = center[:, None, :] * np.conj(k_pre)[None, :, :] * rot[None, :, :]          # [G][N][F]
    return np.real(terms).sum(axis=-1)


def trig_score(center, k_post, pos, t, offsets: Sequence[int], theta, pairing="half"):
    """Mean over the future offsets of trig_score_at_offset  [W3-PRUNE]."""
    acc = None
    for o in offsets:
        T = trig_score_at_offset(center, k_post, pos, t, o, theta, pairing)
        acc = T if acc is None else acc + T
    return acc / float(len(offsets))


def trig_score_closed_form(center, k_post, t, offsets, theta, pairing="half"):
    """The same average written with the per-band offset sum:
    sum_f Re[c_f * e^{i*omega_f*t} * Phi_f * conj(k~_f)],
    Phi_f = (1/|O|) sum_o e^{i*omega_f*o}, k~ the stored post-RoPE key
    (post-RoPE phase = pre-RoPE phase + omega_f*p, so positions cancel)."""
    d = k_post.shape[-1]
    om = band_frequencies(d, theta)
    offs = np.asarray(list(offsets), dtype=np.float64)
    phi = np.exp(1j * om[:, None] * offs[None, :]).mean(axis=1)                      # [F]
    A = center * np.exp(1j * om * float(t))[None, :] * phi[None, :]                   # [G][F]
    kb = to_bands(k_post, pairing)                                                    # [N][F]
    return np.real(A[:, None, :] * np.conj(kb)[None, :, :]).sum(axis=-1)


def norm_score(R, m, k_post, pairing="half"):
    """N_{h,i} = sum_f (1 - R_{h,f}) * m_{h,f} * |k_{i,f}|  [W3-SCORE], [W2]."""
    kabs = np.abs(to_bands(k_post, pairing))                                          # [N][F]
    W = (1.0 - np.asarray(R, dtype=np.float64)) * np.asarray(m, dtype=np.float64)    # [G][F]
    return W @ kabs.T


def key_scores(center, R, m, k_post, pos, t, offsets, theta, pairing="half"):
    """Fused per-head key score s = trig score + norm score, [G][N]."""
    return (trig_score(center, k_post, pos, t, offsets, theta, pairing)
            + norm_score(R, m, k_post, pairing))


def gqa_aggregate(s: np.ndarray) -> np.ndarray:
    """z-score each query head's scores over the unit's keys (population sigma,
    sigma = 0 -> z = 0), then take the max over the heads  [W3-PRUNE].

    The moments are taken of the scores minus the head's first score (z is
    unchanged by a shift), so a head whose scores are all equal has exactly zero
    deviation and gets z = 0 rather than a rounding artefact of the mean."""
    s = np.asarray(s, dtype=np.float64)
    d = s - s[:, :1]
    mu = d.mean(axis=1, keepdims=True)
    sd = np.sqrt(((d - mu) ** 2).mean(axis=1, keepdims=True))
    z = np.where(sd > 0, (d - mu) / np.where(sd > 0, sd, 1.0), 0.0)
    return np.fmax.reduce(z, axis=0)


def select_topb(a: np.ndarray, B: int) -> np.ndarray:
    """Kept slots, ascending: the B largest a (ties -> lower slot, NaN lowest);
    all slots when N <= B  [W3-PRUNE]."""
    a = np.asarray(a)
    N = a.shape[0]
    if N <= B:
        return np.arange(N, dtype=np.int64)
    def key(i):
        v = a[i]
        return (1, 0.0, i) if np.isnan(v) else (0, -float(v), i)
    order = sorted(range(N), key=key)
    return np.array(sorted(order[:B]), dtype=np.int64)


def select_topb_bruteforce(a: np.ndarray, B: int) -> np.ndarray:
    """Exhaustive reference for tiny N: enumerate every B-subset; keep the one whose
    values, sorted descending, are lexicographically largest (i.e. the multiset of
    the B largest values, NaN counted as -inf); among subsets with equal values,
    the lexicographically smallest slot tuple."""
    a = np.where(np.isnan(a), -np.inf, np.asarray(a, dtype=np.float64))
    N = a.shape[0]
    if N <= B:
        return np.arange(N)
    best, best_sum = None, None
    for comb in itertools.combinations(range(N), B):
        vals = sorted((a[i] for i in comb), reverse=True)
        if best is None or vals > best_sum or (vals == best_sum and comb < best):
            best, best_sum = comb, vals
    return np.array(best)


def compact(x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Ordered compaction: row j of the result is row idx_j of x  [W3-PRUNE]."""
    return np.asarray(x)[np.asarray(idx, dtype=np.int64)]


def holefill_layout(kept: np.ndarray, B: int) -> np.ndarray:
    """Hole-fill compaction layout (an alternative to the ordered one; the pages
    fix only that the top-B keys are kept, W3-PRUNE).  kept: the ascending kept
    slots (len B).  Kept slots below B stay where they are; the evicted slots
    below B (the holes, ascending) receive the kept slots at or above B (the
    movers, ascending), the k-th hole the k-th mover.  Returns src[j], the
    original slot of the row that ends at slot j, for j < B."""
    kept = np.asarray(kept, dtype=np.int64)
    assert kept.shape[0] == B
    inside = kept[kept < B]
    movers = kept[kept >= B]
    holes = np.setdiff1d(np.arange(B), inside)
    assert holes.shape[0] == movers.shape[0]
    src = np.arange(B, dtype=np.int64)
    src[holes] = movers
    return src


# ----------------------------------------------------------------------------
# Distance-preference curves  [W3-TRIG]
# ----------------------------------------------------------------------------
def center_curve(cq: np.ndarray, ck: np.ndarray, d: int, theta: float, n_delta: int) -> np.ndarray:
    """The trigonometric series of one query head against its KV head, from the
    centers: C(delta) = sum_f Re[cq_f * conj(ck_f) * e^{i*omega_f*delta}],
    delta = 0..n_delta-1.  cq, ck: [F] complex."""
    om = band_frequencies(d, theta)
    delta = np.arange(n_delta, dtype=np.float64)
    terms = cq[None, :] * np.conj(ck)[None, :] * np.exp(1j * om[None, :] * delta[:, None])
    return np.real(terms).sum(axis=1)


def logit_curve(q_seq: np.ndarray, k_seq: np.ndarray, theta: float, n_delta: int,
                pairing: str = "half") -> np.ndarray:
    """The exact mean RoPE logit at each distance over one sequence: query
    sample j sits at position j, key sample i at position i, and
    E(delta) = mean over i in [0, n - delta) of rope(q_{i+delta}, i+delta) . rope(k_i, i).
    q_seq, k_seq: [n][d] pre-RoPE samples."""
    n = q_seq.shape[0]
    pos = np.arange(n, dtype=np.float64)
    qr = rope(q_seq, pos, theta, pairing)
    kr = rope(k_seq, pos, theta, pairing)
    out = np.empty(n_delta)
    for dl in range(n_delta):
        out[dl] = np.mean(np.sum(qr[dl:] * kr[: n - dl], axis=1))
    return out


def pearson(a: np.ndarray, b: np.ndarray) -> float:
    """Pearson correlation; 0 when either series is constant."""
    a = np.asarray(a, dtype=np.float64) - np.mean(a)
    b = np.asarray(b, dtype=np.float64) - np.mean(b)
    den = math.sqrt(float(np.sum(a * a)) * float(np.sum(b * b)))
    return float(np.sum(a * b)) / den if den > 0 else 0.0


# ----------------------------------------------------------------------------
# Decode attention over a (compressed) cache  [W3-TRIG] (the RoPE attention
# logit), [W3-PRUNE] (online decoding with window pruning every 128 tokens)
# ----------------------------------------------------------------------------
def decode_attention(q_post: np.ndarray, k_post: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of the G post-RoPE query vectors q_post [G][d] of one
    KV head over its N cached post-RoPE keys k_post [N][d] and values v [N][d]:
    out[h] = sum_i w_{h,i} v_i with w_{h,i} proportional to exp(scale * q_h . k_i),
    normalised over i.  fp64; the largest logit of each head is subtracted
    before exp (the weights are unchanged)."""
    q = np.asarray(q_post, dtype=np.float64)
    k = np.asarray(k_post, dtype=np.float64)
    logits = scale * (q @ k.T)                                        # [G][N]
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = e / e.sum(axis=1, keepdims=True)
    return w @ np.asarray(v, dtype=np.float64)


# ----------------------------------------------------------------------------
# One unit (sequence, layer, KV head) end to end
# ----------------------------------------------------------------------------
def compress_unit(center, R, m, k_post, v, pos, t, offsets, theta, B, pairing="half", route="offsets"):
    """Score -> GQA aggregate -> top-B -> compact for one unit.

    center/R/m: [G][F] statistics of the G query heads of this KV head.
    route: "offsets" scores with the per-offset trig score (keys un-rotated by
    their positions `pos`); "closed" with trig_score_closed_form (the same
    average through the per-band offset sum, positions not needed), which is
    far cheaper for long units.
    Returns dict(s=[G][N], a=[N], idx=[min(N,B)], k=[min(N,B)][d], v=...).
    """
    if route == "offsets":
        s = key_scores(center, R, m, k_post, pos, t, offsets, theta, pairing)
    elif route == "closed":
        s = trig_score_closed_form(center, k_post, t, offsets, theta, pairing) + norm_score(R, m, k_post, pairing)
    else:
        raise ValueError(route)
    a = gqa_aggregate(s)
    idx = select_topb(a, B)
    out = {"s": s, "a": a, "idx": idx, "k": compact(k_post, idx), "v": compact(v, idx)}
    if idx.shape[0] == B and k_post.shape[0] > B:
        hf = holefill_layout(idx, B)
        out.update(hf_src=hf, hf_k=compact(k_post, hf), hf_v=compact(v, hf))
    return out


def paged_logical_rows(pool, block_table_row, g, n, block=16):
    """Rows 0..n-1 of KV head g of one sequence from a paged pool
    [nblocks][block][Hkv][d]: logical slot j lives in block block_table_row[j // block],
    row j % block."""
    out = np.empty((n, pool.shape[-1]), dtype=pool.dtype)
    for j in range(n):
        out[j] = pool[block_table_row[j // block], j % block, g]
    return out
