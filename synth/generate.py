"""Seeded synthetic Qwen3-shaped KV caches and calibration queries.

The pages that describe TriAttention measure on real model activations
(Qwen3-8B and others on AIME/MATH500); none of that is available here, so these
generators stand in for them.  They reproduce the structure the pages describe
(TriAttention write-up on yeyulingfeng.com, section 主要方法, paragraph on Q/K
concentration): per attention head and per RoPE band, pre-RoPE query and key
vectors cluster around a fixed non-zero center.

Recipe (per layer, per head, per band f):
  * center   = magnitude * e^{i*phase},  magnitude ~ lognormal(0, 0.5),
               phase ~ U[0, 2*pi).  Query centers per query head, key centers
               per KV head.
  * sample   = center * e^{i*phi} * r,   phi ~ von Mises(0, kappa), r ~ N(1, 0.2).
  * keys are stored post-RoPE: band f of the key at position p is multiplied by
    e^{i*omega_f*p}, omega_f = theta^(-2f/d) (the model's position encoding;
    rotate-half band layout x_f = x[f] + i*x[f+d/2] unless 'interleaved').
  * values ~ N(0, 1).
  * calibration queries: n pre-RoPE samples per query head.

This module contains no part of the compression method (no scoring, no
statistics, no selection); it only synthesises what a model would have cached.
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int                     # layers
    S: int                     # sequences
    Hq: int                    # query heads
    Hkv: int                   # KV heads
    d: int                     # head_dim
    theta: float               # RoPE base
    dtype: str                 # 'f32' | 'bf16' (cache storage type)
    budget: int                # B
    offsets: tuple             # future offsets o
    n_keys: Optional[int] = None          # N for every sequence (dense workloads)
    n_range: Optional[tuple] = None       # (lo, hi) inclusive: N_s ~ U[lo, hi]
    paged: bool = False
    block: int = 16
    kappa: float = 4.0                     # angular concentration, all heads
    mixed_R: bool = False                  # 80% heads R~U[.8,.98], 20% R~U[.2,.5]
    outlier_frac: float = 0.0              # fraction of keys scaled by outlier_scale
    outlier_scale: float = 3.0
    n_calib: int = 4096
    pairing: str = "half"                  # 'half' (rotate-half) | 'interleaved'

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def F(self) -> int:
        return self.d // 2

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def seq_lengths(self) -> List[int]:
        if self.n_keys is not None:
            return [self.n_keys] * self.S
        lo, hi = self.n_range
        rng = np.random.default_rng(seed_for(self.name, "lengths"))
        return [int(x) for x in rng.integers(lo, hi + 1, size=self.S)]

    @property
    def cap(self) -> int:
        """Row capacity per unit (dense) or logical rows per sequence (paged)."""
        m = max(self.seq_lengths())
        if self.paged:
            return -(-m // self.block) * self.block
        return m

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _geo(k: int) -> tuple:
    return tuple(2 ** i for i in range(k + 1))


# The five configurations named for the compression step, by what they are.
WORKLOADS: Dict[str, Workload] = {
    # 1 layer, 1 KV head, GQA 2, d=64 (32 bands, theta 1e4), fp32, N=1024, B=256,
    # t=1024, offsets 1..1024.
    "tiny_d64_gqa2_n1024": Workload(
        name="tiny_d64_gqa2_n1024", L=1, S=1, Hq=2, Hkv=1, d=64, theta=1e4,
        dtype="f32", budget=256, offsets=_geo(10), n_keys=1024),
    # Qwen3-8B-shaped single layer, 32/8 heads, d=128, theta 1e6, bf16, batch 1,
    # N=2176 (2048 + one 128-token window), offsets 2^0..2^16, mixed concentration.
    "qwen3_8b_layer_n2176": Workload(
        name="qwen3_8b_layer_n2176", L=1, S=1, Hq=32, Hkv=8, d=128, theta=1e6,
        dtype="bf16", budget=2048, offsets=_geo(16), n_keys=2176, mixed_R=True),
    # Qwen3-8B-shaped full step: 36 layers, batch 16, N=2176, B=2048.
    "qwen3_8b_36l_b16_n2176": Workload(
        name="qwen3_8b_36l_b16_n2176", L=36, S=16, Hq=32, Hkv=8, d=128, theta=1e6,
        dtype="bf16", budget=2048, offsets=_geo(16), n_keys=2176),
    # Long one-shot compression: 36 layers, batch 4, N=32768 -> B=2048, 10% 3x outliers.
    "qwen3_8b_36l_b4_n32768": Workload(
        name="qwen3_8b_36l_b4_n32768", L=36, S=4, Hq=32, Hkv=8, d=128, theta=1e6,
        dtype="bf16", budget=2048, offsets=_geo(16), n_keys=32768, outlier_frac=0.1),
    # Paged mixed batch, Qwen3-32B shapes: 64 layers, 64/8 heads, batch 64,
    # N_s ~ U[2176, 32768], 16-token blocks, random block table, B=1024.
    "qwen3_32b_64l_b64_paged": Workload(
        name="qwen3_32b_64l_b64_paged", L=64, S=64, Hq=64, Hkv=8, d=128, theta=1e6,
        dtype="bf16", budget=1024, offsets=_geo(16), n_range=(2176, 32768), paged=True),
}


def seed_for(*parts) -> int:
    """Stable 31-bit seed from a tuple of names/indices."""
    return zlib.crc32("/".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(*parts))
    return g


def vonmises(kappa: torch.Tensor, shape, gen: torch.Generator) -> torch.Tensor:
    """Angles ~ von Mises(0, kappa) by the Best & Fisher (1979) rejection sampler.

    kappa broadcasts against `shape`; kappa <= 1e-6 draws uniform angles.
    """
    device = gen.device
    kappa = torch.as_tensor(kappa, dtype=torch.float64, device=device).expand(shape).contiguous()
    out = torch.empty(shape, dtype=torch.float64, device=device)
    flat_k = kappa.reshape(-1)
    flat_o = out.reshape(-1)
    todo = torch.arange(flat_k.numel(), device=device)
    tiny = flat_k[todo] <= 1e-6
    if bool(tiny.any()):
        idx = todo[tiny]
        flat_o[idx] = (torch.rand(idx.numel(), generator=gen, device=device, dtype=torch.float64) * 2 - 1) * math.pi
        todo = todo[~tiny]
    while todo.numel() > 0:
        k = flat_k[todo]
        tau = 1.0 + torch.sqrt(1.0 + 4.0 * k * k)
        rho = (tau - torch.sqrt(2.0 * tau)) / (2.0 * k)
        r = (1.0 + rho * rho) / (2.0 * rho)
        u = torch.rand((3, todo.numel()), generator=gen, device=device, dtype=torch.float64)
        z = torch.cos(math.pi * u[0])
        f = (1.0 + r * z) / (r + z)
        c = k * (r - f)
        u2 = u[1].clamp_min(1e-300)
        accept = (c * (2.0 - c) - u2 > 0) | (torch.log(c / u2) + 1.0 - c >= 0)
        ang = torch.sign(u[2] - 0.5) * torch.acos(f.clamp(-1.0, 1.0))
        flat_o[todo[accept]] = ang[accept]
        todo = todo[~accept]
    return out


def _kappa_for_R(R: float) -> float:
    """kappa such that the von Mises mean resultant length I1(k)/I0(k) equals R."""
    from scipy.optimize import brentq
    from scipy.special import i0e, i1e
    return float(brentq(lambda k: i1e(k) / i0e(k) - R, 1e-9, 1e5, xtol=1e-12))


def head_kappas(w: Workload, layer: int, role: str, H: int) -> np.ndarray:
    """Per-head concentration: constant kappa, or the mixed-R recipe."""
    if not w.mixed_R:
        return np.full(H, w.kappa)
    rng = np.random.default_rng(seed_for(w.name, "kappa", role, layer))
    n_low = int(math.floor(0.2 * H + 0.5))
    low = set(rng.permutation(H)[:n_low].tolist())
    out = np.empty(H)
    for h in range(H):
        R = rng.uniform(0.2, 0.5) if h in low else rng.uniform(0.8, 0.98)
        out[h] = _kappa_for_R(R)
    return out


def _centers(gen, shape, device):
    mag = torch.exp(0.5 * torch.randn(shape, generator=gen, device=device, dtype=torch.float64))
    ph = torch.rand(shape, generator=gen, device=device, dtype=torch.float64) * (2 * math.pi)
    return mag * torch.cos(ph), mag * torch.sin(ph)


def _bands_to_vec(re: torch.Tensor, im: torch.Tensor, pairing: str) -> torch.Tensor:
    if pairing == "half":
        return torch.cat([re, im], dim=-1)
    return torch.stack([re, im], dim=-1).flatten(-2)


def _omega(w: Workload, device) -> torch.Tensor:
    f = torch.arange(w.F, device=device, dtype=torch.float64)
    return w.theta ** (-2.0 * f / w.d)


def generate_layer(w: Workload, layer: int, device="cpu", with_q: bool = True):
    """One layer of the workload.

    Returns dict with
      q_pre [n_calib][Hq][d] float32          (pre-RoPE calibration queries)
      k, v  dense: [S][Hkv][cap][d]; paged: per-sequence list is not used here,
            the caller scatters through the block table (see generate()).
      seq_len [S] (python list), positions are 0..N_s-1, t_s = N_s.
    Keys/values are produced in float64 and cast to the storage dtype.
    """
    device = torch.device(device)
    g = _gen(device, w.name, "layer", layer)
    F, d, S, Hq, Hkv = w.F, w.d, w.S, w.Hq, w.Hkv
    lens = w.seq_lengths()
    cap = max(lens)
    qc_re, qc_im = _centers(g, (Hq, F), device)
    kc_re, kc_im = _centers(g, (Hkv, F), device)
    out = {"seq_len": lens}
    if with_q:
        kq = torch.as_tensor(head_kappas(w, layer, "q", Hq), device=device).view(1, Hq, 1)
        phi = vonmises(kq, (w.n_calib, Hq, F), g)
        r = 1.0 + 0.2 * torch.randn((w.n_calib, Hq, F), generator=g, device=device, dtype=torch.float64)
        cre, cim = qc_re.unsqueeze(0), qc_im.unsqueeze(0)
        cs, sn = torch.cos(phi), torch.sin(phi)
        q_re = r * (cre * cs - cim * sn)
        q_im = r * (cre * sn + cim * cs)
        out["q_pre"] = _bands_to_vec(q_re, q_im, w.pairing).to(torch.float32)
        del phi, r, q_re, q_im, cs, sn
    kk = torch.as_tensor(head_kappas(w, layer, "k", Hkv), device=device).view(Hkv, 1, 1)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    K = torch.zeros((S, Hkv, cap, d), dtype=tdt, device=device)
    V = torch.zeros((S, Hkv, cap, d), dtype=tdt, device=device)
    om = _omega(w, device)
    for s in range(S):
        n = lens[s]
        phi = vonmises(kk, (Hkv, n, F), g)
        r = 1.0 + 0.2 * torch.randn((Hkv, n, F), generator=g, device=device, dtype=torch.float64)
        if w.outlier_frac > 0:
            sel = torch.rand((Hkv, n, 1), generator=g, device=device, dtype=torch.float64) < w.outlier_frac
            r = torch.where(sel, r * w.outlier_scale, r)
        cre, cim = kc_re.unsqueeze(1), kc_im.unsqueeze(1)
        cs, sn = torch.cos(phi), torch.sin(phi)
        k_re = r * (cre * cs - cim * sn)
        k_im = r * (cre * sn + cim * cs)
        # store post-RoPE: band f of the key at position p times e^{i*omega_f*p}
        pos = torch.arange(n, device=device, dtype=torch.float64).view(1, n, 1)
        ang = pos * om.view(1, 1, F)
        rc, rs = torch.cos(ang), torch.sin(ang)
        kr_re = k_re * rc - k_im * rs
        kr_im = k_re * rs + k_im * rc
        K[s, :, :n] = _bands_to_vec(kr_re, kr_im, w.pairing).to(tdt)
        V[s, :, :n] = torch.randn((Hkv, n, d), generator=g, device=device, dtype=torch.float32).to(tdt)
        del phi, r, k_re, k_im, kr_re, kr_im, ang, rc, rs
    out["k"] = K
    out["v"] = V
    return out


def _samples(gen, c_re, c_im, kappa, n, device, outlier_frac=0.0, outlier_scale=3.0):
    """n samples per head around the centers [H][F]: center * e^{i*phi} * r,
    phi ~ von Mises(0, kappa_h), r ~ N(1, 0.2) (optionally scaled outliers).
    Returns (re, im) [n][H][F] float64."""
    H, F = c_re.shape
    kap = torch.as_tensor(kappa, dtype=torch.float64, device=device).view(1, H, 1)
    phi = vonmises(kap, (n, H, F), gen)
    r = 1.0 + 0.2 * torch.randn((n, H, F), generator=gen, device=device, dtype=torch.float64)
    if outlier_frac > 0:
        sel = torch.rand((n, H, 1), generator=gen, device=device, dtype=torch.float64) < outlier_frac
        r = torch.where(sel, r * outlier_scale, r)
    cs, sn = torch.cos(phi), torch.sin(phi)
    return r * (c_re * cs - c_im * sn), r * (c_re * sn + c_im * cs)


def sequence_samples(w: Workload, layer: int, n: int, device="cpu", kappa_q=None, kappa_k=None,
                     tag: str = "seq"):
    """Pre-RoPE samples of one sequence of n tokens for one layer: queries
    q [n][Hq][d], keys k [n][Hkv][d] and values v [n][Hkv][d] (float64), drawn
    with the recipe above from centers of their own seed (name, tag, layer).
    kappa_q / kappa_k override the per-head concentration (a scalar or one
    value per head).  Token i sits at position i; nothing here is rotated."""
    device = torch.device(device)
    g = _gen(device, w.name, tag, layer)
    qc = _centers(g, (w.Hq, w.F), device)
    kc = _centers(g, (w.Hkv, w.F), device)
    kq = head_kappas(w, layer, "q", w.Hq) if kappa_q is None else np.broadcast_to(kappa_q, (w.Hq,))
    kk = head_kappas(w, layer, "k", w.Hkv) if kappa_k is None else np.broadcast_to(kappa_k, (w.Hkv,))
    q = _bands_to_vec(*_samples(g, qc[0], qc[1], np.array(kq, dtype=np.float64), n, device), w.pairing)
    k = _bands_to_vec(*_samples(g, kc[0], kc[1], np.array(kk, dtype=np.float64), n, device,
                                w.outlier_frac, w.outlier_scale), w.pairing)
    v = torch.randn((n, w.Hkv, w.d), generator=g, device=device, dtype=torch.float64)
    return q, k, v


def block_table(w: Workload, device="cpu"):
    """Random block table for a paged workload: [S][max_blocks] int32 (unused = 0),
    plus the number of physical blocks per layer pool."""
    lens = w.seq_lengths()
    need = [-(-n // w.block) for n in lens]
    nblocks = sum(need)
    maxb = max(need)
    rng = np.random.default_rng(seed_for(w.name, "block_table"))
    perm = rng.permutation(nblocks)
    bt = np.zeros((w.S, maxb), dtype=np.int32)
    o = 0
    for s, k in enumerate(need):
        bt[s, :k] = perm[o:o + k]
        o += k
    return torch.as_tensor(bt, device=device), nblocks


def generate(w: Workload, device="cpu", layers: Optional[Sequence[int]] = None, with_q: bool = True):
    """Whole-workload tensors on `device`.

    Dense: k, v [Lsel][S][Hkv][cap][d]; paged: k, v pools [Lsel][nblocks][block][Hkv][d]
    with block_table [S][max_blocks].  Also q_pre [Lsel][n][Hq][d] (float32),
    seq_len [S] int32 and t [S] int32 (t_s = N_s: the next query position).
    `layers` selects a subset of layer indices (each generated from its own seed,
    so a subset is bit-identical to the same layers of the full workload).
    """
    layers = list(range(w.L)) if layers is None else list(layers)
    lens = w.seq_lengths()
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    Lsel = len(layers)
    out = {"layers": layers}
    if w.paged:
        bt, nblocks = block_table(w, device)
        out["block_table"] = bt
        out["nblocks"] = nblocks
        K = torch.zeros((Lsel, nblocks, w.block, w.Hkv, w.d), dtype=tdt, device=device)
        V = torch.zeros_like(K)
    else:
        K = torch.empty((Lsel, w.S, w.Hkv, w.cap, w.d), dtype=tdt, device=device)
        V = torch.empty_like(K)
    Q = torch.empty((Lsel, w.n_calib, w.Hq, w.d), dtype=torch.float32, device=device) if with_q else None
    for li, l in enumerate(layers):
        lay = generate_layer(w, l, device, with_q=with_q)
        if with_q:
            Q[li] = lay["q_pre"]
        if w.paged:
            for s, n in enumerate(lens):
                nb = -(-n // w.block)
                rows = torch.zeros((nb * w.block, w.Hkv, w.d), dtype=tdt, device=device)
                rows[:n] = lay["k"][s, :, :n].transpose(0, 1)
                K[li, bt[s, :nb].long()] = rows.view(nb, w.block, w.Hkv, w.d)
                rows.zero_()
                rows[:n] = lay["v"][s, :, :n].transpose(0, 1)
                V[li, bt[s, :nb].long()] = rows.view(nb, w.block, w.Hkv, w.d)
        else:
            K[li] = lay["k"]
            V[li] = lay["v"]
        del lay
    out["k"], out["v"], out["q_pre"] = K, V, Q
    out["seq_len"] = torch.tensor(lens, dtype=torch.int32, device=device)
    out["t"] = torch.tensor(lens, dtype=torch.int32, device=device)
    return out


def unit_rows(w: Workload, data: dict, li: int, s: int, g: int, which: str = "k") -> torch.Tensor:
    """The rows of one unit (sequence s, layer index li, KV head g) in logical slot
    order, [N_s][d], from a generate() result (dense or paged layout)."""
    n = int(data["seq_len"][s])
    X = data[which]
    if not w.paged:
        return X[li, s, g, :n]
    nb = -(-n // w.block)
    blocks = data["block_table"][s, :nb].long()
    return X[li, blocks, :, g, :].reshape(nb * w.block, w.d)[:n]
