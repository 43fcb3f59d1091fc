"""Guard regions around every buffer the library reads or writes, checked after
every call, and whole-cache checks of every unit (not only sampled ones).

A mistake in the tail arithmetic of a compaction (whole 32-row chunks, whole
paged blocks) or in an output's indexing would write past a unit's rows, a
buffer's end or into a neighbouring unit, which the per-unit parity tests,
comparing only the rows of the units they check, would not see.  Here K, V (or
the paged pools), idx, new_len, agg, raw and the workspace each sit inside a
larger allocation whose head and tail (4 KB each) hold a byte pattern; after
each call the pattern must be intact.  After the step every unit's kept rows
must equal the pristine rows at its indices, and the rows the step has no
business writing must be unchanged:
  dense: rows at or past min(N, B) of every unit (compaction stores end at B);
  paged: every block of a sequence past its first ceil(B/block) blocks, and
         whole sequences with N <= B.
"""
import pytest
import torch

import kv_cache_compression_06_b300 as tk
from synth import Workload, generate

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
GEO16 = tuple(2 ** i for i in range(17))
GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """Tensors carved out of byte buffers with guard bytes on both sides."""

    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype, fill=None):
        numel = 1
        for x in shape:
            numel *= int(x)
        n = torch.tensor([], dtype=dtype).element_size() * numel
        raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)
        t = raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            t.copy_(fill) if torch.is_tensor(fill) else t.fill_(fill)
        self.bufs.append(raw)
        return t

    def check(self, what):
        torch.cuda.synchronize()
        for i, raw in enumerate(self.bufs):
            assert torch.all(raw[:GUARD] == PATTERN), f"{what}: guard before buffer {i} overwritten"
            assert torch.all(raw[-GUARD:] == PATTERN), f"{what}: guard after buffer {i} overwritten"


def W(name, **kw):
    base = dict(L=2, S=4, Hq=8, Hkv=2, d=128, theta=1e6, dtype="bf16", budget=512, offsets=GEO16)
    base.update(kw)
    return Workload(name=name, **base)


CASES = [
    W("guard_fused_dense", n_range=(300, 1900)),
    W("guard_fused_paged16", n_range=(300, 1900), paged=True),
    W("guard_fused_paged32_d64_g2", Hq=4, d=64, n_range=(300, 1900), paged=True, block=32),
    W("guard_long_dense_g4", n_range=(400, 13000), budget=1024),
    W("guard_long_paged_g8", Hq=16, n_range=(400, 16000), budget=1000, paged=True),
    W("guard_long_paged_hg_g4_h8", Hq=32, Hkv=8, n_range=(400, 9000), budget=1000, paged=True, S=3),
    W("guard_long_f32_d64", d=64, dtype="f32", n_range=(20000, 30000), budget=2000, S=2),
]


@pytest.mark.parametrize("compact", ["ordered", "holefill"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_guards_and_every_unit(w, compact):
    data = generate(w, device=DEV)
    g = Guarded()
    K = g.empty(tuple(data["k"].shape), data["k"].dtype, data["k"])
    V = g.empty(tuple(data["v"].shape), data["v"].dtype, data["v"])
    bt = None if not w.paged else g.empty(tuple(data["block_table"].shape), torch.int32, data["block_table"])
    seq_len = g.empty((w.S,), torch.int32, data["seq_len"])
    t = g.empty((w.S,), torch.int32, data["t"])
    q = data["q_pre"]
    cache = tk.KVCache(K, V, seq_len, Hkv=w.Hkv, block_table=bt, block=w.block)
    stats = tk.tri_calibrate_stats(q, pairing=w.pairing)
    params = tk.Params(w.theta, t, w.offsets, w.budget, pairing=w.pairing)
    L = K.shape[0]
    nws = tk.tri_workspace_bytes(cache, stats, params)
    ws = g.empty((nws,), torch.uint8, 0) if nws else None
    agg = g.empty((L, w.S, w.Hkv, w.cap), torch.float32, 0.0)
    raw = g.empty((L, w.S, w.Hq, w.cap), torch.float32, 0.0)
    tk.tri_score(cache, stats, params, agg=agg, raw=raw, ws=ws)
    g.check("tri_score")
    idx_sel = g.empty((L, w.S, w.Hkv, w.budget), torch.int32, -7)
    tk.tri_select_topb(cache, agg, w.budget, idx=idx_sel)
    g.check("tri_select_topb")
    K0, V0 = K.clone(), V.clone()
    idx = g.empty((L, w.S, w.Hkv, w.budget), torch.int32, -7)
    new_len = g.empty((w.S,), torch.int32, -7)
    tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len, ws=ws, compact=compact)
    g.check("tri_compress_step")
    assert tk.tri_get_device_status() == 0
    lens = data["seq_len"].tolist()
    B = w.budget
    assert new_len.tolist() == [min(n, B) for n in lens]
    for s, n in enumerate(lens):
        m = min(n, B)
        for l in range(L):
            for gh in range(w.Hkv):
                gi = idx[l, s, gh].long()
                if n > B:
                    kept = torch.sort(gi).values if compact == "holefill" else gi
                    assert torch.equal(kept, idx_sel[l, s, gh].long()), (l, s, gh)
                else:
                    assert torch.equal(gi[:n], torch.arange(n, device=DEV)) and torch.all(gi[n:] == -1)
                if not w.paged:
                    assert torch.equal(K[l, s, gh, :m], K0[l, s, gh, gi[:m]]), (l, s, gh)
                    assert torch.equal(V[l, s, gh, :m], V0[l, s, gh, gi[:m]]), (l, s, gh)
                    assert torch.equal(K[l, s, gh, m:], K0[l, s, gh, m:]) and torch.equal(V[l, s, gh, m:], V0[l, s, gh, m:])
                else:
                    nb = -(-n // w.block)
                    blocks = data["block_table"][s, :nb].long()
                    rows = lambda X: X[l, blocks, :, gh, :].reshape(nb * w.block, w.d)[:n]
                    assert torch.equal(rows(K)[:m], rows(K0)[gi[:m]]) and torch.equal(rows(V)[:m], rows(V0)[gi[:m]])
        if w.paged:
            nb = -(-n // w.block)
            keep_b = nb if n <= B else -(-B // w.block)
            tail = data["block_table"][s, keep_b:nb].long()
            assert torch.equal(K[:, tail], K0[:, tail]) and torch.equal(V[:, tail], V0[:, tail]), s
            if n <= B:
                head = data["block_table"][s, :nb].long()
                assert torch.equal(K[:, head], K0[:, head]) and torch.equal(V[:, head], V0[:, head])
    # unfused compaction from the selected indices into a second guarded copy
    K2 = g.empty(tuple(K0.shape), K0.dtype, K0)
    V2 = g.empty(tuple(V0.shape), V0.dtype, V0)
    len2 = g.empty((w.S,), torch.int32, -7)
    other = tk.KVCache(K2, V2, seq_len, Hkv=w.Hkv, block_table=bt, block=w.block)
    tk.tri_compact_kv(other, idx_sel, w.budget, new_len=len2, compact=compact)
    g.check("tri_compact_kv")
    assert torch.equal(len2, new_len)
