"""Benchmark of the TriAttention compression step on the Qwen3-8B-shaped full
step (36 layers x 8 KV heads x 32 query heads, d=128, bf16, 16 sequences of
N=2176 keys, budget B=2048, offsets 2^0..2^16).

One step = one call of tri_compress_step over the whole batch (score every key,
GQA z/max, top-B, in-place compaction of K and V), with inputs resident in HBM.
The compaction is in place, so the cache is restored from a pristine copy
before every step (untimed; the 5.1 GB copy also flushes the 126 MB L2).

The same run also times, each in its own timed region with its own clock
record and algorithmic bytes ("extras"): the hole-fill layout on the same
workload, the long 32k-key workload (36 layers x 4 sequences, both layouts), a
layer group of the paged Qwen3-32B-shaped workload (its 64 layers do not fit
HBM) and the decode loop around the step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle
(closed-form route, one process per host core) on a bounded sample of the same
workload.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import time

# The CPU-oracle leg runs one worker process per host core, each with one BLAS
# thread (set before numpy is imported; spawned workers inherit it).
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "cached keys scored+selected+compacted/sec"
WORKLOAD = "qwen3_8b_36l_b16_n2176"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def _config(w, extra=None):
    c = {"workload": w.name, "layers": w.L, "kv_heads": w.Hkv, "q_heads": w.Hq, "head_dim": w.d,
         "dtype_cache": w.dtype, "batch": w.S, "n_keys": w.n_keys or list(w.n_range), "budget": w.budget,
         "paged_block": w.block if w.paged else None,
         "offsets": f"2^0..2^{int(math.log2(max(w.offsets)))}", "theta": w.theta}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------ CPU oracle leg
_ORACLE_STATE = {}


def _oracle_worker_init(w):
    """Pool initialiser: layer 0 of the workload on the CPU and the oracle's
    statistics for it (untimed; every worker builds its own copy)."""
    from oracle import tri_oracle as O
    from synth import generate_layer

    lay = generate_layer(w, 0, "cpu", with_q=True)
    _ORACLE_STATE["w"] = w
    _ORACLE_STATE["layer"] = lay
    _ORACLE_STATE["stats"] = O.calibrate(lay["q_pre"].double().numpy(), w.pairing)


def _oracle_unit(unit):
    """One unit (sequence s, KV head g of layer 0) through the oracle's
    closed-form route: closed-form trig score + norm score, GQA z/max, top-B,
    ordered compaction of K and V.  Returns the unit's key count."""
    from oracle import tri_oracle as O

    s, g = unit
    w, lay, (c, R, m) = _ORACLE_STATE["w"], _ORACLE_STATE["layer"], _ORACLE_STATE["stats"]
    n = lay["seq_len"][s]
    kr = lay["k"][s, g, :n].double().numpy()
    vr = lay["v"][s, g, :n].double().numpy()
    sl = slice(g * w.G, (g + 1) * w.G)
    sc = O.trig_score_closed_form(c[sl], kr, n, list(w.offsets), w.theta, w.pairing) + O.norm_score(
        R[sl], m[sl], kr, w.pairing)
    idx = O.select_topb(O.gqa_aggregate(sc), w.budget)
    O.compact(kr, idx)
    O.compact(vr, idx)
    return n


class OraclePool:
    """The oracle on every host core: one spawned worker process per core (a
    fresh interpreter, started before any GPU work), each with one BLAS thread."""

    def __init__(self, w, cores=None):
        import multiprocessing as mp
        self.w = w
        self.cores = cores or os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_worker_init, initargs=(w,))
        self.rng = np.random.default_rng(0)
        self.pool.map(_oracle_unit, self._units(self.cores))     # every worker has its layer

    def _units(self, k):
        return [(int(self.rng.integers(self.w.S)), int(self.rng.integers(self.w.Hkv))) for _ in range(k)]

    def run(self, n_units):
        """Runs n_units random units of layer 0; returns (keys, seconds)."""
        units = self._units(n_units)
        t0 = time.perf_counter()
        keys = sum(self.pool.map(_oracle_unit, units, chunksize=1))
        return keys, time.perf_counter() - t0

    def run_for(self, budget_s):
        """Batches of 4 units per core until budget_s seconds; returns (keys, seconds, units)."""
        keys = units = 0
        el = 0.0
        while el < budget_s:
            k, t = self.run(4 * self.cores)
            keys, el, units = keys + k, el + t, units + 4 * self.cores
        return keys, el, units

    def close(self):
        self.pool.close()
        self.pool.join()


def _world():
    return int(os.environ.get("WORLD_SIZE", "1"))


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    pool = OraclePool(w)
    per_step, total_keys = [], 0
    for i in range(args.warmup + args.steps):
        keys, el = pool.run(2 * pool.cores)
        if i >= args.warmup:
            per_step.append(el)
            total_keys += keys
    pool.close()
    T = sum(per_step)
    value = total_keys / T
    sample = (f"per step: {2 * pool.cores} random units (seq, KV head) of layer 0 (N={w.n_keys or 'ragged'} keys each), "
              f"closed-form route, fp64 numpy, {pool.cores} worker processes x 1 thread")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": _world(),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * T / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w, {"sample": sample}),
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": pool.cores, "kind": "oracle",
                             "route": "closed form", "sample": sample},
            "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()
                self.out = ""

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ traffic record
def _traffic_record(kernel_src_hash, workload, layers):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source and this workload
    (else None).  A capture taken on the first `captured_layers` layers (a
    case of a few GB, as ncu captures should be) is scaled to `layers`: every
    layer holds the same units, so the traffic grows in proportion."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        if rec.get("kernel_src_sha1") == kernel_src_hash and rec.get("workload") == workload:
            cl = int(rec.get("captured_layers", rec.get("layers", layers)))
            return float(rec["dram_bytes_per_launch"]) * layers / cl
    except Exception:
        pass
    return None


def _hf_apply(w, compact):
    """Hole-fill rows are moved by holefill_apply_kernel after the selection
    when a unit's list and holes (8 B bytes) fit 56 KB of shared memory."""
    return compact == "holefill" and 8 * w.budget <= 57344


def _select_kernel_name(w, cap, compact):
    """The long-unit select/compact kernels tri_compress_step launches:
    select_only_kernel, then holefill_apply_kernel (hole-fill, when _hf_apply)
    or compact_only_kernel, when the compaction's shared memory (a 6 x 16 KB
    ring, 96 barrier bytes, 256 selection bytes, the kept list) fits 227 KB
    and, for hole-fill by compact_only_kernel, the ring holds the hole
    bookkeeping (B + 16 + 4 min(B, cap - B) bytes, rounded to 128) and 16 KB of
    staging; else select_compact_kernel."""
    B = w.budget
    bcap = -(-min(B, cap) // 32) * 32
    total = 6 * 16384 + 2 * 6 * 8 + 256 + -(-bcap * 4 // 128) * 128
    if total <= 232448 and _hf_apply(w, compact):
        return "select_only_kernel+holefill_apply_kernel"
    hf_ok = compact != "holefill" or -(-(B + 16 + 4 * max(min(B, cap - B), 0)) // 128) * 128 + 16384 <= 6 * 16384
    return "select_only_kernel+compact_only_kernel" if total <= 232448 and hf_ok else "select_compact_kernel"


def kernel_src_hash():
    import hashlib
    h = hashlib.sha1()
    from kv_cache_compression_06_b300.build import CSRC
    for f in CSRC:
        with open(os.path.join(ROOT, "kv_cache_compression_06_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# ------------------------------------------------------------------ ranks
def max_over_ranks(x, device):
    """The largest x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_throughput(world, keys_per_rank, t_step):
    """Whole-job keys/s: every rank compresses its own replica of the workload
    (weak scaling), the step ends when the slowest rank ends."""
    return world * keys_per_rank / t_step


# ------------------------------------------------------------------ GPU leg
def _moved_rows(idx, seq_len, B):
    """Rows each compressed unit actually moves: B minus the untouched prefix
    (idx_j == j), summed over units with N > B."""
    import torch
    ii = idx.view(-1, B).long()
    ar = torch.arange(B, device=ii.device)
    e0 = torch.where((ii != ar).any(dim=1), (ii != ar).int().argmax(dim=1), torch.full_like(ii[:, 0], B))
    L, S, Hkv = idx.shape[0], idx.shape[1], idx.shape[2]
    n = seq_len.long().view(1, S, 1).expand(L, S, Hkv).reshape(-1)
    return int(torch.where(n > B, B - e0, torch.zeros_like(e0)).sum())


def _moved_rows_holefill(idx, seq_len, B):
    """Rows a hole-fill compaction moves: slots j < B whose row came from elsewhere."""
    import torch
    ii = idx.view(-1, B).long()
    ar = torch.arange(B, device=ii.device)
    L, S, Hkv = idx.shape[0], idx.shape[1], idx.shape[2]
    n = seq_len.long().view(1, S, 1).expand(L, S, Hkv).reshape(-1)
    moved = ((ii != ar) & (ii >= 0)).sum(dim=1)
    return int(torch.where(n > B, moved, torch.zeros_like(moved)).sum())


def run_e2e(tk, cache, stats, params, k0, v0, idx, new_len, steps, compact):
    """Seconds per step, end to end: every step copies the whole cache in from
    pinned host memory, compresses it with tri_compress_step one layer at a
    time, and copies K, V, idx and the new lengths back.  Layers are pipelined
    over three streams (PCIe is full duplex): layer l goes up while layer l-1
    is compressed and layer l-2 comes down; a layer's upload waits for the
    previous step's download of the same layer."""
    import torch
    L = cache.L
    hk = torch.empty_like(k0, device="cpu").pin_memory()
    hv = torch.empty_like(v0, device="cpu").pin_memory()
    hk.copy_(k0)
    hv.copy_(v0)
    ok_ = torch.empty_like(hk).pin_memory()
    ov = torch.empty_like(hv).pin_memory()
    oi = torch.empty(idx.shape, dtype=torch.int32).pin_memory()
    on = torch.empty(new_len.shape, dtype=torch.int32).pin_memory()
    layers = [tk.KVCache(cache.k[l:l + 1], cache.v[l:l + 1], cache.seq_len, Hkv=cache.Hkv,
                         block_table=cache.block_table, block=cache.block) for l in range(L)]
    lstats = [tk.Stats(stats.center[l:l + 1], stats.R[l:l + 1], stats.mag[l:l + 1]) for l in range(L)]
    ws = tk.workspace(layers[0], lstats[0], params)
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_cmp = [torch.cuda.Event() for _ in range(L)]
    ev_out = [torch.cuda.Event() for _ in range(L)]
    ev_len = torch.cuda.Event()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for it in range(steps):
        if it > 0:
            s_cmp.wait_event(ev_len)   # the previous step's new lengths are down
        for l in range(L):
            if it > 0:
                s_in.wait_event(ev_out[l])
            with torch.cuda.stream(s_in):
                cache.k[l].copy_(hk[l], non_blocking=True)
                cache.v[l].copy_(hv[l], non_blocking=True)
                ev_in[l].record(s_in)
            s_cmp.wait_event(ev_in[l])
            tk.tri_compress_step(layers[l], lstats[l], params, idx_out=idx[l:l + 1], new_len=new_len, ws=ws,
                                 stream=s_cmp, compact=compact)
            ev_cmp[l].record(s_cmp)
            s_out.wait_event(ev_cmp[l])
            with torch.cuda.stream(s_out):
                ok_[l].copy_(cache.k[l], non_blocking=True)
                ov[l].copy_(cache.v[l], non_blocking=True)
                oi[l].copy_(idx[l], non_blocking=True)
                ev_out[l].record(s_out)
        with torch.cuda.stream(s_out):
            on.copy_(new_len, non_blocking=True)
            ev_len.record(s_out)
    torch.cuda.synchronize()
    t = (time.perf_counter() - t0) / steps
    h2d = hk.numel() * hk.element_size() + hv.numel() * hv.element_size()
    d2h = h2d + oi.numel() * 4 + on.numel() * 4
    return t, h2d, d2h


def _step_kernels(w, cap, compact, fused):
    """The kernels one tri_compress_step launches, in order (fused: the unit's
    scores fit one CTA's shared memory; idx_out is always given here)."""
    if fused:
        mma = w.dtype == "bf16" and w.pairing == "half"
        k = f"fused_mma_kernel<{w.d},{w.G}>" if mma else f"fused_kernel<{w.d},{w.G},{w.dtype}>"
        return [k] + (["holefill_apply_kernel"] if _hf_apply(w, compact) else [])
    mma = w.dtype == "bf16" and w.pairing == "half"
    # paged d = 128 caches whose block holds 128 head-rows: every KV head of a block per copy
    heads = mma and w.paged and w.d == 128 and w.Hkv * w.block == 128 and w.block % 16 == 0
    score = "score_heads_mma_kernel" if heads else ("score_keys_mma_kernel" if mma else "score_tiles_kernel")
    return ["phase_kernel", score] + _select_kernel_name(w, cap, compact).split("+")


def _kernel_name(w, cap, compact, fused):
    return "+".join(_step_kernels(w, cap, compact, fused))


class Measured:
    """One workload on the GPU: generated, calibrated, restorable, timed."""

    def __init__(self, tk, w, dev):
        import torch
        from synth import generate
        self.tk, self.w, self.dev = tk, w, dev
        self.data = generate(w, device=dev)
        d = self.data
        self.cache = tk.KVCache(d["k"], d["v"], d["seq_len"], Hkv=w.Hkv, block_table=d.get("block_table"),
                                block=w.block)
        self.stats = tk.tri_calibrate_stats(d["q_pre"], pairing=w.pairing)
        d["q_pre"] = None
        self.params = tk.Params(w.theta, d["t"], w.offsets, w.budget, pairing=w.pairing)
        self.ws = tk.workspace(self.cache, self.stats, self.params)
        self.fused = self.ws is None   # the unit's scores fit one CTA's shared memory
        self.k0, self.v0 = self.cache.k.clone(), self.cache.v.clone()
        self.L = self.cache.L
        self.idx = torch.empty((self.L, w.S, w.Hkv, w.budget), dtype=torch.int32, device=dev)
        self.new_len = torch.empty(w.S, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()
        # A cache smaller than L2 (126 MB) would stay resident across steps: write
        # a 256 MB buffer after each restore so every step starts from a cold L2.
        self.cache_bytes = 2 * self.k0.numel() * self.k0.element_size()
        self.flush = (torch.empty(256 << 20, dtype=torch.uint8, device=dev)
                      if self.cache_bytes < (512 << 20) else None)

    def launches(self, compact):
        return len(_step_kernels(self.w, self.cache.cap, compact, self.fused))

    def restore(self):
        self.cache.k.copy_(self.k0)
        self.cache.v.copy_(self.v0)
        if self.flush is not None:
            self.flush.fill_(1)

    def step(self, compact):
        self.tk.tri_compress_step(self.cache, self.stats, self.params, idx_out=self.idx, new_len=self.new_len,
                                  ws=self.ws, stream=self.stream, compact=compact)

    def time(self, compact, steps, warmup, world, local, min_region_s=0.0):
        """Mean seconds per step (max over ranks), per-step ms, clock summary.
        With min_region_s > 0 the step count grows until the timed region
        (restores included) lasts about that long, so that the clock sampler
        sees it."""
        import torch
        import torch.distributed as dist
        for _ in range(warmup):
            self.restore()
            self.step(compact)
        torch.cuda.synchronize()
        assert self.tk.tri_get_device_status() == 0
        if min_region_s > 0:
            t0 = time.perf_counter()
            self.restore()
            self.step(compact)
            torch.cuda.synchronize()
            steps = max(steps, int(math.ceil(min_region_s / max(time.perf_counter() - t0, 1e-6))))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            torch.cuda.nvtx.range_push("timed")
            for i in range(steps):
                self.restore()
                ev[i][0].record(self.stream)
                self.step(compact)
                ev[i][1].record(self.stream)
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_pop()
        if world > 1:
            dist.barrier()
        ms = [a.elapsed_time(b) for a, b in ev]
        t_step = max_over_ranks(sum(ms) / len(ms) / 1e3, self.dev)
        assert self.tk.tri_get_device_status() == 0
        return t_step, ms, clk.summary()

    def bytes(self, compact):
        """Algorithmic bytes of the last step: K read for scoring + K/V moved
        (read + write) by compaction, over the units the step compresses (N > B)."""
        w = self.w
        B, rb = w.budget, w.d * w.esize
        lens = [int(x) for x in self.data["seq_len"].tolist()]
        M = (_moved_rows(self.idx, self.data["seq_len"], B) if compact == "ordered"
             else _moved_rows_holefill(self.idx, self.data["seq_len"], B))
        scored = self.L * w.Hkv * sum(n for n in lens if n > B)
        units_c = self.L * w.Hkv * sum(1 for n in lens if n > B)
        return {"alg_bytes": scored * rb + 4 * M * rb, "alg_bytes_all_B": scored * rb + 4 * units_c * B * rb,
                "moved_rows": M, "moved_rows_if_all_B": units_c * B, "units": self.L * w.S * w.Hkv,
                "units_compressed": units_c, "n_keys": self.L * w.Hkv * sum(lens)}

    def free(self):
        for a in ("data", "cache", "stats", "params", "ws", "k0", "v0", "idx", "new_len", "flush"):
            setattr(self, a, None)
        import torch
        torch.cuda.empty_cache()


def _extra(m, compact, steps, warmup, world, local, peak, note):
    """A workload timed in its own region: throughput, roofline fraction,
    algorithmic bytes and its own clock record."""
    t, ms, clocks = m.time(compact, steps, warmup, world, local, min_region_s=0.3)
    steps = len(ms)
    b = m.bytes(compact)
    ach = b["alg_bytes"] / t / 1e9
    l2 = (f"cache restored from a pristine {m.cache_bytes / 1e9:.3f} GB copy before every step"
          + (" plus a 256 MB L2 flush" if m.flush is not None else " (flushes L2)") + "; untimed")
    return {"config": _config(m.w, {"layers": m.L, "compaction": compact, "note": note, "l2": l2}),
            "value": job_throughput(world, b["n_keys"], t), "unit": "keys/s", "ms_per_step": t * 1e3,
            "steps": steps, "warmup": warmup, "step_ms_min": min(ms), "step_ms_median": float(np.median(ms)),
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                         "algorithmic_bytes_per_launch": b["alg_bytes"],
                         "algorithmic_bytes_if_all_B_moved": b["alg_bytes_all_B"],
                         "kernel": _kernel_name(m.w, m.cache.cap, compact, m.fused)},
            "moved_rows": b["moved_rows"], "units_compressed": b["units_compressed"],
            "gpu_launches": m.launches(compact) * steps, "clocks": clocks}


def decode_leg(tk, dev, windows, warmup_windows, world, local, peak, layers=None):
    """The decode loop around the step on Qwen3-8B shapes (36 layers, 32/8 heads,
    d = 128, bf16, 16 sequences, paged 16-token blocks, B = 2048): every token
    appends K/V to all units and attends (tri_append_kv + tri_decode_attention
    over all 36 layers at once), every 128 tokens tri_compress_step runs.  The
    caches start at N = B, so each window grows them to 2176 and the step brings
    them back to 2048 (the steady state of the benchmark workload).  Times the
    decode tokens and the step of each window with CUDA events; the overhead is
    the step's time over the window's decode time."""
    import torch
    from synth import WORKLOADS, generate
    w = WORKLOADS[WORKLOAD].with_(name="decode_loop_qwen3_8b_36l_b16_paged", paged=True, block=16)
    if layers:
        w = w.with_(L=layers)
    window, B = 128, w.budget
    data = generate(w, device=dev)                       # 2176 rows per sequence
    cache = tk.KVCache(data["k"], data["v"], torch.full((w.S,), B, dtype=torch.int32, device=dev), Hkv=w.Hkv,
                       block_table=data["block_table"], block=w.block)
    stats = tk.tri_calibrate_stats(data["q_pre"], pairing=w.pairing)
    data["q_pre"] = None
    pos = torch.full((w.S,), B, dtype=torch.int32, device=dev)
    loop = tk.DecodeLoop(cache, stats, w.theta, w.offsets, B, pos, window=window)
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    qs = torch.randn((window, w.L, w.S, w.Hq, w.d), generator=g, device=dev).to(torch.bfloat16)
    ks = torch.randn((window, w.L, w.S, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
    vs = torch.randn((window, w.L, w.S, w.Hkv, w.d), generator=g, device=dev).to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    loop.stream = stream

    def run_window(evs=None):
        if evs is not None:
            evs[0].record(stream)
        for i in range(window):
            loop.append(ks[i], vs[i])
            loop.attend(qs[i])
            trigger = loop.advance()
        if evs is not None:
            evs[1].record(stream)
        assert trigger
        loop.compress()
        if evs is not None:
            evs[2].record(stream)

    for _ in range(warmup_windows):
        run_window()
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == 0
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(windows)]
    with ClockSampler(local) as clk:
        torch.cuda.nvtx.range_push("timed")
        for e in evs:
            run_window(e)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    assert tk.tri_get_device_status() == 0
    dec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    cmp_ms = [e[1].elapsed_time(e[2]) for e in evs]
    d_tok = sum(dec_ms) / len(dec_ms) / window
    d_cmp = sum(cmp_ms) / len(cmp_ms)
    rb = w.d * w.esize
    units = w.L * w.S * w.Hkv
    # decode-step bytes: every unit reads its N K and V rows (N = 2049..2176 over
    # the window, mean 2112.5) and writes one K and one V row
    dec_bytes = units * (2 * rb * (B + (window + 1) / 2.0) + 2 * rb)
    M = _moved_rows(loop.idx, torch.full((w.S,), B + window, dtype=torch.int32, device=dev), B)
    cmp_bytes = units * (B + window) * rb + 4 * M * rb
    d_ach = dec_bytes / (d_tok * 1e-3) / 1e9
    c_ach = cmp_bytes / (d_cmp * 1e-3) / 1e9
    res = {"config": {"workload": w.name, "layers": w.L, "batch": w.S, "q_heads": w.Hq, "kv_heads": w.Hkv,
                      "head_dim": w.d, "budget": B, "window": window, "paged_block": w.block,
                      "start_len": B, "note": "steady state: each window grows N from 2048 to 2176, the step "
                                              "compresses back to 2048; inputs resident in HBM"},
           "windows": windows, "warmup_windows": warmup_windows,
           "decode_ms_per_token": d_tok, "compress_ms_per_trigger": d_cmp,
           "overhead_frac": d_cmp / (window * d_tok),
           "tokens_per_s": w.S * window / ((window * d_tok + d_cmp) * 1e-3),
           "decode_roofline": {"bound": "hbm", "achieved": d_ach, "peak": peak, "unit": "GB/s",
                               "frac": d_ach / peak, "algorithmic_bytes_per_token": dec_bytes,
                               "kernels": "append_kv_kernel + decode_attn_kernel<128,4>"},
           "compress_roofline": {"bound": "hbm", "achieved": c_ach, "peak": peak, "unit": "GB/s",
                                 "frac": c_ach / peak, "algorithmic_bytes_per_launch": cmp_bytes},
           "gpu_launches": windows * (2 * window + (1 if loop.cmp_ws is None else 3)),
           "clocks": clk.summary()}
    del loop, cache, stats, data, qs, ks, vs
    torch.cuda.empty_cache()
    return res


def run_b300(args, w):
    import torch
    import torch.distributed as dist

    import kv_cache_compression_06_b300 as tk
    from synth import WORKLOADS

    world = _world()
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # CPU oracle baseline first (rank 0, N=1), before any GPU work: the worker
    # processes are spawned, not forked from a CUDA process.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and w.name == WORKLOAD:
        pool = OraclePool(w)
        keys, el, units = pool.run_for(args.cpu_seconds)
        pool.close()
        cpu = {"value": keys / el, "unit": "keys/s", "cores": pool.cores, "kind": "oracle", "route": "closed form",
               "sample": f"{units} random units (seq, KV head) of layer 0, {keys} keys in all, {el:.1f} s wall on "
                         f"{pool.cores} worker processes (os.cpu_count()) x 1 BLAS thread; closed-form route, "
                         f"fp64 numpy"}
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    peak, peak_kind = _peaks()

    m = Measured(tk, w, dev)
    t_step, ms, clocks = m.time(args.compact, args.steps, args.warmup, world, local)
    b = m.bytes(args.compact)
    head_kernel = _kernel_name(w, m.cache.cap, args.compact, m.fused)
    head_launches, head_L = m.launches(args.compact), m.L
    l2_note = (f"cache restored from a pristine {m.cache_bytes / 1e9:.3f} GB copy before every step"
               + (" plus a 256 MB L2 flush" if m.flush is not None else " (flushes L2)") + "; untimed")

    # end to end through the public API from pinned host buffers
    e2e = None
    if args.e2e_steps > 0:
        e2e_steps = min(args.steps, args.e2e_steps)
        t_e2e, h2d, d2h = run_e2e(tk, m.cache, m.stats, m.params, m.k0, m.v0, m.idx, m.new_len, e2e_steps,
                                  args.compact)
        e2e = {"value": world * b["n_keys"] / t_e2e, "unit": "keys/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "how": "layer-pipelined: layer l's K/V up, layer l-1 compressed, layer l-2's K/V, idx down, "
                      "on three streams"}

    extras = {}
    if args.extras and w.name == WORKLOAD and args.layers is None and args.seqs is None:
        other = "holefill" if args.compact == "ordered" else "ordered"
        extras[f"{w.name}/{other}"] = _extra(m, other, args.steps, args.warmup, world, local, peak,
                                             "same cache and step, the other compaction layout")
        m.free()
        m = Measured(tk, WORKLOADS["qwen3_8b_36l_b4_n32768"], dev)
        extras["qwen3_8b_36l_b4_n32768"] = _extra(m, "ordered", args.extra_steps, args.warmup, world, local, peak,
                                                  "long one-shot compression, 32768 -> 2048 keys")
        extras["qwen3_8b_36l_b4_n32768/holefill"] = _extra(m, "holefill", args.extra_steps, args.warmup, world,
                                                           local, peak, "same cache and step, hole-fill layout")
        m.free()
        pw = WORKLOADS["qwen3_32b_64l_b64_paged"]
        m = Measured(tk, pw.with_(L=args.paged_layers), dev)
        extras[f"qwen3_32b_64l_b64_paged/layers0-{args.paged_layers - 1}"] = _extra(
            m, "ordered", args.extra_steps, args.warmup, world, local, peak,
            f"layer group of {args.paged_layers} of the 64 layers (K+V of all 64, ~293 GB, exceed HBM); every "
            "layer has the same lengths and block table, so the group's per-key throughput is the step's")
        m.free()
        extras["decode_loop_qwen3_8b_36l_b16_paged"] = decode_leg(tk, dev, args.decode_windows, 1, world, local,
                                                                 peak)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    achieved = b["alg_bytes"] / t_step / 1e9
    line = {
        "metric": METRIC, "value": job_throughput(world, b["n_keys"], t_step), "unit": "keys/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "accum": "f32",
        "data": "synthetic",
        "config": _config(w, {"layers": head_L, "compaction": args.compact,
                              "l2": l2_note,
                              "parallelism": f"replicas x{world}"}),
        "compress_step_us": t_step * 1e6,
        "hbm_gbs": achieved,
        "hbm_frac_of_8tbs": achieved / 8000.0,
        "moved_rows": b["moved_rows"], "moved_rows_if_all_B": b["moved_rows_if_all_B"], "units": b["units"],
        "units_compressed": b["units_compressed"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": _traffic_record(kernel_src_hash(), w.name, w.L),
                     "algorithmic_bytes_per_launch": b["alg_bytes"],
                     "algorithmic_bytes_if_all_B_moved": b["alg_bytes_all_B"],
                     "kernel": head_kernel},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": head_launches * args.steps,
        "step_ms_min": min(ms), "step_ms_median": float(np.median(ms)),
        "extras": extras or None,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1,
                    help="GPUs of this run; for N > 1 launch one rank per GPU with torchrun (WORLD_SIZE must be N)")
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-steps", type=int, default=3,
                    help="end-to-end steps from pinned host buffers (0: skip; the host needs 4x the cache size)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name (default: the 36-layer Qwen3-8B-shaped batch-16 step)")
    ap.add_argument("--layers", type=int, default=None,
                    help="use only the first N layers (small case for ncu captures, or a layer group "
                         "of a workload whose full cache exceeds HBM)")
    ap.add_argument("--compact", default="ordered", choices=["ordered", "holefill"],
                    help="layout of the kept rows (default: ordered, the slot order of the kept keys)")
    ap.add_argument("--seqs", type=int, default=None,
                    help="use only N sequences (small case for ncu captures)")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="time only the headline workload (skip the hole-fill, long and paged extras)")
    ap.add_argument("--extra-steps", type=int, default=20, help="timed steps of each extra workload")
    ap.add_argument("--decode-windows", type=int, default=2,
                    help="timed 128-token windows of the decode-loop extra")
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the decode-loop workload and print its record (for profiling)")
    ap.add_argument("--paged-layers", type=int, default=8,
                    help="layers of the paged Qwen3-32B-shaped workload timed as its extra (a layer group)")
    args = ap.parse_args()
    if args.gpus != _world():
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {_world()}; for N > 1 launch one rank "
                         "per GPU with `python -m torch.distributed.run --nproc-per-node N bench.py --gpus N`\n")
        sys.exit(2)
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(L=args.layers)
    if args.seqs:
        w = w.with_(S=args.seqs)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.decode_only:
        import torch
        import kv_cache_compression_06_b300 as tk
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        res = decode_leg(tk, torch.device("cuda", local), args.decode_windows, 1, 1, local, _peaks()[0],
                         layers=args.layers)
        print(json.dumps(res), flush=True)
    else:
        run_b300(args, w)


if __name__ == "__main__":
    main()
