"""Benchmark of the TriAttention compression step on the Qwen3-8B-shaped full
step (36 layers x 8 KV heads x 32 query heads, d=128, bf16, 16 sequences of
N=2176 keys, budget B=2048, offsets 2^0..2^16).

One step = one call of tri_compress_step over the whole batch (score every key,
GQA z/max, top-B, in-place compaction of K and V), with inputs resident in HBM.
The compaction is in place, so the cache is restored from a pristine copy
before every step (untimed; the 5.1 GB copy also flushes the 126 MB L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle on a
bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import time

# The CPU-oracle leg runs single-threaded: pin numpy's BLAS pool before import.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

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
def oracle_layer(w):
    """Layer 0 of the workload on the CPU with the oracle's statistics (untimed)."""
    from oracle import tri_oracle as O
    from synth import generate_layer

    lay = generate_layer(w, 0, "cpu", with_q=True)
    return lay, O.calibrate(lay["q_pre"].double().numpy(), w.pairing)


def oracle_sample(w, budget_s, max_units=None, seed=0, layer=None):
    """Runs the fp64 oracle on sampled units of layer 0 (generated on the CPU,
    or the given oracle_layer) until budget_s seconds of CPU work; returns
    (keys, seconds, units, threads)."""
    from oracle import tri_oracle as O

    lay, stats = layer if layer is not None else oracle_layer(w)
    rng = np.random.default_rng(seed)
    keys = units = 0
    t0 = time.perf_counter()
    while True:
        s, g = int(rng.integers(w.S)), int(rng.integers(w.Hkv))
        n = lay["seq_len"][s]
        kr = lay["k"][s, g, :n].double().numpy()
        vr = lay["v"][s, g, :n].double().numpy()
        sl = slice(g * w.G, (g + 1) * w.G)
        O.compress_unit(stats[0][sl], stats[1][sl], stats[2][sl], kr, vr, np.arange(n, dtype=np.float64),
                        n, list(w.offsets), w.theta, w.budget, w.pairing)
        keys += n
        units += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_units and units >= max_units):
            return keys, el, units, 1


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = []
    total_keys = 0
    layer = oracle_layer(w)
    for i in range(args.warmup + args.steps):
        keys, el, units, cores = oracle_sample(w, 0.0, max_units=2, seed=1000 + i, layer=layer)
        if i >= args.warmup:
            per_step.append(el)
            total_keys += keys
    T = sum(per_step)
    value = total_keys / T
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * T / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(w, {"sample": "2 units (seq, KV head) of layer 0 per step"}),
            "cpu_baseline": {"value": value, "unit": "keys/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: 2 random units of layer 0 (N=2176 keys each), "
                                       "per-offset route, fp64 numpy, 1 thread"},
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
                                       "--format=csv,noheader,nounits", "-lms", "100"],
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
    (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        if (rec.get("kernel_src_sha1") == kernel_src_hash and rec.get("workload") == workload
                and int(rec.get("layers", layers)) == layers):
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def _select_kernel_name(w, cap, compact):
    """The long-unit select/compact kernel tri_compress_step launches: the
    three-per-SM select2_kernel when its shared memory holds the kept list and,
    for hole-fill, the hole bookkeeping (B + 16 + 4 min(B, cap - B) bytes in a
    4 x 16 KB ring); else select_compact_kernel."""
    B = w.budget
    bcap = -(-min(B, cap) // 32) * 32
    total = 4 * 16384 + 64 + 1024 + 256 + 128 + -(-bcap * 4 // 128) * 128
    hf_ok = compact != "holefill" or B + 16 + 4 * max(min(B, cap - B), 0) <= 4 * 16384
    return "select2_kernel" if total <= 232448 and hf_ok else "select_compact_kernel"


def kernel_src_hash():
    import hashlib
    h = hashlib.sha1()
    for f in ("tri.cu", "tri_path.cuh", "tri_device.cuh", "tri_mma.cuh"):
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


def run_b300(args, w):
    import torch
    import torch.distributed as dist

    import kv_cache_compression_06_b300 as tk
    from synth import generate

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # CPU oracle baseline first (rank 0, N=1), before any GPU work.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and w.name == WORKLOAD:
        keys, el, units, cores = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": keys / el, "unit": "keys/s", "cores": cores, "kind": "oracle",
               "sample": f"{units} random units (seq, KV head) of layer 0, {keys} keys in all, "
                         f"{el:.1f} s; per-offset route, fp64 numpy, 1 thread"}
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    data = generate(w, device=dev)
    cache = tk.KVCache(data["k"], data["v"], data["seq_len"], Hkv=w.Hkv,
                       block_table=data.get("block_table"), block=w.block)
    stats = tk.tri_calibrate_stats(data["q_pre"], pairing=w.pairing)
    del data["q_pre"]
    params = tk.Params(w.theta, data["t"], w.offsets, w.budget, pairing=w.pairing)
    ws = tk.workspace(cache, stats, params)
    launches = 1 if ws is None else 3   # fused kernel, or phases + score tiles + select/compact
    k0, v0 = cache.k.clone(), cache.v.clone()
    L = cache.L
    idx = torch.empty((L, w.S, w.Hkv, w.budget), dtype=torch.int32, device=dev)
    new_len = torch.empty(w.S, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    # A cache smaller than L2 (126 MB) would stay resident across steps: write a
    # 256 MB buffer after each restore so every step starts from a cold L2.
    cache_bytes = 2 * k0.numel() * k0.element_size()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if cache_bytes < (512 << 20) else None

    def restore():
        cache.k.copy_(k0)
        cache.v.copy_(v0)
        if flush is not None:
            flush.fill_(1)

    def step():
        tk.tri_compress_step(cache, stats, params, idx_out=idx, new_len=new_len, ws=ws, stream=stream,
                             compact=args.compact)

    for _ in range(args.warmup):
        restore()
        step()
    torch.cuda.synchronize()
    assert tk.tri_get_device_status() == 0

    # algorithmic bytes: K read for scoring + K/V moved (read + write) by
    # compaction, over the units the step compresses (N > B)
    B, rb = w.budget, w.d * w.esize
    lens = [int(x) for x in data["seq_len"].tolist()]
    M = _moved_rows(idx, data["seq_len"], B) if args.compact == "ordered" else _moved_rows_holefill(idx, data["seq_len"], B)
    units = L * w.S * w.Hkv
    n_keys = L * w.Hkv * sum(lens)
    scored = L * w.Hkv * sum(n for n in lens if n > B)
    units_c = L * w.Hkv * sum(1 for n in lens if n > B)
    alg_bytes = scored * rb + 4 * M * rb
    alg_bytes_full_move = scored * rb + 4 * units_c * B * rb

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        torch.cuda.nvtx.range_push("timed")
        for i in range(args.steps):
            restore()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    if world > 1:
        dist.barrier()
    ms = [a.elapsed_time(b) for a, b in ev]
    t_step = sum(ms) / len(ms) / 1e3
    t_step = max_over_ranks(t_step, dev)
    assert tk.tri_get_device_status() == 0

    # end to end through the public API from pinned host buffers
    e2e = None
    if args.e2e_steps > 0:
        e2e_steps = min(args.steps, args.e2e_steps)
        t_e2e, h2d, d2h = run_e2e(tk, cache, stats, params, k0, v0, idx, new_len, e2e_steps, args.compact)
        e2e = {"value": world * n_keys / t_e2e, "unit": "keys/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "how": "layer-pipelined: layer l's K/V up, layer l-1 compressed, layer l-2's K/V, idx down, "
                      "on three streams"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = _peaks()
    achieved = alg_bytes / t_step / 1e9
    mma = w.dtype == "bf16" and w.pairing == "half"
    if launches == 1:
        kname = f"fused_mma_kernel<{w.d},{w.G}>" if mma else f"fused_kernel<{w.d},{w.G},{w.dtype}>"
    else:
        kname = ("phase_kernel+" + ("score_tiles_mma_kernel" if mma else "score_tiles_kernel")
                 + "+" + _select_kernel_name(w, cache.cap, args.compact))
    line = {
        "metric": METRIC, "value": job_throughput(world, n_keys, t_step), "unit": "keys/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": _config(w, {"layers": L, "compaction": args.compact,
                              "l2": f"cache restored from a pristine {cache_bytes / 1e9:.3f} GB copy before every "
                                    "step" + (" plus a 256 MB L2 flush" if flush is not None else " (flushes L2)")
                                    + "; untimed",
                              "parallelism": f"replicas x{world}"}),
        "compress_step_us": t_step * 1e6,
        "hbm_gbs": achieved,
        "hbm_frac_of_8tbs": achieved / 8000.0,
        "moved_rows": M, "moved_rows_if_all_B": units_c * B, "units": units, "units_compressed": units_c,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": _traffic_record(kernel_src_hash(), w.name, L),
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "algorithmic_bytes_if_all_B_moved": alg_bytes_full_move,
                     "kernel": kname},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clk.summary(),
        "gpu_launches": launches * args.steps,
        "step_ms_min": min(ms), "step_ms_median": float(np.median(ms)),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
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
    args = ap.parse_args()
    from synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(L=args.layers)
    if args.seqs:
        w = w.with_(S=args.seqs)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_b300(args, w)


if __name__ == "__main__":
    main()
