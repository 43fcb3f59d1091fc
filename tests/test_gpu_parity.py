"""GPU parity: libtri (through the C ABI) against the fp64 oracle on the same
seeded inputs, for the five workloads of the compression step.

Small workloads are generated on the CPU and compared on every unit; the large
ones are generated on the GPU and compared on seeded sampled units (plus the
longest and shortest), whose pristine rows are copied to the host before the
kernels run.  What is compared: tests/_gpu_check.py; tolerances:
tests/_helpers.py.
"""
import pytest
import torch

from synth import WORKLOADS, generate
from tests import _gpu_check as C

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def test_tiny_d64_fp32_every_unit():
    w = WORKLOADS["tiny_d64_gqa2_n1024"]
    C.run_and_check(w, generate(w, device="cpu"), [(0, 0, 0)], DEV)


def test_qwen3_8b_single_layer_every_unit():
    w = WORKLOADS["qwen3_8b_layer_n2176"]
    C.run_and_check(w, generate(w, device="cpu"), [(0, 0, g) for g in range(w.Hkv)], DEV)


def test_qwen3_8b_full_step_sampled_units():
    w = WORKLOADS["qwen3_8b_36l_b16_n2176"]
    C.run_and_check(w, generate(w, device=DEV), C.sample_units(w, w.L, 64, 3), DEV)


def test_qwen3_8b_long_32k_sampled_units():
    """64 sampled units plus the longest and shortest; the oracle scores these
    32768-key units through its closed-form route (pinned equal to the
    per-offset route at rel 1e-9); one unit also through the per-offset route."""
    w = WORKLOADS["qwen3_8b_36l_b4_n32768"]
    data = generate(w, device=DEV)
    units = C.sample_units(w, w.L, 64, 4)
    assert len(units) >= 60
    C.run_and_check(w, data, units, DEV, route="closed")


def test_qwen3_8b_long_32k_per_offset_route():
    w = WORKLOADS["qwen3_8b_36l_b4_n32768"]
    C.run_and_check(w, generate(w, device=DEV, layers=[0, 1]), [(1, 3, 7)], DEV)


def test_qwen3_32b_paged_sampled_units_layer_subset():
    """Full per-layer shape (64 sequences, ragged N, 16-token pages, G=8, B=1024);
    K+V for all 64 layers (~293 GB) exceeds HBM, so four of the 64 layers are
    generated (each from its own seed, identical to the full workload's); 64
    sampled units spread over them plus the longest and shortest sequence."""
    w = WORKLOADS["qwen3_32b_64l_b64_paged"]
    data = generate(w, device=DEV, layers=[0, 21, 37, 63])
    units = C.sample_units(w, 4, 64, 5)
    assert len({u[0] for u in units}) == 4 and len(units) >= 60
    C.run_and_check(w, data, units, DEV, route="closed")


def test_qwen3_8b_full_step_holefill_sampled_units():
    w = WORKLOADS["qwen3_8b_36l_b16_n2176"]
    C.run_and_check_holefill(w, generate(w, device=DEV, layers=list(range(8))), C.sample_units(w, 8, 24, 6), DEV)


ERROR_BUDGET_CASES = [
    ("qwen3_8b_layer_n2176", None),                       # G = 4, fused tensor-core kernel
    ("g8_fused", dict(L=1, S=2, Hq=64, Hkv=8, n_keys=3000, budget=1024)),
    ("g8_long_paged", dict(L=1, S=2, Hq=64, Hkv=8, n_keys=14000, budget=1024, paged=True)),
    ("g4_long", dict(L=1, S=2, Hq=32, Hkv=8, n_keys=14000, budget=2048)),
]


@pytest.mark.parametrize("name,shape", ERROR_BUDGET_CASES, ids=[c[0] for c in ERROR_BUDGET_CASES])
def test_score_error_budget(name, shape):
    """The tensor-core score's error against the fp64 oracle, every unit:
    strict relative error over keys with |s_ref| >= std_h (where the tolerance
    is exactly rel 1e-3), and the error in units of std_h over all keys.  Prints
    both (the numbers quoted for the hi/lo split)."""
    import json
    import numpy as np
    from oracle import tri_oracle as O
    from synth import Workload
    from tests import _helpers as H
    if shape is None:
        w = WORKLOADS[name]
    else:
        w = Workload(name=f"err_budget_{name}", d=128, theta=1e6, dtype="bf16", offsets=tuple(2 ** i for i in range(17)),
                     **shape)
    data = generate(w, device=DEV)
    cache, stats, params = C.setup(w, data, DEV)
    L = data["k"].shape[0]
    raw = torch.zeros((L, w.S, w.Hq, w.cap), dtype=torch.float32, device=DEV)
    agg = torch.zeros((L, w.S, w.Hkv, w.cap), dtype=torch.float32, device=DEV)
    import kv_cache_compression_06_b300 as tk
    from synth import unit_rows
    tk.tri_score(cache, stats, params, agg=agg, raw=raw)
    torch.cuda.synchronize()
    ost = O.calibrate(data["q_pre"][0].double().cpu().numpy(), w.pairing)
    strict = floor = 0.0
    for s in range(w.S):
        for g in range(w.Hkv):
            kr = unit_rows(w, data, 0, s, g, "k").double().cpu().numpy()
            ref = H.oracle_unit(w, ost, kr, kr, g, int(data["t"][s]), route="closed")["s"]
            got = raw[0, s, g * w.G:(g + 1) * w.G, : kr.shape[0]].double().cpu().numpy()
            sd = ref.std(axis=1, keepdims=True)
            err = np.abs(got - ref)
            big = np.abs(ref) >= sd
            strict = max(strict, float((err[big] / np.abs(ref[big])).max()))
            floor = max(floor, float((err / sd).max()))
    print(json.dumps({"score_error_budget": name, "G": w.G, "max_rel_err_where_abs_s_ge_std": strict,
                      "max_err_over_std": floor}))
    assert strict <= 1e-3 and floor <= 1e-3
