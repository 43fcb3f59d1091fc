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
    w = WORKLOADS["qwen3_8b_36l_b4_n32768"]
    C.run_and_check(w, generate(w, device=DEV), C.sample_units(w, w.L, 8, 4), DEV)


def test_qwen3_32b_paged_sampled_units_layer_subset():
    """Full per-layer shape (64 sequences, ragged N, 16-token pages, G=8, B=1024);
    K+V for all 64 layers (~293 GB) exceeds HBM, so two of the 64 layers are
    generated (each from its own seed, identical to the full workload's)."""
    w = WORKLOADS["qwen3_32b_64l_b64_paged"]
    C.run_and_check(w, generate(w, device=DEV, layers=[0, 37]), C.sample_units(w, 2, 6, 5), DEV)


def test_qwen3_8b_full_step_holefill_sampled_units():
    w = WORKLOADS["qwen3_8b_36l_b16_n2176"]
    C.run_and_check_holefill(w, generate(w, device=DEV, layers=list(range(8))), C.sample_units(w, 8, 24, 6), DEV)
