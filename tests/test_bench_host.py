"""Host-side checks of bench.py that need no GPU.

The bench line names the kernels a step launches; for long units that name
follows the library's own rule for choosing select_only_kernel +
compact_only_kernel or + holefill_apply_kernel (the compaction's shared-memory
layout and ring size, the hole-fill kernel's shared-memory cap).  These tests restate that rule from the constants in the
CUDA sources and check bench.py's copy of it, so the two cannot drift apart.
"""
import os
import re

import pytest

import bench
from synth import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cache_compression_06_b300", "csrc")


def _const(name):
    for f in ("tri.cu", "tri_device.cuh", "tri_path.cuh"):
        with open(os.path.join(CSRC, f)) as fh:
            m = re.search(r"constexpr int %s = (\d+);" % name, fh.read())
        if m:
            return int(m.group(1))
    raise KeyError(name)


def _rule(B, cap, compact):
    stages, stage, sel_ints, max_smem = (_const("kCoStages"), _const("kStageBytes"), _const("kSelInts"),
                                         _const("kMaxSmem"))
    up = lambda x, a: -(-x // a) * a
    bcap = up(min(B, cap), 32)
    total = stages * stage + 2 * stages * 8 + sel_ints * 4 + up(bcap * 4, 128)
    if total <= max_smem and compact == "holefill" and 8 * B <= _const("kHfMaxSmem"):
        return "select_only_kernel+holefill_apply_kernel"
    hf_ok = compact != "holefill" or up(B + 16 + 4 * max(min(B, cap - B), 0), 128) + 16384 <= stages * stage
    return "select_only_kernel+compact_only_kernel" if total <= max_smem and hf_ok else "select_compact_kernel"


@pytest.mark.parametrize("B", [256, 1024, 2048, 8192, 16000, 40000])
@pytest.mark.parametrize("cap", [2176, 32768, 65536])
@pytest.mark.parametrize("compact", ["ordered", "holefill"])
def test_select_kernel_name_follows_library_rule(B, cap, compact):
    w = WORKLOADS["qwen3_8b_36l_b4_n32768"].with_(budget=B)
    assert bench._select_kernel_name(w, cap, compact) == _rule(B, cap, compact)


def test_moved_rows_counts_only_compressed_units():
    import torch
    B = 4
    idx = torch.tensor([[[[0, 1, 2, 3]], [[0, 2, 5, 7]]]], dtype=torch.int32)   # [L=1][S=2][Hkv=1][B]
    seq_len = torch.tensor([4, 9], dtype=torch.int32)
    # sequence 0 has N <= B (untouched); sequence 1 keeps slot 0 in place and moves 3 rows
    assert bench._moved_rows(idx, seq_len, B) == 3


@pytest.mark.parametrize("compact", ["ordered", "holefill"])
def test_fused_step_kernels(compact):
    w = WORKLOADS["qwen3_8b_36l_b16_n2176"]
    k = bench._step_kernels(w, 2176, compact, fused=True)
    assert k == ["fused_mma_kernel<128,4>"] + (["holefill_apply_kernel"] if compact == "holefill" else [])


def test_paged_step_kernels_name_the_head_grouped_score_kernel():
    w = WORKLOADS["qwen3_32b_64l_b64_paged"]
    assert bench._step_kernels(w, 32768, "ordered", fused=False)[1] == "score_heads_mma_kernel"
    assert bench._step_kernels(w.with_(block=32), 32768, "ordered", fused=False)[1] == "score_keys_mma_kernel"
    assert bench._step_kernels(WORKLOADS["qwen3_8b_36l_b4_n32768"], 32768, "ordered", fused=False)[1] == \
        "score_keys_mma_kernel"
