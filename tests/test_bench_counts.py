"""The bench line's kernel-launch count per step (``gpu_launches``) for each path: the plan and
the attention kernel; three more for the fp8 dequantisation pass (live-tile marking, staging
slots, dequantisation); one for the KV append of the cache-sourced path; one for the split-KV
merge, which runs whenever ``kv_split_tiles`` is non-zero, including -1 (the tuned length)."""
import types

import pytest

import bench
from paged_kv_prefix_gb300 import binding


def _dc(kv_dtype=binding.PPA_KV_BF16, flags=0, split=0):
    dims = binding.PpaDims()
    dims.kv_dtype = kv_dtype
    dims.flags = flags
    dims.kv_split_tiles = split
    return types.SimpleNamespace(dims=dims)


FP8 = binding.PPA_KV_FP8_E4M3
IK = binding.PPA_FLAG_FP8_INKERNEL
CACHED = binding.PPA_FLAG_KV_IN_CACHE


@pytest.mark.parametrize("kv_dtype,flags,split,want", [
    (binding.PPA_KV_BF16, 0, 0, 2),
    (binding.PPA_KV_BF16, 0, 32, 3),
    (binding.PPA_KV_BF16, 0, -1, 3),
    (FP8, 0, 0, 5),
    (FP8, 0, -1, 6),
    (FP8, IK, 0, 2),
    (FP8, IK, -1, 3),
    (binding.PPA_KV_BF16, CACHED, 0, 3),
    (FP8, CACHED, 0, 6),
])
def test_launches_per_step(kv_dtype, flags, split, want):
    assert bench._launches_per_step(_dc(kv_dtype, flags, split)) == want
