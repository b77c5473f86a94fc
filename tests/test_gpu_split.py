"""Split-KV (ppa_dims.kv_split_tiles): sequences whose new tokens fit one query tile are cut
into key-tile segments, attended in parallel and merged by their log-sum-exps. The output
must match the oracle (the same attention, unsplit) and the unsplit kernel run."""
import numpy as np
import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


def _run(case, split, flags=0, append=False):
    dc = binding.DeviceCase(case, flags_extra=flags, kv_split_tiles=split)
    if append:
        dc.append()
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    return dc.out.float().cpu().numpy()


def _decode_batch(D, G, page, kv="bf16", seed=0, **kw):
    """Decode and verify rows (1-8 new tokens) over long contexts, next to a prefill sequence
    (several query tiles: not split) and an empty one."""
    rng = np.random.default_rng(seed)
    tq = 128 // G
    ctx = [int(rng.integers(1500, 3000)), int(rng.integers(300, 900)), 2000, 40, 0, 700]
    qlen = [1, int(rng.integers(2, 9)), tq, 1, 3, 2 * tq + 5]
    return wl.build_case("split", ctx, qlen, 2 * G, 2, D, page, kv_dtype=kv, seed=seed, **kw)


@pytest.mark.parametrize("D,G", [(64, 1), (128, 4), (128, 8), (256, 4)])
@pytest.mark.parametrize("split", [1, 3, 8])
def test_split_kv_matches_oracle_and_unsplit(D, G, split):
    case = _decode_batch(D, G, 37, seed=D + G + split, causal=True)
    got = _run(case, split)
    assert_close(got, ref.attention(case.numpy_inputs()), f"split {split}")
    assert_close(got, _run(case, 0), "split vs unsplit")


@pytest.mark.parametrize("D", [128, 256])
def test_split_kv_with_windows_and_ranges(D):
    mm = np.array([[[100, 900]], [[0, 0]], [[1000, 1990]], [[0, 0]], [[0, 0]], [[0, 300]]])
    case = _decode_batch(D, 4, 16, seed=3, causal=True, window_left=700, mm_ranges=mm,
                         clamp_mm=True)
    assert_close(_run(case, 2), ref.attention(case.numpy_inputs()), "split mm")


@pytest.mark.parametrize("fp8_path", [0, binding.PPA_FLAG_FP8_INKERNEL], ids=["prepass", "inkernel"])
def test_split_kv_fp8(fp8_path):
    case = _decode_batch(128, 4, 544, kv="fp8_e4m3", seed=4, causal=True)
    assert_close(_run(case, 4, fp8_path), ref.attention(case.numpy_inputs()), "split fp8")


def test_split_kv_cache_sourced():
    case = _decode_batch(128, 8, 37, seed=5, causal=True)
    inp = case.numpy_inputs()
    inp["k_cache"], inp["v_cache"] = ref.append_kv(inp)
    inp["kv_in_cache"] = True
    got = _run(case, 2, binding.PPA_FLAG_KV_IN_CACHE, append=True)
    assert_close(got, ref.attention(inp), "split cache-sourced")


def test_split_kv_noncausal_verify_rows():
    """Non-causal rows see keys on both sides: every segment holds some of each row's keys."""
    case = _decode_batch(64, 2, 5, seed=6, causal=False, window_right=40)
    assert_close(_run(case, 3), ref.attention(case.numpy_inputs()), "split non-causal")


def test_rejected_split_batch_writes_nothing_past_the_output():
    """Lengths the plan rejects (a middle sequence runs past total_q) with split-KV on: the
    device reports PPA_ERR_INVALID and neither the attention nor the merge writes a row, in
    particular none past total_q (the output view is the head of a larger, sentinel-filled
    buffer)."""
    case = wl.build_case("bad_split", [300, 40, 20], [1, 1, 1], 2, 1, 128, 16, causal=True,
                         seed=8)
    dc = binding.DeviceCase(case, kv_split_tiles=2)
    big = torch.full((case.total_q + 200, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[: case.total_q]
    dc.cu_query_lens.copy_(torch.tensor([0, 1, 100, 3], dtype=torch.int32))  # sequence 1: n = 99
    dc.run(out=out)
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_ERR_INVALID
    assert bool((big.float() == 7.0).all())
