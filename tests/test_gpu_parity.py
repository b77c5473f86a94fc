"""Attention output of the CUDA path against the CPU oracle (bf16 out, atol = rtol = 2e-2),
on seeded inputs small enough for the oracle, spanning several tiles and ragged tails, plus
the invariances the method guarantees."""
import numpy as np
import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import assert_close, parity, run_gpu

pytestmark = pytest.mark.gpu


def test_tiny_config():
    err, _ = parity(wl.tiny(seed=0))
    assert err < 2e-2


@pytest.mark.parametrize("shape", [0, 1, 2])
def test_nonpow2_pages_scaled(shape):
    parity(wl.nonpow2(shape, seed=1, scale=1 / 8))


def test_swa_noncausal_scaled():
    parity(wl.swa_noncausal(seed=2, scale=1 / 16))


def test_swa_causal_scaled():
    parity(wl.swa_causal(seed=3, seq_len=2048, window=256))


def test_clamped_mm_scaled():
    parity(wl.clamped_mm(seed=4, scale=1 / 16, num_ranges=3))


@pytest.mark.parametrize("page", [128, 544, 1056])
@pytest.mark.parametrize("windowed", [False, True])
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_mixed_scaled(page, windowed, kv):
    parity(wl.mixed(page, windowed, kv_dtype=kv, seed=5, scale=1 / 16, num_seqs=6))


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("group", [1, 3, 8])
@pytest.mark.parametrize("page", [1, 5, 16, 37])
def test_ragged_geometry(head_dim, group, page):
    """Odd page sizes (tiles straddle many pages), empty and one-token sequences, contexts
    that end mid-page, GQA groups that do not divide 128."""
    rng = np.random.default_rng(head_dim * 100 + group * 10 + page)
    ctx = [0, 1, 37, int(rng.integers(100, 400)), 0, 130]
    qlen = [1, 0, 19, int(rng.integers(130, 300)), 200, 3]
    parity(wl.build_case("ragged", ctx, qlen, 2 * group, 2, head_dim, page, causal=True,
                         window_left=int(rng.choice([0, 50])), seed=page))


@pytest.mark.parametrize("causal", [False, True])
def test_windows_and_ranges_combined(causal):
    rng = np.random.default_rng(7)
    mm = np.array([[[10, 90], [150, 400], [0, 0]], [[0, 500], [3, 2], [600, 700]]])
    parity(wl.build_case("combo", [60, 300], [400, 420], 8, 2, 128, 16, causal=causal,
                         window_left=70, window_right=33, mm_ranges=mm, clamp_mm=True,
                         seed=int(rng.integers(1 << 30))))
    parity(wl.build_case("combo_unclamped", [60, 300], [400, 420], 8, 2, 128, 16, causal=causal,
                         window_left=70, window_right=33, mm_ranges=mm, clamp_mm=False, seed=8))


# The two fp8 paths: live cache tiles dequantised into workspace before the attention kernel
# (the default), or widened by the kernel's producers (PPA_FLAG_FP8_INKERNEL).
FP8_PATHS = pytest.mark.parametrize("fp8_path", [0, binding.PPA_FLAG_FP8_INKERNEL],
                                    ids=["prepass", "inkernel"])


@FP8_PATHS
def test_fp8_kv_scaled(fp8_path):
    parity(wl.mixed(544, False, kv_dtype="fp8_e4m3", seed=9, scale=1 / 16, num_seqs=4),
           flags_extra=fp8_path)


@FP8_PATHS
@pytest.mark.parametrize("page", [16, 37])
@pytest.mark.parametrize("windowed", [False, True])
def test_fp8_kv_head_dim_256(page, windowed, fp8_path):
    """fp8 cache at head_dim 256 (in the kernel: each CTA of the pair widens its half of every
    K and V row)."""
    rng = np.random.default_rng(page + 2 * windowed)
    ctx = [0, 45, int(rng.integers(200, 400)), 130]
    qlen = [17, 1, int(rng.integers(150, 300)), 64]
    parity(wl.build_case("fp8_d256", ctx, qlen, 8, 4, 256, page, causal=True,
                         window_left=100 if windowed else 0, kv_dtype="fp8_e4m3", seed=page),
           flags_extra=fp8_path)


@FP8_PATHS
@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("page", [1, 5, 37, 128, 300])
def test_fp8_ragged_geometry(head_dim, page, fp8_path):
    """Contexts that end mid-tile, on a tile boundary or are empty; a window that leaves the
    first cache tiles dead; pages smaller and larger than a key tile."""
    rng = np.random.default_rng(head_dim + page)
    ctx = [0, 1, 127, 128, 129, int(rng.integers(300, 700)), 256]
    qlen = [5, 0, 3, 40, 1, int(rng.integers(100, 260)), 130]
    parity(wl.build_case("fp8_ragged", ctx, qlen, 6, 2, head_dim, page, causal=True,
                         window_left=int(rng.choice([0, 150])), kv_dtype="fp8_e4m3", seed=page),
           flags_extra=fp8_path)


@FP8_PATHS
@pytest.mark.parametrize("head_dim", [128, 256])
def test_fp8_kv_scales_of_2_8_and_above(head_dim, fp8_path):
    """Dequantisation scales >= 2^8 take the widening's two-multiply branch (scale * 2^120
    would overflow fp32). K's scale grows by 2^16 and the softmax scale shrinks by the same
    power of two, so the logits keep their size; V's outputs grow by 2^16."""
    import dataclasses
    base = wl.build_case("fp8_big", [0, 200, 37], [50, 180, 9], 8, 2, head_dim, 37, causal=True,
                         window_left=60, kv_dtype="fp8_e4m3", seed=31 + head_dim)
    big = 2.0 ** 16
    case = dataclasses.replace(base, k_scale=base.k_scale * big, v_scale=base.v_scale * big,
                               sm_scale=head_dim ** -0.5 / big)
    assert case.k_scale >= 256 and case.v_scale >= 256
    got = run_gpu(case, flags_extra=fp8_path).out.float().cpu().numpy()
    want = ref.attention(case.numpy_inputs())
    # the tolerance applies at the outputs' own magnitude: compare both divided by 2^16
    assert_close(got / big, want / big, case.name)


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("chunk,lookback", [(16, 0), (100, 1), (300, 2)])
def test_chunked_local_parity(head_dim, causal, chunk, lookback):
    """Chunked-local attention: the base left edge at a chunk start; key tiles before it are
    skipped (a chunk boundary inside a query tile keeps the earlier chunk's keys live)."""
    rng = np.random.default_rng(head_dim + chunk)
    ctx = [0, int(rng.integers(100, 500)), 37, 300]
    qlen = [int(rng.integers(200, 420)), int(rng.integers(60, 200)), 1, 129]
    parity(wl.build_case("chunked", ctx, qlen, 8, 2, head_dim, 37, causal=causal,
                         window_right=0 if causal else 70, chunk_size=chunk,
                         chunk_lookback=lookback, seed=chunk))


@pytest.mark.parametrize("head_dim", [128, 256])
def test_chunked_local_with_clamped_mm_ranges(head_dim):
    """The review case on the multimodal-pruning page: clamped ranges, OR-ed on with the left
    window as their clamp, re-enable keys before the chunk start."""
    mm = np.array([[[120, 380], [500, 520]], [[0, 0], [40, 90]]])
    parity(wl.build_case("chunked_mm", [0, 200], [600, 300], 8, 4, head_dim, 16, causal=True,
                         window_left=150, mm_ranges=mm, clamp_mm=True, chunk_size=128,
                         chunk_lookback=0, seed=head_dim))


def test_page_permutation_is_bitwise_invariant():
    a = wl.build_case("perm", [300, 1000], [200, 333], 8, 2, 128, 544, causal=True, seed=10,
                      value_rng_seed=77)
    b = wl.build_case("perm", [300, 1000], [200, 333], 8, 2, 128, 544, causal=True, seed=11,
                      value_rng_seed=77)
    assert not torch.equal(a.block_table, b.block_table)
    oa = run_gpu(a).out.cpu()
    ob = run_gpu(b).out.cpu()
    assert torch.equal(oa, ob)


@pytest.mark.parametrize("factory", [
    lambda: wl.swa_noncausal(seed=12, scale=1 / 32),
    lambda: wl.clamped_mm(seed=13, scale=1 / 32, num_ranges=2),
    lambda: wl.mixed(1040, True, seed=14, scale=1 / 16, num_seqs=3),
])
def test_pruned_equals_unpruned_bitwise(factory):
    case = factory()
    pruned = run_gpu(case).out.cpu()
    full = run_gpu(case, flags_extra=binding.PPA_FLAG_NO_PRUNE).out.cpu()
    assert torch.equal(pruned.float(), full.float())


def test_removing_a_range_changes_gpu_output():
    case = wl.clamped_mm(seed=15, scale=1 / 16, num_seqs=1, num_ranges=2, range_width=100)
    with_mm = run_gpu(case).out.float().cpu().numpy()
    a, e = case.mm_ranges[0, 0].tolist()
    case.mm_ranges[0, 0] = torch.tensor([0, 0], dtype=torch.int32)
    without = run_gpu(case).out.float().cpu().numpy()
    assert np.abs(with_mm[a:e - 1] - without[a:e - 1]).max() > 2e-2
    assert_close(without, ref.attention(case.numpy_inputs()), "without range")


def test_single_allowed_key_returns_value_row():
    case = wl.build_case("one", [0, 40], [150, 70], 4, 2, 64, 16, causal=True, window_left=1,
                         seed=16)
    got = run_gpu(case).out.float().cpu()
    want = case.v_new.float().repeat_interleave(2, dim=1)
    assert torch.equal(got, want)


def test_status_reports_bad_page_without_faulting():
    case = wl.build_case("badpage", [40], [10], 2, 1, 64, 16, causal=True, seed=17)
    case.block_table[0, 1] = case.num_pages + 5
    dc = binding.DeviceCase(case)
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_ERR_BAD_PAGE


def test_status_reports_bad_lengths():
    case = wl.tiny(seed=0)
    dc = binding.DeviceCase(case)
    dc.cu_query_lens[1] = -5
    dc.run()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_ERR_INVALID


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("windowed", [False, True])
def test_per_sequence_causal_parity(head_dim, windowed):
    """Per-sequence causal flags: each sequence's key tiles and mask follow its own flag."""
    rng = np.random.default_rng(head_dim + windowed)
    ctx = [0, int(rng.integers(50, 300)), 130, 0]
    qlen = [int(rng.integers(150, 300)), int(rng.integers(40, 150)), 77, 129]
    parity(wl.build_case("seq_causal", ctx, qlen, 8, 4, head_dim, 16, causal=True,
                         window_left=120 if windowed else 0, window_right=60 if windowed else 0,
                         seq_causal=[True, False, False, True], seed=head_dim))


def test_per_sequence_causal_with_ranges_and_tile_bounds():
    mm = np.array([[[30, 90]], [[10, 200]], [[0, 0]]])
    case = wl.build_case("seq_causal_mm", [0, 40, 10], [300, 250, 90], 8, 2, 128, 37, causal=False,
                         window_left=64, window_right=32, mm_ranges=mm, clamp_mm=True,
                         seq_causal=[False, True, True], seed=7)
    parity(case)
    # the plan's per-tile bounds follow each sequence's flag, bit-exact
    dims = binding.dims_for(case)
    sc = case.seq_causal.cuda()
    dims.seq_causal = sc.data_ptr()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cap = -(-case.total_q // 16) + case.num_seqs
    out = torch.full((cap, 2), -7, dtype=torch.int32, device="cuda")
    binding.ppa_tile_bounds(dims, 16, 128, case.cu_query_lens.cuda(), case.context_lens.cuda(),
                            case.mm_ranges.cuda(), out, status)
    assert binding.ppa_read_status(status) == 0
    want = ref.tile_bounds(case.numpy_inputs(), 16, 128)
    assert np.array_equal(out[: len(want)].cpu().numpy(), want)
