"""Host-side checks of the C ABI that need no GPU: the library loads, exports every entry
point include/ppa.h declares, sizes its workspace and rejects invalid arguments before
launching anything."""
import ctypes
import os
import re

import pytest

from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ppa.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ppa_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = binding.lib()
    names = _declared_functions()
    assert "ppa_prefill" in names and len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(binding._SIGNATURES)


def test_status_strings_and_version():
    assert binding.ppa_status_string(0) == "ok"
    assert "timed out" in binding.ppa_status_string(binding.PPA_ERR_TIMEOUT)
    assert binding.ppa_status_string(99) == "unknown status"
    assert binding.ppa_version() == 300  # the ppa_dims layout the binding mirrors


def _dims(**kw):
    d = binding.dims_for(wl.tiny())
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_tiles_and_workspace():
    d = _dims()
    assert binding.ppa_query_tiles(d) == (64, 128)  # G = 2 -> 64 tokens x 2 heads
    assert binding.ppa_workspace_bytes(d) > 0
    assert binding.ppa_query_tiles(_dims(num_q_heads=32, num_kv_heads=4, head_dim=256)) == (16, 128)
    assert binding.ppa_query_tiles(_dims(num_q_heads=6, num_kv_heads=2)) == (42, 128)
    assert binding.ppa_workspace_bytes(_dims(head_dim=96)) == 0
    assert binding.ppa_query_tiles(_dims(head_dim=96)) == (0, 0)


def test_fp8_workspace_holds_the_bf16_staging_unless_widened_in_kernel():
    base = binding.ppa_workspace_bytes(_dims())
    fp8 = _dims(kv_dtype=binding.PPA_KV_FP8_E4M3)
    inkernel = _dims(kv_dtype=binding.PPA_KV_FP8_E4M3, flags=fp8.flags | binding.PPA_FLAG_FP8_INKERNEL)
    assert binding.ppa_workspace_bytes(inkernel) == base
    # K and V tiles of 128 positions for every block-table slot of every sequence
    tiles = fp8.num_seqs * -(-(fp8.max_pages_per_seq * fp8.page_size) // 128)
    staging = 2 * tiles * 128 * fp8.num_kv_heads * fp8.head_dim * 2
    assert staging <= binding.ppa_workspace_bytes(fp8) - base <= staging + 4 * 256 + 8 * tiles


def test_auto_split_is_the_tuned_segment_length():
    d = _dims(num_seqs=4, total_q=4, max_pages_per_seq=200, num_pages=900)
    auto = binding.ppa_workspace_bytes(_dims(kv_split_tiles=-1, num_seqs=4, total_q=4,
                                             max_pages_per_seq=200, num_pages=900))
    tuned = binding.ppa_workspace_bytes(_dims(kv_split_tiles=32, num_seqs=4, total_q=4,
                                              max_pages_per_seq=200, num_pages=900))
    assert auto == tuned > binding.ppa_workspace_bytes(d)


def test_fp8_staging_is_sized_by_the_cache_token_bound():
    """max_cache_tokens > 0: floor(bound / 128) + 2 * num_seqs staging tiles, never more than
    the block-table capacity; the table still covers every block-table slot."""
    big = dict(kv_dtype=binding.PPA_KV_FP8_E4M3, num_seqs=32, total_q=70000, num_q_heads=32,
               num_kv_heads=4, head_dim=128, page_size=544, max_pages_per_seq=61,
               num_pages=2000)
    full = binding.ppa_workspace_bytes(_dims(**big))
    entries = 32 * -(-(61 * 544) // 128)
    tile_bytes = 2 * 128 * 4 * 128 * 2  # K and V
    for bound in (590_000, 131_072, 1):
        got = binding.ppa_workspace_bytes(_dims(max_cache_tokens=bound, **big))
        pages = min(entries, bound // 128 + 64)
        assert full - got == (entries - pages) * tile_bytes
    assert binding.ppa_workspace_bytes(_dims(max_cache_tokens=10**9, **big)) == full
    assert binding.ppa_workspace_bytes(_dims(max_cache_tokens=-1, **big)) == 0


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, binding.PPA_ERR_UNSUPPORTED),
    ("num_kv_heads", 3, binding.PPA_ERR_INVALID),
    ("num_q_heads", 0, binding.PPA_ERR_INVALID),
    ("page_size", 0, binding.PPA_ERR_INVALID),
    ("num_pages", 0, binding.PPA_ERR_INVALID),
    ("num_seqs", -1, binding.PPA_ERR_INVALID),
    ("kv_dtype", 7, binding.PPA_ERR_INVALID),
    ("flags", 64, binding.PPA_ERR_INVALID),
    ("sm_scale", float("nan"), binding.PPA_ERR_INVALID),
    ("max_mm_ranges", -2, binding.PPA_ERR_INVALID),
    ("chunk_size", -1, binding.PPA_ERR_INVALID),
    ("kv_split_tiles", -3, binding.PPA_ERR_INVALID),
    ("kv_split_tiles", -2, binding.PPA_ERR_INVALID),
    ("max_cache_tokens", -1, binding.PPA_ERR_INVALID),
])
def test_invalid_dims_rejected(field, value, code):
    d = _dims(**{field: value})
    fake = 1 << 20  # never dereferenced: validation fails first
    got = binding.ppa_prefill(d, fake, fake, fake, fake, fake, fake, fake, fake, None, None, None,
                              fake, fake, fake, stream=0, check=False)
    assert got == code


def test_chunk_lookback_must_be_non_negative_with_chunks():
    f = 1 << 20
    args = [f] * 8 + [None, None, None, f, f, f]
    d = _dims(chunk_size=16, chunk_lookback=-1)
    assert binding.ppa_prefill(d, *args, stream=0, check=False) == binding.PPA_ERR_INVALID
    assert binding.ppa_workspace_bytes(d) == 0
    assert binding.ppa_workspace_bytes(_dims(chunk_size=16, chunk_lookback=2)) > 0
    # without chunks the lookback is ignored
    assert binding.ppa_workspace_bytes(_dims(chunk_size=0, chunk_lookback=-1)) > 0


def test_split_kv_workspace_holds_the_partials():
    base = _dims()
    split = _dims(kv_split_tiles=4)
    extra = binding.ppa_workspace_bytes(split) - binding.ppa_workspace_bytes(base)
    tq = 128 // (base.num_q_heads // base.num_kv_heads)
    tiles = -(-(base.max_pages_per_seq * base.page_size + tq) // 128)
    nseg = -(-tiles // 4)
    slots = base.num_seqs * nseg * base.num_kv_heads
    partials = slots * 128 * (base.head_dim + 1) * 4  # O rows and log-sum-exps, fp32
    assert partials <= extra <= partials + 4 * 256 + base.num_seqs * (nseg - 1) * (
        36 + 4 * base.num_kv_heads) + 8 * (base.num_seqs + 1)


def test_append_kv_validates_on_the_host():
    d = _dims()
    f = 1 << 20
    # every call below is rejected (or has no work) before anything is launched
    ok = [f, f, f, f, f, f, f, None, None, f]  # k_new .. context_lens, scales, status
    for i, name in [(0, "k_new"), (2, "k_cache"), (4, "block_table"), (9, "status")]:
        a = list(ok)
        a[i] = None
        assert binding.ppa_append_kv(d, *a, stream=0, check=False) == binding.PPA_ERR_INVALID, name
    a = list(ok)
    a[1] = f + 8  # misaligned v_new
    assert binding.ppa_append_kv(d, *a, stream=0, check=False) == binding.PPA_ERR_INVALID
    d8 = _dims(kv_dtype=binding.PPA_KV_FP8_E4M3)  # fp8 without scales
    assert binding.ppa_append_kv(d8, *ok, stream=0, check=False) == binding.PPA_ERR_INVALID
    empty = _dims(num_seqs=0, total_q=0)
    assert binding.ppa_append_kv(empty, *ok, stream=0, check=False) == binding.PPA_OK


def test_null_and_misaligned_pointers_rejected():
    d = _dims()
    f = 1 << 20
    args = [f] * 8 + [None, None, None, f, f, f]  # never launched: each call below is rejected
    # k_new = NULL needs PPA_FLAG_KV_IN_CACHE
    a = list(args)
    a[1] = None
    assert binding.ppa_prefill(d, *a, stream=0, check=False) == binding.PPA_ERR_UNSUPPORTED
    # missing output
    a = list(args)
    a[11] = None
    assert binding.ppa_prefill(d, *a, stream=0, check=False) == binding.PPA_ERR_INVALID
    # misaligned q
    a = list(args)
    a[0] = f + 2
    assert binding.ppa_prefill(d, *a, stream=0, check=False) == binding.PPA_ERR_INVALID
    # multimodal ranges declared but not passed
    d2 = _dims(max_mm_ranges=3)
    assert binding.ppa_prefill(d2, *args, stream=0, check=False) == binding.PPA_ERR_INVALID
    # fp8 without scales
    d3 = _dims(kv_dtype=binding.PPA_KV_FP8_E4M3)
    assert binding.ppa_prefill(d3, *args, stream=0, check=False) == binding.PPA_ERR_INVALID


def test_empty_batch_launches_nothing():
    d = _dims(num_seqs=0, total_q=0)
    f = 1 << 20
    assert binding.ppa_prefill(d, *([f] * 8), None, None, None, f, f, f, stream=0,
                               check=False) == binding.PPA_OK


def test_test_entry_points_validate():
    d = _dims()
    f = 1 << 20
    assert binding.ppa_tile_bounds(d, 0, 32, f, f, None, f, f, stream=0, check=False) == 1
    assert binding.ppa_debug_mask(d, 5, f, f, None, f, 1, 1, stream=0, check=False) == 1
    assert binding.ppa_debug_e4m3_to_bf16(None, None, -1, stream=0, check=False) == 1
    assert binding.ppa_read_status(None, stream=0) == 1
    assert binding.ppa_live_pairs(d, None, f, None, f, stream=0, check=False) == 1
