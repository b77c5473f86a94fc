"""The parity checks can fail: at the sizes the GPU parity tests use, including the full-size
workloads, removing one live key tile (128 keys, the kernels' tile) from the oracle's mask
moves some checked output by more than the rounding-derived bound those tests apply
(``tests/tolerance.py``). The mistake is planted in the oracle, on the CPU: its mask
predicate is wrapped so that one tile's columns read as masked (rows left with no key keep
their mask, as a row is never empty)."""
import numpy as np
import pytest

from oracle import ref
from paged_kv_prefix_gb300 import workloads as wl
from tests import rescale_cases as rc
from tests import tolerance

TN = 128


def _check(case, monkeypatch, rows=8, seed=0):
    inp = case.numpy_inputs()
    cu = inp["cu_query_lens"]
    lens = [(int(inp["context_lens"][b]) + int(cu[b + 1] - cu[b])) if cu[b + 1] > cu[b] else -1
            for b in range(case.num_seqs)]
    b = int(np.argmax(lens))
    c, n = int(inp["context_lens"][b]), int(cu[b + 1] - cu[b])
    rng = np.random.default_rng(seed)
    toks = np.unique(np.concatenate([[n - 1], rng.choice(n, size=min(n, rows), replace=False)]))
    kv = (ref.gather_kv(inp, b, "k"), ref.gather_kv(inp, b, "v"))
    want = ref.attention_rows(inp, b, toks, kv=kv)
    tol = tolerance.tight_tolerance(inp, b, toks, want, kv)
    # a tile live for the last row other than the row's own tile, else the row's own tile
    q_last = c + int(toks.max())
    kt = q_last // TN - 1 if q_last >= TN else 0
    orig = ref.allowed_mask

    def without_tile(*a, **k):
        m = orig(*a, **k)
        m2 = m.copy()
        m2[:, kt * TN:(kt + 1) * TN] = False
        empty = ~m2.any(axis=1)
        m2[empty] = m[empty]
        return m2

    monkeypatch.setattr(ref, "allowed_mask", without_tile)
    dropped = ref.attention_rows(inp, b, toks, kv=kv)
    monkeypatch.setattr(ref, "allowed_mask", orig)
    moved = np.abs(dropped - want)
    assert (moved > tol).any(), (f"{case.name}: dropping key tile {kt} moves the checked rows "
                                 f"by at most {moved.max():.3g}, within the bound")
    return float((moved / tol).max()), bool((~tolerance.within_bar(dropped, want)).any())


SCALED = [
    lambda: wl.nonpow2(0, seed=1, scale=1 / 8),
    lambda: wl.nonpow2(1, seed=1, scale=1 / 8),
    lambda: wl.nonpow2(2, seed=1, scale=1 / 8),
    lambda: wl.swa_noncausal(seed=2, scale=1 / 16),
    lambda: wl.swa_causal(seed=3, seq_len=2048, window=256),
    lambda: wl.clamped_mm(seed=4, scale=1 / 16, num_ranges=3),
    lambda: wl.mixed(544, False, seed=5, scale=1 / 16, num_seqs=6),
    lambda: wl.mixed(1056, True, kv_dtype="fp8_e4m3", seed=5, scale=1 / 16, num_seqs=6),
    lambda: rc.build(rc.PREFILL[3]),
]


@pytest.mark.parametrize("factory", SCALED, ids=range(len(SCALED)))
def test_dropped_tile_is_caught_at_test_sizes(factory, monkeypatch):
    _check(factory(), monkeypatch)


FULL = [
    lambda: wl.nonpow2(0, seed=0),
    lambda: wl.swa_causal(seed=0),
    lambda: wl.clamped_mm(seed=0),
    lambda: wl.mixed(544, False, seed=0),
    lambda: wl.mixed(2048, True, kv_dtype="fp8_e4m3", seed=0),
]


@pytest.mark.parametrize("factory", FULL, ids=range(len(FULL)))
def test_dropped_tile_is_caught_at_full_size(factory, monkeypatch):
    _check(factory(), monkeypatch)
