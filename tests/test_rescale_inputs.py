"""The rescale cases really exercise the online-softmax rescale with mass already in O.

On the oracle's own scores for the inputs the GPU rescale tests use, a large share of rows
have a key, after the row's first live key tile, whose score exceeds that tile's maximum by
more than 8 log2 units (the kernels' rescale threshold), while the keys before it keep a
share of the row's softmax mass that a wrong rescale factor would visibly move. The key tile
width is the library's own (``ppa_query_tiles``)."""
import math

import numpy as np
import pytest

from oracle import ref
from paged_kv_prefix_gb300 import binding
from tests import rescale_cases as rc


def _row_jumps(case, split_tiles=0):
    """Per (row, head): the largest rise, in log2 units, of a later key tile's maximum over
    the running maximum of the row's first live tile (of its segment, with split-KV), and
    the softmax mass of the keys up to the first such tile."""
    inp = case.numpy_inputs()
    _, tn = binding.ppa_query_tiles(binding.dims_for(case))
    Hq, Hkv, D = case.num_q_heads, case.num_kv_heads, case.head_dim
    G = Hq // Hkv
    scale = case.sm_scale if case.sm_scale > 0 else 1.0 / math.sqrt(D)
    cu = inp["cu_query_lens"]
    jumps, masses = [], []
    for b in range(case.num_seqs):
        c, n = int(inp["context_lens"][b]), int(cu[b + 1] - cu[b])
        if n == 0:
            continue
        s = c + n
        K = ref.gather_kv(inp, b, "k").astype(np.float64)
        toks = np.arange(n)
        mask = ref.allowed_mask(c + toks, s, case.causal, case.window_left, case.window_right,
                                None, case.clamp_mm)
        Q = inp["q"][int(cu[b]):int(cu[b]) + n].astype(np.float64)
        for h in range(Hq):
            sc = np.where(mask, (Q[:, h] @ K[:, h // G].T) * scale * math.log2(math.e), -np.inf)
            for j in range(n):
                allowed = np.nonzero(mask[j])[0]
                t_first, t_last = allowed[0] // tn, allowed[-1] // tn
                segs = [(t_first, t_last + 1)]
                if split_tiles > 0:
                    segs = [(t, min(t + split_tiles, t_last + 1))
                            for t in range(t_first, t_last + 1, split_tiles)]
                for lo, hi in segs:
                    tiles = [sc[j, t * tn:(t + 1) * tn].max() for t in range(lo, hi)]
                    run = tiles[0]
                    best, cut = 0.0, None
                    for t in range(1, len(tiles)):
                        if tiles[t] - run > best:
                            best, cut = tiles[t] - run, lo + t
                        run = max(run, tiles[t])
                    jumps.append(best)
                    if cut is not None and best > 8.0:
                        seg = sc[j, lo * tn:hi * tn]
                        w = np.exp2(seg - seg.max())
                        masses.append(w[:(cut - lo) * tn].sum() / w.sum())
    return np.array(jumps), np.array(masses)


@pytest.mark.parametrize("spec", rc.PREFILL + [rc.LARGE_SCALE], ids=lambda s: s[0])
def test_rows_jump_past_the_rescale_threshold_with_mass_in_o(spec):
    jumps, masses = _row_jumps(rc.build(spec))
    assert (jumps > 8.0).mean() > 0.5, f"only {(jumps > 8.0).mean():.2f} of rows jump past 8"
    # the keys before the jump keep a share of the mass that a wrong alpha would change
    assert np.median(masses) > 0.05 and masses.max() > 0.2, (np.median(masses), masses.max())


def test_split_segments_rescale_with_mass_in_o():
    jumps, masses = _row_jumps(rc.build(rc.DECODE), split_tiles=3)
    assert (jumps > 8.0).sum() >= 20
    assert np.median(masses) > 0.05
