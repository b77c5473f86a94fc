"""Helpers shared by the GPU tests: run a case through the C ABI and compare with the oracle."""
import numpy as np
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from tests import tolerance

ATOL = tolerance.ATOL  # bf16 output vs fp32 oracle: max-abs 2e-2 and rtol 2e-2
RTOL = tolerance.RTOL


def run_gpu(case, flags_extra=0, stream=None):
    dc = binding.DeviceCase(case, flags_extra=flags_extra)
    dc.run(stream=stream)
    torch.cuda.synchronize()
    status = dc.read_status()
    assert status == binding.PPA_OK, binding.status_string(status)
    return dc


def assert_close(got, want, what=""):
    assert got.shape == want.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    bad = err > ATOL + RTOL * np.abs(want)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; max abs error "
                             f"{err.max():.4g}; first bad indices {idx.tolist()}")
    return float(err.max())


def assert_tight(inp, got, want, what="", row_chunk=512):
    """Every row of every sequence within the rounding-derived bound (``tests/tolerance.py``);
    returns the largest ratio of error to bound."""
    cu = inp["cu_query_lens"]
    worst = 0.0
    for b in range(len(inp["context_lens"])):
        n = int(cu[b + 1] - cu[b])
        if n == 0:
            continue
        kv = (ref.gather_kv(inp, b, "k"), ref.gather_kv(inp, b, "v"))
        for j0 in range(0, n, row_chunk):
            toks = np.arange(j0, min(n, j0 + row_chunk))
            rows = int(cu[b]) + toks
            ratio = (np.abs(got[rows] - want[rows])
                     / tolerance.tight_tolerance(inp, b, toks, want[rows], kv))
            if (ratio > 1.0).any():
                idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
                raise AssertionError(
                    f"{what} seq {b}: error above the rounding-derived bound by {ratio.max():.3g}x "
                    f"at (token {int(toks[idx[0]])}, head {idx[1]}, col {idx[2]}): "
                    f"got {got[rows][idx]:.6g}, want {want[rows][idx]:.6g}")
            worst = max(worst, float(ratio.max()))
    return worst


def parity(case, flags_extra=0, tight=True, **dc_kw):
    """Whole output against the oracle: the 2e-2 bar, and (``tight``) the rounding-derived
    bound."""
    dc = binding.DeviceCase(case, flags_extra=flags_extra, **dc_kw)
    dc.run()
    torch.cuda.synchronize()
    status = dc.read_status()
    assert status == binding.PPA_OK, binding.status_string(status)
    got = dc.out.float().cpu().numpy()
    inp = case.numpy_inputs()
    if flags_extra & binding.PPA_FLAG_KV_IN_CACHE:
        inp["kv_in_cache"] = True
    want = ref.attention(inp)
    err = assert_close(got, want, case.name)
    if tight:
        assert_tight(inp, got, want, case.name)
    return err, dc


def sampled_parity(case, dc, rows_per_seq=6, seed=0):
    """Compare sampled output rows of a full-size run with the oracle computed one by one:
    each sequence's first and last query token plus ``rows_per_seq`` distinct others, against
    the 2e-2 bar and against the rounding-derived bound of ``tests/tolerance.py``. Returns
    (max abs error, max ratio of error to the rounding-derived bound)."""
    inp = case.numpy_inputs()
    got = dc.out.float().cpu().numpy()
    rng = np.random.default_rng(seed)
    cu = inp["cu_query_lens"]
    worst, worst_ratio = 0.0, 0.0
    for b in range(case.num_seqs):
        n = int(cu[b + 1] - cu[b])
        if n == 0:
            continue
        inner = rng.choice(n, size=min(n, rows_per_seq), replace=False)
        toks = np.unique(np.concatenate([[0, n - 1], inner]))
        kv = (ref.gather_kv(inp, b, "k"), ref.gather_kv(inp, b, "v"))
        want = ref.attention_rows(inp, b, toks, kv=kv)
        g = got[int(cu[b]) + toks]
        worst = max(worst, assert_close(g, want, f"{case.name} seq {b}"))
        ratio = np.abs(g - want) / tolerance.tight_tolerance(inp, b, toks, want, kv)
        if (ratio > 1.0).any():
            idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
            raise AssertionError(
                f"{case.name} seq {b}: error above the rounding-derived bound by "
                f"{ratio.max():.3g}x at (token {int(toks[idx[0]])}, head {idx[1]}, col {idx[2]}): "
                f"got {g[idx]:.6g}, want {want[idx]:.6g}")
        worst_ratio = max(worst_ratio, float(ratio.max()))
    return worst, worst_ratio
