"""Helpers shared by the GPU tests: run a case through the C ABI and compare with the oracle."""
import numpy as np
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding

ATOL = 2e-2  # bf16 output vs fp32 oracle: max-abs 2e-2 and rtol 2e-2
RTOL = 2e-2


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


def parity(case, flags_extra=0):
    dc = run_gpu(case, flags_extra)
    got = dc.out.float().cpu().numpy()
    want = ref.attention(case.numpy_inputs())
    return assert_close(got, want, case.name), dc


def sampled_parity(case, dc, rows_per_seq=6, seed=0):
    """Compare sampled output rows of a full-size run with the oracle computed one by one."""
    inp = case.numpy_inputs()
    got = dc.out.float().cpu().numpy()
    rng = np.random.default_rng(seed)
    cu = inp["cu_query_lens"]
    worst = 0.0
    for b in range(case.num_seqs):
        n = int(cu[b + 1] - cu[b])
        if n == 0:
            continue
        toks = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, size=rows_per_seq)]))
        want = ref.attention_rows(inp, b, toks)
        worst = max(worst, assert_close(got[int(cu[b]) + toks], want, f"{case.name} seq {b}"))
    return worst
