"""Parity on the full-size workloads, in the launch configuration the benchmark times.

The oracle cannot attend every row of these batches in reasonable time, so each sequence is
checked on its first and last query token and six other distinct rows, computed one by one,
against the 2e-2 bar and the rounding-derived bound of ``tests/tolerance.py`` (tight enough
that one missing live key tile shows: ``tests/test_parity_sensitivity.py``). The workloads
are the seeded stand-ins of the pages' experiments (``paged_kv_prefix_gb300/workloads.py``):
the non-power-of-2 page sizes of the PR #54194 report, the windowed prefill of PR #50776, the
clamped multimodal prefix of PR #53147 and the mixed-serving sweep over six page sizes, two
windows and two cache dtypes."""
import pytest
import torch

from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl
from tests.gpu_util import parity, sampled_parity

pytestmark = pytest.mark.gpu


def _run_sampled(case, flags=0):
    dc = binding.DeviceCase(case, flags_extra=flags)
    dc.plan()
    dc.attend()
    torch.cuda.synchronize()
    assert dc.read_status() == binding.PPA_OK
    err, ratio = sampled_parity(case, dc, rows_per_seq=6)
    del dc
    torch.cuda.empty_cache()
    return err, ratio


def test_full_tiny():
    parity(wl.tiny(seed=0))


@pytest.mark.parametrize("shape", [0, 1, 2])
def test_full_nonpow2(shape):
    _run_sampled(wl.nonpow2(shape, seed=0))


def test_full_swa64_noncausal():
    _run_sampled(wl.swa_noncausal(seed=0))


def test_full_swa1024_causal():
    _run_sampled(wl.swa_causal(seed=0))


def test_full_clamped_mm():
    case = wl.clamped_mm(seed=0)
    assert case.max_mm_ranges == 60
    _run_sampled(case)


# every run of the mixed-serving sweep; the page size varies fastest, so consecutive runs
# share one value draw
MIXED = [(kv, windowed, page) for kv in ("bf16", "fp8_e4m3") for windowed in (False, True)
         for page in wl.MIXED_PAGE_SIZES]


@pytest.mark.parametrize("kv,windowed,page", MIXED,
                         ids=[f"{kv}-w{int(w)}-p{p}" for kv, w, p in MIXED])
def test_full_mixed_serving(kv, windowed, page):
    _run_sampled(wl.mixed(page, windowed, kv_dtype=kv, seed=0))


def test_full_mixed_fp8_in_kernel():
    _run_sampled(wl.mixed(544, False, kv_dtype="fp8_e4m3", seed=0),
                 flags=binding.PPA_FLAG_FP8_INKERNEL)
