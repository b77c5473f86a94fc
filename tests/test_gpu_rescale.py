"""The online-softmax rescale of an output accumulator that already holds mass, on both
attention kernels, against the oracle.

The inputs (``tests/rescale_cases.py``) make row maxima jump by about 9.5 log2 units after a
row's first live key tiles; ``tests/test_rescale_inputs.py`` shows on the oracle's own scores
that the jump passes the kernels' rescale threshold (8) while the earlier keys keep a share of
the softmax mass. The rescale multiplies O (in TMEM) by alpha = 2^(m_old - m_new) and the row
sum by the same factor; a wrong, stale or missing alpha, or an O update racing the PV MMA,
moves these outputs far beyond the tolerance. Sources: the dense-reference parity test on
the multimodal-pruning page ("[Kernel][Gemma4] Prune Triton sliding-window tiles for
multimodal prefixes", 评论区精华) and its first risk (风险与影响): bounds, masks and numerics
must agree."""
import pytest

from paged_kv_prefix_gb300 import binding
from tests import rescale_cases as rc
from tests.gpu_util import parity

pytestmark = pytest.mark.gpu

FP8_PATHS = pytest.mark.parametrize("fp8_path", [0, binding.PPA_FLAG_FP8_INKERNEL],
                                    ids=["prepass", "inkernel"])


@pytest.mark.parametrize("spec", rc.PREFILL, ids=lambda s: s[0])
def test_rescale_prefill(spec):
    parity(rc.build(spec))


def test_rescale_large_softmax_scale():
    parity(rc.build(rc.LARGE_SCALE))


@FP8_PATHS
@pytest.mark.parametrize("spec", [rc.PREFILL[1], rc.PREFILL[2], rc.PREFILL[4]],
                         ids=lambda s: s[0])
def test_rescale_fp8(spec, fp8_path):
    parity(rc.build(spec, kv_dtype="fp8_e4m3"), flags_extra=fp8_path)


@pytest.mark.parametrize("split", [2, 3])
def test_rescale_split_kv(split):
    parity(rc.build(rc.DECODE), kv_split_tiles=split)


@FP8_PATHS
def test_rescale_split_kv_fp8(fp8_path):
    parity(rc.build(rc.DECODE, kv_dtype="fp8_e4m3"), flags_extra=fp8_path, kv_split_tiles=3)


def test_rescale_split_kv_head_dim_256():
    parity(rc.build(rc.DECODE, head_dim=256, seed=89), kv_split_tiles=3)
