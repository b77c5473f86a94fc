"""Inputs whose row maxima jump after a row's first live key tile, so that the attention
kernels' online softmax must rescale an output accumulator that already holds mass.

The kernels keep a stale row reference and rescale O only when a key tile's maximum exceeds
it by more than 8 (in log2 units, i.e. a factor 2^8 in the weights). With N(0, 1) inputs
and the default scale 1/sqrt(D) no score ever grows that far after the first tile, so these
cases shape Q and K (``workloads.build_case(logit_jump=...)``): column 0 of every query is 1
and its other columns are small, and column 0 of a sparse set of keys (every ``PERIOD``-th
position from ``FIRST``) is ``boost``. Those keys' scores sit about ``JUMP`` log2 units above
the rest. A row that first attends to ordinary keys and later reaches a boosted one takes the
rescale with alpha = 2^-JUMP or so, and the ordinary keys still carry roughly a fifth of its
softmax mass (one boosted key outweighs 2^JUMP ordinary ones, and there are PERIOD ordinary
keys per boosted one), so a wrong alpha moves the output far beyond the tolerance.

Test infrastructure: only the tests import this module.
"""
from __future__ import annotations

import math

from paged_kv_prefix_gb300 import workloads as wl

JUMP = 9.5      # log2 units; the kernels rescale above 8
FIRST = 330     # first boosted key position (tile 2 of 128-key tiles)
PERIOD = 173    # boosted keys are sparse: about one per 128-key tile


def boost_for(head_dim: int, sm_scale: float = 0.0) -> float:
    """Column-0 key value that lifts a score by JUMP log2 units over an ordinary key."""
    scale = sm_scale if sm_scale > 0 else 1.0 / math.sqrt(head_dim)
    return JUMP / (scale * math.log2(math.e))


def case(name: str, ctx, qlen, num_q_heads: int, num_kv_heads: int, head_dim: int,
         page_size: int = 37, sm_scale: float = 0.0, q_noise: float = 0.1, seed: int = 0,
         **kw):
    return wl.build_case(name, ctx, qlen, num_q_heads, num_kv_heads, head_dim, page_size,
                         causal=True, sm_scale=sm_scale, seed=seed,
                         logit_jump=(boost_for(head_dim, sm_scale), FIRST, PERIOD, q_noise), **kw)


# (name, builder kwargs): prefill rows over several key tiles, for both attention kernels
# (head dims 64/128 single CTA, 256 on CTA pairs), groups of 1 and 8 query heads per KV head.
PREFILL = [
    (f"jump_d{d}_g{g}", dict(ctx=[0, 300, 1000], qlen=[700, 260, 150], num_q_heads=2 * g,
                             num_kv_heads=2, head_dim=d, seed=10 * d + g))
    for d in (64, 128, 256) for g in (1, 8)
]

# A large softmax scale (1.0 instead of 1/sqrt(D)); the query noise shrinks with it so that
# the first tile's maximum stays close to the ordinary scores.
LARGE_SCALE = ("jump_scale1_d128", dict(ctx=[500, 0], qlen=[300, 600], num_q_heads=8,
                                        num_kv_heads=2, head_dim=128, sm_scale=1.0,
                                        q_noise=0.01, seed=77))

# Decode and verification rows over long contexts, for split-KV: segments whose first tile
# holds no boosted key rescale within the segment.
DECODE = ("jump_decode_d128", dict(ctx=[2900, 2100, 3500], qlen=[1, 4, 8], num_q_heads=16,
                                   num_kv_heads=2, head_dim=128, seed=88))


def build(spec, **extra):
    name, kw = spec
    kw = dict(kw)
    kw.update(extra)
    return case(name, **kw)
