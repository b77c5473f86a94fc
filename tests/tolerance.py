"""Tolerances for comparing the library's bf16 attention output with the fp32 oracle.

Two bars, both applied by the parity tests:

* ``within_bar``: the stated acceptance bar, max-abs 2e-2 with rtol 2e-2 (the tolerance of
  the dense-reference parity test on the multimodal-pruning page, "[Kernel][Gemma4] Prune
  Triton sliding-window tiles for multimodal prefixes", 评论区精华).
* ``tight_tolerance``: a per-element bound derived from the rounding the kernels do. It is much
  smaller than 2e-2 on long rows, where an output is an average over thousands of keys and
  one missing key tile moves it by far less than 2e-2. The kernels compute scores and the
  softmax in fp32 and round in three places:

  1. each unnormalised weight p_k (at most 2^8 times the row's running reference) is rounded
     to bf16 for the PV product: a relative error delta_k with |delta_k| <= 2^-9, from round
     to nearest even, so uniform and independent across keys;
  2. with an fp8 cache, each cached K and V element enters the tensor cores as
     bf16(decode(code) * scale): the same kind of relative error per element, which moves
     the score of key k by about ``scale * 2^-9 * sqrt(sum_e (q_e k_e)^2)`` and its value row
     by ``2^-9 * v_k``;
  3. the output O / l is rounded to bf16: at most half an ulp, 2^-8 * |out| (8-bit
     significand).

  The row sum l uses the unrounded p_k, so error (1) adds ``sum_k w_k delta_k v_k`` to the
  output, w the normalised softmax weights; its standard deviation is
  ``2^-9 / sqrt(3) * sqrt(sum_k w_k^2 v_k^2)``. The bound is ``2^-8 |want| + 10 sigma + 1e-5``
  with sigma the combined standard deviation of (1) and, for fp8, (2); 1e-5 covers the fp32
  accumulation in the tensor cores and in the oracle.

Test infrastructure: only the tests import this module.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import ref

ATOL = 2e-2
RTOL = 2e-2


def within_bar(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Elementwise: |got - want| <= 2e-2 + 2e-2 |want|."""
    return np.abs(got - want) <= ATOL + RTOL * np.abs(want)


def _scale(inp: dict) -> float:
    sm = inp["sm_scale"]
    return sm if sm > 0 else 1.0 / math.sqrt(inp["head_dim"])


def tight_tolerance(inp: dict, b: int, toks: np.ndarray, want: np.ndarray, kv: tuple) -> np.ndarray:
    """Per-element bound ``[len(toks), Hq, D]`` for output rows ``toks`` of sequence ``b``
    (``want``: the oracle's rows; ``kv``: the oracle's gathered (K, V) of the sequence)."""
    Hq, Hkv, D = inp["num_q_heads"], inp["num_kv_heads"], inp["head_dim"]
    G = Hq // Hkv
    fp8 = inp["kv_dtype"] != "bf16"
    cu = inp["cu_query_lens"]
    c = int(inp["context_lens"][b])
    s = c + int(cu[b + 1] - cu[b])
    toks = np.asarray(toks, dtype=np.int64)
    sc_causal = inp.get("seq_causal")
    causal = bool(inp["causal"]) if sc_causal is None else bool(sc_causal[b])
    mm = inp.get("mm_ranges")
    mask = ref.allowed_mask(c + toks, s, causal, inp["window_left"], inp["window_right"],
                            None if mm is None else mm[b], inp["clamp_mm"],
                            int(inp.get("chunk_size", 0) or 0),
                            int(inp.get("chunk_lookback", 0) or 0))
    Q = inp["q"][int(cu[b]) + toks].astype(np.float64)
    K = kv[0].astype(np.float64)
    V = kv[1].astype(np.float64)
    scale = _scale(inp)
    tol = np.empty(want.shape, dtype=np.float64)
    for h in range(Hq):
        g = h // G
        scores = np.where(mask, (Q[:, h, :] @ K[:, g, :].T) * scale, -np.inf)
        w = np.exp(scores - scores.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        w2 = w * w
        v2 = V[:, g, :] ** 2
        var = w2 @ v2  # (1): p rounding
        if fp8:
            var += w2 @ v2  # (2): V element rounding
            gk2 = (scale ** 2) * ((Q[:, h, :] ** 2) @ (K[:, g, :] ** 2).T)  # score error scale^2
            wg = w2 * gk2
            out = want[:, h, :].astype(np.float64)
            var += wg @ v2 - 2.0 * (wg @ V[:, g, :]) * out + wg.sum(axis=1, keepdims=True) * out ** 2
        sigma = 2.0 ** -9 / math.sqrt(3.0) * np.sqrt(np.maximum(var, 0.0))
        tol[:, h, :] = 2.0 ** -8 * np.abs(want[:, h, :]) + 10.0 * sigma + 1e-5
    return tol
