"""CPU oracle for chunked-prefill attention over a paged KV cache.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this module. The library (``paged_kv_prefix_gb300``) never does,
and this module imports nothing from the library: the two share only the seeded input
generators in ``paged_kv_prefix_gb300/workloads.py``, which hold no attention arithmetic.

It is the plain definition, written out slowly:

* K/V of a sequence are gathered token by token. A context position ``p < c`` comes from
  physical page ``block_table[b][p // P]``, slot ``p % P``. A new position ``p >= c``
  comes from ``k_new/v_new`` row ``cu_query_lens[b] + p - c``. Every context token is
  resolved to its own (page, slot) pair, so a tile may straddle pages and the page size can
  be any integer.
  Sources: PR #54194 report (prefix-prefill tiles decoupled from page size), sections
  "功能与动机" (motivation) and "关键源码片段" (the note on ``_paged_kv_cache_offsets``).
* The (query, key) mask is the base causal/window mask OR-ed with the multimodal
  ranges. Sources: "[Kernel][Gemma4] Prune Triton sliding-window tiles for multimodal
  prefixes" (PR #53147), sections "实现拆解" items 1-2 and "关键源码片段"
  (``compute_tile_loop_bounds``), and "[Kernel] Skip fully masked key blocks in windowed
  Triton prefill" (PR #50776), "关键源码片段" (``SLIDING_WINDOW_Q``/``SLIDING_WINDOW_K``).
* A dense softmax over the full row, then a weighted sum of V. The computation is fp32,
  as in the fp32 reference of the PR #54194 report ("实现拆解" item 4). Pins may pass
  ``dtype=np.float64``.

Readings where the pages are silent or disagree:

* Window ``W > 0`` on the left admits keys with ``q - k < W``, i.e. ``q-W+1 .. q``
  (PR #53147 ``first_allowed_key = q_abs - SLIDING_WINDOW + 1``). The same convention
  applies on the right: ``k - q < W``. ``W <= 0`` means unbounded on that side. The
  right window only applies when non-causal.
* A multimodal range ``[a, e]`` is inclusive of ``e``. It is valid iff ``a < e``, and its
  end is clipped to ``s - 1``. A query ``q`` inside the range may attend to every key
  inside it (bidirectional). With the clamp flag and a left window, such a key must also
  satisfy ``q - k < W``.
* Chunked-local attention (``chunk_size > 0``, PR #53147 "关键源码片段", the
  ``CHUNK_LOOKBACK >= 0`` branch of ``compute_tile_loop_bounds``): the base mask's left
  edge becomes ``k >= ((q // CS) - LB) * CS`` in place of the left window; the right edge is
  unchanged. Multimodal ranges are still clamped by the ordinary left window (section
  "评论区精华": the MM mask is OR-ed on and clamped by the sliding window, so it can re-enable
  keys before the chunk boundary). The page prints only the tile bound, taken at the block's
  last row; the per-pair predicate is this reading of it.
* Per-sequence causality (``USE_PER_SEQ_CAUSAL`` on the PR #53147 page, where the tile
  bound takes the non-causal right edge because causality is decided per sequence inside
  the mask): ``inp["seq_causal"][b]``, when given, replaces the batch's causal flag for
  sequence ``b``.
* The softmax scale defaults to ``1/sqrt(D)``. Query head ``h`` reads KV head
  ``h // (Hq/Hkv)``.
* fp8 caches hold OCP E4M3 "fn" codes (no infinities, S.1111.111 is NaN). The value is
  ``decode(code) * scale``, with one fp32 scale for K and one for V.
* KV append. The PR #54194 report ("实现拆解" item 4) validates the kernel on a
  ``k=None`` cache-sourced path, where the new tokens' K/V are read from the paged cache;
  the pages print no code that writes them there, so the append is a reading: new token
  ``j`` of sequence ``b`` is written to position ``c + j`` of the sequence, i.e. page ``block_table[b][(c + j) // P]``, slot
  ``(c + j) % P``. A bf16 cache takes the value unchanged. An fp8 cache takes the code
  nearest to ``value / scale`` (the quotient formed in fp32), ties to the even code,
  magnitudes past 448 saturated to 448, NaN to a NaN code. The pages name only the dtype,
  so this encoding is a reading: round to nearest even is the IEEE default, and saturation
  keeps an out-of-range value finite rather than NaN.
* Cache-sourced attention (``inp["kv_in_cache"]``): the new tokens' K/V are read from the
  cache at positions ``c .. s-1`` instead of from ``k_new/v_new``.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

__all__ = [
    "e4m3fn_table",
    "e4m3fn_encode",
    "append_kv",
    "allowed_pair",
    "allowed_mask",
    "gather_kv",
    "attention",
    "attention_rows",
    "tile_bounds",
    "live_pairs",
]


# ---------------------------------------------------------------------------------------
# fp8 e4m3fn decode, from the bit definition (1 sign, 4 exponent bits with bias 7,
# 3 mantissa bits; exponent 0 is subnormal; 0x7F/0xFF are NaN; there is no infinity).
# ---------------------------------------------------------------------------------------
def e4m3fn_table() -> np.ndarray:
    """Value of each of the 256 codes as float64 (NaN for the two NaN codes)."""
    table = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if (code >> 7) & 1 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            table[code] = math.nan
        elif exp == 0:
            table[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)
        else:
            table[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return table


_E4M3 = e4m3fn_table()


def e4m3fn_encode(x) -> np.ndarray:
    """Codes of float32 values ``x``: the nearest finite E4M3 value, ties to the even code,
    magnitudes above the largest finite value (448) saturated to it, NaN to 0x7F. The
    sign bit is the value's (so -0.0 gives 0x80). Finite positive codes 0x00 .. 0x7E
    increase with their value, so the search runs over that table."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    pos = _E4M3[:0x7F]  # codes 0 .. 126, ascending, all finite
    hi = np.clip(np.searchsorted(pos, mag, side="left"), 0, 0x7E)  # first value >= mag
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = np.abs(pos[hi] - mag)
    d_lo = np.abs(mag - pos[lo])
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(take_lo, lo, hi)
    code = np.where(mag >= pos[0x7E], 0x7E, code)  # saturate (also +-inf)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


# ---------------------------------------------------------------------------------------
# The mask.
# ---------------------------------------------------------------------------------------
def _chunk_first_key(q, chunk_size: int, chunk_lookback: int):
    """First key of the chunk ``chunk_lookback`` chunks before query ``q``'s own chunk."""
    return ((q // chunk_size) - chunk_lookback) * chunk_size


def allowed_pair(q: int, k: int, s: int, causal: bool, window_left: int, window_right: int,
                 ranges: Optional[Iterable], clamp: bool, chunk_size: int = 0,
                 chunk_lookback: int = 0) -> bool:
    """Whether query position ``q`` may attend to key position ``k`` (scalar form).

    base: causal ``k <= q`` (else ``k - q < WR`` when ``WR > 0``), and ``q - k < WL``
    when ``WL > 0`` (with ``chunk_size > 0``: ``k >= ((q // CS) - LB) * CS`` instead). mm:
    some valid range contains both q and k (clamped by ``WL`` when ``clamp``). The result is
    base OR mm.
    """
    if k < 0 or k >= s or q < 0 or q >= s:
        return False
    if causal:
        right_ok = k <= q
    else:
        right_ok = window_right <= 0 or (k - q) < window_right
    if chunk_size > 0:
        left_ok = k >= _chunk_first_key(q, chunk_size, chunk_lookback)
    else:
        left_ok = window_left <= 0 or (q - k) < window_left
    if right_ok and left_ok:
        return True
    if ranges is None:
        return False
    for a, e in ranges:
        a, e = int(a), int(e)
        if not a < e:
            continue
        e = min(e, s - 1)
        if a <= q <= e and a <= k <= e:
            if clamp and window_left > 0 and not (q - k) < window_left:
                continue
            return True
    return False


def allowed_mask(q_pos: np.ndarray, s: int, causal: bool, window_left: int, window_right: int,
                 ranges: Optional[np.ndarray], clamp: bool, chunk_size: int = 0,
                 chunk_lookback: int = 0) -> np.ndarray:
    """Dense ``[len(q_pos), s]`` boolean mask, the same predicate as :func:`allowed_pair`."""
    qq = np.asarray(q_pos, dtype=np.int64)[:, None]
    kk = np.arange(s, dtype=np.int64)[None, :]
    if causal:
        right_ok = kk <= qq
    elif window_right > 0:
        right_ok = (kk - qq) < window_right
    else:
        right_ok = np.ones((1, s), dtype=bool)
    if chunk_size > 0:
        left_ok = kk >= _chunk_first_key(qq, chunk_size, chunk_lookback)
    elif window_left > 0:
        left_ok = (qq - kk) < window_left
    else:
        left_ok = np.ones((1, s), dtype=bool)
    mask = np.broadcast_to(right_ok & left_ok, (qq.shape[0], s)).copy()
    if ranges is not None:
        for a, e in np.asarray(ranges, dtype=np.int64).reshape(-1, 2):
            if not a < e:
                continue
            e = min(e, s - 1)
            mm = (a <= qq) & (qq <= e) & (a <= kk) & (kk <= e)
            if clamp and window_left > 0:
                mm = mm & ((qq - kk) < window_left)
            mask = mask | mm
    return mask


# ---------------------------------------------------------------------------------------
# Paged gather, token by token.
# ---------------------------------------------------------------------------------------
def _cache_value(inp: dict, which: str, page: int, slot: int, dtype) -> np.ndarray:
    cache = inp[f"{which}_cache"]
    row = cache[page, slot]  # [Hkv, D]
    if inp["kv_dtype"] == "bf16":
        return row.astype(dtype)
    scale = inp[f"{which}_scale"]
    return (_E4M3[row.astype(np.int64)] * scale).astype(dtype)


def gather_kv(inp: dict, b: int, which: str, dtype=np.float32) -> np.ndarray:
    """K or V of sequence ``b`` at positions ``0 .. s-1``, shape ``[s, Hkv, D]``. With
    ``inp["kv_in_cache"]`` every position comes from the cache."""
    P = inp["page_size"]
    c = int(inp["context_lens"][b])
    cu = inp["cu_query_lens"]
    n = int(cu[b + 1] - cu[b])
    new = inp[f"{which}_new"]
    from_cache = c + n if inp.get("kv_in_cache") else c
    rows = []
    for p in range(c + n):
        if p < from_cache:
            page = int(inp["block_table"][b, p // P])
            rows.append(_cache_value(inp, which, page, p % P, dtype))
        else:
            rows.append(new[int(cu[b]) + p - c].astype(dtype))
    if not rows:
        return np.zeros((0, inp["num_kv_heads"], inp["head_dim"]), dtype=dtype)
    return np.stack(rows)


def _seq_ranges(inp: dict, b: int) -> Optional[np.ndarray]:
    mm = inp.get("mm_ranges")
    return None if mm is None else mm[b]


def _causal(inp: dict, b: int) -> bool:
    """Whether sequence ``b``'s base mask is causal."""
    sc = inp.get("seq_causal")
    return bool(inp["causal"]) if sc is None else bool(sc[b])


def _chunk(inp: dict) -> dict:
    """The chunked-local parameters of a batch (absent: off)."""
    return {"chunk_size": int(inp.get("chunk_size", 0) or 0),
            "chunk_lookback": int(inp.get("chunk_lookback", 0) or 0)}


def _scale(inp: dict) -> float:
    sm = inp["sm_scale"]
    return sm if sm > 0 else 1.0 / math.sqrt(inp["head_dim"])


# ---------------------------------------------------------------------------------------
# Attention.
# ---------------------------------------------------------------------------------------
def _softmax_rows(scores: np.ndarray, mask: np.ndarray) -> np.ndarray:
    scores = np.where(mask, scores, -np.inf)
    m = scores.max(axis=1, keepdims=True)
    p = np.exp(scores - m)
    return p / p.sum(axis=1, keepdims=True)


def attention_rows(inp: dict, b: int, tokens: np.ndarray, dtype=np.float32,
                   kv: Optional[tuple] = None) -> np.ndarray:
    """Output rows ``[len(tokens), Hq, D]`` for query tokens ``tokens`` (indices within
    sequence ``b``'s new tokens)."""
    Hq, Hkv, D = inp["num_q_heads"], inp["num_kv_heads"], inp["head_dim"]
    G = Hq // Hkv
    c = int(inp["context_lens"][b])
    cu = inp["cu_query_lens"]
    n = int(cu[b + 1] - cu[b])
    s = c + n
    K, V = kv if kv is not None else (gather_kv(inp, b, "k", dtype), gather_kv(inp, b, "v", dtype))
    tokens = np.asarray(tokens, dtype=np.int64)
    mask = allowed_mask(c + tokens, s, _causal(inp, b), inp["window_left"], inp["window_right"],
                        _seq_ranges(inp, b), inp["clamp_mm"], **_chunk(inp))
    Q = inp["q"][int(cu[b]) + tokens].astype(dtype)  # [t, Hq, D]
    scale = dtype(_scale(inp))
    out = np.empty((len(tokens), Hq, D), dtype=dtype)
    for h in range(Hq):
        g = h // G
        scores = (Q[:, h, :] @ K[:, g, :].T) * scale
        out[:, h, :] = _softmax_rows(scores, mask) @ V[:, g, :]
    return out


def attention(inp: dict, dtype=np.float32, row_chunk: int = 1024) -> np.ndarray:
    """Full output ``[total_q, Hq, D]``."""
    Hq, D = inp["num_q_heads"], inp["head_dim"]
    cu = inp["cu_query_lens"]
    B = len(inp["context_lens"])
    out = np.zeros((int(cu[-1]), Hq, D), dtype=dtype)
    for b in range(B):
        n = int(cu[b + 1] - cu[b])
        if n == 0:
            continue
        kv = (gather_kv(inp, b, "k", dtype), gather_kv(inp, b, "v", dtype))
        for j0 in range(0, n, row_chunk):
            toks = np.arange(j0, min(n, j0 + row_chunk))
            out[int(cu[b]) + toks] = attention_rows(inp, b, toks, dtype, kv)
    return out


# ---------------------------------------------------------------------------------------
# KV append.
# ---------------------------------------------------------------------------------------
def append_kv(inp: dict) -> tuple:
    """The caches after writing every new token: ``(k_cache, v_cache)`` copies, float32
    values for a bf16 cache, uint8 codes for an fp8 one. Slots no new token maps to keep
    their contents."""
    P = inp["page_size"]
    cu = inp["cu_query_lens"]
    out = []
    for which in ("k", "v"):
        cache = inp[f"{which}_cache"].copy()
        new = inp[f"{which}_new"]
        scale = np.float32(inp[f"{which}_scale"])
        for b in range(len(inp["context_lens"])):
            c = int(inp["context_lens"][b])
            for j in range(int(cu[b + 1] - cu[b])):
                pos = c + j
                page = int(inp["block_table"][b, pos // P])
                row = new[int(cu[b]) + j].astype(np.float32)  # [Hkv, D]
                if inp["kv_dtype"] == "bf16":
                    cache[page, pos % P] = row
                else:
                    cache[page, pos % P] = e4m3fn_encode(row / scale)  # fp32 quotient
        out.append(cache)
    return tuple(out)


# ---------------------------------------------------------------------------------------
# Live key tiles and live pairs, by brute force over the dense mask.
# ---------------------------------------------------------------------------------------
def tile_bounds(inp: dict, tq: int, tn: int) -> np.ndarray:
    """``[query tiles, 2]`` int32: for each (sequence, query tile of ``tq`` tokens) in order,
    ``lo = min(K*) // tn`` and ``hi = max(K*) // tn + 1`` where ``K*`` is the set of keys
    that at least one query of the tile may attend to."""
    cu = inp["cu_query_lens"]
    out = []
    for b in range(len(cu) - 1):
        c = int(inp["context_lens"][b])
        n = int(cu[b + 1] - cu[b])
        s = c + n
        for t in range(-(-n // tq)):
            toks = np.arange(t * tq, min(n, (t + 1) * tq))
            mask = allowed_mask(c + toks, s, _causal(inp, b), inp["window_left"],
                                inp["window_right"], _seq_ranges(inp, b), inp["clamp_mm"],
                                **_chunk(inp))
            live = np.nonzero(mask.any(axis=0))[0]
            out.append((live.min() // tn, live.max() // tn + 1))
    return np.asarray(out, dtype=np.int32).reshape(-1, 2)


def live_pairs(inp: dict, row_chunk: int = 2048) -> int:
    """Number of allowed (query token, key) pairs summed over all sequences (one head)."""
    cu = inp["cu_query_lens"]
    total = 0
    for b in range(len(cu) - 1):
        c = int(inp["context_lens"][b])
        n = int(cu[b + 1] - cu[b])
        for j0 in range(0, n, row_chunk):
            toks = np.arange(j0, min(n, j0 + row_chunk))
            total += int(allowed_mask(c + toks, c + n, _causal(inp, b), inp["window_left"],
                                      inp["window_right"], _seq_ranges(inp, b),
                                      inp["clamp_mm"], **_chunk(inp)).sum())
    return total
