"""Seeded synthetic inputs for chunked-prefill attention over a paged KV cache.

This module only *generates data*: random Q/K/V values, the page permutation, the block
table, ragged lengths and multimodal ranges, laid out as the library's C ABI expects
(``include/ppa.h``). It holds none of the attention arithmetic, so both the CUDA path and
the CPU oracle can take their inputs from it.

Layouts (all row-major, see ``include/ppa.h``):

* ``q``                      ``[total_q, Hq, D]``  bf16
* ``k_new``, ``v_new``       ``[total_q, Hkv, D]`` bf16
* ``k_cache``, ``v_cache``   ``[num_pages, P, Hkv, D]`` bf16, or uint8 e4m3fn codes
* ``block_table``            ``[B, max_pages_per_seq]`` int32 (logical page -> physical page)
* ``cu_query_lens``          ``[B + 1]`` int32, ``context_lens`` ``[B]`` int32
* ``mm_ranges``              ``[B, R, 2]`` int32, ``[start, end]`` with ``end`` inclusive

The pages a sequence owns cover all ``c + n`` of its positions (as a serving engine
allocates them), but only the first ``ceil(c / P)`` are meant to be read. With
``poison=True`` every cache slot that must never be read (slots of new tokens, spare
pages, block-table padding) holds NaN, so an implementation that reads one produces NaN
instead of a silently plausible value.

The named workloads at the bottom follow the shapes of the experiments and tests described
in the vLLM PR reports on prefix-prefill tiles (PR #54194), windowed key-block skipping
(PR #50776) and clamped multimodal prefixes (PR #53147); values are N(0, 1), no dataset is
involved.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass
class PrefillCase:
    """One batch of chunked-prefill work, as host (CPU) tensors."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    causal: bool
    window_left: int
    window_right: int
    clamp_mm: bool
    kv_dtype: str  # "bf16" or "fp8_e4m3"
    sm_scale: float  # <= 0 means 1/sqrt(head_dim)
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_scale: float
    v_scale: float
    block_table: torch.Tensor
    cu_query_lens: torch.Tensor
    context_lens: torch.Tensor
    mm_ranges: Optional[torch.Tensor]
    chunk_size: int = 0      # > 0: chunked-local attention (base left edge at a chunk start)
    chunk_lookback: int = 0  # chunks before the query's own chunk that stay visible
    seq_causal: Optional[torch.Tensor] = None  # int32 [B]: per-sequence causal flags

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.numel())

    @property
    def total_q(self) -> int:
        return int(self.cu_query_lens[-1])

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def max_mm_ranges(self) -> int:
        return 0 if self.mm_ranges is None else int(self.mm_ranges.shape[1])

    @property
    def query_lens(self) -> np.ndarray:
        cu = self.cu_query_lens.numpy()
        return (cu[1:] - cu[:-1]).astype(np.int64)

    @property
    def seq_lens(self) -> np.ndarray:
        return self.context_lens.numpy().astype(np.int64) + self.query_lens

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "seed": self.seed,
            "num_seqs": self.num_seqs,
            "total_q": self.total_q,
            "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "page_size": self.page_size,
            "causal": self.causal,
            "window_left": self.window_left,
            "window_right": self.window_right,
            "mm_ranges_per_seq": self.max_mm_ranges,
            "clamp_mm": self.clamp_mm,
            "kv_dtype": self.kv_dtype,
            "context_tokens": int(self.context_lens.sum()),
        }

    def numpy_inputs(self) -> dict:
        """Plain NumPy copies for CPU consumers (bf16 -> float32 is exact)."""
        out = {
            "q": self.q.float().numpy(),
            "k_new": self.k_new.float().numpy(),
            "v_new": self.v_new.float().numpy(),
            "block_table": self.block_table.numpy().astype(np.int64),
            "cu_query_lens": self.cu_query_lens.numpy().astype(np.int64),
            "context_lens": self.context_lens.numpy().astype(np.int64),
            "mm_ranges": None if self.mm_ranges is None else self.mm_ranges.numpy().astype(np.int64),
            "page_size": self.page_size,
            "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "causal": self.causal,
            "window_left": self.window_left,
            "window_right": self.window_right,
            "clamp_mm": self.clamp_mm,
            "sm_scale": self.sm_scale,
            "chunk_size": self.chunk_size,
            "chunk_lookback": self.chunk_lookback,
            "seq_causal": None if self.seq_causal is None else self.seq_causal.numpy().astype(bool),
            "kv_dtype": self.kv_dtype,
            "k_scale": self.k_scale,
            "v_scale": self.v_scale,
        }
        if self.kv_dtype == "bf16":
            out["k_cache"] = self.k_cache.float().numpy()
            out["v_cache"] = self.v_cache.float().numpy()
        else:
            out["k_cache"] = self.k_cache.numpy()  # uint8 codes
            out["v_cache"] = self.v_cache.numpy()
        return out


def _normal_bf16(rng: np.random.Generator, shape) -> torch.Tensor:
    return torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32)).to(torch.bfloat16)


def _quantize_e4m3(x: torch.Tensor) -> tuple[torch.Tensor, float]:
    """Per-tensor scale amax/448; codes from torch's round-to-nearest-even cast."""
    amax = float(x.abs().max()) if x.numel() else 1.0
    scale = (amax / E4M3_MAX) if amax > 0 else 1.0
    y = (x.float() / scale).clamp(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8), float(scale)


# The last value draw, reused by the next case with the same seed, lengths and head shape (the
# mixed-serving runs differ only in page size and window, so their values are identical).
_VALUE_MEMO: dict = {}


def _draw_values(seed_key, ctx: np.ndarray, qlen: np.ndarray, Hq: int, Hkv: int, D: int,
                 logit_jump: Optional[tuple]):
    """Q, k_new, v_new and every sequence's context K/V, drawn N(0, 1) in a fixed order from
    ``default_rng(seed_key)``; with ``logit_jump`` the Q and K values are then shaped as
    described in :func:`build_case`."""
    key = (seed_key if isinstance(seed_key, int) else tuple(seed_key), tuple(ctx.tolist()),
           tuple(qlen.tolist()), Hq, Hkv, D, logit_jump)
    if _VALUE_MEMO.get("key") == key:
        return _VALUE_MEMO["values"]
    _VALUE_MEMO.clear()
    rng = np.random.default_rng(seed_key)
    total_q = int(qlen.sum())
    q = _normal_bf16(rng, (total_q, Hq, D))
    k_new = _normal_bf16(rng, (total_q, Hkv, D))
    v_new = _normal_bf16(rng, (total_q, Hkv, D))
    ctx_k = [_normal_bf16(rng, (int(c), Hkv, D)) for c in ctx]
    ctx_v = [_normal_bf16(rng, (int(c), Hkv, D)) for c in ctx]
    if logit_jump is not None:
        boost, first, period, q_noise = logit_jump
        q = (q.float() * q_noise).to(torch.bfloat16)
        q[:, :, 0] = 1.0
        cu = np.concatenate([[0], np.cumsum(qlen)])
        for b in range(ctx.size):
            c, n = int(ctx[b]), int(qlen[b])
            pos = np.arange(c + n)
            col = np.where((pos >= first) & ((pos - first) % period == 0), boost, 0.0)
            col = torch.from_numpy(col.astype(np.float32)).to(torch.bfloat16)
            ctx_k[b][:, :, 0] = col[:c, None]
            k_new[int(cu[b]):int(cu[b]) + n, :, 0] = col[c:, None]
    values = (q, k_new, v_new, ctx_k, ctx_v)
    _VALUE_MEMO.update(key=key, values=values)
    return values


def build_case(
    name: str,
    context_lens: Sequence[int],
    query_lens: Sequence[int],
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    page_size: int,
    causal: bool = True,
    window_left: int = 0,
    window_right: int = 0,
    mm_ranges: Optional[np.ndarray] = None,
    clamp_mm: bool = False,
    kv_dtype: str = "bf16",
    sm_scale: float = 0.0,
    seed: int = 0,
    spare_frac: float = 0.10,
    poison: bool = True,
    value_rng_seed: Optional[int] = None,
    chunk_size: int = 0,
    chunk_lookback: int = 0,
    seq_causal: Optional[Sequence[bool]] = None,
    logit_jump: Optional[tuple] = None,
) -> PrefillCase:
    """Build one case. Lengths are per sequence; ``mm_ranges`` is ``[B, R, 2]`` or None.

    ``logit_jump = (boost, first, period, q_noise)`` shapes Q and K so that a row's scores
    jump upward once it reaches a sparse set of keys: every query row becomes
    ``(1, q_noise * N(0,1), ...)`` (column 0 set to 1, the rest scaled down) and column 0 of
    every key is 0, except at absolute positions ``first, first + period, ...`` of each
    sequence, where it is ``boost``. Those keys' scores then exceed the others' by about
    ``boost`` (times the softmax scale), while the rest stay close together."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    qlen = np.asarray(query_lens, dtype=np.int64)
    assert ctx.shape == qlen.shape and ctx.ndim == 1
    assert (ctx >= 0).all() and (qlen >= 0).all()
    B = ctx.size
    P = int(page_size)
    D = int(head_dim)
    Hq, Hkv = int(num_q_heads), int(num_kv_heads)
    layout_rng = np.random.default_rng([seed, 7919])

    total_q = int(qlen.sum())
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(qlen)

    q, k_new, v_new, ctx_k, ctx_v = _draw_values(
        seed if value_rng_seed is None else value_rng_seed, ctx, qlen, Hq, Hkv, D, logit_jump)

    # Pages owned by each sequence cover every position 0..s-1.
    s = ctx + qlen
    pages_per_seq = np.array([max(1, math.ceil(int(x) / P)) for x in s], dtype=np.int64)
    used = int(pages_per_seq.sum())
    spare = max(1, int(math.ceil(used * spare_frac)))
    num_pages = used + spare
    perm = layout_rng.permutation(num_pages)
    maxp = int(pages_per_seq.max()) if B else 1
    poison_page = int(perm[used])  # first spare page
    block_table = np.full((B, maxp), poison_page, dtype=np.int64)
    off = 0
    for b in range(B):
        block_table[b, : pages_per_seq[b]] = perm[off : off + pages_per_seq[b]]
        off += pages_per_seq[b]

    # Context K/V values (contiguous per sequence) are scattered into their pages.
    if kv_dtype == "bf16":
        fill = float("nan") if poison else 0.0
        k_cache = torch.full((num_pages, P, Hkv, D), fill, dtype=torch.bfloat16)
        v_cache = torch.full((num_pages, P, Hkv, D), fill, dtype=torch.bfloat16)
        k_src, v_src = ctx_k, ctx_v
        k_scale = v_scale = 1.0
    elif kv_dtype == "fp8_e4m3":
        allk = torch.cat(ctx_k) if B else torch.zeros(0)
        allv = torch.cat(ctx_v) if B else torch.zeros(0)
        kq, k_scale = _quantize_e4m3(allk)
        vq, v_scale = _quantize_e4m3(allv)
        splits = [int(c) for c in ctx]
        k_src = list(torch.split(kq, splits)) if B else []
        v_src = list(torch.split(vq, splits)) if B else []
        fill = 0x7F if poison else 0
        k_cache = torch.full((num_pages, P, Hkv, D), fill, dtype=torch.uint8)
        v_cache = torch.full((num_pages, P, Hkv, D), fill, dtype=torch.uint8)
    else:
        raise ValueError(f"unknown kv_dtype {kv_dtype!r}")

    for b in range(B):
        c = int(ctx[b])
        for lp in range(math.ceil(c / P)):
            lo, hi = lp * P, min(c, (lp + 1) * P)
            phys = int(block_table[b, lp])
            k_cache[phys, : hi - lo] = k_src[b][lo:hi]
            v_cache[phys, : hi - lo] = v_src[b][lo:hi]

    mm = None
    if mm_ranges is not None:
        mm = torch.from_numpy(np.asarray(mm_ranges, dtype=np.int32).reshape(B, -1, 2).copy())

    return PrefillCase(
        name=name,
        seed=seed,
        num_q_heads=Hq,
        num_kv_heads=Hkv,
        head_dim=D,
        page_size=P,
        causal=bool(causal),
        window_left=int(window_left),
        window_right=int(window_right),
        clamp_mm=bool(clamp_mm),
        kv_dtype=kv_dtype,
        sm_scale=float(sm_scale),
        q=q,
        k_new=k_new,
        v_new=v_new,
        k_cache=k_cache,
        v_cache=v_cache,
        k_scale=float(k_scale),
        v_scale=float(v_scale),
        block_table=torch.from_numpy(block_table.astype(np.int32)),
        cu_query_lens=torch.from_numpy(cu.astype(np.int32)),
        context_lens=torch.from_numpy(ctx.astype(np.int32)),
        mm_ranges=mm,
        chunk_size=int(chunk_size),
        chunk_lookback=int(chunk_lookback),
        seq_causal=None if seq_causal is None
        else torch.tensor([1 if x else 0 for x in seq_causal], dtype=torch.int32),
    )


# ---------------------------------------------------------------------------------------
# The named workloads. Each takes a ``scale`` in (0, 1] that shrinks lengths for parity
# tests the CPU oracle finishes in seconds while keeping the structure.
# ---------------------------------------------------------------------------------------

NONPOW2_SHAPES = [  # (num_q_heads, q heads per kv head, head_dim, page_size)
    (64, 1, 128, 544),
    (8, 4, 256, 1040),
    (8, 4, 256, 1056),
]

MIXED_PAGE_SIZES = [128, 512, 544, 1040, 1056, 2048]


def _scaled(x: int, scale: float, lo: int = 1) -> int:
    return max(lo, int(round(x * scale)))


def tiny(seed: int = 0, **kw) -> PrefillCase:
    """Batch 2, 4 q heads / 2 kv heads, D 64, page 16, context [0, 37], queries [19, 8], causal."""
    return build_case("tiny", [0, 37], [19, 8], 4, 2, 64, 16, causal=True, seed=seed, **kw)


def nonpow2(shape_idx: int, seed: int = 0, scale: float = 1.0, num_seqs: int = 8, **kw) -> PrefillCase:
    """Ragged batch, context U[0, 8192], query U[1, 2048], causal, non-power-of-2 pages."""
    hq, g, d, p = NONPOW2_SHAPES[shape_idx]
    rng = np.random.default_rng([seed, 101, shape_idx])
    ctx = rng.integers(0, _scaled(8192, scale, 0) + 1, size=num_seqs)
    qlen = rng.integers(1, _scaled(2048, scale) + 1, size=num_seqs)
    return build_case(f"nonpow2_h{hq}_g{g}_d{d}_p{p}", ctx, qlen, hq, hq // g, d, p,
                      causal=True, seed=seed, **kw)


def swa_noncausal(seed: int = 0, scale: float = 1.0, **kw) -> PrefillCase:
    """One sequence of 16384 new tokens, 8 heads, D 64, window 64 both sides, non-causal."""
    n = _scaled(16384, scale)
    return build_case("swa64_noncausal", [0], [n], 8, 8, 64, 16, causal=False,
                      window_left=64, window_right=64, seed=seed, **kw)


def swa_causal(seed: int = 0, scale: float = 1.0, seq_len: int = 32768, window: int = 1024,
               **kw) -> PrefillCase:
    """One sequence of 32768 new tokens, 8 heads, D 64, causal, left window 1024."""
    n = _scaled(seq_len, scale)
    return build_case(f"swa{window}_causal_{seq_len}", [0], [n], 8, 8, 64, 16, causal=True,
                      window_left=window, seed=seed, **kw)


def chunked_local(seed: int = 0, scale: float = 1.0, num_seqs: int = 4, seq_len: int = 32768,
                  chunk: int = 8192, lookback: int = 0, **kw) -> PrefillCase:
    """Chunked-local prefill: 4 x 32768 new tokens, 32 q / 8 kv heads, D 128, page 544,
    causal, chunks of 8192 keys (each query sees its own chunk's prefix)."""
    n = _scaled(seq_len, scale)
    c = max(1, _scaled(chunk, scale))
    return build_case(f"chunked{c}_lb{lookback}", [0] * num_seqs, [n] * num_seqs, 32, 8, 128,
                      544, causal=True, chunk_size=c, chunk_lookback=lookback, seed=seed, **kw)


def decode(seed: int = 0, scale: float = 1.0, num_seqs: int = 32, new_tokens: int = 1,
           **kw) -> PrefillCase:
    """Decode over long contexts: 32 sequences, context U[8192, 32768], 1 new token each
    (``new_tokens`` > 1: speculative verification), 32 q / 8 kv heads, D 128, page 544, causal."""
    rng = np.random.default_rng([seed, 404])
    ctx = [_scaled(int(x), scale) for x in rng.integers(8192, 32769, size=num_seqs)]
    return build_case(f"decode_n{new_tokens}", ctx, [new_tokens] * num_seqs, 32, 8, 128, 544,
                      causal=True, seed=seed, **kw)


def mm_ranges_for(seq_len: int, num_ranges: int, width: int, rng: np.random.Generator) -> np.ndarray:
    """Non-overlapping ranges [a, a + width - 1] at seeded random starts."""
    free = seq_len - num_ranges * width
    assert free >= 0
    u = np.sort(rng.integers(0, free + 1, size=num_ranges))
    a = u + width * np.arange(num_ranges)
    return np.stack([a, a + width - 1], axis=-1)


def clamped_mm(seed: int = 0, scale: float = 1.0, num_seqs: int = 4, num_ranges: int = 60,
               range_width: int = 256, **kw) -> PrefillCase:
    """4 x 16384 tokens, 16 q / 8 kv heads, D 256, causal, window 1024, 60 clamped ranges."""
    n = _scaled(16384, scale)
    rng = np.random.default_rng([seed, 303])
    nr = min(num_ranges, n // range_width)
    ranges = np.stack([mm_ranges_for(n, nr, range_width, rng) for _ in range(num_seqs)])
    return build_case("clamped_mm", [0] * num_seqs, [n] * num_seqs, 16, 8, 256, 16, causal=True,
                      window_left=_scaled(1024, scale), mm_ranges=ranges, clamp_mm=True,
                      seed=seed, **kw)


def mixed(page_size: int, windowed: bool, kv_dtype: str = "bf16", seed: int = 0,
          scale: float = 1.0, num_seqs: int = 32, **kw) -> PrefillCase:
    """32 seqs, context U[4096, 32768], query U[512, 4096], 32 q / 4 kv heads, D 128, causal."""
    rng = np.random.default_rng([seed, 505])
    ctx = rng.integers(_scaled(4096, scale, 0), _scaled(32768, scale, 0) + 1, size=num_seqs)
    qlen = rng.integers(_scaled(512, scale), _scaled(4096, scale) + 1, size=num_seqs)
    wl = _scaled(4096, scale) if windowed else 0
    return build_case(f"mixed_p{page_size}_w{wl}_{kv_dtype}", ctx, qlen, 32, 4, 128, page_size,
                      causal=True, window_left=wl, kv_dtype=kv_dtype, seed=seed, **kw)
