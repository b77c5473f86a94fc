"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Nothing here compares the oracle with itself. Each check uses an independent route:
values the pages print, brute force over tiny inputs, closed forms, library routines
(scipy softmax, torch scaled_dot_product_attention, torch's e4m3 conversion), or
invariants a wrong index or sign would break.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inp(case):
    return case.numpy_inputs()


def _manual_inp(q, k_new, v_new, context_k=None, context_v=None, *, causal=True, wl_=0, wr=0,
                ranges=None, clamp=False, page_size=16, sm_scale=0.0):
    """A single-sequence input dict built by hand (no generator), cache laid out
    contiguously: logical page i -> physical page i."""
    n, hq, d = q.shape
    hkv = k_new.shape[1]
    c = 0 if context_k is None else context_k.shape[0]
    npages = max(1, math.ceil((c + n) / page_size))
    kc = np.zeros((npages, page_size, hkv, d))
    vc = np.zeros((npages, page_size, hkv, d))
    for p in range(c):
        kc[p // page_size, p % page_size] = context_k[p]
        vc[p // page_size, p % page_size] = context_v[p]
    return {
        "q": q, "k_new": k_new, "v_new": v_new, "k_cache": kc, "v_cache": vc,
        "block_table": np.arange(npages)[None, :], "cu_query_lens": np.array([0, n]),
        "context_lens": np.array([c]), "mm_ranges": None if ranges is None else np.asarray(ranges)[None],
        "page_size": page_size, "num_q_heads": hq, "num_kv_heads": hkv, "head_dim": d,
        "causal": causal, "window_left": wl_, "window_right": wr, "clamp_mm": clamp,
        "sm_scale": sm_scale, "kv_dtype": "bf16", "k_scale": 1.0, "v_scale": 1.0,
    }


# ---------------------------------------------------------------------------------------
# (a) the mask: brute force on tiny inputs, and the structure pruning relies on
# ---------------------------------------------------------------------------------------
def _random_geometry(rng):
    s = int(rng.integers(1, 64))
    c = int(rng.integers(0, s + 1))
    causal = bool(rng.integers(0, 2))
    wl_ = int(rng.choice([0, 1, 2, 5, 17, 70]))
    wr = int(rng.choice([0, 1, 3, 9, 70]))
    nr = int(rng.integers(0, 4))
    ranges = []
    for _ in range(nr):
        a = int(rng.integers(-2, s + 3))
        e = int(a + rng.integers(-3, 25))
        ranges.append((a, e))
    ranges.append((0, 0))  # padding entry, never valid
    clamp = bool(rng.integers(0, 2))
    return s, c, causal, wl_, wr, np.array(ranges), clamp


def test_mask_vectorised_equals_pairwise_bruteforce():
    rng = np.random.default_rng(1)
    for _ in range(300):
        s, c, causal, wl_, wr, ranges, clamp = _random_geometry(rng)
        qpos = np.arange(c, s)
        dense = ref.allowed_mask(qpos, s, causal, wl_, wr, ranges, clamp)
        brute = np.array([[ref.allowed_pair(int(q), k, s, causal, wl_, wr, ranges, clamp)
                           for k in range(s)] for q in qpos], dtype=bool).reshape(len(qpos), s)
        assert dense.shape == brute.shape and (dense == brute).all()


def test_mask_rows_are_intervals_containing_the_diagonal():
    """Every row's allowed set is one contiguous interval that contains k = q. This is the
    property that makes a per-query-tile key interval exact."""
    rng = np.random.default_rng(2)
    for _ in range(300):
        s, c, causal, wl_, wr, ranges, clamp = _random_geometry(rng)
        qpos = np.arange(c, s)
        mask = ref.allowed_mask(qpos, s, causal, wl_, wr, ranges, clamp)
        for i, q in enumerate(qpos):
            live = np.nonzero(mask[i])[0]
            assert mask[i, q]
            assert live.max() - live.min() + 1 == live.size


def test_mask_textbook_cases():
    s = 40
    q = np.arange(s)
    causal = ref.allowed_mask(q, s, True, 0, 0, None, False)
    assert (causal == np.tril(np.ones((s, s), bool))).all()
    full = ref.allowed_mask(q, s, False, 0, 0, None, False)
    assert full.all()
    band = ref.allowed_mask(q, s, False, 3, 5, None, False)
    expect = np.triu(np.tril(np.ones((s, s), bool), 4), -2)  # k-q <= 4 and q-k <= 2
    assert (band == expect).all()
    # an MM range admits future keys inside it even when causal
    mm = ref.allowed_mask(q, s, True, 0, 0, np.array([[10, 19]]), False)
    assert mm[12, 19] and not mm[12, 20] and not mm[9, 10]
    # range end is inclusive; a < e is required (a 1-token range is invalid)
    assert ref.allowed_mask(q, s, True, 0, 0, np.array([[10, 10]]), False).sum() == causal.sum()
    # the clamp keeps mm keys within the left window
    cl = ref.allowed_mask(q, s, True, 4, 0, np.array([[10, 30]]), True)
    assert cl[20, 17] and not cl[20, 16] and cl[20, 30]


# ---------------------------------------------------------------------------------------
# tile bounds: the page's printed geometry, and the p2 loop-limit formulas
# ---------------------------------------------------------------------------------------
def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _golden_rows("p4_tile_bounds.txt"))
def test_tile_bounds_page_fixture(row):
    c, n, tq, tn, t, wl_, wr, causal, clamp, a1, e1, a2, e2, lo, hi = row
    inp = {
        "cu_query_lens": np.array([0, n]), "context_lens": np.array([c]),
        "mm_ranges": np.array([[[a1, e1], [a2, e2]]]), "causal": bool(causal),
        "window_left": wl_, "window_right": wr, "clamp_mm": bool(clamp),
    }
    bounds = ref.tile_bounds(inp, tq, tn)
    assert tuple(bounds[t]) == (lo, hi)
    # Without the range the causal case prunes to the window alone; the range must widen it.
    if causal:
        inp["mm_ranges"] = np.array([[[0, 0], [0, 0]]])
        assert tuple(ref.tile_bounds(inp, tq, tn)[t]) == (3, 36)


def test_tile_bounds_within_windowed_prefill_loop_limits():
    """The windowed-prefill page clamps the key loop of query block m (rows m*BM..m*BM+BM-1,
    context 0) to start floor((m*BM - SW_Q)/BN)*BN and end min(end, (m+1)*BM - 1 + SW_K + 1),
    and causal to (m+1)*BM. Its left edge admits one key more than ours, so our exact live
    interval must lie inside those limits."""
    rng = np.random.default_rng(3)
    for _ in range(60):
        n = int(rng.integers(1, 300))
        bm = int(rng.choice([8, 16, 32]))
        bn = int(rng.choice([16, 32, 64]))
        causal = bool(rng.integers(0, 2))
        swq = int(rng.integers(1, 80))
        swk = 0 if causal else int(rng.integers(1, 80))
        inp = {"cu_query_lens": np.array([0, n]), "context_lens": np.array([0]),
               "mm_ranges": None, "causal": causal, "window_left": swq, "window_right": swk,
               "clamp_mm": False}
        mask_rows = ref.allowed_mask(np.arange(n), n, causal, swq, swk, None, False)
        for m in range(-(-n // bm)):
            live = np.nonzero(mask_rows[m * bm:(m + 1) * bm].any(axis=0))[0]
            start = max(0, ((m * bm - swq) // bn) * bn)
            end = n
            if causal:
                end = min(end, (m + 1) * bm)
            else:
                end = min(end, (m + 1) * bm - 1 + swk + 1)
            assert live.min() >= start and live.max() < end
            # and the oracle's tile interval is the tight one
            lo, hi = ref.tile_bounds(inp, bm, bn)[m]
            assert lo == live.min() // bn and hi == live.max() // bn + 1


def test_tile_bounds_exact_cover():
    """Pruning is exact: no allowed pair lies outside [lo*TN, hi*TN), and every key tile in
    [lo, hi) holds at least one allowed pair of the query tile."""
    case = wl.build_case("t", [13, 0, 40], [29, 17, 50], 2, 1, 8, 5, causal=True, window_left=9,
                         mm_ranges=np.array([[[3, 20], [30, 35]], [[2, 9], [0, 0]],
                                             [[41, 70], [50, 52]]]), clamp_mm=True, seed=4)
    inp = _inp(case)
    for tq, tn in [(4, 8), (7, 16), (16, 4)]:
        bounds = ref.tile_bounds(inp, tq, tn)
        i = 0
        for b in range(case.num_seqs):
            c = int(inp["context_lens"][b])
            n = int(inp["cu_query_lens"][b + 1] - inp["cu_query_lens"][b])
            for t in range(-(-n // tq)):
                toks = np.arange(t * tq, min(n, (t + 1) * tq))
                m = ref.allowed_mask(c + toks, c + n, True, 9, 0, inp["mm_ranges"][b], True)
                lo, hi = bounds[i]
                assert not m[:, : lo * tn].any() and not m[:, hi * tn:].any()
                for kt in range(lo, hi):
                    assert m[:, kt * tn:(kt + 1) * tn].any()
                i += 1
        assert i == len(bounds)


# ---------------------------------------------------------------------------------------
# (b), (c), (g): closed forms and library routines
# ---------------------------------------------------------------------------------------
def test_single_allowed_key_returns_its_value_row():
    case = wl.build_case("t", [0, 21], [33, 12], 4, 2, 64, 16, causal=True, window_left=1, seed=5)
    inp = _inp(case)
    out = ref.attention(inp)
    # each query sees only itself, a new token: the output is its own v_new row
    G = 2
    expect = np.repeat(inp["v_new"], G, axis=1)
    assert np.array_equal(out, expect)
    one = _manual_inp(inp["q"][:1], inp["k_new"][:1], inp["v_new"][:1])
    assert np.array_equal(ref.attention(one), np.repeat(inp["v_new"][:1], 2, axis=1))


def test_zero_query_returns_mean_of_allowed_values():
    case = wl.build_case("t", [0, 37, 5], [19, 8, 30], 4, 2, 32, 16, causal=True, window_left=11,
                         seed=6)
    inp = _inp(case)
    inp["q"] = np.zeros_like(inp["q"])
    out = ref.attention(inp, dtype=np.float64)
    for b in range(3):
        c = int(inp["context_lens"][b])
        cu = inp["cu_query_lens"]
        V = np.concatenate([
            np.stack([inp["v_cache"][inp["block_table"][b, p // 16], p % 16] for p in range(c)])
            if c else np.zeros((0, 2, 32)),
            inp["v_new"][cu[b]:cu[b + 1]]]).astype(np.float64)
        for j in range(int(cu[b + 1] - cu[b])):
            q = c + j
            keys = np.arange(max(0, q - 11 + 1), q + 1)  # causal with left window 11
            mean = V[keys].mean(axis=0)  # [Hkv, D]
            assert np.allclose(out[cu[b] + j], np.repeat(mean, 2, axis=0), atol=1e-12)


def test_textbook_softmax_attention_noncausal():
    from scipy.special import softmax
    rng = np.random.default_rng(7)
    n, h, d = 37, 3, 16
    q, k, v = (rng.standard_normal((n, h, d)) for _ in range(3))
    inp = _manual_inp(q, k, v, causal=False)
    out = ref.attention(inp, dtype=np.float64)
    for hh in range(h):
        p = softmax(q[:, hh] @ k[:, hh].T / math.sqrt(d), axis=1)
        assert np.allclose(out[:, hh], p @ v[:, hh], atol=1e-12)


@pytest.mark.parametrize("wl_", [0, 7])
def test_causal_prefix_gqa_against_torch_sdpa(wl_):
    """Context + new tokens, GQA 3, causal (bottom-right aligned) with an optional left
    window, against torch SDPA fed a mask built with tril/triu and K/V expanded per head."""
    rng = np.random.default_rng(8)
    c, n, hkv, g, d = 23, 17, 2, 3, 8
    ctx_k, ctx_v = rng.standard_normal((c, hkv, d)), rng.standard_normal((c, hkv, d))
    q = rng.standard_normal((n, hkv * g, d))
    kn, vn = rng.standard_normal((n, hkv, d)), rng.standard_normal((n, hkv, d))
    inp = _manual_inp(q, kn, vn, ctx_k, ctx_v, causal=True, wl_=wl_, page_size=5)
    out = ref.attention(inp, dtype=np.float64)
    K = torch.from_numpy(np.concatenate([ctx_k, kn])).permute(1, 0, 2).repeat_interleave(g, 0)
    V = torch.from_numpy(np.concatenate([ctx_v, vn])).permute(1, 0, 2).repeat_interleave(g, 0)
    Q = torch.from_numpy(q).permute(1, 0, 2)
    s = c + n
    mask = torch.ones(n, s, dtype=torch.bool).tril(diagonal=c)
    if wl_:
        mask &= torch.ones(n, s, dtype=torch.bool).triu(diagonal=c - wl_ + 1)
    expect = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    assert np.allclose(out, expect.permute(1, 0, 2).numpy(), atol=1e-12)


# ---------------------------------------------------------------------------------------
# the paged gather
# ---------------------------------------------------------------------------------------
def test_gather_follows_block_table_token_by_token():
    """A cache scattered by hand with a page size of 5 and a shuffled block table; every
    gathered row must carry its own position id."""
    P, c, n, hkv, d = 5, 23, 4, 2, 3
    npages = 9
    rng = np.random.default_rng(9)
    perm = rng.permutation(npages)
    kc = np.full((npages, P, hkv, d), np.nan)
    vc = np.full((npages, P, hkv, d), np.nan)
    for p in range(c):
        kc[perm[p // P], p % P] = p + np.arange(hkv)[:, None] * 1000
        vc[perm[p // P], p % P] = -p
    kn = (c + np.arange(n))[:, None, None] + np.zeros((n, hkv, d)) + np.arange(hkv)[:, None] * 1000
    inp = _manual_inp(np.zeros((n, hkv, d)), kn, -kn, causal=True, page_size=P)
    inp.update({"k_cache": kc, "v_cache": vc, "block_table": perm[None, :],
                "context_lens": np.array([c])})
    K = ref.gather_kv(inp, 0, "k", np.float64)
    V = ref.gather_kv(inp, 0, "v", np.float64)
    pos = np.arange(c + n)
    assert np.array_equal(K[:, 0, 0], pos) and np.array_equal(K[:, 1, 2], pos + 1000)
    assert np.array_equal(V[:, 0, 0], -pos)


def test_physical_page_permutation_invariance():
    """(d) Shuffling physical pages and rewriting the block table gives bitwise the same
    output."""
    a = wl.build_case("t", [37, 100], [19, 30], 4, 2, 32, 16, causal=True, seed=10,
                      value_rng_seed=99)
    b = wl.build_case("t", [37, 100], [19, 30], 4, 2, 32, 16, causal=True, seed=11,
                      value_rng_seed=99)
    assert not np.array_equal(a.block_table.numpy(), b.block_table.numpy())
    assert np.array_equal(ref.attention(_inp(a)), ref.attention(_inp(b)))


def test_pruned_keys_equal_dense():
    """(e) Attention over only the keys of [lo*TN, hi*TN) equals the dense-mask result."""
    case = wl.clamped_mm(seed=12, scale=1 / 64, num_seqs=2, num_ranges=3, range_width=40)
    inp = _inp(case)
    dense = ref.attention(inp, dtype=np.float64)
    tq, tn = 32, 16
    bounds = ref.tile_bounds(inp, tq, tn)
    i = 0
    for b in range(case.num_seqs):
        c = int(inp["context_lens"][b])
        cu = inp["cu_query_lens"]
        n = int(cu[b + 1] - cu[b])
        K, V = ref.gather_kv(inp, b, "k", np.float64), ref.gather_kv(inp, b, "v", np.float64)
        for t in range(-(-n // tq)):
            lo, hi = bounds[i]
            i += 1
            k0, k1 = lo * tn, min(hi * tn, c + n)
            toks = np.arange(t * tq, min(n, (t + 1) * tq))
            mask = ref.allowed_mask(c + toks, c + n, True, inp["window_left"], 0,
                                    inp["mm_ranges"][b], True)[:, k0:k1]
            for h in range(inp["num_q_heads"]):
                g = h // 2
                sc = inp["q"][cu[b] + toks, h].astype(np.float64) @ K[k0:k1, g].T / 16.0
                sc = np.where(mask, sc, -np.inf)
                p = np.exp(sc - sc.max(axis=1, keepdims=True))
                o = (p / p.sum(axis=1, keepdims=True)) @ V[k0:k1, g]
                assert np.allclose(o, dense[cu[b] + toks, h], atol=1e-12, rtol=0)


def test_removing_an_mm_range_changes_the_output():
    """(f) Negative control: dropping one image range must move the rows inside it by more
    than the parity tolerance."""
    case = wl.clamped_mm(seed=13, scale=1 / 32, num_seqs=1, num_ranges=2, range_width=100)
    inp = _inp(case)
    with_mm = ref.attention(inp)
    a, e = inp["mm_ranges"][0, 0]
    inp2 = dict(inp)
    mm = inp["mm_ranges"].copy()
    mm[0, 0] = (0, 0)
    inp2["mm_ranges"] = mm
    without = ref.attention(inp2)
    rows = slice(int(a), int(e) - 1)  # rows that see future keys inside the range
    assert np.abs(with_mm[rows] - without[rows]).max() > 2e-2
    outside = slice(int(e) + 1, int(inp["mm_ranges"][0, 1, 0]))
    assert np.array_equal(with_mm[outside], without[outside])


# ---------------------------------------------------------------------------------------
# fp8 e4m3fn
# ---------------------------------------------------------------------------------------
def test_e4m3fn_table_matches_torch_and_known_values():
    table = ref.e4m3fn_table()
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(table)
    assert (nan == np.isnan(lib)).all() and nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(table[~nan], lib[~nan])
    assert table[0x7E] == 448.0 and table[0x01] == 2.0 ** -9 and table[0x38] == 1.0
    assert table[0x08] == 2.0 ** -6 and table[0x80] == 0.0 and table[0xB8] == -1.0


def test_fp8_cache_dequantises_with_scale():
    case = wl.build_case("t", [30, 5], [7, 9], 4, 2, 16, 16, causal=True, kv_dtype="fp8_e4m3",
                         seed=14)
    inp = _inp(case)
    assert case.k_cache.dtype == torch.uint8 and inp["k_scale"] > 0
    K = ref.gather_kv(inp, 0, "k", np.float64)
    codes = case.k_cache.numpy()[case.block_table[0, 0].item(), 3]
    expect = codes.view(np.uint8).astype(np.int64)
    lib = torch.from_numpy(expect.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(K[3], lib * inp["k_scale"])


def test_live_pairs_matches_closed_form_for_causal_window():
    case = wl.build_case("t", [10, 0], [20, 50], 2, 1, 8, 16, causal=True, window_left=6, seed=15)
    inp = _inp(case)
    expect = 0
    for c, n in [(10, 20), (0, 50)]:
        for j in range(n):
            q = c + j
            expect += q - max(0, q - 5) + 1
    assert ref.live_pairs(inp) == expect


# ---------------------------------------------------------------------------------------
# e4m3 encoding and KV append (the step before attention: new tokens land in their pages)
# ---------------------------------------------------------------------------------------
def test_e4m3_encode_roundtrips_every_finite_code():
    table = ref.e4m3fn_table()
    fin = ~np.isnan(table)
    codes = np.arange(256)[fin].astype(np.uint8)
    assert np.array_equal(ref.e4m3fn_encode(table[fin].astype(np.float32)), codes)


def test_e4m3_encode_matches_the_library_cast_in_range():
    rng = np.random.default_rng(40)
    x = np.concatenate([rng.standard_normal(50000) * 50, rng.standard_normal(50000) * 0.01,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref.e4m3fn_encode(x), lib)


def test_e4m3_encode_ties_go_to_the_even_code():
    table = ref.e4m3fn_table()
    for k in range(0, 0x7E):  # midpoint of codes k and k+1 (exact in fp32: 5 significant bits)
        mid = np.float32((table[k] + table[k + 1]) / 2)
        assert float(mid) == (table[k] + table[k + 1]) / 2
        want = k if k % 2 == 0 else k + 1
        assert ref.e4m3fn_encode(mid) == want, k
        assert ref.e4m3fn_encode(-mid) == want | 0x80, k


def test_e4m3_encode_saturates_and_keeps_signs():
    enc = ref.e4m3fn_encode(np.array([1e6, -1e6, np.inf, -np.inf, 449.0, 470.0, -0.0, 0.0],
                                     dtype=np.float32))
    assert enc.tolist() == [0x7E, 0xFE, 0x7E, 0xFE, 0x7E, 0x7E, 0x80, 0x00]
    assert ref.e4m3fn_encode(np.float32(np.nan)) & 0x7F == 0x7F


def _appended(case):
    inp = _inp(case)
    k, v = ref.append_kv(inp)
    out = dict(inp)
    out["k_cache"], out["v_cache"], out["kv_in_cache"] = k, v, True
    return inp, out


@pytest.mark.parametrize("page", [1, 5, 16, 37])
def test_append_then_cache_sourced_gather_equals_the_new_token_tensors(page):
    case = wl.build_case("t", [0, 13, 40, 7], [9, 0, 21, 30], 4, 2, 16, page, causal=True,
                         seed=41 + page)
    inp, app = _appended(case)
    for b in range(4):
        for which in ("k", "v"):
            assert np.array_equal(ref.gather_kv(app, b, which, np.float64),
                                  ref.gather_kv(inp, b, which, np.float64)), (b, which)
    assert np.array_equal(ref.attention(app, np.float64), ref.attention(inp, np.float64))


def test_append_touches_only_the_new_tokens_slots():
    case = wl.build_case("t", [3, 20], [6, 11], 4, 2, 16, 8, causal=True, seed=42)
    inp, app = _appended(case)
    P, touched = 8, set()
    for b, (c, n) in enumerate([(3, 6), (20, 11)]):
        for pos in range(c, c + n):
            touched.add((int(inp["block_table"][b, pos // P]), pos % P))
    for page in range(inp["k_cache"].shape[0]):
        for slot in range(P):
            same = np.array_equal(app["k_cache"][page, slot], inp["k_cache"][page, slot],
                                  equal_nan=True)
            # untouched slots keep their contents; touched ones lose the NaN poison
            assert same == ((page, slot) not in touched), (page, slot)


def test_append_fp8_stores_the_encoded_quotient():
    case = wl.build_case("t", [17, 4], [12, 25], 4, 2, 16, 16, causal=True,
                         kv_dtype="fp8_e4m3", seed=43)
    inp, app = _appended(case)
    cu = inp["cu_query_lens"]
    for b, c in enumerate([17, 4]):
        K = ref.gather_kv(app, b, "k", np.float64)
        n = int(cu[b + 1] - cu[b])
        x = inp["k_new"][int(cu[b]):int(cu[b]) + n].astype(np.float32)
        codes = ref.e4m3fn_encode(x / np.float32(inp["k_scale"]))
        assert np.array_equal(K[c:], ref.e4m3fn_table()[codes.astype(np.int64)] * inp["k_scale"])
        assert np.array_equal(K[:c], ref.gather_kv(inp, b, "k", np.float64)[:c])


# ---------------------------------------------------------------------------------------
# chunked-local attention (base left edge at the start of the chunk LB chunks back)
# ---------------------------------------------------------------------------------------
def test_chunked_mask_vectorised_equals_pairwise_and_rows_stay_intervals():
    rng = np.random.default_rng(50)
    for _ in range(200):
        s, c, causal, wl_, wr, ranges, clamp = _random_geometry(rng)
        cs, lb = int(rng.choice([1, 3, 8, 16, 64])), int(rng.integers(0, 3))
        qpos = np.arange(c, s)
        dense = ref.allowed_mask(qpos, s, causal, wl_, wr, ranges, clamp, cs, lb)
        brute = np.array([[ref.allowed_pair(int(q), k, s, causal, wl_, wr, ranges, clamp, cs, lb)
                           for k in range(s)] for q in qpos], dtype=bool).reshape(len(qpos), s)
        assert (dense == brute).all()
        for i, q in enumerate(qpos):
            live = np.nonzero(dense[i])[0]
            assert dense[i, q] and live.max() - live.min() + 1 == live.size


def test_chunked_mask_textbook_cases():
    s = 50
    q = np.arange(s)
    causal = np.tril(np.ones((s, s), bool))
    # chunk 16, lookback 0: block-diagonal causal (each query sees its own chunk's prefix)
    m = ref.allowed_mask(q, s, True, 0, 0, None, False, 16, 0)
    blocks = (q[:, None] // 16) == (q[None, :] // 16)
    assert (m == (causal & blocks)).all()
    # lookback 1: position 37 sees keys 16 .. 37
    m1 = ref.allowed_mask(np.array([37]), s, True, 0, 0, None, False, 16, 1)
    assert np.nonzero(m1[0])[0].tolist() == list(range(16, 38))
    # a chunk at least as long as the sequence leaves the causal mask
    assert (ref.allowed_mask(q, s, True, 0, 0, None, False, 64, 0) == causal).all()
    # chunk 1: only the diagonal; the window_left is not part of the base mask then
    assert (ref.allowed_mask(q, s, True, 9, 0, None, False, 1, 0) == np.eye(s, dtype=bool)).all()
    # a clamped MM range re-enables keys before the chunk start (32), down to the window edge
    # (40 - 12 + 1 = 29, so the range start 30 binds) and up to the range end
    mm = ref.allowed_mask(np.array([40]), s, True, 12, 0, np.array([[30, 45]]), True, 16, 0)
    assert np.nonzero(mm[0])[0].tolist() == list(range(30, 46))
    # with a narrower window the clamped range starts inside the chunk: the chunk edge binds
    mm6 = ref.allowed_mask(np.array([40]), s, True, 6, 0, np.array([[30, 45]]), True, 16, 0)
    assert np.nonzero(mm6[0])[0].tolist() == list(range(32, 46))


def test_chunk_of_one_returns_each_querys_own_value_row():
    """With chunk size 1 and no lookback each causal query sees only itself: the output is
    its own V row, for every head of the group."""
    case = wl.build_case("t", [5, 0], [9, 12], 4, 2, 16, 8, causal=True, seed=51,
                         chunk_size=1, chunk_lookback=0)
    inp = _inp(case)
    out = ref.attention(inp, np.float64)
    cu = inp["cu_query_lens"]
    for b, c in enumerate([5, 0]):
        V = ref.gather_kv(inp, b, "v", np.float64)
        for j in range(int(cu[b + 1] - cu[b])):
            for h in range(4):
                assert np.allclose(out[int(cu[b]) + j, h], V[c + j, h // 2], rtol=0, atol=1e-12)


def test_per_sequence_causal_flags_select_each_sequences_mask():
    """A batch with per-sequence flags [causal, non-causal, causal] gives, row for row, the
    output of the same batch run all-causal for sequences 0 and 2 and all-non-causal for 1."""
    import dataclasses
    base = wl.build_case("t", [7, 20, 0], [15, 9, 11], 4, 2, 16, 8, causal=True,
                         window_right=5, seed=52)
    mixed = dataclasses.replace(base, seq_causal=torch.tensor([1, 0, 1], dtype=torch.int32))
    out = ref.attention(_inp(mixed), np.float64)
    all_c = ref.attention(_inp(base), np.float64)
    all_n = ref.attention(_inp(dataclasses.replace(base, causal=False)), np.float64)
    assert not np.allclose(all_c, all_n)
    rows = [(0, 15, all_c), (15, 24, all_n), (24, 35, all_c)]
    for a, e, want in rows:
        assert np.array_equal(out[a:e], want[a:e])


@pytest.mark.parametrize("chunk,lookback", [(4, 0), (8, 1), (5, 2)])
def test_chunked_local_against_torch_sdpa(chunk, lookback):
    """Chunked-local attention with context and GQA, against torch SDPA fed a block mask built
    from position indices with integer floor division (k // CS >= q // CS - LB) and K/V
    expanded per query head."""
    rng = np.random.default_rng(60 + chunk)
    c, n, hkv, g, d = 19, 14, 2, 2, 8
    ctx_k, ctx_v = rng.standard_normal((c, hkv, d)), rng.standard_normal((c, hkv, d))
    q = rng.standard_normal((n, hkv * g, d))
    kn, vn = rng.standard_normal((n, hkv, d)), rng.standard_normal((n, hkv, d))
    inp = _manual_inp(q, kn, vn, ctx_k, ctx_v, causal=True, page_size=7)
    inp["chunk_size"], inp["chunk_lookback"] = chunk, lookback
    out = ref.attention(inp, dtype=np.float64)
    K = torch.from_numpy(np.concatenate([ctx_k, kn])).permute(1, 0, 2).repeat_interleave(g, 0)
    V = torch.from_numpy(np.concatenate([ctx_v, vn])).permute(1, 0, 2).repeat_interleave(g, 0)
    Q = torch.from_numpy(q).permute(1, 0, 2)
    qpos = torch.arange(c, c + n)[:, None]
    kpos = torch.arange(c + n)[None, :]
    mask = (kpos <= qpos) & (kpos // chunk >= qpos // chunk - lookback)
    expect = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    assert np.allclose(out, expect.permute(1, 0, 2).numpy(), atol=1e-12)


def test_per_sequence_causal_against_torch_sdpa():
    """Two sequences, one causal and one bidirectional with a right window, each against torch
    SDPA with its own mask."""
    rng = np.random.default_rng(61)
    d, hkv, g = 8, 1, 2
    seqs = [(6, 9, True), (4, 11, False)]
    qs, kns, vns, out_want = [], [], [], []
    blocks = []
    for c, n, causal in seqs:
        ck, cv = rng.standard_normal((c, hkv, d)), rng.standard_normal((c, hkv, d))
        q = rng.standard_normal((n, hkv * g, d))
        kn, vn = rng.standard_normal((n, hkv, d)), rng.standard_normal((n, hkv, d))
        K = torch.from_numpy(np.concatenate([ck, kn])).permute(1, 0, 2).repeat_interleave(g, 0)
        V = torch.from_numpy(np.concatenate([cv, vn])).permute(1, 0, 2).repeat_interleave(g, 0)
        qpos = torch.arange(c, c + n)[:, None]
        kpos = torch.arange(c + n)[None, :]
        mask = (kpos <= qpos) if causal else (kpos - qpos < 3)
        out_want.append(torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q).permute(1, 0, 2), K, V, attn_mask=mask).permute(1, 0, 2).numpy())
        blocks.append((ck, cv, q, kn, vn))
    # the batch: both sequences' contexts on contiguous pages of 4
    P = 4
    pages = [math.ceil((c + n) / P) for c, n, _ in seqs]
    kc = np.zeros((sum(pages), P, hkv, d))
    vc = np.zeros_like(kc)
    bt = np.zeros((2, max(pages)), dtype=np.int64)
    base = 0
    for b, ((c, n, _), (ck, cv, *_)) in enumerate(zip(seqs, blocks)):
        bt[b, :pages[b]] = np.arange(base, base + pages[b])
        for p in range(c):
            kc[base + p // P, p % P], vc[base + p // P, p % P] = ck[p], cv[p]
        base += pages[b]
    inp = {
        "q": np.concatenate([blk[2] for blk in blocks]),
        "k_new": np.concatenate([blk[3] for blk in blocks]),
        "v_new": np.concatenate([blk[4] for blk in blocks]),
        "k_cache": kc, "v_cache": vc, "block_table": bt,
        "cu_query_lens": np.array([0, 9, 20]), "context_lens": np.array([6, 4]),
        "mm_ranges": None, "page_size": P, "num_q_heads": hkv * g, "num_kv_heads": hkv,
        "head_dim": d, "causal": True, "window_left": 0, "window_right": 3, "clamp_mm": False,
        "sm_scale": 0.0, "kv_dtype": "bf16", "k_scale": 1.0, "v_scale": 1.0,
        "seq_causal": np.array([True, False]),
    }
    out = ref.attention(inp, dtype=np.float64)
    assert np.allclose(out[:9], out_want[0], atol=1e-12)
    assert np.allclose(out[9:], out_want[1], atol=1e-12)
