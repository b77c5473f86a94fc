"""Bit-exact checks of the integer work on the GPU: live key-tile bounds, the allowed-pair
bitmap the attention kernel evaluates, the live-pair count and the fp8 decode."""
import numpy as np
import pytest
import torch

from oracle import ref
from paged_kv_prefix_gb300 import binding
from paged_kv_prefix_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev(x):
    return None if x is None else x.cuda()


def _geometry_cases():
    rng = np.random.default_rng(20)
    cases = []
    for i in range(24):
        B = int(rng.integers(1, 6))
        ctx = rng.integers(0, 300, size=B)
        qlen = rng.integers(0, 260, size=B)
        qlen[0] = max(qlen[0], 1)
        causal = bool(rng.integers(0, 2))
        wl_ = int(rng.choice([0, 1, 7, 64, 200]))
        wr = int(rng.choice([0, 1, 9, 100]))
        R = int(rng.integers(0, 5))
        mm = None
        if R:
            mm = np.zeros((B, R, 2), dtype=np.int64)
            for b in range(B):
                s = int(ctx[b] + qlen[b])
                for r in range(R):
                    a = int(rng.integers(-3, s + 5))
                    mm[b, r] = (a, a + int(rng.integers(-2, 90)))
        chunk = int(rng.choice([0, 0, 1, 16, 100])) if i >= 12 else 0  # chunked-local rows
        cases.append(wl.build_case(f"geo{i}", ctx, qlen, 2, 1, 64, int(rng.choice([5, 16, 37])),
                                   causal=causal, window_left=wl_, window_right=wr,
                                   mm_ranges=mm, clamp_mm=bool(rng.integers(0, 2)), seed=i,
                                   chunk_size=chunk, chunk_lookback=int(rng.integers(0, 3))))
    cases.append(wl.build_case("page_fixture", [0], [4096], 2, 1, 64, 16, causal=True,
                               window_left=1024, mm_ranges=np.array([[[1024, 2303], [0, 0]]]),
                               clamp_mm=True))
    return cases


@pytest.mark.parametrize("case", _geometry_cases(), ids=lambda c: c.name)
def test_tile_bounds_bit_exact(case):
    inp = case.numpy_inputs()
    dims = binding.dims_for(case)
    cu, ctx, mm = case.cu_query_lens.cuda(), case.context_lens.cuda(), _dev(case.mm_ranges)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tq, tn in [(8, 32), (16, 64), (128, 128), (7, 13), (1, 1)]:
        cap = -(-case.total_q // tq) + case.num_seqs
        out = torch.full((cap, 2), -7, dtype=torch.int32, device="cuda")
        binding.ppa_tile_bounds(dims, tq, tn, cu, ctx, mm, out, status)
        assert binding.ppa_read_status(status) == 0
        want = ref.tile_bounds(inp, tq, tn)
        got = out[: len(want)].cpu().numpy()
        assert np.array_equal(got, want), (tq, tn)


def test_tile_bounds_page_worked_example():
    case = _geometry_cases()[-1]
    dims = binding.dims_for(case)
    cap = 4096 // 8 + 1
    out = torch.zeros((cap, 2), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.ppa_tile_bounds(dims, 8, 32, case.cu_query_lens.cuda(), case.context_lens.cuda(),
                            case.mm_ranges.cuda(), out, status)
    assert out[140].tolist() == [3, 72]


@pytest.mark.parametrize("case", _geometry_cases()[:12] + _geometry_cases()[12:24:2], ids=lambda c: c.name)
def test_debug_mask_bit_exact(case):
    inp = case.numpy_inputs()
    dims = binding.dims_for(case)
    cu, ctx, mm = case.cu_query_lens.cuda(), case.context_lens.cuda(), _dev(case.mm_ranges)
    for b in range(case.num_seqs):
        c = int(inp["context_lens"][b])
        n = int(inp["cu_query_lens"][b + 1] - inp["cu_query_lens"][b])
        if n == 0:
            continue
        s = c + n
        words = -(-s // 32) + 1
        bm = torch.full((n, words), 0x5A5A5A5A, dtype=torch.int64).to(torch.int32).cuda()
        binding.ppa_debug_mask(dims, b, cu, ctx, mm, bm, n, words)
        torch.cuda.synchronize()
        bits = bm.cpu().numpy().view(np.uint32)
        got = ((bits[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(n, words * 32)
        want = ref.allowed_mask(c + np.arange(n), s, case.causal, case.window_left,
                                case.window_right, None if inp["mm_ranges"] is None
                                else inp["mm_ranges"][b], case.clamp_mm, case.chunk_size,
                                case.chunk_lookback)
        assert np.array_equal(got[:, :s].astype(bool), want)
        assert not got[:, s:].any()


@pytest.mark.parametrize("case", _geometry_cases()[:12] + _geometry_cases()[12:24:2], ids=lambda c: c.name)
def test_live_pairs_bit_exact(case):
    dims = binding.dims_for(case)
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    binding.ppa_live_pairs(dims, case.cu_query_lens.cuda(), case.context_lens.cuda(),
                           _dev(case.mm_ranges), out)
    assert int(out.item()) == ref.live_pairs(case.numpy_inputs())


def test_e4m3_decode_bit_exact():
    codes = torch.arange(256, dtype=torch.uint8, device="cuda")
    out = torch.zeros(256, dtype=torch.int16, device="cuda")
    binding.ppa_debug_e4m3_to_bf16(codes, out, 256)
    got = out.view(torch.bfloat16).float().cpu().numpy().astype(np.float64)
    table = ref.e4m3fn_table()
    nan = np.isnan(table)
    assert np.isnan(got[nan]).all()
    assert np.array_equal(got[~nan], table[~nan])
    # odd count and unaligned tail
    out2 = torch.zeros(7, dtype=torch.int16, device="cuda")
    binding.ppa_debug_e4m3_to_bf16(codes[100:107], out2, 7)
    assert np.array_equal(out2.view(torch.bfloat16).float().cpu().numpy(), table[100:107])


@pytest.mark.parametrize("case", _geometry_cases()[:12] + _geometry_cases()[12:24:2], ids=lambda c: c.name)
def test_live_kv_tokens_bit_exact(case):
    """Cached context keys that some query of the sequence may attend to, from the dense mask."""
    inp = case.numpy_inputs()
    want = 0
    for b in range(case.num_seqs):
        c = int(inp["context_lens"][b])
        n = int(inp["cu_query_lens"][b + 1] - inp["cu_query_lens"][b])
        if n == 0 or c == 0:
            continue
        m = ref.allowed_mask(c + np.arange(n), c + n, case.causal, case.window_left,
                             case.window_right, None if inp["mm_ranges"] is None
                             else inp["mm_ranges"][b], case.clamp_mm, case.chunk_size,
                             case.chunk_lookback)
        want += int(m[:, :c].any(axis=0).sum())
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    binding.ppa_live_kv_tokens(binding.dims_for(case), case.cu_query_lens.cuda(),
                               case.context_lens.cuda(), _dev(case.mm_ranges), out)
    assert int(out.item()) == want
