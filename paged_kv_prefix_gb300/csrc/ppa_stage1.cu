// Stage 1: per (sequence, query tile) the exact interval [lo, hi) of live key tiles, and the
// work list the attention kernel consumes, heaviest query tiles first. Plus the small test
// kernels that expose the mask arithmetic (allowed-pair bitmap, live-pair count, fp8 decode).
//
// Sources: "[Kernel] Skip fully masked key blocks in windowed Triton prefill" (PR #50776),
// 功能与动机 / 关键源码片段 (clamp the key loop to the keys that can survive the window);
// "[Kernel][Gemma4] Prune Triton sliding-window tiles for multimodal prefixes" (PR #53147),
// 实现拆解 2 and 关键源码片段 (compute_tile_loop_bounds: union of the base window and every
// intersecting multimodal range, clipped to seq_len - 1, converted with // TILE_SIZE).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ppa_internal.cuh"
#include "ppa_kernels.h"
#include "ppa_ptx.cuh"

namespace ppa {

namespace {

constexpr int kStage1Threads = 1024;

}  // namespace

// Validates sequence b and returns its query length (0 if invalid, with *bad set).
__device__ __forceinline__ int seq_query_len(const Stage1Params& p, int b, int* c_out, bool* bad) {
  const int q0 = p.cu_query_lens[b], q1 = p.cu_query_lens[b + 1];
  const int c = p.context_lens[b];
  const int n = q1 - q0;
  bool ok = (n >= 0) && (c >= 0) && (q0 >= 0) && (c <= INT_MAX - n);
  if (b == 0 && q0 != 0) ok = false;
  if (b == p.num_seqs - 1 && q1 != p.total_q) ok = false;
  // the block-table row covers every cache position read: c of them, or c + n when the new
  // tokens' K/V are read from the cache too
  const int span = p.kv_in_cache ? c + n : c;
  if (ok && span > 0 && (span - 1) / p.page_size >= p.max_pages_per_seq) ok = false;
  *c_out = c;
  if (!ok) *bad = true;
  return ok ? n : 0;
}

// Live keys [klo, khi] of query tile t of a sequence (context c, n queries); every key with
// no_prune (testing) unless `pruned` asks for the live ones regardless.
__device__ __forceinline__ void qtile_keys(const Stage1Params& p, int seq, int c, int n, int t,
                                           int* klo, int* khi, bool pruned = false) {
  const int s = c + n;
  if (p.no_prune && !pruned) {
    *klo = 0;
    *khi = s - 1;
    return;
  }
  const int q_lo = c + t * p.tq;
  const int q_hi = c + min(n, (t + 1) * p.tq) - 1;
  const int32_t* ranges =
      p.mask.mm_ranges ? p.mask.mm_ranges + (size_t)seq * p.mask.max_mm_ranges * 2 : nullptr;
  tile_interval(q_lo, q_hi, s, seq_mask(p.mask, seq), ranges, *klo, *khi);
}

// Live key tiles of query tile t of a sequence, on the grid aligned to multiples of tn.
__device__ __forceinline__ void qtile_bounds(const Stage1Params& p, int seq, int c, int n, int t,
                                             int* lo, int* hi) {
  int klo, khi;
  qtile_keys(p, seq, c, n, t, &klo, &khi);
  *lo = klo / p.tn;
  *hi = khi / p.tn + 1;
}

// Key tiles [lo, hi) covering keys [klo, khi] on the grid shifted by koff.
__device__ __forceinline__ void grid_tiles(int klo, int khi, int koff, int tn, int* lo, int* hi) {
  *lo = (klo + koff) / tn;
  *hi = (khi + koff) / tn + 1;
}

// Last index r in [0, count) with base[r] <= x (base non-decreasing, base[0] <= x).
__device__ __forceinline__ int last_le(const int32_t* base, int count, int x) {
  int lo = 0, hi = count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bounds only (testing): {lo, hi} of every query tile, in (sequence, tile) order.
__global__ void __launch_bounds__(kStage1Threads) tile_bounds_kernel(const Stage1Params p) {
  __shared__ int s_base[kStage1Threads];
  __shared__ int s_c[kStage1Threads];
  __shared__ int s_n[kStage1Threads];
  __shared__ int s_warp[32];
  __shared__ int s_err;
  const int tid = threadIdx.x;
  if (tid == 0) s_err = 0;
  __syncthreads();
  int carry = 0;
  for (int b0 = 0; b0 < p.num_seqs; b0 += kStage1Threads) {
    const int b = b0 + tid;
    int nt = 0, c = 0, n = 0;
    if (b < p.num_seqs) {
      bool bad = false;
      n = seq_query_len(p, b, &c, &bad);
      if (bad) atomicExch(&s_err, 1);
      nt = (n + p.tq - 1) / p.tq;
    }
    int total;
    const int excl = block_exclusive_scan(nt, s_warp, &total);
    s_base[tid] = excl;
    s_c[tid] = c;
    s_n[tid] = n;
    __syncthreads();
    const int nseq = min(kStage1Threads, p.num_seqs - b0);
    for (int i = tid; i < total; i += kStage1Threads) {
      const int sb = last_le(s_base, nseq, i);
      int lo, hi;
      qtile_bounds(p, b0 + sb, s_c[sb], s_n[sb], i - s_base[sb], &lo, &hi);
      const int gi = carry + i;
      if (gi < p.max_qtiles) {
        p.bounds_out[2 * gi] = lo;
        p.bounds_out[2 * gi + 1] = hi;
      } else {
        atomicExch(&s_err, 1);
      }
    }
    carry += total;
    __syncthreads();
  }
  if (s_err && tid == 0) report(p.status, PPA_ERR_INVALID);
}

// The plan (one CTA of 1024 threads):
//   1. validate every sequence and count its units (nq query tiles each); scan -> unit bases;
//   2. every unit's per-tile live key-tile intervals and union cost; per-sequence cost;
//   3. rank sequences by cost, heaviest first (up to kMaxRankedSeqs; beyond that, in order);
//   4. lay the work list out sequence by sequence in that rank order, KV head by KV head,
//      each sequence's units last-to-first. The query tiles of one (sequence, KV head) are
//      thus taken together by neighbouring CTAs and stream the same K/V through L2, while
//      the heaviest sequences start first.
constexpr int kMaxRankedSeqs = 4096;

__global__ void __launch_bounds__(kStage1Threads) plan_kernel(const Stage1Params p) {
  __shared__ int s_warp[32];
  __shared__ int s_err;
  const int tid = threadIdx.x;
  const int B = p.num_seqs;
  if (tid == 0) s_err = 0;
  __syncthreads();

  // 1. units per sequence. With split-KV, a sequence of one query tile whose live key
  //    interval spans more than split_tiles key tiles becomes one unit per segment of
  //    split_tiles key tiles, each with its own partial-result slot.
  int carry = 0, split_carry = 0;
  for (int b0 = 0; b0 < B; b0 += kStage1Threads) {
    const int b = b0 + tid;
    int nu = 0, nseg = 0;
    if (b < B) {
      bool bad = false;
      int c;
      const int n = seq_query_len(p, b, &c, &bad);
      if (bad) atomicExch(&s_err, 1);
      const int nt = (n + p.tq - 1) / p.tq;
      nu = (nt + p.nq - 1) / p.nq;
      if (p.split_tiles > 0 && nt == 1 && !bad) {  // the tiles of step 2's single-tile unit
        int klo, khi, plo, phi, lo, hi;
        qtile_keys(p, b, c, n, 0, &klo, &khi);
        qtile_keys(p, b, c, n, 0, &plo, &phi, true);
        grid_tiles(klo, khi, key_grid_offset(plo, p.tn), p.tn, &lo, &hi);
        const int segs = (hi - lo + p.split_tiles - 1) / p.split_tiles;
        if (segs >= 2) nu = nseg = segs;
      }
      p.seq_cost[b] = 0;
    }
    int total, stotal;
    const int excl = block_exclusive_scan(nu, s_warp, &total);
    if (b < B) p.seq_unit_base[b] = carry + excl;
    carry += total;
    if (p.seq_split_base != nullptr) {
      const int sexcl = block_exclusive_scan(nseg, s_warp, &stotal);
      if (b < B) p.seq_split_base[b] = split_carry + sexcl;
      split_carry += stotal;
    }
  }
  const int n_units = carry;
  if (tid == 0) {
    p.seq_unit_base[B] = n_units;
    if (p.seq_split_base != nullptr) p.seq_split_base[B] = split_carry;
  }
  __syncthreads();
  if (s_err || n_units > p.max_units || (long long)n_units * p.num_kv_heads > INT_MAX) {
    if (p.seq_split_base != nullptr)  // no segment of a rejected batch is merged
      for (int b = tid; b <= B; b += kStage1Threads) p.seq_split_base[b] = 0;
    if (tid == 0) {
      report(p.status, PPA_ERR_INVALID);
      p.ws->n_items = 0;
      p.ws->n_units = 0;
      p.ws->next_item = 0;
      p.ws->done_ctas = 0;
    }
    return;
  }

  // 2. units
  for (int u = tid; u < n_units; u += kStage1Threads) {
    const int b = last_le(p.seq_unit_base, B, u);
    const int c = p.context_lens[b];
    const int n = p.cu_query_lens[b + 1] - p.cu_query_lens[b];
    const int nt = (n + p.tq - 1) / p.tq;
    const int lu = u - p.seq_unit_base[b];
    const bool split =
        p.seq_split_base != nullptr && p.seq_split_base[b + 1] > p.seq_split_base[b];
    const int t0 = split ? 0 : lu * p.nq;
    const int cnt = split ? 1 : min(p.nq, nt - t0);
    Unit un{b, t0, cnt, 0, 0, 0, 0, 0, -1, 0};
    // The grid is the pruned unit's, also without pruning (testing): the tiles of the pruned
    // run are then a subset of the unpruned run's, whose extra tiles are fully masked, and
    // the two outputs agree bit for bit. Its first tile may then hold keys below 0, which
    // the attention kernels read as zeros and mask.
    int klo0, khi0, klo1 = 0, khi1 = 0, plo, phi;
    qtile_keys(p, b, c, n, t0, &klo0, &khi0);
    qtile_keys(p, b, c, n, t0, &plo, &phi, true);
    if (cnt > 1) {
      int plo1, phi1;
      qtile_keys(p, b, c, n, t0 + 1, &klo1, &khi1);
      qtile_keys(p, b, c, n, t0 + 1, &plo1, &phi1, true);
      plo = min(plo, plo1);
    }
    un.koff = key_grid_offset(plo, p.tn);
    grid_tiles(klo0, khi0, un.koff, p.tn, &un.lo0, &un.hi0);
    if (split) {  // segment lu of the tile's key tiles
      un.lo0 += lu * p.split_tiles;
      un.hi0 = min(un.hi0, un.lo0 + p.split_tiles);
      un.part = p.seq_split_base[b] + lu;
    }
    int lo = un.lo0, hi = un.hi0;
    if (cnt > 1) {
      grid_tiles(klo1, khi1, un.koff, p.tn, &un.lo1, &un.hi1);
      lo = min(lo, un.lo1);
      hi = max(hi, un.hi1);
    }
    un.cost = hi - lo;
    p.units[u] = un;
    atomicAdd(&p.seq_cost[b], un.cost);
  }
  __syncthreads();

  // 3. sequences heaviest first (ties by index)
  for (int b = tid; b < B; b += kStage1Threads) {
    int rank = b;
    if (B <= kMaxRankedSeqs) {
      const int cb = p.seq_cost[b];
      rank = 0;
      for (int b2 = 0; b2 < B; ++b2) {
        const int c2 = p.seq_cost[b2];
        rank += (c2 > cb) || (c2 == cb && b2 < b);
      }
    }
    p.seq_order[rank] = b;
  }
  __syncthreads();

  // 4. item bases in rank order, then the items
  carry = 0;
  for (int r0 = 0; r0 < B; r0 += kStage1Threads) {
    const int r = r0 + tid;
    int cnt = 0;
    if (r < B) {
      const int b = p.seq_order[r];
      cnt = (p.seq_unit_base[b + 1] - p.seq_unit_base[b]) * p.num_kv_heads;
    }
    int total;
    const int excl = block_exclusive_scan(cnt, s_warp, &total);
    if (r < B) p.seq_item_base[r] = carry + excl;
    carry += total;
  }
  const int n_items = carry;
  if (tid == 0) p.seq_item_base[B] = n_items;
  __syncthreads();
  for (int i = tid; i < n_items; i += kStage1Threads) {
    const int r = last_le(p.seq_item_base, B, i);
    const int b = p.seq_order[r];
    const int ub = p.seq_unit_base[b];
    const int nu = p.seq_unit_base[b + 1] - ub;
    const int li = i - p.seq_item_base[r];
    const int g = li / nu;
    const int lu = nu - 1 - (li - g * nu);
    p.items[i] = (ub + lu) * p.num_kv_heads + g;
  }
  if (tid == 0) {
    p.ws->n_units = n_units;
    p.ws->n_items = n_items;
    p.ws->next_item = 0;
    p.ws->done_ctas = 0;
  }
}

// ---------------------------------------------------------------------------------------
// Test kernels
// ---------------------------------------------------------------------------------------
__global__ void debug_mask_kernel(const MaskParams mp, int seq, const int32_t* cu,
                                  const int32_t* ctx, uint32_t* bitmap, int max_rows,
                                  int words_per_row) {
  const int c = ctx[seq];
  const int n = cu[seq + 1] - cu[seq];
  const int s = c + n;
  const int rows = min(n, max_rows);
  const int32_t* ranges = mp.mm_ranges ? mp.mm_ranges + (size_t)seq * mp.max_mm_ranges * 2 : nullptr;
  for (int j = blockIdx.x; j < rows; j += gridDim.x) {
    int kmin, kmax;
    row_interval(c + j, s, seq_mask(mp, seq), ranges, kmin, kmax);
    for (int w = threadIdx.x; w < words_per_row; w += blockDim.x) {
      const int k0 = w * 32;
      uint32_t bits = 0;
      for (int i = 0; i < 32; ++i) {
        const int k = k0 + i;
        if (k < s && k >= kmin && k <= kmax) bits |= 1u << i;
      }
      bitmap[(size_t)j * words_per_row + w] = bits;
    }
  }
}

__global__ void live_pairs_kernel(const MaskParams mp, int num_seqs, int total_q,
                                  const int32_t* cu, const int32_t* ctx,
                                  unsigned long long* out) {
  unsigned long long acc = 0;
  for (int tok = blockIdx.x * blockDim.x + threadIdx.x; tok < total_q;
       tok += gridDim.x * blockDim.x) {
    int lo = 0, hi = num_seqs - 1;  // last sequence with cu[b] <= tok
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int c = ctx[b];
    const int n = cu[b + 1] - cu[b];
    const int j = tok - cu[b];
    if (j < 0 || j >= n) continue;
    const int32_t* ranges = mp.mm_ranges ? mp.mm_ranges + (size_t)b * mp.max_mm_ranges * 2 : nullptr;
    int kmin, kmax;
    row_interval(c + j, c + n, seq_mask(mp, b), ranges, kmin, kmax);
    acc += (unsigned long long)(kmax - kmin + 1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc) atomicAdd(out, acc);
}

// One thread per query token: the allowed key interval [kmin, kmax] of its row (row_interval),
// for the attention kernels to load instead of scanning the multimodal ranges once per unit.
// Sequence lookup by binary search over cu_query_lens, as in live_pairs_kernel; tokens of a
// sequence whose lengths are invalid get some interval, but the plan then schedules no work.
__global__ void row_bounds_kernel(const MaskParams mp, int num_seqs, int total_q,
                                  const int32_t* cu, const int32_t* ctx, int32_t* out) {
  for (int tok = blockIdx.x * blockDim.x + threadIdx.x; tok < total_q;
       tok += gridDim.x * blockDim.x) {
    int lo = 0, hi = num_seqs - 1;  // last sequence with cu[b] <= tok
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int c = ctx[b];
    const int n = cu[b + 1] - cu[b];
    const int j = tok - cu[b];
    const int32_t* ranges = mp.mm_ranges ? mp.mm_ranges + (size_t)b * mp.max_mm_ranges * 2 : nullptr;
    int kmin = 0, kmax = 0;
    if (j >= 0 && j < n) row_interval(c + j, c + n, seq_mask(mp, b), ranges, kmin, kmax);
    out[2 * (size_t)tok] = kmin;
    out[2 * (size_t)tok + 1] = kmax;
  }
}

// One CTA per sequence: the cached context keys that at least one of its queries may attend
// to. The union of the rows' allowed intervals is itself an interval (each row's contains the
// row's own position and the positions are consecutive), so it is [min kmin, max kmax].
__global__ void live_kv_tokens_kernel(const MaskParams mp, const int32_t* cu, const int32_t* ctx,
                                      unsigned long long* out) {
  __shared__ int s_lo[32], s_hi[32];
  const int b = blockIdx.x;
  const int c = ctx[b];
  const int n = cu[b + 1] - cu[b];
  const int32_t* ranges = mp.mm_ranges ? mp.mm_ranges + (size_t)b * mp.max_mm_ranges * 2 : nullptr;
  int lo = INT_MAX, hi = INT_MIN;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    int kmin, kmax;
    row_interval(c + j, c + n, seq_mask(mp, b), ranges, kmin, kmax);
    lo = min(lo, kmin);
    hi = max(hi, kmax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_down_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_down_sync(0xffffffffu, hi, o));
  }
  const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if ((threadIdx.x & 31) == 0) { s_lo[warp] = lo; s_hi[warp] = hi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; ++w) { lo = min(lo, s_lo[w]); hi = max(hi, s_hi[w]); }
    const int top = min(hi, c - 1);
    if (n > 0 && top >= lo) atomicAdd(out, (unsigned long long)(top - lo + 1));
  }
}

__global__ void e4m3_decode_kernel(const uint8_t* codes, uint16_t* out, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const uint16_t pair = (uint16_t)codes[i] | (uint16_t)((i + 1 < n ? codes[i + 1] : 0) << 8);
  const uint32_t b2 = e4m3x2_to_bf16x2(pair);
  out[i] = (uint16_t)(b2 & 0xFFFFu);
  if (i + 1 < n) out[i + 1] = (uint16_t)(b2 >> 16);
}

// ---------------------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------------------
cudaError_t launch_plan(const Stage1Params& p, cudaStream_t stream) {
  plan_kernel<<<1, kStage1Threads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tile_bounds(const Stage1Params& p, cudaStream_t stream) {
  tile_bounds_kernel<<<1, kStage1Threads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_debug_mask(const MaskParams& mp, int seq, const int32_t* cu, const int32_t* ctx,
                              uint32_t* bitmap, int max_rows, int words_per_row,
                              cudaStream_t stream) {
  const int grid = max(1, min(max_rows, 4096));
  debug_mask_kernel<<<grid, 128, 0, stream>>>(mp, seq, cu, ctx, bitmap, max_rows, words_per_row);
  return cudaGetLastError();
}

cudaError_t launch_live_pairs(const MaskParams& mp, int num_seqs, int total_q, const int32_t* cu,
                              const int32_t* ctx, unsigned long long* out, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  if (total_q == 0 || num_seqs == 0) return cudaSuccess;
  const int grid = min(1184, (total_q + 255) / 256);
  live_pairs_kernel<<<grid, 256, 0, stream>>>(mp, num_seqs, total_q, cu, ctx, out);
  return cudaGetLastError();
}

cudaError_t launch_live_kv_tokens(const MaskParams& mp, int num_seqs, const int32_t* cu,
                                  const int32_t* ctx, unsigned long long* out,
                                  cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  if (num_seqs == 0) return cudaSuccess;
  live_kv_tokens_kernel<<<num_seqs, 256, 0, stream>>>(mp, cu, ctx, out);
  return cudaGetLastError();
}

cudaError_t launch_row_bounds(const MaskParams& mp, int num_seqs, int total_q, const int32_t* cu,
                              const int32_t* ctx, int32_t* out, cudaStream_t stream) {
  if (num_seqs == 0 || total_q == 0) return cudaSuccess;
  const int blocks = (total_q + 255) / 256;
  row_bounds_kernel<<<blocks < 4096 ? blocks : 4096, 256, 0, stream>>>(mp, num_seqs, total_q, cu,
                                                                       ctx, out);
  return cudaGetLastError();
}

// Split-KV merge: one CTA per (sequence, KV head), threads over the head dimension. For each
// of the tile's rows, the segments' rows O_s (already divided by their own row sums) weigh in
// with 2^(lse_s - max lse): softmax over the union of the segments' keys, exactly.
// A plan that rejected the batch (bad lengths found on the device) leaves no items and no
// partials: the merge then writes nothing. Rows are also bounded by one query tile and by
// total_q, so lengths that changed after the plan cannot send a store outside `out`.
__global__ void split_merge_kernel(const MergeParams p) {
  if (p.ws->n_items == 0) return;
  const int b = blockIdx.x / p.num_kv_heads;
  const int g = blockIdx.x - b * p.num_kv_heads;
  const int s0 = p.seq_split_base[b], ns = p.seq_split_base[b + 1] - s0;
  if (ns <= 0) return;
  const int q0 = p.cu_query_lens[b];
  const int n = p.cu_query_lens[b + 1] - q0;
  if (q0 < 0 || n <= 0 || n > p.total_q - q0) return;
  const int rows = min(n * p.group, kRowsPerTile);
  for (int r = 0; r < rows; ++r) {
    float mx = -__int_as_float(0x7f800000);
    for (int s = 0; s < ns; ++s)
      mx = fmaxf(mx, p.part_lse[((size_t)(s0 + s) * p.num_kv_heads + g) * kRowsPerTile + r]);
    const int tok = r / p.group, hh = r - tok * p.group;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                          ((size_t)(q0 + tok) * p.num_q_heads + g * p.group + hh) * p.head_dim;
    for (int col = threadIdx.x; col < p.head_dim; col += blockDim.x) {
      float num = 0.f, den = 0.f;
      for (int s = 0; s < ns; ++s) {
        const size_t slot = (size_t)(s0 + s) * p.num_kv_heads + g;
        const float lse = p.part_lse[slot * kRowsPerTile + r];
        if (lse == -__int_as_float(0x7f800000)) continue;  // no keys of the row in segment s
        const float w = exp2f(lse - mx);
        den += w;
        num += w * p.part_o[(slot * kRowsPerTile + r) * p.head_dim + col];
      }
      orow[col] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
    }
  }
}

cudaError_t launch_split_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  split_merge_kernel<<<p.num_seqs * p.num_kv_heads, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_decode(const uint8_t* codes, uint16_t* out, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int pairs = (n + 1) / 2;
  e4m3_decode_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(codes, out, n);
  return cudaGetLastError();
}

}  // namespace ppa
