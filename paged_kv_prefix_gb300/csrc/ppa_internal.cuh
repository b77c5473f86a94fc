// Shared device-side definitions: launch parameters, the workspace layout, status
// reporting and the mask arithmetic that both the tile-bounds stage and the attention
// kernel evaluate (so the two can never disagree).
#pragma once

#include <cstdint>

#include "../../include/ppa.h"

namespace ppa {

constexpr int kRowsPerTile = 128;  // rows of one query tile (tokens x heads of a group)
constexpr unsigned long long kWaitNs = 2000000000ull;  // default limit of a device wait: 2 s

// Mask parameters of one call.
struct MaskParams {
  int causal;
  int window_left;   // <= 0: off
  int window_right;  // <= 0: off (ignored when causal)
  int clamp_mm;
  int max_mm_ranges;
  const int32_t* mm_ranges;  // [B][R][2] or nullptr
  int chunk_size;            // > 0: chunked-local base left edge (instead of window_left)
  int chunk_lookback;
  const int32_t* seq_causal;  // [B] per-sequence causal flags, or nullptr (use `causal`)
};

// The mask of sequence b: `causal` taken from the per-sequence flags when given.
__device__ __forceinline__ MaskParams seq_mask(const MaskParams& mp, int b) {
  MaskParams m = mp;
  if (mp.seq_causal != nullptr) m.causal = mp.seq_causal[b] != 0 ? 1 : 0;
  return m;
}

// Lowest key of the base mask for query position q: the start of the chunk chunk_lookback
// chunks before q's own (chunked-local attention), else the left window's edge, else 0. The
// result is non-decreasing in q, so over a run of rows the first row's value bounds them all.
__device__ __forceinline__ int base_first_key(int q, const MaskParams& mp) {
  if (mp.chunk_size > 0) return (q / mp.chunk_size - mp.chunk_lookback) * mp.chunk_size;
  return mp.window_left > 0 ? q - mp.window_left + 1 : 0;
}

// Workspace header; followed by per-sequence arrays, the unit table and the work list.
struct WsHeader {
  int32_t next_item;   // work-stealing counter of the persistent kernel
  int32_t n_items;     // number of (unit, kv head) items, 0 on a device-side error
  int32_t n_units;
  int32_t done_ctas;   // CTAs of the running attention launch that have finished
  int32_t pad[12];
};

// One unit of work: nt (1 or 2) consecutive query tiles t0, t0+1 of sequence `seq` that
// share one K/V stream, with each tile's live key tiles [lo_i, hi_i). `cost` is the number of
// key tiles in the union. The unit's key tiles lie on a grid shifted by `koff` keys: tile kt
// holds keys [kt * TN - koff, kt * TN - koff + TN). The plan starts the grid at the 16-key
// boundary at or below the unit's first live key, so a short window needs no more tiles than
// its span (a 16-key chunk still lies in one page whenever the page size is a multiple of 16).
struct Unit {
  int32_t seq, t0, nt, lo0, hi0, lo1, hi1, cost;
  int32_t part;  // split-KV segment: its partial-result slot (x Hkv + kv head); -1: not split
  int32_t koff;  // key grid offset, 0 .. TN-16 in steps of 16
};

// Offset of the key-tile grid whose first tile starts at the 16-key boundary at or below kmin.
__host__ __device__ __forceinline__ int key_grid_offset(int kmin, int tn) {
  const int kb = kmin & ~15;
  return (tn - kb % tn) % tn;
}

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Allowed keys of one query position q form the single interval [kmin, kmax], which always
// contains q: the base window contains q, every multimodal range that contains q contains q,
// and the union of intervals that share a point is an interval.
//   base: [WL > 0 ? q - WL + 1 : 0,  causal ? q : (WR > 0 ? q + WR - 1 : s - 1)]
//   mm:   for each valid range [a, e'] containing q: [clamp && WL > 0 ? max(a, q - WL + 1) : a, e']
// ("[Kernel][Gemma4] Prune Triton sliding-window tiles for multimodal prefixes", 实现拆解 2:
// the multimodal mask is OR-ed onto the base mask, so bounds take the union.)
__device__ __forceinline__ void row_interval(int q, int s, const MaskParams& mp,
                                             const int32_t* ranges /* this sequence, [R][2] */,
                                             int& kmin, int& kmax) {
  int lo = base_first_key(q, mp);
  int hi;
  if (mp.causal) {
    hi = q;
  } else if (mp.window_right > 0) {
    hi = (mp.window_right - 1 >= s - 1 - q) ? s - 1 : q + mp.window_right - 1;
  } else {
    hi = s - 1;
  }
  if (ranges != nullptr) {
    const bool clamp = mp.clamp_mm && mp.window_left > 0;
    for (int r = 0; r < mp.max_mm_ranges; ++r) {
      const int a = ranges[2 * r];
      const int e = ranges[2 * r + 1];
      if (!(a < e)) continue;
      const int e2 = e < s - 1 ? e : s - 1;
      if (a <= q && q <= e2) {
        const int l = clamp ? max(a, q - mp.window_left + 1) : a;
        lo = min(lo, l);
        hi = max(hi, e2);
      }
    }
  }
  kmin = max(lo, 0);
  kmax = hi;
}

// Union of the row intervals of query positions q_lo .. q_hi (one query tile), in closed
// form. A range contributes iff it shares a row with the tile; its lowest key over those rows
// is max(a, q_lo - WL + 1) when clamped (the window edge of the tile's first row), else a.
// The base lower edge also uses the first row, q_lo (the page computes it from the last row,
// which is not a bound for the earlier rows of the block).
__device__ __forceinline__ void tile_interval(int q_lo, int q_hi, int s, const MaskParams& mp,
                                              const int32_t* ranges, int& klo, int& khi) {
  int lo = base_first_key(q_lo, mp);
  int hi;
  if (mp.causal) {
    hi = q_hi;
  } else if (mp.window_right > 0) {
    hi = (mp.window_right - 1 >= s - 1 - q_hi) ? s - 1 : q_hi + mp.window_right - 1;
  } else {
    hi = s - 1;
  }
  if (ranges != nullptr) {
    const bool clamp = mp.clamp_mm && mp.window_left > 0;
    for (int r = 0; r < mp.max_mm_ranges; ++r) {
      const int a = ranges[2 * r];
      const int e = ranges[2 * r + 1];
      if (!(a < e)) continue;
      const int e2 = e < s - 1 ? e : s - 1;
      if (a <= q_hi && e2 >= q_lo) {
        const int l = clamp ? max(a, q_lo - mp.window_left + 1) : a;
        lo = min(lo, l);
        hi = max(hi, e2);
      }
    }
  }
  klo = max(lo, 0);
  khi = hi;
}

// Scan across a block of 1024 threads (32 warps): returns the exclusive prefix of v and sets
// *total to the block's sum. warp_sums: 32 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

// Tile shape for a head group of G query heads: tq tokens x G heads <= 128 rows.
__host__ __device__ constexpr int tokens_per_qtile(int group) { return kRowsPerTile / group; }
__host__ __device__ constexpr int keys_per_tile(int) { return 128; }

}  // namespace ppa
