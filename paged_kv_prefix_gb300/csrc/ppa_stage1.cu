// Stage 1: per (sequence, query tile) the exact interval [lo, hi) of live key tiles, and the
// work list the attention kernel consumes, heaviest query tiles first. Plus the small test
// kernels that expose the mask arithmetic (allowed-pair bitmap, live-pair count, fp8 decode).
//
// Sources: "[Kernel] Skip fully masked key blocks in windowed Triton prefill" (PR #50776),
// 功能与动机 / 关键源码片段 (clamp the key loop to the keys that can survive the window);
// "[Kernel][Gemma4] Prune Triton sliding-window tiles for multimodal prefixes" (PR #53147),
// 实现拆解 2 and 关键源码片段 (compute_tile_loop_bounds: union of the base window and every
// intersecting multimodal range, clipped to seq_len - 1, converted with // TILE_SIZE).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ppa_internal.cuh"
#include "ppa_kernels.h"
#include "ppa_ptx.cuh"

namespace ppa {

namespace {

constexpr int kStage1Threads = 1024;
constexpr int kCostBins = 2048;  // work-list cost histogram; costs >= 2047 share the last bin

// Inclusive scan across the block (1024 threads); returns the exclusive prefix, sets *total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
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

}  // namespace

// One CTA of 1024 threads. Sequences are taken 1024 at a time: each thread validates one
// sequence and counts its query tiles, a block scan turns counts into tile offsets, then the
// chunk's tiles are spread over the threads (a binary search finds a tile's sequence).
template <bool kWorklist>
__global__ void __launch_bounds__(kStage1Threads) stage1_kernel(const Stage1Params p) {
  __shared__ int s_base[kStage1Threads];
  __shared__ int s_c[kStage1Threads];
  __shared__ int s_n[kStage1Threads];
  __shared__ int s_warp[32];
  __shared__ int s_hist[kWorklist ? kCostBins : 1];
  __shared__ int s_err;

  const int tid = threadIdx.x;
  if (tid == 0) s_err = 0;
  if (kWorklist) {
    for (int i = tid; i < kCostBins; i += kStage1Threads) s_hist[i] = 0;
  }
  __syncthreads();

  int carry = 0;  // query tiles of the sequences before this chunk
  for (int b0 = 0; b0 < p.num_seqs; b0 += kStage1Threads) {
    const int b = b0 + tid;
    int nt = 0, c = 0, n = 0;
    if (b < p.num_seqs) {
      const int q0 = p.cu_query_lens[b], q1 = p.cu_query_lens[b + 1];
      c = p.context_lens[b];
      n = q1 - q0;
      bool ok = (n >= 0) && (c >= 0) && (q0 >= 0) && (c <= INT_MAX - n);
      if (b == 0 && q0 != 0) ok = false;
      if (b == p.num_seqs - 1 && q1 != p.total_q) ok = false;
      if (ok && c > 0 && (c - 1) / p.page_size >= p.max_pages_per_seq) ok = false;
      if (!ok) {
        atomicExch(&s_err, 1);
        n = 0;
      }
      nt = (n + p.tq - 1) / p.tq;
    }
    int total;
    const int excl = block_exclusive_scan(nt, s_warp, &total);
    s_base[tid] = excl;  // offset within this chunk
    s_c[tid] = c;
    s_n[tid] = n;
    __syncthreads();
    const int nseq = min(kStage1Threads, p.num_seqs - b0);
    for (int i = tid; i < total; i += kStage1Threads) {
      // the last sequence of the chunk whose base is <= i
      int lo = 0, hi = nseq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_base[mid] <= i) lo = mid; else hi = mid - 1;
      }
      const int sb = lo;
      const int t = i - s_base[sb];
      const int seq = b0 + sb;
      const int cs = s_c[sb], ns = s_n[sb], s = cs + ns;
      const int q_lo = cs + t * p.tq;
      const int q_hi = cs + min(ns, (t + 1) * p.tq) - 1;
      int lo_t, hi_t;
      if (p.no_prune) {
        lo_t = 0;
        hi_t = (s + p.tn - 1) / p.tn;
      } else {
        const int32_t* ranges =
            p.mask.mm_ranges ? p.mask.mm_ranges + (size_t)seq * p.mask.max_mm_ranges * 2 : nullptr;
        int klo, khi;
        tile_interval(q_lo, q_hi, s, p.mask, ranges, klo, khi);
        lo_t = klo / p.tn;
        hi_t = khi / p.tn + 1;
      }
      const int gi = carry + i;
      if (gi < p.max_qtiles) {
        if (kWorklist) {
          p.qtiles[gi] = QTile{seq, t, lo_t, hi_t};
          atomicAdd(&s_hist[min(hi_t - lo_t, kCostBins - 1)], 1);
        } else {
          p.bounds_out[2 * gi] = lo_t;
          p.bounds_out[2 * gi + 1] = hi_t;
        }
      } else {
        atomicExch(&s_err, 1);
      }
    }
    carry += total;
    __syncthreads();
  }

  if (s_err) {
    if (tid == 0) report(p.status, PPA_ERR_INVALID);
    if (kWorklist && tid == 0) {
      p.ws->n_items = 0;
      p.ws->n_qtiles = 0;
      p.ws->next_item = 0;
      p.ws->done_ctas = 0;
    }
    return;
  }
  if (!kWorklist) return;

  // Counting sort of the query tiles by cost (live key tiles), heaviest first, so that the
  // persistent kernel's work stealing approximates longest-processing-time-first.
  const int n_qtiles = carry;
  if (tid == 0) {
    int run = 0;
    for (int bin = kCostBins - 1; bin >= 0; --bin) {
      const int h = s_hist[bin];
      s_hist[bin] = run;
      run += h;
    }
  }
  __syncthreads();
  for (int i = tid; i < n_qtiles; i += kStage1Threads) {
    const QTile qt = p.qtiles[i];
    const int pos = atomicAdd(&s_hist[min(qt.hi - qt.lo, kCostBins - 1)], 1);
    p.order[pos] = i;
  }
  if (tid == 0) {
    p.ws->n_qtiles = n_qtiles;
    p.ws->n_items = n_qtiles * p.num_kv_heads;
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
    row_interval(c + j, s, mp, ranges, kmin, kmax);
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
    row_interval(c + j, c + n, mp, ranges, kmin, kmax);
    acc += (unsigned long long)(kmax - kmin + 1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0 && acc) atomicAdd(out, acc);
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
cudaError_t launch_stage1(const Stage1Params& p, bool worklist, cudaStream_t stream) {
  if (worklist) {
    stage1_kernel<true><<<1, kStage1Threads, 0, stream>>>(p);
  } else {
    stage1_kernel<false><<<1, kStage1Threads, 0, stream>>>(p);
  }
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

cudaError_t launch_e4m3_decode(const uint8_t* codes, uint16_t* out, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int pairs = (n + 1) / 2;
  e4m3_decode_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(codes, out, n);
  return cudaGetLastError();
}

}  // namespace ppa
