// fp8 caches: dequantise the live cache key tiles of a batch into bf16 scratch, once per call.
//
// Without this pass every unit of work (two query tiles of one sequence and one KV head)
// widens each e4m3 key tile it visits, so a tile shared by the many units of one long
// sequence is converted once per unit, by producer warps that compete with the softmax for
// issue slots. Here each live tile is converted once, by a memory-bound kernel, and the
// attention kernel then runs its bf16 path on the scratch.
//
// Scratch layout: "pages" of TN (=128) tokens, each holding the cache positions
// [t * TN, t * TN + TN) of one live key tile t of one sequence b, each position [Hkv][D] bf16
// like the cache. Only the live tiles (those some unit visits) get a page: they are packed in
// sequence order, and a block table [num_seqs][tiles_per_seq] gives each live tile its page,
// so the attention kernel reads the scratch as a paged cache with page size TN whose key tiles
// never straddle a page (the same live-tile intervals drive both, so it reads no other entry).
// Rows past a sequence's cache positions (its context, or its context and new tokens when
// those were appended first) are not written and not read: the attention kernel takes those
// keys from the new-token tensors, or zero-fills positions past the sequence.
//
// Each value is bf16(decode(code) * scale), the fp32 product rounded once, as in the
// in-kernel path when it applies the scales itself.
#include <cuda_runtime.h>

#include <cstdint>

#include "ppa_internal.cuh"
#include "ppa_kernels.h"
#include "ppa_ptx.cuh"

namespace ppa {
namespace {

// Positions of sequence b that are read from the cache: its context, and its new tokens too
// when they were appended to the cache before the call.
__device__ __forceinline__ int cache_positions(const Fp8DequantParams& p, int b) {
  const int c = p.context_lens[b];
  return p.kv_in_cache ? c + (p.cu_query_lens[b + 1] - p.cu_query_lens[b]) : c;
}

// One thread per unit: marks the cache tiles (TN-aligned, like the staging pages) that the
// unit's key tiles overlap, up to ceil(cs / TN) (cs: the sequence's cache positions), a word
// of 32 tiles per atomic. The unit's tiles lie on its shifted grid: keys [lo * TN - koff,
// hi * TN - koff).
__global__ void fp8_mark_kernel(Fp8DequantParams p) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= p.max_units || u >= p.ws->n_units) return;
  const Unit un = p.units[u];
  const int k_first = (un.nt > 1 ? min(un.lo0, un.lo1) : un.lo0) * p.tn - un.koff;
  const int k_end = (un.nt > 1 ? max(un.hi0, un.hi1) : un.hi0) * p.tn - un.koff;
  const int lo = k_first / p.tn;
  int hi = (k_end + p.tn - 1) / p.tn;
  const int cs = cache_positions(p, un.seq);
  hi = min(hi, (cs + p.tn - 1) / p.tn);
  hi = min(hi, p.tiles_per_seq);
  uint32_t* bits = p.live_bits + (size_t)un.seq * p.words_per_seq;
  for (int t = max(lo, 0); t < hi;) {
    const int w = t >> 5, b0 = t & 31;
    const int b1 = min(32, b0 + (hi - t));  // bits [b0, b1) of word w
    const uint32_t m = (b1 - b0 == 32) ? 0xFFFFFFFFu : (((1u << (b1 - b0)) - 1u) << b0);
    atomicOr(bits + w, m);
    t += b1 - b0;
  }
}

// One CTA of 1024 threads: the staging page of every live tile, in sequence order (a scan of
// the sequences' live-tile counts, then each sequence numbers its live tiles). If they need
// more pages than the staging holds, the batch is rejected: PPA_ERR_INVALID, and the plan's
// item count is cleared, so neither the dequantisation nor the attention does any work.
constexpr int kSlotThreads = 1024;

__global__ void __launch_bounds__(kSlotThreads) fp8_slots_kernel(Fp8DequantParams p) {
  __shared__ int s_warp[32];
  int carry = 0;
  for (int b0 = 0; b0 < p.num_seqs; b0 += kSlotThreads) {
    const int b = b0 + threadIdx.x;
    const uint32_t* bits = p.live_bits + (size_t)b * p.words_per_seq;
    int cnt = 0;
    if (b < p.num_seqs)
      for (int w = 0; w < p.words_per_seq; ++w) cnt += __popc(bits[w]);
    int total;
    const int excl = block_exclusive_scan(cnt, s_warp, &total);
    if (b < p.num_seqs) {
      int page = carry + excl;
      int32_t* row = p.table + (size_t)b * p.tiles_per_seq;
      for (int w = 0; w < p.words_per_seq; ++w) {
        for (uint32_t m = bits[w]; m != 0u; m &= m - 1u) row[32 * w + __ffs(m) - 1] = page++;
      }
    }
    carry += total;
  }
  if (carry > p.capacity && threadIdx.x == 0) {
    report(p.status, PPA_ERR_INVALID);
    p.ws->n_items = 0;
  }
}

// One CTA per (sequence, key tile) and tensor (blockIdx.y: 0 = K, 1 = V): if the tile is live,
// the bf16 rows of its cache positions into its staging page.
constexpr int kDequantThreads = 256;

__global__ void __launch_bounds__(kDequantThreads) fp8_dequant_kernel(Fp8DequantParams p) {
  if (p.ws->n_items == 0) return;  // rejected by the slot pass (or an empty plan)
  const int b = blockIdx.x / p.tiles_per_seq;
  const int t = blockIdx.x - b * p.tiles_per_seq;
  if (!((p.live_bits[(size_t)b * p.words_per_seq + (t >> 5)] >> (t & 31)) & 1u)) return;
  const int page = p.table[blockIdx.x];  // < capacity: the slot pass checked the count
  const bool is_v = blockIdx.y != 0;
  const uint8_t* src = static_cast<const uint8_t*>(is_v ? p.v_cache : p.k_cache);
  uint8_t* dst = static_cast<uint8_t*>(is_v ? p.v_out : p.k_out);
  const float scale = *(is_v ? p.v_scale : p.k_scale);
  const int rows = min(p.tn, cache_positions(p, b) - t * p.tn);  // >= 1: the tile is live
  const int row_bytes = p.row_codes;         // Hkv * D codes per position
  const int pieces_per_row = row_bytes / 16;
  const int pieces = rows * pieces_per_row;
  const int32_t* bt = p.block_table + (size_t)b * p.max_pages_per_seq;
  // Four 16-byte pieces in flight per thread before any is widened.
  constexpr int kUnroll = 4;
  for (int base = threadIdx.x; base < pieces; base += kDequantThreads * kUnroll) {
    uint4 codes[kUnroll];
    int outp[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int i = base + k * kDequantThreads;
      outp[k] = -1;
      codes[k] = make_uint4(0u, 0u, 0u, 0u);
      if (i < pieces) {
        const int r = i / pieces_per_row, pc = i - r * pieces_per_row;
        const int pos = t * p.tn + r;
        const int lp = pos / p.page_size;
        const int pg = bt[lp];
        outp[k] = i;
        if (pg >= 0 && pg < p.num_pages) {
          const size_t off =
              ((size_t)pg * p.page_size + (pos - lp * p.page_size)) * row_bytes + pc * 16;
          codes[k] = ld_global_nc_v4(src + off);
        } else {
          report(p.status, PPA_ERR_BAD_PAGE);  // the row reads as zero, as in the attention
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      if (outp[k] < 0) continue;
      const uint32_t cw[4] = {codes[k].x, codes[k].y, codes[k].z, codes[k].w};
      uint32_t v[8];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        v[2 * q4] = e4m3x2_to_bf16x2_scaled(static_cast<uint16_t>(cw[q4] & 0xFFFFu), scale);
        v[2 * q4 + 1] = e4m3x2_to_bf16x2_scaled(static_cast<uint16_t>(cw[q4] >> 16), scale);
      }
      const int i = outp[k];
      const int r = i / pieces_per_row, pc = i - r * pieces_per_row;
      uint4* o = reinterpret_cast<uint4*>(
          dst + ((size_t)page * p.tn + r) * (size_t)row_bytes * 2 + (size_t)pc * 32);
      o[0] = make_uint4(v[0], v[1], v[2], v[3]);
      o[1] = make_uint4(v[4], v[5], v[6], v[7]);
    }
  }
}

}  // namespace

cudaError_t launch_fp8_dequant(const Fp8DequantParams& p, cudaStream_t stream) {
  const size_t bits_bytes = (size_t)p.num_seqs * p.words_per_seq * sizeof(uint32_t);
  cudaError_t e = cudaMemsetAsync(p.live_bits, 0, bits_bytes, stream);
  if (e != cudaSuccess) return e;
  if (p.max_units > 0) {
    fp8_mark_kernel<<<(p.max_units + 255) / 256, 256, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  fp8_slots_kernel<<<1, kSlotThreads, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.num_seqs * p.tiles_per_seq), 2u);
  fp8_dequant_kernel<<<grid, kDequantThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ppa
