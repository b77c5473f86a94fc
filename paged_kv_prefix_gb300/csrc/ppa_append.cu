// KV append: the new tokens' K/V written into their pages of the paged cache, the step before
// cache-sourced attention. New token j of sequence b goes to position c_b + j: page
// block_table[b][(c_b + j) / P], slot (c_b + j) % P, all KV heads at once (a cache row is
// [Hkv][D] like a k_new row). bf16 caches take the values unchanged; fp8 caches take the E4M3
// code nearest to value / scale (fp32 quotient; ties to even; saturated at 448; NaN to NaN),
// which is what cvt.rn.satfinite computes.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ppa_internal.cuh"
#include "ppa_kernels.h"
#include "ppa_ptx.cuh"

namespace ppa {
namespace {

constexpr int kAppendThreads = 256;

// E4M3 codes of two fp32 values, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight bf16 values (one 16-byte piece) divided by `scale` and encoded: 8 codes.
__device__ __forceinline__ uint2 encode8(uint4 v, float scale) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = e4m3x2_from_f32(__fdiv_rn(bf16_lo(w[i]), scale), __fdiv_rn(bf16_hi(w[i]), scale));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// One thread per 16-byte piece (8 elements) of a new token's row, K and V both.
__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const AppendParams p) {
  const int pieces = p.row_elems / 8;
  const long long total = (long long)p.total_q * pieces;
  const float ks = p.fp8 ? *p.k_scale : 1.f;
  const float vs = p.fp8 ? *p.v_scale : 1.f;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int tok = static_cast<int>(idx / pieces);
    const int pc = static_cast<int>(idx - (long long)tok * pieces);
    int lo = 0, hi = p.num_seqs - 1;  // last sequence with cu[b] <= tok
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu_query_lens[mid] <= tok) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int q0 = p.cu_query_lens[b], q1 = p.cu_query_lens[b + 1];
    const int c = p.context_lens[b];
    const int n = q1 - q0, j = tok - q0;
    bool ok = n >= 0 && c >= 0 && q0 >= 0 && c <= INT_MAX - n && j >= 0 && j < n;
    if (ok && (c + n - 1) / p.page_size >= p.max_pages_per_seq) ok = false;
    if (!ok) {
      report(p.status, PPA_ERR_INVALID);
      continue;
    }
    const int pos = c + j;
    const int lp = pos / p.page_size;
    const int page = p.block_table[(size_t)b * p.max_pages_per_seq + lp];
    if (page < 0 || page >= p.num_pages) {
      report(p.status, PPA_ERR_BAD_PAGE);
      continue;
    }
    const size_t src = ((size_t)tok * p.row_elems + (size_t)pc * 8) * 2;  // bytes
    const size_t row = (size_t)page * p.page_size + (pos - lp * p.page_size);
    const uint4 kv = ld_global_nc_v4(static_cast<const char*>(p.k_new) + src);
    const uint4 vv = ld_global_nc_v4(static_cast<const char*>(p.v_new) + src);
    if (!p.fp8) {
      const size_t dst = (row * p.row_elems + (size_t)pc * 8) * 2;
      *reinterpret_cast<uint4*>(static_cast<char*>(p.k_cache) + dst) = kv;
      *reinterpret_cast<uint4*>(static_cast<char*>(p.v_cache) + dst) = vv;
    } else {
      const size_t dst = row * p.row_elems + (size_t)pc * 8;
      *reinterpret_cast<uint2*>(static_cast<char*>(p.k_cache) + dst) = encode8(kv, ks);
      *reinterpret_cast<uint2*>(static_cast<char*>(p.v_cache) + dst) = encode8(vv, vs);
    }
  }
}

}  // namespace

cudaError_t launch_append_kv(const AppendParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0 || p.total_q == 0) return cudaSuccess;
  const long long total = (long long)p.total_q * (p.row_elems / 8);
  const long long blocks = (total + kAppendThreads - 1) / kAppendThreads;
  const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
  append_kv_kernel<<<grid, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ppa
