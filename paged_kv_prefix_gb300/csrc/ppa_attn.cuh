// Stage 2: the attention kernel for sm_103a (tcgen05 tensor cores, accumulators in TMEM).
//
// One persistent CTA per SM steals work items (query tile, KV head) from the list stage 1
// built. A query tile is 128 rows: tq tokens x the G query heads that share the KV head,
// token-major ("[Kernel][Gemma4] Prune Triton sliding-window tiles for multimodal prefixes",
// 关键源码片段: BLOCK_M = BLOCK_Q * num_queries_per_kv), so every K/V tile loaded is used
// by all G heads. For each live key tile [lo, hi) of the item:
//   1. gather K and V rows into shared memory, 16 bytes per cp.async. Each key position is
//      resolved on its own, to (block_table page, slot) below the context length or to a
//      k_new/v_new row above it, so tiles straddle pages and the context/new boundary and the
//      page size can be any integer (PR #54194 report, 功能与动机 / 关键源码片段). fp8 rows are
//      widened to bf16 on the way (exact);
//   2. S = Q K^T with tcgen05.mma (M=128, N=TN, K=16 steps) into TMEM;
//   3. one thread per row reads its S row from TMEM, masks keys outside the row's allowed
//      interval [kmin, kmax] (only on tiles it does not fully cover), and runs the online
//      softmax in fp32 with exp2; P goes to shared memory as bf16;
//   4. O (in TMEM) is rescaled by exp2(m_old - m_new) when the row maximum moved, then
//      O += P V with tcgen05.mma (M=128, N=D).
// The epilogue divides by the row sum and stores bf16.
//
// Shared-memory operands use the 128-byte swizzled K-major layout (rows of 64 bf16,
// 8-row atoms of 1024 bytes); V is the same bytes read as an MN-major operand.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ppa_internal.cuh"
#include "ppa_kernels.h"
#include "ppa_ptx.cuh"

namespace ppa {

template <int D, bool FP8>
struct AttnCfg {
  static constexpr int M = kRowsPerTile;  // 128 query rows
  static constexpr int TN = D >= 256 ? 64 : 128;
  static constexpr int THREADS = 128;
  static constexpr int CPR = D / 8;  // 16-byte chunks per bf16 row
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int KV_BYTES = TN * D * 2;  // one K (or V) tile
  static constexpr int P_BYTES = M * TN * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = Q_OFF + Q_BYTES;          // stage s: K at +2s*KV, V at +(2s+1)*KV
  static constexpr int P_OFF = KV_OFF + 4 * KV_BYTES;     // two stages of K and V
  static constexpr int MISC_OFF = P_OFF + P_BYTES;
  static constexpr int MISC_BYTES = 64 + 4 * TN * 8;      // barriers, slots, row pointers x2
  static constexpr int SMEM_BYTES = MISC_OFF + MISC_BYTES + 1024;  // + alignment slack
  static constexpr int TMEM_S = 0;
  static constexpr int TMEM_O = TN;
  static constexpr int TMEM_COLS = (TN + D <= 256) ? 256 : 512;
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Byte offset of 16-byte chunk `ch` of row `row` in a 128B-swizzled K-major operand of
// `rows` rows: 64-element column blocks of rows*128 bytes, 128-byte rows, chunk index XOR
// (row % 8) within each 1024-byte atom.
__device__ __forceinline__ uint32_t swz_off(int row, int ch, int rows) {
  return static_cast<uint32_t>((ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

template <int D, bool FP8>
__device__ __forceinline__ void gather_kv_tile(const AttnParams& p, int b, int g, int c, int s,
                                               int q_start, int k0, uint32_t sK, uint32_t sV,
                                               const char** rowK, const char** rowV) {
  using C = AttnCfg<D, FP8>;
  const int tid = threadIdx.x;
  constexpr size_t kCacheElt = FP8 ? 1 : 2;
  for (int r = tid; r < C::TN; r += C::THREADS) {
    const int pos = k0 + r;
    const char* kp = nullptr;
    const char* vp = nullptr;
    if (pos < c) {
      const int lp = pos / p.page_size;
      const int page = p.block_table[(size_t)b * p.max_pages_per_seq + lp];
      if (page >= 0 && page < p.num_pages) {
        const size_t off =
            (((size_t)page * p.page_size + (pos - lp * p.page_size)) * p.num_kv_heads + g) * D;
        kp = static_cast<const char*>(p.k_cache) + off * kCacheElt;
        vp = static_cast<const char*>(p.v_cache) + off * kCacheElt;
      } else {
        report(p.status, PPA_ERR_BAD_PAGE);
      }
    } else if (pos < s) {
      const size_t off = ((size_t)(q_start + pos - c) * p.num_kv_heads + g) * D;
      kp = static_cast<const char*>(p.k_new) + off * 2;
      vp = static_cast<const char*>(p.v_new) + off * 2;
    }
    rowK[r] = kp;
    rowV[r] = vp;
  }
  __syncthreads();
  if constexpr (!FP8) {
    for (int f = tid; f < C::TN * C::CPR; f += C::THREADS) {
      const int row = f / C::CPR, ch = f % C::CPR;
      const char* kp = rowK[row];
      const char* vp = rowV[row];
      const uint32_t o = swz_off(row, ch, C::TN);
      cp_async_16(sK + o, kp ? kp + ch * 16 : static_cast<const char*>(p.k_new), kp ? 16u : 0u);
      cp_async_16(sV + o, vp ? vp + ch * 16 : static_cast<const char*>(p.v_new), vp ? 16u : 0u);
    }
  } else {
    // 16 elements per unit: 16 fp8 bytes from the cache (widened here) or 32 bf16 bytes from
    // k_new / v_new (two cp.async).
    constexpr int UPR = D / 16;
    for (int f = tid; f < C::TN * UPR; f += C::THREADS) {
      const int row = f / UPR, u = f % UPR;
      const uint32_t o0 = swz_off(row, 2 * u, C::TN), o1 = swz_off(row, 2 * u + 1, C::TN);
      const bool cache_row = (k0 + row) < c;
      const char* ptrs[2] = {rowK[row], rowV[row]};
      const uint32_t bases[2] = {sK, sV};
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const char* src = ptrs[w];
        if (cache_row) {
          uint32_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          if (src) {
            const uint4 codes = ld_global_nc_v4(src + u * 16);
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[2 * i] = e4m3x2_to_bf16x2(static_cast<uint16_t>(cw[i] & 0xFFFFu));
              v[2 * i + 1] = e4m3x2_to_bf16x2(static_cast<uint16_t>(cw[i] >> 16));
            }
          }
          st_shared_v4(bases[w] + o0, v[0], v[1], v[2], v[3]);
          st_shared_v4(bases[w] + o1, v[4], v[5], v[6], v[7]);
        } else {
          const char* fallback = static_cast<const char*>(p.k_new);
          cp_async_16(bases[w] + o0, src ? src + u * 32 : fallback, src ? 16u : 0u);
          cp_async_16(bases[w] + o1, src ? src + u * 32 + 16 : fallback, src ? 16u : 0u);
        }
      }
    }
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(128, 1) attn_kernel(const AttnParams p) {
  using C = AttnCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + C::Q_OFF;
  const uint32_t sP = base + C::P_OFF;
  uint8_t* misc = smem + C::MISC_OFF;
  const uint32_t bar_s = smem_u32(misc);       // S = Q K^T complete
  const uint32_t bar_o = smem_u32(misc + 8);   // O += P V complete
  const uint32_t bar_fin = smem_u32(misc + 16);  // teardown: all MMAs retired
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 24);
  int* s_item = reinterpret_cast<int*>(misc + 28);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 32);
  // Row-pointer tables, one per K/V stage: the gather of tile kt+1 fills its table while
  // threads may still be reading tile kt's.
  const char** rowK0 = reinterpret_cast<const char**>(misc + 64);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_fin, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem + C::TMEM_S;
  const uint32_t tO = tmem + C::TMEM_O;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::TN, false, false);
  constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);

  uint32_t phase_s = 0, phase_o = 0;
  const int n_items = p.ws->n_items;
  const float neg_inf = -__int_as_float(0x7f800000);

  while (true) {
    if (tid == 0) *s_item = atomicAdd(&p.ws->next_item, 1);
    __syncthreads();
    const int item = *s_item;
    if (item >= n_items || *s_abort) break;

    const QTile qt = p.qtiles[p.order[item / p.num_kv_heads]];
    const int g = item % p.num_kv_heads;
    const int b = qt.seq, t = qt.t;
    const int c = p.context_lens[b];
    const int q_start = p.cu_query_lens[b];
    const int n = p.cu_query_lens[b + 1] - q_start;
    const int s = c + n;
    const int32_t* ranges =
        p.mask.mm_ranges ? p.mask.mm_ranges + (size_t)b * p.mask.max_mm_ranges * 2 : nullptr;

    // This thread's row: token tok of the tile, head hh of the group.
    const int tok = tid / p.group, hh = tid % p.group;
    const int j = t * p.tq + tok;
    const bool row_valid = tok < p.tq && j < n;
    int kmin = 0, kmax = s - 1;  // padding rows: every key (Q is zero there, values stay finite)
    if (row_valid) row_interval(c + j, s, p.mask, ranges, kmin, kmax);

    // Q tile (zero rows for padding), then the first K/V tile.
    for (int f = tid; f < C::M * C::CPR; f += C::THREADS) {
      const int row = f / C::CPR, ch = f % C::CPR;
      const int rt = row / p.group, rh = row % p.group, rj = t * p.tq + rt;
      const bool v = rt < p.tq && rj < n;
      const char* src = static_cast<const char*>(p.q) +
                        (v ? (((size_t)(q_start + rj) * p.num_q_heads + g * p.group + rh) * D) * 2 +
                                 ch * 16
                           : 0);
      cp_async_16(sQ + swz_off(row, ch, C::M), src, v ? 16u : 0u);
    }
    const int lo = qt.lo, hi = qt.hi;
    if (lo < hi) {
      gather_kv_tile<D, FP8>(p, b, g, c, s, q_start, lo * C::TN, base + C::KV_OFF,
                             base + C::KV_OFF + C::KV_BYTES, rowK0, rowK0 + C::TN);
    }
    cp_async_commit();

    float m_run = neg_inf, l_run = 0.f;
    float ks_ctx = 1.f, vs_ctx = 1.f;
    if constexpr (FP8) {
      ks_ctx = *p.k_scale;
      vs_ctx = *p.v_scale;
    }

    for (int kt = lo; kt < hi; ++kt) {
      const int st = (kt - lo) & 1;
      const uint32_t sK = base + C::KV_OFF + (2 * st) * C::KV_BYTES;
      const uint32_t sV = sK + C::KV_BYTES;
      if (kt + 1 < hi) {
        const uint32_t nK = base + C::KV_OFF + (2 * (st ^ 1)) * C::KV_BYTES;
        const char** rk = rowK0 + 2 * C::TN * (st ^ 1);
        gather_kv_tile<D, FP8>(p, b, g, c, s, q_start, (kt + 1) * C::TN, nK, nK + C::KV_BYTES,
                               rk, rk + C::TN);
      }
      cp_async_commit();
      cp_async_wait<1>();
      fence_proxy_async_smem();
      __syncthreads();

      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t db = kk >> 2, ks = kk & 3;
          const uint64_t a = sdesc_sw128(sQ + db * (C::M * 128) + ks * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sK + db * (C::TN * 128) + ks * 32, 16, 1024);
          mma_bf16_ss(tS, a, bd, kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar_s);
      }
      if (!*s_abort && !mbar_wait(bar_s, phase_s)) {
        report(p.status, PPA_ERR_TIMEOUT);
        *s_abort = 1;
      }
      phase_s ^= 1;
      tc_fence_after();

      // ---- softmax on this thread's row ----
      float sv[C::TN];
#pragma unroll
      for (int cc = 0; cc < C::TN / 32; ++cc) {
        uint32_t r32[32];
        tmem_ld_32(tS + lane_off + cc * 32, r32);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[cc * 32 + i] = __uint_as_float(r32[i]);
      }
      const int k0 = kt * C::TN;
      const int a0 = kmin - k0, a1 = kmax - k0;  // allowed local columns [a0, a1]
      const bool full = a0 <= 0 && a1 >= C::TN - 1;
      int jc = 0;  // columns below jc are fp8 cache keys
      if constexpr (FP8) jc = min(max(c - k0, 0), C::TN);
      float mx = neg_inf;
#pragma unroll
      for (int i = 0; i < C::TN; ++i) {
        float x = sv[i] * p.scale_log2;
        if constexpr (FP8) x = (i < jc) ? x * ks_ctx : x;
        if (!full && (i < a0 || i > a1)) x = neg_inf;
        sv[i] = x;
        mx = fmaxf(mx, x);
      }
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == neg_inf) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - m_use);
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < C::TN; ++i) {
        const float e = ex2_approx(sv[i] - m_use);
        sum += e;
        sv[i] = e;
      }
      l_run = l_run * alpha + sum;
      m_run = m_new;
      if constexpr (FP8) {
#pragma unroll
        for (int i = 0; i < C::TN; ++i) sv[i] = (i < jc) ? sv[i] * vs_ctx : sv[i];
      }
      // P (bf16) into the swizzled K-major operand, row = tid.
#pragma unroll
      for (int cb = 0; cb < C::TN / 8; ++cb) {
        const int i = cb * 8;
        st_shared_v4(sP + swz_off(tid, cb, C::M), pack_bf16x2(sv[i], sv[i + 1]),
                     pack_bf16x2(sv[i + 2], sv[i + 3]), pack_bf16x2(sv[i + 4], sv[i + 5]),
                     pack_bf16x2(sv[i + 6], sv[i + 7]));
      }
      // Rescale O when this row's maximum moved (warp-uniform decision).
      if (kt > lo && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o32[32];
          tmem_ld_32(tO + lane_off + cc * 32, o32);
#pragma unroll
          for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
          tmem_st_32(tO + lane_off + cc * 32, o32);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::TN / 16; ++kk) {
          const uint32_t kb = kk >> 2, ks = kk & 3;
          const uint64_t a = sdesc_sw128(sP + kb * (C::M * 128) + ks * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sV + kk * 16 * 128, C::TN * 128, 1024);
          mma_bf16_ss(tO, a, bd, kIdescO, (kt > lo || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar_o);
      }
      if (!*s_abort && !mbar_wait(bar_o, phase_o)) {
        report(p.status, PPA_ERR_TIMEOUT);
        *s_abort = 1;
      }
      phase_o ^= 1;
      tc_fence_after();
      // After a timeout the remaining waits are skipped but every barrier is still met; the
      // work loop exits at its next (uniform) check.
    }
    cp_async_wait<0>();

    // ---- epilogue: O / l -> bf16 ----
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(p.out) +
        ((size_t)(q_start + (row_valid ? j : 0)) * p.num_q_heads + g * p.group + hh) * D;
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t o32[32];
      tmem_ld_32(tO + lane_off + cc * 32, o32);
      if (row_valid && lo < hi) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o32[2 * i]) * inv_l,
                             __uint_as_float(o32[2 * i + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  // Teardown: retire every MMA this CTA issued (bounded), then free TMEM.
  cp_async_wait<0>();
  if (tid == 0) {
    tc_commit(bar_fin);
    if (!mbar_wait(bar_fin, 0)) report(p.status, PPA_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // The last CTA to finish re-arms the work counter, so the plan in the workspace can serve
  // the next launch on the stream without another stage-1 pass.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ws->done_ctas, 1) == (int)gridDim.x - 1) {
      p.ws->next_item = 0;
      p.ws->done_ctas = 0;
      __threadfence();
    }
  }
}

template <int D, bool FP8>
cudaError_t launch_attn(const AttnParams& p, int max_items, cudaStream_t stream) {
  using C = AttnCfg<D, FP8>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int configured[64] = {0};
  static int sm_count[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attn_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  const int grid = max(1, min(sm_count[dev], max_items));
  attn_kernel<D, FP8><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ppa
