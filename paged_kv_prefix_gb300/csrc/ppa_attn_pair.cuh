// Stage 2 for head_dim 256: a CTA-pair kernel (a cluster of two CTAs on two SMs).
//
// One unit of work is two consecutive 128-row query tiles of one sequence and one KV head;
// CTA r of the pair owns tile r (its Q, S, P and O). The even CTA issues tcgen05 MMAs of
// M = 256 that cover both tiles (cta_group::2): each instruction reads A rows 0-127 from the
// even CTA and 128-255 from the odd one, and half of the B operand from each. So each CTA
// holds half of every key tile: K rows [r*64, r*64 + 64) of a 128-key tile (all 256 columns),
// and V columns [r*128, r*128 + 128) of all 128 keys. With 128-key tiles the S MMA runs at
// N = 128, where a single SM at head_dim 256 only has shared memory for 64-key tiles (N = 64
// MMAs, about two thirds of the tensor rate), and each instruction covers two SMs.
//
// Per key tile kt the even CTA issues S(kt+1) = Q K(kt+1)^T into the other S buffer, then
// O += P(kt) V(kt); the softmax of each CTA overlaps both (S is double-buffered in TMEM:
// O 256 columns + 2 x 128). Both query tiles walk the union of their live key intervals; a
// row's mask removes the keys outside its own interval.
//
// Synchronisation (all waits bounded):
//   MMA -> both CTAs: S_FULL, O_DONE, K/V/Q_EMPTY, FIN by multicast tcgen05.commit.
//   both CTAs -> MMA: P_FULL and O_EMPTY arrive on the even CTA's barriers (one arrival per
//     softmax warp); P(kt) also certifies that CTA's half of V(kt).
//   KQ_READY, KREADY[stage]: warp 9 of each CTA forwards "Q resident" per unit and "K half
//     resident" per key tile, so the issuer waits for K(kt+1) itself: three K stages then
//     give the loads about three key tiles of lead.
//   Work items: the even CTA's Q loader (warp 10) takes items and writes them into both
//     CTAs' rings; every consumer of either CTA releases the slot on the even CTA's barrier.
#pragma once

#include "ppa_attn_ws.cuh"

namespace ppa {

template <int D>
struct PairCfg {
  static_assert(D == 128 || D == 256, "the pair kernel serves head_dim 128 and 256");
  static constexpr int M = kRowsPerTile;  // rows per CTA (one query tile)
  static constexpr int TN = 128;          // keys per key tile
  static constexpr int KH = TN / 2;       // K rows held by each CTA
  static constexpr int DH = D / 2;        // V columns held by each CTA
  static constexpr int NSK = D == 256 ? 3 : 4;  // K stages
  static constexpr int NSV = D == 256 ? 2 : 4;  // V stages
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int KS_BYTES = KH * D * 2;   // one K stage: 64 rows x 256 columns
  static constexpr int VS_BYTES = TN * DH * 2;  // one V stage: 128 rows x 128 columns
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + Q_BYTES;
  static constexpr int V_OFF = K_OFF + NSK * KS_BYTES;
  static constexpr int BAR_OFF = V_OFF + NSV * VS_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = BAR_OFF + BAR_BYTES + 1024;  // + alignment slack
  static constexpr int TM_O = 0;  // O: D columns
  static constexpr int TM_S = D;  // S buffer b at TM_S + b*TN; P over its first TN/2
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 384;
  static_assert(TM_S + 2 * TN <= TMEM_COLS, "TMEM");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(tiles_per_unit(D) == 2, "plan and kernel agree on query tiles per unit");
  static_assert(keys_per_tile(D) == TN, "plan and kernel agree on the key tile");
};


namespace pairbar {
constexpr int KQ_READY = 272;   // both CTAs' Q of the unit resident
constexpr int KREADY = 280;     // [NSK] both CTAs' halves of the K stage resident
// ring consumers: even CTA warps 0-10 (softmax 4, producers 4, MMA, forwarder, Q loader),
// odd CTA the same without the MMA warp
constexpr int kConsumers = 21;
}  // namespace pairbar
static_assert(pairbar::KREADY + 8 * PairCfg<256>::NSK <= wsbar::LIMIT, "barrier block layout");

struct PairShared {
  WsShared ws;
  uint32_t rank;
  __device__ uint32_t bar(int off) const { return ws.bar(off); }
  // the even CTA's copy of barrier `off`, as a cluster address
  __device__ uint32_t lead(int off) const { return mapa_shared(ws.bar(off), 0); }
  // Bounded wait with acquire at cluster scope (barriers that take the peer's arrivals).
  __device__ bool wait_c(int off, uint32_t parity) const {
    const uint32_t b = ws.bars + off;
    if (mbar_try_wait_cluster(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait_cluster(b, parity)) return true;
      if (*ws.abort) return false;
      if (globaltimer_ns() - t0 > ws.limit()) {
        *ws.abort = 1;
        report(ws.status, PPA_ERR_TIMEOUT);
        return false;
      }
    }
  }
};

__device__ __forceinline__ bool wait_c_warp(const PairShared& sh, int off, uint32_t parity) {
  return __all_sync(0xffffffffu, sh.wait_c(off, parity));
}

// Item ring: the even CTA fills both CTAs' slots; consumers release on the even CTA.
__device__ __forceinline__ int pair_ring_get(const PairShared& sh, int k) {
  const int slot = k & 1;
  int item = -1;
  if ((threadIdx.x & 31) == 0) {
    if (sh.wait_c(wsbar::ITEM_FULL + 8 * slot, (k >> 1) & 1)) item = sh.ws.ring[slot];
    mbar_arrive_cluster(sh.lead(wsbar::ITEM_EMPTY + 8 * slot));
  }
  return __shfl_sync(0xffffffffu, item, 0);
}

__device__ __forceinline__ int pair_ring_get1(const PairShared& sh, int k) {
  const int slot = k & 1;
  int item = -1;
  if (sh.wait_c(wsbar::ITEM_FULL + 8 * slot, (k >> 1) & 1)) item = sh.ws.ring[slot];
  mbar_arrive_cluster(sh.lead(wsbar::ITEM_EMPTY + 8 * slot));
  return item;
}

__device__ __forceinline__ void pair_ring_put(const PairShared& sh, const AttnParams& p, int k,
                                              int n_items) {
  const int slot = k & 1;
  int item = -1;
  if (sh.wait_c(wsbar::ITEM_EMPTY + 8 * slot, ((k >> 1) & 1) ^ 1)) {
    item = atomicAdd(&p.ws->next_item, 1);
    if (item >= n_items) item = -1;
  }
  const uint32_t ring_slot = sh.bar(wsbar::RING) + 4 * slot;
  sh.ws.ring[slot] = item;
  st_shared_cluster_u32(mapa_shared(ring_slot, 1), static_cast<uint32_t>(item));
  mbar_arrive(sh.bar(wsbar::ITEM_FULL + 8 * slot));
  mbar_arrive_cluster(mapa_shared(sh.bar(wsbar::ITEM_FULL + 8 * slot), 1));
}

// Row gather (bf16 cache) for one 32-row block: rows row0 .. row0+31 whose bit is set in
// `rowmask`; lane l's source row starts at `mine` (nullptr: zero fill); `cols` elements per
// row land in the 128-byte-swizzled layout with `rows` rows per 64-column block.
__device__ __forceinline__ void pair_gather_rows(const char* zero_src, int row0, uint32_t rowmask,
                                                 const char* mine, uint32_t sX, int rows,
                                                 int cols) {
  const int lane = threadIdx.x & 31;
  const int cpr = cols / 8;  // 16-byte chunks per row
  const int rpi = 32 / cpr;  // rows per warp instruction
  for (int it = 0; it * rpi < 32; ++it) {
    const int lr = it * rpi + lane / cpr;
    const int ch = lane % cpr;
    const char* rp = reinterpret_cast<const char*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine), lr & 31));
    if (lr < 32 && ((rowmask >> lr) & 1u))
      cp_async_16(sX + swz128(row0 + lr, ch, rows), rp ? rp + ch * 16 : zero_src, rp ? 16u : 0u);
  }
}

// ---------------------------------------------------------------------------------------
// Producers (warps 4-7 of each CTA): warps 4-5 load this CTA's K half (32 rows each), warps
// 6-7 its V half (64 rows each). TMA boxes of 16 rows where a chunk lies in one page of cached
// context or in the new tokens; row gathers otherwise (page or context boundary, fp8).
// ---------------------------------------------------------------------------------------
template <int D, bool FP8>
__device__ void pair_producer(const AttnParams& p, const PairShared& sh, uint32_t base,
                              int n_items) {
  using C = PairCfg<D>;
  constexpr uint32_t kChunkBytes = 16 * 128;  // one 64-column block of 16 rows
  constexpr size_t kCacheElt = FP8 ? 1 : 2;
  const int lane = threadIdx.x & 31;
  const int pw = (threadIdx.x >> 5) - 4;  // 0..3
  const int w = pw >> 1;                  // 0: K, 1: V
  const int half = pw & 1;
  const int rpw = w == 0 ? C::KH / 2 : C::TN / 2;  // rows per warp: 32 (K) or 64 (V)
  const int rows = w == 0 ? C::KH : C::TN;         // rows of one stage's column block
  const int ncol_blocks = w == 0 ? D / 64 : C::DH / 64;
  const int col0 = w == 0 ? 0 : static_cast<int>(sh.rank) * C::DH;  // first column loaded
  const void* tm_new = w == 0 ? (const void*)&p.tm.k_new : (const void*)&p.tm.v_new;
  const void* tm_cache = w == 0 ? (const void*)&p.tm.k_cache : (const void*)&p.tm.v_cache;
  const void* tm_new32 = w == 0 ? (const void*)&p.tm.k_new32 : (const void*)&p.tm.v_new32;
  const void* tm_cache32 = w == 0 ? (const void*)&p.tm.k_cache32 : (const void*)&p.tm.v_cache32;
  const char* g_cache = static_cast<const char*>(w == 0 ? p.k_cache : p.v_cache);
  const char* g_new = static_cast<const char*>(w == 0 ? p.k_new : p.v_new);
  if (lane == 0) {
    if (!p.kv_in_cache) {  // the new-token maps are encoded only when k_new / v_new are read
      tma_prefetch_desc(tm_new);
      tma_prefetch_desc(tm_new32);
    }
    if constexpr (!FP8) {
      tma_prefetch_desc(tm_cache);
      tma_prefetch_desc(tm_cache32);
    }
  }
  const int ns = w == 0 ? C::NSK : C::NSV;
  const int empty_bar = w == 0 ? wsbar::K_EMPTY : wsbar::V_EMPTY;
  const int full_bar = w == 0 ? wsbar::K_FULL : wsbar::V_FULL;
  const uint32_t stage0 = base + (w == 0 ? C::K_OFF : C::V_OFF);
  const float kv_scale = FP8 ? *(w == 0 ? p.k_scale : p.v_scale) : 1.f;  // fp8 dequantisation
  const uint32_t stage_bytes = w == 0 ? C::KS_BYTES : C::VS_BYTES;
  uint32_t kv_iter = 0;
  for (int k = 0;; ++k) {
    const int item = pair_ring_get(sh, k);
    if (item < 0) break;
    const UnitInfo u = decode_item(p, item);

    bool ok = true;
    for (int kt = u.lo; kt < u.hi; ++kt, ++kv_iter) {
      const int s = kv_iter % ns;
      const uint32_t ph = (kv_iter / ns) & 1;
      // key position of this CTA's first row of the stage
      const int key0 = kt * C::TN - u.koff + (w == 0 ? static_cast<int>(sh.rank) * C::KH : 0);
      // Classify this warp's 16-row chunks before waiting for the stage, so that the
      // block-table loads overlap the wait. Lane c < rpw/16 takes chunk c.
      int ctype = 0, crow = 0;  // 1 = cache box, 2 = new-token box, 0 = row gather
      if (lane * 16 < rpw) {
        const int p0 = key0 + half * rpw + 16 * lane;
        if (p0 >= u.cs) {
          if (!p.kv_in_cache) {  // new tokens (cache-sourced: past the sequence, zero fill)
            ctype = 2;
            crow = u.q_start + p0 - u.c;
          }
        } else if (!FP8 && p0 >= 0 && p0 + 15 < u.cs) {  // (chunks below key 0: zero fill)
          const int lp = p0 / p.page_size;
          if ((p0 + 15) / p.page_size == lp) {
            const int page = p.block_table[(size_t)u.b * p.max_pages_per_seq + lp];
            if (page >= 0 && page < p.num_pages) {
              ctype = 1;
              crow = page * p.page_size + (p0 - lp * p.page_size);
            }
          }
        }
      }
      if (!wait_warp(sh.ws, empty_bar + 8 * s, ph ^ 1)) { ok = false; break; }
      const uint32_t sX = stage0 + s * stage_bytes;
      const uint32_t bar = sh.bar(full_bar + 8 * s);
      uint32_t bytes = 0;
      bool any_fallback = false;
      for (int sub = 0; sub * 32 < rpw; ++sub) {
        const int row0 = half * rpw + 32 * sub;  // row within the stage
        const int p_row0 = key0 + row0;
        int types[2], crows[2];
        uint32_t fb_mask = 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          types[c] = __shfl_sync(0xffffffffu, ctype, 2 * sub + c);
          crows[c] = __shfl_sync(0xffffffffu, crow, 2 * sub + c);
          if (types[c] == 0) fb_mask |= 0xFFFFu << (16 * c);
        }
        // both chunks from one contiguous source run: one 32-row box per column block
        const bool one_run = types[0] != 0 && types[0] == types[1] && crows[1] == crows[0] + 16;
        if (lane == 0 && one_run) {
          const void* tm32 = types[0] == 1 ? tm_cache32 : tm_new32;
          for (int db = 0; db < ncol_blocks; ++db)
            tma_load_3d(sX + db * (rows * 128) + row0 * 128, tm32, col0 + db * 64, u.g, crows[0], bar);
          bytes += ncol_blocks * 2 * kChunkBytes;
        }
        if (lane == 0 && !one_run) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (types[c] == 0) continue;
            for (int db = 0; db < ncol_blocks; ++db)
              tma_load_3d(sX + db * (rows * 128) + (row0 + 16 * c) * 128,
                          types[c] == 1 ? tm_cache : tm_new, col0 + db * 64, u.g, crows[c], bar);
            bytes += ncol_blocks * kChunkBytes;
          }
        }
        if (fb_mask != 0) {  // row gather; lane r sources row row0 + r
          const char* mine = nullptr;
          const int pos = p_row0 + lane;
          if (pos < 0) {
            // below key 0 (a shifted first tile): zero fill
          } else if (pos < u.cs) {
            const int lp = pos / p.page_size;
            const int page = p.block_table[(size_t)u.b * p.max_pages_per_seq + lp];
            if (page >= 0 && page < p.num_pages) {
              mine = g_cache +
                     ((((size_t)page * p.page_size + (pos - lp * p.page_size)) * p.num_kv_heads +
                       u.g) * D + col0) * kCacheElt;
            } else {
              report(p.status, PPA_ERR_BAD_PAGE);
            }
          } else if (pos < u.s) {
            mine = g_new + (((size_t)(u.q_start + pos - u.c) * p.num_kv_heads + u.g) * D + col0) * 2;
          }
          if constexpr (FP8) {
            if (w == 0)
              gather_rows_fp8<D>(g_cache, row0, fb_mask, u.cs - p_row0,
                                 mine, sX, rows, kv_scale);
            else
              gather_rows_fp8<C::DH>(g_cache, row0, fb_mask,
                                     u.cs - p_row0, mine, sX, rows, kv_scale);
          } else {
            pair_gather_rows(g_cache, row0, fb_mask, mine, sX, rows,
                             ncol_blocks * 64);
          }
          any_fallback = true;
        }
      }
      if (any_fallback) {
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    }
    if (!ok) break;
  }
  cp_async_wait<0>();
  // This warp's TMA copies land before the CTA exits: wait (bounded) for the last fill of
  // every stage (see ws_producer).
  if (lane == 0) {
    for (uint32_t s = 0; s < static_cast<uint32_t>(ns) && s < kv_iter; ++s) {
      const uint32_t f = s + ns * ((kv_iter - 1 - s) / ns);
      sh.ws.drain(full_bar + 8 * s, (f / ns) & 1);
    }
  }
}

// Q loader (warp 10 of each CTA): this CTA's query tile of each unit; in the even CTA, lane 0
// also runs the item ring. Separate from the K and V streams so that they prefetch across
// unit boundaries instead of waiting for Q_EMPTY.
template <int D>
__device__ void pair_qloader(const AttnParams& p, const PairShared& sh, uint32_t base,
                             int n_items) {
  using C = PairCfg<D>;
  const int lane = threadIdx.x & 31;
  if (lane == 0) tma_prefetch_desc(&p.tm.q);
  uint32_t q_phase = 0;
  bool loaded = false;
  for (int k = 0;; ++k) {
    if (sh.rank == 0 && lane == 0) pair_ring_put(sh, p, k, n_items);
    const int item = pair_ring_get(sh, k);
    if (item < 0) break;
    const UnitInfo u = decode_item(p, item);
    if (!wait_warp(sh.ws, wsbar::Q_EMPTY, q_phase ^ 1)) break;
    q_phase ^= 1;
    loaded = true;
    if (lane == 0) {  // rows past the sequence read zeros or foreign rows; the mask drops them
      const uint32_t box_bytes = static_cast<uint32_t>(p.group * p.tq * 128);
      mbar_arrive_expect_tx(sh.bar(wsbar::Q_FULL), (D / 64) * box_bytes);
#pragma unroll
      for (int db = 0; db < D / 64; ++db)
        tma_load_3d(base + C::Q_OFF + db * (C::M * 128), &p.tm.q, db * 64, u.g * p.group,
                    u.q_start + (u.t0 + static_cast<int>(sh.rank)) * p.tq, sh.bar(wsbar::Q_FULL));
    }
  }
  if (loaded && lane == 0) sh.ws.drain(wsbar::Q_FULL, q_phase ^ 1);  // the last load landed
}

// ---------------------------------------------------------------------------------------
// Readiness forwarder (warp 9 of each CTA): the issuer reads both CTAs' shared memory but can
// wait only on its own barriers. Lane 0 waits for this CTA's Q of each unit and for each K
// half in ring order and arrives on the even CTA's KQ_READY / KREADY[stage]. One barrier per
// K stage keeps one CTA's early arrivals out of the other's phase: the fill after next of a
// stage needs the issuer to have consumed this one.
// ---------------------------------------------------------------------------------------
template <int D>
__device__ void pair_forwarder(const AttnParams& p, const PairShared& sh) {
  using C = PairCfg<D>;
  uint32_t kv = 0, q_phase = 0;
  const bool lead = (threadIdx.x & 31) == 0;
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int item = pair_ring_get(sh, k);
    if (item < 0) break;
    const UnitInfo u = decode_item(p, item);
    if (lead) {
      ok = sh.ws.wait(wsbar::Q_FULL, q_phase);
      if (ok) mbar_arrive_cluster(sh.lead(pairbar::KQ_READY));
      // every K fill in ring order: the previous fill of each stage was this thread's own
      // wait, so the parity tests are unambiguous
      for (int kt = u.lo; kt < u.hi && ok; ++kt, ++kv) {
        ok = sh.ws.wait(wsbar::K_FULL + 8 * (kv % C::NSK), (kv / C::NSK) & 1);
        if (ok) mbar_arrive_cluster(sh.lead(pairbar::KREADY + 8 * (kv % C::NSK)));
      }
    }
    q_phase ^= 1;
    ok = __all_sync(0xffffffffu, ok);
  }
}

// ---------------------------------------------------------------------------------------
// MMA issuer (warp 8 lane 0 of the even CTA).
// ---------------------------------------------------------------------------------------
template <int D>
__device__ void pair_mma(const AttnParams& p, const PairShared& sh, uint32_t base, uint32_t tmem) {
  using C = PairCfg<D>;
  if ((threadIdx.x & 31) != 0) return;
  constexpr uint32_t kIdescS = idesc_bf16_f32(256, C::TN, false, false);
  constexpr uint32_t kIdescO = idesc_bf16_f32(256, D, false, true);
  const uint64_t dQ = sdesc_sw128(base + C::Q_OFF, 16, 1024);
  const uint64_t dK0 = sdesc_sw128(base + C::K_OFF, 16, 1024);
  const uint64_t dV0 = sdesc_sw128(base + C::V_OFF, C::TN * 128, 1024);
  constexpr uint32_t kKStep = C::KS_BYTES >> 4, kVStep = C::VS_BYTES >> 4;
  uint32_t kv_iter = 0, kq_phase = 0, pf_phase = 0, oe_phase = 0, sc = 0;
  // both CTAs' halves of the K tile at ring position kv resident
  auto k_ready = [&](uint32_t kv) {
    const bool r = sh.wait_c(pairbar::KREADY + 8 * (kv % C::NSK), (kv / C::NSK) & 1);
    tc_fence_after();
    return r;
  };
  auto issue_s = [&](int stage, uint32_t buf) {
    const uint32_t tS = tmem + C::TM_S + buf * C::TN;
    uint64_t a0 = dQ, b0 = dK0 + stage * kKStep;
    asm volatile("" : "+l"(a0), "+l"(b0));  // keep per-MMA descriptors out of registers
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off_a = ((kk >> 2) * (C::M * 128) + (kk & 3) * 32) >> 4;
      const uint32_t off_b = ((kk >> 2) * (C::KH * 128) + (kk & 3) * 32) >> 4;
      mma2_bf16_ss(tS, a0 + off_a, b0 + off_b, kIdescS, kk > 0 ? 1u : 0u);
    }
    tc_commit_pair(sh.bar(wsbar::S_FULL + 8 * buf));
    tc_commit_pair(sh.bar(wsbar::K_EMPTY + 8 * stage));  // S is K's only reader
  };
  auto issue_pv = [&](int stage, uint32_t buf, uint32_t acc0) {
    const uint32_t tP = tmem + C::TM_S + buf * C::TN;
    uint64_t b0 = dV0 + stage * kVStep;
    asm volatile("" : "+l"(b0));
#pragma unroll
    for (int kk = 0; kk < C::TN / 16; ++kk)
      mma2_bf16_ts(tmem + C::TM_O, tP + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdescO,
                   kk > 0 ? 1u : acc0);
    tc_commit_pair(sh.bar(wsbar::O_DONE));
    tc_commit_pair(sh.bar(wsbar::V_EMPTY + 8 * stage));
  };
  bool ok = true;
  for (int k = 0; ok; ++k) {
    const int item = pair_ring_get1(sh, k);
    if (item < 0) break;
    const UnitInfo u = decode_item(p, item);
    const int n_kt = u.hi - u.lo;
    // both CTAs' Q resident
    if (!sh.wait_c(pairbar::KQ_READY, kq_phase)) break;
    kq_phase ^= 1;
    if (!k_ready(kv_iter)) break;
    issue_s(kv_iter % C::NSK, sc & 1);
    if (n_kt > 1) {
      if (!k_ready(kv_iter + 1)) break;
      issue_s((kv_iter + 1) % C::NSK, (sc + 1) & 1);
    }
    if (n_kt <= 2) tc_commit_pair(sh.bar(wsbar::Q_EMPTY));  // every S of the unit issued
    // O must have been read out by both CTAs' previous epilogues
    if (!sh.wait_c(wsbar::O_EMPTY, oe_phase ^ 1)) break;
    oe_phase ^= 1;
    for (int kt = u.lo; kt < u.hi; ++kt, ++kv_iter, ++sc) {
      if (kt > u.lo && kt + 1 < u.hi) {
        if (!k_ready(kv_iter + 1)) { ok = false; break; }
        issue_s((kv_iter + 1) % C::NSK, (sc + 1) & 1);
        if (kt + 2 == u.hi) tc_commit_pair(sh.bar(wsbar::Q_EMPTY));
      }
      // P(kt) from both CTAs; also certifies V(kt) in both
      if (!sh.wait_c(wsbar::P_FULL, pf_phase)) { ok = false; break; }
      pf_phase ^= 1;
      tc_fence_after();
      issue_pv(kv_iter % C::NSV, sc & 1, kt > u.lo ? 1u : 0u);
    }
  }
}

// ---------------------------------------------------------------------------------------
// Softmax (warps 0-3 of each CTA): thread r owns row r of this CTA's query tile.
// ---------------------------------------------------------------------------------------
template <int D, bool FP8, bool SPLIT>
__device__ void pair_softmax(const AttnParams& p, const PairShared& sh, uint32_t tmem) {
  using C = PairCfg<D>;
  const int warp = threadIdx.x >> 5;
  const int r = threadIdx.x & 127;
  const int i = static_cast<int>(sh.rank);
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tO = tmem + C::TM_O + lane_off;
  const float neg_inf = -__int_as_float(0x7f800000);
  const float scale = p.scale_log2;
  const uint32_t p_full = sh.lead(wsbar::P_FULL), o_empty = sh.lead(wsbar::O_EMPTY);
  uint32_t od_phase = 0, sc = 0;
  const int tok = r / p.group, hh = r % p.group;
  // This thread's row of one unit. The next unit's is prepared right after the last P of the
  // current unit, before its epilogue: the ring's release arrival then has no output stores
  // to wait for, and the item's dependent loads and the range scan overlap the last PV.
  struct RowPlan {
    UnitInfo u;
    uint32_t kv0;  // K/V ring position of the unit's first key tile
    int j, kmin, kmax;
    bool row_valid;
  };
  auto plan_row = [&](int item, uint32_t kv0, RowPlan& rp) {
    rp.u = decode_item(p, item);
    rp.kv0 = kv0;
    rp.j = (rp.u.t0 + i) * p.tq + tok;
    rp.row_valid = i < rp.u.nt && tok < p.tq && rp.j < rp.u.n;
    row_bounds_of(p, rp.u, rp.j, rp.row_valid, rp.kmin, rp.kmax);
  };
  int item = pair_ring_get(sh, 0);
  RowPlan cur;
  if (item >= 0) plan_row(item, 0u, cur);
  for (int k = 0; item >= 0; ++k) {
    const UnitInfo& u = cur.u;
    const uint32_t kv0 = cur.kv0;
    const int lo = u.lo, hi = u.hi;  // the pair walks the union of both tiles' intervals
    const int j = cur.j, kmin = cur.kmin, kmax = cur.kmax;
    const bool row_valid = cur.row_valid;
    float m_ref = neg_inf, l_run = 0.f;
    bool ok = true;
    for (int kt = lo; kt < hi; ++kt) {
      const uint32_t buf = sc & 1;
      const uint32_t tS = tmem + C::TM_S + buf * C::TN + lane_off;
      const uint32_t kv = kv0 + (kt - lo);
      const uint32_t bar_v = wsbar::V_FULL + 8 * (kv % C::NSV), par_v = (kv / C::NSV) & 1;
      if (!wait_warp(sh.ws, wsbar::S_FULL + 8 * buf, (sc >> 1) & 1)) { ok = false; break; }
      ++sc;
      // Probe V(kt) now (after S(kt) landed: every earlier fill of its stage was confirmed
      // before S(kt) could be issued); wait before arriving only if needed.
      const bool v_ready = mbar_test_wait(sh.bar(bar_v), par_v);
      tc_fence_after();
      float sv[C::TN];
#pragma unroll
      for (int cc = 0; cc < C::TN / 64; ++cc) {
        uint32_t r64[64];
        tmem_ld_64(tS + cc * 64, r64);
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[cc * 64 + e] = __uint_as_float(r64[e]);
      }
      const int k0 = kt * C::TN - u.koff;  // key position of the tile's first column
      const int a0 = kmin - k0, a1 = kmax - k0;  // allowed local columns [a0, a1]
      if (!(a0 <= 0 && a1 >= C::TN - 1)) {
#pragma unroll
        for (int e = 0; e < C::TN; ++e) sv[e] = (e < a0 || e > a1) ? neg_inf : sv[e];
      }
      constexpr int kPer = C::TN / 8;
      float mx[8];
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        float m = fmax3(sv[q8], sv[q8 + 8], sv[q8 + 16]);
        int jj = 3;
#pragma unroll
        for (; jj + 1 < kPer; jj += 2) m = fmax3(m, sv[q8 + 8 * jj], sv[q8 + 8 * jj + 8]);
        if (jj < kPer) m = fmaxf(m, sv[q8 + 8 * jj]);
        mx[q8] = m;
      }
      const float tile_max =
          fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      const float m_tile = tile_max * scale;
      bool rescale = false;
      float alpha = 1.f;
      if (m_tile > m_ref + 8.f) {  // stale reference kept unless the maximum grew by > 2^8
        alpha = ex2_approx(m_ref - m_tile);
        rescale = kt > lo;
        m_ref = m_tile;
      }
      const float m_use = m_ref == neg_inf ? 0.f : m_ref;
      const uint64_t scale2 = f2_pack(scale, scale), negm2 = f2_pack(-m_use, -m_use);
      uint64_t sum2[4] = {0, 0, 0, 0};
      uint32_t pk[C::TN / 2];
#pragma unroll
      for (int e = 0; e < C::TN; e += 2) {
        float y0, y1;
        f2_unpack(f2_fma(f2_pack(sv[e], sv[e + 1]), scale2, negm2), y0, y1);
        float p0 = ex2_approx(y0);
        float p1 = ex2_approx(y1);
        sum2[(e >> 1) & 3] = f2_add(sum2[(e >> 1) & 3], f2_pack(p0, p1));
        pk[e >> 1] = pack_bf16x2(p0, p1);
      }
      float sl[8];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) f2_unpack(sum2[q4], sl[2 * q4], sl[2 * q4 + 1]);
      l_run = l_run * alpha +
              (((sl[0] + sl[1]) + (sl[2] + sl[3])) + ((sl[4] + sl[5]) + (sl[6] + sl[7])));
#pragma unroll
      for (int cc = 0; cc < C::TN / 64; ++cc) {
        uint32_t w32[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) w32[e] = pk[cc * 32 + e];
        tmem_st_32(tS + cc * 32, w32);
      }
      // S(kt) was issued before PV(kt-1): O is idle only after that PV completed
      if (kt > lo) {
        if (!wait_warp(sh.ws, wsbar::O_DONE, od_phase)) { ok = false; break; }
        od_phase ^= 1;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o32[32];
          tmem_ld_32(tO + cc * 32, o32);
#pragma unroll
          for (int e = 0; e < 32; ++e) o32[e] = __float_as_uint(__uint_as_float(o32[e]) * alpha);
          tmem_st_32(tO + cc * 32, o32);
        }
      }
      tmem_st_wait();
      if (!__all_sync(0xffffffffu, v_ready) && !wait_warp(sh.ws, bar_v, par_v)) { ok = false; break; }
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive_cluster_relaxed(p_full);  // P is in TMEM
    }
    if (!ok) break;
    const int next = pair_ring_get(sh, k + 1);
    RowPlan nxt = cur;
    if (next >= 0) plan_row(next, kv0 + static_cast<uint32_t>(hi - lo), nxt);
    // ---- epilogue: the last PV; O / l to bf16 ----
    if (!wait_warp(sh.ws, wsbar::O_DONE, od_phase)) break;
    od_phase ^= 1;
    tc_fence_after();
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(p.out) +
        ((size_t)(u.q_start + (row_valid ? j : 0)) * p.num_q_heads + u.g * p.group + hh) * D;
    auto store32 = [&](const uint32_t (&o32)[32], int cc) {
      if (!row_valid) return;
      uint32_t wv[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        wv[e] = pack_bf16x2(__uint_as_float(o32[2 * e]) * inv_l,
                            __uint_as_float(o32[2 * e + 1]) * inv_l);
      uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dst[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
    };
    if (SPLIT && u.part >= 0) {  // a split-KV segment: O / l in fp32 and its log-sum-exp
      if constexpr (SPLIT) split_partial_store<D>(p, u, r, row_valid, m_ref, l_run, inv_l, tO);
    } else {
      // 32-column chunks, the load of the next in flight while one is converted and stored
      static_assert((D / 32) % 2 == 0, "chunk pairs");
      uint32_t oa[32], ob[32];
      tmem_ld_32_async(tO, oa);
      tmem_ld_wait(oa);
#pragma unroll 1
      for (int cc = 0; cc < D / 32; cc += 2) {
        tmem_ld_32_async(tO + (cc + 1) * 32, ob);
        store32(oa, cc);
        tmem_ld_wait(ob);
        if (cc + 2 < D / 32) tmem_ld_32_async(tO + (cc + 2) * 32, oa);
        store32(ob, cc + 1);
        if (cc + 2 < D / 32) tmem_ld_wait(oa);
      }
    }
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_cluster_relaxed(o_empty);  // O was read from TMEM
    item = next;
    cur = nxt;
  }
}

template <int D, bool FP8, bool SPLIT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(384, 1)
    attn_pair_kernel(const __grid_constant__ AttnParams p) {
  using C = PairCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint8_t* barp = smem + C::BAR_OFF;
  PairShared sh;
  sh.ws.bars = base + C::BAR_OFF;
  sh.ws.abort = reinterpret_cast<volatile int*>(barp + wsbar::ABORT);
  sh.ws.ring = reinterpret_cast<volatile int*>(barp + wsbar::RING);
  sh.ws.status = p.status;
  sh.rank = cluster_ctarank();
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) {
    using namespace wsbar;
    for (int s = 0; s < 2; ++s) {
      mbar_init(sh.bar(ITEM_FULL + 8 * s), 1);
      mbar_init(sh.bar(ITEM_EMPTY + 8 * s), pairbar::kConsumers);
      mbar_init(sh.bar(S_FULL + 8 * s), 1);
    }
    mbar_init(sh.bar(Q_FULL), 1);
    mbar_init(sh.bar(Q_EMPTY), 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(sh.bar(K_FULL + 8 * s), 2);  // the two K warps, with their TMA bytes
      mbar_init(sh.bar(K_EMPTY + 8 * s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(sh.bar(V_FULL + 8 * s), 2);
      mbar_init(sh.bar(V_EMPTY + 8 * s), 1);
    }
    mbar_init(sh.bar(P_FULL), 8);   // 4 softmax warps x 2 CTAs
    mbar_init(sh.bar(O_DONE), 1);
    mbar_init(sh.bar(O_EMPTY), 8);
    mbar_init(sh.bar(FIN), 1);
    *reinterpret_cast<unsigned long long*>(barp + LIMIT) = p.wait_ns;
    mbar_init(sh.bar(pairbar::KQ_READY), 2);
    for (int s = 0; s < C::NSK; ++s) mbar_init(sh.bar(pairbar::KREADY + 8 * s), 2);
    *sh.ws.abort = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc_pair(sh.bar(wsbar::TMEM_SLOT), C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(barp + wsbar::TMEM_SLOT);
  const int n_items = p.ws->n_items;

  // 384 threads x 168 registers at launch: softmax warpgroup 232, the other two 136 each.
  if (warp < 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 232;\n" ::: "memory");
    pair_softmax<D, FP8, SPLIT>(p, sh, tmem);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 136;\n" ::: "memory");
  }
  if (warp < 4) {
  } else if (warp < 8) {
    pair_producer<D, FP8>(p, sh, base, n_items);
  } else if (warp == 8) {
    if (sh.rank == 0) {
      pair_mma<D>(p, sh, base, tmem);
      if ((tid & 31) == 0) tc_commit_pair(sh.bar(wsbar::FIN));  // retire every pair MMA
    }
  } else if (warp == 9) {
    pair_forwarder<D>(p, sh);
  } else if (warp == 10) {
    pair_qloader<D>(p, sh, base, n_items);
  }
  // TMEM of both CTAs is written by the even CTA's MMAs: both wait for them to retire.
  if (tid == 0 && !sh.ws.drain(wsbar::FIN, 0)) report(p.status, PPA_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no arrival or store from the peer is still in flight
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
  // The last CTA to finish re-arms the work counter for the next launch on this plan.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ws->done_ctas, 1) == (int)gridDim.x - 1) {
      p.ws->next_item = 0;
      p.ws->done_ctas = 0;
      __threadfence();
    }
  }
}

template <int D, bool FP8, bool SPLIT>
cudaError_t launch_attn_pair(const AttnParams& p, int max_items, cudaStream_t stream) {
  using C = PairCfg<D>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // per-device set-up, once; under a lock so that a concurrent first call cannot read
  // sm_count before it is written
  static std::mutex mu;
  static int configured[64] = {0};
  static int sm_count[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(attn_pair_kernel<D, FP8, SPLIT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      configured[dev] = 1;
    }
    sms = sm_count[dev];
  }
  const int pairs = max(1, min(sms / 2, max_items));
  attn_pair_kernel<D, FP8, SPLIT><<<2 * pairs, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ppa
