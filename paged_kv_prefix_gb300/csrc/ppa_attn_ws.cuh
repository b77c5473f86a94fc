// Stage 2: a warp-specialised, pipelined attention kernel for sm_103a.
//
// One persistent CTA per SM, 16 warps:
//   warps 0-3   softmax for query tile A (one thread per row)     \ 184 registers each
//   warps 4-7   softmax for query tile B                          /
//   warps 8-11  producers: TMA / cp.async paged K/V gather            56 registers each
//   warp  12    MMA issue (lane 0)                                  \ 88 registers each
//   warp  13    Q loads and the item ring                           |
//   warps 14-15 idle                                               /
// A unit of work is two consecutive 128-row query tiles (tq tokens x G heads each, token
// major) of one sequence and one KV head; both tiles consume one stream of K/V tiles, so each
// tile is gathered once for 256 query rows. Per key tile kt the MMA warp issues, for each
// query tile i whose live interval contains kt:
//     O_i += P_i V(kt)        (P_i read from TMEM: the softmax wrote it over S_i)
//     S_i  = Q_i K(kt+1)^T    (next tile, into TMEM)
// so the softmax of one tile overlaps the MMAs of the other ("ping-pong"). S, P and O live in
// TMEM (512 columns: O_A, O_B, S_A, S_B). The softmax keeps a stale row maximum and rescales O
// only when the maximum grows by more than 2^8, so P stays <= 256 and rescales are rare.
//
// Synchronisation is by mbarriers only: producers -> MMA (q_full, k_full, v_full), MMA ->
// producers (q_empty, kv_empty via tcgen05.commit), MMA -> softmax (s_full, o_done), softmax
// -> MMA (p_full, o_empty). Work items come from the plan's list through a two-slot ring
// filled by one producer thread (atomic work stealing). Every wait is bounded; after a
// timeout the CTA raises a shared abort flag, every role leaves its loop, the MMAs in flight
// are retired and TMEM is freed.
//
// Sources: the live-tile intervals and the mask are those of "[Kernel][Gemma4] Prune Triton
// sliding-window tiles for multimodal prefixes" (实现拆解 2, 关键源码片段) and "[Kernel] Skip
// fully masked key blocks in windowed Triton prefill" (功能与动机); the per-token paged gather
// follows the PR #54194 report (功能与动机); the row packing BLOCK_M = BLOCK_Q x
// num_queries_per_kv is the unified-attention layout of PR #53147 (关键源码片段).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "ppa_internal.cuh"
#include "ppa_kernels.h"
#include "ppa_ptx.cuh"

namespace ppa {

template <int D, bool FP8 = false>
struct WsCfg {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128 (256 runs on CTA pairs)");
  static constexpr int M = kRowsPerTile;  // rows per query tile
  // Two query tiles share each 128-key tile (S_A, S_B, O_A, O_B fill TMEM).
  static constexpr int NQ = 2;    // query tiles per unit
  static constexpr int TN = 128;  // keys per key tile
  static constexpr int NSB = 1;   // S buffers per query tile
  static constexpr int NSK = D == 64 ? 4 : 2;  // K stages
  static constexpr int NSV = NSK;              // V stages
  static constexpr int CPR = D / 8;       // 16-byte chunks per bf16 row
  static constexpr int Q_BYTES = M * D * 2;
  static constexpr int KV_BYTES = TN * D * 2;
  static constexpr int Q_OFF = 0;
  // K stage s at KV_OFF + s*STAGE_STRIDE, V stage s at V_OFF + s*STAGE_STRIDE (interleaved)
  static constexpr int KV_OFF = Q_OFF + NQ * Q_BYTES;
  static constexpr int STAGE_STRIDE = 2 * KV_BYTES;
  static constexpr int V_OFF = KV_OFF + KV_BYTES;
  // fp8 caches: per producer warp, a staging area for its 64 rows of raw e4m3 bytes (only
  // the fp8 instantiation reserves it; every other offset is the same in both)
  static constexpr int STG_OFF = KV_OFF + (NSK + NSV) * KV_BYTES;
  static constexpr int STG_ROWS = TN / 2;  // rows per producer warp
  static constexpr int STG_BYTES = FP8 ? 4 * STG_ROWS * D : 0;
  static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM_BYTES = BAR_OFF + BAR_BYTES + 1024;  // + alignment slack
  static constexpr int TM_O = 0;       // O_i at column TM_O + i*D
  static constexpr int TM_S = NQ * D;  // S buffer (i, b) at TM_S + (i*NSB + b)*TN; P over its first TN/2
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 512;
  static_assert(TM_S + NQ * NSB * TN <= TMEM_COLS, "TMEM");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  // The barrier block holds four full and four empty barriers per stream (K_FULL, V_FULL,
  // K_EMPTY and V_EMPTY, 8 bytes each): more stages would overlap the next array.
  static_assert(NSK <= 4 && NSV <= 4, "stages per stream: at most the four barriers of each");
  static_assert(NQ == tiles_per_unit(D), "plan and kernel agree on query tiles per unit");
  static_assert(TN == keys_per_tile(D), "plan and kernel agree on the key tile");
};

// Barrier and slot offsets inside the barrier block.
namespace wsbar {
constexpr int ITEM_FULL = 0, ITEM_EMPTY = 16, Q_FULL = 32, Q_EMPTY = 40, K_FULL = 48,
              V_FULL = 80, K_EMPTY = 112, S_FULL = 144, P_FULL = 160, O_DONE = 176,
              O_EMPTY = 192, FIN = 208, TMEM_SLOT = 216, ABORT = 220, RING = 224,
              V_EMPTY = 240, FOLD = 288,  // FOLD: fp8 scale constants, see Fp8Fold
              LIMIT = 304,  // u64: ns before a wait gives up (read only once a wait is slow)
              STG_FULL = 312;  // [4] fp8: a producer warp's staging boxes landed
constexpr int kRingConsumers = 14;  // warps 0..13 each release a ring slot once
}  // namespace wsbar

struct WsShared {
  uint32_t bars;  // shared address of the barrier block
  volatile int* abort;
  volatile int* ring;
  int32_t* status;
  __device__ uint32_t bar(int off) const { return bars + off; }
  // The wait limit, kept in shared memory rather than in every role's registers.
  __device__ unsigned long long limit() const {
    unsigned long long v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(bars + wsbar::LIMIT));
    return v;
  }
  // Bounded wait; false if the CTA is aborting (this or another role timed out).
  __device__ bool wait(int off, uint32_t parity) const {
    const uint32_t b = bars + off;
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait(b, parity)) return true;
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit()) {
        *abort = 1;
        report(status, PPA_ERR_TIMEOUT);
        return false;
      }
    }
  }
  // Bounded wait that ignores the abort flag: used after an abort, for copies this thread
  // issued that must land before the CTA exits. False if it gave up.
  __device__ bool drain(int off, uint32_t parity) const {
    const uint32_t b = bars + off;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(b, parity))
      if (globaltimer_ns() - t0 > limit()) return false;
    return true;
  }
};

// Bounded wait by a whole warp with a warp-uniform outcome (a lane that gives up makes every
// lane give up, so the warp never splits around later warp-collective operations).
__device__ __forceinline__ bool wait_warp(const WsShared& sh, int off, uint32_t parity) {
  const bool ok = sh.wait(off, parity);
  return __all_sync(0xffffffffu, ok);
}

// Consumer side of the item ring (whole warp): the k-th item of this CTA, or -1 at the end.
__device__ __forceinline__ int ring_get(const WsShared& sh, int k) {
  const int slot = k & 1;
  int item = -1;
  if (sh.wait(wsbar::ITEM_FULL + 8 * slot, (k >> 1) & 1)) item = sh.ring[slot];
  item = __shfl_sync(0xffffffffu, item, 0);  // one outcome for the whole warp
  if ((threadIdx.x & 31) == 0) mbar_arrive(sh.bar(wsbar::ITEM_EMPTY + 8 * slot));
  return item;
}

// Single-thread consumer (the MMA issuer): same protocol without the warp.
__device__ __forceinline__ int ring_get1(const WsShared& sh, int k) {
  const int slot = k & 1;
  int item = -1;
  if (sh.wait(wsbar::ITEM_FULL + 8 * slot, (k >> 1) & 1)) item = sh.ring[slot];
  mbar_arrive(sh.bar(wsbar::ITEM_EMPTY + 8 * slot));
  return item;
}

// Producer side (one thread): fetch the next item and publish it in slot k & 1. Returns the
// item (-1: none left).
__device__ __forceinline__ int ring_put(const WsShared& sh, const AttnParams& p, int k,
                                        int n_items) {
  const int slot = k & 1;
  int item = -1;
  if (sh.wait(wsbar::ITEM_EMPTY + 8 * slot, ((k >> 1) & 1) ^ 1)) {
    item = atomicAdd(&p.ws->next_item, 1);
    if (item >= n_items) item = -1;
  }
  sh.ring[slot] = item;
  mbar_arrive(sh.bar(wsbar::ITEM_FULL + 8 * slot));
  return item;
}

struct UnitInfo {
  int b, g, t0, nt, c, n, s, q_start, lo, hi;
  int cs;  // key positions below cs come from the cache: c, or s when K/V are in the cache
  int part;  // split-KV segment: partial-result slot, -1 when the unit writes the output
  int koff;  // key tile kt holds keys [kt * TN - koff, kt * TN - koff + TN)
  int lo_i[2], hi_i[2];
};

__device__ __forceinline__ UnitInfo decode_item(const AttnParams& p, int item) {
  UnitInfo u;
  const int packed = p.items[item];
  const Unit un = p.units[packed / p.num_kv_heads];
  u.g = packed % p.num_kv_heads;
  u.b = un.seq;
  u.t0 = un.t0;
  u.nt = un.nt;
  u.c = p.context_lens[u.b];
  u.q_start = p.cu_query_lens[u.b];
  u.n = p.cu_query_lens[u.b + 1] - u.q_start;
  u.s = u.c + u.n;
  u.cs = p.kv_in_cache ? u.s : u.c;
  u.part = un.part;
  u.koff = un.koff;
  u.lo_i[0] = un.lo0;
  u.hi_i[0] = un.hi0;
  u.lo_i[1] = un.nt > 1 ? un.lo1 : 0;
  u.hi_i[1] = un.nt > 1 ? un.hi1 : 0;
  u.lo = un.nt > 1 ? min(un.lo0, un.lo1) : un.lo0;
  u.hi = un.nt > 1 ? max(un.hi0, un.hi1) : un.hi0;
  return u;
}

// The allowed key interval of row j (query position c + j) of unit u: with multimodal ranges
// it comes from the per-token table the plan stage wrote (one load instead of a scan over
// every range); otherwise from the closed form. Padding rows (not valid) attend everywhere.
__device__ __forceinline__ void row_bounds_of(const AttnParams& p, const UnitInfo& u, int j,
                                              bool valid, int& kmin, int& kmax) {
  kmin = 0;
  kmax = u.s - 1;
  if (!valid) return;
  if (p.row_bounds != nullptr) {
    const int2 kb = *reinterpret_cast<const int2*>(p.row_bounds + 2 * (size_t)(u.q_start + j));
    kmin = kb.x;
    kmax = kb.y;
  } else {
    row_interval(u.c + j, u.s, seq_mask(p.mask, u.b), nullptr, kmin, kmax);
  }
}

__device__ __forceinline__ uint32_t swz128(int row, int ch, int rows) {
  return static_cast<uint32_t>((ch >> 3) * rows * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------------------
// Producer role (warps 8-11).
//
// Q (the Q loader, warp 13): one TMA box per 64-column block; the box {64 columns, G heads,
// tq tokens} lands as token-major rows, exactly the MMA's A operand.
// K/V: warps 0-1 stream K and warps 2-3 stream V, each owning half of every key tile, with
// separate empty barriers: a K slot frees as soon as the S MMAs that read it are issued, a V
// slot after its PV, so K runs up to two tiles ahead of V. A chunk of 16 keys that are cached
// context in one page, or are all new tokens, is one TMA box per 64-column block from the
// cache or the k_new/v_new tensor (rows past the sequence read the next sequence's tokens or
// the zero fill beyond the tensor: finite values that the mask removes); two such chunks that
// are contiguous in their source are one 32-row box. Any other chunk (it
// straddles the context end or a page boundary; the page id is out of range; the cache is fp8
// and must be widened) is gathered row by row with cp.async, as the PR #54194 report describes
// for per-token offsets. Each warp then arrives once on k_full / v_full with the byte count of
// its boxes.
// ---------------------------------------------------------------------------------------

// Where an fp8 cache's dequantisation scales are applied. With `fold` (the usual case) a
// producer widens a cache row to bf16(decode(code)) * 2^-112 (exact, e4m3x2_to_bf16x2_m112)
// and the softmax applies the scales: on a key tile made only of cache rows the K scale joins
// the row's exp2 multiplier and the V scale joins the exp2 argument as log2(v_scale * 2^112),
// so P carries it into PV. A tile that also holds new tokens is widened with its scales, as
// without folding, so the softmax only tells cache-only tiles from the rest. The bounds keep
// every intermediate finite: scale_log2 * k_scale
// * 2^112 and P * v_scale * 2^112 (P <= 2^8) stay below 2^127. Other scales (non-positive,
// NaN, or too large) are applied by the producer, which then writes bf16(decode * scale).
struct Fp8Fold {
  bool fold;
  float ks;      // k_scale * 2^112: data-domain S -> logit
  float lv;      // log2(v_scale * 2^112)
  float inv_vs;  // 1 / (v_scale * 2^112)
};

__device__ __forceinline__ Fp8Fold fp8_fold(const AttnParams& p) {
  const float k = *p.k_scale, v = *p.v_scale;
  Fp8Fold f;
  f.fold = k > 0.f && v > 0.f && v < 0x1p7f && k < 0x1p15f && k * p.scale_log2 < 0x1p15f;
  f.ks = k * 0x1p112f;
  f.lv = log2f(v) + 112.f;
  f.inv_vs = 1.f / (v * 0x1p112f);
  return f;
}

// Position of 16-byte piece `un` of staging row `row` (rows of D e4m3 codes). It is the layout
// a TMA box lands in with the 128-byte swizzle (D 128: piece ^ row % 8) or the 64-byte one
// (D 64: piece ^ (row / 2) % 4), so cp.async gathers and TMA boxes fill one staging area, and
// the widening, which reads piece un of 32 rows at once, stays free of bank conflicts.
template <int D>
__device__ __forceinline__ int stg_piece(int un, int row) {
  static_assert(D == 64 || D == 128, "staged e4m3 rows of 64 or 128 bytes");
  return D == 128 ? ((un ^ row) & 7) : ((un ^ (row >> 1)) & 3);
}

// fp8 cache, first half of a 32-row block's gather (one row per lane): the lane copies its
// row's raw e4m3 bytes (rows below `cache_rows`) into its staging row with cp.async, or its
// bf16 new-token row straight into the stage. No registers hold the data, so all rows of the
// warp are in flight at once; fp8_stage_widen() finishes the cache rows.
template <int D>
__device__ __forceinline__ void fp8_stage_issue(const char* zero_src, int row0, uint32_t rowmask,
                                                int cache_rows, const char* mine, uint32_t sX,
                                                int rows, uint32_t stg_row) {
  const int lane = threadIdx.x & 31;
  if (!((rowmask >> lane) & 1u)) return;
  if (lane < cache_rows) {
#pragma unroll
    for (int un = 0; un < D / 16; ++un)
      cp_async_16(stg_row + stg_piece<D>(un, lane) * 16, mine ? mine + un * 16 : zero_src,
                  mine ? 16u : 0u);
  } else {
#pragma unroll
    for (int ch = 0; ch < D / 8; ++ch)
      cp_async_16(sX + swz128(row0 + lane, ch, rows), mine ? mine + ch * 16 : zero_src,
                  mine ? 16u : 0u);
  }
}

// Second half: widen the lane's staged e4m3 row to bf16 into the 128-byte-swizzled stage:
// bf16(decode(code)) * 2^-112 when the softmax applies the scales (FOLD), else
// bf16(decode(code) * scale), the fp32 product rounded once.
template <int D, bool FOLD>
__device__ __forceinline__ void fp8_stage_widen(int row0, uint32_t rowmask, int cache_rows,
                                                uint32_t sX, int rows, uint32_t stg_row,
                                                float scale) {
  const int lane = threadIdx.x & 31;
  if (!((rowmask >> lane) & 1u) || lane >= cache_rows) return;
  const int row = row0 + lane;
#pragma unroll
  for (int un = 0; un < D / 16; ++un) {
    const uint4 codes = ld_shared_v4(stg_row + stg_piece<D>(un, lane) * 16);
    const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t v[8];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const uint16_t c0 = static_cast<uint16_t>(cw[q4] & 0xFFFFu);
      const uint16_t c1 = static_cast<uint16_t>(cw[q4] >> 16);
      v[2 * q4] = FOLD ? e4m3x2_to_bf16x2_m112(c0) : e4m3x2_to_bf16x2_scaled(c0, scale);
      v[2 * q4 + 1] = FOLD ? e4m3x2_to_bf16x2_m112(c1) : e4m3x2_to_bf16x2_scaled(c1, scale);
    }
    st_shared_v4(sX + swz128(row, 2 * un, rows), v[0], v[1], v[2], v[3]);
    st_shared_v4(sX + swz128(row, 2 * un + 1, rows), v[4], v[5], v[6], v[7]);
  }
}

// Gather of one 32-row block with an fp8 cache, one row per lane: lane r sources row
// row0 + r (if its bit is set in `rowmask`) from `mine` (nullptr: zero fill). Rows below
// `cache_rows` are fp8 cache rows of COLS codes: the lane issues all its 16-byte loads first,
// so their latency overlaps, then widens them to bf16. Later rows are bf16 new tokens, copied
// with cp.async. `rows` is the number of rows per 64-column block of the destination.
template <int COLS>
__device__ __forceinline__ void gather_rows_fp8(const char* zero_src, int row0, uint32_t rowmask,
                                                int cache_rows, const char* mine, uint32_t sX,
                                                int rows, float scale) {
  const int lane = threadIdx.x & 31;
  if (!((rowmask >> lane) & 1u)) return;
  const int row = row0 + lane;
  if (lane < cache_rows) {
    uint4 codes[COLS / 16];
#pragma unroll
    for (int un = 0; un < COLS / 16; ++un)
      codes[un] = mine ? ld_global_nc_v4(mine + un * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int un = 0; un < COLS / 16; ++un) {
      const uint32_t cw[4] = {codes[un].x, codes[un].y, codes[un].z, codes[un].w};
      uint32_t v[8];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        v[2 * q4] = e4m3x2_to_bf16x2_scaled(static_cast<uint16_t>(cw[q4] & 0xFFFFu), scale);
        v[2 * q4 + 1] = e4m3x2_to_bf16x2_scaled(static_cast<uint16_t>(cw[q4] >> 16), scale);
      }
      st_shared_v4(sX + swz128(row, 2 * un, rows), v[0], v[1], v[2], v[3]);
      st_shared_v4(sX + swz128(row, 2 * un + 1, rows), v[4], v[5], v[6], v[7]);
    }
  } else {
#pragma unroll
    for (int ch = 0; ch < COLS / 8; ++ch)
      cp_async_16(sX + swz128(row, ch, rows), mine ? mine + ch * 16 : zero_src, mine ? 16u : 0u);
  }
}

// Row-wise gather (bf16 cache) of rows row0 .. row0+nrows-1 whose bit is set in `rowmask`;
// `mine` is the source row of lane `lane` (lanes >= nrows unused), nullptr for zero fill.
template <int D>
__device__ __forceinline__ void gather_rows(const AttnParams& p, int row0, int nrows,
                                            uint32_t rowmask, const char* mine, uint32_t sX) {
  using C = WsCfg<D>;
  const int lane = threadIdx.x & 31;
  constexpr int RPI = 32 / C::CPR;  // rows per warp instruction
  for (int it = 0; it * RPI < nrows; ++it) {
    const int lr = it * RPI + lane / C::CPR;
    const int ch = lane % C::CPR;
    const char* rp = reinterpret_cast<const char*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine), lr & 31));
    if (lr < nrows && ((rowmask >> lr) & 1u))
      cp_async_16(sX + swz128(row0 + lr, ch, C::TN),
                  rp ? rp + ch * 16 : static_cast<const char*>(p.k_cache), rp ? 16u : 0u);
  }
}

template <int D, bool FP8>
__device__ void ws_producer(const AttnParams& p, const WsShared& sh, uint32_t base, int n_items) {
  using C = WsCfg<D>;
  constexpr int RPW = C::TN / 2;   // key rows per producer warp (two warps per stream)
  constexpr int NSUB = RPW / 32;   // 32-row blocks per warp
  constexpr uint32_t kChunkBytes = 16 * 128;  // one 64-column block of 16 rows
  constexpr size_t kCacheElt = FP8 ? 1 : 2;
  const int lane = threadIdx.x & 31;
  const int pw = (threadIdx.x >> 5) - 8;  // 0..3
  const int w = pw >> 1;                  // 0: the K stream, 1: the V stream
  const int half = pw & 1;
  const void* tm_new = w == 0 ? (const void*)&p.tm.k_new : (const void*)&p.tm.v_new;
  const void* tm_cache = w == 0 ? (const void*)&p.tm.k_cache : (const void*)&p.tm.v_cache;
  const void* tm_new32 = w == 0 ? (const void*)&p.tm.k_new32 : (const void*)&p.tm.v_new32;
  const void* tm_cache32 = w == 0 ? (const void*)&p.tm.k_cache32 : (const void*)&p.tm.v_cache32;
  // fp8: the cache as e4m3 bytes, boxes of 16 rows into this warp's staging area
  const void* tm_cache8 = w == 0 ? (const void*)&p.tm.k_cache8 : (const void*)&p.tm.v_cache8;
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
    } else {
      tma_prefetch_desc(tm_cache8);
    }
  }
  const int empty_bar = w == 0 ? wsbar::K_EMPTY : wsbar::V_EMPTY;
  const int full_bar = w == 0 ? wsbar::K_FULL : wsbar::V_FULL;
  const float kv_scale = FP8 ? *(w == 0 ? p.k_scale : p.v_scale) : 1.f;  // fp8 dequantisation
  const bool kv_fold = FP8 && fp8_fold(p).fold;
  uint32_t kv_iter = 0;
  bool stg_pending = false;  // fp8: staging boxes of the current tile not yet seen landed
  for (int k = 0;; ++k) {
    const int item = ring_get(sh, k);
    if (item < 0) break;
    const UnitInfo u = decode_item(p, item);

    // ---- this warp's rows of the K (or V) tiles of the union interval ----
    bool ok = true;
    for (int kt = u.lo; kt < u.hi; ++kt, ++kv_iter) {
      const int ns = C::NSK == C::NSV ? C::NSK : (w == 0 ? C::NSK : C::NSV);
      const int s = kv_iter % ns;
      const uint32_t ph = (kv_iter / ns) & 1;
      // Classify this warp's 16-row chunks before waiting for the stage, so that the
      // block-table loads overlap the wait. Lane c < RPW/16 takes chunk c.
      int ctype = 0, crow = 0;  // 1 = cache box, 2 = new-token box, 0 = row gather
      if (lane * 16 < RPW) {
        const int p0 = kt * C::TN - u.koff + half * RPW + 16 * lane;
        if (p0 >= u.cs) {
          if (!p.kv_in_cache) {  // new tokens (cache-sourced: past the sequence, zero fill)
            ctype = 2;
            crow = u.q_start + p0 - u.c;
          }
        } else if (p0 >= 0 && p0 + 15 < u.cs) {  // (chunks below key 0: zero fill)
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
      if (!wait_warp(sh, empty_bar + 8 * s, ph ^ 1)) { ok = false; break; }
      const uint32_t sX = base + (w == 0 ? C::KV_OFF : C::V_OFF) + s * C::STAGE_STRIDE;
      const uint32_t bar = sh.bar(full_bar + 8 * s);
      uint32_t bytes = 0, stg_bytes = 0;
      bool any_fallback = false;
      uint32_t fp8_mask[NSUB];  // fp8: rows of each 32-row block still to widen
      int fp8_cache_rows[NSUB];
      const uint32_t stg = base + C::STG_OFF + pw * (C::STG_ROWS * D);  // this warp's staging
      const uint32_t stg_bar = sh.bar(wsbar::STG_FULL + 8 * pw);
#pragma unroll
      for (int sub = 0; sub < NSUB; ++sub) {
        fp8_mask[sub] = 0;
        fp8_cache_rows[sub] = 0;
        const int row0 = half * RPW + 32 * sub;
        const int p_row0 = kt * C::TN - u.koff + row0;  // key position of the block's first row
        int types[2], rows[2];
        uint32_t fb_mask = 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          types[c] = __shfl_sync(0xffffffffu, ctype, 2 * sub + c);
          rows[c] = __shfl_sync(0xffffffffu, crow, 2 * sub + c);
          if (types[c] == 0) fb_mask |= 0xFFFFu << (16 * c);
        }
        // both chunks from one contiguous source run: one 32-row box per column block (fp8
        // cache chunks go to the staging area in boxes of their own instead)
        const bool one_run = types[0] != 0 && types[0] == types[1] && rows[1] == rows[0] + 16 &&
                             (!FP8 || types[0] == 2);
        if (lane == 0 && one_run) {
          const void* tm32 = types[0] == 1 ? tm_cache32 : tm_new32;
#pragma unroll
          for (int db = 0; db < D / 64; ++db)
            tma_load_3d(sX + db * (C::TN * 128) + row0 * 128, tm32, db * 64, u.g, rows[0], bar);
          bytes += (D / 64) * 2 * kChunkBytes;
        }
        if (lane == 0 && !one_run) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (types[c] == 0) continue;
            if (FP8 && types[c] == 1) {  // e4m3 rows into the staging, widened below
              tma_load_3d(stg + (32 * sub + 16 * c) * D, tm_cache8, 0, u.g, rows[c], stg_bar);
              stg_bytes += 16 * D;
              continue;
            }
#pragma unroll
            for (int db = 0; db < D / 64; ++db)
              tma_load_3d(sX + db * (C::TN * 128) + (row0 + 16 * c) * 128,
                          types[c] == 1 ? tm_cache : tm_new, db * 64, u.g, rows[c], bar);
            bytes += (D / 64) * kChunkBytes;
          }
        }
        if constexpr (FP8) {  // the boxed cache rows are widened like the gathered ones
          for (int c = 0; c < 2; ++c)
            if (types[c] == 1) fp8_mask[sub] |= 0xFFFFu << (16 * c);
          fp8_cache_rows[sub] = u.cs - p_row0;
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
                     (((size_t)page * p.page_size + (pos - lp * p.page_size)) * p.num_kv_heads +
                      u.g) * D * kCacheElt;
            } else {
              report(p.status, PPA_ERR_BAD_PAGE);
            }
          } else if (pos < u.s) {
            mine = g_new + ((size_t)(u.q_start + pos - u.c) * p.num_kv_heads + u.g) * D * 2;
          }
          if constexpr (FP8) {
            fp8_stage_issue<D>(g_cache, row0, fb_mask, u.cs - p_row0, mine,
                               sX, C::TN, stg + (32 * sub + lane) * D);
            fp8_mask[sub] |= fb_mask;
          } else {
            gather_rows<D>(p, row0, 32, fb_mask, mine, sX);
          }
          any_fallback = true;
        }
      }
      if constexpr (FP8) {
        // every staged row has landed: the boxes (this warp's staging barrier, one phase per
        // key tile) and the gathers
        cp_async_commit();
        if (lane == 0) mbar_arrive_expect_tx(stg_bar, stg_bytes);
        stg_pending = true;
        if (!wait_warp(sh, wsbar::STG_FULL + 8 * pw, kv_iter & 1)) { ok = false; break; }
        stg_pending = false;
        cp_async_wait<0>();
        any_fallback = true;  // the widened rows are generic-proxy writes
#pragma unroll
        for (int sub = 0; sub < NSUB; ++sub) {
          if (fp8_mask[sub] != 0) {
            if (kv_fold && u.cs >= (kt + 1) * C::TN - u.koff)  // cache-only: the softmax scales
              fp8_stage_widen<D, true>(half * RPW + 32 * sub, fp8_mask[sub], fp8_cache_rows[sub],
                                       sX, C::TN, stg + (32 * sub + lane) * D, kv_scale);
            else
              fp8_stage_widen<D, false>(half * RPW + 32 * sub, fp8_mask[sub], fp8_cache_rows[sub],
                                        sX, C::TN, stg + (32 * sub + lane) * D, kv_scale);
          }
        }
        if (any_fallback) {
          fence_proxy_async_smem();
          __syncwarp();
        }
      } else if (any_fallback) {
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
  // staging boxes of a tile cut short by an abort (its phase: the current tile's)
  if (FP8 && stg_pending && lane == 0) sh.drain(wsbar::STG_FULL + 8 * pw, kv_iter & 1);
  // This warp's TMA copies must land before the CTA exits: wait for the last fill of every
  // stage. After a normal end those fills are complete or complete shortly. After an abort a
  // fill whose other half was never issued cannot complete, and the wait gives up at the limit,
  // long after the copies themselves have landed.
  if (lane == 0) {
    constexpr uint32_t ns = C::NSK;
    static_assert(C::NSK == C::NSV, "one stage count for K and V");
    for (uint32_t s = 0; s < ns && s < kv_iter; ++s) {
      const uint32_t f = s + ns * ((kv_iter - 1 - s) / ns);  // last fill of stage s
      sh.drain(full_bar + 8 * s, (f / ns) & 1);
    }
  }
}

// Q loader (warp 13): runs the item ring and loads each unit's query tiles, so that the K
// and V streams never wait for Q_EMPTY at a unit boundary and prefetch across units.
template <int D>
__device__ void ws_qloader(const AttnParams& p, const WsShared& sh, uint32_t base, int n_items) {
  using C = WsCfg<D>;
  const int lane = threadIdx.x & 31;
  if (lane == 0) tma_prefetch_desc(&p.tm.q);
  uint32_t q_phase = 0;
  bool loaded = false;
  for (int k = 0;; ++k) {
    if (lane == 0) ring_put(sh, p, k, n_items);
    const int item = ring_get(sh, k);
    if (item < 0) break;
    // Testing the bounded waits: the CTA that took the plan's first item neither loads its
    // queries nor feeds its ring any further, so the waits for them run out.
    if (p.debug_stall && item == 0) break;
    const UnitInfo u = decode_item(p, item);
    if (!wait_warp(sh, wsbar::Q_EMPTY, q_phase ^ 1)) break;
    q_phase ^= 1;
    loaded = true;
    if (lane == 0) {
      const uint32_t box_bytes = static_cast<uint32_t>(p.group * p.tq * 128);
      mbar_arrive_expect_tx(sh.bar(wsbar::Q_FULL), u.nt * (D / 64) * box_bytes);
      for (int i = 0; i < u.nt; ++i) {
#pragma unroll
        for (int db = 0; db < D / 64; ++db)
          tma_load_3d(base + C::Q_OFF + i * C::Q_BYTES + db * (C::M * 128), &p.tm.q, db * 64,
                      u.g * p.group, u.q_start + (u.t0 + i) * p.tq, sh.bar(wsbar::Q_FULL));
      }
    }
  }
  // The last query load must land before the CTA exits (after an abort it may still be in
  // flight): its phase of Q_FULL is the one before q_phase.
  if (loaded && lane == 0) sh.drain(wsbar::Q_FULL, q_phase ^ 1);
}

// The tile intervals of a unit: the part of its decoding that the MMA issuer needs.
struct UnitTiles {
  int nt, lo, hi, lo_i[2], hi_i[2];
};

__device__ __forceinline__ UnitTiles unit_tiles(const Unit& un) {
  UnitTiles t;
  t.nt = un.nt;
  t.lo_i[0] = un.lo0;
  t.hi_i[0] = un.hi0;
  t.lo_i[1] = un.nt > 1 ? un.lo1 : 0;
  t.hi_i[1] = un.nt > 1 ? un.hi1 : 0;
  t.lo = un.nt > 1 ? min(un.lo0, un.lo1) : un.lo0;
  t.hi = un.nt > 1 ? max(un.hi0, un.hi1) : un.hi0;
  return t;
}

// ---------------------------------------------------------------------------------------
// MMA role (warp 12; lane 0 issues).
// ---------------------------------------------------------------------------------------
template <int D>
__device__ void ws_mma(const AttnParams& p, const WsShared& sh, uint32_t base, uint32_t tmem) {
  using C = WsCfg<D>;
  if ((threadIdx.x & 31) != 0) return;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::TN, false, false);
  constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);
  // Descriptors are built once; a K-step adds a compile-time offset (in 16-byte units) to the
  // 14-bit start-address field, which cannot carry because shared addresses stay below 256 KB.
  const uint64_t dQ0 = sdesc_sw128(base + C::Q_OFF, 16, 1024);
  const uint64_t dK0 = sdesc_sw128(base + C::KV_OFF, 16, 1024);
  const uint64_t dV0 = sdesc_sw128(base + C::V_OFF, C::TN * 128, 1024);
  constexpr uint32_t kQStep = C::Q_BYTES >> 4, kStageStep = C::STAGE_STRIDE >> 4;
  static_assert(C::NSK == C::NSV, "two-tile units use one ring position for K and V");
  constexpr int NS = C::NSK;
  // Per-tile phases as bit i of one word, and the tile intervals read through selects: a
  // runtime index into a small array would put it in local memory, on this thread's
  // critical path between MMA batches.
  uint32_t kv_iter = 0, q_phase = 0, pf_bits = 0, oe_bits = 0;
  bool ok = true;
  // The k-th item and its unit. The next one is taken once a unit's first S are issued (the
  // issuer then waits for their softmax anyway), so its dependent loads are done when the
  // unit ends and the next unit's first S follow its last PV without a gap.
  int item = ring_get1(sh, 0);
  Unit un_next{};
  if (item >= 0) un_next = p.units[p.items[item] / p.num_kv_heads];
  for (int k = 0; ok && item >= 0; ++k) {
    const UnitTiles u = unit_tiles(un_next);
    bool fetched = false;
    auto fetch_next = [&]() {
      item = ring_get1(sh, k + 1);
      if (item >= 0) un_next = p.units[p.items[item] / p.num_kv_heads];
      fetched = true;
    };
    const int lo0 = u.lo_i[0], hi0 = u.hi_i[0], lo1 = u.lo_i[1], hi1 = u.hi_i[1];
    uint32_t early = 0;  // tiles whose first S was issued ahead of their first key tile
    if (!sh.wait(wsbar::Q_FULL, q_phase)) break;
    q_phase ^= 1;
    tc_fence_after();
    auto issue_s = [&](int i, int stage) {
      const uint32_t tS = tmem + C::TM_S + i * C::TN;
      uint64_t a0 = dQ0 + i * kQStep, b0 = dK0 + stage * kStageStep;
      // Opaque to the compiler: otherwise it hoists every per-MMA descriptor of the
      // unrolled batches out of the loop into registers and spills them to local memory.
      asm volatile("" : "+l"(a0), "+l"(b0));
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off_a = ((kk >> 2) * (C::M * 128) + (kk & 3) * 32) >> 4;
        const uint32_t off_b = ((kk >> 2) * (C::TN * 128) + (kk & 3) * 32) >> 4;
        mma_bf16_ss(tS, a0 + off_a, b0 + off_b, kIdescS, kk > 0 ? 1u : 0u);
      }
      tc_commit(sh.bar(wsbar::S_FULL + 8 * i));
    };
    // Steady state: both tiles past their first key tile and with a next one. Straight-line
    // code whose only taken branch is the back edge: this thread competes for the
    // instruction cache with the softmax warps' long bodies, and every taken branch into an
    // evicted line stalls it while the tensor pipe, which queues about one MMA, runs dry.
    const int steady_lo = u.nt == 2 ? max(lo0, lo1) + 1 : INT_MAX;
    const int steady_hi = u.nt == 2 ? min(hi0, hi1) - 1 : INT_MIN;
    auto issue_pv = [&](int i, int stage, uint32_t acc0) {
      const uint32_t tP = tmem + C::TM_S + i * C::TN;
      const uint32_t tO = tmem + C::TM_O + i * D;
      uint64_t b0 = dV0 + stage * kStageStep;
      asm volatile("" : "+l"(b0));
#pragma unroll
      for (int kk = 0; kk < C::TN / 16; ++kk)
        mma_bf16_ts(tO, tP + kk * 8, b0 + ((kk * 16 * 128) >> 4), kIdescO, kk > 0 ? 1u : acc0);
    };
    for (int kt = u.lo; kt < u.hi && ok;) {
      if (kt >= steady_lo && kt < steady_hi) {
        for (; kt < steady_hi; ++kt, ++kv_iter) {
          const int s = kv_iter % NS, s1 = (kv_iter + 1) % NS;
          tc_commit(sh.bar(wsbar::K_EMPTY + 8 * s));  // both S(kt) were issued last iteration
          if (!sh.wait(wsbar::P_FULL, pf_bits & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(0, s, 1u);
          issue_s(0, s1);
          if (!sh.wait(wsbar::P_FULL + 8, (pf_bits >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          pf_bits ^= 3u;
          issue_pv(1, s, 1u);
          tc_commit(sh.bar(wsbar::V_EMPTY + 8 * s));
          issue_s(1, s1);
        }
        continue;
      }
      const int s = kv_iter % NS;
      const uint32_t ph = (kv_iter / NS) & 1;
      // first key tile of a query tile: its S (the one S whose K the issuer waits for)
      for (int i = 0; i < u.nt && ok; ++i) {
        if (kt != (i ? lo1 : lo0) || ((early >> i) & 1u)) continue;
        if (!sh.wait(wsbar::K_FULL + 8 * s, ph)) { ok = false; break; }
        tc_fence_after();
        issue_s(i, s);
      }
      // A tile whose interval starts one key tile later (a window or range edge between the
      // two query tiles): issue its first S now, so that its softmax overlaps the other tile's
      // first one instead of following it.
      if (kt == u.lo && u.nt == 2 && ok) {
        for (int i = 0; i < 2 && ok; ++i) {
          if ((i ? lo1 : lo0) != kt + 1) continue;
          const uint32_t kv1 = kv_iter + 1;
          if (!sh.wait(wsbar::K_FULL + 8 * (kv1 % NS), (kv1 / NS) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_s(i, kv1 % NS);
          early |= 1u << i;
        }
      }
      // every S that reads K(kt) has now been issued (in this or the previous iteration)
      tc_commit(sh.bar(wsbar::K_EMPTY + 8 * s));
      if (!fetched) fetch_next();
      // At the unit's last key tile every S has been issued: Q is free once they complete,
      // so the next unit's Q loads while this unit's last PVs and softmax run.
      if (kt == u.hi - 1) tc_commit(sh.bar(wsbar::Q_EMPTY));
      for (int i = 0; i < u.nt && ok; ++i) {
        const int lo_i = i ? lo1 : lo0, hi_i = i ? hi1 : hi0;
        if (kt < lo_i || kt >= hi_i) continue;
        if (kt == lo_i) {  // O_i must have been read out by the previous epilogue
          if (!sh.wait(wsbar::O_EMPTY + 8 * i, ((oe_bits >> i) & 1) ^ 1)) { ok = false; break; }
          oe_bits ^= 1u << i;
        }
        // P_i(kt) also certifies V(kt) and, unless this is the tile's last key tile,
        // K(kt+1): the softmax warps waited for both before arriving. The issuer waits on
        // nothing else here, because each wait leaves the tensor pipe idle (its queue holds
        // about one MMA).
        if (!sh.wait(wsbar::P_FULL + 8 * i, (pf_bits >> i) & 1)) { ok = false; break; }
        pf_bits ^= 1u << i;
        tc_fence_after();
        issue_pv(i, s, kt > lo_i ? 1u : 0u);
        if (kt + 1 < hi_i) {
          issue_s(i, (kv_iter + 1) % NS);
        } else {
          tc_commit(sh.bar(wsbar::O_DONE + 8 * i));
        }
      }
      tc_commit(sh.bar(wsbar::V_EMPTY + 8 * s));
      ++kv_iter;
      ++kt;
    }
    if (ok && !fetched) fetch_next();  // (a unit without key tiles)
  }
}

// ---------------------------------------------------------------------------------------
// Softmax role (warps 0-7): warpgroup i owns query tile i; thread r owns row r.
// ---------------------------------------------------------------------------------------
// Split-KV epilogue of one row (thread `r` of a query tile): O / l as D fp32 values and the
// row's base-2 log-sum-exp over this segment's keys, m + log2(l) with m the exp2 reference the
// row's P used (-inf when none of the segment's keys is allowed), into partial slot
// u.part * Hkv + u.g. The merge kernel combines a sequence's segments.
template <int D>
__device__ __forceinline__ void split_partial_store(const AttnParams& p, const UnitInfo& u, int r,
                                                    bool row_valid, float m_ref, float l_run,
                                                    float inv_l, uint32_t tO) {
  const size_t slot = (size_t)u.part * p.num_kv_heads + u.g;
  float* orow = p.part_o + (slot * kRowsPerTile + r) * D;
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t o32[32];
    tmem_ld_32(tO + cc * 32, o32);
    if (row_valid) {
      float4* dst = reinterpret_cast<float4*>(orow + cc * 32);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        dst[e] = make_float4(__uint_as_float(o32[4 * e]) * inv_l, __uint_as_float(o32[4 * e + 1]) * inv_l,
                             __uint_as_float(o32[4 * e + 2]) * inv_l, __uint_as_float(o32[4 * e + 3]) * inv_l);
    }
  }
  if (row_valid) {
    const float neg_inf = -__int_as_float(0x7f800000);
    const float m_use = m_ref == neg_inf ? 0.f : m_ref;
    p.part_lse[slot * kRowsPerTile + r] = l_run > 0.f ? m_use + log2f(l_run) : neg_inf;
  }
}

template <int D, bool FP8, bool SPLIT>
__device__ void ws_softmax(const AttnParams& p, const WsShared& sh, uint32_t tmem) {
  using C = WsCfg<D>;
  const int warp = threadIdx.x >> 5;
  const int i = warp >> 2;
  const int r = threadIdx.x & 127;
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tO = tmem + C::TM_O + i * D + lane_off;
  const float neg_inf = -__int_as_float(0x7f800000);
  const float scale = p.scale_log2;
  // One S buffer per tile: S_FULL[i] and O_DONE[i] flip once per use.
  uint32_t sf_phase = 0, od_phase = 0;
  uint32_t kv_next = 0;  // K/V ring position of the next unit's first key tile
  for (int k = 0;; ++k) {
    const int item = ring_get(sh, k);
    if (item < 0) break;
    const UnitInfo u = decode_item(p, item);
    const uint32_t kv0 = kv_next;
    kv_next += u.hi - u.lo;
    if (i >= u.nt) continue;
    const int lo = i ? u.lo_i[1] : u.lo_i[0], hi = i ? u.hi_i[1] : u.hi_i[0];
    const int tok = r / p.group, hh = r % p.group;
    const int j = (u.t0 + i) * p.tq + tok;
    const bool row_valid = tok < p.tq && j < u.n;
    int kmin, kmax;  // padding rows attend everywhere (Q is zero: finite)
    row_bounds_of(p, u, j, row_valid, kmin, kmax);
    float m_ref = neg_inf, l_run = 0.f;
    bool ok = true;
    for (int kt = lo; kt < hi; ++kt) {
      const uint32_t tS = tmem + C::TM_S + i * C::TN + lane_off;
      const uint32_t kv = kv0 + (kt - u.lo);  // ring position of key tile kt
      const uint32_t bar_v = wsbar::V_FULL + 8 * (kv % C::NSV), par_v = (kv / C::NSV) & 1;
      const uint32_t bar_k = wsbar::K_FULL + 8 * ((kv + 1) % C::NSK);
      const uint32_t par_k = ((kv + 1) / C::NSK) & 1;
      if (!wait_warp(sh, wsbar::S_FULL + 8 * i, sf_phase)) { ok = false; break; }
      sf_phase ^= 1;
      // V(kt) and K(kt+1) must be resident before P_FULL lets the issuer start PV(kt) and
      // S(kt+1). Probe both now (non-blocking; the latency overlaps the softmax) and wait
      // before the arrival only for what was not ready. Probing after S(kt) has landed is
      // what makes the parity test unambiguous: every earlier fill of these stages that a
      // tile uses was confirmed before the issuer could issue S(kt).
      const bool v_ready = mbar_test_wait(sh.bar(bar_v), par_v);
      const bool k_ready = kt + 1 >= hi || mbar_test_wait(sh.bar(bar_k), par_k);
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
      // fp8 with folded scales: a tile of cache keys only was widened without its scales.
      // The constants come from shared memory each tile (no registers held across tiles).
      float2 fc = make_float2(0.f, 0.f);  // (scale_log2 * k_scale * 2^112, log2(v_scale * 2^112))
      if constexpr (FP8) fc = ld_shared_f2(sh.bar(wsbar::FOLD));
      const bool cache_tile = FP8 && fc.x != 0.f && u.cs - k0 >= C::TN;
      const float sc = cache_tile ? fc.x : scale;  // exp2 multiplier
      const int a0 = kmin - k0, a1 = kmax - k0;  // allowed local columns [a0, a1]
      if (!(a0 <= 0 && a1 >= C::TN - 1)) {
#pragma unroll
        for (int e = 0; e < C::TN; ++e) sv[e] = (e < a0 || e > a1) ? neg_inf : sv[e];
      }
      // row maximum: 8 independent chains of 3-input maxima over columns q, q+8, q+16, ...
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
      const float m_tile = tile_max * sc;  // in exp2 units
      // Keep the stale reference unless the maximum grew by more than 2^8.
      bool rescale = false;
      float alpha = 1.f;
      if (m_tile > m_ref + 8.f) {
        alpha = ex2_approx(m_ref - m_tile);  // 0 when m_ref = -inf
        rescale = kt > lo;
        m_ref = m_tile;
      }
      const float m_use = m_ref == neg_inf ? 0.f : m_ref;
      // p = exp2(s * sc - m): the exponent arguments and the row sums run as packed pairs. On
      // an fp8 cache-only tile the argument also carries log2(v_scale * 2^112), so P is scaled
      // for the PV MMA and its row sum is scaled back once.
      const float lv = cache_tile ? fc.y : 0.f;
      const uint64_t scale2 = f2_pack(sc, sc), negm2 = f2_pack(lv - m_use, lv - m_use);
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
      float l_tile = ((sl[0] + sl[1]) + (sl[2] + sl[3])) + ((sl[4] + sl[5]) + (sl[6] + sl[7]));
      if (cache_tile) l_tile *= ld_shared_f32(sh.bar(wsbar::FOLD + 8));  // 1 / (v_scale 2^112)
      l_run = l_run * alpha + l_tile;
      // P over the first TN/2 columns of this S buffer
#pragma unroll
      for (int cc = 0; cc < C::TN / 64; ++cc) {
        uint32_t w32[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) w32[e] = pk[cc * 32 + e];
        tmem_st_32(tS + cc * 32, w32);
      }
      // O_i is idle here: PV_i(kt-1) completed before S_i(kt) (one issuing thread, in order).
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
      if (!__all_sync(0xffffffffu, v_ready) && !wait_warp(sh, bar_v, par_v)) { ok = false; break; }
      if (!__all_sync(0xffffffffu, k_ready) && !wait_warp(sh, bar_k, par_k)) { ok = false; break; }
      tc_fence_before();
      mbar_arrive(sh.bar(wsbar::P_FULL + 8 * i));
    }
    if (!ok) break;
    // ---- epilogue: the last PV of this tile ----
    if (!wait_warp(sh, wsbar::O_DONE + 8 * i, od_phase)) break;
    od_phase ^= 1;
    tc_fence_after();
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    if constexpr (SPLIT) {  // only launches with split-KV carry this path
      if (u.part >= 0) {  // a split-KV segment: O / l in fp32 and the row's log-sum-exp
        split_partial_store<D>(p, u, r, row_valid, m_ref, l_run, inv_l, tO);
        tc_fence_before();
        mbar_arrive(sh.bar(wsbar::O_EMPTY + 8 * i));
        continue;
      }
    }
    __nv_bfloat16* orow =
        static_cast<__nv_bfloat16*>(p.out) +
        ((size_t)(u.q_start + (row_valid ? j : 0)) * p.num_q_heads + u.g * p.group + hh) * D;
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t o32[32];
      tmem_ld_32(tO + cc * 32, o32);
      if (row_valid) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(o32[2 * e]) * inv_l,
                             __uint_as_float(o32[2 * e + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    }
    tc_fence_before();
    mbar_arrive(sh.bar(wsbar::O_EMPTY + 8 * i));
  }
}

template <int D, bool FP8, bool SPLIT>
__global__ void __launch_bounds__(512, 1) attn_ws_kernel(const __grid_constant__ AttnParams p) {
  using C = WsCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint8_t* barp = smem + C::BAR_OFF;
  WsShared sh;
  sh.bars = base + C::BAR_OFF;
  sh.abort = reinterpret_cast<volatile int*>(barp + wsbar::ABORT);
  sh.ring = reinterpret_cast<volatile int*>(barp + wsbar::RING);
  sh.status = p.status;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  if (tid == 0) {
    using namespace wsbar;
    for (int s = 0; s < 2; ++s) {
      mbar_init(sh.bar(ITEM_FULL + 8 * s), 1);
      mbar_init(sh.bar(ITEM_EMPTY + 8 * s), kRingConsumers);
      mbar_init(sh.bar(S_FULL + 8 * s), 1);
      mbar_init(sh.bar(P_FULL + 8 * s), 128);
      mbar_init(sh.bar(O_DONE + 8 * s), 1);
      mbar_init(sh.bar(O_EMPTY + 8 * s), 128);
    }
    mbar_init(sh.bar(Q_FULL), 1);  // the Q loader, with the TMA byte count
    mbar_init(sh.bar(Q_EMPTY), 1);
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(sh.bar(K_FULL + 8 * s), 2);  // one arrival (with its TMA bytes) per stream warp
      mbar_init(sh.bar(K_EMPTY + 8 * s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(sh.bar(V_FULL + 8 * s), 2);
      mbar_init(sh.bar(V_EMPTY + 8 * s), 1);
    }
    mbar_init(sh.bar(FIN), 1);
    if constexpr (FP8)
      for (int w = 0; w < 4; ++w) mbar_init(sh.bar(STG_FULL + 8 * w), 1);
    *sh.abort = 0;
    *reinterpret_cast<unsigned long long*>(barp + LIMIT) = p.wait_ns;
    if constexpr (FP8) {
      const Fp8Fold f = fp8_fold(p);
      float* fc = reinterpret_cast<float*>(barp + FOLD);
      fc[0] = f.fold ? p.scale_log2 * f.ks : 0.f;  // 0: scales not folded
      fc[1] = f.lv;
      fc[2] = f.inv_vs;
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sh.bar(wsbar::TMEM_SLOT), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(barp + wsbar::TMEM_SLOT);
  const int n_items = p.ws->n_items;

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 184;\n" ::: "memory");
    ws_softmax<D, FP8, SPLIT>(p, sh, tmem);
  } else {
    // One count per warpgroup (setmaxnreg acts on whole warpgroups): the producers' (warps
    // 8-11) 56, the MMA issuer's and query loader's warpgroup (12-15) 88, so that the issuer's
    // state stays in registers. 256 x 184 + 128 x 56 + 128 x 88 = 512 x 128, the launch budget.
    if (warp < 12) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 56;\n" ::: "memory");
    } else {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 88;\n" ::: "memory");
    }
    if (warp < 12) {
      ws_producer<D, FP8>(p, sh, base, n_items);
    } else if (warp == 13) {
      ws_qloader<D>(p, sh, base, n_items);
    } else if (warp == 12) {
      ws_mma<D>(p, sh, base, tmem);
      if ((tid & 31) == 0) {  // retire every MMA this CTA issued before TMEM is freed
        tc_commit(sh.bar(wsbar::FIN));
        if (!sh.drain(wsbar::FIN, 0)) report(p.status, PPA_ERR_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
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
cudaError_t launch_attn_ws(const AttnParams& p, int max_items, cudaStream_t stream) {
  using C = WsCfg<D, FP8>;
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
      e = cudaFuncSetAttribute(attn_ws_kernel<D, FP8, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      configured[dev] = 1;
    }
    sms = sm_count[dev];
  }
  const int grid = max(1, min(sms, max_items));
  attn_ws_kernel<D, FP8, SPLIT><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ppa
