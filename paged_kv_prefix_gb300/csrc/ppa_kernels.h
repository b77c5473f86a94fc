// Launch parameters and launchers shared between the C-ABI layer (ppa_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ppa_internal.cuh"

namespace ppa {

struct Stage1Params {
  int num_seqs, total_q, tq, tn, num_kv_heads, page_size, max_pages_per_seq, no_prune;
  int kv_in_cache;      // block-table rows must cover c + n positions, not c
  int max_qtiles;       // bound on sum_b ceil(n_b / tq); also bounds the number of units
  int nq;               // query tiles per unit (plan mode)
  MaskParams mask;
  const int32_t* cu_query_lens;
  const int32_t* context_lens;
  // plan mode
  WsHeader* ws;
  int32_t* seq_unit_base;  // [B + 1] first unit of each sequence (sequence order)
  int32_t* seq_cost;       // [B]     key tiles summed over the sequence's units
  int32_t* seq_order;      // [B]     sequences, heaviest first
  int32_t* seq_item_base;  // [B + 1] first item of each sequence in heaviest-first order
  Unit* units;             // [max_units]
  int32_t* items;          // [max_units * num_kv_heads]: unit * Hkv + kv head
  // split-KV: a sequence with one query tile becomes segments of split_tiles key tiles
  int split_tiles;         // 0: off
  int max_units;           // capacity of units / items
  int32_t* seq_split_base; // [B + 1] first partial slot of each split sequence (or nullptr)
  // bounds-only mode
  int32_t* bounds_out;     // [max_qtiles][2]
  int32_t* status;
};

// TMA descriptors of one call (encoded on the host per call; passed as a __grid_constant__
// kernel parameter so that the kernel can hand their parameter-space address to the TMA unit).
//   q             [total_q][Hq][D] bf16, box {64, G, tq}: one query tile, token-major rows
//   k_new, v_new  [total_q][Hkv][D] bf16, box {64, 1, 16}: 16 keys of one KV head
//   k_cache, v_cache [num_pages * P][Hkv][D] bf16, box {64, 1, 16} (unused for fp8 caches)
// All use the 128-byte swizzle, matching the operand layout of the MMAs.
// Boxes of {64 columns, 1 head, 16 rows}, and the same tensors with 32-row boxes for key
// blocks that are contiguous in their source (one page, or all new tokens).
struct TmaMaps {
  CUtensorMap q, k_new, v_new, k_cache, v_cache;
  CUtensorMap k_new32, v_new32, k_cache32, v_cache32;
  // fp8 caches widened in the single-CTA kernel: [num_pages * P][Hkv][D] e4m3 bytes, boxes
  // {D, 1, 16} with the 128-byte (D 128) or 64-byte (D 64) swizzle
  CUtensorMap k_cache8, v_cache8;
};

struct AttnParams {
  TmaMaps tm;
  const void* q;
  const void* k_new;
  const void* v_new;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* cu_query_lens;
  const int32_t* context_lens;
  const float* k_scale;  // fp8 only
  const float* v_scale;  // fp8 only
  void* out;
  WsHeader* ws;
  const Unit* units;
  const int32_t* items;
  const int32_t* row_bounds;  // [total_q][2] row intervals when multimodal ranges are given
  int32_t* status;
  int kv_in_cache;  // new tokens' K/V read from the cache (positions c .. s-1); k_new unused
  // split-KV partial results: slot (part * Hkv + g) holds 128 rows of D fp32 (O / l) and 128
  // base-2 log-sum-exps
  float* part_o;
  float* part_lse;
  MaskParams mask;
  int num_q_heads, num_kv_heads, group, tq, page_size, num_pages, max_pages_per_seq;
  float scale_log2;  // softmax scale * log2(e)
  unsigned long long wait_ns;  // limit of every bounded wait in the attention kernels
  int debug_stall;  // testing (single-CTA kernel): the CTA taking item 0 never loads its queries
};

cudaError_t launch_plan(const Stage1Params& p, cudaStream_t stream);
cudaError_t launch_tile_bounds(const Stage1Params& p, cudaStream_t stream);

// Query tiles per unit of work for a head dimension: two 128-row tiles share each K/V tile
// when both fit in TMEM and shared memory (D <= 128), otherwise one.
// Two consecutive query tiles per unit: one CTA's ping-pong pair (head_dim <= 128) or the two
// CTAs of a pair, one tile each (head_dim 256).
__host__ __device__ constexpr int tiles_per_unit(int) { return 2; }
cudaError_t launch_debug_mask(const MaskParams& mp, int seq, const int32_t* cu, const int32_t* ctx,
                              uint32_t* bitmap, int max_rows, int words_per_row,
                              cudaStream_t stream);
cudaError_t launch_live_pairs(const MaskParams& mp, int num_seqs, int total_q, const int32_t* cu,
                              const int32_t* ctx, unsigned long long* out, cudaStream_t stream);
cudaError_t launch_live_kv_tokens(const MaskParams& mp, int num_seqs, const int32_t* cu,
                                  const int32_t* ctx, unsigned long long* out,
                                  cudaStream_t stream);
cudaError_t launch_e4m3_decode(const uint8_t* codes, uint16_t* out, int n, cudaStream_t stream);
// Per query token, its row's allowed key interval [kmin, kmax] (out: [total_q][2]).
cudaError_t launch_row_bounds(const MaskParams& mp, int num_seqs, int total_q, const int32_t* cu,
                              const int32_t* ctx, int32_t* out, cudaStream_t stream);

// fp8 caches: the live cache key tiles of a planned batch, dequantised to bf16 scratch pages of
// TN tokens (ppa_fp8_dequant.cu).
struct Fp8DequantParams {
  WsHeader* ws;        // the plan's header (n_units; n_items cleared if the staging overflows)
  const Unit* units;
  int max_units;       // capacity of `units`
  const int32_t* context_lens;
  const int32_t* block_table;
  const void* k_cache;  // e4m3 codes [num_pages][page_size][Hkv][D]
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  void* k_out;          // bf16 [capacity][tn][Hkv][D]: the live tiles, packed
  void* v_out;
  int32_t* table;       // [num_seqs][tiles_per_seq]: staging page of each live tile
  uint32_t* live_bits;  // [num_seqs][words_per_seq]
  int32_t* status;
  const int32_t* cu_query_lens;
  int kv_in_cache;  // cache positions run to c + n (new tokens already appended), not c
  int num_seqs, tiles_per_seq, words_per_seq, tn, page_size, num_pages, max_pages_per_seq;
  int row_codes;  // Hkv * D
  int capacity;   // staging pages
};
cudaError_t launch_fp8_dequant(const Fp8DequantParams& p, cudaStream_t stream);

// KV append (ppa_append.cu): new token j of sequence b to cache position c_b + j.
struct AppendParams {
  const void* k_new;  // bf16 [total_q][Hkv][D]
  const void* v_new;
  void* k_cache;      // bf16 or e4m3 codes [num_pages][page_size][Hkv][D]
  void* v_cache;
  const int32_t* block_table;
  const int32_t* cu_query_lens;
  const int32_t* context_lens;
  const float* k_scale;  // fp8 only
  const float* v_scale;
  int32_t* status;
  int num_seqs, total_q, row_elems /* Hkv * D */, page_size, num_pages, max_pages_per_seq;
  int fp8;
};
cudaError_t launch_append_kv(const AppendParams& p, cudaStream_t stream);

// Split-KV merge (ppa_stage1.cu): for every split sequence and KV head, the segments' partial
// rows combined by their log-sum-exps into the bf16 output.
struct MergeParams {
  const WsHeader* ws;  // the plan's header: n_items == 0 after the plan rejected the batch
  const float* part_o;
  const float* part_lse;
  const int32_t* seq_split_base;  // [B + 1]
  const int32_t* cu_query_lens;
  void* out;  // bf16 [total_q][Hq][D]
  int num_seqs, total_q, num_kv_heads, group, head_dim, num_q_heads;
};
cudaError_t launch_split_merge(const MergeParams& p, cudaStream_t stream);

// Attention kernels, one translation unit per head dimension. `max_ctas` bounds the
// persistent grid (the number of work items cannot be known on the host).
cudaError_t launch_attn_d64(const AttnParams& p, bool fp8, bool split, int max_items,
                             cudaStream_t stream);
cudaError_t launch_attn_d128(const AttnParams& p, bool fp8, bool split, int max_items,
                             cudaStream_t stream);
cudaError_t launch_attn_d256(const AttnParams& p, bool fp8, bool split, int max_items,
                             cudaStream_t stream);

}  // namespace ppa
