// The C ABI declared in include/ppa.h: argument validation, workspace sizing and the two
// launches of ppa_prefill. Nothing here allocates, frees or synchronises, except
// ppa_read_status, whose job is to synchronise.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/ppa.h"
#include "ppa_internal.cuh"
#include "ppa_kernels.h"

namespace {

using ppa::WsHeader;

constexpr unsigned kKnownFlags = PPA_FLAG_CAUSAL | PPA_FLAG_CLAMP_MM | PPA_FLAG_NO_PRUNE |
                                 PPA_FLAG_FP8_INKERNEL | PPA_FLAG_KV_IN_CACHE;

bool kv_in_cache(const ppa_dims* d) { return (d->flags & PPA_FLAG_KV_IN_CACHE) != 0u; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ppa_status check_dims(const ppa_dims* d) {
  if (d == nullptr) return PPA_ERR_INVALID;
  if (d->num_seqs < 0 || d->total_q < 0) return PPA_ERR_INVALID;
  if (d->num_q_heads < 1 || d->num_kv_heads < 1) return PPA_ERR_INVALID;
  if (d->num_q_heads % d->num_kv_heads != 0) return PPA_ERR_INVALID;
  if (d->page_size < 1 || d->num_pages < 1 || d->max_pages_per_seq < 1) return PPA_ERR_INVALID;
  if (d->max_mm_ranges < 0) return PPA_ERR_INVALID;
  if (d->chunk_size < 0 || (d->chunk_size > 0 && d->chunk_lookback < 0)) return PPA_ERR_INVALID;
  if (d->kv_split_tiles < -1 || d->max_cache_tokens < 0) return PPA_ERR_INVALID;
  if ((d->flags & ~kKnownFlags) != 0u) return PPA_ERR_INVALID;
  if (!std::isfinite(d->sm_scale)) return PPA_ERR_INVALID;
  if (d->kv_dtype != PPA_KV_BF16 && d->kv_dtype != PPA_KV_FP8_E4M3) return PPA_ERR_INVALID;
  if (d->num_q_heads / d->num_kv_heads > ppa::kRowsPerTile) return PPA_ERR_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return PPA_ERR_UNSUPPORTED;
  // element offsets are formed in 64-bit; rows and tokens must fit int32
  if ((long long)d->num_pages * d->page_size > INT_MAX) return PPA_ERR_INVALID;
  if ((long long)d->total_q * d->num_q_heads > INT_MAX) return PPA_ERR_INVALID;
  return PPA_OK;
}

int group_of(const ppa_dims* d) { return d->num_q_heads / d->num_kv_heads; }

// Split-KV segment length in key tiles: the caller's, or with -1 the tuned default. A sweep
// over 4, 8, 16, 32 and 64 tiles (decode and 4-token verification batches of 8 and 32
// sequences over 8K-32K contexts, head dim 128, 8 KV heads) found 32 tiles (4096 keys) best
// or within 4 % of best at every point; shorter segments cost more in merging and partial
// traffic than they gain in balance once rows carry more than one token.
constexpr int kAutoSplitTiles = 32;
int split_tiles_of(const ppa_dims* d) {
  return d->kv_split_tiles < 0 ? kAutoSplitTiles : d->kv_split_tiles;
}

long long max_qtiles_for(const ppa_dims* d, int tq) {
  return ((long long)d->total_q + tq - 1) / tq + d->num_seqs;
}

ppa::MaskParams mask_of(const ppa_dims* d, const int32_t* mm_ranges) {
  ppa::MaskParams m;
  m.causal = (d->flags & PPA_FLAG_CAUSAL) ? 1 : 0;
  m.window_left = d->window_left;
  m.window_right = d->window_right;
  m.clamp_mm = (d->flags & PPA_FLAG_CLAMP_MM) ? 1 : 0;
  m.max_mm_ranges = (mm_ranges != nullptr) ? d->max_mm_ranges : 0;
  m.mm_ranges = (d->max_mm_ranges > 0) ? mm_ranges : nullptr;
  m.chunk_size = d->chunk_size > 0 ? d->chunk_size : 0;
  m.chunk_lookback = d->chunk_size > 0 ? d->chunk_lookback : 0;
  m.seq_causal = d->seq_causal;
  return m;
}

struct WsLayout {
  size_t header, seq_unit_base, seq_cost, seq_order, seq_item_base, units, items;
  // split-KV: unit capacity with the segments, per-sequence partial-slot bases, partials
  long long max_units;
  bool split;
  size_t seq_split_base, part_o, part_lse;
  size_t row_bounds;  // [total_q][2] row intervals; only with multimodal ranges
  bool has_row_bounds;
  // fp8 caches dequantised before the attention kernel (see ppa_fp8_dequant.cu)
  bool fp8_scratch;
  int fp8_tiles_per_seq, fp8_words_per_seq, fp8_pages;
  size_t fp8_bits, fp8_table, fp8_k, fp8_v;
  size_t total;
};

WsLayout ws_layout(const ppa_dims* d) {
  const long long mq = max_qtiles_for(d, ppa::tokens_per_qtile(group_of(d)));
  const size_t seq_ints = (size_t)d->num_seqs + 1;
  WsLayout w;
  w.header = 0;
  w.seq_unit_base = align_up(sizeof(WsHeader), 256);
  w.seq_cost = align_up(w.seq_unit_base + seq_ints * 4, 256);
  w.seq_order = align_up(w.seq_cost + seq_ints * 4, 256);
  w.seq_item_base = align_up(w.seq_order + seq_ints * 4, 256);
  // split-KV: a split sequence has one query tile (n <= tq) and at most
  // ceil((max_pages_per_seq * P + tq) / 128) key tiles, so at most nseg_max segments
  long long nseg_max = 1;
  const int split_tiles = split_tiles_of(d);
  w.split = split_tiles > 0;
  if (w.split) {
    const long long tn = ppa::keys_per_tile(d->head_dim);
    const long long tq = ppa::tokens_per_qtile(group_of(d));
    const long long tiles = ((long long)d->max_pages_per_seq * d->page_size + tq + tn - 1) / tn;
    nseg_max = (tiles + split_tiles - 1) / split_tiles;
    if (nseg_max < 1) nseg_max = 1;
  }
  w.max_units = mq + (w.split ? (long long)d->num_seqs * (nseg_max - 1) : 0);
  w.units = align_up(w.seq_item_base + seq_ints * 4, 256);
  w.items = align_up(w.units + (size_t)w.max_units * sizeof(ppa::Unit), 256);
  w.total = align_up(w.items + (size_t)w.max_units * d->num_kv_heads * 4, 256);
  w.seq_split_base = w.part_o = w.part_lse = w.total;
  if (w.split) {
    const size_t slots = (size_t)d->num_seqs * nseg_max * d->num_kv_heads;
    w.seq_split_base = w.total;
    w.part_o = align_up(w.seq_split_base + seq_ints * 4, 256);
    w.part_lse = align_up(w.part_o + slots * ppa::kRowsPerTile * d->head_dim * 4, 256);
    w.total = align_up(w.part_lse + slots * ppa::kRowsPerTile * 4, 256);
  }
  w.has_row_bounds = d->max_mm_ranges > 0;
  w.row_bounds = w.total;
  if (w.has_row_bounds) w.total = align_up(w.row_bounds + (size_t)d->total_q * 8, 256);
  w.fp8_scratch = false;
  w.fp8_tiles_per_seq = w.fp8_words_per_seq = w.fp8_pages = 0;
  w.fp8_bits = w.fp8_table = w.fp8_k = w.fp8_v = w.total;
  if (d->kv_dtype == PPA_KV_FP8_E4M3 && !(d->flags & PPA_FLAG_FP8_INKERNEL)) {
    const long long tn = ppa::keys_per_tile(d->head_dim);
    const long long tiles = ((long long)d->max_pages_per_seq * d->page_size + tn - 1) / tn;
    const long long entries = tiles * d->num_seqs;  // the table: every tile of every row
    long long pages = entries;
    // The live cache positions of one sequence are consecutive (the allowed keys of each row
    // form an interval containing the row, and the rows are consecutive), so L of them touch
    // at most floor((L - 1) / tn) + 2 tiles.
    if (d->max_cache_tokens > 0)
      pages = std::min(pages, (long long)d->max_cache_tokens / tn + 2LL * d->num_seqs);
    if (pages > 0 && pages * tn <= INT_MAX) {  // scratch rows must fit the kernel's int32 rows
      const size_t row_bytes = (size_t)d->num_kv_heads * d->head_dim * 2;
      w.fp8_scratch = true;
      w.fp8_tiles_per_seq = (int)tiles;
      w.fp8_words_per_seq = (int)((tiles + 31) / 32);
      w.fp8_pages = (int)pages;
      w.fp8_bits = w.total;
      w.fp8_table = align_up(w.fp8_bits + (size_t)d->num_seqs * w.fp8_words_per_seq * 4, 256);
      w.fp8_k = align_up(w.fp8_table + (size_t)entries * 4, 256);
      w.fp8_v = align_up(w.fp8_k + (size_t)pages * tn * row_bytes, 256);
      w.total = align_up(w.fp8_v + (size_t)pages * tn * row_bytes, 256);
    }
  }
  return w;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A 3-D bf16 tensor [rows][heads][D] (row-major) seen as dims {D, heads, rows}, with a box of
// {64, box_heads, box_rows} and the 128-byte swizzle.
bool encode_rows(CUtensorMap* m, const void* ptr, int head_dim, int heads, long long rows,
                 int box_heads, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)heads * head_dim * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An fp8 cache [rows][heads][D] as e4m3 bytes, seen as dims {D, heads, rows}, with a box of
// {D, 1, 16} rows in the swizzle whose span is one row (128-byte rows at D 128, 64 at D 64): the
// layout the attention kernel's staging area and its widening use.
bool encode_rows_u8(CUtensorMap* m, const void* ptr, int head_dim, int heads, long long rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr || (head_dim != 64 && head_dim != 128)) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)head_dim, (cuuint64_t)heads * head_dim};
  const cuuint32_t box[3] = {(cuuint32_t)head_dim, 1u, 16u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

size_t ppa_workspace_bytes(const ppa_dims* dims) {
  if (check_dims(dims) != PPA_OK) return 0;
  return ws_layout(dims).total;
}

void ppa_query_tiles(const ppa_dims* dims, int* tq, int* tn) {
  const bool ok = check_dims(dims) == PPA_OK;
  if (tq) *tq = ok ? ppa::tokens_per_qtile(group_of(dims)) : 0;
  if (tn) *tn = ok ? ppa::keys_per_tile(dims->head_dim) : 0;
}

ppa_status ppa_plan(const ppa_dims* dims, const int32_t* cu_query_lens,
                    const int32_t* context_lens, const int32_t* mm_ranges, void* workspace,
                    int32_t* device_status, void* stream) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  if (cu_query_lens == nullptr || context_lens == nullptr || workspace == nullptr ||
      device_status == nullptr)
    return PPA_ERR_INVALID;
  if (dims->max_mm_ranges > 0 && mm_ranges == nullptr) return PPA_ERR_INVALID;
  if (!aligned16(workspace)) return PPA_ERR_INVALID;
  if (dims->num_seqs == 0 || dims->total_q == 0) return PPA_OK;  // nothing to plan
  const int tq = ppa::tokens_per_qtile(group_of(dims));
  const long long mq = max_qtiles_for(dims, tq);
  if (mq * dims->num_kv_heads > INT_MAX) return PPA_ERR_INVALID;
  const WsLayout w = ws_layout(dims);
  if (w.max_units * dims->num_kv_heads > INT_MAX) return PPA_ERR_INVALID;
  char* ws = static_cast<char*>(workspace);
  ppa::Stage1Params s1{};
  s1.num_seqs = dims->num_seqs;
  s1.total_q = dims->total_q;
  s1.tq = tq;
  s1.tn = ppa::keys_per_tile(dims->head_dim);
  s1.num_kv_heads = dims->num_kv_heads;
  s1.page_size = dims->page_size;
  s1.max_pages_per_seq = dims->max_pages_per_seq;
  s1.no_prune = (dims->flags & PPA_FLAG_NO_PRUNE) ? 1 : 0;
  s1.kv_in_cache = kv_in_cache(dims) ? 1 : 0;
  s1.max_qtiles = (int)mq;
  s1.nq = ppa::tiles_per_unit(dims->head_dim);
  s1.mask = mask_of(dims, mm_ranges);
  s1.cu_query_lens = cu_query_lens;
  s1.context_lens = context_lens;
  s1.ws = reinterpret_cast<WsHeader*>(ws + w.header);
  s1.seq_unit_base = reinterpret_cast<int32_t*>(ws + w.seq_unit_base);
  s1.seq_cost = reinterpret_cast<int32_t*>(ws + w.seq_cost);
  s1.seq_order = reinterpret_cast<int32_t*>(ws + w.seq_order);
  s1.seq_item_base = reinterpret_cast<int32_t*>(ws + w.seq_item_base);
  s1.units = reinterpret_cast<ppa::Unit*>(ws + w.units);
  s1.items = reinterpret_cast<int32_t*>(ws + w.items);
  s1.split_tiles = w.split ? split_tiles_of(dims) : 0;
  s1.max_units = (int)w.max_units;
  s1.seq_split_base = w.split ? reinterpret_cast<int32_t*>(ws + w.seq_split_base) : nullptr;
  s1.bounds_out = nullptr;
  s1.status = device_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ppa::launch_plan(s1, s) != cudaSuccess) return PPA_ERR_CUDA;
  if (w.has_row_bounds &&
      ppa::launch_row_bounds(s1.mask, dims->num_seqs, dims->total_q, cu_query_lens, context_lens,
                             reinterpret_cast<int32_t*>(ws + w.row_bounds), s) != cudaSuccess)
    return PPA_ERR_CUDA;
  return PPA_OK;
}

}  // extern "C"

namespace {

// ppa_attend with the attention kernel's wait limit and the test stall of
// ppa_debug_prefill_stalled.
ppa_status attend_impl(const ppa_dims* dims, const void* q, const void* k_new, const void* v_new,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* cu_query_lens, const int32_t* context_lens,
                       const int32_t* mm_ranges, const float* k_scale, const float* v_scale,
                       void* out, void* workspace, int32_t* device_status, void* stream,
                       unsigned long long wait_ns, int stall) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  const bool in_cache = kv_in_cache(dims);
  if (!in_cache && (k_new == nullptr || v_new == nullptr)) return PPA_ERR_UNSUPPORTED;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      cu_query_lens == nullptr || context_lens == nullptr || out == nullptr ||
      workspace == nullptr || device_status == nullptr)
    return PPA_ERR_INVALID;
  if (dims->max_mm_ranges > 0 && mm_ranges == nullptr) return PPA_ERR_INVALID;
  const bool fp8 = dims->kv_dtype == PPA_KV_FP8_E4M3;
  if (fp8 && (k_scale == nullptr || v_scale == nullptr)) return PPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace))
    return PPA_ERR_INVALID;
  if (!in_cache && (!aligned16(k_new) || !aligned16(v_new))) return PPA_ERR_INVALID;
  if (dims->num_seqs == 0 || dims->total_q == 0) return PPA_OK;  // nothing to compute

  const int G = group_of(dims);
  const int tq = ppa::tokens_per_qtile(G);
  const long long mq = max_qtiles_for(dims, tq);
  if (mq * dims->num_kv_heads > INT_MAX) return PPA_ERR_INVALID;
  const WsLayout w = ws_layout(dims);
  if (w.max_units * dims->num_kv_heads > INT_MAX) return PPA_ERR_INVALID;
  char* ws = static_cast<char*>(workspace);

  ppa::AttnParams a{};
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.cu_query_lens = cu_query_lens;
  a.context_lens = context_lens;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out = out;
  a.ws = reinterpret_cast<WsHeader*>(ws + w.header);
  a.units = reinterpret_cast<const ppa::Unit*>(ws + w.units);
  a.items = reinterpret_cast<const int32_t*>(ws + w.items);
  a.row_bounds = w.has_row_bounds ? reinterpret_cast<const int32_t*>(ws + w.row_bounds) : nullptr;
  a.part_o = w.split ? reinterpret_cast<float*>(ws + w.part_o) : nullptr;
  a.part_lse = w.split ? reinterpret_cast<float*>(ws + w.part_lse) : nullptr;
  a.status = device_status;
  a.kv_in_cache = in_cache ? 1 : 0;
  a.mask = mask_of(dims, mm_ranges);
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.group = G;
  a.tq = tq;
  a.page_size = dims->page_size;
  a.num_pages = dims->num_pages;
  a.max_pages_per_seq = dims->max_pages_per_seq;
  a.wait_ns = wait_ns;
  a.debug_stall = stall;
  const int D = dims->head_dim;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // fp8 with scratch: dequantise the live cache tiles once, then run the bf16 kernel on them,
  // read as a paged cache of 128-token pages through the identity block table.
  const bool prepass = fp8 && w.fp8_scratch;
  if (prepass) {
    ppa::Fp8DequantParams f{};
    f.ws = a.ws;
    f.units = a.units;
    f.max_units = (int)w.max_units;
    f.context_lens = context_lens;
    f.block_table = block_table;
    f.k_cache = k_cache;
    f.v_cache = v_cache;
    f.k_scale = k_scale;
    f.v_scale = v_scale;
    f.k_out = ws + w.fp8_k;
    f.v_out = ws + w.fp8_v;
    f.table = reinterpret_cast<int32_t*>(ws + w.fp8_table);
    f.live_bits = reinterpret_cast<uint32_t*>(ws + w.fp8_bits);
    f.status = device_status;
    f.cu_query_lens = cu_query_lens;
    f.kv_in_cache = in_cache ? 1 : 0;
    f.num_seqs = dims->num_seqs;
    f.tiles_per_seq = w.fp8_tiles_per_seq;
    f.words_per_seq = w.fp8_words_per_seq;
    f.tn = ppa::keys_per_tile(D);
    f.page_size = dims->page_size;
    f.num_pages = dims->num_pages;
    f.max_pages_per_seq = dims->max_pages_per_seq;
    f.row_codes = dims->num_kv_heads * D;
    f.capacity = w.fp8_pages;
    if (ppa::launch_fp8_dequant(f, s) != cudaSuccess) return PPA_ERR_CUDA;
    a.k_cache = f.k_out;
    a.v_cache = f.v_out;
    a.block_table = f.table;
    a.page_size = f.tn;
    a.num_pages = w.fp8_pages;
    a.max_pages_per_seq = w.fp8_tiles_per_seq;
  }
  const bool fp8_kernel = fp8 && !prepass;
  bool maps_ok = encode_rows(&a.tm.q, q, D, dims->num_q_heads, dims->total_q, G, tq);
  if (maps_ok && !in_cache)  // cache-sourced: the kernel never reads k_new / v_new
    maps_ok = encode_rows(&a.tm.k_new, k_new, D, dims->num_kv_heads, dims->total_q, 1, 16) &&
              encode_rows(&a.tm.v_new, v_new, D, dims->num_kv_heads, dims->total_q, 1, 16) &&
              encode_rows(&a.tm.k_new32, k_new, D, dims->num_kv_heads, dims->total_q, 1, 32) &&
              encode_rows(&a.tm.v_new32, v_new, D, dims->num_kv_heads, dims->total_q, 1, 32);
  if (maps_ok && fp8_kernel && D <= 128) {  // e4m3 rows boxed into the producers' staging
    const long long cache_rows = (long long)a.num_pages * a.page_size;
    maps_ok = encode_rows_u8(&a.tm.k_cache8, a.k_cache, D, dims->num_kv_heads, cache_rows) &&
              encode_rows_u8(&a.tm.v_cache8, a.v_cache, D, dims->num_kv_heads, cache_rows);
  }
  if (maps_ok && !fp8_kernel) {
    const long long cache_rows = (long long)a.num_pages * a.page_size;
    maps_ok = encode_rows(&a.tm.k_cache, a.k_cache, D, dims->num_kv_heads, cache_rows, 1, 16) &&
              encode_rows(&a.tm.v_cache, a.v_cache, D, dims->num_kv_heads, cache_rows, 1, 16) &&
              encode_rows(&a.tm.k_cache32, a.k_cache, D, dims->num_kv_heads, cache_rows, 1, 32) &&
              encode_rows(&a.tm.v_cache32, a.v_cache, D, dims->num_kv_heads, cache_rows, 1, 32);
  }
  if (!maps_ok) return PPA_ERR_CUDA;
  const float sm = dims->sm_scale > 0.f ? dims->sm_scale : 1.0f / std::sqrt((float)dims->head_dim);
  a.scale_log2 = sm * 1.4426950408889634f;
  const int max_items = (int)(w.max_units * dims->num_kv_heads);
  cudaError_t e;
  switch (dims->head_dim) {
    case 64: e = ppa::launch_attn_d64(a, fp8_kernel, w.split, max_items, s); break;
    case 128: e = ppa::launch_attn_d128(a, fp8_kernel, w.split, max_items, s); break;
    default: e = ppa::launch_attn_d256(a, fp8_kernel, w.split, max_items, s); break;
  }
  if (e == cudaSuccess && w.split) {  // segments of split sequences -> the output rows
    ppa::MergeParams m{};
    m.ws = a.ws;
    m.part_o = a.part_o;
    m.part_lse = a.part_lse;
    m.seq_split_base = reinterpret_cast<const int32_t*>(ws + w.seq_split_base);
    m.cu_query_lens = cu_query_lens;
    m.out = out;
    m.num_seqs = dims->num_seqs;
    m.total_q = dims->total_q;
    m.num_kv_heads = dims->num_kv_heads;
    m.group = G;
    m.head_dim = D;
    m.num_q_heads = dims->num_q_heads;
    e = ppa::launch_split_merge(m, s);
  }
  return e == cudaSuccess ? PPA_OK : PPA_ERR_CUDA;
}

// Host checks of ppa_prefill, before ppa_plan launches anything.
ppa_status prefill_checks(const ppa_dims* dims, const void* q, const void* k_new,
                          const void* v_new, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const float* k_scale, const float* v_scale,
                          const void* out) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  const bool in_cache = kv_in_cache(dims);
  if (!in_cache && (k_new == nullptr || v_new == nullptr)) return PPA_ERR_UNSUPPORTED;
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || block_table == nullptr ||
      out == nullptr)
    return PPA_ERR_INVALID;
  if (dims->kv_dtype == PPA_KV_FP8_E4M3 && (k_scale == nullptr || v_scale == nullptr))
    return PPA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PPA_ERR_INVALID;
  if (!in_cache && (!aligned16(k_new) || !aligned16(v_new))) return PPA_ERR_INVALID;
  return PPA_OK;
}

}  // namespace

extern "C" {

ppa_status ppa_attend(const ppa_dims* dims, const void* q, const void* k_new, const void* v_new,
                      const void* k_cache, const void* v_cache, const int32_t* block_table,
                      const int32_t* cu_query_lens, const int32_t* context_lens,
                      const int32_t* mm_ranges, const float* k_scale, const float* v_scale,
                      void* out, void* workspace, int32_t* device_status, void* stream) {
  return attend_impl(dims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                     context_lens, mm_ranges, k_scale, v_scale, out, workspace, device_status,
                     stream, ppa::kWaitNs, 0);
}

ppa_status ppa_debug_prefill_stalled(const ppa_dims* dims, const void* q, const void* k_new,
                                     const void* v_new, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, const int32_t* cu_query_lens,
                                     const int32_t* context_lens, const int32_t* mm_ranges,
                                     const float* k_scale, const float* v_scale, void* out,
                                     void* workspace, int32_t* device_status,
                                     unsigned wait_limit_us, void* stream) {
  if (dims != nullptr && dims->head_dim == 256) return PPA_ERR_UNSUPPORTED;
  if (wait_limit_us == 0) return PPA_ERR_INVALID;
  const ppa_status sc = prefill_checks(dims, q, k_new, v_new, k_cache, v_cache, block_table,
                                       k_scale, v_scale, out);
  if (sc != PPA_OK) return sc;
  const ppa_status sp = ppa_plan(dims, cu_query_lens, context_lens, mm_ranges, workspace,
                                 device_status, stream);
  if (sp != PPA_OK) return sp;
  return attend_impl(dims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                     context_lens, mm_ranges, k_scale, v_scale, out, workspace, device_status,
                     stream, 1000ull * wait_limit_us, 1);
}

ppa_status ppa_prefill(const ppa_dims* dims, const void* q, const void* k_new, const void* v_new,
                       const void* k_cache, const void* v_cache, const int32_t* block_table,
                       const int32_t* cu_query_lens, const int32_t* context_lens,
                       const int32_t* mm_ranges, const float* k_scale, const float* v_scale,
                       void* out, void* workspace, int32_t* device_status, void* stream) {
  // Validate everything ppa_attend checks before ppa_plan launches anything.
  const ppa_status sc = prefill_checks(dims, q, k_new, v_new, k_cache, v_cache, block_table,
                                       k_scale, v_scale, out);
  if (sc != PPA_OK) return sc;
  const ppa_status sp = ppa_plan(dims, cu_query_lens, context_lens, mm_ranges, workspace,
                                 device_status, stream);
  if (sp != PPA_OK) return sp;
  return ppa_attend(dims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                    context_lens, mm_ranges, k_scale, v_scale, out, workspace, device_status,
                    stream);
}

ppa_status ppa_append_kv(const ppa_dims* dims, const void* k_new, const void* v_new,
                         void* k_cache, void* v_cache, const int32_t* block_table,
                         const int32_t* cu_query_lens, const int32_t* context_lens,
                         const float* k_scale, const float* v_scale, int32_t* device_status,
                         void* stream) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr ||
      block_table == nullptr || cu_query_lens == nullptr || context_lens == nullptr ||
      device_status == nullptr)
    return PPA_ERR_INVALID;
  const bool fp8 = dims->kv_dtype == PPA_KV_FP8_E4M3;
  if (fp8 && (k_scale == nullptr || v_scale == nullptr)) return PPA_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PPA_ERR_INVALID;
  if (dims->num_seqs == 0 || dims->total_q == 0) return PPA_OK;  // nothing to write
  ppa::AppendParams a{};
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.cu_query_lens = cu_query_lens;
  a.context_lens = context_lens;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.status = device_status;
  a.num_seqs = dims->num_seqs;
  a.total_q = dims->total_q;
  a.row_elems = dims->num_kv_heads * dims->head_dim;
  a.page_size = dims->page_size;
  a.num_pages = dims->num_pages;
  a.max_pages_per_seq = dims->max_pages_per_seq;
  a.fp8 = fp8 ? 1 : 0;
  return ppa::launch_append_kv(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PPA_OK
             : PPA_ERR_CUDA;
}

ppa_status ppa_tile_bounds(const ppa_dims* dims, int tq, int tn, const int32_t* cu_query_lens,
                           const int32_t* context_lens, const int32_t* mm_ranges,
                           int32_t* bounds_out, int32_t* device_status, void* stream) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  if (tq < 1 || tn < 1 || cu_query_lens == nullptr || context_lens == nullptr ||
      bounds_out == nullptr || device_status == nullptr)
    return PPA_ERR_INVALID;
  if (dims->max_mm_ranges > 0 && mm_ranges == nullptr) return PPA_ERR_INVALID;
  if (dims->num_seqs == 0) return PPA_OK;
  ppa::Stage1Params s1{};
  s1.num_seqs = dims->num_seqs;
  s1.total_q = dims->total_q;
  s1.tq = tq;
  s1.tn = tn;
  s1.num_kv_heads = dims->num_kv_heads;
  s1.page_size = dims->page_size;
  s1.max_pages_per_seq = dims->max_pages_per_seq;
  s1.no_prune = (dims->flags & PPA_FLAG_NO_PRUNE) ? 1 : 0;
  s1.kv_in_cache = kv_in_cache(dims) ? 1 : 0;
  const long long mq = max_qtiles_for(dims, tq);
  if (mq > INT_MAX / 2) return PPA_ERR_INVALID;
  s1.max_qtiles = (int)mq;
  s1.mask = mask_of(dims, mm_ranges);
  s1.cu_query_lens = cu_query_lens;
  s1.context_lens = context_lens;
  s1.bounds_out = bounds_out;
  s1.status = device_status;
  return ppa::launch_tile_bounds(s1, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PPA_OK
             : PPA_ERR_CUDA;
}

ppa_status ppa_debug_mask(const ppa_dims* dims, int seq, const int32_t* cu_query_lens,
                          const int32_t* context_lens, const int32_t* mm_ranges,
                          uint32_t* bitmap_out, int max_rows, int words_per_row, void* stream) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  if (seq < 0 || seq >= dims->num_seqs || max_rows < 0 || words_per_row < 1 ||
      cu_query_lens == nullptr || context_lens == nullptr || bitmap_out == nullptr)
    return PPA_ERR_INVALID;
  if (dims->max_mm_ranges > 0 && mm_ranges == nullptr) return PPA_ERR_INVALID;
  if (max_rows == 0) return PPA_OK;
  return ppa::launch_debug_mask(mask_of(dims, mm_ranges), seq, cu_query_lens, context_lens,
                                bitmap_out, max_rows, words_per_row,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PPA_OK
             : PPA_ERR_CUDA;
}

ppa_status ppa_live_pairs(const ppa_dims* dims, const int32_t* cu_query_lens,
                          const int32_t* context_lens, const int32_t* mm_ranges,
                          unsigned long long* count_out, void* stream) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  if (cu_query_lens == nullptr || context_lens == nullptr || count_out == nullptr)
    return PPA_ERR_INVALID;
  if (dims->max_mm_ranges > 0 && mm_ranges == nullptr) return PPA_ERR_INVALID;
  return ppa::launch_live_pairs(mask_of(dims, mm_ranges), dims->num_seqs, dims->total_q,
                                cu_query_lens, context_lens, count_out,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PPA_OK
             : PPA_ERR_CUDA;
}

ppa_status ppa_live_kv_tokens(const ppa_dims* dims, const int32_t* cu_query_lens,
                              const int32_t* context_lens, const int32_t* mm_ranges,
                              unsigned long long* count_out, void* stream) {
  const ppa_status st = check_dims(dims);
  if (st != PPA_OK) return st;
  if (cu_query_lens == nullptr || context_lens == nullptr || count_out == nullptr)
    return PPA_ERR_INVALID;
  if (dims->max_mm_ranges > 0 && mm_ranges == nullptr) return PPA_ERR_INVALID;
  return ppa::launch_live_kv_tokens(mask_of(dims, mm_ranges), dims->num_seqs, cu_query_lens,
                                    context_lens, count_out,
                                    static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PPA_OK
             : PPA_ERR_CUDA;
}

ppa_status ppa_debug_e4m3_to_bf16(const uint8_t* codes, uint16_t* bf16_out, int n, void* stream) {
  if (n < 0 || (n > 0 && (codes == nullptr || bf16_out == nullptr))) return PPA_ERR_INVALID;
  return ppa::launch_e4m3_decode(codes, bf16_out, n, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PPA_OK
             : PPA_ERR_CUDA;
}

ppa_status ppa_read_status(int32_t* device_status, void* stream) {
  if (device_status == nullptr) return PPA_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t code = 0;
  if (cudaMemcpyAsync(&code, device_status, sizeof(code), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return PPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PPA_ERR_CUDA;
  if (cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess) return PPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PPA_ERR_CUDA;
  return static_cast<ppa_status>(code);
}

const char* ppa_status_string(ppa_status status) {
  switch (status) {
    case PPA_OK: return "ok";
    case PPA_ERR_INVALID: return "invalid argument";
    case PPA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PPA_ERR_CUDA: return "CUDA runtime error";
    case PPA_ERR_TIMEOUT: return "device-side wait timed out";
    case PPA_ERR_BAD_PAGE: return "block-table entry out of range";
  }
  return "unknown status";
}

int ppa_version(void) { return PPA_VERSION; }

}  // extern "C"
