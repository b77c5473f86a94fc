// ppa_prefill_noalloc: ppa_prefill for callers that cannot allocate device memory.
//
// ppa_prefill needs a few hundred kilobytes of scratch (the query-tile table and the work
// list) that its caller normally allocates. Some callers cannot: a plugin running inside a host
// framework that owns the whole device memory pool and hands its plugins no allocator, or a
// runtime that forbids device allocation after start-up to keep a fixed, audited memory
// footprint. For them this entry point keeps the scratch in a file-scope device array of fixed
// size, reserved when the library is loaded (every GPU that loads the library holds it until
// the process exits), and allocates nothing per call.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ppa.h"

namespace {

// The scratch. In host code this name is only a host-side stand-in for the symbol, never a
// device address: the address a kernel may use comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_workspace[PPA_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device, looked up once per device (with that
// device current) and cached.
ppa_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PPA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PPA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_device_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr)
      return PPA_ERR_CUDA;
    g_device_ptr[dev] = p;
  }
  *out = g_device_ptr[dev];
  return PPA_OK;
}

}  // namespace

extern "C" ppa_status ppa_prefill_noalloc(const ppa_dims* dims, const void* q, const void* k_new,
                                          const void* v_new, const void* k_cache,
                                          const void* v_cache, const int32_t* block_table,
                                          const int32_t* cu_query_lens,
                                          const int32_t* context_lens, const int32_t* mm_ranges,
                                          const float* k_scale, const float* v_scale, void* out,
                                          int32_t* device_status, void* stream) {
  if (dims == nullptr) return PPA_ERR_INVALID;
  // fp8 caches widen inside the attention kernel here, and split-KV is off: neither the bf16
  // staging of the live cache tiles nor the split partials would fit the fixed scratch. Both
  // change only how the result is computed, not the result.
  ppa_dims d = *dims;
  if (d.kv_dtype == PPA_KV_FP8_E4M3) d.flags |= PPA_FLAG_FP8_INKERNEL;
  d.kv_split_tiles = 0;
  dims = &d;
  const size_t need = ppa_workspace_bytes(dims);
  if (need == 0) {
    // Invalid dims: ppa_prefill checks them before anything else and returns the reason
    // without launching, so the missing workspace is never looked at.
    return ppa_prefill(dims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                       context_lens, mm_ranges, k_scale, v_scale, out, nullptr, device_status,
                       stream);
  }
  if (need > PPA_NOALLOC_WORKSPACE_BYTES) return PPA_ERR_UNSUPPORTED;  // batch too large
  void* scratch = nullptr;
  const ppa_status st = scratch_for_current_device(&scratch);
  if (st != PPA_OK) return st;
  // The plan stage writes every scratch word the attention stage reads (header, tile table,
  // work order) before that stage runs, so stale contents of an earlier call need no clearing.
  return ppa_prefill(dims, q, k_new, v_new, k_cache, v_cache, block_table, cu_query_lens,
                     context_lens, mm_ranges, k_scale, v_scale, out, scratch, device_status,
                     stream);
}
