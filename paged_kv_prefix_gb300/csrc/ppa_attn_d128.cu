// Attention kernel instances for head_dim 128 (bf16 and fp8 e4m3 KV caches): the
// warp-specialised two-query-tile kernel.
#include "ppa_attn_ws.cuh"

namespace ppa {

cudaError_t launch_attn_d128(const AttnParams& p, bool fp8, bool split, int max_items,
                             cudaStream_t stream) {
  if (split)  // the split-KV epilogue is compiled only into these instances
    return fp8 ? launch_attn_ws<128, true, true>(p, max_items, stream)
               : launch_attn_ws<128, false, true>(p, max_items, stream);
  return fp8 ? launch_attn_ws<128, true, false>(p, max_items, stream)
             : launch_attn_ws<128, false, false>(p, max_items, stream);
}

}  // namespace ppa
