// Attention kernel instances for head_dim 256 (bf16 and fp8 e4m3 KV caches): the CTA-pair
// kernel, M = 256 tcgen05 MMAs over two SMs with 128-key tiles.
#include "ppa_attn_pair.cuh"

namespace ppa {

cudaError_t launch_attn_d256(const AttnParams& p, bool fp8, bool split, int max_items,
                             cudaStream_t stream) {
  if (split)  // the split-KV epilogue is compiled only into these instances
    return fp8 ? launch_attn_pair<256, true, true>(p, max_items, stream)
               : launch_attn_pair<256, false, true>(p, max_items, stream);
  return fp8 ? launch_attn_pair<256, true, false>(p, max_items, stream)
             : launch_attn_pair<256, false, false>(p, max_items, stream);
}

}  // namespace ppa
