// attn_decode_paged.cu -- instantiations of the attention kernel over a paged KV cache
// (block table), head dim 128 or 256, 4-stage ring.
#include "attn_decode.cuh"

namespace da {

cudaError_t launch_attention_paged(const AttnParams& p, int grid, int nb, int dim, cudaStream_t stream) {
  if (dim == kHeadDimWide)
    return nb == 1 ? launch_one<1, false, 4, 0, kHeadDimWide, true>(p, grid, stream)
                   : launch_one<2, false, 4, 0, kHeadDimWide, true>(p, grid, stream);
  if (dim != kHeadDim) return cudaErrorInvalidValue;
  return nb == 1 ? launch_one<1, false, 4, 0, kHeadDim, true>(p, grid, stream)
                 : launch_one<2, false, 4, 0, kHeadDim, true>(p, grid, stream);
}

}  // namespace da
