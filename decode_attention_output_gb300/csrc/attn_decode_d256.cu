// attn_decode_d256.cu -- instantiations of the attention kernel at head dim 256
// (4-stage ring of 32-token tiles; attention and scores-only variants).
#include "attn_decode.cuh"

namespace da {

cudaError_t launch_attention_d256(const AttnParams& p, int grid, int nb, bool scores_only, cudaStream_t stream) {
  if (nb == 1)
    return scores_only ? launch_one<1, true, 4, 0, kHeadDimWide>(p, grid, stream)
                       : launch_one<1, false, 4, 0, kHeadDimWide>(p, grid, stream);
  return scores_only ? launch_one<2, true, 4, 0, kHeadDimWide>(p, grid, stream)
                     : launch_one<2, false, 4, 0, kHeadDimWide>(p, grid, stream);
}

}  // namespace da
