// attn_decode_fp8.cu -- instantiations of the attention kernel over an fp8 (e4m3) KV
// cache: head dim 128, 128-token tiles in a 4-stage (or, on request, 6-stage) ring of 32 KB stages.
#include "attn_decode.cuh"

namespace da {

cudaError_t launch_attention_fp8(const AttnParams& p, int grid, int nb, cudaStream_t stream) {
  if (attn_stages_for(p.B, nb, p.stages, p.cluster > 1) == kMaxStages)
    return nb == 1 ? launch_one<1, false, kMaxStages, 0, kHeadDim, false, true>(p, grid, stream)
                   : launch_one<2, false, kMaxStages, 0, kHeadDim, false, true>(p, grid, stream);
  return nb == 1 ? launch_one<1, false, 4, 0, kHeadDim, false, true>(p, grid, stream)
                 : launch_one<2, false, 4, 0, kHeadDim, false, true>(p, grid, stream);
}

}  // namespace da
