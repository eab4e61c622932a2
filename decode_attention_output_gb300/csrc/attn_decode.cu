// attn_decode.cu -- instantiations of the attention kernel at head dim 128 (4- or
// 6-stage ring, scores-only variant, fused step) and the dispatch over head dims.
#include "attn_decode.cuh"

namespace da {
namespace {

template <int NB, bool SCORES>
cudaError_t launch_nb(const AttnParams& p, int grid, cudaStream_t stream) {
  if (attn_stages_for(p.B, NB, p.stages, p.cluster > 1) == kMaxStages)
    return launch_one<NB, SCORES, kMaxStages, 0, kHeadDim>(p, grid, stream);
  return launch_one<NB, SCORES, 4, 0, kHeadDim>(p, grid, stream);
}

template <int NB>
cudaError_t launch_fused(const AttnParams& p, int grid, int npad, cudaStream_t stream) {
  switch (npad) {
    case 16: return launch_one<NB, false, 4, 16, kHeadDim>(p, grid, stream);
    case 32: return launch_one<NB, false, 4, 32, kHeadDim>(p, grid, stream);
    case 64: return launch_one<NB, false, 4, 64, kHeadDim>(p, grid, stream);
    default: return launch_one<NB, false, 4, 128, kHeadDim>(p, grid, stream);
  }
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, int grid, int nb, int dim, bool scores_only, cudaStream_t stream,
                             int npad) {
  if (dim == kHeadDimWide) {
    if (npad > 0) return cudaErrorInvalidValue;  // the fused step is built for D = 128 only
    return launch_attention_d256(p, grid, nb, scores_only, stream);
  }
  if (dim != kHeadDim) return cudaErrorInvalidValue;
  if (npad > 0) return nb == 1 ? launch_fused<1>(p, grid, npad, stream) : launch_fused<2>(p, grid, npad, stream);
  if (nb == 1) return scores_only ? launch_nb<1, true>(p, grid, stream) : launch_nb<1, false>(p, grid, stream);
  return scores_only ? launch_nb<2, true>(p, grid, stream) : launch_nb<2, false>(p, grid, stream);
}

int attn_max_active_clusters(int cluster) {
  // The contiguous instance at D = 128 stands for all: every instance holds one CTA per SM.
  const auto kern = attn_decode_kernel<1, false, 4, 0, kHeadDim>;
  const size_t smem = attn_smem_bytes(1, 1, 4, kHeadDim, kStageBytes, true);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(attn_threads(attn_producers(false, false, false)));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace da
