// kernels.h -- parameter blocks and launchers shared by the C-ABI layer (api.cu)
// and the kernels. Host and device code both include it; it holds no method
// arithmetic beyond the tiling constants.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace da {

// ----------------------------------------------------------- split-KV attention
constexpr int kHeadDim = 128;
constexpr int kTile = 64;                       // tokens per pipeline stage
constexpr int kConsumerWarps = 4;               // each owns 16 tokens of a stage
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;  // + one TMA producer warp
constexpr int kStages = 4;
constexpr int kHalfBytes = kTile * 128;         // 64 tokens x 64 dims x bf16 (one 128B-swizzled box)
constexpr int kKTileBytes = 2 * kHalfBytes;     // 64 tokens x 128 dims
constexpr int kStageBytes = 2 * kKTileBytes;    // K tile + V tile
constexpr int kQRowBytes = 272;                 // 256 B of q + 16 B pad (conflict-free fragment loads)
constexpr int kMaxGroup = 16;
constexpr int kMaxBatch = 1024;
constexpr int kQSlotBytes = kMaxGroup * kQRowBytes;
constexpr int kMergeRow = 132;                  // floats per head row of the merge scratch (128 + pad)

constexpr size_t attn_smem_bytes(int batch) {
  return 1024                                                  // alignment slack
         + (size_t)kStages * kStageBytes                       // K/V ring
         + (size_t)kStages * kQSlotBytes                       // q rows per stage
         + (size_t)kConsumerWarps * kMaxGroup * kMergeRow * 4  // per-warp O
         + (size_t)kConsumerWarps * kMaxGroup * 2 * 4          // per-warp (m, l)
         + (size_t)2 * kStages * 8                             // full/empty barriers
         + 16                                                  // flags
         + (size_t)(batch + 1) * 4;                            // tile prefix over the batch
}

struct AttnParams {
  CUtensorMap tm_k;  // [B][Hkv][Lcap][128] bf16, box 64 dims x 64 tokens, 128B swizzle
  CUtensorMap tm_v;
  const __nv_bfloat16* q;
  long long q_sb, q_sh;  // element strides of q [B][Hq][128]
  const int* seq_lens;
  __nv_bfloat16* attn;   // [B][Hq][128] bf16 result
  long long a_sb, a_sh;
  float* scores;         // [B][Hq][Lcap] fp32 (scores-only mode)
  long long s_sb, s_sh;
  float* part_o;         // [slots][gpad][128] unnormalised partial outputs
  float* part_ml;        // [slots][gpad][2]   (running max in log2 units, sum)
  int* counters;         // [B*Hkv] completion counters (zero between calls)
  int* err;              // device error word
  int B, Hkv, G, Lcap;
  int gpad;              // 8 or 16 (heads per group rounded up to the MMA width)
  float scale_log2;      // scale * log2(e)
};

// grid = number of persistent CTAs; nb = 1 for G <= 8, 2 for G <= 16.
cudaError_t launch_attention(const AttnParams& p, int grid, int nb, bool scores_only, cudaStream_t stream);

// ------------------------------------------------------- projection: GEMV path
constexpr int kGemvThreads = 256;
constexpr int kGemvCols = 256;  // 32 lanes x 8 columns
constexpr int kGemvMaxKc = 1024;

struct GemvParams {
  const __nv_bfloat16* x;  // [B][K]
  long long x_sb;
  const __nv_bfloat16* w;  // [K][N] row-major
  long long w_sk;
  __nv_bfloat16* y;        // [B][N]
  long long y_sb;
  float* part;             // [ksplit][B][N] fp32 split-K partials
  int* counters;           // [batch chunks][column blocks]
  int B, K, N, kc, ksplit;
};

// bt = batch rows per CTA (1, 2, 4 or 8); grid = (col blocks, ksplit, batch chunks).
cudaError_t launch_gemv(const GemvParams& p, int bt, bool pdl, cudaStream_t stream);
size_t gemv_smem_bytes(int bt, int kc);

}  // namespace da
