// oproj_gemv.cu -- output projection for small batches on the CUDA cores:
//   y[b][n] = sum_k x[b][k] * W[k][n]   (bf16 operands, fp32 accumulation, bf16 out)
// the page's `result = matmul(attn_output_flat, o_weight, DT_BF16)` (page "PyPTO
// 开箱性能调优实战 Decode Attention 多 Matmul 独立 TileShape 配置 F-16", section
// "代码对比"; output_proj row of the shape table: M = batch, K = N = 4096).
//
// With M = batch <= 8 the product is a skinny GEMV whose cost is reading W once:
//  * each CTA owns 256 columns and a k-slice of W; a warp reads whole 512-byte row
//    segments (one 16-byte streaming load per lane), all batch rows reuse each load;
//  * the first loads of W are issued before the wait on the attention kernel
//    (programmatic dependent launch), so the W stream overlaps its tail;
//  * split-K partials are summed in a fixed order by the CTA that completes a
//    column block last (atomic counter, no waiting), so results are deterministic.
#include "kernels.h"
#include "ptx.cuh"

namespace da {
namespace {

template <int BT>
struct GemvCfg {
  static constexpr int U = BT <= 2 ? 8 : (BT == 4 ? 6 : 4);  // rows in flight per lane
};

template <int BT>
__global__ void __launch_bounds__(kGemvThreads, 2) oproj_gemv_kernel(const __grid_constant__ GemvParams p) {
  constexpr int U = GemvCfg<BT>::U;
  extern __shared__ float gsm[];
  float* xs = gsm;                   // [BT][kc]
  float* red = gsm + BT * p.kc;      // [8 warps][256]
  int* flag = reinterpret_cast<int*>(red + 8 * kGemvCols);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cb = blockIdx.x, ks = blockIdx.y, b0 = blockIdx.z * BT;
  const int col0 = cb * kGemvCols;
  const int col = col0 + lane * 8;
  const bool col_ok = col < p.N;
  const int k_begin = ks * p.kc;
  const int k_end = min(p.K, k_begin + p.kc);

  // W does not depend on the attention kernel: start streaming it right away.
  uint4 wv[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int kr = k_begin + warp + 8 * u;
    wv[u] = (kr < k_end && col_ok) ? ldg_stream_v4(p.w + (long long)kr * p.w_sk + col) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait_primary();
  for (int i = tid; i < BT * p.kc; i += kGemvThreads) {
    const int b = i / p.kc, kk = i - b * p.kc;
    float v = 0.f;
    if (b0 + b < p.B && k_begin + kk < k_end) v = __bfloat162float(p.x[(long long)(b0 + b) * p.x_sb + k_begin + kk]);
    xs[i] = v;
  }
  __syncthreads();

  float acc[BT][8];
#pragma unroll
  for (int b = 0; b < BT; ++b)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[b][e] = 0.f;

  for (int k = k_begin + warp; k < k_end; k += 8 * U) {
    uint4 nx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kr = k + 8 * U + 8 * u;
      nx[u] = (kr < k_end && col_ok) ? ldg_stream_v4(p.w + (long long)kr * p.w_sk + col) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kr = k + 8 * u;
      if (kr < k_end) {
        const uint32_t wr[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
        float wf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          wf[2 * e] = bf16lo_to_f32(wr[e]);
          wf[2 * e + 1] = bf16hi_to_f32(wr[e]);
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          const float xv = xs[b * p.kc + (kr - k_begin)];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[b][e] = fmaf(xv, wf[e], acc[b][e]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) wv[u] = nx[u];
  }

  // reduce the 8 warps' k-subsets, one batch row at a time
  for (int b = 0; b < BT; ++b) {
    float4* r4 = reinterpret_cast<float4*>(red + warp * kGemvCols + lane * 8);
    r4[0] = make_float4(acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
    r4[1] = make_float4(acc[b][4], acc[b][5], acc[b][6], acc[b][7]);
    __syncthreads();
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w * kGemvCols + tid];
    __syncthreads();
    const int c = col0 + tid;
    if (b0 + b < p.B && c < p.N) {
      if (p.ksplit == 1) p.y[(long long)(b0 + b) * p.y_sb + c] = __float2bfloat16_rn(sum);
      else if (in_bounds(ks < p.ksplit && b0 + b < p.B && c < p.N, p.err)) p.part[((long long)ks * p.B + b0 + b) * p.N + c] = sum;
    }
  }
  if (p.ksplit == 1) return;

  __syncthreads();  // every thread's partial stores precede the release below
  int* counter = p.counters + blockIdx.z * gridDim.x + cb;
  if (tid == 0) *flag = (atomic_add_acq_rel_gpu(counter, 1) == p.ksplit - 1);
  __syncthreads();
  if (*flag) {  // last k-slice of this column block: sum all slices in order
    const int c = col0 + tid;
    const bool c_ok = c < p.N;
    float sum[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) sum[b] = 0.f;
    // slice s is added after slice s-1 (a fixed order); eight slices' loads go out together
    // clamped (always valid) addresses: a batch of loads in flight at once, masked afterwards
    const int cc = c_ok ? c : p.N - 1;
    const int bmax = p.B - 1;
    for (int s0 = 0; s0 < p.ksplit; s0 += 8) {
      float v[8][BT];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = min(s0 + u, p.ksplit - 1);
#pragma unroll
        for (int b = 0; b < BT; ++b) v[u][b] = __ldcg(p.part + ((long long)s * p.B + min(b0 + b, bmax)) * p.N + cc);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int b = 0; b < BT; ++b) sum[b] += (s0 + u < p.ksplit) ? v[u][b] : 0.f;
    }
#pragma unroll
    for (int b = 0; b < BT; ++b)
      if (c_ok && b0 + b < p.B) p.y[(long long)(b0 + b) * p.y_sb + c] = __float2bfloat16_rn(sum[b]);
    if (tid == 0) *counter = 0;
  }
}

template <int BT>
cudaError_t launch_bt(const GemvParams& p, bool pdl, cudaStream_t stream) {
  const size_t smem = gemv_smem_bytes(BT, p.kc);
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(oproj_gemv_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gemv_smem_bytes(BT, kGemvMaxKc));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.N + kGemvCols - 1) / kGemvCols, p.ksplit, (p.B + BT - 1) / BT);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, oproj_gemv_kernel<BT>, p);
}

}  // namespace

size_t gemv_smem_bytes(int bt, int kc) { return (size_t)bt * kc * 4 + 8 * kGemvCols * 4 + 16; }

cudaError_t launch_gemv(const GemvParams& p, int bt, bool pdl, cudaStream_t stream) {
  switch (bt) {
    case 1: return launch_bt<1>(p, pdl, stream);
    case 2: return launch_bt<2>(p, pdl, stream);
    case 4: return launch_bt<4>(p, pdl, stream);
    default: return launch_bt<8>(p, pdl, stream);
  }
}

}  // namespace da
