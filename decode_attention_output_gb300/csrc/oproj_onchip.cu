// oproj_onchip.cu -- output projection of a single-row batch with o_weight staged on chip
// while the attention kernel still runs:
//   y[n] = sum_k x[k] * W[k][n]   (bf16 operands, fp32 accumulation, bf16 out)
// the page's `result = matmul(attn_output_flat, o_weight, DT_BF16)` (page "PyPTO 开箱性能
// 调优实战 Decode Attention 多 Matmul 独立 TileShape 配置 F-16", section "代码对比";
// output_proj row of its shape table: M = 1, K = N = 4096).
//
// At batch 1 the attention kernel occupies a few dozen SMs for a few microseconds, and W
// (K x N bf16, 33.5 MB at K = N = 4096) is four fifths of the step's bytes. This kernel is
// launched right behind the attention's set-up (programmatic dependent launch) with one CTA
// of 512 threads per SM that the attention leaves free. Before it waits for the attention
// grid, every CTA stages its share of W on chip, in shared memory (by TMA) and in registers
// (16-byte loads): the free SMs' shared memory plus register files hold all of W. Once the
// attention's output x is complete the CTA reads x into shared memory and does the
// arithmetic, a few hundred FMAs per thread.
//
// Work split: the CTAs form a grid of column groups (kOnchipCols = 512 columns, 1 KB of every
// row of W) by k-ranges; CTA (g, j) owns columns [512 g, 512 g + 512) of k-blocks (64 rows)
// [j * kb / KG, (j + 1) * kb / KG), so that the CTAs of one k-range read whole rows of W
// together. Its first k-blocks land in shared memory (8 TMA boxes of 64 x 64 per k-block),
// the rest in registers. Thread t owns the 8 columns of 16-byte piece t % 8 of column tile
// t / 64, and rows (t / 8) % 8 + 8 i of every k-block; its 8 sums are reduced over the
// rows in the warp and across the two warps of its column tile, and the k-ranges' fp32
// parts of a column group are summed, in k order, by the CTA that completes the group last
// (atomic counter, no waiting), so results are deterministic.
#include "kernels.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kOcBoxBytes = 64 * 64 * 2;             // one TMA box: 64 columns x 64 rows
constexpr int kOcKbBytes = (kOnchipCols / 64) * kOcBoxBytes;  // one k-block of a column group

__device__ __forceinline__ void fma_piece(float (&acc)[8], const uint4& w, float xv) {
  const uint32_t wr[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc[2 * e] = fmaf(xv, bf16lo_to_f32(wr[e]), acc[2 * e]);
    acc[2 * e + 1] = fmaf(xv, bf16hi_to_f32(wr[e]), acc[2 * e + 1]);
  }
}

__global__ void __launch_bounds__(kOnchipThreads, 1) oproj_onchip_kernel(const __grid_constant__ OnchipParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xs = smem + (size_t)p.smem_kblocks * kOcKbBytes;                           // x [K] bf16
  uint64_t* bars = reinterpret_cast<uint64_t*>(xs + ((size_t)p.K * 2 + 15) / 16 * 16);  // [smem k-blocks], x
  int* flag = reinterpret_cast<int*>(bars + p.smem_kblocks + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, j = blockIdx.y, KG = gridDim.y;
  const int kb0 = (int)((long long)j * p.kb / KG), kb1 = (int)((long long)(j + 1) * p.kb / KG);
  const int nk = kb1 - kb0;
  const int ns = min(nk, p.smem_kblocks);  // k-blocks staged in shared memory
  const int nr = nk - ns;                  // k-blocks held in registers (<= kOnchipRegKblocks: the host checks)
  const int n_base = g * kOnchipCols;
  const uint32_t xbar = smem_u32(bars + p.smem_kblocks);
  if (!in_bounds(nr <= kOnchipRegKblocks && n_base + kOnchipCols <= p.N, p.err)) return;  // (checked build)

  if (tid == 0) {
    prefetch_tensormap(&p.tm_w);
    for (int i = 0; i < ns; ++i) mbar_init(smem_u32(bars + i), 1);
    mbar_init(xbar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // W does not depend on the attention kernel: stage this CTA's k-blocks now.
  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_arrive_expect_tx(smem_u32(bars + i), kOcKbBytes);
      for (int ct = 0; ct < kOnchipCols / 64; ++ct)
        tma_load_2d(smem_u32(smem + (size_t)i * kOcKbBytes + ct * kOcBoxBytes), &p.tm_w, smem_u32(bars + i),
                    n_base + ct * 64, (kb0 + i) * 64);
    }
  }
  const int pc = tid & 7, ro = (tid >> 3) & 7, ct = tid >> 6;  // piece, row offset, column tile
  const int col = n_base + ct * 64 + pc * 8;                     // first of this thread's 8 columns
  uint4 wr[kOnchipRegKblocks][8];
#pragma unroll
  for (int i = 0; i < kOnchipRegKblocks; ++i)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      wr[i][q] = make_uint4(0, 0, 0, 0);
      if (i < nr) wr[i][q] = ldg_stream_v4(p.w + (long long)((kb0 + ns + i) * 64 + ro + 8 * q) * p.w_sk + col);
    }
  // The attention's output is complete (and visible) once its grid has completed.
  pdl_wait_primary();
  if (tid == 0) {
    mbar_arrive_expect_tx(xbar, (uint32_t)p.K * 2);
    bulk_load(smem_u32(xs), p.x, (uint32_t)p.K * 2, xbar);
  }
  mbar_wait_bounded(xbar, 0, p.err, kErrWaitFull, nullptr);
  const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(xs);

  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int i = 0; i < ns; ++i) {
    mbar_wait_bounded(smem_u32(bars + i), 0, p.err, kErrWaitFull, nullptr);
    const uint8_t* box = smem + (size_t)i * kOcKbBytes + ct * kOcBoxBytes;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int r = ro + 8 * q;
      // (a box lands with the tensor map's 128-byte swizzle: chunk pc of row r sits at pc ^ (r % 8))
      const uint4 w = *reinterpret_cast<const uint4*>(box + r * 128 + ((pc ^ (r & 7)) << 4));
      fma_piece(acc, w, __bfloat162float(xv[(kb0 + i) * 64 + r]));
    }
  }
#pragma unroll
  for (int i = 0; i < kOnchipRegKblocks; ++i)
    if (i < nr) {
#pragma unroll
      for (int q = 0; q < 8; ++q) fma_piece(acc, wr[i][q], __bfloat162float(xv[(kb0 + ns + i) * 64 + ro + 8 * q]));
    }
  // The 8 row offsets of a piece: lanes pc + 8 m of a warp (m = 0..3), then the column
  // tile's two warps through shared memory (the staged k-blocks are consumed: their space is free).
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 8);
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 16);
  }
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [2 warps of a tile][512 columns]
  if (lane < 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) red[(warp & 1) * kOnchipCols + ct * 64 + pc * 8 + e] = acc[e];
  }
  __syncthreads();
  const float sum = red[tid] + red[kOnchipCols + tid];  // column n_base + tid
  const int n = n_base + tid;
  if (KG == 1) {
    p.y[n] = __float2bfloat16_rn(sum);
    return;
  }
  // the k-ranges' parts of this column group, summed in k order by the CTA that completes it last
  p.part[((long long)g * KG + j) * kOnchipCols + tid] = sum;
  __syncthreads();  // every part store precedes the release below
  if (tid == 0) *flag = atomic_add_acq_rel_gpu(p.counters + g, 1) == KG - 1;
  __syncthreads();
  if (*flag) {
    float t = 0.f;
    for (int q = 0; q < KG; ++q) t += __ldcg(p.part + ((long long)g * KG + q) * kOnchipCols + tid);
    p.y[n] = __float2bfloat16_rn(t);
    if (tid == 0) p.counters[g] = 0;  // ready for the next call
  }
}

}  // namespace

size_t onchip_smem_bytes(int smem_kblocks, int K) {
  return 1024 + (size_t)smem_kblocks * kOcKbBytes + ((size_t)K * 2 + 15) / 16 * 16 + (size_t)(smem_kblocks + 1) * 8 + 16;
}

int onchip_max_smem_kblocks(int K) {
  int n = 0;
  while (onchip_smem_bytes(n + 1, K) <= kMaxDynSmem) ++n;
  return n;
}

cudaError_t launch_onchip(const OnchipParams& p, int kgroups, bool pdl, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(oproj_onchip_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(oproj_onchip_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.N / kOnchipCols, kgroups);
  cfg.blockDim = dim3(kOnchipThreads);
  cfg.dynamicSmemBytes = onchip_smem_bytes(p.smem_kblocks, p.K);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, oproj_onchip_kernel, p);
}

}  // namespace da
