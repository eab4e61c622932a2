// oproj_umma.cu -- output projection on the 5th-generation tensor cores (tcgen05,
// accumulator in TMEM) for batches where it is a real dense contraction:
//   y[b][n] = sum_k x[b][k] * W[k][n]   (bf16 operands, fp32 accumulation, bf16 out)
// the page's `result = matmul(attn_output_flat, o_weight, DT_BF16)` (page "PyPTO
// 开箱性能调优实战 Decode Attention 多 Matmul 独立 TileShape 配置 F-16", section
// "代码对比"; output_proj row of its shape table: M = batch, K = N = hidden).
//
// Swap-AB: the MMA computes y^T[n][b] = W^T[n][k] . x^T[k][b], so the MMA's M is
// 128 hidden columns and its N is the batch (padded to 16/32/64/128 rows with
// TMA zero fill). W is [K][N] row-major, i.e. the A operand is MN-major: two TMA
// boxes of 64 columns x 64 k-rows (128-byte swizzle) per stage form its canonical
// layout (leading byte offset = distance between the two 64-column atoms, stride
// byte offset = 1024 between groups of eight k-rows). x is K-major (canonical
// 128-byte swizzled rows). One thread issues tcgen05.mma, tcgen05.commit frees
// each stage, and the four warps read the fp32 accumulator out of TMEM.
// The split-K slices of a column tile form a thread-block cluster and sum their fp32
// tiles through distributed shared memory in a fixed order (more than eight slices, on
// request only: through global partials and the CTA that completes the tile last).
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace da {
namespace {

// Two CTAs per SM: each keeps about 100 KB of W in flight (more stages for narrow batches).
template <int NPAD>
struct UmmaCfg {
  static constexpr int kABytes = kUmmaBM * kUmmaBK * 2;  // 16 KB: two 64-column boxes
  static constexpr int kBBytes = NPAD * kUmmaBK * 2;
  static constexpr int kStage = kABytes + ((kBBytes + 1023) / 1024) * 1024;
  static constexpr int kStages = NPAD <= 16 ? 6 : (NPAD <= 32 ? 5 : (NPAD <= 64 ? 4 : 3));
  static constexpr int kTmemCols = NPAD < 32 ? 32 : NPAD;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + (2 * kStages + 1) * 8 + 16;
  static_assert(kSmem <= 113 * 1024, "two CTAs per SM");
  static_assert((size_t)kStages * kStage >= (size_t)NPAD * kUmmaBM * 4, "the fp32 tile fits the ring");
};

template <int NPAD>
__global__ void __launch_bounds__(kUmmaThreads, 2) oproj_umma_kernel(const __grid_constant__ UmmaParams p) {
  using C = UmmaCfg<NPAD>;
  constexpr uint32_t kIdesc = umma_idesc_bf16(kUmmaBM, NPAD, /*A MN-major*/ true, /*B K-major*/ false);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);  // full[S], empty[S], accum
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 1);
  int* flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::kStages + s); };
  const uint32_t accum_bar = smem_u32(bars + 2 * C::kStages);

  const int mt = blockIdx.x, ks = blockIdx.y, bz = blockIdx.z;
  const int n0 = mt * kUmmaBM, b0 = bz * NPAD;
  const int nkb = (p.K + kUmmaBK - 1) / kUmmaBK;
  const int kb0 = (int)((long long)ks * nkb / p.ksplit);
  const int nk = (int)((long long)(ks + 1) * nkb / p.ksplit) - kb0;  // >= 1: the host keeps ksplit <= nkb

  if (warp == 0) {
    if (lane == 0) {  // fetch the tensor maps while TMEM and the barriers are set up
      prefetch_tensormap(&p.tm_w);
      prefetch_tensormap(&p.tm_x);
    }
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accum_bar, 1);
    *flag = 0;
    fence_barrier_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&p.tm_w);
      prefetch_tensormap(&p.tm_x);
      const uint32_t ring = smem_u32(smem);
      const int pre = nk < C::kStages ? nk : C::kStages;
      // W does not depend on the attention kernel: fill the first stages with it
      // before waiting for that grid (programmatic dependent launch).
      for (int it = 0; it < pre; ++it) {
        const uint32_t a = ring + it * C::kStage;
        const int k0 = (kb0 + it) * kUmmaBK;
        mbar_arrive_expect_tx(full_bar(it), C::kABytes + C::kBBytes);
        tma_load_2d(a, &p.tm_w, full_bar(it), n0, k0);
        tma_load_2d(a + kUmmaBK * 128, &p.tm_w, full_bar(it), n0 + 64, k0);
      }
      // ... and pull the rest of this CTA's W slice into L2, so that the refills after
      // the wait come from L2 while the attention kernel's last CTAs still run.
      if (p.prefetch)
        for (int it = pre; it < nk; ++it) {
          tma_prefetch_2d(&p.tm_w, n0, (kb0 + it) * kUmmaBK);
          tma_prefetch_2d(&p.tm_w, n0 + 64, (kb0 + it) * kUmmaBK);
        }
      pdl_wait_primary();
      for (int it = 0; it < pre; ++it)
        tma_load_2d(ring + it * C::kStage + C::kABytes, &p.tm_x, full_bar(it), (kb0 + it) * kUmmaBK, b0);
      for (int it = pre; it < nk; ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        mbar_wait_bounded(empty_bar(s), ph ^ 1, p.err, kErrWaitEmpty, nullptr);
        const uint32_t a = ring + s * C::kStage;
        const int k0 = (kb0 + it) * kUmmaBK;
        mbar_arrive_expect_tx(full_bar(s), C::kABytes + C::kBBytes);
        tma_load_2d(a, &p.tm_w, full_bar(s), n0, k0);
        tma_load_2d(a + kUmmaBK * 128, &p.tm_w, full_bar(s), n0 + 64, k0);
        tma_load_2d(a + C::kABytes, &p.tm_x, full_bar(s), k0, b0);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t ring = smem_u32(smem);
      for (int it = 0; it < nk; ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        mbar_wait_bounded(full_bar(s), ph, p.err, kErrWaitFull, nullptr);
        tc_fence_after_sync();
        const uint32_t a = ring + s * C::kStage;
        const uint32_t bsm = a + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < kUmmaBK / 16; ++kk) {
          // A: 16 k-rows per MMA = two 8-row groups (1024 B apart); the second 64-column
          // atom sits 64 rows x 128 B further. B: 16 k = 32 bytes along each 128-byte row.
          const uint64_t adesc = umma_smem_desc(a + kk * 16 * 128, kUmmaBK * 128, 1024);
          const uint64_t bdesc = umma_smem_desc(bsm + kk * 32, 16, 1024);
          umma_bf16(tmem, adesc, bdesc, kIdesc, (it | kk) != 0);
        }
        umma_commit(empty_bar(s));  // the stage is free once these MMAs have read it
      }
      umma_commit(accum_bar);
    }
  }
  __syncwarp();

  // ------------------------------------------------------------- epilogue
  mbar_wait_bounded(accum_bar, 0, p.err, kErrWaitMma, nullptr);
  tc_fence_after_sync();
  const int n = n0 + warp * 32 + lane;  // TMEM lane = hidden column within the tile
  float acc[NPAD];
#pragma unroll
  for (int c = 0; c < NPAD / 16; ++c) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(tmem + ((uint32_t)(warp * 32) << 16) + c * 16, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[c * 16 + i] = __uint_as_float(r[i]);
  }
  const bool n_ok = n < p.N;
  if (p.ksplit == 1) {
#pragma unroll
    for (int b = 0; b < NPAD; ++b)
      if (n_ok && b0 + b < p.B) p.y[(long long)(b0 + b) * p.y_sb + n] = __float2bfloat16_rn(acc[b]);
  } else if (p.cluster) {
    // The k-slices of this column tile are one cluster: their fp32 tiles meet in
    // distributed shared memory, red[b][m] in the ring (free: every MMA has completed,
    // so every stage was consumed). CTA r of the cluster sums its share of the outputs
    // over the slices in slice order (deterministic) and writes bf16.
    float* red = reinterpret_cast<float*>(smem);
    static_assert(NPAD * kUmmaBM * 4 <= C::kStages * C::kStage, "the fp32 tile fits the ring");
#pragma unroll
    for (int b = 0; b < NPAD; ++b) red[b * kUmmaBM + warp * 32 + lane] = acc[b];
    cluster_sync();  // every slice's tile is in its CTA's shared memory
    const int rank = (int)cluster_ctarank();
    const int nb_valid = p.B - b0 < NPAD ? p.B - b0 : NPAD;
    // shares of four consecutive outputs (one row of the tile: 128 is a multiple of 4), read
    // as 16-byte vectors from the slices that exist (2, 4 or at most 8 of them)
    const int total = nb_valid * kUmmaBM, chunk = ((total + p.ksplit - 1) / p.ksplit + 3) & ~3;
    const int o_end = min(total, (rank + 1) * chunk);
    const uint32_t red_u32 = smem_u32(red);
    const bool red_ok = in_bounds(p.ksplit <= kMaxClusterSplit && rank < p.ksplit && o_end <= NPAD * kUmmaBM, p.err);
    auto reduce = [&](auto ks_max) {
      constexpr int KS = decltype(ks_max)::value;
      for (int o = rank * chunk + 4 * tid; red_ok && o < o_end; o += 4 * kUmmaThreads) {
        float4 v[KS];
#pragma unroll
        for (int q = 0; q < KS; ++q) v[q] = ld_cluster_f32x4(cluster_map(red_u32 + 4u * o, (uint32_t)min(q, p.ksplit - 1)));
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // slices added in order
#pragma unroll
        for (int q = 0; q < KS; ++q)
          if (q < p.ksplit) {
            s0 += v[q].x;
            s1 += v[q].y;
            s2 += v[q].z;
            s3 += v[q].w;
          }
        const int b = o / kUmmaBM, nn = n0 + o % kUmmaBM;  // nn, N multiples of 4: all four or none
        if (nn < p.N && in_bounds(b0 + b < p.B, p.err)) {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(s0, s1), hi = __floats2bfloat162_rn(s2, s3);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(p.y + (long long)(b0 + b) * p.y_sb + nn) = pk;
        }
      }
    };
    if (p.ksplit <= 2) reduce(std::integral_constant<int, 2>());
    else if (p.ksplit <= 4) reduce(std::integral_constant<int, 4>());
    else reduce(std::integral_constant<int, kMaxClusterSplit>());
    cluster_sync();  // no CTA leaves while another still reads its shared memory
  } else {
#pragma unroll
    for (int b = 0; b < NPAD; ++b)
      if (n_ok && b0 + b < p.B && in_bounds(ks < p.ksplit && p.part != nullptr, p.err))
        p.part[((long long)ks * p.B + b0 + b) * p.N + n] = acc[b];
    __syncthreads();  // every thread's partial stores precede the release below
    int* counter = p.counters + blockIdx.z * gridDim.x + mt;
    if (tid == 0) *flag = (atomic_add_acq_rel_gpu(counter, 1) == p.ksplit - 1);
    __syncthreads();
    if (*flag) {  // last k-slice of this column tile: sum all slices in order
      const int nb_valid = p.B - b0 < NPAD ? p.B - b0 : NPAD;
      const int nc = n_ok ? n : p.N - 1;
      // batch rows in chunks of up to 32; per pass about 64 loads from clamped (always
      // valid) addresses are in flight, masked afterwards; slices are added in order
      constexpr int kChunk = NPAD < 32 ? NPAD : 32;
      constexpr int kSlices = 64 / kChunk;
      for (int bc = 0; bc < nb_valid; bc += kChunk) {
        float sum[kChunk];
#pragma unroll
        for (int b = 0; b < kChunk; ++b) sum[b] = 0.f;
        for (int s0 = 0; s0 < p.ksplit; s0 += kSlices) {
          float v[kSlices][kChunk];
#pragma unroll
          for (int u = 0; u < kSlices; ++u) {
            const int sl = min(s0 + u, p.ksplit - 1);
#pragma unroll
            for (int b = 0; b < kChunk; ++b)
              v[u][b] = __ldcg(p.part + ((long long)sl * p.B + b0 + min(bc + b, nb_valid - 1)) * p.N + nc);
          }
#pragma unroll
          for (int u = 0; u < kSlices; ++u)
#pragma unroll
            for (int b = 0; b < kChunk; ++b) sum[b] += (s0 + u < p.ksplit) ? v[u][b] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kChunk; ++b)
          if (n_ok && bc + b < nb_valid) p.y[(long long)(b0 + bc + b) * p.y_sb + n] = __float2bfloat16_rn(sum[b]);
      }
      if (tid == 0) *counter = 0;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

template <int NPAD>
cudaError_t launch_npad(const UmmaParams& p, bool pdl, cudaStream_t stream) {
  using C = UmmaCfg<NPAD>;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(oproj_umma_kernel<NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    // all of the unified L1 as shared memory: two CTAs per SM (a smaller carveout fits one,
    // and the clusters that do not fit wait for a second wave)
    e = cudaFuncSetAttribute(oproj_umma_kernel<NPAD>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.N + kUmmaBM - 1) / kUmmaBM, p.ksplit, (p.B + NPAD - 1) / NPAD);
  cfg.blockDim = dim3(kUmmaThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // the k-slices of a column tile
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = p.cluster ? p.ksplit : 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, oproj_umma_kernel<NPAD>, p);
}

}  // namespace

size_t umma_smem_bytes(int npad) {
  switch (npad) {
    case 16: return UmmaCfg<16>::kSmem;
    case 32: return UmmaCfg<32>::kSmem;
    case 64: return UmmaCfg<64>::kSmem;
    default: return UmmaCfg<128>::kSmem;
  }
}

cudaError_t launch_umma(const UmmaParams& p, int npad, bool pdl, cudaStream_t stream) {
  switch (npad) {
    case 16: return launch_npad<16>(p, pdl, stream);
    case 32: return launch_npad<32>(p, pdl, stream);
    case 64: return launch_npad<64>(p, pdl, stream);
    default: return launch_npad<128>(p, pdl, stream);
  }
}

}  // namespace da
