// oproj_stream.cu -- output projection for batches up to 16, streamed while the
// attention kernel finishes:
//   y[b][n] = sum_k x[b][k] * W[k][n]   (bf16 operands, fp32 accumulation, bf16 out)
// the page's `result = matmul(attn_output_flat, o_weight, DT_BF16)` (page "PyPTO
// 开箱性能调优实战 Decode Attention 多 Matmul 独立 TileShape 配置 F-16", section
// "代码对比"; output_proj row of the shape table: M = batch, K = N = 4096).
//
// The product is bound by reading W once, and W does not depend on the attention
// output x. The kernel is launched behind the attention kernel with programmatic
// dependent launch, so its CTAs start on each SM the attention kernel leaves (the
// attention CTAs end over several microseconds) and bring W in before they wait for x:
//  * work unit = 64 columns x 128 k-rows of W (16 KB, one TMA box with 128-byte
//    swizzle); units are laid column block major;
//  * first wave (the first CTA of each SM): exactly nbuf units, all in its shared-memory
//    ring by TMA before griddepcontrol.wait, plus an L2 prefetch of the second wave's
//    units (an equal share each), so all of W streams from HBM during the attention's
//    tail;
//  * second wave (about two more CTAs per SM): the remaining units in contiguous ranges,
//    read from L2 through their own rings;
//  * after the wait, x for the CTA's units goes to shared memory and warp w multiplies
//    columns [16w, 16w + 16) of every unit with mma.sync m16n8k16 (M = 16 columns of
//    W^T read by ldmatrix.trans, N = 8 batch rows, K = 16 k-rows), so what follows the
//    attention is a few microseconds of L2 reads, not a CUDA-core FMA loop;
//  * a CTA writes one fp32 partial per column block it touches; the CTA completing a
//    block last (atomic counter, no waiting) sums the partials in CTA order, so results
//    are deterministic.
#include "kernels.h"
#include "ptx.cuh"

namespace da {
namespace {

static_assert(kStreamThreads == 128 && kStreamCols == 64, "four warps, 16 columns each");

// Unit range of CTA c: the first wave takes nbuf units each, the second wave splits
// the rest evenly (every second-wave range is non-empty: the host keeps n2 <= rest).
struct StreamRange {
  int u0, u1;
};
__device__ __forceinline__ StreamRange stream_range(const StreamParams& p, int c) {
  const int first = min(p.wave1 * p.nbuf, p.units);
  StreamRange r;
  if (c < p.wave1) {
    r.u0 = min(c * p.nbuf, p.units);
    r.u1 = min((c + 1) * p.nbuf, p.units);
  } else {
    const int n2 = (int)gridDim.x - p.wave1, rest = p.units - first, i = c - p.wave1;
    r.u0 = first + (int)((long long)i * rest / n2);
    r.u1 = first + (int)((long long)(i + 1) * rest / n2);
  }
  return r;
}
// CTA whose range holds unit u.
__device__ __forceinline__ int stream_cta_of(const StreamParams& p, int u) {
  const int first = min(p.wave1 * p.nbuf, p.units);
  if (u < first) return u / p.nbuf;
  const int n2 = (int)gridDim.x - p.wave1, rest = p.units - first;
  return p.wave1 + (int)(((long long)(u - first + 1) * n2 - 1) / rest);
}

template <int NT>
__global__ void __launch_bounds__(kStreamThreads, 4) oproj_stream_kernel(const __grid_constant__ StreamParams p) {
  constexpr int NP = 8 * NT;  // batch rows per unit in the x buffer (the MMA's N, padded)
  constexpr int kXP = kStreamXPitch;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nbuf = p.nbuf;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem + (size_t)nbuf * kStreamUnitBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nbuf * kStreamUnitBytes + (size_t)p.umax * NP * kXP * 2);
  int* flag = reinterpret_cast<int*>(bars + nbuf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const StreamRange rg = stream_range(p, blockIdx.x);
  const int nu = rg.u1 - rg.u0;  // >= 1
  const uint32_t ring = smem_u32(smem);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto issue = [&](int i, uint64_t pol) {  // unit u0 + i into buffer i % nbuf
    const int u = rg.u0 + i, cb = u / p.nkc, kc = u - cb * p.nkc;
    const int s = i % nbuf;
    mbar_arrive_expect_tx(full_bar(s), kStreamUnitBytes);
    tma_load_2d_hint(ring + (uint32_t)s * kStreamUnitBytes, &p.tm_w, full_bar(s), cb * kStreamCols,
                     kc * kStreamRows, pol);
  };

  if (tid == 0) {
    for (int s = 0; s < nbuf; ++s) mbar_init(full_bar(s), 1);
    *flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    // W does not depend on the attention output: fill the ring, then pull this CTA's
    // share of the second wave's units into L2, all before waiting for the attention.
    prefetch_tensormap(&p.tm_w);
    const uint64_t pol = l2_policy_evict_first();  // each W byte is read once
    for (int i = 0; i < nu && i < nbuf; ++i) issue(i, pol);
    if (p.prefetch && (int)blockIdx.x < p.wave1) {
      const int first = min(p.wave1 * p.nbuf, p.units), rest = p.units - first, c = blockIdx.x;
      const int v0 = first + (int)((long long)c * rest / p.wave1);
      const int v1 = first + (int)((long long)(c + 1) * rest / p.wave1);
      for (int u = v0; u < v1; ++u) {
        const int cb = u / p.nkc, kc = u - cb * p.nkc;
        tma_prefetch_2d(&p.tm_w, cb * kStreamCols, kc * kStreamRows);
      }
    }
  }
  pdl_wait_primary();  // x is the previous kernel's output

  // x rows of this CTA's units: xs[i][n][kk] = x[n][k0(i) + kk], zero outside [B) x [K)
  constexpr int kChunks = kStreamRows / 8;  // 16-byte chunks per x row of a unit
  for (int idx = tid; idx < nu * NP * kChunks; idx += kStreamThreads) {
    const int i = idx / (NP * kChunks), rem = idx - i * (NP * kChunks), n = rem / kChunks, ch = rem % kChunks;
    const int u = rg.u0 + i, kc = u % p.nkc, k = kc * kStreamRows + ch * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < p.B && k < p.K) v = __ldcg(reinterpret_cast<const uint4*>(p.x + (long long)n * p.x_sb + k));
    *reinterpret_cast<uint4*>(xs + (i * NP + n) * kXP + ch * 8) = v;
  }
  __syncthreads();

  const uint32_t* xs32 = reinterpret_cast<const uint32_t*>(xs);
  // ldmatrix.trans lane roles: matrix q = lane / 8 (k half q / 2, column half q % 2), row li = lane % 8
  const int lq = lane >> 3, li = lane & 7;
  const uint32_t lane_off = (uint32_t)((lq >> 1) * 8 + li) * 128 + (uint32_t)(((2 * warp + (lq & 1)) ^ li) << 4);
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const uint64_t pol = l2_policy_evict_first();

  for (int i = 0; i < nu; ++i) {
    const int u = rg.u0 + i, cb = u / p.nkc;
    const int s = i % nbuf;
    mbar_wait_bounded(full_bar(s), (uint32_t)(i / nbuf) & 1u, p.err, kErrWaitFull, nullptr);
    const uint32_t tile = ring + (uint32_t)s * kStreamUnitBytes + lane_off;
    const uint32_t* xr = xs32 + (i * NP + g) * (kXP / 2) + t;
#pragma unroll
    for (int ks = 0; ks < kStreamRows / 16; ++ks) {
      uint32_t a[4];
      // rows 16ks .. 16ks + 15 (each 128 bytes); the swizzle depends on row % 8 only
      ldsm_x4_trans(tile + (uint32_t)ks * 16 * 128, a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma_bf16_16816(acc[nt], a, xr[nt * 8 * (kXP / 2) + ks * 8], xr[nt * 8 * (kXP / 2) + ks * 8 + 4]);
    }
    __syncthreads();  // every warp is done with buffer s
    if (tid == 0 && i + nbuf < nu) issue(i + nbuf, pol);

    const bool flush = (i == nu - 1) || ((u + 1) / p.nkc != cb);
    if (!flush) continue;
    // ---- this CTA's part of column block cb: lane holds columns 16w + g (+8), rows 8nt + 2t (+1)
    const int c_first = stream_cta_of(p, cb * p.nkc), c_last = stream_cta_of(p, cb * p.nkc + p.nkc - 1);
    const int nparts = c_last - c_first + 1;
    const int col0 = cb * kStreamCols;
    if (nparts == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = col0 + warp * 16 + g + (e >> 1) * 8, b = nt * 8 + 2 * t + (e & 1);
          if (n < p.N && b < p.B) p.y[(long long)b * p.y_sb + n] = __float2bfloat16_rn(acc[nt][e]);
        }
    } else {
      const long long slot = (long long)blockIdx.x + cb;  // unique: ranges are contiguous and ordered
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = warp * 16 + g + (e >> 1) * 8, b = nt * 8 + 2 * t + (e & 1);
          if (b < p.B) p.part[(slot * p.B + b) * kStreamCols + c] = acc[nt][e];
        }
      __syncthreads();  // every thread's partial stores precede the release below
      if (tid == 0) *flag = (atomic_add_acq_rel_gpu(p.counters + cb, 1) == nparts - 1);
      __syncthreads();
      if (*flag) {
        // Last part of this column block: output o = (b, c) for o = tid + 128 j; each output
        // sums its parts in CTA order, the loads of kPC parts x all of this thread's
        // outputs in flight together (clamped, always valid addresses).
        constexpr int kOut = (kStreamCols * NP + kStreamThreads - 1) / kStreamThreads;
        constexpr int kPC = 32 / kOut;  // parts per batch of loads: 32 values in flight
        float sum[kOut];
#pragma unroll
        for (int j = 0; j < kOut; ++j) sum[j] = 0.f;
        const int nout = kStreamCols * p.B;
        for (int q0 = 0; q0 < nparts; q0 += kPC) {
          float v[kPC][kOut];
#pragma unroll
          for (int k = 0; k < kPC; ++k) {
            const long long sl = (long long)c_first + min(q0 + k, nparts - 1) + cb;
#pragma unroll
            for (int j = 0; j < kOut; ++j) {
              const int o = min(tid + kStreamThreads * j, nout - 1);
              v[k][j] = __ldcg(p.part + sl * p.B * kStreamCols + o);
            }
          }
#pragma unroll
          for (int k = 0; k < kPC; ++k)
#pragma unroll
            for (int j = 0; j < kOut; ++j) sum[j] += (q0 + k < nparts) ? v[k][j] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kOut; ++j) {
          const int o = tid + kStreamThreads * j, b = o / kStreamCols, n = col0 + o % kStreamCols;
          if (o < nout && n < p.N) p.y[(long long)b * p.y_sb + n] = __float2bfloat16_rn(sum[j]);
        }
        if (tid == 0) p.counters[cb] = 0;  // ready for the next call
      }
      __syncthreads();  // flag is reused by the next column block
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  }
}

template <int NT>
cudaError_t launch_nt(const StreamParams& p, int grid, size_t smem, bool pdl, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(oproj_stream_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem);
    if (e != cudaSuccess) return e;
    // the same carveout as the attention kernel, so the SMs need no reconfiguration
    e = cudaFuncSetAttribute(oproj_stream_kernel<NT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, oproj_stream_kernel<NT>, p);
}

}  // namespace

size_t stream_smem_bytes(int nt, int nbuf, int umax) {
  return 1024 + (size_t)nbuf * kStreamUnitBytes + (size_t)umax * 8 * nt * kStreamXPitch * 2 + (size_t)nbuf * 8 + 16;
}

cudaError_t launch_stream(const StreamParams& p, int nt, int grid, bool pdl, cudaStream_t stream) {
  const size_t smem = stream_smem_bytes(nt, p.nbuf, p.umax);
  if (smem > kMaxDynSmem || (nt != 1 && nt != 2) || grid < p.wave1 || p.nbuf < 1) return cudaErrorInvalidValue;
  return nt == 1 ? launch_nt<1>(p, grid, smem, pdl, stream) : launch_nt<2>(p, grid, smem, pdl, stream);
}

}  // namespace da
