// attn_decode.cuh -- persistent split-KV decode attention for sm_103a (the kernel
// template; attn_decode.cu instantiates head dim 128 and the fused step,
// attn_decode_d256.cu head dim 256, attn_decode_paged.cu the paged cache,
// attn_decode_fp8.cu the fp8 cache).
//
// Computes, for every batch row b and query head h (KV head j = h / G),
//   S = q . K^T over t < L_b (the page's scores_fp32, fp32),
//   P = softmax(scale * S),  O = P . V  (the page's attn_output, bf16),
// the three-matmul decode attention of the page "PyPTO 开箱性能调优实战 Decode
// Attention 多 Matmul 独立 TileShape 配置 F-16", section "代码对比", with the
// QK^T and attn.V shapes of its table "三个 Matmul 的 Shape 特征分析".
//
// Design (GB300):
//  * Work unit = one tile of one (batch, KV-head) sequence: 32 KB of K+V (64 tokens at
//    D = 128, 32 at D = 256, 128 with an fp8 cache). All tiles of the batch are laid
//    end to end and each persistent CTA takes an equal, contiguous range of them, so
//    ragged batches stay balanced. A range may end or start inside a sequence: each
//    CTA emits one partial (m, l, O) per sequence it touches; the CTA that finishes a
//    sequence last (an atomic completion counter, no waiting) merges the partials with
//    the log-sum-exp rule and writes bf16.
//  * Start-up: the set-up warp scans the lengths, computes this CTA's range and the cursor
//    at its first tile (division by the worker count as a host-computed multiply and shift,
//    a warp ballot for the batch row) and copies the first tile of each consumer group
//    itself; the consumers read the range's first q straight from global memory.
//  * Two producer lanes, one per consumer group (tiles of alternating parity), stream K
//    and V tiles with one 5-D TMA copy per tile and tensor (the head dim split into
//    128-byte rows of 64-dim boxes, 128-byte swizzle) into a 4-stage shared-memory ring
//    guarded by mbarriers; q rows arrive by 1-D bulk copy with the first tiles of a
//    sequence that starts inside the range.
//    A paged cache is read in boxes of min(block size, tile) tokens, the block ids
//    arriving by TMA a few tiles ahead.
//  * Cluster mode (where there is room for two or more CTAs per sequence): the grid is
//    launched in thread-block clusters. With equal lengths every sequence gets the CTAs
//    of one cluster, which merge their partial states through distributed shared memory
//    after a cluster barrier instead of through L2; with unequal lengths the kernel keeps
//    the flat split and the L2 merge, and no CTA waits at a cluster barrier.
//  * Programmatic dependent launch: the kernel waits for the previous kernel in the
//    stream before its first global access, and lets the next one launch right after its
//    set-up, or, when the projection follows, a few tiles before the end of its range.
//  * Two consumer groups of four warps take alternate stages, so two tiles are
//    in compute at once per SM. Each warp owns 16 tokens of a stage and all G
//    query heads of the group (every K/V byte is read once). S^T = K . Q^T runs
//    on mma.sync m16n8k16 with tokens as M and heads as N (G <= 8 fills one
//    8-wide N block); the online softmax runs in registers (a lagging reference
//    maximum, see kSlack, a running sum, exp2 with scale*log2e folded); P is
//    rounded to bf16 and moved into the B-operand layout with movmatrix;
//    O^T = V^T . P^T accumulates
//    in fp32 registers. At the end of a sequence segment the eight warps' states
//    are merged (pairwise in registers, then across four warps in shared memory).
//  * D = 256 (a GQA decode whose QK^T contracts D in two 128-wide halves and whose
//    attn.V has N = D split in two, page "PyPTO 开箱性能调优实战 Decode Attention
//    多 Matmul 独立 TileShape 配置 F-16", section "仓库源码佐证"): the warps of a group
//    pair up on 16 tokens; both compute the 16 x G scores over all 256 dims (the
//    tensor pipe is mostly idle, so the duplicate QK^T is cheap) and hence the same
//    softmax state, and each accumulates one 128-dim half of O. Registers per
//    thread stay those of D = 128 except the q fragments, which double.
//  * fp8 (e4m3) cache: a warp owns 32 tokens (two 16-row halves, one softmax update);
//    codes are widened to f16 in registers (exact) for f16 MMAs, q and P in f16.
#pragma once
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace da {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
// Online softmax with a lagging reference: a warp takes its weights 2^(x - m) against a
// running reference m that moves to the running maximum (rescaling l and O) only when a
// score of the tile exceeds it by more than kSlack (log2 units). Weights then stay at or
// below 2^kSlack, and most tiles skip the maximum's shuffle reduction and the rescale.
// Every merge takes a part's reference as its m: the result does not depend on it.
constexpr float kSlack = 8.f;

// Position of the current tile in the flattened tile order.
struct Cursor {
  int b, kvh, j, nt;  // batch row, KV head, tile index in the sequence, tiles in the sequence
};

// Advances to the next tile (only called while one exists); prefix[b] = KV heads x tiles of
// all batch rows before b, prefix[B] = total tiles.
__device__ __forceinline__ void cursor_next(Cursor& c, const int* prefix, int B, int Hkv) {
  if (++c.j < c.nt) return;
  c.j = 0;
  if (++c.kvh < Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
  } while (c.b < B - 1 && prefix[c.b + 1] == prefix[c.b]);
  c.nt = (prefix[c.b + 1] - prefix[c.b]) / Hkv;
}

// floor(n / d) for 0 <= n < 2^31 from the host's m = ceil(2^s / d), s = 31 + ceil(log2 d):
// n m / 2^s exceeds n / d by less than n / 2^s < 1 / d, too little to reach the next integer.
__device__ __forceinline__ unsigned div_mul(unsigned n, unsigned long long m, int s) {
  return (unsigned)(((unsigned long long)n * m) >> s);
}

// floor(a / b) for 0 <= a < 2^31, b > 0 and a quotient below 2^16: the float quotient's
// relative error (two roundings to float and a 2-ulp division) stays below 2^-21, so it lies
// within 0.05 of a / b and one step either way corrects its truncation.
__device__ __forceinline__ int div_small(int a, int b) {
  int q = (int)__fdividef((float)a, (float)b);
  const long long r = (long long)a - (long long)q * b;
  if (r < 0) --q;
  else if (r >= b) ++q;
  return q;
}

// Tiles of a range [start, end) copied by the set-up warp (contiguous caches): the first, and
// the second when it lies in the same sequence (its first tile at j, of nt).
__device__ __forceinline__ int early_tiles(long long start, long long end, int j, int nt) {
  return end - start >= 2 && j + 1 < nt ? 2 : (end > start ? 1 : 0);
}

// CTA whose range [i*T/P, (i+1)*T/P) holds tile x.
__device__ __forceinline__ int cta_of(long long x, long long T, int P) {
  return (int)(((x + 1) * (long long)P - 1) / T);
}

__device__ __forceinline__ int clamp_len(int L, int Lcap) { return L < 0 ? 0 : (L > Lcap ? Lcap : L); }

// Keep the bf16 halves of v whose token index (tok for the low half, tok + 1 for
// the high half) is below `valid`.
__device__ __forceinline__ uint32_t mask_tokens(uint32_t v, int tok, int valid) {
  const uint32_t lo = tok < valid ? 0x0000ffffu : 0u;
  const uint32_t hi = tok + 1 < valid ? 0xffff0000u : 0u;
  return v & (lo | hi);
}

// ---------------------------------------------------------------- fused step
// Phase B of the fused step projects the attention output X [B][K] with W_o [K][N]
// on tcgen05: y^T[n][b] = W_o^T[n][k] . X^T[k][b] (swap-AB: M = 128 hidden columns,
// N = batch padded to NPAD). Work unit = one column tile (128 columns) x one 64-row
// k-block of W_o; the units are laid end to end (column tile major) and each CTA
// takes an equal contiguous range, so a CTA covers at most two column tiles (the
// host checks it) and accumulates each in its own TMEM region.
struct ProjSplit {
  int PB;             // CTAs with phase-B work
  long long u0, u1;   // this CTA's units
};

__device__ __forceinline__ ProjSplit proj_split(const AttnParams& p, int cta) {
  ProjSplit r;
  r.PB = min((int)gridDim.x, p.units);
  r.u0 = cta < r.PB ? (long long)cta * p.units / r.PB : 0;
  r.u1 = cta < r.PB ? (long long)(cta + 1) * p.units / r.PB : 0;
  return r;
}

// Waits until n CTAs have arrived (bounded), then counts this CTA's departure; the
// last one to leave resets both counters for the next launch. A CTA that gives up
// records kErrGridSync and carries on without counting its departure (the host's error
// query then resets the counters): the rest of its pipeline is intact, so every later
// wait of the kernel still ends, and only the result is invalid.
__device__ __forceinline__ bool grid_barrier_wait(int* sync, int n, int* err, unsigned long long limit_ns) {
  const unsigned long long t0 = globaltimer_ns();
  while (ld_acquire_gpu(sync) < n) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrGridSync);
      return false;
    }
    __nanosleep(64);
  }
  if (atomic_add_acq_rel_gpu(sync + 1, 1) == n - 1) {
    sync[0] = 0;
    sync[1] = 0;
  }
  return true;
}

// Phase-B producer: refills the (now free) K/V ring with W_o tiles right away, and
// with X tiles once the grid barrier says every attention output is written.
template <int NPAD, int S>
__device__ void fused_producer(const AttnParams& p, uint32_t ring, uint64_t* bars, int it_a, int* flags) {
  constexpr uint32_t kXBytes = NPAD * 128;  // NPAD rows x 64 k x bf16
  constexpr int SB = proj_stages(NPAD), kStageB = proj_stage_bytes(NPAD);
  auto empty_a = [&](int s) { return smem_u32(bars + S + s); };
  auto full_b = [&](int s) { return smem_u32(bars + 2 * S + s); };
  auto empty_b = [&](int s) { return smem_u32(bars + 2 * S + 8 + s); };
  const ProjSplit ps = proj_split(p, blockIdx.x);
  const int nu = (int)(ps.u1 - ps.u0);
  const int pre = nu < SB ? nu : SB;
  prefetch_tensormap(&p.tm_w);
  prefetch_tensormap(&p.tm_x);
  // Fill phase-B stages from the top of the ring down: a stage only waits for the phase-A
  // stages it overlaps that were actually used (their last fill must have been consumed),
  // so CTAs with few attention tiles start on W_o while their attention is still running.
  int released = S;  // phase-A stages [released, S) are known free
  for (int jj = pre - 1; jj >= 0; --jj) {
    const int j = jj;
    const int lo_a = (j * kStageB) / kStageBytes;  // lowest phase-A stage this phase-B stage touches
    while (released > lo_a) {
      --released;
      if (released < it_a) {  // stage used in phase A: wait for the consumers of its last fill
        const int k = released + ((it_a - 1 - released) / S) * S;
        mbar_wait_bounded(empty_a(released), (k / S) & 1, p.err, kErrWaitEmpty, flags);
      }
    }
    const int unit = (int)ps.u0 + j, tile = unit / p.kb_per_tile, kb = unit - tile * p.kb_per_tile;
    const uint32_t dst = ring + j * kStageB;
    mbar_arrive_expect_tx(full_b(j), kProjWBytes + kXBytes);
    tma_load_2d(dst, &p.tm_w, full_b(j), tile * 128, kb * 64);
    tma_load_2d(dst + 8192, &p.tm_w, full_b(j), tile * 128 + 64, kb * 64);
  }
  grid_barrier_wait(p.grid_sync, (int)gridDim.x + p.sync_extra, p.err,
                    p.sync_limit_ns ? p.sync_limit_ns : kWaitLimitNs);
  fence_proxy_async_global();  // X was written by other CTAs' generic stores; TMA reads it
  for (int j = 0; j < pre; ++j) {
    const int unit = (int)ps.u0 + j, tile = unit / p.kb_per_tile, kb = unit - tile * p.kb_per_tile;
    tma_load_2d(ring + j * kStageB + kProjWBytes, &p.tm_x, full_b(j), kb * 64, 0);
  }
  for (int j = pre; j < nu; ++j) {
    const int s = j % SB;
    const uint32_t ph = (j / SB) & 1;
    mbar_wait_bounded(empty_b(s), ph ^ 1, p.err, kErrWaitEmpty, flags);
    const int unit = (int)ps.u0 + j, tile = unit / p.kb_per_tile, kb = unit - tile * p.kb_per_tile;
    const uint32_t dst = ring + s * kStageB;
    mbar_arrive_expect_tx(full_b(s), kProjWBytes + kXBytes);
    tma_load_2d(dst, &p.tm_w, full_b(s), tile * 128, kb * 64);
    tma_load_2d(dst + 8192, &p.tm_w, full_b(s), tile * 128 + 64, kb * 64);
    tma_load_2d(dst + kProjWBytes, &p.tm_x, full_b(s), kb * 64, 0);
  }
  for (int k = nu > SB ? nu - SB : 0; k < nu; ++k)  // no copies in flight at exit
    mbar_wait_bounded(full_b(k % SB), (k / SB) & 1, p.err, kErrWaitDrain, nullptr, kWaitLimitNs / 10);
}

// Phase-B MMA issuer (one thread): four tcgen05.mma per unit into the TMEM region of
// its column tile; each stage is released by tcgen05.commit, each region's
// accumulator is announced when the tile's last unit of this CTA is issued.
template <int NPAD, int S>
__device__ void fused_mma(const AttnParams& p, uint32_t ring, uint64_t* bars, uint32_t tmem, int* flags) {
  constexpr uint32_t kIdesc = umma_idesc_bf16(128, NPAD, /*A MN-major*/ true, /*B K-major*/ false);
  constexpr int SB = proj_stages(NPAD), kStageB = proj_stage_bytes(NPAD);
  auto full_b = [&](int s) { return smem_u32(bars + 2 * S + s); };
  auto empty_b = [&](int s) { return smem_u32(bars + 2 * S + 8 + s); };
  const ProjSplit ps = proj_split(p, blockIdx.x);
  const int nu = (int)(ps.u1 - ps.u0);
  const int tile0 = nu > 0 ? (int)(ps.u0 / p.kb_per_tile) : 0;
  for (int j = 0; j < nu; ++j) {
    const int s = j % SB;
    mbar_wait_bounded(full_b(s), (j / SB) & 1, p.err, kErrWaitFull, flags);
    tc_fence_after_sync();
    const int unit = (int)ps.u0 + j, tile = unit / p.kb_per_tile, kb = unit - tile * p.kb_per_tile;
    const int region = tile - tile0;
    const uint32_t a = ring + s * kStageB, bsm = a + kProjWBytes;
    const bool first = (j == 0) || (kb == 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t adesc = umma_smem_desc(a + kk * 16 * 128, 64 * 128, 1024);
      const uint64_t bdesc = umma_smem_desc(bsm + kk * 32, 16, 1024);
      umma_bf16(tmem + region * NPAD, adesc, bdesc, kIdesc, !(first && kk == 0));
    }
    umma_commit(empty_b(s));
    if (j == nu - 1 || kb == p.kb_per_tile - 1) umma_commit(smem_u32(bars + 2 * S + 16 + region));
  }
}

// CTA of phase B holding unit u.
__device__ __forceinline__ int proj_cta_of(long long u, int units, int PB) {
  return (int)(((u + 1) * (long long)PB - 1) / units);
}

// Phase-B epilogue (warps 0-3, TMEM lanes 0-127 = the tile's 128 columns): bf16 out
// when one CTA covered the whole column tile, else fp32 partials that the last
// CTA of the tile sums in a fixed order (atomic counter, no waiting).
template <int NPAD, int S>
__device__ void fused_epilogue(const AttnParams& p, uint64_t* bars, uint32_t tmem, int* flags, int warp, int lane,
                               int tid) {
  const ProjSplit ps = proj_split(p, blockIdx.x);
  if (ps.u1 <= ps.u0) return;
  const int kb = p.kb_per_tile;
  const int tile0 = (int)(ps.u0 / kb), tile1 = (int)((ps.u1 - 1) / kb);
  for (int tile = tile0; tile <= tile1; ++tile) {
    const int region = tile - tile0;
    mbar_wait_bounded(smem_u32(bars + 2 * S + 16 + region), 0, p.err, kErrWaitMma, flags);
    tc_fence_after_sync();
    float acc[NPAD];
#pragma unroll
    for (int c = 0; c < NPAD / 16; ++c) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(tmem + ((uint32_t)(warp * 32) << 16) + region * NPAD + c * 16, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[c * 16 + i] = __uint_as_float(r[i]);
    }
    const int m = warp * 32 + lane, n = tile * 128 + m;
    const bool n_ok = n < p.N;
    const int first = proj_cta_of((long long)tile * kb, p.units, ps.PB);
    const int last = proj_cta_of((long long)tile * kb + kb - 1, p.units, ps.PB);
    const int np = last - first + 1;
    if (np == 1) {
#pragma unroll
      for (int b = 0; b < NPAD; ++b)
        if (n_ok && b < p.B) p.y[(long long)b * p.y_sb + n] = __float2bfloat16_rn(acc[b]);
      continue;
    }
    const long long slot = (long long)blockIdx.x + tile;
    const bool part_ok = in_bounds((slot * p.B + p.B) * 128 <= p.proj_part_floats, p.err);
#pragma unroll
    for (int b = 0; b < NPAD; ++b)
      if (b < p.B && part_ok) p.proj_part[(slot * p.B + b) * 128 + m] = acc[b];
    named_bar_sync(2, 128);  // every epilogue thread's partial stores precede the release
    if (tid == 0)
      flags[2] = in_bounds(tile * p.kb_per_tile < p.units, p.err) &&
                 atomic_add_acq_rel_gpu(p.proj_counters + tile, 1) == np - 1;
    named_bar_sync(2, 128);
    if (flags[2]) {  // the last part of this column tile: sum all parts in order
      // batch rows in chunks of up to 32; per pass about 64 loads from clamped (always
      // valid) addresses are in flight, masked afterwards; parts are added in order
      constexpr int kChunk = NPAD < 32 ? NPAD : 32;
      constexpr int kParts = 64 / kChunk;
      for (int bc = 0; bc < p.B; bc += kChunk) {
        float sum[kChunk];
#pragma unroll
        for (int b = 0; b < kChunk; ++b) sum[b] = 0.f;
        for (int p0 = 0; p0 < np; p0 += kParts) {
          float v[kParts][kChunk];
#pragma unroll
          for (int u = 0; u < kParts; ++u) {
            int pc = min(p0 + u, np - 1);
            if (!in_bounds(((long long)first + pc + tile + 1) * p.B * 128 <= p.proj_part_floats, p.err)) pc = -first - tile;
#pragma unroll
            for (int b = 0; b < kChunk; ++b)
              v[u][b] = __ldcg(p.proj_part + (((long long)first + pc + tile) * p.B + min(bc + b, p.B - 1)) * 128 + m);
          }
#pragma unroll
          for (int u = 0; u < kParts; ++u)
#pragma unroll
            for (int b = 0; b < kChunk; ++b) sum[b] += (p0 + u < np) ? v[u][b] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < kChunk; ++b)
          if (n_ok && bc + b < p.B) p.y[(long long)(bc + b) * p.y_sb + n] = __float2bfloat16_rn(sum[b]);
      }
      if (tid == 0) p.proj_counters[tile] = 0;  // ready for the next call
    }
    named_bar_sync(2, 128);  // flags[2] is reused by the next tile
  }
}

// ---------------------------------------------------------------- paged cache
// Producer of the paged variant (one lane, like the contiguous producer). A tile of
// kT tokens is cut into boxes of min(block_size, kT) tokens (block sizes are powers of
// two), each read from its own block: box s of tile j of sequence b comes from block
// block_table[b][(j*kT + s*sub_tok) / block_size]. The block ids travel by TMA too: the 16 table entries
// from the tile's first one (rounded down to 16 bytes) are loaded kIdTiles tiles
// ahead into a shared-memory ring, each row completing on its own mbarrier, so no
// table read sits between a stage becoming free and its copies going out (the stream
// is bound by bytes in flight). Entries past a sequence's ceil(L / block_size) may be
// fetched but are never used; boxes that start at or past the sequence's length are
// not loaded (the consumers mask those tokens). A block id outside [0, num_blocks) is
// recorded in the error word and read past the pool's end, which TMA fills with zeros.
template <int S, int DIM>
__device__ __forceinline__ void paged_producer(const AttnParams& p, uint32_t ring, uint8_t* q_slots, size_t q_slot,
                                               uint64_t* bars, int* flags, const int* prefix, const int* lens,
                                               int* ids, long long start, long long end, const Cursor& c_start,
                                               int role) {
  // This lane shares its SM sub-partition with two busy consumer warps, so every
  // instruction per tile costs: block sizes are powers of two (shifts, no divisions),
  // and all but the copies is done before waiting for the stage.
  constexpr int kT = tile_tokens(DIM), kQRow = q_row_bytes(DIM);
  constexpr int kLogT = kT == 64 ? 6 : 5;
  static_assert((1 << kLogT) == kT, "tile tokens are a power of two");
  constexpr int PF = AttnSmem::kIdTiles, kRow = AttnSmem::kIdRow, kStride = AttnSmem::kIdStride;
  static_assert(kStride * 4 % 128 == 0, "ring rows must start 128-byte aligned");
  static_assert((PF & (PF - 1)) == 0, "ring rows are a power of two");
  constexpr int kMaxSub = kT / 8;  // boxes per tile at the smallest block size
  static_assert(kMaxSub + 3 <= kRow, "a tile's ids fit one row after rounding down to 16 bytes");
  if (start >= end) return;
  const int B = p.B, Hkv = p.Hkv, G = p.G;
  const int lbs = p.block_shift;
  const int lsub = lbs < kLogT ? lbs : kLogT;  // log2 of the tokens per box
  const int nsub = 1 << (kLogT - lsub);        // boxes per 64-dim column of a tile
  const uint32_t sub_bytes = (128u * (DIM / 64)) << lsub;  // one box row of K (or V)
  const unsigned nblk = (unsigned)p.num_blocks;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  auto id_bar = [&](int k) { return smem_u32(bars + 2 * S + k); };
  // flat table index of a tile's first entry
  auto entry = [&](const Cursor& a) { return (long long)a.b * p.bt_stride + ((a.j << kLogT) >> lbs); };
  auto fetch = [&](const Cursor& a, int slot) {
    in_bounds(entry(a) >= 0 && entry(a) < p.bt_entries, p.err);  // checked build: record only (TMA fills past the end)
    mbar_arrive_expect_tx(id_bar(slot), kRow * 4);
    tma_load_2d(smem_u32(ids + slot * kStride), &p.tm_table, id_bar(slot), (int)(entry(a) & ~3ll), 0);
  };
  prefetch_tensormap(&p.tm_k);
  prefetch_tensormap(&p.tm_v);
  prefetch_tensormap(&p.tm_table);
  const uint64_t kv_policy = l2_policy_evict_first();
  // Two producers (one per consumer group) share the work: this one issues the tiles whose
  // index in the range has parity `role`, i.e. the stages of group `role` and the block-id
  // ring rows of the same parity (S and PF are even), and walks the same cursor to skip the
  // others.
  static_assert(S % 2 == 0 && PF % 2 == 0, "stages and id rows split by parity");
  Cursor ca = c_start;  // the tile whose ids were fetched last
  for (int k = 0; k < PF && start + k < end; ++k) {
    if (k > 0) cursor_next(ca, prefix, B, Hkv);
    if ((k & 1) == role) fetch(ca, k);
  }
  Cursor c = c_start;
  long long seg0 = start;
  int it = 0;
  for (long long x = start; x < end; ++x, ++it) {
    if (x != start) {
      cursor_next(c, prefix, B, Hkv);
      if (c.j == 0) seg0 = x;
    }
    if ((it & 1) != role) {  // the other producer's tile: keep the id cursor in step
      if (x + PF < end) cursor_next(ca, prefix, B, Hkv);
      continue;
    }
    if (!in_bounds(c.b >= 0 && c.b < B && c.kvh >= 0 && c.kvh < Hkv, p.err)) c.b = c.kvh = 0;  // checked build
    const bool with_q = seg0 != start && x - seg0 < kGroups;  // (the range's first q: the consumers)
    const int stage = it % S;
    const int t0 = c.j << kLogT;
    // boxes holding tokens of the sequence (>= 1: t0 < L); the first row in the block:
    // with bs < kT every box starts a block (t0 % bs == 0), with bs >= kT the tile's one
    // box starts at t0 % bs
    const int n_load = min(nsub, (lens[c.b] - t0 + (1 << lsub) - 1) >> lsub);
    const int row = t0 & ((1 << lbs) - 1);
    const int slot = it & (PF - 1);
    mbar_wait_bounded(id_bar(slot), (it / PF) & 1, p.err, kErrWaitFull, flags);
    const int* idr = ids + slot * kStride + (int)(entry(c) & 3);
    int blk[kMaxSub];
#pragma unroll
    for (int s = 0; s < kMaxSub; ++s) blk[s] = idr[s];  // within the row; checked where used
    const uint32_t fb = full_bar(stage);
    const uint32_t kdst = ring + stage * kStageBytes;
    mbar_wait_bounded(empty_bar(stage), ((it / S) & 1) ^ 1, p.err, kErrWaitEmpty, flags);
    mbar_arrive_expect_tx(fb, 2 * n_load * sub_bytes + (with_q ? G * DIM * 2 : 0));
#pragma unroll
    for (int s = 0; s < kMaxSub; ++s) {
      if (s >= n_load) break;
      int bk = blk[s];
      if ((unsigned)bk >= nblk) {
        atomicOr(p.err, kErrBlockTable);
        bk = (int)nblk;
      }
      // one copy per tensor: box s = all D/64 dim boxes of its rows ([box][dim box][rows])
      const uint32_t off = (uint32_t)(s * 128 * (DIM / 64)) << lsub;
      tma_load_5d_hint(kdst + off, &p.tm_k, fb, 0, row, 0, c.kvh, bk, kv_policy);
      tma_load_5d_hint(kdst + kKTileBytes + off, &p.tm_v, fb, 0, row, 0, c.kvh, bk, kv_policy);
    }
    if (with_q) {
      const uint32_t qdst = smem_u32(q_slots + stage * q_slot);
      const __nv_bfloat16* qsrc = p.q + (long long)c.b * p.q_sb + (long long)(c.kvh * G) * p.q_sh;
      for (int h = 0; h < G; ++h) bulk_load(qdst + h * kQRow, qsrc + (long long)h * p.q_sh, DIM * 2, fb);
    }
    // ids of tile x + PF into the row this tile has just read. The row's reads have
    // completed: their values are operands of the copies issued above, which precede
    // this refill in program order. (A proxy fence here would also wait for the copies
    // in flight.)
    if (x + PF < end) {
      cursor_next(ca, prefix, B, Hkv);
      fetch(ca, slot);
    }
  }
  // do not leave with copies in flight (every id row fetched was waited for above)
  for (int k = it > S ? it - S : 0; k < it; ++k)
    if ((k & 1) == role) mbar_wait_bounded(full_bar(k % S), (k / S) & 1, p.err, kErrWaitDrain, nullptr, kWaitLimitNs / 10);
}

template <int NB, bool SCORES, int S, int NPAD, int DIM, bool PAGED = false, bool KV8 = false>
__global__ void __launch_bounds__(attn_threads(attn_producers(PAGED, NPAD > 0, SCORES)), 1)
    attn_decode_kernel(const __grid_constant__ AttnParams p) {
  constexpr int kProducers = attn_producers(PAGED, NPAD > 0, SCORES);
  constexpr int kThreads = attn_threads(kProducers);
  constexpr bool kFused = NPAD > 0;
  constexpr bool kWide = DIM == kHeadDimWide;
  static_assert(DIM == kHeadDim || (kWide && !kFused), "head dim 128, or 256 without the fused step");
  static_assert(!PAGED || (!kFused && !SCORES), "the paged variant computes attention only");
  static_assert(!KV8 || (DIM == kHeadDim && !kFused && !SCORES && !PAGED),
                "the fp8-cache variant: head dim 128, attention only, contiguous cache");
  // Stage: K tile then V tile, 32 KB (bf16: 64 tokens x 256 B each; fp8: 128 tokens x 128 B).
  constexpr int kSB = kStageBytes;
  constexpr int kKB = kSB / 2;
  // tokens per tile (fp8 cache: 128, so that a stage again holds 32 KB)
  constexpr int kT = KV8 ? kTileFp8 : tile_tokens(DIM);
  constexpr int kQRow = q_row_bytes(DIM);
  constexpr int kKs = DIM / 16;           // k-steps of QK^T
  constexpr int kTmemCols = NPAD <= 16 ? 32 : 2 * NPAD;  // two accumulator regions
  constexpr int HP = 8 * NB;  // heads per group, padded to the MMA width
  const int B = p.B, Hkv = p.Hkv, G = p.G, Lcap = p.Lcap;
  static_assert(S % kGroups == 0, "a stage must always be consumed by the same group");
  constexpr AttnSmem kFixed(NB, 0, S, DIM, kSB);  // offsets that do not depend on the batch size
  const AttnSmem lay(NB, B, S, DIM, kSB);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;

  uint8_t* q_slots = smem + kFixed.off_q();
  float* merge_o = reinterpret_cast<float*>(smem + kFixed.off_merge_o());    // [4][HP][kMergeRow]
  float* merge_ml = reinterpret_cast<float*>(smem + kFixed.off_merge_ml());  // [4][HP][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFixed.off_bars());
  int* flags = reinterpret_cast<int*>(smem + kFixed.off_flags());            // [0] abort, [1] last CTA
  int* prefix = reinterpret_cast<int*>(smem + lay.off_prefix());             // [B + 1]
  int* lens = reinterpret_cast<int*>(smem + lay.off_lens());                 // [B], clamped
  float* cpart_o = reinterpret_cast<float*>(smem + lay.off_cpart());         // [2][HP][DIM] (cluster mode)
  float* cpart_ml = cpart_o + 2 * HP * DIM;                                   // [2][HP][2]
  int* duty = reinterpret_cast<int*>(cpart_ml + 2 * HP * 2);  // [2][4] merges to share
  const uint32_t ring = smem_u32(smem);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  // Guards of the bounds-checked build (constant true otherwise): an index against the
  // extent of its buffer, a shared-memory range against this CTA's dynamic allocation.
  const uint32_t smem_lo = smem_u32(smem_raw);
  auto ok = [&](bool c) { return in_bounds(c, p.err); };
  auto sm_ok = [&](uint32_t addr, uint32_t bytes) { return smem_in_bounds(smem_lo, addr, bytes, p.err); };
  auto attn_ok = [&](int b, int h, int d) { return ok(b >= 0 && b < B && h >= 0 && h < Hkv * G && d >= 0 && d < DIM); };

  // L2 policy of the producers' K/V copies (read exactly once); no memory access, so it is
  // made before the wait below, off the path to the first copy
  const uint64_t kv_policy = l2_policy_evict_first();
  if (warp >= kGroups * kGroupWarps && lane == 0) {
    // The producers' tensor maps first: their fetch then overlaps the set-up below (the
    // sequence lengths' load) instead of delaying the first copy.
    prefetch_tensormap(&p.tm_k);
    if (!SCORES) prefetch_tensormap(&p.tm_v);
    if (PAGED) prefetch_tensormap(&p.tm_table);
    if (kFused) {
      prefetch_tensormap(&p.tm_w);
      prefetch_tensormap(&p.tm_x);
    }
    // The lengths are not known before the wait below, but when every sequence is full (the
    // cache's capacity) this CTA's first tiles are those of the split of B * Hkv full
    // sequences: pull the first ring's worth into L2 now (and the first q), so that the first
    // copies come from L2.
    // (An L2 prefetch only warms the cache, which stays coherent with whatever the previous
    // kernel writes; a wrong guess costs two tiles of bandwidth.)
    if constexpr (!PAGED && !kFused) {
      const int role = warp - kGroups * kGroupWarps;
      const long long nt = (p.Lcap + kT - 1) / kT, per_b = (long long)p.Hkv * nt, Tg = (long long)p.B * per_b;
      int workers = min((int)gridDim.x, p.attn_workers);
      if (p.cluster > 1) workers = min(workers, p.B * p.Hkv * p.cluster);
      const long long Pg = min((long long)workers, Tg);
      const long long x0 = Pg > 0 ? (long long)blockIdx.x * Tg / Pg : 0;
      const long long x1 = Pg > 0 ? ((long long)blockIdx.x + 1) * Tg / Pg : 0;
      for (long long x = x0 + role; Pg > 0 && blockIdx.x < Pg && x < x1 && x < x0 + S; x += kProducers) {
        const int b = (int)(x / per_b), r = (int)(x - (long long)b * per_b), kvh = r / (int)nt, j = r - kvh * (int)nt;
        tma_prefetch_5d(&p.tm_k, 0, j * kT, 0, kvh, b);
        if (!SCORES) tma_prefetch_5d(&p.tm_v, 0, j * kT, 0, kvh, b);
        if (x == x0)  // and the q rows of that sequence, which the consumers read first
          bulk_prefetch_l2(p.q + (long long)b * p.q_sb + (long long)(kvh * p.G) * p.q_sh,
                           (uint32_t)((((long long)(p.G - 1) * p.q_sh + DIM) * 2 + 15) & ~15ll), l2_policy_evict_last());
      }
    }
  }
  if (tid == 32) {  // (the set-up warp's first lane: it copies the first tiles, below)
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kGroupWarps);
    }
    if (PAGED) {  // rows of the block-id ring
      for (int s = 0; s < AttnSmem::kIdTiles; ++s) mbar_init(smem_u32(bars + 2 * S + s), 1);
    }
    if (kFused) {
      for (int s = 0; s < 8; ++s) {
        mbar_init(smem_u32(bars + 2 * S + s), 1);      // phase-B full: the producer's expect-tx
        mbar_init(smem_u32(bars + 2 * S + 8 + s), 1);  // phase-B empty: one tcgen05.commit
      }
      mbar_init(smem_u32(bars + 2 * S + 16), 1);  // accumulator of the first column tile
      mbar_init(smem_u32(bars + 2 * S + 17), 1);  // ... and of the second
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    if (p.cluster > 1) {  // (the region exists in cluster launches only)
      duty[2] = 0;  // no sequence of this CTA merges on chip (yet)
      duty[6] = 0;
    }
    fence_barrier_init();
  }
  if (kFused && warp == 0) {  // TMEM for the projection accumulators (one CTA per SM)
    tmem_alloc(smem_u32(flags + 3), kTmemCols);
    tmem_relinquish();
  }
  // Padded head rows of the q slots stay zero for the whole kernel.
  for (int i = tid; i < (int)(S * kFixed.q_slot() / 16); i += kThreads)
    reinterpret_cast<uint4*>(q_slots)[i] = make_uint4(0, 0, 0, 0);
  // Launched with programmatic dependent launch, this grid may start while the previous
  // kernel in the stream drains; nothing above touched global memory, and nothing below
  // does before the previous kernel has completed and its writes are visible.
  pdl_wait_primary();
  if (warp == 1) {  // clamped lengths, and tiles per batch row scanned into prefix
    int carry = 0, v0 = 0;
    bool unequal = false;  // do the rows differ in tile count?
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int v = 0;
      if (b < B) {
        const int L = clamp_len(__ldg(p.seq_lens + b), Lcap);
        lens[b] = L;
        v = ((L + kT - 1) / kT) * Hkv;
      }
      if (base == 0) v0 = __shfl_sync(0xffffffffu, v, 0);
      unequal |= __any_sync(0xffffffffu, b < B && v != v0);
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
      }
      if (b < B) prefix[b + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) prefix[0] = 0;
    // This CTA's range [start, end) of the T tiles and the cursor at its first tile, for every
    // warp after the barrier. Worker c of P takes [c T / P, (c + 1) T / P), computed as
    // c (T / P) + c (T % P) / P in 32-bit arithmetic (T < 2^31, c <= P <= 512), each division
    // by P a multiply and a shift from the host when P is the worker count it expected.
    __syncwarp();  // prefix[] and lens[] complete
    const int T = carry;
    // Cluster mode with unequal lengths: the cluster CTAs work as the flat grid does
    const bool chip = p.cluster > 1 && !unequal;
    int workers = min((int)gridDim.x, p.attn_workers);
    if (chip) workers = min(workers, B * Hkv * p.cluster);
    const int P = T > 0 ? min(workers, T) : 1;
    const int cta = blockIdx.x;
    int start = 0, end = 0;
    if (T > 0 && cta < P) {
      if (P == T) {  // one tile each
        start = cta;
        end = cta + 1;
      } else {
        unsigned tq, tr, f0, f1;
        if (P == (chip ? p.split_div[1] : p.split_div[0])) {
          const unsigned long long m = chip ? p.split_mul[1] : p.split_mul[0];
          const int sh = chip ? p.split_shift[1] : p.split_shift[0];
          tq = div_mul((unsigned)T, m, sh);
          tr = (unsigned)T - tq * (unsigned)P;
          f0 = div_mul((unsigned)cta * tr, m, sh);
          f1 = div_mul((unsigned)(cta + 1) * tr, m, sh);
        } else {
          tq = (unsigned)T / (unsigned)P;
          tr = (unsigned)T % (unsigned)P;
          f0 = (unsigned)cta * tr / (unsigned)P;
          f1 = (unsigned)(cta + 1) * tr / (unsigned)P;
        }
        start = (int)((unsigned)cta * tq + f0);
        end = (int)((unsigned)(cta + 1) * tq + f1);
      }
    }
    // The cursor at `start`: the last batch row whose first tile is at or before it (prefix
    // is non-decreasing: count the rows at or before it, 32 at a time), then the KV head and
    // the tile within the row's share.
    int cb = 0, ckvh = 0, cj = 0, cnt = 1;
    if (start < end) {
      int rows = 0;
      for (int base = 0; base < B; base += 32) {
        const unsigned at = __ballot_sync(0xffffffffu, base + lane < B && prefix[base + lane] <= start);
        rows += __popc(at);
        if (at != 0xffffffffu) break;
      }
      cb = rows - 1;  // >= 0: prefix[0] = 0
      cnt = (lens[cb] + kT - 1) / kT;
      const int r = start - prefix[cb];
      ckvh = div_small(r, cnt);
      cj = r - ckvh * cnt;
    }
    // The first tile of each consumer group (lane g: group g's, stage g), copied now so that
    // they are in flight while the other warps pass the set-up barrier; the second only if
    // it lies in the same sequence (it then needs no q: the consumers read the range's first
    // q themselves). The barriers are fresh, initialised by lane 0 of this warp.
    if (!PAGED && lane < kGroups && lane < early_tiles(start, end, cj, cnt)) {
      Cursor ce = {cb, ckvh, cj, cnt};
      if (lane == 1) cursor_next(ce, prefix, B, Hkv);
      const uint32_t fb = full_bar(lane), dst = ring + lane * kSB;
      if (!(sm_ok(dst, kSB) && ok(ce.b >= 0 && ce.b < B && ce.kvh >= 0 && ce.kvh < Hkv && ce.j * kT < Lcap)))
        ce.b = ce.kvh = ce.j = 0;  // checked build: record, clamp
      mbar_arrive_expect_tx(fb, SCORES ? kKB : kSB);
      tma_load_5d_hint(dst, &p.tm_k, fb, 0, ce.j * kT, 0, ce.kvh, ce.b, kv_policy);
      if (!SCORES) tma_load_5d_hint(dst + kKB, &p.tm_v, fb, 0, ce.j * kT, 0, ce.kvh, ce.b, kv_policy);
    }
    if (lane == 0) {
      int* rng = flags + 8;
      rng[0] = start;
      rng[1] = end;
      rng[2] = P;
      rng[3] = cb;
      rng[4] = ckvh;
      rng[5] = cj;
      rng[6] = cnt;
      rng[7] = chip ? 1 : 0;
    }
  }
  if (kFused) tc_fence_before_sync();
  __syncthreads();
  if (kFused) tc_fence_after_sync();
  const uint32_t tmem = kFused ? (uint32_t)flags[3] : 0u;
  // The next kernel in the stream (launched with programmatic dependent launch) may now
  // be scheduled; it waits for this grid's completion before it reads our output. When
  // the projection follows, the trigger comes near the end of the CTA's tiles instead
  // (below), so that its W_o loads do not queue in front of this grid's K/V stream.
  if (p.trigger_at <= 0) pdl_launch_dependents();

  const long long T = prefix[B];
  const int cta = blockIdx.x;
  const int* rng = flags + 8;  // range and first cursor (set-up warp)
  // > 1: cluster mode: the grid comes in clusters of `cs` consecutive CTAs. With equal
  // lengths the tiles go to B * Hkv * cs workers, cs per sequence, so that the parts of
  // every sequence lie in one cluster and merge on chip (the grid's other CTAs leave at
  // once); otherwise to every CTA of the grid.
  const int cs = p.cluster;
  // With unequal lengths the cluster CTAs work as the flat grid does, without on-chip
  // merges and without the cluster barriers at the end, which would hold every CTA of a
  // cluster until its slowest one is done (the same flag in every CTA).
  const bool chip = rng[7] != 0;
  // P workers share the T tiles; with P <= T every range is non-empty, so the CTAs
  // cta_of(first tile) .. cta_of(last tile) of a sequence all hold a part of it.
  const int P = rng[2];
  // first tile of worker c, floor(c * T / P) (off the path to the first copy)
  auto split = [&](int c) {
    return (long long)c * ((unsigned)T / (unsigned)P) + (long long)(((unsigned)c * ((unsigned)T % (unsigned)P)) / (unsigned)P);
  };
  const long long start = rng[0], end = rng[1];
  const Cursor c_start = {rng[3], rng[4], rng[5], rng[6]};

  if (warp >= kGroups * kGroupWarps) {
    // ------------------------------------------------------------ producer(s)
    if constexpr (PAGED) {
      if (lane == 0)
        paged_producer<S, DIM>(p, ring, q_slots, kFixed.q_slot(), bars, flags, prefix, lens,
                               reinterpret_cast<int*>(smem + lay.off_ids()), start, end, c_start,
                               warp - kGroups * kGroupWarps);
    } else if (lane == 0) {
     const int role = warp - kGroups * kGroupWarps;  // with two producers: tiles of parity `role`
     int it = 0;
     if (start < end) {
      // This CTA's share of the prefetch region, in 4 KB-aligned pieces, one per tile.
      const uint64_t pf_policy = l2_policy_evict_last();
      long long pf_next = 0, pf_end = 0, pf_piece = 0;
      if (p.prefetch_bytes > 0) {
        const long long pf_per_cta = ((p.prefetch_bytes + P - 1) / P + 4095) & ~4095ll;
        pf_next = min((long long)cta * pf_per_cta, p.prefetch_bytes);
        pf_end = min(pf_next + pf_per_cta, p.prefetch_bytes);
        pf_piece = ((pf_end - pf_next + (end - start) - 1) / (end - start) + 4095) & ~4095ll;
        if (kProducers == 2) {  // the first producer alone pulls the region, per pair of tiles
          if (role) pf_end = pf_next;
          else pf_piece *= 2;
        }
      }
      const int n_early = early_tiles(start, end, c_start.j, c_start.nt);
      Cursor c = c_start;
      long long seg0 = start;
      for (long long x = start; x < end; ++x, ++it) {
        if (x != start) {
          cursor_next(c, prefix, B, Hkv);
          if (c.j == 0) seg0 = x;
        }
        if (kProducers == 2 && (it & 1) != role) continue;  // the other producer's tile
        // each group's first tile of a segment that starts inside the range (the consumers
        // read the range's first q themselves)
        const bool with_q = seg0 != start && x - seg0 < kGroups;
        const int stage = it % S;
        const uint32_t ph = (it / S) & 1;
        const uint32_t fb = full_bar(stage);
        if (it >= n_early) {  // (the first ones: copied by the set-up warp)
          if (it >= S) mbar_wait_bounded(empty_bar(stage), ph ^ 1, p.err, kErrWaitEmpty, flags);  // (fresh before)
          uint32_t bytes = SCORES ? kKB : kSB;
          if (with_q) bytes += G * DIM * 2;
          const uint32_t kdst = ring + stage * kSB;
          const int t0 = c.j * kT;
          // bounds-checked build: a cursor outside the batch is recorded and clamped, so that
          // every copy stays inside the tensors and every wait of the kernel still ends
          if (!(sm_ok(kdst, kSB) && sm_ok(smem_u32(q_slots + stage * kFixed.q_slot()), G * kQRow) &&
                ok(c.b >= 0 && c.b < B && c.kvh >= 0 && c.kvh < Hkv && t0 >= 0 && t0 < Lcap)))
            c.b = c.kvh = 0;
          mbar_arrive_expect_tx(fb, bytes);
          tma_load_5d_hint(kdst, &p.tm_k, fb, 0, t0, 0, c.kvh, c.b, kv_policy);  // all D/64 boxes at once
          if (!SCORES) tma_load_5d_hint(kdst + kKB, &p.tm_v, fb, 0, t0, 0, c.kvh, c.b, kv_policy);
        }
        for (long long todo = min(pf_piece, pf_end - pf_next); todo > 0;) {
          const long long n = min(todo, 32768ll);
          bulk_prefetch_l2(p.prefetch + pf_next, (uint32_t)n, pf_policy);
          pf_next += n;
          todo -= n;
        }
        if (with_q) {
          const uint32_t qdst = smem_u32(q_slots + stage * kFixed.q_slot());
          const __nv_bfloat16* qsrc = p.q + (long long)c.b * p.q_sb + (long long)(c.kvh * G) * p.q_sh;
          for (int h = 0; h < G; ++h) bulk_load(qdst + h * kQRow, qsrc + (long long)h * p.q_sh, DIM * 2, fb);
        }
      }
      // Do not leave with copies in flight (only matters if the consumers gave up; the fused
      // step's consumers wait for these copies before the CTA can end, so it skips this).
      if (!kFused)
      for (int k = it > S ? it - S : 0; k < it; ++k)
        if (kProducers == 1 || (k & 1) == role)
          mbar_wait_bounded(full_bar(k % S), (k / S) & 1, p.err, kErrWaitDrain, nullptr,
                            kWaitLimitNs / 10);
     }
     if constexpr (kFused) fused_producer<NPAD, S>(p, ring, bars, it, flags);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int grp = warp / kGroupWarps;  // consumer group: takes iterations it % kGroups == grp
    const int wg = warp % kGroupWarps;   // warp in group
    // merge/output mapping: thread -> (first head tid / DIM, dim tid % DIM), heads step kHStep
    constexpr int kHStep = kConsumerThreads / DIM;
    if (!SCORES) {  // empty sequences produce zero rows
      for (int s = cta; s < B * Hkv; s += gridDim.x) {
        const int b = s / Hkv;
        if (lens[b] != 0) continue;
        const int kvh = s - b * Hkv;
        for (int h = tid / DIM; h < G; h += kHStep)
          if (attn_ok(b, kvh * G + h, tid % DIM))
            p.attn[(long long)b * p.a_sb + (long long)(kvh * G + h) * p.a_sh + (tid % DIM)] = __float2bfloat16_rn(0.f);
      }
    }
    uint32_t qf[NB][kKs][2];
    float o[8][NB][4];
    float m_run[NB][2], l_run[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      m_run[nb][0] = m_run[nb][1] = kNegInf;
      l_run[nb][0] = l_run[nb][1] = 0.f;
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) o[mb][nb][0] = o[mb][nb][1] = o[mb][nb][2] = o[mb][nb][3] = 0.f;
    }
    // this warp's first token inside a stage, and (D = 256) its 128-dim half of O
    const int tb = KV8 ? wg * 32 : (kWide ? (wg >> 1) * 16 : wg * 16);
    const int dh = kWide ? (wg & 1) : 0;
    // dims (within an m-tile of 16) of this lane's accumulator rows g and g+8
    const int d_lo = KV8 ? 2 * g : g, d_hi = KV8 ? 2 * g + 1 : g + 8;
    // Tile layout in shared memory: [box][dim box][box rows][128 B], one box = the rows
    // one copy brings (the whole tile, or a paged block smaller than a tile). Byte offset
    // of a row inside its dim box, and the distance between dim boxes:
    constexpr int kLogT = kT == 128 ? 7 : (kT == 64 ? 6 : 5);
    const int lbox = PAGED ? min(p.block_shift, kLogT) : kLogT;  // log2 rows per box
    const uint32_t dbox = 128u << lbox;
    auto row_off = [&](int r) {
      return ((uint32_t)((r >> lbox) * (DIM / 64)) << (lbox + 7)) + ((uint32_t)(r & ((1 << lbox) - 1)) << 7);
    };
    const uint32_t qk_row = row_off(tb + (lane & 7) + ((lane >> 3) & 1) * 8);  // ldmatrix rows of S^T
    const uint32_t pv_row = row_off(tb + (lane & 7) + ((lane >> 4) & 1) * 8);  // ldmatrix.trans rows of V
    const float sl2 = p.scale_log2;
    // q fragments of a segment's (batch row, KV head): head h's row at rows + h * stride bytes
    // (in shared memory for the segments that start inside the range, whose first tiles carry
    // q; from global memory for the range's first segment, loaded while its first stages are
    // in flight). Head rows at or past `heads` read as zero.
    auto load_q = [&](const uint8_t* rows, long long stride, int heads, bool global) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int h = nb * 8 + g;
#pragma unroll
        for (int ks = 0; ks < kKs; ++ks) {
          uint32_t w0 = 0, w1 = 0;
          if constexpr (KV8) {
            // k-slots 2t, 2t+1, 2t+8, 2t+9 of step ks hold dims 16ks + 4t .. 4t+3 (the
            // order in which an fp8 K row reaches this lane); q in f16, same order
            const uint8_t* row = rows + h * stride + (ks * 16 + 4 * t) * 2;
            if (h < heads) {
              const uint2 w = global ? __ldg(reinterpret_cast<const uint2*>(row)) : *reinterpret_cast<const uint2*>(row);
              w0 = bf16x2_to_f16x2_clamped(w.x);
              w1 = bf16x2_to_f16x2_clamped(w.y);
            }
          } else {
            const uint8_t* row = rows + h * stride + (ks * 16 + 2 * t) * 2;
            if (h < heads) {
              w0 = global ? __ldg(reinterpret_cast<const uint32_t*>(row)) : *reinterpret_cast<const uint32_t*>(row);
              w1 = global ? __ldg(reinterpret_cast<const uint32_t*>(row + 16)) : *reinterpret_cast<const uint32_t*>(row + 16);
            }
          }
          qf[nb][ks][0] = w0;
          qf[nb][ks][1] = w1;
        }
      }
    };
    Cursor c;
    if (start < end) {
      c = c_start;
      if (ok(c.b >= 0 && c.b < B && c.kvh >= 0 && c.kvh < Hkv))
        load_q(reinterpret_cast<const uint8_t*>(p.q + (long long)c.b * p.q_sb + (long long)(c.kvh * G) * p.q_sh),
               p.q_sh * 2, G, true);
    }
    long long seg0 = start;
    int it = 0;
    for (long long x = start; x < end; ++x, ++it) {
      if (x != start) {
        cursor_next(c, prefix, B, Hkv);
        if (c.j == 0) seg0 = x;
      }
      if (!ok(c.b >= 0 && c.b < B && c.kvh >= 0 && c.kvh < Hkv)) c.b = c.kvh = 0;  // checked build: record, clamp
      const bool last = (x == end - 1) || (c.j == c.nt - 1);
      if (it % kGroups == grp) {
        const int t0 = c.j * kT;
        const int vw = min(kT, lens[c.b] - t0) - tb;  // valid tokens of this warp's 16 (fp8: 32)
        const int stage = it % S;
        const uint32_t ph = (it / S) & 1;
        mbar_wait_bounded(full_bar(stage), ph, p.err, kErrWaitFull, flags);
        if (seg0 != start && x - seg0 < kGroups)  // this group's first tile of the segment carries q
          load_q(q_slots + stage * kFixed.q_slot(), kQRow, HP, false);
        if constexpr (KV8) {
          // fp8 cache: this warp owns 32 tokens (rows tb .. tb+31 of a 128-token tile), two
          // 16-row halves that share one softmax update. K and V rows are 128 bytes.
          if (vw > 0) {
            const uint32_t kbase = ring + stage * kSB;
            // ---- S^T = K . Q^T per half. One ldmatrix.x4 brings two k-steps (rows +0..7 and
            // +8..15 of 16-byte chunks 2kk and 2kk+1); a lane holds 4 dims of a row per matrix,
            // widened to f16 exactly, which is the k-slot order of the q fragments.
            float sa[2][NB][4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float se[NB][4], so[NB][4];
#pragma unroll
              for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int i = 0; i < 4; ++i) se[nb][i] = so[nb][i] = 0.f;
              const int row = tb + 16 * hh + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
              for (int kk = 0; kk < kKs / 2; ++kk) {
                const int chunk = 2 * kk + (lane >> 4);
                uint32_t m[4];
                ldsm_x4(kbase + row * 128 + ((chunk ^ (lane & 7)) << 4), m[0], m[1], m[2], m[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint32_t a[4] = {e4m3x2_to_f16x2(m[2 * h]), e4m3x2_to_f16x2(m[2 * h + 1]),
                                         e4m3x2_to_f16x2(m[2 * h] >> 16), e4m3x2_to_f16x2(m[2 * h + 1] >> 16)};
#pragma unroll
                  for (int nb = 0; nb < NB; ++nb) {
                    if (h) mma_f16_16816(so[nb], a, qf[nb][2 * kk + h][0], qf[nb][2 * kk + h][1]);
                    else mma_f16_16816(se[nb], a, qf[nb][2 * kk + h][0], qf[nb][2 * kk + h][1]);
                  }
                }
              }
#pragma unroll
              for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int i = 0; i < 4; ++i) sa[hh][nb][i] = se[nb][i] + so[nb][i];
            }
            // ---- online softmax over the 32 tokens (element i of half hh: token
            // 16hh + g + 8(i>>1), head 8nb + 2t + (i&1)); P rounded to f16 for P.V
            float xv[NB][2][4];
            bool grow = false;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const bool v0 = 16 * hh + g < vw, v1 = 16 * hh + g + 8 < vw;
                xv[nb][hh][0] = v0 ? sa[hh][nb][0] * sl2 : kNegInf;
                xv[nb][hh][1] = v0 ? sa[hh][nb][1] * sl2 : kNegInf;
                xv[nb][hh][2] = v1 ? sa[hh][nb][2] * sl2 : kNegInf;
                xv[nb][hh][3] = v1 ? sa[hh][nb][3] * sl2 : kNegInf;
                grow |= fmaxf(xv[nb][hh][0], xv[nb][hh][2]) > m_run[nb][0] + kSlack;
                grow |= fmaxf(xv[nb][hh][1], xv[nb][hh][3]) > m_run[nb][1] + kSlack;
              }
            if (__any_sync(0xffffffffu, grow)) {  // the reference moves to the running maximum
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                float mx0 = fmaxf(fmaxf(xv[nb][0][0], xv[nb][0][2]), fmaxf(xv[nb][1][0], xv[nb][1][2]));
                float mx1 = fmaxf(fmaxf(xv[nb][0][1], xv[nb][0][3]), fmaxf(xv[nb][1][1], xv[nb][1][3]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[nb][0], mx0), mn1 = fmaxf(m_run[nb][1], mx1);
                const float al0 = fast_exp2(m_run[nb][0] - mn0), al1 = fast_exp2(m_run[nb][1] - mn1);
                m_run[nb][0] = mn0;
                m_run[nb][1] = mn1;
                l_run[nb][0] *= al0;
                l_run[nb][1] *= al1;
#pragma unroll
                for (int mb = 0; mb < 8; ++mb) {
                  o[mb][nb][0] *= al0;
                  o[mb][nb][1] *= al1;
                  o[mb][nb][2] *= al0;
                  o[mb][nb][3] *= al1;
                }
              }
            }
            uint32_t pb[2][NB][2];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const float m0 = m_run[nb][0], m1 = m_run[nb][1];
              float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const uint32_t r0 = pack_f16x2(fast_exp2(xv[nb][hh][0] - m0), fast_exp2(xv[nb][hh][1] - m1));
                const uint32_t r1 = pack_f16x2(fast_exp2(xv[nb][hh][2] - m0), fast_exp2(xv[nb][hh][3] - m1));
                ls0 += f16lo_to_f32(r0) + f16lo_to_f32(r1);  // the weights that enter P.V
                ls1 += f16hi_to_f32(r0) + f16hi_to_f32(r1);
                pb[hh][nb][0] = movmatrix_trans(r0);  // P[head g][tokens 16hh + 2t, +1]
                pb[hh][nb][1] = movmatrix_trans(r1);  // P[head g][tokens 16hh + 2t + 8, +9]
              }
              l_run[nb][0] += ls0;
              l_run[nb][1] += ls1;
            }
            // ---- O^T += V^T . P^T, one k-step per half. ldmatrix.trans of 16-bit pairs hands
            // a lane tokens 2t, 2t+1 of dims 2g, 2g+1 (a byte each); a byte permute makes
            // (dim 2g: two tokens) and (dim 2g+1: two tokens), widened to f16 exactly, so the
            // MMA's rows g and g+8 of m-tile mb are dims 16mb + 2g and 16mb + 2g + 1.
            const uint32_t vbase = kbase + kKB;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // valid tokens of this half: a half past the length is masked whole (its weights
              // are 0 too), with no branch on the count in the hot loop (measured 28.1 -> 27.5 us
              // for the batch-8 fp8 attention)
              const int vwh = vw - 16 * hh;
              const int row = tb + 16 * hh + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
              for (int mp = 0; mp < 4; ++mp) {
                const int chunk = 2 * mp + (lane >> 4);
                uint32_t m[4];
                ldsm_x4_trans(vbase + row * 128 + ((chunk ^ (lane & 7)) << 4), m[0], m[1], m[2], m[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  uint32_t lo = m[2 * h], hi = m[2 * h + 1];  // tokens 2t, 2t+1 and 2t+8, 2t+9
                  lo = mask_tokens(lo, 2 * t, vwh);  // rows past the sequence may hold anything;
                  hi = mask_tokens(hi, 2 * t + 8, vwh);  // P is 0 there
                  const uint32_t pl = __byte_perm(lo, 0, 0x3120), ph = __byte_perm(hi, 0, 0x3120);
                  const uint32_t a[4] = {e4m3x2_to_f16x2(pl), e4m3x2_to_f16x2(pl >> 16), e4m3x2_to_f16x2(ph),
                                         e4m3x2_to_f16x2(ph >> 16)};
#pragma unroll
                  for (int nb = 0; nb < NB; ++nb) mma_f16_16816(o[2 * mp + h][nb], a, pb[hh][nb][0], pb[hh][nb][1]);
                }
              }
            }
          }
        } else if (vw > 0) {
          const uint32_t kbase = ring + stage * kSB;
          // ---- S^T[16 tokens][8*NB heads] = K_tile . Q^T  (fp32, unscaled)
          float se[NB][4], so[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) se[nb][i] = so[nb][i] = 0.f;
          {
#pragma unroll
            for (int ks = 0; ks < kKs; ++ks) {
              const int chunk = 2 * (ks & 3) + (lane >> 4);
              const uint32_t addr = kbase + (ks >> 2) * dbox + qk_row + ((chunk ^ (lane & 7)) << 4);
              uint32_t a[4];
              ldsm_x4(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                if (ks & 1) mma_bf16_16816(so[nb], a, qf[nb][ks][0], qf[nb][ks][1]);
                else mma_bf16_16816(se[nb], a, qf[nb][ks][0], qf[nb][ks][1]);
              }
            }
          }
          float s[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[nb][i] = se[nb][i] + so[nb][i];
          // fragment element i: token g + 8*(i>>1), head 8*nb + 2t + (i&1)
          if (SCORES) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int head = nb * 8 + 2 * t + (i & 1);
                const int tok = g + 8 * (i >> 1);
                if (head < G && tok < vw && dh == 0 &&  // at D = 256 both warps of a pair hold S
                    ok(t0 + tb + tok >= 0 && t0 + tb + tok < Lcap))
                  p.scores[(long long)c.b * p.s_sb + (long long)(c.kvh * G + head) * p.s_sh + t0 + tb + tok] =
                      s[nb][i];
              }
          } else {
            const bool v0 = g < vw, v1 = g + 8 < vw;
            float xs[NB][4];
            bool grow = false;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              xs[nb][0] = v0 ? s[nb][0] * sl2 : kNegInf;
              xs[nb][1] = v0 ? s[nb][1] * sl2 : kNegInf;
              xs[nb][2] = v1 ? s[nb][2] * sl2 : kNegInf;
              xs[nb][3] = v1 ? s[nb][3] * sl2 : kNegInf;
              grow |= fmaxf(xs[nb][0], xs[nb][2]) > m_run[nb][0] + kSlack;
              grow |= fmaxf(xs[nb][1], xs[nb][3]) > m_run[nb][1] + kSlack;
            }
            if (__any_sync(0xffffffffu, grow)) {  // the reference moves to the running maximum
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                float mx0 = fmaxf(xs[nb][0], xs[nb][2]), mx1 = fmaxf(xs[nb][1], xs[nb][3]);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                }
                const float mn0 = fmaxf(m_run[nb][0], mx0), mn1 = fmaxf(m_run[nb][1], mx1);
                const float al0 = fast_exp2(m_run[nb][0] - mn0), al1 = fast_exp2(m_run[nb][1] - mn1);
                m_run[nb][0] = mn0;
                m_run[nb][1] = mn1;
                l_run[nb][0] *= al0;
                l_run[nb][1] *= al1;
#pragma unroll
                for (int mb = 0; mb < 8; ++mb) {
                  o[mb][nb][0] *= al0;
                  o[mb][nb][1] *= al1;
                  o[mb][nb][2] *= al0;
                  o[mb][nb][3] *= al1;
                }
              }
            }
            uint32_t pb[NB][2];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const float m0 = m_run[nb][0], m1 = m_run[nb][1];
              // the sum uses the bf16-rounded weights that enter P.V
              const uint32_t r0 = pack_bf16x2(fast_exp2(xs[nb][0] - m0), fast_exp2(xs[nb][1] - m1));  // token g
              const uint32_t r1 = pack_bf16x2(fast_exp2(xs[nb][2] - m0), fast_exp2(xs[nb][3] - m1));  // token g+8
              l_run[nb][0] += bf16lo_to_f32(r0) + bf16lo_to_f32(r1);
              l_run[nb][1] += bf16hi_to_f32(r0) + bf16hi_to_f32(r1);
              pb[nb][0] = movmatrix_trans(r0);  // P[head g][tokens 2t, 2t+1]
              pb[nb][1] = movmatrix_trans(r1);  // P[head g][tokens 2t+8, 2t+9]
            }
            // ---- O^T[128 dims (of half dh)][8*NB heads] += V_tile^T . P^T
            const uint32_t vbase = kbase + kKB;
            const int jm = lane >> 3;
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
              const int chunk = 2 * (mb & 3) + (jm & 1);
              const uint32_t addr = vbase + (dh * 2 + (mb >> 2)) * dbox + pv_row + ((chunk ^ (lane & 7)) << 4);
              uint32_t a[4];
              ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
              if (vw < 16) {  // rows past the sequence may hold anything; P is 0 there
                a[0] = mask_tokens(a[0], 2 * t, vw);
                a[1] = mask_tokens(a[1], 2 * t, vw);
                a[2] = mask_tokens(a[2], 2 * t + 8, vw);
                a[3] = mask_tokens(a[3], 2 * t + 8, vw);
              }
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(o[mb][nb], a, pb[nb][0], pb[nb][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
      }

      if (p.trigger_at > 0 && tid == 0 && x == (end - p.trigger_at > start ? end - p.trigger_at : start))
        pdl_launch_dependents();
      if (!SCORES && last) {
        // ---------------------------------------- finish this sequence segment
        const int b = c.b, kvh = c.kvh, seq = b * Hkv + kvh;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) l_run[nb][cc] += __shfl_xor_sync(0xffffffffu, l_run[nb][cc], off);
        float* mo = merge_o + wg * HP * kMergeRow;
        float* ml = merge_ml + wg * HP * 2;
        if (!(sm_ok(smem_u32(mo), HP * kMergeRow * 4) && sm_ok(smem_u32(ml), HP * 2 * 4))) mo = ml = merge_ml;
        // (1) group 1 hands its state to the partner warp of group 0
        if (grp == 1) {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int h0 = nb * 8 + 2 * t;
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
              mo[h0 * kMergeRow + mb * 16 + d_lo] = o[mb][nb][0];
              mo[(h0 + 1) * kMergeRow + mb * 16 + d_lo] = o[mb][nb][1];
              mo[h0 * kMergeRow + mb * 16 + d_hi] = o[mb][nb][2];
              mo[(h0 + 1) * kMergeRow + mb * 16 + d_hi] = o[mb][nb][3];
            }
            if (g == 0) {
              ml[h0 * 2] = m_run[nb][0];
              ml[h0 * 2 + 1] = l_run[nb][0];
              ml[h0 * 2 + 2] = m_run[nb][1];
              ml[h0 * 2 + 3] = l_run[nb][1];
            }
          }
        }
        named_bar_sync(1, kConsumerThreads);
        // (2) group 0 merges it into registers and publishes the pair's state
        if (grp == 0) {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int h = nb * 8 + 2 * t + cc;
              const float mp = ml[h * 2], lp = ml[h * 2 + 1];
              const float mn = fmaxf(m_run[nb][cc], mp);
              const float mref = mn == kNegInf ? 0.f : mn;  // both empty: stay empty
              const float a_self = fast_exp2(m_run[nb][cc] - mref), a_part = fast_exp2(mp - mref);
              l_run[nb][cc] = l_run[nb][cc] * a_self + lp * a_part;
              m_run[nb][cc] = mn;
#pragma unroll
              for (int mb = 0; mb < 8; ++mb) {
                o[mb][nb][cc] = o[mb][nb][cc] * a_self + mo[h * kMergeRow + mb * 16 + d_lo] * a_part;
                o[mb][nb][cc + 2] = o[mb][nb][cc + 2] * a_self + mo[h * kMergeRow + mb * 16 + d_hi] * a_part;
              }
            }
          }
          __syncwarp();
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int h0 = nb * 8 + 2 * t;
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
              mo[h0 * kMergeRow + mb * 16 + d_lo] = o[mb][nb][0];
              mo[(h0 + 1) * kMergeRow + mb * 16 + d_lo] = o[mb][nb][1];
              mo[h0 * kMergeRow + mb * 16 + d_hi] = o[mb][nb][2];
              mo[(h0 + 1) * kMergeRow + mb * 16 + d_hi] = o[mb][nb][3];
            }
            if (g == 0) {
              ml[h0 * 2] = m_run[nb][0];
              ml[h0 * 2 + 1] = l_run[nb][0];
              ml[h0 * 2 + 2] = m_run[nb][1];
              ml[h0 * 2 + 3] = l_run[nb][1];
            }
          }
        }
        named_bar_sync(1, kConsumerThreads);

        // (3) merge the pair states that hold dim d -- all four at D = 128; at D = 256 the
        //     two of half d / 128 (warps w0 and w0 + 2, whose partners hold the same softmax
        //     state for the same tokens): thread -> (head, dim)
        const long long F = prefix[b] + (long long)kvh * c.nt;  // first tile of this sequence
        const int first_cta = cta_of(F, T, P), last_cta = cta_of(F + c.nt - 1, T, P);
        const int n_parts = last_cta - first_cta + 1;
        // Cluster mode: a sequence whose parts all lie in this CTA's cluster leaves its state
        // in shared memory (slot 0 if it is this CTA's first segment, else slot 1) for the
        // on-chip merge after the loop.
        const bool on_chip = chip && n_parts > 1 && first_cta / cs == last_cta / cs;
        const int cslot = seg0 == start ? 0 : 1;
        if (on_chip && tid == 0) {  // this CTA merges its share of the sequence's outputs
          int* dt = duty + 4 * cslot;
          dt[0] = seq;
          dt[1] = first_cta;
          dt[2] = n_parts;
          dt[3] = F == split(first_cta) ? 0 : 1;  // the slot the first part sits in
        }
        constexpr int kHold = kWide ? kGroupWarps / 2 : kGroupWarps;  // warps holding a dim
        constexpr int kWStep = kGroupWarps / kHold;
        const int d = tid % DIM, dl = d & 127, w0 = kWide ? (d >> 7) : 0;
        for (int h = tid / DIM; h < G; h += kHStep) {
          float M = kNegInf;
#pragma unroll
          for (int i = 0; i < kHold; ++i) M = fmaxf(M, merge_ml[((w0 + i * kWStep) * HP + h) * 2]);
          float lsum = 0.f, acc = 0.f;
#pragma unroll
          for (int i = 0; i < kHold; ++i) {
            const int w = w0 + i * kWStep;
            const float f = fast_exp2(merge_ml[(w * HP + h) * 2] - M);  // 0 for a pair with no tokens
            lsum += f * merge_ml[(w * HP + h) * 2 + 1];
            acc += f * merge_o[(w * HP + h) * kMergeRow + dl];
          }
          if constexpr (KV8) acc *= p.v_scale;  // V = v_cache * v_scale (linear through every merge)
          if (on_chip) {
            if (ok(cslot >= 0 && cslot < 2 && h < HP) && sm_ok(smem_u32(cpart_ml + (cslot * HP + h) * 2), 8)) {
              cpart_o[(cslot * HP + h) * DIM + d] = acc;
              if (d == 0) {
                cpart_ml[(cslot * HP + h) * 2] = M;
                cpart_ml[(cslot * HP + h) * 2 + 1] = lsum;
              }
            }
          } else if (n_parts == 1) {
            if (attn_ok(b, kvh * G + h, d))
              p.attn[(long long)b * p.a_sb + (long long)(kvh * G + h) * p.a_sh + d] = __float2bfloat16_rn(acc / lsum);
          } else if (ok((long long)cta + seq < p.part_slots && h < p.gpad)) {
            // evict-last: a part written early in the launch (a range's first segment) must
            // still be in L2 when the sequence's last CTA merges it, after the K/V stream
            const uint64_t keep = l2_policy_evict_last();
            const long long slot = (long long)cta + seq;
            st_global_hint(p.part_o + (slot * p.gpad + h) * DIM + d, acc, keep);
            if (d == 0) {
              st_global_hint(p.part_ml + (slot * p.gpad + h) * 2, M, keep);
              st_global_hint(p.part_ml + (slot * p.gpad + h) * 2 + 1, lsum, keep);
            }
          }
        }
        if (!on_chip && n_parts > 1) {
          named_bar_sync(1, kConsumerThreads);  // every thread's partial stores precede the release
          if (tid == 0)
            flags[1] = ok(seq >= 0 && seq < B * Hkv) && atomic_add_acq_rel_gpu(p.counters + seq, 1) == n_parts - 1;
          named_bar_sync(1, kConsumerThreads);  // ... and the acquire precedes every thread's loads
          if (flags[1]) {  // every other part has landed: merge them all, in one pass
            // Thread (h, d) loads the parts' (m, l, O[h][d]) for two of its heads together,
            // eight parts per batch from clamped (always valid) addresses, masked afterwards,
            // and merges them with a running maximum: one L2 round trip per eight parts and
            // head pair after the counter (a thread holds G / (256 / D) heads: two at G = 4).
            for (int h = tid / DIM; h < G; h += 2 * kHStep) {
              const int hs[2] = {h, h + kHStep < G ? h + kHStep : h};
              float M[2] = {kNegInf, kNegInf}, lsum[2] = {0.f, 0.f}, acc[2] = {0.f, 0.f};
              for (int p0 = 0; p0 < n_parts; p0 += 8) {
                float mv[2][8], lv[2][8], ov[2][8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  long long slot = (long long)first_cta + min(p0 + u, n_parts - 1) + seq;
                  if (!ok(slot >= 0 && slot < p.part_slots)) slot = 0;
#pragma unroll
                  for (int k = 0; k < 2; ++k) {
                    const float* ml = p.part_ml + (slot * p.gpad + hs[k]) * 2;
                    mv[k][u] = __ldcg(ml);
                    lv[k][u] = __ldcg(ml + 1);
                    ov[k][u] = __ldcg(p.part_o + (slot * p.gpad + hs[k]) * DIM + d);
                  }
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                  float Mc = M[k];
#pragma unroll
                  for (int u = 0; u < 8; ++u)
                    if (p0 + u < n_parts) Mc = fmaxf(Mc, mv[k][u]);  // every part holds a token: finite
                  const float r = fast_exp2(M[k] - Mc);              // 0 on the first batch
                  lsum[k] *= r;
                  acc[k] *= r;
#pragma unroll
                  for (int u = 0; u < 8; ++u)
                    if (p0 + u < n_parts) {
                      const float f = fast_exp2(mv[k][u] - Mc);
                      lsum[k] += f * lv[k][u];
                      acc[k] += f * ov[k][u];
                    }
                  M[k] = Mc;
                }
              }
#pragma unroll
              for (int k = 0; k < 2; ++k)
                if ((k == 0 || hs[1] != h) && attn_ok(b, kvh * G + hs[k], d))
                  p.attn[(long long)b * p.a_sb + (long long)(kvh * G + hs[k]) * p.a_sh + d] =
                      __float2bfloat16_rn(acc[k] / lsum[k]);
            }
            if (tid == 0) p.counters[seq] = 0;  // ready for the next call
          }
        }
        named_bar_sync(1, kConsumerThreads);  // merge scratch and flags free again
        // the next segment starts from an empty state
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          m_run[nb][0] = m_run[nb][1] = kNegInf;
          l_run[nb][0] = l_run[nb][1] = 0.f;
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) o[mb][nb][0] = o[mb][nb][1] = o[mb][nb][2] = o[mb][nb][3] = 0.f;
        }
      }
    }
    if constexpr (kFused) {
      // This CTA's attention outputs (its own segments and every merge it performed)
      // are written: arrive at the grid barrier (release covers all consumer stores).
      named_bar_sync(1, kConsumerThreads);
      if (tid == 0) atomic_add_acq_rel_gpu(p.grid_sync, 1);
      if (warp == kGroupWarps) {  // first warp of group 1 issues the MMAs
        if (lane == 0) fused_mma<NPAD, S>(p, ring, bars, tmem, flags);
        __syncwarp();
      } else if (warp < kGroupWarps) {  // group 0 drains TMEM
        fused_epilogue<NPAD, S>(p, bars, tmem, flags, warp, lane, tid);
        tc_fence_before_sync();
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if (!SCORES && chip) {
    // Cluster mode: every sequence whose parts lie in this cluster is merged here. Each CTA
    // holding a part merges its share of the (head, dim) outputs over all the parts, in
    // CTA order, reading their shared memory (distributed shared memory: no global
    // partials, no counter, no L2 round trip).
    cluster_sync();  // every CTA's states are in its shared memory
    const uint32_t o_base = smem_u32(cpart_o), ml_base = smem_u32(cpart_ml);
    for (int k = 0; k < 2; ++k) {
      const int np = duty[4 * k + 2];
      if (np == 0) continue;
      const int sq = duty[4 * k], f = duty[4 * k + 1], fslot = duty[4 * k + 3];
      const int bq = sq / Hkv, kq = sq - bq * Hkv;
      if (!ok(np <= cs && cta >= f && cta - f < np && fslot >= 0 && fslot < 2 && sq >= 0 && sq < B * Hkv)) continue;
      const int items = G * DIM, chunk = (items + np - 1) / np, mine = cta - f;
      const int i_end = min(items, (mine + 1) * chunk);
      // NP >= np parts, all loads of an item in flight together (as many as the parts need)
      auto merge = [&](auto np_max) {
        constexpr int NP = decltype(np_max)::value;
        for (int item = mine * chunk + tid; item < i_end; item += kThreads) {
          const int h = item / DIM, d = item - h * DIM;
          float mv[NP], lv[NP], ov[NP];
#pragma unroll
          for (int q = 0; q < NP; ++q) {
            const int qq = min(q, np - 1);
            // the first part is in the slot its CTA chose; the others are their CTAs' first segments
            const uint32_t slot = qq == 0 ? (uint32_t)fslot : 0u;
            const uint32_t rank = (uint32_t)((f + qq) % cs);
            mv[q] = ld_cluster_f32(cluster_map(ml_base + 8u * (slot * HP + h), rank));
            lv[q] = ld_cluster_f32(cluster_map(ml_base + 8u * (slot * HP + h) + 4u, rank));
            ov[q] = ld_cluster_f32(cluster_map(o_base + 4u * (uint32_t)((slot * HP + h) * DIM + d), rank));
          }
          float M = kNegInf;
#pragma unroll
          for (int q = 0; q < NP; ++q)
            if (q < np) M = fmaxf(M, mv[q]);  // every part holds a token: finite
          float lsum = 0.f, acc = 0.f;
#pragma unroll
          for (int q = 0; q < NP; ++q)
            if (q < np) {
              const float w = fast_exp2(mv[q] - M);
              lsum += w * lv[q];
              acc += w * ov[q];
            }
          if (attn_ok(bq, kq * G + h, d))
            p.attn[(long long)bq * p.a_sb + (long long)(kq * G + h) * p.a_sh + d] = __float2bfloat16_rn(acc / lsum);
        }
      };
      if (np <= 2) merge(std::integral_constant<int, 2>());
      else if (np <= 4) merge(std::integral_constant<int, 4>());
      else merge(std::integral_constant<int, kMaxAttnCluster>());
    }
    cluster_sync();  // no CTA leaves while another still reads its shared memory
  }
  if (kFused && warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NB, bool SCORES, int S, int NPAD, int DIM, bool PAGED = false, bool KV8 = false>
cudaError_t launch_one(const AttnParams& p, int grid, cudaStream_t stream) {
  // The shared-memory opt-in is a per-device function attribute: set it once per device.
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(attn_decode_kernel<NB, SCORES, S, NPAD, DIM, PAGED, KV8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem);
    if (e != cudaSuccess) return e;
    // All of the SM's unified L1 as shared memory, the carveout of the projection kernel
    // too, so that three projection CTAs fit on an SM the moment this kernel leaves it.
    e = cudaFuncSetAttribute(attn_decode_kernel<NB, SCORES, S, NPAD, DIM, PAGED, KV8>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(attn_threads(attn_producers(PAGED, NPAD > 0, SCORES)));
  cfg.dynamicSmemBytes = attn_smem_bytes(p.B, NB, S, DIM, kStageBytes, p.cluster > 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  if (NPAD > 0) {
    attr[0].id = cudaLaunchAttributeCooperative;  // the fused step's grid barrier needs every CTA resident
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeClusterDimension;  // cluster mode: on-chip merges
    attr[0].val.clusterDim.x = p.cluster > 1 ? p.cluster : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  }
  // early launch behind the previous kernel (the kernel waits before any global access)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (NPAD == 0 && p.pdl) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<NB, SCORES, S, NPAD, DIM, PAGED, KV8>, p);
}

}  // namespace
}  // namespace da
