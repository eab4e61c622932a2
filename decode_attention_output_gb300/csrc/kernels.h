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
// Head dims the kernel implements: 128, and 256 (the two-halves contraction of a
// D = 256 GQA decode). A stage always holds 32 KB: a K tile and a V tile of
// tile_tokens(D) tokens x D dims in 64-dim boxes of 128-byte swizzled rows.
constexpr int kHeadDim = 128;
constexpr int kHeadDimWide = 256;
__host__ __device__ constexpr int tile_tokens(int dim) { return dim == kHeadDimWide ? 32 : 64; }
constexpr int kTile = 64;                      // tokens per pipeline stage at D = 128
constexpr int kGroupWarps = 4;                 // consumer warps per group; each owns 16 tokens of a stage
constexpr int kGroups = 2;                     // consumer groups take alternate stages
constexpr int kConsumerThreads = kGroups * kGroupWarps * 32;
// Producer warps of the attention kernel: one per consumer group (each issues the tiles of
// its group's stages) for a paged cache, where small blocks mean several copies per tile and
// one lane's issue rate set the pace; for a contiguous cache when kContigTwoProducers.
constexpr bool kContigTwoProducers = true;
__host__ __device__ constexpr int attn_producers(bool paged, bool fused, bool scores) {
  return paged || (kContigTwoProducers && !fused && !scores) ? 2 : 1;
}
__host__ __device__ constexpr int attn_threads(int producers) { return kConsumerThreads + 32 * producers; }
constexpr int kMaxStages = 6;                  // even stage counts: stage s always belongs to group s % 2
constexpr int kKTileBytes = 16384;             // K tile: tile_tokens(D) x D x bf16 (both head dims)
constexpr int kStageBytes = 2 * kKTileBytes;   // K tile + V tile
__host__ __device__ constexpr int box_bytes(int dim) { return tile_tokens(dim) * 128; }  // 64 dims of a tile
__host__ __device__ constexpr int q_row_bytes(int dim) { return dim * 2 + 16; }  // + 16 B pad: conflict-free
                                                                                 // fragment loads
constexpr int kMaxGroup = 16;
constexpr int kMaxBatch = 1024;
constexpr int kMergeRow = 132;                 // floats per head row of the merge scratch (128 + pad); at
                                               // D = 256 a warp holds one 128-dim half of the output
constexpr int kMaxAttnCtas = 512;              // persistent CTAs of the attention kernel (and so parts
                                               // per sequence) at most
static_assert(tile_tokens(kHeadDim) * kHeadDim * 2 == kKTileBytes, "K tile bytes at D = 128");
static_assert(tile_tokens(kHeadDimWide) * kHeadDimWide * 2 == kKTileBytes, "K tile bytes at D = 256");
// Shared-memory carve-up of the attention kernel; nb = 8-head blocks (1 or 2),
// stages = pipeline depth (even, so that a stage always belongs to one consumer group),
// dim = head dim (128 or 256).
struct AttnSmem {
  int nb, batch, stages, dim, stage_bytes;
  __host__ __device__ constexpr AttnSmem(int nb_, int batch_, int stages_, int dim_ = kHeadDim,
                                         int stage_bytes_ = kStageBytes)
      : nb(nb_), batch(batch_), stages(stages_), dim(dim_), stage_bytes(stage_bytes_) {}
  __host__ __device__ constexpr int heads() const { return 8 * nb; }
  __host__ __device__ constexpr size_t q_slot() const { return (size_t)heads() * q_row_bytes(dim); }
  __host__ __device__ constexpr size_t off_q() const { return (size_t)stages * stage_bytes; }
  __host__ __device__ constexpr size_t off_merge_o() const { return off_q() + stages * q_slot(); }
  __host__ __device__ constexpr size_t off_merge_ml() const {
    return off_merge_o() + (size_t)kGroupWarps * heads() * kMergeRow * 4;
  }
  __host__ __device__ constexpr size_t off_bars() const { return off_merge_ml() + (size_t)kGroupWarps * heads() * 2 * 4; }
  // barriers: full[S], empty[S] (attention); full[8], empty[8], accum[2] (fused projection)
  __host__ __device__ constexpr size_t off_flags() const { return off_bars() + (2 * stages + 18) * 8; }
  // flags: int [16]: [0] abort, [1] last CTA of a sequence, [2] last CTA of a column tile (fused
  // step), [3] TMEM address, [8..15] this CTA's range of tiles and the cursor at its first tile
  __host__ __device__ constexpr size_t off_prefix() const { return off_flags() + 64; }
  __host__ __device__ constexpr size_t off_lens() const { return off_prefix() + (size_t)(batch + 1) * 4; }
  // paged caches: kIdTiles rows of 16 block ids (one 64-byte TMA box per tile), rows
  // 128 bytes apart (a tensor copy's shared-memory destination is 128-byte aligned)
  __host__ __device__ constexpr size_t off_ids() const { return (off_lens() + (size_t)batch * 4 + 127) & ~(size_t)127; }
  // cluster mode: this CTA's merged states of the sequences it shares with other CTAs of its
  // cluster (slot 0: its first segment, slot 1: its last), read by those CTAs:
  // O [2][heads][dim], then (m, l) [2][heads][2], then the merge duties int [2][4] (and 16
  // bytes of padding)
  __host__ __device__ constexpr size_t off_cpart() const { return off_ids() + kIdTiles * kIdStride * 4; }
  __host__ __device__ constexpr size_t cpart_bytes() const { return 2 * (size_t)heads() * (dim + 2) * 4 + 48; }
  // the cluster-mode states only in clusters (at most half as many sequences as SMs)
  __host__ __device__ constexpr size_t total(bool cluster = false) const {
    return 1024 + off_cpart() + (cluster ? cpart_bytes() : 0);
  }
  static constexpr int kIdTiles = 8;
  static constexpr int kIdRow = 16;     // entries a row receives
  static constexpr int kIdStride = 32;  // entries between rows (128 bytes)
};

constexpr size_t kMaxDynSmem = 232448;  // 227 KB per CTA on sm_100-class GPUs
constexpr size_t attn_smem_bytes(int batch, int nb, int stages, int dim = kHeadDim, int stage_bytes = kStageBytes,
                                 bool cluster = false) {
  return AttnSmem(nb, batch, stages, dim, stage_bytes).total(cluster);
}
// fp8 (e4m3) caches: a tile is 128 tokens (128 x 128 dims x 1 byte of K and of V), so a
// stage holds the same 32 KB and the ring the same 4 stages as for bf16.
constexpr int kTileFp8 = 128;
static_assert(AttnSmem(2, kMaxBatch, 4).total() <= kMaxDynSmem, "attention kernel exceeds 227 KB of shared memory");
// Cluster mode needs room for two parked states: every group width at D = 128, up to
// eight heads per group at D = 256 (the host checks each launch; wider groups at D = 256
// merge through L2).
static_assert(AttnSmem(2, 128, 4).total(true) <= kMaxDynSmem, "cluster mode (D = 128) exceeds 227 KB");
static_assert(AttnSmem(1, 128, 4, kHeadDimWide).total(true) <= kMaxDynSmem, "cluster mode (D = 256) exceeds 227 KB");
static_assert(AttnSmem(2, kMaxBatch, 4, kHeadDimWide).total() <= kMaxDynSmem,
              "attention kernel (D = 256) exceeds 227 KB of shared memory");
// 4 stages by default (measured faster than 6 on the GB300: deeper rings slowed the
// stream); 6 on request when it fits this batch and group width (D = 128 only).
constexpr int attn_stages_for(int batch, int nb, int requested, bool cluster = false) {
  return requested == kMaxStages && attn_smem_bytes(batch, nb, kMaxStages, kHeadDim, kStageBytes, cluster) <= kMaxDynSmem
             ? kMaxStages
             : 4;
}

struct AttnParams {
  CUtensorMap tm_k;  // [B][Hkv][Lcap][D] bf16, box 64 dims x tile_tokens(D) tokens, 128B swizzle
  CUtensorMap tm_v;
  const __nv_bfloat16* q;
  long long q_sb, q_sh;  // element strides of q [B][Hq][D]
  const int* seq_lens;
  __nv_bfloat16* attn;   // [B][Hq][D] bf16 result
  long long a_sb, a_sh;
  float* scores;         // [B][Hq][Lcap] fp32 (scores-only mode)
  long long s_sb, s_sh;
  float* part_o;         // [slots][gpad][D] unnormalised partial outputs
  float* part_ml;        // [slots][gpad][2]   (running max in log2 units, sum)
  long long part_slots;  // slots of part_o / part_ml (checked in the bounds-checked build)
  int* counters;         // [B*Hkv] completion counters (zero between calls)
  int* err;              // device error word
  int B, Hkv, G, Lcap;
  int gpad;              // 8 or 16 (heads per group rounded up to the MMA width)
  float scale_log2;      // scale * log2(e)
  // Optional region the next kernel reads (the projection weights): pulled into L2
  // in pieces while the K/V stream runs. prefetch_bytes = 0 disables it.
  const char* prefetch;
  long long prefetch_bytes;
  int stages;            // requested pipeline depth (4 or 6)
  // Fused step only (decode_attn_fwd in one launch): the projection of this kernel's
  // own attention output (attn, contiguous [B][K]) by W_o, on tcgen05 after a grid barrier.
  CUtensorMap tm_w;      // W_o [K][N] bf16: box 64 columns x 64 rows, 128B swizzle
  CUtensorMap tm_x;      // attention output [B][K] bf16: box 64 k x npad rows, 128B swizzle
  __nv_bfloat16* y;      // [B][N]
  long long y_sb;
  float* proj_part;      // [slots][B][128] fp32 split-K partials
  long long proj_part_floats;  // floats of proj_part (checked in the bounds-checked build)
  int* proj_counters;    // [column tiles], zero between calls
  int* grid_sync;        // [2]: arrivals, departures of the grid barrier, zero between calls
  unsigned long long sync_limit_ns;  // the grid barrier's wait limit (0: two seconds)
  int sync_extra;        // arrivals the grid barrier waits for beyond the grid (0; a test sets 1
                         // to make the wait run out)
  int N, K, kb_per_tile, units;  // units = column tiles x k-blocks of 64
  int attn_workers;      // CTAs that take attention tiles (<= grid); the fused step may leave
                         // some CTAs free to start on W_o at once
  // Paged cache only: tm_k / tm_v map [num_blocks][Hkv][block_size][D]; token t of sequence b
  // is row t % block_size of block block_table[b * bt_stride + t / block_size].
  const int* block_table;
  long long bt_stride;
  long long bt_entries;  // flat extent of the table, (B - 1) * bt_stride + max_blocks
  int block_size, num_blocks;
  int block_shift;       // log2(block_size)
  CUtensorMap tm_table;  // the table as one flat int32 array (one row), box 16 entries
  // fp8 (e4m3) caches only: K = k_cache * k_scale, V = v_cache * v_scale
  float k_scale, v_scale;
  // Cluster mode (> 1): the grid is launched in clusters of `cluster` consecutive CTAs; the
  // tiles are split over the CTAs as always, and a sequence whose parts all lie in one
  // cluster merges them in distributed shared memory (the others through L2).
  int cluster;
  int pdl;  // 1: launched with programmatic dependent launch (waits before any global access)
  // > 0: each CTA lets the next kernel launch when it reaches the tile this many before the
  // end of its range; 0: right after set-up
  int trigger_at;
  // floor(n / d) = (n * split_mul) >> split_shift, exact for 0 <= n < 2^31, for the two worker
  // counts d that split the tiles over the CTAs: [0] min(grid, attn_workers), [1] (cluster
  // mode) min(that, B * Hkv * cluster). A worker count that differs is divided the plain way.
  unsigned long long split_mul[2];
  int split_div[2], split_shift[2];
};
constexpr int kMaxAttnCluster = 8;  // portable cluster size

// Paged caches: a power of two from 8 tokens (tiles are cut into blocks, or blocks hold
// whole tiles; the producer's index arithmetic is shifts and masks).
__host__ __device__ constexpr bool paged_block_ok(int block_size, int dim) {
  return block_size >= 8 && block_size <= (1 << 20) && (block_size & (block_size - 1)) == 0 && dim > 0;
}

constexpr int kProjWBytes = 2 * 64 * 128;  // one stage of W_o: 128 columns x 64 k-rows
// Phase-B stages re-cut the attention ring (kStages x kStageBytes) into W_o + X tiles.
__host__ __device__ constexpr int proj_stage_bytes(int npad) { return kProjWBytes + ((npad * 128 + 1023) / 1024) * 1024; }
__host__ __device__ constexpr int proj_stages(int npad) {
  return (4 * kStageBytes) / proj_stage_bytes(npad) < 8 ? (4 * kStageBytes) / proj_stage_bytes(npad) : 8;
}

// grid = number of persistent CTAs; nb = 1 for G <= 8, 2 for G <= 16; dim = head dim
// (128 or 256); npad = 0 for the attention alone, else the batch padding (16/32/64/128)
// of the fused projection (a cooperative launch: every CTA must be resident for the
// grid barrier; D = 128 only).
cudaError_t launch_attention(const AttnParams& p, int grid, int nb, int dim, bool scores_only, cudaStream_t stream,
                             int npad = 0);
// The D = 256 instantiations (their own translation unit).
cudaError_t launch_attention_d256(const AttnParams& p, int grid, int nb, bool scores_only, cudaStream_t stream);
// Attention over a paged cache (p.block_table set), D = 128 or 256.
cudaError_t launch_attention_paged(const AttnParams& p, int grid, int nb, int dim, cudaStream_t stream);
// Attention over an fp8 (e4m3) cache, D = 128 (p.k_scale, p.v_scale set).
cudaError_t launch_attention_fp8(const AttnParams& p, int grid, int nb, cudaStream_t stream);
// Clusters of `cluster` attention CTAs (one per SM) that can be resident at once on the
// current device (the GPCs' SM counts leave some SMs out); 0 if the query fails.
int attn_max_active_clusters(int cluster);

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
  int* err;                // device error word (bounds-checked build)
  int B, K, N, kc, ksplit;
};

// bt = batch rows per CTA (1, 2, 4 or 8); grid = (col blocks, ksplit, batch chunks).
cudaError_t launch_gemv(const GemvParams& p, int bt, bool pdl, cudaStream_t stream);
size_t gemv_smem_bytes(int bt, int kc);


// ------------------------------------------- projection: tcgen05 tensor-core path
constexpr int kUmmaThreads = 128;  // warp 0: TMA producer, warp 1: MMA issuer, all four: epilogue
constexpr int kUmmaBM = 128;       // hidden columns per tile (the MMA's M, swap-AB)
constexpr int kUmmaBK = 64;        // k rows per pipeline stage

struct UmmaParams {
  CUtensorMap tm_w;  // W [K][N] bf16 row-major: box 64 columns x 64 rows, 128B swizzle
  CUtensorMap tm_x;  // X [B][K] bf16: box 64 k x npad batch rows, 128B swizzle
  __nv_bfloat16* y;  // [B][N]
  long long y_sb;
  float* part;       // [ksplit][B][N] fp32 split-K partials (null: the cluster reduction)
  int* counters;     // [batch chunks][column tiles]
  int* err;
  int B, K, N, ksplit;
  int prefetch;      // 1: pull the k-blocks past the first ring fill into L2 before the PDL wait
  int cluster;       // 1: the ksplit slices of a column tile are one cluster (ksplit <= 8)
};
constexpr int kMaxClusterSplit = 8;  // portable cluster size

// ---------------------------- projection of a single-row batch with W staged on chip
constexpr int kOnchipThreads = 512;   // thread t: 8 columns (piece t % 8 of column tile t / 64), rows (t / 8) % 8 + 8 i
constexpr int kOnchipCols = 512;      // columns of a CTA's group (1 KB of every row of W)
constexpr int kOnchipRegKblocks = 3;  // k-blocks (64 rows) a CTA holds in registers (8 x 16 bytes each per thread)

struct OnchipParams {
  CUtensorMap tm_w;          // W [K][N] bf16 row-major: box 64 columns x 64 rows, 128B swizzle
  const __nv_bfloat16* x;    // [K] the attention output of the one batch row (16-byte aligned)
  const __nv_bfloat16* w;    // W, for the register-held k-blocks
  long long w_sk;            // row stride of W in elements
  __nv_bfloat16* y;          // [N]
  float* part;               // [N / 512 groups][k-ranges][512] fp32 parts
  int* counters;             // [N / 512] completion counters, zero between calls
  int* err;
  int K, N;                  // K a multiple of 64, N of 512
  int kb;                    // K / 64
  int smem_kblocks;          // k-blocks a CTA stages in shared memory (the rest of its range in registers)
};
size_t onchip_smem_bytes(int smem_kblocks, int K);
int onchip_max_smem_kblocks(int K);
// grid = (N / 512 column groups, kgroups k-ranges): one CTA per SM that the attention leaves
// free; each CTA's k-range is at most smem_kblocks + kOnchipRegKblocks k-blocks.
cudaError_t launch_onchip(const OnchipParams& p, int kgroups, bool pdl, cudaStream_t stream);

size_t umma_smem_bytes(int npad);
// grid = (ceil(N / 128), ksplit, ceil(B / npad)); npad in {16, 32, 64, 128}.
cudaError_t launch_umma(const UmmaParams& p, int npad, bool pdl, cudaStream_t stream);

}  // namespace da
