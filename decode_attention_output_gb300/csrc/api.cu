// api.cu -- the C ABI declared in include/decode_attn.h: argument validation,
// the per-device workspace, TMA descriptor encoding, launch planning and dispatch.
// No arithmetic of the method happens here; every step runs in the kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "decode_attn.h"
#include "kernels.h"

namespace {

using namespace da;

// ------------------------------------------------------------------ options
struct Options {
  int64_t attn_ctas = 0;
  int64_t oproj_path = 0;  // 0 auto, 1 gemv, 2 tcgen05, 3 on-chip staged (batch 1 behind the attention)
  int64_t oproj_splitk = 0;
  int64_t gemm_min_batch = 1;  // tcgen05 from batch 1 (with the cluster reduction: batch 1 step
                               // 18.9 -> 16.4 us against the CUDA-core GEMV)
  int64_t pdl = 1;
  int64_t l2_prefetch = 0;  // decode_attn_fwd: the attention kernel pulls W_o into L2 while it
                            // streams K/V (measured slower: off)
  int64_t attn_stages = 4;  // attention pipeline depth, 4 or 6 (6 no faster with two producers)
  int64_t fused = 0;        // decode_attn_fwd as one persistent launch (measured slower so far: off)
  int64_t fused_attn_ctas = 0;  // attention workers of the fused step (0: about 4 tiles each)
  int64_t oproj_cluster = 1;    // tcgen05 projection: split-K slices reduce in a cluster
  int64_t attn_cluster = 1;     // attention in thread-block clusters with on-chip merges
  int64_t attn_pdl = 1;         // attention launched with programmatic dependent launch (eager
                                // batch-8 step 54.5 -> 52.2 us: its CTAs start as the previous kernel drains)
  int64_t oproj_prefetch = 0;   // tcgen05 projection behind the attention: pull the rest of each
                                // CTA's W slice into L2 before waiting (measured no faster: off)
  int64_t attn_trigger = 3;     // decode_attn_fwd: each attention CTA lets the projection launch
                                // this many tiles before its end (0: at set-up); 3 against 0:
                                // batch 1 15.9 -> 14.9 us, 131k context 306.2 -> 303.5 us
  int64_t grid_wait_us = 0;     // test hook: the fused step's grid-barrier wait limit (0: 2 s)
  int64_t grid_wait_extra = 0;  // test hook: arrivals that barrier waits for beyond the grid
};
std::mutex g_mu;
Options g_opt;

Options options_snapshot() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_opt;
}

// ---------------------------------------------------------------- workspace
// Fixed header (zeroed once when allocated, kept at zero by the kernels):
//   [0, 256)                      device error word
//   [256, 256 + 256 KiB)          attention completion counters (B*Hkv <= 65536)
//   [.., + 256 KiB)               projection completion counters
// followed by per-call scratch laid out by the caller.
constexpr size_t kMaxCounters = 65536;
constexpr size_t kErrOff = 0;
constexpr size_t kGridSyncOff = 64;  // two ints of the fused step's grid barrier
constexpr size_t kAttnCntOff = 256;
constexpr size_t kGemvCntOff = kAttnCntOff + kMaxCounters * 4;
constexpr size_t kHeaderBytes = kGemvCntOff + kMaxCounters * 4;
constexpr int kMaxDevices = 64;

struct Workspace {
  char* base = nullptr;
  size_t bytes = 0;
};
Workspace g_ws[kMaxDevices];

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Returns the workspace of the current device with at least `scratch` bytes after
// the header, growing it if needed. Growth is stream-ordered on `stream` (no device-wide
// synchronisation): the old block is released with cudaFreeAsync behind the work already
// queued on `stream`, the new one comes from cudaMallocAsync and its header is zeroed by
// cudaMemsetAsync, all on `stream`.
int workspace_get(size_t scratch, cudaStream_t stream, char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& ws = g_ws[dev];
  const size_t need = kHeaderBytes + align_up(scratch, 256);
  if (need > ws.bytes) {
    if (ws.base) {
      if (cudaFreeAsync(ws.base, stream) != cudaSuccess) return DA_ERR_CUDA;
      ws.base = nullptr;
      ws.bytes = 0;
    }
    const size_t bytes = std::max(need, (size_t)32 << 20);
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) {
      cudaGetLastError();
      return DA_ERR_NOMEM;
    }
    if (cudaMemsetAsync(p, 0, kHeaderBytes, stream) != cudaSuccess) {
      cudaFreeAsync(p, stream);
      return DA_ERR_CUDA;
    }
    ws.base = static_cast<char*>(p);
    ws.bytes = bytes;
  }
  *out = ws.base;
  return DA_OK;
}

// --------------------------------------------------------------- device info
int sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// ------------------------------------------------------------ TMA encoding
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 5-D map over a [B][Hkv][Lcap][D] bf16 cache (or a [num_blocks][Hkv][block_size][D]
// page pool) with the head dim split in two: {64 dims, token, D/64 dim boxes, head,
// batch (or block)}. One box = 64 dims x box_tokens tokens x all D/64 dim boxes, which
// lands in shared memory as D/64 consecutive 64-dim boxes of box_tokens rows (128-byte
// rows, 128-byte swizzle): one copy per tile and tensor (box_tokens 0: tile_tokens(D)).
// An fp8 (e4m3) cache is mapped the same way with 128-dim boxes (128-byte rows): at
// D = 128 a tile is one box of 64 tokens x 128 bytes.
int encode_kv_map(CUtensorMap* map, const da_tensor_t* t, int box_tokens = 0) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return DA_ERR_CUDA;
  const int64_t B = t->shape[0], H = t->shape[1], L = t->shape[2], D = t->shape[3];
  const int64_t es = t->dtype == DA_DTYPE_E4M3 ? 1 : 2, inner = 128 / es;  // elements per 128-byte box row
  // a stride of an extent-1 dimension is never used; give it a harmless legal value
  const int64_t st = L == 1 ? D : t->stride[2];
  const int64_t sh = H == 1 ? st * L : t->stride[1];
  const int64_t sb = B == 1 ? sh * H : t->stride[0];
  cuuint64_t dims[5] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)(D / inner), (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[4] = {(cuuint64_t)(st * es), 128, (cuuint64_t)(sh * es), (cuuint64_t)(sb * es)};
  cuuint32_t box[5] = {(cuuint32_t)inner, (cuuint32_t)(box_tokens > 0 ? box_tokens : tile_tokens((int)D)),
                       (cuuint32_t)(D / inner), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUtensorMapDataType type = es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, type, 5, t->data, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_UNSUPPORTED;
}

// Map over a block table seen as one flat int32 array of `entries` (a 2-D map of one
// row); box = 16 entries.
int encode_table_map(CUtensorMap* map, const void* base, int64_t entries) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return DA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)entries, 1};
  cuuint64_t strides[1] = {(cuuint64_t)align_up((size_t)entries * 4, 16)};
  cuuint32_t box[2] = {16, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_UNSUPPORTED;
}

// 2-D map over a row-major bf16 matrix [rows][cols] with row stride `ld` elements;
// box = 64 columns x box_rows rows, 128-byte swizzle.
int encode_2d_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return DA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(rows == 1 ? cols : ld) * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DA_OK : DA_ERR_UNSUPPORTED;
}

// --------------------------------------------------------------- validation
enum Use { kInput16, kOutput };  // inputs feed TMA / 16-byte loads, outputs take scalar stores

int elem_size(int dtype) { return dtype == DA_DTYPE_BF16 ? 2 : (dtype == DA_DTYPE_E4M3 ? 1 : 4); }

int check_tensor(const da_tensor_t* t, int dtype, int ndim, Use use) {
  if (!t) return DA_ERR_NULL;
  if (t->dtype != dtype) return DA_ERR_DTYPE;
  if (t->ndim != ndim) return DA_ERR_SHAPE;
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return DA_ERR_SHAPE;
    numel *= t->shape[i];
  }
  if (numel == 0) return DA_OK;  // empty: the caller decides whether that is allowed
  if (!t->data) return DA_ERR_NULL;
  if (t->shape[ndim - 1] > 1 && t->stride[ndim - 1] != 1) return DA_ERR_STRIDE;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(t->data);
  if (use == kInput16) {
    if (addr % 16) return DA_ERR_ALIGN;
    for (int i = 0; i < ndim - 1; ++i)
      if (t->shape[i] > 1 && (t->stride[i] <= 0 || (t->stride[i] * elem_size(dtype)) % 16)) return DA_ERR_STRIDE;
  } else {
    if (addr % elem_size(dtype)) return DA_ERR_ALIGN;
    for (int i = 0; i < ndim - 1; ++i)
      if (t->shape[i] > 1 && t->stride[i] <= 0) return DA_ERR_STRIDE;
  }
  return DA_OK;
}

#define DA_TRY(expr)          \
  do {                        \
    const int _rc = (expr);   \
    if (_rc != DA_OK) return _rc; \
  } while (0)

struct AttnShape {
  int B, Hq, Hkv, G, Lcap, D;
};

int check_attention_inputs(const da_tensor_t* q, const da_tensor_t* k, const da_tensor_t* v,
                           const da_tensor_t* lens, bool need_v, AttnShape* s, int kv_dtype = DA_DTYPE_BF16) {
  DA_TRY(check_tensor(q, DA_DTYPE_BF16, 3, kInput16));
  DA_TRY(check_tensor(k, kv_dtype, 4, kInput16));
  if (need_v) DA_TRY(check_tensor(v, kv_dtype, 4, kInput16));
  if (!lens) return DA_ERR_NULL;
  if (lens->dtype != DA_DTYPE_I32) return DA_ERR_DTYPE;
  if (lens->ndim != 1) return DA_ERR_SHAPE;
  const int64_t B = q->shape[0], Hq = q->shape[1], Hkv = k->shape[1], Lcap = k->shape[2], D = q->shape[2];
  if (k->shape[3] != D) return DA_ERR_SHAPE;
  if (D != kHeadDim && D != kHeadDimWide) return DA_ERR_SHAPE;
  if (kv_dtype == DA_DTYPE_E4M3 && D != kHeadDim) return DA_ERR_UNSUPPORTED;  // fp8 caches: D = 128
  if (k->shape[0] != B || lens->shape[0] != B) return DA_ERR_SHAPE;
  if (need_v)
    for (int i = 0; i < 4; ++i)
      if (v->shape[i] != k->shape[i]) return DA_ERR_SHAPE;
  if (B > 0) {
    if (!lens->data) return DA_ERR_NULL;
    if (B > 1 && lens->stride[0] != 1) return DA_ERR_STRIDE;
    if (reinterpret_cast<uintptr_t>(lens->data) % 4) return DA_ERR_ALIGN;
  }
  if (Hq <= 0 || Hkv <= 0 || Lcap <= 0) return DA_ERR_SHAPE;
  if (Hq % Hkv) return DA_ERR_SHAPE;
  if (Hq / Hkv > kMaxGroup) return DA_ERR_UNSUPPORTED;
  if (B > DA_MAX_BATCH) return DA_ERR_UNSUPPORTED;
  if (B * Hkv > (int64_t)kMaxCounters) return DA_ERR_UNSUPPORTED;
  if (Lcap > (int64_t)1 << 30) return DA_ERR_UNSUPPORTED;
  const int64_t tt = tile_tokens((int)D);
  if (B * Hkv * ((Lcap + tt - 1) / tt) >= ((int64_t)1 << 31)) return DA_ERR_UNSUPPORTED;
  s->B = (int)B;
  s->Hq = (int)Hq;
  s->Hkv = (int)Hkv;
  s->G = (int)(Hq / Hkv);
  s->Lcap = (int)Lcap;
  s->D = (int)D;
  return DA_OK;
}

// A paged cache: k_pages / v_pages [num_blocks][Hkv][block_size][D] bf16 (any strides obeying
// the conventions), block_table [B][max_blocks] int32 (rows contiguous), seq_lens [B].
// The logical capacity is max_blocks * block_size.
struct PagedShape {
  const int* table;
  long long table_stride, table_entries;  // row stride; flat extent (B-1)*stride + max_blocks
  int block_size, num_blocks;
};

int check_paged_inputs(const da_tensor_t* q, const da_tensor_t* kp, const da_tensor_t* vp,
                       const da_tensor_t* table, const da_tensor_t* lens, AttnShape* s, PagedShape* ps) {
  DA_TRY(check_tensor(q, DA_DTYPE_BF16, 3, kInput16));
  DA_TRY(check_tensor(kp, DA_DTYPE_BF16, 4, kInput16));
  DA_TRY(check_tensor(vp, DA_DTYPE_BF16, 4, kInput16));
  if (!table || !lens) return DA_ERR_NULL;
  if (table->dtype != DA_DTYPE_I32 || lens->dtype != DA_DTYPE_I32) return DA_ERR_DTYPE;
  if (table->ndim != 2 || lens->ndim != 1) return DA_ERR_SHAPE;
  const int64_t B = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t NB = kp->shape[0], Hkv = kp->shape[1], BS = kp->shape[2], MB = table->shape[1];
  if (D != kHeadDim && D != kHeadDimWide) return DA_ERR_SHAPE;
  if (kp->shape[3] != D) return DA_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (vp->shape[i] != kp->shape[i]) return DA_ERR_SHAPE;
  if (table->shape[0] != B || lens->shape[0] != B) return DA_ERR_SHAPE;
  if (Hq <= 0 || Hkv <= 0 || NB <= 0 || BS <= 0 || MB <= 0) return DA_ERR_SHAPE;
  if (Hq % Hkv) return DA_ERR_SHAPE;
  if (!paged_block_ok((int)std::min<int64_t>(BS, 1 << 30), (int)D)) return DA_ERR_UNSUPPORTED;
  if (Hq / Hkv > kMaxGroup) return DA_ERR_UNSUPPORTED;
  if (B > DA_MAX_BATCH) return DA_ERR_UNSUPPORTED;
  if (B * Hkv > (int64_t)kMaxCounters) return DA_ERR_UNSUPPORTED;
  if (NB >= ((int64_t)1 << 31) || BS > ((int64_t)1 << 20)) return DA_ERR_UNSUPPORTED;
  const int64_t Lcap = MB * BS;
  if (MB > ((int64_t)1 << 30) || Lcap > ((int64_t)1 << 30)) return DA_ERR_UNSUPPORTED;
  const int64_t tt = tile_tokens((int)D);
  if (B * Hkv * ((Lcap + tt - 1) / tt) >= ((int64_t)1 << 31)) return DA_ERR_UNSUPPORTED;
  if (B > 0) {
    if (!lens->data || !table->data) return DA_ERR_NULL;
    if (B > 1 && lens->stride[0] != 1) return DA_ERR_STRIDE;
    if (MB > 1 && table->stride[1] != 1) return DA_ERR_STRIDE;
    if (B > 1 && table->stride[0] < MB) return DA_ERR_STRIDE;
    if (reinterpret_cast<uintptr_t>(lens->data) % 4 || reinterpret_cast<uintptr_t>(table->data) % 16)
      return DA_ERR_ALIGN;  // the table is read by TMA: 16-byte aligned base
    if ((B - 1) * table->stride[0] + MB >= ((int64_t)1 << 31)) return DA_ERR_UNSUPPORTED;
  }
  s->B = (int)B;
  s->Hq = (int)Hq;
  s->Hkv = (int)Hkv;
  s->G = (int)(Hq / Hkv);
  s->Lcap = (int)Lcap;
  s->D = (int)D;
  ps->table = static_cast<const int*>(table->data);
  ps->table_stride = B > 1 ? table->stride[0] : MB;
  ps->table_entries = B > 0 ? (B - 1) * ps->table_stride + MB : 0;
  ps->block_size = (int)BS;
  ps->num_blocks = (int)NB;
  return DA_OK;
}

// ------------------------------------------------------------------ planning
struct AttnPlan {
  int grid, nb, gpad;
  long long slots;  // split-KV partial slots in the scratch
  int cluster;    // > 1: CTAs per sequence in cluster mode
  int flat_grid;  // the grid without cluster mode (the fall-back if a cluster launch is refused)
  size_t part_o_off, part_ml_off, bytes;
};

// Persistent CTAs of the attention kernel: one per SM, or fewer for small problems, about
// four tiles each counted from the cache capacity (an upper bound of the device-side
// lengths): at batch 1, kv_len 2048 (256 tiles) 64 CTAs took 9.1 us against 10.1 us for 152
// (fewer parts per sequence to merge, the same bytes in flight). `tile_tok` = tokens per
// tile of the variant (64 at D = 128, 32 at D = 256, 128 for an fp8 cache). The fused
// step keeps one CTA per SM: its projection phase runs on every CTA.
// `clustered`: cluster mode may be used (the attention-only entry points: with the projection
// kernel's CTAs streaming W beside it, the cluster-placed attention streams slower and the
// batch-1 step measured 16.9 against 16.3 us; alone it is 8.0 against 9.1 us).
// Where the cluster mode may be used: nowhere, only above about four tiles per SM, or at
// any size.
enum class ClusterUse { kNever, kLarge, kAny };

ClusterUse cluster_use_only(const Options& o) {  // the attention-only entry points
  return o.attn_cluster ? ClusterUse::kAny : ClusterUse::kNever;
}
// decode_attn_fwd: at batch 1 the flat grid gave the faster step (15.0 vs 15.7 us)
// (2: at every size there too)
ClusterUse cluster_use_fwd(const Options& o) {
  return o.attn_cluster == 2 ? ClusterUse::kAny : (o.attn_cluster ? ClusterUse::kLarge : ClusterUse::kNever);
}

// Clusters of cs attention CTAs resident at once on the current device (cached).
int max_active_clusters(int cs) {
  static std::mutex mu;
  static int cache[kMaxDevices][kMaxAttnCluster + 1];
  static bool known[kMaxDevices][kMaxAttnCluster + 1];
  int dev = 0;
  if (cs < 2 || cs > kMaxAttnCluster || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!known[dev][cs]) {
    cache[dev][cs] = attn_max_active_clusters(cs);
    known[dev][cs] = true;
  }
  return cache[dev][cs];
}

AttnPlan plan_attention(const AttnShape& s, const Options& o, int tile_tok = 0, bool fused = false,
                        ClusterUse clustered = ClusterUse::kNever) {
  AttnPlan pl;
  const int sms = std::max(1, sm_count());
  if (tile_tok <= 0) tile_tok = tile_tokens(s.D);
  const long long seqs = (long long)s.B * s.Hkv, tiles_seq = (s.Lcap + tile_tok - 1) / tile_tok;
  const long long tiles = seqs * tiles_seq;
  const int auto_grid = fused ? sms : (int)std::max<long long>(1, std::min<long long>(sms, (tiles + 3) / 4));
  // at most kMaxAttnCtas workers: a sequence then has at most that many parts, whose merge
  // weights fit the kernel's merge scratch
  pl.grid = std::min(o.attn_ctas > 0 ? (int)o.attn_ctas : auto_grid, kMaxAttnCtas);
  // Cluster mode where there is room for a cluster of cs >= 2 CTAs per sequence (at most 8,
  // at least two tiles each by capacity), as many clusters as are resident at once up to
  // the flat grid's size. The kernel gives each sequence cs CTAs of one cluster when the
  // lengths are equal, so that every sequence merges in distributed shared memory instead
  // of through L2 (batch 8: step 52.9 -> 50.9 us, head dim 256 97.2 -> 95.1 us); with
  // unequal lengths it splits the tiles over the whole grid as the flat mode does (a fixed
  // cs CTAs per sequence would leave the longest sequence to set the pace), and only the
  // sequences whose parts fall in one cluster merge on chip.
  pl.cluster = 0;
  pl.flat_grid = pl.grid;
  const bool small = tiles <= 4ll * sms;
  const bool cluster_ok = (clustered == ClusterUse::kAny || (clustered == ClusterUse::kLarge && !small)) &&
                          attn_smem_bytes(s.B, s.G <= 8 ? 1 : 2, 4, s.D, kStageBytes, true) <= kMaxDynSmem;
  if (!fused && cluster_ok && o.attn_ctas == 0 && 2 * seqs <= sms) {
    const long long cs = std::min<long long>({(long long)kMaxAttnCluster, sms / seqs, (tiles_seq + 1) / 2});
    if (cs >= 2) {
      const long long want = std::max<long long>(seqs, (pl.grid + cs - 1) / cs);  // clusters
      const long long n = std::min<long long>(want, max_active_clusters((int)cs));
      if (n >= seqs) {
        pl.cluster = (int)cs;
        pl.grid = (int)(n * cs);
      }
    }
  }
  pl.nb = s.G <= 8 ? 1 : 2;
  pl.gpad = 8 * pl.nb;
  const size_t slots = (size_t)std::max(pl.grid, pl.flat_grid) + (size_t)s.B * s.Hkv;
  pl.slots = (long long)slots;
  pl.part_ml_off = 0;
  pl.part_o_off = align_up(slots * pl.gpad * 2 * 4, 256);
  pl.bytes = pl.part_o_off + align_up(slots * pl.gpad * s.D * 4, 256);
  return pl;
}

struct GemvPlan {
  int bt, kc, ksplit, ncb, nbz;
  size_t bytes;
};

GemvPlan plan_gemv(int B, int K, int N, const Options& o) {
  GemvPlan pl;
  pl.bt = B <= 1 ? 1 : (B <= 2 ? 2 : (B <= 4 ? 4 : 8));
  pl.nbz = (B + pl.bt - 1) / pl.bt;
  pl.ncb = (N + kGemvCols - 1) / kGemvCols;
  const int sms = std::max(1, sm_count());
  int ksplit = (int)o.oproj_splitk;
  if (ksplit <= 0) {
    const double target = 2.0 * sms;
    ksplit = std::max(1, (int)std::lround(target / (double)(pl.ncb * pl.nbz)));
  }
  ksplit = std::min(ksplit, std::max(1, K / 8));
  int kc = (int)align_up((size_t)((K + ksplit - 1) / ksplit), 8);
  kc = std::min(kc, kGemvMaxKc);
  pl.kc = kc;
  pl.ksplit = (K + kc - 1) / kc;
  pl.bytes = pl.ksplit > 1 ? align_up((size_t)pl.ksplit * B * N * 4, 256) : 0;
  return pl;
}

int run_gemv(const __nv_bfloat16* x, long long x_sb, const da_tensor_t* w, const da_tensor_t* out, int B, int K,
             int N, char* ws, char* scratch, const GemvPlan& pl, bool pdl, cudaStream_t stream) {
  if (pl.nbz * pl.ncb > (int)kMaxCounters) return DA_ERR_UNSUPPORTED;
  GemvParams gp;
  gp.x = x;
  gp.x_sb = x_sb;
  gp.w = static_cast<const __nv_bfloat16*>(w->data);
  gp.w_sk = w->stride[0];
  gp.y = static_cast<__nv_bfloat16*>(out->data);
  gp.y_sb = out->stride[0];
  gp.part = reinterpret_cast<float*>(scratch);
  gp.counters = reinterpret_cast<int*>(ws + kGemvCntOff);
  gp.err = reinterpret_cast<int*>(ws + kErrOff);
  gp.B = B;
  gp.K = K;
  gp.N = N;
  gp.kc = pl.kc;
  gp.ksplit = pl.ksplit;
  return launch_gemv(gp, pl.bt, pdl, stream) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

struct UmmaPlan {
  int npad, ksplit;
  bool cluster;
  size_t bytes;
};

UmmaPlan plan_umma(int B, int K, int N, const Options& o) {
  UmmaPlan pl;
  pl.npad = B <= 16 ? 16 : (B <= 32 ? 32 : (B <= 64 ? 64 : 128));
  const int bchunks = (B + pl.npad - 1) / pl.npad;
  const int mtiles = (N + kUmmaBM - 1) / kUmmaBM;
  const int nkb = (K + kUmmaBK - 1) / kUmmaBK;
  const int sms = std::max(1, sm_count());
  int ks = (int)o.oproj_splitk;
  // two CTAs per SM, at most eight slices (a cluster): batch 8 step 53.0 -> 51.0 us against one
  // per SM; the long-context workloads within 1 % either way
  // With K > 4096 (more than 64 k-blocks) at most six (head dim 256, K = 8192, batch 8,
  // interleaved A/B: 8 slices 96.1 us, 6 93.8, 4 94.7, 2 103.4; batch 64 takes 4 from the
  // grid rule above: 604.7 us against 609.4 at 8 and 614.4 at 6).
  if (ks <= 0) {
    ks = std::min(kMaxClusterSplit, std::max(1, 2 * sms / std::max(1, mtiles * bchunks)));
    if (nkb > 64) ks = std::min(ks, 6);
  }
  pl.ksplit = std::max(1, std::min(ks, nkb));
  // up to eight slices reduce in a cluster; more (on request) through global partials
  pl.cluster = pl.ksplit > 1 && pl.ksplit <= kMaxClusterSplit && o.oproj_cluster;
  pl.bytes = pl.ksplit > 1 && !pl.cluster ? align_up((size_t)pl.ksplit * B * N * 4, 256) : 0;
  return pl;
}

int run_umma(const void* x, long long x_sb, const da_tensor_t* w, const da_tensor_t* out, int B, int K, int N,
             char* ws, char* scratch, const UmmaPlan& pl, bool pdl, cudaStream_t stream) {
  const int bchunks = (B + pl.npad - 1) / pl.npad;
  const int mtiles = (N + kUmmaBM - 1) / kUmmaBM;
  if ((int64_t)bchunks * mtiles > (int64_t)kMaxCounters) return DA_ERR_UNSUPPORTED;
  UmmaParams up;
  memset(&up, 0, sizeof(up));
  DA_TRY(encode_2d_map(&up.tm_w, w->data, K, N, w->stride[0], kUmmaBK));
  DA_TRY(encode_2d_map(&up.tm_x, x, B, K, x_sb, pl.npad));
  up.y = static_cast<__nv_bfloat16*>(out->data);
  up.y_sb = out->stride[0];
  up.part = reinterpret_cast<float*>(scratch);
  up.counters = reinterpret_cast<int*>(ws + kGemvCntOff);
  up.err = reinterpret_cast<int*>(ws + kErrOff);
  up.B = B;
  up.K = K;
  up.N = N;
  up.ksplit = pl.ksplit;
  up.prefetch = pdl && options_snapshot().oproj_prefetch ? 1 : 0;
  up.cluster = pl.cluster ? 1 : 0;
  return launch_umma(up, pl.npad, pdl, stream) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// The batch-1 projection with W staged on chip while the attention runs (oproj_onchip.cu):
// one CTA per SM the attention leaves free, a grid of 512-column groups by k-ranges, each
// CTA holding its rectangle of W in shared memory and registers. Feasible when the free SMs
// can hold all of W that way.
struct OnchipPlan {
  bool ok = false;
  int kgroups = 0, smem_kblocks = 0;
  size_t bytes = 0;  // k-range parts
};

OnchipPlan plan_onchip(int B, int K, int N, int free_sms) {
  OnchipPlan pl;
  if (B != 1 || K % 64 || N % kOnchipCols || K <= 0 || N <= 0 || N / kOnchipCols > (int)kMaxCounters) return pl;
  const int kb = K / 64, groups = N / kOnchipCols;
  pl.smem_kblocks = onchip_max_smem_kblocks(K);
  const int per_cta = pl.smem_kblocks + kOnchipRegKblocks;  // k-blocks one CTA can hold
  if (pl.smem_kblocks <= 0 || free_sms < groups) return pl;
  pl.kgroups = std::min(free_sms / groups, kb);
  if ((kb + pl.kgroups - 1) / pl.kgroups > per_cta) return pl;  // the free SMs cannot hold all of W
  pl.bytes = align_up((size_t)groups * pl.kgroups * kOnchipCols * 4, 256);
  pl.ok = true;
  return pl;
}

int run_onchip(const void* x, const da_tensor_t* w, const da_tensor_t* out, int K, int N, char* ws, char* scratch,
               const OnchipPlan& pl, bool pdl, cudaStream_t stream) {
  OnchipParams op;
  memset(&op, 0, sizeof(op));
  DA_TRY(encode_2d_map(&op.tm_w, w->data, K, N, w->stride[0], 64));
  op.x = static_cast<const __nv_bfloat16*>(x);
  op.w = static_cast<const __nv_bfloat16*>(w->data);
  op.w_sk = w->stride[0];
  op.y = static_cast<__nv_bfloat16*>(out->data);
  op.part = reinterpret_cast<float*>(scratch);
  op.counters = reinterpret_cast<int*>(ws + kGemvCntOff);
  op.err = reinterpret_cast<int*>(ws + kErrOff);
  op.K = K;
  op.N = N;
  op.kb = K / 64;
  op.smem_kblocks = pl.smem_kblocks;
  return launch_onchip(op, pl.kgroups, pdl, stream) == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// The projection step: picks the tcgen05 GEMM, the CUDA-core GEMV or (batch 1 behind the
// attention) the on-chip-staged projection by batch size (or the "oproj_path" option) and
// says how much scratch it needs.
struct ProjPlan {
  bool gemm;
  bool onchip = false;
  GemvPlan gv;
  UmmaPlan um;
  OnchipPlan oc;
  size_t bytes;
};

// free_sms: SMs the attention kernel leaves free when the projection follows it (0: none).
ProjPlan plan_projection(int B, int K, int N, const Options& o, int free_sms = 0) {
  ProjPlan pl;
  // On request only (option 3): measured slower than the tcgen05 path at batch 1 (21.8 against
  // 15.6 us per step): the attention slows by ~2 us under W's concurrent stream, the register
  // part of the staging issues at ~36 GB/s per SM, and the CUDA-core arithmetic after the
  // wait takes ~2.4 us.
  if (o.oproj_path == 3) {
    pl.oc = plan_onchip(B, K, N, free_sms);
    if (pl.oc.ok) {
      pl.onchip = true;
      pl.gemm = false;
      pl.bytes = pl.oc.bytes;
      return pl;
    }
  }
  pl.gemm = o.oproj_path == 2 || ((o.oproj_path == 0 || o.oproj_path == 3) && B >= o.gemm_min_batch);  // 3 where infeasible: auto
  if (pl.gemm) {
    pl.um = plan_umma(B, K, N, o);
    pl.bytes = pl.um.bytes;
  } else {
    pl.gv = plan_gemv(B, K, N, o);
    pl.bytes = pl.gv.bytes;
  }
  return pl;
}

int run_projection(const __nv_bfloat16* x, long long x_sb, const da_tensor_t* w, const da_tensor_t* out, int B,
                   int K, int N, char* ws, char* scratch, const ProjPlan& pl, bool pdl, cudaStream_t stream) {
  if (pl.onchip) return run_onchip(x, w, out, K, N, ws, scratch, pl.oc, pdl, stream);
  if (pl.gemm) return run_umma(x, x_sb, w, out, B, K, N, ws, scratch, pl.um, pdl, stream);
  return run_gemv(x, x_sb, w, out, B, K, N, ws, scratch, pl.gv, pdl, stream);
}

// The fused step: attention, grid barrier and tcgen05 projection in one cooperative launch.
struct FusedPlan {
  bool ok = false;
  int npad = 0, kb_per_tile = 0, mtiles = 0, units = 0, attn_workers = 0;
  size_t part_bytes = 0;
};

FusedPlan plan_fused(const AttnShape& s, int K, int N, const AttnPlan& ap, const Options& o) {
  FusedPlan f;
  if (!o.fused || o.oproj_path == 1 || s.B > 128 || K % 64 || s.D != kHeadDim) return f;
  f.npad = s.B <= 16 ? 16 : (s.B <= 32 ? 32 : (s.B <= 64 ? 64 : 128));
  f.kb_per_tile = K / 64;
  f.mtiles = (N + 127) / 128;
  f.units = f.mtiles * f.kb_per_tile;
  const int pb = std::min(ap.grid, f.units);
  // a CTA must cover at most two column tiles (two TMEM accumulator regions)
  if ((f.units + pb - 1) / pb > f.kb_per_tile + 1) return f;
  if (f.mtiles > (int)kMaxCounters) return f;
  f.part_bytes = align_up((size_t)(pb + f.mtiles) * s.B * 128 * 4, 256);
  // Attention workers: about four tiles each (from the cache capacity, an upper bound
  // of the device-side lengths), so that with short sequences the other CTAs start on
  // W_o at once. The attention partial slots are sized for the full grid anyway.
  const long long tiles = (long long)s.B * s.Hkv * ((s.Lcap + kTile - 1) / kTile);  // D = 128 tiles
  f.attn_workers = o.fused_attn_ctas > 0 ? (int)std::min<long long>(o.fused_attn_ctas, ap.grid)
                                         : (int)std::max<long long>(1, std::min<long long>(ap.grid, (tiles + 3) / 4));
  f.ok = true;
  return f;
}

// Scales of an fp8 (e4m3) cache: K = k_cache * k, V = v_cache * v.
struct KvScales {
  float k, v;
};

struct FusedArgs {
  const FusedPlan* plan;
  const da_tensor_t* w;
  const da_tensor_t* out;
  float* part;
  int K, N;
};

// Multiplier and shift that make floor(n / d) = (n * m) >> sh exact for 0 <= n < 2^31 (d >= 1):
// sh = 31 + ceil(log2 d), m = ceil(2^sh / d) < 2^32 + 1, so n * m < 2^64 and n * m / 2^sh
// exceeds n / d by less than n / 2^sh < 1 / d.
void set_split_divisor(AttnParams& p, int k, int d) {
  d = std::max(d, 1);
  int l = 0;
  while ((1ll << l) < d) ++l;
  p.split_div[k] = d;
  p.split_shift[k] = 31 + l;
  p.split_mul[k] = ((1ull << (31 + l)) + (unsigned long long)d - 1) / (unsigned long long)d;
}

int run_attention(const da_tensor_t* q, const da_tensor_t* k, const da_tensor_t* v, const da_tensor_t* lens,
                  const AttnShape& s, const AttnPlan& pl, char* ws, char* scratch, __nv_bfloat16* attn,
                  long long a_sb, long long a_sh, float* scores, long long s_sb, long long s_sh, float scale,
                  cudaStream_t stream, const void* prefetch = nullptr, long long prefetch_bytes = 0,
                  const FusedArgs* fused = nullptr, const PagedShape* paged = nullptr,
                  const KvScales* kv8 = nullptr, int trigger_at = 0) {
  AttnParams p;
  memset(&p, 0, sizeof(p));
  if (fused) {
    DA_TRY(encode_2d_map(&p.tm_w, fused->w->data, fused->K, fused->N, fused->w->stride[0], 64));
    DA_TRY(encode_2d_map(&p.tm_x, attn, s.B, fused->K, a_sb, fused->plan->npad));
    p.y = static_cast<__nv_bfloat16*>(fused->out->data);
    p.y_sb = fused->out->stride[0];
    p.proj_part = fused->part;
    p.proj_part_floats = (long long)(fused->plan->part_bytes / 4);
    p.proj_counters = reinterpret_cast<int*>(ws + kGemvCntOff);
    p.grid_sync = reinterpret_cast<int*>(ws + kGridSyncOff);
    const Options o = options_snapshot();
    p.sync_limit_ns = (unsigned long long)o.grid_wait_us * 1000ull;  // 0: the kernels' default
    p.sync_extra = (int)o.grid_wait_extra;
    p.N = fused->N;
    p.K = fused->K;
    p.kb_per_tile = fused->plan->kb_per_tile;
    p.units = fused->plan->units;
  }

  const int box_tokens = paged ? std::min(paged->block_size, tile_tokens(s.D)) : (kv8 ? kTileFp8 : 0);
  DA_TRY(encode_kv_map(&p.tm_k, k, box_tokens));
  if (v) DA_TRY(encode_kv_map(&p.tm_v, v, box_tokens));
  else p.tm_v = p.tm_k;
  if (paged) {
    p.block_table = paged->table;
    p.bt_stride = paged->table_stride;
    p.bt_entries = paged->table_entries;
    p.block_size = paged->block_size;
    p.num_blocks = paged->num_blocks;
    p.block_shift = 0;
    while ((1 << p.block_shift) < paged->block_size) ++p.block_shift;
    DA_TRY(encode_table_map(&p.tm_table, paged->table, paged->table_entries));
  }
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_sb = q->stride[0];
  p.q_sh = q->stride[1];
  p.seq_lens = static_cast<const int*>(lens->data);
  p.attn = attn;
  p.a_sb = a_sb;
  p.a_sh = a_sh;
  p.scores = scores;
  p.s_sb = s_sb;
  p.s_sh = s_sh;
  p.part_ml = reinterpret_cast<float*>(scratch + pl.part_ml_off);
  p.part_o = reinterpret_cast<float*>(scratch + pl.part_o_off);
  p.part_slots = pl.slots;
  p.counters = reinterpret_cast<int*>(ws + kAttnCntOff);
  p.err = reinterpret_cast<int*>(ws + kErrOff);
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.G = s.G;
  p.Lcap = s.Lcap;
  p.gpad = pl.gpad;
  // scores are scaled in the exp2 domain; an fp8 cache's k_scale folds in there
  p.scale_log2 = scale * (kv8 ? kv8->k : 1.f) * 1.4426950408889634f;
  p.k_scale = kv8 ? kv8->k : 1.f;
  p.v_scale = kv8 ? kv8->v : 1.f;
  p.stages = (int)options_snapshot().attn_stages;
  p.attn_workers = fused ? fused->plan->attn_workers : pl.grid;
  p.prefetch = static_cast<const char*>(prefetch);
  p.prefetch_bytes = prefetch ? (prefetch_bytes & ~15ll) : 0;
  p.cluster = (fused || scores) ? 0 : pl.cluster;
  p.pdl = options_snapshot().attn_pdl ? 1 : 0;
  p.trigger_at = fused ? 0 : trigger_at;
  auto launch = [&](int grid) {
    // the worker counts the kernel divides the tiles by: the flat grid's and cluster mode's
    const int flat = std::min(grid, p.attn_workers);
    set_split_divisor(p, 0, flat);
    set_split_divisor(p, 1, p.cluster > 1 ? (int)std::min<long long>(flat, (long long)s.B * s.Hkv * p.cluster) : flat);
    return kv8     ? launch_attention_fp8(p, grid, pl.nb, stream)
           : paged ? launch_attention_paged(p, grid, pl.nb, s.D, stream)
                   : launch_attention(p, grid, pl.nb, s.D, scores != nullptr, stream, fused ? fused->plan->npad : 0);
  };
  cudaError_t e = launch(pl.grid);
  if (e != cudaSuccess && p.cluster > 1) {  // clusters of this size refused here: the flat grid
    cudaGetLastError();
    p.cluster = 0;
    p.attn_workers = pl.flat_grid;
    e = launch(pl.flat_grid);
  }
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return DA_ERR_UNSUPPORTED;  // the caller falls back to two launches
  }
  return e == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// decode_attn_only / decode_attn_only_paged after their input checks.
int only_checked(const da_tensor_t* q, const da_tensor_t* k, const da_tensor_t* v, const da_tensor_t* seq_lens,
                 const da_tensor_t* attn_out, float scale, void* stream, const AttnShape& s,
                 const PagedShape* paged, const KvScales* kv8 = nullptr) {
  DA_TRY(check_tensor(attn_out, DA_DTYPE_BF16, 3, kOutput));
  if (attn_out->shape[0] != s.B || attn_out->shape[1] != s.Hq || attn_out->shape[2] != s.D)
    return DA_ERR_SHAPE;
  if (!std::isfinite(scale)) return DA_ERR_UNSUPPORTED;
  if (s.B == 0) return DA_OK;
  const Options o = options_snapshot();
  const AttnPlan pl = plan_attention(s, o, kv8 ? kTileFp8 : 0, false, cluster_use_only(o));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = nullptr;
  DA_TRY(workspace_get(pl.bytes, st, &ws));
  return run_attention(q, k, v, seq_lens, s, pl, ws, ws + kHeaderBytes,
                       static_cast<__nv_bfloat16*>(attn_out->data), attn_out->stride[0], attn_out->stride[1],
                       nullptr, 0, 0, scale, st, nullptr, 0, nullptr, paged, kv8);
}

// decode_attn_fwd / decode_attn_fwd_paged after their input checks. The fused step is
// built for a contiguous cache at head dim 128; everything else takes two launches.
int fwd_checked(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                const da_tensor_t* seq_lens, const da_tensor_t* o_weight, const da_tensor_t* out, float scale,
                void* stream, const AttnShape& s, const PagedShape* paged, const KvScales* kv8 = nullptr) {
  DA_TRY(check_tensor(o_weight, DA_DTYPE_BF16, 2, kInput16));
  DA_TRY(check_tensor(out, DA_DTYPE_BF16, 2, kOutput));
  const int64_t K = (int64_t)s.Hq * s.D, N = o_weight->shape[1];
  if (o_weight->shape[0] != K || out->shape[0] != s.B || out->shape[1] != N) return DA_ERR_SHAPE;
  if (N <= 0 || N % 8) return DA_ERR_SHAPE;
  if (N > (1 << 30) || K > (1 << 30)) return DA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return DA_ERR_UNSUPPORTED;
  if (s.B == 0) return DA_OK;
  const Options o = options_snapshot();
  const AttnPlan ap = plan_attention(s, o, kv8 ? kTileFp8 : 0, false, cluster_use_fwd(o));
  const size_t attn_bytes = align_up((size_t)s.B * K * 2, 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const AttnPlan fap = plan_attention(s, o, 0, true);
  const FusedPlan fp = (paged || kv8) ? FusedPlan() : plan_fused(s, (int)K, (int)N, fap, o);
  if (fp.ok) {  // one launch: attention, grid barrier, projection
    char* ws = nullptr;
    DA_TRY(workspace_get(fap.bytes + attn_bytes + fp.part_bytes, st, &ws));
    char* scratch = ws + kHeaderBytes;
    __nv_bfloat16* attn = reinterpret_cast<__nv_bfloat16*>(scratch + fap.bytes);
    const FusedArgs fa{&fp, o_weight, out, reinterpret_cast<float*>(scratch + fap.bytes + attn_bytes), (int)K, (int)N};
    const long long w_span = ((long long)(K - 1) * o_weight->stride[0] + N) * 2;
    const int rc = run_attention(q, k_cache, v_cache, seq_lens, s, fap, ws, scratch, attn, K, s.D, nullptr, 0, 0,
                                 scale, st, o.l2_prefetch ? o_weight->data : nullptr, w_span, &fa);
    if (rc != DA_ERR_UNSUPPORTED) return rc;  // else: not co-resident here, take two launches
  }
  // Batch 1: the on-chip-staged projection takes the SMs the attention leaves free (it runs
  // beside the attention, so it needs the programmatic dependent launch of both kernels).
  const int free_sms = (o.pdl && o.attn_pdl && !ap.cluster) ? std::max(0, sm_count() - ap.grid) : 0;
  const ProjPlan gp = plan_projection(s.B, (int)K, (int)N, o, free_sms);
  char* ws = nullptr;
  DA_TRY(workspace_get(ap.bytes + attn_bytes + gp.bytes, st, &ws));
  char* scratch = ws + kHeaderBytes;
  __nv_bfloat16* attn = reinterpret_cast<__nv_bfloat16*>(scratch + ap.bytes);
  // W_o span: rows 0..K-1 of stride w_sk, the last row N wide
  const long long w_span = ((long long)(K - 1) * o_weight->stride[0] + N) * 2;
  // The on-chip projection stages W while the attention runs: launched right after its set-up.
  DA_TRY(run_attention(q, k_cache, v_cache, seq_lens, s, ap, ws, scratch, attn, K, s.D, nullptr, 0, 0, scale,
                       st, o.l2_prefetch ? o_weight->data : nullptr, w_span, nullptr, paged, kv8,
                       gp.onchip ? 0 : (int)o.attn_trigger));
  return run_projection(attn, K, o_weight, out, s.B, (int)K, (int)N, ws, scratch + ap.bytes + attn_bytes, gp,
                        o.pdl != 0, st);
}

}  // namespace

// ======================================================================= C ABI
extern "C" {

const char* decode_attn_status_str(int code) {
  switch (code) {
    case DA_OK: return "ok";
    case DA_ERR_NULL: return "null pointer or descriptor";
    case DA_ERR_DTYPE: return "wrong dtype";
    case DA_ERR_SHAPE: return "inconsistent or unsupported shape";
    case DA_ERR_STRIDE: return "bad stride (innermost must be 1, others multiples of 8 elements)";
    case DA_ERR_ALIGN: return "misaligned base pointer";
    case DA_ERR_UNSUPPORTED: return "unsupported configuration";
    case DA_ERR_NOMEM: return "workspace allocation failed";
    case DA_ERR_CUDA: return "CUDA error";
    case DA_ERR_OPTION: return "unknown option or bad value";
    case DA_ERR_DEVICE: return "device-side error recorded";
    case DA_ERR_SCRATCH: return "request needs more than the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int decode_attn_set_option(const char* key, int64_t value) {
  if (!key) return DA_ERR_OPTION;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!strcmp(key, "attn_ctas") && value >= 0 && value <= kMaxAttnCtas) g_opt.attn_ctas = value;
  else if (!strcmp(key, "oproj_path") && value >= 0 && value <= 3) g_opt.oproj_path = value;
  else if (!strcmp(key, "oproj_splitk") && value >= 0 && value <= 4096) g_opt.oproj_splitk = value;
  else if (!strcmp(key, "gemm_min_batch") && value >= 1) g_opt.gemm_min_batch = value;
  else if (!strcmp(key, "pdl") && (value == 0 || value == 1)) g_opt.pdl = value;
  else if (!strcmp(key, "l2_prefetch") && (value == 0 || value == 1)) g_opt.l2_prefetch = value;
  else if (!strcmp(key, "attn_stages") && (value == 4 || value == 6)) g_opt.attn_stages = value;
  else if (!strcmp(key, "fused") && (value == 0 || value == 1)) g_opt.fused = value;
  else if (!strcmp(key, "fused_attn_ctas") && value >= 0 && value <= kMaxAttnCtas) g_opt.fused_attn_ctas = value;
  else if (!strcmp(key, "oproj_prefetch") && (value == 0 || value == 1)) g_opt.oproj_prefetch = value;
  else if (!strcmp(key, "oproj_cluster") && (value == 0 || value == 1)) g_opt.oproj_cluster = value;
  else if (!strcmp(key, "attn_cluster") && value >= 0 && value <= 2) g_opt.attn_cluster = value;
  else if (!strcmp(key, "attn_pdl") && (value == 0 || value == 1)) g_opt.attn_pdl = value;
  else if (!strcmp(key, "attn_trigger") && value >= 0 && value <= (1 << 20)) g_opt.attn_trigger = value;
  else if (!strcmp(key, "grid_wait_us") && value >= 0 && value <= 2000000) g_opt.grid_wait_us = value;
  else if (!strcmp(key, "grid_wait_extra") && (value == 0 || value == 1)) g_opt.grid_wait_extra = value;
  else return DA_ERR_OPTION;
  return DA_OK;
}

int decode_attn_get_option(const char* key, int64_t* value) {
  if (!key || !value) return DA_ERR_OPTION;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!strcmp(key, "attn_ctas")) *value = g_opt.attn_ctas;
  else if (!strcmp(key, "oproj_path")) *value = g_opt.oproj_path;
  else if (!strcmp(key, "oproj_splitk")) *value = g_opt.oproj_splitk;
  else if (!strcmp(key, "gemm_min_batch")) *value = g_opt.gemm_min_batch;
  else if (!strcmp(key, "pdl")) *value = g_opt.pdl;
  else if (!strcmp(key, "l2_prefetch")) *value = g_opt.l2_prefetch;
  else if (!strcmp(key, "attn_stages")) *value = g_opt.attn_stages;
  else if (!strcmp(key, "fused")) *value = g_opt.fused;
  else if (!strcmp(key, "fused_attn_ctas")) *value = g_opt.fused_attn_ctas;
  else if (!strcmp(key, "oproj_prefetch")) *value = g_opt.oproj_prefetch;
  else if (!strcmp(key, "oproj_cluster")) *value = g_opt.oproj_cluster;
  else if (!strcmp(key, "attn_cluster")) *value = g_opt.attn_cluster;
  else if (!strcmp(key, "attn_pdl")) *value = g_opt.attn_pdl;
  else if (!strcmp(key, "attn_trigger")) *value = g_opt.attn_trigger;
  else if (!strcmp(key, "grid_wait_us")) *value = g_opt.grid_wait_us;
  else if (!strcmp(key, "grid_wait_extra")) *value = g_opt.grid_wait_extra;
  else return DA_ERR_OPTION;
  return DA_OK;
}

int decode_attn_only(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                     const da_tensor_t* seq_lens, const da_tensor_t* attn_out, float scale, void* stream) {
  AttnShape s;
  DA_TRY(check_attention_inputs(q, k_cache, v_cache, seq_lens, true, &s));
  return only_checked(q, k_cache, v_cache, seq_lens, attn_out, scale, stream, s, nullptr);
}

int decode_attn_only_paged(const da_tensor_t* q, const da_tensor_t* k_pages, const da_tensor_t* v_pages,
                           const da_tensor_t* block_table, const da_tensor_t* seq_lens, const da_tensor_t* attn_out,
                           float scale, void* stream) {
  AttnShape s;
  PagedShape ps;
  DA_TRY(check_paged_inputs(q, k_pages, v_pages, block_table, seq_lens, &s, &ps));
  return only_checked(q, k_pages, v_pages, seq_lens, attn_out, scale, stream, s, &ps);
}

}  // extern "C"

// ----------------------------------------------- attention without allocation
// Scratch of decode_attn_only_noalloc: a fixed device array that every GPU loading
// this library holds until the process exits. Its layout copies the workspace's:
// the error word and completion counters first (the fixed header), then the
// split-KV partials of one call.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
static_assert(kHeaderBytes < kNoAllocScratchBytes, "header must fit the fixed scratch");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name only stands in for it; the runtime gives the real address, looked up
// once per device (the first call on a device does this lookup).
int noalloc_scratch(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return DA_ERR_CUDA;
    }
    g_noalloc_addr[dev] = ptr;
  }
  *out = static_cast<char*>(g_noalloc_addr[dev]);
  return DA_OK;
}
}  // namespace

extern "C" {

int decode_attn_only_noalloc(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                             const da_tensor_t* seq_lens, const da_tensor_t* attn_out, float scale, void* stream) {
  AttnShape s;
  DA_TRY(check_attention_inputs(q, k_cache, v_cache, seq_lens, true, &s));
  DA_TRY(check_tensor(attn_out, DA_DTYPE_BF16, 3, kOutput));
  if (attn_out->shape[0] != s.B || attn_out->shape[1] != s.Hq || attn_out->shape[2] != s.D)
    return DA_ERR_SHAPE;
  if (!std::isfinite(scale)) return DA_ERR_UNSUPPORTED;
  if (s.B == 0) return DA_OK;
  const Options o = options_snapshot();
  const AttnPlan pl = plan_attention(s, o, 0, false, cluster_use_only(o));
  if (kHeaderBytes + pl.bytes > kNoAllocScratchBytes) return DA_ERR_SCRATCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = nullptr;
  DA_TRY(noalloc_scratch(&base));
  // The array keeps whatever the previous call left: the error word and this call's
  // completion counters must start at zero (a memset allocates nothing).
  if (cudaMemsetAsync(base, 0, kAttnCntOff + (size_t)s.B * s.Hkv * 4, st) != cudaSuccess) return DA_ERR_CUDA;
  return run_attention(q, k_cache, v_cache, seq_lens, s, pl, base, base + kHeaderBytes,
                       static_cast<__nv_bfloat16*>(attn_out->data), attn_out->stride[0], attn_out->stride[1],
                       nullptr, 0, 0, scale, st);
}

int decode_attn_scores(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* seq_lens,
                       const da_tensor_t* scores, void* stream) {
  AttnShape s;
  DA_TRY(check_attention_inputs(q, k_cache, nullptr, seq_lens, false, &s));
  DA_TRY(check_tensor(scores, DA_DTYPE_F32, 3, kOutput));
  if (scores->shape[0] != s.B || scores->shape[1] != s.Hq || scores->shape[2] != s.Lcap) return DA_ERR_SHAPE;
  if (s.B == 0) return DA_OK;
  const Options o = options_snapshot();
  const AttnPlan pl = plan_attention(s, o);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = nullptr;
  DA_TRY(workspace_get(pl.bytes, st, &ws));
  return run_attention(q, k_cache, nullptr, seq_lens, s, pl, ws, ws + kHeaderBytes, nullptr, 0, 0,
                       static_cast<float*>(scores->data), scores->stride[0], scores->stride[1], 1.0f, st);
}

int decode_attn_oproj(const da_tensor_t* attn_flat, const da_tensor_t* o_weight, const da_tensor_t* out,
                      void* stream) {
  DA_TRY(check_tensor(attn_flat, DA_DTYPE_BF16, 2, kInput16));
  DA_TRY(check_tensor(o_weight, DA_DTYPE_BF16, 2, kInput16));
  DA_TRY(check_tensor(out, DA_DTYPE_BF16, 2, kOutput));
  const int64_t B = attn_flat->shape[0], K = attn_flat->shape[1], N = o_weight->shape[1];
  if (o_weight->shape[0] != K || out->shape[0] != B || out->shape[1] != N) return DA_ERR_SHAPE;
  if (B == 0) return DA_OK;
  if (K <= 0 || N <= 0 || K % 8 || N % 8) return DA_ERR_SHAPE;
  if (K > (1 << 30) || N > (1 << 30)) return DA_ERR_UNSUPPORTED;
  const Options o = options_snapshot();
  const ProjPlan pl = plan_projection((int)B, (int)K, (int)N, o);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = nullptr;
  DA_TRY(workspace_get(pl.bytes, st, &ws));
  return run_projection(static_cast<const __nv_bfloat16*>(attn_flat->data), B > 1 ? attn_flat->stride[0] : K,
                        o_weight, out, (int)B, (int)K, (int)N, ws, ws + kHeaderBytes, pl, false, st);
}

int decode_attn_fwd(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                    const da_tensor_t* seq_lens, const da_tensor_t* o_weight, const da_tensor_t* out, float scale,
                    void* stream) {
  AttnShape s;
  DA_TRY(check_attention_inputs(q, k_cache, v_cache, seq_lens, true, &s));
  return fwd_checked(q, k_cache, v_cache, seq_lens, o_weight, out, scale, stream, s, nullptr);
}

int decode_attn_fwd_fp8(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                        const da_tensor_t* seq_lens, const da_tensor_t* o_weight, const da_tensor_t* out, float scale,
                        float k_scale, float v_scale, void* stream) {
  AttnShape s;
  DA_TRY(check_attention_inputs(q, k_cache, v_cache, seq_lens, true, &s, DA_DTYPE_E4M3));
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return DA_ERR_UNSUPPORTED;
  const KvScales kv{k_scale, v_scale};
  return fwd_checked(q, k_cache, v_cache, seq_lens, o_weight, out, scale, stream, s, nullptr, &kv);
}

int decode_attn_only_fp8(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                         const da_tensor_t* seq_lens, const da_tensor_t* attn_out, float scale, float k_scale,
                         float v_scale, void* stream) {
  AttnShape s;
  DA_TRY(check_attention_inputs(q, k_cache, v_cache, seq_lens, true, &s, DA_DTYPE_E4M3));
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return DA_ERR_UNSUPPORTED;
  const KvScales kv{k_scale, v_scale};
  return only_checked(q, k_cache, v_cache, seq_lens, attn_out, scale, stream, s, nullptr, &kv);
}

int decode_attn_fwd_paged(const da_tensor_t* q, const da_tensor_t* k_pages, const da_tensor_t* v_pages,
                          const da_tensor_t* block_table, const da_tensor_t* seq_lens, const da_tensor_t* o_weight,
                          const da_tensor_t* out, float scale, void* stream) {
  AttnShape s;
  PagedShape ps;
  DA_TRY(check_paged_inputs(q, k_pages, v_pages, block_table, seq_lens, &s, &ps));
  return fwd_checked(q, k_pages, v_pages, seq_lens, o_weight, out, scale, stream, s, &ps);
}

int decode_attn_last_device_error(void* stream, int32_t* host_code) {
  if (!host_code) return DA_ERR_NULL;
  *host_code = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return DA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    base = g_ws[dev].base;
  }
  char* fixed = nullptr;  // the no-allocation scratch, once a call has looked it up here
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    fixed = static_cast<char*>(g_noalloc_addr[dev]);
  }
  int32_t code = 0;
  for (char* b : {base, fixed}) {
    if (!b) continue;
    int32_t c = 0;
    if (cudaMemcpy(&c, b + kErrOff, sizeof(c), cudaMemcpyDeviceToHost) != cudaSuccess) return DA_ERR_CUDA;
    // A CTA that gave up waiting left its completion counter (and, in the fused step, the
    // grid barrier) short of the count that resets it: clear the whole header, or the next
    // call would see stale counts.
    if (c && cudaMemset(b, 0, kHeaderBytes) != cudaSuccess) return DA_ERR_CUDA;
    code |= c;
  }
  *host_code = code;
  return DA_OK;
}

int decode_attn_device_error(void* stream, int32_t* host_code) {
  return decode_attn_last_device_error(stream, host_code);
}

void decode_attn_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (int d = 0; d < kMaxDevices; ++d) {
    if (!g_ws[d].base) continue;
    if (cudaSetDevice(d) == cudaSuccess) {
      cudaDeviceSynchronize();
      cudaFree(g_ws[d].base);
    }
    g_ws[d].base = nullptr;
    g_ws[d].bytes = 0;
  }
  cudaSetDevice(cur);
}

}  // extern "C"
