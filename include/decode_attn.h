/*
 * decode_attn.h -- C ABI of libdecode_attn.so: one decode step of grouped-query
 * attention over a bf16 KV cache, followed by the output projection, on one
 * NVIDIA GB300 (sm_103a).
 *
 * The computation is the one of the page "PyPTO 开箱性能调优实战 Decode
 * Attention 多 Matmul 独立 TileShape 配置 F-16" (eliteato.com/news/26629),
 * section "代码对比": three contractions with their own result types
 *
 *   scores_fp32 = q_grouped . k_cache^T                 (fp32 scores)
 *   weights     = softmax(scale * scores_fp32)          (the "vector ops")
 *   attn_output = weights . v_cache                     (bf16)
 *   result      = attn_output_flat . o_weight           (bf16)
 *
 * and the shapes of its table "三个 Matmul 的 Shape 特征分析" (QK^T: M = query
 * heads per KV head, K = head_dim = 128, N = kv_len; attn.V: M = heads per KV
 * head, K = kv_len, N = 128; output_proj: M = batch, K = heads * 128,
 * N = hidden). Head dim 256 is the page's other GQA decode (section "仓库源码
 * 佐证": QK^T contracts D = 256 in two halves of 128, attn.V has N = D = 256);
 * every entry point takes D = 128 or D = 256, read from q's last extent.
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is a da_tensor_t descriptor. Its data pointer is a
 *    DEVICE pointer owned by the caller; the library never frees or keeps it.
 *  - Strides are in elements. The innermost dimension must be contiguous
 *    (stride 1); every other stride of an input must be a multiple of 16 bytes
 *    (8 bf16 elements, 16 e4m3 elements) and every base pointer 16-byte aligned
 *    (TMA and 16-byte vector loads need it).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Every call only enqueues work on it and returns; nothing is
 *    synchronised, nothing is copied back to the host.
 *  - All arguments are validated on the host before anything is launched; on
 *    a failure the call returns a negative da_status_t and launches nothing.
 *    A failed launch returns DA_ERR_CUDA.
 *  - The library owns one workspace per device (partial results of the split
 *    KV pass and of the split-K projection, completion counters, the bf16
 *    attention intermediate). When a call needs more, it is grown in stream
 *    order on that call's stream (cudaFreeAsync of the old block, cudaMallocAsync
 *    of the new one, cudaMemsetAsync of its header; no device-wide
 *    synchronisation), so the first call with the largest shapes should precede
 *    any CUDA graph capture. Calls on different streams of the same device share
 *    it: the caller must order them (their work must not overlap on the GPU).
 *  - seq_lens lives on the device. Each length is clamped to [0, Lcap] on the
 *    device; a length of 0 gives an all-zero attention row.
 *  - Bounded device waits: every wait inside a kernel gives up after about
 *    two seconds, records a code that decode_attn_last_device_error() returns,
 *    and the kernel then finishes without waiting further (its output is not
 *    valid).
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of da_tensor_t.dtype. */
enum { DA_DTYPE_BF16 = 1, DA_DTYPE_F32 = 2, DA_DTYPE_I32 = 3, DA_DTYPE_E4M3 = 4 /* fp8 e4m3 (OCP "fn") */ };

/* A strided view of caller-owned device memory (DLPack-like). */
typedef struct da_tensor {
  void* data;        /* device pointer */
  int32_t dtype;     /* DA_DTYPE_* */
  int32_t ndim;      /* number of valid entries in shape/stride, 1..4 */
  int64_t shape[4];
  int64_t stride[4]; /* in elements */
} da_tensor_t;

typedef enum {
  DA_OK = 0,
  DA_ERR_NULL = -1,        /* a required pointer or descriptor is NULL */
  DA_ERR_DTYPE = -2,       /* wrong element type */
  DA_ERR_SHAPE = -3,       /* inconsistent or unsupported shape */
  DA_ERR_STRIDE = -4,      /* innermost dim not contiguous, or a stride not a multiple of 8 */
  DA_ERR_ALIGN = -5,       /* base pointer not 16-byte aligned */
  DA_ERR_UNSUPPORTED = -6, /* valid request outside what the kernels implement */
  DA_ERR_NOMEM = -7,       /* the workspace could not be grown */
  DA_ERR_CUDA = -8,        /* a CUDA runtime call or launch failed */
  DA_ERR_OPTION = -9,      /* unknown option key or value out of range */
  DA_ERR_DEVICE = -10,     /* a kernel recorded a device-side error (bounded wait ran out) */
  DA_ERR_SCRATCH = -11     /* decode_attn_only_noalloc: the call needs more than its fixed scratch */
} da_status_t;

/* Limits checked on the host. */
#define DA_HEAD_DIM 128      /* D: the default head dim */
#define DA_HEAD_DIM_WIDE 256 /* D: the other head dim the kernels implement */
#define DA_MAX_GROUP 16  /* G = Hq / Hkv */
#define DA_MAX_BATCH 1024

/*
 * decode_attn_fwd -- the whole step: attention, then the output projection.
 * Page: "PyPTO 开箱性能调优实战 Decode Attention 多 Matmul 独立 TileShape 配置
 * F-16", section "代码对比" (the three matmuls) and the shape table.
 *
 *   q        [B, Hq, D]          bf16  the new token's queries, D = 128 or 256
 *   k_cache  [B, Hkv, Lcap, D]   bf16  keys; token t of sequence b is row t
 *   v_cache  [B, Hkv, Lcap, D]   bf16  values, same shape as k_cache
 *   seq_lens [B]                 int32 valid tokens per sequence (device)
 *   o_weight [Hq*D, N]           bf16  row-major; row k = h*D + d
 *   out      [B, N]              bf16  written
 *   scale    softmax scale applied to the fp32 scores (usually 1/sqrt(D))
 *
 * Query head h attends with KV head h / (Hq / Hkv) over tokens t < seq_lens[b].
 * Requires Hq % Hkv == 0, Hq / Hkv <= 16, B <= 1024, N % 8 == 0; any other D
 * returns DA_ERR_SHAPE.
 * Returns DA_OK or a negative da_status_t.
 */
int decode_attn_fwd(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                    const da_tensor_t* seq_lens, const da_tensor_t* o_weight, const da_tensor_t* out,
                    float scale, void* stream);

/*
 * decode_attn_only -- the attention half: attn_out[b, h, :] =
 * softmax(scale * q[b,h] . K[b, h/G]^T) . V[b, h/G] over t < seq_lens[b],
 * written as bf16 (the page's `attn_output`, DT_BF16).
 *   attn_out [B, Hq, D] bf16, caller-allocated, any strides obeying the
 *   conventions. Other arguments as decode_attn_fwd.
 */
int decode_attn_only(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                     const da_tensor_t* seq_lens, const da_tensor_t* attn_out, float scale,
                     void* stream);

/*
 * decode_attn_only_noalloc -- decode_attn_only for callers that must not allocate
 * device memory at run time: for example a serving process whose GPU memory is
 * reserved up front by its own allocator or memory pool (an allocation outside
 * it can fail, or take memory the pool was sized to own), or a request path with
 * a latency bound, where growing the library workspace (a stream-ordered pool
 * allocation that may have to map new device memory) is not allowed. The pages
 * have no counterpart; this is a deployment convenience, with the same arguments
 * and the same result as decode_attn_only.
 *
 * Scratch: a fixed 8 MiB device array inside the library, held by every GPU that
 * loads it until the process exits. It is never allocated or freed and no
 * allocating routine is called. The split-KV partials need one slot per
 * (sequence, KV head) pair plus one per persistent CTA: on a 152-SM GB300 with
 * the default grid that allows B*Hkv up to 1738 when Hq/Hkv <= 8 and up to 793
 * when Hq/Hkv <= 16 at D = 128; at D = 256 up to 800 and 324. A larger call
 * returns DA_ERR_SCRATCH and launches nothing.
 *
 * - The first call on a device looks up the array's device address (no
 *   allocation); make that first call before any stream capture.
 * - Every call clears the error word and its completion counters with
 *   cudaMemsetAsync on `stream` before the kernel, because the array keeps the
 *   previous call's contents.
 * - All calls share the one array: calls whose work overlaps on the GPU (other
 *   streams, other host threads) race on it and must be serialised by the caller.
 * - Device-side wait timeouts are recorded in the array's own error word, which
 *   decode_attn_last_device_error() reads and clears together with the
 *   workspace's (until the next call of this entry point clears it).
 */
int decode_attn_only_noalloc(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                             const da_tensor_t* seq_lens, const da_tensor_t* attn_out, float scale,
                             void* stream);

/*
 * decode_attn_fwd_paged / decode_attn_only_paged -- decode_attn_fwd / decode_attn_only
 * over a paged KV cache: the keys and values live in a pool of fixed-size blocks and
 * a per-sequence block table lists the blocks of each sequence in token order. The
 * pages have no paged cache; the computation is exactly that of the contiguous entry
 * points on the cache the table describes,
 *
 *   K[b, j, t, :] = k_pages[block_table[b, t / block_size], j, t % block_size, :]
 *
 * for t < seq_lens[b] (and the same for V).
 *   k_pages     [num_blocks, Hkv, block_size, D] bf16  the key pool (device). Any strides
 *               obeying the conventions, so a pool stored as [num_blocks, block_size,
 *               Hkv, D] is passed as the view with dims 1 and 2 swapped.
 *   v_pages     same shape as k_pages (its own strides)
 *   block_table [B, max_blocks] int32 (device), rows contiguous, base 16-byte aligned
 *               (it is read by TMA): entry i of row b is the pool block holding tokens
 *               [i * block_size, (i + 1) * block_size) of sequence b. Only the first
 *               ceil(seq_lens[b] / block_size) entries of a row are used (a few entries
 *               past them may be fetched, never past the table's last entry).
 *   seq_lens    [B] int32 (device), clamped to [0, max_blocks * block_size]
 *   q, o_weight, out, attn_out, scale: as decode_attn_fwd / decode_attn_only.
 * block_size: a power of two from 8 to 2^20; anything else returns DA_ERR_UNSUPPORTED.
 * (Blocks of 32 tokens and more stream at 90-95% of the contiguous rate on GB300; 16
 * at about 75%, 8 at about 55%.) A table entry outside [0, num_blocks) that
 * is read sets bit 64 of the device error word (decode_attn_last_device_error) and that
 * block reads as zeros. The fused option does not apply: two launches.
 */
int decode_attn_fwd_paged(const da_tensor_t* q, const da_tensor_t* k_pages, const da_tensor_t* v_pages,
                          const da_tensor_t* block_table, const da_tensor_t* seq_lens, const da_tensor_t* o_weight,
                          const da_tensor_t* out, float scale, void* stream);
int decode_attn_only_paged(const da_tensor_t* q, const da_tensor_t* k_pages, const da_tensor_t* v_pages,
                           const da_tensor_t* block_table, const da_tensor_t* seq_lens, const da_tensor_t* attn_out,
                           float scale, void* stream);

/*
 * decode_attn_fwd_fp8 / decode_attn_only_fp8 -- decode_attn_fwd / decode_attn_only over
 * an fp8 KV cache: k_cache and v_cache hold e4m3 codes (DA_DTYPE_E4M3, the OCP "fn"
 * format: 4 exponent bits with bias 7, 3 mantissa bits, no infinities), and the keys and
 * values are
 *
 *   K = k_cache * k_scale,   V = v_cache * v_scale       (one float scale per cache)
 *
 * The pages have no fp8 cache; the computation is exactly that of the bf16 entry points
 * on these K and V. The cache bytes halve; q, o_weight and the outputs stay bf16.
 *   k_cache, v_cache [B, Hkv, Lcap, 128] e4m3; strides multiples of 16 elements (bytes)
 *   k_scale, v_scale finite floats (DA_ERR_UNSUPPORTED otherwise)
 *   other arguments as decode_attn_fwd / decode_attn_only
 * Head dim 128 only (D = 256 returns DA_ERR_UNSUPPORTED); the fused option does not apply.
 * The kernels widen the codes to f16 (exact) and multiply them with q rounded to f16,
 * which is exact for |q| <= 65504; larger |q| is clamped to 65504. The softmax weights
 * enter P.V as f16 (bf16 on the bf16 path).
 */
int decode_attn_fwd_fp8(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                        const da_tensor_t* seq_lens, const da_tensor_t* o_weight, const da_tensor_t* out, float scale,
                        float k_scale, float v_scale, void* stream);
int decode_attn_only_fp8(const da_tensor_t* q, const da_tensor_t* k_cache, const da_tensor_t* v_cache,
                         const da_tensor_t* seq_lens, const da_tensor_t* attn_out, float scale, float k_scale,
                         float v_scale, void* stream);

/*
 * decode_attn_scores -- the first contraction alone: the page's `scores_fp32`
 * (q_grouped . k_cache^T, b_trans=True), unscaled, in fp32.
 *   scores [B, Hq, Lcap] fp32: scores[b, h, t] is written for t < seq_lens[b]
 *   only; entries at t >= seq_lens[b] are left as they were.
 * A checking and tuning hook; it runs the attention kernel's QK^T code.
 */
int decode_attn_scores(const da_tensor_t* q, const da_tensor_t* k_cache,
                       const da_tensor_t* seq_lens, const da_tensor_t* scores, void* stream);

/*
 * decode_attn_oproj -- the last contraction alone: out = attn_flat . o_weight
 * (the page's output_proj: M = batch, K = Hq*128, N = hidden), bf16 operands,
 * fp32 accumulation, bf16 result.
 *   attn_flat [B, K] bf16;  o_weight [K, N] bf16 row-major;  out [B, N] bf16.
 * Requires N % 8 == 0 and K % 8 == 0.
 */
int decode_attn_oproj(const da_tensor_t* attn_flat, const da_tensor_t* o_weight,
                      const da_tensor_t* out, void* stream);

/*
 * Tuning options (process-wide; 0 = automatic). Keys:
 *   "attn_ctas"     CTAs of the persistent attention kernel (0: one per SM, fewer for
 *                   small problems: about four tiles each by the cache capacity;
 *                   at most 512)
 *   "oproj_path"    0 auto, 1 CUDA-core GEMV, 2 tcgen05 tensor-core GEMM, 3 (decode_attn_fwd
 *                   at batch 1) o_weight staged in the shared memory and registers of the
 *                   SMs the attention leaves free while the attention runs, then a CUDA-core
 *                   product (correct, measured slower on GB300; auto where it does not fit)
 *   "oproj_splitk"  split-K factor of the projection (0: auto, two CTAs per SM, at
 *                   most 8, at most 6 when K > 4096)
 *   "attn_cluster"  1 (default): where there is room for two or more CTAs per
 *                   (batch, KV head) sequence, the attention kernel is launched in
 *                   thread-block clusters of up to 8 CTAs (decode_attn_fwd: only
 *                   above about four tiles per SM). When every sequence has the same
 *                   length, each gets the CTAs of one cluster and their partial
 *                   states merge in distributed shared memory; otherwise the tiles
 *                   are split evenly over the whole grid as in the flat mode, and
 *                   only the sequences whose parts fall in one cluster merge on
 *                   chip (the rest through L2). 2: as 1, and decode_attn_fwd
 *                   takes clusters at every size too. 0: always the flat grid.
 *                   Results agree within the rounding of the merge order.
 *   "oproj_cluster" 1 (default): the split-K slices of a tcgen05 column tile form a
 *                   thread-block cluster and reduce in distributed shared memory
 *                   (split-K <= 8); 0: through global partials and an atomic counter
 *   "gemm_min_batch" smallest batch that takes the tensor-core GEMM in auto mode
 *                   (default 1: every batch; the GEMV measured slower on GB300)
 *   "pdl"           1 (default): launch the projection with programmatic
 *                   dependent launch so it overlaps the attention kernel's tail
 *   "attn_pdl"      1 (default): launch the attention kernel with programmatic
 *                   dependent launch too; it waits for the previous kernel in the
 *                   stream to complete before its first global-memory access (every
 *                   input is read after that), so only its start-up overlaps
 *   "attn_trigger"  3 (default): in decode_attn_fwd each attention CTA lets the
 *                   projection kernel launch when it reaches the tile this many
 *                   before the end of its range, so that the projection's early
 *                   o_weight loads overlap the attention's last tiles and merges
 *                   rather than queue in front of its K/V stream; 0: right after
 *                   the attention's set-up. Timing only: results are identical.
 *   "l2_prefetch"   0 (default) or 1: in decode_attn_fwd the attention kernel
 *                   pulls o_weight into L2 while it streams K/V, so that the
 *                   projection reads o_weight from L2 (measured slower on GB300:
 *                   the prefetch competes with the K/V stream)
 *   "attn_stages"   4 (default) or 6: depth of the attention kernel's K/V ring
 *                   (6 only at D = 128, bf16 or fp8 cache, and when it fits in shared
 *                   memory for the batch)
 *   "fused"         0 (default): decode_attn_fwd runs two launches (attention,
 *                   projection); 1: one persistent cooperative launch (attention,
 *                   a bounded grid barrier, tcgen05 projection) when batch <= 128
 *                   (correct, but measured slower on GB300 so far); head dim 128
 *                   only: at D = 256 decode_attn_fwd always takes two launches
 *   "fused_attn_ctas" attention workers of the fused step (0: about four 64-token
 *                   tiles each, at most one per SM; the other CTAs start on o_weight)
 *   "oproj_prefetch" 0 (default) or 1: in decode_attn_fwd each tcgen05 projection CTA
 *                   pulls the part of its o_weight slice that its ring does not hold
 *                   into L2 before it waits for the attention kernel (measured no
 *                   faster on GB300)
 *   "grid_wait_us"  test hook: the fused step's grid-barrier wait limit in microseconds
 *                   (0, the default: two seconds; at most 2000000)
 *   "grid_wait_extra" test hook, 0 (default) or 1: the fused step's grid barrier waits
 *                   for this many arrivals beyond the grid, so that with 1 the wait runs
 *                   out, records error bit 32 and the kernel completes with an invalid
 *                   result (a failure that touches no bad address and hangs nothing)
 * Returns DA_OK or DA_ERR_OPTION.
 */
int decode_attn_set_option(const char* key, int64_t value);
int decode_attn_get_option(const char* key, int64_t* value);

/*
 * decode_attn_last_device_error -- synchronises `stream`, then reports in
 * *host_code the device error word of the current device (the bitwise OR of the
 * workspace's word and the no-allocation scratch's word): 0 when no kernel
 * recorded an error. Codes (bits): 1 a consumer gave up waiting for a K/V stage,
 * 2 a producer gave up waiting for a free stage, 4 copies still in flight at
 * exit, 8 a tensor-core completion never arrived, 32 the fused step's grid
 * barrier did not complete, 64 a paged cache's block table named a block outside
 * the pool. A non-zero word is cleared, and with it the completion counters and
 * grid-barrier words beside it (a CTA that gave up left them short of the count
 * that resets them), so that the next call starts clean. Returns DA_OK, or
 * DA_ERR_CUDA when the synchronisation or a copy failed.
 */
int decode_attn_last_device_error(void* stream, int32_t* host_code);
/* The same call under its earlier name. */
int decode_attn_device_error(void* stream, int32_t* host_code);

/* Frees the workspace of every device (synchronises those devices). */
void decode_attn_release(void);

/* A static, human-readable name for a da_status_t. */
const char* decode_attn_status_str(int code);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
