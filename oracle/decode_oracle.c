/*
 * decode_oracle.c -- fp64 CPU oracle for one decode step: grouped-query
 * attention over a bf16 KV cache followed by the output projection.
 *
 * TEST INFRASTRUCTURE ONLY. The library (its CUDA kernels, its C-ABI and the
 * Python binding) never links, loads or calls this file; only the tests, the
 * smoke check and the benchmark's CPU-baseline leg do. It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes follows the page "PyPTO 开箱性能调优实战 Decode Attention 多
 * Matmul 独立 TileShape 配置 F-16" (eliteato.com/news/26629): section "代码对比"
 * gives the three contractions and their result types, section "三个 Matmul 的
 * Shape 特征分析" their shapes (QK^T M=4 K=128 N=2048, attn*V M=4 K=2048 N=128,
 * output_proj M=1 K=4096 N=4096):
 *
 *   scores = q_grouped . k_cache^T            fp32 on the page, here fp64
 *   (vector ops: scale, then softmax over the valid keys)
 *   attn   = attn_weights . v_cache           bf16 on the page, here fp64
 *   out    = attn_output_flat . o_weight      bf16 on the page, here fp64
 *
 * Every function is the plain definition written out in double precision from
 * the same bf16 bit patterns the GPU receives (bf16 -> double is exact). There
 * is no online softmax, no blocking and no intermediate rounding; the one
 * exception is oracle_group_attention_split, which states the split-KV
 * log-sum-exp combine on purpose so that it can be checked against the
 * unsplit definition.
 *
 * Readings taken where the page is silent:
 *  - the "vector ops" are: multiply the fp32 scores by `scale`, subtract the
 *    row maximum, exponentiate, divide by the row sum (softmax over t < L);
 *    no mask, bias or soft-cap beyond the sequence length;
 *  - query head h reads KV head h / G (the page's q_grouped: G consecutive
 *    query heads share one KV head);
 *  - o_weight is [Hq*D, hidden] row-major (the page's matmul has no b_trans),
 *    and the flattened attention index is k = h*D + d;
 *  - a sequence of length 0 attends to nothing and its output row is 0.
 *
 * Layouts (elements, all contiguous):
 *   q [B][Hq][D], k_cache and v_cache [B][Hkv][Lcap][D], seq_lens [B],
 *   o_weight [Hq*D][N], attn [B][Hq][D], out [B][N].
 *
 * Build: gcc -O2 -fno-fast-math -fopenmp -shared -fPIC (see oracle/__init__.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Scores of one (batch, KV-head) group: s[g][t] = sum_d q[g][d] * k[t][d].
 * This is QK^T of the page's shape table with M = G, K = D, N = L; the keys are
 * rows of the cache (the page's b_trans=True). Unscaled.
 * q row g starts at q + g*q_row_stride; key t at k + t*k_row_stride.
 */
void oracle_group_scores(const uint16_t* q, int64_t q_row_stride, const uint16_t* k,
                         int64_t k_row_stride, int64_t G, int64_t L, int64_t D,
                         double* s /* [G][L] */) {
  for (int64_t g = 0; g < G; ++g) {
    for (int64_t t = 0; t < L; ++t) {
      double acc = 0.0;
      for (int64_t d = 0; d < D; ++d) {
        acc += bf16_bits_to_double(q[g * q_row_stride + d]) *
               bf16_bits_to_double(k[t * k_row_stride + d]);
      }
      s[g * L + t] = acc;
    }
  }
}

/*
 * One group of G query heads attending to the same L keys and values:
 *   z[t] = scale * s[t];  p[t] = exp(z[t] - max z) / sum_t' exp(z[t'] - max z)
 *   out[g][d] = sum_t p[t] * v[t][d]
 * (attn * V of the shape table: M = G, K = L, N = D). L == 0 gives zeros.
 */
int oracle_group_attention(const uint16_t* q, int64_t q_row_stride, const uint16_t* k,
                           int64_t k_row_stride, const uint16_t* v, int64_t v_row_stride,
                           int64_t G, int64_t L, int64_t D, double scale,
                           double* out /* [G][D] */) {
  if (L == 0) {
    memset(out, 0, (size_t)(G * D) * sizeof(double));
    return 0;
  }
  double* s = (double*)malloc((size_t)(G * L) * sizeof(double));
  if (!s) return -1;
  oracle_group_scores(q, q_row_stride, k, k_row_stride, G, L, D, s);
  for (int64_t g = 0; g < G; ++g) {
    double* z = s + g * L;
    double zmax = -INFINITY;
    for (int64_t t = 0; t < L; ++t) {
      z[t] = scale * z[t];
      if (z[t] > zmax) zmax = z[t];
    }
    double zsum = 0.0;
    for (int64_t t = 0; t < L; ++t) {
      z[t] = exp(z[t] - zmax);
      zsum += z[t];
    }
    for (int64_t t = 0; t < L; ++t) z[t] = z[t] / zsum; /* z now holds p */
    for (int64_t d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int64_t t = 0; t < L; ++t) acc += z[t] * bf16_bits_to_double(v[t * v_row_stride + d]);
      out[g * D + d] = acc;
    }
  }
  free(s);
  return 0;
}

/*
 * The same result computed split-KV: the L keys are cut into chunks of
 * `chunk` tokens; chunk c keeps its own maximum m_c, its own sum
 * l_c = sum exp(z - m_c) and its own unnormalised output O_c = sum exp(z - m_c) v;
 * the chunks are then merged with M = max_c m_c:
 *   out = sum_c exp(m_c - M) O_c / sum_c exp(m_c - M) l_c.
 * Exactly equal to oracle_group_attention up to rounding, because
 * exp(z - M) = exp(z - m_c) * exp(m_c - M).
 */
int oracle_group_attention_split(const uint16_t* q, int64_t q_row_stride, const uint16_t* k,
                                 int64_t k_row_stride, const uint16_t* v, int64_t v_row_stride,
                                 int64_t G, int64_t L, int64_t D, double scale, int64_t chunk,
                                 double* out /* [G][D] */) {
  if (chunk <= 0) return -1;
  if (L == 0) {
    memset(out, 0, (size_t)(G * D) * sizeof(double));
    return 0;
  }
  int64_t n_chunks = (L + chunk - 1) / chunk;
  double* s = (double*)malloc((size_t)(G * L) * sizeof(double));
  double* m_c = (double*)malloc((size_t)n_chunks * sizeof(double));
  double* l_c = (double*)malloc((size_t)n_chunks * sizeof(double));
  double* o_c = (double*)malloc((size_t)(n_chunks * D) * sizeof(double));
  if (!s || !m_c || !l_c || !o_c) {
    free(s); free(m_c); free(l_c); free(o_c);
    return -1;
  }
  oracle_group_scores(q, q_row_stride, k, k_row_stride, G, L, D, s);
  for (int64_t g = 0; g < G; ++g) {
    const double* sg = s + g * L;
    for (int64_t c = 0; c < n_chunks; ++c) {
      int64_t t0 = c * chunk, t1 = t0 + chunk < L ? t0 + chunk : L;
      double m = -INFINITY;
      for (int64_t t = t0; t < t1; ++t)
        if (scale * sg[t] > m) m = scale * sg[t];
      double l = 0.0;
      for (int64_t d = 0; d < D; ++d) o_c[c * D + d] = 0.0;
      for (int64_t t = t0; t < t1; ++t) {
        double e = exp(scale * sg[t] - m);
        l += e;
        for (int64_t d = 0; d < D; ++d) o_c[c * D + d] += e * bf16_bits_to_double(v[t * v_row_stride + d]);
      }
      m_c[c] = m;
      l_c[c] = l;
    }
    double big_m = -INFINITY;
    for (int64_t c = 0; c < n_chunks; ++c)
      if (m_c[c] > big_m) big_m = m_c[c];
    double denom = 0.0;
    for (int64_t c = 0; c < n_chunks; ++c) denom += exp(m_c[c] - big_m) * l_c[c];
    for (int64_t d = 0; d < D; ++d) {
      double num = 0.0;
      for (int64_t c = 0; c < n_chunks; ++c) num += exp(m_c[c] - big_m) * o_c[c * D + d];
      out[g * D + d] = num / denom;
    }
  }
  free(s); free(m_c); free(l_c); free(o_c);
  return 0;
}

/*
 * Output projection (output_proj of the shape table: M = B, K = Kdim, N):
 *   y[b][n] = sum_k x[b][k] * w[k][n],   w row-major [Kdim][N].
 * x is fp64 (the oracle's own attention output, never rounded).
 */
void oracle_oproj(const double* x /* [B][Kdim] */, const uint16_t* w /* [Kdim][N] */, int64_t B,
                  int64_t Kdim, int64_t N, double* y /* [B][N] */) {
  for (int64_t b = 0; b < B; ++b) {
    double* yb = y + b * N;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) yb[n] = 0.0;
    /* accumulate row by row so that w is read along its contiguous axis */
#pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < (N + 255) / 256; ++nb) {
      int64_t n0 = nb * 256, n1 = n0 + 256 < N ? n0 + 256 : N;
      for (int64_t kk = 0; kk < Kdim; ++kk) {
        double xk = x[b * Kdim + kk];
        const uint16_t* wk = w + kk * N;
        for (int64_t n = n0; n < n1; ++n) yb[n] += xk * bf16_bits_to_double(wk[n]);
      }
    }
  }
}

/*
 * Unscaled scores for the whole batch: scores[b][h][t] for t < seq_lens[b];
 * entries t >= seq_lens[b] are left untouched. Returns -1 on bad arguments
 * (Hq not a multiple of Hkv, or a length outside [0, Lcap]).
 */
int oracle_scores(const uint16_t* q, const uint16_t* k, const int32_t* seq_lens, int64_t B,
                  int64_t Hq, int64_t Hkv, int64_t Lcap, int64_t D, double* scores) {
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] > Lcap) return -1;
  int64_t G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic)
  for (int64_t bh = 0; bh < B * Hq; ++bh) {
    int64_t b = bh / Hq, h = bh % Hq, j = h / G;
    int64_t L = seq_lens[b];
    double* tmp = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    if (!tmp) {
      err = -1;
      continue;
    }
    oracle_group_scores(q + (b * Hq + h) * D, D, k + (b * Hkv + j) * Lcap * D, D, 1, L, D, tmp);
    memcpy(scores + (b * Hq + h) * Lcap, tmp, (size_t)L * sizeof(double));
    free(tmp);
  }
  return err;
}

/*
 * Attention for the whole batch: attn[b][h][:] over t < seq_lens[b] with
 * KV head h / G. Returns -1 on bad arguments.
 */
int oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const int32_t* seq_lens, int64_t B, int64_t Hq, int64_t Hkv, int64_t Lcap,
                     int64_t D, double scale, double* attn /* [B][Hq][D] */) {
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] > Lcap) return -1;
  int64_t G = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic)
  for (int64_t bh = 0; bh < B * Hq; ++bh) {
    int64_t b = bh / Hq, h = bh % Hq, j = h / G;
    const uint16_t* kb = k + (b * Hkv + j) * Lcap * D;
    const uint16_t* vb = v + (b * Hkv + j) * Lcap * D;
    if (oracle_group_attention(q + (b * Hq + h) * D, D, kb, D, vb, D, 1, seq_lens[b], D, scale,
                               attn + (b * Hq + h) * D) != 0)
      err = -1;
  }
  return err;
}

/*
 * The whole decode step: attention, then out = attn_flat . o_weight with
 * attn_flat[b][h*D + d] = attn[b][h][d]. `out` may be NULL (attention only).
 */
int oracle_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* seq_lens,
                  const uint16_t* w, int64_t B, int64_t Hq, int64_t Hkv, int64_t Lcap, int64_t D,
                  int64_t N, double scale, double* attn /* [B][Hq][D] */,
                  double* out /* [B][N] or NULL */) {
  int rc = oracle_attention(q, k, v, seq_lens, B, Hq, Hkv, Lcap, D, scale, attn);
  if (rc != 0) return rc;
  if (out) oracle_oproj(attn, w, B, Hq * D, N, out);
  return 0;
}

/*
 * oracle_gather_pages -- the contiguous cache that a paged cache describes, for the
 * library's block-table entry points (the pages describe no paged cache; this is the
 * plain reading of a block table): for t < seq_lens[b] and every KV head j,
 *
 *   cache[b][j][t][:] = pages[table[b][t / bs]][j][t % bs][:]
 *
 * A table entry outside [0, num_blocks) gives a zero row (the library flags it and
 * reads zeros), and rows t >= seq_lens[b] are zero. Only bit patterns are copied.
 *   pages [num_blocks][Hkv][bs][D], table [B][max_blocks], cache [B][Hkv][max_blocks*bs][D]
 * Returns 0, or -1 when a length lies outside [0, max_blocks * bs].
 */
int oracle_gather_pages(const uint16_t* pages, int64_t num_blocks, int64_t Hkv, int64_t bs, int64_t D,
                        const int32_t* table, int64_t B, int64_t max_blocks, const int32_t* seq_lens,
                        uint16_t* cache) {
  const int64_t Lcap = max_blocks * bs;
  for (int64_t b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || seq_lens[b] > Lcap) return -1;
  memset(cache, 0, (size_t)(B * Hkv * Lcap * D) * sizeof(uint16_t));
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t t = 0; t < seq_lens[b]; ++t) {
      const int64_t blk = table[b * max_blocks + t / bs];
      if (blk < 0 || blk >= num_blocks) continue;
      const int64_t row = t % bs;
      for (int64_t j = 0; j < Hkv; ++j) {
        const uint16_t* src = pages + ((blk * Hkv + j) * bs + row) * D;
        uint16_t* dst = cache + ((b * Hkv + j) * Lcap + t) * D;
        memcpy(dst, src, (size_t)D * sizeof(uint16_t));
      }
    }
  }
  return 0;
}

/*
 * oracle_e4m3_to_bf16 -- widens fp8 e4m3 codes (the OCP 8-bit format E4M3 "fn": 1 sign
 * bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN)
 * to the bf16 bit patterns of the same values, for the library's fp8-cache entry points
 * (the pages describe no fp8 cache). Every e4m3 value is a bf16 value, so this is exact:
 *   exponent field 0:      (-1)^s * m * 2^-9            (subnormals and zeros)
 *   exponent field e > 0:  (-1)^s * (1 + m / 8) * 2^(e - 7)
 * NaN codes give the bf16 quiet NaN 0x7fc0 (with the sign). Returns the number of NaN codes.
 */
int64_t oracle_e4m3_to_bf16(const uint8_t* in, int64_t n, uint16_t* out) {
  int64_t nans = 0;
  for (int64_t i = 0; i < n; ++i) {
    const unsigned b = in[i];
    const unsigned s = b >> 7, e = (b >> 3) & 15u, m = b & 7u;
    if (e == 15u && m == 7u) {
      out[i] = (uint16_t)((s << 15) | 0x7fc0u);
      ++nans;
      continue;
    }
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    const float f = (float)(s ? -mag : mag);  /* exact: at most 4 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof(u));
    out[i] = (uint16_t)(u >> 16);  /* exact: the low 16 bits of u are zero */
  }
  return nans;
}
