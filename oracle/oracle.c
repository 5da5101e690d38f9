/*
 * oracle.c -- plain, slow, fp64 CPU statement of what the batch-invariant
 * reduction kernels compute.  TEST INFRASTRUCTURE ONLY: it is linked by the
 * tests, by the smoke check and by the benchmark's CPU-baseline leg, never by
 * the product path.  It shares no code, header or constant with the CUDA
 * library; the two meet only through the seeded inputs the tests hand to both.
 *
 * Sources (three web pages on batch-invariant LLM inference):
 *   [P1] "Reproducible LLM Inference - Batch Invariance, the Cost of
 *        Determinism, and Where Bitwise Identity Is Actually Required"
 *        (hidekazu-konishi.com)
 *   [P3] "Your Answer Depends on Who Else Is in the Batch" (praveentn.live)
 *
 * The method does not change WHAT is computed, only the order of the
 * additions.  So every function here is the plain mathematical definition,
 * evaluated in double precision from bf16 inputs that are widened exactly:
 * no blocking, no splitting, no fusion -- except oracle_attention_splits and
 * the two split planners, which state the split structure itself (P1 §5.5)
 * so that tests can show it is an exact rearrangement of the plain softmax.
 *
 * Every bf16 value is passed as its raw 16-bit pattern (uint16_t).
 * Threads: each function splits independent output rows over nthreads POSIX
 * threads (nthreads <= 0: one per online core).  Rows never interact, so the
 * results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 -> double: a bf16 is the top half of an IEEE binary32, so the
 * widening is exact. */
static double bf16_val(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------ */
/* tiny row-parallel runner                                            */
/* ------------------------------------------------------------------ */
typedef void (*row_fn)(void* ctx, int64_t r);
typedef struct {
  row_fn fn;
  void* ctx;
  int64_t begin, end;
} row_job;

static void* run_rows(void* p) {
  row_job* j = (row_job*)p;
  for (int64_t r = j->begin; r < j->end; ++r) j->fn(j->ctx, r);
  return NULL;
}

int oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void parallel_rows(row_fn fn, void* ctx, int64_t rows, int nthreads) {
  if (nthreads <= 0) nthreads = oracle_default_threads();
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
  if (nthreads <= 1) {
    for (int64_t r = 0; r < rows; ++r) fn(ctx, r);
    return;
  }
  pthread_t th[256];
  row_job jobs[256];
  int64_t per = (rows + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].begin = (int64_t)t * per;
    jobs[t].end = jobs[t].begin + per < rows ? jobs[t].begin + per : rows;
    if (jobs[t].begin >= jobs[t].end) break;
    if (pthread_create(&th[t], NULL, run_rows, &jobs[t]) != 0) {
      run_rows(&jobs[t]); /* no thread available: run inline */
      jobs[t].fn = NULL;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (jobs[t].fn) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* RMSNorm                                                             */
/* ------------------------------------------------------------------ */
/* Root-mean-square normalisation of one token's hidden vector (P3, "Where
 * the reductions are" and "A Concrete Example": a sum of squares across the
 * hidden dimension, then a division by the square root of the mean; the
 * operation of Zhang & Sennrich, cited by P3):
 *     ms[i]   = (1/H) * sum_j x[i,j]^2
 *     y[i,j]  = x[i,j] / sqrt(ms[i] + eps) * w[j]
 * eps sits inside the square root; there is no mean subtraction.
 * mean_sq (may be NULL) receives ms[i]. */
typedef struct {
  const uint16_t *x, *w;
  int64_t H;
  double eps;
  double *y, *mean_sq;
} rms_ctx;

static void rms_row(void* p, int64_t i) {
  rms_ctx* c = (rms_ctx*)p;
  const uint16_t* xr = c->x + i * c->H;
  double ss = 0.0;
  for (int64_t j = 0; j < c->H; ++j) {
    double v = bf16_val(xr[j]);
    ss += v * v;
  }
  double ms = ss / (double)c->H;
  double inv = 1.0 / sqrt(ms + c->eps);
  if (c->mean_sq) c->mean_sq[i] = ms;
  for (int64_t j = 0; j < c->H; ++j)
    c->y[i * c->H + j] = bf16_val(xr[j]) * inv * bf16_val(c->w[j]);
}

int oracle_rmsnorm(const uint16_t* x, const uint16_t* w, int64_t M, int64_t H,
                   double eps, double* y, double* mean_sq, int nthreads) {
  if (M < 0 || H <= 0 || !x || !w || !y) return -1;
  rms_ctx c = {x, w, H, eps, y, mean_sq};
  parallel_rows(rms_row, &c, M, nthreads);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Residual add (the step in front of a pre-norm RMSNorm)              */
/* ------------------------------------------------------------------ */
/* The residual stream is kept in bf16: h = round_bf16(float(x) + float(r)),
 * the sum of the two bf16 values in IEEE single precision (round to nearest
 * even), then rounded once more to bf16, nearest even.  The library's fused
 * add-RMSNorm normalises this h; the RMSNorm itself is oracle_rmsnorm. */
static uint16_t bf16_round_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) /* inf or nan: keep, quiet the nan */
    return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

int oracle_add_bf16(const uint16_t* x, const uint16_t* r, int64_t n, uint16_t* h) {
  if (n < 0 || (n > 0 && (!x || !r || !h))) return -1;
  for (int64_t i = 0; i < n; ++i) {
    const float a = (float)bf16_val(x[i]), b = (float)bf16_val(r[i]);
    volatile float s = a + b; /* one single-precision rounding, no wider intermediate */
    h[i] = bf16_round_rne(s);
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* GEMM                                                                */
/* ------------------------------------------------------------------ */
/* The linear layer: every output element is one dot product over the
 * contraction dimension (P1 §3.3, P3 "Where the reductions are"):
 *     C[i,n] = sum_k A[i,k] * W[n,k]
 * A is [M,K] row-major, W is [N,K] row-major (a Linear layer's weight).
 * rows == NULL: all M rows, C is [M,N].  Otherwise only the listed rows of A
 * are computed and C is [nrows,N] (a sample of a large product). */
typedef struct {
  const uint16_t *A, *W;
  int64_t N, K;
  const int64_t* rows;
  double* C;
} gemm_ctx;

static void gemm_row(void* p, int64_t r) {
  gemm_ctx* c = (gemm_ctx*)p;
  int64_t i = c->rows ? c->rows[r] : r;
  const uint16_t* a = c->A + i * c->K;
  double* a_d = (double*)malloc(sizeof(double) * (size_t)c->K);
  if (!a_d) return;
  for (int64_t k = 0; k < c->K; ++k) a_d[k] = bf16_val(a[k]);
  for (int64_t n = 0; n < c->N; ++n) {
    const uint16_t* wr = c->W + n * c->K;
    double acc = 0.0;
    for (int64_t k = 0; k < c->K; ++k) acc += a_d[k] * bf16_val(wr[k]);
    c->C[r * c->N + n] = acc;
  }
  free(a_d);
}

int oracle_gemm(const uint16_t* A, const uint16_t* W, int64_t M, int64_t N,
                int64_t K, const int64_t* rows, int64_t nrows, double* C,
                int nthreads) {
  if (!A || !W || !C || M < 0 || N <= 0 || K <= 0) return -1;
  if (rows)
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= M) return -2;
  gemm_ctx c = {A, W, N, K, rows, C};
  parallel_rows(gemm_row, &c, rows ? nrows : M, nthreads);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Attention over a paged KV cache                                     */
/* ------------------------------------------------------------------ */
/* Softmax attention for one query row over keys 0..n-1 of its sequence
 * (P1 §5.5; FlashAttention, cited by P3):
 *     s_t   = scale * <q, k_t>
 *     out   = sum_t softmax(s)_t * v_t
 * The keys live in a paged cache (PagedAttention, cited by P1 §1.1 and P3):
 * K and V are [num_pages][Hkv][page_size][D]; token t of sequence b is in
 * page block_table[b*max_blocks + t/page_size], slot t%page_size.
 * Grouped-query attention: q-head h reads kv-head h / (Hq/Hkv).
 * Decode: one row per request, n = kv length.  Causal prefill: one row per
 * prompt token at absolute position p, n = p+1.  Both are this function.
 * q is [R][Hq][D]; out is [R][Hq][D]; row r belongs to sequence row_seq[r]
 * and sees row_nkeys[r] keys. */
typedef struct {
  const uint16_t *q, *k, *v;
  int Hq, Hkv, D, page_size, max_blocks;
  int64_t num_pages;
  const int32_t *row_seq, *row_nkeys, *block_table;
  double scale;
  double* out;
  int64_t split_size, split_count; /* used by the split statement only */
  int status;
} attn_ctx;

static const uint16_t* kv_row(const attn_ctx* c, const uint16_t* base,
                              int32_t seq, int64_t t, int kvh) {
  int32_t page = c->block_table[(int64_t)seq * c->max_blocks + t / c->page_size];
  if (page < 0 || page >= c->num_pages) return NULL;
  return base + ((((int64_t)page * c->Hkv + kvh) * c->page_size +
                  t % c->page_size) * (int64_t)c->D);
}

static void attn_row(void* p, int64_t r) {
  attn_ctx* c = (attn_ctx*)p;
  int32_t seq = c->row_seq[r];
  int64_t n = c->row_nkeys[r];
  int G = c->Hq / c->Hkv;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  if (!s) { c->status = -3; return; }
  for (int h = 0; h < c->Hq; ++h) {
    int kvh = h / G;
    const uint16_t* q = c->q + ((int64_t)r * c->Hq + h) * c->D;
    double* o = c->out + ((int64_t)r * c->Hq + h) * c->D;
    double smax = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
      const uint16_t* kr = kv_row(c, c->k, seq, t, kvh);
      if (!kr) { c->status = -4; free(s); return; }
      double dot = 0.0;
      for (int d = 0; d < c->D; ++d) dot += bf16_val(q[d]) * bf16_val(kr[d]);
      s[t] = c->scale * dot;
      if (s[t] > smax) smax = s[t];
    }
    /* softmax(s)_t = exp(s_t - max) / sum exp(s - max): subtracting the
     * maximum is an exact identity that only keeps exp() in range. */
    double den = 0.0;
    for (int64_t t = 0; t < n; ++t) { s[t] = exp(s[t] - smax); den += s[t]; }
    for (int d = 0; d < c->D; ++d) o[d] = 0.0;
    for (int64_t t = 0; t < n; ++t) {
      const uint16_t* vr = kv_row(c, c->v, seq, t, kvh);
      double wgt = s[t] / den;
      for (int d = 0; d < c->D; ++d) o[d] += wgt * bf16_val(vr[d]);
    }
    if (n == 0)
      for (int d = 0; d < c->D; ++d) o[d] = NAN; /* undefined: no keys */
  }
  free(s);
}

static int attn_check(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      int Hq, int Hkv, int D, int page_size, int max_blocks,
                      const int32_t* row_seq, const int32_t* row_nkeys,
                      const int32_t* block_table, double* out) {
  if (!q || !k || !v || !row_seq || !row_nkeys || !block_table || !out) return -1;
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0 || max_blocks <= 0)
    return -1;
  return 0;
}

int oracle_attention(const uint16_t* q, int64_t R, int Hq, int D,
                     const int32_t* row_seq, const int32_t* row_nkeys,
                     const uint16_t* k_cache, const uint16_t* v_cache, int Hkv,
                     int page_size, int64_t num_pages,
                     const int32_t* block_table, int max_blocks, double scale,
                     double* out, int nthreads) {
  int e = attn_check(q, k_cache, v_cache, Hq, Hkv, D, page_size, max_blocks,
                     row_seq, row_nkeys, block_table, out);
  if (e) return e;
  for (int64_t r = 0; r < R; ++r)
    if (row_nkeys[r] < 0 || row_nkeys[r] > (int64_t)max_blocks * page_size) return -2;
  attn_ctx c = {q, k_cache, v_cache, Hq, Hkv, D, page_size, max_blocks,
                num_pages, row_seq, row_nkeys, block_table, scale, out, 0, 0, 0};
  parallel_rows(attn_row, &c, R, nthreads);
  return c.status;
}

/* ------------------------------------------------------------------ */
/* Split planning (integer work)                                       */
/* ------------------------------------------------------------------ */
/* Fixed split SIZE (P1 §5.5; P3 "The attention detail that gets missed"):
 * a sequence of L keys is cut into chunks of S keys starting at key 0, the
 * last one shorter; the boundaries depend only on absolute key indices.
 * Writes the start of each chunk (and starts[count] = L) and returns the
 * count, or -1 if cap is too small. */
int64_t oracle_split_starts_fixed_size(int64_t L, int64_t S, int64_t* starts,
                                       int64_t cap) {
  if (L < 0 || S <= 0) return -1;
  int64_t n = 0;
  for (int64_t b = 0; b < L; b += S) {
    if (n >= cap) return -1;
    starts[n++] = b;
  }
  if (n >= cap) return -1;
  starts[n] = L;
  return n;
}

/* Fixed split COUNT (the FlashDecoding-style plan the pages reject): L keys
 * cut into c chunks whose boundaries sit at floor(j*L/c), so they move as
 * L grows (P3: 250 at L=1000, 256 at L=1024 with four chunks). */
int64_t oracle_split_starts_fixed_count(int64_t L, int64_t count, int64_t* starts,
                                        int64_t cap) {
  if (L < 0 || count <= 0 || cap < count + 1) return -1;
  for (int64_t j = 0; j <= count; ++j) starts[j] = (j * L) / count;
  return count;
}

/* Attention evaluated split by split and merged in index order: for each
 * chunk j of the split plan, the chunk-local maximum m_j, the sum
 * l_j = sum exp(s - m_j) and the unnormalised o_j = sum exp(s - m_j) v; then
 * a left fold over j = 0,1,... with the log-sum-exp merge
 *     m = max(m_a, m_b), l = l_a e^(m_a-m) + l_b e^(m_b-m), o likewise,
 * and out = o / l (P1 §4.3: partials combined in a fixed, non-parallel
 * clean-up; P1 §5.5: fixed split size).  Exact in real arithmetic, so in
 * fp64 it must agree with oracle_attention to rounding.
 * split_size > 0 selects the fixed-size plan, otherwise split_count > 0 the
 * fixed-count plan. */
static void attn_split_row(void* p, int64_t r) {
  attn_ctx* c = (attn_ctx*)p;
  int32_t seq = c->row_seq[r];
  int64_t n = c->row_nkeys[r];
  int G = c->Hq / c->Hkv;
  int64_t cap = n + 2 + c->split_count;
  int64_t* st = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
  double* o_j = (double*)malloc(sizeof(double) * (size_t)c->D);
  if (!st || !o_j) { c->status = -3; free(st); free(o_j); return; }
  int64_t ns = c->split_size > 0
                   ? oracle_split_starts_fixed_size(n, c->split_size, st, cap)
                   : oracle_split_starts_fixed_count(n, c->split_count, st, cap);
  for (int h = 0; h < c->Hq; ++h) {
    int kvh = h / G;
    const uint16_t* q = c->q + ((int64_t)r * c->Hq + h) * c->D;
    double* o = c->out + ((int64_t)r * c->Hq + h) * c->D;
    double m = -INFINITY, l = 0.0;
    int have = 0;
    for (int d = 0; d < c->D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < ns; ++j) {
      if (st[j] >= st[j + 1]) continue; /* empty chunk (count plan, tiny L) */
      double mj = -INFINITY, lj = 0.0;
      for (int64_t t = st[j]; t < st[j + 1]; ++t) {
        const uint16_t* kr = kv_row(c, c->k, seq, t, kvh);
        if (!kr) { c->status = -4; goto out; }
        double dot = 0.0;
        for (int d = 0; d < c->D; ++d) dot += bf16_val(q[d]) * bf16_val(kr[d]);
        if (c->scale * dot > mj) mj = c->scale * dot;
      }
      for (int d = 0; d < c->D; ++d) o_j[d] = 0.0;
      for (int64_t t = st[j]; t < st[j + 1]; ++t) {
        const uint16_t* kr = kv_row(c, c->k, seq, t, kvh);
        const uint16_t* vr = kv_row(c, c->v, seq, t, kvh);
        double dot = 0.0;
        for (int d = 0; d < c->D; ++d) dot += bf16_val(q[d]) * bf16_val(kr[d]);
        double e = exp(c->scale * dot - mj);
        lj += e;
        for (int d = 0; d < c->D; ++d) o_j[d] += e * bf16_val(vr[d]);
      }
      if (!have) {
        m = mj; l = lj;
        for (int d = 0; d < c->D; ++d) o[d] = o_j[d];
        have = 1;
      } else {
        double mn = m > mj ? m : mj;
        double ca = exp(m - mn), cb = exp(mj - mn);
        l = l * ca + lj * cb;
        for (int d = 0; d < c->D; ++d) o[d] = o[d] * ca + o_j[d] * cb;
        m = mn;
      }
    }
    for (int d = 0; d < c->D; ++d) o[d] = have ? o[d] / l : NAN;
  }
out:
  free(st);
  free(o_j);
}

int oracle_attention_splits(const uint16_t* q, int64_t R, int Hq, int D,
                            const int32_t* row_seq, const int32_t* row_nkeys,
                            const uint16_t* k_cache, const uint16_t* v_cache,
                            int Hkv, int page_size, int64_t num_pages,
                            const int32_t* block_table, int max_blocks,
                            double scale, int64_t split_size, int64_t split_count,
                            double* out, int nthreads) {
  int e = attn_check(q, k_cache, v_cache, Hq, Hkv, D, page_size, max_blocks,
                     row_seq, row_nkeys, block_table, out);
  if (e) return e;
  if (split_size <= 0 && split_count <= 0) return -1;
  for (int64_t r = 0; r < R; ++r)
    if (row_nkeys[r] < 0 || row_nkeys[r] > (int64_t)max_blocks * page_size) return -2;
  attn_ctx c = {q, k_cache, v_cache, Hq, Hkv, D, page_size, max_blocks,
                num_pages, row_seq, row_nkeys, block_table, scale, out,
                split_size, split_count, 0};
  parallel_rows(attn_split_row, &c, R, nthreads);
  return c.status;
}

/* ------------------------------------------------------------------ */
/* Seeded sampling ([P1] §9.2, §9.3)                                   */
/* ------------------------------------------------------------------ */
/* [P1] §9.3: a sampler that is deterministic under batching perturbs the
 * logits with Gumbel noise drawn from a seeded hash and takes the argmax
 * (the Gumbel-max construction: argmax_v (z_v / T + G_v) with G_v i.i.d.
 * standard Gumbel is a draw from softmax(z / T)); §9.2: temperature 0 is the
 * plain argmax.  The pages name no hash; this oracle and the kernel each
 * implement Philox4x64-10 from its publication (Salmon, Moraes, Dror and
 * Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011): a 4 x 64-bit
 * counter and a 2 x 64-bit key, ten rounds of two 64 x 64 -> 128-bit
 * products, the key advanced by two Weyl constants between rounds. */
static void philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B97F4A7C15ull;   /* golden ratio */
      k1 += 0xBB67AE8584CAA73Bull;   /* sqrt(3) - 1 */
    }
    unsigned __int128 p0 = (unsigned __int128)0xD2E7470EE14C6C93ull * c0;
    unsigned __int128 p1 = (unsigned __int128)0xCA5A826395121157ull * c2;
    uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
    uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

void oracle_philox4x64(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  philox4x64_10(ctr, key, out);
}

/* The uniform of vocabulary entry v for (seed, step): one Philox block per 8
 * entries (counter {v / 8, step, 0, 0}, key {seed, 0}); entry v takes 32-bit
 * half v % 2 (0 = low) of 64-bit word (v / 2) % 4, keeps its top 23 bits k
 * and maps them to u = (k + 1/2) 2^-23, strictly inside (0, 1). */
static double sample_uniform(uint64_t seed, uint64_t step, int64_t v) {
  const uint64_t ctr[4] = {(uint64_t)v >> 3, step, 0, 0}, key[2] = {seed, 0};
  uint64_t out[4];
  philox4x64_10(ctr, key, out);
  const uint64_t w = out[(v >> 1) & 3];
  const uint32_t half = (v & 1) ? (uint32_t)(w >> 32) : (uint32_t)w;
  return ((double)(half >> 9) + 0.5) * 0x1p-23;
}

int oracle_sample_uniform(uint64_t seed, uint64_t step, int64_t v0, int64_t n, double* u) {
  if (v0 < 0 || n < 0 || (n && !u)) return -1;
  for (int64_t i = 0; i < n; ++i) u[i] = sample_uniform(seed, step, v0 + i);
  return 0;
}

typedef struct {
  const uint16_t* logits;
  int64_t V;
  const float* temperature;
  const uint64_t* seed;
  const uint64_t* step;
  double* scores;
} sample_ctx;

/* Score of entry v of row b: z / T + G with G = -log(-log(u)) for T > 0,
 * else the logit itself (greedy). */
static void sample_row(void* p, int64_t b) {
  sample_ctx* c = (sample_ctx*)p;
  const uint16_t* z = c->logits + b * c->V;
  double* s = c->scores + b * c->V;
  const double T = (double)c->temperature[b];
  for (int64_t v = 0; v < c->V; ++v) {
    const double x = bf16_val(z[v]);
    if (T > 0.0) {
      const double u = sample_uniform(c->seed[b], c->step[b], v);
      s[v] = x / T - log(-log(u));
    } else {
      s[v] = x;
    }
  }
}

int oracle_sample_scores(const uint16_t* logits, int64_t B, int64_t V, const float* temperature,
                         const uint64_t* seed, const uint64_t* step, double* scores,
                         int nthreads) {
  if (B < 0 || V <= 0) return -1;
  if (B == 0) return 0;
  if (!logits || !temperature || !seed || !step || !scores) return -1;
  sample_ctx c = {logits, V, temperature, seed, step, scores};
  parallel_rows(sample_row, &c, B, nthreads);
  return 0;
}
