/*
 * FP64 CPU oracle for paged MQA/GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * statement of what the GPU path computes. Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it. It shares no
 * code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * What it follows (Loom Kernels landing page, "Supported now", the
 * "Paged MQA/GQA decode" entry: GQA packing + local split-K/LSE; and the
 * benchmark page, "Current qualified results": the D128 long-context
 * split-K/LSE path). The pages name the operator but print no formula, so the
 * operator is the textbook one its name denotes:
 *
 *   for every sequence b and query head hq, with G = Hq / Hkv,
 *   kv head h = floor(hq / G), context length L = context_lens[b]:
 *     k_t = k_cache[block_table[b, floor(t / bs)], t mod bs, h, :]   (t < L)
 *     v_t = v_cache[block_table[b, floor(t / bs)], t mod bs, h, :]
 *     s_t = scale * sum_d q[b, hq, d] * k_t[d]
 *     out[b, hq, :] = sum_t softmax(s)_t * v_t
 *
 * Every input element is converted exactly to double; every sum is a plain
 * left-to-right double sum in token order; softmax subtracts the row maximum
 * before exponentiating. There is no blocking, no online softmax and no
 * re-association: the loops below are the definition written out.
 *
 * Readings where the pages are silent:
 *   - no mask other than t < L (plain decode over the whole context);
 *   - contiguous GQA groups: query head hq reads kv head floor(hq / G);
 *   - block-table entries at page index >= ceil(L / bs) are never read;
 *   - L == 0 yields a zero output row (the GPU path does the same);
 *   - split-K: a sequence's pages are cut into contiguous, page-aligned
 *     chunks of `chunk_pages` pages; a chunk with no tokens has lse = -inf and
 *     o = 0; chunks are merged by log-sum-exp weighting.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BF16 0
#define ORACLE_FP16 1
#define ORACLE_FP8_E4M3 2 /* K/V cache elements only */

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ERANGE (-2)
#define ORACLE_ENOMEM (-3)

/* ---------------------------------------------------------------------------
 * Exact conversions between 16-bit storage formats and double.
 * bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits (the top half of
 * an IEEE binary32). binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
 * ------------------------------------------------------------------------- */

double oracle_bf16_to_f64(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int exp = (bits >> 7) & 0xff;
  int frac = bits & 0x7f;
  double mag;
  if (exp == 0xff) {
    mag = frac ? NAN : INFINITY;
  } else if (exp == 0) {
    mag = ldexp((double)frac, -126 - 7); /* subnormal: frac * 2^-133 */
  } else {
    mag = ldexp((double)(128 + frac), exp - 127 - 7);
  }
  return sign ? -mag : mag;
}

double oracle_fp16_to_f64(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int exp = (bits >> 10) & 0x1f;
  int frac = bits & 0x3ff;
  double mag;
  if (exp == 0x1f) {
    mag = frac ? NAN : INFINITY;
  } else if (exp == 0) {
    mag = ldexp((double)frac, -14 - 10); /* subnormal: frac * 2^-24 */
  } else {
    mag = ldexp((double)(1024 + frac), exp - 15 - 10);
  }
  return sign ? -mag : mag;
}

double oracle_to_f64(uint16_t bits, int dtype) {
  return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(bits) : oracle_fp16_to_f64(bits);
}

/* Round a double to the nearest value with `mant_bits` fraction bits and
 * minimum normal exponent `emin`, ties to even, directly from double (no
 * intermediate float, so no double rounding). Returns the rounded double;
 * values beyond the largest finite number of the format become infinity. */
static double round_to_format(double x, int mant_bits, int emin, double max_finite) {
  if (x == 0.0 || isnan(x) || isinf(x)) return x;
  int e;
  frexp(x, &e);            /* |x| = f * 2^e, f in [0.5, 1) */
  int exp_unbiased = e - 1; /* |x| in [2^(e-1), 2^e) */
  if (exp_unbiased < emin) exp_unbiased = emin; /* subnormal spacing */
  double quantum = ldexp(1.0, exp_unbiased - mant_bits);
  double scaled = x / quantum; /* exact: division by a power of two */
  /* ties to even on the integer grid */
  double fl = floor(scaled);
  double diff = scaled - fl;
  double r;
  if (diff > 0.5) {
    r = fl + 1.0;
  } else if (diff < 0.5) {
    r = fl;
  } else {
    r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  }
  double y = r * quantum;
  if (fabs(y) > max_finite) return x > 0 ? INFINITY : -INFINITY;
  return copysign(y, x); /* a value that rounds to zero keeps its sign */
}

/* bfloat16 largest finite: (2 - 2^-7) * 2^127; binary16: 65504. */
double oracle_round_bf16(double x) {
  return round_to_format(x, 7, -126, ldexp(255.0, 120));
}

double oracle_round_fp16(double x) { return round_to_format(x, 10, -14, 65504.0); }

/* Encode an already-rounded double as a 16-bit pattern. */
static uint16_t encode_bf16(double y) {
  float f = (float)y; /* exact: y is representable in binary32 */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if (isnan(y)) return 0x7fc0;
  return (uint16_t)(u >> 16);
}

static uint16_t encode_fp16(double y) {
  if (isnan(y)) return 0x7e00;
  uint16_t sign = signbit(y) ? 0x8000 : 0;
  double a = fabs(y);
  if (isinf(a)) return sign | 0x7c00;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  int exp_unbiased = e - 1;
  if (exp_unbiased < -14) { /* subnormal: a = frac * 2^-24 */
    return sign | (uint16_t)ldexp(a, 24);
  }
  uint16_t frac = (uint16_t)(ldexp(a, 10 - exp_unbiased) - 1024.0);
  return sign | (uint16_t)((exp_unbiased + 15) << 10) | frac;
}

void oracle_round_array(const double* x, int64_t n, int dtype, uint16_t* bits_out,
                        double* rounded_out) {
  for (int64_t i = 0; i < n; ++i) {
    double y = dtype == ORACLE_BF16 ? oracle_round_bf16(x[i]) : oracle_round_fp16(x[i]);
    if (rounded_out) rounded_out[i] = y;
    if (bits_out) bits_out[i] = dtype == ORACLE_BF16 ? encode_bf16(y) : encode_fp16(y);
  }
}

void oracle_decode_array(const uint16_t* bits, int64_t n, int dtype, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_to_f64(bits[i], dtype);
}

/* FP8 E4M3 (the "fn" variant of the OCP 8-bit formats): 1 sign, 4 exponent
 * (bias 7), 3 fraction bits; exponent 0 holds subnormals m * 2^-9; there is
 * no infinity, and S.1111.111 is NaN. Largest finite value 448. */
double oracle_e4m3_to_f64(uint8_t bits) {
  int sign = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(8.0 + m, e - 7 - 3);
  return sign ? -v : v;
}

void oracle_decode_e4m3_array(const uint8_t* bits, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f64(bits[i]);
}

/* ---------------------------------------------------------------------------
 * Problem description shared by the entry points below.
 * ------------------------------------------------------------------------- */
typedef struct {
  const uint16_t* q;       /* [B, Hq, D] */
  const void* k_cache;     /* [num_blocks, bs, Hkv, D], elements of kv_dtype */
  const void* v_cache;     /* [num_blocks, bs, Hkv, D] */
  const int32_t* block_table; /* [B, max_blocks] */
  const int32_t* context_lens; /* [B] */
  int B, Hq, Hkv, D, bs, max_blocks;
  int64_t num_blocks;
  int dtype;               /* of q */
  double scale;
  int kv_dtype;            /* BF16, FP16 or FP8_E4M3 */
  const double* k_scale;   /* [Hkv] dequantisation scales, NULL = 1 */
  const double* v_scale;
} problem;

static int check_problem(const problem* p) {
  if (!p->q || !p->k_cache || !p->v_cache || !p->block_table || !p->context_lens)
    return ORACLE_EINVAL;
  if (p->B < 0 || p->Hq <= 0 || p->Hkv <= 0 || p->D <= 0 || p->bs <= 0 || p->max_blocks < 0)
    return ORACLE_EINVAL;
  if (p->Hq % p->Hkv != 0) return ORACLE_EINVAL;
  if (p->dtype != ORACLE_BF16 && p->dtype != ORACLE_FP16) return ORACLE_EINVAL;
  if (p->kv_dtype != ORACLE_BF16 && p->kv_dtype != ORACLE_FP16 && p->kv_dtype != ORACLE_FP8_E4M3)
    return ORACLE_EINVAL;
  for (int b = 0; b < p->B; ++b) {
    int L = p->context_lens[b];
    if (L < 0 || (int64_t)L > (int64_t)p->max_blocks * p->bs) return ORACLE_ERANGE;
    int pages = (L + p->bs - 1) / p->bs;
    for (int i = 0; i < pages; ++i) {
      int32_t blk = p->block_table[(int64_t)b * p->max_blocks + i];
      if (blk < 0 || (int64_t)blk >= p->num_blocks) return ORACLE_ERANGE;
    }
  }
  return ORACLE_OK;
}

/* Element index of (token t of sequence b, kv head h, dim 0) in a cache. */
static int64_t cache_row(const problem* p, int b, int t, int h) {
  int32_t blk = p->block_table[(int64_t)b * p->max_blocks + t / p->bs];
  int off = t % p->bs;
  return (((int64_t)blk * p->bs + off) * p->Hkv + h) * p->D;
}

/* Element i of a K or V cache of kv head h: its exact value times the head's
 * dequantisation scale (no scale: the value itself). */
static double kv_value(const problem* p, const void* cache, const double* head_scale, int h,
                       int64_t i) {
  double x = p->kv_dtype == ORACLE_FP8_E4M3
                 ? oracle_e4m3_to_f64(((const uint8_t*)cache)[i])
                 : oracle_to_f64(((const uint16_t*)cache)[i], p->kv_dtype);
  return head_scale ? x * head_scale[h] : x;
}

/* Scaled logit s_t = scale * q[b,hq,:] . k_t */
static double logit(const problem* p, int b, int hq, int h, int t) {
  const uint16_t* qrow = p->q + ((int64_t)b * p->Hq + hq) * p->D;
  const int64_t krow = cache_row(p, b, t, h);
  double dot = 0.0;
  for (int d = 0; d < p->D; ++d)
    dot += oracle_to_f64(qrow[d], p->dtype) * kv_value(p, p->k_cache, p->k_scale, h, krow + d);
  return p->scale * dot;
}

/* softmax(s) . V over tokens [t0, t1) of one (b, hq) row.
 * Writes the normalised output to o[0..D), and returns via *m_out / *l_out
 * the row maximum and the sum of exp(s - max). Empty ranges give m = -inf,
 * l = 0 and o = 0. `s` is caller scratch of length >= t1 - t0. */
static void attend_range(const problem* p, int b, int hq, int t0, int t1, double* s, double* o,
                         double* m_out, double* l_out) {
  int G = p->Hq / p->Hkv;
  int h = hq / G;
  for (int d = 0; d < p->D; ++d) o[d] = 0.0;
  if (t1 <= t0) {
    *m_out = -INFINITY;
    *l_out = 0.0;
    return;
  }
  double m = -INFINITY;
  for (int t = t0; t < t1; ++t) {
    s[t - t0] = logit(p, b, hq, h, t);
    if (s[t - t0] > m) m = s[t - t0];
  }
  double l = 0.0;
  for (int t = t0; t < t1; ++t) {
    double w = exp(s[t - t0] - m);
    l += w;
    const int64_t vrow = cache_row(p, b, t, h);
    for (int d = 0; d < p->D; ++d) o[d] += w * kv_value(p, p->v_cache, p->v_scale, h, vrow + d);
  }
  for (int d = 0; d < p->D; ++d) o[d] /= l;
  *m_out = m;
  *l_out = l;
}

/* ---------------------------------------------------------------------------
 * Row-parallel driver: rows are (b, hq) pairs, handed out in contiguous
 * slices to plain pthreads. Each row is computed independently.
 * ------------------------------------------------------------------------- */
typedef struct {
  const problem* p;
  const int32_t* rows; /* pairs (b, hq); NULL = all rows in order */
  int64_t row_begin, row_end;
  double* out;         /* [n_rows, D] */
  int status;
} row_job;

static void* run_rows(void* arg) {
  row_job* j = (row_job*)arg;
  const problem* p = j->p;
  int max_len = p->max_blocks * p->bs;
  double* s = (double*)malloc(sizeof(double) * (max_len > 0 ? max_len : 1));
  if (!s) {
    j->status = ORACLE_ENOMEM;
    return NULL;
  }
  for (int64_t r = j->row_begin; r < j->row_end; ++r) {
    int b, hq;
    if (j->rows) {
      b = j->rows[2 * r];
      hq = j->rows[2 * r + 1];
    } else {
      b = (int)(r / p->Hq);
      hq = (int)(r % p->Hq);
    }
    double m, l;
    attend_range(p, b, hq, 0, p->context_lens[b], s, j->out + r * p->D, &m, &l);
  }
  free(s);
  j->status = ORACLE_OK;
  return NULL;
}

static int run_parallel(const problem* p, const int32_t* rows, int64_t n_rows, double* out,
                        int num_threads) {
  if (num_threads < 1) num_threads = 1;
  if (num_threads > 256) num_threads = 256;
  if ((int64_t)num_threads > n_rows) num_threads = n_rows > 0 ? (int)n_rows : 1;
  pthread_t tids[256];
  row_job jobs[256];
  int64_t per = (n_rows + num_threads - 1) / num_threads;
  int started = 0;
  for (int i = 0; i < num_threads; ++i) {
    jobs[i].p = p;
    jobs[i].rows = rows;
    jobs[i].row_begin = i * per < n_rows ? i * per : n_rows;
    jobs[i].row_end = (i + 1) * per < n_rows ? (i + 1) * per : n_rows;
    jobs[i].out = out;
    jobs[i].status = ORACLE_OK;
  }
  if (num_threads == 1) {
    run_rows(&jobs[0]);
    return jobs[0].status;
  }
  for (int i = 0; i < num_threads; ++i) {
    if (pthread_create(&tids[i], NULL, run_rows, &jobs[i]) != 0) break;
    ++started;
  }
  for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
  if (started != num_threads) {
    /* fall back to finishing the remaining slices on this thread */
    for (int i = started; i < num_threads; ++i) run_rows(&jobs[i]);
  }
  for (int i = 0; i < num_threads; ++i)
    if (jobs[i].status != ORACLE_OK) return jobs[i].status;
  return ORACLE_OK;
}

/* Full output: out[B, Hq, D] in double. */
int oracle_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_table, const int32_t* context_lens, int B, int Hq,
                        int Hkv, int D, int block_size, int max_blocks, int64_t num_blocks,
                        int dtype, double scale, double* out, int num_threads) {
  problem p = {q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv, D,
               block_size, max_blocks, num_blocks, dtype, scale, dtype, NULL, NULL};
  int st = check_problem(&p);
  if (st != ORACLE_OK) return st;
  if (!out) return ORACLE_EINVAL;
  return run_parallel(&p, NULL, (int64_t)B * Hq, out, num_threads);
}

/* Selected rows only: rows = n_rows pairs (b, hq); out_rows[n_rows, D]. */
int oracle_paged_decode_rows(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* block_table, const int32_t* context_lens, int B,
                             int Hq, int Hkv, int D, int block_size, int max_blocks,
                             int64_t num_blocks, int dtype, double scale, const int32_t* rows,
                             int64_t n_rows, double* out_rows, int num_threads) {
  problem p = {q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv, D,
               block_size, max_blocks, num_blocks, dtype, scale, dtype, NULL, NULL};
  int st = check_problem(&p);
  if (st != ORACLE_OK) return st;
  if (!rows || !out_rows || n_rows < 0) return ORACLE_EINVAL;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[2 * r] < 0 || rows[2 * r] >= B || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= Hq)
      return ORACLE_EINVAL;
  return run_parallel(&p, rows, n_rows, out_rows, num_threads);
}

/* Any K/V element type with per-kv-head dequantisation scales (FP8 KV
 * cache; the pages leave the scale granularity open, so per kv head is the
 * reading and a per-tensor scale is the case of equal entries):
 *   k_t[d] = k_scale[h] * decode(k_cache element), likewise v_t with v_scale.
 * q is bf16/fp16 (q_dtype). rows: n_rows pairs (b, hq), or NULL for all
 * B * Hq rows in order (n_rows ignored). out_rows[rows, D]. */
int oracle_paged_decode_kv(const uint16_t* q, const void* k_cache, const void* v_cache,
                           int kv_dtype, const double* k_scale, const double* v_scale,
                           const int32_t* block_table, const int32_t* context_lens, int B,
                           int Hq, int Hkv, int D, int block_size, int max_blocks,
                           int64_t num_blocks, int q_dtype, double scale, const int32_t* rows,
                           int64_t n_rows, double* out_rows, int num_threads) {
  problem p = {q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv, D,
               block_size, max_blocks, num_blocks, q_dtype, scale, kv_dtype, k_scale, v_scale};
  int st = check_problem(&p);
  if (st != ORACLE_OK) return st;
  if (!out_rows) return ORACLE_EINVAL;
  if (!rows) return run_parallel(&p, NULL, (int64_t)B * Hq, out_rows, num_threads);
  if (n_rows < 0) return ORACLE_EINVAL;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[2 * r] < 0 || rows[2 * r] >= B || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= Hq)
      return ORACLE_EINVAL;
  return run_parallel(&p, rows, n_rows, out_rows, num_threads);
}

/* Split-K partials. Split s of sequence b covers pages
 * [s * chunk_pages, (s + 1) * chunk_pages) clipped to the sequence's
 * ceil(L / bs) pages, i.e. tokens [s * chunk_pages * bs, ...) clipped to L.
 * For every (b, hq, s < num_splits):
 *   lse[b, hq, s] = log sum_{t in split} exp(s_t)   (-inf if the split is empty)
 *   o[b, hq, s, :] = softmax over the split's tokens, applied to V (0 if empty)
 */
int oracle_split_partials(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                          const int32_t* block_table, const int32_t* context_lens, int B, int Hq,
                          int Hkv, int D, int block_size, int max_blocks, int64_t num_blocks,
                          int dtype, double scale, int chunk_pages, int num_splits,
                          double* lse, double* o) {
  problem p = {q, k_cache, v_cache, block_table, context_lens, B, Hq, Hkv, D,
               block_size, max_blocks, num_blocks, dtype, scale, dtype, NULL, NULL};
  int st = check_problem(&p);
  if (st != ORACLE_OK) return st;
  if (chunk_pages < 1 || num_splits < 1 || !lse || !o) return ORACLE_EINVAL;
  int max_len = max_blocks * block_size;
  double* s = (double*)malloc(sizeof(double) * (max_len > 0 ? max_len : 1));
  if (!s) return ORACLE_ENOMEM;
  for (int b = 0; b < B; ++b) {
    int L = context_lens[b];
    for (int hq = 0; hq < Hq; ++hq) {
      for (int sp = 0; sp < num_splits; ++sp) {
        int64_t t0 = (int64_t)sp * chunk_pages * block_size;
        int64_t t1 = t0 + (int64_t)chunk_pages * block_size;
        if (t0 > L) t0 = L;
        if (t1 > L) t1 = L;
        int64_t idx = ((int64_t)b * Hq + hq) * num_splits + sp;
        double m, l;
        attend_range(&p, b, hq, (int)t0, (int)t1, s, o + idx * D, &m, &l);
        lse[idx] = (l > 0.0) ? m + log(l) : -INFINITY;
      }
    }
  }
  free(s);
  return ORACLE_OK;
}

/* Log-sum-exp merge of split partials, per row r < n_rows:
 *   M = max_s lse[r, s]
 *   out[r, :] = sum_s exp(lse[r, s] - M) * o[r, s, :] / sum_s exp(lse[r, s] - M)
 * Splits with lse = -inf carry weight 0; a row whose splits are all empty
 * yields zeros. */
int oracle_lse_merge(const double* lse, const double* o, int64_t n_rows, int num_splits, int D,
                     double* out) {
  if (!lse || !o || !out || n_rows < 0 || num_splits < 1 || D < 1) return ORACLE_EINVAL;
  for (int64_t r = 0; r < n_rows; ++r) {
    double M = -INFINITY;
    for (int sp = 0; sp < num_splits; ++sp)
      if (lse[r * num_splits + sp] > M) M = lse[r * num_splits + sp];
    double* orow = out + r * D;
    for (int d = 0; d < D; ++d) orow[d] = 0.0;
    if (M == -INFINITY) continue;
    double wsum = 0.0;
    for (int sp = 0; sp < num_splits; ++sp) {
      double l = lse[r * num_splits + sp];
      if (l == -INFINITY) continue;
      double w = exp(l - M);
      wsum += w;
      const double* os = o + (r * num_splits + sp) * D;
      for (int d = 0; d < D; ++d) orow[d] += w * os[d];
    }
    for (int d = 0; d < D; ++d) orow[d] /= wsum;
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * RoPE + paged-KV write (Loom Kernels landing page, "Supported now":
 * "RoPE + paged-KV write - packed Q/K rotation + native cache write").
 * The pages name the fused step but not its formula; the reading here is the
 * rotary embedding as commonly defined: for token t at position pos_t, for
 * each rotated pair j < rot_dim / 2 with angle table row cs = cos_sin[pos_t]
 * (cos_j = cs[j], sin_j = cs[rot_dim / 2 + j]) and pair elements
 *   (a, b) = (j, j + rot_dim / 2)   (rotate-halves, "neox")  or
 *   (a, b) = (2j, 2j + 1)           (interleaved pairs),
 *   y_a = x_a cos_j - x_b sin_j,   y_b = x_b cos_j + x_a sin_j;
 * dims >= rot_dim pass through. q is rotated into q_out; the rotated k and
 * the unchanged v go to cache row slot_mapping[t] (block-major layout: row
 * index slot = block * block_size + offset). slot < 0 skips the cache write;
 * a position outside [0, max_position) or a slot beyond the cache leaves the
 * token's outputs untouched. Everything in double, rounded once (RNE) to the
 * storage dtype.
 * ------------------------------------------------------------------------- */
static void rope_row(const uint16_t* x, uint16_t* y, const float* cs, int D, int rot_dim,
                     int neox, int dtype) {
  int half = rot_dim / 2;
  for (int d = 0; d < D; ++d) y[d] = x[d];  /* pass-through dims */
  for (int j = 0; j < half; ++j) {
    int a = neox ? j : 2 * j;
    int b = neox ? j + half : 2 * j + 1;
    double c = (double)cs[j], s = (double)cs[half + j];
    double xa = oracle_to_f64(x[a], dtype), xb = oracle_to_f64(x[b], dtype);
    double ya = xa * c - xb * s;
    double yb = xb * c + xa * s;
    y[a] = dtype == ORACLE_BF16 ? encode_bf16(oracle_round_bf16(ya)) : encode_fp16(oracle_round_fp16(ya));
    y[b] = dtype == ORACLE_BF16 ? encode_bf16(oracle_round_bf16(yb)) : encode_fp16(oracle_round_fp16(yb));
  }
}

int oracle_rope_kv_write(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* positions, const int64_t* slot_mapping,
                         const float* cos_sin, int T, int Hq, int Hkv, int D, int rot_dim,
                         int max_position, int neox, int64_t num_slots, int dtype,
                         uint16_t* q_out, uint16_t* k_cache, uint16_t* v_cache) {
  if (!q || !k || !v || !positions || !slot_mapping || !cos_sin || !q_out || !k_cache || !v_cache)
    return ORACLE_EINVAL;
  if (T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || rot_dim < 0 || rot_dim > D || rot_dim % 2)
    return ORACLE_EINVAL;
  for (int t = 0; t < T; ++t) {
    int pos = positions[t];
    if (pos < 0 || pos >= max_position) continue;
    const float* cs = cos_sin + (int64_t)pos * rot_dim;
    for (int h = 0; h < Hq; ++h) {
      int64_t off = ((int64_t)t * Hq + h) * D;
      rope_row(q + off, q_out + off, cs, D, rot_dim, neox, dtype);
    }
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_slots) continue;
    for (int h = 0; h < Hkv; ++h) {
      int64_t src = ((int64_t)t * Hkv + h) * D;
      int64_t dst = (slot * Hkv + h) * D;
      rope_row(k + src, k_cache + dst, cs, D, rot_dim, neox, dtype);
      for (int d = 0; d < D; ++d) v_cache[dst + d] = v[src + d];
    }
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * KV-cache movement (landing page, "Next boundaries": KV-cache movement,
 * "scheduler-facing block copy, gather, scatter, and compact work for prefix
 * reuse and preemption"). The pages name the operations only; the readings:
 * a cache is [num_blocks, block_size, Hkv, D] of any element type, moved as
 * raw bytes (row_bytes = Hkv * D * element size per token slot), so every
 * operation is an exact copy.
 *   copy_blocks: for each pair i, block pairs[2i+1] of both caches becomes a
 *     copy of block pairs[2i] (destinations distinct and not sources, so the
 *     order of the pairs does not matter);
 *   gather: the tokens t < lens[b] of each sequence, in order, through its
 *     block table, into a contiguous [sum(lens), row] buffer (sequence b
 *     starts at row lens[0] + ... + lens[b-1]);
 *   scatter: contiguous rows into the cache slots slot_mapping[t] (slot =
 *     block * block_size + offset; negative = skip);
 *   remap_table: table[b, p] = new_id[table[b, p]] for the pages p <
 *     ceil(lens[b] / block_size) a sequence uses (compaction's table update).
 * ------------------------------------------------------------------------- */
int oracle_copy_blocks(uint8_t* k_cache, uint8_t* v_cache, int64_t num_blocks,
                       int64_t block_bytes, const int64_t* pairs, int64_t n_pairs) {
  if (!k_cache || !v_cache || num_blocks < 0 || block_bytes < 0 || n_pairs < 0)
    return ORACLE_EINVAL;
  if (n_pairs > 0 && !pairs) return ORACLE_EINVAL;
  for (int64_t i = 0; i < n_pairs; ++i) {
    int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return ORACLE_ERANGE;
    for (int64_t j = 0; j < block_bytes; ++j) {
      k_cache[dst * block_bytes + j] = k_cache[src * block_bytes + j];
      v_cache[dst * block_bytes + j] = v_cache[src * block_bytes + j];
    }
  }
  return ORACLE_OK;
}

int oracle_gather_kv(const uint8_t* k_cache, const uint8_t* v_cache, int64_t num_blocks,
                     int block_size, int64_t row_bytes, const int32_t* block_table,
                     int max_blocks, const int32_t* lens, int B, uint8_t* k_out,
                     uint8_t* v_out) {
  if (!k_cache || !v_cache || !block_table || !lens || !k_out || !v_out) return ORACLE_EINVAL;
  if (block_size < 1 || row_bytes < 0 || B < 0 || max_blocks < 0) return ORACLE_EINVAL;
  int64_t row = 0;
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 0 || (int64_t)lens[b] > (int64_t)max_blocks * block_size) return ORACLE_ERANGE;
    for (int t = 0; t < lens[b]; ++t) {
      int32_t blk = block_table[(int64_t)b * max_blocks + t / block_size];
      if (blk < 0 || blk >= num_blocks) return ORACLE_ERANGE;
      int64_t slot = (int64_t)blk * block_size + t % block_size;
      for (int64_t j = 0; j < row_bytes; ++j) {
        k_out[row * row_bytes + j] = k_cache[slot * row_bytes + j];
        v_out[row * row_bytes + j] = v_cache[slot * row_bytes + j];
      }
      ++row;
    }
  }
  return ORACLE_OK;
}

int oracle_scatter_kv(const uint8_t* k_in, const uint8_t* v_in, int64_t n_rows,
                      int64_t row_bytes, const int64_t* slot_mapping, uint8_t* k_cache,
                      uint8_t* v_cache, int64_t num_slots) {
  if (!k_in || !v_in || !slot_mapping || !k_cache || !v_cache || n_rows < 0 || row_bytes < 0)
    return ORACLE_EINVAL;
  for (int64_t t = 0; t < n_rows; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) return ORACLE_ERANGE;
    for (int64_t j = 0; j < row_bytes; ++j) {
      k_cache[slot * row_bytes + j] = k_in[t * row_bytes + j];
      v_cache[slot * row_bytes + j] = v_in[t * row_bytes + j];
    }
  }
  return ORACLE_OK;
}

int oracle_remap_table(int32_t* block_table, int B, int max_blocks, const int32_t* lens,
                       int block_size, const int32_t* new_id, int64_t num_blocks) {
  if (!block_table || !lens || !new_id || B < 0 || max_blocks < 0 || block_size < 1)
    return ORACLE_EINVAL;
  for (int b = 0; b < B; ++b) {
    int pages = (lens[b] + block_size - 1) / block_size;
    if (lens[b] < 0 || pages > max_blocks) return ORACLE_ERANGE;
    for (int p = 0; p < pages; ++p) {
      int32_t* e = block_table + (int64_t)b * max_blocks + p;
      if (*e < 0 || *e >= num_blocks) return ORACLE_ERANGE;
      *e = new_id[*e];
    }
  }
  return ORACLE_OK;
}
