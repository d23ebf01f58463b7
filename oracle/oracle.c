/*
 * Paged KV-cache attention: the plain CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this code.  It shares nothing with the
 * CUDA library (no header, no helper, no constant) and the CUDA library never
 * calls it.
 *
 * What it computes, and where the pages define it:
 *   - the cache write ("How serving works in Tlaloc", section 1 "From a model
 *     to DXIR", and section 2 "From DXIR to StableHLO", KV_CACHE_WRITE bullet):
 *     every token whose slot is not -1 has its K row and V row copied into the
 *     pool at that slot; slot -1 (padding) writes nothing;
 *   - paged attention (same page, section 2, PAGED_ATTENTION bullet): a query
 *     at position p reads the keys 0..p of its own sequence, found through the
 *     sequence's block table, scores them with a dot product, takes a softmax
 *     and returns the softmax-weighted sum of the values; the causal length is
 *     position + 1 (section 1);
 *   - the sliding window (section 3, "Sliding-window layers"): with window W
 *     only positions p-W+1..p are read;
 *   - the ring (section 2, the bullet on sliding layers whose table is a
 *     ring; section 3, the windowed KV pool): the first ring_pages entries of
 *     the table are a ring of N = ring_pages * page_size slots, logical block
 *     b living on ring page b % ring_pages; slot i holds the position
 *     (L - 1 - i) mod N behind the row's last one, and is read when that age
 *     is less than the window and less than L;
 *   - the blockwise form (section 2, "Blockwise attention"): the same result
 *     folded over key blocks of 2,048 positions with a running max, a running
 *     sum and a running P.V;
 *   - the KV sizing closed form ("Serving Models", "Count KV heads and
 *     distinct stored tensors"): 2 * layers * H_kv * d_head * bytes per token;
 *   - the fp8 KV cache ("How serving works in Tlaloc", the FP8 KV cache
 *     paragraph of its quantisation section, after "Int8 weights (opt-in)"):
 *     pools of e4m3fn codes (1 sign bit, 4 exponent bits with bias 7, 3
 *     mantissa bits, no infinities, S.1111.111 is NaN) with no scale; the
 *     write clamps each value to +-448 (the largest finite code) and rounds
 *     it to the nearest code, ties to an even mantissa (the rounding the same
 *     section states for e4m3 weight codes); attention reads the codes'
 *     exact values;
 *   - int8 KV pools (same page: "What would make it faster" lists int8 KV
 *     pools as a next step without a format; the format is read from its
 *     "Int8 weights (opt-in)" paragraph, one f32 scale per output channel,
 *     max |W| / 127, codes rounded half to even): each (token, KV head) row
 *     of d values gets one scale s = max |x| / 127 and each value the code
 *     round-half-even(x / s), both computed in binary32; attention reads code
 *     x s exactly.
 *
 * Everything is the plain definition written out: widen each stored value
 * exactly to double, accumulate in double, in index order, one output at a
 * time.  The only parallelism is over independent outputs (OpenMP), which does
 * not change any output's arithmetic.
 *
 * Readings taken where the pages are silent:
 *   - pool layout [num_pages][page_size][H_kv][d], so slot s is page s/ps,
 *     offset s%ps;
 *   - query head h reads KV head h / (H_q / H_kv);
 *   - a query with causal length 0 (position -1, i.e. padding) outputs 0;
 *   - the softmax subtracts the running maximum before exponentiating.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1, OR_FP8 = 2, OR_INT8 = 3 };
enum { OR_OK = 0, OR_BAD_ARG = 1, OR_BAD_PAGE = 2, OR_NO_MEM = 3 };

/* Value of one e4m3fn code: (-1)^s 2^(e-7) (1 + m/8) for e > 0,
 * (-1)^s 2^-6 (m/8) for e = 0; e = 15 with m = 7 is NaN. */
static double fp8_value(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* The e4m3fn code nearest to x (ties to the even mantissa), clamped to
 * +-448; NaN gives the NaN code 0x7F.  The sign of zero is kept. */
static uint8_t fp8_code(double x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E; /* clamp (448 itself is a code) */
  int e;                               /* exponent of the code's binade */
  double steps;                        /* a in units of the binade's spacing */
  if (a < ldexp(1.0, -6)) {            /* subnormal codes: spacing 2^-9 */
    e = 0;
    steps = ldexp(a, 9);
  } else {
    int E;
    frexp(a, &E);                      /* a = f 2^E, f in [0.5, 1) */
    e = E - 1 + 7;                     /* biased exponent */
    steps = ldexp(a, 3 - (E - 1));     /* in [8, 16): 8 + mantissa */
  }
  double r = floor(steps);
  const double frac = steps - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  int m;
  if (e == 0) {
    m = (int)r; /* 0..8; 8 is the smallest normal code 0x08 */
    return sign | (uint8_t)m;
  }
  m = (int)r - 8; /* 0..8 */
  if (m == 8) {
    m = 0;
    e += 1;
  }
  if (e > 15 || (e == 15 && m == 7)) return sign | 0x7E; /* rounded past 448 */
  return sign | (uint8_t)((e << 3) | m);
}

/* Exact widening of one stored element to double.  bf16 is the upper half of
 * an IEEE binary32, so the widening is a 16-bit shift; fp8 codes widen to
 * their value. */
static double widen(const void* base, int64_t idx, int dtype) {
  if (dtype == OR_F32) return (double)((const float*)base)[idx];
  if (dtype == OR_FP8) return fp8_value(((const uint8_t*)base)[idx]);
  if (dtype == OR_INT8) return (double)((const int8_t*)base)[idx]; /* the code; x scale apart */
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int64_t elem_size(int dtype) {
  return dtype == OR_F32 ? 4 : (dtype == OR_FP8 || dtype == OR_INT8) ? 1 : 2;
}

/* The query of an fp8 or int8 cache is bf16. */
static int query_dtype(int kv_dtype) {
  return (kv_dtype == OR_FP8 || kv_dtype == OR_INT8) ? OR_BF16 : kv_dtype;
}

double oracle_fp8_value(int32_t code) { return fp8_value((uint8_t)code); }
int32_t oracle_fp8_code(double x) { return fp8_code(x); }

/* ---------------------------------------------------------------- write -- */

int oracle_kv_cache_write(const void* k_new, const void* v_new, void* k_cache,
                          void* v_cache, const int64_t* slot_mapping,
                          int64_t n_tokens, int64_t num_pages, int64_t page_size,
                          int64_t h_kv, int64_t d, int64_t elem_bytes) {
  if (n_tokens < 0 || num_pages <= 0 || page_size <= 0 || h_kv <= 0 || d <= 0 ||
      elem_bytes <= 0)
    return OR_BAD_ARG;
  const int64_t row_bytes = h_kv * d * elem_bytes; /* one token: all KV heads */
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue; /* padding: never written */
    if (slot < 0 || slot >= num_pages * page_size) return OR_BAD_PAGE;
    const int64_t page = slot / page_size;
    const int64_t offset = slot % page_size;
    const int64_t dst = (page * page_size + offset) * row_bytes;
    memcpy((char*)k_cache + dst, (const char*)k_new + t * row_bytes, (size_t)row_bytes);
    memcpy((char*)v_cache + dst, (const char*)v_new + t * row_bytes, (size_t)row_bytes);
  }
  return OR_OK;
}

/* The write into an fp8 pool: each element of the new rows (f32 or bf16) is
 * converted to its e4m3fn code (fp8_code); slot -1 writes nothing. */
int oracle_kv_cache_write_fp8(const void* k_new, const void* v_new, int32_t src_dtype,
                              uint8_t* k_cache, uint8_t* v_cache, const int64_t* slot_mapping,
                              int64_t n_tokens, int64_t num_pages, int64_t page_size,
                              int64_t h_kv, int64_t d) {
  if (n_tokens < 0 || num_pages <= 0 || page_size <= 0 || h_kv <= 0 || d <= 0 ||
      (src_dtype != OR_F32 && src_dtype != OR_BF16))
    return OR_BAD_ARG;
  const int64_t row = h_kv * d; /* elements of one token (all KV heads) */
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_pages * page_size) return OR_BAD_PAGE;
    for (int64_t e = 0; e < row; ++e) {
      k_cache[slot * row + e] = fp8_code(widen(k_new, t * row + e, src_dtype));
      v_cache[slot * row + e] = fp8_code(widen(v_new, t * row + e, src_dtype));
    }
  }
  return OR_OK;
}

/* The write into an int8 pool: each (token, KV head) row of d new values (f32
 * or bf16, widened exactly to binary32) gets the scale s = m / 127 with m the
 * largest magnitude of its finite values, and each finite value x the code
 * round-half-even(x / s), clamped to +-127; s and x / s are binary32 divisions.
 * A row with s = 0 (all zeros, or m so small that m / 127 underflows) writes
 * codes 0 and scale 0.  A non-finite value writes code 0 and is counted in
 * *n_bad.  Codes sit at the pool layout [num_pages][page_size][H_kv][d], the
 * scales at [num_pages][H_kv][page_size] (a page's scales of one head are
 * contiguous).  Slot -1 writes nothing. */
static void quantize_row_int8(const void* src, int64_t idx0, int src_dtype, int64_t d,
                              int8_t* codes, float* scale, int64_t* n_bad) {
  float m = 0.0f;
  for (int64_t e = 0; e < d; ++e) {
    const float x = (float)widen(src, idx0 + e, src_dtype);
    if (!isfinite(x)) {
      ++*n_bad;
      continue;
    }
    if (fabsf(x) > m) m = fabsf(x);
  }
  const float sc = m / 127.0f;
  for (int64_t e = 0; e < d; ++e) {
    const float x = (float)widen(src, idx0 + e, src_dtype);
    float r = 0.0f;
    if (isfinite(x) && sc > 0.0f) {
      r = rintf(x / sc); /* the default rounding mode: to nearest, ties to even */
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
    }
    codes[e] = (int8_t)r;
  }
  *scale = sc;
}

int oracle_kv_cache_write_int8(const void* k_new, const void* v_new, int32_t src_dtype,
                               int8_t* k_codes, int8_t* v_codes, float* k_scales,
                               float* v_scales, const int64_t* slot_mapping, int64_t n_tokens,
                               int64_t num_pages, int64_t page_size, int64_t h_kv, int64_t d,
                               int64_t* n_bad) {
  if (n_tokens < 0 || num_pages <= 0 || page_size <= 0 || h_kv <= 0 || d <= 0 ||
      (src_dtype != OR_F32 && src_dtype != OR_BF16))
    return OR_BAD_ARG;
  *n_bad = 0;
  const int64_t row = h_kv * d; /* elements of one token (all KV heads) */
  for (int64_t t = 0; t < n_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_pages * page_size) return OR_BAD_PAGE;
    const int64_t page = slot / page_size, offset = slot % page_size;
    for (int64_t g = 0; g < h_kv; ++g) {
      const int64_t si = (page * h_kv + g) * page_size + offset;
      quantize_row_int8(k_new, t * row + g * d, src_dtype, d, k_codes + slot * row + g * d,
                        k_scales + si, n_bad);
      quantize_row_int8(v_new, t * row + g * d, src_dtype, d, v_codes + slot * row + g * d,
                        v_scales + si, n_bad);
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------ attention -- */

typedef struct {
  const void* k_cache;
  const void* v_cache;
  int dtype;
  const int32_t* bt_row; /* this sequence's block table row */
  int32_t max_pages_per_seq;
  int32_t num_pages, page_size, h_kv, d;
  const float* k_scales; /* int8 pools: [num_pages][H_kv][page_size] */
  const float* v_scales;
} paged_seq;

/* Element e of the K (or V) row of logical position j, KV head g; *scale_idx
 * is the row's entry in an int8 pool's scales. */
static int kv_index(const paged_seq* s, int64_t j, int64_t g, int64_t* row_base,
                    int64_t* scale_idx) {
  const int64_t logical_block = j / s->page_size;
  if (logical_block >= s->max_pages_per_seq) return OR_BAD_PAGE;
  const int64_t page = s->bt_row[logical_block];
  if (page < 0 || page >= s->num_pages) return OR_BAD_PAGE;
  const int64_t offset = j % s->page_size;
  *row_base = ((page * s->page_size + offset) * s->h_kv + g) * s->d;
  *scale_idx = (page * s->h_kv + g) * s->page_size + offset;
  return OR_OK;
}

/* Stored element e of a row, exactly: the widened value, or for an int8 pool
 * code x scale (8 + 24 significant bits: exact in double). */
static double kv_value(const paged_seq* s, const void* pool, const float* scales,
                       int64_t base, int64_t e, int64_t scale_idx) {
  const double x = widen(pool, base + e, s->dtype);
  return s->dtype == OR_INT8 ? x * (double)scales[scale_idx] : x;
}

static double score(const paged_seq* s, const double* q, int64_t j, int64_t g,
                    double scale, int* err) {
  int64_t base, si;
  if (kv_index(s, j, g, &base, &si) != OR_OK) { *err = OR_BAD_PAGE; return 0.0; }
  double dot = 0.0;
  for (int64_t e = 0; e < s->d; ++e)
    dot += q[e] * kv_value(s, s->k_cache, s->k_scales, base, e, si);
  return scale * dot;
}

static void add_weighted_value(const paged_seq* s, int64_t j, int64_t g, double w,
                               double* acc, int* err) {
  int64_t base, si;
  if (kv_index(s, j, g, &base, &si) != OR_OK) { *err = OR_BAD_PAGE; return; }
  for (int64_t e = 0; e < s->d; ++e)
    acc[e] += w * kv_value(s, s->v_cache, s->v_scales, base, e, si);
}

/* One-pass form: scores of keys lo..p, softmax, weighted sum of values. */
static int attend_one_pass(const paged_seq* s, const double* q, int64_t lo, int64_t p,
                           int64_t g, double scale, double* out) {
  const int64_t d = s->d;
  for (int64_t e = 0; e < d; ++e) out[e] = 0.0;
  if (p < lo) return OR_OK; /* no live key: output 0 */
  const int64_t n = p - lo + 1;
  double* sc = (double*)malloc((size_t)n * sizeof(double));
  if (!sc) return OR_NO_MEM;
  int err = OR_OK;
  double m = -INFINITY;
  for (int64_t j = lo; j <= p; ++j) {
    sc[j - lo] = score(s, q, j, g, scale, &err);
    if (sc[j - lo] > m) m = sc[j - lo];
  }
  double l = 0.0;
  for (int64_t j = lo; j <= p; ++j) {
    const double w = exp(sc[j - lo] - m);
    l += w;
    add_weighted_value(s, j, g, w, out, &err);
  }
  for (int64_t e = 0; e < d; ++e) out[e] /= l;
  free(sc);
  return err;
}

/* Blockwise form: the keys are visited in blocks [kb*blk, (kb+1)*blk) for kb
 * from kb_first to kb_last, and each block is folded into a running max m, a
 * running sum l and a running P.V acc:
 *   m' = max(m, max_j s_j)
 *   l  = l * exp(m - m') + sum_j exp(s_j - m')
 *   acc = acc * exp(m - m') + sum_j exp(s_j - m') v_j
 * A block holding none of the row's keys lo..p is skipped.  out = acc / l. */
static int attend_blockwise(const paged_seq* s, const double* q, int64_t lo, int64_t p,
                            int64_t g, double scale, int64_t blk, int64_t kb_first,
                            int64_t kb_last, double* out) {
  const int64_t d = s->d;
  for (int64_t e = 0; e < d; ++e) out[e] = 0.0;
  if (p < lo) return OR_OK;
  double* sc = (double*)malloc((size_t)blk * sizeof(double));
  double* acc = (double*)calloc((size_t)d, sizeof(double));
  if (!sc || !acc) { free(sc); free(acc); return OR_NO_MEM; }
  int err = OR_OK;
  double m = -INFINITY, l = 0.0;
  for (int64_t kb = kb_first; kb <= kb_last; ++kb) {
    int64_t j0 = kb * blk, j1 = (kb + 1) * blk - 1;
    if (j0 < lo) j0 = lo;
    if (j1 > p) j1 = p;
    if (j1 < j0) continue; /* block fully masked for this row */
    double m_blk = -INFINITY;
    for (int64_t j = j0; j <= j1; ++j) {
      sc[j - j0] = score(s, q, j, g, scale, &err);
      if (sc[j - j0] > m_blk) m_blk = sc[j - j0];
    }
    const double m_new = m > m_blk ? m : m_blk;
    const double carry = exp(m - m_new); /* exp(-inf) = 0 on the first block */
    l *= carry;
    for (int64_t e = 0; e < d; ++e) acc[e] *= carry;
    for (int64_t j = j0; j <= j1; ++j) {
      const double w = exp(sc[j - j0] - m_new);
      l += w;
      add_weighted_value(s, j, g, w, acc, &err);
    }
    m = m_new;
  }
  for (int64_t e = 0; e < d; ++e) out[e] = acc[e] / l;
  free(sc);
  free(acc);
  return err;
}

/* Ring form: the N slots of the ring are visited in slot order; slot i holds
 * position last - ((last - i) mod N), where last is the row's last written
 * position, and is read when that position lies in lo..p (for a decode query,
 * p = last: the slot's age (last - i) mod N is below the window and below
 * L = last + 1).  One pass: scores, max, softmax, weighted sum of values.
 * Slot i is logical position i of the ring's table entries. */
static int attend_ring(const paged_seq* s, const double* q, int64_t lo, int64_t p,
                       int64_t last, int64_t n_slots, int64_t g, double scale, double* out) {
  const int64_t d = s->d;
  for (int64_t e = 0; e < d; ++e) out[e] = 0.0;
  if (p < lo) return OR_OK;
  double* sc = (double*)malloc((size_t)n_slots * sizeof(double));
  if (!sc) return OR_NO_MEM;
  int err = OR_OK;
  double m = -INFINITY;
  for (int64_t i = 0; i < n_slots; ++i) {
    const int64_t age = ((last - i) % n_slots + n_slots) % n_slots;
    const int64_t pos = last - age;
    if (pos < lo || pos > p) { sc[i] = -INFINITY; continue; }
    sc[i] = score(s, q, i, g, scale, &err);
    if (sc[i] > m) m = sc[i];
  }
  double l = 0.0;
  for (int64_t i = 0; i < n_slots; ++i) {
    if (sc[i] == -INFINITY) continue;
    const double w = exp(sc[i] - m);
    l += w;
    add_weighted_value(s, i, g, w, out, &err);
  }
  if (l > 0.0)
    for (int64_t e = 0; e < d; ++e) out[e] /= l;
  free(sc);
  return err;
}

static int64_t window_lo(int64_t p, int64_t window) {
  if (window <= 0) return 0;
  const int64_t lo = p - window + 1;
  return lo < 0 ? 0 : lo;
}

static void set_threads(int32_t n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Decode: one query token per sequence; sequence b has causal length
 * context_lens[b] (its query sits at position context_lens[b] - 1).
 * ring_pages > 0: the table's first ring_pages entries are the sequence's
 * ring (attend_ring); 0: full history.
 * Computes the sequences listed in seqs[0..n_seqs) into out[n_seqs][H_q][d]. */
static int decode_common(const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scales, const float* v_scales, int32_t dtype,
                         const int32_t* block_table, int32_t max_pages_per_seq,
                         const int32_t* context_lens, int32_t B, int32_t h_q, int32_t h_kv,
                         int32_t d, int32_t num_pages, int32_t page_size, int32_t window,
                         int32_t ring_pages, double scale, const int32_t* seqs,
                         int32_t n_seqs, double* out, int32_t n_threads) {
  if (B <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d <= 0 || page_size <= 0 ||
      num_pages <= 0 || max_pages_per_seq <= 0 ||
      (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_FP8 && dtype != OR_INT8) ||
      (dtype == OR_INT8 && (!k_scales || !v_scales)) || ring_pages < 0 ||
      ring_pages > max_pages_per_seq)
    return OR_BAD_ARG;
  for (int32_t i = 0; i < n_seqs; ++i)
    if (seqs[i] < 0 || seqs[i] >= B) return OR_BAD_ARG;
  const int64_t group = h_q / h_kv;
  int status = OR_OK;
  set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t item = 0; item < (int64_t)n_seqs * h_q; ++item) {
    const int64_t b = seqs[item / h_q], h = item % h_q, g = h / group;
    paged_seq s = {k_cache, v_cache, dtype, block_table + b * max_pages_per_seq,
                   max_pages_per_seq, num_pages, page_size, h_kv, d, k_scales, v_scales};
    double* qv = (double*)malloc((size_t)d * sizeof(double));
    double* o = out + item * d;
    if (!qv) { status = OR_NO_MEM; continue; }
    for (int64_t e = 0; e < d; ++e) qv[e] = widen(q, (b * h_q + h) * d + e, query_dtype(dtype));
    const int64_t p = (int64_t)context_lens[b] - 1;
    const int rc = ring_pages > 0
                       ? attend_ring(&s, qv, window_lo(p, window), p, p,
                                     (int64_t)ring_pages * page_size, g, scale, o)
                       : attend_one_pass(&s, qv, window_lo(p, window), p, g, scale, o);
    if (rc != OR_OK) status = rc;
    free(qv);
  }
  return status;
}

int oracle_paged_decode(const void* q, const void* k_cache, const void* v_cache,
                        int32_t dtype, const int32_t* block_table,
                        int32_t max_pages_per_seq, const int32_t* context_lens,
                        int32_t B, int32_t h_q, int32_t h_kv, int32_t d,
                        int32_t num_pages, int32_t page_size, int32_t window,
                        int32_t ring_pages, double scale, const int32_t* seqs, int32_t n_seqs,
                        double* out, int32_t n_threads) {
  if (dtype == OR_INT8) return OR_BAD_ARG; /* int8 pools come with their scales */
  return decode_common(q, k_cache, v_cache, NULL, NULL, dtype, block_table, max_pages_per_seq,
                       context_lens, B, h_q, h_kv, d, num_pages, page_size, window, ring_pages,
                       scale, seqs, n_seqs, out, n_threads);
}

/* Decode over int8 pools: codes k_codes / v_codes at the pool layout, scales
 * [num_pages][H_kv][page_size]; each element read as code x scale. */
int oracle_paged_decode_int8(const void* q, const int8_t* k_codes, const int8_t* v_codes,
                             const float* k_scales, const float* v_scales,
                             const int32_t* block_table, int32_t max_pages_per_seq,
                             const int32_t* context_lens, int32_t B, int32_t h_q, int32_t h_kv,
                             int32_t d, int32_t num_pages, int32_t page_size, int32_t window,
                             int32_t ring_pages, double scale, const int32_t* seqs,
                             int32_t n_seqs, double* out, int32_t n_threads) {
  return decode_common(q, k_codes, v_codes, k_scales, v_scales, OR_INT8, block_table,
                       max_pages_per_seq, context_lens, B, h_q, h_kv, d, num_pages, page_size,
                       window, ring_pages, scale, seqs, n_seqs, out, n_threads);
}

/* Prefill: q[B][T][H_q][d], positions[B][T] (-1 = padding).  Token (b,t) has
 * causal length positions[b][t] + 1 and reads its own row's block table.
 * blockwise = 0: one-pass form; otherwise the blockwise fold over key blocks of
 * key_block positions, visiting the call's block range from the first block
 * any row can see to the block holding the call's last position.
 * ring_pages > 0: the table's first ring_pages entries are the row's ring and
 * every token reads it in one pass (attend_ring), relative to the row's last
 * live position (blockwise is then ignored).
 * Computes the tokens listed (as b*T+t) in tokens[0..n_tokens) into
 * out[n_tokens][H_q][d]. */
static int prefill_common(const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scales, const float* v_scales, int32_t dtype,
                          const int32_t* block_table, int32_t max_pages_per_seq,
                          const int32_t* positions, int32_t B, int32_t T, int32_t h_q,
                          int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size,
                          int32_t window, int32_t ring_pages, double scale, int32_t blockwise,
                          int32_t key_block, const int64_t* tokens, int64_t n_tokens,
                          double* out, int32_t n_threads) {
  if (B <= 0 || T <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d <= 0 ||
      page_size <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 ||
      (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_FP8 && dtype != OR_INT8) ||
      (dtype == OR_INT8 && (!k_scales || !v_scales)) ||
      (blockwise && key_block <= 0) || ring_pages < 0 || ring_pages > max_pages_per_seq)
    return OR_BAD_ARG;
  for (int64_t i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= (int64_t)B * T) return OR_BAD_ARG;
  /* The call's block range, over every live token of the call. */
  int64_t kb_first = INT64_MAX, kb_last = -1;
  for (int64_t i = 0; i < (int64_t)B * T; ++i) {
    const int64_t p = positions[i];
    if (p < 0) continue;
    const int64_t lo = window_lo(p, window);
    if (blockwise) {
      if (lo / key_block < kb_first) kb_first = lo / key_block;
      if (p / key_block > kb_last) kb_last = p / key_block;
    }
  }
  const int64_t group = h_q / h_kv;
  int status = OR_OK;
  set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t item = 0; item < n_tokens * h_q; ++item) {
    const int64_t bt_idx = tokens[item / h_q], h = item % h_q, g = h / group;
    const int64_t b = bt_idx / T;
    paged_seq s = {k_cache, v_cache, dtype, block_table + b * max_pages_per_seq,
                   max_pages_per_seq, num_pages, page_size, h_kv, d, k_scales, v_scales};
    double* qv = (double*)malloc((size_t)d * sizeof(double));
    double* o = out + item * d;
    if (!qv) { status = OR_NO_MEM; continue; }
    for (int64_t e = 0; e < d; ++e)
      qv[e] = widen(q, (bt_idx * h_q + h) * d + e, query_dtype(dtype));
    const int64_t p = positions[bt_idx];
    const int64_t lo = window_lo(p, window);
    int rc;
    if (ring_pages > 0) {
      int64_t last = -1; /* the row's last live position */
      for (int64_t t = 0; t < T; ++t)
        if (positions[b * T + t] > last) last = positions[b * T + t];
      rc = attend_ring(&s, qv, lo, p, last, (int64_t)ring_pages * page_size, g, scale, o);
    } else if (!blockwise || p < 0)
      rc = attend_one_pass(&s, qv, lo, p, g, scale, o);
    else
      rc = attend_blockwise(&s, qv, lo, p, g, scale, key_block, kb_first, kb_last, o);
    if (rc != OR_OK) status = rc;
    free(qv);
  }
  return status;
}

int oracle_paged_prefill(const void* q, const void* k_cache, const void* v_cache,
                         int32_t dtype, const int32_t* block_table,
                         int32_t max_pages_per_seq, const int32_t* positions, int32_t B,
                         int32_t T, int32_t h_q, int32_t h_kv, int32_t d,
                         int32_t num_pages, int32_t page_size, int32_t window,
                         int32_t ring_pages, double scale, int32_t blockwise, int32_t key_block,
                         const int64_t* tokens, int64_t n_tokens, double* out,
                         int32_t n_threads) {
  if (dtype == OR_INT8) return OR_BAD_ARG; /* int8 pools come with their scales */
  return prefill_common(q, k_cache, v_cache, NULL, NULL, dtype, block_table, max_pages_per_seq,
                        positions, B, T, h_q, h_kv, d, num_pages, page_size, window, ring_pages,
                        scale, blockwise, key_block, tokens, n_tokens, out, n_threads);
}

/* Prefill over int8 pools (codes at the pool layout, scales
 * [num_pages][H_kv][page_size]); each element read as code x scale, the rest
 * as oracle_paged_prefill. */
int oracle_paged_prefill_int8(const void* q, const int8_t* k_codes, const int8_t* v_codes,
                              const float* k_scales, const float* v_scales,
                              const int32_t* block_table, int32_t max_pages_per_seq,
                              const int32_t* positions, int32_t B, int32_t T, int32_t h_q,
                              int32_t h_kv, int32_t d, int32_t num_pages, int32_t page_size,
                              int32_t window, int32_t ring_pages, double scale,
                              int32_t blockwise, int32_t key_block, const int64_t* tokens,
                              int64_t n_tokens, double* out, int32_t n_threads) {
  return prefill_common(q, k_codes, v_codes, k_scales, v_scales, OR_INT8, block_table,
                        max_pages_per_seq, positions, B, T, h_q, h_kv, d, num_pages, page_size,
                        window, ring_pages, scale, blockwise, key_block, tokens, n_tokens, out,
                        n_threads);
}

/* ---------------------------------------------------------------- sizing -- */

/* Bytes of K and V one token of one sequence occupies: 2 * L * H_kv * d * q
 * ("Serving Models", "Count KV heads and distinct stored tensors"). */
int64_t oracle_kv_bytes_per_token(int64_t layers, int64_t h_kv, int64_t d_head,
                                  int64_t bytes_per_elem) {
  return 2 * layers * h_kv * d_head * bytes_per_elem;
}

int64_t oracle_elem_size(int32_t dtype) { return elem_size(dtype); }

/* Ring pages a windowed pool needs so that a call writing up to `chunk` tokens
 * fits past the window (section 3 and section 4 of "How serving works in
 * Tlaloc"): a call of n tokens at p0 needs min(p0, W-1) + n positions at once,
 * so the ring is ceil((W - 1 + chunk) / page_size) pages; a decode step
 * (chunk = 1) needs ceil(W / page_size). */
int64_t oracle_ring_pages(int64_t window, int64_t chunk, int64_t page_size) {
  if (window <= 0 || chunk <= 0 || page_size <= 0) return -1;
  return (window - 1 + chunk + page_size - 1) / page_size;
}
