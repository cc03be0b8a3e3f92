/*
 * CPU fp64 oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The
 * product (libpa and its Python binding) never calls into it; the two share
 * no code.
 *
 * What it computes.  The method ("paged_attention_v2", project_6 commit
 * 96f4baf "Dockerfile", section "Implementation") reaches exact softmax
 * attention over each sequence's cached keys and values: the per-partition
 * partials of Phase 1 combined by the log-sum-exp rescale of Phase 2 are
 * algebraically one softmax over all tokens.  So the main entry point,
 * pa_oracle_attention, is that plain definition written out, with no
 * partitioning:
 *
 *   kvh       = h / (H / Hkv)                 (contiguous GQA groups)
 *   K_t, V_t  = cache[block_tables[s][t / bs]][kvh][t % bs][:]
 *   logit_t   = scale * sum_d q[s][h][d] * K_t[d]          t in [0, L_s)
 *   out[s][h] = sum_t softmax(logit)_t * V_t
 *
 * The softmax subtracts the maximum logit before exponentiating (the usual
 * definition; it changes nothing but overflow).  L_s = 0 gives zeros.
 *
 * pa_oracle_partials and pa_oracle_combine are the method's own two phases,
 * written from the same commit note's "Phase 1: Per-partition attention" and
 * "Phase 2: Cross-partition reduction (log-sum-exp)", in that order:
 *   Phase 1, for partition p = tokens [p*P, min((p+1)*P, L)):
 *     max_logits[p] = max_t logit_t
 *     exp_sums[p]   = sum_t exp(logit_t - max_logits[p])
 *     tmp_out[p]    = sum_t exp(logit_t - max_logits[p]) * V_t / exp_sums[p]
 *   Phase 2:
 *     global_max = max_p max_logits[p]
 *     rescale_p  = exp(max_logits[p] - global_max) * exp_sums[p]
 *     out        = sum_p (rescale_p / sum_p' rescale_p') * tmp_out[p]
 * They exist to pin the GPU's two phases separately and to test that the
 * combine equals the unpartitioned definition.
 *
 * Layouts (all row-major, contiguous):
 *   q, out           [B][H][D]
 *   k_cache, v_cache [num_blocks][Hkv][bs][D]
 *   block_tables     int32 [B][max_blocks]
 *   seq_lens         int32 [B]
 *   max_logits, exp_sums [B][H][max_parts]; tmp_out [B][H][max_parts][D]
 * Element types of q / k_cache / v_cache: f64, f32, bf16 or f16 (one code for
 * all three).  Each element is widened to double exactly before any
 * arithmetic, so the oracle consumes exactly the values the GPU sees.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2, ORC_F16 = 3 };

/* bfloat16 is the top half of an IEEE binary32: shift the 16 bits up. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Normal: (1 + f/1024) * 2^(e-15); subnormal: (f/1024) * 2^-14. */
static double f16_bits_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 10) & 0x1f;
  int f = b & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* f/1024 * 2^-14 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp(1024.0 + (double)f, e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -v : v;
}

static double load_elem(const void *base, size_t idx, int dtype) {
  switch (dtype) {
  case ORC_F64: return ((const double *)base)[idx];
  case ORC_F32: return (double)((const float *)base)[idx];
  case ORC_BF16: return bf16_bits_to_double(((const uint16_t *)base)[idx]);
  case ORC_F16: return f16_bits_to_double(((const uint16_t *)base)[idx]);
  default: return NAN;
  }
}

/* Element-wise widening, exposed so that tests can pin the decoders against
 * independent library conversions over every bit pattern. */
void pa_oracle_widen(double *dst, const void *src, int dtype, size_t n) {
  for (size_t i = 0; i < n; ++i) dst[i] = load_elem(src, i, dtype);
}

/* Offset of element d of token t of KV head kvh for sequence s. */
static size_t kv_index(const int32_t *block_tables, int s, int t, int kvh,
                       int d, int Hkv, int D, int bs, int max_blocks) {
  int64_t blk = block_tables[(size_t)s * max_blocks + t / bs];
  int off = t % bs;
  return (((size_t)blk * Hkv + kvh) * bs + off) * D + d;
}

static double logit_of(const void *q, const void *kc, int dtype,
                       const int32_t *bt, int s, int h, int t, int kvh, int H,
                       int Hkv, int D, int bs, int max_blocks, double scale) {
  double dot = 0.0;
  for (int d = 0; d < D; ++d)
    dot += load_elem(q, ((size_t)s * H + h) * D + d, dtype) *
           load_elem(kc, kv_index(bt, s, t, kvh, d, Hkv, D, bs, max_blocks), dtype);
  return scale * dot;
}

/* Softmax attention of query head h of sequence s over tokens [t0, t1).
 * Writes the normalised weighted sum to o[0..D), returns the max logit in
 * *m_out and the sum of exp(logit - max) in *s_out.  Empty range: o = 0,
 * *m_out = -inf, *s_out = 0. */
static void attend_range(double *o, double *m_out, double *s_out,
                         const void *q, const void *kc, const void *vc,
                         int dtype, const int32_t *bt, int s, int h, int t0,
                         int t1, int H, int Hkv, int D, int bs, int max_blocks,
                         double scale, double *logits) {
  int G = H / Hkv;
  int kvh = h / G;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (t1 <= t0) {
    *m_out = -INFINITY;
    *s_out = 0.0;
    return;
  }
  double m = -INFINITY;
  for (int t = t0; t < t1; ++t) {
    logits[t - t0] = logit_of(q, kc, dtype, bt, s, h, t, kvh, H, Hkv, D, bs,
                              max_blocks, scale);
    if (logits[t - t0] > m) m = logits[t - t0];
  }
  double sum = 0.0;
  for (int t = t0; t < t1; ++t) {
    double w = exp(logits[t - t0] - m);
    sum += w;
    for (int d = 0; d < D; ++d)
      o[d] += w * load_elem(vc, kv_index(bt, s, t, kvh, d, Hkv, D, bs, max_blocks), dtype);
  }
  for (int d = 0; d < D; ++d) o[d] /= sum;
  *m_out = m;
  *s_out = sum;
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

int pa_oracle_max_threads(void) { return set_threads(0); }

/* The plain definition: out[s][h][:] for every (s, h).  `logit_scratch` must
 * hold nthreads_used * max_seq_len doubles (see pa_oracle_max_threads). */
void pa_oracle_attention(double *out, const void *q, const void *k_cache,
                         const void *v_cache, int dtype,
                         const int32_t *block_tables, const int32_t *seq_lens,
                         int B, int H, int Hkv, int D, int bs, int max_blocks,
                         double scale, int nthreads, double *logit_scratch,
                         int max_seq_len) {
  set_threads(nthreads);
  long long n = (long long)B * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long i = 0; i < n; ++i) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    int s = (int)(i / H), h = (int)(i % H);
    double m, sum;
    attend_range(out + (size_t)i * D, &m, &sum, q, k_cache, v_cache, dtype,
                 block_tables, s, h, 0, seq_lens[s], H, Hkv, D, bs, max_blocks,
                 scale, logit_scratch + (size_t)tid * max_seq_len);
  }
}

/* The same definition on a list of (s, h) pairs only: out[i][:] for pair i.
 * Used to sample outputs of workloads too large to run whole. */
void pa_oracle_attention_pairs(double *out, const int32_t *pairs, int npairs,
                               const void *q, const void *k_cache,
                               const void *v_cache, int dtype,
                               const int32_t *block_tables,
                               const int32_t *seq_lens, int B, int H, int Hkv,
                               int D, int bs, int max_blocks, double scale,
                               int nthreads, double *logit_scratch,
                               int max_seq_len) {
  (void)B;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < npairs; ++i) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    int s = pairs[2 * i], h = pairs[2 * i + 1];
    double m, sum;
    attend_range(out + (size_t)i * D, &m, &sum, q, k_cache, v_cache, dtype,
                 block_tables, s, h, 0, seq_lens[s], H, Hkv, D, bs, max_blocks,
                 scale, logit_scratch + (size_t)tid * max_seq_len);
  }
}

/* Phase 1: per-partition max logit, exp-sum and normalised weighted V sum.
 * Partitions p >= ceil(L_s / P) are left untouched. */
void pa_oracle_partials(double *max_logits, double *exp_sums, double *tmp_out,
                        const void *q, const void *k_cache, const void *v_cache,
                        int dtype, const int32_t *block_tables,
                        const int32_t *seq_lens, int B, int H, int Hkv, int D,
                        int bs, int max_blocks, double scale, int P,
                        int max_parts, int nthreads, double *logit_scratch) {
  set_threads(nthreads);
  long long n = (long long)B * H * max_parts;
#pragma omp parallel for schedule(dynamic, 4)
  for (long long i = 0; i < n; ++i) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    int p = (int)(i % max_parts);
    long long sh = i / max_parts;
    int s = (int)(sh / H), h = (int)(sh % H);
    int L = seq_lens[s];
    int t0 = p * P;
    if (t0 >= L) continue;
    int t1 = t0 + P < L ? t0 + P : L;
    attend_range(tmp_out + (size_t)i * D, &max_logits[i], &exp_sums[i], q,
                 k_cache, v_cache, dtype, block_tables, s, h, t0, t1, H, Hkv,
                 D, bs, max_blocks, scale, logit_scratch + (size_t)tid * P);
  }
}

/* Phase 2: log-sum-exp combine of the partials of each (s, h) over its
 * num_parts[s] partitions.  num_parts[s] = 0 gives zeros. */
void pa_oracle_combine(double *out, const double *max_logits,
                       const double *exp_sums, const double *tmp_out,
                       const int32_t *num_parts, int B, int H, int D,
                       int max_parts) {
  for (long long sh = 0; sh < (long long)B * H; ++sh) {
    int s = (int)(sh / H);
    int np = num_parts[s];
    const double *ml = max_logits + sh * max_parts;
    const double *es = exp_sums + sh * max_parts;
    const double *to = tmp_out + sh * max_parts * D;
    double *o = out + sh * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (np <= 0) continue;
    double gmax = -INFINITY;
    for (int p = 0; p < np; ++p)
      if (ml[p] > gmax) gmax = ml[p];
    double total = 0.0;
    for (int p = 0; p < np; ++p) total += exp(ml[p] - gmax) * es[p];
    for (int p = 0; p < np; ++p) {
      double w = exp(ml[p] - gmax) * es[p] / total;
      for (int d = 0; d < D; ++d) o[d] += w * to[(size_t)p * D + d];
    }
  }
}

/* Multi-token queries over the paged cache: the query chunk of a sequence is
 * its last few tokens, all of them already in the cache.  The prefill patch
 * of project_6 (optimizations/prefix_prefill_patch.py, module docstring)
 * tunes a kernel that runs attention for blocks of query positions over a
 * paged prefix; the pages give no formula for it, so this is the plain
 * causal reading:
 *
 *   sequence s holds L = seq_lens[s] tokens in the cache; its chunk is the
 *   last n = q_start[s+1] - q_start[s] of them (1 <= n <= L), rows
 *   q_start[s] .. q_start[s+1]-1 of q and out ([rows][H][D]);
 *   chunk token i (cache position L - n + i) attends to cache tokens
 *   [0, L - n + i]:
 *     out[q_start[s] + i][h] = sum_{t <= L-n+i} softmax_t(scale q.K_t) V_t
 *
 * With n = 1 for every sequence this is pa_oracle_attention.  A sequence
 * with n = 0 has no rows; n > L is not a valid input (its rows are left at
 * zero).  Written out here on its own, not through attend_range, so that the
 * two definitions can be checked against each other. */
void pa_oracle_query_chunks(double *out, const void *q, const void *k_cache,
                            const void *v_cache, int dtype,
                            const int32_t *block_tables,
                            const int32_t *seq_lens, const int32_t *q_start,
                            int B, int H, int Hkv, int D, int bs,
                            int max_blocks, double scale, int nthreads,
                            double *logit_scratch, int max_seq_len) {
  set_threads(nthreads);
  const int G = H / Hkv;
  const long long rows = B > 0 ? q_start[B] : 0;
  const long long n_out = rows * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long i = 0; i < n_out; ++i) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double *lg = logit_scratch + (size_t)tid * max_seq_len;
    const long long row = i / H;
    const int h = (int)(i % H), kvh = h / G;
    int s = 0;
    while (s + 1 < B && q_start[s + 1] <= row) ++s;  /* the row's sequence */
    const int L = seq_lens[s], n = q_start[s + 1] - q_start[s];
    const int pos = L - n + (int)(row - q_start[s]);  /* last visible token */
    double *o = out + (size_t)i * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (n > L || pos < 0) continue;
    double m = -INFINITY;
    for (int t = 0; t <= pos; ++t) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += load_elem(q, (size_t)i * D + d, dtype) *
               load_elem(k_cache, kv_index(block_tables, s, t, kvh, d, Hkv, D, bs, max_blocks),
                         dtype);
      lg[t] = scale * dot;
      if (lg[t] > m) m = lg[t];
    }
    double sum = 0.0;
    for (int t = 0; t <= pos; ++t) {
      const double w = exp(lg[t] - m);
      sum += w;
      for (int d = 0; d < D; ++d)
        o[d] += w * load_elem(v_cache, kv_index(block_tables, s, t, kvh, d, Hkv, D, bs, max_blocks),
                              dtype);
    }
    for (int d = 0; d < D; ++d) o[d] = o[d] / sum;
  }
}
