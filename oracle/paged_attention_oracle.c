/*
 * FP64 CPU oracle for batched decode attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the timed CPU
 * baseline can compare the CUDA library against a plain, slow, obviously
 * correct evaluation of what the method computes. It shares no code, header,
 * table or constant with the CUDA library.
 *
 * Sources (the pages this follows):
 *  - "flashinfer.cake_fmha" API page: the paged decode contract
 *    (query, kv_cache, block_tables, seq_lens, max_kv_len) and the
 *    "optimized FP8 decode" paragraph (HND pages, one K/V page table).
 *  - PR #4557 "feat(cake_mla): add generated Blackwell TRT-LLM MLA decode
 *    backend", review thread "Exclusive causal bound drops the newest key":
 *    query row i of a request keeps keys 0 .. seq_len - q_len + i inclusive;
 *    review thread "Hoist the KV gather": the test reference gathers the
 *    request's rows through the page table and slices [: right + 1].
 *  - PR #5952 (fused QK RMSNorm + RoPE + paged KV append), summary: NHD pages
 *    [num_pages, page_size, Hkv, head_dim] addressed through a dense
 *    [B, max_pages] table; commit #5956 "Contract": seq_lens is the total
 *    length after the append, and K/V are stored as x / k_scale, x / v_scale
 *    in round-to-nearest saturating E4M3.
 *  - PR #5552 (Kimi-K3 FP8 latent MLA): latent 512 + 64 rope channels, so an
 *    MLA key is the whole 576-wide cached row and its value the first 512.
 *
 * Plain reading taken where the pages are silent:
 *  - HND pages are [num_pages, Hkv, page_size, head_dim] (the name read like
 *    NHD's).
 *  - LSE is the natural logarithm; a row with no visible key gives out = 0,
 *    lse = -inf.
 *  - E4M3 is OCP E4M3FN: bias 7, no infinities, S.1111.111 is NaN.
 *
 * Method, written without tiling, online softmax or splits: for each request
 * b, query row i and query head h, gather the visible keys through the page
 * table, compute every logit, take the maximum, then a second pass forms the
 * weights, their sum and the weighted sum of values, all in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Mutation switches: the pin tests rebuild this file with one of these
 * defined to show that a plausible mistake fails at least one pin.       */
#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0
#endif

enum { ORACLE_NHD = 0, ORACLE_HND = 1 };
enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1 };

enum {
  ORACLE_OK = 0,
  ORACLE_BAD_ARG = 1,
  ORACLE_BAD_QLEN = 2,   /* q_len > seq_len: the new tokens must be cached */
  ORACLE_BAD_PAGE = 3,   /* a referenced page id lies outside the pool     */
};

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits. Exponent
 * field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities.   */
double oracle_e4m3_to_double(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int expo = (byte >> 3) & 0xF;
  int mant = byte & 0x7;
  double mag;
  if (expo == 0xF && mant == 0x7) return NAN;
#if ORACLE_MUTATION == 5
  /* planted mistake: wrong exponent bias */
  if (expo == 0) mag = ldexp((double)mant / 8.0, -7);
  else mag = ldexp(1.0 + (double)mant / 8.0, expo - 8);
#else
  if (expo == 0) mag = ldexp((double)mant / 8.0, -6);
  else mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
#endif
  return sign ? -mag : mag;
}

static double load_elem(const void* pool, int dtype, int64_t idx) {
  if (dtype == ORACLE_BF16) return oracle_bf16_to_double(((const uint16_t*)pool)[idx]);
  return oracle_e4m3_to_double(((const uint8_t*)pool)[idx]);
}

/* Element offset of (page, slot, kv head, channel 0) in a pool. */
static int64_t row_offset(int layout, int64_t page, int64_t slot, int64_t g,
                          int64_t num_kv_heads, int64_t page_size,
                          int64_t page_stride, int64_t row_stride) {
#if ORACLE_MUTATION == 3
  /* planted mistake: NHD and HND swapped */
  layout = 1 - layout;
#endif
  if (layout == ORACLE_NHD) return page * page_stride + (slot * num_kv_heads + g) * row_stride;
  return page * page_stride + (g * page_size + slot) * row_stride;
}

/*
 * Paged GQA decode (also MHA when Hq == Hkv and MQA when Hkv == 1).
 *
 *  q            [total_q, num_q_heads, head_dim_qk] bf16 bits; request b
 *               owns rows q_indptr[b] .. q_indptr[b+1]-1
 *  k_pool/v_pool element type kv_dtype (bf16 bits or e4m3 bytes); page p,
 *               slot s, kv head g starts at row_offset(...)
 *  block_tables [batch, max_pages_per_seq]; token t of request b lives in
 *               page block_tables[b*max_pages_per_seq + t/page_size],
 *               slot t % page_size
 *  seq_lens     [batch] total cached length including the q_len new tokens
 *  q_indptr     [batch+1], or NULL for one query row per request
 *  kv_lo/kv_hi  keep only keys with kv_lo <= t < kv_hi (kv_hi < 0: no upper
 *               restriction); used to evaluate one split of the key range
 *  out          [total_q, num_q_heads, head_dim_v] double
 *  lse          [total_q, num_q_heads] double (natural log)
 *
 * Logit: sm_scale * sum_d q_d * (k_d * k_scale); value: v_d * v_scale
 * (K/V stored as x / scale). For bf16 pools pass k_scale = v_scale = 1.
 * sinks        [num_q_heads] or NULL: attention sinks, one logit per query
 *              head added to the softmax denominator with no value (the
 *              pages' MLA call takes `sinks`): out = sum_t e^s_t v_t /
 *              (sum_t e^s_t + e^sink), lse = log of that denominator
 */
int oracle_paged_decode(int batch, int num_q_heads, int num_kv_heads,
                        int head_dim_qk, int head_dim_v, int page_size,
                        int num_pages, int max_pages_per_seq, int layout,
                        int kv_dtype, const uint16_t* q, const void* k_pool,
                        const void* v_pool, int64_t k_page_stride,
                        int64_t v_page_stride, int64_t k_row_stride,
                        int64_t v_row_stride, const int32_t* block_tables,
                        const int32_t* seq_lens, const int32_t* q_indptr,
                        double sm_scale, double k_scale, double v_scale,
                        const double* sinks, int64_t kv_lo, int64_t kv_hi, double* out,
                        double* lse, int num_threads) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim_qk <= 0 ||
      head_dim_v <= 0 || page_size <= 0 || num_q_heads % num_kv_heads != 0)
    return ORACLE_BAD_ARG;
  const int group = num_q_heads / num_kv_heads;
  int64_t total_q = q_indptr ? q_indptr[batch] : batch;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t qlen = q_indptr ? (int64_t)q_indptr[b + 1] - q_indptr[b] : 1;
    if (qlen < 0 || seq_lens[b] < 0) return ORACLE_BAD_ARG;
    if (qlen > seq_lens[b]) return ORACLE_BAD_QLEN;
    if ((int64_t)seq_lens[b] > (int64_t)max_pages_per_seq * page_size) return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < seq_lens[b]; t += page_size) {
      int32_t p = block_tables[(int64_t)b * max_pages_per_seq + t / page_size];
      if (p < 0 || p >= num_pages) return ORACLE_BAD_PAGE;
    }
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  }
  if (total_q == 0) return ORACLE_OK;

#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double* logit = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)head_dim_v);
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim_qk);
    if (!logit || !acc || !qd) {
#pragma omp atomic write
      status = ORACLE_BAD_ARG;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t work = 0; work < (int64_t)batch * num_q_heads; ++work) {
        int b = (int)(work / num_q_heads);
        int h = (int)(work % num_q_heads);
#if ORACLE_MUTATION == 2
        int g = h % num_kv_heads; /* planted mistake: interleaved head map */
#else
        int g = h / group;
#endif
        int64_t q0 = q_indptr ? q_indptr[b] : b;
        int64_t qlen = q_indptr ? (int64_t)q_indptr[b + 1] - q_indptr[b] : 1;
        int64_t L = seq_lens[b];
        for (int64_t i = 0; i < qlen; ++i) {
          int64_t row = q0 + i;
          const uint16_t* qrow = q + (row * num_q_heads + h) * (int64_t)head_dim_qk;
          for (int d = 0; d < head_dim_qk; ++d) qd[d] = oracle_bf16_to_double(qrow[d]);
          /* absolute position of this query token; keys 0..pos are visible */
          int64_t pos = L - qlen + i;
#if ORACLE_MUTATION == 1
          int64_t t_end = pos; /* planted mistake: exclusive causal bound */
#else
          int64_t t_end = pos + 1;
#endif
          if (kv_hi >= 0 && kv_hi < t_end) t_end = kv_hi;
          int64_t t_begin = kv_lo > 0 ? kv_lo : 0;
          double* o = out + (row * num_q_heads + h) * (int64_t)head_dim_v;
          const double sink = sinks ? sinks[h] : -INFINITY;
          if (t_end <= t_begin) {
            for (int d = 0; d < head_dim_v; ++d) o[d] = 0.0;
            lse[row * num_q_heads + h] = sink;
            continue;
          }
          /* pass 1: logits and their maximum */
          double m = -INFINITY;
          for (int64_t t = t_begin; t < t_end; ++t) {
            int64_t page = block_tables[(int64_t)b * max_pages_per_seq + t / page_size];
            int64_t slot = t % page_size;
            int64_t base = row_offset(layout, page, slot, g, num_kv_heads, page_size,
                                      k_page_stride, k_row_stride);
            double dot = 0.0;
            for (int d = 0; d < head_dim_qk; ++d)
              dot += qd[d] * (load_elem(k_pool, kv_dtype, base + d) * k_scale);
#if ORACLE_MUTATION == 4
            double s = dot; /* planted mistake: scale dropped */
#else
            double s = sm_scale * dot;
#endif
            logit[t - t_begin] = s;
            if (s > m) m = s;
          }
          /* a sink is one more term of the denominator, with no value */
          if (sink > m) m = sink;
          /* pass 2: weights, their sum and the weighted sum of values */
#if ORACLE_MUTATION == 8
          double l = 0.0; /* planted mistake: the sink left out of the denominator */
#else
          double l = sinks ? exp(sink - m) : 0.0;
#endif
          for (int d = 0; d < head_dim_v; ++d) acc[d] = 0.0;
          for (int64_t t = t_begin; t < t_end; ++t) {
            int64_t page = block_tables[(int64_t)b * max_pages_per_seq + t / page_size];
            int64_t slot = t % page_size;
            int64_t base = row_offset(layout, page, slot, g, num_kv_heads, page_size,
                                      v_page_stride, v_row_stride);
            double w = exp(logit[t - t_begin] - m);
            l += w;
            for (int d = 0; d < head_dim_v; ++d)
              acc[d] += w * (load_elem(v_pool, kv_dtype, base + d) * v_scale);
          }
          for (int d = 0; d < head_dim_v; ++d) o[d] = acc[d] / l;
          lse[row * num_q_heads + h] = m + log(l);
        }
      }
    }
    free(logit);
    free(acc);
    free(qd);
  }
  return status;
}

/*
 * MLA decode: every query head attends over one latent KV head. The cache
 * row of token t is kv[page][slot][0:head_dim_qk] (latent then rope
 * channels); the key is the whole row and the value its first head_dim_v
 * channels.
 *
 *  q        [total_q, num_heads, head_dim_qk] bf16 bits, or E4M3 codes
 *  kv_pool  [num_pages, page_size, head_dim_qk] bf16 bits, or E4M3 codes
 *  kv_dtype ORACLE_E4M3: query and pool are E4M3 codes with values
 *           code * q_scale and code * kv_scale (PR #5552, FP8 query and
 *           FP8 latent cache); ORACLE_BF16: pass scales of 1
 *  out      [total_q, num_heads, head_dim_v] double; lse [total_q, num_heads]
 */
int oracle_mla_decode(int batch, int num_heads, int head_dim_qk, int head_dim_v,
                      int page_size, int num_pages, int max_pages_per_seq, int kv_dtype,
                      double q_scale, double kv_scale, const void* q, const void* kv_pool,
                      const int32_t* block_tables, const int32_t* seq_lens,
                      const int32_t* q_indptr, double sm_scale, const double* sinks,
                      double* out, double* lse, int num_threads) {
  if (batch < 0 || num_heads <= 0 || head_dim_qk <= 0 || head_dim_v <= 0 ||
      head_dim_v > head_dim_qk || page_size <= 0)
    return ORACLE_BAD_ARG;
  int64_t total_q = q_indptr ? q_indptr[batch] : batch;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t qlen = q_indptr ? (int64_t)q_indptr[b + 1] - q_indptr[b] : 1;
    if (qlen < 0 || seq_lens[b] < 0) return ORACLE_BAD_ARG;
    if (qlen > seq_lens[b]) return ORACLE_BAD_QLEN;
    if ((int64_t)seq_lens[b] > (int64_t)max_pages_per_seq * page_size) return ORACLE_BAD_ARG;
    for (int64_t t = 0; t < seq_lens[b]; t += page_size) {
      int32_t p = block_tables[(int64_t)b * max_pages_per_seq + t / page_size];
      if (p < 0 || p >= num_pages) return ORACLE_BAD_PAGE;
    }
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  }
  if (total_q == 0) return ORACLE_OK;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
  int status = ORACLE_OK;
#pragma omp parallel
  {
    double* logit = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)head_dim_v);
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim_qk);
    if (!logit || !acc || !qd) {
#pragma omp atomic write
      status = ORACLE_BAD_ARG;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t row = 0; row < total_q; ++row) {
        /* the request that owns this query row */
        int b = 0;
        if (q_indptr) {
          while (b + 1 < batch && q_indptr[b + 1] <= row) ++b;
        } else {
          b = (int)row;
        }
        int64_t qlen = q_indptr ? (int64_t)q_indptr[b + 1] - q_indptr[b] : 1;
        int64_t i = q_indptr ? row - q_indptr[b] : 0;
        int64_t L = seq_lens[b];
        int64_t t_end = L - qlen + i + 1;
        for (int h = 0; h < num_heads; ++h) {
          const int64_t qbase = (row * num_heads + h) * (int64_t)head_dim_qk;
          for (int d = 0; d < head_dim_qk; ++d) qd[d] = load_elem(q, kv_dtype, qbase + d) * q_scale;
          double m = -INFINITY;
          for (int64_t t = 0; t < t_end; ++t) {
            int64_t page = block_tables[(int64_t)b * max_pages_per_seq + t / page_size];
            const int64_t kbase = (page * page_size + t % page_size) * (int64_t)head_dim_qk;
            double dot = 0.0;
            for (int d = 0; d < head_dim_qk; ++d) dot += qd[d] * (load_elem(kv_pool, kv_dtype, kbase + d) * kv_scale);
            logit[t] = sm_scale * dot;
            if (logit[t] > m) m = logit[t];
          }
          double* o = out + (row * num_heads + h) * (int64_t)head_dim_v;
          const double sink = sinks ? sinks[h] : -INFINITY;
          if (t_end <= 0) {
            for (int d = 0; d < head_dim_v; ++d) o[d] = 0.0;
            lse[row * num_heads + h] = sink;
            continue;
          }
          if (sink > m) m = sink;
          double l = sinks ? exp(sink - m) : 0.0;
          for (int d = 0; d < head_dim_v; ++d) acc[d] = 0.0;
          for (int64_t t = 0; t < t_end; ++t) {
            int64_t page = block_tables[(int64_t)b * max_pages_per_seq + t / page_size];
            const int64_t vbase = (page * page_size + t % page_size) * (int64_t)head_dim_qk;
            double w = exp(logit[t] - m);
            l += w;
            for (int d = 0; d < head_dim_v; ++d)
              acc[d] += w * (load_elem(kv_pool, kv_dtype, vbase + d) * kv_scale);
          }
          for (int d = 0; d < head_dim_v; ++d) o[d] = acc[d] / l;
          lse[row * num_heads + h] = m + log(l);
        }
      }
    }
    free(logit);
    free(acc);
    free(qd);
  }
  return status;
}

/*
 * Merge of attention states computed over disjoint key ranges (the split-KV
 * reduction): lse = log sum_s exp(lse_s), out = sum_s exp(lse_s - lse) out_s.
 * States with lse_s = -inf (no visible key) carry no weight; if every state
 * is empty the result is out = 0, lse = -inf.
 *
 *  o_states   [num_states, rows, dim]; lse_states [num_states, rows]
 */
void oracle_merge_states(int num_states, int64_t rows, int dim,
                         const double* o_states, const double* lse_states,
                         double* out, double* lse) {
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int s = 0; s < num_states; ++s)
      if (lse_states[(int64_t)s * rows + r] > m) m = lse_states[(int64_t)s * rows + r];
    double* o = out + r * dim;
    for (int d = 0; d < dim; ++d) o[d] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double total = 0.0;
    for (int s = 0; s < num_states; ++s) total += exp(lse_states[(int64_t)s * rows + r] - m);
    double l = m + log(total);
    for (int s = 0; s < num_states; ++s) {
      double w = exp(lse_states[(int64_t)s * rows + r] - l);
      const double* os = o_states + ((int64_t)s * rows + r) * dim;
      if (w == 0.0) continue;
      for (int d = 0; d < dim; ++d) o[d] += w * os[d];
    }
    lse[r] = l;
  }
}

/*
 * OCP E4M3FN encoding of a binary32 value, rounding to nearest with ties to
 * even and saturating to the largest finite magnitude (448): the "RN
 * satfinite" conversion in which PR #5952 commit #5956 stores K / k_scale
 * and V / v_scale. NaN encodes as S.1111.111; +-inf saturate like any value
 * beyond 448. Zero keeps its sign.
 */
static double round_half_even(double a) {
  double f = floor(a);
  double d = a - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
#if ORACLE_MUTATION == 7
  /* planted mistake: ties away from zero */
  return f + 1.0;
#else
  return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
#endif
}

uint8_t oracle_e4m3_from_float(float x) {
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  const double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9 (a count of 8 is the smallest normal) */
    const double q = round_half_even(a * 512.0);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int k;
  frexp(a, &k);      /* a = f 2^k, f in [0.5, 1): the unbiased exponent is k - 1 */
  int e = k - 1;
  double q = round_half_even(ldexp(a, 3 - e));  /* 1.mmm in eighths: 8 .. 16 */
  if (q == 16.0) {
    q = 8.0;
    ++e;
  }
  const int code = ((e + 7) << 3) | ((int)q - 8);
  return (uint8_t)(sign | (code > 0x7E ? 0x7E : code));
}

/*
 * Paged KV append: writes the new tokens' K and V rows into the pools, the
 * step before decode (PR #5952, "fused ... paged KV append"; commit #5956
 * "Contract": seq_lens is the total length after the append, and token r of
 * request b sits at position r + seq_lens[b] - q_len_b).
 *
 *  k_new/v_new  [total_new, num_kv_heads, head_dim] bf16 bits; request b owns
 *               rows q_indptr[b] .. q_indptr[b+1]-1 (v_new may be NULL: a
 *               K-only pool such as the MLA latent cache)
 *  pools        as for oracle_paged_decode (compact rows); BF16 pools get the
 *               bits, E4M3 pools get oracle_e4m3_from_float(x / scale) with the
 *               quotient taken in binary32
 *  zero_tail    nonzero: the slots of each request's last page past its
 *               length are zeroed (K and V), as the pages' append does
 *
 * A row whose page id lies outside the pool is not written (the result is
 * ORACLE_BAD_PAGE); a request with q_len > seq_len writes nothing
 * (ORACLE_BAD_QLEN). Every other row is written. Returns the first error.
 */
int oracle_paged_append(int batch, int num_kv_heads, int head_dim, int page_size, int num_pages,
                        int max_pages_per_seq, int layout, int kv_dtype, const uint16_t* k_new,
                        const uint16_t* v_new, const int32_t* q_indptr, const int32_t* seq_lens,
                        const int32_t* block_tables, float k_scale, float v_scale, void* k_pool,
                        void* v_pool, int64_t k_page_stride, int64_t v_page_stride, int zero_tail) {
  if (batch < 0 || num_kv_heads < 1 || head_dim < 1 || page_size < 1 || num_pages < 0) return ORACLE_BAD_ARG;
  int result = ORACLE_OK;
  for (int b = 0; b < batch; ++b) {
    const int n = q_indptr[b + 1] - q_indptr[b];
    const int L = seq_lens[b];
    if (n < 0 || n > L) {
      if (result == ORACLE_OK) result = ORACLE_BAD_QLEN;
      continue;
    }
    for (int i = 0; i < n; ++i) {
#if ORACLE_MUTATION == 6
      /* planted mistake: positions shifted by one */
      const int64_t pos = (int64_t)L - n + i + 1;
#else
      const int64_t pos = (int64_t)L - n + i;
#endif
      const int64_t page = block_tables[(int64_t)b * max_pages_per_seq + pos / page_size];
      const int64_t slot = pos % page_size;
      if (page < 0 || page >= num_pages) {
        if (result == ORACLE_OK) result = ORACLE_BAD_PAGE;
        continue;
      }
      const int64_t row = (int64_t)q_indptr[b] + i;
      for (int g = 0; g < num_kv_heads; ++g) {
        for (int t = 0; t < 2; ++t) {
          const uint16_t* src = t == 0 ? k_new : v_new;
          void* pool = t == 0 ? k_pool : v_pool;
          if (!src || !pool) continue;
          const int64_t stride = t == 0 ? k_page_stride : v_page_stride;
          const int64_t dst = row_offset(layout, page, slot, g, num_kv_heads, page_size, stride, head_dim);
          const uint16_t* in = src + (row * num_kv_heads + g) * head_dim;
          for (int d = 0; d < head_dim; ++d) {
            if (kv_dtype == ORACLE_BF16) {
              ((uint16_t*)pool)[dst + d] = in[d];
            } else {
              const float x = (float)oracle_bf16_to_double(in[d]);
              const float scale = t == 0 ? k_scale : v_scale;
              const float qv = x / scale;
              ((uint8_t*)pool)[dst + d] = oracle_e4m3_from_float(qv);
            }
          }
        }
      }
    }
    if (zero_tail && L > 0 && L % page_size != 0) {
      const int64_t page = block_tables[(int64_t)b * max_pages_per_seq + (L - 1) / page_size];
      if (page < 0 || page >= num_pages) {
        if (result == ORACLE_OK) result = ORACLE_BAD_PAGE;
        continue;
      }
      for (int64_t slot = L % page_size; slot < page_size; ++slot)
        for (int g = 0; g < num_kv_heads; ++g)
          for (int t = 0; t < 2; ++t) {
            void* pool = t == 0 ? k_pool : v_pool;
            if (!pool || (t == 1 && !v_new)) continue;
            const int64_t stride = t == 0 ? k_page_stride : v_page_stride;
            const int64_t dst = row_offset(layout, page, slot, g, num_kv_heads, page_size, stride, head_dim);
            for (int d = 0; d < head_dim; ++d) {
              if (kv_dtype == ORACLE_BF16)
                ((uint16_t*)pool)[dst + d] = 0;
              else
                ((uint8_t*)pool)[dst + d] = 0;
            }
          }
    }
  }
  return result;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
