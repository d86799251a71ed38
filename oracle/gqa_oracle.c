/*
 * gqa_oracle.c — plain, slow, fp64 CPU oracle for the grouped-query attention
 * (GQA) decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, import or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA
 * library; the two meet only through the seeded inputs the tests generate.
 *
 * What it computes, and where the pages define it:
 *
 *  - Scaled dot-product attention per query head: score_t = scale * (q . k_t),
 *    weights = softmax(scores), output = sum_t weights_t * v_t.
 *    ("Grouped Query Attention (GQA): Efficient Multi-Head Attention",
 *    Worked example 2: score = q.k / sqrt(head_dim), softmax, weighted sum of
 *    values.)
 *  - Head mapping: query head h reads KV head floor(h / G), G = Hq / Hkv, so
 *    contiguous groups share a KV head ("Llama-2 70B uses 64 query heads, how
 *    many KV heads ...", What the choice does to attention: heads 0-7 read KV
 *    head 0, 8-15 read KV head 1; "GQA, decode the acronym", same mapping;
 *    "Grouped-Query Attention: How Sharing KV Heads Shrinks Inference Memory",
 *    How grouped-query attention works: floor(h / (H / G)) with G groups).
 *  - Decode step: one new query per head attends over every cached token of
 *    its sequence ("... Efficient Multi-Head Attention", The bottleneck: at each
 *    decoding step attend over the cached K/V of all prior tokens).  The cache
 *    holds exactly seq_lens[b] valid tokens; the caller has appended the current
 *    token already.  A sequence with no valid token yields an all-zero output.
 *  - FP8 cache: each stored byte is an OCP FP8 E4M3 ("e4m3fn") or E5M2 code (the
 *    pages name both 8-bit formats), the value
 *    is decode(code) * scale with one fp32 scale per (sequence, KV head) for K
 *    and one for V ("... Shrinks Inference Memory", FP8 KV cache: 8-bit
 *    floating-point cache with scaling factors).
 *  - KV cache bytes per token = 2 * layers * kv_heads * head_dim * bytes
 *    ("Grouped Query Attention: Why 8 KV Heads Decide Your Batch Size", TL;DR
 *    and "Why does GQA decide your batch size?").
 *
 * Every input element is first converted to fp64 by this file's own decoders
 * (written from the IEEE binary16, bfloat16 and OCP FP8 E4M3 / E5M2 bit
 * layouts);
 * all arithmetic after that is fp64.  The softmax subtracts the row maximum
 * before exponentiating (a rewrite that is exact in real arithmetic).
 *
 * Independent (b, h) rows may be computed on several threads (OpenMP); the
 * arithmetic of one row is a plain sequential loop and does not depend on the
 * thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element type codes understood by the oracle's loaders. */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_F64 = 3, ORC_E5M2 = 4 };

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1F;
  int f = bits & 0x3FF;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
  } else if (e == 31) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(1.0 + (double)f / 1024.0, e - 15);
  }
  return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xFF;
  int f = bits & 0x7F;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -133); /* subnormal: f * 2^-7 * 2^-126 */
  } else if (e == 255) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(1.0 + (double)f / 128.0, e - 127);
  }
  return sign ? -mag : mag;
}

/* OCP FP8 E4M3 ("fn" flavour): 1 sign bit, 4 exponent bits (bias 7), 3
 * fraction bits, no infinities, S.1111.111 is NaN, largest finite 448. */
double oracle_e4m3_to_f64(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xF;
  int f = bits & 0x7;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -9); /* subnormal: f * 2^-3 * 2^-6 */
  } else if (e == 15 && f == 7) {
    mag = NAN;
  } else {
    mag = ldexp(1.0 + (double)f / 8.0, e - 7);
  }
  return sign ? -mag : mag;
}

/* OCP FP8 E5M2: 1 sign bit, 5 exponent bits (bias 15), 2 fraction bits,
 * IEEE-style infinities and NaNs at exponent 31, largest finite 57344. */
double oracle_e5m2_to_f64(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 2) & 0x1F;
  int f = bits & 0x3;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -16); /* subnormal: f * 2^-2 * 2^-14 */
  } else if (e == 31) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp(1.0 + (double)f / 4.0, e - 15);
  }
  return sign ? -mag : mag;
}

static double load_elem(const void* base, size_t idx, int dtype) {
  switch (dtype) {
    case ORC_F16: return oracle_f16_to_f64(((const uint16_t*)base)[idx]);
    case ORC_BF16: return oracle_bf16_to_f64(((const uint16_t*)base)[idx]);
    case ORC_E4M3: return oracle_e4m3_to_f64(((const uint8_t*)base)[idx]);
    case ORC_E5M2: return oracle_e5m2_to_f64(((const uint8_t*)base)[idx]);
    case ORC_F64: return ((const double*)base)[idx];
    default: return NAN;
  }
}

/* ------------------------------------------------------- cache-size formula */

/* 2 (K and V) x layers x kv_heads x head_dim x bytes per element. */
uint64_t oracle_kv_bytes_per_token(int layers, int kv_heads, int head_dim,
                                   int bytes_per_elem) {
  return 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim *
         (uint64_t)bytes_per_elem;
}

/* --------------------------------------------------------- one (b, h) row */

typedef struct {
  const void* q;       /* [B, Hq, D]        q_dtype   */
  const void* k;       /* [B, Hkv, Smax, D] kv_dtype  */
  const void* v;       /* [B, Hkv, Smax, D] kv_dtype  */
  const double* k_scale; /* [B, Hkv] or NULL (then 1) */
  const double* v_scale; /* [B, Hkv] or NULL (then 1) */
  const int32_t* seq_lens; /* [B] */
  double scale;
  int B, Hq, Hkv, Smax, D;
  int q_dtype, kv_dtype;
} orc_problem;

/* Attention of one query row against the first n cached tokens of KV head
 * kvh of sequence b: the query is D elements at q_off of the query tensor.
 * If w is non-NULL it receives the n softmax weights.  `scores` is caller
 * scratch of Smax doubles.  Returns n. */
static int attend(const orc_problem* p, int b, int kvh, size_t q_off, int n,
                  double* out, double* w, double* scores) {
  const size_t kv_off = ((size_t)b * p->Hkv + kvh) * (size_t)p->Smax * p->D;
  const double ks = p->k_scale ? p->k_scale[b * p->Hkv + kvh] : 1.0;
  const double vs = p->v_scale ? p->v_scale[b * p->Hkv + kvh] : 1.0;

  for (int d = 0; d < p->D; ++d) out[d] = 0.0;
  if (n <= 0) return 0;

  /* scores: s_t = scale * sum_d q_d * k_{t,d} */
  for (int t = 0; t < n; ++t) {
    double dot = 0.0;
    for (int d = 0; d < p->D; ++d) {
      double qd = load_elem(p->q, q_off + d, p->q_dtype);
      double kd = load_elem(p->k, kv_off + (size_t)t * p->D + d, p->kv_dtype) * ks;
      dot += qd * kd;
    }
    scores[t] = p->scale * dot;
  }

  /* softmax with the row maximum subtracted */
  double m = scores[0];
  for (int t = 1; t < n; ++t)
    if (scores[t] > m) m = scores[t];
  double z = 0.0;
  for (int t = 0; t < n; ++t) {
    scores[t] = exp(scores[t] - m);
    z += scores[t];
  }
  for (int t = 0; t < n; ++t) scores[t] /= z;
  if (w)
    for (int t = 0; t < n; ++t) w[t] = scores[t];

  /* output: sum_t w_t * v_t */
  for (int t = 0; t < n; ++t) {
    const double wt = scores[t];
    for (int d = 0; d < p->D; ++d) {
      double vd = load_elem(p->v, kv_off + (size_t)t * p->D + d, p->kv_dtype) * vs;
      out[d] += wt * vd;
    }
  }
  return n;
}

static int clamped_len(const orc_problem* p, int b) {
  int L = p->seq_lens[b];
  if (L < 0) L = 0;
  if (L > p->Smax) L = p->Smax;
  return L;
}

/* Computes out[0..D) for query head h of sequence b (one new token, q
 * [B, Hq, D]): attention over all L_b cached tokens of KV head floor(h/G). */
static int attend_row(const orc_problem* p, int b, int h, double* out,
                      double* w, double* scores) {
  const int G = p->Hq / p->Hkv;   /* query heads per KV head */
  const int kvh = h / G;          /* contiguous grouping */
  const size_t q_off = ((size_t)b * p->Hq + h) * p->D;
  return attend(p, b, kvh, q_off, clamped_len(p, b), out, w, scores);
}

static int check_problem(const orc_problem* p) {
  if (!p->q || !p->k || !p->v || !p->seq_lens) return 1;
  if (p->B < 0 || p->Hq < 1 || p->Hkv < 1 || p->Smax < 1 || p->D < 1) return 1;
  if (p->Hq % p->Hkv != 0) return 1;
  if (p->q_dtype == ORC_E4M3 || p->q_dtype == ORC_E5M2) return 1;
  if (p->q_dtype < 0 || p->q_dtype > ORC_E5M2) return 1;
  if (p->kv_dtype < 0 || p->kv_dtype > ORC_E5M2) return 1;
  return 0;
}

/* ------------------------------------------------------------- entry points */

/* Full decode step: out[B, Hq, D] (fp64).  k_scale / v_scale may be NULL
 * (scale 1).  nthreads <= 0 uses the OpenMP default.  Returns 0 on success. */
int oracle_gqa_decode(const void* q, int q_dtype, const void* k, const void* v,
                      int kv_dtype, const double* k_scale,
                      const double* v_scale, const int32_t* seq_lens,
                      double scale, double* out, int B, int Hq, int Hkv,
                      int Smax, int D, int nthreads) {
  orc_problem p = {q, k, v, k_scale, v_scale, seq_lens, scale,
                   B, Hq, Hkv, Smax, D, q_dtype, kv_dtype};
  if (check_problem(&p) || !out) return 1;
  const long rows = (long)B * Hq;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)Smax);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (long r = 0; r < rows; ++r) {
      int b = (int)(r / Hq), h = (int)(r % Hq);
      attend_row(&p, b, h, out + (size_t)r * D, NULL, scores);
    }
    free(scores);
  }
  return 0;
}

/* Sampled rows: for each i < n, computes the output row of (bh[2i], bh[2i+1])
 * into out[i*D .. i*D + D).  Same arithmetic as oracle_gqa_decode. */
int oracle_gqa_decode_rows(const void* q, int q_dtype, const void* k,
                           const void* v, int kv_dtype, const double* k_scale,
                           const double* v_scale, const int32_t* seq_lens,
                           double scale, const int32_t* bh, int n, double* out,
                           int B, int Hq, int Hkv, int Smax, int D,
                           int nthreads) {
  orc_problem p = {q, k, v, k_scale, v_scale, seq_lens, scale,
                   B, Hq, Hkv, Smax, D, q_dtype, kv_dtype};
  if (check_problem(&p) || !out || !bh) return 1;
  for (int i = 0; i < n; ++i)
    if (bh[2 * i] < 0 || bh[2 * i] >= B || bh[2 * i + 1] < 0 ||
        bh[2 * i + 1] >= Hq)
      return 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)Smax);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int i = 0; i < n; ++i)
      attend_row(&p, bh[2 * i], bh[2 * i + 1], out + (size_t)i * D, NULL,
                 scores);
    free(scores);
  }
  return 0;
}

/* Debug entry: the softmax weights of one (b, h) row, w[0..L), and its output
 * row.  Returns L, or -1 on a bad argument. */
int oracle_gqa_weights(const void* q, int q_dtype, const void* k,
                       const void* v, int kv_dtype, const double* k_scale,
                       const double* v_scale, const int32_t* seq_lens,
                       double scale, int b, int h, double* w, double* out_row,
                       int B, int Hq, int Hkv, int Smax, int D) {
  orc_problem p = {q, k, v, k_scale, v_scale, seq_lens, scale,
                   B, Hq, Hkv, Smax, D, q_dtype, kv_dtype};
  if (check_problem(&p) || !w || !out_row) return -1;
  if (b < 0 || b >= B || h < 0 || h >= Hq) return -1;
  double* scores = (double*)malloc(sizeof(double) * (size_t)Smax);
  int L = attend_row(&p, b, h, out_row, w, scores);
  free(scores);
  return L;
}

/* Multi-token step (chunked prefill / speculative decode): q and out are
 * [B, Hq, T, D]; the last T of sequence b's L_b cached tokens are the new
 * ones, and new token i (0-based) attends causally to cached tokens
 * t <= L_b - T + i, i.e. to the first max(0, L_b - T + i + 1) of them
 * (scaled dot-product attention with a causal mask, as in "Grouped Query
 * Attention: Why 8 KV Heads Decide Your Batch Size", The repeat_kv trap:
 * scaled_dot_product_attention(..., is_causal=True, enable_gqa=True)).
 * T = 1 is the decode step.  Returns 0 on success. */
int oracle_gqa_decode_chunk(const void* q, int q_dtype, const void* k,
                            const void* v, int kv_dtype, const double* k_scale,
                            const double* v_scale, const int32_t* seq_lens,
                            double scale, double* out, int B, int Hq, int Hkv,
                            int T, int Smax, int D, int nthreads) {
  orc_problem p = {q, k, v, k_scale, v_scale, seq_lens, scale,
                   B, Hq, Hkv, Smax, D, q_dtype, kv_dtype};
  if (check_problem(&p) || !out || T < 1) return 1;
  const long rows = (long)B * Hq * T;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)Smax);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (long r = 0; r < rows; ++r) {
      const int b = (int)(r / ((long)Hq * T));
      const int h = (int)((r / T) % Hq);
      const int i = (int)(r % T);
      const int L = clamped_len(&p, b);
      int n = L - T + i + 1;
      if (n > L) n = L;
      attend(&p, b, h / G, (size_t)r * D, n, out + (size_t)r * D, NULL,
             scores);
    }
    free(scores);
  }
  return 0;
}

/* ------------------------------------------ cache append (+ FP8 quantise) */

/* Largest finite value of an 8-bit code type. */
static float fp8_max(int dtype) { return dtype == ORC_E5M2 ? 57344.0f : 448.0f; }

/* fp32 -> 8-bit code, round to nearest even on the format's grid, values
 * beyond the largest finite value clamped to it ("satfinite").  Written from
 * the OCP FP8 E4M3 (bias 7, 3 fraction bits, no inf, S.1111.111 NaN) and
 * E5M2 (bias 15, 2 fraction bits, exponent 31 inf/NaN) layouts. */
uint8_t oracle_f32_to_fp8(float v, int dtype) {
  const int mbits = dtype == ORC_E5M2 ? 2 : 3;
  const int bias = dtype == ORC_E5M2 ? 15 : 7;
  const int emax = dtype == ORC_E5M2 ? 15 : 8; /* largest unbiased exponent */
  const double maxv = fp8_max(dtype);
  const uint8_t maxcode = dtype == ORC_E5M2 ? 0x7B : 0x7E;
  if (v != v) return 0x7F; /* NaN */
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= maxv) return sign | maxcode;
  const double min_normal = ldexp(1.0, 1 - bias);
  if (a < min_normal) {
    /* subnormal grid: multiples of 2^(1 - bias - mbits) */
    double q = nearbyint(a / ldexp(1.0, 1 - bias - mbits));
    return sign | (uint8_t)q; /* q == 2^mbits is the smallest normal code */
  }
  int e;
  frexp(a, &e);
  e -= 1; /* a = 1.f * 2^e */
  double r = nearbyint((a / ldexp(1.0, e) - 1.0) * (double)(1 << mbits));
  if (r == (double)(1 << mbits)) {
    r = 0.0;
    e += 1;
  }
  if (e > emax || (dtype != ORC_E5M2 && e == emax && (int)r == 7))
    return sign | maxcode;
  return sign | (uint8_t)(((e + bias) << mbits) | (int)r);
}

/* Appends one token's K and V rows per (sequence, KV head) at position
 * L_b = seq_lens[b] and sets seq_lens[b] = L_b + 1 ("Grouped Query Attention
 * (GQA): Efficient Multi-Head Attention", The bottleneck: the cache grows by
 * one token's K and V per decoding step).  16-bit caches: the rows are copied.
 * 8-bit caches ("Grouped-Query Attention: How Sharing KV Heads Shrinks
 * Inference Memory", FP8 KV cache: codes with scaling factors), per (b, kvh)
 * and tensor, all decisions in fp32:
 *   a = max_d |x_d|;
 *   scale s <= 0 (unset): s' = a / MAX (1 if a == 0), earlier codes kept;
 *   else s' = s doubled until a / s' <= MAX; if it grew, every earlier code
 *        c of the slab becomes encode(decode(c) * (s / s'));
 *   the new row's codes are encode(x_d / s'); the scale becomes s'.
 * A sequence with L_b >= Smax is left unchanged and flags bit 2 (cache full).
 * Returns the flags (0 when every sequence was appended). */
int oracle_append_kv(const void* k_new, const void* v_new, int in_dtype,
                     void* k_cache, void* v_cache, int cache_dtype,
                     float* k_scale, float* v_scale, int32_t* seq_lens, int B,
                     int Hkv, int Smax, int D) {
  int flags = 0;
  const int fp8 = cache_dtype == ORC_E4M3 || cache_dtype == ORC_E5M2;
  const float M = fp8 ? fp8_max(cache_dtype) : 0.0f;
  for (int b = 0; b < B; ++b) {
    int L = seq_lens[b] < 0 ? 0 : seq_lens[b];
    if (L >= Smax) {
      flags |= 4;
      continue;
    }
    for (int j = 0; j < Hkv; ++j) {
      for (int which = 0; which < 2; ++which) {
        const void* src = which ? v_new : k_new;
        void* cache = which ? v_cache : k_cache;
        float* scales = which ? v_scale : k_scale;
        const size_t row = (size_t)b * Hkv + j;
        const size_t slab = row * (size_t)Smax * D;
        if (!fp8) {
          for (int d = 0; d < D; ++d)
            ((uint16_t*)cache)[slab + (size_t)L * D + d] =
                ((const uint16_t*)src)[row * D + d];
          continue;
        }
        uint8_t* codes = (uint8_t*)cache;
        float a = 0.0f;
        for (int d = 0; d < D; ++d) {
          float x = (float)load_elem(src, row * D + d, in_dtype);
          if (fabsf(x) > a) a = fabsf(x);
        }
        float s = scales[row], s2;
        if (!(s > 0.0f)) {
          s2 = a > 0.0f ? a / M : 1.0f;
        } else {
          s2 = s;
          for (int it = 0; it < 256 && a / s2 > M; ++it) s2 = s2 * 2.0f;
          if (s2 != s) {
            const float ratio = s / s2;
            for (size_t i = 0; i < (size_t)L * D; ++i) {
              float c = (float)load_elem(codes, slab + i, cache_dtype);
              codes[slab + i] = oracle_f32_to_fp8(c * ratio, cache_dtype);
            }
          }
        }
        for (int d = 0; d < D; ++d) {
          float x = (float)load_elem(src, row * D + d, in_dtype);
          codes[slab + (size_t)L * D + d] = oracle_f32_to_fp8(x / s2, cache_dtype);
        }
        scales[row] = s2;
      }
    }
    seq_lens[b] = L + 1;
  }
  return flags;
}

/* Number of threads the oracle would use by default. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
