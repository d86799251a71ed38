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

/* Computes out[0..D) for query head h of sequence b.  If w is non-NULL it
 * receives the L softmax weights.  `scores` is caller scratch of Smax doubles.
 * Returns the number of valid tokens L used. */
static int attend_row(const orc_problem* p, int b, int h, double* out,
                      double* w, double* scores) {
  const int G = p->Hq / p->Hkv;   /* query heads per KV head */
  const int kvh = h / G;          /* contiguous grouping */
  int L = p->seq_lens[b];
  if (L < 0) L = 0;
  if (L > p->Smax) L = p->Smax;

  const size_t q_off = ((size_t)b * p->Hq + h) * p->D;
  const size_t kv_off = ((size_t)b * p->Hkv + kvh) * (size_t)p->Smax * p->D;
  const double ks = p->k_scale ? p->k_scale[b * p->Hkv + kvh] : 1.0;
  const double vs = p->v_scale ? p->v_scale[b * p->Hkv + kvh] : 1.0;

  for (int d = 0; d < p->D; ++d) out[d] = 0.0;
  if (L == 0) return 0;

  /* scores: s_t = scale * sum_d q_d * k_{t,d} */
  for (int t = 0; t < L; ++t) {
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
  for (int t = 1; t < L; ++t)
    if (scores[t] > m) m = scores[t];
  double z = 0.0;
  for (int t = 0; t < L; ++t) {
    scores[t] = exp(scores[t] - m);
    z += scores[t];
  }
  for (int t = 0; t < L; ++t) scores[t] /= z;
  if (w)
    for (int t = 0; t < L; ++t) w[t] = scores[t];

  /* output: sum_t w_t * v_t */
  for (int t = 0; t < L; ++t) {
    const double wt = scores[t];
    for (int d = 0; d < p->D; ++d) {
      double vd = load_elem(p->v, kv_off + (size_t)t * p->D + d, p->kv_dtype) * vs;
      out[d] += wt * vd;
    }
  }
  return L;
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

/* Number of threads the oracle would use by default. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
