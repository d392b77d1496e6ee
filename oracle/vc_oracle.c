/*
 * vc_oracle.c -- plain, slow CPU oracle for the ExpCast-FP8 + V-Smooth FP8 attention forward.
 *
 * TEST INFRASTRUCTURE. This library exists only to check the CUDA path. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product path never calls it.
 * It shares no code, header, table or constant generator with the CUDA library.
 *
 * Sources, cited by page title and section/equation:
 *   [VC]  "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention" (arXiv 2609.15810)
 *   [OVC] "Open-VC Attention: an open-source, error-tunable variant of VC-Attention" (MachGen blog)
 *
 * Floating point: sums, means and the exact attention are fp64. Where the method fixes an fp32
 * step that decides an integer (the ExpCast code, an E4M3 code), the step is written in fp32 and
 * the file must be compiled with -ffp-contract=off so that no a*b+c is fused behind our back.
 *
 * Readings taken where the pages are silent (each one also listed in the design notes):
 *   R1  E4M3 follows the OCP FP8 E4M3 format the tensor core consumes: exponent field 0 is
 *       subnormal (m/8 * 2^-6), 0x7F/0xFF are NaN, the largest finite value is 448.
 *   R2  Encoding is round-to-nearest-even with saturation to +-448.
 *   R3  One Q/K scale per 128-token block is one scalar over the 128 x D block, s = amax/448.
 *   R4  k-means: Lloyd iterations (assign -> update) started from c_i = x_{floor(i*S/k)}; ties in
 *       the assignment go to the lowest index; an empty cluster keeps its centroid.
 *   R5  The partial last block's mean is taken over its valid rows only.
 *   R6  The ExpCast pre-round value is computed as one fp32 fused multiply-add
 *       y = fmaf(S32, a_j, 119.65f - M), then rounded to the nearest integer, ties to even, and
 *       clipped to [0, 120]. Codes 1..7 decode as E4M3 subnormals.
 *   R7  Key visit order for query tile qt: start = min(nkb-1, 2*floor(qt/2) + 2), sweep down to 0, then
 *       the tail. The two query tiles 2m and 2m+1 share one order (2 and 1 blocks past their
 *       diagonals), so that one pass over the keys can serve both.
 *   R17 Per-channel V residual scale (an option; one scale per head is the default): the channel's
 *       scale is its residual amax over the whole head / 448 (1 when the channel is all zero), and
 *       the stored block means are bf16(fp32(mean) / scale), so that the single epilogue multiply
 *       by the channel's scale restores both the residual and the mean term.
 *   R18 V residual repair ([OVC]): the budget is a row count n_rep per head (rho*S rounded up by the
 *       caller); the energy of a token is summed in fp32 in channel order from its true-unit rounding
 *       residuals, ties to the lower index; the kept tokens' keys are copied in ascending token order
 *       into extra 128-row blocks quantised like any other key block (own scale per block); their
 *       residuals are coded in E4M3 in the main residual codes' units; repair tiles leave the running
 *       max and the row sum alone (codes clip at 120).  Defined without V-Smooth only.
 *   R19 QK Hadamard rotation (an option): the unnormalised Walsh-Hadamard transform of every Q and K
 *       row (after the K centre), as an fp32 butterfly in a fixed stage order, before the block
 *       quantiser; the score constant takes the 1/D.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BLOCK 128

/* ---------------------------------------------------------------------------------------------
 * E4M3 codec.  [VC] §3.3: "A byte with exponent field e and mantissa field m encodes the value
 * v = 2^(e-7)(1+m/8)".  Subnormals / NaN / saturation follow reading R1/R2.
 * ------------------------------------------------------------------------------------------- */
double orc_e4m3_decode(uint8_t c) {
  int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a > 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid: multiples of 2^-9; m == 8 lands exactly on the smallest normal (code 8) */
    double m = nearbyint(a * 512.0);
    return sign | (uint8_t)m;
  }
  int ex;
  double fr = frexp(a, &ex);      /* a = fr * 2^ex, fr in [0.5, 1) */
  int e = ex - 1;                 /* a = (2 fr) * 2^e, 2fr in [1, 2) */
  double m = nearbyint((2.0 * fr - 1.0) * 8.0); /* exact product, RNE on the 3-bit mantissa */
  if (m == 8.0) { e += 1; m = 0.0; }
  int code = ((e + 7) << 3) | (int)m;
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

void orc_e4m3_decode_n(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}
void orc_e4m3_encode_n(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}

/* bf16 helpers: bf16 -> fp32 is exact; fp64 -> bf16 rounds once, to nearest even. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
uint16_t orc_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int ex;
  double fr = frexp(a, &ex);      /* a = fr 2^ex, fr in [0.5,1) */
  int e = ex - 1;                 /* unbiased exponent of a */
  if (e < -126) {                 /* bf16 subnormal grid: multiples of 2^-133 */
    double m = nearbyint(ldexp(a, 133));
    uint32_t bits = (uint32_t)m;  /* m <= 128 -> may carry into the smallest normal */
    return sign | (uint16_t)bits;
  }
  double m = nearbyint((2.0 * fr) * 128.0); /* 8 significant bits: [128, 256] */
  if (m == 256.0) { m = 128.0; e += 1; }
  if (e > 127) return sign | 0x7F80; /* overflow -> inf */
  uint32_t bits = ((uint32_t)(e + 127) << 7) | ((uint32_t)m - 128u);
  return sign | (uint16_t)bits;
}
void orc_f64_to_bf16_n(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(x[i]);
}

/* ---------------------------------------------------------------------------------------------
 * ExpCast-FP8.  [VC] §3.3 Eq. 7: c(u) = clip_[0,120](Round(8(u+8) + 56 + beta)), beta = -0.35,
 * Round = round-to-nearest-even.  [OVC] "Scheduling around ExpCast": the softmax scale, the Q/K
 * dequantisation scales, log2 e, the factor 8 and the running maximum fold into one FMA a*S + b.
 * With S32 the raw fp32 score and a_j = 8 log2(e)/sqrt(D) * sQ * sK, S32*a_j is the true score in
 * code units, so 8(u+8)+56+beta = S32*a_j + (120 + beta) - M.  Reading R6 fixes the fp32 contract.
 * ------------------------------------------------------------------------------------------- */
static const float ORC_B0 = 119.65f; /* 8*8 + 56 + beta */

int orc_expcast_unclipped(float s32, float a, float b) { return (int)rintf(fmaf(s32, a, b)); }

int orc_expcast_code(float s32, float a, float b) {
  float y = fmaf(s32, a, b);
  if (isnan(y)) return 0;
  float r = rintf(y);
  if (r < 0.0f) return 0;
  if (r > 120.0f) return 120;
  return (int)r;
}

void orc_expcast_codes(const float* s, const float* a, const float* b, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_expcast_code(s[i], a[i], b[i]);
}

/* The conventional path that ExpCast replaces ([VC] §3.3, Fig. 5a): exponentiate, then cast to
 * E4M3.  u is the log2-domain score relative to the row maximum; the row maximum lands at 2^8. */
uint8_t orc_exp_then_cast(double u) { return orc_e4m3_encode((float)exp2(u + 8.0)); }

/* Code of the direct map as a function of u alone (no fp32 score path): the reference formula
 * of Eq. 7 evaluated in double, used by the pins that compare against the printed statistics. */
int orc_expcast_of_u(double u) {
  double r = nearbyint(8.0 * (u + 8.0) + 56.0 - 0.35);
  if (r < 0) r = 0;
  if (r > 120) r = 120;
  return (int)r;
}

/* ---------------------------------------------------------------------------------------------
 * Per-128-token block quantiser for Q and K'.  [OVC] "Scheduling around ExpCast": "Q and K are
 * quantized to FP8 with one scale per 128-token block".  Reading R3: s = amax/448, inverse scale
 * 448/amax computed once in fp32, code = E4M3(x * inv).  An all-zero block gets s = 1.
 * x: [S, D] bf16 bits, codes: [S_pad, D] (pad rows zero), scales: [nkb].
 * ------------------------------------------------------------------------------------------- */
/* center: NULL, or one bf16 value per channel subtracted (in fp32) from every row before the
 * block maximum and the codes are taken (the K channel centering below). */
/* QK Hadamard rotation ([VC] §3.4 "Fused preprocessing", App. B: the Q and K quantisation passes fuse
 * a Hadamard rotation; Fig. 3 / §4: it shrinks the probability term and is free in time).  Reading R19:
 * the unnormalised Sylvester-order Walsh-Hadamard transform of each row, y = H_D x with
 * H_D[i][j] = (-1)^popcount(i & j), computed in fp32 as the usual butterfly: stages s = 1, 2, ..., D/2,
 * each replacing the pair (x[i], x[i+s]) (bit s of i clear) by (x[i] + x[i+s], x[i] - x[i+s]).  The
 * 1/sqrt(D) of the orthonormal rotation cancels in the block quantiser's amax scale and is folded into
 * the score constant instead (scores of rotated operands are D times the plain ones). */
void orc_fwht_f32(float* x, int D) {
  for (int s = 1; s < D; s <<= 1)
    for (int i = 0; i < D; ++i)
      if (!(i & s)) {
        float a = x[i], b = x[i + s];
        x[i] = a + b;
        x[i + s] = a - b;
      }
}

/* Row t of the block quantiser's input in fp32: x - center when a centre is given, then rotated. */
static void orc_quant_row(const uint16_t* x, int64_t t, int D, const uint16_t* center, int rotate, float* v) {
  for (int d = 0; d < D; ++d) {
    v[d] = bf16_to_f32(x[t * D + d]);
    if (center) v[d] = v[d] - bf16_to_f32(center[d]);
  }
  if (rotate) orc_fwht_f32(v, D);
}

void orc_quant_blocks_rot(const uint16_t* x, int64_t S, int D, const uint16_t* center, int rotate, uint8_t* codes,
                          float* scales) {
  int64_t nkb = (S + ORC_BLOCK - 1) / ORC_BLOCK;
  float* v = (float*)malloc((size_t)D * sizeof(float));
  memset(codes, 0, (size_t)(nkb * ORC_BLOCK * D));
  for (int64_t j = 0; j < nkb; ++j) {
    int64_t t0 = j * ORC_BLOCK, t1 = t0 + ORC_BLOCK < S ? t0 + ORC_BLOCK : S;
    float amax = 0.0f;
    for (int64_t t = t0; t < t1; ++t) {
      orc_quant_row(x, t, D, center, rotate, v);
      for (int d = 0; d < D; ++d)
        if (fabsf(v[d]) > amax) amax = fabsf(v[d]);
    }
    if (amax == 0.0f) { scales[j] = 1.0f; continue; }
    float inv = 448.0f / amax;
    scales[j] = amax / 448.0f;
    for (int64_t t = t0; t < t1; ++t) {
      orc_quant_row(x, t, D, center, rotate, v);
      for (int d = 0; d < D; ++d) codes[t * D + d] = orc_e4m3_encode(v[d] * inv);
    }
  }
  free(v);
}

void orc_quant_blocks_centered(const uint16_t* x, int64_t S, int D, const uint16_t* center, uint8_t* codes,
                               float* scales) {
  orc_quant_blocks_rot(x, S, D, center, 0, codes, scales);
}

void orc_quant_blocks(const uint16_t* x, int64_t S, int D, uint8_t* codes, float* scales) {
  orc_quant_blocks_centered(x, S, D, NULL, codes, scales);
}

/* ---------------------------------------------------------------------------------------------
 * K channel centering.  [VC] §3.4 "Fused preprocessing" and App. B: the K quantisation pass fuses
 * "the centering statistics" and "mean subtraction".  Subtracting one vector from every key adds a
 * per-query constant to the scores, which the softmax ignores, while the keys' quantisation range
 * shrinks.  Reading: the statistic is the channel mean over the S tokens of the head, taken in fp64
 * and rounded once to bf16 (mu[d]); the keys are quantised as K - mu in fp32.
 * x: [S, D] bf16 bits, token order.  mu: [D] bf16 bits.
 * ------------------------------------------------------------------------------------------- */
void orc_channel_mean_bf16(const uint16_t* x, int64_t S, int D, uint16_t* mu) {
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int64_t t = 0; t < S; ++t) acc += (double)bf16_to_f32(x[t * D + d]);
    mu[d] = orc_f64_to_bf16(acc / (double)S);
  }
}

/* ---------------------------------------------------------------------------------------------
 * Value-guided grouping.  [VC] §3.2 "Value-guided permutation": per batch and head an online
 * k-means over the value tokens assigns a label z_t; pi = argsort(z); "Unbalanced clusters cost
 * little": plain (unbalanced) k-means.  Reading R4 fixes init, iteration and ties.
 * v: [S, D] bf16 bits.  labels: [S].  centroids: [k, D] (fp64).  J_rounds: [iters] objective of
 * each round's assignment (sum of squared distances to the member means).
 * ------------------------------------------------------------------------------------------- */
double orc_kmeans_objective(const uint16_t* v, int64_t S, int D, int k, const int32_t* labels) {
  double* sum = (double*)calloc((size_t)k * D, sizeof(double));
  int64_t* cnt = (int64_t*)calloc((size_t)k, sizeof(int64_t));
  for (int64_t t = 0; t < S; ++t) {
    int z = labels[t];
    cnt[z]++;
    for (int d = 0; d < D; ++d) sum[(int64_t)z * D + d] += bf16_to_f32(v[t * D + d]);
  }
  for (int i = 0; i < k; ++i)
    if (cnt[i])
      for (int d = 0; d < D; ++d) sum[(int64_t)i * D + d] /= (double)cnt[i];
  double J = 0.0;
  for (int64_t t = 0; t < S; ++t) {
    const double* m = sum + (int64_t)labels[t] * D;
    for (int d = 0; d < D; ++d) {
      double e = bf16_to_f32(v[t * D + d]) - m[d];
      J += e * e;
    }
  }
  free(sum);
  free(cnt);
  return J;
}

/* Lloyd rounds from the centroids already in `centroids` ([k, D], fp64).  Warm start ([VC] §3.2
 * "Unbalanced clusters cost little": "warm-starting each step from the previous step's centroids
 * halves its cost"): the caller passes the previous grouping's centroids here instead of rows. */
void orc_kmeans_from(const uint16_t* v, int64_t S, int D, int k, int iters, int32_t* labels, double* centroids,
                     double* J_rounds) {
  double* sum = (double*)malloc((size_t)k * D * sizeof(double));
  int64_t* cnt = (int64_t*)malloc((size_t)k * sizeof(int64_t));
  for (int it = 0; it < iters; ++it) {
    /* assign: nearest centroid in squared Euclidean distance, ties to the lowest index */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < S; ++t) {
      double best = INFINITY;
      int bi = 0;
      for (int i = 0; i < k; ++i) {
        const double* c = centroids + (int64_t)i * D;
        double dist = 0.0;
        for (int d = 0; d < D; ++d) {
          double e = (double)bf16_to_f32(v[t * D + d]) - c[d];
          dist += e * e;
        }
        if (dist < best) { best = dist; bi = i; }
      }
      labels[t] = bi;
    }
    if (J_rounds) J_rounds[it] = orc_kmeans_objective(v, S, D, k, labels);
    /* update: member mean; an empty cluster keeps its centroid */
    memset(sum, 0, (size_t)k * D * sizeof(double));
    memset(cnt, 0, (size_t)k * sizeof(int64_t));
    for (int64_t t = 0; t < S; ++t) {
      cnt[labels[t]]++;
      for (int d = 0; d < D; ++d) sum[(int64_t)labels[t] * D + d] += bf16_to_f32(v[t * D + d]);
    }
    for (int i = 0; i < k; ++i)
      if (cnt[i])
        for (int d = 0; d < D; ++d) centroids[(int64_t)i * D + d] = sum[(int64_t)i * D + d] / (double)cnt[i];
  }
  free(sum);
  free(cnt);
}

void orc_kmeans(const uint16_t* v, int64_t S, int D, int k, int iters, int32_t* labels, double* centroids,
                double* J_rounds) {
  for (int i = 0; i < k; ++i) {
    int64_t src = (int64_t)((double)i * (double)S / (double)k);
    for (int d = 0; d < D; ++d) centroids[(int64_t)i * D + d] = bf16_to_f32(v[src * D + d]);
  }
  orc_kmeans_from(v, S, D, k, iters, labels, centroids, J_rounds);
}

/* ---------------------------------------------------------------------------------------------
 * Grouping schedule over a run of n denoising steps.  [VC] §3.4 "Amortized grouping schedule" and
 * App. A "Grouping schedule": grouping and demeaning run on the first 25% of the steps, a window of
 * ceil(n/4) steps; inside it the permutation is computed once and reused for `reuse` adjacent steps
 * (4 in the pages: steps 0, 4, 8 of a 40-step run); after the window the plain low-bit kernel runs on
 * the permutation the window left behind (reading R12: pi kept, no means).
 * Returns 0 = group from scratch, 1 = group warm-started from the previous centroids, 2 = reuse pi
 * with V-Smooth, 3 = plain kernel on the kept pi.
 * ------------------------------------------------------------------------------------------- */
int orc_schedule_action(int step, int n_steps, int reuse) {
  const int window = (n_steps + 3) / 4;
  if (step >= window) return 3;
  if (step % reuse != 0) return 2;
  return step == 0 ? 0 : 1;
}

/* Stable argsort of the labels by counting sort: pi lists the tokens of cluster 0 in token order,
 * then cluster 1, ...  ([VC] §3.2 Eq. 3: pi = argsort(z), applied to K and V, Q keeps its order.) */
void orc_stable_argsort(const int32_t* z, int64_t S, int k, int32_t* perm) {
  int64_t* start = (int64_t*)calloc((size_t)k + 1, sizeof(int64_t));
  for (int64_t t = 0; t < S; ++t) start[z[t] + 1]++;
  for (int i = 0; i < k; ++i) start[i + 1] += start[i];
  for (int64_t t = 0; t < S; ++t) perm[start[z[t]]++] = (int32_t)t;
  free(start);
}

/* ---------------------------------------------------------------------------------------------
 * Gather, block demeaning and residual quantisation of V.  [VC] §3.2 "Block demeaning" Eq. 4:
 * mu_j = mean of the rows of block j of V' = V[pi], R_j = V'_j - 1 mu_j^T, each mean one 16-bit
 * vector.  [OVC] "Scheduling around ExpCast": V (here its residual) gets one scale per head.
 * The residual is taken against the stored bf16 mean, so R + mu_b reconstructs V' (reading R5 for
 * the partial block).  perm may be NULL (identity); subtract_mean = 0 gives R = V' and mu = 0.
 * Outputs: mu [nkb, D] fp64 (exact mean), mub [nkb, D] bf16 bits, resid [S_pad, D] fp32 (pad rows
 * zero), rcodes [S_pad, D] E4M3 codes of R * 448/amax, *amax_out, *sv_out = amax/448.
 * ------------------------------------------------------------------------------------------- */
/* per_channel = 0: one residual scale per head ([OVC]); amax_out[0], sv_out[0] and mut unused.
 * per_channel = 1: one scale per channel ([VC] §3.2 "Block demeaning": the residual goes through
 * "per-channel E4M3 at 8 bits"; App. B: "the means are stored divided by the per-channel value
 * scale, so the kernel's single epilogue multiply applies to both terms of Eq. 6").  Reading R17:
 * amax_out[d] = max_t |R[t,d]| over the head, sv_out[d] = amax_d/448 (1 for an all-zero channel),
 * codes E4M3(R * (448/amax_d)), and the stored means mut[j,d] = bf16(fp32(mub[j,d]) / sv[d]). */
void orc_demean_ex(const uint16_t* v, const int32_t* perm, int64_t S, int D, int subtract_mean, int per_channel,
                   double* mu, uint16_t* mub, uint16_t* mut, float* resid, uint8_t* rcodes, float* amax_out,
                   float* sv_out) {
  int64_t nkb = (S + ORC_BLOCK - 1) / ORC_BLOCK;
  memset(resid, 0, (size_t)(nkb * ORC_BLOCK * D) * sizeof(float));
  memset(rcodes, 0, (size_t)(nkb * ORC_BLOCK * D));
  float* amax = (float*)calloc((size_t)D, sizeof(float));
  for (int64_t j = 0; j < nkb; ++j) {
    int64_t t0 = j * ORC_BLOCK, t1 = t0 + ORC_BLOCK < S ? t0 + ORC_BLOCK : S;
    for (int d = 0; d < D; ++d) {
      double s = 0.0;
      for (int64_t t = t0; t < t1; ++t) {
        int64_t src = perm ? perm[t] : t;
        s += bf16_to_f32(v[src * D + d]);
      }
      double m = subtract_mean ? s / (double)(t1 - t0) : 0.0;
      mu[j * D + d] = m;
      mub[j * D + d] = orc_f64_to_bf16(m);
    }
    for (int64_t t = t0; t < t1; ++t) {
      int64_t src = perm ? perm[t] : t;
      for (int d = 0; d < D; ++d) {
        float r = bf16_to_f32(v[src * D + d]) - bf16_to_f32(mub[j * D + d]);
        resid[t * D + d] = r;
        if (fabsf(r) > amax[d]) amax[d] = fabsf(r);
      }
    }
  }
  if (!per_channel) {  /* one scale over the whole head */
    float a = 0.0f;
    for (int d = 0; d < D; ++d) a = amax[d] > a ? amax[d] : a;
    for (int d = 0; d < D; ++d) amax[d] = a;
  }
  for (int d = 0; d < D; ++d) {
    float inv = amax[d] > 0.0f ? 448.0f / amax[d] : 1.0f;
    for (int64_t t = 0; t < S; ++t) rcodes[t * D + d] = orc_e4m3_encode(resid[t * D + d] * inv);
  }
  for (int d = 0; d < (per_channel ? D : 1); ++d) {
    amax_out[d] = amax[d];
    sv_out[d] = amax[d] > 0.0f ? amax[d] / 448.0f : 1.0f;
  }
  if (per_channel && mut)
    for (int64_t j = 0; j < nkb; ++j)
      for (int d = 0; d < D; ++d) mut[j * D + d] = orc_f64_to_bf16((double)(bf16_to_f32(mub[j * D + d]) / sv_out[d]));
  free(amax);
}

void orc_demean(const uint16_t* v, const int32_t* perm, int64_t S, int D, int subtract_mean, double* mu,
                uint16_t* mub, float* resid, uint8_t* rcodes, float* amax_out, float* sv_out) {
  orc_demean_ex(v, perm, S, D, subtract_mean, 0, mu, mub, NULL, resid, rcodes, amax_out, sv_out);
}

/* ---------------------------------------------------------------------------------------------
 * V residual repair selection ([OVC] "Why V residual repair"): with the residual quantised without
 * V-Smooth (R = V, one scale per head or per channel), every token j leaves the rounding residual
 * r_j,c = s_c (x_j,c - dec(E4M3(x_j,c))), x_j,c = fl32(v_j,c * inv_c); tokens are ranked by the residual
 * energy sum_c r_j,c^2 and the top n_rep kept.  Reading R18: the energy is taken in fp32 exactly as the
 * kernel does, t = fl32(s_c * (x - dec)) (the subtraction is exact) and e = fmaf(t, t, e) over
 * c = 0..D-1 in order; ties go to the lower token index; the kept tokens are listed in ascending
 * index order.  inv_c = 448/amax_c (1 if amax_c is 0), s_c = amax_c/448 (1 if 0), from the amax of
 * the residual quantiser (per head: all channels equal).
 * Outputs: idx [n_rep] ascending, energy [S] (may be NULL), rep [nrt*128, D] E4M3 codes of
 * (x - dec) for the kept tokens (code units of the main residual codes), pad rows 0. */
typedef struct {
  float e;
  int32_t j;
} orc_ej;

static int orc_cmp_energy(const void* a, const void* b) {
  const orc_ej* x = (const orc_ej*)a;
  const orc_ej* y = (const orc_ej*)b;
  if (x->e != y->e) return x->e > y->e ? -1 : 1;
  return x->j < y->j ? -1 : (x->j > y->j);
}

static int orc_cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return x < y ? -1 : (x > y);
}

void orc_repair_select(const uint16_t* v, int64_t S, int D, const float* amax, int64_t n_rep, int32_t* idx,
                       float* energy, uint8_t* rep) {
  float* inv = (float*)malloc((size_t)D * sizeof(float));
  float* sc = (float*)malloc((size_t)D * sizeof(float));
  for (int d = 0; d < D; ++d) {
    inv[d] = amax[d] > 0.0f ? 448.0f / amax[d] : 1.0f;
    sc[d] = amax[d] > 0.0f ? amax[d] / 448.0f : 1.0f;
  }
  orc_ej* all = (orc_ej*)malloc((size_t)(S > 0 ? S : 1) * sizeof(orc_ej));
  for (int64_t j = 0; j < S; ++j) {
    float e = 0.0f;
    for (int d = 0; d < D; ++d) {
      float x = bf16_to_f32(v[j * D + d]) * inv[d];
      float r = x - (float)orc_e4m3_decode(orc_e4m3_encode(x));
      float t = sc[d] * r;
      e = fmaf(t, t, e);
    }
    all[j].e = e;
    all[j].j = (int32_t)j;
    if (energy) energy[j] = e;
  }
  qsort(all, (size_t)S, sizeof(orc_ej), orc_cmp_energy);
  for (int64_t i = 0; i < n_rep; ++i) idx[i] = all[i].j;
  qsort(idx, (size_t)n_rep, sizeof(int32_t), orc_cmp_i32);
  int64_t rpad = (n_rep + ORC_BLOCK - 1) / ORC_BLOCK * ORC_BLOCK;
  memset(rep, 0, (size_t)(rpad * D));
  for (int64_t i = 0; i < n_rep; ++i)
    for (int d = 0; d < D; ++d) {
      float x = bf16_to_f32(v[(int64_t)idx[i] * D + d]) * inv[d];
      rep[i * D + d] = orc_e4m3_encode(x - (float)orc_e4m3_decode(orc_e4m3_encode(x)));
    }
  free(all);
  free(inv);
  free(sc);
}

/* Gather rows of a [S, D] bf16 tensor by pi: out[t] = x[pi[t]]  ([VC] §3.2 Eq. 3: K' = K[pi]). */
void orc_gather_rows(const uint16_t* x, const int32_t* perm, int64_t S, int D, uint16_t* out) {
  for (int64_t t = 0; t < S; ++t) memcpy(out + t * D, x + (int64_t)perm[t] * D, (size_t)D * 2);
}

/* ---------------------------------------------------------------------------------------------
 * Key visit order.  [OVC] "Scheduling around ExpCast", mid-window key traversal: start a few
 * blocks past the query's diagonal block, sweep down to block 0, then visit the tail; every block
 * once.  Reading R7: the pair of query tiles (2m, 2m+1) starts at block 2m+2, i.e. "a few" = 2 for
 * the even tile and 1 for the odd one.  midwindow = 0 gives the linear order 0..nkb-1.
 * ------------------------------------------------------------------------------------------- */
void orc_visit_order(int nkb, int qt, int midwindow, int32_t* order) {
  if (!midwindow) {
    for (int i = 0; i < nkb; ++i) order[i] = i;
    return;
  }
  const int pair_start = (qt / 2) * 2 + 2;
  int start = pair_start < nkb - 1 ? pair_start : nkb - 1;
  int n = 0;
  for (int j = start; j >= 0; --j) order[n++] = j;
  for (int j = start + 1; j < nkb; ++j) order[n++] = j;
}

/* ---------------------------------------------------------------------------------------------
 * (i) The quantised attention forward, one query row at a time.
 *   [VC] §3.1 Eq. 1 (online softmax), §3.2 Eq. 6 (online mean restoration
 *   A <- alpha A + P~ R_q + r mu^T, l <- alpha l + r, r = P~ 1), §3.3 Eq. 7 (ExpCast);
 *   [OVC] "Scheduling around ExpCast": running max on the true score, every increase applied with
 *   an output rescale, row sum of the decoded FP8 probabilities that feed PV, mid-window order.
 * Inputs (one batch-head): qc,kc,rc [S_pad, D] E4M3 codes (K and R already permuted), sq,sk [nkb],
 * sv the per-head residual scale, mub [nkb, D] bf16 means (NULL: no mean term).
 * flags: 1 = ExpCast (else exponentiate then cast), 2 = mid-window order (else linear), 4 = Q and K
 * rotated (R19).
 * rows: query token indices.  Outputs per row: out [D] fp64 = sv*A/l, l, final max M (code units).
 * ------------------------------------------------------------------------------------------- */
#define ORC_EXPCAST 1
#define ORC_MIDWINDOW 2
#define ORC_HADAMARD 4 /* Q and K were rotated (R19): the score constant carries 1/D more */

float orc_code_scale(int D) { return (float)(8.0 * 1.4426950408889634 / sqrt((double)D)); }
/* With rotated Q and K (R19) the scores carry a factor D. */
float orc_code_scale_rot(int D) { return (float)(8.0 * 1.4426950408889634 / ((double)D * sqrt((double)D))); }

/* svc: NULL (one residual scale sv per head, means mub in true units) or [D] per-channel scales with mut
 * the means already divided by them (R17): then the mean term is r_j * mut[j,d] and O[d] = svc[d] A[d] / l. */
/* V residual repair ([OVC] "Why V residual repair"), reading R18: n_rep extra key rows visited after
 * every regular tile, in tiles of 128 (kc_rep [nrt*128, D] codes of the copied keys with one scale per
 * repair tile sk_rep [nrt]; rc_rep [nrt*128, D] the E4M3 codes of the selected tokens' residuals in the
 * same code units as rc).  Their probabilities come from the same code formula with the running max M
 * left as it is (no update, no rescale; ExpCast clips at 120), they add P~ R to the numerator only,
 * and l is left unchanged.  n_rep = 0: no repair. */
void orc_attention_quant_rep(const uint8_t* qc, const float* sq, const uint8_t* kc, const float* sk,
                             const uint8_t* rc, float sv, const float* svc, const uint16_t* mub,
                             const uint16_t* mut, const uint8_t* kc_rep, const float* sk_rep, const uint8_t* rc_rep,
                             int64_t n_rep, int64_t S, int D, int flags, const int64_t* rows, int64_t nrows,
                             double* out, double* l_out, float* m_out) {
  int nrt = (int)((n_rep + ORC_BLOCK - 1) / ORC_BLOCK);
  int nkb = (int)((S + ORC_BLOCK - 1) / ORC_BLOCK);
  float C = (flags & ORC_HADAMARD) ? orc_code_scale_rot(D) : orc_code_scale(D);
#pragma omp parallel
  {
    int32_t* order = (int32_t*)malloc((size_t)nkb * sizeof(int32_t));
    double* A = (double*)malloc((size_t)D * sizeof(double));
    double* qd = (double*)malloc((size_t)D * sizeof(double));
    float s32[ORC_BLOCK];
    uint8_t code[ORC_BLOCK];
#pragma omp for schedule(dynamic, 1)
    for (int64_t ri = 0; ri < nrows; ++ri) {
      int64_t r = rows[ri];
      int qt = (int)(r / ORC_BLOCK);
      orc_visit_order(nkb, qt, flags & ORC_MIDWINDOW, order);
      for (int d = 0; d < D; ++d) qd[d] = orc_e4m3_decode(qc[r * D + d]);
      float aq = C * sq[qt];
      float M = -INFINITY;
      double l = 0.0;
      for (int d = 0; d < D; ++d) A[d] = 0.0;
      for (int oi = 0; oi < nkb; ++oi) {
        int j = order[oi];
        int ncols = (int)((int64_t)(j + 1) * ORC_BLOCK <= S ? ORC_BLOCK : S - (int64_t)j * ORC_BLOCK);
        float aj = aq * sk[j];
        /* raw score: exact in fp64 (at most 50 significant bits), then one rounding to fp32 */
        float t = -INFINITY;
        for (int c = 0; c < ncols; ++c) {
          const uint8_t* kr = kc + ((int64_t)j * ORC_BLOCK + c) * D;
          double acc = 0.0;
          for (int d = 0; d < D; ++d) acc += qd[d] * orc_e4m3_decode(kr[d]);
          s32[c] = (float)acc;
          float sc = s32[c] * aj;
          if (sc > t) t = sc;
        }
        float Mn = M > t ? M : t;
        if (Mn > M && M > -INFINITY) {
          double alpha = exp2(((double)M - (double)Mn) / 8.0);
          for (int d = 0; d < D; ++d) A[d] *= alpha;
          l *= alpha;
        }
        M = Mn;
        float b = ORC_B0 - M;
        double rj = 0.0;
        for (int c = 0; c < ncols; ++c) {
          if (flags & ORC_EXPCAST) {
            code[c] = (uint8_t)orc_expcast_code(s32[c], aj, b);
          } else {
            float y = fmaf(s32[c], aj, b);
            float ze = (y - ORC_B0) * 0.125f + 8.0f;
            code[c] = orc_e4m3_encode((float)exp2((double)ze));
          }
          rj += orc_e4m3_decode(code[c]);
        }
        for (int d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int c = 0; c < ncols; ++c)
            acc += orc_e4m3_decode(code[c]) * orc_e4m3_decode(rc[((int64_t)j * ORC_BLOCK + c) * D + d]);
          double mean_term = 0.0;
          if (mub && svc && mut) mean_term = rj * (double)bf16_to_f32(mut[(int64_t)j * D + d]);
          else if (mub) mean_term = rj * ((double)bf16_to_f32(mub[(int64_t)j * D + d]) / (double)sv);
          A[d] += acc + mean_term;
        }
        l += rj;
      }
      for (int jr = 0; jr < nrt; ++jr) {  /* repair tiles: numerator only, M kept */
        int ncols = (int)((int64_t)(jr + 1) * ORC_BLOCK <= n_rep ? ORC_BLOCK : n_rep - (int64_t)jr * ORC_BLOCK);
        float aj = aq * sk_rep[jr];
        float b = ORC_B0 - M;
        for (int c = 0; c < ncols; ++c) {
          const uint8_t* kr = kc_rep + ((int64_t)jr * ORC_BLOCK + c) * D;
          double acc = 0.0;
          for (int d = 0; d < D; ++d) acc += qd[d] * orc_e4m3_decode(kr[d]);
          float sc = (float)acc;
          if (flags & ORC_EXPCAST) {
            code[c] = (uint8_t)orc_expcast_code(sc, aj, b);
          } else {
            float y = fmaf(sc, aj, b);
            float ze = (y - ORC_B0) * 0.125f + 8.0f;
            code[c] = orc_e4m3_encode((float)exp2((double)ze));
          }
        }
        for (int d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int c = 0; c < ncols; ++c)
            acc += orc_e4m3_decode(code[c]) * orc_e4m3_decode(rc_rep[((int64_t)jr * ORC_BLOCK + c) * D + d]);
          A[d] += acc;
        }
      }
      for (int d = 0; d < D; ++d) out[ri * D + d] = (double)(svc ? svc[d] : sv) * A[d] / l;
      if (l_out) l_out[ri] = l;
      if (m_out) m_out[ri] = M;
    }
    free(order);
    free(A);
    free(qd);
  }
}

void orc_attention_quant_ex(const uint8_t* qc, const float* sq, const uint8_t* kc, const float* sk,
                            const uint8_t* rc, float sv, const float* svc, const uint16_t* mub, const uint16_t* mut,
                            int64_t S, int D, int flags, const int64_t* rows, int64_t nrows, double* out,
                            double* l_out, float* m_out) {
  orc_attention_quant_rep(qc, sq, kc, sk, rc, sv, svc, mub, mut, NULL, NULL, NULL, 0, S, D, flags, rows, nrows, out,
                          l_out, m_out);
}

void orc_attention_quant(const uint8_t* qc, const float* sq, const uint8_t* kc, const float* sk, const uint8_t* rc,
                         float sv, const uint16_t* mub, int64_t S, int D, int flags, const int64_t* rows,
                         int64_t nrows, double* out, double* l_out, float* m_out) {
  orc_attention_quant_ex(qc, sq, kc, sk, rc, sv, NULL, mub, NULL, S, D, flags, rows, nrows, out, l_out, m_out);
}

/* ---------------------------------------------------------------------------------------------
 * (ii) Exact softmax attention in fp64 on the unquantised, unpermuted inputs.
 * [VC] §3.1: S = Q K^T / sqrt(d), P = softmax(S), O = P V.  q,k,v: [S, D] bf16 bits.
 * ------------------------------------------------------------------------------------------- */
void orc_attention_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t S, int D,
                         const int64_t* rows, int64_t nrows, double* out) {
  double scale = 1.0 / sqrt((double)D);
#pragma omp parallel
  {
    double* s = (double*)malloc((size_t)S * sizeof(double));
#pragma omp for schedule(dynamic, 1)
    for (int64_t ri = 0; ri < nrows; ++ri) {
      int64_t r = rows[ri];
      double mx = -INFINITY;
      for (int64_t t = 0; t < S; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)bf16_to_f32(q[r * D + d]) * (double)bf16_to_f32(k[t * D + d]);
        s[t] = acc * scale;
        if (s[t] > mx) mx = s[t];
      }
      double den = 0.0;
      for (int64_t t = 0; t < S; ++t) {
        s[t] = exp(s[t] - mx);
        den += s[t];
      }
      for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t t = 0; t < S; ++t) acc += s[t] * (double)bf16_to_f32(v[t * D + d]);
        out[ri * D + d] = acc / den;
      }
    }
    free(s);
  }
}

/* ---------------------------------------------------------------------------------------------
 * The same tiled recurrence with every quantiser switched off, for the mean-restoration check of
 * [VC] §3.2 "Online mean restoration": scores exact (fp64, natural-log domain), probabilities the
 * exact exp, V' = R + 1 mu^T with R and mu kept in fp64.  It must reproduce (ii) to rounding.
 * q,k,v: [S, D] fp64 (K, V already permuted), perm unused here.
 * ------------------------------------------------------------------------------------------- */
void orc_attention_demeaned_exact(const double* q, const double* k, const double* v, int64_t S, int D, int flags,
                                  const int64_t* rows, int64_t nrows, double* out) {
  int nkb = (int)((S + ORC_BLOCK - 1) / ORC_BLOCK);
  double scale = 1.0 / sqrt((double)D);
  double* mu = (double*)malloc((size_t)nkb * D * sizeof(double));
  for (int j = 0; j < nkb; ++j) {
    int64_t t0 = (int64_t)j * ORC_BLOCK, t1 = t0 + ORC_BLOCK < S ? t0 + ORC_BLOCK : S;
    for (int d = 0; d < D; ++d) {
      double s = 0.0;
      for (int64_t t = t0; t < t1; ++t) s += v[t * D + d];
      mu[j * D + d] = s / (double)(t1 - t0);
    }
  }
#pragma omp parallel
  {
    int32_t* order = (int32_t*)malloc((size_t)nkb * sizeof(int32_t));
    double* A = (double*)malloc((size_t)D * sizeof(double));
    double p[ORC_BLOCK];
#pragma omp for schedule(dynamic, 1)
    for (int64_t ri = 0; ri < nrows; ++ri) {
      int64_t r = rows[ri];
      orc_visit_order(nkb, (int)(r / ORC_BLOCK), flags & ORC_MIDWINDOW, order);
      double m = -INFINITY, l = 0.0;
      for (int d = 0; d < D; ++d) A[d] = 0.0;
      for (int oi = 0; oi < nkb; ++oi) {
        int j = order[oi];
        int ncols = (int)((int64_t)(j + 1) * ORC_BLOCK <= S ? ORC_BLOCK : S - (int64_t)j * ORC_BLOCK);
        double tmax = -INFINITY;
        for (int c = 0; c < ncols; ++c) {
          double acc = 0.0;
          for (int d = 0; d < D; ++d) acc += q[r * D + d] * k[((int64_t)j * ORC_BLOCK + c) * D + d];
          p[c] = acc * scale;
          if (p[c] > tmax) tmax = p[c];
        }
        double mn = m > tmax ? m : tmax;
        double alpha = (m == -INFINITY) ? 0.0 : exp(m - mn);
        double rj = 0.0;
        for (int c = 0; c < ncols; ++c) {
          p[c] = exp(p[c] - mn);
          rj += p[c];
        }
        for (int d = 0; d < D; ++d) {
          double acc = 0.0;
          for (int c = 0; c < ncols; ++c)
            acc += p[c] * (v[((int64_t)j * ORC_BLOCK + c) * D + d] - mu[(int64_t)j * D + d]);
          A[d] = alpha * A[d] + acc + rj * mu[(int64_t)j * D + d];
        }
        l = alpha * l + rj;
        m = mn;
      }
      for (int d = 0; d < D; ++d) out[ri * D + d] = A[d] / l;
    }
    free(order);
    free(A);
  }
  free(mu);
}
