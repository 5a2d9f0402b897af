/*
 * lmoe_oracle.c -- plain, slow, obviously correct CPU oracle of the Stable Latent MoE
 * feed-forward layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file;
 * only the test-suite, the smoke check and the CPU-baseline leg of the benchmark do.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Precision: every step runs in IEEE double from the bf16 bit patterns of the inputs,
 * widened exactly, with no intermediate rounding -- except the routing decision (score,
 * threshold, top-K, gates), which is defined in fp32 so that a device implementation can
 * reproduce it bit for bit.  Build with -ffp-contract=off: the fp32 routing arithmetic must
 * not be fused by the compiler (fmaf is called explicitly where a fused op is meant).
 *
 * Sources (web pages on Kimi K3; none prints an equation, so each formula below is the
 * plainest reading of the words, and the readings are listed where they are made):
 *   [TPP]  "The 2.8-Trillion-Parameter Problem: Why Bigger Models Break the Old Playbook",
 *          aitrending.vip summary -- sections "TL;DR" and "Technical Details".
 *   [IK3]  the same title, "Part 1 of Inside Kimi K3" (Towards AI article, wpnews.pro copy) --
 *          its passages on Mixture of Experts, Stable LatentMoE, the stabilizers, and
 *          Quantile Balancing.
 *   [SU]   "苏神复盘 Kimi K3：896 个专家背后，藏着哪些关键技术取舍？" (daily-ai-frontier),
 *          "Merged summary", bullets "LatentMoE" and "Stable LatentMoE".
 *
 * Layout conventions: all matrices row-major; weights stored [out, in].
 *   x        [n, d]        bf16 bits      hidden state (7168 wide in K3)
 *   w_down   [L, d]        bf16 bits      latent down-projection (L = d/2)
 *   w_router [E, L]        bf16 bits      router
 *   w_gate   [E, I, L]     bf16 bits      routed expert gate branch
 *   w_value  [E, I, L]     bf16 bits      routed expert value branch
 *   w_edown  [E, L, I]     bf16 bits      routed expert down projection
 *   gamma    [L]           fp32           RMSNorm weight
 *   w_up     [d, L]        bf16 bits      up-projection back to the hidden width
 *   w_sgate  [S, Is, d]    bf16 bits      shared experts, gate branch
 *   w_svalue [S, Is, d]    bf16 bits      shared experts, value branch
 *   w_sdown  [S, d, Is]    bf16 bits      shared experts, down projection
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exactly (bf16 is the top half of an fp32). */
static double bf(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
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

/* ------------------------------------------------------------------------------------ */
/* Latent down-projection.  [TPP] Technical Details, "Stable Latent MoE with Compression":
 * the 7168-wide hidden state is projected to 3584 dimensions before routing; [IK3] Stable
 * LatentMoE passage: the projection happens first, experts then work in the latent.
 * No bias is mentioned anywhere, so none is used.
 *   lat[t, l] = sum_i x[t, i] * w_down[l, i]                                               */
void oracle_latent(int n, int d, int L, const uint16_t *x, const uint16_t *w_down,
                   double *lat) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    for (int l = 0; l < L; ++l) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += bf(x[(size_t)t * d + i]) * bf(w_down[(size_t)l * d + i]);
      lat[(size_t)t * L + l] = acc;
    }
  }
}

/* Router logits.  [IK3] Mixture-of-Experts passage: a lightweight router looks at each
 * token; [SU] LatentMoE bullet: routing happens in the latent space.  Reading: a linear
 * router without bias on the latent, z[t, e] = sum_l lat[t, l] * w_router[e, l].         */
void oracle_router_logits(int n, int L, int E, const double *lat, const uint16_t *w_router,
                          double *logits) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int l = 0; l < L; ++l)
        acc += lat[(size_t)t * L + l] * bf(w_router[(size_t)e * L + l]);
      logits[(size_t)t * E + e] = acc;
    }
  }
}

/* ------------------------------------------------------------------------------------ */
/* Router score s = sigmoid(z), in fp32, specified to the last bit.  The pages name no
 * score function; the reading is the logistic sigmoid.  So that routing decisions can be
 * reproduced exactly, the fp32 evaluation is fixed here step by step:
 *   1. clamp z to [-88, 88];  x = -z
 *   2. Cody-Waite range reduction (W. J. Cody and W. Waite, "Software Manual for the
 *      Elementary Functions", 1980): n = rint(fl(x * log2(e))),
 *      r = fma(-n, LN2_HI, x), r = fma(-n, LN2_LO, r), where LN2_HI = 22713/32768 has 15
 *      significant bits (so n * LN2_HI is exact for |n| <= 127) and LN2_LO = fl32(ln2 - LN2_HI)
 *   3. p = Taylor polynomial of exp(r) of degree 7, coefficients fl32(1/k!), by Horner's
 *      rule with one fma per step, highest degree first
 *   4. e = (p * 2^n1) * 2^n2 with n1 = n/2 (toward zero), n2 = n - n1 (both powers normal)
 *   5. s = 1 / (1 + e), each operation one IEEE round-to-nearest fp32 operation.        */
float oracle_sigmoid32(float z) {
  const float LOG2E = 0x1.715476p+0f;      /* fl32(1/ln 2) */
  const float LN2_HI = 0x1.62e4p-1f;       /* 22713/32768 */
  const float LN2_LO = 0x1.7f7d1cp-20f;    /* fl32(ln 2 - 22713/32768) */
  const float C7 = 0x1.a01a02p-13f;        /* fl32(1/5040) */
  const float C6 = 0x1.6c16c2p-10f;        /* fl32(1/720)  */
  const float C5 = 0x1.111112p-7f;         /* fl32(1/120)  */
  const float C4 = 0x1.555556p-5f;         /* fl32(1/24)   */
  const float C3 = 0x1.555556p-3f;         /* fl32(1/6)    */
  const float C2 = 0.5f, C1 = 1.0f, C0 = 1.0f;
  if (z > 88.0f) z = 88.0f;
  if (z < -88.0f) z = -88.0f;
  float x = -z;
  float t = x * LOG2E;
  float nf = rintf(t);
  float r = fmaf(-nf, LN2_HI, x);
  r = fmaf(-nf, LN2_LO, r);
  float p = C7;
  p = fmaf(p, r, C6);
  p = fmaf(p, r, C5);
  p = fmaf(p, r, C4);
  p = fmaf(p, r, C3);
  p = fmaf(p, r, C2);
  p = fmaf(p, r, C1);
  p = fmaf(p, r, C0);
  int n = (int)nf;
  int n1 = n / 2, n2 = n - n1;
  uint32_t b1 = (uint32_t)(n1 + 127) << 23, b2 = (uint32_t)(n2 + 127) << 23;
  float s1, s2;
  memcpy(&s1, &b1, 4);
  memcpy(&s2, &b2, 4);
  float e = (p * s1) * s2;
  float den = 1.0f + e;
  return 1.0f / den;
}

/* Decreases of the routing score between consecutive fp32 inputs, over every fp32 value in
 * [-88, 88] in increasing order (outside it the clamp makes the score constant): *one_ulp
 * counts steps down by exactly one ulp, *more counts larger ones.  The sequence of fp32
 * roundings is not monotone everywhere, so the k-th largest score of a set of logits need
 * not be the score of its k-th largest logit: selections are made on the scores. */
void oracle_sigmoid_decreases(long long *one_ulp, long long *more) {
  const uint32_t NEG = 0xC2B00000u; /* -88.0f */
  const uint32_t POS = 0x42B00000u; /* +88.0f */
  const long long nneg = (long long)(NEG - 0x80000000u) + 1; /* -88 ... -0 */
  const long long n = nneg + (long long)POS + 1;               /* ... +0 ... +88 */
  long long c1 = 0, c2 = 0;
#pragma omp parallel for schedule(static) reduction(+ : c1, c2)
  for (long long c = 0; c < 4096; ++c) {
    const long long i0 = n * c / 4096, i1 = n * (c + 1) / 4096;
    float prev = 0.0f;
    for (long long i = (i0 > 0 ? i0 - 1 : 0); i < i1; ++i) {
      const uint32_t bits = i < nneg ? NEG - (uint32_t)i : (uint32_t)(i - nneg);
      float z;
      memcpy(&z, &bits, 4);
      const float sc = oracle_sigmoid32(z);
      if (i >= i0 && i > 0 && sc < prev) {
        if (nextafterf(sc, 2.0f) == prev)
          ++c1;
        else
          ++c2;
      }
      prev = sc;
    }
  }
  *one_ulp = c1;
  *more = c2;
}

void oracle_scores(long long count, const float *logits, float *scores) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < count; ++i) scores[i] = oracle_sigmoid32(logits[i]);
}

static int cmp_float_desc(const void *a, const void *b) {
  float x = *(const float *)a, y = *(const float *)b;
  return (x < y) - (x > y);
}

/* Quantile-Balancing threshold.  [IK3] Quantile Balancing passage: the threshold is read
 * off the batch's score distribution -- the score an expert needs to stay within its fair
 * share of tokens; [SU] Stable LatentMoE bullet: it solves directly for per-expert Top-K
 * thresholds.  Reading: tau[e] = the k-th largest score in column e of the batch's score
 * matrix, k = max(1, floor(T*K/E)), at most T (the caller passes k).  Computed by sorting
 * each column in full.                                                                   */
void oracle_thresholds(int T, int E, int k, const float *logits, float *tau) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int e = 0; e < E; ++e) {
    float *col = (float *)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) col[t] = oracle_sigmoid32(logits[(size_t)t * E + e]);
    qsort(col, (size_t)T, sizeof(float), cmp_float_desc);
    tau[e] = (T > 0 && k >= 1 && k <= T) ? col[k - 1] : 0.0f;
    free(col);
  }
}

typedef struct {
  float a;
  int e;
} route_key;

/* Order: larger a first; equal a (IEEE equality, so -0 == +0) -> smaller expert id first. */
static int cmp_route(const void *pa, const void *pb) {
  const route_key *x = (const route_key *)pa, *y = (const route_key *)pb;
  if (x->a > y->a) return -1;
  if (x->a < y->a) return 1;
  return (x->e > y->e) - (x->e < y->e);
}

/* Top-K routing.  [TPP] Technical Details: a lightweight router selects 16 of the 896
 * routed experts per token; [SU]: Quantile Balancing replaces the bias updates of the
 * predecessor, so the thresholds take the bias's place.  Reading:
 *   a[t, e] = fl32(s[t, e] - tau[e])          (tau == NULL: no balancing, a = s)
 *   the K experts with the largest a, ties to the smaller expert id, listed in that order
 *   gate[t, j] = fl32(s_j / S), S = fl32 sum of the selected s in slot order j = 0..K-1.  */
void oracle_route(int T, int E, int K, const float *logits, const float *tau, int32_t *idx,
                  float *gate, float *scores) {
#pragma omp parallel for schedule(dynamic, 16)
  for (int t = 0; t < T; ++t) {
    route_key *keys = (route_key *)malloc(sizeof(route_key) * (size_t)E);
    float *s = (float *)malloc(sizeof(float) * (size_t)E);
    for (int e = 0; e < E; ++e) {
      s[e] = oracle_sigmoid32(logits[(size_t)t * E + e]);
      if (scores) scores[(size_t)t * E + e] = s[e];
      keys[e].a = tau ? (s[e] - tau[e]) : s[e];
      keys[e].e = e;
    }
    qsort(keys, (size_t)E, sizeof(route_key), cmp_route);
    float sum = 0.0f;
    for (int j = 0; j < K; ++j) sum = sum + s[keys[j].e];
    for (int j = 0; j < K; ++j) {
      idx[(size_t)t * K + j] = keys[j].e;
      gate[(size_t)t * K + j] = s[keys[j].e] / sum;
    }
    free(keys);
    free(s);
  }
}

/* ------------------------------------------------------------------------------------ */
/* SiTU-GLU.  [TPP] Technical Details, "Stabilization Mechanisms", and [IK3] stabilizers
 * passage: the gate and the value branch are smoothly capped to about +-100 in magnitude,
 * and the activation behaves like SwiGLU near zero; [SU] Stable LatentMoE bullet: it
 * soft-caps SwiGLU outliers.  Reading: each branch goes through c*tanh(./c), c = 100, and
 * the capped branches are combined as in SwiGLU:  silu(c tanh(g/c)) * c tanh(v/c).        */
double oracle_situ(double g, double v, double c) {
  double gc = c * tanh(g / c);
  double vc = c * tanh(v / c);
  return gc / (1.0 + exp(-gc)) * vc;
}

void oracle_situ_vec(long long count, const double *g, const double *v, double c,
                     double *out) {
  for (long long i = 0; i < count; ++i) out[i] = oracle_situ(g[i], v[i], c);
}

/* Routed experts in the latent, gate-weighted aggregation, RMSNorm.
 * [TPP] Technical Details: experts operate in the compressed latent space and their
 * outputs are projected back to full width; [IK3]: their outputs are combined, then
 * projected back up; RMSNorm sits right before the up-projection; [SU]: RMSNorm after
 * expert aggregation and before up-projection.
 *   h = SiTU(lat . Wg[e]^T, lat . Wv[e]^T)          [I]
 *   o = h . Wed[e]^T                                [L]
 *   u = sum_j gate[t, j] * o_j
 *   z = gamma * u / sqrt(mean(u^2) + eps)                                                  */
void oracle_routed(int n, int L, int E, int K, int I, const double *lat, const int32_t *idx,
                   const float *gate, const uint16_t *w_gate, const uint16_t *w_value,
                   const uint16_t *w_edown, const float *gamma, double c, double eps,
                   double *z) {
  (void)E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    double *u = (double *)calloc((size_t)L, sizeof(double));
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    const double *lt = lat + (size_t)t * L;
    for (int j = 0; j < K; ++j) {
      int e = idx[(size_t)t * K + j];
      double g = (double)gate[(size_t)t * K + j];
      const uint16_t *Wg = w_gate + (size_t)e * I * L;
      const uint16_t *Wv = w_value + (size_t)e * I * L;
      const uint16_t *Wd = w_edown + (size_t)e * L * I;
      for (int i = 0; i < I; ++i) {
        double ag = 0.0, av = 0.0;
        for (int l = 0; l < L; ++l) {
          ag += lt[l] * bf(Wg[(size_t)i * L + l]);
          av += lt[l] * bf(Wv[(size_t)i * L + l]);
        }
        h[i] = oracle_situ(ag, av, c);
      }
      for (int l = 0; l < L; ++l) {
        double o = 0.0;
        for (int i = 0; i < I; ++i) o += h[i] * bf(Wd[(size_t)l * I + i]);
        u[l] += g * o;
      }
    }
    double ms = 0.0;
    for (int l = 0; l < L; ++l) ms += u[l] * u[l];
    ms /= (double)L;
    double inv = 1.0 / sqrt(ms + eps);
    for (int l = 0; l < L; ++l) z[(size_t)t * L + l] = (double)gamma[l] * u[l] * inv;
    free(u);
    free(h);
  }
}

/* Shared experts.  [TPP] TL;DR and Technical Details: 2 shared experts next to the 896
 * routed ones; [SU] LatentMoE bullet: 2 always-on shared experts offset the latent
 * bottleneck.  Reading: they see the full-width hidden state (only the routed path is
 * compressed, [TPP] Technical Details) and use the same SiTU-GLU FFN form; every token
 * passes through every shared expert with weight 1.
 *   ys[t] = sum_s SiTU(x . Wsg[s]^T, x . Wsv[s]^T) . Wsd[s]^T                               */
void oracle_shared(int n, int d, int S, int Is, const uint16_t *x, const uint16_t *w_sgate,
                   const uint16_t *w_svalue, const uint16_t *w_sdown, double c, double *ys) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    double *h = (double *)malloc(sizeof(double) * (size_t)Is);
    double *out = ys + (size_t)t * d;
    for (int m = 0; m < d; ++m) out[m] = 0.0;
    for (int s = 0; s < S; ++s) {
      const uint16_t *Wg = w_sgate + (size_t)s * Is * d;
      const uint16_t *Wv = w_svalue + (size_t)s * Is * d;
      const uint16_t *Wd = w_sdown + (size_t)s * d * Is;
      for (int i = 0; i < Is; ++i) {
        double ag = 0.0, av = 0.0;
        for (int k = 0; k < d; ++k) {
          double xv = bf(x[(size_t)t * d + k]);
          ag += xv * bf(Wg[(size_t)i * d + k]);
          av += xv * bf(Wv[(size_t)i * d + k]);
        }
        h[i] = oracle_situ(ag, av, c);
      }
      for (int m = 0; m < d; ++m) {
        double acc = 0.0;
        for (int i = 0; i < Is; ++i) acc += h[i] * bf(Wd[(size_t)m * Is + i]);
        out[m] += acc;
      }
    }
    free(h);
  }
}

/* Up-projection and residual.  [TPP] Technical Details: outputs are projected back to
 * full width; the residual stream stays 7168 wide; [IK3] baseline decoder passage: the FFN
 * is wrapped in a residual connection.
 *   y[t, m] = residual[t, m] + sum_l z[t, l] * w_up[m, l] + ys[t, m]
 * (residual == NULL: no residual term).                                                   */
void oracle_output(int n, int d, int L, const double *z, const double *ys,
                   const uint16_t *w_up, const uint16_t *residual, double *y) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    for (int m = 0; m < d; ++m) {
      double acc = 0.0;
      for (int l = 0; l < L; ++l) acc += z[(size_t)t * L + l] * bf(w_up[(size_t)m * L + l]);
      double r = residual ? bf(residual[(size_t)t * d + m]) : 0.0;
      y[(size_t)t * d + m] = r + acc + ys[(size_t)t * d + m];
    }
  }
}

/* ------------------------------------------------------------------------------------ */
/* FP8 (e4m3) variant of the routed experts.  [SU] Stable LatentMoE bullet: SiTU-GLU
 * soft-caps the outliers that would otherwise blow up the BF16/FP8 dynamic range, i.e. the
 * routed experts are meant to run in FP8.  The pages give no quantisation recipe; the
 * reading used here (stated once, followed by both sides):
 *   - e4m3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; subnormal step 2^-9; largest
 *     finite 448; the code S.1111.111 is NaN; no infinities;
 *   - rounding to e4m3: to nearest, ties to an even mantissa; magnitudes above 448 (and
 *     infinities) saturate to 448; NaN -> NaN;
 *   - a row x (fp32 values) is quantised with one scale: amax = max |x|,
 *     s = fl32(amax / 448) (s = 1 when that is 0), q = e4m3(fl32(x / s)); x ~ q * s;
 *   - the routed GEMMs take quantised rows on both sides: each weight row (one output
 *     feature of one expert) and each activation row (the bf16 latent of a token; the
 *     bf16 SiTU output of one (token, expert) pair); products are summed and the sum is
 *     multiplied by both rows' scales.                                                      */

/* e4m3 code -> value (exact in double). */
double oracle_e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* fp32 -> nearest e4m3 code, ties to even, saturating. */
uint8_t oracle_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  uint8_t code;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal, code 0x08 */
    double q = nearbyint(a * 512.0); /* exact scaling; default rounding is to nearest even */
    code = (uint8_t)q;
  } else {
    int ex;
    frexp(a, &ex);  /* a = f * 2^ex, f in [0.5, 1) -> a in [2^(ex-1), 2^ex) */
    const int E = ex - 1;
    double q = nearbyint(ldexp(a, 3 - E)); /* in [8, 16]: 8 + mantissa, 16 = next binade */
    int Ef = E, mq = (int)q;
    if (mq == 16) {
      Ef += 1;
      mq = 8;
    }
    if (Ef > 8 || (Ef == 8 && mq > 14)) return sign | 0x7E; /* rounded past 448 */
    code = (uint8_t)(((Ef + 7) << 3) | (mq - 8));
  }
  return sign | code;
}

/* Quantise `rows` rows of `cols` fp32 values each: codes [rows, cols], scales [rows]. */
void oracle_quantize_rows(long long rows, int cols, const float *x, uint8_t *codes,
                          float *scales) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < rows; ++r) {
    const float *xr = x + (size_t)r * cols;
    float amax = 0.0f;
    for (int i = 0; i < cols; ++i) {
      const float a = fabsf(xr[i]);
      if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    if (!(s > 0.0f)) s = 1.0f;
    scales[r] = s;
    for (int i = 0; i < cols; ++i) codes[(size_t)r * cols + i] = oracle_e4m3_encode(xr[i] / s);
  }
}

/* double -> nearest bf16 value (ties to even), returned as the exact fp32 it is. */
float oracle_bf16_round(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return (float)x;
  int ex;
  frexp(x, &ex); /* |x| in [2^(ex-1), 2^ex) */
  double q = nearbyint(ldexp(x, 8 - ex)); /* 8 significant bits */
  return (float)ldexp(q, ex - 8);
}

/* Relative distance of x from the nearest bf16 rounding tie (the midpoint between two
 * neighbouring bf16 values).  Small values mean that a slightly different evaluation of x
 * may round to the other neighbour. */
double oracle_bf16_tie_distance(double x) {
  if (x == 0.0 || isnan(x) || isinf(x)) return INFINITY;
  int ex;
  frexp(x, &ex);
  const double ulp = ldexp(1.0, ex - 8);          /* bf16 spacing at |x| */
  const double a = fabs(x);
  const double lo = floor(a / ulp) * ulp;          /* bf16 neighbour below |x| */
  return fabs(a - (lo + 0.5 * ulp)) / a;
}

/* 1 when the scale of a row of values (quantised from their bf16 roundings) depends on a
 * near-tie: some element within 2^-6 of the row's largest bf16 magnitude lies within
 * `margin` (relative) of a bf16 rounding tie, so that an evaluation of the row that differs
 * in the last fp32 bits may pick another amax, another scale, and other codes. */
static int scale_near_tie(const double *x, int n, double margin) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float a = fabsf(oracle_bf16_round(x[i]));
    if (a > amax) amax = a;
  }
  for (int i = 0; i < n; ++i)
    if (fabs(x[i]) >= (double)amax * (1.0 - ldexp(1.0, -6)) &&
        oracle_bf16_tie_distance(x[i]) < margin)
      return 1;
  return 0;
}

/* Routed experts with e4m3 operands, aggregation and RMSNorm (the fp8 reading above).
 * Weights arrive quantised: qg, qv [E, I, L] with sg, sv [E, I]; qd [E, L, I] with sd [E, L].
 * The latent row of a token is rounded to bf16 and quantised; the SiTU output of each
 * (token, expert) pair is rounded to bf16 and quantised; everything else is fp64.
 *   g_i = sg_i * s_lat * sum_l dq(qg_il) dq(q_lat_l)     (v likewise)
 *   h_i = SiTU(g_i, v_i);  q_h, s_h = quantise(bf16(h))
 *   o_l = sd_l * s_h * sum_i dq(qd_li) dq(q_h_i);  u = sum_j gate_j o_j;  z = RMSNorm(u)   */
void oracle_routed_fp8(int n, int L, int E, int K, int I, const double *lat,
                       const int32_t *idx, const float *gate, const uint8_t *qg,
                       const float *sg, const uint8_t *qv, const float *sv,
                       const uint8_t *qd, const float *sd, const float *gamma, double c,
                       double eps, double *z, int32_t *scale_ties, double tie_margin) {
  (void)E;
  double dq[256];
  for (int i = 0; i < 256; ++i) dq[i] = oracle_e4m3_decode((uint8_t)i);
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t) {
    double *u = (double *)calloc((size_t)L, sizeof(double));
    float *row = (float *)malloc(sizeof(float) * (size_t)(L > I ? L : I));
    double *hx = (double *)malloc(sizeof(double) * (size_t)I);
    uint8_t *ql = (uint8_t *)malloc((size_t)L);
    uint8_t *qh = (uint8_t *)malloc((size_t)I);
    float s_lat, s_h;
    int ties = scale_near_tie(lat + (size_t)t * L, L, tie_margin);
    for (int l = 0; l < L; ++l) row[l] = oracle_bf16_round(lat[(size_t)t * L + l]);
    oracle_quantize_rows(1, L, row, ql, &s_lat);
    for (int j = 0; j < K; ++j) {
      const int e = idx[(size_t)t * K + j];
      const double g = (double)gate[(size_t)t * K + j];
      for (int i = 0; i < I; ++i) {
        const size_t wr = (size_t)e * I + i;
        double ag = 0.0, av = 0.0;
        for (int l = 0; l < L; ++l) {
          ag += dq[qg[wr * L + l]] * dq[ql[l]];
          av += dq[qv[wr * L + l]] * dq[ql[l]];
        }
        ag *= (double)sg[wr] * (double)s_lat;
        av *= (double)sv[wr] * (double)s_lat;
        hx[i] = oracle_situ(ag, av, c);
        row[i] = oracle_bf16_round(hx[i]);
      }
      ties += scale_near_tie(hx, I, tie_margin);
      oracle_quantize_rows(1, I, row, qh, &s_h);
      for (int l = 0; l < L; ++l) {
        const size_t wr = (size_t)e * L + l;
        double o = 0.0;
        for (int i = 0; i < I; ++i) o += dq[qd[wr * I + i]] * dq[qh[i]];
        u[l] += g * o * (double)sd[wr] * (double)s_h;
      }
    }
    double ms = 0.0;
    for (int l = 0; l < L; ++l) ms += u[l] * u[l];
    ms /= (double)L;
    const double inv = 1.0 / sqrt(ms + eps);
    for (int l = 0; l < L; ++l) z[(size_t)t * L + l] = (double)gamma[l] * u[l] * inv;
    if (scale_ties) scale_ties[t] = ties;
    free(u);
    free(row);
    free(hx);
    free(ql);
    free(qh);
  }
}

/* ------------------------------------------------------------------------------------ */
/* Streaming thresholds.  [IK3] Quantile Balancing passage: thresholds are read off the
 * distribution of the router scores at each step.  A threshold that persists across steps
 * (for decode batches too small to carry a quantile, or to damp step-to-step noise) is the
 * exponential moving average of the per-step thresholds -- a reading; the pages do not
 * name one.  In fp32, one subtraction and one fused multiply-add:
 *   tau_ema <- fma(beta, tau_ema - tau_step, tau_step)   (= beta tau_ema + (1-beta) tau_step)
 * and on the first step tau_ema <- tau_step.                                              */
void oracle_tau_ema(int E, float beta, int first, const float *tau_step, float *tau_ema) {
  for (int e = 0; e < E; ++e)
    tau_ema[e] = first ? tau_step[e] : fmaf(beta, tau_ema[e] - tau_step[e], tau_step[e]);
}

/* Load statistics over steps ([IK3]: the balancing exists so that no expert sits idle while
 * a few monopolise the traffic).  acc, 64-bit counters (4 + 4E), updated from one step's
 * per-expert token counts:
 *   acc[0] steps, acc[1] routed pairs, acc[2] sum over steps of max_e count,
 *   acc[3] largest count of any expert in any step,
 *   acc[4 + e] sum of counts of e, acc[4 + E + e] sum of squared counts of e,
 *   acc[4 + 2E + e] steps in which e received no token, acc[4 + 3E + e] largest count of e. */
void oracle_load_stats_update(int E, const int32_t *counts, unsigned long long *acc) {
  unsigned long long pairs = 0, mx = 0;
  for (int e = 0; e < E; ++e) {
    const unsigned long long c = (unsigned long long)counts[e];
    pairs += c;
    if (c > mx) mx = c;
    acc[4 + e] += c;
    acc[4 + E + e] += c * c;
    acc[4 + 2 * E + e] += c == 0 ? 1 : 0;
    if (c > acc[4 + 3 * E + e]) acc[4 + 3 * E + e] = c;
  }
  acc[0] += 1;
  acc[1] += pairs;
  acc[2] += mx;
  if (mx > acc[3]) acc[3] = mx;
}

/* ------------------------------------------------------------------------------------ */
/* Expert-parallel dispatch and combine (the pages' layout, on one device).  [IK3] Stable
 * LatentMoE and communication passages: experts live on different GPUs, each selected
 * expert receives the token's (latent) vector, and the outputs travel back to be combined;
 * compressing before the trip halves the bytes.  [TPP] Technical Details: 7168 -> 3584.
 * Readings: R ranks host the E experts in equal contiguous blocks (expert e on rank
 * e / (E/R)); a token's row travels once to every rank hosting at least one of its experts
 * (with the mask of its slots served there); the expert side returns one row per such
 * (token, rank) pair, the gate-weighted sum of its slots' outputs; the source sums the
 * returned rows. */

/* Dispatch: pairs (token, rank) in (rank, token) order.  send_off [R + 1], send_tok [P],
 * send_slots [P] (bit j: slot j of the token goes to that rank), send_rows [P, W] (copies of
 * the token's row, bf16 bits).  Returns P. */
long long oracle_ep_dispatch(int T, int K, int E, int R, const int32_t *idx, int W,
                             const uint16_t *rows, int32_t *send_off, int32_t *send_tok,
                             uint32_t *send_slots, uint16_t *send_rows) {
  const int per = E / R;
  long long p = 0;
  for (int r = 0; r < R; ++r) {
    send_off[r] = (int32_t)p;
    for (int t = 0; t < T; ++t) {
      uint32_t slots = 0;
      for (int j = 0; j < K; ++j)
        if (idx[(size_t)t * K + j] / per == r) slots |= 1u << j;
      if (!slots) continue;
      send_tok[p] = t;
      send_slots[p] = slots;
      if (send_rows) memcpy(send_rows + (size_t)p * W, rows + (size_t)t * W, sizeof(uint16_t) * W);
      ++p;
    }
  }
  send_off[R] = (int32_t)p;
  return p;
}

/* Combine, expert side: for each pair p, part[p] = bf16(sum over its slots j, ascending, of
 * gate[t, j] * o_j accumulated in fp32 by fused multiply-adds), where o_j is the row
 * o[inv[t, j]] (bf16 bits).  Source side: u[t] = sum over its pairs in rank order of the
 * returned rows, in fp32. */
static uint16_t f32_to_bf16_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)(u >> 16 | ((u & 0xFFFF) ? 0x40 : 0));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void oracle_ep_combine(int T, int K, long long P, const int32_t *send_tok,
                       const uint32_t *send_slots, const int32_t *inv, const float *gate,
                       int W, const uint16_t *o, uint16_t *part, float *u) {
  for (long long p = 0; p < P; ++p) {
    const int t = send_tok[p];
    for (int w = 0; w < W; ++w) {
      float acc = 0.0f;
      for (int j = 0; j < K; ++j)
        if (send_slots[p] >> j & 1u)
          acc = fmaf(gate[(size_t)t * K + j], (float)bf(o[(size_t)inv[(size_t)t * K + j] * W + w]),
                     acc);
      part[(size_t)p * W + w] = f32_to_bf16_rn(acc);
    }
  }
  for (size_t i = 0; i < (size_t)T * W; ++i) u[i] = 0.0f;
  for (long long p = 0; p < P; ++p) { /* pairs are in rank order, so each u[t] sums ranks in order */
    const int t = send_tok[p];
    for (int w = 0; w < W; ++w) u[(size_t)t * W + w] += (float)bf(part[(size_t)p * W + w]);
  }
}
