/*
 * attn_oracle.c -- plain fp64 CPU oracle for ragged GQA attention with its
 * full vector-Jacobian product.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes (the plain definition; one sequence b, query head h,
 * local query position i in [0, Lq), local key position j in [0, Lk); the
 * Hq query heads share Hkv key/value heads, query head h reading K/V head
 * g(h) = floor(h / (Hq / Hkv)), so consecutive query heads form a group):
 *
 *   s_ij  = sigma * sum_f q[i,h,f] k[j,g(h),f],  sigma = scale_multiplier/sqrt(d)
 *           ("Noncausal Global Extreme-GQA Ragged Attention Full VJP",
 *            section "What You Have": scaled logits use 0.75/sqrt(head_dim))
 *   t_ij  = c * tanh(s_ij / c)   (c = softcap; t = s when c <= 0)
 *           (same page, "Hard Constraints": the soft cap acts on the scaled
 *            dot product before ALiBi and before masking)
 *   z_ij  = t_ij - slope[b,h] * |i + Lk - Lq - j|
 *           (same page, "What You Have": the ALiBi distance)
 *   z_ij  = -inf where the mask forbids (i, j)
 *   lse_i = log sum_j exp(z_ij)                (natural log)
 *   P_ij  = exp(z_ij - lse_i);  out_i = sum_j P_ij v_j,g(h)
 *   D_i   = dO_i . out_i
 *   dP_ij = dO_i . v_j,g(h);   dZ_ij = P_ij (dP_ij - D_i)
 *   dS_ij = dZ_ij * (1 - (t_ij/c)^2)   (dZ_ij when c <= 0)
 *   dq_i  = sigma sum_j dS_ij k_j,g(h)
 *   dk_j,g = sigma sum_{h: g(h)=g} sum_i dS_ij q_i   (h outer, i inner)
 *   dv_j,g = sum_{h: g(h)=g} sum_i P_ij dO_i         (h outer, i inner)
 *
 * With Hkv = 1 (the pages' case, "Hard Constraints": one K/V head shared by
 * every query head) g(h) = 0 and dk/dv sum over all heads.  The grouping of
 * consecutive query heads for Hkv > 1 is the usual grouped-query reading;
 * the pages fix only Hkv = 1.
 *
 * Dropout (optional; "ragged flash attention gradient recompute", "Root
 * causes addressed": a counter-based splitmix64 hash of (seed, b, h, row,
 * col), independent of tiling, with one rate or one rate per row):
 *   K_b    = splitmix64(seed ^ b)
 *   x_hij  = splitmix64(K_b ^ (h << 48 | i << 24 | floor(j / 4)))  (i, j local
 *            positions below 2^24, h below 2^16: one hash per four keys)
 *   u_hij  = the 16-bit field j mod 4 of x_hij, (x_hij >> 16 (j mod 4)) & 0xFFFF
 *   keep   = u_ij >= T,  T = (uint32)(rate * 2^16) in fp32 (2^16 when
 *            rate >= 1),  scale = 1 / (1 - rate)  (0 when rate >= 1)
 *   with rate = the call's rate, or rates[token] per query token when given.
 *   out_i  = sum_j P_ij keep_ij scale v_j     (lse and P undropped)
 *   dZ_ij  = P_ij (keep_ij scale dP_ij - D_i),  dv_j += P_ij keep_ij scale dO_i
 *   (D_i = dO_i . out_i of the dropped out, as above).
 *
 * Gate (optional; "Pairwise-Gated Attention Engine", "Why it is hard": each
 * query-key pair also gets a sigmoid gate from separate low-dimensional
 * projections that scales the softmax weight after normalisation):
 *   G_ij = 1 / (1 + exp(-qg_i . kg_j,g(h) / sqrt(R)))    (qg, kg of width R)
 *   out_i = sum_j P_ij G_ij (keep scale)_ij v_j
 *   dW_ij = dO_i . v_j;  dZ_ij = P_ij (G_ij (keep scale)_ij dW_ij - D_i)
 *   dg_ij = dW_ij P_ij (keep scale)_ij G_ij (1 - G_ij)
 *   dqg_i = sum_j dg_ij kg_j / sqrt(R);  dkg_j = sum_h sum_i dg_ij qg_i / sqrt(R)
 *   dv_j += P_ij G_ij (keep scale)_ij dO_i;  D_i = dO_i . out_i as before.
 *
 * Rows with no admissible key ("ragged flash attention gradient recompute",
 * "Root causes addressed", empty rows) have lse = -inf, out = 0, and add
 * nothing to any gradient.
 *
 * Mask reading (the pages accept causal/window arguments but never define
 * them): with k0 = i + Lk - Lq, key j is admissible iff
 *   (wl < 0 or j >= k0 - wl) and (wr' < 0 or j <= k0 + wr'),
 * where wr' = 0 when causal, else wr.
 *
 * The inputs are fp16 or bf16 bit patterns (or, for finite-difference checks,
 * doubles) read through their strides and decoded exactly to double by the
 * converters below; every later step is double precision.  Work is spread over POSIX threads, but every sum is taken
 * in the fixed order written above, so results do not depend on the thread
 * count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---- exact decoding of the 16-bit input formats ---------------------- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    mag = m ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16: the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---- problem description --------------------------------------------- */

typedef struct {
  int dtype; /* 0 = fp16, 1 = bf16, 2 = fp64 */
  int B, Hq, Hkv, d;
  const void *q;
  int64_t q_ts, q_hs;
  const void *k;
  int64_t k_ts, k_hs;
  const void *v;
  int64_t v_ts, v_hs;
  const void *dout;
  int64_t do_ts, do_hs;
  const int32_t *cu_q, *cu_k;
  const float *slopes; /* [B, Hq] with batch stride; NULL means all zero */
  int64_t slopes_bs;
  int causal, wl, wr;
  double softcap, scale_multiplier;
  int dropout;               /* 0: none */
  uint64_t seed;
  float rate;                /* used when rates is NULL */
  const float *rates;        /* per query token [total_q], or NULL */
  int R;                     /* gate width; 0: no gate */
  const void *qg;            /* [T_q][Hq][R] with strides */
  int64_t qg_ts, qg_hs;
  const void *kg;            /* [T_k][Hkv][R] with strides */
  int64_t kg_ts, kg_hs;
} problem;

/* ---- counter-based dropout ------------------------------------------- */

/* SplitMix64's output function (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014): a Weyl increment, then two
 * xor-shift-multiply rounds and a final xor-shift. */
static uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Threshold of a 16-bit draw and scale of a dropout rate (fp32 rate, as the
 * caller gives it). */
static void drop_params(float rate, uint32_t *T, double *scale) {
  if (!(rate < 1.0f)) {
    *T = 1u << 16;
    *scale = 0.0;
    return;
  }
  if (!(rate > 0.0f)) {
    *T = 0;
    *scale = 1.0;
    return;
  }
  *T = (uint32_t)(rate * 65536.0f);
  *scale = 1.0 / (1.0 - (double)rate);
}

/* The dropout factor keep * scale of element (b, h, i, j); 1 without dropout.
 * `token` is the packed query token (for per-token rates).  One SplitMix64
 * output serves the four keys 4m .. 4m + 3 of a row: key j takes the 16-bit
 * field j mod 4 (bits 16 (j mod 4) and up). */
static double drop_factor(const problem *p, int b, int h, int64_t token, int i, int j) {
  if (!p->dropout) return 1.0;
  const float rate = p->rates ? p->rates[token] : p->rate;
  uint32_t T;
  double scale;
  drop_params(rate, &T, &scale);
  const uint64_t kb = splitmix64(p->seed ^ (uint64_t)b);
  const uint64_t x = splitmix64(kb ^ (((uint64_t)h << 48) | ((uint64_t)(uint32_t)i << 24) |
                                      (uint64_t)((uint32_t)j >> 2)));
  const uint32_t u = (uint32_t)(x >> (16 * (j & 3))) & 0xFFFFu;
  return u >= T ? scale : 0.0;
}

/* Element idx (in elements, strides already applied) of input array a. */
static double decode(const problem *p, const void *a, int64_t idx) {
  if (p->dtype == 2) return ((const double *)a)[idx];
  uint16_t x = ((const uint16_t *)a)[idx];
  return p->dtype == 1 ? bf16_bits_to_double(x) : half_bits_to_double(x);
}

/* Decoded rows, gathered once per sequence so the inner loops stay plain. */
typedef struct {
  const problem *p;
  int b, Lq, Lk;
  int64_t q0, k0;     /* first packed token of the sequence */
  double *Q;          /* [Lq][Hq][d] */
  double *dO;         /* [Lq][Hq][d] */
  double *K, *V;      /* [Lk][Hkv][d] */
  double *Qg, *Kg;    /* [Lq][Hq][R], [Lk][Hkv][R] (NULL without a gate) */
} seqdata;

/* The K/V head that query head h reads. */
static int kv_head(const problem *p, int h) { return h / (p->Hq / p->Hkv); }

/* Decoded K (or V) row of key j, K/V head g. */
static const double *kv_row(const seqdata *s, const double *a, int j, int g) {
  return a + ((size_t)j * s->p->Hkv + g) * s->p->d;
}

static void seq_load(const problem *p, int b, seqdata *s) {
  int d = p->d, H = p->Hq;
  s->p = p;
  s->b = b;
  s->q0 = p->cu_q[b];
  s->k0 = p->cu_k[b];
  s->Lq = p->cu_q[b + 1] - p->cu_q[b];
  s->Lk = p->cu_k[b + 1] - p->cu_k[b];
  s->Q = malloc(sizeof(double) * ((size_t)s->Lq * H * d + 1));
  s->dO = malloc(sizeof(double) * ((size_t)s->Lq * H * d + 1));
  s->K = malloc(sizeof(double) * ((size_t)s->Lk * p->Hkv * d + 1));
  s->V = malloc(sizeof(double) * ((size_t)s->Lk * p->Hkv * d + 1));
  for (int i = 0; i < s->Lq; i++)
    for (int h = 0; h < H; h++)
      for (int f = 0; f < d; f++) {
        int64_t t = s->q0 + i;
        s->Q[((size_t)i * H + h) * d + f] = decode(p, p->q, t * p->q_ts + h * p->q_hs + f);
        s->dO[((size_t)i * H + h) * d + f] = decode(p, p->dout, t * p->do_ts + h * p->do_hs + f);
      }
  for (int j = 0; j < s->Lk; j++)
    for (int g = 0; g < p->Hkv; g++)
      for (int f = 0; f < d; f++) {
        int64_t t = s->k0 + j;
        size_t at = ((size_t)j * p->Hkv + g) * d + f;
        s->K[at] = decode(p, p->k, t * p->k_ts + g * p->k_hs + f);
        s->V[at] = decode(p, p->v, t * p->v_ts + g * p->v_hs + f);
      }
  s->Qg = s->Kg = NULL;
  if (p->R > 0) {
    const int R = p->R;
    s->Qg = malloc(sizeof(double) * ((size_t)s->Lq * H * R + 1));
    s->Kg = malloc(sizeof(double) * ((size_t)s->Lk * p->Hkv * R + 1));
    for (int i = 0; i < s->Lq; i++)
      for (int h = 0; h < H; h++)
        for (int f = 0; f < R; f++)
          s->Qg[((size_t)i * H + h) * R + f] =
              decode(p, p->qg, (s->q0 + i) * p->qg_ts + h * p->qg_hs + f);
    for (int j = 0; j < s->Lk; j++)
      for (int g = 0; g < p->Hkv; g++)
        for (int f = 0; f < R; f++)
          s->Kg[((size_t)j * p->Hkv + g) * R + f] =
              decode(p, p->kg, (s->k0 + j) * p->kg_ts + g * p->kg_hs + f);
  }
}

/* The gate of query row (i, h) and key j of K/V head kh (1 without a gate). */
static double gate_of(const seqdata *s, int h, int i, int j, int kh) {
  const problem *p = s->p;
  if (p->R == 0) return 1.0;
  const double *qg = s->Qg + ((size_t)i * p->Hq + h) * p->R;
  const double *kg = s->Kg + ((size_t)j * p->Hkv + kh) * p->R;
  double g = 0.0;
  for (int f = 0; f < p->R; f++) g += qg[f] * kg[f];
  g /= sqrt((double)p->R);
  return 1.0 / (1.0 + exp(-g));
}

static void seq_free(seqdata *s) {
  free(s->Q);
  free(s->dO);
  free(s->K);
  free(s->V);
  free(s->Qg);
  free(s->Kg);
}

static int admissible(const problem *p, int Lq, int Lk, int i, int j) {
  long k0 = (long)i + Lk - Lq;
  int wr = p->causal ? 0 : p->wr;
  if (p->wl >= 0 && (long)j < k0 - p->wl) return 0;
  if (wr >= 0 && (long)j > k0 + wr) return 0;
  return 1;
}

static double slope_of(const problem *p, int b, int h) {
  return p->slopes ? (double)p->slopes[(int64_t)b * p->slopes_bs + h] : 0.0;
}

/* Logit of (i, h) against key j of K/V head kh before masking: returns z,
 * and the softcap derivative factor 1 - (t/c)^2 through *g. */
static double logit(const seqdata *s, const double *qi, int i, int j, int kh, double slope,
                    double *g) {
  const problem *p = s->p;
  int d = p->d;
  const double *kj = kv_row(s, s->K, j, kh);
  double dot = 0.0;
  for (int f = 0; f < d; f++) dot += qi[f] * kj[f];
  double sigma = p->scale_multiplier / sqrt((double)d);
  double sc = sigma * dot;
  double t;
  if (p->softcap > 0.0) {
    double th = tanh(sc / p->softcap);
    t = p->softcap * th;
    *g = 1.0 - th * th;
  } else {
    t = sc;
    *g = 1.0;
  }
  double dist = fabs((double)((long)i + s->Lk - s->Lq - j));
  return t - slope * dist;
}

/* ---- per-row pass: out, lse, D, dq and row diagnostics ----------------- */

typedef struct {
  double *out, *lse, *dq, *Dpre; /* out/dq [T_q][Hq][d]; lse/Dpre [T_q][Hq] */
  double *dz_rowsum, *p_rowsum;  /* optional [T_q][Hq] */
  double *dk, *dv;               /* [T_k][Hkv][d] */
  double *dqg, *dkg;             /* [T_q][Hq][R], [T_k][Hkv][R] with a gate */
} outputs;

/* Where one query row's results go. */
typedef struct {
  double *out, *dq; /* [d] each */
  double *lse, *D;
  double *dz_sum, *p_sum; /* optional */
  double *dqg;            /* [R] with a gate, else NULL */
  int stats_only;         /* stop after lse, out and D (no dq): feeds a key pass */
} rowdest;

/* One query row (i, h) of sequence s, whose decoded q and dO rows are qi and
 * dOi.  z, P, gv are caller scratch of length >= Lk. */
static void row_pass(const seqdata *s, int h, int i, const double *qi, const double *dOi,
                     const rowdest *o, double *z, double *P, double *gv) {
  const problem *p = s->p;
  int d = p->d, Lk = s->Lk;
  double slope = slope_of(p, s->b, h);
  int kh = kv_head(p, h);
  double m = -INFINITY;
  for (int j = 0; j < Lk; j++) {
    z[j] = logit(s, qi, i, j, kh, slope, &gv[j]);
    if (!admissible(p, s->Lq, Lk, i, j)) z[j] = -INFINITY;
    if (z[j] > m) m = z[j];
  }
  for (int f = 0; f < d; f++) {
    o->out[f] = 0.0;
    if (o->dq) o->dq[f] = 0.0;
  }
  for (int f = 0; o->dqg && f < p->R; f++) o->dqg[f] = 0.0;
  if (m == -INFINITY) { /* empty row */
    *o->lse = -INFINITY;
    *o->D = 0.0;
    if (o->dz_sum) *o->dz_sum = 0.0;
    if (o->p_sum) *o->p_sum = 0.0;
    return;
  }
  double l = 0.0;
  for (int j = 0; j < Lk; j++) l += exp(z[j] - m);
  double lse = m + log(l);
  *o->lse = lse;
  double psum = 0.0;
  for (int j = 0; j < Lk; j++) {
    P[j] = exp(z[j] - lse);
    psum += P[j];
  }
  const int64_t token = s->q0 + i;
  for (int j = 0; j < Lk; j++) {
    const double pd = P[j] * gate_of(s, h, i, j, kh) * drop_factor(p, s->b, h, token, i, j);
    for (int f = 0; f < d; f++) o->out[f] += pd * kv_row(s, s->V, j, kh)[f];
  }
  double D = 0.0;
  for (int f = 0; f < d; f++) D += dOi[f] * o->out[f];
  *o->D = D;
  if (o->stats_only) return;
  double dzsum = 0.0;
  double sigma = p->scale_multiplier / sqrt((double)d);
  for (int j = 0; j < Lk; j++) {
    double dp = 0.0;
    for (int f = 0; f < d; f++) dp += dOi[f] * kv_row(s, s->V, j, kh)[f];
    const double fd = drop_factor(p, s->b, h, token, i, j);
    const double G = gate_of(s, h, i, j, kh);
    double dz = P[j] * (G * fd * dp - D);
    dzsum += dz;
    double ds = dz * gv[j];
    for (int f = 0; f < d; f++) o->dq[f] += sigma * ds * kv_row(s, s->K, j, kh)[f];
    if (o->dqg) {
      const double dg = dp * P[j] * fd * G * (1.0 - G) / sqrt((double)p->R);
      const double *kg = s->Kg + ((size_t)j * p->Hkv + kh) * p->R;
      for (int f = 0; f < p->R; f++) o->dqg[f] += dg * kg[f];
    }
  }
  if (o->dz_sum) *o->dz_sum = dzsum;
  if (o->p_sum) *o->p_sum = psum;
}

/* Row pass for row i of every head of a loaded sequence, into the packed
 * output arrays. */
static void row_pass_packed(const seqdata *s, int h, int i, const outputs *o, double *z,
                            double *P, double *gv) {
  int d = s->p->d, H = s->p->Hq;
  int64_t rowid = (s->q0 + i) * (int64_t)H + h;
  rowdest r = {o->out + rowid * d, o->dq ? o->dq + rowid * d : NULL, o->lse + rowid,
               o->Dpre + rowid,
               o->dz_rowsum ? o->dz_rowsum + rowid : NULL,
               o->p_rowsum ? o->p_rowsum + rowid : NULL,
               o->dqg ? o->dqg + rowid * s->p->R : NULL, o->dq == NULL};
  const double *qi = s->Q + ((size_t)i * H + h) * d;
  const double *dOi = s->dO + ((size_t)i * H + h) * d;
  row_pass(s, h, i, qi, dOi, &r, z, P, gv);
}

/* ---- per-key pass: dk, dv (needs every row's lse and D) ---------------- */

/* Key j of K/V head kh: sums over the query heads of its group, into the
 * rows dkrow, dvrow (and dkgrow with a gate). */
static void key_pass_to(const seqdata *s, int j, int kh, const outputs *o, double *dkrow,
                        double *dvrow, double *dkgrow) {
  const problem *p = s->p;
  int d = p->d, H = p->Hq, R = p->Hq / p->Hkv;
  double sigma = p->scale_multiplier / sqrt((double)d);
  for (int f = 0; f < d; f++) {
    dkrow[f] = 0.0;
    dvrow[f] = 0.0;
  }
  const double *vj = kv_row(s, s->V, j, kh);
  for (int f = 0; dkgrow && f < p->R; f++) dkgrow[f] = 0.0;
  for (int h = kh * R; h < (kh + 1) * R; h++) {
    double slope = slope_of(p, s->b, h);
    for (int i = 0; i < s->Lq; i++) {
      int64_t rowid = (s->q0 + i) * (int64_t)H + h;
      double lse = o->lse[rowid];
      if (lse == -INFINITY) continue; /* empty row contributes nothing */
      if (!admissible(p, s->Lq, s->Lk, i, j)) continue;
      const double *qi = s->Q + ((size_t)i * H + h) * d;
      const double *dOi = s->dO + ((size_t)i * H + h) * d;
      double g;
      double z = logit(s, qi, i, j, kh, slope, &g);
      double P = exp(z - lse);
      double dp = 0.0;
      for (int f = 0; f < d; f++) dp += dOi[f] * vj[f];
      const double fd = drop_factor(p, s->b, h, s->q0 + i, i, j);
      const double G = gate_of(s, h, i, j, kh);
      double ds = P * (G * fd * dp - o->Dpre[rowid]) * g;
      for (int f = 0; f < d; f++) {
        dvrow[f] += P * G * fd * dOi[f];
        dkrow[f] += ds * qi[f];
      }
      if (dkgrow) {
        const double dg = dp * P * fd * G * (1.0 - G) / sqrt((double)p->R);
        const double *qg = s->Qg + ((size_t)i * H + h) * p->R;
        for (int f = 0; f < p->R; f++) dkgrow[f] += dg * qg[f];
      }
    }
  }
  for (int f = 0; f < d; f++) dkrow[f] *= sigma;
}

/* Key j of K/V head kh into the packed dk, dv (and dkg) outputs. */
static void key_pass(const seqdata *s, int j, int kh, const outputs *o) {
  const problem *p = s->p;
  int64_t at = ((s->k0 + j) * (int64_t)p->Hkv + kh) * p->d;
  double *dkgrow = o->dkg ? o->dkg + ((s->k0 + j) * (int64_t)p->Hkv + kh) * p->R : NULL;
  key_pass_to(s, j, kh, o, o->dk + at, o->dv + at, dkgrow);
}

/* ---- a tiny thread pool over a fixed unit list ------------------------- */

typedef struct {
  const problem *p;
  const outputs *o;
  const seqdata *seqs; /* indexed by sequence */
  const int *unit_b;   /* unit -> sequence */
  const int *unit_a;   /* unit -> head (phase 1) or key * Hkv + K/V head (phase 2) */
  int n_units;
  int phase; /* 1: rows of (sequence, head); 2: keys; 3: sampled keys into dk_r/dv_r */
  double *dk_r, *dv_r; /* phase 3: [n_units][d] */
  int next; /* shared counter */
  pthread_mutex_t mu;
} pool;

static void *worker(void *arg) {
  pool *w = (pool *)arg;
  int Lmax = 1;
  for (int u = 0; u < w->n_units; u++) {
    int L = w->seqs[w->unit_b[u]].Lk;
    if (L > Lmax) Lmax = L;
  }
  double *z = malloc(sizeof(double) * Lmax);
  double *P = malloc(sizeof(double) * Lmax);
  double *g = malloc(sizeof(double) * Lmax);
  for (;;) {
    pthread_mutex_lock(&w->mu);
    int u = w->next++;
    pthread_mutex_unlock(&w->mu);
    if (u >= w->n_units) break;
    const seqdata *s = &w->seqs[w->unit_b[u]];
    if (w->phase == 1) {
      for (int i = 0; i < s->Lq; i++) row_pass_packed(s, w->unit_a[u], i, w->o, z, P, g);
    } else if (w->phase == 2) {
      key_pass(s, w->unit_a[u] / w->p->Hkv, w->unit_a[u] % w->p->Hkv, w->o);
    } else {
      const int64_t d = w->p->d;
      key_pass_to(s, w->unit_a[u] / w->p->Hkv, w->unit_a[u] % w->p->Hkv, w->o,
                  w->dk_r + u * d, w->dv_r + u * d, NULL);
    }
  }
  free(z);
  free(P);
  free(g);
  return NULL;
}

static int thread_count(int requested) {
  if (requested > 0) return requested;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void run_pool(pool *w, int nthreads) {
  pthread_t *tid = malloc(sizeof(pthread_t) * nthreads);
  w->next = 0;
  pthread_mutex_init(&w->mu, NULL);
  for (int t = 0; t < nthreads; t++) pthread_create(&tid[t], NULL, worker, w);
  for (int t = 0; t < nthreads; t++) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&w->mu);
  free(tid);
}

/* ---- exported entry points --------------------------------------------- */

/* Full forward + VJP for the sequences with seq_sel[b] != 0 (all of them when
 * seq_sel is NULL).  Output rows of unselected sequences are left untouched.
 * All output arrays are dense fp64: out, dq [T_q][Hq][d]; lse, Dpre [T_q][Hq];
 * dk, dv [T_k][Hkv][d]; dz_rowsum and p_rowsum [T_q][Hq] are optional (NULL).
 * Hq must be a multiple of Hkv.  Returns the number of threads used (0 for
 * an invalid head split). */
int oracle_fvjp(int dtype, int B, int Hq, int Hkv, int d, const void *q, int64_t q_ts,
                int64_t q_hs, const void *k, int64_t k_ts, int64_t k_hs, const void *v,
                int64_t v_ts, int64_t v_hs,
                const void *dout, int64_t do_ts, int64_t do_hs, const int32_t *cu_q,
                const int32_t *cu_k, const float *slopes, int64_t slopes_bs, int causal, int wl,
                int wr, double softcap, double scale_multiplier, int dropout, uint64_t seed,
                float rate, const float *rates, int R, const void *qg, int64_t qg_ts,
                int64_t qg_hs, const void *kg, int64_t kg_ts, int64_t kg_hs,
                const uint8_t *seq_sel, double *out, double *lse, double *dq, double *dk,
                double *dv, double *Dpre, double *dz_rowsum, double *p_rowsum, double *dqg,
                double *dkg, int nthreads) {
  if (Hkv < 1 || Hq % Hkv) return 0;
  problem p = {dtype, B,     Hq,    Hkv,  d,     q,  q_ts,  q_hs,    k,
               k_ts,  k_hs,  v,     v_ts, v_hs,  dout, do_ts, do_hs,  cu_q,
               cu_k,  slopes, slopes_bs, causal, wl, wr, softcap, scale_multiplier,
               dropout, seed, rate, rates, R, qg, qg_ts, qg_hs, kg, kg_ts, kg_hs};
  if (R < 0 || (R > 0 && (!qg || !kg || !dqg || !dkg))) return 0;
  outputs o = {out, lse, dq, Dpre, dz_rowsum, p_rowsum, dk, dv, dqg, dkg};
  int nt = thread_count(nthreads);
  seqdata *seqs = calloc((size_t)B + 1, sizeof(seqdata));
  int n1 = 0, n2 = 0;
  for (int b = 0; b < B; b++) {
    if (seq_sel && !seq_sel[b]) continue;
    seq_load(&p, b, &seqs[b]);
    n1 += Hq;
    n2 += seqs[b].Lk * Hkv;
  }
  int *ub = malloc(sizeof(int) * (size_t)(n1 + n2 + 1));
  int *ua = malloc(sizeof(int) * (size_t)(n1 + n2 + 1));
  /* phase 1: one unit per (sequence, head) */
  int n = 0;
  for (int b = 0; b < B; b++) {
    if (seq_sel && !seq_sel[b]) continue;
    for (int h = 0; h < Hq; h++) {
      ub[n] = b;
      ua[n] = h;
      n++;
    }
  }
  pool w1 = {.p = &p, .o = &o, .seqs = seqs, .unit_b = ub, .unit_a = ua, .n_units = n, .phase = 1};
  run_pool(&w1, nt);
  /* phase 2: one unit per (sequence, key, K/V head) */
  n = 0;
  for (int b = 0; b < B; b++) {
    if (seq_sel && !seq_sel[b]) continue;
    for (int j = 0; j < seqs[b].Lk * Hkv; j++) {
      ub[n] = b;
      ua[n] = j;
      n++;
    }
  }
  pool w2 = {.p = &p, .o = &o, .seqs = seqs, .unit_b = ub, .unit_a = ua, .n_units = n, .phase = 2};
  run_pool(&w2, nt);
  for (int b = 0; b < B; b++)
    if (!seq_sel || seq_sel[b]) seq_free(&seqs[b]);
  free(seqs);
  free(ub);
  free(ua);
  return nt;
}

/* Row-sampled forward and dq: for each sampled packed row (token tok[r], head
 * head[r]) compute out, lse, D and dq, written densely at index r of the
 * out_r/dq_r [n][d] and lse_r/D_r [n] arrays.  The sequence of each token is
 * found from cu_q.  Costs O(Lk * d) per row, so it serves full-size checks. */
typedef struct {
  const problem *p;
  int n;
  const int64_t *tok;
  const int32_t *head;
  double *out_r, *lse_r, *dq_r, *D_r;
  int next;
  pthread_mutex_t mu;
} rowpool;

static int seq_of_token(const problem *p, int64_t t) {
  int lo = 0, hi = p->B - 1; /* last b with cu_q[b] <= t, among non-empty */
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (p->cu_q[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  while (lo < p->B && p->cu_q[lo + 1] <= t) lo++; /* skip empty sequences */
  return lo;
}

static void *row_worker(void *arg) {
  rowpool *w = (rowpool *)arg;
  const problem *p = w->p;
  int d = p->d, H = p->Hq;
  for (;;) {
    pthread_mutex_lock(&w->mu);
    int r = w->next++;
    pthread_mutex_unlock(&w->mu);
    if (r >= w->n) break;
    int64_t t = w->tok[r];
    int h = w->head[r];
    int b = seq_of_token(p, t);
    /* The sequence's keys are decoded; of the queries only row t, head h. */
    seqdata s;
    s.p = p;
    s.b = b;
    s.q0 = p->cu_q[b];
    s.k0 = p->cu_k[b];
    s.Lq = p->cu_q[b + 1] - p->cu_q[b];
    s.Lk = p->cu_k[b + 1] - p->cu_k[b];
    s.Q = s.dO = NULL;
    s.Qg = s.Kg = NULL;
    int i = (int)(t - s.q0);
    double *qi = malloc(sizeof(double) * d);
    double *dOi = malloc(sizeof(double) * d);
    for (int f = 0; f < d; f++) {
      qi[f] = decode(p, p->q, t * p->q_ts + (int64_t)h * p->q_hs + f);
      dOi[f] = decode(p, p->dout, t * p->do_ts + (int64_t)h * p->do_hs + f);
    }
    s.K = malloc(sizeof(double) * ((size_t)s.Lk * p->Hkv * d + 1));
    s.V = malloc(sizeof(double) * ((size_t)s.Lk * p->Hkv * d + 1));
    for (int j = 0; j < s.Lk; j++)
      for (int g = 0; g < p->Hkv; g++)
        for (int f = 0; f < d; f++) {
          int64_t tk = s.k0 + j;
          size_t at = ((size_t)j * p->Hkv + g) * d + f;
          s.K[at] = decode(p, p->k, tk * p->k_ts + g * p->k_hs + f);
          s.V[at] = decode(p, p->v, tk * p->v_ts + g * p->v_hs + f);
        }
    rowdest o = {w->out_r + (int64_t)r * d, w->dq_r + (int64_t)r * d, w->lse_r + r, w->D_r + r,
                 NULL, NULL, NULL};
    int Lk1 = s.Lk > 0 ? s.Lk : 1;
    double *z = malloc(sizeof(double) * Lk1), *P = malloc(sizeof(double) * Lk1);
    double *g = malloc(sizeof(double) * Lk1);
    row_pass(&s, h, i, qi, dOi, &o, z, P, g);
    (void)H;
    free(z);
    free(P);
    free(g);
    free(qi);
    free(dOi);
    free(s.K);
    free(s.V);
  }
  return NULL;
}

int oracle_rows(int dtype, int B, int Hq, int Hkv, int d, const void *q, int64_t q_ts,
                int64_t q_hs, const void *k, int64_t k_ts, int64_t k_hs, const void *v,
                int64_t v_ts, int64_t v_hs,
                const void *dout, int64_t do_ts, int64_t do_hs, const int32_t *cu_q,
                const int32_t *cu_k, const float *slopes, int64_t slopes_bs, int causal, int wl,
                int wr, double softcap, double scale_multiplier, int dropout, uint64_t seed,
                float rate, const float *rates, int R, const void *qg, int64_t qg_ts,
                int64_t qg_hs, const void *kg, int64_t kg_ts, int64_t kg_hs, int n,
                const int64_t *tok,
                const int32_t *head, double *out_r, double *lse_r, double *dq_r, double *D_r,
                int nthreads) {
  if (Hkv < 1 || Hq % Hkv) return 0;
  problem p = {dtype, B,     Hq,    Hkv,  d,     q,  q_ts,  q_hs,    k,
               k_ts,  k_hs,  v,     v_ts, v_hs,  dout, do_ts, do_hs,  cu_q,
               cu_k,  slopes, slopes_bs, causal, wl, wr, softcap, scale_multiplier,
               dropout, seed, rate, rates, R, qg, qg_ts, qg_hs, kg, kg_ts, kg_hs};
  if (R != 0) return 0; /* the row sampler serves the ungated path */
  rowpool w;
  w.p = &p;
  w.n = n;
  w.tok = tok;
  w.head = head;
  w.out_r = out_r;
  w.lse_r = lse_r;
  w.dq_r = dq_r;
  w.D_r = D_r;
  w.next = 0;
  pthread_mutex_init(&w.mu, NULL);
  int nt = thread_count(nthreads);
  pthread_t *tid = malloc(sizeof(pthread_t) * nt);
  for (int t = 0; t < nt; t++) pthread_create(&tid[t], NULL, row_worker, &w);
  for (int t = 0; t < nt; t++) pthread_join(tid[t], NULL);
  pthread_mutex_destroy(&w.mu);
  free(tid);
  return nt;
}

/* Key-sampled dk and dv: for each sampled key (packed key token key_tok[r],
 * K/V head key_head[r]) its dk and dv rows, written densely at index r of
 * dk_r/dv_r [n][d].  Every sequence holding a sampled key first takes the
 * row pass of oracle_fvjp with the dq part left out (lse and D are computed
 * the same way, operation for operation), then each sampled key takes
 * oracle_fvjp's key pass: the rows equal oracle_fvjp's dk and dv bit for
 * bit, at about a quarter of its cost per sequence.  Ungated problems only.
 * Returns the number of threads used (0 for invalid arguments). */
int oracle_keys(int dtype, int B, int Hq, int Hkv, int d, const void *q, int64_t q_ts,
                int64_t q_hs, const void *k, int64_t k_ts, int64_t k_hs, const void *v,
                int64_t v_ts, int64_t v_hs,
                const void *dout, int64_t do_ts, int64_t do_hs, const int32_t *cu_q,
                const int32_t *cu_k, const float *slopes, int64_t slopes_bs, int causal, int wl,
                int wr, double softcap, double scale_multiplier, int dropout, uint64_t seed,
                float rate, const float *rates, int R, const void *qg, int64_t qg_ts,
                int64_t qg_hs, const void *kg, int64_t kg_ts, int64_t kg_hs, int n,
                const int64_t *key_tok, const int32_t *key_head, double *dk_r, double *dv_r,
                int nthreads) {
  if (Hkv < 1 || Hq % Hkv || R != 0 || n < 0) return 0;
  problem p = {dtype, B,     Hq,    Hkv,  d,     q,  q_ts,  q_hs,    k,
               k_ts,  k_hs,  v,     v_ts, v_hs,  dout, do_ts, do_hs,  cu_q,
               cu_k,  slopes, slopes_bs, causal, wl, wr, softcap, scale_multiplier,
               dropout, seed, rate, rates, R, qg, qg_ts, qg_hs, kg, kg_ts, kg_hs};
  int64_t Tq = B > 0 ? cu_q[B] : 0;
  for (int r = 0; r < n; r++) {
    if (key_head[r] < 0 || key_head[r] >= Hkv || key_tok[r] < 0 || key_tok[r] >= cu_k[B])
      return 0;
  }
  /* the sequence of each sampled key (last b with cu_k[b] <= t, non-empty) */
  int *kb = malloc(sizeof(int) * ((size_t)n + 1));
  uint8_t *need = calloc((size_t)B + 1, 1);
  for (int r = 0; r < n; r++) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if (cu_k[mid] <= key_tok[r])
        lo = mid;
      else
        hi = mid - 1;
    }
    while (lo < B && cu_k[lo + 1] <= key_tok[r]) lo++;
    kb[r] = lo;
    need[lo] = 1;
  }
  double *out = malloc(sizeof(double) * ((size_t)Tq * Hq * d + 1));
  double *lse = malloc(sizeof(double) * ((size_t)Tq * Hq + 1));
  double *Dpre = malloc(sizeof(double) * ((size_t)Tq * Hq + 1));
  outputs o = {out, lse, NULL, Dpre, NULL, NULL, NULL, NULL, NULL, NULL};
  int nt = thread_count(nthreads);
  seqdata *seqs = calloc((size_t)B + 1, sizeof(seqdata));
  int n1 = 0;
  for (int b = 0; b < B; b++)
    if (need[b]) {
      seq_load(&p, b, &seqs[b]);
      n1 += Hq;
    }
  int *ub = malloc(sizeof(int) * (size_t)(n1 + n + 1));
  int *ua = malloc(sizeof(int) * (size_t)(n1 + n + 1));
  int m = 0;
  for (int b = 0; b < B; b++)
    for (int h = 0; need[b] && h < Hq; h++) {
      ub[m] = b;
      ua[m] = h;
      m++;
    }
  pool w1 = {.p = &p, .o = &o, .seqs = seqs, .unit_b = ub, .unit_a = ua, .n_units = m, .phase = 1};
  run_pool(&w1, nt);
  for (int r = 0; r < n; r++) {
    ub[r] = kb[r];
    ua[r] = (int)(key_tok[r] - cu_k[kb[r]]) * Hkv + key_head[r];
  }
  pool w3 = {.p = &p, .o = &o, .seqs = seqs, .unit_b = ub, .unit_a = ua, .n_units = n,
             .phase = 3, .dk_r = dk_r, .dv_r = dv_r};
  run_pool(&w3, nt);
  for (int b = 0; b < B; b++)
    if (need[b]) seq_free(&seqs[b]);
  free(seqs);
  free(ub);
  free(ua);
  free(kb);
  free(need);
  free(out);
  free(lse);
  free(Dpre);
  return nt;
}

/* Exposed for the dropout pins in the test-suite. */
uint64_t oracle_splitmix64(uint64_t x) { return splitmix64(x); }

double oracle_drop_factor(uint64_t seed, float rate, int b, int h, int i, int j) {
  problem p;
  memset(&p, 0, sizeof p);
  p.dropout = 1;
  p.seed = seed;
  p.rate = rate;
  return drop_factor(&p, b, h, 0, i, j);
}

/* Exposed for the decoder pins in the test-suite. */
double oracle_decode(int dtype, uint16_t x) {
  return dtype == 1 ? bf16_bits_to_double(x) : half_bits_to_double(x);
}
