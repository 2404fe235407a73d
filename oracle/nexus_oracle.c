/*
 * nexus_oracle.c -- plain CPU oracle for one Nexus Sampling eviction step.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm load this library. The product path (the CUDA
 * library) never calls it, and this file shares no code, header or constant
 * table with it.
 *
 * What it follows:
 *   "Forget Without Compromise: Nexus Sampling for Streaming KV-Cache Eviction
 *    Under Fixed Budgets" (full text):
 *     §2.1 streaming view          -- keep B of T rows, continue with K_S, V_S
 *     §2.1 Eq. (1)                 -- S = rownorm(BlockSum_b(softmax(Q K^T / sqrt(D))))
 *     §2.2 Eq. (3)                 -- a = (1/W) sum_q a^(q)
 *     §2.2 Eq. (4)                 -- walk: gamma_q = 1 + <a^(q), C>, C += gamma_q a^(q)
 *     §2.2 Eq. (2)                 -- s = a + lambda * c~,   c~ = C / ||C||_1
 *     §2.2 Eq. (5)                 -- w = s + eps_tie * j / (N_k - 1)
 *     §2.3                         -- forced sink + recency slots, K = B - B_forced
 *     §2.3 Eq. (6), n = 1          -- priority u^(1/w); same order as ln(u)/w
 *   Efraimidis & Spirakis, "Weighted random sampling with a reservoir" (IPL 2006):
 *     keep the K largest keys u^(1/w).
 *   Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 *     (SC'11): the Philox4x32 bijection with 10 rounds.
 *
 * Readings where §2.1-§2.3 leave a detail unstated (each the plainest reading of the
 * surrounding text):
 *   block size b = 1 (BlockSum and rownorm are identities); the window query Q
 *   is the mean of the G query heads that share the KV head, in the model's dtype
 *   (for a bf16 cache: the mean rounded once to bf16); no causal mask;
 *   the walk uses the last H window rows oldest first, without damping, and
 *   c~ = 0 when H = 0; forced slots are the first n_sink and the last n_recent
 *   slots; ties in the key are broken by the larger slot (the newer token).
 *
 * Precision: every score is computed in double. The weight w is rounded once to
 * float; from there the key path is exactly specified float arithmetic (each
 * +, -, *, / rounded to nearest, compiled with -ffp-contract=off), so any
 * correct implementation of the same specification gives the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Input decoding                                                            */
/* ------------------------------------------------------------------------ */

enum { NXO_F32 = 0, NXO_BF16 = 1 };

/* bfloat16 is the upper half of an IEEE binary32 word. */
static double nxo_bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

static double nxo_load(const void* base, int dtype, int64_t idx) {
  if (dtype == NXO_BF16) return nxo_bf16_to_double(((const uint16_t*)base)[idx]);
  return (double)((const float*)base)[idx];
}

/* bfloat16 rounding of a double: to the nearest value with 8 significant bits (binary32's
 * exponent range, so below 2^-126 to a multiple of 2^-133), ties to even. Finite inputs
 * within the bf16 range only. */
static double nxo_round_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  if (fabs(x) < ldexp(1.0, -126)) return ldexp(nearbyint(ldexp(x, 133)), -133);
  int e;
  const double m = frexp(x, &e);            /* x = m 2^e, 0.5 <= |m| < 1 */
  return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

/* ------------------------------------------------------------------------ */
/* Scoring: Eqs. (1)-(5) for one slice (one layer, sequence and KV head)     */
/* ------------------------------------------------------------------------ */

/*
 * Eq. (1), the part before BlockSum: for every window row w, the logits
 * Q_w . K_j / sqrt(D) over the whole cache (no mask) and their softmax, into
 * P (W x T, row-major). rowmax / rowsum (optional) receive each row's maximum
 * logit and sum of exp(logit - max).
 */
static void nxo_softmax_rows(int T, int d, int W, const double* K, const double* Qbar,
                             double* P, double* rowmax, double* rowsum) {
  const double scale = 1.0 / sqrt((double)d);
  for (int w = 0; w < W; ++w) {
    double* row = P + (size_t)w * T;
    double m = -INFINITY;
    for (int j = 0; j < T; ++j) {
      double dot = 0.0;
      for (int k = 0; k < d; ++k) dot += Qbar[(size_t)w * d + k] * K[(size_t)j * d + k];
      row[j] = dot * scale;
      if (row[j] > m) m = row[j];
    }
    double z = 0.0;
    for (int j = 0; j < T; ++j) {
      row[j] = exp(row[j] - m);
      z += row[j];
    }
    for (int j = 0; j < T; ++j) row[j] /= z;
    if (rowmax) rowmax[w] = m;
    if (rowsum) rowsum[w] = z;
  }
}

/*
 * Eqs. (3), (4), (2), (5) over N scoring units (tokens at b = 1, blocks at
 * b > 1), from the W per-row distributions P (W x N). Outputs as in
 * nxo_slice_scores. Returns 0, or -1 on allocation failure.
 */
static int nxo_weights_from_rows(int N, int W, int H, double lambda, double eps_tie,
                                 const double* P, double* a, double* ctilde, double* s,
                                 float* w32, double* gamma) {
  double* C = (double*)calloc((size_t)N, sizeof(double));
  double* ab = (double*)malloc(sizeof(double) * (size_t)N);
  double* cb = (double*)malloc(sizeof(double) * (size_t)N);
  if (!C || !ab || !cb) {
    free(C); free(ab); free(cb);
    return -1;
  }
  /* Eq. (3): the direct score is the uniform average of the W rows. */
  for (int j = 0; j < N; ++j) {
    double acc = 0.0;
    for (int w = 0; w < W; ++w) acc += P[(size_t)w * N + j];
    ab[j] = acc / (double)W;
  }

  /* Eq. (4): C starts at 0; each of the last H rows, oldest first, is plugged
   * in once: gamma = 1 + <a^(q), C>, then C += gamma a^(q). */
  for (int t = 0; t < H; ++t) {
    const double* row = P + (size_t)(W - H + t) * N;
    double inner = 0.0;
    for (int j = 0; j < N; ++j) inner += row[j] * C[j];
    double g = 1.0 + inner;
    if (gamma) gamma[t] = g;
    for (int j = 0; j < N; ++j) C[j] += g * row[j];
  }
  /* c~ = C / ||C||_1; an empty walk (H = 0) leaves c~ = 0. */
  double l1 = 0.0;
  for (int j = 0; j < N; ++j) l1 += fabs(C[j]);
  for (int j = 0; j < N; ++j) cb[j] = (H > 0 && l1 > 0.0) ? C[j] / l1 : 0.0;

  /* Eq. (2) and Eq. (5): s = a + lambda c~, w = s + eps_tie * j / (N - 1). */
  for (int j = 0; j < N; ++j) {
    double sj = ab[j] + lambda * cb[j];
    double r = (N > 1) ? (double)j / (double)(N - 1) : 0.0;
    double wj = sj + eps_tie * r;
    if (a) a[j] = ab[j];
    if (ctilde) ctilde[j] = cb[j];
    if (s) s[j] = sj;
    if (w32) w32[j] = (float)wj;
  }
  free(C); free(ab); free(cb);
  return 0;
}

/*
 * K: T x d rows of cached keys; Qbar: W x d window queries (already averaged
 * over the query heads of the group). All outputs are optional (NULL skips);
 * P (W x T) is the per-row distribution a^(q) of Eq. (3). Block size b = 1:
 * BlockSum and rownorm of Eq. (1) are identities.
 *
 * Returns 0 on success, -1 on bad sizes or allocation failure.
 */
int nxo_slice_scores(int T, int d, int W, int H, double lambda, double eps_tie,
                     const double* K, const double* Qbar, double* P_out,
                     double* a, double* ctilde, double* s, float* w32,
                     double* rowmax, double* rowsum, double* gamma) {
  if (T < 1 || d < 1 || W < 1 || H < 0 || H > W) return -1;
  double* P = P_out ? P_out : (double*)malloc(sizeof(double) * (size_t)W * T);
  if (!P) return -1;
  nxo_softmax_rows(T, d, W, K, Qbar, P, rowmax, rowsum);
  int rc = nxo_weights_from_rows(T, W, H, lambda, eps_tie, P, a, ctilde, s, w32, gamma);
  if (!P_out) free(P);
  return rc;
}

/*
 * Eq. (1) at block size b > 1 (§2.1 "Block granularity"): the token softmax rows
 * are summed over blocks of b consecutive slots (BlockSum_b; the last block
 * holds the T mod b remaining slots when b does not divide T) and each row is
 * renormalised to sum 1 (rownorm), giving W rows over N_k = ceil(T / b) blocks;
 * then Eqs. (3), (4), (2), (5) run over blocks, the tie-break ramp over the
 * block index j / (N_k - 1). Outputs have N_k entries; Pb_out (optional) is the
 * W x N_k block distribution. Returns N_k, or -1 on bad sizes / allocation.
 */
int nxo_block_scores(int T, int d, int W, int H, int b, double lambda, double eps_tie,
                     const double* K, const double* Qbar, double* Pb_out, double* a,
                     double* ctilde, double* s, float* w32, double* gamma) {
  if (T < 1 || d < 1 || W < 1 || H < 0 || H > W || b < 1) return -1;
  const int N = (T + b - 1) / b;
  double* P = (double*)malloc(sizeof(double) * (size_t)W * T);
  double* Pb = Pb_out ? Pb_out : (double*)malloc(sizeof(double) * (size_t)W * N);
  if (!P || !Pb) {
    free(P);
    if (!Pb_out) free(Pb);
    return -1;
  }
  nxo_softmax_rows(T, d, W, K, Qbar, P, NULL, NULL);
  for (int w = 0; w < W; ++w) {
    const double* row = P + (size_t)w * T;
    double* brow = Pb + (size_t)w * N;
    double tot = 0.0;
    for (int B = 0; B < N; ++B) {
      double acc = 0.0;
      for (int j = B * b; j < T && j < (B + 1) * b; ++j) acc += row[j];
      brow[B] = acc;
      tot += acc;
    }
    for (int B = 0; B < N; ++B) brow[B] /= tot;   /* rownorm */
  }
  int rc = nxo_weights_from_rows(N, W, H, lambda, eps_tie, Pb, a, ctilde, s, w32, gamma);
  free(P);
  if (!Pb_out) free(Pb);
  return rc == 0 ? N : -1;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11)                                      */
/* ------------------------------------------------------------------------ */

/*
 * One Philox4x32 round: two 32x32->64 multiplications of words 0 and 2 by the
 * round multipliers; the high halves are mixed into words 1 and 3 with the key.
 * Ten rounds; the key is bumped by the Weyl constants between rounds.
 */
void nxo_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t MUL0 = 0xD2511F53u, MUL1 = 0xCD9E8D57u;
  const uint32_t WEYL0 = 0x9E3779B9u, WEYL1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += WEYL0;
      k1 += WEYL1;
    }
    uint64_t p0 = (uint64_t)MUL0 * (uint64_t)x0;
    uint64_t p1 = (uint64_t)MUL1 * (uint64_t)x2;
    uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
    uint32_t y1 = (uint32_t)p1;
    uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
    uint32_t y3 = (uint32_t)p0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* A 32-bit word to a uniform in (0, 1): the top 23 bits k give (2k + 1) 2^-24,
 * exact in binary32 and never 0 or 1. */
float nxo_uniform(uint32_t x) {
  uint32_t k = x >> 9;
  return (float)(2u * k + 1u) * (1.0f / 16777216.0f);
}

/* ------------------------------------------------------------------------ */
/* ln_spec: a fully specified binary32 natural logarithm                     */
/* ------------------------------------------------------------------------ */

/*
 * Textbook method (argument reduction by the exponent, then the atanh series):
 *   u = 2^e m with m in [sqrt(1/2), sqrt(2)],
 *   f = (m - 1) / (m + 1),  ln m = 2 atanh f = 2f (1 + f^2/3 + f^4/5 + ...),
 *   ln u = e ln2_hi + (e ln2_lo + ln m), with ln 2 split Cody-Waite style into
 *   ln2_hi (16 significant bits, so e * ln2_hi is exact) and ln2_lo.
 * The series is truncated after the f^12/13 term and evaluated by Horner in
 * s = f^2 with separately rounded multiplies and adds, in the fixed order
 * below. Defined for normal u in (0, 1); that is all the key path needs.
 */
float nxo_ln_spec(float u) {
  const float ln2_hi = 45426.0f / 65536.0f;  /* round(ln2 * 2^16) / 2^16 */
  const float ln2_lo = (float)(0.69314718055994530942 - 45426.0 / 65536.0);
  const float c3 = 1.0f / 3.0f, c5 = 1.0f / 5.0f, c7 = 1.0f / 7.0f, c9 = 1.0f / 9.0f;
  const float c11 = 1.0f / 11.0f, c13 = 1.0f / 13.0f;
  uint32_t b;
  memcpy(&b, &u, 4);
  int e = (int)((b >> 23) & 0xFFu) - 127;
  uint32_t frac = b & 0x7FFFFFu;
  uint32_t mbits;
  if (frac > 0x3504F3u) {       /* 1.frac > sqrt(2): use m/2 and e + 1 */
    mbits = frac | 0x3F000000u;
    e += 1;
  } else {
    mbits = frac | 0x3F800000u;
  }
  float m;
  memcpy(&m, &mbits, 4);
  float num = m - 1.0f;
  float den = m + 1.0f;
  float f = num / den;
  float s = f * f;
  float t = f + f;
  float q = c13;
  q = q * s; q = q + c11;
  q = q * s; q = q + c9;
  q = q * s; q = q + c7;
  q = q * s; q = q + c5;
  q = q * s; q = q + c3;
  float sq = s * q;
  float r = t * sq;
  float lnm = t + r;
  float ef = (float)e;
  float hi = ef * ln2_hi;
  float lo = ef * ln2_lo;
  float tail = lo + lnm;
  return hi + tail;
}

void nxo_ln_spec_many(int64_t n, const float* u, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = nxo_ln_spec(u[i]);
}

/* ------------------------------------------------------------------------ */
/* exp_spec: a fully specified binary32 exponential                          */
/* ------------------------------------------------------------------------ */

/*
 * Textbook method (Cody & Waite argument reduction, then the Taylor series):
 *   k = round-to-nearest-even(x / ln 2) (x * (1/ln 2) rounded to binary32 first),
 *   r = (x - k ln2_hi) - k ln2_lo   with ln 2 = ln2_hi + ln2_lo as in ln_spec
 *                                   (16-bit ln2_hi, so k ln2_hi is exact),
 *   e^r = 1 + r + r^2/2! + ... + r^7/7!  by Horner from the r^7/7! term,
 *   e^x = e^r * 2^k.
 * |r| <= ln(2)/2, so the truncated series is within 1e-8 relative. Results with
 * k < -126 (below the smallest normal scale) are flushed to 0, k > 127 gives
 * +inf. Every + and * is one binary32 rounding, in the fixed order below.
 */
float nxo_exp_spec(float x) {
  const float inv_ln2 = 1.44269504088896340736f;
  const float ln2_hi = 45426.0f / 65536.0f;
  const float ln2_lo = (float)(0.69314718055994530942 - 45426.0 / 65536.0);
  const float c2 = 1.0f / 2.0f, c3 = 1.0f / 6.0f, c4 = 1.0f / 24.0f, c5 = 1.0f / 120.0f;
  const float c6 = 1.0f / 720.0f, c7 = 1.0f / 5040.0f;
  if (x != x) return x;
  float t = x * inv_ln2;
  float kf = rintf(t);
  if (kf < -126.0f) return 0.0f;
  if (kf > 127.0f) return INFINITY;
  float hi = kf * ln2_hi;
  float lo = kf * ln2_lo;
  float r = x - hi;
  r = r - lo;
  float p = c7;
  p = p * r; p = p + c6;
  p = p * r; p = p + c5;
  p = p * r; p = p + c4;
  p = p * r; p = p + c3;
  p = p * r; p = p + c2;
  p = p * r; p = p + 1.0f;
  p = p * r; p = p + 1.0f;
  uint32_t sbits = (uint32_t)((int)kf + 127) << 23;
  float scale;
  memcpy(&scale, &sbits, 4);
  return p * scale;
}

/* bfloat16 rounding of the window queries (the model's dtype), elementwise over doubles. */
void nxo_round_bf16_many(int64_t n, const double* x, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = nxo_round_bf16(x[i]);
}

void nxo_exp_spec_many(int64_t n, const float* x, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = nxo_exp_spec(x[i]);
}

void nxo_philox_many(int64_t n, const uint32_t* ctr4, const uint32_t* key2, uint32_t* out4) {
  for (int64_t i = 0; i < n; ++i) nxo_philox4x32_10(ctr4 + 4 * i, key2, out4 + 4 * i);
}

/* ------------------------------------------------------------------------ */
/* Selection: forced slots, then the K largest reservoir keys (§2.3)         */
/* ------------------------------------------------------------------------ */

enum { NXO_RESERVOIR = 0, NXO_TOPK = 1 };

typedef struct {
  float key;
  int32_t slot;
} nxo_cand;

/* Descending by key, then by slot (the newer token wins a tie). */
static int nxo_cand_cmp(const void* pa, const void* pb) {
  const nxo_cand* x = (const nxo_cand*)pa;
  const nxo_cand* y = (const nxo_cand*)pb;
  if (x->key > y->key) return -1;
  if (x->key < y->key) return 1;
  return (x->slot > y->slot) ? -1 : (x->slot < y->slot) ? 1 : 0;
}

static int nxo_int_cmp(const void* pa, const void* pb) {
  int32_t x = *(const int32_t*)pa, y = *(const int32_t*)pb;
  return (x > y) - (x < y);
}

/*
 * The reservoir key of slot j. Counter = (pos_j, step, head_id, seq_id) with
 * the draw group in bits 24..31 of word 3 (group 0 here); key = the 64-bit seed.
 * The uniform is word 0 of the Philox output; the key is ln(u) / w in binary32
 * (n = 1 of Eq. (6): u^(1/w) and ln(u)/w give the same order).
 */
float nxo_reservoir_key(float w, int32_t pos, uint64_t seed, uint32_t step, uint32_t head_id,
                        uint32_t seq_id) {
  uint32_t ctr[4] = {(uint32_t)pos, step, head_id, seq_id & 0x00FFFFFFu};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  nxo_philox4x32_10(ctr, key, out);
  float u = nxo_uniform(out[0]);
  return nxo_ln_spec(u) / w;
}

/*
 * The n-averaged priority of Eq. (6), pi_j = (1/n) sum_i (u_j^(i))^(1/w_j), in the
 * log domain (at token-sized weights u^(1/w) underflows even in double):
 *   l_i = ln(u_i), M = max_i l_i, r = 1 / w (one IEEE division),
 *   key = M r + ln( sum_i exp((l_i - M) r) )  =  ln(n pi_j).
 * The constant -ln n is left out: it does not change the order. Draw i uses
 * word i mod 4 of the Philox block with draw group g = i / 4 in bits 24..31 of
 * counter word 3 (so draws 0..3 share one block, and draw 0 is the n = 1 draw).
 * Every operation is one binary32 rounding in the order written (ln_spec,
 * exp_spec; the sum runs i = 0 .. n - 1). A zero weight (r = +inf) gives -inf.
 * n = 1 is the plain key ln(u)/w above. n is at most 1024 (256 draw groups).
 */
float nxo_reservoir_key_n(float w, int32_t pos, uint64_t seed, uint32_t step, uint32_t head_id,
                          uint32_t seq_id, int n) {
  if (n <= 1) return nxo_reservoir_key(w, pos, seed, step, head_id, seq_id);
  if (n > 1024) return NAN;
  float l[1024];
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4] = {0, 0, 0, 0};
  float M = -INFINITY;
  for (int i = 0; i < n; ++i) {
    if (i % 4 == 0) {
      uint32_t g = (uint32_t)(i / 4);
      uint32_t ctr[4] = {(uint32_t)pos, step, head_id, (seq_id & 0x00FFFFFFu) | (g << 24)};
      nxo_philox4x32_10(ctr, key, out);
    }
    l[i] = nxo_ln_spec(nxo_uniform(out[i % 4]));
    if (l[i] > M) M = l[i];
  }
  float r = 1.0f / w;
  if (!(r < INFINITY)) return -INFINITY;
  float S = 0.0f;
  for (int i = 0; i < n; ++i) {
    float dlt = l[i] - M;
    float x = dlt * r;
    S = S + nxo_exp_spec(x);
  }
  float head = M * r;
  return head + nxo_ln_spec(S);
}

/*
 * Retention set S_t of one slice over T decision units (slots at b = 1, blocks
 * at b > 1; pos is each unit's absolute position, a block's being that of its
 * first token). Writes the min(T, B) kept units, ascending, into keep_idx and
 * returns that count. kappa (length T, optional) receives the key of every
 * candidate unit (NaN for forced units). n_avg is the averaging count n of
 * Eq. (6) (1: Efraimidis-Spirakis keys). Returns -1 on invalid arguments.
 */
int nxo_select_slice(int T, const float* w32, const int32_t* pos, int B, int n_sink, int n_recent,
                     int mode, uint64_t seed, uint32_t step, uint32_t head_id, uint32_t seq_id,
                     int n_avg, int32_t* keep_idx, float* kappa) {
  if (T < 0 || B < 0 || n_sink < 0 || n_recent < 0 || n_sink + n_recent > B) return -1;
  if (T <= B) {
    for (int j = 0; j < T; ++j) keep_idx[j] = j;
    if (kappa) for (int j = 0; j < T; ++j) kappa[j] = NAN;
    return T;
  }
  int n_forced = n_sink + n_recent; /* disjoint because n_sink + n_recent <= B < T */
  int K = B - n_forced;
  int n_cand = T - n_forced;
  nxo_cand* cand = (nxo_cand*)malloc(sizeof(nxo_cand) * (size_t)(n_cand > 0 ? n_cand : 1));
  if (!cand) return -1;
  int c = 0, o = 0;
  for (int j = 0; j < T; ++j) {
    int forced = (j < n_sink) || (j >= T - n_recent);
    if (forced) {
      keep_idx[o++] = j;
      if (kappa) kappa[j] = NAN;
      continue;
    }
    float key = (mode == NXO_TOPK)
                    ? w32[j]
                    : nxo_reservoir_key_n(w32[j], pos[j], seed, step, head_id, seq_id, n_avg);
    if (kappa) kappa[j] = key;
    cand[c].key = key;
    cand[c].slot = j;
    ++c;
  }
  qsort(cand, (size_t)n_cand, sizeof(nxo_cand), nxo_cand_cmp);
  for (int i = 0; i < K; ++i) keep_idx[o++] = cand[i].slot;
  qsort(keep_idx, (size_t)B, sizeof(int32_t), nxo_int_cmp);
  free(cand);
  return B;
}

/* ------------------------------------------------------------------------ */
/* The whole step over a cache (§2.1): score, select, keep K_S and V_S       */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t layers, seqs, kv_heads, group, head_dim;
  int32_t capacity;          /* rows per slice (paged: max_pages_per_seq * page_size) */
  int32_t page_size;         /* 0: contiguous [L][S][Hkv][cap][d] */
  int32_t num_pages;         /* paged: pages per layer, pool [L][pages][Hkv][page][d] */
  int32_t max_pages_per_seq;
  int32_t dtype;             /* NXO_F32 or NXO_BF16 */
  void* k;
  void* v;
  int32_t* pos;              /* one per row, same row layout as k */
  int32_t* lens;             /* [L][S][Hkv] */
  const int32_t* block_table;/* [S][max_pages_per_seq] */
} nxo_cache;

typedef struct {
  int32_t window, walk_len, n_sink, n_recent, mode;
  double lambda, eps_tie;
  const int32_t* budget;     /* [S]: units kept per slice of sequence s */
  uint64_t seed;
  uint32_t step;
  int32_t seq_id_base, layer_id_base;
  int32_t n_avg;             /* averaging count n of Eq. (6) (1: plain ES keys) */
  int32_t block_size;        /* b: tokens per decision unit (1 or more) */
  const int32_t* slice_budget; /* optional [L*S*Hkv]: overrides budget[s] per slice */
} nxo_params;

/* Row index (in units of rows) of slot j of slice (l, s, h). */
static int64_t nxo_row(const nxo_cache* c, int l, int s, int h, int j) {
  if (c->page_size == 0)
    return (((int64_t)l * c->seqs + s) * c->kv_heads + h) * c->capacity + j;
  int32_t page = c->block_table[(int64_t)s * c->max_pages_per_seq + j / c->page_size];
  return (((int64_t)l * c->num_pages + page) * c->kv_heads + h) * c->page_size + j % c->page_size;
}

/*
 * One eviction step for the listed slices (slice id = (l * S + s) * Hkv + h;
 * sel == NULL means every slice). Decisions are made per unit of b = block_size
 * consecutive slots (b = 1: per token; the last block of a slice holds the
 * T mod b remaining slots when b does not divide T); the budget B, n_sink and
 * n_recent count units. For slice number i of the list:
 *   keep_out[i * cap ...]  the kept units, ascending (first min(N, B) entries,
 *                          N = ceil(T / b) units),
 *   w_out[i * cap ...]     the binary32 weight w of every unit,
 *   a_out[i * cap ...]     the direct score a (double) of every unit,
 *   newlen_out[i]          the rows left: the total size of the kept units.
 * Any of the outputs may be NULL. With mutate != 0 the K, V and pos rows of the
 * listed slices are compacted in place (the kept units' rows, in order, become
 * slots 0 .. newlen - 1) and lens updated.
 * Returns 0, or -1 on an invalid argument or allocation failure.
 */
int nxo_evict_step(nxo_cache* c, const void* q, const nxo_params* p, int n_sel,
                   const int32_t* sel, int32_t* keep_out, float* w_out, double* a_out,
                   int32_t* newlen_out, int mutate, int nthreads) {
  const int L = c->layers, S = c->seqs, Hk = c->kv_heads, G = c->group, d = c->head_dim;
  const int W = p->window, H = p->walk_len, cap = c->capacity, bs = p->block_size;
  if (H > W || H < 0 || W < 1 || G < 1 || d < 1 || bs < 1) return -1;
  int n = sel ? n_sel : L * S * Hk;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
  for (int i = 0; i < n; ++i) {
    int sid = sel ? sel[i] : i;
    int h = sid % Hk, s = (sid / Hk) % S, l = sid / (Hk * S);
    int T = c->lens[sid];
    int B = p->slice_budget ? p->slice_budget[sid] : p->budget[s];
    int N = (T + bs - 1) / bs;                     /* decision units */
    double* K = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * d);
    double* Qb = (double*)calloc((size_t)W * d, sizeof(double));
    double* a = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    float* w = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
    int32_t* pj = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    int32_t* keep = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!K || !Qb || !a || !w || !pj || !keep) {
      failed |= 1;
    } else {
      for (int j = 0; j < T; ++j) {
        int64_t r = nxo_row(c, l, s, h, j);
        for (int k = 0; k < d; ++k) K[(size_t)j * d + k] = nxo_load(c->k, c->dtype, r * d + k);
      }
      /* a unit's position is that of its first slot */
      for (int u = 0; u < N; ++u) pj[u] = c->pos[nxo_row(c, l, s, h, u * bs)];
      /* The window query of the KV group: mean of its G query heads, a tensor of the
       * model's dtype (a bf16 model's head average is bf16: the mean rounded once). */
      for (int w_ = 0; w_ < W; ++w_)
        for (int k = 0; k < d; ++k) {
          double acc = 0.0;
          for (int g = 0; g < G; ++g) {
            int64_t hq = (int64_t)h * G + g;
            int64_t idx = ((((int64_t)l * S + s) * (Hk * G) + hq) * W + w_) * d + k;
            acc += nxo_load(q, c->dtype, idx);
          }
          const double mean = acc / (double)G;
          Qb[(size_t)w_ * d + k] = c->dtype == NXO_BF16 ? nxo_round_bf16(mean) : mean;
        }
      int rc = 0, nk = 0;
      if (T > 0) {
        if (bs == 1)
          rc = nxo_slice_scores(T, d, W, H, p->lambda, p->eps_tie, K, Qb, NULL, a, NULL, NULL, w,
                                NULL, NULL, NULL);
        else
          rc = nxo_block_scores(T, d, W, H, bs, p->lambda, p->eps_tie, K, Qb, NULL, a, NULL,
                                NULL, w, NULL) == N ? 0 : -1;
      }
      if (rc == 0) {
        uint32_t head_id = (uint32_t)((p->layer_id_base + l) * Hk + h);
        uint32_t seq_id = (uint32_t)(p->seq_id_base + s);
        nk = nxo_select_slice(N, w, pj, B, p->n_sink, p->n_recent, p->mode, p->seed, p->step,
                              head_id, seq_id, p->n_avg, keep, NULL);
      }
      if (rc != 0 || nk < 0) {
        failed |= 1;
      } else {
        /* rows kept: whole units, the last (partial) unit with its own size */
        int nl = 0;
        for (int u = 0; u < nk; ++u) {
          int size = T - keep[u] * bs;
          nl += size < bs ? size : bs;
        }
        if (keep_out) {
          for (int u = 0; u < nk; ++u) keep_out[(size_t)i * cap + u] = keep[u];
        }
        if (w_out) for (int u = 0; u < N; ++u) w_out[(size_t)i * cap + u] = w[u];
        if (a_out) for (int u = 0; u < N; ++u) a_out[(size_t)i * cap + u] = a[u];
        if (newlen_out) newlen_out[i] = nl;
        if (mutate && nl < T) {
          /* §2.1: inference continues with K_S, V_S -- copy out, then back. */
          size_t eb = (c->dtype == NXO_BF16) ? 2 : 4;
          size_t rb = eb * (size_t)d;
          unsigned char* kt = (unsigned char*)malloc(rb * (size_t)nl);
          unsigned char* vt = (unsigned char*)malloc(rb * (size_t)nl);
          int32_t* pt = (int32_t*)malloc(sizeof(int32_t) * (size_t)nl);
          if (!kt || !vt || !pt) {
            failed |= 1;
          } else {
            int o = 0;
            for (int u = 0; u < nk; ++u)
              for (int j = keep[u] * bs; j < T && j < (keep[u] + 1) * bs; ++j, ++o) {
                int64_t r = nxo_row(c, l, s, h, j);
                memcpy(kt + rb * o, (unsigned char*)c->k + rb * r, rb);
                memcpy(vt + rb * o, (unsigned char*)c->v + rb * r, rb);
                pt[o] = c->pos[r];
              }
            for (int j = 0; j < nl; ++j) {
              int64_t r = nxo_row(c, l, s, h, j);
              memcpy((unsigned char*)c->k + rb * r, kt + rb * j, rb);
              memcpy((unsigned char*)c->v + rb * r, vt + rb * j, rb);
              c->pos[r] = pt[j];
            }
            c->lens[sid] = nl;
          }
          free(kt); free(vt); free(pt);
        }
      }
    }
    free(K); free(Qb); free(a); free(w); free(pj); free(keep);
  }
  return failed ? -1 : 0;
}

/*
 * Stand-alone compaction of one slice's rows given a kept-slot list: the
 * out-of-place definition (copy rows keep[0..n) aside, then write them to
 * slots 0..n). Used to check an in-place implementation.
 */
int nxo_compact_slice(nxo_cache* c, int sid, const int32_t* keep, int nl) {
  const int Hk = c->kv_heads, S = c->seqs, d = c->head_dim;
  int h = sid % Hk, s = (sid / Hk) % S, l = sid / (Hk * S);
  size_t eb = (c->dtype == NXO_BF16) ? 2 : 4, rb = eb * (size_t)d;
  unsigned char* kt = (unsigned char*)malloc(rb * (size_t)(nl > 0 ? nl : 1));
  unsigned char* vt = (unsigned char*)malloc(rb * (size_t)(nl > 0 ? nl : 1));
  int32_t* pt = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nl > 0 ? nl : 1));
  if (!kt || !vt || !pt) { free(kt); free(vt); free(pt); return -1; }
  for (int j = 0; j < nl; ++j) {
    int64_t r = nxo_row(c, l, s, h, keep[j]);
    memcpy(kt + rb * j, (unsigned char*)c->k + rb * r, rb);
    memcpy(vt + rb * j, (unsigned char*)c->v + rb * r, rb);
    pt[j] = c->pos[r];
  }
  for (int j = 0; j < nl; ++j) {
    int64_t r = nxo_row(c, l, s, h, j);
    memcpy((unsigned char*)c->k + rb * r, kt + rb * j, rb);
    memcpy((unsigned char*)c->v + rb * r, vt + rb * j, rb);
    c->pos[r] = pt[j];
  }
  c->lens[sid] = nl;
  free(kt); free(vt); free(pt);
  return 0;
}
