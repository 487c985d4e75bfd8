/*
 * sv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, CPU oracle for the batched verify-and-accept step of
 * speculative decoding (Leviathan rejection sampling as used by EAGLE /
 * EAGLE-2 / EAGLE-3).  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [Lesson]  "Decodificação Especulativa e EAGLE-3" (ai-engineering.academy,
 *             Phase 10 Lesson 15) and its Persian twin "دیکودینگ حدسی و
 *             EAGLE-3" (nextadmin.net) -- same lesson, same sections.
 *   [Blog]    "投机解码发展" (caijizhuo.github.io).  NOTE: the blog swaps the
 *             letters (its p is the verifier, its q the draft).  This file uses
 *             the lesson's notation throughout: p = draft, q = verifier.
 *
 * Precision.  Probabilities, ratios and the accept test are computed in
 * double from logits widened exactly to double.  The inverse-CDF token
 * choice (residual / bonus sampling) is a floating-point quantity deciding an
 * integer; it is taken in the kernel's arithmetic, fully specified below
 * (sample_repro): IEEE fp32 operations in a fixed order, an fp32 exponential
 * built from Cody-Waite range reduction and a degree-7 Taylor polynomial, and
 * exact 64-bit fixed-point sums, so that the order of summation cannot change
 * the chosen token.  The tests pin that arithmetic against libm exp and
 * against the double-precision residual law.
 *
 * Compile with -ffp-contract=off: every fused multiply-add below is explicit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_DRAW_ACCEPT 0u
#define ORC_DRAW_SAMPLE 1u
#define ORC_DRAW_DRAFT 2u
#define ORC_DRAW_TREE 3u

#define ORC_ROW_NAN 1u
#define ORC_ROW_BAD_TOKEN 2u
#define ORC_ROW_RESID_ZERO 4u
#define ORC_ROW_P_ZERO 8u
#define ORC_ROW_BAD_TREE 16u

/* ------------------------------------------------------------------------
 * Philox4x32-10 counter-based generator.
 * Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 * (SC'11), section on the Philox family: ten rounds of two 32x32->64
 * multiplies (multipliers 0xD2511F53, 0xCD9E8D57), a word permutation with
 * XOR of the high halves into the other words and the round key, and a Weyl
 * key schedule (increments 0x9E3779B9, 0xBB67AE85) between rounds.
 * ---------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                       uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform the pages call uniform() ([Lesson] Passo 1; [Blog] section 4,
 * spec_decode / eagle_round pseudocode).  The pages leave the generator open;
 * this build keys Philox on the seed and counts on (position, draw, sequence,
 * step mod 2^32), and takes the top 24 bits of the first output word:
 * u = u24 * 2^-24 in [0, 1 - 2^-24], exact in fp32 and fp64. */
uint32_t orc_u24(uint64_t seed, uint64_t step, uint32_t seq, uint32_t pos,
                 uint32_t draw) {
  uint32_t ctr[4] = {pos, draw, seq, (uint32_t)step};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[0] >> 8;
}

/* ------------------------------------------------------------------------
 * Double-precision softmax pieces.  The verifier returns q_1..q_{N+1} and the
 * draft supplies p_1..p_N as full-vocabulary distributions ([Lesson] "O
 * invariante"; [Blog] section 2, step 2 "verify").  Temperature scales the
 * logits before the softmax (the pages name temperature as the knob that
 * lowers acceptance: [Lesson] "Quando não recorrer"; [Blog] section 6).
 * ---------------------------------------------------------------------- */

/* 1 if the row is unusable: a NaN or +inf logit, or every logit -inf. */
int orc_row_bad(const float *x, int V) {
  int all_minf = 1;
  for (int v = 0; v < V; ++v) {
    float a = x[v];
    if (isnan(a) || (isinf(a) && a > 0)) return 1;
    if (!(isinf(a) && a < 0)) all_minf = 0;
  }
  return (V <= 0 || all_minf) ? 1 : 0;
}

/* max_v x_v / T and sum_v exp(x_v/T - max), sequential in index order. */
void orc_row_stats(const float *x, int V, double T, double *m_out,
                   double *s_out) {
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double z = (double)x[v] / T;
    if (z > m) m = z;
  }
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += exp((double)x[v] / T - m);
  *m_out = m;
  *s_out = s;
}

/* Full softmax row in double (used by the pins and the probability outputs). */
void orc_softmax(const float *x, int V, double T, double *prob) {
  double m, s;
  orc_row_stats(x, V, T, &m, &s);
  for (int v = 0; v < V; ++v) prob[v] = exp((double)x[v] / T - m) / s;
}

/* ------------------------------------------------------------------------
 * Step 1 of the lesson ("Passo 1: a regra de rejeição"): accept the draft
 * token d with probability min(1, q(d)/p(d)); a draft probability <= 0 is
 * accepted outright.  The test is u < min(1, q/p), strict.
 * ---------------------------------------------------------------------- */
int orc_accept(double q_prob, double p_prob, double u) {
  if (p_prob <= 0.0) return 1;
  double r = q_prob / p_prob;
  return u < (r < 1.0 ? r : 1.0);
}

/* Step 2 of the lesson ("Passo 2: distribuição residual"): the residual is
 * (q - p)_+ normalised by its L1 norm; when that norm is zero, q itself. */
void orc_residual(const double *q, const double *p, int V, double *out) {
  double s = 0.0;
  for (int v = 0; v < V; ++v) {
    double r = q[v] - p[v];
    out[v] = r > 0.0 ? r : 0.0;
    s += out[v];
  }
  if (s == 0.0) {
    for (int v = 0; v < V; ++v) out[v] = q[v];
    return;
  }
  for (int v = 0; v < V; ++v) out[v] /= s;
}

/* Inverse CDF in ascending token order: the smallest k whose cumulative
 * weight exceeds t (the pages' sample() is unspecified; this is the plainest
 * reading, and it is what Python's weighted choice does).  If rounding leaves
 * no such k, the last k with positive weight. */
int orc_invcdf_f64(const double *w, int V, double t) {
  double c = 0.0;
  int last_pos = -1;
  for (int k = 0; k < V; ++k) {
    c += w[k];
    if (w[k] > 0.0) last_pos = k;
    if (c > t) return k;
  }
  return last_pos;
}

/* ------------------------------------------------------------------------
 * The sampling arithmetic (fp32 + exact fixed point), shared *by
 * specification* with the GPU kernels (each side has its own code).
 *
 *   z_v   = fl32(x_v * invT),     invT = fl32(1 / T)
 *   m     = max_v z_v             (exact)
 *   e_v   = exp32(z_v - m)        (fl32 subtraction, then exp32 below)
 *   E_v   = floor(e_v * 2^40);  S_E = sum_v E_v         (exact uint64)
 *
 * A draw from q -- the bonus token from q_{N+1} ([Lesson] "O invariante"),
 * or the correction when the residual mass is zero ([Lesson] Passo 2) --
 * takes the weights W_v = E_v, S = S_E: q_v = e_v / sum e, and E_v is e_v
 * on a 2^-40 grid, so these weights are q up to that truncation.
 *
 * A residual draw at a rejection ([Lesson] Passo 2) normalises both rows:
 *   inv_s = fl32( 2^40 / fl64(S_E) )                    (per row, fl64 divide)
 *   q_v   = fl32(e_v * inv_s),  p_v likewise from the draft row
 *   w_v   = max(0, fl32(q_v - p_v));  W_v = floor(w_v * 2^62);  S = sum_v W_v
 *   if S == 0 (q == p to the last bit): the draw from q above
 *
 *   t     = floor(u24 * S / 2^24)                       (exact, 128-bit)
 *   token = min { k : sum_{v<=k} W_v > t }
 *
 * exp32(a): 0 if a < -80; else n = rint(a*log2e) via the 1.5*2^23 shift,
 * r = a - n*ln2 (Cody & Waite two-constant reduction, "Software Manual for the
 * Elementary Functions", 1980), e^r by the Taylor series to degree 7 in
 * Horner form with fused multiply-adds, scaled by 2^n.
 * ---------------------------------------------------------------------- */
static const float ORC_LOG2E = 0x1.715476p+0f;  /* fl32(1/ln 2) */
static const float ORC_LN2_HI = 0x1.62e4p-1f;   /* ln 2 to 15 bits */
static const float ORC_LN2_LO = 0x1.7f7d1cp-20f; /* fl32(ln 2 - LN2_HI) */
static const float ORC_SHIFTER = 0x1.8p+23f;     /* 1.5 * 2^23 */

float orc_exp32(float a) {
  if (!(a >= -80.0f)) return 0.0f;
  float t = fmaf(a, ORC_LOG2E, ORC_SHIFTER);
  float n = t - ORC_SHIFTER;
  float r = fmaf(-n, ORC_LN2_HI, a);
  r = fmaf(-n, ORC_LN2_LO, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  uint32_t bits = (uint32_t)(ni + 127) << 23;
  float scale;
  memcpy(&scale, &bits, sizeof scale);
  return p * scale;
}

static float orc_zmax32(const float *x, int V, float invT) {
  float m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    float z = x[v] * invT;
    if (z > m) m = z;
  }
  return m;
}

/* E_v = floor(exp32(fl32(x_v * invT) - m) * 2^40) of one row; returns S_E */
static uint64_t orc_fixed_exp40(const float *x, int V, float invT, float m, uint64_t *E) {
  uint64_t se = 0;
  for (int v = 0; v < V; ++v) {
    float e = orc_exp32(x[v] * invT - m);
    E[v] = (uint64_t)(e * 0x1p40f);
    se += E[v];
  }
  return se;
}

static float orc_inv_sum(uint64_t se) { return (float)(0x1p40 / (double)se); }

/* The weights W_v and their sum S of a residual (xp != NULL) or a draw from q
 * (xp == NULL), as specified above.  *resid_zero is set when a residual had
 * zero mass and q was used. */
static uint64_t orc_sample_weights(const float *xq, const float *xp, int V, float invT,
                                   uint64_t *W, int *resid_zero) {
  *resid_zero = 0;
  float mq = orc_zmax32(xq, V, invT);
  uint64_t se_q = orc_fixed_exp40(xq, V, invT, mq, W);
  if (!xp) return se_q;
  float iq = orc_inv_sum(se_q);
  float mp = orc_zmax32(xp, V, invT);
  uint64_t *Ep = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
  float ip = orc_inv_sum(orc_fixed_exp40(xp, V, invT, mp, Ep));
  free(Ep);
  uint64_t *R = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
  uint64_t S = 0;
  for (int v = 0; v < V; ++v) {
    float q = orc_exp32(xq[v] * invT - mq) * iq;
    float p = orc_exp32(xp[v] * invT - mp) * ip;
    float d = q - p;
    R[v] = (uint64_t)((d > 0.0f ? d : 0.0f) * 0x1p62f);
    S += R[v];
  }
  if (S != 0) memcpy(W, R, sizeof(uint64_t) * (size_t)V);
  free(R);
  if (S == 0) { /* residual mass zero: fall back to q ([Lesson] Passo 2) */
    *resid_zero = 1;
    return se_q;
  }
  return S;
}

/* The token of uniform u24 over weights W (cumulative sums C, total S):
 * the smallest k with C_k > t, t = floor(u24 S / 2^24); *gap gets
 * min(t - C_{k-1}, C_k - 1 - t) / S, the distance to the nearer boundary. */
static int orc_pick(const uint64_t *C, int V, uint64_t S, uint32_t u24, double *gap) {
  uint64_t t = (uint64_t)(((unsigned __int128)u24 * (unsigned __int128)S) >> 24);
  int lo = 0, hi = V - 1; /* C[V-1] = S > t, so the answer exists */
  while (lo < hi) {
    int mid = lo + (hi - lo) / 2;
    if (C[mid] > t) hi = mid;
    else lo = mid + 1;
  }
  uint64_t prev = lo ? C[lo - 1] : 0;
  uint64_t below = t - prev, above = C[lo] - 1 - t;
  *gap = (double)(below < above ? below : above) / (double)S;
  return lo;
}

/* n draws on one row (pair): tokens[i] for uniform u24[i].  Returns 0, or -1
 * when V < 1. */
int orc_sample_repro_many(const float *xq, const float *xp, int V, float invT,
                          const uint32_t *u24, int n, int32_t *tokens, double *gaps,
                          int *resid_zero) {
  if (V < 1) return -1;
  uint64_t *W = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
  uint64_t S = orc_sample_weights(xq, xp, V, invT, W, resid_zero);
  for (int v = 1; v < V; ++v) W[v] += W[v - 1]; /* cumulative sums in place */
  for (int i = 0; i < n; ++i) {
    double g;
    tokens[i] = orc_pick(W, V, S, u24[i], &g);
    if (gaps) gaps[i] = g;
  }
  free(W);
  return 0;
}

/* One draw: residual (xp != NULL) or from q (xp == NULL).  Returns the token;
 * *gap and *resid_zero as above. */
int orc_sample_repro(const float *xq, const float *xp, int V, float invT,
                     uint32_t u24, double *gap, int *resid_zero) {
  int32_t k = -1;
  orc_sample_repro_many(xq, xp, V, invT, &u24, 1, &k, gap, resid_zero);
  return k;
}

/* ------------------------------------------------------------------------
 * The verify walk ([Lesson] "O invariante" and Passo 3; [Blog] section 4,
 * spec_decode pseudocode): walk positions left to right; at the first
 * rejection j sample from residual(q_j, p_j) and stop; if every draft is
 * accepted, sample a bonus token from q_{N+1}.  The bonus is emitted only on
 * full acceptance (the blog's eagle_round listing appends it unconditionally,
 * which contradicts its own worked example of 2 accepted + 1 correction = 3
 * tokens in section 2; the lesson's reading is used).
 *
 * Generic over chain and tree: position i (0-based) is judged by verifier row
 * path[i] and draft row path[i] of the sequence, and tests token tok[i]; the
 * bonus row is verifier row path[npos].  A chain is path[i] = i.  The ratio
 * q(d)/p(d) is evaluated as exp of its logarithm so that tiny probabilities do
 * not underflow to 0/0; p(d) <= 0 means the draft logit is -inf.
 *
 * u_acc / u_samp (optional) replace the Philox uniforms, for enumeration;
 * seq_ids (optional) gives each row of the batch its sequence number in the
 * Philox counter, so that a subset of a batch can be replayed.
 * ---------------------------------------------------------------------- */
/* ------------------------------------------------------------------------
 * Greedy verification: the temperature -> 0 limit of the rule above.  Every
 * softmax becomes the point mass at the row's arg max (ties: the lowest
 * token id), so min(1, q(d)/p(d)) is 1 when d is the verifier's arg max and
 * 0 otherwise, the residual (q - p)+ is the point mass at the verifier's arg
 * max, and so is the bonus.  Only verifier rows are read: a draft token is
 * accepted iff it equals the verifier row's arg max; the first mismatch
 * emits that arg max and stops; full acceptance emits the arg max of the last
 * verifier row.  q_prob = 1 or 0 (the limit of q(d)); p_prob, margins and
 * gap are NaN (not defined in the limit).
 * ---------------------------------------------------------------------- */
int orc_argmax(const float *x, int V) {
  int k = 0;
  for (int v = 1; v < V; ++v)
    if (x[v] > x[k]) k = v;
  return k;
}

static int orc_verify_greedy(const float *vlog, int64_t v_bstride, int B, int V,
                             const int32_t *path, int path_stride, const int32_t *npos_arr,
                             const int32_t *tok, int tok_stride, int32_t *out_tokens,
                             int out_stride, int32_t *out_accept, double *out_q, double *out_p,
                             double *out_margin, int margin_stride, double *out_gap,
                             uint32_t *out_status) {
  for (int b = 0; b < B; ++b) {
    const float *vb = vlog + (int64_t)b * v_bstride;
    int npos = npos_arr[b];
    const int32_t *pb = path ? path + (int64_t)b * path_stride : NULL;
    const int32_t *tb = tok + (int64_t)b * tok_stride;
    uint32_t status = 0;
    int32_t *ot = out_tokens + (int64_t)b * out_stride;
    for (int i = 0; i < out_stride; ++i) ot[i] = -1;
    for (int i = 0; i < margin_stride; ++i) {
      if (out_q) out_q[(int64_t)b * margin_stride + i] = NAN;
      if (out_p) out_p[(int64_t)b * margin_stride + i] = NAN;
    }
    if (out_margin)
      for (int i = 0; i <= margin_stride; ++i)
        out_margin[(int64_t)b * (margin_stride + 1) + i] = NAN;
    if (out_gap) out_gap[b] = NAN;
    for (int i = 0; i <= npos; ++i) {
      int r = pb ? pb[i] : i;
      if (orc_row_bad(vb + (int64_t)r * V, V)) status |= ORC_ROW_NAN;
      if (i < npos && (tb[i] < 0 || tb[i] >= V)) status |= ORC_ROW_BAD_TOKEN;
    }
    if (status) {
      out_accept[b] = 0;
      out_status[b] = status;
      continue;
    }
    int a = npos;
    for (int i = 0; i < npos; ++i) {
      int r = pb ? pb[i] : i;
      int k = orc_argmax(vb + (int64_t)r * V, V);
      if (out_q) out_q[(int64_t)b * margin_stride + i] = (tb[i] == k) ? 1.0 : 0.0;
      if (a == npos && tb[i] != k) a = i;
    }
    for (int i = 0; i < a; ++i) ot[i] = tb[i];
    int r = pb ? pb[a] : a;
    ot[a] = orc_argmax(vb + (int64_t)r * V, V);
    out_accept[b] = a;
    out_status[b] = 0;
  }
  return 0;
}

/* The verify walk of every sequence.  Two readings of which rows a round
 * touches:
 *   early_exit = 0  every row and token of the round is checked before the
 *                   walk (any bad row or token faults the sequence), and q(d),
 *                   p(d) and the margin are reported for every position;
 *   early_exit = 1  only the rows the walk reaches, in its order ([Lesson]
 *                   Passo 3 and [Blog] section 4 spec_decode: the walk ends at
 *                   the first rejection, so nothing after it is needed): at
 *                   position i the verifier and draft rows of i and token i
 *                   are checked first (a bad one faults the sequence with the
 *                   bits found there), then judged; the bonus row is checked
 *                   only when every position passes.  q(d), p(d) and the margin
 *                   exist for positions up to the first rejection, NaN after.
 * Accepted tokens, the correction / bonus token and the accept length are the
 * same in both readings whenever neither faults. */
int orc_verify_ex(const float *vlog, int64_t v_bstride, const float *dlog,
                  int64_t d_bstride, int B, int V, float T,
                  const int32_t *path, int path_stride, const int32_t *npos_arr,
                  const int32_t *tok, int tok_stride, uint64_t seed,
                  uint64_t step, const uint32_t *u_acc, int u_acc_stride,
                  const uint32_t *u_samp, const int32_t *seq_ids,
                  int32_t *out_tokens, int out_stride,
                  int32_t *out_accept, double *out_q, double *out_p,
                  double *out_margin, int margin_stride, double *out_gap,
                  uint32_t *out_status, int early_exit) {
  if (B < 0 || V <= 0 || !(T >= 0.0f)) return -1;
  if (early_exit && T == 0.0f) return -1;
  if (T == 0.0f)
    return orc_verify_greedy(vlog, v_bstride, B, V, path, path_stride, npos_arr, tok,
                             tok_stride, out_tokens, out_stride, out_accept, out_q, out_p,
                             out_margin, margin_stride, out_gap, out_status);
  float invT = 1.0f / T;
  double Td = (double)T;
  for (int b = 0; b < B; ++b) {
    const uint32_t sid = seq_ids ? (uint32_t)seq_ids[b] : (uint32_t)b;
    const float *vb = vlog + (int64_t)b * v_bstride;
    const float *db = dlog + (int64_t)b * d_bstride;
    int npos = npos_arr[b];
    const int32_t *pb = path ? path + (int64_t)b * path_stride : NULL;
    const int32_t *tb = tok + (int64_t)b * tok_stride;
    uint32_t status = 0;
    int p_zero_seen = 0;
    int32_t *ot = out_tokens + (int64_t)b * out_stride;
    for (int i = 0; i < out_stride; ++i) ot[i] = -1;
    for (int i = 0; i < margin_stride; ++i) {
      if (out_q) out_q[(int64_t)b * margin_stride + i] = NAN;
      if (out_p) out_p[(int64_t)b * margin_stride + i] = NAN;
    }
    if (out_margin)
      for (int i = 0; i <= margin_stride; ++i)
        out_margin[(int64_t)b * (margin_stride + 1) + i] = NAN;
    /* full reading: every row / token the round could touch, before the walk */
    for (int i = 0; i <= npos && !early_exit; ++i) {
      int r = pb ? pb[i] : i;
      if (orc_row_bad(vb + (int64_t)r * V, V)) status |= ORC_ROW_NAN;
      if (i < npos && orc_row_bad(db + (int64_t)r * V, V)) status |= ORC_ROW_NAN;
      if (i < npos && (tb[i] < 0 || tb[i] >= V)) status |= ORC_ROW_BAD_TOKEN;
    }
    int a = 0, stopped = 0;
    for (int i = 0; i < npos && !status && !(early_exit && stopped); ++i) {
      int r = pb ? pb[i] : i;
      const float *xq = vb + (int64_t)r * V, *xp = db + (int64_t)r * V;
      if (early_exit) {
        /* early exit: this position's rows and token, as the walk reaches them */
        if (orc_row_bad(xq, V) || orc_row_bad(xp, V)) status |= ORC_ROW_NAN;
        if (tb[i] < 0 || tb[i] >= V) status |= ORC_ROW_BAD_TOKEN;
        if (status) break;
      }
      int d = tb[i];
      double mq, sq, mp, sp;
      orc_row_stats(xq, V, Td, &mq, &sq);
      orc_row_stats(xp, V, Td, &mp, &sp);
      double zq = (double)xq[d] / Td, zp = (double)xp[d] / Td;
      double qd = exp(zq - mq) / sq, pd = exp(zp - mp) / sp;
      double ratio;
      int p_zero = isinf(zp) && zp < 0;
      if (p_zero)
        ratio = INFINITY;
      else if (isinf(zq) && zq < 0)
        ratio = 0.0;
      else
        ratio = exp(((zq - mq) - (zp - mp)) + (log(sp) - log(sq)));
      uint32_t u24 = u_acc ? u_acc[(int64_t)b * u_acc_stride + i]
                           : orc_u24(seed, step, sid, (uint32_t)i, ORC_DRAW_ACCEPT);
      double u = (double)u24 * 0x1p-24;
      if (out_q) out_q[(int64_t)b * margin_stride + i] = qd;
      if (out_p) out_p[(int64_t)b * margin_stride + i] = pd;
      double rc = ratio < 1.0 ? ratio : 1.0;
      if (out_margin) out_margin[(int64_t)b * (margin_stride + 1) + i] = rc - u;
      if (stopped) continue;
      int acc = p_zero ? 1 : (u < rc);
      if (p_zero) p_zero_seen = 1;
      if (acc) {
        ot[i] = d;
        a = i + 1;
      } else {
        stopped = 1;
      }
    }
    if (early_exit && !status && a == npos &&
        orc_row_bad(vb + (int64_t)(pb ? pb[npos] : npos) * V, V))
      status |= ORC_ROW_NAN; /* early exit: the bonus row, reached */
    if (status) {
      /* a fault: nothing is emitted and no probability reported */
      for (int i = 0; i < out_stride; ++i) ot[i] = -1;
      for (int i = 0; i < margin_stride; ++i) {
        if (out_q) out_q[(int64_t)b * margin_stride + i] = NAN;
        if (out_p) out_p[(int64_t)b * margin_stride + i] = NAN;
      }
      if (out_margin)
        for (int i = 0; i <= margin_stride; ++i)
          out_margin[(int64_t)b * (margin_stride + 1) + i] = NAN;
      out_accept[b] = 0;
      out_status[b] = status;
      if (out_gap) out_gap[b] = NAN;
      continue;
    }
    if (p_zero_seen) status |= ORC_ROW_P_ZERO;
    /* correction (residual at position a) or bonus (verifier row path[npos]) */
    uint32_t us = u_samp ? u_samp[b]
                         : orc_u24(seed, step, sid, (uint32_t)a, ORC_DRAW_SAMPLE);
    double gap = NAN;
    int rz = 0, k;
    if (a < npos) {
      int r = pb ? pb[a] : a;
      k = orc_sample_repro(vb + (int64_t)r * V, db + (int64_t)r * V, V, invT,
                           us, &gap, &rz);
    } else {
      int r = pb ? pb[npos] : npos;
      k = orc_sample_repro(vb + (int64_t)r * V, NULL, V, invT, us, &gap, &rz);
    }
    if (rz) status |= ORC_ROW_RESID_ZERO;
    ot[a] = k;
    out_accept[b] = a;
    out_status[b] = status;
    if (out_gap) out_gap[b] = gap;
    if (out_margin)
      out_margin[(int64_t)b * (margin_stride + 1) + margin_stride] = gap;
  }
  return 0;
}

int orc_verify(const float *vlog, int64_t v_bstride, const float *dlog,
               int64_t d_bstride, int B, int V, float T,
               const int32_t *path, int path_stride, const int32_t *npos_arr,
               const int32_t *tok, int tok_stride, uint64_t seed,
               uint64_t step, const uint32_t *u_acc, int u_acc_stride,
               const uint32_t *u_samp, const int32_t *seq_ids,
               int32_t *out_tokens, int out_stride,
               int32_t *out_accept, double *out_q, double *out_p,
               double *out_margin, int margin_stride, double *out_gap,
               uint32_t *out_status) {
  return orc_verify_ex(vlog, v_bstride, dlog, d_bstride, B, V, T, path, path_stride,
                       npos_arr, tok, tok_stride, seed, step, u_acc, u_acc_stride, u_samp,
                       seq_ids, out_tokens, out_stride, out_accept, out_q, out_p,
                       out_margin, margin_stride, out_gap, out_status, 0);
}

/* ------------------------------------------------------------------------
 * Tree helpers.  A flattened draft tree of T slots per sequence: parent[0] ==
 * -1 is the root (the last committed token), parent[c] in [0, c) for a node,
 * -2 for an unused slot.  [Blog] "为什么要树，以及树怎么一次验完": number the
 * flattened nodes; each node sees only itself and its ancestors.
 * ---------------------------------------------------------------------- */
int orc_tree_valid(const int32_t *parent, const float *score, int T) {
  if (T < 1 || parent[0] != -1) return 0;
  for (int c = 1; c < T; ++c) {
    if (parent[c] == -2) continue;
    if (parent[c] < 0 || parent[c] >= c) return 0;
    if (parent[parent[c]] == -2) return 0;
    if (score && isnan(score[c])) return 0;
  }
  return 1;
}

/* Best-child walk ([Blog] section 4, eagle_round: "walk the tree along
 * best_child").  best_child is not defined on the page; read as the child with
 * the highest path score (the score the drafter attaches: parent score times
 * draft probability, same listing), ties to the lower slot index, none at a
 * leaf.  At most max_depth steps.  Returns the depth D; path[0..D]. */
int orc_tree_best_path(const int32_t *parent, const float *score, int T,
                       int max_depth, int32_t *path) {
  int D = 0, cur = 0;
  path[0] = 0;
  while (D < max_depth) {
    int best = -1;
    for (int c = 1; c < T; ++c) {
      if (parent[c] != cur) continue;
      if (best < 0 || score[c] > score[best]) best = c;
    }
    if (best < 0) break;
    path[++D] = best;
    cur = best;
  }
  return D;
}

/* Tree verify: path from the best-child walk, then the verify walk with
 * verifier row n_{k-1} judging token[n_k] (the parent's distribution is the
 * one over the token that follows it; reading of the listing, whose p_all[child]
 * indexes the node whose distribution predicts the *next* token). */
int orc_verify_tree(const float *vlog, const float *dlog, const int32_t *parent,
                    const int32_t *token, const float *score, int B, int T,
                    int max_depth, int V, float temperature, uint64_t seed,
                    uint64_t step, const int32_t *seq_ids, int32_t *out_path,
                    int32_t *out_tokens,
                    int32_t *out_accept, double *out_q, double *out_p,
                    double *out_margin, double *out_gap, uint32_t *out_status) {
  int P = max_depth + 1;
  int32_t *path = (int32_t *)calloc((size_t)B * P + 1, sizeof(int32_t));
  int32_t *tok = (int32_t *)calloc((size_t)B * (P > 1 ? P - 1 : 1) + 1, sizeof(int32_t));
  int32_t *npos = (int32_t *)calloc((size_t)(B > 0 ? B : 1), sizeof(int32_t));
  uint8_t *bad = (uint8_t *)calloc((size_t)(B > 0 ? B : 1), 1);
  for (int b = 0; b < B; ++b) {
    const int32_t *pa = parent + (int64_t)b * T;
    const float *sc = score + (int64_t)b * T;
    int32_t *pth = path + (int64_t)b * P;
    for (int i = 0; i < P; ++i) pth[i] = -1;
    if (!orc_tree_valid(pa, sc, T)) {
      bad[b] = 1;
      npos[b] = 0;
      pth[0] = 0;
      continue;
    }
    int D = orc_tree_best_path(pa, sc, T, max_depth, pth);
    npos[b] = D;
    for (int i = 0; i < D; ++i) tok[(int64_t)b * (P - 1) + i] = token[(int64_t)b * T + pth[i + 1]];
  }
  int rc = orc_verify(vlog, (int64_t)T * V, dlog, (int64_t)T * V, B, V,
                      temperature, path, P, npos, tok, P - 1, seed, step, NULL,
                      0, NULL, seq_ids, out_tokens, P, out_accept, out_q, out_p,
                      out_margin, P - 1, out_gap, out_status);
  for (int b = 0; b < B; ++b) {
    int32_t *op = out_path + (int64_t)b * P;
    for (int i = 0; i < P; ++i) op[i] = -1;
    op[0] = 0; /* the root (last committed token) is always kept */
    if (bad[b]) {
      out_status[b] = ORC_ROW_BAD_TREE;
      out_accept[b] = 0;
      for (int i = 0; i < P; ++i) out_tokens[(int64_t)b * P + i] = -1;
      if (out_gap) out_gap[b] = NAN;
      if (out_margin)
        for (int i = 0; i < P; ++i) out_margin[(int64_t)b * P + i] = NAN;
      if (out_q)
        for (int i = 0; i < P - 1; ++i) out_q[(int64_t)b * (P - 1) + i] = NAN;
      if (out_p)
        for (int i = 0; i < P - 1; ++i) out_p[(int64_t)b * (P - 1) + i] = NAN;
      continue;
    }
    if (out_status[b] & (ORC_ROW_NAN | ORC_ROW_BAD_TOKEN)) continue;
    int a = out_accept[b];
    for (int i = 0; i <= a; ++i) op[i] = path[(int64_t)b * P + i];
  }
  free(path);
  free(tok);
  free(npos);
  free(bad);
  return rc;
}

/* Ancestor mask: bit j of node n is set iff j == n or j is an ancestor of n;
 * depth = number of ancestors.  Unused slots get an empty mask and depth -1. */
void orc_tree_mask(const int32_t *parent, int B, int T, uint64_t *mask,
                   int32_t *depth) {
  int W = (T + 63) / 64;
  for (int b = 0; b < B; ++b) {
    const int32_t *pa = parent + (int64_t)b * T;
    int ok = orc_tree_valid(pa, NULL, T);
    for (int n = 0; n < T; ++n) {
      uint64_t *mk = mask + ((int64_t)b * T + n) * W;
      for (int w = 0; w < W; ++w) mk[w] = 0;
      depth[(int64_t)b * T + n] = -1;
      if (!ok || pa[n] == -2) continue;
      int d = -1;
      for (int j = n; j >= 0; j = pa[j]) {
        mk[j / 64] |= (uint64_t)1 << (j % 64);
        ++d;
      }
      depth[(int64_t)b * T + n] = d;
    }
  }
}

/* ------------------------------------------------------------------------
 * KV rollback / compaction ([Lesson] "Reversão de KV cache" and Passo 4;
 * [Blog] section 3 "copy the accepted path's KV rows together, drop the other
 * branches" and the compact_kv step of eagle_round).  Cache layout
 * [L][2][B][S][H][D] of elem_bytes each.  For every sequence, layer and K/V:
 * dst row dst_base+k <- src row src_base+rows[k], k < n_rows, all reads
 * before any write.  kv_len = dst_base + n_rows, or -1 (nothing moved) when a
 * row is out of range, n_rows is out of [0, P], or an in-place call (src ==
 * dst) has dst_base != src_base or rows not strictly increasing with
 * rows[k] >= k.  The pages put no bound on the number of rows kept, and
 * neither does this definition.
 * ---------------------------------------------------------------------- */
void orc_kv_compact(const uint8_t *src, uint8_t *dst, int L, int B, int S_src,
                    int S_dst, int H, int D, int elem_bytes,
                    const int32_t *src_base, const int32_t *dst_base,
                    const int32_t *rows, const int32_t *n_rows, int P,
                    int32_t *out_kv_len) {
  size_t rb = (size_t)H * D * elem_bytes;
  int inplace = (src == dst);
  uint8_t *tmp = (uint8_t *)malloc(rb * (size_t)(P > 0 ? P : 1));
  for (int b = 0; b < B; ++b) {
    int n = n_rows[b];
    int ok = (n >= 0 && n <= P && src_base[b] >= 0 && dst_base[b] >= 0 &&
              dst_base[b] + n <= S_dst);
    if (inplace && src_base[b] != dst_base[b]) ok = 0;
    for (int k = 0; ok && k < n; ++k) {
      int r = rows[(int64_t)b * P + k];
      if (r < 0 || src_base[b] + r >= S_src) ok = 0;
      if (inplace && (r < k || (k > 0 && r <= rows[(int64_t)b * P + k - 1]))) ok = 0;
    }
    if (!ok) {
      out_kv_len[b] = -1;
      continue;
    }
    for (int l = 0; l < L; ++l) {
      for (int kv = 0; kv < 2; ++kv) {
        size_t slab = ((size_t)l * 2 + kv) * (size_t)B + (size_t)b;
        const uint8_t *sb = src + slab * (size_t)S_src * rb;
        uint8_t *db = dst + slab * (size_t)S_dst * rb;
        for (int k = 0; k < n; ++k)
          memcpy(tmp + (size_t)k * rb,
                 sb + (size_t)(src_base[b] + rows[(int64_t)b * P + k]) * rb, rb);
        for (int k = 0; k < n; ++k)
          memcpy(db + (size_t)(dst_base[b] + k) * rb, tmp + (size_t)k * rb, rb);
      }
    }
    out_kv_len[b] = dst_base[b] + n;
  }
  free(tmp);
}

/* ------------------------------------------------------------------------
 * Speedup model ([Lesson] "O que determina a aceleração"): expected tokens
 * per verifier pass (1 - a^(N+1)) / (1 - a); wall time per token
 * (N c + 1) / E; speedup = E / (N c + 1).
 * ---------------------------------------------------------------------- */
double orc_expected_tokens(double alpha, int N) {
  if (alpha == 1.0) return (double)(N + 1);
  return (1.0 - pow(alpha, N + 1)) / (1.0 - alpha);
}

double orc_speedup(double alpha, int N, double c) {
  return orc_expected_tokens(alpha, N) / ((double)N * c + 1.0);
}

/* ------------------------------------------------------------------------
 * Dynamic draft tree (EAGLE-2; [Blog] section 5, "三代之间的变化": the tree
 * grows where the draft is confident -- a node's score is the product of the
 * draft probabilities along its path, the best-scored nodes are expanded,
 * and the tree is pruned to a node budget).  Three steps, called per level
 * by the caller that runs the draft model:
 *
 * expand:   for each frontier row (a draft logit row and the path score of
 *           the node it belongs to) the K tokens with the largest logits
 *           (equal logits in ascending token id) and their child scores
 *           = frontier score * softmax(x / T)[token] (T = 0: 1 for the
 *           first arg max, 0 for the others).  A row with a NaN or +inf
 *           logit, or all -inf, or a NaN frontier score (an empty frontier
 *           entry), proposes nothing: tokens -1, scores -inf.
 * select:   per sequence the K best candidates of a level, by score, equal
 *           scores in ascending candidate index; candidates with token -1
 *           are never chosen; missing picks are -1.
 * finalize: per sequence the T best candidates overall (score descending,
 *           then level ascending, then index ascending; candidate 0 is the
 *           root), numbered level by level (score descending, index
 *           ascending within a level); a kept node's parent is the slot of
 *           its parent candidate (-1 for the root; -2 if that candidate was
 *           not kept, which cannot happen when child scores never exceed
 *           their parent's); unused slots get parent -2, token -1, score 0.
 * ---------------------------------------------------------------------- */
int orc_tree_expand(const float *dlog, int R, int V, float T, const float *fscore, int K,
                    int32_t *out_tok, double *out_score) {
  if (R < 0 || V < 1 || K < 1 || K > V || !(T >= 0.0f)) return -1;
  double *prob = (double *)malloc(sizeof(double) * (size_t)V);
  uint8_t *taken = (uint8_t *)malloc((size_t)V);
  for (int r = 0; r < R; ++r) {
    const float *x = dlog + (int64_t)r * V;
    int32_t *ot = out_tok + (int64_t)r * K;
    double *os = out_score + (int64_t)r * K;
    if (orc_row_bad(x, V) || isnan(fscore[r])) {
      for (int k = 0; k < K; ++k) {
        ot[k] = -1;
        os[k] = -INFINITY;
      }
      continue;
    }
    int am = orc_argmax(x, V);
    if (T > 0.0f) orc_softmax(x, V, (double)T, prob);
    memset(taken, 0, (size_t)V);
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int v = 0; v < V; ++v)
        if (!taken[v] && (best < 0 || x[v] > x[best])) best = v;
      taken[best] = 1;
      ot[k] = best;
      double p = T > 0.0f ? prob[best] : (best == am ? 1.0 : 0.0);
      os[k] = (double)fscore[r] * p;
    }
  }
  free(prob);
  free(taken);
  return 0;
}

int orc_tree_select(const float *score, const int32_t *token, int B, int C, int K,
                    int32_t *out_idx) {
  if (B < 0 || C < 1 || K < 1) return -1;
  uint8_t *taken = (uint8_t *)malloc((size_t)C);
  for (int b = 0; b < B; ++b) {
    const float *s = score + (int64_t)b * C;
    const int32_t *t = token + (int64_t)b * C;
    memset(taken, 0, (size_t)C);
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int c = 0; c < C; ++c)
        if (!taken[c] && t[c] >= 0 && (best < 0 || s[c] > s[best])) best = c;
      out_idx[(int64_t)b * K + k] = best;
      if (best >= 0) taken[best] = 1;
    }
  }
  free(taken);
  return 0;
}

/* a before b in the keep order: score desc, level asc, index asc */
static int orc_keep_before(const float *s, const int32_t *lv, int a, int b) {
  if (s[a] != s[b]) return s[a] > s[b];
  if (lv[a] != lv[b]) return lv[a] < lv[b];
  return a < b;
}
/* a before b in the slot order: level asc, score desc, index asc */
static int orc_slot_before(const float *s, const int32_t *lv, int a, int b) {
  if (lv[a] != lv[b]) return lv[a] < lv[b];
  if (s[a] != s[b]) return s[a] > s[b];
  return a < b;
}

int orc_tree_finalize(const int32_t *cparent, const int32_t *ctoken, const float *cscore,
                      const int32_t *clevel, int B, int C, int Tn, int32_t *parent,
                      int32_t *token, float *score) {
  if (B < 0 || C < 1 || Tn < 1) return -1;
  int *keep = (int *)malloc(sizeof(int) * (size_t)Tn);
  int *slot = (int *)malloc(sizeof(int) * (size_t)C);
  uint8_t *taken = (uint8_t *)malloc((size_t)C);
  for (int b = 0; b < B; ++b) {
    const int32_t *cp = cparent + (int64_t)b * C, *ct = ctoken + (int64_t)b * C;
    const int32_t *cl = clevel + (int64_t)b * C;
    const float *cs = cscore + (int64_t)b * C;
    memset(taken, 0, (size_t)C);
    int n = 0;
    for (; n < Tn; ++n) { /* selection of the keep set, one pick at a time */
      int best = -1;
      for (int c = 0; c < C; ++c)
        if (!taken[c] && (c == 0 || ct[c] >= 0) && (best < 0 || orc_keep_before(cs, cl, c, best)))
          best = c;
      if (best < 0) break;
      taken[best] = 1;
      keep[n] = best;
    }
    /* slot order among the kept: insertion sort */
    for (int i = 1; i < n; ++i) {
      int v = keep[i], j = i - 1;
      while (j >= 0 && orc_slot_before(cs, cl, v, keep[j])) {
        keep[j + 1] = keep[j];
        --j;
      }
      keep[j + 1] = v;
    }
    for (int c = 0; c < C; ++c) slot[c] = -1;
    for (int i = 0; i < n; ++i) slot[keep[i]] = i;
    int32_t *op = parent + (int64_t)b * Tn, *otk = token + (int64_t)b * Tn;
    float *os = score + (int64_t)b * Tn;
    for (int i = 0; i < Tn; ++i) {
      if (i >= n) {
        op[i] = -2;
        otk[i] = -1;
        os[i] = 0.0f;
        continue;
      }
      int c = keep[i];
      op[i] = cp[c] < 0 ? -1 : (slot[cp[c]] >= 0 ? slot[cp[c]] : -2);
      otk[i] = ct[c];
      os[i] = cs[c];
    }
  }
  free(keep);
  free(slot);
  free(taken);
  return 0;
}

/* ------------------------------------------------------------------------
 * Tree-masked verifier attention, one layer.  [Blog] section 3: the verifier
 * scores the whole flattened draft tree in one forward pass, and the
 * attention mask lets every node see the committed context, itself and its
 * ancestors, never a sibling or another branch; [Lesson] "Reversão de KV
 * cache": the verifier pass over a tree runs a non-causal mask that follows
 * the tree.  Grouped-query heads: query head h reads KV head h / (Hq / Hkv).
 *
 *   q    [B][T][Hq][D]        queries of the T tree nodes (node 0 = root)
 *   kv   [2][B][S][Hkv][D]    this layer's cache, K then V; node n's own
 *                             K/V row is slot base[b] + n
 *   mask [B][T][(T+63)/64]    ancestor bitmask (orc_tree_mask)
 *
 * Row (b, n, h) sees key slots j < base[b] and j = base[b] + m for every
 * m < T whose bit is set in node n's mask.  Scores s_j = scale * <q, k_j>;
 * out = sum_j exp(s_j - M) v_j / sum_j exp(s_j - M) with M = max_j s_j, and
 * lse = M + log(sum_j exp(s_j - M)).  No visible key: out 0, lse -inf.
 * base[b] < 0 or base[b] + T > S: out and lse NaN.
 * sel lists n_sel (b, n, h) triples to compute (sel == NULL: every row in
 * [B][T][Hq] order); out is [rows][D], lse [rows] (lse may be NULL).
 * Plain double arithmetic, keys in slot order.
 * ---------------------------------------------------------------------- */
int orc_tree_attention(const float *q, const float *kv, const int32_t *base,
                       const uint64_t *mask, int B, int T, int Hq, int Hkv,
                       int D, int S, double scale, const int32_t *sel,
                       int n_sel, double *out, double *lse) {
  if (B < 1 || T < 1 || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 || D < 1 || S < 1)
    return -1;
  const int G = Hq / Hkv, W = (T + 63) / 64;
  const int64_t rows = sel ? n_sel : (int64_t)B * T * Hq;
  int32_t *vis = (int32_t *)malloc(sizeof(int32_t) * ((size_t)S + 1));
  double *s = (double *)malloc(sizeof(double) * ((size_t)S + 1));
  if (!vis || !s) {
    free(vis);
    free(s);
    return -2;
  }
  for (int64_t r = 0; r < rows; ++r) {
    int b, n, h;
    if (sel) {
      b = sel[3 * r];
      n = sel[3 * r + 1];
      h = sel[3 * r + 2];
    } else {
      b = (int)(r / ((int64_t)T * Hq));
      n = (int)(r / Hq % T);
      h = (int)(r % Hq);
    }
    double *o = out + r * D;
    const int bs = base[b];
    if (bs < 0 || (int64_t)bs + T > S) {
      for (int d = 0; d < D; ++d) o[d] = NAN;
      if (lse) lse[r] = NAN;
      continue;
    }
    const float *qr = q + (((int64_t)b * T + n) * Hq + h) * D;
    const int kh = h / G;
    const float *K = kv + (int64_t)b * S * Hkv * D;
    const float *V = kv + ((int64_t)B + b) * S * Hkv * D;
    const uint64_t *mk = mask + ((int64_t)b * T + n) * W;
    int nv = 0;
    for (int j = 0; j < bs; ++j) vis[nv++] = j;
    for (int m = 0; m < T; ++m)
      if ((mk[m / 64] >> (m % 64)) & 1) vis[nv++] = bs + m;
    if (nv == 0) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (lse) lse[r] = -INFINITY;
      continue;
    }
    double M = -INFINITY;
    for (int i = 0; i < nv; ++i) {
      const float *kr = K + ((int64_t)vis[i] * Hkv + kh) * D;
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += (double)qr[d] * (double)kr[d];
      s[i] = scale * acc;
      if (s[i] > M) M = s[i];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int i = 0; i < nv; ++i) {
      const double w = exp(s[i] - M);
      const float *vr = V + ((int64_t)vis[i] * Hkv + kh) * D;
      l += w;
      for (int d = 0; d < D; ++d) o[d] += w * (double)vr[d];
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    if (lse) lse[r] = M + log(l);
  }
  free(vis);
  free(s);
  return 0;
}
