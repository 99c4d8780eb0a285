/*
 * Oracle for the attention forward pass: a plain, slow, float64 CPU implementation.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the benchmark's CPU
 * baseline call this file. It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, step by step, for every batch row b and head h (inputs are bf16 bit
 * patterns in [B, T, H, D] layout, widened exactly to double):
 *
 *  1. RoPE at position t (habr "Autoresearch" deep dive, train.py listing, apply_rotary_emb and
 *     _precompute_rotary_embeddings): head_dim is split in halves x1 = x[0:D/2], x2 = x[D/2:D];
 *     y1 = x1*cos + x2*sin, y2 = -x1*sin + x2*cos, with angle t * base^(-2i/D) for pair i.
 *     The angles, cos and sin are evaluated in double here (the listing stores them in bf16;
 *     that storage choice is not reproduced).
 *  2. QK RMSNorm without gain (same listing, norm(): F.rms_norm over the last dim):
 *     x / sqrt(mean(x^2) + eps). The listing applies RoPE first, then the norm
 *     (CausalSelfAttention.forward); both steps commute exactly because a rotation of each
 *     pair keeps the sum of squares. Steps 1-2 are evaluated in double in the listing's order.
 *  3. The rotated, normalised q and k are rounded once to bf16 (nearest, ties to even),
 *     because the listing runs under bf16 autocast and hands bf16 q, k to the attention call.
 *     round_qk = 0 skips this rounding (information only).
 *
 *     Near ties. Any implementation evaluates steps 1-2 in some finite precision before it
 *     rounds to bf16, and where the exact value lies closer to a bf16 rounding midpoint than
 *     that evaluation's error, either neighbouring bf16 value is a correct result. The oracle
 *     therefore also reports, for every rounded element, its ambiguity radius: the largest
 *     distance from the oracle's bf16 value to any bf16 value that an evaluation within the
 *     error budget below can round to (0 for almost every element). The budget is that of an
 *     IEEE-754 single-precision evaluation in which every addition, multiplication, fused
 *     multiply-add, square root and division (or reciprocal) is correctly rounded, the squares
 *     are summed in any order, and cos / sin are those of the double angle rounded to single
 *     precision. To first order in u = 2^-24:
 *       - the sum of D squares (each exact in single precision: a bf16 value has 8 significant
 *         bits) in any order: relative error <= (D - 1) u (all terms are non-negative);
 *       - mean + eps (eps itself rounded to single precision): 2 u more; the square root
 *         halves the relative error and adds u; the reciprocal adds u: r is within
 *         (D/2 + 3) u of 1/sqrt(mean + eps) relative;
 *       - each output is a sum of two products of |x1|, |x2| with |cos| r, |sin| r (RoPE), or
 *         |x| r (no RoPE); the table entries, the products and the sum add at most 4 u of
 *         (|x1| + |x2|) r (respectively |x| r).
 *     The budget used is delta = (D/2 + 16) u * mag, mag = (|x1| + |x2|) r with RoPE and |x| r
 *     without (the margin of 9 u covers a reciprocal square root a few units in the last place
 *     from correctly rounded, second-order terms and the double evaluation here). The valid
 *     bf16 values are those between round(y - delta) and round(y + delta).
 *  4. Allowed keys of query i ("geometry_of_andrea" page, "A Máscara Causal": token t sees
 *     tokens 0..t; habr listing, flash_attn_func(..., causal=True, window_size=(W, 0))):
 *     J(i) = { j in [0, T) : (causal => j <= i),
 *                            (window >= 0 => j >= i - window and (not causal => j <= i + window)) }.
 *  4b. Grouped K/V heads (habr "Autoresearch" deep dive, train.py listing, GPTConfig.n_kv_head and
 *     CausalSelfAttention: k and v carry n_kv_head <= n_head heads with n_head % n_kv_head == 0 and
 *     go to the attention call as they are): query head h attends with K/V head
 *     h / (n_head / n_kv_head), the convention of the FlashAttention call the listing makes.
 *     n_kv_head = n_head is plain multi-head attention.
 *  5. softmax(Q K^T / sqrt(d_k)) V ("geometry_of_andrea", "O que a Atenção Calcula" and
 *     "Escalonamento por sqrt(d_k)"): s_ij = q_i . k_j / sqrt(D) for j in J(i); m = max s;
 *     Z = sum exp(s - m); p_ij = exp(s_ij - m) / Z; out_i = sum p_ij v_j; lse_i = m + ln Z.
 *     This is the two-pass exact softmax, the plain definition.
 *  6. Slack (optional outputs). With a^q, a^k the ambiguity radii of step 3, every valid choice
 *     of q^, k^ moves s_ij by at most
 *       e_ij = sum_d (a^q_id |k^_jd| + |q^_id| a^k_jd + a^q_id a^k_jd) / sqrt(D).
 *     The log-sum-exp is monotone and moves by at most lse_slack_i = ln sum_j p_ij exp(e_ij)
 *     (Jensen's inequality bounds the downward move by the same value). A weight moves to
 *     p'_ij = p_ij exp(D_j) / (p_ij exp(D_j) + R_j) with |D_j| <= e_ij and the other keys' part
 *     R_j between Rmin_j = sum_{k != j} p_ik exp(-e_ik) and Rmax_j = sum_{k != j} p_ik exp(e_ik);
 *     that ratio grows with D_j and falls with R_j, so |p'_ij - p_ij| <= p_ij g_ij with
 *     g_ij = max(exp(e_ij) / (p_ij exp(e_ij) + Rmin_j) - 1, 1 - exp(-e_ij) / (p_ij exp(-e_ij) + Rmax_j)).
 *     The weights' changes sum to zero, so output element d moves by at most
 *     out_slack_id = sum_j p_ij g_ij |v_jd - out_id|. Both are 0 when no element is ambiguous.
 *
 * eps < 0 turns the norm off; rope_base <= 0 turns RoPE off (raw mode).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* Widen a bf16 bit pattern to double (exact). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 value (8 significant bits, ties to even). */
double oracle_round_bf16(double x) {
  if (!isfinite(x) || x == 0.0) return x;
  int e;
  frexp(x, &e);             /* |x| in [2^(e-1), 2^e) */
  int ulp_exp = e - 8;      /* spacing of bf16 values in that binade */
  if (ulp_exp < -133) ulp_exp = -133; /* subnormal spacing: 2^-126 * 2^-7 */
  double y = ldexp(nearbyint(ldexp(x, -ulp_exp)), ulp_exp);
  if (fabs(y) > 3.3895313892515355e38) y = copysign(INFINITY, x); /* above the largest bf16 */
  return y;
}

/* Step 3's evaluation budget factor: delta = budget_units(D) * 2^-24 * mag. */
static double budget_units(int D) { return (double)D / 2.0 + 16.0; }

/* Steps 1-3 for one row x[0..D) at position t; the result goes to y[0..D) and, if amb is not
 * NULL, the ambiguity radius of each element to amb[0..D) (step 3; amb_scale multiplies the
 * budget, 1 for the stated one). */
static void prologue_row(const double *x, double *y, double *amb, int D, int t, double base, double eps,
                         int round_qk, double amb_scale) {
  double tmp[1024], mag[1024];
  int half = D / 2;
  for (int d = 0; d < D; ++d) {
    tmp[d] = x[d];
    mag[d] = fabs(x[d]);
  }
  if (base > 0.0) {
    for (int i = 0; i < half; ++i) {
      double theta = (double)t * pow(base, -2.0 * (double)i / (double)D);
      double c = cos(theta), s = sin(theta);
      double x1 = x[i], x2 = x[i + half];
      tmp[i] = x1 * c + x2 * s;
      tmp[i + half] = -x1 * s + x2 * c;
      mag[i] = mag[i + half] = fabs(x1) + fabs(x2);
    }
  }
  double r = 1.0;
  if (eps >= 0.0) {
    double ms = 0.0;
    for (int d = 0; d < D; ++d) ms += tmp[d] * tmp[d];
    ms /= (double)D;
    r = 1.0 / sqrt(ms + eps);
  }
  const double units = amb_scale * (budget_units(D) * ldexp(1.0, -24));
  for (int d = 0; d < D; ++d) {
    double val = tmp[d] * r;
    if (!round_qk) {
      y[d] = val;
      if (amb) amb[d] = 0.0;
      continue;
    }
    y[d] = oracle_round_bf16(val);
    if (amb) {
      double delta = units * mag[d] * r;
      double lo = oracle_round_bf16(val - delta), hi = oracle_round_bf16(val + delta);
      double a = fmax(hi - y[d], y[d] - lo);
      amb[d] = a > 0.0 ? a : 0.0;
    }
  }
}

static int key_allowed(int i, int j, int T, int window, int causal) {
  if (j < 0 || j >= T) return 0;
  if (causal && j > i) return 0;
  if (window >= 0) {
    if (j < i - window) return 0;
    if (!causal && j > i + window) return 0;
  }
  return 1;
}

static int check_dims(int B, int H, int T, int D, double base) {
  if (B < 1 || H < 1 || T < 1 || D < 1 || D > 1024) return 0;
  if (base > 0.0 && (D % 2) != 0) return 0;
  return 1;
}

/* K/V head count: 1 <= Hkv <= H and H a multiple of Hkv (step 4b). */
static int check_kv_heads(int H, int Hkv) { return Hkv >= 1 && Hkv <= H && H % Hkv == 0; }

/* Index of element (b, t, h, d) in a [B, T, H, D] tensor. */
static size_t idx4(int b, int t, int h, int d, int T, int H, int D) {
  return (((size_t)b * T + t) * H + h) * D + d;
}

/* Steps 1-3 for a whole [B, T, H, D] tensor of bf16 bits; y is [B, T, H, D] doubles and amb
 * (may be NULL) the ambiguity radii of step 3. */
int oracle_qk_prologue(const uint16_t *x, double *y, double *amb, int B, int T, int H, int D,
                       double rope_base, double eps, int round_qk, double amb_scale, int nthreads) {
  if (!x || !y || !check_dims(B, H, T, D, rope_base)) return ORACLE_EINVAL;
  long n = (long)B * T * H;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  for (long row = 0; row < n; ++row) {
    int t = (int)((row / H) % T);
    double xr[1024];
    for (int d = 0; d < D; ++d) xr[d] = bf16_to_double(x[row * D + d]);
    prologue_row(xr, y + row * D, amb ? amb + row * D : NULL, D, t, rope_base, eps, round_qk, amb_scale);
  }
  return ORACLE_OK;
}

/* Steps 4-5 for query row i of head (b, h), given prologue outputs qh ([B,T,H,D] doubles) and kh
 * ([B,T,Hkv,D] doubles) and v ([B,T,Hkv,D] bf16); the row uses K/V head hk (step 4b).
 * Writes out[0..D) and *lse; if p is non-NULL also writes the T weights p[0..T). If out_slack is
 * non-NULL, aq / ak are the ambiguity radii laid out like qh / kh, and step 6 writes
 * out_slack[0..D) and *lse_slack. */
static void attend_row(const double *qh, const double *kh, const uint16_t *v, const double *aq,
                       const double *ak, int b, int h, int hk, int i, int T, int H, int Hkv, int D,
                       int window, int causal, double *out, double *lse, double *p, double *out_slack,
                       double *lse_slack) {
  double *s = (double *)malloc(sizeof(double) * (size_t)T);
  const double scale = 1.0 / sqrt((double)D);
  const double *qi = qh + idx4(b, i, h, 0, T, H, D);
  double m = -INFINITY;
  for (int j = 0; j < T; ++j) {
    if (!key_allowed(i, j, T, window, causal)) {
      s[j] = -INFINITY;
      continue;
    }
    const double *kj = kh + idx4(b, j, hk, 0, T, Hkv, D);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
    s[j] = dot * scale;
    if (s[j] > m) m = s[j];
  }
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (out_slack)
    for (int d = 0; d < D; ++d) out_slack[d] = 0.0;
  if (lse_slack) *lse_slack = 0.0;
  if (m == -INFINITY) { /* no allowed key: empty row (only possible for an invalid mask) */
    *lse = -INFINITY;
    if (p) for (int j = 0; j < T; ++j) p[j] = 0.0;
    free(s);
    return;
  }
  double Z = 0.0;
  for (int j = 0; j < T; ++j)
    if (s[j] != -INFINITY) Z += exp(s[j] - m);
  for (int j = 0; j < T; ++j) {
    double pj = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m) / Z;
    if (p) p[j] = pj;
    if (pj == 0.0) continue;
    for (int d = 0; d < D; ++d) out[d] += pj * bf16_to_double(v[idx4(b, j, hk, d, T, Hkv, D)]);
  }
  *lse = m + log(Z);
  if (out_slack && aq && ak) {
    /* step 6: e_ij over the allowed keys, then the lse and output bounds */
    const double *aqi = aq + idx4(b, i, h, 0, T, H, D);
    int flagged[1024], nf = 0;
    for (int d = 0; d < D; ++d)
      if (aqi[d] > 0.0) flagged[nf++] = d;
    double *e = (double *)malloc(sizeof(double) * (size_t)T);
    double up = 0.0, down = 0.0; /* sum p (exp(e) - 1), sum p (exp(-e) - 1) */
    int any = 0;
    for (int j = 0; j < T; ++j) {
      e[j] = 0.0;
      if (s[j] == -INFINITY) continue;
      const double *kj = kh + idx4(b, j, hk, 0, T, Hkv, D);
      const double *akj = ak + idx4(b, j, hk, 0, T, Hkv, D);
      double acc = 0.0;
      for (int f = 0; f < nf; ++f) acc += aqi[flagged[f]] * fabs(kj[flagged[f]]);
      for (int d = 0; d < D; ++d)
        if (akj[d] > 0.0) acc += (fabs(qi[d]) + aqi[d]) * akj[d];
      e[j] = acc * scale;
      if (e[j] > 0.0) {
        double pj = exp(s[j] - m) / Z;
        up += pj * expm1(e[j]);
        down += pj * expm1(-e[j]);
        any = 1;
      }
    }
    if (any) {
      *lse_slack = log1p(up);
      const double zmax = 1.0 + up, zmin = 1.0 + down;
      for (int j = 0; j < T; ++j) {
        if (s[j] == -INFINITY) continue;
        double pj = exp(s[j] - m) / Z;
        if (pj == 0.0) continue;
        /* the other keys' share of the normaliser lies in [rmin, rmax] */
        double ep = exp(e[j]), em = exp(-e[j]);
        double rmin = fmax(zmin - pj * em, 0.0), rmax = fmax(zmax - pj * ep, 0.0);
        double g = fmax(ep / (pj * ep + rmin) - 1.0, 1.0 - em / (pj * em + rmax));
        if (g <= 0.0) continue;
        for (int d = 0; d < D; ++d)
          out_slack[d] += pj * g * fabs(bf16_to_double(v[idx4(b, j, hk, d, T, Hkv, D)]) - out[d]);
      }
    }
    free(e);
  }
  free(s);
}

/* Full forward: q is [B, T, H, D], k and v are [B, T, Hkv, D] (bf16 bits); out is [B, T, H, D]
 * doubles, lse is [B, H, T] doubles (either may be NULL). out_slack ([B, T, H, D]) and lse_slack
 * ([B, H, T]) are step 6's bounds; both NULL to skip step 6, both non-NULL to compute it.
 * amb_scale multiplies step 3's budget (1 for the stated one; tests widen it). */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                    double *lse, double *out_slack, double *lse_slack, int B, int H, int Hkv, int T,
                    int D, int window, int causal, double rope_base, double eps, int round_qk,
                    double amb_scale, int nthreads) {
  if (!q || !k || !v || !check_dims(B, H, T, D, rope_base) || !check_kv_heads(H, Hkv)) return ORACLE_EINVAL;
  if ((out_slack == NULL) != (lse_slack == NULL)) return ORACLE_EINVAL;
  const int slack = out_slack != NULL;
  size_t nq = (size_t)B * T * H * D, nk = (size_t)B * T * Hkv * D;
  double *qh = (double *)malloc(sizeof(double) * nq);
  double *kh = (double *)malloc(sizeof(double) * nk);
  double *aq = slack ? (double *)malloc(sizeof(double) * nq) : NULL;
  double *ak = slack ? (double *)malloc(sizeof(double) * nk) : NULL;
  if (!qh || !kh || (slack && (!aq || !ak))) {
    free(qh);
    free(kh);
    free(aq);
    free(ak);
    return ORACLE_ENOMEM;
  }
  int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
  oracle_qk_prologue(q, qh, aq, B, T, H, D, rope_base, eps, round_qk, amb_scale, nt);
  oracle_qk_prologue(k, kh, ak, B, T, Hkv, D, rope_base, eps, round_qk, amb_scale, nt);
  long rows = (long)B * H * T;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
  for (long r = 0; r < rows; ++r) {
    int i = (int)(r % T);
    int h = (int)((r / T) % H);
    int b = (int)(r / ((long)T * H));
    double o[1024], l, os[1024], ls;
    attend_row(qh, kh, v, aq, ak, b, h, h / (H / Hkv), i, T, H, Hkv, D, window, causal, o, &l, NULL,
               slack ? os : NULL, slack ? &ls : NULL);
    if (out)
      for (int d = 0; d < D; ++d) out[idx4(b, i, h, d, T, H, D)] = o[d];
    if (lse) lse[((size_t)b * H + h) * T + i] = l;
    if (slack) {
      for (int d = 0; d < D; ++d) out_slack[idx4(b, i, h, d, T, H, D)] = os[d];
      lse_slack[((size_t)b * H + h) * T + i] = ls;
    }
  }
  free(qh);
  free(kh);
  free(aq);
  free(ak);
  return ORACLE_OK;
}

/* Selected rows only: rows is n triples (b, h, i); out is [n, D], lse is [n], and (optional,
 * both or neither) out_slack [n, D] and lse_slack [n] are step 6's bounds.
 * The prologue is evaluated for the query row and for every allowed key of it. */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *rows,
                     long n, double *out, double *lse, double *out_slack, double *lse_slack, int B,
                     int H, int Hkv, int T, int D, int window, int causal, double rope_base,
                     double eps, int round_qk, double amb_scale, int nthreads) {
  if (!q || !k || !v || !rows || n < 0 || !check_dims(B, H, T, D, rope_base) || !check_kv_heads(H, Hkv))
    return ORACLE_EINVAL;
  if ((out_slack == NULL) != (lse_slack == NULL)) return ORACLE_EINVAL;
  const int slack = out_slack != NULL;
  for (long r = 0; r < n; ++r) {
    const int32_t *t3 = rows + 3 * r;
    if (t3[0] < 0 || t3[0] >= B || t3[1] < 0 || t3[1] >= H || t3[2] < 0 || t3[2] >= T)
      return ORACLE_EINVAL;
  }
  int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (long r = 0; r < n; ++r) {
    int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
    int hk = h / (H / Hkv);
    /* a private [1, T, 1, D] copy of the prologue for this head's needed rows */
    double *qh = (double *)calloc((size_t)T * D, sizeof(double));
    double *kh = (double *)calloc((size_t)T * D, sizeof(double));
    double *aq = slack ? (double *)calloc((size_t)T * D, sizeof(double)) : NULL;
    double *ak = slack ? (double *)calloc((size_t)T * D, sizeof(double)) : NULL;
    double xr[1024];
    for (int d = 0; d < D; ++d) xr[d] = bf16_to_double(q[idx4(b, i, h, d, T, H, D)]);
    prologue_row(xr, qh + (size_t)i * D, slack ? aq + (size_t)i * D : NULL, D, i, rope_base, eps, round_qk,
                 amb_scale);
    for (int j = 0; j < T; ++j) {
      if (!key_allowed(i, j, T, window, causal)) continue;
      for (int d = 0; d < D; ++d) xr[d] = bf16_to_double(k[idx4(b, j, hk, d, T, Hkv, D)]);
      prologue_row(xr, kh + (size_t)j * D, slack ? ak + (size_t)j * D : NULL, D, j, rope_base, eps, round_qk,
                   amb_scale);
    }
    /* attend_row indexes a [B, T, H, D] tensor; view the private copy as B = H = 1 and
       gather v into the same [1, T, 1, D] view. */
    uint16_t *vv = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * D);
    for (int j = 0; j < T; ++j)
      for (int d = 0; d < D; ++d) vv[(size_t)j * D + d] = v[idx4(b, j, hk, d, T, Hkv, D)];
    attend_row(qh, kh, vv, aq, ak, 0, 0, 0, i, T, 1, 1, D, window, causal, out + r * D, lse + r, NULL,
               slack ? out_slack + r * D : NULL, slack ? lse_slack + r : NULL);
    free(vv);
    free(qh);
    free(kh);
    free(aq);
    free(ak);
  }
  return ORACLE_OK;
}

/* The full weight matrix p[T][T] of head (b, h) (rows: queries, columns: keys). */
int oracle_attn_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v, int b, int h,
                      double *p, int B, int H, int Hkv, int T, int D, int window, int causal,
                      double rope_base, double eps, int round_qk) {
  if (!q || !k || !v || !p || !check_dims(B, H, T, D, rope_base) || !check_kv_heads(H, Hkv) || b < 0 ||
      b >= B || h < 0 || h >= H)
    return ORACLE_EINVAL;
  size_t n = (size_t)B * T * H * D;
  double *qh = (double *)malloc(sizeof(double) * n);
  double *kh = (double *)malloc(sizeof(double) * ((size_t)B * T * Hkv * D));
  if (!qh || !kh) {
    free(qh);
    free(kh);
    return ORACLE_ENOMEM;
  }
  oracle_qk_prologue(q, qh, NULL, B, T, H, D, rope_base, eps, round_qk, 1.0, 1);
  oracle_qk_prologue(k, kh, NULL, B, T, Hkv, D, rope_base, eps, round_qk, 1.0, 1);
  double o[1024], l;
  for (int i = 0; i < T; ++i)
    attend_row(qh, kh, v, NULL, NULL, b, h, h / (H / Hkv), i, T, H, Hkv, D, window, causal, o, &l,
               p + (size_t)i * T, NULL, NULL);
  free(qh);
  free(kh);
  return ORACLE_OK;
}

int oracle_num_threads(void) { return omp_get_max_threads(); }
