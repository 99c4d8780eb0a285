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
 *     pair keeps the sum of squares.
 *  3. The rotated, normalised q and k are rounded once to bf16 (nearest, ties to even),
 *     because the listing runs under bf16 autocast and hands bf16 q, k to the attention call.
 *     round_qk = 0 skips this rounding (information only).
 *
 *     This rounding is a quantisation decision, so it is taken in the same precision as the
 *     CUDA kernel takes it (prec = ORACLE_PREC_F32, the mode used for parity): steps 1-2 are
 *     then evaluated with this fixed sequence of IEEE-754 single-precision operations, each
 *     correctly rounded (fmaf, *, +, sqrtf, /):
 *         P[m] = 0 for m = 0..7; for d = 0..D-1 in order: P[d % 8] = fmaf(x[d], x[d], P[d % 8])
 *         ss = ((P[0] + P[2]) + (P[4] + P[6])) + ((P[1] + P[3]) + (P[5] + P[7]))
 *         r  = 1 / sqrtf(ss * (1/D) + eps)                      (r = 1 without the norm)
 *         c  = cos32(theta_i) * r,  s = sin32(theta_i) * r       (c = r, s = 0 without RoPE)
 *         y[i] = fmaf(x1, c, x2 * s),  y[i + D/2] = fmaf(x2, c, -(x1 * s))
 *     where cos32 / sin32 are the double cos / sin of the double angle rounded to float. In
 *     exact arithmetic this is the same function as steps 1-2 (the norm is a per-row scale and
 *     commutes with the rotation). prec = ORACLE_PREC_F64 evaluates steps 1-2 in double, in the
 *     listing's order; the pins use it.
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

#define ORACLE_PREC_F64 0
#define ORACLE_PREC_F32 1

/* Round a float to the nearest bf16 value (ties to even), returned as double (exact). */
static double round_bf16_from_float(float f) { return oracle_round_bf16((double)f); }

/* Steps 1-3 in the single-precision sequence described in the header comment. */
static void prologue_row_f32(const double *x, double *y, int D, int t, double base, double eps,
                             int round_qk) {
  base = (double)(float)base; /* the kernel receives the base as a float */
  float xf[1024];
  for (int d = 0; d < D; ++d) xf[d] = (float)x[d]; /* x holds bf16 values: exact */
  float r = 1.0f;
  if (eps >= 0.0) {
    float part[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    for (int d = 0; d < D; ++d) part[d % 8] = fmaf(xf[d], xf[d], part[d % 8]);
    float even = (part[0] + part[2]) + (part[4] + part[6]);
    float odd = (part[1] + part[3]) + (part[5] + part[7]);
    float ss = even + odd;
    float ms = ss * (1.0f / (float)D);
    float den = sqrtf(ms + (float)eps);
    r = 1.0f / den;
  }
  if (base > 0.0) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
      double theta = (double)t * pow(base, -2.0 * (double)i / (double)D);
      float c = (float)cos(theta) * r, s = (float)sin(theta) * r;
      float x1 = xf[i], x2 = xf[i + half];
      float y1 = fmaf(x1, c, x2 * s);
      float y2 = fmaf(x2, c, -(x1 * s));
      y[i] = round_qk ? round_bf16_from_float(y1) : (double)y1;
      y[i + half] = round_qk ? round_bf16_from_float(y2) : (double)y2;
    }
  } else {
    for (int d = 0; d < D; ++d) {
      float v = xf[d] * r;
      y[d] = round_qk ? round_bf16_from_float(v) : (double)v;
    }
  }
}

/* Step 1 and 2 for one row x[0..D) at position t; the result goes to y[0..D). */
static void prologue_row_f64(const double *x, double *y, int D, int t, double base, double eps,
                             int round_qk) {
  double tmp[1024];
  for (int d = 0; d < D; ++d) tmp[d] = x[d];
  if (base > 0.0) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
      double theta = (double)t * pow(base, -2.0 * (double)i / (double)D);
      double c = cos(theta), s = sin(theta);
      double x1 = x[i], x2 = x[i + half];
      tmp[i] = x1 * c + x2 * s;
      tmp[i + half] = -x1 * s + x2 * c;
    }
  }
  double r = 1.0;
  if (eps >= 0.0) {
    double ms = 0.0;
    for (int d = 0; d < D; ++d) ms += tmp[d] * tmp[d];
    ms /= (double)D;
    r = 1.0 / sqrt(ms + eps);
  }
  for (int d = 0; d < D; ++d) {
    double val = tmp[d] * r;
    y[d] = round_qk ? oracle_round_bf16(val) : val;
  }
}

static void prologue_row(const double *x, double *y, int D, int t, double base, double eps,
                         int round_qk, int prec) {
  if (prec == ORACLE_PREC_F32)
    prologue_row_f32(x, y, D, t, base, eps, round_qk);
  else
    prologue_row_f64(x, y, D, t, base, eps, round_qk);
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

/* Steps 1-3 for a whole [B, T, H, D] tensor of bf16 bits; y is [B, T, H, D] doubles. */
int oracle_qk_prologue(const uint16_t *x, double *y, int B, int T, int H, int D,
                       double rope_base, double eps, int round_qk, int prec, int nthreads) {
  if (!x || !y || !check_dims(B, H, T, D, rope_base)) return ORACLE_EINVAL;
  long n = (long)B * T * H;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  for (long row = 0; row < n; ++row) {
    int t = (int)((row / H) % T);
    double xr[1024];
    for (int d = 0; d < D; ++d) xr[d] = bf16_to_double(x[row * D + d]);
    prologue_row(xr, y + row * D, D, t, rope_base, eps, round_qk, prec);
  }
  return ORACLE_OK;
}

/* Step 4-5 for query row i of head (b, h), given prologue outputs qh ([B,T,H,D] doubles) and kh
 * ([B,T,Hkv,D] doubles) and v ([B,T,Hkv,D] bf16); the row uses K/V head hk (step 4b).
 * Writes out[0..D) and *lse; if p is non-NULL also writes the T weights p[0..T). */
static void attend_row(const double *qh, const double *kh, const uint16_t *v, int b, int h, int hk,
                       int i, int T, int H, int Hkv, int D, int window, int causal, double *out,
                       double *lse, double *p) {
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
  free(s);
}

/* Full forward: q is [B, T, H, D], k and v are [B, T, Hkv, D] (bf16 bits); out is [B, T, H, D]
 * doubles, lse is [B, H, T] doubles (either may be NULL). */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *out,
                    double *lse, int B, int H, int Hkv, int T, int D, int window, int causal,
                    double rope_base, double eps, int round_qk, int prec, int nthreads) {
  if (!q || !k || !v || !check_dims(B, H, T, D, rope_base) || !check_kv_heads(H, Hkv)) return ORACLE_EINVAL;
  size_t n = (size_t)B * T * H * D;
  double *qh = (double *)malloc(sizeof(double) * n);
  double *kh = (double *)malloc(sizeof(double) * ((size_t)B * T * Hkv * D));
  if (!qh || !kh) {
    free(qh);
    free(kh);
    return ORACLE_ENOMEM;
  }
  int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
  oracle_qk_prologue(q, qh, B, T, H, D, rope_base, eps, round_qk, prec, nt);
  oracle_qk_prologue(k, kh, B, T, Hkv, D, rope_base, eps, round_qk, prec, nt);
  long rows = (long)B * H * T;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
  for (long r = 0; r < rows; ++r) {
    int i = (int)(r % T);
    int h = (int)((r / T) % H);
    int b = (int)(r / ((long)T * H));
    double o[1024], l;
    attend_row(qh, kh, v, b, h, h / (H / Hkv), i, T, H, Hkv, D, window, causal, o, &l, NULL);
    if (out)
      for (int d = 0; d < D; ++d) out[idx4(b, i, h, d, T, H, D)] = o[d];
    if (lse) lse[((size_t)b * H + h) * T + i] = l;
  }
  free(qh);
  free(kh);
  return ORACLE_OK;
}

/* Selected rows only: rows is n triples (b, h, i); out is [n, D], lse is [n].
 * The prologue is evaluated for the query row and for every allowed key of it. */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, const int32_t *rows,
                     long n, double *out, double *lse, int B, int H, int Hkv, int T, int D,
                     int window, int causal, double rope_base, double eps, int round_qk, int prec,
                     int nthreads) {
  if (!q || !k || !v || !rows || n < 0 || !check_dims(B, H, T, D, rope_base) || !check_kv_heads(H, Hkv))
    return ORACLE_EINVAL;
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
    double xr[1024];
    for (int d = 0; d < D; ++d) xr[d] = bf16_to_double(q[idx4(b, i, h, d, T, H, D)]);
    prologue_row(xr, qh + (size_t)i * D, D, i, rope_base, eps, round_qk, prec);
    for (int j = 0; j < T; ++j) {
      if (!key_allowed(i, j, T, window, causal)) continue;
      for (int d = 0; d < D; ++d) xr[d] = bf16_to_double(k[idx4(b, j, hk, d, T, Hkv, D)]);
      prologue_row(xr, kh + (size_t)j * D, D, j, rope_base, eps, round_qk, prec);
    }
    /* attend_row indexes a [B, T, H, D] tensor; view the private copy as B = H = 1 and
       gather v into the same [1, T, 1, D] view. */
    uint16_t *vv = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)T * D);
    for (int j = 0; j < T; ++j)
      for (int d = 0; d < D; ++d) vv[(size_t)j * D + d] = v[idx4(b, j, hk, d, T, Hkv, D)];
    attend_row(qh, kh, vv, 0, 0, 0, i, T, 1, 1, D, window, causal, out + r * D, lse + r, NULL);
    free(vv);
    free(qh);
    free(kh);
  }
  return ORACLE_OK;
}

/* The full weight matrix p[T][T] of head (b, h) (rows: queries, columns: keys). */
int oracle_attn_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v, int b, int h,
                      double *p, int B, int H, int Hkv, int T, int D, int window, int causal,
                      double rope_base, double eps, int round_qk, int prec) {
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
  oracle_qk_prologue(q, qh, B, T, H, D, rope_base, eps, round_qk, prec, 1);
  oracle_qk_prologue(k, kh, B, T, Hkv, D, rope_base, eps, round_qk, prec, 1);
  double o[1024], l;
  for (int i = 0; i < T; ++i)
    attend_row(qh, kh, v, b, h, h / (H / Hkv), i, T, H, Hkv, D, window, causal, o, &l, p + (size_t)i * T);
  free(qh);
  free(kh);
  return ORACLE_OK;
}

int oracle_num_threads(void) { return omp_get_max_threads(); }
