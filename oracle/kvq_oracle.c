/*
 * CPU oracle for the quantized KV cache -- TEST INFRASTRUCTURE ONLY.
 * See kvq_oracle.h for the sources cited below ([KIVI], [HF], [INNERQ] ...).
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared.
 * float arithmetic is IEEE single precision with round-to-nearest-even and
 * no fused multiply-add, so every quantization decision below is the plain
 * fp32 formula evaluated one operation at a time.
 */
#include "kvq_oracle.h"

#include <fenv.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

int orc_rounding_is_nearest(void) { return fegetround() == FE_TONEAREST; }

/* IEEE binary16 -> binary32, exact. */
float orc_half_to_float(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int man = h & 0x3ff;
  float v;
  if (expo == 0)
    v = ldexpf((float)man, -24); /* zero or subnormal: man * 2^-24 */
  else if (expo == 31)
    v = man ? NAN : INFINITY;
  else
    v = ldexpf((float)(man | 0x400), expo - 25); /* (1024 + man) * 2^(e-25) */
  return sign ? -v : v;
}

/*
 * IEEE binary32 -> binary16, round to nearest even; overflow gives infinity,
 * NaN stays NaN.  Written from the two formats' definitions: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; subnormals in units of 2^-24.
 */
uint16_t orc_float_to_half(float f) {
  uint32_t x;
  memcpy(&x, &f, sizeof(x));
  const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  const uint32_t ax = x & 0x7fffffffu;
  if (ax >= 0x7f800000u) return sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u);
  if (ax >= 0x477ff000u) return sign | 0x7c00u;  /* >= 65520: rounds past 65504 */
  const int e = (int)(ax >> 23) - 127;           /* unbiased exponent */
  if (e < -25) return sign;                      /* below 2^-25: rounds to zero */
  const uint32_t m = (ax & 0x7fffffu) | 0x800000u;  /* 24-bit significand */
  /* keep 11 significant bits for a normal result; a subnormal result counts
   * units of 2^-24, i.e. m * 2^(e+1) */
  const int shift = e >= -14 ? 13 : -(e + 1);
  uint32_t q = m >> shift;
  const uint32_t rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1;
  if (e >= -14) /* q in [0x400, 0x800]; a carry to 0x800 moves to the next exponent */
    return sign | (uint16_t)((((uint32_t)(e + 15)) << 10) + (q - 0x400u));
  return sign | (uint16_t)q;                     /* 0x400 = the smallest normal */
}

static float round_to_half(float f) { return orc_half_to_float(orc_float_to_half(f)); }

static void min_max(const float *x, int n, float *mn, float *mx) {
  float lo = x[0], hi = x[0];
  for (int i = 1; i < n; ++i) {
    if (x[i] < lo) lo = x[i];
    if (x[i] > hi) hi = x[i];
  }
  /* -0 and +0 compare equal; keep the result independent of their order. */
  *mn = lo + 0.0f;
  *mx = hi + 0.0f;
}

/*
 * Asymmetric uniform quantizer of one group ([HF] §2.1: X_Q = round(X/S) - Z
 * with scale S and zero offset Z; [KIVI] 2-bit asymmetric).  Written in the
 * min/scale form: scale = (max - min) / (2^b - 1), zero = min,
 * u = clamp(rint((x - min) / scale), 0, 2^b - 1), dequantized u*scale + zero.
 * A constant group (max == min) stores scale 0 and all codes 0.
 */
void orc_quant_asym(const float *x, int n, int bits, float *scale, float *zero,
                    uint8_t *u, int64_t ustride) {
  const float top = (float)((1 << bits) - 1);
  float mn, mx;
  min_max(x, n, &mn, &mx);
  *zero = mn;
  if (mx == mn) {
    *scale = 0.0f;
    for (int i = 0; i < n; ++i) u[i * ustride] = 0;
    return;
  }
  const float s = (mx - mn) / top;
  *scale = s;
  for (int i = 0; i < n; ++i) {
    float r = rintf((x[i] - mn) / s);
    if (r < 0.0f) r = 0.0f;
    if (r > top) r = top;
    u[i * ustride] = (uint8_t)r;
  }
}

/*
 * Symmetric quantizer of one group ([HF] §2.1: range symmetric about zero;
 * [INNERQ] 方法论 2).  a = max(|min|, |max|), scale = a / (2^(b-1) - 1),
 * q = clamp(rint(x / scale), -(2^(b-1) - 1), 2^(b-1) - 1).  Stored as the
 * unsigned code u = q + 2^(b-1) with zero = -2^(b-1) * scale, so that
 * u*scale + zero = q*scale dequantizes both modes with one formula.
 */
void orc_quant_sym(const float *x, int n, int bits, float *scale, float *zero,
                   uint8_t *u, int64_t ustride) {
  const int half = 1 << (bits - 1);
  const float lim = (float)(half - 1);
  float mn, mx;
  min_max(x, n, &mn, &mx);
  const float a = fmaxf(fabsf(mn), fabsf(mx));
  const float s = a / lim;
  *scale = s;
  *zero = -(float)half * s;
  for (int i = 0; i < n; ++i) {
    float r = rintf(x[i] / s);
    if (r < -lim) r = -lim;
    if (r > lim) r = lim;
    u[i * ustride] = (uint8_t)((int)r + half);
  }
}

/*
 * fp16 metadata (a cache-format variant; the pages fix no storage precision
 * for scales and zero points).  Reading: the fp32 scale and zero above are
 * rounded once to fp16, and the codes are taken with the stored values, so
 * dequantization u*scale + zero uses exactly what is stored.  A scale that
 * rounds to 0 is a constant group (all codes 0, or q = 0 when symmetric).
 */
void orc_quant_asym_f16(const float *x, int n, int bits, float *scale, float *zero,
                        uint8_t *u, int64_t ustride) {
  const float top = (float)((1 << bits) - 1);
  float mn, mx;
  min_max(x, n, &mn, &mx);
  const float z = round_to_half(mn);
  const float s = mx == mn ? 0.0f : round_to_half((mx - mn) / top);
  *zero = z;
  *scale = s;
  for (int i = 0; i < n; ++i) {
    float r = s == 0.0f ? 0.0f : rintf((x[i] - z) / s);
    if (r < 0.0f) r = 0.0f;
    if (r > top) r = top;
    u[i * ustride] = (uint8_t)r;
  }
}

void orc_quant_sym_f16(const float *x, int n, int bits, float *scale, float *zero,
                       uint8_t *u, int64_t ustride) {
  const int half = 1 << (bits - 1);
  const float lim = (float)(half - 1);
  float mn, mx;
  min_max(x, n, &mn, &mx);
  const float a = fmaxf(fabsf(mn), fabsf(mx));
  const float s = round_to_half(a / lim);
  *scale = s;
  *zero = -(float)half * s;
  for (int i = 0; i < n; ++i) {
    float r = s == 0.0f ? 0.0f : rintf(x[i] / s);
    if (r < -lim) r = -lim;
    if (r > lim) r = lim;
    u[i * ustride] = (uint8_t)((int)r + half);
  }
}

/*
 * Per-group choice between the two ([INNERQ] 方法论 2: symmetric when the group
 * is centred at zero, asymmetric otherwise; the page gives no threshold).
 * Reading used: symmetric iff the group is not constant and its midpoint
 * (max + min) / 2 lies within half an asymmetric step of zero, i.e.
 * |max + min| <= (max - min) / (2^b - 1).
 */
int orc_choose_symmetric(float mn, float mx, int bits) {
  if (mx == mn) return 0;
  const float step = (mx - mn) / (float)((1 << bits) - 1);
  return fabsf(mx + mn) <= step;
}

/* ---- dense-and-sparse outliers ([KVQ4]) -------------------------------- */

/*
 * The k elements of largest magnitude of one fp16 row ([d] bits): those are
 * the row's outliers.  The page computes per-token outlier thresholds online
 * and keeps about 1 % of the elements; read as a fixed count k per token
 * (1 % of d rounded up, chosen by the caller), equal magnitudes going to the
 * lower channel.  idx receives the k channels in ascending order.
 */
void orc_select_outliers(const uint16_t *row, int d, int k, uint16_t *idx) {
  uint8_t taken[256] = {0};
  for (int j = 0; j < k; ++j) {
    int best = -1;
    float bm = -1.0f;
    for (int c = 0; c < d; ++c) {
      const float m = fabsf(orc_half_to_float(row[c]));
      if (!taken[c] && m > bm) {
        bm = m;
        best = c;
      }
    }
    taken[best] = 1;
  }
  int n = 0;
  for (int c = 0; c < d; ++c)
    if (taken[c]) idx[n++] = (uint16_t)c;
}

/* Records the outliers of the token row src (fp16, [d]) as token t's list
 * and marks them in is_out[d]. */
static void record_outliers(const orc_head *s, const uint16_t *src, int64_t t,
                            uint16_t *oidx, uint16_t *oval, uint8_t *is_out) {
  const int k = s->outliers;
  memset(is_out, 0, (size_t)s->d);
  orc_select_outliers(src, s->d, k, oidx + t * k);
  for (int j = 0; j < k; ++j) {
    const int c = oidx[t * k + j];
    oval[t * k + j] = src[c];
    is_out[c] = 1;
  }
}

/*
 * Asymmetric quantization of the inliers of one group: the statistics come
 * from the elements with is_out == 0 only ([KVQ4]: removing the outliers
 * narrows the range the codes span); outlier positions store code 0 (the
 * decode reads their fp16 value instead).  No inlier: scale 0, zero 0.
 */
static void quant_inliers(const orc_head *s, const float *x, const uint8_t *is_out, int n,
                          float *scale, float *zero, uint8_t *u, int64_t ustride) {
  float in[256];
  uint8_t code[256];
  int m = 0;
  for (int i = 0; i < n; ++i)
    if (!is_out[i]) in[m++] = x[i];
  if (m == 0) {
    *scale = 0.0f;
    *zero = 0.0f;
  } else {
    (s->meta_f16 ? orc_quant_asym_f16 : orc_quant_asym)(in, m, s->bits, scale, zero, code, 1);
  }
  m = 0;
  for (int i = 0; i < n; ++i) u[i * ustride] = is_out[i] ? 0 : code[m++];
}

/* ---- KIVI ------------------------------------------------------------- */

/* Key group: G consecutive tokens (rows of src, stride d) quantized per
 * channel ([KIVI] 工作原理: keys grouped every G tokens, quantized along the
 * channel dimension).  Destination: tokens t0 .. t0+G-1, t0 a multiple of G. */
static void kivi_quant_key_group(orc_head *s, const uint16_t *src, int64_t t0) {
  const int d = s->d, G = s->k_group;
  float *x = (float *)malloc(sizeof(float) * (size_t)G);
  /* with outliers: each token's are found over its own row ([KVQ4]: per
   * token, online), and each channel's statistics skip the group's tokens
   * that hold an outlier there */
  uint8_t *mask = s->outliers ? (uint8_t *)malloc((size_t)G * (size_t)d) : 0, col[256];
  if (mask)
    for (int i = 0; i < G; ++i)
      record_outliers(s, src + (int64_t)i * d, t0 + i, s->k_oidx, s->k_oval, mask + i * d);
  for (int c = 0; c < d; ++c) {
    for (int i = 0; i < G; ++i) x[i] = orc_half_to_float(src[(int64_t)i * d + c]);
    float *scale = &s->k_scale[(t0 / G) * d + c], *zero = &s->k_zero[(t0 / G) * d + c];
    if (mask) {
      for (int i = 0; i < G; ++i) col[i] = mask[i * d + c];
      quant_inliers(s, x, col, G, scale, zero, &s->k_u[t0 * d + c], d);
    } else {
      (s->meta_f16 ? orc_quant_asym_f16 : orc_quant_asym)(x, G, s->bits, scale, zero,
                                                           &s->k_u[t0 * d + c], d);
    }
  }
  free(mask);
  free(x);
}

/* Value token: quantized per token in groups of v_group channels
 * ([KIVI] 为什么…: values per token); with outliers, the token's are found
 * over the whole row and each group's statistics skip them. */
static void kivi_quant_value_token(orc_head *s, const uint16_t *src, int64_t t) {
  const int d = s->d, Gv = s->v_group, ng = d / Gv;
  float x[256];
  uint8_t is_out[256];
  if (s->outliers) record_outliers(s, src, t, s->v_oidx, s->v_oval, is_out);
  for (int j = 0; j < ng; ++j) {
    for (int i = 0; i < Gv; ++i) x[i] = orc_half_to_float(src[j * Gv + i]);
    float *scale = &s->v_scale[t * ng + j], *zero = &s->v_zero[t * ng + j];
    if (s->outliers)
      quant_inliers(s, x, is_out + j * Gv, Gv, scale, zero, &s->v_u[t * d + j * Gv], 1);
    else
      (s->meta_f16 ? orc_quant_asym_f16 : orc_quant_asym)(x, Gv, s->bits, scale, zero,
                                                           &s->v_u[t * d + j * Gv], 1);
  }
}

/* ---- InnerQ ----------------------------------------------------------- */

/* One token, groups of `group` consecutive channels along the inner (head)
 * dimension, each group symmetric or asymmetric ([INNERQ] 方法论 1-2).  With
 * `norm` (keys under the one-shot normalization) channel c is first scaled
 * by 1 / norm[c]: the fp32 reciprocal, then one fp32 product. */
static void innerq_quant_token(const orc_head *s, const uint16_t *src, int group,
                               int64_t t, uint8_t *u, float *scale, float *zero,
                               uint8_t *sym, const float *norm) {
  const int d = s->d, ng = d / group;
  float x[256];
  for (int j = 0; j < ng; ++j) {
    for (int i = 0; i < group; ++i) {
      x[i] = orc_half_to_float(src[j * group + i]);
      if (norm) {
        const float r = 1.0f / norm[j * group + i];
        x[i] = x[i] * r;
      }
    }
    float mn, mx;
    min_max(x, group, &mn, &mx);
    const int is_sym = orc_choose_symmetric(mn, mx, s->bits);
    sym[t * ng + j] = (uint8_t)is_sym;
    if (is_sym)
      (s->meta_f16 ? orc_quant_sym_f16 : orc_quant_sym)(
          x, group, s->bits, &scale[t * ng + j], &zero[t * ng + j], &u[t * d + j * group], 1);
    else
      (s->meta_f16 ? orc_quant_asym_f16 : orc_quant_asym)(
          x, group, s->bits, &scale[t * ng + j], &zero[t * ng + j], &u[t * d + j * group], 1);
  }
}

static void innerq_quant_kv(orc_head *s, const uint16_t *k, const uint16_t *v, int64_t t) {
  innerq_quant_token(s, k, s->k_group, t, s->k_u, s->k_scale, s->k_zero, s->k_sym,
                     s->k_normalize ? s->k_norm : 0);
  innerq_quant_token(s, v, s->v_group, t, s->v_u, s->v_scale, s->v_zero, s->v_sym, 0);
}

/* One-shot per-channel key normalization ([INNERQ] 关键贡献, 方法论 4): the
 * prompt's keys are scaled once per channel and the factor is folded into
 * the query.  The pages fix no statistic; the factor of channel c is the
 * largest |K[t][c]| over the T prompt tokens (sinks and window included), 1
 * when that is 0 (or T = 0).  Keys appended later use the same factors. */
static void innerq_key_norms(orc_head *s, const uint16_t *K, int64_t T) {
  const int d = s->d;
  for (int c = 0; c < d; ++c) {
    float a = 0.0f;
    for (int64_t t = 0; t < T; ++t) {
      const float x = fabsf(orc_half_to_float(K[t * d + c]));
      if (x > a) a = x;
    }
    s->k_norm[c] = a > 0.0f ? a : 1.0f;
  }
}

/* ---- cache state machine ---------------------------------------------- */

/* Values held quantized: they follow the keys (batch flush), except for
 * KIVI's value queue, which keeps its own count. */
static int64_t values_quantized(const orc_head *s) {
  return s->v_queue ? s->n_vquant : s->n_quant;
}

/*
 * Prefill of one head's prompt K, V ([T][d] fp16).
 * KIVI ([KIVI] 工作原理): the first l - r tokens, l - r a multiple of R (hence
 *   of G), are quantized; the last r = T mod R stay fp16 in the residual.
 *   With v_queue the values are a queue instead (the page's value
 *   paragraph): the last min(T, R - 1) values stay fp16, the rest are
 *   quantized per token.
 * InnerQ ([INNERQ] 方法论 4; [KVQ5]): the first S tokens stay fp16 as sinks,
 *   the last W as the recent window, the tokens between are quantized.
 * Returns 0, or -1 when the quantized region would exceed the capacity.
 */
int orc_prefill(orc_head *s, const uint16_t *K, const uint16_t *V, int64_t T) {
  const int d = s->d;
  s->n_flush = 0;
  if (s->scheme == ORC_KIVI) {
    const int R = s->residual, G = s->k_group;
    const int64_t nq = T - T % R;
    /* the value queue ([KIVI] 工作原理, value paragraph) holds the newest
     * values until it reaches R, then its oldest is quantized: after the
     * prompt it holds the last min(T, R - 1) values */
    const int64_t nvq = !s->v_queue ? nq : (T >= R ? T - (R - 1) : 0);
    if (nq > s->cap || nvq > s->cap) return -1;
    for (int64_t g = 0; g < nq / G; ++g) kivi_quant_key_group(s, K + g * G * d, g * G);
    for (int64_t t = 0; t < nvq; ++t) kivi_quant_value_token(s, V + t * d, t);
    memcpy(s->k_res, K + nq * d, sizeof(uint16_t) * (size_t)((T - nq) * d));
    memcpy(s->v_res, V + nvq * d, sizeof(uint16_t) * (size_t)((T - nvq) * d));
    s->n_quant = nq;
    s->n_resid = T - nq;
    s->n_vquant = nvq;
    s->n_sink_used = 0;
    return 0;
  }
  const int64_t ns = T < s->n_sink ? T : s->n_sink;
  const int64_t rest = T - ns;
  const int64_t nw = rest < s->residual ? rest : s->residual;
  const int64_t nq = rest - nw;
  if (nq > s->cap) return -1;
  if (s->k_normalize) innerq_key_norms(s, K, T);
  memcpy(s->k_sink, K, sizeof(uint16_t) * (size_t)(ns * d));
  memcpy(s->v_sink, V, sizeof(uint16_t) * (size_t)(ns * d));
  for (int64_t t = 0; t < nq; ++t) innerq_quant_kv(s, K + (ns + t) * d, V + (ns + t) * d, t);
  memcpy(s->k_res, K + (T - nw) * d, sizeof(uint16_t) * (size_t)(nw * d));
  memcpy(s->v_res, V + (T - nw) * d, sizeof(uint16_t) * (size_t)(nw * d));
  s->n_sink_used = ns;
  s->n_quant = nq;
  s->n_resid = nw;
  return 0;
}

/*
 * One decode token (k, v: [d] fp16).
 * KIVI ([KIVI] 工作原理; [HF] §3.1): the token joins the fp16 residual; when the
 *   residual reaches R tokens all R are quantized (keys as R/G groups, values
 *   per token), appended to the quantized region, and the residual empties.
 *   With v_queue only the keys flush so; the value is pushed onto the value
 *   queue, and once the queue holds R values its oldest is quantized per
 *   token and appended to the quantized values.
 * InnerQ ([INNERQ] 方法论 4): sinks fill first, then the window; once the
 *   window holds W tokens its oldest token is quantized and appended to the
 *   quantized region, and the new token takes its place.
 * Returns 0, or -1 (state unchanged) when the quantized region is full.
 */
int orc_append(orc_head *s, const uint16_t *k, const uint16_t *v) {
  const int d = s->d;
  const size_t row = sizeof(uint16_t) * (size_t)d;
  if (s->scheme == ORC_KIVI) {
    const int R = s->residual, G = s->k_group;
    const int64_t held = s->n_quant + s->n_resid;  /* tokens before this one */
    int64_t nv = held - s->n_vquant;               /* queued fp16 values (queue) */
    if (s->n_resid + 1 == R && s->n_quant + R > s->cap) return -1;
    if (s->v_queue && nv + 1 == R && s->n_vquant + 1 > s->cap) return -1;
    if (s->v_queue && (nv < 0 || nv >= R)) return -1;  /* not a reachable queue state */
    memcpy(s->k_res + s->n_resid * d, k, row);
    if (!s->v_queue) memcpy(s->v_res + s->n_resid * d, v, row);
    s->n_resid += 1;
    if (s->n_resid == R) {
      for (int g = 0; g < R / G; ++g)
        kivi_quant_key_group(s, s->k_res + (int64_t)g * G * d, s->n_quant + (int64_t)g * G);
      if (!s->v_queue)
        for (int t = 0; t < R; ++t)
          kivi_quant_value_token(s, s->v_res + (int64_t)t * d, s->n_quant + t);
      s->n_quant += R;
      s->n_resid = 0;
      s->n_flush += 1;
    }
    if (s->v_queue) {
      /* push the value; once the queue holds R, its oldest is quantized */
      memcpy(s->v_res + nv * d, v, row);
      nv += 1;
      if (nv == R) {
        kivi_quant_value_token(s, s->v_res, s->n_vquant);
        s->n_vquant += 1;
        memmove(s->v_res, s->v_res + d, row * (size_t)(R - 1));
      }
    }
    return 0;
  }
  if (s->n_sink_used < s->n_sink) {
    memcpy(s->k_sink + s->n_sink_used * d, k, row);
    memcpy(s->v_sink + s->n_sink_used * d, v, row);
    s->n_sink_used += 1;
    return 0;
  }
  if (s->n_resid < s->residual) {
    memcpy(s->k_res + s->n_resid * d, k, row);
    memcpy(s->v_res + s->n_resid * d, v, row);
    s->n_resid += 1;
    return 0;
  }
  if (s->n_quant + 1 > s->cap) return -1;
  if (s->residual == 0) { /* no window: the token itself is quantized */
    innerq_quant_kv(s, k, v, s->n_quant);
    s->n_quant += 1;
    return 0;
  }
  innerq_quant_kv(s, s->k_res, s->v_res, s->n_quant);
  s->n_quant += 1;
  memmove(s->k_res, s->k_res + d, row * (size_t)(s->residual - 1));
  memmove(s->v_res, s->v_res + d, row * (size_t)(s->residual - 1));
  memcpy(s->k_res + (int64_t)(s->residual - 1) * d, k, row);
  memcpy(s->v_res + (int64_t)(s->residual - 1) * d, v, row);
  return 0;
}

/* fp16 outlier of token t at channel c from its list, or -1 when c is an
 * inlier ([KVQ4]: the sparse part holds the outliers at full precision). */
static int outlier_slot(const orc_head *s, const uint16_t *oidx, int64_t t, int c) {
  for (int j = 0; j < s->outliers; ++j)
    if (oidx[t * s->outliers + j] == c) return j;
  return -1;
}

/* Dequantized key / value element of quantized token t, channel c, in fp64
 * (an outlier: its fp16 value). */
static double key_hat(const orc_head *s, int64_t t, int c) {
  const int d = s->d;
  const int o = s->outliers ? outlier_slot(s, s->k_oidx, t, c) : -1;
  if (o >= 0) return (double)orc_half_to_float(s->k_oval[t * s->outliers + o]);
  const double u = (double)s->k_u[t * d + c];
  if (s->scheme == ORC_KIVI) {
    const int64_t i = (t / s->k_group) * d + c;
    return u * (double)s->k_scale[i] + (double)s->k_zero[i];
  }
  const int64_t i = t * (d / s->k_group) + c / s->k_group;
  return u * (double)s->k_scale[i] + (double)s->k_zero[i];
}

static double value_hat(const orc_head *s, int64_t t, int c) {
  const int d = s->d;
  const int o = s->outliers ? outlier_slot(s, s->v_oidx, t, c) : -1;
  if (o >= 0) return (double)orc_half_to_float(s->v_oval[t * s->outliers + o]);
  const int64_t i = t * (d / s->v_group) + c / s->v_group;
  return (double)s->v_u[t * d + c] * (double)s->v_scale[i] + (double)s->v_zero[i];
}

/*
 * Decode attention of one query head q ([d] fp16) over the whole cache in
 * fp64: softmax(tau * q . k) . v over the fp16 sink tokens, the dequantized
 * tokens and the fp16 residual / window tokens ([IKV]: fp16 tokens joined
 * with the dequantized cache; [KIVI] 背景: every decode step reads the whole
 * cache).  Max-subtracted softmax.  An empty cache gives a zero output.
 * Returns 0, or -1 on allocation failure.
 */
int orc_attend(const orc_head *s, const uint16_t *q, double tau, double *out) {
  const int d = s->d;
  const int64_t n = s->n_sink_used + s->n_quant + s->n_resid;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (n == 0) return 0;
  double *sc = (double *)malloc(sizeof(double) * (size_t)n);
  double *qd = (double *)malloc(sizeof(double) * (size_t)d);
  if (!sc || !qd) { free(sc); free(qd); return -1; }
  for (int c = 0; c < d; ++c) qd[c] = (double)orc_half_to_float(q[c]);

  int64_t i = 0;
  for (int64_t t = 0; t < s->n_sink_used; ++t, ++i) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += qd[c] * (double)orc_half_to_float(s->k_sink[t * d + c]);
    sc[i] = tau * acc;
  }
  for (int64_t t = 0; t < s->n_quant; ++t, ++i) {
    /* normalized keys: the factor is folded into the query */
    double acc = 0.0;
    for (int c = 0; c < d; ++c)
      acc += qd[c] * (s->k_normalize ? (double)s->k_norm[c] : 1.0) * key_hat(s, t, c);
    sc[i] = tau * acc;
  }
  for (int64_t t = 0; t < s->n_resid; ++t, ++i) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += qd[c] * (double)orc_half_to_float(s->k_res[t * d + c]);
    sc[i] = tau * acc;
  }

  double m = sc[0];
  for (int64_t j = 1; j < n; ++j) if (sc[j] > m) m = sc[j];
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) { sc[j] = exp(sc[j] - m); l += sc[j]; }

  i = 0;
  for (int64_t t = 0; t < s->n_sink_used; ++t, ++i)
    for (int c = 0; c < d; ++c) out[c] += sc[i] * (double)orc_half_to_float(s->v_sink[t * d + c]);
  const int64_t nvq = values_quantized(s);
  for (int64_t t = 0; t < nvq; ++t, ++i)
    for (int c = 0; c < d; ++c) out[c] += sc[i] * value_hat(s, t, c);
  for (int64_t t = 0; t < n - s->n_sink_used - nvq; ++t, ++i)
    for (int c = 0; c < d; ++c) out[c] += sc[i] * (double)orc_half_to_float(s->v_res[t * d + c]);
  for (int c = 0; c < d; ++c) out[c] /= l;

  free(sc);
  free(qd);
  return 0;
}

/*
 * Rotary position embedding of one vector x ([d], fp64) at position p.  The
 * pages say only that RoPE turns pairs of channels by position-dependent
 * amounts ([KVQ2]); the rotation itself is RoFormer's, as LLaMA applies it:
 * channels 2i and 2i+1 form pair i, turned counter-clockwise by the angle
 * p * theta_i with theta_i = base^(-2i/d).
 */
static void rope_rotate(double *x, int d, double base, double p) {
  for (int i = 0; i < d / 2; ++i) {
    const int ca = 2 * i, cb = 2 * i + 1;
    const double theta = pow(base, -2.0 * i / d);
    const double c = cos(p * theta), sn = sin(p * theta);
    const double a = x[ca], b = x[cb];
    x[ca] = a * c - b * sn;
    x[cb] = a * sn + b * c;
  }
}

/*
 * Key (k != 0) or value row of the j-th token the cache holds, in arrival
 * order: the fp16 sinks, the quantized tokens (dequantized in fp64; a
 * normalized key is multiplied back by its channel factor), then the fp16
 * residual / window tokens, oldest first.
 */
static void token_row(const orc_head *s, int64_t j, int k, double *row) {
  const int d = s->d;
  if (j < s->n_sink_used) {
    const uint16_t *src = (k ? s->k_sink : s->v_sink) + j * d;
    for (int c = 0; c < d; ++c) row[c] = (double)orc_half_to_float(src[c]);
    return;
  }
  j -= s->n_sink_used;
  const int64_t nq = k ? s->n_quant : values_quantized(s);
  if (j < nq) {
    for (int c = 0; c < d; ++c)
      row[c] = k ? (s->k_normalize ? (double)s->k_norm[c] : 1.0) * key_hat(s, j, c)
                 : value_hat(s, j, c);
    return;
  }
  j -= nq;
  const uint16_t *src = (k ? s->k_res : s->v_res) + j * d;
  for (int c = 0; c < d; ++c) row[c] = (double)orc_half_to_float(src[c]);
}

/*
 * Decode attention over keys cached BEFORE the rotary position embedding
 * ([KVQ2]: keys quantized pre-RoPE, the embedding applied after
 * dequantization, at attention time).  The j-th token held (arrival order,
 * as token_row) sits at position pos0 + j; the query belongs to the newest
 * token, position pos0 + n - 1.  Every key and the query are rotated
 * (rope_rotate) and then attended exactly as orc_attend does, in fp64.
 * Returns 0, or -1 on allocation failure.
 */
int orc_attend_rope(const orc_head *s, const uint16_t *q, double tau, double base,
                    int64_t pos0, double *out) {
  const int d = s->d;
  const int64_t n = s->n_sink_used + s->n_quant + s->n_resid;
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (n == 0) return 0;
  double *sc = (double *)malloc(sizeof(double) * (size_t)n);
  double *qd = (double *)malloc(sizeof(double) * (size_t)d);
  double *row = (double *)malloc(sizeof(double) * (size_t)d);
  if (!sc || !qd || !row) { free(sc); free(qd); free(row); return -1; }
  for (int c = 0; c < d; ++c) qd[c] = (double)orc_half_to_float(q[c]);
  rope_rotate(qd, d, base, (double)(pos0 + n - 1));
  for (int64_t j = 0; j < n; ++j) {
    token_row(s, j, 1, row);
    rope_rotate(row, d, base, (double)(pos0 + j));
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += qd[c] * row[c];
    sc[j] = tau * acc;
  }
  double m = sc[0];
  for (int64_t j = 1; j < n; ++j) if (sc[j] > m) m = sc[j];
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) { sc[j] = exp(sc[j] - m); l += sc[j]; }
  for (int64_t j = 0; j < n; ++j) {
    token_row(s, j, 0, row);
    for (int c = 0; c < d; ++c) out[c] += sc[j] * row[c];
  }
  for (int c = 0; c < d; ++c) out[c] /= l;
  free(sc);
  free(qd);
  free(row);
  return 0;
}

/*
 * Bit packing of code rows ([n_rows][d], one code per byte) into
 * [n_rows][d*bits/8] bytes: along the channels of a token, little-endian
 * within each byte, channel c at bits (c mod (8/bits))*bits of byte
 * c / (8/bits).  The pages fix no layout; this one is the library's.
 */
void orc_pack(const uint8_t *u, int64_t n_rows, int d, int bits, uint8_t *out) {
  const int per = 8 / bits;
  const int rb = d / per;
  memset(out, 0, (size_t)(n_rows * rb));
  for (int64_t t = 0; t < n_rows; ++t)
    for (int c = 0; c < d; ++c)
      out[t * rb + c / per] |= (uint8_t)(u[t * d + c] << ((c % per) * bits));
}

/* Mode flags (one per group, token-major) as bits: flag i is bit i % 32 of
 * word i / 32.  `out` holds ceil(n / 32) words. */
void orc_pack_modes(const uint8_t *sym, int64_t n, uint32_t *out) {
  memset(out, 0, sizeof(uint32_t) * (size_t)((n + 31) / 32));
  for (int64_t i = 0; i < n; ++i)
    if (sym[i]) out[i / 32] |= (uint32_t)1 << (i % 32);
}
