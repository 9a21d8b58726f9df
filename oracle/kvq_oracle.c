/*
 * kvq_oracle.c — plain, slow, single-threaded CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY: the product library never links, loads or calls
 * this file.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg execute it.  It shares no source, header, table or helper with the CUDA
 * path.
 *
 * Sources (web pages on KV-cache quantization; cited by title and section):
 *  [KIVI]   "KIVI: KV cache axes" article — §1 attention s = qK^T/sqrt(D),
 *           p = softmax(s), o = pV and the output-error decomposition;
 *           §2 the per-group contract m = min, step = (max-m)/(2^b-1),
 *           c = RNE((x-m)/step), x^ = m + step*c, constant group special case;
 *           §3 grouping axes (Key per-channel over consecutive tokens, Value
 *           per-token over consecutive channels) and LSB-first 2-bit packing;
 *           §4/§5 residual buffer and flush; §6 one global softmax over the
 *           quantized and the full-precision parts; §7 byte accounting.
 *  [MixKVQ] "MixKVQ: Query-Aware Mixed-Precision KV Cache Quantization for
 *           Long-Context Reasoning" — "KV cache quantization principle" (z =
 *           min, s = (max-min)/(2^B-1), round), appendix error bound |x-x^| <=
 *           s/2, salience A_d = I_d * S_d, importance I_d = mean |Q_{i,d}|,
 *           sensitivity S_d, the three tiers BF16/UINT4/UINT2, GQA
 *           aggregation ("system-level implementation details"), Algorithm 1.
 *  [PN-Mix] "PN-Mix" reproduction notes — "core formulas" Eq. 2 (codes
 *           clipped to [0, 2^b-1]; constant group stored with zero scale and
 *           the original offset); App. G (codes packed along tokens).
 *
 * Readings where the pages are silent or disagree (each listed in the design
 * notes): codes use round-half-to-even; step is an IEEE fp32 division; a
 * constant group stores step 0 with origin = the value (reconstruction equals
 * the KIVI article's step-1 variant); origin is stored as bf16 (lossless, it
 * is an input value) and step as fp32; among equal minima -0.0 is preferred,
 * among equal maxima +0.0.
 */
#include "kvq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

float orc_bf16_to_f32(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t orc_f32_to_bf16_exact(float value) {
  uint32_t u;
  memcpy(&u, &value, sizeof u);
  return (uint16_t)(u >> 16);
}

/* Total order on finite floats used for min/max: -0.0 sorts below +0.0. */
static int orc_less(float a, float b) {
  if (a < b) return 1;
  if (a == b && signbit(a) && !signbit(b)) return 1;
  return 0;
}

/*
 * [KIVI] §2 and [MixKVQ] "KV cache quantization principle":
 *   m = min x,  step = (max x - m) / (2^b - 1),  c = RNE((x - m)/step),
 * with the codes clipped to [0, 2^b - 1] ([PN-Mix] Eq. 2).  Rejects
 * non-finite inputs and a step that is not a positive finite number
 * ([KIVI] §3 reference's validation).  Constant group: step stored as 0,
 * all codes 0, origin = the value ([PN-Mix] "core formulas").
 */
int orc_quantize_group(const float* x, long n, long stride, int bits,
                       uint8_t* codes, float* origin, float* step) {
  if (n <= 0 || stride <= 0 || bits < 1 || bits > 8) return ORC_ERR_ARG;
  for (long i = 0; i < n; ++i)
    if (!isfinite(x[i * stride])) return ORC_ERR_NONFINITE;

  float lo = x[0];
  float hi = x[0];
  for (long i = 1; i < n; ++i) {
    float v = x[i * stride];
    if (orc_less(v, lo)) lo = v;
    if (orc_less(hi, v)) hi = v;
  }

  *origin = lo;
  if (hi == lo) {
    *step = 0.0f;
    for (long i = 0; i < n; ++i) codes[i] = 0;
    return ORC_OK;
  }

  const int top = (1 << bits) - 1;
  volatile float range = hi - lo;             /* one fp32 rounding */
  volatile float delta = range / (float)top;  /* IEEE fp32 division */
  if (!(delta > 0.0f) || !isfinite(delta)) return ORC_ERR_RANGE;
  *step = delta;

  for (long i = 0; i < n; ++i) {
    volatile float diff = x[i * stride] - lo;  /* fp32 */
    volatile float y = diff / delta;           /* fp32, IEEE division */
    float r = nearbyintf(y);                   /* ties to even */
    if (r < 0.0f) r = 0.0f;
    if (r > (float)top) r = (float)top;
    codes[i] = (uint8_t)r;
  }
  return ORC_OK;
}

uint16_t orc_f32_to_bf16_rn(float value) {
  uint32_t u;
  memcpy(&u, &value, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);   /* ties to the even bf16 pattern */
  return (uint16_t)(u >> 16);
}

static float orc_bf16_round(float x) { return orc_bf16_to_f32(orc_f32_to_bf16_rn(x)); }

/* [KIVI] §7: the fixed pack path keeps the minimum in a tensor of the
 * input's dtype and computes the step from it in that dtype; here every
 * operation is an fp32 operation whose result is rounded to bf16. */
int orc_quantize_group_bf16(const float* x, long n, long stride, int bits,
                            uint8_t* codes, uint16_t* origin, uint16_t* step) {
  if (n <= 0 || stride <= 0 || bits < 1 || bits > 8) return ORC_ERR_ARG;
  for (long i = 0; i < n; ++i)
    if (!isfinite(x[i * stride])) return ORC_ERR_NONFINITE;

  float lo = x[0];
  float hi = x[0];
  for (long i = 1; i < n; ++i) {
    float v = x[i * stride];
    if (orc_less(v, lo)) lo = v;
    if (orc_less(hi, v)) hi = v;
  }

  *origin = orc_f32_to_bf16_exact(lo);
  if (hi == lo) {
    *step = 0;
    for (long i = 0; i < n; ++i) codes[i] = 0;
    return ORC_OK;
  }

  const int top = (1 << bits) - 1;
  volatile float range = orc_bf16_round(hi - lo);
  volatile float delta = orc_bf16_round(range / (float)top);
  if (!(delta > 0.0f) || !isfinite(delta)) return ORC_ERR_RANGE;
  *step = orc_f32_to_bf16_exact(delta);

  for (long i = 0; i < n; ++i) {
    volatile float diff = orc_bf16_round(x[i * stride] - lo);
    volatile float y = orc_bf16_round(diff / delta);
    float r = nearbyintf(y);                   /* ties to even */
    if (r < 0.0f) r = 0.0f;
    if (r > (float)top) r = (float)top;
    codes[i] = (uint8_t)r;
  }
  return ORC_OK;
}

/* [PN-Mix] Eq. 7 (quarter-point 1-bit groups). */
int orc_quantize_group_1bit_mid(const float* x, long n, long stride, uint8_t* codes,
                                float* offset, float* scale) {
  if (n <= 0 || stride <= 0) return ORC_ERR_ARG;
  for (long i = 0; i < n; ++i)
    if (!isfinite(x[i * stride])) return ORC_ERR_NONFINITE;
  float lo = x[0], hi = x[0];
  for (long i = 1; i < n; ++i) {
    float v = x[i * stride];
    if (orc_less(v, lo)) lo = v;
    if (orc_less(hi, v)) hi = v;
  }
  if (hi == lo) {
    *offset = lo;
    *scale = 0.0f;
    for (long i = 0; i < n; ++i) codes[i] = 0;
    return ORC_OK;
  }
  volatile float range = hi - lo;
  volatile float s = range / 2.0f;
  volatile float three_lo = 3.0f * lo;
  volatile float num = three_lo + hi;
  volatile float z = num / 4.0f;
  if (!(s > 0.0f) || !isfinite(s) || !isfinite(z)) return ORC_ERR_RANGE;
  *offset = z;
  *scale = s;
  for (long i = 0; i < n; ++i) {
    volatile float diff = x[i * stride] - z;
    volatile float y = diff / s;
    float r = nearbyintf(y);
    if (r < 0.0f) r = 0.0f;
    if (r > 1.0f) r = 1.0f;
    codes[i] = (uint8_t)r;
  }
  return ORC_OK;
}

/* [PN-Mix] Eq. 6 (pair-norm scores, fp32 in a fixed order). */
int orc_pair_scores(const uint16_t* q, int Hg, int Lq, const uint16_t* k, int Lk, int D,
                    int layout, float* sigma) {
  if (!q || !k || !sigma || Hg <= 0 || Lq <= 0 || Lk <= 0 || D <= 0 || D % 2 ||
      (layout != 0 && layout != 1))
    return ORC_ERR_ARG;
  const int P = D / 2;
  for (int i = 0; i < P; ++i) {
    const int ca = layout == 0 ? 2 * i : i;
    const int cb = layout == 0 ? 2 * i + 1 : i + P;
    volatile float qsum = 0.0f;
    for (int h = 0; h < Hg; ++h) {
      volatile float acc = 0.0f;
      for (int t = 0; t < Lq; ++t) {
        const float a = orc_bf16_to_f32(q[((long)h * Lq + t) * D + ca]);
        const float b = orc_bf16_to_f32(q[((long)h * Lq + t) * D + cb]);
        if (!isfinite(a) || !isfinite(b)) return ORC_ERR_NONFINITE;
        volatile float aa = a * a, bb = b * b;
        volatile float ss = aa + bb;
        acc = acc + sqrtf(ss);
      }
      volatile float mean = acc / (float)Lq;
      qsum = qsum + mean;
    }
    volatile float qbar = qsum / (float)Hg;
    volatile float kacc = 0.0f;
    for (int t = 0; t < Lk; ++t) {
      const float a = orc_bf16_to_f32(k[(long)t * D + ca]);
      const float b = orc_bf16_to_f32(k[(long)t * D + cb]);
      if (!isfinite(a) || !isfinite(b)) return ORC_ERR_NONFINITE;
      volatile float aa = a * a, bb = b * b;
      volatile float ss = aa + bb;
      kacc = kacc + sqrtf(ss);
    }
    volatile float kbar = kacc / (float)Lk;
    sigma[i] = qbar * kbar;
  }
  return ORC_OK;
}

/* [KIVI] §3 teaching packer: code i goes to byte i/(8/b) at bit offset
 * b*(i mod 8/b), low bits first; the logical length is carried separately. */
void orc_pack_lsb(const uint8_t* codes, long n, int bits, uint8_t* out) {
  const int per = 8 / bits;
  const long nbytes = (n + per - 1) / per;
  memset(out, 0, (size_t)nbytes);
  for (long i = 0; i < n; ++i)
    out[i / per] |= (uint8_t)(codes[i] << (bits * (int)(i % per)));
}

void orc_unpack_lsb(const uint8_t* packed, long n, int bits, uint8_t* codes) {
  const int per = 8 / bits;
  const uint8_t mask = (uint8_t)((1u << bits) - 1u);
  for (long i = 0; i < n; ++i)
    codes[i] = (uint8_t)((packed[i / per] >> (bits * (int)(i % per))) & mask);
}

/*
 * [KIVI] §3 grouping table, Key row: one parameter set per channel d over G
 * consecutive tokens K[t:t+G, d].  [PN-Mix] App. G: Key codes are packed
 * along tokens.  [MixKVQ] workflow: Key cache is quantized per channel.
 */
int orc_quantize_k_unit(const uint16_t* k, long T, int D, int G, int bits,
                        uint8_t* codes, uint16_t* kmin, float* kscale) {
  if (T < 0 || D <= 0 || G <= 0 || T % G != 0 || bits < 1 || bits > 8)
    return ORC_ERR_ARG;
  const long groups = T / G;
  const long bytes_per_channel = ((long)G * bits + 7) / 8;  /* padded */
  float* x = (float*)malloc(sizeof(float) * (size_t)G);
  uint8_t* c = (uint8_t*)malloc((size_t)G);
  int status = ORC_OK;
  for (long g = 0; g < groups && status == ORC_OK; ++g) {
    for (int d = 0; d < D; ++d) {
      for (int i = 0; i < G; ++i) x[i] = orc_bf16_to_f32(k[(g * G + i) * D + d]);
      float m, s;
      status = orc_quantize_group(x, G, 1, bits, c, &m, &s);
      if (status != ORC_OK) break;
      orc_pack_lsb(c, G, bits, codes + (g * D + d) * bytes_per_channel);
      kmin[g * D + d] = orc_f32_to_bf16_exact(m);
      kscale[g * D + d] = s;
    }
  }
  free(x);
  free(c);
  return status;
}

/* [KIVI] §3 grouping table, Value row: one parameter set per token t over G
 * consecutive channels V[t, d:d+G].  [MixKVQ] workflow: Value per token. */
int orc_quantize_v_unit(const uint16_t* v, long T, int D, int G, int bits,
                        uint8_t* codes, uint16_t* vmin, float* vscale) {
  if (T < 0 || D <= 0 || G <= 0 || D % G != 0 || (D * bits) % 8 != 0)
    return ORC_ERR_ARG;
  const int groups = D / G;
  const long row_bytes = (long)D * bits / 8;
  float* x = (float*)malloc(sizeof(float) * (size_t)G);
  uint8_t* c = (uint8_t*)malloc((size_t)D);
  int status = ORC_OK;
  for (long t = 0; t < T && status == ORC_OK; ++t) {
    for (int j = 0; j < groups; ++j) {
      for (int i = 0; i < G; ++i) x[i] = orc_bf16_to_f32(v[t * D + j * G + i]);
      float m, s;
      status = orc_quantize_group(x, G, 1, bits, c + j * G, &m, &s);
      if (status != ORC_OK) break;
      vmin[t * groups + j] = orc_f32_to_bf16_exact(m);
      vscale[t * groups + j] = s;
    }
    /* the token's D codes, packed LSB first along channels */
    if (status == ORC_OK) orc_pack_lsb(c, D, bits, codes + t * row_bytes);
  }
  free(x);
  free(c);
  return status;
}

/* [KIVI] §2: x^ = m + step * c, evaluated in fp64. */
void orc_dequant_k_unit(const uint8_t* codes, const uint16_t* kmin,
                        const float* kscale, long T, int D, int G, int bits,
                        double* out) {
  const long groups = T / G;
  const long bytes_per_channel = ((long)G * bits + 7) / 8;
  uint8_t* c = (uint8_t*)malloc((size_t)G);
  for (long g = 0; g < groups; ++g) {
    for (int d = 0; d < D; ++d) {
      orc_unpack_lsb(codes + (g * D + d) * bytes_per_channel, G, bits, c);
      const double m = (double)orc_bf16_to_f32(kmin[g * D + d]);
      const double s = (double)kscale[g * D + d];
      for (int i = 0; i < G; ++i) out[(g * G + i) * D + d] = m + s * (double)c[i];
    }
  }
  free(c);
}

void orc_dequant_v_unit(const uint8_t* codes, const uint16_t* vmin,
                        const float* vscale, long T, int D, int G, int bits,
                        double* out) {
  const int groups = D / G;
  const long row_bytes = (long)D * bits / 8;
  uint8_t* c = (uint8_t*)malloc((size_t)D);
  for (long t = 0; t < T; ++t) {
    orc_unpack_lsb(codes + t * row_bytes, D, bits, c);
    for (int d = 0; d < D; ++d) {
      const int j = d / G;
      const double m = (double)orc_bf16_to_f32(vmin[t * groups + j]);
      const double s = (double)vscale[t * groups + j];
      out[t * D + d] = m + s * (double)c[d];
    }
  }
  free(c);
}

/*
 * [KIVI] §1: s = q K^T / sqrt(D), p = softmax(s), o = p V, and §6: a single
 * softmax over all visible rows (quantized history and full-precision
 * residual together).  Plain fp64, max-shifted exponentials.
 */
int orc_attention(const double* q, const double* k, const double* v, long n,
                  int D, double* o, double* p_out) {
  if (n <= 0 || D <= 0) return ORC_ERR_ARG;
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  double peak = -INFINITY;
  for (long t = 0; t < n; ++t) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * k[t * D + d];
    s[t] = dot * inv_sqrt_d;
    if (!isfinite(s[t])) {
      free(s);
      return ORC_ERR_NONFINITE;
    }
    if (s[t] > peak) peak = s[t];
  }
  double total = 0.0;
  for (long t = 0; t < n; ++t) {
    s[t] = exp(s[t] - peak);
    total += s[t];
  }
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (long t = 0; t < n; ++t) {
    const double p = s[t] / total;
    if (p_out) p_out[t] = p;
    for (int d = 0; d < D; ++d) o[d] += p * v[t * D + d];
  }
  free(s);
  return ORC_OK;
}

/*
 * [MixKVQ] importance I_d = (1/L_q) sum_i |Q_{i,d}|, aggregated over the
 * query heads that share one KV head ("system-level implementation
 * details"): a mean over n_rep heads x L_q tokens, summed in fp32 in the
 * order token ascending, then head ascending, then one IEEE division.
 */
int orc_importance(const uint16_t* q_group, int n_rep, int Lq, int D,
                   float* I) {
  if (n_rep <= 0 || Lq <= 0 || D <= 0) return ORC_ERR_ARG;
  for (int d = 0; d < D; ++d) {
    volatile float acc = 0.0f;
    for (int i = 0; i < Lq; ++i) {
      for (int h = 0; h < n_rep; ++h) {
        const float x = orc_bf16_to_f32(q_group[((long)h * Lq + i) * D + d]);
        if (!isfinite(x)) return ORC_ERR_NONFINITE;
        acc = acc + fabsf(x);
      }
    }
    volatile float count = (float)(n_rep * Lq);
    I[d] = acc / count;
  }
  return ORC_OK;
}

/* [MixKVQ] sensitivity S_d = (max k_d - min k_d) / (2^B - 1) over the
 * group's tokens, from the raw range in fp32. */
int orc_sensitivity(const uint16_t* k, int G, int D, int bits, float* S) {
  if (G <= 0 || D <= 0 || bits < 1 || bits > 8) return ORC_ERR_ARG;
  const float top = (float)((1 << bits) - 1);
  for (int d = 0; d < D; ++d) {
    float lo = orc_bf16_to_f32(k[d]);
    float hi = lo;
    for (int i = 0; i < G; ++i) {
      const float x = orc_bf16_to_f32(k[(long)i * D + d]);
      if (!isfinite(x)) return ORC_ERR_NONFINITE;
      if (x < lo) lo = x;
      if (x > hi) hi = x;
    }
    volatile float range = hi - lo;
    volatile float s = range / top;
    if (!isfinite(s)) return ORC_ERR_RANGE;
    S[d] = s;
  }
  return ORC_OK;
}

/* [MixKVQ] salience A_d = I_d * S_d (one fp32 product). */
void orc_salience(const float* I, const float* S, int D, float* A) {
  for (int d = 0; d < D; ++d) {
    volatile float a = I[d] * S[d];
    A[d] = a;
  }
}

/*
 * Rank form of the three tiers: the n_bf16 channels of largest A_d keep
 * BF16, the next n_uint4 go to UINT4, the rest to UINT2 ([MixKVQ] three-tier
 * strategy; counts stand for its thresholds).  Ties go to the lower channel
 * index.  Plain selection: repeatedly pick the best unassigned channel.
 */
int orc_tiers_rank(const float* A, int D, int n_bf16, int n_uint4,
                   uint8_t* tiers) {
  if (D <= 0 || n_bf16 < 0 || n_uint4 < 0 || n_bf16 + n_uint4 > D)
    return ORC_ERR_ARG;
  for (int d = 0; d < D; ++d)
    if (!isfinite(A[d])) return ORC_ERR_NONFINITE;
  uint8_t* taken = (uint8_t*)calloc((size_t)D, 1);
  for (int rank = 0; rank < D; ++rank) {
    int best = -1;
    for (int d = 0; d < D; ++d) {
      if (taken[d]) continue;
      if (best < 0 || A[d] > A[best]) best = d;  /* strict: lower d wins ties */
    }
    taken[best] = 1;
    tiers[best] = rank < n_bf16 ? ORC_TIER_BF16
                  : rank < n_bf16 + n_uint4 ? ORC_TIER_UINT4
                                            : ORC_TIER_UINT2;
  }
  free(taken);
  return ORC_OK;
}

/* [MixKVQ] threshold form: A > tau_BF16 -> BF16; tau_UINT4 < A <= tau_BF16
 * -> UINT4; A <= tau_UINT4 -> UINT2. */
int orc_tiers_threshold(const float* A, int D, float tau_bf16, float tau_uint4,
                        uint8_t* tiers) {
  if (D <= 0) return ORC_ERR_ARG;
  for (int d = 0; d < D; ++d) {
    if (!isfinite(A[d])) return ORC_ERR_NONFINITE;
    if (A[d] > tau_bf16)
      tiers[d] = ORC_TIER_BF16;
    else if (A[d] > tau_uint4)
      tiers[d] = ORC_TIER_UINT4;
    else
      tiers[d] = ORC_TIER_UINT2;
  }
  return ORC_OK;
}

/*
 * [MixKVQ] threshold tiers in a key record of fixed capacity (at most
 * cap_bf16 BF16 and cap_uint4 UINT4 channels a group).  Channels are taken
 * from the largest A_d down (ties: lower index first); each one is BF16 if
 * A_d > tau_bf16 and fewer than cap_bf16 channels are BF16 so far, else
 * UINT4 if A_d > tau_uint4 and fewer than cap_uint4 are UINT4, else UINT2.
 * With both caps = D this is the plain threshold rule; with both thresholds
 * at -infinity it is the rank rule with counts cap_bf16, cap_uint4.
 */
int orc_tiers_capped(const float* A, int D, float tau_bf16, float tau_uint4,
                     int cap_bf16, int cap_uint4, uint8_t* tiers) {
  if (D <= 0 || cap_bf16 < 0 || cap_uint4 < 0) return ORC_ERR_ARG;
  for (int d = 0; d < D; ++d)
    if (!isfinite(A[d])) return ORC_ERR_NONFINITE;
  uint8_t* taken = (uint8_t*)calloc((size_t)D, 1);
  int nb = 0, n4 = 0;
  for (int k = 0; k < D; ++k) {
    int best = -1;
    for (int d = 0; d < D; ++d) {
      if (taken[d]) continue;
      if (best < 0 || A[d] > A[best]) best = d;  /* strict: lower d wins ties */
    }
    taken[best] = 1;
    if (A[best] > tau_bf16 && nb < cap_bf16) {
      tiers[best] = ORC_TIER_BF16;
      ++nb;
    } else if (A[best] > tau_uint4 && n4 < cap_uint4) {
      tiers[best] = ORC_TIER_UINT4;
      ++n4;
    } else {
      tiers[best] = ORC_TIER_UINT2;
    }
  }
  free(taken);
  return ORC_OK;
}

/*
 * [MixKVQ] online saliency estimation: the cache keeps a running fp32 sum
 * of query magnitudes per key channel, and every decode step adds the
 * current query token's |q| of each head of the KV group, heads in order
 * (q_step: n_rep rows of D bf16).  Summed over the steps of a window this is
 * the importance sum of orc_importance in the same order (token, then head).
 */
int orc_observe_query(float* acc, const uint16_t* q_step, int n_rep, int D) {
  if (n_rep <= 0 || D <= 0) return ORC_ERR_ARG;
  for (int h = 0; h < n_rep; ++h)
    for (int d = 0; d < D; ++d)
      if (!isfinite(orc_bf16_to_f32(q_step[(long)h * D + d]))) return ORC_ERR_NONFINITE;
  for (int d = 0; d < D; ++d) {
    volatile float a = acc[d];
    for (int h = 0; h < n_rep; ++h) a = a + fabsf(orc_bf16_to_f32(q_step[(long)h * D + d]));
    acc[d] = a;
  }
  return ORC_OK;
}

/* I_d of the window the accumulator covers: acc_d / (n_rep * steps). */
int orc_importance_from_sum(const float* acc, int n_rep, int steps, int D, float* I) {
  if (n_rep <= 0 || steps <= 0 || D <= 0) return ORC_ERR_ARG;
  for (int d = 0; d < D; ++d) {
    volatile float count = (float)(n_rep * steps);
    I[d] = acc[d] / count;
  }
  return ORC_OK;
}

/*
 * [MixKVQ] Algorithm 1 KeyQuant: OutlierReserve splits the key channels by
 * tier; BF16 channels are kept as they are ("sparse outlier store"), UINT4
 * and UINT2 channels are group-quantized along tokens at 4 and 2 bits.
 * Storage order: BF16 channels, then UINT4, then UINT2, each ascending.
 */
int orc_quantize_k_mixed_group(const uint16_t* k, int G, int D,
                               const uint8_t* tiers, uint8_t* perm,
                               uint16_t* raw, uint8_t* c4, uint16_t* m4,
                               float* s4, uint8_t* c2, uint16_t* m2,
                               float* s2) {
  if (G <= 0 || D <= 0 || G % 4 != 0) return ORC_ERR_ARG;
  float* x = (float*)malloc(sizeof(float) * (size_t)G);
  uint8_t* c = (uint8_t*)malloc((size_t)G);
  int slot = 0, n_b = 0, n_4 = 0, n_2 = 0;
  int status = ORC_OK;
  for (int tier = ORC_TIER_BF16; tier <= ORC_TIER_UINT2 && status == ORC_OK;
       ++tier) {
    for (int d = 0; d < D; ++d) {
      if (tiers[d] != tier) continue;
      perm[slot++] = (uint8_t)d;
      for (int i = 0; i < G; ++i) x[i] = orc_bf16_to_f32(k[(long)i * D + d]);
      if (tier == ORC_TIER_BF16) {
        for (int i = 0; i < G; ++i) {
          if (!isfinite(x[i])) status = ORC_ERR_NONFINITE;
          raw[(long)n_b * G + i] = k[(long)i * D + d];
        }
        ++n_b;
      } else {
        const int bits = tier == ORC_TIER_UINT4 ? 4 : 2;
        float m, s;
        status = orc_quantize_group(x, G, 1, bits, c, &m, &s);
        if (status != ORC_OK) break;
        if (bits == 4) {
          orc_pack_lsb(c, G, 4, c4 + (long)n_4 * (G / 2));
          m4[n_4] = orc_f32_to_bf16_exact(m);
          s4[n_4] = s;
          ++n_4;
        } else {
          orc_pack_lsb(c, G, 2, c2 + (long)n_2 * (G / 4));
          m2[n_2] = orc_f32_to_bf16_exact(m);
          s2[n_2] = s;
          ++n_2;
        }
      }
    }
  }
  free(x);
  free(c);
  if (status == ORC_OK && slot != D) status = ORC_ERR_ARG;
  return status;
}

void orc_dequant_k_mixed_group(int G, int D, const uint8_t* perm, int n_bf16,
                               int n_uint4, const uint16_t* raw,
                               const uint8_t* c4, const uint16_t* m4,
                               const float* s4, const uint8_t* c2,
                               const uint16_t* m2, const float* s2,
                               double* out) {
  uint8_t* c = (uint8_t*)malloc((size_t)G);
  for (int slot = 0; slot < D; ++slot) {
    const int d = perm[slot];
    if (slot < n_bf16) {
      for (int i = 0; i < G; ++i)
        out[(long)i * D + d] = (double)orc_bf16_to_f32(raw[(long)slot * G + i]);
    } else if (slot < n_bf16 + n_uint4) {
      const int j = slot - n_bf16;
      orc_unpack_lsb(c4 + (long)j * (G / 2), G, 4, c);
      const double m = (double)orc_bf16_to_f32(m4[j]);
      const double s = (double)s4[j];
      for (int i = 0; i < G; ++i) out[(long)i * D + d] = m + s * (double)c[i];
    } else {
      const int j = slot - n_bf16 - n_uint4;
      orc_unpack_lsb(c2 + (long)j * (G / 4), G, 2, c);
      const double m = (double)orc_bf16_to_f32(m2[j]);
      const double s = (double)s2[j];
      for (int i = 0; i < G; ++i) out[(long)i * D + d] = m + s * (double)c[i];
    }
  }
  free(c);
}

/*
 * [KIVI] §7 per-(layer, KV head, request) persistent bytes: the quantized
 * elements of both caches, (2T - rK - rV) per channel, each costing b/8
 * bytes of code plus one origin and one step per G elements; the float
 * residual elements cost f bytes each.  Generalized to separate Key/Value
 * bit widths and group sizes and to separate origin/step widths; with
 * k_bits = v_bits = b, Gk = Gv = G and origin = step = e it is the page's
 * formula M = D[(2T - rK - rV)(b/8 + 2e/G) + (rK + rV) f].
 */
double orc_cache_bytes(long T, long rK, long rV, int D, int k_bits, int v_bits,
                       int Gk, int Gv, int origin_bytes, int step_bytes,
                       int float_bytes) {
  const double meta = (double)(origin_bytes + step_bytes);
  const double per_k = (double)k_bits / 8.0 + meta / (double)Gk;
  const double per_v = (double)v_bits / 8.0 + meta / (double)Gv;
  return (double)D * ((double)(T - rK) * per_k + (double)(T - rV) * per_v +
                      (double)(rK + rV) * (double)float_bytes);
}
