/*
 * kvq_oracle.h — plain, single-threaded CPU oracle for low-bit KV-cache
 * quantization (KIVI-style asymmetric min–max, MixKVQ query-aware key tiers)
 * and decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this code; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no source with the CUDA path.
 *
 * Precision contract: quantization arithmetic in IEEE fp32 (one rounding per
 * operation, division by true division, codes rounded to nearest-even),
 * compiled with -ffp-contract=off; dequantization and attention in fp64.
 *
 * bf16 values travel as their raw 16-bit patterns (uint16_t).
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORC_OK = 0,
  ORC_ERR_ARG = 1,        /* malformed arguments                           */
  ORC_ERR_NONFINITE = 2,  /* a non-finite input value                      */
  ORC_ERR_RANGE = 3       /* step not a positive finite fp32 number        */
};

enum { ORC_TIER_BF16 = 0, ORC_TIER_UINT4 = 1, ORC_TIER_UINT2 = 2 };

/* Exact bf16 <-> fp32 conversions (fp32 -> bf16 only for values that are
 * already bf16-representable; the oracle never needs a rounding one). */
float orc_bf16_to_f32(uint16_t bits);
uint16_t orc_f32_to_bf16_exact(float value);

/* One quantization group of n values x[i*stride], b-bit codes. */
int orc_quantize_group(const float* x, long n, long stride, int bits,
                       uint8_t* codes, float* origin, float* step);

/* Nearest-even rounding of a finite fp32 value to bf16 (the bf16
 * arithmetic below computes each operation in fp32 and rounds the result to
 * bf16, as arithmetic on a bf16 tensor dtype does). */
uint16_t orc_f32_to_bf16_rn(float value);

/* [KIVI] §7 metadata in the input dtype: one group of n bf16-valued x with
 * its origin (the minimum) and step kept as bf16 and computed in bf16:
 *   R = bf16(M - m), step = bf16(R / (2^b - 1)),
 *   c = clip(RNE(bf16(bf16(x - m) / step)), 0, 2^b - 1);
 * a constant group (M == m) has step 0 and codes 0.  Errors as for
 * orc_quantize_group (RANGE when the bf16 step is 0 or not finite). */
int orc_quantize_group_bf16(const float* x, long n, long stride, int bits,
                            uint8_t* codes, uint16_t* origin, uint16_t* step);

/* [PN-Mix] Eq. 7: a 1-bit group whose two reconstructions sit at the
 * quarter points: s = fl32(fl32(M - m) / 2), z = fl32(fl32(fl32(3 m) + M) / 4),
 * c = clip(RNE(fl32(fl32(x - z) / s)), 0, 1), x^ = z + s c; a constant
 * group (M == m) has s = 0 and z = m (zero scale, original offset). */
int orc_quantize_group_1bit_mid(const float* x, long n, long stride, uint8_t* codes,
                                float* offset, float* scale);

/* [PN-Mix] Eq. 6 pair scores of one KV head: q bf16 [Hg][Lq][D] (the query
 * heads of its GQA group, in order), k bf16 [Lk][D]; pair i is channels
 * (2i, 2i+1) for layout 0 (adjacent) or (i, i + D/2) for layout 1 (split
 * halves).  In fp32: a token's pair norm is the correctly rounded
 * sqrt(a*a + b*b); per head the norms are summed in token order and divided
 * by Lq, the head means summed in head order and divided by Hg, the key
 * norms summed in token order and divided by Lk; sigma = the product. */
int orc_pair_scores(const uint16_t* q, int Hg, int Lq, const uint16_t* k, int Lk, int D,
                    int layout, float* sigma);

/* LSB-first packing of b-bit codes (b in {1,2,4,8}). */
void orc_pack_lsb(const uint8_t* codes, long n, int bits, uint8_t* out);
void orc_unpack_lsb(const uint8_t* packed, long n, int bits, uint8_t* codes);

/* Key history of one (batch row, KV head): k is bf16 [T][D] (token-major),
 * T a multiple of the token group G.  Outputs in canonical layout:
 *   codes  [T/G][D][ceil(G*bits/8)]  (each channel's G codes packed along
 *          tokens, LSB first, padded to a whole byte)
 *   kmin   [T/G][D] bf16,  kscale [T/G][D] fp32                           */
int orc_quantize_k_unit(const uint16_t* k, long T, int D, int G, int bits,
                        uint8_t* codes, uint16_t* kmin, float* kscale);

/* Value history of one unit: v bf16 [T][D]; groups of G consecutive channels
 * of one token.  codes [T][D*bits/8] (a token's D codes packed LSB first
 * along channels), vmin [T][D/G] bf16, vscale [T][D/G] fp32.              */
int orc_quantize_v_unit(const uint16_t* v, long T, int D, int G, int bits,
                        uint8_t* codes, uint16_t* vmin, float* vscale);

/* Reconstruction m + step*c in fp64, written token-major [T][D]. */
void orc_dequant_k_unit(const uint8_t* codes, const uint16_t* kmin,
                        const float* kscale, long T, int D, int G, int bits,
                        double* out);
void orc_dequant_v_unit(const uint8_t* codes, const uint16_t* vmin,
                        const float* vscale, long T, int D, int G, int bits,
                        double* out);

/* Decode attention for one query vector over n rows, all in fp64:
 * s = q K^T / sqrt(D), p = softmax(s), o = p V.  p_out may be NULL. */
int orc_attention(const double* q, const double* k, const double* v, long n,
                  int D, double* o, double* p_out);

/* MixKVQ statistics for one (batch row, KV head).
 * importance: q_group bf16 [n_rep][Lq][D] (the query heads sharing the KV
 * head); I_d = sum over (token i ascending, head ascending) of |Q|, divided
 * by n_rep*Lq.  sensitivity: k bf16 [G][D], S_d = (max-min)/(2^bits-1). */
int orc_importance(const uint16_t* q_group, int n_rep, int Lq, int D, float* I);
int orc_sensitivity(const uint16_t* k, int G, int D, int bits, float* S);
void orc_salience(const float* I, const float* S, int D, float* A);
int orc_tiers_rank(const float* A, int D, int n_bf16, int n_uint4,
                   uint8_t* tiers);
int orc_tiers_threshold(const float* A, int D, float tau_bf16, float tau_uint4,
                        uint8_t* tiers);
int orc_tiers_capped(const float* A, int D, float tau_bf16, float tau_uint4,
                     int cap_bf16, int cap_uint4, uint8_t* tiers);
int orc_observe_query(float* acc, const uint16_t* q_step, int n_rep, int D);
int orc_importance_from_sum(const float* acc, int n_rep, int steps, int D, float* I);

/* One mixed-precision key group: k bf16 [G][D], tiers[D] given.
 *   perm     [D]                   channels: BF16 tier, then UINT4, then
 *                                  UINT2, each in ascending channel order
 *   raw      [n_bf16][G] bf16      BF16-tier channels, token order
 *   c4       [n_uint4][G/2]        4-bit codes packed along tokens
 *   m4, s4   [n_uint4]             bf16 origin, fp32 step
 *   c2       [n_uint2][G/4]        2-bit codes packed along tokens
 *   m2, s2   [n_uint2]                                                    */
int orc_quantize_k_mixed_group(const uint16_t* k, int G, int D,
                               const uint8_t* tiers, uint8_t* perm,
                               uint16_t* raw, uint8_t* c4, uint16_t* m4,
                               float* s4, uint8_t* c2, uint16_t* m2, float* s2);
void orc_dequant_k_mixed_group(int G, int D, const uint8_t* perm, int n_bf16,
                               int n_uint4, const uint16_t* raw,
                               const uint8_t* c4, const uint16_t* m4,
                               const float* s4, const uint8_t* c2,
                               const uint16_t* m2, const float* s2,
                               double* out);

/* Persistent bytes of one (batch row, KV head) holding T visible tokens, of
 * which the last rK keys and rV values are kept in floating point (f bytes
 * each) and the rest are b-bit codes plus one origin and one step per group
 * (Gk tokens for keys, Gv channels for values). */
double orc_cache_bytes(long T, long rK, long rV, int D, int k_bits, int v_bits,
                       int Gk, int Gv, int origin_bytes, int step_bytes,
                       int float_bytes);

#ifdef __cplusplus
}
#endif
#endif
