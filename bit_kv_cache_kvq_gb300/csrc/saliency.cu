// MixKVQ channel salience and tiers ("MixKVQ: Query-Aware Mixed-Precision
// KV Cache Quantization for Long-Context Reasoning": salience score
// derivation, three-tier strategy, GQA aggregation in the system-level
// implementation details).
//
// One CTA per (batch row, KV head), one thread per channel d:
//   I_d = (fp32 sum, token i ascending then GQA head ascending, of |Q|)
//         / (n_rep * Lq)                         -- one IEEE division
//   S_d = fl32(fl32(max_t k - min_t k) / (2^B - 1))
//   A_d = fl32(I_d * S_d)
// The summation order is fixed so the result is bit-reproducible.
//
// Online form (MixKVQ "efficient online salience estimation"): the cache
// keeps the running |q| sum per (batch row, KV head, channel); each decode
// step adds its query heads' magnitudes in head order, so a window of steps
// sums in exactly the order above and its I_d is the same number.
#include <cuda_runtime.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ float bf2f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__global__ void __launch_bounds__(kD) saliency_kernel(
    const uint16_t* __restrict__ q_win, int Hq, int Lq,
    const uint16_t* __restrict__ k_grp, int Hkv, int G, int sal_bits,
    kvq_tier_spec spec, float* I_out, float* A_out, uint8_t* tiers_out) {
  __shared__ float sA[kD];
  const int u = blockIdx.x;
  const int b = u / Hkv, kvh = u % Hkv;
  const int d = threadIdx.x;
  const int n_rep = Hq / Hkv;

  float acc = 0.0f;
  const uint16_t* qb = q_win + (static_cast<long long>(b) * Hq + kvh * n_rep) * Lq * kD + d;
  for (int i = 0; i < Lq; ++i)
    for (int h = 0; h < n_rep; ++h)
      acc = __fadd_rn(acc, fabsf(bf2f(qb[(static_cast<long long>(h) * Lq + i) * kD])));
  const float I = __fdiv_rn(acc, static_cast<float>(n_rep * Lq));

  const uint16_t* kb = k_grp + static_cast<long long>(u) * G * kD + d;
  float lo = bf2f(kb[0]), hi = lo;
  bool bad = !isfinite(lo);
  for (int t = 1; t < G; ++t) {
    const float x = bf2f(kb[static_cast<long long>(t) * kD]);
    bad |= !isfinite(x);
    lo = fminf(lo, x);
    hi = fmaxf(hi, x);
  }
  const float S = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>((1 << sal_bits) - 1));
  const float A = bad ? __int_as_float(0x7fc00000) : __fmul_rn(I, S);
  sA[d] = A;
  __syncthreads();

  int tier;
  if (spec.mode == KVQ_TIERS_RANK) {
    int rank = 0;
    for (int e = 0; e < kD; ++e) {
      const float Ae = sA[e];
      rank += (Ae > A || (Ae == A && e < d)) ? 1 : 0;
    }
    tier = rank < spec.n_bf16 ? KVQ_TIER_BF16
           : rank < spec.n_bf16 + spec.n_uint4 ? KVQ_TIER_UINT4
                                               : KVQ_TIER_UINT2;
  } else {
    tier = A > spec.tau_bf16 ? KVQ_TIER_BF16
           : A > spec.tau_uint4 ? KVQ_TIER_UINT4
                                : KVQ_TIER_UINT2;
  }
  const long long o = static_cast<long long>(u) * kD + d;
  if (I_out) I_out[o] = I;
  if (A_out) A_out[o] = A;
  if (tiers_out) tiers_out[o] = static_cast<uint8_t>(tier);
}

// One decode step into the running sums: block = unit, thread = channel.
__global__ void __launch_bounds__(kD) observe_query_kernel(const uint16_t* __restrict__ q,
                                                           int Hq, int Hkv, float* acc,
                                                           unsigned* status) {
  const int u = blockIdx.x, d = threadIdx.x;
  const int b = u / Hkv, kvh = u % Hkv, n_rep = Hq / Hkv;
  const uint16_t* qb = q + (static_cast<long long>(b) * Hq + kvh * n_rep) * kD + d;
  const long long o = static_cast<long long>(u) * kD + d;
  float a = acc[o];
  bool bad = false;
  for (int h = 0; h < n_rep; ++h) {
    const float x = bf2f(qb[h * kD]);
    bad |= !isfinite(x);
    a = __fadd_rn(a, fabsf(x));
  }
  acc[o] = a;
  if (bad) atomicOr(status, static_cast<unsigned>(KVQ_FLAG_NONFINITE));
}

__global__ void __launch_bounds__(kD) window_importance_kernel(const float* __restrict__ acc,
                                                               float count, float* I) {
  const long long o = static_cast<long long>(blockIdx.x) * kD + threadIdx.x;
  I[o] = __fdiv_rn(acc[o], count);
}

}  // namespace

cudaError_t launch_observe_query(const kvq_cache* c, const kvq_bf16* q, int Hq, cudaStream_t s) {
  observe_query_kernel<<<c->cfg.batch * c->cfg.kv_heads, kD, 0, s>>>(
      q, Hq, c->cfg.kv_heads, c->qacc, c->status);
  return cudaGetLastError();
}

cudaError_t launch_window_importance(const kvq_cache* c, float* I, cudaStream_t s) {
  window_importance_kernel<<<c->cfg.batch * c->cfg.kv_heads, kD, 0, s>>>(
      c->qacc, static_cast<float>(c->q_rep * c->q_steps), I);
  return cudaGetLastError();
}

cudaError_t launch_saliency(const kvq_bf16* q_win, int Hq, int Lq,
                            const kvq_bf16* k_grp, int B, int Hkv, int G,
                            int sal_bits, const kvq_tier_spec* spec,
                            float* I_out, float* A_out, uint8_t* tiers_out,
                            cudaStream_t s) {
  saliency_kernel<<<B * Hkv, kD, 0, s>>>(q_win, Hq, Lq, k_grp, Hkv, G, sal_bits,
                                         *spec, I_out, A_out, tiers_out);
  return cudaGetLastError();
}

}  // namespace kvq
