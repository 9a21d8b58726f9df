// PN-Mix H3/L1 keys (PN-Mix reproduction notes): the once-per-prefill pair
// selection of Eq. 6 and the canonical export of the H3/L1 key groups.  The
// key groups themselves are quantized in quant.cu; the decode reads them in
// decode_mma.cuh.
#include <cuda_runtime.h>

#include "frag_layout.h"
#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ float bfv(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Mean pair norm of rows [0, L) of x (bf16 [L][D]): (1/L) sum_t
// sqrt(a^2 + b^2), every operation fp32 rounded, the sum in token order.
__device__ float mean_pair_norm(const uint16_t* x, int L, int ca, int cb, bool& bad) {
  float acc = 0.0f;
  for (int t = 0; t < L; ++t) {
    const float a = bfv(x[static_cast<long long>(t) * kD + ca]);
    const float b = bfv(x[static_cast<long long>(t) * kD + cb]);
    if (!isfinite(a) || !isfinite(b)) bad = true;
    const float ss = __fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b));
    acc = __fadd_rn(acc, __fsqrt_rn(ss));
  }
  return __fdiv_rn(acc, static_cast<float>(L));
}

// Eq. 6 for one (b, KV head): block = unit, thread = pair i.  sigma_i =
// qbar_i * kbar_i (qbar: the mean over the GQA group's heads, in order, of
// the heads' mean pair norms).  Then the n_high largest sigma (ties: lower
// pair; a NaN counts as the smallest) are selected, and the unit's stored
// channel order is written: the selected pairs' channels ascending, then
// the others ascending.
__global__ void __launch_bounds__(kD / 2) pnmix_pairs_kernel(
    const uint16_t* __restrict__ q, int Hq, int Lq, const uint16_t* __restrict__ k, int Lk,
    int Hkv, int layout, int n_high, float* sigma_out, uint8_t* perm, unsigned* status) {
  constexpr int P = kD / 2;
  __shared__ float sig[P];
  __shared__ uint8_t high[kD];
  const int u = blockIdx.x, i = threadIdx.x;
  const int b = u / Hkv, kvh = u % Hkv, hg = Hq / Hkv;
  const int ca = layout == KVQ_PAIRS_ADJACENT ? 2 * i : i;
  const int cb = layout == KVQ_PAIRS_ADJACENT ? 2 * i + 1 : i + P;
  bool bad = false;
  float qsum = 0.0f;
  for (int h = 0; h < hg; ++h) {
    const uint16_t* qh = q + (static_cast<long long>(b) * Hq + kvh * hg + h) * Lq * kD;
    qsum = __fadd_rn(qsum, mean_pair_norm(qh, Lq, ca, cb, bad));
  }
  const float qbar = __fdiv_rn(qsum, static_cast<float>(hg));
  const float kbar = mean_pair_norm(k + static_cast<long long>(u) * Lk * kD, Lk, ca, cb, bad);
  const float s = __fmul_rn(qbar, kbar);
  sig[i] = s;
  if (sigma_out) sigma_out[static_cast<long long>(u) * P + i] = s;
  if (bad && status) atomicOr(status, static_cast<unsigned>(KVQ_FLAG_NONFINITE));
  __syncthreads();
  int rank = 0;
  for (int j = 0; j < P; ++j) {
    const float sj = sig[j];
    const bool before = s != s ? (sj == sj || j < i)                 // NaN: last
                               : (sj > s || (sj == s && j < i));
    rank += before ? 1 : 0;
  }
  const bool sel = rank < n_high;
  high[ca] = sel;
  high[cb] = sel;
  __syncthreads();
  // stored position of channels ca, cb: selected channels first, each part ascending
  for (int c = i; c < kD; c += P) {
    int pos = 0;
    const int nh = 2 * n_high;
    if (high[c]) {
      for (int e = 0; e < c; ++e) pos += high[e];
    } else {
      pos = nh;
      for (int e = 0; e < c; ++e) pos += !high[e];
    }
    perm[static_cast<long long>(u) * kD + pos] = static_cast<uint8_t>(c);
  }
}

// Canonical export of the H3/L1 key groups: block (group, unit), thread =
// stored position p (channel perm[p]): the code of every token (LSB plane
// bit, plus the upper-plane bits for the high channels), offset, scale.
__global__ void pnmix_export_kernel(const uint8_t* __restrict__ records, long long rec_bytes,
                                    int max_groups, RecLayout L, const uint8_t* __restrict__ perm,
                                    uint8_t* codes, float* offset, float* scale, int n) {
  const int g = blockIdx.x, u = blockIdx.y, p = threadIdx.x;
  const uint8_t* rec = records + (static_cast<long long>(u) * max_groups + g) * rec_bytes;
  const uint32_t* lsb = reinterpret_cast<const uint32_t*>(rec + L.k_codes);
  const uint32_t* up = reinterpret_cast<const uint32_t*>(rec + L.kc);
  const int ch = perm[static_cast<long long>(u) * kD + p];
  const long long ug = static_cast<long long>(u) * n + g;
  offset[ug * kD + ch] = reinterpret_cast<const float*>(rec + L.k_min)[p];
  scale[ug * kD + ch] = reinterpret_cast<const float*>(rec + L.k_scale)[p];
  for (int tok = 0; tok < kKG; ++tok) {
    int mt, ks, lane, reg, half;
    frag_coords(tok, p, mt, ks, lane, reg, half);
    const int rhi = reg & 1, chi = reg >> 1;
    const int word = (mt * 2 + (ks >> 2)) * 32 + lane;
    const int bit = 2 * (ks & 3) + chi + 8 * rhi + 16 * half;
    uint32_t c = (lsb[word] >> bit) & 1u;
    if (p < L.nh) {
      const CodePos q = mixed_code_pos(tok, p, L.kw2);
      c |= ((up[q.word] >> q.bit) & 3u) << 1;
    }
    codes[(ug * kKG + tok) * kD + ch] = static_cast<uint8_t>(c);
  }
}

__global__ void pnmix_high_kernel(const uint8_t* __restrict__ perm, int nh, uint8_t* high) {
  const int u = blockIdx.x, p = threadIdx.x;
  high[static_cast<long long>(u) * kD + perm[static_cast<long long>(u) * kD + p]] = p < nh;
}

}  // namespace

cudaError_t launch_pnmix_pairs(const kvq_cache* c, const kvq_bf16* q, int Hq, int Lq,
                               const kvq_bf16* k, int Lk, float* sigma, cudaStream_t s) {
  const int units = c->cfg.batch * c->cfg.kv_heads;
  pnmix_pairs_kernel<<<units, kD / 2, 0, s>>>(reinterpret_cast<const uint16_t*>(q), Hq, Lq,
                                              reinterpret_cast<const uint16_t*>(k), Lk,
                                              c->cfg.kv_heads, c->cfg.pair_layout,
                                              c->cfg.n_high_pairs, sigma, c->pn_perm, c->status);
  return cudaGetLastError();
}

cudaError_t launch_export_pnmix(const kvq_cache* c, uint8_t* codes, float* offset, float* scale,
                                uint8_t* high, cudaStream_t s) {
  const int n = c->t_q / kKG, units = c->cfg.batch * c->cfg.kv_heads;
  if (high) pnmix_high_kernel<<<units, kD, 0, s>>>(c->pn_perm, c->lay.nh, high);
  if (n > 0)
    pnmix_export_kernel<<<dim3(n, units), kD, 0, s>>>(c->records, c->lay.bytes, c->max_groups,
                                                       c->lay, c->pn_perm, codes, offset, scale, n);
  return cudaGetLastError();
}

}  // namespace kvq
