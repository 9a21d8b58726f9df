// PN-Mix H3/L1 keys (PN-Mix reproduction notes): the once-per-prefill pair
// selection of Eq. 6 and the canonical export of the H3/L1 key groups.  The
// key groups themselves are quantized in quant.cu; the decode reads them in
// decode_mma.cuh.
#include <cuda_runtime.h>

#include "frag_layout.h"
#include "kvq_internal.h"
#include "sqrt_rn.h"

namespace kvq {
namespace {

__device__ __forceinline__ float bfv(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Eq. 6 for one (b, KV head): block = unit.  sigma_i = qbar_i * kbar_i
// (qbar: the mean over the GQA group's heads, in order, of the heads' mean
// pair norms).  The unit's key rows stream through a ring of kPairStages
// shared-memory slots of kPairRows rows (one bulk copy a slot, on an
// mbarrier).  Threads 64 and up compute a chunk's pair norms (thread ->
// pair tid mod 64, rows tid / 64 - 1 + 7k) into one half of a term table
// while thread i < 64 adds the previous chunk's terms of pair i in token
// order from the other half; the query window goes through the table with
// every thread computing terms.  Then the n_high largest sigma (ties: lower
// pair; a NaN counts as the smallest) are selected, and the unit's stored
// channel order is written: the selected pairs' channels ascending, then
// the others ascending.
constexpr int kPairRows = 128;
constexpr int kPairStages = 4;
constexpr int kPairThreads = 512;
constexpr int kPairWaitPolls = 1 << 20;
constexpr size_t kPairRing = static_cast<size_t>(kPairStages) * kPairRows * kD * 2;
constexpr size_t kPairTerms = 2 * static_cast<size_t>(kPairRows) * (kD / 2) * 4;   // two halves
constexpr size_t kPairSmem = kPairRing + kPairTerms + kPairStages * 8 + 16;

__device__ __forceinline__ bool pair_wait(uint32_t mb, uint32_t parity, int polls) {
  for (int i = 0; i < polls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(mb), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// sqrt(a^2 + b^2), every operation fp32 rounded (the root correctly rounded)
__device__ __forceinline__ float pair_norm(uint16_t xa, uint16_t xb, bool& bad) {
  const float x = bfv(xa), y = bfv(xb);
  const float s = __fadd_rn(__fmul_rn(x, x), __fmul_rn(y, y));
  // a non-finite input leaves s infinite or NaN; only then (or when finite
  // inputs overflow) are the inputs themselves tested
  if (!(s <= 3.40282346638528860e38f) && (!isfinite(x) || !isfinite(y))) bad = true;
  return sqrt_rn(s);
}

__global__ void __launch_bounds__(kPairThreads) pnmix_pairs_kernel(
    const uint16_t* __restrict__ q, int Hq, int Lq, const uint16_t* __restrict__ k, int Lk,
    int Hkv, int layout, int n_high, float* sigma_out, uint8_t* perm, unsigned* status) {
  constexpr int P = kD / 2;
  constexpr int kRowStep = kPairThreads / P;   // 4 rows in flight per pass of the threads
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* ring = reinterpret_cast<uint16_t*>(smem);                   // [stage][row][D]
  float* terms = reinterpret_cast<float*>(smem + kPairRing);            // [row][pair]
  const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem + kPairRing + kPairTerms));
  __shared__ float sig[P];
  __shared__ uint8_t high[kD];
  __shared__ int stop;
  const int u = blockIdx.x, tid = threadIdx.x, i = tid & (P - 1), r0 = tid / P;
  const int b = u / Hkv, kvh = u % Hkv, hg = Hq / Hkv;
  const int ca = layout == KVQ_PAIRS_ADJACENT ? 2 * i : i;
  const int cb = layout == KVQ_PAIRS_ADJACENT ? 2 * i + 1 : i + P;
  const uint8_t* ku = reinterpret_cast<const uint8_t*>(k + static_cast<long long>(u) * Lk * kD);
  const int nch = (Lk + kPairRows - 1) / kPairRows;
  if (tid == 0) {
    for (int st = 0; st < kPairStages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(bar0 + 8 * st) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    stop = 0;
  }
  __syncthreads();
  // chunk c (rows 64c ..) into stage c % kPairStages (thread 0)
  auto issue = [&](int c) {
    const uint32_t bytes = static_cast<uint32_t>(min(kPairRows, Lk - kPairRows * c) * kD * 2);
    const uint32_t mb = bar0 + 8 * (c % kPairStages);
    const uint32_t dst = static_cast<uint32_t>(
        __cvta_generic_to_shared(ring + static_cast<size_t>(c % kPairStages) * kPairRows * kD));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mb), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(ku + static_cast<long long>(c) * kPairRows * kD * 2), "r"(bytes), "r"(mb)
        : "memory");
  };
  int issued = 0;
  if (tid == 0)
    for (; issued < min(kPairStages, nch); ++issued) issue(issued);
  bool bad = false;
  // Key means, two chunks in flight: in pass c the producer threads (P and
  // up) write chunk c's pair norms into table half c & 1 while thread i < P
  // adds chunk c - 1's terms of pair i, in token order, from the other half.
  constexpr int kProdRows = (kPairThreads - P) / P;   // 7 rows in flight per pass of the producers
  float kacc = 0.0f;
  int c = 0;
  for (; c <= nch; ++c) {
    const bool produce = c < nch;
    const int st = c % kPairStages;
    if (produce && tid >= P && !pair_wait(bar0 + 8 * st, (c / kPairStages) & 1, kPairWaitPolls))
      atomicOr(&stop, 1);
    __syncthreads();   // every producer has waited (or given up)
    if (stop) break;   // block-uniform
    if (tid >= P) {
      if (produce) {
        const uint16_t* rows = ring + static_cast<size_t>(st) * kPairRows * kD;
        float* tb = terms + (c & 1) * (kPairRows * P);
        const int n = min(kPairRows, Lk - kPairRows * c);
#pragma unroll 4
        for (int r = tid / P - 1; r < n; r += kProdRows)
          tb[r * P + i] = pair_norm(rows[r * kD + ca], rows[r * kD + cb], bad);
      }
    } else if (c > 0) {
      const float* tb = terms + ((c - 1) & 1) * (kPairRows * P);
      const int n = min(kPairRows, Lk - kPairRows * (c - 1));
      // sixteen terms' loads ahead of their additions (in token order)
      for (int r0s = 0; r0s < n; r0s += 16) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = tb[min(r0s + j, n - 1) * P + i];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (r0s + j < n) kacc = __fadd_rn(kacc, v[j]);
      }
    }
    __syncthreads();   // chunk c's stage consumed and its terms written, chunk c - 1's added
    if (tid == 0 && produce && issued < nch) issue(issued++);
  }
  if (stop && tid == 0) {
    // a wait gave up: every copy still in flight lands before the block
    // leaves (full limit), and the selection is flagged invalid
    atomicOr(status, static_cast<unsigned>(KVQ_FLAG_TIMEOUT));
    for (int cc = c; cc < issued; ++cc)
      pair_wait(bar0 + 8 * (cc % kPairStages), (cc / kPairStages) & 1, kPairWaitPolls);
  }
  // query means: per head, chunks of 64 tokens through the same table
  float qsum = 0.0f;
  for (int h = 0; h < hg; ++h) {
    const uint16_t* qh = q + (static_cast<long long>(b) * Hq + kvh * hg + h) * Lq * kD;
    float acc = 0.0f;
    for (int t0 = 0; t0 < Lq; t0 += kPairRows) {
      const int n = min(kPairRows, Lq - t0);
#pragma unroll 4
      for (int r = r0; r < n; r += kRowStep) {
        const long long row = static_cast<long long>(t0 + r) * kD;
        terms[r * P + i] = pair_norm(qh[row + ca], qh[row + cb], bad);
      }
      __syncthreads();
      if (tid < P) {
        for (int r0s = 0; r0s < n; r0s += 16) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = terms[min(r0s + j, n - 1) * P + i];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (r0s + j < n) acc = __fadd_rn(acc, v[j]);
        }
      }
      __syncthreads();
    }
    qsum = __fadd_rn(qsum, __fdiv_rn(acc, static_cast<float>(Lq)));
  }
  if (tid < P) {
    const float kbar = __fdiv_rn(kacc, static_cast<float>(Lk));
    const float s = __fmul_rn(__fdiv_rn(qsum, static_cast<float>(hg)), kbar);
    sig[i] = s;
    if (sigma_out) sigma_out[static_cast<long long>(u) * P + i] = s;
  }
  if (bad && status) atomicOr(status, static_cast<unsigned>(KVQ_FLAG_NONFINITE));
  __syncthreads();
  if (tid < P) {
    const float s = sig[i];
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
  }
  __syncthreads();
  // stored position of every channel: selected channels first, each part ascending
  for (int ch = tid; ch < kD; ch += kPairThreads) {
    int pos = 0;
    const int nh = 2 * n_high;
    if (high[ch]) {
      for (int e = 0; e < ch; ++e) pos += high[e];
    } else {
      pos = nh;
      for (int e = 0; e < ch; ++e) pos += !high[e];
    }
    perm[static_cast<long long>(u) * kD + pos] = static_cast<uint8_t>(ch);
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
  static SmemOptIn opt_in;
  cudaError_t e = opt_in.ensure(pnmix_pairs_kernel);
  if (e != cudaSuccess) return e;
  pnmix_pairs_kernel<<<units, kPairThreads, kPairSmem, s>>>(
      reinterpret_cast<const uint16_t*>(q), Hq, Lq, reinterpret_cast<const uint16_t*>(k), Lk,
      c->cfg.kv_heads, c->cfg.pair_layout, c->cfg.n_high_pairs, sigma, c->pn_perm, c->status);
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
