// KIVI streaming variant ("KIVI: KV cache axes" §4–§7): keys quantized per
// channel in groups of G = 32 tokens, sealed R = 128 tokens at a time; values
// a FIFO residual of R tokens, the token leaving it quantized per token in
// groups of 32 channels; origin and step kept in the input dtype (bf16) and
// computed in it (every operation an fp32 operation rounded to bf16).
//
// Record of 128 key tokens (RecLayout with kivi = 1):
//   key part:   codes in the key fragment order (frag_layout.h), then steps
//               bf16 [4 sub-groups][D] and origins bf16 [4][D]
//   value part: codes in the value fragment order for the record's tokens
//               whose values have left the FIFO, steps bf16 [128][D/32] and
//               origins bf16 [128][D/32]; zero for the others
// The value FIFO is the cache's residual V window used as a ring: token t
// sits in slot t mod 128.  With T_k = 128 n quantized keys and r_K key
// residual tokens, slot i < r_K holds token T_k + i (a key residual token)
// and slot i >= r_K token T_k - 128 + i (of the last record, not yet
// quantized), so the last record's value i comes from the codes for i < r_K
// and from ring slot i otherwise.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "frag_layout.h"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kSub = 32;                  // KIVI group: tokens (keys) / channels (values)
constexpr int kSubs = kKG / kSub;         // key sub-groups per record

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ float bfr(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ uint16_t bf_bits(float exact) {
  return static_cast<uint16_t>(__float_as_uint(exact) >> 16);
}
// -0.0 below +0.0 (the oracle's order of values)
__device__ __forceinline__ bool less_signed(float a, float b) {
  return a < b || (a == b && (__float_as_uint(a) & 0x80000000u) && !(__float_as_uint(b) & 0x80000000u));
}

struct KiviGroup {
  float m, step;      // bf16 values
  unsigned flags;
};

// The KIVI quantizer of one group (bf16 arithmetic): R = bf16(M - m), step =
// bf16(R / (2^b - 1)); a constant group keeps step 0.
__device__ __forceinline__ KiviGroup kivi_params(float lo, float hi, bool nonfinite, int top) {
  KiviGroup p{lo, 0.0f, nonfinite ? static_cast<unsigned>(KVQ_FLAG_NONFINITE) : 0u};
  if (nonfinite || hi == lo) return p;
  const float range = bfr(__fsub_rn(hi, lo));
  const float step = bfr(__fdiv_rn(range, static_cast<float>(top)));
  if (!(step > 0.0f) || !isfinite(step)) p.flags |= KVQ_FLAG_RANGE;
  p.step = step;
  return p;
}
// code = clip(RNE(bf16(bf16(x - m) / step)), 0, top); 0 for a constant group
__device__ __forceinline__ uint32_t kivi_code(float x, const KiviGroup& p, int top) {
  if (p.step == 0.0f || p.flags) return 0u;
  const float diff = bfr(__fsub_rn(x, p.m));
  const float y = bfr(__fdiv_rn(diff, p.step));
  return static_cast<uint32_t>(fminf(fmaxf(rintf(y), 0.0f), static_cast<float>(top)));
}

// The same code without a division for most elements.  With rcp =
// RN(1/step), z = RN(diff * rcp) lies within 2.5 fp32 ulps of the IEEE
// quotient RN(diff / step), so both round to the same bf16 value unless a
// bf16 rounding boundary (an fp32 value whose low 16 bits are 0x8000) lies
// within 3 ulps of z; those elements, and groups whose step is below
// 2^-100 (rcp could overflow), take the quotient.
struct KiviFast {
  float rcp;
  bool exact;   // every element by the quotient (a constant, flagged or tiny-step group too)
};
__device__ __forceinline__ KiviFast kivi_fast(const KiviGroup& p) {
  return {p.step > 0.0f ? __frcp_rn(p.step) : 0.0f, !(p.step >= 0x1p-100f) || p.flags != 0u};
}
__device__ __forceinline__ uint32_t kivi_code_fast(float x, const KiviGroup& p, const KiviFast& f,
                                                   int top) {
  if (f.exact) return kivi_code(x, p, top);
  const float diff = bfr(__fsub_rn(x, p.m));
  const float z = __fmul_rn(diff, f.rcp);
  const uint32_t lo = __float_as_uint(z) & 0xFFFFu;
  const float y = lo - (0x8000u - 3u) <= 6u ? bfr(__fdiv_rn(diff, p.step)) : bfr(z);
  return static_cast<uint32_t>(fminf(fmaxf(rintf(y), 0.0f), static_cast<float>(top)));
}

// 128 bf16 rows of D channels into shared memory (row t at t * D), rows
// [0, n) from src + t * D; 16-byte copies.
__device__ __forceinline__ void stage_rows(const kvq_bf16* src, int n, uint16_t* s) {
  const uint4* g = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(s);
  for (int i = threadIdx.x; i < n * (kD / 8); i += blockDim.x) d[i] = g[i];
}

struct KiviArgs {
  QuantSrc src;           // rows: unit u, record k, token t at k * group_stride + t * D
  uint8_t* records;
  long long rec_bytes;
  int max_groups;
  int first_group;        // record of blockIdx.x = 0
  RecLayout lay;
  int t0, t1;             // value kernel: tokens [t0, t1) of the record (clamped per record)
  int n_valid;            // value kernel: tokens of the records that are quantized (prefill)
  unsigned* status;
};

__device__ __forceinline__ uint8_t* kivi_record(const KiviArgs& a) {
  return a.records + (static_cast<long long>(blockIdx.y) * a.max_groups + a.first_group + blockIdx.x) *
                         a.rec_bytes;
}

// Seal 128 key tokens into a record: per (sub-group, channel) one group of 32
// tokens; codes staged as bytes, then packed into fragment-order words.  The
// record's value part is zeroed (its values arrive token by token).
template <int KB>
__global__ void __launch_bounds__(256) kivi_seal_keys_kernel(KiviArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem);        // [128][D]
  uint8_t* cB = smem + kKG * kD * 2;                       // codes [128][D]
  constexpr int top = (1 << KB) - 1;
  const long long off = static_cast<long long>(blockIdx.y) * a.src.unit_stride +
                        static_cast<long long>(blockIdx.x) * a.src.group_stride;
  stage_rows(a.src.k + off, kKG, sK);
  __syncthreads();
  uint8_t* rec = kivi_record(a);
  const RecLayout& L = a.lay;
  uint16_t* kst = reinterpret_cast<uint16_t*>(rec + L.k_scale);
  uint16_t* kmn = reinterpret_cast<uint16_t*>(rec + L.k_min);
  unsigned flags = 0;
  for (int gi = threadIdx.x; gi < kSubs * kD; gi += blockDim.x) {
    const int sg = gi / kD, d = gi % kD;
    float lo = bf(sK[(kSub * sg) * kD + d]), hi = lo;
    bool nf = false;
    for (int t = kSub * sg; t < kSub * sg + kSub; ++t) {
      const float x = bf(sK[t * kD + d]);
      nf |= !isfinite(x);
      if (less_signed(x, lo)) lo = x;
      if (less_signed(hi, x)) hi = x;
    }
    const KiviGroup p = kivi_params(lo, hi, nf, top);
    flags |= p.flags;
    kst[sg * kD + d] = bf_bits(p.step);
    kmn[sg * kD + d] = nf ? 0 : bf_bits(p.m);
    const KiviFast f = kivi_fast(p);
    for (int t = kSub * sg; t < kSub * sg + kSub; ++t)
      cB[t * kD + d] = static_cast<uint8_t>(kivi_code_fast(bf(sK[t * kD + d]), p, f, top));
  }
  // value part of the record: empty until tokens leave the FIFO
  uint4* vz = reinterpret_cast<uint4*>(rec + L.v_codes);
  for (int i = threadIdx.x; i < (static_cast<int>(a.rec_bytes) - L.v_codes) / 16; i += blockDim.x)
    vz[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  uint32_t* dst = reinterpret_cast<uint32_t*>(rec + L.k_codes);
  constexpr int per = 32 / KB;
  for (int w = threadIdx.x; w < kKG * kD * KB / 32; w += blockDim.x) {
    uint32_t acc = 0;
    for (int s = 0; s < per; ++s) {
      int tok, ch;
      key_word_code(w, s, KB, tok, ch);
      acc |= static_cast<uint32_t>(cB[tok * kD + ch]) << (KB * s);
    }
    dst[w] = acc;
  }
  if (flags) atomicOr(a.status, flags);
}

// Quantize the values of tokens [t0, t1) of a record (clamped to the
// record's quantized tokens n_valid - 128 * record for a prefill): per token
// 4 groups of 32 channels; the codes are OR-ed into the fragment-order words
// (the other tokens' bits are kept) and the metadata written.
template <int VB>
__global__ void __launch_bounds__(256) kivi_values_kernel(KiviArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* sV = reinterpret_cast<uint16_t*>(smem);        // [128][D]
  uint8_t* cB = smem + kKG * kD * 2;                       // codes [128][D]
  constexpr int top = (1 << VB) - 1;
  const int rec_idx = a.first_group + blockIdx.x;
  const int t0 = a.t0;
  const int t1 = min(a.t1, a.n_valid - kKG * rec_idx);
  if (t1 <= t0) return;   // block-uniform
  const long long off = static_cast<long long>(blockIdx.y) * a.src.unit_stride +
                        static_cast<long long>(blockIdx.x) * a.src.group_stride;
  stage_rows(a.src.v + off + static_cast<long long>(t0) * kD, t1 - t0, sV + t0 * kD);
  __syncthreads();
  uint8_t* rec = kivi_record(a);
  const RecLayout& L = a.lay;
  uint16_t* vst = reinterpret_cast<uint16_t*>(rec + L.v_scale);
  uint16_t* vmn = reinterpret_cast<uint16_t*>(rec + L.v_min);
  unsigned flags = 0;
  for (int gi = threadIdx.x + t0 * kVGroups; gi < t1 * kVGroups; gi += blockDim.x) {
    const int t = gi / kVGroups, j = gi % kVGroups;
    const uint16_t* row = sV + t * kD + kSub * j;
    float lo = bf(row[0]), hi = lo;
    bool nf = false;
    for (int c = 0; c < kSub; ++c) {
      const float x = bf(row[c]);
      nf |= !isfinite(x);
      if (less_signed(x, lo)) lo = x;
      if (less_signed(hi, x)) hi = x;
    }
    const KiviGroup p = kivi_params(lo, hi, nf, top);
    flags |= p.flags;
    vst[t * kVGroups + j] = bf_bits(p.step);
    vmn[t * kVGroups + j] = nf ? 0 : bf_bits(p.m);
    const KiviFast f = kivi_fast(p);
    for (int c = 0; c < kSub; ++c)
      cB[t * kD + kSub * j + c] = static_cast<uint8_t>(kivi_code_fast(bf(row[c]), p, f, top));
  }
  __syncthreads();
  uint32_t* dst = reinterpret_cast<uint32_t*>(rec + L.v_codes);
  constexpr int per = 32 / VB;
  for (int w = threadIdx.x; w < kKG * kD * VB / 32; w += blockDim.x) {
    uint32_t acc = 0;
    bool any = false;
    for (int s = 0; s < per; ++s) {
      int tok, ch;
      value_word_code(w, s, VB, tok, ch);
      if (tok >= t0 && tok < t1) {
        acc |= static_cast<uint32_t>(cB[tok * kD + ch]) << (VB * s);
        any = true;
      }
    }
    if (any) dst[w] |= acc;
  }
  if (flags) atomicOr(a.status, flags);
}

constexpr int kKiviSmem = kKG * kD * 2 + kKG * kD;   // staged rows + code bytes (48 KB)

template <typename K>
cudaError_t launch_kivi(K kernel, const KiviArgs& a, int n_records, int units, cudaStream_t s) {
  static SmemOptIn opt_in;
  cudaError_t e = opt_in.ensure(kernel);
  if (e != cudaSuccess) return e;
  kernel<<<dim3(n_records, units), 256, kKiviSmem, s>>>(a);
  return cudaGetLastError();
}

KiviArgs kivi_args(const kvq_cache* c, QuantSrc src, int first_group) {
  KiviArgs a;
  a.src = src;
  a.records = c->records;
  a.rec_bytes = c->lay.bytes;
  a.max_groups = c->max_groups;
  a.first_group = first_group;
  a.lay = c->lay;
  a.t0 = 0;
  a.t1 = kKG;
  a.n_valid = 1 << 30;
  a.status = c->status;
  return a;
}

// Export of the KIVI key codes: block (record, unit), thread = channel;
// per 32-token sub-group the channel's codes LSB first along its tokens.
__global__ void kivi_export_k_kernel(const uint8_t* __restrict__ records, long long rec_bytes,
                                     int max_groups, int kb, uint8_t* dst, int n) {
  const int g = blockIdx.x, u = blockIdx.y, d = threadIdx.x;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(
      records + (static_cast<long long>(u) * max_groups + g) * rec_bytes);
  const int per = 8 / kb, nbytes = kSub * kb / 8;
  const uint32_t mask = (1u << kb) - 1u;
  for (int sg = 0; sg < kSubs; ++sg) {
    uint8_t* out = dst + ((static_cast<long long>(u) * n + g) * kSubs + sg) * kD * nbytes +
                   static_cast<long long>(d) * nbytes;
    for (int i = 0; i < nbytes; ++i) {
      uint32_t byte = 0;
      for (int e = 0; e < per; ++e) {
        const CodePos p = key_code_pos(kSub * sg + i * per + e, d, kb);
        byte |= ((words[p.word] >> p.bit) & mask) << (kb * e);
      }
      out[i] = static_cast<uint8_t>(byte);
    }
  }
}

// Export of the KIVI value codes: block (record, unit), thread = token;
// the token's codes LSB first along channels.
__global__ void kivi_export_v_kernel(const uint8_t* __restrict__ records, long long rec_bytes,
                                     int max_groups, int off, int vb, uint8_t* dst, int n) {
  const int g = blockIdx.x, u = blockIdx.y, tok = threadIdx.x;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(
      records + (static_cast<long long>(u) * max_groups + g) * rec_bytes + off);
  const int per = 8 / vb, row = kD * vb / 8;
  const uint32_t mask = (1u << vb) - 1u;
  uint8_t* out = dst + ((static_cast<long long>(u) * n + g) * kKG + tok) * row;
  for (int i = 0; i < row; ++i) {
    uint32_t byte = 0;
    for (int e = 0; e < per; ++e) {
      const CodePos p = value_code_pos(tok, i * per + e, vb);
      byte |= ((words[p.word] >> p.bit) & mask) << (vb * e);
    }
    out[i] = static_cast<uint8_t>(byte);
  }
}

// Bytes [off, off + bytes) of records [u][0..n) into dst [u][n][bytes].
__global__ void kivi_gather_kernel(const uint8_t* __restrict__ records, long long rec_bytes,
                                   int max_groups, int off, int bytes, uint8_t* dst, int n) {
  const int g = blockIdx.x, u = blockIdx.y;
  const uint8_t* src = records + (static_cast<long long>(u) * max_groups + g) * rec_bytes + off;
  uint8_t* out = dst + (static_cast<long long>(u) * n + g) * bytes;
  for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(src)[i];
}

}  // namespace

cudaError_t launch_export_kivi(const kvq_cache* c, uint8_t* k_codes, kvq_bf16* k_origin,
                               kvq_bf16* k_step, uint8_t* v_codes, kvq_bf16* v_origin,
                               kvq_bf16* v_step, cudaStream_t s) {
  const int n = c->t_q / kKG, units = c->cfg.batch * c->cfg.kv_heads;
  if (n == 0) return cudaSuccess;
  const RecLayout& L = c->lay;
  const dim3 grid(n, units);
  kivi_export_k_kernel<<<grid, kD, 0, s>>>(c->records, L.bytes, c->max_groups, L.kb, k_codes, n);
  kivi_export_v_kernel<<<grid, kKG, 0, s>>>(c->records, L.bytes, c->max_groups, L.v_codes, L.vb,
                                            v_codes, n);
  const int kmeta = kSubs * kD * 2, vmeta = kKG * kVGroups * 2;
  kivi_gather_kernel<<<grid, 64, 0, s>>>(c->records, L.bytes, c->max_groups, L.k_min, kmeta,
                                         reinterpret_cast<uint8_t*>(k_origin), n);
  kivi_gather_kernel<<<grid, 64, 0, s>>>(c->records, L.bytes, c->max_groups, L.k_scale, kmeta,
                                         reinterpret_cast<uint8_t*>(k_step), n);
  kivi_gather_kernel<<<grid, 64, 0, s>>>(c->records, L.bytes, c->max_groups, L.v_min, vmeta,
                                         reinterpret_cast<uint8_t*>(v_origin), n);
  kivi_gather_kernel<<<grid, 64, 0, s>>>(c->records, L.bytes, c->max_groups, L.v_scale, vmeta,
                                         reinterpret_cast<uint8_t*>(v_step), n);
  return cudaGetLastError();
}

cudaError_t launch_kivi_seal(const kvq_cache* c, QuantSrc src, int n_records, int first_record,
                             cudaStream_t s) {
  if (n_records == 0) return cudaSuccess;
  const KiviArgs a = kivi_args(c, src, first_record);
  const int units = c->cfg.batch * c->cfg.kv_heads;
  return c->cfg.k_bits == 2 ? launch_kivi(kivi_seal_keys_kernel<2>, a, n_records, units, s)
                            : launch_kivi(kivi_seal_keys_kernel<4>, a, n_records, units, s);
}

cudaError_t launch_kivi_values(const kvq_cache* c, QuantSrc src, int n_records, int first_record,
                               int t0, int t1, int n_valid, cudaStream_t s) {
  if (n_records == 0 || t1 <= t0) return cudaSuccess;
  KiviArgs a = kivi_args(c, src, first_record);
  a.t0 = t0;
  a.t1 = t1;
  a.n_valid = n_valid;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  return c->cfg.v_bits == 2 ? launch_kivi(kivi_values_kernel<2>, a, n_records, units, s)
                            : launch_kivi(kivi_values_kernel<4>, a, n_records, units, s);
}

}  // namespace kvq
