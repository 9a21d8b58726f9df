// Residual append, group quantization (flush and prefill, uniform and mixed
// keys) and canonical export of the packed cache.
//
// Quantizer ("KIVI: KV cache axes" §2; MixKVQ "KV cache quantization
// principle"; PN-Mix Eq. 2): per group m = min, M = max,
//   step = fl32(fl32(M - m) / (2^b - 1)),  c = clip(RNE(fl32(fl32(x - m) / step)))
// with IEEE fp32 subtraction and division (__fsub_rn / __fdiv_rn), codes
// rounded half-to-even, and a constant group (M == m) stored as step 0,
// codes 0, origin m.  Groups: Key per channel over the 128 tokens of a tile,
// Value per token over 32 consecutive channels (KIVI §3).  Codes are first
// staged as bytes in shared memory and then packed word by word into the
// tensor-core fragment order of frag_layout.h; kvq_export_* converts back to
// the canonical LSB-first layout.
#include <cuda_runtime.h>

#include "frag_layout.h"
#include "kvq_internal.h"

namespace kvq {
namespace {


__device__ __forceinline__ float bf2f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Order-preserving key of a finite float; -0.0 sorts below +0.0.
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Params {
  float m;
  float step;
  unsigned flags;
};

__device__ __forceinline__ Params group_params(float lo, float hi, int top,
                                               bool nonfinite) {
  Params p{lo, 0.0f, nonfinite ? (unsigned)KVQ_FLAG_NONFINITE : 0u};
  if (nonfinite || hi == lo) return p;
  const float range = __fsub_rn(hi, lo);
  const float step = __fdiv_rn(range, static_cast<float>(top));
  if (!(step > 0.0f) || !isfinite(step)) p.flags |= KVQ_FLAG_RANGE;
  p.step = step;
  return p;
}


__device__ __forceinline__ uint16_t f2bf_bits(float exact_bf16_value) {
  return static_cast<uint16_t>(__float_as_uint(exact_bf16_value) >> 16);
}

struct QuantArgs {
  QuantSrc src;
  uint8_t* records;
  long long rec_bytes;
  int max_groups;
  int first_group;
  RecLayout lay;
  const float* importance;  // mixed: [units][D], or NULL: qacc / q_count
  const float* qacc;        // mixed: the online window's |q| sums [units][D]
  float q_count;            // (query heads per KV head) * (steps observed)
  float tau_bf16, tau_uint4;  // threshold tiers (lay.thresh)
  unsigned* status;
};

// Staged tiles: bf16 [128 tokens][128 channels], the 16-byte piece ch/8 of
// row t at piece (ch/8) ^ (t & 7), so column reads (a channel over tokens)
// and row reads (a token's channels) are both free of bank conflicts.
__device__ __forceinline__ int swz(int t, int ch) {
  return t * kD + ((((ch >> 3) ^ (t & 7)) << 3) | (ch & 7));
}

// Stage one 128-token bf16 tile (K or V) in shared memory (cp.async, 16 bytes).
__device__ __forceinline__ void load_tile(const QuantArgs& a, const kvq_bf16* src, uint16_t* sT) {
  const long long off = static_cast<long long>(blockIdx.y) * a.src.unit_stride +
                        static_cast<long long>(blockIdx.x) * a.src.group_stride;
  const uint8_t* gs = reinterpret_cast<const uint8_t*>(src + off);
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(sT));
  for (int i = threadIdx.x; i < kKG * kD * 2 / 16; i += blockDim.x) {
    const int t = i >> 4, pc = i & 15;
    const uint32_t o = static_cast<uint32_t>((t * 16 + (pc ^ (t & 7))) * 16);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d + o), "l"(gs + 16 * i));
  }
  asm volatile("cp.async.commit_group;\n" ::);
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

// Per-group quantizer parameters kept for the code pass: origin m and
// rcp = RN(1 / step) (0 for a constant group), plus the step itself for the
// exact fallback.
struct GroupQ {
  float m, rcp;
};

__device__ __forceinline__ GroupQ make_q(const Params& p) {
  return {p.m, p.step > 0.0f ? __frcp_rn(p.step) : 0.0f};
}

// c = clip(RNE(fl32(fl32(x - m) / step)), 0, top), fast form.  With
// q' = RN(d * RN(1/step)), |q' - RN(d / step)| <= 2^-22 q <= 2^-18 (q <= 15
// plus a rounding, as x <= the group max), so the two round to the same
// integer unless q' lies within 2^-17 of a half-integer; such codes (and
// non-finite q') set `exact` and the caller recomputes with the IEEE
// quotient (code_exact).  Rounding: adding 1.5 * 2^23 rounds q in [0, 2^22)
// to the nearest integer, ties to even, into the low mantissa bits; no
// clamp is needed since 0 <= q < top + 1/2.
constexpr float kTieMargin = 0.4999923706054688f;   // 0.5 - 2^-17
__device__ __forceinline__ uint32_t code_fast(float x, GroupQ g, float& rmax) {
  constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
  const float d = __fsub_rn(x, g.m);
  const float q = __fmul_rn(d, g.rcp);
  const float tq = __fadd_rn(q, kMagic);
  const float n = __fsub_rn(tq, kMagic);
  // NaN (a non-finite group) must reach the exact path: fmaxf would drop it
  const float r = fabsf(__fsub_rn(q, n));
  rmax = r == r ? fmaxf(rmax, r) : 1.0f;
  return __float_as_uint(tq) & 0xFFu;
}
__device__ __forceinline__ uint32_t code_exact(float x, float m, float step, int top) {
  if (step == 0.0f) return 0u;
  const float q = __fdiv_rn(__fsub_rn(x, m), step);
  return static_cast<uint32_t>(fminf(fmaxf(rintf(q), 0.0f), static_cast<float>(top)));
}

// Two bf16 values in a 32-bit word -> two 16-bit order keys (key order =
// value order, -0.0 below +0.0, NaN beyond the infinities).
__device__ __forceinline__ uint32_t key2(uint32_t x) {
  return x ^ (((x >> 15) & 0x00010001u) * 0x7FFFu) ^ 0x80008000u;
}
__device__ __forceinline__ float unkey16(uint32_t k) {
  const uint32_t u = (k & 0x8000u) ? (k ^ 0x8000u) : (~k & 0xFFFFu);
  return __uint_as_float(u << 16);
}
// a 16-bit key range holds a non-finite value iff an extreme is beyond +-inf
__device__ __forceinline__ bool bad_range(uint32_t kmin, uint32_t kmax) {
  return kmax >= 0xFF80u || kmin <= 0x007Fu;
}

// Key channel ranges: thread (pair p = tid & 63 of channels 2p, 2p+1,
// quarter tid >> 6 of 32 tokens), packed keys, merged through shared memory.
// Threads 0..127 return the range of channel tid.
__device__ __forceinline__ void key_ranges(const uint16_t* sK, uint32_t* sRed, float& lo,
                                           float& hi, bool& bad) {
  const int p = threadIdx.x & 63, qq = threadIdx.x >> 6;
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(sK);
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll 8
  for (int t = 32 * qq; t < 32 * qq + 32; ++t) {
    const uint32_t k = key2(t32[t * 64 + ((((p >> 2) ^ (t & 7)) << 2) | (p & 3))]);
    kmin = __vminu2(kmin, k);
    kmax = __vmaxu2(kmax, k);
  }
  sRed[qq * 64 + p] = kmin;
  sRed[256 + qq * 64 + p] = kmax;
  __syncthreads();
  if (threadIdx.x < kD) {
    const int c = threadIdx.x, pp = c >> 1, sh = 16 * (c & 1);
    uint32_t mn = 0xFFFFu, mx = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mn = min(mn, (sRed[i * 64 + pp] >> sh) & 0xFFFFu);
      mx = max(mx, (sRed[256 + i * 64 + pp] >> sh) & 0xFFFFu);
    }
    lo = unkey16(mn);
    hi = unkey16(mx);
    bad = bad_range(mn, mx);
  }
}

// Value groups: thread (token t = tid / 2, h = tid & 1) takes two of the
// token's four 32-channel groups (h = 0: 0, 1; h = 1: 3, 2 -- the order keeps
// a quarter warp's 16-byte reads on distinct banks).  Writes the steps and
// origins to the record and the parameters to vq / vstep [t * 4 + j].
template <int VB>
__device__ __forceinline__ unsigned value_groups(const QuantArgs& a, const uint16_t* sV,
                                                 GroupQ* vq, float* vstep, uint8_t* rec) {
  constexpr int top = (1 << VB) - 1;
  const int t = threadIdx.x >> 1, h = threadIdx.x & 1;
  float* vscale = reinterpret_cast<float*>(rec + a.lay.v_scale);
  uint16_t* vmin = reinterpret_cast<uint16_t*>(rec + a.lay.v_min);
  const uint4* row = reinterpret_cast<const uint4*>(sV + t * kD);
  unsigned flags = 0;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = h ? 3 - jj : jj;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w = row[(4 * j + k) ^ (t & 7)];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t kk = key2(ws[e]);
        kmin = __vminu2(kmin, kk);
        kmax = __vmaxu2(kmax, kk);
      }
    }
    const uint32_t mn = min(kmin & 0xFFFFu, kmin >> 16), mx = max(kmax & 0xFFFFu, kmax >> 16);
    const Params p = group_params(unkey16(mn), unkey16(mx), top, bad_range(mn, mx));
    vq[t * kVGroups + j] = make_q(p);
    vstep[t * kVGroups + j] = p.step;
    vscale[t * kVGroups + j] = p.step;
    vmin[t * kVGroups + j] = f2bf_bits(p.m);
    flags |= p.flags;
  }
  return flags;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Rare exact recomputation of one key word (kept out of line so the fast
// loop stays small in the instruction cache).
template <int KB>
__device__ __noinline__ uint32_t key_word_exact(const uint32_t* t32, const GroupQ* kq,
                                                const float* kstep, int mt, int ks0, int g,
                                                int t) {
  constexpr int top = (1 << KB) - 1;
  constexpr int KSW = KB == 2 ? 2 : 1;
  uint32_t acc = 0;
  for (int kl = 0; kl < KSW; ++kl)
    for (int r = 0; r < 4; ++r) {
      const int tok = 16 * mt + g + 8 * (r & 1);
      const int ch0 = 16 * (ks0 + kl) + 2 * t + 8 * (r >> 1);
      const uint32_t xw = t32[tok * 64 + ((((ch0 >> 3) ^ (tok & 7)) << 2) | ((ch0 & 7) >> 1))];
      for (int hh = 0; hh < 2; ++hh) {
        const float x = hh ? __uint_as_float(xw & 0xFFFF0000u) : __uint_as_float(xw << 16);
        const int ch = ch0 + hh;
        const int pos = KB == 2 ? 2 * pair_2bit(kl, r) + 16 * hh : 4 * nibble_4bit(r) + 16 * hh;
        acc |= code_exact(x, kq[ch].m, kstep[ch], top) << pos;
      }
    }
  return acc;
}

// Rare exact recomputation of one value word.
template <int VB>
__device__ __noinline__ uint32_t value_word_exact(const uint16_t* sV, const GroupQ* vq,
                                                  const float* vstep, int mc, int kt0, int g,
                                                  int t) {
  constexpr int top = (1 << VB) - 1;
  constexpr int KSW = VB == 2 ? 2 : 1;
  const int j = mc >> 1;
  uint32_t acc = 0;
  for (int kl = 0; kl < KSW; ++kl)
    for (int r = 0; r < 4; ++r)
      for (int hh = 0; hh < 2; ++hh) {
        const int ch = 16 * mc + g + 8 * (r & 1);
        const int tok = 16 * (kt0 + kl) + 2 * t + 8 * (r >> 1) + hh;
        const int pos = VB == 2 ? 2 * pair_2bit(kl, r) + 16 * hh : 4 * nibble_4bit(r) + 16 * hh;
        acc |= code_exact(bf2f(sV[swz(tok, ch)]), vq[tok * kVGroups + j].m,
                          vstep[tok * kVGroups + j], top) << pos;
      }
  return acc;
}

// Key codes straight into fragment-order words (frag_layout.h).  A word of
// (tile mt, k-step pair or k-step, lane g,t) holds tokens g, g+8 of the tile
// and channels 2t, 2t+1, 2t+8, 2t+9 of its k-step(s); each register's pair of
// adjacent channels is one 32-bit read of the staged tile.  A thread's words
// share their lane and k-steps (only the tile differs), so the channel
// parameters and the swizzled column offsets are set up once.
template <int KB>
__device__ __forceinline__ void pack_key_words(const uint16_t* sK, const GroupQ* kq,
                                               const float* kstep, uint32_t* dst) {
  constexpr int KSW = KB == 2 ? 2 : 1;   // k-steps per word
  constexpr int NWT = KB == 2 ? 4 : 8;   // words per thread (256 threads)
  const uint32_t* t32 = reinterpret_cast<const uint32_t*>(sK);
  const int tid = threadIdx.x;
  int lane, ks0, mt0, mstep;
  if (KB == 2) {   // word (mt*4 + ks/2)*32 + lane = tid + 256 k
    lane = tid & 31;
    ks0 = 2 * ((tid >> 5) & 3);
    mt0 = tid >> 7;
    mstep = 2;
  } else {         // word ((mt*4 + ks/2)*32 + lane)*2 + ks%2 = tid + 256 k
    lane = (tid >> 1) & 31;
    ks0 = 2 * ((tid >> 6) & 3) + (tid & 1);
    mt0 = 0;
    mstep = 1;
  }
  const int g = lane >> 2, t = lane & 3;
  GroupQ gq[KSW][4];
  int col[KSW][2];   // 32-bit column offset of channels 2t (+8) in rows with t & 7 = g
#pragma unroll
  for (int kl = 0; kl < KSW; ++kl) {
#pragma unroll
    for (int r2 = 0; r2 < 4; ++r2)   // channels 2t, 2t+1, 2t+8, 2t+9
      gq[kl][r2] = kq[16 * (ks0 + kl) + 2 * t + (r2 & 1) + 8 * (r2 >> 1)];
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      const int ch = 16 * (ks0 + kl) + 2 * t + 8 * hb;
      col[kl][hb] = (((ch >> 3) ^ g) << 2) | ((ch & 7) >> 1);
    }
  }
#pragma unroll 1
  for (int k = 0; k < NWT; ++k) {
    const int mt = mt0 + mstep * k;
    const uint32_t* row0 = t32 + (16 * mt + g) * 64;   // token g of the tile (row + 8: token g+8)
    float rmax = 0.0f;
    uint32_t acc = 0;
#pragma unroll
    for (int kl = 0; kl < KSW; ++kl)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t xw = row0[8 * 64 * (r & 1) + col[kl][r >> 1]];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float x = hh ? bf_hi(xw) : bf_lo(xw);
          const int pos = KB == 2 ? 2 * pair_2bit(kl, r) + 16 * hh : 4 * nibble_4bit(r) + 16 * hh;
          acc |= code_fast(x, gq[kl][2 * (r >> 1) + hh], rmax) << pos;
        }
      }
    if (!(rmax < kTieMargin)) acc = key_word_exact<KB>(t32, kq, kstep, mt, ks0, g, t);   // rare
    dst[tid + 256 * k] = acc;
  }
}

// Value codes straight into fragment-order words: thread (channel tile mc,
// lane g,t) builds the words of all the group's token k-steps (2-bit: 4
// words, k-step pairs; 4-bit: 8) and stores them as 16-byte vectors.  A word
// holds channels g, g+8 of the tile and tokens 2t, 2t+1, 2t+8, 2t+9 of its
// k-step(s); parameters per (token, 32-channel group).
template <int VB>
__device__ __forceinline__ void pack_value_words(const uint16_t* sV, const GroupQ* vq,
                                                 const float* vstep, uint32_t* dst) {
  constexpr int KSW = VB == 2 ? 2 : 1;
  constexpr int NW = VB == 2 ? 4 : 8;   // words per (mc, lane)
  const int mc = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3, j = mc >> 1;
  uint32_t* out4 = dst + (mc * (NW / 4)) * 128 + lane * 4;   // word (mc, lane, wi)
#pragma unroll 1
  for (int wi = 0; wi < NW; ++wi) {
    float rmax = 0.0f;
    uint32_t acc = 0;
    float xs[KSW][4][2];
#pragma unroll
    for (int kl = 0; kl < KSW; ++kl)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kt = KSW * wi + kl;
          const int ch = 16 * mc + g + 8 * (r & 1);
          const int tok = 16 * kt + 2 * t + 8 * (r >> 1) + hh;
          xs[kl][r][hh] = bf2f(sV[swz(tok, ch)]);
        }
#pragma unroll
    for (int kl = 0; kl < KSW; ++kl)
#pragma unroll
      for (int r2 = 0; r2 < 4; ++r2) {   // tokens 2t, 2t+1, 2t+8, 2t+9
        const int tok = 16 * (KSW * wi + kl) + 2 * t + (r2 & 1) + 8 * (r2 >> 1);
        const GroupQ gq = vq[tok * kVGroups + j];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {   // the two registers holding this token
          const int r = 2 * (r2 >> 1) + rr, hh = r2 & 1;
          const int pos = VB == 2 ? 2 * pair_2bit(kl, r) + 16 * hh : 4 * nibble_4bit(r) + 16 * hh;
          acc |= code_fast(xs[kl][r][hh], gq, rmax) << pos;
        }
      }
    if (!(rmax < kTieMargin)) acc = value_word_exact<VB>(sV, vq, vstep, mc, KSW * wi, g, t);   // rare
    // word index of (mc, lane, wi): 2-bit (mc*32 + lane)*4 + wi; 4-bit
    // ((mc*2 + wi/4)*32 + lane)*4 + wi%4
    out4[(wi >> 2) * 128 + (wi & 3)] = acc;
  }
}

__device__ __forceinline__ uint8_t* group_record(const QuantArgs& a) {
  return a.records + (static_cast<long long>(blockIdx.y) * a.max_groups + a.first_group +
                      blockIdx.x) * a.rec_bytes;
}

// Dynamic shared memory of a quantize block: the staged tile (32 KB), then
// the parameter area (kParamBytes): values use vq [512] and vstep [512];
// keys use kq [128], kstep [128], a 2 KB reduction buffer and (mixed keys)
// the rank keys and tiers; mixed key blocks add their virtual codes after.
constexpr int kTileBytes = kKG * kD * 2;
constexpr int kParamBytes = kKG * kVGroups * (8 + 4);   // 6 KB, the larger of the two uses

// Value half of a group (block z = 1 of every quantize launch).
template <int VB>
__device__ __forceinline__ void value_part(const QuantArgs& a, uint8_t* smem) {
  uint16_t* sV = reinterpret_cast<uint16_t*>(smem);
  GroupQ* vq = reinterpret_cast<GroupQ*>(smem + kTileBytes);
  float* vstep = reinterpret_cast<float*>(smem + kTileBytes + kKG * kVGroups * 8);
  load_tile(a, a.src.v, sV);
  __syncthreads();
  uint8_t* rec = group_record(a);
  const unsigned flags = value_groups<VB>(a, sV, vq, vstep, rec);
  __syncthreads();
  pack_value_words<VB>(sV, vq, vstep, reinterpret_cast<uint32_t*>(rec + a.lay.v_codes));
  if (flags) atomicOr(a.status, flags);
}

// Uniform keys and values of one 128-token group: block (group, unit, z),
// z = 0 the keys, z = 1 the values, each from its own 32 KB staged tile.
template <int KB, int VB>
__global__ void __launch_bounds__(256) quantize_uniform_kernel(QuantArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  if (blockIdx.z) {
    value_part<VB>(a, smem);
    return;
  }
  uint16_t* sT = reinterpret_cast<uint16_t*>(smem);
  GroupQ* kq = reinterpret_cast<GroupQ*>(smem + kTileBytes);
  float* kstep = reinterpret_cast<float*>(smem + kTileBytes + kD * 8);
  uint32_t* sRed = reinterpret_cast<uint32_t*>(smem + kTileBytes + kD * 12);
  load_tile(a, a.src.k, sT);
  __syncthreads();
  uint8_t* rec = group_record(a);
  unsigned flags = 0;
  float lo, hi;
  bool bad;
  key_ranges(sT, sRed, lo, hi, bad);
  if (threadIdx.x < kD) {
    const int d = threadIdx.x;
    const Params p = group_params(lo, hi, (1 << KB) - 1, bad);
    kq[d] = make_q(p);
    kstep[d] = p.step;
    reinterpret_cast<float*>(rec + a.lay.k_scale)[d] = p.step;
    reinterpret_cast<uint16_t*>(rec + a.lay.k_min)[d] = f2bf_bits(p.m);
    flags = p.flags;
  }
  __syncthreads();
  pack_key_words<KB>(sT, kq, kstep, reinterpret_cast<uint32_t*>(rec + a.lay.k_codes));
  if (flags) atomicOr(a.status, flags);
}

// Mixed keys (MixKVQ KeyQuant): per channel S_d = fl32(fl32(M - m)/3) over
// the tile, A_d = fl32(I_d * S_d), with I_d given or taken from the online
// window (fl32(sum |q| / count)).  Channels are ranked by A (descending,
// channel ascending on ties).  Rank tiers: the first n_bf16 BF16, the next
// n_uint4 UINT4, the rest UINT2.  Threshold tiers: the channels with
// A > tau_bf16 lead the ranking, so the first min(#{A > tau_bf16}, n_bf16)
// are BF16; of the rest, those with A > tau_uint4 (again a prefix) are
// UINT4 up to n_uint4; the others UINT2 (channels over a capacity drop one
// tier, smallest A first).  The counts go to the record's header.  Storage
// order BF16, UINT4, UINT2 channels, each ascending (the permutation).  The
// BF16 tier is stored raw, channel-major and piece-swizzled; the UINT4 and
// UINT2 codes become 2-bit virtual channels (kvq_internal.h), staged as
// bytes cKv[tok][v] and packed in the key fragment order.
template <int VB>
__global__ void __launch_bounds__(256) quantize_mixed_kernel(QuantArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const RecLayout& L = a.lay;
  const int kvs = 32 * L.kw2;   // staged virtual channels per token
  if (blockIdx.z) {
    value_part<VB>(a, smem);
    return;
  }
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem);
  uint32_t* sRed = reinterpret_cast<uint32_t*>(smem + kTileBytes);             // 2 KB
  uint32_t* sKey = reinterpret_cast<uint32_t*>(smem + kTileBytes + 2048);     // 512 B
  uint8_t* sTier = smem + kTileBytes + 2048 + 512;                            // 128 B
  float* sA = reinterpret_cast<float*>(smem + kTileBytes + 2048 + 512 + 128);  // 512 B
  uint8_t* cKv = smem + kTileBytes + kParamBytes;
  load_tile(a, a.src.k, sK);
  // virtual channels past this group's count stay zero
  for (int i = threadIdx.x; i < kKG * kvs / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(cKv)[i] = 0u;
  __syncthreads();

  const int u = blockIdx.y;
  uint8_t* rec = group_record(a);
  unsigned flags = 0;
  float lo, hi;
  bool bad;
  key_ranges(sK, sRed, lo, hi, bad);
  if (threadIdx.x < kD) {
    const int d = threadIdx.x;
    float S = 0.0f;
    if (!bad) S = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    const long long ud = static_cast<long long>(u) * kD + d;
    const float I = a.importance ? a.importance[ud] : __fdiv_rn(a.qacc[ud], a.q_count);
    if (!isfinite(I)) flags |= KVQ_FLAG_NONFINITE;
    if (bad) flags |= KVQ_FLAG_NONFINITE;
    else if (!isfinite(S)) flags |= KVQ_FLAG_RANGE;
    const float A = __fmul_rn(I, S);
    // Rank by a total-order key (NaN, only possible on a flagged group,
    // sorts last) so ranks are always a permutation and every slot stays
    // inside its tier's region.
    const uint32_t key = isnan(A) ? 0u : fkey(A);
    sKey[d] = key;
    sA[d] = A;
    asm volatile("bar.sync 1, 128;");
    // rank, and how many channels pass each threshold (NaN passes none)
    int rank = 0, above_b = 0, above_4 = 0;
    for (int e = 0; e < kD; ++e) {
      const uint32_t ke = sKey[e];
      rank += (ke > key || (ke == key && e < d)) ? 1 : 0;
      if (L.thresh) {
        const float Ae = sA[e];
        above_b += Ae > a.tau_bf16 ? 1 : 0;
        above_4 += Ae > a.tau_uint4 ? 1 : 0;
      }
    }
    int nb = L.nb, n4 = L.n4;
    if (L.thresh) {
      nb = min(above_b, L.nb);
      n4 = max(0, min(above_4 - nb, L.n4));
    }
    const int tier = rank < nb ? KVQ_TIER_BF16
                     : rank < nb + n4 ? KVQ_TIER_UINT4
                                      : KVQ_TIER_UINT2;
    sTier[d] = static_cast<uint8_t>(tier);
    if (d == 0) {
      rec[L.hdr] = static_cast<uint8_t>(nb);
      rec[L.hdr + 1] = static_cast<uint8_t>(n4);
    }
    asm volatile("bar.sync 1, 128;");
    int slot = tier == KVQ_TIER_BF16 ? 0 : tier == KVQ_TIER_UINT4 ? nb : nb + n4;
    for (int e = 0; e < d; ++e) slot += (sTier[e] == tier) ? 1 : 0;
    rec[L.perm + slot] = static_cast<uint8_t>(d);
    if (tier == KVQ_TIER_BF16) {
      uint16_t* raw = reinterpret_cast<uint16_t*>(rec + L.raw) + slot * kKG;
      for (int t = 0; t < kKG; ++t) raw[(((t >> 3) ^ (slot & 7)) << 3) | (t & 7)] = sK[swz(t, d)];
    } else {
      const int bits = tier == KVQ_TIER_UINT4 ? 4 : 2;
      const int top = (1 << bits) - 1;
      const Params p = group_params(lo, hi, top, bad);
      flags |= p.flags;
      const int j = slot - nb;   // index among the quantized channels
      reinterpret_cast<float*>(rec + L.s4)[j] = p.step;
      reinterpret_cast<uint16_t*>(rec + L.m4)[j] = f2bf_bits(p.m);
      if (bits == 4) {
        for (int t = 0; t < kKG; ++t) {
          const uint32_t c = code_exact(bf2f(sK[swz(t, d)]), p.m, p.step, top);
          cKv[t * kvs + j] = static_cast<uint8_t>(c & 3u);
          cKv[t * kvs + n4 + j] = static_cast<uint8_t>(c >> 2);
        }
      } else {
        for (int t = 0; t < kKG; ++t)
          cKv[t * kvs + n4 + j] = static_cast<uint8_t>(code_exact(bf2f(sK[swz(t, d)]), p.m, p.step, top));
      }
    }
  }
  __syncthreads();
  {
    uint32_t* dst = reinterpret_cast<uint32_t*>(rec + L.kc);
    const int words = 8 * L.kw2 * 32;
    for (int w = threadIdx.x; w < words; w += blockDim.x) {
      uint32_t acc = 0;
#pragma unroll
      for (int s2 = 0; s2 < 16; ++s2) {
        int tok, v;
        mixed_word_code(w, s2, L.kw2, tok, v);
        acc |= static_cast<uint32_t>(cKv[tok * kvs + v]) << (2 * s2);
      }
      dst[w] = acc;
    }
  }
  if (flags) atomicOr(a.status, flags);
}

__global__ void append_kernel(const uint4* __restrict__ k_new,
                              const uint4* __restrict__ v_new, uint4* dst_k,
                              uint4* dst_v, int cap, int slot) {
  // one (b, kv head) per block; 16 x 16 bytes per row of D bf16
  constexpr int kRow = kD * 2 / 16;
  const int u = blockIdx.x;
  const int i = threadIdx.x;
  const long long dst = (static_cast<long long>(u) * cap + slot) * kRow;
  if (i < kRow)
    dst_k[dst + i] = __ldg(k_new + static_cast<long long>(u) * kRow + i);
  else if (i < 2 * kRow)
    dst_v[dst + i - kRow] = __ldg(v_new + static_cast<long long>(u) * kRow + i - kRow);
}

// Copy one section (bytes at offset off of every group record) of records
// [u][g0 .. g0+n) into dst [u][n][bytes].
__global__ void gather_section_kernel(const uint8_t* __restrict__ records,
                                      long long rec_bytes, int max_groups,
                                      int off, int bytes, uint8_t* dst, int n) {
  const int g = blockIdx.x;
  const int u = blockIdx.y;
  const uint8_t* src = records + (static_cast<long long>(u) * max_groups + g) * rec_bytes + off;
  uint8_t* out = dst + (static_cast<long long>(u) * n + g) * bytes;
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(out) |
                     static_cast<uintptr_t>(bytes)) & 15) == 0;
  if (vec) {
    for (int i = threadIdx.x; i < bytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(src)[i];
  } else {
    for (int i = threadIdx.x; i < bytes; i += blockDim.x) out[i] = src[i];
  }
}

// Canonical export of the fragment-order codes of records [u][0..n).
// Keys: dst [u][n][D][128*bits/8], channel d's codes LSB first along tokens.
// Values: dst [u][n*128][D*bits/8], token t's codes LSB first along channels.
__global__ void export_codes_kernel(const uint8_t* __restrict__ records, long long rec_bytes,
                                    int max_groups, int off, int bits, bool key,
                                    uint8_t* dst, int n) {
  const int g = blockIdx.x;
  const int u = blockIdx.y;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(
      records + (static_cast<long long>(u) * max_groups + g) * rec_bytes + off);
  const int x = threadIdx.x;  // channel (keys) or token (values)
  const int per = 8 / bits, row_bytes = 128 * bits / 8;
  const uint32_t mask = (1u << bits) - 1u;
  uint8_t* out = dst + ((static_cast<long long>(u) * n + g) * 128 + x) * row_bytes;
  for (int i = 0; i < row_bytes; ++i) {
    uint32_t byte = 0;
    for (int e = 0; e < per; ++e) {
      const int y = i * per + e;  // token (keys) or channel (values)
      const CodePos p = key ? key_code_pos(y, x, bits) : value_code_pos(x, y, bits);
      byte |= ((words[p.word] >> p.bit) & mask) << (bits * e);
    }
    out[i] = static_cast<uint8_t>(byte);
  }
}

// Canonical export of mixed key groups [u][0..n) at the record capacities
// (cb = n_bf16, c4 = n_uint4 of the config, c2 = n2cap; the group's own
// counts nb, n4 go to counts[..][0..1] if counts is not NULL, n2 = D - nb -
// n4): perm [..][D], raw [..][cb][128] in token order, UINT4 codes
// [..][c4][64] with origins and steps [..][c4], UINT2 codes [..][c2][32]
// with origins and steps [..][c2], codes LSB first along tokens, rebuilt
// from the virtual 2-bit channels; entries past a group's count are zero.
__global__ void export_mixed_kernel(const uint8_t* __restrict__ records, long long rec_bytes,
                                    int max_groups, RecLayout L, uint8_t* counts,
                                    uint8_t* perm, uint16_t* raw, uint8_t* c4, uint16_t* m4,
                                    float* s4, uint8_t* c2, uint16_t* m2, float* s2, int n) {
  const int g = blockIdx.x;
  const int u = blockIdx.y;
  const uint8_t* rec = records + (static_cast<long long>(u) * max_groups + g) * rec_bytes;
  const long long ug = static_cast<long long>(u) * n + g;
  const int nb = rec[L.hdr], n4 = rec[L.hdr + 1], n2 = kD - nb - n4;
  if (counts && threadIdx.x == 0) {
    counts[ug * 2] = static_cast<uint8_t>(nb);
    counts[ug * 2 + 1] = static_cast<uint8_t>(n4);
  }
  if (threadIdx.x < kD) perm[ug * kD + threadIdx.x] = rec[L.perm + threadIdx.x];
  const uint16_t* rraw = reinterpret_cast<const uint16_t*>(rec + L.raw);
  for (int e = threadIdx.x; e < L.nb * kKG; e += blockDim.x) {
    const int i = e >> 7, t = e & 127;
    raw[ug * L.nb * kKG + e] =
        i < nb ? rraw[i * kKG + ((((t >> 3) ^ (i & 7)) << 3) | (t & 7))] : 0;
  }
  const uint32_t* words = reinterpret_cast<const uint32_t*>(rec + L.kc);
  const float* steps = reinterpret_cast<const float*>(rec + L.s4);
  const uint16_t* mins = reinterpret_cast<const uint16_t*>(rec + L.m4);
  auto code2 = [&](int tok, int v) {
    const CodePos p = mixed_code_pos(tok, v, L.kw2);
    return (words[p.word] >> p.bit) & 3u;
  };
  const int j = threadIdx.x;
  if (j < L.n4) {   // UINT4 slot j: lo plane v = j, hi plane v = n4 + j
    uint8_t* out = c4 + (ug * L.n4 + j) * (kKG / 2);
    for (int i = 0; i < kKG / 2; ++i) {
      uint32_t byte = 0;
      for (int e = 0; e < 2 && j < n4; ++e) {
        const int t = 2 * i + e;
        byte |= (code2(t, j) | (code2(t, n4 + j) << 2)) << (4 * e);
      }
      out[i] = static_cast<uint8_t>(byte);
    }
    m4[ug * L.n4 + j] = j < n4 ? mins[j] : 0;
    s4[ug * L.n4 + j] = j < n4 ? steps[j] : 0.0f;
  }
  if (j < L.n2cap) {   // UINT2 slot j: virtual channel 2 n4 + j
    uint8_t* out = c2 + (ug * L.n2cap + j) * (kKG / 4);
    for (int i = 0; i < kKG / 4; ++i) {
      uint32_t byte = 0;
      for (int e = 0; e < 4 && j < n2; ++e) byte |= code2(4 * i + e, 2 * n4 + j) << (2 * e);
      out[i] = static_cast<uint8_t>(byte);
    }
    m2[ug * L.n2cap + j] = j < n2 ? mins[n4 + j] : 0;
    s2[ug * L.n2cap + j] = j < n2 ? steps[n4 + j] : 0.0f;
  }
}

cudaError_t export_codes(const kvq_cache* c, int off, int bits, bool key, void* dst,
                         cudaStream_t s) {
  const int n = c->t_q / kKG;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  if (n == 0) return cudaSuccess;
  export_codes_kernel<<<dim3(n, units), 128, 0, s>>>(c->records, c->lay.bytes, c->max_groups,
                                                     off, bits, key,
                                                     static_cast<uint8_t*>(dst), n);
  return cudaGetLastError();
}

cudaError_t gather(const kvq_cache* c, int off, int bytes, void* dst,
                   cudaStream_t s) {
  const int n = c->t_q / kKG;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  if (n == 0 || bytes == 0) return cudaSuccess;
  gather_section_kernel<<<dim3(n, units), 128, 0, s>>>(
      c->records, c->lay.bytes, c->max_groups, off, bytes,
      static_cast<uint8_t*>(dst), n);
  return cudaGetLastError();
}

constexpr int kQuantSmem = kTileBytes + kParamBytes;  // 38 KB


}  // namespace

cudaError_t launch_append(const kvq_cache* c, const kvq_bf16* k_new, const kvq_bf16* v_new,
                          kvq_bf16* dst_k, kvq_bf16* dst_v, int cap, int slot, cudaStream_t s) {
  const int units = c->cfg.batch * c->cfg.kv_heads;
  // same shared-memory split as the decode grid that usually follows
  static const cudaError_t carve = cudaFuncSetAttribute(
      append_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
      cudaSharedmemCarveoutMaxShared);
  if (carve != cudaSuccess) return carve;
  append_kernel<<<units, 32, 0, s>>>(reinterpret_cast<const uint4*>(k_new),
                                     reinterpret_cast<const uint4*>(v_new),
                                     reinterpret_cast<uint4*>(dst_k),
                                     reinterpret_cast<uint4*>(dst_v), cap, slot);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const kvq_cache* c, QuantSrc src, int n_groups,
                            int first_group, const float* importance,
                            cudaStream_t s) {
  if (n_groups == 0) return cudaSuccess;
  QuantArgs a;
  a.src = src;
  a.records = c->records;
  a.rec_bytes = c->lay.bytes;
  a.max_groups = c->max_groups;
  a.first_group = first_group;
  a.lay = c->lay;
  a.importance = importance;
  a.qacc = c->qacc;
  a.q_count = static_cast<float>(c->q_rep * c->q_steps);
  // +0.0f turns a threshold of -0 into +0, so A = +0 is not above it
  a.tau_bf16 = c->cfg.tau_bf16 + 0.0f;
  a.tau_uint4 = c->cfg.tau_uint4 + 0.0f;
  a.status = c->status;
  const dim3 grid(n_groups, c->cfg.batch * c->cfg.kv_heads, 2);   // z: keys, values
  const int kb = c->cfg.k_bits, vb = c->cfg.v_bits;
  cudaError_t e = cudaSuccess;
#define KVQ_LAUNCH(KERNEL, SMEM)                             \
  do {                                                       \
    static SmemOptIn opt_in;                                 \
    e = opt_in.ensure(KERNEL);                               \
    if (e != cudaSuccess) return e;                          \
    KERNEL<<<grid, 256, SMEM, s>>>(a);                       \
  } while (0)
  if (c->cfg.k_mode == KVQ_K_MIXED) {
    const int smem = kTileBytes + kParamBytes + kKG * 32 * c->lay.kw2;   // + virtual codes
    if (vb == 2) KVQ_LAUNCH(quantize_mixed_kernel<2>, smem);
    else KVQ_LAUNCH(quantize_mixed_kernel<4>, smem);
  } else if (kb == 2 && vb == 2) {
    KVQ_LAUNCH((quantize_uniform_kernel<2, 2>), kQuantSmem);
  } else if (kb == 2 && vb == 4) {
    KVQ_LAUNCH((quantize_uniform_kernel<2, 4>), kQuantSmem);
  } else if (kb == 4 && vb == 2) {
    KVQ_LAUNCH((quantize_uniform_kernel<4, 2>), kQuantSmem);
  } else {
    KVQ_LAUNCH((quantize_uniform_kernel<4, 4>), kQuantSmem);
  }
#undef KVQ_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_copy_tokens(const kvq_bf16* k, const kvq_bf16* v, int L, int first, int count,
                               kvq_bf16* dst_k, kvq_bf16* dst_v, int cap, int units,
                               cudaStream_t s) {
  if (count == 0) return cudaSuccess;
  const size_t row = static_cast<size_t>(kD) * sizeof(kvq_bf16);
  cudaError_t e = cudaMemcpy2DAsync(dst_k, cap * row, k + static_cast<size_t>(first) * kD,
                                    static_cast<size_t>(L) * row, count * row, units,
                                    cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaMemcpy2DAsync(dst_v, cap * row, v + static_cast<size_t>(first) * kD,
                           static_cast<size_t>(L) * row, count * row, units,
                           cudaMemcpyDeviceToDevice, s);
}

cudaError_t launch_export_k_uniform(const kvq_cache* c, uint8_t* codes,
                                    kvq_bf16* kmin, float* kscale,
                                    cudaStream_t s) {
  const RecLayout& L = c->lay;
  cudaError_t e = export_codes(c, L.k_codes, L.kb, true, codes, s);
  if (e == cudaSuccess) e = gather(c, L.k_min, kD * 2, kmin, s);
  if (e == cudaSuccess) e = gather(c, L.k_scale, kD * 4, kscale, s);
  return e;
}

cudaError_t launch_export_v(const kvq_cache* c, uint8_t* codes, kvq_bf16* vmin,
                            float* vscale, cudaStream_t s) {
  const RecLayout& L = c->lay;
  cudaError_t e = export_codes(c, L.v_codes, L.vb, false, codes, s);
  if (e == cudaSuccess) e = gather(c, L.v_min, kKG * kVGroups * 2, vmin, s);
  if (e == cudaSuccess) e = gather(c, L.v_scale, kKG * kVGroups * 4, vscale, s);
  return e;
}

cudaError_t launch_export_k_mixed(const kvq_cache* c, uint8_t* counts, uint8_t* perm,
                                  kvq_bf16* raw, uint8_t* c4, kvq_bf16* m4,
                                  float* s4, uint8_t* c2, kvq_bf16* m2,
                                  float* s2, cudaStream_t s) {
  const int n = c->t_q / kKG;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  if (n == 0) return cudaSuccess;
  export_mixed_kernel<<<dim3(n, units), 128, 0, s>>>(
      c->records, c->lay.bytes, c->max_groups, c->lay, counts, perm,
      reinterpret_cast<uint16_t*>(raw), c4, reinterpret_cast<uint16_t*>(m4), s4, c2,
      reinterpret_cast<uint16_t*>(m2), s2, n);
  return cudaGetLastError();
}

}  // namespace kvq
