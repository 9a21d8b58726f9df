// Residual append, group quantization (flush and prefill, uniform and mixed
// keys) and canonical export of the packed cache.
//
// Quantizer ("KIVI: KV cache axes" §2; MixKVQ "KV cache quantization
// principle"; PN-Mix Eq. 2): per group m = min, M = max,
//   step = fl32(fl32(M - m) / (2^b - 1)),  c = clip(RNE(fl32(fl32(x - m) / step)))
// with IEEE fp32 subtraction and division (__fsub_rn / __fdiv_rn), codes
// rounded half-to-even, and a constant group (M == m) stored as step 0,
// codes 0, origin m.  Every pass reaches these codes bit for bit without a
// division per element (code_bits and near_bits below; KIVI's bf16 rule in
// kivi_bits); only flagged groups and steps below 2^-100 divide, out of
// line.  Groups: Key per channel over the 128 tokens of a tile,
// Value per token over 32 consecutive channels (KIVI §3).  The uniform and
// KIVI-prefill passes build whole words of the tensor-core fragment order
// of frag_layout.h in registers; the mixed and PN-Mix passes stage codes as
// bytes and pack them word by word; kvq_export_* converts back to the
// canonical LSB-first layout.
#include <cuda_bf16.h>
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
  const uint8_t* perm;      // PN-Mix: [units][D] stored position -> channel
  int kivi_valid;           // KIVI prefill: value tokens quantized, from the first record on
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

// Exact code of one element, IEEE quotient (the definition): the rare path.
__device__ __forceinline__ uint32_t code_exact(float x, float m, float step, int top) {
  if (step == 0.0f) return 0u;
  const float q = __fdiv_rn(__fsub_rn(x, m), step);
  return static_cast<uint32_t>(fminf(fmaxf(rintf(q), 0.0f), static_cast<float>(top)));
}

// code_exact out of line, for loops whose fast path is inlined many times
// and whose exact path is rare (flagged or tiny-step groups)
__device__ __noinline__ uint32_t code_exact_rare(float x, float m, float step, int top) {
  return code_exact(x, m, step, top);
}

// ---- bf16x2 helpers
// Elementwise min / max of two bf16 pairs; a NaN in either operand gives NaN.
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.NaN.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t swap_halves(uint32_t a) { return __byte_perm(a, 0, 0x1032); }

// d = RN(x - m) for the bf16 x in the low (high) half of w, given nm = -m:
// one mixed-precision FMA x * 1 + nm (x * 1 is exact, so this is fl32(x - m)).
__device__ __forceinline__ float sub_lo(uint32_t w, float nm) {
  float d;
  asm("{\n .reg .b16 l, h, one;\n mov.b32 {l, h}, %1;\n mov.b16 one, 0x3F80;\n"
      " fma.rn.f32.bf16 %0, l, one, %2;\n}\n" : "=f"(d) : "r"(w), "f"(nm));
  return d;
}
__device__ __forceinline__ float sub_hi(uint32_t w, float nm) {
  float d;
  asm("{\n .reg .b16 l, h, one;\n mov.b32 {l, h}, %1;\n mov.b16 one, 0x3F80;\n"
      " fma.rn.f32.bf16 %0, h, one, %2;\n}\n" : "=f"(d) : "r"(w), "f"(nm));
  return d;
}

// The code of d = fl32(x - m) in the fast form.  y = RN(d * r + 32) with r =
// RN(1/step) lies in [32, 64) (codes <= 15), where the fp32 spacing is
// 2^-18, so the bits of y hold (d/step) with 18 fraction bits.  |y - 32 -
// d/step| <= 2^-19 + 16 * 2^-24 and |RN(d/step) - d/step| <= 2^-21, so y -
// 32 is within 1.2 units of 2^-18 of the IEEE quotient RN(d/step).  Adding
// 1/2 + 2 units and keeping the integer part gives RNE(RN(d/step)) unless
// the fraction lies within 2 units of 1/2, below 1/2 or 5 above ("near"):
// then the element takes the exact path.  The addition rides in the FMA:
// 1/2 + 2^-17 is an even multiple of the spacing, so RN(d * r + 32 + 1/2 +
// 2^-17) is y plus 1/2 + 2 units exactly (ties included) and stays below
// 64.  Returns those bits v: the code is (v >> 18) & (2^b - 1).
constexpr float kCodeMagic = 32.500007629394531f;   // 32 + 1/2 + 2^-17
constexpr uint32_t kHalfPlus = 0x20002u;    // 1/2 + 2 units of 2^-18
constexpr uint32_t kNearMask = 0x3FFF8u;    // fraction within [1/2 - 2, 1/2 + 5] units
__device__ __forceinline__ uint32_t code_bits(float d, float r) {
  return __float_as_uint(fmaf(d, r, kCodeMagic));
}
__device__ __forceinline__ bool is_near(uint32_t v) { return (v & kNearMask) == 0u; }
// A near element: its quotient z = d/step lies close to h = n + 1/2, n =
// floor(y - 32), so its code is n or n + 1, decided by RNE(RN(z)).  With
// rem = d - h * step, exact in one FMA (the operands nearly cancel: h has at
// most 5 significant bits and |rem| < 2^-14 d), RN(z) = h exactly when
// -step * ulp-(h)/2 <= rem <= step * ulp(h)/2 (h has an even significand, so
// it wins both ties), and then the code is RNE(h) = n + (n & 1); above that
// band RN(z) > h (code n + 1), below it RN(z) < h (code n).  Needs step >=
// 2^-100 (no underflow in the bounds); smaller steps take the exact tile
// path.  Returns the code in code_bits' position.  Out of line: elements
// come here rarely (ties of bf16 data, about one in 2^15 otherwise), and
// an inline copy at each of a thread's 64 unrolled elements would grow the
// code passes past the instruction cache.
__device__ __noinline__ uint32_t near_bits(uint32_t v, float d, float step, uint32_t top) {
  const uint32_t n = ((v - kHalfPlus) >> 18) & 15u;
  const float h = static_cast<float>(n) + 0.5f;
  const float rem = fmaf(-h, step, d);
  // step * 2^(e - 24), e = floor(log2 h): the distance from h to its upper
  // neighbour, halved (and to its lower one, except for h = 1/2)
  const uint32_t e = __float_as_uint(h) >> 23;   // biased exponent of h
  const float up = step * __uint_as_float((e - 24u) << 23);
  const float dn = n == 0u ? 0.5f * up : up;
  const uint32_t c = rem > up ? n + 1u : rem < -dn ? n : n + (n & 1u);
  return min(c, top) << 18;
}
// The code in v (bits 18..) moved to bit `pos` of a word, masked.
template <int BITS>
__device__ __forceinline__ uint32_t place(uint32_t v, int pos) {
  constexpr uint32_t m = (1u << BITS) - 1u;
  return (pos >= 18 ? v << (pos - 18) : v >> (18 - pos)) & (m << pos);
}

// Range of a group from its bf16 min / max bits (NaN-propagating), with
// the pages' order of signed zeros (-0 below +0): a zero minimum is -0 iff
// the group holds a -0 (looked up by the caller only then).
__device__ __forceinline__ bool nonfinite_bits(uint32_t b) { return (b & 0x7F80u) == 0x7F80u; }

// Per-group parameters of the code pass: -m and RN(1/step) (0 for a constant
// or non-finite group); the step itself is kept apart for the exact path.
struct GroupQ {
  float nm, rcp;
};

// ---- KIVI streaming variant ("KIVI: KV cache axes" §7): origin and step in
// bf16, computed in bf16 (every operation an fp32 operation rounded to
// bf16), code = clip(RNE(bf16(bf16(x - m) / step)), 0, top).
__device__ __forceinline__ float bfr(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
struct KiviGroupP {
  float m, step;
  unsigned flags;
};
__device__ __forceinline__ KiviGroupP kivi_group(float lo, float hi, bool nonfinite, int top) {
  KiviGroupP p{lo, 0.0f, nonfinite ? static_cast<unsigned>(KVQ_FLAG_NONFINITE) : 0u};
  if (nonfinite || hi == lo) return p;
  const float step = bfr(__fdiv_rn(bfr(__fsub_rn(hi, lo)), static_cast<float>(top)));
  if (!(step > 0.0f) || !isfinite(step)) p.flags |= KVQ_FLAG_RANGE;
  p.step = step;
  return p;
}
// The (-m, rcp) pair the code pass uses: rcp = RN(1/step); 0 for a constant
// or flagged group (every code 0: with -m = 0 the product is 0, or NaN for a
// non-finite x, which the clip sends to 0); -1 for a step below 2^-100, which
// sends every element of the group to the exact quotient.
__device__ __forceinline__ GroupQ kivi_q(const KiviGroupP& p) {
  if (p.flags || p.step == 0.0f) return {0.0f, 0.0f};
  return {-p.m, p.step < 0x1p-100f ? -1.0f : __frcp_rn(p.step)};
}
// The rare path of kivi_bits: bf16(RN(diff / step)) with the step read
// back from the record (bf16).  Out of line, as near_bits: an inline IEEE
// division at each of a thread's unrolled elements overflows the
// instruction cache.
__device__ __noinline__ float kivi_exact(float diff, const uint16_t* step_bf16) {
  return bfr(__fdiv_rn(diff, bf2f(*step_bf16)));
}
// The code of d32 = fl32(x - m) in code_bits' position.  diff = bf16(d32);
// z = RN(diff * rcp) lies within 2.5 fp32 ulps of RN(diff / step), so both
// round to the same bf16 value unless a bf16 rounding boundary (an fp32 value
// whose low 16 bits are 0x8000) lies within 3 ulps of z; such elements (and
// tiny-step groups) take the IEEE quotient.  The code is clip(RNE(y), 0,
// top): the clip first (the same result: RNE is monotonic and the bounds
// are integers; a NaN y clips to 0 either way), then RNE by adding 1.5 *
// 2^23, which rounds any value in [0, top] to the nearest integer, ties to
// even, into the low bits.
template <int BITS>
__device__ __forceinline__ uint32_t kivi_bits(float d32, float rcp, const uint16_t* step_bf16) {
  constexpr float top = static_cast<float>((1 << BITS) - 1);
  const float diff = bfr(d32);
  const float z = __fmul_rn(diff, rcp);
  float y;
  if ((__float_as_uint(z) & 0xFFFFu) - 0x7FFDu <= 6u || rcp < 0.0f)   // rare
    y = kivi_exact(diff, step_bf16);
  else
    y = bfr(z);
  const float c = __fadd_rn(fminf(fmaxf(y, 0.0f), top), 12582912.0f);   // 1.5 * 2^23
  return (__float_as_uint(c) & 15u) << 18;
}


// A tile takes the exact path everywhere when a group is non-finite or has
// a step in (0, 2^-100) (the near-element bounds would underflow).
constexpr float kTinyStep = 7.888609052210118e-31f;   // 2^-100
__device__ __forceinline__ GroupQ make_q(const Params& p, bool& exact_tile) {
  const float r = p.step > 0.0f ? __frcp_rn(p.step) : 0.0f;
  if (p.flags) exact_tile = true;
  if (p.step > 0.0f && p.step < kTinyStep) exact_tile = true;
  return {-p.m, r};
}

// ---- Key half: ranges per channel over the tile's 128 tokens.
// Thread (piece o = tid & 15: channels 8o..8o+7, tokens 8s..8s+7 with s =
// tid >> 4) reduces its 8 rows with bf16x2 min/max; lanes o and o + 16 merge
// by a shuffle, the 8 warps through shared memory (sRed: [8][16][8] words).
// Threads 0..127 return channel tid's range (lo with the signed-zero rule).
__device__ __forceinline__ void key_ranges(const uint16_t* sK, uint32_t* sRed, float& lo,
                                           float& hi, bool& bad) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int o = lane & 15, s = tid >> 4;
  const uint4* rows = reinterpret_cast<const uint4*>(sK);
  uint4 w = rows[(8 * s) * 16 + o];   // token 8s: (8s & 7) = 0
  uint32_t mn[4] = {w.x, w.y, w.z, w.w}, mx[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 1; i < 8; ++i) {
    w = rows[(8 * s + i) * 16 + (o ^ i)];
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mn[k] = bmin2(mn[k], ww[k]);
      mx[k] = bmax2(mx[k], ww[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    mn[k] = bmin2(mn[k], __shfl_xor_sync(0xffffffffu, mn[k], 16));
    mx[k] = bmax2(mx[k], __shfl_xor_sync(0xffffffffu, mx[k], 16));
  }
  if (lane < 16) {
    uint4* dst = reinterpret_cast<uint4*>(sRed + (warp * 16 + o) * 8);
    dst[0] = make_uint4(mn[0], mn[1], mn[2], mn[3]);
    dst[1] = make_uint4(mx[0], mx[1], mx[2], mx[3]);
  }
  __syncthreads();
  if (tid < kD) {
    const int d = tid, oo = d >> 3, k = (d & 7) >> 1, sh = 16 * (d & 1);
    uint32_t m2 = sRed[oo * 8 + k], x2 = sRed[oo * 8 + 4 + k];
#pragma unroll
    for (int wv = 1; wv < 8; ++wv) {
      m2 = bmin2(m2, sRed[(wv * 16 + oo) * 8 + k]);
      x2 = bmax2(x2, sRed[(wv * 16 + oo) * 8 + 4 + k]);
    }
    uint32_t lb = (m2 >> sh) & 0xFFFFu;
    const uint32_t hb = (x2 >> sh) & 0xFFFFu;
    bad = nonfinite_bits(lb) || nonfinite_bits(hb);
    if (!bad && (lb & 0x7FFFu) == 0u) {   // a zero minimum: -0 iff the channel holds one
      lb = 0u;
      for (int t = 0; t < kKG; ++t)
        if (sK[swz(t, d)] == 0x8000u) lb = 0x8000u;
    }
    lo = bf2f(static_cast<uint16_t>(lb));
    hi = bf2f(static_cast<uint16_t>(hb));
  }
}

// Key codes straight into fragment-order words (frag_layout.h).  Thread
// (tile mt, row g, word column w) takes tokens 16 mt + g and + 8 and
// channels 32 w .. 32 w + 31: one 16-byte read gives channels 2t, 2t+1 of
// lanes t = 0..3 for one (k-step, half of the k-step, token row), and the
// thread's words are the 4 (2-bit) or 8 (4-bit) consecutive words of lanes
// (g, 0..3), stored as 16-byte vectors.  Lanes 0..7 of a warp are the eight
// rows g, so each quarter warp's reads fall on eight different pieces.
// Exact path of a whole tile (a non-finite group or a step below 2^-100):
// every code from the IEEE quotient; the same words as key_codes.
template <int KB>
__device__ __noinline__ void key_codes_slow(const uint16_t* sK, const GroupQ* kq,
                                            const float* kstep, uint32_t* dst) {
  constexpr int NW = KB == 2 ? 4 : 8;
  constexpr int top = (1 << KB) - 1;
  const int tid = threadIdx.x;
  const int g = tid & 7, w = (tid >> 3) & 3, mt = tid >> 5;
  uint32_t* out = dst + ((mt * 4 + w) * 32 + 4 * g) * (NW / 4);
#pragma unroll 1
  for (int i = 0; i < NW; ++i) {
    const int t = KB == 2 ? i : i >> 1;
    uint32_t acc = 0;
#pragma unroll 1
    for (int e = 0; e < 32 / KB; ++e) {
      // code slot e of word i: (rhi, kl, chi, half) of this thread's elements
      int rhi, kl, chi, half;
      if (KB == 2) {
        half = e >> 3;
        const int P = e & 7;
        rhi = P >> 2;
        kl = (P >> 1) & 1;
        chi = P & 1;
      } else {
        half = e >> 2;
        kl = i & 1;
        rhi = (e >> 1) & 1;
        chi = e & 1;
      }
      const int tok = 16 * mt + g + 8 * rhi;
      const int ch = 32 * w + 16 * kl + 8 * chi + 2 * t + half;
      acc |= code_exact(bf2f(sK[swz(tok, ch)]), -kq[ch].nm, kstep[ch], top) << (KB * e);
    }
    out[i] = acc;
  }
}

// KIVI (f1): the channel parameters are per 32-token sub-group ([4][128]),
// the steps bf16 ([4][128]); a thread's tokens all lie in sub-group mt / 2.
template <int KB, bool KIVI = false>
__device__ __forceinline__ void key_codes(const uint16_t* sK, const GroupQ* kq,
                                          const void* steps, bool exact_tile, uint32_t* dst) {
  constexpr int NW = KB == 2 ? 4 : 8;
  constexpr int top = (1 << KB) - 1;
  const float* kstep = static_cast<const float*>(steps);
  if (!KIVI && exact_tile) {   // block-uniform, rare
    key_codes_slow<KB>(sK, kq, kstep, dst);
    return;
  }
  const int tid = threadIdx.x;
  const int g = tid & 7, w = (tid >> 3) & 3, mt = tid >> 5;
  const uint4* rows = reinterpret_cast<const uint4*>(sK);
  const float4* kq4 = reinterpret_cast<const float4*>(kq) + (KIVI ? (mt >> 1) * (kD / 2) : 0);
  const uint16_t* kst = static_cast<const uint16_t*>(steps) + (KIVI ? (mt >> 1) * kD : 0);
  uint32_t acc[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) acc[i] = 0u;
#pragma unroll
  for (int kl = 0; kl < 2; ++kl)
#pragma unroll
    for (int chi = 0; chi < 2; ++chi) {
      const int p = 4 * w + 2 * kl + chi;   // piece: channels 8p .. 8p + 7
      // (-m, rcp) of channels 8p + e, e = 2t + half
      float4 q4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q4[i] = kq4[4 * p + i];
      const float nm[8] = {q4[0].x, q4[0].z, q4[1].x, q4[1].z, q4[2].x, q4[2].z, q4[3].x, q4[3].z};
      const float rc[8] = {q4[0].y, q4[0].w, q4[1].y, q4[1].w, q4[2].y, q4[2].w, q4[3].y, q4[3].w};
#pragma unroll
      for (int rhi = 0; rhi < 2; ++rhi) {
        const uint4 x4 = rows[(16 * mt + g + 8 * rhi) * 16 + (p ^ g)];
        const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int e = 2 * t + half;
            const float d = half ? sub_hi(xw[t], nm[e]) : sub_lo(xw[t], nm[e]);
            uint32_t v;
            if constexpr (KIVI) {
              v = kivi_bits<KB>(d, rc[e], kst + 8 * p + e);
            } else {
              v = code_bits(d, rc[e]);
              if (is_near(v)) v = near_bits(v, d, kstep[8 * p + e], top);   // rare
            }
            if (KB == 2) acc[t] |= place<2>(v, 2 * (4 * rhi + 2 * kl + chi) + 16 * half);
            else acc[2 * t + kl] |= place<4>(v, 4 * (2 * rhi + chi) + 16 * half);
          }
      }
    }
  // 2-bit: words (mt*4 + w)*32 + 4g + t; 4-bit: ((mt*4 + w)*32 + 4g + t)*2 + kl
  uint4* out = reinterpret_cast<uint4*>(dst + ((mt * 4 + w) * 32 + 4 * g) * (NW / 4));
  out[0] = make_uint4(acc[0], acc[1], acc[2], acc[3]);
  if (NW == 8) out[1] = make_uint4(acc[4 % NW], acc[5 % NW], acc[6 % NW], acc[7 % NW]);
}

// ---- Value half: ranges per (token, 32-channel group).  Thread (token tid
// >> 1, h = tid & 1) takes groups j = 2h, 2h + 1 (h = 1 in the order 3, 2 so
// a quarter warp's 16-byte reads fall on distinct banks).  Writes steps and
// origins to the record and (-m, rcp) to vq[tok * 4 + j], steps to vstep.
template <int VB>
__device__ __forceinline__ unsigned value_ranges(const uint16_t* sV, GroupQ* vq, float* vstep,
                                                 uint8_t* rec, const RecLayout& L,
                                                 bool& exact_tile) {
  constexpr int top = (1 << VB) - 1;
  const int t = threadIdx.x >> 1, h = threadIdx.x & 1;
  float* vscale = reinterpret_cast<float*>(rec + L.v_scale);
  uint16_t* vmin = reinterpret_cast<uint16_t*>(rec + L.v_min);
  const uint4* row = reinterpret_cast<const uint4*>(sV + t * kD);
  unsigned flags = 0;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = h ? 3 - jj : jj;
    uint32_t mn = 0u, mx = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w = row[(4 * j + k) ^ (t & 7)];
      const uint32_t a = bmin2(bmin2(w.x, w.y), bmin2(w.z, w.w));
      const uint32_t b = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
      mn = k ? bmin2(mn, a) : a;
      mx = k ? bmax2(mx, b) : b;
    }
    mn = bmin2(mn, swap_halves(mn));
    mx = bmax2(mx, swap_halves(mx));
    uint32_t lb = mn & 0xFFFFu;
    const uint32_t hb = mx & 0xFFFFu;
    const bool bad = nonfinite_bits(lb) || nonfinite_bits(hb);
    if (!bad && (lb & 0x7FFFu) == 0u) {   // a zero minimum: -0 iff the group holds one
      lb = 0u;
      for (int c = 32 * j; c < 32 * j + 32; ++c)
        if (sV[swz(t, c)] == 0x8000u) lb = 0x8000u;
    }
    const Params p = group_params(bf2f(static_cast<uint16_t>(lb)),
                                  bf2f(static_cast<uint16_t>(hb)), top, bad);
    vq[t * kVGroups + j] = make_q(p, exact_tile);
    vstep[t * kVGroups + j] = p.step;
    vscale[t * kVGroups + j] = p.step;
    vmin[t * kVGroups + j] = f2bf_bits(p.m);
    flags |= p.flags;
  }
  return flags;
}

// Value codes straight into fragment-order words.  A word (tile mc, lane
// (g, t), k-step column) holds channels 16 mc + g and + 8 of tokens 16 kt +
// 2t + {0, 1, 8, 9}.  Thread (t, token parity half, g-half gh, w-half wh,
// mc) takes channels 16 mc + 4 gh + {0..3} (and + 8) of its tokens 16 kt +
// 2t + 8 chi + half, kt in 4 wh .. 4 wh + 3: an 8-byte read per (token,
// channel half) gives the four channels of lanes g = 4 gh .. 4 gh + 3.  The
// two lanes of a token pair (half = 0, 1) OR their words together; lanes
// 0..15 read sixteen different 8-byte places of the swizzled tile.
// Exact path of a whole value tile: every code from the IEEE quotient, each
// word built by one thread (words w of lanes (g, t) of tile mc).
template <int VB>
__device__ __noinline__ void value_codes_slow(const uint16_t* sV, const GroupQ* vq,
                                              const float* vstep, uint32_t* dst) {
  constexpr int top = (1 << VB) - 1;
  constexpr int per = 32 / VB;
#pragma unroll 1
  for (int wd = threadIdx.x; wd < kKG * kD * VB / 32; wd += blockDim.x) {
    uint32_t acc = 0;
#pragma unroll 1
    for (int sl = 0; sl < per; ++sl) {
      int tok, ch;
      value_word_code(wd, sl, VB, tok, ch);
      const int gi = tok * kVGroups + ch / kVG;
      acc |= code_exact(bf2f(sV[swz(tok, ch)]), -vq[gi].nm, vstep[gi], top) << (VB * sl);
    }
    dst[wd] = acc;
  }
}

template <int VB, bool KIVI = false>
__device__ __forceinline__ void value_codes(const uint16_t* sV, const GroupQ* vq,
                                            const void* steps, bool exact_tile, uint32_t* dst) {
  const float* vstep = static_cast<const float*>(steps);
  const uint16_t* vst = static_cast<const uint16_t*>(steps);   // KIVI: bf16 [128][4]
  constexpr int top = (1 << VB) - 1;
  constexpr int NW = VB == 2 ? 8 : 16;   // words before the pair merge: (w, i) or (kt, i)
  if (!KIVI && exact_tile) {   // block-uniform, rare
    value_codes_slow<VB>(sV, vq, vstep, dst);
    return;
  }
  const int tid = threadIdx.x;
  const int t = tid & 3, half = (tid >> 2) & 1, gh = (tid >> 3) & 1, wh = (tid >> 4) & 1,
            mc = tid >> 5;
  const int j = mc >> 1;
  const uint2* rows = reinterpret_cast<const uint2*>(sV);   // [128 tokens][32 half pieces]
  uint32_t acc[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) acc[i] = 0u;
#pragma unroll
  for (int wl = 0; wl < 2; ++wl)
#pragma unroll
    for (int kl = 0; kl < 2; ++kl)
#pragma unroll
      for (int chi = 0; chi < 2; ++chi) {
        const int w = 2 * wh + wl;
        const int tok = 16 * (2 * w + kl) + 2 * t + 8 * chi + half;
        const GroupQ q = vq[tok * kVGroups + j];
#pragma unroll
        for (int rhi = 0; rhi < 2; ++rhi) {
          const uint2 x2 = rows[tok * 32 + 2 * ((2 * mc + rhi) ^ (tok & 7)) + gh];
          const uint32_t xw[2] = {x2.x, x2.y};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float d = (i & 1) ? sub_hi(xw[i >> 1], q.nm) : sub_lo(xw[i >> 1], q.nm);
            uint32_t v;
            if constexpr (KIVI) {
              v = kivi_bits<VB>(d, q.rcp, vst + tok * kVGroups + j);
            } else {
              v = code_bits(d, q.rcp);
              if (is_near(v)) v = near_bits(v, d, vstep[tok * kVGroups + j], top);   // rare
            }
            if (VB == 2) acc[4 * wl + i] |= place<2>(v, 2 * (4 * rhi + 2 * kl + chi) + 16 * half);
            else acc[8 * wl + 4 * kl + i] |= place<4>(v, 4 * (2 * rhi + chi) + 16 * half);
          }
        }
      }
  // the other token of each pair (lane ^ 4) holds the other half of every word
#pragma unroll
  for (int i = 0; i < NW; ++i) acc[i] |= __shfl_xor_sync(0xffffffffu, acc[i], 4);
  // lane half = 0 stores the words of w = 2 wh, half = 1 those of 2 wh + 1
  const int w = 2 * wh + half;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int g = 4 * gh + i;
    if (VB == 2) {   // word (mc*32 + 4g + t)*4 + w
      dst[(mc * 32 + 4 * g + t) * 4 + w] = half ? acc[4 + i] : acc[i];
    } else {         // words ((mc*2 + w/2)*32 + 4g + t)*4 + 2(w%2) + kl
      const uint32_t a0 = half ? acc[8 + i] : acc[i], a1 = half ? acc[12 + i] : acc[4 + i];
      *reinterpret_cast<uint2*>(dst + ((mc * 2 + (w >> 1)) * 32 + 4 * g + t) * 4 + 2 * (w & 1)) =
          make_uint2(a0, a1);
    }
  }
}

__device__ __forceinline__ uint8_t* group_record(const QuantArgs& a) {
  return a.records + (static_cast<long long>(blockIdx.y) * a.max_groups + a.first_group +
                      blockIdx.x) * a.rec_bytes;
}

// Dynamic shared memory of a quantize block: the staged tile (32 KB), then
// the parameter area (kParamBytes): values use vq [512] and vstep [512];
// keys use kq [128], kstep [128] and a 4 KB reduction buffer; mixed key
// blocks keep their rank keys and tiers after the reduction buffer and add
// their virtual codes after the parameter area.
constexpr int kTileBytes = kKG * kD * 2;
constexpr int kParamBytes = kKG * kVGroups * (8 + 4);   // 6 KB, the larger of the uses
constexpr int kRedBytes = 8 * 16 * 8 * 4;               // key range reduction buffer
static_assert(kD * 12 + kRedBytes <= kParamBytes, "key parameters fit the area");
static_assert(kRedBytes + 512 + 128 + 512 <= kParamBytes, "mixed ranking area fits");

// Value half of a group (block z = 1 of every quantize launch).
template <int VB>
__device__ __forceinline__ void value_part(const QuantArgs& a, uint8_t* smem) {
  uint16_t* sV = reinterpret_cast<uint16_t*>(smem);
  GroupQ* vq = reinterpret_cast<GroupQ*>(smem + kTileBytes);
  float* vstep = reinterpret_cast<float*>(smem + kTileBytes + kKG * kVGroups * 8);
  load_tile(a, a.src.v, sV);
  __syncthreads();
  uint8_t* rec = group_record(a);
  bool exact_tile = false;
  const unsigned flags = value_ranges<VB>(sV, vq, vstep, rec, a.lay, exact_tile);
  exact_tile = __syncthreads_or(exact_tile);
  value_codes<VB>(sV, vq, vstep, exact_tile, reinterpret_cast<uint32_t*>(rec + a.lay.v_codes));
  if (flags) atomicOr(a.status, flags);
}

// Uniform keys and values of one 128-token group: block (group, unit, z),
// z = 0 the keys, z = 1 the values, each from its own 32 KB staged tile.
// At most 48 registers a thread, so five blocks (40 warps) share an SM:
// each block waits on its tile load alone, and more blocks keep more loads
// in flight.
template <int KB, int VB>
__global__ void __launch_bounds__(256, 5) quantize_uniform_kernel(QuantArgs a) {
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
  bool bad, exact_tile = false;
  key_ranges(sT, sRed, lo, hi, bad);
  if (threadIdx.x < kD) {
    const int d = threadIdx.x;
    const Params p = group_params(lo, hi, (1 << KB) - 1, bad);
    kq[d] = make_q(p, exact_tile);
    kstep[d] = p.step;
    reinterpret_cast<float*>(rec + a.lay.k_scale)[d] = p.step;
    reinterpret_cast<uint16_t*>(rec + a.lay.k_min)[d] = f2bf_bits(p.m);
    flags = p.flags;
  }
  exact_tile = __syncthreads_or(exact_tile);
  key_codes<KB>(sT, kq, kstep, exact_tile, reinterpret_cast<uint32_t*>(rec + a.lay.k_codes));
  if (flags) atomicOr(a.status, flags);
}

// ---- KIVI streaming variant, prefill (f1; "KIVI: KV cache axes" §4–§7).
// The records of a prefill in one launch: block (record, unit, z).  z = 0
// seals the record's 128 keys: per channel four 32-token groups (origin and
// step bf16, [4][D]), codes in the key fragment order.  z = 1 quantizes the
// values of the record's tokens that have left the FIFO (kivi_valid counts
// them from the launch's first record on): per token four 32-channel groups
// (bf16 [128][4]); the other tokens' codes and metadata are written zero.
// Ranges are bf16x2 min / max (NaN-propagating) with -0 below +0 (the
// oracle's order); a non-finite group keeps step 0, origin 0 and zero codes,
// flagged.
template <int B>
__global__ void __launch_bounds__(256, 5) quantize_kivi_kernel(QuantArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int top = (1 << B) - 1;
  constexpr int kSub = 32, kSubs = kKG / kSub;
  uint8_t* rec = group_record(a);
  const RecLayout& L = a.lay;
  uint16_t* sT = reinterpret_cast<uint16_t*>(smem);
  GroupQ* q = reinterpret_cast<GroupQ*>(smem + kTileBytes);   // 512 groups
  unsigned flags = 0;
  if (blockIdx.z == 0) {
    load_tile(a, a.src.k, sT);
    __syncthreads();
    uint16_t* kst = reinterpret_cast<uint16_t*>(rec + L.k_scale);
    uint16_t* kmn = reinterpret_cast<uint16_t*>(rec + L.k_min);
    {
      // thread = (sub-group sg, channel pair 2c, 2c + 1): bf16x2 min / max
      // (NaN-propagating) over the sub-group's 32 rows, one word a row
      const int sg = threadIdx.x >> 6, c = threadIdx.x & 63;
      const uint32_t* rows = reinterpret_cast<const uint32_t*>(sT);
      uint32_t mn = 0u, mx = 0u;
      for (int t = kSub * sg; t < kSub * sg + kSub; ++t) {
        const uint32_t w = rows[swz(t, 2 * c) >> 1];
        mn = t == kSub * sg ? w : bmin2(mn, w);
        mx = t == kSub * sg ? w : bmax2(mx, w);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int d = 2 * c + h, gi = sg * kD + d;
        uint32_t lb = (mn >> (16 * h)) & 0xFFFFu;
        const uint32_t hb = (mx >> (16 * h)) & 0xFFFFu;
        const bool nf = nonfinite_bits(lb) || nonfinite_bits(hb);
        if (!nf && (lb & 0x7FFFu) == 0u) {   // a zero minimum: -0 iff the group holds one
          lb = 0u;
          for (int t = kSub * sg; t < kSub * sg + kSub; ++t)
            if (sT[swz(t, d)] == 0x8000u) lb = 0x8000u;
        }
        const KiviGroupP p = kivi_group(bf2f(static_cast<uint16_t>(lb)),
                                        bf2f(static_cast<uint16_t>(hb)), nf, top);
        flags |= p.flags;
        kst[gi] = f2bf_bits(p.step);
        kmn[gi] = nf ? 0 : f2bf_bits(p.m);
        q[gi] = kivi_q(p);
      }
    }
    __syncthreads();   // the steps reach the record before the code pass reads them back
    key_codes<B, true>(sT, q, kst, false, reinterpret_cast<uint32_t*>(rec + L.k_codes));
  } else {
    const int nv = min(kKG, a.kivi_valid - kKG * static_cast<int>(blockIdx.x));
    uint16_t* vst = reinterpret_cast<uint16_t*>(rec + L.v_scale);
    uint16_t* vmn = reinterpret_cast<uint16_t*>(rec + L.v_min);
    if (nv <= 0) {   // every value of the record is still in the FIFO: an empty value part
      uint4* z = reinterpret_cast<uint4*>(rec + L.v_codes);
      for (int i = threadIdx.x; i < (static_cast<int>(a.rec_bytes) - L.v_codes) / 16; i += blockDim.x)
        z[i] = make_uint4(0u, 0u, 0u, 0u);
      return;
    }
    load_tile(a, a.src.v, sT);
    __syncthreads();
    {
      // thread = (token t, groups j = 2h, 2h + 1; h = 1 in the order 3, 2):
      // bf16x2 min / max over the group's four 16-byte pieces
      const int t = threadIdx.x >> 1, h = threadIdx.x & 1;
      const uint4* row = reinterpret_cast<const uint4*>(sT + t * kD);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = h ? 3 - jj : jj, gi = t * kVGroups + j;
        if (t >= nv) {   // still in the FIFO
          vst[gi] = 0;
          vmn[gi] = 0;
          q[gi] = {0.0f, 0.0f};
          continue;
        }
        uint32_t mn = 0u, mx = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 w = row[(4 * j + k) ^ (t & 7)];
          const uint32_t lo2 = bmin2(bmin2(w.x, w.y), bmin2(w.z, w.w));
          const uint32_t hi2 = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
          mn = k ? bmin2(mn, lo2) : lo2;
          mx = k ? bmax2(mx, hi2) : hi2;
        }
        mn = bmin2(mn, swap_halves(mn));
        mx = bmax2(mx, swap_halves(mx));
        uint32_t lb = mn & 0xFFFFu;
        const uint32_t hb = mx & 0xFFFFu;
        const bool nf = nonfinite_bits(lb) || nonfinite_bits(hb);
        if (!nf && (lb & 0x7FFFu) == 0u) {   // a zero minimum: -0 iff the group holds one
          lb = 0u;
          for (int cc = kSub * j; cc < kSub * j + kSub; ++cc)
            if (sT[swz(t, cc)] == 0x8000u) lb = 0x8000u;
        }
        const KiviGroupP p = kivi_group(bf2f(static_cast<uint16_t>(lb)),
                                        bf2f(static_cast<uint16_t>(hb)), nf, top);
        flags |= p.flags;
        vst[gi] = f2bf_bits(p.step);
        vmn[gi] = nf ? 0 : f2bf_bits(p.m);
        q[gi] = kivi_q(p);
      }
    }
    __syncthreads();
    value_codes<B, true>(sT, q, vst, false, reinterpret_cast<uint32_t*>(rec + L.v_codes));
  }
  if (flags) atomicOr(a.status, flags);
}

// PN-Mix H3/L1 keys and uniform values of one 128-token group (z = 1: the
// values).  Keys: thread p < 128 takes the unit's stored position p
// (channel perm[p]; the first nh positions are the selected pairs' channels):
// high channels by Eq. 2 at 3 bits (origin the minimum, step (M - m)/7),
// the others by Eq. 7 (s = (M - m)/2, z = (3m + M)/4, code RNE((x - z)/s)
// clipped to 0..1), every operation fp32 rounded; codes staged as bytes,
// then the LSB plane and the upper plane packed word by word.
// The code of a position whose scale is below 2^-100 (or whose offset
// overflowed): clip(RNE(RN((x - off) / sc)), 0, top) by the IEEE quotient.
// Out of line, as near_bits: rare, and the code loop is unrolled.
__device__ __noinline__ uint32_t pnmix_exact_code(float x, float off, float sc, float top) {
  const float y = __fdiv_rn(__fsub_rn(x, off), sc);
  return static_cast<uint32_t>(fminf(fmaxf(rintf(y), 0.0f), top));
}

template <int VB>
__global__ void __launch_bounds__(256) quantize_pnmix_kernel(QuantArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const RecLayout& L = a.lay;
  if (blockIdx.z) {
    value_part<VB>(a, smem);
    return;
  }
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem);
  uint8_t* cB = smem + kTileBytes;   // codes [128 tokens][128 positions]
  // per stored position: channel, offset, scale, RN(1/scale); mode 0 = all
  // codes 0, 1 = fast decision, 2 = IEEE quotient for every element
  __shared__ float s_off[kD], s_sc[kD], s_rcp[kD];
  __shared__ uint8_t s_ch[kD], s_mode[kD];
  load_tile(a, a.src.k, sK);
  __syncthreads();
  uint8_t* rec = group_record(a);
  unsigned flags = 0;
  // channel ranges (all threads; the code area is free until the codes),
  // then each stored position takes its channel's
  {
    float* s_clo = reinterpret_cast<float*>(cB + kRedBytes);
    float* s_chi = s_clo + kD;
    uint8_t* s_cbad = reinterpret_cast<uint8_t*>(s_chi + kD);
    float lo, hi;
    bool bad;
    key_ranges(sK, reinterpret_cast<uint32_t*>(cB), lo, hi, bad);
    if (threadIdx.x < kD) {
      s_clo[threadIdx.x] = lo;
      s_chi[threadIdx.x] = hi;
      s_cbad[threadIdx.x] = bad;
    }
    __syncthreads();
  }
  if (threadIdx.x < kD) {
    const int p = threadIdx.x;
    const int ch = a.perm[static_cast<long long>(blockIdx.y) * kD + p];
    const float* s_clo = reinterpret_cast<const float*>(cB + kRedBytes);
    const float lo = s_clo[ch], hi = s_clo[kD + ch];
    const bool bad = (cB + kRedBytes + 2 * kD * 4)[ch] != 0;
    float off = lo, sc = 0.0f;
    if (bad) {
      flags |= KVQ_FLAG_NONFINITE;
    } else if (hi != lo) {
      if (p < L.nh) {   // Eq. 2 at 3 bits
        sc = __fdiv_rn(__fsub_rn(hi, lo), 7.0f);
        if (!(sc > 0.0f) || !isfinite(sc)) flags |= KVQ_FLAG_RANGE;
      } else {          // Eq. 7
        sc = __fdiv_rn(__fsub_rn(hi, lo), 2.0f);
        off = __fdiv_rn(__fadd_rn(__fmul_rn(3.0f, lo), hi), 4.0f);
        if (!(sc > 0.0f) || !isfinite(sc) || !isfinite(off)) flags |= KVQ_FLAG_RANGE;
      }
    }
    reinterpret_cast<float*>(rec + L.k_scale)[p] = sc;
    reinterpret_cast<float*>(rec + L.k_min)[p] = off;
    s_ch[p] = static_cast<uint8_t>(ch);
    s_off[p] = off;
    s_sc[p] = sc;
    s_rcp[p] = sc > 0.0f ? __frcp_rn(sc) : 0.0f;
    s_mode[p] = (bad || !(sc > 0.0f)) ? 0 : (sc < kTinyStep || !isfinite(sc) || !isfinite(off)) ? 2 : 1;
  }
  __syncthreads();
  // Codes, two threads a position (64 tokens each).  High positions (Eq. 2,
  // 3 bits): the uniform quantizer's decision (code_bits, and near_bits
  // near a rounding boundary), RNE(RN(d / s)) bit for bit.  Low positions
  // (Eq. 7): clip(RNE(RN(d / s)), 0, 1) is 1 iff RN(d / s) > 1/2, i.e. iff
  // d - s/2 > s 2^-25; the remainder by one FMA is exact wherever the
  // comparison is close (Sterbenz: d within [s/4, s]), and far from it the
  // rounding cannot change its sign or its side of s 2^-25.
  {
    const int p = threadIdx.x & (kD - 1), t0 = (threadIdx.x >> 7) * (kKG / 2);
    const int ch = s_ch[p], mode = s_mode[p];
    const float off = s_off[p], sc = s_sc[p], rcp = s_rcp[p];
    const bool hi3 = p < L.nh;
    const float half_ulp = sc * 0x1p-25f;
    // unrolled by the swizzle period, so each element's tile offset is a constant
#pragma unroll 8
    for (int t = t0; t < t0 + kKG / 2; ++t) {
      uint32_t c = 0;
      const float x = bf2f(sK[swz(t, ch)]);
      if (mode == 1) {
        const float d = __fsub_rn(x, off);
        if (hi3) {
          uint32_t v = code_bits(d, rcp);
          if (is_near(v)) v = near_bits(v, d, sc, 7u);   // rare
          c = (v >> 18) & 7u;
        } else {
          c = __fmaf_rn(-0.5f, sc, d) > half_ulp ? 1u : 0u;
        }
      } else if (mode == 2) {   // rare: the IEEE quotient
        c = pnmix_exact_code(x, off, sc, hi3 ? 7.0f : 1.0f);
      }
      cB[t * kD + p] = static_cast<uint8_t>(c);
    }
  }
  __syncthreads();
  // LSB plane: word (mt*2 + ks/4)*32 + lane, bit 2*(ks%4) + chi + 8*rhi + 16*half
  // for token 16 mt + g + 8 rhi and position 16 ks + 2t + 8 chi + half; the
  // two halves are adjacent positions, read together
  const uint16_t* cB2 = reinterpret_cast<const uint16_t*>(cB);
  uint32_t* lsb = reinterpret_cast<uint32_t*>(rec + L.k_codes);
  for (int w = threadIdx.x; w < kKG * kD / 32; w += blockDim.x) {
    const int lane = w & 31, kq = (w >> 5) & 1, mt = w >> 6;
    const int g = lane >> 2, t = lane & 3;
    uint32_t acc = 0;
#pragma unroll
    for (int rhi = 0; rhi < 2; ++rhi)
#pragma unroll
      for (int kl4 = 0; kl4 < 4; ++kl4)
#pragma unroll
        for (int chi = 0; chi < 2; ++chi) {
          const int tok = 16 * mt + g + 8 * rhi, p = 16 * (4 * kq + kl4) + 2 * t + 8 * chi;
          const uint32_t two = cB2[(tok * kD + p) >> 1];   // positions p, p + 1
          const int bit = 2 * kl4 + chi + 8 * rhi;
          acc |= (two & 1u) << bit;
          acc |= ((two >> 8) & 1u) << (bit + 16);
        }
    lsb[w] = acc;
  }
  // upper plane of the high positions: 2-bit key fragment order, kw2 words a
  // (tile, lane): word (mt kw2 + wi) 32 + lane, slot P + 8 half for token
  // 16 mt + g + 8 (P >> 2) and position 32 wi + 16 ((P >> 1) & 1) + 8 (P & 1)
  // + 2t + half (the fragment pair order of the mixed key records)
  uint32_t* up = reinterpret_cast<uint32_t*>(rec + L.kc);
  for (int w = threadIdx.x; w < 8 * L.kw2 * 32; w += blockDim.x) {
    const int lane = w & 31, qw = w >> 5, mt = qw / L.kw2, wi = qw - mt * L.kw2;
    const int g = lane >> 2, t = lane & 3;
    uint32_t acc = 0;
#pragma unroll
    for (int P = 0; P < 8; ++P) {
      const int tok = 16 * mt + g + 8 * (P >> 2);
      const int v = 32 * wi + 16 * ((P >> 1) & 1) + 8 * (P & 1) + 2 * t;
      const uint32_t two = cB2[(tok * kD + v) >> 1];   // positions v, v + 1
      acc |= ((two >> 1) & 3u) << (2 * P);
      acc |= ((two >> 9) & 3u) << (2 * P + 16);
    }
    up[w] = acc;
  }
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
  uint32_t* sRed = reinterpret_cast<uint32_t*>(smem + kTileBytes);                   // 4 KB
  uint32_t* sKey = reinterpret_cast<uint32_t*>(smem + kTileBytes + kRedBytes);      // 512 B
  uint8_t* sTier = smem + kTileBytes + kRedBytes + 512;                             // 128 B
  float* sA = reinterpret_cast<float*>(smem + kTileBytes + kRedBytes + 512 + 128);  // 512 B
  uint8_t* cKv = smem + kTileBytes + kParamBytes;
  // per channel, for the code pass: origin, step, RN(1/step), code slots, fast path
  __shared__ float s_mx[kD], s_st[kD], s_rc[kD];
  __shared__ int16_t s_at[kD], s_at4[kD];
  __shared__ bool s_fast[kD];
  // ranking: second halves' counts, per-warp tier ballots, BF16 slot -> channel
  __shared__ int s_rk[kD];
  __shared__ uint32_t s_tm[3][kD / 32];
  __shared__ uint8_t s_bf[kD];
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
  // per channel (threads below 128): importance, saliency A = I * S, and a
  // total-order rank key (NaN, only possible on a flagged group, sorts last,
  // so ranks are always a permutation and every slot stays inside its
  // tier's region)
  const int d = threadIdx.x & (kD - 1);
  const bool chan = threadIdx.x < kD;
  float A = 0.0f;
  if (chan) {
    float S = 0.0f;
    if (!bad) S = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    const long long ud = static_cast<long long>(u) * kD + d;
    const float I = a.importance ? a.importance[ud] : __fdiv_rn(a.qacc[ud], a.q_count);
    if (!isfinite(I)) flags |= KVQ_FLAG_NONFINITE;
    if (bad) flags |= KVQ_FLAG_NONFINITE;
    else if (!isfinite(S)) flags |= KVQ_FLAG_RANGE;
    A = __fmul_rn(I, S);
    sKey[d] = isnan(A) ? 0u : fkey(A);
  }
  // how many channels pass each threshold (NaN passes none); each count is
  // also a barrier, the first one after the keys
  const int above_b = __syncthreads_count(chan && A > a.tau_bf16);
  const int above_4 = __syncthreads_count(chan && A > a.tau_uint4);
  int nb = L.nb, n4 = L.n4;
  if (L.thresh) {
    nb = min(above_b, L.nb);
    n4 = max(0, min(above_4 - nb, L.n4));
  }
  // rank: the keys above this channel's, or equal at a lower channel; two
  // threads a channel, half of the keys each
  int rank = 0;
  {
    const uint32_t key = sKey[d];
    const int e0 = (threadIdx.x >> 7) * (kD / 2);
    int part = 0;
#pragma unroll 8
    for (int e = e0; e < e0 + kD / 2; ++e) {
      const uint32_t ke = sKey[e];
      part += (ke > key || (ke == key && e < d)) ? 1 : 0;
    }
    if (!chan) s_rk[d] = part;
    __syncthreads();
    if (chan) rank = part + s_rk[d];
  }
  // tiers; a channel's slot in its tier is the number of lower channels of
  // that tier (per-warp ballots)
  int tier = KVQ_TIER_UINT2;
  if (chan) {
    tier = rank < nb ? KVQ_TIER_BF16 : rank < nb + n4 ? KVQ_TIER_UINT4 : KVQ_TIER_UINT2;
    sTier[d] = static_cast<uint8_t>(tier);
    if (d == 0) {
      rec[L.hdr] = static_cast<uint8_t>(nb);
      rec[L.hdr + 1] = static_cast<uint8_t>(n4);
    }
    const unsigned mb = __ballot_sync(0xffffffffu, tier == KVQ_TIER_BF16);
    const unsigned m4 = __ballot_sync(0xffffffffu, tier == KVQ_TIER_UINT4);
    const unsigned m2 = __ballot_sync(0xffffffffu, tier == KVQ_TIER_UINT2);
    if ((d & 31) == 0) {
      s_tm[0][d >> 5] = mb;
      s_tm[1][d >> 5] = m4;
      s_tm[2][d >> 5] = m2;
    }
  }
  __syncthreads();
  if (chan) {
    const int ti = tier == KVQ_TIER_BF16 ? 0 : tier == KVQ_TIER_UINT4 ? 1 : 2;
    int slot = ti == 0 ? 0 : ti == 1 ? nb : nb + n4;
    for (int w = 0; w < (d >> 5); ++w) slot += __popc(s_tm[ti][w]);
    slot += __popc(s_tm[ti][d >> 5] & ((1u << (d & 31)) - 1u));
    rec[L.perm + slot] = static_cast<uint8_t>(d);
    if (tier == KVQ_TIER_BF16) {
      s_bf[slot] = static_cast<uint8_t>(d);
    } else {
      const int bits = tier == KVQ_TIER_UINT4 ? 4 : 2;
      const int top = (1 << bits) - 1;
      const Params p = group_params(lo, hi, top, bad);
      flags |= p.flags;
      const int j = slot - nb;   // index among the quantized channels
      reinterpret_cast<float*>(rec + L.s4)[j] = p.step;
      reinterpret_cast<uint16_t*>(rec + L.m4)[j] = f2bf_bits(p.m);
      // codes below, two threads a channel
      s_mx[d] = p.m;
      s_st[d] = p.step;
      s_rc[d] = p.step > 0.0f ? __frcp_rn(p.step) : 0.0f;
      s_at[d] = static_cast<int16_t>(bits == 4 ? j : n4 + j);
      s_at4[d] = static_cast<int16_t>(n4 + j);
      // flagged channels and steps below 2^-100 take the IEEE quotient
      s_fast[d] = p.flags == 0u && !(p.step > 0.0f && p.step < kTinyStep);
    }
  }
  __syncthreads();
  // the BF16 tier's raw keys, all threads: slot s holds channel s_bf[s]'s
  // 128 tokens, 16-byte pieces rotated by the slot
  {
    uint16_t* raw = reinterpret_cast<uint16_t*>(rec + L.raw);
    for (int i = threadIdx.x; i < nb * kKG; i += blockDim.x) {
      const int slot = i >> 7, t = i & (kKG - 1);
      raw[slot * kKG + ((((t >> 3) ^ (slot & 7)) << 3) | (t & 7))] = sK[swz(t, s_bf[slot])];
    }
  }
  // UINT4 / UINT2 codes, two threads a channel (64 tokens each), by the
  // uniform quantizer's decision (code_bits, near_bits for the elements near
  // a rounding boundary): RNE(RN(d / step)) bit for bit
  {
    const int d = threadIdx.x & (kD - 1), t0 = (threadIdx.x >> 7) * (kKG / 2);
    const int tier = sTier[d];
    if (tier != KVQ_TIER_BF16) {
      const int bits = tier == KVQ_TIER_UINT4 ? 4 : 2;
      const int top = (1 << bits) - 1;
      const float m = s_mx[d], step = s_st[d], r = s_rc[d];
      const int lo_at = s_at[d], hi_at = s_at4[d];
      const bool fast = s_fast[d];
      // unrolled by the tile's swizzle period, so each element's offset is a constant
#pragma unroll 8
      for (int t = t0; t < t0 + kKG / 2; ++t) {
        const float x = bf2f(sK[swz(t, d)]);
        uint32_t c;
        if (fast) {
          const float dd = __fsub_rn(x, m);
          uint32_t v = code_bits(dd, r);
          if (is_near(v)) v = near_bits(v, dd, step, top);   // rare
          c = (v >> 18) & static_cast<uint32_t>(top);
        } else {
          c = code_exact_rare(x, m, step, top);
        }
        cKv[t * kvs + lo_at] = static_cast<uint8_t>(bits == 4 ? (c & 3u) : c);
        if (bits == 4) cKv[t * kvs + hi_at] = static_cast<uint8_t>(c >> 2);
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
  a.perm = c->pn_perm;
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
  if (c->cfg.k_mode == KVQ_K_PNMIX) {
    const int smem = kTileBytes + kKG * kD;   // the tile, then the code bytes (>= values' need)
    static_assert(kKG * kD >= kParamBytes, "PN-Mix code bytes cover the value parameters");
    if (vb == 2) KVQ_LAUNCH(quantize_pnmix_kernel<2>, smem);
    else KVQ_LAUNCH(quantize_pnmix_kernel<4>, smem);
  } else if (c->cfg.k_mode == KVQ_K_MIXED) {
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

cudaError_t launch_kivi_prefill(const kvq_cache* c, QuantSrc src, int n_records, int n_valid,
                                cudaStream_t s) {
  if (n_records == 0) return cudaSuccess;
  QuantArgs a = {};
  a.src = src;
  a.records = c->records;
  a.rec_bytes = c->lay.bytes;
  a.max_groups = c->max_groups;
  a.first_group = 0;
  a.lay = c->lay;
  a.kivi_valid = n_valid;
  a.status = c->status;
  const dim3 grid(n_records, c->cfg.batch * c->cfg.kv_heads, 2);   // z: keys, values
  cudaError_t e;
  if (c->cfg.k_bits == 2) {
    static SmemOptIn opt_in;
    if ((e = opt_in.ensure(quantize_kivi_kernel<2>)) != cudaSuccess) return e;
    quantize_kivi_kernel<2><<<grid, 256, kQuantSmem, s>>>(a);
  } else {
    static SmemOptIn opt_in;
    if ((e = opt_in.ensure(quantize_kivi_kernel<4>)) != cudaSuccess) return e;
    quantize_kivi_kernel<4><<<grid, 256, kQuantSmem, s>>>(a);
  }
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
