// Tensor-core split-K decode attention over the packed cache (uniform keys).
//
// Math as in the CUDA-core version ("KIVI: KV cache axes" §1, §6; MixKVQ
// Algorithm 1): s = q·k^/sqrt(D) over history and residual, one softmax,
// o = sum p v^.  Per 128-token group g of one (b, kv head) the two dense
// contractions run on mma.sync.m16n8k16 (f16 operands, fp32 accumulators):
//
//   S[tok][h]  = sum_ch C_K[tok][ch] Q'[ch][h],   Q' = q * step_K * log2e/sqrt(D)
//   O^T[ch][h] = sum_tok C_V^T[ch][tok] P'[tok][h], P' = p * step_V(tok, ch/32)
//
// with the origins added on the side: bias_h = sum_ch q m_K (CUDA cores) and
// sum_tok p m_V (a fifth small MMA whose A rows are the value origins).
// Codes are exact in f16.  A pair of codes becomes an f16x2 register with
// one shift and one LOP3: the code lands in the mantissa of 1.0, giving
// 1 + c/4 or 1 + c/16, the B rows carry the matching factor 4 or 16, and
// the constant part sum_k B[k][h] of the scores is removed with one more
// MMA whose A tile is all ones (exactly the same B values, so it cancels to
// fp32 rounding).  Value codes are made exact (c, one HFMA2 per pair) so the
// running output accumulates offset-free in the MMA accumulators across
// groups.
// Q' and P' are normalized by powers of two per group (and V channel group)
// so every f16 operand stays in range for any bf16 input.  Q' is split into
// an f16 high part and an f16 low part (the rounding error of the high part)
// so the scores carry ~22 bits of Q': with at most 4 query heads per KV head
// the low part rides in the 4 otherwise unused B columns (lanes of columns
// 4-7 hold head (column - 4)) and one shuffle adds it back; with 8 heads a
// second MMA per k-step accumulates it.
//
// Work split ("stream-K"): the flattened sequence of items (for each unit
// its groups, then its residual as one item of weight kResidualWeight) is
// cut into equal contiguous slices, one per warp; a warp keeps one online-
// softmax state per unit it touches and writes one partial per unit.  Each
// warp stages one record at a time in its own shared memory, in two parts:
// the key part of the next group loads while the current group's softmax and
// P·V run, the value part of the next group while its QK runs.  Warps never
// wait on each other.  The combine kernel merges each query head's partials
// with the exact log-sum-exp rule.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "frag_layout.h"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr uint32_t kOne2 = 0x3C003C00u;  // f16x2 (1.0, 1.0)
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kResidualWeight = 3;       // residual item ~ 3 groups of work
constexpr float kSentinel = 4.2535295865117308e37f;  // 2^125: "no group yet"

// Per-warp shared memory after the record buffer (key part, then value
// part): the value-step table (256 words), the value-origin table (4 rows of
// 72 words) and the unit's query, [8 heads][136] bf16 or, with at most 4
// heads per KV head, [4 heads][136] fp32 pre-scaled by log2(e)/sqrt(D)
// (rows padded so head rows fall in different banks).
constexpr int kVsbBytes = 256 * 4;
constexpr int kVmbBytes = 4 * 72 * 4;
constexpr int kQRow = 136;
constexpr int kQBytes = 8 * kQRow * 2;   // = 4 * kQRow * 4
constexpr int kWarpExtra = kVsbBytes + kVmbBytes + kQBytes;

__device__ __forceinline__ float bf2f(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Power-of-two normalizer for a non-negative magnitude x: returns s with
// x*s in [0.5, 1) for ordinary x (clamped at the extremes), and 1/s.
__device__ __forceinline__ void pow2_norm(float x, float& s, float& inv) {
  int e = (__float_as_uint(x) >> 23) & 0xff;
  e = min(max(e, 1), 252);
  s = __uint_as_float(static_cast<uint32_t>(253 - e) << 23);
  inv = __uint_as_float(static_cast<uint32_t>(e + 1) << 23);
}

// 1/x for x an exact power of two in the normal range (exponent arithmetic).
__device__ __forceinline__ float pow2_rcp(float x) {
  return __uint_as_float((254u << 23) - __float_as_uint(x));
}

// Swizzled positions in the per-warp value tables (u32 index), chosen so
// both the writers (lane = 4 tokens) and the readers (lane = fragment
// position) hit distinct shared-memory banks.
// vsb: per (kt, t) 8 words (j = 0..3, slot = b0/b1), stored as two 16-byte
//      chunks c = 2t + (j >> 1) placed at chunk c ^ kt of row kt.
__device__ __forceinline__ int vsb_index(int kt, int t, int j, int slot) {
  const int c = (2 * t + (j >> 1)) ^ kt;
  return kt * 32 + c * 4 + (j & 1) * 2 + slot;
}
// vmb: per (j, kt) 8 words (t = 0..3, slot = a0/a2), rows of j padded to 72
//      words so the four j rows start in different banks.
__device__ __forceinline__ int vmb_index(int kt, int j, int t, int slot) {
  return j * 72 + kt * 8 + t * 2 + slot;
}

// (a & b) | c in one three-input logic instruction (lookup table 0xEA).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// --- code unpacking: word -> A fragment registers (see frag_layout.h)
template <int KL>
__device__ __forceinline__ void unpack2(uint32_t x, uint32_t (&a)[4]) {
  constexpr uint32_t M4 = 0x03000300u, M16 = 0x00C000C0u;
  if (KL == 0) {
    const uint32_t l8 = x << 8, l4 = x << 4;
    a[0] = and_or(l8, M4, kOne2);
    a[1] = and_or(l4, M4, kOne2);
    a[2] = and_or(l4, M16, kOne2);
    a[3] = and_or(x, M16, kOne2);
  } else {
    const uint32_t r4 = x >> 4, r8 = x >> 8;
    a[0] = and_or(x, M4, kOne2);
    a[1] = and_or(r4, M4, kOne2);
    a[2] = and_or(r4, M16, kOne2);
    a[3] = and_or(r8, M16, kOne2);
  }
}

// Value codes exact: (1 + c/s)*s - s = c for the s = 4 and s = 16 pairs.
template <int KL>
__device__ __forceinline__ void unpack2_exact(uint32_t x, uint32_t (&a)[4]) {
  constexpr uint32_t s4 = 0x44004400u, n4 = 0xC400C400u;     // (4, 4), (-4, -4)
  constexpr uint32_t s16 = 0x4C004C00u, n16 = 0xCC00CC00u;   // (16, 16), (-16, -16)
  unpack2<KL>(x, a);
  a[0] = hfma2_u(a[0], s4, n4);
  a[1] = hfma2_u(a[1], s4, n4);
  a[2] = hfma2_u(a[2], s16, n16);
  a[3] = hfma2_u(a[3], s16, n16);
}

__device__ __forceinline__ void unpack4(uint32_t x, uint32_t (&a)[4]) {
  constexpr uint32_t M = 0x03C003C0u;
  a[0] = and_or(x << 6, M, kOne2);
  a[1] = and_or(x << 2, M, kOne2);
  a[2] = and_or(x >> 2, M, kOne2);
  a[3] = and_or(x >> 6, M, kOne2);
}

__device__ __forceinline__ void unpack4_exact(uint32_t x, uint32_t (&a)[4]) {
  constexpr uint32_t s16 = 0x4C004C00u, n16 = 0xCC00CC00u;
  unpack4(x, a);
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = hfma2_u(a[i], s16, n16);
}

struct MmaArgs {
  const uint8_t* records;
  long long rec_bytes;
  int max_groups;
  RecLayout lay;
  int n_groups;           // quantized groups per unit
  int r;                  // residual tokens
  const uint16_t* res_k;  // [units][128][D]
  const uint16_t* res_v;
  const uint16_t* q;      // [B][Hq][D]
  int Hkv, Hq, units;
  long long unit_len;     // weighted positions per unit
  long long total;        // units * unit_len
  int n_slots;            // warps with work
  int max_parts;          // partial slots per unit in ws
  float* ws;              // [units][max_parts][NREP][D + 2]
};

__device__ __forceinline__ long long slot_start(const MmaArgs& a, int w) {
  return (static_cast<long long>(w) * a.total) / a.n_slots;
}
__device__ __forceinline__ int slot_of(const MmaArgs& a, long long p) {
  return static_cast<int>(((p + 1) * a.n_slots - 1) / a.total);
}

template <int KB, int VB, int NREP>
struct Warp {
  static constexpr int KSCALE_B = KB == 2 ? 4 : 16;   // B-row factor for a0/a1
  static constexpr int KSCALE_T = 16;                  // B-row factor for a2/a3
  static constexpr bool SPARE = NREP <= 4;             // Q' low part in columns 4-7
  static constexpr int NL = SPARE ? 1 : 8;             // low-part fragments kept

  const MmaArgs& a;
  const int lane, g, t;
  uint8_t* kbuf;   // key part of the staged record
  uint8_t* vbuf;   // value part of the staged record
  uint32_t* vsb;   // value-step table, B order (vsb_index)
  uint32_t* vmb;   // value-origin table, A order (vmb_index)
  void* qs;        // the unit's query (see kQBytes)

  // online-softmax state (heads 2t, 2t+1 of this lane)
  float O[8][4];   // running O^T in units of sv[j] (channel tiles mc = 0..7)
  float vm[2];     // origin term (lanes g < 4: channel group j = g)
  float mrun[2], lrun[2];
  float sv[4], inv_sv[4];  // current units of O per j

  __device__ __forceinline__ Warp(const MmaArgs& args, uint8_t* base)
      : a(args), lane(threadIdx.x & 31), g((threadIdx.x & 31) >> 2), t(threadIdx.x & 3) {
    const int rb = static_cast<int>(a.rec_bytes);
    kbuf = base;
    vbuf = base + a.lay.kpart;
    vsb = reinterpret_cast<uint32_t*>(base + rb);
    vmb = reinterpret_cast<uint32_t*>(base + rb + kVsbBytes);
    qs = base + rb + kVsbBytes + kVmbBytes;
  }

  // x rounded to 11 significant bits (an f16 value for the normalized
  // range used here); x - result is exact in fp32
  __device__ __forceinline__ static float round_f16_precision(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x00001000u) & 0xFFFFE000u);
  }

  __device__ __forceinline__ static void qk_mma(float (&s)[4], const uint32_t (&A)[4],
                                                const uint32_t (&bq)[8][2],
                                                const uint32_t (&bl)[NL][2], int ks) {
    mma_f16(s, A[0], A[1], A[2], A[3], bq[ks][0], bq[ks][1]);
    if (!SPARE) mma_f16(s, A[0], A[1], A[2], A[3], bl[ks % NL][0], bl[ks % NL][1]);
  }

  __device__ __forceinline__ void begin_unit(int u) {
    const int b = u / a.Hkv, kvh = u % a.Hkv;
    const uint16_t* qg = a.q + (static_cast<long long>(b) * a.Hq + kvh * NREP) * kD;
    const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
    __syncwarp();
    if (SPARE) {   // fp32 [4][kQRow], pre-scaled
      float* q = static_cast<float*>(qs);
      for (int i = lane; i < 4 * kD; i += 32) {
        const int h = i / kD, c = i % kD;
        q[h * kQRow + c] = h < NREP ? bf2f(qg[h * kD + c]) * c0 : 0.0f;
      }
    } else {       // bf16 [8][kQRow]
      uint32_t* q = static_cast<uint32_t*>(qs);
      for (int i = lane; i < 8 * (kD / 2); i += 32) {
        const int h = i / (kD / 2), c2 = i % (kD / 2);
        q[h * (kQRow / 2) + c2] = reinterpret_cast<const uint32_t*>(qg + h * kD)[c2];
      }
    }
    __syncwarp();
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) O[m][c] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sv[j] = kSentinel;
      inv_sv[j] = 1.0f / kSentinel;
    }
    vm[0] = vm[1] = 0.0f;
    mrun[0] = mrun[1] = -INFINITY;
    lrun[0] = lrun[1] = 0.0f;
  }

  // cp.async of bytes [lo, hi) of group record grp of unit u into dst.
  __device__ __forceinline__ void issue(int u, int grp, uint8_t* dst, int lo, int hi) {
    const uint8_t* src = a.records + (static_cast<long long>(u) * a.max_groups + grp) * a.rec_bytes + lo;
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const int chunks = (hi - lo) >> 4;
    for (int c = lane; c < chunks; c += 32)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d + 16 * c),
                   "l"(src + 16 * c));
  }
  __device__ __forceinline__ void issue_k(int u, int grp) { issue(u, grp, kbuf, 0, a.lay.kpart); }
  __device__ __forceinline__ void issue_v(int u, int grp) {
    issue(u, grp, vbuf, a.lay.kpart, static_cast<int>(a.rec_bytes));
  }

  // Scores of one group (keys in kbuf), softmax folded into the running
  // state; returns p in S (C-fragment layout) and the rescale factors.
  __device__ __forceinline__ void qk_softmax(float (&S)[8][4], float (&alpha)[2]) {
    const RecLayout& L = a.lay;
    const float* kscale = reinterpret_cast<const float*>(kbuf + L.k_scale);
    const uint32_t* kmin2 = reinterpret_cast<const uint32_t*>(kbuf + L.k_min);
    float qk[32];
    float mx = 0.0f, bias = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const float2 s01 = *reinterpret_cast<const float2*>(kscale + 16 * ks + 2 * t);
      const float2 s89 = *reinterpret_cast<const float2*>(kscale + 16 * ks + 2 * t + 8);
      const uint32_t m01 = kmin2[8 * ks + t];
      const uint32_t m89 = kmin2[8 * ks + t + 4];
      float qa, qb, qc, qd;
      if (SPARE) {
        const float* qrow = static_cast<const float*>(qs) + (g & 3) * kQRow;
        const float2 q01 = *reinterpret_cast<const float2*>(qrow + 16 * ks + 2 * t);
        const float2 q89 = *reinterpret_cast<const float2*>(qrow + 16 * ks + 2 * t + 8);
        qa = q01.x; qb = q01.y; qc = q89.x; qd = q89.y;
      } else {
        const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
        const uint32_t* qrow = static_cast<const uint32_t*>(qs) + g * (kQRow / 2);
        const uint32_t q01 = qrow[8 * ks + t], q89 = qrow[8 * ks + t + 4];
        qa = bf2f(q01 & 0xffffu) * c0; qb = bf2f(q01 >> 16) * c0;
        qc = bf2f(q89 & 0xffffu) * c0; qd = bf2f(q89 >> 16) * c0;
      }
      qk[4 * ks + 0] = qa * s01.x;
      qk[4 * ks + 1] = qb * s01.y;
      qk[4 * ks + 2] = qc * s89.x;
      qk[4 * ks + 3] = qd * s89.y;
      bias = fmaf(qa, bf2f(m01 & 0xffffu), bias);
      bias = fmaf(qb, bf2f(m01 >> 16), bias);
      bias = fmaf(qc, bf2f(m89 & 0xffffu), bias);
      bias = fmaf(qd, bf2f(m89 >> 16), bias);
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fabsf(qk[4 * ks + i]));
    }
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    bias += __shfl_xor_sync(kFull, bias, 1);
    bias += __shfl_xor_sync(kFull, bias, 2);
    float sq, inv_sq;
    pow2_norm(mx, sq, inv_sq);
    // high part: the value rounded to f16 precision; low part: the rest
    uint32_t bq[8][2], bl[NL][2];
    {
      const float fb = sq * KSCALE_B, ft = sq * KSCALE_T;
      const bool low_lane = SPARE && g >= 4;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        float x[4] = {qk[4 * ks + 0] * fb, qk[4 * ks + 1] * fb, qk[4 * ks + 2] * ft,
                      qk[4 * ks + 3] * ft};
        float hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          hi[i] = round_f16_precision(x[i]);
          lo[i] = x[i] - hi[i];
        }
        if (SPARE) {
#pragma unroll
          for (int i = 0; i < 4; ++i) x[i] = low_lane ? lo[i] : hi[i];
          bq[ks][0] = pack_h2(x[0], x[1]);
          bq[ks][1] = pack_h2(x[2], x[3]);
        } else {
          bq[ks][0] = pack_h2(hi[0], hi[1]);
          bq[ks][1] = pack_h2(hi[2], hi[3]);
          bl[ks % NL][0] = pack_h2(lo[0], lo[1]);
          bl[ks % NL][1] = pack_h2(lo[2], lo[3]);
        }
      }
    }
    // per head of this lane's C columns: 1/sq and bias from that head's lanes
    float hinv[2], hbias[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int src = 4 * (SPARE ? ((2 * t + h) & 3) : (2 * t + h));
      hinv[h] = __shfl_sync(kFull, inv_sq, src);
      hbias[h] = __shfl_sync(kFull, bias, src);
    }

    // ---- QK on tensor cores, k-step outer: eight independent accumulator chains
    float Ck[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      mma_f16(Ck, kOne2, kOne2, kOne2, kOne2, bq[ks][0], bq[ks][1]);
      if (!SPARE) mma_f16(Ck, kOne2, kOne2, kOne2, kOne2, bl[ks % NL][0], bl[ks % NL][1]);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[mt][c] = 0.0f;
    const uint8_t* kc = kbuf + L.k_codes;
    if (KB == 2) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t kw[8];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          kw[mt] = reinterpret_cast<const uint32_t*>(kc)[(mt * 4 + w) * 32 + lane];
#pragma unroll
        for (int kl = 0; kl < 2; ++kl) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t A[4];
            if (kl) unpack2<1>(kw[mt], A);
            else unpack2<0>(kw[mt], A);
            qk_mma(S[mt], A, bq, bl, 2 * w + kl);
          }
        }
      }
    } else {
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint2 kw[8];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          kw[mt] = reinterpret_cast<const uint2*>(kc)[(mt * 4 + kp) * 32 + lane];
#pragma unroll
        for (int kl = 0; kl < 2; ++kl) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t A[4];
            unpack4(kl ? kw[mt].y : kw[mt].x, A);
            qk_mma(S[mt], A, bq, bl, 2 * kp + kl);
          }
        }
      }
    }

    // ---- scores in log2 units and the online softmax
    if (SPARE) {   // columns c and c + 4 hold the high and low parts of one head
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) S[mt][c] += __shfl_xor_sync(kFull, S[mt][c], 2);
      Ck[0] += __shfl_xor_sync(kFull, Ck[0], 2);
      Ck[1] += __shfl_xor_sync(kFull, Ck[1], 2);
    }
    // score = acc * hinv + off with hinv > 0, so the max is taken on the raw
    // accumulators and p = 2^(acc * hinv + off - m) is one FMA and one ex2
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float off = hbias[h] - Ck[h] * hinv[h];
      float m = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) m = fmaxf(m, fmaxf(S[mt][h], S[mt][h + 2]));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
      const float m_new = fmaxf(mrun[h], fmaf(m, hinv[h], off));
      alpha[h] = ex2(mrun[h] - m_new);
      mrun[h] = m_new;
      const float shift = off - m_new;
      float ls = 0.0f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        S[mt][h] = ex2(fmaf(S[mt][h], hinv[h], shift));
        S[mt][h + 2] = ex2(fmaf(S[mt][h + 2], hinv[h], shift));
        ls += S[mt][h] + S[mt][h + 2];
      }
      lrun[h] = fmaf(lrun[h], alpha[h], ls);
    }
  }

  // Value-side tables of one group (values in vbuf): lane l handles tokens
  // 4l..4l+3.  Returns this group's units per j and the origin scale.
  __device__ __forceinline__ void value_tables(float (&svn)[4], float (&inv_svm)[4]) {
    const RecLayout& L = a.lay;
    const float* vscale = reinterpret_cast<const float*>(vbuf + (L.v_scale - L.kpart));
    const uint2* vmin2 = reinterpret_cast<const uint2*>(vbuf + (L.v_min - L.kpart));
    float vs[4][4], vmn[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = reinterpret_cast<const float4*>(vscale)[4 * lane + i];
      vs[i][0] = f.x; vs[i][1] = f.y; vs[i][2] = f.z; vs[i][3] = f.w;
      const uint2 m = vmin2[4 * lane + i];
      vmn[i][0] = bf2f(m.x & 0xffffu); vmn[i][1] = bf2f(m.x >> 16);
      vmn[i][2] = bf2f(m.y & 0xffffu); vmn[i][3] = bf2f(m.y >> 16);
    }
    float svm[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float mx = fmaxf(fmaxf(vs[0][j], vs[1][j]), fmaxf(vs[2][j], vs[3][j]));
      float mm = fmaxf(fmaxf(fabsf(vmn[0][j]), fabsf(vmn[1][j])),
                       fmaxf(fabsf(vmn[2][j]), fabsf(vmn[3][j])));
      mx = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(mx)));
      mm = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(mm)));
      float s_new, inv_new;
      pow2_norm(mx, s_new, inv_new);
      (void)inv_new;
      // the units of this group's P' never exceed the running ones
      svn[j] = fminf(s_new, sv[j]);
      pow2_norm(mm, svm[j], inv_svm[j]);
    }
    const int kt = lane >> 2, q4 = lane & 3;
    const int t0 = 2 * (q4 & 1), chi = q4 >> 1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float sc = svn[j];
      vsb[vsb_index(kt, t0, j, chi)] = pack_h2(vs[0][j] * sc, vs[1][j] * sc);
      vsb[vsb_index(kt, t0 + 1, j, chi)] = pack_h2(vs[2][j] * sc, vs[3][j] * sc);
      const float sm = svm[j];
      vmb[vmb_index(kt, j, t0, chi)] = pack_h2(vmn[0][j] * sm, vmn[1][j] * sm);
      vmb[vmb_index(kt, j, t0 + 1, chi)] = pack_h2(vmn[2][j] * sm, vmn[3][j] * sm);
    }
  }

  // P·V of one group (values in vbuf) into the running output.
  __device__ __forceinline__ void pv(float (&S)[8][4], const float (&alpha)[2]) {
    const RecLayout& L = a.lay;
    float svn[4], inv_svm[4];
    value_tables(svn, inv_svm);
    // running output to this group's units
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float ratio = svn[j] * inv_sv[j];
      const float f0 = alpha[0] * ratio, f1 = alpha[1] * ratio;
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        O[2 * j + mm][0] *= f0; O[2 * j + mm][2] *= f0;
        O[2 * j + mm][1] *= f1; O[2 * j + mm][3] *= f1;
      }
      sv[j] = svn[j];
      inv_sv[j] = pow2_rcp(svn[j]);
    }
    __syncwarp();   // value tables written by all lanes

    float Dvm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const uint8_t* vc = vbuf + (L.v_codes - L.kpart);
    uint32_t vw[8];
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      const uint32_t b0 = movmatrix_t(pack_h2(S[kt][0], S[kt][1]));
      const uint32_t b1 = movmatrix_t(pack_h2(S[kt][2], S[kt][3]));
      {
        const uint2 av = *reinterpret_cast<const uint2*>(vmb + vmb_index(kt, g & 3, t, 0));
        const uint32_t a0 = g < 4 ? av.x : 0u, a2 = g < 4 ? av.y : 0u;
        mma_f16(Dvm, a0, 0u, a2, 0u, b0, b1);
      }
      const uint4 vsA = *reinterpret_cast<const uint4*>(vsb + vsb_index(kt, t, 0, 0));
      const uint4 vsB = *reinterpret_cast<const uint4*>(vsb + vsb_index(kt, t, 2, 0));
      const uint32_t vsr[4][2] = {{vsA.x, vsA.y}, {vsA.z, vsA.w}, {vsB.x, vsB.y}, {vsB.z, vsB.w}};
      if (VB == 4 || (kt & 1) == 0) {
        const int row = VB == 2 ? (kt >> 1) : kt;
        const uint4 lo = *reinterpret_cast<const uint4*>(vc + ((row * 2 + 0) * 32 + lane) * 16);
        const uint4 hi = *reinterpret_cast<const uint4*>(vc + ((row * 2 + 1) * 32 + lane) * 16);
        vw[0] = lo.x; vw[1] = lo.y; vw[2] = lo.z; vw[3] = lo.w;
        vw[4] = hi.x; vw[5] = hi.y; vw[6] = hi.z; vw[7] = hi.w;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t bj0 = hmul2_u(b0, vsr[j][0]);
        const uint32_t bj1 = hmul2_u(b1, vsr[j][1]);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          const int mc = 2 * j + mm;
          uint32_t A[4];
          if (VB == 2) {
            if (kt & 1) unpack2_exact<1>(vw[mc], A);
            else unpack2_exact<0>(vw[mc], A);
          } else {
            unpack4_exact(vw[mc], A);
          }
          mma_f16(O[mc], A[0], A[1], A[2], A[3], bj0, bj1);
        }
      }
    }
    // origin term in true units (lanes g < 4 hold channel group j = g)
    {
      const float im = g == 0 ? inv_svm[0] : g == 1 ? inv_svm[1] : g == 2 ? inv_svm[2]
                       : g == 3 ? inv_svm[3] : 0.0f;
      vm[0] = fmaf(vm[0], alpha[0], Dvm[0] * im);
      vm[1] = fmaf(vm[1], alpha[1], Dvm[1] * im);
    }
  }

  // The bf16 residual window (r tokens) on CUDA cores, with the record
  // buffer as scratch.  Added into the same online-softmax state.
  __device__ __forceinline__ void residual(int u) {
    float* qf = reinterpret_cast<float*>(kbuf);             // [NREP][128], later o_r
    float* pb = qf + NREP * kD;                             // [NREP][128]
    const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
    __syncwarp();
    for (int i = lane; i < NREP * kD; i += 32) {
      const int h = i / kD, c = i % kD;
      qf[i] = SPARE ? static_cast<const float*>(qs)[h * kQRow + c]
                    : bf2f(static_cast<const uint16_t*>(qs)[h * kQRow + c]) * c0;
    }
    __syncwarp();
    const uint16_t* kr = a.res_k + static_cast<long long>(u) * kR * kD;
    const uint16_t* vr = a.res_v + static_cast<long long>(u) * kR * kD;
    float s[4][NREP];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tk = lane + 32 * i;
#pragma unroll
      for (int h = 0; h < NREP; ++h) s[i][h] = 0.0f;
      if (tk < a.r) {
        const uint4* row = reinterpret_cast<const uint4*>(kr + tk * kD);
        for (int c8 = 0; c8 < kD / 8; ++c8) {
          const uint4 w = __ldg(row + c8);
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float k0 = bf2f(wv[e] & 0xffffu), k1 = bf2f(wv[e] >> 16);
#pragma unroll
            for (int h = 0; h < NREP; ++h)
              s[i][h] = fmaf(qf[h * kD + c8 * 8 + 2 * e], k0,
                             fmaf(qf[h * kD + c8 * 8 + 2 * e + 1], k1, s[i][h]));
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < NREP; ++h) s[i][h] = -INFINITY;
      }
    }
    float alpha_all[NREP], lsum_all[NREP];
#pragma unroll
    for (int h = 0; h < NREP; ++h) {
      float m = fmaxf(fmaxf(s[0][h], s[1][h]), fmaxf(s[2][h], s[3][h]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
      const float m_old = __shfl_sync(kFull, mrun[h & 1], h >> 1);  // lane (0, h/2)
      const float m_new = fmaxf(m_old, m);
      alpha_all[h] = ex2(m_old - m_new);
      float ls = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float p = ex2(s[i][h] - m_new);
        ls += p;
        pb[h * kD + lane + 32 * i] = p;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(kFull, ls, o);
      lsum_all[h] = ls;
      if ((h >> 1) == t) mrun[h & 1] = m_new;
    }
    float al[2] = {1.0f, 1.0f}, lsn[2] = {0.0f, 0.0f};
#pragma unroll
    for (int h = 0; h < NREP; ++h) {
      if ((h >> 1) == t) {
        al[h & 1] = alpha_all[h];
        lsn[h & 1] = lsum_all[h];
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) lrun[h] = lrun[h] * al[h] + (g == 0 ? lsn[h] : 0.0f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (sv[j] == kSentinel) {   // no group in this segment: O is still zero
        sv[j] = 1.0f;
        inv_sv[j] = 1.0f;
      }
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        O[2 * j + mm][0] *= al[0]; O[2 * j + mm][2] *= al[0];
        O[2 * j + mm][1] *= al[1]; O[2 * j + mm][3] *= al[1];
      }
    }
    vm[0] *= al[0];
    vm[1] *= al[1];
    __syncwarp();
    // o_r[h][ch] for channels 4*lane .. 4*lane+3
    float o[NREP][4];
#pragma unroll
    for (int h = 0; h < NREP; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[h][e] = 0.0f;
    for (int tk = 0; tk < a.r; ++tk) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(vr + tk * kD + 4 * lane));
      const float v0 = bf2f(w.x & 0xffffu), v1 = bf2f(w.x >> 16);
      const float v2 = bf2f(w.y & 0xffffu), v3 = bf2f(w.y >> 16);
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        const float p = pb[h * kD + tk];
        o[h][0] = fmaf(p, v0, o[h][0]);
        o[h][1] = fmaf(p, v1, o[h][1]);
        o[h][2] = fmaf(p, v2, o[h][2]);
        o[h][3] = fmaf(p, v3, o[h][3]);
      }
    }
    float* ob = qf;   // q no longer needed
#pragma unroll
    for (int h = 0; h < NREP; ++h)
      *reinterpret_cast<float4*>(ob + h * kD + 4 * lane) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    __syncwarp();
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      const int j = mc >> 1;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int h = 2 * t + (c & 1);
        const int ch = 16 * mc + g + 8 * (c >> 1);
        if (h < NREP) O[mc][c] = fmaf(ob[h * kD + ch], sv[j], O[mc][c]);
      }
    }
    __syncwarp();
  }

  // Merge the lanes and write this unit's partial (o, m, l) per query head.
  __device__ __forceinline__ void finish(int u, int part) {
    float l[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float x = lrun[h];
      x += __shfl_xor_sync(kFull, x, 4);
      x += __shfl_xor_sync(kFull, x, 8);
      x += __shfl_xor_sync(kFull, x, 16);
      l[h] = x;
    }
    float* base = a.ws + (static_cast<long long>(u) * a.max_parts + part) * NREP * (kD + 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float vm0 = __shfl_sync(kFull, vm[0], 4 * j + t);
      const float vm1 = __shfl_sync(kFull, vm[1], 4 * j + t);
#pragma unroll
      for (int mm = 0; mm < 2; ++mm) {
        const int mc = 2 * j + mm;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int h = 2 * t + (c & 1);
          const int ch = 16 * mc + g + 8 * (c >> 1);
          const float val = O[mc][c] * inv_sv[j] + ((c & 1) ? vm1 : vm0);
          if (h < NREP) base[h * (kD + 2) + ch] = val;
        }
      }
    }
    if (g == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int hh = 2 * t + h;
        if (hh < NREP) {
          base[hh * (kD + 2) + kD] = mrun[h];
          base[hh * (kD + 2) + kD + 1] = l[h];
        }
      }
    }
  }
};

template <int KB, int VB, int NREP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) decode_mma_kernel(MmaArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int slot = blockIdx.x * WARPS + warp;
  if (slot >= a.n_slots) return;            // warp-uniform
  uint8_t* mine = smem + static_cast<size_t>(warp) * (a.rec_bytes + kWarpExtra);
  Warp<KB, VB, NREP> W(a, mine);
  const long long p0 = slot_start(a, slot), p1 = slot_start(a, slot + 1);
  for (int u = static_cast<int>(p0 / a.unit_len); u <= static_cast<int>((p1 - 1) / a.unit_len); ++u) {
    const long long ub = static_cast<long long>(u) * a.unit_len;
    const long long lo = max(p0, ub) - ub, hi = min(p1, ub + a.unit_len) - ub;
    const int g0 = static_cast<int>(lo);
    const int g1 = static_cast<int>(min(hi, static_cast<long long>(a.n_groups)));
    const bool res = a.r > 0 && lo <= a.n_groups && a.n_groups < hi;
    W.begin_unit(u);
    if (g0 < g1) {
      // keys of group i+1 load during the softmax and P·V of group i; values
      // of group i+1 during its QK.  One commit group per part, in order.
      W.issue_k(u, g0);
      asm volatile("cp.async.commit_group;\n" ::);
      W.issue_v(u, g0);
      asm volatile("cp.async.commit_group;\n" ::);
      for (int gi = g0; gi < g1; ++gi) {
        const bool more = gi + 1 < g1;
        asm volatile("cp.async.wait_group 1;\n" ::);   // keys of gi
        __syncwarp();
        float S[8][4], alpha[2];
        W.qk_softmax(S, alpha);
        __syncwarp();                                  // key part consumed
        if (more) W.issue_k(u, gi + 1);
        asm volatile("cp.async.commit_group;\n" ::);
        asm volatile("cp.async.wait_group 1;\n" ::);   // values of gi
        __syncwarp();
        W.pv(S, alpha);
        __syncwarp();                                  // value part consumed
        if (more) W.issue_v(u, gi + 1);
        asm volatile("cp.async.commit_group;\n" ::);
      }
      asm volatile("cp.async.wait_group 0;\n" ::);
      __syncwarp();
    }
    if (res) W.residual(u);
    W.finish(u, slot - slot_of(a, ub));
  }
}

__global__ void __launch_bounds__(128) combine_parts_kernel(const float* __restrict__ ws,
                                                           int Hkv, int Hq, int max_parts,
                                                           long long unit_len, long long total,
                                                           int n_slots, float* __restrict__ out) {
  const int row = blockIdx.x;                 // b * Hq + hq
  const int n_rep = Hq / Hkv;
  const int b = row / Hq, hq = row % Hq;
  const int u = b * Hkv + hq / n_rep, h = hq % n_rep;
  const long long ub = static_cast<long long>(u) * unit_len;
  const int first = static_cast<int>(((ub + 1) * n_slots - 1) / total);
  const int last = static_cast<int>(((ub + unit_len) * n_slots - 1) / total);
  const int n = last - first + 1;
  const float* base = ws + static_cast<long long>(u) * max_parts * n_rep * (kD + 2) + h * (kD + 2);
  const long long stride = static_cast<long long>(n_rep) * (kD + 2);
  float M = -INFINITY;
  for (int k = 0; k < n; ++k) M = fmaxf(M, base[k * stride + kD]);
  float o = 0.0f, l = 0.0f;
  for (int k = 0; k < n; ++k) {
    const float mk = base[k * stride + kD];
    if (mk == -INFINITY) continue;
    const float w = exp2f(mk - M);
    o = fmaf(w, base[k * stride + threadIdx.x], o);
    l = fmaf(w, base[k * stride + kD + 1], l);
  }
  out[static_cast<long long>(row) * kD + threadIdx.x] = o / l;
}

template <int KB, int VB, int NREP, int WARPS>
cudaError_t launch_cfg(const MmaArgs& a, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(WARPS) * (a.rec_bytes + kWarpExtra);
  auto kern = decode_mma_kernel<KB, VB, NREP, WARPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = (a.n_slots + WARPS - 1) / WARPS;
  kern<<<grid, WARPS * 32, smem, s>>>(a);
  return cudaGetLastError();
}

template <int KB, int VB, int WARPS>
cudaError_t launch_rep(const MmaArgs& a, int nrep, cudaStream_t s) {
  switch (nrep) {
    case 1: return launch_cfg<KB, VB, 1, WARPS>(a, s);
    case 2: return launch_cfg<KB, VB, 2, WARPS>(a, s);
    case 4: return launch_cfg<KB, VB, 4, WARPS>(a, s);
    case 8: return launch_cfg<KB, VB, 8, WARPS>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int mma_warps_per_cta(int rec_bytes) {
  // one record buffer plus the tables and the query per warp, within the
  // 227 KB of shared memory a block may use; at most 12 warps so a thread
  // keeps up to 168 registers
  const int per = rec_bytes + kWarpExtra;
  return max(1, min(12, (227 * 1024) / per));
}

bool mma_plan(int num_sms, int units, int n_rep, int n_groups, int r, int rec_bytes,
              size_t ws_cap, MmaPlan* plan) {
  plan->unit_len = n_groups + (r > 0 ? kResidualWeight : 0);
  const long long total = static_cast<long long>(units) * plan->unit_len;
  const long long resident = static_cast<long long>(num_sms) * mma_warps_per_cta(rec_bytes);
  long long slots = total < resident ? total : resident;
  if (ws_cap) {
    // each unit's positions meet at most ceil(slots / units) + 1 slots
    const size_t per_part = static_cast<size_t>(units) * n_rep * (kD + 2) * sizeof(float);
    const long long fit = static_cast<long long>(ws_cap / per_part);
    if (fit < 2) return false;
    const long long lim = static_cast<long long>(units) * (fit - 1);
    if (slots > lim) slots = lim;
  }
  plan->n_slots = static_cast<int>(slots);
  plan->max_parts = static_cast<int>((slots + units - 1) / units) + 1;
  return true;
}

size_t mma_ws_bytes(int num_sms, int B, int Hkv, int Hq, int max_groups, int rec_bytes) {
  // worst case over the lengths this cache can hold: one warp slot per
  // weighted position or all resident warps, whichever is fewer
  const int units = B * Hkv;
  const long long resident = static_cast<long long>(num_sms) * mma_warps_per_cta(rec_bytes);
  const long long per_unit = (resident + units - 1) / units + 2;
  const long long cap = static_cast<long long>(max_groups) + kResidualWeight + 1;
  const long long parts = per_unit < cap ? per_unit : cap;
  return static_cast<size_t>(units) * parts * (Hq / Hkv) * (kD + 2) * sizeof(float);
}

cudaError_t launch_decode_mma(const kvq_cache* c, const kvq_bf16* q, int Hq, float* out,
                              float* ws, const MmaPlan& plan, cudaStream_t s) {
  MmaArgs a;
  a.records = c->records;
  a.rec_bytes = c->lay.bytes;
  a.max_groups = c->max_groups;
  a.lay = c->lay;
  a.n_groups = c->t_q / kKG;
  a.r = c->r;
  a.res_k = c->res_k;
  a.res_v = c->res_v;
  a.q = q;
  a.Hkv = c->cfg.kv_heads;
  a.Hq = Hq;
  a.units = c->cfg.batch * c->cfg.kv_heads;
  a.unit_len = plan.unit_len;
  a.n_slots = plan.n_slots;
  a.max_parts = plan.max_parts;
  a.total = static_cast<long long>(a.units) * a.unit_len;
  a.ws = ws;
  const int nrep = Hq / c->cfg.kv_heads;
  const int kb = c->cfg.k_bits, vb = c->cfg.v_bits;
  if (mma_warps_per_cta(c->lay.bytes) != (kb == 2 && vb == 2 ? 12 : kb == 4 && vb == 4 ? 9 : 11))
    return cudaErrorInvalidConfiguration;
  cudaError_t e;
  if (kb == 2 && vb == 2) e = launch_rep<2, 2, 12>(a, nrep, s);
  else if (kb == 2 && vb == 4) e = launch_rep<2, 4, 11>(a, nrep, s);
  else if (kb == 4 && vb == 2) e = launch_rep<4, 2, 11>(a, nrep, s);
  else e = launch_rep<4, 4, 9>(a, nrep, s);
  if (e != cudaSuccess) return e;
  combine_parts_kernel<<<c->cfg.batch * Hq, kD, 0, s>>>(ws, a.Hkv, Hq, a.max_parts, a.unit_len,
                                                        a.total, a.n_slots, out);
  return cudaGetLastError();
}

}  // namespace kvq
