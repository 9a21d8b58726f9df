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
// A pair of codes becomes an f16x2 register with one AND (frag_layout.h):
// the masked half is the subnormal c * 2^(pos - 24), exact, and the B rows
// that meet it carry 2^(15 - pos), so every product is c * B' * 2^-9 with
// B' the normalized Q' or P' entry.  No offset enters the sums, so the
// running output accumulates across groups in the MMA accumulators.
// Q' and P' are normalized by powers of two per group (and V channel group)
// so every f16 operand stays in range (at most 2^15) for any bf16 input.
// Scores need more than f16's 11 bits of Q' (a large score's error is its
// size times the operand rounding), so Q' is split into an f16 high part
// and an f16 low part (the rounding error of the high part), ~22 bits in
// all: with at most 4 query heads per KV head, B column 2h holds head h's
// high part and column 2h + 1 its low part, so a lane's two accumulator
// columns are one head and one add merges them (the softmax then runs once
// per score, on lane (g, t) for head t); with 8 heads a second MMA per
// k-step adds the low part.
//
// Work split ("stream-K"): the flattened sequence of items (for each unit
// its groups, then its residual window and its attention-sink window, one
// item each) is cut into equal contiguous slices, one per warp, and
// consecutive slices run on different SMs; a warp keeps one online-softmax
// state per unit it touches and writes one partial per unit.  Each warp
// stages one record at a time in its own shared memory, in two parts: the
// key part of the next group loads while the current group's softmax and
// P·V run, the value part of the next group while its QK runs.  Warps never
// wait on each other.  The combine kernels merge each query head's partials
// with the exact log-sum-exp rule.
#pragma once

#include <atomic>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "frag_layout.h"
#include "kvq_internal.h"
#include "mma_util.h"

namespace kvq {

// Arguments of one decode launch (one type for every translation unit that
// instantiates the kernel).
struct MmaArgs {
  const uint8_t* records;
  long long rec_bytes;
  int max_groups;
  RecLayout lay;
  int n_groups;           // quantized groups per unit
  int r;                  // residual tokens
  const uint16_t* res_k;  // [units][128][D]
  const uint16_t* res_v;
  int s, n_sink;          // sink tokens, sink window capacity
  const uint16_t* sink_k; // [units][n_sink][D]
  const uint16_t* sink_v;
  const uint16_t* q;      // [B][Hq][D]
  const uint4* new_k;     // fused append: token [units][D] for residual slot r - 1 (or NULL)
  const uint4* new_v;
  int Hkv, Hq, units;
  long long unit_len;     // weighted positions per unit
  long long total;        // units * unit_len
  int n_slots;            // warps with work
  int max_parts;          // partial slots per unit in ws
  float* ws;              // [units][max_parts][NREP][D + 2]
  unsigned* status;       // sticky KVQ_FLAG_* word of the cache
  int wait_polls;         // try_wait polls before a wait for a staged part gives up
  const uint8_t* perm;    // PN-Mix: [units][D] stored position -> channel
};

cudaError_t launch_decode_kivi(const MmaArgs& a, int nrep, int bits, int warps, cudaStream_t s);
cudaError_t launch_decode_pnmix(const MmaArgs& a, int nrep, int vbits, int warps, cudaStream_t s);

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
// Split positions of a bf16 window item (the residual or the sink; a group
// is 1): a window's 16-token chunks stream through two buffer slots, so it
// takes about as long as two groups, and slices holding one get fewer.
constexpr int kResidualWeight = 2;
constexpr float kSentinel = 4.2535295865117308e37f;  // 2^125: "no group yet"
constexpr float kCodeUnit = 512.0f;      // 2^9: products carry c * B' / 2^9
constexpr float kInvCodeUnit = 1.0f / 512.0f;

// Per-warp shared memory after the record buffer (key part, then value
// part): with mixed keys the value-step table (256 words) and the
// value-origin table (4 rows of 72 words), then the unit's query, [8
// heads][136] bf16 or, with at most 4 heads per KV head, [4 heads][136] fp32
// pre-scaled by log2(e)/sqrt(D) (rows padded so head rows fall in different
// banks).  The padding of the first row, never read as query, holds the 16
// zero bytes ldmatrix reads for absent rows.  With uniform keys the two
// value tables are built in place over the staged value steps and origins
// they are computed from (3072 bytes, read into registers first).
constexpr int kVsbBytes = 256 * 4;
constexpr int kVmbBytes = 4 * 72 * 4;   // 4 origin rows
constexpr int kQRow = 136;
constexpr int kQBytes = 8 * kQRow * 2;   // = 4 * kQRow * 4
static_assert(kVsbBytes + kVmbBytes <= 4 * kKG * kVGroups + 2 * kKG * kVGroups,
              "value tables must fit over the staged value metadata");
// Per-warp regions stay multiples of 128 bytes: cp.async copies of 128-byte
// aligned record lines into misaligned shared memory cost ~10% of the
// decode time.
__host__ __device__ constexpr int warp_extra(bool mix) {
  return (mix ? kVsbBytes + kVmbBytes : 0) + kQBytes;
}
static_assert(warp_extra(false) % 128 == 0 && warp_extra(true) % 128 == 0,
              "per-warp extra must keep 128-byte alignment");
// Warps per block.  Two-bit uniform records with at most 4 query heads per
// KV head fit 16 warps (4 per scheduler, up to 128 registers a thread) in
// shared memory; the other variants run 12 (up to 168 registers).
__host__ __device__ constexpr int max_warps(int kb, int vb, int nrep, bool mix) {
  return (!mix && kb == 2 && vb == 2 && nrep <= 4) ? 16 : 12;
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

// --- code unpacking: word x and y = x >> 8 -> A fragment registers
// (frag_layout.h).  Each register is one AND; its halves are f16 subnormals.
// B-row factor of register pair (a0, a1) / (a2, a3) is 2^(15 - pos).
template <int KL>
__device__ __forceinline__ void unpack2(uint32_t x, uint32_t y, uint32_t (&a)[4]) {
  constexpr uint32_t Mb = 0x00030003u << (4 * KL), Mt = 0x000C000Cu << (4 * KL);
  a[0] = x & Mb;
  a[1] = y & Mb;
  a[2] = x & Mt;
  a[3] = y & Mt;
}
__device__ __forceinline__ void unpack4(uint32_t x, uint32_t y, uint32_t (&a)[4]) {
  constexpr uint32_t Mb = 0x000F000Fu, Mt = 0x00F000F0u;
  a[0] = x & Mb;
  a[1] = y & Mb;
  a[2] = x & Mt;
  a[3] = y & Mt;
}
// PN-Mix LSB plane (1 bit a code): a word holds four k-steps (k_local4 =
// k & 3); registers a0, a2 from x, a1, a3 from y = x >> 8, each masked to
// the bits 2 * k_local4 + (reg >> 1) of both halves.
template <int KL4>
__device__ __forceinline__ void unpack1(uint32_t x, uint32_t y, uint32_t (&a)[4]) {
  constexpr uint32_t Mb = 0x00010001u << (2 * KL4), Mt = 0x00020002u << (2 * KL4);
  a[0] = x & Mb;
  a[1] = y & Mb;
  a[2] = x & Mt;
  a[3] = y & Mt;
}
// 2^(15 - pos) for B rows b0 (slot 0: rows 2t, 2t+1) and b1 (slot 1: rows
// 2t+8, 2t+9) of k-step k (BITS = 1: the PN-Mix LSB plane).
template <int BITS>
__host__ __device__ constexpr float row_factor(int k, int slot) {
  return BITS == 2   ? static_cast<float>(1 << (15 - 4 * (k & 1) - 2 * slot))
         : BITS == 1 ? static_cast<float>(1 << (15 - 2 * (k & 3) - slot))
                     : static_cast<float>(1 << (15 - 4 * slot));
}


// mbarrier helpers for the bulk staging of records.
__device__ __forceinline__ void mbar_init(uint32_t mb) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(mb) : "memory");
}
// Wait for phase `parity` of mbarrier mb; false if it did not complete
// within `polls` polls (each try_wait also suspends for a while).
constexpr int kWaitPolls = 1 << 20;
__device__ __forceinline__ bool mbar_wait(uint32_t mb, uint32_t parity, int polls) {
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

// Bring `bytes` (a multiple of 16) at p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, int bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ long long slot_start(const MmaArgs& a, int w) {
  return (static_cast<long long>(w) * a.total) / a.n_slots;
}
__device__ __forceinline__ int slot_of(const MmaArgs& a, long long p) {
  return static_cast<int>(((p + 1) * a.n_slots - 1) / a.total);
}

template <int KB, int VB, int NREP, bool MIX, bool KIVI = false, bool PNMIX = false>
struct Warp {
  static constexpr bool SEP = MIX || KIVI;  // value tables in their own area
  static constexpr bool SPARE = NREP <= 4;  // Q' low part in odd columns;
                                            // query kept as pre-scaled fp32
  static constexpr int NL = SPARE ? 1 : 8;  // low-part fragments kept

  const MmaArgs& a;
  const int lane, g, t;
  uint8_t* kbuf;   // key part of the staged record
  uint8_t* vbuf;   // value part of the staged record
  uint32_t* vsb;   // value-step table, B order (vsb_index)
  uint32_t* vmb;   // value-origin table, A order (vmb_index)
  void* qs;        // the unit's query (see kQBytes)
  uint32_t mb_k, mb_v;        // mbarriers of the staged key / value parts
  uint32_t ph_k = 0, ph_v = 0;  // their current phase parities
  // mixed keys only:
  const uint16_t* qg_row;  // this lane's query head (g, capped at NREP - 1) in global memory
  float qmax;      // max |query| of the head row this lane builds B columns for

  // online-softmax state (heads 2t, 2t+1 of this lane)
  // Running O^T in units of sv / 2^9: channel tiles mc = 0..7, or with at
  // most 4 heads only the 4 tiles whose accumulator columns this lane keeps
  // (tile_of: channel groups of odd j keep columns 4..7, lanes t >= 2).
  static constexpr int NO = SPARE ? 4 : 8;
  float O[NO][4];
  float vm[2];     // origin term (lanes g < 4: channel group j = g)
  float mrun[2], lrun[2];
  float sv, inv_sv;  // current units of O

  __device__ __forceinline__ Warp(const MmaArgs& args, uint8_t* base)
      : a(args), lane(threadIdx.x & 31), g((threadIdx.x & 31) >> 2), t(threadIdx.x & 3) {
    const int rb = static_cast<int>(a.rec_bytes);
    kbuf = base;
    vbuf = base + a.lay.kpart;
    uint8_t* tables = SEP ? base + rb : vbuf + (a.lay.v_scale - a.lay.kpart);
    vsb = reinterpret_cast<uint32_t*>(tables);
    vmb = reinterpret_cast<uint32_t*>(tables + kVsbBytes);
    qs = base + rb + (SEP ? kVsbBytes + kVmbBytes : 0);
    // the two mbarriers sit in the padding of query row 1
    mb_k = static_cast<uint32_t>(__cvta_generic_to_shared(qs)) + (SPARE ? (kQRow + kD) * 4 : (kQRow + kD) * 2);
    mb_v = mb_k + 8;
    if (lane == 0) {
      mbar_init(mb_k);
      mbar_init(mb_v);
      asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncwarp();
    if (MIX) {
      if (lane < 4) reinterpret_cast<uint32_t*>(zero_row())[lane] = 0u;
      __syncwarp();
    }
  }

  // 16 zero bytes in the padding of query row 0 (fp32 rows: 128 floats used
  // of 136; bf16 rows: 128 of 136)
  __device__ __forceinline__ uint8_t* zero_row() const {
    return static_cast<uint8_t*>(qs) + (SPARE ? kD * 4 : kD * 2);
  }

  // Channel tile of output slot i (see O).
  __device__ __forceinline__ int tile_of(int i) const {
    return SPARE ? 4 * (i >> 1) + (i & 1) + 2 * (t >> 1) : i;
  }

  // Query head of the B column this lane builds (column g): with at most 4
  // heads, column 2h holds head h's high part and column 2h + 1 its low
  // part; with 8 heads column g is head g.
  __device__ __forceinline__ int hrow() const { return SPARE ? (g >> 1) : g; }
  __device__ __forceinline__ bool low_col() const { return SPARE && (g & 1); }
  // Lane of this lane's quad holding head hh's scores (one head per lane,
  // at most 4 heads): lane (g, hh & 3).
  __device__ __forceinline__ int head_lane(int hh) const { return (lane & ~3) | (hh & 3); }

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
    if (MIX) qg_row = qg + min(hrow(), NREP - 1) * kD;
    const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
    __syncwarp();
    if (SPARE) {   // fp32 [4][kQRow], pre-scaled; lane = 16 channels of one head
      float* q = static_cast<float*>(qs);
      const int h = lane >> 3, c = (lane & 7) * 16;
      float v[16];
      if (h >= NREP) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
      } else if (PNMIX) {   // the unit's stored channel order
        const uint8_t* pm = a.perm + static_cast<long long>(u) * kD + c;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = bf2f(qg[h * kD + pm[i]]) * c0;
      } else if ((reinterpret_cast<uintptr_t>(a.q) & 15) == 0) {
        const uint4* src = reinterpret_cast<const uint4*>(qg + h * kD + c);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint4 w = __ldg(src + k);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[8 * k + 2 * i] = bf2f(ww[i] & 0xffffu) * c0;
            v[8 * k + 2 * i + 1] = bf2f(ww[i] >> 16) * c0;
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = bf2f(qg[h * kD + c + i]) * c0;
      }
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(q + h * kQRow + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {       // bf16 [8][kQRow]; lane = 8-channel pieces lane + 32 i of the 128
      // all loads are issued before any store: at the start of a call they
      // queue behind every warp's first records, so one round trip, not 16
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int piece = lane + 32 * i, h = piece >> 4, c = (piece & 15) * 8;
        if (PNMIX) {   // the unit's stored channel order
          const uint8_t* pm = a.perm + static_cast<long long>(u) * kD + c;
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(qg[h * kD + pm[2 * k]]) |
                   (static_cast<uint32_t>(qg[h * kD + pm[2 * k + 1]]) << 16);
          v[i] = make_uint4(w[0], w[1], w[2], w[3]);
        } else if ((reinterpret_cast<uintptr_t>(a.q) & 15) == 0) {
          v[i] = __ldg(reinterpret_cast<const uint4*>(qg + h * kD + c));
        } else {
          const uint16_t* src = qg + h * kD + c;   // any 2-byte aligned q
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(src[2 * k]) | (static_cast<uint32_t>(src[2 * k + 1]) << 16);
          v[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      uint16_t* q = static_cast<uint16_t*>(qs);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int piece = lane + 32 * i, h = piece >> 4, c = (piece & 15) * 8;
        *reinterpret_cast<uint4*>(q + h * kQRow + c) = v[i];
      }
    }
    __syncwarp();
    if (MIX) {   // max |q| of this lane's head row (fp32 pre-scaled, or bf16)
      float mx = 0.0f;
      for (int c = t; c < kD; c += 4)
        mx = fmaxf(mx, SPARE ? fabsf(static_cast<const float*>(qs)[hrow() * kQRow + c])
                             : fabsf(bf2f(static_cast<const uint16_t*>(qs)[g * kQRow + c])));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      qmax = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    }
#pragma unroll
    for (int m = 0; m < NO; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) O[m][c] = 0.0f;
    sv = kSentinel;
    inv_sv = 1.0f / kSentinel;
    vm[0] = vm[1] = 0.0f;
    mrun[0] = mrun[1] = -INFINITY;
    lrun[0] = lrun[1] = 0.0f;
  }

  // Bytes [lo, hi) of group record grp of unit u into dst with one bulk
  // copy issued by lane 0, completing on mbarrier mb (the warp has read
  // dst's previous contents: __syncwarp before, then the proxy fence).
  __device__ __forceinline__ void issue(int u, int grp, uint8_t* dst, int lo, int hi, uint32_t mb) {
    // every lane orders its earlier shared-memory accesses (reads of the
    // buffer, the in-place tables) before the copy that overwrites them
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const uint8_t* src = a.records + (static_cast<long long>(u) * a.max_groups + grp) * a.rec_bytes + lo;
      const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
      const uint32_t bytes = static_cast<uint32_t>(hi - lo);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mb), "r"(bytes)
                   : "memory");
      // records are read once per call: first out of L2, which keeps the
      // split-K partials there for the combine
      uint64_t pol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
          " [%0], [%1], %2, [%3], %4;\n"
          ::"r"(d), "l"(src), "r"(bytes), "r"(mb), "l"(pol)
          : "memory");
    }
  }
  __device__ __forceinline__ void issue_k(int u, int grp) { issue(u, grp, kbuf, 0, a.lay.kpart, mb_k); }
  __device__ __forceinline__ void issue_v(int u, int grp) {
    issue(u, grp, vbuf, a.lay.kpart, static_cast<int>(a.rec_bytes), mb_v);
  }
  // Wait for the staged key (value) part; on a timeout record the flag and
  // return false (the caller stops; the copy in flight is then waited for
  // with the full limit, so it has landed before the warp leaves).
  __device__ __forceinline__ bool wait_part(uint32_t mb, uint32_t& phase) {
    const bool ok = mbar_wait(mb, phase, a.wait_polls);
    phase ^= 1u;
    if (!ok) {
      if (lane == 0) atomicOr(a.status, static_cast<unsigned>(KVQ_FLAG_TIMEOUT));
      mbar_wait(mb, phase ^ 1u, kWaitPolls);
    }
    return ok;
  }

  // Scores of one group (keys in kbuf) in C-fragment layout, with their
  // unit hinv and origin term hbias per head (the softmax comes later).
  __device__ __forceinline__ void scores(float (&S)[8][4], float (&hinv)[2], float (&hbias)[2]) {
    if constexpr (KIVI) {
      scores_kivi(S, hinv, hbias);
      return;
    }
    if constexpr (MIX) scores_mixed(S, hinv, hbias);
    else if constexpr (PNMIX) scores_pnmix(S, hinv, hbias);
    else scores_uniform(S, hinv, hbias);
    if (SPARE) {   // columns 2t and 2t + 1: the high and low parts of head t
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        S[mt][0] += S[mt][1];
        S[mt][2] += S[mt][3];
      }
    }
  }

  // Q' = q * step * log2(e)/sqrt(D) of one key record (or sub-group) as B
  // fragments: steps of channels c, c + 1 from step2(c) (c even), bf16
  // origins in pairs from kmin2.  Also the unit inv_sq of the scores (per
  // head, on the lane that builds its high column) and the origin term
  // bias = sum_ch q m (log2 units, shared by a head's lanes).
  template <class StepPair>
  __device__ __forceinline__ void build_q(StepPair step2, const uint32_t* kmin2,
                                          uint32_t (&bq)[8][2], uint32_t (&bl)[NL][2],
                                          float& inv_sq, float& bias) {
    float sq;
    bias = 0.0f;
    if constexpr (SPARE) {
      // The two lanes of a head (columns 2h: high part, 2h + 1: low part)
      // share the work: the even lane takes the rows of b0 (channels 2t,
      // 2t + 1 of each k-step), the odd lane those of b1 (2t + 8, 2t + 9);
      // each rounds its Q' into high and low parts and hands the part it
      // does not keep to its partner (lane ^ 4) in one shuffle per k-step.
      const int par = g & 1;
      const int c_off = 2 * t + 8 * par;
      const float* qrow = static_cast<const float*>(qs) + hrow() * kQRow;
      float qk[16];
      float mx = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const float2 sc = step2(16 * ks + c_off);
        const float2 qv = *reinterpret_cast<const float2*>(qrow + 16 * ks + c_off);
        const uint32_t m2 = kmin2[8 * ks + t + 4 * par];
        qk[2 * ks + 0] = qv.x * sc.x;
        qk[2 * ks + 1] = qv.y * sc.y;
        bias = fmaf(qv.x, bf16_lo(m2), bias);
        bias = fmaf(qv.y, bf16_hi(m2), bias);
        mx = max3_abs(mx, qk[2 * ks], qk[2 * ks + 1]);
      }
      mx = fabsf(mx);
#pragma unroll
      for (int x = 1; x <= 4; x <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, x));
        bias += __shfl_xor_sync(kFull, bias, x);
      }
      pow2_norm(mx, sq, inv_sq);
      // the row factor of this lane's slot (b0 or b1), times the norm
      const float sp = sq * (par ? row_factor<KB>(0, 1) : row_factor<KB>(0, 0));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const float f = sp * (row_factor<KB>(ks, 0) / row_factor<KB>(0, 0));
        const float x0 = qk[2 * ks] * f, x1 = qk[2 * ks + 1] * f;
        // high part: x rounded to f16; low part: the (exact) rest, rounded
        const uint32_t H = pack_h2(x0, x1);
        const float2 hf = h2_to_f2(H);
        const uint32_t Lo = pack_h2(x0 - hf.x, x1 - hf.y);
        const uint32_t recv = __shfl_xor_sync(kFull, par ? H : Lo, 4);
        bq[ks][0] = par ? recv : H;
        bq[ks][1] = par ? Lo : recv;
      }
    } else {
      float qk[32];
      float mx = 0.0f;
      const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
      const uint32_t* qrow = static_cast<const uint32_t*>(qs) + g * (kQRow / 2);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const float2 s01 = step2(16 * ks + 2 * t);
        const float2 s89 = step2(16 * ks + 2 * t + 8);
        const uint32_t m01 = kmin2[8 * ks + t];
        const uint32_t m89 = kmin2[8 * ks + t + 4];
        const uint32_t q01 = qrow[8 * ks + t], q89 = qrow[8 * ks + t + 4];
        const float qa = bf16_lo(q01) * c0, qb = bf16_hi(q01) * c0;
        const float qc = bf16_lo(q89) * c0, qd = bf16_hi(q89) * c0;
        qk[4 * ks + 0] = qa * s01.x;
        qk[4 * ks + 1] = qb * s01.y;
        qk[4 * ks + 2] = qc * s89.x;
        qk[4 * ks + 3] = qd * s89.y;
        bias = fmaf(qa, bf16_lo(m01), bias);
        bias = fmaf(qb, bf16_hi(m01), bias);
        bias = fmaf(qc, bf16_lo(m89), bias);
        bias = fmaf(qd, bf16_hi(m89), bias);
        mx = max3_abs(mx, max3_abs(qk[4 * ks], qk[4 * ks + 1], qk[4 * ks + 2]), qk[4 * ks + 3]);
      }
      mx = fabsf(mx);
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      bias += __shfl_xor_sync(kFull, bias, 1);
      bias += __shfl_xor_sync(kFull, bias, 2);
      pow2_norm(mx, sq, inv_sq);
      // B' = Q' * sq in [0, 1), times the row factor of its code position;
      // high part: B' rounded to f16 precision, low part: the rest
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const float f0 = sq * row_factor<KB>(ks, 0), f1 = sq * row_factor<KB>(ks, 1);
        float x[4] = {qk[4 * ks + 0] * f0, qk[4 * ks + 1] * f0, qk[4 * ks + 2] * f1,
                      qk[4 * ks + 3] * f1};
        bq[ks][0] = pack_h2(x[0], x[1]);
        bq[ks][1] = pack_h2(x[2], x[3]);
        const float2 h01 = h2_to_f2(bq[ks][0]), h23 = h2_to_f2(bq[ks][1]);
        bl[ks % NL][0] = pack_h2(x[0] - h01.x, x[1] - h01.y);
        bl[ks % NL][1] = pack_h2(x[2] - h23.x, x[3] - h23.y);
      }
    }
  }

  // Per head of this lane's C columns: the score unit and origin term from
  // the lane that built that head's (high) B column.
  __device__ __forceinline__ void head_units(float inv_sq, float bias, float (&hinv)[2],
                                             float (&hbias)[2]) const {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int src = SPARE ? 8 * t : 4 * (2 * t + h);
      hinv[h] = __shfl_sync(kFull, inv_sq, src) * kCodeUnit;
      hbias[h] = __shfl_sync(kFull, bias, src);
    }
  }

  // QK on tensor cores for the key m-tiles MT0 .. MT0 + NMT - 1, k-step
  // outer: NMT independent accumulator chains (S zeroed first).
  template <int MT0, int NMT>
  __device__ __forceinline__ void qk_tiles(float (&S)[8][4], const uint32_t (&bq)[8][2],
                                           const uint32_t (&bl)[NL][2]) const {
#pragma unroll
    for (int mt = MT0; mt < MT0 + NMT; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[mt][c] = 0.0f;
    const uint8_t* kc = kbuf + a.lay.k_codes;
    if (KB == 2) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t kx[NMT], ky[NMT];
#pragma unroll
        for (int i = 0; i < NMT; ++i) {
          kx[i] = reinterpret_cast<const uint32_t*>(kc)[((MT0 + i) * 4 + w) * 32 + lane];
          ky[i] = kx[i] >> 8;
        }
#pragma unroll
        for (int kl = 0; kl < 2; ++kl) {
          const int ks = 2 * w + kl;
#pragma unroll
          for (int i = 0; i < NMT; ++i) {
            uint32_t A[4];
            if (kl) unpack2<1>(kx[i], ky[i], A);
            else unpack2<0>(kx[i], ky[i], A);
            qk_mma(S[MT0 + i], A, bq, bl, ks);
          }
        }
      }
    } else {
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint2 kw[NMT];
#pragma unroll
        for (int i = 0; i < NMT; ++i)
          kw[i] = reinterpret_cast<const uint2*>(kc)[((MT0 + i) * 4 + kp) * 32 + lane];
#pragma unroll
        for (int kl = 0; kl < 2; ++kl) {
          const int ks = 2 * kp + kl;
#pragma unroll
          for (int i = 0; i < NMT; ++i) {
            const uint32_t x = kl ? kw[i].y : kw[i].x;
            uint32_t A[4];
            unpack4(x, x >> 8, A);
            qk_mma(S[MT0 + i], A, bq, bl, ks);
          }
        }
      }
    }
  }

  // Uniform keys: score accumulators S (code units), their unit hinv and the
  // origin term hbias per head of this lane's C columns, in log2 units.
  __device__ __forceinline__ void scores_uniform(float (&S)[8][4], float (&hinv)[2],
                                                 float (&hbias)[2]) {
    const float* kscale = reinterpret_cast<const float*>(kbuf + a.lay.k_scale);
    const uint32_t* kmin2 = reinterpret_cast<const uint32_t*>(kbuf + a.lay.k_min);
    uint32_t bq[8][2], bl[NL][2];
    float inv_sq, bias;
    build_q([&](int c) { return *reinterpret_cast<const float2*>(kscale + c); }, kmin2, bq, bl,
            inv_sq, bias);
    head_units(inv_sq, bias, hinv, hbias);
    qk_tiles<0, 8>(S, bq, bl);
  }

  // PN-Mix H3/L1 keys (PN-Mix reproduction notes, Eq. 2, Eq. 7, App. G), in
  // the unit's stored channel order (the query in shared memory is in it
  // too): a code is c = c0 + 2 c12 with c0 its LSB (every channel) and c12
  // its upper two bits (the nh high channels, stored first), so
  //   s = sum_p q_p z_p + sum_p (q_p s_p) c0_p + sum_{p < nh} (2 q_p s_p) c12_p
  // with z the origins / Eq. 7 offsets and s the steps / Eq. 7 scales.  The
  // LSB plane runs as 1-bit codes over all eight k-steps, the upper plane as
  // 2-bit codes over the first nh / 16; one power-of-two unit for both.
  __device__ __forceinline__ void scores_pnmix(float (&S)[8][4], float (&hinv)[2],
                                               float (&hbias)[2]) {
    const RecLayout& L = a.lay;
    const float* ksc = reinterpret_cast<const float*>(kbuf + L.k_scale);
    const float* kof = reinterpret_cast<const float*>(kbuf + L.k_min);
    const int nh16 = L.nh >> 4;   // upper-plane k-steps
    uint32_t b1[8][2], b2[8][2], l1[NL][2], l2[NL][2];
    float sq, inv_sq, bias = 0.0f;
    const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
    // Q' of this lane's rows (SPARE: 16 channels of one head, the pair's two
    // lanes splitting b0 / b1 rows; else 32 channels of head g)
    constexpr int NQ = SPARE ? 16 : 32;
    float qk[NQ];
    float mx = 0.0f;
    const int par = g & 1;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int j = 0; j < (SPARE ? 2 : 4); ++j) {
        const int ch = SPARE ? 16 * ks + 2 * t + 8 * par + j : 16 * ks + 2 * t + (j & 1) + 8 * (j >> 1);
        const float qv = SPARE ? static_cast<const float*>(qs)[hrow() * kQRow + ch]
                               : bf2f(static_cast<const uint16_t*>(qs)[g * kQRow + ch]) * c0;
        const float x = qv * ksc[ch];
        bias = fmaf(qv, kof[ch], bias);
        qk[(SPARE ? 2 : 4) * ks + j] = x;
        mx = fmaxf(mx, fabsf(x) * (ch < L.nh ? 2.0f : 1.0f));
      }
    }
    if (SPARE) {
#pragma unroll
      for (int x = 1; x <= 4; x <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, x));
        bias += __shfl_xor_sync(kFull, bias, x);
      }
    } else {
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      bias += __shfl_xor_sync(kFull, bias, 1);
      bias += __shfl_xor_sync(kFull, bias, 2);
    }
    pow2_norm(mx, sq, inv_sq);
    // B fragments of both planes: x * sq * row factor (times 2 for the upper
    // plane), split into an f16 high part and an f16 low part
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int plane = 0; plane < 2; ++plane) {
        if (plane == 1 && ks >= nh16) continue;
        if constexpr (SPARE) {
          const float f = sq * (plane ? 2.0f * row_factor<2>(ks, par) : row_factor<1>(ks, par));
          const float x0 = qk[2 * ks] * f, x1 = qk[2 * ks + 1] * f;
          const uint32_t H = pack_h2(x0, x1);
          const float2 hf = h2_to_f2(H);
          const uint32_t Lo = pack_h2(x0 - hf.x, x1 - hf.y);
          const uint32_t recv = __shfl_xor_sync(kFull, par ? H : Lo, 4);
          uint32_t (&bb)[8][2] = plane ? b2 : b1;
          bb[ks][0] = par ? recv : H;
          bb[ks][1] = par ? Lo : recv;
        } else {
          const float f0 = sq * (plane ? 2.0f * row_factor<2>(ks, 0) : row_factor<1>(ks, 0));
          const float f1 = sq * (plane ? 2.0f * row_factor<2>(ks, 1) : row_factor<1>(ks, 1));
          const float x[4] = {qk[4 * ks] * f0, qk[4 * ks + 1] * f0, qk[4 * ks + 2] * f1,
                              qk[4 * ks + 3] * f1};
          uint32_t (&bb)[8][2] = plane ? b2 : b1;
          uint32_t (&ll)[NL][2] = plane ? l2 : l1;
          bb[ks][0] = pack_h2(x[0], x[1]);
          bb[ks][1] = pack_h2(x[2], x[3]);
          const float2 h01 = h2_to_f2(bb[ks][0]), h23 = h2_to_f2(bb[ks][1]);
          ll[ks % NL][0] = pack_h2(x[0] - h01.x, x[1] - h01.y);
          ll[ks % NL][1] = pack_h2(x[2] - h23.x, x[3] - h23.y);
        }
      }
    }
    head_units(inv_sq, bias, hinv, hbias);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[mt][c] = 0.0f;
    // LSB plane: word (mt*2 + ks/4)*32 + lane, four k-steps a word
    const uint32_t* lsb = reinterpret_cast<const uint32_t*>(kbuf + L.k_codes);
#pragma unroll
    for (int kq = 0; kq < 2; ++kq) {
      uint32_t kx[8], ky[8];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        kx[mt] = lsb[(mt * 2 + kq) * 32 + lane];
        ky[mt] = kx[mt] >> 8;
      }
#pragma unroll
      for (int kl4 = 0; kl4 < 4; ++kl4) {
        const int ks = 4 * kq + kl4;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t A[4];
          if (kl4 == 0) unpack1<0>(kx[mt], ky[mt], A);
          else if (kl4 == 1) unpack1<1>(kx[mt], ky[mt], A);
          else if (kl4 == 2) unpack1<2>(kx[mt], ky[mt], A);
          else unpack1<3>(kx[mt], ky[mt], A);
          qk_mma(S[mt], A, b1, l1, ks);
        }
      }
    }
    // upper plane: 2-bit words (mt*kw2 + w)*32 + lane over the first nh channels
    const uint32_t* up = reinterpret_cast<const uint32_t*>(kbuf + L.kc);
    const int kw2 = L.kw2;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (w >= kw2) break;
      uint32_t kx[8], ky[8];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        kx[mt] = up[(mt * kw2 + w) * 32 + lane];
        ky[mt] = kx[mt] >> 8;
      }
#pragma unroll
      for (int kl = 0; kl < 2; ++kl) {
        const int ks = 2 * w + kl;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t A[4];
          if (kl) unpack2<1>(kx[mt], ky[mt], A);
          else unpack2<0>(kx[mt], ky[mt], A);
          qk_mma(S[mt], A, b2, l2, ks);
        }
      }
    }
  }

  // KIVI keys ("KIVI: KV cache axes" §3–§4: keys grouped along tokens): four
  // 32-token sub-groups per record, each with its own bf16 step and origin
  // per channel.  Each sub-group's Q' and origin term drive the QK MMAs of
  // its two m-tiles, whose scores then move to log2 units; the softmax gets
  // unit 1 and no origin term.
  __device__ __forceinline__ void scores_kivi(float (&S)[8][4], float (&hinv)[2],
                                              float (&hbias)[2]) {
    const uint32_t* kst2 = reinterpret_cast<const uint32_t*>(kbuf + a.lay.k_scale);
    const uint32_t* kmn2 = reinterpret_cast<const uint32_t*>(kbuf + a.lay.k_min);
#pragma unroll
    for (int sg = 0; sg < 4; ++sg) {
      uint32_t bq[8][2], bl[NL][2];
      float inv_sq, bias, hi[2], hb[2];
      const uint32_t* st = kst2 + sg * (kD / 2);
      build_q([&](int c) {
                const uint32_t w = st[c >> 1];
                return make_float2(bf16_lo(w), bf16_hi(w));
              },
              kmn2 + sg * (kD / 2), bq, bl, inv_sq, bias);
      head_units(inv_sq, bias, hi, hb);
      if (sg == 0) qk_tiles<0, 2>(S, bq, bl);
      else if (sg == 1) qk_tiles<2, 2>(S, bq, bl);
      else if (sg == 2) qk_tiles<4, 2>(S, bq, bl);
      else qk_tiles<6, 2>(S, bq, bl);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float (&s)[4] = S[2 * sg + i];
        if (SPARE) {   // columns 2t, 2t + 1: head t's high and low parts
          s[0] = fmaf(s[0] + s[1], hi[0], hb[0]);
          s[2] = fmaf(s[2] + s[3], hi[0], hb[0]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) s[c] = fmaf(s[c], hi[c & 1], hb[c & 1]);
        }
      }
    }
    hinv[0] = hinv[1] = 1.0f;
    hbias[0] = hbias[1] = 0.0f;
  }

  // Mixed keys (MixKVQ): the BF16 tier on bf16 MMAs of the raw keys and the
  // exact query (ldmatrix transposes the channel-major raw rows), rescaled
  // into the code path's units; the UINT4 and UINT2 tiers as 2-bit virtual
  // channels on the code path.  A per-group table, built in the mixed warps'
  // own table area (free until this group's value tables), gives each virtual channel its key
  // channel, step (times 4 for the high half of a UINT4 code, times the row
  // factor) and origin (zero for a high half).  Q' is normalized by the bound
  // max|q| * max step, so the table needs no pass over the products.
  __device__ __forceinline__ void scores_mixed(float (&S)[8][4], float (&hinv)[2],
                                               float (&hbias)[2]) {
    const RecLayout& L = a.lay;
    // this group's tier counts (its header); kw2 is the record's room
    const int nb = kbuf[L.hdr], n4 = kbuf[L.hdr + 1], nv = kD + n4 - nb, kw2 = L.kw2;
    const int kw_used = (nv + 31) >> 5;   // words of the group's virtual channels
    const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
    uint2* tab = reinterpret_cast<uint2*>(vsb);
    const float* sc = reinterpret_cast<const float*>(kbuf + L.s4);
    const uint16_t* mn = reinterpret_cast<const uint16_t*>(kbuf + L.m4);
    const uint8_t* perm = kbuf + L.perm;
    uint32_t smax = 0u;
    for (int v = lane; v < 32 * kw2; v += 32) {
      float sm = 0.0f;
      uint32_t mc = 0u;
      if (v < nv) {
        const bool hi = v >= n4 && v < 2 * n4;
        const int idx = v < n4 ? v : v - n4;
        const float st = sc[idx] * (hi ? 4.0f : 1.0f);
        smax = max(smax, __float_as_uint(st));   // steps are >= 0
        const float rf = __uint_as_float((142u - 4u * ((v >> 4) & 1) - 2u * ((v >> 3) & 1)) << 23);
        sm = st * rf * (SPARE ? 1.0f : c0);
        mc = (hi ? 0u : static_cast<uint32_t>(mn[idx])) | (static_cast<uint32_t>(perm[nb + idx]) << 16);
      }
      tab[v] = make_uint2(__float_as_uint(sm), mc);
    }
    smax = __reduce_max_sync(kFull, smax);
    float sq, inv_sq;
    pow2_norm(qmax * __uint_as_float(smax) * (SPARE ? 1.0f : c0), sq, inv_sq);
    if (sq > 1.099511627776e12f) {   // cap at 2^40: raw scores stay finite in code units
      sq = 1.099511627776e12f;
      inv_sq = 1.0f / 1.099511627776e12f;
    }
    __syncwarp();   // table written by all lanes

#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int c = 0; c < 4; ++c) S[mt][c] = 0.0f;
    // ---- BF16 tier: raw keys (A, via ldmatrix.trans) times the exact query
    if (nb > 0) {
      const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(kbuf + L.raw));
      const uint32_t zaddr = static_cast<uint32_t>(__cvta_generic_to_shared(zero_row()));
      for (int k16 = 0; k16 < (nb + 15) >> 4; ++k16) {
        uint32_t qb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 16 * k16 + 2 * t + (e & 1) + 8 * (e >> 1);
          // exact bf16 query: the staged copy (8 heads) or global memory
          // (with at most 4 heads the staged copy is pre-scaled fp32)
          qb[e] = (i < nb && !low_col() && hrow() < NREP)
                      ? static_cast<uint32_t>(SPARE ? __ldg(qg_row + perm[i])
                                                    : static_cast<const uint16_t*>(qs)[g * kQRow + perm[i]])
                      : 0u;
        }
        const uint32_t b0 = qb[0] | (qb[1] << 16), b1 = qb[2] | (qb[3] << 16);
        const int i = 16 * k16 + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int pc = 2 * mt + ((lane >> 3) & 1);
          uint32_t A[4];
          ldsm_x4_t(A, i < nb ? raw + i * 256 + ((pc ^ (i & 7)) << 4) : zaddr);
          mma_bf16(S[mt], A, b0, b1);
        }
      }
      // raw dot products -> code units: * c0 * sq / 2^9 per head
      float rr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int src = SPARE ? 8 * t : 4 * (2 * t + h);
        rr[h] = c0 * __shfl_sync(kFull, sq, src) * kInvCodeUnit;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) S[mt][c] *= rr[c & 1];
    }

    // ---- UINT4 and UINT2 tiers: virtual 2-bit channels
    const uint32_t* kcw = reinterpret_cast<const uint32_t*>(kbuf + L.kc);
    float bias = 0.0f;
    for (int w = 0; w < kw_used; ++w) {
      uint32_t kx[8], ky[8];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        kx[mt] = kcw[(mt * kw2 + w) * 32 + lane];
        ky[mt] = kx[mt] >> 8;
      }
#pragma unroll
      for (int kl = 0; kl < 2; ++kl) {
        const int v0 = 32 * w + 16 * kl + 2 * t;
        uint32_t bq0, bq1, bl0 = 0u, bl1 = 0u;
        if constexpr (SPARE) {
          // a head's two lanes share the build (as for uniform keys): the
          // even lane takes the b0 rows (v0, v0 + 1), the odd lane the b1
          // rows (v0 + 8, v0 + 9), and they swap the part they do not keep
          const int par = g & 1;
          const uint4 e = *reinterpret_cast<const uint4*>(tab + v0 + 8 * par);
          const uint32_t es[2] = {e.x, e.z}, em[2] = {e.y, e.w};
          float x[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int ch = static_cast<int>(em[i] >> 16);
            const float qv = static_cast<const float*>(qs)[hrow() * kQRow + ch];
            bias = fmaf(qv, bf16_lo(em[i]), bias);
            x[i] = qv * __uint_as_float(es[i]) * sq;
          }
          const uint32_t H = pack_h2(x[0], x[1]);
          const float2 hf = h2_to_f2(H);
          const uint32_t Lo = pack_h2(x[0] - hf.x, x[1] - hf.y);
          const uint32_t recv = __shfl_xor_sync(kFull, par ? H : Lo, 4);
          bq0 = par ? recv : H;
          bq1 = par ? Lo : recv;
        } else {
          const uint4 e01 = *reinterpret_cast<const uint4*>(tab + v0);
          const uint4 e89 = *reinterpret_cast<const uint4*>(tab + v0 + 8);
          const uint32_t es[4] = {e01.x, e01.z, e89.x, e89.z};
          const uint32_t em[4] = {e01.y, e01.w, e89.y, e89.w};
          float x[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int ch = static_cast<int>(em[i] >> 16);
            const float qv = bf2f(static_cast<const uint16_t*>(qs)[g * kQRow + ch]);
            bias = fmaf(qv, bf16_lo(em[i]), bias);
            x[i] = qv * __uint_as_float(es[i]) * sq;
          }
          bq0 = pack_h2(x[0], x[1]);
          bq1 = pack_h2(x[2], x[3]);
          const float2 h01 = h2_to_f2(bq0), h23 = h2_to_f2(bq1);
          bl0 = pack_h2(x[0] - h01.x, x[1] - h01.y);
          bl1 = pack_h2(x[2] - h23.x, x[3] - h23.y);
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t A[4];
          if (kl) unpack2<1>(kx[mt], ky[mt], A);
          else unpack2<0>(kx[mt], ky[mt], A);
          mma_f16(S[mt], A[0], A[1], A[2], A[3], bq0, bq1);
          if (!SPARE) mma_f16(S[mt], A[0], A[1], A[2], A[3], bl0, bl1);
        }
      }
    }
    bias += __shfl_xor_sync(kFull, bias, 1);
    bias += __shfl_xor_sync(kFull, bias, 2);
    if (SPARE) bias += __shfl_xor_sync(kFull, bias, 4);   // the pair's halves
    else bias *= c0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int src = SPARE ? 8 * t : 4 * (2 * t + h);
      hinv[h] = __shfl_sync(kFull, inv_sq, src) * kCodeUnit;
      hbias[h] = __shfl_sync(kFull, bias, src);
    }
  }

  // One online-softmax step over 128 scores in C layout (rows = tokens):
  // score = acc * hinv + off in log2 units with hinv > 0, so the max is taken
  // on the raw accumulators and p = 2^(acc * hinv + off - m) is one FMA and
  // one ex2.  With at most 4 heads lane (g, t) holds head t in columns 0 and
  // 2 (rows g, g + 8; the state is in mrun[0], lrun[0]), else heads 2t,
  // 2t + 1 in columns (0, 2) and (1, 3).  Returns p in S and the factors
  // that rescale the earlier state of heads 2t, 2t + 1 (the output's columns).
  __device__ __forceinline__ void softmax_update(float (&S)[8][4], const float (&hinv)[2],
                                                 const float (&hoff)[2], float (&alpha)[2]) {
    if constexpr (SPARE) {
      float m = max3(max3(S[0][0], S[0][2], S[1][0]), max3(S[1][2], S[2][0], S[2][2]),
                     max3(S[3][0], S[3][2], S[4][0]));
      m = max3(m, max3(S[4][2], S[5][0], S[5][2]), max3(S[6][0], S[6][2], S[7][0]));
      m = fmaxf(m, S[7][2]);
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
      m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
      const float m_new = fmaxf(mrun[0], fmaf(m, hinv[0], hoff[0]));
      const float al = ex2(mrun[0] - m_new);
      mrun[0] = m_new;
      const float shift = hoff[0] - m_new;
      float ls = 0.0f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        S[mt][0] = ex2(fmaf(S[mt][0], hinv[0], shift));
        S[mt][2] = ex2(fmaf(S[mt][2], hinv[0], shift));
        ls += S[mt][0] + S[mt][2];
      }
      lrun[0] = fmaf(lrun[0], al, ls);
      alpha[0] = __shfl_sync(kFull, al, head_lane(2 * t));
      alpha[1] = __shfl_sync(kFull, al, head_lane(2 * t + 1));
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float off = hoff[h];
        float m = max3(max3(S[0][h], S[0][h + 2], S[1][h]), max3(S[1][h + 2], S[2][h], S[2][h + 2]),
                       max3(S[3][h], S[3][h + 2], S[4][h]));
        m = max3(m, max3(S[4][h + 2], S[5][h], S[5][h + 2]), max3(S[6][h], S[6][h + 2], S[7][h]));
        m = fmaxf(m, S[7][h + 2]);
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
  }

  // Value-side tables of one group (values in vbuf): lane l handles tokens
  // 4l..4l+3.  Returns this group's units per j and the origin scale.
  __device__ __forceinline__ void value_tables(float& svn, float& inv_svm) {
    const RecLayout& L = a.lay;
    const float* vscale = reinterpret_cast<const float*>(vbuf + (L.v_scale - L.kpart));
    const uint2* vmin2 = reinterpret_cast<const uint2*>(vbuf + (L.v_min - L.kpart));
    float vs[4][4], vmn[4][4];
    float mx = 0.0f, mm = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (KIVI) {   // bf16 steps [tok][4]
        const uint2 f = reinterpret_cast<const uint2*>(vscale)[4 * lane + i];
        vs[i][0] = bf16_lo(f.x); vs[i][1] = bf16_hi(f.x);
        vs[i][2] = bf16_lo(f.y); vs[i][3] = bf16_hi(f.y);
      } else {
        const float4 f = reinterpret_cast<const float4*>(vscale)[4 * lane + i];
        vs[i][0] = f.x; vs[i][1] = f.y; vs[i][2] = f.z; vs[i][3] = f.w;
      }
      const uint2 m = vmin2[4 * lane + i];
      vmn[i][0] = bf16_lo(m.x); vmn[i][1] = bf16_hi(m.x);
      vmn[i][2] = bf16_lo(m.y); vmn[i][3] = bf16_hi(m.y);
      mx = max3(mx, max3(vs[i][0], vs[i][1], vs[i][2]), vs[i][3]);
      mm = max3_abs(mm, max3_abs(vmn[i][0], vmn[i][1], vmn[i][2]), vmn[i][3]);
    }
    mm = fabsf(mm);
    // one power-of-two unit for the group's steps and one for its origins
    // (steps are >= 0, so their bit patterns order like their values)
    mx = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(mx)));
    mm = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(mm)));
    // uniform keys: the tables overwrite the metadata every lane has read
    if (!SEP) __syncwarp();
    float s_new, inv_new, svm;
    // a group whose steps are all zero (constant value groups, or a KIVI
    // record whose values are all still in the FIFO) gets unit 1: its
    // tables are zero either way, and a unit from a zero maximum would
    // overflow with the row factor (0 * inf)
    pow2_norm(mx > 0.0f ? mx : 1.0f, s_new, inv_new);
    (void)inv_new;
    // the units of this group's P' never exceed the running ones
    svn = fminf(s_new, sv);
    pow2_norm(mm, svm, inv_svm);
    const int kt = lane >> 2, q4 = lane & 3;
    const int t0 = 2 * (q4 & 1), chi = q4 >> 1;
    // the row factor of the code position these tokens meet (frag_layout.h)
    const float rf = VB == 2 ? __uint_as_float((142u - 4u * (kt & 1) - 2u * chi) << 23)
                             : __uint_as_float((142u - 4u * chi) << 23);
    const float sc = svn * rf;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      vsb[vsb_index(kt, t0, j, chi)] = pack_h2(vs[0][j] * sc, vs[1][j] * sc);
      vsb[vsb_index(kt, t0 + 1, j, chi)] = pack_h2(vs[2][j] * sc, vs[3][j] * sc);
      vmb[vmb_index(kt, j, t0, chi)] = pack_h2(vmn[0][j] * svm, vmn[1][j] * svm);
      vmb[vmb_index(kt, j, t0 + 1, chi)] = pack_h2(vmn[2][j] * svm, vmn[3][j] * svm);
    }
  }

  // Channel tile mc (16 channels) of one group's P·V with B fragments bj,
  // summed in a fresh accumulator acc.
  __device__ __forceinline__ void pv_tile(const uint8_t* vc, int mc, const uint32_t (&bj)[8][2],
                                          float (&acc)[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = 0.0f;
    if (VB == 2) {
      const uint4 w4 = *reinterpret_cast<const uint4*>(vc + (mc * 32 + lane) * 16);
      const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x = wv[w], y = x >> 8;
        uint32_t A[4];
        unpack2<0>(x, y, A);
        mma_f16(acc, A[0], A[1], A[2], A[3], bj[2 * w][0], bj[2 * w][1]);
        unpack2<1>(x, y, A);
        mma_f16(acc, A[0], A[1], A[2], A[3], bj[2 * w + 1][0], bj[2 * w + 1][1]);
      }
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(vc + ((mc * 2 + hh) * 32 + lane) * 16);
        const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t A[4];
          unpack4(wv[i], wv[i] >> 8, A);
          mma_f16(acc, A[0], A[1], A[2], A[3], bj[4 * hh + i][0], bj[4 * hh + i][1]);
        }
      }
    }
  }
  // One FFMA per accumulator folds a group's tile into the rescaled output.
  __device__ __forceinline__ void fold(int i, const float (&acc)[4], float f0, float f1) {
    O[i][0] = fmaf(O[i][0], f0, acc[0]);
    O[i][2] = fmaf(O[i][2], f0, acc[2]);
    O[i][1] = fmaf(O[i][1], f1, acc[1]);
    O[i][3] = fmaf(O[i][3], f1, acc[3]);
  }

  // P·V of one group (values in vbuf) into the running output.  Each
  // channel tile sums the group in a fresh accumulator and one FFMA folds it
  // into the rescaled running output: the running sum of the (always
  // non-negative) code terms never passes through the tensor cores'
  // accumulation, whose truncation would otherwise grow with the context.
  __device__ __forceinline__ void pv(float (&S)[8][4], const float (&alpha)[2], float svn,
                                     float inv_svm) {
    const RecLayout& L = a.lay;
    // rescale of the running output to this group's units, per head
    float f0, f1;
    {
      const float ratio = svn * inv_sv;
      f0 = alpha[0] * ratio;
      f1 = alpha[1] * ratio;
      sv = svn;
      inv_sv = pow2_rcp(svn);
    }
    __syncwarp();   // value tables written by all lanes

    // B fragments of p for the 8 token k-steps; origin term on the side
    uint32_t pb[8][2];
    float Dvm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      if constexpr (SPARE) {   // rows g, g + 8 of heads 2t, 2t + 1 from their lanes
        const uint32_t pk = pack_h2(S[kt][0], S[kt][2]);
        const uint32_t x0 = __shfl_sync(kFull, pk, head_lane(2 * t));
        const uint32_t x1 = __shfl_sync(kFull, pk, head_lane(2 * t + 1));
        pb[kt][0] = movmatrix_t(__byte_perm(x0, x1, 0x5410));
        pb[kt][1] = movmatrix_t(__byte_perm(x0, x1, 0x7632));
      } else {
        pb[kt][0] = movmatrix_t(pack_h2(S[kt][0], S[kt][1]));
        pb[kt][1] = movmatrix_t(pack_h2(S[kt][2], S[kt][3]));
      }
      // lanes g >= 4 (A rows 4..7) take zeros
      const uint2 av = *reinterpret_cast<const uint2*>(vmb + vmb_index(kt, g & 3, t, 0));
      const uint32_t a0 = g < 4 ? av.x : 0u, a2 = g < 4 ? av.y : 0u;
      mma_f16(Dvm, a0, 0u, a2, 0u, pb[kt][0], pb[kt][1]);
    }
    const uint8_t* vc = vbuf + (L.v_codes - L.kpart);
    if constexpr (SPARE) {
      // B columns 4..7 repeat heads 0..3, so they carry the next channel
      // group's P': one set of B fragments serves groups 2jp and 2jp + 1
      // (their channel tiles keep the results of columns 0..3 and 4..7).
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        const int jl = 2 * jp + (g >> 2);
        uint32_t bj[8][2];
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          const uint2 vs = *reinterpret_cast<const uint2*>(vsb + vsb_index(kt, t, jl, 0));
          bj[kt][0] = hmul2_u(pb[kt][0], vs.x);
          bj[kt][1] = hmul2_u(pb[kt][1], vs.y);
        }
        // tiles 4jp + k (group 2jp, columns 0..3) and 4jp + k + 2 (group
        // 2jp + 1, columns 4..7): each lane keeps the one of its columns
        const bool hi = t >= 2;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float acc_e[4], acc_o[4], acc[4];
          pv_tile(vc, 4 * jp + k, bj, acc_e);
          pv_tile(vc, 4 * jp + k + 2, bj, acc_o);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[c] = hi ? acc_o[c] : acc_e[c];
          fold(2 * jp + k, acc, f0, f1);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // P' = p * step of this channel group (with the row factors)
        uint32_t bj[8][2];
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
          const uint2 vs = *reinterpret_cast<const uint2*>(vsb + vsb_index(kt, t, j, 0));
          bj[kt][0] = hmul2_u(pb[kt][0], vs.x);
          bj[kt][1] = hmul2_u(pb[kt][1], vs.y);
        }
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
          float acc[4];
          pv_tile(vc, 2 * j + mm, bj, acc);
          fold(2 * j + mm, acc, f0, f1);
        }
      }
    }
    // origin term in true units (lanes g < 4 hold channel group j = g)
    {
      const float im = g < 4 ? inv_svm : 0.0f;
      vm[0] = fmaf(vm[0], alpha[0], Dvm[0] * im);
      vm[1] = fmaf(vm[1], alpha[1], Dvm[1] * im);
    }
  }

  // Fused append: the unit's new token into residual slot `slot` (lanes
  // 0..15 the key row, 16..31 the value row), visible to the chunk copies
  // that read the window next.
  __device__ __forceinline__ void put_token(int u, int slot) {
    const int piece = lane & 15;
    const uint4* src = (lane < 16 ? a.new_k : a.new_v) + static_cast<long long>(u) * (kD / 8) + piece;
    uint4* dst = reinterpret_cast<uint4*>(const_cast<uint16_t*>(lane < 16 ? a.res_k : a.res_v)) +
                 (static_cast<long long>(u) * kR + slot) * (kD / 8) + piece;
    *dst = __ldg(src);
    __threadfence();
    __syncwarp();
  }

  // 16-token chunk c (16 rows x 256 B) of a residual tensor into chunk slot
  // `slot` of the record buffer, 16-byte pieces placed at column piece
  // (col ^ (row & 7)) so the ldmatrix row reads are free of bank conflicts.
  __device__ __forceinline__ void stage_chunk(const uint8_t* src, int c, int slot) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(kbuf)) + slot * 4096;
    const uint8_t* s0 = src + c * 4096;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lane + 32 * k, row = i >> 4, col = i & 15;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                       d + row * 256 + ((col ^ (row & 7)) << 4)),
                   "l"(s0 + 16 * i));
    }
  }
  __device__ __forceinline__ uint32_t chunk_addr(int slot, int row, int col16) const {
    return static_cast<uint32_t>(__cvta_generic_to_shared(kbuf)) + slot * 4096 + row * 256 +
           ((col16 ^ (row & 7)) << 4);
  }

  // A bf16 window (the residual, or the attention sinks: count tokens of a
  // [units][cap][D] pair) on tensor cores, folded into the same
  // online-softmax state.  Scores: bf16 MMA of the exact bf16 keys and
  // query (exact products, fp32 sums).  P·V: the values transposed by
  // ldmatrix, p split into bf16 high and low parts (16 bits in all), one
  // fresh accumulator per chunk and channel tile.  Keys and values stream
  // through two 4 KB chunk slots of the record buffer.
  __device__ __forceinline__ void window(int u, const uint16_t* kbase, const uint16_t* vbase,
                                        int count, int cap) {
    const int r = count, nc = (r + 15) >> 4;
    const uint8_t* kr = reinterpret_cast<const uint8_t*>(kbase + static_cast<long long>(u) * cap * kD);
    const uint8_t* vr = reinterpret_cast<const uint8_t*>(vbase + static_cast<long long>(u) * cap * kD);
    // query B fragments: the high-part columns of the code path hold the
    // exact query (column 2h with at most 4 heads, else g), the others zero
    uint32_t bqr[8][2];
    {
      const int b = u / a.Hkv, kvh = u % a.Hkv;
      const bool on = !low_col() && hrow() < NREP;
      const uint32_t* qg = reinterpret_cast<const uint32_t*>(
          a.q + (static_cast<long long>(b) * a.Hq + kvh * NREP + min(hrow(), NREP - 1)) * kD);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        bqr[ks][0] = on ? __ldg(qg + 8 * ks + t) : 0u;
        bqr[ks][1] = on ? __ldg(qg + 8 * ks + t + 4) : 0u;
      }
    }
    __syncwarp();
    float S[8][4];
    stage_chunk(kr, 0, 0);
    asm volatile("cp.async.commit_group;\n" ::);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (c < nc) {
        if (c + 1 < nc) stage_chunk(kr, c + 1, (c + 1) & 1);
        asm volatile("cp.async.commit_group;\n" ::);
        asm volatile("cp.async.wait_group 1;\n" ::);
        __syncwarp();
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t A[4];
          ldsm_x4(A, chunk_addr(c & 1, row, 2 * ks + (lane >> 4)));
          mma_bf16(acc, A, bqr[ks][0], bqr[ks][1]);
        }
        __syncwarp();   // slot read before it is staged again
#pragma unroll
        for (int i = 0; i < 4; ++i) S[c][i] = 16 * c + g + 8 * (i >> 1) < r ? acc[i] : -INFINITY;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) S[c][i] = -INFINITY;
      }
    }
    // the first value chunk loads during the softmax
    stage_chunk(vr, 0, 0);
    asm volatile("cp.async.commit_group;\n" ::);
    {
      const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
      const float hinv[2] = {c0, c0}, hoff[2] = {0.0f, 0.0f};
      float alpha[2];
      softmax_update(S, hinv, hoff, alpha);
      if (sv == kSentinel) {   // no group in this segment: O is still zero
        sv = 1.0f;
        inv_sv = 1.0f;
      }
#pragma unroll
      for (int mc = 0; mc < NO; ++mc) {
        O[mc][0] *= alpha[0]; O[mc][2] *= alpha[0];
        O[mc][1] *= alpha[1]; O[mc][3] *= alpha[1];
      }
      vm[0] *= alpha[0];
      vm[1] *= alpha[1];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (c < nc) {
        if (c + 1 < nc) stage_chunk(vr, c + 1, (c + 1) & 1);
        asm volatile("cp.async.commit_group;\n" ::);
        // p of this chunk as bf16 B fragments: high part, then the rest
        uint32_t ph[2], pl[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          // row g (i = 0) or g + 8 (i = 1) of heads 2t, 2t + 1
          const float p0 = SPARE ? __shfl_sync(kFull, S[c][2 * i], head_lane(2 * t)) : S[c][2 * i];
          const float p1 = SPARE ? __shfl_sync(kFull, S[c][2 * i], head_lane(2 * t + 1))
                                 : S[c][2 * i + 1];
          const uint32_t hi = pack_bf2(p0, p1);
          const float l0 = p0 - __uint_as_float(hi << 16);
          const float l1 = p1 - __uint_as_float(hi & 0xffff0000u);
          ph[i] = movmatrix_t(hi);
          pl[i] = movmatrix_t(pack_bf2(l0, l1));
        }
        // tokens past r (last chunk): zero their value columns, whatever
        // the buffer holds there
        const int t0 = 16 * c + 2 * t;
        const uint32_t m01 = (t0 < r ? 0xffffu : 0u) | (t0 + 1 < r ? 0xffff0000u : 0u);
        const uint32_t m89 = (t0 + 8 < r ? 0xffffu : 0u) | (t0 + 9 < r ? 0xffff0000u : 0u);
        asm volatile("cp.async.wait_group 1;\n" ::);
        __syncwarp();
        const int row = (lane & 7) + 8 * (lane >> 4);
        const float sc = sv * kInvCodeUnit;
        float acc8[8][4];
#pragma unroll
        for (int mc = 0; mc < 8; ++mc) {
          uint32_t A[4];
          ldsm_x4_t(A, chunk_addr(c & 1, row, 2 * mc + ((lane >> 3) & 1)));
          A[0] &= m01; A[1] &= m01; A[2] &= m89; A[3] &= m89;
#pragma unroll
          for (int i = 0; i < 4; ++i) acc8[mc][i] = 0.0f;
          mma_bf16(acc8[mc], A, ph[0], ph[1]);
          mma_bf16(acc8[mc], A, pl[0], pl[1]);
        }
#pragma unroll
        for (int k = 0; k < NO; ++k) {
          // with at most 4 heads: the tile of this lane's kept columns
          const int me = SPARE ? 4 * (k >> 1) + (k & 1) : k;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float v = SPARE ? (t >= 2 ? acc8[me + 2][i] : acc8[me][i]) : acc8[me][i];
            O[k][i] = fmaf(v, sc, O[k][i]);
          }
        }
        __syncwarp();   // slot read before it is staged again
      }
    }
    asm volatile("cp.async.wait_group 0;\n" ::);
    __syncwarp();
  }

  // KIVI: P·V over tokens first .. 127 of a unit's newest record, whose
  // values are still in the value FIFO (ring slots first .. 127 of the
  // unit's residual V window), with the probabilities the softmax left in
  // S.  The window's value path: 16-token chunks staged in two 4 KB slots of
  // the record buffer (free once the record's P·V is done), values
  // transposed by ldmatrix, p split into bf16 high and low parts, one fresh
  // accumulator per chunk and channel tile folded into the running output.
  __device__ __forceinline__ void ring_values(int u, const float (&S)[8][4], int first) {
    const uint8_t* vr = reinterpret_cast<const uint8_t*>(a.res_v + static_cast<long long>(u) * kR * kD);
    const int c0 = first >> 4;
    __syncwarp();
    stage_chunk(vr, c0, c0 & 1);
    asm volatile("cp.async.commit_group;\n" ::);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (c >= c0) {
        if (c + 1 < 8) stage_chunk(vr, c + 1, (c + 1) & 1);
        asm volatile("cp.async.commit_group;\n" ::);
        uint32_t ph[2], pl[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          // row g (i = 0) or g + 8 (i = 1) of heads 2t, 2t + 1
          const float p0 = SPARE ? __shfl_sync(kFull, S[c][2 * i], head_lane(2 * t)) : S[c][2 * i];
          const float p1 = SPARE ? __shfl_sync(kFull, S[c][2 * i], head_lane(2 * t + 1))
                                 : S[c][2 * i + 1];
          const uint32_t hi = pack_bf2(p0, p1);
          const float l0 = p0 - __uint_as_float(hi << 16);
          const float l1 = p1 - __uint_as_float(hi & 0xffff0000u);
          ph[i] = movmatrix_t(hi);
          pl[i] = movmatrix_t(pack_bf2(l0, l1));
        }
        // tokens before `first` have their values in the codes: zero their
        // value columns here
        const int t0 = 16 * c + 2 * t;
        const uint32_t m01 = (t0 >= first ? 0xffffu : 0u) | (t0 + 1 >= first ? 0xffff0000u : 0u);
        const uint32_t m89 = (t0 + 8 >= first ? 0xffffu : 0u) | (t0 + 9 >= first ? 0xffff0000u : 0u);
        asm volatile("cp.async.wait_group 1;\n" ::);
        __syncwarp();
        const int row = (lane & 7) + 8 * (lane >> 4);
        const float sc = sv * kInvCodeUnit;
        float acc8[8][4];
#pragma unroll
        for (int mc = 0; mc < 8; ++mc) {
          uint32_t A[4];
          ldsm_x4_t(A, chunk_addr(c & 1, row, 2 * mc + ((lane >> 3) & 1)));
          A[0] &= m01; A[1] &= m01; A[2] &= m89; A[3] &= m89;
#pragma unroll
          for (int i = 0; i < 4; ++i) acc8[mc][i] = 0.0f;
          mma_bf16(acc8[mc], A, ph[0], ph[1]);
          mma_bf16(acc8[mc], A, pl[0], pl[1]);
        }
#pragma unroll
        for (int k = 0; k < NO; ++k) {
          const int me = SPARE ? 4 * (k >> 1) + (k & 1) : k;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float v = SPARE ? (t >= 2 ? acc8[me + 2][i] : acc8[me][i]) : acc8[me][i];
            O[k][i] = fmaf(v, sc, O[k][i]);
          }
        }
        __syncwarp();   // slot read before it is staged again
      }
    }
    asm volatile("cp.async.wait_group 0;\n" ::);
    __syncwarp();
  }

  // Merge the lanes and write this unit's partial (o, m, l) per query head.
  __device__ __forceinline__ void finish(int u, int part) {
    float l[2];
#pragma unroll
    for (int h = 0; h < (SPARE ? 1 : 2); ++h) {
      float x = lrun[h];
      x += __shfl_xor_sync(kFull, x, 4);
      x += __shfl_xor_sync(kFull, x, 8);
      x += __shfl_xor_sync(kFull, x, 16);
      l[h] = x;
    }
    float* base = a.ws + (static_cast<long long>(u) * a.max_parts + part) * NREP * (kD + 2);
#pragma unroll
    for (int i = 0; i < NO; ++i) {
      // with at most 4 heads, the tiles of odd channel groups keep columns
      // 4..7 (lanes t >= 2), which hold heads 2t - 4 and 2t - 3
      const int mc = tile_of(i), j = mc >> 1;
      const float vm0 = __shfl_sync(kFull, vm[0], 4 * j + t);
      const float vm1 = __shfl_sync(kFull, vm[1], 4 * j + t);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int h = SPARE ? ((2 * t + (c & 1)) & 3) : 2 * t + (c & 1);
        const int ch = 16 * mc + g + 8 * (c >> 1);
        const float val = O[i][c] * (inv_sv * kCodeUnit) + ((c & 1) ? vm1 : vm0);
        if (h < NREP) base[h * (kD + 2) + ch] = val;
      }
    }
    if (SPARE) {   // lane (0, t): head t
      if (g == 0 && t < NREP) {
        base[t * (kD + 2) + kD] = mrun[0];
        base[t * (kD + 2) + kD + 1] = l[0];
      }
    } else if (g == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int hh = 2 * t + h;
        base[hh * (kD + 2) + kD] = mrun[h];
        base[hh * (kD + 2) + kD + 1] = l[h];
      }
    }
  }

  // An empty partial (o = 0, m = -inf, l = 0: it weighs nothing in the
  // merge) for a unit this warp gave up on, so the combine never reads a
  // slot left over from an earlier call.
  __device__ __forceinline__ void empty_part(int u, int part) {
    float* base = a.ws + (static_cast<long long>(u) * a.max_parts + part) * NREP * (kD + 2);
    for (int i = lane; i < NREP * (kD + 2); i += 32) {
      const int c = i % (kD + 2);
      base[i] = c == kD ? -INFINITY : 0.0f;
    }
  }
};


template <int KB, int VB, int NREP, bool MIX, bool KIVI = false, bool PNMIX = false>
__global__ void __launch_bounds__(max_warps(KB, VB, NREP, MIX || KIVI || PNMIX) * 32, 1) decode_mma_kernel(MmaArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  // Consecutive slices (records of one unit, contiguous in memory) run on
  // different SMs, so each SM's warps read from several places at once; row
  // w of the grid is rotated by w, so a block's warps take slices from
  // different places of the unit pattern.  (Unrotated, with every unit
  // spanning a multiple of the grid width in slices, a block's slices all
  // sat at the same place: blocks carried unequal numbers of groups and the
  // units' window items all landed on a few SMs.)
  const int slot = warp * gridDim.x + (blockIdx.x + warp) % gridDim.x;
  // the combine kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  if (slot >= a.n_slots) return;            // warp-uniform
  uint8_t* mine = smem + static_cast<size_t>(warp) * (a.rec_bytes + warp_extra(MIX || KIVI));
  Warp<KB, VB, NREP, MIX, KIVI, PNMIX> W(a, mine);
  const long long p0 = slot_start(a, slot), p1 = slot_start(a, slot + 1);
  const int u_last = static_cast<int>((p1 - 1) / a.unit_len);
  // after a wait gave up: empty partials for this unit and the rest of the slice
  auto abandon = [&](int u0) {
    for (int uu = u0; uu <= u_last; ++uu)
      W.empty_part(uu, slot - slot_of(a, static_cast<long long>(uu) * a.unit_len));
  };
  // The bf16 windows this slice reads last go to L2 now, so their chunk
  // copies (two in flight) do not wait on HBM at the end of the slice.
  if (W.lane == 0) {
    for (int u = static_cast<int>(p0 / a.unit_len); u <= u_last; ++u) {
      const long long ub = static_cast<long long>(u) * a.unit_len;
      const long long lo = max(p0, ub) - ub, hi = min(p1, ub + a.unit_len) - ub;
      if (a.r > 0 && lo <= a.n_groups && a.n_groups < hi) {
        prefetch_l2(a.res_k + static_cast<long long>(u) * kR * kD, a.r * kD * 2);
        prefetch_l2(a.res_v + static_cast<long long>(u) * kR * kD, a.r * kD * 2);
      }
      const long long ps = a.n_groups + (a.r > 0 ? kResidualWeight : 0);
      if (a.s > 0 && lo <= ps && ps < hi) {
        prefetch_l2(a.sink_k + static_cast<long long>(u) * a.n_sink * kD, a.s * kD * 2);
        prefetch_l2(a.sink_v + static_cast<long long>(u) * a.n_sink * kD, a.s * kD * 2);
      }
    }
  }
  for (int u = static_cast<int>(p0 / a.unit_len); u <= u_last; ++u) {
    const long long ub = static_cast<long long>(u) * a.unit_len;
    const long long lo = max(p0, ub) - ub, hi = min(p1, ub + a.unit_len) - ub;
    const int g0 = static_cast<int>(lo);
    const int g1 = static_cast<int>(min(hi, static_cast<long long>(a.n_groups)));
    const bool res = a.r > 0 && lo <= a.n_groups && a.n_groups < hi;
    const int ps = a.n_groups + (a.r > 0 ? kResidualWeight : 0);   // position of the sink item
    const bool snk = a.s > 0 && lo <= ps && ps < hi;
    // keys of group i+1 load during the P·V of group i, values of group
    // i+1 during its QK: one bulk copy and one mbarrier per part.  The
    // unit's first group is requested before its query is read.
    if (g0 < g1) {
      W.issue_k(u, g0);
      W.issue_v(u, g0);
    }
    W.begin_unit(u);
    bool gave_up = false;
    if (g0 < g1) {
      for (int gi = g0; gi < g1; ++gi) {
        const bool more = gi + 1 < g1;
        if (!W.wait_part(W.mb_k, W.ph_k)) {   // keys of gi (bounded wait)
          W.wait_part(W.mb_v, W.ph_v);        // the value copy in flight
          gave_up = true;
          break;
        }
        float S[8][4], hinv[2], hbias[2], alpha[2], svn, inv_svm;
        W.scores(S, hinv, hbias);
        __syncwarp();                          // key part (and mixed table) consumed
        if (more) W.issue_k(u, gi + 1);
        if (!W.wait_part(W.mb_v, W.ph_v)) {   // values of gi
          if (more) W.wait_part(W.mb_k, W.ph_k);
          gave_up = true;
          break;
        }
        // the value tables' shared-memory round trip overlaps the softmax
        W.value_tables(svn, inv_svm);
        W.softmax_update(S, hinv, hbias, alpha);
        W.pv(S, alpha, svn, inv_svm);
        __syncwarp();                          // value part consumed
        if (more) W.issue_v(u, gi + 1);
        // KIVI: the newest record's values from token r on are still in the
        // value FIFO (ring slots r..127); its codes there are zero
        if (KIVI && gi == a.n_groups - 1) W.ring_values(u, S, a.r);
      }
    }
    // out of the group loop, so the loop keeps no state for it
    if (gave_up) {
      abandon(u);
      return;
    }
    if (res) {
      if (a.new_k != nullptr) W.put_token(u, a.r - 1);
      W.window(u, a.res_k, a.res_v, a.r, kR);
    }
    if (snk) W.window(u, a.sink_k, a.sink_v, a.s, a.n_sink);
    W.finish(u, slot - slot_of(a, ub));
  }
}

template <int KB, int VB, int NREP, bool MIX, bool KIVI = false, bool PNMIX = false>
cudaError_t launch_cfg(const MmaArgs& a, int warps, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(warps) * (a.rec_bytes + warp_extra(MIX || KIVI));
  auto kern = decode_mma_kernel<KB, VB, NREP, MIX, KIVI, PNMIX>;
  static SmemOptIn opt_in;
  cudaError_t e = opt_in.ensure(kern);
  if (e != cudaSuccess) return e;
  const int grid = (a.n_slots + warps - 1) / warps;
  kern<<<grid, warps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

template <int KB, int VB, bool MIX, bool KIVI = false, bool PNMIX = false>
cudaError_t launch_rep(const MmaArgs& a, int nrep, int warps, cudaStream_t s) {
  switch (nrep) {
    case 1: return launch_cfg<KB, VB, 1, MIX, KIVI, PNMIX>(a, warps, s);
    case 2: return launch_cfg<KB, VB, 2, MIX, KIVI, PNMIX>(a, warps, s);
    case 4: return launch_cfg<KB, VB, 4, MIX, KIVI, PNMIX>(a, warps, s);
    case 8: return launch_cfg<KB, VB, 8, MIX, KIVI, PNMIX>(a, warps, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace kvq
