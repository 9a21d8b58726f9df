// Internal definitions of libkvq: HBM layout of the packed cache, the cache
// handle and the kernel launchers shared between translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

constexpr int kD = KVQ_HEAD_DIM;   // head_dim
constexpr int kKG = KVQ_K_GROUP;   // tokens per key group
constexpr int kVG = KVQ_V_GROUP;   // channels per value group
constexpr int kR = KVQ_RESIDUAL;   // residual capacity
constexpr int kVGroups = kD / kVG; // value groups per token (4)
constexpr int kMaxRep = 8;         // query heads per KV head

// ---------------------------------------------------------------------------
// One "group record" holds everything the decode kernel reads for 128
// consecutive tokens of one (batch row, KV head): the Key codes and per-
// channel (step, origin), then the Value codes and per-token (step, origin).
// Records of one (b, kv head) are contiguous, so a split of the token axis
// is one contiguous byte range (streamed with 16-byte cp.async copies).
//
// Uniform key (k_bits = kb):
//   [0]            K codes  128*128*kb/8 bytes in tensor-core fragment
//                           order (frag_layout.h)
//   [kc]           kscale   fp32  [D]
//   [kc+4D]        kmin     bf16  [D]
// PN-Mix key (H3/L1, App. G packing), channels in the unit's stored order
// (the high channels first, each part ascending; the cache's pn_perm):
//   [0]            LSB plane 2048 B: bit 0 of every code, 1-bit fragment
//                  order: word (mt*2 + ks/4)*32 + lane, bit 2*(ks%4) + chi +
//                  8*rhi + 16*half (frag_layout.h coordinates)
//   [kc]           upper plane: bits 1-2 of the high channels' codes, nh/32
//                  words per (tile, lane) in the 2-bit key fragment order
//   [k_scale]      fp32 [D] steps (high) or Eq. 7 scales (low)
//   [k_min]        fp32 [D] origins (high) or Eq. 7 offsets (low)
// KIVI key (KIVI article: keys per channel in groups of 32 tokens, metadata
// in the input dtype):
//   [0]            K codes  128*128*kb/8 bytes, fragment order as uniform
//   [kc]           kstep    bf16  [4][D]   per 32-token sub-group and channel
//   [kc+8D]        kmin     bf16  [4][D]
//   value part:    codes as uniform, vstep bf16 [128][D/32], vmin bf16
//                  [128][D/32]; zero for tokens still in the value FIFO
// Mixed key: the group's own counts nb (BF16), n4 (UINT4), n2 = D - nb - n4
// (UINT2) are in its header; rank tiers fix them to the config's n_bf16,
// n_uint4, threshold tiers bound them by those (the sections are sized for
// the largest case):
//   [0]            perm     uint8 [D]   BF16, UINT4, UINT2 channels, ascending
//   [D]            raw      bf16  [n_bf16][128] channel-major; the 16-byte
//                           piece p of tier channel i sits at piece p ^ (i & 7)
//   [kc]           codes    2-bit "virtual channels" in the key fragment
//                           order (frag_layout.h) with kw2 words per (tile,
//                           lane): v < n4 the low two bits of UINT4 channel
//                           v, n4 <= v < 2 n4 its high two bits, then the
//                           n2 UINT2 channels, zero up to 32 kw2 channels
//   [s4]           steps    fp32  [nq]  UINT4 channels, then UINT2 (perm order)
//   [m4]           origins  bf16  [nq]  same order
//   [hdr]          counts   uint8 nb, n4 (16 bytes reserved)
// Value (v_bits = vb), after the key part at offset kpart:
//   [kpart]        V codes  128*128*vb/8 bytes in fragment order
//   [+vc]          vscale   fp32  [128][D/32]
//   [+vc+2048]     vmin     bf16  [128][D/32]
// Every section starts on a 16-byte boundary; the value part and the
// record size are multiples of 128 bytes (uniform layouts are by
// construction, mixed key parts are padded), so records and their parts
// start on 128-byte lines.
// ---------------------------------------------------------------------------
struct RecLayout {
  int mixed;
  int kivi;      // KIVI variant: bf16 metadata, keys in four 32-token sub-groups
  int pnmix;     // PN-Mix H3/L1 keys: LSB plane + upper plane of the high channels
  int nh;        // PN-Mix: high channels (2 * n_high_pairs), first in the stored order
  int kb, vb;
  int thresh;    // mixed: threshold tiers (per-group counts up to nb, n4)
  int nb, n4;    // mixed: BF16 / UINT4 channels a group (rank tiers) or at most
  // key (uniform)
  int k_codes, k_scale, k_min;
  // key (mixed): perm [D], raw [nb][128], virtual 2-bit channel words, the
  // quantized channels' steps [nq] (fp32) and origins [nq] (bf16) in perm
  // order (UINT4 first), then the header: the group's BF16 and UINT4
  // channel counts (one byte each)
  int perm, raw, kc, s4, m4, hdr;
  int nq;       // capacity of the step / origin tables
  int n2cap;    // UINT2 channels a group at most (D - nb - n4, or D)
  int nv, kw2;  // virtual 2-bit channels (2 n4 + n2) at most, words per (tile, lane)
  int kpart;  // bytes of the key part
  // value
  int v_codes, v_scale, v_min;
  int bytes;  // total record bytes (multiple of 16)
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline RecLayout make_layout(int mixed, int kb, int vb,
                                                 int nb, int n4, int thresh, int kivi = 0,
                                                 int pnmix_high = -1) {
  RecLayout L{};
  L.mixed = mixed;
  L.kivi = kivi;
  L.kb = kb;
  L.vb = vb;
  if (pnmix_high >= 0) {
    // PN-Mix: LSB plane (1 bit, all channels), upper plane (2 bits, the
    // nh high channels), then fp32 scales and offsets, channels in the
    // unit's stored order (high channels first)
    L.pnmix = 1;
    L.kb = 2;
    L.nh = pnmix_high;
    L.k_codes = 0;
    L.kc = kD * kKG / 8;
    L.kw2 = pnmix_high / 32;
    L.k_scale = L.kc + pnmix_high * kKG * 2 / 8;
    L.k_min = L.k_scale + 4 * kD;
    L.kpart = (L.k_min + 4 * kD + 127) & ~127;
    L.v_codes = L.kpart;
    L.v_scale = L.v_codes + kKG * kD * vb / 8;
    L.v_min = L.v_scale + 4 * kKG * kVGroups;
    L.bytes = align16(L.v_min + 2 * kKG * kVGroups);
    return L;
  }
  if (kivi) {
    // KIVI: steps then origins, bf16 [4 sub-groups of 32 tokens][D]
    L.k_codes = 0;
    L.k_scale = kD * kKG * kb / 8;
    L.k_min = L.k_scale + 2 * 4 * kD;
    L.kpart = (L.k_min + 2 * 4 * kD + 127) & ~127;
    L.v_codes = L.kpart;
    L.v_scale = L.v_codes + kKG * kD * vb / 8;        // bf16 [128][D/32]
    L.v_min = L.v_scale + 2 * kKG * kVGroups;
    L.bytes = (L.v_min + 2 * kKG * kVGroups + 127) & ~127;
    return L;
  }
  if (!mixed) {
    L.k_codes = 0;
    L.k_scale = kD * kKG * kb / 8;
    L.k_min = L.k_scale + 4 * kD;
    L.kpart = align16(L.k_min + 2 * kD);
  } else {
    // rank tiers: exactly nb BF16 and n4 UINT4 channels a group; threshold
    // tiers: any counts up to those, so the tables take the largest case
    // (no BF16 channel, n4 UINT4 channels: D + n4 virtual channels)
    L.thresh = thresh;
    L.nb = nb;
    L.n4 = n4;
    L.perm = 0;
    L.raw = kD;
    L.nq = thresh ? kD : kD - nb;
    L.n2cap = thresh ? kD : kD - nb - n4;
    L.nv = kD + n4 - (thresh ? 0 : nb);
    L.kw2 = (L.nv + 31) / 32;
    L.kc = align16(L.raw + nb * kKG * 2);
    L.s4 = L.kc + L.kw2 * 8 * 32 * 4;
    L.m4 = L.s4 + 4 * L.nq;
    L.hdr = align16(L.m4 + 2 * L.nq);
    L.kpart = (L.hdr + 16 + 127) & ~127;   // value part on a 128-byte line
  }
  L.v_codes = L.kpart;
  L.v_scale = L.v_codes + kKG * kD * vb / 8;
  L.v_min = L.v_scale + 4 * kKG * kVGroups;
  L.bytes = align16(L.v_min + 2 * kKG * kVGroups);
  return L;
}

}  // namespace kvq

// The opaque handle.
struct kvq_cache {
  kvq_config cfg;
  kvq::RecLayout lay;
  int device;
  int num_sms;
  uint8_t* base;       // whole device allocation
  bool owned;          // allocated by the library
  size_t bytes;
  uint8_t* records;    // [B*Hkv][max_groups][lay.bytes]
  int max_groups;
  kvq_bf16* res_k;     // [B*Hkv][128][D]
  kvq_bf16* res_v;
  kvq_bf16* sink_k;    // [B*Hkv][n_sink][D] (attention-sink window)
  kvq_bf16* sink_v;
  unsigned* status;    // sticky KVQ_FLAG_* word
  float* qacc;         // mixed: running sum of |q| [B*Hkv][D] (online saliency)
  uint8_t* pn_perm;    // PN-Mix: [B*Hkv][D] stored position -> channel (high first)
  bool pn_ready;       // PN-Mix: pairs selected (kvq_pnmix_pairs)
  int q_steps;         // decode steps summed in qacc since the last flush
  int q_rep;           // query heads per KV head of those steps
  int t_q;             // quantized tokens (multiple of 128)
  int r;               // residual tokens (0..128)
  int s;               // sink tokens (0..n_sink)
};

namespace kvq {

// Raises one kernel's dynamic shared-memory limit to the device's opt-in
// maximum (less the kernel's static shared memory), once per device (a cudaFuncSetAttribute round trip on every
// launch would add host time to every call).  One instance per kernel.
struct SmemOptIn {
  std::atomic<unsigned long long> done{0};   // bit d: device d is set up
  template <typename K>
  cudaError_t ensure(K kernel) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    // the opt-in maximum less the kernel's static shared memory
    int most = 0;
    cudaFuncAttributes fa;
    e = cudaDeviceGetAttribute(&most, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               most - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// Polls a decode warp makes before its wait for a staged record part gives
// up (KVQ_FLAG_TIMEOUT); kvq_set_wait_limit changes it for failure tests.
int decode_wait_polls();
void set_decode_wait_polls(int polls);
void set_decode_split_event(cudaEvent_t ev);

// Where the quantize kernel reads its 128-token tiles from.
struct QuantSrc {
  const kvq_bf16* k;
  const kvq_bf16* v;
  long long unit_stride;   // elements between consecutive (b, kv head)
  long long group_stride;  // elements between consecutive 128-token tiles
};

// One token into slot `slot` of a [units][cap][D] bf16 window pair (the
// residual or the sink).
cudaError_t launch_append(const kvq_cache* c, const kvq_bf16* k_new, const kvq_bf16* v_new,
                          kvq_bf16* dst_k, kvq_bf16* dst_v, int cap, int slot, cudaStream_t s);
// Tokens [first, first + count) of k, v [units][L][D] into rows 0..count-1
// of a [units][cap][D] window pair.
cudaError_t launch_copy_tokens(const kvq_bf16* k, const kvq_bf16* v, int L, int first, int count,
                               kvq_bf16* dst_k, kvq_bf16* dst_v, int cap, int units,
                               cudaStream_t s);
// importance: mixed keys' I_d [units][D]; NULL takes it from the cache's
// online window (qacc / (q_rep * q_steps)).
cudaError_t launch_quantize(const kvq_cache* c, QuantSrc src, int n_groups,
                            int first_group, const float* importance,
                            cudaStream_t s);


// KIVI variant (kivi.cu): seal n_records key records from 128-token tiles of
// src.k (unit u, record k at u * unit_stride + k * group_stride elements),
// zeroing their value parts; quantize the values of tokens [t0, t1) of
// records first_record.. from src.v rows (record k's token t at k *
// group_stride + t * D), limited to the first n_valid tokens of the history.
cudaError_t launch_kivi_seal(const kvq_cache* c, QuantSrc src, int n_records, int first_record,
                             cudaStream_t s);
// KIVI prefill: records 0 .. n_records - 1 sealed and the values of tokens
// [0, n_valid) quantized, in one launch (quant.cu).
cudaError_t launch_kivi_prefill(const kvq_cache* c, QuantSrc src, int n_records, int n_valid,
                                cudaStream_t s);
cudaError_t launch_kivi_values(const kvq_cache* c, QuantSrc src, int n_records, int first_record,
                               int t0, int t1, int n_valid, cudaStream_t s);
// Canonical KIVI export of records [u][0 .. t_q/128): key codes [u][n*4][D]
// [32*bits/8] (per 32-token group and channel, LSB first along tokens),
// origins and steps bf16 [u][n*4][D]; value codes [u][n*128][D*bits/8],
// origins and steps bf16 [u][n*128][D/32] (zero for tokens in the FIFO).
// PN-Mix (pnmix.cu): Eq. 6 pair scores and the selection into c->pn_perm;
// export of the H3/L1 key groups.
cudaError_t launch_pnmix_pairs(const kvq_cache* c, const kvq_bf16* q, int Hq, int Lq,
                               const kvq_bf16* k, int Lk, float* sigma, cudaStream_t s);
cudaError_t launch_export_pnmix(const kvq_cache* c, uint8_t* codes, float* offset, float* scale,
                                uint8_t* high, cudaStream_t s);
cudaError_t launch_export_kivi(const kvq_cache* c, uint8_t* k_codes, kvq_bf16* k_origin,
                               kvq_bf16* k_step, uint8_t* v_codes, kvq_bf16* v_origin,
                               kvq_bf16* v_step, cudaStream_t s);

// Tensor-core decode (decode_mma.cu).  The plan cuts the weighted item
// sequence (per unit: its groups, then its residual) into n_slots warp
// slices; each unit's partials occupy max_parts slots of the workspace.
struct MmaPlan {
  long long unit_len;
  int n_slots;
  int max_parts;
};
int mma_warps_per_cta(const RecLayout& lay, int n_rep);
// false if even two partial slots per unit exceed ws_cap (0 = no cap)
bool mma_plan(int num_sms, int units, int n_rep, int n_groups, int r, int sink,
              const RecLayout& lay, size_t ws_cap, MmaPlan* plan);
size_t mma_ws_bytes(int num_sms, int B, int Hkv, int Hq, int max_groups, const RecLayout& lay);
// new_k, new_v (or NULL): a token [B][Hkv][D] the kernel writes into
// residual slot c->r - 1 before reading the residual (a fused append).
cudaError_t launch_decode_mma(const kvq_cache* c, const kvq_bf16* q, int Hq, float* out,
                              float* ws, const MmaPlan& plan, const kvq_bf16* new_k,
                              const kvq_bf16* new_v, cudaStream_t s);
// Merge split-K partials [units][max_parts][n_rep][D + 2] (o, m, l) of the
// slots of a plan into out [B][Hq][D]; launched as a programmatic dependent
// of the kernel that wrote them.
cudaError_t launch_combine_parts(const float* ws, int B, int Hkv, int Hq, int max_parts,
                                 long long unit_len, long long total, int n_slots, float* out,
                                 cudaStream_t s);

// bf16 comparator (decode.cu): stream-K over 16-token chunks of plain bf16
// K, V; workspace as the quantized decode's.
size_t bf16_ws_bytes(int num_sms, int B, int Hkv, int Hq, int T);
cudaError_t launch_decode_bf16(const kvq_bf16* k, const kvq_bf16* v, int B, int Hkv, int T,
                               const kvq_bf16* q, int Hq, float* out, float* ws,
                               size_t ws_bytes, int num_sms, cudaStream_t s);

cudaError_t launch_saliency(const kvq_bf16* q_win, int Hq, int Lq,
                            const kvq_bf16* k_grp, int B, int Hkv, int G,
                            int sal_bits, const kvq_tier_spec* spec,
                            float* I_out, float* A_out, uint8_t* tiers_out,
                            cudaStream_t s);
// Online saliency (saliency.cu): qacc[u][d] += |q| of the unit's query
// heads, in head order; I[u][d] = qacc[u][d] / count.
cudaError_t launch_observe_query(const kvq_cache* c, const kvq_bf16* q, int Hq, cudaStream_t s);
cudaError_t launch_window_importance(const kvq_cache* c, float* I, cudaStream_t s);

cudaError_t launch_export_k_uniform(const kvq_cache* c, uint8_t* codes,
                                    kvq_bf16* kmin, float* kscale,
                                    cudaStream_t s);
cudaError_t launch_export_v(const kvq_cache* c, uint8_t* codes, kvq_bf16* vmin,
                            float* vscale, cudaStream_t s);
cudaError_t launch_export_k_mixed(const kvq_cache* c, uint8_t* counts, uint8_t* perm,
                                  kvq_bf16* raw, uint8_t* c4, kvq_bf16* m4,
                                  float* s4, uint8_t* c2, kvq_bf16* m2,
                                  float* s2, cudaStream_t s);


}  // namespace kvq
