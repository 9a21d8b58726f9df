// Unquantized comparator: decode attention over plain bf16 K, V (the 16-bit
// baseline the pages measure against: MixKVQ "BF16" rows, PN-Mix FP16).
//
// Same math as the quantized path (KIVI: KV cache axes §1, §6): s = q·k /
// sqrt(D) in log2 units, one softmax over all tokens, o = sum p v, split-K
// with an exact log-sum-exp combine.  Tensor cores do both contractions of
// every 16-token chunk: scores from bf16 MMAs of the exact keys and query
// (exact products, fp32 sums), P·V from the values transposed by ldmatrix
// and p split into bf16 high and low parts (16 bits), each chunk summed in a
// fresh accumulator and folded into the running output in fp32.
//
// Work split ("stream-K"): the (unit, chunk) items, units = (b, kv head),
// are cut into equal contiguous slices, one per warp of a persistent grid
// (12 warps per SM); each warp streams its chunks through two 8 KB slots
// (K and V of one chunk) of its own shared memory with 16-byte cp.async,
// the next chunk loading while the current one computes, and writes one
// partial per unit it touches.  combine_parts_kernel merges them.
#include <cuda_runtime.h>

#include "kvq_internal.h"
#include "mma_util.h"

namespace kvq {
namespace {

constexpr int kChunk = 16;                       // tokens per item
constexpr int kChunkBytes = kChunk * kD * 2;     // 4 KB of K (or V)
constexpr int kSlotBytes = 2 * kChunkBytes;      // K then V
constexpr int kWarps = 12;
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

struct Bf16Args {
  const uint8_t* k;   // [units][T][D] bf16
  const uint8_t* v;
  const uint16_t* q;  // [B][Hq][D]
  int Hkv, Hq, T, n_chunks;
  long long total;    // units * n_chunks
  int n_slots, max_parts;
  float* ws;          // [units][max_parts][n_rep][D + 2]
};

__device__ __forceinline__ long long slice_start(const Bf16Args& a, int w) {
  return (static_cast<long long>(w) * a.total) / a.n_slots;
}
__device__ __forceinline__ int slice_of(const Bf16Args& a, long long p) {
  return static_cast<int>(((p + 1) * a.n_slots - 1) / a.total);
}

// Chunk c of unit u (K and V, 16 rows of 256 B) into slot `slot`: 16-byte
// piece p of row t at piece p ^ (t & 7), so ldmatrix row reads are free of
// bank conflicts.  Rows past T repeat row T - 1 (never read past the
// tensor); their scores are masked.
__device__ __forceinline__ void stage(const Bf16Args& a, int u, int c, uint32_t slot_addr,
                                      int lane) {
  const long long ubase = static_cast<long long>(u) * a.T;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i, row = e >> 4, pc = e & 15;
    const int tok = min(c * kChunk + row, a.T - 1);
    const long long off = ((ubase + tok) * kD) * 2 + pc * 16;
    const uint32_t d = slot_addr + row * 256 + ((pc ^ (row & 7)) << 4);
    cp_async16(d, a.k + off);
    cp_async16(d + kChunkBytes, a.v + off);
  }
}

template <int NREP>
__global__ void __launch_bounds__(kWarps * 32, 1) decode_bf16_kernel(Bf16Args a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // the combine kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int slot = blockIdx.x * kWarps + warp;
  if (slot >= a.n_slots) return;   // warp-uniform
  const uint32_t buf = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) +
                       warp * 2 * kSlotBytes;
  const float c0 = kLog2e * rsqrtf(static_cast<float>(kD));
  const long long p0 = slice_start(a, slot), p1 = slice_start(a, slot + 1);
  for (int u = static_cast<int>(p0 / a.n_chunks); u <= static_cast<int>((p1 - 1) / a.n_chunks);
       ++u) {
    const long long ub = static_cast<long long>(u) * a.n_chunks;
    const int c_lo = static_cast<int>(max(p0, ub) - ub);
    const int c_hi = static_cast<int>(min(p1, ub + a.n_chunks) - ub);
    // query B fragments: column g = head g (zero for g >= NREP), exact bf16
    uint32_t bq[8][2];
    {
      const int b = u / a.Hkv, kvh = u % a.Hkv;
      const uint32_t* qg = reinterpret_cast<const uint32_t*>(
          a.q + (static_cast<long long>(b) * a.Hq + kvh * NREP + min(g, NREP - 1)) * kD);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        bq[ks][0] = g < NREP ? __ldg(qg + 8 * ks + t) : 0u;
        bq[ks][1] = g < NREP ? __ldg(qg + 8 * ks + t + 4) : 0u;
      }
    }
    float O[8][4];
#pragma unroll
    for (int mc = 0; mc < 8; ++mc)
#pragma unroll
      for (int i = 0; i < 4; ++i) O[mc][i] = 0.0f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.0f, 0.0f};

    __syncwarp();
    stage(a, u, c_lo, buf, lane);
    cp_async_commit();
    for (int c = c_lo; c < c_hi; ++c) {
      const uint32_t cur = buf + ((c - c_lo) & 1) * kSlotBytes;
      if (c + 1 < c_hi) stage(a, u, c + 1, buf + ((c + 1 - c_lo) & 1) * kSlotBytes, lane);
      cp_async_commit();
      cp_async_wait<1>();
      __syncwarp();
      // ---- scores of the chunk's 16 tokens
      float S[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      {
        const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int pc = 2 * ks + (lane >> 4);
          uint32_t A[4];
          ldsm_x4(A, cur + row * 256 + ((pc ^ (row & 7)) << 4));
          mma_bf16(S, A, bq[ks][0], bq[ks][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (c * kChunk + g + 8 * (i >> 1) >= a.T) S[i] = -INFINITY;
      // ---- online softmax (log2 units), per head column 2t + h
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float m = fmaxf(S[h], S[h + 2]);
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
        m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
        const float m_new = fmaxf(mrun[h], m * c0);
        alpha[h] = ex2(mrun[h] - m_new);
        mrun[h] = m_new;
        S[h] = ex2(fmaf(S[h], c0, -m_new));
        S[h + 2] = ex2(fmaf(S[h + 2], c0, -m_new));
        lrun[h] = fmaf(lrun[h], alpha[h], S[h] + S[h + 2]);
      }
      if (__any_sync(kFull, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
        for (int mc = 0; mc < 8; ++mc) {
          O[mc][0] *= alpha[0]; O[mc][2] *= alpha[0];
          O[mc][1] *= alpha[1]; O[mc][3] *= alpha[1];
        }
      }
      // ---- P·V: p as bf16 high + low B fragments, values transposed
      uint32_t ph[2], pl[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float x0 = S[2 * i], x1 = S[2 * i + 1];
        const uint32_t hi = pack_bf2(x0, x1);
        const float l0 = x0 - __uint_as_float(hi << 16);
        const float l1 = x1 - __uint_as_float(hi & 0xffff0000u);
        ph[i] = movmatrix_t(hi);
        pl[i] = movmatrix_t(pack_bf2(l0, l1));
      }
      {
        const uint32_t vb = cur + kChunkBytes;
        const int row = (lane & 7) + 8 * (lane >> 4);
#pragma unroll
        for (int mc = 0; mc < 8; ++mc) {
          const int pc = 2 * mc + ((lane >> 3) & 1);
          uint32_t A[4];
          ldsm_x4_t(A, vb + row * 256 + ((pc ^ (row & 7)) << 4));
          float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma_bf16(acc, A, ph[0], ph[1]);
          mma_bf16(acc, A, pl[0], pl[1]);
#pragma unroll
          for (int i = 0; i < 4; ++i) O[mc][i] += acc[i];
        }
      }
      __syncwarp();   // slot read before it is staged again
    }
    cp_async_wait<0>();
    __syncwarp();
    // ---- partial (o, m, l) of this unit's slice
    float l[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float x = lrun[h];
      x += __shfl_xor_sync(kFull, x, 4);
      x += __shfl_xor_sync(kFull, x, 8);
      x += __shfl_xor_sync(kFull, x, 16);
      l[h] = x;
    }
    const int part = slot - slice_of(a, ub);
    float* base = a.ws + (static_cast<long long>(u) * a.max_parts + part) * NREP * (kD + 2);
#pragma unroll
    for (int mc = 0; mc < 8; ++mc)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int h = 2 * t + (i & 1);
        if (h < NREP) base[h * (kD + 2) + 16 * mc + g + 8 * (i >> 1)] = O[mc][i];
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
}

struct Bf16Plan {
  int n_chunks;
  long long total;
  int n_slots, max_parts;
};

Bf16Plan plan_bf16(int num_sms, int units, int T) {
  Bf16Plan p;
  p.n_chunks = (T + kChunk - 1) / kChunk;
  p.total = static_cast<long long>(units) * p.n_chunks;
  const long long resident = static_cast<long long>(num_sms) * kWarps;
  p.n_slots = static_cast<int>(p.total < resident ? p.total : resident);
  // each unit's chunks meet at most ceil(slots / units) + 1 slots
  p.max_parts = (p.n_slots + units - 1) / units + 1;
  return p;
}

template <int NREP>
cudaError_t launch_nrep(const Bf16Args& a, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(kWarps) * 2 * kSlotBytes;
  auto kern = decode_bf16_kernel<NREP>;
  static SmemOptIn opt_in;
  cudaError_t e = opt_in.ensure(kern);
  if (e != cudaSuccess) return e;
  kern<<<(a.n_slots + kWarps - 1) / kWarps, kWarps * 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t bf16_ws_bytes(int num_sms, int B, int Hkv, int Hq, int T) {
  const int units = B * Hkv;
  const Bf16Plan p = plan_bf16(num_sms, units, T);
  return static_cast<size_t>(units) * p.max_parts * (Hq / Hkv) * (kD + 2) * sizeof(float);
}

cudaError_t launch_decode_bf16(const kvq_bf16* k, const kvq_bf16* v, int B, int Hkv, int T,
                               const kvq_bf16* q, int Hq, float* out, float* ws,
                               size_t ws_bytes, int num_sms, cudaStream_t s) {
  const int units = B * Hkv, nrep = Hq / Hkv;
  const Bf16Plan p = plan_bf16(num_sms, units, T);
  if (ws_bytes < bf16_ws_bytes(num_sms, B, Hkv, Hq, T)) return cudaErrorInvalidValue;
  Bf16Args a;
  a.k = reinterpret_cast<const uint8_t*>(k);
  a.v = reinterpret_cast<const uint8_t*>(v);
  a.q = q;
  a.Hkv = Hkv;
  a.Hq = Hq;
  a.T = T;
  a.n_chunks = p.n_chunks;
  a.total = p.total;
  a.n_slots = p.n_slots;
  a.max_parts = p.max_parts;
  a.ws = ws;
  cudaError_t e;
  switch (nrep) {
    case 1: e = launch_nrep<1>(a, s); break;
    case 2: e = launch_nrep<2>(a, s); break;
    case 4: e = launch_nrep<4>(a, s); break;
    case 8: e = launch_nrep<8>(a, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_combine_parts(ws, B, Hkv, Hq, p.max_parts, p.n_chunks, p.total, p.n_slots, out,
                              s);
}

}  // namespace kvq
