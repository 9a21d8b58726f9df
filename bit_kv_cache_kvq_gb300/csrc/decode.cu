// Unquantized bf16 comparator: split-K ("flash-decoding") decode attention
// over plain bf16 K, V on CUDA cores, plus its combine kernel.
//
// Math ("KIVI: KV cache axes" §1 and §6; MixKVQ Algorithm 1): for query
// head h of KV head kvh, s_t = q·k^_t / sqrt(D) over the dequantized
// history and the residual tokens, p = softmax over all of them together,
// o = sum_t p_t v^_t.  Scores are kept in log2 units (q pre-scaled by
// log2(e)/sqrt(D)) so p = exp2(s - max).
//
// Work split: grid (n_split, B*Hkv).  A CTA streams a contiguous range of
// 128-token blocks of one (b, kv head) for all n_rep query heads that share
// it (GQA: each byte is read once).  Inside the CTA, teams of TL lanes each
// own whole blocks and keep their own online-softmax state; teams merge
// once at the end.  A second kernel merges the splits with the exact
// log-sum-exp rule (KIVI §6: blockwise softmax is allowed when the blocks
// share one global normalization).
#include <cuda_runtime.h>

#include <cfloat>

#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ float bf2f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void bf2x8(const uint4& w, float* f) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(v[i] << 16);
    f[2 * i + 1] = __uint_as_float(v[i] & 0xffff0000u);
  }
}

// Reductions over one team of TL lanes.  Teams of a warp run different
// numbers of groups (and only one team takes the residual), so every
// shuffle names the calling team's lanes only.
template <int TL>
__device__ __forceinline__ unsigned team_mask_of() {
  return (TL == 32 ? 0xffffffffu : ((1u << TL) - 1u)) << ((threadIdx.x & 31) / TL * TL);
}
template <int TL>
__device__ __forceinline__ float team_sum(float x) {
  const unsigned m = team_mask_of<TL>();
#pragma unroll
  for (int o = TL / 2; o > 0; o >>= 1) x += __shfl_xor_sync(m, x, o);
  return x;
}
template <int TL>
__device__ __forceinline__ float team_max(float x) {
  const unsigned m = team_mask_of<TL>();
#pragma unroll
  for (int o = TL / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(m, x, o));
  return x;
}

// Fields the partial writer needs.
struct DecodeArgs {
  int Hkv, Hq;
  int n_split;
  float* ws;              // o [rows][n_split][D], then (m, l) [rows][n_split][2]
};

template <int NREP>
struct TeamShape {
  static constexpr int TL = NREP <= 4 ? 8 : 16;  // lanes per team
  static constexpr int CPT = 128 / TL;           // tokens (QK) / channels (PV) per lane
  static constexpr int TEAMS = 128 / TL;         // teams per 128-thread CTA
};

// Online-softmax state of one lane: its running max (team-uniform), its
// share of the normalizer, and the output accumulators of its CPT channels.
template <int NREP, int CPT>
struct SoftState {
  float m[NREP];
  float l[NREP];
  float o[CPT][NREP];
  __device__ void init() {
#pragma unroll
    for (int h = 0; h < NREP; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
#pragma unroll
      for (int i = 0; i < CPT; ++i) o[i][h] = 0.0f;
    }
  }
  // Fold a block of scores s[CPT][NREP] (masked entries -inf) into the
  // state and write exp2(s - m_new) to p_out[h][lane*CPT + i].
  template <int TL>
  __device__ void absorb(float (&s)[CPT][NREP], float* p_out, int li) {
#pragma unroll
    for (int h = 0; h < NREP; ++h) {
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < CPT; ++i) bm = fmaxf(bm, s[i][h]);
      bm = team_max<TL>(bm);
      const float m_new = fmaxf(m[h], bm);
      const float alpha = (m[h] == -INFINITY) ? 0.0f : exp2f(m[h] - m_new);
      l[h] *= alpha;
#pragma unroll
      for (int i = 0; i < CPT; ++i) o[i][h] *= alpha;
      m[h] = m_new;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const float p = (s[i][h] == -INFINITY) ? 0.0f : exp2f(s[i][h] - m_new);
        l[h] += p;
        p_out[h * 128 + li * CPT + i] = p;
      }
    }
  }
};

// Merge the teams of a CTA and write its partial (o, m, l) per query head.
template <int NREP, int TL, int CPT, int TEAMS, typename State>
__device__ void write_partial(const DecodeArgs& a, State& st, float* s_o,
                              float* s_ml, int team, int li, int b, int kvh,
                              int split) {
  __syncthreads();  // all teams done with their probability buffers
#pragma unroll
  for (int h = 0; h < NREP; ++h) {
    const float l = team_sum<TL>(st.l[h]);
#pragma unroll
    for (int i = 0; i < CPT; ++i) s_o[(team * NREP + h) * 128 + li * CPT + i] = st.o[i][h];
    if (li == 0) {
      s_ml[(team * NREP + h) * 2 + 0] = st.m[h];
      s_ml[(team * NREP + h) * 2 + 1] = l;
    }
  }
  __syncthreads();
  const int ch = threadIdx.x;  // 128 threads = 128 channels
  const long long rows = static_cast<long long>(gridDim.y / a.Hkv) * a.Hq;
  float* ws_o = a.ws;
  float* ws_ml = a.ws + rows * a.n_split * kD;
#pragma unroll
  for (int h = 0; h < NREP; ++h) {
    float M = -INFINITY;
    for (int t = 0; t < TEAMS; ++t) M = fmaxf(M, s_ml[(t * NREP + h) * 2]);
    float o = 0.0f, l = 0.0f;
    if (M != -INFINITY) {
      for (int t = 0; t < TEAMS; ++t) {
        const float mt = s_ml[(t * NREP + h) * 2];
        const float w = (mt == -INFINITY) ? 0.0f : exp2f(mt - M);
        o += w * s_o[(t * NREP + h) * 128 + ch];
        l += w * s_ml[(t * NREP + h) * 2 + 1];
      }
    }
    const long long row = static_cast<long long>(b) * a.Hq + kvh * NREP + h;
    ws_o[(row * a.n_split + split) * kD + ch] = o;
    if (ch == 0) {
      ws_ml[(row * a.n_split + split) * 2 + 0] = M;
      ws_ml[(row * a.n_split + split) * 2 + 1] = l;
    }
  }
}

// ---------------------------------------------------------------------------
// Unquantized comparator: identical split-K skeleton over bf16 K, V
// [units][T][D].  A "group" is 128 consecutive tokens; the last is ragged.
struct Bf16Args {
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* q;
  int T, Hkv, Hq;
  int n_groups, n_split, gps;
  float* ws;
  float qscale;
  // fields read by write_partial
};

template <int NREP>
__global__ void __launch_bounds__(128) decode_bf16_kernel(Bf16Args a, DecodeArgs shape) {
  using Shape = TeamShape<NREP>;
  constexpr int TL = Shape::TL, CPT = Shape::CPT, TEAMS = Shape::TEAMS;
  __shared__ float s_q[NREP * kD];
  __shared__ float s_p[TEAMS * NREP * 128];
  __shared__ float s_ml[TEAMS * NREP * 2];
  const int split = blockIdx.x;
  const int u = blockIdx.y;
  const int b = u / a.Hkv, kvh = u % a.Hkv;
  const int team = threadIdx.x / TL, li = threadIdx.x % TL;
  const unsigned team_mask = team_mask_of<TL>();
  for (int i = threadIdx.x; i < NREP * kD; i += blockDim.x) {
    const int h = i / kD, d = i % kD;
    s_q[i] = bf2f(a.q[(static_cast<long long>(b) * a.Hq + kvh * NREP + h) * kD + d]) * a.qscale;
  }
  __syncthreads();
  SoftState<NREP, CPT> st;
  st.init();
  float* p_buf = s_p + team * NREP * 128;
  const uint16_t* kbase = a.k + static_cast<long long>(u) * a.T * kD;
  const uint16_t* vbase = a.v + static_cast<long long>(u) * a.T * kD;
  const int g_begin = split * a.gps;
  const int g_end = min(g_begin + a.gps, a.n_groups);
  for (int g = g_begin + team; g < g_end; g += TEAMS) {
    const int t0 = g * 128;
    const int nt = min(128, a.T - t0);
    float s[CPT][NREP];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const int t = li * CPT + i;
      float acc[NREP];
#pragma unroll
      for (int h = 0; h < NREP; ++h) acc[h] = 0.0f;
      if (t < nt) {
        const uint4* row = reinterpret_cast<const uint4*>(kbase + static_cast<long long>(t0 + t) * kD);
#pragma unroll 4
        for (int dc = 0; dc < kD / 8; ++dc) {
          float f[8];
          bf2x8(__ldg(row + dc), f);
#pragma unroll
          for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int h = 0; h < NREP; ++h) acc[h] = fmaf(s_q[h * kD + dc * 8 + e], f[e], acc[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < NREP; ++h) s[i][h] = (t < nt) ? acc[h] : -INFINITY;
    }
    st.template absorb<TL>(s, p_buf, li);
    __syncwarp(team_mask);
    const uint16_t* vrow0 = vbase + static_cast<long long>(t0) * kD + li * CPT;
#pragma unroll 2
    for (int t = 0; t < nt; ++t) {
      float vf[CPT];
#pragma unroll
      for (int c8 = 0; c8 < CPT / 8; ++c8)
        bf2x8(__ldg(reinterpret_cast<const uint4*>(vrow0 + static_cast<long long>(t) * kD) + c8), vf + 8 * c8);
#pragma unroll
      for (int h = 0; h < NREP; ++h) {
        const float p = p_buf[h * 128 + t];
#pragma unroll
        for (int i = 0; i < CPT; ++i) st.o[i][h] = fmaf(p, vf[i], st.o[i][h]);
      }
    }
    __syncwarp(team_mask);
  }
  write_partial<NREP, TL, CPT, TEAMS>(shape, st, s_p, s_ml, team, li, b, kvh, split);
}

// Exact merge of the split partials: M = max m_i, o = sum 2^(m_i-M) o_i /
// sum 2^(m_i-M) l_i.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ ws,
                                                     int rows, int n_split,
                                                     float* __restrict__ out) {
  const long long row = blockIdx.x;
  const int ch = threadIdx.x;
  const float* ws_o = ws;
  const float* ws_ml = ws + static_cast<long long>(rows) * n_split * kD;
  float M = -INFINITY;
  for (int i = 0; i < n_split; ++i) M = fmaxf(M, ws_ml[(row * n_split + i) * 2]);
  float o = 0.0f, l = 0.0f;
  for (int i = 0; i < n_split; ++i) {
    const float mi = ws_ml[(row * n_split + i) * 2];
    if (mi == -INFINITY) continue;
    const float w = exp2f(mi - M);
    o = fmaf(w, ws_o[(row * n_split + i) * kD + ch], o);
    l = fmaf(w, ws_ml[(row * n_split + i) * 2 + 1], l);
  }
  out[row * kD + ch] = o / l;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

int choose_splits(int num_sms, int units, int n_chunks) {
  const int target = 4 * num_sms;  // CTAs wanted in flight
  int n = (target + units - 1) / units;
  n = min(n, max(n_chunks, 1));
  n = min(n, kMaxSplits);
  return max(n, 1);
}

cudaError_t launch_combine(const float* ws, int rows, int n_split, float* out,
                           cudaStream_t s) {
  combine_kernel<<<rows, kD, 0, s>>>(ws, rows, n_split, out);
  return cudaGetLastError();
}

cudaError_t launch_decode_bf16(const kvq_bf16* k, const kvq_bf16* v, int B,
                               int Hkv, int T, const kvq_bf16* q, int Hq,
                               float* out, float* ws, int n_split, int num_sms,
                               cudaStream_t s) {
  (void)num_sms;
  Bf16Args a;
  a.k = k;
  a.v = v;
  a.q = q;
  a.T = T;
  a.Hkv = Hkv;
  a.Hq = Hq;
  a.n_groups = (T + 127) / 128;
  a.n_split = n_split;
  a.gps = (a.n_groups + n_split - 1) / n_split;
  a.ws = ws;
  a.qscale = kLog2e / sqrtf(static_cast<float>(kD));
  DecodeArgs shape{};
  shape.Hkv = Hkv;
  shape.Hq = Hq;
  shape.n_split = n_split;
  shape.ws = ws;
  const dim3 grid(n_split, B * Hkv);
  switch (Hq / Hkv) {
    case 1: decode_bf16_kernel<1><<<grid, 128, 0, s>>>(a, shape); break;
    case 2: decode_bf16_kernel<2><<<grid, 128, 0, s>>>(a, shape); break;
    case 4: decode_bf16_kernel<4><<<grid, 128, 0, s>>>(a, shape); break;
    case 8: decode_bf16_kernel<8><<<grid, 128, 0, s>>>(a, shape); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(ws, B * Hq, n_split, out, s);
}

}  // namespace kvq
