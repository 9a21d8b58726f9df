// Split-K partial merge (combine kernels), split planning and the launch of
// the tensor-core decode (the kernel itself is in decode_mma.cuh).
#include "decode_mma.cuh"

namespace kvq {
namespace {

// Merge the partials (o, m, l) of one query head (block = (b, hq), thread =
// channel) with the log-sum-exp rule: M = max m_k, w_k = 2^(m_k - M),
// o = sum w_k o_k / sum w_k l_k.  Every warp takes the weights itself (lane
// k % 32 holds part k's), so no block barrier is needed, and the values of
// the first 32 parts load together with the maxima: for up to 32 parts the
// merge is one round trip to memory.  Launched as a programmatic dependent
// of the decode kernel: it may start while that kernel drains and waits for
// its results with griddepcontrol.wait.
__global__ void __launch_bounds__(128) combine_parts_kernel(const float* __restrict__ ws,
                                                           int Hkv, int Hq, int max_parts,
                                                           long long unit_len, long long total,
                                                           int n_slots, float* __restrict__ out) {
  constexpr int kEarly = 32;
  const int row = blockIdx.x;                 // b * Hq + hq
  const int n_rep = Hq / Hkv;
  const int b = row / Hq, hq = row % Hq;
  const int u = b * Hkv + hq / n_rep, h = hq % n_rep;
  const long long ub = static_cast<long long>(u) * unit_len;
  const int first = static_cast<int>(((ub + 1) * n_slots - 1) / total);
  const int last = static_cast<int>(((ub + unit_len) * n_slots - 1) / total);
  const int n = last - first + 1;
  const int c = threadIdx.x, lane = c & 31;
  const float* base = ws + static_cast<long long>(u) * max_parts * n_rep * (kD + 2) + h * (kD + 2);
  const long long stride = static_cast<long long>(n_rep) * (kD + 2);
  // Two passes over the same code: the first, with no parts, runs before
  // the wait and only brings the merge's instructions into the SM's
  // instruction cache (after an L2 flush every first fetch would otherwise
  // go to memory once the decode grid is done); the second merges.
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int np = pass ? n : 0;
    float o[kEarly];
#pragma unroll
    for (int j = 0; j < kEarly; ++j) o[j] = j < np ? base[j * stride + c] : 0.0f;
    const float m0 = lane < np ? base[lane * stride + kD] : -INFINITY;
    const float l0 = lane < np ? base[lane * stride + kD + 1] : 0.0f;
    float M = m0;
    for (int k = lane + 32; k < np; k += 32) M = fmaxf(M, base[k * stride + kD]);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, x));
    // parts 0..31: weights from lane k; a part that saw no token weighs 0
    float w = m0 == -INFINITY ? 0.0f : exp2f(m0 - M);
    float L = w * l0, O = 0.0f;
#pragma unroll
    for (int j = 0; j < kEarly; ++j) O = fmaf(__shfl_sync(kFull, w, j), o[j], O);
    // parts 32 and up, 32 at a time
    for (int k0 = 32; k0 < np; k0 += 32) {
      const int k = k0 + lane;
      const float mk = k < np ? base[k * stride + kD] : -INFINITY;
      w = mk == -INFINITY ? 0.0f : exp2f(mk - M);
      L = fmaf(w, k < np ? base[k * stride + kD + 1] : 0.0f, L);
      const int cnt = min(32, np - k0);
#pragma unroll 4
      for (int j = 0; j < cnt; ++j)
        O = fmaf(__shfl_sync(kFull, w, j), base[(k0 + j) * stride + c], O);
    }
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) L += __shfl_xor_sync(kFull, L, x);
    if (pass) out[static_cast<long long>(row) * kD + c] = O / L;
  }
}

// The same merge for rows with many partials (small batches split over
// the whole GPU): w warps a row, w = ceil(parts / 20) from 4 to 16.  Warp i
// takes parts 20 i .. 20 i + 19, then 20 (i + w) .., ...: per chunk the
// twenty parts' values (lane = channels 2l, 2l + 1, 64 + 2l, 65 + 2l), maxima
// and normalizers load together, and the chunk folds into the warp's
// running (M, L, O) by the log-sum-exp rule; the warps' states merge
// through shared memory by the same rule.  For up to 320 parts a row that
// is one round trip to memory.
constexpr int kWideParts = 20;   // parts a warp keeps in flight
constexpr int kWideWarps = 16;
constexpr size_t kSpreadSmem = 48 * 1024;
__global__ void __launch_bounds__(kWideWarps * 32) combine_wide_kernel(
    const float* __restrict__ ws, int Hkv, int Hq, int max_parts, long long unit_len,
    long long total, int n_slots, float* __restrict__ out) {
  __shared__ float sO[kWideWarps][kD];
  __shared__ float sM[kWideWarps], sL[kWideWarps];
  const int row = blockIdx.x;                 // b * Hq + hq
  const int n_rep = Hq / Hkv;
  const int b = row / Hq, hq = row % Hq;
  const int u = b * Hkv + hq / n_rep, h = hq % n_rep;
  const long long ub = static_cast<long long>(u) * unit_len;
  const int first = static_cast<int>(((ub + 1) * n_slots - 1) / total);
  const int last = static_cast<int>(((ub + unit_len) * n_slots - 1) / total);
  const int n = last - first + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const float* base = ws + static_cast<long long>(u) * max_parts * n_rep * (kD + 2) + h * (kD + 2);
  const long long stride = static_cast<long long>(n_rep) * (kD + 2);
  // Two passes over the same code, as in combine_parts_kernel: the first
  // (before the wait) runs one chunk with every load and the store turned
  // off; it only brings the instructions into the SM's instruction cache.
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass) asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int np = pass ? n : 0;
    float M = -INFINITY, L = 0.0f;
    float2 o0 = make_float2(0.0f, 0.0f), o1 = make_float2(0.0f, 0.0f);
    for (int c0 = warp * kWideParts; c0 < (pass ? np : kWideParts); c0 += nw * kWideParts) {
      float2 va[kWideParts], vb[kWideParts];
#pragma unroll
      for (int j = 0; j < kWideParts; ++j) {
        const bool ok = c0 + j < np;
        const float* pj = base + static_cast<long long>(c0 + j) * stride;
        va[j] = ok ? *reinterpret_cast<const float2*>(pj + 2 * lane) : make_float2(0.0f, 0.0f);
        vb[j] = ok ? *reinterpret_cast<const float2*>(pj + 64 + 2 * lane) : make_float2(0.0f, 0.0f);
      }
      const int kl = c0 + lane;
      const bool okl = lane < kWideParts && kl < np;
      const float mk = okl ? base[static_cast<long long>(kl) * stride + kD] : -INFINITY;
      const float lk = okl ? base[static_cast<long long>(kl) * stride + kD + 1] : 0.0f;
      float mc = mk;
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFull, mc, x));
      const float mn = fmaxf(M, mc);
      // running state rescaled to the new maximum; a part (or a state) that
      // saw no token weighs 0
      const float f = M == -INFINITY ? 0.0f : exp2f(M - mn);
      const float wk = mk == -INFINITY ? 0.0f : exp2f(mk - mn);
      float lw = wk * lk;
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) lw += __shfl_xor_sync(kFull, lw, x);
      L = fmaf(L, f, lw);
      o0.x *= f; o0.y *= f; o1.x *= f; o1.y *= f;
#pragma unroll
      for (int j = 0; j < kWideParts; ++j) {
        const float wj = __shfl_sync(kFull, wk, j);
        o0.x = fmaf(wj, va[j].x, o0.x); o0.y = fmaf(wj, va[j].y, o0.y);
        o1.x = fmaf(wj, vb[j].x, o1.x); o1.y = fmaf(wj, vb[j].y, o1.y);
      }
      M = mn;
    }
    sO[warp][2 * lane] = o0.x;
    sO[warp][2 * lane + 1] = o0.y;
    sO[warp][64 + 2 * lane] = o1.x;
    sO[warp][65 + 2 * lane] = o1.y;
    if (lane == 0) {
      sM[warp] = M;
      sL[warp] = L;
    }
    __syncthreads();
    if (threadIdx.x < kD) {
      const int ch = threadIdx.x;
      float Mx = -INFINITY;
      for (int w = 0; w < nw; ++w) Mx = fmaxf(Mx, sM[w]);
      float O = 0.0f, Lt = 0.0f;
      for (int w = 0; w < nw; ++w) {
        const float f = sM[w] == -INFINITY ? 0.0f : exp2f(sM[w] - Mx);
        O = fmaf(f, sO[w][ch], O);
        Lt = fmaf(f, sL[w], Lt);
      }
      if (pass) out[static_cast<long long>(row) * kD + ch] = O / Lt;
    }
    __syncthreads();   // the first pass's reads of the tables before the second's writes
  }
}

std::atomic<int> g_wait_polls{kWaitPolls};
std::atomic<cudaEvent_t> g_split_event{nullptr};

}  // namespace

void set_decode_split_event(cudaEvent_t ev) { g_split_event.store(ev, std::memory_order_relaxed); }

int decode_wait_polls() { return g_wait_polls.load(std::memory_order_relaxed); }
void set_decode_wait_polls(int polls) {
  g_wait_polls.store(polls < 0 ? kWaitPolls : polls, std::memory_order_relaxed);
}

int mma_warps_per_cta(const RecLayout& lay, int n_rep) {
  // one record buffer plus the query (and, with mixed keys, the tables) per
  // warp, within the 227 KB of shared memory a block may use, and at most
  // the variant's register-bound warp count
  const bool sep = lay.mixed != 0 || lay.kivi != 0;   // value tables in their own area
  const int per = lay.bytes + warp_extra(sep);
  return max(1, min(max_warps(lay.kb, lay.vb, n_rep, sep || lay.pnmix != 0), (227 * 1024) / per));
}

bool mma_plan(int num_sms, int units, int n_rep, int n_groups, int r, int sink,
              const RecLayout& lay, size_t ws_cap, MmaPlan* plan) {
  plan->unit_len = n_groups + (r > 0 ? kResidualWeight : 0) + (sink > 0 ? kResidualWeight : 0);
  const long long total = static_cast<long long>(units) * plan->unit_len;
  const long long resident = static_cast<long long>(num_sms) * mma_warps_per_cta(lay, n_rep);
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

size_t mma_ws_bytes(int num_sms, int B, int Hkv, int Hq, int max_groups, const RecLayout& lay) {
  // worst case over the lengths this cache can hold: one warp slot per
  // weighted position or all resident warps, whichever is fewer
  const int units = B * Hkv;
  const long long resident = static_cast<long long>(num_sms) * mma_warps_per_cta(lay, Hq / Hkv);
  const long long per_unit = (resident + units - 1) / units + 2;
  const long long cap = static_cast<long long>(max_groups) + 2 * kResidualWeight + 1;
  const long long parts = per_unit < cap ? per_unit : cap;
  return static_cast<size_t>(units) * parts * (Hq / Hkv) * (kD + 2) * sizeof(float);
}

cudaError_t launch_combine_parts(const float* ws, int B, int Hkv, int Hq, int max_parts,
                                 long long unit_len, long long total, int n_slots, float* out,
                                 cudaStream_t s) {
  // the combine's blocks land on SMs configured for the decode grid's
  // shared memory: ask for the same split so none has to reconfigure
  static const cudaError_t carve = cudaFuncSetAttribute(
      combine_parts_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
      cudaSharedmemCarveoutMaxShared);
  if (carve != cudaSuccess) return carve;
  static const cudaError_t carve_wide = cudaFuncSetAttribute(
      combine_wide_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
      cudaSharedmemCarveoutMaxShared);
  if (carve_wide != cudaSuccess) return carve_wide;
  // rows of up to 32 partials: one block of 128 threads a row; more: one
  // warp per 20 partials a row, at least 4 (the final merge takes a thread
  // per channel) and at most 16
  const bool many = max_parts > 32;
  const int wide_warps =
      max(kD / 32, min(kWideWarps, (max_parts + kWideParts - 1) / kWideParts));
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(B * Hq);
  lc.blockDim = dim3(many ? wide_warps * 32 : kD);
  // The decode blocks leave their SMs at different times and the first
  // SMs to free up would take every combine block (16 a SM), sharing their
  // L2 bandwidth; 48 KB of (unused) shared memory a block caps it at 4 a
  // SM, so the rows spread over ~B * Hq / 4 SMs.
  lc.dynamicSmemBytes = many ? 0 : kSpreadSmem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (many)
    return cudaLaunchKernelEx(&lc, combine_wide_kernel, ws, Hkv, Hq, max_parts, unit_len, total,
                              n_slots, out);
  return cudaLaunchKernelEx(&lc, combine_parts_kernel, ws, Hkv, Hq, max_parts, unit_len, total,
                            n_slots, out);
}

cudaError_t launch_decode_mma(const kvq_cache* c, const kvq_bf16* q, int Hq, float* out,
                              float* ws, const MmaPlan& plan, const kvq_bf16* new_k,
                              const kvq_bf16* new_v, cudaStream_t s) {
  MmaArgs a;
  a.records = c->records;
  a.rec_bytes = c->lay.bytes;
  a.max_groups = c->max_groups;
  a.lay = c->lay;
  a.n_groups = c->t_q / kKG;
  a.r = c->r;
  a.res_k = c->res_k;
  a.res_v = c->res_v;
  a.s = c->s;
  a.n_sink = c->cfg.n_sink;
  a.sink_k = c->sink_k;
  a.sink_v = c->sink_v;
  a.q = q;
  a.new_k = reinterpret_cast<const uint4*>(new_k);
  a.new_v = reinterpret_cast<const uint4*>(new_v);
  a.Hkv = c->cfg.kv_heads;
  a.Hq = Hq;
  a.units = c->cfg.batch * c->cfg.kv_heads;
  a.unit_len = plan.unit_len;
  a.n_slots = plan.n_slots;
  a.max_parts = plan.max_parts;
  a.total = static_cast<long long>(a.units) * a.unit_len;
  a.ws = ws;
  a.status = c->status;
  a.wait_polls = decode_wait_polls();
  a.perm = c->pn_perm;
  const int nrep = Hq / c->cfg.kv_heads;
  const int kb = c->cfg.k_bits, vb = c->cfg.v_bits;
  const int warps = mma_warps_per_cta(c->lay, nrep);
  cudaError_t e;
  if (c->lay.pnmix) {
    e = launch_decode_pnmix(a, nrep, vb, warps, s);
  } else if (c->lay.kivi) {
    e = launch_decode_kivi(a, nrep, kb, warps, s);
  } else if (c->cfg.k_mode == KVQ_K_MIXED) {
    if (vb == 2) e = launch_rep<2, 2, true>(a, nrep, warps, s);
    else e = launch_rep<2, 4, true>(a, nrep, warps, s);
  } else if (kb == 2 && vb == 2) {
    e = launch_rep<2, 2, false>(a, nrep, warps, s);
  } else if (kb == 2 && vb == 4) {
    e = launch_rep<2, 4, false>(a, nrep, warps, s);
  } else if (kb == 4 && vb == 2) {
    e = launch_rep<4, 2, false>(a, nrep, warps, s);
  } else {
    e = launch_rep<4, 4, false>(a, nrep, warps, s);
  }
  if (e != cudaSuccess) return e;
  // measurement hook: an event between the decode kernel and its combine
  if (cudaEvent_t ev = g_split_event.exchange(nullptr, std::memory_order_relaxed)) {
    e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) return e;
  }
  return launch_combine_parts(ws, c->cfg.batch, a.Hkv, Hq, a.max_parts, a.unit_len, a.total,
                              a.n_slots, out, s);
}

}  // namespace kvq
