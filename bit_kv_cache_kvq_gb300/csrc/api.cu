// extern "C" entry points of libkvq.so (declared and documented in kvq.h).
// Host side only: argument checks, the cache handle and its lengths, and the
// kernel launches.  Every check runs before anything is enqueued, so a call
// that returns an error leaves the cache unchanged.
#include <cuda_runtime.h>

#include <new>

#include "kvq_internal.h"

using namespace kvq;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool valid_config(const kvq_config* c) {
  if (!c) return false;
  if (c->batch < 1 || c->kv_heads < 1 || c->max_tokens < 0) return false;
  if (c->head_dim != kD) return false;
  if (c->max_tokens % kKG) return false;
  if (c->v_bits != 2 && c->v_bits != 4) return false;
  if (c->n_sink < 0 || c->n_sink > kR) return false;
  if (c->k_mode == KVQ_K_UNIFORM) {
    if (c->k_bits != 2 && c->k_bits != 4) return false;
  } else if (c->k_mode == KVQ_K_PNMIX) {
    if (c->n_high_pairs < 0 || c->n_high_pairs > kD / 2 || c->n_high_pairs % 16) return false;
    if (c->pair_layout != KVQ_PAIRS_ADJACENT && c->pair_layout != KVQ_PAIRS_SPLIT) return false;
    if (c->n_sink != 0) return false;
  } else if (c->k_mode == KVQ_K_KIVI) {
    // KIVI-2 and KIVI-4: keys and values at the same width; no sink window
    if ((c->k_bits != 2 && c->k_bits != 4) || c->v_bits != c->k_bits) return false;
    if (c->n_sink != 0) return false;
  } else if (c->k_mode == KVQ_K_MIXED) {
    if (c->n_bf16 < 0 || c->n_uint4 < 0 || c->n_bf16 + c->n_uint4 > kD) return false;
    if (c->tier_mode == KVQ_TIERS_THRESHOLD) {
      if (c->tau_bf16 != c->tau_bf16 || c->tau_uint4 != c->tau_uint4) return false;  // NaN
    } else if (c->tier_mode != KVQ_TIERS_RANK) {
      return false;
    }
  } else {
    return false;
  }
  return true;
}

RecLayout layout_of(const kvq_config* c) {
  return make_layout(c->k_mode == KVQ_K_MIXED, c->k_mode == KVQ_K_MIXED ? 2 : c->k_bits,
                     c->v_bits, c->n_bf16, c->n_uint4,
                     c->k_mode == KVQ_K_MIXED && c->tier_mode == KVQ_TIERS_THRESHOLD,
                     c->k_mode == KVQ_K_KIVI,
                     c->k_mode == KVQ_K_PNMIX ? 2 * c->n_high_pairs : -1);
}

bool is_pnmix(const kvq_cache* c) { return c->cfg.k_mode == KVQ_K_PNMIX; }

bool is_kivi(const kvq_cache* c) { return c->cfg.k_mode == KVQ_K_KIVI; }

// Rows [first, first + count) of src [units][L][D] into rows [dst_first,
// dst_first + count) of dst [units][cap][D].
cudaError_t copy_rows(const kvq_bf16* src, int L, int first, int count, kvq_bf16* dst, int cap,
                      int dst_first, int units, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const size_t row = static_cast<size_t>(kD) * sizeof(kvq_bf16);
  return cudaMemcpy2DAsync(dst + static_cast<size_t>(dst_first) * kD, cap * row,
                           src + static_cast<size_t>(first) * kD, static_cast<size_t>(L) * row,
                           count * row, units, cudaMemcpyDeviceToDevice, s);
}

// KIVI prefill of L tokens: the persisted state of L appends ("KIVI: KV
// cache axes" §5).  Keys: L - L mod 128 sealed in records; values: the
// first L - min(L, 128) quantized token by token into their records; the
// last min(L, 128) values in the FIFO ring (token t in slot t mod 128); the
// key residual holds the last L mod 128 keys.
int kivi_prefill(kvq_cache* c, const kvq_bf16* k, const kvq_bf16* v, int L, cudaStream_t s) {
  const int n_rec = L / kKG, r = L % kKG;
  if (n_rec * kKG > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  if (L == 0) return KVQ_OK;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  const QuantSrc src{k, v, static_cast<long long>(L) * kD, static_cast<long long>(kKG) * kD};
  cudaError_t e = launch_kivi_prefill(c, src, n_rec, L - kKG, s);
  if (e == cudaSuccess) e = copy_rows(k, L, n_rec * kKG, r, c->res_k, kR, 0, units, s);
  if (e == cudaSuccess && n_rec > 0)   // tokens L - 128 .. 128 n_rec - 1 -> slots r .. 127
    e = copy_rows(v, L, L - kKG, kKG - r, c->res_v, kR, r, units, s);
  if (e == cudaSuccess) e = copy_rows(v, L, n_rec * kKG, r, c->res_v, kR, 0, units, s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  c->t_q = n_rec * kKG;
  c->r = r;
  return KVQ_OK;
}

// KIVI append ("KIVI: KV cache axes" §4, Algorithm 1 order): once the FIFO
// holds 128 values, the one the new token displaces (slot r, token T_k -
// 128 + r of the newest record) is quantized into that record; the new key
// and value take slot r; a key residual reaching 128 tokens is sealed into
// a new record (four 32-token groups) and empties.
int kivi_append(kvq_cache* c, const kvq_bf16* k_new, const kvq_bf16* v_new, cudaStream_t s) {
  const bool seal = c->r + 1 == kR;
  if (seal && c->t_q + kKG > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  cudaError_t e = cudaSuccess;
  if (c->t_q > 0) {
    const QuantSrc ring{nullptr, c->res_v, static_cast<long long>(kR) * kD, 0};
    e = launch_kivi_values(c, ring, 1, c->t_q / kKG - 1, c->r, c->r + 1, 1 << 30, s);
  }
  if (e == cudaSuccess) e = launch_append(c, k_new, v_new, c->res_k, c->res_v, kR, c->r, s);
  if (e == cudaSuccess && seal) {
    const QuantSrc res{c->res_k, nullptr, static_cast<long long>(kR) * kD, 0};
    e = launch_kivi_seal(c, res, 1, c->t_q / kKG, s);
  }
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  if (seal) {
    c->t_q += kKG;
    c->r = 0;
  } else {
    c->r += 1;
  }
  return KVQ_OK;
}

struct Sizes {
  size_t records, residual, sink, qacc, perm, status, total;
};

Sizes sizes_of(const kvq_config* c) {
  const RecLayout L = layout_of(c);
  const size_t units = static_cast<size_t>(c->batch) * c->kv_heads;
  Sizes s;
  s.records = round_up(units * (c->max_tokens / kKG) * static_cast<size_t>(L.bytes));
  s.residual = round_up(units * kR * kD * sizeof(kvq_bf16));
  s.sink = round_up(units * static_cast<size_t>(c->n_sink) * kD * sizeof(kvq_bf16));
  s.qacc = c->k_mode == KVQ_K_MIXED ? round_up(units * kD * sizeof(float)) : 0;
  s.perm = c->k_mode == KVQ_K_PNMIX ? round_up(units * kD) : 0;
  s.status = kAlign;
  s.total = s.records + 2 * s.residual + 2 * s.sink + s.qacc + s.perm + s.status;
  return s;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" {

size_t kvq_cache_bytes(const kvq_config* cfg) {
  if (!valid_config(cfg)) return 0;
  return sizes_of(cfg).total;
}

int kvq_cache_alloc(const kvq_config* cfg, void* dev_buf, size_t buf_bytes,
                    cudaStream_t s, kvq_cache** out) {
  if (!out || !cfg) return KVQ_ERR_ARG;
  *out = nullptr;
  if (cfg->head_dim != kD) return KVQ_ERR_SHAPE;
  if (!valid_config(cfg)) return KVQ_ERR_ARG;
  const Sizes sz = sizes_of(cfg);
  if (dev_buf) {
    if (buf_bytes < sz.total) return KVQ_ERR_CAPACITY;
    if (reinterpret_cast<uintptr_t>(dev_buf) % kAlign) return KVQ_ERR_ARG;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KVQ_ERR_CUDA;
  kvq_cache* c = new (std::nothrow) kvq_cache{};
  if (!c) return KVQ_ERR_CUDA;
  c->cfg = *cfg;
  if (cfg->k_mode == KVQ_K_MIXED) c->cfg.k_bits = 2;
  c->lay = layout_of(cfg);
  c->device = dev;
  c->num_sms = sms;
  c->bytes = sz.total;
  c->owned = dev_buf == nullptr;
  if (c->owned) {
    void* p = nullptr;
    if (cudaMallocAsync(&p, sz.total, s) != cudaSuccess) {
      delete c;
      return KVQ_ERR_CUDA;
    }
    c->base = static_cast<uint8_t*>(p);
  } else {
    c->base = static_cast<uint8_t*>(dev_buf);
  }
  c->records = c->base;
  c->max_groups = cfg->max_tokens / kKG;
  c->res_k = reinterpret_cast<kvq_bf16*>(c->base + sz.records);
  c->res_v = reinterpret_cast<kvq_bf16*>(c->base + sz.records + sz.residual);
  c->sink_k = reinterpret_cast<kvq_bf16*>(c->base + sz.records + 2 * sz.residual);
  c->sink_v = reinterpret_cast<kvq_bf16*>(c->base + sz.records + 2 * sz.residual + sz.sink);
  uint8_t* tail = c->base + sz.records + 2 * sz.residual + 2 * sz.sink;
  c->qacc = sz.qacc ? reinterpret_cast<float*>(tail) : nullptr;
  c->pn_perm = sz.perm ? tail + sz.qacc : nullptr;
  c->pn_ready = false;
  c->status = reinterpret_cast<unsigned*>(tail + sz.qacc + sz.perm);
  c->t_q = 0;
  c->r = 0;
  c->s = 0;
  c->q_steps = 0;
  c->q_rep = 0;
  // the online |q| sums, the PN-Mix order and the status word are adjacent
  if (cudaMemsetAsync(tail, 0, sz.qacc + sz.perm + sizeof(unsigned), s) != cudaSuccess) {
    if (c->owned) cudaFreeAsync(c->base, s);
    delete c;
    return KVQ_ERR_CUDA;
  }
  *out = c;
  return KVQ_OK;
}

int kvq_cache_free(kvq_cache* c, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  cudaError_t e = cudaSuccess;
  if (c->owned) e = cudaFreeAsync(c->base, s);
  delete c;
  return cuda_status(e);
}

int kvq_cache_lengths(const kvq_cache* c, int* quantized_tokens, int* residual_tokens) {
  if (!c) return KVQ_ERR_ARG;
  if (quantized_tokens) *quantized_tokens = c->t_q;
  if (residual_tokens) *residual_tokens = c->r;
  return KVQ_OK;
}

int kvq_cache_sink_tokens(const kvq_cache* c, int* sink_tokens) {
  if (!c || !sink_tokens) return KVQ_ERR_ARG;
  *sink_tokens = c->s;
  return KVQ_OK;
}

int kvq_cache_reset(kvq_cache* c, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (cudaMemsetAsync(c->status, 0, sizeof(unsigned), s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (c->qacc && cudaMemsetAsync(c->qacc, 0, sizeof(float) * kD * c->cfg.batch * c->cfg.kv_heads,
                                 s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  c->t_q = 0;
  c->r = 0;
  c->s = 0;
  c->q_steps = 0;
  c->q_rep = 0;
  c->pn_ready = false;   // a new prefill selects its pairs again
  return KVQ_OK;
}

int kvq_pnmix_pairs(kvq_cache* c, const kvq_bf16* q, int Hq, int Lq, const kvq_bf16* k, int Lk,
                    float* sigma, cudaStream_t s) {
  if (!c || !q || !k || Lq < 1 || Lk < 1 || !aligned16(k)) return KVQ_ERR_ARG;
  if (!is_pnmix(c)) return KVQ_ERR_MODE;
  if (Hq < c->cfg.kv_heads || Hq % c->cfg.kv_heads) return KVQ_ERR_SHAPE;
  if (c->t_q != 0 || c->r != 0) return KVQ_ERR_NOT_EMPTY;
  if (launch_pnmix_pairs(c, q, Hq, Lq, k, Lk, sigma, s) != cudaSuccess) return KVQ_ERR_CUDA;
  c->pn_ready = true;
  return KVQ_OK;
}

int kvq_export_pnmix(const kvq_cache* c, uint8_t* codes, float* offset, float* scale,
                     uint8_t* high, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (!is_pnmix(c)) return KVQ_ERR_MODE;
  if (c->t_q > 0 && (!codes || !offset || !scale)) return KVQ_ERR_ARG;
  return cuda_status(launch_export_pnmix(c, codes, offset, scale, high, s));
}

int kvq_append_residual(kvq_cache* c, const kvq_bf16* k_new, const kvq_bf16* v_new,
                        cudaStream_t s) {
  if (!c || !k_new || !v_new) return KVQ_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if (is_kivi(c)) return kivi_append(c, k_new, v_new, s);
  if (c->s < c->cfg.n_sink) {   // the sequence's first tokens are the sinks
    const cudaError_t e = launch_append(c, k_new, v_new, c->sink_k, c->sink_v, c->cfg.n_sink,
                                        c->s, s);
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    c->s += 1;
    return KVQ_OK;
  }
  if (c->r >= kR) return KVQ_ERR_RESIDUAL_FULL;
  const cudaError_t e = launch_append(c, k_new, v_new, c->res_k, c->res_v, kR, c->r, s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  c->r += 1;
  return KVQ_OK;
}

static int check_importance(const kvq_cache* c, const float* importance) {
  if (c->cfg.k_mode == KVQ_K_MIXED) return importance ? KVQ_OK : KVQ_ERR_MODE;
  return importance ? KVQ_ERR_MODE : KVQ_OK;
}

int kvq_flush_group(kvq_cache* c, const float* importance, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (is_kivi(c)) return KVQ_ERR_MODE;   // KIVI seals its keys inside the append
  const bool mixed = c->cfg.k_mode == KVQ_K_MIXED;
  if (!mixed && importance) return KVQ_ERR_MODE;
  const bool window = mixed && !importance;   // I_d from the online window
  if (window && c->q_steps == 0) return KVQ_ERR_EMPTY;
  if (c->r != kR) return KVQ_ERR_RESIDUAL_NOT_FULL;
  if (c->t_q + kKG > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  if (is_pnmix(c) && !c->pn_ready) return KVQ_ERR_EMPTY;
  QuantSrc src{c->res_k, c->res_v, static_cast<long long>(kR) * kD, 0};
  cudaError_t e = launch_quantize(c, src, 1, c->t_q / kKG, importance, s);
  if (e == cudaSuccess && window)   // the next window starts from zero
    e = cudaMemsetAsync(c->qacc, 0, sizeof(float) * kD * c->cfg.batch * c->cfg.kv_heads, s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  c->t_q += kKG;
  c->r = 0;
  if (window) {
    c->q_steps = 0;
    c->q_rep = 0;
  }
  return KVQ_OK;
}

int kvq_observe_query(kvq_cache* c, const kvq_bf16* q, int Hq, cudaStream_t s) {
  if (!c || !q) return KVQ_ERR_ARG;
  if (c->cfg.k_mode != KVQ_K_MIXED) return KVQ_ERR_MODE;
  const int Hkv = c->cfg.kv_heads;
  if (Hq < Hkv || Hq % Hkv) return KVQ_ERR_SHAPE;
  if (c->q_steps && Hq / Hkv != c->q_rep) return KVQ_ERR_SHAPE;
  if (launch_observe_query(c, q, Hq, s) != cudaSuccess) return KVQ_ERR_CUDA;
  c->q_rep = Hq / Hkv;
  c->q_steps += 1;
  return KVQ_OK;
}

int kvq_quantize_prefill(kvq_cache* c, const kvq_bf16* k, const kvq_bf16* v, int L,
                         const float* importance, cudaStream_t s) {
  if (!c || L < 0) return KVQ_ERR_ARG;
  if (L > 0 && (!k || !v)) return KVQ_ERR_ARG;
  if (L > 0 && (!aligned16(k) || !aligned16(v))) return KVQ_ERR_ARG;
  const int m = check_importance(c, importance);
  if (m != KVQ_OK) return m;
  if (c->t_q != 0 || c->r != 0 || c->s != 0) return KVQ_ERR_NOT_EMPTY;
  if (is_kivi(c)) return kivi_prefill(c, k, v, L, s);
  if (is_pnmix(c) && !c->pn_ready && L >= kKG) return KVQ_ERR_EMPTY;   // pairs not selected
  const int sk = L < c->cfg.n_sink ? L : c->cfg.n_sink;   // sink tokens
  const int n_q = (L - sk) / kKG;
  const int r = (L - sk) % kKG;
  if (n_q * kKG > c->cfg.max_tokens) return KVQ_ERR_CAPACITY;
  if (L == 0) return KVQ_OK;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  cudaError_t e = launch_copy_tokens(k, v, L, 0, sk, c->sink_k, c->sink_v, c->cfg.n_sink, units, s);
  QuantSrc src{k + static_cast<size_t>(sk) * kD, v + static_cast<size_t>(sk) * kD,
               static_cast<long long>(L) * kD, static_cast<long long>(kKG) * kD};
  if (e == cudaSuccess) e = launch_quantize(c, src, n_q, 0, importance, s);
  if (e == cudaSuccess)
    e = launch_copy_tokens(k, v, L, sk + n_q * kKG, r, c->res_k, c->res_v, kR, units, s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  c->s = sk;
  c->t_q = n_q * kKG;
  c->r = r;
  return KVQ_OK;
}

size_t kvq_decode_workspace_bytes(const kvq_cache* c, int Hq) {
  if (!c || Hq < 1 || Hq % c->cfg.kv_heads) return 0;
  return mma_ws_bytes(c->num_sms, c->cfg.batch, c->cfg.kv_heads, Hq, c->max_groups, c->lay);
}

static bool valid_rep(int Hq, int Hkv) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return false;
  const int n = Hq / Hkv;
  return n == 1 || n == 2 || n == 4 || n == 8;
}

int kvq_decode_attention(const kvq_cache* c, const kvq_bf16* q, int Hq, float* out,
                         void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!c || !q || !out) return KVQ_ERR_ARG;
  if (!valid_rep(Hq, c->cfg.kv_heads)) return KVQ_ERR_SHAPE;
  if (c->s + c->t_q + c->r == 0) return KVQ_ERR_EMPTY;
  if (!ws || ws_bytes < kvq_decode_workspace_bytes(c, Hq) || !aligned16(ws))
    return KVQ_ERR_WORKSPACE;
  MmaPlan plan;
  if (!mma_plan(c->num_sms, c->cfg.batch * c->cfg.kv_heads, Hq / c->cfg.kv_heads,
                c->t_q / kKG, c->r, c->s, c->lay, ws_bytes, &plan))
    return KVQ_ERR_WORKSPACE;
  return cuda_status(
      launch_decode_mma(c, q, Hq, out, static_cast<float*>(ws), plan, nullptr, nullptr, s));
}

int kvq_decode_step(kvq_cache* c, const kvq_bf16* k_new, const kvq_bf16* v_new,
                    const float* importance, const kvq_bf16* q, int Hq, float* out, void* ws,
                    size_t ws_bytes, cudaStream_t s) {
  if (!c || !k_new || !v_new || !q || !out) return KVQ_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_ARG;
  if (!valid_rep(Hq, c->cfg.kv_heads)) return KVQ_ERR_SHAPE;
  if (!ws || ws_bytes < kvq_decode_workspace_bytes(c, Hq) || !aligned16(ws))
    return KVQ_ERR_WORKSPACE;
  if (is_kivi(c) || c->s < c->cfg.n_sink || c->r + 1 >= kR) {
    // the token goes to the sink window, or fills the residual (a flush
    // comes before the attention): the three calls in sequence
    int e = kvq_append_residual(c, k_new, v_new, s);
    if (e != KVQ_OK) return e;
    if (c->r == kR && (e = kvq_flush_group(c, importance, s)) != KVQ_OK) return e;
    return kvq_decode_attention(c, q, Hq, out, ws, ws_bytes, s);
  }
  // the decode kernel writes the token into residual slot r itself
  MmaPlan plan;
  if (!mma_plan(c->num_sms, c->cfg.batch * c->cfg.kv_heads, Hq / c->cfg.kv_heads,
                c->t_q / kKG, c->r + 1, c->s, c->lay, ws_bytes, &plan))
    return KVQ_ERR_WORKSPACE;
  c->r += 1;
  const cudaError_t e =
      launch_decode_mma(c, q, Hq, out, static_cast<float*>(ws), plan, k_new, v_new, s);
  if (e != cudaSuccess) {
    c->r -= 1;
    return KVQ_ERR_CUDA;
  }
  return KVQ_OK;
}

static int current_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

size_t kvq_decode_bf16_workspace_bytes(int B, int Hkv, int T, int Hq) {
  if (B < 1 || Hkv < 1 || T < 1 || !valid_rep(Hq, Hkv)) return 0;
  const int sms = current_sms();
  return sms ? bf16_ws_bytes(sms, B, Hkv, Hq, T) : 0;
}

int kvq_decode_bf16(const kvq_bf16* k, const kvq_bf16* v, int B, int Hkv, int T,
                    const kvq_bf16* q, int Hq, float* out, void* ws, size_t ws_bytes,
                    cudaStream_t s) {
  if (!k || !v || !q || !out || B < 1 || Hkv < 1 || T < 1) return KVQ_ERR_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q)) return KVQ_ERR_ARG;
  if (!valid_rep(Hq, Hkv)) return KVQ_ERR_SHAPE;
  const int sms = current_sms();
  if (!sms) return KVQ_ERR_CUDA;
  if (!ws || ws_bytes < bf16_ws_bytes(sms, B, Hkv, Hq, T) || !aligned16(ws))
    return KVQ_ERR_WORKSPACE;
  return cuda_status(launch_decode_bf16(k, v, B, Hkv, T, q, Hq, out, static_cast<float*>(ws),
                                        ws_bytes, sms, s));
}

int kvq_channel_saliency(const kvq_bf16* q_win, int Hq, int Lq, const kvq_bf16* k_grp,
                         int B, int Hkv, int G, int sal_bits, const kvq_tier_spec* spec,
                         float* I_out, float* A_out, uint8_t* tiers_out, cudaStream_t s) {
  if (!q_win || !k_grp || !spec || B < 1 || Hkv < 1 || Lq < 1 || G < 1) return KVQ_ERR_ARG;
  if (Hq < Hkv || Hq % Hkv) return KVQ_ERR_SHAPE;
  if (sal_bits < 1 || sal_bits > 8) return KVQ_ERR_ARG;
  if (spec->mode == KVQ_TIERS_RANK) {
    if (spec->n_bf16 < 0 || spec->n_uint4 < 0 || spec->n_bf16 + spec->n_uint4 > kD)
      return KVQ_ERR_ARG;
  } else if (spec->mode != KVQ_TIERS_THRESHOLD) {
    return KVQ_ERR_ARG;
  }
  return cuda_status(launch_saliency(q_win, Hq, Lq, k_grp, B, Hkv, G, sal_bits, spec,
                                     I_out, A_out, tiers_out, s));
}

int kvq_cache_status(kvq_cache* c, cudaStream_t s, int* status) {
  if (!c || !status) return KVQ_ERR_ARG;
  unsigned host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, c->status, sizeof host, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  *status = static_cast<int>(host);
  return KVQ_OK;
}

int kvq_export_k(const kvq_cache* c, uint8_t* codes, kvq_bf16* kmin, float* kscale,
                 cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (c->cfg.k_mode != KVQ_K_UNIFORM) return KVQ_ERR_MODE;
  if (c->t_q == 0) return KVQ_OK;   // nothing to copy; empty buffers may be NULL
  if (!codes || !kmin || !kscale) return KVQ_ERR_ARG;
  return cuda_status(launch_export_k_uniform(c, codes, kmin, kscale, s));
}

int kvq_export_v(const kvq_cache* c, uint8_t* codes, kvq_bf16* vmin, float* vscale,
                 cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (c->t_q == 0) return KVQ_OK;
  if (!codes || !vmin || !vscale) return KVQ_ERR_ARG;
  return cuda_status(launch_export_v(c, codes, vmin, vscale, s));
}

int kvq_export_residual(const kvq_cache* c, kvq_bf16* k_r, kvq_bf16* v_r, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (c->r == 0) return KVQ_OK;   // nothing to copy; empty buffers may be NULL
  if (!k_r || !v_r) return KVQ_ERR_ARG;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  const size_t row = kD * sizeof(kvq_bf16);
  cudaError_t e = cudaMemcpy2DAsync(k_r, c->r * row, c->res_k, kR * row, c->r * row, units,
                                    cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(v_r, c->r * row, c->res_v, kR * row, c->r * row, units,
                          cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

int kvq_export_sink(const kvq_cache* c, kvq_bf16* k, kvq_bf16* v, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (c->s == 0) return KVQ_OK;   // nothing to copy; empty buffers may be NULL
  if (!k || !v) return KVQ_ERR_ARG;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  const size_t row = kD * sizeof(kvq_bf16);
  const size_t cap = static_cast<size_t>(c->cfg.n_sink) * row;
  cudaError_t e = cudaMemcpy2DAsync(k, c->s * row, c->sink_k, cap, c->s * row, units,
                                    cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(v, c->s * row, c->sink_v, cap, c->s * row, units,
                          cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

int kvq_export_k_mixed(const kvq_cache* c, uint8_t* counts, uint8_t* perm, kvq_bf16* raw,
                       uint8_t* c4, kvq_bf16* m4, float* s4, uint8_t* c2, kvq_bf16* m2,
                       float* s2, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (c->cfg.k_mode != KVQ_K_MIXED) return KVQ_ERR_MODE;
  if (c->t_q == 0) return KVQ_OK;
  // a tier with no room has an empty (possibly NULL) destination
  const RecLayout& L = c->lay;
  if (!perm || (L.nb && !raw) || (L.n4 && (!c4 || !m4 || !s4)) ||
      (L.n2cap && (!c2 || !m2 || !s2)))
    return KVQ_ERR_ARG;
  return cuda_status(launch_export_k_mixed(c, counts, perm, raw, c4, m4, s4, c2, m2, s2, s));
}

int kvq_set_wait_limit(int polls) {
  const int previous = decode_wait_polls();
  set_decode_wait_polls(polls);
  return previous;
}

int kvq_set_decode_split_event(cudaEvent_t ev) {
  set_decode_split_event(ev);
  return KVQ_OK;
}

int kvq_export_kivi(const kvq_cache* c, uint8_t* k_codes, kvq_bf16* k_origin, kvq_bf16* k_step,
                    uint8_t* v_codes, kvq_bf16* v_origin, kvq_bf16* v_step, kvq_bf16* k_res,
                    kvq_bf16* v_res, cudaStream_t s) {
  if (!c) return KVQ_ERR_ARG;
  if (!is_kivi(c)) return KVQ_ERR_MODE;
  const int units = c->cfg.batch * c->cfg.kv_heads;
  const int total = c->t_q + c->r, rv = total < kR ? total : kR;
  cudaError_t e = cudaSuccess;
  if (c->t_q > 0) {
    if (!k_codes || !k_origin || !k_step || !v_codes || !v_origin || !v_step) return KVQ_ERR_ARG;
    e = launch_export_kivi(c, k_codes, k_origin, k_step, v_codes, v_origin, v_step, s);
  }
  if (e == cudaSuccess && c->r > 0) {
    if (!k_res) return KVQ_ERR_ARG;
    e = copy_rows(c->res_k, kR, 0, c->r, k_res, c->r, 0, units, s);
  }
  if (e == cudaSuccess && rv > 0) {   // the FIFO oldest first: slots r .. 127, then 0 .. r - 1
    if (!v_res) return KVQ_ERR_ARG;
    if (c->t_q > 0) e = copy_rows(c->res_v, kR, c->r, kR - c->r, v_res, rv, 0, units, s);
    if (e == cudaSuccess) e = copy_rows(c->res_v, kR, 0, c->r, v_res, rv, rv - c->r, units, s);
  }
  return cuda_status(e);
}

const char* kvq_status_string(int code) {
  switch (code) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_ARG: return "KVQ_ERR_ARG";
    case KVQ_ERR_SHAPE: return "KVQ_ERR_SHAPE";
    case KVQ_ERR_CAPACITY: return "KVQ_ERR_CAPACITY";
    case KVQ_ERR_RESIDUAL_FULL: return "KVQ_ERR_RESIDUAL_FULL";
    case KVQ_ERR_RESIDUAL_NOT_FULL: return "KVQ_ERR_RESIDUAL_NOT_FULL";
    case KVQ_ERR_EMPTY: return "KVQ_ERR_EMPTY";
    case KVQ_ERR_NOT_EMPTY: return "KVQ_ERR_NOT_EMPTY";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
    case KVQ_ERR_MODE: return "KVQ_ERR_MODE";
    default: return "KVQ_ERR_UNKNOWN";
  }
}

}  // extern "C"
