// Decode attention for callers that cannot allocate device memory.
//
// kvq_decode_attention needs a caller-provided workspace for its split-K
// partials.  Some callers cannot provide one: code running where every
// allocation must happen up front (an inference server that reserves all
// device memory at start-up and forbids cudaMalloc on the request path), a
// host that owns no allocator of its own (a plain C caller without a memory
// pool), or a step replayed from a recorded launch sequence where a fresh
// allocation would break the recording.  kvq_decode_attention_static serves
// them: its workspace is a fixed array in this library's device memory.
//
// The array below is a file-scope __device__ variable.  Every GPU that loads
// libkvq.so holds it (KVQ_STATIC_WORKSPACE_BYTES) until the process exits.
// Host code must not pass the name `g_static_ws` to a kernel: on the host it
// is only a stand-in symbol, not a device address.  The device address is
// looked up once per device with cudaGetSymbolAddress, on the first call made
// with that device current, and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

__device__ __align__(256) unsigned char g_static_ws[KVQ_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (looked up once).
cudaError_t static_ws_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int kvq_decode_attention_static(const kvq_cache* c, const kvq_bf16* q, int Hq,
                                           float* out, cudaStream_t s) {
  using namespace kvq;
  if (!c || !q || !out) return KVQ_ERR_ARG;
  if (Hq < 1 || Hq % c->cfg.kv_heads) return KVQ_ERR_SHAPE;
  const int n_rep = Hq / c->cfg.kv_heads;
  if (n_rep != 1 && n_rep != 2 && n_rep != 4 && n_rep != 8) return KVQ_ERR_SHAPE;
  if (c->s + c->t_q + c->r == 0) return KVQ_ERR_EMPTY;

  // Plan the split so its partials fit the fixed array; reject what cannot
  // fit with two partial slots per (batch row, KV head).
  MmaPlan plan;
  if (!mma_plan(c->num_sms, c->cfg.batch * c->cfg.kv_heads, n_rep, c->t_q / kKG, c->r, c->s,
                c->lay, KVQ_STATIC_WORKSPACE_BYTES, &plan))
    return KVQ_ERR_WORKSPACE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev != c->device) return KVQ_ERR_ARG;   // the array of the cache's own device
  void* ws = nullptr;
  if (static_ws_address(dev, &ws) != cudaSuccess) return KVQ_ERR_CUDA;
  // Every partial the combine reads is rewritten by this call (a warp whose
  // wait gave up writes empty partials for the units it leaves), so nothing
  // in the array has to start at zero.
  return launch_decode_mma(c, q, Hq, out, static_cast<float*>(ws), plan, nullptr, nullptr, s) ==
                 cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}
