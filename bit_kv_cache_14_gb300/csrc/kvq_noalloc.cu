// Decode attention whose scratch lives in a fixed device array, for callers
// that cannot allocate device memory (see kvq_decode_attention_noalloc in
// include/kvq.h).  Nothing here allocates: the scratch is a file-scope device
// array that exists on every GPU that loads the library, and its device
// address is looked up once per device.
#include <mutex>

#include "kvq_internal.cuh"

// The shared scratch.  Host code only sees a stand-in symbol; its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_mu;
void *g_scratch_addr[kvq::kMaxDevices] = {nullptr};

// Device address of the scratch on the current device (its primary
// context); looked up on the first call made with that device current.
int scratch_address(void **out) {
  const int dev = kvq::device_slot();
  if (dev < 0) return KVQ_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, kvq_noalloc_scratch) != cudaSuccess || p == nullptr)
      return KVQ_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" int kvq_decode_attention_noalloc(const kvq_config *cfg, const kvq_cache *cache,
                                            const uint16_t *q, float *out,
                                            float softmax_scale, void *stream) {
  kvq::Geometry g;
  int r = kvq::resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  const size_t need = kvq::decode_workspace_bytes(g);
  if (need > (size_t)KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ECAPACITY;
  void *ws = nullptr;
  if ((r = scratch_address(&ws)) != KVQ_OK) return r;
  // every check of the regular decode first: a rejected call enqueues nothing
  // and leaves the shared array alone
  if ((r = kvq::check_decode_call(g, cache, q, out, softmax_scale, ws,
                                  (size_t)KVQ_NOALLOC_SCRATCH_BYTES)) != KVQ_OK)
    return r;
  // The scratch must read zero when a decode starts; a successful decode
  // leaves it so, but another call may have stopped early: clear the part
  // this configuration uses.
  if (cudaMemsetAsync(ws, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVQ_ECUDA;
  return kvq_decode_attention(cfg, cache, q, out, softmax_scale, ws,
                              (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
}
