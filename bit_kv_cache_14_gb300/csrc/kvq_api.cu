// C ABI of libkvq: validation, buffer sizes, host counters, launches.
// Declarations and contracts: include/kvq.h.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "kvq_internal.cuh"
#include "kvq_rope.cuh"

namespace kvq {

namespace {
thread_local int t_last_launches = 0;

bool pow2_group(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// SM count per device, looked up once; calls from several host threads may
// race to fill an entry, and all of them store the same value.
int num_sms_cached() {
  static std::atomic<int> cache[kMaxDevices];
  const int dev = device_slot();
  if (dev < 0) return 152;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace

void note_launch(int n) { t_last_launches = n; }

int device_slot() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int resolve(const kvq_config *cfg, Geometry *g) {
  if (!cfg || !g) return KVQ_EINVAL;
  const kvq_config &c = *cfg;
  if (c.batch < 1 || c.n_kv_heads < 1 || c.n_q_heads < 1 || c.max_ctx < 1) return KVQ_EINVAL;
  // at most 2^30 tokens per sequence: every byte size below stays far from
  // overflow (65535 heads x 2^25 blocks x < 2^15 bytes)
  if (c.max_ctx > (1LL << 30)) return KVQ_EUNSUPPORTED;
  if (c.n_q_heads % c.n_kv_heads != 0) return KVQ_EINVAL;
  if (c.scheme != KVQ_KIVI && c.scheme != KVQ_INNERQ && c.scheme != KVQ_INNERQ_KNORM)
    return KVQ_EINVAL;
  if (c.residual < 0 || c.n_sink < 0 || c.k_group < 1 || c.v_group < 1) return KVQ_EINVAL;
  const int rg = c.n_q_heads / c.n_kv_heads;
  if (rg != 1 && rg != 2 && rg != 4 && rg != 8) return KVQ_EUNSUPPORTED;
  if (c.head_dim != 64 && c.head_dim != 128) return KVQ_EUNSUPPORTED;
  if (c.bits != 2 && c.bits != 4) return KVQ_EUNSUPPORTED;
  if ((int64_t)c.batch * c.n_kv_heads > 65535) return KVQ_EUNSUPPORTED;
  if (!pow2_group(c.v_group) || c.head_dim % c.v_group != 0) return KVQ_EUNSUPPORTED;
  if (c.residual > kMaxResidual || c.n_sink > kMaxResidual) return KVQ_EUNSUPPORTED;
  if (c.scheme == KVQ_KIVI) {
    if (c.n_sink != 0) return KVQ_EINVAL;
    if (c.residual < 1 || c.residual % c.k_group != 0) return KVQ_EINVAL;
    if (!pow2_group(c.k_group)) return KVQ_EUNSUPPORTED;
  } else {
    if (!pow2_group(c.k_group) || c.head_dim % c.k_group != 0) return KVQ_EUNSUPPORTED;
  }
  if ((c.flags & ~(KVQ_META_F16 | KVQ_VALUE_QUEUE | KVQ_RAGGED)) != 0) return KVQ_EINVAL;
  if (c.outliers < 0 || c.outliers > 8) return KVQ_EINVAL;
  if (c.scheme != KVQ_KIVI && ((c.flags & KVQ_VALUE_QUEUE) || c.outliers > 0)) return KVQ_EINVAL;
  g->B = c.batch;
  g->H = c.n_kv_heads;
  g->Hq = c.n_q_heads;
  g->d = c.head_dim;
  g->bits = c.bits;
  // the normalization is an InnerQ option: internally the scheme is InnerQ
  g->scheme = c.scheme == KVQ_INNERQ_KNORM ? KVQ_INNERQ : c.scheme;
  g->knorm = c.scheme == KVQ_INNERQ_KNORM ? 1 : 0;
  g->k_group = c.k_group;
  g->v_group = c.v_group;
  g->residual = c.residual;
  g->n_sink = c.n_sink;
  g->max_ctx = c.max_ctx;
  g->meta16 = (c.flags & KVQ_META_F16) ? 1 : 0;
  g->msz = g->meta16 ? 2 : 4;
  g->vq = (c.flags & KVQ_VALUE_QUEUE) ? 1 : 0;
  g->ragged = (c.flags & KVQ_RAGGED) ? 1 : 0;
  g->n_out = c.outliers;
  g->cap = (c.max_ctx + kCapAlign - 1) / kCapAlign * kCapAlign;
  g->row_bytes = c.head_dim * c.bits / 8;
  g->v_meta_cols = c.head_dim / c.v_group;
  if (g->scheme == KVQ_KIVI) {
    g->k_meta_cols = c.head_dim;
    g->k_meta_rows = g->cap / c.k_group;
    g->mode_words = 0;
  } else {
    g->k_meta_cols = c.head_dim / c.k_group;
    g->k_meta_rows = g->cap;
    g->mode_words = g->cap * (c.head_dim / c.k_group) / 32;
    const int64_t vw = g->cap * (c.head_dim / c.v_group) / 32;
    if (vw > g->mode_words) g->mode_words = vw;
  }
  const int vmeta = kBlockTokens * g->v_meta_cols * g->msz;
  g->blk_vc = kBlockTokens * g->row_bytes;
  g->blk_vs = 2 * kBlockTokens * g->row_bytes;
  g->blk_vz = g->blk_vs + vmeta;
  g->blk_ks = g->blk_vz + vmeta;
  int end;
  if (g->scheme == KVQ_INNERQ) {
    const int kmeta = kBlockTokens * g->k_meta_cols * g->msz;
    g->blk_kz = g->blk_ks + kmeta;
    end = g->blk_kz + kmeta;
  } else {
    // G <= 32: the statistics of the block's 32 / G key groups follow
    g->blk_kz = g->blk_ks;
    end = g->blk_ks + (c.k_group <= kBlockTokens
                           ? (kBlockTokens / c.k_group) * 2 * c.head_dim * g->msz
                           : 0);
  }
  // outlier lists: n_out words per token, keys then values
  g->blk_ko = end;
  g->blk_vo = g->blk_ko + kBlockTokens * g->n_out * 4;
  g->block_bytes = g->blk_vo + kBlockTokens * g->n_out * 4;
  g->knorm_off = (int64_t)g->B * g->H * (g->cap / kBlockTokens) * g->block_bytes;
  return KVQ_OK;
}

CachePtrs ptrs_of(const Geometry &g, const kvq_cache *c) {
  CachePtrs p;
  p.blocks = static_cast<uint8_t *>(c->blocks);
  p.k_norm = g.knorm ? reinterpret_cast<float *>(p.blocks + g.knorm_off) : nullptr;
  p.k_meta = static_cast<uint8_t *>(c->k_meta);
  p.k_mode = c->k_mode;
  p.v_mode = c->v_mode;
  p.k_res = reinterpret_cast<__half *>(c->k_res);
  p.v_res = reinterpret_cast<__half *>(c->v_res);
  p.k_sink = reinterpret_cast<__half *>(c->k_sink);
  p.v_sink = reinterpret_cast<__half *>(c->v_sink);
  p.status = c->dev_status;
  p.seq_prompt = g.ragged ? c->seq_prompt : nullptr;
  p.appended = c->n_appended;
  return p;
}

// The host counters as a Counts (n_vq: the value queue's count follows from
// the length).
static Counts host_counts(const Geometry &g, const kvq_cache *c) {
  Counts k;
  k.n_quant = c->n_quant;
  k.n_resid = c->n_resid;
  k.n_sink = c->n_sink;
  k.ring_head = c->ring_head;
  const int64_t n = c->n_quant + c->n_resid + c->n_sink;
  k.n_vq = (g.scheme == KVQ_KIVI && g.vq) ? (n >= g.residual ? n - g.residual + 1 : 0) : c->n_quant;
  return k;
}

// The buffers a configuration uses must be present and 16-byte aligned.
static int check_cache(const Geometry &g, const kvq_cache *c) {
  if (!c) return KVQ_EINVAL;
  if (!c->blocks) return KVQ_EINVAL;
  if (!aligned16(c->blocks)) return KVQ_EALIGN;
  if (g.scheme == KVQ_KIVI && g.k_group > kBlockTokens) {
    if (!c->k_meta) return KVQ_EINVAL;
    if (!aligned16(c->k_meta)) return KVQ_EALIGN;
  }
  if (g.residual > 0) {
    if (!c->k_res || !c->v_res) return KVQ_EINVAL;
    if (!aligned16(c->k_res) || !aligned16(c->v_res)) return KVQ_EALIGN;
  }
  if (g.scheme == KVQ_INNERQ) {
    if (!c->k_mode || !c->v_mode) return KVQ_EINVAL;
    if (!aligned16(c->k_mode) || !aligned16(c->v_mode)) return KVQ_EALIGN;
    if (g.n_sink > 0) {
      if (!c->k_sink || !c->v_sink) return KVQ_EINVAL;
      if (!aligned16(c->k_sink) || !aligned16(c->v_sink)) return KVQ_EALIGN;
    }
  }
  if (g.ragged) {
    if (!c->seq_prompt) return KVQ_EINVAL;
    if (!aligned16(c->seq_prompt)) return KVQ_EALIGN;
  }
  if (c->n_quant < 0 || c->n_resid < 0 || c->n_sink < 0 || c->ring_head < 0) return KVQ_EINVAL;
  return KVQ_OK;
}

// The host counters the library maintains must describe a state it can
// reach (a corrupted struct must not steer a kernel past the buffers): every
// call but prefill, which resets them, checks them first.
static int check_counters(const Geometry &g, const kvq_cache *c) {
  if (c->n_quant > g.cap || c->n_resid > g.residual || c->n_sink > g.n_sink) return KVQ_EINVAL;
  if (c->n_quant + c->n_resid + c->n_sink > g.max_ctx) return KVQ_EINVAL;
  if (c->n_appended < 0 || c->n_appended > c->n_quant + c->n_resid + c->n_sink) return KVQ_EINVAL;
  if (g.scheme == KVQ_KIVI && (c->n_resid >= g.residual || c->n_quant % g.residual != 0))
    return KVQ_EINVAL;
  if (g.scheme == KVQ_INNERQ && g.residual > 0 && c->ring_head >= g.residual) return KVQ_EINVAL;
  if (g.scheme == KVQ_INNERQ && g.residual == 0 && c->ring_head != 0) return KVQ_EINVAL;
  return KVQ_OK;
}

static int check_state(const Geometry &g, const kvq_cache *c) {
  const int r = check_cache(g, c);
  return r != KVQ_OK ? r : check_counters(g, c);
}

static int from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA; }

int check_decode_call(const Geometry &g, const kvq_cache *cache, const uint16_t *q,
                      const float *out, float softmax_scale, const void *ws, size_t ws_bytes) {
  int r;
  if ((r = check_state(g, cache)) != KVQ_OK) return r;
  if (!q || !out || !ws) return KVQ_EINVAL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(ws)) return KVQ_EALIGN;
  if (ws_bytes < decode_workspace_bytes(g)) return KVQ_ECAPACITY;
  if (!(softmax_scale == softmax_scale)) return KVQ_EINVAL;
  return KVQ_OK;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

int kvq_cache_sizes(const kvq_config *cfg, kvq_sizes *out) {
  if (!out) return KVQ_EINVAL;
  Geometry g;
  const int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  memset(out, 0, sizeof(*out));
  const size_t BH = (size_t)g.B * g.H;
  out->blocks = BH * (size_t)(g.cap / kBlockTokens) * g.block_bytes +
                (g.knorm ? BH * (size_t)g.d * sizeof(float) : 0);
  if (g.scheme == KVQ_KIVI && g.k_group > kBlockTokens)
    out->k_meta = BH * (size_t)g.k_meta_rows * 2 * g.d * g.msz + kMetaPad;
  if (g.scheme == KVQ_INNERQ) out->k_mode = out->v_mode = BH * (size_t)g.mode_words * 4;
  out->k_res = out->v_res = BH * (size_t)g.residual * g.d * 2;
  out->k_sink = out->v_sink = BH * (size_t)g.n_sink * g.d * 2;
  out->status = sizeof(int32_t);
  out->seq_prompt = g.ragged ? (size_t)g.B * sizeof(int32_t) : 0;
  return KVQ_OK;
}

int kvq_workspace_bytes(const kvq_config *cfg, size_t *bytes) {
  if (!bytes) return KVQ_EINVAL;
  Geometry g;
  const int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  *bytes = decode_workspace_bytes(g);
  return KVQ_OK;
}

// Both prefills.  lens (host, ragged only) null: every sequence has T tokens.
static int prefill(const kvq_config *cfg, kvq_cache *cache, const uint16_t *K, const uint16_t *V,
                   int64_t T, const int32_t *lens, bool ragged_call, void *stream) {
  Geometry g;
  int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  if (ragged_call && (!g.ragged || !lens)) return KVQ_EINVAL;
  if ((r = check_cache(g, cache)) != KVQ_OK) return r;  // counters: reset below
  if (T < 0) return KVQ_EINVAL;
  if (T > 0 && (!K || !V)) return KVQ_EINVAL;
  if (T > 0 && (!aligned16(K) || !aligned16(V))) return KVQ_EALIGN;
  if (T > g.max_ctx) return KVQ_ECAPACITY;
  int64_t longest = T;
  if (lens) {
    longest = 0;
    for (int b = 0; b < g.B; ++b) {
      if (lens[b] < 0 || lens[b] > T) return KVQ_EINVAL;
      if (lens[b] > longest) longest = lens[b];
    }
  }
  const Counts c = counts_of(g, longest, 0);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CachePtrs p = ptrs_of(g, cache);
  p.appended = 0;
  int launches = 0;
  if (g.ragged) {
    // every sequence's prompt length, read by the kernels below and by every
    // later call
    if (lens)
      r = from_cuda(cudaMemcpyAsync(cache->seq_prompt, lens, (size_t)g.B * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, st));
    else
      r = from_cuda(launch_fill_i32(cache->seq_prompt, g.B, (int32_t)T, st)), ++launches;
    if (r != KVQ_OK) return r;
  }
  int n = 0;
  r = from_cuda(launch_prefill(g, p, reinterpret_cast<const __half *>(K),
                               reinterpret_cast<const __half *>(V), T, c, st, &n));
  if (r != KVQ_OK) return r;
  cache->n_quant = c.n_quant;
  cache->n_resid = c.n_resid;
  cache->n_sink = c.n_sink;
  cache->ring_head = 0;
  cache->n_appended = 0;
  note_launch(launches + n);
  return KVQ_OK;
}

int kvq_quantize_prefill(const kvq_config *cfg, kvq_cache *cache, const uint16_t *K,
                         const uint16_t *V, int64_t T, void *stream) {
  return prefill(cfg, cache, K, V, T, nullptr, false, stream);
}

int kvq_quantize_prefill_ragged(const kvq_config *cfg, kvq_cache *cache, const uint16_t *K,
                                const uint16_t *V, int64_t T_max, const int32_t *lens,
                                void *stream) {
  return prefill(cfg, cache, K, V, T_max, lens, true, stream);
}

int kvq_append(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k, const uint16_t *v,
               void *stream) {
  Geometry g;
  int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  if ((r = check_state(g, cache)) != KVQ_OK) return r;
  if (!k || !v) return KVQ_EINVAL;
  if (!aligned16(k) || !aligned16(v)) return KVQ_EALIGN;
  if (cache->n_quant + cache->n_resid + cache->n_sink + 1 > g.max_ctx) return KVQ_ECAPACITY;
  if (g.scheme == KVQ_KIVI && cache->n_resid >= g.residual) return KVQ_EINVAL;
  if (g.scheme == KVQ_INNERQ && g.residual > 0 && cache->ring_head >= g.residual) return KVQ_EINVAL;
  r = from_cuda(launch_append(g, ptrs_of(g, cache), reinterpret_cast<const __half *>(k),
                              reinterpret_cast<const __half *>(v), host_counts(g, cache),
                              static_cast<cudaStream_t>(stream)));
  if (r != KVQ_OK) return r;
  cache->n_appended += 1;
  if (g.scheme == KVQ_KIVI) {
    if (cache->n_resid + 1 == g.residual) {
      cache->n_quant += g.residual;
      cache->n_resid = 0;
    } else {
      cache->n_resid += 1;
    }
  } else if (cache->n_sink < g.n_sink) {
    cache->n_sink += 1;
  } else if (cache->n_resid < g.residual) {
    cache->n_resid += 1;
  } else {
    cache->n_quant += 1;
    if (g.residual > 0) cache->ring_head = (cache->ring_head + 1) % g.residual;
  }
  note_launch(1);
  return KVQ_OK;
}

int kvq_decode_attention(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                         float *out, float softmax_scale, void *ws, size_t ws_bytes,
                         void *stream) {
  Geometry g;
  int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  if ((r = check_decode_call(g, cache, q, out, softmax_scale, ws, ws_bytes)) != KVQ_OK) return r;
  const Counts c = host_counts(g, cache);
  const DecodePlan plan = plan_decode(g, c.n_quant, g.ragged ? (int64_t)g.residual + g.n_sink
                                                             : c.n_resid + c.n_sink,
                                      num_sms_cached());
  r = from_cuda(launch_decode(g, ptrs_of(g, cache), plan, c, reinterpret_cast<const __half *>(q),
                              out, softmax_scale, ws, num_sms_cached(),
                              static_cast<cudaStream_t>(stream)));
  if (r != KVQ_OK) return r;
  note_launch(1);
  return KVQ_OK;
}

int kvq_decode_attention_rope(const kvq_config *cfg, const kvq_cache *cache, const uint16_t *q,
                              float *out, float softmax_scale, double rope_base, void *ws,
                              size_t ws_bytes, void *stream) {
  Geometry g;
  int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  if ((r = check_state(g, cache)) != KVQ_OK) return r;
  if (!q || !out || !ws) return KVQ_EINVAL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(ws)) return KVQ_EALIGN;
  if (ws_bytes < decode_workspace_bytes(g)) return KVQ_ECAPACITY;
  if (!(softmax_scale == softmax_scale)) return KVQ_EINVAL;
  if (!(rope_base > 0.0) || !isfinite(rope_base)) return KVQ_EINVAL;
  if (!rope_group_supported(g.Hq / g.H) || g.max_ctx > kRopeMaxPositions) return KVQ_EUNSUPPORTED;
  if (g.meta16 || g.vq || g.n_out || g.ragged) return KVQ_EUNSUPPORTED;
  if (cache->n_quant > 0 && tc_rope_supported(g))
    r = from_cuda(launch_decode_tc_rope(g, ptrs_of(g, cache), cache->n_quant, cache->n_resid,
                                        reinterpret_cast<const __half *>(q), out, softmax_scale,
                                        rope_base, ws, num_sms_cached(),
                                        static_cast<cudaStream_t>(stream)));
  else
    r = from_cuda(launch_decode_rope(g, ptrs_of(g, cache), cache->n_quant, cache->n_resid,
                                     cache->n_sink, cache->ring_head,
                                     reinterpret_cast<const __half *>(q), out, softmax_scale,
                                     rope_base, ws, num_sms_cached(),
                                     static_cast<cudaStream_t>(stream)));
  if (r != KVQ_OK) return r;
  note_launch(1);
  return KVQ_OK;
}

int kvq_append_decode(const kvq_config *cfg, kvq_cache *cache, const uint16_t *k,
                      const uint16_t *v, const uint16_t *q, float *out, float softmax_scale,
                      void *ws, size_t ws_bytes, void *stream) {
  Geometry g;
  int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  if ((r = check_state(g, cache)) != KVQ_OK) return r;
  if (!k || !v || !q || !out || !ws) return KVQ_EINVAL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out) || !aligned16(ws))
    return KVQ_EALIGN;
  if (cache->n_quant + cache->n_resid + cache->n_sink + 1 > g.max_ctx) return KVQ_ECAPACITY;
  if (ws_bytes < decode_workspace_bytes(g)) return KVQ_ECAPACITY;
  if (!(softmax_scale == softmax_scale)) return KVQ_EINVAL;
  // One launch when the append only stores the new token (KIVI, no flush)
  // and the decode runs on the tensor-core path; two launches otherwise.
  // (not under the value queue, whose append may quantize a value, nor with
  // per-sequence lengths, whose residual slots differ between sequences)
  const bool fuse = g.scheme == KVQ_KIVI && cache->n_resid + 1 < g.residual &&
                    cache->n_quant > 0 && !g.vq && !g.ragged && tc_decode_supported(g);
  if (!fuse) {
    if ((r = kvq_append(cfg, cache, k, v, stream)) != KVQ_OK) return r;
    if ((r = kvq_decode_attention(cfg, cache, q, out, softmax_scale, ws, ws_bytes, stream)) !=
        KVQ_OK)
      return r;
    note_launch(2);
    return KVQ_OK;
  }
  r = from_cuda(launch_decode_tc(g, ptrs_of(g, cache), cache->n_quant, cache->n_resid + 1,
                                 cache->n_sink, reinterpret_cast<const __half *>(q), out,
                                 softmax_scale, ws, num_sms_cached(),
                                 static_cast<cudaStream_t>(stream),
                                 reinterpret_cast<const __half *>(k),
                                 reinterpret_cast<const __half *>(v)));
  if (r != KVQ_OK) return r;
  cache->n_resid += 1;
  cache->n_appended += 1;
  note_launch(1);
  return KVQ_OK;
}

int kvq_decode_step_host(const kvq_config *cfg, kvq_cache *cache, const uint16_t *h_in,
                         float *h_out, uint16_t *d_in, float *d_out, float softmax_scale,
                         void *ws, size_t ws_bytes, void *stream) {
  Geometry g;
  int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  if (!h_in || !h_out || !d_in || !d_out) return KVQ_EINVAL;
  if ((r = check_state(g, cache)) != KVQ_OK) return r;
  if (!aligned16(d_in) || !aligned16(d_out)) return KVQ_EALIGN;
  if (cache->n_quant + cache->n_resid + cache->n_sink + 1 > g.max_ctx) return KVQ_ECAPACITY;
  if (ws_bytes < decode_workspace_bytes(g)) return KVQ_ECAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // [k | v | q]: each part is a multiple of 8 halves (d is), so every part
  // of the device staging buffer stays 16-byte aligned
  const size_t kv = (size_t)g.B * g.H * g.d, qn = (size_t)g.B * g.Hq * g.d;
  const size_t in_bytes = (2 * kv + qn) * 2, o_bytes = qn * 4;
  if (cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return KVQ_ECUDA;
  if ((r = kvq_append_decode(cfg, cache, d_in, d_in + kv, d_in + 2 * kv, d_out, softmax_scale, ws,
                             ws_bytes, stream)) != KVQ_OK)
    return r;
  const int launches = kvq_last_launch_count();
  if (cudaMemcpyAsync(h_out, d_out, o_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return KVQ_ECUDA;
  note_launch(launches);
  return KVQ_OK;
}

int kvq_get_device_status(kvq_cache *cache, void *stream) {
  if (!cache || !cache->dev_status) return KVQ_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ECUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, cache->dev_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVQ_ECUDA;
  if (v != 0) {
    const int32_t zero = 0;
    if (cudaMemcpy(cache->dev_status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return KVQ_ECUDA;
  }
  return v == 0 ? KVQ_OK : (int)v;
}

int kvq_last_launch_count(void) { return t_last_launches; }

int kvq_decode_kernel_name(const kvq_config *cfg, int64_t n_quant, char *buf, size_t len) {
  if (!buf || len == 0 || n_quant < 0) return KVQ_EINVAL;
  Geometry g;
  const int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  int n;
  if (n_quant > 0 && tc_decode_supported(g))
    n = tc_variant_name(g, buf, len);
  else if (n_quant > 0 && gqa_decode_supported(g))
    n = gqa_variant_name(g, buf, len);
  else
    n = snprintf(buf, len, "decode_kernel<d=%d,bits=%d,rg=%d,scheme=%s>", g.d, g.bits, g.Hq / g.H,
                 g.scheme == KVQ_KIVI ? "kivi" : "innerq");
  return (n < 0 || (size_t)n >= len) ? KVQ_EINVAL : KVQ_OK;
}

int kvq_rope_kernel_name(const kvq_config *cfg, int64_t n_quant, char *buf, size_t len) {
  if (!buf || len == 0 || n_quant < 0) return KVQ_EINVAL;
  Geometry g;
  const int r = resolve(cfg, &g);
  if (r != KVQ_OK) return r;
  int n;
  if (n_quant > 0 && tc_rope_supported(g))
    n = tc_rope_variant_name(g, buf, len);
  else
    n = snprintf(buf, len, "rope_decode_kernel<d=%d,bits=%d,rg=%d,scheme=%s>", g.d, g.bits,
                 g.Hq / g.H, g.scheme == KVQ_KIVI ? "kivi" : "innerq");
  return (n < 0 || (size_t)n >= len) ? KVQ_EINVAL : KVQ_OK;
}

void kvq_debug_stall_waits(int64_t iterations) {
  set_debug_stall(iterations < 0 ? 0 : (long long)iterations);
}

const char *kvq_strerror(int code) {
  switch (code) {
    case KVQ_OK: return "ok";
    case KVQ_EINVAL: return "invalid argument";
    case KVQ_EUNSUPPORTED: return "unsupported configuration";
    case KVQ_ECAPACITY: return "capacity exceeded (max_ctx or workspace)";
    case KVQ_EALIGN: return "device buffer not 16-byte aligned";
    case KVQ_ECUDA: return "CUDA error";
    case KVQ_ETIMEOUT: return "device-side wait timed out";
  }
  return "unknown error";
}

}  // extern "C"
