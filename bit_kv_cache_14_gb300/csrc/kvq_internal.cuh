// Internal declarations shared by the libkvq translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kMaxHeadDim = 128;
constexpr int kMaxResidual = 1024;
constexpr int kCapAlign = 128;     // token-stride granularity of the cache layout
constexpr int kMetaPad = 64;       // slack bytes after the KIVI key-statistics buffer
constexpr int kBlockTokens = 32;   // tokens per block of the quantized region

// Geometry of one cache, resolved on the host from kvq_config and copied by
// value into every kernel.
struct Geometry {
  int B, H, Hq, d, bits, scheme, k_group, v_group, residual, n_sink;
  int64_t max_ctx;
  int64_t cap;        // per-head token capacity: max_ctx rounded up to kCapAlign
  int row_bytes;      // packed bytes per token row: d * bits / 8
  int k_meta_cols;    // KIVI: d; InnerQ: d / k_group
  int v_meta_cols;    // d / v_group
  int64_t k_meta_rows;  // KIVI: cap / G key groups per head; InnerQ: cap
  int64_t mode_words;   // per head, InnerQ only
  int block_bytes;      // one 32-token block
  int blk_vc, blk_vs, blk_vz, blk_ks, blk_kz;  // byte offsets inside a block
  int blk_ko, blk_vo;   // outlier lists (KIVI with n_out > 0)
  int knorm;            // InnerQ key normalization (KVQ_INNERQ_KNORM)
  int64_t knorm_off;    // byte offset of the key factors f32 [B][H][d] in blocks
  int meta16;           // scales and zeros stored in fp16 (KVQ_META_F16)
  int msz;              // bytes per stored scale / zero: 4 or 2
  int vq;               // KIVI value queue (KVQ_VALUE_QUEUE)
  int n_out;            // KIVI outliers per token and tensor (0 = none)
  int ragged;           // per-sequence prompt lengths (KVQ_RAGGED)
};

// Device pointers of a cache (same meaning as kvq_cache).
struct CachePtrs {
  uint8_t *blocks;
  uint8_t *k_meta;
  uint32_t *k_mode, *v_mode;
  __half *k_res, *v_res, *k_sink, *v_sink;
  int32_t *status;
  float *k_norm;  // key factors [B*H][d] (KVQ_INNERQ_KNORM), else nullptr
  const int32_t *seq_prompt;  // KVQ_RAGGED: prompt length per sequence, else nullptr
  int64_t appended;           // tokens appended to every sequence since the prefill
};

// Counters of one sequence (the kvq_cache counters, plus the number of
// values held quantized: n_quant, or under the value queue its own count).
struct Counts {
  int64_t n_quant, n_resid, n_sink, ring_head, n_vq;
};

// The counters of a sequence that received `prompt` tokens at prefill and
// `appended` single appends since: every counter is a function of those two
// (KIVI residual = length mod R; InnerQ sinks, then window, then quantized,
// with one ring step per eviction; value queue max(0, n - R + 1)).
__host__ __device__ inline Counts counts_of(const Geometry &g, int64_t prompt, int64_t appended) {
  Counts c;
  const int64_t n = prompt + appended;
  if (g.scheme == KVQ_KIVI) {
    c.n_resid = n % g.residual;
    c.n_quant = n - c.n_resid;
    c.n_sink = 0;
    c.ring_head = 0;
    c.n_vq = g.vq ? (n >= g.residual ? n - g.residual + 1 : 0) : c.n_quant;
  } else {
    c.n_sink = n < g.n_sink ? n : g.n_sink;
    const int64_t rest = n - c.n_sink;
    c.n_resid = rest < g.residual ? rest : g.residual;
    c.n_quant = rest - c.n_resid;
    const int64_t ps = prompt < g.n_sink ? prompt : g.n_sink, prest = prompt - ps;
    const int64_t pq = prest - (prest < g.residual ? prest : g.residual);
    c.ring_head = g.residual > 0 ? (c.n_quant - pq) % g.residual : 0;
    c.n_vq = c.n_quant;
  }
  return c;
}

// Counters of sequence b: the uniform ones, or (KVQ_RAGGED) its own.
__device__ __forceinline__ Counts seq_counts(const Geometry &g, const CachePtrs &p,
                                             const Counts &uniform, int b) {
  return g.ragged ? counts_of(g, p.seq_prompt[b], p.appended) : uniform;
}

// ---- addressing of the block layout (include/kvq.h, "Packed layout") ------
__host__ __device__ __forceinline__ int64_t block_index(const Geometry &g, int64_t bh,
                                                        int64_t t) {
  return bh * (g.cap / kBlockTokens) + t / kBlockTokens;
}
__device__ __forceinline__ uint8_t *tok_block(const Geometry &g, const CachePtrs &p, int64_t bh,
                                              int64_t t) {
  return p.blocks + block_index(g, bh, t) * g.block_bytes;
}
// Packed code row of token t (off = 0 for keys, g.blk_vc for values).
__device__ __forceinline__ uint8_t *code_row(const Geometry &g, const CachePtrs &p, int64_t bh,
                                             int64_t t, int off) {
  return tok_block(g, p, bh, t) + off + (int)(t % kBlockTokens) * g.row_bytes;
}
// Per-token statistics row of token t: `cols` stored values at block offset `off`.
__device__ __forceinline__ uint8_t *tok_meta(const Geometry &g, const CachePtrs &p, int64_t bh,
                                             int64_t t, int off, int cols) {
  return tok_block(g, p, bh, t) + off + (int)(t % kBlockTokens) * cols * g.msz;
}
// KIVI key group grp of head bh: scale row (d stored values); the zero row
// follows at + d * msz bytes.  G <= 32: at the end of the group's block;
// G >= 64: in the k_meta array.
__device__ __forceinline__ uint8_t *kivi_key_meta(const Geometry &g, const CachePtrs &p,
                                                  int64_t bh, int64_t grp) {
  if (g.k_group <= kBlockTokens) {
    const int64_t t0 = grp * g.k_group;
    return tok_block(g, p, bh, t0) + g.blk_ks +
           (int)((t0 % kBlockTokens) / g.k_group) * 2 * g.d * g.msz;
  }
  return p.k_meta + (bh * g.k_meta_rows + grp) * 2 * g.d * g.msz;
}
// Outlier list of token t (off = g.blk_ko for keys, g.blk_vo for values):
// n_out words (channel << 16) | fp16 bits, channels ascending.
__device__ __forceinline__ uint32_t *tok_outliers(const Geometry &g, const CachePtrs &p,
                                                  int64_t bh, int64_t t, int off) {
  return reinterpret_cast<uint32_t *>(tok_block(g, p, bh, t) + off) +
         (int)(t % kBlockTokens) * g.n_out;
}

// A stored statistic as fp32, and its store (under KVQ_META_F16 the value is
// already an fp16 value, so the conversion is exact).
__device__ __forceinline__ float ld_meta(const Geometry &g, const uint8_t *row, int i) {
  return g.meta16 ? __half2float(reinterpret_cast<const __half *>(row)[i])
                  : reinterpret_cast<const float *>(row)[i];
}
__device__ __forceinline__ void st_meta(const Geometry &g, uint8_t *row, int i, float v) {
  if (g.meta16)
    reinterpret_cast<__half *>(row)[i] = __float2half_rn(v);
  else
    reinterpret_cast<float *>(row)[i] = v;
}

int resolve(const kvq_config *cfg, Geometry *g);

// ---- per-device launch set-up ----------------------------------------------
// Function attributes and occupancy belong to a device: every cache below is
// indexed by the current device (0 .. kMaxDevices - 1).
constexpr int kMaxDevices = 64;
// The current device, or -1 when there is none or its ordinal is too large.
int device_slot();

// Launch set-up of one kernel: the dynamic shared memory its attribute allows
// and its resident blocks per SM at that size, per device, filled on first use
// with the device current.  The fast path is two relaxed loads; the first use
// (per device and size) takes a lock.
struct KernelSetup {
  std::atomic<int> smem[kMaxDevices];  // bytes the attribute allows (0: not set)
  std::atomic<int> occ[kMaxDevices];   // blocks per SM at occ_smem
  std::atomic<int> occ_smem[kMaxDevices];
  std::mutex mu;
};

// Makes `kern` launchable with smem_bytes of dynamic shared memory and
// `threads` threads on the current device; *occ (if given) receives its
// resident blocks per SM there.
template <typename F>
cudaError_t kernel_setup(KernelSetup &s, F kern, int threads, int smem_bytes, int *occ) {
  const int dev = device_slot();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (s.smem[dev].load(std::memory_order_acquire) >= smem_bytes &&
      (!occ || s.occ_smem[dev].load(std::memory_order_acquire) == smem_bytes)) {
    if (occ) *occ = s.occ[dev].load(std::memory_order_relaxed);
    return cudaSuccess;
  }
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.smem[dev].load(std::memory_order_relaxed) < smem_bytes) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    s.smem[dev].store(smem_bytes, std::memory_order_release);
  }
  if (occ) {
    if (s.occ_smem[dev].load(std::memory_order_relaxed) != smem_bytes) {
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem_bytes);
      if (e != cudaSuccess) return e;
      s.occ[dev].store(n > 0 ? n : 1, std::memory_order_relaxed);
      s.occ_smem[dev].store(smem_bytes, std::memory_order_release);
    }
    *occ = s.occ[dev].load(std::memory_order_relaxed);
  }
  return cudaSuccess;
}

// Launch of a persistent grid whose blocks wait on one another (the
// tensor-core decode merges): cooperative, so the launch fails unless every
// block can be resident at once, instead of leaving a poll to time out.
template <typename... P, typename... A>
cudaError_t launch_cooperative(void (*kern)(P...), unsigned grid, unsigned threads, int smem,
                               cudaStream_t st, A &&...args) {
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3(grid);
  c.blockDim = dim3(threads);
  c.dynamicSmemBytes = (size_t)smem;
  c.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  // programmatic dependent launch: the kernel may start while the previous
  // grid on the stream drains; it waits for it (griddepcontrol.wait) before
  // its first access to global memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  c.attrs = attr;
  c.numAttrs = 2;
  return cudaLaunchKernelEx(&c, kern, static_cast<A &&>(args)...);
}
CachePtrs ptrs_of(const Geometry &g, const kvq_cache *c);
// Every check kvq_decode_attention makes before it enqueues anything (cache
// buffers and counters, pointers, alignment, workspace size, scale); KVQ_OK
// or the error it would return.
int check_decode_call(const Geometry &g, const kvq_cache *cache, const uint16_t *q,
                      const float *out, float softmax_scale, const void *ws, size_t ws_bytes);
void note_launch(int n);

// ---- launchers (return cudaError_t of the launch) ------------------------
// Prefill of K, V [B][H][T][d] (T = the row stride; under KVQ_RAGGED each
// sequence's own prompt length is read from p.seq_prompt) into an empty
// cache; c = the counters after it (the longest sequence's when ragged).
cudaError_t launch_prefill(const Geometry &g, const CachePtrs &p, const __half *K,
                           const __half *V, int64_t T, const Counts &c, cudaStream_t st,
                           int *launches);
// One appended token per (batch, kv head); c = the counters before it.
cudaError_t launch_append(const Geometry &g, const CachePtrs &p, const __half *k,
                          const __half *v, const Counts &c, cudaStream_t st);
// dst[0 .. n) = v.
cudaError_t launch_fill_i32(int32_t *dst, int n, int32_t v, cudaStream_t st);

// Partial (m, l, o) slots per head in the decode workspace: enough for one
// per 128 quantized tokens plus the fp16 segment.
inline int part_slots(const Geometry &g) { return (int)(g.cap / kCapAlign) + 2; }

// Partial slots per head of the tensor-core decode kernels, a bound for both
// splits.  The grouped-query kernel cuts each head into 128-token units plus
// fp16 units and leaves one partial per warp (8 per block) for every block
// that touches a head; the MHA kernel gives every warp an equal range of
// 32-token tiles, fp16 chunks (tc_fp16_chunk tokens, two units each) and two
// empty units per head, one partial per warp touching the head, i.e. at most
// cap/32 + 2 * chunks + 3 per head (each warp holds at least one unit), which
// 8 * (cap/128 + chunks + 2) covers.  At most kTcMaxBlocks blocks.
constexpr int kTcWarps = 8;
constexpr int kTcMaxBlocks = 1024;
inline int tc_fp16_chunk(const Geometry &g) {
  const int kmb = (g.scheme == KVQ_KIVI && g.k_group > kBlockTokens) ? 2 * g.d * g.msz : 0;
  const int ch = (g.block_bytes + kmb) / (4 * g.d);
  return ch < 8 ? ch : 8;
}
inline int tc_part_slots(const Geometry &g) {
  const int ch = tc_fp16_chunk(g) > 0 ? tc_fp16_chunk(g) : 1;
  int64_t u = g.cap / kCapAlign + (g.residual + g.n_sink + ch - 1) / ch + 1;
  if (u > kTcMaxBlocks + 1) u = kTcMaxBlocks + 1;
  return (int)(kTcWarps * (u + 1));
}

struct DecodePlan {
  int n_qsplit;        // splits over the quantized region
  int n_split;         // n_qsplit + (fp16 segment present ? 1 : 0)
  int64_t chunk;       // quantized tokens per split
};
size_t decode_workspace_bytes(const Geometry &g);
DecodePlan plan_decode(const Geometry &g, int64_t n_quant, int64_t n_fp16, int num_sms);
cudaError_t launch_decode(const Geometry &g, const CachePtrs &p, const DecodePlan &plan,
                          const Counts &c, const __half *q, float *out, float scale, void *ws,
                          int num_sms, cudaStream_t st);

// Tensor-core decode path (MHA, head_dim 128, 2 or 4 value groups).
bool tc_decode_supported(const Geometry &g);
// k_new, v_new non-null: fused append -- the last of the n_resid residual
// rows is the step's new token, read from k_new / v_new ([B][H][d]) and
// stored into the residual by the kernel.
cudaError_t launch_decode_tc(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                             int64_t n_resid, int64_t n_sink, const __half *q, float *out,
                             float scale, void *ws, int num_sms, cudaStream_t st,
                             const __half *k_new = nullptr, const __half *v_new = nullptr);
void set_debug_stall(long long iterations);

// Name of the kernel instantiation each tensor-core path launches for g
// (snprintf semantics).
int tc_variant_name(const Geometry &g, char *buf, size_t len);
int gqa_variant_name(const Geometry &g, char *buf, size_t len);

// Tensor-core grouped-query path (head_dim 128, 2 or 4 query heads per KV
// head, 2 or 4 value groups; 2- or 4-bit KIVI with G >= 32, or InnerQ with
// key channel groups of 32 or 64; statistics in fp32 or fp16).
bool gqa_decode_supported(const Geometry &g);
cudaError_t launch_decode_gqa(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                              int64_t n_resid, int64_t n_sink, const __half *q, float *out,
                              float scale, void *ws, int num_sms, cudaStream_t st);

// ---- quantization arithmetic (bit-exact contract with the formula) -------
// Asymmetric: scale = (max - min) / (2^b - 1), zero = min,
// code = clamp(rint((x - min) / scale), 0, 2^b - 1); constant group: 0, 0.
__device__ __forceinline__ float canon_zero(float x) { return __fadd_rn(x, 0.0f); }

__device__ __forceinline__ float asym_scale(float mn, float mx, int bits) {
  return mx == mn ? 0.0f : __fdiv_rn(__fsub_rn(mx, mn), (float)((1 << bits) - 1));
}

__device__ __forceinline__ uint32_t asym_code(float x, float mn, float scale, int bits) {
  if (scale == 0.0f) return 0u;
  float r = rintf(__fdiv_rn(__fsub_rn(x, mn), scale));
  const float top = (float)((1 << bits) - 1);
  r = fminf(fmaxf(r, 0.0f), top);
  return (uint32_t)r;
}

// Symmetric: scale = max(|min|, |max|) / (2^(b-1) - 1),
// code = clamp(rint(x / scale), -lim, lim) + 2^(b-1), zero = -2^(b-1) * scale.
__device__ __forceinline__ float sym_scale(float mn, float mx, int bits) {
  return __fdiv_rn(fmaxf(fabsf(mn), fabsf(mx)), (float)((1 << (bits - 1)) - 1));
}

__device__ __forceinline__ uint32_t sym_code(float x, float scale, int bits) {
  const int half = 1 << (bits - 1);
  const float lim = (float)(half - 1);
  float r = rintf(__fdiv_rn(x, scale));
  r = fminf(fmaxf(r, -lim), lim);
  return (uint32_t)((int)r + half);
}

// The same codes with one reciprocal per group instead of one division per
// element, and bit for bit the same: with inv the hardware reciprocal of the
// scale (rcp.approx: at most 1 ulp, a relative error below 2^-23), the
// product rn(d * inv) differs from the IEEE quotient rn(d / scale) by less
// than 2^-21 of its magnitude, under 2^-15 while |d / scale| < 64, so rint
// gives the same integer for both unless the product lies within kTieGuard
// (2^-12) of a half-integer; there -- and for a quotient out of that range --
// the IEEE division decides.
constexpr float kTieGuard = 1.0f / 4096.0f;
__device__ __forceinline__ float rint_quotient(float d, float scale, float inv) {
  const float r = __fmul_rn(d, inv);
  const float f = __fsub_rn(r, floorf(r));
  if (!(fabsf(r) < 64.0f) || fabsf(__fsub_rn(f, 0.5f)) < kTieGuard)
    return rintf(__fdiv_rn(d, scale));
  return rintf(r);
}
__device__ __forceinline__ uint32_t asym_code_inv(float x, float mn, float scale, float inv,
                                                  int bits) {
  if (scale == 0.0f) return 0u;
  float r = rint_quotient(__fsub_rn(x, mn), scale, inv);
  r = fminf(fmaxf(r, 0.0f), (float)((1 << bits) - 1));
  return (uint32_t)r;
}
// Symmetric (a scale of 0, possible only for fp16 statistics, gives q = 0).
__device__ __forceinline__ uint32_t sym_code_inv(float x, float scale, float inv, int bits) {
  const int half = 1 << (bits - 1);
  if (scale == 0.0f) return (uint32_t)half;
  const float lim = (float)(half - 1);
  float r = rint_quotient(x, scale, inv);
  r = fminf(fmaxf(r, -lim), lim);
  return (uint32_t)((int)r + half);
}
// The reciprocal of a scale for the products above (the hardware
// approximation; scales are normal numbers), 0 for a zero scale (then no
// code uses it).
__device__ __forceinline__ float recip_or_zero(float scale) {
  if (scale == 0.0f) return 0.0f;
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(scale));
  return r;
}

// InnerQ mode rule: symmetric iff not constant and |max + min| <= (max - min)/(2^b - 1).
__device__ __forceinline__ bool choose_symmetric(float mn, float mx, int bits) {
  if (mx == mn) return false;
  const float step = __fdiv_rn(__fsub_rn(mx, mn), (float)((1 << bits) - 1));
  return fabsf(__fadd_rn(mx, mn)) <= step;
}

}  // namespace kvq
