// Prefill quantize+pack and append/flush kernels.
//
// Method: keys per channel over G-token groups, values per token over channel
// groups ("大模型量化技术原理：KIVI、IntactKV、KVQuant", KIVI / 工作原理); residual
// flushed in one batch when it holds R tokens (pgsm.cn how-to §3.1); InnerQ
// per-token groups along the head dimension with a per-group symmetric /
// asymmetric choice, fp16 sinks and recent window (InnerQ page, 方法论 1-4).
// Options: statistics stored in fp16 (codes taken with the stored values);
// KIVI's value queue (the same page, KIVI / 工作原理, value paragraph: a value
// is quantized when R newer ones wait behind it); dense-and-sparse outliers
// (the same page, KVQuant / 技术原理 四: each token's largest elements kept in
// fp16, the group statistics taken over the rest); per-sequence lengths.
//
// Work mapping: one thread owns 8 consecutive channels of one token (one
// 16-byte fp16 load, 2 or 4 packed output bytes), so a warp reads whole
// 256-byte token rows and writes whole packed rows, and the d/8 lanes of a
// row are consecutive lanes of one warp.  Per-token group min/max is a
// butterfly over the lanes of the group; a token's outliers are k rounds of a
// max over its row's lanes; per-channel key statistics combine 16-byte row
// loads over the row lanes in shared memory.
#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kQuantBlock = 256;

__device__ __forceinline__ void load8(const __half *p, float (&x)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4 *>(p);
  const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Store the packed codes of one 8-channel chunk: 2 bytes (2-bit) or 4 (4-bit).
__device__ __forceinline__ void store_chunk(uint8_t *row, int chunk, uint32_t w, int bits) {
  if (bits == 2)
    reinterpret_cast<uint16_t *>(row)[chunk] = (uint16_t)w;
  else
    reinterpret_cast<uint32_t *>(row)[chunk] = w;
}

// ---- statistics of one group (the formula; fp16 storage option) -----------
__device__ __forceinline__ float rn16(float x) { return __half2float(__float2half_rn(x)); }

struct Stats {
  float scale, zero;
};

// Asymmetric: scale = (max - min) / (2^b - 1), zero = min; with fp16 storage
// both are rounded to fp16 once (a constant group keeps scale 0) and the codes
// use the rounded values.
__device__ __forceinline__ Stats asym_stats(float mn, float mx, int bits, bool f16) {
  if (!f16) return Stats{asym_scale(mn, mx, bits), mn};
  const float s = mx == mn ? 0.0f : rn16(__fdiv_rn(__fsub_rn(mx, mn), (float)((1 << bits) - 1)));
  return Stats{s, rn16(mn)};
}

// Symmetric: scale = max(|min|, |max|) / (2^(b-1) - 1) (fp16: rounded once),
// zero = -2^(b-1) * scale (an exact product).
__device__ __forceinline__ Stats sym_stats(float mn, float mx, int bits, bool f16) {
  float s = sym_scale(mn, mx, bits);
  if (f16) s = rn16(s);
  return Stats{s, __fmul_rn(-(float)(1 << (bits - 1)), s)};
}

// Symmetric code; a scale of 0 (an fp16 scale that rounded to zero) gives q = 0.
__device__ __forceinline__ uint32_t sym_code_z(float x, float scale, int bits) {
  return scale == 0.0f ? (uint32_t)(1 << (bits - 1)) : sym_code(x, scale, bits);
}

// ---- dense-and-sparse outliers ---------------------------------------------
// The k largest-magnitude elements of one token row held as 8-channel chunks
// by `chunks` aligned consecutive lanes (this lane holds chunk j), equal
// magnitudes going to the lower channel: k rounds of a maximum over the row's
// lanes of (|x| as fp16 bits, 255 - channel).  Every lane of the warp calls it
// (rows of other lane groups run their own rounds).  Returns the bitmask of
// this lane's 8 elements that are outliers.
__device__ __forceinline__ uint32_t outlier_mask(const float (&x)[8], int j, int chunks, int k) {
  uint32_t key[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    key[e] = ((uint32_t)__half_as_ushort(__float2half_rn(fabsf(x[e]))) << 8) |
             (uint32_t)(255 - (8 * j + e));
  uint32_t taken = 0;
  for (int r = 0; r < k; ++r) {
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (!((taken >> e) & 1u)) m = max(m, key[e]);
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, m, off);
      if (off < chunks) m = max(m, o);
    }
    const int c = 255 - (int)(m & 255u);
    if ((c >> 3) == j) taken |= 1u << (c & 7);
  }
  return taken;
}

// Writes the row's outlier list (words (channel << 16) | fp16 bits, channels
// ascending) to `list` when `valid`: each lane writes its own outliers at the
// position given by the outliers of the lanes before it.  Every lane calls it.
__device__ __forceinline__ void store_outliers(uint32_t *list, const float (&x)[8], int j,
                                               int chunks, uint32_t taken, bool valid) {
  const int cnt = __popc(taken);
  int pre = cnt;
  for (int dlt = 1; dlt < chunks; dlt <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, pre, dlt, chunks);
    if (j >= dlt) pre += y;
  }
  int pos = pre - cnt;
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if ((taken >> e) & 1u)
      list[pos++] = ((uint32_t)(8 * j + e) << 16) | (uint32_t)__half_as_ushort(__float2half_rn(x[e]));
}

// Shared scratch of key_group_per_channel: per-row-lane partial minima and
// maxima, [blockDim / (d / 8)][d] each (2048 floats for any d), and the
// outlier bitmask of every (row, chunk) of the group.
constexpr int kKeyPart = kQuantBlock * 8;
constexpr int kMaskBytes = 128 * 16;  // G <= 128 rows, d / 8 <= 16 chunks

// One key group (G tokens of src, row stride d) quantized per channel into
// token slots [t0, t0 + G), t0 a multiple of G.  All threads of the block call
// it.  A thread reads 8-channel chunks (16-byte loads) of rows r0, r0 +
// lanes, ...; the per-channel minimum and maximum are then combined over the
// row lanes (min / max are order-free, so the result is that of one pass).
// With outliers, each token's are found over its own row first, written as
// its list, and skipped by the statistics (code 0 at their positions).
__device__ void key_group_per_channel(const Geometry &g, const CachePtrs &p, int64_t bh,
                                      const __half *src, int64_t t0, float *s_scale,
                                      float *s_mn, float *s_pmn, float *s_pmx, uint8_t *s_om) {
  const int d = g.d, G = g.k_group;
  const int chunks = d / 8, lanes = blockDim.x / chunks;
  const int j = threadIdx.x % chunks, r0 = threadIdx.x / chunks;
  if (g.n_out > 0) {
    for (int base = 0; base < G; base += lanes) {
      const int i = base + r0;
      const bool valid = i < G;
      float x[8];
      if (valid) {
        load8(src + (int64_t)i * d + 8 * j, x);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.0f;
      }
      const uint32_t taken = outlier_mask(x, j, chunks, g.n_out);
      store_outliers(valid ? tok_outliers(g, p, bh, t0 + i, g.blk_ko) : nullptr, x, j, chunks,
                     taken, valid);
      if (valid) s_om[i * chunks + j] = (uint8_t)taken;
    }
    __syncthreads();
  }
  {
    float mn8[8], mx8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      mn8[k] = INFINITY;
      mx8[k] = -INFINITY;
    }
    for (int i = r0; i < G; i += lanes) {
      float x[8];
      load8(src + (int64_t)i * d + 8 * j, x);
      const uint32_t om = g.n_out > 0 ? s_om[i * chunks + j] : 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if ((om >> k) & 1u) continue;
        mn8[k] = fminf(mn8[k], x[k]);
        mx8[k] = fmaxf(mx8[k], x[k]);
      }
    }
    if (r0 < lanes) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        s_pmn[r0 * d + 8 * j + k] = mn8[k];
        s_pmx[r0 * d + 8 * j + k] = mx8[k];
      }
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float mn = s_pmn[c], mx = s_pmx[c];
    for (int r = 1; r < lanes; ++r) {
      mn = fminf(mn, s_pmn[r * d + c]);
      mx = fmaxf(mx, s_pmx[r * d + c]);
    }
    Stats st;
    if (mn > mx) {
      st = Stats{0.0f, 0.0f};  // no inlier in the group (every element an outlier)
    } else {
      st = asym_stats(canon_zero(mn), canon_zero(mx), g.bits, g.meta16);
    }
    s_scale[c] = st.scale;
    s_mn[c] = st.zero;
    uint8_t *km = kivi_key_meta(g, p, bh, t0 / G);
    st_meta(g, km, c, st.scale);
    st_meta(g, km + d * g.msz, c, st.zero);
  }
  __syncthreads();
  for (int it = threadIdx.x; it < G * chunks; it += blockDim.x) {
    const int i = it / chunks, jj = it - i * chunks;
    float x[8];
    load8(src + (int64_t)i * d + 8 * jj, x);
    const uint32_t om = g.n_out > 0 ? s_om[it] : 0u;
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = 8 * jj + k;
      if (!((om >> k) & 1u)) w |= asym_code(x[k], s_mn[c], s_scale[c], g.bits) << (k * g.bits);
    }
    store_chunk(code_row(g, p, bh, t0 + i, 0), jj, w, g.bits);
  }
  __syncthreads();
}

// One-shot per-channel key normalization ("InnerQ" summary, key
// contributions and methodology 4): keys of channel c are multiplied by
// r_c = 1 / n_c before they are quantized (fp32 division, then an fp32
// product), n_c the largest |K[t][c]| of the prompt (1 if 0).
__device__ __forceinline__ void normalize8(const float *k_norm_row, int c0, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(k_norm_row + c0)[0];
  const float4 b = reinterpret_cast<const float4 *>(k_norm_row + c0)[1];
  const float n[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = __fmul_rn(x[k], __fdiv_rn(1.0f, n[k]));
}

// Prompt length of sequence b: T, or its own under KVQ_RAGGED.
__device__ __forceinline__ int64_t prompt_len(const Geometry &g, const CachePtrs &p, int b,
                                              int64_t T) {
  return g.ragged ? (int64_t)p.seq_prompt[b] : T;
}

// Key factors, pass 1: the largest |K[t][c]| of tokens [t0, t0 + kNormTokens)
// of head blockIdx.y into n[bh][c] by an atomic max on the bit pattern
// (non-negative floats order like their bits); n starts at 0.
constexpr int kNormTokens = 4096;
__global__ void __launch_bounds__(kQuantBlock)
    key_absmax_kernel(Geometry g, CachePtrs p, const __half *K, int64_t T) {
  __shared__ unsigned int s_max[kMaxHeadDim];
  const int d = g.d;
  float *n = p.k_norm;
  const int64_t bh = blockIdx.y;
  const int64_t Tb = prompt_len(g, p, (int)(bh / g.H), T);
  const int chunks = d / 8, rows = kQuantBlock / chunks;
  const int j = threadIdx.x % chunks, r = threadIdx.x / chunks;
  for (int c = threadIdx.x; c < d; c += blockDim.x) s_max[c] = 0u;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kNormTokens;
  const int64_t t1 = min(t0 + kNormTokens, Tb);
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int64_t t = t0 + r; t < t1; t += rows) {
    float x[8];
    load8(K + (bh * T + t) * d + 8 * j, x);
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], fabsf(x[k]));
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) atomicMax(&s_max[8 * j + k], __float_as_uint(m[k]));
  __syncthreads();
  for (int c = threadIdx.x; c < d; c += blockDim.x)
    atomicMax(reinterpret_cast<unsigned int *>(n + bh * d + c), s_max[c]);
}

// Key factors, pass 2: an all-zero channel (or an empty prompt) gets 1.
__global__ void key_norm_finish_kernel(float *n, int64_t count) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    if (!(n[i] > 0.0f)) n[i] = 1.0f;
}

// Result of quantizing one 8-channel chunk inside a per-token group.
struct ChunkQ {
  uint32_t codes;
  float scale, zero;
  bool sym;
};

// Per-token group quantization of the 8 values x of this lane; the group is
// `lanes` consecutive, aligned lanes (lanes = group / 8, a power of two <= 16;
// it may differ between lanes of a warp).  Every lane of the warp must call it:
// the butterfly always runs its four full-mask rounds and each lane only
// combines the rounds inside its own group.  om: this lane's outliers (they
// take no part in the statistics and store code 0); a group left without an
// element stores scale 0 and zero 0.
__device__ __forceinline__ ChunkQ quant_chunk(const float (&x)[8], int lanes, int bits,
                                              bool allow_sym, bool f16, uint32_t om) {
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if ((om >> k) & 1u) continue;
    mn = fminf(mn, x[k]);
    mx = fmaxf(mx, x[k]);
  }
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) {
    const float omn = __shfl_xor_sync(0xffffffffu, mn, off);
    const float omx = __shfl_xor_sync(0xffffffffu, mx, off);
    if (off < lanes) {
      mn = fminf(mn, omn);
      mx = fmaxf(mx, omx);
    }
  }
  ChunkQ r;
  r.codes = 0;
  if (mn > mx) {  // no inlier in the group
    r.scale = r.zero = 0.0f;
    r.sym = false;
    return r;
  }
  mn = canon_zero(mn);
  mx = canon_zero(mx);
  r.sym = allow_sym && choose_symmetric(mn, mx, bits);
  if (r.sym) {
    const Stats st = sym_stats(mn, mx, bits, f16);
    r.scale = st.scale;
    r.zero = st.zero;
#pragma unroll
    for (int k = 0; k < 8; ++k) r.codes |= sym_code_z(x[k], r.scale, bits) << (k * bits);
  } else {
    const Stats st = asym_stats(mn, mx, bits, f16);
    r.scale = st.scale;
    r.zero = st.zero;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (!((om >> k) & 1u)) r.codes |= asym_code(x[k], r.zero, r.scale, bits) << (k * bits);
  }
  return r;
}

// Where one per-token quantization writes: block offsets of the code rows
// and of the scale / zero rows, optional mode bits.
struct TokenDst {
  int off_codes, off_scale, off_zero;
  uint32_t *mode;  // nullptr for KIVI values
  int group;       // channels per group
  int meta_cols;   // d / group
};

__device__ __forceinline__ TokenDst key_dst(const Geometry &g, const CachePtrs &p) {
  return TokenDst{0, g.blk_ks, g.blk_kz, p.k_mode, g.k_group, g.d / g.k_group};
}
__device__ __forceinline__ TokenDst value_dst(const Geometry &g, const CachePtrs &p) {
  return TokenDst{g.blk_vc, g.blk_vs, g.blk_vz, g.scheme == KVQ_INNERQ ? p.v_mode : nullptr,
                  g.v_group, g.d / g.v_group};
}

__device__ __forceinline__ void store_token(const Geometry &g, const CachePtrs &p,
                                            const TokenDst &dst, int64_t bh, int64_t t, int j,
                                            int lanes, const ChunkQ &q) {
  store_chunk(code_row(g, p, bh, t, dst.off_codes), j, q.codes, g.bits);
  if ((j & (lanes - 1)) == 0) {
    const int gi = j / lanes;
    st_meta(g, tok_meta(g, p, bh, t, dst.off_scale, dst.meta_cols), gi, q.scale);
    st_meta(g, tok_meta(g, p, bh, t, dst.off_zero, dst.meta_cols), gi, q.zero);
  }
}

// A KIVI value token held by the `chunks` lanes of its row (this lane: chunk
// j): outliers (if any) found and listed, then quantized per group into slot
// t.  Every lane of the warp calls it; `valid` guards the stores.
__device__ __forceinline__ void quant_value_token(const Geometry &g, const CachePtrs &p,
                                                  int64_t bh, int64_t t, int j, int chunks,
                                                  const float (&x)[8], bool valid) {
  const TokenDst dst = value_dst(g, p);
  uint32_t om = 0;
  if (g.n_out > 0) {
    om = outlier_mask(x, j, chunks, g.n_out);
    store_outliers(valid ? tok_outliers(g, p, bh, t, g.blk_vo) : nullptr, x, j, chunks, om,
                   valid);
  }
  const int lanes = g.v_group / 8;
  const ChunkQ q = quant_chunk(x, lanes, g.bits, false, g.meta16, om);
  if (valid) store_token(g, p, dst, bh, t, j, lanes, q);
}

// Prefill, per-token groups: the quantized tokens of every head of X
// [B*H][T][d] (InnerQ keys and values from row n_sink on; KIVI values from
// row 0, the first n_vq of them) into slots [0, n).  blockIdx.y = head,
// blockIdx.z = 0 keys / 1 values (keys only under InnerQ).  A block takes
// kTokIter rounds of kQuantBlock / (d/8) tokens.
constexpr int kTokIter = 4;
__global__ void __launch_bounds__(kQuantBlock)
    per_token_prefill_kernel(Geometry g, CachePtrs p, const __half *K, const __half *V,
                             int64_t T, Counts uni) {
  const bool is_key = blockIdx.z == 0 && g.scheme == KVQ_INNERQ;
  const TokenDst dst = is_key ? key_dst(g, p) : value_dst(g, p);
  const __half *X = is_key ? K : V;
  const int64_t bh = blockIdx.y;
  const Counts c = seq_counts(g, p, uni, (int)(bh / g.H));
  const int64_t src0 = c.n_sink;
  const int64_t n_tok = (g.scheme == KVQ_KIVI) ? c.n_vq : c.n_quant;
  const int chunks = g.d / 8;
  const int tpr = kQuantBlock / chunks;  // tokens per round
  const int64_t tok0 = (int64_t)blockIdx.x * tpr * kTokIter;
  if (tok0 >= n_tok) return;  // (uniform per block)
  const int lt = threadIdx.x / chunks, j = threadIdx.x - lt * chunks;
  const int lanes = dst.group / 8;

  // Mode bits of this block's tokens, assembled in shared memory (at most
  // kTokIter * kQuantBlock * 8 / 16 bits: groups of >= 16 channels).
  __shared__ uint32_t s_bits[kTokIter * kQuantBlock / 64 + 2];
  const int ng = dst.meta_cols;
  const int64_t bit0 = tok0 * ng;
  const int64_t wbase = bit0 >> 5;
  if (dst.mode) {
    for (int i = threadIdx.x; i < kTokIter * kQuantBlock / 64 + 2; i += blockDim.x) s_bits[i] = 0;
    __syncthreads();
  }

  for (int it = 0; it < kTokIter; ++it) {
    const int64_t t = tok0 + (int64_t)it * tpr + lt;
    const bool valid = t < n_tok;
    float x[8];
    if (valid) {
      load8(X + (bh * T + src0 + t) * g.d + 8 * j, x);
      if (is_key && g.knorm) normalize8(p.k_norm + bh * g.d, 8 * j, x);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = 0.0f;
    }
    if (!dst.mode) {  // KIVI values (outliers, fp16 statistics)
      quant_value_token(g, p, bh, t, j, chunks, x, valid);
      continue;
    }
    const ChunkQ q = quant_chunk(x, lanes, g.bits, true, g.meta16, 0u);
    if (valid) {
      store_token(g, p, dst, bh, t, j, lanes, q);
      if ((j & (lanes - 1)) == 0) {
        const int gi = j / lanes;
        if (q.sym) {
          const int64_t bit = t * ng + gi;
          atomicOr(&s_bits[(bit >> 5) - wbase], 1u << (bit & 31));
        }
      }
    }
  }
  if (!dst.mode) return;
  __syncthreads();
  // Write back the words this block owns.  Blocks own disjoint bit ranges;
  // the block holding the last token also owns the rest of its last word.
  const int64_t tok_end = min(tok0 + (int64_t)tpr * kTokIter, n_tok);
  int64_t bit1 = tok_end * ng;
  if (tok_end == n_tok) bit1 = (bit1 + 31) & ~(int64_t)31;
  const int64_t wlast = (bit1 - 1) >> 5;
  uint32_t *words = dst.mode + bh * g.mode_words;
  for (int64_t w = wbase + threadIdx.x; w <= wlast; w += blockDim.x) {
    const int64_t lo = max(bit0, w * 32) - w * 32, hi = min(bit1, w * 32 + 32) - w * 32;
    const uint32_t mask = (hi - lo == 32) ? 0xffffffffu : (((1u << (hi - lo)) - 1u) << lo);
    const uint32_t bits = s_bits[w - wbase] & mask;
    if (mask == 0xffffffffu) {
      words[w] = bits;
    } else {
      atomicAnd(&words[w], ~mask);
      atomicOr(&words[w], bits);
    }
  }
}

// Prefill, KIVI keys: one block per (G-token group, head).
__global__ void __launch_bounds__(kQuantBlock)
    kivi_key_prefill_kernel(Geometry g, CachePtrs p, const __half *K, int64_t T, Counts uni) {
  __shared__ float s_scale[kMaxHeadDim], s_mn[kMaxHeadDim], s_pmn[kKeyPart], s_pmx[kKeyPart];
  __shared__ uint8_t s_om[kMaskBytes];
  const int64_t bh = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * g.k_group;
  if (t0 >= seq_counts(g, p, uni, (int)(bh / g.H)).n_quant) return;  // (ragged: shorter)
  key_group_per_channel(g, p, bh, K + (bh * T + t0) * g.d, t0, s_scale, s_mn, s_pmn, s_pmx,
                        s_om);
}

// fp16 rows of a prefill, every head: blockIdx.z = 0 the residual / window
// keys, 1 their values, 2 the sink keys, 3 the sink values.  KIVI residual
// rows hold tokens [n_quant, n) in slots 0.. (values under the queue: tokens
// [n_vq, n) in ring slots t mod R); InnerQ window rows hold the last n_resid
// tokens oldest first, sinks the first n_sink.
__global__ void prefill_rows_kernel(Geometry g, CachePtrs p, const __half *K, const __half *V,
                                    int64_t T, Counts uni, int max_rows) {
  const int kind = blockIdx.z;
  const bool val = kind & 1;
  const __half *X = val ? V : K;
  const int vec = g.d / 8;
  const int64_t BH = (int64_t)g.B * g.H;
  const int64_t total = BH * max_rows * vec;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bh = i / ((int64_t)max_rows * vec);
    const int r = (int)((i / vec) % max_rows);
    const int jv = (int)(i % vec);
    const Counts c = seq_counts(g, p, uni, (int)(bh / g.H));
    const int64_t n = c.n_quant + c.n_resid + c.n_sink;  // the sequence's prompt length
    int64_t src;
    __half *dst;
    if (kind >= 2) {
      if (r >= c.n_sink) continue;
      src = r;
      dst = (val ? p.v_sink : p.k_sink) + (bh * g.n_sink + r) * g.d;
    } else if (g.scheme == KVQ_KIVI && val && g.vq) {
      if (r >= n - c.n_vq) continue;
      src = c.n_vq + r;
      dst = p.v_res + (bh * g.residual + src % g.residual) * g.d;
    } else {
      if (r >= c.n_resid) continue;
      src = n - c.n_resid + r;
      dst = (val ? p.v_res : p.k_res) + (bh * g.residual + r) * g.d;
    }
    reinterpret_cast<uint4 *>(dst)[jv] = reinterpret_cast<const uint4 *>(X + (bh * T + src) * g.d)[jv];
  }
}

// KIVI append (one block per head): the token's key enters residual slot
// n_resid and its value slot n_resid (the value queue: ring slot n mod R, n
// the tokens held before).  When the residual reaches R its R keys are
// quantized as R/G groups into slots [n_quant, n_quant + R), and (without the
// queue) its R values per token.  Under the queue, once R values wait the
// oldest (token n_vq) is quantized into value slot n_vq.
__global__ void __launch_bounds__(kQuantBlock)
    kivi_append_kernel(Geometry g, CachePtrs p, const __half *k, const __half *v, Counts uni) {
  __shared__ float s_scale[kMaxHeadDim], s_mn[kMaxHeadDim], s_pmn[kKeyPart], s_pmx[kKeyPart];
  __shared__ uint8_t s_om[kMaskBytes];
  const int64_t bh = blockIdx.x;
  const int d = g.d, R = g.residual;
  const Counts c = seq_counts(g, p, uni, (int)(bh / g.H));
  const int64_t slot = c.n_resid, n = c.n_quant + c.n_resid;
  const bool flush = slot + 1 == R;
  __half *kr = p.k_res + bh * R * d, *vr = p.v_res + bh * R * d;
  const int64_t vslot = g.vq ? n % R : slot;
  for (int cc = threadIdx.x; cc < d / 8; cc += blockDim.x) {
    reinterpret_cast<uint4 *>(kr + slot * d)[cc] = reinterpret_cast<const uint4 *>(k + bh * d)[cc];
    reinterpret_cast<uint4 *>(vr + vslot * d)[cc] = reinterpret_cast<const uint4 *>(v + bh * d)[cc];
  }
  const bool pop = g.vq && n - c.n_vq + 1 == R;
  if (!flush && !pop) return;
  __syncthreads();
  const int chunks = d / 8;
  if (flush) {
    for (int grp = 0; grp < R / g.k_group; ++grp)
      key_group_per_channel(g, p, bh, kr + (int64_t)grp * g.k_group * d,
                            c.n_quant + (int64_t)grp * g.k_group, s_scale, s_mn, s_pmn, s_pmx,
                            s_om);
    if (!g.vq) {
      const int tpr = blockDim.x / chunks;
      for (int t0 = 0; t0 < R; t0 += tpr) {
        const int t = t0 + (int)threadIdx.x / chunks, j = (int)threadIdx.x % chunks;
        const bool valid = t < R;
        float x[8];
        load8(vr + (int64_t)(valid ? t : 0) * d + 8 * j, x);
        quant_value_token(g, p, bh, c.n_quant + t, j, chunks, x, valid);
      }
    }
  }
  if (pop && threadIdx.x < 32) {
    // the oldest queued value (token n_vq, ring slot n_vq mod R) leaves the queue
    const int j = threadIdx.x % chunks;
    const bool valid = (int)threadIdx.x < chunks;
    float x[8];
    load8(vr + (c.n_vq % R) * d + 8 * j, x);
    quant_value_token(g, p, bh, c.n_vq, j, chunks, x, valid);
  }
}

// InnerQ append (one warp per head): the sink fills first, then the window;
// once the window holds W tokens the one in ring slot ring_head (the oldest;
// or the new token itself when there is no window) is quantized into slot
// n_quant and the new token takes its window slot.
__global__ void __launch_bounds__(32)
    innerq_append_kernel(Geometry g, CachePtrs p, const __half *k, const __half *v, Counts uni) {
  const int64_t bh = blockIdx.x;
  const int d = g.d, W = g.residual, S = g.n_sink;
  const Counts c = seq_counts(g, p, uni, (int)(bh / g.H));
  const uint4 *kn = reinterpret_cast<const uint4 *>(k + bh * d);
  const uint4 *vn = reinterpret_cast<const uint4 *>(v + bh * d);
  const int lane = threadIdx.x;
  if (c.n_sink < S || c.n_resid < W) {
    const bool sink = c.n_sink < S;
    const int64_t slot = sink ? c.n_sink : c.n_resid;
    __half *dk = sink ? p.k_sink + (bh * S + slot) * d : p.k_res + (bh * W + slot) * d;
    __half *dv = sink ? p.v_sink + (bh * S + slot) * d : p.v_res + (bh * W + slot) * d;
    for (int cc = lane; cc < d / 8; cc += 32) {
      reinterpret_cast<uint4 *>(dk)[cc] = kn[cc];
      reinterpret_cast<uint4 *>(dv)[cc] = vn[cc];
    }
    return;
  }
  const int64_t slot = c.ring_head, n_quant = c.n_quant;
  const __half *srck = W > 0 ? p.k_res + (bh * W + slot) * d : k + bh * d;
  const __half *srcv = W > 0 ? p.v_res + (bh * W + slot) * d : v + bh * d;
  const int chunks = d / 8;
  for (int it0 = 0; it0 < 2 * chunks; it0 += 32) {
    const int it = it0 + lane;
    const bool valid = it < 2 * chunks;
    const bool is_key = it < chunks;
    const int j = is_key ? it : it - chunks;
    const TokenDst dst = is_key ? key_dst(g, p) : value_dst(g, p);
    float x[8];
    if (valid) {
      load8((is_key ? srck : srcv) + 8 * j, x);
      if (is_key && g.knorm) normalize8(p.k_norm + bh * d, 8 * j, x);
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) x[kk] = 0.0f;
    }
    // Keys and values may use different group sizes: lanes of one group are
    // consecutive and never straddle the key/value boundary (chunks is a
    // multiple of both group widths).
    const int lanes = (valid ? dst.group : 8) / 8;
    const ChunkQ q = quant_chunk(x, lanes, g.bits, true, g.meta16, 0u);
    if (valid) {
      store_token(g, p, dst, bh, n_quant, j, lanes, q);
      if ((j & (lanes - 1)) == 0) {
        const int ng = dst.meta_cols, gi = j / lanes;
        const int64_t bit = n_quant * ng + gi;
        uint32_t *word = dst.mode + bh * g.mode_words + (bit >> 5);
        if (q.sym)
          atomicOr(word, 1u << (bit & 31));
        else
          atomicAnd(word, ~(1u << (bit & 31)));
      }
    }
  }
  if (W == 0) return;
  __syncwarp();
  __half *dk = p.k_res + (bh * W + slot) * d, *dv = p.v_res + (bh * W + slot) * d;
  for (int cc = lane; cc < d / 8; cc += 32) {
    reinterpret_cast<uint4 *>(dk)[cc] = kn[cc];
    reinterpret_cast<uint4 *>(dv)[cc] = vn[cc];
  }
}

__global__ void fill_i32_kernel(int32_t *dst, int n, int32_t v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) dst[i] = v;
}

int copy_blocks(int64_t total_vec) {
  int64_t b = (total_vec + 255) / 256;
  return (int)(b < 1 ? 1 : (b > 65535 ? 65535 : b));
}

}  // namespace

cudaError_t launch_fill_i32(int32_t *dst, int n, int32_t v, cudaStream_t st) {
  fill_i32_kernel<<<copy_blocks(n), 256, 0, st>>>(dst, n, v);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const Geometry &g, const CachePtrs &p, const __half *K,
                           const __half *V, int64_t T, const Counts &c, cudaStream_t st,
                           int *launches) {
  const int64_t BH = (int64_t)g.B * g.H;
  const int chunks = g.d / 8;
  const int tpb = kQuantBlock / chunks;
  const int64_t per_block = (int64_t)tpb * kTokIter;
  int n = 0;
  if (g.scheme == KVQ_INNERQ && g.knorm) {
    // key factors over the whole prompt, before any key is quantized
    const cudaError_t e = cudaMemsetAsync(p.k_norm, 0, sizeof(float) * BH * g.d, st);
    if (e != cudaSuccess) return e;
    if (T > 0) {
      key_absmax_kernel<<<dim3((unsigned)((T + kNormTokens - 1) / kNormTokens), (unsigned)BH),
                          kQuantBlock, 0, st>>>(g, p, K, T);
      ++n;
    }
    key_norm_finish_kernel<<<copy_blocks(BH * g.d), 256, 0, st>>>(p.k_norm, BH * g.d);
    ++n;
  }
  if (g.scheme == KVQ_KIVI) {
    if (c.n_quant > 0) {
      kivi_key_prefill_kernel<<<dim3((unsigned)(c.n_quant / g.k_group), (unsigned)BH),
                                kQuantBlock, 0, st>>>(g, p, K, T, c);
      ++n;
    }
    if (c.n_vq > 0) {
      per_token_prefill_kernel<<<dim3((unsigned)((c.n_vq + per_block - 1) / per_block),
                                      (unsigned)BH, 1),
                                 kQuantBlock, 0, st>>>(g, p, K, V, T, c);
      ++n;
    }
  } else if (c.n_quant > 0) {
    per_token_prefill_kernel<<<dim3((unsigned)((c.n_quant + per_block - 1) / per_block),
                                    (unsigned)BH, 2),
                               kQuantBlock, 0, st>>>(g, p, K, V, T, c);
    ++n;
  }
  // fp16 rows: residual / window keys and values (up to R rows: the value
  // queue holds at most R - 1), sinks
  const int max_rows = g.residual > g.n_sink ? g.residual : g.n_sink;
  if (max_rows > 0 && T > 0) {
    prefill_rows_kernel<<<dim3(copy_blocks(BH * max_rows * chunks), 1, g.n_sink > 0 ? 4 : 2), 256,
                          0, st>>>(g, p, K, V, T, c, max_rows);
    ++n;
  }
  *launches = n;
  return cudaGetLastError();
}

cudaError_t launch_append(const Geometry &g, const CachePtrs &p, const __half *k,
                          const __half *v, const Counts &c, cudaStream_t st) {
  const unsigned BH = (unsigned)(g.B * g.H);
  if (g.scheme == KVQ_KIVI)
    kivi_append_kernel<<<BH, kQuantBlock, 0, st>>>(g, p, k, v, c);
  else
    innerq_append_kernel<<<BH, 32, 0, st>>>(g, p, k, v, c);
  return cudaGetLastError();
}

}  // namespace kvq
