// Prefill quantize+pack and append/flush kernels.
//
// Method: keys per channel over G-token groups, values per token over channel
// groups ("大模型量化技术原理：KIVI、IntactKV、KVQuant", KIVI / 工作原理); residual
// flushed in one batch when it holds R tokens (pgsm.cn how-to §3.1); InnerQ
// per-token groups along the head dimension with a per-group symmetric /
// asymmetric choice, fp16 sinks and recent window (InnerQ page, 方法论 1-4).
//
// Work mapping: one thread owns 8 consecutive channels of one token (one
// 16-byte fp16 load, 2 or 4 packed output bytes), so a warp reads whole
// 256-byte token rows and writes whole packed rows.  Per-token group min/max
// is a butterfly over the lanes of the group; per-channel key statistics are
// one thread per channel walking the G tokens of the group.
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

// Shared scratch of key_group_per_channel: per-row-lane partial minima and
// maxima, [blockDim / (d / 8)][d] each (2048 floats for any d).
constexpr int kKeyPart = kQuantBlock * 8;

// One key group (G tokens of src, row stride d) quantized per channel into
// token slots [t0, t0 + G), t0 a multiple of G.  All threads of the block call
// it; s_scale / s_mn are d-float shared arrays, s_pmn / s_pmx kKeyPart-float
// scratch.  A thread reads 8-channel chunks (16-byte loads) of rows r0, r0 +
// lanes, ...; the per-channel minimum and maximum are then combined over the
// row lanes (min / max are order-free, so the result is that of one pass).
__device__ void key_group_per_channel(const Geometry &g, const CachePtrs &p, int64_t bh,
                                      const __half *src, int64_t t0, float *s_scale,
                                      float *s_mn, float *s_pmn, float *s_pmx) {
  const int d = g.d, G = g.k_group;
  {
    const int chunks = d / 8, lanes = blockDim.x / chunks;
    const int j = threadIdx.x % chunks, r0 = threadIdx.x / chunks;
    float mn8[8], mx8[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      mn8[k] = INFINITY;
      mx8[k] = -INFINITY;
    }
    for (int i = r0; i < G; i += lanes) {
      float x[8];
      load8(src + (int64_t)i * d + 8 * j, x);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
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
  const int lanes = blockDim.x / (d / 8);
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float mn = s_pmn[c], mx = s_pmx[c];
    for (int r = 1; r < lanes; ++r) {
      mn = fminf(mn, s_pmn[r * d + c]);
      mx = fmaxf(mx, s_pmx[r * d + c]);
    }
    mn = canon_zero(mn);
    mx = canon_zero(mx);
    const float sc = asym_scale(mn, mx, g.bits);
    s_scale[c] = sc;
    s_mn[c] = mn;
    float *km = kivi_key_meta(g, p, bh, t0 / G);
    km[c] = sc;
    km[d + c] = mn;
  }
  __syncthreads();
  const int chunks = d / 8;
  for (int it = threadIdx.x; it < G * chunks; it += blockDim.x) {
    const int i = it / chunks, j = it - i * chunks;
    float x[8];
    load8(src + (int64_t)i * d + 8 * j, x);
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = 8 * j + k;
      w |= asym_code(x[k], s_mn[c], s_scale[c], g.bits) << (k * g.bits);
    }
    store_chunk(code_row(g, p, bh, t0 + i, 0), j, w, g.bits);
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

// Key factors, pass 1: the largest |K[t][c]| of tokens [t0, t0 + kNormTokens)
// of head blockIdx.y into n[bh][c] by an atomic max on the bit pattern
// (non-negative floats order like their bits); n starts at 0.
constexpr int kNormTokens = 4096;
__global__ void __launch_bounds__(kQuantBlock)
    key_absmax_kernel(const __half *K, int64_t T, int d, float *n) {
  __shared__ unsigned int s_max[kMaxHeadDim];
  const int64_t bh = blockIdx.y;
  const int chunks = d / 8, rows = kQuantBlock / chunks;
  const int j = threadIdx.x % chunks, r = threadIdx.x / chunks;
  for (int c = threadIdx.x; c < d; c += blockDim.x) s_max[c] = 0u;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kNormTokens;
  const int64_t t1 = min(t0 + kNormTokens, T);
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
// combines the rounds inside its own group.
__device__ __forceinline__ ChunkQ quant_chunk(const float (&x)[8], int lanes, int bits,
                                              bool allow_sym) {
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) {
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
  mn = canon_zero(mn);
  mx = canon_zero(mx);
  ChunkQ r;
  r.sym = allow_sym && choose_symmetric(mn, mx, bits);
  r.codes = 0;
  if (r.sym) {
    r.scale = sym_scale(mn, mx, bits);
    r.zero = __fmul_rn(-(float)(1 << (bits - 1)), r.scale);
#pragma unroll
    for (int k = 0; k < 8; ++k) r.codes |= sym_code(x[k], r.scale, bits) << (k * bits);
  } else {
    r.scale = asym_scale(mn, mx, bits);
    r.zero = mn;
#pragma unroll
    for (int k = 0; k < 8; ++k) r.codes |= asym_code(x[k], mn, r.scale, bits) << (k * bits);
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
    tok_meta(g, p, bh, t, dst.off_scale, dst.meta_cols)[gi] = q.scale;
    tok_meta(g, p, bh, t, dst.off_zero, dst.meta_cols)[gi] = q.zero;
  }
}

// Prefill, per-token groups: tokens [src0, src0 + n_tok) of every head of
// X [B*H][T][d] quantized into slots [0, n_tok).  blockIdx.y = head,
// blockIdx.z = 0 keys / 1 values (keys only under InnerQ).  A block takes
// kTokIter rounds of kQuantBlock / (d/8) tokens.
constexpr int kTokIter = 4;
__global__ void __launch_bounds__(kQuantBlock)
    per_token_prefill_kernel(Geometry g, CachePtrs p, const __half *K, const __half *V,
                             int64_t T, int64_t src0, int64_t n_tok) {
  const bool is_key = blockIdx.z == 0 && g.scheme == KVQ_INNERQ;
  const TokenDst dst = is_key ? key_dst(g, p) : value_dst(g, p);
  const __half *X = is_key ? K : V;
  const int64_t bh = blockIdx.y;
  const int chunks = g.d / 8;
  const int tpr = kQuantBlock / chunks;  // tokens per round
  const int64_t tok0 = (int64_t)blockIdx.x * tpr * kTokIter;
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
    const ChunkQ q = quant_chunk(x, lanes, g.bits, dst.mode != nullptr);
    if (valid) {
      store_token(g, p, dst, bh, t, j, lanes, q);
      if ((j & (lanes - 1)) == 0) {
        const int gi = j / lanes;
        if (dst.mode && q.sym) {
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
  if (tok_end <= tok0) return;
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
    kivi_key_prefill_kernel(Geometry g, CachePtrs p, const __half *K, int64_t T) {
  __shared__ float s_scale[kMaxHeadDim], s_mn[kMaxHeadDim], s_pmn[kKeyPart], s_pmx[kKeyPart];
  const int64_t bh = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * g.k_group;
  key_group_per_channel(g, p, bh, K + (bh * T + t0) * g.d, t0, s_scale, s_mn, s_pmn, s_pmx);
}

// fp16 row copy: rows [src0, src0 + n) of every head of X [B*H][T][d] into
// rows [0, n) of dst [B*H][dst_rows][d].  blockIdx.z: 0 keys, 1 values.
__global__ void copy_rows_kernel(const __half *K, const __half *V, int64_t T, int64_t src0,
                                 int64_t n, __half *dk, __half *dv, int64_t dst_rows, int d,
                                 int64_t n_heads) {
  const __half *X = blockIdx.z == 0 ? K : V;
  __half *D = blockIdx.z == 0 ? dk : dv;
  const int vec = d / 8;
  const int64_t total = n_heads * n * vec;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bh = i / (n * vec);
    const int64_t r = (i / vec) % n;
    const int j = (int)(i % vec);
    const uint4 v = *reinterpret_cast<const uint4 *>(X + (bh * T + src0 + r) * d + 8 * j);
    *reinterpret_cast<uint4 *>(D + (bh * dst_rows + r) * d + 8 * j) = v;
  }
}

// KIVI append: token into residual slot `slot`; on `flush` the whole residual
// (R tokens) is quantized into slots [n_quant, n_quant + R).  One block per head.
__global__ void __launch_bounds__(kQuantBlock)
    kivi_append_kernel(Geometry g, CachePtrs p, const __half *k, const __half *v,
                       int64_t slot, int flush, int64_t n_quant) {
  __shared__ float s_scale[kMaxHeadDim], s_mn[kMaxHeadDim], s_pmn[kKeyPart], s_pmx[kKeyPart];
  const int64_t bh = blockIdx.x;
  const int d = g.d, R = g.residual;
  __half *kr = p.k_res + bh * R * d, *vr = p.v_res + bh * R * d;
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    reinterpret_cast<uint4 *>(kr + slot * d)[c] = reinterpret_cast<const uint4 *>(k + bh * d)[c];
    reinterpret_cast<uint4 *>(vr + slot * d)[c] = reinterpret_cast<const uint4 *>(v + bh * d)[c];
  }
  if (!flush) return;
  __syncthreads();
  for (int grp = 0; grp < R / g.k_group; ++grp)
    key_group_per_channel(g, p, bh, kr + (int64_t)grp * g.k_group * d,
                          n_quant + (int64_t)grp * g.k_group, s_scale, s_mn, s_pmn, s_pmx);
  const TokenDst dst = value_dst(g, p);
  const int chunks = d / 8, lanes = g.v_group / 8;
  const int items = R * chunks;
  const int rounds = (items + blockDim.x - 1) / blockDim.x;
  for (int rd = 0; rd < rounds; ++rd) {
    const int it = rd * blockDim.x + threadIdx.x;
    const bool valid = it < items;
    const int t = valid ? it / chunks : 0, j = valid ? it - t * chunks : 0;
    float x[8];
    load8(vr + (int64_t)t * d + 8 * j, x);
    const ChunkQ q = quant_chunk(x, lanes, g.bits, false);
    if (valid) store_token(g, p, dst, bh, n_quant + t, j, lanes, q);
  }
}

// InnerQ append.  action 0: token into sink slot; 1: into window slot;
// 2: quantize the token in window slot `slot` (the oldest; or the new token
// itself when there is no window) into quantized slot n_quant, then put the
// new token in that window slot.  One warp per head.
__global__ void __launch_bounds__(32)
    innerq_append_kernel(Geometry g, CachePtrs p, const __half *k, const __half *v, int action,
                         int64_t slot, int64_t n_quant) {
  const int64_t bh = blockIdx.x;
  const int d = g.d, W = g.residual, S = g.n_sink;
  const uint4 *kn = reinterpret_cast<const uint4 *>(k + bh * d);
  const uint4 *vn = reinterpret_cast<const uint4 *>(v + bh * d);
  const int lane = threadIdx.x;
  if (action == 0 || action == 1) {
    __half *dk = action == 0 ? p.k_sink + (bh * S + slot) * d : p.k_res + (bh * W + slot) * d;
    __half *dv = action == 0 ? p.v_sink + (bh * S + slot) * d : p.v_res + (bh * W + slot) * d;
    for (int c = lane; c < d / 8; c += 32) {
      reinterpret_cast<uint4 *>(dk)[c] = kn[c];
      reinterpret_cast<uint4 *>(dv)[c] = vn[c];
    }
    return;
  }
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
    const ChunkQ q = quant_chunk(x, lanes, g.bits, true);
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
  for (int c = lane; c < d / 8; c += 32) {
    reinterpret_cast<uint4 *>(dk)[c] = kn[c];
    reinterpret_cast<uint4 *>(dv)[c] = vn[c];
  }
}

int copy_blocks(int64_t total_vec) {
  int64_t b = (total_vec + 255) / 256;
  return (int)(b < 1 ? 1 : (b > 65535 ? 65535 : b));
}

}  // namespace

cudaError_t launch_prefill(const Geometry &g, const CachePtrs &p, const __half *K,
                           const __half *V, int64_t T, int64_t n_quant, int64_t n_resid,
                           int64_t n_sink, cudaStream_t st, int *launches) {
  const int64_t BH = (int64_t)g.B * g.H;
  const int chunks = g.d / 8;
  const int tpb = kQuantBlock / chunks;
  int n = 0;
  if (g.scheme == KVQ_KIVI) {
    if (n_quant > 0) {
      kivi_key_prefill_kernel<<<dim3((unsigned)(n_quant / g.k_group), (unsigned)BH), kQuantBlock, 0,
                                st>>>(g, p, K, T);
      per_token_prefill_kernel<<<dim3((unsigned)((n_quant + tpb * kTokIter - 1) / (tpb * kTokIter)),
                                      (unsigned)BH, 1),
                                 kQuantBlock, 0, st>>>(g, p, K, V, T, 0, n_quant);
      n += 2;
    }
    if (n_resid > 0) {
      copy_rows_kernel<<<dim3(copy_blocks(BH * n_resid * chunks), 1, 2), 256, 0, st>>>(
          K, V, T, n_quant, n_resid, p.k_res, p.v_res, g.residual, g.d, BH);
      ++n;
    }
  } else {
    if (g.knorm) {
      // key factors over the whole prompt, before any key is quantized
      const cudaError_t e = cudaMemsetAsync(p.k_norm, 0, sizeof(float) * BH * g.d, st);
      if (e != cudaSuccess) return e;
      if (T > 0) {
        key_absmax_kernel<<<dim3((unsigned)((T + kNormTokens - 1) / kNormTokens), (unsigned)BH),
                            kQuantBlock, 0, st>>>(K, T, g.d, p.k_norm);
        ++n;
      }
      key_norm_finish_kernel<<<copy_blocks(BH * g.d), 256, 0, st>>>(p.k_norm, BH * g.d);
      ++n;
    }
    if (n_sink > 0) {
      copy_rows_kernel<<<dim3(copy_blocks(BH * n_sink * chunks), 1, 2), 256, 0, st>>>(
          K, V, T, 0, n_sink, p.k_sink, p.v_sink, g.n_sink, g.d, BH);
      ++n;
    }
    if (n_quant > 0) {
      per_token_prefill_kernel<<<dim3((unsigned)((n_quant + tpb * kTokIter - 1) / (tpb * kTokIter)),
                                      (unsigned)BH, 2),
                                 kQuantBlock, 0, st>>>(g, p, K, V, T, n_sink, n_quant);
      ++n;
    }
    if (n_resid > 0) {
      copy_rows_kernel<<<dim3(copy_blocks(BH * n_resid * chunks), 1, 2), 256, 0, st>>>(
          K, V, T, T - n_resid, n_resid, p.k_res, p.v_res, g.residual, g.d, BH);
      ++n;
    }
  }
  *launches = n;
  return cudaGetLastError();
}

cudaError_t launch_append(const Geometry &g, const CachePtrs &p, const __half *k,
                          const __half *v, int64_t n_quant, int64_t n_resid, int64_t n_sink,
                          int64_t ring_head, cudaStream_t st) {
  const unsigned BH = (unsigned)(g.B * g.H);
  if (g.scheme == KVQ_KIVI) {
    const int flush = (n_resid + 1 == g.residual) ? 1 : 0;
    kivi_append_kernel<<<BH, kQuantBlock, 0, st>>>(g, p, k, v, n_resid, flush, n_quant);
  } else {
    int action;
    int64_t slot;
    if (n_sink < g.n_sink) {
      action = 0;
      slot = n_sink;
    } else if (n_resid < g.residual) {
      action = 1;
      slot = n_resid;
    } else {
      action = 2;
      slot = ring_head;
    }
    innerq_append_kernel<<<BH, 32, 0, st>>>(g, p, k, v, action, slot, n_quant);
  }
  return cudaGetLastError();
}

}  // namespace kvq
