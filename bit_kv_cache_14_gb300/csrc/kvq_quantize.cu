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

// ---- codes of 8 elements ---------------------------------------------------
// The product r = d * (1 / scale) is rounded to an integer by adding 1.5 *
// 2^23 (round to nearest even, |r| < 2^22), clamped in that domain and read
// from the low mantissa bits: about ten instructions an element.  A lane whose
// product lies within kTieGuard of a half-integer for any element (rare; or a
// product out of range) redoes its 8 codes with asym_code_inv / sym_code_inv,
// where the IEEE quotient decides: the codes are exactly those of the formula.
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr int kMagicBits = 0x4B400000;

__device__ __forceinline__ float magic_round(float r, bool &tie) {
  const float m = __fadd_rn(r, kMagic);
  tie |= !(fabsf(__fsub_rn(r, __fsub_rn(m, kMagic))) < 0.5f - kTieGuard);
  return m;
}

// Asymmetric codes; z / s / inv hold one value per element (PER, the KIVI
// key channels) or one for all 8 (a per-token group).  om: outliers, code 0.
template <int BITS, bool PER>
__device__ __forceinline__ uint32_t pack_asym(const float (&x)[8], uint32_t om, const float *z,
                                              const float *s, const float *inv) {
  constexpr float top = (float)((1 << BITS) - 1);
  bool tie = false;
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int i = PER ? e : 0;
    bool te = false;
    const float m = magic_round(__fmul_rn(__fsub_rn(x[e], z[i]), inv[i]), te);
    const float mc = fminf(fmaxf(m, kMagic), kMagic + top);
    const uint32_t c = (uint32_t)(__float_as_int(mc) - kMagicBits);
    if (!((om >> e) & 1u)) {  // (an outlier's product does not count)
      w |= c << (e * BITS);
      tie |= te;
    }
  }
  if (tie) {
    w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = PER ? e : 0;
      if (!((om >> e) & 1u)) w |= asym_code_inv(x[e], z[i], s[i], inv[i], BITS) << (e * BITS);
    }
  }
  return w;
}

// Symmetric codes of one group: q + 2^(b-1), q = clamp(rint(x / scale)).
template <int BITS>
__device__ __forceinline__ uint32_t pack_sym(const float (&x)[8], float s, float inv) {
  constexpr int half = 1 << (BITS - 1);
  constexpr float lim = (float)(half - 1);
  bool tie = false;
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float m = magic_round(__fmul_rn(x[e], inv), tie);
    const float mc = fminf(fmaxf(m, kMagic - lim), kMagic + lim);
    w |= (uint32_t)(__float_as_int(mc) - kMagicBits + half) << (e * BITS);
  }
  if (tie) {
    w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) w |= sym_code_inv(x[e], s, inv, BITS) << (e * BITS);
  }
  return w;
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
                                      float *s_mn, float *s_inv, float *s_pmn, float *s_pmx,
                                      uint8_t *s_om) {
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
    s_inv[c] = recip_or_zero(st.scale);
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
    const int c0 = 8 * jj;
    const uint32_t w =
        g.bits == 2 ? pack_asym<2, true>(x, om, s_mn + c0, s_scale + c0, s_inv + c0)
                    : pack_asym<4, true>(x, om, s_mn + c0, s_scale + c0, s_inv + c0);
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
// it may differ between lanes of a warp).  Every lane of the warp must call it
// with the same `rounds` (a power of two >= every calling lane's `lanes`): the
// butterfly runs its full-mask rounds up to it and each lane only combines the
// rounds inside its own group.  om: this lane's outliers (they take no part in
// the statistics and store code 0); a group left without an element stores
// scale 0 and zero 0.
template <int BITS>
__device__ __forceinline__ ChunkQ quant_chunk(const float (&x)[8], int lanes, int rounds,
                                              bool allow_sym, bool f16, uint32_t om) {
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if ((om >> k) & 1u) continue;
    mn = fminf(mn, x[k]);
    mx = fmaxf(mx, x[k]);
  }
  for (int off = 1; off < rounds; off <<= 1) {
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
  r.sym = allow_sym && choose_symmetric(mn, mx, BITS);
  const Stats st = r.sym ? sym_stats(mn, mx, BITS, f16) : asym_stats(mn, mx, BITS, f16);
  r.scale = st.scale;
  r.zero = st.zero;
  const float inv = recip_or_zero(r.scale);
  r.codes = r.sym ? pack_sym<BITS>(x, r.scale, inv)
                  : pack_asym<BITS, false>(x, om, &r.zero, &r.scale, &inv);
  return r;
}

// quant_chunk for a width known only at run time.
__device__ __forceinline__ ChunkQ quant_chunk_b(const float (&x)[8], int lanes, int rounds,
                                                int bits, bool allow_sym, bool f16, uint32_t om) {
  return bits == 2 ? quant_chunk<2>(x, lanes, rounds, allow_sym, f16, om)
                   : quant_chunk<4>(x, lanes, rounds, allow_sym, f16, om);
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
  const ChunkQ q = quant_chunk_b(x, lanes, lanes, g.bits, false, g.meta16, om);
  if (valid) store_token(g, p, dst, bh, t, j, lanes, q);
}

// ---- prefill of per-token groups, one lane per (token, group) --------------
// Codes of n_el elements of one group, two at a time with the packed fp32x2
// IEEE operations (each component rounded exactly as the scalar one), the
// rint by the 1.5 * 2^23 addition; `tie` collects |r - rint(r)| close to 1/2
// (the caller then redoes the group with the IEEE quotient).  CLAMP: clamp to
// the code range (needed only when the stored statistics are rounded to fp16:
// with fp32 statistics every product already lies in range).
template <int BITS, bool SYM, bool CLAMP>
__device__ __forceinline__ uint32_t codes_pair(float2 x, float2 nz, float2 inv, float &tie_max) {
  constexpr int half = 1 << (BITS - 1);
  constexpr float lo = SYM ? -(float)(half - 1) : 0.0f;
  constexpr float hi = SYM ? (float)(half - 1) : (float)((1 << BITS) - 1);
  const float2 d = SYM ? x : __fadd2_rn(x, nz);
  const float2 r = __fmul2_rn(d, inv);
  float2 m = __fadd2_rn(r, make_float2(kMagic, kMagic));
  const float2 ri = __fadd2_rn(m, make_float2(-kMagic, -kMagic));  // rint(r), exact
  const float2 e = __fadd2_rn(r, make_float2(-ri.x, -ri.y));
  tie_max = fmaxf(tie_max, fmaxf(fabsf(e.x), fabsf(e.y)));
  if (CLAMP || SYM) {
    m.x = fminf(fmaxf(m.x, kMagic + lo), kMagic + hi);
    m.y = fminf(fmaxf(m.y, kMagic + lo), kMagic + hi);
  }
  const uint32_t c0 = (uint32_t)(__float_as_int(m.x) - kMagicBits + (SYM ? half : 0));
  const uint32_t c1 = (uint32_t)(__float_as_int(m.y) - kMagicBits + (SYM ? half : 0));
  return c0 | (c1 << BITS);
}

// Codes of an element pair against per-lane parameters: r = (x + nz) * inv,
// rint by the 1.5 * 2^23 addition, clamped to [lo, hi], plus off (asymmetric:
// nz = -zero, [0, 2^b - 1], off 0; symmetric: nz = 0, [-(2^(b-1) - 1),
// 2^(b-1) - 1], off 2^(b-1)) -- one branch-free path for both modes.
template <int BITS>
__device__ __forceinline__ uint32_t codes_pair_any(float2 x, float2 nz, float2 inv, float lo,
                                                   float hi, int off, float &tie_max) {
  const float2 r = __fmul2_rn(__fadd2_rn(x, nz), inv);
  float2 m = __fadd2_rn(r, make_float2(kMagic, kMagic));
  const float2 ri = __fadd2_rn(m, make_float2(-kMagic, -kMagic));  // rint(r), exact
  const float2 e = __fadd2_rn(r, make_float2(-ri.x, -ri.y));
  tie_max = fmaxf(tie_max, fmaxf(fabsf(e.x), fabsf(e.y)));
  m.x = fminf(fmaxf(m.x, kMagic + lo), kMagic + hi);
  m.y = fminf(fmaxf(m.y, kMagic + lo), kMagic + hi);
  const uint32_t c0 = (uint32_t)(__float_as_int(m.x) - kMagicBits + off);
  const uint32_t c1 = (uint32_t)(__float_as_int(m.y) - kMagicBits + off);
  return c0 | (c1 << BITS);
}

// Outliers of one token row of raw fp16 values spread over `nl` aligned
// consecutive lanes, each holding GC of them (lane position li, channels
// li*GC ..): the k largest magnitudes, equal ones to the lower channel (k
// rounds of a maximum over the row's lanes of (|x| bits, 255 - channel)).
// Sets taken[] (this lane's outlier bits) and writes the row's list
// ((channel << 16) | fp16 bits, channels ascending) to `list` when valid.
// Every lane calls it.
template <int GC>
__device__ __forceinline__ void row_outliers(const __half *xh, int li, int nl, int k,
                                             uint32_t (&taken)[(GC + 31) / 32], uint32_t *list,
                                             bool valid) {
#pragma unroll
  for (int w = 0; w < (GC + 31) / 32; ++w) taken[w] = 0u;
  for (int r = 0; r < k; ++r) {
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < GC; ++e)
      if (!((taken[e >> 5] >> (e & 31)) & 1u))
        m = max(m, ((uint32_t)(__half_as_ushort(xh[e]) & 0x7fffu) << 8) |
                       (uint32_t)(255 - (li * GC + e)));
    for (int off = 1; off < 8; off <<= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, m, off);
      if (off < nl) m = max(m, o);
    }
    const int c = 255 - (int)(m & 255u);
    if (c / GC == li) taken[(c % GC) >> 5] |= 1u << ((c % GC) & 31);
  }
  int cnt = 0;
#pragma unroll
  for (int w = 0; w < (GC + 31) / 32; ++w) cnt += __popc(taken[w]);
  int pre = cnt;
  for (int dlt = 1; dlt < nl; dlt <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, pre, dlt, nl);
    if (li >= dlt) pre += y;
  }
  int pos = pre - cnt;
  if (!valid) return;
#pragma unroll
  for (int e = 0; e < GC; ++e)
    if ((taken[e >> 5] >> (e & 31)) & 1u)
      list[pos++] = ((uint32_t)(li * GC + e) << 16) | (uint32_t)__half_as_ushort(xh[e]);
}

// Prefill of per-token groups: every lane quantizes one (token, group) of
// GL 16-byte chunks (GC = 8 GL channels) -- its statistics once, no shuffle
// but for outliers, one branch-free code path for both modes -- and a warp
// covers 32 / (d / GC) whole tokens, so the InnerQ mode bits of a warp are
// one 32-bit word (a ballot).  The row stays in registers as its raw fp16
// pairs.  KIND 0: InnerQ keys (from row n_sink on; normalized under
// KVQ_INNERQ_KNORM), 1: InnerQ values, 2: KIVI values (from row 0, the first
// n_vq of them; outliers).
template <int BITS, int GL, int KIND>
__global__ void __launch_bounds__(kQuantBlock)
    group_prefill_kernel(Geometry g, CachePtrs p, const __half *X, int64_t T, Counts uni) {
  constexpr int GC = GL * 8, NP = GC / 2;  // elements, element pairs
  constexpr bool KEY = KIND == 0, MODE = KIND != 2;
  __shared__ float s_rk[kMaxHeadDim];  // reciprocal key factors (KVQ_INNERQ_KNORM)
  const int d = g.d, ng = d / GC, tpw = 32 / ng;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t bh = blockIdx.y;
  const Counts c = seq_counts(g, p, uni, (int)(bh / g.H));
  const int64_t src0 = c.n_sink;
  const int64_t n_tok = KIND == 2 ? c.n_vq : c.n_quant;
  const bool norm = KEY && g.knorm;
  if (norm) {
    for (int i = threadIdx.x; i < d; i += blockDim.x)
      s_rk[i] = __fdiv_rn(1.0f, p.k_norm[bh * d + i]);
    __syncthreads();
  }
  const int64_t tw = ((int64_t)blockIdx.x * (kQuantBlock / 32) + warp) * tpw;  // first token
  if (tw >= n_tok) return;  // (whole warps)
  const int gi = lane % ng;
  const int64_t t = tw + lane / ng;
  const bool valid = t < n_tok;
  __half2 xh[NP];
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(
        X + (bh * T + src0 + (valid ? t : tw)) * d + gi * GC);
#pragma unroll
    for (int k = 0; k < GL; ++k) {
      const uint4 raw = src[k];
      xh[4 * k] = *reinterpret_cast<const __half2 *>(&raw.x);
      xh[4 * k + 1] = *reinterpret_cast<const __half2 *>(&raw.y);
      xh[4 * k + 2] = *reinterpret_cast<const __half2 *>(&raw.z);
      xh[4 * k + 3] = *reinterpret_cast<const __half2 *>(&raw.w);
    }
  }
  // element pair i as fp32 (normalized keys: times the reciprocal factors)
  auto pair = [&](int i) -> float2 {
    const float2 f = __half22float2(xh[i]);
    if (!norm) return f;
    return __fmul2_rn(f, make_float2(s_rk[gi * GC + 2 * i], s_rk[gi * GC + 2 * i + 1]));
  };
  uint32_t taken[(GC + 31) / 32];
#pragma unroll
  for (int w = 0; w < (GC + 31) / 32; ++w) taken[w] = 0u;
  const bool outl = KIND == 2 && g.n_out > 0;
  if (outl)
    row_outliers<GC>(reinterpret_cast<const __half *>(xh), gi, ng, g.n_out, taken,
                     valid ? tok_outliers(g, p, bh, t, g.blk_vo) : nullptr, valid);
  float mn, mx;
  if (!norm && !outl) {
    __half2 a = xh[0], b = xh[0];
#pragma unroll
    for (int i = 1; i < NP; ++i) {
      a = __hmin2(a, xh[i]);
      b = __hmax2(b, xh[i]);
    }
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    mn = fminf(fa.x, fa.y);
    mx = fmaxf(fb.x, fb.y);
  } else {
    mn = INFINITY;
    mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const float2 f = pair(i);
      if (!((taken[(2 * i) >> 5] >> ((2 * i) & 31)) & 1u)) {
        mn = fminf(mn, f.x);
        mx = fmaxf(mx, f.x);
      }
      if (!((taken[(2 * i + 1) >> 5] >> ((2 * i + 1) & 31)) & 1u)) {
        mn = fminf(mn, f.y);
        mx = fmaxf(mx, f.y);
      }
    }
  }
  bool sym = false;
  Stats st{0.0f, 0.0f};
  if (!(mn > mx)) {  // (else no inlier: scale 0, zero 0)
    mn = canon_zero(mn);
    mx = canon_zero(mx);
    sym = MODE && choose_symmetric(mn, mx, BITS);
    st = sym ? sym_stats(mn, mx, BITS, g.meta16) : asym_stats(mn, mx, BITS, g.meta16);
  }
  const float inv = recip_or_zero(st.scale);
  constexpr int WPG = GC * BITS / 32;  // code words of a group
  constexpr int PPW = 16 / BITS;       // element pairs a code word holds
  uint32_t cw[WPG];
  {
    constexpr int half = 1 << (BITS - 1);
    const float lo = sym ? -(float)(half - 1) : 0.0f;
    const float hi = sym ? (float)(half - 1) : (float)((1 << BITS) - 1);
    const int off = sym ? half : 0;
    const float nzv = sym ? 0.0f : -st.zero;
    const float2 nz = make_float2(nzv, nzv), iv = make_float2(inv, inv);
    float tie = 0.0f;
    if (MODE || g.meta16 || outl) {
      // both modes (per-lane range and offset), or codes that can leave
      // their range: the clamped path
#pragma unroll
      for (int w = 0; w < WPG; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < PPW; ++i)
          word |= codes_pair_any<BITS>(pair(w * PPW + i), nz, iv, lo, hi, off, tie)
                  << (2 * i * BITS);
        cw[w] = word;
      }
    } else {
      // KIVI values with fp32 statistics: every product lies in the code range
#pragma unroll
      for (int w = 0; w < WPG; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < PPW; ++i)
          word |= codes_pair<BITS, false, false>(pair(w * PPW + i), nz, iv, tie) << (2 * i * BITS);
        cw[w] = word;
      }
    }
    if (!(tie < 0.5f - kTieGuard)) {
      // a product close to a tie (or out of range): the IEEE quotient decides
      for (int w = 0; w < WPG; ++w) {
        uint32_t word = 0;
        for (int i = 0; i < PPW; ++i) {
          const float2 f = pair(w * PPW + i);
          const uint32_t c0 = sym ? sym_code_inv(f.x, st.scale, inv, BITS)
                                  : asym_code_inv(f.x, st.zero, st.scale, inv, BITS);
          const uint32_t c1 = sym ? sym_code_inv(f.y, st.scale, inv, BITS)
                                  : asym_code_inv(f.y, st.zero, st.scale, inv, BITS);
          word |= (c0 | (c1 << BITS)) << (2 * i * BITS);
        }
        cw[w] = word;
      }
    }
  }
  if (outl) {  // outliers store code 0
#pragma unroll
    for (int e = 0; e < GC; ++e)
      if ((taken[e >> 5] >> (e & 31)) & 1u)
        cw[e / (32 / BITS)] &= ~(((1u << BITS) - 1u) << ((e % (32 / BITS)) * BITS));
  }
  const TokenDst dst = KEY ? key_dst(g, p) : value_dst(g, p);
  if (valid) {
    uint8_t *blk = tok_block(g, p, bh, t);
    const int row = (int)(t % kBlockTokens);
    uint32_t *code = reinterpret_cast<uint32_t *>(blk + dst.off_codes + row * g.row_bytes) + gi * WPG;
    if (WPG == 1) {
      code[0] = cw[0];
    } else if (WPG == 2) {
      *reinterpret_cast<uint2 *>(code) = make_uint2(cw[0], cw[1 % WPG]);
    } else {
#pragma unroll
      for (int w = 0; w < WPG; w += 4)
        *reinterpret_cast<uint4 *>(code + w) =
            make_uint4(cw[w % WPG], cw[(w + 1) % WPG], cw[(w + 2) % WPG], cw[(w + 3) % WPG]);
    }
    st_meta(g, blk + dst.off_scale + row * ng * g.msz, gi, st.scale);
    st_meta(g, blk + dst.off_zero + row * ng * g.msz, gi, st.zero);
  }
  if (MODE) {
    // the warp's 32 mode bits are one word: tokens tw .. tw + tpw, groups in order
    const uint32_t bits = __ballot_sync(0xffffffffu, valid && sym);
    if (lane == 0) dst.mode[bh * g.mode_words + (tw * ng >> 5)] = bits;
  }
}

// One KIVI key group (G tokens of src, row stride D) quantized per channel by
// ONE warp, with no shared memory and no block barrier: lane (rs, j) holds the
// 8 channels of chunk j (a 16-byte load per row) for the rows rs, rs + RL,
// ... (RL = 32 / (D/8) row slices); the per-channel minimum and maximum are
// combined over the slices by shuffles, each lane takes its 8 channels'
// statistics and reciprocals, and a second pass over the same rows (L1 hits)
// packs the codes.  With outliers each row's are found by the 16 (or 8) lanes
// of its slice, listed in the first pass, and found again in the second.
// GT > 0 (the group size, 16 or 32, known at compile time; no outliers): each
// lane issues the loads of all its rows at once for the first pass, so a warp
// has the whole group in flight; the second pass reads them again from L1.
template <int D, int BITS, int GT = 0>
__device__ __forceinline__ void key_group_warp(const Geometry &g, const CachePtrs &p, int64_t bh,
                                               const __half *src, int64_t t0) {
  constexpr int CH = D / 8, RL = 32 / CH;
  constexpr int NR = GT > 0 ? GT / RL : 1;  // rows a lane holds (GT > 0)
  const int lane = threadIdx.x & 31, j = lane % CH, rs = lane / CH;
  const int G = GT > 0 ? GT : g.k_group;
  uint4 held[NR];
  if constexpr (GT > 0) {
#pragma unroll
    for (int r = 0; r < NR; ++r)
      held[r] = *reinterpret_cast<const uint4 *>(src + (int64_t)(rs + r * RL) * D + 8 * j);
  }
  float mn[8], mx[8];
  if (GT > 0 || g.n_out == 0) {
    // raw fp16 keys: the minimum and maximum on half2 pairs (exact)
    __half2 hmn[4], hmx[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hmn[e] = __float2half2_rn(INFINITY);
      hmx[e] = __float2half2_rn(-INFINITY);
    }
    auto fold = [&](const uint4 &raw) {
      const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hmn[e] = __hmin2(hmn[e], h[e]);
        hmx[e] = __hmax2(hmx[e], h[e]);
      }
    };
    if constexpr (GT > 0) {
#pragma unroll
      for (int r = 0; r < NR; ++r) fold(held[r]);
    } else {
      for (int i = rs; i < G; i += RL)
        fold(*reinterpret_cast<const uint4 *>(src + (int64_t)i * D + 8 * j));
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = __half22float2(hmn[e]), b = __half22float2(hmx[e]);
      mn[2 * e] = a.x;
      mn[2 * e + 1] = a.y;
      mx[2 * e] = b.x;
      mx[2 * e + 1] = b.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      mn[e] = INFINITY;
      mx[e] = -INFINITY;
    }
    for (int i = rs; i < G; i += RL) {
      float x[8];
      load8(src + (int64_t)i * D + 8 * j, x);
      const uint32_t om = outlier_mask(x, j, CH, g.n_out);
      store_outliers(tok_outliers(g, p, bh, t0 + i, g.blk_ko), x, j, CH, om, true);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if ((om >> e) & 1u) continue;
        mn[e] = fminf(mn[e], x[e]);
        mx[e] = fmaxf(mx[e], x[e]);
      }
    }
  }
#pragma unroll
  for (int off = CH; off < 32; off <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      mn[e] = fminf(mn[e], __shfl_xor_sync(0xffffffffu, mn[e], off));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], off));
    }
  float sc[8], zr[8], inv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    // no inlier in the group (every element an outlier): scale 0, zero 0
    const Stats st = mn[e] > mx[e] ? Stats{0.0f, 0.0f}
                                   : asym_stats(canon_zero(mn[e]), canon_zero(mx[e]), BITS,
                                                g.meta16);
    sc[e] = st.scale;
    zr[e] = st.zero;
    inv[e] = recip_or_zero(st.scale);
  }
  if (rs == 0) {
    uint8_t *km = kivi_key_meta(g, p, bh, t0 / G);
    if (g.meta16) {
      __half2 hs[4], hz[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hs[e] = __floats2half2_rn(sc[2 * e], sc[2 * e + 1]);
        hz[e] = __floats2half2_rn(zr[2 * e], zr[2 * e + 1]);
      }
      reinterpret_cast<uint4 *>(km)[j] = *reinterpret_cast<const uint4 *>(hs);
      reinterpret_cast<uint4 *>(km + D * 2)[j] = *reinterpret_cast<const uint4 *>(hz);
    } else {
      float4 *ks = reinterpret_cast<float4 *>(km) + 2 * j;
      float4 *kz = reinterpret_cast<float4 *>(km + D * 4) + 2 * j;
      ks[0] = make_float4(sc[0], sc[1], sc[2], sc[3]);
      ks[1] = make_float4(sc[4], sc[5], sc[6], sc[7]);
      kz[0] = make_float4(zr[0], zr[1], zr[2], zr[3]);
      kz[1] = make_float4(zr[4], zr[5], zr[6], zr[7]);
    }
  }
  float2 nz[4], iv[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    nz[e] = make_float2(-zr[2 * e], -zr[2 * e + 1]);
    iv[e] = make_float2(inv[2 * e], inv[2 * e + 1]);
  }
  // codes leave their range only for outliers or fp16-rounded statistics
  const bool clamp = g.meta16 || g.n_out > 0;
  // the group's rows are consecutive token rows of one block (G <= 32) or of
  // G / 32 consecutive blocks of the head
  uint8_t *blk0 = tok_block(g, p, bh, t0);
  const int r0 = (int)(t0 % kBlockTokens);
  for (int i = rs; i < G; i += RL) {
    float x[8];
    load8(src + (int64_t)i * D + 8 * j, x);
    const uint32_t om = GT == 0 && g.n_out > 0 ? outlier_mask(x, j, CH, g.n_out) : 0u;
    float tie = 0.0f;
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 xv = make_float2(x[2 * e], x[2 * e + 1]);
      const uint32_t cc = clamp ? codes_pair<BITS, false, true>(xv, nz[e], iv[e], tie)
                                : codes_pair<BITS, false, false>(xv, nz[e], iv[e], tie);
      w |= cc << (2 * e * BITS);
    }
    if (!(tie < 0.5f - kTieGuard)) w = pack_asym<BITS, true>(x, 0u, zr, sc, inv);
    if (om) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if ((om >> e) & 1u) w &= ~(((1u << BITS) - 1u) << (e * BITS));
    }
    const int row = r0 + i;
    store_chunk(blk0 + (int64_t)(row / kBlockTokens) * g.block_bytes +
                    (row % kBlockTokens) * g.row_bytes,
                j, w, BITS);
  }
}

// Prefill, KIVI keys: one warp per (head, G-token group), 8 warps a block.
template <int D, int BITS, int GT>
__global__ void __launch_bounds__(kQuantBlock)
    kivi_key_prefill_kernel(Geometry g, CachePtrs p, const __half *K, int64_t T, Counts uni,
                            int64_t groups_per_head) {
  const int64_t gi = (int64_t)blockIdx.x * (kQuantBlock / 32) + (threadIdx.x >> 5);
  if (gi >= (int64_t)g.B * g.H * groups_per_head) return;  // (whole warps)
  const int64_t bh = gi / groups_per_head;
  const int64_t t0 = (gi - bh * groups_per_head) * g.k_group;
  if (t0 >= seq_counts(g, p, uni, (int)(bh / g.H)).n_quant) return;  // (ragged: shorter)
  key_group_warp<D, BITS, GT>(g, p, bh, K + (bh * T + t0) * D, t0);
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
  __shared__ float s_scale[kMaxHeadDim], s_mn[kMaxHeadDim], s_inv[kMaxHeadDim];
  __shared__ float s_pmn[kKeyPart], s_pmx[kKeyPart];
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
                            c.n_quant + (int64_t)grp * g.k_group, s_scale, s_mn, s_inv, s_pmn,
                            s_pmx, s_om);
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
    const ChunkQ q = quant_chunk_b(x, lanes, 16, g.bits, true, g.meta16, 0u);
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

// group_prefill_kernel for a kind, group width and code width known at run
// time.
template <int BITS, int KIND>
cudaError_t launch_group_prefill_b(const Geometry &g, const CachePtrs &p, const __half *X,
                                   int64_t T, const Counts &c, int group, int64_t n_tok,
                                   cudaStream_t st) {
  const int ng = g.d / group, tpb = (kQuantBlock / 32) * (32 / ng);
  const dim3 grid((unsigned)((n_tok + tpb - 1) / tpb), (unsigned)(g.B * g.H));
  switch (group) {
    case 16: group_prefill_kernel<BITS, 2, KIND><<<grid, kQuantBlock, 0, st>>>(g, p, X, T, c); break;
    case 32: group_prefill_kernel<BITS, 4, KIND><<<grid, kQuantBlock, 0, st>>>(g, p, X, T, c); break;
    case 64: group_prefill_kernel<BITS, 8, KIND><<<grid, kQuantBlock, 0, st>>>(g, p, X, T, c); break;
    case 128: group_prefill_kernel<BITS, 16, KIND><<<grid, kQuantBlock, 0, st>>>(g, p, X, T, c); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_group_prefill_k(const Geometry &g, const CachePtrs &p, const __half *X,
                                   int64_t T, const Counts &c, int group, int64_t n_tok,
                                   cudaStream_t st) {
  return g.bits == 2 ? launch_group_prefill_b<2, KIND>(g, p, X, T, c, group, n_tok, st)
                     : launch_group_prefill_b<4, KIND>(g, p, X, T, c, group, n_tok, st);
}

cudaError_t launch_group_prefill(const Geometry &g, const CachePtrs &p, const __half *X,
                                 int64_t T, const Counts &c, int kind, int group, int64_t n_tok,
                                 cudaStream_t st) {
  if (kind == 0) return launch_group_prefill_k<0>(g, p, X, T, c, group, n_tok, st);
  if (kind == 1) return launch_group_prefill_k<1>(g, p, X, T, c, group, n_tok, st);
  return launch_group_prefill_k<2>(g, p, X, T, c, group, n_tok, st);
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
      const int64_t gph = c.n_quant / g.k_group;
      const int64_t warps = BH * gph, per = kQuantBlock / 32;
      const unsigned blocks = (unsigned)((warps + per - 1) / per);
      // groups of 16 or 32 tokens without outliers: the register-resident form
      const int gt = g.n_out > 0 ? 0 : g.k_group == 32 ? 32 : g.k_group == 16 ? 16 : 0;
      auto pick = [&](auto d_c, auto b_c) {
        constexpr int D = decltype(d_c)::value, B = decltype(b_c)::value;
        return gt == 32 ? kivi_key_prefill_kernel<D, B, 32>
             : gt == 16 ? kivi_key_prefill_kernel<D, B, 16> : kivi_key_prefill_kernel<D, B, 0>;
      };
      using I64 = std::integral_constant<int, 64>;
      using I128 = std::integral_constant<int, 128>;
      using B2 = std::integral_constant<int, 2>;
      using B4 = std::integral_constant<int, 4>;
      auto kern = g.d == 64 ? (g.bits == 2 ? pick(I64{}, B2{}) : pick(I64{}, B4{}))
                            : (g.bits == 2 ? pick(I128{}, B2{}) : pick(I128{}, B4{}));
      kern<<<blocks, kQuantBlock, 0, st>>>(g, p, K, T, c, gph);
      ++n;
    }
    if (c.n_vq > 0) {
      const cudaError_t e = launch_group_prefill(g, p, V, T, c, 2, g.v_group, c.n_vq, st);
      if (e != cudaSuccess) return e;
      ++n;
    }
  } else if (c.n_quant > 0) {
    cudaError_t e = launch_group_prefill(g, p, K, T, c, 0, g.k_group, c.n_quant, st);
    if (e == cudaSuccess) e = launch_group_prefill(g, p, V, T, c, 1, g.v_group, c.n_quant, st);
    if (e != cudaSuccess) return e;
    n += 2;
  }
  // fp16 rows: residual / window keys and values (up to R rows: the value
  // queue holds at most R - 1), sinks
  const int max_rows = g.residual > g.n_sink ? g.residual : g.n_sink;
  // (uniform lengths: nothing to copy when the prompt left no fp16 row)
  const int64_t n_all = c.n_quant + c.n_resid + c.n_sink;
  const bool rows = g.ragged || c.n_resid > 0 || c.n_sink > 0 || c.n_vq < n_all;
  if (max_rows > 0 && T > 0 && rows) {
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
