// Decode attention over keys cached BEFORE the rotary position embedding.
//
// Method ("大模型量化技术原理：KIVI、IntactKV、KVQuant", KVQuant / 技术原理 二):
// keys are quantized before RoPE, and the embedding is applied after
// dequantization inside the q.K^T kernel.  RoPE turns channel pair i =
// (2i, 2i+1) of a vector at position p by the angle p * theta_i, theta_i =
// base^(-2i/d) (RoFormer's rotation).  Rotations compose, so
//     score(t) = R(p_t) k_t . R(s) q = k_t . R(s - p_t) q:
// the kernel turns the query, never a key, and never materialises a rotated
// or dequantized key.
//   * A 32-token sub-tile whose first token sits at position p0 gets the
//     anchor query A = R(s - p0) q (d/2 angles, two per lane).
//   * Its token j needs R(-j) A; pair i then contributes
//         cos(j theta_i) (k_a A_a + k_b A_b) + sin(j theta_i) (k_a A_b - k_b A_a),
//     with cos / sin of j theta_i from a 32 x d/2 table in shared memory that
//     every sub-tile and head shares.
//   * The dequantization k = code * scale + zero (KIVI: per channel of the
//     key group; InnerQ: per token group, times the channel factor of the key
//     normalization) is folded into six per-pair weights computed with the
//     anchor, so a token costs six FMAs per channel pair and head (KIVI).
//   * Codes become floats exactly without a conversion instruction: a code
//     masked in place inside its 16-bit half, OR-ed into the mantissa of
//     2^23, minus 2^23, is code * 2^offset; the weights carry 2^-offset.
// Angles: positions below 2^24 are exact in fp32.  p * theta is formed as a
// float-float product (theta split into hi + lo), reduced by 2 pi with a
// three-part constant (W. J. Cody, W. Waite, "Software Manual for the
// Elementary Functions", 1980), and its cosine and sine come from __sincosf
// of the reduced angle (|error| ~ 1e-6 rad in all).
// Values are not rotated; their codes use the same in-place conversion, the
// power of two applied once to each accumulator at the end.
// Work split: one block per (split, KV head); the quantized tokens are cut
// into splits so that one wave of blocks fills every SM (blocks per SM from
// the occupancy calculator), plus one split for the fp16 sink / residual /
// window tokens (each with its own angle).  Each warp loads its sub-tile's
// code rows before computing the sub-tile's weights, so the two loads'
// latencies overlap.  The block that finishes a head last merges the splits'
// (m, l, o) by log-sum-exp (IntactKV / KV Cache量化 on the same page: fp16
// tokens joined with the dequantized ones).
#include <math.h>

#include "kvq_rope.cuh"

namespace kvq {

namespace {

constexpr int kRBlock = 256;            // threads per block
constexpr int kRWarps = kRBlock / 32;
constexpr int kSub = 32;                // tokens per sub-tile: one per lane
constexpr int kRChunkMin = 128;         // quantized tokens per split: at least this
constexpr int kRChunkCap = 2048;        // ... and at most this
constexpr int kRBlockFixed = 128;       // a block's fixed work, in token-equivalents

struct RopeArgs {
  Geometry g;
  CachePtrs p;
  const __half *q;
  float *out;
  float scale_log2;        // softmax scale * log2(e): scores in the exp2 domain
  int64_t n_quant, n_resid, n_sink, ring_head;
  int64_t qpos;            // position of the query: the newest token
  int64_t chunk;
  int n_qsplit, n_split, s_max, sc_max;
  float *ws_ml;            // [BH][s_max][RG][2]
  float *ws_o;             // [BH][s_max][RG][D]
  int *ws_cnt;             // [BH]
  float c1, c2, c3;        // 2 pi = c1 + c2 + c3
  float2 theta[kMaxHeadDim / 2];  // theta_i = hi + lo
};

// Shared-memory layout in floats, identical on host and device.
struct RSmem {
  int q, cs, w, z, sc, misc, total;
};

__host__ __device__ inline RSmem rope_smem(int D, int RG, int NGS, int sc_max) {
  RSmem s;
  const int P = D / 2;
  const int TL = kRBlock / (D / 8);
  const int wf = kRWarps * NGS * RG * P * 4;   // float4 per-pair weights, per warp
  const int zf = kRWarps * NGS * RG * P * 2;   // float2 zero terms
  int region = wf + zf;
  if (TL * RG * D > region) region = TL * RG * D;  // the value reduction reuses it
  s.q = 0;
  s.cs = s.q + RG * D;            // float2 [P][kSub]
  s.w = s.cs + P * kSub * 2;
  s.z = s.w + wf;
  s.sc = s.w + region;            // [RG][sc_max]
  s.misc = s.sc + RG * sc_max;
  s.total = s.misc + 8 * RG + 64;
  return s;
}

// cos and sin of delta * theta (delta a non-negative integer below 2^24).
__device__ __forceinline__ float2 rope_cs(float delta, float2 th, const RopeArgs &a) {
  return rope_cos_sin(delta, th, a.c1, a.c2, a.c3);
}

// x < 2^16: its value as a float, exactly.
__device__ __forceinline__ float small_uint_to_float(uint32_t x) {
  return __uint_as_float(0x4B000000u | x) - 8388608.0f;
}

template <int RG>
__device__ __forceinline__ void block_reduce(float (&v)[RG], bool is_max, float *scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int h = 0; h < RG; ++h) {
    float x = v[h];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, x, off);
      x = is_max ? fmaxf(x, o) : x + o;
    }
    if (lane == 0) scratch[h * kRWarps + wid] = x;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < RG; ++h) {
    float x = scratch[h * kRWarps];
#pragma unroll
    for (int w = 1; w < kRWarps; ++w)
      x = is_max ? fmaxf(x, scratch[h * kRWarps + w]) : x + scratch[h * kRWarps + w];
    v[h] = x;
  }
  __syncthreads();
}

// One query head per KV head (KIVI): registers capped so five blocks fit an SM.
template <int RG, int SCHEME>
constexpr int rope_min_blocks() { return (RG == 1 && SCHEME == KVQ_KIVI) ? 5 : 1; }

template <int D, int BITS, int RG, int SCHEME>
__global__ void __launch_bounds__(kRBlock, rope_min_blocks<RG, SCHEME>())
    rope_decode_kernel(const RopeArgs a) {
  extern __shared__ float4 smem4[];
  float *smem = reinterpret_cast<float *>(smem4);
  constexpr int P = D / 2;              // channel pairs
  constexpr int NW = D * BITS / 32;     // 32-bit code words per token row
  constexpr int CH = D / 8;             // 8-channel chunks per row (value pass)
  constexpr int TL = kRBlock / CH;      // token lanes of the value pass
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  const Geometry &g = a.g;
  const int NGS = (SCHEME == KVQ_KIVI && g.k_group < kSub) ? kSub / g.k_group : 1;
  const RSmem L = rope_smem(D, RG, NGS, a.sc_max);
  float *q_s = smem + L.q, *sc = smem + L.sc, *misc = smem + L.misc;
  float2 *cs = reinterpret_cast<float2 *>(smem + L.cs);
  float4 *w_s = reinterpret_cast<float4 *>(smem + L.w);
  float2 *z_s = reinterpret_cast<float2 *>(smem + L.z);
  float *u_s = smem + L.w;

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int split = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / g.H), h = (int)(bh % g.H);
  const bool fp16_split = split == a.n_qsplit;

  for (int i = tid; i < RG * D; i += kRBlock) {
    const int hq = h * RG + i / D;
    q_s[i] = __half2float(a.q[((int64_t)b * g.Hq + hq) * D + i % D]) * a.scale_log2;
  }
  if (!fp16_split)
    for (int i = tid; i < P * kSub; i += kRBlock) cs[i] = rope_cs((float)(i % kSub), a.theta[i / kSub], a);

  int64_t t0 = 0, n_tok;
  if (fp16_split) {
    n_tok = a.n_sink + a.n_resid;
  } else {
    t0 = (int64_t)split * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, a.n_quant);
    n_tok = t1 > t0 ? t1 - t0 : 0;
  }
  __syncthreads();

  // ---------------- key pass: scores (exp2 domain) into sc[h][i] ----------
  if (fp16_split) {
    // sinks at positions 0..; residual / window slot r holds the token that
    // arrived k-th among them (KIVI: k = r; InnerQ ring: k = r - ring_head mod W)
    for (int64_t i = tid; i < n_tok; i += kRBlock) {
      const __half *row;
      int64_t pos;
      if (i < a.n_sink) {
        row = a.p.k_sink + (bh * g.n_sink + i) * D;
        pos = i;
      } else {
        const int64_t r = i - a.n_sink;
        row = a.p.k_res + (bh * g.residual + r) * D;
        const int64_t k = SCHEME == KVQ_KIVI ? r : (r - a.ring_head + g.residual) % g.residual;
        pos = a.n_sink + a.n_quant + k;
      }
      const float delta = (float)(a.qpos - pos);
      float s[RG];
#pragma unroll
      for (int hh = 0; hh < RG; ++hh) s[hh] = 0.0f;
#pragma unroll 2
      for (int c8 = 0; c8 < CH; ++c8) {
        const uint4 raw = reinterpret_cast<const uint4 *>(row)[c8];
        const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const int pr = 4 * c8 + k2;
          const float2 kk = __half22float2(hv[k2]);
          const float2 r = rope_cs(delta, a.theta[pr], a);
#pragma unroll
          for (int hh = 0; hh < RG; ++hh) {
            const float qa = q_s[hh * D + 2 * pr], qb = q_s[hh * D + 2 * pr + 1];
            s[hh] += kk.x * (r.x * qa - r.y * qb) + kk.y * (r.y * qa + r.x * qb);  // k . R q
          }
        }
      }
#pragma unroll
      for (int hh = 0; hh < RG; ++hh) sc[hh * a.sc_max + i] = s[hh];
    }
  } else {
    const int n_sub = (int)((n_tok + kSub - 1) / kSub);
    const int64_t pos_base = SCHEME == KVQ_KIVI ? 0 : a.n_sink;  // position of slot 0
    float4 *w_me = w_s + wid * NGS * RG * P;
    float2 *z_me = z_s + wid * NGS * RG * P;
    const int lgk = __ffs(g.k_group) - 1;
    for (int st = wid; st < n_sub; st += kRWarps) {
      const int64_t tb = t0 + (int64_t)st * kSub;
      const float delta0 = (float)(a.qpos - (pos_base + tb));
      // the lane's code row is loaded first, so its latency overlaps the
      // key statistics' and the weights' computation
      const int j = lane;
      const bool live = tb + j < t0 + n_tok;
      uint32_t wd[NW];
      if (live) {
        const uint4 *row = reinterpret_cast<const uint4 *>(code_row(g, a.p, bh, tb + j, 0));
#pragma unroll
        for (int v = 0; v < NW / 4; ++v) {
          const uint4 x = row[v];
          wd[4 * v] = x.x;
          wd[4 * v + 1] = x.y;
          wd[4 * v + 2] = x.z;
          wd[4 * v + 3] = x.w;
        }
      }
      // per-pair weights of the anchor query A = R(delta0) q
#pragma unroll
      for (int pp = 0; pp < (P + 31) / 32; ++pp) {
        const int pr = lane + 32 * pp;
        if (pr < P) {
          const float2 r = rope_cs(delta0, a.theta[pr], a);
          const int oa = (2 * pr * BITS) & 15, ob = oa + BITS;  // offsets in the 16-bit half
          const float fa = __int_as_float((127 - oa) << 23), fb = __int_as_float((127 - ob) << 23);
          float na = 1.0f, nb = 1.0f;
          if (SCHEME == KVQ_INNERQ && g.knorm) {
            na = a.p.k_norm[bh * D + 2 * pr];
            nb = a.p.k_norm[bh * D + 2 * pr + 1];
          }
          for (int gi = 0; gi < NGS; ++gi) {
            float sa = na, sb = nb, za = 0.0f, zb = 0.0f;
            if (SCHEME == KVQ_KIVI) {
              // (fp32 statistics: the options are refused for this kernel)
              const float *km = reinterpret_cast<const float *>(
                  kivi_key_meta(g, a.p, bh, (tb + (int64_t)gi * g.k_group) >> lgk));
              sa = km[2 * pr];
              sb = km[2 * pr + 1];
              za = km[D + 2 * pr];
              zb = km[D + 2 * pr + 1];
            }
#pragma unroll
            for (int hh = 0; hh < RG; ++hh) {
              const float qa = q_s[hh * D + 2 * pr], qb = q_s[hh * D + 2 * pr + 1];
              const float Aa = r.x * qa - r.y * qb, Ab = r.y * qa + r.x * qb;
              w_me[(gi * RG + hh) * P + pr] =
                  make_float4(sa * Aa * fa, sb * Ab * fb, sa * Ab * fa, -(sb * Aa) * fb);
              // KIVI: the zeros' terms; InnerQ: the unscaled pair sums (times z_j later)
              z_me[(gi * RG + hh) * P + pr] =
                  SCHEME == KVQ_KIVI ? make_float2(za * Aa + zb * Ab, za * Ab - zb * Aa)
                                     : make_float2(sa * Aa + sb * Ab, sa * Ab - sb * Aa);
            }
          }
        }
      }
      __syncwarp();
      if (live) {
        const int64_t t = tb + j;
        const int gi = NGS > 1 ? (j >> lgk) : 0;
        const float4 *wt = w_me + gi * RG * P;
        const float2 *zt = z_me + gi * RG * P;
        const float2 *csj = cs + j;
        float acc[RG];
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) acc[hh] = 0.0f;
        if (SCHEME == KVQ_KIVI) {
#pragma unroll
          for (int pr = 0; pr < P; ++pr) {
            const uint32_t word = wd[(2 * pr * BITS) / 32];
            const uint32_t half = ((2 * pr * BITS) % 32) >= 16 ? word >> 16 : word;
            const int o = (2 * pr * BITS) & 15;
            const float ua = small_uint_to_float(half & (kMask << o));
            const float ub = small_uint_to_float(half & (kMask << (o + BITS)));
            const float2 cj = csj[pr * kSub];
#pragma unroll
            for (int hh = 0; hh < RG; ++hh) {
              const float4 w = wt[hh * P + pr];
              const float2 z = zt[hh * P + pr];
              const float X = fmaf(ua, w.x, fmaf(ub, w.y, z.x));
              const float Y = fmaf(ua, w.z, fmaf(ub, w.w, z.y));
              acc[hh] = fmaf(cj.x, X, fmaf(cj.y, Y, acc[hh]));
            }
          }
        } else {
          const int GK = g.k_group;
          const int ngk = D / GK;
          const float *ks = reinterpret_cast<const float *>(tok_meta(g, a.p, bh, t, g.blk_ks, ngk));
          const float *kz = reinterpret_cast<const float *>(tok_meta(g, a.p, bh, t, g.blk_kz, ngk));
          float accg[RG], zg[RG];
#pragma unroll
          for (int hh = 0; hh < RG; ++hh) accg[hh] = zg[hh] = 0.0f;
          float sj = 0.0f, zj = 0.0f;
#pragma unroll
          for (int pr = 0; pr < P; ++pr) {
            if (((2 * pr) & (GK - 1)) == 0) {
              sj = ks[(2 * pr) >> lgk];
              zj = kz[(2 * pr) >> lgk];
            }
            const uint32_t word = wd[(2 * pr * BITS) / 32];
            const uint32_t half = ((2 * pr * BITS) % 32) >= 16 ? word >> 16 : word;
            const int o = (2 * pr * BITS) & 15;
            const float ua = small_uint_to_float(half & (kMask << o));
            const float ub = small_uint_to_float(half & (kMask << (o + BITS)));
            const float2 cj = csj[pr * kSub];
#pragma unroll
            for (int hh = 0; hh < RG; ++hh) {
              const float4 w = wt[hh * P + pr];
              const float2 z = zt[hh * P + pr];
              const float X = fmaf(ua, w.x, ub * w.y);
              const float Y = fmaf(ua, w.z, ub * w.w);
              accg[hh] = fmaf(cj.x, X, fmaf(cj.y, Y, accg[hh]));
              zg[hh] = fmaf(cj.x, z.x, fmaf(cj.y, z.y, zg[hh]));
            }
            if (((2 * pr + 2) & (GK - 1)) == 0) {
#pragma unroll
              for (int hh = 0; hh < RG; ++hh) {
                acc[hh] = fmaf(sj, accg[hh], fmaf(zj, zg[hh], acc[hh]));
                accg[hh] = zg[hh] = 0.0f;
              }
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) sc[hh * a.sc_max + (t - t0)] = acc[hh];
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // ---------------- softmax statistics of this split ----------------------
  float m[RG], l[RG];
#pragma unroll
  for (int hh = 0; hh < RG; ++hh) m[hh] = -INFINITY;
  for (int64_t i = tid; i < n_tok; i += kRBlock)
#pragma unroll
    for (int hh = 0; hh < RG; ++hh) m[hh] = fmaxf(m[hh], sc[hh * a.sc_max + i]);
  block_reduce<RG>(m, true, misc);
#pragma unroll
  for (int hh = 0; hh < RG; ++hh) l[hh] = 0.0f;
  for (int64_t i = tid; i < n_tok; i += kRBlock)
#pragma unroll
    for (int hh = 0; hh < RG; ++hh) {
      const float pv = exp2f(sc[hh * a.sc_max + i] - m[hh]);
      sc[hh * a.sc_max + i] = pv;
      l[hh] += pv;
    }
  block_reduce<RG>(l, false, misc);

  // ---------------- value pass: o[h][c] = sum_t p_t v_hat_tc ---------------
  const int jc = tid % CH, tl = tid / CH;
  float acc[RG][8], zacc[RG];
#pragma unroll
  for (int hh = 0; hh < RG; ++hh) {
    zacc[hh] = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[hh][k] = 0.0f;
  }
  if (fp16_split) {
    for (int64_t i = tl; i < n_tok; i += TL) {
      const __half *row = i < a.n_sink ? a.p.v_sink + (bh * g.n_sink + i) * D
                                       : a.p.v_res + (bh * g.residual + (i - a.n_sink)) * D;
      const uint4 raw = reinterpret_cast<const uint4 *>(row)[jc];
      const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
      for (int hh = 0; hh < RG; ++hh) {
        const float pv = sc[hh * a.sc_max + i];
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const float2 f = __half22float2(hv[k2]);
          acc[hh][2 * k2] += pv * f.x;
          acc[hh][2 * k2 + 1] += pv * f.y;
        }
      }
    }
  } else {
    // Codes stay in place in their 16-bit half: acc[h][k] collects
    // p * scale * (code << offset_k), and the power of two comes out once at
    // the end.  Split starts are multiples of the 32-token block.
    const int ngv = D / g.v_group;
    const int gv = (8 * jc) / g.v_group;
    for (int64_t bt = 0; bt < n_tok; bt += kBlockTokens) {
      const uint8_t *blk = tok_block(g, a.p, bh, t0 + bt);
      const uint8_t *vrow = blk + g.blk_vc;
      const float *vsr = reinterpret_cast<const float *>(blk + g.blk_vs);
      const float *vzr = reinterpret_cast<const float *>(blk + g.blk_vz);
      for (int r = tl; r < kBlockTokens; r += TL) {
        if (bt + r >= n_tok) break;
        const uint8_t *row = vrow + r * g.row_bytes;
        const uint32_t word = BITS == 2 ? (uint32_t)reinterpret_cast<const uint16_t *>(row)[jc]
                                        : reinterpret_cast<const uint32_t *>(row)[jc];
        const float vs = vsr[r * ngv + gv];
        const float vz = vzr[r * ngv + gv];
        float cv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t half = (k * BITS) >= 16 ? word >> 16 : word;
          cv[k] = small_uint_to_float(half & (kMask << ((k * BITS) & 15)));
        }
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) {
          const float pv = sc[hh * a.sc_max + bt + r];
          const float ps = pv * vs;
          zacc[hh] = fmaf(pv, vz, zacc[hh]);
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[hh][k] = fmaf(ps, cv[k], acc[hh][k]);
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < RG; ++hh)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[hh][k] *= __int_as_float((127 - ((k * BITS) & 15)) << 23);
  }
  // reduce the TL token lanes through shared memory (the weights are dead)
  __syncthreads();
#pragma unroll
  for (int hh = 0; hh < RG; ++hh)
#pragma unroll
    for (int k = 0; k < 8; ++k) u_s[(tl * RG + hh) * D + 8 * jc + k] = acc[hh][k] + zacc[hh];
  __syncthreads();

  const int64_t part = bh * a.s_max + split;
  for (int i = tid; i < RG * D; i += kRBlock) {
    const int hh = i / D, c = i % D;
    float s = 0.0f;
    for (int r = 0; r < TL; ++r) s += u_s[(r * RG + hh) * D + c];
    a.ws_o[(part * RG + hh) * D + c] = s;
  }
  if (tid < RG) {
    float mv = m[0], lv = l[0];
#pragma unroll
    for (int hh = 0; hh < RG; ++hh)
      if (hh == tid) {
        mv = m[hh];
        lv = l[hh];
      }
    a.ws_ml[(part * RG + tid) * 2 + 0] = n_tok > 0 ? mv : -INFINITY;
    a.ws_ml[(part * RG + tid) * 2 + 1] = n_tok > 0 ? lv : 0.0f;
  }

  // ---------------- the last block of the head merges the splits ----------
  __threadfence();
  __syncthreads();
  int *flag = reinterpret_cast<int *>(misc);
  if (tid == 0) {
    const int prev = atomicAdd(&a.ws_cnt[bh], 1);
    flag[0] = prev == a.n_split - 1;
  }
  __syncthreads();
  if (!flag[0]) return;
  __threadfence();
  for (int i = tid; i < RG * D; i += kRBlock) {
    const int hh = i / D, c = i % D;
    float M = -INFINITY;
    for (int sp = 0; sp < a.n_split; ++sp)
      M = fmaxf(M, __ldcg(&a.ws_ml[((bh * a.s_max + sp) * RG + hh) * 2]));
    float Lsum = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < a.n_split; ++sp) {
        const int64_t pi = (bh * a.s_max + sp) * RG + hh;
        const float ms = __ldcg(&a.ws_ml[pi * 2]);
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        Lsum += w * __ldcg(&a.ws_ml[pi * 2 + 1]);
        O += w * __ldcg(&a.ws_o[pi * D + c]);
      }
    }
    a.out[((int64_t)b * g.Hq + h * RG + hh) * D + c] = Lsum > 0.0f ? O / Lsum : 0.0f;
  }
  // leave the workspace zero, as every decode path expects it
  __syncthreads();
  const int64_t p0 = (int64_t)bh * a.s_max * RG;
  for (int i = tid; i < a.n_split * RG * D; i += kRBlock) a.ws_o[p0 * D + i] = 0.0f;
  for (int i = tid; i < a.n_split * RG * 2; i += kRBlock) a.ws_ml[p0 * 2 + i] = 0.0f;
  if (tid == 0) atomicExch(&a.ws_cnt[bh], 0);  // an atomic, like the tickets it resets
}

// Splits over the quantized tokens, plus the fp16 split.  A split's block
// costs about its tokens plus a fixed part (kRBlockFixed token-equivalents:
// the cos / sin table, the reductions, the partial row); blocks run in waves
// of per_sm * num_sms, so the plan minimises waves * (chunk + fixed) over the
// number of splits.  chunk: a multiple of 32 tokens (sub-tiles and blocks
// start aligned), at least kRChunkMin (the partial slots per head suffice),
// at most kRChunkCap (the score buffer).
void plan_rope(RopeArgs &a, int per_sm, int num_sms) {
  const int64_t BH = (int64_t)a.g.B * a.g.H;
  const int64_t slots = (int64_t)per_sm * num_sms;
  int64_t chunk = kRChunkMin, best = -1;
  const int64_t s0 = (a.n_quant + kRChunkCap - 1) / kRChunkCap;
  for (int64_t s = s0 > 0 ? s0 : 1; s < s0 + 64; ++s) {
    int64_t c = (a.n_quant + s - 1) / s;
    c = (c + kSub - 1) / kSub * kSub;
    if (c < kRChunkMin) c = kRChunkMin;
    if (c > kRChunkCap) continue;
    const int64_t ns = (a.n_quant + c - 1) / c;
    const int64_t cost = ((BH * ns + slots - 1) / slots) * (c + kRBlockFixed);
    if (best < 0 || cost < best) {
      best = cost;
      chunk = c;
    }
  }
  a.chunk = chunk;
  a.n_qsplit = (int)((a.n_quant + chunk - 1) / chunk);
  a.n_split = a.n_qsplit + (a.n_resid + a.n_sink > 0 ? 1 : 0);
  if (a.n_split == 0) a.n_split = 1;  // empty cache: one empty split writes zeros
}

template <int D, int BITS, int RG, int SCHEME>
cudaError_t launch_t(RopeArgs a, int smem_bytes, int num_sms, cudaStream_t st) {
  static KernelSetup setup;
  int per_sm = 1;
  const cudaError_t e =
      kernel_setup(setup, rope_decode_kernel<D, BITS, RG, SCHEME>, kRBlock, smem_bytes, &per_sm);
  if (e != cudaSuccess) return e;
  plan_rope(a, per_sm, num_sms);
  rope_decode_kernel<D, BITS, RG, SCHEME>
      <<<dim3((unsigned)a.n_split, (unsigned)(a.g.B * a.g.H)), kRBlock, smem_bytes, st>>>(a);
  return cudaGetLastError();
}

template <int D, int BITS, int RG>
cudaError_t launch_s(const RopeArgs &a, int smem, int num_sms, cudaStream_t st) {
  return a.g.scheme == KVQ_KIVI ? launch_t<D, BITS, RG, KVQ_KIVI>(a, smem, num_sms, st)
                                : launch_t<D, BITS, RG, KVQ_INNERQ>(a, smem, num_sms, st);
}

template <int D, int BITS>
cudaError_t launch_r(const RopeArgs &a, int rg, int smem, int num_sms, cudaStream_t st) {
  switch (rg) {
    case 1: return launch_s<D, BITS, 1>(a, smem, num_sms, st);
    case 2: return launch_s<D, BITS, 2>(a, smem, num_sms, st);
    case 4: return launch_s<D, BITS, 4>(a, smem, num_sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_rope(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                               int64_t n_resid, int64_t n_sink, int64_t ring_head,
                               const __half *q, float *out, float scale, double rope_base,
                               void *ws, int num_sms, cudaStream_t st) {
  const int rg = g.Hq / g.H;
  if (!rope_group_supported(rg)) return cudaErrorInvalidValue;
  RopeArgs a;
  a.g = g;
  a.p = p;
  a.q = q;
  a.out = out;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_quant = n_quant;
  a.n_resid = n_resid;
  a.n_sink = n_sink;
  a.ring_head = ring_head;
  a.qpos = n_sink + n_quant + n_resid - 1;
  const int64_t BH = (int64_t)g.B * g.H;
  a.s_max = part_slots(g);
  a.sc_max = kRChunkCap > g.residual + g.n_sink ? kRChunkCap : g.residual + g.n_sink;
  // theta_i = base^(-2i/d) as hi + lo; 2 pi in three parts
  rope_constants(rope_base, g.d, a.theta, a.c1, a.c2, a.c3);
  // workspace: counters, then (m, l) and o rows (the general decode layout)
  const int64_t parts = BH * a.s_max * rg;
  char *base = static_cast<char *>(ws);
  const size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  a.ws_cnt = reinterpret_cast<int *>(base);
  a.ws_ml = reinterpret_cast<float *>(base + cnt);
  a.ws_o = a.ws_ml + parts * 2;
  const int ngs = (g.scheme == KVQ_KIVI && g.k_group < kSub) ? kSub / g.k_group : 1;
  const int smem = rope_smem(g.d, rg, ngs, a.sc_max).total * (int)sizeof(float);
  if (g.d == 64) return g.bits == 2 ? launch_r<64, 2>(a, rg, smem, num_sms, st)
                                    : launch_r<64, 4>(a, rg, smem, num_sms, st);
  return g.bits == 2 ? launch_r<128, 2>(a, rg, smem, num_sms, st)
                     : launch_r<128, 4>(a, rg, smem, num_sms, st);
}

}  // namespace kvq
