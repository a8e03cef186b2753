// Fused decode attention over the packed cache (split-K over tokens, one
// launch, in-kernel merge by the last block of each head).
//
// Method: every decode step reads the whole cache ("大模型量化技术原理：KIVI、
// IntactKV、KVQuant", KIVI / 背景), so the kernel streams the packed codes with
// their scale / zero once and never materialises a dequantized K or V.  The
// dequantization is folded into the two GEMVs (InnerQ page, 方法论 3: one
// shared scale per group, loaded once and reused):
//   KIVI keys (per channel c, G-token group g):
//     s_t = sum_c (q_c s_gc) u_tc + sum_c q_c z_gc       -- q~ and the bias once per group
//   per-token groups j (KIVI values, InnerQ keys and values):
//     s_t = sum_j s_tj (sum_{c in j} q_c u_tc) + sum_j z_tj Q_j,   Q_j = sum_{c in j} q_c
//     o_c = sum_t (p_t s_tj) u_tc + sum_t p_t z_tj
// The fp16 sink / residual / window tokens form one more split; every split
// leaves (m, l, o) and the last block of the head merges them with the
// log-sum-exp rule (the fp16 part joins the dequantized part, IntactKV /
// KV Cache量化 on the same page).
#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kBlock = 256;
constexpr int kTile = 256;  // tokens per key tile (one thread per token)
constexpr int kMinKeyGroup = 16;

struct DecodeArgs {
  Geometry g;
  CachePtrs p;
  const __half *q;
  float *out;
  float scale_log2;  // softmax_scale * log2(e): scores live in the exp2 domain
  Counts cnt;        // counters (the longest sequence's under KVQ_RAGGED)
  int64_t chunk;
  int n_qsplit, n_split, s_max;
  int sc_max;        // score slots per head in shared memory
  float *ws_ml;      // [BH][s_max][RG][2]
  float *ws_o;       // [BH][s_max][RG][D]
  int *ws_cnt;       // [BH]
};

// Shared-memory layout (floats), identical on host and device.
struct Smem {
  int q, qj, bias, sc, u, misc, total;
};

__host__ __device__ inline Smem smem_layout(int D, int RG, int sc_max, int ngk) {
  Smem s;
  const int TL = kBlock / (D / 8);
  const int ngt = kTile / kMinKeyGroup;
  int a_floats = ngt * RG * D;
  const int red_floats = TL * RG * D;
  if (red_floats > a_floats) a_floats = red_floats;
  s.q = 0;
  s.qj = s.q + RG * D;
  s.bias = s.qj + RG * ngk;
  s.sc = s.bias + ngt * RG;
  s.u = s.sc + RG * sc_max;
  s.misc = s.u + a_floats;
  s.total = s.misc + 4 * RG + 64;
  return s;
}

template <int BITS>
__device__ __forceinline__ float code_at(uint32_t word, int k) {
  return (float)((word >> (k * BITS)) & ((1u << BITS) - 1u));
}

// Block-wide max and sum for RG values per thread; results broadcast.
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
    if (lane == 0) scratch[h * 8 + wid] = x;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < RG; ++h) {
    float x = scratch[h * 8];
#pragma unroll
    for (int w = 1; w < kBlock / 32; ++w) x = is_max ? fmaxf(x, scratch[h * 8 + w]) : x + scratch[h * 8 + w];
    v[h] = x;
  }
  __syncthreads();
}

template <int D, int BITS, int RG, int SCHEME>
__global__ void __launch_bounds__(kBlock) decode_kernel(const DecodeArgs a) {
  extern __shared__ float smem[];
  constexpr int NW = D * BITS / 32;  // 32-bit code words per token row
  constexpr int CPW = 32 / BITS;     // codes per word
  constexpr int CH = D / 8;          // 8-channel chunks per row
  constexpr int TL = kBlock / CH;    // token lanes in the value pass
  const Geometry &g = a.g;
  const int ngk = SCHEME == KVQ_KIVI ? 1 : D / g.k_group;
  const Smem L = smem_layout(D, RG, a.sc_max, ngk);
  float *q_s = smem + L.q, *qj_s = smem + L.qj, *bias_s = smem + L.bias;
  float *sc = smem + L.sc, *u_s = smem + L.u, *misc = smem + L.misc;

  const int tid = threadIdx.x;
  const int split = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / g.H), h = (int)(bh % g.H);
  const Counts cn = seq_counts(g, a.p, a.cnt, b);  // this sequence's counters

  const bool fp16_split = split == a.n_qsplit;
  for (int i = tid; i < RG * D; i += kBlock) {
    const int hq = h * RG + i / D;
    q_s[i] = __half2float(a.q[((int64_t)b * g.Hq + hq) * D + i % D]) * a.scale_log2;
    // quantized keys are normalized per channel: the factor goes into q
    if (SCHEME == KVQ_INNERQ && g.knorm && !fp16_split) q_s[i] *= a.p.k_norm[bh * D + i % D];
  }
  __syncthreads();
  if (SCHEME == KVQ_INNERQ) {
    for (int i = tid; i < RG * ngk; i += kBlock) {
      const int hh = i / ngk, j = i % ngk;
      float s = 0.0f;
      for (int c = j * g.k_group; c < (j + 1) * g.k_group; ++c) s += q_s[hh * D + c];
      qj_s[i] = s;
    }
  }

  int64_t t0 = 0, n_tok;
  if (fp16_split) {
    n_tok = cn.n_sink + cn.n_resid;
  } else {
    t0 = (int64_t)split * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, cn.n_quant);
    n_tok = t1 > t0 ? t1 - t0 : 0;
  }
  __syncthreads();

  // ---------------- key pass: scores (exp2 domain) into sc[h][i] ----------
  if (fp16_split) {
    for (int64_t i = tid; i < n_tok; i += kBlock) {
      const __half *row = i < cn.n_sink ? a.p.k_sink + (bh * g.n_sink + i) * D
                                        : a.p.k_res + (bh * g.residual + (i - cn.n_sink)) * D;
      float s[RG] = {};
#pragma unroll 4
      for (int c8 = 0; c8 < CH; ++c8) {
        const uint4 raw = reinterpret_cast<const uint4 *>(row)[c8];
        const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const float2 f = __half22float2(hv[k2]);
#pragma unroll
          for (int hh = 0; hh < RG; ++hh)
            s[hh] += q_s[hh * D + 8 * c8 + 2 * k2] * f.x + q_s[hh * D + 8 * c8 + 2 * k2 + 1] * f.y;
        }
      }
#pragma unroll
      for (int hh = 0; hh < RG; ++hh) sc[hh * a.sc_max + i] = s[hh];
    }
  } else if (SCHEME == KVQ_KIVI) {
    const int G = g.k_group;
    for (int64_t tt = 0; tt < n_tok; tt += kTile) {
      const int ngt = kTile / G;
      // q~ = q * scale and bias = q . zero for the groups of this tile
      const int64_t g0 = (t0 + tt) / G;
      const int ng_here = (int)min((int64_t)ngt, (n_tok - tt + G - 1) / G);
      for (int i = tid; i < ng_here * D; i += kBlock) {
        const int gl = i / D, c = i % D;
        const float sk = ld_meta(g, kivi_key_meta(g, a.p, bh, g0 + gl), c);
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) u_s[(gl * RG + hh) * D + c] = q_s[hh * D + c] * sk;
      }
      const int lane = tid & 31, wid = tid >> 5;
      for (int pr = wid; pr < ng_here * RG; pr += kBlock / 32) {
        const int gl = pr / RG, hh = pr % RG;
        const uint8_t *zr = kivi_key_meta(g, a.p, bh, g0 + gl) + D * g.msz;
        float s = 0.0f;
        for (int c = lane; c < D; c += 32) s += q_s[hh * D + c] * ld_meta(g, zr, c);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) bias_s[pr] = s;
      }
      __syncthreads();
      const int64_t i = tt + tid;
      if (i < n_tok) {
        const int gl = tid / G;
        const uint4 *row = reinterpret_cast<const uint4 *>(code_row(g, a.p, bh, t0 + i, 0));
        float s[RG];
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) s[hh] = bias_s[gl * RG + hh];
#pragma unroll
        for (int w4 = 0; w4 < NW / 4; ++w4) {
          const uint4 v = row[w4];
          const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
            for (int k = 0; k < CPW; ++k) {
              const float u = code_at<BITS>(words[wi], k);
              const int c = (w4 * 4 + wi) * CPW + k;
#pragma unroll
              for (int hh = 0; hh < RG; ++hh) s[hh] += u_s[(gl * RG + hh) * D + c] * u;
            }
          }
        }
        if (g.n_out > 0) {
          // dense-and-sparse: an outlier's code is 0, so the dense sum holds
          // q_c * zero there; its fp16 value replaces it
          const int64_t t = t0 + i;
          const uint32_t *ol = tok_outliers(g, a.p, bh, t, g.blk_ko);
          const uint8_t *zr = kivi_key_meta(g, a.p, bh, t / G) + D * g.msz;
          for (int e = 0; e < g.n_out; ++e) {
            const uint32_t w = ol[e];
            const int c = (int)(w >> 16);
            const float dv = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))) -
                             ld_meta(g, zr, c);
#pragma unroll
            for (int hh = 0; hh < RG; ++hh) s[hh] += q_s[hh * D + c] * dv;
          }
        }
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) sc[hh * a.sc_max + i] = s[hh];
      }
      __syncthreads();
    }
  } else {  // InnerQ keys: per-token groups of k_group channels
    const int GK = g.k_group;
    for (int64_t i = tid; i < n_tok; i += kBlock) {
      const int64_t t = t0 + i;
      const uint32_t *row = reinterpret_cast<const uint32_t *>(code_row(g, a.p, bh, t, 0));
      const uint8_t *ks = tok_meta(g, a.p, bh, t, g.blk_ks, ngk);
      const uint8_t *kz = tok_meta(g, a.p, bh, t, g.blk_kz, ngk);
      float s[RG] = {};
      for (int j = 0; j < ngk; ++j) {
        float part[RG] = {};
        for (int w = j * GK / CPW; w < (j + 1) * GK / CPW; ++w) {
          const uint32_t word = row[w];
#pragma unroll
          for (int k = 0; k < CPW; ++k) {
            const float u = code_at<BITS>(word, k);
#pragma unroll
            for (int hh = 0; hh < RG; ++hh) part[hh] += q_s[hh * D + w * CPW + k] * u;
          }
        }
        const float sj = ld_meta(g, ks, j), zj = ld_meta(g, kz, j);
#pragma unroll
        for (int hh = 0; hh < RG; ++hh) s[hh] += sj * part[hh] + zj * qj_s[hh * ngk + j];
      }
#pragma unroll
      for (int hh = 0; hh < RG; ++hh) sc[hh * a.sc_max + i] = s[hh];
    }
  }
  __syncthreads();

  // ---------------- softmax statistics of this split ----------------------
  float m[RG], l[RG];
#pragma unroll
  for (int hh = 0; hh < RG; ++hh) m[hh] = -INFINITY;
  for (int64_t i = tid; i < n_tok; i += kBlock)
#pragma unroll
    for (int hh = 0; hh < RG; ++hh) m[hh] = fmaxf(m[hh], sc[hh * a.sc_max + i]);
  block_reduce<RG>(m, true, misc);
#pragma unroll
  for (int hh = 0; hh < RG; ++hh) l[hh] = 0.0f;
  for (int64_t i = tid; i < n_tok; i += kBlock)
#pragma unroll
    for (int hh = 0; hh < RG; ++hh) {
      const float pv = exp2f(sc[hh * a.sc_max + i] - m[hh]);
      sc[hh * a.sc_max + i] = pv;
      l[hh] += pv;
    }
  block_reduce<RG>(l, false, misc);

  // ---------------- value pass: o[h][c] = sum_t p_t v_hat_tc ---------------
  const int j = tid % CH, tl = tid / CH;
  float acc[RG][8], zacc[RG];
#pragma unroll
  for (int hh = 0; hh < RG; ++hh) {
    zacc[hh] = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[hh][k] = 0.0f;
  }
  if (fp16_split) {
    for (int64_t i = tl; i < n_tok; i += TL) {
      // (value queue: the residual token n_quant + r sits in ring slot r)
      const __half *row = i < cn.n_sink ? a.p.v_sink + (bh * g.n_sink + i) * D
                                        : a.p.v_res + (bh * g.residual + (i - cn.n_sink)) * D;
      const uint4 raw = reinterpret_cast<const uint4 *>(row)[j];
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
    const int ngv = D / g.v_group;
    const int gv = (8 * j) / g.v_group;
    for (int64_t i = tl; i < n_tok; i += TL) {
      const int64_t t = t0 + i;
      if (t >= cn.n_vq) {
        // value queue: the token's key is quantized, its value still fp16 in
        // ring slot t mod R
        const uint4 raw = reinterpret_cast<const uint4 *>(
            a.p.v_res + (bh * g.residual + t % g.residual) * D)[j];
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
        continue;
      }
      const uint8_t *row = code_row(g, a.p, bh, t, g.blk_vc);
      const uint32_t word = BITS == 2 ? (uint32_t)reinterpret_cast<const uint16_t *>(row)[j]
                                      : reinterpret_cast<const uint32_t *>(row)[j];
      const float vs = ld_meta(g, tok_meta(g, a.p, bh, t, g.blk_vs, ngv), gv);
      const float vz = ld_meta(g, tok_meta(g, a.p, bh, t, g.blk_vz, ngv), gv);
#pragma unroll
      for (int hh = 0; hh < RG; ++hh) {
        const float pv = sc[hh * a.sc_max + i];
        const float ps = pv * vs;
        zacc[hh] += pv * vz;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[hh][k] += ps * code_at<BITS>(word, k);
      }
      if (g.n_out > 0) {
        // this chunk's outliers: code 0 gave p * zero, the fp16 value replaces it
        const uint32_t *ol = tok_outliers(g, a.p, bh, t, g.blk_vo);
        for (int e = 0; e < g.n_out; ++e) {
          const uint32_t w = ol[e];
          const int c = (int)(w >> 16);
          if ((c >> 3) != j) continue;
          const float dv = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))) - vz;
#pragma unroll
          for (int hh = 0; hh < RG; ++hh)
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (k == (c & 7)) acc[hh][k] += sc[hh * a.sc_max + i] * dv;
        }
      }
    }
  }
  // reduce the TL token lanes through shared memory
#pragma unroll
  for (int hh = 0; hh < RG; ++hh)
#pragma unroll
    for (int k = 0; k < 8; ++k) u_s[(tl * RG + hh) * D + 8 * j + k] = acc[hh][k] + zacc[hh];
  __syncthreads();

  const int64_t part = bh * a.s_max + split;
  for (int i = tid; i < RG * D; i += kBlock) {
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

  // ---------------- last block of the head merges the splits --------------
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
  for (int i = tid; i < RG * D; i += kBlock) {
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
  // leave the workspace zero, as the tensor-core path expects it
  __syncthreads();
  const int64_t p0 = (int64_t)bh * a.s_max * RG;
  for (int i = tid; i < a.n_split * RG * D; i += kBlock) a.ws_o[p0 * D + i] = 0.0f;
  for (int i = tid; i < a.n_split * RG * 2; i += kBlock) a.ws_ml[p0 * 2 + i] = 0.0f;
  if (tid == 0) atomicExch(&a.ws_cnt[bh], 0);  // an atomic, like the tickets it resets
}

template <int D, int BITS, int RG, int SCHEME>
cudaError_t launch_t(const DecodeArgs &a, int smem_bytes, cudaStream_t st) {
  static KernelSetup setup;
  const cudaError_t e = kernel_setup(setup, decode_kernel<D, BITS, RG, SCHEME>, kBlock, smem_bytes,
                                     nullptr);
  if (e != cudaSuccess) return e;
  decode_kernel<D, BITS, RG, SCHEME>
      <<<dim3((unsigned)a.n_split, (unsigned)(a.g.B * a.g.H)), kBlock, smem_bytes, st>>>(a);
  return cudaGetLastError();
}

template <int D, int BITS, int RG>
cudaError_t launch_s(const DecodeArgs &a, int smem, cudaStream_t st) {
  return a.g.scheme == KVQ_KIVI ? launch_t<D, BITS, RG, KVQ_KIVI>(a, smem, st)
                                : launch_t<D, BITS, RG, KVQ_INNERQ>(a, smem, st);
}

template <int D, int BITS>
cudaError_t launch_r(const DecodeArgs &a, int rg, int smem, cudaStream_t st) {
  switch (rg) {
    case 1: return launch_s<D, BITS, 1>(a, smem, st);
    case 2: return launch_s<D, BITS, 2>(a, smem, st);
    case 4: return launch_s<D, BITS, 4>(a, smem, st);
    case 8: return launch_s<D, BITS, 8>(a, smem, st);
  }
  return cudaErrorInvalidValue;
}

int chunk_cap(int rg) { return rg <= 4 ? 2048 : 1024; }

int64_t fp16_cap(const Geometry &g) { return (int64_t)g.residual + g.n_sink; }

int sc_slots(const Geometry &g) {
  const int rg = g.Hq / g.H;
  int64_t s = chunk_cap(rg);
  if (fp16_cap(g) > s) s = fp16_cap(g);
  return (int)s;
}

int s_max_of(const Geometry &g) { return part_slots(g); }

}  // namespace

size_t decode_workspace_bytes(const Geometry &g) {
  // the larger of the two decode paths' partial arrays
  const int64_t BH = (int64_t)g.B * g.H, rg = g.Hq / g.H;
  int64_t parts = BH * s_max_of(g) * rg;
  const int64_t tc_parts = BH * tc_part_slots(g) * rg;  // the grouped-query kernel: rg rows a slot
  if (tc_parts > parts) parts = tc_parts;
  size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  return cnt + (size_t)parts * 2 * sizeof(float) + (size_t)parts * g.d * sizeof(float) + 256;
}

DecodePlan plan_decode(const Geometry &g, int64_t n_quant, int64_t n_fp16, int num_sms) {
  DecodePlan pl;
  const int64_t BH = (int64_t)g.B * g.H;
  const int rg = g.Hq / g.H;
  int64_t want = (3LL * num_sms + BH - 1) / BH;
  if (want < 1) want = 1;
  int64_t chunk = (n_quant + want - 1) / want;
  chunk = (chunk + kTile - 1) / kTile * kTile;
  if (chunk < kTile) chunk = kTile;
  if (chunk > chunk_cap(rg)) chunk = chunk_cap(rg);
  pl.chunk = chunk;
  pl.n_qsplit = (int)((n_quant + chunk - 1) / chunk);
  pl.n_split = pl.n_qsplit + (n_fp16 > 0 ? 1 : 0);
  if (pl.n_split == 0) pl.n_split = 1;  // empty cache: one empty split writes zeros
  return pl;
}

cudaError_t launch_decode(const Geometry &g, const CachePtrs &p, const DecodePlan &plan,
                          const Counts &c, const __half *q, float *out, float scale, void *ws,
                          int num_sms, cudaStream_t st) {
  // (attention does not depend on the order of window tokens: no ring_head)
  if (c.n_quant > 0 && tc_decode_supported(g))
    return launch_decode_tc(g, p, c.n_quant, c.n_resid, c.n_sink, q, out, scale, ws, num_sms, st);
  if (c.n_quant > 0 && gqa_decode_supported(g))
    return launch_decode_gqa(g, p, c.n_quant, c.n_resid, c.n_sink, q, out, scale, ws, num_sms,
                             st);
  DecodeArgs a;
  a.g = g;
  a.p = p;
  a.q = q;
  a.out = out;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.cnt = c;
  a.chunk = plan.chunk;
  a.n_qsplit = plan.n_qsplit;
  a.n_split = plan.n_split;
  a.s_max = s_max_of(g);
  a.sc_max = sc_slots(g);
  const int64_t BH = (int64_t)g.B * g.H, rg = g.Hq / g.H;
  const int64_t parts = BH * a.s_max * rg;
  char *base = static_cast<char *>(ws);
  size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  a.ws_cnt = reinterpret_cast<int *>(base);
  a.ws_ml = reinterpret_cast<float *>(base + cnt);
  a.ws_o = a.ws_ml + parts * 2;
  const int ngk = g.scheme == KVQ_KIVI ? 1 : g.d / g.k_group;
  const int smem = smem_layout(g.d, (int)rg, a.sc_max, ngk).total * (int)sizeof(float);
  if (g.d == 64) return g.bits == 2 ? launch_r<64, 2>(a, (int)rg, smem, st)
                                    : launch_r<64, 4>(a, (int)rg, smem, st);
  return g.bits == 2 ? launch_r<128, 2>(a, (int)rg, smem, st)
                     : launch_r<128, 4>(a, (int)rg, smem, st);
}

}  // namespace kvq
