// Fused decode attention on the tensor cores (MHA, head_dim 128).
//
// Same computation as decode_kernel (softmax(scale * q.K^T) V over the packed
// cache, dequantization folded into both GEMVs -- "大模型量化技术原理：KIVI、
// IntactKV、KVQuant", KIVI / 背景; InnerQ page, 方法论 3), arranged for GB300:
//
//  * Persistent, stream-K: the (head, 128-token stage) list of the whole batch,
//    plus one fp16 item per head (sink + residual / window tokens), is cut into
//    equal contiguous ranges, one per resident block.  A head split across
//    blocks leaves one partial (m, l, o) per block; the last block to finish a
//    head (atomic ticket, no spinning) merges them with the log-sum-exp rule.
//  * Each 128-token stage (codes + scale/zero of K and V) is fetched with 1-D
//    cp.async.bulk into a 4-slot shared-memory ring completed on mbarriers.
//    Every wait is bounded; a timeout sets the status word and the block
//    drains its own copies before it returns.
//  * Both GEMVs run as mma.sync m16n8k16 (fp16 in, fp32 accumulate).  2/4-bit
//    codes become exact fp16 integers with one LOP3 per two codes (the code
//    bits are OR-ed into the mantissa of 1024.0) and one HSUB2; the position
//    of a code inside its 16-bit half multiplies it by a power of two that the
//    other operand (or the final output row) divides out exactly.  The channel
//    order inside each MMA is a permutation chosen so a thread consumes whole
//    32-bit code words; the matching operand uses the same permutation.
//      keys   D[token][n] = sum_c code_tc * B[c][n],  B = q~ = q*scale split
//             into fp16 hi + lo (n = hi, lo); KIVI: rebuilt per G-token group,
//             InnerQ: q per channel group j (n = (j, hi/lo)), scale applied after.
//      values D[c][n] = sum_t code_tc * B[t][n],  B = p_t * scale_tj split into
//             hi + lo, n = (value group j, hi/lo); row c keeps column j(c).
//    zero points enter as q.zero per key group and sum_t p_t zero_tj per value
//    group (CUDA cores).  q is normalised by a power of two so no fp16 operand
//    can overflow (|q| <= 1, scales <= 65504).
#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTT = 128;      // tokens per stage (one 16-token MMA tile per warp)
constexpr int kStages = 4;
constexpr int kD = 128;
constexpr int kScrFloats = 4096 + 64;  // fp16 item: 2048 scores + 16x128 reduce
constexpr uint32_t kMagic = 0x64006400u;  // half2(1024, 1024)
constexpr long long kDrainLimit = 1LL << 26;

struct TcArgs {
  Geometry g;
  CachePtrs p;
  const __half *q;
  float *out;
  float scale_log2;
  int64_t n_quant, n_fp16, n_sink;
  int S_h, F_h, U;  // quantized stages, fp16 units, units per head
  int64_t total;    // BH * U
  int nc;           // resident blocks
  int slot_bytes, off_vc, off_ks, off_kz, off_vs, off_vz;
  float *ws_ml, *ws_o;
  int *ws_cnt;
  int part_stride;
  long long wait_limit;   // poll cap of every pipeline wait
  long long stall_limit;  // debug: > 0 = first wait on a barrier nothing completes
};

struct TcLayout {
  int ring, sB, sBias, sQf, sScr, sFlag, bars, total;
};

__host__ __device__ inline TcLayout tc_layout(int slot_bytes) {
  TcLayout L;
  L.ring = 0;
  L.sB = L.ring + kStages * slot_bytes;       // 8 key groups x 128 u32
  L.sBias = L.sB + 8 * 128 * 4;               // [8 groups][2] floats
  L.sQf = L.sBias + 16 * 4;                   // [128] floats
  L.sScr = L.sQf + kD * 4;                    // scratch floats
  L.sFlag = L.sScr + kScrFloats * 4;          // [8] ints / floats
  L.bars = L.sFlag + 8 * 4;                   // kStages mbarriers + 1 never completed
  L.total = L.bars + (kStages + 1) * 8;
  return L;
}

// ---- PTX helpers --------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void bar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void bar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool bar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity, long long limit) {
  for (long long it = 0;; ++it) {
    if (bar_try_wait(bar, parity)) return true;
    if (it >= limit) return false;
  }
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t lop_or_and(uint32_t a, uint32_t mask, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hsub_magic(uint32_t x) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(kMagic));
  return d;
}

// Code pair at position p of a word holding two 16-bit halves of codes:
// returns half2(code_lo * f, code_hi * f) exactly, f = 4^p' / 16^p' below.
// ws = w >> 10 (2-bit) or w >> 8 (4-bit), precomputed by the caller.
template <int BITS>
__device__ __forceinline__ uint32_t ext(uint32_t w, uint32_t ws, int p) {
  if (BITS == 2) {
    return p <= 4 ? hsub_magic(lop_or_and(w, 0x00030003u << (2 * p), kMagic))
                  : hsub_magic(lop_or_and(ws, 0x00030003u << (2 * (p - 5)), kMagic));
  }
  return p <= 1 ? hsub_magic(lop_or_and(w, 0x000F000Fu << (4 * p), kMagic))
                : hsub_magic(lop_or_and(ws, 0x000F000Fu << (4 * (p - 2)), kMagic));
}

template <int BITS>
__device__ __forceinline__ uint32_t shifted(uint32_t w) {
  return BITS == 2 ? (w >> 10) : (w >> 8);
}

// Multiplier carried by the code at position p (see ext).
template <int BITS>
__host__ __device__ __forceinline__ float pos_factor(int p) {
  if (BITS == 2) return (float)(1 << (2 * (p <= 4 ? p : p - 5)));
  return (p & 1) ? 16.0f : 1.0f;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// fp16 hi + lo split of two fp32 values (hi = rn(x), lo = rn(x - hi)).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  hi = h2u(h);
  lo = h2u(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}

// Key-operand channel pair (c_lo, c_hi = c_lo + half word) of MMA column pair
// (tig, kb, reg); see the key extraction in process_tile.
template <int BITS>
__device__ __forceinline__ void key_pair(int tig, int kb, int reg, int &c_lo, int &c_hi, int &p) {
  if (BITS == 2) {
    const int W = 2 * tig + (kb >> 2);
    p = 2 * (kb & 3) + reg;
    c_lo = 16 * W + p;
    c_hi = c_lo + 8;
  } else {
    const int W = 4 * tig + (kb >> 1);
    p = 2 * (kb & 1) + reg;
    c_lo = 8 * W + p;
    c_hi = c_lo + 4;
  }
}

__device__ __forceinline__ int64_t owner_of(int64_t x, int64_t total, int nc) {
  return ((x + 1) * nc - 1) / total;
}

// Number of partials head bh produces, and the index of the fp16 one.
__device__ __forceinline__ void head_parts(const TcArgs &a, int64_t bh, int &nseg, int &nparts) {
  const int64_t base = bh * a.U;
  nseg = a.S_h > 0 ? (int)(owner_of(base + a.S_h - 1, a.total, a.nc) -
                           owner_of(base, a.total, a.nc) + 1)
                   : 0;
  nparts = nseg + (a.F_h > 0 ? 1 : 0);
}

// Threads 0..127 hold (M, L, O_c) of one partial of head bh in registers;
// publish it, take a ticket, and let the last block of the head merge.
__device__ void publish(const TcArgs &a, int64_t bh, int slot, float M, float L, float O,
                        int *sflag) {
  const int tid = threadIdx.x;
  const int64_t pi = bh * a.part_stride + slot;
  if (tid < kD) a.ws_o[pi * kD + tid] = O;
  if (tid == 0) {
    a.ws_ml[pi * 2] = M;
    a.ws_ml[pi * 2 + 1] = L;
  }
  int nseg, nparts;
  head_parts(a, bh, nseg, nparts);
  __threadfence();
  __syncthreads();
  if (tid == 0) sflag[1] = atomicAdd(&a.ws_cnt[bh], 1) == nparts - 1;
  __syncthreads();
  if (sflag[1]) {
    __threadfence();
    if (tid < kD) {
      float Mx = -INFINITY;
      for (int s = 0; s < nparts; ++s) Mx = fmaxf(Mx, __ldcg(&a.ws_ml[(bh * a.part_stride + s) * 2]));
      float Ls = 0.0f, Os = 0.0f;
      if (Mx != -INFINITY) {
        for (int s = 0; s < nparts; ++s) {
          const int64_t q = bh * a.part_stride + s;
          const float ms = __ldcg(&a.ws_ml[q * 2]);
          if (ms == -INFINITY) continue;
          const float w = exp2f(ms - Mx);
          Ls += w * __ldcg(&a.ws_ml[q * 2 + 1]);
          Os += w * __ldcg(&a.ws_o[q * kD + tid]);
        }
      }
      const int b = (int)(bh / a.g.H), h = (int)(bh % a.g.H);
      a.out[((int64_t)b * a.g.Hq + h) * kD + tid] = Ls > 0.0f ? Os / Ls : 0.0f;
    }
    if (tid == 0) a.ws_cnt[bh] = 0;
  }
  __syncthreads();
}

// fp16 sink + residual / window tokens of head bh on CUDA cores (<= 2048
// tokens); publishes partial `slot`.
__device__ void fp16_item(const TcArgs &a, int64_t bh, int slot, const float *sQf, float *scr,
                          int *sflag) {
  const Geometry &g = a.g;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = (int)a.n_fp16, ns = (int)a.n_sink;
  float *sc = scr;          // [2048]
  float *red = scr + 2048;  // [16][128]
  float *wred = scr + 4096; // [8]
  float mloc = -INFINITY;
  for (int i = tid; i < n; i += kThreads) {
    const __half *row = i < ns ? a.p.k_sink + (bh * g.n_sink + i) * kD
                               : a.p.k_res + (bh * g.residual + (i - ns)) * kD;
    float s = 0.0f;
#pragma unroll 4
    for (int c8 = 0; c8 < kD / 8; ++c8) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(row) + c8);
      const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __half22float2(hv[k]);
        s = fmaf(sQf[8 * c8 + 2 * k], f.x, s);
        s = fmaf(sQf[8 * c8 + 2 * k + 1], f.y, s);
      }
    }
    sc[i] = s;
    mloc = fmaxf(mloc, s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
  if (lane == 0) wred[warp] = mloc;
  __syncthreads();
  float M = wred[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, wred[w]);
  __syncthreads();
  float lloc = 0.0f;
  for (int i = tid; i < n; i += kThreads) {
    const float p = exp2f(sc[i] - M);
    sc[i] = p;
    lloc += p;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, off);
  if (lane == 0) wred[warp] = lloc;
  __syncthreads();
  float L = 0.0f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) L += wred[w];
  const int j = tid & 15, tl = tid >> 4;
  float acc[8] = {};
  for (int i = tl; i < n; i += 16) {
    const __half *row = i < ns ? a.p.v_sink + (bh * g.n_sink + i) * kD
                               : a.p.v_res + (bh * g.residual + (i - ns)) * kD;
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(row) + j);
    const __half2 *hv = reinterpret_cast<const __half2 *>(&raw);
    const float p = sc[i];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(hv[k]);
      acc[2 * k] = fmaf(p, f.x, acc[2 * k]);
      acc[2 * k + 1] = fmaf(p, f.y, acc[2 * k + 1]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) red[tl * kD + 8 * j + k] = acc[k];
  __syncthreads();
  float O = 0.0f;
  if (tid < kD)
    for (int r = 0; r < 16; ++r) O += red[r * kD + tid];
  publish(a, bh, slot, n > 0 ? M : -INFINITY, n > 0 ? L : 0.0f, O, sflag);
}

template <int BITS, int SCHEME, int NGV, int NGK>
__global__ void __launch_bounds__(kThreads, 2) tc_decode_kernel(const TcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int RB = kD * BITS / 8;  // packed bytes per token row
  const Geometry &g = a.g;
  const TcLayout Ly = tc_layout(a.slot_bytes);
  uint8_t *ring = smem + Ly.ring;
  uint32_t *sB = reinterpret_cast<uint32_t *>(smem + Ly.sB);
  float *sBias = reinterpret_cast<float *>(smem + Ly.sBias);
  float *sQf = reinterpret_cast<float *>(smem + Ly.sQf);
  float *sScr = reinterpret_cast<float *>(smem + Ly.sScr);
  int *sFlag = reinterpret_cast<int *>(smem + Ly.sFlag);
  float *sFlagF = reinterpret_cast<float *>(smem + Ly.sFlag);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Ly.bars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  const int64_t x0 = (int64_t)blockIdx.x * a.total / a.nc;
  const int64_t x1 = (int64_t)(blockIdx.x + 1) * a.total / a.nc;

  // zero the ring once so stale bytes are always finite; barriers
  for (int i = tid; i < kStages * a.slot_bytes / 16; i += kThreads)
    reinterpret_cast<uint4 *>(ring)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int s = 0; s <= kStages; ++s) bar_init(&bars[s], 1);
    sFlag[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();

  // ---- producer (thread 0): next quantized unit to fetch -----------------
  int64_t px = x0;
  int issued = 0;
  auto issue_next = [&]() {
    while (px < x1 && (int)(px % a.U) >= a.S_h) ++px;
    if (px >= x1) return;
    const int64_t bh = px / a.U;
    const int u = (int)(px % a.U);
    const int64_t tok0 = (int64_t)u * kTT;
    const int n = (int)min((int64_t)kTT, a.n_quant - tok0);
    uint8_t *dst = ring + (issued % kStages) * a.slot_bytes;
    uint64_t *bar = &bars[issued % kStages];
    const uint32_t cb = (uint32_t)(n * RB);
    uint32_t kmb, vmb = (uint32_t)((n * NGV * 4 + 15) & ~15);
    const float *ks, *kz;
    if (SCHEME == KVQ_KIVI) {
      kmb = (uint32_t)((n / g.k_group) * kD * 4);
      ks = a.p.k_scale + (bh * g.k_meta_rows + tok0 / g.k_group) * kD;
      kz = a.p.k_zero + (bh * g.k_meta_rows + tok0 / g.k_group) * kD;
    } else {
      kmb = (uint32_t)((n * NGK * 4 + 15) & ~15);
      ks = a.p.k_scale + (bh * g.cap + tok0) * NGK;
      kz = a.p.k_zero + (bh * g.cap + tok0) * NGK;
    }
    bar_expect_tx(bar, 2 * cb + 2 * kmb + 2 * vmb);
    bulk_g2s(dst, a.p.k_codes + (bh * g.cap + tok0) * RB, cb, bar);
    bulk_g2s(dst + a.off_vc, a.p.v_codes + (bh * g.cap + tok0) * RB, cb, bar);
    bulk_g2s(dst + a.off_ks, ks, kmb, bar);
    bulk_g2s(dst + a.off_kz, kz, kmb, bar);
    bulk_g2s(dst + a.off_vs, a.p.v_scale + (bh * g.cap + tok0) * NGV, vmb, bar);
    bulk_g2s(dst + a.off_vz, a.p.v_zero + (bh * g.cap + tok0) * NGV, vmb, bar);
    ++issued;
    ++px;
  };
  if (tid == 0)
    for (int s = 0; s < kStages - 1; ++s) issue_next();

  // ---- per-head constants --------------------------------------------------
  float pow2E = 1.0f;  // scores = raw * 2^E (q normalised by 2^-E)
  // KIVI key-operand build: this thread's channel pair (ip = tid % 64)
  const int ip = tid & 63;
  int bW, bp, b_clo, b_chi, b_tig, b_kb, b_reg;
  if (BITS == 2) {
    bW = ip >> 3;
    bp = ip & 7;
    b_clo = 16 * bW + bp;
    b_chi = b_clo + 8;
    b_tig = bW >> 1;
    b_kb = 4 * (bW & 1) + (bp >> 1);
  } else {
    bW = ip >> 2;
    bp = ip & 3;
    b_clo = 8 * bW + bp;
    b_chi = b_clo + 4;
    b_tig = bW >> 2;
    b_kb = 2 * (bW & 3) + (bp >> 1);
  }
  b_reg = bp & 1;
  float qn_lo = 0.f, qn_hi = 0.f, qf_lo = 0.f, qf_hi = 0.f;
  // InnerQ: fixed key operand and per-group sums of q
  uint32_t bqi[8][2];
  float Qj[NGK];

  // ---- per-warp online-softmax state --------------------------------------
  float m_run = -INFINITY, l_lane = 0.0f, z_lane[NGV];
  float dv[8][4];
  auto reset_state = [&]() {
    m_run = -INFINITY;
    l_lane = 0.0f;
#pragma unroll
    for (int j = 0; j < NGV; ++j) z_lane[j] = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) dv[mt][r] = 0.0f;
  };
  reset_state();

  auto start_head = [&](int64_t bh) {
    const int b = (int)(bh / g.H), h = (int)(bh % g.H);
    float v = 0.0f;
    if (tid < kD) {
      v = __half2float(a.q[((int64_t)b * g.Hq + h) * kD + tid]) * a.scale_log2;
      sQf[tid] = v;
    }
    float mx = fabsf(v);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0 && warp < 4) sFlagF[4 + warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(sFlagF[4], sFlagF[5]), fmaxf(sFlagF[6], sFlagF[7]));
    int E = 0;
    if (mx > 0.0f && mx < INFINITY) frexpf(mx, &E);
    pow2E = ldexpf(1.0f, E);
    const float inv = ldexpf(1.0f, -E);
    if (SCHEME == KVQ_KIVI) {
      const float f = pos_factor<BITS>(bp);
      qf_lo = sQf[b_clo];
      qf_hi = sQf[b_chi];
      qn_lo = qf_lo * inv / f;
      qn_hi = qf_hi * inv / f;
    } else {
      const int GK = kD / NGK;
#pragma unroll
      for (int j = 0; j < NGK; ++j) {
        float s = 0.0f;
        for (int c = j * GK; c < (j + 1) * GK; ++c) s += sQf[c];
        Qj[j] = s;
      }
      // columns n = gid = (group j = gid/2, part = gid%2); zero for gid >= 2*NGK
      const int jn = gid >> 1, part = gid & 1;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          int clo, chi, p;
          key_pair<BITS>(tig, kb, r, clo, chi, p);
          const float f = pos_factor<BITS>(p);
          const float vlo = (clo / GK == jn) ? sQf[clo] * inv / f : 0.0f;
          const float vhi = (chi / GK == jn) ? sQf[chi] * inv / f : 0.0f;
          uint32_t hi, lo;
          split2(vlo, vhi, hi, lo);
          bqi[kb][r] = gid < 2 * NGK ? (part ? lo : hi) : 0u;
        }
    }
    __syncthreads();
  };

  // Warp states -> one partial for head bh (slot = segment index).
  auto flush = [&](int64_t bh) {
    float l = l_lane;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    float Z[NGV];
#pragma unroll
    for (int j = 0; j < NGV; ++j) {
      float z = z_lane[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      Z[j] = z;
    }
    float *ws = sScr + warp * (kD + 2);
    const int gc = (gid * NGV) >> 3;  // value group of this thread's 16 channels
    if (tig == gc) {
      float zc = Z[0];
#pragma unroll
      for (int j = 1; j < NGV; ++j)
        if (j == gc) zc = Z[j];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float invf = 1.0f / pos_factor<BITS>(BITS == 2 ? mt : (mt & 3));
        ws[2 + 16 * gid + mt] = (dv[mt][0] + dv[mt][1]) * invf + zc;
        ws[2 + 16 * gid + 8 + mt] = (dv[mt][2] + dv[mt][3]) * invf + zc;
      }
    }
    if (lane == 0) {
      ws[0] = m_run;
      ws[1] = l;
    }
    __syncthreads();
    float M = -INFINITY, L = 0.0f, O = 0.0f;
    if (tid < kD) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sScr[w * (kD + 2)]);
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = sScr[w * (kD + 2)];
          if (mw == -INFINITY) continue;
          const float s = exp2f(mw - M);
          L += s * sScr[w * (kD + 2) + 1];
          O += s * sScr[w * (kD + 2) + 2 + tid];
        }
      }
    }
    const int seg = (int)(blockIdx.x - owner_of(bh * a.U, a.total, a.nc));
    publish(a, bh, seg, M, L, O, sFlag);
    reset_state();
  };

  int qi = 0;
  int64_t cur = -1;
  bool seg_open = false;
  bool aborted = false;
  for (int64_t x = x0; x < x1; ++x) {
    const int64_t bh = x / a.U;
    const int u = (int)(x % a.U);
    if (bh != cur) {
      if (seg_open) flush(cur);
      seg_open = false;
      start_head(bh);
      cur = bh;
    }
    if (u >= a.S_h) {
      if (u == a.S_h) {
        if (seg_open) flush(bh);
        seg_open = false;
        int nseg, nparts;
        head_parts(a, bh, nseg, nparts);
        fp16_item(a, bh, nseg, sQf, sScr, sFlag);
      }
      continue;
    }
    seg_open = true;
    if (tid == 0) issue_next();
    const int s = qi % kStages;
    const uint8_t *slot = ring + s * a.slot_bytes;
    bool ok = true;
    if (qi == 0 && a.stall_limit > 0) ok = bar_wait(&bars[kStages], 0u, a.stall_limit);
    if (!ok || !bar_wait(&bars[s], (uint32_t)((qi / kStages) & 1), a.wait_limit)) {
      sFlag[0] = 1;
      if (a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
    }
    const int n_stage = (int)min((int64_t)kTT, a.n_quant - (int64_t)u * kTT);

    if (SCHEME == KVQ_KIVI) {
      // q~ = q * scale (normalised, position factor divided out) as fp16
      // hi/lo in the B-fragment order, and q . zero per group.
      const int ngs = n_stage / g.k_group;
      const float *ks = reinterpret_cast<const float *>(slot + a.off_ks);
      const float *kz = reinterpret_cast<const float *>(slot + a.off_kz);
      for (int it = tid; it < ngs * 64; it += kThreads) {
        const int gl = it >> 6;
        const float v_lo = qn_lo * ks[gl * kD + b_clo], v_hi = qn_hi * ks[gl * kD + b_chi];
        uint32_t hi, lo;
        split2(v_lo, v_hi, hi, lo);
        uint32_t *dstB = sB + gl * 128;
        dstB[(0 * 4 + b_tig) * 16 + b_kb * 2 + b_reg] = hi;
        dstB[(1 * 4 + b_tig) * 16 + b_kb * 2 + b_reg] = lo;
        float bz = fmaf(qf_lo, kz[gl * kD + b_clo], qf_hi * kz[gl * kD + b_chi]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bz += __shfl_xor_sync(0xffffffffu, bz, off);
        if (lane == 0) sBias[gl * 2 + ((it >> 5) & 1)] = bz;
      }
    }
    __syncthreads();
    if (sFlag[0]) {
      aborted = true;
      break;
    }

    const int r0 = warp * 16;
    if (r0 < n_stage) {
      const uint8_t *kc = slot;
      const uint8_t *vc = slot + a.off_vc;
      // ---------------- keys: D[token][n] --------------------------------
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t bk[8][2];
      if (SCHEME == KVQ_KIVI) {
        const int gl = r0 / g.k_group;
        if (gid < 2) {
          const uint4 *src = reinterpret_cast<const uint4 *>(sB + gl * 128 + (gid * 4 + tig) * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v4 = src[i];
            bk[2 * i][0] = v4.x;
            bk[2 * i][1] = v4.y;
            bk[2 * i + 1][0] = v4.z;
            bk[2 * i + 1][1] = v4.w;
          }
        } else {
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) bk[kb][0] = bk[kb][1] = 0u;
        }
      } else {
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          bk[kb][0] = bqi[kb][0];
          bk[kb][1] = bqi[kb][1];
        }
      }
      if (BITS == 2) {
        const uint2 wa = *reinterpret_cast<const uint2 *>(kc + (r0 + gid) * RB + 8 * tig);
        const uint2 wb = *reinterpret_cast<const uint2 *>(kc + (r0 + gid + 8) * RB + 8 * tig);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t w0 = m ? wa.y : wa.x, w1 = m ? wb.y : wb.x;
          const uint32_t s0 = shifted<2>(w0), s1 = shifted<2>(w1);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            mma16816(d, ext<2>(w0, s0, 2 * j), ext<2>(w1, s1, 2 * j), ext<2>(w0, s0, 2 * j + 1),
                     ext<2>(w1, s1, 2 * j + 1), bk[4 * m + j][0], bk[4 * m + j][1]);
          }
        }
      } else {
        const uint4 wa = *reinterpret_cast<const uint4 *>(kc + (r0 + gid) * RB + 16 * tig);
        const uint4 wb = *reinterpret_cast<const uint4 *>(kc + (r0 + gid + 8) * RB + 16 * tig);
        const uint32_t A0[4] = {wa.x, wa.y, wa.z, wa.w}, A1[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t s0 = shifted<4>(A0[m]), s1 = shifted<4>(A1[m]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            mma16816(d, ext<4>(A0[m], s0, 2 * j), ext<4>(A1[m], s1, 2 * j),
                     ext<4>(A0[m], s0, 2 * j + 1), ext<4>(A1[m], s1, 2 * j + 1),
                     bk[2 * m + j][0], bk[2 * m + j][1]);
          }
        }
      }
      // ---------------- scores -> one token per lane (t = lane & 15) ------
      float ra, rb;
      if (SCHEME == KVQ_KIVI) {
        ra = d[0] + d[1];
        rb = d[2] + d[3];
      } else {
        const float *ks = reinterpret_cast<const float *>(slot + a.off_ks);
        const float *kz = reinterpret_cast<const float *>(slot + a.off_kz);
        const int jj = tig < NGK ? tig : NGK - 1;
        float qj = Qj[0];
#pragma unroll
        for (int j = 1; j < NGK; ++j)
          if (j == jj) qj = Qj[j];
        ra = fmaf(ks[(r0 + gid) * NGK + jj], (d[0] + d[1]) * pow2E, kz[(r0 + gid) * NGK + jj] * qj);
        rb = fmaf(ks[(r0 + gid + 8) * NGK + jj], (d[2] + d[3]) * pow2E,
                  kz[(r0 + gid + 8) * NGK + jj] * qj);
        if (tig >= NGK) ra = rb = 0.0f;
#pragma unroll
        for (int off = 1; off < NGK; off <<= 1) {
          ra += __shfl_xor_sync(0xffffffffu, ra, off);
          rb += __shfl_xor_sync(0xffffffffu, rb, off);
        }
      }
      const int t = lane & 15;
      const float xa = __shfl_sync(0xffffffffu, ra, 4 * (t & 7));
      const float xb = __shfl_sync(0xffffffffu, rb, 4 * (t & 7));
      float score = (t & 8) ? xb : xa;
      if (SCHEME == KVQ_KIVI) {
        const int gl = r0 / g.k_group;
        score = fmaf(score, pow2E, sBias[gl * 2] + sBias[gl * 2 + 1]);
      }
      const bool valid = r0 + t < n_stage;
      score = valid ? score : -INFINITY;
      float mt_ = score;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, off));
      if (mt_ > m_run) {
        const float alpha = exp2f(m_run - mt_);
        l_lane *= alpha;
#pragma unroll
        for (int j = 0; j < NGV; ++j) z_lane[j] *= alpha;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) dv[mt][r] *= alpha;
        m_run = mt_;
      }
      const float p = exp2f(score - m_run);
      const float pc = (lane < 16 && valid) ? p : 0.0f;
      l_lane += pc;
      {
        const float *vz = reinterpret_cast<const float *>(slot + a.off_vz);
#pragma unroll
        for (int j = 0; j < NGV; ++j)
          z_lane[j] = pc > 0.0f ? fmaf(pc, vz[(r0 + t) * NGV + j], z_lane[j]) : z_lane[j];
      }
      // ---------------- values: B = p * scale (hi/lo), A = codes ----------
      const float *vs = reinterpret_cast<const float *>(slot + a.off_vs);
      const int jg = (gid >> 1) < NGV ? (gid >> 1) : NGV - 1;
      const int tk0 = 2 * tig, tk1 = 2 * tig + 1, tk2 = 2 * tig + 8, tk3 = 2 * tig + 9;
      const float p0 = __shfl_sync(0xffffffffu, p, tk0), p1 = __shfl_sync(0xffffffffu, p, tk1);
      const float p2 = __shfl_sync(0xffffffffu, p, tk2), p3 = __shfl_sync(0xffffffffu, p, tk3);
      const float x0 = p0 > 0.0f ? p0 * vs[(r0 + tk0) * NGV + jg] : 0.0f;
      const float x1 = p1 > 0.0f ? p1 * vs[(r0 + tk1) * NGV + jg] : 0.0f;
      const float x2 = p2 > 0.0f ? p2 * vs[(r0 + tk2) * NGV + jg] : 0.0f;
      const float x3 = p3 > 0.0f ? p3 * vs[(r0 + tk3) * NGV + jg] : 0.0f;
      uint32_t h01, l01, h23, l23;
      split2(x0, x1, h01, l01);
      split2(x2, x3, h23, l23);
      const bool bact = gid < 2 * NGV;
      const uint32_t bv0 = bact ? ((gid & 1) ? l01 : h01) : 0u;
      const uint32_t bv1 = bact ? ((gid & 1) ? l23 : h23) : 0u;
      if (BITS == 2) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(vc + (r0 + tk0) * RB + 4 * gid);
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(vc + (r0 + tk1) * RB + 4 * gid);
        const uint32_t w2 = *reinterpret_cast<const uint32_t *>(vc + (r0 + tk2) * RB + 4 * gid);
        const uint32_t w3 = *reinterpret_cast<const uint32_t *>(vc + (r0 + tk3) * RB + 4 * gid);
        const uint32_t xa_ = __byte_perm(w0, w1, 0x5410), ya_ = __byte_perm(w0, w1, 0x7632);
        const uint32_t xb_ = __byte_perm(w2, w3, 0x5410), yb_ = __byte_perm(w2, w3, 0x7632);
        const uint32_t xas = shifted<2>(xa_), yas = shifted<2>(ya_);
        const uint32_t xbs = shifted<2>(xb_), ybs = shifted<2>(yb_);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma16816(dv[mt], ext<2>(xa_, xas, mt), ext<2>(ya_, yas, mt), ext<2>(xb_, xbs, mt),
                   ext<2>(yb_, ybs, mt), bv0, bv1);
      } else {
        const uint2 w0 = *reinterpret_cast<const uint2 *>(vc + (r0 + tk0) * RB + 8 * gid);
        const uint2 w1 = *reinterpret_cast<const uint2 *>(vc + (r0 + tk1) * RB + 8 * gid);
        const uint2 w2 = *reinterpret_cast<const uint2 *>(vc + (r0 + tk2) * RB + 8 * gid);
        const uint2 w3 = *reinterpret_cast<const uint2 *>(vc + (r0 + tk3) * RB + 8 * gid);
        // [0]: channels 16gid+0..3, [1]: +4..7, [2]: +8..11, [3]: +12..15
        const uint32_t xa4[4] = {__byte_perm(w0.x, w1.x, 0x5410), __byte_perm(w0.x, w1.x, 0x7632),
                                 __byte_perm(w0.y, w1.y, 0x5410), __byte_perm(w0.y, w1.y, 0x7632)};
        const uint32_t xb4[4] = {__byte_perm(w2.x, w3.x, 0x5410), __byte_perm(w2.x, w3.x, 0x7632),
                                 __byte_perm(w2.y, w3.y, 0x5410), __byte_perm(w2.y, w3.y, 0x7632)};
        uint32_t sa4[4], sb4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sa4[i] = shifted<4>(xa4[i]);
          sb4[i] = shifted<4>(xb4[i]);
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int lo = mt < 4 ? 0 : 1, hi = mt < 4 ? 2 : 3, pos = mt & 3;
          mma16816(dv[mt], ext<4>(xa4[lo], sa4[lo], pos), ext<4>(xa4[hi], sa4[hi], pos),
                   ext<4>(xb4[lo], sb4[lo], pos), ext<4>(xb4[hi], sb4[hi], pos), bv0, bv1);
        }
      }
    }
    __syncthreads();
    ++qi;
  }
  if (aborted) {
    if (tid == 0)
      for (int i = qi; i < issued; ++i)
        bar_wait(&bars[i % kStages], (uint32_t)((i / kStages) & 1), kDrainLimit);
    return;
  }
  if (seg_open) flush(cur);
}

template <int BITS, int SCHEME, int NGV, int NGK>
cudaError_t launch_tc_t(TcArgs &a, int smem, int num_sms, cudaStream_t st) {
  auto kern = tc_decode_kernel<BITS, SCHEME, NGV, NGK>;
  static int configured = 0;
  static int occ = 0;
  if (configured != smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    configured = smem;
  }
  int64_t nc = (int64_t)num_sms * occ;
  if (nc > a.total) nc = a.total;
  if (nc < 1) nc = 1;
  a.nc = (int)nc;
  kern<<<(unsigned)nc, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int BITS, int SCHEME>
cudaError_t launch_tc_v(TcArgs &a, int smem, int num_sms, cudaStream_t st) {
  const int ngv = kD / a.g.v_group;
  if constexpr (SCHEME == KVQ_KIVI) {
    return ngv == 4 ? launch_tc_t<BITS, SCHEME, 4, 1>(a, smem, num_sms, st)
                    : launch_tc_t<BITS, SCHEME, 2, 1>(a, smem, num_sms, st);
  } else {
  const int ngk = kD / a.g.k_group;
  if (ngv == 4)
    return ngk == 4 ? launch_tc_t<BITS, SCHEME, 4, 4>(a, smem, num_sms, st)
                    : launch_tc_t<BITS, SCHEME, 4, 2>(a, smem, num_sms, st);
  return ngk == 4 ? launch_tc_t<BITS, SCHEME, 2, 4>(a, smem, num_sms, st)
                  : launch_tc_t<BITS, SCHEME, 2, 2>(a, smem, num_sms, st);
  }
}

long long g_stall_limit = 0;

}  // namespace

void set_debug_stall(long long n) { g_stall_limit = n; }

bool tc_decode_supported(const Geometry &g) {
  if (g.d != kD || g.Hq != g.H) return false;
  const int ngv = kD / g.v_group;
  if (ngv != 2 && ngv != 4) return false;
  if (g.scheme == KVQ_KIVI) return g.k_group >= 16 && g.k_group <= 128;
  const int ngk = kD / g.k_group;
  return ngk == 2 || ngk == 4;
}

cudaError_t launch_decode_tc(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                             int64_t n_resid, int64_t n_sink, const __half *q, float *out,
                             float scale, void *ws, int num_sms, cudaStream_t st) {
  TcArgs a;
  a.g = g;
  a.p = p;
  a.q = q;
  a.out = out;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_quant = n_quant;
  a.n_fp16 = n_resid + n_sink;
  a.n_sink = n_sink;
  const int RB = kD * g.bits / 8;
  const int ngv = kD / g.v_group;
  const int kmb = g.scheme == KVQ_KIVI ? (kTT / g.k_group) * kD * 4 : kTT * (kD / g.k_group) * 4;
  const int vmb = kTT * ngv * 4;
  a.off_vc = kTT * RB;
  a.off_ks = 2 * kTT * RB;
  a.off_kz = a.off_ks + kmb;
  a.off_vs = a.off_kz + kmb;
  a.off_vz = a.off_vs + vmb;
  a.slot_bytes = (a.off_vz + vmb + 127) & ~127;
  a.S_h = (int)((n_quant + kTT - 1) / kTT);
  const int64_t payload = 2LL * kTT * RB + 2 * kmb + 2 * vmb;
  a.F_h = a.n_fp16 > 0 ? (int)((a.n_fp16 * kD * 2 * 2 * 2 + payload - 1) / payload) : 0;
  a.U = a.S_h + a.F_h;
  a.total = (int64_t)g.B * g.H * a.U;
  a.part_stride = part_slots(g);
  const int64_t BH = (int64_t)g.B * g.H;
  char *base = static_cast<char *>(ws);
  const size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  a.ws_cnt = reinterpret_cast<int *>(base);
  a.ws_ml = reinterpret_cast<float *>(base + cnt);
  a.ws_o = a.ws_ml + (size_t)BH * a.part_stride * 2;
  a.wait_limit = 1LL << 24;
  a.stall_limit = g_stall_limit;
  const int smem = tc_layout(a.slot_bytes).total;
  if (g.bits == 2)
    return g.scheme == KVQ_KIVI ? launch_tc_v<2, KVQ_KIVI>(a, smem, num_sms, st)
                                : launch_tc_v<2, KVQ_INNERQ>(a, smem, num_sms, st);
  return g.scheme == KVQ_KIVI ? launch_tc_v<4, KVQ_KIVI>(a, smem, num_sms, st)
                              : launch_tc_v<4, KVQ_INNERQ>(a, smem, num_sms, st);
}

}  // namespace kvq
