// Fused decode attention on the tensor cores (MHA, head_dim 128).
//
// Same computation as decode_kernel (softmax(scale * q.K^T) V over the packed
// cache, dequantization folded into both GEMVs -- "大模型量化技术原理：KIVI、
// IntactKV、KVQuant", KIVI / 背景; InnerQ page, 方法论 3), arranged for GB300:
//
//  * Persistent, stream-K: the (head, 128-token unit) list of the whole batch,
//    plus one cost-weighted fp16 item per head (sink + residual / window
//    tokens), is cut into equal contiguous ranges, one per resident block.  A
//    head split across blocks leaves one partial (m, l, o) per block; the last
//    block to finish a head (atomic ticket, no spinning) merges them with the
//    log-sum-exp rule.
//  * Warp-autonomous consumers: inside a block, the 32-token tiles of each
//    head segment go round-robin to the warps.  Each warp owns a small ring of
//    shared-memory slots that its lane 0 fills with 1-D cp.async.bulk copies
//    (codes + scale/zero of K and V of one tile) completed on the warp's own
//    mbarriers, and keeps its own online-softmax state; the block synchronises
//    only at head-segment ends, to merge the warps.  The ring runs ahead across
//    segment ends, so the copies never stop.  Every wait is bounded; a timeout
//    sets the status word and the warp drains its own copies before the block
//    returns.
//  * Both GEMVs run as mma.sync m16n8k16 (fp16 in, fp32 accumulate), two
//    independent 16-token MMA tiles per warp tile.  2/4-bit codes become exact
//    fp16 operands with one AND per two codes: the masked code bits, left in
//    place in the low ten bits of a 16-bit half, read as the subnormal
//    code * 2^(position bits) * 2^-24.  The position power of two is divided
//    out of the other operand (or the final output row) and the 2^-24 out of
//    the fp32 result, both exactly.  The channel order inside each MMA
//    is a permutation chosen so a thread consumes whole 32-bit code words; the
//    matching operand uses the same permutation.
//      keys   D[token][n] = sum_c code_tc * B[c][n],  B = q~ = q*scale split
//             into fp16 hi + lo (n = hi, lo); KIVI: rebuilt per G-token group,
//             InnerQ: q per channel group j (n = (j, hi/lo)), scale applied after.
//      values D[c][n] = sum_t code_tc * B[t][n],  B = p_t * scale_tj split into
//             hi + lo, n = (value group j, hi/lo); row c keeps column j(c).
//    zero points enter as q.zero per key group and sum_t p_t zero_tj per value
//    group (CUDA cores).  q is normalised by a power of two so no fp16 operand
//    can overflow (|q| <= 1, scales <= 65504).
#include <math.h>

#include <type_traits>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnit = 128;    // tokens per stream-K work unit
constexpr int kTile = 32;     // tokens per warp tile (two 16-token MMA tiles)
constexpr int kD = 128;
constexpr float kSub = 16777216.0f;  // 2^24: undoes the subnormal scale of the code operands
constexpr int kDrainLimit = 1 << 26;

struct TcArgs {
  Geometry g;
  CachePtrs p;
  const __half *q;
  float *out;
  float scale_log2;
  int64_t n_quant, n_fp16, n_sink;
  int S_h, F_h, U;  // quantized units, fp16 units, units per head
  int total;        // BH * U
  int nc;           // resident blocks
  float *ws_ml, *ws_o;
  int *ws_cnt;
  int part_stride;
  int wait_limit;   // poll cap of every pipeline wait
  int stall_limit;  // debug: > 0 = first wait on a barrier nothing completes
};

struct TcLayout {
  int ring, sB, bars, total;
};

__host__ __device__ constexpr TcLayout tc_layout(int slot_bytes, int nslot, int sb_bytes) {
  TcLayout L{};
  L.ring = 0;
  L.sB = L.ring + kWarps * nslot * slot_bytes;  // per warp: key operand + zero block
  L.bars = L.sB + kWarps * sb_bytes;            // per warp: nslot + 1 mbarriers
  L.total = L.bars + kWarps * (nslot + 1) * 8;
  return L;
}

// Compile-time layout of one warp-ring slot (one 32-token tile).  The first
// BB bytes are a copy of the cache block (K codes, V codes, V scale, V zero,
// InnerQ K scale, K zero; KIVI G <= 32 key statistics); for KIVI G >= 64 the
// statistics of the tile's key group (scale row, zero row); the query row
// on the first tile of a head.  Outside the ring each warp keeps its KIVI key
// operand (fp16 hi/lo words in fragment order, per key group) and 64 bytes
// that stay zero.
// KM (KIVI): 2 = G 16, two key groups per tile, statistics inside the block;
// 1 = G 32, one group, inside the block; 0 = G >= 64, the tile's group read
// from the separate key-statistics array.
template <int BITS, int SCHEME, int NGV, int NGK, int KM>
struct SlotCfg {
  static constexpr int RB = kD * BITS / 8;
  static constexpr int off_vc = kTile * RB;
  static constexpr int off_vs = 2 * kTile * RB;
  static constexpr int off_vz = off_vs + kTile * NGV * 4;
  static constexpr int off_ks = off_vz + kTile * NGV * 4;  // InnerQ
  static constexpr int off_kz = off_ks + kTile * NGK * 4;  // InnerQ
  static constexpr bool KIN = SCHEME == KVQ_KIVI && KM >= 1;
  static constexpr int KGB = (KM == 2 ? 2 : 1) * 2 * kD * 4;  // KIVI key statistics of a tile
  static constexpr int BB = SCHEME == KVQ_KIVI ? off_ks + (KIN ? KGB : 0) : off_kz + kTile * NGK * 4;
  static constexpr int KMB = SCHEME == KVQ_KIVI && !KIN ? KGB : 0;  // separate copy
  static constexpr int off_km = KIN ? off_ks : BB;
  static constexpr int off_q = BB + KMB;
  static constexpr int bytes = off_q + kD * 2;
  static constexpr int SBB = (SCHEME == KVQ_KIVI ? (KM == 2 ? 2 : 1) * 512 : 0) + 64;
  static constexpr int sb_zero = SBB / 4 - 16;  // word offset of the zero block
  static constexpr int nslot = tc_layout(bytes, 3, SBB).total <= 112 * 1024 ? 3 : 2;
  static constexpr int smem = tc_layout(bytes, nslot, SBB).total;
};


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
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity, int limit) {
  if (bar_try_wait(bar, parity)) return true;
  for (int it = 0; it < limit; ++it)
    if (bar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Code pair at position p of a word holding two 16-bit halves of codes:
// returns half2(code_lo * f, code_hi * f) * 2^-24 exactly, f = 4^p' (2-bit)
// or 16^p' (4-bit).  The masked bits sit in the low ten bits of each half, so
// each half reads as the fp16 subnormal (code * f) * 2^-24: one AND per pair.
// ws = w >> 10 (2-bit) or w >> 8 (4-bit), precomputed by the caller.
template <int BITS>
__device__ __forceinline__ uint32_t ext(uint32_t w, uint32_t ws, int p) {
  if (BITS == 2) return p <= 4 ? (w & (0x00030003u << (2 * p))) : (ws & (0x00030003u << (2 * (p - 5))));
  return p <= 1 ? (w & (0x000F000Fu << (4 * p))) : (ws & (0x000F000Fu << (4 * (p - 2))));
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
  asm(
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

__device__ __forceinline__ int owner_of(int x, int total, int nc) {
  return (int)(((int64_t)(x + 1) * nc - 1) / total);
}

// Quantized segments of head bh (one per block touching its quantized units)
// and the head's partial count: every warp of every such block leaves one
// partial, and so does every warp of the block owning the fp16 item.
__device__ __forceinline__ void head_parts(const TcArgs &a, int bh, int &nseg, int &nparts) {
  const int base = bh * a.U;
  nseg = a.S_h > 0 ? owner_of(base + a.S_h - 1, a.total, a.nc) - owner_of(base, a.total, a.nc) + 1
                   : 0;
  nparts = kWarps * (nseg + (a.F_h > 0 ? 1 : 0));
}

// One warp publishes partial `slot` of head bh (its o values are already
// stored), takes a ticket, and if it is the head's last partial, merges all
// of them with the log-sum-exp rule and writes the output row.
__device__ void warp_publish(const TcArgs &a, int bh, int slot, float m, float l) {
  const int lane = threadIdx.x & 31;
  const int64_t base = (int64_t)bh * a.part_stride;
  if (lane == 0) {
    a.ws_ml[(base + slot) * 2] = m;
    a.ws_ml[(base + slot) * 2 + 1] = l;
  }
  int nseg, nparts;
  head_parts(a, bh, nseg, nparts);
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&a.ws_cnt[bh], 1) == nparts - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  float Mx = -INFINITY;
  for (int s = lane; s < nparts; s += 32) Mx = fmaxf(Mx, __ldcg(&a.ws_ml[(base + s) * 2]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
  float Ls = 0.0f, O[4] = {0.f, 0.f, 0.f, 0.f};
  if (Mx != -INFINITY) {
    for (int s = 0; s < nparts; ++s) {
      const float ms = __ldcg(&a.ws_ml[(base + s) * 2]);
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - Mx);
      Ls = fmaf(w, __ldcg(&a.ws_ml[(base + s) * 2 + 1]), Ls);
      const float4 o = __ldcg(reinterpret_cast<const float4 *>(a.ws_o + (base + s) * kD) + lane);
      O[0] = fmaf(w, o.x, O[0]);
      O[1] = fmaf(w, o.y, O[1]);
      O[2] = fmaf(w, o.z, O[2]);
      O[3] = fmaf(w, o.w, O[3]);
    }
  }
  const int b = bh / a.g.H, h = bh % a.g.H;
  const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
  float4 r;
  r.x = O[0] * inv;
  r.y = O[1] * inv;
  r.z = O[2] * inv;
  r.w = O[3] * inv;
  reinterpret_cast<float4 *>(a.out + ((int64_t)b * a.g.Hq + h) * kD)[lane] = r;
  if (lane == 0) a.ws_cnt[bh] = 0;
}

template <int BITS, int SCHEME, int NGV, int NGK, int KM>
__global__ void __launch_bounds__(kThreads, 2) tc_decode_kernel(const TcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using SC = SlotCfg<BITS, SCHEME, NGV, NGK, KM>;
  constexpr bool G16 = SCHEME == KVQ_KIVI && KM == 2;
  constexpr int RB = SC::RB;  // packed bytes per token row
  constexpr int nslot = SC::nslot;
  constexpr int SLOT = SC::bytes;
  const Geometry &g = a.g;
  constexpr TcLayout Ly = tc_layout(SLOT, nslot, SC::SBB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  uint8_t *wring = smem + Ly.ring + warp * nslot * SLOT;
  uint64_t *wbars = reinterpret_cast<uint64_t *>(smem + Ly.bars) + warp * (nslot + 1);
  uint32_t *sBw = reinterpret_cast<uint32_t *>(smem + Ly.sB + warp * SC::SBB);

  const int x0 = (int)((int64_t)blockIdx.x * a.total / a.nc);
  const int x1 = (int)((int64_t)(blockIdx.x + 1) * a.total / a.nc);
  const int bh_first = x0 / a.U, bh_last = (x1 - 1) / a.U;

  // Each warp owns its ring and barriers; nothing below synchronises warps.
  for (int i = lane; i < nslot * SLOT / 16; i += 32)
    reinterpret_cast<uint4 *>(wring)[i] = make_uint4(0, 0, 0, 0);
  if (lane < 16) sBw[SC::sb_zero + lane] = 0u;
  if (lane == 0) {
    for (int s = 0; s <= nslot; ++s) bar_init(&wbars[s], 1);  // [nslot]: never completed
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();

  // quantized token range [tq0, tq1) of head bh inside this block's units
  auto seg_of = [&](int bh, int &tq0, int &tq1) {
    const int base = bh * a.U;
    const int ua = max(x0, base) - base;
    const int ub = min(min(x1, base + a.U) - base, a.S_h);
    tq0 = ua * kUnit;
    tq1 = ua < ub ? (int)min((int64_t)ub * kUnit, a.n_quant) : tq0;
  };

  // ---- producer: this warp's tiles in the order the consumer visits them --
  int pc_bh = -1, pc_tq0 = 0, pc_tq1 = 0, pc_lt = 0, issued = 0, ps = 0;
  auto pc_settle = [&]() {
    while (pc_bh >= 0 && pc_tq0 + kTile * pc_lt >= pc_tq1) {
      if (++pc_bh > bh_last) {
        pc_bh = -1;
        return;
      }
      seg_of(pc_bh, pc_tq0, pc_tq1);
      pc_lt = warp;
    }
  };
  // Called by the whole warp; lane 0 posts the byte count and issues the
  // copies of the next tile of this warp: its cache block, the KIVI key
  // statistics of its group(s), and the query row on the first tile of a head.
  auto issue_next = [&]() {
    if (pc_bh < 0) return;
    const int tok0 = pc_tq0 + kTile * pc_lt;
    const bool first = pc_lt == warp;
    uint8_t *dst = wring + ps * SLOT;
    uint64_t *bar = &wbars[ps];
    ps = ps + 1 == nslot ? 0 : ps + 1;
    if (lane == 0) {
      bar_expect_tx(bar, (uint32_t)(SC::BB + SC::KMB + (first ? kD * 2 : 0)));
      bulk_g2s(dst, a.p.blocks + ((int64_t)pc_bh * (g.cap / kTile) + tok0 / kTile) * SC::BB,
               SC::BB, bar);
      if (SCHEME == KVQ_KIVI && !SC::KIN)
        bulk_g2s(dst + SC::off_km,
                 a.p.k_meta + ((int64_t)pc_bh * g.k_meta_rows + tok0 / g.k_group) * 2 * kD,
                 SC::KMB, bar);
      if (first)
        bulk_g2s(dst + SC::off_q, a.q + ((int64_t)(pc_bh / g.H) * g.Hq + pc_bh % g.H) * kD,
                 kD * 2, bar);
    }
    ++issued;
    pc_lt += kWarps;
    pc_settle();
  };
  pc_bh = bh_first;
  seg_of(pc_bh, pc_tq0, pc_tq1);
  pc_lt = warp;
  pc_settle();
  for (int s = 0; s < nslot; ++s) issue_next();

  // ---- per-head constants (each warp for itself) --------------------------
  float pow2E = 1.0f;  // scores = raw * 2^(E+24) (q normalised by 2^-E, codes by 2^-24)
  float q4[4];         // q of channels 4*lane .. 4*lane+3 (exp2 domain)
  // KIVI key operand: this lane builds channel pairs ip = lane and lane + 32
  constexpr int kHalf = BITS == 2 ? 8 : 4;  // channel offset of the high half of a pair
  int b_clo[2], b_sidx[2];
  float qn_lo[2], qn_hi[2], qf_lo[2], qf_hi[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int ip = lane + 32 * r;
    int W, p, tg, kb;
    if (BITS == 2) {
      W = ip >> 3;
      p = ip & 7;
      b_clo[r] = 16 * W + p;
      tg = W >> 1;
      kb = 4 * (W & 1) + (p >> 1);
    } else {
      W = ip >> 2;
      p = ip & 3;
      b_clo[r] = 8 * W + p;
      tg = W >> 2;
      kb = 2 * (W & 3) + (p >> 1);
    }
    b_sidx[r] = tg * 16 + kb * 2 + (p & 1);
    qn_lo[r] = qn_hi[r] = qf_lo[r] = qf_hi[r] = 0.0f;
  }
  // InnerQ: fixed key operand and per-group sums of q
  uint32_t bqi[8][2];
  float Qj[NGK];

  // Per-head constants from the query row that rode along with the head's
  // first tile of this warp.
  auto start_head = [&](const uint8_t *slot) {
    const __half *qh = reinterpret_cast<const __half *>(slot + SC::off_q);
    const uint2 qr = reinterpret_cast<const uint2 *>(qh)[lane];
    const float2 q01 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.x));
    const float2 q23 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.y));
    q4[0] = q01.x * a.scale_log2;
    q4[1] = q01.y * a.scale_log2;
    q4[2] = q23.x * a.scale_log2;
    q4[3] = q23.y * a.scale_log2;
    float mx = fmaxf(fmaxf(fabsf(q4[0]), fabsf(q4[1])), fmaxf(fabsf(q4[2]), fabsf(q4[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    int E = 0;
    if (mx > 0.0f && mx < INFINITY) frexpf(mx, &E);
    pow2E = ldexpf(1.0f, E) * kSub;
    const float inv = ldexpf(1.0f, -E);
    auto qf = [&](int c) { return __half2float(qh[c]) * a.scale_log2; };
    if (SCHEME == KVQ_KIVI) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int p = BITS == 2 ? (b_clo[r] & 7) : (b_clo[r] & 3);
        const float invf = inv / pos_factor<BITS>(p);
        qf_lo[r] = qf(b_clo[r]);
        qf_hi[r] = qf(b_clo[r] + kHalf);
        qn_lo[r] = qf_lo[r] * invf;
        qn_hi[r] = qf_hi[r] * invf;
      }
    } else {
      const int GK = kD / NGK;
      const float s4 = (q4[0] + q4[1]) + (q4[2] + q4[3]);
#pragma unroll
      for (int j = 0; j < NGK; ++j) {
        float sj = (4 * lane) / GK == j ? s4 : 0.0f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sj += __shfl_xor_sync(0xffffffffu, sj, off);
        Qj[j] = sj;
      }
      // columns n = gid = (group j = gid/2, part = gid%2); zero for gid >= 2*NGK
      const int jn = gid >> 1, part = gid & 1;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          int clo, chi, p;
          key_pair<BITS>(tig, kb, r, clo, chi, p);
          const float invf = inv / pos_factor<BITS>(p);
          const float vlo = (clo / GK == jn) ? qf(clo) * invf : 0.0f;
          const float vhi = (chi / GK == jn) ? qf(chi) * invf : 0.0f;
          uint32_t hi, lo;
          split2(vlo, vhi, hi, lo);
          bqi[kb][r] = gid < 2 * NGK ? (part ? lo : hi) : 0u;
        }
    }
  };

  // ---- per-warp online-softmax state ----------------------------------------
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

  // Warp state -> partial `slot` of head bh (lanes hold one token each, so
  // every lane counts).
  auto flush = [&](int bh, int slot) {
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
    float *wo = a.ws_o + ((int64_t)bh * a.part_stride + slot) * kD;
    const int gc = (gid * NGV) >> 3;  // value group of this thread's 16 channels
    if (tig == gc) {
      float zc = Z[0];
#pragma unroll
      for (int j = 1; j < NGV; ++j)
        if (j == gc) zc = Z[j];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float invf = kSub / pos_factor<BITS>(BITS == 2 ? mt : (mt & 3));
        wo[16 * gid + mt] = fmaf(dv[mt][0] + dv[mt][1], invf, zc);
        wo[16 * gid + 8 + mt] = fmaf(dv[mt][2] + dv[mt][3], invf, zc);
      }
    }
    warp_publish(a, bh, slot, m_run, l);
    reset_state();
  };

  // fp16 sink + residual / window tokens of head bh: this warp takes every
  // kWarps-th token (a lane owns 4 channels) and publishes partial `slot`.
  auto fp16_item = [&](int bh, int slot) {
    const int n = (int)a.n_fp16, ns = (int)a.n_sink;
    float qq[4];
    {
      const uint2 qr = __ldg(reinterpret_cast<const uint2 *>(
                                 a.q + ((int64_t)(bh / g.H) * g.Hq + bh % g.H) * kD) + lane);
      const float2 q01 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.x));
      const float2 q23 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.y));
      qq[0] = q01.x * a.scale_log2;
      qq[1] = q01.y * a.scale_log2;
      qq[2] = q23.x * a.scale_log2;
      qq[3] = q23.y * a.scale_log2;
    }
    float m = -INFINITY, l = 0.0f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = warp; i < n; i += kWarps) {
      const int64_t kr = i < ns ? ((int64_t)bh * g.n_sink + i) : ((int64_t)bh * g.residual + (i - ns));
      const __half *krow = (i < ns ? a.p.k_sink : a.p.k_res) + kr * kD;
      const __half *vrow = (i < ns ? a.p.v_sink : a.p.v_res) + kr * kD;
      const uint2 kw = __ldg(reinterpret_cast<const uint2 *>(krow) + lane);
      const uint2 vw = __ldg(reinterpret_cast<const uint2 *>(vrow) + lane);
      const float2 k01 = __half22float2(*reinterpret_cast<const __half2 *>(&kw.x));
      const float2 k23 = __half22float2(*reinterpret_cast<const __half2 *>(&kw.y));
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.y));
      float sc = fmaf(qq[0], k01.x, fmaf(qq[1], k01.y, fmaf(qq[2], k23.x, qq[3] * k23.y)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
      const float mn = fmaxf(m, sc);
      const float al = exp2f(m - mn), pp = exp2f(sc - mn);
      l = fmaf(l, al, pp);
      acc[0] = fmaf(acc[0], al, pp * v01.x);
      acc[1] = fmaf(acc[1], al, pp * v01.y);
      acc[2] = fmaf(acc[2], al, pp * v23.x);
      acc[3] = fmaf(acc[3], al, pp * v23.y);
      m = mn;
    }
    float4 o;
    o.x = acc[0];
    o.y = acc[1];
    o.z = acc[2];
    o.w = acc[3];
    reinterpret_cast<float4 *>(a.ws_o + ((int64_t)bh * a.part_stride + slot) * kD)[lane] = o;
    warp_publish(a, bh, slot, m, l);
  };

  int done = 0;          // tiles whose copies completed
  int cs = 0;            // ring slot of the next tile
  uint32_t cph = 0;      // its barrier phase parity
  bool first = true;
  for (int bh = bh_first; bh <= bh_last; ++bh) {
    int tq0, tq1;
    seg_of(bh, tq0, tq1);
    const int base = bh * a.U;
    const bool own_fp16 = a.F_h > 0 && x0 <= base + a.S_h && base + a.S_h < x1;
    if (tq1 <= tq0 && !own_fp16) continue;
    if (tq1 > tq0) {
      const int nt = (tq1 - tq0 + kTile - 1) / kTile;
      bool aborted = false;
      for (int lt = warp; lt < nt; lt += kWarps) {
        const int s = cs;
        const uint32_t par = cph;
        if (++cs == nslot) {
          cs = 0;
          cph ^= 1u;
        }
        bool ok = true;
        if (first && a.stall_limit > 0) ok = bar_wait(&wbars[nslot], 0u, a.stall_limit);
        first = false;
        if (ok) ok = bar_wait(&wbars[s], par, a.wait_limit);
        // one verdict per warp: every lane takes the same path from here
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
          aborted = true;
          break;
        }
        ++done;
        const uint8_t *slot = wring + s * SLOT;
        if (lt == warp) start_head(slot);
        const int tok0 = tq0 + kTile * lt;
        const int n = min(kTile, tq1 - tok0);
        auto tile = [&](auto full_c) {
          constexpr bool FULL = decltype(full_c)::value;
          const uint8_t *kc = slot;
          const uint8_t *vc = slot + SC::off_vc;
          // ------------- keys: two 16-token MMA tiles ------------------------
          float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
          float bias0 = 0.0f, bias1 = 0.0f;
          uint32_t bk[8][2];
          auto load_bk = [&](int gl) {
            if (SCHEME == KVQ_KIVI) {
              // lanes of columns >= 2 read the zero block: no divergent branch
              const uint4 *src = reinterpret_cast<const uint4 *>(
                  gid < 2 ? sBw + gl * 128 + (gid * 4 + tig) * 16 : sBw + SC::sb_zero);
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
              for (int kb = 0; kb < 8; ++kb) {
                bk[kb][0] = bqi[kb][0];
                bk[kb][1] = bqi[kb][1];
              }
            }
          };
          bool two_groups = false;
          if (SCHEME == KVQ_KIVI) {
            // q~ = q * scale (normalised, position factor divided out) as fp16
            // hi/lo in B-fragment order, and q . zero, per key group of the tile
            const float *km = reinterpret_cast<const float *>(slot + SC::off_km);
            two_groups = G16 && (FULL || n > 16);
  #pragma unroll
            for (int gl = 0; gl < (G16 ? 2 : 1); ++gl) {
              if (gl == 1 && !two_groups) break;
              const float *ks = km + gl * 2 * kD, *kz = ks + kD;
              float bz = 0.0f;
  #pragma unroll
              for (int r = 0; r < 2; ++r) {
                const int clo = b_clo[r], chi = b_clo[r] + kHalf;
                uint32_t hi, lo;
                split2(qn_lo[r] * ks[clo], qn_hi[r] * ks[chi], hi, lo);
                sBw[gl * 128 + b_sidx[r]] = hi;
                sBw[gl * 128 + 64 + b_sidx[r]] = lo;
                bz = fmaf(qf_lo[r], kz[clo], fmaf(qf_hi[r], kz[chi], bz));
              }
  #pragma unroll
              for (int off = 16; off > 0; off >>= 1) bz += __shfl_xor_sync(0xffffffffu, bz, off);
              if (gl == 0) bias0 = bz;
              bias1 = bz;
            }
            __syncwarp();
          }
          load_bk(0);
          if (BITS == 2) {
            const uint2 wa0 = *reinterpret_cast<const uint2 *>(kc + gid * RB + 8 * tig);
            const uint2 wb0 = *reinterpret_cast<const uint2 *>(kc + (gid + 8) * RB + 8 * tig);
            const uint2 wa1 = *reinterpret_cast<const uint2 *>(kc + (gid + 16) * RB + 8 * tig);
            const uint2 wb1 = *reinterpret_cast<const uint2 *>(kc + (gid + 24) * RB + 8 * tig);
            if (!two_groups) {
  #pragma unroll
              for (int m = 0; m < 2; ++m) {
                const uint32_t w00 = m ? wa0.y : wa0.x, w01 = m ? wb0.y : wb0.x;
                const uint32_t w10 = m ? wa1.y : wa1.x, w11 = m ? wb1.y : wb1.x;
                const uint32_t s00 = shifted<2>(w00), s01 = shifted<2>(w01);
                const uint32_t s10 = shifted<2>(w10), s11 = shifted<2>(w11);
  #pragma unroll
                for (int j = 0; j < 4; ++j) {
                  mma16816(d0, ext<2>(w00, s00, 2 * j), ext<2>(w01, s01, 2 * j),
                           ext<2>(w00, s00, 2 * j + 1), ext<2>(w01, s01, 2 * j + 1),
                           bk[4 * m + j][0], bk[4 * m + j][1]);
                  mma16816(d1, ext<2>(w10, s10, 2 * j), ext<2>(w11, s11, 2 * j),
                           ext<2>(w10, s10, 2 * j + 1), ext<2>(w11, s11, 2 * j + 1),
                           bk[4 * m + j][0], bk[4 * m + j][1]);
                }
              }
            } else {
  #pragma unroll
              for (int t2 = 0; t2 < 2; ++t2) {
                if (t2 == 1) load_bk(1);
                const uint2 wa = t2 ? wa1 : wa0, wb = t2 ? wb1 : wb0;
  #pragma unroll
                for (int m = 0; m < 2; ++m) {
                  const uint32_t w0 = m ? wa.y : wa.x, w1 = m ? wb.y : wb.x;
                  const uint32_t s0 = shifted<2>(w0), s1 = shifted<2>(w1);
  #pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    if (t2 == 0)
                      mma16816(d0, ext<2>(w0, s0, 2 * j), ext<2>(w1, s1, 2 * j),
                               ext<2>(w0, s0, 2 * j + 1), ext<2>(w1, s1, 2 * j + 1),
                               bk[4 * m + j][0], bk[4 * m + j][1]);
                    else
                      mma16816(d1, ext<2>(w0, s0, 2 * j), ext<2>(w1, s1, 2 * j),
                               ext<2>(w0, s0, 2 * j + 1), ext<2>(w1, s1, 2 * j + 1),
                               bk[4 * m + j][0], bk[4 * m + j][1]);
                  }
                }
              }
            }
          } else {
            // 4-bit keys: G >= 32 always gives one key group per tile here
            // (the 4-bit group-16 case takes the same path with two groups)
  #pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {
              if (two_groups && t2 == 1) load_bk(1);
              const uint4 wa = *reinterpret_cast<const uint4 *>(kc + (16 * t2 + gid) * RB + 16 * tig);
              const uint4 wb = *reinterpret_cast<const uint4 *>(kc + (16 * t2 + gid + 8) * RB + 16 * tig);
              const uint32_t A0[4] = {wa.x, wa.y, wa.z, wa.w}, A1[4] = {wb.x, wb.y, wb.z, wb.w};
  #pragma unroll
              for (int m = 0; m < 4; ++m) {
                const uint32_t s0 = shifted<4>(A0[m]), s1 = shifted<4>(A1[m]);
  #pragma unroll
                for (int j = 0; j < 2; ++j) {
                  if (t2 == 0)
                    mma16816(d0, ext<4>(A0[m], s0, 2 * j), ext<4>(A1[m], s1, 2 * j),
                             ext<4>(A0[m], s0, 2 * j + 1), ext<4>(A1[m], s1, 2 * j + 1),
                             bk[2 * m + j][0], bk[2 * m + j][1]);
                  else
                    mma16816(d1, ext<4>(A0[m], s0, 2 * j), ext<4>(A1[m], s1, 2 * j),
                             ext<4>(A0[m], s0, 2 * j + 1), ext<4>(A1[m], s1, 2 * j + 1),
                             bk[2 * m + j][0], bk[2 * m + j][1]);
                }
              }
            }
          }
          // ------------- scores -> one token per lane ------------------------
          float ra0, rb0, ra1, rb1;
          if (SCHEME == KVQ_KIVI) {
            ra0 = d0[0] + d0[1];
            rb0 = d0[2] + d0[3];
            ra1 = d1[0] + d1[1];
            rb1 = d1[2] + d1[3];
          } else {
            const float *ks = reinterpret_cast<const float *>(slot + SC::off_ks);
            const float *kz = reinterpret_cast<const float *>(slot + SC::off_kz);
            const int jj = tig < NGK ? tig : NGK - 1;
            float qj = Qj[0];
  #pragma unroll
            for (int j = 1; j < NGK; ++j)
              if (j == jj) qj = Qj[j];
            auto term = [&](int row, float dd) {
              return fmaf(ks[row * NGK + jj], dd * pow2E, kz[row * NGK + jj] * qj);
            };
            ra0 = term(gid, d0[0] + d0[1]);
            rb0 = term(gid + 8, d0[2] + d0[3]);
            ra1 = term(gid + 16, d1[0] + d1[1]);
            rb1 = term(gid + 24, d1[2] + d1[3]);
            if (tig >= NGK) ra0 = rb0 = ra1 = rb1 = 0.0f;
  #pragma unroll
            for (int off = 1; off < NGK; off <<= 1) {
              ra0 += __shfl_xor_sync(0xffffffffu, ra0, off);
              rb0 += __shfl_xor_sync(0xffffffffu, rb0, off);
              ra1 += __shfl_xor_sync(0xffffffffu, ra1, off);
              rb1 += __shfl_xor_sync(0xffffffffu, rb1, off);
            }
          }
          const int t = lane;
          const int src = 4 * (t & 7);
          const float xa0 = __shfl_sync(0xffffffffu, ra0, src), xb0 = __shfl_sync(0xffffffffu, rb0, src);
          const float xa1 = __shfl_sync(0xffffffffu, ra1, src), xb1 = __shfl_sync(0xffffffffu, rb1, src);
          float score = t < 16 ? ((t & 8) ? xb0 : xa0) : ((t & 8) ? xb1 : xa1);
          if (SCHEME == KVQ_KIVI) score = fmaf(score, pow2E, t < 16 ? bias0 : bias1);
          const bool valid = FULL || t < n;
          score = valid ? score : -INFINITY;
          float mt_ = score;
  #pragma unroll
          for (int off = 1; off < 32; off <<= 1) mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, off));
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
          l_lane += p;
          {
            const float *vz = reinterpret_cast<const float *>(slot + SC::off_vz) + t * NGV;
            float zr[NGV];
            if (NGV == 4) {
              const float4 z4 = *reinterpret_cast<const float4 *>(vz);
              zr[0] = z4.x;
              zr[1] = z4.y;
              zr[2 % NGV] = z4.z;
              zr[3 % NGV] = z4.w;
            } else {
              const float2 z2 = *reinterpret_cast<const float2 *>(vz);
              zr[0] = z2.x;
              zr[1 % NGV] = z2.y;
            }
  #pragma unroll
            for (int j = 0; j < NGV; ++j)
              z_lane[j] = (FULL || p > 0.0f) ? fmaf(p, zr[j], z_lane[j]) : z_lane[j];
          }
          // ------------- values: B = p * scale (hi/lo), A = codes ------------
          const float *vs = reinterpret_cast<const float *>(slot + SC::off_vs);
          const int jg = (gid >> 1) < NGV ? (gid >> 1) : NGV - 1;
          const bool bact = gid < 2 * NGV;
          const int nkb = (FULL || n > 16) ? 2 : 1;
          for (int kb = 0; kb < nkb; ++kb) {
            // MMA k pairs (2tig, 2tig+1) and (2tig+8, 2tig+9) carry tokens
            // tig + {0, 4} and tig + {8, 12}: rows 4 apart hit distinct banks
            const int tk0 = 16 * kb + tig, tk1 = tk0 + 4, tk2 = tk0 + 8, tk3 = tk0 + 12;
            const float p0 = __shfl_sync(0xffffffffu, p, tk0), p1 = __shfl_sync(0xffffffffu, p, tk1);
            const float p2 = __shfl_sync(0xffffffffu, p, tk2), p3 = __shfl_sync(0xffffffffu, p, tk3);
            const float x0 = (FULL || p0 > 0.0f) ? p0 * vs[tk0 * NGV + jg] : 0.0f;
            const float x1 = (FULL || p1 > 0.0f) ? p1 * vs[tk1 * NGV + jg] : 0.0f;
            const float x2 = (FULL || p2 > 0.0f) ? p2 * vs[tk2 * NGV + jg] : 0.0f;
            const float x3 = (FULL || p3 > 0.0f) ? p3 * vs[tk3 * NGV + jg] : 0.0f;
            uint32_t h01, l01, h23, l23;
            split2(x0, x1, h01, l01);
            split2(x2, x3, h23, l23);
            const uint32_t bv0 = bact ? ((gid & 1) ? l01 : h01) : 0u;
            const uint32_t bv1 = bact ? ((gid & 1) ? l23 : h23) : 0u;
            if (BITS == 2) {
              const uint32_t w0 = *reinterpret_cast<const uint32_t *>(vc + tk0 * RB + 4 * gid);
              const uint32_t w1 = *reinterpret_cast<const uint32_t *>(vc + tk1 * RB + 4 * gid);
              const uint32_t w2 = *reinterpret_cast<const uint32_t *>(vc + tk2 * RB + 4 * gid);
              const uint32_t w3 = *reinterpret_cast<const uint32_t *>(vc + tk3 * RB + 4 * gid);
              const uint32_t xa_ = __byte_perm(w0, w1, 0x5410), ya_ = __byte_perm(w0, w1, 0x7632);
              const uint32_t xb_ = __byte_perm(w2, w3, 0x5410), yb_ = __byte_perm(w2, w3, 0x7632);
              const uint32_t xas = shifted<2>(xa_), yas = shifted<2>(ya_);
              const uint32_t xbs = shifted<2>(xb_), ybs = shifted<2>(yb_);
  #pragma unroll
              for (int mt = 0; mt < 8; ++mt)
                mma16816(dv[mt], ext<2>(xa_, xas, mt), ext<2>(ya_, yas, mt), ext<2>(xb_, xbs, mt),
                         ext<2>(yb_, ybs, mt), bv0, bv1);
            } else {
              const uint2 w0 = *reinterpret_cast<const uint2 *>(vc + tk0 * RB + 8 * gid);
              const uint2 w1 = *reinterpret_cast<const uint2 *>(vc + tk1 * RB + 8 * gid);
              const uint2 w2 = *reinterpret_cast<const uint2 *>(vc + tk2 * RB + 8 * gid);
              const uint2 w3 = *reinterpret_cast<const uint2 *>(vc + tk3 * RB + 8 * gid);
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
        };
        if (n == kTile)
          tile(std::true_type{});
        else
          tile(std::false_type{});
        __syncwarp();
        issue_next();  // refill the slot just consumed
      }
      if (aborted) {
        // give up this block's work for this warp; its copies complete first
        if (lane == 0)
          for (int i = done; i < issued; ++i)
            bar_wait(&wbars[i % nslot], (uint32_t)((i / nslot) & 1), kDrainLimit);
        return;
      }
      const int seg = (int)blockIdx.x - owner_of(base, a.total, a.nc);
      flush(bh, seg * kWarps + warp);
    }
    if (own_fp16) {
      int nseg, nparts;
      head_parts(a, bh, nseg, nparts);
      fp16_item(bh, nseg * kWarps + warp);
    }
  }
}

template <int BITS, int SCHEME, int NGV, int NGK, int KM>
cudaError_t launch_tc_t(TcArgs &a, int num_sms, cudaStream_t st) {
  auto kern = tc_decode_kernel<BITS, SCHEME, NGV, NGK, KM>;
  constexpr int smem = SlotCfg<BITS, SCHEME, NGV, NGK, KM>::smem;
  if (a.g.block_bytes != SlotCfg<BITS, SCHEME, NGV, NGK, KM>::BB) return cudaErrorInvalidValue;
  static int occ = 0;
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int o = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    occ = o < 1 ? 1 : o;
  }
  int64_t nc = (int64_t)num_sms * occ;
  if (nc > kTcMaxBlocks) nc = kTcMaxBlocks;
  if (nc > a.total) nc = a.total;
  if (nc < 1) nc = 1;
  a.nc = (int)nc;
  kern<<<(unsigned)nc, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int BITS, int SCHEME>
cudaError_t launch_tc_v(TcArgs &a, int num_sms, cudaStream_t st) {
  const int ngv = kD / a.g.v_group;
  if constexpr (SCHEME == KVQ_KIVI) {
    const int G = a.g.k_group;
    if (ngv == 4)
      return G == 16 ? launch_tc_t<BITS, SCHEME, 4, 1, 2>(a, num_sms, st)
           : G == 32 ? launch_tc_t<BITS, SCHEME, 4, 1, 1>(a, num_sms, st)
                     : launch_tc_t<BITS, SCHEME, 4, 1, 0>(a, num_sms, st);
    return G == 16 ? launch_tc_t<BITS, SCHEME, 2, 1, 2>(a, num_sms, st)
         : G == 32 ? launch_tc_t<BITS, SCHEME, 2, 1, 1>(a, num_sms, st)
                   : launch_tc_t<BITS, SCHEME, 2, 1, 0>(a, num_sms, st);
  } else {
    const int ngk = kD / a.g.k_group;
    if (ngv == 4)
      return ngk == 4 ? launch_tc_t<BITS, SCHEME, 4, 4, 0>(a, num_sms, st)
                      : launch_tc_t<BITS, SCHEME, 4, 2, 0>(a, num_sms, st);
    return ngk == 4 ? launch_tc_t<BITS, SCHEME, 2, 4, 0>(a, num_sms, st)
                    : launch_tc_t<BITS, SCHEME, 2, 2, 0>(a, num_sms, st);
  }
}

int g_stall_limit = 0;

}  // namespace

void set_debug_stall(long long n) { g_stall_limit = n > (1 << 30) ? (1 << 30) : (int)n; }

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
  a.S_h = (int)((n_quant + kUnit - 1) / kUnit);
  // fp16 item weight in units: its bytes against a unit's bytes, x2 for the
  // CUDA-core path
  const int64_t unit_bytes = 2LL * kUnit * RB + 2LL * kUnit * ngv * 4 +
                             (g.scheme == KVQ_KIVI ? 2LL * (kUnit / g.k_group) * kD * 4
                                                   : 2LL * kUnit * (kD / g.k_group) * 4);
  a.F_h = a.n_fp16 > 0 ? (int)((a.n_fp16 * kD * 2 * 2 * 2 + unit_bytes - 1) / unit_bytes) : 0;
  a.U = a.S_h + a.F_h;
  const int64_t total = (int64_t)g.B * g.H * a.U;
  if (total >= (1LL << 31)) return cudaErrorInvalidValue;
  a.total = (int)total;
  a.part_stride = tc_part_slots(g);
  const int64_t BH = (int64_t)g.B * g.H;
  char *base = static_cast<char *>(ws);
  const size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  a.ws_cnt = reinterpret_cast<int *>(base);
  a.ws_ml = reinterpret_cast<float *>(base + cnt);
  a.ws_o = a.ws_ml + (size_t)BH * a.part_stride * 2;
  a.wait_limit = 1 << 24;
  a.stall_limit = g_stall_limit;
  if (g.bits == 2)
    return g.scheme == KVQ_KIVI ? launch_tc_v<2, KVQ_KIVI>(a, num_sms, st)
                                : launch_tc_v<2, KVQ_INNERQ>(a, num_sms, st);
  return g.scheme == KVQ_KIVI ? launch_tc_v<4, KVQ_KIVI>(a, num_sms, st)
                              : launch_tc_v<4, KVQ_INNERQ>(a, num_sms, st);
}

}  // namespace kvq
