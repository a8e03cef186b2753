// The tensor-core MHA decode kernel and its launch templates, shared by the
// translation units that instantiate them (fp32 statistics:
// kvq_decode_tc.cu; fp16 statistics: kvq_decode_tc16.cu).  See
// kvq_decode_tc.cu for the design.
#pragma once

#include "kvq_rope.cuh"
#include "kvq_tc_common.cuh"

namespace kvq {

namespace {


// Work units: a quantized tile is one unit, an fp16 chunk kChunkUnits (its
// dot products run on the CUDA cores in a long dependent chain), and every
// head starts with kHeadUnits units that hold no data.  They fall to the
// warp that holds the head's first unit: the warp that changes heads there
// and merges the head's partials at the end, both costs of about a tile.
constexpr int kHeadUnits = 2;
constexpr int kChunkUnits = 2;
constexpr int kMinWarpUnits = 6;

// Counters of head bh: the launch's, or (per-sequence lengths) its
// sequence's own; nf = fp16 tokens (sinks + residual / window), nvq = tokens
// whose values are quantized (the value queue keeps [nvq, nq) in fp16).
struct HeadCnt {
  int nq, nf, ns, nvq;
};
// The counters of a sequence with n = prompt + appended tokens: counts_of's
// rules in 32-bit arithmetic (a cache holds at most 2^30 tokens).
__device__ __forceinline__ HeadCnt seq_cnt(const Geometry &g, int n) {
  if (g.scheme == KVQ_KIVI) {
    const int nr = n % g.residual;
    return HeadCnt{n - nr, nr, 0, g.vq ? (n >= g.residual ? n - g.residual + 1 : 0) : n - nr};
  }
  const int ns = min(n, g.n_sink), rest = n - ns, nr = min(rest, g.residual);
  return HeadCnt{rest - nr, nr + ns, ns, rest - nr};
}
template <int EXT>
__device__ __forceinline__ HeadCnt head_cnt(const TcArgs &a, int bh) {
  if (!EXT || !a.g.ragged) return HeadCnt{(int)a.n_quant, (int)a.n_fp16, (int)a.n_sink, (int)a.n_vq};
  return seq_cnt(a.g, a.p.seq_prompt[bh / a.g.H] + (int)a.p.appended);
}

// What unit range [x0, x1) holds of head bh: its U units are HU empty ones,
// S_h quantized tiles of kTile tokens, then F_h = nch * UPC fp16 units; a
// chunk belongs to the warp that holds its first unit.  (Per-sequence lengths:
// the unit layout is the longest sequence's, with room for the most fp16
// tokens a sequence can hold; a shorter head's units past its own tokens are
// empty.)
template <int EXT>
__device__ __forceinline__ Seg warp_seg(const TcArgs &a, const HeadCnt &hc, int bh, int x0,
                                        int x1) {
  Seg s;
  const int base = bh * a.U;
  const int ua = max(x0, base) - base, ub = min(x1, base + a.U) - base;
  const int qa = max(ua - a.HU, 0), qb = min(ub - a.HU, a.S_h);
  const int fa = max(ua - a.HU - a.S_h, 0), fb = min(ub - a.HU - a.S_h, a.F_h);
  s.tq0 = qa * kTile;
  s.c0 = (fa + a.UPC - 1) / a.UPC;
  if (!EXT) {
    s.tq1 = qa < qb ? (int)min((int64_t)qb * kTile, a.n_quant) : s.tq0;
    s.c1 = fa < fb ? min((fb + a.UPC - 1) / a.UPC, a.nch) : s.c0;
  } else {
    const int nch = (hc.nf + a.CH - 1) / a.CH;
    s.tq1 = qa < qb ? max(min(qb * kTile, hc.nq), s.tq0) : s.tq0;
    s.c1 = fa < fb ? max(min((fb + a.UPC - 1) / a.UPC, nch), s.c0) : s.c0;
  }
  return s;
}

// Per-sequence lengths (the extended kernel): every head holds only its own
// sequence's tiles and chunks -- kHeadUnits empty units, S quantized tiles,
// F = chunks * UPC fp16 units -- heads in batch order, so the warps' equal
// ranges are equal work (with the uniform layout every head would take the
// longest sequence's units).  A head's first unit is a prefix sum over the
// batch that each warp takes itself (ragged_locate); its span follows from
// that and its counters.
struct HeadSpan {
  int base, U, S, F;
};

template <int EXT>
__device__ __forceinline__ HeadSpan span_at(const TcArgs &a, int base, const HeadCnt &hc) {
  if (!EXT) return HeadSpan{base, a.U, a.S_h, a.F_h};
  const int S = (hc.nq + kTile - 1) / kTile, F = (hc.nf + a.CH - 1) / a.CH * a.UPC;
  return HeadSpan{base, a.HU + S + F, S, F};
}

// Units of one head of sequence b.
__device__ __forceinline__ int seq_units(const TcArgs &a, int b) {
  const HeadCnt c = seq_cnt(a.g, a.p.seq_prompt[b] + (int)a.p.appended);
  return a.HU + (c.nq + kTile - 1) / kTile + (c.nf + a.CH - 1) / a.CH * a.UPC;
}

// Run by the whole warp: the units of every head (`total`) and, for x >= 0,
// the head bh that holds unit x and its first unit (returned).
__device__ int ragged_locate(const TcArgs &a, int x, int &bh, int &total) {
  const int lane = threadIdx.x & 31, B = a.g.B, H = a.g.H;
  int base = 0;
  bh = -1;
  int acc = 0;  // units of the sequences before this round
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int uh = b < B ? seq_units(a, b) : 0;
    const int ub = H * uh;  // units of sequence b, all its heads
    int inc = ub;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    const int tot = __shfl_sync(0xffffffffu, inc, 31);
    if (bh < 0 && x >= acc && x < acc + tot) {  // (warp-uniform)
      const int L = __ffs(__ballot_sync(0xffffffffu, acc + inc > x)) - 1;
      const int start = acc + __shfl_sync(0xffffffffu, inc - ub, L);
      const int U = __shfl_sync(0xffffffffu, uh, L);
      const int h = (x - start) / U;
      bh = (b0 + L) * H + h;
      base = start + h * U;
    }
    acc += tot;
  }
  total = acc;
  return base;
}

// The extended kernel's unit layout for warp gw: the units' total, the
// working warps (every one owns at least one unit, so the warps touching a
// head are consecutive: its partial slots), the warp's range, its first and
// last heads and the first unit of the first.  Uniform lengths: the launch's.
struct ExtRange {
  int total, nw, x0, x1, bh_first, bh_last, base_first;
};
__device__ ExtRange ext_range(const TcArgs &a, int gw) {
  ExtRange r;
  r.total = a.total;
  r.nw = a.nw;
  int t_;
  if (a.g.ragged && a.g.B <= 32) {
    // one pass: lane b holds sequence b's units; their prefix sum gives the
    // total, then both ends of the warp's range
    const int lane = threadIdx.x & 31, H = a.g.H;
    const int uh = lane < a.g.B ? seq_units(a, lane) : 0, ub = H * uh;
    int inc = ub;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    r.total = __shfl_sync(0xffffffffu, inc, 31);
    r.nw = min(a.nw, r.total);
    r.x0 = (int)((int64_t)gw * r.total / r.nw);
    r.x1 = (int)((int64_t)(gw + 1) * r.total / r.nw);
    if (gw >= r.nw) return r;
    auto head_of = [&](int x, int &bh) {
      const int L = __ffs(__ballot_sync(0xffffffffu, inc > x)) - 1;
      const int start = __shfl_sync(0xffffffffu, inc - ub, L);
      const int U = __shfl_sync(0xffffffffu, uh, L);
      const int h = (x - start) / U;
      bh = L * H + h;
      return start + h * U;
    };
    r.base_first = head_of(r.x0, r.bh_first);
    head_of(r.x1 - 1, r.bh_last);
    return r;
  }
  if (a.g.ragged) {
    ragged_locate(a, -1, r.bh_first, r.total);
    r.nw = min(a.nw, r.total);
  }
  r.x0 = (int)((int64_t)gw * r.total / r.nw);
  r.x1 = (int)((int64_t)(gw + 1) * r.total / r.nw);
  if (gw >= r.nw) return r;
  if (a.g.ragged) {
    r.base_first = ragged_locate(a, r.x0, r.bh_first, t_);
    ragged_locate(a, r.x1 - 1, r.bh_last, t_);
  } else {
    r.bh_first = r.x0 / a.U;
    r.bh_last = (r.x1 - 1) / a.U;
    r.base_first = r.bh_first * a.U;
  }
  return r;
}

// warp_seg for a head whose first unit is head_base (the extended kernel).
template <int EXT>
__device__ __forceinline__ Seg warp_seg_at(const TcArgs &a, const HeadCnt &hc, int head_base,
                                           int x0, int x1) {
  const HeadSpan hs = span_at<EXT>(a, head_base, hc);
  Seg s;
  const int base = hs.base;
  const int ua = max(x0, base) - base, ub = min(x1, base + hs.U) - base;
  const int qa = max(ua - a.HU, 0), qb = min(ub - a.HU, hs.S);
  const int fa = max(ua - a.HU - hs.S, 0), fb = min(ub - a.HU - hs.S, hs.F);
  const int nch = (hc.nf + a.CH - 1) / a.CH;
  s.tq0 = qa * kTile;
  s.c0 = (fa + a.UPC - 1) / a.UPC;
  s.tq1 = qa < qb ? max(min(qb * kTile, hc.nq), s.tq0) : s.tq0;
  s.c1 = fa < fb ? max(min((fb + a.UPC - 1) / a.UPC, nch), s.c0) : s.c0;
  return s;
}

// OUT = 1: the extended kernel -- per-sequence lengths, the value queue and
// outlier lists, each a run-time option; OUT = 2: per-sequence lengths only;
// OUT = 0 compiles none of them.
// RP = 1: the rotary form (keys cached before RoPE; KIVI, key groups of 32 or
// more, fp32 statistics, no options): key scores on the CUDA cores, one token
// per lane, the rest as above.
template <int BITS, int SCHEME, int NGV, int NGK, int KM, int MF, int OUT, int RP = 0>
__global__ void __launch_bounds__(kThreads, 2) tc_decode_kernel(const TcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using SC = SlotCfg<BITS, SCHEME, NGV, NGK, KM, MF, OUT, RP>;
  static_assert(!RP || (SCHEME == KVQ_KIVI && KM <= 1 && MF == 0 && OUT == 0),
                "the rotary form: KIVI, one key group per tile, fp32 statistics, no options");
  // OUT: 0 = no options; 1 = outlier lists and the value queue compiled in
  // (and per-sequence lengths, if the cache has them); 2 = per-sequence
  // lengths only.  XO: the outlier and value-queue code.
  constexpr bool XO = OUT == 1;
  constexpr bool G16 = SCHEME == KVQ_KIVI && KM == 2;
  constexpr int RB = SC::RB;  // packed bytes per token row
  constexpr int nslot = SC::nslot;
  constexpr int SLOT = SC::bytes;
  const Geometry &g = a.g;
  constexpr TcLayout Ly = tc_layout(SLOT, nslot, SC::SBB, SC::CSB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  grid_dep_trigger();  // the next decode's blocks may take the SMs this grid leaves
  // The rotary form's table: entry [L][j] = (cos j theta_2L, cos j theta_2L+1,
  // sin j theta_2L, sin j theta_2L+1) for token offsets j < 32 (pair-pair L =
  // channels 4L .. 4L + 3), built once by the block.
  const float4 *cs_tab = reinterpret_cast<const float4 *>(smem);
  if constexpr (RP != 0) {
    float4 *tab = reinterpret_cast<float4 *>(smem);
    for (int i = tid; i < 32 * 32; i += kThreads) {
      const int L = i >> 5, j = i & 31;
      const float2 r0 = rope_cos_sin((float)j, a.theta[2 * L], a.c1, a.c2, a.c3);
      const float2 r1 = rope_cos_sin((float)j, a.theta[2 * L + 1], a.c1, a.c2, a.c3);
      tab[i] = make_float4(r0.x, r1.x, r0.y, r1.y);
    }
    __syncthreads();
  }
  uint8_t *wring = smem + Ly.ring + warp * nslot * SLOT;
  uint64_t *wbars = reinterpret_cast<uint64_t *>(smem + Ly.bars) + warp * (nslot + 1);
  uint32_t *sBw = reinterpret_cast<uint32_t *>(smem + Ly.sB + warp * SC::SBB);
  const uint32_t wring_s = smem_u32(wring), wbars_s = smem_u32(wbars);  // shared-window addresses

  // Warp-level stream-K: logical warp gw owns units [x0, x1) of the
  // concatenated per-head unit lists (units of one tile or fp16 chunk).
  // When fewer warps than the grid holds have work, logical warps go
  // round-robin over the blocks, so every SM gets about the same number.
  const int gw = a.nw < (int)gridDim.x * kWarps ? warp * (int)gridDim.x + (int)blockIdx.x
                                                : (int)blockIdx.x * kWarps + warp;
  if (gw >= a.nw) return;
  // (OUT: per-sequence lengths lay the heads out by their own units)
  ExtRange rx{};
  if constexpr (OUT != 0) {
    grid_dep_wait();  // the per-sequence counters are device data
    rx = ext_range(a, gw);
    if (gw >= rx.nw) return;
  }
  const int x0 = OUT ? rx.x0 : (int)((int64_t)gw * a.total / a.nw);
  const int x1 = OUT ? rx.x1 : (int)((int64_t)(gw + 1) * a.total / a.nw);
  const int bh_first = OUT ? rx.bh_first : x0 / a.U, bh_last = OUT ? rx.bh_last : (x1 - 1) / a.U;
  // fp16 tokens per chunk: a chunk's K and V rows fill the slot up to the
  // query (with outlier lists the block size, so CH, is a run-time value)
  const int CH = XO ? a.CH : SC::CH;
  const int BBr = XO ? g.block_bytes : SC::BB;  // bytes of a cache block
  const int n_out = XO ? g.n_out : 0;
  float *qf_s = reinterpret_cast<float *>(sBw + SC::sb_xtra);  // OUT: q, score domain
  float *xo_s = qf_s + kD;  // OUT: outliers' value corrections, m_run frame

  // Each warp owns its ring and barriers; nothing below synchronises warps.
  // Ring bytes are only read where a copy wrote them (rows past a segment's
  // end are masked), so the ring needs no clearing; the zero block does.
  if (lane < 16) sBw[SC::sb_zero + lane] = 0u;
  if (XO)
#pragma unroll
    for (int i = 0; i < 4; ++i) xo_s[4 * lane + i] = 0.0f;
  if (lane == 0) {
    for (int s = 0; s <= nslot; ++s) bar_init(&wbars[s], 1);  // [nslot]: never completed
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();

  // ---- producer: this warp's items in the order the consumer visits them:
  // per head, its quantized tiles, then its fp16 chunks.
  int pc_bh = bh_first, pc_ph = 0, pc_lt = 0, pc_n = 0, issued = 0, ps = 0;
  const uint64_t pol_once = l2_evict_first();  // cache blocks are read once
  HeadCnt pc_hc = head_cnt<OUT>(a, pc_bh);
  int pc_base = OUT ? rx.base_first : 0;  // (OUT) first unit of head pc_bh
  Seg pc_seg = OUT ? warp_seg_at<OUT>(a, pc_hc, pc_base, x0, x1)
                   : warp_seg<OUT>(a, pc_hc, pc_bh, x0, x1);
  pc_n = (pc_seg.tq1 - pc_seg.tq0 + kTile - 1) / kTile;
  auto pc_settle = [&]() {
    while (pc_bh >= 0 && pc_lt >= pc_n) {
      if (pc_ph == 0) {
        pc_ph = 1;
        pc_n = pc_seg.c1 - pc_seg.c0;
      } else {
        if constexpr (OUT != 0) pc_base += span_at<OUT>(a, pc_base, pc_hc).U;
        if (++pc_bh > bh_last) {
          pc_bh = -1;
          return;
        }
        pc_ph = 0;
        pc_hc = head_cnt<OUT>(a, pc_bh);
        pc_seg = OUT ? warp_seg_at<OUT>(a, pc_hc, pc_base, x0, x1)
                     : warp_seg<OUT>(a, pc_hc, pc_bh, x0, x1);
        pc_n = (pc_seg.tq1 - pc_seg.tq0 + kTile - 1) / kTile;
      }
      pc_lt = 0;
    }
  };
  // Called by the whole warp; lane 0 posts the byte count and issues the
  // copies of the next item of this warp.  A quantized tile: its cache block
  // and, for KIVI G >= 64, its key group's statistics.  An fp16 chunk: its K
  // rows, then its V rows (sink rows before residual / window rows).  The
  // query row rides along with the warp's first item of each phase of a head.
  auto issue_next = [&]() {
    if (pc_bh < 0) return;
    const bool first = pc_lt == 0;
    uint8_t *dst = wring + ps * SLOT;
    uint64_t *bar = &wbars[ps];
    const uint32_t dst_s = wring_s + ps * SLOT, bar_s = wbars_s + 8 * ps;
    ps = ps + 1 == nslot ? 0 : ps + 1;
    if (pc_ph == 0) {
      // a cache block: the common case, issued without a branch on the lane
      const int tok0 = pc_seg.tq0 + kTile * pc_lt;
      bulk_g2s_pred(lane == 0, bar_s, (uint32_t)(BBr + SC::KMB + (first ? kD * 2 : 0)), dst_s,
                    a.p.blocks + ((int64_t)pc_bh * (g.cap / kTile) + tok0 / kTile) * BBr, BBr,
                    pol_once);
      if (SCHEME == KVQ_KIVI && !SC::KIN && lane == 0)
        bulk_g2s(dst + SC::off_km,
                 a.p.k_meta + ((int64_t)pc_bh * g.k_meta_rows + tok0 / g.k_group) * 2 * kD * g.msz,
                 SC::KMB, bar);
      if (first && lane == 0)
        bulk_g2s(dst + SC::off_q, a.q + ((int64_t)(pc_bh / g.H) * g.Hq + pc_bh % g.H) * kD, kD * 2,
                 bar);
    } else if (lane == 0) {
      const __half *qrow = a.q + ((int64_t)(pc_bh / g.H) * g.Hq + pc_bh % g.H) * kD;
      const int ns = pc_hc.ns;
      const int i0 = (pc_seg.c0 + pc_lt) * CH, i1 = min(i0 + CH, pc_hc.nf);
      const int s0 = min(i0, ns), s1 = min(i1, ns);            // sink rows
      const int r0 = max(i0, ns) - ns, r1 = max(i1, ns) - ns;  // residual / window rows
      bar_expect_tx(bar, (uint32_t)(2 * (i1 - i0) * kD * 2 + (first ? kD * 2 : 0)));
      if (s1 > s0) {
        const int64_t row = (int64_t)pc_bh * g.n_sink + s0;
        bulk_g2s(dst, a.p.k_sink + row * kD, (uint32_t)((s1 - s0) * kD * 2), bar);
        bulk_g2s(dst + CH * kD * 2, a.p.v_sink + row * kD, (uint32_t)((s1 - s0) * kD * 2), bar);
      }
      if (r1 > r0) {
        // a fused append's new row is not in the residual yet: it comes from
        // the step's input rows
        const int rn = (a.new_row >= 0 && r1 - 1 == a.new_row) ? r1 - 1 : r1;
        const int64_t row = (int64_t)pc_bh * g.residual + r0;
        const int o = (s1 - s0) * kD * 2;
        if (rn > r0) {
          bulk_g2s(dst + o, a.p.k_res + row * kD, (uint32_t)((rn - r0) * kD * 2), bar);
          bulk_g2s(dst + CH * kD * 2 + o, a.p.v_res + row * kD,
                   (uint32_t)((rn - r0) * kD * 2), bar);
        }
        if (rn < r1) {
          const int on = o + (rn - r0) * kD * 2;
          bulk_g2s(dst + on, a.k_new + (int64_t)pc_bh * kD, kD * 2, bar);
          bulk_g2s(dst + CH * kD * 2 + on, a.v_new + (int64_t)pc_bh * kD, kD * 2, bar);
        }
      }
      if (first) bulk_g2s(dst + SC::off_q, qrow, kD * 2, bar);
    }
    ++issued;
    ++pc_lt;
    pc_settle();
  };
  pc_settle();
  // the previous grid on the stream has drained: device data from here on
  // (under per-sequence lengths the wait came before the counters' reads)
  if constexpr (OUT == 0) grid_dep_wait();
  for (int s = 0; s < nslot; ++s) issue_next();

  // ---- per-head constants (each warp for itself) --------------------------
  float pow2E = 1.0f;  // scores = raw * 2^(E+24) (q normalised by 2^-E, codes by 2^-24)
  float q4[4];         // q of channels 4*lane .. 4*lane+3 (exp2 domain)
  // KIVI key operand: this lane builds the channel pairs (c, c + kHalf) of
  // c = b_clo and c = b_clo + 1 (even positions p and p + 1 of word W), whose
  // B-fragment words sit next to each other at b_sidx, b_sidx + 1
  constexpr int kHalf = BITS == 2 ? 8 : 4;  // channel offset of the high half of a pair
  int b_clo, b_sidx;
  float qn_lo[2], qn_hi[2], qf_lo[2], qf_hi[2];
  {
    int W, p, tg, kb;
    if (BITS == 2) {
      W = lane >> 2;
      p = 2 * (lane & 3);
      b_clo = 16 * W + p;
      tg = W >> 1;
      kb = 4 * (W & 1) + (p >> 1);
    } else {
      W = lane >> 1;
      p = 2 * (lane & 1);
      b_clo = 8 * W + p;
      tg = W >> 2;
      kb = 2 * (W & 3) + (p >> 1);
    }
    b_sidx = tg * 16 + kb * 2;
#pragma unroll
    for (int r = 0; r < 2; ++r) qn_lo[r] = qn_hi[r] = qf_lo[r] = qf_hi[r] = 0.0f;
  }
  // InnerQ: fixed key operand and per-group sums of q
  uint32_t bqi[8][2];
  float Qj[NGK];

  // Per-head constants from the query row that rode along with the head's
  // first tile of this warp.
  auto start_head = [&](const uint8_t *slot, int cur_bh) {
    const __half *qh = reinterpret_cast<const __half *>(slot + SC::off_q);
    const uint2 qr = reinterpret_cast<const uint2 *>(qh)[lane];
    const float2 q01 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.x));
    const float2 q23 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.y));
    q4[0] = q01.x * a.scale_log2;
    q4[1] = q01.y * a.scale_log2;
    q4[2] = q23.x * a.scale_log2;
    q4[3] = q23.y * a.scale_log2;
    // InnerQ with normalized keys: the per-channel factors go into q (the
    // quantized tokens only; the fp16 rows reload the raw query)
    const float *knr = SCHEME == KVQ_INNERQ && g.knorm ? a.p.k_norm + (int64_t)cur_bh * kD : nullptr;
    if (knr) {
      const float4 n4 = reinterpret_cast<const float4 *>(knr)[lane];
      q4[0] *= n4.x;
      q4[1] *= n4.y;
      q4[2] *= n4.z;
      q4[3] *= n4.w;
    }
    if (XO) {
      // the query in the score domain, for the outliers' key corrections
      __syncwarp();
      reinterpret_cast<float4 *>(qf_s)[lane] = make_float4(q4[0], q4[1], q4[2], q4[3]);
      __syncwarp();
    }
    float mx = fmaxf(fmaxf(fabsf(q4[0]), fabsf(q4[1])), fmaxf(fabsf(q4[2]), fabsf(q4[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    int E = 0;
    if (mx > 0.0f && mx < INFINITY) frexpf(mx, &E);
    pow2E = ldexpf(1.0f, E) * kSub;
    const float inv = ldexpf(1.0f, -E);
    auto qf = [&](int c) { return __half2float(qh[c]) * a.scale_log2 * (knr ? knr[c] : 1.0f); };
    if (SCHEME == KVQ_KIVI) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int c = b_clo + r;
        const int p = BITS == 2 ? (c & 7) : (c & 3);
        const float invf = inv * inv_pos_factor<BITS>(p);
        qf_lo[r] = qf(c);
        qf_hi[r] = qf(c + kHalf);
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
          const float invf = inv * inv_pos_factor<BITS>(p);
          const float vlo = (clo / GK == jn) ? qf(clo) * invf : 0.0f;
          const float vhi = (chi / GK == jn) ? qf(chi) * invf : 0.0f;
          uint32_t hi, lo;
          split2(vlo, vhi, hi, lo);
          bqi[kb][r] = gid < 2 * NGK ? (part ? lo : hi) : 0u;
        }
    }
  };

  // ---- the rotary form's key scores (RP) -------------------------------------
  // Token t (lane t) of the tile at `slot`, token 0 at position tok0: with the
  // anchor A = R(qpos - tok0) q, score = k_t . R(-t) A, and per channel pair
  // (a, b) that is cos(t theta) X + sin(t theta) Y with X = k_a A_a + k_b A_b,
  // Y = k_a A_b - k_b A_a (the rotation moved onto the query: RoPE rotations
  // compose).  Lane L first writes the weights of its pair-pair L (channels
  // 4L .. 4L + 3) into the warp's area, the dequantization k = code * scale +
  // zero folded in; then every lane runs its own token through the 32
  // pair-pairs, two pairs per packed instruction.  A code is read in place:
  // masked inside its 16-bit half and OR-ed into the mantissa of 2^23, minus
  // 2^23, the code at bit offset o reads as code * 2^o; the weights carry 2^-o.
  auto rope_score = [&](const uint8_t *slot, int t, int tok0) -> float {
    float4 *wt = reinterpret_cast<float4 *>(sBw);
    auto pow2i = [](int e) { return __int_as_float((127 + e) << 23); };
    {
      const float delta0 = (float)(a.qpos - tok0);
      const float2 r0 = rope_cos_sin(delta0, a.theta[2 * lane], a.c1, a.c2, a.c3);
      const float2 r1 = rope_cos_sin(delta0, a.theta[2 * lane + 1], a.c1, a.c2, a.c3);
      const float a0a = r0.x * q4[0] - r0.y * q4[1], a0b = r0.y * q4[0] + r0.x * q4[1];
      const float a1a = r1.x * q4[2] - r1.y * q4[3], a1b = r1.y * q4[2] + r1.x * q4[3];
      const float4 sc4 = reinterpret_cast<const float4 *>(slot + SC::off_km)[lane];
      const float4 zr4 = reinterpret_cast<const float4 *>(slot + SC::off_km + kD * 4)[lane];
      const int o = BITS == 2 ? 8 * (lane & 1) : 0;  // offset of channel 4L in its half
      const float f0 = pow2i(-o), f1 = pow2i(-(o + BITS));
      const float f2 = pow2i(-(o + 2 * BITS)), f3 = pow2i(-(o + 3 * BITS));
      // [L]: X weights of the a channels (pairs 2L, 2L + 1), then of the b
      // channels; [32 + L]: the same for Y; [64 + L]: the zeros' X, Y terms
      wt[lane] = make_float4(sc4.x * a0a * f0, sc4.z * a1a * f2, sc4.y * a0b * f1, sc4.w * a1b * f3);
      wt[32 + lane] =
          make_float4(sc4.x * a0b * f0, sc4.z * a1b * f2, -(sc4.y * a0a) * f1, -(sc4.w * a1a) * f3);
      wt[64 + lane] = make_float4(fmaf(zr4.x, a0a, zr4.y * a0b), fmaf(zr4.z, a1a, zr4.w * a1b),
                                  fmaf(zr4.x, a0b, -(zr4.y * a0a)), fmaf(zr4.z, a1b, -(zr4.w * a1a)));
      __syncwarp();
    }
    constexpr int NW = SC::RB / 4;  // code words of a token row
    uint32_t wd[NW];
    const uint4 *row = reinterpret_cast<const uint4 *>(slot + t * SC::RB);
#pragma unroll
    for (int v = 0; v < NW / 4; ++v) {
      const uint4 x = row[v];
      wd[4 * v] = x.x;
      wd[4 * v + 1] = x.y;
      wd[4 * v + 2] = x.z;
      wd[4 * v + 3] = x.w;
    }
    constexpr uint32_t M = (1u << BITS) - 1u;
    const uint32_t magic = 0x4B000000u;  // 2^23
    const float2 unmagic = make_float2(-8388608.0f, -8388608.0f);
    const float4 *cst = cs_tab + t;
    // four independent accumulators (pair-pairs L mod 4) keep the dependent
    // chains short; each step's shared loads are issued a step ahead
    float2 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.0f, 0.0f);
    float4 wa = wt[0], wb = wt[32], wz = wt[64], c = cst[0];
#pragma unroll
    for (int L = 0; L < 32; ++L) {
      float4 wa_n, wb_n, wz_n, c_n;
      if (L + 1 < 32) {
        wa_n = wt[L + 1];
        wb_n = wt[33 + L];
        wz_n = wt[65 + L];
        c_n = cst[32 * (L + 1)];
      }
      const int bit0 = 4 * L * BITS;  // first bit of channel 4L in the row
      const uint32_t w = wd[bit0 >> 5];
      const uint32_t h = (bit0 & 16) ? (w >> 16) : w;
      const int o = bit0 & 15;
      const float2 u = __fadd2_rn(make_float2(__uint_as_float(and_or(h, M << o, magic)),
                                              __uint_as_float(and_or(h, M << (o + 2 * BITS), magic))),
                                  unmagic);  // channels 4L, 4L + 2
      const float2 v = __fadd2_rn(make_float2(__uint_as_float(and_or(h, M << (o + BITS), magic)),
                                              __uint_as_float(and_or(h, M << (o + 3 * BITS), magic))),
                                  unmagic);  // channels 4L + 1, 4L + 3
      const float2 X = __ffma2_rn(u, make_float2(wa.x, wa.y),
                                  __ffma2_rn(v, make_float2(wa.z, wa.w), make_float2(wz.x, wz.y)));
      const float2 Y = __ffma2_rn(u, make_float2(wb.x, wb.y),
                                  __ffma2_rn(v, make_float2(wb.z, wb.w), make_float2(wz.z, wz.w)));
      acc[L & 3] = __ffma2_rn(make_float2(c.x, c.y), X, __ffma2_rn(make_float2(c.z, c.w), Y, acc[L & 3]));
      if (L + 1 < 32) {
        wa = wa_n;
        wb = wb_n;
        wz = wz_n;
        c = c_n;
      }
    }
    const float2 s01 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
    return s01.x + s01.y;
  };
  // The rotary form's fp16 rows: row tt of the chunk that starts at fp16
  // index i0 is the token at position n_quant + i0 + tt (KIVI keeps no
  // sinks).  Each lane turns the query by R(qpos - position) on its channels
  // 4 lane .. 4 lane + 3 and the warp sums; returns the score of row gid
  // (rows past nv: 0).
  auto rope_chunk_score = [&](const uint8_t *slot, int i0, int nv) -> float {
    const float2 th0 = a.theta[2 * lane], th1 = a.theta[2 * lane + 1];
    const uint2 *kr = reinterpret_cast<const uint2 *>(slot);
    float sp = 0.0f;
    for (int tt = 0; tt < nv; ++tt) {
      const uint2 kw = kr[tt * (kD / 4) + lane];
      const float2 k01 = __half22float2(*reinterpret_cast<const __half2 *>(&kw.x));
      const float2 k23 = __half22float2(*reinterpret_cast<const __half2 *>(&kw.y));
      const float delta = (float)(a.qpos - ((int)a.n_quant + i0 + tt));
      const float2 r0 = rope_cos_sin(delta, th0, a.c1, a.c2, a.c3);
      const float2 r1 = rope_cos_sin(delta, th1, a.c1, a.c2, a.c3);
      float x = fmaf(k01.x, r0.x * q4[0] - r0.y * q4[1], k01.y * (r0.y * q4[0] + r0.x * q4[1]));
      x = fmaf(k23.x, r1.x * q4[2] - r1.y * q4[3], fmaf(k23.y, r1.y * q4[2] + r1.x * q4[3], x));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      sp = gid == tt ? x : sp;
    }
    return sp;
  };

  // ---- per-warp online-softmax state ----------------------------------------
  float m_run = -INFINITY, l_lane = 0.0f, z_lane[NGV];
  float dv[8][4];
  // value queue: p_t * v_t of tokens whose key is quantized but whose value
  // is still fp16 (channels 4*lane .. 4*lane + 3, m_run frame)
  float xv[4];
  auto reset_state = [&]() {
    m_run = -INFINITY;
    l_lane = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < NGV; ++j) z_lane[j] = 0.0f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) dv[mt][r] = 0.0f;
  };
  reset_state();

  // Warp state -> partial `slot` of head bh.  The quantized-token state
  // (online softmax over MMA fragments; lanes hold one token each for l and
  // z) and the fp16-token state (mf, lf, af: a lane owns channels 4*lane ..
  // 4*lane + 3) are joined with the log-sum-exp rule; the quantized output
  // row goes through the warp's operand area to reach the lane layout.
  int pend_bh = -1;  // head this warp merges (slot 0), once it has published
  int pend_np = 0, cur_np = 0;  // (OUT) its partial count, the current head's
  auto flush = [&](int bh, int slot, float mf, float lf, const float (&af)[4]) -> bool {
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
    float *so = reinterpret_cast<float *>(sBw);
    const int gc = (gid * NGV) >> 3;  // value group of this thread's 16 channels
    if (tig == gc) {
      float zc = Z[0];
#pragma unroll
      for (int j = 1; j < NGV; ++j)
        if (j == gc) zc = Z[j];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float invf = kSub * kSlackScale / pos_factor<BITS>(BITS == 2 ? mt : (mt & 3));
        so[16 * gid + mt] = fmaf(dv[mt][0] + dv[mt][1], invf, zc);
        so[16 * gid + 8 + mt] = fmaf(dv[mt][2] + dv[mt][3], invf, zc);
      }
    }
    __syncwarp();
    float4 oq = reinterpret_cast<const float4 *>(so)[lane];
    if (XO) {
      oq.x += xv[0];
      oq.y += xv[1];
      oq.z += xv[2];
      oq.w += xv[3];
      // the outliers' value corrections (every lane's atomics are done)
      const float4 xo = reinterpret_cast<const float4 *>(xo_s)[lane];
      oq.x += xo.x;
      oq.y += xo.y;
      oq.z += xo.z;
      oq.w += xo.w;
      reinterpret_cast<float4 *>(xo_s)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncwarp();
    const float m = fmaxf(m_run, mf);
    const float wq = m_run == -INFINITY ? 0.0f : exp2_approx(m_run - m);
    const float wf = mf == -INFINITY ? 0.0f : exp2_approx(mf - m);
    float4 o;
    o.x = fmaf(oq.x, wq, af[0] * wf);
    o.y = fmaf(oq.y, wq, af[1] * wf);
    o.z = fmaf(oq.z, wq, af[2] * wf);
    o.w = fmaf(oq.w, wq, af[3] * wf);
    const float lt = fmaf(l, wq, lf * wf);
    reset_state();
    // a merge still owed (a head this warp held whole) comes first; the
    // merge of the warp's last head waits until after the tile loop
    if (pend_bh >= 0 && !merge_head<8>(a, pend_bh, OUT ? pend_np : -1)) return false;
    publish_partial(a, bh, slot, o, m, lt);
    pend_bh = slot == 0 ? bh : -1;
    if constexpr (OUT != 0) pend_np = cur_np;
    return true;
  };

  int done = 0;          // items whose copies completed
  int cs = 0;            // ring slot of the next item
  uint32_t cph = 0;      // its barrier phase parity
  // Waits for the next ring slot.  One verdict per warp: every lane takes
  // the same path; false (status word set) on timeout.
  auto wait_slot = [&](int &s_out) -> bool {
    const int s = cs;
    const uint32_t par = cph;
    if (++cs == nslot) {
      cs = 0;
      cph ^= 1u;
    }
    const bool ok = bar_wait(wbars_s + 8 * s, par, a.wait_limit);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
      return false;
    }
    ++done;
    s_out = s;
    return true;
  };
  bool aborted = false;
  if (a.stall_limit > 0) {
    // debug: the warp's first wait is on a barrier nothing completes
    const bool ok = bar_wait(&wbars[nslot], 0u, a.stall_limit);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
      aborted = true;
    }
  }
  int base_t = OUT ? rx.base_first : 0;  // (OUT) first unit of head bh
  for (int bh = bh_first; bh <= bh_last && !aborted; ++bh) {
    const HeadCnt hc = head_cnt<OUT>(a, bh);
    const Seg sg = OUT ? warp_seg_at<OUT>(a, hc, base_t, x0, x1)
                       : warp_seg<OUT>(a, hc, bh, x0, x1);
    const int tq0 = sg.tq0, tq1 = sg.tq1;
    // fp16 sink + residual / window chunks of this warp's segment
    const int nchk = sg.c1 - sg.c0;
    const int base = OUT ? base_t : bh * a.U;
    if (tq1 > tq0) {
      const int nt = (tq1 - tq0 + kTile - 1) / kTile;
      for (int lt = 0; lt < nt; ++lt) {
        int s;
        if (!wait_slot(s)) {
          aborted = true;
          break;
        }
        const uint8_t *slot = wring + s * SLOT;
        if (lt == 0) start_head(slot, bh);
        const int tok0 = tq0 + kTile * lt;
        const int n = min(kTile, tq1 - tok0);
        auto tile = [&](auto full_c) {
          constexpr bool FULL = decltype(full_c)::value;
          const uint8_t *vc = slot + SC::off_vc;
          const int t = lane;
          float score;
          if constexpr (RP != 0) {
            score = rope_score(slot, t, tok0);
          } else {
            const uint8_t *kc = slot;
            // ------------- keys: two 16-token MMA tiles ------------------------
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            float bias0 = 0.0f, bias1 = 0.0f;
            // key operand words of MMA k-block kb for key group gl (loaded next
            // to their use to keep few registers live)
            auto bk_at = [&](int gl, int kb) -> uint2 {
              if (SCHEME == KVQ_KIVI) {
                // lanes of columns >= 2 read the zero block: no divergent branch
                const uint32_t *src = gid < 2 ? sBw + gl * 128 + (gid * 4 + tig) * 16 : sBw + SC::sb_zero;
                return *reinterpret_cast<const uint2 *>(src + 2 * kb);
              } else {
                return make_uint2(bqi[kb][0], bqi[kb][1]);
              }
            };
            bool two_groups = false;
            if (SCHEME == KVQ_KIVI) {
              // q~ = q * scale (normalised, position factor divided out) as fp16
              // hi/lo in B-fragment order, and q . zero, per key group of the tile
              const uint8_t *km = slot + SC::off_km;
              two_groups = G16 && (FULL || n > 16);
    #pragma unroll
              for (int gl = 0; gl < (G16 ? 2 : 1); ++gl) {
                if (gl == 1 && !two_groups) break;
                const uint8_t *ks = km + gl * 2 * kD * SC::MSZ, *kz = ks + kD * SC::MSZ;
                const float2 s_lo = ld_stat2<MF>(ks, b_clo);
                const float2 s_hi = ld_stat2<MF>(ks, b_clo + kHalf);
                const float2 z_lo = ld_stat2<MF>(kz, b_clo);
                const float2 z_hi = ld_stat2<MF>(kz, b_clo + kHalf);
                uint32_t h0, l0, h1, l1;
                split2(qn_lo[0] * s_lo.x, qn_hi[0] * s_hi.x, h0, l0);
                split2(qn_lo[1] * s_lo.y, qn_hi[1] * s_hi.y, h1, l1);
                *reinterpret_cast<uint2 *>(sBw + gl * 128 + b_sidx) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(sBw + gl * 128 + 64 + b_sidx) = make_uint2(l0, l1);
                float bz = fmaf(qf_lo[0], z_lo.x, fmaf(qf_hi[0], z_hi.x, fmaf(qf_lo[1], z_lo.y, qf_hi[1] * z_hi.y)));
    #pragma unroll
                for (int off = 16; off > 0; off >>= 1) bz += __shfl_xor_sync(0xffffffffu, bz, off);
                if (gl == 0) bias0 = bz;
                bias1 = bz;
              }
              __syncwarp();
            }
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
                    const uint2 b = bk_at(0, 4 * m + j);
                    mma16816(d0, ext<2>(w00, s00, 2 * j), ext<2>(w01, s01, 2 * j),
                             ext<2>(w00, s00, 2 * j + 1), ext<2>(w01, s01, 2 * j + 1), b.x, b.y);
                    mma16816(d1, ext<2>(w10, s10, 2 * j), ext<2>(w11, s11, 2 * j),
                             ext<2>(w10, s10, 2 * j + 1), ext<2>(w11, s11, 2 * j + 1), b.x, b.y);
                  }
                }
              } else {
    #pragma unroll
                for (int t2 = 0; t2 < 2; ++t2) {
                  const uint2 wa = t2 ? wa1 : wa0, wb = t2 ? wb1 : wb0;
    #pragma unroll
                  for (int m = 0; m < 2; ++m) {
                    const uint32_t w0 = m ? wa.y : wa.x, w1 = m ? wb.y : wb.x;
                    const uint32_t s0 = shifted<2>(w0), s1 = shifted<2>(w1);
    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                      const uint2 b = bk_at(t2, 4 * m + j);
                      if (t2 == 0)
                        mma16816(d0, ext<2>(w0, s0, 2 * j), ext<2>(w1, s1, 2 * j),
                                 ext<2>(w0, s0, 2 * j + 1), ext<2>(w1, s1, 2 * j + 1), b.x, b.y);
                      else
                        mma16816(d1, ext<2>(w0, s0, 2 * j), ext<2>(w1, s1, 2 * j),
                                 ext<2>(w0, s0, 2 * j + 1), ext<2>(w1, s1, 2 * j + 1), b.x, b.y);
                    }
                  }
                }
              }
            } else {
              // 4-bit keys: G >= 32 always gives one key group per tile here
              // (the 4-bit group-16 case takes the same path with two groups)
    #pragma unroll
              for (int t2 = 0; t2 < 2; ++t2) {
                const int gl = two_groups ? t2 : 0;
                const uint4 wa = *reinterpret_cast<const uint4 *>(kc + (16 * t2 + gid) * RB + 16 * tig);
                const uint4 wb = *reinterpret_cast<const uint4 *>(kc + (16 * t2 + gid + 8) * RB + 16 * tig);
                const uint32_t A0[4] = {wa.x, wa.y, wa.z, wa.w}, A1[4] = {wb.x, wb.y, wb.z, wb.w};
    #pragma unroll
                for (int m = 0; m < 4; ++m) {
                  const uint32_t s0 = shifted<4>(A0[m]), s1 = shifted<4>(A1[m]);
    #pragma unroll
                  for (int j = 0; j < 2; ++j) {
                    const uint2 b = bk_at(gl, 2 * m + j);
                    if (t2 == 0)
                      mma16816(d0, ext<4>(A0[m], s0, 2 * j), ext<4>(A1[m], s1, 2 * j),
                               ext<4>(A0[m], s0, 2 * j + 1), ext<4>(A1[m], s1, 2 * j + 1), b.x, b.y);
                    else
                      mma16816(d1, ext<4>(A0[m], s0, 2 * j), ext<4>(A1[m], s1, 2 * j),
                               ext<4>(A0[m], s0, 2 * j + 1), ext<4>(A1[m], s1, 2 * j + 1), b.x, b.y);
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
              const uint8_t *ks = slot + SC::off_ks;
              const uint8_t *kz = slot + SC::off_kz;
              const int jj = tig < NGK ? tig : NGK - 1;
              float qj = Qj[0];
    #pragma unroll
              for (int j = 1; j < NGK; ++j)
                if (j == jj) qj = Qj[j];
              auto term = [&](int row, float dd) {
                return fmaf(ld_stat<MF>(ks, row * NGK + jj), dd * pow2E,
                            ld_stat<MF>(kz, row * NGK + jj) * qj);
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
          
            const int src = 4 * (t & 7);
            const float xa0 = __shfl_sync(0xffffffffu, ra0, src), xb0 = __shfl_sync(0xffffffffu, rb0, src);
            const float xa1 = __shfl_sync(0xffffffffu, ra1, src), xb1 = __shfl_sync(0xffffffffu, rb1, src);
            score = t < 16 ? ((t & 8) ? xb0 : xa0) : ((t & 8) ? xb1 : xa1);
            if (SCHEME == KVQ_KIVI) score = fmaf(score, pow2E, t < 16 ? bias0 : bias1);
          }
          const bool valid = FULL || t < n;
          if (XO && valid) {
            // dense-and-sparse keys: an outlier's code is 0, so the dense score
            // holds q_c * zero_c there; its fp16 value replaces it
            const uint32_t *ol = reinterpret_cast<const uint32_t *>(slot + g.blk_ko) + t * n_out;
            const uint8_t *kz = slot + SC::off_km + ((G16 ? (t >> 4) : 0) * 2 + 1) * kD * SC::MSZ;
            for (int e = 0; e < n_out; ++e) {
              const uint32_t w = ol[e];
              const int c = (int)(w >> 16);
              const float v = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
              score = fmaf(qf_s[c], v - ld_stat<MF>(kz, c), score);
            }
          }
          score = valid ? score : -INFINITY;
          // value queue: tokens [vq_from, ...) of the head keep fp16 values
          const int vq_from = XO ? hc.nvq - tok0 : kTile;
          const bool valid_v = XO ? valid && t < vq_from : valid;
          // lazy rescaling: the reference m_run moves only when a score passes
          // it by more than kSlack (one vote, no reduction on most tiles)
          if (__any_sync(0xffffffffu, score > m_run + kSlack)) {
            float mt_ = score;
  #pragma unroll
            for (int off = 1; off < 32; off <<= 1) mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, off));
            const float alpha = exp2_approx(m_run - mt_);
            l_lane *= alpha;
  #pragma unroll
            for (int j = 0; j < NGV; ++j) z_lane[j] *= alpha;
            if (XO) {
  #pragma unroll
              for (int i = 0; i < 4; ++i) xv[i] *= alpha;
              __syncwarp();  // the previous tiles' corrections are in
  #pragma unroll
              for (int i = 0; i < 4; ++i) xo_s[4 * lane + i] *= alpha;
              __syncwarp();
            }
  #pragma unroll
            for (int mt = 0; mt < 8; ++mt)
  #pragma unroll
              for (int r = 0; r < 4; ++r) dv[mt][r] *= alpha;
            m_run = mt_;
          }
          const float p = exp2_approx(score - m_run);  // <= 2^kSlack
          const float pv = p * kInvSlack;          // value operand scale: stays in fp16 range
          l_lane += p;
          {
            float zr[NGV];
            ld_stat_row<MF, NGV>(slot + SC::off_vz + t * NGV * SC::MSZ, zr);
  #pragma unroll
            for (int j = 0; j < NGV; ++j)
              z_lane[j] = (XO ? valid_v : (FULL || p > 0.0f)) ? fmaf(p, zr[j], z_lane[j])
                                                                : z_lane[j];
            if (XO && valid_v) {
              // dense-and-sparse values: code 0 gave p * zero, the fp16 value
              // replaces it (channel c of an arbitrary lane: shared atomics)
              const uint32_t *ol = reinterpret_cast<const uint32_t *>(slot + g.blk_vo) + t * n_out;
              for (int e = 0; e < n_out; ++e) {
                const uint32_t w = ol[e];
                const int c = (int)(w >> 16);
                const float v = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
                float zc = zr[0];
  #pragma unroll
                for (int j = 1; j < NGV; ++j)
                  if (j == c / (kD / NGV)) zc = zr[j];
                atomicAdd(&xo_s[c], p * (v - zc));
              }
            }
          }
          if (XO && vq_from < n) {
            // (warp-uniform) the tile's value-queue tokens: p_t * v_t from their
            // fp16 ring rows (slot t mod R), on CUDA cores, in token order; the
            // rows of four tokens are loaded before their products
            const int t_first = max(vq_from, 0);
            const uint2 *ring = reinterpret_cast<const uint2 *>(a.p.v_res + (int64_t)bh * g.residual * kD);
            int rs = (int)((tok0 + t_first) % g.residual);
            for (int tt0 = t_first; tt0 < n; tt0 += 4) {
              uint2 vw[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                vw[u] = tt0 + u < n ? ring[(int64_t)rs * (kD / 4) + lane] : make_uint2(0u, 0u);
                rs = rs + 1 == g.residual ? 0 : rs + 1;
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float pt = __shfl_sync(0xffffffffu, p, (tt0 + u) & 31);
                if (tt0 + u < n) {
                  const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vw[u].x));
                  const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vw[u].y));
                  xv[0] = fmaf(pt, v01.x, xv[0]);
                  xv[1] = fmaf(pt, v01.y, xv[1]);
                  xv[2] = fmaf(pt, v23.x, xv[2]);
                  xv[3] = fmaf(pt, v23.y, xv[3]);
                }
              }
            }
          }
          // ------------- values: B = p * scale (hi/lo), A = codes ------------
          // MMA k pairs (2tig, 2tig+1) and (2tig+8, 2tig+9) of k-block kb carry
          // tokens 16kb + tig + {0, 4} and + {8, 12} (code rows 4 apart hit
          // distinct banks).  Each token's lane writes its operand row
          // B[t][(j, hi/lo)] = p_t * scale_tj * 2^-kSlack as fp16 hi + lo into the
          // warp's operand area (the key operand is consumed by now), laid out
          // [column][kb][tig][4 tokens] so each lane then loads the fragment of
          // a k-block with one 64-bit load.
          {
            float sv[NGV];
            ld_stat_row<MF, NGV>(slot + SC::off_vs + t * NGV * SC::MSZ, sv);
            __syncwarp();  // every lane's key-operand loads are done
            __half *orow = reinterpret_cast<__half *>(sBw) + 16 * (t >> 4) + 4 * (t & 3) + ((t & 15) >> 2);
  #pragma unroll
            for (int j = 0; j < NGV; ++j) {
              const float x = valid_v ? pv * sv[j] : 0.0f;
              const __half h = __float2half_rn(x);
              orow[64 * j] = h;
              orow[64 * j + 32] = __float2half_rn(x - __half2float(h));
            }
            __syncwarp();
          }
          const bool bact = gid < 2 * NGV;
          const uint32_t *bsrc = sBw + 16 * gid + 2 * tig;
          const int nkb = (FULL || n > 16) ? 2 : 1;
          for (int kb = 0; kb < nkb; ++kb) {
            const int tk0 = 16 * kb + tig, tk1 = tk0 + 4, tk2 = tk0 + 8, tk3 = tk0 + 12;
            const uint2 bw = *reinterpret_cast<const uint2 *>(bsrc + 8 * kb);
            const uint32_t bv0 = bact ? bw.x : 0u;
            const uint32_t bv1 = bact ? bw.y : 0u;
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
      if (aborted) break;
    }
    // fp16 chunks; a lane owns channels 4*lane .. 4*lane + 3.  A warp whose
    // range holds only a head's empty unit still publishes (an empty
    // partial): the head's partial count includes every warp it touches.
    float mf = -INFINITY, lf = 0.0f, af[4] = {0.f, 0.f, 0.f, 0.f};
    float pow2F = 1.0f;  // fp16 scores = MMA result * 2^F (q normalised by 2^-F)
    {
      for (int lt = 0; lt < nchk; ++lt) {
        int s;
        if (!wait_slot(s)) {
          aborted = true;
          break;
        }
        const uint8_t *slot = wring + s * SLOT;
        if (lt == 0) {
          const uint2 qr = reinterpret_cast<const uint2 *>(slot + SC::off_q)[lane];
          const float2 q01 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.x));
          const float2 q23 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.y));
          q4[0] = q01.x * a.scale_log2;
          q4[1] = q01.y * a.scale_log2;
          q4[2] = q23.x * a.scale_log2;
          q4[3] = q23.y * a.scale_log2;
          // key-score operand of the fp16 rows: q / 2^F as fp16 hi/lo.  With
          // channels 16kb + 4tig .. + 3 on k-pairs (2tig, 2tig+1), (2tig+8,
          // 2tig+9) of k-block kb, lane L's own 4 channels are the B words of
          // (kb, tig) = (L >> 2, L & 3).
          float mx = fmaxf(fmaxf(fabsf(q4[0]), fabsf(q4[1])), fmaxf(fabsf(q4[2]), fabsf(q4[3])));
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          int F = 0;
          if (mx > 0.0f && mx < INFINITY) frexpf(mx, &F);
          pow2F = ldexpf(1.0f, F);
          const float inv = ldexpf(1.0f, -F);
          uint32_t h0, l0, h1, l1;
          split2(q4[0] * inv, q4[1] * inv, h0, l0);
          split2(q4[2] * inv, q4[3] * inv, h1, l1);
          __syncwarp();  // the quantized tiles' operand loads are done
          *reinterpret_cast<uint2 *>(sBw + (lane & 3) * 16 + 2 * (lane >> 2)) = make_uint2(h0, h1);
          *reinterpret_cast<uint2 *>(sBw + (4 + (lane & 3)) * 16 + 2 * (lane >> 2)) = make_uint2(l0, l1);
          __syncwarp();
        }
        const int i0 = (sg.c0 + lt) * CH;
        const int nv = min(CH, hc.nf - i0);  // valid rows of the chunk
        if (a.new_row >= 0) {
          // fused append: the warp holding the new token stores it in the residual
          const int tn = hc.ns + a.new_row - i0;
          if (tn >= 0 && tn < nv) {
            const int half = lane >> 4, j = lane & 15;
            const uint4 v4 = reinterpret_cast<const uint4 *>(slot + half * CH * kD * 2 + tn * kD * 2)[j];
            __half *dstrow = (half ? a.p.v_res : a.p.k_res) + ((int64_t)bh * g.residual + a.new_row) * kD;
            reinterpret_cast<uint4 *>(dstrow)[j] = v4;
          }
        }
        const uint2 *vr = reinterpret_cast<const uint2 *>(slot + CH * kD * 2);
        // scores on the tensor cores: A = the chunk's K rows (token rows 0..7;
        // rows 8..15 zero), B = the query operand; rows past the chunk's valid
        // ones are masked below.  Lane (gid, 0) ends with token gid's score.
        float sp;
        if constexpr (RP != 0) {
          sp = rope_chunk_score(slot, i0, nv);
        } else {
          const uint2 *ka = reinterpret_cast<const uint2 *>(slot + gid * kD * 2) + tig;
          const uint32_t *bq = gid < 2 ? sBw + (gid * 4 + tig) * 16 : sBw + SC::sb_zero;
          float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            const uint2 av = ka[4 * kb];
            const uint2 bv = *reinterpret_cast<const uint2 *>(bq + 2 * kb);
            mma16816((kb & 1) ? e1 : e0, av.x, 0u, av.y, 0u, bv.x, bv.y);
          }
          sp = __shfl_sync(0xffffffffu, (e0[0] + e0[1]) + (e1[0] + e1[1]), lane & ~3) * pow2F;
        }
        const int row = gid;
        const float sc = row < nv ? sp : -INFINITY;
        float mc = sc;
        mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 4));
        mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 8));
        mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, 16));
        const float mn = fmaxf(mf, mc);
        const float al = exp2_approx(mf - mn);
        const float pr = exp2_approx(sc - mn);  // 0 for rows past the chunk's end
        float ps_ = pr;
        ps_ += __shfl_xor_sync(0xffffffffu, ps_, 4);
        ps_ += __shfl_xor_sync(0xffffffffu, ps_, 8);
        ps_ += __shfl_xor_sync(0xffffffffu, ps_, 16);
        lf = fmaf(lf, al, ps_);
#pragma unroll
        for (int i = 0; i < 4; ++i) af[i] *= al;
        mf = mn;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < CH && t < nv) {
            // row t's probability sits in lanes whose bits 4,3,2 spell t
            const float pt = __shfl_sync(0xffffffffu, pr, ((t >> 2) << 4) | (((t >> 1) & 1) << 3) | ((t & 1) << 2));
            const uint2 vw = vr[t * (kD / 4) + lane];
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.y));
            af[0] = fmaf(pt, v01.x, af[0]);
            af[1] = fmaf(pt, v01.y, af[1]);
            af[2] = fmaf(pt, v23.x, af[2]);
            af[3] = fmaf(pt, v23.y, af[3]);
          }
        }
        __syncwarp();
        issue_next();
      }
      if (aborted) break;
    }
    if constexpr (OUT != 0) {
      // partials of the head: one per warp whose range touches it
      const int U = span_at<OUT>(a, base, hc).U;
      cur_np = owner_of(base + U - 1, rx.total, rx.nw) - owner_of(base, rx.total, rx.nw) + 1;
      base_t += U;
      if (cur_np > a.part_stride) {
        // (cannot happen: a head's partials are at most its units) never
        // touch rows past the head's slots
        if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ECAPACITY);
        aborted = true;
        break;
      }
    }
    if (!flush(bh, gw - owner_of(base, OUT ? rx.total : a.total, OUT ? rx.nw : a.nw), mf, lf,
               af)) {
      aborted = true;
      break;
    }
  }
  if (!aborted && pend_bh >= 0 && !merge_head<24>(a, pend_bh, OUT ? pend_np : -1)) aborted = true;
  if (aborted) {
    // give up this warp's work; its copies complete first
    if (lane == 0)
      for (int i = done; i < issued; ++i)
        bar_wait(&wbars[i % nslot], (uint32_t)((i / nslot) & 1), kDrainLimit);
  }
}

template <int BITS, int SCHEME, int NGV, int NGK, int KM, int MF, int OUT, int RP = 0>
cudaError_t launch_tc_t(TcArgs &a, int num_sms, cudaStream_t st) {
  using SC = SlotCfg<BITS, SCHEME, NGV, NGK, KM, MF, OUT, RP>;
  auto kern = tc_decode_kernel<BITS, SCHEME, NGV, NGK, KM, MF, OUT, RP>;
  constexpr int smem = SC::smem;
  if (a.g.meta16 != MF || tc_ext_kind(a.g) != OUT) return cudaErrorInvalidValue;
  // the block and the fp16 chunk fit the slot (the block size, and so the
  // chunk, is compile-time without outlier lists)
  if (OUT == 1 ? (a.g.block_bytes > SC::BBX || a.g.n_out > kMaxOutliers ||
             2 * a.CH * kD * 2 > SC::off_q)
          : (a.g.block_bytes != SC::BB || a.CH != SC::CH))
    return cudaErrorInvalidValue;
  static KernelSetup setup;
  int occ = 0;
  const cudaError_t e = kernel_setup(setup, kern, kThreads, smem, &occ);
  if (e != cudaSuccess) return e;
  int64_t nc = (int64_t)num_sms * occ;
  if (nc > kTcMaxBlocks) nc = kTcMaxBlocks;
  // every working warp gets at least kMinWarpUnits units (or all of them):
  // a head's partials are the warps its units span, and its merger reads
  // them in rounds, so cutting small batches across the whole grid costs
  // more in merging than the extra warps bring
  int64_t nw = nc * kWarps;
  if (nw > (a.total + kMinWarpUnits - 1) / kMinWarpUnits)
    nw = (a.total + kMinWarpUnits - 1) / kMinWarpUnits;
  if (nw < 1) nw = 1;
  // blocks: enough for the working warps, rounded up to a whole number per
  // SM (the working warps spread over them, see the kernel)
  const int64_t need = (nw + kWarps - 1) / kWarps;
  const int64_t per = ((need + num_sms - 1) / num_sms) * num_sms;
  if (per < nc) nc = per;
  a.nc = (int)nc;
  a.nw = (int)nw;
  // every block must be resident: the merging warps wait for other blocks
  if (nc > (int64_t)num_sms * occ) return cudaErrorCooperativeLaunchTooLarge;
  const cudaError_t le = launch_cooperative(kern, (unsigned)nc, kThreads, smem, st, a);
  return le != cudaSuccess ? le : cudaGetLastError();
}

// The template arguments the dispatch picks for a geometry (one function, so
// the launch and kvq_decode_kernel_name cannot disagree).
struct TcVariant {
  int ngv, ngk, km;
};
TcVariant tc_variant(const Geometry &g) {
  TcVariant v{kD / g.v_group, 1, 0};
  if (g.scheme == KVQ_KIVI)
    v.km = g.k_group == 16 ? 2 : g.k_group == 32 ? 1 : 0;
  else
    v.ngk = kD / g.k_group;
  return v;
}

template <int BITS, int SCHEME, int MF, int OUT>
cudaError_t launch_tc_v(TcArgs &a, int num_sms, cudaStream_t st) {
  const TcVariant v = tc_variant(a.g);
  if constexpr (SCHEME == KVQ_KIVI) {
    if (v.ngv == 4)
      return v.km == 2 ? launch_tc_t<BITS, SCHEME, 4, 1, 2, MF, OUT>(a, num_sms, st)
           : v.km == 1 ? launch_tc_t<BITS, SCHEME, 4, 1, 1, MF, OUT>(a, num_sms, st)
                       : launch_tc_t<BITS, SCHEME, 4, 1, 0, MF, OUT>(a, num_sms, st);
    return v.km == 2 ? launch_tc_t<BITS, SCHEME, 2, 1, 2, MF, OUT>(a, num_sms, st)
         : v.km == 1 ? launch_tc_t<BITS, SCHEME, 2, 1, 1, MF, OUT>(a, num_sms, st)
                     : launch_tc_t<BITS, SCHEME, 2, 1, 0, MF, OUT>(a, num_sms, st);
  } else {
    if (v.ngv == 4)
      return v.ngk == 4 ? launch_tc_t<BITS, SCHEME, 4, 4, 0, MF, OUT>(a, num_sms, st)
                        : launch_tc_t<BITS, SCHEME, 4, 2, 0, MF, OUT>(a, num_sms, st);
    return v.ngk == 4 ? launch_tc_t<BITS, SCHEME, 2, 4, 0, MF, OUT>(a, num_sms, st)
                      : launch_tc_t<BITS, SCHEME, 2, 2, 0, MF, OUT>(a, num_sms, st);
  }
}

// Every instantiation of one statistics width, dispatched on bits and scheme
// (OUT: the extended kernel).
template <int MF, int OUT = 0>
cudaError_t launch_tc_mf(TcArgs &a, int num_sms, cudaStream_t st) {
  if (a.g.bits == 2)
    return a.g.scheme == KVQ_KIVI ? launch_tc_v<2, KVQ_KIVI, MF, OUT>(a, num_sms, st)
                                  : launch_tc_v<2, KVQ_INNERQ, MF, OUT>(a, num_sms, st);
  return a.g.scheme == KVQ_KIVI ? launch_tc_v<4, KVQ_KIVI, MF, OUT>(a, num_sms, st)
                                : launch_tc_v<4, KVQ_INNERQ, MF, OUT>(a, num_sms, st);
}

}  // namespace

}  // namespace kvq
