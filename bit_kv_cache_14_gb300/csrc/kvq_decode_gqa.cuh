// Grouped-query decode attention on the tensor cores: head_dim 128, 2- or
// 4-bit KIVI codes, RG = 2 or 4 query heads per KV head.
//
// Same computation as the MHA kernel (softmax(scale * q.K^T) V over the
// packed cache, dequantization folded into both GEMVs -- "大模型量化技术原理：
// KIVI、IntactKV、KVQuant", KIVI / 背景; GQA maps query head hq to KV head
// hq / RG), arranged so one pass over the cache serves all RG query heads:
//
//  * Keys: D[token][n] = sum_c code * B[c][n] with the 8 MMA columns n =
//    (query head r, fp16 hi/lo) -- every column carries data.  The operand
//    is rebuilt per key group from a per-warp table of the normalised
//    queries.  A lane of the accumulator holds head tig's scores for 4
//    tokens, so the online softmax runs per lane with no transposition.
//  * Values: each 16-row MMA tile holds channels of ONE value group (word
//    W = group * words-per-group + gid mod words-per-group, code position
//    chosen per lane by a shift), so its operand is that group's columns
//    n = (r, hi/lo) of p_tr * scale_tj and every accumulator entry is used:
//    lane (gid, tig) accumulates head tig.
//  * fp16 sink / residual tokens ride the same ring in 8-token chunks and are
//    folded on CUDA cores one head at a time into a second partial.
//  * Work split by block (each block an equal range of (head, 128-token unit)
//    plus fp16 units; a segment's tiles go round-robin to the block's warps).
//    Rings and bounded waits are the MHA kernel's (kvq_tc_common.cuh); a
//    warp publishes its partial (RG rows) and takes a ticket with a relaxed
//    atomic, and the last ticket's holder merges (fence-free, the same
//    encoding as the MHA merge).
#pragma once

#include <stdio.h>

#include "kvq_tc_common.cuh"

namespace kvq {

namespace {

// NGK = 0: KIVI keys (per-channel statistics over G tokens; KM = 1 when G =
// 32 puts them inside the block); NGK = 2 or 4: InnerQ keys (per token, NGK
// groups of channels; KM unused).  MF: statistics stored in fp16.
template <int BITS, int NGV, int KM, int RG, int NGK = 0, int MF = 0>
struct GqaCfg {
  static constexpr bool INQ = NGK > 0;
  static constexpr int MSZ = MF ? 2 : 4;    // bytes per stored statistic
  static constexpr int RB = kD * BITS / 8;  // bytes per token row of codes
  static constexpr int off_vc = kTile * RB;
  static constexpr int off_vs = 2 * kTile * RB;
  static constexpr int off_vz = off_vs + kTile * NGV * MSZ;
  static constexpr int off_ks = off_vz + kTile * NGV * MSZ;
  static constexpr int off_kz = off_ks + kTile * NGK * MSZ;  // InnerQ: [token][group]
  static constexpr bool KIN = !INQ && KM >= 1;  // KIVI G = 32: key statistics inside the block
  static constexpr int KGB = 2 * kD * MSZ;
  static constexpr int BB = INQ ? off_kz + kTile * NGK * MSZ : off_ks + (KIN ? KGB : 0);
  static constexpr int KMB = (INQ || KIN) ? 0 : KGB;
  static constexpr int off_km = KIN ? off_ks : BB;
  static constexpr int bytes = BB + KMB;  // one slot (no query rows in the ring)
  static constexpr int CH = bytes / (4 * kD) < 8 ? bytes / (4 * kD) : 8;
  // code words: a 32-bit word holds CPW channels, PH per 16-bit half (the
  // low half channels 0..PH-1 of the word, the high half PH..CPW-1)
  static constexpr int CPW = 32 / BITS, PH = 16 / BITS;
  static constexpr int KWL = kD / CPW / 4;      // key words per lane group (2 or 4)
  static constexpr int SPW = 8 / KWL;           // key k-steps per word
  static constexpr int SPG = INQ ? 8 / NGK : 0;  // InnerQ: key k-steps per channel group
  static constexpr int WPG = kD / NGV / CPW;    // code words per value group
  static constexpr int NV = 8 / WPG;            // code positions dealt over a tile's rows
  static constexpr int MPJ = PH / NV;           // value MMAs per value group and k-block
  // per warp: key operand (8 columns, each a row of KROW words: lane group
  // tig's 2-word fragment of k-step s at tig * KTIG + 2 s; the pitches put
  // the 16 fragments a half-warp reads, and the 32 words one store writes,
  // on distinct banks), also the value operand (2 NGV blocks of 64 words) and
  // the output transpose of RG x 128 floats; query table [c][4] fp32 + 2^E
  // per head
  static constexpr int KTIG = 24, KROW = 98;
  static constexpr int SBB = 8 * KROW * 4;
  static constexpr int QTB = kD * 4 * 4 + 16;
  __host__ __device__ static constexpr int lay(int nslot, int what) {
    // what: 0 sB offset, 1 QT offset, 2 bars offset, 3 total
    return what == 0 ? kWarps * nslot * bytes
         : what == 1 ? kWarps * nslot * bytes + kWarps * SBB
         : what == 2 ? kWarps * nslot * bytes + kWarps * (SBB + QTB)
                     : kWarps * nslot * bytes + kWarps * (SBB + QTB) + kWarps * (nslot + 1) * 8;
  }
  // two blocks per SM where two ring slots fit in half the shared memory
  // (2-bit), else one block per SM with three slots (4-bit: 6 KB blocks)
  static constexpr int MINB = lay(2, 3) <= 112 * 1024 ? 2 : 1;
  static constexpr int nslot = MINB == 2 ? (lay(3, 3) <= 112 * 1024 ? 3 : 2) : 3;
  static constexpr int smem = lay(nslot, 3);
  static_assert(smem <= 227 * 1024, "shared memory");
  static_assert(MPJ * NGV == 8, "eight value MMAs per k-block");
};

// Partial slots of head bh (RG rows each): 8 per block holding quantized
// units of it (every warp, by block order), then one per warp with at least
// one of the block's fp16 chunks (by block order, no gaps).  gqa_slot0(a, bh,
// xe) is the first fp16 slot of block xe; for xe past the last block it is
// the head's slot count.
__device__ __forceinline__ int gqa_slot0(const TcArgs &a, int bh, int xe) {
  const int base = bh * a.U;
  int np = 0;
  if (a.S_h > 0)
    np = kWarps * (owner_of(base + a.S_h - 1, a.total, a.nc) - owner_of(base, a.total, a.nc) + 1);
  if (a.F_h > 0) {
    const int xa = owner_of(base + a.S_h, a.total, a.nc);
    const int xb = min(owner_of(base + a.U - 1, a.total, a.nc), xe - 1);
    for (int x = xa; x <= xb; ++x) {
      int x0, x1;
      block_range(a, x, x0, x1);
      const Seg sg = seg_in(a, bh, x0, x1);
      np += min(kWarps, sg.c1 - sg.c0);
    }
  }
  return np;
}

// Merge of n encoded partial rows row0, row0 + stride, ... (see merge in
// kvq_tc_common.cuh): (M, L, O) for this lane's 4 channels; rows zeroed.
__device__ bool merge_strided(const TcArgs &a, int64_t row0, int stride, int n, float &M,
                              float &L, float4 &O) {
  const int lane = threadIdx.x & 31;
  const uint2 *ml = reinterpret_cast<const uint2 *>(a.ws_ml);
  const uint4 *wo = reinterpret_cast<const uint4 *>(a.ws_o);
  bool ok = true;
  M = -INFINITY;
  for (int s = lane; s < n; s += 32) {
    const int64_t row = row0 + (int64_t)s * stride;
    uint2 v = ld_relaxed(ml + row);
    for (int it = 0; it < kMergePolls && (v.x == 0u || v.y == 0u); ++it) {
      __nanosleep(32);
      v = ld_relaxed(ml + row);
    }
    ok = ok && v.x != 0u && v.y != 0u;
    M = fmaxf(M, __uint_as_float(v.x ^ kEnc));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  L = 0.0f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s0 = 0; s0 < n && ok; s0 += 32) {
    float w = 0.0f;
    if (s0 + lane < n) {
      const uint2 v = ld_relaxed(ml + row0 + (int64_t)(s0 + lane) * stride);
      const float ms = __uint_as_float(v.x ^ kEnc);
      if (ms != -INFINITY) {
        w = exp2f(ms - M);
        L = fmaf(w, __uint_as_float(v.y ^ kEnc), L);
      }
    }
    const int nb = min(32, n - s0);
    for (int j0 = 0; j0 < nb; j0 += 8) {
      uint4 o[8];
      bool ready = false;
      for (int it = 0; it < kMergePolls && !ready; ++it) {
        bool mine = true;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o[j] = j0 + j < nb
                     ? ld_relaxed(wo + (row0 + (int64_t)(s0 + j0 + j) * stride) * (kD / 4) + lane)
                     : make_uint4(1, 1, 1, 1);
          mine = mine && o[j].x != 0u && o[j].y != 0u && o[j].z != 0u && o[j].w != 0u;
        }
        ready = __all_sync(0xffffffffu, mine);
        if (!ready) __nanosleep(32);
      }
      ok = ok && ready;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
        if (j0 + j < nb && wj != 0.0f) {
          acc[0] = fmaf(wj, __uint_as_float(o[j].x ^ kEnc), acc[0]);
          acc[1] = fmaf(wj, __uint_as_float(o[j].y ^ kEnc), acc[1]);
          acc[2] = fmaf(wj, __uint_as_float(o[j].z ^ kEnc), acc[2]);
          acc[3] = fmaf(wj, __uint_as_float(o[j].w ^ kEnc), acc[3]);
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  O = make_float4(acc[0], acc[1], acc[2], acc[3]);
  for (int s = 0; s < n; ++s)
    st_relaxed(reinterpret_cast<uint4 *>(a.ws_o) + (row0 + (int64_t)s * stride) * (kD / 4) + lane,
               make_uint4(0, 0, 0, 0));
  for (int s = lane; s < n; s += 32)
    st_relaxed(reinterpret_cast<uint2 *>(a.ws_ml) + row0 + (int64_t)s * stride, make_uint2(0, 0));
  if (!__all_sync(0xffffffffu, ok)) {
    if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
    return false;
  }
  return true;
}

// The warp holding head bh's last ticket merges its partials, head by head.
template <int RG>
__device__ bool gqa_finish(const TcArgs &a, int bh, int ticket) {
  const int lane = threadIdx.x & 31;
  const int nparts = gqa_slot0(a, bh, a.nc);
  if (__shfl_sync(0xffffffffu, ticket, 0) != nparts - 1) return true;
  const int b = bh / a.g.H, h = bh % a.g.H;
  for (int r = 0; r < RG; ++r) {
    float M, L;
    float4 O;
    if (!merge_strided(a, (int64_t)bh * a.part_stride * RG + r, RG, nparts, M, L, O))
      return false;
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    reinterpret_cast<float4 *>(a.out + ((int64_t)b * a.g.Hq + h * RG + r) * kD)[lane] =
        make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
  }
  if (lane == 0) atomicExch(&a.ws_cnt[bh], 0);  // an atomic, like the tickets it resets
  return true;
}

// Key-operand pair ip (0..63: lane ip mod 32, pass ip / 32) builds channels
// c = CPW W + p and c + PH of code word W at position p.  2-bit: p = ip mod 8,
// W = kw_of(ip / 8) with bits 1 and 2 swapped; 4-bit: p = ip mod 4, W =
// kw_of(ip / 4) with bits 2 and 3 swapped.  Either way one pass writes the
// fragments of lane groups 0 and 2 (or 1 and 3); the map is its own inverse.
template <int BITS>
__device__ __forceinline__ int kw_of(int q) {
  if (BITS == 2) return (q & 1) | ((q & 2) << 1) | ((q & 4) >> 1);
  return (q & 3) | ((q & 4) << 1) | ((q & 8) >> 1);
}

// Position of q_r[c] in the query table: channel c = CPW W + PH e + p (p <
// PH) belongs to key-operand pair ip = PH kw_of(W) + p; the table is
// [ip / 32][r / 2][ip mod 32][r mod 2][e].
template <int BITS>
__device__ __forceinline__ int qt_index(int c, int r) {
  constexpr int CPW = 32 / BITS, PH = 16 / BITS;
  const int ip = PH * kw_of<BITS>(c / CPW) + (c % PH), e = (c / PH) & 1;
  return (((ip >> 5) * 2 + (r >> 1)) * 32 + (ip & 31)) * 4 + (r & 1) * 2 + e;
}

// InnerQ keys: MMA k-step s covers channels 16 s .. 16 s + 15 (inside one
// channel group).  2-bit: every lane group reads code word s, lane group t
// takes positions 2t, 2t + 1 of both halves (the word shifted right by 4t
// bits); 4-bit: lane group t reads word 2s + t / 2 and takes positions
// 2 (t mod 2), + 1 (shifted by 8 (t mod 2) bits).  Either way lane group t's
// k pairs (2t, 2t + 1) and (2t + 8, 2t + 9) hold channels (c1, c2) and
// (c1 + 1, c2 + 1), c2 = c1 + PH.  The query table is [r][lane L = 4 s + t]
// of float4 (q[c1], q[c2], q[c1 + 1], q[c2 + 1]); iq_index gives channel c's
// place in it.
template <int BITS>
__device__ __forceinline__ int iq_c1(int L) {
  const int s = L >> 2, t = L & 3;
  return BITS == 2 ? 16 * s + 2 * t : 8 * (2 * s + (t >> 1)) + 2 * (t & 1);
}
template <int BITS>
__device__ __forceinline__ int iq_index(int c, int r) {
  int L, h;
  if (BITS == 2) {
    L = 4 * (c >> 4) + ((c & 7) >> 1);
    h = (c >> 3) & 1;
  } else {
    const int W = c >> 3;
    L = 4 * (W >> 1) + 2 * (W & 1) + ((c >> 1) & 1);
    h = (c >> 2) & 1;
  }
  return (r * 32 + L) * 4 + 2 * (c & 1) + h;
}

template <int BITS, int NGV, int KM, int RG, int NGK = 0, int MF = 0>
__global__ void __launch_bounds__(kThreads, (GqaCfg<BITS, NGV, KM, RG, NGK, MF>::MINB))
    tc_gqa_kernel(const TcArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  using C = GqaCfg<BITS, NGV, KM, RG, NGK, MF>;
  constexpr bool INQ = C::INQ;
  constexpr int RB = C::RB;
  constexpr int nslot = C::nslot;
  constexpr int SLOT = C::bytes;
  constexpr int CH = C::CH;
  constexpr int WPG = C::WPG, MPJ = C::MPJ, NV = C::NV, CPW = C::CPW, PH = C::PH;
  constexpr int KWL = C::KWL, SPW = C::SPW;
  const Geometry &g = a.g;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  uint8_t *wring = smem + warp * nslot * SLOT;
  uint32_t *sBw = reinterpret_cast<uint32_t *>(smem + C::lay(nslot, 0) + warp * C::SBB);
  float *QT = reinterpret_cast<float *>(smem + C::lay(nslot, 1) + warp * C::QTB);
  uint64_t *wbars = reinterpret_cast<uint64_t *>(smem + C::lay(nslot, 2)) + warp * (nslot + 1);

  grid_dep_trigger();  // the next decode's blocks may take the SMs this grid leaves
  int x0, x1;
  block_range(a, blockIdx.x, x0, x1);
  const int bh_first = x0 / a.U, bh_last = (x1 - 1) / a.U;

  if (lane == 0) {
    for (int s = 0; s <= nslot; ++s) bar_init(&wbars[s], 1);  // [nslot]: never completed
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();

  // ---- producer: per head, quantized tiles lt = warp, warp + 8, ..., then
  // fp16 chunks lt = warp, warp + 8, ... of this block's segments
  int pc_bh = bh_first, pc_ph = 0, pc_lt = warp, pc_n = 0, issued = 0, ps = 0;
  const uint8_t *pc_src = nullptr, *pc_meta = nullptr;  // next block / key statistics
  const uint64_t pol_once = l2_evict_first();  // cache blocks are read once
  const uint32_t wring_s = smem_u32(wring), wbars_s = smem_u32(wbars);
  Seg pc_seg = seg_in(a, pc_bh, x0, x1);
  pc_n = (pc_seg.tq1 - pc_seg.tq0 + kTile - 1) / kTile;
  auto pc_settle = [&]() {
    while (pc_bh >= 0 && pc_lt >= pc_n) {
      if (pc_ph == 0) {
        pc_ph = 1;
        pc_n = pc_seg.c1 - pc_seg.c0;
      } else {
        if (++pc_bh > bh_last) {
          pc_bh = -1;
          return;
        }
        pc_ph = 0;
        pc_seg = seg_in(a, pc_bh, x0, x1);
        pc_n = (pc_seg.tq1 - pc_seg.tq0 + kTile - 1) / kTile;
      }
      pc_lt = warp;
    }
  };
  auto issue_next = [&]() {
    if (pc_bh < 0) return;
    uint8_t *dst = wring + ps * SLOT;
    uint64_t *bar = &wbars[ps];
    const uint32_t dst_s = wring_s + ps * SLOT, bar_s = wbars_s + 8 * ps;
    ps = ps + 1 == nslot ? 0 : ps + 1;
    if (pc_ph == 0) {
      // a cache block: posted by one lane without a branch.  The warp's blocks
      // of one head are kWarps apart, and so are their key-statistics rows
      // (kWarps * kTile tokens is a whole number of key groups).
      if (pc_lt == warp) {
        const int tok0 = pc_seg.tq0 + kTile * pc_lt;
        pc_src = a.p.blocks + ((int64_t)pc_bh * (g.cap / kTile) + tok0 / kTile) * C::BB;
        if constexpr (C::KMB > 0)
          pc_meta = a.p.k_meta + ((int64_t)pc_bh * g.k_meta_rows + tok0 / g.k_group) * 2 * kD * g.msz;
      }
      bulk_g2s_pred(lane == 0, bar_s, (uint32_t)(C::BB + C::KMB), dst_s, pc_src, C::BB, pol_once);
      pc_src += kWarps * C::BB;
      if constexpr (C::KMB > 0) {
        if (lane == 0) bulk_g2s(dst + C::off_km, pc_meta, C::KMB, bar);
        pc_meta += (kWarps * kTile / g.k_group) * 2 * kD * g.msz;
      }
    } else if (lane == 0) {
      const int ns = (int)a.n_sink;
      const int i0 = (pc_seg.c0 + pc_lt) * CH, i1 = min(i0 + CH, (int)a.n_fp16);
      const int s0 = min(i0, ns), s1 = min(i1, ns);
      const int r0 = max(i0, ns) - ns, r1 = max(i1, ns) - ns;
      bar_expect_tx(bar, (uint32_t)(2 * (i1 - i0) * kD * 2));
      if (s1 > s0) {
        const int64_t row = (int64_t)pc_bh * g.n_sink + s0;
        bulk_g2s(dst, a.p.k_sink + row * kD, (uint32_t)((s1 - s0) * kD * 2), bar);
        bulk_g2s(dst + CH * kD * 2, a.p.v_sink + row * kD, (uint32_t)((s1 - s0) * kD * 2), bar);
      }
      if (r1 > r0) {
        const int64_t row = (int64_t)pc_bh * g.residual + r0;
        const int o = (s1 - s0) * kD * 2;
        bulk_g2s(dst + o, a.p.k_res + row * kD, (uint32_t)((r1 - r0) * kD * 2), bar);
        bulk_g2s(dst + CH * kD * 2 + o, a.p.v_res + row * kD, (uint32_t)((r1 - r0) * kD * 2),
                 bar);
      }
    }
    ++issued;
    pc_lt += kWarps;
    pc_settle();
  };
  pc_settle();
  grid_dep_wait();  // the previous grid on the stream has drained: device data from here on
  for (int s = 0; s < nslot; ++s) issue_next();

  // ---- per-head query table: q_r[c] * scale_log2 * 2^-E_r at qt_index(c, r),
  // then 2^E_r at [4 kD + r]; written with plain stores when the warp starts a
  // head.  The order serves the key-operand build: the lane that builds
  // channel pair (c, c + 8) finds (q_r[c], q_r[c + 8]) for r = 0, 1 in one
  // float4 and for r = 2, 3 in the next 32 lanes' float4 row.
  float pow2 = 1.0f;  // 2^E of this lane's softmax head (tig)
  float qsum[NGK > 0 ? NGK : 1];  // InnerQ: head tig's query summed per channel group
#pragma unroll
  for (int gq = 0; gq < (NGK > 0 ? NGK : 1); ++gq) qsum[gq] = 0.0f;
  int q_head = -1;
  // query head r of KV head bh, this lane's channels 4 lane .. 4 lane + 3,
  // times scale_log2
  auto raw_q = [&](int bh, int r, float (&v)[4]) {
    const int b = bh / g.H, h = bh % g.H;
    const uint2 qr =
        __ldg(reinterpret_cast<const uint2 *>(a.q + ((int64_t)b * g.Hq + h * RG + r) * kD) + lane);
    const float2 q01 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.x));
    const float2 q23 = __half22float2(*reinterpret_cast<const __half2 *>(&qr.y));
    v[0] = q01.x * a.scale_log2;
    v[1] = q01.y * a.scale_log2;
    v[2] = q23.x * a.scale_log2;
    v[3] = q23.y * a.scale_log2;
  };
  // InnerQ with normalized keys: the per-channel factors go into the table's
  // query (the codes' side; the fp16 rows take the raw query)
  const bool knorm = INQ && g.knorm;
  auto load_q = [&](int bh) {
    float qv[RG][4];
#pragma unroll
    for (int r = 0; r < RG; ++r) raw_q(bh, r, qv[r]);
    if (knorm) {
      const float4 n4 = reinterpret_cast<const float4 *>(a.p.k_norm + (int64_t)bh * kD)[lane];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        qv[r][0] *= n4.x;
        qv[r][1] *= n4.y;
        qv[r][2] *= n4.z;
        qv[r][3] *= n4.w;
      }
    }
    float e2[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      float mx = fmaxf(fmaxf(fabsf(qv[r][0]), fabsf(qv[r][1])), fmaxf(fabsf(qv[r][2]), fabsf(qv[r][3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      int E = 0;
      if (mx > 0.0f && mx < INFINITY) frexpf(mx, &E);
      e2[r] = ldexpf(1.0f, E);
      const float inv = ldexpf(1.0f, -E);
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[r][i] *= inv;
    }
    __syncwarp();  // the previous head's readers are done with the table
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < RG; ++r)
        QT[INQ ? iq_index<BITS>(4 * lane + i, r) : qt_index<BITS>(4 * lane + i, r)] = qv[r][i];
    if (lane < RG) QT[4 * kD + lane] = e2[lane < RG ? lane : 0];
    if constexpr (INQ) {
      // per channel group: the sum of head tig's normalised query (the zero
      // points' term of the scores)
#pragma unroll
      for (int r = 0; r < RG; ++r)
#pragma unroll
        for (int gq = 0; gq < NGK; ++gq) {
          float sq = (4 * lane) / (kD / NGK) == gq ? (qv[r][0] + qv[r][1]) + (qv[r][2] + qv[r][3]) : 0.0f;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
          if (r == tig) qsum[gq] = sq;
        }
    }
    __syncwarp();
    pow2 = tig < RG ? QT[4 * kD + tig] : 1.0f;
    q_head = bh;
  };

  // key-operand channel pairs this lane builds (as in the MHA kernel), and
  // the factor 1 / pos_factor(p) that undoes the code position p; lane group
  // tig holds words W = KWL tig + w, k-step SPW w + p / 2, register p mod 2
  int b_clo[2];
  uint32_t *b_dst[2];
  float2 b_ipf[2];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int ip = lane + 32 * m;
    const int W = kw_of<BITS>(ip / PH), p = ip % PH;
    b_clo[m] = CPW * W + p;
    b_dst[m] = sBw + (W / KWL) * C::KTIG + (SPW * (W % KWL) + (p >> 1)) * 2 + (p & 1);
    const float f = inv_pos_factor<BITS>(p);
    b_ipf[m] = make_float2(f, f);
  }
  // InnerQ: the key-operand words lane L = 4 s + t writes (k-step s, lane
  // group t; column n at + n KROW), the factor of its second k pair (relative
  // position 1 after the shift), and the reader's shift and word choice
  uint32_t *const iq_wr = sBw + (lane & 3) * C::KTIG + 2 * (lane >> 2);
  const float2 iq_f1 = make_float2(inv_pos_factor<BITS>(1), inv_pos_factor<BITS>(1));
  const int iq_sh = BITS == 2 ? 4 * tig : 8 * (tig & 1);
  const bool iq_hiw = (tig >> 1) != 0;  // 4-bit: the odd word of the k-step's pair
  // value operand: the writer's columns (r = tig, hi / lo) and the reader's
  // column gid sit at column slot n ^ (n >> 2), which keeps the writers' 32-bit
  // stores (columns 0, 2, 4, 6 or 1, 3, 5, 7) and each half-warp's 64-bit
  // loads (columns 0-3 or 4-7) on distinct banks
  const int wofs = 2 * (gid & 3) + (gid >> 2);  // word of token pair (gid, gid + 8)
  uint32_t *const v_hi = sBw + (2 * tig + (tig >> 1)) * 8 + wofs;
  uint32_t *const v_lo = sBw + (2 * tig + 1 - (tig >> 1)) * 8 + wofs;
  const uint32_t *const v_rd = sBw + (gid ^ (gid >> 2)) * 8 + 2 * tig;
  // value codes: this lane's rows take code position NV m + v_off of each
  // half word (m the MMA's index in its value group), read in place by a
  // mask: the low half of the positions (0-3 of 2-bit, 0-1 of 4-bit) from the
  // token pair's half words, the high half from them shifted down a byte
  const int v_off = gid / WPG;
  const uint32_t vm0 = (BITS == 2 ? 0x00030003u : 0x000F000Fu) << (BITS * v_off), vm1 = vm0 << 4;
  const float2 neg1 = make_float2(-1.0f, -1.0f);
  const bool head_lane = tig < RG;

  // ---- online-softmax state: lane (gid, tig) holds head tig ---------------
  // (lanes of absent heads keep a finite reference, so their weights are 0)
  float m_run = -INFINITY;
  float2 l2, z2[NGV / 2];
  float dv[8][4];
  auto reset_state = [&]() {
    m_run = head_lane ? -INFINITY : 0.0f;
    l2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NGV / 2; ++j) z2[j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) dv[mt][r] = 0.0f;
  };
  reset_state();

  int pend_bh = -1, pend_ticket = 0;
  auto publish = [&](int bh, int slot, const float4 (&o)[RG], const float (&m)[RG],
                     const float (&l)[RG]) -> bool {
    if (pend_bh >= 0 && !gqa_finish<RG>(a, pend_bh, pend_ticket)) return false;
    const int64_t row0 = ((int64_t)bh * a.part_stride + slot) * RG;
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      st_relaxed(reinterpret_cast<uint4 *>(a.ws_o + (row0 + r) * kD) + lane, enc4(o[r]));
      if (lane == 0)
        st_relaxed(reinterpret_cast<uint2 *>(a.ws_ml) + row0 + r,
                   make_uint2(__float_as_uint(m[r]) ^ kEnc, __float_as_uint(l[r]) ^ kEnc));
    }
    pend_ticket = 0;
    if (lane == 0) pend_ticket = atomicAdd(&a.ws_cnt[bh], 1);
    pend_bh = bh;
    return true;
  };

  // quantized state -> partial `slot` of head bh
  auto flush_quant = [&](int bh, int slot) -> bool {
    float l = l2.x + l2.y, Z[NGV];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
    for (int j = 0; j < NGV; ++j) {
      float z = (j & 1) ? z2[j / 2].y : z2[j / 2].x;
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      Z[j] = z;
    }
    float *so = reinterpret_cast<float *>(sBw);
    __syncwarp();
    if (head_lane) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int j = mt / MPJ, m = mt % MPJ;
        const int W = j * WPG + gid % WPG, p = m * NV + v_off;
        // the code sat at position ps of its source half word (the high
        // positions after the shift by a byte): 2^24 * 2^kSlack / pos_factor
        const int ps = p % (PH / 2);
        const float f = __int_as_float((127 + 24 + kSlackLog2 - BITS * ps) << 23);
        so[tig * kD + CPW * W + p] = fmaf(dv[mt][0] + dv[mt][1], f, Z[j]);
        so[tig * kD + CPW * W + PH + p] = fmaf(dv[mt][2] + dv[mt][3], f, Z[j]);
      }
    }
    __syncwarp();
    float4 o[RG];
    float mm[RG], ll[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      o[r] = reinterpret_cast<const float4 *>(so)[r * (kD / 4) + lane];
      mm[r] = __shfl_sync(0xffffffffu, m_run, r);
      ll[r] = __shfl_sync(0xffffffffu, l, r);
    }
    __syncwarp();
    reset_state();
    return publish(bh, slot, o, mm, ll);
  };

  int cs = 0, done = 0;
  uint32_t cph = 0;
  bool first = true;
  auto wait_slot = [&](int &s_out) -> bool {
    bool ok = true;
    if (first && a.stall_limit > 0) ok = bar_wait(&wbars[nslot], 0u, a.stall_limit);
    first = false;
    if (ok) ok = bar_wait(wbars_s + 8 * cs, cph, a.wait_limit);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
      return false;
    }
    s_out = cs;
    if (++cs == nslot) {
      cs = 0;
      cph ^= 1u;
    }
    ++done;
    return true;
  };

  bool aborted = false;
  for (int bh = bh_first; bh <= bh_last && !aborted; ++bh) {
    const Seg sg = seg_in(a, bh, x0, x1);
    const int base = bh * a.U;
    const int tq0 = sg.tq0, tq1 = sg.tq1;
    if (tq1 > tq0) {
      if (q_head != bh) load_q(bh);
      // KIVI: every tile is whole (the quantized length is a multiple of the
      // key group >= 32, which the launch checks); InnerQ: the last may end early
      const int nt = (tq1 - tq0 + kTile - 1) / kTile;
      for (int lt = warp; lt < nt; lt += kWarps) {
        int s;
        if (!wait_slot(s)) {
          aborted = true;
          break;
        }
        const uint8_t *slot = wring + s * SLOT;
        const uint8_t *kc = slot;
        const uint8_t *vc = slot + C::off_vc;
        const int tok0 = tq0 + kTile * lt;
        const bool full = !INQ || tok0 + kTile <= tq1;
        float sc[4];
        if constexpr (INQ) {
          // ---- key operand: columns (r, hi/lo) of QT / pos_factor (the fixed
          // normalised query: the per-token scales enter after the MMAs)
#pragma unroll
          for (int r = 0; r < RG; ++r) {
            const float4 qv4 = reinterpret_cast<const float4 *>(QT)[r * 32 + lane];
            const float2 x0 = make_float2(qv4.x, qv4.y);
            const float2 x1 = __fmul2_rn(make_float2(qv4.z, qv4.w), iq_f1);
            const __half2 h0 = __float22half2_rn(x0), h1 = __float22half2_rn(x1);
            const __half2 l0 = __float22half2_rn(__ffma2_rn(__half22float2(h0), neg1, x0));
            const __half2 l1 = __float22half2_rn(__ffma2_rn(__half22float2(h1), neg1, x1));
            *reinterpret_cast<uint2 *>(iq_wr + (2 * r) * C::KROW) = make_uint2(h2u(h0), h2u(h1));
            *reinterpret_cast<uint2 *>(iq_wr + (2 * r + 1) * C::KROW) = make_uint2(h2u(l0), h2u(l1));
          }
          // per-token scales and zeros: [token][group] rows, read per group
          // next to their use
          const uint8_t *ksr = slot + C::off_ks + gid * NGK * C::MSZ;
          __syncwarp();
          // ---- keys: per channel group, D_g[token][(r, hi/lo)] over its
          // k-steps, weighted by the token's scale of that group
          const uint32_t *bsrc = sBw + gid * C::KROW + tig * C::KTIG;
          constexpr uint32_t M0 = BITS == 2 ? 0x00030003u : 0x000F000Fu, M1 = M0 << BITS;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          // code bytes of rows gid + 8 i: 2-bit, words (st, st + 1) of an even
          // k-step st (8 bytes); 4-bit, words 2 st .. 2 st + 3 (16 bytes)
          uint4 ch[4];
#pragma unroll
          for (int gq = 0; gq < NGK; ++gq) {
            float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ss = 0; ss < C::SPG; ++ss) {
              const int st = gq * C::SPG + ss;
              if ((st & 1) == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint8_t *row = kc + (gid + 8 * i) * RB;
                  if (BITS == 2) {
                    const uint2 x = *reinterpret_cast<const uint2 *>(row + 4 * st);
                    ch[i].x = x.x, ch[i].y = x.y;
                  } else {
                    ch[i] = *reinterpret_cast<const uint4 *>(row + 8 * st);
                  }
                }
              }
              uint32_t w[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t x;
                if (BITS == 2)
                  x = (st & 1) ? ch[i].y : ch[i].x;
                else
                  x = (st & 1) ? (iq_hiw ? ch[i].w : ch[i].z) : (iq_hiw ? ch[i].y : ch[i].x);
                w[i] = x >> iq_sh;
              }
              const uint2 b = *reinterpret_cast<const uint2 *>(bsrc + 2 * st);
              mma16816(e0, w[0] & M0, w[1] & M0, w[0] & M1, w[1] & M1, b.x, b.y);
              mma16816(e1, w[2] & M0, w[3] & M0, w[2] & M1, w[3] & M1, b.x, b.y);
            }
            acc[0] = fmaf(ld_stat<MF>(ksr, gq), e0[0] + e0[1], acc[0]);
            acc[1] = fmaf(ld_stat<MF>(ksr, 8 * NGK + gq), e0[2] + e0[3], acc[1]);
            acc[2] = fmaf(ld_stat<MF>(ksr, 16 * NGK + gq), e1[0] + e1[1], acc[2]);
            acc[3] = fmaf(ld_stat<MF>(ksr, 24 * NGK + gq), e1[2] + e1[3], acc[3]);
          }
          // ---- scores: (sum_g scale * D_g * 2^24 + sum_g zero * q-sum_g) * 2^E;
          // tokens past the head's quantized end (a short last tile) -inf
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float zk[NGK];
            ld_stat_row<MF, NGK>(slot + C::off_kz + (gid + 8 * i) * NGK * C::MSZ, zk);
            float zt = 0.0f;
#pragma unroll
            for (int gq = 0; gq < NGK; ++gq) zt = fmaf(zk[gq], qsum[gq], zt);
            sc[i] = fmaf(acc[i], kSub, zt) * pow2;
            if (!full) sc[i] = tok0 + gid + 8 * i < tq1 ? sc[i] : -INFINITY;
          }
        } else {
          // ---- key operand: columns (r, hi/lo) of QT * scale / pos_factor(p), and the
          // per-head bias sum_c QT * zero, for this tile's key group
          const uint8_t *ks = slot + C::off_km, *kz = ks + kD * C::MSZ;
          float2 bacc[RG];
#pragma unroll
          for (int r = 0; r < RG; ++r) bacc[r] = make_float2(0.f, 0.f);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int clo = b_clo[m], chi = clo + PH;
            const float2 s2 =
                __fmul2_rn(make_float2(ld_stat<MF>(ks, clo), ld_stat<MF>(ks, chi)), b_ipf[m]);
            const float2 zz = make_float2(ld_stat<MF>(kz, clo), ld_stat<MF>(kz, chi));
            const float4 q01 = reinterpret_cast<const float4 *>(QT)[(2 * m) * 32 + lane];
            const float4 q23 = RG > 2 ? reinterpret_cast<const float4 *>(QT)[(2 * m + 1) * 32 + lane] : q01;
#pragma unroll
            for (int r = 0; r < RG; ++r) {
              const float4 &qq = r < 2 ? q01 : q23;
              const float2 qr = (r & 1) ? make_float2(qq.z, qq.w) : make_float2(qq.x, qq.y);
              const float2 x = __fmul2_rn(qr, s2);
              const __half2 h = __float22half2_rn(x);
              b_dst[m][(2 * r) * C::KROW] = h2u(h);
              b_dst[m][(2 * r + 1) * C::KROW] =
                  h2u(__float22half2_rn(__ffma2_rn(__half22float2(h), neg1, x)));
              bacc[r] = __ffma2_rn(qr, zz, bacc[r]);
            }
          }
          float bpart[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) bpart[r] = r < RG ? bacc[r < RG ? r : 0].x + bacc[r < RG ? r : 0].y : 0.0f;
          // reduce-scatter of the 4 bias sums: lane L ends with head (L >> 3)
          {
            const bool h4 = lane & 16;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float mine = h4 ? bpart[j + 2] : bpart[j], other = h4 ? bpart[j] : bpart[j + 2];
              bpart[j] = mine + __shfl_xor_sync(0xffffffffu, other, 16);
            }
            const bool h3 = lane & 8;
            const float mine = h3 ? bpart[1] : bpart[0], other = h3 ? bpart[0] : bpart[1];
            bpart[0] = mine + __shfl_xor_sync(0xffffffffu, other, 8);
            bpart[0] += __shfl_xor_sync(0xffffffffu, bpart[0], 4);
            bpart[0] += __shfl_xor_sync(0xffffffffu, bpart[0], 2);
            bpart[0] += __shfl_xor_sync(0xffffffffu, bpart[0], 1);
          }
          const float bias = __shfl_sync(0xffffffffu, bpart[0], (tig & 3) << 3);
          __syncwarp();
          // ---- keys: D[token][(r, hi/lo)]
          // (two accumulators per 16-token half, one per code word, keep the
          // dependent MMA chains four long)
          float d0[4], d1[4];
          {
            float e0[2][4] = {}, e1[2][4] = {};
            const uint32_t *bsrc = sBw + gid * C::KROW + tig * C::KTIG;
            // rows gid, gid + 8, gid + 16, gid + 24: this lane group's KWL words
            uint32_t w[KWL][4], sw[KWL][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint8_t *row = kc + (gid + 8 * i) * RB + 4 * KWL * tig;
              if constexpr (KWL == 2) {
                const uint2 x = *reinterpret_cast<const uint2 *>(row);
                w[0][i] = x.x, w[1][i] = x.y;
              } else {
                const uint4 x = *reinterpret_cast<const uint4 *>(row);
                w[0][i] = x.x, w[1][i] = x.y, w[2][i] = x.z, w[3][i] = x.w;
              }
            }
#pragma unroll
            for (int m = 0; m < KWL; ++m)
#pragma unroll
              for (int i = 0; i < 4; ++i) sw[m][i] = shifted<BITS>(w[m][i]);
#pragma unroll
            for (int jj = 0; jj < SPW; ++jj)
#pragma unroll
              for (int m = 0; m < KWL; ++m) {
                const uint2 b = *reinterpret_cast<const uint2 *>(bsrc + 2 * (SPW * m + jj));
                float(&f0)[4] = e0[m & 1];
                float(&f1)[4] = e1[m & 1];
                mma16816(f0, ext<BITS>(w[m][0], sw[m][0], 2 * jj), ext<BITS>(w[m][1], sw[m][1], 2 * jj),
                         ext<BITS>(w[m][0], sw[m][0], 2 * jj + 1),
                         ext<BITS>(w[m][1], sw[m][1], 2 * jj + 1), b.x, b.y);
                mma16816(f1, ext<BITS>(w[m][2], sw[m][2], 2 * jj), ext<BITS>(w[m][3], sw[m][3], 2 * jj),
                         ext<BITS>(w[m][2], sw[m][2], 2 * jj + 1),
                         ext<BITS>(w[m][3], sw[m][3], 2 * jj + 1), b.x, b.y);
              }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              d0[i] = e0[0][i] + e0[1][i];
              d1[i] = e1[0][i] + e1[1][i];
            }
          }
          // ---- scores of head tig for tokens gid, gid + 8, gid + 16, gid + 24
          const float2 ksub2 = make_float2(kSub, kSub), bias2 = make_float2(bias, bias);
          const float2 pw2 = make_float2(pow2, pow2);
          const float2 s01 =
              __fmul2_rn(__ffma2_rn(make_float2(d0[0] + d0[1], d0[2] + d0[3]), ksub2, bias2), pw2);
          const float2 s23 =
              __fmul2_rn(__ffma2_rn(make_float2(d1[0] + d1[1], d1[2] + d1[3]), ksub2, bias2), pw2);
          sc[0] = s01.x, sc[1] = s01.y, sc[2] = s23.x, sc[3] = s23.y;
        }
        if constexpr (RG < 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[i] = head_lane ? sc[i] : -INFINITY;
        }
        const float lim = m_run + kSlack;
        const bool grow = sc[0] > lim || sc[1] > lim || sc[2] > lim || sc[3] > lim;
        if (__any_sync(0xffffffffu, grow)) {
          float mt_ = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, off));
          if (mt_ > m_run) {
            const float alpha = exp2_approx(m_run - mt_);
            const float2 al2 = make_float2(alpha, alpha);
            l2 = __fmul2_rn(l2, al2);
#pragma unroll
            for (int j = 0; j < NGV / 2; ++j) z2[j] = __fmul2_rn(z2[j], al2);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              const float2 x = __fmul2_rn(make_float2(dv[mt][0], dv[mt][1]), al2);
              const float2 y = __fmul2_rn(make_float2(dv[mt][2], dv[mt][3]), al2);
              dv[mt][0] = x.x;
              dv[mt][1] = x.y;
              dv[mt][2] = y.x;
              dv[mt][3] = y.y;
            }
            m_run = mt_;
          }
        }
        // weights 2^(s - m) (0 for an absent head: its reference is finite)
        float2 pv[2];
        {
          const float2 mr = make_float2(m_run, m_run);
          const uint8_t *vz = slot + C::off_vz;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float2 e = __ffma2_rn(mr, neg1, make_float2(sc[2 * k], sc[2 * k + 1]));
            const float2 p = make_float2(exp2_approx(e.x), exp2_approx(e.y));
            l2 = __fadd2_rn(l2, p);
            pv[k] = __fmul2_rn(p, make_float2(kInvSlack, kInvSlack));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float pi = h ? p.y : p.x;
              const float2 pp = make_float2(pi, pi);
              float zv[NGV];
              ld_stat_row<MF, NGV>(vz + (gid + 8 * (2 * k + h)) * NGV * C::MSZ, zv);
              // (a token past a short tile's end has weight 0; its statistics
              // need not be finite)
              const bool okz = full || tok0 + gid + 8 * (2 * k + h) < tq1;
#pragma unroll
              for (int j = 0; j < NGV; ++j) zv[j] = okz ? zv[j] : 0.0f;
#pragma unroll
              for (int jp = 0; jp < NGV / 2; ++jp)
                z2[jp] = __ffma2_rn(pp, make_float2(zv[2 * jp], zv[2 * jp + 1]), z2[jp]);
            }
          }
        }
        // ---- values: per value group j, its 16-row tiles and columns (r, hi/lo)
        // MMA k pairs (2tig, 2tig+1) and (2tig+8, 2tig+9) of k-block kb carry
        // tokens 16kb + tig + {0, 8} and + {4, 12}.  The operand B[t][(r,
        // hi/lo)] = p_tr * scale_tj * 2^-kSlack is written once, by the lane that
        // holds p_tr (head tig, tokens gid + 8i): a token pair (t, t + 8) of one
        // column is one 32-bit word, at [j][kb][column slot][tig'][2 words] in
        // the warp's operand area (the key operand is consumed by now); each
        // lane then loads its fragment of (kb, j) with one 64-bit load.
        {
          const uint8_t *vs = slot + C::off_vs;
          __syncwarp();  // every lane's key-operand loads are done
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            // tokens a = gid + 16 kb and b = a + 8: products taken in pairs of
            // value groups (j, j + 1), then packed per group as (a, b)
            const float2 paa = make_float2(pv[kb].x, pv[kb].x), pbb = make_float2(pv[kb].y, pv[kb].y);
            float2 sa[NGV / 2], sb[NGV / 2];
            {
              float xa[NGV], xb[NGV];
              ld_stat_row<MF, NGV>(vs + (gid + 16 * kb) * NGV * C::MSZ, xa);
              ld_stat_row<MF, NGV>(vs + (gid + 16 * kb + 8) * NGV * C::MSZ, xb);
#pragma unroll
              for (int jp = 0; jp < NGV / 2; ++jp) {
                sa[jp] = make_float2(xa[2 * jp], xa[2 * jp + 1]);
                sb[jp] = make_float2(xb[2 * jp], xb[2 * jp + 1]);
              }
            }
            if (!full) {
              const bool oka = tok0 + gid + 16 * kb < tq1, okb = tok0 + gid + 16 * kb + 8 < tq1;
#pragma unroll
              for (int jp = 0; jp < NGV / 2; ++jp) {
                if (!oka) sa[jp] = make_float2(0.f, 0.f);
                if (!okb) sb[jp] = make_float2(0.f, 0.f);
              }
            }
#pragma unroll
            for (int jp = 0; jp < NGV / 2; ++jp) {
              const float2 xa = __fmul2_rn(paa, sa[jp]), xb = __fmul2_rn(pbb, sb[jp]);
              const __half2 h0 = __floats2half2_rn(xa.x, xb.x), h1 = __floats2half2_rn(xa.y, xb.y);
              const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
              const float2 ea = __ffma2_rn(make_float2(f0.x, f1.x), neg1, xa);
              const float2 eb = __ffma2_rn(make_float2(f0.y, f1.y), neg1, xb);
              v_hi[(4 * jp + kb) * 64] = h2u(h0);
              v_lo[(4 * jp + kb) * 64] = h2u(__floats2half2_rn(ea.x, eb.x));
              v_hi[(4 * jp + 2 + kb) * 64] = h2u(h1);
              v_lo[(4 * jp + 2 + kb) * 64] = h2u(__floats2half2_rn(ea.y, eb.y));
            }
          }
          __syncwarp();
        }
        {
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint8_t *vr = vc + (16 * kb + tig) * RB + 4 * (gid % WPG);
#pragma unroll
            for (int j = 0; j < NGV; ++j) {
              const uint2 bw = *reinterpret_cast<const uint2 *>(v_rd + (j * 2 + kb) * 64);
              const uint8_t *vw = vr + 4 * j * WPG;
              const uint32_t w0 = *reinterpret_cast<const uint32_t *>(vw);
              const uint32_t w1 = *reinterpret_cast<const uint32_t *>(vw + 8 * RB);
              const uint32_t w2 = *reinterpret_cast<const uint32_t *>(vw + 4 * RB);
              const uint32_t w3 = *reinterpret_cast<const uint32_t *>(vw + 12 * RB);
              const uint32_t ya = __byte_perm(w0, w1, 0x5410), yb = __byte_perm(w0, w1, 0x7632);
              const uint32_t yc = __byte_perm(w2, w3, 0x5410), yd = __byte_perm(w2, w3, 0x7632);
              const uint32_t za = ya >> 8, zb = yb >> 8, zc = yc >> 8, zd = yd >> 8;
              if constexpr (MPJ == 2) {
                mma16816(dv[2 * j], ya & vm0, yb & vm0, yc & vm0, yd & vm0, bw.x, bw.y);
                mma16816(dv[2 * j + 1], za & vm0, zb & vm0, zc & vm0, zd & vm0, bw.x, bw.y);
              } else {
                mma16816(dv[4 * j], ya & vm0, yb & vm0, yc & vm0, yd & vm0, bw.x, bw.y);
                mma16816(dv[4 * j + 1], ya & vm1, yb & vm1, yc & vm1, yd & vm1, bw.x, bw.y);
                mma16816(dv[4 * j + 2], za & vm0, zb & vm0, zc & vm0, zd & vm0, bw.x, bw.y);
                mma16816(dv[4 * j + 3], za & vm1, zb & vm1, zc & vm1, zd & vm1, bw.x, bw.y);
              }
            }
          }
        }
        __syncwarp();
        issue_next();
      }
      if (aborted) break;
      if (!flush_quant(bh, kWarps * ((int)blockIdx.x - owner_of(base, a.total, a.nc)) + warp)) {
        aborted = true;
        break;
      }
    }
    // ---- fp16 chunks of this block's segment, one head at a time ----------
    const int nchk = sg.c1 - sg.c0;
    if (warp < nchk) {
      if (q_head != bh) load_q(bh);
      float qq[RG][4], mf[RG], lf[RG], af[RG][4];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const float e = QT[4 * kD + r];
        if (knorm) {
          raw_q(bh, r, qq[r]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            qq[r][i] = QT[INQ ? iq_index<BITS>(4 * lane + i, r) : qt_index<BITS>(4 * lane + i, r)] * e;
        }
        mf[r] = -INFINITY;
        lf[r] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) af[r][i] = 0.0f;
      }
      for (int lt = warp; lt < nchk; lt += kWarps) {
        int s;
        if (!wait_slot(s)) {
          aborted = true;
          break;
        }
        const uint8_t *slot = wring + s * SLOT;
        const int i0 = (sg.c0 + lt) * CH;
        const int nv = min(CH, (int)a.n_fp16 - i0);
        const uint2 *kr = reinterpret_cast<const uint2 *>(slot);
        const uint2 *vr = reinterpret_cast<const uint2 *>(slot + CH * kD * 2);
        for (int t = 0; t < nv; ++t) {
          const uint2 kw = kr[t * (kD / 4) + lane], vw = vr[t * (kD / 4) + lane];
          const float2 k01 = __half22float2(*reinterpret_cast<const __half2 *>(&kw.x));
          const float2 k23 = __half22float2(*reinterpret_cast<const __half2 *>(&kw.y));
          const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.x));
          const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&vw.y));
#pragma unroll
          for (int r = 0; r < RG; ++r) {
            float sc_ = fmaf(qq[r][0], k01.x, fmaf(qq[r][1], k01.y, fmaf(qq[r][2], k23.x, qq[r][3] * k23.y)));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sc_ += __shfl_xor_sync(0xffffffffu, sc_, off);
            const float mn = fmaxf(mf[r], sc_);
            const float al = exp2_approx(mf[r] - mn), pp = exp2_approx(sc_ - mn);
            lf[r] = fmaf(lf[r], al, pp);
            af[r][0] = fmaf(af[r][0], al, pp * v01.x);
            af[r][1] = fmaf(af[r][1], al, pp * v01.y);
            af[r][2] = fmaf(af[r][2], al, pp * v23.x);
            af[r][3] = fmaf(af[r][3], al, pp * v23.y);
            mf[r] = mn;
          }
        }
        __syncwarp();
        issue_next();
      }
      if (aborted) break;
      float4 o[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) o[r] = make_float4(af[r][0], af[r][1], af[r][2], af[r][3]);
      if (!publish(bh, gqa_slot0(a, bh, blockIdx.x) + warp, o, mf, lf)) {
        aborted = true;
        break;
      }
    }
  }
  if (!aborted && pend_bh >= 0 && !gqa_finish<RG>(a, pend_bh, pend_ticket)) aborted = true;
  if (aborted && lane == 0)
    for (int i = done; i < issued; ++i)
      bar_wait(&wbars[i % nslot], (uint32_t)((i / nslot) & 1), kDrainLimit);
}

template <int BITS, int NGV, int KM, int RG, int NGK = 0, int MF = 0>
cudaError_t launch_gqa_t(TcArgs &a, int num_sms, cudaStream_t st) {
  using C = GqaCfg<BITS, NGV, KM, RG, NGK, MF>;
  auto kern = tc_gqa_kernel<BITS, NGV, KM, RG, NGK, MF>;
  if (a.g.block_bytes != C::BB || tc_fp16_chunk(a.g) != C::CH) return cudaErrorInvalidValue;
  static KernelSetup setup;
  int occ = 0;
  const cudaError_t e = kernel_setup(setup, kern, kThreads, C::smem, &occ);
  if (e != cudaSuccess) return e;
  int64_t nc = (int64_t)num_sms * occ;
  if (nc > kTcMaxBlocks) nc = kTcMaxBlocks;
  if (nc > a.total) nc = a.total;
  if (nc < 1) nc = 1;
  a.nc = (int)nc;
  // every block must be resident: the last ticket's holder waits for the others
  if (nc > (int64_t)num_sms * occ) return cudaErrorCooperativeLaunchTooLarge;
  const cudaError_t le = launch_cooperative(kern, (unsigned)nc, kThreads, C::smem, st, a);
  return le != cudaSuccess ? le : cudaGetLastError();
}

// The instantiation the geometry names, for statistics in fp32 (MF = 0) or
// fp16 (MF = 1): KIVI keys (value groups, key statistics inside the block or
// not) and InnerQ keys (value groups, key channel groups), over the code width
// and the query heads per KV head.
template <int MF, int BITS, int RG>
cudaError_t launch_kivi_br(TcArgs &a, int num_sms, cudaStream_t st) {
  const int ngv = kD / a.g.v_group, km = a.g.k_group == 32 ? 1 : 0;
  if (ngv == 4)
    return km ? launch_gqa_t<BITS, 4, 1, RG, 0, MF>(a, num_sms, st)
              : launch_gqa_t<BITS, 4, 0, RG, 0, MF>(a, num_sms, st);
  return km ? launch_gqa_t<BITS, 2, 1, RG, 0, MF>(a, num_sms, st)
            : launch_gqa_t<BITS, 2, 0, RG, 0, MF>(a, num_sms, st);
}
template <int MF>
cudaError_t launch_kivi(TcArgs &a, int num_sms, cudaStream_t st) {
  const int rg = a.g.Hq / a.g.H;
  if (a.g.bits == 4)
    return rg == 4 ? launch_kivi_br<MF, 4, 4>(a, num_sms, st) : launch_kivi_br<MF, 4, 2>(a, num_sms, st);
  return rg == 4 ? launch_kivi_br<MF, 2, 4>(a, num_sms, st) : launch_kivi_br<MF, 2, 2>(a, num_sms, st);
}
template <int MF, int BITS, int RG>
cudaError_t launch_innerq_br(TcArgs &a, int num_sms, cudaStream_t st) {
  const int ngv = kD / a.g.v_group, ngk = kD / a.g.k_group;
  if (ngv == 4)
    return ngk == 4 ? launch_gqa_t<BITS, 4, 0, RG, 4, MF>(a, num_sms, st)
                    : launch_gqa_t<BITS, 4, 0, RG, 2, MF>(a, num_sms, st);
  return ngk == 4 ? launch_gqa_t<BITS, 2, 0, RG, 4, MF>(a, num_sms, st)
                  : launch_gqa_t<BITS, 2, 0, RG, 2, MF>(a, num_sms, st);
}
template <int MF>
cudaError_t launch_innerq(TcArgs &a, int num_sms, cudaStream_t st) {
  const int rg = a.g.Hq / a.g.H;
  if (a.g.bits == 4)
    return rg == 4 ? launch_innerq_br<MF, 4, 4>(a, num_sms, st)
                   : launch_innerq_br<MF, 4, 2>(a, num_sms, st);
  return rg == 4 ? launch_innerq_br<MF, 2, 4>(a, num_sms, st)
                 : launch_innerq_br<MF, 2, 2>(a, num_sms, st);
}

}  // namespace

// The other families' launches, each in a translation unit of its own so the
// instantiations compile in parallel (arguments filled in by
// launch_decode_gqa): InnerQ keys (kvq_decode_gqa_iq.cu), KIVI keys with fp16
// statistics (kvq_decode_gqa_f16.cu), InnerQ keys with fp16 statistics
// (kvq_decode_gqa_iq16.cu).
cudaError_t launch_gqa_innerq(TcArgs &a, int num_sms, cudaStream_t st);
cudaError_t launch_gqa_kivi_f16(TcArgs &a, int num_sms, cudaStream_t st);
cudaError_t launch_gqa_innerq_f16(TcArgs &a, int num_sms, cudaStream_t st);

}  // namespace kvq
