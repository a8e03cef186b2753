// Shared pieces of the tensor-core decode kernels (MHA: kvq_decode_tc.cu,
// grouped-query: kvq_decode_gqa.cu): launch arguments, PTX wrappers (mbarriers,
// bulk copies, mma.sync), the code-extraction helpers, the stream-K work
// split and the fence-free merge of partials.  Everything sits in an unnamed
// namespace: each translation unit gets its own internal copy.
#pragma once

#include <math.h>

#include <type_traits>

#include "kvq_internal.cuh"

namespace kvq {

// Launch arguments of the tensor-core decode kernels (one definition for
// every translation unit that launches them).
struct TcArgs {
  Geometry g;
  CachePtrs p;
  const __half *q;
  float *out;
  const __half *k_new, *v_new;  // fused append: the step's new K, V rows [B][H][d]
  int new_row;                  // their residual row (the last one), or -1
  float scale_log2;
  int64_t n_quant, n_fp16, n_sink;
  int S_h, F_h, U;  // quantized units, fp16 units, units per head
  int CPU;          // fp16 chunks per fp16 unit (grouped-query kernel)
  int UPC;          // units per fp16 chunk (warp-level split)
  int nch;          // fp16 chunks per head
  int total;        // BH * U
  int nc;           // resident blocks
  int HU;           // leading units of a head that hold no data (a head change's cost)
  int nw;           // warps given work (warp-level split; 0 where work is split by block)
  float *ws_ml, *ws_o;
  int *ws_cnt;
  int part_stride;
  int wait_limit;   // poll cap of every pipeline wait
  int stall_limit;  // debug: > 0 = first wait on a barrier nothing completes
  int64_t n_vq;     // values held quantized (the value queue's count; else n_quant)
  int CH;           // fp16 tokens per chunk (tc_fp16_chunk)
  // keys cached before RoPE (the rotary form of the MHA kernel only): the
  // query's position, 2 pi = c1 + c2 + c3, theta_i = theta[i].x + .y
  int qpos;
  float c1, c2, c3;
  float2 theta[64];
};

// Common arguments of the MHA tensor-core decode (work split, workspace);
// k_new / v_new: a fused append's rows, or null.
cudaError_t tc_fill_args(TcArgs &a, const Geometry &g, const CachePtrs &p, int64_t n_quant,
                         int64_t n_resid, int64_t n_sink, const __half *q, float *out, float scale,
                         void *ws, const __half *k_new, const __half *v_new);

// The MHA tensor-core decode with fp16 statistics (KVQ_META_F16), the
// extended one (outlier lists, the value queue, per-sequence lengths) and
// the one with per-sequence lengths only, each built in its own translation
// unit.
cudaError_t launch_tc_f16(TcArgs &a, int num_sms, cudaStream_t st);
cudaError_t launch_tc_ext(TcArgs &a, int num_sms, cudaStream_t st);
cudaError_t launch_tc_rag(TcArgs &a, int num_sms, cudaStream_t st);

// The MHA tensor-core family a cache takes: 0 = no options; 1 = outlier
// lists or the value queue (per-sequence lengths too, if the cache has them);
// 2 = per-sequence lengths only.
inline int tc_ext_kind(const Geometry &g) {
  if (g.n_out > 0 || g.vq) return 1;
  return g.ragged ? 2 : 0;
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnit = 128;    // tokens per stream-K work unit (grouped-query kernel)
constexpr int kTile = 32;     // tokens per warp tile (two 16-token MMA tiles)
constexpr int kD = 128;
constexpr float kSub = 16777216.0f;  // 2^24: undoes the subnormal scale of the code operands
// Lazy online softmax: probabilities are taken against a running reference
// that may sit up to kSlack (log2 units) below the true maximum, so p <=
// 2^kSlack; the value operand carries p * 2^-kSlack * scale (at most the
// value scale: within fp16 range) and the output row multiplies it back.
// The slack is small because the operand's fp16 hi + lo split is exact to
// about 2^-22 only above fp16's normal minimum 2^-14: a weight p whose
// p * 2^-kSlack * scale falls below it keeps only an absolute 2^-25, and
// over thousands of tokens those errors add up to an offset of the output
// (on a head whose softmax is held by a few tokens, 2e-3 with a slack of 8).
// A larger reference jump costs one rescale of the accumulators.
constexpr int kSlackLog2 = 2;
constexpr float kSlack = (float)kSlackLog2;
constexpr float kSlackScale = (float)(1 << kSlackLog2);
constexpr float kInvSlack = 1.0f / kSlackScale;
constexpr int kDrainLimit = 1 << 26;



struct TcLayout {
  int ring, sB, bars, total;
};

// pre: bytes the block keeps ahead of the rings (the rotary form's cos / sin
// table)
__host__ __device__ constexpr TcLayout tc_layout(int slot_bytes, int nslot, int sb_bytes,
                                                 int pre = 0) {
  TcLayout L{};
  L.ring = pre;
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
// operand (fp16 hi/lo words in fragment order, per key group), reused to
// transpose the output row at a head's end, and 64 bytes that stay zero.
// KM (KIVI): 2 = G 16, two key groups per tile, statistics inside the block;
// 1 = G 32, one group, inside the block; 0 = G >= 64, the tile's group read
// from the separate key-statistics array.  MF: statistics stored in fp16
// (MSZ = 2 bytes each) instead of fp32.
// OUT = 1 (the extended kernel with outliers or the value queue): the block
// may carry outlier lists (up to
// kMaxOutliers words per token and tensor), so its size is known only at run
// time: the slot reserves room for the largest, and the per-warp area adds
// the query in the score domain and the outliers' value corrections (128
// floats each).
// RP (the rotary form, keys cached before RoPE): the key scores run on the
// CUDA cores, so the per-warp area holds the tile's per-pair key weights
// (3 x 32 float4) instead of the key operand, and the block keeps a 32 x 32
// float4 table of cos / sin ahead of the rings.
constexpr int kMaxOutliers = 8;
template <int BITS, int SCHEME, int NGV, int NGK, int KM, int MF = 0, int OUT = 0, int RP = 0>
struct SlotCfg {
  static constexpr int MSZ = MF ? 2 : 4;
  static constexpr int RB = kD * BITS / 8;
  static constexpr int off_vc = kTile * RB;
  static constexpr int off_vs = 2 * kTile * RB;
  static constexpr int off_vz = off_vs + kTile * NGV * MSZ;
  static constexpr int off_ks = off_vz + kTile * NGV * MSZ;  // InnerQ
  static constexpr int off_kz = off_ks + kTile * NGK * MSZ;  // InnerQ
  static constexpr bool KIN = SCHEME == KVQ_KIVI && KM >= 1;
  static constexpr int KGB = (KM == 2 ? 2 : 1) * 2 * kD * MSZ;  // KIVI key statistics of a tile
  static constexpr int BB = SCHEME == KVQ_KIVI ? off_ks + (KIN ? KGB : 0) : off_kz + kTile * NGK * MSZ;
  static constexpr int BBX = BB + (OUT == 1 ? 2 * kTile * kMaxOutliers * 4 : 0);  // room in the slot
  static constexpr int KMB = SCHEME == KVQ_KIVI && !KIN ? KGB : 0;  // separate copy
  static constexpr int off_km = KIN ? off_ks : BBX;
  static constexpr int off_q = BBX + KMB;
  static constexpr int bytes = off_q + kD * 2;
  static constexpr int CH = off_q / (4 * kD) < 8 ? off_q / (4 * kD) : 8;  // fp16 tokens per chunk
  // per warp: KIVI key operand (512 B per group; also the 512 B output
  // transpose at a head's end), the outlier extras, 64 zero bytes
  static constexpr int SBO = RP ? 3 * 32 * 16 : (SCHEME == KVQ_KIVI && KM == 2 ? 1024 : 512);
  static constexpr int SBB = SBO + (OUT == 1 ? 1024 : 0) + 64;
  static constexpr int sb_xtra = SBO / 4;       // word offset of the extras (OUT)
  static constexpr int sb_zero = SBB / 4 - 16;  // word offset of the zero block
  static constexpr int CSB = RP ? 32 * 32 * 16 : 0;  // the rotary form's cos / sin table
  static constexpr int nslot = tc_layout(bytes, 3, SBB, CSB).total <= 112 * 1024 ? 3 : 2;
  static constexpr int smem = tc_layout(bytes, nslot, SBB, CSB).total;
};

// Stored statistics as fp32: element i of a row at `base`, the pair (i, i +
// 1) (i even), and N consecutive values (a per-token row of N groups).
template <int MF>
__device__ __forceinline__ float ld_stat(const uint8_t *base, int i) {
  if (MF) return __half2float(reinterpret_cast<const __half *>(base)[i]);
  return reinterpret_cast<const float *>(base)[i];
}
template <int MF>
__device__ __forceinline__ float2 ld_stat2(const uint8_t *base, int i) {
  // (byte offset i * size: i is even, so the pair is aligned)
  if (MF) return __half22float2(*reinterpret_cast<const __half2 *>(base + i * 2));
  return *reinterpret_cast<const float2 *>(base + i * 4);
}
template <int MF, int N>
__device__ __forceinline__ void ld_stat_row(const uint8_t *base, float (&out)[N]) {
  static_assert(N == 2 || N == 4, "rows of 2 or 4 groups");
  if (MF) {
    if (N == 4) {
      const uint2 w = *reinterpret_cast<const uint2 *>(base);
      const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
      out[0] = a.x;
      out[1] = a.y;
      out[2 % N] = b.x;
      out[3 % N] = b.y;
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(base));
      out[0] = a.x;
      out[1 % N] = a.y;
    }
  } else if (N == 4) {
    const float4 a = *reinterpret_cast<const float4 *>(base);
    out[0] = a.x;
    out[1] = a.y;
    out[2 % N] = a.z;
    out[3 % N] = a.w;
  } else {
    const float2 a = *reinterpret_cast<const float2 *>(base);
    out[0] = a.x;
    out[1 % N] = a.y;
  }
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

// Barrier waits on a shared-window address (bar_s) or a pointer.
__device__ __forceinline__ bool bar_try_wait(uint32_t bar_s, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar_s), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool bar_wait(uint32_t bar_s, uint32_t parity, int limit) {
  if (bar_try_wait(bar_s, parity)) return true;
  for (int it = 0; it < limit; ++it)
    if (bar_try_wait(bar_s, parity)) return true;
  return false;
}

__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity, int limit) {
  return bar_wait(smem_u32(bar), parity, limit);
}

// Programmatic dependent launch (the launch attribute set by
// launch_cooperative).  grid_dep_trigger: the next launch on the stream may
// start its blocks as this grid's blocks leave the SMs.  grid_dep_wait: wait
// until the previous grid on the stream has completed and its writes are
// visible; nothing before it may read or write global memory that another
// kernel writes (a launch without the attribute returns at once).
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once per launch: evicted first, so the stream of
// cache blocks does not push out the partials and other rows read again.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Predicated on `on` (one lane), without a branch: posts tx expected bytes on
// the barrier at bar_s and copies `bytes` from src to dst_s (shared-window
// addresses) with L2 policy pol.
__device__ __forceinline__ void bulk_g2s_pred(bool on, uint32_t bar_s, uint32_t tx, uint32_t dst_s,
                                              const void *src, uint32_t bytes, uint64_t pol) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %0, 0;\n"
      " @p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n"
      " @p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%3], "
      "[%4], %5, [%1], %6;\n}\n" ::"r"((int)on),
      "r"(bar_s), "r"(tx), "r"(dst_s), "l"(src), "r"(bytes), "l"(pol)
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

// (x & m) | c in one instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(m), "r"(c));
  return d;
}

template <int BITS>
__device__ __forceinline__ uint32_t shifted(uint32_t w) {
  return BITS == 2 ? (w >> 10) : (w >> 8);
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz: relative error about
// 2^-22; 2^-inf = 0).  Softmax weights only.
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Multiplier carried by the code at position p (see ext).
template <int BITS>
__host__ __device__ __forceinline__ float pos_factor(int p) {
  if (BITS == 2) return (float)(1 << (2 * (p <= 4 ? p : p - 5)));
  return (p & 1) ? 16.0f : 1.0f;
}

// 1 / pos_factor(p), exact (a power of two).
template <int BITS>
__device__ __forceinline__ float inv_pos_factor(int p) {
  const int e = BITS == 2 ? 2 * (p <= 4 ? p : p - 5) : ((p & 1) ? 4 : 0);
  return __int_as_float((127 - e) << 23);
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

// Unit range [x0, x1) of block x.
__device__ __forceinline__ void block_range(const TcArgs &a, int x, int &x0, int &x1) {
  x0 = (int)((int64_t)x * a.total / a.nc);
  x1 = (int)((int64_t)(x + 1) * a.total / a.nc);
}

// What block range [x0, x1) holds of head bh: quantized tokens [tq0, tq1)
// (from its units [0, S_h)) and fp16 chunks [c0, c1) (from its units
// [S_h, U), CPU chunks each).
struct Seg {
  int tq0, tq1, c0, c1;
};
__device__ __forceinline__ Seg seg_in(const TcArgs &a, int bh, int x0, int x1) {
  Seg s;
  const int base = bh * a.U;
  const int ua = max(x0, base) - base;
  const int ub = min(min(x1, base + a.U) - base, a.S_h);
  s.tq0 = ua * kUnit;
  s.tq1 = ua < ub ? (int)min((int64_t)ub * kUnit, a.n_quant) : s.tq0;
  const int fa = max(x0 - base - a.S_h, 0), fb = min(x1 - base - a.S_h, a.F_h);
  s.c0 = fa * a.CPU;
  s.c1 = fa < fb ? min(fb * a.CPU, a.nch) : s.c0;
  return s;
}

// Partials of head bh under the warp-level split: one per warp whose unit
// range touches the head, slot (warp - first such warp).
__device__ __forceinline__ int head_nparts(const TcArgs &a, int bh) {
  const int base = bh * a.U;
  return owner_of(base + a.U - 1, a.total, a.nw) - owner_of(base, a.total, a.nw) + 1;
}

// Partials are stored XOR-ed with kEnc: no float that arithmetic produces
// (kEnc is a signalling NaN) encodes to 0, so a zero word means "not
// written yet" and the zero-filled workspace starts empty.  The head's merger
// is fixed in advance: the warp in slot 0, whose range holds the head's first
// unit and so ends in this head (or holds all of it).  After publishing its
// own partial it polls (bounded) until the others are visible, merges them
// with the log-sum-exp rule, writes the output row and zeroes the partials
// again.
//
// Memory model: every access to a partial word -- the writer's store, the
// merger's polling loads and its zeroing stores -- is a relaxed access at GPU
// scope (st.relaxed.gpu / ld.relaxed.gpu), so the accesses are morally strong
// and there is no data race; the data is its own flag (each 32-bit word is
// written once per launch, and a non-zero word is the final value), so no
// release / acquire ordering between words is needed.  The loads are asm
// volatile with a memory clobber: the compiler cannot hoist them out of the
// poll loop.  The grids that merge this way are launched cooperatively, so
// every block of the grid is resident and every poll can end.
constexpr uint32_t kEnc = 0x7fbadbadu;
constexpr int kMergePolls = 1 << 22;

__device__ __forceinline__ void st_relaxed(uint4 *p, uint4 v) {
  asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_relaxed(uint2 *p, uint2 v) {
  asm volatile("st.relaxed.gpu.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y)
               : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed(const uint4 *p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_relaxed(const uint2 *p) {
  uint2 v;
  asm volatile("ld.relaxed.gpu.global.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint4 enc4(float4 v) {
  return make_uint4(__float_as_uint(v.x) ^ kEnc, __float_as_uint(v.y) ^ kEnc,
                    __float_as_uint(v.z) ^ kEnc, __float_as_uint(v.w) ^ kEnc);
}

__device__ __forceinline__ bool vis4(uint4 v) {
  return v.x != 0u && v.y != 0u && v.z != 0u && v.w != 0u;
}

// Stores partial `slot` of head bh: the lane's 4 output channels and (lane 0)
// m, l.
__device__ __forceinline__ void publish_partial(const TcArgs &a, int bh, int slot, float4 o,
                                                float m, float l) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)bh * a.part_stride + slot;
  st_relaxed(reinterpret_cast<uint4 *>(a.ws_o + row * kD) + lane, enc4(o));
  if (lane == 0)
    st_relaxed(reinterpret_cast<uint2 *>(a.ws_ml) + row,
               make_uint2(__float_as_uint(m) ^ kEnc, __float_as_uint(l) ^ kEnc));
}

// Run by the whole warp in slot 0 of head bh after it published its own
// partial (a lane reads back only what it wrote itself there): merges the
// head's partials (nparts_given, or by the uniform unit layout) and writes
// the output row.  Returns false if they did not
// all appear within the poll bound (status word set).
// MB: partial rows fetched in one round of loads when nparts <= MB (the
// kernel's last call can afford many registers).
template <int MB>
__device__ bool merge_head(const TcArgs &a, int bh, int nparts_given = -1) {
  const int lane = threadIdx.x & 31;
  const int nparts = nparts_given >= 0 ? nparts_given : head_nparts(a, bh);
  const int64_t base = (int64_t)bh * a.part_stride;
  const uint2 *ml = reinterpret_cast<const uint2 *>(a.ws_ml) + base;
  const uint4 *wo = reinterpret_cast<const uint4 *>(a.ws_o + base * kD);
  bool ok = true;
  float Ls = 0.0f, O[4] = {0.f, 0.f, 0.f, 0.f};
  if (nparts <= MB) {
    // every (m, l) and o row in one round of loads, repeated until all are
    // visible
    uint2 v = make_uint2(1u, 1u);
    uint4 o[MB];
    bool all = false;
    for (int it = 0; it < kMergePolls && !all; ++it) {
      if (it > 0) __nanosleep(32);
      v = lane < nparts ? ld_relaxed(ml + lane) : make_uint2(1u, 1u);
      bool mine = v.x != 0u && v.y != 0u;
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        o[j] = j < nparts ? ld_relaxed(wo + (int64_t)j * (kD / 4) + lane) : make_uint4(1, 1, 1, 1);
        mine = mine && vis4(o[j]);
      }
      all = __all_sync(0xffffffffu, mine);
    }
    ok = all;
    if (ok) {
      const float ms = lane < nparts ? __uint_as_float(v.x ^ kEnc) : -INFINITY;
      float M = ms;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      const float w = ms != -INFINITY ? exp2_approx(ms - M) : 0.0f;
      Ls = w * (lane < nparts ? __uint_as_float(v.y ^ kEnc) : 0.0f);
#pragma unroll
      for (int j = 0; j < MB; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, j & 31);
        if (j < nparts && wj != 0.0f) {
          O[0] = fmaf(wj, __uint_as_float(o[j].x ^ kEnc), O[0]);
          O[1] = fmaf(wj, __uint_as_float(o[j].y ^ kEnc), O[1]);
          O[2] = fmaf(wj, __uint_as_float(o[j].z ^ kEnc), O[2]);
          O[3] = fmaf(wj, __uint_as_float(o[j].w ^ kEnc), O[3]);
        }
      }
    }
  } else {
    // (m, l) of partial s sits in lane s % 32; every load is re-polled
    // (bounded) until its words are non-zero
    auto ml_of = [&](int s) -> uint2 {
      uint2 v = ld_relaxed(ml + s);
      for (int it = 0; it < kMergePolls && (v.x == 0u || v.y == 0u); ++it) {
        __nanosleep(32);
        v = ld_relaxed(ml + s);
      }
      return v;
    };
    float M = -INFINITY;
    for (int s = lane; s < nparts; s += 32) {
      const uint2 v = ml_of(s);
      ok = ok && v.x != 0u && v.y != 0u;
      M = fmaxf(M, __uint_as_float(v.x ^ kEnc));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    ok = __all_sync(0xffffffffu, ok);
    for (int s0 = 0; s0 < nparts && ok; s0 += 32) {
      float w = 0.0f;
      if (s0 + lane < nparts) {
        const uint2 v = ld_relaxed(ml + s0 + lane);
        const float ms = __uint_as_float(v.x ^ kEnc);
        if (ms != -INFINITY) {
          w = exp2_approx(ms - M);
          Ls = fmaf(w, __uint_as_float(v.y ^ kEnc), Ls);
        }
      }
      const int nb = min(32, nparts - s0);
      for (int j0 = 0; j0 < nb; j0 += 8) {
        uint4 o[8];
        bool ready = false;
        for (int it = 0; it < kMergePolls && !ready; ++it) {
          bool mine = true;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            o[j] = j0 + j < nb ? ld_relaxed(wo + (int64_t)(s0 + j0 + j) * (kD / 4) + lane)
                               : make_uint4(1, 1, 1, 1);
            mine = mine && vis4(o[j]);
          }
          ready = __all_sync(0xffffffffu, mine);
          if (!ready) __nanosleep(32);
        }
        ok = ok && ready;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
          if (j0 + j < nb && wj != 0.0f) {
            O[0] = fmaf(wj, __uint_as_float(o[j].x ^ kEnc), O[0]);
            O[1] = fmaf(wj, __uint_as_float(o[j].y ^ kEnc), O[1]);
            O[2] = fmaf(wj, __uint_as_float(o[j].z ^ kEnc), O[2]);
            O[3] = fmaf(wj, __uint_as_float(o[j].w ^ kEnc), O[3]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
  if (!__all_sync(0xffffffffu, ok)) {
    if (lane == 0 && a.p.status) atomicExch(a.p.status, KVQ_ETIMEOUT);
    return false;
  }
  const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
  reinterpret_cast<float4 *>(a.out + ((int64_t)(bh / a.g.H) * a.g.Hq + bh % a.g.H) * kD)[lane] =
      make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
  // leave the workspace as found: partials zero
  for (int s = 0; s < nparts; ++s)
    st_relaxed(reinterpret_cast<uint4 *>(a.ws_o + base * kD) + (int64_t)s * (kD / 4) + lane,
               make_uint4(0, 0, 0, 0));
  for (int s = lane; s < nparts; s += 32)
    st_relaxed(reinterpret_cast<uint2 *>(a.ws_ml) + base + s, make_uint2(0, 0));
  return true;
}

}  // namespace

// Poll cap of the debug stall (kvq_debug_stall_waits); 0 = off.
int debug_stall_limit();

}  // namespace kvq
