// Fused decode attention on the tensor cores (MHA, head_dim 128).
//
// Same computation as decode_kernel (softmax(scale * q.K^T) V over the packed
// cache, dequantization folded into both GEMVs -- "大模型量化技术原理：KIVI、
// IntactKV、KVQuant", KIVI / 背景; InnerQ page, 方法论 3), arranged for GB300:
//
//  * Persistent, stream-K over warps: every head is a list of work units (a
//    32-token tile is one unit, an 8-token fp16 chunk of sink / residual /
//    window tokens two, plus two empty units at the head's start), and the
//    list of the whole batch is cut into equal contiguous ranges, one per
//    warp of the resident grid.  A warp leaves one partial (m, l, o) per head
//    it touches; the warp holding a head's first unit (its range ends in that
//    head, and the empty units give it less data) merges them with the
//    log-sum-exp rule once they are all visible.  No atomics, no fences.
//  * Warp-autonomous: each warp owns a small ring of shared-memory slots that
//    one lane fills with 1-D cp.async.bulk copies (a tile's whole 32-token
//    block, issued by a predicated instruction) completed on the warp's own
//    mbarriers, and keeps its own online-softmax state; nothing synchronises
//    the warps of a block.  The ring runs ahead across head ends, so the
//    copies never stop.  Every wait is bounded; a timeout sets the status
//    word and the warp drains its own copies before it returns.
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
//             hi + lo, n = (value group j, hi/lo), written once per token by
//             the token's lane; row c keeps column j(c).
//    zero points enter as q.zero per key group and sum_t p_t zero_tj per value
//    group (CUDA cores).  q is normalised by a power of two so no fp16 operand
//    can overflow (|q| <= 1, scales <= 65504).
#include <stdio.h>

#include "kvq_decode_tc.cuh"

namespace kvq {

namespace {

int g_stall_limit = 0;

}  // namespace

void set_debug_stall(long long n) { g_stall_limit = n > (1 << 30) ? (1 << 30) : (int)n; }
int debug_stall_limit() { return g_stall_limit; }

int tc_variant_name(const Geometry &g, char *buf, size_t len) {
  const TcVariant v = tc_variant(g);
  return snprintf(buf, len, "tc_decode_kernel<bits=%d,scheme=%s,ngv=%d,ngk=%d,km=%d,mf=%d,ext=%d>",
                  g.bits, g.scheme == KVQ_KIVI ? "kivi" : "innerq", v.ngv, v.ngk, v.km, g.meta16,
                  tc_ext_kind(g));
}

bool tc_decode_supported(const Geometry &g) {
  if (g.d != kD || g.Hq != g.H) return false;
  const int ngv = kD / g.v_group;
  if (ngv != 2 && ngv != 4) return false;
  if (g.scheme == KVQ_KIVI) return g.k_group >= 16 && g.k_group <= 128;
  const int ngk = kD / g.k_group;
  return ngk == 2 || ngk == 4;
}

cudaError_t tc_fill_args(TcArgs &a, const Geometry &g, const CachePtrs &p, int64_t n_quant,
                         int64_t n_resid, int64_t n_sink, const __half *q, float *out, float scale,
                         void *ws, const __half *k_new, const __half *v_new) {
  a.g = g;
  a.p = p;
  a.q = q;
  a.out = out;
  a.k_new = k_new;
  a.v_new = v_new;
  a.new_row = k_new ? (int)n_resid - 1 : -1;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_quant = n_quant;
  a.n_fp16 = n_resid + n_sink;
  a.n_sink = n_sink;
  const int64_t n_all = n_quant + n_resid + n_sink;
  a.n_vq = (g.scheme == KVQ_KIVI && g.vq) ? (n_all >= g.residual ? n_all - g.residual + 1 : 0)
                                           : n_quant;
  a.S_h = (int)((n_quant + kTile - 1) / kTile);
  // fp16 rows travel in chunks of CH tokens (K and V rows fill a ring slot up
  // to its query row; without outlier lists the kernel's SlotCfg::CH is the
  // same expression)
  const int CH = tc_fp16_chunk(g);
  a.CH = CH;
  a.CPU = 1;
  a.UPC = kChunkUnits;
  // per-sequence lengths: the counters are the longest sequence's, and any
  // sequence may hold up to R - 1 (KIVI) or S + W (InnerQ) fp16 tokens
  const int64_t fp16_units = g.ragged ? (g.scheme == KVQ_KIVI ? g.residual - 1
                                                               : (int64_t)g.residual + g.n_sink)
                                      : a.n_fp16;
  a.nch = (int)((fp16_units + CH - 1) / CH);
  a.F_h = a.nch * a.UPC;
  a.HU = kHeadUnits;
  a.U = a.HU + a.S_h + a.F_h;
  const int64_t total = (int64_t)g.B * g.H * a.U;
  if (total >= (1LL << 31)) return cudaErrorInvalidValue;
  a.total = (int)total;
  a.part_stride = tc_part_slots(g);
  // ws_o must stay 16-byte aligned (uint4 rows): BH * part_stride * 8 bytes
  // past ws_ml, so the stride is even
  if (a.part_stride & 1) return cudaErrorInvalidValue;
  const int64_t BH = (int64_t)g.B * g.H;
  char *base = static_cast<char *>(ws);
  const size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  a.ws_cnt = reinterpret_cast<int *>(base);
  a.ws_ml = reinterpret_cast<float *>(base + cnt);
  a.ws_o = a.ws_ml + (size_t)BH * a.part_stride * 2;
  a.wait_limit = 1 << 24;
  a.stall_limit = g_stall_limit;
  a.qpos = 0;
  a.c1 = a.c2 = a.c3 = 0.0f;
  return cudaSuccess;
}

cudaError_t launch_decode_tc(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                             int64_t n_resid, int64_t n_sink, const __half *q, float *out,
                             float scale, void *ws, int num_sms, cudaStream_t st,
                             const __half *k_new, const __half *v_new) {
  TcArgs a;
  const cudaError_t e =
      tc_fill_args(a, g, p, n_quant, n_resid, n_sink, q, out, scale, ws, k_new, v_new);
  if (e != cudaSuccess) return e;
  const int kind = tc_ext_kind(g);
  if (kind == 1) return launch_tc_ext(a, num_sms, st);
  if (kind == 2) return launch_tc_rag(a, num_sms, st);
  return g.meta16 ? launch_tc_f16(a, num_sms, st) : launch_tc_mf<0>(a, num_sms, st);
}

}  // namespace kvq
