// Decode attention over keys cached before RoPE, tensor-core form (head_dim
// 128, one query head per KV head, KIVI with key groups of 32 or more, fp32
// statistics, no cache options): the MHA tensor-core kernel with RP = 1.
//
// Method ("大模型量化技术原理：KIVI、IntactKV、KVQuant", KVQuant / 技术原理 二):
// keys are quantized before the rotary embedding, which is applied inside
// q.K^T after dequantization.  Everything but the key scores is the MHA
// kernel's (ring of bulk copies per warp, value pass on the tensor cores,
// stream-K merge); the key scores turn the query instead of the keys
// (R(p) k . R(s) q = k . R(s - p) q): one anchor R(qpos - p0) q per 32-token
// tile, the per-token turn R(-t) from a cos / sin table the block builds
// once, the dequantization folded into per-pair weights (see rope_score in
// kvq_decode_tc.cuh).  Other shapes take rope_decode_kernel (kvq_rope.cu).
#include <stdio.h>

#include "kvq_decode_tc.cuh"

namespace kvq {

namespace {

template <int BITS>
cudaError_t launch_rope_b(TcArgs &a, int num_sms, cudaStream_t st) {
  const TcVariant v = tc_variant(a.g);
  if (v.ngv == 4)
    return v.km == 1 ? launch_tc_t<BITS, KVQ_KIVI, 4, 1, 1, 0, 0, 1>(a, num_sms, st)
                     : launch_tc_t<BITS, KVQ_KIVI, 4, 1, 0, 0, 0, 1>(a, num_sms, st);
  return v.km == 1 ? launch_tc_t<BITS, KVQ_KIVI, 2, 1, 1, 0, 0, 1>(a, num_sms, st)
                   : launch_tc_t<BITS, KVQ_KIVI, 2, 1, 0, 0, 0, 1>(a, num_sms, st);
}

}  // namespace

bool tc_rope_supported(const Geometry &g) {
  if (g.d != kD || g.Hq != g.H || g.scheme != KVQ_KIVI) return false;
  if (g.meta16 || g.vq || g.ragged || g.n_out) return false;
  const int ngv = kD / g.v_group;
  return (ngv == 2 || ngv == 4) && g.k_group >= 32 && g.k_group <= 128;
}

int tc_rope_variant_name(const Geometry &g, char *buf, size_t len) {
  const TcVariant v = tc_variant(g);
  return snprintf(buf, len, "tc_decode_kernel<bits=%d,scheme=kivi,ngv=%d,km=%d,rope=1>", g.bits,
                  v.ngv, v.km);
}

cudaError_t launch_decode_tc_rope(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                                  int64_t n_resid, const __half *q, float *out, float scale,
                                  double rope_base, void *ws, int num_sms, cudaStream_t st) {
  if (!tc_rope_supported(g)) return cudaErrorInvalidValue;
  TcArgs a;
  const cudaError_t e =
      tc_fill_args(a, g, p, n_quant, n_resid, 0, q, out, scale, ws, nullptr, nullptr);
  if (e != cudaSuccess) return e;
  a.qpos = (int)(n_quant + n_resid - 1);
  rope_constants(rope_base, kD, a.theta, a.c1, a.c2, a.c3);
  return g.bits == 2 ? launch_rope_b<2>(a, num_sms, st) : launch_rope_b<4>(a, num_sms, st);
}

}  // namespace kvq
