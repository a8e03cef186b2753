// Grouped-query decode attention on the tensor cores: the dispatch over the
// instantiations of tc_gqa_kernel (kvq_decode_gqa.cuh) and the launch.
#include "kvq_decode_gqa.cuh"

namespace kvq {

namespace {

// The template arguments the dispatch picks for a geometry.
struct GqaVariant {
  int bits, ngv, km, rg, ngk, mf;  // ngk: InnerQ key channel groups (0: KIVI)
};
GqaVariant gqa_variant(const Geometry &g) {
  const int mf = g.meta16 ? 1 : 0;
  if (g.scheme == KVQ_INNERQ)
    return GqaVariant{g.bits, kD / g.v_group, 0, g.Hq / g.H, kD / g.k_group, mf};
  return GqaVariant{g.bits, kD / g.v_group, g.k_group == 32 ? 1 : 0, g.Hq / g.H, 0, mf};
}

}  // namespace

int gqa_variant_name(const Geometry &g, char *buf, size_t len) {
  const GqaVariant v = gqa_variant(g);
  const char *mf = v.mf ? ",mf=1" : "";
  if (v.ngk)
    return snprintf(buf, len, "tc_gqa_kernel<bits=%d,scheme=innerq,ngv=%d,ngk=%d,rg=%d%s>", v.bits,
                    v.ngv, v.ngk, v.rg, mf);
  return snprintf(buf, len, "tc_gqa_kernel<bits=%d,ngv=%d,km=%d,rg=%d%s>", v.bits, v.ngv, v.km,
                  v.rg, mf);
}

bool gqa_decode_supported(const Geometry &g) {
  if (g.d != kD || (g.bits != 2 && g.bits != 4)) return false;
  if (g.vq || g.n_out || g.ragged) return false;
  const int rg = g.Hq / g.H;
  if (rg != 2 && rg != 4) return false;
  const int ngv = kD / g.v_group;
  if (ngv != 2 && ngv != 4) return false;
  if (g.scheme == KVQ_INNERQ)  // channel groups of 32 or 64
    return g.k_group == 32 || g.k_group == 64;
  return g.scheme == KVQ_KIVI && g.k_group >= 32 && g.k_group <= 128;
}

cudaError_t launch_decode_gqa(const Geometry &g, const CachePtrs &p, int64_t n_quant,
                              int64_t n_resid, int64_t n_sink, const __half *q, float *out,
                              float scale, void *ws, int num_sms, cudaStream_t st) {
  TcArgs a;
  a.g = g;
  a.p = p;
  a.q = q;
  a.out = out;
  a.k_new = nullptr;
  a.v_new = nullptr;
  a.new_row = -1;
  a.scale_log2 = scale * 1.4426950408889634f;
  // KIVI: the kernel takes whole tiles only (InnerQ masks a short last tile)
  if (g.scheme == KVQ_KIVI && n_quant % kTile != 0) return cudaErrorInvalidValue;
  a.n_quant = n_quant;
  a.n_fp16 = n_resid + n_sink;
  a.n_sink = n_sink;
  a.S_h = (int)((n_quant + kUnit - 1) / kUnit);
  const int kmb = g.scheme == KVQ_KIVI && g.k_group > kBlockTokens ? 2 * kD * 4 : 0;
  const int CH = tc_fp16_chunk(g);
  const int64_t unit_bytes = (int64_t)(kUnit / kBlockTokens) * (g.block_bytes + kmb);
  a.CPU = (int)(unit_bytes / (CH * 4 * kD));
  if (a.CPU < 1) a.CPU = 1;
  a.nch = (int)((a.n_fp16 + CH - 1) / CH);
  a.F_h = (a.nch + a.CPU - 1) / a.CPU;
  a.U = a.S_h + a.F_h;
  a.HU = 0;
  a.nw = 0;
  a.UPC = 0;
  const int64_t total = (int64_t)g.B * g.H * a.U;
  if (total >= (1LL << 31)) return cudaErrorInvalidValue;
  a.total = (int)total;
  a.part_stride = tc_part_slots(g);
  if (a.part_stride & 1) return cudaErrorInvalidValue;  // keeps ws_o 16-byte aligned
  const int rg = g.Hq / g.H;
  const int64_t BH = (int64_t)g.B * g.H;
  char *base = static_cast<char *>(ws);
  const size_t cnt = ((size_t)BH * sizeof(int) + 255) & ~(size_t)255;
  a.ws_cnt = reinterpret_cast<int *>(base);
  a.ws_ml = reinterpret_cast<float *>(base + cnt);
  a.ws_o = a.ws_ml + (size_t)BH * a.part_stride * rg * 2;
  a.wait_limit = 1 << 24;
  a.stall_limit = debug_stall_limit();
  if (g.scheme == KVQ_INNERQ)
    return g.meta16 ? launch_gqa_innerq_f16(a, num_sms, st) : launch_gqa_innerq(a, num_sms, st);
  return g.meta16 ? launch_gqa_kivi_f16(a, num_sms, st) : launch_kivi<0>(a, num_sms, st);
}

}  // namespace kvq
