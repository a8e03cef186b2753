// Grouped-query decode attention on the tensor cores, InnerQ keys: the
// instantiations of tc_gqa_kernel for per-token channel groups (NGK = 2 or 4;
// kvq_decode_gqa.cuh), kept in a translation unit of their own so the two
// families compile in parallel.
#include "kvq_decode_gqa.cuh"

namespace kvq {

namespace {

template <int BITS, int RG>
cudaError_t launch_iq_br(TcArgs &a, int num_sms, cudaStream_t st) {
  const int ngv = kD / a.g.v_group, ngk = kD / a.g.k_group;
  if (ngv == 4)
    return ngk == 4 ? launch_gqa_t<BITS, 4, 0, RG, 4>(a, num_sms, st)
                    : launch_gqa_t<BITS, 4, 0, RG, 2>(a, num_sms, st);
  return ngk == 4 ? launch_gqa_t<BITS, 2, 0, RG, 4>(a, num_sms, st)
                  : launch_gqa_t<BITS, 2, 0, RG, 2>(a, num_sms, st);
}

}  // namespace

cudaError_t launch_gqa_innerq(TcArgs &a, int num_sms, cudaStream_t st) {
  const int rg = a.g.Hq / a.g.H;
  if (a.g.bits == 4)
    return rg == 4 ? launch_iq_br<4, 4>(a, num_sms, st) : launch_iq_br<4, 2>(a, num_sms, st);
  return rg == 4 ? launch_iq_br<2, 4>(a, num_sms, st) : launch_iq_br<2, 2>(a, num_sms, st);
}

}  // namespace kvq
