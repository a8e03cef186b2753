// The tensor-core MHA decode with per-sequence lengths and no other option
// (continuous batching): the same kernel (kvq_decode_tc.cuh) with OUT = 2 --
// each head's counters from its sequence's prompt length and the unit layout
// by sequence -- without the outlier and value-queue code, for fp32 and fp16
// statistics, in a translation unit of its own.
#include "kvq_decode_tc.cuh"

namespace kvq {

cudaError_t launch_tc_rag(TcArgs &a, int num_sms, cudaStream_t st) {
  return a.g.meta16 ? launch_tc_mf<1, 2>(a, num_sms, st) : launch_tc_mf<0, 2>(a, num_sms, st);
}

}  // namespace kvq
