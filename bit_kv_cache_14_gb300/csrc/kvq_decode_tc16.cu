// The tensor-core MHA decode for caches whose scales and zero points are
// stored in fp16 (KVQ_META_F16): the same kernel (kvq_decode_tc.cuh) reading
// 16-bit statistics, in a translation unit of its own so the two widths
// compile in parallel.
#include "kvq_decode_tc.cuh"

namespace kvq {

cudaError_t launch_tc_f16(TcArgs &a, int num_sms, cudaStream_t st) {
  return launch_tc_mf<1>(a, num_sms, st);
}

}  // namespace kvq
