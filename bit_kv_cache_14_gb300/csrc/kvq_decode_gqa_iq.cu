// Grouped-query decode attention on the tensor cores, InnerQ keys with fp32
// statistics: the instantiations of tc_gqa_kernel for per-token key channel
// groups (NGK = 2 or 4; kvq_decode_gqa.cuh).
#include "kvq_decode_gqa.cuh"

namespace kvq {

cudaError_t launch_gqa_innerq(TcArgs &a, int num_sms, cudaStream_t st) {
  return launch_innerq<0>(a, num_sms, st);
}

}  // namespace kvq
