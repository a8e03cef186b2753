// Grouped-query decode attention on the tensor cores, InnerQ keys with fp16
// statistics (KVQ_META_F16; kvq_decode_gqa.cuh).
#include "kvq_decode_gqa.cuh"

namespace kvq {

cudaError_t launch_gqa_innerq_f16(TcArgs &a, int num_sms, cudaStream_t st) {
  return launch_innerq<1>(a, num_sms, st);
}

}  // namespace kvq
