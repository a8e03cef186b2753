// The tensor-core MHA decode for KIVI caches with dense-and-sparse outlier
// lists ("大模型量化技术原理：KIVI、IntactKV、KVQuant", KVQuant / 技术原理 四):
// the same kernel (kvq_decode_tc.cuh) with the lists' corrections (keys: the
// fp16 value replaces q_c * zero_c in the score; values: p * (v - zero) into
// the channel), for fp32 and fp16 statistics, in a translation unit of its
// own so the instantiations compile in parallel.
#include "kvq_decode_tc.cuh"

namespace kvq {

cudaError_t launch_tc_out(TcArgs &a, int num_sms, cudaStream_t st) {
  return a.g.meta16 ? launch_tc_mf<1, 1>(a, num_sms, st) : launch_tc_mf<0, 1>(a, num_sms, st);
}

}  // namespace kvq
