// The extended tensor-core MHA decode: the same kernel (kvq_decode_tc.cuh)
// with the run-time cache-format options compiled in -- per-sequence lengths
// (each head's counters from its sequence's prompt length), KIVI's value queue
// (fp16 values of tokens whose key is quantized, on CUDA cores in the same
// softmax frame), and dense-and-sparse outlier lists ("大模型量化技术原理：
// KIVI、IntactKV、KVQuant", KVQuant / 技术原理 四: the fp16 value replaces
// q_c * zero_c in the score, and p * (v - zero) goes into the value channel)
// -- for fp32 and fp16 statistics, in a translation unit of its own so the
// instantiations compile in parallel with the plain ones.
#include "kvq_decode_tc.cuh"

namespace kvq {

cudaError_t launch_tc_ext(TcArgs &a, int num_sms, cudaStream_t st) {
  return a.g.meta16 ? launch_tc_mf<1, 1>(a, num_sms, st) : launch_tc_mf<0, 1>(a, num_sms, st);
}

}  // namespace kvq
