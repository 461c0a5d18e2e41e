// attention_q8_q8.cu -- instantiation of the mixed-batch attention kernels for
// K format MIXATTN_KV_Q8_0 and V format MIXATTN_KV_Q8_0 (one translation unit per format pair so the
// build compiles them in parallel).
#include "attention_kernel.cuh"

namespace mixattn {

cudaError_t launch_attention_q8_q8(int head_dim, const AttnParams& p, unsigned int* err, cudaStream_t s) {
  if (head_dim == 64) return launch_attention_t<MIXATTN_KV_Q8_0, MIXATTN_KV_Q8_0, 64>(p, err, s);
  return launch_attention_t<MIXATTN_KV_Q8_0, MIXATTN_KV_Q8_0, 128>(p, err, s);
}

}  // namespace mixattn
