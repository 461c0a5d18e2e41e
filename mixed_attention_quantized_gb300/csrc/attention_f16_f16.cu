// attention_f16_f16.cu -- instantiation of the mixed-batch attention kernels for
// K format MIXATTN_KV_F16 and V format MIXATTN_KV_F16 (one translation unit per format pair so the
// build compiles them in parallel).
#include "attention_kernel.cuh"

namespace mixattn {

cudaError_t launch_attention_f16_f16(int head_dim, const AttnParams& p, unsigned int* err, cudaStream_t s) {
  if (head_dim == 64) return launch_attention_t<MIXATTN_KV_F16, MIXATTN_KV_F16, 64>(p, err, s);
  return launch_attention_t<MIXATTN_KV_F16, MIXATTN_KV_F16, 128>(p, err, s);
}

}  // namespace mixattn
