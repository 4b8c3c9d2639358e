// attn_tc_f16_d64.cu -- instantiates the tcgen05 attention kernels for
// f16 inputs and head dim 64 (one translation unit per type and head
// dim, so they compile in parallel).
#include "attn_tc.cuh"

namespace gb300_attn {

cudaError_t launch_attn_tc_f16_d64(const TcParams& P, cudaStream_t stream) {
  return launch_attn_tc_dd<64, false>(P, stream);
}

}  // namespace gb300_attn
