// attn_tc.cu -- dispatch of the tcgen05 attention kernels by input type and
// head dim (the kernels live in attn_tc.cuh, instantiated per type and head
// dim in attn_tc_<type>_d<D>.cu).
#include "attn_internal.h"

namespace gb300_attn {

cudaError_t launch_attn_tc_bf16_d64(const TcParams& P, cudaStream_t stream);
cudaError_t launch_attn_tc_bf16_d128(const TcParams& P, cudaStream_t stream);
cudaError_t launch_attn_tc_f16_d64(const TcParams& P, cudaStream_t stream);
cudaError_t launch_attn_tc_f16_d128(const TcParams& P, cudaStream_t stream);

cudaError_t launch_attn_tc(const TcParams& P, bool bf16, cudaStream_t stream) {
  if (P.c.D == 64) return bf16 ? launch_attn_tc_bf16_d64(P, stream) : launch_attn_tc_f16_d64(P, stream);
  return bf16 ? launch_attn_tc_bf16_d128(P, stream) : launch_attn_tc_f16_d128(P, stream);
}

}  // namespace gb300_attn
