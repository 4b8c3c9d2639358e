// attn_lane16.cu -- bf16 / f16 attention forward with head dim 256 or 384 on
// the tensor cores (sm_103a): the 16-bit instances of the single-lane kernel
// in attn_lane1.cuh.
//
// "pictor-kernels 0.1.0, src/gpu_backend/cuda_imagen_attn_kernels.rs"
// ("Kernel structure") compiles a wider head-dim variant of its attention
// kernel next to the D = 128 one.  For D = 256 the ping-pong tile kernel's
// two query tiles no longer fit tensor memory (S and O of one tile take
// 128 + 256 columns), so this path keeps one query tile per CTA with Q in
// tensor memory (128 columns), two 64-key S buffers and O (256 columns).
// K and V tiles come straight from the caller's tensors by TMA; V rows past
// the valid length are zeroed in shared memory before the P.V products.
// For D = 384 (the page's widest variant) O takes 384 columns, so Q moves to
// shared memory (by TMA, read by an SS-MMA), two 64-column S buffers sit
// below O, K and V stream in units (128-dim K chunks, 16-key V sub-tiles),
// and each 16-key step of P.V runs as N = 256 and N = 128 parts.
#include "attn_lane1.cuh"

namespace gb300_attn {

cudaError_t launch_attn_lane16(const LaneParams& P, bool bf16, cudaStream_t stream) {
  if (P.c.D == 384)
    return bf16 ? lane1::launch_lane1<384, lane1::kInBF16>(P, stream)
                : lane1::launch_lane1<384, lane1::kInF16>(P, stream);
  return bf16 ? lane1::launch_lane1<256, lane1::kInBF16>(P, stream)
              : lane1::launch_lane1<256, lane1::kInF16>(P, stream);
}

}  // namespace gb300_attn
