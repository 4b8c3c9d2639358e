// attn_f32tc.cu -- fp32 attention forward on the tensor cores (sm_103a) by
// error-compensated bf16 splits: the fp32 instance of the single-lane kernel
// in attn_lane1.cuh, and the pre-pass that splits K and V.
//
// The method is the tiled online softmax of "onnx-runtime-ep-cuda
// 0.1.0-dev.5, src/kernels/flash_attention.rs" on fp32 inputs, as
// "pictor-kernels 0.1.0, src/gpu_backend/cuda_imagen_attn_kernels.rs"
// ("Parity-first design") requires for its DiT joint attention: fp32 in,
// fp32 out, every intermediate in fp32 accuracy.  That page runs the products
// on CUDA cores and leaves tensor-core tuning for later; here both products
// run as bf16 tcgen05 MMAs with fp32 accumulation in tensor memory, each fp32
// operand carried as a sum of bf16 pieces (x0 = bf16(x), x1 = bf16(x - x0),
// ..., every subtraction exact in fp32):
//   S = Q K^T   three pieces of Q and of K (residual <= 2^-24 |x|), six
//               products q0k0 + q0k1 + q1k0 + q0k2 + q1k1 + q2k0 (the dropped
//               terms are below 3 * 2^-24 |q k|): the scores, which the
//               exponential turns into relative errors of P, keep fp32
//               accuracy even for large |s|;
//   O = P V     two pieces of P and of V (residual <= 2^-16), three products
//               p0v0 + p0v1 + p1v0; P's error is relative to each term and
//               the output is a weighted average of V, so its error stays
//               near 2^-16 max|v| at worst.
#include "attn_lane1.cuh"

namespace gb300_attn {
namespace {

using lane1::split_pair;
constexpr int kKP = lane1::In<lane1::kInF32Split>::KP;  // pieces of K
constexpr int kVP = lane1::In<lane1::kInF32Split>::VP;  // pieces of V

// ------------------------------------------------------------------ pre-pass
// One thread per four consecutive elements of K and of V: K -> three pieces,
// V -> two, or zeros for rows at or past the batch's valid length
// min(total_lengths[b] (else Sk), Sk).  D is a multiple of 4.  Workspace
// layout: [k0, k1, k2, v0, v1], each [B, Hkv, kv_capacity, D] bf16.
__global__ void __launch_bounds__(256) f32_split_kv_kernel(const float* __restrict__ k,
                                                           const float* __restrict__ v,
                                                           __nv_bfloat16* __restrict__ ws,
                                                           const int32_t* __restrict__ total_lengths,
                                                           int Hkv, int kv_capacity, int Sk, int D,
                                                           int64_t n_elems) {
  // the attention kernel (a programmatic dependent) may start its prologue
  // and its first Q rows now; it waits for this grid before reading the pieces
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t n4 = n_elems / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i * 4;
    const int64_t row_all = e / D;  // plane * kv_capacity + row
    const int64_t plane = row_all / kv_capacity;
    const int row = (int)(row_all - plane * kv_capacity);
    const int b = (int)(plane / Hkv);
    int valid = total_lengths ? __ldg(total_lengths + b) : Sk;
    valid = valid < Sk ? valid : Sk;
    float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
    if (row < valid) {
      kx = __ldg(reinterpret_cast<const float4*>(k + e));
      vx = __ldg(reinterpret_cast<const float4*>(v + e));
    }
    uint32_t k01[kKP], k23[kKP], v01[kVP], v23[kVP];
    split_pair<kKP>(kx.x, kx.y, k01);
    split_pair<kKP>(kx.z, kx.w, k23);
    split_pair<kVP>(vx.x, vx.y, v01);
    split_pair<kVP>(vx.z, vx.w, v23);
#pragma unroll
    for (int pc = 0; pc < kKP; ++pc)
      *reinterpret_cast<uint2*>(ws + pc * n_elems + e) = make_uint2(k01[pc], k23[pc]);
#pragma unroll
    for (int pc = 0; pc < kVP; ++pc)
      *reinterpret_cast<uint2*>(ws + (kKP + pc) * n_elems + e) = make_uint2(v01[pc], v23[pc]);
  }
}

}  // namespace

// Splits K and V into the workspace, then runs the attention kernel; both on
// `stream`.  The parameters are validated by the caller.
cudaError_t launch_attn_f32tc(const LaneParams& P, const float* k, const float* v, void* ws, cudaStream_t stream) {
  const CommonParams& c = P.c;
  const int64_t n = (int64_t)c.B * c.Hkv * c.kv_capacity * c.D;
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t want = (n / 4 + 255) / 256;
  const int blocks = (int)(want < (int64_t)sms * 16 ? (want > 0 ? want : 1) : (int64_t)sms * 16);
  f32_split_kv_kernel<<<blocks, 256, 0, stream>>>(k, v, static_cast<__nv_bfloat16*>(ws), c.total_lengths,
                                                   c.Hkv, c.kv_capacity, c.Sk, c.D, n);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return c.D == 64 ? lane1::launch_lane1<64, lane1::kInF32Split>(P, stream)
                   : lane1::launch_lane1<128, lane1::kInF32Split>(P, stream);
}

size_t f32tc_workspace_bytes(int64_t kv_elems) { return (size_t)kv_elems * 2 * (kKP + kVP); }

}  // namespace gb300_attn
