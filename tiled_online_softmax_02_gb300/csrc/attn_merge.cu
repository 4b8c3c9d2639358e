// attn_merge.cu -- the merge step of split-KV attention: each query row was
// computed over num_splits key ranges by different CTAs, each leaving its
// normalised partial row O_s and log-sum-exp L_s.  The row is
//   O = sum_s w_s O_s / sum_s w_s,  w_s = exp(L_s - max_s L_s),
//   L = max_s L_s + log(sum_s w_s),
// which is the online-softmax rescale of "onnx-runtime-ep-cuda 0.1.0-dev.5,
// src/kernels/flash_attention.rs" (`flash_attention_body`: alpha / beta
// rescale of two partial sums) applied across whole key ranges.  Rows with no
// finite score in any range are 0 with L = -inf.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"

namespace gb300_attn {
namespace {

// One warp per row, lanes over the columns (VEC = D / 32 each, D = 64 or
// 128).  Lane l fetches the log-sum-exps of ranges l and l + 32 (one round
// trip for up to 64 ranges); the maximum, the weights and their sum are
// formed with shuffles.  Then every lane issues its loads of all the
// partial rows unconditionally (a range without keys holds -inf and weight
// 0, and its partial row is never multiplied in), so they overlap.
//
// Launched as a programmatic dependent of the split kernel: its CTAs may be
// scheduled as that grid drains, and every thread waits for the whole grid
// (and its writes to the workspace) before reading.
template <int VEC>
__global__ void attn_merge_kernel(const MergeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  const int64_t plane = rows * p.D;  // floats per split in ws_o
  for (int64_t row = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); row < rows;
       row += (int64_t)gridDim.x * warps) {  // (b * Hq + h) * Sq + qi
    const float l0 = lane < p.num_splits ? __ldg(p.ws_lse + lane * rows + row) : -INFINITY;
    const float l1 = lane + 32 < p.num_splits ? __ldg(p.ws_lse + (lane + 32) * rows + row) : -INFINITY;
    float m = fmaxf(l0, l1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float w0 = (m != -INFINITY && l0 != -INFINITY) ? __expf(l0 - m) : 0.f;
    const float w1 = (m != -INFINITY && l1 != -INFINITY) ? __expf(l1 - m) : 0.f;
    float wsum = w0 + w1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    const float* src = p.ws_o + row * p.D + lane * VEC;
#pragma unroll 8
    for (int sp = 0; sp < p.num_splits; ++sp) {
      const float w = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
      float o[VEC];
      if constexpr (VEC == 4) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(src + sp * plane));
        o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
      } else {
        const float2 x = __ldg(reinterpret_cast<const float2*>(src + sp * plane));
        o[0] = x.x; o[1] = x.y;
      }
      const bool live = w != 0.f;
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += live ? w * o[v] : 0.f;
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    const int64_t qi = row % p.Sq;
    const int64_t bh = row / p.Sq;
    const int64_t h = bh % p.Hq, b = bh / p.Hq;
    const int64_t base = (p.out_layout == 0 ? row * p.D : ((b * p.Sq + qi) * p.Hq + h) * p.D) + lane * VEC;
    uint32_t packed[VEC / 2];
#pragma unroll
    for (int v = 0; v < VEC / 2; ++v) {
      if (p.bf16) {
        __nv_bfloat162 x = __floats2bfloat162_rn(acc[2 * v] * inv, acc[2 * v + 1] * inv);
        packed[v] = *reinterpret_cast<uint32_t*>(&x);
      } else {
        __half2 x = __floats2half2_rn(acc[2 * v] * inv, acc[2 * v + 1] * inv);
        packed[v] = *reinterpret_cast<uint32_t*>(&x);
      }
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + base;
    if constexpr (VEC == 4)
      *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    else
      *reinterpret_cast<uint32_t*>(dst) = packed[0];
    if (p.lse != nullptr && lane == 0) p.lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

__global__ void fill_f32_kernel(float* dst, int64_t n, float value) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = value;
}

}  // namespace

cudaError_t launch_attn_merge(const MergeParams& p, cudaStream_t stream) {
  if (p.D != 64 && p.D != 128) return cudaErrorInvalidValue;  // the split path's head dims
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  const int threads = 128;  // four rows a CTA
  const int64_t blocks = (rows + 3) / 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks < 65535 * 8 ? blocks : 65535 * 8), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.D == 128 ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<4>, p) : cudaLaunchKernelEx(&cfg, attn_merge_kernel<2>, p);
}

cudaError_t launch_fill_f32(float* dst, int64_t n, float value, cudaStream_t stream) {
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  fill_f32_kernel<<<(unsigned)(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096), threads, 0, stream>>>(dst, n, value);
  return cudaGetLastError();
}

}  // namespace gb300_attn
