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

// One thread per (row, 2 output columns); the per-split loads are issued
// unconditionally (a range without keys holds -inf and weight 0, and its
// partial row is never multiplied in), so they overlap instead of forming a
// chain of dependent branches.
//
// Launched as a programmatic dependent of the split kernel: its CTAs may be
// scheduled as that grid drains, and every thread waits for the whole grid
// (and its writes to the workspace) before reading.
__global__ void attn_merge_kernel(const MergeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t groups = p.D / 2;
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  const int64_t plane = rows * p.D;  // floats per split in ws_o
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < rows * groups;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = idx / groups;  // (b * Hq + h) * Sq + qi
    const int c = (int)(idx - row * groups) * 2;
    float m = -INFINITY;
#pragma unroll 8
    for (int s = 0; s < p.num_splits; ++s) m = fmaxf(m, __ldg(p.ws_lse + s * rows + row));
    float2 acc = make_float2(0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
#pragma unroll 8
      for (int s = 0; s < p.num_splits; ++s) {
        const float ls = __ldg(p.ws_lse + s * rows + row);
        const float2 o = __ldg(reinterpret_cast<const float2*>(p.ws_o + s * plane + row * p.D + c));
        const bool live = ls != -INFINITY;
        const float w = live ? __expf(ls - m) : 0.f;
        acc.x += live ? w * o.x : 0.f;
        acc.y += live ? w * o.y : 0.f;
        wsum += w;
      }
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    const int64_t qi = row % p.Sq;
    const int64_t bh = row / p.Sq;
    const int64_t h = bh % p.Hq, b = bh / p.Hq;
    const int64_t base = p.out_layout == 0 ? row * p.D : ((b * p.Sq + qi) * p.Hq + h) * p.D;
    uint32_t packed;
    if (p.bf16) {
      __nv_bfloat162 v = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      packed = *reinterpret_cast<uint32_t*>(&v);
    } else {
      __half2 v = __floats2half2_rn(acc.x * inv, acc.y * inv);
      packed = *reinterpret_cast<uint32_t*>(&v);
    }
    *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + base + c) = packed;
    if (p.lse != nullptr && c == 0) p.lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

__global__ void fill_f32_kernel(float* dst, int64_t n, float value) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = value;
}

}  // namespace

cudaError_t launch_attn_merge(const MergeParams& p, cudaStream_t stream) {
  const int64_t work = (int64_t)p.B * p.Hq * p.Sq * (p.D / 2);
  const int threads = 128;
  const int64_t blocks = (work + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks < 65535 * 8 ? blocks : 65535 * 8), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_merge_kernel, p);
}

cudaError_t launch_fill_f32(float* dst, int64_t n, float value, cudaStream_t stream) {
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  fill_f32_kernel<<<(unsigned)(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096), threads, 0, stream>>>(dst, n, value);
  return cudaGetLastError();
}

}  // namespace gb300_attn
