// attn_internal.h -- parameter blocks and launchers shared between the C ABI
// layer (attn_api.cu) and the kernels (attn_tc.cu, attn_f32.cu).  Not part
// of the public interface.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300_attn {

// Problem description common to every kernel.  Sizes are validated by the
// API layer before any kernel sees them.
struct CommonParams {
  const int32_t* total_lengths;  // [B] or nullptr
  const int32_t* past_lengths;   // [B] or nullptr
  const float* mask;             // [mask_planes, Sq, Sk] or nullptr
  void* out;
  int B, Hq, Hkv, Sq, Sk, kv_capacity, D, group;
  int causal, local_window, out_layout, mask_planes;
  int mask_vec4;      // 1: every mask row starts 16-byte aligned (Sk % 4 == 0)
  float scale;        // softmax scale
  float scale_log2;   // scale * log2(e)
  float softcap;      // > 0: soft-cap value c
  float inv_softcap;  // 1 / c
  // soft-cap folded into log2 units: softcap(scale*s)*log2(e) = k2 * r + k3,
  // r = 1 / (2^(k1 * s) + 1), k1 = 2 log2(e) scale / c, k2 = -2 c log2(e), k3 = c log2(e)
  float sc_k1, sc_k2, sc_k3;
  // the same through the hardware tanh: softcap(scale*s)*log2(e) = sc_out * tanh(sc_in * s),
  // sc_in = scale / c, sc_out = c log2(e) (tensor-core kernels)
  float sc_in, sc_out;
  uint64_t timeout_ns;
  int* status;        // device status word (timeouts)
  // split-KV (tensor-core kernel): each query tile's key tiles are cut into
  // num_splits contiguous ranges handled by different CTAs
  int num_splits;     // 1: no split, rows are finished in the kernel
  float* ws_o;        // num_splits > 1: partial rows [num_splits, B, Hq, Sq, D], each O / l
  float* ws_lse;      // num_splits > 1: partial log-sum-exp [num_splits, B, Hq, Sq]
  float* lse;         // nullable: the row log-sum-exp [B, Hq, Sq] (natural log)
};

// Combines split-KV partial rows into the output (and the log-sum-exp).
struct MergeParams {
  const float* ws_o;
  const float* ws_lse;
  void* out;
  float* lse;  // nullable
  int B, Hq, Sq, D, num_splits, out_layout;
  bool bf16;
};

// tcgen05 kernel: Q / K / V reach shared memory through TMA tensor maps.
struct TcParams {
  CUtensorMap tmap_q;  // dims {D, Sq, B*Hq},          box {64, 128, 1}, 128B swizzle
  CUtensorMap tmap_k;  // dims {D, kv_capacity, B*Hkv}, box {64, 128, 1}, 128B swizzle
  CUtensorMap tmap_v;  // same as tmap_k
  CommonParams c;
};

// fp32 CUDA-core kernel.
struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  CommonParams c;
};

// Single-lane tensor-core kernel (one query tile per CTA, Q in tensor
// memory): fp32 inputs as bf16 pieces (K / V split into a workspace by a
// pre-pass: k0, k1, k2, v0, v1, each [B, Hkv, kv_capacity, D], read through
// one TMA map over [5 * B * Hkv planes, kv_capacity rows, D]), or bf16 / f16
// inputs with D = 256 or 384 (maps over the caller's k and v; at D = 384 Q
// goes to shared memory by TMA as well).  K piece t of kv
// plane i is plane t * B * Hkv + i of tmap_k; V piece t is plane
// v_plane0 + t * B * Hkv + i of tmap_v.
struct LaneParams {
  CUtensorMap tmap_q;  // 16-bit D = 384 only: Q [B*Hq planes, Sq rows, D], box {64, 128, 1}
  CUtensorMap tmap_k;  // box {64, key tile (64, or 32 at D = 384), 1}, 128B swizzle
  CUtensorMap tmap_v;
  const void* q;       // [B, Hq, Sq, D] fp32 or 16-bit, split / stored to tensor memory in the kernel
  int v_plane0;
  CommonParams c;
};

constexpr int kTcBlockM = 128;  // query rows per tcgen05 CTA
constexpr int kTcBlockN = 128;  // keys per tcgen05 tile
constexpr int kF32BlockM = 64;  // query rows per fp32 CTA
constexpr int kF32MaxHeadDim = 384;  // fp32-exact kernel: any head dim up to this

// Launchers.  They assume validated parameters.
cudaError_t launch_attn_tc(const TcParams& p, bool bf16, cudaStream_t stream);
cudaError_t launch_attn_f32(const F32Params& p, cudaStream_t stream);
cudaError_t launch_attn_f32tc(const LaneParams& p, const float* k, const float* v, void* ws, cudaStream_t stream);
cudaError_t launch_attn_lane16(const LaneParams& p, bool bf16, cudaStream_t stream);
// workspace bytes of the fp32 tensor-core path for B * Hkv * kv_capacity * D elements of K (and of V)
size_t f32tc_workspace_bytes(int64_t kv_elems);
constexpr int kF32TcPlanesPerKv = 5;  // k0, k1, k2, v0, v1
cudaError_t launch_selftest_wait(uint64_t timeout_ns, int* status, cudaStream_t stream);
cudaError_t launch_attn_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_fill_f32(float* dst, int64_t n, float value, cudaStream_t stream);

}  // namespace gb300_attn
