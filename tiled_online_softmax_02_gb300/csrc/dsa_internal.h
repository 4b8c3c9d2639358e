// dsa_internal.h -- internal interface of the DSA indexer's index selection
// (dsa_select.cu) to the C ABI (attn_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace gb300_attn {

// DSA indexer index selection (dsa_select.cu).
struct DsaParams {
  CUtensorMap tmap_key;  // key as {D, T, B}, box {64 bytes of dims, 64, 1}, 64B swizzle (tile path)
  int tile_path;         // 1: the TMA-fed score kernel (tmap_key valid), 0: the general one
  const void* query;    // [B, S, H, D] of dtype
  const void* key;      // [B, T, D]
  const void* weights;  // [B, S, H]
  const float* bias;    // [B, 1, S, T]
  float* scores;        // workspace [B * S, T]: fp32 scores, 0xFFFFFFFF where not allowed
  int64_t* out;         // [B, 1, S, top_k]
  int B, S, H, D, T, top_k, dtype;  // dtype: 0 f32, 1 f16, 2 bf16
  float scale, weights_scale;
  uint64_t timeout_ns;
  int* status;          // device status word (timeouts)
  uint64_t neg_zero2;   // (-0.0f, -0.0f) as a packed pair: the addend of the rounded products
  unsigned long long* unit_counter;  // tile path: units handed out past the grid size, zero at launch (in the workspace)
};

// Whether the TMA-fed score kernel takes a problem: key / query rows of
// whole chunks of its K rows, q of a row in shared memory.
bool dsa_tile_path_ok(int dtype, int H, int D);
// The key tensor map the TMA-fed score kernel reads (its box and swizzle
// follow the kernel's K rows); encoder = cuTensorMapEncodeTiled.  0 on success.
int dsa_encode_key_map(CUtensorMap* map, void* encoder, const void* key, int dtype, int B, int T, int D);

// Bytes of the workspace after the scores: the tile kernel's unit counter.
constexpr size_t kDsaCounterBytes = 256;
cudaError_t launch_dsa_select(const DsaParams& p, cudaStream_t stream);

}  // namespace gb300_attn
