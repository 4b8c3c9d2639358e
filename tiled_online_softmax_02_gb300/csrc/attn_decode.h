// attn_decode.h -- parameters and launcher of the few-rows (decode) kernel,
// shared between the C ABI layer and attn_decode.cu.  Not part of the public
// interface.
#pragma once

#include "attn_internal.h"

namespace gb300_attn {

// Query rows per kv head (group * Sq) the decode kernel takes at most.
constexpr int kDecodeMaxRows = 32;

// Few query rows per kv head: every CTA takes one (batch, kv head) and a
// contiguous part of its key tiles, with all group * Sq query rows of that kv
// head in the N dimension of one tcgen05 product (S^T = K Q^T, O^T = V^T P^T).
struct DecodeParams {
  CUtensorMap tmap_k;  // dims {D, kv_capacity, B*Hkv}, box {64, 128, 1}, 128B swizzle
  CUtensorMap tmap_v;  // same as tmap_k
  const void* q;       // [B, Hq, Sq, D]
  int cluster;         // CTAs per thread-block cluster (1..8): each takes a part of the key
                       // tiles, and the cluster merges its partial rows in shared memory
  CommonParams c;      // c.num_splits key ranges per kv head (each one cluster); > 1 writes
                       // partial rows to c.ws_o / c.ws_lse for the merge kernel
};

cudaError_t launch_attn_decode(const DecodeParams& p, bool bf16, cudaStream_t stream);

}  // namespace gb300_attn
