// dsa_select.cu -- sparse index selection of the DSA indexer on GB300
// (sm_103a): for every (batch, query) row, score every key position and keep
// the top_k positions.
//
// Definition: "onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/dsa_index_select.rs"
// (module doc and score kernel).  For row (b, s) and key t:
//   allowed = bias[b, 0, s, t] > -1e30
//   score   = sum_h (ascending) relu(scale * sum_d (ascending) q[b,s,h,d] k[b,t,d])
//             * (w[b,s,h] * weights_scale)  +  bias[b, 0, s, t]
// in fp32 with every multiply and add rounded separately, NaN replaced by the
// positive quiet NaN; the top min(#allowed, top_k) allowed keys by (score desc
// in f32 total order, index asc), emitted ascending and padded with -1.  The
// page fixes the precision because the output is an index set: the score
// kernel keeps that exact arithmetic (no fused multiply-add, no reordering),
// so it runs on the CUDA cores -- a tensor-core product would round
// differently and move near-tied selections.
//
//   dsa_score_kernel   one CTA per (row, 256-key block).  K arrives in
//                      32-dim chunks, transposed into shared memory; each
//                      thread keeps two keys' dot products for every head in
//                      registers (heads padded with zeros to HP, which adds
//                      exactly nothing), then takes the head sum in order.
//                      Blocks whose keys are all masked write the "not
//                      allowed" mark without computing (causal prefill skips
//                      about half the grid).
//   dsa_select_kernel  one CTA per row: 8-bit radix select over the
//                      total-order keys (four histogram passes) finds the
//                      top_k-th key, then an ordered block compaction keeps
//                      the larger keys and the lowest-index ties.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "attn_internal.h"

namespace gb300_attn {
namespace {

constexpr int kScoreThreads = 128;
constexpr int kDChunk = 32;                  // head-dim columns per shared-memory chunk
constexpr int kSelectThreads = 256;
constexpr uint32_t kNotAllowed = 0xFFFFFFFFu;  // score bits of a cell that is not allowed

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// -------------------------------------------------------------- scores
// Unit u = (row, key block of KPT * 128 keys); thread tid takes keys
// t0 + tid + 128 j, j < KPT.  HP = heads rounded up (16, 32 or 64); the
// per-thread accumulators are KPT x HP.
template <typename T, int HP, int KPT>
__global__ void __launch_bounds__(kScoreThreads) dsa_score_kernel(const DsaParams p) {
  constexpr int kKeys = KPT * kScoreThreads;
  constexpr int kStride = kKeys + 1;  // padded row of the transposed K chunk
  __shared__ float k_s[kDChunk * kStride];  // [d][key]
  __shared__ float q_s[HP * kDChunk];       // [h][d]
  __shared__ float w_s[HP];
  const T* __restrict__ query = static_cast<const T*>(p.query);
  const T* __restrict__ key = static_cast<const T*>(p.key);
  const T* __restrict__ weights = static_cast<const T*>(p.weights);
  const int tid = threadIdx.x;
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t kblocks = ((int64_t)p.T + kKeys - 1) / kKeys;
  const int64_t units = rows * kblocks;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t row = u / kblocks;
    const int64_t t0 = (u - row * kblocks) * kKeys;
    const int64_t b = row / p.S;
    const float* brow = p.bias + row * (int64_t)p.T;
    uint32_t* out_bits = reinterpret_cast<uint32_t*>(p.scores) + row * (int64_t)p.T;
    float bias_v[KPT];
    bool ok[KPT];
    bool any = false;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int64_t t = t0 + tid + j * kScoreThreads;
      bias_v[j] = t < p.T ? brow[t] : -INFINITY;
      ok[j] = bias_v[j] > -1e30f;
      any = any || ok[j];
    }
    if (!__syncthreads_or(any)) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int64_t t = t0 + tid + j * kScoreThreads;
        if (t < p.T) out_bits[t] = kNotAllowed;
      }
      continue;  // no allowed key in this block
    }
    float acc[KPT][HP];
#pragma unroll
    for (int j = 0; j < KPT; ++j)
#pragma unroll
      for (int h = 0; h < HP; ++h) acc[j][h] = 0.0f;
    if (tid < HP) w_s[tid] = tid < p.H ? to_f32(weights[row * p.H + tid]) : 0.0f;
    for (int d0 = 0; d0 < p.D; d0 += kDChunk) {
      __syncthreads();  // the previous chunk has been read
      // K chunk: key kk, dims [d0, d0 + 32), transposed; zeros outside
      for (int i = tid; i < kKeys * kDChunk; i += kScoreThreads) {
        const int kk = i / kDChunk, dd = i - kk * kDChunk;
        const int64_t t = t0 + kk;
        const int d = d0 + dd;
        k_s[dd * kStride + kk] = (t < p.T && d < p.D) ? to_f32(key[(b * p.T + t) * p.D + d]) : 0.0f;
      }
      // Q chunk of this row: heads padded with zeros
      for (int i = tid; i < HP * kDChunk; i += kScoreThreads) {
        const int h = i / kDChunk, dd = i - h * kDChunk;
        const int d = d0 + dd;
        q_s[i] = (h < p.H && d < p.D) ? to_f32(query[(row * p.H + h) * p.D + d]) : 0.0f;
      }
      __syncthreads();
      // dot products, head_dim ascending, multiply and add rounded separately
#pragma unroll 2
      for (int dd = 0; dd < kDChunk; ++dd) {
        float kv[KPT];
#pragma unroll
        for (int j = 0; j < KPT; ++j) kv[j] = k_s[dd * kStride + tid + j * kScoreThreads];
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          const float qv = q_s[h * kDChunk + dd];
#pragma unroll
          for (int j = 0; j < KPT; ++j) acc[j][h] = __fadd_rn(acc[j][h], __fmul_rn(qv, kv[j]));
        }
      }
    }
    // head sum, heads ascending
    float wsum[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) wsum[j] = 0.0f;
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      const float wprod = __fmul_rn(w_s[h], p.weights_scale);
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        float sc = __fmul_rn(p.scale, acc[j][h]);
        sc = sc > 0.0f ? sc : 0.0f;  // ReLU (a NaN dot gives 0)
        wsum[j] = __fadd_rn(wsum[j], __fmul_rn(sc, wprod));
      }
    }
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int64_t t = t0 + tid + j * kScoreThreads;
      if (t < p.T) {
        const float s = __fadd_rn(wsum[j], bias_v[j]);
        out_bits[t] = ok[j] ? (isnan(s) ? 0x7FC00000u : __float_as_uint(s)) : kNotAllowed;
      }
    }
    __syncthreads();  // w_s is rewritten by the next unit
  }
}

// -------------------------------------------------------------- selection
// Unsigned key whose order is the f32 total order (negative values reversed
// under the sign bit); the "not allowed" mark maps to 0, below every score
// (scores are never negative NaNs: NaNs were made positive).
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Exclusive prefix sum over the CTA (kSelectThreads); also returns the total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kSelectThreads / 32 ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kSelectThreads / 32) warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
  *total = warp_sums[kSelectThreads / 32 - 1];
  return before;
}

__global__ void __launch_bounds__(kSelectThreads) dsa_select_kernel(const DsaParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[kSelectThreads / 32];
  __shared__ uint32_t digit_s, rank_s;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t T = p.T;
  const int64_t chunk = (T + kSelectThreads - 1) / kSelectThreads;  // contiguous keys per thread
  const int64_t beg = tid * chunk < T ? tid * chunk : T;
  const int64_t end = beg + chunk < T ? beg + chunk : T;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint32_t* bits = reinterpret_cast<const uint32_t*>(p.scores) + row * (int64_t)T;
    int64_t* out = p.out + row * (int64_t)p.top_k;
    uint32_t n_ok = 0;
    for (int64_t t = beg; t < end; ++t) n_ok += bits[t] != kNotAllowed;
    uint32_t allowed;
    block_exclusive_scan(n_ok, warp_sums, &allowed);
    const uint32_t keep = allowed < (uint32_t)p.top_k ? allowed : (uint32_t)p.top_k;
    for (int64_t i = keep + tid; i < p.top_k; i += kSelectThreads) out[i] = -1;
    if (keep == 0) continue;
    // radix select of the keep-th largest key, 8 bits at a time from the top
    uint32_t prefix = 0, pmask = 0, rank = keep;
    for (int shift = 24; shift >= 0; shift -= 8) {
      hist[tid] = 0u;  // kSelectThreads == 256 bins
      __syncthreads();
      for (int64_t t = beg; t < end; ++t) {
        const uint32_t k = order_key(bits[t]);
        // cells that are not allowed (key 0) sit below every allowed one and
        // rank <= #allowed, so they never decide a digit: leave them out
        if (k != 0u && (k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l holds bins 255 - 8l ... 248 - 8l (descending); count from the top
        uint32_t c[8], s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = hist[255 - 8 * lane - i];
          s += c[i];
        }
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - s;
        if (excl < rank && rank <= incl) {  // exactly one lane
          uint32_t acc = excl;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (acc < rank && rank <= acc + c[i]) {
              digit_s = 255u - 8u * lane - i;
              rank_s = rank - acc;
            }
            acc += c[i];
          }
        }
      }
      __syncthreads();
      prefix |= digit_s << shift;
      pmask |= 255u << shift;
      rank = rank_s;
      __syncthreads();
    }
    const uint32_t thr = prefix;  // the keep-th largest key
    // ordered compaction: keys above thr, and the lowest-index keys equal to it
    uint32_t n_gt = 0, n_eq = 0;
    for (int64_t t = beg; t < end; ++t) {
      const uint32_t k = order_key(bits[t]);
      n_gt += k > thr;
      n_eq += k == thr;
    }
    uint32_t total_gt, total_eq;
    block_exclusive_scan(n_gt, warp_sums, &total_gt);
    const uint32_t eq_before = block_exclusive_scan(n_eq, warp_sums, &total_eq);
    const uint32_t ties = keep - total_gt;  // equal keys to take, lowest indices first
    const uint32_t my_ties = eq_before >= ties ? 0u : (n_eq < ties - eq_before ? n_eq : ties - eq_before);
    uint32_t n_sel_total;
    uint32_t slot = block_exclusive_scan(n_gt + my_ties, warp_sums, &n_sel_total);
    uint32_t taken = 0;
    for (int64_t t = beg; t < end; ++t) {
      const uint32_t k = order_key(bits[t]);
      const bool take = k > thr || (k == thr && taken < my_ties);
      taken += k == thr;
      if (take) out[slot++] = t;
    }
    __syncthreads();
  }
}

template <typename T, int HP, int KPT>
void launch_score_v(const DsaParams& p, int sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t keys = (int64_t)KPT * kScoreThreads;
  const int64_t units = rows * (((int64_t)p.T + keys - 1) / keys);
  const int64_t cap = (int64_t)sms * 16;
  const int grid = (int)(units < cap ? units : cap);
  dsa_score_kernel<T, HP, KPT><<<grid, kScoreThreads, 0, stream>>>(p);
}

template <typename T>
cudaError_t launch_score_t(const DsaParams& p, int sms, cudaStream_t stream) {
  if (p.H <= 16) launch_score_v<T, 16, 2>(p, sms, stream);
  else if (p.H <= 32) launch_score_v<T, 32, 2>(p, sms, stream);
  else launch_score_v<T, 64, 1>(p, sms, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dsa_select(const DsaParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t rows = (int64_t)p.B * p.S;
  if (p.T > 0) {
    if (p.dtype == 0) e = launch_score_t<float>(p, sms, stream);
    else if (p.dtype == 1) e = launch_score_t<__half>(p, sms, stream);
    else e = launch_score_t<__nv_bfloat16>(p, sms, stream);
    if (e != cudaSuccess) return e;
  }
  const int64_t cap = (int64_t)sms * 8;
  const int grid = (int)(rows < cap ? rows : cap);
  dsa_select_kernel<<<grid, kSelectThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gb300_attn
