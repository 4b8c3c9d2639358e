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
// kernels keep that exact arithmetic (no fused multiply-add, no reordering),
// so they run on the CUDA cores -- a tensor-core product would round
// differently and move near-tied selections.
//
//   dsa_tile_kernel     the score kernel for rows of whole 64-byte chunks.
//                       CTAs take (row, key block) units from a counter; a
//                       staging warp posts each unit's q (fp32 [d][h] in
//                       shared memory, one broadcast 128-bit load feeding
//                       two head pairs), head weights and bias into one of
//                       two slots, and four compute warps each stream their
//                       own keys of K through a private two-stage TMA ring
//                       (64-byte swizzled rows).  Dot products sit in
//                       registers as packed pairs (two heads per
//                       fma.rn.f32x2 with a -0 addend / add.rn.f32x2: each
//                       element still rounded on its own; a pair takes one
//                       issue slot, leaving slots for the loads while the
//                       fp32 pipe, not issue, bounds the loop).  Units whose
//                       keys are all masked are marked and skipped.
//   dsa_score_kernel    the general score kernel (any head dim / alignment):
//                       K chunks transposed into shared memory by the CTA,
//                       scalar rounded multiplies and adds.
//   dsa_select_cluster  selection with the row's slice resident in shared
//                       memory: a cluster of C CTAs splits a row (C > 1 when
//                       rows are few), 8-bit radix select whose per-CTA
//                       histograms (warp-aggregated atomics) are merged over
//                       distributed shared memory, then an ordered tile
//                       compaction.
//   dsa_select_kernel   selection streaming the row from global memory
//                       (rows too long for the cluster's shared memory).
//
// The selection kernels are launched as programmatic dependents of the score
// kernel: their CTAs may become resident while its last units run, and each
// thread waits (griddepcontrol.wait, a hardware dependency on the whole score
// grid and its memory) before it reads anything.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "attn_internal.h"
#include "dsa_internal.h"
#include "device_common.cuh"

namespace gb300_attn {
namespace {

constexpr int kScoreThreads = 128;
constexpr int kDChunk = 32;                  // head-dim columns per shared-memory chunk
constexpr int kSelectThreads = 256;
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kMaxCluster = 8;  // CTAs splitting one row in the selection (16, non-portable, measured slower)
constexpr uint32_t kNotAllowed = 0xFFFFFFFFu;  // score bits of a cell that is not allowed

// Programmatic dependent launch.  The dependents may launch once every CTA
// of this grid has signalled (or exited); they still see this grid's writes
// only after their own wait, which returns once the whole grid is complete.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Packed fp32 pairs with IEEE round-to-nearest on each element and no flush
// of subnormals: the same results as two scalar __fmul_rn / __fadd_rn.  The
// rounded product is formed as fma(a, b, z) with z = (-0, -0) taken from the
// launch parameters: q * k + (-0) is q * k rounded once, for zeros, infinities
// and NaNs too, and an addend the assembler cannot see keeps it from fusing
// the product into the following add (which it does for a packed mul.rn /
// add.rn pair even when contraction is switched off).
__device__ __forceinline__ uint64_t mul_rn2(uint64_t a, uint64_t b, uint64_t z) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(z));
  return d;
}
__device__ __forceinline__ uint64_t add_rn2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ uint64_t pack2u(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Final score bits of a cell: the head sum plus the bias, NaN made the
// positive quiet NaN; a cell that is not allowed gets the mark.
__device__ __forceinline__ uint32_t score_bits(float wsum, float bias, bool ok) {
  const float s = __fadd_rn(wsum, bias);
  return ok ? (isnan(s) ? 0x7FC00000u : __float_as_uint(s)) : kNotAllowed;
}

// -------------------------------------------------------------- general scores
// Unit u = (row, key block of KPT * 128 keys); thread tid takes keys
// t0 + tid + 128 j, j < KPT.  HP = heads rounded up (16, 32 or 64); the
// per-thread accumulators are KPT x HP.
template <typename T, int HP, int KPT>
__global__ void __launch_bounds__(kScoreThreads) dsa_score_kernel(const __grid_constant__ DsaParams p) {
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
    const int64_t row = u % rows;  // row-fastest: a grid stride sees every key block
    const int64_t t0 = (u / rows) * kKeys;
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
      if (t < p.T) out_bits[t] = score_bits(wsum[j], bias_v[j], ok[j]);
    }
    __syncthreads();  // w_s is rewritten by the next unit
  }
}

// -------------------------------------------------------------- tile scores
constexpr int kTileWarps = 4;                          // compute warps
constexpr int kTileThreads = (kTileWarps + 1) * 32;    // + the staging warp
constexpr int kBoxRows = 64;                           // key rows per TMA box
constexpr int kRowBytes = 64;                          // one swizzled shared-memory row of K
constexpr int kGroupHeads = 16;                        // heads per pass over K
constexpr int kMaxQFloats = 8192;                      // q of a row in shared memory: D * heads (padded)
// KPT keys per lane: 4 for throughput (per dim a lane loads 16 broadcast q
// values for 4 keys, so shared-memory delivery stays under the fp32 pipe),
// 2 when rows are few and smaller units spread better over the SMs.
template <int KPT>
struct Tile {
  static constexpr int kWarpKeys = 32 * KPT;                // keys of one compute warp in a unit
  static constexpr int kKeys = kTileWarps * kWarpKeys;      // keys per unit
  static constexpr int kStageBytes = kWarpKeys * kRowBytes; // one stage of one warp's ring
  static constexpr int kBoxes = kWarpKeys / kBoxRows;
  // K ring depth of each compute warp: with 2 keys a lane a chunk's compute
  // is short against an HBM round trip, and the smaller stages leave room
  // for a third at two CTAs per SM
  static constexpr int kStages = KPT == 2 ? 3 : 2;
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}


// Element e of a 16-byte group of K as fp32.
template <typename T>
__device__ __forceinline__ float group_elem(const uint4& g, int e);
template <>
__device__ __forceinline__ float group_elem<float>(const uint4& g, int e) {
  const uint32_t w = e == 0 ? g.x : e == 1 ? g.y : e == 2 ? g.z : g.w;
  return __uint_as_float(w);
}
template <>
__device__ __forceinline__ float group_elem<__nv_bfloat16>(const uint4& g, int e) {
  const int i = e >> 1;
  const uint32_t w = i == 0 ? g.x : i == 1 ? g.y : i == 2 ? g.z : g.w;
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}
template <>
__device__ __forceinline__ float group_elem<__half>(const uint4& g, int e) {
  const int i = e >> 1;
  const uint32_t w = i == 0 ? g.x : i == 1 ? g.y : i == 2 ? g.z : g.w;
  return __half2float(__ushort_as_half((unsigned short)((e & 1) ? (w >> 16) : (w & 0xFFFFu))));
}

// One chunk of 32 bytes of dims for this lane's KPT keys and one group of
// 16 heads: acc[j][hp] holds heads (2 hp, 2 hp + 1) of the group for key
// r0 + 32 j.  q_c is the shared-memory address of the chunk's first dim and
// the group's first head in q_s ([d][hs], row stride hs); each accumulator
// takes its dims in ascending order.
template <typename T, int KPT>
__device__ __forceinline__ void tile_chunk(uint64_t (&acc)[KPT][kGroupHeads / 2], uint32_t kst, uint32_t q_c,
                                           int hs, int r0, uint64_t z) {
  constexpr int kGroups = kRowBytes / 16;
  constexpr int kVec = 16 / (int)sizeof(T);
#pragma unroll 1
  for (int g = 0; g < kGroups; ++g) {
    uint4 raw[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const uint32_t off = (uint32_t)(r0 + 32 * j) * kRowBytes + (uint32_t)g * 16u;
      raw[j] = lds128(kst + (off ^ ((off >> 3) & 0x30u)));  // 64-byte swizzle
    }
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      uint64_t kd[KPT];
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const float kv = group_elem<T>(raw[j], e);
        kd[j] = pack2(kv, kv);
      }
      const uint32_t qd = q_c + (uint32_t)((g * kVec + e) * hs) * 4u;
#pragma unroll
      for (int hq = 0; hq < kGroupHeads / 4; ++hq) {
        const uint4 qv = lds128(qd + 16u * hq);  // broadcast: every lane the same heads
        const uint64_t q01 = pack2u(qv.x, qv.y), q23 = pack2u(qv.z, qv.w);
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
          acc[j][2 * hq] = add_rn2(acc[j][2 * hq], mul_rn2(q01, kd[j], z));
          acc[j][2 * hq + 1] = add_rn2(acc[j][2 * hq + 1], mul_rn2(q23, kd[j], z));
        }
      }
    }
  }
}

// q of one row as fp32 [d][h] over hs (padded) heads, zeros past H, and the
// head weights times weights_scale, staged by one warp.
template <typename T>
__device__ __forceinline__ void stage_q_warp(const DsaParams& p, int64_t row, int hs, float* q_s, float* w_s,
                                             int lane) {
  constexpr int kVec = 16 / (int)sizeof(T);
  const T* qrow = static_cast<const T*>(p.query) + row * (int64_t)p.H * p.D;
  // lanes over heads (hs is a multiple of 16: whole half-warps), dims in
  // 16-byte groups
  const int gstep = hs >= 32 ? 1 : 2;  // hs == 16: two dim groups a pass
  const int h0 = hs >= 32 ? lane : lane & 15;
  const int g0 = hs >= 32 ? 0 : lane >> 4;
  for (int hb = 0; hb < hs; hb += 32) {
    const int h = hb + h0;
    if (h >= hs) break;
    const T* src = qrow + (int64_t)h * p.D;
#pragma unroll 4
    for (int g = g0; g < p.D / kVec; g += gstep) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (h < p.H) raw = __ldg(reinterpret_cast<const uint4*>(src + g * kVec));
      float* dst = q_s + g * kVec * hs + h;
#pragma unroll
      for (int e = 0; e < kVec; ++e) dst[e * hs] = group_elem<T>(raw, e);
    }
  }
  for (int h = lane; h < hs; h += 32)
    w_s[h] = h < p.H ? __fmul_rn(to_f32(static_cast<const T*>(p.weights)[row * p.H + h]), p.weights_scale) : 0.0f;
}

// How a unit is split over the four compute warps.  G groups of 16 heads;
// Gs warps share one key block (each takes G / Gs groups) and a unit holds
// 4 / Gs key blocks.  With 2 keys a lane (small problems) and G = 2 or 4,
// the heads are split over warps so a unit holds fewer keys and the units
// spread over more SMs; otherwise every warp takes all groups (Gs = 1).
struct TileShape {
  int G, Gs, KB, gpw, unit_keys, term_floats;
};
__host__ __device__ inline TileShape tile_shape(int H, int kpt) {
  TileShape t;
  t.G = (H + kGroupHeads - 1) / kGroupHeads;
  t.Gs = (kpt == 2 && (t.G == 2 || t.G == 4)) ? t.G : 1;
  t.KB = kTileWarps / t.Gs;
  t.gpw = t.G / t.Gs;
  t.unit_keys = t.KB * 32 * kpt;
  // per slot: the terms the other warps of a key block hand to its first
  t.term_floats = t.KB * (t.Gs - 1) * t.gpw * kGroupHeads * 32 * kpt;
  return t;
}

// Shared-memory plan of the tile kernel: the compute warps' K rings, then
// two unit slots (q [D][hs], head weights [hs], the unit's bias [keys],
// handed-over terms), the slots' unit indices and the mbarriers.
template <int KPT>
struct TileSmem {
  static constexpr int kSlots = 2;
  static constexpr int kBars = kTileWarps * Tile<KPT>::kStages + 2 * kSlots + kSlots * kTileWarps;
  __host__ __device__ static size_t slot_floats(int D, int hs, int terms) {
    return (size_t)D * hs + hs + Tile<KPT>::kKeys + terms;
  }
  __host__ __device__ static size_t bytes(int D, int hs, int terms) {
    return 1024 + (size_t)kTileWarps * Tile<KPT>::kStages * Tile<KPT>::kStageBytes + kSlots * slot_floats(D, hs, terms) * 4 +
           kSlots * 8 + kBars * 8;
  }
};

// The staging warp's look at unit v of `ukeys` keys: whether a key is
// allowed, with this lane's bias values (keys t0 + lane + 32 i) kept for the
// unit's slot.
template <int KPT>
__device__ __forceinline__ bool unit_bias(const DsaParams& p, int64_t rows, int64_t v, int ukeys, int lane,
                                          float (&bv)[Tile<KPT>::kKeys / 32]) {
  const int64_t row = v % rows, t0 = (v / rows) * ukeys;
  const float* brow = p.bias + row * (int64_t)p.T;
  bool any = false;
#pragma unroll
  for (int i = 0; i < Tile<KPT>::kKeys / 32; ++i) {
    const int64_t t = t0 + lane + 32 * i;
    bv[i] = (32 * i < ukeys && t < p.T) ? brow[t] : -INFINITY;
    any = any || bv[i] > -1e30f;
  }
  return __any_sync(0xffffffffu, any);
}

// Unit u = (row, unit_keys keys), rows fastest (CTAs working at the same
// time then share key blocks in L2); CTAs take units from a counter in the
// workspace, zeroed before the launch.  Warp 4 looks at each unit's bias
// first: a unit without an allowed key gets the "not allowed" mark from it
// and nothing else; every other unit it stages into a slot (q, head weights,
// bias) ahead of the compute warps.  Warps 0..3 take the posted units in
// order.  Compute warp w works on key block (w / Gs + n) mod KB of the n-th
// unit (lane: keys r0 + 32 j), so masked blocks fall on every warp alike,
// and on head groups [(w % Gs) gpw, + gpw).  Each streams its block's K
// through its own TMA ring -- every chunk of dims once per group -- so no
// warp waits for another's stage.  The first warp of a key block sums the
// heads in order: its own groups, then the relu-weighted terms the other
// warps of the block left in the slot.  A warp whose keys are all masked
// loads and computes nothing.
template <typename T, int KPT>
__global__ void __launch_bounds__(kTileThreads, 2) dsa_tile_kernel(const __grid_constant__ DsaParams p) {
  constexpr int kDims = kRowBytes / (int)sizeof(T);  // dims per chunk
  constexpr int kTileKeys = Tile<KPT>::kKeys;
  constexpr int kWarpKeys = Tile<KPT>::kWarpKeys;
  constexpr int kStageBytes = Tile<KPT>::kStageBytes;
  constexpr int kTileStages = Tile<KPT>::kStages;
  constexpr int kSlots = TileSmem<KPT>::kSlots;
  extern __shared__ uint8_t smem_raw[];
  const TileShape sh = tile_shape(p.H, KPT);
  const int hs = sh.G * kGroupHeads;  // heads padded to whole groups
  const int slot_floats = (int)TileSmem<KPT>::slot_floats(p.D, hs, sh.term_floats);
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;  // stages on the swizzle period
  uint8_t* gbase = smem_raw + (sbase - raw_addr);
  float* slots = reinterpret_cast<float*>(gbase + kTileWarps * kTileStages * kStageBytes);
  int64_t* unit_s = reinterpret_cast<int64_t*>(slots + kSlots * slot_floats);
  uint64_t* bars = reinterpret_cast<uint64_t*>(unit_s + kSlots);
  const uint32_t full0 = smem_u32(bars);  // [warp][stage]
  const uint32_t ufull0 = full0 + 8u * kTileWarps * kTileStages, uempty0 = ufull0 + 8u * kSlots;
  const uint32_t tfull0 = uempty0 + 8u * kSlots;  // [slot][key block]: the other warps' terms
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();  // the selection may take SMs this grid leaves idle
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTileWarps * kTileStages; ++i) mbar_init(full0 + 8u * i, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(ufull0 + 8u * s, 1);
      mbar_init(uempty0 + 8u * s, kTileWarps);
      for (int k = 0; k < kTileWarps; ++k) mbar_init(tfull0 + 8u * (s * kTileWarps + k), sh.Gs > 1 ? sh.Gs - 1 : 1);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t kblocks = ((int64_t)p.T + sh.unit_keys - 1) / sh.unit_keys;
  const int64_t units = rows * kblocks;
  const int nchunks = p.D / kDims;

  if (warp == kTileWarps) {  // ---------------- staging warp
    int slot = 0;
    uint32_t uphase[kSlots] = {};
    float bv[kTileKeys / 32];
    // the next unit this CTA takes from the shared counter (units in
    // increasing order over all CTAs, so an SM that finishes early takes
    // more) that has an allowed key; units passed over get the mark; bv then
    // holds its bias
    // (a CTA's first unit is its own index: the grid is never larger than
    // the unit count, and the counter hands out units from gridDim.x on)
    bool first = true;
    auto next_active = [&]() -> int64_t {
      for (;;) {
        unsigned long long w = 0;
        if (lane == 0 && !first) w = atomicAdd(p.unit_counter, 1ull);
        const int64_t v = first ? (int64_t)blockIdx.x : (int64_t)gridDim.x + (int64_t)__shfl_sync(0xffffffffu, w, 0);
        first = false;
        if (v >= units) return units;
        if (unit_bias<KPT>(p, rows, v, sh.unit_keys, lane, bv)) return v;
        const int64_t row = v % rows, t0 = (v / rows) * sh.unit_keys;
        uint32_t* ob = reinterpret_cast<uint32_t*>(p.scores) + row * (int64_t)p.T;
#pragma unroll
        for (int i = 0; i < kTileKeys / 32; ++i) {
          const int64_t t = t0 + lane + 32 * i;
          if (32 * i < sh.unit_keys && t < p.T) ob[t] = kNotAllowed;
        }
      }
    };
    for (;;) {
      const int64_t v = next_active();
      // unit v (v == units: the end mark) into the next slot
      bool w = true;
      if (lane == 0) w = mbar_wait(uempty0 + 8u * slot, uphase[slot] ^ 1u, p.timeout_ns, p.status);
      if (!__shfl_sync(0xffffffffu, w, 0)) return;  // timed out (recorded)
      float* sl = slots + slot * slot_floats;
      if (v < units) {
        stage_q_warp<T>(p, v % rows, hs, sl, sl + p.D * hs, lane);
        float* bs = sl + p.D * hs + hs;
#pragma unroll
        for (int i = 0; i < kTileKeys / 32; ++i)
          if (32 * i < sh.unit_keys) bs[lane + 32 * i] = bv[i];
      }
      if (lane == 0) unit_s[slot] = v < units ? v : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(ufull0 + 8u * slot);  // release: the slot's contents
      uphase[slot] ^= 1u;
      slot ^= 1;
      if (v >= units) return;
    }
  }

  // ---------------- compute warps
  const uint32_t my_full = full0 + 8u * warp * kTileStages;
  const uint32_t my_ring = sbase + (uint32_t)warp * kTileStages * kStageBytes;
  const int kb0 = warp / sh.Gs, gw = warp - kb0 * sh.Gs;  // key block share and group share
  const int g_first = gw * sh.gpw;
  const int per_unit = sh.gpw * nchunks;
  const int term_block = (sh.Gs - 1) * sh.gpw * kGroupHeads * kWarpKeys;  // floats per key block
  uint32_t n_issued = 0, n_used = 0;  // chunks through this warp's ring
  int slot = 0;
  uint32_t uphase[kSlots] = {};
  for (uint32_t seq = 0;; ++seq) {
    if (!mbar_wait_warp(ufull0 + 8u * slot, uphase[slot], p.timeout_ns, p.status)) return;
    const int64_t u = unit_s[slot];
    if (u < 0) return;  // the end mark (every chunk issued has been waited on)
    const float* q_s = slots + slot * slot_floats;
    const float* w_s = q_s + p.D * hs;
    const float* b_s = w_s + hs;
    const int kb = (int)((kb0 + seq) % sh.KB);  // this warp's key block in the unit
    float* terms = const_cast<float*>(b_s) + kTileKeys + kb * term_block;
    const int rw = kb * kWarpKeys;
    const int64_t row = u % rows;
    const int64_t t0 = (u / rows) * sh.unit_keys + rw;
    bool mine = false;
#pragma unroll
    for (int j = 0; j < KPT; ++j) mine = mine || b_s[rw + lane + 32 * j] > -1e30f;
    const bool warp_any = __any_sync(0xffffffffu, mine);
    float wsum[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) wsum[j] = 0.0f;
    if (warp_any) {
      const int64_t b = row / p.S;
      // chunk `it` of this warp's groups ((group, chunk of dims) order) into the ring
      auto issue = [&](int it) {
        const uint32_t st = n_issued % kTileStages;
        if (lane == 0) {
          fence_proxy_async_smem();  // this warp's reads of the stage come first
          mbar_arrive_expect_tx(my_full + 8u * st, kStageBytes);
#pragma unroll
          for (int x = 0; x < Tile<KPT>::kBoxes; ++x)
            tma_load_3d(my_ring + st * kStageBytes + (uint32_t)x * kBoxRows * kRowBytes, &p.tmap_key,
                        my_full + 8u * st, (it % nchunks) * kDims, (int)(t0 + x * kBoxRows), (int)b);
        }
        ++n_issued;
      };
      const int head = per_unit < kTileStages ? per_unit : kTileStages;
      for (int it = 0; it < head; ++it) issue(it);
      uint64_t acc[KPT][kGroupHeads / 2];
      for (int it = 0; it < per_unit; ++it) {
        const int gl = it / nchunks, c = it - gl * nchunks;
        const int grp = g_first + gl;
        if (c == 0) {
#pragma unroll
          for (int j = 0; j < KPT; ++j)
#pragma unroll
            for (int h = 0; h < kGroupHeads / 2; ++h) acc[j][h] = 0ull;
        }
        const uint32_t st = n_used % kTileStages;
        if (!mbar_wait_warp(my_full + 8u * st, (n_used / kTileStages) & 1u, p.timeout_ns, p.status)) {
          // timed out (recorded): let the other copies in flight land first
          if (lane == 0)
            for (uint32_t o = n_used + 1; o < n_issued; ++o)
              mbar_wait(my_full + 8u * (o % kTileStages), (o / kTileStages) & 1u, p.timeout_ns, p.status);
          return;
        }
        ++n_used;
        const uint32_t q_c = smem_u32(q_s + c * kDims * hs + grp * kGroupHeads);
        tile_chunk<T, KPT>(acc, my_ring + st * kStageBytes, q_c, hs, lane, p.neg_zero2);
        __syncwarp();
        if (it + kTileStages < per_unit) issue(it + kTileStages);
        if (c == nchunks - 1) {
          // this group's heads, heads ascending: into the head sum (the
          // block's first warp) or handed over as terms (the others)
          const float* wg = w_s + grp * kGroupHeads;
          float* tg = terms + ((gw - 1) * sh.gpw + gl) * kGroupHeads * kWarpKeys;
#pragma unroll
          for (int hp = 0; hp < kGroupHeads / 2; ++hp) {
            const float w0 = wg[2 * hp], w1 = wg[2 * hp + 1];
#pragma unroll
            for (int j = 0; j < KPT; ++j) {
              float a0, a1;
              unpack2(acc[j][hp], a0, a1);
              float s0 = __fmul_rn(p.scale, a0);
              s0 = s0 > 0.0f ? s0 : 0.0f;  // ReLU (a NaN dot gives 0)
              float s1 = __fmul_rn(p.scale, a1);
              s1 = s1 > 0.0f ? s1 : 0.0f;
              const float e0 = __fmul_rn(s0, w0), e1 = __fmul_rn(s1, w1);
              if (gw == 0) {
                wsum[j] = __fadd_rn(wsum[j], e0);
                wsum[j] = __fadd_rn(wsum[j], e1);
              } else {
                tg[(2 * hp) * kWarpKeys + lane + 32 * j] = e0;
                tg[(2 * hp + 1) * kWarpKeys + lane + 32 * j] = e1;
              }
            }
          }
        }
      }
    }
    if (gw > 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(tfull0 + 8u * (slot * kTileWarps + kb));  // release: the terms (every unit)
    } else {
      if (warp_any && sh.Gs > 1) {
        // the other warps' heads, in order, after this warp's own
        if (!mbar_wait_warp(tfull0 + 8u * (slot * kTileWarps + kb), uphase[slot], p.timeout_ns, p.status)) return;
        const int nt = (sh.Gs - 1) * sh.gpw * kGroupHeads;
        for (int h = 0; h < nt; ++h)
#pragma unroll
          for (int j = 0; j < KPT; ++j) wsum[j] = __fadd_rn(wsum[j], terms[h * kWarpKeys + lane + 32 * j]);
      }
      uint32_t* out_bits = reinterpret_cast<uint32_t*>(p.scores) + row * (int64_t)p.T;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int64_t t = t0 + lane + 32 * j;
        if (t < p.T) {
          const float bv = b_s[rw + lane + 32 * j];
          out_bits[t] = score_bits(wsum[j], bv, bv > -1e30f);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(uempty0 + 8u * slot);  // this warp is done with the slot
    uphase[slot] ^= 1u;
    slot ^= 1;
  }
}

// -------------------------------------------------------------- selection
// Unsigned key whose order is the f32 total order (negative values reversed
// under the sign bit); the "not allowed" mark maps to 0, below every score
// (scores are never negative NaNs: NaNs were made positive).
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Adds one to bin `bin` of h for every lane with `active`: one shared atomic
// per distinct bin in the warp (scores of a row crowd into few top digits).
// Warp-collective and branch-free (inactive lanes match among themselves on
// a key no bin has), so the updates of several keys can overlap.
__device__ __forceinline__ void hist_add(uint32_t* h, uint32_t bin, bool active) {
  const uint32_t peers = __match_any_sync(0xffffffffu, active ? bin : 0xFFFFFFFFu);
  if (active && __ffs(peers) - 1 == (int)(threadIdx.x & 31)) atomicAdd(&h[bin], (uint32_t)__popc(peers));
}


// Warp 0: the bin of histogram gh (counted from the top) holding the
// rank-th largest element, and the rank within it.
__device__ __forceinline__ void find_digit(const uint32_t* gh, uint32_t rank, uint32_t* digit_s, uint32_t* rank_s) {
  const int lane = threadIdx.x & 31;
  // lane l holds bins 255 - 8l ... 248 - 8l (descending)
  uint32_t c[8], s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = gh[255 - 8 * lane - i];
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
        *digit_s = 255u - 8u * lane - i;
        *rank_s = rank - acc;
      }
      acc += c[i];
    }
  }
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Barrier over every thread of every CTA of the cluster, with release /
// acquire ordering of shared memory (a hardware barrier: all CTAs of a
// cluster are resident together).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared word `a` summed over CTAs r0 .. r0 + 7 of the cluster's csize: the
// eight remote loads go out in one block (ranks past csize read the last CTA
// and are not added), so they cost one latency.
__device__ __forceinline__ uint32_t cluster_sum8(const uint32_t* a, int r0, int csize) {
  uint32_t r[8], v[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) r[c] = (uint32_t)(r0 + c < csize ? r0 + c : csize - 1);
  asm volatile(
      "{\n\t.reg .u32 a<8>;\n\t"
      "mapa.shared::cluster.u32 a0, %8, %9;\n\tmapa.shared::cluster.u32 a1, %8, %10;\n\t"
      "mapa.shared::cluster.u32 a2, %8, %11;\n\tmapa.shared::cluster.u32 a3, %8, %12;\n\t"
      "mapa.shared::cluster.u32 a4, %8, %13;\n\tmapa.shared::cluster.u32 a5, %8, %14;\n\t"
      "mapa.shared::cluster.u32 a6, %8, %15;\n\tmapa.shared::cluster.u32 a7, %8, %16;\n\t"
      "ld.shared::cluster.u32 %0, [a0];\n\tld.shared::cluster.u32 %1, [a1];\n\t"
      "ld.shared::cluster.u32 %2, [a2];\n\tld.shared::cluster.u32 %3, [a3];\n\t"
      "ld.shared::cluster.u32 %4, [a4];\n\tld.shared::cluster.u32 %5, [a5];\n\t"
      "ld.shared::cluster.u32 %6, [a6];\n\tld.shared::cluster.u32 %7, [a7];\n\t}"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
      : "r"(smem_u32(a)), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
  uint32_t sum = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c) sum += r0 + c < csize ? v[c] : 0u;
  return sum;
}

// Words a[0..7] of CTA `cta`'s copy, summed (eight loads in one block).
__device__ __forceinline__ uint32_t peer_sum8(const uint32_t* a, uint32_t cta) {
  uint32_t v[8];
  asm volatile(
      "{\n\t.reg .u32 b;\n\t"
      "mapa.shared::cluster.u32 b, %8, %9;\n\t"
      "ld.shared::cluster.u32 %0, [b];\n\tld.shared::cluster.u32 %1, [b+4];\n\t"
      "ld.shared::cluster.u32 %2, [b+8];\n\tld.shared::cluster.u32 %3, [b+12];\n\t"
      "ld.shared::cluster.u32 %4, [b+16];\n\tld.shared::cluster.u32 %5, [b+20];\n\t"
      "ld.shared::cluster.u32 %6, [b+24];\n\tld.shared::cluster.u32 %7, [b+28];\n\t}"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
      : "r"(smem_u32(a)), "r"(cta)
      : "memory");
  return v[0] + v[1] + v[2] + v[3] + v[4] + v[5] + v[6] + v[7];
}

// A cluster of csize CTAs per row (grid-stride over rows by cluster); CTA c
// holds keys [c * slice, (c + 1) * slice) of the row in shared memory, and
// warp w of it the contiguous segment [w * seg, (w + 1) * seg) of that slice
// for the ordered compaction.  Per row: 7 cluster barriers and no other.
__global__ void __launch_bounds__(kSelectThreads) dsa_select_cluster(const __grid_constant__ DsaParams p, int csize,
                                                                     int slice) {
  extern __shared__ uint32_t keys_s[];  // this CTA's slice as order keys (0: not allowed)
  __shared__ uint32_t hist[3][256];     // per radix pass, three in rotation (peers read them)
  __shared__ uint32_t gh[256];          // the cluster's histogram of a pass (clusters of 2 or more)
  __shared__ __align__(16) uint32_t w_ok[kSelectWarps];  // per-warp counts, read by peers
  // per-warp counts of keys above / at the threshold, packed (above) | (at << 16):
  // a slice holds at most kSliceMaxBytes / 4 < 65536 keys, so the sums of
  // eight warps never carry across the halves
  __shared__ __align__(16) uint32_t w_ge[kSelectWarps];
  static_assert(kSelectWarps == 8, "peer_sum8 reads eight per-warp counts");
  static_assert(kMaxCluster <= 8, "cluster_sum8 sums eight CTAs");
  pdl_wait();  // the score grid is complete and its scores visible
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t T = p.T;
  const int64_t base = (int64_t)crank * slice;
  const int n = (int)(T - base < 0 ? 0 : (T - base < slice ? T - base : slice));
  const int seg = ((n + kSelectWarps - 1) / kSelectWarps + 31) & ~31;
  const int s0 = warp * seg < n ? warp * seg : n;
  const int s1 = s0 + seg < n ? s0 + seg : n;
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t row = cluster_index(); row < rows; row += cluster_count()) {
    const uint32_t* bits = reinterpret_cast<const uint32_t*>(p.scores) + row * T + base;
    int64_t* out = p.out + row * (int64_t)p.top_k;
    uint32_t mine = 0;
    int i0 = 0;
    if ((reinterpret_cast<uintptr_t>(bits) & 15u) == 0) {  // 16-byte loads and stores for whole quads
      const int n4 = n >> 2;
      const uint4* b4 = reinterpret_cast<const uint4*>(bits);
      uint4* k4 = reinterpret_cast<uint4*>(keys_s);
      for (int v = tid; v < n4; v += kSelectThreads) {
        const uint4 x = b4[v];
        const uint4 k = make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
        k4[v] = k;
        mine += (k.x != 0u) + (k.y != 0u) + (k.z != 0u) + (k.w != 0u);
      }
      i0 = n4 << 2;
    }
    for (int i = i0 + tid; i < n; i += kSelectThreads) {
      const uint32_t k = order_key(bits[i]);
      keys_s[i] = k;
      mine += k != 0u;
    }
    mine = __reduce_add_sync(0xffffffffu, mine);
    if (lane == 0) w_ok[warp] = mine;
    hist[0][tid] = 0u;  // the first two passes' histograms (kSelectThreads == 256 bins)
    hist[1][tid] = 0u;
    cluster_sync_all();  // slices, counts and zeroed histograms, cluster-wide
    uint32_t a = 0;
    if (lane < csize) {
      if (csize == 1)
        for (int w = 0; w < kSelectWarps; ++w) a += w_ok[w];
      else
        a = peer_sum8(w_ok, (uint32_t)lane);
    }
    const uint32_t allowed = __reduce_add_sync(0xffffffffu, a);
    const uint32_t keep = allowed < (uint32_t)p.top_k ? allowed : (uint32_t)p.top_k;
    for (int64_t i = keep + (int64_t)crank * kSelectThreads + tid; i < p.top_k; i += (int64_t)csize * kSelectThreads)
      out[i] = -1;
    if (keep > 0) {  // the same in every CTA of the cluster
      // radix select of the keep-th largest key, 8 bits at a time from the
      // top; when every allowed key is kept the threshold is simply 0 (the
      // "not allowed" key), and the passes are skipped
      uint32_t prefix = 0, pmask = 0, rank = keep;
#pragma unroll 1
      for (int pass = 0; pass < (keep < allowed ? 4 : 0); ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t* h = hist[pass % 3];
        // the next pass's buffer, last read by the peers two passes ago
        if (pass == 1 || pass == 2) hist[(pass + 1) % 3][tid] = 0u;
        // four keys a thread per step, loaded first (independent updates)
        for (int i0 = 0; i0 < n; i0 += 4 * kSelectThreads) {
          uint32_t k[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kSelectThreads + tid;
            k[u] = i < n ? keys_s[i] : 0u;
          }
          // cells that are not allowed (key 0) sit below every allowed one
          // and rank <= #allowed, so they never decide a digit
#pragma unroll
          for (int u = 0; u < 4; ++u) hist_add(h, (k[u] >> shift) & 255u, k[u] != 0u && (k[u] & pmask) == prefix);
        }
        cluster_sync_all();  // every CTA's histogram of this pass is complete
        const uint32_t* hc = h;
        if (csize > 1) {
          // the cluster's histogram, one bin a thread (gh is rewritten only
          // after the next pass's cluster barrier, when every warp has read it)
          gh[tid] = cluster_sum8(&h[tid], 0, csize);  // csize <= kMaxCluster == 8
          __syncthreads();
          hc = gh;
        }
        // every warp: bins 255 - 8 lane .. 248 - 8 lane, counted from the top
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = hc[255 - 8 * lane - i];
          sum += c[i];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t excl = incl - sum;
        const int owner = __ffs(__ballot_sync(0xffffffffu, excl < rank && rank <= incl)) - 1;
        uint32_t digit = 0, rin = 0, cnt = 0, acc = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc < rank && rank <= acc + c[i]) {
            digit = 255u - 8u * lane - i;
            rin = rank - acc;
            cnt = c[i];
          }
          acc += c[i];
        }
        digit = __shfl_sync(0xffffffffu, digit, owner);
        rank = __shfl_sync(0xffffffffu, rin, owner);
        cnt = __shfl_sync(0xffffffffu, cnt, owner);
        prefix |= digit << shift;
        pmask |= 255u << shift;
        // the whole bin is kept: its lowest key (lower bits 0) serves as the
        // threshold -- every key of the bin is >= it, those equal to it are
        // all taken as ties -- and the remaining passes are not needed (the
        // same decision in every CTA: they share the cluster's histogram)
        if (rank == cnt) break;
      }
      const uint32_t thr = prefix;  // the keep-th largest key
      uint32_t g = 0, e = 0;
      for (int i = s0 + lane; i < s1; i += 32) {
        const uint32_t k = keys_s[i];
        g += k > thr;
        e += k == thr;
      }
      g = __reduce_add_sync(0xffffffffu, g);
      e = __reduce_add_sync(0xffffffffu, e);
      if (lane == 0) w_ge[warp] = g | (e << 16);
      cluster_sync_all();
      // keys above / at thr in the CTAs before this one (slices in key order),
      // over the cluster, and in this CTA's warps before this one
      uint32_t pge = 0;  // CTA `lane`'s packed counts
      if (lane < csize) {
        if (csize == 1)
          for (int w = 0; w < kSelectWarps; ++w) pge += w_ge[w];
        else
          pge = peer_sum8(w_ge, (uint32_t)lane);
      }
      const uint32_t pg = pge & 0xFFFFu, pe = pge >> 16;
      const uint32_t gt_total = __reduce_add_sync(0xffffffffu, pg);
      uint32_t gt_before = __reduce_add_sync(0xffffffffu, (uint32_t)lane < crank ? pg : 0u);
      uint32_t eq_before = __reduce_add_sync(0xffffffffu, (uint32_t)lane < crank ? pe : 0u);
      for (int w = 0; w < warp; ++w) {
        gt_before += w_ge[w] & 0xFFFFu;
        eq_before += w_ge[w] >> 16;
      }
      // keys equal to thr are taken lowest index first
      const uint32_t ties = keep - gt_total;
      // ordered compaction of this warp's segment, 32 keys a step
      for (int i0 = s0; i0 < s1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t k = i < s1 ? keys_s[i] : 0u;
        const bool kg = k > thr, ke = k == thr;
        const uint32_t bg = __ballot_sync(0xffffffffu, kg), be = __ballot_sync(0xffffffffu, ke);
        const uint32_t eb = eq_before + (uint32_t)__popc(be & lt);  // equal keys before this one
        if (kg || (ke && eb < ties))
          out[gt_before + (uint32_t)__popc(bg & lt) + (eb < ties ? eb : ties)] = base + i;
        gt_before += (uint32_t)__popc(bg);
        eq_before += (uint32_t)__popc(be);
      }
    }
    cluster_sync_all();  // peers are done with this row's counts and histograms
  }
}

// One CTA per row (grid-stride), the row streamed from global memory: rows
// too long for the cluster kernel's shared memory.
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
    uint32_t s = lane < kSelectWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kSelectWarps) warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
  *total = warp_sums[kSelectWarps - 1];
  return before;
}

__global__ void __launch_bounds__(kSelectThreads) dsa_select_kernel(const __grid_constant__ DsaParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_sums[kSelectWarps];
  __shared__ uint32_t digit_s, rank_s;
  pdl_wait();  // the score grid is complete and its scores visible
  const int tid = threadIdx.x;
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t T = p.T;
  const int64_t chunk = (T + kSelectThreads - 1) / kSelectThreads;  // contiguous keys per thread
  const int64_t beg = tid * chunk < T ? tid * chunk : T;
  const int64_t end = beg + chunk < T ? beg + chunk : T;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const uint32_t* bits = reinterpret_cast<const uint32_t*>(p.scores) + row * T;
    int64_t* out = p.out + row * (int64_t)p.top_k;
    uint32_t n_ok = 0;
    for (int64_t t = beg; t < end; ++t) n_ok += bits[t] != kNotAllowed;
    uint32_t allowed;
    block_exclusive_scan(n_ok, warp_sums, &allowed);
    const uint32_t keep = allowed < (uint32_t)p.top_k ? allowed : (uint32_t)p.top_k;
    for (int64_t i = keep + tid; i < p.top_k; i += kSelectThreads) out[i] = -1;
    if (keep == 0) continue;
    uint32_t prefix = 0, pmask = 0, rank = keep;
    for (int shift = 24; shift >= 0; shift -= 8) {
      hist[tid] = 0u;
      __syncthreads();
      for (int64_t m = 0; m < chunk; ++m) {  // the same trip count in every lane
        const int64_t t = beg + m;
        const uint32_t k = t < end ? order_key(bits[t]) : 0u;
        hist_add(hist, (k >> shift) & 255u, k != 0u && (k & pmask) == prefix);
      }
      __syncthreads();
      if (tid < 32) find_digit(hist, rank, &digit_s, &rank_s);
      __syncthreads();
      prefix |= digit_s << shift;
      pmask |= 255u << shift;
      rank = rank_s;
      __syncthreads();
    }
    const uint32_t thr = prefix;
    uint32_t n_gt = 0, n_eq = 0;
    for (int64_t t = beg; t < end; ++t) {
      const uint32_t k = order_key(bits[t]);
      n_gt += k > thr;
      n_eq += k == thr;
    }
    uint32_t total_gt, total_eq;
    block_exclusive_scan(n_gt, warp_sums, &total_gt);
    const uint32_t eq_before = block_exclusive_scan(n_eq, warp_sums, &total_eq);
    const uint32_t ties = keep - total_gt;
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

// -------------------------------------------------------------- launchers

template <typename T, int KPT>
cudaError_t launch_tile(const DsaParams& p, int sms, cudaStream_t stream) {
  const TileShape sh = tile_shape(p.H, KPT);
  const size_t smem = TileSmem<KPT>::bytes(p.D, sh.G * kGroupHeads, sh.term_floats);
  static bool attr_set = false;  // the same value from every caller
  if (!attr_set) {
    // the largest plan: D * hs at its cap, hs = 64, the most terms
    const cudaError_t e = cudaFuncSetAttribute(dsa_tile_kernel<T, KPT>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)TileSmem<KPT>::bytes(kMaxQFloats / 64, 64,
                                                                         tile_shape(64, KPT).term_floats));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t units = rows * (((int64_t)p.T + sh.unit_keys - 1) / sh.unit_keys);
  const int64_t cap = (int64_t)sms * 2;
  const int grid = (int)(units < cap ? units : cap);
  dsa_tile_kernel<T, KPT><<<grid, kTileThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// 4 keys per lane when that still gives every resident CTA four units or
// more, else 2.
template <typename T>
cudaError_t launch_tile_any(const DsaParams& p, int sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.S;
  const int64_t units4 = rows * (((int64_t)p.T + Tile<4>::kKeys - 1) / Tile<4>::kKeys);
  if (units4 >= (int64_t)sms * 2 * 4) return launch_tile<T, 4>(p, sms, stream);
  return launch_tile<T, 2>(p, sms, stream);
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
  if (p.tile_path) return launch_tile_any<T>(p, sms, stream);
  if (p.H <= 16) launch_score_v<T, 16, 2>(p, sms, stream);
  else if (p.H <= 32) launch_score_v<T, 32, 2>(p, sms, stream);
  else launch_score_v<T, 64, 1>(p, sms, stream);
  return cudaGetLastError();
}

constexpr int64_t kSliceMaxBytes = 160 * 1024;  // a CTA's slice of a row in shared memory
static_assert(kSliceMaxBytes / 4 < 65536, "dsa_select_cluster packs per-CTA key counts in 16 bits");

// Cluster size for the resident selection (0: stream from global memory):
// the smallest of 1, 2, 4, ... kMaxCluster that gives every SM a CTA, else
// kMaxCluster, as long as the slice fits.
int select_cluster_size(int64_t rows, int64_t T, int sms, int* slice) {
  for (int c = 1; c <= kMaxCluster; c *= 2) {
    const int64_t L = (T + c - 1) / c;
    if (L * 4 <= kSliceMaxBytes && (rows * c >= sms || c == kMaxCluster)) {
      *slice = (int)L;
      return c;
    }
  }
  return 0;
}

cudaError_t launch_select(const DsaParams& p, int sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.S;
  int slice = 0;
  const int c = select_cluster_size(rows, p.T, sms, &slice);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kSelectThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (p.T > 0) {  // a programmatic dependent of the score kernel just enqueued
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (c == 0) {
    const int64_t cap = (int64_t)sms * 8;
    cfg.gridDim = dim3((unsigned)(rows < cap ? rows : cap), 1, 1);
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)na;
    return cudaLaunchKernelEx(&cfg, dsa_select_kernel, p);
  }
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(dsa_select_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSliceMaxBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t max_clusters = (int64_t)sms * 8 / c;
  const int64_t clusters = rows < max_clusters ? rows : max_clusters;
  cfg.gridDim = dim3((unsigned)(clusters * c), 1, 1);
  cfg.dynamicSmemBytes = (size_t)slice * 4;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)c;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)na;
  return cudaLaunchKernelEx(&cfg, dsa_select_cluster, p, c, slice);
}

}  // namespace

bool dsa_tile_path_ok(int dtype, int H, int D) {
  if (H < 1 || H > 64 || D < 1) return false;
  const int dims = kRowBytes / (dtype == 0 ? 4 : 2);  // dims in one row of K
  const int64_t hs = (H + kGroupHeads - 1) / kGroupHeads * kGroupHeads;
  return D % dims == 0 && (int64_t)D * hs <= kMaxQFloats;
}

// key [B, T, D] as a 3-D TMA map {D, T, B}: a box of one K row of dims by
// 128 keys with the matching swizzle; keys past T read as zero.
int dsa_encode_key_map(CUtensorMap* map, void* encoder, const void* key, int dtype, int B, int T, int D) {
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(encoder);
  const int es = dtype == 0 ? 4 : 2;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)D * es, (cuuint64_t)T * (cuuint64_t)D * es};
  const cuuint32_t box[3] = {(cuuint32_t)(kRowBytes / es), (cuuint32_t)kBoxRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType ty = dtype == 0   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_64B;  // kRowBytes
  const CUresult r = fn(map, ty, 3, const_cast<void*>(key), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : 1;
}

cudaError_t launch_dsa_select(const DsaParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (p.T > 0) {
    if (p.dtype == 0) e = launch_score_t<float>(p, sms, stream);
    else if (p.dtype == 1) e = launch_score_t<__half>(p, sms, stream);
    else e = launch_score_t<__nv_bfloat16>(p, sms, stream);
    if (e != cudaSuccess) return e;
  }
  return launch_select(p, sms, stream);
}

}  // namespace gb300_attn
