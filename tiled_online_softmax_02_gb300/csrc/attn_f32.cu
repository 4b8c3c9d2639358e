// attn_f32.cu -- fp32-exact attention forward on CUDA cores (FFMA), for
// callers that need fp32 parity (no tensor cores, no 16-bit staging).
//
// Same method as the tensor-core kernel -- the tiled online softmax of
// "onnx-runtime-ep-cuda 0.1.0-dev.5, src/kernels/flash_attention.rs"
// (`flash_attention_body`) with every operand, score, probability and
// accumulator in fp32, as the parity-first design of "pictor-kernels 0.1.0,
// src/gpu_backend/cuda_imagen_attn_kernels.rs" (module doc "Parity-first
// design") asks.  The pages' scalar kernels give each warp one query row and
// re-read Q per key; here a 256-thread CTA owns 64 query rows and walks the
// keys in tiles of BN, with both products register-tiled:
//   S tile (64 x BN): thread (ty, tx) owns rows ty + 16 i and keys tx + 16 j
//                     (i < 4, j < BN / 16), 16 FFMA per 8 shared-memory
//                     vector loads at BN = 64, 12 per 7 at BN = 48;
//   O tile (64 x D):  thread owns rows ty + 16 i and columns 4 tx + 64 g.
// At head dims 256 and 384, whose CTAs take a whole SM, a grid of 64-row
// tiles smaller than the SM count runs as 32-row CTAs instead (i < 2), twice
// as many.
// Row max / sum reductions run over the 16 lanes that share a row.
// Head dims are padded to DP = 64, 128, 256 or 384 (the page's wider VAE
// variant compiles the same kernel for head dims up to 384, "Kernel
// structure"); columns past D are zero in shared memory and never stored.
// Q, a K tile, a V tile and P must fit in shared memory: BN = 48 keys up to
// DP = 128 (95 KB, so two CTAs share an SM), 64 at DP = 256 (211 KB), 32 at
// DP = 384 (203 KB).
// With one 256-thread CTA per SM nothing else covers a tile's load latency,
// so the loads run under the arithmetic: V of tile t is requested (cp.async,
// global -> shared, no registers) before S of tile t is computed, and K of
// tile t + 1 before the P.V products of tile t; each buffer is rewritten only
// after the barrier that ends its last reads.
#include "device_common.cuh"

namespace gb300_attn {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// RI = query rows per thread: a CTA owns 16 RI rows (64, or 32 where 64-row
// tiles would leave SMs without a CTA).
template <int DP, int RI = 4>
struct F32Config {
  static constexpr int BMr = 16 * RI;             // query rows per CTA
  static constexpr int BN = DP <= 128 ? 48 : DP <= 256 ? 64 : 32;  // keys per tile
  static constexpr int kKeysPerThread = BN / 16;
  static constexpr int kQStride = DP + 4;  // padded rows: conflict-free float4 reads
  static constexpr int kKStride = DP + 4;
  static constexpr int kVStride = DP;
  static constexpr int kPStride = BN + 4;
  static constexpr int kGroups = DP / 64;  // float4 column groups per O row per thread
  static constexpr size_t kSmemFloats =
      (size_t)BMr * kQStride + (size_t)BN * kKStride + (size_t)BN * kVStride + (size_t)BMr * kPStride;
  static constexpr size_t kSmemBytes = kSmemFloats * sizeof(float);
  // Head dims up to 128: 48-key tiles leave room for two CTAs an SM, and the
  // register budget is set to match (128 a thread), so 16 warps cover each
  // other's shared-memory latency (measured 5% faster on DiT than one CTA with
  // 64-key tiles and the full register budget); at 256 and 384 a CTA takes the
  // SM and the compiler's own register choice measured fastest.
  static constexpr int kMinBlocks = DP <= 128 ? 2 : 0;
  static constexpr int kUnrollS = 4;
  static constexpr int kUnrollPV = 2;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Loads rows [row0, row0 + nrows) of a [rows, D] fp32 matrix into shared memory
// with row stride `sstride`, zero-filling rows >= valid_rows and columns >= D.
template <int DP>
__device__ __forceinline__ void load_rows(float* dst, int sstride, const float* src, int64_t row0,
                                          int nrows, int64_t valid_rows, int D, bool vec4) {
  if (vec4) {
    constexpr int kVecPerRow = DP / 4;
    for (int idx = threadIdx.x; idx < nrows * kVecPerRow; idx += kThreads) {
      const int r = idx / kVecPerRow;
      const int c = (idx % kVecPerRow) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row0 + r < valid_rows && c < D)
        v = __ldg(reinterpret_cast<const float4*>(src + (row0 + r) * (int64_t)D + c));
      *reinterpret_cast<float4*>(dst + r * sstride + c) = v;
    }
  } else {
    for (int idx = threadIdx.x; idx < nrows * DP; idx += kThreads) {
      const int r = idx / DP;
      const int c = idx % DP;
      float v = 0.f;
      if (row0 + r < valid_rows && c < D) v = __ldg(src + (row0 + r) * (int64_t)D + c);
      dst[r * sstride + c] = v;
    }
  }
}

// The same rows as load_rows, as 16-byte cp.async copies (rows of whole
// 16-byte chunks: D % 4 == 0 and 16-byte aligned planes), zero-filled outside
// the valid rows and past D; one commit group per call.  Without vec4 the
// rows are loaded synchronously, and the barrier before their first use makes
// them visible all the same.
template <int DP>
__device__ __forceinline__ void load_rows_async(float* dst, int sstride, const float* src, int64_t row0,
                                                int nrows, int64_t valid_rows, int D, bool vec4) {
  if (!vec4) {
    load_rows<DP>(dst, sstride, src, row0, nrows, valid_rows, D, false);
    return;
  }
  constexpr int kVecPerRow = DP / 4;
  for (int idx = threadIdx.x; idx < nrows * kVecPerRow; idx += kThreads) {
    const int r = idx / kVecPerRow;
    const int c = (idx % kVecPerRow) * 4;
    const bool valid = row0 + r < valid_rows && c < D;
    const float* g = valid ? src + (row0 + r) * (int64_t)D + c : src;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + r * sstride + c)), "l"(g),
                 "r"(valid ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void async_rows_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int DP, int RI, bool SOFTCAP, bool MASK>
__global__ void __launch_bounds__(kThreads, F32Config<DP, RI>::kMinBlocks) attn_fwd_f32_kernel(const __grid_constant__ F32Params P) {
  using Cfg = F32Config<DP, RI>;
  constexpr int BM = Cfg::BMr;
  constexpr int BN = Cfg::BN;
  constexpr int KJ = Cfg::kKeysPerThread;
  const CommonParams& p = P.c;
  extern __shared__ __align__(16) float fsm[];
  float* Qs = fsm;
  float* Ks = Qs + BM * Cfg::kQStride;
  float* Vs = Ks + BN * Cfg::kKStride;
  float* Ps = Vs + BN * Cfg::kVStride;

  const int tx = threadIdx.x & 15;
  const int ty = threadIdx.x >> 4;
  const int n_qt = (p.Sq + BM - 1) / BM;
  const int qt = n_qt - 1 - (int)blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / p.group;
  const int64_t q0 = (int64_t)qt * BM;
  const int D = p.D;
  const bool vec4 = (D % 4) == 0;

  const BatchLimits L = batch_limits(p, b);
  const TileRange T = tile_range(p, L, q0, BM, BN);
  int64_t zero_from = L.lsk < (int64_t)p.Sk ? L.lsk : (int64_t)p.Sk;  // garbage slots start here
  if (zero_from < 0) zero_from = 0;

  const float* qplane = P.q + ((int64_t)b * p.Hq + h) * (int64_t)p.Sq * D;
  const float* kplane = P.k + ((int64_t)b * p.Hkv + kvh) * (int64_t)p.kv_capacity * D;
  const float* vplane = P.v + ((int64_t)b * p.Hkv + kvh) * (int64_t)p.kv_capacity * D;
  load_rows<DP>(Qs, Cfg::kQStride, qplane, q0, BM, p.Sq, D, vec4);

  RowLimits R[RI];
  const float* mrow[RI];
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    const int64_t qi = q0 + ty + 16 * i;
    R[i] = row_limits(p, L, qi);
    mrow[i] = nullptr;
    if constexpr (MASK) {
      int64_t plane = 0;
      if (p.mask_planes == p.B) plane = b;
      else if (p.mask_planes == p.B * p.Hq) plane = (int64_t)b * p.Hq + h;
      if (qi < p.Sq) mrow[i] = p.mask + (plane * p.Sq + qi) * (int64_t)p.Sk;
    }
  }

  float m[RI], l[RI];
  float o[RI][Cfg::kGroups][4];
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int g = 0; g < Cfg::kGroups; ++g)
#pragma unroll
      for (int u = 0; u < 4; ++u) o[i][g][u] = 0.f;
  }

  if (T.t_begin < T.t_end)
    load_rows_async<DP>(Ks, Cfg::kKStride, kplane, (int64_t)T.t_begin * BN, BN, zero_from, D, vec4);
  for (int t = T.t_begin; t < T.t_end; ++t) {
    const int64_t key0 = (int64_t)t * BN;
    const bool more = t + 1 < T.t_end;
    async_rows_wait<0>();  // this thread's copies of K(t)
    __syncthreads();       // K(t) (and Q) visible; the previous tile's P.V no longer reads V / P
    load_rows_async<DP>(Vs, Cfg::kVStride, vplane, key0, BN, zero_from, D, vec4);

    // S = Q K^T for this thread's RI x KJ block
    float s[RI][KJ];
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
      for (int j = 0; j < KJ; ++j) s[i][j] = 0.f;
#pragma unroll Cfg::kUnrollS
    for (int d0 = 0; d0 < DP; d0 += 4) {
      float4 qa[RI], kb[KJ];
#pragma unroll
      for (int i = 0; i < RI; ++i)
        qa[i] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * i) * Cfg::kQStride + d0);
#pragma unroll
      for (int j = 0; j < KJ; ++j)
        kb[j] = *reinterpret_cast<const float4*>(Ks + (tx + 16 * j) * Cfg::kKStride + d0);
#pragma unroll
      for (int i = 0; i < RI; ++i)
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
          s[i][j] = fmaf(qa[i].x, kb[j].x, s[i][j]);
          s[i][j] = fmaf(qa[i].y, kb[j].y, s[i][j]);
          s[i][j] = fmaf(qa[i].z, kb[j].z, s[i][j]);
          s[i][j] = fmaf(qa[i].w, kb[j].w, s[i][j]);
        }
    }

    // scores in log2 units; invisible keys -> -inf (a select)
    const bool need_mask = !(key0 >= T.full_lo && key0 + BN <= T.full_hi);
#pragma unroll
    for (int i = 0; i < RI; ++i) {
#pragma unroll
      for (int j = 0; j < KJ; ++j) {
        const int64_t kj = key0 + tx + 16 * j;
        float v;
        if (SOFTCAP || MASK) {
          v = s[i][j] * p.scale;
          if constexpr (SOFTCAP) v = soft_cap(v, p.softcap, p.inv_softcap);
          if constexpr (MASK) {
            if (mrow[i] != nullptr && kj < (int64_t)p.Sk) v += __ldg(mrow[i] + kj);
          }
          v *= kLog2e;
        } else {
          v = s[i][j] * p.scale_log2;
        }
        if (need_mask && !(kj >= R[i].lo && kj < R[i].hi)) v = -INFINITY;
        s[i][j] = v;
      }
    }

    // online softmax update per row (the tile update of the page's kernel)
#pragma unroll
    for (int i = 0; i < RI; ++i) {
      float mt = s[i][0];
#pragma unroll
      for (int j = 1; j < KJ; ++j) mt = fmaxf(mt, s[i][j]);
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m[i], mt);
      const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m[i] == -INFINITY) ? 0.f : fast_exp2(m[i] - m_new);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < KJ; ++j) {
        const float e = fast_exp2(s[i][j] - m_sub);
        s[i][j] = e;
        rs += e;
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l[i] = l[i] * alpha + rs;
      m[i] = m_new;
#pragma unroll
      for (int g = 0; g < Cfg::kGroups; ++g)
#pragma unroll
        for (int u = 0; u < 4; ++u) o[i][g][u] *= alpha;
#pragma unroll
      for (int j = 0; j < KJ; ++j) Ps[(ty + 16 * i) * Cfg::kPStride + tx + 16 * j] = s[i][j];
    }
    __syncthreads();  // P complete; S no longer reads K
    if (more) load_rows_async<DP>(Ks, Cfg::kKStride, kplane, key0 + BN, BN, zero_from, D, vec4);
    if (more) async_rows_wait<1>();  // V(t) landed; K(t + 1) may still be in flight
    else async_rows_wait<0>();
    __syncthreads();  // V(t) visible

    // O += P V
#pragma unroll Cfg::kUnrollPV
    for (int k0 = 0; k0 < BN; k0 += 4) {
      float4 pa[RI];
#pragma unroll
      for (int i = 0; i < RI; ++i)
        pa[i] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * i) * Cfg::kPStride + k0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int g = 0; g < Cfg::kGroups; ++g) {
          const float4 vb = *reinterpret_cast<const float4*>(Vs + (k0 + kk) * Cfg::kVStride + g * 64 + tx * 4);
#pragma unroll
          for (int i = 0; i < RI; ++i) {
            const float pk = kk == 0 ? pa[i].x : kk == 1 ? pa[i].y : kk == 2 ? pa[i].z : pa[i].w;
            o[i][g][0] = fmaf(pk, vb.x, o[i][g][0]);
            o[i][g][1] = fmaf(pk, vb.y, o[i][g][1]);
            o[i][g][2] = fmaf(pk, vb.z, o[i][g][2]);
            o[i][g][3] = fmaf(pk, vb.w, o[i][g][3]);
          }
        }
      }
    }
  }

  // normalise and store
  float* out = reinterpret_cast<float*>(p.out);
#pragma unroll
  for (int i = 0; i < RI; ++i) {
    const int64_t qi = q0 + ty + 16 * i;
    if (qi >= p.Sq) continue;
    const float inv = l[i] > 0.f ? 1.0f / l[i] : 0.f;
    int64_t base;
    if (p.out_layout == 0)
      base = (((int64_t)b * p.Hq + h) * p.Sq + qi) * D;
    else
      base = (((int64_t)b * p.Sq + qi) * p.Hq + h) * D;
#pragma unroll
    for (int g = 0; g < Cfg::kGroups; ++g) {
      const int c = g * 64 + tx * 4;
      if (vec4) {
        if (c < D)
          *reinterpret_cast<float4*>(out + base + c) =
              make_float4(o[i][g][0] * inv, o[i][g][1] * inv, o[i][g][2] * inv, o[i][g][3] * inv);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c + u < D) out[base + c + u] = o[i][g][u] * inv;
      }
    }
  }
}

template <int DP, int RI, bool SOFTCAP, bool MASK>
cudaError_t launch_variant(const F32Params& P, cudaStream_t stream) {
  auto kernel = attn_fwd_f32_kernel<DP, RI, SOFTCAP, MASK>;
  constexpr size_t smem = F32Config<DP, RI>::kSmemBytes;
  constexpr int rows = F32Config<DP, RI>::BMr;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((P.c.Sq + rows - 1) / rows), (unsigned)P.c.Hq, (unsigned)P.c.B);
  kernel<<<grid, kThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

template <int DP, int RI>
cudaError_t launch_dp_ri(const F32Params& P, cudaStream_t stream) {
  const bool sc = P.c.softcap > 0.0f;
  const bool mk = P.c.mask != nullptr && P.c.mask_planes > 0;
  if (sc && mk) return launch_variant<DP, RI, true, true>(P, stream);
  if (sc) return launch_variant<DP, RI, true, false>(P, stream);
  if (mk) return launch_variant<DP, RI, false, true>(P, stream);
  return launch_variant<DP, RI, false, false>(P, stream);
}

// 64-row CTAs, or (wide head dims, whose CTAs take a whole SM) 32-row CTAs
// when 64-row tiles would leave SMs without a CTA.
template <int DP>
cudaError_t launch_dp(const F32Params& P, cudaStream_t stream) {
  if constexpr (DP >= 256) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t tiles64 = (int64_t)((P.c.Sq + 63) / 64) * P.c.Hq * P.c.B;
    if (tiles64 < sms) return launch_dp_ri<DP, 2>(P, stream);
  }
  return launch_dp_ri<DP, 4>(P, stream);
}

}  // namespace

cudaError_t launch_attn_f32(const F32Params& P, cudaStream_t stream) {
  if (P.c.D <= 64) return launch_dp<64>(P, stream);
  if (P.c.D <= 128) return launch_dp<128>(P, stream);
  if (P.c.D <= 256) return launch_dp<256>(P, stream);
  if (P.c.D <= kF32MaxHeadDim) return launch_dp<384>(P, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gb300_attn
