// attn_tc.cu -- tensor-core (tcgen05) attention forward for bf16 / f16 inputs
// on GB300 (sm_103a).
//
// The method is the tiled online softmax of "onnx-runtime-ep-cuda
// 0.1.0-dev.5, src/kernels/flash_attention.rs" (module doc and
// `flash_attention_body`): scores of one key tile at a time, a running row
// maximum and denominator, and the output numerator rescaled when the maximum
// moves, so no [B,H,Sq,Sk] score tensor ever exists.  The page's kernel stages
// 8 query rows x 16 keys through shared memory with scalar FMAs (and a wmma
// variant with 16x16 tiles); this kernel is a GB300 design of the same method:
//
//   CTA = 128 query rows of one (b, h).  One tile = 128 keys.
//   warp 4      TMA producer: Q once, then K_j / V_j into a stage ring.
//   warp 5      MMA issuer (one thread): S_j = Q K_j^T into tensor memory
//               (two S buffers, fp32), then O += P_j V_j with P_j read from
//               tensor memory.  Owns the tensor-memory allocation.
//   warps 0-3   softmax: thread r owns query row r (= TMEM lane r).  Reads
//               its S row with tcgen05.ld, applies the structural masks
//               (select to -inf), soft-cap and additive mask, updates the
//               running max / sum in registers, writes P (input dtype) back
//               over its S row, and rescales its O row when the max grew by
//               more than 2^8 (otherwise the old max is kept: the final
//               O / l is exact either way).  Then normalises and stores.
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O [256, 256+D).
// Shared memory: Q tile, kStages x (K tile, V tile), barriers; every tile is
// stored as 64-column (128-byte) blocks in the 128-byte swizzle TMA writes.
//
// Every barrier wait is bounded (see mbar_wait); on a timeout the kernel
// records ATTN_ERR_TIMEOUT in the status word, drains what it issued, frees
// tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"

namespace gb300_attn {
namespace {

constexpr int BM = kTcBlockM;
constexpr int BN = kTcBlockN;
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;  // keep the old max while it is within 2^8
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct TcConfig {
  static constexpr int kSub = D / 64;                   // 128-byte column blocks per row
  static constexpr uint32_t kSubBytes = BM * 128;       // [128 rows][64 cols] of 16-bit
  static constexpr uint32_t kTileBytes = kSub * kSubBytes;
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
  // q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2], pv_done, drain, o_final
  static constexpr int kNumBars = 1 + 3 * kStages + 2 + 2 + 1 + 1 + 1;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffTmemSlot + 16 + 1024;  // + 1024 alignment slack
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int D, bool BF16, bool SOFTCAP, bool MASK>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc_kernel(const __grid_constant__ TcParams P) {
  using Cfg = TcConfig<D>;
  constexpr int S = Cfg::kStages;
  const CommonParams& p = P.c;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + Cfg::kOffQ;
  const uint32_t sK = sbase + Cfg::kOffK;
  const uint32_t sV = sbase + Cfg::kOffV;
  const uint32_t bar0 = sbase + Cfg::kOffBar;
  const uint32_t bar_q = bar0;
  auto bar_k = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_v = [&](int s) { return bar0 + 8u * (1 + S + s); };
  auto bar_empty = [&](int s) { return bar0 + 8u * (1 + 2 * S + s); };
  auto bar_s = [&](int i) { return bar0 + 8u * (1 + 3 * S + i); };
  auto bar_p = [&](int i) { return bar0 + 8u * (1 + 3 * S + 2 + i); };
  const uint32_t bar_pv = bar0 + 8u * (1 + 3 * S + 4);
  const uint32_t bar_drain = bar0 + 8u * (1 + 3 * S + 5);
  // Completes once, after the last P.V.  The epilogue cannot wait on pv_done:
  // by then pv_done may still be two phases short, which a parity wait cannot
  // tell from done.
  const uint32_t bar_o_final = bar0 + 8u * (1 + 3 * S + 6);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (p.Sq + BM - 1) / BM;
  const int qt = n_qt - 1 - (int)blockIdx.x;  // longest causal rows first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / p.group;
  const int64_t q0 = (int64_t)qt * BM;

  const BatchLimits L = batch_limits(p, b);
  const TileRange T = tile_range(p, L, q0, BM, BN);
  const int n_tiles = T.t_end - T.t_begin;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_k(s), 1);
      mbar_init(bar_v(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s(i), 1);
      mbar_init(bar_p(i), 4);  // one arrival per softmax warp
    }
    mbar_init(bar_pv, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_o_final, 1);
    mbar_init_fence();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&P.tmap_q);
    tma_prefetch_desc(&P.tmap_k);
    tma_prefetch_desc(&P.tmap_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0) {
      const int q_plane = b * p.Hq + h;
      const int kv_plane = b * p.Hkv + kvh;
      mbar_arrive_expect_tx(bar_q, Cfg::kTileBytes);
      for (int s = 0; s < Cfg::kSub; ++s)
        tma_load_3d(sQ + s * Cfg::kSubBytes, &P.tmap_q, bar_q, s * 64, (int)q0, q_plane);
      int issued = 0;
      for (int n = 0; n < n_tiles; ++n) {
        const int st = n % S;
        const int key0 = (T.t_begin + n) * BN;
        if (n >= S && !mbar_wait(bar_empty(st), ((n / S) - 1) & 1, p.timeout_ns, p.status)) break;
        mbar_arrive_expect_tx(bar_k(st), Cfg::kTileBytes);
        for (int s = 0; s < Cfg::kSub; ++s)
          tma_load_3d(sK + st * Cfg::kTileBytes + s * Cfg::kSubBytes, &P.tmap_k, bar_k(st), s * 64,
                      key0, kv_plane);
        mbar_arrive_expect_tx(bar_v(st), Cfg::kTileBytes);
        for (int s = 0; s < Cfg::kSub; ++s)
          tma_load_3d(sV + st * Cfg::kTileBytes + s * Cfg::kSubBytes, &P.tmap_v, bar_v(st), s * 64,
                      key0, kv_plane);
        issued = n + 1;
      }
      // Let every copy this thread started land before the CTA can exit.
      for (int n = (issued > S ? issued - S : 0); n < issued; ++n) {
        mbar_wait(bar_k(n % S), (n / S) & 1, p.timeout_ns, p.status);
        mbar_wait(bar_v(n % S), (n / S) & 1, p.timeout_ns, p.status);
      }
      mbar_wait(bar_q, 0, p.timeout_ns, p.status);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (n_tiles > 0) {
      constexpr uint32_t idesc_qk = make_idesc_f16kind(BF16, BM, BN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16kind(BF16, BM, D, true);
      int64_t zero_from = L.lsk < (int64_t)p.Sk ? L.lsk : (int64_t)p.Sk;
      if (zero_from < 0) zero_from = 0;

      // O += P_m V_m for tile m (P_m lives in S buffer m & 1).
      auto issue_pv = [&](int m) -> bool {
        const int st = m % S;
        const int buf = m & 1;
        const int64_t key0 = (int64_t)(T.t_begin + m) * BN;
        if (!mbar_wait_warp(bar_v(st), (m / S) & 1, p.timeout_ns, p.status)) return false;
        if (zero_from < key0 + BN && zero_from < (int64_t)p.kv_capacity) {
          // Cache slots past the valid length may hold NaN / Inf; P is 0 there
          // but 0 * NaN is not, so zero those V rows (whole 128-byte rows, so
          // the swizzle does not matter).
          const int r0 = zero_from > key0 ? (int)(zero_from - key0) : 0;
          const int chunks = (BN - r0) * 8;  // 16-byte chunks per column block
          for (int s = 0; s < Cfg::kSub; ++s) {
            uint8_t* vblk = smem + Cfg::kOffV + st * Cfg::kTileBytes + s * Cfg::kSubBytes;
            for (int c = lane; c < chunks; c += 32)
              *reinterpret_cast<uint4*>(vblk + (size_t)(r0 + (c >> 3)) * 128 + (c & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!mbar_wait_warp(bar_p(buf), (m >> 1) & 1, p.timeout_ns, p.status)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vaddr = sV + st * Cfg::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            // B = V[keys 16kk.., 0..D): MN-major; 8-key groups 1024 B apart,
            // 64-column blocks kSubBytes apart.
            const uint64_t bdesc = make_sdesc_sw128(vaddr + kk * 2048, Cfg::kSubBytes, 1024);
            const uint32_t a_tmem = tmem + kColS0 + buf * 128 + kk * 8;
            mma_ts(tmem + kColO, a_tmem, bdesc, idesc_pv, (m > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar_pv);
          tc_commit(bar_empty(st));
        }
        __syncwarp();
        return true;
      };

      bool ok = mbar_wait_warp(bar_q, 0, p.timeout_ns, p.status);
      for (int n = 0; ok && n < n_tiles; ++n) {
        const int st = n % S;
        const int buf = n & 1;
        if (!mbar_wait_warp(bar_k(st), (n / S) & 1, p.timeout_ns, p.status)) { ok = false; break; }
        // S buffer `buf` holds P_{n-2} until PV_{n-2} has completed.
        if (n >= 2 && !mbar_wait_warp(bar_pv, (n - 2) & 1, p.timeout_ns, p.status)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kaddr = sK + st * Cfg::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * Cfg::kSubBytes + (kk & 3) * 32;
            const uint64_t adesc = make_sdesc_sw128(sQ + off, 16, 1024);
            const uint64_t bdesc = make_sdesc_sw128(kaddr + off, 16, 1024);
            mma_ss(tmem + kColS0 + buf * 128, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          }
          tc_commit(bar_s(buf));
        }
        __syncwarp();
        if (n >= 1 && !issue_pv(n - 1)) { ok = false; break; }
      }
      if (ok && issue_pv(n_tiles - 1) && lane == 0) tc_commit(bar_o_final);
      // Wait for every MMA this warp issued before tensor memory is freed.
      if (lane == 0) tc_commit(bar_drain);
      __syncwarp();
      mbar_wait_warp(bar_drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = warp * 32 + lane;
    const int64_t qi = q0 + row;
    const RowLimits R = row_limits(p, L, qi);
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float* mrow = nullptr;
    if constexpr (MASK) {
      int64_t plane = 0;
      if (p.mask_planes == p.B) plane = b;
      else if (p.mask_planes == p.B * p.Hq) plane = (int64_t)b * p.Hq + h;
      if (qi < p.Sq) mrow = p.mask + (plane * p.Sq + qi) * (int64_t)p.Sk;
    }

    float m_run = -INFINITY;  // running max, log2 units
    float l_run = 0.0f;       // running denominator
    bool ok = true;
    for (int n = 0; n < n_tiles; ++n) {
      const int buf = n & 1;
      const int64_t key0 = (int64_t)(T.t_begin + n) * BN;
      if (!mbar_wait_warp(bar_s(buf), (n >> 1) & 1, p.timeout_ns, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_base + kColS0 + buf * 128;
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
      tmem_wait_ld();
      float x[BN];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(sr[c][i]);

      const bool need_mask = !(key0 >= T.full_lo && key0 + BN <= T.full_hi);
      float m_tile;
      bool scaled;  // x already in log2 units (else raw Q.K, scaled inside the exp)
      if (SOFTCAP || MASK || need_mask) {
        // general path: x_j = ((softcap(scale s_j)) + mask_j) * log2 e, or -inf
        m_tile = -INFINITY;
#pragma unroll
        for (int c4 = 0; c4 < BN; c4 += 4) {
          float mv[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (MASK) {
            const int64_t j0 = key0 + c4;
            if (mrow != nullptr) {
              if (p.mask_vec4 && j0 + 3 < (int64_t)p.Sk) {
                const float4 m4 = __ldg(reinterpret_cast<const float4*>(mrow + j0));
                mv[0] = m4.x; mv[1] = m4.y; mv[2] = m4.z; mv[3] = m4.w;
              } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (j0 + u < (int64_t)p.Sk) mv[u] = __ldg(mrow + j0 + u);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t j = key0 + c4 + u;
            float v = x[c4 + u] * p.scale;
            if constexpr (SOFTCAP) v = soft_cap(v, p.softcap, p.inv_softcap);
            if constexpr (MASK) v += mv[u];
            v *= kLog2e;
            x[c4 + u] = (j >= R.lo && j < R.hi) ? v : -INFINITY;
            m_tile = fmaxf(m_tile, x[c4 + u]);
          }
        }
        scaled = true;
      } else {
        // every key of this tile is visible to every row: the extreme raw
        // score times the (signed) scale is the max of the scaled scores
        float ext = x[0];
        if (p.scale_log2 >= 0.0f) {
#pragma unroll
          for (int i = 1; i < BN; ++i) ext = fmaxf(ext, x[i]);
        } else {
#pragma unroll
          for (int i = 1; i < BN; ++i) ext = fminf(ext, x[i]);
        }
        m_tile = ext * p.scale_log2;
        scaled = false;
      }

      // online update, keeping the old max unless it grew by more than 2^8
      const float m_new = fmaxf(m_run, m_tile);
      float alpha = 1.0f;
      bool rescale = false;
      float m_use = m_run;
      if (m_run == -INFINITY) {
        m_use = m_new;  // first live tile: this row's O is still exactly 0
      } else if (m_new - m_run > kRescaleLog2) {
        m_use = m_new;
        alpha = fast_exp2(m_run - m_new);
        rescale = true;
      }
      const float m_sub = (m_use == -INFINITY) ? 0.0f : m_use;

      uint32_t pr[2][32];
      float sum = 0.0f;
#pragma unroll
      for (int i = 0; i < BN / 2; ++i) {
        float e0, e1;
        if (scaled) {
          e0 = fast_exp2(x[2 * i] - m_sub);
          e1 = fast_exp2(x[2 * i + 1] - m_sub);
        } else {
          e0 = fast_exp2(fmaf(x[2 * i], p.scale_log2, -m_sub));
          e1 = fast_exp2(fmaf(x[2 * i + 1], p.scale_log2, -m_sub));
        }
        sum += e0 + e1;
        pr[i >> 5][i & 31] = pack2<BF16>(e0, e1);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;

      // P (16-bit, 64 columns) over the first half of this S buffer
      tmem_st32(s_addr, pr[0]);
      tmem_st32(s_addr + 32, pr[1]);

      if (__any_sync(0xffffffffu, rescale)) {
        // O holds P_{n-1} V_{n-1} once PV_{n-1} completes (n >= 1 here).
        if (!mbar_wait_warp(bar_pv, (n - 1) & 1, p.timeout_ns, p.status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + kColO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_base + kColO + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(buf));
    }

    // ---------------------------------------------------------- epilogue
    bool have_o = ok && n_tiles > 0;
    if (have_o) {
      have_o = mbar_wait_warp(bar_o_final, 0, p.timeout_ns, p.status);
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
      using T16 = uint16_t;
      T16* out = reinterpret_cast<T16*>(p.out);
      int64_t base;
      if (p.out_layout == 0)
        base = (((int64_t)b * p.Hq + h) * p.Sq + qi) * D;
      else
        base = (((int64_t)b * p.Sq + qi) * p.Hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (have_o) {
          tmem_ld32(tmem + lane_base + kColO + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (qi < p.Sq) {
          uint4* dst = reinterpret_cast<uint4*>(out + base + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16, bool SOFTCAP, bool MASK>
cudaError_t launch_variant(const TcParams& P, cudaStream_t stream) {
  auto kernel = attn_fwd_tc_kernel<D, BF16, SOFTCAP, MASK>;
  constexpr uint32_t smem = TcConfig<D>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((P.c.Sq + BM - 1) / BM), (unsigned)P.c.Hq, (unsigned)P.c.B);
  kernel<<<grid, kThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_d(const TcParams& P, cudaStream_t stream) {
  const bool sc = P.c.softcap > 0.0f;
  const bool mk = P.c.mask != nullptr && P.c.mask_planes > 0;
  if (sc && mk) return launch_variant<D, BF16, true, true>(P, stream);
  if (sc) return launch_variant<D, BF16, true, false>(P, stream);
  if (mk) return launch_variant<D, BF16, false, true>(P, stream);
  return launch_variant<D, BF16, false, false>(P, stream);
}

}  // namespace

cudaError_t launch_attn_tc(const TcParams& P, bool bf16, cudaStream_t stream) {
  if (P.c.D == 64) return bf16 ? launch_d<64, true>(P, stream) : launch_d<64, false>(P, stream);
  return bf16 ? launch_d<128, true>(P, stream) : launch_d<128, false>(P, stream);
}

}  // namespace gb300_attn
