// attn_tc.cu -- tensor-core (tcgen05) attention forward for bf16 / f16 inputs
// on GB300 (sm_103a).
//
// The method is the tiled online softmax of "onnx-runtime-ep-cuda
// 0.1.0-dev.5, src/kernels/flash_attention.rs" (module doc and
// `flash_attention_body`): scores of one key tile at a time, a running row
// maximum and denominator, and the output numerator rescaled when the maximum
// moves, so no [B,H,Sq,Sk] score tensor ever exists.  The page's kernel stages
// 8 query rows x 16 keys through shared memory with scalar FMAs (and a wmma
// variant with 16x16 tiles); this kernel is a GB300 design of the same method.
//
// CTA = two 128-row query tiles (t = 0, 1) of one (b, h); key tiles of 128.
//   warps 0-3   softmax for query tile 0, warps 4-7 for query tile 1: thread
//               r of a warpgroup owns query row r (= TMEM lane r).  Reads its
//               S row with tcgen05.ld, applies the structural masks (select to
//               -inf), soft-cap and additive mask, updates the running max /
//               sum in registers, writes P (input dtype) back over its S row,
//               and rescales its O row when the max grew by more than 2^8
//               (otherwise the old max is kept: the final O / l is exact
//               either way).  Then normalises and stores the row.
//   warp 8      TMA producer: both Q tiles once, then K_j / V_j into a ring.
//   warp 9      MMA issuer (one thread) and owner of tensor memory.  Per key
//               tile j, for t = 0, 1:  O_t += P_t(j-1) V(j-1), then
//               S_t(j) = Q_t K(j)^T.  While warpgroup 0 turns S_0 into P_0,
//               the tensor core works on tile 1, and the other way round.
//               Because S_t(j) is issued after O_t's P.V and a commit covers
//               every earlier MMA of the thread, "S_t(j) ready" also means
//               "O_t up to date", so a rescale never waits.
// Each query tile visits only its own key-tile range (causal / window /
// length limits), so the diagonal and window edges cost no extra MMAs.
//
// Tensor memory (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384),
// O_1 [384,512).  Shared memory: Q_0, Q_1, kStages x (K, V) tiles, barriers;
// every tile is stored as 64-column (128-byte) blocks in the 128-byte swizzle
// TMA writes.
//
// Every barrier wait is bounded (mbar_wait); on a timeout the kernel records
// ATTN_ERR_TIMEOUT in the status word, drains what it issued, frees tensor
// memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"

namespace gb300_attn {
namespace {

constexpr int BM = kTcBlockM;   // rows per query tile
constexpr int BN = kTcBlockN;   // keys per key tile
constexpr int kQTiles = 2;      // query tiles per CTA
constexpr int kThreads = 320;   // 8 softmax warps + producer + MMA
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
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
  static constexpr uint32_t kOffK = kOffQ + kQTiles * kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kTileBytes;
  // q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], p_full[2], o_final[2], drain
  static constexpr int kNumBars = 1 + 3 * kStages + 2 + 2 + 2 + 1;
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

// Maximum / minimum of 128 values as eight independent chains (short
// dependency depth instead of one 127-long chain).
__device__ __forceinline__ float max128(const float (&x)[BN]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = x[k];
#pragma unroll
  for (int i = 8; i < BN; i += 8)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], x[i + k]);
  return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

__device__ __forceinline__ float min128(const float (&x)[BN]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = x[k];
#pragma unroll
  for (int i = 8; i < BN; i += 8)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fminf(m[k], x[i + k]);
  return fminf(fminf(fminf(m[0], m[1]), fminf(m[2], m[3])), fminf(fminf(m[4], m[5]), fminf(m[6], m[7])));
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
  auto bar_s = [&](int t) { return bar0 + 8u * (1 + 3 * S + t); };
  auto bar_p = [&](int t) { return bar0 + 8u * (1 + 3 * S + 2 + t); };
  // completes once, after query tile t's last P.V (the epilogue's wait)
  auto bar_o = [&](int t) { return bar0 + 8u * (1 + 3 * S + 4 + t); };
  const uint32_t bar_drain = bar0 + 8u * (1 + 3 * S + 6);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (p.Sq + kQTiles * BM - 1) / (kQTiles * BM);
  const int qt = n_qt - 1 - (int)blockIdx.x;  // longest causal rows first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / p.group;
  const int64_t q0 = (int64_t)qt * (kQTiles * BM);

  // key-tile range of each query tile, and their union [tb, te)
  const BatchLimits L = batch_limits(p, b);
  TileRange tr[kQTiles];
  int tb = 0, te = 0;
  bool any = false;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    tr[t] = tile_range(p, L, q0 + t * BM, BM, BN);
    if (tr[t].t_end > tr[t].t_begin) {
      tb = any ? min(tb, tr[t].t_begin) : tr[t].t_begin;
      te = any ? max(te, tr[t].t_end) : tr[t].t_end;
      any = true;
    }
  }
  const int N = te - tb;  // key tiles the CTA streams
  auto active = [&](int t, int j) { return j >= tr[t].t_begin && j < tr[t].t_end; };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_k(s), 1);
      mbar_init(bar_v(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(bar_s(t), 1);
      mbar_init(bar_p(t), 4);  // one arrival per softmax warp of the tile
      mbar_init(bar_o(t), 1);
    }
    mbar_init(bar_drain, 1);
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
    if (lane == 0 && N > 0) {
      const int q_plane = b * p.Hq + h;
      const int kv_plane = b * p.Hkv + kvh;
      mbar_arrive_expect_tx(bar_q, kQTiles * Cfg::kTileBytes);
      for (int t = 0; t < kQTiles; ++t)
        for (int s = 0; s < Cfg::kSub; ++s)
          tma_load_3d(sQ + t * Cfg::kTileBytes + s * Cfg::kSubBytes, &P.tmap_q, bar_q, s * 64,
                      (int)(q0 + t * BM), q_plane);
      int issued = 0;
      for (int n = 0; n < N; ++n) {
        const int st = n % S;
        const int key0 = (tb + n) * BN;
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
    if (N > 0) {
      constexpr uint32_t idesc_qk = make_idesc_f16kind(BF16, BM, BN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16kind(BF16, BM, D, true);
      int64_t zero_from = L.lsk < (int64_t)p.Sk ? L.lsk : (int64_t)p.Sk;
      if (zero_from < 0) zero_from = 0;
      int pc[kQTiles] = {0, 0};  // P.V products issued per query tile

      bool ok = mbar_wait_warp(bar_q, 0, p.timeout_ns, p.status);
      // iteration n: P.V of key tile tb+n-1 (if n >= 1), S of key tile tb+n (if n < N)
      for (int n = 0; ok && n <= N; ++n) {
        const int j = tb + n;
        bool k_ready = false;  // K(j) is waited for only before its first use
        if (n >= 1) {
          const int ps = (n - 1) % S;
          if (!mbar_wait_warp(bar_v(ps), ((n - 1) / S) & 1, p.timeout_ns, p.status)) {
            ok = false;
            break;
          }
          const int64_t key0 = (int64_t)(j - 1) * BN;
          if (zero_from < key0 + BN && zero_from < (int64_t)p.kv_capacity) {
            // Cache slots past the valid length may hold NaN / Inf; P is 0
            // there but 0 * NaN is not, so zero those V rows (whole 128-byte
            // rows, so the swizzle does not matter).
            const int r0 = zero_from > key0 ? (int)(zero_from - key0) : 0;
            const int chunks = (BN - r0) * 8;
            for (int s = 0; s < Cfg::kSub; ++s) {
              uint8_t* vblk = smem + Cfg::kOffV + ps * Cfg::kTileBytes + s * Cfg::kSubBytes;
              for (int c = lane; c < chunks; c += 32)
                *reinterpret_cast<uint4*>(vblk + (size_t)(r0 + (c >> 3)) * 128 + (c & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < kQTiles; ++t) {
          const bool do_pv = n >= 1 && active(t, j - 1);
          const bool do_s = n < N && active(t, j);
          if (do_pv) {
            if (!mbar_wait_warp(bar_p(t), pc[t] & 1, p.timeout_ns, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (lane == 0) {
              const uint32_t vaddr = sV + ((n - 1) % S) * Cfg::kTileBytes;
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk) {
                // B = V[keys 16kk.., 0..D): MN-major; 8-key groups 1024 B
                // apart, 64-column blocks kSubBytes apart.
                const uint64_t bdesc = make_sdesc_sw128(vaddr + kk * 2048, Cfg::kSubBytes, 1024);
                mma_ts(tmem + kColO + t * 128, tmem + t * 128 + kk * 8, bdesc, idesc_pv,
                       (pc[t] > 0 || kk > 0) ? 1u : 0u);
              }
              if (!do_s) tc_commit(bar_o(t));  // query tile t has seen its last key tile
            }
            ++pc[t];
          }
          if (do_s && !k_ready) {
            if (!mbar_wait_warp(bar_k(n % S), (n / S) & 1, p.timeout_ns, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            k_ready = true;
          }
          if (do_s && lane == 0) {
            const uint32_t kaddr = sK + (n % S) * Cfg::kTileBytes;
            const uint32_t qaddr = sQ + t * Cfg::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * Cfg::kSubBytes + (kk & 3) * 32;
              const uint64_t adesc = make_sdesc_sw128(qaddr + off, 16, 1024);
              const uint64_t bdesc = make_sdesc_sw128(kaddr + off, 16, 1024);
              mma_ss(tmem + t * 128, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar_s(t));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (n >= 1 && lane == 0) tc_commit(bar_empty((n - 1) % S));
        __syncwarp();
      }
      // Wait for every MMA this warp issued before tensor memory is freed.
      if (lane == 0) tc_commit(bar_drain);
      __syncwarp();
      mbar_wait_warp(bar_drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;  // query tile of this warpgroup
    const int wq = warp & 3;  // TMEM lane quarter
    const int row = wq * 32 + lane;
    const int64_t qi = q0 + t * BM + row;
    const TileRange T = t == 0 ? tr[0] : tr[1];  // a select keeps tr[] in registers
    const int nt = T.t_end - T.t_begin;
    const RowLimits R = row_limits(p, L, qi);
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + t * 128;
    const uint32_t o_addr = tmem + lane_base + kColO + t * 128;
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
    for (int c = 0; c < nt; ++c) {
      const int64_t key0 = (int64_t)(T.t_begin + c) * BN;
      if (!mbar_wait_warp(bar_s(t), c & 1, p.timeout_ns, p.status)) { ok = false; break; }
      tc_fence_after();
      float x[BN];
      {
        uint32_t sr[4][32];
#pragma unroll
        for (int k = 0; k < 4; ++k) tmem_ld32(s_addr + k * 32, sr[k]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 32; ++i) x[k * 32 + i] = __uint_as_float(sr[k][i]);
      }

      const bool need_mask = !(key0 >= T.full_lo && key0 + BN <= T.full_hi);
      float m_tile;
      bool scaled;  // x already in log2 units (else raw Q.K, scaled inside the exp)
      if (SOFTCAP || MASK || need_mask) {
        // general path: x_j = ((softcap(scale s_j)) + mask_j) * log2 e, or -inf
        int64_t lo = R.lo - key0, hi = R.hi - key0;
        lo = lo < 0 ? 0 : (lo > BN ? BN : lo);
        hi = hi < 0 ? 0 : (hi > BN ? BN : hi);
        const int lo_rel = (int)lo;
        const uint32_t span = hi > lo ? (uint32_t)(hi - lo) : 0u;
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
            float v;
            if constexpr (SOFTCAP || MASK) {
              v = x[c4 + u] * p.scale;
              if constexpr (SOFTCAP) v = soft_cap(v, p.softcap, p.inv_softcap);
              if constexpr (MASK) v += mv[u];
              v *= kLog2e;
            } else {
              v = x[c4 + u] * p.scale_log2;
            }
            x[c4 + u] = ((uint32_t)(c4 + u - lo_rel) < span) ? v : -INFINITY;
          }
        }
        m_tile = max128(x);
        scaled = true;
      } else {
        // every key of this tile is visible to every row: the extreme raw
        // score times the (signed) scale is the max of the scaled scores
        m_tile = (p.scale_log2 >= 0.0f ? max128(x) : min128(x)) * p.scale_log2;
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
      const float xmul = scaled ? 1.0f : p.scale_log2;  // brings x to log2 units

      // P = 2^(x - m) in four 32-column chunks, each packed into 16 columns
      // of 16-bit pairs over the first half of this S row
      float sum = 0.0f;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = x[ch * 32 + 2 * i], a1 = x[ch * 32 + 2 * i + 1];
          const float e0 = fast_exp2(fmaf(a0, xmul, -m_sub));
          const float e1 = fast_exp2(fmaf(a1, xmul, -m_sub));
          sum += e0 + e1;
          pk[i] = pack2<BF16>(e0, e1);
        }
        tmem_st16(s_addr + ch * 16, pk);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;

      if (__any_sync(0xffffffffu, rescale)) {
        // O_t already holds every earlier P.V (see the header)
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          uint32_t o[32];
          tmem_ld32(o_addr + k * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(o_addr + k * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(t));
    }

    // ---------------------------------------------------------- epilogue
    bool have_o = ok && nt > 0;
    if (have_o) {
      have_o = mbar_wait_warp(bar_o(t), 0, p.timeout_ns, p.status);
      tc_fence_after();
    }
    if (ok) {
      const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
      uint16_t* out = reinterpret_cast<uint16_t*>(p.out);
      int64_t base;
      if (p.out_layout == 0)
        base = (((int64_t)b * p.Hq + h) * p.Sq + qi) * D;
      else
        base = (((int64_t)b * p.Sq + qi) * p.Hq + h) * D;
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        uint32_t o[32];
        if (have_o) {
          tmem_ld32(o_addr + k * 32, o);
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
          uint4* dst = reinterpret_cast<uint4*>(out + base + k * 32);
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
  const dim3 grid((unsigned)((P.c.Sq + kQTiles * BM - 1) / (kQTiles * BM)), (unsigned)P.c.Hq,
                  (unsigned)P.c.B);
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
