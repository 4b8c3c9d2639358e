// attn_decode.cu -- attention forward for few query rows per kv head (decode:
// one or a few new tokens per sequence over a long KV cache), on tcgen05.
//
// The definition is the one of "onnx-runtime-ep-cuda 0.1.0-dev.5,
// src/kernels/flash_attention.rs" (kernel `flash_attention_body`): per row the
// visible keys, scale, soft-cap, additive mask and an online softmax over key
// tiles.  That page sends Sq = 1 to a separate decode kernel
// (`gqa_decode_fp16`, named at its dispatch in `run`); this file is that case,
// designed for this GPU.
//
// With group * Sq <= 32 query rows per kv head, a 128-row query tile would be
// nearly empty and every query head would stream the same K / V again.  Here
// one CTA takes one (batch, kv head) and a part of its key tiles, and puts
// every query row of that kv head in the N dimension of the tensor-core
// products, keys in M:
//   S^T[key, row] = K_tile Q^T          (M = 128 keys, N = 16 or 32 rows, K = D)
//   O^T[d, row]  += V_tile^T P^T        (M = 128 (d),   N = 16 or 32 rows, K = 128 keys)
// so K and V are read once per kv head and the launch streams them at HBM
// rate.  Each of the 128 softmax threads owns one key (one TMEM lane of S^T);
// row maxima and sums are reduced across threads (warp shuffles, then one
// shared-memory exchange through a bounded mbarrier).
//
// Roles (224 threads): warps 0-3 softmax, warp 4 K loads (TMA), warp 5 V loads
// (TMA), warp 6 MMA issue.  A kv head's key tiles can be cut into parts in two
// ways, combinable: a thread-block cluster of up to 8 CTAs whose partial rows
// are merged through distributed shared memory by the cluster's first CTA,
// and num_splits key ranges whose partial O / l and log-sum-exp go to a
// workspace for the merge kernel.  With neither, the CTA writes the output.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_decode.h"
#include "device_common.cuh"

namespace gb300_attn {
namespace {

constexpr int kDecThreads = 224;
constexpr int kDecKeys = 128;  // keys per tile (M of S^T)
constexpr int kKWarp = 4, kVWarp = 5, kMmaWarp = 6;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past a 256x growth

// Stage counts of the K and V rings for D = 128 (D = 64 uses 3 and 2) and the
// CTAs per SM the 16-row variant is compiled for.
#ifndef GB300_DEC_K_STAGES
#define GB300_DEC_K_STAGES 2
#endif
#ifndef GB300_DEC_V_STAGES
#define GB300_DEC_V_STAGES 1
#endif
#ifndef GB300_DEC_MIN_BLOCKS
#define GB300_DEC_MIN_BLOCKS 2
#endif

template <int D, int NR>
struct DecConfig {
  static constexpr int kSub = D / 64;                  // 64-column (128-byte) blocks per row
  static constexpr int kSubBytes = kDecKeys * 128;      // one 64-column block of a K / V tile
  static constexpr int kTileBytes = kSub * kSubBytes;   // one K or V tile
  static constexpr int kSK = D == 128 ? GB300_DEC_K_STAGES : 3;  // K stages
  static constexpr int kSV = D == 128 ? GB300_DEC_V_STAGES : 2;  // V stages
  static constexpr int kRowBlock = NR * 128;            // one 64-column block of Q or P^T
  static constexpr int kQBytes = kSub * kRowBlock;
  static constexpr int kPBytes = 2 * kRowBlock;         // 128 keys = two 64-key blocks
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kSK * kTileBytes;
  static constexpr int kOffQ = kOffV + kSV * kTileBytes;
  static constexpr int kOffP = kOffQ + kQBytes;         // two buffers
  static constexpr int kOffRed = kOffP + 2 * kPBytes;   // float [2][4][NR]
  static constexpr int kOffLim = kOffRed + 2 * 4 * NR * 4;  // int2 [NR]: visible keys per row
  static constexpr int kOffMrow = kOffLim + NR * 8;     // int64 [NR]: mask row offset per row
  static constexpr int kOffBar = kOffMrow + NR * 8;
  // k_full[kSK] k_empty[kSK] v_full[kSV] v_empty[kSV] s_full[2] p_full[2] pv_done[2] red
  static constexpr int kNumBars = 2 * kSK + 2 * kSV + 7;
  static constexpr int kOffSlot = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffSlot + 16 + 1024;  // + 1024-byte alignment slack
  static constexpr int kColO = 2 * NR;                      // TMEM: S^T x2, then O^T
  static constexpr uint32_t kTmemCols = 3 * NR <= 64 ? 64u : 128u;
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kRowBlock % 1024 == 0, "SW128 alignment");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert((NR * D + NR) * 4 <= kSK * kTileBytes, "cluster exchange fits in the K ring");
};

template <int D, int NR>
struct DecLayout {
  using C = DecConfig<D, NR>;
  uint8_t* base;
  uint32_t s;  // shared address of base
  __device__ uint32_t k_tile(int st) const { return s + C::kOffK + st * C::kTileBytes; }
  __device__ uint32_t v_tile(int st) const { return s + C::kOffV + st * C::kTileBytes; }
  __device__ uint8_t* v_ptr(int st) const { return base + C::kOffV + st * C::kTileBytes; }
  __device__ uint32_t q() const { return s + C::kOffQ; }
  __device__ uint8_t* q_ptr() const { return base + C::kOffQ; }
  __device__ uint32_t p_buf(int i) const { return s + C::kOffP + i * C::kPBytes; }
  __device__ uint8_t* p_ptr(int i) const { return base + C::kOffP + i * C::kPBytes; }
  __device__ float* red(int slot) const { return reinterpret_cast<float*>(base + C::kOffRed) + slot * 4 * NR; }
  __device__ int2* lim() const { return reinterpret_cast<int2*>(base + C::kOffLim); }
  __device__ int64_t* mrow() const { return reinterpret_cast<int64_t*>(base + C::kOffMrow); }
  __device__ uint32_t k_full(int i) const { return s + C::kOffBar + i * 8; }
  __device__ uint32_t k_empty(int i) const { return s + C::kOffBar + (C::kSK + i) * 8; }
  __device__ uint32_t v_full(int i) const { return s + C::kOffBar + (2 * C::kSK + i) * 8; }
  __device__ uint32_t v_empty(int i) const { return s + C::kOffBar + (2 * C::kSK + C::kSV + i) * 8; }
  __device__ uint32_t s_full(int i) const { return s + C::kOffBar + (2 * C::kSK + 2 * C::kSV + i) * 8; }
  __device__ uint32_t p_full(int i) const { return s + C::kOffBar + (2 * C::kSK + 2 * C::kSV + 2 + i) * 8; }
  __device__ uint32_t pv_done(int i) const { return s + C::kOffBar + (2 * C::kSK + 2 * C::kSV + 4 + i) * 8; }
  __device__ uint32_t red_bar() const { return s + C::kOffBar + (2 * C::kSK + 2 * C::kSV + 6) * 8; }
  __device__ uint32_t* slot() const { return reinterpret_cast<uint32_t*>(base + C::kOffSlot); }
  // softmax warps that finished their partial rows (4 when the CTA's part is
  // complete; fewer after a timed-out wait)
  __device__ int* done_warps() const { return reinterpret_cast<int*>(base + C::kOffSlot + 8); }
  // cluster exchange, over the K ring once every S^T product is done:
  // normalised partial rows [NR][D] and their log-sum-exps (log2 units) [NR]
  __device__ float* xo() const { return reinterpret_cast<float*>(base + C::kOffK); }
  __device__ float* xl() const { return xo() + NR * D; }
};

// The (batch, kv head, part) of a CTA and its key tiles.
struct DecUnit {
  int b, kvh;
  int part;        // key range (split) index; its partial row goes to the workspace
  int rank;        // CTA index within the cluster
  int R;           // query rows of this kv head: group * Sq
  int64_t row0;    // first row (b * Hq + kvh * group) * Sq in [B*Hq*Sq]
  int t0, n;       // key tiles [t0, t0 + n)
  int64_t zero_from;  // V rows at or past this key hold no valid data
};

__device__ __forceinline__ DecUnit dec_unit(const CommonParams& p, int P_cluster) {
  DecUnit u;
  u.part = blockIdx.x / P_cluster;
  u.rank = blockIdx.x % P_cluster;
  u.kvh = blockIdx.y;
  u.b = blockIdx.z;
  u.R = p.group * p.Sq;
  u.row0 = ((int64_t)u.b * p.Hq + (int64_t)u.kvh * p.group) * p.Sq;
  const BatchLimits L = batch_limits(p, u.b);
  // visible ranges grow with qi: the union is [lo(0), hi(Sq-1))
  const RowLimits first = row_limits(p, L, 0), last = row_limits(p, L, p.Sq - 1);
  int tb = 0, te = 0;
  if (last.hi > first.lo) {
    tb = first.lo / kDecKeys;
    te = (last.hi + kDecKeys - 1) / kDecKeys;
  }
  const int total = te - tb;
  const int parts = p.num_splits * P_cluster;  // = gridDim.x
  const int per = (total + parts - 1) / parts;
  int a = tb + (int)blockIdx.x * per, e = a + per;
  if (a > te) a = te;
  if (e > te) e = te;
  u.t0 = a;
  u.n = e - a;
  int64_t zf = L.lsk < (int64_t)p.Sk ? L.lsk : (int64_t)p.Sk;
  u.zero_from = zf < 0 ? 0 : zf;
  return u;
}

// tcgen05 instruction descriptor, kind::f16, fp32 accumulator, with both
// operand major-nesses selectable (bit 15 A, bit 16 B; 1 = MN-major).
__host__ __device__ constexpr uint32_t dec_idesc(bool bf16, int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Loads NR consecutive 32-bit TMEM columns of this thread's lane.
template <int NR>
__device__ __forceinline__ void tmem_ld_nr(uint32_t taddr, uint32_t (&r)[NR]);

template <>
__device__ __forceinline__ void tmem_ld_nr<16>(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld_nr<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}

template <int NR>
__device__ __forceinline__ void tmem_st_nr(uint32_t taddr, const uint32_t (&r)[NR]);

template <>
__device__ __forceinline__ void tmem_st_nr<16>(uint32_t taddr, const uint32_t (&r)[16]) {
  tmem_st16(taddr, r);
}

template <>
__device__ __forceinline__ void tmem_st_nr<32>(uint32_t taddr, const uint32_t (&r)[32]) {
  tmem_st32(taddr, r);
}

// Reduce-scatter across the warp: on entry every lane holds NR values (one
// per row); on exit lane l holds, for row dec_row_of_lane<NR>(l), the max (or
// sum) over all 32 lanes.  NR - 1 + (32 / NR == 2 ? 1 : 0) shuffles.
template <int NR>
__device__ __forceinline__ int dec_row_of_lane(int lane) {
  // halving steps over lane bits 4, 3, ... keep the upper half in lanes with the bit set
  int r = 0, half = NR / 2;
#pragma unroll
  for (int bit = 4; half >= 1; --bit, half >>= 1)
    if (lane & (1 << bit)) r += half;
  return r;
}

template <int NR, bool MAX>
__device__ __forceinline__ float dec_reduce_scatter(float (&v)[NR], int lane) {
#pragma unroll
  for (int half = NR / 2, bit = 4; half >= 1; half >>= 1, --bit) {
    const bool upper = (lane >> bit) & 1;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = upper ? v[k] : v[k + half];
      const float keep = upper ? v[k + half] : v[k];
      const float got = __shfl_xor_sync(0xffffffffu, send, 1 << bit);
      v[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float x = v[0];
  // lanes not yet combined: the remaining low bits (NR = 16: bit 0)
#pragma unroll
  for (int bit = 0; (1 << bit) < 32 / NR; ++bit) {
    const float got = __shfl_xor_sync(0xffffffffu, x, 1 << bit);
    x = MAX ? fmaxf(x, got) : x + got;
  }
  return x;
}

// ------------------------------------------------------------------ loaders
// One thread streams the unit's K (or V) tiles through a ring of NS stages.
// Stage st is refilled once the MMA that read it has committed `empty(st)`.
template <int D, int NR, int NS>
__device__ __forceinline__ void dec_loader(const CommonParams& p, const CUtensorMap* tmap,
                                           const DecUnit& u, uint32_t ring, uint32_t full0,
                                           uint32_t empty0) {
  using C = DecConfig<D, NR>;
  const int plane = u.b * p.Hkv + u.kvh;
  for (int n = 0; n < u.n; ++n) {
    const int st = n % NS;
    if (n >= NS && !mbar_wait(empty0 + st * 8, ((n / NS) - 1) & 1, p.timeout_ns, p.status)) return;
    const uint32_t full = full0 + st * 8;
    mbar_arrive_expect_tx(full, C::kTileBytes);
    const int key0 = (u.t0 + n) * kDecKeys;
#pragma unroll
    for (int s = 0; s < C::kSub; ++s)
      tma_load_3d(ring + st * C::kTileBytes + s * C::kSubBytes, tmap, full, s * 64, key0, plane);
  }
  // let every copy land before the CTA may exit
  for (int n = u.n > NS ? u.n - NS : 0; n < u.n; ++n)
    mbar_wait(full0 + (n % NS) * 8, (n / NS) & 1, p.timeout_ns, p.status);
}

// ---------------------------------------------------------------- MMA issuer
// Whole warp waits, lane 0 issues.  Iteration n: S^T(n) into S buffer n % 2,
// then O^T += V^T(n-1) P^T(n-1).  S buffer n % 2 is free because P(n-2),
// which the softmax wrote after reading S(n-2), was waited for one iteration
// earlier.
template <int D, int NR, bool BF16>
__device__ __forceinline__ void dec_mma(const CommonParams& p, const DecLayout<D, NR>& sm,
                                        const DecUnit& u, uint32_t tmem, int lane) {
  using C = DecConfig<D, NR>;
  constexpr uint32_t idesc_s = dec_idesc(BF16, kDecKeys, NR, false, false);
  constexpr uint32_t idesc_o = dec_idesc(BF16, 128, NR, true, false);
  // V^T as the M-major A operand: d in 64-column blocks kSubBytes apart (for
  // D = 64 both halves of M = 128 read the same block, so O^T lanes 64-127
  // repeat lanes 0-63), 8-key groups 1024 bytes apart, 2048 bytes per 16 keys.
  constexpr uint32_t v_lbo = D == 128 ? (uint32_t)C::kSubBytes : 0u;

  auto pv = [&](int t) -> bool {
    if (!mbar_wait_warp(sm.p_full(t & 1), (t >> 1) & 1, p.timeout_ns, p.status)) return false;
    const int vs = t % C::kSV;
    if (!mbar_wait_warp(sm.v_full(vs), (t / C::kSV) & 1, p.timeout_ns, p.status)) return false;
    const int64_t key0 = (int64_t)(u.t0 + t) * kDecKeys;
    if (u.zero_from < key0 + kDecKeys) {
      // cache slots past the valid length may hold NaN / Inf; P is 0 there but
      // 0 * NaN is not, so those V rows are zeroed (whole 128-byte rows)
      const int r0 = u.zero_from > key0 ? (int)(u.zero_from - key0) : 0;
      const int chunks = (kDecKeys - r0) * 8;
      for (int s = 0; s < C::kSub; ++s) {
        uint8_t* blk = sm.v_ptr(vs) + s * C::kSubBytes;
        for (int c = lane; c < chunks; c += 32)
          *reinterpret_cast<uint4*>(blk + (size_t)(r0 + (c >> 3)) * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    tc_fence_after();
    // the converged warp issues; one elected lane starts the MMAs (see mma_ss_elect)
    const uint64_t adesc0 = make_sdesc_sw128(sm.v_tile(vs), v_lbo, 1024);
    const uint64_t bdesc0 = make_sdesc_sw128(sm.p_buf(t & 1), 16, 1024);
#pragma unroll
    for (int kk = 0; kk < kDecKeys / 16; ++kk)
      mma_ss_elect(tmem + C::kColO, adesc0 + (uint32_t)((kk * 2048) >> 4),
                   bdesc0 + (uint32_t)(((kk >> 2) * C::kRowBlock + (kk & 3) * 32) >> 4), idesc_o,
                   (t > 0 || kk > 0) ? 1u : 0u);
    tc_commit_elect(sm.pv_done(t & 1));
    tc_commit_elect(sm.v_empty(vs));
    return true;
  };

  for (int n = 0; n < u.n; ++n) {
    const int ks = n % C::kSK;
    if (!mbar_wait_warp(sm.k_full(ks), (n / C::kSK) & 1, p.timeout_ns, p.status)) return;
    tc_fence_after();
    {
      const uint64_t adesc0 = make_sdesc_sw128(sm.k_tile(ks), 16, 1024);
      const uint64_t bdesc0 = make_sdesc_sw128(sm.q(), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(tmem + (n & 1) * NR, adesc0 + (uint32_t)(((kk >> 2) * C::kSubBytes + (kk & 3) * 32) >> 4),
                     bdesc0 + (uint32_t)(((kk >> 2) * C::kRowBlock + (kk & 3) * 32) >> 4), idesc_s,
                     kk > 0 ? 1u : 0u);
      tc_commit_elect(sm.s_full(n & 1));
      tc_commit_elect(sm.k_empty(ks));
    }
    if (n >= 1 && !pv(n - 1)) return;
  }
  if (u.n >= 1) pv(u.n - 1);
}

template <bool BF16>
__device__ __forceinline__ uint16_t dec_to_bits(float x) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

// Row r of the unit, column d = tid: the normalised value and the row's
// log-sum-exp in log2 units, to the workspace (split) or the output.
template <int D, bool BF16>
__device__ __forceinline__ void dec_store_row(const CommonParams& p, const DecUnit& u, int r, int tid,
                                              float val, float lse2) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  const int64_t row = u.row0 + r;
  const float lse = lse2 * kLn2;  // -inf stays -inf
  if (p.num_splits > 1) {
    if (tid < D) p.ws_o[((int64_t)u.part * rows + row) * D + tid] = val;
    if (tid == r) p.ws_lse[(int64_t)u.part * rows + row] = lse;
    return;
  }
  if (tid < D) {
    int64_t idx = row * D + tid;
    if (p.out_layout != 0) {
      const int qi = r % p.Sq, h = u.kvh * p.group + r / p.Sq;
      idx = (((int64_t)u.b * p.Sq + qi) * p.Hq + h) * D + tid;
    }
    reinterpret_cast<uint16_t*>(p.out)[idx] = dec_to_bits<BF16>(val);
  }
  if (p.lse != nullptr && tid == r) p.lse[row] = lse;
}

// Distributed shared memory: a 32-bit load from CTA `rank` of the cluster at
// the offset of this CTA's shared address `saddr`.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t saddr, int rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Every thread of every CTA of the cluster arrives; release / acquire order
// shared-memory writes before the other CTAs' reads.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ------------------------------------------------------------------ softmax
// Thread tid of warps 0-3 owns key tid of every tile (TMEM lane tid of S^T)
// and, in the epilogue, column d = tid of O^T.  Scores are kept in log2
// units; the running maximum m of a row moves (and O^T and l are rescaled)
// only when a tile raises it by more than kRescaleThreshold.
template <int D, int NR, bool BF16>
__device__ __forceinline__ void dec_softmax(const CommonParams& p, const DecLayout<D, NR>& sm,
                                            const DecUnit& u, uint32_t tmem, int cluster, int warp,
                                            int lane) {
  using C = DecConfig<D, NR>;
  const int tid = warp * 32 + lane;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const bool has_mask = p.mask != nullptr;
  const bool has_cap = p.softcap > 0.0f;
  const int2* lim = sm.lim();
  const int64_t* mrow = sm.mrow();
  float m[NR], l[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
  }
  bool ok = true;
  int use = 0;  // completed phases of red_bar
  for (int n = 0; n < u.n; ++n) {
    const int j = (u.t0 + n) * kDecKeys + tid;
    float t[NR];  // the mask term first (its loads issued before the S wait), then the score
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int2 lr = lim[r];  // rows past R have empty limits
      t[r] = (has_mask && j >= lr.x && j < lr.y) ? __ldg(p.mask + mrow[r] + j) * kLog2e : 0.0f;
    }
    if (!mbar_wait_warp(sm.s_full(n & 1), (n >> 1) & 1, p.timeout_ns, p.status)) { ok = false; break; }
    tc_fence_after();
    float x[NR];
    tmem_ld_nr<NR>(tmem + lane_base + (uint32_t)((n & 1) * NR), reinterpret_cast<uint32_t(&)[NR]>(x));
    tmem_wait_ld();
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float v = t[r] + (has_cap ? soft_cap_log2(x[r], p.sc_k1, p.sc_k2, p.sc_k3) : x[r] * p.scale_log2);
      const int2 lr = lim[r];
      t[r] = (j >= lr.x && j < lr.y) ? v : -INFINITY;  // a select: invisible keys never add
      x[r] = t[r];
    }
    // tile maximum of every row over the 128 keys
    const float wmax = dec_reduce_scatter<NR, true>(x, lane);
    float* red = sm.red(use & 1);
    if (NR == 32 || (lane & 1) == 0) red[warp * NR + dec_row_of_lane<NR>(lane)] = wmax;
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.red_bar());
    if (!mbar_wait_warp(sm.red_bar(), use & 1, p.timeout_ns, p.status)) { ok = false; break; }
    ++use;
    float* alpha = x;  // reused: 1 for rows whose maximum stays
    bool any = false;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float tm = fmaxf(fmaxf(red[r], red[NR + r]), fmaxf(red[2 * NR + r], red[3 * NR + r]));
      const float mn = fmaxf(m[r], tm);
      const bool up = mn > m[r] + kRescaleThreshold;  // false while the row has seen nothing
      alpha[r] = up ? fast_exp2(m[r] - mn) : 1.0f;     // m = -inf gives 0
      if (up) m[r] = mn;
      l[r] *= alpha[r];
      any |= up;
    }
    if (any) {  // the same decision in every thread: m is uniform
      if (n > 0) {  // O^T holds tiles < n once P.V(n-1) has completed
        if (!mbar_wait_warp(sm.pv_done((n - 1) & 1), ((n - 1) >> 1) & 1, p.timeout_ns, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t o[NR];
        tmem_ld_nr<NR>(tmem + lane_base + (uint32_t)C::kColO, o);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
        tmem_st_nr<NR>(tmem + lane_base + (uint32_t)C::kColO, o);
        tmem_wait_st();
      }
    }
    // P buffer n % 2 was last read by P.V(n-2)
    if (n >= 2 && !mbar_wait_warp(sm.pv_done(n & 1), ((n - 2) >> 1) & 1, p.timeout_ns, p.status)) {
      ok = false;
      break;
    }
    // P^T[row r][key tid], K-major with 128-byte swizzle: 64-key blocks
    // kRowBlock apart, rows 128 bytes apart in groups of 8 (1024 bytes),
    // 16-byte chunk index XOR (row % 8).
    uint8_t* pb = sm.p_ptr(n & 1) + (tid >> 6) * C::kRowBlock + (tid & 7) * 2;
    const int kc = (tid >> 3) & 7;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float pr = t[r] == -INFINITY ? 0.0f : fast_exp2(t[r] - m[r]);
      l[r] += pr;
      *reinterpret_cast<uint16_t*>(pb + (r >> 3) * 1024 + (r & 7) * 128 + ((kc ^ (r & 7)) << 4)) =
          dec_to_bits<BF16>(pr);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.p_full(n & 1));
  }
  if (!ok) return;

  // ---- epilogue: row sums over the 128 threads, then O^T / l per row
  float x[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) x[r] = l[r];
  const float wsum = dec_reduce_scatter<NR, false>(x, lane);
  float* red = sm.red(use & 1);
  if (NR == 32 || (lane & 1) == 0) red[warp * NR + dec_row_of_lane<NR>(lane)] = wsum;
  __syncwarp();
  if (lane == 0) mbar_arrive(sm.red_bar());
  if (!mbar_wait_warp(sm.red_bar(), use & 1, p.timeout_ns, p.status)) return;
  float o[NR];
  if (u.n > 0) {
    if (!mbar_wait_warp(sm.pv_done((u.n - 1) & 1), ((u.n - 1) >> 1) & 1, p.timeout_ns, p.status)) return;
    tc_fence_after();
    uint32_t ob[NR];
    tmem_ld_nr<NR>(tmem + lane_base + (uint32_t)C::kColO, ob);
    tmem_wait_ld();
#pragma unroll
    for (int r = 0; r < NR; ++r) o[r] = __uint_as_float(ob[r]);
  } else {
#pragma unroll
    for (int r = 0; r < NR; ++r) o[r] = 0.0f;
  }
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    if (r >= u.R) break;
    const float Lr = red[r] + red[NR + r] + red[2 * NR + r] + red[3 * NR + r];
    const float inv = Lr > 0.0f ? 1.0f / Lr : 0.0f;
    const float lse2 = Lr > 0.0f ? m[r] + log2f(Lr) : -INFINITY;
    if (cluster > 1) {  // to shared memory, for the cluster's first CTA to merge
      if (tid < D) sm.xo()[r * D + tid] = o[r] * inv;
      if (tid == r) sm.xl()[r] = lse2;
    } else {
      dec_store_row<D, BF16>(p, u, r, tid, o[r] * inv, lse2);
    }
  }
  if (cluster > 1) {
    __syncwarp();
    if (lane == 0) atomicAdd(sm.done_warps(), 1);  // this warp's share of the part is written
  }
}

__device__ __forceinline__ int ld_dsmem_s32(uint32_t saddr, int rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(rank));
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

// Cluster merge, by the softmax threads of the cluster's first CTA: row r of
// the CTAs' parts combines as O = sum_k w_k O_k / sum_k w_k with
// w_k = 2^(lse_k - max lse), read from each CTA's shared memory.
template <int D, int NR, bool BF16>
__device__ __forceinline__ void dec_cluster_merge(const CommonParams& p, const DecLayout<D, NR>& sm,
                                                  const DecUnit& u, int cluster, int tid) {
  const uint32_t xo = smem_u32(sm.xo()), xl = smem_u32(sm.xl());
  // A CTA whose wait timed out left its part unwritten (the status word has
  // the timeout): its rows are then written as 0 with log-sum-exp -inf rather
  // than merged from stale shared memory.
  bool complete = true;
  for (int k = 0; k < cluster; ++k) complete &= ld_dsmem_s32(smem_u32(sm.done_warps()), k) == 4;
  if (!complete) {
    for (int r = 0; r < u.R; ++r) dec_store_row<D, BF16>(p, u, r, tid, 0.0f, -INFINITY);
    return;
  }
  for (int r = 0; r < u.R; ++r) {
    float lk[8];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      lk[k] = k < cluster ? ld_dsmem_f32(xl + r * 4, k) : -INFINITY;
      mx = fmaxf(mx, lk[k]);
    }
    float wsum = 0.0f, acc = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float w = lk[k] == -INFINITY ? 0.0f : exp2f(lk[k] - mx);
      wsum += w;
      if (w > 0.0f && tid < D) acc = fmaf(w, ld_dsmem_f32(xo + (uint32_t)(r * D + tid) * 4, k), acc);
    }
    dec_store_row<D, BF16>(p, u, r, tid, wsum > 0.0f ? acc / wsum : 0.0f,
                           wsum > 0.0f ? mx + log2f(wsum) : -INFINITY);
  }
}

// -------------------------------------------------------------------- kernel
template <int D, int NR, bool BF16>
__global__ void __launch_bounds__(kDecThreads, NR == 16 ? GB300_DEC_MIN_BLOCKS : 1) attn_decode_kernel(const __grid_constant__ DecodeParams P) {
  using C = DecConfig<D, NR>;
  const CommonParams& p = P.c;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecLayout<D, NR> sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  sm.s = smem_u32(sm.base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DecUnit u = dec_unit(p, P.cluster);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSK; ++i) {
      mbar_init(sm.k_full(i), 1);
      mbar_init(sm.k_empty(i), 1);
    }
    for (int i = 0; i < C::kSV; ++i) {
      mbar_init(sm.v_full(i), 1);
      mbar_init(sm.v_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sm.s_full(i), 1);
      mbar_init(sm.p_full(i), 4);  // one arrival per softmax warp
      mbar_init(sm.pv_done(i), 1);
    }
    mbar_init(sm.red_bar(), 4);
    *sm.done_warps() = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < NR) {  // visible keys and mask row of every query row
    const int r = threadIdx.x;
    int2 lr = make_int2(0, 0);
    int64_t mo = 0;
    if (r < u.R) {
      const int qi = r % p.Sq, h = u.kvh * p.group + r / p.Sq;
      const RowLimits rl = row_limits(p, batch_limits(p, u.b), qi);
      lr = make_int2(rl.lo, rl.hi);
      if (p.mask != nullptr) {
        int64_t plane = 0;
        if (p.mask_planes == p.B) plane = u.b;
        else if ((int64_t)p.mask_planes == (int64_t)p.B * p.Hq) plane = (int64_t)u.b * p.Hq + h;
        mo = (plane * p.Sq + qi) * (int64_t)p.Sk;
      }
    }
    sm.lim()[r] = lr;
    sm.mrow()[r] = mo;
  }
  {  // Q rows of this kv head, K-major with 128-byte swizzle; rows past R are 0
    constexpr int kChunks = D / 8;  // 16-byte chunks per row
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(P.q) + u.row0 * D);
    for (int c = threadIdx.x; c < NR * kChunks; c += kDecThreads) {
      const int r = c / kChunks, k = c % kChunks;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (r < u.R) val = __ldg(q + (int64_t)r * kChunks + k);
      *reinterpret_cast<uint4*>(sm.q_ptr() + (k >> 3) * C::kRowBlock + (r >> 3) * 1024 + (r & 7) * 128 +
                                (((k & 7) ^ (r & 7)) << 4)) = val;
    }
    fence_proxy_async_smem();
  }
  if (warp == kKWarp && lane == 0) tma_prefetch_desc(&P.tmap_k);
  if (warp == kVWarp && lane == 0) tma_prefetch_desc(&P.tmap_v);
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(sm.slot()), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm.slot());

  if (warp < 4) {
    dec_softmax<D, NR, BF16>(p, sm, u, tmem, P.cluster, warp, lane);
  } else if (warp == kKWarp) {
    if (lane == 0) dec_loader<D, NR, C::kSK>(p, &P.tmap_k, u, sm.k_tile(0), sm.k_full(0), sm.k_empty(0));
  } else if (warp == kVWarp) {
    if (lane == 0) dec_loader<D, NR, C::kSV>(p, &P.tmap_v, u, sm.v_tile(0), sm.v_full(0), sm.v_empty(0));
  } else {
    dec_mma<D, NR, BF16>(p, sm, u, tmem, lane);
  }
  if (P.cluster > 1) {
    cluster_sync_all();  // every CTA's partial rows are in its shared memory
    if (u.rank == 0 && warp < 4) dec_cluster_merge<D, NR, BF16>(p, sm, u, P.cluster, threadIdx.x);
    cluster_sync_all();  // ... and have been read: no CTA's shared memory goes away earlier
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int NR, bool BF16>
cudaError_t launch_dec(const DecodeParams& P, cudaStream_t stream) {
  auto kernel = attn_decode_kernel<D, NR, BF16>;
  constexpr int smem = DecConfig<D, NR>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the whole carve-out as shared memory, so two CTAs fit on an SM where the size allows
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(P.c.num_splits * P.cluster), (unsigned)P.c.Hkv, (unsigned)P.c.B);
  if (P.cluster <= 1) {
    kernel<<<grid, kDecThreads, smem, stream>>>(P);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kDecThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

template <int D, bool BF16>
cudaError_t launch_dec_d(const DecodeParams& P, cudaStream_t stream) {
  return P.c.group * P.c.Sq <= 16 ? launch_dec<D, 16, BF16>(P, stream) : launch_dec<D, 32, BF16>(P, stream);
}

}  // namespace

cudaError_t launch_attn_decode(const DecodeParams& P, bool bf16, cudaStream_t stream) {
  const int64_t rows = (int64_t)P.c.group * P.c.Sq;
  if (rows < 1 || rows > kDecodeMaxRows || P.c.num_splits < 1 || P.cluster < 1 || P.cluster > 8 ||
      (P.c.D != 64 && P.c.D != 128))
    return cudaErrorInvalidValue;
  if (P.c.D == 128) return bf16 ? launch_dec_d<128, true>(P, stream) : launch_dec_d<128, false>(P, stream);
  return bf16 ? launch_dec_d<64, true>(P, stream) : launch_dec_d<64, false>(P, stream);
}

}  // namespace gb300_attn
