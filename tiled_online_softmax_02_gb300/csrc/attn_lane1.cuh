#pragma once
// attn_lane1.cuh -- single-lane tensor-core attention forward for sm_103a:
// one softmax warpgroup per CTA, two MMA issuers, two or three S buffers.
// Used where the ping-pong tile kernel's tensor-memory layout does not fit:
//   - fp32 inputs as error-compensated bf16 pieces (attn_f32tc.cu, D 64 /
//     128): Q and K in three pieces, P and V in two, six products for QK^T
//     and three for P.V;
//   - bf16 / f16 inputs with D = 256 or 384 (attn_lane16.cu): one piece
//     each.  At D = 384, O alone takes 384 of the 512 tensor-memory columns,
//     so Q goes to shared memory by TMA instead (QK^T as an SS-MMA, 96 KB),
//     and K and V stream through their rings in units (K in 128-dim chunks
//     of 16 KB, V in 16-key sub-tiles of 12 KB), which keeps Q, the rings
//     and the mask buffers within the 227 KB of shared memory a CTA may use.
//
// The method is the tiled online softmax of "onnx-runtime-ep-cuda
// 0.1.0-dev.5, src/kernels/flash_attention.rs" (module doc and
// `flash_attention_body`): scores of one key tile at a time, running row
// max and denominator, O rescaled when the max moves.  Work item = one
// 128-row query tile of one (b, h); its 64-key tiles run in order; key tile
// g of the CTA (counted over all its items) uses S buffer g % SB.
//   warps 0-3   softmax: thread = query row.  They write each item's Q rows
//               (split into pieces for fp32) to tensor memory (except at
//               D = 384) as soon as the previous item's last P is written,
//               ahead of that item's epilogue.
//   warp 4      TMA producer: the K and V units of each key tile into their
//               rings (unit u in slot u % KS or u % VS), each ring with its
//               own barriers, V one tile behind K; it also prefetches each
//               item's Q block into L2 (at D = 384: loads it into shared
//               memory).
//   warp 5      QK^T issuer (converged warp, elect.sync) and owner of tensor
//               memory: S_g = Q K_g^T once K_g is in and the P.V of tile
//               g - SB (whose P the buffer holds) has finished.
//   warp 6      P.V issuer: O += P_g V_g once P_g is written.
// Tensor memory (512 columns): Q pieces [0, KP D/2), SB S buffers of 64
// columns from kColS, O (D columns) after them; P_b
// over S_b (as VP bf16 / f16 pieces of FN / 2 columns).  Every barrier wait
// is bounded; a timeout sets ATTN_ERR_TIMEOUT in the device status word and
// the kernel drains and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"

namespace gb300_attn {
namespace lane1 {

constexpr int FM = 128;          // query rows per item
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;      // issues every MMA, or QK^T only with a second issuer
constexpr int kPvWarp = 6;       // the second issuer (P.V), where there is one
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;  // keep the old max while it is within 2^8
constexpr float kLog2e = 1.4426950408889634f;

// Input kinds.
constexpr int kInF32Split = 0;  // fp32 q / k / v, K / V pre-split in a workspace, fp32 out
constexpr int kInF16 = 1;
constexpr int kInBF16 = 2;

template <int IN>
struct In {
  static constexpr int KP = IN == kInF32Split ? 3 : 1;   // pieces of Q and K
  static constexpr int VP = IN == kInF32Split ? 2 : 1;   // pieces of P and V
  static constexpr bool kBF16 = IN != kInF16;            // MMA operand type (pieces are bf16)
};

template <int D, int IN>
struct Cfg {
  static constexpr int KP = In<IN>::KP, VP = In<IN>::VP;
  // Q in shared memory (SS-MMA) when O leaves no tensor-memory room for it
  static constexpr bool kQSmem = IN != kInF32Split && D > 256;
  static constexpr int FN = 64;                                // keys per key tile
  static constexpr int kSub = D / 64;                          // 128-byte column blocks per row
  static constexpr uint32_t kSubBytes = FN * 128;              // [FN rows][64 cols] of 16-bit
  static constexpr uint32_t kPieceBytes = kSub * kSubBytes;    // one piece of one tile
  static constexpr uint32_t kKTileBytes = KP * kPieceBytes;
  static constexpr uint32_t kVTileBytes = VP * kPieceBytes;
  static constexpr uint32_t kQSubBytes = FM * 128;             // [128 rows][64 cols] of 16-bit
  static constexpr uint32_t kQBytes = kQSmem ? kSub * kQSubBytes : 0;
  // The K and V rings hold units: a whole key tile, or at D = 384 (whose Q
  // takes 96 KB of shared memory) K in chunks of 128 dims (16 KB) and V in
  // sub-tiles of 16 keys (12 KB), so that 64-key tiles still stream through
  // a few slots.  A K unit is freed by its QK^T products, a V unit by its
  // P.V products; the producer loads V one tile behind K.
  static constexpr int kKUnits = kQSmem ? D / 128 : 1;         // K units per key tile
  static constexpr int kVUnits = kQSmem ? FN / 16 : 1;         // V units per key tile
  static constexpr uint32_t kKUnitBytes = kKTileBytes / kKUnits;
  static constexpr uint32_t kVUnitBytes = kVTileBytes / kVUnits;
  static constexpr uint32_t kVUnitSubBytes = kSubBytes / kVUnits;  // [16 rows][64 cols] at D = 384
  // ring slots (units): 4 / 5 at fp32 D = 64, 2 / 3 at fp32 D = 128, 3 / 3 at
  // D = 256, 4 / 4 at D = 384
  static constexpr int kKStages = kQSmem ? 4 : (kKTileBytes <= 24576 ? 4 : (IN == kInF32Split ? 2 : 3));
  static constexpr int kVStages = kQSmem ? 4 : (IN != kInF32Split ? kKStages : kKStages + 1);
  // S buffers: three where tensor memory has room for them (fp32 pieces),
  // else two.  Two MMA warps issue (QK^T and P.V), so that neither issuer's
  // barrier waits leave the tensor core without queued work.
  static constexpr int kSBufs = IN == kInF32Split ? 3 : 2;
  static constexpr int kThreads = 224;  // 4 softmax warps, producer, two MMA issuers
  // mask staging per softmax warp: 32 rows x kMaskKeys keys of f32
  static constexpr int kMaskKeys = kQSmem ? 16 : 32;
  static constexpr uint32_t kMaskBufBytes = 32 * kMaskKeys * 4;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kKUnitBytes;
  static constexpr uint32_t kOffMaskBuf = kOffV + kVStages * kVUnitBytes;
  static constexpr uint32_t kOffBar = kOffMaskBuf + 4 * kMaskBufBytes;
  // k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], q_full, q_empty,
  // s_full[SB], p_full[SB], s_free[SB], pv_done, o_final, drain
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 + 3 * kSBufs + 3;
  static constexpr uint32_t kOffSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffSlot + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  // tensor memory columns
  static constexpr uint32_t kQPiece = D / 2;                       // columns per piece of Q
  static constexpr uint32_t kColQ = 0;
  static constexpr uint32_t kColS = kQSmem ? 0 : (KP * kQPiece + 63) / 64 * 64;  // + buffer * 64
  static constexpr uint32_t kColO = kColS + 64 * kSBufs;
  static_assert(kColO + D <= kTmemCols, "tensor memory columns");
};

template <int D, int IN>
struct Smem {
  using C = Cfg<D, IN>;
  static constexpr int KS = C::kKStages, VS = C::kVStages, SB = C::kSBufs;
  static constexpr int kB = 2 * KS + 2 * VS;  // first barrier after the rings
  uint8_t* base;
  uint32_t sQ, sK, sV, bar0;
  // K unit u (counted over the CTA's key tiles) in K slot u % KS, V unit u in V slot u % VS
  __device__ uint32_t k_full(int s) const { return bar0 + 8u * s; }
  __device__ uint32_t k_empty(int s) const { return bar0 + 8u * (KS + s); }
  __device__ uint32_t v_full(int s) const { return bar0 + 8u * (2 * KS + s); }
  __device__ uint32_t v_empty(int s) const { return bar0 + 8u * (2 * KS + VS + s); }
  __device__ uint32_t q_full() const { return bar0 + 8u * kB; }
  __device__ uint32_t q_empty() const { return bar0 + 8u * (kB + 1); }
  // per S buffer b: the scores of its next tile are in (s_full), its P is
  // written (p_full, 4 arrivals).  A buffer's next scores wait for the P.V of
  // its previous P, so neither barrier can run two phases ahead of its waiter.
  __device__ uint32_t s_full(int b) const { return bar0 + 8u * (kB + 2 + b); }
  __device__ uint32_t p_full(int b) const { return bar0 + 8u * (kB + 2 + SB + b); }
  // (two issuers) the P.V products of buffer b's P finished: its next S may go in
  __device__ uint32_t s_free(int b) const { return bar0 + 8u * (kB + 2 + 2 * SB + b); }
  // one completion per P.V (the softmax waits on it only before rescaling O)
  __device__ uint32_t pv_done() const { return bar0 + 8u * (kB + 2 + 3 * SB); }
  __device__ uint32_t o_final() const { return bar0 + 8u * (kB + 3 + 3 * SB); }
  __device__ uint32_t drain() const { return bar0 + 8u * (kB + 4 + 3 * SB); }
  __device__ uint8_t* mask_buf(int warp) const { return base + C::kOffMaskBuf + warp * C::kMaskBufBytes; }
};

// ------------------------------------------------------------------ pieces
// bf16 pieces of fp32 values; each subtraction is exact in fp32.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xffff0000u); }

__device__ __forceinline__ uint32_t bf16_pair(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// (a, b) -> n pieces, each a packed bf16 pair (first value in the low half,
// as the MMA's K order wants).
template <int N>
__device__ __forceinline__ void split_pair(float a, float b, uint32_t (&out)[N]) {
#pragma unroll
  for (int k = 0; k < N; ++k) {
    out[k] = bf16_pair(a, b);
    if (k + 1 < N) {
      // (a, b) - piece, two lanes in one packed FMA
      f2_split(ffma2(f2(bf16_lo(out[k]), bf16_hi(out[k])), f2(-1.0f, -1.0f), f2(a, b)), a, b);
    }
  }
}

// A pair of fp32 values rounded to the 16-bit type, packed (first value low).
template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// ------------------------------------------------------------------ work items
// One 128-row query tile of one (b, h) and the 64-key tiles [tb, tb + N) its
// rows can see.
struct FItem {
  int b, h, kvh;
  int64_t q0;
  BatchLimits L;
  TileRange T;
  int tb, N;
};

// Latest query tiles (longest causal rows) first; the heads of one kv group
// are consecutive items, so their K / V tiles come from L2.  FN: keys per tile.
template <int FN>
__device__ __forceinline__ FItem make_fitem(const CommonParams& p, int idx) {
  const int bh = p.B * p.Hq;
  const int nqt = (p.Sq + FM - 1) / FM;
  FItem it;
  const int qt = nqt - 1 - idx / bh;
  const int rem = idx - (idx / bh) * bh;
  it.b = rem / p.Hq;
  it.h = rem - it.b * p.Hq;
  it.kvh = it.h / p.group;
  it.q0 = (int64_t)qt * FM;
  it.L = batch_limits(p, it.b);
  it.T = tile_range(p, it.L, it.q0, FM, FN);
  it.tb = it.T.t_begin;
  it.N = it.T.t_end - it.T.t_begin;
  return it;
}

// Static snake schedule over the persistent CTAs.
__device__ __forceinline__ int f_item_of_round(int r, int n_items) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const int idx = r * G + ((r & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

// ------------------------------------------------------------------ producer
// One thread.  Per key tile: its K units into the K ring (k_full) and its V
// units into the V ring (v_full).  A K unit is freed by its QK^T products, a
// V unit by its P.V products; since P.V runs about a tile after QK^T, V is
// loaded one tile behind K, so a wait for a V slot never holds back the next
// K.  At each item start it also prefetches the item's Q rows into L2, so
// the softmax warps' Q loads come from L2 (at D = 384 it loads Q into shared
// memory instead).  K / V tiles are read by every query tile of their kv
// head, Q and O once: K / V are loaded as L2 evict_last, and the softmax
// warps read Q and write O as evict_first, so a Q / O stream larger than L2
// does not push K / V out between the query tiles that share them (the
// prefetch keeps the default policy: an evict_first prefetch measured a few
// MB more DRAM reads).
template <int D, int IN>
__device__ __forceinline__ void f_producer(const LaneParams& P, const Smem<D, IN>& sm, int n_items) {
  using C = Cfg<D, IN>;
  constexpr int KP = C::KP, VP = C::VP;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  constexpr int FN = C::FN;
  const CommonParams& p = P.c;
  const int kvp = p.B * p.Hkv;  // planes per piece
  int g = 0;
  int q_items = 0;  // items whose Q was loaded into shared memory (kQSmem)
  const uint64_t keep = l2_evict_last_policy(), stream = l2_evict_first_policy();
  int k_issued = 0, v_issued = 0;  // units whose K / V copies were started
  // fp32: K / V pieces come from the pre-pass grid; wait until it finished
  // (its writes are then visible).  Everything before this point, and Q,
  // is independent of it.
  if constexpr (IN == kInF32Split) asm volatile("griddepcontrol.wait;" ::: "memory");
  // K unit c of key tile gt (key0, kv plane) into K slot (gt kKUnits + c) % KS
  auto load_k = [&](int gt, int c, int key0, int kv_plane) -> bool {
    const int gu = gt * C::kKUnits + c, ks = gu % KS;
    if (gu >= KS && !mbar_wait(sm.k_empty(ks), ((gu / KS) - 1) & 1, p.timeout_ns, p.status)) return false;
    mbar_arrive_expect_tx(sm.k_full(ks), C::kKUnitBytes);
    ++k_issued;
    const uint32_t dst = sm.sK + ks * C::kKUnitBytes;
    if constexpr (C::kKUnits == 1) {
      for (int pc = 0; pc < KP; ++pc)
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(dst + pc * C::kPieceBytes + s * C::kSubBytes, &P.tmap_k, sm.k_full(ks), s * 64, key0,
                           pc * kvp + kv_plane, keep);
    } else {
      // dims [128 c, 128 c + 128): two 64-column blocks
      for (int s = 0; s < 2; ++s)
        tma_load_3d_hint(dst + s * C::kSubBytes, &P.tmap_k, sm.k_full(ks), (2 * c + s) * 64, key0, kv_plane, keep);
    }
    return true;
  };
  // V unit u of key tile gt into V slot (gt kVUnits + u) % VS
  auto load_v = [&](int gt, int u, int key0, int kv_plane) -> bool {
    const int gu = gt * C::kVUnits + u, vs = gu % VS;
    if (gu >= VS && !mbar_wait(sm.v_empty(vs), ((gu / VS) - 1) & 1, p.timeout_ns, p.status)) return false;
    mbar_arrive_expect_tx(sm.v_full(vs), C::kVUnitBytes);
    ++v_issued;
    const uint32_t dst = sm.sV + vs * C::kVUnitBytes;
    if constexpr (C::kVUnits == 1) {
      for (int pc = 0; pc < VP; ++pc)
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(dst + pc * C::kPieceBytes + s * C::kSubBytes, &P.tmap_v, sm.v_full(vs), s * 64, key0,
                           P.v_plane0 + pc * kvp + kv_plane, keep);
    } else {
      // keys [key0 + 16 u, + 16): kSub [16 rows][64 cols] blocks
      for (int s = 0; s < C::kSub; ++s)
        tma_load_3d_hint(dst + s * C::kVUnitSubBytes, &P.tmap_v, sm.v_full(vs), s * 64, key0 + 16 * u, kv_plane,
                         keep);
    }
    return true;
  };
  // V of tile g - 1, not yet loaded: key0 and plane, or vplane < 0
  int vkey0 = 0, vplane = -1;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = f_item_of_round(r, n_items);
    if (idx < 0) break;
    const FItem it = make_fitem<C::FN>(p, idx);
    if (it.N == 0) continue;
    if constexpr (C::kQSmem) {
      // Q into shared memory once the previous item's QK^T products are done
      if (q_items > 0 && !mbar_wait(sm.q_empty(), (q_items - 1) & 1, p.timeout_ns, p.status)) break;
      mbar_arrive_expect_tx(sm.q_full(), C::kQBytes);
      for (int s = 0; s < C::kSub; ++s)
        tma_load_3d_hint(sm.sQ + s * C::kQSubBytes, &P.tmap_q, sm.q_full(), s * 64, (int)it.q0,
                         it.b * p.Hq + it.h, stream);
      ++q_items;
    } else {
      const int64_t rows = (int64_t)p.Sq - it.q0 < FM ? (int64_t)p.Sq - it.q0 : FM;
      constexpr int kQElem = IN == kInF32Split ? 4 : 2;  // bytes per Q element
      const uint8_t* qsrc = static_cast<const uint8_t*>(P.q) + (((int64_t)it.b * p.Hq + it.h) * p.Sq + it.q0) * D * kQElem;
      bulk_prefetch_l2(qsrc, (uint32_t)(rows * D * kQElem));
    }
    const int kv_plane = it.b * p.Hkv + it.kvh;
    for (int n = 0; n < it.N; ++n, ++g) {
      const int key0 = (it.tb + n) * FN;
      for (int c = 0; c < C::kKUnits && ok; ++c) ok = load_k(g, c, key0, kv_plane);
      for (int u = 0; u < C::kVUnits && ok && vplane >= 0; ++u) ok = load_v(g - 1, u, vkey0, vplane);
      if (!ok) break;
      vkey0 = key0;
      vplane = kv_plane;
    }
  }
  for (int u = 0; u < C::kVUnits && ok && vplane >= 0; ++u) ok = load_v(g - 1, u, vkey0, vplane);
  // Let every copy this thread started land before the CTA can exit.
  for (int n = (k_issued > KS ? k_issued - KS : 0); n < k_issued; ++n)
    mbar_wait(sm.k_full(n % KS), (n / KS) & 1, p.timeout_ns, p.status);
  for (int n = (v_issued > VS ? v_issued - VS : 0); n < v_issued; ++n)
    mbar_wait(sm.v_full(n % VS), (n / VS) & 1, p.timeout_ns, p.status);
  if (C::kQSmem && q_items > 0) mbar_wait(sm.q_full(), (q_items - 1) & 1, p.timeout_ns, p.status);
}

// ------------------------------------------------------------------ MMA issuers
// Two warps issue: ROLE 1 the scores S = Q K^T of every key tile, ROLE 2 the
// products O += P V, both on the CTA's running key tile count g, tile g in S
// buffer g % SB.  The whole warp runs this; elect.sync picks the issuing lane.
// An issuing warp is held until only a few MMAs are queued, so a single
// issuer's barrier waits would each leave the tensor core idle for most of
// their duration; with two, one issuer's MMAs keep the queue busy while the
// other waits.  The scores of tile g go into the buffer of tile g - SB's P,
// so they wait until that tile's P.V products finished (s_free).
// For inputs read straight from the caller's cache (16-bit), V rows at or
// past the valid length may hold any bits (NaN / Inf included): P is 0 there
// but 0 * NaN is not, so those rows are zeroed in shared memory before the
// P.V products read them.
template <int D, int IN, int ROLE>
__device__ __forceinline__ void f_mma(const LaneParams& P, const Smem<D, IN>& sm, uint32_t tmem, int n_items,
                                      int lane) {
  using C = Cfg<D, IN>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  constexpr int KP = C::KP, VP = C::VP;
  constexpr bool kBF16 = In<IN>::kBF16;
  constexpr int FN = C::FN;
  constexpr int SB = C::kSBufs;
  constexpr bool kQK = ROLE == 1, kPV = ROLE == 2;
  static_assert(ROLE == 1 || ROLE == 2, "issuer roles");
  constexpr uint32_t id_qk = make_idesc_f16kind(kBF16, FM, FN, false);
  // one MMA's N is at most 256: D = 384 runs as N = 256 and N = 128 parts
  constexpr int kN0 = D > 256 ? 256 : D;
  constexpr uint32_t id_pv = make_idesc_f16kind(kBF16, FM, kN0, true);
  constexpr uint32_t id_pv1 = make_idesc_f16kind(kBF16, FM, D > 256 ? D - 256 : 64, true);
  const CommonParams& p = P.c;
  int g0 = 0;          // ring position of the item's first key tile
  int q_items = 0;     // items whose Q was consumed
  int pb[3] = {0, 0, 0};  // P tiles consumed per S buffer (all items)
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = f_item_of_round(r, n_items);
    if (idx < 0) break;
    const FItem it = make_fitem<C::FN>(p, idx);
    if (it.N == 0) continue;
    if constexpr (kQK) {
      if (!mbar_wait_warp(sm.q_full(), q_items & 1, p.timeout_ns, p.status)) break;
      ++q_items;
      tc_fence_after();
    }
    int64_t zero_from = it.L.lsk < (int64_t)p.Sk ? it.L.lsk : (int64_t)p.Sk;
    if (zero_from < 0) zero_from = 0;
    for (int n = 0; ok && n <= it.N; ++n) {
      if (kQK && n < it.N) {
        // S = Q K_n^T (pieces: q0k0 + q0k1 + q1k0 + q0k2 + q1k1 + q2k0)
        const int gs = g0 + n;
        const int bs = gs % SB;
        // Of the two waits before a tile's first products, the one measured
        // to complete later goes last, so the products follow it at once:
        // the buffer (s_free) with two S buffers, K with three.
        auto wait_buffer = [&]() -> bool {
          return gs < SB || mbar_wait_warp(sm.s_free(bs), ((gs / SB) - 1) & 1, p.timeout_ns, p.status);
        };
        if (SB == 3 && !wait_buffer()) { ok = false; break; }
        const uint32_t sd = tmem + C::kColS + 64 * bs;
        if constexpr (C::kKUnits == 1) {
          const int ks = gs % KS;
          if (!mbar_wait_warp(sm.k_full(ks), (gs / KS) & 1, p.timeout_ns, p.status)) { ok = false; break; }
          if (SB != 3 && !wait_buffer()) { ok = false; break; }
          tc_fence_after();
          const uint32_t kb = sm.sK + ks * C::kKUnitBytes;
          if constexpr (KP == 3) {
            uint64_t kd[3];
#pragma unroll
            for (int pc = 0; pc < 3; ++pc) kd[pc] = make_sdesc_sw128(kb + pc * C::kPieceBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              // K step kk: 32 bytes into a 128-byte row, 64-column blocks kSubBytes apart
              const uint32_t off16 = ((kk >> 2) * C::kSubBytes + (kk & 3) * 32) >> 4;
              const uint32_t q0 = tmem + C::kColQ + kk * 8, q1 = q0 + C::kQPiece, q2 = q0 + 2 * C::kQPiece;
              mma_ts6_elect(sd, q0, kd[0] + off16, q0, kd[1] + off16, q1, kd[0] + off16, q0, kd[2] + off16,
                            q1, kd[1] + off16, q2, kd[0] + off16, id_qk, kk > 0 ? 1u : 0u);
            }
          } else {
            const uint64_t kd = make_sdesc_sw128(kb, 16, 1024);
            // K steps 4s..4s+3 lie in 64-column block s
#pragma unroll
            for (int s = 0; s < D / 64; ++s) {
              const uint32_t o = (s * C::kSubBytes) >> 4;
              const uint32_t q = tmem + C::kColQ + s * 32;
              mma_ts4_elect(sd, q, kd + o, q + 8, kd + o + 2, q + 16, kd + o + 4, q + 24, kd + o + 6, id_qk,
                            s > 0 ? 1u : 0u);
            }
          }
          tc_commit_elect(sm.k_empty(ks));
        } else {
          // D = 384: Q and K both K-major in shared memory.  K unit c holds
          // dims [128 c, 128 c + 128) as two 64-column blocks (kSubBytes
          // apart); Q's 64-column blocks are kQSubBytes apart.  Each unit is
          // freed as soon as its products finish.
          const uint64_t qd = make_sdesc_sw128(sm.sQ, 16, 1024);
#pragma unroll
          for (int c = 0; c < C::kKUnits; ++c) {
            const int gu = gs * C::kKUnits + c, ks = gu % KS;
            if (!mbar_wait_warp(sm.k_full(ks), (gu / KS) & 1, p.timeout_ns, p.status)) { ok = false; break; }
            if (SB != 3 && c == 0 && !wait_buffer()) { ok = false; break; }
            tc_fence_after();
            const uint64_t kd = make_sdesc_sw128(sm.sK + ks * C::kKUnitBytes, 16, 1024);
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              const uint32_t oq = ((2 * c + s) * C::kQSubBytes) >> 4, okk = (s * C::kSubBytes) >> 4;
              mma_ss4_elect(sd, qd + oq, kd + okk, qd + oq + 2, kd + okk + 2, qd + oq + 4, kd + okk + 4,
                            qd + oq + 6, kd + okk + 6, id_qk, (c > 0 || s > 0) ? 1u : 0u);
            }
            tc_commit_elect(sm.k_empty(ks));
          }
          if (!ok) break;
        }
        tc_commit_elect(sm.s_full(bs));
        // the item's last QK^T products are issued: Q may be replaced once they finish
        if (n == it.N - 1) tc_commit_elect(sm.q_empty());
      }
      if (kPV && n >= 1) {
        // O (+)= P_{n-1} V_{n-1} (pieces: p0 v0 + p0 v1 + p1 v0), V unit by unit
        const int m = n - 1;
        const int gv = g0 + m;
        const int bp = gv % SB;
        const uint32_t pa = tmem + C::kColS + 64 * bp;  // P piece t over 32 columns from pa + 32 t
        // P and the first V unit, the one measured to complete later last:
        // V with the fp32 pieces (three S buffers), P otherwise
        auto wait_p = [&]() -> bool {
          if (!mbar_wait_warp(sm.p_full(bp), pb[bp] & 1, p.timeout_ns, p.status)) return false;
          ++pb[bp];
          return true;
        };
        if (SB == 3 && !wait_p()) { ok = false; break; }
        constexpr int kUKeys = FN / C::kVUnits;          // keys per V unit
        const int64_t key0 = (int64_t)(it.tb + m) * FN;
#pragma unroll
        for (int u = 0; u < C::kVUnits; ++u) {
          const int gu = gv * C::kVUnits + u, vs = gu % VS;
          if (!mbar_wait_warp(sm.v_full(vs), (gu / VS) & 1, p.timeout_ns, p.status)) { ok = false; break; }
          if (SB != 3 && u == 0 && !wait_p()) { ok = false; break; }
          const uint32_t vb = sm.sV + vs * C::kVUnitBytes;
          if constexpr (IN != kInF32Split) {
            const int64_t ukey0 = key0 + u * kUKeys;
            if (zero_from < ukey0 + kUKeys && zero_from < (int64_t)p.kv_capacity) {
              const int r0 = zero_from > ukey0 ? (int)(zero_from - ukey0) : 0;
              const int chunks = (kUKeys - r0) * 8;  // 16-byte chunks of whole 128-byte rows
              for (int s = 0; s < C::kSub; ++s) {
                uint8_t* blk = sm.base + C::kOffV + vs * C::kVUnitBytes + s * C::kVUnitSubBytes;
                for (int c = lane; c < chunks; c += 32)
                  *reinterpret_cast<uint4*>(blk + (size_t)(r0 + (c >> 3)) * 128 + (c & 7) * 16) =
                      make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
          }
          tc_fence_after();
          // B = V[keys 16kk.., 0..D): MN-major; 8-key groups 1024 B apart,
          // 64-column blocks kVUnitSubBytes apart
          const uint64_t d0 = make_sdesc_sw128(vb, C::kVUnitSubBytes, 1024);
          if constexpr (VP == 2) {
            const uint64_t d1 = make_sdesc_sw128(vb + C::kPieceBytes, C::kSubBytes, 1024);
            // two K steps (16 keys each, 2048 bytes of V apart) per issue block
#pragma unroll
            for (int kk = 0; kk < FN / 16; kk += 2) {
              const uint32_t o0 = (uint32_t)(kk * 2048) >> 4, o1 = (uint32_t)((kk + 1) * 2048) >> 4;
              mma_ts6_elect(tmem + C::kColO, pa + kk * 8, d0 + o0, pa + kk * 8, d1 + o0, pa + 32 + kk * 8, d0 + o0,
                            pa + (kk + 1) * 8, d0 + o1, pa + (kk + 1) * 8, d1 + o1, pa + 32 + (kk + 1) * 8,
                            d0 + o1, id_pv, (m == 0 && kk == 0) ? 0u : 1u);
            }
          } else if constexpr (D > 256) {
            // one K step (16 keys): columns [0, 256) from V blocks 0-3 (N = 256),
            // [256, D) from blocks 4.. into O + 256
            const uint64_t d1 = make_sdesc_sw128(vb + 4 * C::kVUnitSubBytes, C::kVUnitSubBytes, 1024);
            const uint32_t acc = (m == 0 && u == 0) ? 0u : 1u;
            mma_ts_elect(tmem + C::kColO, pa + 8 * u, d0, id_pv, acc);
            mma_ts_elect(tmem + C::kColO + 256, pa + 8 * u, d1, id_pv1, acc);
          } else {
            static_assert(FN == 64, "four K steps per key tile");
            mma_ts4_elect(tmem + C::kColO, pa, d0, pa + 8, d0 + 128, pa + 16, d0 + 256, pa + 24, d0 + 384, id_pv,
                          m == 0 ? 0u : 1u);
          }
          tc_commit_elect(sm.v_empty(vs));
        }
        if (!ok) break;
        tc_commit_elect(sm.s_free(bp));
        tc_commit_elect(sm.pv_done());
        if (m == it.N - 1) tc_commit_elect(sm.o_final());  // the item's last P.V
      }
    }
    if (!ok) break;
    g0 += it.N;
  }
  // Wait for every MMA this warp issued before tensor memory is freed.
  tc_commit_elect(sm.drain());
  mbar_wait_warp(sm.drain(), 0, p.timeout_ns, p.status);
}

// ------------------------------------------------------------------ softmax
// Maximum / minimum of N values (N a multiple of 16) in eight chains.
template <int N>
__device__ __forceinline__ float maxn(const float (&x)[N]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(x[k], x[k + 8]);
#pragma unroll
  for (int i = 16; i < N; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmax3(m[k], x[i + k], x[i + 8 + k]);
  return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], fmax3(m[5], m[6], m[7])));
}

template <int N>
__device__ __forceinline__ float minn(const float (&x)[N]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fminf(x[k], x[k + 8]);
#pragma unroll
  for (int i = 16; i < N; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmin3(m[k], x[i + k], x[i + 8 + k]);
  return fminf(fmin3(m[0], m[1], m[2]), fmin3(m[3], m[4], fmin3(m[5], m[6], m[7])));
}

// Rows of a warp move between global memory and the threads that own them
// (thread = row) through the warp's staging buffer, 32 columns at a time:
// each global load or store instruction then covers whole 32-column row
// segments of several rows (128 bytes of fp32 or 64 of 16-bit per row)
// instead of one 16-byte piece of 32 rows.  Segment chunks are XOR-swizzled
// by row, so both the row-wise and the lane-per-row accesses are free of
// bank conflicts.
template <int ES>
struct RowStage {
  static constexpr int kSegBytes = 32 * ES;      // one row's 32 columns
  static constexpr int kCps = kSegBytes / 16;    // 16-byte chunks per segment
  static constexpr int kRpi = 32 / kCps;         // rows per instruction
  static constexpr int kInstr = 32 / kRpi;       // instructions per 32 rows
  __device__ static int swz(int r) { return kCps == 8 ? (r & 7) : ((r >> 1) & 3); }
  __device__ static uint32_t at(int r, int c) { return (uint32_t)(r * kSegBytes + ((c ^ swz(r)) << 4)); }
};

// This thread's Q row in tensor memory: piece t over columns [t D/2,
// (t+1) D/2), column c holding d = 2c, 2c + 1.  fp32 rows are split into KP
// bf16 pieces; 16-bit rows are stored as they are.  The warp's 32 rows are
// read with coalesced loads (all in flight at once) and handed to their
// threads through `buf` (at least 32 rows x 32 columns).
template <int D, int IN>
__device__ __forceinline__ void store_q_row(const CommonParams& p, const void* q, const FItem& it, int warp,
                                            int lane, uint32_t tlane, uint8_t* buf) {
  using C = Cfg<D, IN>;
  constexpr int ES = IN == kInF32Split ? 4 : 2;
  using RS = RowStage<ES>;
  constexpr int kChunks = D / 32;
  const int rsub = lane / RS::kCps, csub = lane % RS::kCps;
  const int64_t qw0 = it.q0 + warp * 32;  // first row of the warp
  const uint8_t* base =
      static_cast<const uint8_t*>(q) + ((((int64_t)it.b * p.Hq + it.h) * p.Sq + qw0) * D) * ES + csub * 16;
  const uint64_t stream = l2_evict_first_policy();
  uint4 v[kChunks][RS::kInstr];
#pragma unroll
  for (int ch = 0; ch < kChunks; ++ch)
#pragma unroll
    for (int i = 0; i < RS::kInstr; ++i) {
      const int r = i * RS::kRpi + rsub;
      v[ch][i] = qw0 + r < p.Sq ? ld_nc_hint(base + (int64_t)r * D * ES + ch * RS::kSegBytes, stream)
                                : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
  for (int ch = 0; ch < kChunks; ++ch) {
#pragma unroll
    for (int i = 0; i < RS::kInstr; ++i)
      *reinterpret_cast<uint4*>(buf + RS::at(i * RS::kRpi + rsub, csub)) = v[ch][i];
    __syncwarp();
    uint4 mine[RS::kCps];
#pragma unroll
    for (int c = 0; c < RS::kCps; ++c) mine[c] = *reinterpret_cast<const uint4*>(buf + RS::at(lane, c));
    __syncwarp();
    if constexpr (IN == kInF32Split) {
      uint32_t pcs[C::KP][16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t a[C::KP], b[C::KP];
        split_pair<C::KP>(__uint_as_float(mine[i].x), __uint_as_float(mine[i].y), a);
        split_pair<C::KP>(__uint_as_float(mine[i].z), __uint_as_float(mine[i].w), b);
#pragma unroll
        for (int t = 0; t < C::KP; ++t) {
          pcs[t][2 * i] = a[t];
          pcs[t][2 * i + 1] = b[t];
        }
      }
#pragma unroll
      for (int t = 0; t < C::KP; ++t) tmem_st16(tlane + C::kColQ + t * C::kQPiece + ch * 16, pcs[t]);
    } else {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[4 * i] = mine[i].x;
        w[4 * i + 1] = mine[i].y;
        w[4 * i + 2] = mine[i].z;
        w[4 * i + 3] = mine[i].w;
      }
      tmem_st16(tlane + C::kColQ + ch * 16, w);
    }
  }
}

// Mask block of one warp -- 32 rows by the N keys [key0, key0 + N) -- into
// x of the lane that owns each row (natural units; 0 outside), KC keys (32
// or 16) at a time.  Each instruction loads rows of KC * 4 contiguous bytes
// (4 rows x 128 bytes, or 8 rows x 64 bytes); a per-warp
// buffer of 32 rows x KC keys (16-byte chunks XOR-swizzled by row so that
// both the row-wise stores and the lane-per-row reads are conflict-free)
// turns rows into lanes.  vec4 needs 16-byte aligned mask rows (Sk % 4 == 0).
template <int N, int KC>
__device__ __forceinline__ void mask_rows(float (&x)[N], const float* mwarp, int nrows, int Sk, int key0,
                                          bool vec4, uint8_t* buf, int lane) {
  static_assert(KC == 32 || KC == 16, "chunk of 32 or 16 keys");
  constexpr int kCpr = KC / 4;     // 16-byte chunks per buffered row
  constexpr int kRpi = 32 / kCpr;  // rows per load instruction
  constexpr int kRowBytes = KC * 4;
  const int rsub = lane / kCpr;
  const int csub = lane % kCpr;
  auto swz = [](int row) { return KC == 32 ? (row & 7) : ((row >> 1) & 3); };
#pragma unroll
  for (int k = 0; k < N / KC; ++k) {
    float4 v[32 / kRpi];
#pragma unroll
    for (int i = 0; i < 32 / kRpi; ++i) {
      const int row = kRpi * i + rsub;
      const int key = key0 + KC * k + 4 * csub;
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      const float* src = mwarp + (int64_t)row * Sk + key;
      if (vec4) {
        if (row < nrows && key + 3 < Sk) t = __ldg(reinterpret_cast<const float4*>(src));
      } else if (row < nrows) {
        if (key + 0 < Sk) t.x = __ldg(src + 0);
        if (key + 1 < Sk) t.y = __ldg(src + 1);
        if (key + 2 < Sk) t.z = __ldg(src + 2);
        if (key + 3 < Sk) t.w = __ldg(src + 3);
      }
      v[i] = t;
    }
#pragma unroll
    for (int i = 0; i < 32 / kRpi; ++i) {
      const int row = kRpi * i + rsub;
      *reinterpret_cast<float4*>(buf + row * kRowBytes + ((csub ^ swz(row)) << 4)) = v[i];
    }
    __syncwarp();
#pragma unroll
    for (int c = 0; c < kCpr; ++c) {
      const float4 t = *reinterpret_cast<const float4*>(buf + lane * kRowBytes + ((c ^ swz(lane)) << 4));
      x[KC * k + 4 * c + 0] = t.x;
      x[KC * k + 4 * c + 1] = t.y;
      x[KC * k + 4 * c + 2] = t.z;
      x[KC * k + 4 * c + 3] = t.w;
    }
    __syncwarp();
  }
}

// Warps 0-3: thread = one query row of the item.
template <int D, int IN, bool SOFTCAP, bool MASK>
__device__ __forceinline__ void f_softmax(const LaneParams& P, const Smem<D, IN>& sm, uint32_t tmem, int n_items,
                                          int warp, int lane) {
  using C = Cfg<D, IN>;
  constexpr bool kF32 = IN == kInF32Split;
  constexpr int FN = C::FN;
  const CommonParams& p = P.c;
  const int row = warp * 32 + lane;
  const uint32_t tlane = tmem + ((uint32_t)(warp * 32) << 16);
  const uint32_t o_addr = tlane + C::kColO;
  int sb[3] = {0, 0, 0};  // S tiles consumed per buffer (all items)
  int tiles = 0;       // key tiles consumed (all items): P.V completions to wait for
  int qn = 0;          // items whose Q was stored
  int on = 0;          // o_final completions
  // Q rows of the first item at or after round r0 that has keys, into tensor
  // memory once the QK^T products of the item before it have finished.  The
  // next item's Q goes in right after this item's last P, before its
  // epilogue, so the MMA warp starts the next item's QK^T while the
  // epilogue runs.  Warp-collective; false on a timeout.
  auto stage_q = [&](int r0) -> bool {
    for (int r2 = r0;; ++r2) {
      const int idx2 = f_item_of_round(r2, n_items);
      if (idx2 < 0) return true;
      const FItem it2 = make_fitem<C::FN>(p, idx2);
      if (it2.N == 0) continue;
      if (qn > 0 && !mbar_wait_warp(sm.q_empty(), (qn - 1) & 1, p.timeout_ns, p.status)) return false;
      ++qn;
      store_q_row<D, IN>(p, P.q, it2, warp, lane, tlane, sm.mask_buf(warp));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.q_full());
      return true;
    }
  };
  bool ok = true;
  if constexpr (!C::kQSmem) ok = stage_q(0);
  for (int r = 0; ok; ++r) {
    const int idx = f_item_of_round(r, n_items);
    if (idx < 0) break;
    const FItem it = make_fitem<C::FN>(p, idx);
    const int64_t qi = it.q0 + row;
    const int64_t row_id = ((int64_t)it.b * p.Hq + it.h) * p.Sq + qi;
    const int64_t obase = p.out_layout == 0 ? row_id * D : (((int64_t)it.b * p.Sq + qi) * p.Hq + it.h) * D;
    // the output row as 16-byte units: 4 fp32 or 8 16-bit values each
    uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + obase * (kF32 ? 4 : 2));
    if (it.N == 0) {
      // no visible key for any row of the tile: the rows are 0
      if (qi < p.Sq) {
#pragma unroll 4
        for (int i = 0; i < D / (kF32 ? 4 : 8); ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      continue;
    }

    const RowLimits R = row_limits(p, it.L, qi);
    const float* mwarp = nullptr;
    int mrows = 0;
    if constexpr (MASK) {
      int64_t plane = 0;
      if (p.mask_planes == p.B) plane = it.b;
      else if (p.mask_planes == p.B * p.Hq) plane = (int64_t)it.b * p.Hq + it.h;
      const int64_t qw0 = qi - lane;
      mwarp = p.mask + (plane * p.Sq + (qw0 < p.Sq ? qw0 : 0)) * (int64_t)p.Sk;
      mrows = qw0 < p.Sq ? (int)min((int64_t)32, (int64_t)p.Sq - qw0) : 0;
    }
    const float xs = SOFTCAP ? p.sc_out : p.scale_log2;  // brings a raw x to log2 units
    float m_run = -INFINITY;  // running max, log2 units
    float l_run = 0.0f;
    for (int n = 0; n < it.N; ++n, ++tiles) {
      // the MMA warps' buffer order: the running key tile count
      const int bsel = tiles % C::kSBufs;
      const uint32_t s_addr = tlane + C::kColS + 64 * bsel;
      const int64_t key0 = (int64_t)(it.tb + n) * FN;
      float x[FN];
      if constexpr (MASK)
        mask_rows<FN, C::kMaskKeys>(x, mwarp, mrows, p.Sk, (int)key0, p.mask_vec4 != 0, sm.mask_buf(warp), lane);
      if (!mbar_wait_warp(sm.s_full(bsel), sb[bsel] & 1, p.timeout_ns, p.status)) { ok = false; break; }
      ++sb[bsel];
      tc_fence_after();
      const bool need_mask = !(key0 >= it.T.full_lo && key0 + FN <= it.T.full_hi);
      bool scaled = false;
      {
        uint32_t sr[FN / 32][32];
#pragma unroll
        for (int k = 0; k < FN / 32; ++k) tmem_ld32(s_addr + 32 * k, sr[k]);
        tmem_wait_ld();
        if constexpr (MASK) {
          const uint64_t le2 = f2(kLog2e, kLog2e);
          if constexpr (SOFTCAP) {
            const uint64_t in2 = f2(p.sc_in, p.sc_in), out2 = f2(p.sc_out, p.sc_out);
#pragma unroll
            for (int i = 0; i < FN; i += 2) {
              float a0, a1;
              f2_split(fmul2(f2(__uint_as_float(sr[i >> 5][i & 31]), __uint_as_float(sr[i >> 5][(i & 31) + 1])), in2),
                       a0, a1);
              f2_split(ffma2(f2(fast_tanh(a0), fast_tanh(a1)), out2, fmul2(f2(x[i], x[i + 1]), le2)), x[i], x[i + 1]);
            }
          } else {
            const uint64_t sc2 = f2(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int i = 0; i < FN; i += 2) {
              const uint64_t sv =
                  fmul2(f2(__uint_as_float(sr[i >> 5][i & 31]), __uint_as_float(sr[i >> 5][(i & 31) + 1])), sc2);
              f2_split(ffma2(f2(x[i], x[i + 1]), le2, sv), x[i], x[i + 1]);
            }
          }
          scaled = true;
        } else if constexpr (SOFTCAP) {
          const uint64_t in2 = f2(p.sc_in, p.sc_in);
#pragma unroll
          for (int i = 0; i < FN; i += 2) {
            float a0, a1;
            f2_split(fmul2(f2(__uint_as_float(sr[i >> 5][i & 31]), __uint_as_float(sr[i >> 5][(i & 31) + 1])), in2),
                     a0, a1);
            x[i] = fast_tanh(a0);
            x[i + 1] = fast_tanh(a1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < FN; ++i) x[i] = __uint_as_float(sr[i >> 5][i & 31]);
        }
      }
      if (need_mask) {
        // structural limits of this row: keys outside [lo, hi) become -inf
        if (!scaled && !(xs > 0.0f)) {
#pragma unroll
          for (int i = 0; i < FN; ++i) x[i] *= xs;
          scaled = true;
        }
        int lo = R.lo - (int)key0, hi = R.hi - (int)key0;
        lo = lo < 0 ? 0 : (lo > FN ? FN : lo);
        hi = hi < 0 ? 0 : (hi > FN ? FN : hi);
        const uint32_t span = hi > lo ? (uint32_t)(hi - lo) : 0u;
#pragma unroll
        for (int i = 0; i < FN; ++i) x[i] = ((uint32_t)(i - lo) < span) ? x[i] : -INFINITY;
      }
      float m_tile;
      if (scaled) {
        m_tile = maxn<FN>(x);
      } else if (!need_mask) {
        m_tile = (xs >= 0.0f ? maxn<FN>(x) : minn<FN>(x)) * xs;
      } else {
        const float mr = maxn<FN>(x);
        m_tile = mr == -INFINITY ? -INFINITY : mr * xs;
      }
      // online update, keeping the old max unless it grew by more than 2^8
      const float m_new = fmaxf(m_run, m_tile);
      float alpha = 1.0f;
      bool rescale = false;
      float m_use = m_run;
      if (m_run == -INFINITY) {
        m_use = m_new;
      } else if (m_new - m_run > kRescaleLog2) {
        m_use = m_new;
        alpha = fast_exp2(m_run - m_new);
        rescale = true;
      }
      const float m_sub = (m_use == -INFINITY) ? 0.0f : m_use;
      const float xmul = scaled ? 1.0f : xs;
      const uint64_t mul2 = f2(xmul, xmul), sub2 = f2(-m_sub, -m_sub);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
      // P = 2^(x - m) over this row's S columns, 16 columns per store: for
      // fp32 two bf16 pieces (p0 in columns [0, 32), p1 in [32, 64)), else
      // rounded to the input type (columns [0, 32))
#pragma unroll
      for (int ch = 0; ch < FN / 32; ++ch) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a0, a1;
          f2_split(ffma2(f2(x[ch * 32 + 2 * i], x[ch * 32 + 2 * i + 1]), mul2, sub2), a0, a1);
          const float e0 = fast_exp2(a0), e1 = fast_exp2(a1);
          acc[i & 3] = fadd2(acc[i & 3], f2(e0, e1));
          if constexpr (C::VP == 2) {
            uint32_t pc[2];
            split_pair<2>(e0, e1, pc);
            ph[i] = pc[0];
            pl[i] = pc[1];
          } else {
            ph[i] = pack16<In<IN>::kBF16>(e0, e1);
          }
        }
        tmem_st16(s_addr + ch * 16, ph);
        if constexpr (C::VP == 2) tmem_st16(s_addr + 32 + ch * 16, pl);
      }
      float sum, sum_hi;
      f2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), sum, sum_hi);
      l_run = l_run * alpha + sum + sum_hi;
      m_run = m_use;
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold every earlier P.V of the item first: wait for the P.V of
        // the previous key tile (the tiles - 1 -th completion of pv_done)
        if (!mbar_wait_warp(sm.pv_done(), (tiles - 1) & 1, p.timeout_ns, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          uint32_t o[32];
          tmem_ld32(o_addr + k * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float u0, u1;
            f2_split(fmul2(f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), u0, u1);
            o[i] = __float_as_uint(u0);
            o[i + 1] = __float_as_uint(u1);
          }
          tmem_st32(o_addr + k * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full(bsel));
    }
    if (!ok) break;
    if constexpr (!C::kQSmem) {
      if (!stage_q(r + 1)) { ok = false; break; }
    }

    // ------------------------------------------------------------ epilogue
    if (!mbar_wait_warp(sm.o_final(), on & 1, p.timeout_ns, p.status)) { ok = false; break; }
    ++on;
    tc_fence_after();
    const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    // O is written once: evict_first, so it does not displace K / V in L2
    const uint64_t o_policy = l2_evict_first_policy();
    const uint64_t w2 = f2(inv_l, inv_l);
    {
      // through the staging buffer: coalesced row segments (see RowStage)
      using RS = RowStage<kF32 ? 4 : 2>;
      uint8_t* buf = sm.mask_buf(warp);
      const int rsub = lane / RS::kCps, csub = lane % RS::kCps;
      const int64_t qw0 = it.q0 + warp * 32;
      uint8_t* odst[RS::kInstr];
#pragma unroll
      for (int i = 0; i < RS::kInstr; ++i) {
        const int64_t qr = qw0 + i * RS::kRpi + rsub;
        const int64_t e = p.out_layout == 0 ? (((int64_t)it.b * p.Hq + it.h) * p.Sq + qr) * D
                                            : (((int64_t)it.b * p.Sq + qr) * p.Hq + it.h) * D;
        odst[i] = qr < p.Sq ? static_cast<uint8_t*>(p.out) + e * (kF32 ? 4 : 2) + csub * 16 : nullptr;
      }
      // the next 32 columns' tensor-memory load is in flight while these
      // are converted and stored (tcgen05.wait::ld waits for every earlier
      // load, so the load of chunk k + 1 is issued right after the wait for k)
      uint32_t ob[2][32];
      tmem_ld32(o_addr, ob[0]);
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        tmem_wait_ld();
        if (k + 1 < D / 32) tmem_ld32(o_addr + (k + 1) * 32, ob[(k + 1) & 1]);
        const uint32_t(&o)[32] = ob[k & 1];
        float r[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          f2_split(fmul2(f2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), w2), r[i], r[i + 1]);
#pragma unroll
        for (int c = 0; c < RS::kCps; ++c) {
          uint4 u;
          if constexpr (kF32) {
            u = make_uint4(__float_as_uint(r[4 * c]), __float_as_uint(r[4 * c + 1]), __float_as_uint(r[4 * c + 2]),
                           __float_as_uint(r[4 * c + 3]));
          } else {
            u = make_uint4(pack16<In<IN>::kBF16>(r[8 * c], r[8 * c + 1]),
                           pack16<In<IN>::kBF16>(r[8 * c + 2], r[8 * c + 3]),
                           pack16<In<IN>::kBF16>(r[8 * c + 4], r[8 * c + 5]),
                           pack16<In<IN>::kBF16>(r[8 * c + 6], r[8 * c + 7]));
          }
          *reinterpret_cast<uint4*>(buf + RS::at(lane, c)) = u;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < RS::kInstr; ++i) {
          const uint4 u = *reinterpret_cast<const uint4*>(buf + RS::at(i * RS::kRpi + rsub, csub));
          if (odst[i]) st_hint(odst[i] + k * RS::kSegBytes, u, o_policy);
        }
        __syncwarp();
      }
    }
    // The next item's first P.V (which overwrites O) waits for this
    // warpgroup's next P, written after these reads (fence before arrive).
    tc_fence_before();
  }
}

// ------------------------------------------------------------------ kernel
template <int D, int IN, bool SOFTCAP, bool MASK>
__global__ void __launch_bounds__(Cfg<D, IN>::kThreads, 1) attn_fwd_lane1_kernel(const __grid_constant__ LaneParams P) {
  using C = Cfg<D, IN>;
  const CommonParams& p = P.c;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem<D, IN> sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm.base);
  sm.sQ = sbase + C::kOffQ;
  sm.sK = sbase + C::kOffK;
  sm.sV = sbase + C::kOffV;
  sm.bar0 = sbase + C::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.base + C::kOffSlot);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = ((p.Sq + FM - 1) / FM) * p.B * p.Hq;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(sm.k_full(s), 1);
      mbar_init(sm.k_empty(s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.v_empty(s), 1);
    }
    mbar_init(sm.q_full(), C::kQSmem ? 1 : 4);  // the producer's TMA, or one arrival per softmax warp
    mbar_init(sm.q_empty(), 1);
    for (int b = 0; b < C::kSBufs; ++b) {
      mbar_init(sm.s_full(b), 1);
      mbar_init(sm.p_full(b), 4);  // one arrival per softmax warp
      mbar_init(sm.s_free(b), 1);
    }
    mbar_init(sm.pv_done(), 1);
    mbar_init(sm.o_final(), 1);
    mbar_init(sm.drain(), 2);  // one commit per issuing warp
    mbar_init_fence();
  }
  if (warp == kTmaWarp && lane == 0) {
    if (C::kQSmem) tma_prefetch_desc(&P.tmap_q);
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
    if (lane == 0) f_producer<D, IN>(P, sm, n_items);
  } else if (warp == kMmaWarp) {
    f_mma<D, IN, 1>(P, sm, tmem, n_items, lane);
  } else if (warp == kPvWarp) {
    f_mma<D, IN, 2>(P, sm, tmem, n_items, lane);
  } else {
    f_softmax<D, IN, SOFTCAP, MASK>(P, sm, tmem, n_items, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int IN, bool SOFTCAP, bool MASK>
cudaError_t launch_lane1_variant(const LaneParams& P, cudaStream_t stream) {
  auto kernel = attn_fwd_lane1_kernel<D, IN, SOFTCAP, MASK>;
  constexpr uint32_t smem = Cfg<D, IN>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t n_items = (int64_t)((P.c.Sq + FM - 1) / FM) * P.c.B * P.c.Hq;
  if (n_items > INT32_MAX) return cudaErrorInvalidConfiguration;
  const int grid = (int)(n_items < sms ? n_items : sms);  // one persistent CTA per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(Cfg<D, IN>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // fp32: a programmatic dependent of the K / V pre-pass, so the prologue and
  // the first item's Q rows overlap its tail (the producer waits for it in
  // hardware before the first K / V load)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = IN == kInF32Split ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

// One head dim and input kind: the four soft-cap / mask variants.
template <int D, int IN>
cudaError_t launch_lane1(const LaneParams& P, cudaStream_t stream) {
  const bool sc = P.c.softcap > 0.0f;
  const bool mk = P.c.mask != nullptr && P.c.mask_planes > 0;
  if (sc && mk) return launch_lane1_variant<D, IN, true, true>(P, stream);
  if (sc) return launch_lane1_variant<D, IN, true, false>(P, stream);
  if (mk) return launch_lane1_variant<D, IN, false, true>(P, stream);
  return launch_lane1_variant<D, IN, false, false>(P, stream);
}

}  // namespace lane1
}  // namespace gb300_attn
