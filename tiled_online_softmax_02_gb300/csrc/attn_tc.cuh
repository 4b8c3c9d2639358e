#pragma once
// attn_tc.cuh -- tensor-core (tcgen05) attention forward for bf16 / f16 inputs
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
// Work item = two 128-row query tiles (t = 0, 1) of one (b, h).  The kernel is
// persistent: one CTA per SM walks a static snake order over the items
// (latest query rows -- the longest causal rows -- first), and the K/V ring,
// barrier phases and tensor memory carry over from item to item, so the next
// item's loads overlap the current item's tail.
//   warps 0-3   softmax for query tile 0, warps 4-7 for query tile 1: thread
//               r of a warpgroup owns query row r (= TMEM lane r).  Reads its
//               S row with tcgen05.ld, applies the structural masks (select to
//               -inf), soft-cap and additive mask, updates the running max /
//               sum in registers, writes P (input dtype) back over its S row,
//               and rescales its O row when the max grew by more than 2^8
//               (otherwise the old max is kept: the final O / l is exact
//               either way).  Then normalises and stores the row.
//   warp 8      TMA producer: both Q tiles per item, K_j / V_j into a ring.
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
// O_1 [384,512).  Shared memory: Q_0, Q_1, the K and V rings (2 + 2 stages
// at D = 128 with a mask, 2 + 3 without, 4 + 4 at D = 64), barriers and the
// per-warp mask buffers; every tile is stored as 64-column (128-byte) blocks
// in the 128-byte swizzle TMA writes.
//
// Every barrier wait is bounded (mbar_wait); on a timeout the kernel records
// ATTN_ERR_TIMEOUT in the status word, drains what it issued, frees tensor
// memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"

// Included by the attn_tc_<dtype>_d<D>.cu translation units; each
// instantiates launch_attn_tc_dd for one input type and head dim.
namespace gb300_attn {
namespace {

constexpr int BM = kTcBlockM;   // rows per query tile
constexpr int BN = kTcBlockN;   // keys per key tile
constexpr int kQTiles = 2;      // query tiles per work item
constexpr int kThreads = 320;   // 8 softmax warps + producer + MMA
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;  // keep the old max while it is within 2^8
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxOrderB = 64;   // batches ranked by cost when B <= this
constexpr uint32_t kMaskBufBytes = 32 * 32 * 4;  // per softmax warp: 32 rows x 32 keys of f32

// MB: the variant stages the mask through per-warp buffers.  Without a mask
// (MB false) that space holds a third V stage at D = 128, and K and V of key
// tile g complete one barrier (k_full of K's slot): the QK^T products of a
// tile already wait for it, so the MMA warp's wait before the P.V products
// of that tile, a step later, goes away (with three V stages V's load starts
// about two steps before its P.V, so a tile's barrier is not held back by
// its V).  With a mask, K and V keep their own barriers and two stages each.
template <int D, bool MB = true>
struct TcConfig {
  static constexpr int kSub = D / 64;                   // 128-byte column blocks per row
  static constexpr uint32_t kSubBytes = BM * 128;       // [128 rows][64 cols] of 16-bit
  static constexpr uint32_t kTileBytes = kSub * kSubBytes;
  static constexpr int kKStages = (D == 64) ? 4 : 2;
  static constexpr int kVStages = (D == 64) ? 4 : (MB ? 2 : 3);
  static constexpr bool kCombined = !MB;  // V(g) completes k_full(g % kKStages)
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQTiles * kTileBytes;
  static constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
  static constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
  // q_full, q_empty, k_full[SK], v_full[SV], k_empty[SK], v_empty[SV], s_full[2],
  // p_full[2], o_final[2], drain, merge_full, merge_done
  static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 3;
  static constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffMerge = kOffTmemSlot + 16;          // float2 [128] (key-split merge)
  static constexpr uint32_t kOffOrder = kOffMerge + BM * 8;         // int [kMaxOrderB] batch order
  static constexpr uint32_t kOffMaskBuf = (kOffOrder + kMaxOrderB * 4 + 127) / 128 * 128;
  static constexpr uint32_t kSmemBytes = kOffMaskBuf + (MB ? 8 * kMaskBufBytes : 0) + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Shared-memory addresses of the tiles and barriers.
template <int D, bool MB = true>
struct Smem {
  using Cfg = TcConfig<D, MB>;
  static constexpr int SK = Cfg::kKStages, SV = Cfg::kVStages;
  static constexpr int kR = 2 + 2 * SK + 2 * SV;  // first barrier after the rings
  uint8_t* base;
  uint32_t sQ, sK, sV, bar0;
  __device__ uint32_t q_full() const { return bar0; }
  __device__ uint32_t q_empty() const { return bar0 + 8u; }
  __device__ uint32_t k_full(int s) const { return bar0 + 8u * (2 + s); }
  __device__ uint32_t v_full(int s) const { return bar0 + 8u * (2 + SK + s); }
  // K and V slots are released separately: a K tile is free once both
  // query tiles' QK^T products read it, one key tile before its V is
  __device__ uint32_t k_empty(int s) const { return bar0 + 8u * (2 + SK + SV + s); }
  __device__ uint32_t v_empty(int s) const { return bar0 + 8u * (2 + 2 * SK + SV + s); }
  __device__ uint32_t s_full(int t) const { return bar0 + 8u * (kR + t); }
  __device__ uint32_t p_full(int t) const { return bar0 + 8u * (kR + 2 + t); }
  // completes once per item, after query tile t's last P.V (the epilogue's wait)
  __device__ uint32_t o_final(int t) const { return bar0 + 8u * (kR + 4 + t); }
  __device__ uint32_t drain() const { return bar0 + 8u * (kR + 6); }
  // key-split merge hand-over: lane 1's row max / sum written (128 arrivals),
  // then lane 1's O read by warpgroup 0 (128 arrivals)
  __device__ uint32_t merge_full() const { return bar0 + 8u * (kR + 7); }
  __device__ uint32_t merge_done() const { return bar0 + 8u * (kR + 8); }
  __device__ float2* merge() const { return reinterpret_cast<float2*>(base + Cfg::kOffMerge); }
  __device__ const int* order() const { return reinterpret_cast<const int*>(base + Cfg::kOffOrder); }
  __device__ uint8_t* mask_buf(int warp) const { return base + Cfg::kOffMaskBuf + warp * kMaskBufBytes; }
};

// One work item of one (b, h): two lanes t = 0, 1, each a 128-row query tile
// with its own S / O in tensor memory, visiting key tiles
// tr[t].t_begin, + stride, ... < tr[t].t_end.  Normally lane t is query tile t
// (stride 1).  When the second query tile would have no rows (short Sq, e.g.
// decode or chunked prefill), both lanes take the same 128 rows and split the
// key tiles even / odd (stride 2), so the tensor core still alternates
// between two softmax warpgroups; warpgroup 0 merges the two partial rows.
// The item streams the key tiles [tb, tb + N).
struct Item {
  int b, h, kvh;
  int kvsplit;  // split-KV range index (0 when the key tiles are not split)
  int64_t q0;
  BatchLimits L;
  TileRange tr[kQTiles];
  int tb, N, stride;
  bool lanesplit;  // both lanes on query tile 0's rows, alternate key tiles
  __device__ bool active(int t, int j) const {
    return j >= tr[t].t_begin && j < tr[t].t_end && ((j - tr[t].t_begin) & (stride - 1)) == 0;
  }
  __device__ bool last(int t, int j) const { return j + stride >= tr[t].t_end; }
  __device__ int tiles(int t) const {
    return tr[t].t_end > tr[t].t_begin ? (tr[t].t_end - tr[t].t_begin + stride - 1) / stride : 0;
  }
  __device__ int64_t row0(int t) const { return q0 + (lanesplit ? 0 : t * BM); }
};

template <bool KSPLIT>
__device__ __forceinline__ Item make_item(const CommonParams& p, int idx, const int* border) {
  const int bh = p.B * p.Hq;
  const int per_qp = bh * p.num_splits;
  const int n_qp = (p.Sq + kQTiles * BM - 1) / (kQTiles * BM);
  Item it;
  const int qp = n_qp - 1 - idx / per_qp;  // latest query rows first
  int rem = idx - (idx / per_qp) * per_qp;
  it.kvsplit = rem / bh;  // items of one split range of one kv group are consecutive
  rem -= it.kvsplit * bh;
  const int br = rem / p.Hq;
  it.b = border ? border[br] : br;  // costliest batches first
  it.h = rem - br * p.Hq;           // heads of one kv group are consecutive items
  it.kvh = it.h / p.group;
  it.q0 = (int64_t)qp * (kQTiles * BM);
  it.L = batch_limits(p, it.b);
  // key tiles of the item before any split-KV cut: both query tiles' ranges
  TileRange tq[kQTiles];
  int tb = 0, te = 0;
  bool any = false;
  const bool lanesplit = KSPLIT && it.q0 + BM >= (int64_t)p.Sq;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    tq[t] = (lanesplit && t == 1) ? tq[0] : tile_range(p, it.L, it.q0 + t * BM, BM, BN);
    if (tq[t].t_end > tq[t].t_begin) {
      tb = any ? min(tb, tq[t].t_begin) : tq[t].t_begin;
      te = any ? max(te, tq[t].t_end) : tq[t].t_end;
      any = true;
    }
  }
  // split-KV: this item keeps the split-th of num_splits contiguous pieces
  if (p.num_splits > 1 && te > tb) {
    const int cs = (te - tb + p.num_splits - 1) / p.num_splits;
    const int c0 = min(te, tb + it.kvsplit * cs);
    te = min(te, c0 + cs);
    tb = c0;
  }
  it.tb = tb;
  it.N = te - tb;
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    it.tr[t] = tq[t];
    it.tr[t].t_begin = max(tq[t].t_begin, tb);
    it.tr[t].t_end = min(tq[t].t_end, te);
    if (it.tr[t].t_end <= it.tr[t].t_begin) it.tr[t].t_begin = it.tr[t].t_end = 0;
  }
  it.lanesplit = lanesplit;
  it.stride = 1;
  if (lanesplit) {
    // both lanes on query tile 0's rows, alternate key tiles
    it.stride = 2;
    if (it.tr[0].t_end > it.tr[0].t_begin + 1) {
      it.tr[1] = it.tr[0];
      it.tr[1].t_begin = it.tr[0].t_begin + 1;
    } else {
      it.tr[1].t_begin = it.tr[1].t_end = 0;  // one key tile: lane 1 stays empty
    }
  }
  return it;
}

// Batches ranked by their number of valid key tiles (descending, ties by
// index), written to order[rank] = b.  Threads 0..B-1 each rank one batch.
__device__ __forceinline__ void rank_batches(const CommonParams& p, int* order) {
  const int b = threadIdx.x;
  if (b >= p.B) return;
  auto cost = [&](int i) {
    const BatchLimits L = batch_limits(p, i);
    int64_t n = L.lsk < (int64_t)p.Sk ? L.lsk : (int64_t)p.Sk;
    return n > 0 ? n : (int64_t)0;
  };
  const int64_t c = cost(b);
  int rank = 0;
  for (int i = 0; i < p.B; ++i) {
    const int64_t ci = cost(i);
    rank += (ci > c || (ci == c && i < b)) ? 1 : 0;
  }
  order[rank] = b;
}

// Static snake schedule: round r gives CTA c item r*G + c (r even) or
// r*G + G-1-c (r odd), so heavy and light items alternate between CTAs.
__device__ __forceinline__ int item_of_round(int r, int n_items) {
  const int G = gridDim.x;
  const int c = blockIdx.x;
  const int idx = r * G + ((r & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

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

// Maximum / minimum of 128 values: three-input max / min in eight
// independent chains (68 instructions, dependency depth 9).
__device__ __forceinline__ float max128(const float (&x)[BN]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(x[k], x[k + 8]);
#pragma unroll
  for (int i = 16; i < BN; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmax3(m[k], x[i + k], x[i + 8 + k]);
  return fmaxf(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], fmax3(m[5], m[6], m[7])));
}

__device__ __forceinline__ float min128(const float (&x)[BN]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fminf(x[k], x[k + 8]);
#pragma unroll
  for (int i = 16; i < BN; i += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmin3(m[k], x[i + k], x[i + 8 + k]);
  return fminf(fmin3(m[0], m[1], m[2]), fmin3(m[3], m[4], fmin3(m[5], m[6], m[7])));
}

// Prefetch of one box of a 3-D tensor map into L2 (no shared memory, no
// completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tmap), "r"(c0),
               "r"(c1), "r"(c2)
               : "memory");
}

// ------------------------------------------------------------------ producer
// One thread.  Q tiles per item (after the previous item's QK^T products
// released them), then the item's K / V tiles into the stage ring; the ring
// index g runs on across items.
template <int D, bool KSPLIT, bool MB>
__device__ __forceinline__ void producer_role(const TcParams& P, const Smem<D, MB>& sm, int n_items) {
  using Cfg = TcConfig<D, MB>;
  constexpr int SK = Cfg::kKStages, SV = Cfg::kVStages;
  const CommonParams& p = P.c;
  int g = 0;        // K / V tiles issued so far (ring position)
  int k_issued = 0, v_issued = 0;  // tiles whose K / V copies were started
  int q_items = 0;  // items whose Q was loaded
  // batch ranking only in the key-split variant (short query ranges, where
  // ragged lengths decide the cost); elsewhere the pointer stays out of registers
  const int* border = (KSPLIT && p.B <= kMaxOrderB) ? sm.order() : nullptr;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = item_of_round(r, n_items);
    if (idx < 0) break;
    const Item it = make_item<KSPLIT>(p, idx, border);
    if (it.N == 0) continue;
    const int q_plane = it.b * p.Hq + it.h;
    const int kv_plane = it.b * p.Hkv + it.kvh;
    // a lane-split item's two lanes share query tile 0's rows: one Q tile
    const int nq = it.lanesplit ? 1 : kQTiles;
    // This point is reached once the previous item's K / V are all issued,
    // a few key tiles before its last QK^T frees the Q buffer: the Q rows go
    // into L2 now, so the load below (which a whole item boundary waits for)
    // does not wait on DRAM.  Key-split items are a few key tiles long, too
    // short for the prefetch to run ahead (measured slightly slower there).
    if (!KSPLIT && q_items > 0)
      for (int t = 0; t < nq; ++t)
        for (int s = 0; s < Cfg::kSub; ++s) tma_prefetch_l2_3d(&P.tmap_q, s * 64, (int)it.row0(t), q_plane);
    if (q_items > 0 && !mbar_wait(sm.q_empty(), (q_items - 1) & 1, p.timeout_ns, p.status)) break;
    mbar_arrive_expect_tx(sm.q_full(), nq * Cfg::kTileBytes);
    for (int t = 0; t < nq; ++t)
      for (int s = 0; s < Cfg::kSub; ++s)
        tma_load_3d(sm.sQ + t * Cfg::kTileBytes + s * Cfg::kSubBytes, &P.tmap_q, sm.q_full(), s * 64,
                    (int)it.row0(t), q_plane);
    ++q_items;
    for (int n = 0; n < it.N; ++n, ++g) {
      const int sk = g % SK, sv = g % SV;
      const int key0 = (it.tb + n) * BN;
      // K(g) reuses the slot of K(g - SK), freed after that tile's QK^T
      // products; V(g) the slot of V(g - SV), freed after its P.V products,
      // which come a key tile later.  So K runs ahead of V.
      if (g >= SK && !mbar_wait(sm.k_empty(sk), ((g / SK) - 1) & 1, p.timeout_ns, p.status)) {
        ok = false;
        break;
      }
      // combined: this phase of k_full(sk) completes when K and V both landed
      mbar_arrive_expect_tx(sm.k_full(sk), Cfg::kCombined ? 2 * Cfg::kTileBytes : Cfg::kTileBytes);
      for (int s = 0; s < Cfg::kSub; ++s)
        tma_load_3d(sm.sK + sk * Cfg::kTileBytes + s * Cfg::kSubBytes, &P.tmap_k, sm.k_full(sk), s * 64,
                    key0, kv_plane);
      ++k_issued;
      if (g >= SV && !mbar_wait(sm.v_empty(sv), ((g / SV) - 1) & 1, p.timeout_ns, p.status)) {
        ok = false;
        break;
      }
      const uint32_t vbar = Cfg::kCombined ? sm.k_full(sk) : sm.v_full(sv);
      if (!Cfg::kCombined) mbar_arrive_expect_tx(vbar, Cfg::kTileBytes);
      for (int s = 0; s < Cfg::kSub; ++s)
        tma_load_3d(sm.sV + sv * Cfg::kTileBytes + s * Cfg::kSubBytes, &P.tmap_v, vbar, s * 64, key0, kv_plane);
      ++v_issued;
    }
  }
  // Let every copy this thread started land before the CTA can exit (with
  // the combined barrier, k_full covers V as well).
  for (int n = (k_issued > SK ? k_issued - SK : 0); n < k_issued; ++n)
    mbar_wait(sm.k_full(n % SK), (n / SK) & 1, p.timeout_ns, p.status);
  if (!Cfg::kCombined)
    for (int n = (v_issued > SV ? v_issued - SV : 0); n < v_issued; ++n)
      mbar_wait(sm.v_full(n % SV), (n / SV) & 1, p.timeout_ns, p.status);
  if (q_items > 0) mbar_wait(sm.q_full(), (q_items - 1) & 1, p.timeout_ns, p.status);
}

// S_t = Q K^T for one key tile (K tile at kaddr, Q from query tile slot qt:
// t, or 0 for both lanes of a lane-split item), then commit s_full(t).
// Warp-collective: the whole MMA warp calls it, one elected lane issues.
template <int D, bool BF16, bool MB>
__device__ __forceinline__ void issue_qk(const Smem<D, MB>& sm, uint32_t tmem, int t, int qt, uint32_t kaddr) {
  using Cfg = TcConfig<D, MB>;
  constexpr uint32_t idesc_qk = make_idesc_f16kind(BF16, BM, BN, false);
  const uint64_t adesc0 = make_sdesc_sw128(sm.sQ + qt * Cfg::kTileBytes, 16, 1024);
  const uint64_t bdesc0 = make_sdesc_sw128(kaddr, 16, 1024);
  // K steps kk = 4s..4s+3 lie in 64-column block s (kSubBytes apart), 32
  // bytes into each 128-byte row; the start address field counts 16 bytes
#pragma unroll
  for (int s = 0; s < D / 64; ++s) {
    const uint32_t o = (s * Cfg::kSubBytes) >> 4;
    mma_ss4_elect(tmem + t * 128, adesc0 + o, bdesc0 + o, adesc0 + o + 2, bdesc0 + o + 2, adesc0 + o + 4,
                  bdesc0 + o + 4, adesc0 + o + 6, bdesc0 + o + 6, idesc_qk, s > 0 ? 1u : 0u);
  }
  tc_commit_elect(sm.s_full(t));
}

// O_t (+)= P_t V for one key tile (V tile at vaddr; P_t in tensor memory over
// the first half of S_t).
// Warp-collective, like issue_qk.
template <int D, bool BF16, bool MB>
__device__ __forceinline__ void issue_pv(const Smem<D, MB>& sm, uint32_t tmem, int t, uint32_t vaddr,
                                         bool accumulate) {
  using Cfg = TcConfig<D, MB>;
  constexpr uint32_t idesc_pv = make_idesc_f16kind(BF16, BM, D, true);
  // B = V[keys 16kk.., 0..D): MN-major; 8-key groups 1024 B apart, 64-column
  // blocks kSubBytes apart.
  const uint64_t bdesc0 = make_sdesc_sw128(vaddr, Cfg::kSubBytes, 1024);
  // four K steps (16 keys, 2048 bytes of V, 8 columns of P each) per issue block
  const uint32_t d = tmem + kColO + t * 128, a = tmem + t * 128;
#pragma unroll
  for (int kk = 0; kk < BN / 16; kk += 4)
    mma_ts4_elect(d, a + kk * 8, bdesc0 + (uint32_t)(kk * 128), a + (kk + 1) * 8,
                  bdesc0 + (uint32_t)((kk + 1) * 128), a + (kk + 2) * 8, bdesc0 + (uint32_t)((kk + 2) * 128),
                  a + (kk + 3) * 8, bdesc0 + (uint32_t)((kk + 3) * 128), idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
}

// ------------------------------------------------------------------ MMA issuer
// Whole warp waits; lane 0 issues.  Per item and key tile j (iteration n):
// the P.V products of tile j-1, then the QK^T products of tile j, per query
// tile in turn.  Returns after every MMA it issued has completed.
template <int D, bool BF16, bool KSPLIT, bool MB>
__device__ __forceinline__ void mma_role(const TcParams& P, const Smem<D, MB>& sm, uint32_t tmem,
                                         int n_items, int lane) {
  using Cfg = TcConfig<D, MB>;
  constexpr int SK = Cfg::kKStages, SV = Cfg::kVStages;
  const CommonParams& p = P.c;
  int g0 = 0;                 // ring position of the item's first key tile
  int q_items = 0;            // items whose Q was consumed
  int pc[kQTiles] = {0, 0};   // P tiles consumed per lane (all items)
  // batch ranking only in the key-split variant (short query ranges, where
  // ragged lengths decide the cost); elsewhere the pointer stays out of registers
  const int* border = (KSPLIT && p.B <= kMaxOrderB) ? sm.order() : nullptr;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = item_of_round(r, n_items);
    if (idx < 0) break;
    const Item it = make_item<KSPLIT>(p, idx, border);
    if (it.N == 0) continue;
    if (!mbar_wait_warp(sm.q_full(), q_items & 1, p.timeout_ns, p.status)) { ok = false; break; }
    ++q_items;
    int64_t zero_from = it.L.lsk < (int64_t)p.Sk ? it.L.lsk : (int64_t)p.Sk;
    if (zero_from < 0) zero_from = 0;
    bool first_pv[kQTiles] = {true, true};
    for (int n = 0; ok && n <= it.N; ++n) {
      const int j = it.tb + n;
      bool k_ready = false;  // K(j) is waited for only before its first use
      if (n >= 1) {
        const int gp = g0 + n - 1;
        const int ps = gp % SV;
        // combined barrier: V(j - 1) landed with K(j - 1), which this warp
        // waited for before that tile's QK^T products
        if (!Cfg::kCombined && !mbar_wait_warp(sm.v_full(ps), (gp / SV) & 1, p.timeout_ns, p.status)) {
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
            uint8_t* vblk = sm.base + Cfg::kOffV + ps * Cfg::kTileBytes + s * Cfg::kSubBytes;
            for (int c = lane; c < chunks; c += 32)
              *reinterpret_cast<uint4*>(vblk + (size_t)(r0 + (c >> 3)) * 128 + (c & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
      }
      tc_fence_after();
      const bool pv0 = n >= 1 && it.active(0, j - 1), pv1 = n >= 1 && it.active(1, j - 1);
      const bool s0 = n < it.N && it.active(0, j), s1 = n < it.N && it.active(1, j);
      const uint32_t kaddr = sm.sK + ((g0 + n) % SK) * Cfg::kTileBytes;
      const uint32_t vaddr = sm.sV + ((g0 + n - 1 + SV) % SV) * Cfg::kTileBytes;
      // K(j) is waited for only right before the first S that reads it, so a
      // late K never holds back the P.V products of tile j-1.
      auto wait_k = [&]() -> bool {
        if (k_ready) return true;
        const int gs = g0 + n;
        if (!mbar_wait_warp(sm.k_full(gs % SK), (gs / SK) & 1, p.timeout_ns, p.status)) return false;
        tc_fence_after();
        k_ready = true;
        return true;
      };
      // A lane with no P.V pending gets its S first (key-split lanes
      // alternate), so the tensor core has work while the other lane's
      // softmax runs.  S_t(j) overwrites the S region that held the lane's
      // previous P, whose P.V this thread issued earlier.
      if (!KSPLIT) {
        // both lanes are query tiles: P.V then S, lane by lane
        if (pv0) {
          if (!mbar_wait_warp(sm.p_full(0), pc[0] & 1, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          issue_pv<D, BF16, MB>(sm, tmem, 0, vaddr, !first_pv[0]);
          if (it.last(0, j - 1)) tc_commit_elect(sm.o_final(0));  // lane 0 has seen its last key tile
          first_pv[0] = false;
          ++pc[0];
        }
        if (s0) {
          if (!wait_k()) { ok = false; break; }
          issue_qk<D, BF16, MB>(sm, tmem, 0, 0, kaddr);
        }
        __syncwarp();
        if (pv1) {
          if (!mbar_wait_warp(sm.p_full(1), pc[1] & 1, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          issue_pv<D, BF16, MB>(sm, tmem, 1, vaddr, !first_pv[1]);
          if (it.last(1, j - 1)) tc_commit_elect(sm.o_final(1));
          first_pv[1] = false;
          ++pc[1];
        }
        if (s1) {
          if (!wait_k()) { ok = false; break; }
          issue_qk<D, BF16, MB>(sm, tmem, 1, it.lanesplit ? 0 : 1, kaddr);
        }
        __syncwarp();
      } else {
      if (s0 && !pv0) {
        if (!wait_k()) { ok = false; break; }
        issue_qk<D, BF16, MB>(sm, tmem, 0, 0, kaddr);
      }
      if (s1 && !pv1) {
        if (!wait_k()) { ok = false; break; }
        issue_qk<D, BF16, MB>(sm, tmem, 1, it.lanesplit ? 0 : 1, kaddr);
      }
      if (pv0) {
        if (!mbar_wait_warp(sm.p_full(0), pc[0] & 1, p.timeout_ns, p.status)) { ok = false; break; }
        tc_fence_after();
        issue_pv<D, BF16, MB>(sm, tmem, 0, vaddr, !first_pv[0]);
        if (it.last(0, j - 1)) tc_commit_elect(sm.o_final(0));  // lane 0 has seen its last key tile
        first_pv[0] = false;
        ++pc[0];
        if (s0) {
          if (!wait_k()) { ok = false; break; }
          issue_qk<D, BF16, MB>(sm, tmem, 0, 0, kaddr);
        }
      }
      if (pv1) {
        if (!mbar_wait_warp(sm.p_full(1), pc[1] & 1, p.timeout_ns, p.status)) { ok = false; break; }
        tc_fence_after();
        issue_pv<D, BF16, MB>(sm, tmem, 1, vaddr, !first_pv[1]);
        if (it.last(1, j - 1)) tc_commit_elect(sm.o_final(1));
        first_pv[1] = false;
        ++pc[1];
        if (s1) {
          if (!wait_k()) { ok = false; break; }
          issue_qk<D, BF16, MB>(sm, tmem, 1, it.lanesplit ? 0 : 1, kaddr);
        }
      }
      }  // KSPLIT
      __syncwarp();
      if (!ok) break;
      // K(j) was read by this iteration's QK^T products, V(j-1) by its P.V
      if (n < it.N) tc_commit_elect(sm.k_empty((g0 + n) % SK));
      if (n >= 1) tc_commit_elect(sm.v_empty((g0 + n - 1) % SV));
      // the item's last QK^T products are issued: Q may be replaced once they finish
      if (n == it.N - 1) tc_commit_elect(sm.q_empty());
      __syncwarp();
    }
    if (!ok) break;
    g0 += it.N;
  }
  // Wait for every MMA this warp issued before tensor memory is freed.
  tc_commit_elect(sm.drain());
  mbar_wait_warp(sm.drain(), 0, p.timeout_ns, p.status);
}

// Mask block of one warp -- 32 rows (mask rows mwarp, mwarp + Sk, ...) by the
// 128 keys [key0, key0 + 128) -- into x of the lane that owns each row
// (natural units; 0 for rows >= nrows and keys >= Sk).  A lane-per-row load
// would touch 32 cache lines per instruction; instead each instruction loads
// 4 rows x 128 contiguous bytes, and a 4 KB per-warp buffer (16-byte chunks
// XOR-swizzled by row, conflict-free both ways) turns rows into lanes.  Needs
// vec4: mask rows are 16-byte aligned (Sk % 4 == 0) and loads are float4;
// otherwise each 16-byte chunk is four scalar loads with per-element bounds.
__device__ __forceinline__ void mask_rows_coalesced(float (&x)[BN], const float* mwarp, int nrows,
                                                    int Sk, int key0, bool vec4, uint8_t* buf,
                                                    int lane) {
  const int rsub = lane >> 3;  // row within a group of 4
  const int csub = lane & 7;   // 16-byte chunk within a 128-byte row segment
  // one 32-key chunk in flight per lane (8 float4); the other lane's warps
  // cover the latency
  float4 v[8];
  auto load = [&](int k, float4 (&dst)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = 4 * i + rsub;
      const int key = key0 + 32 * k + 4 * csub;
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
      dst[i] = t;
    }
  };
  load(0, v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = 4 * i + rsub;
      *reinterpret_cast<float4*>(buf + row * 128 + ((csub ^ (row & 7)) << 4)) = v[i];
    }
    if (k + 1 < 4) load(k + 1, v);
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 t = *reinterpret_cast<const float4*>(buf + lane * 128 + ((c ^ (lane & 7)) << 4));
      x[32 * k + 4 * c + 0] = t.x;
      x[32 * k + 4 * c + 1] = t.y;
      x[32 * k + 4 * c + 2] = t.z;
      x[32 * k + 4 * c + 3] = t.w;
    }
    __syncwarp();
  }
}

// The asynchronous form of the same staging, for rows of whole 16-byte
// chunks (vec4) when a second 4 KB buffer per warp is free (key-split
// kernels whose items all share one query tile leave query tile 1's shared
// memory unused): chunk k of 32 keys goes to buffer k & 1 by cp.async
// (zero-filled outside the mask), so two chunks are in flight and no
// registers hold them, and the next key tile's first two chunks are
// requested as soon as their buffers are read, to land during this tile's
// softmax.
__device__ __forceinline__ void mask_chunk_async(uint8_t* buf, const float* mwarp, int nrows, int Sk, int key0,
                                                 int k, int lane) {
  const int rsub = lane >> 3, csub = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = 4 * i + rsub;
    const int key = key0 + 32 * k + 4 * csub;
    const bool valid = row < nrows && key + 3 < Sk;
    const float* src = valid ? mwarp + (int64_t)row * Sk + key : mwarp;
    const uint32_t dst = smem_u32(buf + row * 128 + ((csub ^ (row & 7)) << 4));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void mask_chunk_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
  __syncwarp();  // every lane's copies of the chunk have landed
}
__device__ __forceinline__ void mask_chunk_read(float (&x)[BN], const uint8_t* buf, int k, int lane) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float4 t = *reinterpret_cast<const float4*>(buf + lane * 128 + ((c ^ (lane & 7)) << 4));
    x[32 * k + 4 * c + 0] = t.x;
    x[32 * k + 4 * c + 1] = t.y;
    x[32 * k + 4 * c + 2] = t.z;
    x[32 * k + 4 * c + 3] = t.w;
  }
  __syncwarp();  // every lane has read the buffer before it is refilled
}

// ------------------------------------------------------------------ softmax
// Warpgroup t (warps 4t..4t+3); thread = one query row of query tile t.
template <int D, bool BF16, bool SOFTCAP, bool MASK, bool KSPLIT, bool SPLITKV>
__device__ __forceinline__ void softmax_role(const TcParams& P, const Smem<D, MASK>& sm, uint32_t tmem,
                                             int n_items, int warp, int lane) {
  using Cfg = TcConfig<D, MASK>;
  const CommonParams& p = P.c;
  const int t = warp >> 2;  // query tile of this warpgroup
  const int wq = warp & 3;  // TMEM lane quarter
  const int row = wq * 32 + lane;
  const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
  const uint32_t s_addr = tmem + lane_base + t * 128;
  const uint32_t o_addr = tmem + lane_base + kColO + t * 128;
  int sc = 0;                // S tiles this lane consumed (all items)
  int oc[kQTiles] = {0, 0};  // o_final completions per lane so far (both warpgroups track both)
  int mc = 0;                // key-split items merged so far
  // batch ranking only in the key-split variant (short query ranges, where
  // ragged lengths decide the cost); elsewhere the pointer stays out of registers
  const int* border = (KSPLIT && p.B <= kMaxOrderB) ? sm.order() : nullptr;
  bool ok = true;
  for (int r = 0; ok; ++r) {
    const int idx = item_of_round(r, n_items);
    if (idx < 0) break;
    const Item it = make_item<KSPLIT>(p, idx, border);
    // selects, not it.tr[t]: a runtime index would put the item in local memory
    const TileRange T = t == 0 ? it.tr[0] : it.tr[1];
    const int nt0 = it.tiles(0), nt1 = it.tiles(1);
    const int nt = t == 0 ? nt0 : nt1;
    const int64_t qi = (t == 0 ? it.row0(0) : it.row0(1)) + row;
    const RowLimits R = row_limits(p, it.L, qi);
    const float* mwarp = nullptr;  // this warp's first mask row
    int mrows = 0;
    if constexpr (MASK) {
      int64_t plane = 0;
      if (p.mask_planes == p.B) plane = it.b;
      else if (p.mask_planes == p.B * p.Hq) plane = (int64_t)it.b * p.Hq + it.h;
      const int64_t qw0 = qi - lane;  // this warp's first row
      mwarp = p.mask + (plane * p.Sq + (qw0 < p.Sq ? qw0 : 0)) * (int64_t)p.Sk;
      mrows = qw0 < p.Sq ? (int)min((int64_t)32, (int64_t)p.Sq - qw0) : 0;
    }

    float m_run = -INFINITY;  // running max, log2 units
    float l_run = 0.0f;       // running denominator
    // asynchronous mask staging: key-split kernel, every item one query tile
    // (query tile 1's shared memory is then never used), 16-byte mask rows
    const bool mpipe = MASK && KSPLIT && D == 128 && p.Sq <= BM && p.mask_vec4 != 0;
    uint8_t* mb0 = sm.mask_buf(warp);
    uint8_t* mb1 = sm.base + Cfg::kOffQ + Cfg::kTileBytes + warp * kMaskBufBytes;
    const int kstep = (KSPLIT ? it.stride : 1) * BN;
    if (mpipe && nt > 0) {
      mask_chunk_async(mb0, mwarp, mrows, p.Sk, T.t_begin * BN, 0, lane);
      mask_chunk_async(mb1, mwarp, mrows, p.Sk, T.t_begin * BN, 1, lane);
    }
    for (int c = 0; c < nt; ++c, ++sc) {
      const int64_t key0 = (int64_t)(T.t_begin + c * (KSPLIT ? it.stride : 1)) * BN;
      float x[BN];
      if constexpr (MASK) {
        // this tile's mask rows into x (natural units), before the S wait:
        // the loads overlap the tensor core's work
        if (mpipe) {
          const bool more = c + 1 < nt;
          const int kn = (int)key0 + kstep;
          mask_chunk_wait<1>();
          mask_chunk_read(x, mb0, 0, lane);
          mask_chunk_async(mb0, mwarp, mrows, p.Sk, (int)key0, 2, lane);
          mask_chunk_wait<1>();
          mask_chunk_read(x, mb1, 1, lane);
          mask_chunk_async(mb1, mwarp, mrows, p.Sk, (int)key0, 3, lane);
          mask_chunk_wait<1>();
          mask_chunk_read(x, mb0, 2, lane);
          if (more) {
            mask_chunk_async(mb0, mwarp, mrows, p.Sk, kn, 0, lane);
            mask_chunk_wait<1>();
          } else {
            mask_chunk_wait<0>();
          }
          mask_chunk_read(x, mb1, 3, lane);
          if (more) mask_chunk_async(mb1, mwarp, mrows, p.Sk, kn, 1, lane);
        } else {
          mask_rows_coalesced(x, mwarp, mrows, p.Sk, (int)key0, p.mask_vec4 != 0, sm.mask_buf(warp), lane);
        }
      }
      if (!mbar_wait_warp(sm.s_full(t), sc & 1, p.timeout_ns, p.status)) { ok = false; break; }
      tc_fence_after();

      const bool need_mask = !(key0 >= T.full_lo && key0 + BN <= T.full_hi);
      float m_tile;
      // x is either already in log2 units (scaled) or a raw value that xs
      // brings there: the raw Q.K (xs = scale log2 e) or, with a soft-cap,
      // tanh(scale Q.K / c) (xs = c log2 e > 0)
      bool scaled = false;
      const float xs = SOFTCAP ? p.sc_out : p.scale_log2;
      if constexpr (MASK) {
        // x = transform(S) + mask * log2 e, 32 columns at a time
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t sr[32];
          tmem_ld32(s_addr + k * 32, sr);
          tmem_wait_ld();
          if constexpr (SOFTCAP) {
            // (mask, mask) * log2 e + c log2 e * tanh(scale s / c)
            const uint64_t in2 = f2(p.sc_in, p.sc_in), out2 = f2(p.sc_out, p.sc_out);
            const uint64_t le2 = f2(kLog2e, kLog2e);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float a0, a1;
              f2_split(fmul2(f2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), in2), a0, a1);
              const uint64_t tv = f2(fast_tanh(a0), fast_tanh(a1));
              f2_split(ffma2(tv, out2, fmul2(f2(x[32 * k + i], x[32 * k + i + 1]), le2)), x[32 * k + i],
                       x[32 * k + i + 1]);
            }
          } else {
            // (mask, mask) * log2 e + (s, s) * scale log2 e, two keys per instruction
            const uint64_t sc2 = f2(p.scale_log2, p.scale_log2);
            const uint64_t le2 = f2(kLog2e, kLog2e);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const uint64_t sv = fmul2(f2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sc2);
              f2_split(ffma2(f2(x[32 * k + i], x[32 * k + i + 1]), le2, sv), x[32 * k + i], x[32 * k + i + 1]);
            }
          }
        }
        scaled = true;
      } else {
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
        if constexpr (SOFTCAP) {
          // tanh(scale s / c); xs = c log2 e brings it to log2 units
          const uint64_t in2 = f2(p.sc_in, p.sc_in);
#pragma unroll
          for (int i = 0; i < BN; i += 2) {
            float a0, a1;
            f2_split(fmul2(f2(x[i], x[i + 1]), in2), a0, a1);
            x[i] = fast_tanh(a0);
            x[i + 1] = fast_tanh(a1);
          }
        }
      }
      if (need_mask) {
        // structural limits of this row: keys outside [lo, hi) become -inf;
        // with a positive scale the raw scores can be selected directly
        if (!scaled && !(xs > 0.0f)) {
#pragma unroll
          for (int i = 0; i < BN; ++i) x[i] *= xs;
          scaled = true;
        }
        int lo = R.lo - (int)key0, hi = R.hi - (int)key0;
        lo = lo < 0 ? 0 : (lo > BN ? BN : lo);
        hi = hi < 0 ? 0 : (hi > BN ? BN : hi);
        const int lo_rel = (int)lo;
        const uint32_t span = hi > lo ? (uint32_t)(hi - lo) : 0u;
#pragma unroll
        for (int i = 0; i < BN; ++i) x[i] = ((uint32_t)(i - lo_rel) < span) ? x[i] : -INFINITY;
      }
      if (scaled) {
        m_tile = max128(x);
      } else if (!need_mask) {
        // every key of this tile is visible to every row: the extreme raw
        // score times the (signed) scale is the max of the scaled scores
        m_tile = (xs >= 0.0f ? max128(x) : min128(x)) * xs;
      } else {
        // raw scores with -inf outside the row's keys, positive scale
        const float mr = max128(x);
        m_tile = mr == -INFINITY ? -INFINITY : mr * xs;
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
      const float xmul = scaled ? 1.0f : xs;  // brings x to log2 units

      // P = 2^(x - m) in four 32-column chunks, each packed into 16 columns
      // of 16-bit pairs over the first half of this S row.  The argument and
      // the row sum take one packed instruction per two keys; the sum runs
      // in four independent pairs of accumulators.
      const uint64_t mul2 = f2(xmul, xmul), sub2 = f2(-m_sub, -m_sub);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float a0, a1;
          f2_split(ffma2(f2(x[ch * 32 + 2 * i], x[ch * 32 + 2 * i + 1]), mul2, sub2), a0, a1);
          const float e0 = fast_exp2(a0);
          const float e1 = fast_exp2(a1);
          acc[i & 3] = fadd2(acc[i & 3], f2(e0, e1));
          pk[i] = pack2<BF16>(e0, e1);
        }
        tmem_st16(s_addr + ch * 16, pk);
      }
      float sum, sum_hi;
      f2_split(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])), sum, sum_hi);
      sum += sum_hi;
      l_run = l_run * alpha + sum;
      m_run = m_use;

      if (__any_sync(0xffffffffu, rescale)) {
        // O_t already holds every earlier P.V of this item (see the header)
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
      if (lane == 0) mbar_arrive(sm.p_full(t));
    }
    if (!ok) break;

    // ---------------------------------------------------------- epilogue
    float2* merge = sm.merge();
    float a0 = 1.0f, a1 = 0.0f, inv_l = 0.0f;  // out = (a0 O_t + a1 O_1) * inv_l
    float m_fin = m_run, l_fin = l_run;        // the row's reference max (log2 units) and sum
    bool have_o = nt > 0, have_o1 = false;
    if (KSPLIT && it.lanesplit) {
      // key-split lanes: warpgroup 1 hands its row max / sum to warpgroup 0,
      // which combines both partial rows
      if (t == 1) {
        merge[row] = make_float2(m_run, l_run);
        mbar_arrive(sm.merge_full());
        // O_1 must not be overwritten by this lane's next item before warpgroup 0 read it
        if (!mbar_wait_warp(sm.merge_done(), mc & 1, p.timeout_ns, p.status)) { ok = false; break; }
        tc_fence_after();
        ++mc;
        oc[0] += nt0 > 0;
        oc[1] += nt1 > 0;
        continue;
      }
      if (nt1 > 0) {
        if (!mbar_wait_warp(sm.o_final(1), oc[1] & 1, p.timeout_ns, p.status)) { ok = false; break; }
        have_o1 = true;
      }
      if (!mbar_wait_warp(sm.merge_full(), mc & 1, p.timeout_ns, p.status)) { ok = false; break; }
      const float2 ml1 = merge[row];
      const float m = fmaxf(m_run, ml1.x);
      a0 = m_run == -INFINITY ? 0.0f : fast_exp2(m_run - m);
      a1 = ml1.x == -INFINITY ? 0.0f : fast_exp2(ml1.x - m);
      const float l = a0 * l_run + a1 * ml1.y;
      inv_l = l > 0.0f ? 1.0f / l : 0.0f;
      m_fin = m;
      l_fin = l;
    } else {
      inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    }
    if (have_o) {
      if (!mbar_wait_warp(sm.o_final(t), (t == 0 ? oc[0] : oc[1]) & 1, p.timeout_ns, p.status)) { ok = false; break; }
    }
    oc[0] += nt0 > 0;
    oc[1] += nt1 > 0;
    tc_fence_after();
    // natural-log log-sum-exp of the row's scores (-inf without a finite score)
    const float lse_row = l_fin > 0.0f ? (m_fin + __log2f(l_fin)) * 0.6931471805599453f : -INFINITY;
    const bool partial = SPLITKV && p.num_splits > 1;  // split-KV: a normalised fp32 partial row
    const int64_t row_id = ((int64_t)it.b * p.Hq + it.h) * p.Sq + qi;
    int64_t base;
    if (partial)
      base = ((int64_t)it.kvsplit * p.B * p.Hq * p.Sq + row_id) * D;
    else if (p.out_layout == 0)
      base = row_id * D;
    else
      base = (((int64_t)it.b * p.Sq + qi) * p.Hq + it.h) * D;
    const uint32_t o1_addr = tmem + lane_base + kColO + 128;
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
      if (KSPLIT && have_o1) {  // key-split: fold in lane 1's partial row
        uint32_t o1[32];
        tmem_ld32(o1_addr + k * 32, o1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[i] = __float_as_uint(a0 * __uint_as_float(o[i]) + a1 * __uint_as_float(o1[i]));
      }
      if (qi < p.Sq) {
        if (partial) {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + base + k * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                 __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
        } else {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + base + k * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
    if (qi < p.Sq) {
      if (partial)
        p.ws_lse[(int64_t)it.kvsplit * p.B * p.Hq * p.Sq + row_id] = lse_row;
      else if (SPLITKV && p.lse != nullptr)
        p.lse[row_id] = lse_row;
    }
    if (KSPLIT && it.lanesplit) {
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(sm.merge_done());  // lane 1 may now start its next item
      ++mc;
    }
    // The next item's first P.V into O_t waits for this warpgroup's next
    // p_full arrival, which comes after these reads (fence before arrive).
  }
  // mask copies still in flight after an early stop land before the exit
  if (MASK) asm volatile("cp.async.wait_all;" ::: "memory");
}

template <int D, bool BF16, bool SOFTCAP, bool MASK, bool KSPLIT, bool SPLITKV>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc_kernel(const __grid_constant__ TcParams P) {
  using Cfg = TcConfig<D, MASK>;
  const CommonParams& p = P.c;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem<D, MASK> sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm.base);
  sm.sQ = sbase + Cfg::kOffQ;
  sm.sK = sbase + Cfg::kOffK;
  sm.sV = sbase + Cfg::kOffV;
  sm.bar0 = sbase + Cfg::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm.base + Cfg::kOffTmemSlot);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = ((p.Sq + kQTiles * BM - 1) / (kQTiles * BM)) * p.B * p.Hq * p.num_splits;

  if (threadIdx.x == 0) {
    mbar_init(sm.q_full(), 1);
    mbar_init(sm.q_empty(), 1);
    for (int s = 0; s < Cfg::kKStages; ++s) {
      mbar_init(sm.k_full(s), 1);
      mbar_init(sm.k_empty(s), 1);
    }
    for (int s = 0; s < Cfg::kVStages; ++s) {
      mbar_init(sm.v_full(s), 1);
      mbar_init(sm.v_empty(s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(sm.s_full(t), 1);
      mbar_init(sm.p_full(t), 4);  // one arrival per softmax warp of the tile
      mbar_init(sm.o_final(t), 1);
    }
    mbar_init(sm.drain(), 1);
    mbar_init(sm.merge_full(), BM);
    mbar_init(sm.merge_done(), BM);
    mbar_init_fence();
  }
  if (KSPLIT && p.B <= kMaxOrderB) rank_batches(p, reinterpret_cast<int*>(sm.base + Cfg::kOffOrder));
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
    if (lane == 0) producer_role<D, KSPLIT, MASK>(P, sm, n_items);
  } else if (warp == kMmaWarp) {
    mma_role<D, BF16, KSPLIT, MASK>(P, sm, tmem, n_items, lane);
  } else {
    softmax_role<D, BF16, SOFTCAP, MASK, KSPLIT, SPLITKV>(P, sm, tmem, n_items, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16, bool SOFTCAP, bool MASK, bool KSPLIT, bool SPLITKV>
cudaError_t launch_variant(const TcParams& P, cudaStream_t stream) {
  auto kernel = attn_fwd_tc_kernel<D, BF16, SOFTCAP, MASK, KSPLIT, SPLITKV>;
  constexpr uint32_t smem = TcConfig<D, MASK>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t n_items =
      (int64_t)((P.c.Sq + kQTiles * BM - 1) / (kQTiles * BM)) * P.c.B * P.c.Hq * P.c.num_splits;
  if (n_items > INT32_MAX) return cudaErrorInvalidConfiguration;
  const int grid = (int)(n_items < sms ? n_items : sms);  // one persistent CTA per SM
  kernel<<<grid, kThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

template <int D, bool BF16, bool KSPLIT, bool SPLITKV>
cudaError_t launch_k(const TcParams& P, cudaStream_t stream) {
  const bool sc = P.c.softcap > 0.0f;
  const bool mk = P.c.mask != nullptr && P.c.mask_planes > 0;
  if (sc && mk) return launch_variant<D, BF16, true, true, KSPLIT, SPLITKV>(P, stream);
  if (sc) return launch_variant<D, BF16, true, false, KSPLIT, SPLITKV>(P, stream);
  if (mk) return launch_variant<D, BF16, false, true, KSPLIT, SPLITKV>(P, stream);
  return launch_variant<D, BF16, false, false, KSPLIT, SPLITKV>(P, stream);
}

}  // namespace

// One head dim and input type; split into translation units by attn_tc_*.cu.
template <int D, bool BF16>
cudaError_t launch_attn_tc_dd(const TcParams& P, cudaStream_t stream) {
  // Key-split lanes are compiled in only when some item has an empty second
  // query tile: the last query pair holds at most 128 rows.
  const int rem = P.c.Sq - ((P.c.Sq - 1) / (kQTiles * BM)) * (kQTiles * BM);
  const bool ksplit = rem <= BM;
  // split-KV partial rows and the log-sum-exp output only in the variants
  // that need them
  const bool splitkv = P.c.num_splits > 1 || P.c.lse != nullptr;
  if (ksplit) return splitkv ? launch_k<D, BF16, true, true>(P, stream) : launch_k<D, BF16, true, false>(P, stream);
  return splitkv ? launch_k<D, BF16, false, true>(P, stream) : launch_k<D, BF16, false, false>(P, stream);
}

}  // namespace gb300_attn
