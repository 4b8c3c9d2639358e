// device_common.cuh -- device-side building blocks shared by the attention
// kernels of this library: per-row visibility limits, bounded mbarrier waits,
// TMA loads and the tcgen05 (5th-generation tensor core / tensor memory)
// instructions, written as inline PTX for sm_103a.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "attn_internal.h"

namespace gb300_attn {

// ---------------------------------------------------------------------------
// Per-row limits.  "onnx-runtime-ep-cuda 0.1.0-dev.5,
// src/kernels/flash_attention.rs", kernel `flash_attention_body`: the valid
// length lsk, the causal bound causal_max (from past_lengths, else aligned to
// the end of the valid keys) and the window lower bound local_min.  A key j
// is visible to row qi iff lo <= j < hi with
//   lo = local_min,  hi = min(lsk, Sk, causal ? causal_max + 1 : +inf).
// Rows outside [0, Sq) see nothing.  64-bit arithmetic throughout.
// ---------------------------------------------------------------------------
struct RowLimits {
  int lo, hi;  // visible keys are [lo, hi), 0 <= lo <= hi <= Sk (empty when equal)
};

struct BatchLimits {
  int64_t lsk;          // total_lengths[b] or Sk (unclamped, as on the page)
  int64_t causal_base;  // causal_max = causal_base + qi
};

__device__ __forceinline__ BatchLimits batch_limits(const CommonParams& p, int b) {
  BatchLimits L;
  L.lsk = p.total_lengths ? (int64_t)__ldg(p.total_lengths + b) : (int64_t)p.Sk;
  L.causal_base = p.past_lengths ? (int64_t)__ldg(p.past_lengths + b) : L.lsk - (int64_t)p.Sq;
  return L;
}

__device__ __forceinline__ RowLimits row_limits(const CommonParams& p, const BatchLimits& L,
                                                int64_t qi) {
  const int64_t causal_max = L.causal_base + qi;
  int64_t lo = 0;
  if (p.local_window > 0) {
    lo = causal_max + 1 - (int64_t)p.local_window;
    if (lo < 0) lo = 0;
  }
  int64_t hi = L.lsk < (int64_t)p.Sk ? L.lsk : (int64_t)p.Sk;
  if (p.causal && causal_max + 1 < hi) hi = causal_max + 1;
  if (qi < 0 || qi >= (int64_t)p.Sq) hi = lo;  // rows past Sq see nothing
  // clamp into [0, Sk] (keeps the visible set; fits 32 bits)
  if (lo > (int64_t)p.Sk) lo = p.Sk;
  if (hi < lo) hi = lo;
  RowLimits r;
  r.lo = (int)lo;
  r.hi = (int)hi;
  return r;
}

// Key-tile range [t_begin, t_end) of tiles of `bn` keys that a block of query
// rows [q0, q0 + bm) must visit, plus the range of tiles where every row in
// the block sees every key (no per-element masking needed there).  lo and hi
// are non-decreasing in qi, so the extremes come from the first and last row.
struct TileRange {
  int t_begin, t_end;  // tiles to visit
  int full_lo, full_hi;  // keys [full_lo, full_hi) visible to every row
};

__device__ __forceinline__ TileRange tile_range(const CommonParams& p, const BatchLimits& L,
                                                int64_t q0, int bm, int bn) {
  TileRange t;
  int64_t q_last = q0 + bm - 1;
  if (q_last >= (int64_t)p.Sq) q_last = (int64_t)p.Sq - 1;
  const RowLimits first = row_limits(p, L, q0);
  const RowLimits last = row_limits(p, L, q_last);
  // union of the visible ranges of all rows (rows with an empty range included
  // in the bounds is harmless: their scores are all masked)
  const int lo = first.lo;
  const int hi = last.hi;
  if (hi <= lo || q0 >= (int64_t)p.Sq) {
    t.t_begin = t.t_end = 0;
  } else {
    t.t_begin = (int)(lo / bn);
    t.t_end = (int)((hi + bn - 1) / bn);
  }
  // keys every row sees: [max lo, min hi) = [last.lo, first.hi)
  t.full_lo = last.lo;
  t.full_hi = first.hi;
  return t;
}

// ---------------------------------------------------------------------------
// Status word.  A kernel that gives up on a bounded wait ORs this bit into the
// device status word the host reads back (attn_get_device_status).
// ---------------------------------------------------------------------------
constexpr int kStatusTimeout = 1;

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

// ---------------------------------------------------------------------------
// mbarrier (shared memory barrier objects)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Optional suspend-time hint for try_wait (ns).  0 (the default) uses the
// plain form, whose suspension limit the hardware picks.
#ifndef GB300_WAIT_HINT_NS
#define GB300_WAIT_HINT_NS 0
#endif

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
#if GB300_WAIT_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"((uint32_t)GB300_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

// Waits until the phase with the given parity of barrier `bar` completes.
// Gives up after `timeout_ns` of %globaltimer: records the timeout in the
// status word and returns false.  Every wait in this library goes through
// here, so no kernel can spin forever.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u && global_timer_ns() - t0 > timeout_ns) {
      if (status) atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// Warp-collective form: every lane waits, and the warp agrees on the outcome,
// so a timeout can never split a warp in front of a .sync.aligned instruction.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                               int* status) {
  const bool ok = mbar_wait(bar, parity, timeout_ns, status);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// L2 eviction policies (createpolicy) for the cache-hinted accesses below:
// lines loaded as evict_last stay in L2 ahead of lines marked evict_first,
// so tiles read many times (K / V) outlive data streamed once (Q, O).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// tma_load_3d with an L2 cache policy
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1,
                                                 int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
// 16-byte read-only load / store with an L2 cache policy
__device__ __forceinline__ uint4 ld_nc_hint(const void* ptr, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(policy));
  return v;
}
__device__ __forceinline__ void st_hint(void* ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}
// Bulk prefetch of [src, src + bytes) into L2 (no completion to wait for);
// src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA, commit, loads / stores
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives once on `bar` when every tcgen05 async operation this thread issued
// so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Warp-collective forms: every lane of the warp executes the call and one
// lane, chosen by elect.sync (the lowest active lane, so always the same one
// for a converged warp), issues the instruction.  Keeping the issuing warp
// converged matters on this GPU: issued from a one-lane divergent branch,
// MMAs started up to three times slower whenever other warps of the same SM
// sub-partition had arithmetic ready to issue (the softmax warps).
__device__ __forceinline__ void mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %4, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Several MMAs into one accumulator from one asm block and one elect.sync:
// the issuing lane then needs no further issue slots between them, which
// keeps MMAs back to back even while other warps of the sub-partition issue
// (N = 64 MMAs: 32 cycles each this way, 39 when issued one asm block at a
// time next to one arithmetic-heavy warp).  The first MMA accumulates iff
// acc0 != 0, the others always.
__device__ __forceinline__ void mma_ss4_elect(uint32_t d, uint64_t a0, uint64_t b0, uint64_t a1, uint64_t b1,
                                              uint64_t a2, uint64_t b2, uint64_t a3, uint64_t b3,
                                              uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %10, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %9, q;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %9, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %9, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %9, 1;\n\t}" ::"r"(d),
      "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc), "r"(acc0)
      : "memory");
}

// Four MMAs with A in tensor memory (addresses a_i).
__device__ __forceinline__ void mma_ts4_elect(uint32_t d, uint32_t a0, uint64_t b0, uint32_t a1, uint64_t b1,
                                              uint32_t a2, uint64_t b2, uint32_t a3, uint64_t b3,
                                              uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %10, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %9, q;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %9, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %9, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %9, 1;\n\t}" ::"r"(d),
      "r"(a0), "l"(b0), "r"(a1), "l"(b1), "r"(a2), "l"(b2), "r"(a3), "l"(b3), "r"(idesc), "r"(acc0)
      : "memory");
}

// Six MMAs with A in tensor memory.
__device__ __forceinline__ void mma_ts6_elect(uint32_t d, uint32_t a0, uint64_t b0, uint32_t a1, uint64_t b1,
                                              uint32_t a2, uint64_t b2, uint32_t a3, uint64_t b3,
                                              uint32_t a4, uint64_t b4, uint32_t a5, uint64_t b5,
                                              uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "setp.ne.b32 q, %14, 0;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %13, q;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %13, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %13, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %13, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %13, 1;\n\t"
      "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%11], %12, %13, 1;\n\t}" ::"r"(d),
      "r"(a0), "l"(b0), "r"(a1), "l"(b1), "r"(a2), "l"(b2), "r"(a3), "l"(b3), "r"(a4), "l"(b4),
      "r"(a5), "l"(b5), "r"(idesc), "r"(acc0)
      : "memory");
}

// tc_commit by the elected lane (the lane that issued the warp's MMAs).
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Instruction descriptor of tcgen05.mma .kind::f16 (dense, fp32 accumulator):
// bits 4-5 D format (1 = f32), 7-9 A format and 10-12 B format (0 = f16,
// 1 = bf16), 15 / 16 A / B major-ness (0 = K-major, 1 = MN-major),
// 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_f16kind(bool bf16, int M, int N, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand:
// bits 0-13 start address >> 4, 16-29 leading-dimension byte offset >> 4,
// 32-45 stride-dimension byte offset >> 4, 46-47 = 1 (descriptor version),
// 49-51 base offset (0: tiles are 1024-byte aligned), 61-63 = 2 (128B swizzle).
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                     uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

#define GB300_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                    "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define GB300_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                    "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM
// lane (lane = warp's lane quarter base + lane id).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : GB300_R8(0), GB300_R8(8), GB300_R8(16), GB300_R8(24)
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      GB300_W8(0), GB300_W8(8), GB300_W8(16), GB300_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      GB300_W8(0), GB300_W8(8)
      : "memory");
}

#undef GB300_R8
#undef GB300_W8

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Math helpers (hardware instructions)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (sm_100+ f32x2 arithmetic): one instruction does two
// lanes' worth of FMA / ADD / MUL, which halves the issue slots the softmax
// warps take from the MMA-issuing warp on the same SM sub-partition.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// max / min of three (one instruction on sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Hardware tanh (one MUFU op; relative error about 2^-11).
__device__ __forceinline__ float fast_tanh(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// c * tanh(s / c) through tanh(y) = 1 - 2 / (2^(2 y log2 e) + 1): one ex2 and
// one reciprocal; exact limits +-c for |y| -> inf, absolute error ~1e-7 * c.
// The same soft-cap on a raw score s, returned in log2 units, with the
// constants folded (see CommonParams::sc_k*): one FMUL, ex2, FADD, rcp, FFMA.
__device__ __forceinline__ float soft_cap_log2(float s, float k1, float k2, float k3) {
  return fmaf(k2, fast_rcp(fast_exp2(s * k1) + 1.0f), k3);
}

__device__ __forceinline__ float soft_cap(float s, float cap, float inv_cap) {
  const float e = fast_exp2(s * inv_cap * 2.8853900817779268f);  // 2 * log2(e)
  return cap * (1.0f - 2.0f * fast_rcp(e + 1.0f));
}

}  // namespace gb300_attn
