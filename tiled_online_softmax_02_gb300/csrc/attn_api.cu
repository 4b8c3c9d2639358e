// attn_api.cu -- the C ABI of libattn.so (declared in include/attn.h):
// argument validation, tensor-map encoding, kernel dispatch and the device
// status word.
//
// Host entry modelled on `run` of "onnx-runtime-ep-cuda 0.1.0-dev.5,
// src/kernels/flash_attention.rs": a capability gate (unsupported requests
// return a distinct status, never a silent fallback), dtype dispatch, checked
// narrowing of sizes and of the grid, then one launch.  Unlike that host code
// the call is asynchronous (no synchronisation after the launch) and an
// empty key range (Sk == 0) writes zeros instead of leaving the output
// untouched.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/attn.h"
#include "attn_decode.h"
#include "attn_internal.h"
#include "dsa_internal.h"
#include "device_common.cuh"

namespace gb300_attn {
namespace {

__device__ int g_status_word;  // ORed kStatus* bits from every kernel

thread_local int t_last_cuda_error = 0;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return ATTN_ERR_CUDA;
}

// Device address of g_status_word on the current device (looked up once per
// device with that device current).
int* status_ptr(int* err) {
  static std::mutex mu;
  static int* cache[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    *err = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_status_word);
    if (e != cudaSuccess) {
      *err = cuda_fail(e);
      return nullptr;
    }
    cache[dev] = static_cast<int*>(ptr);
  }
  return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(int* err) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static cudaError_t init_err = cudaSuccess;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    init_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                cudaEnableDefault, &q);
    if (init_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else if (init_err == cudaSuccess)
      init_err = cudaErrorSymbolNotFound;
  });
  if (!fn) *err = cuda_fail(init_err);
  return fn;
}

// 16-bit tensor [planes, rows, D] as a 3-D TMA map with a {64, box_rows, 1}
// box and the 128-byte swizzle the tcgen05 shared-memory descriptors expect.
// Rows and planes out of range read as zero.
int encode_map(CUtensorMap* map, const void* base, bool bf16, int64_t planes, int64_t rows, int D,
               int box_rows = kTcBlockM) {
  int err = ATTN_OK;
  auto fn = encode_fn(&err);
  if (!fn) return err;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * (cuuint64_t)D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return ATTN_OK;
}

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > (INT64_C(1) << 62) / a) return false;
  *out = a * b;
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

__global__ void selftest_wait_kernel(uint64_t timeout_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    mbar_init_fence();
  }
  __syncthreads();
  // Nobody arrives on this barrier: the wait must run out and record it.
  if (threadIdx.x == 0) mbar_wait(a, 0, timeout_ns, status);
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t timeout_ns, int* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace gb300_attn

using namespace gb300_attn;

namespace {

constexpr int kMaxSplits = 64;

int tile_count(int Sk) { return (Sk + kTcBlockN - 1) / kTcBlockN; }

int64_t splitkv_rows(int B, int Hq, int Sq) { return (int64_t)B * Hq * Sq; }

// Few query rows per kv head go to the decode kernel (16-bit types).
bool decode_shape(int Hq, int Hkv, int Sq) {
  return Hkv > 0 && Hq % Hkv == 0 && (int64_t)(Hq / Hkv) * Sq <= kDecodeMaxRows;
}

// Thread-block cluster size of the decode kernel when the key tiles are not
// split across launches: enough CTAs for about two waves of two per SM, at
// most 8 (the portable cluster size) and at most one CTA per key tile.
int decode_cluster(int B, int Hkv, int Sk) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t units = (int64_t)B * Hkv;
  int64_t cl = (4 * (int64_t)sms + units - 1) / units;
  if (cl > tile_count(Sk)) cl = tile_count(Sk);
  if (cl > 8) cl = 8;
  return cl < 1 ? 1 : (int)cl;
}

// Split count chosen when the caller passes 0, never more splits than key
// tiles.  Decode kernel: CTAs = B * Hkv * splits, about two waves of two CTAs
// per SM.  Tensor-core kernel: about two work items per SM.
int auto_splits(int B, int Hq, int Hkv, int Sq, int Sk) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t items = decode_shape(Hq, Hkv, Sq)
                            ? (int64_t)B * Hkv
                            : (int64_t)((Sq + 2 * kTcBlockM - 1) / (2 * kTcBlockM)) * B * Hq;
  if (items <= 0) return 1;
  const int64_t target = decode_shape(Hq, Hkv, Sq) ? 4 * (int64_t)sms : 2 * (int64_t)sms;
  int64_t s = (target + items - 1) / items;
  const int tiles = tile_count(Sk);
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : (int)s;
}

int fwd_impl(const void* q, const void* k, const void* v, const float* mask,
             const int32_t* total_lengths, const int32_t* past_lengths, void* out,
             int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
             int causal, int local_window, float scale, float softcap, int out_layout,
             int mask_planes, int dtype, void* stream, bool splitkv_api, int num_splits, float* lse,
             void* workspace, size_t workspace_bytes, bool f32split = false, bool validate_only = false) {
  // ---------------------------------------------------------------- validation
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (B < 0 || Sq < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (Sk < 0 || kv_capacity < Sk) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (out_layout != ATTN_OUT_HEAD_MAJOR && out_layout != ATTN_OUT_TOKEN_MAJOR) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !std::isfinite(softcap)) return ATTN_ERR_INVALID_ARG;
  const int64_t BHq = (int64_t)B * Hq;
  if (mask_planes < 0) return ATTN_ERR_INVALID_ARG;
  if (mask_planes == 0 && mask != nullptr) return ATTN_ERR_INVALID_ARG;
  if (mask_planes > 0) {
    if (mask == nullptr) return ATTN_ERR_INVALID_ARG;
    if (mask_planes != 1 && mask_planes != B && (int64_t)mask_planes != BHq) return ATTN_ERR_INVALID_ARG;
  }
  const int64_t esize = dtype == ATTN_F32 ? 4 : 2;
  int64_t q_elems, kv_elems, mask_elems = 0, t;
  if (!mul_ok(BHq, Sq, &t) || !mul_ok(t, D, &q_elems)) return ATTN_ERR_INVALID_ARG;
  if (!mul_ok((int64_t)B * Hkv, kv_capacity, &t) || !mul_ok(t, D, &kv_elems)) return ATTN_ERR_INVALID_ARG;
  if (mask_planes > 0 && (!mul_ok(mask_planes, Sq, &t) || !mul_ok(t, Sk, &mask_elems)))
    return ATTN_ERR_INVALID_ARG;
  if (q_elems > (INT64_C(1) << 60) / esize || kv_elems > (INT64_C(1) << 60) / esize)
    return ATTN_ERR_INVALID_ARG;
  if (B == 0 || Sq == 0) return ATTN_OK;  // empty problem: nothing to write
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return ATTN_ERR_INVALID_ARG;  // grid.z / grid.y
  if ((int64_t)((Sq + 2 * kTcBlockM - 1) / (2 * kTcBlockM)) * BHq > INT32_MAX)
    return ATTN_ERR_INVALID_ARG;  // work items of the persistent tensor-core kernel
  const int64_t qbytes = q_elems * esize, kvbytes = kv_elems * esize, mbytes = mask_elems * 4;
  const int64_t lenbytes = (int64_t)B * 4;
  // every buffer the call writes (out, and below the log-sum-exp and the
  // workspace) must be disjoint from every buffer it reads
  auto hits_inputs = [&](const void* p, int64_t bytes) {
    return overlaps(p, bytes, q, qbytes) || overlaps(p, bytes, k, kvbytes) || overlaps(p, bytes, v, kvbytes) ||
           overlaps(p, bytes, mask, mbytes) || overlaps(p, bytes, total_lengths, lenbytes) ||
           overlaps(p, bytes, past_lengths, lenbytes);
  };
  if (hits_inputs(out, qbytes)) return ATTN_ERR_INVALID_ARG;

  // capability gate: no kernel, no launch
  if (dtype == ATTN_F32 && D > kF32MaxHeadDim) return ATTN_ERR_UNSUPPORTED;
  if (f32split) {
    if (dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)B * Hkv > INT32_MAX / kF32TcPlanesPerKv) return ATTN_ERR_INVALID_ARG;  // TMA planes
    const size_t need = f32tc_workspace_bytes(kv_elems);
    if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return ATTN_ERR_UNSUPPORTED;
    if (overlaps(workspace, (int64_t)need, out, qbytes) || hits_inputs(workspace, (int64_t)need))
      return ATTN_ERR_INVALID_ARG;
  }
  if (splitkv_api) {
    if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
    if (dtype == ATTN_F32) return ATTN_ERR_UNSUPPORTED;  // split-KV is a tensor-core path
    if (lse && !aligned(lse, 4)) return ATTN_ERR_UNSUPPORTED;
    if (lse && (overlaps(lse, splitkv_rows(B, Hq, Sq) * 4, out, qbytes) ||
                hits_inputs(lse, splitkv_rows(B, Hq, Sq) * 4)))
      return ATTN_ERR_INVALID_ARG;
  }
  // 16-bit: D 64 / 128 on every entry, D 256 / 384 on attn_fwd (the single-lane kernel)
  const bool wide16 = dtype != ATTN_F32 && (D == 256 || D == 384) && !splitkv_api;
  if (dtype != ATTN_F32 && D != 64 && D != 128 && !wide16) return ATTN_ERR_UNSUPPORTED;
  if ((wide16 || f32split) && (int64_t)((Sq + 127) / 128) * BHq > INT32_MAX)
    return ATTN_ERR_INVALID_ARG;  // work items of the single-lane kernel
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return ATTN_ERR_UNSUPPORTED;
  if (mask && !aligned(mask, 4)) return ATTN_ERR_UNSUPPORTED;
  if ((total_lengths && !aligned(total_lengths, 4)) || (past_lengths && !aligned(past_lengths, 4)))
    return ATTN_ERR_UNSUPPORTED;

  if (validate_only) return ATTN_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (Sk == 0) {  // no key at all: every row is 0 (and its log-sum-exp -inf)
    cudaError_t e = cudaMemsetAsync(out, 0, (size_t)qbytes, st);
    if (e == cudaSuccess && lse) e = launch_fill_f32(lse, splitkv_rows(B, Hq, Sq), -INFINITY, st);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
  }
  int splits = 1;
  if (splitkv_api) {
    splits = num_splits == 0 ? auto_splits(B, Hq, Hkv, Sq, Sk) : num_splits;
    if (splits > 1) {
      const size_t need = (size_t)splits * (size_t)splitkv_rows(B, Hq, Sq) * (size_t)(D + 1) * 4;
      if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
      if (!aligned(workspace, 16)) return ATTN_ERR_UNSUPPORTED;
      if (overlaps(workspace, (int64_t)need, out, qbytes) || hits_inputs(workspace, (int64_t)need) ||
          (lse && overlaps(workspace, (int64_t)need, lse, splitkv_rows(B, Hq, Sq) * 4)))
        return ATTN_ERR_INVALID_ARG;
    }
  }

  int err = ATTN_OK;
  int* status = status_ptr(&err);
  if (!status) return err;

  CommonParams c{};
  c.total_lengths = total_lengths;
  c.past_lengths = past_lengths;
  c.mask = mask_planes > 0 ? mask : nullptr;
  c.out = out;
  c.B = B; c.Hq = Hq; c.Hkv = Hkv; c.Sq = Sq; c.Sk = Sk; c.kv_capacity = kv_capacity; c.D = D;
  c.group = Hq / Hkv;
  c.causal = causal;
  c.local_window = local_window > 0 ? local_window : 0;
  c.out_layout = out_layout;
  c.mask_planes = mask_planes;
  c.mask_vec4 = (mask && aligned(mask, 16) && (Sk % 4) == 0) ? 1 : 0;
  c.scale = scale;
  c.scale_log2 = (float)((double)scale * 1.4426950408889634);
  c.softcap = softcap > 0.0f ? softcap : 0.0f;
  c.inv_softcap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
  if (softcap > 0.0f) {
    const double l2e = 1.4426950408889634;
    c.sc_k1 = (float)(2.0 * l2e * (double)scale / (double)softcap);
    c.sc_k2 = (float)(-2.0 * (double)softcap * l2e);
    c.sc_k3 = (float)((double)softcap * l2e);
    c.sc_in = (float)((double)scale / (double)softcap);
    c.sc_out = (float)((double)softcap * l2e);
  }
  c.timeout_ns = g_timeout_ns.load();
  c.status = status;
  c.num_splits = splits;
  c.lse = lse;
  if (splits > 1) {
    c.ws_o = static_cast<float*>(workspace);
    c.ws_lse = c.ws_o + (size_t)splits * (size_t)splitkv_rows(B, Hq, Sq) * D;
  }

  cudaError_t e;
  if (f32split) {
    // K / V pieces in the workspace: k0, k1, k2 then v0, v1, B * Hkv planes each
    LaneParams lp{};
    lp.q = q;
    lp.c = c;
    lp.v_plane0 = 3 * B * Hkv;
    int rc = encode_map(&lp.tmap_k, workspace, true, kF32TcPlanesPerKv * (int64_t)B * Hkv, kv_capacity, D, 64);
    if (rc != ATTN_OK) return rc;
    lp.tmap_v = lp.tmap_k;
    e = launch_attn_f32tc(lp, static_cast<const float*>(k), static_cast<const float*>(v), workspace, st);
  } else if (wide16) {
    const bool bf16 = dtype == ATTN_BF16;
    LaneParams lp{};
    lp.q = q;
    lp.c = c;
    lp.v_plane0 = 0;
    // 64-key tiles; at D = 384 V streams in 16-key units (one box of 16 rows)
    const int v_box = D == 384 ? 16 : 64;
    int rc = encode_map(&lp.tmap_k, k, bf16, (int64_t)B * Hkv, kv_capacity, D, 64);
    if (rc == ATTN_OK) rc = encode_map(&lp.tmap_v, v, bf16, (int64_t)B * Hkv, kv_capacity, D, v_box);
    if (rc == ATTN_OK && D == 384) rc = encode_map(&lp.tmap_q, q, bf16, BHq, Sq, D);  // Q by TMA
    if (rc != ATTN_OK) return rc;
    e = launch_attn_lane16(lp, bf16, st);
  } else if (dtype == ATTN_F32) {
    F32Params fp{};
    fp.q = static_cast<const float*>(q);
    fp.k = static_cast<const float*>(k);
    fp.v = static_cast<const float*>(v);
    fp.c = c;
    e = launch_attn_f32(fp, st);
  } else if (decode_shape(Hq, Hkv, Sq)) {
    const bool bf16 = dtype == ATTN_BF16;
    DecodeParams dp{};
    dp.q = q;
    dp.c = c;
    dp.cluster = splits == 1 ? decode_cluster(B, Hkv, Sk) : 1;
    int rc = encode_map(&dp.tmap_k, k, bf16, (int64_t)B * Hkv, kv_capacity, D);
    if (rc == ATTN_OK) rc = encode_map(&dp.tmap_v, v, bf16, (int64_t)B * Hkv, kv_capacity, D);
    if (rc != ATTN_OK) return rc;
    e = launch_attn_decode(dp, bf16, st);
  } else {
    const bool bf16 = dtype == ATTN_BF16;
    TcParams tp{};
    tp.c = c;
    int rc = encode_map(&tp.tmap_q, q, bf16, BHq, Sq, D);
    if (rc == ATTN_OK) rc = encode_map(&tp.tmap_k, k, bf16, (int64_t)B * Hkv, kv_capacity, D);
    if (rc == ATTN_OK) rc = encode_map(&tp.tmap_v, v, bf16, (int64_t)B * Hkv, kv_capacity, D);
    if (rc != ATTN_OK) return rc;
    e = launch_attn_tc(tp, bf16, st);
  }
  if (dtype != ATTN_F32) {
    const bool bf16 = dtype == ATTN_BF16;
    if (e == cudaSuccess && splits > 1) {
      MergeParams mp{};
      mp.ws_o = c.ws_o;
      mp.ws_lse = c.ws_lse;
      mp.out = out;
      mp.lse = lse;
      mp.B = B; mp.Hq = Hq; mp.Sq = Sq; mp.D = D;
      mp.num_splits = splits;
      mp.out_layout = out_layout;
      mp.bf16 = bf16;
      e = launch_attn_merge(mp, st);
    }
  }
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, const float* mask,
                        const int32_t* total_lengths, const int32_t* past_lengths, void* out,
                        int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
                        int causal, int local_window, float scale, float softcap, int out_layout,
                        int mask_planes, int dtype, void* stream) {
  return fwd_impl(q, k, v, mask, total_lengths, past_lengths, out, B, Hq, Hkv, Sq, Sk, kv_capacity,
                  D, causal, local_window, scale, softcap, out_layout, mask_planes, dtype, stream,
                  false, 1, nullptr, nullptr, 0);
}

// ---------------------------------------------------------------------------
// End-to-end call on host buffers (attn_fwd_host): the problem is cut into
// pieces -- runs of whole batches, at most 64 pieces, and for head-major
// output, with fewer than eight batches, each batch cut further by whole
// kv-head groups -- and the library's own streams overlap piece i + 1's
// upload, piece i's kernel and piece i - 1's download.  Each piece is an ordinary attn_fwd call
// on its slices, so the result is the whole call's bit for bit.  Issuing this
// natively keeps the host's cost per piece to a few microseconds, well under
// a piece's copy time.
namespace {

struct HostPiece {
  int b0, b1, h0, h1, kv0, kv1;
};

constexpr int kMaxHostPieces = 64;
constexpr int kHostComputeStreams = 4;

// The host path's own streams on one device: uploads, downloads, and a few
// compute streams so that the kernels of small pieces (fewer work items than
// SMs) run side by side.  Created on first use, kept for the process.
struct HostStreams {
  cudaStream_t in, out, compute[kHostComputeStreams];
};

HostStreams* host_streams(int* err) {
  static std::mutex mu;
  static HostStreams* cache[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    *err = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    HostStreams hs{};
    cudaStream_t* all[2 + kHostComputeStreams] = {&hs.in, &hs.out};
    for (int i = 0; i < kHostComputeStreams; ++i) all[2 + i] = &hs.compute[i];
    for (int i = 0; i < 2 + kHostComputeStreams; ++i)
      if ((e = cudaStreamCreateWithFlags(all[i], cudaStreamNonBlocking)) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaStreamDestroy(*all[j]);
        *err = cuda_fail(e);
        return nullptr;
      }
    cache[dev] = new HostStreams(hs);
  }
  return cache[dev];
}

int host_pieces(int B, int Hq, int Hkv, int out_layout, HostPiece* pieces) {
  const int group = Hq / Hkv;
  int n = 0;
  if (out_layout == ATTN_OUT_HEAD_MAJOR && B < 8) {
    const int per_batch = std::min(Hkv, (8 + B - 1) / B);
    for (int b = 0; b < B; ++b)
      for (int i = 0; i < per_batch; ++i) {
        const int kv0 = (int)((int64_t)Hkv * i / per_batch), kv1 = (int)((int64_t)Hkv * (i + 1) / per_batch);
        if (kv1 > kv0) pieces[n++] = HostPiece{b, b + 1, kv0 * group, kv1 * group, kv0, kv1};
      }
    return n;
  }
  const int chunks = std::min(B, kMaxHostPieces);
  for (int i = 0; i < chunks; ++i) {
    const int b0 = (int)((int64_t)B * i / chunks), b1 = (int)((int64_t)B * (i + 1) / chunks);
    if (b1 > b0) pieces[n++] = HostPiece{b0, b1, 0, Hq, 0, Hkv};
  }
  return n;
}

}  // namespace

extern "C" int attn_fwd_host(const void* q, const void* k, const void* v, const float* mask,
                             const int32_t* total_lengths, const int32_t* past_lengths, void* out, void* dq,
                             void* dk, void* dv, float* dmask, int32_t* dtotal, int32_t* dpast, void* dout, int B,
                             int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D, int causal,
                             int local_window, float scale, float softcap, int out_layout, int mask_planes,
                             int dtype, void* stream, uint64_t* copied_bytes) {
  if (copied_bytes) copied_bytes[0] = copied_bytes[1] = 0;
  if ((mask == nullptr) != (dmask == nullptr) || (total_lengths == nullptr) != (dtotal == nullptr) ||
      (past_lengths == nullptr) != (dpast == nullptr))
    return ATTN_ERR_INVALID_ARG;
  // the whole problem, as attn_fwd would see it on the device buffers
  int rc = fwd_impl(dq, dk, dv, dmask, dtotal, dpast, dout, B, Hq, Hkv, Sq, Sk, kv_capacity, D, causal,
                    local_window, scale, softcap, out_layout, mask_planes, dtype, stream, false, 1, nullptr,
                    nullptr, 0, false, /*validate_only=*/true);
  if (rc != ATTN_OK) return rc;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;

  const size_t es = dtype == ATTN_F32 ? 4 : 2;
  const size_t q_head = (size_t)Sq * D * es, kv_head = (size_t)kv_capacity * D * es;
  const size_t m_plane = (size_t)Sq * Sk * 4;
  const size_t o_batch = (size_t)Sq * Hq * D * es;
  HostPiece pieces[kMaxHostPieces];
  int n;
  if (q_head % 16 == 0 && kv_head % 16 == 0) {
    n = host_pieces(B, Hq, Hkv, out_layout, pieces);
  } else {  // a piece would start off the 16-byte alignment the kernels need: one piece
    pieces[0] = HostPiece{0, B, 0, Hq, 0, Hkv};
    n = 1;
  }
  const bool per_head_mask = mask != nullptr && (int64_t)mask_planes == (int64_t)B * Hq && Hq > 1;
  const bool per_batch_mask = mask != nullptr && !per_head_mask && mask_planes == B && B > 1;

  HostStreams* hs = host_streams(&rc);
  if (!hs) return rc;
  cudaStream_t cs = static_cast<cudaStream_t>(stream), si = hs->in, so = hs->out;
  uint64_t up_bytes = 0, down_bytes = 0;
  // `height` rows of `width` bytes, `pitch` apart, from host h + off to device d + off
  auto h2d = [&](void* d, const void* h, size_t off, size_t width, size_t pitch, size_t height) {
    if (width == 0 || height == 0) return cudaSuccess;
    up_bytes += (uint64_t)width * height;
    uint8_t* dst = static_cast<uint8_t*>(d) + off;
    const uint8_t* src = static_cast<const uint8_t*>(h) + off;
    if (width == pitch || height == 1)
      return cudaMemcpyAsync(dst, src, width * height, cudaMemcpyHostToDevice, si);
    if (pitch <= (size_t)INT32_MAX)
      return cudaMemcpy2DAsync(dst, pitch, src, pitch, width, height, cudaMemcpyHostToDevice, si);
    for (size_t r = 0; r < height; ++r) {  // pitches past the 2-D copy's limit: one copy per row
      cudaError_t err = cudaMemcpyAsync(dst + r * pitch, src + r * pitch, width, cudaMemcpyHostToDevice, si);
      if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
  };
  // Only keys j < min(lsk, Sk) can be visible (attn_fwd's definition), and
  // the kernels never let a cache slot or mask column past that reach the
  // output: those are not uploaded.
  auto key_rows = [&](int b) -> size_t {
    if (!total_lengths) return (size_t)Sk;
    return (size_t)std::min(std::max(total_lengths[b], 0), Sk);
  };
  cudaEvent_t events[2 * kMaxHostPieces + 3 + kHostComputeStreams];
  int n_events = 0;
  auto new_event = [&](cudaEvent_t* e) {
    cudaError_t err = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    if (err == cudaSuccess) events[n_events++] = *e;
    return err;
  };
  int used_compute = 0;  // compute streams that got a piece
  auto finish = [&](int status) {
    // `stream` joins the internal streams (work queued on it after this call
    // is ordered after all of it) ...
    cudaStream_t mine[2 + kHostComputeStreams] = {si, so};
    for (int i = 0; i < used_compute; ++i) mine[2 + i] = hs->compute[i];
    for (int i = 0; i < 2 + used_compute; ++i) {
      cudaEvent_t j;
      if (new_event(&j) == cudaSuccess && cudaEventRecord(j, mine[i]) == cudaSuccess)
        cudaStreamWaitEvent(cs, j, 0);
    }
    // ... and nothing of this call may still use the caller's buffers when it returns
    for (int i = 0; i < 2 + used_compute; ++i) cudaStreamSynchronize(mine[i]);
    cudaStreamSynchronize(cs);
    for (int i = 0; i < n_events; ++i) cudaEventDestroy(events[i]);
    if (copied_bytes && status == ATTN_OK) {
      copied_bytes[0] = up_bytes;
      copied_bytes[1] = down_bytes;
    }
    return status;
  };
  cudaError_t e;
  cudaEvent_t start;
  // the device buffers may still be in use by earlier work on `stream`
  used_compute = std::min(n, kHostComputeStreams);
  if ((e = new_event(&start)) != cudaSuccess || (e = cudaEventRecord(start, cs)) != cudaSuccess)
    return finish(cuda_fail(e));
  if ((e = cudaStreamWaitEvent(si, start, 0)) != cudaSuccess || (e = cudaStreamWaitEvent(so, start, 0)) != cudaSuccess)
    return finish(cuda_fail(e));
  for (int i = 0; i < used_compute; ++i)
    if ((e = cudaStreamWaitEvent(hs->compute[i], start, 0)) != cudaSuccess) return finish(cuda_fail(e));
  size_t shared_cols = 0;  // a shared mask plane serves every batch: the widest key range
  for (int b = 0; b < B && mask && !per_head_mask && !per_batch_mask; ++b)
    shared_cols = std::max(shared_cols, key_rows(b));
  const size_t m_row = (size_t)Sk * 4;
  if ((total_lengths && (e = h2d(dtotal, total_lengths, 0, (size_t)B * 4, 0, 1)) != cudaSuccess) ||
      (past_lengths && (e = h2d(dpast, past_lengths, 0, (size_t)B * 4, 0, 1)) != cudaSuccess) ||
      (mask && !per_head_mask && !per_batch_mask &&
       (e = h2d(dmask, mask, 0, shared_cols * 4, m_row, (size_t)Sq)) != cudaSuccess))
    return finish(cuda_fail(e));  // lengths, and a mask plane shared by every piece
  int mask_next = 0;  // first batch whose plane has not gone up yet (one plane per batch)
  for (int i = 0; i < n; ++i) {
    const HostPiece& pc = pieces[i];
    const int nb = pc.b1 - pc.b0, hq = pc.h1 - pc.h0, hkv = pc.kv1 - pc.kv0;
    const size_t qo = ((size_t)pc.b0 * Hq + pc.h0) * q_head, ko = ((size_t)pc.b0 * Hkv + pc.kv0) * kv_head;
    const size_t qb = (size_t)nb * hq * q_head;
    float* m_dev = dmask;
    int planes = mask ? 1 : 0;
    size_t mo = 0;
    if (per_head_mask) {
      mo = ((size_t)pc.b0 * Hq + pc.h0) * m_plane;
      planes = nb * hq;
      for (int b = pc.b0; b < pc.b1; ++b)
        if ((e = h2d(dmask, mask, ((size_t)b * Hq + pc.h0) * m_plane, key_rows(b) * 4, m_row,
                     (size_t)hq * Sq)) != cudaSuccess)
          return finish(cuda_fail(e));
    } else if (per_batch_mask) {
      mo = (size_t)pc.b0 * m_plane;
      planes = nb;
      for (int b = std::max(pc.b0, mask_next); b < pc.b1; ++b)  // once per batch, with its first piece
        if ((e = h2d(dmask, mask, (size_t)b * m_plane, key_rows(b) * 4, m_row, (size_t)Sq)) != cudaSuccess)
          return finish(cuda_fail(e));
      mask_next = std::max(mask_next, pc.b1);
    }
    if (mask) m_dev = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(dmask) + mo);
    if ((e = h2d(dq, q, qo, qb, qb, 1)) != cudaSuccess) return finish(cuda_fail(e));
    const size_t row = (size_t)D * es;
    for (int b = pc.b0; b < pc.b1; ++b) {
      const size_t off = ((size_t)b * Hkv + pc.kv0) * kv_head, w = key_rows(b) * row;
      if ((e = h2d(dk, k, off, w, kv_head, (size_t)hkv)) != cudaSuccess ||
          (e = h2d(dv, v, off, w, kv_head, (size_t)hkv)) != cudaSuccess)
        return finish(cuda_fail(e));
    }
    cudaEvent_t up, done;
    if ((e = new_event(&up)) != cudaSuccess || (e = new_event(&done)) != cudaSuccess) return finish(cuda_fail(e));
    cudaStream_t ks = hs->compute[i % kHostComputeStreams];
    if ((e = cudaEventRecord(up, si)) != cudaSuccess || (e = cudaStreamWaitEvent(ks, up, 0)) != cudaSuccess)
      return finish(cuda_fail(e));
    const bool head_major = out_layout == ATTN_OUT_HEAD_MAJOR;
    const size_t oo = head_major ? qo : (size_t)pc.b0 * o_batch, ob = head_major ? qb : (size_t)nb * o_batch;
    rc = fwd_impl(static_cast<uint8_t*>(dq) + qo, static_cast<uint8_t*>(dk) + ko, static_cast<uint8_t*>(dv) + ko,
                  m_dev, dtotal ? dtotal + pc.b0 : nullptr, dpast ? dpast + pc.b0 : nullptr,
                  static_cast<uint8_t*>(dout) + oo, nb, hq, hkv, Sq, Sk, kv_capacity, D, causal, local_window,
                  scale, softcap, out_layout, planes, dtype, ks, false, 1, nullptr, nullptr, 0);
    if (rc != ATTN_OK) return finish(rc);
    if ((e = cudaEventRecord(done, ks)) != cudaSuccess || (e = cudaStreamWaitEvent(so, done, 0)) != cudaSuccess)
      return finish(cuda_fail(e));
    if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(out) + oo, static_cast<const uint8_t*>(dout) + oo, ob,
                             cudaMemcpyDeviceToHost, so)) != cudaSuccess)
      return finish(cuda_fail(e));
    down_bytes += ob;
  }
  return finish(ATTN_OK);
}

extern "C" int attn_fwd_splitkv(const void* q, const void* k, const void* v, const float* mask,
                                const int32_t* total_lengths, const int32_t* past_lengths,
                                void* out, int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity,
                                int D, int causal, int local_window, float scale, float softcap,
                                int out_layout, int mask_planes, int dtype, int num_splits,
                                float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, mask, total_lengths, past_lengths, out, B, Hq, Hkv, Sq, Sk, kv_capacity,
                  D, causal, local_window, scale, softcap, out_layout, mask_planes, dtype, stream,
                  true, num_splits, lse, workspace, workspace_bytes);
}

extern "C" int attn_fwd_f32_split(const float* q, const float* k, const float* v, const float* mask,
                                  const int32_t* total_lengths, const int32_t* past_lengths, float* out,
                                  int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
                                  int causal, int local_window, float scale, float softcap,
                                  int out_layout, int mask_planes, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, mask, total_lengths, past_lengths, out, B, Hq, Hkv, Sq, Sk, kv_capacity,
                  D, causal, local_window, scale, softcap, out_layout, mask_planes, ATTN_F32, stream,
                  false, 1, nullptr, workspace, workspace_bytes, true);
}

extern "C" size_t attn_f32_split_workspace_bytes(int B, int Hkv, int kv_capacity, int D) {
  if (B <= 0 || Hkv <= 0 || kv_capacity <= 0 || D <= 0) return 0;
  return f32tc_workspace_bytes((int64_t)B * Hkv * kv_capacity * D);
}

// ---------------------------------------------------------------------------
// DSA indexer index selection ("onnx-runtime-ep-cuda 0.1.0-dev.6,
// src/kernels/dsa_index_select.rs"): validation, then the score and the
// selection kernels on `stream`.
extern "C" size_t dsa_index_select_workspace_bytes(int B, int S, int T) {
  if (B <= 0 || S <= 0 || T <= 0) return 0;
  return (size_t)B * (size_t)S * (size_t)T * 4 + kDsaCounterBytes;
}

extern "C" int dsa_index_select(const void* query, const void* key, const void* weights, const float* bias,
                                int64_t* out, int B, int S, int H, int D, int T, int top_k, float scale,
                                float weights_scale, int dtype, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (dtype != 0 && dtype != 1 && dtype != 2) return ATTN_ERR_INVALID_ARG;
  if (B < 0 || S < 0 || H <= 0 || D <= 0 || T < 0 || top_k <= 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale <= 0.0f) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(weights_scale) || weights_scale <= 0.0f) return ATTN_ERR_INVALID_ARG;
  const int64_t es = dtype == 0 ? 4 : 2;
  int64_t rows, q_el, k_el, w_el, b_el, o_el, t;
  if (!mul_ok(B, S, &rows) || !mul_ok(rows, H, &t) || !mul_ok(t, D, &q_el)) return ATTN_ERR_INVALID_ARG;
  if (!mul_ok(B, T, &t) || !mul_ok(t, D, &k_el)) return ATTN_ERR_INVALID_ARG;
  if (!mul_ok(rows, H, &w_el) || !mul_ok(rows, T, &b_el) || !mul_ok(rows, top_k, &o_el))
    return ATTN_ERR_INVALID_ARG;
  if (q_el > (INT64_C(1) << 60) / 4 || k_el > (INT64_C(1) << 60) / 4 || b_el > (INT64_C(1) << 60) / 4 ||
      o_el > (INT64_C(1) << 60) / 8)
    return ATTN_ERR_INVALID_ARG;
  if (rows == 0) return ATTN_OK;  // empty problem: nothing to write
  // key and bias hold no element when T == 0 and may then be NULL
  if (!query || !weights || !out || (T > 0 && (!key || !bias))) return ATTN_ERR_INVALID_ARG;
  if (H > 64) return ATTN_ERR_UNSUPPORTED;  // heads are held in registers, up to 64
  const int64_t ws_need = b_el * 4 + (int64_t)kDsaCounterBytes;  // scores, then the unit counter
  if (T > 0 && (!workspace || workspace_bytes < (size_t)ws_need)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(query, es) || !aligned(key, es) || !aligned(weights, es) || !aligned(bias, 4) ||
      !aligned(out, 8) || (T > 0 && !aligned(workspace, 16)))
    return ATTN_ERR_UNSUPPORTED;
  const int64_t ob = o_el * 8;
  if (overlaps(out, ob, query, q_el * es) || overlaps(out, ob, key, k_el * es) ||
      overlaps(out, ob, weights, w_el * es) || overlaps(out, ob, bias, b_el * 4))
    return ATTN_ERR_INVALID_ARG;
  if (T > 0 && (overlaps(workspace, ws_need, out, ob) || overlaps(workspace, ws_need, query, q_el * es) ||
                overlaps(workspace, ws_need, key, k_el * es) || overlaps(workspace, ws_need, weights, w_el * es) ||
                overlaps(workspace, ws_need, bias, b_el * 4)))
    return ATTN_ERR_INVALID_ARG;
  DsaParams dp{};
  dp.query = query;
  dp.key = key;
  dp.weights = weights;
  dp.bias = bias;
  dp.scores = static_cast<float*>(workspace);
  dp.out = out;
  dp.B = B; dp.S = S; dp.H = H; dp.D = D; dp.T = T; dp.top_k = top_k; dp.dtype = dtype;
  dp.scale = scale;
  dp.weights_scale = weights_scale;
  dp.timeout_ns = g_timeout_ns.load();
  dp.neg_zero2 = 0x8000000080000000ull;
  int err = ATTN_OK;
  dp.status = status_ptr(&err);
  if (!dp.status) return err;
  // the TMA-fed score kernel: whole 64-byte chunks of dims, 16-byte aligned
  // rows of q and K, TMA coordinates within range
  dp.tile_path = T > 0 && T <= (1 << 30) && dsa_tile_path_ok(dtype, H, D) && aligned(key, 16) &&
                 aligned(query, 16);
  if (dp.tile_path) {
    // the counter sits 16-byte aligned after the scores; zeroed on the stream
    const size_t off = ((size_t)b_el * 4 + 15) & ~(size_t)15;
    dp.unit_counter = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + off);
    const cudaError_t me = cudaMemsetAsync(dp.unit_counter, 0, sizeof(unsigned long long),
                                           static_cast<cudaStream_t>(stream));
    if (me != cudaSuccess) return cuda_fail(me);
    int rc = ATTN_OK;
    auto fn = encode_fn(&rc);
    if (!fn) return rc;
    if (dsa_encode_key_map(&dp.tmap_key, reinterpret_cast<void*>(fn), key, dtype, B, T, D) != 0)
      return cuda_fail(cudaErrorInvalidValue);
    if (rc != ATTN_OK) return rc;
  }
  const cudaError_t e = launch_dsa_select(dp, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

extern "C" int attn_splitkv_num_splits(int B, int Hq, int Hkv, int Sq, int Sk) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0) return 1;
  return auto_splits(B, Hq, Hkv, Sq, Sk);
}

extern "C" size_t attn_splitkv_workspace_bytes(int B, int Hq, int Sq, int D, int num_splits) {
  if (B <= 0 || Hq <= 0 || Sq <= 0 || D <= 0 || num_splits <= 1) return 0;
  return (size_t)num_splits * (size_t)splitkv_rows(B, Hq, Sq) * (size_t)(D + 1) * 4;
}

extern "C" const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_UNKNOWN_STATUS";
  }
}

extern "C" int attn_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int attn_get_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  if (word != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return (word & kStatusTimeout) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

extern "C" int attn_set_wait_timeout_ns(uint64_t timeout_ns) {
  g_timeout_ns.store(timeout_ns == 0 ? 2000000000ull : timeout_ns);
  return ATTN_OK;
}

extern "C" int attn_selftest_bounded_wait(uint64_t timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return ATTN_ERR_INVALID_ARG;
  int err = ATTN_OK;
  int* status = status_ptr(&err);
  if (!status) return err;
  cudaError_t e = launch_selftest_wait(timeout_ns, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return attn_get_device_status(stream);
}

extern "C" int attn_version(void) { return 100; }

// ---------------------------------------------------------------------------
// Allocation-free split-KV entry point.
//
// Some callers cannot allocate device memory at the point where they run
// attention: inference runtimes and plugin hosts that plan all device memory
// ahead of time and forbid allocation while executing, code running inside a
// region where cudaMalloc would synchronise the device or disturb other work,
// or embedded integrations with no allocator at hand.  For them this entry
// point keeps the split-KV scratch in a fixed buffer that the library itself
// owns.  The buffer below lives in every GPU's memory once the library is
// loaded on it, until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch on the current device.  Host code may
// not use the symbol itself as a device pointer, so it is looked up once per
// device, with that device current, and cached.
void* noalloc_scratch(int* err) {
  static std::mutex mu;
  static void* cache[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    *err = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = cuda_fail(e);
      return nullptr;
    }
    cache[dev] = ptr;
  }
  return cache[dev];
}

}  // namespace

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v,
                                        const float* mask, const int32_t* total_lengths,
                                        const int32_t* past_lengths, void* out, int B, int Hq,
                                        int Hkv, int Sq, int Sk, int kv_capacity, int D,
                                        int causal, int local_window, float scale, float softcap,
                                        int out_layout, int mask_planes, int dtype, int num_splits,
                                        float* lse, void* stream) {
  // Problems whose partial rows do not fit the fixed buffer are refused up
  // front, before anything is launched.
  if (B > 0 && Hq > 0 && Hkv > 0 && Sq > 0 && Sk > 0 && D > 0 && num_splits >= 0 &&
      num_splits <= kMaxSplits) {
    const int splits = num_splits == 0 ? auto_splits(B, Hq, Hkv, Sq, Sk) : num_splits;
    if (attn_splitkv_workspace_bytes(B, Hq, Sq, D, splits) > (size_t)ATTN_NOALLOC_SCRATCH_BYTES)
      return ATTN_ERR_INVALID_ARG;
  }
  int err = ATTN_OK;
  void* scratch = noalloc_scratch(&err);
  if (!scratch) return err;
  return fwd_impl(q, k, v, mask, total_lengths, past_lengths, out, B, Hq, Hkv, Sq, Sk, kv_capacity,
                  D, causal, local_window, scale, softcap, out_layout, mask_planes, dtype, stream,
                  true, num_splits, lse, scratch, (size_t)ATTN_NOALLOC_SCRATCH_BYTES);
}
