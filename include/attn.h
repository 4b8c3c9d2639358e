/*
 * attn.h -- C ABI of libattn.so: tiled online-softmax scaled dot-product
 * attention forward for NVIDIA GB300 (sm_103a).
 *
 * Plain C: every argument is a pointer or a scalar, no C++ or framework
 * types.  All tensor pointers are DEVICE pointers owned by the caller; the
 * library keeps no reference to them after the call returns, allocates no
 * device memory and never synchronises inside attn_fwd.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* a bad size, flag, null pointer or overlapping output      */
    ATTN_ERR_UNSUPPORTED = 2, /* a valid request the library has no kernel for             */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed (see attn_last_cuda_error) */
    ATTN_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait (see attn_get_device_status) */
};

/* Element type of q, k, v and out. */
enum attn_dtype { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 };

/* Layout of out. */
enum attn_out_layout {
    ATTN_OUT_HEAD_MAJOR = 0, /* [B, Hq, Sq, D]                                  */
    ATTN_OUT_TOKEN_MAJOR = 1 /* [B, Sq, Hq*D]: out[(b*Sq + qi)*Hq*D + h*D + d]  */
};

/*
 * attn_fwd -- attention forward for one batch of heads.
 *
 * Defined by "onnx-runtime-ep-cuda 0.1.0-dev.5, src/kernels/flash_attention.rs"
 * (the kernel `flash_attention_body` and the host entry `run`): for every batch
 * b, query head h and query row qi, with kv_head = h / (Hq / Hkv),
 *
 *   lsk        = total_lengths ? total_lengths[b] : Sk
 *   causal_max = past_lengths ? past_lengths[b] + qi : lsk - Sq + qi
 *   local_min  = local_window > 0 ? max(0, causal_max + 1 - local_window) : 0
 *   key j in [0, Sk) is visible iff j < lsk, j >= local_min and
 *                                     (causal == 0 or j <= causal_max)
 *   s_j = scale * <q[b,h,qi,:], k[b,kv_head,j,:]>,
 *         then softcap * tanh(s_j / softcap) when softcap > 0,
 *         then + mask[plane, qi, j] when mask != NULL;
 *   invisible keys get s_j = -inf (a select, never an add);
 *   out[b,h,qi,:] = sum_j softmax(s)_j v[b,kv_head,j,:], or 0 when no key
 *   has a finite score.
 * The token-major layout is the transposed output of "pictor-kernels 0.1.0,
 * src/gpu_backend/cuda_imagen_attn_kernels.rs" (module doc "The op"), with
 * the batch outermost.
 *
 * Arguments (all pointers are device pointers, 16-byte aligned, caller-owned):
 *   q             [B, Hq, Sq, D]            dtype
 *   k, v          [B, Hkv, kv_capacity, D]  dtype; slots j >= min(lsk, Sk) may
 *                                            hold any bits, NaN / Inf included:
 *                                            they never reach the output
 *   mask          NULL or f32 [mask_planes, Sq, Sk] (row stride Sk, 4-byte
 *                 aligned); plane = b when mask_planes == B, b*Hq + h when
 *                 mask_planes == B*Hq, else 0 (mask_planes == 1)
 *   total_lengths NULL or int32 [B] (device): valid cache length per batch
 *   past_lengths  NULL or int32 [B] (device): cached tokens before query row 0
 *   out           output in the chosen layout, dtype; must not overlap q, k, v
 *   B, Sq         >= 0 (0 is an empty problem: OK, nothing written)
 *   Hq, Hkv, D    > 0, Hq % Hkv == 0
 *   Sk            0 <= Sk <= kv_capacity; Sk == 0 writes zeros to out
 *   causal        0 or 1;  local_window <= 0 means no window
 *   scale         finite (callers usually pass 1/sqrt(D))
 *   softcap       finite; <= 0 means no soft-capping
 *   out_layout    enum attn_out_layout
 *   mask_planes   0 (mask must be NULL), 1, B or B*Hq (mask must be non-NULL)
 *   dtype         enum attn_dtype.  ATTN_F32 runs the fp32-exact CUDA-core
 *                 kernel, any 1 <= D <= 384 (the DiT page's kernel is
 *                 compiled up to head dim 384 for its VAE variant, "Kernel
 *                 structure").  ATTN_F16 / ATTN_BF16 run the
 *                 tensor-core (tcgen05) kernels: D must be 64, 128, 256 or
 *                 384 (256 and 384 on attn_fwd only), fp32 accumulation, P
 *                 rounded to the input type before P.V, output rounded to
 *                 nearest even.
 *   stream        a cudaStream_t (NULL = the legacy default stream)
 *
 * Behaviour: validates everything it can see on the host first; on any error
 * it returns the status without launching or writing anything.  On success
 * the work is enqueued on `stream` and the call returns without waiting.
 * It allocates nothing, so it may be captured into a CUDA graph.
 * Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED (D or dtype without a
 * kernel, misaligned pointers or rows), ATTN_ERR_CUDA (launch failure).
 * A kernel that times out on an internal wait is reported by
 * attn_get_device_status, not by this call.
 */
int attn_fwd(const void *q, const void *k, const void *v, const float *mask,
             const int32_t *total_lengths, const int32_t *past_lengths, void *out,
             int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
             int causal, int local_window, float scale, float softcap, int out_layout,
             int mask_planes, int dtype, void *stream);

/*
 * attn_fwd_host -- attn_fwd end to end from host memory: uploads the inputs,
 * runs the attention and downloads the output, with the copies of one piece
 * overlapped with the kernels of its neighbours.  Same operation as attn_fwd
 * (every output element is bit-identical to attn_fwd on the same inputs).
 *
 * The problem is cut into pieces: runs of whole batches, at most 64 pieces,
 * and for ATTN_OUT_HEAD_MAJOR with fewer than eight batches each batch cut
 * further by whole kv-head groups, about eight pieces in all.  When a
 * piece's slices would not start on a 16-byte boundary (fp32 with Sq * D or
 * kv_capacity * D not a multiple of 4) the whole problem is one piece.
 * For each piece, in order: its q / k / v slices (and mask planes) are
 * copied up on an upload stream; one of a few compute streams waits for them
 * and runs attn_fwd on the piece (so the kernels of small pieces can run
 * side by side); a download stream waits for that and copies the piece's
 * output down.  These streams are the library's own (created once per
 * device, kept for the process), forked from and joined back into `stream`.
 * Lengths and a shared mask plane go up first.  Only what can reach the
 * output is uploaded: of each batch's cache rows and mask columns, those
 * j < min(total_lengths[b], Sk) (all Sk when total_lengths is NULL); the
 * other slots of dk / dv / dmask are left as they were.
 *
 * Arguments as attn_fwd, except:
 *   q, k, v, mask, total_lengths, past_lengths, out
 *                 HOST buffers with attn_fwd's shapes (page-locked memory is
 *                 needed for the copies to overlap; pageable memory works,
 *                 serialised).  mask / lengths NULL exactly when their device
 *                 counterparts are NULL.
 *   dq, dk, dv, dmask, dtotal, dpast, dout
 *                 caller-owned DEVICE buffers of the same sizes, the device
 *                 arguments of attn_fwd (alignment and overlap rules as there).
 *   stream        a cudaStream_t: work already on it finishes before the
 *                 device buffers are written, and work queued on it after
 *                 the call is ordered after all of the call's work.
 *   copied_bytes  NULL or uint64_t[2]: on success receives the bytes copied
 *                 host to device and device to host.
 * Behaviour: validates the whole problem as attn_fwd would before touching
 * anything.  BLOCKS until the output is in `out` (and on any error, until
 * nothing it enqueued still runs), so the host buffers may be reused as
 * soon as it returns.  Creates and destroys its own events; allocates no
 * device memory.  Errors as attn_fwd.
 */
int attn_fwd_host(const void *q, const void *k, const void *v, const float *mask,
                  const int32_t *total_lengths, const int32_t *past_lengths, void *out,
                  void *dq, void *dk, void *dv, float *dmask, int32_t *dtotal, int32_t *dpast,
                  void *dout, int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
                  int causal, int local_window, float scale, float softcap, int out_layout,
                  int mask_planes, int dtype, void *stream, uint64_t *copied_bytes);

/*
 * attn_fwd_splitkv -- attn_fwd with each query tile's keys split into
 * `num_splits` contiguous ranges computed by different CTAs, then merged
 * (the flash-decoding arrangement: for decode-like shapes with few query rows
 * and long key ranges).  The result is the same attention output; it can
 * also return each row's log-sum-exp of its scores.
 *
 * The definition is attn_fwd's.  The merge combines ranges r with partial
 * outputs O_r and log-sum-exps L_r as O = sum_r w_r O_r / sum_r w_r,
 * w_r = exp(L_r - max L), L = max L + log sum_r w_r -- the online-softmax
 * rescale of "onnx-runtime-ep-cuda 0.1.0-dev.5, src/kernels/flash_attention.rs"
 * (`flash_attention_body`, alpha / beta update) applied to whole key ranges.
 *
 * Arguments as attn_fwd, plus:
 *   dtype           ATTN_F16 or ATTN_BF16 only (ATTN_F32: ATTN_ERR_UNSUPPORTED),
 *                   with D 64 or 128 (256, 384: ATTN_ERR_UNSUPPORTED)
 *   num_splits      0 = chosen by the library (attn_splitkv_num_splits), else 1..64
 *   lse             NULL or f32 [B, Hq, Sq] device: log sum_j exp(s_j) per row,
 *                   natural log, -inf for rows without a finite score
 *   workspace       device scratch of at least attn_splitkv_workspace_bytes(
 *                   B, Hq, Sq, D, splits) bytes, 16-byte aligned, caller-owned,
 *                   not overlapping any other argument; unused (may be NULL)
 *                   when the split count is 1.  Calls that share a workspace
 *                   must not overlap on the GPU.
 * Launches the attention kernel and, when split, one merge kernel, on
 * `stream`; allocates and synchronises nothing.  The merge kernel is a
 * programmatic dependent of the attention kernel (it may be scheduled while
 * that kernel drains and waits for it in hardware; under stream capture the
 * two are joined by a programmatic graph edge).  Errors as attn_fwd;
 * ATTN_ERR_INVALID_ARG also for a split count outside 0..64 or a missing /
 * too small workspace.
 */
int attn_fwd_splitkv(const void *q, const void *k, const void *v, const float *mask,
                     const int32_t *total_lengths, const int32_t *past_lengths, void *out,
                     int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
                     int causal, int local_window, float scale, float softcap, int out_layout,
                     int mask_planes, int dtype, int num_splits, float *lse, void *workspace,
                     size_t workspace_bytes, void *stream);

/* The split count attn_fwd_splitkv uses for num_splits == 0 on the current
 * device, at most one split per 128-key tile: with (Hq / Hkv) * Sq <= 32 query
 * rows per kv head (the decode kernel) about four CTAs per SM over
 * B * Hkv * splits, otherwise about two query-tile work items per SM. */
int attn_splitkv_num_splits(int B, int Hq, int Hkv, int Sq, int Sk);

/* Workspace bytes attn_fwd_splitkv needs for a split count (0 when <= 1):
 * num_splits * B * Hq * Sq * (D + 1) * 4. */
size_t attn_splitkv_workspace_bytes(int B, int Hq, int Sq, int D, int num_splits);

/*
 * attn_fwd_f32_split -- attn_fwd for fp32 q, k, v, out on the tensor cores.
 *
 * The definition is attn_fwd's, in fp32 as "pictor-kernels 0.1.0,
 * src/gpu_backend/cuda_imagen_attn_kernels.rs" ("Parity-first design") asks
 * of its DiT joint attention. That page keeps the products on CUDA cores and
 * leaves tensor-core tuning for later. This entry runs both products as bf16
 * tcgen05 MMAs with fp32 accumulation, each fp32 operand carried as a sum of
 * bf16 pieces (x0 = bf16(x), x1 = bf16(x - x0), x2 = bf16(x - x0 - x1)):
 *   S = Q K^T   three pieces of Q and K, six products
 *               (q0k0 + q0k1 + q1k0 + q0k2 + q1k1 + q2k0). The dropped terms
 *               are below about 3 * 2^-24 |q k|, so the scores keep fp32
 *               accuracy even where |s| is large.
 *   O = P V     two pieces of P and V (residual <= 2^-16), three products
 *               (p0v0 + p0v1 + p1v0). The output is a P-weighted average of
 *               V, so its error stays near 2^-16 max|v|.
 * The result is held to the fp32 path's 1e-4 bound, including on sharply
 * peaked softmax rows. The fp32-exact CUDA-core kernel stays available as
 * attn_fwd with ATTN_F32.
 *
 * Arguments as attn_fwd with dtype fixed to fp32, plus:
 *   D               64 or 128 (others: ATTN_ERR_UNSUPPORTED)
 *   workspace       device scratch of at least attn_f32_split_workspace_bytes(
 *                   B, Hkv, kv_capacity, D) bytes, 16-byte aligned,
 *                   caller-owned, not overlapping any other argument.  The
 *                   call first writes the bf16 pieces of k (three) and v (two) there (rows
 *                   at or past a batch's valid length as zeros), then runs
 *                   the attention kernel.  Calls that share a workspace must
 *                   not overlap on the GPU.
 * Launches two kernels on `stream`; allocates and synchronises nothing.
 * Errors as attn_fwd; ATTN_ERR_INVALID_ARG also for a missing or too small
 * workspace, or more than 2^31 / 5 key-value planes (B * Hkv).
 */
int attn_fwd_f32_split(const float *q, const float *k, const float *v, const float *mask,
                       const int32_t *total_lengths, const int32_t *past_lengths, float *out,
                       int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
                       int causal, int local_window, float scale, float softcap, int out_layout,
                       int mask_planes, void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes attn_fwd_f32_split needs: 5 * B * Hkv * kv_capacity * D * 2
 * (three bf16 pieces of k, two of v); 0 for non-positive sizes. */
size_t attn_f32_split_workspace_bytes(int B, int Hkv, int kv_capacity, int D);

/*
 * dsa_index_select -- sparse index selection of the DSA indexer.
 *
 * Defined by "onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/dsa_index_select.rs"
 * (module doc and score kernel).  For every batch b, query s and key t:
 *   allowed = bias[b, 0, s, t] > -1e30
 *   score   = sum over heads h = 0..H-1 of
 *               max(scale * sum over d = 0..D-1 of q[b,s,h,d] * k[b,t,d], 0)
 *               * (w[b,s,h] * weights_scale)
 *             + bias[b, 0, s, t]
 * computed in fp32, each multiply and add rounded separately, in exactly
 * that order (d ascending, then h ascending); a NaN score becomes the
 * positive quiet NaN.  out[b, 0, s, :] holds the min(#allowed, top_k)
 * allowed keys with the largest scores (f32 total order: NaN above +inf,
 * -0 below +0; ties to the lower index), in ascending order, then -1s.
 * The scores run on the CUDA cores in that exact order: the result is an
 * index set, and any other rounding could change it.
 *
 * Arguments (device pointers, caller-owned):
 *   query    [B, S, H, D]   dtype;  key [B, T, D] dtype;  weights [B, S, H] dtype
 *   bias     [B, 1, S, T]   f32
 *   out      [B, 1, S, top_k] int64; must not overlap the inputs
 *   B, S, T  >= 0 (B * S == 0: OK, nothing written; T == 0: every slot -1,
 *            and key / bias may be NULL)
 *   H        1..64 (more: ATTN_ERR_UNSUPPORTED);  D >= 1;  top_k >= 1
 *   scale, weights_scale  finite and > 0
 *   dtype    0 f32, 1 f16, 2 bf16 (query, key and weights share it)
 *   workspace  at least dsa_index_select_workspace_bytes(B, S, T) bytes,
 *            16-byte aligned, not overlapping any other argument (the fp32
 *            scores, then a work counter the call zeroes on `stream`); may be
 *            NULL when T == 0.  Calls that share a workspace must not overlap
 *            on the GPU.
 * Enqueues an 8-byte memset (for the counter) and two kernels on
 * `stream`; allocates and synchronises nothing, so it may be captured into
 * a CUDA graph (make one call on the device before capturing: the first call
 * sets kernel attributes and looks up the tensor-map encoder).  The second
 * kernel (the selection) is a programmatic dependent of the first (the
 * scores): it may be scheduled while the first drains and waits for it in
 * hardware before reading a score.
 * Errors: ATTN_ERR_INVALID_ARG (bad size, attribute, dtype, null or
 * overlapping pointer, small workspace), ATTN_ERR_UNSUPPORTED (H > 64,
 * misaligned pointers), ATTN_ERR_CUDA (launch failure).
 */
int dsa_index_select(const void *query, const void *key, const void *weights, const float *bias,
                     int64_t *out, int B, int S, int H, int D, int T, int top_k, float scale,
                     float weights_scale, int dtype, void *workspace, size_t workspace_bytes,
                     void *stream);

/* Workspace bytes dsa_index_select needs: B * S * T * 4 + 256 (0 for non-positive sizes). */
size_t dsa_index_select_workspace_bytes(int B, int S, int T);

/* Size of the library-owned buffer attn_fwd_splitkv_noalloc uses (8 MiB). */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv for callers that cannot
 * allocate device memory when they run attention: runtimes and plugin hosts
 * that plan all device memory ahead of time and forbid allocation during
 * execution, code where a cudaMalloc would synchronise the device or disturb
 * other work, or integrations with no allocator available.  The split-KV
 * scratch lives in a buffer the library owns, ATTN_NOALLOC_SCRATCH_BYTES in
 * size, present on every GPU the library is loaded on until the process
 * exits.  This entry point has no counterpart in the source pages; it is a
 * deployment convenience around the same kernels.
 *
 * Arguments and results as attn_fwd_splitkv, without the workspace.  It calls
 * no cudaMalloc / cudaFree and no allocating library routine.
 *   - Problems whose partial rows need more than ATTN_NOALLOC_SCRATCH_BYTES
 *     (attn_splitkv_workspace_bytes for the split count used) are refused
 *     with ATTN_ERR_INVALID_ARG before anything is launched.
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call uses the same buffer and leaves its partial rows there.
 *     Nothing in it has to start at zero: each call writes every value it
 *     later reads.  Calls that overlap on the GPU (different streams, or
 *     different host threads) race on the buffer; serialise them.
 */
int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, const float *mask,
                             const int32_t *total_lengths, const int32_t *past_lengths, void *out,
                             int B, int Hq, int Hkv, int Sq, int Sk, int kv_capacity, int D,
                             int causal, int local_window, float scale, float softcap,
                             int out_layout, int mask_planes, int dtype, int num_splits,
                             float *lse, void *stream);

/* Human-readable name of a status code; never NULL. */
const char *attn_status_string(int status);

/* The cudaError_t of the last CUDA failure seen by this library on the
 * calling thread (0 if none). */
int attn_last_cuda_error(void);

/*
 * attn_get_device_status -- synchronises `stream`, then reports and clears
 * the device-side status word of the current device: ATTN_ERR_TIMEOUT if any
 * kernel of this library gave up on a bounded wait since the last query,
 * else ATTN_OK (or ATTN_ERR_CUDA if the synchronisation failed).
 */
int attn_get_device_status(void *stream);

/*
 * attn_set_wait_timeout_ns -- limit, in nanoseconds of %globaltimer, after
 * which a kernel stops waiting on an internal barrier, records
 * ATTN_ERR_TIMEOUT and exits.  Applies to launches made after the call.
 * 0 restores the default (2 s).  Returns ATTN_OK.
 * After a timeout the outputs of the launches involved are not valid: rows a
 * kernel could not finish keep what the buffer held before, except rows
 * merged across a thread-block cluster from an unfinished part, which are
 * written as 0 (log-sum-exp -inf) rather than from stale partial results.
 */
int attn_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * attn_selftest_bounded_wait -- launches one small kernel that waits on a
 * shared-memory barrier nobody arrives at, with the given limit, so that the
 * timeout path can be exercised without hanging the GPU.  Synchronises
 * `stream` and returns what attn_get_device_status would: ATTN_ERR_TIMEOUT
 * when the wait ran out as designed.  timeout_ns must be in (0, 1e9].
 */
int attn_selftest_bounded_wait(uint64_t timeout_ns, void *stream);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
