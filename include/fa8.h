/*
 * fa8.h -- C ABI of the GB300 (sm_103a) fused FP8 attention forward.
 *
 *   O   = softmax( softmax_scale * dq * dk * Q K^T  [+ causal / left-window mask]
 *                  [+ learnable sink in the denominator] ) * V * dv
 *   LSE = natural-log log-sum-exp of the masked, scaled scores (and the sink)
 *
 * with Q, K, V in E4M3, O in bf16 or fp16 and LSE in fp32.
 *
 * Where the operation is defined (page title, section):
 *  - "PyTorch ... FlashAttention-4 MXFP8", 2.1 Attention Forward: S = Q K^T,
 *    P = softmax(S), O = P V.
 *  - "[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward for Hopper":
 *    Design/"Descales" (q/k descales fold into the softmax scale, v descale into the
 *    final normalisation; each 0-d or (batch, kv_heads)); Design/"Paged K/V";
 *    Design/"Decode launches" (host-known launch choices); "Supported" (head dims,
 *    causal, sliding window, varlen, paged K/V, PackGQA, SplitKV, learnable sink,
 *    fp16/bf16 output) and "Rejected with an error" (E5M2, mixed dtypes).
 *  - "tml-fa4 PR #4", Summary: P carries a 2^8 bias that cancels in the O
 *    normalisation and is removed from the LSE.
 *
 * Every pointer argument is owned by the caller.  The library keeps no pointer after
 * a call returns other than inside the work it enqueued on `stream`.  Arguments are
 * validated on the host before anything is enqueued; on an error nothing is enqueued,
 * a status code is returned and fa8_last_error() gives a one-line reason.
 */
#ifndef FA8_H_
#define FA8_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA8_VERSION 100 /* 1.0.0 */

#if defined(__GNUC__)
#define FA8_API __attribute__((visibility("default")))
#else
#define FA8_API
#endif

typedef enum {
    FA8_SUCCESS = 0,
    FA8_ERR_INVALID_ARG = 1,    /* malformed shape, stride, pointer or flag           */
    FA8_ERR_UNSUPPORTED = 2,    /* well-formed but not implemented (e.g. E5M2, d=80)  */
    FA8_ERR_WORKSPACE = 3,      /* split-KV workspace missing or too small            */
    FA8_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed                  */
    FA8_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up a bounded wait (see fa8_check)    */
    FA8_ERR_DEVICE_BOUNDS = 6   /* a kernel saw a block-table entry out of range      */
} fa8_status;

typedef enum {
    FA8_DTYPE_E4M3 = 1, /* float8_e4m3fn */
    FA8_DTYPE_E5M2 = 2, /* float8_e5m2 (rejected as Q/K/V) */
    FA8_DTYPE_BF16 = 3,
    FA8_DTYPE_F16 = 4,
    FA8_DTYPE_F32 = 5,
    FA8_DTYPE_I32 = 6
} fa8_dtype;

/*
 * A strided view of device memory.  `stride` is in elements; unused trailing entries of
 * `shape`/`stride` are ignored.  A 0-d tensor has ndim == 0.
 */
typedef struct {
    void *data;
    int32_t dtype; /* fa8_dtype */
    int32_t ndim;  /* 0..4 */
    int64_t shape[4];
    int64_t stride[4];
} fa8_tensor;

/*
 * fa8_fwd -- enqueue the fused FP8 attention forward on `stream` (a cudaStream_t).
 *
 * Layouts (the last dimension is always contiguous):
 *   q   batched (B, Sq, Hq, D)            or varlen (total_q, Hq, D) with cu_seqlens_q
 *   k   batched (B, Sk, Hkv, D)           or varlen (total_k, Hkv, D) with cu_seqlens_k
 *       or paged (num_pages, page_size, Hkv, D) with block_table and cu_seqlens_k
 *   v   as k with DV in place of D
 *   out like q with DV in place of D; bf16 or fp16
 *   lse batched (B, Hq, Sq) or varlen (Hq, total_q); fp32; may be NULL
 * Q/K/V are E4M3 (E5M2 or mixed dtypes -> FA8_ERR_UNSUPPORTED).  (D, DV) is one of
 * (64,64), (96,96), (128,128), (192,128), (192,192), (256,256).  Hq % Hkv == 0 and Hq/Hkv <= 128;
 * q-head h reads kv-head h / (Hq/Hkv).  Row strides of q/k/v must be multiples of 16
 * bytes and their base pointers 16-byte aligned (they are read by TMA).
 *
 * cu_seqlens_q / cu_seqlens_k: int32 (B+1) prefix sums of the per-request query / key
 *   lengths.  For paged K/V, cu_seqlens_k gives each request's key count (its
 *   differences); keys are read only from the first ceil(len/page_size) entries of the
 *   request's block_table row.
 * block_table: int32 (B, max_pages), stride(1) == 1, entries are page indices into
 *   k/v dim 0.  page_size must equal k.shape[1] and be a multiple of 8.
 *   Entries out of range read as zeros (TMA bounds) and raise FA8_ERR_DEVICE_BOUNDS in
 *   fa8_check; they never make the kernel touch memory outside k/v.
 * descale_q/k/v: fp32, 0-d or (B, Hkv) with any strides (0 = broadcast); NULL = 1.0.
 *   They must be positive.
 * sink: fp32 (Hq,) natural-log logits added to every row's denominator; NULL = none.
 * causal: 0/1, bottom-right aligned (key j visible to query i when j <= i + Lk - Lq).
 * window_left: -1 = unbounded, else keys j >= i + Lk - Lq - window_left stay visible.
 * softmax_scale: <= 0 selects 1/sqrt(D).
 * num_splits: 0 = heuristic, 1 = no split, n > 1 = launch n splits of each tile's key
 *   range and merge them with a second kernel.  The launch depends only on shapes and the
 *   device's SM count, never on device values, so a call can be graph-captured.  On the
 *   device, a tile whose visible keys span t KV tiles of 128 keys runs
 *   min(n, max(1, ceil(t / cap))) of the launched splits; the other splits exit at once and
 *   the merge does not read them.  cap (2 to 512 KV tiles per split) is chosen once per
 *   call from the requests' key counts: the choice that minimises a model of the run time
 *   (a fixed cost per work unit, the units spread over the CTAs that run at once, and the
 *   longest unit's tail).  The heuristic launches about eight waves of CTAs, or one wave
 *   when there are few (query tile, kv-head) pairs; when every launched split fits in one
 *   wave the finest cap is used, and with dense K/V and batched q (every length known from
 *   the shapes) the host chooses the cap and launches only the splits that run.
 * workspace / workspace_bytes: device scratch for the split partials and the split cap the
 *   forward kernel passes to the merge kernel, at least fa8_fwd_workspace_size() bytes
 *   (may be NULL/0 when that size is 0).
 */
FA8_API fa8_status fa8_fwd(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v,
                   const fa8_tensor *descale_q, const fa8_tensor *descale_k,
                   const fa8_tensor *descale_v, fa8_tensor *out, fa8_tensor *lse,
                   const fa8_tensor *cu_seqlens_q, const fa8_tensor *cu_seqlens_k,
                   const fa8_tensor *block_table, int page_size, int causal, int window_left,
                   const fa8_tensor *sink, float softmax_scale, int num_splits,
                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * fa8_fwd_workspace_size -- validates the shape arguments of fa8_fwd (no data is read)
 * and reports the split count fa8_fwd would use and the workspace it needs.
 * Either output pointer may be NULL.
 */
FA8_API fa8_status fa8_fwd_workspace_size(const fa8_tensor *q, const fa8_tensor *k,
                                  const fa8_tensor *v, const fa8_tensor *cu_seqlens_q,
                                  const fa8_tensor *cu_seqlens_k, const fa8_tensor *block_table,
                                  int page_size, int num_splits, int *splits_out,
                                  size_t *bytes_out);

/*
 * fa8_fwd_plan -- the launch plan fa8_fwd would use on a device with `sm_count` SMs,
 * computed on the host only (no CUDA call): the split count, the workspace bytes and the
 * forward's work grid (grid_out[0] = Q-tile slots, grid_out[1] = kv_heads x splits; the
 * prefill kernel for dv <= 128 is persistent and walks these units with min(units, SMs)
 * CTAs).  It runs the same shape validation as fa8_fwd.  Any output pointer may be NULL.
 */
FA8_API fa8_status fa8_fwd_plan(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v,
                                const fa8_tensor *cu_seqlens_q, const fa8_tensor *cu_seqlens_k,
                                const fa8_tensor *block_table, int page_size, int num_splits,
                                int sm_count, int *splits_out, size_t *bytes_out,
                                int64_t *grid_out);

/*
 * fa8_fwd_static_scratch -- fa8_fwd without a caller-provided workspace.  The attention
 * it computes is fa8_fwd's, argument for argument; nothing in the published method
 * corresponds to this entry point, which only changes where the split partials live.
 *
 * Who it is for: callers that cannot hand the library a device buffer -- a runtime whose
 * device memory is carved up once at start-up and that may not allocate afterwards, or
 * plain C code that links only this library and has no allocator of its own.  Neither
 * this function nor anything it calls allocates or frees device memory.
 *
 * Where the partials go: one array of FA8_STATIC_SCRATCH_BYTES (32 MiB) of device memory
 * that the library declares statically, so it exists once per device for as long as the
 * library is loaded.  A call whose split plan (see fa8_fwd_workspace_size) needs more
 * than that returns FA8_ERR_WORKSPACE before anything is enqueued; lower num_splits or
 * use fa8_fwd with a workspace of your own.  Calls whose plan has one split do not touch
 * the array.  Nothing in it has to start at zero: every call writes each partial before
 * the merge kernel reads it.
 *
 * Sharing: every call on a device uses the same array.  Two calls that can run at the
 * same time on one device (different streams without an event between them, or different
 * host threads) overwrite each other's partials and give wrong results; order them on one
 * stream, or use fa8_fwd with separate workspaces.
 *
 * Set-up: the first call on each device, made with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and keeps it; make that first call
 * before capturing a stream.  A failure there returns FA8_ERR_CUDA.
 */
#define FA8_STATIC_SCRATCH_BYTES ((size_t)32 * 1024 * 1024)
FA8_API fa8_status fa8_fwd_static_scratch(const fa8_tensor *q, const fa8_tensor *k,
                                          const fa8_tensor *v, const fa8_tensor *descale_q,
                                          const fa8_tensor *descale_k,
                                          const fa8_tensor *descale_v, fa8_tensor *out,
                                          fa8_tensor *lse, const fa8_tensor *cu_seqlens_q,
                                          const fa8_tensor *cu_seqlens_k,
                                          const fa8_tensor *block_table, int page_size,
                                          int causal, int window_left, const fa8_tensor *sink,
                                          float softmax_scale, int num_splits, void *stream);

/*
 * fa8_check -- reads the library's device status word of the current device on `stream`
 * (ordered after the work enqueued there), waits for that read, and clears the word if it
 * was set: FA8_SUCCESS, FA8_ERR_DEVICE_TIMEOUT (a kernel gave up a bounded wait and
 * returned early; its outputs are undefined) or FA8_ERR_DEVICE_BOUNDS.
 *
 * The status word is one per device, shared by every stream and host thread that calls the
 * library on that device: a kernel on any stream sets its bits, and a check on any stream
 * reads and clears them all.  So a check may report (and clear) an error raised by another
 * stream's work, and work still running on another stream may set the word after the read.
 * Callers that run forwards on several streams at once and need to know which call failed
 * should check from one place after joining the streams.
 */
FA8_API fa8_status fa8_check(void *stream);

/*
 * fa8_set_decode_kernel -- 1 (the default): shapes with batched q and at most 16 query rows
 * per kv-head (Sq x Hq/Hkv <= 16, Hq/Hkv dividing 16, dv a multiple of 128) run the decode
 * kernel, which puts the keys of a tile on the MMA's M dimension and the few query rows on
 * N; 0: every shape runs the 128-row forward kernel.  Both compute the same attention (not
 * bit-identically).  A process-wide setting, safe to change from any host thread: each
 * fa8_fwd call reads it once, so one call uses one setting throughout.
 */
FA8_API fa8_status fa8_set_decode_kernel(int enable);

/* Sets the bound on every in-kernel wait (nanoseconds; default 2e9, minimum 1e5); a
 * process-wide setting, read once by each later fa8_fwd call, safe from any host thread. */
FA8_API fa8_status fa8_set_wait_timeout_ns(uint64_t ns);

/*
 * fa8_debug_wait_probe -- DEBUG ONLY.  Launches a one-CTA kernel whose only work is a bounded wait on a
 * barrier that nothing completes, then returns fa8_check(stream).  It exists to test the
 * timeout path: with the default bound it returns FA8_ERR_DEVICE_TIMEOUT after ~2 s.
 */
FA8_API fa8_status fa8_debug_wait_probe(void *stream);

/*
 * fa8_debug_set_trace_buffer -- in a library built with -DFA8_TRACE, later forward launches
 * record clock64() at each pipeline event (TMA issue, MMA issue, softmax and fold
 * hand-offs) of the first 8 CTAs into `device_buffer`, laid out [cta 8][event 16][tile 64]
 * as uint64 (needs 65536 bytes); NULL turns it off.  Other builds return
 * FA8_ERR_UNSUPPORTED.  DEBUG ONLY: for pipeline tuning with a trace build; production
 * builds do not record anything.
 */
FA8_API fa8_status fa8_debug_set_trace_buffer(void *device_buffer, size_t bytes);

FA8_API const char *fa8_status_string(fa8_status s);
/* Reason for the last error returned on the calling thread ("" if none). */
FA8_API const char *fa8_last_error(void);
FA8_API int fa8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA8_H_ */
