/*
 * psa_attn.h -- C ABI of the GB300 (sm_103a) PSA self-attention library.
 *
 * PSA attention runs two softmax-attention calls, "lo" and "hi", over one
 * packed per-(batch, head) buffer.  The calls share the Q and K sections, and
 * each owns one V section ("Struct PsaFa2Backward", vision_rs yolo attention
 * psa page: description and "Atomicity" paragraphs).  It is self-attention:
 * the query and key counts are both N (same page, description).  Because the
 * two calls share Q, K and therefore one softmax P, this library runs them as
 * ONE attention with a 2d-wide value [V_lo | V_hi]; the gradients it returns are
 * exactly those of the two calls, with dQ and dK summed over both.
 *
 * Notation, per (b, h) slice, all matrices [N, d] row-major:
 *   S = scale * Q K^T, LSE_i = ln sum_j exp(S_ij), P = exp(S - LSE 1^T),
 *   O_lo = P V_lo, O_hi = P V_hi.
 *
 * Common conventions
 *   - BH = B * heads slices; the slice index is the outermost index of every
 *     tensor.  packed / d_packed are [BH, 4, N, d]: sections 0..3 are
 *     Q, K, V_lo, V_hi (resp. dQ, dK, dV_lo, dV_hi).  o_lo, o_hi, do_lo, do_hi
 *     are [BH, N, d]; lse is [BH, N] fp32 (natural log, always fp32, whatever
 *     the storage type).  All contiguous, no padding.
 *   - Storage dtype: PSA_F32 or PSA_BF16 for every non-lse tensor; arithmetic
 *     accumulates in fp32.
 *   - head_dim (d) is one of 16, 32, 64.
 *   - All pointers are DEVICE pointers, 16-byte aligned.  The caller allocates
 *     and owns every buffer, including the backward workspace; the library
 *     allocates no device memory per call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it and do not synchronise the host.
 *   - Return: 0 on success, a negative psa_status on error.  Arguments are
 *     checked before anything is launched; on an argument error nothing is
 *     launched and no buffer is touched.  psa_attn_last_error() returns a
 *     message for the calling thread's last error.
 *   - B*heads == 0 or N == 0 is a valid empty call (returns 0, launches nothing).
 */
#ifndef PSA_ATTN_H
#define PSA_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PSA_F32 = 0, PSA_BF16 = 1 } psa_dtype;

typedef enum {
    PSA_OK = 0,
    PSA_ERR_ARG = -1,          /* null pointer, negative size, non-finite scale, bad dtype */
    PSA_ERR_ALIGN = -2,        /* a pointer is not 16-byte aligned */
    PSA_ERR_UNSUPPORTED = -3,  /* head_dim not in {16, 32, 64}, or a size over the limits */
    PSA_ERR_WORKSPACE = -4,    /* workspace missing or smaller than psa_attn_bwd_workspace_bytes */
    PSA_ERR_CUDA = -5,         /* a CUDA launch / driver call failed (message has the CUDA error) */
    PSA_ERR_TIMEOUT = -6       /* a device-side bounded wait gave up (see psa_attn_sync_status) */
} psa_status;

/* Backward kernel choice.  AUTO picks the tensor-core (tcgen05) path where it
 * exists for the (dtype, head_dim) and the CUDA-core (SIMT) path elsewhere.
 *   PSA_ALGO_TC        one key-outer pass; dQ partial sums are added to an
 *                      fp32 accumulator by bulk reduce operations, and the
 *                      dK/dV products of neighbouring query sub-tiles come
 *                      from two issuing threads, in orders that can differ
 *                      from run to run, and so can the rounding of dQ, dK and
 *                      dV.  (The units of its last, partial wave are split
 *                      along the queries; their dK/dV partials are summed in
 *                      a fixed order.)
 *   PSA_ALGO_TC_2PASS  a key-outer dK/dV pass and a query-outer dQ pass
 *                      (the split of "Struct PsaFa2Backward", description:
 *                      query gradients from a sweep over keys, key gradients
 *                      from a sweep over queries); no atomics,
 *                      bit-for-bit reproducible.  Backward only (the forward
 *                      entry points reject it). */
typedef enum { PSA_ALGO_AUTO = 0, PSA_ALGO_SIMT = 1, PSA_ALGO_TC = 2, PSA_ALGO_TC_2PASS = 3 } psa_algo;

/*
 * psa_attn_fwd -- PSA forward: O_lo = P V_lo, O_hi = P V_hi and LSE.
 * Produces the forward outputs that the backward consumes; "Struct
 * PsaFa2Backward", "Grid" paragraph (the backward shares the forward pass's
 * decomposition).
 *   packed  [BH,4,N,d] dtype, read
 *   o_lo, o_hi [BH,N,d] dtype, written
 *   lse     [BH,N] fp32, written (natural log of the softmax denominator of scale*q.k)
 *   scale   softmax scale applied to q.k (finite)
 */
int psa_attn_fwd(const void* packed, void* o_lo, void* o_hi, float* lse,
                 int B, int heads, int N, int head_dim, float scale,
                 int dtype, void* stream);

/* Like psa_attn_fwd, with an explicit kernel choice (psa_algo): the
 * tensor-core forward (bf16 storage) or the CUDA-core forward (any storage).
 * PSA_ALGO_TC returns PSA_ERR_UNSUPPORTED for fp32 storage. */
int psa_attn_fwd_algo(const void* packed, void* o_lo, void* o_hi, float* lse,
                      int B, int heads, int N, int head_dim, float scale,
                      int dtype, int algo, void* stream);

/*
 * Bytes of device workspace psa_attn_bwd needs for these sizes and the kernel
 * AUTO would pick: the fp32 row statistics D (the CUDA-core and two-pass
 * paths), or on the fused tensor-core path 8 bytes of row statistics per query
 * (LSE and D, padded to whole 64-query tiles), an fp32 dQ accumulator and room
 * for the fp32 dK/dV partials of split units.  The size does not depend on the
 * GPU.  Returns 0 for an empty or invalid problem.
 */
size_t psa_attn_bwd_workspace_bytes(int B, int heads, int N, int head_dim, int dtype);

/*
 * psa_attn_bwd -- PSA backward (the lo/hi pair of FA2 backward calls).
 * "Struct PsaFa2Backward": description (P is recomputed from Q, K and the row
 * statistics; query gradients need a sweep over keys, key gradients a sweep
 * over queries),
 * "Atomicity" (dQ, dK summed over lo and hi; each call owns its dV section).
 *   packed       [BH,4,N,d] dtype, read (Q, K, V_lo, V_hi)
 *   o_lo, o_hi   [BH,N,d] dtype, read (forward outputs)
 *   lse          [BH,N] fp32, read (from psa_attn_fwd)
 *   do_lo, do_hi [BH,N,d] dtype, read (upstream gradients)
 *   d_packed     [BH,4,N,d] dtype, OVERWRITTEN with dQ, dK, dV_lo, dV_hi
 *                (the page's kernel adds into a zeroed buffer; this call writes
 *                the gradients, so d_packed need not be zeroed first)
 *   workspace    device scratch of at least workspace_bytes; contents on entry
 *                are ignored, contents on exit are unspecified
 * Calls that share a workspace must not overlap on the GPU.
 */
int psa_attn_bwd(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                 const void* do_lo, const void* do_hi, void* d_packed,
                 void* workspace, size_t workspace_bytes,
                 int B, int heads, int N, int head_dim, float scale,
                 int dtype, void* stream);

/* Like psa_attn_bwd, with an explicit kernel choice (psa_algo).  PSA_ALGO_TC
 * and PSA_ALGO_TC_2PASS return PSA_ERR_UNSUPPORTED where no tensor-core kernel
 * exists for the (dtype, head_dim). */
int psa_attn_bwd_algo(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                      const void* do_lo, const void* do_hi, void* d_packed,
                      void* workspace, size_t workspace_bytes,
                      int B, int heads, int N, int head_dim, float scale,
                      int dtype, int algo, void* stream);

/*
 * psa_attn_view -- a strided view of a [B, heads, N, d] tensor: element
 * (b, h, n, j) (batch, head, position, feature) is at
 *   base + b*batch_stride + h*head_stride + n*pos_stride + j*feat_stride
 * with strides in elements.  Row-major rows ([N, d] per slice, as
 * psa_attn_bwd takes dO): feat_stride = 1, pos_stride >= d (a padded row when
 * larger).  Channel-major ([d, N] per slice, as a [B, c, H, W] feature map
 * holds it): pos_stride = 1, feat_stride >= N.
 */
typedef struct {
    const void* base;
    long long batch_stride, head_stride, pos_stride, feat_stride;
} psa_attn_view;

/*
 * psa_attn_bwd_ex -- psa_attn_bwd on strided layouts.  "Struct
 * PsaMergeAttnRuntimeOp" (forward_output_row_stride,
 * backward_grad_output_row_stride: a buffer's row stride may be rounded up
 * past the row length so that every row starts on a 16-byte boundary, as TMA
 * copies need) and the channel-major feature maps of the model around the op.
 *   packed          [BH, 4, N, qkv_row_stride] dtype, read: rows of d used
 *                   (section stride N*qkv_row_stride, slice stride 4*N*qkv_row_stride)
 *   qkv_row_stride  >= head_dim; also the row stride of d_packed
 *   o_lo, o_hi      [BH, N, o_row_stride] dtype, read; o_row_stride >= head_dim
 *   lse             [BH, N] fp32, read
 *   do_lo, do_hi    views (above) of the upstream gradients, read
 *   d_packed        [BH, 4, N, qkv_row_stride] dtype: the first head_dim
 *                   elements of every row are OVERWRITTEN, the padding is not
 *                   touched
 *   workspace       at least psa_attn_bwd_ex_workspace_bytes(...) bytes
 *   algo            PSA_ALGO_AUTO, PSA_ALGO_TC (fused tensor-core kernel, bf16)
 *                   or PSA_ALGO_SIMT; the two-pass mode takes contiguous
 *                   tensors only (psa_attn_bwd_algo)
 * Alignment: every pointer 16-byte aligned.  The tensor-core path also needs
 * every stride other than a unit one to be a multiple of 16 bytes (TMA); the
 * CUDA-core path needs qkv_row_stride = o_row_stride = head_dim (it gathers
 * strided dO views into the workspace first).  Violations return
 * PSA_ERR_ALIGN or PSA_ERR_UNSUPPORTED before anything is launched.
 * Other arguments, results and errors as psa_attn_bwd_algo.
 */
int psa_attn_bwd_ex(const void* packed, long long qkv_row_stride,
                    const void* o_lo, const void* o_hi, long long o_row_stride,
                    const float* lse, const psa_attn_view* do_lo, const psa_attn_view* do_hi,
                    void* d_packed, void* workspace, size_t workspace_bytes,
                    int B, int heads, int N, int head_dim, float scale,
                    int dtype, int algo, void* stream);

/* Workspace bytes psa_attn_bwd_ex needs (0 for an empty or invalid problem). */
size_t psa_attn_bwd_ex_workspace_bytes(const psa_attn_view* do_lo, const psa_attn_view* do_hi,
                                       int B, int heads, int N, int head_dim, int dtype, int algo);

/*
 * psa_merge_bwd -- the backward of the PSA attention merge alone
 * ("Struct PsaMergeAttnRuntimeOp", pack_backward_args: d_merged, d_lo, d_hi,
 * c, H, W, num_heads; backward_grid: one block per (batch*head, position)).
 * The merged tensor is [B, c, H, W], c = 2 * heads * head_dim, N = H * W;
 * its channels hold the lo outputs of every head in the low half and the hi
 * outputs in the high half, head-major in each half (a reading: the pages
 * name the arguments, not the order):
 *   d_lo[b*heads + h, n, j] = d_merged[b, h*head_dim + j, n]
 *   d_hi[b*heads + h, n, j] = d_merged[b, heads*head_dim + h*head_dim + j, n]
 *   d_merged  [B, c, H, W] dtype, read;  d_lo, d_hi  [B*heads, N, d] dtype, written
 */
int psa_merge_bwd(const void* d_merged, void* d_lo, void* d_hi, int B, int heads, int H, int W,
                  int head_dim, int dtype, void* stream);

/*
 * psa_merge_attn_bwd -- the merge's backward fused into the attention
 * backward: the kernels read dO_lo and dO_hi straight out of d_merged (the
 * views of psa_merge_bwd's mapping), so d_lo / d_hi are never written.
 * Arguments as psa_attn_bwd, with d_merged [B, 2*heads*head_dim, H, W] in
 * place of do_lo / do_hi and N = H * W; the workspace is
 * psa_merge_attn_bwd_workspace_bytes(...) bytes.  The tensor-core path needs
 * H * W a multiple of 8 (rows of d_merged 16-byte aligned).
 */
int psa_merge_attn_bwd(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                       const void* d_merged, void* d_packed, void* workspace, size_t workspace_bytes,
                       int B, int heads, int H, int W, int head_dim, float scale,
                       int dtype, int algo, void* stream);
size_t psa_merge_attn_bwd_workspace_bytes(int B, int heads, int H, int W, int head_dim, int dtype, int algo);

/*
 * psa_attn_bwd_noalloc -- the backward for callers that cannot allocate device
 * memory.  (The pages have no counterpart of this entry point; it is a
 * convenience of this library.)
 *
 * Some callers cannot call cudaMalloc or any allocating routine: a plugin that
 * is handed only its input and output buffers by a host runtime that owns all
 * device memory, or an application whose memory budget is fixed after start-up
 * and forbids libraries from allocating later.  psa_attn_bwd needs a workspace
 * from its caller; this variant needs none.  It runs the CUDA-core backward
 * (PSA_ALGO_SIMT) and keeps its only scratch -- the fp32 row statistics D, one
 * value per query row -- in a static array inside this library's device
 * memory, 2 MiB per GPU, which every GPU that loads the library holds until the
 * process exits.  The call itself allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   Arguments and results are those of psa_attn_bwd without the workspace.
 *   Limit: B*heads*N <= psa_attn_bwd_noalloc_max_rows() (524288); larger
 *   problems return PSA_ERR_UNSUPPORTED before anything is launched.
 *   Set-up: the first call on each device looks up the device address of the
 *   static array (with that device current) and caches it; make that first
 *   call before any stream capture.
 *   Sharing: every call on a device uses the same array.  D is rewritten in
 *   full by each call before it is read, so a call never sees an earlier
 *   call's values, but calls that overlap on the GPU (different streams, or
 *   different host threads, without ordering between them) race on it.
 */
int psa_attn_bwd_noalloc(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                         const void* do_lo, const void* do_hi, void* d_packed,
                         int B, int heads, int N, int head_dim, float scale,
                         int dtype, void* stream);

/* Largest B*heads*N psa_attn_bwd_noalloc accepts. */
long long psa_attn_bwd_noalloc_max_rows(void);

/* Workspace bytes for an explicit kernel choice (0 if unsupported). */
size_t psa_attn_bwd_workspace_bytes_algo(int B, int heads, int N, int head_dim, int dtype, int algo);

/*
 * psa_attn_bwd_host -- the backward on HOST buffers: copies the inputs to the
 * device, runs psa_attn_bwd_algo and copies d_packed back, all enqueued on
 * `stream`.  (The pages have no counterpart; it is this library's end-to-end
 * entry point.)  The (batch*head) slices are independent, so they are split
 * into `chunks` groups whose copy in, backward and copy back are pipelined:
 * the copies run on two streams this library creates once per device, and the
 * kernels on `stream`.
 *   packed ... d_packed  HOST pointers, layouts as in psa_attn_bwd (d_packed is
 *                written).  Page-locked memory (cudaHostAlloc or
 *                cudaHostRegister) makes the copies asynchronous; with pageable
 *                memory the call still works, but the copies block the host.
 *   dev_buf      DEVICE scratch, 256-byte aligned, at least
 *                psa_attn_bwd_host_buffer_bytes(...) bytes: the device copies of
 *                every input and of d_packed, then the backward workspace.
 *                Contents on entry are ignored; on exit unspecified.
 *   algo         as psa_attn_bwd_algo.
 *   chunks       0 = chosen by the library from the sizes and the GPU
 *                (psa_attn_bwd_host_chunks); else 1..64, capped at B*heads.
 *                With N % 4 != 0 the call runs as one chunk (every chunk's lse
 *                must start on a 16-byte boundary).
 *   stream       the call starts after earlier work on `stream`; work enqueued
 *                on `stream` after the call starts after d_packed has landed in
 *                host memory.  Asynchronous: synchronise `stream` before reading
 *                d_packed.
 * Returns as psa_attn_bwd (PSA_ERR_WORKSPACE: dev_buf missing or too small;
 * PSA_ERR_ALIGN: dev_buf not 256-byte aligned).  An empty problem returns 0
 * and touches nothing.  Calls that share dev_buf must not overlap on the GPU;
 * calls from several host threads are serialised while they enqueue.
 */
int psa_attn_bwd_host(const void* packed, const void* o_lo, const void* o_hi, const float* lse,
                      const void* do_lo, const void* do_hi, void* d_packed,
                      void* dev_buf, size_t dev_buf_bytes,
                      int B, int heads, int N, int head_dim, float scale,
                      int dtype, int algo, int chunks, void* stream);

/* Device buffer bytes psa_attn_bwd_host needs (0 for an empty or invalid
 * problem); they do not depend on the chunk count. */
size_t psa_attn_bwd_host_buffer_bytes(int B, int heads, int N, int head_dim, int dtype, int algo);

/* The chunk count psa_attn_bwd_host uses for chunks = 0 on the current device
 * (1 when no device is available). */
int psa_attn_bwd_host_chunks(int B, int heads, int N, int head_dim, int dtype, int algo);

/*
 * Synchronises `stream`, then reports whether any kernel of this library gave
 * up on a bounded device-side wait since the last check (PSA_ERR_TIMEOUT, and
 * the flag is cleared), or whether the stream has a CUDA error (PSA_ERR_CUDA).
 * Returns 0 otherwise.
 */
int psa_attn_sync_status(void* stream);

/*
 * Failure-detection self-test (the pages have no counterpart).  Launches, on
 * `stream`, one small kernel that waits -- through the same bounded device-side
 * wait the backward kernels use -- on a barrier nothing ever arrives on, with
 * a 20 ms limit.  The wait gives up, records the timeout in the device error
 * word and the kernel exits normally; no fault, no trap, and the CUDA context
 * stays usable.  A following psa_attn_sync_status(stream) returns
 * PSA_ERR_TIMEOUT and clears the word.  Returns 0 if the launch succeeded.
 */
int psa_attn_selftest_wait_timeout(void* stream);

/*
 * Kernel timing (instrumentation; it changes no result and skips no work).
 * While enabled, every launch this library makes records a pair of CUDA events
 * around itself on the call's stream, tagged with a slot: 0 = forward,
 * 1 = backward preprocess (D), 2 = backward main (dK/dV, and dQ on the
 * tensor-core path), 3 = backward dQ (CUDA-core path) / dQ finalize.
 * psa_attn_profile_read() synchronises those events, writes per-slot total
 * milliseconds and launch counts into the caller's arrays (length >= 4) and
 * clears the records.  Returns the number of slots, or a negative psa_status.
 * Without timing, the tensor-core backward's main and finalize kernels start
 * as programmatic dependents of the kernel before them (their blocks are
 * scheduled while it finishes); with timing on they start after it, one by
 * one, so that each pair of events measures one kernel.
 */
int psa_attn_profile_enable(int on);
int psa_attn_profile_read(float* total_ms, int* launches, int n_slots);
const char* psa_attn_profile_slot_name(int slot);

/* Message for the calling thread's most recent error ("" if none). */
const char* psa_attn_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int psa_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PSA_ATTN_H */
