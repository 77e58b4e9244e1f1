/*
 * evo_attn.h — C ABI of the GB300 (sm_103a) memory-efficient biased
 * Evoformer attention library (libevo_attn.so).
 *
 * What it computes.  For each batch b, row n and head h, with L queries and
 * L keys of head dimension D:
 *
 *     O = softmax(Q Kᵀ · D^-1/2 + bias1 + bias2) · V
 *
 * with the key mask bias1 broadcast over heads and queries and the pair
 * bias bias2 shared by all N rows.  Source: the web page "DeepSpeed4Science
 * 技术指南：AI4Science 大模型长序列训练与 Evoformer 内存高效注意力内核实战"
 * — §3.5 (the reference test scales Q·Kᵀ, adds the bias, applies softmax and
 * multiplies by V), §3.6 (the layouts below and the four Evoformer usages),
 * §3.7 (inputs fp16/bf16 on the device; bias1 shaped (B, N, 1, 1, L) and
 * bias2 (B, 1, H, L, L); the forward saves an fp32 log-sum-exp for the
 * backward; the backward forms delta first, then dQ, dK, dV and the bias
 * gradients, accumulating bias gradients in fp32 before casting back).
 *
 * Layouts (dense, row-major, no padding; the *_strided entry points also take
 * strided q, k, v, out, dout, dq, dk, dv, see evo_layout_t):
 *     q, k, v, out, dout, dq, dk, dv : [B, N, L, H, D]   dtype
 *     bias1 (key mask)               : [B, N, 1, 1, L]   dtype, nullable
 *     bias2 (pair bias)              : [B, 1, H, L, L]   dtype, nullable
 *     dbias2                         : [B, 1, H, L, L]   dtype
 *     lse                            : [B, N, H, L]      float32, natural log
 *
 * Readings where the page is silent: the scale is D^-1/2 with D the true head
 * dimension; lse is the natural log of the scaled, biased scores; a query row
 * whose every key score is -inf (an fp16 -1e9 mask over all keys) has an
 * empty softmax: its output row is 0, its lse is -inf and it contributes no
 * gradient.
 *
 * Supported: B, N, H >= 1; 1 <= L <= 32768; D in {8, 16, 24, ..., 64};
 * fp16 or bf16 with fp32 accumulation.  The page's own limits (forward
 * sequence length > 16, backward head dimension <= 64) are relaxed to L >= 1
 * and kept at D <= 64.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must point to memory of the current
 *    CUDA device; the caller owns all buffers.  The library allocates no
 *    device memory and has no settings: everything a call does is decided by
 *    its arguments (evo_options_t for what goes beyond the tensors), so calls
 *    from several threads or on several streams do not affect each other.
 *    What the library itself holds is fixed at load: a per-device cache of
 *    device properties, one fallback device status word per device (for
 *    calls given no status location, see evo_attn_device_status), the
 *    calling thread's last-error text, and the scratch array of
 *    evo_attn_bwd_noalloc.
 *  - Device buffers of the tensors above must be 16-byte aligned, except
 *    bias1 (2-byte) and lse (4-byte); the backward workspace 256-byte.
 *  - Outputs are overwritten, never accumulated into, and must not overlap
 *    any input (EVO_ERR_ALIASING).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are reported synchronously, before
 *    anything is launched, and leave every buffer untouched.  A failed kernel
 *    launch returns EVO_ERR_CUDA.
 *  - Every device-side wait is bounded.  A wait that runs out sets a device
 *    status word instead of hanging: the location the call's options give,
 *    else the backward workspace's own word (evo_attn_bwd_opts, read with
 *    evo_attn_bwd_status), else the fallback word (read with
 *    evo_attn_device_status).
 */
#ifndef EVO_ATTN_H
#define EVO_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EVO_ATTN_ABI_VERSION 4

/* Every entry point below is exported from libevo_attn.so; nothing else is. */
#if defined(__GNUC__)
#define EVO_API __attribute__((visibility("default")))
#else
#define EVO_API
#endif

typedef enum {
  EVO_OK = 0,
  EVO_ERR_NULL_POINTER = 1,        /* a required pointer is NULL                    */
  EVO_ERR_BAD_SHAPE = 2,           /* B,N,H < 1, L outside [1, 32768], D not 8..64 step 8,
                                      or an element count that overflows           */
  EVO_ERR_BAD_DTYPE = 3,           /* dtype is neither EVO_F16 nor EVO_BF16         */
  EVO_ERR_MISALIGNED = 4,          /* a pointer breaks the alignment rule above     */
  EVO_ERR_WORKSPACE_TOO_SMALL = 5, /* workspace_bytes < evo_attn_bwd_workspace_bytes */
  EVO_ERR_ARCH = 6,                /* current device is not compute capability 10.3 */
  EVO_ERR_CUDA = 7,                /* a CUDA runtime/driver call or launch failed   */
  EVO_ERR_DEVICE_TIMEOUT = 8,      /* a bounded device-side wait ran out            */
  EVO_ERR_ALIASING = 9,            /* an output overlaps an input                   */
  EVO_ERR_BAD_ARGUMENT = 10,       /* any other invalid argument (e.g. dbias2 given
                                      without bias2, or missing with bias2)         */
  EVO_ERR_SCRATCH_LIMIT = 11,      /* evo_attn_bwd_noalloc: the problem needs more
                                      scratch than EVO_NOALLOC_SCRATCH_BYTES         */
  EVO_ERR_BAD_LAYOUT = 12          /* a stride of evo_layout_t breaks its rules      */
} evo_status_t;

typedef enum { EVO_F16 = 0, EVO_BF16 = 1 } evo_dtype_t;

typedef struct {
  int64_t B, N, L, H, D;
} evo_shape_t;

/*
 * Strided layout of one [B,N,L,H,D] tensor (evo_attn_fwd_strided,
 * evo_attn_bwd_strided): the element strides of its B, N and L dimensions.
 * Its H and D dimensions stay packed (strides D and 1), so each token row of
 * H*D elements is contiguous.  Packed: b = N*L*H*D, n = L*H*D, l = H*D.
 *
 * This is how the Evoformer's transposed usages reach the kernels without a
 * copy (page §3.6: column-wise MSA attention runs over the other axis of the
 * MSA; triangle attention around the ending node over the other axis of the
 * pair representation): pass the [B, N_res, N_seq, H, D] view of a
 * [B, N_seq, N_res, H, D] buffer as b = N_seq*N_res*H*D, n = H*D,
 * l = N_res*H*D.
 *
 * Rules (else EVO_ERR_BAD_LAYOUT): the strides of dimensions of extent > 1 are
 * positive multiples of 8 below 2^36; no two token rows overlap (taken in
 * order of stride, each stride is at least the extent in elements of the
 * dimensions inside it, the innermost at least H*D); the whole span is below
 * 2^44 elements.  Strides of dimensions of extent 1 are ignored.
 *
 * The aliasing rule (EVO_ERR_ALIASING) compares each tensor's span, from its
 * first element to its last: tensors interleaved in one buffer (for instance
 * q and out as two slots of one [.., 4, H, D] buffer) count as overlapping
 * even where their elements are disjoint.
 */
typedef struct {
  int64_t b, n, l;
} evo_strides_t;

/* Layouts of the [B,N,L,H,D] tensors of one call.  The forward reads q, k, v
 * and out; the backward all eight.  bias1, bias2, lse and the bias gradients
 * keep their packed layouts. */
typedef struct {
  evo_strides_t q, k, v, out, dout, dq, dk, dv;
} evo_layout_t;

/*
 * Per-call options of evo_attn_fwd_opts and evo_attn_bwd_opts.  Zero the
 * struct, set `size` to sizeof(evo_options_t), then set what the call needs;
 * a NULL options pointer means the defaults (all zero).  Nothing is kept after
 * the call returns.  A struct whose size is too small, with unknown flag bits,
 * or with num_events > 0 and events == NULL is EVO_ERR_BAD_ARGUMENT.
 *
 *   flags          EVO_OPT_SKIP_MASKED_TILES: masked key-tile skipping.  A key
 *                  j of row (b, n) counts as masked when bias1[b,n,j] <=
 *                  skip_threshold (a NaN counts as kept); every 128-key tile of
 *                  a row whose keys are all masked is skipped, as long as the
 *                  row keeps some key.  The forward skips on every shape with
 *                  L <= 8192; the backward on the shapes whose dQ tiles do not
 *                  fit in tensor memory (its per-key-tile schedule), writing the
 *                  skipped tiles' dK and dV as zeros.  The results are those of
 *                  the unskipped computation whenever each masked key's scaled,
 *                  biased score lies more than 88 below its row's largest one:
 *                  its fp32 exponential is then exactly 0 either way (page
 *                  §3.6's key mask, a very large negative bias, meets this by
 *                  far).  Skipped tiles still count in any nominal FLOP figure
 *                  derived from the shape.
 *                  EVO_OPT_NO_DBIAS2 (backward only): do not compute the
 *                  pair-bias gradient; dbias2 must then be NULL even with a
 *                  bias2, and the workspace may be sized with EVO_WS_NO_DBIAS2.
 *   skip_threshold see EVO_OPT_SKIP_MASKED_TILES (e.g. -1e4).
 *   wait_limit_ns  bound on every device-side wait of the call (0 = 2e9; values
 *                  below 1000 are raised to 1000).
 *   status         device int the call's kernels set to EVO_ERR_DEVICE_TIMEOUT
 *                  if a wait runs out (the caller clears it); NULL: the forward
 *                  uses the fallback word, the backward its workspace's word.
 *   events, num_events
 *                  profiling: caller-owned CUDA events (cudaEvent_t, timing
 *                  enabled), at most 8 used, recorded on the call's stream
 *                  around each kernel it launches:
 *                    forward:  events[0] before its kernel, events[1] after it;
 *                    backward: events[2] before its first kernel, then one
 *                    event after each kernel in launch order — events[3] after
 *                    delta, events[4] after the main backward kernel (with
 *                    masked-tile skipping on the per-key-tile schedule its
 *                    skip-bit kernel runs between events[3] and events[4]),
 *                    events[5] recorded right after events[4], and with the
 *                    pair-bias gradient events[6] after its per-group partials
 *                    and events[7] after their fixed-order sum.  With dbias1,
 *                    its partial and sum kernels run between events[5] and
 *                    events[6].  A call split batch by batch (strided layouts)
 *                    records them for its last batch.  Indices >= num_events
 *                    are skipped.  Recording works inside stream capture (the
 *                    records become graph nodes).
 */
#define EVO_OPT_SKIP_MASKED_TILES 1u
#define EVO_OPT_NO_DBIAS2 2u

typedef struct {
  uint32_t size;
  uint32_t flags;
  float skip_threshold;
  uint32_t reserved;
  uint64_t wait_limit_ns;
  int* status;
  void* const* events;
  int32_t num_events;
} evo_options_t;

/* For the calling thread's last call that returned EVO_ERR_CUDA: which step
 * failed and the CUDA error name and code (static thread-local text, valid
 * until this thread's next failing call; "" if none failed). */
EVO_API const char* evo_attn_last_error_detail(void);

/* ABI version of the loaded library (EVO_ATTN_ABI_VERSION at build time). */
EVO_API int evo_attn_abi_version(void);

/* Static, NUL-terminated description of a status code. */
EVO_API const char* evo_status_string(evo_status_t status);

/*
 * Forward (page §3.5-§3.7).  Device pointers:
 *   q, k, v  [B,N,L,H,D] inputs; bias1 [B,N,1,1,L] or NULL; bias2 [B,1,H,L,L] or NULL;
 *   out      [B,N,L,H,D] output O, rounded to nearest in dtype;
 *   lse      [B,N,H,L]   fp32 output, natural-log log-sum-exp of each query row.
 * The L×L score matrix never exists in device memory.
 */
EVO_API evo_status_t evo_attn_fwd(const void* q, const void* k, const void* v,
                          const void* bias1, const void* bias2,
                          void* out, float* lse,
                          evo_shape_t shape, evo_dtype_t dtype, void* stream);

/*
 * evo_attn_fwd on strided tensors: q, k, v and out laid out as `layout` says
 * (NULL = packed, exactly evo_attn_fwd).  The alignment rule applies to the
 * first element.  Tensors whose batch stride is not N times their row stride
 * (with B > 1 and N > 1) are processed one batch at a time, one launch each.
 */
EVO_API evo_status_t evo_attn_fwd_strided(const void* q, const void* k, const void* v,
                                          const void* bias1, const void* bias2,
                                          void* out, float* lse,
                                          evo_shape_t shape, evo_dtype_t dtype,
                                          const evo_layout_t* layout, void* stream);

/*
 * evo_attn_fwd_strided with per-call options (evo_options_t; NULL = defaults,
 * exactly evo_attn_fwd_strided).  EVO_OPT_NO_DBIAS2 is EVO_ERR_BAD_ARGUMENT here.
 */
EVO_API evo_status_t evo_attn_fwd_opts(const void* q, const void* k, const void* v,
                                       const void* bias1, const void* bias2,
                                       void* out, float* lse,
                                       evo_shape_t shape, evo_dtype_t dtype,
                                       const evo_layout_t* layout, const evo_options_t* opts,
                                       void* stream);

/* Flags of evo_attn_bwd_workspace_bytes (bit 0 keeps the meaning of the
 * former has_bias2 argument, so passing 0 / 1 still works). */
#define EVO_WS_BIAS2 1     /* the call has a pair bias (and computes dbias2)     */
#define EVO_WS_DBIAS1 2    /* the call computes dbias1 (evo_attn_bwd_ex)          */
#define EVO_WS_NO_DBIAS2 4 /* with a pair bias, no dbias2 (EVO_OPT_NO_DBIAS2)     */

/*
 * Bytes of device workspace the backward needs for this problem (0 on a bad
 * shape, dtype or flag).  It holds the call's status word (256 bytes); the
 * fp32 row terms delta [B,N,H,L]; for the shapes whose dQ tiles do not fit in
 * tensor memory, L x DP fp32 dQ rows (DP = D rounded up to 16, 32 or 64) for
 * each of at most 256 CTAs, and the skip bits of masked key-tile skipping;
 * with EVO_WS_BIAS2, where a key-major kernel runs, a transposed copy of the
 * pair bias, and unless EVO_WS_NO_DBIAS2 the fp32 per-group partial sums of the
 * pair-bias gradient; with EVO_WS_DBIAS1, fp32 per-(b, n, h) partial sums of
 * the key-mask gradient.  Depends only on its arguments; enough for every
 * layout of evo_attn_bwd_strided.
 */
EVO_API size_t evo_attn_bwd_workspace_bytes(evo_shape_t shape, evo_dtype_t dtype, int flags);

/*
 * Backward (page §3.7: delta first, then dQ/dK/dV and the bias gradient).
 * Device pointers:
 *   q, k, v, bias1, bias2 : the forward's inputs (bias1/bias2 nullable as there);
 *   out, lse              : the forward's outputs;
 *   dout                  : [B,N,L,H,D] gradient of the loss with respect to out;
 *   dq, dk, dv            : [B,N,L,H,D] outputs;
 *   dbias2                : [B,1,H,L,L] output, required iff bias2 != NULL.
 *                           Summed over N in fp32 in a fixed order (two stages:
 *                           per-group partials, then a fixed-order sum of the
 *                           groups).  Every gradient is summed in a fixed order,
 *                           so repeated calls give identical bytes;
 *   workspace             : >= evo_attn_bwd_workspace_bytes(...) bytes, caller-owned,
 *                           contents need not be initialised; clobbered.
 * The gradient of bias1 is produced by evo_attn_bwd_ex.
 */
EVO_API evo_status_t evo_attn_bwd(const void* q, const void* k, const void* v,
                          const void* bias1, const void* bias2,
                          const void* out, const float* lse, const void* dout,
                          void* dq, void* dk, void* dv, void* dbias2,
                          void* workspace, size_t workspace_bytes,
                          evo_shape_t shape, evo_dtype_t dtype, void* stream);

/*
 * evo_attn_bwd plus the key-mask gradient (page §3.7: the backward returns the
 * gradients of both biases):
 *   dbias1 : [B,N,1,1,L] output in dtype, or NULL (then exactly evo_attn_bwd).
 *            dbias1[b,n,j] = Σ_h Σ_i dS[b,n,h,i,j], summed in fp32 in a fixed
 *            order (per-(b,n,h) partials, then a fixed-order sum over h), so
 *            repeated calls give identical bytes.  Requires bias1 != NULL.
 *   workspace : >= evo_attn_bwd_workspace_bytes(shape, dtype,
 *               (bias2 ? EVO_WS_BIAS2 : 0) | (dbias1 ? EVO_WS_DBIAS1 : 0)).
 * Errors as evo_attn_bwd; EVO_ERR_BAD_ARGUMENT if dbias1 is given without bias1.
 */
EVO_API evo_status_t evo_attn_bwd_ex(const void* q, const void* k, const void* v,
                             const void* bias1, const void* bias2,
                             const void* out, const float* lse, const void* dout,
                             void* dq, void* dk, void* dv, void* dbias1, void* dbias2,
                             void* workspace, size_t workspace_bytes,
                             evo_shape_t shape, evo_dtype_t dtype, void* stream);

/*
 * evo_attn_bwd_ex on strided tensors: q, k, v, out, dout, dq, dk and dv laid
 * out as `layout` says (NULL = packed, exactly evo_attn_bwd_ex).  Outputs are
 * written only at their own elements; bytes between rows are left alone.
 * With B > 1 and a tensor whose batch stride is not N times its row stride the
 * call runs one batch at a time (the workspace is reused by each; the
 * profiling events then bracket the last batch).
 */
EVO_API evo_status_t evo_attn_bwd_strided(const void* q, const void* k, const void* v,
                                          const void* bias1, const void* bias2,
                                          const void* out, const float* lse, const void* dout,
                                          void* dq, void* dk, void* dv, void* dbias1, void* dbias2,
                                          void* workspace, size_t workspace_bytes,
                                          evo_shape_t shape, evo_dtype_t dtype,
                                          const evo_layout_t* layout, void* stream);

/*
 * evo_attn_bwd_strided with per-call options (evo_options_t; NULL = defaults).
 * Unlike the entry points above, which record a timeout in the fallback word,
 * this one records it in its workspace's own status word (cleared by the
 * call's first kernel) unless opts->status is given; read it with
 * evo_attn_bwd_status.  With EVO_OPT_NO_DBIAS2, dbias2 must be NULL and no
 * pair-bias gradient is computed.
 */
EVO_API evo_status_t evo_attn_bwd_opts(const void* q, const void* k, const void* v,
                                       const void* bias1, const void* bias2,
                                       const void* out, const float* lse, const void* dout,
                                       void* dq, void* dk, void* dv, void* dbias1, void* dbias2,
                                       void* workspace, size_t workspace_bytes,
                                       evo_shape_t shape, evo_dtype_t dtype,
                                       const evo_layout_t* layout, const evo_options_t* opts,
                                       void* stream);

/*
 * Synchronises `stream`, then reads the status word of a workspace last used
 * by evo_attn_bwd_opts (device pointer, 256-byte aligned): EVO_OK, or
 * EVO_ERR_DEVICE_TIMEOUT if one of that call's kernels gave up on a bounded
 * wait (its outputs are then undefined).  EVO_ERR_CUDA if the synchronisation
 * or the read failed.
 */
EVO_API evo_status_t evo_attn_bwd_status(const void* workspace, void* stream);

/*
 * Synchronises `stream`, then reads and clears the fallback device status
 * word on the current device: EVO_OK, or EVO_ERR_DEVICE_TIMEOUT if some
 * kernel of a call given no status location of its own gave up on a bounded
 * wait since the last read (its outputs are then undefined).  EVO_ERR_CUDA
 * if the synchronisation itself failed.
 */
EVO_API evo_status_t evo_attn_device_status(void* stream);

/*
 * Self-test of the bounded-wait path: launches one block that waits on a
 * shared-memory barrier nothing ever signals, with the wait limit given here
 * (clamped to [1000 ns, 1e9 ns]).  The block gives up, records
 * EVO_ERR_DEVICE_TIMEOUT in *status (a device int, 4-byte aligned; NULL = the
 * fallback word, read with evo_attn_device_status) and exits.  Faults nothing
 * and leaves the context usable.
 */
EVO_API evo_status_t evo_attn_selftest_wait_timeout(uint64_t limit_ns, int* status, void* stream);

/*
 * Bytes of device arena evo_attn_step_host needs for this problem (0 on a bad
 * shape or dtype): room for the inputs, outputs, lse and backward workspace
 * (and, with a pair bias and B = 1, the fp32 partial planes of its gradient).
 */
EVO_API size_t evo_attn_step_host_arena_bytes(evo_shape_t shape, evo_dtype_t dtype, int has_bias1,
                                              int has_bias2);

/*
 * One forward + backward step from and to HOST memory.  Copies q, k, v,
 * bias1, bias2 (nullable as in evo_attn_fwd) and dout from host buffers into
 * the caller's device arena (one cudaMemcpyAsync per tensor), runs
 * evo_attn_fwd and evo_attn_bwd there, and copies out, dq, dk, dv, dbias2
 * (required iff bias2 != NULL) and, when lse != NULL, lse back to host
 * buffers.  The work runs in chunks of rows (b, n), so that the copies of one
 * chunk overlap another's compute; with a pair bias and B = 1 each chunk's
 * backward writes the partial sums of its own n-groups of the pair-bias
 * gradient and one fixed-order sum follows, so every output is the same bytes
 * as evo_attn_fwd + evo_attn_bwd on device buffers give.  Host buffers should
 * be page-locked for the copies to be asynchronous; all work is queued on
 * `stream`, so synchronise it before reading the outputs.  arena: device memory of at least
 * evo_attn_step_host_arena_bytes(...) bytes, 256-byte aligned, caller-owned.
 * Host pointers have no alignment rule.  Validation as in evo_attn_fwd/bwd.
 */
EVO_API evo_status_t evo_attn_step_host(const void* q, const void* k, const void* v, const void* bias1,
                                        const void* bias2, const void* dout, void* out, float* lse, void* dq,
                                        void* dk, void* dv, void* dbias2, void* arena, size_t arena_bytes,
                                        evo_shape_t shape, evo_dtype_t dtype, void* stream);

/*
 * Backward for callers that cannot allocate device memory.
 *
 * The method's pages have no counterpart to this entry point; it exists for
 * the library's users.  evo_attn_bwd needs a device workspace from its
 * caller, and some callers cannot provide one: code that runs where
 * cudaMalloc is unavailable or forbidden (inside a memory-pool-managed
 * framework that owns every allocation, a real-time or embedded loop that
 * must not allocate after start-up, a plugin without access to the host
 * application's allocator).  This variant runs the same backward but takes
 * its scratch from a fixed array inside the library: a file-scope
 * __device__ array of EVO_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU
 * which loads this part of the library holds until the process exits.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments and outputs are those of evo_attn_bwd without the workspace.
 * Problems whose backward workspace (evo_attn_bwd_workspace_bytes) exceeds
 * EVO_NOALLOC_SCRATCH_BYTES are rejected with EVO_ERR_SCRATCH_LIMIT before
 * anything is launched.
 *
 * When the array is reserved: with lazy module loading (CUDA_MODULE_LOADING=
 * LAZY, the default) at the first call on each device, which therefore can
 * fail with EVO_ERR_CUDA if the device has no 16 MiB left (the reason is in
 * evo_attn_last_error_detail; a later call tries again); with eager loading,
 * on every GPU where the process creates a context.  So a caller that must
 * not allocate after start-up makes one call per device during start-up.
 * That first call also looks up the array's device address on that device
 * (cudaGetSymbolAddress, with the device current); make it before any stream
 * capture on the device.  The address is cached per device index; after a
 * cudaDeviceReset it is stale, and this entry point must not be used on that
 * device again in the process.  Every call on a device shares the one array,
 * which keeps the previous call's contents (the kernels write every byte
 * before reading it): calls whose work overlaps on the GPU — on different
 * streams, or from different host threads — race on the scratch and give
 * wrong results.  Serialise them.  Timeouts of its kernels are recorded in
 * the fallback status word (evo_attn_device_status).
 */
#define EVO_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

EVO_API evo_status_t evo_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                          const void* bias1, const void* bias2,
                                          const void* out, const float* lse, const void* dout,
                                          void* dq, void* dk, void* dv, void* dbias2,
                                          evo_shape_t shape, evo_dtype_t dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EVO_ATTN_H */
