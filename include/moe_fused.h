/* moe_fused.h -- C ABI of the GB300 fused MoE expert block.
 *
 * The block (FusedDeepMoE analysis, §1.2 operator signature and §9.1 the
 * DeepSeek-style MoE it implements) computes, on one GPU, for a batch of bs
 * tokens already routed by an external router:
 *
 *   dispatch   counting sort of the active (token, k) pairs by expert
 *              (§4.1 local token counting and the prefix-sum expand index);
 *   quant      per-token dynamic INT8 quantisation of x (§4.1, §7.3);
 *   GEMM1      grouped INT8 x INT8 -> INT32, dequantised by per-output-channel
 *              x per-token FP32 scales, SwiGLU (§3.3, §6.1);
 *   requant    per-row dynamic INT8 quantisation of the SwiGLU output (§7.2);
 *   GEMM2      grouped INT8 GEMM, dequantised to bf16 (§3.4, §6.2);
 *   combine    output[t] = sum_k expert_scales[t,k] * row(t,k), in fp32,
 *              k ascending, rounded once to bf16 (§4.2 LocalWindowCopy);
 *   shared     an optional shared expert on every active token, written to
 *              share_output.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; all are
 *     owned by the caller.  The library allocates no device memory and never
 *     copies weights; it owns only the host-side handle.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously; only argument checks are synchronous.
 *   - Return 0 on success or a negative MOE_ERR_* code.  A call that returns an
 *     error before launching leaves every output untouched.
 *   - Tensors are dense, row-major, with the innermost dimension contiguous.
 *     Every pointer must be 16-byte aligned unless its entry point states
 *     another rule.
 */
#ifndef MOE_FUSED_H
#define MOE_FUSED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)          /* NULL where a tensor is required, bad count, bad handle  */
#define MOE_ERR_UNSUPPORTED_SHAPE (-2)    /* shape outside the limits below                           */
#define MOE_ERR_WORKSPACE_TOO_SMALL (-3)  /* workspace_bytes below what create() reported             */
#define MOE_ERR_CUDA (-4)                 /* a CUDA runtime call failed (launch, attribute, memcpy)  */
#define MOE_ERR_DEVICE_TIMEOUT (-5)       /* a bounded in-kernel wait gave up (see get_status)        */
#define MOE_ERR_UNIMPLEMENTED (-6)
#define MOE_ERR_ALIGNMENT (-7)            /* a pointer is not aligned as its entry point requires       */

/* Static shape of one block.  Limits: 1 <= hidden, inter <= 16384 and both
 * multiples of 64; 1 <= num_experts <= 1024; 1 <= topk <= min(num_experts, 16);
 * 0 <= bs_max <= 65536.  GEMM1 has N = 2*inter outputs (gate rows 0..inter-1,
 * up rows inter..2*inter-1); GEMM2 maps inter -> hidden.  `flags` is a
 * combination of the MOE_FLAG_* bits below (MOE_FLAG_SCALE_BF16 and
 * MOE_FLAG_SCALE_FP16 exclude each other); other bits are reserved
 * (MOE_ERR_INVALID_ARG).  The pages' supported ranges (§9.4) are not
 * enforced. */

/* Every expert takes the tensor-core path with separate requant and combine
 * kernels: the unfused chain (FusedDeepMoE analysis §9.3, the "SmallOps"
 * sequence of dispatch+quant, GEMM1, requant, GEMM2, combine) kept as an A/B
 * baseline for the fused weight-streaming path that experts with at most 8
 * rows take by default.  Results are the same either way (the same
 * operations in the same order). */
#define MOE_FLAG_UNFUSED 1

/* The routing weight of pair (t, k) is folded into its row's GEMM2 dequant
 * scale (DeepSeek-V4 decode case study §2.3: the per-row dequant scale and
 * the routing weight fused into one row scale computed once per row):
 *   y2[r][j] = bf16((float(acc2[r][j]) * w2_scale[e][j]) * (s2[r] * expert_scales[t][k]))
 *   output[t] = bf16(sum over k ascending of float(y2[row(t,k)])), from 0.0f.
 * The shared expert is unchanged.  This rounds differently from the default
 * (routing weight applied in the combine after each row's bf16 rounding). */
#define MOE_FLAG_FOLD_ROUTING 2

/* Signature variants of the operator's input table (§1.2: x bf16 or fp16;
 * routed weight scales fp32, bf16 or fp16; smooth scales optional, shape not
 * given).
 * MOE_FLAG_FP16_ACT: x is fp16, and y2, output and share_output are fp16
 *   (round to nearest even, IEEE overflow to infinity) instead of bf16.
 * MOE_FLAG_SCALE_BF16 / MOE_FLAG_SCALE_FP16: gmm1_weight_scale and
 *   gmm2_weight_scale hold bf16 / fp16 values, widened exactly to fp32 before
 *   the same arithmetic.  The shared expert's scales stay fp32.
 * MOE_FLAG_EXPERT_SMOOTH: expert_smooth_scales is [num_experts, hidden]; the
 *   routed row of pair (t, k) with expert e is quantised from
 *   x[t] * expert_smooth_scales[e] (a per-row quant: the workspace holds one
 *   int8 row per routed pair).  The shared expert keeps its [hidden] vector. */
#define MOE_FLAG_FP16_ACT 4
#define MOE_FLAG_SCALE_BF16 8
#define MOE_FLAG_SCALE_FP16 16
#define MOE_FLAG_EXPERT_SMOOTH 32
typedef struct {
  int32_t bs_max;
  int32_t hidden;
  int32_t num_experts;
  int32_t topk;
  int32_t inter;
  int32_t has_shared;
  int32_t flags;
} moe_fused_config_t;

/* Per-call tensors, following the operator signature (§1.2):
 *   x                  [bs, hidden] bf16 (fp16 with MOE_FLAG_FP16_ACT)
 *   expert_ids         [bs, topk] int32; a pair whose id is outside
 *                      [0, num_experts) is skipped (not counted, adds nothing)
 *   expert_scales      [bs, topk] fp32 routing weights
 *   gmm1_weight        [num_experts, 2*inter, hidden] int8, K (hidden) contiguous
 *   gmm1_weight_scale  [num_experts, 2*inter] fp32 per output channel (bf16 / fp16
 *                      with MOE_FLAG_SCALE_BF16 / MOE_FLAG_SCALE_FP16)
 *   gmm2_weight        [num_experts, hidden, inter] int8, K (inter) contiguous
 *   gmm2_weight_scale  [num_experts, hidden] fp32 (or as gmm1_weight_scale)
 *   share_gmm1_weight / _scale   [2*inter, hidden] / [2*inter]  (has_shared)
 *   share_gmm2_weight / _scale   [hidden, inter] / [hidden]     (has_shared)
 *   expert_smooth_scales  [hidden] fp32 or NULL: multiplies x per channel
 *                      before the routed experts' quant ([num_experts, hidden]
 *                      with MOE_FLAG_EXPERT_SMOOTH: expert e's own row)
 *   share_smooth_scales   [hidden] fp32 or NULL: same for the shared expert
 *   x_active_mask      [bs] bool (one byte, 0 = inactive) or NULL (all active);
 *                      inactive tokens are not dispatched and get zero rows in
 *                      output and share_output
 * Outputs:
 *   output             [bs, hidden] bf16 (x's dtype)
 *   share_output       [bs, hidden] bf16 (x's dtype), required iff has_shared, else NULL
 *   expert_token_nums  [num_experts] int32: rows each expert received (counts,
 *                      not a prefix sum)
 * bs: 0 <= bs <= bs_max.  bs == 0 zeroes expert_token_nums and leaves the other
 * outputs untouched. */
typedef struct {
  const void* x;
  const int32_t* expert_ids;
  const float* expert_scales;
  const int8_t* gmm1_weight;
  const void* gmm1_weight_scale;   /* fp32, or bf16 / fp16 bits (flags) */
  const int8_t* gmm2_weight;
  const void* gmm2_weight_scale;
  const int8_t* share_gmm1_weight;
  const float* share_gmm1_weight_scale;
  const int8_t* share_gmm2_weight;
  const float* share_gmm2_weight_scale;
  const float* expert_smooth_scales;
  const float* share_smooth_scales;
  const uint8_t* x_active_mask;
  void* output;
  void* share_output;
  int32_t* expert_token_nums;
  int32_t bs;
} moe_fused_args_t;

/* Device-side status of the last forward that used a workspace. */
typedef struct {
  int32_t skipped_pairs;   /* active pairs whose expert id was outside [0, E) */
  int32_t error_flags;     /* bit 0: an in-kernel wait gave up                 */
  int32_t error_site;      /* which wait gave up (kernel id * 16 + site)       */
  int32_t dispatched_rows; /* R: routed rows dispatched                        */
  int32_t shared_rows;     /* S: rows run through the shared expert            */
  int32_t active_slots;    /* GEMM slots: experts with at least one row, +1    */
                           /* for the shared expert (in a batch of at most 8   */
                           /* tokens an expert with more rows, from repeated   */
                           /* ids, counts once per slot of at most 8 rows)     */
  int32_t reserved[2];
} moe_fused_status_t;

/* A handle holds host-side state between calls (tensor maps, timing records,
 * its own stream): one host thread at a time may call into a given handle.  Distinct handles share no
 * host state.  On the GPU, forwards must not overlap one another: the
 * one-launch forward (a grid barrier) and the small experts' streamed launch
 * (GEMM2 work that waits on other CTAs' GEMM1 work) count on every CTA of
 * the launch getting an SM, one CTA per SM.  Forwards issued in sequence
 * (one stream, or streams ordered by events) meet that.  Two forwards in
 * flight at once on one GPU (one handle or several, on unordered streams)
 * can each hold SMs the other's waiting CTAs need; their bounded waits then
 * give up after 2 s and get_status reports MOE_ERR_DEVICE_TIMEOUT. */
typedef struct moe_fused_handle moe_fused_handle_t;

/* Validate `cfg`, allocate the host handle and report the workspace size in
 * bytes (device memory the caller allocates, 256-byte aligned, and passes to
 * every forward).  The device current at this call is the device the handle
 * launches on.  The handle also creates one non-blocking stream and three
 * events of its own (the second engine's stream, see moe_fused_forward);
 * moe_fused_destroy releases them.  Errors: INVALID_ARG, UNSUPPORTED_SHAPE,
 * CUDA. */
int moe_fused_create(const moe_fused_config_t* cfg, moe_fused_handle_t** out_handle,
                     size_t* workspace_bytes);

/* Workspace bytes for `cfg` without creating a handle. */
int moe_fused_workspace_size(const moe_fused_config_t* cfg, size_t* workspace_bytes);

/* Enqueue one forward of the block on `stream`.  `workspace` must hold at least
 * the reported bytes; its contents need no initialisation and are overwritten.
 * Two forwards that share a workspace must be ordered on the GPU.
 * A batch of at most 8 tokens (without MOE_FLAG_EXPERT_SMOOTH smooth scales,
 * and unless MOE_FLAG_UNFUSED is set) runs as one launch whose CTAs meet at
 * one grid barrier; its words (a workspace region of their own) need no
 * initial value: each CTA's arrival tag carries the barrier's generation
 * mixed with a random constant of the handle.  A larger batch on the fused
 * path runs the dp4a launch on `stream` beside the tensor-core GEMMs on the
 * handle's own stream, forked from `stream` after the dispatch and joined
 * back before the combine (so a CUDA graph captured from `stream` holds
 * both); launches whose CTAs take their work in arrival order count arrivals
 * in status words 40..42, which the forward's dispatch zeroes first.  So no
 * state carries from one forward to the next: between forwards the caller
 * may overwrite any part of the workspace (moe_fused_get_status reads the
 * status words the last forward left).  Errors: INVALID_ARG,
 * UNSUPPORTED_SHAPE (bs > bs_max), WORKSPACE_TOO_SMALL, ALIGNMENT, CUDA
 * (launch failure). */
int moe_fused_forward(moe_fused_handle_t* handle, const moe_fused_args_t* args, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Synchronise `stream` and read the status words of the last forward that used
 * `workspace` into *out (host memory).  Returns DEVICE_TIMEOUT if a wait gave
 * up, otherwise 0 (or CUDA). */
int moe_fused_get_status(moe_fused_handle_t* handle, const void* workspace, void* stream,
                         moe_fused_status_t* out);

/* Free the handle, its stream and events (no device memory is owned).  NULL
 * is accepted. */
int moe_fused_destroy(moe_fused_handle_t* handle);

/* Static string for an error code. */
const char* moe_fused_strerror(int code);

/* ---- dispatch for callers that cannot allocate device memory ------------
 * The pages have no counterpart of this entry point; it exists for callers
 * that may not allocate device memory at all -- a plugin or custom op inside
 * a host framework that owns every device allocation, or a process running
 * on a fixed, pre-reserved device-memory budget -- and therefore cannot
 * provide the workspace that moe_fused_forward needs.
 *
 * It runs only the dispatch step (the counting sort of the active (t, k)
 * pairs by expert, stable by flat index t*topk+k) and writes
 *   expert_token_nums  [num_experts] int32 (device): rows per expert, exactly
 *                      as moe_fused_forward writes it;
 *   expand_row         [bs, topk] int32 (device) or NULL: the row of each pair
 *                      in expert-sorted order, -1 for pairs not dispatched
 *                      (masked token or id outside [0, num_experts)).
 * Inputs: expert_ids [bs, topk] int32 and x_active_mask [bs] (or NULL), device.
 *
 * Its scratch lives in one library-owned static device array of 2 MiB, which
 * every GPU that loads the library keeps until the process exits.  Limits:
 * bs * topk <= 65536, num_experts <= 1024, 1 <= topk <= min(16, num_experts);
 * larger sizes return MOE_ERR_UNSUPPORTED_SHAPE before any launch.  It calls
 * no allocating routine.  The first call in each CUDA context (per device,
 * and again after that device's context is destroyed and recreated, e.g. by
 * cudaDeviceReset) looks up the array's device address and sets the kernel's
 * shared-memory attribute with that context current; make that first call
 * before any stream capture.  The set-up is guarded by a lock, so host
 * threads may make their first calls concurrently.  Every call on a device
 * shares the one array: calls that may overlap on the GPU (on different
 * streams without ordering) race and must not be issued.  Nothing in the
 * array needs clearing between calls: the kernel initialises all it reads.
 * Errors: INVALID_ARG (NULL expert_token_nums, or NULL expert_ids with
 * bs > 0), ALIGNMENT (expert_ids, expert_token_nums or a non-NULL expand_row
 * not 4-byte aligned), UNSUPPORTED_SHAPE, CUDA. */
int moe_fused_dispatch_noalloc(const int32_t* expert_ids, const uint8_t* x_active_mask, int32_t bs, int32_t topk,
                               int32_t num_experts, int32_t* expert_token_nums, int32_t* expand_row, void* stream);

/* ---- per-kernel timing (used by the benchmark) ---------------------------
 * With timing enabled, forward brackets each kernel launch with CUDA events on
 * `stream`.  get_timing synchronises the recorded events, writes for each
 * kernel id k < max_kernels the summed milliseconds ms[k] and launch count
 * launches[k] (host arrays), returns the number of kernel ids, and clears the
 * record.  Kernel ids: 0 dispatch + quant, 1 dispatch finish (multi-CTA
 * dispatch of batches with bs*topk > 8192; not launched otherwise), 2 expand
 * (f16 token rows for the tensor-core GEMMs), 3 GEMM1 + SwiGLU (+ requant)
 * for experts with at most 8 rows (dp4a weight streaming), 4 GEMM1 + dequant
 * for the other experts (tcgen05), 5 SwiGLU + requant of their rows, 6 GEMM2
 * + dequant (+ combine when every expert has at most 8 rows), 7 GEMM2 +
 * dequant (tcgen05), 8 combine.  A batch of at most 8 tokens runs every
 * expert through kernels 3 and 6 (an expert that repeated ids give more than
 * 8 rows in several slots of at most 8), so kernels 2, 4, 5, 7 and 8 are not
 * launched for it (2 still is with per-expert smooth scales, for the per-row
 * quant). */
int moe_fused_set_timing(moe_fused_handle_t* handle, int enable);
int moe_fused_get_timing(moe_fused_handle_t* handle, float* ms, int32_t* launches, int max_kernels);
const char* moe_fused_kernel_name(int kernel_id);

/* ---- test-only entry points (prefix moe_fused_debug_) -------------------
 * Workspace regions, so a test can read the intermediates of the last forward
 * or plant inputs for a single stage.  Region ids:
 *   0 status  1 counts [E]  2 offsets [E+1]  3 row_of [bs*topk]
 *   4 tk_of_row [bs*topk]  5 active tokens [bs]  6 x_q [bs_max,h] int8
 *   7 x_scale [bs_max] f32  8 xs_q [bs_max,h] int8  9 xs_scale [bs_max]
 *   10 h [rows,2*inter] f32 (the SwiGLU output of each GEMM1 row in its
 *      first inter floats, on both GEMM engines)  11 x2 [rows,inter] int8
 *      (codes of weight-streaming rows)  12 s2 [rows] f32
 *   13 y2 [bs_max*topk,h] in x's dtype  14 slot table
 *   15 row_token [rows] int32  16 shared_row [bs_max] int32
 *   17 row-block counters  18 token counters [bs_max]  19 token totals [bs_max]
 *   20 small-expert item ranges  21 x1h [rows,h] f16  22 x2h [rows,inter] f16
 *   23 multi-CTA dispatch counts [chunks][E] then skipped ids [chunks]
 *      (empty when bs_max*topk <= 8192: one CTA dispatches alone)
 *   24 amax2 [rows] f32: max |h| of each row of a tensor-core block (the
 *      GEMM1 epilogue's atomic maximum, read by the requant kernel)
 * `rows` = bs*topk + bs: routed row r at index r (r < R), the shared expert's
 * i-th active token at index bs*topk + i.  Writes *offset and *bytes. */
int moe_fused_debug_region(moe_fused_handle_t* handle, int region, size_t* offset, size_t* bytes);

/* Phase-stop forward: enqueue kernels 0..last_kernel of the forward (kernel
 * ids as for get_timing) and stop, so that a test can read the intermediates
 * of that stage before a later stage changes them (a forward that stops
 * before GEMM2 runs the small experts' GEMM1 in a launch of its own, without
 * the GEMM2 that otherwise streams behind it).  Same arguments, checks and
 * errors as moe_fused_forward. */
int moe_fused_debug_forward_until(moe_fused_handle_t* handle, const moe_fused_args_t* args, void* workspace,
                                  size_t workspace_bytes, int last_kernel, void* stream);

/* Range forward: enqueue kernels first_kernel..last_kernel of the forward
 * (kernel ids as for get_timing) on the state the workspace already holds
 * from an earlier call with the same args, e.g. GEMM2 and the combine after
 * a test has planted requantised codes and row scales (regions 11, 12 and
 * 22) into a workspace left by moe_fused_debug_forward_until(..., 5, ...).
 * A range that starts after kernel 3 runs the small experts' GEMM2 as a
 * launch of its own.  The per-token combine counters are reset by kernel 0
 * only, so GEMM2 and the combine may run once per dispatch.  Same checks
 * and errors as moe_fused_forward, plus INVALID_ARG for a bad range. */
int moe_fused_debug_forward_range(moe_fused_handle_t* handle, const moe_fused_args_t* args, void* workspace,
                                  size_t workspace_bytes, int first_kernel, int last_kernel, void* stream);

/* Run one grouped GEMM with a raw INT32 epilogue on the dispatch state and
 * operands currently in `workspace` (left by a forward with the same args):
 * which = 1: acc1[r, n] = sum_c xq(r)[c] * W1[e(r)][n][c] for every row
 *            r of the routed and shared groups, n < 2*inter;
 * which = 2: acc2[r, j] = sum_i x2[r][i] * W2[e(r)][j][i], j < hidden.
 * `acc` is a device int32 buffer [rows, N] (rows as for region 10); rows not
 * dispatched are left untouched. */
int moe_fused_debug_gemm_acc(moe_fused_handle_t* handle, const moe_fused_args_t* args, void* workspace,
                             size_t workspace_bytes, int which, int32_t* acc, void* stream);

/* Exercise the kernels' bounded waits: one thread waits for something that
 * never happens -- which = 0: an mbarrier phase nobody arrives on; which = 1:
 * a workspace flag nobody sets (the cross-CTA ready-flag spin) -- gives up
 * after the wait budget (2 s), records kErrWaitTimeout and site
 * MOE_DEBUG_WAIT_SITE + which in the workspace's status word, and returns.
 * Nothing faults or traps; the next forward clears the status.  Asynchronous
 * on `stream`; read the result with moe_fused_get_status, which then returns
 * MOE_ERR_DEVICE_TIMEOUT.  MOE_ERR_INVALID_ARG for a bad handle, workspace or
 * `which`, MOE_ERR_WORKSPACE_TOO_SMALL below the reported size. */
#define MOE_DEBUG_WAIT_SITE 240
int moe_fused_debug_wait_timeout(moe_fused_handle_t* handle, void* workspace, size_t workspace_bytes, int which,
                                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FUSED_H */
