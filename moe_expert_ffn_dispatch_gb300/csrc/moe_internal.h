// Internal host/device declarations shared by the kernels and the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// status word indices (int32) at the start of the workspace
enum StatusWord : int {
  kStSkipped = 0,
  kStErrorFlags = 1,
  kStErrorSite = 2,
  kStRows = 3,
  kStSharedRows = 4,
  kStSlots = 5,
  // arrival counters of the GEMM launches whose CTAs take their work in
  // arrival order (engines side by side): small, big GEMM1, big GEMM2; the
  // dispatch zeroes them every forward, before those launches start
  kStCtaCounter = 40,
};
constexpr int kErrWaitTimeout = 1;

// ---------------------------------------------------------------- layout
// Workspace regions (byte offsets, 256-byte aligned).  `rows` = bs_max*topk
// routed rows + bs_max shared rows.  y2 has a region of its own (it no
// longer aliases h: the small experts' GEMM2 runs in the same launch as
// their GEMM1, while other CTAs may still write and read h).
struct WsLayout {
  size_t status;     // 64 int32 status words
  size_t counts;     // [E] int32
  size_t offsets;    // [E+1] int32
  size_t row_of;     // [bs_max*topk] int32
  size_t tk_of_row;  // [bs_max*topk] int32
  size_t active;     // [bs_max] int32: i-th active token
  size_t x_q;        // [bs_max, h] int8
  size_t x_scale;    // [bs_max] f32
  size_t xs_q;       // [bs_max, h] int8 (shared-expert quant)
  size_t xs_scale;   // [bs_max] f32
  size_t hbuf;       // [rows, 2I] f32: the SwiGLU output h of each GEMM1 row in [0, I)
  size_t x2;         // [rows, I] int8
  size_t s2;         // [rows] f32
  size_t y2;         // [bs_max*topk, h] bf16 (x's dtype)
  size_t slots;      // slot table (int32), see SlotTable
  size_t row_token;  // [rows] int32: token of each GEMM row (routed and shared)
  size_t shared_row; // [bs_max] int32: shared-expert row of token t, -1 if inactive
  size_t blk_ticket; // int32 per row block: GEMM1 tiles done (last one requantises)
  size_t tok_ticket; // [bs_max] int32: GEMM2 output columns done per token
  size_t tok_expect; // [bs_max] int32: columns that complete a token (rows * h)
  size_t ranges;     // [2][kMaxCtas + 1] int32: small-phase item range of each CTA (GEMM1, GEMM2)
  size_t x1h;        // [rows, h] f16: GEMM1 token operand of the rows in big blocks (codes as f16)
  size_t x2h;        // [rows, I] f16: GEMM2 token operand of the rows in big blocks
  size_t dcnt;       // multi-CTA dispatch: [chunks][E] rows per (chunk, expert), then [chunks] skipped ids
  size_t amax2;      // [rows] f32 bits: max |h| of each tensor-core row (atomic max from the GEMM1 epilogue)
  size_t bar_tags;   // [kMaxCtas] u64: the one-launch kernel's grid barrier (word 0 its generation, word b
                     // the arrival tag of CTA b); any initial content works
  size_t total;
  size_t sizes[32];  // bytes per region id (debug_region)
};

// Region ids (moe_fused_debug_region); the order of WsLayout's fields.
enum Region : int {
  kRegStatus = 0, kRegCounts, kRegOffsets, kRegRowOf, kRegTkOfRow, kRegActive, kRegXq, kRegXScale,
  kRegXsq, kRegXsScale, kRegH, kRegX2, kRegS2, kRegY2, kRegSlots, kRegRowToken, kRegSharedRow,
  kRegBlkTicket, kRegTokTicket, kRegTokExpect, kRegRanges, kRegX1h, kRegX2h, kRegDcnt, kRegAmax2, kRegBarTags,
  kNumRegions
};

constexpr int kMaxCtas = 1023;  // persistent grid size limit (one CTA per SM)

// Slot table: the experts that received rows, split by row count.  Experts
// with at most kSmallRows rows ("small", decode-like) go to the weight-
// streaming dp4a kernel, the others ("big") to the tensor-core kernel in
// token blocks of kTokenBlock rows.  The shared expert is one more slot in
// whichever list its row count selects (expert id -1).  In a batch of at
// most kSmallRows tokens every expert is small: one whose repeated ids give
// it more rows takes several small slots of at most kSmallRows rows (see
// FwdParams::small_only).  Stored as int32 words at layout.slots:
//   header: [0] n_big  [1] token blocks over big slots  [2] R  [3] S
//           [4] n_small  [5] CTAs of the small phase (the item ranges are
//           split over these)  [6] engines side by side (the GEMM launches'
//           CTAs take their work in arrival order; the big launches use the
//           num_ctas - [5] CTAs the small phase leaves)  [7] reserved
//   then seven arrays of stride (E + 2 + kSplitSlots):
//     big:   expert id, first row, row count, exclusive prefix of blocks
//     small: expert id, first row, row count
constexpr int kMaxTopk = 16;
// Extra small slots a batch of at most kSmallRows tokens can need: an expert
// with c rows takes ceil(c / kSmallRows) slots, one more than its share of
// the at most kSmallRows * kMaxTopk routed rows, kSmallRows rows a slot.
constexpr int kSplitSlots = kMaxTopk;
struct SlotTable {
  static constexpr int kHeader = 8;
  static constexpr int kNumBig = 0, kBigBlocks = 1, kRows = 2, kSharedRows = 3, kNumSmall = 4;
  static constexpr int kSmallCtas = 5, kSplit = 6;
  static __host__ __device__ int stride(int E) { return E + 2 + kSplitSlots; }
  static __host__ __device__ int words(int E) { return kHeader + 7 * stride(E); }
};

constexpr int kSmallRows = 8;     // experts with <= this many rows take the dp4a path ...
constexpr int kSmallMaxK = 4096;  // ... when both contraction lengths are at most this
constexpr int kTokenBlock = 128;  // token rows per big-phase work item (the MMA's N)
constexpr int kDispChunk = 2048;  // flat (t, k) pairs per CTA of the multi-CTA dispatch

// ---------------------------------------------------------------- params
struct FwdParams {
  int32_t bs, h, E, topk, I, has_shared;
  int32_t share_uses_xq;  // shared quant identical to routed quant (same smooth vector)
  int32_t fold_routing;   // routing weight folded into the GEMM2 row scale; combine is a plain sum
  int32_t disp_chunks;    // dispatch chunks of kDispChunk pairs; <= 1: one CTA dispatches alone
  int32_t with_tickets;   // dispatch resets the GEMM epilogue counters (forward path)
  int32_t small_rows;     // row count up to which an expert takes the dp4a path (0: never)
  int32_t small_only;     // bs <= small_rows: every expert takes the dp4a path (an expert with
                          // more rows, from repeated ids, in slots of at most small_rows rows), so
                          // no big block exists and the tensor-core launches are skipped
  int32_t num_ctas;       // grid of the GEMM launches (<= kMaxCtas)
  int32_t split_engines;  // the dp4a launch and the tensor-core chain run side by side on disjoint CTA
                          // sets, split by the dispatch (slot table words 5 and 6)
  int32_t act_fp16;       // x, y2 and the outputs are fp16 (else bf16)
  int32_t scale_dtype;    // routed weight scales: 0 fp32, 1 bf16, 2 fp16
  int32_t xq_per_row;     // per-expert smooth: routed x_q / x_scale are indexed by row, not token
  uint64_t bar_salt;      // the handle's random constant mixed into the grid barrier's arrival tags
  const uint16_t* x;
  const int32_t* ids;
  const float* scales;
  const int8_t* w1;
  const void* w1s;        // dtype scale_dtype
  const int8_t* w2;
  const void* w2s;        // dtype scale_dtype
  const int8_t* sw1;
  const float* sw1s;
  const int8_t* sw2;
  const float* sw2s;
  const float* smooth;
  const float* ssmooth;
  const uint8_t* mask;
  uint16_t* out;
  uint16_t* sout;
  int32_t* token_nums;
  char* ws;
  WsLayout L;
};

template <typename T>
__host__ __device__ inline T* ws_ptr(const FwdParams& p, size_t off) {
  return reinterpret_cast<T*>(p.ws + off);
}

// kernel ids (timing / status sites)
enum KernelId : int {
  kKDispatchQuant = 0,
  kKDispatchFinish = 1,
  kKExpand = 2,
  kKGemm1Small = 3,
  kKGemm1Big = 4,
  kKRequantBig = 5,
  kKGemm2Small = 6,
  kKGemm2Big = 7,
  kKCombine = 8,
  kNumKernels = 9
};

// TMA descriptors of the big-phase operands (built on the host per forward).
struct alignas(64) TcMaps {
  CUtensorMap a1;   // W1 [E*2I, h] int8, box {128, 16} (16-row gate / up groups), 128-byte swizzle
  CUtensorMap a1s;  // shared W1 [2I, h] int8, box {128, 16}, 128-byte swizzle
  CUtensorMap a2;   // W2 [E*h, I] int8, box {128, 128}, 128-byte swizzle
  CUtensorMap a2s;  // shared W2 [h, I] int8, box {128, 128}, 128-byte swizzle
  CUtensorMap b1;   // x1h [rows, h] f16, box {64, 128}, 128-byte swizzle
  CUtensorMap b2;   // x2h [rows, I] f16, box {64, 128}, 128-byte swizzle
  CUtensorMap b1n;  // x1h, box {64, 16}: blocks of at most 64 rows
  CUtensorMap b2n;  // x2h, box {64, 16}
};

// GEMM modes
enum GemmMode : int { kGemm1SwiGLU = 0, kGemm2Bf16 = 1, kGemm1Raw = 2, kGemm2Raw = 3 };

// How a launch joins its stream: programmatic stream serialisation (the
// kernel may start while its predecessor drains and waits for it in-kernel;
// the default), and optionally an event recorded once every CTA of the launch
// has begun (launch completion).
struct LaunchOpts {
  bool pdl = true;
  cudaEvent_t started = nullptr;
};

inline cudaLaunchConfig_t launch_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr,
                                        const LaunchOpts& o) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  unsigned n = 0;
  if (o.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (o.started) {
    attr[n].id = cudaLaunchAttributeLaunchCompletionEvent;
    attr[n].val.launchCompletionEvent.event = o.started;
    attr[n].val.launchCompletionEvent.flags = 0;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

// The default: programmatic stream serialisation only.  attr: 2 entries.
inline cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, cudaLaunchAttribute* attr) {
  return launch_config(grid, block, smem, s, attr, LaunchOpts());
}

// ---------------------------------------------------------------- launches
size_t dispatch_smem_bytes(int E);
cudaError_t launch_dispatch_quant(const FwdParams& p, cudaStream_t s);
cudaError_t launch_expand(const FwdParams& p, cudaStream_t s);
cudaError_t launch_dispatch_finish(const FwdParams& p, cudaStream_t s);
cudaError_t launch_requant_big(const FwdParams& p, cudaStream_t s, const LaunchOpts& o = LaunchOpts());
cudaError_t launch_combine(const FwdParams& p, cudaStream_t s);
cudaError_t launch_moe_gemm_small(const FwdParams& p, int mode, int32_t* raw_acc, int num_ctas, cudaStream_t s);
// GEMM1 then GEMM2 of the small experts in one launch (GEMM2 streamed behind GEMM1)
cudaError_t launch_moe_gemm_small_streamed(const FwdParams& p, int num_ctas, cudaStream_t s,
                                           const LaunchOpts& o = LaunchOpts());
// the whole forward of a batch of at most small_rows tokens (small_only, token
// quant) in one launch of num_ctas CTAs: dispatch, quant, GEMM1, GEMM2, combine
cudaError_t launch_moe_decode_one_launch(const FwdParams& p, cudaStream_t s);
cudaError_t launch_moe_gemm_big(const FwdParams& p, const TcMaps& maps, int mode, int32_t* raw_acc, int num_ctas,
                                cudaStream_t s, const LaunchOpts& o = LaunchOpts());
cudaError_t moe_gemm_small_prepare_attributes();
cudaError_t moe_gemm_big_prepare_attributes();
cudaError_t dispatch_prepare_attributes(int E);
int dispatch_noalloc(const int32_t* expert_ids, const uint8_t* mask, int bs, int topk, int E,
                     int32_t* expert_token_nums, int32_t* expand_row, cudaStream_t s);

}  // namespace moe
