// C ABI of the fused MoE expert block: argument checks, workspace planning,
// launch sequence, per-kernel timing and the test-only entry points.
//
// Launch sequence of one forward (Process() of the FusedDeepMoE analysis
// §3.2: dispatch, GMM1 with SwiGLU + quant, GMM2 with combine):
//   dispatch + quant -> expand (f16 token rows of big blocks) ->
//   GEMM1 + SwiGLU (+ requant, small experts) -> GEMM1 + SwiGLU (big) ->
//   requant of big blocks -> GEMM2 + bf16 dequant (+ combine when no big
//   blocks) -> GEMM2 (big) -> combine (when big blocks exist).
// Kernel boundaries carry the dependencies; inside a GEMM launch the fused
// epilogues run in the CTA that finishes a block last, and a GEMM2 streamed
// behind GEMM1 waits (bounded) for the requant of its rows.  A batch of at
// most 8 tokens with per-token quant runs the whole forward as one launch
// (moe_decode_one_launch_kernel).
#include <cstdio>
#include <cstring>
#include <chrono>
#include <new>
#include <random>
#include <vector>

#include <cuda.h>

#include "device_prims.cuh"
#include "moe_fused.h"
#include "moe_internal.h"

struct TimingRecord {
  int kernel;
  cudaEvent_t start, stop;
};

struct moe_fused_handle {
  moe_fused_config_t cfg;
  int device;
  int num_sms;
  moe::WsLayout L;
  bool timing;
  std::vector<TimingRecord> records;
  std::vector<cudaEvent_t> pool;
  moe::TcMaps maps;          // tensor maps of the last forward's operands
  const void* map_key[5];    // pointers they were built for
  bool maps_valid;
  // random constant mixed into the one-launch grid barrier's arrival tags
  uint64_t bar_salt;
  // engines side by side: the tensor-core chain's stream, and the events of
  // the fork (after expand), of the tensor-core GEMM1's launch completion
  // (every CTA begun) and of the join (before the combine)
  cudaStream_t side;
  cudaEvent_t ev_fork, ev_started, ev_join;
};

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

int check_config(const moe_fused_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const int32_t known = MOE_FLAG_UNFUSED | MOE_FLAG_FOLD_ROUTING | MOE_FLAG_FP16_ACT | MOE_FLAG_SCALE_BF16 |
                        MOE_FLAG_SCALE_FP16 | MOE_FLAG_EXPERT_SMOOTH;
  if ((c->flags & ~known) != 0) return MOE_ERR_INVALID_ARG;
  if ((c->flags & MOE_FLAG_SCALE_BF16) && (c->flags & MOE_FLAG_SCALE_FP16)) return MOE_ERR_INVALID_ARG;
  if (c->hidden < 64 || c->hidden > 16384 || c->hidden % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->inter < 64 || c->inter > 16384 || c->inter % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->num_experts < 1 || c->num_experts > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->topk < 1 || c->topk > 16 || c->topk > c->num_experts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->bs_max < 0 || c->bs_max > 65536) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c->has_shared != 0 && c->has_shared != 1) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe::WsLayout plan(const moe_fused_config_t& c) {
  moe::WsLayout L{};
  const size_t bs = static_cast<size_t>(c.bs_max), E = static_cast<size_t>(c.num_experts);
  const size_t h = static_cast<size_t>(c.hidden), I = static_cast<size_t>(c.inter), K = static_cast<size_t>(c.topk);
  const size_t routed = bs * K;
  const size_t rows = routed + (c.has_shared ? bs : 0);
  size_t off = 0;
  auto take = [&](size_t& field, size_t bytes, int id) {
    field = off;
    L.sizes[id] = bytes;
    off = align_up(off + (bytes ? bytes : 1));
  };
  const size_t big_blocks = (rows + moe::kTokenBlock - 1) / moe::kTokenBlock + E + 2;
  take(L.status, 64 * sizeof(int32_t), moe::kRegStatus);
  take(L.counts, E * 4, moe::kRegCounts);
  take(L.offsets, (E + 1) * 4, moe::kRegOffsets);
  take(L.row_of, routed * 4, moe::kRegRowOf);
  take(L.tk_of_row, routed * 4, moe::kRegTkOfRow);
  take(L.active, bs * 4, moe::kRegActive);
  // per-expert smooth scales quantise every routed row on its own
  const size_t xq_rows = (c.flags & MOE_FLAG_EXPERT_SMOOTH) ? routed : bs;
  take(L.x_q, xq_rows * h, moe::kRegXq);
  take(L.x_scale, xq_rows * 4, moe::kRegXScale);
  take(L.xs_q, c.has_shared ? bs * h : 0, moe::kRegXsq);
  take(L.xs_scale, c.has_shared ? bs * 4 : 0, moe::kRegXsScale);
  // h rows are 2I floats wide (both GEMM1 engines store the SwiGLU output in
  // the first I)
  // y2 has its own region: the small experts' GEMM2 runs in the same launch
  // as their GEMM1, while other CTAs may still write and read h
  const size_t hbytes = rows * 2 * I * 4, ybytes = routed * h * 2;
  take(L.hbuf, hbytes, moe::kRegH);
  take(L.x2, rows * I, moe::kRegX2);
  take(L.s2, rows * 4, moe::kRegS2);
  take(L.y2, ybytes, moe::kRegY2);
  take(L.slots, static_cast<size_t>(moe::SlotTable::words(c.num_experts)) * 4, moe::kRegSlots);
  take(L.row_token, rows * 4, moe::kRegRowToken);
  take(L.shared_row, bs * 4, moe::kRegSharedRow);
  take(L.blk_ticket, (static_cast<size_t>(moe::SlotTable::stride(c.num_experts)) + big_blocks) * 4, moe::kRegBlkTicket);
  take(L.tok_ticket, bs * 4, moe::kRegTokTicket);
  take(L.tok_expect, bs * 4, moe::kRegTokExpect);
  take(L.ranges, 2 * (moe::kMaxCtas + 1) * 4, moe::kRegRanges);
  take(L.x1h, rows * h * 2, moe::kRegX1h);
  take(L.x2h, rows * I * 2, moe::kRegX2h);
  const size_t chunks = routed > 4 * moe::kDispChunk ? (routed + moe::kDispChunk - 1) / moe::kDispChunk : 1;
  take(L.dcnt, chunks > 1 ? (chunks * E + chunks) * 4 : 0, moe::kRegDcnt);
  take(L.amax2, rows * 4, moe::kRegAmax2);
  take(L.bar_tags, moe::kMaxCtas * sizeof(uint64_t), moe::kRegBarTags);
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int build_params(moe_fused_handle* hd, const moe_fused_args_t* a, void* ws, size_t ws_bytes, moe::FwdParams* p) {
  if (!hd || !a) return MOE_ERR_INVALID_ARG;
  const moe_fused_config_t& c = hd->cfg;
  if (a->bs < 0 || a->bs > c.bs_max) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < hd->L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_ALIGNMENT;
  if (!a->expert_token_nums) return MOE_ERR_INVALID_ARG;
  if (a->bs > 0) {
    if (!a->x || !a->expert_ids || !a->expert_scales || !a->gmm1_weight || !a->gmm1_weight_scale ||
        !a->gmm2_weight || !a->gmm2_weight_scale || !a->output)
      return MOE_ERR_INVALID_ARG;
    if (c.has_shared) {
      if (!a->share_gmm1_weight || !a->share_gmm1_weight_scale || !a->share_gmm2_weight ||
          !a->share_gmm2_weight_scale || !a->share_output)
        return MOE_ERR_INVALID_ARG;
    } else if (a->share_output) {
      return MOE_ERR_INVALID_ARG;
    }
    const void* ptrs[] = {a->x, a->expert_ids, a->expert_scales, a->gmm1_weight, a->gmm1_weight_scale,
                          a->gmm2_weight, a->gmm2_weight_scale, a->share_gmm1_weight, a->share_gmm1_weight_scale,
                          a->share_gmm2_weight, a->share_gmm2_weight_scale, a->expert_smooth_scales,
                          a->share_smooth_scales, a->x_active_mask, a->output, a->share_output,
                          a->expert_token_nums};
    for (const void* q : ptrs)
      if (q && !aligned16(q)) return MOE_ERR_ALIGNMENT;
  }
  std::memset(p, 0, sizeof(*p));
  p->bs = a->bs;
  p->h = c.hidden;
  p->E = c.num_experts;
  p->topk = c.topk;
  p->I = c.inter;
  p->has_shared = c.has_shared;
  // [E, h] smooth scales (when given) make the routed quant per row
  p->xq_per_row = (c.flags & MOE_FLAG_EXPERT_SMOOTH) != 0 && a->expert_smooth_scales != nullptr;
  p->share_uses_xq = c.has_shared && !p->xq_per_row && (a->expert_smooth_scales == a->share_smooth_scales);
  p->act_fp16 = (c.flags & MOE_FLAG_FP16_ACT) != 0;
  p->scale_dtype = (c.flags & MOE_FLAG_SCALE_BF16) ? 1 : (c.flags & MOE_FLAG_SCALE_FP16) ? 2 : 0;
  p->fold_routing = (c.flags & MOE_FLAG_FOLD_ROUTING) != 0;
  // the second launch of the multi-CTA dispatch pays off above a few chunks
  const int nf = a->bs * c.topk;
  p->disp_chunks = nf > 4 * moe::kDispChunk ? (nf + moe::kDispChunk - 1) / moe::kDispChunk : 1;
  p->with_tickets = 1;
  const bool fused_ok = (c.flags & MOE_FLAG_UNFUSED) == 0 && c.hidden <= moe::kSmallMaxK && c.inter <= moe::kSmallMaxK;
  p->small_rows = fused_ok ? moe::kSmallRows : 0;
  // a batch of at most small_rows tokens never needs the tensor-core path: an
  // expert can exceed small_rows rows only through repeated ids, and then takes
  // several small slots (its weights streamed once per slot)
  p->small_only = p->small_rows > 0 && a->bs <= p->small_rows;
  p->num_ctas = hd->num_sms < moe::kMaxCtas ? hd->num_sms : moe::kMaxCtas;
  p->x = static_cast<const uint16_t*>(a->x);
  p->ids = a->expert_ids;
  p->scales = a->expert_scales;
  p->w1 = a->gmm1_weight;
  p->w1s = a->gmm1_weight_scale;
  p->w2 = a->gmm2_weight;
  p->w2s = a->gmm2_weight_scale;
  p->sw1 = a->share_gmm1_weight;
  p->sw1s = a->share_gmm1_weight_scale;
  p->sw2 = a->share_gmm2_weight;
  p->sw2s = a->share_gmm2_weight_scale;
  p->smooth = a->expert_smooth_scales;
  p->ssmooth = a->share_smooth_scales;
  p->mask = a->x_active_mask;
  p->out = static_cast<uint16_t*>(a->output);
  p->sout = static_cast<uint16_t*>(a->share_output);
  p->token_nums = a->expert_token_nums;
  p->ws = static_cast<char*>(ws);
  p->L = hd->L;
  p->bar_salt = hd->bar_salt;
  return MOE_OK;
}

cudaEvent_t take_event(moe_fused_handle* hd) {
  if (!hd->pool.empty()) {
    cudaEvent_t e = hd->pool.back();
    hd->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launch `fn` bracketed by timing events when enabled.
template <typename F>
cudaError_t timed(moe_fused_handle* hd, int kernel, cudaStream_t s, F fn) {
  if (!hd->timing) return fn();
  TimingRecord r{kernel, take_event(hd), take_event(hd)};
  if (!r.start || !r.stop) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaEventRecord(r.start, s);
  if (e != cudaSuccess) return e;
  e = fn();
  if (e != cudaSuccess) return e;
  e = cudaEventRecord(r.stop, s);
  if (e != cudaSuccess) return e;
  try {
    hd->records.push_back(r);
  } catch (...) {  // no exception leaves a C entry point
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
    return cudaErrorMemoryAllocation;
  }
  return cudaSuccess;
}

// ---- TMA descriptors for the tensor-core path -----------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// 2-D row-major [rows][cols] tensor, box {box_cols, box_rows}
bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, size_t elem, uint64_t rows, uint64_t cols,
               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * elem};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Build (or reuse) the tensor maps of this forward's operands.
int prepare_maps(moe_fused_handle* hd, const moe::FwdParams& p) {
  const void* key[5] = {p.w1, p.w2, p.sw1, p.sw2, p.ws};
  if (hd->maps_valid && std::memcmp(key, hd->map_key, sizeof(key)) == 0) return MOE_OK;
  const moe_fused_config_t& c = hd->cfg;
  const uint64_t E = c.num_experts, h = c.hidden, I = c.inter;
  const uint64_t rows = static_cast<uint64_t>(c.bs_max) * c.topk + (c.has_shared ? c.bs_max : 0);
  const uint64_t brows = rows > 0 ? rows : 1;
  const void* sw1 = p.sw1 ? p.sw1 : p.w1;
  const void* sw2 = p.sw2 ? p.sw2 : p.w2;
  moe::TcMaps& m = hd->maps;
  bool ok = encode_2d(&m.a1, p.w1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, E * 2 * I, h, 128, 16, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.a1s, sw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 2 * I, h, 128, 16, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.a2, p.w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, E * h, I, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.a2s, sw2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, h, I, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.b1, p.ws + p.L.x1h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, brows, h, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.b2, p.ws + p.L.x2h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, brows, I, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.b1n, p.ws + p.L.x1h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, brows, h, 64, 16,
                      CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode_2d(&m.b2n, p.ws + p.L.x2h, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, brows, I, 64, 16,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) {
    hd->maps_valid = false;
    return MOE_ERR_CUDA;
  }
  std::memcpy(hd->map_key, key, sizeof(key));
  hd->maps_valid = true;
  return MOE_OK;
}

// One thread waits for what never comes (see moe_fused_debug_wait_timeout):
// an mbarrier phase without arrivals, or a flag nobody sets.  The bounded
// wait records the timeout in the status word and returns.
__global__ void debug_wait_kernel(int32_t* status, const int32_t* flag, int which) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bar, 1);
    abort_flag = 0;
    moe::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  volatile int* ab = &abort_flag;
  if (which == 0) moe::mbar_wait_bounded(&bar, 0, ab, status, MOE_DEBUG_WAIT_SITE);
  else moe::spin_until_ge(flag, 1, ab, status, MOE_DEBUG_WAIT_SITE + 1);
}

int cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  std::fprintf(stderr, "moe_fused: CUDA error %s\n", cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

int moe_fused_workspace_size(const moe_fused_config_t* cfg, size_t* workspace_bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!workspace_bytes) return MOE_ERR_INVALID_ARG;
  *workspace_bytes = plan(*cfg).total;
  return MOE_OK;
}

int moe_fused_create(const moe_fused_config_t* cfg, moe_fused_handle_t** out_handle, size_t* workspace_bytes) {
  int rc = check_config(cfg);
  if (rc) return rc;
  if (!out_handle) return MOE_ERR_INVALID_ARG;
  *out_handle = nullptr;
  moe_fused_handle* hd = new (std::nothrow) moe_fused_handle();
  if (!hd) return MOE_ERR_INVALID_ARG;
  hd->cfg = *cfg;
  hd->timing = false;
  hd->maps_valid = false;
  hd->side = nullptr;
  hd->ev_fork = hd->ev_started = hd->ev_join = nullptr;
  {
    // the grid barrier's salt: random where the platform has an entropy
    // source, else the clock and the handle's address alone (no exception
    // leaves this C entry point)
    const uint64_t t = static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
    uint64_t r = 0;
    try {
      std::random_device rd;
      r = (static_cast<uint64_t>(rd()) << 32) ^ rd();
    } catch (...) {
      r = 0;
    }
    hd->bar_salt = r ^ (t * 0x9E3779B97F4A7C15ull) ^ static_cast<uint64_t>(reinterpret_cast<uintptr_t>(hd));
  }
  cudaError_t e = cudaGetDevice(&hd->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&hd->num_sms, cudaDevAttrMultiProcessorCount, hd->device);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hd->side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hd->ev_fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hd->ev_started, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hd->ev_join, cudaEventDisableTiming);
  if (e == cudaSuccess) e = moe::moe_gemm_small_prepare_attributes();
  if (e == cudaSuccess) e = moe::moe_gemm_big_prepare_attributes();
  if (e == cudaSuccess) e = moe::dispatch_prepare_attributes(1024);
  if (e != cudaSuccess) {
    moe_fused_destroy(hd);
    return cuda_fail(e);
  }
  hd->L = plan(*cfg);
  if (workspace_bytes) *workspace_bytes = hd->L.total;
  *out_handle = hd;
  return MOE_OK;
}

int moe_fused_forward(moe_fused_handle_t* hd, const moe_fused_args_t* args, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return moe_fused_debug_forward_range(hd, args, workspace, workspace_bytes, 0, moe::kNumKernels - 1, stream);
}

int moe_fused_debug_forward_until(moe_fused_handle_t* hd, const moe_fused_args_t* args, void* workspace,
                                  size_t workspace_bytes, int last_kernel, void* stream) {
  return moe_fused_debug_forward_range(hd, args, workspace, workspace_bytes, 0, last_kernel, stream);
}

int moe_fused_debug_forward_range(moe_fused_handle_t* hd, const moe_fused_args_t* args, void* workspace,
                                  size_t workspace_bytes, int first_kernel, int last_kernel, void* stream) {
  moe::FwdParams p;
  int rc = build_params(hd, args, workspace, workspace_bytes, &p);
  if (rc) return rc;
  if (first_kernel < 0 || last_kernel >= moe::kNumKernels || first_kernel > last_kernel) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p.bs == 0) {
    if (first_kernel > 0) return MOE_OK;  // nothing was dispatched: later stages have no work
    e = cudaMemsetAsync(args->expert_token_nums, 0, sizeof(int32_t) * hd->cfg.num_experts, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.ws + p.L.status, 0, 64 * sizeof(int32_t), s);
    return cuda_fail(e);
  }
  // A batch of at most small_rows tokens with per-token quant: the whole
  // forward is one launch (dispatch and quant repeated per CTA, then the
  // streamed GEMMs behind a grid barrier that needs no initial state).
  const bool one_launch =
      p.small_only && !p.xq_per_row && first_kernel == moe::kKDispatchQuant && last_kernel >= moe::kKGemm2Small;
  // A whole forward of a larger batch on the fused path runs the dp4a launch
  // and the tensor-core chain side by side (below); the dispatch splits the
  // CTAs between them and zeroes the launches' arrival counters.
  p.split_engines = p.small_rows > 0 && !p.small_only && first_kernel == moe::kKDispatchQuant &&
                    last_kernel == moe::kKCombine;
  if (one_launch)
    return cuda_fail(timed(hd, moe::kKGemm1Small, s, [&] { return moe::launch_moe_decode_one_launch(p, s); }));
  rc = prepare_maps(hd, p);
  if (rc) return rc;
  const int sms = p.num_ctas;
  const moe::TcMaps& maps = hd->maps;
  // the small experts' GEMM2 streams behind their GEMM1 in one launch when
  // the range holds both (a range that stops after GEMM1 keeps h intact; one
  // that starts after it runs the small GEMM2 as a launch of its own)
  const bool streamed =
      p.small_rows > 0 && first_kernel <= moe::kKGemm1Small && last_kernel >= moe::kKGemm2Small;
  auto run = [&](int k) -> cudaError_t {
    switch (k) {
      case moe::kKDispatchQuant: return moe::launch_dispatch_quant(p, s);
      case moe::kKDispatchFinish: return moe::launch_dispatch_finish(p, s);
      case moe::kKExpand: return moe::launch_expand(p, s);
      case moe::kKGemm1Small:
        return streamed ? moe::launch_moe_gemm_small_streamed(p, sms, s)
                        : moe::launch_moe_gemm_small(p, moe::kGemm1SwiGLU, nullptr, sms, s);
      case moe::kKGemm1Big: return moe::launch_moe_gemm_big(p, maps, moe::kGemm1SwiGLU, nullptr, sms, s);
      case moe::kKRequantBig: return moe::launch_requant_big(p, s);
      case moe::kKGemm2Small: return moe::launch_moe_gemm_small(p, moe::kGemm2Bf16, nullptr, sms, s);
      case moe::kKGemm2Big: return moe::launch_moe_gemm_big(p, maps, moe::kGemm2Bf16, nullptr, sms, s);
      default: return moe::launch_combine(p, s);
    }
  };
  if (p.split_engines) {
    // Stream s: dispatch (+ finish) and expand.  Side stream: the tensor-core
    // GEMM1, the requant, GEMM2.  Stream s again, once every CTA of the
    // tensor-core GEMM1 has begun (so that its CTAs hold their SMs before the
    // dp4a launch fills the rest): the dp4a launch; then, after the side
    // stream, the combine.  Neither the tensor-core GEMM1 nor the requant
    // starts early behind its predecessor: CTAs waiting for a predecessor
    // would hold SMs that the other engine's CTAs need.
    e = cudaSuccess;
    for (int k = moe::kKDispatchQuant; k <= moe::kKExpand && e == cudaSuccess; ++k) {
      if (k == moe::kKDispatchFinish && p.disp_chunks <= 1) continue;
      e = timed(hd, k, s, [&] { return run(k); });
    }
    if (e == cudaSuccess) e = cudaEventRecord(hd->ev_fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hd->side, hd->ev_fork, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    moe::LaunchOpts first_big;
    first_big.pdl = false;
    first_big.started = hd->ev_started;
    moe::LaunchOpts no_pdl;
    no_pdl.pdl = false;
    e = timed(hd, moe::kKGemm1Big, hd->side, [&] {
      return moe::launch_moe_gemm_big(p, maps, moe::kGemm1SwiGLU, nullptr, sms, hd->side, first_big);
    });
    if (e == cudaSuccess)
      e = timed(hd, moe::kKRequantBig, hd->side, [&] { return moe::launch_requant_big(p, hd->side, no_pdl); });
    if (e == cudaSuccess)
      e = timed(hd, moe::kKGemm2Big, hd->side,
                [&] { return moe::launch_moe_gemm_big(p, maps, moe::kGemm2Bf16, nullptr, sms, hd->side); });
    // the side stream always rejoins s (a capture must not be left forked)
    const cudaError_t ej = cudaEventRecord(hd->ev_join, hd->side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hd->ev_started, 0);
    if (e == cudaSuccess)
      e = timed(hd, moe::kKGemm1Small, s, [&] { return moe::launch_moe_gemm_small_streamed(p, sms, s, no_pdl); });
    const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(s, hd->ev_join, 0) : ej;
    if (e == cudaSuccess) e = ew;
    if (e == cudaSuccess) e = timed(hd, moe::kKCombine, s, [&] { return run(moe::kKCombine); });
    return cuda_fail(e);
  }
  e = cudaSuccess;
  for (int k = first_kernel; k <= last_kernel && e == cudaSuccess; ++k) {
    if (k == moe::kKDispatchFinish && p.disp_chunks <= 1) continue;  // one-CTA dispatch: nothing to launch
    if (k == moe::kKGemm2Small && streamed) continue;                 // ran inside the GEMM1 launch
    // no big block can exist: the tensor-core GEMMs, their requant and the
    // combine kernel would return at once (the small GEMM2 combines every
    // token), and the expand kernel too unless it quantises per routed row
    if (p.small_only && (k == moe::kKGemm1Big || k == moe::kKRequantBig || k == moe::kKGemm2Big ||
                         k == moe::kKCombine || (k == moe::kKExpand && !p.xq_per_row)))
      continue;
    e = timed(hd, k, s, [&] { return run(k); });
  }
  return cuda_fail(e);
}

int moe_fused_get_status(moe_fused_handle_t* hd, const void* workspace, void* stream, moe_fused_status_t* out) {
  if (!hd || !workspace || !out) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t w[8];
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpy(w, static_cast<const char*>(workspace) + hd->L.status, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  out->skipped_pairs = w[moe::kStSkipped];
  out->error_flags = w[moe::kStErrorFlags];
  out->error_site = w[moe::kStErrorSite];
  out->dispatched_rows = w[moe::kStRows];
  out->shared_rows = w[moe::kStSharedRows];
  out->active_slots = w[moe::kStSlots];
  out->reserved[0] = out->reserved[1] = 0;
  if (out->error_flags & moe::kErrWaitTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  return MOE_OK;
}

int moe_fused_destroy(moe_fused_handle_t* hd) {
  if (!hd) return MOE_OK;
  for (auto& r : hd->records) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  for (auto e : hd->pool) cudaEventDestroy(e);
  for (cudaEvent_t e : {hd->ev_fork, hd->ev_started, hd->ev_join})
    if (e) cudaEventDestroy(e);
  if (hd->side) cudaStreamDestroy(hd->side);
  delete hd;
  return MOE_OK;
}

const char* moe_fused_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_UNIMPLEMENTED: return "not implemented";
    case MOE_ERR_ALIGNMENT: return "pointer not aligned (forward: 16-byte, workspace 256-byte; no-alloc dispatch: 4-byte)";
    default: return "unknown error";
  }
}

int moe_fused_set_timing(moe_fused_handle_t* hd, int enable) {
  if (!hd) return MOE_ERR_INVALID_ARG;
  hd->timing = enable != 0;
  return MOE_OK;
}

int moe_fused_get_timing(moe_fused_handle_t* hd, float* ms, int32_t* launches, int max_kernels) {
  if (!hd || max_kernels < 0 || (max_kernels > 0 && (!ms || !launches))) return MOE_ERR_INVALID_ARG;
  for (int k = 0; k < max_kernels; ++k) {
    ms[k] = 0.0f;
    launches[k] = 0;
  }
  cudaError_t err = cudaSuccess;
  for (auto& r : hd->records) {
    cudaError_t e = cudaEventSynchronize(r.stop);
    float t = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
    if (e != cudaSuccess) err = e;
    if (r.kernel < max_kernels) {
      ms[r.kernel] += t;
      launches[r.kernel] += 1;
    }
    try {
      hd->pool.push_back(r.start);
    } catch (...) {
      cudaEventDestroy(r.start);
    }
    try {
      hd->pool.push_back(r.stop);
    } catch (...) {
      cudaEventDestroy(r.stop);
    }
  }
  hd->records.clear();
  if (err != cudaSuccess) return cuda_fail(err);
  return moe::kNumKernels;
}

const char* moe_fused_kernel_name(int k) {
  static const char* names[] = {"dispatch_quant", "dispatch_finish", "expand",    "gemm1_small", "gemm1_big",
                                "requant_big",    "gemm2_small",     "gemm2_big", "combine"};
  return (k >= 0 && k < moe::kNumKernels) ? names[k] : "unknown";
}

int moe_fused_dispatch_noalloc(const int32_t* expert_ids, const uint8_t* x_active_mask, int32_t bs, int32_t topk,
                               int32_t num_experts, int32_t* expert_token_nums, int32_t* expand_row, void* stream) {
  return moe::dispatch_noalloc(expert_ids, x_active_mask, bs, topk, num_experts, expert_token_nums, expand_row,
                               static_cast<cudaStream_t>(stream));
}

int moe_fused_debug_region(moe_fused_handle_t* hd, int region, size_t* offset, size_t* bytes) {
  if (!hd || !offset || !bytes) return MOE_ERR_INVALID_ARG;
  const moe::WsLayout& L = hd->L;
  const size_t offs[moe::kNumRegions] = {L.status, L.counts, L.offsets, L.row_of, L.tk_of_row, L.active, L.x_q,
                                         L.x_scale, L.xs_q, L.xs_scale, L.hbuf, L.x2, L.s2, L.y2, L.slots,
                                         L.row_token, L.shared_row, L.blk_ticket, L.tok_ticket, L.tok_expect,
                                         L.ranges, L.x1h, L.x2h, L.dcnt, L.amax2, L.bar_tags};
  if (region < 0 || region >= moe::kNumRegions) return MOE_ERR_INVALID_ARG;
  *offset = offs[region];
  *bytes = L.sizes[region];
  return MOE_OK;
}

int moe_fused_debug_gemm_acc(moe_fused_handle_t* hd, const moe_fused_args_t* args, void* workspace,
                             size_t workspace_bytes, int which, int32_t* acc, void* stream) {
  moe::FwdParams p;
  int rc = build_params(hd, args, workspace, workspace_bytes, &p);
  if (rc) return rc;
  if ((which != 1 && which != 2) || !acc) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int mode = which == 1 ? moe::kGemm1Raw : moe::kGemm2Raw;
  rc = prepare_maps(hd, p);
  if (rc) return rc;
  cudaError_t e = moe::launch_moe_gemm_small(p, mode, acc, p.num_ctas, s);
  if (e == cudaSuccess) e = moe::launch_moe_gemm_big(p, hd->maps, mode, acc, p.num_ctas, s);
  return cuda_fail(e);
}

int moe_fused_debug_wait_timeout(moe_fused_handle_t* hd, void* workspace, size_t workspace_bytes, int which,
                                 void* stream) {
  if (!hd || !workspace || (which != 0 && which != 1)) return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < hd->L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* status = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + hd->L.status);
  // status words 0..31 start clean; word 32 is the flag that nobody sets
  cudaError_t e = cudaMemsetAsync(status, 0, 64 * sizeof(int32_t), s);
  if (e == cudaSuccess) {
    debug_wait_kernel<<<1, 32, 0, s>>>(status, status + 32, which);
    e = cudaGetLastError();
  }
  return cuda_fail(e);
}

}  // extern "C"
