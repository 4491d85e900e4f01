// The two grouped INT8 expert GEMMs with their fused epilogues.
//
//   GEMM1 (FusedDeepMoE analysis §3.3, §5.2.1; epilogue §6.1; BlockQuant §7.2):
//     acc1[r, n] = sum_c x_q[t(r), c] * W1[e][n][c]               int8 x int8 -> int32
//     y1 = (float(acc1) * w1_scale[e][n]) * x_scale[t(r)]
//     h[r, j] = silu(y1[r, j]) * y1[r, I + j],   silu(g) = g / (1 + exp(-g))
//     then, once every column tile of a block of rows is done, the per-row
//     requant: amax = max(max|h|, 1e-4), s2 = amax * (1/127),
//     x2 = RNE((h * 127) * (1/amax)) clamped to +-127.
//   GEMM2 (§3.4, §5.2.2; epilogue §6.2; combine §4.2):
//     acc2[r, j] = sum_i x2[r, i] * W2[e][j][i]
//     y2[r, j] = act((float(acc2) * w2_scale[e][j]) * s2[r])   (act: bf16, or fp16)
//     then, once every row of a token is done, the combine:
//     output[t] = act(sum_k float(y2[row(t,k)]) * expert_scales[t, k]),
//     fp32 sum from 0, k ascending, multiply and add rounded separately.
//
// This file holds the small-expert kernel; tc_gemm.cu the big-expert one.
// Both walk the slot table that dispatch built:
//   small experts: <= kSmallRows rows (decode; in a batch of at most
//     kSmallRows tokens every expert, one that repeated ids give more rows
//     taking several slots of at most kSmallRows rows).  The weights are
//     read once from HBM and used for M <= 8 multiply-adds each, so the work
//     is a batch of matrix-vector products: dp4a on exactly M rows, fed by
//     2 KiB-per-row bulk copies (one producer warp, a 3-stage mbarrier
//     full/empty ring -- the FIFO of the Mega-MoE analysis §4), items of 32
//     weight rows, each CTA one contiguous run of items; the token rows of a
//     run of items on one expert are loaded once and stay resident.
//   big experts: blocks of up to 128 rows on the tcgen05 tensor cores
//     (tc_gemm.cu).
// The requant and the combine run in the CTA that completes the last tile of
// a row block (GEMM1) or of a token (GEMM2): each such CTA fences its
// writes and bumps a per-forward counter (reset by the dispatch kernel); the
// one that brings a counter to its total does the work.  In a forward, GEMM2
// streams behind GEMM1 in the same launch (moe_gemm_small_streamed_kernel):
// the only wait on another CTA is a GEMM2 slot's bounded wait for the requant
// of its rows, marked on the same counter.
#include "device_prims.cuh"
#include "epilogue_ops.cuh"
#include "moe_internal.h"
#include "quant_ops.cuh"

namespace moe {

namespace {

// ===================================================================== small
namespace small_path {

constexpr int BN = 32;                 // weight rows per item
constexpr int MT = kSmallRows;         // token rows per item (<= 8)
constexpr int KC = 2048;               // K bytes per stage (one bulk copy per row)
constexpr int STAGES = 3;
constexpr int kMaxK = kSmallMaxK;      // token rows of a run stay resident: MT x K bytes
constexpr int kInfoSlots = 6;          // > STAGES: per-item token info ring
constexpr int kSlotCache = 8;          // small-slot table entries a CTA can touch, per GEMM
constexpr int kRowsPerWarp = BN / kConsumerWarps;  // 4

constexpr int OFF_W = 0;                                        // STAGES x [BN][KC] weights
constexpr int OFF_T = OFF_W + STAGES * BN * KC;                 // [m][K] token rows of the current run
constexpr int OFF_Y = OFF_T + MT * kMaxK;                       // 2 x [BN][MT] fp32
constexpr int kNumBars = 2 * STAGES + 3;                        // full, empty [STAGES]; tok_full, tok_empty; ready
constexpr int OFF_BAR = OFF_Y + 2 * BN * MT * 4;
constexpr int OFF_INFO = OFF_BAR + kNumBars * 8;                // kInfoSlots x {scale, row, token}[MT]
constexpr int OFF_SLOT = OFF_INFO + kInfoSlots * 3 * MT * 4;    // 2 x kSlotCache x {e, row0, rows}: GEMM1, GEMM2
constexpr int OFF_MISC = OFF_SLOT + 2 * kSlotCache * 3 * 4;     // abort, flag, red[8], tok[MT], range[4], lid
constexpr int MISC_RANGE = 2 + kConsumerWarps + MT;             // item range {begin, end} of GEMM1, GEMM2
constexpr int MISC_LID = MISC_RANGE + 4;                        // this CTA's index in arrival order
constexpr int SMEM_BYTES = OFF_MISC + (MISC_LID + 1) * 4;
static_assert(kRowsPerWarp * MT == 32, "one reduced value per lane");
static_assert(kInfoSlots > STAGES, "info ring must outlive the stage ring");

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Butterfly reduce-scatter over the warp of the 4 * MP partial sums a lane
// holds: its warp's 4 weight rows x the first MP token slots (MP a power of
// two >= the item's token rows; the slots past them hold zeros).  The
// log2(4 MP) highest lane bits scatter the values and the remaining bits sum
// them, so lane L ends with the full sum of index L >> (5 - log2(4 MP)) =
// rr * MP + t: 4 MP - 1 + 5 - log2(4 MP) shuffles (6 for one token row, 31
// for eight), exact int32 adds.
template <int MP>
__device__ __forceinline__ int warp_reduce_scatter(const int (&acc)[kRowsPerWarp * MT], int lane) {
  constexpr int N = kRowsPerWarp * MP;
  constexpr int LG = N == 4 ? 2 : N == 8 ? 3 : N == 16 ? 4 : 5;
  int v[N];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
    for (int t = 0; t < MP; ++t) v[rr * MP + t] = acc[rr * MT + t];
#pragma unroll
  for (int lv = 0; lv < LG; ++lv) {
    const int hv = N >> (lv + 1), bit = 16 >> lv;
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int k = 0; k < hv; ++k) {
      const int send = upper ? v[k] : v[k + hv];
      const int keep = upper ? v[k + hv] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
    }
  }
#pragma unroll
  for (int bit = 16 >> LG; bit >= 1; bit >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], bit);
  return v[0];
}

// log2 of the token slots an item of m rows reduces over (1, 2, 4 or 8 slots)
__device__ __forceinline__ int slot_log2(int m) { return m <= 1 ? 0 : m <= 2 ? 1 : m <= 4 ? 2 : 3; }

__device__ __forceinline__ int reduce_item(int lgmp, const int (&acc)[kRowsPerWarp * MT], int lane) {
  switch (lgmp) {
    case 0: return warp_reduce_scatter<1>(acc, lane);
    case 1: return warp_reduce_scatter<2>(acc, lane);
    case 2: return warp_reduce_scatter<4>(acc, lane);
    default: return warp_reduce_scatter<MT>(acc, lane);
  }
}
static_assert(MT == 8, "reduce_item covers 1, 2, 4 and 8 token slots");

// One stage of dot products for a warp: kRowsPerWarp weight rows (at Ws,
// stride KC) against M token rows (at Ts, stride KC), lane-strided 16-byte
// column slices.  M is a template argument so the loop body is straight-line
// code with 4*M independent dp4a chains.
template <int M, bool FULL>
__device__ __forceinline__ void stage_dot(const char* __restrict__ Ws, const char* __restrict__ Ts, int tstride,
                                          int bytes, int lane, int (&acc)[kRowsPerWarp * MT]) {
  constexpr int kSteps = KC / 512;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int c = i * 512 + lane * 16;
    if (!FULL && c >= bytes) break;
    uint4 tv[M];
#pragma unroll
    for (int t = 0; t < M; ++t) tv[t] = *reinterpret_cast<const uint4*>(Ts + t * tstride + c);
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const uint4 wv = *reinterpret_cast<const uint4*>(Ws + rr * KC + c);
#pragma unroll
      for (int t = 0; t < M; ++t) {
        int a = acc[rr * MT + t];
        a = dp4a(wv.x, tv[t].x, a);
        a = dp4a(wv.y, tv[t].y, a);
        a = dp4a(wv.z, tv[t].z, a);
        a = dp4a(wv.w, tv[t].w, a);
        acc[rr * MT + t] = a;
      }
    }
  }
}

template <bool FULL>
__device__ __forceinline__ void stage_dot_m(int m, const char* Ws, const char* Ts, int tstride, int bytes, int lane,
                                            int (&acc)[kRowsPerWarp * MT]) {
  switch (m) {
    case 1: stage_dot<1, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    case 2: stage_dot<2, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    case 3: stage_dot<3, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    case 4: stage_dot<4, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    case 5: stage_dot<5, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    case 6: stage_dot<6, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    case 7: stage_dot<7, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
    default: stage_dot<MT, FULL>(Ws, Ts, tstride, bytes, lane, acc); break;
  }
}

struct SmallItem {
  int slot, e, row0, m, jt;
};

// Ring positions of a thread's role, carried from GEMM1 into GEMM2 when both
// run in one launch (the rings and barriers are not re-initialised between).
struct SmallState {
  int stage_it = 0, item_no = 0, run_no = 0;
  bool ready_seen = false;  // the producer has seen the one-launch kernel's `ready` barrier complete
};

// This CTA's contiguous run of items of one GEMM (consecutive tiles of one
// expert are contiguous in memory), and whether the forward has big blocks
// (then the combine kernel, not the small GEMM2, combines the tokens).
struct SmallRange {
  int it_begin, it_end;
  bool has_big;
};

// The range of CTA `cta` as the dispatch kernel left it in the workspace.
template <bool G1>
__device__ __forceinline__ SmallRange global_range(const FwdParams& p, int cta) {
  const int32_t* ranges = ws_ptr<int32_t>(p, p.L.ranges) + (G1 ? 0 : kMaxCtas + 1);
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  return SmallRange{ranges[cta], ranges[cta + 1], slots[SlotTable::kBigBlocks] > 0};
}

// This CTA's index among the small phase's CTAs, or -1 if the phase has no
// work for it: blockIdx.x, or, with the engines side by side (the tensor-core
// chain holding some SMs), the CTA's place in arrival order, so that the
// CTAs that work are the ones that got an SM first (the streamed GEMM2 waits
// on other CTAs' GEMM1 work).  Called by every thread.
__device__ __forceinline__ int small_cta(const FwdParams& p, char* smem) {
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int lid = blockIdx.x;
  if (slots[SlotTable::kSplit])
    lid = arrival_index(ws_ptr<int32_t>(p, p.L.status) + kStCtaCounter,
                        reinterpret_cast<int*>(smem + OFF_MISC) + MISC_LID);
  return lid < slots[SlotTable::kSmallCtas] ? lid : -1;
}

__device__ __forceinline__ void init_rings(char* smem) {
  if (threadIdx.x == 0) {
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    for (int s = 0; s < kNumBars; ++s)
      mbar_init(&full[s], (s < STAGES || s == 2 * STAGES || s == 2 * STAGES + 2) ? 1 : kConsumerWarps);
    *reinterpret_cast<volatile int*>(smem + OFF_MISC) = 0;  // abort flag
    fence_barrier_init();
  }
}

// The producer's exit: wait (bounded, and not cut short by an abort) until
// every bulk copy it issued has landed -- the last phase it armed on each
// weight stage and on the token-row barrier -- so that no copy still writes
// into this CTA's shared memory once the CTA ends.  Called by the whole
// producer warp after its last GEMM phase.
__device__ __forceinline__ void drain_copies(char* smem, const SmallState& ss, int32_t* status, int site) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* tok_full = full + 2 * STAGES;
  for (int s = 0; s < STAGES && s < ss.stage_it; ++s) {
    const int last_round = (ss.stage_it - 1 - s) / STAGES;
    mbar_wait_bounded(&full[s], last_round & 1, nullptr, status, site);
  }
  if (ss.run_no > 0) mbar_wait_bounded(tok_full, (ss.run_no - 1) & 1, nullptr, status, site);
}

// this CTA's slots of one GEMM's item range into its shared-memory cache, by
// threads [0, kSlotCache): `sm_exp` is the small slots' expert array, the
// first-row and row-count arrays follow it at `stride` (the workspace's slot
// table, or the one-launch kernel's own copy in shared memory).  The caller
// synchronises the block afterwards.
template <bool G1>
__device__ __forceinline__ void cache_slots(const FwdParams& p, char* smem, const SmallRange& rg,
                                            const int32_t* sm_exp, int stride) {
  const int J = G1 ? p.I / (BN / 2) : p.h / BN;
  const int slot_first = rg.it_begin / J;
  const int n_cached = rg.it_end > rg.it_begin ? (rg.it_end - 1) / J - slot_first + 1 : 0;
  int32_t* cache = reinterpret_cast<int32_t*>(smem + OFF_SLOT) + (G1 ? 0 : 3 * kSlotCache);
  if (threadIdx.x < kSlotCache && threadIdx.x < n_cached) {
    const int sl = slot_first + threadIdx.x;
    cache[3 * threadIdx.x + 0] = sm_exp[sl];
    cache[3 * threadIdx.x + 1] = sm_exp[stride + sl];
    cache[3 * threadIdx.x + 2] = sm_exp[2 * stride + sl];
  }
}

template <bool G1>
__device__ __forceinline__ void cache_slots_global(const FwdParams& p, char* smem, const SmallRange& rg) {
  const int st = SlotTable::stride(p.E);
  cache_slots<G1>(p, smem, rg, ws_ptr<int32_t>(p, p.L.slots) + SlotTable::kHeader + 4 * st, st);
}

// One GEMM over this CTA's item range `rg`.  `streamed`: GEMM2 running in
// the same launch right after GEMM1 -- each small slot's rows are read only
// once the CTA that requantised them has marked the slot's ticket (tiles + 1).
// `ready` (one-launch kernel, else null): the producer reads nothing another
// CTA writes in this launch -- the slot table in the workspace, the token
// rows, the row info, the tickets -- before this barrier's first phase has
// completed (the grid barrier behind the dispatch); its weight copies need
// only the slot cache and may start earlier.
template <int MODE>
__device__ void run(const FwdParams& p, int32_t* raw, char* smem, SmallState& ss, bool streamed, const SmallRange& rg,
                    uint64_t* ready) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tok_full = empty + STAGES;
  uint64_t* tok_empty = tok_full + 1;
  float* info_scale = reinterpret_cast<float*>(smem + OFF_INFO);                 // [slot][MT]
  int32_t* info_row = reinterpret_cast<int32_t*>(smem + OFF_INFO) + kInfoSlots * MT;
  int32_t* info_tok = info_row + kInfoSlots * MT;
  int32_t* slot_cache = reinterpret_cast<int32_t*>(smem + OFF_SLOT) + (G1 ? 0 : 3 * kSlotCache);  // [kSlotCache][3]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  int* s_flag = reinterpret_cast<int*>(smem + OFF_MISC) + 1;
  float* s_red = reinterpret_cast<float*>(smem + OFF_MISC) + 2;
  int* s_tok = reinterpret_cast<int*>(smem + OFF_MISC) + 2 + kConsumerWarps;

  const int K = G1 ? p.h : p.I;
  const int NW = G1 ? 2 * p.I : p.h;
  const int J = G1 ? p.I / (BN / 2) : p.h / BN;
  const int n_kc = (K + KC - 1) / KC;
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  const int st = SlotTable::stride(p.E);
  const int32_t* sm_exp = slots + SlotTable::kHeader + 4 * st;
  const int32_t* sm_row0 = sm_exp + st;
  const int32_t* sm_rows = sm_row0 + st;
  const bool has_big = rg.has_big;
  const long it_begin = rg.it_begin;
  const long it_end = rg.it_end;
  const int slot_first = static_cast<int>(it_begin / J);
  const int n_cached = it_end > it_begin ? static_cast<int>((it_end - 1) / J) - slot_first + 1 : 0;
  const int site = (G1 ? kKGemm1Small : kKGemm2Small) * 16;

  const bool cached = n_cached <= kSlotCache;
  // items are walked as (slot, tile) pairs advanced one by one: no 64-bit
  // division by J per item
  const int jt_first = static_cast<int>(it_begin - static_cast<long>(slot_first) * J);
  auto item_of = [&](int slot, int jt) {
    SmallItem x;
    x.slot = slot;
    x.jt = jt;
    if (cached) {
      const int c = x.slot - slot_first;
      x.e = slot_cache[3 * c];
      x.row0 = slot_cache[3 * c + 1];
      x.m = slot_cache[3 * c + 2];
    } else {
      x.e = sm_exp[x.slot];
      x.row0 = sm_row0[x.slot];
      x.m = sm_rows[x.slot];
    }
    return x;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_t = policy_evict_last();
    const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
    const float* xsc = ws_ptr<float>(p, p.L.x_scale);
    const float* xssc = p.share_uses_xq ? xsc : ws_ptr<float>(p, p.L.xs_scale);
    const float* s2 = ws_ptr<float>(p, p.L.s2);
    const int8_t* xq = ws_ptr<int8_t>(p, p.L.x_q);
    const int8_t* xsq = p.share_uses_xq ? xq : ws_ptr<int8_t>(p, p.L.xs_q);
    const int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
    const int32_t* tk_of_row = ws_ptr<int32_t>(p, p.L.tk_of_row);
    // streamed GEMM2: a slot's s2 and x2 are read only after its requant is
    // marked done (ticket = GEMM1 tiles + 1), by any CTA of this launch
    const int32_t* blk_ticket = ws_ptr<int32_t>(p, p.L.blk_ticket);
    const int g1_tiles = p.I / (BN / 2);
    auto load_info = [&](const SmallItem& x, int& tok, float& sc) -> bool {
      if (!G1 && streamed &&
          !__all_sync(0xffffffffu, spin_until_ge(blk_ticket + x.slot, g1_tiles + 1, abort_flag, status, site + 5)))
        return false;
      if (lane < x.m) {
        const int r = x.row0 + lane;
        tok = row_token[r];
        // routed x_scale is per token, or per row with per-expert smooth scales
        if (G1) sc = x.e >= 0 ? xsc[p.xq_per_row ? r : tok] : xssc[tok];
        else if (p.fold_routing && x.e >= 0) sc = __fmul_rn(s2[r], p.scales[tk_of_row[r]]);  // folded row scale
        else sc = s2[r];
      }
      return true;
    };
    // Each run's weight copies are issued first: they need only the slot
    // table.  The run's row info (token, scale) and its token rows follow,
    // for a streamed GEMM2 once the slot's rows are requantised.  The
    // consumers acquire tok_full before they compute a run's first item and
    // read its info only after that, so tok_full's release publishes that
    // item's info entry; the run's later items publish theirs through the
    // full[s] arrive of their first stage.
    auto wait_ready = [&]() -> bool {
      if (ready == nullptr || ss.ready_seen) return true;
      if (!mbar_wait_bounded(ready, 0, abort_flag, status, site + 6, false)) return false;
      ss.ready_seen = true;
      return *abort_flag == 0;
    };
    // slots beyond the cache are read from the workspace's slot table
    if (!cached && it_begin < it_end && !wait_ready()) return;
    int run_tok = 0;
    float run_scale = 0.0f;
    SmallItem nx{};
    int ps = slot_first, pj = jt_first;  // position of nx
    if (it_begin < it_end) nx = item_of(ps, pj);
    int &stage_it = ss.stage_it, &item_no = ss.item_no, &run_no = ss.run_no;
    int run_slot = -1;
    // token rows of a new run (whole K), once the consumers are done with the
    // previous run's rows
    auto load_run_rows = [&](const SmallItem& x, int tok) -> bool {
      if (run_no > 0) {
        if (!mbar_wait_bounded(tok_empty, (run_no - 1) & 1, abort_flag, status, site + 3, false)) return false;
      }
      if (lane == 0) mbar_arrive_expect_tx(tok_full, static_cast<uint32_t>(x.m * K));
      __syncwarp();
      // x2 (or, in the one-launch kernel, x_q) written by another CTA's
      // generic stores, read here by a bulk copy
      if ((!G1 && streamed) || ready != nullptr) fence_proxy_async_global();
      if (lane < x.m) {
        const int8_t* trow =
            !G1 ? x2 + static_cast<size_t>(x.row0 + lane) * p.I
            : x.e < 0 ? xsq + static_cast<size_t>(tok) * p.h
                      : xq + static_cast<size_t>(p.xq_per_row ? x.row0 + lane : tok) * p.h;
        bulk_g2s(smem + OFF_T + lane * K, trow, static_cast<uint32_t>(K), tok_full, pol_t);
      }
      run_slot = x.slot;
      ++run_no;
      return true;
    };
    for (long it = it_begin; it < it_end; ++it, ++item_no) {
      const SmallItem cur = nx;
      const int8_t* wbase = G1 ? (cur.e >= 0 ? p.w1 + static_cast<size_t>(cur.e) * NW * K : p.sw1)
                               : (cur.e >= 0 ? p.w2 + static_cast<size_t>(cur.e) * NW * K : p.sw2);
      int n;
      if (G1) n = (lane < BN / 2) ? cur.jt * (BN / 2) + lane : p.I + cur.jt * (BN / 2) + (lane - BN / 2);
      else n = cur.jt * BN + lane;
      const int8_t* wrow = wbase + static_cast<size_t>(n) * K;
      const bool new_run = cur.slot != run_slot;
      const int is = item_no % kInfoSlots;
      for (int kc = 0; kc < n_kc; ++kc, ++stage_it) {
        const int s = stage_it % STAGES;
        const int round = stage_it / STAGES;
        if (round > 0) {
          if (!mbar_wait_bounded(&empty[s], (round - 1) & 1, abort_flag, status, site + 1, false)) return;
        }
        if (kc == 0 && !new_run && lane < cur.m) {
          // published to the consumers by the release of the arrive below
          info_scale[is * MT + lane] = run_scale;
          info_row[is * MT + lane] = cur.row0 + lane;
          info_tok[is * MT + lane] = run_tok;
        }
        const int k0 = kc * KC;
        const int bytes = min(KC, K - k0);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(BN * bytes));
        __syncwarp();
        bulk_g2s(smem + OFF_W + (s * BN + lane) * KC, wrow + k0, bytes, &full[s], pol_w);
      }
      if (new_run) {
        if (!wait_ready()) return;
        if (!load_info(cur, run_tok, run_scale)) return;
        if (lane < cur.m) {
          info_scale[is * MT + lane] = run_scale;
          info_row[is * MT + lane] = cur.row0 + lane;
          info_tok[is * MT + lane] = run_tok;
        }
        __syncwarp();
        if (!load_run_rows(cur, run_tok)) return;
      }
      if (it + 1 < it_end) {
        if (++pj == J) {
          pj = 0;
          ++ps;
        }
        nx = item_of(ps, pj);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;
  float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
  int &stage_it = ss.stage_it, &item_no = ss.item_no, &run_no = ss.run_no;
  int run_items = 0, run_slot = -1;
  bool tok_ok = true;
  int cs = slot_first, cj = jt_first;  // position of the current item
  for (long it = it_begin; it < it_end; ++it, ++item_no) {
    const SmallItem cur = item_of(cs, cj);
    const bool run_end = (it + 1 == it_end) || (cj + 1 == J);
    if (++cj == J) {
      cj = 0;
      ++cs;
    }
    const int m = cur.m, jt = cur.jt;
    const int is = item_no % kInfoSlots;
    // after the reduce, lane L holds (row rr of this warp, token t) with
    // rr * mp + t = L >> sh; one owner lane per pair writes it
    const int lgmp = slot_log2(m), sh = 3 - lgmp;
    const int idx = lane >> sh;
    const int rr = idx >> lgmp, t = idx & ((1 << lgmp) - 1);
    const bool owner = (lane & ((1 << sh) - 1)) == 0 && t < m;
    const int nl = kRowsPerWarp * warp + rr;  // row inside the item
    int ng;
    if (G1) ng = (nl < BN / 2) ? jt * (BN / 2) + nl : p.I + jt * (BN / 2) + (nl - BN / 2);
    else ng = jt * BN + nl;
    // this lane's weight scale, loaded now and used after the dot products
    float ws = 0.0f;
    if (!RAW) {
      if (cur.e >= 0) ws = wscale_at(G1 ? p.w1s : p.w2s, static_cast<size_t>(cur.e) * NW + ng, p.scale_dtype);
      else ws = (G1 ? p.sw1s : p.sw2s)[ng];
    }
    if (cur.slot != run_slot) {
      tok_ok = mbar_wait_bounded(tok_full, run_no & 1, abort_flag, status, site + 4);
      run_slot = cur.slot;
      ++run_no;
    }
    float* ytile = reinterpret_cast<float*>(smem + OFF_Y) + (item_no & 1) * BN * MT;  // [BN][MT]

    int acc[kRowsPerWarp * MT];
#pragma unroll
    for (int a = 0; a < kRowsPerWarp * MT; ++a) acc[a] = 0;

    for (int kc = 0; kc < n_kc; ++kc, ++stage_it) {
      const int s = stage_it % STAGES;
      const int round = stage_it / STAGES;
      const bool ok = mbar_wait_bounded(&full[s], round & 1, abort_flag, status, site + 2);
      if (ok && tok_ok) {
        const int bytes = min(KC, K - kc * KC);
        const char* Ws = smem + OFF_W + (s * BN + kRowsPerWarp * warp) * KC;
        const char* Ts = smem + OFF_T + kc * KC;
        if (bytes == KC) stage_dot_m<true>(m, Ws, Ts, K, bytes, lane, acc);
        else stage_dot_m<false>(m, Ws, Ts, K, bytes, lane, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (run_end && lane == 0) mbar_arrive(tok_empty);  // this run's token rows are no longer read

    const int mine = reduce_item(lgmp, acc, lane);
    // the abort flag is read only right after a CTA-wide barrier, so that
    // every consumer thread leaves the loop at the same item
    bool stop = false;
    if (RAW) {
      if (owner) raw[static_cast<size_t>(info_row[is * MT + t]) * NW + ng] = mine;
      consumer_sync();
      stop = *abort_flag != 0;
    } else if (G1) {
      // gate and up rows of a column sit in different warps: meet in shared memory
      if (owner) ytile[nl * MT + t] = __fmul_rn(__fmul_rn(__int2float_rn(mine), ws), info_scale[is * MT + t]);
      consumer_sync();
      stop = *abort_flag != 0;
      if (ctid < (BN / 2) * m) {
        const int tt = ctid / (BN / 2), j = ctid % (BN / 2);
        const float g = ytile[j * MT + tt];
        const float u = ytile[(BN / 2 + j) * MT + tt];
        const float d = __fadd_rn(1.0f, expf(-g));
        hbuf[static_cast<size_t>(info_row[is * MT + tt]) * (2 * p.I) + jt * (BN / 2) + j] =
            __fmul_rn(__fdiv_rn(g, d), u);
      }
    } else {
      // GEMM2: each lane owns one (row, token) result and stores it straight
      // away: no shared-memory staging, no CTA barrier per item
      if (owner) {
        const uint16_t b =
            f32_to_act_bits(__fmul_rn(__fmul_rn(__int2float_rn(mine), ws), info_scale[is * MT + t]), p.act_fp16);
        if (cur.e >= 0) y2[static_cast<size_t>(info_row[is * MT + t]) * p.h + ng] = b;
        else p.sout[static_cast<size_t>(info_tok[is * MT + t]) * p.h + ng] = b;
      }
    }
    if (!RAW) {
      // report once per run of this CTA's items on one expert
      ++run_items;
      if (run_end) {
        __threadfence();
        consumer_sync();
        if (!G1) stop = *abort_flag != 0;
        if (G1) gemm1_item_done(p, cur.slot, J, run_items, cur.row0, m, s_flag, s_red, ctid, false);
        else if (!has_big) gemm2_item_done(p, cur.e >= 0, m, info_tok + is * MT, BN * run_items, s_tok, ctid);
        run_items = 0;
      }
    }
    if (stop) break;
  }
}


// ================================================================ one launch
// A batch of at most kSmallRows tokens (every expert small) runs its whole
// forward in one launch, the persistent single launch of the Mega-MoE FIFO
// analysis (§5.1-§5.2) at decode batch sizes.  Each CTA repeats the dispatch
// of the at most kSmallRows * kMaxTopk (t, k) pairs in its own shared memory
// (the dispatch kernel's counting-sort order, slot table and cost split), so
// its weight copies can start at once; CTA 0 writes the dispatch arrays into
// the workspace, CTAs 1 .. bs quantise one token each, every CTA clears a
// share of the tickets, and one grid barrier later the GEMM1 -> GEMM2 stream
// runs as in the streamed kernel.

// Scratch of the per-CTA dispatch: int32 words in the token-row area, which
// receives no token row before the grid barrier.
constexpr int kMaxPairs = kSmallRows * kMaxTopk;     // (t, k) pairs of a batch
constexpr int kMaxSmallSlots = kMaxPairs + 1;        // a slot per routed row, plus the shared expert's
constexpr int TD_PE = 0;                             // [kMaxPairs] expert of pair f, -1 if not routed
constexpr int TD_ROW = TD_PE + kMaxPairs;            // [kMaxPairs] rank of pair f in its expert, then its row
constexpr int TD_SCAN = TD_ROW + kMaxPairs;          // [8] warp totals of a scan
constexpr int TD_MISC = TD_SCAN + 8;                 // [8] skipped pairs, R, small slots, active tokens, shared rows
constexpr int TD_AFLAG = TD_MISC + 8;                // [kSmallRows] token t active
constexpr int TD_ACT = TD_AFLAG + kSmallRows;        // [kSmallRows] active tokens in ascending order
constexpr int TD_SROW = TD_ACT + kSmallRows;         // [kSmallRows] shared-expert row of token t, -1 if inactive
constexpr int TD_SLOT = TD_SROW + kSmallRows;        // 3 x [kMaxSmallSlots] small slots: expert, first row, rows
constexpr int TD_WP = TD_SLOT + 3 * kMaxSmallSlots;  // [kMaxSmallSlots + 1] exclusive prefix of the slot costs
constexpr int TD_CNT = TD_WP + kMaxSmallSlots + 1;   // [1024] rows per expert
constexpr int TD_OFF = TD_CNT + 1024;                // [1024] first row per expert
constexpr int TD_WORDS = TD_OFF + 1024;
static_assert(TD_WORDS * 4 <= MT * kMaxK, "dispatch scratch fits the token-row area");
static_assert(4 * kConsumers >= 1024, "four experts per consumer thread cover E <= 1024");
static_assert(kMaxSmallSlots < kConsumers, "one slot per consumer thread in the cost scan");

// Exclusive prefix sum of one int per consumer thread, and the total.  s_w:
// kConsumerWarps ints of scratch.  Both consumer barriers are inside.
__device__ __forceinline__ int consumer_excl_scan(int v, int32_t* s_w, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_w[warp] = incl;
  consumer_sync();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) {
    const int x = s_w[w];
    before += w < warp ? x : 0;
    tot += x;
  }
  *total = tot;
  consumer_sync();
  return incl - v + before;
}

// The dispatch of the batch into this CTA's shared memory, by the consumer
// threads: the rows of every pair (rank by flat index t * topk + k inside its
// expert, experts in ascending id), the small slots (an expert with c rows in
// ceil(c / small_rows) slots, then the shared expert on the active tokens),
// this CTA's item ranges of both GEMMs and its slot caches.
__device__ void local_dispatch(const FwdParams& p, char* smem) {
  int32_t* td = reinterpret_cast<int32_t*>(smem + OFF_T);
  int32_t* rng = reinterpret_cast<int32_t*>(smem + OFF_MISC) + MISC_RANGE;
  int32_t* s_exp = td + TD_SLOT;
  int32_t* s_row0 = s_exp + kMaxSmallSlots;
  int32_t* s_rows = s_row0 + kMaxSmallSlots;
  const int ctid = threadIdx.x;
  const int E = p.E, K = p.topk, bs = p.bs, P = bs * K, sr = p.small_rows;
  // 1. the expert of every pair (-1: token masked out, or id outside [0, E))
  for (int e = ctid; e < E; e += kConsumers) td[TD_CNT + e] = 0;
  bool skip = false;
  if (ctid < P) {
    const int t = ctid / K;
    const bool act = p.mask == nullptr || p.mask[t] != 0;
    const int id = p.ids[ctid];
    const bool valid = act && id >= 0 && id < E;
    skip = act && !valid;
    td[TD_PE + ctid] = valid ? id : -1;
  }
  if (ctid < bs) td[TD_AFLAG + ctid] = (p.mask == nullptr || p.mask[ctid] != 0) ? 1 : 0;
  const int skipped = named_barrier_count(1, kConsumers, skip);
  // 2. rank of each pair among its expert's pairs; rows per expert
  if (ctid < P) {
    const int e = td[TD_PE + ctid];
    if (e >= 0) {
      int rank = 0;
      for (int f = 0; f < ctid; ++f) rank += td[TD_PE + f] == e;
      td[TD_ROW + ctid] = rank;
      atomicAdd(&td[TD_CNT + e], 1);
    }
  }
  consumer_sync();
  // 3. first row and first slot of every expert: one scan of the row count
  //    and the slot count packed in 16-bit halves (both totals <= kMaxPairs)
  int c[4], n[4], mine = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * ctid + j;
    c[j] = e < E ? td[TD_CNT + e] : 0;
    n[j] = (c[j] + sr - 1) / sr;
    mine += c[j] | (n[j] << 16);
  }
  int tot;
  const int ex = consumer_excl_scan(mine, td + TD_SCAN, &tot);
  {
    int rc = ex & 0xFFFF, rn = ex >> 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * ctid + j;
      if (e < E) {
        td[TD_OFF + e] = rc;
        for (int q = 0; q < n[j]; ++q) {
          s_exp[rn + q] = e;
          s_row0[rn + q] = rc + q * sr;
          s_rows[rn + q] = min(sr, c[j] - q * sr);
        }
      }
      rc += c[j];
      rn += n[j];
    }
  }
  const int R = tot & 0xFFFF, ns_routed = tot >> 16;
  consumer_sync();
  // 4. row of every pair; the active tokens and the shared expert's slot
  if (ctid < P) {
    const int e = td[TD_PE + ctid];
    if (e >= 0) td[TD_ROW + ctid] += td[TD_OFF + e];
  }
  if (ctid == 0) {
    int S = 0;
    for (int t = 0; t < bs; ++t) {
      if (td[TD_AFLAG + t]) {
        td[TD_ACT + S] = t;
        td[TD_SROW + t] = bs * K + S;
        ++S;
      } else {
        td[TD_SROW + t] = -1;
      }
    }
    int ns = ns_routed;
    const int shared_rows = p.has_shared ? S : 0;  // S <= bs <= small_rows: one small slot
    if (shared_rows > 0) {
      s_exp[ns] = -1;
      s_row0[ns] = bs * K;
      s_rows[ns] = shared_rows;
      ++ns;
    }
    td[TD_MISC + 0] = skipped;
    td[TD_MISC + 1] = R;
    td[TD_MISC + 2] = ns;
    td[TD_MISC + 3] = S;
    td[TD_MISC + 4] = shared_rows;
  }
  consumer_sync();
  // 5. cost prefix of the small slots, this CTA's item ranges, its caches
  const int ns = td[TD_MISC + 2];
  int wtot;
  const int wex = consumer_excl_scan(ctid < ns ? 12 + s_rows[ctid] : 0, td + TD_SCAN, &wtot);
  if (ctid <= ns) td[TD_WP + ctid] = wex;
  consumer_sync();
  if (ctid < 4) {
    const int J = (ctid >> 1) == 0 ? p.I / (BN / 2) : p.h / BN;
    rng[ctid] = small_item_start(td + TD_WP, ns, J, p.num_ctas, blockIdx.x + (ctid & 1));
  }
  consumer_sync();
  cache_slots<true>(p, smem, SmallRange{rng[0], rng[1], false}, s_exp, kMaxSmallSlots);
  cache_slots<false>(p, smem, SmallRange{rng[2], rng[3], false}, s_exp, kMaxSmallSlots);
}

// CTA 0's copy of the dispatch into the workspace: what the dispatch kernel
// writes for the same batch (counts, offsets, expert_token_nums, row maps,
// active list, slot table, status words, the item ranges of every CTA, the
// per-token GEMM2 counters).  By the consumer threads.
__device__ void publish_dispatch(const FwdParams& p, const int32_t* td) {
  const int ctid = threadIdx.x;
  const int E = p.E, K = p.topk, bs = p.bs, P = bs * K, G = p.num_ctas;
  const int skipped = td[TD_MISC], R = td[TD_MISC + 1], ns = td[TD_MISC + 2], S = td[TD_MISC + 3];
  const int shared_rows = td[TD_MISC + 4];
  const int32_t* s_exp = td + TD_SLOT;
  int32_t* counts = ws_ptr<int32_t>(p, p.L.counts);
  int32_t* offsets = ws_ptr<int32_t>(p, p.L.offsets);
  int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  int32_t* tk_of_row = ws_ptr<int32_t>(p, p.L.tk_of_row);
  int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  int32_t* active = ws_ptr<int32_t>(p, p.L.active);
  int32_t* shared_row = ws_ptr<int32_t>(p, p.L.shared_row);
  int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  int32_t* ranges = ws_ptr<int32_t>(p, p.L.ranges);
  for (int e = ctid; e < E; e += kConsumers) {
    const int c = td[TD_CNT + e];
    counts[e] = c;
    offsets[e] = td[TD_OFF + e];
    p.token_nums[e] = c;
  }
  if (ctid < P) {
    const int r = td[TD_PE + ctid] >= 0 ? td[TD_ROW + ctid] : -1;
    row_of[ctid] = r;
    if (r >= 0) {
      tk_of_row[r] = ctid;
      row_token[r] = ctid / K;
    }
  }
  if (ctid < S) {
    active[ctid] = td[TD_ACT + ctid];
    if (p.has_shared) row_token[bs * K + ctid] = td[TD_ACT + ctid];
  }
  if (p.has_shared && ctid < bs) shared_row[ctid] = td[TD_SROW + ctid];
  const int st = SlotTable::stride(E);
  int32_t* b_blk = slots + SlotTable::kHeader + 3 * st;
  int32_t* g_exp = b_blk + st;
  if (ctid < ns) {
    g_exp[ctid] = s_exp[ctid];
    g_exp[st + ctid] = s_exp[kMaxSmallSlots + ctid];
    g_exp[2 * st + ctid] = s_exp[2 * kMaxSmallSlots + ctid];
  }
  if (ctid == 0) {
    offsets[E] = R;
    b_blk[0] = 0;
    slots[SlotTable::kNumBig] = 0;
    slots[SlotTable::kBigBlocks] = 0;
    slots[SlotTable::kRows] = R;
    slots[SlotTable::kSharedRows] = shared_rows;
    slots[SlotTable::kNumSmall] = ns;
    slots[SlotTable::kSmallCtas] = G;
    slots[SlotTable::kSplit] = 0;
    status[kStSkipped] = skipped;
    status[kStErrorFlags] = 0;
    status[kStErrorSite] = 0;
    status[kStRows] = R;
    status[kStSharedRows] = shared_rows;
    status[kStSlots] = ns;
  }
  for (int b = ctid; b <= G; b += kConsumers) {
    ranges[b] = small_item_start(td + TD_WP, ns, p.I / (BN / 2), G, b);
    ranges[kMaxCtas + 1 + b] = small_item_start(td + TD_WP, ns, p.h / BN, G, b);
  }
  if (ctid < bs) {
    int nvalid = 0;
    for (int k = 0; k < K; ++k) nvalid += td[TD_PE + ctid * K + k] >= 0;
    ws_ptr<int32_t>(p, p.L.tok_ticket)[ctid] = 0;
    ws_ptr<int32_t>(p, p.L.tok_expect)[ctid] = nvalid * p.h;
  }
}

// The consumers' part of the one-launch prologue after the local dispatch:
// CTA 0 publishes it, every CTA clears its share of the row-block tickets,
// CTA (1 + t) mod G quantises token t (and writes the zero rows of tokens
// that nothing combines into); then the grid barrier (run by the first
// consumer warp), and the `ready` barrier tells this CTA's producer that it
// may read what other CTAs wrote.
// false (for every consumer) if the grid barrier gave up.
__device__ bool publish_and_quant(const FwdParams& p, char* smem) {
  const int ctid = threadIdx.x;
  const int G = p.num_ctas, b = blockIdx.x;
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  float* s_red = reinterpret_cast<float*>(smem + OFF_MISC) + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  uint64_t* ready = reinterpret_cast<uint64_t*>(smem + OFF_BAR) + 2 * STAGES + 2;
  if (b == 0) publish_dispatch(p, reinterpret_cast<const int32_t*>(smem + OFF_T));
  int32_t* blk_ticket = ws_ptr<int32_t>(p, p.L.blk_ticket);
  const int nt = static_cast<int>(p.L.sizes[kRegBlkTicket] / 4), per = (nt + G - 1) / G;
  const int i_end = min(nt, (b + 1) * per);
  for (int i = b * per + ctid; i < i_end; i += kConsumers) blk_ticket[i] = 0;
  for (int t = 0; t < p.bs; ++t)
    if ((1 + t) % G == b) quant_token(p, t, s_red, 0);
  consumer_sync();
  bool ok = true;
  if (ctid < 32) {  // the first consumer warp
    ok = grid_barrier_tagged(ws_ptr<uint64_t>(p, p.L.bar_tags), p.bar_salt, G, status, kKGemm1Small * 16 + 7);
    if (ctid == 0) {
      if (!ok) *abort_flag = 1;
      mbar_arrive(ready);
    }
  }
  return !consumer_sync_or(!ok);
}

}  // namespace small_path

constexpr int SMEM_BYTES = small_path::SMEM_BYTES;
static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_small_kernel(FwdParams p, int32_t* raw) {
  extern __shared__ __align__(128) char smem[];
  // everything below reads what the preceding kernel wrote
  grid_dependency_wait();
  grid_launch_dependents();
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  const int cta = small_path::small_cta(p, smem);
  if (cta < 0) return;
  small_path::init_rings(smem);
  const small_path::SmallRange rg = small_path::global_range<G1>(p, cta);
  small_path::cache_slots_global<G1>(p, smem, rg);
  __syncthreads();
  small_path::SmallState ss;
  small_path::run<MODE>(p, raw, smem, ss, false, rg, nullptr);
  if ((threadIdx.x >> 5) == kConsumerWarps)
    small_path::drain_copies(smem, ss, ws_ptr<int32_t>(p, p.L.status), (G1 ? kKGemm1Small : kKGemm2Small) * 16 + 14);
}

// GEMM2 streamed behind GEMM1 in one persistent launch (one CTA per SM, all
// resident): each CTA runs its GEMM1 items, then its GEMM2 items through the
// same rings, so its weight stream moves on to GEMM2 as soon as its own
// GEMM1 work is issued; a GEMM2 slot waits (bounded) only for the requant of
// that slot's rows, which the CTA completing the slot's GEMM1 tiles marks on
// the slot's ticket.  GEMM1 work never waits on GEMM2, so every wait ends.
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_small_streamed_kernel(FwdParams p) {
  extern __shared__ __align__(128) char smem[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int cta = small_path::small_cta(p, smem);
  if (cta < 0) return;
  small_path::init_rings(smem);
  const small_path::SmallRange rg1 = small_path::global_range<true>(p, cta);
  const small_path::SmallRange rg2 = small_path::global_range<false>(p, cta);
  small_path::cache_slots_global<true>(p, smem, rg1);
  small_path::cache_slots_global<false>(p, smem, rg2);
  __syncthreads();
  small_path::SmallState ss;
  small_path::run<kGemm1SwiGLU>(p, nullptr, smem, ss, false, rg1, nullptr);
  small_path::run<kGemm2Bf16>(p, nullptr, smem, ss, true, rg2, nullptr);
  if ((threadIdx.x >> 5) == kConsumerWarps)
    small_path::drain_copies(smem, ss, ws_ptr<int32_t>(p, p.L.status), kKGemm1Small * 16 + 14);
}

// The whole forward of a batch of at most kSmallRows tokens in one launch
// (num_ctas CTAs, one per SM, all resident): dispatch and quant as above,
// then GEMM1 -> GEMM2 -> combine streamed as in the streamed kernel.
__global__ void __launch_bounds__(kThreads, 1) moe_decode_one_launch_kernel(FwdParams p) {
  extern __shared__ __align__(128) char smem[];
  // the previous forward may still read the workspace and write the outputs
  grid_dependency_wait();
  grid_launch_dependents();
  small_path::init_rings(smem);
  __syncthreads();
  const bool consumer = (threadIdx.x >> 5) < kConsumerWarps;
  if (consumer) small_path::local_dispatch(p, smem);
  __syncthreads();
  const int32_t* rng = reinterpret_cast<const int32_t*>(smem + small_path::OFF_MISC) + small_path::MISC_RANGE;
  const small_path::SmallRange rg1{rng[0], rng[1], false}, rg2{rng[2], rng[3], false};
  uint64_t* ready = reinterpret_cast<uint64_t*>(smem + small_path::OFF_BAR) + 2 * small_path::STAGES + 2;
  const bool go = consumer ? small_path::publish_and_quant(p, smem) : true;
  small_path::SmallState ss;
  if (go) {
    small_path::run<kGemm1SwiGLU>(p, nullptr, smem, ss, false, rg1, ready);
    small_path::run<kGemm2Bf16>(p, nullptr, smem, ss, true, rg2, ready);
  }
  if (!consumer) small_path::drain_copies(smem, ss, ws_ptr<int32_t>(p, p.L.status), kKGemm1Small * 16 + 14);
}

}  // namespace

cudaError_t moe_gemm_small_prepare_attributes() {
  const void* fns[] = {reinterpret_cast<const void*>(moe_gemm_small_kernel<kGemm1SwiGLU>),
                       reinterpret_cast<const void*>(moe_gemm_small_kernel<kGemm2Bf16>),
                       reinterpret_cast<const void*>(moe_gemm_small_kernel<kGemm1Raw>),
                       reinterpret_cast<const void*>(moe_gemm_small_kernel<kGemm2Raw>),
                       reinterpret_cast<const void*>(moe_gemm_small_streamed_kernel),
                       reinterpret_cast<const void*>(moe_decode_one_launch_kernel)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_moe_gemm_small(const FwdParams& p, int mode, int32_t* raw_acc, int num_ctas, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(num_ctas), dim3(kThreads), SMEM_BYTES, s, attr);
  switch (mode) {
    case kGemm1SwiGLU: return cudaLaunchKernelEx(&cfg, moe_gemm_small_kernel<kGemm1SwiGLU>, p, raw_acc);
    case kGemm2Bf16: return cudaLaunchKernelEx(&cfg, moe_gemm_small_kernel<kGemm2Bf16>, p, raw_acc);
    case kGemm1Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_small_kernel<kGemm1Raw>, p, raw_acc);
    case kGemm2Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_small_kernel<kGemm2Raw>, p, raw_acc);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_moe_gemm_small_streamed(const FwdParams& p, int num_ctas, cudaStream_t s, const LaunchOpts& o) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(dim3(num_ctas), dim3(kThreads), SMEM_BYTES, s, attr, o);
  return cudaLaunchKernelEx(&cfg, moe_gemm_small_streamed_kernel, p);
}

cudaError_t launch_moe_decode_one_launch(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.num_ctas), dim3(kThreads), SMEM_BYTES, s, attr);
  return cudaLaunchKernelEx(&cfg, moe_decode_one_launch_kernel, p);
}

}  // namespace moe
