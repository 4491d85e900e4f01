// Dispatch (counting sort by expert) and per-token dynamic INT8 quantisation.
//
// Dispatch follows the FusedDeepMoE analysis §4.1 (local token counting into
// expert_token_nums; for small batches a (bs+1) x E table whose prefix sums
// give the expand index, §8.4).  On the GPU the table becomes a (warp,
// expert) count table: each warp of one CTA ranks a contiguous segment of the
// flat (t, k) order 32 pairs at a time (equal experts inside a step found by
// one ballot per expert-id bit), and an exclusive prefix over the warps turns
// segment ranks into group ranks, so every row's position inside its expert
// group is its rank by flat index t*topk + k -- the same stable order a
// sequential counting sort produces, with no atomics deciding the order.
//
// Both run in one launch: CTA 0 dispatches while the other CTAs quantise
// (they are independent; the GEMM kernels join them).
//
// Quant follows §4.1 / §7.3 and the W8A8 contract of the DeepSeek-V4 decode
// case study: xs = x * smooth, amax = max(max|xs|, 1e-4), m = 127 / amax,
// q = RNE(xs * m) clamped to +-127, scale = 1 / m.  Every fp32 operation is an
// explicit round-to-nearest intrinsic so no contraction can change a code.
#include <cstring>
#include <mutex>

#include "device_prims.cuh"
#include "moe_fused.h"
#include "moe_internal.h"
#include "quant_ops.cuh"

namespace moe {

namespace {

constexpr int kDispatchThreads = 1024;

// Exclusive scan of one int per thread over a 1024-thread block.
template <typename T>
__device__ T block_exclusive_scan(T v, T* total, T* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    T w = s_warp[lane];
    T wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    s_warp[lane] = wi;  // inclusive over warps
  }
  __syncthreads();
  T excl = incl - v + (warp > 0 ? s_warp[warp - 1] : T(0));
  *total = s_warp[31];
  __syncthreads();
  return excl;
}

// Lanes of the warp whose key equals this lane's, for keys in [0, 2^nbits):
// one ballot per key bit (the warp multi-split), far cheaper than match_any.
__device__ __forceinline__ unsigned warp_peers(int key, int nbits) {
  unsigned m = 0xffffffffu;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1;
    const unsigned bb = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bb : ~bb;
  }
  return m;
}

// Step 1 of the dispatch over the flat pairs [f_lo, f_hi) by one 1024-thread
// CTA: warp w ranks the contiguous segment [f_lo + w seg, f_lo + (w+1) seg)
// 32 pairs at a time (equal experts inside a step found by one ballot per
// expert-id bit; wcnt[w][e] keeps the warp's running count).  On return
// (after a CTA barrier): row_of[f] = rank of pair f inside (its warp's
// segment, its expert), or -1 for a pair that is not routed; wcnt[w][e] =
// rows of expert e in the segments of warps before w; running[e] (e < E) =
// rows of expert e in the range; [seg_lo, seg_hi) = this warp's segment.
__device__ void rank_range(const FwdParams& p, int32_t* running, int32_t* wcnt, int f_lo, int f_hi,
                           int* s_skipped, int& seg_lo, int& seg_hi) {
  const int E = p.E, K = p.topk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  const int nfr = f_hi - f_lo;
  const int seg = ((nfr + 31) / 32 + 31) & ~31;  // pairs per warp, a multiple of 32
  const int key_bits = 32 - __clz(E);            // keys 0..E (E = not routed)
  seg_lo = min(f_hi, f_lo + warp * seg);
  seg_hi = min(f_hi, f_lo + (warp + 1) * seg);
  for (int i = tid; i < 32 * E; i += kDispatchThreads) wcnt[i] = 0;
  __syncthreads();
  {
    int32_t* mycnt = wcnt + warp * E;
    for (int f0 = seg_lo; f0 < seg_hi; f0 += 32 * 8) {
      int ev[8];  // the ids of 8 steps are loaded before any is ranked
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f = f0 + 32 * u + lane;
        int e = E;
        if (f < seg_hi) {
          const int t = f / K;
          const bool act = (p.mask == nullptr) || (p.mask[t] != 0);
          const int id = p.ids[f];
          if (act) {
            if (id >= 0 && id < E) e = id;
            else atomicAdd(s_skipped, 1);
          }
        }
        ev[u] = e;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (f0 + 32 * u >= seg_hi) break;  // warp-uniform
        const int f = f0 + 32 * u + lane;
        const int e = ev[u];
        const unsigned peers = warp_peers(e, key_bits);
        const int rank_w = __popc(peers & ((1u << lane) - 1u));
        const int before = (e < E) ? mycnt[e] : 0;
        __syncwarp();
        if (f < seg_hi) row_of[f] = (e < E) ? before + rank_w : -1;
        if (e < E && rank_w == 0) mycnt[e] = before + __popc(peers);
        __syncwarp();
      }
    }
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = wcnt[w * E + tid];
      wcnt[w * E + tid] = run;  // rows of expert tid in the segments before warp w
      run += v;
    }
    running[tid] = run;
  }
  __syncthreads();
}

// Engines side by side: how many of the num_ctas CTAs the small phase (the
// dp4a launch) gets when the tensor-core chain (GEMM1, requant, GEMM2 of the
// big blocks) runs at the same time on the others.  Each side's time is its
// weight bytes over its CTAs' streaming rate, plus a fixed cost on the
// tensor-core side (the requant between its GEMMs, launch gaps); the split
// minimises the larger of the two.  Rates per CTA, measured with the engines
// side by side on the decode workloads: dp4a 43 GB/s, the tensor-core chain
// 29 GB/s, fixed cost 15 us.  Every small slot and every big token block
// streams one expert's weights (3 h I bytes).  With ts, tb the two sides'
// CTA-us and F the fixed cost, the sides meet where ts / g = F + tb / (G - g),
// the smaller root of F g^2 - (F G + ts + tb) g + ts G = 0; the better of
// the two integers around it is taken.  0 when there is no small work,
// num_ctas when there is no big work.
__device__ int small_phase_ctas(const FwdParams& p, int n_small, int big_blocks) {
  const int G = p.num_ctas;
  if (n_small == 0) return 0;
  if (big_blocks == 0 || G < 2) return G;
  constexpr float kRateSmall = 43e3f, kRateBig = 29e3f;  // bytes per us per CTA
  constexpr float kFixedBig = 15.0f;                      // us
  const float wb = 3.0f * static_cast<float>(p.h) * static_cast<float>(p.I);
  const float ts = static_cast<float>(n_small) * wb / kRateSmall;
  const float tb = static_cast<float>(big_blocks) * wb / kRateBig;
  const float g = static_cast<float>(G);
  const float b = kFixedBig * g + ts + tb;
  const float disc = fmaxf(b * b - 4.0f * kFixedBig * ts * g, 0.0f);
  const float root = (b - sqrtf(disc)) / (2.0f * kFixedBig);
  int lo = static_cast<int>(floorf(root));
  lo = lo < 1 ? 1 : lo > G - 1 ? G - 1 : lo;
  const int hi = lo + 1 < G ? lo + 1 : lo;
  auto t_of = [&](int gs) {
    return fmaxf(ts / static_cast<float>(gs), kFixedBig + tb / static_cast<float>(G - gs));
  };
  return t_of(hi) < t_of(lo) ? hi : lo;
}

// Everything after the rows are placed, by one CTA: counts, offsets and
// expert_token_nums; the active-token list and shared rows; the slot tables;
// the status words; the small-phase item ranges and the per-forward ticket
// reset.  Thread tid < E holds its expert's count c and first row off; R is
// the number of routed rows.  dsm: at least SlotTable::stride(E) ints of scratch.
__device__ void dispatch_tail(const FwdParams& p, int32_t* dsm, int c, int off, int R, int skipped) {
  __shared__ int s_warp[32];
  __shared__ unsigned long long s_warp64[32];
  const int E = p.E, K = p.topk, bs = p.bs;
  const int tid = threadIdx.x;
  int32_t* counts = ws_ptr<int32_t>(p, p.L.counts);
  int32_t* offsets = ws_ptr<int32_t>(p, p.L.offsets);
  int32_t* active = ws_ptr<int32_t>(p, p.L.active);
  int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  int32_t* shared_row = ws_ptr<int32_t>(p, p.L.shared_row);
  const int s_skipped = skipped;
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = off;
    p.token_nums[tid] = c;
  }
  if (tid == 0) offsets[E] = R;

  // 4. active tokens in ascending order (rows of the shared expert)
  int S = 0;
  for (int base = 0; base < bs; base += kDispatchThreads) {
    const int t = base + tid;
    const int a = (t < bs) && ((p.mask == nullptr) || (p.mask[t] != 0));
    int chunk_total = 0;
    const int pos = block_exclusive_scan(a, &chunk_total, s_warp);
    if (a) {
      active[S + pos] = t;
      if (p.has_shared) row_token[bs * K + S + pos] = t;
    }
    if (t < bs && p.has_shared) shared_row[t] = a ? bs * K + S + pos : -1;
    S += chunk_total;
  }

  // 5. slot tables: experts with rows in ascending id, split by row count,
  //    then the shared expert in the list its row count selects.  In a batch
  //    of at most small_rows tokens (small_only) every expert is small: one
  //    with more rows (repeated ids) takes consecutive slots of at most
  //    small_rows rows each, so the tensor-core launches have nothing to do.
  const int st = SlotTable::stride(E);
  int32_t* b_exp = slots + SlotTable::kHeader;
  int32_t* b_row0 = b_exp + st;
  int32_t* b_rows = b_row0 + st;
  int32_t* b_blk = b_rows + st;
  int32_t* s_exp = b_blk + st;
  int32_t* s_row0 = s_exp + st;
  int32_t* s_rows = s_row0 + st;
  const int n_sub = (tid < E && c > 0) ? (p.small_only ? (c + p.small_rows - 1) / p.small_rows
                                                       : (c <= p.small_rows ? 1 : 0))
                                       : 0;
  const int is_big = (tid < E) && !p.small_only && (c > p.small_rows);
  const int nblk = is_big ? (c + kTokenBlock - 1) / kTokenBlock : 0;
  // one scan of the three counters packed in 21-bit fields (each total < 2^21)
  unsigned long long packed_total = 0;
  const unsigned long long packed = block_exclusive_scan<unsigned long long>(
      static_cast<unsigned long long>(n_sub) | (static_cast<unsigned long long>(is_big) << 21) |
          (static_cast<unsigned long long>(nblk) << 42),
      &packed_total, s_warp64);
  constexpr unsigned long long kField = (1ull << 21) - 1;
  const int si = static_cast<int>(packed & kField);
  const int bi = static_cast<int>((packed >> 21) & kField);
  const int ki = static_cast<int>(packed >> 42);
  int n_small = static_cast<int>(packed_total & kField);
  int n_big = static_cast<int>((packed_total >> 21) & kField);
  int big_blk = static_cast<int>(packed_total >> 42);
  for (int j = 0; j < n_sub; ++j) {
    s_exp[si + j] = tid;
    s_row0[si + j] = off + j * p.small_rows;
    s_rows[si + j] = min(p.small_rows, c - j * p.small_rows);
  }
  if (is_big) {
    b_exp[bi] = tid;
    b_row0[bi] = off;
    b_rows[bi] = c;
    b_blk[bi] = ki;
  }
  if (tid == 0) {
    const int shared_rows = p.has_shared ? S : 0;
    if (shared_rows > 0 && shared_rows <= p.small_rows) {
      s_exp[n_small] = -1;
      s_row0[n_small] = bs * K;
      s_rows[n_small] = shared_rows;
      n_small += 1;
    } else if (shared_rows > p.small_rows) {
      b_exp[n_big] = -1;
      b_row0[n_big] = bs * K;
      b_rows[n_big] = shared_rows;
      b_blk[n_big] = big_blk;
      big_blk += (shared_rows + kTokenBlock - 1) / kTokenBlock;
      n_big += 1;
    }
    b_blk[n_big] = big_blk;
    slots[SlotTable::kNumBig] = n_big;
    slots[SlotTable::kBigBlocks] = big_blk;
    slots[SlotTable::kRows] = R;
    slots[SlotTable::kSharedRows] = shared_rows;
    slots[SlotTable::kNumSmall] = n_small;
    slots[SlotTable::kSmallCtas] = p.split_engines ? small_phase_ctas(p, n_small, big_blk) : p.num_ctas;
    slots[SlotTable::kSplit] = p.split_engines ? 1 : 0;
    // the arrival counters of the launches that follow (engines side by side)
    for (int i = 0; i < 3; ++i) status[kStCtaCounter + i] = 0;
    status[kStSkipped] = s_skipped;
    status[kStErrorFlags] = 0;
    status[kStErrorSite] = 0;
    status[kStRows] = R;
    status[kStSharedRows] = shared_rows;
    status[kStSlots] = n_small + n_big;
  }
  if (p.with_tickets) {
    // Split of the small-phase items over the GEMM CTAs, by cost: an item of
    // an expert with m rows streams the same weight bytes as any other but
    // does m dot products per weight, so it counts 12 + m (the base measured
    // best among 4 .. 128 on the decode workloads; a near-uniform split, base
    // 128, made GEMM1 20 % slower).  CTA b takes the items whose cumulative
    // cost starts in [total*b/G, total*(b+1)/G).
    __syncthreads();
    const int ns = slots[SlotTable::kNumSmall];  // written by thread 0 above
    int32_t* wp = dsm;       // exclusive prefix of (12 + m) over the small slots; [ns + 1]
    int carry = 0;
    for (int base = 0; base <= ns; base += kDispatchThreads) {
      const int i = base + tid;
      const int cost = (i < ns) ? 12 + s_rows[i] : 0;
      int tot = 0;
      const int ex = block_exclusive_scan(cost, &tot, s_warp);
      if (i <= ns) wp[i] = carry + ex;
      carry += tot;
    }
    __syncthreads();
    const int G = slots[SlotTable::kSmallCtas];  // written by thread 0 above
    int32_t* ranges = ws_ptr<int32_t>(p, p.L.ranges);
    for (int g = 0; g < 2; ++g) {
      const int J = g == 0 ? p.I / 16 : p.h / 32;   // items per small slot, GEMM1 / GEMM2
      for (int b = tid; b <= G; b += kDispatchThreads)
        ranges[g * (kMaxCtas + 1) + b] = small_item_start(wp, ns, J, G, b);
    }
    // the last-arriver counters used by the GEMM kernels start from zero
    int32_t* blk_ticket = ws_ptr<int32_t>(p, p.L.blk_ticket);
    const int nt = static_cast<int>(p.L.sizes[kRegBlkTicket] / 4);
    for (int i = tid; i < nt; i += kDispatchThreads) blk_ticket[i] = 0;
    int32_t* tok_ticket = ws_ptr<int32_t>(p, p.L.tok_ticket);
    int32_t* tok_expect = ws_ptr<int32_t>(p, p.L.tok_expect);
    for (int t = tid; t < bs; t += kDispatchThreads) {
      int nvalid = 0;
      if ((p.mask == nullptr) || (p.mask[t] != 0)) {
        for (int k = 0; k < K; ++k) {
          const int id = p.ids[t * K + k];
          nvalid += (id >= 0 && id < E);
        }
      }
      tok_ticket[t] = 0;
      tok_expect[t] = nvalid * p.h;
    }
  }
}

// Dispatch of the whole batch by one 1024-thread CTA.  dsm: dynamic shared
// memory of dispatch_smem_bytes(E).
__device__ void dispatch_block(const FwdParams& p, int32_t* dsm) {
  __shared__ int s_warp1[32];
  __shared__ int s_skipped;
  const int E = p.E, K = p.topk, bs = p.bs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* running = dsm;    // [E]: rows per expert, later the offsets
  int32_t* wcnt = dsm + E;   // [32][E]: rows per (warp, expert)
  int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  int32_t* tk_of_row = ws_ptr<int32_t>(p, p.L.tk_of_row);
  int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  if (tid == 0) s_skipped = 0;
  __syncthreads();

  // 1. ranks inside (warp segment, expert)
  int seg_lo, seg_hi;
  rank_range(p, running, wcnt, 0, bs * K, &s_skipped, seg_lo, seg_hi);

  // 2. counts -> exclusive offsets (E <= 1024: one expert per thread)
  const int c = tid < E ? running[tid] : 0;
  int R = 0;
  const int off = block_exclusive_scan(c, &R, s_warp1);
  if (tid < E) running[tid] = off;
  __syncthreads();

  // 3. final row index and its inverse: each warp walks its own segment
  //    again (its ranks were written by the same lanes), 8 steps of loads at
  //    a time before the writes.
  {
    const int32_t* mypre = wcnt + warp * E;
    for (int f0 = seg_lo; f0 < seg_hi; f0 += 32 * 8) {
      int rk[8], ev[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f = f0 + 32 * u + lane;
        rk[u] = (f < seg_hi) ? row_of[f] : -1;
        ev[u] = (f < seg_hi) ? p.ids[f] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (rk[u] >= 0) {
          const int f = f0 + 32 * u + lane;
          const int e = ev[u];
          const int r = running[e] + mypre[e] + rk[u];
          row_of[f] = r;
          tk_of_row[r] = f;
          row_token[r] = f / K;
        }
      }
    }
  }
  __syncthreads();
  dispatch_tail(p, dsm, c, off, R, s_skipped);
}

// Multi-CTA dispatch, first phase: CTA g ranks chunk g of the flat pairs
// (kDispChunk pairs) and leaves each routed pair's rank inside (chunk,
// expert) in row_of, its per-expert totals in dcnt[g][0..E) and its count of
// skipped ids in dcnt[G E + g].
__device__ void dispatch_chunk(const FwdParams& p, int32_t* dsm, int g) {
  __shared__ int s_skipped;
  const int E = p.E, nf = p.bs * p.topk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* running = dsm;
  int32_t* wcnt = dsm + E;
  int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  int32_t* dcnt = ws_ptr<int32_t>(p, p.L.dcnt);
  const int G = p.disp_chunks;
  if (tid == 0) s_skipped = 0;
  __syncthreads();
  int seg_lo, seg_hi;
  const int f_lo = g * kDispChunk, f_hi = min(nf, f_lo + kDispChunk);
  rank_range(p, running, wcnt, f_lo, f_hi, &s_skipped, seg_lo, seg_hi);
  {
    const int32_t* mypre = wcnt + warp * E;
    for (int f = seg_lo + lane; f < seg_hi; f += 32) {
      const int rk = row_of[f];
      if (rk >= 0) row_of[f] = mypre[p.ids[f]] + rk;
    }
  }
  if (tid < E) dcnt[static_cast<size_t>(g) * E + tid] = running[tid];
  if (tid == 0) dcnt[static_cast<size_t>(G) * E + g] = s_skipped;
}

__global__ void __launch_bounds__(kDispatchThreads, 1) dispatch_kernel(FwdParams p) {
  extern __shared__ int32_t dsm[];
  dispatch_block(p, dsm);
}

constexpr int kQuantGroups = kDispatchThreads / kQuantThreads;  // tokens per quant CTA in flight, 256-thread groups
constexpr int kQuantWarps = kDispatchThreads / 32;               // tokens per quant CTA in flight, one warp each
constexpr int kGroupQuantMaxBs = 1216;  // the batch one pass of 304 quant CTAs covers with 256-thread groups

// The first CTA (or the first disp_chunks CTAs, for large batches) dispatch;
// the others quantise tokens.  The two halves are independent: nothing the
// quant writes depends on the dispatch.
__global__ void __launch_bounds__(kDispatchThreads, 1) dispatch_quant_kernel(FwdParams p) {
  extern __shared__ int32_t dsm[];
  // the previous forward's GEMM2 may still read the workspace and write outputs
  grid_dependency_wait();
  grid_launch_dependents();
  const int nd = p.disp_chunks > 1 ? p.disp_chunks : 1;  // dispatch CTAs
  if (blockIdx.x < nd) {
    if (nd == 1) dispatch_block(p, dsm);
    else dispatch_chunk(p, dsm, blockIdx.x);
    return;
  }
  // quant CTAs loop over tokens (at most two CTAs per SM).  Up to
  // kGroupQuantMaxBs tokens, one token per 256-thread group at a time (4 a
  // CTA in flight, one pass over the grid, and eight warps' loads in flight
  // per token); above it, one token per warp (32 a CTA in flight): a prefill
  // batch then takes one pass over the grid instead of several.
  if (p.bs <= kGroupQuantMaxBs) {
    __shared__ float s_red[kQuantGroups][8];
    const int group = threadIdx.x / kQuantThreads;
    const int stride = (gridDim.x - nd) * kQuantGroups;
    for (int t = (blockIdx.x - nd) * kQuantGroups + group; t < p.bs; t += stride)
      quant_token(p, t, s_red[group], group);
  } else {
    const int warp = threadIdx.x >> 5;
    const int stride = (gridDim.x - nd) * kQuantWarps;
    for (int t = (blockIdx.x - nd) * kQuantWarps + warp; t < p.bs; t += stride) quant_token_warp(p, t);
  }
}

// Multi-CTA dispatch, second phase: CTA g < G places the routed pairs of
// chunk g -- expert e's rows of chunk g start at offsets[e] + (rows of e in
// the chunks before g) -- while CTA G runs the tail (counts, offsets, active
// list, slot tables, status, tickets), which reads none of the placement.
__global__ void __launch_bounds__(kDispatchThreads, 1) dispatch_finish_kernel(FwdParams p) {
  extern __shared__ int32_t dsm[];
  __shared__ int s_warp1[32];
  grid_dependency_wait();
  grid_launch_dependents();
  const int E = p.E, K = p.topk, nf = p.bs * K, G = p.disp_chunks;
  const int tid = threadIdx.x, g = blockIdx.x;
  const bool tail = g == G;
  const int32_t* dcnt = ws_ptr<int32_t>(p, p.L.dcnt);
  int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  int32_t* tk_of_row = ws_ptr<int32_t>(p, p.L.tk_of_row);
  int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  int pre = 0, tot = 0;
  if (tid < E) {
    for (int j = 0; j < G; ++j) {
      const int v = dcnt[static_cast<size_t>(j) * E + tid];
      if (j < g) pre += v;
      tot += v;
    }
  }
  int R = 0;
  const int off = block_exclusive_scan(tot, &R, s_warp1);
  if (tail) {
    // skipped ids of all chunks (G < 1024: one per thread), then the tail
    const int sk = tid < G ? dcnt[static_cast<size_t>(G) * E + tid] : 0;
    int skipped = 0;
    block_exclusive_scan(sk, &skipped, s_warp1);
    dispatch_tail(p, dsm, tot, off, R, skipped);
    return;
  }
  if (tid < E) dsm[tid] = off + pre;
  __syncthreads();
  const int f_lo = g * kDispChunk, f_hi = min(nf, f_lo + kDispChunk);
  for (int f0 = f_lo + tid; f0 < f_hi; f0 += 4 * kDispatchThreads) {
    int rk[4], ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = f0 + u * kDispatchThreads;
      rk[u] = f < f_hi ? row_of[f] : -1;
      ev[u] = f < f_hi ? p.ids[f] : 0;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (rk[u] >= 0) {
        const int f = f0 + u * kDispatchThreads;
        const int r = dsm[ev[u]] + rk[u];
        row_of[f] = r;
        tk_of_row[r] = f;
        row_token[r] = f / K;
      }
    }
  }
}

}  // namespace

// [E] + [32][E] of the ranking, and at least stride(E) + 1 ints for the
// tail's prefix of the small slots' costs
size_t dispatch_smem_bytes(int E) {
  const int a = 33 * E, b = SlotTable::stride(E) + 1;
  return sizeof(int32_t) * static_cast<size_t>(a > b ? a : b);
}

cudaError_t launch_dispatch_quant(const FwdParams& p, cudaStream_t s) {
  const int nd = p.disp_chunks > 1 ? p.disp_chunks : 1;
  const int per_cta = p.bs <= kGroupQuantMaxBs ? kQuantGroups : kQuantWarps;
  const int qblocks = (p.bs + per_cta - 1) / per_cta;
  const int blocks = nd + (qblocks < 2 * p.num_ctas ? qblocks : 2 * p.num_ctas);
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(blocks), dim3(kDispatchThreads), dispatch_smem_bytes(p.E), s, attr);
  return cudaLaunchKernelEx(&cfg, dispatch_quant_kernel, p);
}

cudaError_t launch_dispatch_finish(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0 || p.disp_chunks <= 1) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg =
      pdl_config(dim3(p.disp_chunks + 1), dim3(kDispatchThreads), dispatch_smem_bytes(p.E), s, attr);
  return cudaLaunchKernelEx(&cfg, dispatch_finish_kernel, p);
}

cudaError_t dispatch_prepare_attributes(int E) {
  cudaError_t e = cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(dispatch_smem_bytes(E)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(dispatch_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(dispatch_smem_bytes(E)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dispatch_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(dispatch_smem_bytes(E)));
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Dispatch without caller-provided scratch (moe_fused_dispatch_noalloc).
//
// Some callers cannot allocate device memory at all: plugins and custom ops
// inside a host framework that owns every device allocation, or processes
// that run on a fixed, pre-reserved device-memory budget.  For them the
// dispatch kernel above can run with its scratch (offsets, inverse index,
// active-token list, slot table, status words) in the file-scope array
// below, which every GPU that loads this library holds until the process
// exits.  Host code must not pass the array's name to a kernel: on the host
// that name is only a stand-in, so its device address is looked up with
// cudaGetSymbolAddress, once per CUDA context (the module, and with it the
// array's address, is loaded per context: after cudaDeviceReset the next
// primary context gets a fresh copy, so the cache is keyed on the context's
// process-unique id, not on the device number).
namespace moe {

constexpr size_t kNoallocScratchBytes = size_t(2) << 20;  // 2 MiB
constexpr int kNoallocMaxPairs = 65536;                   // bs * topk
constexpr int kNoallocMaxExperts = 1024;

}  // namespace moe

static __device__ __align__(256) char g_noalloc_dispatch_scratch[moe::kNoallocScratchBytes];

namespace moe {

namespace {

// Set-up results per CUDA context: the array's device address in that
// context (and the dispatch kernel's shared-memory attribute, set there).
// A small table guarded by a mutex: host threads may make their first call
// at the same time.
struct NoallocCtx {
  unsigned long long ctx_id;
  char* ptr;
};
constexpr int kNoallocCtxSlots = 64;
std::mutex g_noalloc_mu;
NoallocCtx g_noalloc_ctx[kNoallocCtxSlots];
int g_noalloc_used = 0;
int g_noalloc_next = 0;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Process-unique id of the context current on this thread (0 if none).
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_current || !get_id) {  // called under g_noalloc_mu
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    get_id = reinterpret_cast<CtxGetIdFn>(f);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  if (!ctx) {
    *id = 0;
    return true;
  }
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the static scratch in the current context; the first
// call in a context looks it up (and sets the dispatch kernel's attribute).
// Called under g_noalloc_mu.
char* noalloc_scratch_locked() {
  unsigned long long id = 0;
  if (!current_context_id(&id)) return nullptr;
  if (id == 0) {
    // no context current yet: make the current device's primary context
    // current (cudaSetDevice initialises it), then read its id
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return nullptr;
    if (!current_context_id(&id) || id == 0) return nullptr;
  }
  for (int i = 0; i < g_noalloc_used; ++i)
    if (g_noalloc_ctx[i].ctx_id == id) return g_noalloc_ctx[i].ptr;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_dispatch_scratch) != cudaSuccess || !ptr) return nullptr;
  if (dispatch_prepare_attributes(kNoallocMaxExperts) != cudaSuccess) return nullptr;
  int slot;
  if (g_noalloc_used < kNoallocCtxSlots) {
    slot = g_noalloc_used++;
  } else {
    slot = g_noalloc_next;  // more contexts than slots: replace the oldest entry
    g_noalloc_next = (g_noalloc_next + 1) % kNoallocCtxSlots;
  }
  g_noalloc_ctx[slot] = NoallocCtx{id, static_cast<char*>(ptr)};
  return static_cast<char*>(ptr);
}

// noalloc_scratch_locked under the lock; nullptr also if taking the lock
// fails (no exception leaves the C entry point that calls this)
char* noalloc_scratch() {
  try {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    return noalloc_scratch_locked();
  } catch (...) {
    return nullptr;
  }
}

// Scratch layout inside the static array for (bs, topk, E).
WsLayout noalloc_layout(int bs, int topk, int E) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t& field, size_t bytes) {
    field = off;
    off = (off + (bytes ? bytes : 1) + 255) / 256 * 256;
  };
  const size_t pairs = static_cast<size_t>(bs) * topk;
  take(L.status, 64 * sizeof(int32_t));
  take(L.counts, static_cast<size_t>(E) * 4);
  take(L.offsets, static_cast<size_t>(E + 1) * 4);
  take(L.row_of, pairs * 4);
  take(L.tk_of_row, pairs * 4);
  take(L.active, static_cast<size_t>(bs) * 4);
  take(L.row_token, pairs * 4);
  take(L.shared_row, static_cast<size_t>(bs) * 4);
  take(L.slots, static_cast<size_t>(SlotTable::words(E)) * 4);
  L.total = off;
  return L;
}

bool aligned4(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; }

}  // namespace

// Returns 0, or a negative MOE_ERR_* value (see moe_fused.h).
int dispatch_noalloc(const int32_t* expert_ids, const uint8_t* mask, int bs, int topk, int E,
                     int32_t* expert_token_nums, int32_t* expand_row, cudaStream_t s) {
  if (bs < 0 || topk < 1 || topk > 16 || E < 1 || E > kNoallocMaxExperts || topk > E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(bs) * topk > kNoallocMaxPairs) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!expert_token_nums || (bs > 0 && !expert_ids)) return MOE_ERR_INVALID_ARG;
  // the kernel reads ids and writes counts as int32 words
  if (!aligned4(expert_token_nums) || (expert_ids && !aligned4(expert_ids)) || (expand_row && !aligned4(expand_row)))
    return MOE_ERR_ALIGNMENT;
  const WsLayout L = noalloc_layout(bs, topk, E);
  if (L.total > kNoallocScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
  char* scratch = noalloc_scratch();
  if (!scratch) return MOE_ERR_CUDA;
  if (bs == 0) {
    return cudaMemsetAsync(expert_token_nums, 0, sizeof(int32_t) * E, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.bs = bs;
  p.E = E;
  p.topk = topk;
  p.has_shared = 0;
  p.with_tickets = 0;
  p.small_rows = kSmallRows;
  p.ids = expert_ids;
  p.mask = mask;
  p.token_nums = expert_token_nums;
  p.ws = scratch;
  p.L = L;
  dispatch_kernel<<<1, kDispatchThreads, dispatch_smem_bytes(E), s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (expand_row) {
    if (cudaMemcpyAsync(expand_row, p.ws + L.row_of, sizeof(int32_t) * static_cast<size_t>(bs) * topk,
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
