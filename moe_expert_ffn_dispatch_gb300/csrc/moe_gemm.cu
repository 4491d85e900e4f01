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
//     y2[r, j] = bf16((float(acc2) * w2_scale[e][j]) * s2[r])
//     then, once every row of a token is done, the combine:
//     output[t] = bf16(sum_k float(y2[row(t,k)]) * expert_scales[t, k]),
//     fp32 sum from 0, k ascending, multiply and add rounded separately.
//
// One persistent launch per GEMM runs two phases over the slot table that
// dispatch built:
//   small phase: experts with <= kSmallRows rows (decode).  The weights are
//     read once from HBM and used for M <= 8 multiply-adds each, so the work
//     is a batch of matrix-vector products: dp4a on exactly M rows, fed by
//     2 KiB-per-row bulk copies (one producer warp, a 3-stage mbarrier
//     full/empty ring -- the FIFO of the Mega-MoE analysis §4), items of 32
//     weight rows, each CTA one contiguous run of items; the token rows of a
//     run of items on one expert are loaded once and stay resident.
//   big phase: the other experts in blocks of 64 rows, mma.sync s8 m16n8k32
//     with the weights as the M operand ("swap AB"), 128 weight rows per item,
//     3-stage ring of 256-byte chunks with padded rows for ldmatrix.
// The requant and the combine run in the CTA that completes the last tile of
// a row block (GEMM1) or of a token (GEMM2): each such CTA fences its
// writes and bumps a per-forward counter (reset by the dispatch kernel); the
// one that brings a counter to its total does the work.  No CTA waits for
// another.
#include "device_prims.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr float kAmaxEps = 1e-4f;
constexpr float kInv127 = 1.0f / 127.0f;  // the fp32 nearest to 1/127

__device__ __forceinline__ void consumer_sync() { named_barrier_sync(1, kConsumers); }

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------ epilogue ops
// Requant of rows [r0, r0 + n) of h into x2 / s2, by the consumer threads.
// h was written by other CTAs in this launch: read it through L2 (ld.cg).
__device__ void requant_rows(const FwdParams& p, int r0, int n, float* s_red, int ctid) {
  const int I = p.I, n4 = I >> 2;
  const float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
  float* s2 = ws_ptr<float>(p, p.L.s2);
  const int lane = ctid & 31, warp = ctid >> 5;
  for (int i = 0; i < n; ++i) {
    const int r = r0 + i;
    const float4* hr = reinterpret_cast<const float4*>(hbuf + static_cast<size_t>(r) * I);
    float amax = 0.0f;
    for (int c = ctid; c < n4; c += kConsumers) {
      const float4 v = __ldcg(hr + c);
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_red[warp] = amax;
    consumer_sync();
    amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) amax = fmaxf(amax, s_red[w]);
    consumer_sync();
    if (amax < kAmaxEps) amax = kAmaxEps;
    const float inv = __fdiv_rn(1.0f, amax);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(x2 + static_cast<size_t>(r) * I);
    for (int c = ctid; c < n4; c += kConsumers) {
      const float4 v = __ldcg(hr + c);
      const float f[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t b = static_cast<uint8_t>(f32_to_q(__fmul_rn(__fmul_rn(f[j], 127.0f), inv)));
        packed |= b << (8 * j);
      }
      q4[c] = packed;
    }
    if (ctid == 0) s2[r] = __fmul_rn(amax, kInv127);
  }
}

// Combine of token t, by the consumer threads (y2 through L2).
__device__ void combine_token(const FwdParams& p, int t, int ctid) {
  const int h = p.h, K = p.topk, n8 = h >> 3;
  const int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  const uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
  uint4* out = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * h);
  for (int i = ctid; i < n8; i += kConsumers) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int r = row_of[t * K + k];
      if (r < 0) continue;
      const float sc = p.scales[t * K + k];
      const uint4 v = __ldcg(reinterpret_cast<const uint4*>(y2 + static_cast<size_t>(r) * h) + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float f = bf16_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu));
        acc[j] = __fadd_rn(acc[j], __fmul_rn(f, sc));
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * j])) |
             (static_cast<uint32_t>(f32_to_bf16_bits(acc[2 * j + 1])) << 16);
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// After a CTA's outputs for a row block are written (every writer fenced,
// then a consumer barrier): GEMM1 adds the tiles it finished to the block's
// counter; the CTA that completes the block requantises its rows.
// `done` tiles of the block were finished by this CTA since its last report.
__device__ void gemm1_item_done(const FwdParams& p, int blk, int tiles, int done, int r0, int n, int* s_flag,
                                float* s_red, int ctid) {
  if (ctid == 0) {
    const int old = atomicAdd(ws_ptr<int32_t>(p, p.L.blk_ticket) + blk, done);
    *s_flag = (old + done == tiles);
  }
  consumer_sync();
  if (*s_flag) {
    __threadfence();
    requant_rows(p, r0, n, s_red, ctid);
  }
}

// GEMM2: each routed row of the item adds the columns it completed to its
// token's counter; tokens that reach rows * h are combined by this CTA.
// s_tok: at least m ints of scratch.
__device__ void gemm2_item_done(const FwdParams& p, bool routed, int m, const int32_t* tok_of, int cols,
                                int* s_tok, int ctid) {
  if (ctid < m) {
    int done = -1;
    if (routed) {
      const int t = tok_of[ctid];
      const int old = atomicAdd(ws_ptr<int32_t>(p, p.L.tok_ticket) + t, cols);
      if (old + cols == ws_ptr<int32_t>(p, p.L.tok_expect)[t]) done = t;
    }
    s_tok[ctid] = done;
  }
  consumer_sync();
  for (int i = 0; i < m; ++i) {
    const int t = s_tok[i];
    if (t >= 0) {
      __threadfence();
      combine_token(p, t, ctid);
    }
  }
}

// ===================================================================== small
namespace small_path {

constexpr int BN = 32;                 // weight rows per item
constexpr int MT = kSmallRows;         // token rows per item (<= 8)
constexpr int KC = 2048;               // K bytes per stage (one bulk copy per row)
constexpr int STAGES = 3;
constexpr int kMaxK = kSmallMaxK;      // token rows of a run stay resident: MT x K bytes
constexpr int kInfoSlots = 6;          // > STAGES: per-item token info ring
constexpr int kSlotCache = 16;         // small-slot table entries a CTA can touch
constexpr int kRowsPerWarp = BN / kConsumerWarps;  // 4

constexpr int OFF_W = 0;                                        // STAGES x [BN][KC] weights
constexpr int OFF_T = OFF_W + STAGES * BN * KC;                 // [m][K] token rows of the current run
constexpr int OFF_Y = OFF_T + MT * kMaxK;                       // 2 x [BN][MT] fp32
constexpr int OFF_BAR = OFF_Y + 2 * BN * MT * 4;                // full, empty [STAGES]; tok_full, tok_empty
constexpr int OFF_INFO = OFF_BAR + (2 * STAGES + 2) * 8;        // kInfoSlots x {scale, row, token}[MT]
constexpr int OFF_SLOT = OFF_INFO + kInfoSlots * 3 * MT * 4;    // kSlotCache x {e, row0, rows}
constexpr int OFF_MISC = OFF_SLOT + kSlotCache * 3 * 4;         // abort, flag, red[8], tok[MT]
constexpr int SMEM_BYTES = OFF_MISC + (2 + kConsumerWarps + MT) * 4;
static_assert(kRowsPerWarp * MT == 32, "one reduced value per lane");
static_assert(kInfoSlots > STAGES, "info ring must outlive the stage ring");

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Butterfly reduce-scatter over the warp: on entry every lane holds 32 partial
// sums v[0..31]; on exit lane L holds the full sum of index L (31 shuffles,
// exact int32 adds).
__device__ __forceinline__ int warp_reduce_scatter32(int (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const int send = upper ? v[k] : v[k + half];
      const int keep = upper ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

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

template <int MODE>
__device__ void run(const FwdParams& p, int32_t* raw, char* smem) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tok_full = empty + STAGES;
  uint64_t* tok_empty = tok_full + 1;
  float* info_scale = reinterpret_cast<float*>(smem + OFF_INFO);                 // [slot][MT]
  int32_t* info_row = reinterpret_cast<int32_t*>(smem + OFF_INFO) + kInfoSlots * MT;
  int32_t* info_tok = info_row + kInfoSlots * MT;
  int32_t* slot_cache = reinterpret_cast<int32_t*>(smem + OFF_SLOT);            // [kSlotCache][3]
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
  // contiguous run of items for this CTA (consecutive tiles of one expert are
  // contiguous in memory), split by cost in the dispatch kernel
  const int32_t* ranges = ws_ptr<int32_t>(p, p.L.ranges) + (G1 ? 0 : kMaxCtas + 1);
  const long it_begin = ranges[blockIdx.x];
  const long it_end = ranges[blockIdx.x + 1];
  const int slot_first = static_cast<int>(it_begin / J);
  const int n_cached = it_end > it_begin ? static_cast<int>((it_end - 1) / J) - slot_first + 1 : 0;
  const int site = (G1 ? kKGemm1 : kKGemm2) * 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(tok_full, 1);
    mbar_init(tok_empty, kConsumerWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < kSlotCache && threadIdx.x < n_cached) {
    const int sl = slot_first + threadIdx.x;
    slot_cache[3 * threadIdx.x + 0] = sm_exp[sl];
    slot_cache[3 * threadIdx.x + 1] = sm_row0[sl];
    slot_cache[3 * threadIdx.x + 2] = sm_rows[sl];
  }
  __syncthreads();
  const bool cached = n_cached <= kSlotCache;
  auto item_at = [&](long it) {
    SmallItem x;
    x.slot = static_cast<int>(it / J);
    x.jt = static_cast<int>(it % J);
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
    // token info is loaded one item ahead so its latency hides behind the copies
    auto load_info = [&](const SmallItem& x, int& tok, float& sc) {
      if (lane < x.m) {
        const int r = x.row0 + lane;
        tok = row_token[r];
        sc = G1 ? (x.e >= 0 ? xsc : xssc)[tok] : s2[r];
      }
    };
    int nx_tok = 0;
    float nx_scale = 0.0f;
    SmallItem nx{};
    if (it_begin < it_end) {
      nx = item_at(it_begin);
      load_info(nx, nx_tok, nx_scale);
    }
    int stage_it = 0, item_no = 0, run_slot = -1, run_no = 0;
    for (long it = it_begin; it < it_end; ++it, ++item_no) {
      const SmallItem cur = nx;
      const int cur_tok = nx_tok;
      const float cur_scale = nx_scale;
      const int8_t* wbase = G1 ? (cur.e >= 0 ? p.w1 + static_cast<size_t>(cur.e) * NW * K : p.sw1)
                               : (cur.e >= 0 ? p.w2 + static_cast<size_t>(cur.e) * NW * K : p.sw2);
      int n;
      if (G1) n = (lane < BN / 2) ? cur.jt * (BN / 2) + lane : p.I + cur.jt * (BN / 2) + (lane - BN / 2);
      else n = cur.jt * BN + lane;
      const int8_t* wrow = wbase + static_cast<size_t>(n) * K;
      if (cur.slot != run_slot) {
        // a new run of items on one expert: load its token rows (whole K) once,
        // after the consumers are done with the previous run's rows
        if (run_no > 0) {
          if (!mbar_wait_bounded(tok_empty, (run_no - 1) & 1, abort_flag, status, site + 3, false)) return;
        }
        if (lane == 0) mbar_arrive_expect_tx(tok_full, static_cast<uint32_t>(cur.m * K));
        __syncwarp();
        if (lane < cur.m) {
          const int8_t* trow = G1 ? (cur.e >= 0 ? xq : xsq) + static_cast<size_t>(cur_tok) * p.h
                                  : x2 + static_cast<size_t>(cur.row0 + lane) * p.I;
          bulk_g2s(smem + OFF_T + lane * K, trow, static_cast<uint32_t>(K), tok_full, pol_t);
        }
        run_slot = cur.slot;
        ++run_no;
      }
      for (int kc = 0; kc < n_kc; ++kc, ++stage_it) {
        const int s = stage_it % STAGES;
        const int round = stage_it / STAGES;
        if (round > 0) {
          if (!mbar_wait_bounded(&empty[s], (round - 1) & 1, abort_flag, status, site + 1, false)) return;
        }
        if (kc == 0 && lane < cur.m) {
          // published to the consumers by the release of the arrive below
          const int is = item_no % kInfoSlots;
          info_scale[is * MT + lane] = cur_scale;
          info_row[is * MT + lane] = cur.row0 + lane;
          info_tok[is * MT + lane] = cur_tok;
        }
        const int k0 = kc * KC;
        const int bytes = min(KC, K - k0);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(BN * bytes));
        __syncwarp();
        bulk_g2s(smem + OFF_W + (s * BN + lane) * KC, wrow + k0, bytes, &full[s], pol_w);
      }
      // next item's token info: its dependent loads run while this item's copies fly
      if (it + 1 < it_end) {
        nx = item_at(it + 1);
        load_info(nx, nx_tok, nx_scale);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;
  float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
  int stage_it = 0, item_no = 0, run_items = 0, run_slot = -1, run_no = 0;
  bool tok_ok = true;
  for (long it = it_begin; it < it_end; ++it, ++item_no) {
    const SmallItem cur = item_at(it);
    const int m = cur.m, jt = cur.jt;
    const int is = item_no % kInfoSlots;
    const bool run_end = (it + 1 == it_end) || ((it + 1) / J != cur.slot);
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

    // lane (rr * MT + t) receives the dot product of row rr of this warp with token t
    const int mine = warp_reduce_scatter32(acc, lane);
    {
      const int rr = lane / MT, t = lane % MT;
      const int nl = kRowsPerWarp * warp + rr;  // row inside the item
      int ng;
      if (G1) ng = (nl < BN / 2) ? jt * (BN / 2) + nl : p.I + jt * (BN / 2) + (nl - BN / 2);
      else ng = jt * BN + nl;
      if (RAW) {
        if (t < m) raw[static_cast<size_t>(info_row[is * MT + t]) * NW + ng] = mine;
      } else {
        const float* wsc = G1 ? (cur.e >= 0 ? p.w1s + static_cast<size_t>(cur.e) * NW : p.sw1s)
                              : (cur.e >= 0 ? p.w2s + static_cast<size_t>(cur.e) * NW : p.sw2s);
        float y = 0.0f;
        if (t < m) y = __fmul_rn(__fmul_rn(__int2float_rn(mine), wsc[ng]), info_scale[is * MT + t]);
        ytile[nl * MT + t] = y;
      }
    }
    consumer_sync();
    const bool stop = *abort_flag != 0;
    if (!RAW) {
      if (G1) {
        if (ctid < (BN / 2) * m) {
          const int t = ctid / (BN / 2), j = ctid % (BN / 2);
          const float g = ytile[j * MT + t];
          const float u = ytile[(BN / 2 + j) * MT + t];
          const float d = __fadd_rn(1.0f, expf(-g));
          hbuf[static_cast<size_t>(info_row[is * MT + t]) * p.I + jt * (BN / 2) + j] =
              __fmul_rn(__fdiv_rn(g, d), u);
        }
      } else {
        if (ctid < BN * m) {
          const int t = ctid / BN, j = ctid % BN;
          const uint16_t b = f32_to_bf16_bits(ytile[j * MT + t]);
          if (cur.e >= 0) y2[static_cast<size_t>(info_row[is * MT + t]) * p.h + jt * BN + j] = b;
          else p.sout[static_cast<size_t>(info_tok[is * MT + t]) * p.h + jt * BN + j] = b;
        }
      }
      // report once per run of this CTA's items on one expert
      ++run_items;
      if (run_end) {
        __threadfence();
        consumer_sync();
        if (G1) gemm1_item_done(p, cur.slot, J, run_items, cur.row0, m, s_flag, s_red, ctid);
        else gemm2_item_done(p, cur.e >= 0, m, info_tok + is * MT, BN * run_items, s_tok, ctid);
        run_items = 0;
      }
    }
    if (stop) break;
  }
}

__device__ void inval_barriers(char* smem) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  for (int s = 0; s < 2 * STAGES + 2; ++s) mbar_inval(full + s);
}

}  // namespace small_path

// ======================================================================= big
namespace big_path {

constexpr int BM = 128;                  // weight rows per item
constexpr int TB = kTokenBlock;          // token rows per item
constexpr int KC = 256;                  // K bytes per stage
constexpr int ROWB = KC + 16;            // smem row stride (16 B pad: conflict-free ldmatrix)
constexpr int STAGES = 3;
constexpr int EPI_STRIDE = BM + 4;       // floats per token row of the epilogue tile

constexpr int OFF_W = 0;
constexpr int OFF_T = OFF_W + STAGES * BM * ROWB;
constexpr int OFF_EPI = OFF_T + STAGES * TB * ROWB;
constexpr int OFF_BAR = OFF_EPI + TB * EPI_STRIDE * 4;
constexpr int OFF_INFO = OFF_BAR + 2 * STAGES * 8;
constexpr int OFF_MISC = OFF_INFO + 3 * TB * 4;                // abort, flag, red[8], tok[256]
constexpr int SMEM_BYTES = OFF_MISC + (2 + kConsumerWarps + kConsumers) * 4;
static_assert(OFF_T % 16 == 0 && OFF_EPI % 16 == 0 && OFF_BAR % 8 == 0, "smem alignment");

struct Item {
  int slot, e, row0, rows, tb, jt;
};

__device__ __forceinline__ Item decode_item(long it, int J, const int32_t* slots, int E) {
  const int st = SlotTable::stride(E);
  const int32_t* s_exp = slots + SlotTable::kHeader;
  const int32_t* s_row0 = s_exp + st;
  const int32_t* s_rows = s_row0 + st;
  const int32_t* s_blk = s_rows + st;
  const int n_slots = slots[SlotTable::kNumBig];
  // last slot s with J * blk[s] <= it
  int lo = 0, hi = n_slots - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long>(J) * s_blk[mid] <= it) lo = mid;
    else hi = mid - 1;
  }
  const int s = lo;
  const long local = it - static_cast<long>(J) * s_blk[s];
  const int T = s_blk[s + 1] - s_blk[s];
  Item item;
  item.slot = s;
  item.e = s_exp[s];
  item.row0 = s_row0[s];
  item.rows = s_rows[s];
  item.jt = static_cast<int>(local / T);
  item.tb = static_cast<int>(local % T);
  return item;
}

template <int MODE>
__device__ void run(const FwdParams& p, int32_t* raw, char* smem) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + STAGES;
  float* tok_scale = reinterpret_cast<float*>(smem + OFF_INFO);
  int32_t* tok_row = reinterpret_cast<int32_t*>(smem + OFF_INFO + TB * 4);
  int32_t* tok_tok = reinterpret_cast<int32_t*>(smem + OFF_INFO + 2 * TB * 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC);
  int* s_flag = reinterpret_cast<int*>(smem + OFF_MISC) + 1;
  float* s_red = reinterpret_cast<float*>(smem + OFF_MISC) + 2;
  int* s_tok = reinterpret_cast<int*>(smem + OFF_MISC) + 2 + kConsumerWarps;

  const int K = G1 ? p.h : p.I;                       // contraction length
  const int NW = G1 ? 2 * p.I : p.h;                  // weight rows per expert
  const int J = G1 ? p.I / 64 : (p.h + BM - 1) / BM;  // output tiles per token block
  const int n_kc = (K + KC - 1) / KC;
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  const int32_t* s_blk = slots + SlotTable::kHeader + 3 * SlotTable::stride(p.E);
  const long total_items = static_cast<long>(slots[SlotTable::kBigBlocks]) * J;
  const int site = (G1 ? kKGemm1 : kKGemm2) * 16 + 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_t = policy_evict_last();
    const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
    const int8_t* xq = ws_ptr<int8_t>(p, p.L.x_q);
    const int8_t* xsq = p.share_uses_xq ? xq : ws_ptr<int8_t>(p, p.L.xs_q);
    const int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
    int stage_it = 0;
    for (long it = blockIdx.x; it < total_items; it += gridDim.x) {
      const Item item = decode_item(it, J, slots, p.E);
      const int tok0 = item.tb * TB;
      const int mblk = min(TB, item.rows - tok0);
      const int8_t* wbase = G1 ? (item.e >= 0 ? p.w1 + static_cast<size_t>(item.e) * NW * K : p.sw1)
                               : (item.e >= 0 ? p.w2 + static_cast<size_t>(item.e) * NW * K : p.sw2);
      const int rows_valid = G1 ? BM : min(BM, p.h - item.jt * BM);
      const int8_t* wrow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = lane + 32 * q;
        int n;
        if (G1) n = (i < 64) ? item.jt * 64 + i : p.I + item.jt * 64 + (i - 64);
        else n = item.jt * BM + i;
        wrow[q] = (i < rows_valid) ? wbase + static_cast<size_t>(n) * K : nullptr;
      }
      const int8_t* trow[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int i = lane + 32 * q;
        trow[q] = nullptr;
        if (i < mblk) {
          const int r = item.row0 + tok0 + i;
          if (G1) trow[q] = (item.e >= 0 ? xq : xsq) + static_cast<size_t>(row_token[r]) * p.h;
          else trow[q] = x2 + static_cast<size_t>(r) * p.I;
        }
      }
      for (int kc = 0; kc < n_kc; ++kc, ++stage_it) {
        const int s = stage_it % STAGES;
        const int round = stage_it / STAGES;
        if (round > 0) {
          if (!mbar_wait_bounded(&empty[s], (round - 1) & 1, abort_flag, status, site + 1, false)) return;
        }
        const int k0 = kc * KC;
        const int bytes = min(KC, K - k0);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>((rows_valid + mblk) * bytes));
        __syncwarp();
        char* wdst = smem + OFF_W + s * BM * ROWB;
        char* tdst = smem + OFF_T + s * TB * ROWB;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (wrow[q]) bulk_g2s(wdst + (lane + 32 * q) * ROWB, wrow[q] + k0, bytes, &full[s], pol_w);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (trow[q]) bulk_g2s(tdst + (lane + 32 * q) * ROWB, trow[q] + k0, bytes, &full[s], pol_t);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;       // 0..255
  const int mg = warp & 3;            // rows 32*mg .. 32*mg+31
  const int kh = warp >> 2;           // K-step parity handled by this warp
  const int gid = lane >> 2, tig = lane & 3;
  int32_t* epii = reinterpret_cast<int32_t*>(smem + OFF_EPI);
  float* epif = reinterpret_cast<float*>(smem + OFF_EPI);
  const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  const float* xsc = ws_ptr<float>(p, p.L.x_scale);
  const float* xssc = p.share_uses_xq ? xsc : ws_ptr<float>(p, p.L.xs_scale);
  const float* s2 = ws_ptr<float>(p, p.L.s2);
  float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);

  int stage_it = 0;
  for (long it = blockIdx.x; it < total_items; it += gridDim.x) {
    const Item item = decode_item(it, J, slots, p.E);
    const int tok0 = item.tb * TB;
    const int mblk = min(TB, item.rows - tok0);
    const int nblk = (mblk + 7) >> 3;

    consumer_sync();  // previous epilogue is done with info / epi
    if (ctid < mblk) {
      const int r = item.row0 + tok0 + ctid;
      const int t = row_token[r];
      tok_row[ctid] = r;
      tok_tok[ctid] = t;
      tok_scale[ctid] = G1 ? (item.e >= 0 ? xsc : xssc)[t] : s2[r];
    }

    int32_t acc[2][8][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][b][c] = 0;

    for (int kc = 0; kc < n_kc; ++kc, ++stage_it) {
      const int s = stage_it % STAGES;
      const int round = stage_it / STAGES;
      const bool ok = mbar_wait_bounded(&full[s], round & 1, abort_flag, status, site + 2);
      if (ok) {
        const int bytes = min(KC, K - kc * KC);
        const int nks = bytes >> 5;
        const char* Ws = smem + OFF_W + s * BM * ROWB;
        const char* Ts = smem + OFF_T + s * TB * ROWB;
        for (int ks = kh; ks < nks; ks += 2) {
          uint32_t a[2][4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int row = 32 * mg + 16 * mt + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int col = ks * 32 + (lane >> 4) * 16;
            ldmatrix_x4(a[mt][0], a[mt][1], a[mt][2], a[mt][3], Ws + row * ROWB + col);
          }
#pragma unroll
          for (int nbp = 0; nbp < 8; nbp += 2) {
            if (nbp < nblk) {
              const int tok = nbp * 8 + (lane & 7) + (lane >> 4) * 8;
              const int col = ks * 32 + ((lane >> 3) & 1) * 16;
              uint32_t b0, b1, b2, b3;
              ldmatrix_x4(b0, b1, b2, b3, Ts + tok * ROWB + col);
#pragma unroll
              for (int mt = 0; mt < 2; ++mt) {
                mma_s8_16832(acc[mt][nbp], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b0, b1);
                if (nbp + 1 < nblk)
                  mma_s8_16832(acc[mt][nbp + 1], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b2, b3);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- epilogue: combine the two K halves in smem, dequantise, activate
    if (kh == 1) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
          if (nb < nblk)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int n = 32 * mg + 16 * mt + gid + (c >> 1) * 8;
              const int tok = 8 * nb + 2 * tig + (c & 1);
              epii[tok * EPI_STRIDE + n] = acc[mt][nb][c];
            }
    }
    consumer_sync();
    // every consumer warp has left its K loop: the abort flag is final for this item
    const bool stop = *abort_flag != 0;
    if (kh == 0) {
      const float* wsc;
      if (G1) wsc = item.e >= 0 ? p.w1s + static_cast<size_t>(item.e) * NW : p.sw1s;
      else wsc = item.e >= 0 ? p.w2s + static_cast<size_t>(item.e) * NW : p.sw2s;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
          if (nb < nblk)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int n = 32 * mg + 16 * mt + gid + (c >> 1) * 8;
              const int tok = 8 * nb + 2 * tig + (c & 1);
              const int v = acc[mt][nb][c] + epii[tok * EPI_STRIDE + n];
              int ng;
              if (G1) ng = (n < 64) ? item.jt * 64 + n : p.I + item.jt * 64 + (n - 64);
              else ng = item.jt * BM + n;
              if (RAW) {
                if (tok < mblk && ng < NW) raw[static_cast<size_t>(tok_row[tok]) * NW + ng] = v;
              } else {
                float y = 0.0f;
                if (tok < mblk && ng < NW) y = __fmul_rn(__fmul_rn(__int2float_rn(v), wsc[ng]), tok_scale[tok]);
                epif[tok * EPI_STRIDE + n] = y;
              }
            }
    }
    if (!RAW) {
      consumer_sync();
      if (G1) {
        const int jbase = item.jt * 64;
        for (int idx = ctid; idx < mblk * 64; idx += kConsumers) {
          const int tok = idx >> 6, j = idx & 63;
          const float g = epif[tok * EPI_STRIDE + j];
          const float u = epif[tok * EPI_STRIDE + 64 + j];
          const float d = __fadd_rn(1.0f, expf(-g));
          const float hv = __fmul_rn(__fdiv_rn(g, d), u);
          hbuf[static_cast<size_t>(tok_row[tok]) * p.I + jbase + j] = hv;
        }
        __threadfence();
        consumer_sync();
        gemm1_item_done(p, SlotTable::stride(p.E) + s_blk[item.slot] + item.tb, J, 1, item.row0 + tok0, mblk,
                        s_flag, s_red, ctid);
      } else {
        const int nbase = item.jt * BM;
        const int nvalid = min(BM, p.h - nbase);
        for (int idx = ctid; idx < mblk * BM; idx += kConsumers) {
          const int tok = idx >> 7, n = idx & (BM - 1);
          if (n >= nvalid) continue;
          const uint16_t b = f32_to_bf16_bits(epif[tok * EPI_STRIDE + n]);
          if (item.e >= 0) y2[static_cast<size_t>(tok_row[tok]) * p.h + nbase + n] = b;
          else p.sout[static_cast<size_t>(tok_tok[tok]) * p.h + nbase + n] = b;
        }
        __threadfence();
        consumer_sync();
        gemm2_item_done(p, item.e >= 0, mblk, tok_tok, nvalid, s_tok, ctid);
      }
    }
    if (stop) break;
  }
}

}  // namespace big_path

constexpr int SMEM_BYTES = small_path::SMEM_BYTES > big_path::SMEM_BYTES ? small_path::SMEM_BYTES
                                                                          : big_path::SMEM_BYTES;
static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");

// Small phase, then big phase, in one persistent launch.  The phases reuse
// the same shared memory: every copy of the small phase has landed before
// its consumers finish, and its barriers are invalidated before reuse.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_kernel(FwdParams p, int32_t* raw) {
  extern __shared__ __align__(128) char smem[];
  // everything below reads what the preceding kernel wrote
  grid_dependency_wait();
  grid_launch_dependents();
  small_path::run<MODE>(p, raw, smem);
  __syncthreads();
  if (threadIdx.x == 0) small_path::inval_barriers(smem);
  __syncthreads();
  big_path::run<MODE>(p, raw, smem);
}

}  // namespace

cudaError_t moe_gemm_prepare_attributes() {
  const void* fns[] = {reinterpret_cast<const void*>(moe_gemm_kernel<kGemm1SwiGLU>),
                       reinterpret_cast<const void*>(moe_gemm_kernel<kGemm2Bf16>),
                       reinterpret_cast<const void*>(moe_gemm_kernel<kGemm1Raw>),
                       reinterpret_cast<const void*>(moe_gemm_kernel<kGemm2Raw>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_moe_gemm(const FwdParams& p, int mode, int32_t* raw_acc, int num_ctas, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(num_ctas), dim3(kThreads), SMEM_BYTES, s, attr);
  switch (mode) {
    case kGemm1SwiGLU: return cudaLaunchKernelEx(&cfg, moe_gemm_kernel<kGemm1SwiGLU>, p, raw_acc);
    case kGemm2Bf16: return cudaLaunchKernelEx(&cfg, moe_gemm_kernel<kGemm2Bf16>, p, raw_acc);
    case kGemm1Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_kernel<kGemm1Raw>, p, raw_acc);
    case kGemm2Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_kernel<kGemm2Raw>, p, raw_acc);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
