// Weight-streaming grouped INT8 GEMM for experts with few rows (decode).
//
// Same contractions and epilogues as grouped_gemm.cu (FusedDeepMoE analysis
// §3.3/§6.1 for GEMM1 + SwiGLU, §3.4/§6.2 for GEMM2 + bf16 dequant), for the
// experts whose row count is at most kSmallRows.  With 1..8 rows per expert
// the block is a batch of matrix-vector products bound by HBM: every weight
// byte is read once and used for M <= 8 multiply-adds.  The int8 tensor path
// of this chip would pad M to 8 columns and run at the legacy rate, so these
// items use dp4a on exactly M rows instead.
//
// Work item = (expert, tile of 32 weight rows): GEMM1 takes 16 gate rows and
// the 16 matching up rows; GEMM2 takes 32 output rows.  Each CTA owns one
// contiguous run of items, so it streams contiguous 64 KiB weight regions.
// One producer warp feeds a 2-stage ring of 2 KiB-per-row bulk copies
// (mbarrier full/empty FIFO of the Mega-MoE analysis §4); eight consumer
// warps each own 4 weight rows, every lane a 16-byte column slice, and a warp
// reduction (exact int32 adds) finishes each dot product.
#include "device_prims.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BN = 32;                 // weight rows per item
constexpr int MT = kSmallRows;         // token rows per item (<= 8)
constexpr int KC = 2048;               // K bytes per stage (one bulk copy per row)
constexpr int STAGES = 2;
constexpr int kInfoSlots = 8;          // > STAGES: per-item token info ring
constexpr int kSlotCache = 16;         // small-slot table entries a CTA can touch
constexpr int kConsumerWarps = 8;
constexpr int kRowsPerWarp = BN / kConsumerWarps;  // 4
constexpr int kThreads = (kConsumerWarps + 1) * 32;

constexpr int OFF_W = 0;
constexpr int OFF_T = OFF_W + STAGES * BN * KC;
constexpr int OFF_Y = OFF_T + STAGES * MT * KC;                 // 2 x [BN][MT] fp32
constexpr int OFF_BAR = OFF_Y + 2 * BN * MT * 4;
constexpr int OFF_INFO = OFF_BAR + 2 * STAGES * 8;              // kInfoSlots x {scale, row, token}[MT]
constexpr int OFF_SLOT = OFF_INFO + kInfoSlots * 3 * MT * 4;    // kSlotCache x {e, row0, rows}
constexpr int OFF_ABORT = OFF_SLOT + kSlotCache * 3 * 4;
constexpr int SMEM_BYTES = OFF_ABORT + 16;
static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
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

struct SmallItem {
  int e, row0, m, jt;
};

// One stage of dot products for a warp: kRowsPerWarp weight rows (at Ws,
// stride KC) against M token rows (at Ts, stride KC), lane-strided 16-byte
// column slices.  M is a template argument so the loop body is straight-line
// code with 4*M independent dp4a chains.
template <int M, bool FULL>
__device__ __forceinline__ void stage_dot(const char* __restrict__ Ws, const char* __restrict__ Ts, int bytes,
                                          int lane, int (&acc)[kRowsPerWarp * MT]) {
  constexpr int kSteps = KC / 512;
#pragma unroll
  for (int i = 0; i < kSteps; ++i) {
    const int c = i * 512 + lane * 16;
    if (!FULL && c >= bytes) break;
    uint4 tv[M];
#pragma unroll
    for (int t = 0; t < M; ++t) tv[t] = *reinterpret_cast<const uint4*>(Ts + t * KC + c);
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
__device__ __forceinline__ void stage_dot_m(int m, const char* Ws, const char* Ts, int bytes, int lane,
                                            int (&acc)[kRowsPerWarp * MT]) {
  switch (m) {
    case 1: stage_dot<1, FULL>(Ws, Ts, bytes, lane, acc); break;
    case 2: stage_dot<2, FULL>(Ws, Ts, bytes, lane, acc); break;
    case 3: stage_dot<3, FULL>(Ws, Ts, bytes, lane, acc); break;
    case 4: stage_dot<4, FULL>(Ws, Ts, bytes, lane, acc); break;
    case 5: stage_dot<5, FULL>(Ws, Ts, bytes, lane, acc); break;
    case 6: stage_dot<6, FULL>(Ws, Ts, bytes, lane, acc); break;
    case 7: stage_dot<7, FULL>(Ws, Ts, bytes, lane, acc); break;
    default: stage_dot<MT, FULL>(Ws, Ts, bytes, lane, acc); break;
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemv_kernel(FwdParams p, int32_t* raw) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  extern __shared__ __align__(128) char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + STAGES;
  float* info_scale = reinterpret_cast<float*>(smem + OFF_INFO);                 // [slot][MT]
  int32_t* info_row = reinterpret_cast<int32_t*>(smem + OFF_INFO) + kInfoSlots * MT;
  int32_t* info_tok = info_row + kInfoSlots * MT;
  int32_t* slot_cache = reinterpret_cast<int32_t*>(smem + OFF_SLOT);            // [kSlotCache][3]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

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
  const long total = static_cast<long>(slots[SlotTable::kNumSmall]) * J;
  // contiguous run of items for this CTA: consecutive tiles of the same expert
  // are contiguous in memory
  const long it_begin = total * blockIdx.x / gridDim.x;
  const long it_end = total * (blockIdx.x + 1) / gridDim.x;
  const int slot_first = static_cast<int>(it_begin / J);
  const int n_cached = it_end > it_begin ? static_cast<int>((it_end - 1) / J) - slot_first + 1 : 0;
  const int site = (G1 ? kKGemm1Small : kKGemm2Small) * 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
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
    const int sl = static_cast<int>(it / J);
    x.jt = static_cast<int>(it % J);
    if (cached) {
      const int c = sl - slot_first;
      x.e = slot_cache[3 * c];
      x.row0 = slot_cache[3 * c + 1];
      x.m = slot_cache[3 * c + 2];
    } else {
      x.e = sm_exp[sl];
      x.row0 = sm_row0[sl];
      x.m = sm_rows[sl];
    }
    return x;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_t = policy_evict_last();
    const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
    const float* row_scale = G1 ? ws_ptr<float>(p, p.L.row_scale) : ws_ptr<float>(p, p.L.s2);
    const int8_t* xq = ws_ptr<int8_t>(p, p.L.x_q);
    const int8_t* xsq = p.share_uses_xq ? xq : ws_ptr<int8_t>(p, p.L.xs_q);
    const int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
    // token info is loaded one item ahead so its latency hides behind the copies
    int nx_tok = 0;
    float nx_scale = 0.0f;
    SmallItem nx{};
    if (it_begin < it_end) {
      nx = item_at(it_begin);
      if (lane < nx.m) {
        nx_tok = row_token[nx.row0 + lane];
        nx_scale = row_scale[nx.row0 + lane];
      }
    }
    int stage_it = 0, item_no = 0;
    for (long it = it_begin; it < it_end; ++it, ++item_no) {
      const SmallItem cur = nx;
      const int cur_tok = nx_tok;
      const float cur_scale = nx_scale;
      if (it + 1 < it_end) {
        nx = item_at(it + 1);
        if (lane < nx.m) {
          nx_tok = row_token[nx.row0 + lane];
          nx_scale = row_scale[nx.row0 + lane];
        }
      }
      const int8_t* wbase = G1 ? (cur.e >= 0 ? p.w1 + static_cast<size_t>(cur.e) * NW * K : p.sw1)
                               : (cur.e >= 0 ? p.w2 + static_cast<size_t>(cur.e) * NW * K : p.sw2);
      int n;
      if (G1) n = (lane < BN / 2) ? cur.jt * (BN / 2) + lane : p.I + cur.jt * (BN / 2) + (lane - BN / 2);
      else n = cur.jt * BN + lane;
      const int8_t* wrow = wbase + static_cast<size_t>(n) * K;
      const int8_t* trow = nullptr;
      if (lane < cur.m) {
        if (G1) trow = (cur.e >= 0 ? xq : xsq) + static_cast<size_t>(cur_tok) * p.h;
        else trow = x2 + static_cast<size_t>(cur.row0 + lane) * p.I;
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
        if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>((BN + cur.m) * bytes));
        __syncwarp();
        bulk_g2s(smem + OFF_W + (s * BN + lane) * KC, wrow + k0, bytes, &full[s], pol_w);
        if (trow) bulk_g2s(smem + OFF_T + (s * MT + lane) * KC, trow + k0, bytes, &full[s], pol_t);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;
  float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
  int stage_it = 0, item_no = 0;
  for (long it = it_begin; it < it_end; ++it, ++item_no) {
    const SmallItem cur = item_at(it);
    const int m = cur.m, jt = cur.jt;
    const int is = item_no % kInfoSlots;
    float* ytile = reinterpret_cast<float*>(smem + OFF_Y) + (item_no & 1) * BN * MT;  // [BN][MT]

    int acc[kRowsPerWarp * MT];
#pragma unroll
    for (int a = 0; a < kRowsPerWarp * MT; ++a) acc[a] = 0;

    for (int kc = 0; kc < n_kc; ++kc, ++stage_it) {
      const int s = stage_it % STAGES;
      const int round = stage_it / STAGES;
      const bool ok = mbar_wait_bounded(&full[s], round & 1, abort_flag, status, site + 2);
      if (ok) {
        const int bytes = min(KC, K - kc * KC);
        const char* Ws = smem + OFF_W + (s * BN + kRowsPerWarp * warp) * KC;
        const char* Ts = smem + OFF_T + s * MT * KC;
        if (bytes == KC) stage_dot_m<true>(m, Ws, Ts, bytes, lane, acc);
        else stage_dot_m<false>(m, Ws, Ts, bytes, lane, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

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
    named_barrier_sync(1, kConsumerWarps * 32);
    const bool stop = *abort_flag != 0;
    if (RAW) {
      // accumulators already stored
    } else if (G1) {
      if (ctid < (BN / 2) * m) {
        const int t = ctid / (BN / 2), j = ctid % (BN / 2);
        const float g = ytile[j * MT + t];
        const float u = ytile[(BN / 2 + j) * MT + t];
        const float d = __fadd_rn(1.0f, expf(-g));
        hbuf[static_cast<size_t>(info_row[is * MT + t]) * p.I + jt * (BN / 2) + j] = __fmul_rn(__fdiv_rn(g, d), u);
      }
    } else {
      if (ctid < BN * m) {
        const int t = ctid / BN, j = ctid % BN;
        const uint16_t b = f32_to_bf16_bits(ytile[j * MT + t]);
        if (cur.e >= 0) y2[static_cast<size_t>(info_row[is * MT + t]) * p.h + jt * BN + j] = b;
        else p.sout[static_cast<size_t>(info_tok[is * MT + t]) * p.h + jt * BN + j] = b;
      }
    }
    if (stop) break;
  }
}

}  // namespace

cudaError_t gemv_prepare_attributes() {
  const void* fns[] = {reinterpret_cast<const void*>(grouped_gemv_kernel<kGemm1SwiGLU>),
                       reinterpret_cast<const void*>(grouped_gemv_kernel<kGemm2Bf16>),
                       reinterpret_cast<const void*>(grouped_gemv_kernel<kGemm1Raw>),
                       reinterpret_cast<const void*>(grouped_gemv_kernel<kGemm2Raw>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gemv(const FwdParams& p, int mode, int32_t* raw_acc, int num_ctas, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  switch (mode) {
    case kGemm1SwiGLU: grouped_gemv_kernel<kGemm1SwiGLU><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    case kGemm2Bf16: grouped_gemv_kernel<kGemm2Bf16><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    case kGemm1Raw: grouped_gemv_kernel<kGemm1Raw><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    case kGemm2Raw: grouped_gemv_kernel<kGemm2Raw><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
