// Persistent grouped INT8 GEMM for the two expert contractions.
//
//   GEMM1 (FusedDeepMoE analysis §3.3, §5.2.1, epilogue §6.1):
//     acc1[r, n] = sum_c x_q[t(r), c] * W1[e][n][c]          (int8 x int8 -> int32)
//     y1 = (float(acc1) * w1_scale[e][n]) * x_scale[t(r)]
//     h[r, j] = silu(y1[r, j]) * y1[r, I + j],  silu(g) = g / (1 + exp(-g))
//   GEMM2 (§3.4, §5.2.2, epilogue §6.2):
//     acc2[r, j] = sum_i x2[r, i] * W2[e][j][i]
//     y2[r, j] = bf16((float(acc2) * w2_scale[e][j]) * s2[r])
//
// Work item = (expert slot, output tile of 128 weight rows, block of <= 64
// token rows).  For GEMM1 the 128 rows are 64 gate rows and the 64 matching up
// rows, so SwiGLU completes inside the CTA.  The weights are the M operand of
// the MMA and the few token rows the N operand ("swap AB"): decode batches
// give an expert 1..64 rows, so the weights stream once from HBM while the
// token rows stay in shared memory and L2.
//
// Pipeline (the full/empty mbarrier FIFO of the Mega-MoE analysis §4): one
// producer warp issues 1-D bulk async copies of the weight rows and the
// gathered token rows for each K chunk into a 3-stage ring; eight consumer
// warps run mma.sync m16n8k32 s8 (exact int32), four per half of the K
// steps, and meet in a fused epilogue.  The grid is persistent (one CTA per
// SM) and walks the items in order, so consecutive CTAs share weight tiles
// through L2 when an expert has several token blocks.
#include "device_prims.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BM = 128;                  // weight rows per item
constexpr int TB = kTokenBlock;          // token rows per item
constexpr int KC = 256;                  // K bytes per stage
constexpr int ROWB = KC + 16;            // smem row stride (16 B pad: conflict-free ldmatrix)
constexpr int STAGES = 3;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int EPI_STRIDE = BM + 4;       // floats per token row of the epilogue tile

constexpr int OFF_W = 0;
constexpr int OFF_T = OFF_W + STAGES * BM * ROWB;
constexpr int OFF_EPI = OFF_T + STAGES * TB * ROWB;
constexpr int OFF_BAR = OFF_EPI + TB * EPI_STRIDE * 4;
constexpr int OFF_INFO = OFF_BAR + 2 * STAGES * 8;
constexpr int OFF_ABORT = OFF_INFO + 3 * TB * 4;
constexpr int SMEM_BYTES = OFF_ABORT + 16;

static_assert(OFF_T % 16 == 0 && OFF_EPI % 16 == 0 && OFF_BAR % 8 == 0, "smem alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");

struct Item {
  int e, row0, rows, tb, jt;
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
  item.e = s_exp[s];
  item.row0 = s_row0[s];
  item.rows = s_rows[s];
  item.jt = static_cast<int>(local / T);
  item.tb = static_cast<int>(local % T);
  return item;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(FwdParams p, int32_t* raw) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  extern __shared__ __align__(128) char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + STAGES;
  float* tok_scale = reinterpret_cast<float*>(smem + OFF_INFO);
  int32_t* tok_row = reinterpret_cast<int32_t*>(smem + OFF_INFO + TB * 4);
  int32_t* tok_tok = reinterpret_cast<int32_t*>(smem + OFF_INFO + 2 * TB * 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);

  const int K = G1 ? p.h : p.I;                       // contraction length
  const int NW = G1 ? 2 * p.I : p.h;                  // weight rows per expert
  const int J = G1 ? p.I / 64 : (p.h + BM - 1) / BM;  // output tiles per token block
  const int n_kc = (K + KC - 1) / KC;
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  const long total_items = static_cast<long>(slots[SlotTable::kBigBlocks]) * J;
  const int site = (G1 ? kKGemm1 : kKGemm2) * 16;

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
          if (G1) {
            trow[q] = (item.e >= 0 ? xq : xsq) + static_cast<size_t>(row_token[r]) * p.h;
          } else {
            trow[q] = x2 + static_cast<size_t>(r) * p.I;
          }
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
  const float* row_scale = G1 ? ws_ptr<float>(p, p.L.row_scale) : ws_ptr<float>(p, p.L.s2);
  const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);

  int stage_it = 0;
  for (long it = blockIdx.x; it < total_items; it += gridDim.x) {
    const Item item = decode_item(it, J, slots, p.E);
    const int tok0 = item.tb * TB;
    const int mblk = min(TB, item.rows - tok0);
    const int nblk = (mblk + 7) >> 3;

    named_barrier_sync(1, kConsumerWarps * 32);  // previous epilogue is done with info / epi
    if (ctid < mblk) {
      const int r = item.row0 + tok0 + ctid;
      tok_row[ctid] = r;
      tok_tok[ctid] = row_token[r];
      tok_scale[ctid] = row_scale[r];
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
    named_barrier_sync(1, kConsumerWarps * 32);
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
      named_barrier_sync(1, kConsumerWarps * 32);
      if (G1) {
        const int jbase = item.jt * 64;
        for (int idx = ctid; idx < mblk * 64; idx += kConsumerWarps * 32) {
          const int tok = idx >> 6, j = idx & 63;
          const float g = epif[tok * EPI_STRIDE + j];
          const float u = epif[tok * EPI_STRIDE + 64 + j];
          const float d = __fadd_rn(1.0f, expf(-g));
          const float hv = __fmul_rn(__fdiv_rn(g, d), u);
          hbuf[static_cast<size_t>(tok_row[tok]) * p.I + jbase + j] = hv;
        }
      } else {
        const int nbase = item.jt * BM;
        const int nvalid = min(BM, p.h - nbase);
        for (int idx = ctid; idx < mblk * BM; idx += kConsumerWarps * 32) {
          const int tok = idx >> 7, n = idx & (BM - 1);
          if (n >= nvalid) continue;
          const uint16_t b = f32_to_bf16_bits(epif[tok * EPI_STRIDE + n]);
          if (item.e >= 0) y2[static_cast<size_t>(tok_row[tok]) * p.h + nbase + n] = b;
          else p.sout[static_cast<size_t>(tok_tok[tok]) * p.h + nbase + n] = b;
        }
      }
    }
    if (stop) break;
  }
}

}  // namespace

cudaError_t gemm_prepare_attributes() {
  cudaError_t e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemm1SwiGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemm2Bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<kGemm1Raw>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_kernel<kGemm2Raw>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t launch_gemm(const FwdParams& p, int mode, int32_t* raw_acc, int num_ctas, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  switch (mode) {
    case kGemm1SwiGLU: grouped_gemm_kernel<kGemm1SwiGLU><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    case kGemm2Bf16: grouped_gemm_kernel<kGemm2Bf16><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    case kGemm1Raw: grouped_gemm_kernel<kGemm1Raw><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    case kGemm2Raw: grouped_gemm_kernel<kGemm2Raw><<<num_ctas, kThreads, SMEM_BYTES, s>>>(p, raw_acc); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
