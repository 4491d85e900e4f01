// Big-expert GEMMs on the tcgen05 tensor cores, exact in int32.
//
// Same contractions and epilogues as the small-expert kernel (FusedDeepMoE
// analysis §3.3/§6.1 GEMM1 + SwiGLU, §7.2 requant, §3.4/§6.2 GEMM2 + bf16
// dequant, §4.2 combine), for experts whose row blocks are large enough for
// the tensor cores to pay.
//
// There is no integer MMA kind on this chip's fifth-generation tensor cores,
// so the int8 codes run as f16 values (every integer in [-128, 127] is exact
// in f16) with fp32 accumulation in tensor memory.  A product of two codes is
// at most 128 * 127 in magnitude, so any 1024 consecutive K terms sum to less
// than 2^24 and every partial sum is an exactly representable integer: each
// accumulator covers 1024 K at most and is then drained into int32 registers,
// which keeps the result bit-identical to an int32 GEMM.
//
// Tile: 128 weight rows (GEMM1: 64 gate + the 64 matching up rows) x up to
// 128 token rows of one expert x all of K, weights as the MMA's M operand.
// The requant of big blocks and the combine of forwards with big blocks run
// as separate parallel kernels (below): done by the CTA that finishes a block
// last, they would serialise 128-row blocks and 128-token tiles on a few SMs.
// Warp roles (one CTA per SM, persistent):
//   warp 0      TMA of the int8 weight boxes into an 8-deep staging ring
//   warp 2      TMA of the f16 token boxes (128-byte swizzle) into a 3-deep ring
//   warps 4..7  convert int8 weight stages to f16 tiles in the 128-byte swizzle
//   warp 1      one thread issues tcgen05.mma (M128, N = rows rounded to 16,
//               K16) into two tensor-memory accumulators, alternating per
//               1024 of K, and commits to the ring and accumulator barriers
//   warps 8..15 drain accumulators (tcgen05.ld) into int32, then the fused
//               epilogue; two warps per tensor-memory lane quadrant
// All rings are mbarrier full/empty pairs (the FIFO of the Mega-MoE
// analysis §4); every wait is bounded.
#include <cuda_fp16.h>

#include "device_prims.cuh"
#include "epilogue_ops.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int BM = 128;               // weight rows per tile (MMA M)
constexpr int TB = kTokenBlock;       // token rows per tile (MMA N <= 128)
constexpr int KB = 64;                // K elements per stage: one 128-byte f16 row
constexpr int CHUNK_KB = 16;          // stages per exact accumulation chunk (1024 of K)
constexpr int S8 = 8;                 // int8 weight staging ring
constexpr int S16 = 3;                // f16 operand ring
constexpr int kTmemCols = 2 * TB;     // two accumulators

constexpr int kBigWarps = 16;
constexpr int kBigThreads = kBigWarps * 32;
constexpr int kWarpA = 0, kWarpMma = 1, kWarpB = 2;
constexpr int kConvWarp0 = 4, kConvWarps = 4;
constexpr int kEpiWarp0 = 8;          // epilogue warps 8..15 = the 256 "consumer" threads
constexpr int XSTRIDE = TB + 1;       // floats per row of the exchange tile (bank spread)

constexpr int A8_BYTES = BM * KB;                    // 8 KB
constexpr int F16_TILE = 128 * KB * 2;               // 16 KB
constexpr int OFF_A16 = 0;                           // S16 x [128][64] f16, swizzled
constexpr int OFF_B16 = OFF_A16 + S16 * F16_TILE;    // S16 x [128][64] f16, swizzled (TMA)
constexpr int OFF_A8 = OFF_B16 + S16 * F16_TILE;     // S8 x [128][64] int8
constexpr int OFF_X = OFF_A8 + S8 * A8_BYTES;        // [64][XSTRIDE] fp32 (GEMM1 up half)
constexpr int OFF_BAR = OFF_X + 64 * XSTRIDE * 4;
constexpr int NBAR = 2 * S8 + 3 * S16 + 4;
constexpr int OFF_INFO = OFF_BAR + NBAR * 8;         // tok_scale, tok_row, tok_tok [TB]
constexpr int OFF_MISC = OFF_INFO + 3 * TB * 4;      // tmem slot, abort flag
constexpr int SMEM_BYTES = OFF_MISC + (3 + kConsumerWarps + TB) * 4;
static_assert(OFF_B16 % 1024 == 0 && OFF_A8 % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");

struct BigItem {
  int slot, e, row0, rows, tb, jt;
};

__device__ __forceinline__ BigItem decode_item(long it, int J, const int32_t* slots, int E) {
  const int st = SlotTable::stride(E);
  const int32_t* s_exp = slots + SlotTable::kHeader;
  const int32_t* s_row0 = s_exp + st;
  const int32_t* s_rows = s_row0 + st;
  const int32_t* s_blk = s_rows + st;
  const int n_slots = slots[SlotTable::kNumBig];
  int lo = 0, hi = n_slots - 1;  // last slot s with J * blk[s] <= it
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long>(J) * s_blk[mid] <= it) lo = mid;
    else hi = mid - 1;
  }
  const long local = it - static_cast<long>(J) * s_blk[lo];
  const int T = s_blk[lo + 1] - s_blk[lo];
  BigItem x;
  x.slot = lo;
  x.e = s_exp[lo];
  x.row0 = s_row0[lo];
  x.rows = s_rows[lo];
  x.jt = static_cast<int>(local / T);
  x.tb = static_cast<int>(local % T);
  return x;
}

// 16 int8 codes -> 16 f16 values, exactly: byte v + 128 under the f16
// exponent of 1024 reads as 1024 + v + 128; subtracting 1152 leaves v.
__device__ __forceinline__ void int8x16_to_f16(uint4 in, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {in.x ^ 0x80808080u, in.y ^ 0x80808080u, in.z ^ 0x80808080u, in.w ^ 0x80808080u};
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t a = __byte_perm(w[i], 0x64646464u, 0x4140);  // v0 + 1152, v1 + 1152 as f16
    uint32_t b = __byte_perm(w[i], 0x64646464u, 0x4342);  // v2, v3
    __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    o[2 * i] = *reinterpret_cast<uint32_t*>(&ha);
    o[2 * i + 1] = *reinterpret_cast<uint32_t*>(&hb);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// byte offset of 16-byte chunk j of row r in a [rows][64] f16 tile with the
// 128-byte swizzle (the layout the UMMA descriptor and the TMA expect)
__device__ __forceinline__ int sw128_chunk(int r, int j) { return (r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4); }

template <int MODE>
__global__ void __launch_bounds__(kBigThreads, 1)
    moe_gemm_big_kernel(const __grid_constant__ TcMaps maps, FwdParams p, int32_t* raw) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  extern __shared__ __align__(1024) char smem[];
  uint64_t* a8_full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* a8_empty = a8_full + S8;
  uint64_t* b_full = a8_empty + S8;
  uint64_t* f16_empty = b_full + S16;
  uint64_t* cv_full = f16_empty + S16;
  uint64_t* acc_full = cv_full + S16;
  uint64_t* acc_empty = acc_full + 2;
  float* tok_scale = reinterpret_cast<float*>(smem + OFF_INFO);
  int32_t* tok_row = reinterpret_cast<int32_t*>(smem + OFF_INFO) + TB;
  int32_t* tok_tok = tok_row + TB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC) + 1;

  grid_dependency_wait();
  grid_launch_dependents();

  const int K = G1 ? p.h : p.I;
  const int NW = G1 ? 2 * p.I : p.h;
  const int J = G1 ? p.I / 64 : (p.h + BM - 1) / BM;   // weight tiles per token block
  const int n_kb = K / KB;
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  const int32_t* s_blk = slots + SlotTable::kHeader + 3 * SlotTable::stride(p.E);
  const long total = static_cast<long>(slots[SlotTable::kBigBlocks]) * J;
  const int site = (G1 ? kKGemm1Big : kKGemm2Big) * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (total <= blockIdx.x) return;  // uniform: no item for this CTA (before any barrier or allocation)

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) report_timeout(status, site + 15);  // swizzle alignment broken
    for (int s = 0; s < S8; ++s) {
      mbar_init(&a8_full[s], 1);
      mbar_init(&a8_empty[s], kConvWarps);
    }
    for (int s = 0; s < S16; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&f16_empty[s], 1);
      mbar_init(&cv_full[s], kConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kBigWarps - kEpiWarp0);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  if (aligned && warp == kWarpA) {
    // ---------------------------------------------------- weight TMA (int8)
    if (lane == 0) {
      const void* map = G1 ? &maps.a1 : &maps.a2;
      const void* map_s = G1 ? &maps.a1s : &maps.a2s;
      long n = 0;
      for (long it = blockIdx.x; it < total; it += gridDim.x) {
        const BigItem x = decode_item(it, J, slots, p.E);
        const bool sh = x.e < 0;
        const int rbase = sh ? 0 : x.e * NW;
        for (int kb = 0; kb < n_kb; ++kb, ++n) {
          const int s = static_cast<int>(n % S8);
          const long round = n / S8;
          if (round > 0 && !mbar_wait_bounded(&a8_empty[s], (round - 1) & 1, abort_flag, status, site + 1, false))
            goto done_a;
          mbar_arrive_expect_tx(&a8_full[s], A8_BYTES);
          char* dst = smem + OFF_A8 + s * A8_BYTES;
          if (G1) {
            tma_load_2d(dst, sh ? map_s : map, kb * KB, rbase + x.jt * 64, &a8_full[s]);
            tma_load_2d(dst + 64 * KB, sh ? map_s : map, kb * KB, rbase + p.I + x.jt * 64, &a8_full[s]);
          } else {
            tma_load_2d(dst, sh ? map_s : map, kb * KB, rbase + x.jt * BM, &a8_full[s]);
          }
        }
      }
    done_a:;
    }
  } else if (aligned && warp == kWarpB) {
    // ---------------------------------------------------- token TMA (f16)
    if (lane == 0) {
      const void* map = G1 ? &maps.b1 : &maps.b2;
      long n = 0;
      for (long it = blockIdx.x; it < total; it += gridDim.x) {
        const BigItem x = decode_item(it, J, slots, p.E);
        const int r0 = x.row0 + x.tb * TB;
        for (int kb = 0; kb < n_kb; ++kb, ++n) {
          const int s = static_cast<int>(n % S16);
          const long round = n / S16;
          if (round > 0 && !mbar_wait_bounded(&f16_empty[s], (round - 1) & 1, abort_flag, status, site + 2, false))
            goto done_b;
          mbar_arrive_expect_tx(&b_full[s], F16_TILE);
          tma_load_2d(smem + OFF_B16 + s * F16_TILE, map, kb * KB, r0, &b_full[s]);
        }
      }
    done_b:;
    }
  } else if (aligned && warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
    // ------------------------------------------- int8 -> f16 weight stages
    const int ct = threadIdx.x - kConvWarp0 * 32;  // 0..127
    long n = 0;
    for (long it = blockIdx.x; it < total; it += gridDim.x) {
      for (int kb = 0; kb < n_kb; ++kb, ++n) {
        const int s8 = static_cast<int>(n % S8), s16 = static_cast<int>(n % S16);
        const long r8 = n / S8, r16 = n / S16;
        bool ok = mbar_wait_bounded(&a8_full[s8], r8 & 1, abort_flag, status, site + 3);
        if (ok && r16 > 0) ok = mbar_wait_bounded(&f16_empty[s16], (r16 - 1) & 1, abort_flag, status, site + 4);
        if (ok) {
          const char* src = smem + OFF_A8 + s8 * A8_BYTES;
          char* dst = smem + OFF_A16 + s16 * F16_TILE;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int task = ct + 128 * i;
            const int row = task >> 2, c = task & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(src + row * KB + c * 16);
            uint4 lo, hi;
            int8x16_to_f16(v, lo, hi);
            *reinterpret_cast<uint4*>(dst + sw128_chunk(row, 2 * c)) = lo;
            *reinterpret_cast<uint4*>(dst + sw128_chunk(row, 2 * c + 1)) = hi;
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&a8_empty[s8]);
          mbar_arrive(&cv_full[s16]);
        }
        if (!ok) break;
      }
      if (*abort_flag) break;
    }
  } else if (aligned && warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      long n = 0, acc_n = 0;
      bool ok = true;
      for (long it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const BigItem x = decode_item(it, J, slots, p.E);
        const int mblk = min(TB, x.rows - x.tb * TB);
        const uint32_t idesc = umma_idesc_f16(BM, (mblk + 15) & ~15);
        int buf = 0;
        for (int kb = 0; kb < n_kb && ok; ++kb, ++n) {
          const int s16 = static_cast<int>(n % S16);
          const long r16 = n / S16;
          if (kb % CHUNK_KB == 0) {
            buf = static_cast<int>(acc_n & 1);
            if (acc_n >= 2) ok = mbar_wait_bounded(&acc_empty[buf], ((acc_n >> 1) - 1) & 1, abort_flag, status, site + 5);
            tc_fence_after();
          }
          if (ok) ok = mbar_wait_bounded(&cv_full[s16], r16 & 1, abort_flag, status, site + 6);
          if (ok) ok = mbar_wait_bounded(&b_full[s16], r16 & 1, abort_flag, status, site + 7);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + OFF_A16 + s16 * F16_TILE);
          const uint32_t b_base = smem_u32(smem + OFF_B16 + s16 * F16_TILE);
#pragma unroll
          for (int ks = 0; ks < KB / 16; ++ks) {
            umma_f16(tmem + buf * TB, umma_desc_sw128(a_base + ks * 32), umma_desc_sw128(b_base + ks * 32), idesc,
                     (kb % CHUNK_KB != 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(&f16_empty[s16]);
          if (kb % CHUNK_KB == CHUNK_KB - 1 || kb == n_kb - 1) {
            umma_commit(&acc_full[buf]);
            ++acc_n;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int ctid = threadIdx.x - kEpiWarp0 * 32;   // 0..255
    const int q = warp & 3;                           // tensor-memory lane quadrant
    const int half = (warp - kEpiWarp0) >> 2;         // token columns [64 half, 64 half + 64)
    const int m = 32 * q + lane;                      // weight row inside the tile
    const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
    const float* xsc = ws_ptr<float>(p, p.L.x_scale);
    const float* xssc = p.share_uses_xq ? xsc : ws_ptr<float>(p, p.L.xs_scale);
    const float* s2 = ws_ptr<float>(p, p.L.s2);
    float* hbuf = ws_ptr<float>(p, p.L.hbuf);
    uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
    float* xch = reinterpret_cast<float*>(smem + OFF_X);
    long acc_n = 0;
    for (long it = blockIdx.x; it < total; it += gridDim.x) {
      const BigItem x = decode_item(it, J, slots, p.E);
      const int tok0 = x.tb * TB;
      const int mblk = min(TB, x.rows - tok0);
      consumer_sync();  // the previous item's epilogue is done with the token info
      if (ctid < mblk) {
        const int r = x.row0 + tok0 + ctid;
        const int t = row_token[r];
        tok_row[ctid] = r;
        tok_tok[ctid] = t;
        tok_scale[ctid] = G1 ? (x.e >= 0 ? xsc : xssc)[t] : s2[r];
      }
      consumer_sync();
      int acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0;
      const int n_chunks = (n_kb + CHUNK_KB - 1) / CHUNK_KB;
      bool ok = aligned;
      for (int c = 0; c < n_chunks && ok; ++c, ++acc_n) {
        const int buf = static_cast<int>(acc_n & 1);
        ok = mbar_wait_bounded(&acc_full[buf], (acc_n >> 1) & 1, abort_flag, status, site + 8);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if (64 * half + 32 * cc < mblk) {
            uint32_t v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * TB + 64 * half + 32 * cc, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[32 * cc + j] += __float2int_rn(__uint_as_float(v[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      consumer_sync();
      const bool stop = *abort_flag != 0;  // a failed wait raised it before this barrier
      if (!aligned) break;
      int ng;
      if (G1) ng = (m < 64) ? x.jt * 64 + m : p.I + x.jt * 64 + (m - 64);
      else ng = x.jt * BM + m;
      if (RAW) {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int tok = 64 * half + j;
          if (tok < mblk && ng < NW) raw[static_cast<size_t>(tok_row[tok]) * NW + ng] = acc[j];
        }
      } else if (G1) {
        const float ws = (x.e >= 0 ? p.w1s + static_cast<size_t>(x.e) * NW : p.sw1s)[ng];
        if (m >= 64) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int tok = 64 * half + j;
            if (tok < mblk) xch[(m - 64) * XSTRIDE + tok] = __fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tok_scale[tok]);
          }
        }
        consumer_sync();
        if (m < 64) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int tok = 64 * half + j;
            if (tok < mblk) {
              const float g = __fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tok_scale[tok]);
              const float u = xch[m * XSTRIDE + tok];
              const float d = __fadd_rn(1.0f, expf(-g));
              hbuf[static_cast<size_t>(tok_row[tok]) * p.I + x.jt * 64 + m] = __fmul_rn(__fdiv_rn(g, d), u);
            }
          }
        }
      } else {
        const float ws = (x.e >= 0 ? p.w2s + static_cast<size_t>(x.e) * NW : p.sw2s)[ng];
        const bool valid_n = ng < p.h;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int tok = 64 * half + j;
          if (tok < mblk && valid_n) {
            const uint16_t b = f32_to_bf16_bits(__fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tok_scale[tok]));
            if (x.e >= 0) y2[static_cast<size_t>(tok_row[tok]) * p.h + ng] = b;
            else p.sout[static_cast<size_t>(tok_tok[tok]) * p.h + ng] = b;
          }
        }
      }
      if (stop) break;
    }
  }
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// f16 copies of the token codes of every row in a big block: the GEMM1
// operand that the tensor-memory path reads with TMA.
__global__ void __launch_bounds__(256) expand_kernel(FwdParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  const int total = slots[SlotTable::kBigBlocks];
  if (total == 0) return;
  const int st = SlotTable::stride(p.E);
  const int32_t* s_exp = slots + SlotTable::kHeader;
  const int32_t* s_row0 = s_exp + st;
  const int32_t* s_rows = s_row0 + st;
  const int32_t* s_blk = s_rows + st;
  const int n_slots = slots[SlotTable::kNumBig];
  const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  const int8_t* xq = ws_ptr<int8_t>(p, p.L.x_q);
  const int8_t* xsq = p.share_uses_xq ? xq : ws_ptr<int8_t>(p, p.L.xs_q);
  __half* x1h = ws_ptr<__half>(p, p.L.x1h);
  const int n16 = p.h >> 4;
  for (int b = blockIdx.x; b < total; b += gridDim.x) {
    int lo = 0, hi = n_slots - 1;  // slot of block b
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_blk[mid] <= b) lo = mid;
      else hi = mid - 1;
    }
    const int tb = b - s_blk[lo];
    const int r0 = s_row0[lo] + tb * TB;
    const int n = min(TB, s_rows[lo] - tb * TB);
    const int8_t* src = s_exp[lo] >= 0 ? xq : xsq;
    for (int idx = threadIdx.x; idx < n * n16; idx += blockDim.x) {
      const int i = idx / n16, c = idx % n16;
      const int r = r0 + i;
      const uint4 v = reinterpret_cast<const uint4*>(src + static_cast<size_t>(row_token[r]) * p.h)[c];
      uint4 lo16, hi16;
      int8x16_to_f16(v, lo16, hi16);
      uint4* dst = reinterpret_cast<uint4*>(x1h + static_cast<size_t>(r) * p.h) + 2 * c;
      dst[0] = lo16;
      dst[1] = hi16;
    }
  }
}

// Requant of the rows of big blocks (FusedDeepMoE analysis §7.2), one warp
// per row: amax = max(max|h|, 1e-4), s2 = amax * (1/127),
// q = RNE((h * 127) * (1/amax)); writes the int8 codes, their f16 copy (the
// tensor-core GEMM2 operand) and s2.
__global__ void __launch_bounds__(256) requant_big_kernel(FwdParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  const int total = slots[SlotTable::kBigBlocks];
  if (total == 0) return;
  const int st = SlotTable::stride(p.E);
  const int32_t* s_row0 = slots + SlotTable::kHeader + st;
  const int32_t* s_rows = s_row0 + st;
  const int32_t* s_blk = s_rows + st;
  const int n_slots = slots[SlotTable::kNumBig];
  const int I = p.I, n4 = I >> 2;
  const float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
  __half* x2h = ws_ptr<__half>(p, p.L.x2h);
  float* s2 = ws_ptr<float>(p, p.L.s2);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const long nrows = static_cast<long>(total) * TB;  // block-major row slots (some empty)
  for (long g = gw; g < nrows; g += nw) {
    const int b = static_cast<int>(g / TB), i = static_cast<int>(g % TB);
    int lo = 0, hi = n_slots - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_blk[mid] <= b) lo = mid;
      else hi = mid - 1;
    }
    const int tb = b - s_blk[lo];
    if (tb * TB + i >= s_rows[lo]) continue;
    const int r = s_row0[lo] + tb * TB + i;
    const float4* hr = reinterpret_cast<const float4*>(hbuf + static_cast<size_t>(r) * I);
    float amax = 0.0f;
    for (int c = lane; c < n4; c += 32) {
      const float4 v = hr[c];
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (amax < 1e-4f) amax = 1e-4f;
    const float inv = __fdiv_rn(1.0f, amax);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(x2 + static_cast<size_t>(r) * I);
    __half2* h2 = reinterpret_cast<__half2*>(x2h + static_cast<size_t>(r) * I);
    for (int c = lane; c < n4; c += 32) {
      const float4 v = hr[c];
      const float f[4] = {v.x, v.y, v.z, v.w};
      int8_t q[4];
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        q[j] = f32_to_q(__fmul_rn(__fmul_rn(f[j], 127.0f), inv));
        packed |= static_cast<uint32_t>(static_cast<uint8_t>(q[j])) << (8 * j);
      }
      q4[c] = packed;
      h2[2 * c] = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[1]));
      h2[2 * c + 1] = __halves2half2(__int2half_rn(q[2]), __int2half_rn(q[3]));
    }
    if (lane == 0) s2[r] = __fmul_rn(amax, 1.0f / 127.0f);
  }
}

// Combine of every token (FusedDeepMoE analysis §4.2) when the forward has big
// blocks; otherwise the small-expert GEMM2 already combined every token.
__global__ void __launch_bounds__(256) combine_kernel(FwdParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  if (slots[SlotTable::kBigBlocks] == 0) return;
  const int32_t* tok_expect = ws_ptr<int32_t>(p, p.L.tok_expect);
  for (int t = blockIdx.x; t < p.bs; t += gridDim.x) {
    if (tok_expect[t] == 0) continue;  // inactive, or no valid id: zeroed by the quant
    combine_token(p, t, threadIdx.x);
  }
}

}  // namespace

cudaError_t launch_requant_big(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.num_ctas * 4), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, requant_big_kernel, p);
}

cudaError_t launch_combine(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.num_ctas * 4), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

cudaError_t moe_gemm_big_prepare_attributes() {
  const void* fns[] = {reinterpret_cast<const void*>(moe_gemm_big_kernel<kGemm1SwiGLU>),
                       reinterpret_cast<const void*>(moe_gemm_big_kernel<kGemm2Bf16>),
                       reinterpret_cast<const void*>(moe_gemm_big_kernel<kGemm1Raw>),
                       reinterpret_cast<const void*>(moe_gemm_big_kernel<kGemm2Raw>)};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_expand(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.num_ctas), dim3(256), 0, s, attr);
  return cudaLaunchKernelEx(&cfg, expand_kernel, p);
}

cudaError_t launch_moe_gemm_big(const FwdParams& p, const TcMaps& maps, int mode, int32_t* raw_acc, int num_ctas,
                                cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(dim3(num_ctas), dim3(kBigThreads), SMEM_BYTES, s, attr);
  switch (mode) {
    case kGemm1SwiGLU: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm1SwiGLU>, maps, p, raw_acc);
    case kGemm2Bf16: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm2Bf16>, maps, p, raw_acc);
    case kGemm1Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm1Raw>, maps, p, raw_acc);
    case kGemm2Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm2Raw>, maps, p, raw_acc);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
