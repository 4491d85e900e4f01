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
// Tile: 128 weight rows x up to 128 token rows of one expert x all of K,
// weights as the MMA's M operand (tensor-memory lanes, read by the MMA from
// tensor memory), tokens as N (shared memory).  Per 128 of K the int8 weight
// stage passes through shared memory once (TMA write, converter read) and so
// does the f16 token stage (TMA write, MMA read).  What bounds the kernel is
// the stage loop between the producers, the converter warps and the MMA: at
// full tiles a stage takes about 1050 cycles against 512 cycles of tensor
// work (an isolated M128 N128 K16 MMA takes 64 cycles, random operands or
// not), and taking out the token copies, the conversion arithmetic, the
// tensor-memory stores or half of the MMAs each gains only 1-4 %.  With all
// of them taken out the bare handshake ring (the same waits, arrivals and
// commits) still costs about 470 cycles a stage under this kernel's load,
// and each kind of work adds to it instead of hiding under it; 256-K stages,
// one accumulator with six weight slots, converting ahead of the free slot
// and sleeping pollers were each no faster.  For
// GEMM1 the 128 rows are 64 gate rows and the 64 matching up rows, laid out
// so that each 32-lane quadrant of tensor memory holds 16 gate rows in its
// lanes 0..15 and the 16 matching up rows in lanes 16..31 (every warp
// store then covers one 64-byte run of gate and one of up values, and the
// gate and up values of one output column meet in one warp for SwiGLU).
// The requant of big blocks and the combine of forwards with big blocks run
// as separate parallel kernels (below): done by the CTA that finishes a block
// last, they would serialise 128-row blocks and 128-token tiles on a few SMs.
// Warp roles (one CTA per SM, persistent):
// A stage is 128 of K: two 64-wide atoms of the 128-byte swizzle per f16 tile.
//   warp 0      TMA of the int8 weight boxes into a 6-deep staging ring
//   warp 2      TMA of the f16 token boxes (128-byte swizzle) into a 4-deep
//               ring; 16-row boxes when the block has at most 64 rows
//   warp 3      item scheduler: decodes the CTA's work items (slot-table
//               search, a chain of dependent global loads) into a 4-deep
//               shared-memory ring that the other roles read
//   warps 4..7  convert int8 weight stages to f16, one weight row per
//               thread, into a 4-deep ring in tensor memory (the MMA's A
//               operand), which keeps the f16 weights off shared memory;
//               software-pipelined when the launch's blocks are short
//   warp 1      one elected lane issues tcgen05.mma (M128, N = rows rounded
//               to 16, K16) stage by stage into two tensor-memory
//               accumulators, alternating per 1024 of K, and commits to the
//               ring and accumulator barriers
//   warps 8..15 drain accumulators (tcgen05.ld) into int32, then the
//               epilogue (GEMM1: dequant, SwiGLU, h and the row maxima of
//               |h| for the requant kernel; GEMM2: dequant to the activation
//               dtype); two warps per tensor-memory lane quadrant
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
constexpr int KB = 128;               // K elements per stage
constexpr int KA = 64;                // K elements per swizzle atom (one 128-byte f16 row)
constexpr int ATOMS = KB / KA;        // swizzle atoms per f16 stage
constexpr int CHUNK_KB = 1024 / KB;   // stages per exact accumulation chunk (1024 of K)
constexpr int S8 = 6;                 // int8 weight staging ring (from HBM)
constexpr int SA = 4;                 // f16 weight ring in tensor memory (converted in the CTA)
constexpr int SB = 4;                 // f16 token ring (from L2)
constexpr int SI = 4;                 // decoded work-item ring (item scheduler -> the other roles)
constexpr int kAccCols = 2 * TB;      // two fp32 accumulators of TB columns
constexpr int kAStageCols = KB / 2;   // one f16 weight stage: 128 lanes x 64 columns of f16 pairs
constexpr int kTmemCols = 512;        // kAccCols + SA * kAStageCols, rounded to a power of two
static_assert(kAccCols + SA * kAStageCols <= kTmemCols, "tensor memory budget");
constexpr int kSmallBox = 16;         // rows of the narrow token box

constexpr int kBigWarps = 16;
constexpr int kBigThreads = kBigWarps * 32;
constexpr int kWarpA = 0, kWarpMma = 1, kWarpB = 2, kWarpSched = 3;
constexpr int kConvWarp0 = 4, kConvWarps = 4;
constexpr int kEpiWarp0 = 8;          // epilogue warps 8..15 = the 256 "consumer" threads

constexpr int A8_BYTES = BM * KB;                    // 16 KB: [128 rows][128] int8, 128-byte swizzle
constexpr int F16_ATOM = 128 * KA * 2;               // 16 KB: [128 rows][64] f16, 128-byte swizzle
constexpr int F16_TILE = ATOMS * F16_ATOM;           // 32 KB
constexpr int OFF_B16 = 0;                           // SB x ATOMS x [128][64] f16, swizzled (TMA)
constexpr int OFF_A8 = OFF_B16 + SB * F16_TILE;      // S8 x [128][128] int8, swizzled (TMA)
constexpr int OFF_BAR = OFF_A8 + S8 * A8_BYTES;
constexpr int NBAR = 2 * S8 + 2 * SA + 2 * SB + 4 + 2 * SI + 1;
constexpr int OFF_INFO = OFF_BAR + NBAR * 8;         // tok_scale, tok_row, tok_tok [TB]
constexpr int OFF_ITEM = OFF_INFO + 3 * TB * 4;      // SI decoded items, 8 ints each
constexpr int OFF_MISC = OFF_ITEM + SI * 8 * 4;      // tmem slot, abort flag, arrival index
constexpr int SMEM_BYTES = OFF_MISC + 16;
constexpr int kItemReaders = 4;                      // weight TMA, token TMA, MMA, epilogue
static_assert(KB == 128 && KA == 64, "the MMA loop issues two atoms of four K16 steps per stage");
static_assert(OFF_B16 % 1024 == 0 && OFF_A8 % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(OFF_BAR % 8 == 0, "mbarrier alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");

struct BigItem {
  int slot, e, row0, rows, tb, jt, mblk;
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
  x.mblk = min(TB, x.rows - x.tb * TB);
  return x;
}

// Decoded items pass from the scheduler warp to the other roles through a
// shared-memory ring (one 8-int entry per item): the decode's chain of
// dependent global loads then runs ahead of the pipeline instead of stalling
// every role at each item boundary.
__device__ __forceinline__ void put_item(int32_t* ent, const BigItem& x) {
  ent[0] = x.slot; ent[1] = x.e; ent[2] = x.row0; ent[3] = x.rows;
  ent[4] = x.tb; ent[5] = x.jt; ent[6] = x.mblk;
}
__device__ __forceinline__ BigItem get_item(const volatile int32_t* ent) {
  BigItem x;
  x.slot = ent[0]; x.e = ent[1]; x.row0 = ent[2]; x.rows = ent[3];
  x.tb = ent[4]; x.jt = ent[5]; x.mblk = ent[6];
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

// A TMA producer's exit: wait (bounded, and not cut short by an abort) until
// every copy it issued has landed, i.e. the last phase it armed on each slot
// of its ring has completed, so that no copy still writes into this CTA's
// shared memory once the CTA ends.  `s` / `ph`: the next slot and its phase
// parity; slots before `s` were last armed in the current lap, the others
// (once the ring has wrapped) in the previous one.  Called by the whole warp.
__device__ __forceinline__ void drain_ring(uint64_t* full, int n, int s, uint32_t ph, bool wrapped,
                                           int32_t* status, int site) {
  for (int i = 0; i < n; ++i) {
    if (i < s) mbar_wait_bounded(&full[i], ph, nullptr, status, site);
    else if (wrapped) mbar_wait_bounded(&full[i], ph ^ 1u, nullptr, status, site);
  }
}

// SwiGLU of one dequantised gate / up pair (FusedDeepMoE analysis §6.1):
// t = exp(-g), d = 1 + t, h = (g / d) * u, each step rounded once.
__device__ __forceinline__ float swiglu_1(float g, float u) {
  const float d = __fadd_rn(1.0f, expf(-g));
  return __fmul_rn(__fdiv_rn(g, d), u);
}

// Max over the 16 lanes of each half-warp of 32 values per lane, scattered:
// on return lane L (of 16) holds in v[0], v[1] the maxima of entries 2L and
// 2L + 1 (four butterfly steps, each halving the entries a lane keeps; the
// kept half is chosen by selects, so the array stays in registers).
__device__ __forceinline__ void halfwarp_max_scatter(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int o = 8 >> step;       // lane distance 8, 4, 2, 1
    const int n = 16 >> step;      // entries kept after this step
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float keep = hi ? v[n + i] : v[i];
      const float give = hi ? v[i] : v[n + i];
      v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, o));
    }
  }
}

// Dequant (§6.1: (float(acc) * w_scale) * x_scale) and SwiGLU of one half
// tile in the GEMM1 epilogue: 64 token slots of one output column.  Lane
// l < 16 holds the gate values of the column's slots (acc, gate scale ws),
// lane l + 16 the matching up values (up scale).  Gate lanes take slots
// 0 .. S-1, up lanes S .. 2S-1, and each trades the other S values with its
// partner, one shuffle a slot; S (8 or 16) is the smaller that covers the
// vt <= 32 slots the half holds, so a short block evaluates its own rows
// only (a half of more than 32 rows takes the epilogue's own code).
// h goes to the row's first I floats; max |h| over the tile's columns is
// published per row by an atomic maximum on the float bits (h >= 0 bits
// order as integers), so that the requant needs one pass over h.
template <int S>
__device__ __forceinline__ void swiglu_half_tile(const int (&acc)[64], const float* tscale, const int32_t* trow,
                                                 float ws, bool gate, int lane, int vt, float* hbuf, size_t hstride,
                                                 int col, int32_t* amax2) {
  float hv[32];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (8 * c < S && 8 * c < vt) {  // 8-slot chunks past the half's rows skipped (warp-uniform)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = 8 * c + jj;
        // this lane's dequantised values of slots j and S + j
        const float lo = __fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tscale[j]);
        const float hi = __fmul_rn(__fmul_rn(__int2float_rn(acc[S + j]), ws), tscale[S + j]);
        // gate lanes send gate(S + j) and receive up(j); up lanes the reverse
        const float other = __shfl_xor_sync(0xffffffffu, gate ? hi : lo, 16);
        hv[j] = gate ? swiglu_1(lo, other) : swiglu_1(other, hi);
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) hv[8 * c + jj] = 0.0f;
    }
  }
  const int t0 = gate ? 0 : S;  // slot of hv[0]
#pragma unroll
  for (int j = 0; j < S; ++j)
    if (t0 + j < vt) hbuf[static_cast<size_t>(trow[t0 + j]) * hstride + col] = hv[j];
#pragma unroll
  for (int j = 0; j < 32; ++j) hv[j] = fabsf(hv[j]);
  halfwarp_max_scatter(hv, lane & 15);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int k = 2 * (lane & 15) + u;
    if (k < S && t0 + k < vt) atomicMax(amax2 + trow[t0 + k], __float_as_int(hv[u]));
  }
}

template <int MODE>
__global__ void __launch_bounds__(kBigThreads, 1)
    moe_gemm_big_kernel(const __grid_constant__ TcMaps maps, FwdParams p, int32_t* raw) {
  constexpr bool G1 = (MODE == kGemm1SwiGLU || MODE == kGemm1Raw);
  constexpr bool RAW = (MODE == kGemm1Raw || MODE == kGemm2Raw);
  extern __shared__ __align__(1024) char smem[];
  uint64_t* a8_full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* a8_empty = a8_full + S8;
  uint64_t* a16_full = a8_empty + S8;
  uint64_t* a16_empty = a16_full + SA;
  uint64_t* b_full = a16_empty + SA;
  uint64_t* b_empty = b_full + SB;
  uint64_t* acc_full = b_empty + SB;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* it_full = acc_empty + 2;
  uint64_t* it_empty = it_full + SI;
  uint64_t* drain_bar = it_empty + SI;  // the MMA thread's final commit
  volatile int32_t* items = reinterpret_cast<volatile int32_t*>(smem + OFF_ITEM);
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
  const int n_kb = (K + KB - 1) / KB;  // a last half stage reads zeros beyond K (TMA fill)
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  int32_t* status = ws_ptr<int32_t>(p, p.L.status);
  const long total = static_cast<long>(slots[SlotTable::kBigBlocks]) * J;
  const int site = (G1 ? kKGemm1Big : kKGemm2Big) * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // This CTA's first item and the item stride: blockIdx.x and gridDim.x, or,
  // with the engines side by side (the dp4a launch holding the other SMs),
  // the CTA's place in arrival order among the num_ctas - (small-phase CTAs)
  // that work, so that those are the ones that got an SM.
  long cta0 = blockIdx.x, ncta = gridDim.x;
  if (slots[SlotTable::kSplit]) {
    cta0 = arrival_index(status + kStCtaCounter + (G1 ? 1 : 2), reinterpret_cast<int*>(smem + OFF_MISC) + 2);
    ncta = p.num_ctas - slots[SlotTable::kSmallCtas];
  }
  if (total <= cta0 || cta0 >= ncta) return;  // uniform: no item for this CTA (before any barrier or allocation)

  if (threadIdx.x == 0) {
    if ((smem_u32(smem) & 1023u) != 0) report_timeout(status, site + 15);  // swizzle alignment broken
    for (int s = 0; s < S8; ++s) {
      mbar_init(&a8_full[s], 1);
      mbar_init(&a8_empty[s], kConvWarps);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(&a16_full[s], kConvWarps);
      mbar_init(&a16_empty[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kBigWarps - kEpiWarp0);
    }
    for (int s = 0; s < SI; ++s) {
      mbar_init(&it_full[s], 1);
      mbar_init(&it_empty[s], kItemReaders);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool aligned = (smem_u32(smem) & 1023u) == 0;

  // The single-issuer roles (the two TMA producers and the MMA issuer) run
  // their loops on the whole warp, so every address and descriptor is
  // warp-uniform; one elected lane issues the copies and tensor-core work.
  // Every role walks the same item sequence (cta0, + ncta, ...)
  // and takes each item's decoded form from the scheduler's ring.
  int si = 0;
  uint32_t pi = 0;
  if (aligned && warp == kWarpSched) {
    // ------------------------------------------------------- item scheduler
    bool wrapped = false;
    for (long it = cta0; it < total; it += ncta) {
      const BigItem x = decode_item(it, J, slots, p.E);
      if (wrapped &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(&it_empty[si], pi ^ 1u, abort_flag, status, site + 9, false)))
        break;
      if (lane == 0) {
        put_item(const_cast<int32_t*>(items) + 8 * si, x);
        mbar_arrive(&it_full[si]);
      }
      __syncwarp();
      if (++si == SI) { si = 0; pi ^= 1u; wrapped = true; }
    }
  } else if (aligned && warp == kWarpA) {
    // ---------------------------------------------------- weight TMA (int8)
    int s = 0;
    uint32_t ph = 0;
    bool wrapped = false;
    for (long it = cta0; it < total; it += ncta) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&it_full[si], pi, abort_flag, status, site + 10))) goto done_a;
      const BigItem x = get_item(items + 8 * si);
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[si]);
      if (++si == SI) { si = 0; pi ^= 1u; }
      const bool sh = x.e < 0;
      const int rbase = sh ? 0 : x.e * NW;
      const void* mp = sh ? (G1 ? &maps.a1s : &maps.a2s) : (G1 ? &maps.a1 : &maps.a2);
      for (int kb = 0; kb < n_kb; ++kb) {
        if (wrapped &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(&a8_empty[s], ph ^ 1u, abort_flag, status, site + 1, false)))
          goto done_a;
        if (elect_one()) {
          mbar_arrive_expect_tx(&a8_full[s], A8_BYTES);
          char* dst = smem + OFF_A8 + s * A8_BYTES;
          if (G1) {
            // tile rows 32 g .. 32 g + 15: gate rows 16 g ..; 32 g + 16 ..: the matching up rows
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const int gate = rbase + x.jt * 64 + 16 * g;
              tma_load_2d(dst + (32 * g) * KB, mp, kb * KB, gate, &a8_full[s]);
              tma_load_2d(dst + (32 * g + 16) * KB, mp, kb * KB, gate + p.I, &a8_full[s]);
            }
          } else {
            tma_load_2d(dst, mp, kb * KB, rbase + x.jt * BM, &a8_full[s]);
          }
        }
        __syncwarp();
        if (++s == S8) { s = 0; ph ^= 1u; wrapped = true; }
      }
    }
  done_a:
    drain_ring(a8_full, S8, s, ph, wrapped, status, site + 12);
  } else if (aligned && warp == kWarpB) {
    // ---------------------------------------------------- token TMA (f16)
    int s = 0;
    uint32_t ph = 0;
    bool wrapped = false;
    for (long it = cta0; it < total; it += ncta) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&it_full[si], pi, abort_flag, status, site + 10))) goto done_b;
      const BigItem x = get_item(items + 8 * si);
      __syncwarp();
      if (lane == 0) mbar_arrive(&it_empty[si]);
      if (++si == SI) { si = 0; pi ^= 1u; }
      const int r0 = x.row0 + x.tb * TB;
      const int mblk = x.mblk;
      // narrow boxes for short blocks: the MMA reads only the first mblk rows
      const int nbox = mblk > 64 ? 1 : (mblk + kSmallBox - 1) / kSmallBox;
      const uint32_t bytes = ATOMS * (mblk > 64 ? F16_ATOM : nbox * kSmallBox * KA * 2);
      const void* map = G1 ? &maps.b1 : &maps.b2;
      const void* map_n = G1 ? &maps.b1n : &maps.b2n;
      for (int kb = 0; kb < n_kb; ++kb) {
        if (wrapped &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(&b_empty[s], ph ^ 1u, abort_flag, status, site + 2, false)))
          goto done_b;
        if (elect_one()) {
          mbar_arrive_expect_tx(&b_full[s], bytes);
          char* dst = smem + OFF_B16 + s * F16_TILE;
#pragma unroll
          for (int a = 0; a < ATOMS; ++a) {
            const int kx = kb * KB + a * KA;
            if (mblk > 64) {
              tma_load_2d(dst + a * F16_ATOM, map, kx, r0, &b_full[s]);
            } else {
              for (int b = 0; b < nbox; ++b)
                tma_load_2d(dst + a * F16_ATOM + b * kSmallBox * KA * 2, map_n, kx, r0 + b * kSmallBox, &b_full[s]);
            }
          }
        }
        __syncwarp();
        if (++s == SB) { s = 0; ph ^= 1u; wrapped = true; }
      }
    }
  done_b:
    drain_ring(b_full, SB, s, ph, wrapped, status, site + 13);
  } else if (aligned && warp >= kConvWarp0 && warp < kConvWarp0 + kConvWarps) {
    // ------------------------------- int8 -> f16 weight rows, into tensor memory
    // Thread = weight row = tensor-memory lane (warp 4 + q owns lanes 32 q ..).
    // Row r's 16-byte chunk j sits at chunk j ^ (r % 8) of its 128-byte line
    // (the TMA's 128-byte swizzle), so the 32 rows of a warp read 8 distinct
    // bank groups per load.  Codes 16 j .. 16 j + 15 become the f16 pairs of
    // columns 8 j .. 8 j + 7 of the stage.
    // Two loop orders, chosen per launch from the big blocks' mean row count:
    //  * short blocks (<= 64 rows: the MMA of a stage is cheap, conversion
    //    bounds the kernel): software-pipelined over the CTA's stages.  Stage
    //    k's tensor-memory stores are issued, then stage k + 1's codes are
    //    loaded (and their staging slot released), and only then does the
    //    warp wait for stage k's stores and hand the slot to the MMA, so the
    //    store latency overlaps the next stage's loads;
    //  * full blocks (the tensor pipe bounds the kernel): stage by stage, each
    //    stage handed over as soon as its own stores complete.
    // (Each order measured about 5 % slower than the other on the other kind
    // of workload; loading the next stage only when a non-blocking probe finds
    // it arrived was slower than both.)
    const int row = (warp - kConvWarp0) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kAccCols;
    const int n_big = slots[SlotTable::kNumBig];
    const int32_t* big_rows = slots + SlotTable::kHeader + 2 * SlotTable::stride(p.E);
    int rows_sum = 0;
    for (int i = lane; i < n_big; i += 32) rows_sum += big_rows[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rows_sum += __shfl_xor_sync(0xffffffffu, rows_sum, o);
    const bool pipelined = rows_sum <= 64 * slots[SlotTable::kBigBlocks];
    if (pipelined) {
      const long n_items = (total - cta0 + ncta - 1) / ncta;
      const long n_stages = n_items * n_kb;
      int s8 = 0, sa = 0;
      uint32_t p8 = 0, pa = 0;
      uint4 c[8];
      // codes of the next stage into c, then its staging slot goes back to the weight TMA
      auto load_codes = [&]() -> bool {
        const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&a8_full[s8], p8, abort_flag, status, site + 3));
        if (got) {
          const char* src = smem + OFF_A8 + s8 * A8_BYTES + row * KB;
#pragma unroll
          for (int j = 0; j < 8; ++j) c[j] = *reinterpret_cast<const uint4*>(src + ((j ^ (row & 7)) << 4));
        }
        __syncwarp();
        if (got && lane == 0) mbar_arrive(&a8_empty[s8]);
        if (++s8 == S8) { s8 = 0; p8 ^= 1u; }
        return got;
      };
      bool ok = n_stages > 0 && load_codes();
      for (long k = 0; k < n_stages && ok; ++k) {
        if (k >= SA)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&a16_empty[sa], pa ^ 1u, abort_flag, status, site + 4));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t v[32];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint4 lo, hi;
            int8x16_to_f16(c[4 * h2 + jj], lo, hi);
            v[8 * jj + 0] = lo.x; v[8 * jj + 1] = lo.y; v[8 * jj + 2] = lo.z; v[8 * jj + 3] = lo.w;
            v[8 * jj + 4] = hi.x; v[8 * jj + 5] = hi.y; v[8 * jj + 6] = hi.z; v[8 * jj + 7] = hi.w;
          }
          tmem_st32(lane_base + sa * kAStageCols + 32 * h2, v);
        }
        if (k + 1 < n_stages) ok = load_codes();
        tmem_st_wait();  // also on the way out after a failed wait: no store left in flight
        tc_fence_before();
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&a16_full[sa]);
        if (++sa == SA) { sa = 0; pa ^= 1u; }
      }
    } else {
      int s8 = 0, sa = 0;
      uint32_t p8 = 0, pa = 0;
      bool wrapped = false;
      bool ok = true;
      for (long it = cta0; it < total && ok; it += ncta) {
        for (int kb = 0; kb < n_kb; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&a8_full[s8], p8, abort_flag, status, site + 3));
          if (ok && wrapped)
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&a16_empty[sa], pa ^ 1u, abort_flag, status, site + 4));
          if (ok) {
            tc_fence_after();
            const char* src = smem + OFF_A8 + s8 * A8_BYTES + row * KB;
            // all eight loads first: the tensor-memory stores below are
            // ordered asm statements that later loads cannot move above
            uint4 c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = *reinterpret_cast<const uint4*>(src + ((j ^ (row & 7)) << 4));
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t v[32];
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                uint4 lo, hi;
                int8x16_to_f16(c[4 * h2 + jj], lo, hi);
                v[8 * jj + 0] = lo.x; v[8 * jj + 1] = lo.y; v[8 * jj + 2] = lo.z; v[8 * jj + 3] = lo.w;
                v[8 * jj + 4] = hi.x; v[8 * jj + 5] = hi.y; v[8 * jj + 6] = hi.z; v[8 * jj + 7] = hi.w;
              }
              tmem_st32(lane_base + sa * kAStageCols + 32 * h2, v);
            }
            tmem_st_wait();
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&a8_empty[s8]);
            mbar_arrive(&a16_full[sa]);
          }
          if (!ok) break;
          if (++s8 == S8) { s8 = 0; p8 ^= 1u; }
          if (++sa == SA) { sa = 0; pa ^= 1u; wrapped = true; }
        }
        if (*abort_flag) break;
      }
    }
  } else if (aligned && warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    // One 128-K stage per iteration: wait for its weight slot (tensor
    // memory) and token stage (shared memory), then one elected lane issues
    // its eight K16 MMAs and commits the slot, the stage and, at the end of a
    // 1024-K chunk, the accumulator.  (One thread running the role alone, or
    // rounds of two or four stages, measured slower.)  Ring slots and phases are running counters; the token
    // descriptor advances by addition in its address field (16-byte units: +2
    // per K16 step, +1024 per 16 KB atom); the weight operand is read from
    // tensor memory, 8 columns per K16 step.
    {
      const uint32_t a_tmem0 = tmem + kAccCols;
      const uint64_t b_desc0 = umma_desc_sw128(smem_u32(smem + OFF_B16));
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      long acc_n = 0;
      bool ok = true;
      for (long it = cta0; it < total && ok; it += ncta) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&it_full[si], pi, abort_flag, status, site + 10))) break;
        const int mblk = items[8 * si + 6];
        __syncwarp();
        if (lane == 0) mbar_arrive(&it_empty[si]);
        if (++si == SI) { si = 0; pi ^= 1u; }
        const uint32_t idesc = umma_idesc_f16(BM, (mblk + 15) & ~15);
        uint32_t d_tmem = tmem;
        int kc = 0;  // stage inside the current 1024-K chunk
        for (int kb = 0; kb < n_kb; ++kb) {
          if (kc == 0) {
            const int buf = static_cast<int>(acc_n & 1);
            d_tmem = tmem + buf * TB;
            if (acc_n >= 2 &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(&acc_empty[buf], ((acc_n >> 1) - 1) & 1, abort_flag,
                                                           status, site + 5))) {
              ok = false;
              break;
            }
          }
          const bool w = mbar_wait_bounded(&a16_full[sa], pa, abort_flag, status, site + 6) &&
                         mbar_wait_bounded(&b_full[sb], pb, abort_flag, status, site + 7);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool last = (kc + 1 == CHUNK_KB || kb + 1 == n_kb);
          if (elect_one()) {
            constexpr uint64_t kAtom = F16_ATOM >> 4;
            const uint32_t at = a_tmem0 + sa * kAStageCols;
            const uint64_t bd = b_desc0 + static_cast<uint64_t>(sb * (F16_TILE >> 4));
            umma_f16_ts(d_tmem, at, bd, idesc, kc != 0 ? 1u : 0u);
            umma_f16_ts(d_tmem, at + 8, bd + 2, idesc, 1u);
            umma_f16_ts(d_tmem, at + 16, bd + 4, idesc, 1u);
            umma_f16_ts(d_tmem, at + 24, bd + 6, idesc, 1u);
            umma_f16_ts(d_tmem, at + 32, bd + kAtom, idesc, 1u);
            umma_f16_ts(d_tmem, at + 40, bd + kAtom + 2, idesc, 1u);
            umma_f16_ts(d_tmem, at + 48, bd + kAtom + 4, idesc, 1u);
            umma_f16_ts(d_tmem, at + 56, bd + kAtom + 6, idesc, 1u);
            umma_commit(&a16_empty[sa]);
            umma_commit(&b_empty[sb]);
            if (last) umma_commit(&acc_full[acc_n & 1]);
          }
          __syncwarp();
          if (++sa == SA) { sa = 0; pa ^= 1u; }
          if (++sb == SB) { sb = 0; pb ^= 1u; }
          if (last) {
            ++acc_n;
            kc = 0;
          } else {
            ++kc;
          }
        }
      }
      // every MMA the elected lane issued completes before the CTA frees
      // tensor memory: in a normal run the epilogue already waited for the
      // last accumulator; after a wait gave up this bounded wait covers the
      // MMAs still in flight (elect.sync picks the same lane in a converged warp)
      if (elect_one()) umma_commit(drain_bar);
      __syncwarp();
      mbar_wait_bounded(drain_bar, 0, nullptr, status, site + 11);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int ctid = threadIdx.x - kEpiWarp0 * 32;   // 0..255
    const int q = warp & 3;                           // tensor-memory lane quadrant
    const int half = (warp - kEpiWarp0) >> 2;         // token columns [64 half, 64 half + 64)
    const int m = 32 * q + lane;                      // weight row inside the tile
    const bool gate = lane < 16;                      // GEMM1: gate lane (else the matching up lane)
    const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
    const float* xsc = ws_ptr<float>(p, p.L.x_scale);
    const float* xssc = p.share_uses_xq ? xsc : ws_ptr<float>(p, p.L.xs_scale);
    const float* s2 = ws_ptr<float>(p, p.L.s2);
    const int32_t* tk_of_row_g = ws_ptr<int32_t>(p, p.L.tk_of_row);
    float* hbuf = ws_ptr<float>(p, p.L.hbuf);
    int32_t* amax2 = ws_ptr<int32_t>(p, p.L.amax2);
    uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
    long acc_n = 0;
    for (long it = cta0; it < total && aligned; it += ncta) {
      const bool got = mbar_wait_bounded(&it_full[si], pi, abort_flag, status, site + 10);
      const BigItem x = get_item(items + 8 * si);
      // the previous item's epilogue is done with the token info, and every
      // thread has read the ring entry
      const bool failed = consumer_sync_or(!got || *abort_flag != 0);
      if (ctid == 0) mbar_arrive(&it_empty[si]);
      if (++si == SI) { si = 0; pi ^= 1u; }
      if (failed) break;
      const int tok0 = x.tb * TB;
      const int mblk = x.mblk;
      if (ctid < mblk) {
        const int r = x.row0 + tok0 + ctid;
        const int t = row_token[r];
        tok_row[ctid] = r;
        tok_tok[ctid] = t;
        if (G1) tok_scale[ctid] = x.e >= 0 ? xsc[p.xq_per_row ? r : t] : xssc[t];
        else if (p.fold_routing && x.e >= 0) tok_scale[ctid] = __fmul_rn(s2[r], p.scales[tk_of_row_g[r]]);
        else tok_scale[ctid] = s2[r];
      }
      consumer_sync();
      int acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0;
      const int n_chunks = (n_kb + CHUNK_KB - 1) / CHUNK_KB;
      bool ok = true;
      for (int c = 0; c < n_chunks && ok; ++c, ++acc_n) {
        const int buf = static_cast<int>(acc_n & 1);
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[buf], (acc_n >> 1) & 1, abort_flag, status, site + 8));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        // 16 columns at a time: columns past the block's rows are not read
        // (at 16 rows a block, 32-column loads read twice what it needs and
        // compete with the MMA for tensor memory)
        for (int cc = 0; cc < 4; ++cc) {
          if (64 * half + 16 * cc < mblk) {
            uint32_t v[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * TB + 64 * half + 16 * cc, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[16 * cc + j] += __float2int_rn(__uint_as_float(v[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      }
      const bool stop = consumer_sync_or(*abort_flag != 0);  // uniform over the epilogue threads
      // GEMM1: output column of this lane's gate / up pair; GEMM2: output column
      const int col = G1 ? x.jt * 64 + 16 * q + (lane & 15) : x.jt * BM + m;
      if (RAW) {
        const int ng = G1 ? (gate ? col : p.I + col) : col;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int tok = 64 * half + j;
          if (tok < mblk && ng < NW) raw[static_cast<size_t>(tok_row[tok]) * NW + ng] = acc[j];
        }
      } else if (G1) {
        // Dequant (§6.1: (float(acc) * w_scale) * x_scale) and SwiGLU.  Lane
        // l < 16 holds the gate row of output column `col` for the 64 tokens
        // of this half, lane l + 16 the matching up row; each lane takes 32
        // of the tokens (gate lanes the first 32, up lanes the last 32) and
        // trades the other 32 values with its partner.  h goes to the row's
        // first I floats; max |h| over this tile's columns is published per
        // row by an atomic maximum on the float bits (h >= 0 bits order as
        // integers), so that the requant needs one pass over h.
        const int ncol = gate ? col : p.I + col;
        const float ws = x.e >= 0 ? wscale_at(p.w1s, static_cast<size_t>(x.e) * NW + ncol, p.scale_dtype)
                                  : p.sw1s[ncol];
        // token slots of this half that hold rows of the block: gate lanes
        // take the first 32, up lanes the next ones, 8-token chunks past the
        // block's rows skipped (warp-uniform).  A half of at most 32 rows
        // goes to swiglu_half_tile, whose 16 or 8 slots a lane evaluate only
        // the rows it has (mid512 GEMM1 836 -> 783 us); the full-half case
        // keeps this code: written through the same template it compiled
        // 7 % slower at prefill.
        const int vt = mblk - 64 * half;
        if (vt > 32) {
          const int n_g = vt < 32 ? vt : 32;
          float hv[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (8 * c < n_g) {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int j = 8 * c + jj;
                // this lane's dequantised values of tokens j and 32 + j
                const float lo = __fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tok_scale[64 * half + j]);
                const float hi =
                    __fmul_rn(__fmul_rn(__int2float_rn(acc[32 + j]), ws), tok_scale[64 * half + 32 + j]);
                // gate lanes send gate(32 + j) and receive up(j); up lanes the reverse
                const float other = __shfl_xor_sync(0xffffffffu, gate ? hi : lo, 16);
                hv[j] = gate ? swiglu_1(lo, other) : swiglu_1(other, hi);
              }
            } else {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) hv[8 * c + jj] = 0.0f;
            }
          }
          const int tbase = 64 * half + (gate ? 0 : 32);  // token of hv[0]
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tok = tbase + j;
            if (tok < mblk) hbuf[static_cast<size_t>(tok_row[tok]) * (2 * p.I) + col] = hv[j];
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) hv[j] = fabsf(hv[j]);
          halfwarp_max_scatter(hv, lane & 15);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int tok = tbase + 2 * (lane & 15) + u;
            if (tok < mblk) atomicMax(amax2 + tok_row[tok], __float_as_int(hv[u]));
          }
        } else if (vt > 16) {
          swiglu_half_tile<16>(acc, tok_scale + 64 * half, tok_row + 64 * half, ws, gate, lane, vt, hbuf,
                               2 * static_cast<size_t>(p.I), col, amax2);
        } else if (vt > 0) {
          swiglu_half_tile<8>(acc, tok_scale + 64 * half, tok_row + 64 * half, ws, gate, lane, vt, hbuf,
                              2 * static_cast<size_t>(p.I), col, amax2);
        }
      } else {
        const bool valid_n = col < p.h;
        const float ws = !valid_n ? 0.0f
                         : x.e >= 0 ? wscale_at(p.w2s, static_cast<size_t>(x.e) * NW + col, p.scale_dtype)
                                    : p.sw2s[col];
        // A full half walks its 64 token slots; a shorter one skips the
        // 8-slot chunks past the block's rows (warp-uniform).  Measured
        // against one loop for both: mid512 GEMM2 428 -> 410 us, prefill
        // 530 -> 524 us (the chunked loop alone made prefill 13 us slower).
        if (64 * half + 64 <= mblk) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int tok = 64 * half + j;
            if (tok < mblk && valid_n) {
              const uint16_t b =
                  f32_to_act_bits(__fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tok_scale[tok]), p.act_fp16);
              if (x.e >= 0) y2[static_cast<size_t>(tok_row[tok]) * p.h + col] = b;
              else p.sout[static_cast<size_t>(tok_tok[tok]) * p.h + col] = b;
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if (64 * half + 8 * c < mblk) {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int j = 8 * c + jj;
                const int tok = 64 * half + j;
                if (tok < mblk && valid_n) {
                  const uint16_t b =
                      f32_to_act_bits(__fmul_rn(__fmul_rn(__int2float_rn(acc[j]), ws), tok_scale[tok]), p.act_fp16);
                  if (x.e >= 0) y2[static_cast<size_t>(tok_row[tok]) * p.h + col] = b;
                  else p.sout[static_cast<size_t>(tok_tok[tok]) * p.h + col] = b;
                }
              }
            }
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

// The big slots' tables (block prefix, first row, row count, expert, and a
// prefix of their row counts) staged in shared memory once per CTA, so that
// kernels working row by row find the slot of a row in a few shared-memory
// probes instead of a chain of dependent global loads.  Layout: 5 arrays of
// the slot table's stride (at most E + 1 big slots), i.e. big_slots_smem_bytes(E).
__host__ __device__ inline size_t big_slots_smem_bytes(int E) { return 5u * SlotTable::stride(E) * sizeof(int32_t); }

struct BigSlots {
  const int32_t* pre;   // first block of each slot (n + 1 entries)
  const int32_t* row0;
  const int32_t* rows;
  const int32_t* exp;
  const int32_t* rpre;  // rows of the slots before each slot (n + 1 entries: rpre[n] = all big rows)
  int n;
};

// Called by every thread of the block (blockDim a multiple of 32, <= 1024).
__device__ __forceinline__ BigSlots stage_big_slots(const FwdParams& p, const int32_t* slots, int32_t* t) {
  __shared__ int s_wsum[32];
  const int st = SlotTable::stride(p.E);
  const int32_t* s_exp = slots + SlotTable::kHeader;
  const int32_t* s_row0 = s_exp + st;
  const int32_t* s_rows = s_row0 + st;
  const int32_t* s_blk = s_rows + st;
  const int n = slots[SlotTable::kNumBig];
  for (int i = threadIdx.x; i <= n; i += blockDim.x) {
    t[i] = s_blk[i];
    if (i < n) {
      t[st + i] = s_row0[i];
      t[2 * st + i] = s_rows[i];
      t[3 * st + i] = s_exp[i];
    }
  }
  __syncthreads();
  // row prefix: each thread sums a contiguous chunk of slots, the chunk sums
  // are scanned across the block, then each thread writes its chunk's prefixes
  int32_t* rpre = t + 4 * st;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nwarp = blockDim.x >> 5;
  const int chunk = (n + blockDim.x - 1) / blockDim.x;
  const int c0 = min(n, tid * chunk), c1 = min(n, c0 + chunk);
  int sum = 0;
  for (int i = c0; i < c1; ++i) sum += t[2 * st + i];
  int x = sum;  // inclusive scan over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_wsum[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nwarp ? s_wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarp) s_wsum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  int run = x - sum + (wid > 0 ? s_wsum[wid - 1] : 0);
  for (int i = c0; i < c1; ++i) {
    rpre[i] = run;
    run += t[2 * st + i];
  }
  if (tid == 0) rpre[n] = s_wsum[nwarp - 1];
  __syncthreads();
  return BigSlots{t, t + st, t + 2 * st, t + 3 * st, rpre, n};
}

// slot of big row g (0 <= g < rpre[n], counting only real rows of big slots):
// the last slot whose first row index is <= g
__device__ __forceinline__ int big_row_slot(const BigSlots& t, int g) {
  int lo = 0, hi = t.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.rpre[mid] <= g) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Per-row quant of routed row r with per-expert smooth scales (the operator
// input table's smooth scales read as [E, h]): the same steps as the token
// quant (xs = x[t] * smooth[e], amax floored at 1e-4, m = 127 / amax,
// q = RNE(xs * m), scale = 1 / m), by one warp; rows of big blocks also get
// their f16 copy for the tensor-core GEMM1.
__device__ __forceinline__ void quant_routed_row(const FwdParams& p, int r, int lane, const int32_t* tk_of_row,
                                                 const int32_t* counts, int8_t* xq, float* xsc, __half* x1h) {
  const int f = tk_of_row[r];
  const int t = f / p.topk, e = p.ids[f];
  const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * p.h);
  const float4* sm = reinterpret_cast<const float4*>(p.smooth + static_cast<size_t>(e) * p.h);
  const int n8 = p.h >> 3;
  const bool fp16 = p.act_fp16 != 0;
  auto load8 = [&](int c, float (&v)[8]) {
    const uint4 w4 = xr[c];
    const float4 s0 = sm[2 * c], s1 = sm[2 * c + 1];
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
    const float s8[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      v[j] = __fmul_rn(act_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu), fp16), s8[j]);
  };
  float amax = 0.0f;
  for (int c = lane; c < n8; c += 32) {
    float v[8];
    load8(c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (amax < kAmaxEps) amax = kAmaxEps;
  const float m = __fdiv_rn(127.0f, amax);
  const bool big = counts[e] > p.small_rows;
  uint2* qrow = reinterpret_cast<uint2*>(xq + static_cast<size_t>(r) * p.h);
  uint4* hrow = reinterpret_cast<uint4*>(x1h + static_cast<size_t>(r) * p.h);
  for (int c = lane; c < n8; c += 32) {
    float v[8];
    load8(c, v);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      packed[j >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(f32_to_q(__fmul_rn(v[j], m)))) << ((j & 3) * 8);
    qrow[c] = make_uint2(packed[0], packed[1]);
    if (big) {
      uint4 lo16, hi16;
      int8x16_to_f16(make_uint4(packed[0], packed[1], 0u, 0u), lo16, hi16);
      hrow[c] = lo16;
    }
  }
  if (lane == 0) xsc[r] = __fdiv_rn(1.0f, m);
}

// f16 copies of the token codes of every row in a big block: the GEMM1
// operand that the tensor-memory path reads with TMA.  One warp per row of
// the big slots at a time, the rows spread evenly over the grid.
// With per-expert smooth scales the routed rows are quantised here first
// (every routed row, one warp each, their f16 copies included), and the slot
// loop then copies only the shared expert's rows.
__global__ void __launch_bounds__(256) expand_kernel(FwdParams p) {
  extern __shared__ int32_t ex_smem[];  // big_slots_smem_bytes(E)
  grid_dependency_wait();
  grid_launch_dependents();
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  if (p.xq_per_row) {
    const int R = slots[SlotTable::kRows];
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int r = gw; r < R; r += nw)
      quant_routed_row(p, r, lane, ws_ptr<int32_t>(p, p.L.tk_of_row), ws_ptr<int32_t>(p, p.L.counts),
                       ws_ptr<int8_t>(p, p.L.x_q), ws_ptr<float>(p, p.L.x_scale), ws_ptr<__half>(p, p.L.x1h));
  }
  const int total = slots[SlotTable::kBigBlocks];

  if (total == 0) return;
  const BigSlots tab = stage_big_slots(p, slots, ex_smem);
  {
    // clear the row maxima that the tensor-core GEMM1 epilogue raises
    int32_t* amax2 = ws_ptr<int32_t>(p, p.L.amax2);
    const int R = slots[SlotTable::kRows], S = slots[SlotTable::kSharedRows];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < R + S; i += gridDim.x * blockDim.x)
      amax2[i < R ? i : p.bs * p.topk + (i - R)] = 0;
  }
  const int32_t* row_token = ws_ptr<int32_t>(p, p.L.row_token);
  const int8_t* xq = ws_ptr<int8_t>(p, p.L.x_q);
  const int8_t* xsq = p.share_uses_xq ? xq : ws_ptr<int8_t>(p, p.L.xs_q);
  __half* x1h = ws_ptr<__half>(p, p.L.x1h);
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  // real rows of the big slots, spread evenly over the warps
  const int nreal = tab.rpre[tab.n];
  for (int g = gw; g < nreal; g += nw) {
    const int sl = big_row_slot(tab, g);
    if (p.xq_per_row && tab.exp[sl] >= 0) continue;  // quantised and copied above
    const int r = tab.row0[sl] + (g - tab.rpre[sl]);
    // lane l converts codes 8 c .. 8 c + 7 for c = l, l + 32, ...: every warp
    // store covers 512 contiguous bytes of the f16 row; streaming (evict-first)
    // stores, since GEMM1 reads these rows once, after the whole pass
    const uint2* src = reinterpret_cast<const uint2*>((tab.exp[sl] >= 0 ? xq : xsq) +
                                                      static_cast<size_t>(row_token[r]) * p.h);
    uint4* dst = reinterpret_cast<uint4*>(x1h + static_cast<size_t>(r) * p.h);
    const int n8 = p.h >> 3;
    for (int c0 = lane; c0 < n8; c0 += 4 * 32) {
      uint2 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + 32 * u < n8) v[u] = src[c0 + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
        if (c < n8) {
          uint4 lo16, hi16;
          int8x16_to_f16(make_uint4(v[u].x, v[u].y, 0u, 0u), lo16, hi16);
          __stcs(dst + c, lo16);
        }
      }
    }
  }
}

// Requant of the rows of big blocks (FusedDeepMoE analysis §7.2), one warp
// per row, one pass: the GEMM1 epilogue left the row's SwiGLU output h in
// the first I floats of its h row and max |h| in amax2; amax = max(that,
// 1e-4), s2 = amax * (1/127), q = RNE((h * 127) * (1/amax)) clamped to +-127.
// Writes the codes as f16 (the tensor-core GEMM2 operand, exact) and s2.
__device__ __forceinline__ void quant_store4(float4 v, float inv, int c, __half2* h2) {
  const float f[4] = {v.x, v.y, v.z, v.w};
  int8_t q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) q[j] = f32_to_q(__fmul_rn(__fmul_rn(f[j], 127.0f), inv));
  const __half2 a = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[1]));
  const __half2 b = __halves2half2(__int2half_rn(q[2]), __int2half_rn(q[3]));
  // one streaming 8-byte store of the four codes (GEMM2 reads them once)
  __stcs(reinterpret_cast<uint2*>(h2) + c,
         make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b)));
}

constexpr int kRqWarps = 8;          // rows in flight per CTA (one per warp)

__global__ void __launch_bounds__(kRqWarps * 32) requant_big_kernel(FwdParams p) {
  extern __shared__ int32_t rq_smem[];  // big_slots_smem_bytes(E)
  grid_dependency_wait();
  grid_launch_dependents();
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  const int total = slots[SlotTable::kBigBlocks];
  if (total == 0) return;
  const int I = p.I, n4 = I >> 2;
  const BigSlots tab = stage_big_slots(p, slots, rq_smem);
  const float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  const int32_t* amax2 = ws_ptr<int32_t>(p, p.L.amax2);
  __half* x2h = ws_ptr<__half>(p, p.L.x2h);
  float* s2 = ws_ptr<float>(p, p.L.s2);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gw = blockIdx.x * kRqWarps + wid;
  const int nw = gridDim.x * kRqWarps;
  // real rows of the big slots, spread evenly over the warps (row slots of
  // the 128-row blocks would leave most warps idle when blocks are short)
  const int nreal = tab.rpre[tab.n];
  for (int g = gw; g < nreal; g += nw) {
    const int sl = big_row_slot(tab, g);
    const int r = tab.row0[sl] + (g - tab.rpre[sl]);
    float amax = __int_as_float(amax2[r]);
    if (amax < 1e-4f) amax = 1e-4f;
    const float inv = __fdiv_rn(1.0f, amax);
    const float4* hr = reinterpret_cast<const float4*>(hbuf + static_cast<size_t>(r) * (2 * I));
    __half2* h2 = reinterpret_cast<__half2*>(x2h + static_cast<size_t>(r) * I);
    // four loads in flight per lane before any is used
    for (int c0 = lane; c0 < n4; c0 += 4 * 32) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + 32 * u < n4) v[u] = __ldcs(hr + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (c0 + 32 * u < n4) quant_store4(v[u], inv, c0 + 32 * u, h2);
    }
    if (lane == 0) s2[r] = __fmul_rn(amax, 1.0f / 127.0f);
  }
}

// Combine of every token (FusedDeepMoE analysis §4.2) when the forward has big
// blocks; otherwise the small-expert GEMM2 already combined every token.
// 4 CTAs of 256 threads resident per SM (at most 64 registers a thread), so
// the grid of 4 per SM runs as one wave: uncapped (72 registers) only 3 fit
// and a quarter of the grid ran as a second, partial wave.
__global__ void __launch_bounds__(256, 4) combine_kernel(FwdParams p) {
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

cudaError_t launch_requant_big(const FwdParams& p, cudaStream_t s, const LaunchOpts& o) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  const size_t smem = big_slots_smem_bytes(p.E);
  cudaLaunchConfig_t cfg = launch_config(dim3(p.num_ctas * 4), dim3(kRqWarps * 32), smem, s, attr, o);
  return cudaLaunchKernelEx(&cfg, requant_big_kernel, p);
}

cudaError_t launch_combine(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
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
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(requant_big_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(big_slots_smem_bytes(1024)));
}

cudaError_t launch_expand(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pdl_config(dim3(p.num_ctas * 4), dim3(256), big_slots_smem_bytes(p.E), s, attr);
  return cudaLaunchKernelEx(&cfg, expand_kernel, p);
}

cudaError_t launch_moe_gemm_big(const FwdParams& p, const TcMaps& maps, int mode, int32_t* raw_acc, int num_ctas,
                                cudaStream_t s, const LaunchOpts& o) {
  if (p.bs == 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(dim3(num_ctas), dim3(kBigThreads), SMEM_BYTES, s, attr, o);
  switch (mode) {
    case kGemm1SwiGLU: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm1SwiGLU>, maps, p, raw_acc);
    case kGemm2Bf16: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm2Bf16>, maps, p, raw_acc);
    case kGemm1Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm1Raw>, maps, p, raw_acc);
    case kGemm2Raw: return cudaLaunchKernelEx(&cfg, moe_gemm_big_kernel<kGemm2Raw>, maps, p, raw_acc);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
