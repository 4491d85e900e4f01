// Per-token dynamic INT8 quantisation of the activations and the split of
// the small experts' items over the GEMM CTAs: shared by the dispatch kernel
// and the one-launch decode kernel, so that both produce the same codes, the
// same scales and the same item ranges.
//
// Quant follows the FusedDeepMoE analysis §4.1 / §7.3 and the W8A8 contract
// of the DeepSeek-V4 decode case study: xs = x * smooth,
// amax = max(max|xs|, 1e-4), m = 127 / amax, q = RNE(xs * m) clamped to
// +-127, scale = 1 / m.  Every fp32 operation is an explicit round-to-nearest
// intrinsic so no contraction can change a code.
#pragma once

#include "device_prims.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kQuantThreads = 256;   // threads that quantise one row together
constexpr float kAmaxEps = 1e-4f;    // floor of a row's amax (quant and requant)

// max over the 256 threads of one quant group (named barrier 1 + group)
__device__ __forceinline__ float group_max(float v, float* s_red, int group) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int gt = threadIdx.x & (kQuantThreads - 1);
  const int lane = gt & 31, warp = gt >> 5;
  if (lane == 0) s_red[warp] = v;
  named_barrier_sync(1 + group, kQuantThreads);
  float r = s_red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) r = fmaxf(r, s_red[w]);
  named_barrier_sync(1 + group, kQuantThreads);
  return r;
}

// Quantise one bf16 (fp16 when `fp16`) row (h multiple of 64) with optional
// smooth scales, by the 256 threads of one group.
__device__ void quant_row(const uint16_t* __restrict__ x, bool fp16, const float* __restrict__ smooth, int h,
                          int8_t* __restrict__ q, float* __restrict__ scale_out, float* s_red, int group) {
  const int gt = threadIdx.x & (kQuantThreads - 1);
  const int n8 = h >> 3;
  float amax = 0.0f;
  for (int i = gt; i < n8; i += kQuantThreads) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float f = act_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu), fp16);
      if (smooth) f = __fmul_rn(f, smooth[i * 8 + j]);
      amax = fmaxf(amax, fabsf(f));
    }
  }
  amax = group_max(amax, s_red, group);
  if (amax < kAmaxEps) amax = kAmaxEps;
  const float m = __fdiv_rn(127.0f, amax);
  for (int i = gt; i < n8; i += kQuantThreads) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float f = act_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu), fp16);
      if (smooth) f = __fmul_rn(f, smooth[i * 8 + j]);
      const uint32_t b = static_cast<uint8_t>(f32_to_q(__fmul_rn(f, m)));
      packed[j >> 2] |= b << ((j & 3) * 8);
    }
    reinterpret_cast<uint2*>(q)[i] = make_uint2(packed[0], packed[1]);
  }
  if (gt == 0) *scale_out = __fdiv_rn(1.0f, m);
}

// Quant of token t by one 256-thread group.  Tokens that no expert row will
// combine into get their zero output rows here: inactive tokens (output and
// share_output) and active tokens whose ids are all outside [0, E) (output).
__device__ void quant_token(const FwdParams& p, int t, float* s_red, int group) {
  const int gt = threadIdx.x & (kQuantThreads - 1);
  const bool act = (p.mask == nullptr) || (p.mask[t] != 0);
  int nvalid = 0;
  if (act)
    for (int k = 0; k < p.topk; ++k) {
      const int id = p.ids[t * p.topk + k];
      nvalid += (id >= 0 && id < p.E);
    }
  const int n8 = p.h >> 3;
  if (nvalid == 0) {
    uint4* out = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * p.h);
    for (int i = gt; i < n8; i += kQuantThreads) out[i] = make_uint4(0, 0, 0, 0);
  }
  if (!act) {
    if (p.has_shared) {
      uint4* so = reinterpret_cast<uint4*>(p.sout + static_cast<size_t>(t) * p.h);
      for (int i = gt; i < n8; i += kQuantThreads) so[i] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const uint16_t* xr = p.x + static_cast<size_t>(t) * p.h;
  // per-expert smooth scales: the routed rows are quantised one by one after
  // the dispatch (expand kernel); only the shared expert's quant runs here
  if (!p.xq_per_row)
    quant_row(xr, p.act_fp16, p.smooth, p.h, ws_ptr<int8_t>(p, p.L.x_q) + static_cast<size_t>(t) * p.h,
              ws_ptr<float>(p, p.L.x_scale) + t, s_red, group);
  if (p.has_shared && !p.share_uses_xq) {
    quant_row(xr, p.act_fp16, p.ssmooth, p.h, ws_ptr<int8_t>(p, p.L.xs_q) + static_cast<size_t>(t) * p.h,
              ws_ptr<float>(p, p.L.xs_scale) + t, s_red, group);
  }
}

// The same quant of one row by one warp (no block barrier): each lane takes
// every 32nd group of 8 values; the row maximum is a warp reduction, so the
// codes and the scale are the ones quant_row computes.
__device__ void quant_row_warp(const uint16_t* __restrict__ x, bool fp16, const float* __restrict__ smooth, int h,
                               int8_t* __restrict__ q, float* __restrict__ scale_out) {
  const int lane = threadIdx.x & 31;
  const int n8 = h >> 3;
  float amax = 0.0f;
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float f = act_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu), fp16);
      if (smooth) f = __fmul_rn(f, smooth[i * 8 + j]);
      amax = fmaxf(amax, fabsf(f));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (amax < kAmaxEps) amax = kAmaxEps;
  const float m = __fdiv_rn(127.0f, amax);
  for (int i = lane; i < n8; i += 32) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float f = act_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu), fp16);
      if (smooth) f = __fmul_rn(f, smooth[i * 8 + j]);
      const uint32_t b = static_cast<uint8_t>(f32_to_q(__fmul_rn(f, m)));
      packed[j >> 2] |= b << ((j & 3) * 8);
    }
    reinterpret_cast<uint2*>(q)[i] = make_uint2(packed[0], packed[1]);
  }
  if (lane == 0) *scale_out = __fdiv_rn(1.0f, m);
}

// quant_token by one warp.
__device__ void quant_token_warp(const FwdParams& p, int t) {
  const int lane = threadIdx.x & 31;
  const bool act = (p.mask == nullptr) || (p.mask[t] != 0);
  int nvalid = 0;
  if (act)
    for (int k = 0; k < p.topk; ++k) {
      const int id = p.ids[t * p.topk + k];
      nvalid += (id >= 0 && id < p.E);
    }
  const int n8 = p.h >> 3;
  if (nvalid == 0) {
    uint4* out = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * p.h);
    for (int i = lane; i < n8; i += 32) out[i] = make_uint4(0, 0, 0, 0);
  }
  if (!act) {
    if (p.has_shared) {
      uint4* so = reinterpret_cast<uint4*>(p.sout + static_cast<size_t>(t) * p.h);
      for (int i = lane; i < n8; i += 32) so[i] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const uint16_t* xr = p.x + static_cast<size_t>(t) * p.h;
  if (!p.xq_per_row)
    quant_row_warp(xr, p.act_fp16, p.smooth, p.h, ws_ptr<int8_t>(p, p.L.x_q) + static_cast<size_t>(t) * p.h,
                   ws_ptr<float>(p, p.L.x_scale) + t);
  if (p.has_shared && !p.share_uses_xq)
    quant_row_warp(xr, p.act_fp16, p.ssmooth, p.h, ws_ptr<int8_t>(p, p.L.xs_q) + static_cast<size_t>(t) * p.h,
                   ws_ptr<float>(p, p.L.xs_scale) + t);
}

// First item of CTA b (of G) in the small phase of one GEMM.  The small slots'
// items are split by cost: an item of an expert with m rows streams the same
// weight bytes as any other but does m dot products per weight, so it counts
// 12 + m; wp[i] is the exclusive prefix of those costs over the ns slots
// (wp[ns] the total) and J the items per slot.  CTA b starts at the first
// item whose cumulative cost reaches b * q + min(b, r), q, r = total divmod
// G; CTA G "starts" at ns * J.  32-bit throughout
// (J * wp[ns] <= 1024 * 1025 * 20 < 2^31).
__device__ __forceinline__ int small_item_start(const int32_t* wp, int ns, int J, int G, int b) {
  if (b == G || ns == 0) return ns * J;
  const int total = J * wp[ns];
  const int q = total / G, r = total - q * G;
  const int target = b * q + (b < r ? b : r);
  int lo = 0, hi = ns - 1;  // last slot whose first item starts at or before target
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (J * wp[mid] <= target) lo = mid;
    else hi = mid - 1;
  }
  const int cost = wp[lo + 1] - wp[lo];
  const int k = (target - J * wp[lo] + cost - 1) / cost;
  return lo * J + (k < J ? k : J);
}

}  // namespace
}  // namespace moe
