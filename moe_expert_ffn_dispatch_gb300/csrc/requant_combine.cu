// Per-row requantisation of the SwiGLU output and the top-k combine.
//
// Requant follows the FusedDeepMoE analysis §7.2 (BlockQuant): amax over the
// row (floored at 1e-4 as the W8A8 contract of the DeepSeek-V4 decode case
// study floors every dynamic quant), scale = amax * (1/127),
// q = RNE((h * 127) * (1 / amax)) clamped to +-127.
//
// Combine follows §4.2 (LocalWindowCopy): per token an fp32 sum starting at
// 0, for k ascending add float(row) * expert_scale (multiply and add rounded
// separately), one final RNE cast to bf16.  Inactive tokens get zero rows in
// output and share_output.
#include "device_prims.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRequantThreads = 256;
constexpr int kCombineThreads = 256;
constexpr float kAmaxEps = 1e-4f;
constexpr float kInv127 = 1.0f / 127.0f;  // the fp32 nearest to 1/127

__global__ void __launch_bounds__(kRequantThreads) requant_kernel(FwdParams p) {
  __shared__ float s_red[33];
  const int32_t* slots = ws_ptr<int32_t>(p, p.L.slots);
  const int R = slots[SlotTable::kRows], S = slots[SlotTable::kSharedRows];
  const int I = p.I;
  const float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
  float* s2 = ws_ptr<float>(p, p.L.s2);
  const int n4 = I >> 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = blockIdx.x; i < R + S; i += gridDim.x) {
    const int r = i < R ? i : p.bs * p.topk + (i - R);
    const float4* hr = reinterpret_cast<const float4*>(hbuf + static_cast<size_t>(r) * I);
    float amax = 0.0f;
    for (int c = threadIdx.x; c < n4; c += kRequantThreads) {
      const float4 v = hr[c];
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    if (warp == 0) {
      float m = lane < kRequantThreads / 32 ? s_red[lane] : 0.0f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) s_red[32] = m;
    }
    __syncthreads();
    amax = s_red[32];
    __syncthreads();
    if (amax < kAmaxEps) amax = kAmaxEps;
    const float inv = __fdiv_rn(1.0f, amax);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(x2 + static_cast<size_t>(r) * I);
    for (int c = threadIdx.x; c < n4; c += kRequantThreads) {
      const float4 v = hr[c];
      const float f[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t b = static_cast<uint8_t>(f32_to_q(__fmul_rn(__fmul_rn(f[j], 127.0f), inv)));
        packed |= b << (8 * j);
      }
      q4[c] = packed;
    }
    if (threadIdx.x == 0) s2[r] = __fmul_rn(amax, kInv127);
  }
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(FwdParams p) {
  __shared__ int s_row[16];
  __shared__ float s_scale[16];
  const int t = blockIdx.x;
  const int h = p.h, K = p.topk;
  const int n8 = h >> 3;
  uint4* out = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * h);
  const bool act = (p.mask == nullptr) || (p.mask[t] != 0);
  if (!act) {
    for (int i = threadIdx.x; i < n8; i += kCombineThreads) out[i] = make_uint4(0, 0, 0, 0);
    if (p.has_shared) {
      uint4* so = reinterpret_cast<uint4*>(p.sout + static_cast<size_t>(t) * h);
      for (int i = threadIdx.x; i < n8; i += kCombineThreads) so[i] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of);
  if (threadIdx.x < K) {
    s_row[threadIdx.x] = row_of[t * K + threadIdx.x];
    s_scale[threadIdx.x] = p.scales[t * K + threadIdx.x];
  }
  __syncthreads();
  const uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
  for (int i = threadIdx.x; i < n8; i += kCombineThreads) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int r = s_row[k];
      if (r < 0) continue;
      const float sc = s_scale[k];
      const uint4 v = reinterpret_cast<const uint4*>(y2 + static_cast<size_t>(r) * h)[i];
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

}  // namespace

cudaError_t launch_requant(const FwdParams& p, int num_ctas, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  requant_kernel<<<num_ctas, kRequantThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const FwdParams& p, cudaStream_t s) {
  if (p.bs == 0) return cudaSuccess;
  combine_kernel<<<p.bs, kCombineThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
