// Epilogue operations shared by the small- and big-expert GEMM kernels:
// per-row requant (FusedDeepMoE analysis §7.2 BlockQuant) and the top-k
// combine (§4.2 LocalWindowCopy), run by the CTA that completes a row block
// (GEMM1) or a token (GEMM2) last, plus the counters that decide it.  Executed
// by the 256 "consumer" threads of a CTA (named barrier 1).
#pragma once

#include <cuda_fp16.h>

#include "device_prims.cuh"
#include "moe_internal.h"
#include "quant_ops.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr float kInv127 = 1.0f / 127.0f;  // the fp32 nearest to 1/127

__device__ __forceinline__ void consumer_sync() { named_barrier_sync(1, kConsumers); }
__device__ __forceinline__ bool consumer_sync_or(bool pred) { return named_barrier_or(1, kConsumers, pred); }

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------ epilogue ops
// Requant of rows [r0, r0 + n) of h into x2 / s2, by the consumer threads.
// h was written by other CTAs in this launch: read it through L2 (ld.cg).
// Rows of big blocks also get their codes as f16 (x2h), the operand of the
// tensor-core GEMM2.
__device__ void requant_rows(const FwdParams& p, int r0, int n, float* s_red, int ctid, bool write_f16) {
  const int I = p.I, n4 = I >> 2;
  const float* hbuf = ws_ptr<float>(p, p.L.hbuf);
  int8_t* x2 = ws_ptr<int8_t>(p, p.L.x2);
  __half* x2h = ws_ptr<__half>(p, p.L.x2h);
  float* s2 = ws_ptr<float>(p, p.L.s2);
  const int lane = ctid & 31, warp = ctid >> 5;
  for (int i = 0; i < n; ++i) {
    const int r = r0 + i;
    const float4* hr = reinterpret_cast<const float4*>(hbuf + static_cast<size_t>(r) * (2 * I));
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
      int8_t q[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        q[j] = f32_to_q(__fmul_rn(__fmul_rn(f[j], 127.0f), inv));
        packed |= static_cast<uint32_t>(static_cast<uint8_t>(q[j])) << (8 * j);
      }
      q4[c] = packed;
      if (write_f16) {
        __half2* dst = reinterpret_cast<__half2*>(x2h + static_cast<size_t>(r) * I) + 2 * c;
        dst[0] = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[1]));
        dst[1] = __halves2half2(__int2half_rn(q[2]), __int2half_rn(q[3]));
      }
    }
    if (ctid == 0) s2[r] = __fmul_rn(amax, kInv127);
  }
}

// Combine of token t, by the consumer threads (y2 through L2, evict-first:
// each row is read once): each thread owns 8 output columns at a time, issues
// the loads of up to 8 expert rows before using any, and adds the terms in
// ascending k (fp32, each product and each sum rounded once, from 0.0f).
__device__ void combine_token(const FwdParams& p, int t, int ctid) {
  const int h = p.h, K = p.topk, n8 = h >> 3;
  const int32_t* row_of = ws_ptr<int32_t>(p, p.L.row_of) + static_cast<size_t>(t) * K;
  const float* scales = p.scales + static_cast<size_t>(t) * K;
  const uint16_t* y2 = ws_ptr<uint16_t>(p, p.L.y2);
  uint4* out = reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * h);
  for (int i = ctid; i < n8; i += kConsumers) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 8) {
      int r[8];
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        r[u] = (k0 + u < K) ? row_of[k0 + u] : -1;
        if (r[u] >= 0) v[u] = __ldcs(reinterpret_cast<const uint4*>(y2 + static_cast<size_t>(r[u]) * h) + i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (r[u] < 0) continue;
        const float sc = scales[k0 + u];
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float f = act_bits_to_f32(static_cast<uint16_t>((w[j >> 1] >> ((j & 1) * 16)) & 0xFFFFu), p.act_fp16);
          // folded mode: the rows already carry their routing weight
          acc[j] = __fadd_rn(acc[j], p.fold_routing ? f : __fmul_rn(f, sc));
        }
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = static_cast<uint32_t>(f32_to_act_bits(acc[2 * j], p.act_fp16)) |
             (static_cast<uint32_t>(f32_to_act_bits(acc[2 * j + 1], p.act_fp16)) << 16);
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// After a CTA's outputs for a row block are written (every writer fenced,
// then a consumer barrier): GEMM1 adds the tiles it finished to the block's
// counter; the CTA that completes the block requantises its rows.
// `done` tiles of the block were finished by this CTA since its last report.
__device__ void gemm1_item_done(const FwdParams& p, int blk, int tiles, int done, int r0, int n, int* s_flag,
                                float* s_red, int ctid, bool big) {
  if (ctid == 0) {
    const int old = atomicAdd(ws_ptr<int32_t>(p, p.L.blk_ticket) + blk, done);
    *s_flag = (old + done == tiles);
  }
  consumer_sync();
  if (*s_flag) {
    __threadfence();
    requant_rows(p, r0, n, s_red, ctid, big);
    // the block's x2 / s2 are complete: one more count on its ticket
    // (tiles + 1) tells a GEMM2 running in the same launch that it may read them
    consumer_sync();
    if (ctid == 0) {
      __threadfence();
      atomicAdd(ws_ptr<int32_t>(p, p.L.blk_ticket) + blk, 1);
    }
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

}  // namespace
}  // namespace moe
