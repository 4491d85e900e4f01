// Peak-rate probe of this GPU for the block's roofline denominators: the
// exact-integer contraction rates that the two GEMM engines can reach and a
// read-only HBM stream (the measured copy rate and cuBLAS bf16 rate come
// from elsewhere).  A standalone program, built and run by `bench.py --peaks`;
// it prints one JSON object.
//
//   dp4a              int8 dot products of 4 (the small-expert engine)
//   mma_sync_s8       legacy warp-level int8 tensor MMA, m16n8k32
//   tcgen05_f16_ss    tcgen05 kind::f16, M128 x N128 x K16, A and B in shared memory
//   tcgen05_f16_ts    the same with A in tensor memory (the big-expert engine's form)
//   hbm_read          a streaming read of 4 GiB (16-byte loads, evict-first)
//   exact_k1024       all-127 x all-127 codes as f16 over K = 1024 with fp32
//                     accumulation in tensor memory: the largest partial sum
//                     (127 * 127 * 1024 < 2^24) must come back exactly
//
// Every kernel is timed with CUDA events after a warm-up launch.  The one
// wait (for the MMAs' commit) gives up after a 2 s budget and sets an error
// flag; nothing traps.
#include <cstdio>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_prims.cuh"

using namespace moe;

#define CK(x)                                                                              \
  do {                                                                                     \
    cudaError_t e_ = (x);                                                                  \
    if (e_ != cudaSuccess) {                                                               \
      std::printf("{\"error\": \"%s at line %d\"}\n", cudaGetErrorString(e_), __LINE__);   \
      return 1;                                                                            \
    }                                                                                      \
  } while (0)

namespace {

__global__ void dp4a_kernel(int iters, int* sink) {
  int a[4] = {static_cast<int>(threadIdx.x), static_cast<int>(threadIdx.x) * 3, 7, 11};
  const int b = 0x01020304 ^ static_cast<int>(blockIdx.x);
  int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = __dp4a(a[j & 3], b + j, c[j]);
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += c[j];
  if (s == 0x7fffffff) *sink = s;
}

__global__ void mma_s8_kernel(int iters, int* sink) {
  const uint32_t a = threadIdx.x, b = blockIdx.x;
  int acc[8][4] = {};
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) mma_s8_16832(acc[j], a, a + 1, a + 2, a + 3, b, b + j);
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
  if (s == 0x7fffffff) *sink = s;
}

// Streaming read: each thread sums 16-byte words of its grid-stride range.
__global__ void hbm_read_kernel(const uint4* src, size_t n, uint32_t* sink) {
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldcs(src + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  if (acc == 0x9e3779b9u) *sink = acc;
}

constexpr int kTile = 128 * 64 * 2;  // [128][64] f16, 128-byte swizzle: 16 KB

// element (r, k) of a [128][64] f16 tile in the K-major 128-byte swizzle
__device__ __forceinline__ int sw128(int r, int k) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) + (k & 7) * 2;
}

// One CTA of 128 threads per SM: A and B tiles ([128][64] f16 each) filled
// with the value `val`, then `reps` rounds of four K16 MMAs (M128 x N128) into
// one accumulator, A from shared memory (ts = false) or tensor memory (ts =
// true), committed to one mbarrier at the end.  Thread t then reads lane t's
// 128 accumulator columns; out[blockIdx][t] = the first column's value (the
// exactness check reads it), err set if a wait ran out.
template <bool TS>
__global__ void __launch_bounds__(128, 1) umma_kernel(float val, long reps, float* out, int* err) {
  extern __shared__ __align__(1024) char smem[];
  char* a = smem;
  char* b = smem + kTile;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * kTile);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const __half hv = __float2half_rn(val);
  for (int i = tid; i < 128 * 64; i += 128) {
    *reinterpret_cast<__half*>(a + sw128(i >> 6, i & 63)) = hv;
    *reinterpret_cast<__half*>(b + sw128(i >> 6, i & 63)) = hv;
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(slot, 256);  // 128 accumulator columns + 32 columns of A
  fence_proxy_async_smem();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const uint32_t a_tmem = tmem + 128;
  if (TS) {
    // A (lane = row, 32 columns of f16 pairs = K 64) into tensor memory
    uint32_t v[32];
    const uint32_t pair = static_cast<uint32_t>(__half_as_ushort(hv)) * 0x10001u;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = pair;
    tmem_st32(a_tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
    tmem_st_wait();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t idesc = umma_idesc_f16(128, 128);
  if (tid == 0) {
    const uint64_t ad = umma_desc_sw128(smem_u32(a)), bd = umma_desc_sw128(smem_u32(b));
    for (long r = 0; r < reps; ++r) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t acc = (r > 0 || ks > 0) ? 1u : 0u;
        if (TS) umma_f16_ts(tmem, a_tmem + 8 * ks, bd + 2 * ks, idesc, acc);
        else umma_f16(tmem, ad + 2 * ks, bd + 2 * ks, idesc, acc);
      }
    }
    umma_commit(bar);
  }
  __syncwarp();
  const bool ok = mbar_wait_bounded(bar, 0, nullptr, nullptr, 0);  // 2 s budget, then give up
  if (!ok && tid == 0) atomicExch(err, 1);
  tc_fence_after();
  uint32_t v[16];
  tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
  out[blockIdx.x * 128 + tid] = __uint_as_float(v[0]);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <typename F>
float time_ms(F launch) {
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  launch();  // warm-up
  cudaDeviceSynchronize();
  cudaEventRecord(e0);
  launch();
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  float ms = 0.0f;
  cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return ms;
}

}  // namespace

int main() {
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, dev));
  int* d_sink = nullptr;
  int* d_err = nullptr;
  float* d_out = nullptr;
  CK(cudaMalloc(&d_sink, 64));
  CK(cudaMalloc(&d_err, 4));
  CK(cudaMalloc(&d_out, sizeof(float) * sms * 128));
  CK(cudaMemset(d_err, 0, 4));

  // dp4a: 8 per iteration per thread, 4 MACs each
  const int it_dp4a = 1 << 16, blocks = sms * 8, threads = 256;
  const float ms_dp4a = time_ms([&] { dp4a_kernel<<<blocks, threads>>>(it_dp4a, d_sink); });
  CK(cudaGetLastError());
  const double ops_dp4a = 2.0 * 4 * 8 * static_cast<double>(it_dp4a) * blocks * threads;

  // mma.sync s8 m16n8k32: 8 per iteration per warp, 16*8*32 MACs each
  const int it_mma = 1 << 14;
  const float ms_mma = time_ms([&] { mma_s8_kernel<<<blocks, threads>>>(it_mma, d_sink); });
  CK(cudaGetLastError());
  const double ops_mma = 2.0 * 16 * 8 * 32 * 8 * static_cast<double>(it_mma) * blocks * (threads / 32);

  // tcgen05 kind::f16 M128 N128 K16, one CTA per SM
  const int smem = 2 * kTile + 64;
  CK(cudaFuncSetAttribute(umma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  CK(cudaFuncSetAttribute(umma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  const long reps = 1 << 15;
  const float ms_ss = time_ms([&] { umma_kernel<false><<<sms, 128, smem>>>(1.0f, reps, d_out, d_err); });
  CK(cudaGetLastError());
  const float ms_ts = time_ms([&] { umma_kernel<true><<<sms, 128, smem>>>(1.0f, reps, d_out, d_err); });
  CK(cudaGetLastError());
  const double ops_umma = 2.0 * 128 * 128 * 16 * 4 * static_cast<double>(reps) * sms;

  // exactness: 127 * 127 over K = 1024 (16 rounds of K 64), both operand forms
  float got_ss = 0.0f, got_ts = 0.0f;
  umma_kernel<false><<<1, 128, smem>>>(127.0f, 16, d_out, d_err);
  CK(cudaMemcpy(&got_ss, d_out, 4, cudaMemcpyDeviceToHost));
  umma_kernel<true><<<1, 128, smem>>>(127.0f, 16, d_out, d_err);
  CK(cudaMemcpy(&got_ts, d_out + 0, 4, cudaMemcpyDeviceToHost));
  const double want = 127.0 * 127.0 * 1024.0;

  // read-only HBM stream over 4 GiB
  const size_t bytes = size_t(4) << 30;
  uint4* buf = nullptr;
  CK(cudaMalloc(&buf, bytes));
  CK(cudaMemset(buf, 1, bytes));
  const float ms_rd = time_ms([&] {
    hbm_read_kernel<<<sms * 8, 512>>>(buf, bytes / 16, reinterpret_cast<uint32_t*>(d_sink));
  });
  CK(cudaGetLastError());
  int err = 0;
  CK(cudaMemcpy(&err, d_err, 4, cudaMemcpyDeviceToHost));

  std::printf(
      "{\"device\": \"%s\", \"sms\": %d, \"dp4a_tops\": %.1f, \"mma_sync_s8_tops\": %.1f, "
      "\"tcgen05_f16_ss_tflops\": %.1f, \"tcgen05_f16_ts_tflops\": %.1f, \"hbm_read_gbs\": %.1f, "
      "\"exact_k1024\": %s, \"exact_k1024_values\": [%.1f, %.1f, %.1f], \"wait_error\": %d}\n",
      prop.name, sms, ops_dp4a / ms_dp4a / 1e9, ops_mma / ms_mma / 1e9, ops_umma / ms_ss / 1e9,
      ops_umma / ms_ts / 1e9, bytes / ms_rd / 1e6,
      (got_ss == want && got_ts == want) ? "true" : "false", got_ss, got_ts, want, err);
  cudaFree(buf);
  cudaFree(d_out);
  cudaFree(d_err);
  cudaFree(d_sink);
  return err != 0;
}
