// Device primitives for the sm_103a kernels: mbarrier full/empty rings fed by
// bulk async copies (the producer/consumer FIFO of the Mega-MoE pipeline
// analysis, §4.1-4.3), warp-level int8 tensor-core MMA, and bounded waits.
//
// Every spin in this library is bounded: a wait that exceeds its budget
// records an error in the workspace status words and returns false, and the
// caller unwinds.  Nothing traps.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {

// bounded wait budget in nanoseconds of %globaltimer
constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: has phase `parity` of `bar` completed?  (acquire)
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Record a wait that gave up: flag + site, first writer wins the site.
__device__ __forceinline__ void report_timeout(int32_t* status, int site) {
  if (status) {
    atomicOr(status + kStErrorFlags, kErrWaitTimeout);
    atomicCAS(status + kStErrorSite, 0, site);
  }
}

// Wait for phase `parity` of `bar`; false after the time budget (or as soon
// as *abort is nonzero, so that sibling warps unwind together).  Only waiters
// with `raise_abort` publish their own timeout through *abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  int32_t* status, int site, bool raise_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 255u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > kWaitBudgetNs) {
        report_timeout(status, site);
        if (abort && raise_abort) *abort = 1;
        return false;
      }
    }
  }
}

// L2 policies for the bulk copies: weights stream through once, activations
// are re-read by every N-tile of an expert.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk async copy global -> shared, completing bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}

// D(16x8, s32) += A(16x32, s8, row) * B(32x8, s8, col)
__device__ __forceinline__ void mma_s8_16832(int32_t* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible; then let the next grid launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Named barrier that also returns the OR of a predicate over its threads,
// so that a decision taken after it (stop on an error) is uniform.
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// Named barrier that also returns how many of its threads had `pred` set.
__device__ __forceinline__ int named_barrier_count(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.popc.u32 %0, %2, %3, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return static_cast<int>(r);
}

// ------------------------------------------------------------ TMA tensor
// 2-D tiled bulk tensor copy global -> shared, completing bytes on `bar`.
// `tmap` is the address of a CUtensorMap kernel parameter (__grid_constant__).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// generic-proxy shared-memory writes -> visible to the async proxy (tensor core, TMA)
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// global-memory data written by generic stores (of other CTAs, acquired
// through a flag) -> visible to this thread's later bulk copies
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Spin until *flag >= want (acquire), with the same bound as the mbarrier
// waits: false if the budget ran out (reported, abort raised) or another
// role raised abort.
__device__ __forceinline__ bool spin_until_ge(const int32_t* flag, int want, volatile int* abort, int32_t* status,
                                              int site) {
  if (ld_acquire_gpu(flag) >= want) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (ld_acquire_gpu(flag) >= want) return true;
    __nanosleep(64);
    if ((++n & 255u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > kWaitBudgetNs) {
        report_timeout(status, site);
        if (abort) *abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Grid-wide barrier of a launch whose CTAs are all resident (one per SM),
// called by one full warp of each CTA after a CTA barrier that orders the
// CTA's other writes before it.  It needs no initial state: tags[0] (the
// generation) and tags[1 .. G-1] may hold anything when the launch starts.
// Every CTA reads the generation g; CTA b > 0 then writes its arrival tag
// (g + 1) ^ salt to tags[b] and waits for the generation to change; CTA 0
// waits until every tag reads (g + 1) ^ salt and then sets the generation to
// g + 1.  The generation changes only after every CTA has arrived, so all
// read the same g; the salt (a random constant of the caller) keeps any
// earlier content of the words from passing for an arrival, and tags of an
// earlier barrier carry an older generation.  Ordering: the tag and the new
// generation are release stores (after the CTA barrier, and after CTA 0's
// warp barrier), the generation is polled with acquire loads, and CTA 0's
// lanes fence after the relaxed loads that saw the tags.  Bounded: a CTA
// whose wait runs out reports it in the status and adds 2 to the
// generation, so that the waiting CTAs stop (they see neither g nor g + 1)
// and no tag written here matches a later barrier.  Returns false (on every
// lane) if this CTA's barrier failed.
__device__ __forceinline__ bool grid_barrier_tagged(uint64_t* tags, uint64_t salt, int G, int32_t* status,
                                                    int site) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  const uint64_t g = __shfl_sync(0xffffffffu, lane == 0 ? ld_relaxed_gpu_u64(tags) : 0ull, 0);
  const uint64_t want = (g + 1) ^ salt;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  bool ok = true;
  if (blockIdx.x == 0) {
    while (true) {
      // every tag of a pass loaded before any is compared: one round trip a pass
      bool all = true;
      for (int base = 1; base < G; base += 8 * 32) {
        uint64_t v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int b = base + lane + 32 * j;
          v[j] = b < G ? ld_relaxed_gpu_u64(tags + b) : want;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) all &= v[j] == want;
      }
      if (__all_sync(0xffffffffu, all)) break;
      if ((++n & 63u) == 0 && __shfl_sync(0xffffffffu, global_timer_ns() - t0 > kWaitBudgetNs, 0)) {
        ok = false;
        break;
      }
    }
    fence_acq_rel_gpu();  // acquire: what the CTAs wrote before their tags
    __syncwarp();
    if (ok && lane == 0) st_release_gpu_u64(tags, g + 1);
  } else {
    uint64_t v = g;
    if (lane == 0) {
      st_release_gpu_u64(tags + blockIdx.x, want);
      while ((v = ld_acquire_gpu_u64(tags)) == g) {
        if ((++n & 255u) == 0 && global_timer_ns() - t0 > kWaitBudgetNs) break;
      }
    }
    v = __shfl_sync(0xffffffffu, v, 0);
    __syncwarp();
    ok = v == g + 1;
  }
  if (!ok && lane == 0) {
    atomicAdd(reinterpret_cast<unsigned long long*>(tags), 2ull);
    report_timeout(status, site);
  }
  return ok;
}

// Logical index of this CTA in a launch whose CTAs take their work in
// arrival order: the i-th CTA to get here gets i.  *counter is zero before
// the launch; the last CTA to arrive (every CTA of the grid calls this once)
// puts it back to zero.  Called by every thread of the CTA after the
// launch's grid-dependency wait; s_lid: one int of shared memory.
__device__ __forceinline__ int arrival_index(int32_t* counter, int* s_lid) {
  if (threadIdx.x == 0) {
    const int i = atomicAdd(counter, 1);
    if (i == static_cast<int>(gridDim.x) - 1) atomicExch(counter, 0);
    *s_lid = i;
  }
  __syncthreads();
  return *s_lid;
}

// true in exactly one lane of the (converged) warp: lets a warp run a loop
// with warp-uniform values while a single lane issues TMA / tcgen05 work
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand tile in the 128-byte swizzle layout: rows of 128 bytes,
// 8-row atoms of 1024 bytes (stride between atoms = 1024).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused by swizzled K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: f16 A and B (K-major), f32 accumulator, M x N
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A(smem desc) * B(smem desc)^T, issued by one thread
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A(tmem) * B(smem desc)^T: A as M lanes x K/2 columns of packed
// f16 pairs (lane = row, lower K in the low half), issued by one thread
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes (one lane per
// thread), then wait until the stores are done
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// arrive on `bar` once every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes (one lane per thread)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// fp32 -> int8 code, round half to even, clamped to [-127, 127]
__device__ __forceinline__ int8_t f32_to_q(float v) {
  int r = __float2int_rn(v);
  r = r > 127 ? 127 : (r < -127 ? -127 : r);
  return static_cast<int8_t>(r);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// fp32 -> bf16 bits, round half to even (inputs are finite)
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// Activation elements (x, y2, the outputs) are bf16, or fp16 when `fp16`.
__device__ __forceinline__ float act_bits_to_f32(uint16_t b, bool fp16) {
  return fp16 ? __half2float(__ushort_as_half(b)) : bf16_bits_to_f32(b);
}
// fp32 -> activation bits, round half to even (fp16: IEEE, overflow to infinity)
__device__ __forceinline__ uint16_t f32_to_act_bits(float f, bool fp16) {
  return fp16 ? __half_as_ushort(__float2half_rn(f)) : f32_to_bf16_bits(f);
}

// Element i of a routed weight-scale array of dtype code dt (0 fp32, 1 bf16,
// 2 fp16), widened exactly to fp32.
__device__ __forceinline__ float wscale_at(const void* base, size_t i, int dt) {
  if (dt == 0) return static_cast<const float*>(base)[i];
  const uint16_t b = static_cast<const uint16_t*>(base)[i];
  return dt == 1 ? bf16_bits_to_f32(b) : __half2float(__ushort_as_half(b));
}

}  // namespace moe
