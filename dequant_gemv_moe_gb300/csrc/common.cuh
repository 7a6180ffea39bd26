// common.cuh — device helpers shared by the kernels of the dqmoe library:
// inline-PTX wrappers for mbarriers, 1-D bulk (TMA) copies, cluster shared
// memory and the m16n8k16 tensor-core instruction, plus the device status word.
// Target: sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/dqmoe.h"

namespace dqmoe {

// Bytes of one 256-weight "super-block row unit" per format.  Q8_0 stores 8
// blocks of 34 bytes per 256 weights, Q4_0 8 blocks of 18.
template <int FMT> struct Fmt;
template <> struct Fmt<DQ_Q4_K> { static constexpr int SB_BYTES = 144; };
template <> struct Fmt<DQ_Q6_K> { static constexpr int SB_BYTES = 210; };
template <> struct Fmt<DQ_Q8_0> { static constexpr int SB_BYTES = 272; };
template <> struct Fmt<DQ_Q4_0> { static constexpr int SB_BYTES = 144; };   // 8 blocks of 18
template <> struct Fmt<DQ_Q5_K> { static constexpr int SB_BYTES = 176; };
template <> struct Fmt<DQ_NVFP4> { static constexpr int SB_BYTES = 144; };
template <> struct Fmt<DQ_Q2_K> { static constexpr int SB_BYTES = 84; };
template <> struct Fmt<DQ_Q3_K> { static constexpr int SB_BYTES = 110; };

// Hardware FP4/FP8 -> fp16 conversions (exact).  e2m1x8: the 8 E2M1 codes of
// a word (byte j: codes 2j low nibble, 2j+1 high nibble) as 4 fp16 pairs in
// code order; e4m3x2: two E4M3 bytes (low byte first) as one fp16 pair.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// Device status word: a kernel whose bounded wait runs out sets it to
// DQ_ERR_DEVICE_TIMEOUT and returns instead of hanging.  Read by
// dq_device_status().
extern __device__ int g_device_status;

__device__ __forceinline__ void report_timeout() {
  atomicExch(&g_device_status, (int)DQ_ERR_DEVICE_TIMEOUT);
}

// A wait that polls longer than this many SM clock cycles (~1 s) gives up.
// DQ_WAIT_LIMIT_CYCLES overrides it for a test build only (the library is
// always built with the default).
#ifndef DQ_WAIT_LIMIT_CYCLES
#define DQ_WAIT_LIMIT_CYCLES 2000000000LL
#endif
constexpr long long kWaitLimitCycles = DQ_WAIT_LIMIT_CYCLES;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
// Relaxed: what the phase waits for (the TMA bytes) is tracked by the count.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

// Arrive on the barrier at the same offset in the shared memory of CTA
// `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar)),
      "r"(rank)
      : "memory");
}

// Relaxed arrival: for a consumer releasing a stage it has finished reading.
// Every shared-memory load of the stage has returned its data (each result
// was consumed by an instruction earlier in program order), so no fence is
// needed before the producer's next asynchronous overwrite.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.relaxed.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
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

// Cluster-scope acquire variant, for barriers that remote CTAs arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with `parity` to complete.  Returns false (and
// records a timeout) if it does not complete within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) {
      report_timeout();
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) {
      report_timeout();
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on
// an mbarrier.  dst, src 16-byte aligned, bytes a multiple of 16.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2-D tiled TMA load of box (x, y) of `map` into shared memory, completion
// counted in bytes on `bar`.  x * element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Prefetch box (x, y) of `map` into L2: no shared memory, no completion
// signal; a later load of the same box finds it in L2.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   (uint64_t)map),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// 16-byte asynchronous copy global -> shared (LDGSTS), and an mbarrier
// arrival that fires once all of this thread's earlier cp.async copies have
// landed (counts as the thread's arrival: .noinc).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store a float into the shared memory of CTA `rank` at this CTA's address.
__device__ __forceinline__ void st_cluster_f32x4(float* local_addr, uint32_t rank, float a,
                                                 float b, float c, float d) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "st.shared::cluster.v4.f32 [ra], {%2, %3, %4, %5};\n\t}" ::"r"(smem_u32(local_addr)),
      "r"(rank), "f"(a), "f"(b), "f"(c), "f"(d)
      : "memory");
}

// ---------------------------------------------------------------------------
// tensor core: D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// packed fp32 pairs (one instruction for two lanes of fp32 arithmetic)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// The same product as a plain (non-volatile) asm: the compiler may schedule
// it freely among independent work.
__device__ __forceinline__ void mma_16816_nv(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// small bit helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  // (a & mask) | orv in one LOP3
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(orv));
  return r;
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) {
  return *reinterpret_cast<__half2*>(&v);
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// Shared loads the compiler may reorder among themselves and other work.  The
// caller orders them after the data is ready by deriving every address from
// a value passed through order_after_wait(), and before the data is released
// by consuming the results in keep_before_release().
__device__ __forceinline__ uint2 lds_u64_nv(uint32_t addr) {
  uint2 v;
  asm("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds_u128_nv(uint32_t addr) {
  uint4 v;
  asm("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32_nv(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16_nv(uint32_t addr) {
  unsigned short v;
  asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// 32-bit load from a 2-byte aligned shared address.
__device__ __forceinline__ uint32_t lds_u32_a2_nv(uint32_t addr) {
  const uint32_t base = addr & ~3u;
  const uint32_t lo = lds_u32_nv(base);
  if ((addr & 2u) == 0) return lo;
  const uint32_t hi = lds_u32_nv(base + 4);
  return __funnelshift_r(lo, hi, 16);
}
__device__ __forceinline__ uint32_t order_after_wait(uint32_t v) {
  asm volatile("mov.b32 %0, %1;" : "=r"(v) : "r"(v) : "memory");
  return v;
}
__device__ __forceinline__ void keep_before_release(float a, float b, float c, float d) {
  asm volatile("" ::"f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
// every element of a float array whose size is a multiple of 4
template <int N>
__device__ __forceinline__ void keep_before_release(const float* a) {
#pragma unroll
  for (int i = 0; i < N; i += 4) keep_before_release(a[i], a[i + 1], a[i + 2], a[i + 3]);
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// 32-bit load from a 2-byte aligned shared address.
__device__ __forceinline__ uint32_t lds_u32_a2(uint32_t addr) {
  const uint32_t base = addr & ~3u;
  const uint32_t lo = lds_u32(base);
  if ((addr & 2u) == 0) return lo;
  const uint32_t hi = lds_u32(base + 4);
  return __funnelshift_r(lo, hi, 16);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization: it may be scheduled while the kernel
// before it in the stream is still finishing.  pdl_wait() blocks the calling
// thread until that kernel has completed and its memory is visible (it returns
// at once when there is none), so every thread calls it before its first read
// of data another kernel may produce and before its first global write.
// pdl_trigger() lets the next kernel be scheduled; issued once every CTA of
// this grid is resident, it only shortens the gap between kernels.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization and, for cluster > 0, a
// thread-block cluster of `cluster` CTAs along x, placed by the load-balancing
// policy (measured on the Llama-3-8B layer step, whose o and down GEMVs run
// in clusters of 8: 32.72 -> 32.24 us; the spread policy equals the default).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    attr[n].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[n].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace dqmoe

