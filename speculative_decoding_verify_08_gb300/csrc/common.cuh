// common.cuh -- helpers shared by the verify-step kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA bulk and tensor copies,
// programmatic dependent launch and warp-level tensor-core MMA; bounded
// waits; and the host-side launcher that applies the library's launch flags.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/specverify.h"

namespace sv {

// ---------------------------------------------------------------- errors --
// Bits of the device error word (one word per device, see api.cu).
constexpr unsigned ERR_TIMEOUT = 1u;
constexpr unsigned ERR_OVERFLOW = 2u;
constexpr unsigned ERR_LISTS = 4u;  // candidate lists made for other rows or a smaller top-k

// A bounded wait gives up after this many SM clock cycles (~1-2 s).
constexpr long long WAIT_LIMIT_CYCLES = 3000000000LL;

// ------------------------------------------------------------ host state --
unsigned *device_error_word();  // device address of this device's word
int device_sm_count();          // SMs of the current device
unsigned launch_flags();
void count_launch();

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ __forceinline__ long long lmin(long long a, long long b) { return a < b ? a : b; }

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device (remembered per kernel and device; see api.cu).
cudaError_t raise_smem_limit(const void *kernel, size_t bytes);

inline sv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

// Launches `kern` on `stream` with the library's launch flags (PDL when
// requested) and counts the launch.  Raises the kernel's dynamic shared
// memory limit to `smem` first, whatever its size: the default limit covers
// static and dynamic shared memory together, so a kernel with static arrays
// can exceed it with less than 48 KB of dynamic memory.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, Args &&...args) {
  if (smem > 0) {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (launch_flags() & SV_LAUNCH_PDL) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e == cudaSuccess) count_launch();
  return e;
}

// The same launch with thread-block clusters of `cl` CTAs along x (cl >= 2;
// the grid is a multiple of cl).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, int cl, Args &&...args) {
  if (smem > 0) {
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void *>(kern), smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (launch_flags() & SV_LAUNCH_PDL) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e == cudaSuccess) count_launch();
  return e;
}

// How many clusters of `cl` CTAs of `kern` (block threads, smem bytes of
// dynamic shared memory) the device runs at once; 0 if the query fails.
// Cached per (kernel, cl, smem, device).
int max_active_clusters(const void *kern, int block, size_t smem, int cl);
template <typename... KArgs>
int max_active_clusters(void (*kern)(KArgs...), int block, size_t smem, int cl) {
  return max_active_clusters(reinterpret_cast<const void *>(kern), block, smem, cl);
}

// ---------------------------------------------------------- device PTX --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Programmatic dependent launch: wait for the predecessor grid's memory,
// and allow the successor grid to be scheduled.  No-ops without PDL.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Makes initialised mbarriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Potentially blocking test: the thread may sleep (up to `ns` nanoseconds)
// until the phase completes, so waiting warps do not take issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete, sleeping between
// checks; gives up after WAIT_LIMIT_CYCLES, records ERR_TIMEOUT in *err and
// returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 200000u)) {
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
      atomicOr(err, ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Bounded wait without the sleep hint, for warps on a latency-critical path
// that have nothing else to do: they resume as soon as the phase completes.
__device__ __forceinline__ bool spin_wait(uint64_t *bar, uint32_t parity, unsigned *err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
      atomicOr(err, ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// L2 policy: stream once, evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Ask L2 to load [p, p + bytes) from memory (16-byte aligned start, bytes a
// multiple of 16); nothing waits for it.
__device__ __forceinline__ void l2_prefetch_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Thread-block clusters: rank in the cluster, the shared-memory address of
// the same variable in CTA `rank` of the cluster, loads from it, and the
// cluster-wide barrier (every thread of every CTA of the cluster, each warp
// converged; release/acquire at cluster scope).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_cluster(uint32_t a, float2) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster(uint32_t a, float4) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                            uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy global -> shared (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2^x by the MUFU approximation (flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 4-byte asynchronous copy global -> shared (completed by cp_async_wait_all).
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// D = A(16x16, row) * B(16x8, col) + C, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same MMA with a zero accumulator input (the first k16 step of a sum).
__device__ __forceinline__ void mma_bf16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same MMA with a zero accumulator input.
__device__ __forceinline__ void mma_f16_16816_zc(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// The k-th largest of the n unsigned keys a[0..n) (shared memory; every lane
// of the warp calls it with the same arguments): the largest t such that at
// least k keys are >= t, built from the highest bit that differs between
// the largest and the smallest key down (the bits above it are common to
// every key).  0 when n <= k (every key qualifies).
// Register variant for n <= 32 * E: the keys are read once.
template <int E>
__device__ __forceinline__ uint32_t warp_kth_largest_regs(const uint32_t *a, int n, int k) {
  const int lane = threadIdx.x & 31;
  uint32_t v[E], mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane + 32 * e;
    v[e] = i < n ? a[i] : 0u;  // absent keys count as 0: never >= a candidate (> 0)
    if (i < n) {
      mx = max(mx, v[e]);
      mn = min(mn, v[e]);
    }
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  const uint32_t d = mx ^ mn;
  if (d == 0u) return mx;
  const int hb = 31 - __clz(d);
  uint32_t t = hb == 31 ? 0u : (mx & ~((2u << hb) - 1u));
  for (int b = hb; b >= 0; --b) {
    const uint32_t cand = t | (1u << b);
    unsigned c = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) c += v[e] >= cand ? 1u : 0u;
    if (__reduce_add_sync(0xffffffffu, c) >= (unsigned)k) t = cand;
  }
  return t;
}

__device__ __forceinline__ uint32_t warp_kth_largest(const uint32_t *a, int n, int k) {
  if (n <= k) return 0u;
  if (n <= 256) return warp_kth_largest_regs<8>(a, n, k);
  if (n <= 512) return warp_kth_largest_regs<16>(a, n, k);
  const int lane = threadIdx.x & 31;
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
  for (int i = lane; i < n; i += 32) {
    mx = max(mx, a[i]);
    mn = min(mn, a[i]);
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  const uint32_t d = mx ^ mn;
  if (d == 0u) return mx;
  const int hb = 31 - __clz(d);
  uint32_t t = hb == 31 ? 0u : (mx & ~((2u << hb) - 1u));
  for (int b = hb; b >= 0; --b) {
    const uint32_t cand = t | (1u << b);
    unsigned c = 0;
    for (int i = lane; i < n; i += 32) c += a[i] >= cand ? 1u : 0u;
    if (__reduce_add_sync(0xffffffffu, c) >= (unsigned)k) t = cand;
  }
  return t;
}

// (a & B) | C as one three-input logic operation (lookup table 0xEA).
template <uint32_t B, uint32_t C>
__device__ __forceinline__ uint32_t and_or(uint32_t a) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(B), "n"(C));
  return d;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Explicit shared-memory loads on 32-bit shared addresses.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float f16lo(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16hi(uint32_t v) {
  return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

}  // namespace sv
