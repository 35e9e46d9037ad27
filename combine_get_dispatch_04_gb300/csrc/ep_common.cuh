// ep_common.cuh -- helpers shared by the layout, dispatch and combine kernels:
// host-side status/validation utilities, per-device properties, and inline
// PTX for 128-bit cache-hinted global accesses, mbarriers and 1-D bulk (TMA)
// copies on sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ep.h"

namespace ep {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline cudaStream_t to_cuda(ep_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline ep_status_t launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

struct DeviceProps {
  int sm_count = 0;
  int smem_optin = 0;   // max dynamic shared memory per block (opt-in)
  int smem_per_sm = 0;  // shared memory per SM, shared by its resident blocks
};

// Cached per device; returns false if the CUDA runtime cannot be queried.
bool device_props(DeviceProps* out);

// Common argument checks for the routing description; the layout also needs
// T % R == 0 (routing_ok), dispatch and combine do not (routing_ok_any_t):
// there the slots, not the source ranks, place the rows.
inline bool routing_ok_any_t(int64_t T, int K, int E, int R) {
  if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS) return false;
  if (R < 1 || R > EP_MAX_RANKS || E % R != 0) return false;
  if (T * (int64_t)R >= (int64_t(1) << 31)) return false;
  return true;
}
inline bool routing_ok(int64_t T, int K, int E, int R) {
  return routing_ok_any_t(T, K, E, R) && T % R == 0;
}

// Launch with programmatic dependent launch (PDL): the kernel may be
// scheduled while the previous kernel in the stream finishes, and waits for
// it in pdl_wait() before touching global memory.  Every kernel of this
// library calls pdl_wait() before its first global access, so all data
// dependences between consecutive launches are kept.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl for a grid of thread-block clusters of `cluster_x` CTAs each
// (grid.x must be a multiple of cluster_x).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                      size_t smem, int cluster_x, cudaStream_t st,
                                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Per-device set-up of a single-cluster kernel, done once by the caller
// (under its own lock): raises the kernel's dynamic shared-memory limit to
// `smem`, and returns in *out the largest cluster it can run: 16 CTAs (a
// non-portable size) when the device schedules a cluster of 16 blocks of
// `block` threads and `smem` bytes, else 8.
template <typename... KArgs>
inline cudaError_t setup_single_cluster(void (*kernel)(KArgs...), int block, size_t smem,
                                        int* out) {
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int ctas = 8;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0) ctas = 16;
  }
  cudaGetLastError();  // a refused non-portable size is not the caller's error
  *out = ctas;
  return cudaSuccess;
}

// Per-device cache of setup_single_cluster's answer for one kernel.
struct ClusterSizeCache {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  int ctas[kMaxDevices] = {};  // 0 = not yet set up

  template <typename... KArgs>
  cudaError_t get(void (*kernel)(KArgs...), int block, size_t smem, int* out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (ctas[dev] == 0) {
      e = setup_single_cluster(kernel, block, smem, &ctas[dev]);
      if (e != cudaSuccess) return e;
    }
    *out = ctas[dev];
    return cudaSuccess;
  }
};

// ---------------------------------------------------------------------------
// device side
// ---------------------------------------------------------------------------

// Waits until the previous kernel in the stream has completed and its
// memory is visible (a no-op without PDL), then lets the next kernel be
// scheduled as this grid's blocks retire.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits like pdl_wait_then_release but leaves the release to the implicit
// one at block exit: the next kernel is scheduled only once every block of
// this grid has finished.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // bounded pipeline waits: 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 128-bit read-only load that does not allocate in L1 (data is touched once).
__device__ __forceinline__ int4 ld_stream_v4(const int4* p) {
  int4 v;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// 128-bit store with the streaming (evict-first) cache policy.
__device__ __forceinline__ void st_stream_v4(int4* p, const int4& v) {
  asm volatile("st.global.cs.v4.s32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream_v2(uint2* p, const uint2& v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// --- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when *abort becomes non-zero or after kWaitTimeoutNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const volatile int* abort) {
  for (int i = 0; i < 32; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// --- 1-D bulk copy (TMA engine), global -> shared, completion on an mbarrier --
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_g2s(void* dst_smem, const void* src_global,
                                              uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_global), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Stores with an L2 cache-policy hint (from createpolicy).
__device__ __forceinline__ void st_hint_b32(void* p, uint32_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void st_hint_b64(void* p, uint64_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(p), "l"(v), "l"(policy)
               : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// --- thread-block cluster ----------------------------------------------------
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Cluster-wide barrier in two halves, executed by every thread of every CTA
// of the cluster.  arrive releases this thread's earlier writes (shared and
// global) at cluster scope; wait blocks until all threads have arrived and
// acquires their writes.  A hardware barrier: it needs no timeout.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address, in the cluster's shared window, of the variable at `p` (a shared
// address of this CTA) in the shared memory of CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_map(const void* p, uint32_t rank) {
  uint32_t out;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(p)), "r"(rank));
  return out;
}

// Load from another CTA's shared memory (distributed shared memory).
// Volatile, so that it stays after the cluster barrier that publishes the
// data; loads issued back to back still overlap until their values are used.
__device__ __forceinline__ int32_t dsmem_ld(uint32_t addr) {
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// --- bf16 packing -----------------------------------------------------------
__device__ __forceinline__ void unpack_bf16x8(const int4& v, float (&f)[8]) {
  const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

}  // namespace ep
