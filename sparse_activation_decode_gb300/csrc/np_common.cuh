// Device helpers shared by the decode-path kernels (sm_103a).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "np_kernels.h"

namespace np {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s

// Raise a kernel's dynamic shared-memory limit only when a launch needs more
// than it was last set to on this device (the attribute call costs host time
// on every launch otherwise).  One cache per kernel function (`Tag`) and
// device; the attribute is idempotent, so a race between threads only
// repeats the call.
template <typename Tag>
inline cudaError_t ensure_dyn_smem(const void* kern, size_t bytes) {
  constexpr int kDevices = 64;
  static size_t set_to[kDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kDevices && bytes <= set_to[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kDevices) set_to[dev] = bytes;
  return e;
}

// ---------------------------------------------------------------------------
// Element types: a 16-byte chunk holds E elements.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int E = 4;
  __device__ __forceinline__ static void load(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
};
template <> struct Elem<__half> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void load(const uint4& v, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) { float2 t = __half22float2(h[i]); f[2 * i] = t.x; f[2 * i + 1] = t.y; }
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int E = 8;
  __device__ __forceinline__ static void load(const uint4& v, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) { float2 t = __bfloat1622float2(h[i]); f[2 * i] = t.x; f[2 * i + 1] = t.y; }
  }
};

// ---------------------------------------------------------------------------
// Shared-memory barriers and 1-D bulk copies (TMA engine, no tensor map).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait until the previous kernel in the stream has completed
// and its writes are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A launch configuration that allows programmatic dependent launch.
struct PdlConfig {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr{};
  PdlConfig(dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
  }
};

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`, giving up after about one second; on
// timeout the error word gets kDevErrTimeout and false is returned.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
      if (err) atomicExch(err, kDevErrTimeout);
      return false;
    }
  }
}

// Bulk copy `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

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

// ---------------------------------------------------------------------------
// Reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of one value per thread over the CTA; every thread gets the total.
// `red` must hold kThreads/32 floats; the summation order is fixed.
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) s += red[i];
  return s;
}

// x_hat = h / sqrt(mean(h^2) + 1e-6) into shared memory (fp32, D values),
// with h = h1 + h2 (h2 may be null).
__device__ __forceinline__ void rmsnorm_to_smem(const float* __restrict__ h, const float* __restrict__ h2, float* xs,
                                                int D, float* red) {
  float ss = 0.f;
  for (int j = threadIdx.x; j < D; j += kThreads) {
    const float v = h2 ? h[j] + h2[j] : h[j];
    xs[j] = v;
    ss = fmaf(v, v, ss);
  }
  const float tot = block_sum(ss, red);
  const float inv = rsqrtf(tot / (float)D + 1e-6f);
  for (int j = threadIdx.x; j < D; j += kThreads) xs[j] *= inv;
  __syncthreads();
}

}  // namespace np
