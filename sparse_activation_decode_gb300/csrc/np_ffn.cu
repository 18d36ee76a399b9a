// FFN over a list of neuron rows, batch 1 (sm_103a).
//
// For each listed row r (a slot of a sparse layer's resident buffers, or a
// neuron of a dense layer):
//     h_r = relu(g_r . x) * (u_r . x)      (or relu(u_r . x) without a gate)
//     y  += h_r * d_r
// with x = rmsnorm(h), h = h_base + y_prev (NeuroPrefetcher full text, delta
// runtime: row i of the gate, up and down^T projections serves active neuron
// i; ReLU-fied form of the activation).  Consecutive layers chain through the
// residual stream as base + previous y: the CTA that reads first stores h for
// the next layer and clears the accumulator after next, so no separate
// residual-add kernel runs between layers.
//
// Design (HBM-bound: 2 flops per weight element):
//  * one CTA per SM per launch, sized so that two fit: consecutive launches
//    in a stream overlap (see below); warp-specialized: warp 8 is the
//    producer, warps 0-7 consume;
//  * whole neuron records (gate|up|down^T rows) stream into a shared-memory
//    ring through 1-D bulk copies (TMA engine); a "full" mbarrier per slot
//    counts the bytes in, an "empty" mbarrier per slot counts the consumer
//    warps done with it, so the producer refills a slot the moment it frees
//    up and keeps the whole ring in flight;
//  * programmatic dependent launch: the weights do not depend on the previous
//    layer, so the producer starts streaming as soon as the CTA is resident,
//    while the previous kernel in the stream may still be finishing; only the
//    consumers wait for it (griddepcontrol.wait) before reading h;
//  * thread t owns 16-byte column chunks t, t+256, ... of every row and keeps
//    the matching x values and y accumulators in registers; products use
//    packed FP32x2 FMAs.  Rows are consumed two at a time: the four dot
//    products of a pair are reduce-scattered across each warp (6 shuffles),
//    one block barrier combines the warps, and the down projection needs no
//    reduction at all;
//  * split-K over CTAs: each CTA adds its partial y to the layer's
//    accumulator with vector atomics (fp32; the order of the CTAs' additions
//    is not fixed).
#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

constexpr int kFfnThreads = 256;                 // consumer threads
constexpr int kFfnWarps = kFfnThreads / 32;      // consumer warps
constexpr int kFfnBlock = kFfnThreads + 32;      // plus one producer warp
constexpr int kRowCache = 64;                    // row indices cached per CTA

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}

// 16 bytes of T as E/2 float pairs
template <typename T> struct Pairs;
template <> struct Pairs<float> {
  static constexpr int N = 2;
  __device__ __forceinline__ static void load(const uint4& v, float2* f) {
    f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};
template <> struct Pairs<__half> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const uint4& v, float2* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __half22float2(h[i]);
  }
};
template <> struct Pairs<__nv_bfloat16> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const uint4& v, float2* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void consumer_sync() {  // warps 0-7 only
  asm volatile("bar.sync 1, %0;" ::"n"(kFfnThreads) : "memory");
}

// Named barrier over the consumer warps that also ORs a predicate: every
// consumer thread gets the same answer.
__device__ __forceinline__ bool consumer_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kFfnThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename T, bool GATED, int MAXC>
__global__ void __launch_bounds__(kFfnBlock, 2) ffn_rows_kernel(FfnLaunch a) {
  constexpr int P = Pairs<T>::N;      // float pairs per 16-byte chunk
  constexpr int E = 2 * P;            // elements per chunk
  constexpr int NPROJ = GATED ? 3 : 2;
  constexpr int NV = GATED ? 4 : 2;   // dot products per pair of rows
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [16]
  uint64_t* empty = full + 16;                           // [16]
  int* rows_s = reinterpret_cast<int*>(smem + 256);      // [kRowCache]
  const int D = a.D, n_slots = a.n_stages;
  const uint32_t row_bytes = (uint32_t)D * sizeof(T);
  const uint32_t slot_bytes = NPROJ * row_bytes;
  unsigned char* ring = smem + 512;
  float* red = reinterpret_cast<float*>(ring + (size_t)n_slots * slot_bytes);
  __shared__ int s_abort, s_issued;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = D / E;

  grid_dependents_launch();  // the next layer may start prefetching its weights
  int n = a.n_rows_dev ? *a.n_rows_dev : a.n_rows_host;
  if (n > a.list_cap) n = a.list_cap;
  if (n < 0) n = 0;
  const int G = (int)gridDim.x;
  const int my_n = (n > (int)blockIdx.x) ? (n - 1 - (int)blockIdx.x) / G + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < n_slots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kFfnWarps);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
  }
  if (a.row_list)
    for (int j = tid; j < my_n && j < kRowCache; j += kFfnBlock) rows_s[j] = a.row_list[blockIdx.x + j * G];
  __syncthreads();

  float2 acc[MAXC][P];
#pragma unroll
  for (int k = 0; k < MAXC; ++k)
#pragma unroll
    for (int q = 0; q < P; ++q) acc[k][q] = make_float2(0.f, 0.f);

  if (warp == kFfnWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const T* w_gate = static_cast<const T*>(a.w_gate);
      const T* w_up = static_cast<const T*>(a.w_up);
      const T* w_down = static_cast<const T*>(a.w_down);
      for (int j = 0; j < my_n; ++j) {
        const int s = j % n_slots;
        if (j >= n_slots && !mbar_wait(&empty[s], (uint32_t)(j / n_slots - 1) & 1u, a.err)) {
          s_abort = 1;
          break;
        }
        int r = a.row_list ? (j < kRowCache ? rows_s[j] : a.row_list[blockIdx.x + j * G]) : (int)blockIdx.x + j * G;
        if ((unsigned)r >= (unsigned)a.row_limit) {
          atomicExch(a.err, kDevErrBounds);
          r = 0;
        }
        unsigned char* dst = ring + (size_t)s * slot_bytes;
        mbar_arrive_expect_tx(&full[s], slot_bytes);
        int p = 0;
        if (GATED) bulk_load(dst + (p++) * row_bytes, w_gate + (size_t)r * D, row_bytes, &full[s], pol);
        bulk_load(dst + (p++) * row_bytes, w_up + (size_t)r * D, row_bytes, &full[s], pol);
        bulk_load(dst + p * row_bytes, w_down + (size_t)r * D, row_bytes, &full[s], pol);
        s_issued = j + 1;
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // x = rmsnorm(h_in + yprev): each thread reads its own chunks of h, once
    // the previous kernel's writes are visible.  CTA 0 stores h for the next
    // layer and clears the accumulator after next.
    grid_dependency_wait();
    float2 xr[MAXC][P];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < MAXC; ++k) {
      const int c = tid + k * kFfnThreads;
#pragma unroll
      for (int q = 0; q < P; ++q) {
        float2 v = make_float2(0.f, 0.f);
        if (c < NC) {
          v = *reinterpret_cast<const float2*>(a.h_in + c * E + 2 * q);
          if (a.yprev) {
            const float2 w = *reinterpret_cast<const float2*>(a.yprev + c * E + 2 * q);
            v.x += w.x;
            v.y += w.y;
          }
          if (blockIdx.x == 0) {
            if (a.hb_out) *reinterpret_cast<float2*>(a.hb_out + c * E + 2 * q) = v;
            if (a.y_zero) *reinterpret_cast<float2*>(a.y_zero + c * E + 2 * q) = make_float2(0.f, 0.f);
          }
        }
        xr[k][q] = v;
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, ss));
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kFfnWarps; ++w) tot += red[w];
    const float inv = rsqrtf(tot / (float)D + 1e-6f);
#pragma unroll
    for (int k = 0; k < MAXC; ++k)
#pragma unroll
      for (int q = 0; q < P; ++q) {
        xr[k][q].x *= inv;
        xr[k][q].y *= inv;
      }
    consumer_sync();  // red is reused below

    for (int j = 0; j < my_n; j += 2) {
      const bool two = j + 1 < my_n;
      const int s0 = j % n_slots, s1 = (j + 1) % n_slots;
      bool ok = mbar_wait(&full[s0], (uint32_t)(j / n_slots) & 1u, a.err);
      if (two) ok = mbar_wait(&full[s1], (uint32_t)((j + 1) / n_slots) & 1u, a.err) && ok;
      const uint4* r0 = reinterpret_cast<const uint4*>(ring + (size_t)s0 * slot_bytes);
      const uint4* r1 = reinterpret_cast<const uint4*>(ring + (size_t)s1 * slot_bytes);
      float2 d2[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) d2[v] = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < MAXC; ++k) {
        const int c = tid + k * kFfnThreads;
        if (c < NC) {
          float2 f[P];
#pragma unroll
          for (int row = 0; row < 2; ++row) {
            if (row == 1 && !two) break;
            const uint4* rr = row ? r1 : r0;
            if (GATED) {
              Pairs<T>::load(rr[c], f);
#pragma unroll
              for (int q = 0; q < P; ++q) d2[row * 2] = ffma2(f[q], xr[k][q], d2[row * 2]);
              Pairs<T>::load(rr[NC + c], f);
#pragma unroll
              for (int q = 0; q < P; ++q) d2[row * 2 + 1] = ffma2(f[q], xr[k][q], d2[row * 2 + 1]);
            } else {
              Pairs<T>::load(rr[c], f);
#pragma unroll
              for (int q = 0; q < P; ++q) d2[row] = ffma2(f[q], xr[k][q], d2[row]);
            }
          }
        }
      }
      // warp reduce-scatter: lane l ends with the warp sum of value vi(l)
      float pv[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) pv[v] = d2[v].x + d2[v].y;
      int cnt = NV, vi = 0;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        if (cnt > 1) {
          const bool up = (lane & off) != 0;
          const int half = cnt >> 1;
#pragma unroll
          for (int q = 0; q < NV / 2; ++q) {
            if (q < half) {
              const float send = up ? pv[q] : pv[q + half];
              const float keep = up ? pv[q + half] : pv[q];
              pv[q] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
          }
          vi = vi * 2 + (up ? 1 : 0);
          cnt = half;
        } else {
          pv[0] += __shfl_xor_sync(0xffffffffu, pv[0], off);
        }
      }
      float* rb = red + ((j >> 1) & 1) * kFfnWarps * NV;
      if ((lane & (32 / NV - 1)) == 0) rb[warp * NV + vi] = pv[0];
      if (consumer_sync_or(!ok)) {  // a copy never arrived: all consumers stop
        if (tid == 0) s_abort = 1;
        break;
      }
      float t[NV];
#pragma unroll
      for (int v = 0; v < NV; ++v) t[v] = 0.f;
#pragma unroll
      for (int w = 0; w < kFfnWarps; ++w) {
        if (NV == 4) {
          const float4 x4 = reinterpret_cast<const float4*>(rb)[w];
          t[0] += x4.x; t[1] += x4.y; t[2 % NV] += x4.z; t[3 % NV] += x4.w;
        } else {
          const float2 x2 = reinterpret_cast<const float2*>(rb)[w];
          t[0] += x2.x; t[1] += x2.y;
        }
      }
      float hv0, hv1;
      if (GATED) {
        hv0 = (t[0] > 0.f ? t[0] : 0.f) * t[1];
        hv1 = (t[2 % NV] > 0.f ? t[2 % NV] : 0.f) * t[3 % NV];
      } else {
        hv0 = t[0] > 0.f ? t[0] : 0.f;
        hv1 = t[1] > 0.f ? t[1] : 0.f;
      }
      const float2 h0 = make_float2(hv0, hv0), h1 = make_float2(hv1, hv1);
      const int dn = (NPROJ - 1) * NC;
#pragma unroll
      for (int k = 0; k < MAXC; ++k) {
        const int c = tid + k * kFfnThreads;
        if (c < NC) {
          float2 f[P];
          Pairs<T>::load(r0[dn + c], f);
#pragma unroll
          for (int q = 0; q < P; ++q) acc[k][q] = ffma2(h0, f[q], acc[k][q]);
          if (two) {
            Pairs<T>::load(r1[dn + c], f);
#pragma unroll
            for (int q = 0; q < P; ++q) acc[k][q] = ffma2(h1, f[q], acc[k][q]);
          }
        }
      }
      // this warp is done with both slots
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[s0]);
        if (two) mbar_arrive(&empty[s1]);
      }
    }
  }
  __syncthreads();
  if (s_abort && tid == kFfnThreads) {
    // drain copies still in flight before the CTA's shared memory goes away
    atomicExch(a.err, kDevErrTimeout);
    const int issued = s_issued;
    const int first = issued > n_slots ? issued - n_slots : 0;
    for (int j = first; j < issued; ++j) mbar_wait(&full[j % n_slots], (uint32_t)(j / n_slots) & 1u, nullptr);
  }

  // ---- split-K: this CTA's partial y into the layer's accumulator
  if (tid < kFfnThreads && !s_abort) {
#pragma unroll
    for (int k = 0; k < MAXC; ++k) {
      const int c = tid + k * kFfnThreads;
      if (c < NC) {
#pragma unroll
        for (int q = 0; q < P; q += 2)
          atomicAdd(reinterpret_cast<float4*>(a.y_acc + c * E + 2 * q),
                    make_float4(acc[k][q].x, acc[k][q].y, acc[k][q + 1].x, acc[k][q + 1].y));
      }
    }
  }
}

template <typename T, bool GATED>
static void* kernel_for(int maxc) {
  switch (maxc) {
    case 1: return reinterpret_cast<void*>(ffn_rows_kernel<T, GATED, 1>);
    case 2: return reinterpret_cast<void*>(ffn_rows_kernel<T, GATED, 2>);
    case 3: return reinterpret_cast<void*>(ffn_rows_kernel<T, GATED, 3>);
    default: return reinterpret_cast<void*>(ffn_rows_kernel<T, GATED, 4>);
  }
}

static int chunks_per_thread(int D, int dtype_bytes) {
  const int nc = D * dtype_bytes / 16;
  return (nc + kFfnThreads - 1) / kFfnThreads;
}

static void* pick_kernel(int dtype, bool gated, int D, int dtype_bytes) {
  const int mc = chunks_per_thread(D, dtype_bytes);
  if (gated) return dtype == 0 ? kernel_for<float, true>(mc) : dtype == 1 ? kernel_for<__half, true>(mc)
                                                                         : kernel_for<__nv_bfloat16, true>(mc);
  return dtype == 0 ? kernel_for<float, false>(mc) : dtype == 1 ? kernel_for<__half, false>(mc)
                                                               : kernel_for<__nv_bfloat16, false>(mc);
}

size_t ffn_smem_bytes(int D, int dtype_bytes, int nproj, int n_stages) {
  return 512 + (size_t)n_stages * nproj * D * dtype_bytes + 64 * 4;
}

int ffn_max_chunks() { return kFfnThreads * 4; }

cudaError_t ffn_plan(int dtype, int gated, int D, int dtype_bytes, size_t smem_per_sm, int n_sms, int* n_stages,
                     int* grid) {
  const int nproj = gated ? 3 : 2;
  // shared memory for two CTAs per SM (so the next layer's CTAs can prefetch
  // beside the current ones), each with as many ring slots (2..16) as fit
  const size_t per_cta = smem_per_sm / 2 > 1024 ? smem_per_sm / 2 - 1024 : 0;
  int ns = 16;
  while (ns > 2 && ffn_smem_bytes(D, dtype_bytes, nproj, ns) > per_cta) --ns;
  if (ffn_smem_bytes(D, dtype_bytes, nproj, ns) > per_cta) return cudaErrorInvalidValue;
  void* k = pick_kernel(dtype, gated != 0, D, dtype_bytes);
  const size_t smem = ffn_smem_bytes(D, dtype_bytes, nproj, ns);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kFfnBlock, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // one CTA per SM per launch: the second slot of every SM is left to the
  // next launch in the stream, which then streams beside this one
  *n_stages = ns;
  *grid = n_sms;
  return cudaSuccess;
}

cudaError_t ffn_set_smem(int dtype, int gated, int D, int dtype_bytes, int n_stages) {
  void* k = pick_kernel(dtype, gated != 0, D, dtype_bytes);
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)ffn_smem_bytes(D, dtype_bytes, gated ? 3 : 2, n_stages));
}

cudaError_t launch_ffn_rows(const FfnLaunch& a, cudaStream_t st) {
  void* k = pick_kernel(a.dtype, a.gated != 0, a.D, a.dtype_bytes);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid, 1, 1);
  cfg.blockDim = dim3(kFfnBlock, 1, 1);
  cfg.dynamicSmemBytes = ffn_smem_bytes(a.D, a.dtype_bytes, a.gated ? 3 : 2, a.n_stages);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  FfnLaunch arg = a;
  void* params[] = {&arg};
  return cudaLaunchKernelExC(&cfg, k, params);
}

}  // namespace np
