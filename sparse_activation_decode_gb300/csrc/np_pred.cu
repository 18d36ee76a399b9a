// Predictor kernels (sm_103a): matrix-vector products over row-major weights
// with fused epilogues.
//
// Shared predictor (NeuroPrefetcher section 3.3, "Shared Activation
// Predictor"): z = relu(W1 x) with x = rmsnorm(h after layer 0), then
// logits = W2 z and, per head of C logits, the index of the maximum (ties to
// the lowest index).  Per-layer predictor (LLM in a flash, section 3.1): the
// same two products plus an output bias, and neuron n fires when its logit is
// positive (sigmoid > 0.5).
//
// The argmax is computed without a second pass: every logit is folded into a
// 64-bit key (order-preserving bits of the fp32 value in the high word, the
// complement of the centroid index in the low word) and combined with
// atomicMax per head, which is order independent and so deterministic.
//
// Streaming: groups of `rows_per_stage` consecutive rows are fetched with one
// 1-D bulk copy each into an n_stages ring; thread t owns 16-byte column
// chunks t, t+256, ... and keeps the matching input values in registers.
#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  v = v + 0.0f;  // -0 -> +0 so that equal values compare equal
  const uint32_t u = __float_as_uint(v);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

namespace {
// d = a * b + c on a pair of floats (one packed FP32x2 FMA)
__device__ __forceinline__ float2 fma_pair(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
}  // namespace

template <typename T, int RPS>
__global__ void __launch_bounds__(kThreads, 2) rowdot_kernel(RowdotLaunch a) {
  static_assert(RPS <= 32 && 32 % RPS == 0, "a group's rows must share one mask word");
  constexpr int E = Elem<T>::E;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  const int len = a.len;
  const uint32_t row_bytes = (uint32_t)len * sizeof(T);
  const uint32_t stage_bytes = RPS * row_bytes;
  unsigned char* stages = smem + 128;
  float* xs = reinterpret_cast<float*>(stages + (size_t)a.n_stages * stage_bytes);
  float* red = xs + len;            // [2][8][RPS]
  float* red1 = red + 2 * 8 * RPS;  // [8]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = len / E;
  const int n_groups = (a.n_rows + RPS - 1) / RPS;
  const int my_n = (n_groups > (int)blockIdx.x) ? (n_groups - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const T* W = static_cast<const T*>(a.W);

  grid_dependents_launch();  // the next kernel may start its own prologue
  if (tid == 0) {
    for (int s = 0; s < a.n_stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t pol = policy_evict_first();
  auto rows_in = [&](int j) {
    const int g = (int)blockIdx.x + j * (int)gridDim.x;
    const int r = a.n_rows - g * RPS;
    return r < RPS ? r : RPS;
  };
  auto issue = [&](int j) {
    const int s = j % a.n_stages;
    const int g = (int)blockIdx.x + j * (int)gridDim.x;
    const uint32_t bytes = (uint32_t)rows_in(j) * row_bytes;
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_load(stages + (size_t)s * stage_bytes, W + (size_t)g * RPS * len, bytes, &bars[s], pol);
  };
  if (tid == 0) {
    const int pre = my_n < a.n_stages ? my_n : a.n_stages;
    for (int j = 0; j < pre; ++j) issue(j);
  }
  // the weights are constant; the input and the buffer cleared here belong
  // to the kernels before this one
  grid_dependency_wait();
  if (blockIdx.x == 0 && a.zero_ptr)
    for (int i = tid; i < a.zero_words; i += kThreads) a.zero_ptr[i] = 0u;

  if (a.vec_rmsnorm) {
    rmsnorm_to_smem(a.vec, a.vec2, xs, len, red1);
  } else {
    for (int j = tid; j < len; j += kThreads) xs[j] = a.vec[j];
    __syncthreads();
  }
  // x in registers as float pairs: each row's dot product runs as two
  // interleaved fp32 sums (even and odd elements), added at the end
  float2 xr[kMaxChunksPerThread][E / 2];
#pragma unroll
  for (int k = 0; k < kMaxChunksPerThread; ++k) {
    const int c = tid + k * kThreads;
#pragma unroll
    for (int e = 0; e < E / 2; ++e)
      xr[k][e] = (c < NC) ? make_float2(xs[c * E + 2 * e], xs[c * E + 2 * e + 1]) : make_float2(0.f, 0.f);
  }

  int issued_upto = my_n < a.n_stages ? my_n : a.n_stages;
  bool aborted = false;
  for (int j = 0; j < my_n; ++j) {
    const int s = j % a.n_stages;
    const bool ok = mbar_wait(&bars[s], (uint32_t)(j / a.n_stages) & 1u, a.err);
    const int nr = rows_in(j);
    const uint4* st = reinterpret_cast<const uint4*>(stages + (size_t)s * stage_bytes);
    float2 p2[RPS];
#pragma unroll
    for (int r = 0; r < RPS; ++r) p2[r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kMaxChunksPerThread; ++k) {
      const int c = tid + k * kThreads;
      if (c < NC) {
#pragma unroll
        for (int r = 0; r < RPS; ++r) {
          if (r < nr) {
            float f[E];
            Elem<T>::load(st[r * NC + c], f);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) p2[r] = fma_pair(make_float2(f[2 * e], f[2 * e + 1]), xr[k][e], p2[r]);
          }
        }
      }
    }
    float p[RPS];
#pragma unroll
    for (int r = 0; r < RPS; ++r) p[r] = p2[r].x + p2[r].y;
    float* rb = red + (j & 1) * 8 * RPS;
#pragma unroll
    for (int r = 0; r < RPS; ++r) {
      const float v = warp_sum(p[r]);
      if (lane == 0) rb[warp * RPS + r] = v;
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    // every thread has read stage j (the barrier above): refill it
    if (tid == 0 && j + a.n_stages < my_n) {
      issue(j + a.n_stages);
      ++issued_upto;
    }
    const int row0 = ((int)blockIdx.x + j * (int)gridDim.x) * RPS;
    if (a.mode == 2) {
      // the group's RPS rows share one 32-bit word of the firing mask (RPS
      // divides 32 and row0 is a multiple of RPS): one OR per group
      if (warp == 0) {
        bool fires = false;
        if (tid < nr) {
          float dot = 0.f;
#pragma unroll
          for (int w = 0; w < kThreads / 32; ++w) dot += rb[w * RPS + tid];
          const float logit = dot + to_f32<T>(static_cast<const T*>(a.bias)[row0 + tid]);
          if (a.out_f) a.out_f[row0 + tid] = logit;
          fires = logit > 0.f;
        }
        const uint32_t bits = __ballot_sync(0xffffffffu, fires);
        if (tid == 0 && bits) atomicOr(&a.fire_bits[row0 >> 5], bits << (row0 & 31));
      }
    } else if (tid < nr) {
      float dot = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) dot += rb[w * RPS + tid];
      const int row = row0 + tid;
      if (a.mode == 0) a.out_f[row] = dot > 0.f ? dot : 0.f;
      else atomicMax(&a.keys[row / a.C], argmax_key(dot, row % a.C));
    }
  }
  if (aborted && tid == 0) {
    const int first = issued_upto > a.n_stages ? issued_upto - a.n_stages : 0;
    for (int j = first; j < issued_upto; ++j)
      mbar_wait(&bars[j % a.n_stages], (uint32_t)(j / a.n_stages) & 1u, nullptr);
  }
}

__global__ void keys_to_ids_kernel(const unsigned long long* __restrict__ keys, int n, int* __restrict__ ids) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) ids[i] = (int)(0xFFFFFFFFu - (uint32_t)(keys[i] & 0xFFFFFFFFull));
}

size_t rowdot_smem_bytes(int len, int dtype_bytes, int rows_per_stage, int n_stages) {
  return 128 + (size_t)n_stages * rows_per_stage * len * dtype_bytes + (size_t)len * 4 +
         (2 * 8 * rows_per_stage + 8) * 4;
}

template <typename T, int RPS>
struct RowdotSmemTag {};

template <typename T, int RPS>
static cudaError_t launch_t(const RowdotLaunch& a, cudaStream_t st) {
  const size_t smem = rowdot_smem_bytes(a.len, a.dtype_bytes, RPS, a.n_stages);
  auto kern = rowdot_kernel<T, RPS>;
  cudaError_t e = ensure_dyn_smem<RowdotSmemTag<T, RPS>>(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  PdlConfig c(dim3(a.grid), dim3(kThreads), smem, st);
  c.cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&c.cfg, kern, a);
}

template <typename T>
static cudaError_t launch_rps(const RowdotLaunch& a, cudaStream_t st) {
  switch (a.rows_per_stage) {
    case 1: return launch_t<T, 1>(a, st);
    case 2: return launch_t<T, 2>(a, st);
    case 4: return launch_t<T, 4>(a, st);
    default: return launch_t<T, 8>(a, st);
  }
}

cudaError_t launch_rowdot(const RowdotLaunch& a, cudaStream_t st) {
  if (a.dtype == 0) return launch_rps<float>(a, st);
  if (a.dtype == 1) return launch_rps<__half>(a, st);
  return launch_rps<__nv_bfloat16>(a, st);
}

cudaError_t launch_keys_to_ids(const unsigned long long* keys, int n, int* ids, cudaStream_t st) {
  keys_to_ids_kernel<<<(n + 255) / 256, 256, 0, st>>>(keys, n, ids);
  return cudaGetLastError();
}

}  // namespace np
