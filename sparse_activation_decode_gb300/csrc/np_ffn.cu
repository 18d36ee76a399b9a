// FFN over a list of neuron rows, batch 1 (sm_103a).
//
// For each listed row r (a slot of a sparse layer's resident buffers, or a
// neuron of a dense layer):
//     h_r = relu(g_r . x) * (u_r . x)      (or relu(u_r . x) without a gate)
//     y  += h_r * d_r
// with x = rmsnorm(h_in) (NeuroPrefetcher full text, delta runtime: row i of
// the gate, up and down^T projections serves active neuron i; the ReLU-fied
// form of the activation).
//
// Design: the kernel is HBM-bound (2 flops per weight element).  Each CTA
// streams whole rows into shared memory with 1-D bulk copies (TMA engine)
// through an n_stages-deep ring guarded by mbarriers; one thread issues the
// copies.  Thread t owns 16-byte column chunks t, t+256, ... of every row and
// keeps the matching x values and y accumulators in registers, so a row
// costs one block reduction (for its two dot products) and no reduction for
// the down projection.  Each CTA writes its partial y; ffn_finish_kernel
// sums the partials in CTA order (deterministic) and adds the residual.
#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

template <typename T, bool GATED>
__global__ void __launch_bounds__(kThreads, 2)
    ffn_rows_kernel(const float* __restrict__ h_in, const T* __restrict__ w_gate, const T* __restrict__ w_up,
                    const T* __restrict__ w_down, const int* __restrict__ row_list, const int* __restrict__ n_rows_dev,
                    int n_rows_host, int list_cap, int row_limit, float* __restrict__ part, int D, int n_stages,
                    int* err) {
  constexpr int E = Elem<T>::E;
  constexpr int NPROJ = GATED ? 3 : 2;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // up to 16 stages
  const uint32_t row_bytes = (uint32_t)D * sizeof(T);
  const uint32_t stage_bytes = NPROJ * row_bytes;
  unsigned char* stages = smem + 128;
  float* xs = reinterpret_cast<float*>(stages + (size_t)n_stages * stage_bytes);
  float* red = xs + D;              // [2][8][2] per-row partial dots
  float* red1 = red + 32;           // [8] rmsnorm scratch

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = D / E;  // 16-byte chunks per row

  int n = n_rows_dev ? *n_rows_dev : n_rows_host;
  if (n > list_cap) n = list_cap;
  if (n < 0) n = 0;
  const int my_n = (n > (int)blockIdx.x) ? (n - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < n_stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t pol = policy_evict_first();
  auto issue = [&](int j) {
    const int s = j % n_stages;
    const int i = (int)blockIdx.x + j * (int)gridDim.x;
    int r = row_list ? row_list[i] : i;
    if ((unsigned)r >= (unsigned)row_limit) {
      atomicExch(err, kDevErrBounds);
      r = 0;
    }
    unsigned char* dst = stages + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&bars[s], stage_bytes);
    int p = 0;
    if (GATED) bulk_load(dst + (p++) * row_bytes, w_gate + (size_t)r * D, row_bytes, &bars[s], pol);
    bulk_load(dst + (p++) * row_bytes, w_up + (size_t)r * D, row_bytes, &bars[s], pol);
    bulk_load(dst + p * row_bytes, w_down + (size_t)r * D, row_bytes, &bars[s], pol);
  };
  if (tid == 0) {
    const int pre = my_n < n_stages ? my_n : n_stages;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  // x = rmsnorm(h_in) while the first rows stream in.
  rmsnorm_to_smem(h_in, xs, D, red1);
  float xr[kMaxChunksPerThread][E];
  float acc[kMaxChunksPerThread][E];
#pragma unroll
  for (int k = 0; k < kMaxChunksPerThread; ++k) {
    const int c = tid + k * kThreads;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      xr[k][e] = (c < NC) ? xs[c * E + e] : 0.f;
      acc[k][e] = 0.f;
    }
  }

  int issued_upto = my_n < n_stages ? my_n : n_stages;
  bool aborted = false;
  for (int j = 0; j < my_n; ++j) {
    const int s = j % n_stages;
    const uint32_t parity = (uint32_t)(j / n_stages) & 1u;
    const bool ok = mbar_wait(&bars[s], parity, err);
    const uint4* st = reinterpret_cast<const uint4*>(stages + (size_t)s * stage_bytes);
    const uint4* st_up = st + (GATED ? NC : 0);
    const uint4* st_dn = st + (GATED ? 2 * NC : NC);
    float pa = 0.f, pb = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxChunksPerThread; ++k) {
      const int c = tid + k * kThreads;
      if (c < NC) {
        float f[E];
        if (GATED) {
          Elem<T>::load(st[c], f);
#pragma unroll
          for (int e = 0; e < E; ++e) pa = fmaf(f[e], xr[k][e], pa);
        }
        Elem<T>::load(st_up[c], f);
#pragma unroll
        for (int e = 0; e < E; ++e) pb = fmaf(f[e], xr[k][e], pb);
      }
    }
    if (GATED) pa = warp_sum(pa);
    pb = warp_sum(pb);
    float* rb = red + (j & 1) * 16;
    if (lane == 0) {
      rb[warp * 2] = pa;
      rb[warp * 2 + 1] = pb;
    }
    if (__syncthreads_or(!ok)) {  // uniform: every thread leaves together
      aborted = true;
      break;
    }
    // every thread is past row j-1: its stage can be refilled
    if (tid == 0 && j >= 1 && j - 1 + n_stages < my_n) {
      issue(j - 1 + n_stages);
      ++issued_upto;
    }
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      a += rb[w * 2];
      b += rb[w * 2 + 1];
    }
    const float hv = GATED ? (a > 0.f ? a : 0.f) * b : (b > 0.f ? b : 0.f);
#pragma unroll
    for (int k = 0; k < kMaxChunksPerThread; ++k) {
      const int c = tid + k * kThreads;
      if (c < NC) {
        float f[E];
        Elem<T>::load(st_dn[c], f);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[k][e] = fmaf(hv, f[e], acc[k][e]);
      }
    }
  }
  if (aborted && tid == 0) {
    // drain copies still in flight before the CTA's shared memory goes away
    const int first = issued_upto > n_stages ? issued_upto - n_stages : 0;
    for (int j = first; j < issued_upto; ++j) mbar_wait(&bars[j % n_stages], (uint32_t)(j / n_stages) & 1u, nullptr);
  }

  float* out = part + (size_t)blockIdx.x * D;
#pragma unroll
  for (int k = 0; k < kMaxChunksPerThread; ++k) {
    const int c = tid + k * kThreads;
    if (c < NC) {
#pragma unroll
      for (int e = 0; e < E; e += 4)
        *reinterpret_cast<float4*>(out + c * E + e) = make_float4(acc[k][e], acc[k][e + 1], acc[k][e + 2], acc[k][e + 3]);
    }
  }
}

// y[j] = sum over CTAs b (in order) of part[b][j]; h_out = h_in + y; y_out = y.
// Block: 256 threads = 8 warps over 32 columns; warp w sums partials w, w+8, ...
__global__ void __launch_bounds__(256) ffn_finish_kernel(const float* __restrict__ part, int n_part, int D,
                                                         const float* h_in, float* h_out, float* y_out) {
  __shared__ float s[8][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + lane;
  float v = 0.f;
  if (j < D)
    for (int b = warp; b < n_part; b += 8) v += part[(size_t)b * D + j];
  s[warp][lane] = v;
  __syncthreads();
  if (warp == 0 && j < D) {
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) y += s[w][lane];
    if (y_out) y_out[j] = y;
    if (h_out) h_out[j] = h_in[j] + y;
  }
}

template <typename T, bool GATED>
static cudaError_t launch_rows_t(const FfnLaunch& a, cudaStream_t st) {
  const size_t smem = ffn_smem_bytes(a.D, a.dtype_bytes, GATED ? 3 : 2, a.n_stages);
  auto kern = ffn_rows_kernel<T, GATED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, kThreads, smem, st>>>(a.h_in, (const T*)a.w_gate, (const T*)a.w_up, (const T*)a.w_down, a.row_list,
                                       a.n_rows_dev, a.n_rows_host, a.list_cap, a.row_limit, a.part, a.D, a.n_stages,
                                       a.err);
  return cudaGetLastError();
}

size_t ffn_smem_bytes(int D, int dtype_bytes, int nproj, int n_stages) {
  return 128 + (size_t)n_stages * nproj * D * dtype_bytes + (size_t)D * 4 + 64 * 4;
}

int ffn_pick_stages(int D, int dtype_bytes, int nproj, size_t smem_limit) {
  int ns = 8;
  while (ns > 2 && ffn_smem_bytes(D, dtype_bytes, nproj, ns) > smem_limit) --ns;
  return ffn_smem_bytes(D, dtype_bytes, nproj, ns) <= smem_limit ? ns : 0;
}

cudaError_t launch_ffn_rows(const FfnLaunch& a, cudaStream_t st) {
  if (a.gated) {
    if (a.dtype == 0) return launch_rows_t<float, true>(a, st);
    if (a.dtype == 1) return launch_rows_t<__half, true>(a, st);
    return launch_rows_t<__nv_bfloat16, true>(a, st);
  }
  if (a.dtype == 0) return launch_rows_t<float, false>(a, st);
  if (a.dtype == 1) return launch_rows_t<__half, false>(a, st);
  return launch_rows_t<__nv_bfloat16, false>(a, st);
}

cudaError_t launch_ffn_finish(const float* part, int n_part, int D, const float* h_in, float* h_out, float* y_out,
                              cudaStream_t st) {
  ffn_finish_kernel<<<(D + 31) / 32, 256, 0, st>>>(part, n_part, D, h_in, h_out, y_out);
  return cudaGetLastError();
}

}  // namespace np
