// Incoming-row movement (sm_103a): host weight store -> device staging ->
// projection buffers, and the row moves of the compact placement.
//
// NeuroPrefetcher section 3.5 ("I/O Path") and its full text: incoming
// neuron IDs are sorted and read as neuron-centric records (gate | up |
// down^T rows of one neuron, contiguous in a layer-major file) into a
// capacity-bounded staging buffer; a fused deinterleave-and-scatter kernel
// writes each record's rows into the slot the delta runtime assigned, and a
// delta larger than the staging capacity is processed as independent
// read+scatter chunks.
//
// Here the storage tier is CPU memory that the GPU reads over the host link
// (NVLink-C2C on GB300).  Individual host-to-device copies per record are
// limited by per-call overhead, so the read is a gather kernel: one CTA per
// record, every thread keeping eight 16-byte loads in flight, which
// saturates the link with a few dozen CTAs.  The scatter kernel works in
// device memory and is HBM-bound: one warp per (record, projection row), 16
// loads in flight per lane.
#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

constexpr int kMoveThreads = 256;
constexpr int kIlp = 8;

__device__ __forceinline__ void copy_vecs(const uint4* __restrict__ src, uint4* __restrict__ dst, int n) {
  for (int base = threadIdx.x; base < n; base += kMoveThreads * kIlp) {
    uint4 v[kIlp];
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int j = base + u * kMoveThreads;
      if (j < n) v[u] = src[j];
    }
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int j = base + u * kMoveThreads;
      if (j < n) dst[j] = v[u];
    }
  }
}

// One warp copies n 16-byte vectors, 16 loads in flight per lane.
constexpr int kWarpIlp = 16;
__device__ __forceinline__ void warp_copy(const uint4* __restrict__ src, uint4* __restrict__ dst, int n, int lane) {
  for (int base = lane; base < n; base += 32 * kWarpIlp) {
    uint4 v[kWarpIlp];
#pragma unroll
    for (int u = 0; u < kWarpIlp; ++u) {
      const int j = base + u * 32;
      if (j < n) v[u] = src[j];
    }
#pragma unroll
    for (int u = 0; u < kWarpIlp; ++u) {
      const int j = base + u * 32;
      if (j < n) dst[j] = v[u];
    }
  }
}

__device__ __forceinline__ int chunk_end(const MoveLaunch& a) {
  int cnt = *a.count;
  if (cnt > a.K) cnt = a.K;
  const int end = a.chunk_begin + a.chunk_cap;
  return cnt < end ? cnt : end;
}

// staging[i - begin] = store[din_n[i]] for the chunk's records
__global__ void __launch_bounds__(kMoveThreads) gather_kernel(MoveLaunch a) {
  const int end = chunk_end(a);
  const uint4* store = static_cast<const uint4*>(a.store_layer);
  uint4* stg = static_cast<uint4*>(a.staging);
  for (int i = a.chunk_begin + blockIdx.x; i < end; i += gridDim.x) {
    const int n = a.din_n[i];
    if ((unsigned)n >= (unsigned)a.F) {
      if (threadIdx.x == 0) atomicExch(a.err, kDevErrBounds);
      continue;
    }
    copy_vecs(store + (size_t)n * a.rec_vec, stg + (size_t)(i - a.chunk_begin) * a.rec_vec, a.rec_vec);
  }
}

// bufs[p][din_s[i]] = staging[i - begin].row[p]: one warp per (record, row)
__global__ void __launch_bounds__(kMoveThreads) scatter_kernel(MoveLaunch a) {
  const int end = chunk_end(a);
  const int units = (end - a.chunk_begin) * a.n_proj;
  const uint4* stg = static_cast<const uint4*>(a.staging);
  uint4* bufs = static_cast<uint4*>(a.bufs_layer);
  const int lane = threadIdx.x & 31, wpb = kMoveThreads / 32;
  for (int u = blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += gridDim.x * wpb) {
    const int r = u / a.n_proj, p = u - r * a.n_proj;
    const int slot = a.din_s[a.chunk_begin + r];
    if ((unsigned)slot >= (unsigned)a.K) {
      if (lane == 0) atomicExch(a.err, kDevErrBounds);
      continue;
    }
    warp_copy(stg + (size_t)r * a.rec_vec + (size_t)p * a.row_vec, bufs + ((size_t)p * a.K + slot) * a.row_vec,
              a.row_vec, lane);
  }
}

// store record -> buffers directly (no staging)
__global__ void __launch_bounds__(kMoveThreads) fused_kernel(MoveLaunch a) {
  const int end = chunk_end(a);
  const uint4* store = static_cast<const uint4*>(a.store_layer);
  uint4* bufs = static_cast<uint4*>(a.bufs_layer);
  for (int i = a.chunk_begin + blockIdx.x; i < end; i += gridDim.x) {
    const int n = a.din_n[i], slot = a.din_s[i];
    if ((unsigned)n >= (unsigned)a.F || (unsigned)slot >= (unsigned)a.K) {
      if (threadIdx.x == 0) atomicExch(a.err, kDevErrBounds);
      continue;
    }
    const uint4* src = store + (size_t)n * a.rec_vec;
    for (int p = 0; p < a.n_proj; ++p)
      copy_vecs(src + (size_t)p * a.row_vec, bufs + ((size_t)p * a.K + slot) * a.row_vec, a.row_vec);
  }
}

// Compact placement: bufs[p][mv_dst[i]] = bufs[p][mv_src[i]], one warp per
// (move, projection row).  Sources lie at or above the region's new end and
// targets below it, so no copy reads a row another one writes.
__global__ void __launch_bounds__(kMoveThreads) move_rows_kernel(MoveLaunch a) {
  int cnt = *a.mv_count;
  if (cnt > a.K) cnt = a.K;
  const int units = cnt * a.n_proj;
  uint4* bufs = static_cast<uint4*>(a.bufs_layer);
  const int lane = threadIdx.x & 31, wpb = kMoveThreads / 32;
  for (int u = blockIdx.x * wpb + (threadIdx.x >> 5); u < units; u += gridDim.x * wpb) {
    const int i = u / a.n_proj, p = u - i * a.n_proj;
    const int src = a.mv_src[i], dst = a.mv_dst[i];
    if ((unsigned)src >= (unsigned)a.K || (unsigned)dst >= (unsigned)a.K) {
      if (lane == 0) atomicExch(a.err, kDevErrBounds);
      continue;
    }
    warp_copy(bufs + ((size_t)p * a.K + src) * a.row_vec, bufs + ((size_t)p * a.K + dst) * a.row_vec, a.row_vec,
              lane);
  }
}

// One slot's rows back to the record of neuron n, or zeros (n < 0: the slot
// never held a row).
__device__ __forceinline__ void restore_slot(const MoveLaunch& a, int slot, int n) {
  const uint4* store = static_cast<const uint4*>(a.store_layer);
  uint4* bufs = static_cast<uint4*>(a.bufs_layer);
  for (int p = 0; p < a.n_proj; ++p) {
    uint4* dst = bufs + ((size_t)p * a.K + slot) * a.row_vec;
    if ((unsigned)n < (unsigned)a.F) {
      copy_vecs(store + (size_t)n * a.rec_vec + (size_t)p * a.row_vec, dst, a.row_vec);
    } else {
      for (int j = threadIdx.x; j < a.row_vec; j += kMoveThreads) dst[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Put back what the slots written by this delta held before it: the slots
// assigned to D_in (din_oldct) and, under the compact placement, the move
// targets (mv_oldct).  The two sets of slots are disjoint.
__global__ void __launch_bounds__(kMoveThreads) restore_kernel(MoveLaunch a) {
  const int end = chunk_end(a);
  for (int i = a.chunk_begin + blockIdx.x; i < end; i += gridDim.x) {
    const int slot = a.din_s[i];
    if ((unsigned)slot < (unsigned)a.K) restore_slot(a, slot, a.din_oldct[i]);
  }
  if (a.mv_count) {
    int cnt = *a.mv_count;
    if (cnt > a.K) cnt = a.K;
    for (int i = blockIdx.x; i < cnt; i += gridDim.x) {
      const int slot = a.mv_dst[i];
      if ((unsigned)slot < (unsigned)a.K) restore_slot(a, slot, a.mv_oldct[i]);
    }
  }
}

cudaError_t launch_gather(const MoveLaunch& a, cudaStream_t st) {
  gather_kernel<<<a.grid, kMoveThreads, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_scatter(const MoveLaunch& a, cudaStream_t st) {
  scatter_kernel<<<a.grid, kMoveThreads, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_fused(const MoveLaunch& a, cudaStream_t st) {
  fused_kernel<<<a.grid, kMoveThreads, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_move_rows(const MoveLaunch& a, cudaStream_t st) {
  move_rows_kernel<<<a.grid, kMoveThreads, 0, st>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_restore(const MoveLaunch& a, cudaStream_t st) {
  restore_kernel<<<a.grid, kMoveThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace np
