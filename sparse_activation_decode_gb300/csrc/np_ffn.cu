// FFN over a list of neuron rows, batch 1 (sm_103a).
//
// For each listed row r (a slot of a sparse layer's resident buffers, or a
// neuron of a dense layer):
//     h_r = relu(g_r . x) * (u_r . x)      (or relu(u_r . x) without a gate,
//                                          or silu(g_r . x) * (u_r . x): SwiGLU)
//     y  += h_r * d_r
// with x = rmsnorm(h), h = h_base + y_prev (NeuroPrefetcher full text, delta
// runtime: an active neuron is computed from its own gate, up and down^T
// rows; ReLU-fied form of the activation).  Consecutive layers chain through the
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
#include <mutex>
#include <tuple>
#include <vector>

#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

constexpr int kFfnThreads = 256;                 // consumer threads of the per-layer kernel
constexpr int kFfnWarps = kFfnThreads / 32;      // consumer warps
constexpr int kFfnBlock = kFfnThreads + 32;      // plus one producer warp
constexpr int kChainThreads = 512;               // consumer threads of the persistent chain
constexpr int kChainReaders = 64;                // host-store reader threads of the persistent chain
constexpr int kChainBlock = kChainThreads + 32 + kChainReaders;
constexpr int kChainGroup = 4;                   // rows per block barrier in the chain (2 for wide rows)
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

// Named barrier 1 over the NT consumer threads (the producer warp never joins).
template <int NT> __device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// The same barrier, also ORing a predicate: every consumer gets the answer.
template <int NT> __device__ __forceinline__ bool consumer_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(NT)
      : "memory");
  return r != 0;
}

// silu(v) = v * sigmoid(v), the SwiGLU gate
__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }


// ---------------------------------------------------------------------------
// Pieces shared by the per-layer kernel and the persistent chain kernel.
// ---------------------------------------------------------------------------
// x = rmsnorm(h_in + yprev) into registers: consumer thread t holds the
// chunks t, t+NT, ... it multiplies.  A writer CTA also stores h (hb_out)
// and clears y_zero.
template <typename T, int MAXC, int NT>
__device__ __forceinline__ void load_x(const float* __restrict__ h_in, const float* __restrict__ yprev,
                                       float* hb_out, float* y_zero, bool writer, int D,
                                       float2 (&xr)[MAXC][Pairs<T>::N], float* red) {
  constexpr int P = Pairs<T>::N, E = 2 * P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = D / E;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < MAXC; ++k) {
    const int c = tid + k * NT;
#pragma unroll
    for (int q = 0; q < P; q += 2) {  // 16-byte loads: two pairs at a time
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < NC) {
        v = *reinterpret_cast<const float4*>(h_in + c * E + 2 * q);
        if (yprev) {
          const float4 w = *reinterpret_cast<const float4*>(yprev + c * E + 2 * q);
          v.x += w.x;
          v.y += w.y;
          v.z += w.z;
          v.w += w.w;
        }
        if (writer) {
          if (hb_out) *reinterpret_cast<float4*>(hb_out + c * E + 2 * q) = v;
          if (y_zero) *reinterpret_cast<float4*>(y_zero + c * E + 2 * q) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      xr[k][q] = make_float2(v.x, v.y);
      xr[k][q + 1] = make_float2(v.z, v.w);
      ss = fmaf(v.x, v.x, fmaf(v.y, v.y, ss));
      ss = fmaf(v.z, v.z, fmaf(v.w, v.w, ss));
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  consumer_sync<NT>();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) tot += red[w];
  const float inv = rsqrtf(tot / (float)D + 1e-6f);
#pragma unroll
  for (int k = 0; k < MAXC; ++k)
#pragma unroll
    for (int q = 0; q < P; ++q) {
      xr[k][q].x *= inv;
      xr[k][q].y *= inv;
    }
  consumer_sync<NT>();  // red is reused by the rows
}

// A group of up to GR records (rr[0..nrow) in shared memory): GR gate and up
// dot products per thread, reduce-scattered over each warp, one named
// barrier (that also ORs !ok) to publish the warps' partials, then every warp
// adds the partials itself, forms the GR activations and applies the down
// projection to its chunks.  Returns false, for every consumer alike, if
// any thread's record never arrived.  `grp` alternates the halves of `red`.
template <typename T, bool GATED, int MAXC, int NT, int GR>
__device__ __forceinline__ bool consume_group(const uint4* __restrict__ sm4, const int (&off)[GR], int nrow, bool ok,
                                              int grp, int NC, const float2 (&xr)[MAXC][Pairs<T>::N],
                                              float2 (&acc)[MAXC][Pairs<T>::N], float* red, bool swiglu) {
  constexpr int P = Pairs<T>::N;
  constexpr int NPROJ = GATED ? 3 : 2;
  constexpr int NV = (GATED ? 2 : 1) * GR;  // dot products per group
  constexpr int NW = NT / 32;
  static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "values per group must be a power of two");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float2 d2[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) d2[v] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < MAXC; ++k) {
    const int c = tid + k * NT;
    if (c < NC) {
      float2 f[P];
#pragma unroll
      for (int r = 0; r < GR; ++r) {
        if (r < nrow) {
          if (GATED) {
            Pairs<T>::load(sm4[off[r] + c], f);
#pragma unroll
            for (int q = 0; q < P; ++q) d2[2 * r] = ffma2(f[q], xr[k][q], d2[2 * r]);
            Pairs<T>::load(sm4[off[r] + NC + c], f);
#pragma unroll
            for (int q = 0; q < P; ++q) d2[2 * r + 1] = ffma2(f[q], xr[k][q], d2[2 * r + 1]);
          } else {
            Pairs<T>::load(sm4[off[r] + c], f);
#pragma unroll
            for (int q = 0; q < P; ++q) d2[r] = ffma2(f[q], xr[k][q], d2[r]);
          }
        }
      }
    }
  }
  // warp reduce-scatter: the lanes with (lane & (32/NV - 1)) == 0 end with
  // the warp sum of value vi(lane)
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
  float* rb = red + (grp & 1) * NW * NV;
  if ((lane & (32 / NV - 1)) == 0) rb[warp * NV + vi] = pv[0];
  if (consumer_sync_or<NT>(!ok)) return false;  // a copy never arrived: all consumers stop
  // lane v < NV adds value v over the warps (fixed order), then the
  // activations go to every lane
  float tot = 0.f;
  if (lane < NV) {
#pragma unroll
    for (int w = 0; w < NW; ++w) tot += rb[w * NV + lane];
  }
  float hv[GR];
#pragma unroll
  for (int r = 0; r < GR; ++r) {
    if (GATED) {
      const float g = __shfl_sync(0xffffffffu, tot, 2 * r);
      const float u = __shfl_sync(0xffffffffu, tot, 2 * r + 1);
      hv[r] = (swiglu ? silu(g) : (g > 0.f ? g : 0.f)) * u;
    } else {
      const float u = __shfl_sync(0xffffffffu, tot, r);
      hv[r] = u > 0.f ? u : 0.f;
    }
  }
  const int dn = (NPROJ - 1) * NC;
#pragma unroll
  for (int k = 0; k < MAXC; ++k) {
    const int c = tid + k * NT;
    if (c < NC) {
      float2 f[P];
#pragma unroll
      for (int r = 0; r < GR; ++r) {
        if (r < nrow) {
          const float2 h2 = make_float2(hv[r], hv[r]);
          Pairs<T>::load(sm4[off[r] + dn + c], f);
#pragma unroll
          for (int q = 0; q < P; ++q) acc[k][q] = ffma2(h2, f[q], acc[k][q]);
        }
      }
    }
  }
  return true;
}

// The same group computation, but every chunk of the group's records (gate,
// up and down^T) is read into registers first and the slots are released
// right away (one arrive per warp on each slot's `empty` barrier), so the
// producer refills them while this group's reduction and down projection
// run.
//
// Each row's slot is waited for, read and released on its own (per warp), so
// a slot goes back to the producer as soon as its row is in registers.
template <typename T, bool GATED, int MAXC, int NT, int GR>
__device__ __forceinline__ bool consume_group_early(const uint4* __restrict__ sm4, const int (&off)[GR],
                                                    const int (&slot)[GR], const uint32_t (&par)[GR],
                                                    uint64_t* full, uint64_t* empty, int nrow, int* err, int grp,
                                                    int NC, const float2 (&xr)[MAXC][Pairs<T>::N],
                                                    float2 (&acc)[MAXC][Pairs<T>::N], float* red, bool swiglu) {
  constexpr int P = Pairs<T>::N;
  constexpr int NPROJ = GATED ? 3 : 2;
  constexpr int NV = (GATED ? 2 : 1) * GR;
  constexpr int NW = NT / 32;
  static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "values per group must be a power of two");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  bool ok = true;
  uint4 w[GR][NPROJ][MAXC];
#pragma unroll
  for (int r = 0; r < GR; ++r) {
    const bool have = r < nrow;
    if (have) ok = mbar_wait(&full[slot[r]], par[r], err) && ok;
#pragma unroll
    for (int p = 0; p < NPROJ; ++p)
#pragma unroll
      for (int k = 0; k < MAXC; ++k) {
        const int c = tid + k * NT;
        w[r][p][k] = (have && c < NC) ? sm4[off[r] + p * NC + c] : make_uint4(0u, 0u, 0u, 0u);
      }
    if (have) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot[r]]);
    }
  }
  float2 d2[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) d2[v] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < MAXC; ++k) {
    float2 f[P];
#pragma unroll
    for (int r = 0; r < GR; ++r) {
      if (GATED) {
        Pairs<T>::load(w[r][0][k], f);
#pragma unroll
        for (int q = 0; q < P; ++q) d2[2 * r] = ffma2(f[q], xr[k][q], d2[2 * r]);
        Pairs<T>::load(w[r][1][k], f);
#pragma unroll
        for (int q = 0; q < P; ++q) d2[2 * r + 1] = ffma2(f[q], xr[k][q], d2[2 * r + 1]);
      } else {
        Pairs<T>::load(w[r][0][k], f);
#pragma unroll
        for (int q = 0; q < P; ++q) d2[r] = ffma2(f[q], xr[k][q], d2[r]);
      }
    }
  }
  float pv[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) pv[v] = d2[v].x + d2[v].y;
  int cnt = NV, vi = 0;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (cnt > 1) {
      const bool up = (lane & o) != 0;
      const int half = cnt >> 1;
#pragma unroll
      for (int q = 0; q < NV / 2; ++q) {
        if (q < half) {
          const float send = up ? pv[q] : pv[q + half];
          const float keep = up ? pv[q + half] : pv[q];
          pv[q] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      vi = vi * 2 + (up ? 1 : 0);
      cnt = half;
    } else {
      pv[0] += __shfl_xor_sync(0xffffffffu, pv[0], o);
    }
  }
  float* rb = red + (grp & 1) * NW * NV;
  if ((lane & (32 / NV - 1)) == 0) rb[warp * NV + vi] = pv[0];
  if (consumer_sync_or<NT>(!ok)) return false;
  float tot = 0.f;
  if (lane < NV) {
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) tot += rb[ww * NV + lane];
  }
#pragma unroll
  for (int r = 0; r < GR; ++r) {
    float hv;
    if (GATED) {
      const float g = __shfl_sync(0xffffffffu, tot, 2 * r);
      const float u = __shfl_sync(0xffffffffu, tot, 2 * r + 1);
      hv = (swiglu ? silu(g) : (g > 0.f ? g : 0.f)) * u;
    } else {
      const float u = __shfl_sync(0xffffffffu, tot, r);
      hv = u > 0.f ? u : 0.f;
    }
    const float2 h2 = make_float2(hv, hv);
#pragma unroll
    for (int k = 0; k < MAXC; ++k) {
      float2 f[P];
      Pairs<T>::load(w[r][NPROJ - 1][k], f);  // zero chunks add nothing
#pragma unroll
      for (int q = 0; q < P; ++q) acc[k][q] = ffma2(h2, f[q], acc[k][q]);
    }
  }
  return true;
}

// This CTA's partial y into the layer's accumulator (vector atomics).
template <typename T, int MAXC, int NT>
__device__ __forceinline__ void add_partial_y(const float2 (&acc)[MAXC][Pairs<T>::N], float* y_acc, int NC) {
  constexpr int P = Pairs<T>::N, E = 2 * P;
  const int tid = threadIdx.x;
#pragma unroll
  for (int k = 0; k < MAXC; ++k) {
    const int c = tid + k * NT;
    if (c < NC) {
#pragma unroll
      for (int q = 0; q < P; q += 2)
        atomicAdd(reinterpret_cast<float4*>(y_acc + c * E + 2 * q),
                  make_float4(acc[k][q].x, acc[k][q].y, acc[k][q + 1].x, acc[k][q + 1].y));
    }
  }
}

template <typename T, bool GATED, int MAXC>
__global__ void __launch_bounds__(kFfnBlock, 2) ffn_rows_kernel(FfnLaunch a) {
  constexpr int P = Pairs<T>::N;      // float pairs per 16-byte chunk
  constexpr int E = 2 * P;            // elements per chunk
  constexpr int NPROJ = GATED ? 3 : 2;
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
      int s = 0;
      uint32_t wrap = 0;  // ring position without divisions: slot s, pass `wrap`
      for (int j = 0; j < my_n; ++j) {
        if (wrap > 0 && !mbar_wait(&empty[s], (wrap - 1) & 1u, a.err)) {
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
        if (++s == n_slots) {
          s = 0;
          ++wrap;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // x = rmsnorm(h_in + yprev), once the previous kernel's writes are
    // visible; CTA 0 stores h for the next layer and clears the accumulator
    // after next.
    grid_dependency_wait();
    float2 xr[MAXC][P];
    load_x<T, MAXC, kFfnThreads>(a.h_in, a.yprev, a.hb_out, a.y_zero, blockIdx.x == 0, D, xr, red);
    int cs = 0;
    uint32_t cwrap = 0;  // ring position of row j: slot cs, pass cwrap
    for (int j = 0; j < my_n; j += 2) {
      const bool two = j + 1 < my_n;
      const int s0 = cs;
      const bool w1 = cs + 1 == n_slots;
      const int s1 = w1 ? 0 : cs + 1;
      bool ok = mbar_wait(&full[s0], cwrap & 1u, a.err);
      if (two) ok = mbar_wait(&full[s1], (cwrap + (w1 ? 1u : 0u)) & 1u, a.err) && ok;
      if (two) {
        cs = w1 ? 1 : (cs + 2 == n_slots ? 0 : cs + 2);
        cwrap += (w1 || cs == 0) ? 1u : 0u;
      } else {
        cs = w1 ? 0 : cs + 1;
        cwrap += w1 ? 1u : 0u;
      }
      const int off[2] = {(int)((512 + (size_t)s0 * slot_bytes) >> 4), (int)((512 + (size_t)s1 * slot_bytes) >> 4)};
      if (!consume_group<T, GATED, MAXC, kFfnThreads, 2>(reinterpret_cast<const uint4*>(smem), off, two ? 2 : 1, ok,
                                                          j >> 1, NC, xr, acc, red, a.swiglu != 0)) {
        if (tid == 0) s_abort = 1;
        break;
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
  if (tid < kFfnThreads && !s_abort) add_partial_y<T, MAXC, kFfnThreads>(acc, a.y_acc, NC);
}

// ---------------------------------------------------------------------------
// Persistent chain over consecutive layers (np_ffn_layers, batch 1).  One
// cooperative launch, one CTA per SM.  The producer streams every layer's
// records without a break (the weights do not depend on h); the consumers
// of layer i wait until every CTA has added its part of layer i-1 (an
// arrival counter per layer, bounded spin) and then read h.  The ring keeps
// the copies going while the consumers wait, so the per-layer barrier costs
// little bandwidth.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until *cnt reaches `target` (bounded: about one second).
__device__ __forceinline__ bool wait_count(const unsigned* cnt, unsigned target, int* err) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_u32(cnt) >= target) return true;
    if ((it & 63u) == 63u && global_ns() - t0 > kWaitLimitNs) {
      atomicExch(err, kDevErrTimeout);
      return false;
    }
  }
}

template <typename T, bool GATED, int MAXC>
__global__ void __launch_bounds__(kChainBlock, 1) ffn_chain_kernel(FfnChainLaunch a) {
  constexpr int P = Pairs<T>::N;
  constexpr int E = 2 * P;
  constexpr int NPROJ = GATED ? 3 : 2;
  // rows per block barrier: a group's rows sit in registers, so rows of
  // several chunks per thread come two or one at a time
  constexpr int GRP = MAXC == 1 ? kChainGroup : (MAXC == 2 ? 2 : 1);
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [16]
  uint64_t* empty = full + 16;                           // [16]
  const int D = a.D, n_slots = a.n_stages;
  const uint32_t row_bytes = (uint32_t)D * sizeof(T);
  const uint32_t slot_bytes = NPROJ * row_bytes;
  unsigned char* ring = smem + 512;
  float* red = reinterpret_cast<float*>(ring + (size_t)n_slots * slot_bytes);
  __shared__ int s_abort, s_issued;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int NC = D / E;
  const int G = (int)gridDim.x;
  const size_t BD = (size_t)D;
  const int n_slices = (D + 31) / 32;            // 32-column slices of y
  const int n_red = n_slices < G ? n_slices : G;  // CTAs that sum slices

  // layer i of the chain: weights, rows and this CTA's share of them
  auto layer_rows = [&](int i, const T** wg, const T** wu, const T** wd, const int** list, int* limit) -> int {
    const int l = a.first + i;
    const unsigned char* base;
    size_t proj;
    int n;
    if (l < a.n_dense) {
      proj = (size_t)a.F * row_bytes;
      base = static_cast<const unsigned char*>(a.dense_w) + (size_t)l * NPROJ * proj;
      *list = nullptr;
      n = a.F;
      *limit = a.F;
    } else {
      const int s = l - a.n_dense;
      proj = (size_t)a.K * row_bytes;
      base = static_cast<const unsigned char*>(a.bufs) + (size_t)s * NPROJ * proj;
      // compact placement: the occupied region [0, n_rows); else the active rows
      *list = a.compact ? nullptr : a.active_slot + (size_t)s * a.K;
      n = a.compact ? a.n_rows[s] : a.counts[(size_t)s * 4];
      n = n < 0 ? 0 : (n > a.K ? a.K : n);
      *limit = a.K;
    }
    int p = 0;
    *wg = GATED ? reinterpret_cast<const T*>(base + (p++) * proj) : nullptr;
    *wu = reinterpret_cast<const T*>(base + (p++) * proj);
    *wd = reinterpret_cast<const T*>(base + p * proj);
    return n > (int)blockIdx.x ? (n - 1 - (int)blockIdx.x) / G + 1 : 0;
  };

  if (tid == 0) {
    for (int s = 0; s < n_slots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kChainThreads / 32);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
  }
  __syncthreads();

  if (warp == kChainThreads / 32) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the rows: each lane fetches one of the next 32
    // row indices, lane 0 takes them by shuffle and issues the copies, so no
    // index load sits on the issue path.
    const uint64_t pol = policy_evict_first();
    int j = 0;
    int ps = 0;          // slot of row j
    uint32_t pwrap = 0;  // passes over the ring so far
    bool stop = false;
    for (int i = 0; i < a.count && !stop; ++i) {
      const T *wg, *wu, *wd;
      const int* list;
      int limit;
      const int my_n = layer_rows(i, &wg, &wu, &wd, &list, &limit);
      if (a.g_store && a.first + i >= a.n_dense) {
        // every CTA has written this layer's incoming rows: the async-proxy
        // reads below must see those generic-proxy writes
        int fail = 0;
        if (lane == 0) {
          fail = wait_count(a.gdone + i, (unsigned)G, a.err) ? 0 : 1;
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        if (__shfl_sync(0xffffffffu, fail, 0)) {
          if (lane == 0) s_abort = 1;
          stop = true;
          break;
        }
      }
      for (int b0 = 0; b0 < my_n && !stop; b0 += 32) {
        int mine = 0;
        if (b0 + lane < my_n) {
          mine = list ? list[blockIdx.x + (b0 + lane) * G] : (int)blockIdx.x + (b0 + lane) * G;
          if ((unsigned)mine >= (unsigned)limit) {
            atomicExch(a.err, kDevErrBounds);
            mine = 0;
          }
        }
        const int cnt = my_n - b0 < 32 ? my_n - b0 : 32;
        for (int q = 0; q < cnt; ++q, ++j) {
          const int r = __shfl_sync(0xffffffffu, mine, q);
          int fail = 0;
          if (lane == 0) {
            const int s = ps;
            if (pwrap > 0 && !mbar_wait(&empty[s], (pwrap - 1) & 1u, a.err)) {
              fail = 1;
            } else {
              unsigned char* dst = ring + (size_t)s * slot_bytes;
              mbar_arrive_expect_tx(&full[s], slot_bytes);
              int p = 0;
              if (GATED) bulk_load(dst + (p++) * row_bytes, wg + (size_t)r * D, row_bytes, &full[s], pol);
              bulk_load(dst + (p++) * row_bytes, wu + (size_t)r * D, row_bytes, &full[s], pol);
              bulk_load(dst + p * row_bytes, wd + (size_t)r * D, row_bytes, &full[s], pol);
              s_issued = j + 1;
            }
          }
          if (++ps == n_slots) {
            ps = 0;
            ++pwrap;
          }
          if (__shfl_sync(0xffffffffu, fail, 0)) {
            if (lane == 0) s_abort = 1;
            stop = true;
            break;
          }
        }
      }
    }
  } else if (warp > kChainThreads / 32) {
    // ------------------------------------------------------------ readers
    // Incoming records of each sparse layer, straight from the host store
    // into their slots (CTA c takes records c, c + G, ...); the rows of a
    // record are copied by the reader threads with eight 16-byte loads in
    // flight each.  Once a CTA's readers are done with a layer, one release
    // per CTA counts it in gdone.  They run ahead of the FFNs, bounded only
    // by the host link.
    if (a.g_store) {
      constexpr int kIlpR = 8;
      const int rt = tid - (kChainThreads + 32);
      const int row_vec = (int)(row_bytes / 16u);
      const int rec_vec = NPROJ * row_vec;
      for (int i = 0; i < a.count; ++i) {
        const int l = a.first + i;
        if (l < a.n_dense) continue;
        const int s = l - a.n_dense;
        int n_in = a.counts[(size_t)s * 4 + 1];
        n_in = n_in < 0 ? 0 : (n_in > a.K ? a.K : n_in);
        const uint4* store = static_cast<const uint4*>(a.g_store) + (size_t)s * a.F * rec_vec;
        uint4* bufs = reinterpret_cast<uint4*>(const_cast<void*>(a.bufs)) + (size_t)s * NPROJ * a.K * row_vec;
        for (int r = (int)blockIdx.x; r < n_in; r += G) {
          const int n = a.din_n[(size_t)s * a.K + r], slot = a.din_s[(size_t)s * a.K + r];
          if ((unsigned)n >= (unsigned)a.F || (unsigned)slot >= (unsigned)a.K) {
            if (rt == 0) atomicExch(a.err, kDevErrBounds);
            continue;
          }
          const uint4* src = store + (size_t)n * rec_vec;
          for (int p = 0; p < NPROJ; ++p) {
            uint4* dst = bufs + ((size_t)p * a.K + slot) * row_vec;
            for (int b = rt; b < row_vec; b += kChainReaders * kIlpR) {
              uint4 v[kIlpR];
#pragma unroll
              for (int u = 0; u < kIlpR; ++u) {
                const int j = b + u * kChainReaders;
                if (j < row_vec) v[u] = src[(size_t)p * row_vec + j];
              }
#pragma unroll
              for (int u = 0; u < kIlpR; ++u) {
                const int j = b + u * kChainReaders;
                if (j < row_vec) dst[j] = v[u];
              }
            }
          }
        }
        // the rows written by every reader of this CTA, then one arrival
        asm volatile("fence.proxy.async.global;" ::: "memory");
        asm volatile("bar.sync 2, %0;" ::"n"(kChainReaders) : "memory");
        if (rt == 0 && !(i == a.withhold && blockIdx.x == 0)) {
          __threadfence();
          atomicAdd(a.gdone + i, 1u);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    int cs = 0;          // slot of the next row
    uint32_t cwrap = 0;  // passes over the ring so far
    for (int i = 0; i < a.count; ++i) {
      if (i > 0) {  // every slice of y(i-1) has been summed
        bool ok = true;
        if (tid == 0) ok = wait_count(a.arrive + 2 * (i - 1) + 1, (unsigned)n_red, a.err);
        if (consumer_sync_or<kChainThreads>(!ok)) {
          if (tid == 0) s_abort = 1;
          break;
        }
      }
      const float* hb = i <= 1 ? a.h : a.hbase + (size_t)((i - 1) & 1) * BD;
      const float* yp = i == 0 ? nullptr : a.yacc + (size_t)((i - 1) % 3) * BD;
      float* hb_out = i >= 1 ? a.hbase + (size_t)(i & 1) * BD : nullptr;
      float* yi = a.yacc + (size_t)(i % 3) * BD;
      float2 xr[MAXC][P];
      load_x<T, MAXC, kChainThreads>(hb, yp, hb_out, nullptr, blockIdx.x == 0, D, xr, red);
      float2 acc[MAXC][P];
#pragma unroll
      for (int k = 0; k < MAXC; ++k)
#pragma unroll
        for (int q = 0; q < P; ++q) acc[k][q] = make_float2(0.f, 0.f);
      const T *wg, *wu, *wd;
      const int* list;
      int limit;
      const int my_n = layer_rows(i, &wg, &wu, &wd, &list, &limit);
      bool aborted = false;
      for (int jj = 0; jj < my_n; jj += GRP) {
        const int nrow = my_n - jj < GRP ? my_n - jj : GRP;
        int off[GRP], slot[GRP];
        uint32_t par[GRP];
#pragma unroll
        for (int r = 0; r < GRP; ++r) {
          slot[r] = cs;
          par[r] = cwrap & 1u;
          off[r] = (int)((512 + (size_t)cs * slot_bytes) >> 4);
          if (r < nrow) {
            if (++cs == n_slots) {
              cs = 0;
              ++cwrap;
            }
          }
        }
        if (!consume_group_early<T, GATED, MAXC, kChainThreads, GRP>(
                reinterpret_cast<const uint4*>(smem), off, slot, par, full, empty, nrow, a.err, jj / GRP, NC,
                xr, acc, red, a.swiglu != 0)) {
          aborted = true;
          break;
        }
      }
      if (aborted) {
        if (tid == 0) s_abort = 1;
        break;
      }
      // split-K in two fixed-order steps: every CTA stores its partial y;
      // once all have, CTA r sums column slice r over the CTAs in order
      {
        float* mine = a.part + (size_t)blockIdx.x * BD;
#pragma unroll
        for (int k = 0; k < MAXC; ++k) {
          const int c = tid + k * kChainThreads;
          if (c < NC)
#pragma unroll
            for (int q = 0; q < P; q += 2)
              *reinterpret_cast<float4*>(mine + c * E + 2 * q) =
                  make_float4(acc[k][q].x, acc[k][q].y, acc[k][q + 1].x, acc[k][q + 1].y);
        }
      }
      // one release per CTA: the barrier orders every thread's stores before
      // thread 0's fence, which makes them visible before its arrival
      consumer_sync<kChainThreads>();
      if (tid == 0) {
        __threadfence();
        atomicAdd(a.arrive + 2 * i, 1u);
      }
      if ((int)blockIdx.x < n_red) {
        bool ok = true;
        if (tid == 0) ok = wait_count(a.arrive + 2 * i, (unsigned)G, a.err);
        if (consumer_sync_or<kChainThreads>(!ok)) {
          if (tid == 0) s_abort = 1;
          break;
        }
        float4* tmp = reinterpret_cast<float4*>(red + 64);  // [64][8]
        const int f = tid & 7, g = tid >> 3;
        for (int sl = (int)blockIdx.x; sl < n_slices; sl += G) {
          // threads (g, f): float4 f of the slice, partials g, g + 64, ...
          const int col = sl * 32 + 4 * f;
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
          if (col < D) {
            // the first three partials of this thread in flight together
            constexpr int GS = kChainThreads / 8;
            float4 v[3];
#pragma unroll
            for (int u = 0; u < 3; ++u) {
              const int cta = g + u * GS;
              v[u] = cta < G ? __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)cta * BD + col))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 3; ++u) {
              sum.x += v[u].x; sum.y += v[u].y; sum.z += v[u].z; sum.w += v[u].w;
            }
            for (int cta = g + 3 * GS; cta < G; cta += GS) {
              const float4 w = __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)cta * BD + col));
              sum.x += w.x; sum.y += w.y; sum.z += w.z; sum.w += w.w;
            }
          }
          tmp[g * 8 + f] = sum;
          consumer_sync<kChainThreads>();
          if (warp == 0) {
            // lane (part, f): every fourth group, then the four parts in a
            // fixed tree (both lanes of a pair get the same, commutative sum)
            const int f2 = lane & 7, part = lane >> 3;
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int gg = part; gg < kChainThreads / 8; gg += 4) {
              const float4 v = tmp[gg * 8 + f2];
              t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
            }
#pragma unroll
            for (int o = 8; o <= 16; o <<= 1) {
              t.x += __shfl_xor_sync(0xffffffffu, t.x, o);
              t.y += __shfl_xor_sync(0xffffffffu, t.y, o);
              t.z += __shfl_xor_sync(0xffffffffu, t.z, o);
              t.w += __shfl_xor_sync(0xffffffffu, t.w, o);
            }
            if (lane < 8 && sl * 32 + 4 * lane < D) *reinterpret_cast<float4*>(yi + sl * 32 + 4 * lane) = t;
          }
          consumer_sync<kChainThreads>();  // tmp is reused by the next slice
        }
        consumer_sync<kChainThreads>();
        if (tid == 0) {
          __threadfence();
          atomicAdd(a.arrive + 2 * i + 1, 1u);
        }
      }
    }
    // the residual stream after the last layer: h = h_last + y_last
    if (blockIdx.x == 0 && !s_abort) {
      bool ok = true;
      if (tid == 0) ok = wait_count(a.arrive + 2 * (a.count - 1) + 1, (unsigned)n_red, a.err);
      if (!consumer_sync_or<kChainThreads>(!ok)) {
        const int i = a.count - 1;
        const float* hl = i == 0 ? a.h : a.hbase + (size_t)(i & 1) * BD;
        const float* yl = a.yacc + (size_t)(i % 3) * BD;
        for (int d = tid; d < D; d += kChainThreads) a.h[d] = hl[d] + yl[d];
      }
    }
  }
  __syncthreads();
  if (s_abort && tid == kChainThreads) {
    atomicExch(a.err, kDevErrTimeout);
    const int issued = s_issued;
    const int first = issued > n_slots ? issued - n_slots : 0;
    for (int j = first; j < issued; ++j) mbar_wait(&full[j % n_slots], (uint32_t)(j / n_slots) & 1u, nullptr);
  }
}

template <typename T, bool GATED>
static void* chain_kernel_for(int maxc) {
  switch (maxc) {
    case 1: return reinterpret_cast<void*>(ffn_chain_kernel<T, GATED, 1>);
    case 2: return reinterpret_cast<void*>(ffn_chain_kernel<T, GATED, 2>);
    case 3: return reinterpret_cast<void*>(ffn_chain_kernel<T, GATED, 3>);
    default: return reinterpret_cast<void*>(ffn_chain_kernel<T, GATED, 4>);
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

static void* pick_chain_kernel(int dtype, bool gated, int D, int dtype_bytes) {
  const int mc = (D * dtype_bytes / 16 + kChainThreads - 1) / kChainThreads;
  if (gated)
    return dtype == 0 ? chain_kernel_for<float, true>(mc)
                      : dtype == 1 ? chain_kernel_for<__half, true>(mc) : chain_kernel_for<__nv_bfloat16, true>(mc);
  return dtype == 0 ? chain_kernel_for<float, false>(mc)
                    : dtype == 1 ? chain_kernel_for<__half, false>(mc) : chain_kernel_for<__nv_bfloat16, false>(mc);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` unless it is
// already at least that on this device.  The limit is per kernel, not per
// model, so it never goes down: a model planned later with smaller rings
// leaves the launches of a model planned earlier valid.
static cudaError_t raise_smem(const void* k, size_t bytes) {
  static std::mutex mu;
  static std::vector<std::tuple<const void*, int, size_t>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& t : done)
    if (std::get<0>(t) == k && std::get<1>(t) == dev) {
      if (bytes <= std::get<2>(t)) return cudaSuccess;
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (e == cudaSuccess) std::get<2>(t) = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.emplace_back(k, dev, bytes);
  return e;
}

size_t ffn_smem_bytes(int D, int dtype_bytes, int nproj, int n_stages) {
  return 512 + (size_t)n_stages * nproj * D * dtype_bytes + 1024;  // barriers/rows, ring, partial sums
}

// the chain kernel also sums y slices in shared memory: 64 x 8 float4 more
static size_t chain_smem_bytes(int D, int dtype_bytes, int nproj, int n_stages) {
  return ffn_smem_bytes(D, dtype_bytes, nproj, n_stages) + 256 + 64 * 8 * 16;
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
  cudaError_t e = raise_smem(k, smem);
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
  return raise_smem(k, ffn_smem_bytes(D, dtype_bytes, gated ? 3 : 2, n_stages));
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
  cfg.numAttrs = a.pdl ? 1 : 0;
  FfnLaunch arg = a;
  void* params[] = {&arg};
  return cudaLaunchKernelExC(&cfg, k, params);
}

cudaError_t ffn_chain_plan(int dtype, int gated, int D, int dtype_bytes, size_t smem_optin, int n_sms,
                           int* n_stages, int* grid) {
  const int nproj = gated ? 3 : 2;
  int ns = 16;  // one CTA per SM with as many ring slots as fit
  while (ns > 2 && chain_smem_bytes(D, dtype_bytes, nproj, ns) > smem_optin) --ns;
  const size_t smem = chain_smem_bytes(D, dtype_bytes, nproj, ns);
  if (smem > smem_optin) return cudaErrorInvalidValue;
  void* k = pick_chain_kernel(dtype, gated != 0, D, dtype_bytes);
  cudaError_t e = raise_smem(k, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kChainBlock, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  *n_stages = ns;
  *grid = n_sms;  // every CTA co-resident (cooperative launch)
  return cudaSuccess;
}

cudaError_t launch_ffn_chain(const FfnChainLaunch& a, cudaStream_t st) {
  void* k = pick_chain_kernel(a.dtype, a.gated != 0, a.D, a.dtype_bytes);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid, 1, 1);
  cfg.blockDim = dim3(kChainBlock, 1, 1);
  cfg.dynamicSmemBytes = chain_smem_bytes(a.D, a.dtype_bytes, a.gated ? 3 : 2, a.n_stages);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  FfnChainLaunch arg = a;
  void* params[] = {&arg};
  return cudaLaunchKernelExC(&cfg, k, params);
}

}  // namespace np
