// Active set, delta and slot assignment for every sparse layer (sm_103a).
//
// One CTA per sparse layer, thread i owns 32-bit word i of the layer's
// neuron bitmasks (F <= 16384).  All set work is bitwise, compaction is a
// block-wide exclusive scan of popcounts, so every output is bit-exact:
//
//  1. A = mask_gate[id_g] (op) mask_up[id_u], op = intersection (NeuroPrefetcher
//     section 3.4) or union, OR-ed over the sequences of a batch; or A = the
//     per-layer predictor's firing mask.
//  2. If |A| > K_max keep the K_max lowest neuron IDs.
//  3. Resident set: R_next = A (slot map, NeuroPrefetcher full text delta
//     runtime), or with windowing (LLM in a flash 3.1) the neurons of R_prev
//     still used within the last W tokens plus A, evicting the oldest last
//     use first (ties: lowest ID first) while more than K_max remain.
//  4. D_in = A \ R_prev, D_out = R_prev \ R_next.  Slots of R_prev ∩ R_next
//     stay; the free slots in ascending order go to D_in in ascending ID
//     order.  New slot map, inverse map and slot contents are written to the
//     other half of the double-buffered state, which becomes the committed
//     state once the rows have been scattered.
#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

constexpr int kSetThreads = 512;
constexpr int kMaxKmax = 8192;

// Exclusive prefix sum of v over the 512-thread block; *total = sum.
__device__ __forceinline__ int block_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSetThreads / 32 ? wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSetThreads / 32) wsum[lane] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? wsum[warp - 1] : 0;
  *total = wsum[kSetThreads / 32 - 1];
  __syncthreads();
  return base + x - v;
}

__device__ __forceinline__ uint32_t lowest_bits(uint32_t w, int m) {
  uint32_t r = 0;
  for (int t = 0; t < m && w; ++t) {
    const uint32_t low = w & (0u - w);
    r |= low;
    w ^= low;
  }
  return r;
}

__global__ void __launch_bounds__(kSetThreads) set_kernel(SetLaunch a) {
  __shared__ int wsum[32];
  __shared__ uint32_t occ[kMaxKmax / 32];
  __shared__ int free_list[kMaxKmax];
  __shared__ int hist[33];
  __shared__ int cut_age, cut_need;

  const int tid = threadIdx.x;
  const int s = a.first_sparse + blockIdx.x;
  const int layer = a.n_dense + s;
  const int F = a.F, K = a.K, W = a.words;
  const int pb = (int)((a.cur_bits >> s) & 1ull), nb = pb ^ 1;
  const size_t S = a.S;
  const int* sm_prev = a.slotmap + ((size_t)pb * S + s) * F;
  int* sm_next = a.slotmap + ((size_t)nb * S + s) * F;
  int* inv_next = a.inv + ((size_t)nb * S + s) * K;
  const int* ct_prev = a.content + ((size_t)pb * S + s) * K;
  int* ct_next = a.content + ((size_t)nb * S + s) * K;
  const uint32_t* res_prev = a.resbits + ((size_t)pb * S + s) * W;
  uint32_t* res_next = a.resbits + ((size_t)nb * S + s) * W;
  const int* ls_prev = a.window > 1 ? a.last_seen + ((size_t)pb * S + s) * F : nullptr;
  int* ls_next = a.window > 1 ? a.last_seen + ((size_t)nb * S + s) * F : nullptr;

  const int i = tid;
  const bool has_word = i < W;
  const uint32_t word_mask =
      (has_word && i == W - 1 && (F & 31)) ? ((1u << (F & 31)) - 1u) : (has_word ? 0xffffffffu : 0u);

  // 1. active set words
  uint32_t aw = 0;
  if (has_word) {
    if (a.ids) {
      for (int b = 0; b < a.batch; ++b) {
        int ig = a.ids[b * a.n_heads + 2 * (layer - 1)];
        int iu = a.ids[b * a.n_heads + 2 * (layer - 1) + 1];
        if ((unsigned)ig >= (unsigned)a.C || (unsigned)iu >= (unsigned)a.C) {
          atomicExch(a.err, kDevErrBounds);
          ig = iu = 0;
        }
        const uint32_t g = a.centroids[(((size_t)s * 2 + 0) * a.C + ig) * W + i];
        const uint32_t u = a.centroids[(((size_t)s * 2 + 1) * a.C + iu) * W + i];
        aw |= a.combine ? (g | u) : (g & u);
      }
    } else {
      aw = a.fire[(size_t)blockIdx.x * W + i];
    }
    aw &= word_mask;
  }

  // 2. cap to the K lowest IDs
  int total;
  int excl = block_scan(__popc(aw), wsum, &total);
  const int dropped = total > K ? total - K : 0;
  if (total > K) {
    if (excl >= K) aw = 0;
    else if (excl + __popc(aw) > K) aw = lowest_bits(aw, K - excl);
  }

  // 3. resident set after this token
  const uint32_t rw = has_word ? res_prev[i] : 0u;
  uint32_t nw = aw;
  if (a.window > 1) {
    // candidates: A plus resident neurons used within the window
    uint32_t old = rw & ~aw;  // resident, not active now
    uint32_t keep_old = 0;
    for (uint32_t w = old; w;) {
      const int b = __ffs(w) - 1;
      w &= w - 1;
      const int n = i * 32 + b;
      const int age = a.token - ls_prev[n];
      if (age >= 0 && age < a.window) keep_old |= 1u << b;
    }
    uint32_t cand = aw | keep_old;
    int ctot;
    (void)block_scan(__popc(cand), wsum, &ctot);
    if (ctot > K) {
      if (tid < 33) hist[tid] = 0;
      __syncthreads();
      for (uint32_t w = keep_old; w;) {
        const int b = __ffs(w) - 1;
        w &= w - 1;
        atomicAdd(&hist[a.token - ls_prev[i * 32 + b]], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int excess = ctot - K, age = a.window - 1;
        while (age > 0 && hist[age] < excess) {
          excess -= hist[age];
          --age;
        }
        cut_age = age;    // evict all older than age, and `excess` lowest IDs of age
        cut_need = excess;
      }
      __syncthreads();
      uint32_t bucket = 0, older = 0;
      for (uint32_t w = keep_old; w;) {
        const int b = __ffs(w) - 1;
        w &= w - 1;
        const int age = a.token - ls_prev[i * 32 + b];
        if (age > cut_age) older |= 1u << b;
        else if (age == cut_age) bucket |= 1u << b;
      }
      int btot;
      const int bexcl = block_scan(__popc(bucket), wsum, &btot);
      uint32_t evict_b = 0;
      if (bexcl < cut_need) evict_b = lowest_bits(bucket, cut_need - bexcl);
      cand &= ~(older | evict_b);
    }
    nw = cand;
  }
  const uint32_t dinw = aw & ~rw;
  const uint32_t doutw = rw & ~nw;
  const uint32_t keptw = rw & nw;

  // 4. compact A, D_in, D_out (ascending IDs)
  int n_a, n_in, n_out;
  const int ea = block_scan(__popc(aw), wsum, &n_a);
  const int ein = block_scan(__popc(dinw), wsum, &n_in);
  const int eout = block_scan(__popc(doutw), wsum, &n_out);
  int* out_a = a.active + (size_t)s * K;
  int* out_in = a.din_n + (size_t)s * K;
  int* out_out = a.dout_n + (size_t)s * K;
  {
    int p = ea;
    for (uint32_t w = aw; w; w &= w - 1) out_a[p++] = i * 32 + __ffs(w) - 1;
    p = ein;
    for (uint32_t w = dinw; w; w &= w - 1) out_in[p++] = i * 32 + __ffs(w) - 1;
    p = eout;
    for (uint32_t w = doutw; w; w &= w - 1) out_out[p++] = i * 32 + __ffs(w) - 1;
  }

  // 5. free slots = [0, K) minus the slots of kept neurons, ascending
  const int KW = (K + 31) / 32;
  if (tid < KW) occ[tid] = 0u;
  __syncthreads();
  for (uint32_t w = keptw; w; w &= w - 1) {
    const int n = i * 32 + __ffs(w) - 1;
    const int slot = sm_prev[n];
    if ((unsigned)slot >= (unsigned)K) {
      atomicExch(a.err, kDevErrBounds);
      continue;
    }
    atomicOr(&occ[slot >> 5], 1u << (slot & 31));
  }
  __syncthreads();
  uint32_t fw = 0;
  if (tid < KW) {
    fw = ~occ[tid];
    if (tid == KW - 1 && (K & 31)) fw &= (1u << (K & 31)) - 1u;
  }
  int n_free;
  const int efree = block_scan(__popc(fw), wsum, &n_free);
  {
    int p = efree;
    for (uint32_t w = fw; w; w &= w - 1) free_list[p++] = tid * 32 + __ffs(w) - 1;
  }
  __syncthreads();
  if (n_in > n_free && tid == 0) atomicExch(a.err, kDevErrBounds);

  // 6. slot map of the next state; D_in slots
  int* out_ins = a.din_s + (size_t)s * K;
  if (has_word) {
    for (int b = 0; b < 32; ++b) {
      const int n = i * 32 + b;
      if (n >= F) break;
      const uint32_t bit = 1u << b;
      int v = -1;
      if (keptw & bit) {
        v = sm_prev[n];
      } else if (dinw & bit) {
        const int r = ein + __popc(dinw & (bit - 1u));
        v = r < n_free ? free_list[r] : 0;
        out_ins[r] = v;
      }
      sm_next[n] = v;
    }
    res_next[i] = nw;
    if (ls_next)
      for (uint32_t w = nw; w; w &= w - 1) {
        const int n = i * 32 + __ffs(w) - 1;
        ls_next[n] = (aw >> (n & 31)) & 1u ? a.token : ls_prev[n];
      }
  }
  // slots of the active neurons, in active-list order
  {
    int* out_as = a.active_slot + (size_t)s * K;
    int p = ea;
    for (uint32_t w = aw; w; w &= w - 1) {
      const int b = __ffs(w) - 1;
      const int n = i * 32 + b;
      int v;
      if ((rw >> b) & 1u) {
        v = sm_prev[n];
      } else {
        const int r = ein + __popc(dinw & ((1u << b) - 1u));
        v = r < n_free ? free_list[r] : 0;
      }
      out_as[p++] = v;
    }
  }
  // inverse map and slot contents of the next state
  for (int k = tid; k < K; k += kSetThreads) {
    inv_next[k] = -1;
    ct_next[k] = ct_prev[k];
  }
  __syncthreads();
  for (uint32_t w = keptw; w; w &= w - 1) {
    const int n = i * 32 + __ffs(w) - 1;
    const int slot = sm_prev[n];
    if ((unsigned)slot < (unsigned)K) inv_next[slot] = n;
  }
  for (uint32_t w = dinw; w; w &= w - 1) {
    const int b = __ffs(w) - 1;
    const int r = ein + __popc(dinw & ((1u << b) - 1u));
    if (r < n_free) {
      const int slot = free_list[r];
      inv_next[slot] = i * 32 + b;
      ct_next[slot] = i * 32 + b;
    }
  }
  if (tid == 0) {
    int* c = a.counts + (size_t)s * 4;
    c[0] = n_a;
    c[1] = n_in;
    c[2] = n_out;
    c[3] = dropped;
    if (a.totals) {
      atomicAdd(&a.totals[0], (unsigned long long)n_a);
      atomicAdd(&a.totals[1], (unsigned long long)n_in);
      atomicAdd(&a.totals[2], (unsigned long long)n_out);
      atomicAdd(&a.totals[3], (unsigned long long)dropped);
    }
  }
}

__global__ void reset_state_kernel(int* slotmap, int* inv, uint32_t* resbits, size_t n_sm, size_t n_inv,
                                   size_t n_res) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_sm; k += stride) slotmap[k] = -1;
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_inv; k += stride) inv[k] = -1;
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_res; k += stride) resbits[k] = 0u;
}

cudaError_t launch_set(const SetLaunch& a, cudaStream_t st) {
  if (a.words > kSetThreads || a.K > kMaxKmax) return cudaErrorInvalidValue;
  set_kernel<<<a.n_layers_launch, kSetThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reset_state(int* slotmap, int* inv, uint32_t* resbits, int* last_seen, int S, int F, int K,
                               int words, cudaStream_t st) {
  (void)last_seen;
  reset_state_kernel<<<256, 256, 0, st>>>(slotmap, inv, resbits, 2ull * S * F, 2ull * S * K, 2ull * S * words);
  return cudaGetLastError();
}

}  // namespace np
