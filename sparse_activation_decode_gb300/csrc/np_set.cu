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
//     order.
//
// The state (slot map S, inverse map inv, slot contents, resident bitmask,
// last use) is updated in place and only where it changes; every value
// overwritten is recorded in the delta lists so that rollback_kernel can put
// the previous state back if the incoming rows cannot be read.  Slots are
// derived from the inverse map (one coalesced pass over the K slots), so the
// F-long slot map is only written, never read.
#include "np_common.cuh"
#include "np_kernels.h"

namespace np {

constexpr int kSetThreads = 512;
constexpr int kMaxKmax = 8192;
constexpr int kMaxWords = kSetThreads;

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

// rank of neuron n among the set bits of `words` (per-word exclusive counts in excl)
__device__ __forceinline__ int bit_rank(const uint32_t* words, const int* excl, int n) {
  const int w = n >> 5;
  return excl[w] + __popc(words[w] & ((1u << (n & 31)) - 1u));
}

__global__ void __launch_bounds__(kSetThreads) set_kernel(SetLaunch a) {
  __shared__ int wsum[32];
  __shared__ uint32_t occ[kMaxKmax / 32];
  __shared__ int hist[33];
  __shared__ int cut_age, cut_need, s_hw;
  __shared__ uint32_t s_a[kMaxWords], s_out[kMaxWords], s_keep[kMaxWords];
  __shared__ int s_ea[kMaxWords], s_eout[kMaxWords];
  extern __shared__ int free_list[];  // [K]

  const int tid = threadIdx.x;
  const int s = a.first_sparse + blockIdx.x;
  const int layer = a.n_dense + s;
  const int F = a.F, K = a.K, W = a.words;
  int* __restrict__ S = a.slotmap + (size_t)s * F;
  int* __restrict__ inv = a.inv + (size_t)s * K;
  int* __restrict__ ct = a.content + (size_t)s * K;
  uint32_t* __restrict__ res = a.resbits + (size_t)s * W;
  int* __restrict__ ls = a.window > 1 ? a.last_seen + (size_t)s * F : nullptr;
  int* __restrict__ out_a = a.active + (size_t)s * K;
  int* __restrict__ out_as = a.active_slot + (size_t)s * K;
  int* __restrict__ out_in = a.din_n + (size_t)s * K;
  int* __restrict__ out_ins = a.din_s + (size_t)s * K;
  int* __restrict__ out_inct = a.din_oldct + (size_t)s * K;
  int* __restrict__ out_out = a.dout_n + (size_t)s * K;
  int* __restrict__ out_outs = a.dout_s + (size_t)s * K;
  int* __restrict__ out_lsold = a.ls_old + (size_t)s * K;

  if (a.keys && a.ids_out && blockIdx.x == 0)
    for (int h = tid; h < a.batch * a.n_heads; h += kSetThreads)
      a.ids_out[h] = (int)(0xFFFFFFFFu - (uint32_t)(a.keys[h] & 0xFFFFFFFFull));

  const int i = tid;
  const bool has_word = i < W;
  const uint32_t word_mask =
      (has_word && i == W - 1 && (F & 31)) ? ((1u << (F & 31)) - 1u) : (has_word ? 0xffffffffu : 0u);

  // 1. active set words and resident words
  uint32_t aw = 0;
  const uint32_t rw = has_word ? res[i] : 0u;
  if (has_word) {
    if (a.ids || a.keys) {
      for (int b = 0; b < a.batch; ++b) {
        const int hg = b * a.n_heads + 2 * (layer - 1);
        int ig, iu;
        if (a.keys) {  // packed argmax keys: low word = ~centroid index
          ig = (int)(0xFFFFFFFFu - (uint32_t)(a.keys[hg] & 0xFFFFFFFFull));
          iu = (int)(0xFFFFFFFFu - (uint32_t)(a.keys[hg + 1] & 0xFFFFFFFFull));
        } else {
          ig = a.ids[hg];
          iu = a.ids[hg + 1];
        }
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
  const int excl = block_scan(__popc(aw), wsum, &total);
  const int dropped = total > K ? total - K : 0;
  if (total > K) {
    if (excl >= K) aw = 0;
    else if (excl + __popc(aw) > K) aw = lowest_bits(aw, K - excl);
  }

  // 3. resident set after this token
  uint32_t nw = aw;
  if (a.window > 1) {
    const uint32_t old = rw & ~aw;  // resident, not active now
    uint32_t keep_old = 0;
    for (uint32_t w = old; w;) {
      const int b = __ffs(w) - 1;
      w &= w - 1;
      const int age = a.token - ls[i * 32 + b];
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
        atomicAdd(&hist[a.token - ls[i * 32 + b]], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int excess = ctot - K, age = a.window - 1;
        while (age > 0 && hist[age] < excess) {
          excess -= hist[age];
          --age;
        }
        cut_age = age;  // evict all older than age, and `excess` lowest IDs of age
        cut_need = excess;
      }
      __syncthreads();
      uint32_t bucket = 0, older = 0;
      for (uint32_t w = keep_old; w;) {
        const int b = __ffs(w) - 1;
        w &= w - 1;
        const int age = a.token - ls[i * 32 + b];
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

  // 4. ranks within A, D_in, D_out; the lists in ascending ID order
  int n_a, n_in, n_out;
  const int ea = block_scan(__popc(aw), wsum, &n_a);
  const int ein = block_scan(__popc(dinw), wsum, &n_in);
  const int eout = block_scan(__popc(doutw), wsum, &n_out);
  if (has_word) {
    s_a[i] = aw;
    s_out[i] = doutw;
    s_keep[i] = rw & nw;
    s_ea[i] = ea;
    s_eout[i] = eout;
    int p = ea;
    for (uint32_t w = aw; w; w &= w - 1) out_a[p++] = i * 32 + __ffs(w) - 1;
    p = ein;
    for (uint32_t w = dinw; w; w &= w - 1) out_in[p++] = i * 32 + __ffs(w) - 1;
    p = eout;
    for (uint32_t w = doutw; w; w &= w - 1) out_out[p++] = i * 32 + __ffs(w) - 1;
  }
  const int KW = (K + 31) / 32;
  if (tid < KW) occ[tid] = 0u;
  if (tid == 0) s_hw = 0;
  __syncthreads();

  // 5. one pass over the slots: occupied = holds a neuron that stays;
  //    kept active neurons get their slot, outgoing neurons record theirs
  for (int k = tid; k < K; k += kSetThreads) {
    const int n = inv[k];
    if ((unsigned)n >= (unsigned)F) continue;
    const uint32_t bit = 1u << (n & 31);
    const int w = n >> 5;
    if (s_out[w] & bit) {
      out_outs[bit_rank(s_out, s_eout, n)] = k;
    } else if (s_keep[w] & bit) {
      atomicOr(&occ[k >> 5], 1u << (k & 31));
      if (s_a[w] & bit) out_as[bit_rank(s_a, s_ea, n)] = k;
    }
  }
  __syncthreads();
  // free slots in ascending order
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
  if (tid < KW && occ[tid]) atomicMax(&s_hw, tid * 32 + 32 - __clz(occ[tid]));
  __syncthreads();
  if (n_in > n_free && tid == 0) atomicExch(a.err, kDevErrBounds);
  // one past the highest occupied slot after this delta (kept slots, and the
  // free slots handed out in ascending order)
  if (tid == 0 && a.slot_hw) {
    const int na = n_in < n_free ? n_in : n_free;
    int hw = s_hw;
    if (na > 0 && free_list[na - 1] + 1 > hw) hw = free_list[na - 1] + 1;
    a.slot_hw[s] = hw;
  }

  // 6. outgoing neurons leave (before incoming ones may take their slots)
  for (int r = tid; r < n_out; r += kSetThreads) {
    const int n = out_out[r];
    const int k = out_outs[r];
    S[n] = -1;
    if ((unsigned)k < (unsigned)K) inv[k] = -1;
  }
  __syncthreads();
  // 7. incoming neurons take the free slots; remember what the slots held
  for (int r = tid; r < n_in; r += kSetThreads) {
    const int n = out_in[r];
    const int k = r < n_free ? free_list[r] : 0;
    out_ins[r] = k;
    out_inct[r] = ct[k];
    ct[k] = n;
    inv[k] = n;
    S[n] = k;
    out_as[bit_rank(s_a, s_ea, n)] = k;
  }
  if (has_word) res[i] = nw;
  if (ls)
    for (int r = tid; r < n_a; r += kSetThreads) {
      const int n = out_a[r];
      out_lsold[r] = ls[n];
      ls[n] = a.token;
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

// Undo set_kernel for one layer per CTA from the recorded delta lists.
__global__ void __launch_bounds__(kSetThreads) rollback_kernel(SetLaunch a) {
  const int s = a.first_sparse + blockIdx.x;
  const int F = a.F, K = a.K, W = a.words;
  int* S = a.slotmap + (size_t)s * F;
  int* inv = a.inv + (size_t)s * K;
  int* ct = a.content + (size_t)s * K;
  uint32_t* res = a.resbits + (size_t)s * W;
  int* ls = a.window > 1 ? a.last_seen + (size_t)s * F : nullptr;
  const int* c = a.counts + (size_t)s * 4;
  const int n_a = c[0], n_in = c[1], n_out = c[2];
  const int* din = a.din_n + (size_t)s * K;
  const int* dins = a.din_s + (size_t)s * K;
  const int* dinct = a.din_oldct + (size_t)s * K;
  const int* dout = a.dout_n + (size_t)s * K;
  const int* douts = a.dout_s + (size_t)s * K;
  if (threadIdx.x == 0 && a.slot_hw) a.slot_hw[s] = K;  // an upper bound is always safe
  for (int r = threadIdx.x; r < n_in; r += kSetThreads) {
    const int n = din[r], k = dins[r];
    if ((unsigned)n >= (unsigned)F || (unsigned)k >= (unsigned)K) continue;
    S[n] = -1;
    inv[k] = -1;
    ct[k] = dinct[r];
    atomicAnd(&res[n >> 5], ~(1u << (n & 31)));
  }
  __syncthreads();
  for (int r = threadIdx.x; r < n_out; r += kSetThreads) {
    const int n = dout[r], k = douts[r];
    if ((unsigned)n >= (unsigned)F || (unsigned)k >= (unsigned)K) continue;
    S[n] = k;
    inv[k] = n;
    atomicOr(&res[n >> 5], 1u << (n & 31));
  }
  if (ls) {
    const int* act = a.active + (size_t)s * K;
    const int* old = a.ls_old + (size_t)s * K;
    for (int r = threadIdx.x; r < n_a; r += kSetThreads) {
      const int n = act[r];
      if ((unsigned)n < (unsigned)F) ls[n] = old[r];
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
  if (a.words > kMaxWords || a.K > kMaxKmax) return cudaErrorInvalidValue;
  const size_t dyn = (size_t)a.K * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(set_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  set_kernel<<<a.n_layers_launch, kSetThreads, dyn, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rollback(const SetLaunch& a, cudaStream_t st) {
  rollback_kernel<<<a.n_layers_launch, kSetThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reset_state(int* slotmap, int* inv, uint32_t* resbits, int S, int F, int K, int words,
                               cudaStream_t st) {
  reset_state_kernel<<<256, 256, 0, st>>>(slotmap, inv, resbits, (size_t)S * F, (size_t)S * K, (size_t)S * words);
  return cudaGetLastError();
}

}  // namespace np
