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
//     use first (ties: lowest ID first) while more than K_max remain, or
//     with frequency-weighted caching (DynamicInfer, importance a + lambda f)
//     R_prev plus A, evicting the non-active neurons active in the fewest
//     tokens of the sequence first (ties: lowest ID first) while more than
//     K_max remain.
//  4. D_in = A \ R_prev, D_out = R_prev \ R_next.  Slot reuse: slots of
//     R_prev ∩ R_next stay; the free slots in ascending order go to D_in in
//     ascending ID order.  Compact placement (LLM in a flash 3.3): the rows
//     occupy exactly [0, |R|); with n = |R_prev| - |D_out|, each slot below n
//     freed by D_out takes a kept row from [n, |R_prev|) (both in ascending
//     slot order, one row move each), and D_in is appended at n, n + 1, ...
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

// The same scan over 64-bit values (three counts packed in 21-bit fields).
__device__ __forceinline__ unsigned long long block_scan64(unsigned long long v, unsigned long long* wsum,
                                                           unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < kSetThreads / 32 ? wsum[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSetThreads / 32) wsum[lane] = w;
  }
  __syncthreads();
  const unsigned long long base = warp > 0 ? wsum[warp - 1] : 0ull;
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

// Slot reuse: the free slots (not held by a kept neuron) in ascending order
// into free_list; *n_free and the high-water mark are published by thread 0.
__device__ __forceinline__ void reuse_assign(const SetLaunch& a, int s, int tid, int KW, int n_in,
                                             const uint32_t* occ, int* wsum, int* s_hw, int* free_list,
                                             int* nfree_out) {
  const int K = a.K;
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
  if (tid < KW && occ[tid]) atomicMax(s_hw, tid * 32 + 32 - __clz(occ[tid]));
  __syncthreads();
  if (tid == 0) {
    if (n_in > n_free) atomicExch(a.err, kDevErrBounds);
    *nfree_out = n_free;
    // one past the highest occupied slot after this delta (kept slots, and
    // the free slots handed out in ascending order)
    if (a.slot_hw) {
      const int na = n_in < n_free ? n_in : n_free;
      int hw = *s_hw;
      if (na > 0 && free_list[na - 1] + 1 > hw) hw = free_list[na - 1] + 1;
      a.slot_hw[s] = hw;
    }
    if (a.mv_count) a.mv_count[s] = 0;
  }
}

// Compact placement: the i-th freed slot below n_keep (ascending) takes the
// row of the i-th kept slot at or above n_keep (ascending); the moves are
// written to the layer's move lists.  Incoming rows go to n_keep, n_keep+1...
__device__ __forceinline__ void compact_assign(const SetLaunch& a, int s, int tid, int KW, int n_keep, int n_in,
                                               const uint32_t* s_hole, const uint32_t* s_mov, int* wsum,
                                               int* hole_list, int* nfree_out) {
  const uint32_t hw = tid < KW ? s_hole[tid] : 0u;
  const uint32_t mw = tid < KW ? s_mov[tid] : 0u;
  int n_holes, n_mov;
  const int eh = block_scan(__popc(hw), wsum, &n_holes);
  const int em = block_scan(__popc(mw), wsum, &n_mov);
  {
    int p = eh;
    for (uint32_t w = hw; w; w &= w - 1) hole_list[p++] = tid * 32 + __ffs(w) - 1;
  }
  __syncthreads();
  const int n_mv = n_holes < n_mov ? n_holes : n_mov;
  int* msrc = a.mv_src + (size_t)s * a.K;
  int* mdst = a.mv_dst + (size_t)s * a.K;
  {
    int p = em;
    for (uint32_t w = mw; w && p < n_mv; w &= w - 1, ++p) {
      msrc[p] = tid * 32 + __ffs(w) - 1;
      mdst[p] = hole_list[p];
    }
  }
  if (tid == 0) {
    if (n_holes != n_mov || n_keep < 0 || n_keep + n_in > a.K) atomicExch(a.err, kDevErrBounds);
    *nfree_out = a.K - (n_keep < 0 ? 0 : n_keep);  // slots left for appends
    a.mv_count[s] = n_mv;
    if (a.slot_hw) a.slot_hw[s] = n_keep + n_in;
  }
}

// HIST: window or frequency residency, which keeps a per-neuron history (the
// last token a neuron was active, or its count).  Without it the kernel has
// no history registers and needs half the register file, so its CTA fits
// beside another kernel's CTAs on one SM.
template <bool HIST>
__global__ void __launch_bounds__(kSetThreads) set_kernel(SetLaunch a) {
  __shared__ int wsum[32];
  __shared__ unsigned long long wsum64[32];
  __shared__ uint32_t occ[kMaxKmax / 32];
  __shared__ uint32_t s_hole[kMaxKmax / 32], s_mov[kMaxKmax / 32];  // compact: slots to refill / to move
  __shared__ int hist[256];
  __shared__ int cut_age, cut_need, s_hw, s_nfree;
  __shared__ uint32_t s_a[kMaxWords], s_out[kMaxWords], s_keep[kMaxWords];
  __shared__ int s_ea[kMaxWords], s_eout[kMaxWords];
  // [K] free slots, then [K] copies of the inverse map and the slot contents,
  // then [K] each: outgoing neurons, their slots, incoming neurons
  extern __shared__ int free_list[];
  int* inv_s = free_list + a.K;
  int* ct_s = inv_s + a.K;
  int* l_out = ct_s + a.K;
  int* l_outs = l_out + a.K;
  int* l_in = l_outs + a.K;

  const int tid = threadIdx.x;
  const int s = a.first_sparse + blockIdx.x;
  const int layer = a.n_dense + s;
  const int F = a.F, K = a.K, W = a.words;
  int* __restrict__ S = a.slotmap + (size_t)s * F;
  int* __restrict__ inv = a.inv + (size_t)s * K;
  int* __restrict__ ct = a.content + (size_t)s * K;
  uint32_t* __restrict__ res = a.resbits + (size_t)s * W;
  int* __restrict__ ls = HIST ? a.last_seen + (size_t)s * F : nullptr;
  int* __restrict__ out_a = a.active + (size_t)s * K;
  int* __restrict__ out_as = a.active_slot + (size_t)s * K;
  int* __restrict__ out_in = a.din_n + (size_t)s * K;
  int* __restrict__ out_ins = a.din_s + (size_t)s * K;
  int* __restrict__ out_inct = a.din_oldct + (size_t)s * K;
  int* __restrict__ out_out = a.dout_n + (size_t)s * K;
  int* __restrict__ out_outs = a.dout_s + (size_t)s * K;
  int* __restrict__ out_lsold = a.ls_old + (size_t)s * K;
  const bool compact = a.compact != 0;

  const int i = tid;
  const bool has_word = i < W;
  const uint32_t word_mask =
      (has_word && i == W - 1 && (F & 31)) ? ((1u << (F & 31)) - 1u) : (has_word ? 0xffffffffu : 0u);

  // The layer's own state does not depend on the prediction: read it while
  // the kernel before this one (the predictor) finishes.  Resident words,
  // the history (last use or count) of this word's 32 neurons, all loads in
  // flight together, and a copy of the inverse map in shared memory.
  grid_dependents_launch();
  const uint32_t rw = has_word ? res[i] : 0u;
  int lsv[32];  // history of the resident neurons now, of the newly active ones below
  if (HIST) {
#pragma unroll
    for (int b = 0; b < 32; ++b) lsv[b] = ((rw >> b) & 1u) ? ls[i * 32 + b] : 0;
  }
  for (int k = tid; k < K; k += kSetThreads) {
    inv_s[k] = inv[k];
    ct_s[k] = ct[k];
  }
  // the prediction and the token counter come from earlier kernels
  grid_dependency_wait();
  const int token = a.token_dev ? *a.token_dev : a.token;

  if (a.keys && a.ids_out && blockIdx.x == 0)
    for (int h = tid; h < a.batch * a.n_heads; h += kSetThreads)
      a.ids_out[h] = (int)(0xFFFFFFFFu - (uint32_t)(a.keys[h] & 0xFFFFFFFFull));

  // 1. active set words
  uint32_t aw = 0;
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

  // 3. resident set after this token (bit loops are unrolled so that the
  //    history stays in registers)
  uint32_t nw = aw;
  if (HIST) {
    const uint32_t fresh = aw & ~rw;
#pragma unroll
    for (int b = 0; b < 32; ++b)
      if ((fresh >> b) & 1u) lsv[b] = ls[i * 32 + b];
  }
  if (HIST && a.window > 1) {
    const uint32_t old = rw & ~aw;  // resident, not active now
    uint32_t keep_old = 0;
#pragma unroll
    for (int b = 0; b < 32; ++b) {
      const int age = token - lsv[b];
      if (((old >> b) & 1u) && age >= 0 && age < a.window) keep_old |= 1u << b;
    }
    uint32_t cand = aw | keep_old;
    int ctot;
    (void)block_scan(__popc(cand), wsum, &ctot);
    if (ctot > K) {
      if (tid < 33) hist[tid] = 0;
      __syncthreads();
#pragma unroll
      for (int b = 0; b < 32; ++b)
        if ((keep_old >> b) & 1u) atomicAdd(&hist[token - lsv[b]], 1);
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
#pragma unroll
      for (int b = 0; b < 32; ++b) {
        if (!((keep_old >> b) & 1u)) continue;
        const int age = token - lsv[b];
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
  } else if (HIST && a.frequency) {
    uint32_t old = rw & ~aw;  // resident, not active now
    int ctot;
    (void)block_scan(__popc(aw | old), wsum, &ctot);
    if (ctot > K) {
      // the (ctot - K) smallest (count, ID) among `old`: radix selection of
      // the count (saturated to 16 bits) in two 8-bit passes, then the
      // lowest IDs of the boundary count
      int need = ctot - K, prefix = 0;
      for (int pass = 0; pass < 2; ++pass) {
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
#pragma unroll
        for (int b = 0; b < 32; ++b) {
          if (!((old >> b) & 1u)) continue;
          const int key = min(lsv[b], 65535);
          if (pass == 0) atomicAdd(&hist[key >> 8], 1);
          else if ((key >> 8) == prefix) atomicAdd(&hist[key & 255], 1);
        }
        __syncthreads();
        if (tid == 0) {
          int d = 0;
          while (d < 255 && hist[d] < need) need -= hist[d++];
          cut_age = d;
          cut_need = need;
        }
        __syncthreads();
        prefix = pass == 0 ? cut_age : (prefix << 8) | cut_age;
        need = cut_need;
      }
      uint32_t bucket = 0, lower = 0;
#pragma unroll
      for (int b = 0; b < 32; ++b) {
        if (!((old >> b) & 1u)) continue;
        const int key = min(lsv[b], 65535);
        if (key < prefix) lower |= 1u << b;
        else if (key == prefix) bucket |= 1u << b;
      }
      int btot;
      const int bexcl = block_scan(__popc(bucket), wsum, &btot);
      uint32_t evict_b = 0;
      if (bexcl < need) evict_b = lowest_bits(bucket, need - bexcl);
      old &= ~(lower | evict_b);
    }
    nw = aw | old;
  }
  const uint32_t dinw = aw & ~rw;
  const uint32_t doutw = rw & ~nw;

  // 4. ranks within A, D_in, D_out (one scan of the three counts packed in
  //    21-bit fields); the lists in ascending ID order, D_in and D_out also
  //    in shared memory for the steps below
  int n_old = 0;
  if (compact) (void)block_scan(__popc(rw), wsum, &n_old);
  constexpr unsigned long long kF21 = (1ull << 21) - 1;
  unsigned long long tot3;
  const unsigned long long ex3 = block_scan64(
      (unsigned long long)__popc(aw) | ((unsigned long long)__popc(dinw) << 21) |
          ((unsigned long long)__popc(doutw) << 42),
      wsum64, &tot3);
  const int ea = (int)(ex3 & kF21), ein = (int)((ex3 >> 21) & kF21), eout = (int)((ex3 >> 42) & kF21);
  const int n_a = (int)(tot3 & kF21), n_in = (int)((tot3 >> 21) & kF21), n_out = (int)((tot3 >> 42) & kF21);
  if (has_word) {
    s_a[i] = aw;
    s_out[i] = doutw;
    s_keep[i] = rw & nw;
    s_ea[i] = ea;
    s_eout[i] = eout;
    int p = ea;
    for (uint32_t w = aw; w; w &= w - 1) out_a[p++] = i * 32 + __ffs(w) - 1;
    p = ein;
    for (uint32_t w = dinw; w; w &= w - 1, ++p) {
      const int n = i * 32 + __ffs(w) - 1;
      out_in[p] = n;
      l_in[p] = n;
    }
    p = eout;
    for (uint32_t w = doutw; w; w &= w - 1, ++p) {
      const int n = i * 32 + __ffs(w) - 1;
      out_out[p] = n;
      l_out[p] = n;
    }
  }
  const int KW = (K + 31) / 32;
  if (tid < KW) {
    occ[tid] = 0u;
    s_hole[tid] = 0u;
    s_mov[tid] = 0u;
  }
  if (tid == 0) s_hw = 0;
  __syncthreads();
  const int n_keep = n_old - n_out;  // compact: rows that stay below this count

  // 5. one pass over the slots: occupied = holds a neuron that stays;
  //    kept active neurons get their slot, outgoing neurons record theirs.
  //    (from the shared copy of the inverse map)
  for (int k = tid; k < K; k += kSetThreads) {
    const int n = inv_s[k];
    if ((unsigned)n >= (unsigned)F) continue;
    const uint32_t bit = 1u << (n & 31);
    const int w = n >> 5;
    const uint32_t kbit = 1u << (k & 31);
    if (s_out[w] & bit) {
      const int r = bit_rank(s_out, s_eout, n);
      out_outs[r] = k;
      l_outs[r] = k;
      if (compact && k < n_keep) atomicOr(&s_hole[k >> 5], kbit);
    } else if (s_keep[w] & bit) {
      atomicOr(&occ[k >> 5], kbit);
      if (compact && k >= n_keep) atomicOr(&s_mov[k >> 5], kbit);
      if (s_a[w] & bit) out_as[bit_rank(s_a, s_ea, n)] = k;
    }
    if (compact && k >= n_old) atomicExch(a.err, kDevErrBounds);  // region not contiguous
  }
  __syncthreads();
  if (compact) {
    compact_assign(a, s, tid, KW, n_keep, n_in, s_hole, s_mov, wsum, free_list, &s_nfree);
  } else {
    reuse_assign(a, s, tid, KW, n_in, occ, wsum, &s_hw, free_list, &s_nfree);
  }
  __syncthreads();

  // 6. outgoing neurons leave (before incoming ones may take their slots)
  for (int r = tid; r < n_out; r += kSetThreads) {
    const int n = l_out[r];
    const int k = l_outs[r];
    S[n] = -1;
    if ((unsigned)k < (unsigned)K) inv[k] = -1;
  }
  __syncthreads();
  // 6b. compact: kept rows from the end of the region fill the freed slots
  if (compact) {
    const int n_mv = a.mv_count[s];
    const int* msrc = a.mv_src + (size_t)s * K;
    const int* mdst = a.mv_dst + (size_t)s * K;
    int* mold = a.mv_oldct + (size_t)s * K;
    for (int r = tid; r < n_mv; r += kSetThreads) {
      const int src = msrc[r], dst = mdst[r];
      const int n = inv[src];
      if ((unsigned)n >= (unsigned)F) continue;
      S[n] = dst;
      inv[dst] = n;
      inv[src] = -1;
      mold[r] = ct[dst];
      ct[dst] = n;
      if (s_a[n >> 5] & (1u << (n & 31))) out_as[bit_rank(s_a, s_ea, n)] = dst;
    }
    __syncthreads();
  }
  // 7. incoming neurons take the free slots (slot reuse) or are appended
  //    (compact); remember what the slots held
  const int n_free = s_nfree;
  for (int r = tid; r < n_in; r += kSetThreads) {
    const int n = l_in[r];
    const int k = r < n_free ? (compact ? n_keep + r : free_list[r]) : 0;
    out_ins[r] = k;
    out_inct[r] = ct_s[k];  // untouched above: appended or free slots are not move targets
    ct[k] = n;
    inv[k] = n;
    S[n] = k;
    out_as[bit_rank(s_a, s_ea, n)] = k;
  }
  if (has_word) res[i] = nw;
  if (HIST && has_word) {  // this word's active neurons, history from registers
    int r = ea;
#pragma unroll
    for (int b = 0; b < 32; ++b) {
      if (!((aw >> b) & 1u)) continue;
      const int n = i * 32 + b;
      out_lsold[r++] = lsv[b];
      ls[n] = a.frequency ? lsv[b] + 1 : token;
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

// Undo set_kernel for one layer per CTA from the recorded delta lists.
__global__ void __launch_bounds__(kSetThreads) rollback_kernel(SetLaunch a) {
  const int s = a.first_sparse + blockIdx.x;
  const int F = a.F, K = a.K, W = a.words;
  int* S = a.slotmap + (size_t)s * F;
  int* inv = a.inv + (size_t)s * K;
  int* ct = a.content + (size_t)s * K;
  uint32_t* res = a.resbits + (size_t)s * W;
  int* ls = (a.window > 1 || a.frequency) ? a.last_seen + (size_t)s * F : nullptr;
  const int* c = a.counts + (size_t)s * 4;
  const int n_a = c[0], n_in = c[1], n_out = c[2];
  const int* din = a.din_n + (size_t)s * K;
  const int* dins = a.din_s + (size_t)s * K;
  const int* dinct = a.din_oldct + (size_t)s * K;
  const int* dout = a.dout_n + (size_t)s * K;
  const int* douts = a.dout_s + (size_t)s * K;
  // slot reuse: an upper bound of the high-water mark is always safe
  if (threadIdx.x == 0 && a.slot_hw && !a.compact) a.slot_hw[s] = K;
  for (int r = threadIdx.x; r < n_in; r += kSetThreads) {
    const int n = din[r], k = dins[r];
    if ((unsigned)n >= (unsigned)F || (unsigned)k >= (unsigned)K) continue;
    S[n] = -1;
    inv[k] = -1;
    ct[k] = dinct[r];
    atomicAnd(&res[n >> 5], ~(1u << (n & 31)));
  }
  __syncthreads();
  if (a.compact) {  // moved rows go back to the end of the region
    const int n_mv = a.mv_count[s];
    const int* msrc = a.mv_src + (size_t)s * K;
    const int* mdst = a.mv_dst + (size_t)s * K;
    const int* mold = a.mv_oldct + (size_t)s * K;
    for (int r = threadIdx.x; r < n_mv; r += kSetThreads) {
      const int src = msrc[r], dst = mdst[r];
      if ((unsigned)src >= (unsigned)K || (unsigned)dst >= (unsigned)K) continue;
      const int n = inv[dst];
      if ((unsigned)n >= (unsigned)F) continue;
      S[n] = src;
      inv[src] = n;
      inv[dst] = -1;
      ct[dst] = mold[r];
    }
    __syncthreads();
  }
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
  if (a.compact) {  // the region is [0, |R_prev|) again
    __shared__ int wsum[32];
    __syncthreads();
    int n_res;
    (void)block_scan(threadIdx.x < W ? __popc(res[threadIdx.x]) : 0, wsum, &n_res);
    if (threadIdx.x == 0) {
      if (a.slot_hw) a.slot_hw[s] = n_res;
      a.mv_count[s] = 0;
    }
  }
}

__global__ void reset_state_kernel(int* slotmap, int* inv, uint32_t* resbits, int* slot_hw, int* counts,
                                   int n_layers, size_t n_sm, size_t n_inv, size_t n_res) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  if (counts)
    for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_sm; k += stride) counts[k] = 0;
  if (slot_hw && blockIdx.x == 0)
    for (int s = threadIdx.x; s < n_layers; s += blockDim.x) slot_hw[s] = 0;
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_sm; k += stride) slotmap[k] = -1;
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_inv; k += stride) inv[k] = -1;
  for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < n_res; k += stride) resbits[k] = 0u;
}

template <bool HIST> struct SetTag {};

cudaError_t launch_set(const SetLaunch& a, cudaStream_t st) {
  if (a.words > kMaxWords || a.K > kMaxKmax) return cudaErrorInvalidValue;
  const size_t dyn = 6 * (size_t)a.K * sizeof(int);
  const bool hist = a.window > 1 || a.frequency;
  cudaError_t e = hist ? ensure_dyn_smem<SetTag<true>>(reinterpret_cast<const void*>(set_kernel<true>), dyn)
                       : ensure_dyn_smem<SetTag<false>>(reinterpret_cast<const void*>(set_kernel<false>), dyn);
  if (e != cudaSuccess) return e;
  PdlConfig c(dim3(a.n_layers_launch), dim3(kSetThreads), dyn, st);
  c.cfg.numAttrs = a.pdl ? 1 : 0;
  return hist ? cudaLaunchKernelEx(&c.cfg, set_kernel<true>, a) : cudaLaunchKernelEx(&c.cfg, set_kernel<false>, a);
}

cudaError_t launch_rollback(const SetLaunch& a, cudaStream_t st) {
  rollback_kernel<<<a.n_layers_launch, kSetThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reset_state(int* slotmap, int* inv, uint32_t* resbits, int* slot_hw, int* counts, int S, int F,
                               int K, int words, cudaStream_t st) {
  reset_state_kernel<<<256, 256, 0, st>>>(slotmap, inv, resbits, slot_hw, counts, S, (size_t)S * F, (size_t)S * K,
                                          (size_t)S * words);
  return cudaGetLastError();
}

}  // namespace np
