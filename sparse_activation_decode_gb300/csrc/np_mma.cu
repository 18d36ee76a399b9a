// Batched row products on the tensor cores (sm_103a): the FFN, the predictor
// hidden layer and the predictor heads for B <= 8 sequences decoded together.
//
// With B sequences the FFN over the union active set (NeuroPrefetcher
// sections 3.3-3.4; every sequence uses the layer's union of predicted rows)
// is a real contraction: for a tile of 128 resident rows,
//     A = W_tile x X^T       (128 rows x B columns, contraction over d_model)
// and the down projection
//     Y = Dt_tile^T x H      (d_model x B, contraction over the tile's rows).
// Both run as tcgen05 MMAs with M = 128, N = 16, fp32 accumulators in tensor
// memory.  The 16 columns carry each sequence's input twice, as a sum of two
// 16-bit values (hi = round(v), lo = round(v - hi)): column j holds hi_j and
// column j + 8 holds lo_j, and the epilogue adds the two accumulator columns,
// so the inputs keep about 16 significant bits and no rounding of x or of the
// activations is needed.  The weights are used exactly as stored.
//
// Work split: thread-block clusters of CS CTAs; the clusters split the row
// list evenly; inside a cluster CTA r owns the column slice
// [r*Kdim/CS, (r+1)*Kdim/CS) of every row.  For each tile of 128 rows:
//   1. a producer warp loads the tile's rows of the slice, 64 columns at a
//      time, with 2-D tensor-map boxes of 32 and 8 rows (4 KB / 1 KB per
//      copy: the copy engine's cost is per request, so requests stay large)
//      into a shared-memory ring.  Sparse layers are walked in slot order,
//      over slots [0, high-water mark) of the resident buffers, and a slot
//      whose inverse map entry is -1 (free) contributes nothing;
//   2. one thread issues the MMAs of the slice for gate and up;
//   3. four epilogue warps read the partial dot products from tensor memory
//      and send them to the CTA of the cluster that owns the row (remote
//      shared-memory stores + cluster-scope mbarrier arrives); the owner adds
//      the CS partials in a fixed order and forms the activation
//      h = relu(g.x)(u.x), which it writes, split into hi/lo, into the
//      operand buffer of every CTA of the cluster;
//   4. (FFN) the MMA thread multiplies the slice's down^T rows of the tile by
//      h, accumulating the slice of y in tensor memory over all tiles.
// At the end every CTA adds its slice of y into the output with fp32 atomic
// adds (the only order-dependent step).
//
// The residual stream is passed as base + previous layer's y (both [B][Kdim]
// fp32); every CTA forms h = base + y_prev for all sequences and its rmsnorm,
// and the CTAs of cluster 0 store h and clear the next accumulator, so
// consecutive layers chain without an extra kernel.
//
// Programmatic dependent launch: the weights and the row count do not depend
// on the previous kernel in the stream (the set kernel and the reads that
// fill the resident buffers reach this stream through events, which stay
// full dependencies), so the producer streams as soon as the CTA is
// resident; the epilogue warps wait for the previous kernel before they read
// its outputs or write anything.  Every CTA waits, so a kernel that follows
// this one also follows its predecessor.
//
// Every wait is bounded (about one second): a timeout records an error word,
// lets the other roles of the CTA stop early, waits for the copies and MMAs
// already in flight, frees the tensor memory and returns.
#include <cstring>
#include <mutex>

#include "np_tc.cuh"

namespace np {

namespace {

constexpr int kMmaThreads = 192;     // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kTileRows = 128;
constexpr uint32_t kTmemCols = 256;
constexpr int kMaxStages = 16;
constexpr uint32_t kSmemHeader = 18432;  // barriers, exchange buffers, activation operand, y staging

// barrier slots
constexpr int kBarFull = 0, kBarEmpty = 16, kBarAccFull = 32, kBarAccEmpty = 33, kBarXReady = 34, kBarRed = 35,
              kBarXFree = 36, kBarHFull = 37, kBarYFull = 38, kBarDone = 39, kBarSS = 40;

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// AND of a flag over the 128 epilogue threads (all of them must arrive).
__device__ __forceinline__ bool epi_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

template <bool BF16> __device__ __forceinline__ uint16_t to16(float v);
template <> __device__ __forceinline__ uint16_t to16<true>(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
template <> __device__ __forceinline__ uint16_t to16<false>(float v) { return __half_as_ushort(__float2half_rn(v)); }
template <bool BF16> __device__ __forceinline__ float from16(uint16_t v);
template <> __device__ __forceinline__ float from16<true>(uint16_t v) {
  return __bfloat162float(__ushort_as_bfloat16(v));
}
template <> __device__ __forceinline__ float from16<false>(uint16_t v) { return __half2float(__ushort_as_half(v)); }

// hi/lo split of v: v ~ hi + lo with hi, lo 16-bit values
template <bool BF16> __device__ __forceinline__ void split16(float v, uint16_t& hi, uint16_t& lo) {
  hi = to16<BF16>(v);
  lo = to16<BF16>(v - from16<BF16>(hi));
}

__device__ __forceinline__ unsigned long long argmax_key_tc(float v, int idx) {
  v = v + 0.0f;
  const uint32_t u = __float_as_uint(v);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}

// Bounded wait that ignores the abort flag (used to drain work in flight).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cl(bar, parity))
    if (global_ns() - t0 > kWaitLimitNs) break;
}

template <int MODE, bool BF16>
__global__ void __launch_bounds__(kMmaThreads, 1) mma_rows_kernel(const __grid_constant__ CUtensorMap tmap32,
                                                                  const __grid_constant__ CUtensorMap tmap8,
                                                                  const MmaArgs a) {
  constexpr bool kFfn = MODE == kMmaFfnGated || MODE == kMmaFfnUp;
  constexpr bool kGated = MODE == kMmaFfnGated;
  constexpr int kProj = kGated ? 2 : 1;  // projections in the first product
  constexpr uint32_t kIdescK = idesc_f16(BF16, false, 128, 16);
  constexpr uint32_t kIdescMN = idesc_f16(BF16, true, 128, 16);

  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (sbase - raw);
  volatile int* misc = reinterpret_cast<volatile int*>(sm + 512);  // [0] tmem base, [1] abort
  float* ssred = reinterpret_cast<float*>(sm + 512 + 64);          // [4 warps][8]
  const uint32_t ssx_a = sbase + 512 + 256;                        // [cs][8] slice sums of squares
  const float* ssx = reinterpret_cast<const float*>(sm + 512 + 256);
  float* ystage = reinterpret_cast<float*>(sm + 14336);            // [8][128] y of one M tile
  float* recv = reinterpret_cast<float*>(sm + 2048);               // [128][16]
  const uint32_t recv_a = sbase + 2048;
  const uint32_t hbuf_a = sbase + 10240;                           // 4 KB activation operand
  const uint32_t xb_a = sbase + kSmemHeader;                       // input operand [ks/64][16 x 64]
  const int ks = a.ks_len;
  const uint32_t ring_a = xb_a + (uint32_t)(ks / 64) * 2048u;
  const int NS = a.n_stages;
  const uint32_t stage_bytes = a.stage_bytes;
  auto bar = [&](int i) -> uint32_t { return sbase + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = a.cs;
  const uint32_t rank = cluster_rank();
  const int cid = (int)cluster_id_x();
  const int slice0 = (int)rank * ks;
  const int Kd = a.Kdim;

  grid_dependents_launch();  // the next layer may start streaming its weights
  // the row count is loaded while the barriers are set up
  int n = a.n_rows_dev ? *a.n_rows_dev : a.n_rows_host;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(reinterpret_cast<uint64_t*>(sm) + kBarFull + s, 1);
      mbar_init(reinterpret_cast<uint64_t*>(sm) + kBarEmpty + s, 1);
    }
    uint64_t* b = reinterpret_cast<uint64_t*>(sm);
    mbar_init(b + kBarAccFull, 1);
    mbar_init(b + kBarAccEmpty, 128);
    mbar_init(b + kBarXReady, 128);
    // cross-CTA barriers count one arrive per epilogue warp of the cluster
    // that writes (each warp's 32 rows have a single owner)
    mbar_init(b + kBarRed, 4);
    mbar_init(b + kBarXFree, 4);
    mbar_init(b + kBarHFull, 4);
    mbar_init(b + kBarYFull, 1);
    mbar_init(b + kBarDone, 1);
    mbar_init(b + kBarSS, (uint32_t)a.cs);
    misc[1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + 512, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = (uint32_t)misc[0];
  volatile int* abort = misc + 1;
  cluster_sync_all();  // every barrier of the cluster is initialised

  n = n < 0 ? 0 : (n > a.row_cap ? a.row_cap : n);
  const int G = a.n_clusters;
  const int r_begin = (int)((long long)cid * n / G), r_end = (int)((long long)(cid + 1) * n / G);
  const int n_tiles = (r_end - r_begin + kTileRows - 1) / kTileRows;
  const int n_kb = ks / 64, n_mt = kFfn ? ks / 128 : 0;

  if (warp == 0) {
    // ---------------- producer: tensor-map gathers into the ring ----------------
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    int ps = 0;          // ring slot of copy `it`
    uint32_t pph = 0;    // its pass parity
    bool ok = true;
    for (int tile = 0; tile < n_tiles && ok; ++tile) {
      const int t0 = r_begin + tile * kTileRows;
      const int nr = min(kTileRows, r_end - t0);
      // boxes: n32 of 32 rows, then 8-row boxes up to a multiple of 8 rows
      // (first product) or of 16 rows (down projection: whole MMA K steps)
      const int n32 = nr >> 5;
      const int nb_gu = n32 + ((((nr + 7) & ~7) - 32 * n32) >> 3);
      const int rows_gu = 32 * n32 + 8 * (nb_gu - n32);
      for (int kb = 0; kb < n_kb && ok; ++kb) {
        const int s = ps;
        int w = 1;
        if (lane == 0) {
          w = wait_phase(bar(kBarEmpty + s), pph ^ 1u, abort, a.err);
          if (w) mbar_arrive_expect_tx_a(bar(kBarFull + s), (uint32_t)(kProj * rows_gu * 128));
        }
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
        const uint32_t dst0 = ring_a + (uint32_t)s * stage_bytes;
        const int x = slice0 + kb * 64;
        for (int q = lane; q < kProj * nb_gu; q += 32) {
          const int p = q / nb_gu, b = q - p * nb_gu;
          const int rb = (p == 0 ? a.row_base0 : a.row_base1) + t0;
          const int r = b < n32 ? 32 * b : 32 * n32 + 8 * (b - n32);
          tma_load_2d(dst0 + (uint32_t)p * 16384u + (uint32_t)r * 128u, b < n32 ? &tmap32 : &tmap8, x, rb + r,
                      bar(kBarFull + s), pol);
        }
        ++it;
        if (++ps == NS) {
          ps = 0;
          pph ^= 1u;
        }
      }
      if (kFfn) {
        const int nb_dt = n32 + ((((nr + 15) & ~15) - 32 * n32) >> 3);
        const int rows_dt = 32 * n32 + 8 * (nb_dt - n32);
        for (int mt = 0; mt < n_mt && ok; ++mt) {
          const int s = ps;
          int w = 1;
          if (lane == 0) {
            w = wait_phase(bar(kBarEmpty + s), pph ^ 1u, abort, a.err);
            if (w) mbar_arrive_expect_tx_a(bar(kBarFull + s), (uint32_t)(2 * rows_dt * 128));
          }
          ok = __shfl_sync(0xffffffffu, w, 0) != 0;
          if (!ok) break;
          const uint32_t dst0 = ring_a + (uint32_t)s * stage_bytes;
          for (int q = lane; q < 2 * nb_dt; q += 32) {
            const int grp = q / nb_dt, b = q - grp * nb_dt;
            const int r = b < n32 ? 32 * b : 32 * n32 + 8 * (b - n32);
            tma_load_2d(dst0 + (uint32_t)grp * 16384u + (uint32_t)r * 128u, b < n32 ? &tmap32 : &tmap8,
                        slice0 + mt * 128 + grp * 64, a.row_base2 + t0 + r, bar(kBarFull + s), pol);
          }
          ++it;
          if (++ps == NS) {
            ps = 0;
            pph ^= 1u;
          }
        }
      }
    }
    // copies still in flight must land before the CTA leaves
    if (lane == 0 && !ok) {
      const uint32_t first = it > (uint32_t)NS ? it - (uint32_t)NS : 0u;
      for (uint32_t j = first; j < it; ++j) wait_drain(bar(kBarFull + (int)(j % (uint32_t)NS)), (j / NS) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = wait_phase(bar(kBarXReady), 0, abort, a.err);
      fence_proxy_async_cta();
      tc_fence_after();
      uint32_t it = 0;
      int ms = 0;          // ring slot of copy `it`
      uint32_t mph = 0;    // its pass parity
      for (int tile = 0; tile < n_tiles && ok; ++tile) {
        const int nr = min(kTileRows, r_end - (r_begin + tile * kTileRows));
        if (tile > 0) {
          ok = wait_phase(bar(kBarAccEmpty), (uint32_t)(tile - 1) & 1u, abort, a.err);
          tc_fence_after();
        }
        for (int kb = 0; kb < n_kb && ok; ++kb) {
          const int s = ms;
          ok = wait_phase(bar(kBarFull + s), mph, abort, a.err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st_a = ring_a + (uint32_t)s * stage_bytes;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const uint64_t bd = smem_desc_sw128(xb_a + (uint32_t)kb * 2048u + (uint32_t)k4 * 32u, 16u, 1024u);
#pragma unroll
            for (int p = 0; p < kProj; ++p) {
              const uint64_t ad = smem_desc_sw128(st_a + (uint32_t)p * 16384u + (uint32_t)k4 * 32u, 16u, 1024u);
              tc_mma(tbase + 16u * (uint32_t)p, ad, bd, kIdescK, (kb | k4) != 0);
            }
          }
          tc_commit(bar(kBarEmpty + s));
          ++it;
          if (++ms == NS) {
            ms = 0;
            mph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(bar(kBarAccFull));
        if (kFfn) {
          ok = wait_phase(bar(kBarHFull), (uint32_t)tile & 1u, abort, a.err);
          if (!ok) break;
          fence_proxy_async_cta();
          tc_fence_after();
          const int nks = (nr + 15) >> 4;
          for (int mt = 0; mt < n_mt && ok; ++mt) {
            const int s = ms;
            ok = wait_phase(bar(kBarFull + s), mph, abort, a.err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t st_a = ring_a + (uint32_t)s * stage_bytes;
            for (int k = 0; k < nks; ++k) {
              const uint64_t ad = smem_desc_sw128(st_a + (uint32_t)k * 2048u, 16384u, 1024u);
              const uint64_t bd =
                  smem_desc_sw128(hbuf_a + (uint32_t)(k >> 2) * 2048u + (uint32_t)(k & 3) * 32u, 16u, 1024u);
              tc_mma(tbase + 32u + 16u * (uint32_t)mt, ad, bd, kIdescMN, (tile > 0 || k > 0) ? 1u : 0u);
            }
            tc_commit(bar(kBarEmpty + s));
            ++it;
            if (++ms == NS) {
              ms = 0;
              mph ^= 1u;
            }
          }
        }
      }
      if (kFfn && ok && n_tiles > 0) tc_commit(bar(kBarYFull));
      // every MMA issued so far has finished before the tensor memory is freed
      tc_commit(bar(kBarDone));
      wait_drain(bar(kBarDone), 0);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (128 threads) ----------------
    const int e = threadIdx.x - 64;
    const int ew = e >> 5;
    const int Q = warp & 3;
    const int t = 32 * Q + lane;  // tile row <-> tensor-memory lane
    const int B = a.B;
    grid_dependency_wait();  // the previous kernel's outputs are visible from here on

    // prologue: input operand of this CTA's column slice
    if (MODE == kMmaHeads) {
      uint32_t* xw = reinterpret_cast<uint32_t*>(sm + kSmemHeader);
      const int q4 = ks / 8;  // 16-byte chunks per operand row
      for (int idx = e; idx < 16 * q4; idx += 128) {
        const int nn = idx / q4, c = idx - nn * q4;
        const uint4 wv = reinterpret_cast<const uint4*>(a.zin + (size_t)nn * Kd + slice0)[c];
        *reinterpret_cast<uint4*>(xw + (kmajor_off(nn, 8 * c, 16) >> 2)) = wv;
      }
    } else {
      // sum of squares of h = hb + yprev over this CTA's slice; the CTAs of
      // the cluster cover every column once, so the slice sums are exchanged
      // and added in rank order.  A slice of at most 256 four-column groups
      // (two per thread) stays in registers: every load is issued at once
      // and the operand is written from the same values after the exchange.
      const int S4 = ks / 4;
      const bool resident = S4 <= 256;
      auto load_h = [&](int i, float4 (&v)[8]) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (b < B) v[b] = reinterpret_cast<const float4*>(a.hb + (size_t)b * Kd + slice0)[i];
        }
        if (a.yprev) {
#pragma unroll
          for (int b = 0; b < 8; ++b)
            if (b < B) {
              const float4 w = reinterpret_cast<const float4*>(a.yprev + (size_t)b * Kd + slice0)[i];
              v[b].x += w.x; v[b].y += w.y; v[b].z += w.z; v[b].w += w.w;
            }
        }
      };
      float ss[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) ss[b] = 0.f;
      auto add_ss = [&](const float4 (&v)[8]) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          ss[b] = fmaf(v[b].x, v[b].x, ss[b]);
          ss[b] = fmaf(v[b].y, v[b].y, ss[b]);
          ss[b] = fmaf(v[b].z, v[b].z, ss[b]);
          ss[b] = fmaf(v[b].w, v[b].w, ss[b]);
        }
      };
      float4 hr[2][8];
      if (resident) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (e + 128 * q < S4) {
            load_h(e + 128 * q, hr[q]);
          } else {
#pragma unroll
            for (int b = 0; b < 8; ++b) hr[q][b] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) add_ss(hr[q]);
      } else {
        for (int i = e; i < S4; i += 128) {
          float4 v[8];
          load_h(i, v);
          add_ss(v);
        }
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) ss[b] = warp_sum(ss[b]);
      if (lane == 0)
#pragma unroll
        for (int b = 0; b < 8; ++b) ssred[ew * 8 + b] = ss[b];
      epi_sync();
      if (e == 0) {
        float part[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) part[b] = ssred[b] + ssred[8 + b] + ssred[16 + b] + ssred[24 + b];
        for (int dst = 0; dst < cs; ++dst) {
          const uint32_t ra = cluster_map(ssx_a + rank * 32u, (uint32_t)dst);
          st_cluster_f4(ra, part[0], part[1], part[2], part[3]);
          st_cluster_f4(ra + 16, part[4], part[5], part[6], part[7]);
        }
        fence_acq_rel_cluster();
        for (int dst = 0; dst < cs; ++dst) mbar_arrive_cluster_relaxed(cluster_map(bar(kBarSS), (uint32_t)dst));
      }
      const bool ss_ok = wait_phase(bar(kBarSS), 0, abort, a.err);
      float inv[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        float tot = 0.f;
        for (int r = 0; r < cs; ++r) tot += ssx[r * 8 + b];
        inv[b] = ss_ok ? rsqrtf(tot / (float)Kd + 1e-6f) : 0.f;
      }
      // x = h * inv as hi/lo operand rows (row b = hi, row 8 + b = lo), four
      // columns per step; cluster 0 also stores h and clears the next y
      uint32_t* xw = reinterpret_cast<uint32_t*>(sm + kSmemHeader);
      auto emit = [&](int i, const float4 (&v)[8]) {
        const int k = 4 * i, d = slice0 + k;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (cid == 0 && b < B) {
            if (a.hb_out) *reinterpret_cast<float4*>(a.hb_out + (size_t)b * Kd + d) = v[b];
            if (a.y_zero) *reinterpret_cast<float4*>(a.y_zero + (size_t)b * Kd + d) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
          uint16_t hi[4], lo[4];
          split16<BF16>(v[b].x * inv[b], hi[0], lo[0]);
          split16<BF16>(v[b].y * inv[b], hi[1], lo[1]);
          split16<BF16>(v[b].z * inv[b], hi[2], lo[2]);
          split16<BF16>(v[b].w * inv[b], hi[3], lo[3]);
          // columns k..k+3 share one 16-byte chunk of their operand row
          xw[kmajor_off(b, k, 16) >> 2] = (uint32_t)hi[0] | ((uint32_t)hi[1] << 16);
          xw[kmajor_off(b, k + 2, 16) >> 2] = (uint32_t)hi[2] | ((uint32_t)hi[3] << 16);
          xw[kmajor_off(8 + b, k, 16) >> 2] = (uint32_t)lo[0] | ((uint32_t)lo[1] << 16);
          xw[kmajor_off(8 + b, k + 2, 16) >> 2] = (uint32_t)lo[2] | ((uint32_t)lo[3] << 16);
        }
      };
      if (resident) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (e + 128 * q < S4) emit(e + 128 * q, hr[q]);
      } else {
        for (int i = e; i < S4; i += 128) {
          float4 v[8];
          load_h(i, v);
          emit(i, v);
        }
      }
      if (MODE == kMmaHidden && a.keys_zero && blockIdx.x == 0)
        for (int i = e; i < a.n_keys_zero; i += 128) a.keys_zero[i] = 0ull;
    }
    fence_proxy_async_cta();
    mbar_arrive_local(bar(kBarXReady));

    const int rpo = kTileRows / cs;  // rows owned per CTA of the cluster
    const uint32_t owner = (uint32_t)(t / rpo);
    const int tl = t - (int)owner * rpo;
    const bool reducer = owner == rank;  // uniform over the warp (rpo >= 32)
    bool ok = true;
    for (int tile = 0; tile < n_tiles && ok; ++tile) {
      const int t0 = r_begin + tile * kTileRows;
      const int nr = min(kTileRows, r_end - t0);
      ok = wait_phase(bar(kBarAccFull), (uint32_t)tile & 1u, abort, a.err);
      if (!ok) break;
      tc_fence_after();
      float g[16], u[16];
      tmem_ld16(tbase + ((uint32_t)(32 * Q) << 16), g);
      if (kGated) tmem_ld16(tbase + ((uint32_t)(32 * Q) << 16) + 16u, u);
      tc_fence_before();
      mbar_arrive_local(bar(kBarAccEmpty));
      if (tile > 0) {
        // the owner has read this CTA's previous partials: it broadcast h
        // after reading them (FFN), or released the buffer (other modes)
        ok = wait_phase(bar(kFfn ? kBarHFull : kBarXFree), (uint32_t)(tile - 1) & 1u, abort, a.err);
        if (!ok) break;
      }
      {
        const uint32_t dst = cluster_map(recv_a + (uint32_t)((rank * rpo + tl) * 64), owner);
        st_cluster_f4(dst, g[0] + g[8], g[1] + g[9], g[2] + g[10], g[3] + g[11]);
        st_cluster_f4(dst + 16, g[4] + g[12], g[5] + g[13], g[6] + g[14], g[7] + g[15]);
        if (kGated) {
          st_cluster_f4(dst + 32, u[0] + u[8], u[1] + u[9], u[2] + u[10], u[3] + u[11]);
          st_cluster_f4(dst + 48, u[4] + u[12], u[5] + u[13], u[6] + u[14], u[7] + u[15]);
        }
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          mbar_arrive_cluster_relaxed(cluster_map(bar(kBarRed), owner));
        }
      }
      if (!reducer) continue;
      ok = wait_phase(bar(kBarRed), (uint32_t)tile & 1u, abort, a.err);
      if (!ok) break;
      float av[8], bv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) av[j] = bv[j] = 0.f;
      for (int src = 0; src < cs; ++src) {
        const float* r = recv + (size_t)(src * rpo + tl) * 16;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          av[j] += r[j];
          if (kGated) bv[j] += r[8 + j];
        }
      }
      if (!kFfn) {
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          for (int src = 0; src < cs; ++src) mbar_arrive_cluster_relaxed(cluster_map(bar(kBarXFree), (uint32_t)src));
        }
      }
      const bool valid = t < nr && (a.occ_inv == nullptr || a.occ_inv[t0 + t] >= 0);
      if (kFfn) {
        uint16_t v16[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float hv = 0.f;
          if (valid && j < B)
            hv = kGated ? (a.swiglu ? av[j] / (1.f + expf(-av[j])) : fmaxf(av[j], 0.f)) * bv[j] : fmaxf(av[j], 0.f);
          split16<BF16>(hv, v16[j], v16[8 + j]);
        }
        // write this row's 16 operand values into the local buffer, then copy
        // the warp's 64 16-byte chunks (16 operand rows x 4 groups of 8 tile
        // rows) to the same place in every other CTA of the cluster
        uint16_t* hw16 = reinterpret_cast<uint16_t*>(sm + 10240);
#pragma unroll
        for (int nn = 0; nn < 16; ++nn) hw16[kmajor_off(nn, t, 16) >> 1] = v16[nn];
        __syncwarp();
        for (int c = lane; c < 64; c += 32) {
          const int nn = c >> 2, kr = 32 * Q + 8 * (c & 3);
          const uint32_t off = kmajor_off(nn, kr, 16);
          const uint4 val = *reinterpret_cast<const uint4*>(sm + 10240 + off);
          for (int dst = 0; dst < cs; ++dst) {
            if (dst == (int)rank) continue;
            const uint32_t ra = cluster_map(hbuf_a + off, (uint32_t)dst);
            asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "r"(val.x), "r"(val.y),
                         "r"(val.z), "r"(val.w)
                         : "memory");
          }
        }
        fence_proxy_async_cluster();
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_cluster();
          for (int dst = 0; dst < cs; ++dst) mbar_arrive_cluster_relaxed(cluster_map(bar(kBarHFull), (uint32_t)dst));
        }
      } else if (MODE == kMmaHidden) {
        if (valid) {
          const int row = t0 + t;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint16_t hi, lo;
            split16<BF16>(j < B ? fmaxf(av[j], 0.f) : 0.f, hi, lo);
            a.zout[(size_t)j * a.zout_stride + row] = hi;
            a.zout[(size_t)(8 + j) * a.zout_stride + row] = lo;
          }
        }
      } else {  // heads: per sequence, argmax over each head's C logits
        const int grow = a.row_base0 + t0 + t;
        const int head = valid ? grow / a.C : -1;
        const int cix = grow - (grow / a.C) * a.C;
        const int nxt_head = __shfl_down_sync(0xffffffffu, head, 1);
        const bool seg_end = lane == 31 || nxt_head != head;
        for (int j = 0; j < B; ++j) {
          unsigned long long key = valid ? argmax_key_tc(av[j], cix) : 0ull;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long other = __shfl_up_sync(0xffffffffu, key, o);
            const int oh = __shfl_up_sync(0xffffffffu, head, o);
            if (lane >= o && oh == head && other > key) key = other;
          }
          if (valid && seg_end) atomicMax(a.keys + (size_t)j * a.n_heads + head, key);
        }
      }
    }
    if (kFfn && n_tiles > 0) {
      if (ok) ok = wait_phase(bar(kBarYFull), 0, abort, a.err);
      ok = epi_and(ok);  // the stores below synchronise all 128 threads
      if (ok) {
        tc_fence_after();
        for (int mt = 0; mt < n_mt; ++mt) {
          float v[16];
          tmem_ld16(tbase + ((uint32_t)(32 * Q) << 16) + 32u + 16u * (uint32_t)mt, v);
#pragma unroll
          for (int j = 0; j < 8; ++j) ystage[j * 128 + t] = v[j] + v[8 + j];
          epi_sync();
          // four consecutive columns of one sequence per vector atomic
          for (int idx = e; idx < B * 32; idx += 128) {
            const int j = idx >> 5, q = idx & 31;
            const float4 y4 = *reinterpret_cast<const float4*>(ystage + j * 128 + 4 * q);
            atomicAdd(reinterpret_cast<float4*>(a.y_acc + (size_t)j * Kd + slice0 + mt * 128 + 4 * q), y4);
          }
          epi_sync();
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  cluster_sync_all();  // no CTA leaves while another may still write into its shared memory
}

template <int MODE, bool BF16> struct MmaSmemTag {};

template <int MODE, bool BF16>
cudaError_t launch_mode(const RowMaps& maps, const MmaArgs& a, size_t smem, cudaStream_t st) {
  auto kern = mma_rows_kernel<MODE, BF16>;
  cudaError_t e = ensure_dyn_smem<MmaSmemTag<MODE, BF16>>(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(a.n_clusters * a.cs));
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, maps.m32, maps.m8, a);
}

template <int MODE, bool BF16>
cudaError_t max_clusters(int cs, size_t smem, int* out) {
  auto kern = mma_rows_kernel<MODE, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(cs * 64));
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

__global__ void add_kernel(float* __restrict__ out, const float* __restrict__ x, const float* __restrict__ y, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = x[i] + y[i];
}

}  // namespace

cudaError_t launch_add(float* out, const float* x, const float* y, int n, cudaStream_t st) {
  add_kernel<<<(n + 255) / 256, 256, 0, st>>>(out, x, y, n);
  return cudaGetLastError();
}

cudaError_t make_row_maps(RowMaps* out, const void* base, int dtype, uint64_t rows, uint64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if (dtype != 1 && dtype != 2) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || cols % 64 || rows == 0 || rows >= (1ull << 31))
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t estr[2] = {1, 1};
  const cuuint32_t heights[2] = {32, 8};
  CUtensorMap* maps[2] = {&out->m32, &out->m8};
  for (int i = 0; i < 2; ++i) {
    std::memset(maps[i], 0, sizeof(CUtensorMap));
    const cuuint32_t box[2] = {64, heights[i]};
    const CUresult r =
        fn(maps[i], dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
           const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

size_t mma_smem_bytes(int mode, int ks_len, int n_stages) {
  const uint32_t stage = (mode == kMmaFfnGated || mode == kMmaFfnUp) ? 32768u : 16384u;
  return 1024 + kSmemHeader + (size_t)(ks_len / 64) * 2048 + (size_t)n_stages * stage;
}

cudaError_t mma_plan(int mode, int bf16, int Kdim, size_t smem_optin, int n_sms, int want_clusters, int max_stages,
                     MmaPlan* p) {
  const bool ffn = mode == kMmaFfnGated || mode == kMmaFfnUp;
  const int unit = ffn ? 128 : 64;
  int cs = 0;
  for (int c : {4, 2, 1})
    if (Kdim % (unit * c) == 0) {
      cs = c;
      break;
    }
  if (cs == 0) return cudaErrorInvalidValue;
  const int ks = Kdim / cs;
  if (ffn && ks / 128 > 14) return cudaErrorInvalidValue;  // y accumulators must fit the tensor memory
  const uint32_t stage = ffn ? 32768u : 16384u;
  const size_t fixed = mma_smem_bytes(mode, ks, 0);
  if (fixed + 2 * stage > smem_optin) return cudaErrorInvalidValue;
  int ns = (int)((smem_optin - fixed) / stage);
  if (ns > kMaxStages) ns = kMaxStages;
  if (max_stages > 1 && ns > max_stages) ns = max_stages;  // fewer stages: more CTAs per SM
  const size_t smem = mma_smem_bytes(mode, ks, ns);
  int nc = 0;
  cudaError_t e = cudaSuccess;
  switch (mode * 2 + (bf16 ? 1 : 0)) {
    case kMmaFfnGated * 2: e = max_clusters<kMmaFfnGated, false>(cs, smem, &nc); break;
    case kMmaFfnGated * 2 + 1: e = max_clusters<kMmaFfnGated, true>(cs, smem, &nc); break;
    case kMmaFfnUp * 2: e = max_clusters<kMmaFfnUp, false>(cs, smem, &nc); break;
    case kMmaFfnUp * 2 + 1: e = max_clusters<kMmaFfnUp, true>(cs, smem, &nc); break;
    case kMmaHidden * 2: e = max_clusters<kMmaHidden, false>(cs, smem, &nc); break;
    case kMmaHidden * 2 + 1: e = max_clusters<kMmaHidden, true>(cs, smem, &nc); break;
    case kMmaHeads * 2: e = max_clusters<kMmaHeads, false>(cs, smem, &nc); break;
    case kMmaHeads * 2 + 1: e = max_clusters<kMmaHeads, true>(cs, smem, &nc); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if (nc < 1) nc = 1;
  if (nc * cs > n_sms) nc = n_sms / cs;
  if (want_clusters > 0 && want_clusters < nc) nc = want_clusters;
  p->cs = cs;
  p->ks_len = ks;
  p->n_clusters = nc;
  p->n_stages = ns;
  p->stage_bytes = stage;
  p->smem = smem;
  return cudaSuccess;
}

cudaError_t launch_mma_rows(int mode, int bf16, const RowMaps& map, const MmaArgs& a_in, const MmaPlan& p,
                            cudaStream_t st) {
  MmaArgs a = a_in;
  a.cs = p.cs;
  a.ks_len = p.ks_len;
  a.n_clusters = p.n_clusters;
  a.n_stages = p.n_stages;
  a.stage_bytes = p.stage_bytes;
  if (a.B < 1 || a.B > 8 || a.Kdim != p.ks_len * p.cs) return cudaErrorInvalidValue;
  switch (mode * 2 + (bf16 ? 1 : 0)) {
    case kMmaFfnGated * 2: return launch_mode<kMmaFfnGated, false>(map, a, p.smem, st);
    case kMmaFfnGated * 2 + 1: return launch_mode<kMmaFfnGated, true>(map, a, p.smem, st);
    case kMmaFfnUp * 2: return launch_mode<kMmaFfnUp, false>(map, a, p.smem, st);
    case kMmaFfnUp * 2 + 1: return launch_mode<kMmaFfnUp, true>(map, a, p.smem, st);
    case kMmaHidden * 2: return launch_mode<kMmaHidden, false>(map, a, p.smem, st);
    case kMmaHidden * 2 + 1: return launch_mode<kMmaHidden, true>(map, a, p.smem, st);
    case kMmaHeads * 2: return launch_mode<kMmaHeads, false>(map, a, p.smem, st);
    case kMmaHeads * 2 + 1: return launch_mode<kMmaHeads, true>(map, a, p.smem, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace np
