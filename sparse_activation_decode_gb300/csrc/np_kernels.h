// Host-side launch interfaces of the decode-path kernels (internal to the
// library; the public boundary is include/np.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace np {

// Device error codes written to the model's error word.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrBounds = 2;

constexpr int kThreads = 256;          // CTA size of the streaming kernels
constexpr int kMaxChunksPerThread = 4; // 16-byte chunks per row <= kThreads * 4

// ---- FFN over a row list (np_ffn.cu) -------------------------------------
struct FfnLaunch {
  const float* h_in;      // [D] residual stream entering the layer
  const void* w_gate;     // [rows][D] or null when !gated
  const void* w_up;       // [rows][D]
  const void* w_down;     // [rows][D] (down^T rows)
  const int* row_list;    // rows to use, or null for rows 0..n-1
  const int* n_rows_dev;  // device count, or null to use n_rows_host
  int n_rows_host;
  int list_cap;           // capacity of row_list (upper bound of the count)
  int row_limit;          // rows present in the weight buffers
  float* part;            // [grid][D] per-CTA partial y
  int D;
  int dtype;              // 0 f32, 1 f16, 2 bf16
  int dtype_bytes;
  int gated;
  int n_stages;
  int grid;
  int* err;
};
size_t ffn_smem_bytes(int D, int dtype_bytes, int nproj, int n_stages);
int ffn_pick_stages(int D, int dtype_bytes, int nproj, size_t smem_limit);
cudaError_t launch_ffn_rows(const FfnLaunch& a, cudaStream_t st);
cudaError_t launch_ffn_finish(const float* part, int n_part, int D, const float* h_in, float* h_out, float* y_out,
                              cudaStream_t st);

// ---- row dot products: predictor layers (np_pred.cu) ----------------------
// out mode: 0 = relu(dot) -> out_f[row]; 1 = argmax key per head of C rows;
//           2 = dot + bias -> out_f[row], bit set in fire_bits where > 0.
struct RowdotLaunch {
  const void* W;          // [n_rows][len]
  int n_rows;
  int len;
  const float* vec;       // [len] fp32 input vector
  int vec_rmsnorm;        // 1: use rmsnorm(vec) instead of vec
  int mode;
  const void* bias;       // mode 2: [n_rows] of dtype
  float* out_f;           // modes 0, 2
  unsigned long long* keys;  // mode 1: [n_rows / C]
  int C;
  uint32_t* fire_bits;    // mode 2
  uint32_t* zero_ptr;     // words cleared by CTA 0 before anything else (may be null)
  int zero_words;
  int dtype;
  int dtype_bytes;
  int rows_per_stage;
  int n_stages;
  int grid;
  int* err;
};
size_t rowdot_smem_bytes(int len, int dtype_bytes, int rows_per_stage, int n_stages);
cudaError_t launch_rowdot(const RowdotLaunch& a, cudaStream_t st);
cudaError_t launch_keys_to_ids(const unsigned long long* keys, int n, int* ids, cudaStream_t st);

// ---- active set, delta, slot assignment (np_set.cu) -----------------------
struct SetLaunch {
  int n_layers_launch;    // CTAs: layers handled by this launch
  int first_sparse;       // sparse index of CTA 0
  int n_dense;            // absolute layer of sparse index 0
  int F, K, C, words;
  int combine;            // 0 intersect, 1 union
  int window;             // 1 = slot-map policy (R = A)
  int batch;
  int n_heads;
  int token;
  const int* ids;         // [batch][n_heads] or null (fire mask mode)
  const uint32_t* fire;   // [n_layers_launch][words] or null
  const uint32_t* centroids;  // [S][2][C][words]
  uint64_t cur_bits;      // bit s: committed state lives in buffer 1 (else 0)
  // double-buffered state, each [2][S][...]
  int* slotmap;           // [2][S][F]
  int* inv;               // [2][S][K]
  int* content;           // [2][S][K]
  uint32_t* resbits;      // [2][S][words]
  int* last_seen;         // [2][S][F] (window > 1)
  int S;
  // outputs [S][...]
  int* counts;            // [S][4]
  int* active;            // [S][K]
  int* active_slot;       // [S][K]
  int* din_n;             // [S][K]
  int* din_s;             // [S][K]
  int* dout_n;            // [S][K]
  unsigned long long* totals;  // running sums: |A|, |D_in|, |D_out|, dropped
  int* err;
};
cudaError_t launch_set(const SetLaunch& a, cudaStream_t st);
cudaError_t launch_reset_state(int* slotmap, int* inv, uint32_t* resbits, int* last_seen, int S, int F, int K,
                               int words, cudaStream_t st);

// ---- host-link gather and deinterleave-scatter (np_scatter.cu) -----------
struct MoveLaunch {
  const void* store_layer;  // device-visible host store, base of this layer's records
  int rec_vec;              // record size in 16-byte units
  int row_vec;              // row size in 16-byte units
  int n_proj;
  int F;
  int K;
  const int* din_n;         // [K] incoming neurons (ascending)
  const int* din_s;         // [K] their slots
  const int* count;         // device |D_in|
  int chunk_begin;
  int chunk_cap;
  void* staging;            // [chunk_cap][rec_vec] device
  void* bufs_layer;         // [n_proj][K][row_vec] device
  const int* content_old;   // restore: neuron whose bytes were in each slot (-1: zero)
  int grid;
  int* err;
};
cudaError_t launch_gather(const MoveLaunch& a, cudaStream_t st);    // host store -> staging
cudaError_t launch_scatter(const MoveLaunch& a, cudaStream_t st);   // staging -> buffers
cudaError_t launch_fused(const MoveLaunch& a, cudaStream_t st);     // host store -> buffers
cudaError_t launch_restore(const MoveLaunch& a, cudaStream_t st);   // previous slot contents back

}  // namespace np
