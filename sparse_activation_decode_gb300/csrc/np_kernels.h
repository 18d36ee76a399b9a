// Host-side launch interfaces of the decode-path kernels (internal to the
// library; the public boundary is include/np.h).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace np {

// Device error codes written to the model's error word.
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrBounds = 2;

constexpr int kThreads = 256;          // CTA size of the streaming kernels
constexpr int kMaxChunksPerThread = 4; // 16-byte chunks per row <= kThreads * 4

// ---- FFN over a row list (np_ffn.cu) -------------------------------------
struct FfnLaunch {
  const float* h_in;      // [D] residual base entering the layer
  const float* yprev;     // [D] previous layer's y (h = h_in + yprev), or null
  float* hb_out;          // CTA 0 stores h here, or null
  float* y_acc;           // [D] y is added here (cleared beforehand)
  float* y_zero;          // [D] CTA 0 clears it (the accumulator after next), or null
  const void* w_gate;     // [rows][D] or null when !gated
  const void* w_up;       // [rows][D]
  const void* w_down;     // [rows][D] (down^T rows)
  const int* row_list;    // rows to use, or null for rows 0..n-1
  const int* n_rows_dev;  // device count, or null to use n_rows_host
  int n_rows_host;
  int list_cap;           // capacity of row_list (upper bound of the count)
  int row_limit;          // rows present in the weight buffers
  int D;
  int dtype;              // 0 f32, 1 f16, 2 bf16
  int dtype_bytes;
  int gated;
  int swiglu;             // gated: silu(g.x) instead of relu(g.x)
  int n_stages;
  int grid;
  int pdl;                  // launch with programmatic dependent launch
  int* err;
};
size_t ffn_smem_bytes(int D, int dtype_bytes, int nproj, int n_stages);
// Ring depth and grid (two CTAs per SM) of the FFN launch.
cudaError_t ffn_plan(int dtype, int gated, int D, int dtype_bytes, size_t smem_per_sm, int n_sms, int* n_stages,
                     int* grid);
int ffn_max_chunks();        // 16-byte chunks per row the FFN supports
void set_last_error(const char* what);  // text returned by np_last_error() on this thread
// Persistent FFN over consecutive layers first..first+count-1 (batch 1),
// launched cooperatively: one CTA per SM, two arrival counters per layer
// (partials stored; y slices summed).  The split-K order is fixed.
struct FfnChainLaunch {
  const void* dense_w;       // [n_dense][n_proj][F][D]
  const void* bufs;          // [S][n_proj][K][D] resident rows
  const int* active_slot;    // [S][K]
  const int* counts;         // [S][4] (|A| first)
  const int* n_rows;         // [S] occupied rows; with `compact` the FFN covers rows [0, n_rows)
  int compact;
  int n_dense, F, K;
  int first, count;
  float* h;                  // [D] residual stream, in and out
  float* hbase;              // [2][D] residual bases
  float* yacc;               // [3][D] layer outputs y
  float* part;               // [grid][D] per-CTA partial y
  unsigned* arrive;          // [2 count] arrival counters, zero beforehand
  int D, dtype, dtype_bytes, gated, swiglu, n_stages, grid;
  int* err;
  // Optional reads of each sparse layer's incoming records inside the same
  // launch (per-token pipeline); g_store = null: the rows are resident.
  const void* g_store;       // device-visible host store [S][F][n_proj][D]
  const int* din_n;          // [S][K] incoming neurons
  const int* din_s;          // [S][K] their slots
  unsigned* gdone;           // [count] CTAs done reading layer first+i, zero beforehand
  // Failure test hook: CTA 0's readers skip their arrival for chain layer
  // `withhold` (-1: none), so that layer's count never completes and the
  // bounded waits behind it run out (the kernel reports a timeout and exits).
  int withhold;
};
cudaError_t ffn_chain_plan(int dtype, int gated, int D, int dtype_bytes, size_t smem_optin, int n_sms,
                           int* n_stages, int* grid);
cudaError_t launch_ffn_chain(const FfnChainLaunch& a, cudaStream_t st);
// Allow the dynamic shared memory of an n_stages ring (after changing it).
cudaError_t ffn_set_smem(int dtype, int gated, int D, int dtype_bytes, int n_stages);
cudaError_t launch_ffn_rows(const FfnLaunch& a, cudaStream_t st);

// ---- row dot products: predictor layers (np_pred.cu) ----------------------
// out mode: 0 = relu(dot) -> out_f[row]; 1 = argmax key per head of C rows;
//           2 = dot + bias -> out_f[row], bit set in fire_bits where > 0.
struct RowdotLaunch {
  const void* W;          // [n_rows][len]
  int n_rows;
  int len;
  const float* vec;       // [len] fp32 input vector
  const float* vec2;      // added to vec before the rmsnorm, or null
  int vec_rmsnorm;        // 1: use rmsnorm(vec + vec2) instead of vec
  int mode;
  const void* bias;       // mode 2: [n_rows] of dtype
  float* out_f;           // modes 0, 2
  unsigned long long* keys;  // mode 1: [n_rows / C]
  int C;
  uint32_t* fire_bits;    // mode 2
  uint32_t* zero_ptr;     // words cleared by CTA 0 once the previous kernel has completed (may be null)
  int zero_words;
  int dtype;
  int dtype_bytes;
  int rows_per_stage;
  int n_stages;
  int grid;
  int pdl;                // launch with programmatic dependent launch
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
  int window;             // > 1: window residency over the last `window` tokens
  int frequency;          // 1: frequency-weighted residency (last_seen holds activation counts)
  int batch;
  int n_heads;
  int token;
  const int* token_dev;   // device token counter, read instead of `token` when set
  const int* ids;         // [batch][n_heads] or null
  const unsigned long long* keys;  // packed argmax keys [batch][n_heads] (used if ids null)
  int* ids_out;           // with keys: CTA 0 also writes the decoded IDs here
  const uint32_t* fire;   // [n_layers_launch][words] or null
  const uint32_t* centroids;  // [S][2][C][words]
  // decode state, updated in place: [S][...]
  int* slotmap;           // [S][F] slot of each neuron or -1
  int* inv;               // [S][K] neuron in each slot or -1
  int* content;           // [S][K] neuron whose rows the slot's bytes hold or -1
  uint32_t* resbits;      // [S][words] resident set
  int* last_seen;         // [S][F] last active token (window > 1) or activation count (frequency)
  int S;
  // delta lists [S][...]
  int* counts;            // [S][4]
  int* active;            // [S][K]
  int* active_slot;       // [S][K]
  int* din_n;             // [S][K]
  int* din_s;             // [S][K]
  int* din_oldct;         // [S][K] previous content of each incoming slot
  int* dout_n;            // [S][K]
  int* dout_s;            // [S][K] slot each outgoing neuron held
  int* ls_old;            // [S][K] previous last use of each active neuron
  unsigned long long* totals;  // running sums: |A|, |D_in|, |D_out|, dropped
  int pdl;                // launch with programmatic dependent launch
  int* slot_hw;           // [S] one past the highest occupied slot (an upper bound), or null;
                          // exactly |R| under the compact placement
  // compact placement: rows stay in [0, |R|); freed slots below the new count
  // are refilled from the end of the region, incoming rows are appended
  int compact;
  int* mv_src;            // [S][K] row moves, slot read
  int* mv_dst;            // [S][K] slot written (a slot freed by D_out)
  int* mv_oldct;          // [S][K] previous content of each written slot
  int* mv_count;          // [S] number of moves
  int* err;
};
cudaError_t launch_set(const SetLaunch& a, cudaStream_t st);
cudaError_t launch_rollback(const SetLaunch& a, cudaStream_t st);  // undo launch_set from its lists
// Cold state: empty maps and resident sets, zero high-water marks and (if
// given) zero activation counts [S][F].
cudaError_t launch_reset_state(int* slotmap, int* inv, uint32_t* resbits, int* slot_hw, int* counts, int S, int F,
                               int K, int words, cudaStream_t st);

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
  const int* din_oldct;     // restore: neuron whose bytes each incoming slot held (-1: zero)
  const int* mv_src;        // compact placement: row moves inside the buffers
  const int* mv_dst;
  const int* mv_oldct;      // restore: neuron whose bytes each move target held
  const int* mv_count;      // device number of moves, or null (no moves)
  int grid;
  int* err;
};
cudaError_t launch_gather(const MoveLaunch& a, cudaStream_t st);    // host store -> staging
cudaError_t launch_scatter(const MoveLaunch& a, cudaStream_t st);   // staging -> buffers
cudaError_t launch_fused(const MoveLaunch& a, cudaStream_t st);     // host store -> buffers
cudaError_t launch_restore(const MoveLaunch& a, cudaStream_t st);   // previous slot contents back
cudaError_t launch_move_rows(const MoveLaunch& a, cudaStream_t st); // bufs[dst] = bufs[src] per move


// ---- batched row products on the tensor cores (np_mma.cu) ----------------
// Modes: FFN with gate (gate, up, down^T), FFN without gate (up, down^T),
// predictor hidden layer (relu, written as hi/lo 16-bit operands), predictor
// heads (argmax keys per head of C rows).
enum { kMmaFfnGated = 0, kMmaFfnUp = 1, kMmaHidden = 2, kMmaHeads = 3 };
struct MmaArgs {
  int Kdim;                 // contraction length (d_model, or the hidden width for the heads)
  int ks_len, cs, n_clusters, B;  // column slice per CTA, cluster size, clusters, sequences (<= 8)
  const int* occ_inv;       // row r is used only if occ_inv[r] >= 0 (slot occupancy), or null: all rows
  const int* n_rows_dev;    // device row count (rows 0..n-1), or null to use n_rows_host
  int n_rows_host;
  int row_cap;              // upper bound of the row count
  int row_base0, row_base1, row_base2;  // tensor-map row of row 0 for each projection
  int oob_row;              // a tensor-map row past the end (reads as zeros)
  const float* hb;          // [B][Kdim] residual base (FFN, hidden)
  const float* yprev;       // [B][Kdim] previous layer's y, or null
  float* hb_out;            // hb + yprev is stored here (cluster 0), or null
  float* y_acc;             // FFN: y is added here, [B][Kdim]
  float* y_zero;            // cleared by cluster 0 (the next layer's accumulator), or null
  const uint16_t* zin;      // heads: [16][Kdim] hi/lo input operand
  uint16_t* zout;           // hidden: [16][zout_stride] hi/lo output
  int zout_stride;
  unsigned long long* keys; // heads: [B][n_heads] packed argmax keys
  int n_heads, C;
  unsigned long long* keys_zero;  // hidden: cleared before the heads run
  int n_keys_zero;
  int swiglu;               // gated FFN: silu(g.x) instead of relu(g.x)
  int n_stages;
  uint32_t stage_bytes;
  int pdl;                  // launch with programmatic dependent launch
  int* err;
};
struct MmaPlan {
  int cs, ks_len, n_clusters, n_stages;
  uint32_t stage_bytes;
  size_t smem;
};
// Two 2-D tensor maps over [rows][cols] 16-bit values with 128-byte swizzle
// and boxes of {64, 32} and {64, 8} (dtype 1 = f16, 2 = bf16).
struct RowMaps {
  CUtensorMap m32, m8;
};
cudaError_t make_row_maps(RowMaps* out, const void* base, int dtype, uint64_t rows, uint64_t cols);
size_t mma_smem_bytes(int mode, int ks_len, int n_stages);
// want_clusters > 0 caps the clusters; max_stages > 1 caps the ring depth.
cudaError_t mma_plan(int mode, int bf16, int Kdim, size_t smem_optin, int n_sms, int want_clusters, int max_stages,
                     MmaPlan* p);
cudaError_t launch_mma_rows(int mode, int bf16, const RowMaps& maps, const MmaArgs& a, const MmaPlan& p,
                            cudaStream_t st);
// out[i] = x[i] + y[i] (the residual stream after the last layer)
cudaError_t launch_add(float* out, const float* x, const float* y, int n, cudaStream_t st);

}  // namespace np
