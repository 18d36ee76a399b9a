/*
 * np.h — C ABI of the per-token sparse-MLP decode path on one GB300 (sm_103a).
 *
 * The path (NeuroPrefetcher: Storage-Aware Sparse LLM Inference via Delta
 * Prefetching, section 3.1 System Overview and the full text's Figure 2
 * execution flow): run the dense prefix, run the shared predictor once after
 * layer 0, turn its centroid IDs into each sparse layer's active set, diff
 * that set against the rows already resident in the layer's K_max-row buffer,
 * fetch only the incoming rows from the storage tier and scatter them into
 * the buffer, then run the sparse FFN over the resident active rows.
 *
 * Storage tier: a host weight store in CPU memory that the GPU can read
 * (page-locked, host-registered, or ATS-visible), standing in for the NVMe
 * file of neuron-centric records.  Records are read by a gather kernel over
 * the host link into a device staging buffer; a deinterleave-scatter kernel
 * then writes each record's rows into the projection buffers.
 *
 * Conventions for every call:
 *  - Work is enqueued on the model's streams and is asynchronous unless the
 *    call says otherwise.  Results in device memory are valid once the caller
 *    has synchronised `main_stream`.
 *  - Buffers passed in are owned by the caller and must stay valid until the
 *    work using them has completed.  The library owns the resident projection
 *    buffers, slot maps, staging buffer and workspaces it allocates in
 *    np_init_model and frees in np_free_model.
 *  - Every call returns an np_status.  No C++ exception and no process exit
 *    crosses this boundary.  On error the call has enqueued nothing that
 *    changes the committed decode state (slot maps, resident buffers, window
 *    history), except where a call says otherwise.
 *  - Device-side waits are bounded: a kernel that waits longer than about one
 *    second records NP_ERR_TIMEOUT in the model's error word, which the next
 *    synchronising call (np_decode_token with stats, np_get_state,
 *    np_check_error) reports.
 */
#ifndef NP_H
#define NP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t np_status;
#define NP_OK 0
#define NP_ERR_ARG (-1)     /* invalid argument: null pointer, size out of range, bad layer */
#define NP_ERR_OOM (-2)     /* a device allocation failed */
#define NP_ERR_CUDA (-3)    /* a CUDA runtime call failed; np_last_error() has its text */
#define NP_ERR_IO (-4)      /* the storage read hook reported a failed read */
#define NP_ERR_TIMEOUT (-5) /* a bounded device wait expired */
#define NP_ERR_STATE (-6)   /* call out of order, e.g. np_scatter with no pending delta */

/* element type of every weight tensor */
#define NP_F32 0
#define NP_F16 1
#define NP_BF16 2

/* how the gate and up centroid masks form the active set (NeuroPrefetcher
 * section 3.4: the masks are intersected; the measured configuration here
 * uses their union) */
#define NP_COMBINE_INTERSECT 0
#define NP_COMBINE_UNION 1

/* residency policy: slot map with resident set = active set (NeuroPrefetcher
 * full text, delta runtime), or the last `window` tokens' active sets (LLM in
 * a flash, section 3.1 Windowing), or frequency-weighted caching (DynamicInfer,
 * hierarchical neuron cache, importance a + lambda f): the active set plus
 * the previous residents, the non-active ones active in the fewest tokens of
 * the sequence evicted first (ties: lowest ID) while more than k_max remain */
#define NP_RES_SLOTMAP 0
#define NP_RES_WINDOW 1
#define NP_RES_FREQUENCY 2

/* predictor: one shared predictor after layer 0 with a per-head argmax over
 * the centroid vocabulary (NeuroPrefetcher section 3.3), or one low-rank
 * predictor per layer firing where its logit is positive (LLM in a flash,
 * section 3.1) */
#define NP_PRED_SHARED_ARGMAX 0
#define NP_PRED_PERLAYER_SIGMOID 1

/* host-to-device path of the incoming rows: gather into the device staging
 * buffer then deinterleave-scatter (NeuroPrefetcher section 3.5), or one fused
 * kernel that reads host records and writes the projection buffers */
#define NP_H2D_STAGED 0
#define NP_H2D_FUSED 1

/* activation of a gated FFN: relu(g.x) * (u.x) (ReLU-fied), or
 * silu(g.x) * (u.x) (SwiGLU, NeuroPrefetcher "Predictive Delta Prefetching")
 * over the same predicted rows.  Models without a gate use relu(u.x). */
#define NP_ACT_RELU 0
#define NP_ACT_SWIGLU 1

/* placement of resident rows in a layer's buffers: freed slots are reused
 * in place (NeuroPrefetcher full text, delta runtime), or the rows are kept
 * contiguous in [0, |R|) (LLM in a flash, section 3.3 "Optimized Data
 * Management in DRAM"): with n = |R_prev| - |D_out|, each slot below n freed
 * by D_out receives a kept row from [n, |R_prev|) (the i-th freed slot in
 * ascending order the i-th such row in ascending order, one device-side row
 * copy each) and D_in is appended at n, n + 1, ... in ascending ID order.
 * Under the compact placement the sparse FFN covers the whole occupied
 * region (that section's [:num_rows] views): the active set, plus the rows
 * that windowing keeps. */
#define NP_SLOTS_REUSE 0
#define NP_SLOTS_COMPACT 1

/* Optional storage read hook, called on the host once per sparse layer before
 * that layer's records are read, with the layer index (absolute) and the
 * token counter.  A non-zero return makes the read fail with NP_ERR_IO. */
typedef int32_t (*np_read_hook_fn)(void* ctx, int32_t layer, int32_t token);

typedef struct np_model np_model; /* opaque, library-owned */

typedef struct {
  int32_t n_layers;     /* L: total layers */
  int32_t n_dense;      /* d: layers 0..d-1 have fully resident FFNs (0..L) */
  int32_t d_model;      /* D: multiple of 8 (16-bit types) or 4 (f32), <= 8192 */
  int32_t d_ff;         /* F: intermediate width */
  int32_t k_max;        /* K: resident rows per sparse layer, 1..F */
  int32_t n_centroids;  /* C: centroids per (layer, projection), shared predictor */
  int32_t dtype;        /* NP_F32 | NP_F16 | NP_BF16 */
  int32_t has_gate;     /* 1: records gate|up|down^T; 0: up|down^T (OPT) */
  int32_t combine;      /* NP_COMBINE_* */
  int32_t residency;    /* NP_RES_* */
  int32_t window;       /* W for NP_RES_WINDOW, 1..32 */
  int32_t batch;        /* sequences decoded together, 1..8 */
  int32_t staging_rows; /* staging capacity in records; 0 means k_max.  A
                           layer delta larger than this is processed in
                           several gather+scatter chunks */
  int32_t pred_hidden;  /* H: predictor hidden width */
  int32_t pred_kind;    /* NP_PRED_* */
  int32_t h2d_mode;     /* NP_H2D_* */
  int32_t activation;   /* NP_ACT_* (NP_ACT_SWIGLU needs has_gate = 1) */
  int32_t slots;        /* NP_SLOTS_* (batch > 1 with NP_RES_WINDOW or
                           NP_RES_FREQUENCY needs NP_SLOTS_COMPACT) */
  int32_t lookahead;    /* per-layer predictor only: the predictor of layer l
                           reads the input of layer max(l - lookahead, 0)
                           (DynamicInfer, cross-layer sparse prediction), so
                           np_decode_token starts layer l's reads `lookahead`
                           layers early; 0..n_layers, 0 = its own input */
  /* Host weight store (caller-owned, CPU memory the device can read; e.g.
   * registered with np_host_register).  Layout: record-major per sparse
   * layer, [L-d][F][n_proj][D] elements of `dtype`, n_proj = 3 (gate, up,
   * down^T row of neuron n) or 2 (up, down^T) — the neuron-centric record of
   * NeuroPrefetcher section 3.5 / LLM in a flash section 3.2. */
  const void* host_store;
  /* Dense-prefix weights (device, caller-owned): [d][3][F][D] = gate rows,
   * up rows, down^T rows (2 instead of 3 when has_gate = 0). */
  const void* dense_w;
  /* Predictor (device, caller-owned).  Shared: W1 [H][D], W2 [2(L-1) C][H],
   * b2 NULL.  Per layer: W1 [L][H][D], W2 [L][F][H], b2 [L][F]. */
  const void* pred_w1;
  const void* pred_w2;
  const void* pred_b2;
  /* Centroid masks (device, caller-owned), shared predictor only:
   * [L-d][2][C][ceil(F/32)] uint32, bit n of a mask in word n/32, bit n%32;
   * projection 0 = gate, 1 = up. */
  const uint32_t* centroids;
  void* main_stream;    /* cudaStream_t for the FFN / predictor / set kernels */
  void* side_stream;    /* cudaStream_t for the host-link gather and scatter */
  np_read_hook_fn read_hook; /* optional, may be NULL */
  void* read_ctx;
} np_model_desc;

/* Device views of the last delta (library-owned, valid until the next
 * np_delta / np_decode_token).  Per sparse layer s = layer - n_dense, arrays
 * of k_max int32 each; only the first count entries are meaningful. */
typedef struct {
  int32_t n_sparse;
  int32_t k_max;
  const int32_t* counts;      /* [S][4]: |A|, |D_in|, |D_out|, dropped by the K_max cap */
  const int32_t* active;      /* [S][K]: active neuron IDs, ascending */
  const int32_t* active_slot; /* [S][K]: slot of each active neuron */
  const int32_t* din_neuron;  /* [S][K]: incoming neuron IDs, ascending */
  const int32_t* din_slot;    /* [S][K]: slot assigned to each incoming neuron */
  const int32_t* dout_neuron; /* [S][K]: outgoing neuron IDs, ascending */
  const int32_t* ids;         /* shared predictor: [batch][2(L-1)] centroid IDs of the
                                 last prediction; NULL for the per-layer predictor */
  const int32_t* move_count;  /* [S]: row moves of the compact placement (0 otherwise) */
  const int32_t* move_src;    /* [S][K]: slot each moved row came from; NULL unless compact */
  const int32_t* move_dst;    /* [S][K]: slot it went to (a slot freed by D_out) */
} np_delta_view;

typedef struct {
  int64_t token;         /* tokens decoded since the last cold start, before this one */
  int64_t active_rows;   /* sum over sparse layers of |A| */
  int64_t din_rows;      /* sum of |D_in| (rows read from the storage tier) */
  int64_t dout_rows;     /* sum of |D_out| */
  int64_t dropped_rows;  /* rows removed by the K_max cap */
  int64_t h2d_bytes;     /* din_rows * record bytes */
  int64_t moved_rows;    /* records copied inside device memory by the compact placement */
} np_stats;

/* Create a model from `desc`; allocates device state (resident buffers
 * [L-d][n_proj][K][D], slot maps, staging, workspaces).  The first token
 * after creation is a cold start.  Synchronous.  Errors: NP_ERR_ARG,
 * NP_ERR_OOM, NP_ERR_CUDA; *out is set only on NP_OK. */
np_status np_init_model(const np_model_desc* desc, np_model** out);

/* Wait for the model's streams and free everything it allocated.  NULL is
 * accepted.  Synchronous. */
np_status np_free_model(np_model* m);

/* Forget the resident sets: the next token loads its full predicted set, as
 * at a sequence's first token (NeuroPrefetcher section 3.4 cold start).
 * Resident buffer bytes are kept. */
np_status np_reset_sequence(np_model* m);

/* Predictor.  Shared kind: layer must be 0; h_dev = residual stream after
 * layer 0, float32 [batch][D]; out_dev = int32 [batch][2(L-1)] centroid IDs,
 * head 2(l-1) = gate of layer l, 2(l-1)+1 = up (NeuroPrefetcher section 3.3;
 * ties go to the lowest centroid index).  Per-layer kind: layer = the sparse
 * layer to predict, h_dev = that layer's input [D]; out_dev = uint32
 * [ceil(F/32)] firing mask, bit n set where logit_n > 0. */
np_status np_predict(np_model* m, int32_t layer, const float* h_dev, void* out_dev);

/* Active set, delta and slot assignment.  layer = -1: every sparse layer from
 * the shared predictor's IDs (pred_dev = int32 [batch][2(L-1)]).  layer = l:
 * only sparse layer l; pred_dev is the IDs (shared) or the firing mask
 * (per layer).  A = gate mask combined with up mask (union over the batch),
 * capped to the K_max lowest IDs; D_in = A minus R_prev, D_out = R_prev minus
 * R_next; incoming neurons in ascending ID order take free slots in ascending
 * slot order (NeuroPrefetcher full text, delta runtime and slot map).  The
 * new state is written in place and stays pending until np_scatter succeeds
 * (a failed read rolls it back).  `out` may be NULL.  Errors: NP_ERR_ARG,
 * NP_ERR_STATE (a delta for that layer is already pending). */
np_status np_delta(np_model* m, int32_t layer, const void* pred_dev, np_delta_view* out);

/* Views of the last computed delta and predictor output (e.g. after
 * np_decode_token).  Does not synchronise. */
np_status np_last_delta(np_model* m, np_delta_view* out);

/* Read the pending delta's incoming records from the host store and scatter
 * their rows into the resident buffers at the assigned slots, chunked by the
 * staging capacity (NeuroPrefetcher section 3.5, launch_deinterleave_scatter;
 * "independent submit-and-scatter chunks"); under the compact placement the
 * delta's row moves inside the buffers run first.  layer = -1: all pending layers;
 * layer = l: that layer only.  On success the pending state is committed.
 * If the read hook fails, rows already written are restored from the store,
 * every pending delta is rolled back, and NP_ERR_IO is returned with the
 * state as before the deltas. */
np_status np_scatter(np_model* m, int32_t layer);

/* Sparse FFN of sparse layer `layer` over its resident active rows, read
 * through the slot map (the occupied rows [0, |R|) under the compact
 * placement): x = rmsnorm(h) (no weight, eps 1e-6),
 * h_n = relu(g_n . x)(u_n . x) (or relu(u_n . x) without a gate),
 * y = sum_n h_n d_n.  h_dev, y_dev: float32 [batch][D]; y_dev may not alias
 * h_dev.  Uses the committed state. */
np_status np_sparse_mlp(np_model* m, int32_t layer, const float* h_dev, float* y_dev);

/* Full FFN of dense layer `layer` < n_dense, same formula over all F neurons. */
np_status np_dense_mlp(np_model* m, int32_t layer, const float* h_dev, float* y_dev);

/* FFNs of layers first .. first+count-1 (dense or sparse) for every
 * sequence on the committed resident rows, one after another, with the
 * residual stream h_dev [batch][D] float32 updated in place: for each layer
 * h += FFN(rmsnorm(h)) — the FFN part of np_decode_token, without the
 * prediction and transfer steps (for callers that run np_predict, np_delta
 * and np_scatter themselves).  Errors: NP_ERR_ARG for a bad range,
 * NP_ERR_STATE if a delta is pending for a layer in the range. */
np_status np_ffn_layers(np_model* m, int32_t first, int32_t count, float* h_dev);

/* One decode step for all sequences: dense prefix, predictor, delta,
 * host-link gather and scatter on the side stream overlapped with the FFNs on
 * the main stream (each sparse layer waits only for its own rows), sparse
 * suffix; h_dev [batch][D] float32 is the residual stream in and out.
 * stats_host may be NULL; when given, the call synchronises and fills it.
 * On an error return the contents of h_dev are unspecified; the committed
 * decode state is unchanged.
 * The first call issues its kernels one by one; later calls replay a CUDA
 * graph of one token captured once (h_dev is copied into and out of an
 * internal buffer on main_stream), except while a read hook is set or
 * profiling is on, which issue the kernels one by one.  Both ways enqueue the
 * same kernels on the same data.  The environment variable NP_TUNE_GRAPH=0
 * (read at np_init_model) turns replay off. */
np_status np_decode_token(np_model* m, float* h_dev, np_stats* stats_host);

/* Copy the committed slot map [F] and inverse map [K] of sparse layer
 * `layer` to host memory (either pointer may be NULL).  Synchronous.
 * NP_ERR_STATE while a delta is pending for that layer. */
np_status np_get_state(np_model* m, int32_t layer, int32_t* slotmap_host, int32_t* inv_host);

/* Device pointer to resident buffer `proj` (0..n_proj-1) of sparse layer
 * `layer`: [K][D] elements of dtype, row = slot.  Library-owned. */
np_status np_resident_rows(np_model* m, int32_t layer, int32_t proj, const void** dev_ptr);

/* Read the counts of the last delta into host memory: [S][4] as in
 * np_delta_view.counts.  Synchronous. */
np_status np_get_counts(np_model* m, int32_t* counts_host);

/* Synchronise the model's streams and report a device-side error
 * (NP_ERR_TIMEOUT) or an asynchronous CUDA error, clearing it. */
np_status np_check_error(np_model* m);

/* Per-kernel timing with CUDA events recorded on each kernel's own stream.
 * When enabled, every launch of the kinds below is bracketed by events and
 * the summed durations are available from np_get_profile (synchronous).
 * enable = 1: plain events; a launch that waits on another stream may be
 * stamped as starting before its wait is over (an upper bound of its
 * duration).  enable = 2: an empty kernel is launched in front of each start
 * event so that it follows the launch's dependencies (exact durations, one
 * extra launch per kernel).  0 turns timing off. */
#define NP_KIND_DENSE 0
#define NP_KIND_PRED 1
#define NP_KIND_SET 2
#define NP_KIND_GATHER 3
#define NP_KIND_SCATTER 4
#define NP_KIND_FFN 5
#define NP_KIND_FINISH 6
#define NP_N_KINDS 7
np_status np_set_profiling(np_model* m, int32_t enable);
/* ms_out[NP_N_KINDS]: summed milliseconds; launches_out[NP_N_KINDS]: launch
 * counts; bytes_out[NP_N_KINDS]: algorithmic bytes moved by those launches.
 * Any pointer may be NULL.  Resets the accumulators. */
np_status np_get_profile(np_model* m, double* ms_out, int64_t* launches_out, int64_t* bytes_out);

/* Timeline of the launches timed since the last np_get_profile, in issue
 * order: kind (NP_KIND_*), start and end in milliseconds relative to the
 * first one (events recorded on each launch's own stream).  Writes at most
 * max_entries entries and their count to *n_out.  Synchronous. */
np_status np_get_timeline(np_model* m, int32_t* kinds, float* start_ms, float* end_ms, int32_t max_entries,
                          int32_t* n_out);

/* Make a caller-owned host range readable by the device (page-locked,
 * mapped).  Synchronous.  Unregister before freeing the memory. */
np_status np_host_register(void* ptr, size_t bytes);
np_status np_host_unregister(void* ptr);

/* Allocation-free FFN over caller-provided rows (no counterpart on the
 * pages: an addition for callers that cannot allocate device memory, e.g. a
 * serving loop whose allocator owns a fixed memory budget, or a
 * latency-critical path where cudaMalloc would synchronize the device).
 * Computes y = sum over the listed rows r of relu(g_r . x)(u_r . x) d_r
 * (relu(u_r . x) d_r when has_gate = 0) with x = rmsnorm(h) — the kernel of
 * np_sparse_mlp — and writes y_dev [d_model].  Rows: rows_dev[0..n_rows) are
 * int32 row indices into w_gate/w_up/w_down ([row_limit][d_model] each, all
 * three of that size), or NULL for rows 0..n_rows-1; n_rows = 0 gives y = 0.
 * All pointers are device pointers, 16-byte aligned (rows_dev: 4-byte);
 * dtype NP_F32/NP_F16/NP_BF16; d_model in [8, 8192], rows a multiple of 16
 * bytes.  y_dev may share no byte with h_dev, the weights or the row list
 * (it is cleared on the stream before the kernel runs).  Enqueued on
 * `stream` (cudaStream_t); the call allocates nothing: y_dev is cleared on
 * the stream and then accumulated into, and the kernel's error word lives
 * in a file-scope device array (256 bytes) whose address the first call on
 * each device looks up, so make that first call before any stream capture.
 * All calls share the array: calls that overlap on the GPU race.
 * Errors returned: NP_ERR_ARG for sizes, pointers or overlaps out of range,
 * NP_ERR_CUDA if a launch fails.  Errors found by the kernel (a row index
 * >= row_limit, for which it reads row 0 instead and so returns a wrong y;
 * a bounded wait that expired, leaving y partial) are recorded in the shared
 * error word and reported by np_ffn_rows_noalloc_check. */
np_status np_ffn_rows_noalloc(const float* h_dev, const void* w_gate, const void* w_up, const void* w_down,
                              const int32_t* rows_dev, int32_t n_rows, int32_t row_limit, int32_t d_model,
                              int32_t dtype, int32_t has_gate, float* y_dev, void* stream);

/* Synchronise `stream`, then read and clear the current device's error word
 * of np_ffn_rows_noalloc: NP_ERR_STATE if a row index was out of range,
 * NP_ERR_TIMEOUT if a device wait expired, in any call since the previous
 * check (the last such error wins); NP_OK if none; NP_ERR_CUDA if the stream
 * holds an asynchronous CUDA error.  Allocates nothing. */
np_status np_ffn_rows_noalloc_check(void* stream);

/* Number of kernel launches the model has issued since creation. */
int64_t np_launch_count(np_model* m);

const char* np_status_str(np_status s);
/* Text of the last CUDA error seen by any call on this thread. */
const char* np_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* NP_H */
