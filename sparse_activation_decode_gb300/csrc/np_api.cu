// Host runtime behind the C ABI in include/np.h.
//
// Owns the per-model device state and orders the kernels of one decode step
// on two streams (NeuroPrefetcher full text, Figure 2 execution flow):
//
//   main: dense layer 0 -> predictor -> set/delta kernel -> [event set]
//         -> dense layers 1..d-1 -> for each sparse layer: wait for that
//         layer's rows, FFN, residual update
//   side: wait [event set] -> for each sparse layer: gather its incoming
//         records over the host link into staging, deinterleave-scatter them
//         into the layer's buffers (chunked by the staging capacity)
//         -> [event layer s]
//
// Decode state (slot maps, inverse maps, slot contents, resident bitmasks,
// window history) is double-buffered per sparse layer: the set kernel reads
// the committed half and writes the other; the host flips the layer's bit
// once its rows are in place, so a failed read leaves the committed state
// untouched (rows already overwritten are restored from the store).
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "np.h"
#include "np_kernels.h"

using namespace np;

namespace {
thread_local std::string g_last_err;

np_status cuda_fail(cudaError_t e, const char* what) {
  g_last_err = std::string(what) + ": " + cudaGetErrorString(e);
  return NP_ERR_CUDA;
}
np_status arg_fail(const char* what) {
  g_last_err = what;
  return NP_ERR_ARG;
}
}  // namespace

#define CUDA_TRY(expr)                                      \
  do {                                                      \
    cudaError_t _e = (expr);                                \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr);     \
  } while (0)

#define NP_TRY(expr)                     \
  do {                                   \
    np_status _s = (expr);               \
    if (_s != NP_OK) return _s;          \
  } while (0)

struct EventPair {
  cudaEvent_t a, b;
};

struct np_model {
  np_model_desc d{};
  int L = 0, dn = 0, S = 0, D = 0, F = 0, K = 0, C = 0, W = 0, B = 1, H = 0, NH = 0;
  int nproj = 3, esz = 2, staging_rows = 0, window = 1;
  int sms = 0;
  size_t smem_optin = 0;
  size_t row_bytes = 0, rec_bytes = 0;
  cudaStream_t main = nullptr, side = nullptr;
  const unsigned char* store_dev = nullptr;
  // device allocations
  void* bufs = nullptr;
  void* staging = nullptr;
  int *slotmap = nullptr, *inv = nullptr, *content = nullptr, *last_seen = nullptr;
  uint32_t* resbits = nullptr;
  int *counts = nullptr, *active = nullptr, *active_slot = nullptr, *din_n = nullptr, *din_s = nullptr,
      *dout_n = nullptr;
  unsigned long long* totals = nullptr;
  int* err = nullptr;
  float* z = nullptr;
  unsigned long long* keys = nullptr;
  int* ids = nullptr;
  uint32_t* fire = nullptr;
  float* logits = nullptr;
  float* part = nullptr;
  std::vector<void*> allocs;
  // launch shapes
  int ffn_grid = 0, ffn_stages = 0, ffn_stages_dense = 0;
  int gather_grid = 0, scatter_grid = 0, pred_grid = 0;
  int rps1 = 1, rps2 = 1, ns1 = 2, ns2 = 2;
  // state
  uint64_t cur_bits = 0, pending_bits = 0, committed_since_token = 0;
  int64_t token = 0;
  int64_t launches = 0;
  cudaEvent_t ev_set = nullptr, ev_side_done = nullptr;
  std::vector<cudaEvent_t> ev_layer;
  // profiling
  bool prof = false;
  std::vector<EventPair> prof_pending[NP_N_KINDS];
  std::vector<EventPair> prof_free;
  double prof_ms[NP_N_KINDS] = {};
  int64_t prof_launches[NP_N_KINDS] = {};
  int64_t prof_fixed_bytes[NP_N_KINDS] = {};
};

namespace {

uint64_t all_layers(const np_model* m) { return m->S >= 64 ? ~0ull : ((1ull << m->S) - 1ull); }

template <typename T>
np_status dev_alloc(np_model* m, T** p, size_t count, int fill_byte = 0) {
  void* q = nullptr;
  const size_t bytes = count * sizeof(T) > 0 ? count * sizeof(T) : 16;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    g_last_err = std::string("cudaMalloc: ") + cudaGetErrorString(e);
    return NP_ERR_OOM;
  }
  m->allocs.push_back(q);
  CUDA_TRY(cudaMemset(q, fill_byte, bytes));
  *p = static_cast<T*>(q);
  return NP_OK;
}

np_status prof_begin(np_model* m, int kind, cudaStream_t st, EventPair* ep) {
  (void)kind;
  if (m->prof_free.empty()) {
    EventPair p;
    CUDA_TRY(cudaEventCreate(&p.a));
    CUDA_TRY(cudaEventCreate(&p.b));
    m->prof_free.push_back(p);
  }
  *ep = m->prof_free.back();
  m->prof_free.pop_back();
  CUDA_TRY(cudaEventRecord(ep->a, st));
  return NP_OK;
}

np_status prof_fold(np_model* m, int kind, size_t keep) {
  auto& v = m->prof_pending[kind];
  if (v.size() <= keep) return NP_OK;
  const size_t n = v.size() - keep;
  for (size_t i = 0; i < n; ++i) {
    CUDA_TRY(cudaEventSynchronize(v[i].b));
    float ms = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&ms, v[i].a, v[i].b));
    m->prof_ms[kind] += ms;
    m->prof_free.push_back(v[i]);
  }
  v.erase(v.begin(), v.begin() + n);
  return NP_OK;
}

np_status prof_end(np_model* m, int kind, cudaStream_t st, const EventPair& ep) {
  CUDA_TRY(cudaEventRecord(ep.b, st));
  m->prof_pending[kind].push_back(ep);
  m->prof_launches[kind] += 1;
  if (m->prof_pending[kind].size() > 4096) NP_TRY(prof_fold(m, kind, 1024));
  return NP_OK;
}

// Launch one kernel (a callable returning cudaError_t), optionally timed.
template <typename Fn>
np_status launch(np_model* m, int kind, cudaStream_t st, int64_t fixed_bytes, Fn fn) {
  EventPair ep{};
  if (m->prof) NP_TRY(prof_begin(m, kind, st, &ep));
  cudaError_t e = fn();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  m->launches += 1;
  if (m->prof) {
    m->prof_fixed_bytes[kind] += fixed_bytes;
    NP_TRY(prof_end(m, kind, st, ep));
  }
  return NP_OK;
}

const unsigned char* layer_bufs(const np_model* m, int s) {
  return static_cast<const unsigned char*>(m->bufs) + (size_t)s * m->nproj * m->K * m->row_bytes;
}

// FFN over a row list followed by the partial-sum finish.
np_status enqueue_ffn(np_model* m, int kind, const unsigned char* base, size_t proj_stride, const int* rows,
                      const int* n_dev, int n_host, int list_cap, int row_limit, int stages, const float* h_in,
                      float* h_out, float* y_out, int64_t fixed_bytes) {
  FfnLaunch a{};
  a.h_in = h_in;
  int p = 0;
  a.w_gate = m->d.has_gate ? base + (p++) * proj_stride : nullptr;
  a.w_up = base + (p++) * proj_stride;
  a.w_down = base + p * proj_stride;
  a.row_list = rows;
  a.n_rows_dev = n_dev;
  a.n_rows_host = n_host;
  a.list_cap = list_cap;
  a.row_limit = row_limit;
  a.part = m->part;
  a.D = m->D;
  a.dtype = m->d.dtype;
  a.dtype_bytes = m->esz;
  a.gated = m->d.has_gate;
  a.n_stages = stages;
  a.grid = m->ffn_grid;
  a.err = m->err;
  cudaStream_t st = m->main;
  NP_TRY(launch(m, kind, st, fixed_bytes, [&] { return launch_ffn_rows(a, st); }));
  NP_TRY(launch(m, NP_KIND_FINISH, st, 0,
                [&] { return launch_ffn_finish(m->part, m->ffn_grid, m->D, h_in, h_out, y_out, st); }));
  return NP_OK;
}

np_status enqueue_dense(np_model* m, int layer, const float* h_in, float* h_out, float* y_out) {
  const size_t proj_stride = (size_t)m->F * m->row_bytes;
  const unsigned char* base =
      static_cast<const unsigned char*>(m->d.dense_w) + (size_t)layer * m->nproj * proj_stride;
  return enqueue_ffn(m, NP_KIND_DENSE, base, proj_stride, nullptr, nullptr, m->F, m->F, m->F, m->ffn_stages_dense,
                     h_in, h_out, y_out, (int64_t)m->nproj * m->F * m->row_bytes);
}

np_status enqueue_sparse(np_model* m, int s, const float* h_in, float* h_out, float* y_out) {
  const size_t proj_stride = (size_t)m->K * m->row_bytes;
  return enqueue_ffn(m, NP_KIND_FFN, layer_bufs(m, s), proj_stride, m->active_slot + (size_t)s * m->K,
                     m->counts + (size_t)s * 4, 0, m->K, m->K, m->ffn_stages, h_in, h_out, y_out, 0);
}

np_status enqueue_rowdot(np_model* m, const void* W, int n_rows, int len, const float* vec, int rms, int mode,
                         const void* bias, float* out_f, unsigned long long* keys, int C, uint32_t* fire,
                         uint32_t* zero_ptr, int zero_words, int rps, int ns) {
  RowdotLaunch a{};
  a.W = W;
  a.n_rows = n_rows;
  a.len = len;
  a.vec = vec;
  a.vec_rmsnorm = rms;
  a.mode = mode;
  a.bias = bias;
  a.out_f = out_f;
  a.keys = keys;
  a.C = C;
  a.fire_bits = fire;
  a.zero_ptr = zero_ptr;
  a.zero_words = zero_words;
  a.dtype = m->d.dtype;
  a.dtype_bytes = m->esz;
  a.rows_per_stage = rps;
  a.n_stages = ns;
  a.grid = m->pred_grid;
  a.err = m->err;
  cudaStream_t st = m->main;
  return launch(m, NP_KIND_PRED, st, (int64_t)n_rows * len * m->esz, [&] { return launch_rowdot(a, st); });
}

np_status enqueue_predict(np_model* m, int layer, const float* h) {
  if (m->d.pred_kind == NP_PRED_SHARED_ARGMAX) {
    NP_TRY(enqueue_rowdot(m, m->d.pred_w1, m->H, m->D, h, 1, 0, nullptr, m->z, nullptr, 0, nullptr,
                          reinterpret_cast<uint32_t*>(m->keys), 2 * m->NH, m->rps1, m->ns1));
    NP_TRY(enqueue_rowdot(m, m->d.pred_w2, m->NH * m->C, m->H, m->z, 0, 1, nullptr, nullptr, m->keys, m->C,
                          nullptr, nullptr, 0, m->rps2, m->ns2));
    cudaStream_t st = m->main;
    return launch(m, NP_KIND_PRED, st, 0, [&] { return launch_keys_to_ids(m->keys, m->NH, m->ids, st); });
  }
  const unsigned char* w1 = static_cast<const unsigned char*>(m->d.pred_w1) + (size_t)layer * m->H * m->row_bytes;
  const unsigned char* w2 =
      static_cast<const unsigned char*>(m->d.pred_w2) + (size_t)layer * m->F * m->H * m->esz;
  const unsigned char* b2 = static_cast<const unsigned char*>(m->d.pred_b2) + (size_t)layer * m->F * m->esz;
  NP_TRY(enqueue_rowdot(m, w1, m->H, m->D, h, 1, 0, nullptr, m->z, nullptr, 0, nullptr, m->fire, m->W, m->rps1,
                        m->ns1));
  return enqueue_rowdot(m, w2, m->F, m->H, m->z, 0, 2, b2, m->logits, nullptr, 0, m->fire, nullptr, 0, m->rps2,
                        m->ns2);
}

np_status enqueue_set(np_model* m, int first_sparse, int n_layers, const int* ids, const uint32_t* fire) {
  SetLaunch a{};
  a.n_layers_launch = n_layers;
  a.first_sparse = first_sparse;
  a.n_dense = m->dn;
  a.F = m->F;
  a.K = m->K;
  a.C = m->C;
  a.words = m->W;
  a.combine = m->d.combine;
  a.window = m->window;
  a.batch = m->B;
  a.n_heads = m->NH;
  a.token = (int)m->token;
  a.ids = ids;
  a.fire = fire;
  a.centroids = m->d.centroids;
  a.cur_bits = m->cur_bits;
  a.slotmap = m->slotmap;
  a.inv = m->inv;
  a.content = m->content;
  a.resbits = m->resbits;
  a.last_seen = m->last_seen;
  a.S = m->S;
  a.counts = m->counts;
  a.active = m->active;
  a.active_slot = m->active_slot;
  a.din_n = m->din_n;
  a.din_s = m->din_s;
  a.dout_n = m->dout_n;
  a.totals = m->totals;
  a.err = m->err;
  cudaStream_t st = m->main;
  NP_TRY(launch(m, NP_KIND_SET, st, (int64_t)n_layers * m->W * 4 * 2 * m->B, [&] { return launch_set(a, st); }));
  CUDA_TRY(cudaEventRecord(m->ev_set, st));
  return NP_OK;
}

MoveLaunch move_args(const np_model* m, int s) {
  MoveLaunch a{};
  a.store_layer = m->store_dev + (size_t)s * m->F * m->rec_bytes;
  a.rec_vec = (int)(m->rec_bytes / 16);
  a.row_vec = (int)(m->row_bytes / 16);
  a.n_proj = m->nproj;
  a.F = m->F;
  a.K = m->K;
  a.din_n = m->din_n + (size_t)s * m->K;
  a.din_s = m->din_s + (size_t)s * m->K;
  a.count = m->counts + (size_t)s * 4 + 1;
  a.staging = m->staging;
  a.bufs_layer = const_cast<unsigned char*>(layer_bufs(m, s));
  a.err = m->err;
  return a;
}

// Enqueue the reads and scatters of sparse layer s on the side stream.
np_status enqueue_move(np_model* m, int s) {
  cudaStream_t st = m->side;
  MoveLaunch a = move_args(m, s);
  if (m->d.h2d_mode == NP_H2D_FUSED) {
    a.chunk_begin = 0;
    a.chunk_cap = m->K;
    a.grid = m->gather_grid;
    NP_TRY(launch(m, NP_KIND_GATHER, st, 0, [&] { return launch_fused(a, st); }));
  } else {
    for (int c = 0; c * m->staging_rows < m->K; ++c) {
      a.chunk_begin = c * m->staging_rows;
      a.chunk_cap = m->staging_rows;
      a.grid = m->gather_grid;
      NP_TRY(launch(m, NP_KIND_GATHER, st, 0, [&] { return launch_gather(a, st); }));
      a.grid = m->scatter_grid;
      NP_TRY(launch(m, NP_KIND_SCATTER, st, 0, [&] { return launch_scatter(a, st); }));
    }
  }
  CUDA_TRY(cudaEventRecord(m->ev_layer[s], st));
  return NP_OK;
}

// Restore the slots written for sparse layer s by the pending delta.
np_status enqueue_restore(np_model* m, int s) {
  cudaStream_t st = m->side;
  MoveLaunch a = move_args(m, s);
  const int cb = (int)((m->cur_bits >> s) & 1ull);
  a.content_old = m->content + ((size_t)cb * m->S + s) * m->K;
  a.chunk_begin = 0;
  a.chunk_cap = m->K;
  a.grid = m->gather_grid;
  return launch(m, NP_KIND_GATHER, st, 0, [&] { return launch_restore(a, st); });
}

// Reads for the pending layers in `layers` (ascending), with the read hook.
// On a hook failure the already-enqueued layers are restored and the pending
// delta of every layer in `layers` is dropped.
np_status move_layers(np_model* m, const std::vector<int>& layers) {
  CUDA_TRY(cudaStreamWaitEvent(m->side, m->ev_set, 0));
  for (size_t k = 0; k < layers.size(); ++k) {
    const int s = layers[k];
    if (m->d.read_hook && m->d.read_hook(m->d.read_ctx, m->dn + s, (int32_t)m->token) != 0) {
      for (size_t q = 0; q < k; ++q) NP_TRY(enqueue_restore(m, layers[q]));
      for (int s2 : layers) m->pending_bits &= ~(1ull << s2);
      CUDA_TRY(cudaEventRecord(m->ev_side_done, m->side));
      CUDA_TRY(cudaStreamWaitEvent(m->main, m->ev_side_done, 0));
      g_last_err = "storage read hook failed";
      return NP_ERR_IO;
    }
    NP_TRY(enqueue_move(m, s));
  }
  return NP_OK;
}

void commit(np_model* m, uint64_t bits) {
  m->cur_bits ^= bits;
  m->pending_bits &= ~bits;
  m->committed_since_token |= bits;
  if ((m->committed_since_token & all_layers(m)) == all_layers(m)) {
    m->committed_since_token = 0;
    m->token += 1;
  }
}

np_status read_device_error(np_model* m) {
  int e = 0;
  CUDA_TRY(cudaMemcpy(&e, m->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (e != 0) {
    CUDA_TRY(cudaMemset(m->err, 0, sizeof(int)));
    g_last_err = e == kDevErrTimeout ? "device wait timed out" : "device bounds check failed";
    return e == kDevErrTimeout ? NP_ERR_TIMEOUT : NP_ERR_STATE;
  }
  return NP_OK;
}

np_status sync_model(np_model* m) {
  CUDA_TRY(cudaStreamSynchronize(m->side));
  CUDA_TRY(cudaStreamSynchronize(m->main));
  return NP_OK;
}

int pick_rps(size_t row_bytes) {
  int r = 1;
  while (r < 8 && (size_t)(r * 2) * row_bytes <= 24576) r *= 2;
  return r;
}

int pick_stages(size_t stage_bytes, size_t fixed, size_t limit) {
  int ns = 8;
  while (ns > 2 && fixed + ns * stage_bytes > limit) --ns;
  return fixed + ns * stage_bytes <= limit ? ns : 0;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

const char* np_status_str(np_status s) {
  switch (s) {
    case NP_OK: return "ok";
    case NP_ERR_ARG: return "invalid argument";
    case NP_ERR_OOM: return "out of device memory";
    case NP_ERR_CUDA: return "CUDA error";
    case NP_ERR_IO: return "storage read failed";
    case NP_ERR_TIMEOUT: return "device wait timed out";
    case NP_ERR_STATE: return "call out of order or corrupt state";
    default: return "unknown status";
  }
}

const char* np_last_error(void) { return g_last_err.c_str(); }

np_status np_host_register(void* ptr, size_t bytes) {
  if (!ptr || bytes == 0) return arg_fail("np_host_register: null pointer or zero size");
  CUDA_TRY(cudaHostRegister(ptr, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable));
  return NP_OK;
}

np_status np_host_unregister(void* ptr) {
  if (!ptr) return arg_fail("np_host_unregister: null pointer");
  CUDA_TRY(cudaHostUnregister(ptr));
  return NP_OK;
}

static np_status validate(const np_model_desc* d) {
  if (!d) return arg_fail("desc is null");
  if (d->n_layers < 1 || d->n_dense < 0 || d->n_dense > d->n_layers) return arg_fail("bad n_layers / n_dense");
  if (d->n_layers - d->n_dense > 64) return arg_fail("at most 64 sparse layers");
  if (d->dtype < NP_F32 || d->dtype > NP_BF16) return arg_fail("bad dtype");
  const int esz = d->dtype == NP_F32 ? 4 : 2;
  if (d->d_model < 8 || d->d_model > 8192 || (d->d_model * esz) % 16 != 0)
    return arg_fail("d_model must be in [8, 8192] with rows a multiple of 16 bytes");
  if (d->d_model / (16 / esz) > kThreads * kMaxChunksPerThread) return arg_fail("d_model too large for dtype");
  if (d->d_ff < 1 || d->d_ff > 16384) return arg_fail("d_ff must be in [1, 16384]");
  if (d->k_max < 1 || d->k_max > d->d_ff || d->k_max > 8192) return arg_fail("k_max must be in [1, min(d_ff, 8192)]");
  if (d->has_gate != 0 && d->has_gate != 1) return arg_fail("has_gate must be 0 or 1");
  if (d->combine != NP_COMBINE_INTERSECT && d->combine != NP_COMBINE_UNION) return arg_fail("bad combine");
  if (d->residency != NP_RES_SLOTMAP && d->residency != NP_RES_WINDOW) return arg_fail("bad residency");
  if (d->residency == NP_RES_WINDOW && (d->window < 1 || d->window > 32)) return arg_fail("window must be 1..32");
  if (d->batch != 1) return arg_fail("batch must be 1");
  if (d->staging_rows < 0 || d->staging_rows > d->k_max) return arg_fail("staging_rows must be in [0, k_max]");
  if (d->h2d_mode != NP_H2D_STAGED && d->h2d_mode != NP_H2D_FUSED) return arg_fail("bad h2d_mode");
  if (d->pred_hidden < 1 || (d->pred_hidden * esz) % 16 != 0 ||
      d->pred_hidden / (16 / esz) > kThreads * kMaxChunksPerThread)
    return arg_fail("pred_hidden must be positive, rows a multiple of 16 bytes, <= 8192");
  if (d->n_dense > 0 && !d->dense_w) return arg_fail("dense_w is null");
  if (d->n_layers > d->n_dense && !d->host_store) return arg_fail("host_store is null");
  if (!d->pred_w1 || !d->pred_w2) return arg_fail("predictor weights are null");
  if (d->pred_kind == NP_PRED_SHARED_ARGMAX) {
    if (d->n_dense < 1) return arg_fail("the shared predictor runs after dense layer 0: n_dense >= 1");
    if (d->n_centroids < 1 || !d->centroids) return arg_fail("centroids missing");
  } else if (d->pred_kind == NP_PRED_PERLAYER_SIGMOID) {
    if (!d->pred_b2) return arg_fail("pred_b2 is null");
  } else {
    return arg_fail("bad pred_kind");
  }
  return NP_OK;
}

np_status np_init_model(const np_model_desc* desc, np_model** out) {
  if (!out) return arg_fail("out is null");
  NP_TRY(validate(desc));
  np_model* m = new (std::nothrow) np_model();
  if (!m) return NP_ERR_OOM;
  m->d = *desc;
  np_status st = NP_OK;
  auto fail = [&](np_status s) {
    np_free_model(m);
    return s;
  };
  m->L = desc->n_layers;
  m->dn = desc->n_dense;
  m->S = m->L - m->dn;
  m->D = desc->d_model;
  m->F = desc->d_ff;
  m->K = desc->k_max;
  m->C = desc->n_centroids;
  m->W = (m->F + 31) / 32;
  m->B = desc->batch;
  m->H = desc->pred_hidden;
  m->NH = desc->pred_kind == NP_PRED_SHARED_ARGMAX ? 2 * (m->L - 1) : 0;
  m->nproj = desc->has_gate ? 3 : 2;
  m->esz = desc->dtype == NP_F32 ? 4 : 2;
  m->staging_rows = desc->staging_rows > 0 ? desc->staging_rows : m->K;
  m->window = desc->residency == NP_RES_WINDOW ? desc->window : 1;
  m->row_bytes = (size_t)m->D * m->esz;
  m->rec_bytes = m->nproj * m->row_bytes;
  m->main = static_cast<cudaStream_t>(desc->main_stream);
  m->side = static_cast<cudaStream_t>(desc->side_stream);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaGetDevice"));
  int optin = 0;
  cudaDeviceGetAttribute(&m->sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  m->smem_optin = (size_t)optin;

  // device-visible address of the host store
  if (m->S > 0) {
    cudaPointerAttributes pa{};
    e = cudaPointerGetAttributes(&pa, desc->host_store);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaPointerGetAttributes(host_store)"));
    if (pa.type == cudaMemoryTypeHost && pa.devicePointer) {
      m->store_dev = static_cast<const unsigned char*>(pa.devicePointer);
    } else if (pa.type == cudaMemoryTypeUnregistered) {
      int pageable = 0;
      cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
      if (!pageable) return fail(arg_fail("host_store is not registered and the device cannot read pageable memory"));
      m->store_dev = static_cast<const unsigned char*>(desc->host_store);
    } else {
      return fail(arg_fail("host_store must be CPU memory"));
    }
    if (reinterpret_cast<uintptr_t>(m->store_dev) % 16 != 0) return fail(arg_fail("host_store not 16-byte aligned"));
  }

  // launch shapes: two streaming CTAs per SM
  const size_t per_cta = m->smem_optin > 2048 ? (m->smem_optin / 2) - 1024 : m->smem_optin;
  m->ffn_stages = ffn_pick_stages(m->D, m->esz, m->nproj, per_cta);
  m->ffn_stages_dense = m->ffn_stages;
  if (m->ffn_stages < 2) return fail(arg_fail("d_model too large for the shared-memory ring"));
  m->ffn_grid = 2 * m->sms;
  m->gather_grid = 2 * m->sms;
  m->scatter_grid = 4 * m->sms;
  m->pred_grid = 2 * m->sms;
  m->rps1 = pick_rps(m->row_bytes);
  m->rps2 = pick_rps((size_t)m->H * m->esz);
  m->ns1 = pick_stages(m->rps1 * m->row_bytes, rowdot_smem_bytes(m->D, m->esz, m->rps1, 0), per_cta);
  m->ns2 = pick_stages(m->rps2 * (size_t)m->H * m->esz, rowdot_smem_bytes(m->H, m->esz, m->rps2, 0), per_cta);
  if (m->ns1 < 2 || m->ns2 < 2) return fail(arg_fail("predictor rows too large for the shared-memory ring"));

  // allocations
  const size_t S = (size_t)m->S, F = m->F, K = m->K;
  const size_t Sa = S > 0 ? S : 1;
  if ((st = dev_alloc(m, reinterpret_cast<unsigned char**>(&m->bufs), Sa * m->nproj * K * m->row_bytes)) != NP_OK)
    return fail(st);
  if ((st = dev_alloc(m, reinterpret_cast<unsigned char**>(&m->staging), (size_t)m->staging_rows * m->rec_bytes)) !=
      NP_OK)
    return fail(st);
  if ((st = dev_alloc(m, &m->slotmap, 2 * Sa * F, 0xff)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->inv, 2 * Sa * K, 0xff)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->content, 2 * Sa * K, 0xff)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->resbits, 2 * Sa * m->W)) != NP_OK) return fail(st);
  if (m->window > 1 && (st = dev_alloc(m, &m->last_seen, 2 * Sa * F)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->counts, Sa * 4)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->active, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->active_slot, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->din_n, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->din_s, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->dout_n, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->totals, 8)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->err, 4)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->z, (size_t)m->B * m->H)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->keys, (size_t)m->B * (m->NH > 0 ? m->NH : 1))) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->ids, (size_t)m->B * (m->NH > 0 ? m->NH : 1))) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->fire, (size_t)m->W)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->logits, F)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->part, (size_t)m->ffn_grid * m->B * m->D)) != NP_OK) return fail(st);

  e = cudaEventCreateWithFlags(&m->ev_set, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  e = cudaEventCreateWithFlags(&m->ev_side_done, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  m->ev_layer.assign(Sa, nullptr);
  for (size_t s = 0; s < S; ++s) {
    e = cudaEventCreateWithFlags(&m->ev_layer[s], cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaDeviceSynchronize"));
  *out = m;
  return NP_OK;
}

np_status np_free_model(np_model* m) {
  if (!m) return NP_OK;
  if (m->main) cudaStreamSynchronize(m->main);
  if (m->side) cudaStreamSynchronize(m->side);
  cudaDeviceSynchronize();
  for (void* p : m->allocs) cudaFree(p);
  if (m->ev_set) cudaEventDestroy(m->ev_set);
  if (m->ev_side_done) cudaEventDestroy(m->ev_side_done);
  for (cudaEvent_t ev : m->ev_layer)
    if (ev) cudaEventDestroy(ev);
  for (auto& v : m->prof_pending)
    for (auto& p : v) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
  for (auto& p : m->prof_free) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  delete m;
  return NP_OK;
}

np_status np_reset_sequence(np_model* m) {
  if (!m) return arg_fail("model is null");
  m->pending_bits = 0;
  m->committed_since_token = 0;
  m->token = 0;
  if (m->S == 0) return NP_OK;
  cudaStream_t st = m->main;
  CUDA_TRY(cudaStreamWaitEvent(st, m->ev_set, 0));
  CUDA_TRY(cudaEventRecord(m->ev_side_done, m->side));
  CUDA_TRY(cudaStreamWaitEvent(st, m->ev_side_done, 0));
  return launch(m, NP_KIND_SET, st, 0, [&] {
    return launch_reset_state(m->slotmap, m->inv, m->resbits, m->last_seen, m->S, m->F, m->K, m->W, st);
  });
}

np_status np_predict(np_model* m, int32_t layer, const float* h_dev, void* out_dev) {
  if (!m || !h_dev || !out_dev) return arg_fail("null argument");
  if (m->d.pred_kind == NP_PRED_SHARED_ARGMAX) {
    if (layer != 0) return arg_fail("the shared predictor takes layer 0");
    NP_TRY(enqueue_predict(m, 0, h_dev));
    CUDA_TRY(cudaMemcpyAsync(out_dev, m->ids, sizeof(int) * m->B * m->NH, cudaMemcpyDeviceToDevice, m->main));
    return NP_OK;
  }
  if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
  NP_TRY(enqueue_predict(m, layer, h_dev));
  CUDA_TRY(cudaMemcpyAsync(out_dev, m->fire, sizeof(uint32_t) * m->W, cudaMemcpyDeviceToDevice, m->main));
  return NP_OK;
}

static void fill_view(const np_model* m, np_delta_view* v) {
  v->n_sparse = m->S;
  v->k_max = m->K;
  v->counts = m->counts;
  v->active = m->active;
  v->active_slot = m->active_slot;
  v->din_neuron = m->din_n;
  v->din_slot = m->din_s;
  v->dout_neuron = m->dout_n;
  v->ids = m->d.pred_kind == NP_PRED_SHARED_ARGMAX ? m->ids : nullptr;
}

np_status np_last_delta(np_model* m, np_delta_view* out) {
  if (!m || !out) return arg_fail("null argument");
  fill_view(m, out);
  return NP_OK;
}

np_status np_delta(np_model* m, int32_t layer, const void* pred_dev, np_delta_view* out) {
  if (!m || !pred_dev) return arg_fail("null argument");
  if (m->S == 0) return arg_fail("model has no sparse layers");
  const bool shared = m->d.pred_kind == NP_PRED_SHARED_ARGMAX;
  if (layer == -1) {
    if (!shared) return arg_fail("layer -1 needs the shared predictor");
    if (m->pending_bits) {
      g_last_err = "a delta is already pending";
      return NP_ERR_STATE;
    }
    NP_TRY(enqueue_set(m, 0, m->S, static_cast<const int*>(pred_dev), nullptr));
    m->pending_bits = all_layers(m);
  } else {
    if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
    const int s = layer - m->dn;
    if (m->pending_bits & (1ull << s)) {
      g_last_err = "a delta is already pending for this layer";
      return NP_ERR_STATE;
    }
    if (shared) NP_TRY(enqueue_set(m, s, 1, static_cast<const int*>(pred_dev), nullptr));
    else NP_TRY(enqueue_set(m, s, 1, nullptr, static_cast<const uint32_t*>(pred_dev)));
    m->pending_bits |= 1ull << s;
  }
  if (out) fill_view(m, out);
  return NP_OK;
}

np_status np_scatter(np_model* m, int32_t layer) {
  if (!m) return arg_fail("model is null");
  std::vector<int> layers;
  if (layer == -1) {
    for (int s = 0; s < m->S; ++s)
      if (m->pending_bits & (1ull << s)) layers.push_back(s);
  } else {
    if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
    const int s = layer - m->dn;
    if (m->pending_bits & (1ull << s)) layers.push_back(s);
  }
  if (layers.empty()) {
    g_last_err = "no pending delta";
    return NP_ERR_STATE;
  }
  NP_TRY(move_layers(m, layers));
  CUDA_TRY(cudaEventRecord(m->ev_side_done, m->side));
  CUDA_TRY(cudaStreamWaitEvent(m->main, m->ev_side_done, 0));
  uint64_t bits = 0;
  for (int s : layers) bits |= 1ull << s;
  commit(m, bits);
  return NP_OK;
}

np_status np_sparse_mlp(np_model* m, int32_t layer, const float* h_dev, float* y_dev) {
  if (!m || !h_dev || !y_dev) return arg_fail("null argument");
  if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
  if (h_dev == y_dev) return arg_fail("y_dev may not alias h_dev");
  return enqueue_sparse(m, layer - m->dn, h_dev, nullptr, y_dev);
}

np_status np_dense_mlp(np_model* m, int32_t layer, const float* h_dev, float* y_dev) {
  if (!m || !h_dev || !y_dev) return arg_fail("null argument");
  if (layer < 0 || layer >= m->dn) return arg_fail("layer is not a dense layer");
  if (h_dev == y_dev) return arg_fail("y_dev may not alias h_dev");
  return enqueue_dense(m, layer, h_dev, nullptr, y_dev);
}

np_status np_decode_token(np_model* m, float* h_dev, np_stats* stats_host) {
  if (!m || !h_dev) return arg_fail("null argument");
  if (m->pending_bits) {
    g_last_err = "a delta is pending; call np_scatter first";
    return NP_ERR_STATE;
  }
  const int64_t token = m->token;
  const bool shared = m->d.pred_kind == NP_PRED_SHARED_ARGMAX;
  for (int l = 0; l < m->dn; ++l) {
    NP_TRY(enqueue_dense(m, l, h_dev, h_dev, nullptr));
    if (l == 0 && shared && m->S > 0) {
      NP_TRY(enqueue_predict(m, 0, h_dev));
      NP_TRY(enqueue_set(m, 0, m->S, m->ids, nullptr));
      m->pending_bits = all_layers(m);
      std::vector<int> layers(m->S);
      for (int s = 0; s < m->S; ++s) layers[s] = s;
      NP_TRY(move_layers(m, layers));
    }
  }
  for (int s = 0; s < m->S; ++s) {
    if (!shared) {
      NP_TRY(enqueue_predict(m, m->dn + s, h_dev));
      NP_TRY(enqueue_set(m, s, 1, nullptr, m->fire));
      m->pending_bits |= 1ull << s;
      const np_status rs = move_layers(m, std::vector<int>{s});
      if (rs != NP_OK) {
        // earlier layers of this token already hold their new rows: put the
        // committed contents back and drop the whole token's delta
        for (int q = 0; q < s; ++q) NP_TRY(enqueue_restore(m, q));
        m->pending_bits = 0;
        CUDA_TRY(cudaEventRecord(m->ev_side_done, m->side));
        CUDA_TRY(cudaStreamWaitEvent(m->main, m->ev_side_done, 0));
        return rs;
      }
    }
    CUDA_TRY(cudaStreamWaitEvent(m->main, m->ev_layer[s], 0));
    NP_TRY(enqueue_sparse(m, s, h_dev, h_dev, nullptr));
  }
  if (m->S > 0) {
    m->committed_since_token = 0;
    m->cur_bits ^= all_layers(m);
    m->pending_bits = 0;
    m->token += 1;
  }
  if (stats_host) {
    std::memset(stats_host, 0, sizeof(*stats_host));
    stats_host->token = token;
    NP_TRY(sync_model(m));
    NP_TRY(read_device_error(m));
    if (m->S > 0) {
      std::vector<int> c((size_t)m->S * 4);
      CUDA_TRY(cudaMemcpy(c.data(), m->counts, c.size() * sizeof(int), cudaMemcpyDeviceToHost));
      for (int s = 0; s < m->S; ++s) {
        stats_host->active_rows += c[s * 4 + 0];
        stats_host->din_rows += c[s * 4 + 1];
        stats_host->dout_rows += c[s * 4 + 2];
        stats_host->dropped_rows += c[s * 4 + 3];
      }
      stats_host->h2d_bytes = stats_host->din_rows * (int64_t)m->rec_bytes;
    }
  }
  return NP_OK;
}

np_status np_get_state(np_model* m, int32_t layer, int32_t* slotmap_host, int32_t* inv_host) {
  if (!m) return arg_fail("model is null");
  if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
  const int s = layer - m->dn;
  NP_TRY(sync_model(m));
  const int cb = (int)((m->cur_bits >> s) & 1ull);
  if (slotmap_host)
    CUDA_TRY(cudaMemcpy(slotmap_host, m->slotmap + ((size_t)cb * m->S + s) * m->F, sizeof(int) * m->F,
                        cudaMemcpyDeviceToHost));
  if (inv_host)
    CUDA_TRY(cudaMemcpy(inv_host, m->inv + ((size_t)cb * m->S + s) * m->K, sizeof(int) * m->K,
                        cudaMemcpyDeviceToHost));
  return read_device_error(m);
}

np_status np_resident_rows(np_model* m, int32_t layer, int32_t proj, const void** dev_ptr) {
  if (!m || !dev_ptr) return arg_fail("null argument");
  if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
  if (proj < 0 || proj >= m->nproj) return arg_fail("bad projection");
  *dev_ptr = layer_bufs(m, layer - m->dn) + (size_t)proj * m->K * m->row_bytes;
  return NP_OK;
}

np_status np_get_counts(np_model* m, int32_t* counts_host) {
  if (!m || !counts_host) return arg_fail("null argument");
  NP_TRY(sync_model(m));
  if (m->S > 0)
    CUDA_TRY(cudaMemcpy(counts_host, m->counts, sizeof(int) * 4 * m->S, cudaMemcpyDeviceToHost));
  return NP_OK;
}

np_status np_check_error(np_model* m) {
  if (!m) return arg_fail("model is null");
  NP_TRY(sync_model(m));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "asynchronous error");
  return read_device_error(m);
}

np_status np_set_profiling(np_model* m, int32_t enable) {
  if (!m) return arg_fail("model is null");
  m->prof = enable != 0;
  return NP_OK;
}

np_status np_get_profile(np_model* m, double* ms_out, int64_t* launches_out, int64_t* bytes_out) {
  if (!m) return arg_fail("model is null");
  NP_TRY(sync_model(m));
  for (int k = 0; k < NP_N_KINDS; ++k) NP_TRY(prof_fold(m, k, 0));
  unsigned long long tot[8] = {};
  CUDA_TRY(cudaMemcpy(tot, m->totals, sizeof(tot), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(m->totals, 0, sizeof(tot)));
  int64_t bytes[NP_N_KINDS];
  for (int k = 0; k < NP_N_KINDS; ++k) bytes[k] = m->prof_fixed_bytes[k];
  const int64_t din = (int64_t)tot[1], act = (int64_t)tot[0];
  bytes[NP_KIND_FFN] += act * (int64_t)m->rec_bytes;
  if (m->d.h2d_mode == NP_H2D_FUSED) {
    bytes[NP_KIND_GATHER] += din * (int64_t)m->rec_bytes;
  } else {
    bytes[NP_KIND_GATHER] += din * (int64_t)m->rec_bytes;
    bytes[NP_KIND_SCATTER] += 2 * din * (int64_t)m->rec_bytes;
  }
  for (int k = 0; k < NP_N_KINDS; ++k) {
    if (ms_out) ms_out[k] = m->prof_ms[k];
    if (launches_out) launches_out[k] = m->prof_launches[k];
    if (bytes_out) bytes_out[k] = bytes[k];
    m->prof_ms[k] = 0;
    m->prof_launches[k] = 0;
    m->prof_fixed_bytes[k] = 0;
  }
  return NP_OK;
}

int64_t np_launch_count(np_model* m) { return m ? m->launches : 0; }

}  // extern "C"
