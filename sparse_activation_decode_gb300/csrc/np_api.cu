// Host runtime behind the C ABI in include/np.h.
//
// Owns the per-model device state and orders the kernels of one decode step
// on two streams (NeuroPrefetcher full text, Figure 2 execution flow):
//
//   main: dense layer 0 -> predictor -> set/delta kernel -> [event set]
//         -> dense layers 1..d-1 -> for each sparse layer: wait for that
//         layer's rows, FFN, residual update
//   gather streams G0 (the caller's side stream) and G1, alternating by
//         layer: wait [event set] -> gather the layer's incoming records over
//         the host link into staging buffer s%2 -> [event gathered s]
//   scatter stream X: wait [gathered s] -> deinterleave-scatter staging into
//         the layer's buffers -> [event ready s]
//   (chunked by the staging capacity; two layers' gathers can be in flight
//   at once, so the host link does not idle while a layer is scattered)
//
// Decode state (slot maps, inverse maps, slot contents, resident bitmasks,
// window history) is updated in place by the set kernel, which records every
// value it overwrites in the delta lists.  If the incoming rows cannot be
// read, a rollback kernel restores the previous state from those lists and
// the rows already overwritten are copied back from the store.
#include <algorithm>
#include <cuda_runtime.h>

#include <climits>
#include <cstdio>
#include <cstdlib>
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

void np::set_last_error(const char* what) { g_last_err = what; }

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
  int frequency = 0;  // frequency-weighted residency: last_seen holds activation counts
  int lookahead = 0;  // per-layer predictor of layer l reads the input of layer max(l - k, 0)
  int sms = 0;
  size_t smem_optin = 0;
  size_t row_bytes = 0, rec_bytes = 0;
  cudaStream_t main = nullptr, side = nullptr;  // side = gather stream G0
  cudaStream_t g1 = nullptr, xs = nullptr;        // gather stream G1, scatter stream X
  cudaStream_t fs = nullptr;                      // sparse-FFN stream
  const unsigned char* store_dev = nullptr;
  // device allocations
  void* bufs = nullptr;
  void* staging = nullptr;  // two buffers of staging_rows records
  int *slotmap = nullptr, *inv = nullptr, *content = nullptr, *last_seen = nullptr;
  uint32_t* resbits = nullptr;
  int *counts = nullptr, *active = nullptr, *active_slot = nullptr, *din_n = nullptr, *din_s = nullptr,
      *din_oldct = nullptr, *dout_n = nullptr, *dout_s = nullptr, *ls_old = nullptr;
  unsigned long long* totals = nullptr;
  int* err = nullptr;
  float* z = nullptr;
  unsigned long long* keys = nullptr;
  int* ids = nullptr;
  uint32_t* fire = nullptr;
  float* logits = nullptr;
  // batched (B > 1) tensor-core path: tensor maps over the weight blocks,
  // launch plans, residual bases [2][B][D], y accumulators [3][B][D], the
  // predictor hidden layer as hi/lo 16-bit operands [16][H]
  bool tc = false;
  RowMaps map_bufs{}, map_dense{}, map_w1{}, map_w2{};
  int* slot_hw = nullptr;  // [S] one past the highest occupied slot (|R| when compact)
  // compact placement (rows in [0, |R|)): row moves of the last delta
  bool compact = false;
  int *mv_src = nullptr, *mv_dst = nullptr, *mv_oldct = nullptr, *mv_count = nullptr;
  MmaPlan plan_ffn{}, plan_hid{}, plan_heads{};
  uint16_t* zhl = nullptr;
  // residual chaining (every batch size): bases [2][B][D], accumulators [3][B][D]
  float* hbase = nullptr;
  float* yacc = nullptr;
  std::vector<void*> allocs;
  // launch shapes
  int ffn_grid = 0, ffn_stages = 0;
  int ffn_stages_dense = 0;              // ring of the dense layers' FFN launches
  int chain_grid = 0, chain_stages = 0;  // persistent FFN chain (batch 1)
  int pdl_mask = 5;                      // programmatic dependent launch: 1 predictor, 2 set kernel, 4 tensor-core kernels
  // streams whose last operation is a kernel launched by the current API
  // call (only the next kernel on such a stream may use programmatic
  // dependent launch, see join())
  cudaStream_t ours[8] = {};
  int n_ours = 0;
  unsigned* arrive = nullptr;            // [2L] arrival counters of the chain
  unsigned* gdone = nullptr;             // [L] per-layer read counters of the per-token pipeline
  bool token_chain = false;              // one persistent launch reads and runs every layer after layer 0
  int withhold_layer = -1;               // failure test hook, see NP_TEST_WITHHOLD_ARRIVAL
  float* chain_part = nullptr;           // [chain_grid][D] partial y of the chain
  int gather_grid = 0, scatter_grid = 0, pred_grid = 0;
  int rps1 = 1, rps2 = 1, ns1 = 2, ns2 = 2;
  int ns1_side = 2, ns2_side = 2;  // predictor rings beside an FFN (lookahead stream)
  // state
  uint64_t pending_bits = 0, committed_since_token = 0;
  int64_t token = 0;
  int64_t launches = 0;
  cudaEvent_t ev_set = nullptr, ev_side_done = nullptr, ev_j[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  cudaEvent_t ev_pre = nullptr, ev_ffn = nullptr;
  std::vector<cudaEvent_t> ev_g, ev_layer;  // per sparse layer: gathered, ready
  // profiling
  bool prof = false;
  bool prof_markers = false;  // an empty kernel before each start event
  // token counter on the device (the set kernel's window ages), and the
  // captured token: replayed with the caller's h staged through h_io
  int* token_dev = nullptr;
  float* h_io = nullptr;
  cudaGraphExec_t graph = nullptr;
  cudaStream_t gs = nullptr;    // capture and replay stream (the caller's main stream may be the legacy one)
  cudaEvent_t ev_gin = nullptr, ev_gout = nullptr;
  // per-layer predictor with a lookahead: predictor and set kernels on their
  // own stream beside the FFNs (ev_pin: a source layer's input is final;
  // ev_psrc: the predictions reading it are done)
  cudaStream_t ps = nullptr;
  cudaEvent_t ev_pin = nullptr, ev_psrc = nullptr;
  // and the set kernels on a stream of their own (ss), so that layer j's set
  // kernel runs beside layer j+1's predictor: two firing-mask buffers
  // alternate by layer; ev_pdone[b]: the predictor that wrote buffer b is
  // done; ev_sdone[b]: the set kernel that read it is done
  bool set_stream = true;
  cudaStream_t ss = nullptr;
  cudaEvent_t ev_pdone[2] = {nullptr, nullptr}, ev_sdone[2] = {nullptr, nullptr};
  uint32_t* fire2 = nullptr;
  bool graph_off = false;       // disabled, or the capture failed
  // token capture: the per-layer FFN kernel nodes in issue order, and the
  // edges between consecutive ones made programmatic (relax_ffn_edges)
  struct CapNode {
    cudaStream_t st;
    cudaGraphNode_t node;
  };
  bool capturing = false;
  bool graph_pdl = true;
  std::vector<CapNode> cap_ffn;
  std::vector<std::pair<cudaGraphNode_t, cudaGraphNode_t>> relaxed;  // valid until the graph is destroyed
  size_t graph_pdl_edges = 0;   // programmatic FFN edges in the instantiated token
  int64_t graph_launches = 0;   // kernels in one replay
  int64_t eager_tokens = 0;     // tokens issued launch by launch (the first one sets kernel attributes)
  std::vector<EventPair> prof_free;
  double prof_ms[NP_N_KINDS] = {};
  int64_t prof_launches[NP_N_KINDS] = {};
  int64_t prof_fixed_bytes[NP_N_KINDS] = {};
  // timeline of timed launches in issue order: (kind, events)
  std::vector<std::pair<int, EventPair>> trace;
};

namespace {

// An integer tuning switch from the environment: its value when set to a
// decimal integer (0 included), else `dflt`.
int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  const long x = std::strtol(v, &end, 10);
  if (end == v || *end != '\0' || x < INT_MIN || x > INT_MAX) return dflt;
  return (int)x;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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

// An empty one-warp kernel (profiling: orders a timing event after the
// stream's pending waits).
__global__ void marker_kernel() {}

cudaError_t launch_marker(cudaStream_t st) {
  marker_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError();
}

// The device token counter advances once a token's deltas are all committed.
__global__ void bump_kernel(int* counter) {
  if (threadIdx.x == 0) *counter += 1;
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
  // A start event placed right after a wait on another stream's event is
  // stamped before that wait is satisfied; an empty kernel in front of it
  // makes the stamp follow everything the launch depends on.
  if (m->prof_markers) CUDA_TRY(launch_marker(st));
  CUDA_TRY(cudaEventRecord(ep->a, st));
  return NP_OK;
}

// Accumulate the durations of the oldest `n` traced launches and recycle
// their events.
np_status prof_fold(np_model* m, size_t n) {
  if (n > m->trace.size()) n = m->trace.size();
  for (size_t i = 0; i < n; ++i) {
    const auto& t = m->trace[i];
    CUDA_TRY(cudaEventSynchronize(t.second.b));
    float ms = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&ms, t.second.a, t.second.b));
    m->prof_ms[t.first] += ms;
    m->prof_free.push_back(t.second);
  }
  m->trace.erase(m->trace.begin(), m->trace.begin() + n);
  return NP_OK;
}

np_status prof_end(np_model* m, int kind, cudaStream_t st, const EventPair& ep) {
  CUDA_TRY(cudaEventRecord(ep.b, st));
  m->trace.push_back({kind, ep});
  m->prof_launches[kind] += 1;
  if (m->trace.size() > 16384) NP_TRY(prof_fold(m, 8192));
  return NP_OK;
}

bool is_ours(const np_model* m, cudaStream_t st) {
  for (int i = 0; i < m->n_ours; ++i)
    if (m->ours[i] == st) return true;
  return false;
}

// The next kernel on `st` follows something other than one of this call's
// kernels (an event wait, a copy, or the caller's own work).
void forget(np_model* m, cudaStream_t st) {
  for (int i = 0; i < m->n_ours; ++i)
    if (m->ours[i] == st) {
      m->ours[i] = m->ours[--m->n_ours];
      return;
    }
}

// Programmatic dependent launch is used only between two kernels of one
// call, back to back on one stream.  Kernels launched with it read data that
// does not depend on the previous kernel (weights, the row count) before
// their griddepcontrol.wait, which is sound only when the relaxed dependency
// is that previous kernel.  Measured on this GPU and driver: eagerly, a
// kernel after an event wait keeps full dependencies anyway; under stream
// capture, a kernel whose only dependency is one kernel node gets a
// programmatic edge even when that node comes from another stream through
// the event, so the kernel could read rows before the copy that wrote them
// is visible.  Hence every event wait, copy and API entry ends the chain.
np_status join(np_model* m, cudaStream_t st, cudaEvent_t ev) {
  CUDA_TRY(cudaStreamWaitEvent(st, ev, 0));
  forget(m, st);
  return NP_OK;
}

// Programmatic dependent launch for the next kernel on `st`: allowed by the
// mask `bit` (0: always) and the stream's last operation is one of this
// call's kernels.
int pdl_for(const np_model* m, cudaStream_t st, int bit) {
  return (bit == 0 || (m->pdl_mask & bit) != 0) && is_ours(m, st) ? 1 : 0;
}

// Start of a public call: no stream's last operation is one of its kernels.
void begin_call(np_model* m) { m->n_ours = 0; }

// Launch one kernel (a callable returning cudaError_t), optionally timed.
template <typename Fn>
np_status launch(np_model* m, int kind, cudaStream_t st, int64_t fixed_bytes, Fn fn) {
  EventPair ep{};
  if (m->prof) NP_TRY(prof_begin(m, kind, st, &ep));
  cudaError_t e = fn();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (!is_ours(m, st) && m->n_ours < 8) m->ours[m->n_ours++] = st;
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

// FFN over a row list: x = rmsnorm(hb + yprev), y added into y_acc; CTA 0
// stores hb + yprev into hb_out and clears y_zero (both optional).
np_status enqueue_ffn(np_model* m, cudaStream_t st, int kind, const unsigned char* base, size_t proj_stride,
                      const int* rows, const int* n_dev, int n_host, int list_cap, int row_limit,
                      const float* hb, const float* yprev, float* hb_out, float* y_acc, float* y_zero,
                      int64_t fixed_bytes) {
  FfnLaunch a{};
  a.h_in = hb;
  a.yprev = yprev;
  a.hb_out = hb_out;
  a.y_acc = y_acc;
  a.y_zero = y_zero;
  int p = 0;
  a.w_gate = m->d.has_gate ? base + (p++) * proj_stride : nullptr;
  a.w_up = base + (p++) * proj_stride;
  a.w_down = base + p * proj_stride;
  a.row_list = rows;
  a.n_rows_dev = n_dev;
  a.n_rows_host = n_host;
  a.list_cap = list_cap;
  a.row_limit = row_limit;
  a.D = m->D;
  a.dtype = m->d.dtype;
  a.dtype_bytes = m->esz;
  a.gated = m->d.has_gate;
  a.swiglu = m->d.activation == NP_ACT_SWIGLU;
  a.n_stages = kind == NP_KIND_DENSE ? m->ffn_stages_dense : m->ffn_stages;
  a.grid = m->ffn_grid;
  a.err = m->err;
  a.pdl = pdl_for(m, st, 0);
  return launch(m, kind, st, fixed_bytes, [&] { return launch_ffn_rows(a, st); });
}

np_status enqueue_tc_ffn(np_model* m, cudaStream_t st, int l, const float* hb, const float* yprev, float* hb_out,
                         float* y_acc, float* y_zero);

// During the token capture, remember the kernel node just added to `st`.
void note_ffn_node(np_model* m, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaGraphNode_t* deps = nullptr;
  size_t nd = 0;
  if (cudaStreamGetCaptureInfo(st, &cs, nullptr, nullptr, &deps, nullptr, &nd) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  if (cs == cudaStreamCaptureStatusActive && nd == 1) m->cap_ffn.push_back({st, deps[0]});
}

np_status enqueue_layer_ffn_kernel(np_model* m, cudaStream_t st, int l, const float* hb, const float* yprev,
                                   float* hb_out, float* y_acc, float* y_zero);

// One layer's FFN kernel; under the token capture its node is recorded when
// the kernel may take a programmatic edge from the previous layer's FFN.
np_status enqueue_layer_ffn(np_model* m, cudaStream_t st, int l, const float* hb, const float* yprev,
                            float* hb_out, float* y_acc, float* y_zero) {
  NP_TRY(enqueue_layer_ffn_kernel(m, st, l, hb, yprev, hb_out, y_acc, y_zero));
  if (m->capturing && (!m->tc || (m->pdl_mask & 4) != 0)) note_ffn_node(m, st);
  return NP_OK;
}

// FFN of layer l (dense or sparse) for every sequence, on the kernel that
// fits the batch: x = rmsnorm(hb + yprev), y added into y_acc.
np_status enqueue_layer_ffn_kernel(np_model* m, cudaStream_t st, int l, const float* hb, const float* yprev,
                                   float* hb_out, float* y_acc, float* y_zero) {
  if (m->tc) return enqueue_tc_ffn(m, st, l, hb, yprev, hb_out, y_acc, y_zero);
  if (l < m->dn) {
    const size_t proj_stride = (size_t)m->F * m->row_bytes;
    const unsigned char* base =
        static_cast<const unsigned char*>(m->d.dense_w) + (size_t)l * m->nproj * proj_stride;
    return enqueue_ffn(m, st, NP_KIND_DENSE, base, proj_stride, nullptr, nullptr, m->F, m->F, m->F, hb, yprev,
                       hb_out, y_acc, y_zero, (int64_t)m->nproj * m->F * m->row_bytes);
  }
  const int s = l - m->dn;
  const size_t proj_stride = (size_t)m->K * m->row_bytes;
  if (m->compact)  // the occupied region [0, |R|)
    return enqueue_ffn(m, st, NP_KIND_FFN, layer_bufs(m, s), proj_stride, nullptr, m->slot_hw + s, 0, m->K, m->K,
                       hb, yprev, hb_out, y_acc, y_zero, 0);
  return enqueue_ffn(m, st, NP_KIND_FFN, layer_bufs(m, s), proj_stride, m->active_slot + (size_t)s * m->K,
                     m->counts + (size_t)s * 4, 0, m->K, m->K, hb, yprev, hb_out, y_acc, y_zero, 0);
}

// Residual chaining across layers: layer l reads base(l) + y(l-1), adds its
// y into y(l) and stores its input h_l as base(l+1); y(l+1) is cleared by
// layer l.  Two bases and three accumulators rotate.
float* chain_base(np_model* m, int i) { return m->hbase + (size_t)(i & 1) * m->B * m->D; }
float* chain_y(np_model* m, int i) { return m->yacc + (size_t)(i % 3) * m->B * m->D; }

// ---- batched path (tensor cores) -------------------------------------------

np_status enqueue_mma(np_model* m, cudaStream_t st, int kind, int mode, const RowMaps& map, const MmaPlan& p,
                      MmaArgs& a, int64_t fixed_bytes) {
  a.B = m->B;
  a.swiglu = m->d.activation == NP_ACT_SWIGLU;
  a.pdl = pdl_for(m, st, 4);
  a.err = m->err;
  const int bf16 = m->d.dtype == NP_BF16;
  return launch(m, kind, st, fixed_bytes, [&] { return launch_mma_rows(mode, bf16, map, a, p, st); });
}

// FFN of layer l for all sequences: x = rmsnorm(hb + yprev), y added into
// y_acc; hb + yprev stored into hb_out and y_zero cleared (both optional).
np_status enqueue_tc_ffn(np_model* m, cudaStream_t st, int l, const float* hb, const float* yprev, float* hb_out,
                         float* y_acc, float* y_zero) {
  MmaArgs a{};
  a.Kdim = m->D;
  a.hb = hb;
  a.yprev = yprev;
  a.hb_out = hb_out;
  a.y_acc = y_acc;
  a.y_zero = y_zero;
  const int g = m->d.has_gate ? 1 : 0;
  const int mode = g ? kMmaFfnGated : kMmaFfnUp;
  if (l < m->dn) {
    const int base = l * m->nproj * m->F;
    a.row_base0 = base;
    a.row_base1 = base + m->F;
    a.row_base2 = base + (1 + g) * m->F;
    a.n_rows_host = m->F;
    a.row_cap = m->F;
    return enqueue_mma(m, st, NP_KIND_DENSE, mode, m->map_dense, m->plan_ffn, a,
                       (int64_t)m->nproj * m->F * m->row_bytes);
  }
  const int s = l - m->dn;
  const int base = s * m->nproj * m->K;
  a.row_base0 = base;
  a.row_base1 = base + m->K;
  a.row_base2 = base + (1 + g) * m->K;
  // slot order over [0, high-water mark); free slots are skipped
  a.occ_inv = m->inv + (size_t)s * m->K;
  a.n_rows_dev = m->slot_hw + s;
  a.row_cap = m->K;
  return enqueue_mma(m, st, NP_KIND_FFN, mode, m->map_bufs, m->plan_ffn, a, 0);
}

// Predictor hidden layer for all sequences (x = rmsnorm(hb + yprev)); the
// argmax keys are cleared for the heads that follow.
np_status enqueue_tc_hidden(np_model* m, const float* hb, const float* yprev) {
  MmaArgs a{};
  a.Kdim = m->D;
  a.hb = hb;
  a.yprev = yprev;
  a.n_rows_host = m->H;
  a.row_cap = m->H;
  a.zout = m->zhl;
  a.zout_stride = m->H;
  a.keys_zero = m->keys;
  a.n_keys_zero = m->B * m->NH;
  return enqueue_mma(m, m->main, NP_KIND_PRED, kMmaHidden, m->map_w1, m->plan_hid, a,
                     (int64_t)m->H * m->D * m->esz);
}

np_status enqueue_tc_heads(np_model* m, int h0, int h1) {
  if (h1 <= h0) return NP_OK;
  MmaArgs a{};
  a.Kdim = m->H;
  a.row_base0 = h0 * m->C;
  a.n_rows_host = (h1 - h0) * m->C;
  a.row_cap = a.n_rows_host;
  a.zin = m->zhl;
  a.keys = m->keys;
  a.n_heads = m->NH;
  a.C = m->C;
  return enqueue_mma(m, m->main, NP_KIND_PRED, kMmaHeads, m->map_w2, m->plan_heads, a,
                     (int64_t)(h1 - h0) * m->C * m->H * m->esz);
}

np_status enqueue_rowdot(np_model* m, const void* W, int n_rows, int len, const float* vec, int rms, int mode,
                         const void* bias, float* out_f, unsigned long long* keys, int C, uint32_t* fire,
                         uint32_t* zero_ptr, int zero_words, int rps, int ns, const float* vec2 = nullptr) {
  RowdotLaunch a{};
  a.W = W;
  a.vec2 = vec2;
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
  a.pdl = pdl_for(m, st, 1);
  return launch(m, NP_KIND_PRED, st, (int64_t)n_rows * len * m->esz, [&] { return launch_rowdot(a, st); });
}

// Second predictor product for heads [h0, h1) only (shared predictor).
np_status enqueue_pred_heads(np_model* m, int h0, int h1) {
  if (m->tc) return enqueue_tc_heads(m, h0, h1);
  if (h1 <= h0) return NP_OK;
  const unsigned char* w2 = static_cast<const unsigned char*>(m->d.pred_w2) + (size_t)h0 * m->C * m->H * m->esz;
  return enqueue_rowdot(m, w2, (h1 - h0) * m->C, m->H, m->z, 0, 1, nullptr, nullptr, m->keys + h0, m->C, nullptr,
                        nullptr, 0, m->rps2, m->ns2);
}

// Hidden layer of the shared predictor on x = rmsnorm(h + h2) (h2 may be null).
np_status enqueue_pred_hidden(np_model* m, const float* h, const float* h2) {
  if (m->tc) return enqueue_tc_hidden(m, h, h2);
  return enqueue_rowdot(m, m->d.pred_w1, m->H, m->D, h, 1, 0, nullptr, m->z, nullptr, 0, nullptr,
                        reinterpret_cast<uint32_t*>(m->keys), 2 * m->NH, m->rps1, m->ns1, h2);
}

np_status enqueue_predict(np_model* m, int layer, const float* h, bool want_ids = true, const float* h2 = nullptr,
                          uint32_t* fire = nullptr) {
  if (!fire) fire = m->fire;
  if (m->tc) {
    NP_TRY(enqueue_tc_hidden(m, h, nullptr));
    NP_TRY(enqueue_tc_heads(m, 0, m->NH));
    if (!want_ids) return NP_OK;
    cudaStream_t st = m->main;
    return launch(m, NP_KIND_PRED, st, 0, [&] { return launch_keys_to_ids(m->keys, m->B * m->NH, m->ids, st); });
  }
  if (m->d.pred_kind == NP_PRED_SHARED_ARGMAX) {
    NP_TRY(enqueue_rowdot(m, m->d.pred_w1, m->H, m->D, h, 1, 0, nullptr, m->z, nullptr, 0, nullptr,
                          reinterpret_cast<uint32_t*>(m->keys), 2 * m->NH, m->rps1, m->ns1));
    NP_TRY(enqueue_rowdot(m, m->d.pred_w2, m->NH * m->C, m->H, m->z, 0, 1, nullptr, nullptr, m->keys, m->C,
                          nullptr, nullptr, 0, m->rps2, m->ns2));
    if (!want_ids) return NP_OK;
    cudaStream_t st = m->main;
    return launch(m, NP_KIND_PRED, st, 0, [&] { return launch_keys_to_ids(m->keys, m->NH, m->ids, st); });
  }
  const unsigned char* w1 = static_cast<const unsigned char*>(m->d.pred_w1) + (size_t)layer * m->H * m->row_bytes;
  const unsigned char* w2 =
      static_cast<const unsigned char*>(m->d.pred_w2) + (size_t)layer * m->F * m->H * m->esz;
  const unsigned char* b2 = static_cast<const unsigned char*>(m->d.pred_b2) + (size_t)layer * m->F * m->esz;
  const bool side = m->ps && m->main == m->ps;  // beside the FFN stream
  NP_TRY(enqueue_rowdot(m, w1, m->H, m->D, h, 1, 0, nullptr, m->z, nullptr, 0, nullptr, fire, m->W, m->rps1,
                        side ? m->ns1_side : m->ns1, h2));
  return enqueue_rowdot(m, w2, m->F, m->H, m->z, 0, 2, b2, m->logits, nullptr, 0, fire, nullptr, 0, m->rps2,
                        side ? m->ns2_side : m->ns2);
}

SetLaunch set_args(np_model* m, int first_sparse, int n_layers);

np_status enqueue_set(np_model* m, int first_sparse, int n_layers, const int* ids, const uint32_t* fire,
                      const unsigned long long* keys = nullptr) {
  SetLaunch a = set_args(m, first_sparse, n_layers);
  a.ids = ids;
  a.keys = keys;
  a.ids_out = keys ? m->ids : nullptr;
  a.fire = fire;
  cudaStream_t st = m->main;
  a.pdl = pdl_for(m, st, 2);
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
  a.staging = static_cast<unsigned char*>(m->staging) + (size_t)(s & 1) * m->staging_rows * m->rec_bytes;
  a.bufs_layer = const_cast<unsigned char*>(layer_bufs(m, s));
  if (m->compact) {
    a.mv_src = m->mv_src + (size_t)s * m->K;
    a.mv_dst = m->mv_dst + (size_t)s * m->K;
    a.mv_oldct = m->mv_oldct + (size_t)s * m->K;
    a.mv_count = m->mv_count + s;
  }
  a.err = m->err;
  return a;
}

cudaStream_t gather_stream(const np_model* m, int s) { return (s & 1) ? m->g1 : m->side; }

// Make `st` wait for all work queued so far on the gather and scatter streams.
np_status join_side(np_model* m, cudaStream_t st) {
  const cudaStream_t src[6] = {m->side, m->g1, m->xs, m->fs, m->ps, m->ss};
  for (int k = 0; k < 6; ++k) {
    CUDA_TRY(cudaEventRecord(m->ev_j[k], src[k]));
    NP_TRY(join(m, st, m->ev_j[k]));
  }
  return NP_OK;
}

// Enqueue the reads and scatters of sparse layer s: gathers on G[s%2] into
// staging buffer s%2, scatters on X; ev_layer[s] marks the rows in place.
np_status enqueue_move(np_model* m, int s) {
  cudaStream_t g = gather_stream(m, s), x = m->xs;
  MoveLaunch a = move_args(m, s);
  if (m->compact) {
    // kept rows fill the freed slots before incoming rows may overwrite the
    // end of the region (device to device, HBM-bound)
    a.grid = m->scatter_grid;
    NP_TRY(launch(m, NP_KIND_SCATTER, g, 0, [&] { return launch_move_rows(a, g); }));
  }
  if (m->d.h2d_mode == NP_H2D_FUSED) {
    a.chunk_begin = 0;
    a.chunk_cap = m->K;
    a.grid = m->gather_grid;
    NP_TRY(launch(m, NP_KIND_GATHER, g, 0, [&] { return launch_fused(a, g); }));
    CUDA_TRY(cudaEventRecord(m->ev_layer[s], g));
    return NP_OK;
  }
  for (int c = 0; c * m->staging_rows < m->K; ++c) {
    // staging buffer s%2 is free once the scatter that last read it is done
    if (c > 0) NP_TRY(join(m, g, m->ev_layer[s]));
    else if (s >= 2) NP_TRY(join(m, g, m->ev_layer[s - 2]));
    a.chunk_begin = c * m->staging_rows;
    a.chunk_cap = m->staging_rows;
    a.grid = m->gather_grid;
    NP_TRY(launch(m, NP_KIND_GATHER, g, 0, [&] { return launch_gather(a, g); }));
    CUDA_TRY(cudaEventRecord(m->ev_g[s], g));
    NP_TRY(join(m, x, m->ev_g[s]));
    a.grid = m->scatter_grid;
    NP_TRY(launch(m, NP_KIND_SCATTER, x, 0, [&] { return launch_scatter(a, x); }));
    CUDA_TRY(cudaEventRecord(m->ev_layer[s], x));
  }
  return NP_OK;
}

// Restore the slots written for sparse layer s by the pending delta.
np_status enqueue_restore(np_model* m, int s) {
  cudaStream_t st = m->xs;
  NP_TRY(join(m, st, m->ev_layer[s]));
  MoveLaunch a = move_args(m, s);
  a.din_oldct = m->din_oldct + (size_t)s * m->K;
  a.chunk_begin = 0;
  a.chunk_cap = m->K;
  a.grid = m->gather_grid;
  return launch(m, NP_KIND_GATHER, st, 0, [&] { return launch_restore(a, st); });
}

SetLaunch set_args(np_model* m, int first_sparse, int n_layers) {
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
  a.frequency = m->frequency;
  a.batch = m->B;
  a.n_heads = m->NH;
  a.token = (int)m->token;
  a.token_dev = m->token_dev;
  a.centroids = m->d.centroids;
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
  a.din_oldct = m->din_oldct;
  a.dout_n = m->dout_n;
  a.dout_s = m->dout_s;
  a.ls_old = m->ls_old;
  a.totals = m->totals;
  a.slot_hw = m->slot_hw;
  a.compact = m->compact;
  a.mv_src = m->mv_src;
  a.mv_dst = m->mv_dst;
  a.mv_oldct = m->mv_oldct;
  a.mv_count = m->mv_count;
  a.err = m->err;
  return a;
}

// Drop every pending delta: copy back the bytes of the slots already written
// for the layers in `moved`, then undo the state changes of all pending
// layers from the recorded lists.
np_status abort_pending(np_model* m, const std::vector<int>& moved) {
  for (int s : moved) NP_TRY(enqueue_restore(m, s));
  NP_TRY(join_side(m, m->main));
  cudaStream_t st = m->main;
  for (int s = 0; s < m->S; ++s) {
    if (!(m->pending_bits & (1ull << s))) continue;
    SetLaunch a = set_args(m, s, 1);
    NP_TRY(launch(m, NP_KIND_SET, st, 0, [&] { return launch_rollback(a, st); }));
  }
  m->pending_bits = 0;
  return NP_OK;
}

// Reads for the pending layers in `layers` (ascending), with the read hook.
// On a hook failure returns NP_ERR_IO with *n_moved = layers whose reads were
// enqueued; the caller aborts the pending deltas.
np_status move_layers(np_model* m, const std::vector<int>& layers, size_t* n_moved) {
  *n_moved = 0;
  NP_TRY(join(m, m->side, m->ev_set));
  NP_TRY(join(m, m->g1, m->ev_set));
  for (size_t k = 0; k < layers.size(); ++k) {
    const int s = layers[k];
    if (m->d.read_hook && m->d.read_hook(m->d.read_ctx, m->dn + s, (int32_t)m->token) != 0) {
      g_last_err = "storage read hook failed";
      return NP_ERR_IO;
    }
    NP_TRY(enqueue_move(m, s));
    *n_moved = k + 1;
  }
  return NP_OK;
}

np_status bump_token(np_model* m) {
  cudaStream_t st = m->main;
  return launch(m, NP_KIND_FINISH, st, 0, [&] {
    bump_kernel<<<1, 32, 0, st>>>(m->token_dev);
    return cudaGetLastError();
  });
}

np_status commit(np_model* m, uint64_t bits) {
  m->pending_bits &= ~bits;
  m->committed_since_token |= bits;
  if ((m->committed_since_token & all_layers(m)) == all_layers(m)) {
    m->committed_since_token = 0;
    m->token += 1;
    return bump_token(m);
  }
  return NP_OK;
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
  CUDA_TRY(cudaStreamSynchronize(m->g1));
  CUDA_TRY(cudaStreamSynchronize(m->xs));
  CUDA_TRY(cudaStreamSynchronize(m->fs));
  if (m->gs) CUDA_TRY(cudaStreamSynchronize(m->gs));
  if (m->ps) CUDA_TRY(cudaStreamSynchronize(m->ps));
  if (m->ss) CUDA_TRY(cudaStreamSynchronize(m->ss));
  CUDA_TRY(cudaStreamSynchronize(m->main));
  return NP_OK;
}

// Rows per predictor ring stage: powers of two up to 8 whose stage stays
// within `stage_cap` bytes (NP_TUNE_PRED_STAGE_BYTES, default 24 KiB).
int pick_rps(size_t row_bytes, size_t stage_cap) {
  int r = 1;
  while (r < 8 && (size_t)(r * 2) * row_bytes <= stage_cap) r *= 2;
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
  if (d->d_model / (16 / esz) > kThreads * kMaxChunksPerThread || d->d_model / (16 / esz) > ffn_max_chunks())
    return arg_fail("d_model too large for dtype");
  if (d->d_ff < 1 || d->d_ff > 16384) return arg_fail("d_ff must be in [1, 16384]");
  if (d->k_max < 1 || d->k_max > d->d_ff || d->k_max > 8192) return arg_fail("k_max must be in [1, min(d_ff, 8192)]");
  if (d->has_gate != 0 && d->has_gate != 1) return arg_fail("has_gate must be 0 or 1");
  if (d->combine != NP_COMBINE_INTERSECT && d->combine != NP_COMBINE_UNION) return arg_fail("bad combine");
  if (d->residency != NP_RES_SLOTMAP && d->residency != NP_RES_WINDOW && d->residency != NP_RES_FREQUENCY)
    return arg_fail("bad residency");
  if (d->lookahead < 0 || d->lookahead > d->n_layers) return arg_fail("lookahead must be in [0, n_layers]");
  if (d->lookahead > 0 && d->pred_kind != NP_PRED_PERLAYER_SIGMOID)
    return arg_fail("lookahead applies to the per-layer predictor");
  if (d->residency == NP_RES_WINDOW && (d->window < 1 || d->window > 32)) return arg_fail("window must be 1..32");
  if (d->batch < 1 || d->batch > 8) return arg_fail("batch must be in 1..8");
  if (d->batch > 1) {
    if (d->dtype == NP_F32) return arg_fail("batched decoding needs f16 or bf16 weights");
    if (d->pred_kind != NP_PRED_SHARED_ARGMAX) return arg_fail("batched decoding uses the shared predictor");
    if (d->d_model % 128 != 0) return arg_fail("batched decoding needs d_model a multiple of 128");
    if (d->pred_hidden % 64 != 0) return arg_fail("batched decoding needs pred_hidden a multiple of 64");
  }
  if (d->staging_rows < 0 || d->staging_rows > d->k_max) return arg_fail("staging_rows must be in [0, k_max]");
  if (d->h2d_mode != NP_H2D_STAGED && d->h2d_mode != NP_H2D_FUSED) return arg_fail("bad h2d_mode");
  if (d->activation != NP_ACT_RELU && d->activation != NP_ACT_SWIGLU) return arg_fail("bad activation");
  if (d->activation == NP_ACT_SWIGLU && !d->has_gate) return arg_fail("SwiGLU needs a gate projection");
  if (d->slots != NP_SLOTS_REUSE && d->slots != NP_SLOTS_COMPACT) return arg_fail("bad slots");
  if (d->batch > 1 && d->residency != NP_RES_SLOTMAP && d->slots != NP_SLOTS_COMPACT)
    return arg_fail("batched decoding with a window or frequency residency needs the compact placement (its FFN "
                    "covers the occupied rows)");
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
  m->compact = desc->slots == NP_SLOTS_COMPACT;
  m->frequency = desc->residency == NP_RES_FREQUENCY;
  m->lookahead = desc->lookahead;
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
  {
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    e = ffn_plan(m->d.dtype, m->d.has_gate, m->D, m->esz, (size_t)smem_sm, m->sms, &m->ffn_stages, &m->ffn_grid);
    if (e != cudaSuccess) return fail(cuda_fail(e, "ffn_plan"));
    // NP_TUNE_FFN_SLOTS sets the ring depth (one CTA per SM fits up to the
    // per-block limit), NP_TUNE_FFN_CTAS the grid
    const int slots = env_int("NP_TUNE_FFN_SLOTS", 0);
    if (slots > 0) {
      if (slots > 16 || ffn_smem_bytes(m->D, m->esz, m->nproj, slots) > m->smem_optin - 1024)
        return fail(arg_fail("NP_TUNE_FFN_SLOTS does not fit in shared memory"));
      m->ffn_stages = slots;
      if ((e = ffn_set_smem(m->d.dtype, m->d.has_gate, m->D, m->esz, slots)) != cudaSuccess)
        return fail(cuda_fail(e, "ffn_set_smem"));
    }
    const int ctas = env_int("NP_TUNE_FFN_CTAS", 0);
    if (ctas > 0) m->ffn_grid = ctas;
    // A dense layer streams every row of d_ff (72 per CTA at the 7B shape)
    // and, as the token's first kernel, runs alone: a deeper ring with one
    // CTA per SM keeps the rows ahead of the consumers (7B dense layer 0 in
    // the decode: 54 -> 49 us).  The sparse layers keep the two-per-SM ring,
    // so that the next layer's CTAs and the reads fit beside them.
    // NP_TUNE_DENSE_SLOTS sets the dense ring (default 6).
    m->ffn_stages_dense = m->ffn_stages;
    int ds = env_int("NP_TUNE_DENSE_SLOTS", 6);
    if (ds > 16) ds = 16;
    while (ds > m->ffn_stages && ffn_smem_bytes(m->D, m->esz, m->nproj, ds) > m->smem_optin - 1024) --ds;
    if (m->dn > 0 && ds > m->ffn_stages) {
      if ((e = ffn_set_smem(m->d.dtype, m->d.has_gate, m->D, m->esz, ds)) != cudaSuccess)
        return fail(cuda_fail(e, "ffn_set_smem"));
      m->ffn_stages_dense = ds;
    }
    if (m->B == 1) {
      e = ffn_chain_plan(m->d.dtype, m->d.has_gate, m->D, m->esz, m->smem_optin - 1024, m->sms, &m->chain_stages,
                         &m->chain_grid);
      if (e != cudaSuccess) return fail(cuda_fail(e, "ffn_chain_plan"));
    }
  }
  // Host-link gathers need only a few MB in flight to fill the link; keeping
  // their grids small leaves the SMs to the FFN running beside them.
  // NP_TUNE_GATHER_CTAS / NP_TUNE_SCATTER_CTAS override the defaults.
  m->graph_off = env_int("NP_TUNE_GRAPH", 1) == 0;
  m->graph_pdl = env_int("NP_TUNE_GRAPH_PDL", 1) != 0;
  // Per-token pipeline: by default where a dense prefix of two or more
  // layers sits on the stream pipeline's FFN stream ahead of the sparse
  // layers (measured: Llama-2-13B shape 516 -> 540 tok/s; the 7B shape, one
  // dense layer, is faster on the stream pipeline, 756 vs 702, because its
  // reads start after the first predictor group instead of after all of
  // them).  NP_TUNE_TOKEN_CHAIN=0/1 forces it off/on.
  const int tc_env = env_int("NP_TUNE_TOKEN_CHAIN", -1);
  m->token_chain = (tc_env == 1 || (tc_env == -1 && m->dn >= 2)) && m->B == 1 && m->S > 0 &&
                   m->d.pred_kind == NP_PRED_SHARED_ARGMAX && !m->compact && m->d.h2d_mode == NP_H2D_FUSED;
  // Failure test hook (never set in normal use): NP_TEST_WITHHOLD_ARRIVAL=l
  // withholds one reader arrival for layer l in the per-token pipeline, so
  // that token ends with NP_ERR_TIMEOUT after the kernel's bounded waits.
  m->withhold_layer = env_int("NP_TEST_WITHHOLD_ARRIVAL", -1);
  m->set_stream = env_int("NP_TUNE_SET_STREAM", 1) != 0;
  m->pdl_mask = env_int("NP_TUNE_PDL", 5);
  m->gather_grid = env_int("NP_TUNE_GATHER_CTAS", 32);
  m->scatter_grid = env_int("NP_TUNE_SCATTER_CTAS", 4 * m->sms);
  if (m->gather_grid < 1) m->gather_grid = 32;
  if (m->scatter_grid < 1) m->scatter_grid = 4 * m->sms;
  m->pred_grid = 2 * m->sms;
  const int pred_ctas = env_int("NP_TUNE_PRED_CTAS", 0);
  if (pred_ctas > 0) m->pred_grid = pred_ctas;
  if (env_int("NP_TUNE_VERBOSE", 0) == 1)
    std::fprintf(stderr, "np: ffn grid %d, ring %d slots; gather %d scatter %d CTAs\n", m->ffn_grid, m->ffn_stages,
                 m->gather_grid, m->scatter_grid);
  {
    // The shared predictor streams long runs of rows alone or beside the
    // sparse FFNs: 48 KiB stages halve its block barriers per byte (7B heads
    // alone 93.5 -> 90.6 us, 13B 117 -> 114 us).  The per-layer predictor
    // keeps 24 KiB stages, so that its rings still fit beside an FFN CTA.
    const int dflt = m->d.pred_kind == NP_PRED_SHARED_ARGMAX ? 49152 : 24576;
    const int cap = env_int("NP_TUNE_PRED_STAGE_BYTES", dflt);
    const size_t stage_cap = cap > 0 ? (size_t)cap : (size_t)dflt;
    m->rps1 = pick_rps(m->row_bytes, stage_cap);
    m->rps2 = pick_rps((size_t)m->H * m->esz, stage_cap);
  }
  m->ns1 = pick_stages(m->rps1 * m->row_bytes, rowdot_smem_bytes(m->D, m->esz, m->rps1, 0), per_cta);
  m->ns2 = pick_stages(m->rps2 * (size_t)m->H * m->esz, rowdot_smem_bytes(m->H, m->esz, m->rps2, 0), per_cta);
  if (m->ns1 < 2 || m->ns2 < 2) return fail(arg_fail("predictor rows too large for the shared-memory ring"));
  {
    // The per-layer predictor with a lookahead runs on its own stream beside
    // the FFN.  Its CTAs (two per SM) then share each SM with one FFN CTA, so
    // their rings are cut to what fits beside it; otherwise a second
    // predictor CTA finds no room on SMs that hold an FFN CTA and the
    // predictor runs in two waves.  Measured on the OPT window workload
    // (lookahead 2, from its warm fill): 935 tok/s with the full rings,
    // 1030-1049 with rings that fit; alone, the full rings stream faster
    // (0.59 vs 0.47 of HBM).
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    const size_t ffn_cta = ffn_smem_bytes(m->D, m->esz, m->nproj, m->ffn_stages) + 1024;
    const size_t pair = (size_t)smem_sm > ffn_cta ? ((size_t)smem_sm - ffn_cta) / 2 : 0;
    const size_t side = pair > 1024 ? pair - 1024 : 0;
    const int s1 = pick_stages(m->rps1 * m->row_bytes, rowdot_smem_bytes(m->D, m->esz, m->rps1, 0), side);
    const int s2 = pick_stages(m->rps2 * (size_t)m->H * m->esz, rowdot_smem_bytes(m->H, m->esz, m->rps2, 0), side);
    m->ns1_side = s1 >= 2 ? std::min(s1, m->ns1) : m->ns1;
    m->ns2_side = s2 >= 2 ? std::min(s2, m->ns2) : m->ns2;
    if (env_int("NP_TUNE_PRED_SIDE_FIT", 1) == 0) {  // full rings on the lookahead stream too
      m->ns1_side = m->ns1;
      m->ns2_side = m->ns2;
    }
    // NP_TUNE_PRED_STAGES caps every predictor ring (for sweeps)
    const int cap = env_int("NP_TUNE_PRED_STAGES", 0);
    if (cap >= 2) {
      m->ns1 = std::min(m->ns1, cap);
      m->ns2 = std::min(m->ns2, cap);
      m->ns1_side = std::min(m->ns1_side, cap);
      m->ns2_side = std::min(m->ns2_side, cap);
    }
  }

  // allocations
  const size_t S = (size_t)m->S, F = m->F, K = m->K;
  const size_t Sa = S > 0 ? S : 1;
  if ((st = dev_alloc(m, reinterpret_cast<unsigned char**>(&m->bufs), Sa * m->nproj * K * m->row_bytes)) != NP_OK)
    return fail(st);
  if (m->d.h2d_mode == NP_H2D_STAGED &&
      (st = dev_alloc(m, reinterpret_cast<unsigned char**>(&m->staging), 2 * (size_t)m->staging_rows * m->rec_bytes)) !=
          NP_OK)
    return fail(st);
  if ((st = dev_alloc(m, &m->slotmap, Sa * F, 0xff)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->inv, Sa * K, 0xff)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->content, Sa * K, 0xff)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->resbits, Sa * m->W)) != NP_OK) return fail(st);
  if ((m->window > 1 || m->frequency) && (st = dev_alloc(m, &m->last_seen, Sa * F)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->counts, Sa * 4)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->active, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->active_slot, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->din_n, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->din_s, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->din_oldct, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->dout_n, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->dout_s, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->ls_old, Sa * K)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->slot_hw, Sa)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->token_dev, 1)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->h_io, (size_t)m->B * m->D)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->mv_count, Sa)) != NP_OK) return fail(st);
  if (m->compact && ((st = dev_alloc(m, &m->mv_src, Sa * K)) != NP_OK || (st = dev_alloc(m, &m->mv_dst, Sa * K)) != NP_OK ||
                     (st = dev_alloc(m, &m->mv_oldct, Sa * K)) != NP_OK))
    return fail(st);
  if ((st = dev_alloc(m, &m->totals, 8)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->err, 4)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->z, (size_t)m->B * m->H)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->keys, (size_t)m->B * (m->NH > 0 ? m->NH : 1))) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->ids, (size_t)m->B * (m->NH > 0 ? m->NH : 1))) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->fire, (size_t)m->W)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->fire2, (size_t)m->W)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->logits, F)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->arrive, 2 * (size_t)m->L)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->gdone, (size_t)m->L)) != NP_OK) return fail(st);
  if (m->B == 1 && (st = dev_alloc(m, &m->chain_part, (size_t)m->chain_grid * m->D)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->hbase, 2 * (size_t)m->B * m->D)) != NP_OK) return fail(st);
  if ((st = dev_alloc(m, &m->yacc, 3 * (size_t)m->B * m->D)) != NP_OK) return fail(st);

  if (m->B > 1) {
    // tensor-core path: maps over every weight block the gathers read
    m->tc = true;
    const int dt = m->d.dtype;
    const size_t optin = m->smem_optin - 1024;
    int want = env_int("NP_TUNE_MMA_CLUSTERS", 0);
    int max_st = env_int("NP_TUNE_MMA_STAGES", 0);
    if (want < 0) want = 0;
    if (max_st < 0) max_st = 0;
    const int ffn_mode = m->d.has_gate ? kMmaFfnGated : kMmaFfnUp;
    // At most two CTAs of these kernels on one SM: each allocates 256 of the
    // SM's 512 tensor-memory columns, and a third would wait for columns
    // inside the kernel.  A stage cap that would leave three CTAs' shared
    // memory on one SM is raised until it does not.
    int smem_sm = 0;
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    auto plan2 = [&](int mode, int Kdim, MmaPlan* p) -> cudaError_t {
      for (int st = max_st;; ++st) {
        const cudaError_t pe = mma_plan(mode, dt == NP_BF16, Kdim, optin, m->sms, want, st, p);
        if (pe != cudaSuccess) return pe;
        if (3 * (p->smem + 1024) > (size_t)smem_sm) return cudaSuccess;
        if (st == 0 || p->n_stages < st) return cudaErrorInvalidConfiguration;  // no deeper ring fits
      }
    };
    if ((e = plan2(ffn_mode, m->D, &m->plan_ffn)) != cudaSuccess ||
        (e = plan2(kMmaHidden, m->D, &m->plan_hid)) != cudaSuccess ||
        (e = plan2(kMmaHeads, m->H, &m->plan_heads)) != cudaSuccess)
      return fail(cuda_fail(e, "mma_plan"));
    if (m->S > 0 && (e = make_row_maps(&m->map_bufs, m->bufs, dt, (uint64_t)m->S * m->nproj * K, m->D)) != cudaSuccess)
      return fail(cuda_fail(e, "tensor map of the resident rows"));
    if (m->dn > 0 &&
        (e = make_row_maps(&m->map_dense, m->d.dense_w, dt, (uint64_t)m->dn * m->nproj * F, m->D)) != cudaSuccess)
      return fail(cuda_fail(e, "tensor map of the dense layers"));
    if ((e = make_row_maps(&m->map_w1, m->d.pred_w1, dt, (uint64_t)m->H, m->D)) != cudaSuccess ||
        (e = make_row_maps(&m->map_w2, m->d.pred_w2, dt, (uint64_t)m->NH * m->C, m->H)) != cudaSuccess)
      return fail(cuda_fail(e, "tensor map of the predictor"));
    if ((st = dev_alloc(m, &m->zhl, 16 * (size_t)m->H)) != NP_OK) return fail(st);
    if (env_int("NP_TUNE_VERBOSE", 0) == 1)
      std::fprintf(stderr, "np: tensor-core ffn %d clusters x %d, %d stages; hidden %d x %d; heads %d x %d\n",
                   m->plan_ffn.n_clusters, m->plan_ffn.cs, m->plan_ffn.n_stages, m->plan_hid.n_clusters,
                   m->plan_hid.cs, m->plan_heads.n_clusters, m->plan_heads.cs);
  }

  e = cudaEventCreateWithFlags(&m->ev_set, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  e = cudaEventCreateWithFlags(&m->ev_side_done, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  for (int k = 0; k < 6; ++k) {
    e = cudaEventCreateWithFlags(&m->ev_j[k], cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  }
  m->ev_layer.assign(Sa, nullptr);
  m->ev_g.assign(Sa, nullptr);
  for (size_t s = 0; s < S; ++s) {
    e = cudaEventCreateWithFlags(&m->ev_layer[s], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_g[s], cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaEventCreate"));
  }
  {
    int lo = 0, hi = 0;
    cudaDeviceGetStreamPriorityRange(&lo, &hi);
    // NP_TUNE_SIDE_PRIORITY=0 puts the internal gather/scatter streams at the
    // default priority instead of the highest
    const int pr = env_int("NP_TUNE_SIDE_PRIORITY", 1) != 0 ? hi : lo;
    e = cudaStreamCreateWithPriority(&m->g1, cudaStreamNonBlocking, pr);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&m->xs, cudaStreamNonBlocking, pr);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->fs, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_pre, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_ffn, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->gs, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->ps, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_pin, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_psrc, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&m->ss, cudaStreamNonBlocking);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
      e = cudaEventCreateWithFlags(&m->ev_pdone[b], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_sdone[b], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_gin, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->ev_gout, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(cuda_fail(e, "cudaStreamCreate"));
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
  if (m->g1) cudaStreamSynchronize(m->g1);
  if (m->xs) cudaStreamSynchronize(m->xs);
  cudaDeviceSynchronize();
  if (m->fs) cudaStreamSynchronize(m->fs);
  if (m->g1) cudaStreamDestroy(m->g1);
  if (m->xs) cudaStreamDestroy(m->xs);
  if (m->fs) cudaStreamDestroy(m->fs);
  if (m->gs) cudaStreamDestroy(m->gs);
  if (m->ps) cudaStreamDestroy(m->ps);
  if (m->ss) cudaStreamDestroy(m->ss);
  for (int b = 0; b < 2; ++b) {
    if (m->ev_pdone[b]) cudaEventDestroy(m->ev_pdone[b]);
    if (m->ev_sdone[b]) cudaEventDestroy(m->ev_sdone[b]);
  }
  if (m->ev_pin) cudaEventDestroy(m->ev_pin);
  if (m->ev_psrc) cudaEventDestroy(m->ev_psrc);
  if (m->ev_gin) cudaEventDestroy(m->ev_gin);
  if (m->ev_gout) cudaEventDestroy(m->ev_gout);
  if (m->ev_pre) cudaEventDestroy(m->ev_pre);
  if (m->graph) cudaGraphExecDestroy(m->graph);
  if (m->ev_ffn) cudaEventDestroy(m->ev_ffn);
  for (cudaEvent_t ev : m->ev_j)
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : m->ev_g)
    if (ev) cudaEventDestroy(ev);
  for (void* p : m->allocs) cudaFree(p);
  if (m->ev_set) cudaEventDestroy(m->ev_set);
  if (m->ev_side_done) cudaEventDestroy(m->ev_side_done);
  for (cudaEvent_t ev : m->ev_layer)
    if (ev) cudaEventDestroy(ev);
  for (auto& t : m->trace) {
    cudaEventDestroy(t.second.a);
    cudaEventDestroy(t.second.b);
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
  begin_call(m);
  // a delta that was never scattered already changed the slot contents
  if (m->pending_bits) NP_TRY(abort_pending(m, std::vector<int>()));
  m->pending_bits = 0;
  m->committed_since_token = 0;
  m->token = 0;
  if (m->S == 0) return NP_OK;
  cudaStream_t st = m->main;
  NP_TRY(join_side(m, st));
  CUDA_TRY(cudaMemsetAsync(m->token_dev, 0, sizeof(int), st));
  forget(m, st);
  return launch(m, NP_KIND_SET, st, 0, [&] {
    return launch_reset_state(m->slotmap, m->inv, m->resbits, m->slot_hw, m->frequency ? m->last_seen : nullptr, m->S,
                              m->F, m->K, m->W, st);
  });
}

np_status np_predict(np_model* m, int32_t layer, const float* h_dev, void* out_dev) {
  if (!m || !h_dev || !out_dev) return arg_fail("null argument");
  begin_call(m);
  if (!aligned16(h_dev)) return arg_fail("h_dev must be 16-byte aligned");
  if (m->d.pred_kind == NP_PRED_SHARED_ARGMAX) {
    if (layer != 0) return arg_fail("the shared predictor takes layer 0");
    NP_TRY(enqueue_predict(m, 0, h_dev));
    CUDA_TRY(cudaMemcpyAsync(out_dev, m->ids, sizeof(int) * m->B * m->NH, cudaMemcpyDeviceToDevice, m->main));
    forget(m, m->main);
    return NP_OK;
  }
  if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
  NP_TRY(enqueue_predict(m, layer, h_dev));
  CUDA_TRY(cudaMemcpyAsync(out_dev, m->fire, sizeof(uint32_t) * m->W, cudaMemcpyDeviceToDevice, m->main));
  forget(m, m->main);
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
  v->move_count = m->mv_count;
  v->move_src = m->mv_src;
  v->move_dst = m->mv_dst;
}

np_status np_last_delta(np_model* m, np_delta_view* out) {
  if (!m || !out) return arg_fail("null argument");
  fill_view(m, out);
  return NP_OK;
}

np_status np_delta(np_model* m, int32_t layer, const void* pred_dev, np_delta_view* out) {
  if (!m || !pred_dev) return arg_fail("null argument");
  begin_call(m);
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
  begin_call(m);
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
  size_t n_moved = 0;
  const np_status rs = move_layers(m, layers, &n_moved);
  if (rs != NP_OK) {
    NP_TRY(abort_pending(m, std::vector<int>(layers.begin(), layers.begin() + n_moved)));
    return rs;
  }
  NP_TRY(join_side(m, m->main));
  uint64_t bits = 0;
  for (int s : layers) bits |= 1ull << s;
  return commit(m, bits);
}

np_status np_sparse_mlp(np_model* m, int32_t layer, const float* h_dev, float* y_dev) {
  if (!m || !h_dev || !y_dev) return arg_fail("null argument");
  begin_call(m);
  if (!aligned16(h_dev) || !aligned16(y_dev)) return arg_fail("h_dev and y_dev must be 16-byte aligned");
  if (layer < m->dn || layer >= m->L) return arg_fail("layer is not a sparse layer");
  if (h_dev == y_dev) return arg_fail("y_dev may not alias h_dev");
  CUDA_TRY(cudaMemsetAsync(y_dev, 0, sizeof(float) * m->B * m->D, m->main));
  forget(m, m->main);
  return enqueue_layer_ffn(m, m->main, layer, h_dev, nullptr, nullptr, y_dev, nullptr);
}

np_status np_dense_mlp(np_model* m, int32_t layer, const float* h_dev, float* y_dev) {
  if (!m || !h_dev || !y_dev) return arg_fail("null argument");
  begin_call(m);
  if (!aligned16(h_dev) || !aligned16(y_dev)) return arg_fail("h_dev and y_dev must be 16-byte aligned");
  if (layer < 0 || layer >= m->dn) return arg_fail("layer is not a dense layer");
  if (h_dev == y_dev) return arg_fail("y_dev may not alias h_dev");
  CUDA_TRY(cudaMemsetAsync(y_dev, 0, sizeof(float) * m->B * m->D, m->main));
  forget(m, m->main);
  return enqueue_layer_ffn(m, m->main, layer, h_dev, nullptr, nullptr, y_dev, nullptr);
}

// The persistent chain over layers first .. first+count-1 (batch 1) on the
// residual stream h_dev; the arrival counters must be zero.
FfnChainLaunch chain_args(np_model* m, int first, int count, float* h_dev) {
  FfnChainLaunch a{};
  a.dense_w = m->d.dense_w;
  a.bufs = m->bufs;
  a.active_slot = m->active_slot;
  a.counts = m->counts;
  a.n_rows = m->slot_hw;
  a.compact = m->compact;
  a.n_dense = m->dn;
  a.F = m->F;
  a.K = m->K;
  a.first = first;
  a.count = count;
  a.h = h_dev;
  a.hbase = m->hbase;
  a.yacc = m->yacc;
  a.part = m->chain_part;
  a.arrive = m->arrive;
  a.D = m->D;
  a.dtype = m->d.dtype;
  a.dtype_bytes = m->esz;
  a.gated = m->d.has_gate;
  a.swiglu = m->d.activation == NP_ACT_SWIGLU;
  a.n_stages = m->chain_stages;
  a.grid = m->chain_grid;
  a.err = m->err;
  a.withhold = -1;
  return a;
}

np_status np_ffn_layers(np_model* m, int32_t first, int32_t count, float* h_dev) {
  if (!m || !h_dev) return arg_fail("null argument");
  begin_call(m);
  if (!aligned16(h_dev)) return arg_fail("h_dev must be 16-byte aligned");
  if (first < 0 || count < 1 || first + count > m->L) return arg_fail("layer range out of bounds");
  for (int l = first; l < first + count; ++l)
    if (l >= m->dn && (m->pending_bits & (1ull << (l - m->dn)))) {
      g_last_err = "a delta is pending for a layer in the range";
      return NP_ERR_STATE;
    }
  // the same chaining as np_decode_token, relative to `first`
  cudaStream_t st = m->main;
  CUDA_TRY(cudaMemsetAsync(chain_y(m, 0), 0, sizeof(float) * m->B * m->D, st));
  forget(m, st);
  if (!m->tc) {
    // batch 1: one persistent kernel streams the whole range
    CUDA_TRY(cudaMemsetAsync(m->arrive, 0, sizeof(unsigned) * 2 * (size_t)count, st));
    forget(m, st);
    const FfnChainLaunch a = chain_args(m, first, count, h_dev);
    return launch(m, NP_KIND_FFN, st, 0, [&] { return launch_ffn_chain(a, st); });
  }
  for (int i = 0; i < count; ++i) {
    const float* hb = i <= 1 ? h_dev : chain_base(m, i - 1);
    NP_TRY(enqueue_layer_ffn(m, st, first + i, hb, i == 0 ? nullptr : chain_y(m, i - 1),
                             i >= 1 ? chain_base(m, i) : nullptr, chain_y(m, i), chain_y(m, i + 1)));
  }
  const float* hb = count == 1 ? h_dev : chain_base(m, count - 1);
  return launch(m, NP_KIND_FINISH, st, 0,
                [&] { return launch_add(h_dev, hb, chain_y(m, count - 1), m->B * m->D, st); });
}

// Everything one token enqueues, with h_dev as the residual stream (in and
// out).  On a failed read the token's deltas are rolled back and NP_ERR_IO
// returned.  Ends with the device token counter advanced.
np_status enqueue_token(np_model* m, float* h_dev) {
  const bool shared = m->d.pred_kind == NP_PRED_SHARED_ARGMAX;
  // Residual chaining: layer l reads base(l) + y(l-1) and adds its y into
  // y(l); the residual stream after the last layer is written back by a
  // final add.  y(0) starts cleared; layer l clears y(l+1).
  auto base_of = [&](int l) -> const float* { return l <= 1 ? h_dev : chain_base(m, l - 1); };
  auto ffn_layer = [&](cudaStream_t st, int l) -> np_status {
    return enqueue_layer_ffn(m, st, l, base_of(l), l == 0 ? nullptr : chain_y(m, l - 1),
                             l >= 1 ? chain_base(m, l) : nullptr, chain_y(m, l), chain_y(m, l + 1));
  };
  CUDA_TRY(cudaMemsetAsync(chain_y(m, 0), 0, sizeof(float) * m->B * m->D, m->main));
  forget(m, m->main);
  cudaStream_t fin = m->main;
  if (shared && m->S > 0 && m->token_chain && !m->d.read_hook) {
    // Per-token pipeline (one persistent launch for layers 1..L-1): dense
    // layer 0, the predictor, one set kernel for every sparse layer, then a
    // cooperative kernel whose reader warps bring each sparse layer's
    // incoming records from the host store into their slots while its FFN
    // producers wait, per layer, until every CTA's readers are done.
    // Layer 0 also runs on the chain kernel (fixed-order split-K), so the
    // whole token is reproducible bit for bit.
    cudaStream_t st = m->main;
    CUDA_TRY(cudaMemsetAsync(m->arrive, 0, sizeof(unsigned) * 2, st));
    forget(m, st);
    const FfnChainLaunch a0 = chain_args(m, 0, 1, h_dev);
    NP_TRY(launch(m, NP_KIND_DENSE, st, (int64_t)m->nproj * m->F * m->row_bytes,
                  [&] { return launch_ffn_chain(a0, st); }));
    NP_TRY(enqueue_pred_hidden(m, h_dev, nullptr));
    NP_TRY(enqueue_pred_heads(m, 0, m->NH));
    m->pending_bits = all_layers(m);
    SetLaunch sa = set_args(m, 0, m->S);
    sa.keys = m->keys;
    sa.ids_out = m->ids;
    sa.pdl = pdl_for(m, st, 2);
    NP_TRY(launch(m, NP_KIND_SET, st, (int64_t)m->S * m->W * 8, [&] { return launch_set(sa, st); }));
    CUDA_TRY(cudaMemsetAsync(m->arrive, 0, sizeof(unsigned) * 2 * (size_t)(m->L - 1), st));
    CUDA_TRY(cudaMemsetAsync(m->gdone, 0, sizeof(unsigned) * (size_t)(m->L - 1), st));
    forget(m, st);
    FfnChainLaunch a = chain_args(m, 1, m->L - 1, h_dev);
    a.g_store = m->store_dev;
    a.din_n = m->din_n;
    a.din_s = m->din_s;
    a.gdone = m->gdone;
    a.withhold = m->withhold_layer >= 1 ? m->withhold_layer - 1 : -1;
    NP_TRY(launch(m, NP_KIND_FFN, st, 0, [&] { return launch_ffn_chain(a, st); }));
    return bump_token(m);
  }
  if (shared && m->S > 0) {
    // main: dense layer 0, the predictor's hidden layer, then per layer
    // group the group's predictor heads, its set kernel and its reads on the
    // gather streams, so that transfers start after the first small group.
    // The FFN stream runs dense layers 1..d-1 (once the predictor has read
    // h) and then the sparse FFNs, each after its own rows have arrived.
    NP_TRY(ffn_layer(m->main, 0));
    NP_TRY(enqueue_pred_hidden(m, h_dev, chain_y(m, 0)));
    CUDA_TRY(cudaEventRecord(m->ev_pre, m->main));
    NP_TRY(join(m, m->fs, m->ev_pre));
    for (int l = 1; l < m->dn; ++l) NP_TRY(ffn_layer(m->fs, l));
    m->pending_bits = all_layers(m);
    std::vector<int> moved;
    int s0 = 0;
    for (int g = 1; s0 < m->S; g *= 2) {
      const int cnt = g < m->S - s0 ? g : m->S - s0;
      const bool last = s0 + cnt == m->S;
      const int l0 = m->dn + s0;
      NP_TRY(enqueue_pred_heads(m, 2 * (l0 - 1), 2 * (l0 - 1 + cnt)));
      if (last) NP_TRY(enqueue_pred_heads(m, 0, 2 * (m->dn - 1)));  // heads of dense layers 1..d-1
      SetLaunch sa = set_args(m, s0, cnt);
      sa.keys = m->keys;
      sa.ids_out = last ? m->ids : nullptr;
      cudaStream_t st = m->main;
      sa.pdl = pdl_for(m, st, 2);
      NP_TRY(launch(m, NP_KIND_SET, st, (int64_t)cnt * m->W * 8, [&] { return launch_set(sa, st); }));
      CUDA_TRY(cudaEventRecord(m->ev_set, st));
      std::vector<int> layers;
      for (int s = s0; s < s0 + cnt; ++s) layers.push_back(s);
      size_t n_moved = 0;
      const np_status rs = move_layers(m, layers, &n_moved);
      for (size_t q = 0; q < n_moved; ++q) moved.push_back(layers[q]);
      if (rs != NP_OK) {
        // layers of later groups have no delta yet
        for (int s = s0 + cnt; s < m->S; ++s) m->pending_bits &= ~(1ull << s);
        NP_TRY(abort_pending(m, moved));
        return rs;
      }
      s0 += cnt;
    }
    for (int s = 0; s < m->S; ++s) {
      NP_TRY(join(m, m->fs, m->ev_layer[s]));
      NP_TRY(ffn_layer(m->fs, m->dn + s));
    }
    fin = m->fs;
  } else {
    // Per-layer predictor: the prediction, delta and reads of sparse layer j
    // are enqueued once the input of layer max(j - k, 0) is final, i.e. just
    // before that layer's FFN, so with a lookahead k > 0 the reads of layer
    // j run on the gather streams during the FFNs of layers j - k .. j - 1.
    // (A model with the shared predictor gets here only without sparse layers.)
    // With a lookahead the predictor and set kernels run on their own stream
    // (ps) beside the FFNs: the predictions reading the input of layer l wait
    // for the FFN of layer l - 1, and the FFN of layer l + 1, which reuses the
    // buffers holding that input, waits for them.
    const int k = m->lookahead;
    const bool split = !shared && k > 0;
    cudaStream_t main_st = m->main;
    bool pred_pending = false;  // predictions of the previous source layer on ps
    bool fire_used[2] = {false, false};  // firing-mask buffers read by a set kernel this token
    int next = m->dn;           // next sparse layer to predict
    for (int l = 0; l < m->L; ++l) {
      if (split && pred_pending) {
        NP_TRY(join(m, main_st, m->ev_psrc));
        pred_pending = false;
      }
      const int upto = l == 0 ? k : l + k;  // layers whose predictor reads the input of layer l
      if (split && !shared && next < m->L && next <= upto) {
        CUDA_TRY(cudaEventRecord(m->ev_pin, main_st));
        NP_TRY(join(m, m->ps, m->ev_pin));
      }
      for (; !shared && next < m->L && next <= upto; ++next) {
        const int s = next - m->dn;
        const int src = next - k > 0 ? next - k : 0;
        np_status rs = NP_OK;
        if (split && m->set_stream) {
          // ps: the predictor writes firing-mask buffer b, once the set
          // kernel two layers back has read it; ss: the set kernel reads it
          const int b = s & 1;
          uint32_t* fire = b ? m->fire2 : m->fire;
          if (fire_used[b]) NP_TRY(join(m, m->ps, m->ev_sdone[b]));
          m->main = m->ps;
          rs = enqueue_predict(m, next, base_of(src), true, src == 0 ? nullptr : chain_y(m, src - 1), fire);
          m->main = main_st;
          NP_TRY(rs);
          CUDA_TRY(cudaEventRecord(m->ev_psrc, m->ps));  // the source layer's input has been read
          pred_pending = true;
          CUDA_TRY(cudaEventRecord(m->ev_pdone[b], m->ps));
          NP_TRY(join(m, m->ss, m->ev_pdone[b]));
          m->main = m->ss;
          rs = enqueue_set(m, s, 1, nullptr, fire);  // records ev_set on ss for the reads below
          m->main = main_st;
          NP_TRY(rs);
          CUDA_TRY(cudaEventRecord(m->ev_sdone[b], m->ss));
          fire_used[b] = true;
        } else {
          if (split) m->main = m->ps;
          rs = enqueue_predict(m, next, base_of(src), true, src == 0 ? nullptr : chain_y(m, src - 1));
          if (rs == NP_OK) rs = enqueue_set(m, s, 1, nullptr, m->fire);
          m->main = main_st;
          NP_TRY(rs);
          if (split) {
            CUDA_TRY(cudaEventRecord(m->ev_psrc, m->ps));
            pred_pending = true;
          }
        }
        m->pending_bits |= 1ull << s;
        size_t n_moved = 0;
        rs = move_layers(m, std::vector<int>{s}, &n_moved);
        if (rs != NP_OK) {
          // earlier layers of this token already hold their new rows: put the
          // previous contents back and undo the whole token's delta
          std::vector<int> moved;
          for (int q = 0; q < s; ++q) moved.push_back(q);
          NP_TRY(abort_pending(m, moved));
          return rs;
        }
      }
      if (l >= m->dn) NP_TRY(join(m, m->main, m->ev_layer[l - m->dn]));
      NP_TRY(ffn_layer(m->main, l));
    }
    if (split && pred_pending) NP_TRY(join(m, main_st, m->ev_psrc));
  }
  if (m->L > 0) {
    const int l = m->L - 1;
    const float* hb = l == 0 ? h_dev : chain_base(m, l);  // layer l stored its input h_l there
    NP_TRY(launch(m, NP_KIND_FINISH, fin, 0,
                  [&] { return launch_add(h_dev, hb, chain_y(m, l), m->B * m->D, fin); }));
  }
  if (fin != m->main) {
    CUDA_TRY(cudaEventRecord(m->ev_ffn, fin));
    NP_TRY(join(m, m->main, m->ev_ffn));
  }
  if (m->S > 0) NP_TRY(bump_token(m));
  return NP_OK;
}

// Put back the full edges that relax_ffn_edges made programmatic.
bool restore_ffn_edges(np_model* m, cudaGraph_t g) {
  cudaGraphEdgeData prog{};
  prog.from_port = cudaGraphKernelNodePortProgrammatic;
  prog.type = cudaGraphDependencyTypeProgrammatic;
  const cudaGraphEdgeData full{};
  bool ok = true;
  for (auto& e : m->relaxed) {
    if (cudaGraphRemoveDependencies(g, &e.first, &e.second, &prog, 1) != cudaSuccess ||
        cudaGraphAddDependencies(g, &e.first, &e.second, &full, 1) != cudaSuccess)
      ok = false;
  }
  m->relaxed.clear();
  cudaGetLastError();
  return ok;
}

// In the captured token, a layer's FFN that follows the previous layer's FFN
// on its stream after event waits (its rows' reads, the predictions that
// read its input buffers) has full edges from all of them: capture keeps a
// programmatic edge only for a launch with one dependency, and one from
// another stream would be unsound (that stream's kernel writes the rows).
// Here the edge from the previous FFN alone becomes programmatic.  Both FFN
// kernels trigger their dependents as they start; before griddepcontrol.wait
// they read only weights, row counts, row lists and slot maps, which come
// from the set kernel and the layer's reads through the full edges that
// stay; every CTA waits before it reads h or y or writes anything.  So
// layer l's rows stream while layer l-1 finishes, as between back-to-back
// launches on one stream.  Returns false on an API error (edges changed so
// far are put back).
bool relax_ffn_edges(np_model* m, cudaGraph_t g) {
  cudaGraphEdgeData prog{};
  prog.from_port = cudaGraphKernelNodePortProgrammatic;
  prog.type = cudaGraphDependencyTypeProgrammatic;
  m->relaxed.clear();
  auto fail = [&] {
    restore_ffn_edges(m, g);
    return false;
  };
  for (size_t i = 1; i < m->cap_ffn.size(); ++i) {
    cudaGraphNode_t prev = nullptr;  // the previous FFN node on the same stream
    for (size_t j = i; j-- > 0;)
      if (m->cap_ffn[j].st == m->cap_ffn[i].st) {
        prev = m->cap_ffn[j].node;
        break;
      }
    if (!prev) continue;
    cudaGraphNode_t node = m->cap_ffn[i].node;
    size_t nd = 0;
    if (cudaGraphNodeGetDependencies(node, nullptr, nullptr, &nd) != cudaSuccess) return fail();
    std::vector<cudaGraphNode_t> deps(nd);
    std::vector<cudaGraphEdgeData> ed(nd);
    if (nd > 0 && cudaGraphNodeGetDependencies(node, deps.data(), ed.data(), &nd) != cudaSuccess) return fail();
    for (size_t k = 0; k < nd; ++k) {
      // only a full edge straight from the previous FFN (another operation
      // between the two on the stream would be the dependency instead)
      if (deps[k] != prev || ed[k].type != cudaGraphDependencyTypeDefault || ed[k].from_port != 0) continue;
      if (cudaGraphRemoveDependencies(g, &prev, &node, &ed[k], 1) != cudaSuccess) return fail();
      if (cudaGraphAddDependencies(g, &prev, &node, &prog, 1) != cudaSuccess) {
        cudaGraphAddDependencies(g, &prev, &node, &ed[k], 1);
        return fail();
      }
      m->relaxed.push_back({prev, node});
    }
  }
  return true;
}

// Capture one token's launches (every stream, forked from and joined back to
// the main stream) as a graph over h_io.  A failed capture leaves the model
// on eager launches.
np_status capture_token(np_model* m) {
  const int64_t l0 = m->launches;
  cudaStream_t user_main = m->main;
  m->main = m->gs;  // the capture runs on the library's own stream
  begin_call(m);    // the graph's first kernels follow its input copy
  cudaError_t e = cudaStreamBeginCapture(m->main, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) {
    if (env_int("NP_TUNE_VERBOSE", 0) == 1) std::fprintf(stderr, "np: no capture: %s\n", cudaGetErrorString(e));
    cudaGetLastError();
    m->main = user_main;
    m->graph_off = true;
    return NP_OK;
  }
  m->capturing = true;
  m->cap_ffn.clear();
  const np_status st = enqueue_token(m, m->h_io);
  m->capturing = false;
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(m->main, &g);
  begin_call(m);
  m->main = user_main;
  m->pending_bits = 0;  // the capture only recorded the work
  m->committed_since_token = 0;
  if (st == NP_OK && e == cudaSuccess && g) {
    if (m->graph_pdl && !relax_ffn_edges(m, g) && env_int("NP_TUNE_VERBOSE", 0) == 1)
      std::fprintf(stderr, "np: FFN edges left full (%s)\n", cudaGetErrorString(cudaGetLastError()));
    e = cudaGraphInstantiate(&m->graph, g, 0);
    if (e != cudaSuccess && !m->relaxed.empty()) {
      // instantiate the token with full edges instead
      cudaGetLastError();
      m->graph = nullptr;
      e = restore_ffn_edges(m, g) ? cudaGraphInstantiate(&m->graph, g, 0) : cudaErrorUnknown;
    }
  }
  m->graph_pdl_edges = m->graph ? m->relaxed.size() : 0;
  m->relaxed.clear();  // node handles of the graph destroyed below
  if (g) cudaGraphDestroy(g);
  m->cap_ffn.clear();
  if (st != NP_OK || e != cudaSuccess || !m->graph) {
    if (env_int("NP_TUNE_VERBOSE", 0) == 1)
      std::fprintf(stderr, "np: token capture failed (status %d, %s; %s)\n", (int)st, cudaGetErrorString(e),
                   g_last_err.c_str());
    cudaGetLastError();
    m->graph = nullptr;
    m->graph_off = true;
  }
  m->graph_launches = m->launches - l0;
  m->launches = l0;
  if (m->graph && env_int("NP_TUNE_VERBOSE", 0) == 1)
    std::fprintf(stderr, "np: token captured (%lld kernels, %zu programmatic FFN edges)\n",
                 (long long)m->graph_launches, m->graph_pdl_edges);
  return NP_OK;
}

np_status np_decode_token(np_model* m, float* h_dev, np_stats* stats_host) {
  if (!m || !h_dev) return arg_fail("null argument");
  begin_call(m);
  if (!aligned16(h_dev)) return arg_fail("h_dev must be 16-byte aligned");
  if (m->pending_bits) {
    g_last_err = "a delta is pending; call np_scatter first";
    return NP_ERR_STATE;
  }
  const int64_t token = m->token;
  // Replay the captured token unless a read hook (a host call per layer) or
  // the per-launch profiler needs the launches issued one by one.
  const bool replay = !m->graph_off && !m->d.read_hook && !m->prof && m->S > 0 && m->eager_tokens > 0;
  if (replay && !m->graph) NP_TRY(capture_token(m));
  if (replay && m->graph) {
    const size_t bytes = sizeof(float) * m->B * m->D;
    CUDA_TRY(cudaMemcpyAsync(m->h_io, h_dev, bytes, cudaMemcpyDeviceToDevice, m->main));
    forget(m, m->main);
    CUDA_TRY(cudaEventRecord(m->ev_gin, m->main));
    NP_TRY(join(m, m->gs, m->ev_gin));
    CUDA_TRY(cudaGraphLaunch(m->graph, m->gs));
    CUDA_TRY(cudaEventRecord(m->ev_gout, m->gs));
    NP_TRY(join(m, m->main, m->ev_gout));
    CUDA_TRY(cudaMemcpyAsync(h_dev, m->h_io, bytes, cudaMemcpyDeviceToDevice, m->main));
    forget(m, m->main);
    m->launches += m->graph_launches;
  } else {
    NP_TRY(enqueue_token(m, h_dev));
    m->eager_tokens += 1;
  }
  if (m->S > 0) {
    m->committed_since_token = 0;
    m->pending_bits = 0;
    m->token += 1;
  }
  if (stats_host) {
    std::memset(stats_host, 0, sizeof(*stats_host));
    stats_host->token = token;
    NP_TRY(sync_model(m));
    NP_TRY(read_device_error(m));
    if (m->S > 0) {
      std::vector<int> c((size_t)m->S * 4), mv((size_t)m->S);
      CUDA_TRY(cudaMemcpy(c.data(), m->counts, c.size() * sizeof(int), cudaMemcpyDeviceToHost));
      CUDA_TRY(cudaMemcpy(mv.data(), m->mv_count, mv.size() * sizeof(int), cudaMemcpyDeviceToHost));
      for (int s = 0; s < m->S; ++s) stats_host->moved_rows += mv[s];
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
  if (m->pending_bits & (1ull << s)) {
    g_last_err = "a delta is pending for this layer";
    return NP_ERR_STATE;
  }
  NP_TRY(sync_model(m));
  if (slotmap_host)
    CUDA_TRY(cudaMemcpy(slotmap_host, m->slotmap + (size_t)s * m->F, sizeof(int) * m->F, cudaMemcpyDeviceToHost));
  if (inv_host)
    CUDA_TRY(cudaMemcpy(inv_host, m->inv + (size_t)s * m->K, sizeof(int) * m->K, cudaMemcpyDeviceToHost));
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
  if (enable < 0 || enable > 2) return arg_fail("profiling mode must be 0, 1 or 2");
  m->prof = enable != 0;
  m->prof_markers = enable == 2;
  return NP_OK;
}

np_status np_get_profile(np_model* m, double* ms_out, int64_t* launches_out, int64_t* bytes_out) {
  if (!m) return arg_fail("model is null");
  NP_TRY(sync_model(m));
  NP_TRY(prof_fold(m, m->trace.size()));
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

np_status np_get_timeline(np_model* m, int32_t* kinds, float* start_ms, float* end_ms, int32_t max_entries,
                          int32_t* n_out) {
  if (!m || !n_out) return arg_fail("null argument");
  NP_TRY(sync_model(m));
  const size_t n = m->trace.size() < (size_t)(max_entries > 0 ? max_entries : 0) ? m->trace.size()
                                                                                  : (size_t)(max_entries > 0 ? max_entries : 0);
  for (size_t i = 0; i < n; ++i) {
    float a = 0.f, b = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&a, m->trace[0].second.a, m->trace[i].second.a));
    CUDA_TRY(cudaEventElapsedTime(&b, m->trace[0].second.a, m->trace[i].second.b));
    if (kinds) kinds[i] = m->trace[i].first;
    if (start_ms) start_ms[i] = a;
    if (end_ms) end_ms[i] = b;
  }
  *n_out = (int32_t)n;
  return NP_OK;
}

int64_t np_launch_count(np_model* m) { return m ? m->launches : 0; }

}  // extern "C"
