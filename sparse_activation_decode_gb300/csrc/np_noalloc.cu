// Allocation-free FFN entry point (np_ffn_rows_noalloc) and its error check
// (np_ffn_rows_noalloc_check).
//
// Some callers cannot call cudaMalloc: a serving loop that runs under a
// fixed, pre-planned memory budget owned by its own allocator, or code on a
// latency-critical path where a device allocation would implicitly
// synchronize the device.  For them this entry point runs the same FFN
// kernel as np_sparse_mlp / np_dense_mlp on caller-provided weights, row
// list, input and output.  The kernel's only state besides the caller's
// buffers is its error word, which lives in one file-scope __device__ array
// of fixed size instead of a model-owned device allocation.
//
// The array is a host-side stand-in in host code: its device address is
// looked up once per device with cudaGetSymbolAddress while that device is
// current (the first call on a device does this, so that first call should
// come before any stream capture), and only that address is passed to the
// kernel.  Every call on a device shares the array and it keeps its
// contents between calls: a bounds or wait error recorded by any call stays
// in the error word until np_ffn_rows_noalloc_check reads and clears it (the
// word starts at zero when the library is loaded).  The output is cleared
// on the caller's stream before each launch.  Calls whose kernels overlap on
// the GPU race on the array: serialize them (one stream, or events).
#include <mutex>

#include "np.h"
#include "np_kernels.h"

namespace np {

constexpr int kNoallocMaxDevices = 64;
constexpr size_t kNoallocWords = 64;  // error word (and room to grow)

struct NoallocScratch {
  int words[kNoallocWords];
};

static __device__ __align__(256) NoallocScratch g_noalloc_scratch;

static std::mutex g_noalloc_mu;
static NoallocScratch* g_noalloc_ptr[kNoallocMaxDevices] = {};

static cudaError_t noalloc_scratch_for_current_device(NoallocScratch** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<NoallocScratch*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace np

namespace {

// [a, a + na) and [b, b + nb) share a byte
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

np_status noalloc_fail(np_status s, const char* what) {
  np::set_last_error(what);
  return s;
}

}  // namespace

extern "C" np_status np_ffn_rows_noalloc(const float* h_dev, const void* w_gate, const void* w_up,
                                         const void* w_down, const int32_t* rows_dev, int32_t n_rows,
                                         int32_t row_limit, int32_t d_model, int32_t dtype, int32_t has_gate,
                                         float* y_dev, void* stream) {
  using namespace np;
  if (!h_dev || !w_up || !w_down || !y_dev || (has_gate && !w_gate))
    return noalloc_fail(NP_ERR_ARG, "np_ffn_rows_noalloc: null pointer");
  if (dtype < NP_F32 || dtype > NP_BF16 || (has_gate != 0 && has_gate != 1))
    return noalloc_fail(NP_ERR_ARG, "np_ffn_rows_noalloc: bad dtype or has_gate");
  const int esz = dtype == NP_F32 ? 4 : 2;
  if (d_model < 8 || d_model > 8192 || (d_model * esz) % 16 != 0 || d_model / (16 / esz) > ffn_max_chunks())
    return noalloc_fail(NP_ERR_ARG, "np_ffn_rows_noalloc: d_model out of range");
  if (n_rows < 0 || row_limit < 1 || (!rows_dev && n_rows > row_limit))
    return noalloc_fail(NP_ERR_ARG, "np_ffn_rows_noalloc: n_rows or row_limit out of range");
  const uintptr_t align_or = reinterpret_cast<uintptr_t>(h_dev) | reinterpret_cast<uintptr_t>(y_dev) |
                             reinterpret_cast<uintptr_t>(w_gate) | reinterpret_cast<uintptr_t>(w_up) |
                             reinterpret_cast<uintptr_t>(w_down);
  if (align_or & 15u) return noalloc_fail(NP_ERR_ARG, "np_ffn_rows_noalloc: pointer not 16-byte aligned");
  // y is cleared on the stream before the kernel reads its inputs, so it may
  // share no byte with any of them
  const size_t vec_bytes = sizeof(float) * (size_t)d_model;
  const size_t w_bytes = (size_t)row_limit * (size_t)d_model * (size_t)esz;
  if (overlaps(y_dev, vec_bytes, h_dev, vec_bytes) || overlaps(y_dev, vec_bytes, w_up, w_bytes) ||
      overlaps(y_dev, vec_bytes, w_down, w_bytes) || (has_gate && overlaps(y_dev, vec_bytes, w_gate, w_bytes)) ||
      overlaps(y_dev, vec_bytes, rows_dev, sizeof(int32_t) * (size_t)n_rows))
    return noalloc_fail(NP_ERR_ARG, "np_ffn_rows_noalloc: y_dev overlaps an input");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  NoallocScratch* scratch = nullptr;
  if (noalloc_scratch_for_current_device(&scratch) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc: cudaGetSymbolAddress");
  int dev = 0, sms = 0, smem_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc: cudaGetDevice");
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  int n_stages = 0, grid = 0;
  if (ffn_plan(dtype, has_gate, d_model, esz, (size_t)smem_sm, sms, &n_stages, &grid) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc: ffn_plan");
  if (cudaMemsetAsync(y_dev, 0, vec_bytes, st) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc: clearing y");

  FfnLaunch a{};
  a.h_in = h_dev;
  a.y_acc = y_dev;
  a.w_gate = has_gate ? w_gate : nullptr;
  a.w_up = w_up;
  a.w_down = w_down;
  a.row_list = rows_dev;
  a.n_rows_dev = nullptr;
  a.n_rows_host = n_rows;
  a.list_cap = rows_dev ? n_rows : row_limit;
  a.row_limit = row_limit;
  a.D = d_model;
  a.dtype = dtype;
  a.dtype_bytes = esz;
  a.gated = has_gate;
  a.n_stages = n_stages;
  a.grid = grid;
  a.err = scratch->words;
  return launch_ffn_rows(a, st) == cudaSuccess ? NP_OK
                                               : noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc: kernel launch");
}

extern "C" np_status np_ffn_rows_noalloc_check(void* stream) {
  using namespace np;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  NoallocScratch* scratch = nullptr;
  if (noalloc_scratch_for_current_device(&scratch) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc_check: cudaGetSymbolAddress");
  if (cudaStreamSynchronize(st) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc_check: stream synchronize");
  int word = 0;
  if (cudaMemcpyAsync(&word, scratch->words, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc_check: reading the error word");
  if (word == 0) return NP_OK;
  if (cudaMemsetAsync(scratch->words, 0, sizeof(int), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return noalloc_fail(NP_ERR_CUDA, "np_ffn_rows_noalloc_check: clearing the error word");
  if (word == kDevErrTimeout) return noalloc_fail(NP_ERR_TIMEOUT, "np_ffn_rows_noalloc: a device wait timed out");
  return noalloc_fail(NP_ERR_STATE, "np_ffn_rows_noalloc: a row index was out of range");
}
