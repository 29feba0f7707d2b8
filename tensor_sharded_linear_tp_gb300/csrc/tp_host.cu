// Plan validation, diagnostics and per-device state of libtp.
//
// The plan rules follow the diffusers "Tensor parallelism" page:
// §Load a sharded model (tp_degree divides the attention-head count),
// §Fused projections (packed blocks with absolute sizes) and
// §Constraints and verification (each packed block divisible on its own,
// all checked before any weight is copied).
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "tp_internal.h"

namespace tp {

namespace {
thread_local std::string g_last_error;
std::mutex g_dev_mutex;
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
unsigned int* g_status_ptr[kMaxDevices] = {nullptr};
unsigned long long g_status_ctx[kMaxDevices] = {0};
}  // namespace

// One status word per device: kernels OR flags into it, tp_device_status reads and clears it.
__device__ unsigned int tp_kernel_status_word;

tp_status fail(tp_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = std::string(tp_status_name(st)) + ": " + buf;
  return st;
}

void clear_error() { g_last_error.clear(); }

tp_status cuda_fail(cudaError_t err, const char* what) {
  return fail(TP_ERR_CUDA, "%s failed: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

int sm_count() {
  int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

constexpr uint64_t kDefaultTileWaitNs = 2000000000ull;
std::atomic<uint64_t> g_tile_wait_ns{kDefaultTileWaitNs};

uint64_t tile_wait_limit_ns() { return g_tile_wait_ns.load(std::memory_order_relaxed); }

unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

unsigned int* status_word() {
  int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  // Cached per device and context: a new context (after cudaDeviceReset, or a caller's own
  // context) loads the module again, possibly at another address.
  if (g_status_ptr[dev] == nullptr || ctx == 0 || g_status_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, tp_kernel_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
    g_status_ctx[dev] = current_context_id();
  }
  return g_status_ptr[dev];
}

tp_status validate_plan(int64_t rows, int64_t cols, tp_style style, int tp_degree, int rank, int64_t num_heads,
                        int64_t head_dim, const int64_t* splits, int n_splits, int64_t* sizes, int* n_sizes) {
  // 1. Arguments.
  if (style != TP_COLWISE && style != TP_ROWWISE) return fail(TP_ERR_INVALID_ARG, "unknown style %d", (int)style);
  if (tp_degree < 1) return fail(TP_ERR_INVALID_ARG, "tp_degree must be >= 1, got %d", tp_degree);
  if (rank != -1 && (rank < 0 || rank >= tp_degree))
    return fail(TP_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, tp_degree);
  if (rows < 0 || cols < 0 || num_heads < 0 || head_dim < 0)
    return fail(TP_ERR_INVALID_ARG, "sizes must be non-negative");
  if (n_splits < 0 || n_splits > TP_MAX_SPLITS)
    return fail(TP_ERR_INVALID_ARG, "n_splits=%d outside [0, %d]", n_splits, TP_MAX_SPLITS);
  if (n_splits > 0 && splits == nullptr) return fail(TP_ERR_INVALID_ARG, "fused_splits is NULL with n_splits=%d", n_splits);
  const int64_t dim = (style == TP_COLWISE) ? rows : cols;
  int n = 0;
  if (n_splits == 0) {
    sizes[0] = dim;
    n = 1;
  } else {
    for (int b = 0; b < n_splits; ++b) {
      if (splits[b] <= 0) return fail(TP_ERR_INVALID_ARG, "split %d has size %lld", b, (long long)splits[b]);
      sizes[b] = splits[b];
    }
    n = n_splits;
  }
  // 2. tp_degree divides the head count.
  if (num_heads > 0 && num_heads % tp_degree != 0)
    return fail(TP_ERR_HEADS_NOT_DIVISIBLE, "tp_degree=%d does not divide num_heads=%lld", tp_degree,
                (long long)num_heads);
  // 3. Blocks cover the sharded dimension.
  int64_t sum = 0;
  for (int b = 0; b < n; ++b) sum += sizes[b];
  if (sum != dim)
    return fail(TP_ERR_SPLIT_SUM, "packed blocks sum to %lld, sharded dimension is %lld", (long long)sum,
                (long long)dim);
  // 4. Every block divisible on its own.
  for (int b = 0; b < n; ++b)
    if (sizes[b] % tp_degree != 0)
      return fail(TP_ERR_SPLIT_NOT_DIVISIBLE, "block %d of %lld not divisible by tp_degree=%d", b,
                  (long long)sizes[b], tp_degree);
  // 5. Whole heads per rank.
  if (head_dim > 0)
    for (int b = 0; b < n; ++b)
      if ((sizes[b] / tp_degree) % head_dim != 0)
        return fail(TP_ERR_NOT_WHOLE_HEADS, "block %d of %lld split %d ways is not whole heads of %lld", b,
                    (long long)sizes[b], tp_degree, (long long)head_dim);
  *n_sizes = n;
  return TP_OK;
}

}  // namespace tp

extern "C" {

tp_status tp_validate(int64_t rows, int64_t cols, tp_style style, int tp_degree, int64_t num_heads,
                      int64_t head_dim, const int64_t* fused_splits, int n_splits) {
  tp::clear_error();
  int64_t sizes[TP_MAX_SPLITS];
  int n = 0;
  return tp::validate_plan(rows, cols, style, tp_degree, -1, num_heads, head_dim, fused_splits, n_splits, sizes, &n);
}

tp_status tp_shard_shape(int64_t rows, int64_t cols, tp_style style, int tp_degree, const int64_t* fused_splits,
                         int n_splits, int64_t* out_rows, int64_t* out_cols) {
  tp::clear_error();
  if (out_rows == nullptr || out_cols == nullptr) return tp::fail(TP_ERR_INVALID_ARG, "output pointers are NULL");
  int64_t sizes[TP_MAX_SPLITS];
  int n = 0;
  tp_status st = tp::validate_plan(rows, cols, style, tp_degree, -1, 0, 0, fused_splits, n_splits, sizes, &n);
  if (st != TP_OK) return st;
  *out_rows = (style == TP_COLWISE) ? rows / tp_degree : rows;
  *out_cols = (style == TP_COLWISE) ? cols : cols / tp_degree;
  return TP_OK;
}

const char* tp_last_error(void) { return tp::g_last_error.c_str(); }

const char* tp_status_name(tp_status status) {
  switch (status) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG";
    case TP_ERR_HEADS_NOT_DIVISIBLE: return "TP_ERR_HEADS_NOT_DIVISIBLE";
    case TP_ERR_SPLIT_NOT_DIVISIBLE: return "TP_ERR_SPLIT_NOT_DIVISIBLE";
    case TP_ERR_SPLIT_SUM: return "TP_ERR_SPLIT_SUM";
    case TP_ERR_NOT_WHOLE_HEADS: return "TP_ERR_NOT_WHOLE_HEADS";
    case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT";
    case TP_ERR_NOT_PINNED: return "TP_ERR_NOT_PINNED";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE";
    case TP_ERR_CUDA: return "TP_ERR_CUDA";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    case TP_ERR_IO: return "TP_ERR_IO";
    case TP_ERR_FORMAT: return "TP_ERR_FORMAT";
    case TP_ERR_NOT_FOUND: return "TP_ERR_NOT_FOUND";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
  }
  return "TP_ERR_UNKNOWN";
}

tp_status tp_device_status(tp_stream_t stream) {
  tp::clear_error();
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tp::cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, tp::tp_kernel_status_word, sizeof(word));
  if (e != cudaSuccess) return tp::cuda_fail(e, "reading the kernel status word");
  if (word != 0) {
    unsigned int zero = 0;
    e = cudaMemcpyToSymbol(tp::tp_kernel_status_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return tp::cuda_fail(e, "clearing the kernel status word");
    return tp::fail(TP_ERR_TIMEOUT, "a kernel gave up on a bounded wait (status word 0x%x)", word);
  }
  return TP_OK;
}

void tp_set_tile_wait_limit_ns(uint64_t ns) {
  tp::g_tile_wait_ns.store(ns == 0 ? tp::kDefaultTileWaitNs : ns, std::memory_order_relaxed);
}

uint64_t tp_tile_wait_limit_ns(void) { return tp::tile_wait_limit_ns(); }

int tp_abi_version(void) { return 103; }

}  // extern "C"
