// Host-side helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>

#include "tp.h"

namespace tp {

// Record a message for tp_last_error() and return `st`.
tp_status fail(tp_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));

// Clear the calling thread's last error.
void clear_error();

// Convert a CUDA error into TP_ERR_CUDA with a message naming `what`.
tp_status cuda_fail(cudaError_t err, const char* what);

// Number of SMs of the current device (cached per device).
int sm_count();

// Device address of the library's kernel status word on the current device
// (bit 0: a kernel gave up on a bounded wait).  Looked up once per device.
unsigned int* status_word();

// Identity of the calling thread's current CUDA context, unique over the process's lifetime
// (0 when no context is current).  Device addresses of the library's own arrays are cached
// under it: a new context loads the library's modules again, possibly elsewhere.
unsigned long long current_context_id();

// The bound on a CTA's wait for other CTAs' tile partials (tp_set_tile_wait_limit_ns), in ns.
uint64_t tile_wait_limit_ns();

// Plan validation shared by every entry point.  On TP_OK, `sizes` holds the
// n_sizes absolute block sizes along the sharded dimension.
tp_status validate_plan(int64_t rows, int64_t cols, tp_style style, int tp_degree, int rank, int64_t num_heads,
                        int64_t head_dim, const int64_t* splits, int n_splits, int64_t* sizes, int* n_sizes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic dependent launch allowed: the kernel's blocks may be scheduled
// while the previous kernel in the stream is still finishing.  Every kernel launched this way
// calls pdl_launch_dependents() (its successor may be scheduled) and pdl_wait() before its
// first global-memory access (it waits for its predecessor's completion and the visibility of
// its writes), so the order of the results is that of plain stream order; what overlaps is
// launch latency and each kernel's prologue (barrier set-up, tensor-memory allocation).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

}  // namespace tp

// Bit 0 of the status word: a bounded wait gave up.
#define TP_DEVSTATUS_TIMEOUT 1u

namespace tp {
// Library-internal batched GEMM (tp_gemm.cu): out_g = A_g . B_g^T for up to TP_MAX_DEGREE groups.
tp_status gemm_batched(int groups, const void* const* a, int64_t lda, const void* const* b, int64_t ldb,
                       void* const* out, int64_t ldo, bool out_f32, int64_t M, int64_t N, int64_t K,
                       cudaStream_t stream);
}  // namespace tp

namespace tp {
// bf16 2-D tensor map over a row-major [outer, inner] matrix (row stride ld elements), cached (tp_gemm.cu).
tp_status encode_bf16_2d(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, uint32_t box_inner,
                         uint32_t box_outer, bool swizzle128);
// Fused attention for head_dim 64 or 128 over n_ranks ranks in one launch (tp_flash.cu), straight
// from each rank's QKV buffer; TP_ERR_UNSUPPORTED for other head sizes.
constexpr bool fused_attention_head_dim(int head_dim) { return head_dim == 64 || head_dim == 128; }
tp_status flash_attention_fused(int head_dim, int n_ranks, const void* const* qkv, int64_t ld_qkv, int64_t T,
                                int n_heads, void* const* out, int64_t ldo, float scale_log2e, cudaStream_t stream);
}  // namespace tp
