// Attention over the local heads of one rank or several (tp_attention_heads, tp_attention_heads_ranks).
//
// diffusers "Tensor parallelism" page, §Colwise and rowwise: the colwise Q, K
// and V projections give each rank a subset of heads, so attention needs no
// communication -- each rank attends over its own heads and its output feeds
// the rowwise out-projection directly.  For local head h (columns
// [h*d, (h+1)*d) of each of Q, K, V in the rank's QKV output):
//     O_h = softmax(Q_h K_h^T / sqrt(d)) V_h        (no mask)
//
// head_dim 64 and 128 run the fused kernel of tp_flash.cu (scores and
// probabilities stay on chip).  Other head sizes take these steps, per batch of
// up to 16 heads:
//   1. S_h = Q_h . K_h^T   -- batched tcgen05 GEMM, fp32 scores [T, T];
//   2. P_h = softmax(S_h / sqrt(d)) row by row, fp32 math, written over its own
//      score row as two bf16 terms, P = P_hi + P_lo with P_hi = bf16(P) and
//      P_lo = bf16(P - P_hi) (P to about 2^-17 relative; one bf16 term would
//      carry 2^-9): each group of 8 scores becomes its 8 P_hi then its 8 P_lo
//      (one warp per row);
//   3. O_h = P_h . V_h     -- batched tcgen05 GEMM over K = 2T with B = V_h^T in
//      the same order (V is transposed once per call, every group of 8 keys
//      written twice), so one product sums P_hi V + P_lo V; bf16 written
//      straight into the rank's attention output columns [h*d, (h+1)*d).
// The score matrices are memory traffic (about 10 bytes per score).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "tp_internal.h"

namespace tp {
namespace {

constexpr int kHeadBatch = TP_MAX_DEGREE;

// The transpose of V with every group of 8 keys written twice, for the two-term P.V product:
// Vt_r[j][16c + i] = Vt_r[j][16c + 8 + i] = V_r[8c + i][j] for keys t = 8c + i < T and
// j < width, for every rank r = blockIdx.z (one launch for all ranks): V_r is [T, width] with
// row stride ld_v elements, Vt_r dense [width, 2T].
struct TransposeRanks {
  const __nv_bfloat16* v[TP_MAX_DEGREE];
  __nv_bfloat16* vt[TP_MAX_DEGREE];
  int64_t ld_v, T, width;
};

// 64 x 64 tiles through shared memory, two bf16 per 4-byte access on both sides, so a warp
// reads 128 contiguous bytes of a V row and writes 128 contiguous bytes of a V^T row.
// T and width are multiples of 8, so a pair never straddles the edge.
__global__ void __launch_bounds__(256) transpose_ranks_bf16(const __grid_constant__ TransposeRanks p) {
  __shared__ __align__(4) __nv_bfloat16 tile[64][66];  // [t][j]; 66: 4-byte rows, 2-way reads
  pdl_launch_dependents();
  pdl_wait();
  const __nv_bfloat16* v = p.v[blockIdx.z];
  __nv_bfloat16* vt = p.vt[blockIdx.z];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 64;
  const int64_t j0 = static_cast<int64_t>(blockIdx.y) * 64;
  const int lane = threadIdx.x & 31, wy = threadIdx.x >> 5;  // 32 lanes x 8 warps
#pragma unroll
  for (int k = 0; k < 64; k += 8) {
    const int64_t t = t0 + wy + k, j = j0 + 2 * lane;
    if (t < p.T && j < p.width)
      *reinterpret_cast<uint32_t*>(&tile[wy + k][2 * lane]) =
          *reinterpret_cast<const uint32_t*>(v + t * p.ld_v + j);
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 64; k += 8) {
    const int64_t j = j0 + wy + k, t = t0 + 2 * lane;
    if (j < p.width && t < p.T) {
      __nv_bfloat162 pr;
      pr.x = tile[2 * lane][wy + k];
      pr.y = tile[2 * lane + 1][wy + k];
      // t is even, so t and t + 1 share a group of 8; the pair is 4-byte aligned.
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(vt + j * 2 * p.T + 2 * t - (t & 7));
      dst[0] = pr;
      dst[4] = pr;
    }
  }
}

// Launch the transpose of n_ranks V_r slices (n_ranks <= TP_MAX_DEGREE).
tp_status transpose_ranks(int n_ranks, const __nv_bfloat16* const* v, int64_t ld_v, __nv_bfloat16* const* vt, int64_t T,
                          int64_t width, cudaStream_t s) {
  TransposeRanks prm{};
  for (int r = 0; r < n_ranks; ++r) {
    prm.v[r] = v[r];
    prm.vt[r] = vt[r];
  }
  prm.ld_v = ld_v;
  prm.T = T;
  prm.width = width;
  const dim3 grid(static_cast<unsigned>((T + 63) / 64), static_cast<unsigned>((width + 63) / 64),
                  static_cast<unsigned>(n_ranks));
  cudaError_t e = launch_pdl(transpose_ranks_bf16, grid, dim3(256), 0, s, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "transpose launch");
  return TP_OK;
}

// Row softmax of fp32 scores scaled by `scale`, written over the same row as two bf16
// terms: the 32 bytes of scores 8c..8c+7 become P_hi of those keys (8 bf16) followed by
// their P_lo (8 bf16), P_hi = bf16(P), P_lo = bf16(P - P_hi).  One warp per row; pass 1
// keeps a running (max, sum of exponentials) per lane and merges them across the warp,
// pass 2 writes P = exp(scale*(s - max)) / sum.  Each lane overwrites exactly the 32
// bytes it has just read, so no score is overwritten before it is read.
__global__ void __launch_bounds__(256) softmax_rows_inplace(float* s, int64_t rows, int T, float scale_log2e) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  float* srow = s + row * T;
  float m = -INFINITY, l = 0.f;
  for (int i = lane * 4; i < T; i += 128) {
    const float4 v = *reinterpret_cast<const float4*>(srow + i);
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float mn = fmaxf(m, x[k]);
      l = l * exp2f((m - mn) * scale_log2e) + exp2f((x[k] - mn) * scale_log2e);
      m = mn;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, mo);
    l = (m == -INFINITY ? 0.f : l * exp2f((m - mn) * scale_log2e)) +
        (mo == -INFINITY ? 0.f : lo * exp2f((mo - mn) * scale_log2e));
    m = mn;
  }
  const float inv = 1.0f / l;
  __nv_bfloat16* prow = reinterpret_cast<__nv_bfloat16*>(srow);
  for (int base = 0; base < T; base += 256) {
    const int i = base + lane * 8;
    if (i < T) {
      float x[8];
      const float4 a = *reinterpret_cast<const float4*>(srow + i);
      const float4 b = *reinterpret_cast<const float4*>(srow + i + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float p0 = exp2f((x[2 * k] - m) * scale_log2e) * inv;
        const float p1 = exp2f((x[2 * k + 1] - m) * scale_log2e) * inv;
        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        hi[k] = *reinterpret_cast<uint32_t*>(&h);
        // bf16 -> fp32 is exact, so p - P_hi is the exact residual before its own rounding.
        __nv_bfloat162 r = __floats2bfloat162_rn(p0 - __bfloat162float(h.x), p1 - __bfloat162float(h.y));
        lo[k] = *reinterpret_cast<uint32_t*>(&r);
      }
      uint4* dst = reinterpret_cast<uint4*>(prow + 2 * static_cast<int64_t>(i));
      dst[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      dst[1] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace tp

namespace tp {
namespace {

// Unfused path for one rank (head sizes other than 64 and 128), using the whole workspace.
tp_status attention_unfused(const void* qkv, int64_t ld_qkv, int64_t T, int n_heads, int head_dim, void* workspace,
                            void* out, int64_t ldo, float scale_log2e, cudaStream_t s) {
  const int64_t width = static_cast<int64_t>(n_heads) * head_dim;
  const size_t hb = static_cast<size_t>(n_heads < kHeadBatch ? n_heads : kHeadBatch);
  float* scores = static_cast<float*>(workspace);
  __nv_bfloat16* vt = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(workspace) +
                                                       align256(hb * static_cast<size_t>(T) * T * 4));
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(qkv);
  const __nv_bfloat16* k = q + width;
  const __nv_bfloat16* v = q + 2 * width;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  // V^T once for all heads, each group of 8 keys twice: [width, 2T].
  tp_status ts = transpose_ranks(1, &v, ld_qkv, &vt, T, width, s);
  if (ts != TP_OK) return ts;
  for (int h0 = 0; h0 < n_heads; h0 += kHeadBatch) {
    const int nb = (n_heads - h0) < kHeadBatch ? (n_heads - h0) : kHeadBatch;
    const void* a[kHeadBatch];
    const void* b[kHeadBatch];
    void* c[kHeadBatch];
    // 1. Scores: S_j = Q_h . K_h^T (fp32).
    for (int j = 0; j < nb; ++j) {
      a[j] = q + static_cast<int64_t>(h0 + j) * head_dim;
      b[j] = k + static_cast<int64_t>(h0 + j) * head_dim;
      c[j] = scores + static_cast<int64_t>(j) * T * T;
    }
    tp_status st = gemm_batched(nb, a, ld_qkv, b, ld_qkv, c, T, true, T, T, head_dim, s);
    if (st != TP_OK) return st;
    // 2. Softmax rows in place: P as P_hi/P_lo groups (bf16, row stride 2T elements) over S.
    const int64_t rows = static_cast<int64_t>(nb) * T;
    softmax_rows_inplace<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(scores, rows, static_cast<int>(T),
                                                                                scale_log2e);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "softmax launch");
    // 3. O_h = P_h . V_h = P_hi V_h + P_lo V_h: K = 2T, B = V_h^T with doubled key groups [head_dim, 2T].
    for (int j = 0; j < nb; ++j) {
      a[j] = scores + static_cast<int64_t>(j) * T * T;  // bf16 view: row stride 2T elements
      b[j] = vt + static_cast<int64_t>(h0 + j) * head_dim * 2 * T;
      c[j] = o + static_cast<int64_t>(h0 + j) * head_dim;
    }
    st = gemm_batched(nb, a, 2 * T, b, 2 * T, c, ldo, false, T, head_dim, 2 * T, s);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

tp_status attention_ranks(int n_ranks, const void* const* qkv, int64_t ld_qkv, int64_t T, int n_heads, int head_dim,
                          void* workspace, size_t ws_bytes, void* const* out, int64_t ldo, cudaStream_t s) {
  if (n_ranks < 1 || n_ranks > TP_MAX_DEGREE)
    return fail(n_ranks < 1 ? TP_ERR_INVALID_ARG : TP_ERR_UNSUPPORTED, "n_ranks=%d outside [1, %d]", n_ranks,
                TP_MAX_DEGREE);
  if (T < 0 || n_heads < 1 || head_dim < 1) return fail(TP_ERR_INVALID_ARG, "T >= 0, n_heads >= 1, head_dim >= 1");
  const int64_t width = static_cast<int64_t>(n_heads) * head_dim;
  if (ld_qkv == 0) ld_qkv = 3 * width;
  if (ldo == 0) ldo = width;
  if (ld_qkv < 3 * width || ldo < width) return fail(TP_ERR_INVALID_ARG, "ld_qkv or ldo smaller than the rows");
  if (T == 0) return TP_OK;
  if (qkv == nullptr || out == nullptr) return fail(TP_ERR_INVALID_ARG, "qkv or out is NULL");
  for (int r = 0; r < n_ranks; ++r)
    if (qkv[r] == nullptr || out[r] == nullptr) return fail(TP_ERR_INVALID_ARG, "qkv[%d] or out[%d] is NULL", r, r);
  if ((T % 8) || (head_dim % 8) || (ld_qkv % 8) || (ldo % 8))
    return fail(TP_ERR_ALIGNMENT, "T, head_dim, ld_qkv and ldo must be multiples of 8");
  if (T > 0x7FFFFFFF / 2) return fail(TP_ERR_UNSUPPORTED, "T=%lld too large", (long long)T);
  for (int r = 0; r < n_ranks; ++r)
    if (!aligned16(qkv[r]) || !aligned16(out[r]))
      return fail(TP_ERR_ALIGNMENT, "qkv[%d] or out[%d] is not 16-byte aligned", r, r);
  if (workspace && !aligned16(workspace)) return fail(TP_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  const size_t need = tp_attention_ranks_workspace_bytes(n_ranks, T, n_heads, head_dim);
  if (need > 0 && (workspace == nullptr || ws_bytes < need))
    return fail(TP_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace ? ws_bytes : 0, need);
  const float scale_log2e = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(head_dim)));
  if (!fused_attention_head_dim(head_dim)) {
    // One rank after another through the same workspace (stream order keeps them apart).
    for (int r = 0; r < n_ranks; ++r) {
      tp_status st = attention_unfused(qkv[r], ld_qkv, T, n_heads, head_dim, workspace, out[r], ldo, scale_log2e, s);
      if (st != TP_OK) return st;
    }
    return TP_OK;
  }
  // Fused: one launch over every rank's heads, K and V read as they are.
  return flash_attention_fused(head_dim, n_ranks, qkv, ld_qkv, T, n_heads, out, ldo, scale_log2e, s);
}

}  // namespace
}  // namespace tp

extern "C" {

size_t tp_attention_workspace_bytes(int64_t T, int n_heads, int head_dim) {
  return tp_attention_ranks_workspace_bytes(1, T, n_heads, head_dim);
}

size_t tp_attention_ranks_workspace_bytes(int n_ranks, int64_t T, int n_heads, int head_dim) {
  if (n_ranks <= 0 || T <= 0 || n_heads <= 0 || head_dim <= 0) return 0;
  if (tp::fused_attention_head_dim(head_dim)) return 0;  // the fused kernel reads Q, K and V in place
  const size_t hb = static_cast<size_t>(n_heads < tp::kHeadBatch ? n_heads : tp::kHeadBatch);
  return tp::align256(hb * static_cast<size_t>(T) * static_cast<size_t>(T) * 4) +
         tp::align256(static_cast<size_t>(n_heads) * static_cast<size_t>(head_dim) * static_cast<size_t>(T) * 4);
}

tp_status tp_attention_heads(const void* qkv, int64_t ld_qkv, int64_t T, int n_heads, int head_dim, void* workspace,
                             size_t ws_bytes, void* out, int64_t ldo, tp_stream_t stream) {
  tp::clear_error();
  const void* q[1] = {qkv};
  void* o[1] = {out};
  return tp::attention_ranks(1, q, ld_qkv, T, n_heads, head_dim, workspace, ws_bytes, o, ldo,
                             reinterpret_cast<cudaStream_t>(stream));
}

tp_status tp_attention_heads_ranks(int n_ranks, const void* const* qkv, int64_t ld_qkv, int64_t T, int n_heads,
                                   int head_dim, void* workspace, size_t ws_bytes, void* const* out, int64_t ldo,
                                   tp_stream_t stream) {
  tp::clear_error();
  return tp::attention_ranks(n_ranks, qkv, ld_qkv, T, n_heads, head_dim, workspace, ws_bytes, out, ldo,
                             reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
