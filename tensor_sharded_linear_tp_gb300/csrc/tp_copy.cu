// Shard extraction (tp_plan_shard) and the in-memory joins (tp_combine).
//
// Both extraction styles and the gather are the same memory operation: a list
// of up to 64 strided 2-D copies ("segments"), each `rows` rows of `row_bytes`
// bytes, between two row strides.  One launch moves every segment:
//   * colwise (packed): one segment per packed block -- the rank's part of a
//     block is (s_b / p) consecutive rows, i.e. one contiguous run;
//   * rowwise (packed): one segment per block -- a column window of every row;
//   * gather: one segment per rank -- rank r's [T, N_each] into columns
//     [r*N_each, (r+1)*N_each) of the joined output.
// A segment whose rows are back to back in both source and destination is
// copied as one long row.  From device memory, rows are cut into pieces of at
// most 4 KiB; a warp copies one piece with 16-byte vector loads and stores, all
// of the piece's loads (up to 8 per lane) issued before its stores.  Grid: up to
// 8 blocks of 256 threads per SM, grid-stride over pieces.  HBM-bound: the
// algorithmic traffic is exactly 2 x the bytes copied.  From page-locked host
// memory (shard-on-read), each segment is one copy-engine transfer
// (cudaMemcpyAsync, or cudaMemcpy2DAsync for a column window of every row): the
// CPU-GPU link bounds it either way, and the copy engines leave the SMs to the
// GEMMs that run beside a load.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include <string>

#include "tp_internal.h"

namespace tp {
namespace {

constexpr int kMaxSegs = 64;
constexpr int64_t kPieceBytes = 4096;
constexpr int kCopyThreads = 256;

struct CopySeg {
  const uint8_t* src;
  uint8_t* dst;
  int64_t rows;
  int64_t row_bytes;
  int64_t src_stride;  // bytes between consecutive rows of the source
  int64_t dst_stride;  // bytes between consecutive rows of the destination
  int64_t pieces;      // pieces per row
  int64_t unit_begin;  // first work unit (row x piece) of this segment
};

struct CopyParams {
  CopySeg seg[kMaxSegs];
  int nseg;
  int64_t total_units;
};

__device__ __forceinline__ uint4 load16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte path: every pointer, stride and row length is a multiple of 16 bytes.
__global__ void __launch_bounds__(kCopyThreads) copy_segments_v16(const __grid_constant__ CopyParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t u = warp; u < p.total_units; u += nwarps) {
    int s = 0;
    while (s + 1 < p.nseg && u >= p.seg[s + 1].unit_begin) ++s;
    const CopySeg& g = p.seg[s];
    const int64_t lu = u - g.unit_begin;
    const int64_t row = lu / g.pieces;
    const int64_t piece = lu - row * g.pieces;
    const int64_t off = piece * kPieceBytes;
    const int64_t nbytes = min(kPieceBytes, g.row_bytes - off);
    const uint4* src = reinterpret_cast<const uint4*>(g.src + row * g.src_stride + off);
    uint4* dst = reinterpret_cast<uint4*>(g.dst + row * g.dst_stride + off);
    const int n = static_cast<int>(nbytes >> 4);  // <= 256 chunks: 8 per lane
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < n) v[j] = load16(src + lane + 32 * j);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < n) dst[lane + 32 * j] = v[j];
  }
}

// 2-byte path for shapes whose rows are not 16-byte multiples (same work split).
__global__ void __launch_bounds__(kCopyThreads) copy_segments_b16(const __grid_constant__ CopyParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t u = warp; u < p.total_units; u += nwarps) {
    int s = 0;
    while (s + 1 < p.nseg && u >= p.seg[s + 1].unit_begin) ++s;
    const CopySeg& g = p.seg[s];
    const int64_t lu = u - g.unit_begin;
    const int64_t row = lu / g.pieces;
    const int64_t piece = lu - row * g.pieces;
    const int64_t off = piece * kPieceBytes;
    const int64_t nbytes = min(kPieceBytes, g.row_bytes - off);
    const uint16_t* src = reinterpret_cast<const uint16_t*>(g.src + row * g.src_stride + off);
    uint16_t* dst = reinterpret_cast<uint16_t*>(g.dst + row * g.dst_stride + off);
    const int n = static_cast<int>(nbytes >> 1);
    for (int i = lane; i < n; i += 32) dst[i] = src[i];
  }
}

struct SegBuilder {
  CopyParams p{};
  bool vec_ok = true;
  bool full() const { return p.nseg == kMaxSegs; }
  void add(const void* src, void* dst, int64_t rows, int64_t row_bytes, int64_t src_stride, int64_t dst_stride) {
    if (rows <= 0 || row_bytes <= 0) return;
    if (rows > 1 && src_stride == row_bytes && dst_stride == row_bytes) {
      // Back-to-back rows on both sides: one long row.
      row_bytes *= rows;
      rows = 1;
    }
    CopySeg& g = p.seg[p.nseg++];
    g.src = static_cast<const uint8_t*>(src);
    g.dst = static_cast<uint8_t*>(dst);
    g.rows = rows;
    g.row_bytes = row_bytes;
    g.src_stride = src_stride;
    g.dst_stride = dst_stride;
    g.pieces = (row_bytes + kPieceBytes - 1) / kPieceBytes;
    g.unit_begin = p.total_units;
    p.total_units += rows * g.pieces;
    if (!aligned16(src) || !aligned16(dst) || (row_bytes & 15) || (rows > 1 && ((src_stride & 15) || (dst_stride & 15))))
      vec_ok = false;
  }
  void reset() {
    p = CopyParams{};
    vec_ok = true;
  }
};

tp_status launch_copy(SegBuilder& b, bool host_src, cudaStream_t stream) {
  if (b.p.total_units == 0) return TP_OK;
  if (host_src) {
    // Page-locked host source: one copy-engine transfer per segment (segment sources are host
    // addresses here).
    for (int i = 0; i < b.p.nseg; ++i) {
      const CopySeg& g = b.p.seg[i];
      const cudaError_t e =
          g.rows == 1 ? cudaMemcpyAsync(g.dst, g.src, static_cast<size_t>(g.row_bytes), cudaMemcpyHostToDevice, stream)
                      : cudaMemcpy2DAsync(g.dst, static_cast<size_t>(g.dst_stride), g.src,
                                          static_cast<size_t>(g.src_stride), static_cast<size_t>(g.row_bytes),
                                          static_cast<size_t>(g.rows), cudaMemcpyHostToDevice, stream);
      if (e != cudaSuccess) return cuda_fail(e, "host-to-device shard copy");
    }
    return TP_OK;
  }
  const int sms = sm_count();
  if (sms <= 0) return fail(TP_ERR_CUDA, "cannot query the SM count of the current device");
  const int64_t warps_needed = b.p.total_units;
  const int64_t blocks_needed = (warps_needed * 32 + kCopyThreads - 1) / kCopyThreads;
  // Up to 8 resident blocks of 256 threads per SM; grid is a multiple of the SM count when large.
  int64_t grid = blocks_needed;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (grid > cap) grid = cap;
  const dim3 g(static_cast<unsigned>(grid)), blk(kCopyThreads);
  cudaError_t e;
  if (b.vec_ok)
    e = launch_pdl(copy_segments_v16, g, blk, 0, stream, b.p);
  else
    e = launch_pdl(copy_segments_b16, g, blk, 0, stream, b.p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "copy kernel launch");
  return TP_OK;
}

// ---------------------------------------------------------------------------
// Reduce: out[i] = bf16_rne(sum_r partials[r][i]), fp32 sum in rank order.
// ---------------------------------------------------------------------------

struct ReduceParams {
  const float* part[TP_MAX_DEGREE];
  __nv_bfloat16* out;
  int64_t n;  // elements
  int p;
};

__global__ void __launch_bounds__(256) reduce_partials_v8(const __grid_constant__ ReduceParams p) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t groups = p.n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += stride) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    // Four ranks' loads are issued before any of their sums, so a thread keeps up to 128 bytes
    // in flight; the sums still run in rank order.
    for (int r0 = 0; r0 < p.p; r0 += 4) {
      float4 a[4], b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (r0 + k < p.p) {
          const float4* src = reinterpret_cast<const float4*>(p.part[r0 + k]) + 2 * g;
          a[k] = __ldcs(src);
          b[k] = __ldcs(src + 1);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (r0 + k < p.p) {
          acc[0] += a[k].x; acc[1] += a[k].y; acc[2] += a[k].z; acc[3] += a[k].w;
          acc[4] += b[k].x; acc[5] += b[k].y; acc[6] += b[k].z; acc[7] += b[k].w;
        }
      }
    }
    __align__(16) __nv_bfloat162 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    reinterpret_cast<uint4*>(p.out)[g] = *reinterpret_cast<const uint4*>(o);
  }
}

// Resident blocks of 256 threads per SM for reduce_partials_v8 (its register count sets it),
// queried once.
int reduce_blocks_per_sm() {
  static std::once_flag once;
  static int blocks = 1;
  std::call_once(once, [] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, reduce_partials_v8, 256, 0) == cudaSuccess && b > 0)
      blocks = b;
    else
      (void)cudaGetLastError();
  });
  return blocks;
}

__global__ void __launch_bounds__(256) reduce_partials_scalar(const __grid_constant__ ReduceParams p, int64_t begin) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n; i += stride) {
    float acc = 0.f;
    for (int r = 0; r < p.p; ++r) acc += p.part[r][i];
    p.out[i] = __float2bfloat16_rn(acc);
  }
}

}  // namespace
}  // namespace tp

namespace tp {
namespace {

// One validated extraction: the source (device memory, or page-locked host memory that the
// copy engines read), the plan's block sizes and the ranks' outputs.
struct ShardJob {
  const uint8_t* src = nullptr;
  bool host_src = false;
  bool empty = true;  // nothing to copy (no ranks, or an empty shard)
  int64_t rows = 0, cols = 0;
  tp_style style = TP_COLWISE;
  int tp_degree = 1, rank_begin = 0, rank_count = 0;
  int64_t sizes[TP_MAX_SPLITS] = {0};
  int n = 0;
  void* const* outs = nullptr;
};

// The plan checks of tp_plan_shard_ranks, in its order (host only, nothing is touched).
tp_status prepare_plan(const void* weight, int64_t rows, int64_t cols, tp_style style, int tp_degree, int rank_begin,
                      int rank_count, const int64_t* fused_splits, int n_splits, int64_t num_heads, int64_t head_dim,
                      void* const* dev_outs, ShardJob* job) {
  if (rank_count < 0) return fail(TP_ERR_INVALID_ARG, "rank_count %d is negative", rank_count);
  if (rank_begin < 0) return fail(TP_ERR_INVALID_ARG, "rank %d is negative", rank_begin);
  // Validate the whole plan (and the first and last rank) before touching any memory.
  tp_status st = validate_plan(rows, cols, style, tp_degree, rank_count > 0 ? rank_begin : -1, num_heads, head_dim,
                               fused_splits, n_splits, job->sizes, &job->n);
  if (st != TP_OK) return st;
  // rank_begin is in [0, tp_degree) here (validate_plan checked it), so the difference cannot overflow.
  if (rank_count > 0 && rank_count > tp_degree - rank_begin)
    return fail(TP_ERR_INVALID_ARG, "ranks [%d, %lld) outside [0, %d)", rank_begin,
                static_cast<long long>(rank_begin) + rank_count, tp_degree);
  job->rows = rows;
  job->cols = cols;
  job->style = style;
  job->tp_degree = tp_degree;
  job->rank_begin = rank_begin;
  job->rank_count = rank_count;
  job->outs = dev_outs;
  job->empty = (rows * cols / tp_degree == 0 || rank_count == 0);
  return TP_OK;
}

// The pointer checks of a job whose plan passed: NULLs, where the source lives, device outputs.
tp_status prepare_pointers(const void* weight, void* const* dev_outs, ShardJob* job) {
  if (job->empty) return TP_OK;
  const int rank_count = job->rank_count;
  if (weight == nullptr || dev_outs == nullptr) return fail(TP_ERR_INVALID_ARG, "weight or dev_outs is NULL");
  for (int i = 0; i < rank_count; ++i)
    if (dev_outs[i] == nullptr) return fail(TP_ERR_INVALID_ARG, "dev_outs[%d] is NULL", i);

  // Where does the source live?  Page-locked host memory is read by the copy engines;
  // pageable host memory is refused rather than staged.
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, weight);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(weight)");
  job->src = static_cast<const uint8_t*>(weight);
  job->host_src = false;
  if (attr.type == cudaMemoryTypeHost) {
    job->host_src = true;
  } else if (attr.type == cudaMemoryTypeUnregistered) {
    return fail(TP_ERR_NOT_PINNED, "weight is pageable host memory; page-lock it (cudaHostAlloc/cudaHostRegister)");
  }
  for (int i = 0; i < rank_count; ++i) {
    cudaPointerAttributes oattr{};
    e = cudaPointerGetAttributes(&oattr, dev_outs[i]);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes(dev_out)");
    if (oattr.type != cudaMemoryTypeDevice && oattr.type != cudaMemoryTypeManaged)
      return fail(TP_ERR_INVALID_ARG, "dev_outs[%d] is not device memory", i);
  }
  return TP_OK;
}

// Add a job's segments to `b` (launching it whenever it fills up).
tp_status append_job(SegBuilder& b, const ShardJob& j, cudaStream_t s) {
  if (j.empty) return TP_OK;
  const int64_t esz = 2;  // bf16
  for (int i = 0; i < j.rank_count; ++i) {
    const int rank = j.rank_begin + i;
    uint8_t* d8 = static_cast<uint8_t*>(j.outs[i]);
    int64_t offset = 0;      // block offset along the sharded dimension
    int64_t out_offset = 0;  // where this block's part starts in the shard
    for (int bi = 0; bi < j.n; ++bi) {
      const int64_t part = j.sizes[bi] / j.tp_degree;
      const int64_t lo = offset + static_cast<int64_t>(rank) * part;
      if (b.full()) {
        tp_status st = launch_copy(b, j.host_src, s);
        if (st != TP_OK) return st;
        b.reset();
      }
      if (j.style == TP_COLWISE) {
        // Rows [lo, lo+part) of W -> rows [out_offset, out_offset+part) of the shard.
        b.add(j.src + lo * j.cols * esz, d8 + out_offset * j.cols * esz, part, j.cols * esz, j.cols * esz,
              j.cols * esz);
      } else {
        // Columns [lo, lo+part) of every row -> columns [out_offset, ...) of the shard.
        const int64_t shard_cols = j.cols / j.tp_degree;
        b.add(j.src + lo * esz, d8 + out_offset * esz, j.rows, part * esz, j.cols * esz, shard_cols * esz);
      }
      offset += j.sizes[bi];
      out_offset += part;
    }
  }
  return TP_OK;
}

}  // namespace
}  // namespace tp

extern "C" {

tp_status tp_plan_shard_ranks(const void* weight, int64_t rows, int64_t cols, tp_style style, int tp_degree,
                              int rank_begin, int rank_count, const int64_t* fused_splits, int n_splits,
                              int64_t num_heads, int64_t head_dim, void* const* dev_outs, tp_stream_t stream) {
  using namespace tp;
  clear_error();
  ShardJob job;
  tp_status st = prepare_plan(weight, rows, cols, style, tp_degree, rank_begin, rank_count, fused_splits, n_splits,
                              num_heads, head_dim, dev_outs, &job);
  if (st == TP_OK) st = prepare_pointers(weight, dev_outs, &job);
  if (st != TP_OK || job.empty) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  SegBuilder b;
  st = append_job(b, job, s);
  if (st != TP_OK) return st;
  return launch_copy(b, job.host_src, s);
}

tp_status tp_plan_shard_many(const tp_shard_request* requests, int n_requests, tp_stream_t stream) {
  using namespace tp;
  clear_error();
  if (n_requests < 0 || n_requests > TP_MAX_SHARD_REQUESTS)
    return fail(n_requests < 0 ? TP_ERR_INVALID_ARG : TP_ERR_UNSUPPORTED, "n_requests=%d outside [0, %d]",
                n_requests, TP_MAX_SHARD_REQUESTS);
  if (n_requests > 0 && requests == nullptr) return fail(TP_ERR_INVALID_ARG, "requests is NULL");
  ShardJob jobs[TP_MAX_SHARD_REQUESTS];
  // Every request's plan first, then every request's pointers: nothing is copied unless all pass.
  for (int pass = 0; pass < 2; ++pass) {
    for (int q = 0; q < n_requests; ++q) {
      const tp_shard_request& r = requests[q];
      tp_status st = pass == 0 ? prepare_plan(r.weight, r.rows, r.cols, r.style, r.tp_degree, r.rank_begin,
                                              r.rank_count, r.fused_splits, r.n_splits, r.num_heads, r.head_dim,
                                              r.dev_outs, &jobs[q])
                               : prepare_pointers(r.weight, r.dev_outs, &jobs[q]);
      if (st != TP_OK) {
        const std::string msg = tp_last_error();
        return fail(st, "request %d: %s", q, msg.c_str());
      }
    }
  }
  // Every check passed: copy, device sources in one launch and host sources in another
  // (more only past 64 segments).
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int kind = 0; kind < 2; ++kind) {
    SegBuilder b;
    bool any = false;
    for (int q = 0; q < n_requests; ++q) {
      if (jobs[q].empty || static_cast<int>(jobs[q].host_src) != kind) continue;
      any = true;
      tp_status st = append_job(b, jobs[q], s);
      if (st != TP_OK) return st;
    }
    if (any) {
      tp_status st = launch_copy(b, kind == 1, s);
      if (st != TP_OK) return st;
    }
  }
  return TP_OK;
}

tp_status tp_plan_shard(const void* weight, int64_t rows, int64_t cols, tp_style style, int tp_degree, int rank,
                        const int64_t* fused_splits, int n_splits, int64_t num_heads, int64_t head_dim, void* dev_out,
                        tp_stream_t stream) {
  using namespace tp;
  if (rank < 0 || rank >= tp_degree) {
    clear_error();
    // Report plan errors first (they do not depend on the rank), then the rank itself.
    int64_t sizes[TP_MAX_SPLITS];
    int n = 0;
    tp_status st = validate_plan(rows, cols, style, tp_degree, -1, num_heads, head_dim, fused_splits, n_splits,
                                 sizes, &n);
    if (st != TP_OK) return st;
    return fail(TP_ERR_INVALID_ARG, "rank %d outside [0, %d)", rank, tp_degree);
  }
  void* outs[1] = {dev_out};
  if (dev_out == nullptr && rows * cols != 0) {
    clear_error();
    int64_t sizes[TP_MAX_SPLITS];
    int n = 0;
    tp_status st = validate_plan(rows, cols, style, tp_degree, rank, num_heads, head_dim, fused_splits, n_splits,
                                 sizes, &n);
    if (st != TP_OK) return st;
    return fail(TP_ERR_INVALID_ARG, "dev_out is NULL");
  }
  return tp_plan_shard_ranks(weight, rows, cols, style, tp_degree, rank, 1, fused_splits, n_splits, num_heads,
                             head_dim, outs, stream);
}

tp_status tp_combine(tp_combine_mode mode, const void* const* partials, int tp_degree, int64_t T, int64_t N_each,
                     void* out, tp_stream_t stream) {
  using namespace tp;
  clear_error();
  if (mode != TP_GATHER && mode != TP_REDUCE) return fail(TP_ERR_INVALID_ARG, "unknown combine mode %d", (int)mode);
  if (tp_degree < 1 || tp_degree > TP_MAX_DEGREE)
    return fail(tp_degree < 1 ? TP_ERR_INVALID_ARG : TP_ERR_UNSUPPORTED, "tp_degree=%d outside [1, %d]", tp_degree,
                TP_MAX_DEGREE);
  if (T < 0 || N_each < 0) return fail(TP_ERR_INVALID_ARG, "negative size");
  if (T == 0 || N_each == 0) return TP_OK;
  if (partials == nullptr || out == nullptr) return fail(TP_ERR_INVALID_ARG, "partials or out is NULL");
  for (int r = 0; r < tp_degree; ++r)
    if (partials[r] == nullptr) return fail(TP_ERR_INVALID_ARG, "partials[%d] is NULL", r);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode == TP_GATHER) {
    SegBuilder b;
    const int64_t row_bytes = N_each * 2;
    for (int r = 0; r < tp_degree; ++r)
      b.add(partials[r], static_cast<uint8_t*>(out) + r * row_bytes, T, row_bytes, row_bytes, row_bytes * tp_degree);
    return launch_copy(b, false, s);
  }
  ReduceParams p{};
  for (int r = 0; r < tp_degree; ++r) p.part[r] = static_cast<const float*>(partials[r]);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.n = T * N_each;
  p.p = tp_degree;
  const int sms = sm_count();
  if (sms <= 0) return fail(TP_ERR_CUDA, "cannot query the SM count of the current device");
  bool vec = aligned16(out);
  for (int r = 0; r < tp_degree; ++r) vec = vec && aligned16(partials[r]);
  int64_t begin = 0;
  if (vec && p.n >= 8) {
    const int64_t groups = p.n >> 3;
    // One wave: as many blocks as the SMs hold at once (the loop strides over the rest).
    int64_t grid = (groups + 255) / 256;
    const int64_t resident = static_cast<int64_t>(sms) * reduce_blocks_per_sm();
    if (grid > resident) grid = resident;
    cudaError_t le = launch_pdl(reduce_partials_v8, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, p);
    if (le != cudaSuccess) return cuda_fail(le, "reduce kernel launch");
    begin = groups << 3;
  }
  if (begin < p.n) {
    int64_t rem = p.n - begin;
    int64_t grid = (rem + 255) / 256;
    if (grid > static_cast<int64_t>(sms) * 8) grid = static_cast<int64_t>(sms) * 8;
    cudaError_t le = launch_pdl(reduce_partials_scalar, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, p, begin);
    if (le != cudaSuccess) return cuda_fail(le, "reduce kernel launch");
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
  return TP_OK;
}

}  // extern "C"
