// Sharded projections on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One persistent kernel runs every rank of a tensor-parallel projection:
//
//   colwise  (tp_linear_colwise): work item = (rank r, m-tile, n-tile),
//            Y_r = act(X . W_r^T + b_r); X is shared by all ranks.
//   rowwise  (tp_linear_rowwise):
//     ACCUM      work item = (m-tile, n-tile); its K loop walks rank 0's
//                [X_0, W_0] slice, then rank 1's, ... accumulating into the
//                same fp32 TMEM accumulator -- the partial sums are joined on
//                chip, in rank order, and written once as bf16.
//     WORKSPACE  work item = (rank, m-tile, n-tile) with the rank varying
//                fastest; each rank writes its fp32 partial tile to the
//                workspace and counts it on an atomic per-tile counter; once
//                all tp_degree partials are in (bounded wait), each rank sums
//                its 1/tp_degree share of the tile's rows in rank order and
//                writes bf16.
//     NONE       work item = (rank, m-tile, n-tile); fp32 partials out.
//
// Two tile shapes share one kernel template:
//   single CTA  128 x 256 output tile per CTA, grid = min(#tiles, #SMs),
//               4-stage ring of A (128 x 64) + B (256 x 64) bf16 boxes;
//   CTA pair    256 x 256 output tile per cluster of two CTAs (used when the
//               output has more than 128 rows): each CTA stages its 128 rows
//               of A and 128 rows of B (3-stage ring, 64 KB per stage), and
//               the even CTA issues cta_group::2 MMAs (M=256) that read both
//               CTAs' shared memory -- half the B traffic per SM of the
//               single-CTA tile, which is shared-memory-bandwidth bound.
// CTA layout (192 threads, one CTA per SM):
//   warp 0      TMA producer, 128-byte swizzled boxes of 64 columns into the
//               ring.  A CTA pair's stage is K = 128, two boxes per operand
//               (eight K=16 MMAs per wait on a full stage: measured 1.3-2.5 %
//               faster than six stages of one box, whose fixed cost per stage
//               showed in the MMA issue); a single CTA's is one box (its two-box
//               stages would leave two of them, 17 % slower at T 128).  Each box
//               has its own empty barrier: it is refilled as soon as its four
//               MMAs are done, so the copy the MMAs next wait on is one box,
//               not a whole stage (measured 4 % on the SwiGLU gate/up GEMM and
//               7 % on a 3-wave out-projection, bit-identical).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (K=16 steps) into
//               one of two TMEM accumulators (2 x 256 columns), so the
//               epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, bias, activation
//               (GELU-tanh or SwiGLU) in fp32, round to bf16, store.
// Chunked accumulation (EPI_BF16_CHUNKED, 320 threads): the MMA warp hands an
// accumulator to the epilogue every 1024 of K, each chunk summed from zero,
// and warps 2..9 (two per TMEM lane quarter, half of the tile's columns each)
// add the chunks into fp32 registers with round-to-nearest (epilogue_chunked).
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); a wait that
// gives up sets a flag in the library's status word and the CTA drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

#include "tp_internal.h"
#include "tp_ptx.cuh"

namespace tp {
namespace {

constexpr int BM = 128;        // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;        // accumulator columns per tile
constexpr int KBOX = 64;       // K per TMA box (one 128-byte swizzle row of bf16)
constexpr int GROUP_M = 16;
constexpr int kTmemCols = 512; // two accumulators of BN columns
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// EPI_BF16_CHUNKED: the K sum is formed on the tensor core in chunks of Cfg::CHUNK_STAGES stages
// (K = 1024), each started from zero in one of the two accumulators, and the epilogue adds the
// chunks in fp32 with round-to-nearest (see epilogue_chunked).  The chunk length is set by the
// epilogue: pulling a chunk's 128 KB out of tensor memory while the tensor core runs takes each
// epilogue warp about 2 us, so a chunk must hold more MMA work than that.  Measured on the
// Q/K/V projection of the block (T 4608, K 6144, 4 x 4608 columns): chunks of K 256 / 512 / 1024 /
// 1536 took 1.51 / 1.14 / 1.09 / 1.10 times the plain launch, and 0.020 / 0.033 / 0.068 /
// 0.100 % of outputs differ from the correctly rounded value (0.35 % plain); one chunk per tile
// takes 1.07 times as long, the cost of the 8-warp epilogue itself.
enum Epi : int { EPI_BF16 = 0, EPI_GELU = 1, EPI_SWIGLU = 2, EPI_F32 = 3, EPI_WS_REDUCE = 4, EPI_BF16_CHUNKED = 5 };

// Epilogue warps: 4 (one per TMEM lane quarter), or 8 for the chunked sum (two per lane quarter,
// each holding the running sums of half of the tile's columns in registers).
__host__ __device__ constexpr int epilogue_warps(int epi) { return epi == EPI_BF16_CHUNKED ? 8 : 4; }
__host__ __device__ constexpr int threads_of(int epi) { return 64 + 32 * epilogue_warps(epi); }

// Tile shape of the single-CTA (kPair = false) and CTA-pair (kPair = true) kernels.
template <bool kPair>
struct Cfg {
  static constexpr int TILE_M = kPair ? 2 * BM : BM;   // output rows per work tile
  static constexpr int B_ROWS = kPair ? BN / 2 : BN;   // B rows each CTA stages
  // K per stage: two boxes per operand for CTA pairs (eight K=16 MMAs per wait on a full stage),
  // one for a single CTA, whose larger B tile leaves room for only two stages of two boxes.
  static constexpr int BK = kPair ? 2 * KBOX : KBOX;
  static constexpr int STAGES = kPair ? 3 : 4;
  static constexpr int CHUNK_STAGES = 1024 / BK;   // EPI_BF16_CHUNKED: stages per chunk (K 1024)
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = B_ROWS * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t A_BOX = BM * KBOX * 2;        // one K box of A
  static constexpr uint32_t B_BOX = B_ROWS * KBOX * 2;    // one K box of B
};

struct GemmParams {
  CUtensorMap map_a[TP_MAX_DEGREE];
  CUtensorMap map_b[TP_MAX_DEGREE];
  CUtensorMap map_out[TP_MAX_DEGREE];        // per output group: 64 x 32 bf16 or 32 x 32 fp32 store boxes
  CUtensorMap map_out_tail[TP_MAX_DEGREE];   // per output group: 32 x 32 bf16 boxes (odd multiples of 32)
  void* out[TP_MAX_DEGREE];                  // per output group
  const __nv_bfloat16* bias[TP_MAX_DEGREE];  // per output group, nullable
  float* ws;                                 // WS_REDUCE: fp32 partials [n_groups][M][N]
  int* counters;                             // WS_REDUCE: one per 128 x 256 output block
  __nv_bfloat16* reduce_out;                 // WS_REDUCE: bf16 [M][ldo]
  const __nv_bfloat16* reduce_bias;          // WS_REDUCE: nullable [N]
  unsigned int* status;
  uint64_t tile_wait_ns;  // WS_REDUCE: bound on the wait for the other ranks' partials of a tile
  int64_t ldo;        // row stride of the outputs, elements
  int M, N;           // output rows; output columns per group
  int n_groups;       // independent outputs (ranks) -- 1 for ACCUM
  int n_ksegs;        // K segments per tile (ranks) -- >1 only for ACCUM
  int kblocks;        // K stages (Cfg::BK wide) per segment
  int m_tiles, n_tiles;
  int bn;             // accumulator columns per tile: a multiple of 32, <= 256 (256 for SwiGLU)
  int n_counters;     // WS_REDUCE: counters per 128-row block (one per n-tile)
  int b_up_row;       // SwiGLU: first row of the up block inside W_r
  int rank_fastest;   // tile order with the rank varying fastest
  int group_m;        // m-tiles per raster group (choose_group_m)
  int a_shared;       // one A map for every rank (colwise)
  int quad;           // 0: CTA pairs alone; 1: clusters of two pairs on n-adjacent tiles sharing A by
                      // multicast (A maps of BM/2 rows); 2: on m-adjacent tiles sharing B (B maps of
                      // a quarter of the tile width)
};

constexpr int kMaxStages = 8;  // stage barriers held in SmemCtrl
static_assert(Cfg<true>::STAGES <= kMaxStages && Cfg<false>::STAGES <= kMaxStages,
              "the control block holds kMaxStages full barriers");
static_assert(Cfg<true>::BK / KBOX <= 2 && Cfg<false>::BK / KBOX <= 2,
              "the control block holds two empty barriers (one per K box) for each stage");

struct alignas(8) SmemCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages * 2];  // [stage * boxes + box]: a box is refilled once its MMAs are done
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int is_last;
};

// Epilogue staging: every epilogue warp owns two 4 KB buffers (a 32 x 32 fp32 or bf16 chunk each),
// written with swizzled 16-byte stores and sent to global memory by TMA stores.
constexpr uint32_t kStageBuf = 4096;
constexpr uint32_t kStagingBytes = 4 /*warps*/ * 2 * kStageBuf;

template <bool kPair>
constexpr size_t smem_bytes() {
  return 1024 /*alignment slack*/ + Cfg<kPair>::STAGES * Cfg<kPair>::STAGE_BYTES + kStagingBytes + sizeof(SmemCtrl);
}

// (With a multicast launch a work item is two adjacent tiles: the tile counts are then counts of
// such items along the paired dimension, and mb or nb the item's index.)
__device__ __forceinline__ void decode_tile(const GemmParams& p, int t, int& g, int& mb, int& nb,
                                            int n_tiles_override = 0, int m_tiles_override = 0,
                                            int group_m_override = 0) {
  const int n_tiles = n_tiles_override > 0 ? n_tiles_override : p.n_tiles;
  const int m_tiles = m_tiles_override > 0 ? m_tiles_override : p.m_tiles;
  const int group_m = group_m_override > 0 ? group_m_override : p.group_m;
  const int tiles_mn = m_tiles * n_tiles;
  int mn;
  if (p.rank_fastest) {
    // The ranks of one (m, n) tile are consecutive work items, so they run at the
    // same time on different CTAs and their partials meet in L2.  The rank is
    // rotated by the tile index so that a persistent CTA does not get the same
    // rank on every tile (with #CTAs a multiple of tp_degree it would).
    mn = t / p.n_groups;
    g = (t + mn) % p.n_groups;
  } else {
    g = t / tiles_mn;
    mn = t - g * tiles_mn;
  }
  // Grouped raster: group_m m-tiles sweep the n-tiles together so the CTAs
  // running at the same time share A and B tiles through L2.
  const int span = group_m * n_tiles;
  const int sr = mn / span;
  const int first_m = sr * group_m;
  const int gm = min(m_tiles - first_m, group_m);
  const int in = mn - sr * span;
  mb = first_m + in % gm;
  nb = in / gm;
}

// Bounded wait: true when the phase completed; false when this CTA is aborting
// (another role gave up) or the wait itself ran out of time.
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* status, bool ignore_abort) {
  auto probe = [&]() {
    return kClusterScope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (probe()) return true;
    if ((i & 63u) == 0) {
      if (!ignore_abort && *abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(status, TP_DEVSTATUS_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait until *ctr >= target (a tile counter other CTAs increment); false on abort or
// timeout.  The bound is the caller's (tp_set_tile_wait_limit_ns), read at launch.
__device__ __noinline__ bool wait_counter(const int* ctr, int target, volatile int* abort_flag, unsigned int* status,
                                          uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(status, TP_DEVSTATUS_TIMEOUT);
      return false;
    }
    __nanosleep(100);
  }
}

// GELU with the tanh approximation, 0.5 x (1 + tanh(u)) with u = sqrt(2/pi) (x + 0.044715 x^3),
// evaluated as x / (1 + e^(-2u)): the same function (1 + tanh(u) = 2 / (1 + e^(-2u))), one fast
// exponential and one fast division (a reciprocal and a product) instead of a full tanh.  With
// the correctly rounded division instead, a 64-token GELU launch ran 2.8x slower than with tanh.
// Large negative u gives x * (1 / inf) = 0, large positive u gives x / 1 = x.
__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  const float u = k0 * (x + k1 * x * x * x);
  return __fdividef(x, 1.0f + __expf(-2.0f * u));
}
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Two fp32 values in one 64-bit register for the paired fp32 instructions of sm_100 and later.
__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack_f2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// silu(g) * u for two columns, g / (1 + e^-g) * u with e^-g = 2^(-g log2(e)): the exponential
// and the reciprocal on the special-function unit, the products and the sum two at a time (the
// epilogue warp of TMEM lane quarter 1 shares its issue slots with the MMA thread; measured:
// the SwiGLU gate/up launch 0.7 % shorter than with the scalar forms, bit-identical).
__device__ __forceinline__ void swiglu_pair(float g0, float g1, float u0, float u1, float& y0, float& y1) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  const uint64_t g2 = pack_f2(g0, g1);
  float t0, t1;
  unpack_f2(mul_f2(g2, pack_f2(kNegLog2e, kNegLog2e)), t0, t1);
  float d0, d1;
  unpack_f2(add_f2(pack_f2(ex2_approx(t0), ex2_approx(t1)), pack_f2(1.0f, 1.0f)), d0, d1);
  unpack_f2(mul_f2(mul_f2(g2, pack_f2(rcp_approx(d0), rcp_approx(d1))), pack_f2(u0, u1)), y0, y1);
}

// Epilogue output path.  A warp drains its 32 rows (one row per lane) in chunks:
// 64 bf16 columns or 32 fp32 columns (128-byte rows, 4 KB per chunk), plus a
// 32-column bf16 chunk for a tile width that is an odd multiple of 32.  A chunk is
// written to one of the warp's two shared-memory buffers with 16-byte stores in
// the tensor map's swizzled order -- 128-byte swizzle: 16-byte piece j of row r
// sits in slot j ^ (r & 7); 64-byte swizzle (32 bf16 columns): slot j ^ ((r >> 1) & 3)
// -- so the 32 lanes hit all banks, and then sent to global memory by one TMA store
// (rows and columns outside the output are clipped).  A buffer is reused only after
// its previous store has finished reading it.
__device__ __forceinline__ uint32_t stage_buffer(uint32_t wbuf, int nchunk, int lane, bool single = false) {
  if (single) {  // one buffer: the previous store must have finished reading it
    if (nchunk >= 1) {
      if (lane == 0) ptx::bulk_wait_read_0();
      __syncwarp();
    }
    return wbuf;
  }
  const uint32_t buf = wbuf + static_cast<uint32_t>(nchunk & 1) * kStageBuf;
  if (nchunk >= 2) {
    if (lane == 0) ptx::bulk_wait_read_1();
    __syncwarp();
  }
  return buf;
}

__device__ __forceinline__ void stage_issue(const CUtensorMap* map, uint32_t buf, int& nchunk, int lane, int x,
                                            int y) {
  ptx::fence_proxy_async_smem();  // make the generic-proxy writes visible to the TMA engine
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(map, buf, x, y);
    ptx::bulk_commit();
  }
  ++nchunk;
}

__device__ __forceinline__ void pack_bf16x32(const float (&f)[32], uint32_t (&packed)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    packed[j] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// fp32: 32 columns.
__device__ __forceinline__ void stage_store_f32(const CUtensorMap* map, uint32_t wbuf, int& nchunk, int lane,
                                                const float (&f)[32], int x, int y) {
  const uint32_t buf = stage_buffer(wbuf, nchunk, lane);
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    ptx::st_shared_v4(row + (static_cast<uint32_t>(j ^ (lane & 7)) << 4), __float_as_uint(f[4 * j]),
                      __float_as_uint(f[4 * j + 1]), __float_as_uint(f[4 * j + 2]), __float_as_uint(f[4 * j + 3]));
  stage_issue(map, buf, nchunk, lane, x, y);
}

// bf16: 64 columns given as two halves of 32.
__device__ __forceinline__ void stage_store_bf16x64(const CUtensorMap* map, uint32_t wbuf, int& nchunk, int lane,
                                                    const float (&lo)[32], const float (&hi)[32], int x, int y,
                                                    bool single = false) {
  const uint32_t buf = stage_buffer(wbuf, nchunk, lane, single);
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 128;
  uint32_t packed[16];
  pack_bf16x32(lo, packed);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::st_shared_v4(row + (static_cast<uint32_t>(j ^ (lane & 7)) << 4), packed[4 * j], packed[4 * j + 1],
                      packed[4 * j + 2], packed[4 * j + 3]);
  pack_bf16x32(hi, packed);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::st_shared_v4(row + (static_cast<uint32_t>((4 + j) ^ (lane & 7)) << 4), packed[4 * j], packed[4 * j + 1],
                      packed[4 * j + 2], packed[4 * j + 3]);
  stage_issue(map, buf, nchunk, lane, x, y);
}

// bf16: 32 columns (the last chunk of a tile whose width is an odd multiple of 32).
__device__ __forceinline__ void stage_store_bf16x32(const CUtensorMap* map, uint32_t wbuf, int& nchunk, int lane,
                                                    const float (&f)[32], int x, int y, bool single = false) {
  const uint32_t buf = stage_buffer(wbuf, nchunk, lane, single);
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 64;
  uint32_t packed[16];
  pack_bf16x32(f, packed);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::st_shared_v4(row + (static_cast<uint32_t>(j ^ ((lane >> 1) & 3)) << 4), packed[4 * j], packed[4 * j + 1],
                      packed[4 * j + 2], packed[4 * j + 3]);
  stage_issue(map, buf, nchunk, lane, x, y);
}

// bf16, 64 columns of a warp tile that lies wholly inside the output, by plain stores: the chunk
// is staged in the warp's buffer (the same 128-byte swizzled rows as for a TMA store), then read
// back four rows at a time, so that each warp store writes four whole 128-byte row pieces.  The
// operand copies the GEMM waits on share the TMA engine with its stores; these stores do not use
// it (a test build writing every tile this way made the SwiGLU gate/up launch about 1 % shorter,
// bit-identical).  A TMA store of an earlier, ragged tile may still be reading a staging buffer:
// that is waited for first.
__device__ __forceinline__ void stage_store_bf16x64_plain(__nv_bfloat16* out, int64_t ldo, uint32_t wbuf, int& nchunk,
                                                          int lane, const float (&lo)[32], const float (&hi)[32], int x,
                                                          int y) {
  if (lane == 0) ptx::bulk_wait_read_0();
  __syncwarp();
  const uint32_t buf = wbuf + static_cast<uint32_t>(nchunk & 1) * kStageBuf;
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 128;
  uint32_t packed[16];
  pack_bf16x32(lo, packed);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::st_shared_v4(row + (static_cast<uint32_t>(j ^ (lane & 7)) << 4), packed[4 * j], packed[4 * j + 1],
                      packed[4 * j + 2], packed[4 * j + 3]);
  pack_bf16x32(hi, packed);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    ptx::st_shared_v4(row + (static_cast<uint32_t>((4 + j) ^ (lane & 7)) << 4), packed[4 * j], packed[4 * j + 1],
                      packed[4 * j + 2], packed[4 * j + 3]);
  __syncwarp();
  const int piece = lane & 7;  // 16-byte piece of a row: 8 columns
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    uint32_t v0, v1, v2, v3;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                 : "r"(buf + static_cast<uint32_t>(r) * 128 + (static_cast<uint32_t>(piece ^ (r & 7)) << 4)));
    *reinterpret_cast<uint4*>(out + static_cast<int64_t>(y + r) * ldo + x + piece * 8) = make_uint4(v0, v1, v2, v3);
  }
  __syncwarp();  // every lane has read the buffer before any lane stages into it again
  ++nchunk;
}

// One accumulator tile: 128 rows (this CTA's TMEM lanes) x p.bn columns; this warp drains
// its 32 rows [row0, row0 + 32), one row per lane, 32 columns at a time.
// `release` is called once, right after the last TMEM read, to hand the accumulator back to
// the MMA warp.  Out-of-range rows and columns are clipped by the TMA stores.
template <int kEpi, typename Release>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, SmemCtrl* ctl, uint32_t taddr, uint32_t wbuf,
                                              int& nchunk, int g, int row0, int mb128, int nb, int lane, int epi_tid,
                                              Release release) {
  const CUtensorMap* omap = &p.map_out[g];
  if constexpr (kEpi == EPI_SWIGLU) {
    const __nv_bfloat16* bias = p.bias[g];
    const int n_out = p.N, up_row = p.b_up_row;
    auto swiglu32 = [&](const uint32_t (&gv)[32], const uint32_t (&uv)[32], int col0, float (&f)[32]) {
      if (bias == nullptr) {  // warp-uniform: no per-element test on the common path
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          swiglu_pair(__uint_as_float(gv[j]), __uint_as_float(gv[j + 1]), __uint_as_float(uv[j]),
                      __uint_as_float(uv[j + 1]), f[j], f[j + 1]);
        return;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int col = col0 + j;
        float gg = __uint_as_float(gv[j]);
        float uu = __uint_as_float(uv[j]);
        if (col < n_out) {
          gg += __bfloat162float(bias[col]);
          uu += __bfloat162float(bias[up_row + col]);
        }
        f[j] = silu_f(gg) * uu;
      }
    };
    // This warp's 32 rows x BN/2 output columns: wholly inside the output -> plain stores,
    // else TMA stores (which clip the rows and columns past the output).
    const bool plain = (row0 + 32 <= p.M) && (nb * (BN / 2) + BN / 2 <= p.N);
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 64) {
      const int col0 = nb * (BN / 2) + c;
      float lo[32], hi[32];
      {
        uint32_t gv[32], uv[32];
        ptx::tmem_ld_32x32b_x32(taddr + c, gv);
        ptx::tmem_ld_32x32b_x32(taddr + BN / 2 + c, uv);
        ptx::tmem_ld_wait();
        swiglu32(gv, uv, col0, lo);
      }
      {
        uint32_t gv[32], uv[32];
        ptx::tmem_ld_32x32b_x32(taddr + c + 32, gv);
        ptx::tmem_ld_32x32b_x32(taddr + BN / 2 + c + 32, uv);
        ptx::tmem_ld_wait();
        if (c + 64 >= BN / 2) release();
        swiglu32(gv, uv, col0 + 32, hi);
      }
      if (plain)
        stage_store_bf16x64_plain(static_cast<__nv_bfloat16*>(p.out[g]), p.ldo, wbuf, nchunk, lane, lo, hi, col0,
                                  row0);
      else if (col0 < p.N)
        stage_store_bf16x64(omap, wbuf, nchunk, lane, lo, hi, col0, row0);
    }
  } else if constexpr (kEpi == EPI_BF16 || kEpi == EPI_GELU) {
    const __nv_bfloat16* bias = p.bias[g];
    const int n_out = p.N;
    auto act32 = [&](const uint32_t (&v)[32], int col0, float (&f)[32]) {
      if (bias == nullptr) {  // warp-uniform: no per-element test on the common path
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = __uint_as_float(v[j]);
          f[j] = (kEpi == EPI_GELU) ? gelu_tanh_f(x) : x;
        }
        return;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float x = __uint_as_float(v[j]);
        if (col0 + j < n_out) x += __bfloat162float(bias[col0 + j]);
        f[j] = (kEpi == EPI_GELU) ? gelu_tanh_f(x) : x;
      }
    };
#pragma unroll 1
    for (int c = 0; c < p.bn; c += 64) {
      const int col0 = nb * p.bn + c;
      const bool pair64 = c + 64 <= p.bn;
      float lo[32], hi[32];
      {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c, v);
        ptx::tmem_ld_wait();
        if (!pair64) release();
        act32(v, col0, lo);
      }
      if (pair64) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + c + 32, v);
        ptx::tmem_ld_wait();
        if (c + 64 >= p.bn) release();
        act32(v, col0 + 32, hi);
        if (col0 < p.N) stage_store_bf16x64(omap, wbuf, nchunk, lane, lo, hi, col0, row0);
      } else if (col0 < p.N) {
        stage_store_bf16x32(&p.map_out_tail[g], wbuf, nchunk, lane, lo, col0, row0);
      }
    }
  } else {
    // fp32 partial tile: to the caller's buffer (EPI_F32) or this rank's workspace plane (EPI_WS_REDUCE).
    const __nv_bfloat16* bias = (kEpi == EPI_F32) ? p.bias[g] : nullptr;
#pragma unroll 1
    for (int c = 0; c < p.bn; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(taddr + c, v);
      ptx::tmem_ld_wait();
      if (c + 32 >= p.bn) release();
      const int col0 = nb * p.bn + c;
      if (col0 < p.N) {
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        if (bias != nullptr) {  // warp-uniform
          const int n_out = p.N;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < n_out) f[j] += __bfloat162float(bias[col0 + j]);
        }
        stage_store_f32(omap, wbuf, nchunk, lane, f, col0, row0);
      }
    }
    if constexpr (kEpi == EPI_WS_REDUCE) {
      // Publish this rank's partial of the 128-row block, count it, wait until every
      // rank's partial is in, then sum this rank's 1/tp_degree share of the block's rows
      // (all partials, in rank order).  Every CTA of the tile sums an equal share, so no
      // CTA is left with all the sums; the launch is cooperative, so the CTAs that wait
      // on each other are resident together, and the wait is bounded.
      if (mb128 * BM < p.M) {
        if (lane == 0) {
          ptx::bulk_wait_all();             // this warp's partial stores are complete ...
          ptx::fence_proxy_async_global();  // ... and ordered before what follows
        }
        __syncwarp();
        __threadfence();
        ptx::named_bar_sync(1, 128);
        int* ctr = &p.counters[mb128 * p.n_counters + nb];
        if (epi_tid == 0) {
          atomicAdd(ctr, 1);
          const bool ready =
              wait_counter(ctr, p.n_groups, reinterpret_cast<volatile int*>(&ctl->abort), p.status, p.tile_wait_ns);
          *reinterpret_cast<volatile int*>(&ctl->is_last) = ready ? 1 : 0;
        }
        ptx::named_bar_sync(1, 128);
        if (*reinterpret_cast<volatile int*>(&ctl->is_last) != 0) {
          __threadfence();
          const int block0 = mb128 * BM;
          const int rows = min(BM, p.M - block0);
          const int lo = block0 + g * rows / p.n_groups;
          const int hi = block0 + (g + 1) * rows / p.n_groups;
          const int col = nb * p.bn + lane * 8;
          const bool col_ok = lane * 8 < p.bn && col < p.N;
          const int64_t plane = static_cast<int64_t>(p.M) * p.N;
          const int warp_e = epi_tid >> 5;
#pragma unroll 1
          for (int row = lo + warp_e; row < hi; row += 8) {
            // Two rows per pass (row and row + 4), every rank's loads in flight before the adds.
            const bool ok1 = row + 4 < hi;
            float a8[2][8];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int j = 0; j < 8; ++j) a8[u][j] = 0.f;
            if (col_ok) {
              const float* src0 = p.ws + static_cast<int64_t>(row) * p.N + col;
              const float* src1 = src0 + 4 * static_cast<int64_t>(p.N);
#pragma unroll 1
              for (int r0 = 0; r0 < p.n_groups; r0 += 4) {
                float4 v[4][2][2];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  if (r0 + u < p.n_groups) {
                    const float4* s0 = reinterpret_cast<const float4*>(src0 + (r0 + u) * plane);
                    v[u][0][0] = __ldcg(s0);
                    v[u][0][1] = __ldcg(s0 + 1);
                    if (ok1) {
                      const float4* s1 = reinterpret_cast<const float4*>(src1 + (r0 + u) * plane);
                      v[u][1][0] = __ldcg(s1);
                      v[u][1][1] = __ldcg(s1 + 1);
                    }
                  }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  if (r0 + u < p.n_groups) {
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                      if (w == 1 && !ok1) continue;
                      a8[w][0] += v[u][w][0].x; a8[w][1] += v[u][w][0].y;
                      a8[w][2] += v[u][w][0].z; a8[w][3] += v[u][w][0].w;
                      a8[w][4] += v[u][w][1].x; a8[w][5] += v[u][w][1].y;
                      a8[w][6] += v[u][w][1].z; a8[w][7] += v[u][w][1].w;
                    }
                  }
                }
              }
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                if (w == 1 && !ok1) continue;
                if (p.reduce_bias != nullptr) {
#pragma unroll
                  for (int j = 0; j < 8; ++j) a8[w][j] += __bfloat162float(p.reduce_bias[col + j]);
                }
                uint32_t pk[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  __nv_bfloat162 h = __floats2bfloat162_rn(a8[w][2 * j], a8[w][2 * j + 1]);
                  pk[j] = *reinterpret_cast<uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(p.reduce_out + static_cast<int64_t>(row + 4 * w) * p.ldo + col) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
        }
      }
    }
  }
}

// Epilogue of EPI_BF16_CHUNKED: 8 warps, warp w (2..9) reading TMEM lane quarter w % 4 and
// owning column half (w - 2) / 4 of the tile (p.bn / 2 = 64, 96 or 128 columns).  Each chunk of
// Cfg::CHUNK_STAGES stages arrives in one of the two accumulators, summed on the tensor core from
// zero; the warp adds it to its running sums (fp32, round to nearest) and releases the
// accumulator at once, so the MMA warp runs one chunk ahead.  After a tile's last chunk the sums
// get the bias, are rounded to bf16 and stored (one 4 KB staging buffer per warp).
//
// Why: the tensor core adds each K=16 step into the fp32 accumulator without rounding to
// nearest, so over K = 6144 the sum drifts (measured on the GB300: 0.35 % of bf16 outputs round
// to the other neighbour of the exact value, against 0.02 % for a round-to-nearest fp32 sum);
// sums of K = 1024 started from zero and added with round-to-nearest bring it to 0.07 %.
template <bool kPair, bool kQuad>
__device__ __forceinline__ void epilogue_chunked(const GemmParams& p, SmemCtrl* ctl, uint8_t* staging, uint32_t tmem,
                                                 int warp, int lane, int unit, int nunits, int total, int n_items,
                                                 int m_items, int gm_items, int quad, uint32_t pq, uint32_t cta,
                                                 uint32_t leader) {
  using C = Cfg<kPair>;
  volatile int* abort_flag = &ctl->abort;
  const int q = warp & 3;            // TMEM lane quarter this warp may read
  const int h = (warp - 2) >> 2;     // column half of the tile
  const int half = p.bn / 2;
  const uint32_t wbuf = ptx::smem_addr(staging) + static_cast<uint32_t>(warp - 2) * kStageBuf;
  const int nchunks = (p.n_ksegs * p.kblocks + C::CHUNK_STAGES - 1) / C::CHUNK_STAGES;
  int nstore = 0;
  uint32_t ccount = 0;
  bool ok = true;
  for (int t = unit; t < total && ok; t += nunits) {
    int g, mb, nb;
    decode_tile(p, t, g, mb, nb, n_items, m_items, gm_items);
    if (quad == 1) nb = 2 * nb + static_cast<int>(pq);
    if (quad == 2) mb = 2 * mb + static_cast<int>(pq);
    float sum[128];
    for (int c = 0; c < nchunks; ++c, ++ccount) {
      const uint32_t acc = ccount & 1u;
      // Warp-uniform outcome: the TMEM loads below are warp-collective.
      if (!__all_sync(0xffffffffu, wait_bounded(ptx::smem_addr(&ctl->tfull[acc]), (ccount >> 1) & 1u, abort_flag,
                                                p.status, false))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * static_cast<uint32_t>(p.bn) +
                             static_cast<uint32_t>(h * half);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (16 * j < half) {  // warp-uniform
          uint32_t v[16];
          ptx::tmem_ld_32x32b_x16(taddr + 16 * j, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            sum[16 * j + i] = (c == 0) ? __uint_as_float(v[i]) : sum[16 * j + i] + __uint_as_float(v[i]);
        }
      }
      ptx::tc_fence_before();
      const uint32_t tempty = ptx::smem_addr(&ctl->tempty[acc]);
      if constexpr (kPair)
        ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty, leader));  // the leader's MMA warp owns the accumulator
      else
        ptx::mbar_arrive(tempty);
    }
    if (!ok) break;
    const int mb128 = mb * (C::TILE_M / BM) + static_cast<int>(cta);
    const int row0 = mb128 * BM + q * 32;
    const __nv_bfloat16* bias = p.bias[g];
    const int colh = nb * p.bn + h * half;   // first output column of this warp's half
    if (bias != nullptr) {  // warp-uniform
#pragma unroll
      for (int i = 0; i < 128; ++i)
        if (i < half && colh + i < p.N) sum[i] += __bfloat162float(bias[colh + i]);
    }
    // Stored straight from the sums: 64 columns (two halves of 32), or 32 for a 96-column half.
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const int col0 = colh + 32 * j;
      if (32 * j >= half || col0 >= p.N) break;
      const float(&lo)[32] = *reinterpret_cast<const float(*)[32]>(&sum[32 * j]);
      const float(&hi)[32] = *reinterpret_cast<const float(*)[32]>(&sum[32 * j + 32]);
      if (32 * j + 64 <= half)
        stage_store_bf16x64(&p.map_out[g], wbuf, nstore, lane, lo, hi, col0, row0, true);
      else
        stage_store_bf16x32(&p.map_out_tail[g], wbuf, nstore, lane, lo, col0, row0, true);
    }
  }
  if (lane == 0) ptx::bulk_wait_all();  // every output store of this warp has landed
}

// kPair = false: one CTA per 128 x 256 tile.  kPair = true: a cluster of two
// CTAs per 256 x 256 tile -- each CTA stages its own 128 rows of A and half of
// B, the even CTA issues cta_group::2 MMAs that read both CTAs' shared memory
// and write both CTAs' tensor memory, and each CTA's epilogue drains its own
// 128 rows.
// kQuad (with kPair): clusters of two CTA pairs that work on n-adjacent tiles of the same 256
// rows, so their A tiles are the same: each CTA loads half of its A rows and multicasts them to
// the CTA in the same position of the other pair, halving the A traffic from L2.  A box of
// either pair is then written by both pairs' producers, so it is free again only once both
// pairs' MMAs are done with it (two arrivals on every box's empty barrier).
template <int kEpi, bool kPair, bool kQuad = false>
__global__ void __launch_bounds__(threads_of(kEpi), 1) tp_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<kPair>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = base + C::STAGES * C::STAGE_BYTES;
  SmemCtrl* ctl = reinterpret_cast<SmemCtrl*>(staging + kStagingBytes);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  static_assert(kPair || !kQuad, "multicast clusters are made of CTA pairs");
  const uint32_t crank = kPair ? ptx::cluster_ctarank() : 0u;
  const uint32_t cta = crank & 1u;              // 0 = leader of the pair
  const uint32_t pq = kQuad ? crank >> 1 : 0u;  // which pair of the cluster
  const uint32_t leader = crank & ~1u;          // cluster rank of this pair's leader
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (2 * pq));
  constexpr int kCtasPerUnit = kQuad ? 4 : (kPair ? 2 : 1);
  const int unit = static_cast<int>(blockIdx.x) / kCtasPerUnit;
  const int nunits = static_cast<int>(gridDim.x) / kCtasPerUnit;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    // Pull every tensor map this launch uses into the TMA descriptor cache while the
    // prologue runs (the maps are launch parameters, not the previous kernel's output), so
    // neither the first copy nor a switch of rank inside a tile waits on a descriptor fetch.
    const int nmaps = (p.n_ksegs > 1) ? p.n_ksegs : p.n_groups;
    for (int r = 0; r < nmaps; ++r) {
      ptx::prefetch_tensormap(&p.map_b[r]);
      if (!p.a_shared || r == 0) ptx::prefetch_tensormap(&p.map_a[r]);
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl->full[s]), 1);
      for (int bx = 0; bx < C::BK / KBOX; ++bx)
        ptx::mbar_init(ptx::smem_addr(&ctl->empty[s * (C::BK / KBOX) + bx]), kQuad ? 2 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&ctl->tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->tempty[a]), (kPair ? 2 : 1) * 32 * epilogue_warps(kEpi));
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ctl->abort = 0;
    ctl->is_last = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    if constexpr (kPair) {
      ptx::tmem_alloc_pair(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if constexpr (kPair) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_wait();  // the previous kernel's writes (operands, output buffers) are complete from here on

  // Work items: tiles, or (kQuad) two adjacent tiles, one per pair: n-adjacent (quad 1, A shared)
  // or m-adjacent (quad 2, B shared).  The host pairs along a dimension with an even tile count.
  const int quad = kQuad ? p.quad : 0;
  const int n_items = quad == 1 ? p.n_tiles / 2 : p.n_tiles;
  const int m_items = quad == 2 ? p.m_tiles / 2 : p.m_tiles;
  const int gm_items = quad == 2 ? (p.group_m + 1) / 2 : p.group_m;
  const int total = p.n_groups * m_items * n_items;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t it = 0;
      bool ok = true;
      for (int t = unit; t < total && ok; t += nunits) {
        int g, mb, nb;
        decode_tile(p, t, g, mb, nb, n_items, m_items, gm_items);
        if (quad == 1) nb = 2 * nb + static_cast<int>(pq);
        if (quad == 2) mb = 2 * mb + static_cast<int>(pq);
        const int a_row = mb * C::TILE_M + static_cast<int>(cta) * BM;
        for (int seg = 0; seg < p.n_ksegs && ok; ++seg) {
          const int r = (p.n_ksegs > 1) ? seg : g;
          const CUtensorMap* ma = &p.map_a[p.a_shared ? 0 : r];
          const CUtensorMap* mbm = &p.map_b[r];
          for (int kb = 0; kb < p.kblocks; ++kb) {
            const uint32_t s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1u;
            const uint32_t full = ptx::smem_addr(&ctl->full[s]);
            const uint32_t sa = ptx::smem_addr(base + s * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
            for (int bx = 0; bx < C::BK / KBOX; ++bx) {
              // Each box is free again once the MMAs that read it are done.
              if (!wait_bounded(ptx::smem_addr(&ctl->empty[s * (C::BK / KBOX) + bx]), ph ^ 1u, abort_flag, p.status,
                                false)) {
                ok = false;
                break;
              }
              const int kx = kb * C::BK + bx * KBOX;
              if constexpr (kPair) {
                // Both CTAs' copies complete on the leader's barrier; the leader expects all of them.
                const uint32_t full_leader = ptx::mapa_shared(full, leader);
                if (cta == 0 && bx == 0)
                  ptx::mbar_arrive_expect_tx(full, 2 * C::A_BYTES + static_cast<uint32_t>(p.bn) * (C::BK * 2));
                // quad: half of this CTA's shared operand rows, to the same position in both pairs.
                const uint16_t qmask = static_cast<uint16_t>((1u << cta) | (1u << (2 + cta)));
                if (quad == 1)
                  ptx::tma_load_2d_pair_mc(sa + bx * C::A_BOX + pq * (C::A_BOX / 2), ma, full_leader, kx,
                                           a_row + static_cast<int>(pq) * (BM / 2), qmask);
                else
                  ptx::tma_load_2d_pair(sa + bx * C::A_BOX, ma, full_leader, kx, a_row);
                int b_row;
                if (kEpi == EPI_SWIGLU)
                  b_row = (cta == 0 ? 0 : p.b_up_row) + nb * (BN / 2);  // leader: gate rows, peer: up rows
                else
                  b_row = nb * p.bn + static_cast<int>(cta) * (p.bn / 2);
                if (quad == 2) {
                  const int half = ((kEpi == EPI_SWIGLU) ? BN : p.bn) / 4;  // rows of each pair's part
                  ptx::tma_load_2d_pair_mc(sb + bx * C::B_BOX + pq * static_cast<uint32_t>(half * KBOX * 2), mbm,
                                           full_leader, kx, b_row + static_cast<int>(pq) * half, qmask);
                } else {
                  ptx::tma_load_2d_pair(sb + bx * C::B_BOX, mbm, full_leader, kx, b_row);
                }
              } else {
                if (bx == 0) ptx::mbar_arrive_expect_tx(full, C::A_BYTES + static_cast<uint32_t>(p.bn) * (C::BK * 2));
                ptx::tma_load_2d(sa + bx * C::A_BOX, ma, full, kx, a_row);
                if (kEpi == EPI_SWIGLU) {
                  ptx::tma_load_2d(sb + bx * C::B_BOX, mbm, full, kx, nb * (BN / 2));
                  ptx::tma_load_2d(sb + bx * C::B_BOX + C::B_BOX / 2, mbm, full, kx, p.b_up_row + nb * (BN / 2));
                } else {
                  ptx::tma_load_2d(sb + bx * C::B_BOX, mbm, full, kx, nb * p.bn);
                }
              }
            }
            if (!ok) break;
            ++it;
          }
        }
      }
      // Let every copy this thread issued land before the CTA can exit.  In a
      // pair, the leader's full barriers count both CTAs' copies.
      if (!kPair || cta == 0) {
        const uint32_t first = it > C::STAGES ? it - C::STAGES : 0;
        for (uint32_t j = first; j < it; ++j)
          wait_bounded(ptx::smem_addr(&ctl->full[j % C::STAGES]), (j / C::STAGES) & 1u, abort_flag, p.status, true);
      } else if (*abort_flag) {
        // The peer cannot observe its own copies; give any in flight time to land (abort path only).
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && cta == 0) {
      // ------------------------------------------------------------ MMA issuer (leader CTA)
      const uint32_t idesc = ptx::idesc_bf16_f32(C::TILE_M, p.bn);
      // An accumulator is taken (wait until the epilogue has released it) and handed to the
      // epilogue (commit) once per tile -- or, for EPI_BF16_CHUNKED, once per chunk of
      // Cfg::CHUNK_STAGES stages (K 1024), each chunk summed from zero; the two accumulators alternate.
      uint32_t it = 0, ccount = 0;
      uint32_t acc = 0, accumulate = 0, d_tmem = tmem;
      bool ok = true;
      auto take = [&]() -> bool {
        acc = ccount & 1u;
        if (!wait_bounded<kPair>(ptx::smem_addr(&ctl->tempty[acc]), ((ccount >> 1) & 1u) ^ 1u, abort_flag, p.status,
                                 false))
          return false;
        ptx::tc_fence_after();
        d_tmem = tmem + acc * static_cast<uint32_t>(p.bn);
        accumulate = 0;
        return true;
      };
      auto hand_over = [&]() {
        if constexpr (kPair)
          ptx::umma_commit_pair(ptx::smem_addr(&ctl->tfull[acc]), pair_mask);
        else
          ptx::umma_commit(ptx::smem_addr(&ctl->tfull[acc]));
        ++ccount;
      };
      for (int t = unit; t < total && ok; t += nunits) {
        if (!take()) break;
        int kdone = 0;
        for (int seg = 0; seg < p.n_ksegs && ok; ++seg) {
          for (int kb = 0; kb < p.kblocks; ++kb, ++kdone) {
            if (kEpi == EPI_BF16_CHUNKED && kdone > 0 && kdone % C::CHUNK_STAGES == 0) {
              hand_over();
              if (!take()) {
                ok = false;
                break;
              }
            }
            const uint32_t s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1u;
            if (!wait_bounded(ptx::smem_addr(&ctl->full[s]), ph, abort_flag, p.status, false)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_addr(base + s * C::STAGE_BYTES);
#pragma unroll
            for (int k = 0; k < C::BK / 16; ++k) {
              // Box k / 4 of each operand; +32 bytes along K inside its 128-byte swizzled row = +2
              // in the >>4 address field.
              const uint64_t adesc = ptx::sw128_kmajor_desc(sa + (k >> 2) * C::A_BOX) + 2u * (k & 3);
              const uint64_t bdesc = ptx::sw128_kmajor_desc(sa + C::A_BYTES + (k >> 2) * C::B_BOX) + 2u * (k & 3);
              if constexpr (kPair)
                ptx::umma_bf16_pair(d_tmem, adesc, bdesc, idesc, accumulate);
              else
                ptx::umma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
              accumulate = 1;
              if ((k & 3) == 3) {  // the box's last MMA: the box is free once these complete
                const uint32_t eb = ptx::smem_addr(&ctl->empty[s * (C::BK / KBOX) + (k >> 2)]);
                if constexpr (kPair)  // (kQuad: free in all four CTAs once both pairs arrive)
                  ptx::umma_commit_pair(eb, kQuad ? 0xF : pair_mask);
                else
                  ptx::umma_commit(eb);
              }
            }
            ++it;
          }
        }
        if (!ok) break;
        hand_over();
      }
      // Wait for every MMA issued before TMEM and shared memory go away (in both CTAs of a pair).
      if constexpr (kPair)
        ptx::umma_commit_pair(ptx::smem_addr(&ctl->drain), pair_mask);
      else
        ptx::umma_commit(ptx::smem_addr(&ctl->drain));
      wait_bounded(ptx::smem_addr(&ctl->drain), 0, abort_flag, p.status, true);
    } else if (kPair && lane == 0) {
      // The peer CTA: its shared memory feeds the leader's MMAs until the final drain arrives.
      wait_bounded(ptx::smem_addr(&ctl->drain), 0, abort_flag, p.status, true);
    }
  } else if constexpr (kEpi == EPI_BF16_CHUNKED) {
    // ---------------------------------------------------------------- epilogue, chunked sum
    epilogue_chunked<kPair, kQuad>(p, ctl, staging, tmem, warp, lane, unit, nunits, total, n_items, m_items,
                                   gm_items, quad, pq, cta, leader);
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int epi_tid = threadIdx.x - 64;
    const uint32_t wbuf = ptx::smem_addr(staging) + static_cast<uint32_t>(warp - 2) * 2 * kStageBuf;
    int nchunk = 0;
    uint32_t tcount = 0;
    for (int t = unit; t < total; t += nunits, ++tcount) {
      int g, mb, nb;
      decode_tile(p, t, g, mb, nb, n_items, m_items, gm_items);
      if (quad == 1) nb = 2 * nb + static_cast<int>(pq);
      if (quad == 2) mb = 2 * mb + static_cast<int>(pq);
      const uint32_t acc = tcount & 1u;
      const uint32_t aph = (tcount >> 1) & 1u;
      // Warp-uniform outcome: the epilogue's TMEM loads are warp-collective.
      if (!__all_sync(0xffffffffu, wait_bounded(ptx::smem_addr(&ctl->tfull[acc]), aph, abort_flag, p.status, false)))
        break;
      ptx::tc_fence_after();
      const int mb128 = mb * (C::TILE_M / BM) + static_cast<int>(cta);
      const int row0 = mb128 * BM + q * 32;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * static_cast<uint32_t>(p.bn);
      const uint32_t tempty = ptx::smem_addr(&ctl->tempty[acc]);
      auto release = [&]() {
        ptx::tc_fence_before();
        if constexpr (kPair)
          ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty, leader));  // the leader's MMA warp owns the accumulator
        else
          ptx::mbar_arrive(tempty);
      };
      epilogue_tile<kEpi>(p, ctl, taddr, wbuf, nchunk, g, row0, mb128, nb, lane, epi_tid, release);
    }
    if (lane == 0) ptx::bulk_wait_all();  // every output store of this warp has landed
  }

  __syncwarp();
  ptx::tc_fence_before();
  if constexpr (kPair) ptx::cluster_sync(); else __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    if constexpr (kPair)
      ptx::tmem_dealloc_pair(tmem, kTmemCols);
    else
      ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Encoded tensor maps are cached: a call that reuses the buffers of an earlier
// call (the usual case in a model's forward pass) skips the driver encode.  The
// key is every argument of the encode, so a cached map is exactly what the
// encode would return now, even if the memory was freed and reallocated at the
// same address.  The cache is cleared when it reaches kMapCacheMax entries.
struct MapKey {
  uint64_t ptr, inner, outer, stride;
  uint32_t box_inner, box_outer, dtype, swizzle;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = 1469598103934665603ull;
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ b[i]) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
constexpr size_t kMapCacheMax = 4096;
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

tp_status encode_2d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, int esz, int64_t inner, int64_t outer,
                    int64_t ld, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle,
                    CUtensorMapL2promotion promo) {
  MapKey key{};
  key.ptr = reinterpret_cast<uint64_t>(ptr);
  key.inner = static_cast<uint64_t>(inner);
  key.outer = static_cast<uint64_t>(outer);
  key.stride = static_cast<uint64_t>(ld) * esz;
  key.box_inner = box_inner;
  key.box_outer = box_outer;
  key.dtype = static_cast<uint32_t>(dtype) | (static_cast<uint32_t>(promo) << 16);
  key.swizzle = static_cast<uint32_t>(swizzle);
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *m = it->second;
      return TP_OK;
    }
  }
  auto enc = encoder();
  if (enc == nullptr) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  std::lock_guard<std::mutex> lock(g_map_mutex);
  if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
  g_map_cache.emplace(key, *m);
  return TP_OK;
}

// 2-D bf16 operand map over a row-major [outer, inner] matrix with row stride `ld`
// elements: box = 64 (inner) x box_outer rows, 128-byte swizzle, out-of-range reads as zero.
tp_status make_map(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
  return encode_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, ld, KBOX,
                   static_cast<uint32_t>(box_outer), CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// Largest number of CTA-pair clusters (kQuad: clusters of two pairs) that can be resident at
// once (cached per device and kernel).
template <int kEpi, bool kQuad = false>
int max_active_pairs(int sms) {
  static int cached[64] = {0};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev & 63] == 0) {
    cudaLaunchConfig_t cfg{};
    constexpr int kCluster = kQuad ? 4 : 2;
    cfg.gridDim = dim3(kCluster * (sms / kCluster), 1, 1);
    cfg.blockDim = dim3(threads_of(kEpi), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<true>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tp_gemm_kernel<kEpi, true, kQuad>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = kQuad ? 0 : sms / 2;  // no multicast launch then (launch_gemm falls back to pairs)
    }
    cached[dev & 63] = n;
  }
  return cached[dev & 63];
}

template <int kEpi, bool kPair, bool kQuad = false>
tp_status set_smem_attr() {
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    err = cudaFuncSetAttribute(tp_gemm_kernel<kEpi, kPair, kQuad>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes<kPair>()));
  });
  if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(max dynamic shared memory)");
  return TP_OK;
}

// Launch the single-CTA kernel (pair == false: 128-row tiles) or the CTA-pair kernel
// (pair == true: 256-row tiles, clusters of two CTAs).  p.m_tiles must match.
// Output map: a row-major [rows, cols] matrix (bf16 or fp32) with row stride `ld` elements,
// written in boxes of 32 rows from the epilogue's swizzled staging buffers: 64 bf16 or
// 32 fp32 columns (128-byte rows, 128-byte swizzle), or, for `narrow` bf16 maps, 32
// columns (64-byte rows, 64-byte swizzle).
tp_status make_out_map(CUtensorMap* m, void* ptr, bool f32, int64_t cols, int64_t rows, int64_t ld,
                       bool narrow = false) {
  const bool sw64 = !f32 && narrow;
  return encode_2d(m, ptr, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f32 ? 4 : 2,
                   cols, rows, ld, (f32 || narrow) ? 32u : 64u, 32u,
                   sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

template <int kEpi>
tp_status launch_gemm(const GemmParams& p, bool pair, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return fail(TP_ERR_CUDA, "cannot query the SM count of the current device");
  const int64_t total = static_cast<int64_t>(p.n_groups) * p.m_tiles * p.n_tiles;
  if (total <= 0) return TP_OK;
  if (total > 0x7FFFFFFF) return fail(TP_ERR_UNSUPPORTED, "too many tiles (%lld)", (long long)total);
  if (p.group_m < 1) return fail(TP_ERR_INVALID_ARG, "GEMM raster group size not set");
  // The workspace mode's CTAs wait on each other (bounded), so that launch is
  // cooperative: it is refused rather than started if they cannot all be resident.
  const bool coop = (kEpi == EPI_WS_REDUCE);
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[3];
  int nattr = 0;
  cfg.blockDim = dim3(threads_of(kEpi), 1, 1);
  cfg.stream = stream;
  if (coop) {
    attr[nattr].id = cudaLaunchAttributeCooperative;
    attr[nattr].val.cooperative = 1;
    ++nattr;
  } else {
    // Programmatic dependent launch (see launch_pdl): the kernel waits for its predecessor
    // after its prologue.
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  cudaError_t e;
  if constexpr (kEpi != EPI_WS_REDUCE) {
    if (pair && p.quad) {
      // Clusters of two CTA pairs, A shared by multicast (see tp_gemm_kernel).
      tp_status st = set_smem_attr<kEpi, true, true>();
      if (st != TP_OK) return st;
      const int quads_max = max_active_pairs<kEpi, true>(sms);
      if (quads_max < 1) return fail(TP_ERR_UNSUPPORTED, "no cluster of four CTAs fits on this device");
      const int64_t items = static_cast<int64_t>(p.n_groups) * p.m_tiles * p.n_tiles / 2;
      const int quads = static_cast<int>(items < quads_max ? items : quads_max);
      cfg.gridDim = dim3(4 * quads, 1, 1);
      cfg.dynamicSmemBytes = smem_bytes<true>();
      attr[nattr].id = cudaLaunchAttributeClusterDimension;
      attr[nattr].val.clusterDim.x = 4;
      attr[nattr].val.clusterDim.y = 1;
      attr[nattr].val.clusterDim.z = 1;
      ++nattr;
      cfg.attrs = attr;
      cfg.numAttrs = nattr;
      e = cudaLaunchKernelEx(&cfg, tp_gemm_kernel<kEpi, true, true>, p);
      if (e != cudaSuccess) return cuda_fail(e, "GEMM (clusters of CTA pairs) launch");
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "GEMM kernel launch");
      return TP_OK;
    }
  }
  if (!pair) {
    tp_status st = set_smem_attr<kEpi, false>();
    if (st != TP_OK) return st;
    cfg.gridDim = dim3(static_cast<unsigned>(total < sms ? total : sms), 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<false>();
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    e = cudaLaunchKernelEx(&cfg, tp_gemm_kernel<kEpi, false>, p);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
  } else {
    tp_status st = set_smem_attr<kEpi, true>();
    if (st != TP_OK) return st;
    const int pairs_max = max_active_pairs<kEpi>(sms);
    const int pairs = static_cast<int>(total < pairs_max ? total : pairs_max);
    if (coop && pairs < p.n_groups)  // each rank of a tile needs its own resident CTA pair
      return fail(TP_ERR_UNSUPPORTED, "%d resident CTA pairs cannot hold %d ranks", pairs, p.n_groups);
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<true>();
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = 2;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    e = cudaLaunchKernelEx(&cfg, tp_gemm_kernel<kEpi, true>, p);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM (CTA pair) launch");
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "GEMM kernel launch");
  return TP_OK;
}

// CTA pairs (256-row tiles) pay off once there is more than one 128-row block of output rows.
inline bool use_pair(int64_t T) { return T > BM; }

// Work units (CTAs, or CTA pairs) that run at the same time.
int resident_units(bool pair) {
  const int sms = sm_count();
  if (!pair) return sms;
  if (set_smem_attr<EPI_BF16, true>() != TP_OK) return sms / 2;
  return max_active_pairs<EPI_BF16>(sms);
}

// CTA-pair launches run as clusters of two pairs (tp_gemm_kernel's kQuad) when a tile count is
// even and the clusters' waves, each about 4 % shorter (measured: fewer operand bytes from L2),
// take no longer than the pairs' (fewer clusters of four than pairs fit: 36 x 4 CTAs against
// 76 x 2 on a 152-SM GB300; e.g. 2592 SwiGLU tiles make 36 cluster waves against 35 pair
// waves, and the clusters still win).  1 = pairs on n-adjacent tiles
// sharing A (even n_tiles), 2 = on m-adjacent tiles sharing B (even m_tiles), 0 = pairs alone.
// Decided before the operand maps are built: the shared operand's boxes are half as high.
int quad_mode(bool pair, int64_t groups, int64_t m_tiles, int64_t n_tiles) {
  if (!pair) return 0;
  if (n_tiles % 2 != 0 && m_tiles % 2 != 0) return 0;
  if (set_smem_attr<EPI_BF16, true, true>() != TP_OK) return 0;
  const int quads = max_active_pairs<EPI_BF16, true>(sm_count());
  const int pairs = resident_units(true);
  if (quads < 1 || pairs < 1) return 0;
  const int64_t tiles = groups * m_tiles * n_tiles;
  const int64_t waves_quad = (tiles / 2 + quads - 1) / quads, waves_pair = (tiles + pairs - 1) / pairs;
  if (waves_quad * 24 > waves_pair * 25) return 0;
  return (n_tiles % 2 == 0) ? 1 : 2;
}

// m-tiles per raster group.  When the A rows of every m-tile fit comfortably in L2, one group
// spans them all: each B panel is then read from DRAM once, by all m-tiles at about the same
// time, and A stays in L2 for the whole sweep.  Otherwise groups of about GROUP_M m-tiles,
// sized evenly, so that no small last group re-reads all of B for a few m-tiles (18 m-tiles
// make groups of 9 and 9, not 16 and 2).
constexpr int64_t kAResidentBytes = 64ll << 20;
int choose_group_m(int m_tiles, int64_t a_bytes) {
  if (a_bytes <= kAResidentBytes) return m_tiles;
  const int groups = (m_tiles + GROUP_M - 1) / GROUP_M;
  return (m_tiles + groups - 1) / groups;
}

// Accumulator width of a launch without SwiGLU: among the widths the epilogue
// supports (multiples of 32 up to 256), the one whose tiles finish in the fewest
// waves; ties go to the narrowest tile.  A launch's time follows its wave count first
// (a stage's fixed cost does not shrink with the width), then the width of its tiles:
// the 16 x N 3072 out-projection (K 4 x 768) took 58.0 / 54.0 / 64.2 / 72.3 / 80.5 us at
// widths 256 / 224 / 192 / 160 / 128 (3 / 3 / 4 / 5 / 6 waves of resident CTA pairs;
// 224 runs as plain pairs on all 152 SMs, 256 as clusters of two pairs on 144), and with a
// box refilled as soon as its MMAs are done 55.9 / 52.9 us at 256 / 224 (each launch alone
// after an L2 flush).
int choose_bn(int64_t n_out, int64_t groups_x_mtiles, int units, bool halves_of_32 = false) {
  static const int kWidths[] = {256, 224, 192, 160, 128};
  int best = 256;
  int64_t best_waves = -1;
  for (int bn : kWidths) {
    if (halves_of_32 && (bn / 2) % 32 != 0) continue;  // the chunked epilogue's halves: 128, 96 or 64 columns
    const int64_t tiles = groups_x_mtiles * ((n_out + bn - 1) / bn);
    const int64_t waves = (tiles + units - 1) / units;
    if (best_waves < 0 || waves <= best_waves) {
      best = bn;
      best_waves = waves;
    }
  }
  return best;
}

inline int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }
inline int stage_k(bool pair) { return pair ? Cfg<true>::BK : Cfg<false>::BK; }

tp_status check_dims(int64_t T, int64_t K, int64_t N) {
  if (T < 0 || K < 0 || N < 0) return fail(TP_ERR_INVALID_ARG, "negative size");
  if (T > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
    return fail(TP_ERR_UNSUPPORTED, "sizes above 2^31-1 are not supported");
  return TP_OK;
}

}  // namespace
}  // namespace tp

extern "C" {

tp_status tp_linear_colwise(const void* x, const void* const* w_shards, const void* const* bias_shards, tp_act act,
                            int tp_degree, int64_t T, int64_t K, int64_t N_r, void* const* y_shards, int64_t ldy,
                            tp_stream_t stream) {
  using namespace tp;
  clear_error();
  if (tp_degree < 1) return fail(TP_ERR_INVALID_ARG, "tp_degree must be >= 1, got %d", tp_degree);
  if (tp_degree > TP_MAX_DEGREE)
    return fail(TP_ERR_UNSUPPORTED, "tp_degree=%d above TP_MAX_DEGREE=%d", tp_degree, TP_MAX_DEGREE);
  const bool chunked = (static_cast<int>(act) & TP_ACCUM_CHUNKED) != 0;
  act = static_cast<tp_act>(static_cast<int>(act) & ~TP_ACCUM_CHUNKED);
  if (act != TP_ACT_NONE && act != TP_ACT_GELU_TANH && act != TP_ACT_SWIGLU)
    return fail(TP_ERR_INVALID_ARG, "unknown activation %d", (int)act);
  if (chunked && act != TP_ACT_NONE)
    return fail(TP_ERR_UNSUPPORTED, "TP_ACCUM_CHUNKED is supported with TP_ACT_NONE only");
  tp_status st = check_dims(T, K, N_r);
  if (st != TP_OK) return st;
  if (act == TP_ACT_SWIGLU && (N_r % 2) != 0)
    return fail(TP_ERR_INVALID_ARG, "SwiGLU needs an even shard width ([gate_r; up_r]), got N_r=%lld", (long long)N_r);
  const int64_t n_out = (act == TP_ACT_SWIGLU) ? N_r / 2 : N_r;
  if (ldy == 0) ldy = n_out;
  if (ldy < n_out) return fail(TP_ERR_INVALID_ARG, "ldy=%lld smaller than the output width %lld", (long long)ldy,
                               (long long)n_out);
  if (T == 0 || N_r == 0) return TP_OK;
  if (K == 0) return fail(TP_ERR_INVALID_ARG, "K (in_features) must be positive");
  if (x == nullptr || w_shards == nullptr || y_shards == nullptr)
    return fail(TP_ERR_INVALID_ARG, "x, w_shards or y_shards is NULL");
  if ((K % 8) != 0 || (n_out % 8) != 0 || (ldy % 8) != 0)
    return fail(TP_ERR_ALIGNMENT, "K (%lld), output width (%lld) and ldy (%lld) must be multiples of 8",
                (long long)K, (long long)n_out, (long long)ldy);
  if (!aligned16(x)) return fail(TP_ERR_ALIGNMENT, "x is not 16-byte aligned");
  for (int r = 0; r < tp_degree; ++r) {
    if (w_shards[r] == nullptr || y_shards[r] == nullptr)
      return fail(TP_ERR_INVALID_ARG, "w_shards[%d] or y_shards[%d] is NULL", r, r);
    if (!aligned16(w_shards[r]) || !aligned16(y_shards[r]))
      return fail(TP_ERR_ALIGNMENT, "w_shards[%d] or y_shards[%d] is not 16-byte aligned", r, r);
  }
  unsigned int* status = status_word();
  if (status == nullptr) return fail(TP_ERR_CUDA, "cannot locate the kernel status word");

  const bool pair = use_pair(T);
  GemmParams p{};
  const int64_t m_tiles = (T + (pair ? 2 * BM : BM) - 1) / (pair ? 2 * BM : BM);
  const int bn = (act == TP_ACT_SWIGLU) ? BN : choose_bn(n_out, tp_degree * m_tiles, resident_units(pair), chunked);
  const int quad = quad_mode(pair, tp_degree, m_tiles, ceil_div(n_out, (act == TP_ACT_SWIGLU) ? BN / 2 : bn));
  p.quad = quad;
  st = make_map(&p.map_a[0], x, K, T, K, quad == 1 ? BM / 2 : BM);
  if (st != TP_OK) return st;
  const int box_b = ((act == TP_ACT_SWIGLU) ? BN / 2 : (pair ? bn / 2 : bn)) / (quad == 2 ? 2 : 1);
  for (int r = 0; r < tp_degree; ++r) {
    st = make_map(&p.map_b[r], w_shards[r], K, N_r, K, box_b);
    if (st != TP_OK) return st;
    p.out[r] = y_shards[r];
    p.bias[r] = bias_shards ? static_cast<const __nv_bfloat16*>(bias_shards[r]) : nullptr;
    st = make_out_map(&p.map_out[r], y_shards[r], false, n_out, T, ldy);
    if (st == TP_OK) st = make_out_map(&p.map_out_tail[r], y_shards[r], false, n_out, T, ldy, true);
    if (st != TP_OK) return st;
  }
  p.status = status;
  p.tile_wait_ns = tile_wait_limit_ns();
  p.ldo = ldy;
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(n_out);
  p.n_groups = tp_degree;
  p.n_ksegs = 1;
  p.kblocks = ceil_div(K, stage_k(pair));
  p.m_tiles = ceil_div(T, pair ? 2 * BM : BM);
  p.group_m = choose_group_m(p.m_tiles, T * K * 2);  // A = X, shared by every rank
  p.n_tiles = ceil_div(n_out, (act == TP_ACT_SWIGLU) ? BN / 2 : bn);
  p.bn = bn;
  p.b_up_row = static_cast<int>(N_r / 2);
  p.rank_fastest = 0;
  p.a_shared = 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (act) {
    case TP_ACT_GELU_TANH: return launch_gemm<EPI_GELU>(p, pair, s);
    case TP_ACT_SWIGLU: return launch_gemm<EPI_SWIGLU>(p, pair, s);
    default: return chunked ? launch_gemm<EPI_BF16_CHUNKED>(p, pair, s) : launch_gemm<EPI_BF16>(p, pair, s);
  }
}

size_t tp_rowwise_workspace_bytes(int tp_degree, int64_t T, int64_t N, tp_reduce_mode mode) {
  if (mode != TP_REDUCE_WORKSPACE || tp_degree < 1 || T <= 0 || N <= 0) return 0;
  const size_t partials = static_cast<size_t>(tp_degree) * static_cast<size_t>(T) * static_cast<size_t>(N) * 4;
  const size_t aligned = (partials + 255) & ~static_cast<size_t>(255);
  // One counter per 128-row block and n-tile, sized for the narrowest tile (128 columns).
  const size_t tiles = static_cast<size_t>((T + tp::BM - 1) / tp::BM) * static_cast<size_t>((N + 127) / 128);
  return aligned + tiles * sizeof(int);
}

}  // extern "C"

namespace tp {
namespace {
tp_status rowwise_impl(const void* const* x_shards, int64_t ldx, const void* const* w_shards, const void* bias,
                       int tp_degree, int64_t T, int64_t K_r, int64_t N, tp_reduce_mode mode, void* workspace,
                       size_t ws_bytes, void* out, tp_stream_t stream);
}  // namespace
}  // namespace tp

extern "C" {

tp_status tp_linear_rowwise(const void* const* x_shards, const void* const* w_shards, const void* bias, int tp_degree,
                            int64_t T, int64_t K_r, int64_t N, tp_reduce_mode mode, void* workspace, size_t ws_bytes,
                            void* out, tp_stream_t stream) {
  tp::clear_error();
  return tp::rowwise_impl(x_shards, K_r, w_shards, bias, tp_degree, T, K_r, N, mode, workspace, ws_bytes, out,
                          stream);
}

tp_status tp_linear_rowwise_split_input(const void* x, int64_t ldx, const void* const* w_shards, const void* bias,
                                        int tp_degree, int64_t T, int64_t K, int64_t N, tp_reduce_mode mode,
                                        void* workspace, size_t ws_bytes, void* out, tp_stream_t stream) {
  using namespace tp;
  clear_error();
  if (tp_degree < 1) return fail(TP_ERR_INVALID_ARG, "tp_degree must be >= 1, got %d", tp_degree);
  if (tp_degree > TP_MAX_DEGREE)
    return fail(TP_ERR_UNSUPPORTED, "tp_degree=%d above TP_MAX_DEGREE=%d", tp_degree, TP_MAX_DEGREE);
  if (K < 0 || T < 0 || N < 0) return fail(TP_ERR_INVALID_ARG, "negative size");
  if (K % tp_degree != 0)
    return fail(TP_ERR_SPLIT_NOT_DIVISIBLE, "K=%lld not divisible by tp_degree=%d", (long long)K, tp_degree);
  if (ldx == 0) ldx = K;
  if (ldx < K) return fail(TP_ERR_INVALID_ARG, "ldx=%lld smaller than K=%lld", (long long)ldx, (long long)K);
  if (T == 0 || N == 0) return TP_OK;
  if (x == nullptr) return fail(TP_ERR_INVALID_ARG, "x is NULL");
  // Rank r's input is the column window [r*K/p, (r+1)*K/p) of the replicated X: a strided view, no copy.
  const int64_t K_r = K / tp_degree;
  const void* xs[TP_MAX_DEGREE];
  for (int r = 0; r < tp_degree; ++r) xs[r] = static_cast<const uint16_t*>(x) + static_cast<int64_t>(r) * K_r;
  return rowwise_impl(xs, ldx, w_shards, bias, tp_degree, T, K_r, N, mode, workspace, ws_bytes, out, stream);
}

}  // extern "C"

namespace tp {
namespace {
tp_status rowwise_impl(const void* const* x_shards, int64_t ldx, const void* const* w_shards, const void* bias,
                       int tp_degree, int64_t T, int64_t K_r, int64_t N, tp_reduce_mode mode, void* workspace,
                       size_t ws_bytes, void* out, tp_stream_t stream) {
  if (tp_degree < 1) return fail(TP_ERR_INVALID_ARG, "tp_degree must be >= 1, got %d", tp_degree);
  if (tp_degree > TP_MAX_DEGREE)
    return fail(TP_ERR_UNSUPPORTED, "tp_degree=%d above TP_MAX_DEGREE=%d", tp_degree, TP_MAX_DEGREE);
  if (mode != TP_REDUCE_NONE && mode != TP_REDUCE_WORKSPACE && mode != TP_REDUCE_ACCUM)
    return fail(TP_ERR_INVALID_ARG, "unknown reduce mode %d", (int)mode);
  tp_status st = check_dims(T, K_r, N);
  if (st != TP_OK) return st;
  if (T == 0 || N == 0) return TP_OK;
  if (K_r == 0) return fail(TP_ERR_INVALID_ARG, "K_r (input features per rank) must be positive");
  if (x_shards == nullptr || w_shards == nullptr || out == nullptr)
    return fail(TP_ERR_INVALID_ARG, "x_shards, w_shards or out is NULL");
  if ((K_r % 8) != 0 || (N % 8) != 0 || (ldx % 8) != 0)
    return fail(TP_ERR_ALIGNMENT, "K_r (%lld), N (%lld) and the input row stride (%lld) must be multiples of 8",
                (long long)K_r, (long long)N, (long long)ldx);
  if (!aligned16(out) || (bias != nullptr && !aligned16(bias)))
    return fail(TP_ERR_ALIGNMENT, "out or bias is not 16-byte aligned");
  for (int r = 0; r < tp_degree; ++r) {
    if (x_shards[r] == nullptr || w_shards[r] == nullptr)
      return fail(TP_ERR_INVALID_ARG, "x_shards[%d] or w_shards[%d] is NULL", r, r);
    if (!aligned16(x_shards[r]) || !aligned16(w_shards[r]))
      return fail(TP_ERR_ALIGNMENT, "x_shards[%d] or w_shards[%d] is not 16-byte aligned", r, r);
  }
  const size_t need = tp_rowwise_workspace_bytes(tp_degree, T, N, mode);
  if (mode == TP_REDUCE_WORKSPACE) {
    if (workspace == nullptr || ws_bytes < need)
      return fail(TP_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace ? ws_bytes : 0, need);
    if (!aligned16(workspace)) return fail(TP_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
  }
  unsigned int* status = status_word();
  if (status == nullptr) return fail(TP_ERR_CUDA, "cannot locate the kernel status word");

  const bool pair = use_pair(T);
  const int64_t m_tiles = (T + (pair ? 2 * BM : BM) - 1) / (pair ? 2 * BM : BM);
  const int groups = (mode == TP_REDUCE_ACCUM) ? 1 : tp_degree;
  const int bn = choose_bn(N, groups * m_tiles, resident_units(pair));
  // (the workspace mode stays in pairs)
  const int quad = mode == TP_REDUCE_WORKSPACE ? 0 : quad_mode(pair, groups, m_tiles, ceil_div(N, bn));
  GemmParams p{};
  p.quad = quad;
  for (int r = 0; r < tp_degree; ++r) {
    st = make_map(&p.map_a[r], x_shards[r], K_r, T, ldx, quad == 1 ? BM / 2 : BM);
    if (st != TP_OK) return st;
    st = make_map(&p.map_b[r], w_shards[r], K_r, N, K_r, (pair ? bn / 2 : bn) / (quad == 2 ? 2 : 1));
    if (st != TP_OK) return st;
  }
  p.status = status;
  p.tile_wait_ns = tile_wait_limit_ns();
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(N);
  p.kblocks = ceil_div(K_r, stage_k(pair));
  p.m_tiles = ceil_div(T, pair ? 2 * BM : BM);
  // A of one tile sweep: every rank's X_r when the ranks are k-segments of one accumulator.
  p.group_m = choose_group_m(p.m_tiles, T * K_r * 2 * (mode == TP_REDUCE_ACCUM ? tp_degree : 1));
  p.n_tiles = ceil_div(N, bn);
  p.bn = bn;
  p.n_counters = ceil_div(N, 128);
  p.a_shared = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode == TP_REDUCE_ACCUM) {
    st = make_out_map(&p.map_out[0], out, false, N, T, N);
    if (st == TP_OK) st = make_out_map(&p.map_out_tail[0], out, false, N, T, N, true);
    if (st != TP_OK) return st;
    p.out[0] = out;
    p.bias[0] = static_cast<const __nv_bfloat16*>(bias);
    p.ldo = N;
    p.n_groups = 1;
    p.n_ksegs = tp_degree;
    p.rank_fastest = 0;
    return launch_gemm<EPI_BF16>(p, pair, s);
  }
  if (mode == TP_REDUCE_NONE) {
    for (int r = 0; r < tp_degree; ++r) {
      p.out[r] = static_cast<float*>(out) + static_cast<int64_t>(r) * T * N;
      p.bias[r] = (r == 0) ? static_cast<const __nv_bfloat16*>(bias) : nullptr;
      st = make_out_map(&p.map_out[r], p.out[r], true, N, T, N);
      if (st != TP_OK) return st;
    }
    p.ldo = N;
    p.n_groups = tp_degree;
    p.n_ksegs = 1;
    p.rank_fastest = 0;
    return launch_gemm<EPI_F32>(p, pair, s);
  }
  // TP_REDUCE_WORKSPACE
  const size_t partial_bytes = (static_cast<size_t>(tp_degree) * T * N * 4 + 255) & ~static_cast<size_t>(255);
  p.ws = static_cast<float*>(workspace);
  for (int r = 0; r < tp_degree; ++r) {
    st = make_out_map(&p.map_out[r], p.ws + static_cast<int64_t>(r) * T * N, true, N, T, N);
    if (st != TP_OK) return st;
  }
  p.counters = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + partial_bytes);
  p.reduce_out = static_cast<__nv_bfloat16*>(out);
  p.reduce_bias = static_cast<const __nv_bfloat16*>(bias);
  p.ldo = N;
  p.n_groups = tp_degree;
  p.n_ksegs = 1;
  p.rank_fastest = 1;
  cudaError_t e = cudaMemsetAsync(p.counters, 0, need - partial_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the tile counters");
  return launch_gemm<EPI_WS_REDUCE>(p, pair, s);
}
}  // namespace
}  // namespace tp

// ---------------------------------------------------------------------------
// Rowwise workspace mode for callers that cannot allocate: the scratch is a
// fixed array compiled into the library.  Host code must not pass the
// array's name to a kernel (on the host it is only a stand-in symbol); its
// device address is looked up once per device and context and cached.
// ---------------------------------------------------------------------------

namespace tp {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TP_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {nullptr};
unsigned long long g_noalloc_ctx[64] = {0};

tp_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TP_ERR_UNSUPPORTED, "device index %d above 63", dev);
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  // Looked up again in a new context (after cudaDeviceReset, or a caller's own context): the
  // module, and with it the array, is loaded anew there.
  if (g_noalloc_ptr[dev] == nullptr || ctx == 0 || g_noalloc_ctx[dev] != ctx) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(built-in scratch)");
    g_noalloc_ptr[dev] = ptr;
    g_noalloc_ctx[dev] = current_context_id();
  }
  *out = g_noalloc_ptr[dev];
  return TP_OK;
}

}  // namespace
}  // namespace tp

extern "C" tp_status tp_linear_rowwise_noalloc(const void* const* x_shards, const void* const* w_shards,
                                               const void* bias, int tp_degree, int64_t T, int64_t K_r, int64_t N,
                                               void* out, tp_stream_t stream) {
  using namespace tp;
  clear_error();
  if (tp_degree < 1 || tp_degree > TP_MAX_DEGREE || T < 0 || N < 0 || K_r < 0)
    // Argument errors are reported by the shared entry point, before any device work.
    return tp_linear_rowwise(x_shards, w_shards, bias, tp_degree, T, K_r, N, TP_REDUCE_WORKSPACE, nullptr, 0, out,
                             stream);
  const size_t need = tp_rowwise_workspace_bytes(tp_degree, T, N, TP_REDUCE_WORKSPACE);
  if (need > TP_NOALLOC_SCRATCH_BYTES)
    return fail(TP_ERR_WORKSPACE,
                "tp_degree=%d, T=%lld, N=%lld needs %zu bytes of scratch; the built-in array holds %zu "
                "(TP_NOALLOC_SCRATCH_BYTES): pass a workspace to tp_linear_rowwise instead",
                tp_degree, (long long)T, (long long)N, need, (size_t)TP_NOALLOC_SCRATCH_BYTES);
  if (need == 0)  // empty problem: nothing to launch, nothing to look up
    return tp_linear_rowwise(x_shards, w_shards, bias, tp_degree, T, K_r, N, TP_REDUCE_WORKSPACE, nullptr, 0, out,
                             stream);
  void* scratch = nullptr;
  tp_status st = noalloc_scratch(&scratch);
  if (st != TP_OK) return st;
  return tp_linear_rowwise(x_shards, w_shards, bias, tp_degree, T, K_r, N, TP_REDUCE_WORKSPACE, scratch,
                           TP_NOALLOC_SCRATCH_BYTES, out, stream);
}

// ---------------------------------------------------------------------------
// Batched GEMM for the attention core (library-internal): group i computes
// out_i = A_i . B_i^T with A_i [M, K] (row stride lda), B_i [N, K] (row stride
// ldb), out_i [M, N] (row stride ldo, bf16 or fp32), K-major bf16 operands.
// ---------------------------------------------------------------------------

namespace tp {

tp_status gemm_batched(int groups, const void* const* a, int64_t lda, const void* const* b, int64_t ldb,
                       void* const* out, int64_t ldo, bool out_f32, int64_t M, int64_t N, int64_t K,
                       cudaStream_t stream) {
  if (groups < 1 || groups > TP_MAX_DEGREE) return fail(TP_ERR_INVALID_ARG, "batched GEMM of %d groups", groups);
  if (M == 0 || N == 0) return TP_OK;
  if (K <= 0 || (K % 8) || (N % 8) || (lda % 8) || (ldb % 8) || (ldo % 8))
    return fail(TP_ERR_ALIGNMENT, "batched GEMM needs K, N and leading dimensions that are multiples of 8");
  unsigned int* status = status_word();
  if (status == nullptr) return fail(TP_ERR_CUDA, "cannot locate the kernel status word");
  const bool pair = use_pair(M);
  const int64_t m_tiles = (M + (pair ? 2 * BM : BM) - 1) / (pair ? 2 * BM : BM);
  const int bn = choose_bn(N, groups * m_tiles, resident_units(pair));
  const int quad = quad_mode(pair, groups, m_tiles, ceil_div(N, bn));
  GemmParams p{};
  p.quad = quad;
  for (int g = 0; g < groups; ++g) {
    if (!aligned16(a[g]) || !aligned16(b[g]) || !aligned16(out[g]))
      return fail(TP_ERR_ALIGNMENT, "batched GEMM operand of group %d is not 16-byte aligned", g);
    tp_status st = make_map(&p.map_a[g], a[g], K, M, lda, quad == 1 ? BM / 2 : BM);
    if (st == TP_OK) st = make_map(&p.map_b[g], b[g], K, N, ldb, (pair ? bn / 2 : bn) / (quad == 2 ? 2 : 1));
    if (st == TP_OK) st = make_out_map(&p.map_out[g], out[g], out_f32, N, M, ldo);
    if (st == TP_OK && !out_f32) st = make_out_map(&p.map_out_tail[g], out[g], false, N, M, ldo, true);
    if (st != TP_OK) return st;
    p.out[g] = out[g];
  }
  p.status = status;
  p.tile_wait_ns = tile_wait_limit_ns();
  p.ldo = ldo;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.n_groups = groups;
  p.n_ksegs = 1;
  p.kblocks = ceil_div(K, stage_k(pair));
  p.m_tiles = static_cast<int>(m_tiles);
  p.group_m = choose_group_m(p.m_tiles, M * K * 2);
  p.n_tiles = ceil_div(N, bn);
  p.bn = bn;
  p.a_shared = 0;
  p.rank_fastest = 0;
  return out_f32 ? launch_gemm<EPI_F32>(p, pair, stream) : launch_gemm<EPI_BF16>(p, pair, stream);
}

}  // namespace tp

namespace tp {

// bf16 2-D tensor map for other kernels of the library (cached like the GEMM's own).
tp_status encode_bf16_2d(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, uint32_t box_inner,
                         uint32_t box_outer, bool swizzle128) {
  return encode_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, ld, box_inner, box_outer,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

}  // namespace tp
