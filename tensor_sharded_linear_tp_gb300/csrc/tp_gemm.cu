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
//                fastest; each rank writes its fp32 partial tile, then an
//                atomic per-tile counter elects the last rank to finish, which
//                sums the partials in rank order and writes bf16 (no spin).
//     NONE       work item = (rank, m-tile, n-tile); fp32 partials out.
//
// CTA layout (192 threads, one CTA per SM, grid = min(#tiles, #SMs)):
//   warp 0      TMA producer: A (128 x 64) and B (256 x 64) bf16 boxes with
//               128-byte swizzle into a 4-stage shared-memory ring.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=256,
//               K=16) into one of two TMEM accumulators (2 x 256 columns),
//               so the epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, bias, activation
//               (GELU-tanh or SwiGLU) in fp32, round to bf16, store.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); a wait that
// gives up sets a flag in the library's status word and the CTA drains its
// in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tp_internal.h"
#include "tp_ptx.cuh"

namespace tp {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int GROUP_M = 16;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum Epi : int { EPI_BF16 = 0, EPI_GELU = 1, EPI_SWIGLU = 2, EPI_F32 = 3, EPI_WS_REDUCE = 4 };

struct GemmParams {
  CUtensorMap map_a[TP_MAX_DEGREE];
  CUtensorMap map_b[TP_MAX_DEGREE];
  void* out[TP_MAX_DEGREE];                  // per output group
  const __nv_bfloat16* bias[TP_MAX_DEGREE];  // per output group, nullable
  float* ws;                                 // WS_REDUCE: fp32 partials [n_groups][M][N]
  int* counters;                             // WS_REDUCE: [m_tiles * n_tiles]
  __nv_bfloat16* reduce_out;                 // WS_REDUCE: bf16 [M][ldo]
  const __nv_bfloat16* reduce_bias;          // WS_REDUCE: nullable [N]
  unsigned int* status;
  int64_t ldo;        // row stride of the outputs, elements
  int M, N;           // output rows; output columns per group
  int n_groups;       // independent outputs (ranks) -- 1 for ACCUM
  int n_ksegs;        // K segments per tile (ranks) -- >1 only for ACCUM
  int kblocks;        // 64-wide K blocks per segment
  int m_tiles, n_tiles;
  int b_up_row;       // SwiGLU: first row of the up block inside W_r
  int rank_fastest;   // tile order with the rank varying fastest
  int a_shared;       // one A map for every rank (colwise)
};

struct alignas(8) SmemCtrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int is_last;
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + sizeof(SmemCtrl);

__device__ __forceinline__ void decode_tile(const GemmParams& p, int t, int& g, int& mb, int& nb) {
  const int tiles_mn = p.m_tiles * p.n_tiles;
  int mn;
  if (p.rank_fastest) {
    g = t % p.n_groups;
    mn = t / p.n_groups;
  } else {
    g = t / tiles_mn;
    mn = t - g * tiles_mn;
  }
  // Grouped raster: GROUP_M m-tiles sweep the n-tiles together so the CTAs
  // running at the same time share A and B tiles through L2.
  const int span = GROUP_M * p.n_tiles;
  const int sr = mn / span;
  const int first_m = sr * GROUP_M;
  const int gm = min(p.m_tiles - first_m, GROUP_M);
  const int in = mn - sr * span;
  mb = first_m + in % gm;
  nb = in / gm;
}

// Bounded wait: true when the phase completed; false when this CTA is aborting
// (another role gave up) or the wait itself ran out of time.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* status, bool ignore_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
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

__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  return 0.5f * x * (1.0f + tanhf(k0 * (x + k1 * x * x * x)));
}
__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + __expf(-x)); }

// Store 32 consecutive fp32 values as bf16 (64 bytes), masked at 8-column granularity.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&f)[32], int valid_cols) {
  uint32_t packed[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
    packed[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (8 * q < valid_cols) d[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
}

__device__ __forceinline__ void store_f32x32(float* dst, const uint32_t (&v)[32], float b0, const float* bvec,
                                             int valid_cols) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (4 * q < valid_cols) {
      float4 o;
      o.x = __uint_as_float(v[4 * q + 0]) + (bvec ? bvec[4 * q + 0] : b0);
      o.y = __uint_as_float(v[4 * q + 1]) + (bvec ? bvec[4 * q + 1] : b0);
      o.z = __uint_as_float(v[4 * q + 2]) + (bvec ? bvec[4 * q + 2] : b0);
      o.w = __uint_as_float(v[4 * q + 3]) + (bvec ? bvec[4 * q + 3] : b0);
      d[q] = o;
    }
  }
}

template <int kEpi>
__global__ void __launch_bounds__(kThreads, 1) tp_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SmemCtrl* ctl = reinterpret_cast<SmemCtrl*>(base + STAGES * STAGE_BYTES);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl->full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&ctl->tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->tempty[a]), 128);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ctl->abort = 0;
    ctl->is_last = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  const int total = p.n_groups * p.m_tiles * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int g, mb, nb;
        decode_tile(p, t, g, mb, nb);
        for (int seg = 0; seg < p.n_ksegs && ok; ++seg) {
          const int r = (p.n_ksegs > 1) ? seg : g;
          const CUtensorMap* ma = &p.map_a[p.a_shared ? 0 : r];
          const CUtensorMap* mbm = &p.map_b[r];
          for (int kb = 0; kb < p.kblocks; ++kb) {
            const uint32_t s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!wait_bounded(ptx::smem_addr(&ctl->empty[s]), ph ^ 1u, abort_flag, p.status, false)) {
              ok = false;
              break;
            }
            const uint32_t full = ptx::smem_addr(&ctl->full[s]);
            const uint32_t sa = ptx::smem_addr(base + s * STAGE_BYTES);
            const uint32_t sb = sa + A_BYTES;
            ptx::mbar_arrive_expect_tx(full, STAGE_BYTES);
            ptx::tma_load_2d(sa, ma, full, kb * BK, mb * BM);
            if (kEpi == EPI_SWIGLU) {
              ptx::tma_load_2d(sb, mbm, full, kb * BK, nb * (BN / 2));
              ptx::tma_load_2d(sb + B_BYTES / 2, mbm, full, kb * BK, p.b_up_row + nb * (BN / 2));
            } else {
              ptx::tma_load_2d(sb, mbm, full, kb * BK, nb * BN);
            }
            ++it;
          }
        }
      }
      // Let every copy this thread issued land before the CTA can exit.
      const uint32_t first = it > STAGES ? it - STAGES : 0;
      for (uint32_t j = first; j < it; ++j)
        wait_bounded(ptx::smem_addr(&ctl->full[j % STAGES]), (j / STAGES) & 1u, abort_flag, p.status, true);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tcount) {
        const uint32_t acc = tcount & 1u;
        const uint32_t aph = (tcount >> 1) & 1u;
        if (!wait_bounded(ptx::smem_addr(&ctl->tempty[acc]), aph ^ 1u, abort_flag, p.status, false)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * BN;
        uint32_t accumulate = 0;
        for (int seg = 0; seg < p.n_ksegs && ok; ++seg) {
          for (int kb = 0; kb < p.kblocks; ++kb) {
            const uint32_t s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1u;
            if (!wait_bounded(ptx::smem_addr(&ctl->full[s]), ph, abort_flag, p.status, false)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t sa = ptx::smem_addr(base + s * STAGE_BYTES);
            const uint64_t adesc = ptx::sw128_kmajor_desc(sa);
            const uint64_t bdesc = ptx::sw128_kmajor_desc(sa + A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              // +32 bytes along K inside the 128-byte swizzled row = +2 in the >>4 address field.
              ptx::umma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, accumulate);
              accumulate = 1;
            }
            ptx::umma_commit(ptx::smem_addr(&ctl->empty[s]));
            ++it;
          }
        }
        if (!ok) break;
        ptx::umma_commit(ptx::smem_addr(&ctl->tfull[acc]));
      }
      // Wait for every MMA this thread issued before TMEM and shared memory go away.
      ptx::umma_commit(ptx::smem_addr(&ctl->drain));
      wait_bounded(ptx::smem_addr(&ctl->drain), 0, abort_flag, p.status, true);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int epi_tid = threadIdx.x - 64;
    uint32_t tcount = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tcount) {
      int g, mb, nb;
      decode_tile(p, t, g, mb, nb);
      const uint32_t acc = tcount & 1u;
      const uint32_t aph = (tcount >> 1) & 1u;
      if (!wait_bounded(ptx::smem_addr(&ctl->tfull[acc]), aph, abort_flag, p.status, false)) break;
      ptx::tc_fence_after();
      const int row = mb * BM + q * 32 + lane;
      const bool row_ok = row < p.M;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      const uint32_t tempty = ptx::smem_addr(&ctl->tempty[acc]);

      if constexpr (kEpi == EPI_SWIGLU) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[g]);
        const __nv_bfloat16* bias = p.bias[g];
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld_32x32b_x32(taddr + c, gv);
          ptx::tmem_ld_32x32b_x32(taddr + BN / 2 + c, uv);
          ptx::tmem_ld_wait();
          if (c + 32 >= BN / 2) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(tempty);
          }
          const int col0 = nb * (BN / 2) + c;
          if (row_ok && col0 < p.N) {
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = col0 + j;
              float gg = __uint_as_float(gv[j]);
              float uu = __uint_as_float(uv[j]);
              if (bias != nullptr && col < p.N) {
                gg += __bfloat162float(bias[col]);
                uu += __bfloat162float(bias[p.b_up_row + col]);
              }
              f[j] = silu_f(gg) * uu;
            }
            store_bf16x32(out + static_cast<int64_t>(row) * p.ldo + col0, f, p.N - col0);
          }
        }
      } else if constexpr (kEpi == EPI_BF16 || kEpi == EPI_GELU) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out[g]);
        const __nv_bfloat16* bias = p.bias[g];
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(taddr + c, v);
          ptx::tmem_ld_wait();
          if (c + 32 >= BN) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(tempty);
          }
          const int col0 = nb * BN + c;
          if (row_ok && col0 < p.N) {
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float x = __uint_as_float(v[j]);
              if (bias != nullptr && col0 + j < p.N) x += __bfloat162float(bias[col0 + j]);
              f[j] = (kEpi == EPI_GELU) ? gelu_tanh_f(x) : x;
            }
            store_bf16x32(out + static_cast<int64_t>(row) * p.ldo + col0, f, p.N - col0);
          }
        }
      } else {
        // fp32 partial tile: to the caller's buffer (EPI_F32) or the workspace (EPI_WS_REDUCE).
        float* out;
        int64_t ld;
        const __nv_bfloat16* bias;
        if constexpr (kEpi == EPI_F32) {
          out = static_cast<float*>(p.out[g]);
          ld = p.ldo;
          bias = p.bias[g];
        } else {
          out = p.ws + static_cast<int64_t>(g) * p.M * p.N;
          ld = p.N;
          bias = nullptr;
        }
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(taddr + c, v);
          ptx::tmem_ld_wait();
          if (c + 32 >= BN) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(tempty);
          }
          const int col0 = nb * BN + c;
          if (row_ok && col0 < p.N) {
            float bv[32];
            if (bias != nullptr) {
#pragma unroll
              for (int j = 0; j < 32; ++j) bv[j] = (col0 + j < p.N) ? __bfloat162float(bias[col0 + j]) : 0.f;
            }
            store_f32x32(out + static_cast<int64_t>(row) * ld + col0, v, 0.f, bias ? bv : nullptr, p.N - col0);
          }
        }
        if constexpr (kEpi == EPI_WS_REDUCE) {
          // Publish this rank's partial tile, count it, and let the last rank to arrive sum all of them.
          __threadfence();
          ptx::named_bar_sync(1, 128);
          if (epi_tid == 0) {
            const int old = atomicAdd(&p.counters[mb * p.n_tiles + nb], 1);
            *reinterpret_cast<volatile int*>(&ctl->is_last) = (old == p.n_groups - 1);
          }
          ptx::named_bar_sync(1, 128);
          const bool last = *reinterpret_cast<volatile int*>(&ctl->is_last) != 0;
          if (last) {
            __threadfence();
            if (row_ok) {
              const int64_t plane = static_cast<int64_t>(p.M) * p.N;
#pragma unroll 1
              for (int c = 0; c < BN; c += 8) {
                const int col = nb * BN + c;
                if (col >= p.N) break;
                float a8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) a8[j] = 0.f;
                const float* src = p.ws + static_cast<int64_t>(row) * p.N + col;
                for (int r = 0; r < p.n_groups; ++r) {
                  const float4* s4 = reinterpret_cast<const float4*>(src + r * plane);
                  const float4 x0 = __ldcg(s4);
                  const float4 x1 = __ldcg(s4 + 1);
                  a8[0] += x0.x; a8[1] += x0.y; a8[2] += x0.z; a8[3] += x0.w;
                  a8[4] += x1.x; a8[5] += x1.y; a8[6] += x1.z; a8[7] += x1.w;
                }
                if (p.reduce_bias != nullptr) {
#pragma unroll
                  for (int j = 0; j < 8; ++j) a8[j] += __bfloat162float(p.reduce_bias[col + j]);
                }
                uint32_t pk[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  __nv_bfloat162 h = __floats2bfloat162_rn(a8[2 * j], a8[2 * j + 1]);
                  pk[j] = *reinterpret_cast<uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(p.reduce_out + static_cast<int64_t>(row) * p.ldo + col) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
            if (epi_tid == 0) p.counters[mb * p.n_tiles + nb] = 0;  // ready for the next call
          }
        }
      }
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
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

// 2-D bf16 map over a row-major [outer, inner] matrix with row stride `ld` elements,
// box = 64 (inner) x box_outer rows, 128-byte swizzle, out-of-range reads as zero.
tp_status make_map(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
  auto enc = encoder();
  if (enc == nullptr) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return TP_OK;
}

template <int kEpi>
tp_status launch_gemm(const GemmParams& p, cudaStream_t stream) {
  const int sms = sm_count();
  if (sms <= 0) return fail(TP_ERR_CUDA, "cannot query the SM count of the current device");
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(tp_gemm_kernel<kEpi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBytes));
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(max dynamic shared memory)");
  const int64_t total = static_cast<int64_t>(p.n_groups) * p.m_tiles * p.n_tiles;
  if (total <= 0) return TP_OK;
  if (total > 0x7FFFFFFF) return fail(TP_ERR_UNSUPPORTED, "too many tiles (%lld)", (long long)total);
  const int grid = static_cast<int>(total < sms ? total : sms);
  tp_gemm_kernel<kEpi><<<grid, kThreads, kSmemBytes, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "GEMM kernel launch");
  return TP_OK;
}

inline int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

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
  if (act != TP_ACT_NONE && act != TP_ACT_GELU_TANH && act != TP_ACT_SWIGLU)
    return fail(TP_ERR_INVALID_ARG, "unknown activation %d", (int)act);
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

  GemmParams p{};
  st = make_map(&p.map_a[0], x, K, T, K, BM);
  if (st != TP_OK) return st;
  const int box_b = (act == TP_ACT_SWIGLU) ? BN / 2 : BN;
  for (int r = 0; r < tp_degree; ++r) {
    st = make_map(&p.map_b[r], w_shards[r], K, N_r, K, box_b);
    if (st != TP_OK) return st;
    p.out[r] = y_shards[r];
    p.bias[r] = bias_shards ? static_cast<const __nv_bfloat16*>(bias_shards[r]) : nullptr;
  }
  p.status = status;
  p.ldo = ldy;
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(n_out);
  p.n_groups = tp_degree;
  p.n_ksegs = 1;
  p.kblocks = ceil_div(K, BK);
  p.m_tiles = ceil_div(T, BM);
  p.n_tiles = ceil_div(n_out, (act == TP_ACT_SWIGLU) ? BN / 2 : BN);
  p.b_up_row = static_cast<int>(N_r / 2);
  p.rank_fastest = 0;
  p.a_shared = 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (act) {
    case TP_ACT_GELU_TANH: return launch_gemm<EPI_GELU>(p, s);
    case TP_ACT_SWIGLU: return launch_gemm<EPI_SWIGLU>(p, s);
    default: return launch_gemm<EPI_BF16>(p, s);
  }
}

size_t tp_rowwise_workspace_bytes(int tp_degree, int64_t T, int64_t N, tp_reduce_mode mode) {
  if (mode != TP_REDUCE_WORKSPACE || tp_degree < 1 || T <= 0 || N <= 0) return 0;
  const size_t partials = static_cast<size_t>(tp_degree) * static_cast<size_t>(T) * static_cast<size_t>(N) * 4;
  const size_t aligned = (partials + 255) & ~static_cast<size_t>(255);
  const size_t tiles = static_cast<size_t>((T + tp::BM - 1) / tp::BM) * static_cast<size_t>((N + tp::BN - 1) / tp::BN);
  return aligned + tiles * sizeof(int);
}

tp_status tp_linear_rowwise(const void* const* x_shards, const void* const* w_shards, const void* bias, int tp_degree,
                            int64_t T, int64_t K_r, int64_t N, tp_reduce_mode mode, void* workspace, size_t ws_bytes,
                            void* out, tp_stream_t stream) {
  using namespace tp;
  clear_error();
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
  if ((K_r % 8) != 0 || (N % 8) != 0)
    return fail(TP_ERR_ALIGNMENT, "K_r (%lld) and N (%lld) must be multiples of 8", (long long)K_r, (long long)N);
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

  GemmParams p{};
  for (int r = 0; r < tp_degree; ++r) {
    st = make_map(&p.map_a[r], x_shards[r], K_r, T, K_r, BM);
    if (st != TP_OK) return st;
    st = make_map(&p.map_b[r], w_shards[r], K_r, N, K_r, BN);
    if (st != TP_OK) return st;
  }
  p.status = status;
  p.M = static_cast<int>(T);
  p.N = static_cast<int>(N);
  p.kblocks = ceil_div(K_r, BK);
  p.m_tiles = ceil_div(T, BM);
  p.n_tiles = ceil_div(N, BN);
  p.a_shared = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (mode == TP_REDUCE_ACCUM) {
    p.out[0] = out;
    p.bias[0] = static_cast<const __nv_bfloat16*>(bias);
    p.ldo = N;
    p.n_groups = 1;
    p.n_ksegs = tp_degree;
    p.rank_fastest = 0;
    return launch_gemm<EPI_BF16>(p, s);
  }
  if (mode == TP_REDUCE_NONE) {
    for (int r = 0; r < tp_degree; ++r) {
      p.out[r] = static_cast<float*>(out) + static_cast<int64_t>(r) * T * N;
      p.bias[r] = (r == 0) ? static_cast<const __nv_bfloat16*>(bias) : nullptr;
    }
    p.ldo = N;
    p.n_groups = tp_degree;
    p.n_ksegs = 1;
    p.rank_fastest = 0;
    return launch_gemm<EPI_F32>(p, s);
  }
  // TP_REDUCE_WORKSPACE
  const size_t partial_bytes = (static_cast<size_t>(tp_degree) * T * N * 4 + 255) & ~static_cast<size_t>(255);
  p.ws = static_cast<float*>(workspace);
  p.counters = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + partial_bytes);
  p.reduce_out = static_cast<__nv_bfloat16*>(out);
  p.reduce_bias = static_cast<const __nv_bfloat16*>(bias);
  p.ldo = N;
  p.n_groups = tp_degree;
  p.n_ksegs = 1;
  p.rank_fastest = 1;
  cudaError_t e = cudaMemsetAsync(p.counters, 0, need - partial_bytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the tile counters");
  return launch_gemm<EPI_WS_REDUCE>(p, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Rowwise workspace mode for callers that cannot allocate: the scratch is a
// fixed array compiled into the library.  Host code must not pass the
// array's name to a kernel (on the host it is only a stand-in symbol); its
// device address is looked up once per device and cached.
// ---------------------------------------------------------------------------

namespace tp {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TP_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {nullptr};

tp_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(TP_ERR_UNSUPPORTED, "device index %d above 63", dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(built-in scratch)");
    g_noalloc_ptr[dev] = ptr;
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
