// Fused attention over a rank's local heads for head_dim 128 (tp_attention_heads).
//
// diffusers "Tensor parallelism" page, §Colwise and rowwise: the colwise Q, K
// and V projections give each rank a subset of heads; each rank attends over
// its own heads.  This kernel computes, for one 128-query tile of one head,
//     O = softmax(Q K^T / sqrt(d)) V
// without writing scores to memory: scores live in tensor memory, the
// probabilities in shared memory.
//
// CTA (192 threads, one per SM), grid = (query tiles, heads):
//   warp 0      TMA producer: Q once (128 x 128), then K and V^T tiles of 128
//               keys through a 2-stage ring (128-byte swizzle).
//   warp 1      one thread issues tcgen05.mma: S_j = Q K_j^T into one of two
//               TMEM score buffers (columns [0,128) and [128,256)), and
//               O += P_j V_j into the TMEM output accumulator (columns [256,384)).
//               The S MMA of tile j+1 runs while the softmax warps work on j.
//   warps 2..5  online softmax, one query row per thread: row max of S_j,
//               P_j = 2^(s*scale*log2e - m) written as bf16 to shared memory
//               in the MMA's K-major swizzled layout, running sum l.  The
//               running max m is raised (and O rescaled in TMEM by 2^(m_old -
//               m_new)) only when a tile's max exceeds it by more than 8 (in
//               log2 units), so P stays below 2^8; the final O / l uses the
//               same m, so the result is exact either way.  Then O / l is
//               rounded to bf16 and written by TMA stores.
// Keys past the end of the sequence are masked (weight 0); queries past it are
// computed and clipped by the store.  Every wait is bounded (~2 s).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tp_internal.h"
#include "tp_ptx.cuh"

namespace tp {
namespace {

constexpr int FD = 128;   // head_dim
constexpr int FQ = 128;   // queries per CTA
constexpr int FK = 128;   // keys per tile
constexpr uint32_t SUB = 16384;             // one 128-row x 64-element bf16 swizzled sub-tile
constexpr uint32_t OFF_Q = 0;               // Q: 2 sub-tiles (d 0..63, 64..127)
constexpr uint32_t OFF_KV = 32768;          // stage s: K (2 sub-tiles) then V^T (2 sub-tiles), 64 KB
constexpr uint32_t OFF_P = 32768 + 2 * 65536;  // P buffer b: 2 sub-tiles (keys 0..63, 64..127), 32 KB each
constexpr uint32_t SMEM_DATA = OFF_P + 2 * 32768;
constexpr uint64_t kFlashWaitLimitNs = 2000000000ull;

struct FlashParams {
  CUtensorMap map_qk;  // the rank's QKV output [T, 3*H*d], boxes of 64 columns x 128 rows
  CUtensorMap map_vt;  // V^T [H*d, T], boxes of 64 keys x 128 rows
  CUtensorMap map_o;   // attention output [T, H*d] (row stride ldo), boxes of 64 columns x 32 rows
  int T;
  int n_heads;
  float scale_log2e;
  unsigned int* status;
};

struct alignas(8) FlashCtrl {
  uint64_t q_full;
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_free[2];
  uint64_t o_full, drain;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kFlashSmem = 1024 + SMEM_DATA + sizeof(FlashCtrl);

__device__ __forceinline__ bool fwait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned int* status,
                                      bool ignore_abort = false) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (!ignore_abort && *abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > kFlashWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(status, TP_DEVSTATUS_TIMEOUT);
        return false;
      }
    }
  }
}

// 2^x with the hardware's approximate exponential (one MUFU operation); x <= 8 here.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(192, 1) tp_flash_kernel(const __grid_constant__ FlashParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FlashCtrl* ctl = reinterpret_cast<FlashCtrl*>(base + SMEM_DATA);
  volatile int* abort_flag = &ctl->abort;
  const uint32_t sbase = ptx::smem_addr(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y;
  const int q0 = qt * FQ;
  const int nkv = (p.T + FK - 1) / FK;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&ctl->q_full), 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->kv_empty[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->s_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->s_free[i]), 128);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_full[i]), 128);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_free[i]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->o_full), 1);
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      const uint32_t qf = ptx::smem_addr(&ctl->q_full);
      ptx::mbar_arrive_expect_tx(qf, 2 * SUB);
      ptx::tma_load_2d(sbase + OFF_Q, &p.map_qk, qf, h * FD, q0);
      ptx::tma_load_2d(sbase + OFF_Q + SUB, &p.map_qk, qf, h * FD + 64, q0);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!fwait(ptx::smem_addr(&ctl->kv_empty[s]), ph ^ 1u, abort_flag, p.status)) break;
        const uint32_t full = ptx::smem_addr(&ctl->kv_full[s]);
        const uint32_t kv = sbase + OFF_KV + s * 65536;
        ptx::mbar_arrive_expect_tx(full, 4 * SUB);
        const int kx = (p.n_heads + h) * FD;
        ptx::tma_load_2d(kv, &p.map_qk, full, kx, j * FK);
        ptx::tma_load_2d(kv + SUB, &p.map_qk, full, kx + 64, j * FK);
        ptx::tma_load_2d(kv + 2 * SUB, &p.map_vt, full, j * FK, h * FD);
        ptx::tma_load_2d(kv + 3 * SUB, &p.map_vt, full, j * FK + 64, h * FD);
        ++issued;
      }
      // Let every copy land before the CTA can exit.
      fwait(qf, 0, abort_flag, p.status, true);
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
        fwait(ptx::smem_addr(&ctl->kv_full[j & 1]), (j >> 1) & 1, abort_flag, p.status, true);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(FQ, FK);
      bool ok = fwait(ptx::smem_addr(&ctl->q_full), 0, abort_flag, p.status);
      for (int j = 0; ok && j <= nkv; ++j) {
        if (j < nkv) {
          const int s = j & 1;
          const uint32_t ph = (j >> 1) & 1;
          if (!fwait(ptx::smem_addr(&ctl->kv_full[s]), ph, abort_flag, p.status) ||
              !fwait(ptx::smem_addr(&ctl->s_free[s]), ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t kbase = sbase + OFF_KV + s * 65536;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t sub = (kk >> 2) * SUB, k4 = 2u * (kk & 3);
            ptx::umma_bf16(tmem + s * FK, ptx::sw128_kmajor_desc(sbase + OFF_Q + sub) + k4,
                           ptx::sw128_kmajor_desc(kbase + sub) + k4, idesc, kk > 0 ? 1u : 0u);
          }
          ptx::umma_commit(ptx::smem_addr(&ctl->s_full[s]));
        }
        if (j >= 1) {
          const int i = j - 1, b = i & 1;
          if (!fwait(ptx::smem_addr(&ctl->p_full[b]), (i >> 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t pbase = sbase + OFF_P + b * 32768;
          const uint32_t vbase = sbase + OFF_KV + b * 65536 + 2 * SUB;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t sub = (kk >> 2) * SUB, k4 = 2u * (kk & 3);
            ptx::umma_bf16(tmem + 2 * FK, ptx::sw128_kmajor_desc(pbase + sub) + k4,
                           ptx::sw128_kmajor_desc(vbase + sub) + k4, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::umma_commit(ptx::smem_addr(&ctl->p_free[b]));
          ptx::umma_commit(ptx::smem_addr(&ctl->kv_empty[b]));
        }
      }
      if (ok) ptx::umma_commit(ptx::smem_addr(&ctl->o_full));
      ptx::umma_commit(ptx::smem_addr(&ctl->drain));
      fwait(ptx::smem_addr(&ctl->drain), 0, abort_flag, p.status, true);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;                 // TMEM lane quarter: query rows [32q, 32q+32)
    const int row = q * 32 + lane;          // this thread's query row inside the tile
    const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float k = p.scale_log2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      const int b = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      // Every wait's outcome is made warp-uniform: the TMEM loads and stores below are
      // warp-collective and must never run in a partial warp.
      if (!__all_sync(0xffffffffu, fwait(ptx::smem_addr(&ctl->s_full[b]), ph, abort_flag, p.status))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int valid = min(FK, p.T - j * FK);
      const uint32_t sbuf = trow + b * FK;
      const bool full = (valid == FK);   // only the last key tile can be partial (warp-uniform)
      // Pass 1: the tile's row max (scaled, log2 units), four independent chains.
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int c = 0; c < FK; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(sbuf + c, v);
        ptx::tmem_ld_wait();
        if (full) {
#pragma unroll
          for (int t = 0; t < 32; ++t) mx[t & 3] = fmaxf(mx[t & 3], __uint_as_float(v[t]));
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (c + t < valid) mx[t & 3] = fmaxf(mx[t & 3], __uint_as_float(v[t]));
        }
      }
      float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * k;
      if (j == 0) {
        m = mt;
      } else {
        // Raise the running max of the rows whose tile max exceeds it by more than 8:
        // their O (complete through tile j-1) and l scale by 2^(m - mt).  The decision is
        // per row but the TMEM read-modify-write is per warp, so the whole warp does it
        // when any of its rows needs it (alpha = 1 for the others).
        const bool need = mt > m + 8.0f;
        if (__any_sync(0xffffffffu, need)) {
          if (!__all_sync(0xffffffffu, fwait(ptx::smem_addr(&ctl->p_free[(j - 1) & 1]), ((j - 1) >> 1) & 1,
                                             abort_flag, p.status))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const float alpha = need ? ex2(m - mt) : 1.0f;
          l *= alpha;
          if (need) m = mt;
#pragma unroll 1
          for (int c = 0; c < FD; c += 32) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(trow + 2 * FK + c, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
            ptx::tmem_st_32x32b_x32(trow + 2 * FK + c, v);
          }
          ptx::tmem_st_wait();
        }
      }
      // P buffer b is free once the P.V MMA of tile j-2 has completed.
      if (!__all_sync(0xffffffffu, fwait(ptx::smem_addr(&ctl->p_free[b]), ph ^ 1u, abort_flag, p.status))) {
        ok = false;
        break;
      }
      // Pass 2: P = 2^(s*k - m) as bf16 into the swizzled K-major P tile; l += sum(P)
      // (the sum of the unrounded values, four independent chains).
      const uint32_t pbase = sbase + OFF_P + b * 32768;
      const float negm = -m;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int c = 0; c < FK; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(sbuf + c, v);
        ptx::tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          float p0 = ex2(fmaf(__uint_as_float(v[2 * t]), k, negm));
          float p1 = ex2(fmaf(__uint_as_float(v[2 * t + 1]), k, negm));
          if (!full) {
            p0 = (c + 2 * t < valid) ? p0 : 0.f;
            p1 = (c + 2 * t + 1 < valid) ? p1 : 0.f;
          }
          ls[t & 3] += p0 + p1;
          __nv_bfloat162 hp = __floats2bfloat162_rn(p0, p1);
          pk[t] = *reinterpret_cast<uint32_t*>(&hp);
        }
        const uint32_t sub = pbase + (c >> 6) * SUB + static_cast<uint32_t>(row) * 128;
        const int chunk0 = (c & 63) >> 3;  // 16-byte piece index of column c within the 64-key row
#pragma unroll
        for (int t = 0; t < 4; ++t)
          ptx::st_shared_v4(sub + (static_cast<uint32_t>((chunk0 + t) ^ (row & 7)) << 4), pk[4 * t], pk[4 * t + 1],
                            pk[4 * t + 2], pk[4 * t + 3]);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&ctl->s_free[b]));
      ptx::fence_proxy_async_smem();  // P (generic-proxy writes) becomes visible to the MMA
      ptx::mbar_arrive(ptx::smem_addr(&ctl->p_full[b]));
    }
    if (ok && __all_sync(0xffffffffu, fwait(ptx::smem_addr(&ctl->o_full), 0, abort_flag, p.status))) {
      ptx::tc_fence_after();
      // Epilogue: O / l in bf16, staged in the (now idle) Q buffer, written by TMA stores.
      const float inv = 1.0f / l;
      const uint32_t stage = sbase + OFF_Q + static_cast<uint32_t>(q) * 8192;
#pragma unroll 1
      for (int c = 0; c < FD; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(trow + 2 * FK + c, v);
        ptx::tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          __nv_bfloat162 ho =
              __floats2bfloat162_rn(__uint_as_float(v[2 * t]) * inv, __uint_as_float(v[2 * t + 1]) * inv);
          pk[t] = *reinterpret_cast<uint32_t*>(&ho);
        }
        const uint32_t dst = stage + (c >> 6) * 4096 + static_cast<uint32_t>(lane) * 128;
        const int chunk0 = (c & 63) >> 3;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          ptx::st_shared_v4(dst + (static_cast<uint32_t>((chunk0 + t) ^ (lane & 7)) << 4), pk[4 * t], pk[4 * t + 1],
                            pk[4 * t + 2], pk[4 * t + 3]);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        ptx::tma_store_2d(&p.map_o, stage, h * FD, q0 + q * 32);
        ptx::tma_store_2d(&p.map_o, stage + 4096, h * FD + 64, q0 + q * 32);
        ptx::bulk_commit();
        ptx::bulk_wait_all();
      }
      __syncwarp();
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Fused attention for head_dim 128 (see the file comment).  vt: V^T [n_heads*128, T].
tp_status flash_attention_d128(const void* qkv, int64_t ld_qkv, int64_t T, int n_heads, const void* vt, void* out,
                               int64_t ldo, float scale_log2e, cudaStream_t stream) {
  unsigned int* status = status_word();
  if (status == nullptr) return fail(TP_ERR_CUDA, "cannot locate the kernel status word");
  FlashParams prm{};
  const int64_t width = static_cast<int64_t>(n_heads) * FD;
  tp_status st = encode_bf16_2d(&prm.map_qk, qkv, 3 * width, T, ld_qkv, 64, 128, true);
  if (st == TP_OK) st = encode_bf16_2d(&prm.map_vt, vt, T, width, T, 64, 128, true);
  if (st == TP_OK) st = encode_bf16_2d(&prm.map_o, out, width, T, ldo, 64, 32, true);
  if (st != TP_OK) return st;
  prm.T = static_cast<int>(T);
  prm.n_heads = n_heads;
  prm.scale_log2e = scale_log2e;
  prm.status = status;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    err = cudaFuncSetAttribute(tp_flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kFlashSmem));
  });
  if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(flash attention)");
  dim3 grid(static_cast<unsigned>((T + FQ - 1) / FQ), static_cast<unsigned>(n_heads));
  tp_flash_kernel<<<grid, 192, kFlashSmem, stream>>>(prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "flash attention launch");
  return TP_OK;
}

}  // namespace tp
