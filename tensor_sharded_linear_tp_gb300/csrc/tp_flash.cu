// Fused attention over the local heads of one or more ranks, head_dim 64 or 128 (tp_attention_heads*).
//
// diffusers "Tensor parallelism" page, §Colwise and rowwise: the colwise Q, K
// and V projections give each rank a subset of heads; each rank attends over
// its own heads.  This kernel computes, for 256 queries (two 128-query tiles)
// of one head of one rank,
//     O = softmax(Q K^T / sqrt(d)) V
// without writing scores to memory: scores and probabilities live in tensor
// memory (TMEM), K and V tiles stream through shared memory, both straight from
// the rank's QKV buffer (V is the B operand of P.V in its own [key][d] layout,
// MN-major, so it needs no transpose).
//
// CTA (320 threads, one per SM), grid = (query-tile pairs, heads, ranks):
//   warp 0       TMA producer: both Q tiles once, then K and V tiles of 128
//                keys, each through its own 2-stage ring (128-byte swizzle).
//   warp 1       one thread issues tcgen05.mma.  For tile g (0, 1) and key tile j:
//                  S_g = Q_g K_j^T        into TMEM columns [128g, 128g+128)
//                  O_g += P_g V_j         P_g read from TMEM as two bf16 terms,
//                                         P_hi (the first 64 columns of S_g's
//                                         region, bf16 pairs) and P_lo (the last
//                                         64), two products into O_g in columns
//                                         [256+d*g, 256+d*g+d) (d = head_dim)
//                Per tile the order is PV_g(j), then S_g(j+1): S_g(j+1) may only
//                overwrite P_g(j) after PV_g(j) read it, which the tensor core's
//                in-order execution of one thread's MMAs guarantees.
//   warps 2..5   softmax of tile 0; warps 6..9 softmax of tile 1 (one query row
//                per thread).  While one tile's softmax runs, the tensor core
//                works on the other tile's P.V and next S.  Per key tile: the
//                row of S into registers, its max; if the max exceeds the
//                running max m by more than 8 (log2 units), m is raised and O
//                and l rescale by 2^(m_old - m_new) (the whole warp does the TMEM
//                read-modify-write when any of its rows needs it); P =
//                2^(s*scale*log2e - m) stored to TMEM as P_hi (P truncated to bf16)
//                and P_lo = bf16(P - P_hi); l += sum of the unrounded P.  Finally O / l in bf16, staged in the
//                tile's (now idle) Q buffer and written by TMA stores.
// Keys past the end of the sequence are masked (weight 0); queries past it are
// computed on zero rows and clipped by the store.  Every wait is bounded (~2 s);
// a CTA that gives up records it in the library status word, lets its copies
// and MMAs drain, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "tp_internal.h"
#include "tp_ptx.cuh"

namespace tp {
namespace {

constexpr int FQ = 128;   // queries per tile; two tiles per CTA
constexpr int FK = 128;   // keys per tile
constexpr int KS = 2;     // K ring stages
constexpr int VS = 2;     // V ring stages
constexpr int kMaxRanks = 16;
constexpr uint32_t SUB = 16384;                         // 128 rows x 64 bf16, 128-byte swizzled
constexpr uint64_t kFlashWaitLimitNs = 2000000000ull;
constexpr int kThreads = 320;

struct FlashParams {
  CUtensorMap map_qk[kMaxRanks];  // rank r's QKV output [T, 3*H*d], boxes of 64 columns x 128 rows (Q, K, V)
  CUtensorMap map_o[kMaxRanks];   // rank r's attention output [T, H*d], boxes of 64 columns x 32 rows
  int T;
  int n_heads;
  float scale_log2e;
  unsigned int* status;
};

struct alignas(8) FlashCtrl {
  uint64_t q_full;
  uint64_t k_full[KS], k_empty[KS];
  uint64_t v_full[VS], v_empty[VS];
  uint64_t s_full[2];   // S_g(j) computed (and every MMA before it, PV_g(j-1) included)
  uint64_t p_full[2];   // P_g(j) stored in TMEM by the tile's 128 softmax threads
  uint64_t o_done[2];   // the tile's last P.V completed
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Shared-memory layout for head_dim kFD (64 or 128): a 128-row tile of Q, K or V is kFD / 64
// sub-tiles of 64 columns (d 0..63, then 64..127), each 128 rows x 128 B, 128-byte swizzled.
template <int kFD>
struct FlashDims {
  static_assert(kFD == 64 || kFD == 128, "the fused kernel covers head_dim 64 and 128");
  static constexpr int HALVES = kFD / 64;
  static constexpr uint32_t TILE = HALVES * SUB;
  static constexpr uint32_t OFF_Q = 0;                     // query tile g at g * TILE
  static constexpr uint32_t OFF_K = 2 * TILE;              // K stage s at OFF_K + s * TILE
  static constexpr uint32_t OFF_V = OFF_K + KS * TILE;     // V stage s, 128 key rows
  static constexpr uint32_t SMEM_DATA = OFF_V + VS * TILE; // 192 KB at head_dim 128, 96 KB at 64
  static constexpr size_t SMEM = 1024 + SMEM_DATA + sizeof(FlashCtrl);
  static_assert(SMEM <= 232448, "flash attention shared memory exceeds the per-CTA limit");
};

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

// Packed pairs of fp32 values for the sm_100 two-wide FMA/ADD instructions (half the
// instruction count of the scalar forms; the softmax is bound by instruction issue).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One key tile of one query row's online softmax (the row is this thread's TMEM lane): sv holds
// the row of S_g = Q K^T for key tile j (in registers).  Masks keys past T, updates the running
// max m (raising it, and rescaling l and O in TMEM, only when the tile's max exceeds it by more
// than 8 in log2 units), writes P = 2^(s*k - m) as bf16 pairs over the first 64 columns of the
// tile's S region and adds the unrounded P to l.  Warp-collective (TMEM access).
template <int FD>
__device__ __forceinline__ void softmax_tile(uint32_t (&sv)[FK], int j, int T, float k, uint32_t s_addr,
                                             uint32_t o_addr, float& m, float& l) {
  const int valid = min(FK, T - j * FK);
  if (valid < FK) {   // only the last key tile can be partial (warp-uniform)
#pragma unroll
    for (int t = 0; t < FK; ++t)
      if (t >= valid) sv[t] = __float_as_uint(-INFINITY);
  }
  float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int t = 0; t < FK; t += 2)
    mx[(t >> 1) & 3] = max3(mx[(t >> 1) & 3], __uint_as_float(sv[t]), __uint_as_float(sv[t + 1]));
  const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * k;
  // Raise the running max of the rows whose tile max exceeds it by more than 8: their
  // l and O (complete through key tile j-1: s_full_g(j) arrived after every MMA issued
  // before S_g(j), PV_g(j-1) included) scale by alpha = 2^(m_old - m_new).  The O
  // rescale is per warp (TMEM access is warp-collective): the whole warp does it when
  // any of its rows needs it, with alpha = 1 for the others.  It runs after P is stored,
  // when the S registers are free.
  bool rescale = false;
  float alpha = 1.0f;
  if (j == 0) {
    m = mt;
  } else {
    const bool need = mt > m + 8.0f;
    rescale = __any_sync(0xffffffffu, need);
    if (need) {
      alpha = ex2(m - mt);
      m = mt;
    }
    l *= alpha;
  }
  // P = 2^(s*k - m) as two bf16 terms, P = P_hi + P_lo: P_hi = P truncated to bf16 (its top
  // 16 bits) as pairs into the first 64 columns of S_g's region, P_lo = bf16(P - P_hi) into
  // the last 64.  The residual P - P_hi is exact in fp32 and below one bf16 ulp of P, so
  // P_hi + P_lo carries P to about 2^-16 relative instead of the 2^-9 of one bf16 term;
  // l += sum(P) (the unrounded values, four independent chains).  Masked keys give
  // 2^-inf = 0 in both terms.
  const uint64_t k2 = f2(k, k), nm2 = f2(-m, -m);
  uint64_t ls[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    // Packed in place: the pair for column t comes from entries 2t, 2t+1 (>= t), so
    // entry t of this half is already consumed when it is overwritten.  The whole row of
    // S is in registers, so the P_lo stores may overwrite S columns 64..127 in TMEM.
    uint32_t* pk = &sv[64 * half];
#pragma unroll
    for (int t8 = 0; t8 < 32; t8 += 8) {
      uint32_t lo[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int t = t8 + u;
        const uint64_t x2 = fma2(
            f2(__uint_as_float(sv[64 * half + 2 * t]), __uint_as_float(sv[64 * half + 2 * t + 1])), k2, nm2);
        float x0, x1;
        f2_split(x2, x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        const uint64_t pp = f2(p0, p1);
        ls[t & 3] = add2(ls[t & 3], pp);
        const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
        pk[t] = __byte_perm(u0, u1, 0x7632);   // the top halves: P_hi of p0 (low), of p1 (high)
        // -P_hi in one logic operation each (keep the top 16 bits, flip the sign), then both
        // residuals P - P_hi in one two-wide add (5 % faster than rounding P_hi and shifting
        // it back, measured on the block's attention).
        const uint64_t res = add2(pp, f2(__uint_as_float((u0 & 0xffff0000u) ^ 0x80000000u),
                                         __uint_as_float((u1 & 0xffff0000u) ^ 0x80000000u)));
        float r0, r1;
        f2_split(res, r0, r1);
        lo[u] = pack_bf16(r0, r1);
      }
      ptx::tmem_st_32x32b_x8(s_addr + 64 + 32 * half + t8, lo);
    }
    ptx::tmem_st_32x32b_x32(s_addr + 32 * half, *reinterpret_cast<uint32_t(*)[32]>(pk));
  }
  if (rescale) {
#pragma unroll 1
    for (int c = 0; c < FD; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(o_addr + c, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * alpha);
      ptx::tmem_st_32x32b_x32(o_addr + c, v);
    }
  }
  ptx::tmem_st_wait();
  {
    float a0, a1;
    f2_split(add2(add2(ls[0], ls[1]), add2(ls[2], ls[3])), a0, a1);
    l += a0 + a1;
  }
}

// The tile's output rows of this warp: O / l in bf16, staged in the (idle) Q buffer `qbuf` of
// the tile and written by two TMA stores of 32 rows x 64 columns (rows past T are skipped or
// clipped).  Warp-collective.
template <int FD>
__device__ __forceinline__ void write_output(const CUtensorMap& map_o, uint32_t o_addr, float l, uint32_t qbuf,
                                             int q, int lane, int h, int row0, int T) {
  // Epilogue: O / l in bf16, staged in the tile's Q buffer (idle: every S MMA of this tile
  // completed before o_done), written by TMA stores of 32 rows x 64 columns.
  const float inv = 1.0f / l;
  const uint32_t stage = qbuf + static_cast<uint32_t>(q) * (FD / 64) * 4096;  // 32 rows x FD bf16 per warp
#pragma unroll 1
  for (int c = 0; c < FD; c += 32) {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(o_addr + c, v);
    ptx::tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) pk[t] = pack_bf16(__uint_as_float(v[2 * t]) * inv, __uint_as_float(v[2 * t + 1]) * inv);
    const uint32_t dst = stage + (c >> 6) * 4096 + static_cast<uint32_t>(lane) * 128;
    const int chunk0 = (c & 63) >> 3;
#pragma unroll
    for (int t = 0; t < 4; ++t)
      ptx::st_shared_v4(dst + (static_cast<uint32_t>((chunk0 + t) ^ (lane & 7)) << 4), pk[4 * t], pk[4 * t + 1],
                        pk[4 * t + 2], pk[4 * t + 3]);
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < T) {
#pragma unroll
    for (int h2 = 0; h2 < FD / 64; ++h2) ptx::tma_store_2d(&map_o, stage + h2 * 4096, h * FD + 64 * h2, row0);
    ptx::bulk_commit();
    ptx::bulk_wait_all();
  }
  __syncwarp();
}

template <int kFD>
__global__ void __launch_bounds__(kThreads, 1) tp_flash_kernel(const __grid_constant__ FlashParams p) {
  using D = FlashDims<kFD>;
  constexpr int FD = kFD;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FlashCtrl* ctl = reinterpret_cast<FlashCtrl*>(base + D::SMEM_DATA);
  volatile int* abort_flag = &ctl->abort;
  const uint32_t sbase = ptx::smem_addr(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, rank = blockIdx.z;
  const int q0 = blockIdx.x * 2 * FQ;
  const int nkv = (p.T + FK - 1) / FK;
  const CUtensorMap* map_qk = &p.map_qk[rank];
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&ctl->q_full), 1);
    for (int i = 0; i < KS; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->k_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->k_empty[i]), 1);
    }
    for (int i = 0; i < VS; ++i) {
      ptx::mbar_init(ptx::smem_addr(&ctl->v_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->v_empty[i]), 1);
    }
    for (int g = 0; g < 2; ++g) {
      ptx::mbar_init(ptx::smem_addr(&ctl->s_full[g]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl->p_full[g]), 128);
      ptx::mbar_init(ptx::smem_addr(&ctl->o_done[g]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
    ctl->abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_wait();  // the previous kernel's writes (Q, K, V) are complete and visible from here on

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      ptx::prefetch_tensormap(map_qk);
      const uint32_t qf = ptx::smem_addr(&ctl->q_full);
      ptx::mbar_arrive_expect_tx(qf, 2 * D::TILE);
      for (int g = 0; g < 2; ++g)
        for (int h2 = 0; h2 < D::HALVES; ++h2)
          ptx::tma_load_2d(sbase + D::OFF_Q + g * D::TILE + h2 * SUB, map_qk, qf, h * FD + 64 * h2, q0 + g * FQ);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int ks = j % KS, vs = j % VS;
        if (!fwait(ptx::smem_addr(&ctl->k_empty[ks]), ((j / KS) & 1) ^ 1u, abort_flag, p.status)) break;
        const uint32_t kf = ptx::smem_addr(&ctl->k_full[ks]);
        const uint32_t kdst = sbase + D::OFF_K + ks * D::TILE;
        const int kx = (p.n_heads + h) * FD;
        ptx::mbar_arrive_expect_tx(kf, D::TILE);
        for (int h2 = 0; h2 < D::HALVES; ++h2) ptx::tma_load_2d(kdst + h2 * SUB, map_qk, kf, kx + 64 * h2, j * FK);
        ++k_issued;
        if (!fwait(ptx::smem_addr(&ctl->v_empty[vs]), ((j / VS) & 1) ^ 1u, abort_flag, p.status)) break;
        const uint32_t vf = ptx::smem_addr(&ctl->v_full[vs]);
        const uint32_t vdst = sbase + D::OFF_V + vs * D::TILE;
        const int vx = (2 * p.n_heads + h) * FD;
        ptx::mbar_arrive_expect_tx(vf, D::TILE);
        for (int h2 = 0; h2 < D::HALVES; ++h2) ptx::tma_load_2d(vdst + h2 * SUB, map_qk, vf, vx + 64 * h2, j * FK);
        ++v_issued;
      }
      // Let every copy land before the CTA can exit.
      fwait(qf, 0, abort_flag, p.status, true);
      for (int j = (k_issued > KS ? k_issued - KS : 0); j < k_issued; ++j)
        fwait(ptx::smem_addr(&ctl->k_full[j % KS]), (j / KS) & 1, abort_flag, p.status, true);
      for (int j = (v_issued > VS ? v_issued - VS : 0); j < v_issued; ++j)
        fwait(ptx::smem_addr(&ctl->v_full[j % VS]), (j / VS) & 1, abort_flag, p.status, true);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(FQ, FK);   // S: M 128 queries, N 128 keys
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(FQ, FD) | ptx::kIdescMnMajorB;  // P.V: N = head_dim;
                                                                                      // V as stored, d contiguous
      auto issue_s = [&](int g, int j) {
        const uint32_t kb = sbase + D::OFF_K + (j % KS) * D::TILE;
        const uint32_t qb = sbase + D::OFF_Q + g * D::TILE;
#pragma unroll
        for (int kk = 0; kk < FD / 16; ++kk) {
          const uint32_t sub = (kk >> 2) * SUB, k4 = 2u * (kk & 3);
          ptx::umma_bf16(tmem + g * FK, ptx::sw128_kmajor_desc(qb + sub) + k4, ptx::sw128_kmajor_desc(kb + sub) + k4,
                         idesc, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int g, int j) {
        // B = V tile: 128 key rows of 128 B per 64-wide d half; the halves are SUB apart (LBO),
        // 8-key groups 1024 B apart (SBO); 16 keys per MMA = 2048 B of rows.
        const uint32_t vb = sbase + D::OFF_V + (j % VS) * D::TILE;
        const uint64_t vdesc = ptx::sw128_mnmajor_desc(vb, SUB, 1024);
        // O_g += P_hi V, then O_g += P_lo V (P_lo in columns 64..127 of the region).
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          ptx::umma_bf16_ts(tmem + 2 * FK + g * FD, tmem + g * FK + kk * 8, vdesc + (kk & 7) * (2048u >> 4),
                            idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
      };
      bool ok = fwait(ptx::smem_addr(&ctl->q_full), 0, abort_flag, p.status) &&
                fwait(ptx::smem_addr(&ctl->k_full[0]), 0, abort_flag, p.status);
      if (ok) {
        ptx::tc_fence_after();
        for (int g = 0; g < 2; ++g) {
          issue_s(g, 0);
          ptx::umma_commit(ptx::smem_addr(&ctl->s_full[g]));
        }
        ptx::umma_commit(ptx::smem_addr(&ctl->k_empty[0]));
      }
      for (int j = 0; ok && j < nkv; ++j) {
        if (!fwait(ptx::smem_addr(&ctl->v_full[j % VS]), (j / VS) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const bool more = j + 1 < nkv;
        for (int g = 0; g < 2 && ok; ++g) {
          if (!fwait(ptx::smem_addr(&ctl->p_full[g]), j & 1, abort_flag, p.status) ||
              (more && g == 0 &&
               !fwait(ptx::smem_addr(&ctl->k_full[(j + 1) % KS]), ((j + 1) / KS) & 1, abort_flag, p.status))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_pv(g, j);
          if (more) {
            issue_s(g, j + 1);
            ptx::umma_commit(ptx::smem_addr(&ctl->s_full[g]));
          } else {
            ptx::umma_commit(ptx::smem_addr(&ctl->o_done[g]));
          }
        }
        if (!ok) break;
        ptx::umma_commit(ptx::smem_addr(&ctl->v_empty[j % VS]));
        if (more) ptx::umma_commit(ptx::smem_addr(&ctl->k_empty[(j + 1) % KS]));
      }
      ptx::umma_commit(ptx::smem_addr(&ctl->drain));
      fwait(ptx::smem_addr(&ctl->drain), 0, abort_flag, p.status, true);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int g = (warp - 2) >> 2;            // query tile of this warpgroup
    const int q = warp & 3;                   // TMEM lane quarter: rows [32q, 32q+32) of the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + g * FK;        // S_g, then P_g in its first 64 columns
    const uint32_t o_addr = tmem + lane_base + 2 * FK + g * FD;
    const float k = p.scale_log2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv && ok; ++j) {
      // Every wait's outcome is made warp-uniform: the TMEM loads and stores below are
      // warp-collective and must never run in a partial warp.
      if (!__all_sync(0xffffffffu, fwait(ptx::smem_addr(&ctl->s_full[g]), j & 1, abort_flag, p.status))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t sv[FK];
      ptx::tmem_ld_32x32b_x32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      ptx::tmem_ld_32x32b_x32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      ptx::tmem_ld_32x32b_x32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[64]));
      ptx::tmem_ld_32x32b_x32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sv[96]));
      ptx::tmem_ld_wait();
      softmax_tile<FD>(sv, j, p.T, k, s_addr, o_addr, m, l);
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&ctl->p_full[g]));
    }
    if (ok && __all_sync(0xffffffffu, fwait(ptx::smem_addr(&ctl->o_done[g]), 0, abort_flag, p.status))) {
      ptx::tc_fence_after();
      write_output<FD>(p.map_o[rank], o_addr, l, sbase + D::OFF_Q + g * D::TILE, q, lane, h, q0 + g * FQ + q * 32,
                       p.T);
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Fused attention for head_dim 64 or 128 over n_ranks ranks in one launch (see the file comment).
template <int kFD>
tp_status flash_attention(int n_ranks, const void* const* qkv, int64_t ld_qkv, int64_t T, int n_heads,
                          void* const* out, int64_t ldo, float scale_log2e, cudaStream_t stream) {
  using D = FlashDims<kFD>;
  if (n_ranks < 1 || n_ranks > kMaxRanks)
    return fail(TP_ERR_UNSUPPORTED, "fused attention over %d ranks in one launch (at most %d)", n_ranks, kMaxRanks);
  unsigned int* status = status_word();
  if (status == nullptr) return fail(TP_ERR_CUDA, "cannot locate the kernel status word");
  FlashParams prm{};
  const int64_t width = static_cast<int64_t>(n_heads) * kFD;
  for (int r = 0; r < n_ranks; ++r) {
    tp_status st = encode_bf16_2d(&prm.map_qk[r], qkv[r], 3 * width, T, ld_qkv, 64, 128, true);
    if (st == TP_OK) st = encode_bf16_2d(&prm.map_o[r], out[r], width, T, ldo, 64, 32, true);
    if (st != TP_OK) return st;
  }
  prm.T = static_cast<int>(T);
  prm.n_heads = n_heads;
  prm.scale_log2e = scale_log2e;
  prm.status = status;
  // The dynamic shared-memory limit, raised once per device (a failure is retried next time).
  static std::atomic<bool> raised[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!raised[dev & 63].load(std::memory_order_acquire)) {
    cudaError_t err = cudaFuncSetAttribute(tp_flash_kernel<kFD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(D::SMEM));
    if (err != cudaSuccess) return cuda_fail(err, "cudaFuncSetAttribute(flash attention)");
    raised[dev & 63].store(true, std::memory_order_release);
  }
  dim3 grid(static_cast<unsigned>((T + 2 * FQ - 1) / (2 * FQ)), static_cast<unsigned>(n_heads),
            static_cast<unsigned>(n_ranks));
  cudaError_t e = launch_pdl(tp_flash_kernel<kFD>, grid, dim3(kThreads), D::SMEM, stream, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "flash attention launch");
  return TP_OK;
}

}  // namespace

tp_status flash_attention_fused(int head_dim, int n_ranks, const void* const* qkv, int64_t ld_qkv, int64_t T,
                                int n_heads, void* const* out, int64_t ldo, float scale_log2e, cudaStream_t stream) {
  if (head_dim == 128)
    return flash_attention<128>(n_ranks, qkv, ld_qkv, T, n_heads, out, ldo, scale_log2e, stream);
  if (head_dim == 64)
    return flash_attention<64>(n_ranks, qkv, ld_qkv, T, n_heads, out, ldo, scale_log2e, stream);
  return fail(TP_ERR_UNSUPPORTED, "the fused attention covers head_dim 64 and 128, not %d", head_dim);
}

}  // namespace tp
