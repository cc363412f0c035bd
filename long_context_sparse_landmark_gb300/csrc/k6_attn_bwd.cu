// K6: backward pass of window + landmark attention (bf16 Q/K/V/dO, d = 128)
// on the tensor cores -- the gradients that training with the sparse
// pattern needs ("Training at 1M+ Token Context: Ring Attention, YaRN,
// NTK-Aware Scaling GPU Cost", Block-Sparse Flash Attention paragraph,
// trains with block-sparse attention).  With A(i) the attended set of row
// i (window keys, visible landmarks), P_ia = exp(scale <q_i, k_a> - lse_i)
// recomputed from the forward's lse:
//   D_i = <dO_i, O_i>,  dS_ia = P_ia (<dO_i, v_a> - D_i),
//   dQ_i = scale sum_a dS_ia k_a,  dK_a = scale sum_i dS_ia q_i,
//   dV_a = sum_i P_ia dO_i,
// and the gradient of a landmark (a block mean) reaches each of its B
// tokens divided by B.
//
// Launches, in stream order:
//   1. bwd_preprocess_kernel: D [Hq, n] (fp32);
//   2. bwd_dkdv_tc_kernel, landmark mode: per (landmark tile, KV head,
//      query chunk) partial dK_lm / dV_lm over the rows that see the
//      landmarks (up to all n rows per landmark, hence the chunks);
//   3. lm_grad_reduce_kernel: sums the chunks (fp32 [2][G][Hkv][d]);
//   4. bwd_dkdv_tc_kernel, window mode: per (128-key tile, KV head) over the
//      query tiles whose windows reach it and every head of the group; the
//      epilogue adds the token's share of its landmark gradient and writes
//      dK, dV;
//   5. bwd_dq_tc_kernel: per (128-row query tile, head) over the landmark
//      and window key tiles, as the forward.
// Each tensor-core kernel: warps 0-3 elementwise (one TMEM lane = one row
// each), warp 4 TMA producer, warp 5 TMEM allocation and MMA issue.  Per
// iteration the two score-like MMAs run, the elementwise warps turn them
// into bf16 P / dS in the same TMEM columns, and the two gradient MMAs
// accumulate in TMEM; tcgen05 MMAs from one thread execute in issue order,
// so the next iteration's score MMAs may be issued right after.  Every wait
// is bounded; a wait that runs out aborts the CTA cleanly.
#include <cuda.h>
#include <math.h>
#include <string.h>

#include "msa_common.cuh"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"
#include "tma_map.h"

namespace msa {
namespace {

constexpr int kD = 128;
constexpr int kT = 128;                      // rows per tile (queries or keys)
constexpr int kChunkBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kChunkBytes;  // 128 rows x 128 bf16
constexpr uint32_t kTileLo = kTileBytes >> 4;
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory of both kernels: a fixed pair of tiles (dQ: Q, dO; dK/dV:
// K, V) and a 2-stage ring of tile pairs (dQ: K, V; dK/dV: Q, dO).
constexpr int kOffFixA = 0;
constexpr int kOffFixB = kTileBytes;
constexpr int kOffRingA = 2 * kTileBytes;                 // 2 stages
constexpr int kOffRingB = kOffRingA + 2 * kTileBytes;     // 2 stages
constexpr int kOffBar = kOffRingB + 2 * kTileBytes;       // 192 KB
enum {
  BAR_FIX = 0,      // fixed tiles landed
  BAR_FULL0 = 1,    // ring stage b landed (1, 2)
  BAR_EMPTY0 = 3,   // ring stage b consumed (3, 4)
  BAR_SF = 5,       // score-like MMAs done
  BAR_EF = 6,       // elementwise results written (4 warp arrivals)
  BAR_ACC = 7,      // gradient accumulators final
  BAR_CLEAN = 8,
  kNumBars = 9
};
constexpr int kOffStats = kOffBar + 8 * kNumBars;  // dK/dV: [4 warps][lse, D][128] fp32
constexpr int kOffTmemSlot = kOffStats + 4 * 2 * kT * 4;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;

struct BwdParams {
  CUtensorMap tm_q, tm_do, tm_k, tm_v, tm_klm, tm_vlm;
  const float* lse;   // [Hq, n]
  const float* D;     // [Hq, n]
  void* dq;           // [n, Hq, d]
  void* dk;           // [n, Hkv, d]
  void* dv;
  float* lm_part;     // [chunks][2][G][Hkv][d]
  const float* lm_grad;  // [2][G][Hkv][d]
  int64_t n, window, block;
  int Hq, Hkv, G, group, grad_bf16;
  int lm_mode, lm_chunks, chunk_tiles;
  float scale, scale_log2;
  int* status;
  uint64_t wait_ns;
};

__device__ __forceinline__ void store_row(void* base, int64_t off, const float (&o)[32], float w,
                                          int bf16) {
  if (bf16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint4 q4;
      q4.x = ptx::pack_bf16x2(o[8 * v + 0] * w, o[8 * v + 1] * w);
      q4.y = ptx::pack_bf16x2(o[8 * v + 2] * w, o[8 * v + 3] * w);
      q4.z = ptx::pack_bf16x2(o[8 * v + 4] * w, o[8 * v + 5] * w);
      q4.w = ptx::pack_bf16x2(o[8 * v + 6] * w, o[8 * v + 7] * w);
      dst[v] = q4;
    }
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int v = 0; v < 8; ++v)
      dst[v] = make_float4(o[4 * v] * w, o[4 * v + 1] * w, o[4 * v + 2] * w, o[4 * v + 3] * w);
  }
}

// Shared set-up of both kernels: barriers, TMEM (512 columns).
__device__ __forceinline__ uint32_t bwd_setup(uint8_t* smem, uint32_t sb, int warp) {
  if (threadIdx.x == 0) {
    ptx::mbar_init(sb + kOffBar + 8 * BAR_FIX, 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(sb + kOffBar + 8 * (BAR_FULL0 + b), 1);
      ptx::mbar_init(sb + kOffBar + 8 * (BAR_EMPTY0 + b), 1);
    }
    ptx::mbar_init(sb + kOffBar + 8 * BAR_SF, 1);
    ptx::mbar_init(sb + kOffBar + 8 * BAR_EF, 4);
    ptx::mbar_init(sb + kOffBar + 8 * BAR_ACC, 1);
    ptx::mbar_init(sb + kOffBar + 8 * BAR_CLEAN, 1);
    *reinterpret_cast<volatile int*>(smem + kOffAbort) = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(smem + kOffTmemSlot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
}

__device__ __forceinline__ void bwd_teardown(uint32_t tmem, int warp) {
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Producer: the fixed pair once, then `iters` ring pairs; `coord(it, &map_a,
// &map_b, &y_a, &y_b, &row)` names the tensors and coordinates of pair it.
template <typename Coord>
__device__ __forceinline__ void produce(uint32_t sb, const CUtensorMap* fa, const CUtensorMap* fb,
                                        int fy, int frow, int iters, Coord coord,
                                        const WaitCtl& ctl, int* status) {
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };
  ptx::mbar_arrive_expect_tx(bar(BAR_FIX), 2 * kTileBytes);
  for (int ch = 0; ch < 2; ++ch) {
    ptx::tma_load_3d(sb + kOffFixA + ch * kChunkBytes, fa, bar(BAR_FIX), ch * 64, fy, frow);
    ptx::tma_load_3d(sb + kOffFixB + ch * kChunkBytes, fb, bar(BAR_FIX), ch * 64, fy, frow);
  }
  int issued = 0;
  for (int it = 0; it < iters; ++it) {
    const int b = it & 1;
    if (it >= 2 && !wait_bar(bar(BAR_EMPTY0 + b), ((it >> 1) - 1) & 1, ctl)) break;
    const CUtensorMap *ma, *mb;
    int ya, yb, row;
    coord(it, &ma, &mb, &ya, &yb, &row);
    ptx::mbar_arrive_expect_tx(bar(BAR_FULL0 + b), 2 * kTileBytes);
    for (int ch = 0; ch < 2; ++ch) {
      ptx::tma_load_3d(sb + kOffRingA + b * kTileBytes + ch * kChunkBytes, ma,
                       bar(BAR_FULL0 + b), ch * 64, ya, row);
      ptx::tma_load_3d(sb + kOffRingB + b * kTileBytes + ch * kChunkBytes, mb,
                       bar(BAR_FULL0 + b), ch * 64, yb, row);
    }
    issued = it + 1;
  }
  drain_bar(bar(BAR_FIX), 0, status);
  for (int b = 0; b < 2; ++b) {
    int last = issued - 1;
    if (last >= 0 && (last & 1) != b) --last;
    if (last >= 0) drain_bar(bar(BAR_FULL0 + b), (last >> 1) & 1, status);
  }
}

// 8 SS MMAs (K = 128 in steps of 16): D[128 x 128] = A[128 x 128] B[128 x 128]^T,
// both operands K-major tiles in shared memory.
__device__ __forceinline__ void mma_scores(uint32_t d, uint32_t a_lo, uint32_t b_lo) {
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kT, kT, false);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
    ptx::mma_ss_lohi(d, a_lo + off, ptx::kDescHiSw128, b_lo + off, ptx::kDescHiSw128, kIdesc,
                     kk > 0 ? 1u : 0u);
  }
}

// 8 TS MMAs: D[128 x 128] += A (bf16 in TMEM columns a..a+63) B, B an
// MN-major tile in shared memory (128 rows of K, 128 of N).
__device__ __forceinline__ void mma_grad(uint32_t d, uint32_t a_tmem, uint32_t b_lo, bool first) {
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kT, kD, true);
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    ptx::mma_ts_lohi(d, a_tmem + kk * 8, b_lo + ((kk * 2048) >> 4), ptx::kDescHiSw128, kIdesc,
                     (!first || kk > 0) ? 1u : 0u);
}

// --------------------------------------------------------------------- dQ
// CTA = (query tile, query head).  TMEM: S 0..127 (dS over 0..63), dP
// 128..255, dQ 256..383.
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_tc_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t qr0 = static_cast<int64_t>(blockIdx.x) * kT;
  const int h = blockIdx.y;
  const int c = h / p.group;
  // Key tiles: landmark tiles first, then the window tiles of the rows.
  const int64_t q_last = min64(qr0 + kT, p.n) - 1;
  const int64_t n_lm = visible_landmarks(q_last, p.window, p.block, p.G);
  const int n_lm_tiles = static_cast<int>((n_lm + kT - 1) / kT);
  const int64_t j_lo = max64(qr0 - p.window + 1, 0);
  const int kt_lo = static_cast<int>(j_lo / kT);
  const int T = n_lm_tiles + static_cast<int>(q_last / kT) - kt_lo + 1;

  const uint32_t tmem = bwd_setup(smem, sb, warp);
  WaitCtl ctl{reinterpret_cast<volatile int*>(smem + kOffAbort), p.status, p.wait_ns};

  if (warp == 4) {
    if (lane == 0) {
      auto coord = [&](int t, const CUtensorMap** ma, const CUtensorMap** mb, int* ya, int* yb,
                       int* row) {
        const bool lm = t < n_lm_tiles;
        *ma = lm ? &p.tm_klm : &p.tm_k;
        *mb = lm ? &p.tm_vlm : &p.tm_v;
        *ya = *yb = c;
        *row = lm ? t * kT : (kt_lo + t - n_lm_tiles) * kT;
      };
      produce(sb, &p.tm_q, &p.tm_do, h, static_cast<int>(qr0), T, coord, ctl, p.status);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t q_lo = ptx::desc_lo(sb + kOffFixA, 16);
      const uint32_t do_lo = ptx::desc_lo(sb + kOffFixB, 16);
      const uint32_t k_lo = ptx::desc_lo(sb + kOffRingA, 16);
      const uint32_t v_lo = ptx::desc_lo(sb + kOffRingB, 16);
      const uint32_t k_mn = ptx::desc_lo(sb + kOffRingA, kChunkBytes);
      bool ok = wait_bar(bar(BAR_FIX), 0, ctl);
      for (int t = 0; ok && t < T; ++t) {
        const int b = t & 1;
        if (!(ok = wait_bar(bar(BAR_FULL0 + b), (t >> 1) & 1, ctl))) break;
        ptx::tc_fence_after();
        mma_scores(tmem, q_lo, k_lo + b * kTileLo);          // S  = Q K^T
        mma_scores(tmem + 128, do_lo, v_lo + b * kTileLo);   // dP = dO V^T
        ptx::mma_commit(bar(BAR_SF));
        if (!(ok = wait_bar(bar(BAR_EF), t & 1, ctl))) break;
        ptx::tc_fence_after();
        mma_grad(tmem + 256, tmem, k_mn + b * kTileLo, t == 0);  // dQ += dS K
        ptx::mma_commit(bar(BAR_EMPTY0 + b));
      }
      if (ok) ptx::mma_commit(bar(BAR_ACC));
      ptx::mma_commit(bar(BAR_CLEAN));
      drain_bar(bar(BAR_CLEAN), 0, p.status);
    }
  } else if (warp < 4) {
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int64_t i = qr0 + threadIdx.x;
    const bool row_ok = i < p.n;
    const float L2 = row_ok ? p.lse[static_cast<int64_t>(h) * p.n + i] * kLog2e : INFINITY;
    const float Di = row_ok ? p.D[static_cast<int64_t>(h) * p.n + i] : 0.f;
    const int64_t my_lm = visible_landmarks(i, p.window, p.block, p.G);
    const int64_t my_lo = max64(i - p.window + 1, 0);
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF), t & 1, ctl));
      if (!ok) break;
      ptx::tc_fence_after();
      int64_t lo, hi;  // valid columns [lo, hi) of this key tile for row i
      if (t < n_lm_tiles) {
        lo = 0;
        hi = my_lm - static_cast<int64_t>(t) * kT;
      } else {
        const int64_t kb = static_cast<int64_t>(kt_lo + t - n_lm_tiles) * kT;
        lo = my_lo - kb;
        hi = i - kb + 1;
      }
      if (!row_ok) hi = lo;
      const int lo_c = static_cast<int>(max64(0, min64(kT, lo)));
      const int hi_c = static_cast<int>(max64(0, min64(kT, hi)));
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float s[32], dp[32];
        ptx::tmem_ld32(tl + cc * 32, s);
        ptx::tmem_ld32(tl + 128 + cc * 32, dp);
        ptx::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float ds[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = cc * 32 + 2 * e + u;
            const bool valid = col >= lo_c && col < hi_c;
            const float pr = valid ? ptx::ex2(fmaf(s[2 * e + u], sl2, -L2)) : 0.f;
            ds[u] = pr * (dp[2 * e + u] - Di);
          }
          pk[e] = ptx::pack_bf16x2(ds[0], ds[1]);
        }
        ptx::tmem_st16(tl + cc * 16, pk);  // dS over columns already read
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(BAR_EF));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_ACC), 0, ctl));
    if (ok) {
      ptx::tc_fence_after();
      const int64_t off = (i * p.Hq + h) * static_cast<int64_t>(kD);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float o[32];
        ptx::tmem_ld32(tl + 256 + cc * 32, o);
        ptx::tmem_wait_ld();
        if (row_ok) store_row(p.dq, off + cc * 32, o, p.scale, p.grad_bf16);
      }
    }
  }
  bwd_teardown(tmem, warp);
}

// ------------------------------------------------------------------ dK, dV
// CTA = (key tile or landmark tile, KV head[, query chunk]).  TMEM: S^T
// 0..127 (P^T over 0..63), dP^T 128..255 (dS^T over 128..191), dV
// 256..383, dK 384..511.
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t kb = static_cast<int64_t>(blockIdx.x) * kT;  // first key / landmark
  const int c = blockIdx.y;
  const int chunk = blockIdx.z;
  const int64_t n_qt = (p.n + kT - 1) / kT;
  // Query tiles [qt_lo, qt_hi] whose rows see some key of the tile.
  int64_t qt_lo, qt_hi;
  if (p.lm_mode) {
    const int64_t first_row = (kb + 1) * p.block + p.window - 1;  // sees landmark kb
    const int64_t base = first_row / kT;
    qt_lo = base + static_cast<int64_t>(chunk) * p.chunk_tiles;
    qt_hi = min64(base + static_cast<int64_t>(chunk + 1) * p.chunk_tiles, n_qt) - 1;
  } else {
    qt_lo = kb / kT;
    qt_hi = min64(p.n - 1, kb + kT - 1 + p.window - 1) / kT;
  }
  const int iters = qt_hi >= qt_lo ? static_cast<int>((qt_hi - qt_lo + 1) * p.group) : 0;
  if (iters == 0) {  // landmark chunk beyond the last row: a zero partial
    if (p.lm_mode && threadIdx.x < kT && kb + threadIdx.x < p.G) {
      for (int which = 0; which < 2; ++which) {
        float* dst = p.lm_part + ((((static_cast<int64_t>(chunk) * 2 + which) * p.G + kb +
                                    threadIdx.x) * p.Hkv + c) * kD);
        for (int e = 0; e < kD; ++e) dst[e] = 0.f;
      }
    }
    return;
  }

  const uint32_t tmem = bwd_setup(smem, sb, warp);
  WaitCtl ctl{reinterpret_cast<volatile int*>(smem + kOffAbort), p.status, p.wait_ns};

  if (warp == 4) {
    if (lane == 0) {
      auto coord = [&](int it, const CUtensorMap** ma, const CUtensorMap** mb, int* ya, int* yb,
                       int* row) {
        *ma = &p.tm_q;
        *mb = &p.tm_do;
        *ya = *yb = c * p.group + it % p.group;
        *row = static_cast<int>((qt_lo + it / p.group) * kT);
      };
      produce(sb, p.lm_mode ? &p.tm_klm : &p.tm_k, p.lm_mode ? &p.tm_vlm : &p.tm_v, c,
              static_cast<int>(kb), iters, coord, ctl, p.status);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t k_lo = ptx::desc_lo(sb + kOffFixA, 16);
      const uint32_t v_lo = ptx::desc_lo(sb + kOffFixB, 16);
      const uint32_t q_lo = ptx::desc_lo(sb + kOffRingA, 16);
      const uint32_t do_lo = ptx::desc_lo(sb + kOffRingB, 16);
      const uint32_t q_mn = ptx::desc_lo(sb + kOffRingA, kChunkBytes);
      const uint32_t do_mn = ptx::desc_lo(sb + kOffRingB, kChunkBytes);
      bool ok = wait_bar(bar(BAR_FIX), 0, ctl);
      for (int it = 0; ok && it < iters; ++it) {
        const int b = it & 1;
        if (!(ok = wait_bar(bar(BAR_FULL0 + b), (it >> 1) & 1, ctl))) break;
        ptx::tc_fence_after();
        mma_scores(tmem, k_lo, q_lo + b * kTileLo);          // S^T  = K Q^T
        mma_scores(tmem + 128, v_lo, do_lo + b * kTileLo);   // dP^T = V dO^T
        ptx::mma_commit(bar(BAR_SF));
        if (!(ok = wait_bar(bar(BAR_EF), it & 1, ctl))) break;
        ptx::tc_fence_after();
        mma_grad(tmem + 256, tmem, do_mn + b * kTileLo, it == 0);       // dV += P^T dO
        mma_grad(tmem + 384, tmem + 128, q_mn + b * kTileLo, it == 0);  // dK += dS^T Q
        ptx::mma_commit(bar(BAR_EMPTY0 + b));
      }
      if (ok) ptx::mma_commit(bar(BAR_ACC));
      ptx::mma_commit(bar(BAR_CLEAN));
      drain_bar(bar(BAR_CLEAN), 0, p.status);
    }
  } else if (warp < 4) {
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int64_t j = kb + threadIdx.x;  // key (window mode) or landmark (landmark mode)
    float* stats = reinterpret_cast<float*>(smem + kOffStats);
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < iters; ++it) {
      const int64_t qr0 = (qt_lo + it / p.group) * kT;
      const int h = c * p.group + it % p.group;
      // This iteration's per-query lse (log2 units) and D in a warp-private
      // copy (no cross-warp barrier, so an aborting warp cannot stall the
      // others).
      float* sL = stats + warp * 2 * kT;
      float* sD = sL + kT;
      __syncwarp();  // every lane is done with the previous iteration's copy
#pragma unroll
      for (int u = 0; u < kT / 32; ++u) {
        const int col = lane + 32 * u;
        const int64_t i = qr0 + col;
        sL[col] = i < p.n ? p.lse[static_cast<int64_t>(h) * p.n + i] * kLog2e : INFINITY;
        sD[col] = i < p.n ? p.D[static_cast<int64_t>(h) * p.n + i] : 0.f;
      }
      __syncwarp();
      // Rows i of this query tile that see key/landmark j: [lo, hi) columns.
      int64_t lo, hi;
      if (p.lm_mode) {
        lo = j < p.G ? (j + 1) * p.block + p.window - 1 - qr0 : kT;
        hi = kT;
      } else {
        lo = j - qr0;
        hi = j + p.window - qr0;
      }
      const int lo_c = static_cast<int>(max64(0, min64(kT, lo)));
      const int hi_c = static_cast<int>(max64(0, min64(kT, hi)));
      ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF), it & 1, ctl));
      if (!ok) break;
      ptx::tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float s[32], dp[32];
        ptx::tmem_ld32(tl + cc * 32, s);
        ptx::tmem_ld32(tl + 128 + cc * 32, dp);
        ptx::tmem_wait_ld();
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pr[2], ds[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = cc * 32 + 2 * e + u;
            const bool valid = col >= lo_c && col < hi_c;
            pr[u] = valid ? ptx::ex2(fmaf(s[2 * e + u], sl2, -sL[col])) : 0.f;
            ds[u] = pr[u] * (dp[2 * e + u] - sD[col]);
          }
          pp[e] = ptx::pack_bf16x2(pr[0], pr[1]);
          dd[e] = ptx::pack_bf16x2(ds[0], ds[1]);
        }
        ptx::tmem_st16(tl + cc * 16, pp);        // P^T over columns already read
        ptx::tmem_st16(tl + 128 + cc * 16, dd);  // dS^T likewise
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(BAR_EF));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_ACC), 0, ctl));
    if (ok) {
      ptx::tc_fence_after();
      if (p.lm_mode) {
        const bool row_ok = j < p.G;
        for (int which = 0; which < 2; ++which) {  // 0: dK_lm, 1: dV_lm
          float* dst = p.lm_part + ((((static_cast<int64_t>(chunk) * 2 + which) * p.G + j) *
                                     p.Hkv + c) * kD);
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            float o[32];
            ptx::tmem_ld32(tl + (which == 0 ? 384 : 256) + cc * 32, o);
            ptx::tmem_wait_ld();
            if (row_ok) store_row(dst, cc * 32, o, which == 0 ? p.scale : 1.f, 0);
          }
        }
      } else {
        const bool row_ok = j < p.n;
        const int64_t off = (j * p.Hkv + c) * static_cast<int64_t>(kD);
        // The token's share of its landmark's gradient.
        const float* lmk = nullptr;
        const float* lmv = nullptr;
        if (p.G > 0 && row_ok) {
          const int64_t l = j / p.block;
          lmk = p.lm_grad + (l * p.Hkv + c) * kD;
          lmv = p.lm_grad + ((static_cast<int64_t>(p.G) + l) * p.Hkv + c) * kD;
        }
        const float invB = 1.f / static_cast<float>(p.block);
        for (int which = 0; which < 2; ++which) {  // 0: dK, 1: dV
          const float* lm = which == 0 ? lmk : lmv;
          const float w = which == 0 ? p.scale : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            float o[32];
            ptx::tmem_ld32(tl + (which == 0 ? 384 : 256) + cc * 32, o);
            ptx::tmem_wait_ld();
            if (lm) {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = fmaf(lm[cc * 32 + e], invB / w, o[e]);
            }
            if (row_ok) store_row(which == 0 ? p.dk : p.dv, off + cc * 32, o, w, p.grad_bf16);
          }
        }
      }
    }
  }
  bwd_teardown(tmem, warp);
}

// ----------------------------------------------------------- small kernels
// D[h, i] = <dO[i, h], O[i, h]>: one warp per (row, head), 4 elements a lane.
template <bool kOutBf16>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const void* out, const uint16_t* dout, float* D, int64_t n, int Hq) {
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= n * Hq) return;
  const int64_t base = pair * kD + lane * 4;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float o = kOutBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(out)[base + e])
                             : static_cast<const float*>(out)[base + e];
    acc = fmaf(o, bf16_bits_to_float(dout[base + e]), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const int64_t i = pair / Hq;
    const int h = static_cast<int>(pair % Hq);
    D[static_cast<int64_t>(h) * n + i] = acc;
  }
}

// lm_grad[e] = sum over chunks of lm_part[chunk][e] (fixed order).
__global__ void __launch_bounds__(256)
    lm_grad_reduce_kernel(const float* part, float* grad, int64_t per_chunk, int chunks) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= per_chunk) return;
  float s = 0.f;
  for (int ch = 0; ch < chunks; ++ch) s += part[ch * per_chunk + e];
  grad[e] = s;
}

}  // namespace

bool attn_bwd_supported(int d, int in_bf16) { return in_bf16 && d == kD; }

cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t s, const char** why) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  BwdParams p;
  memset(&p, 0, sizeof(p));
  struct {
    CUtensorMap* m;
    const void* ptr;
    int64_t rows;
    int H;
    const char* name;
  } maps[] = {{&p.tm_q, a.q, a.n, a.Hq, "cuTensorMapEncodeTiled rejected q"},
              {&p.tm_do, a.dout, a.n, a.Hq, "cuTensorMapEncodeTiled rejected dout"},
              {&p.tm_k, a.k, a.n, a.Hkv, "cuTensorMapEncodeTiled rejected k"},
              {&p.tm_v, a.v, a.n, a.Hkv, "cuTensorMapEncodeTiled rejected v"},
              {&p.tm_klm, a.k_lm, a.G, a.Hkv, "cuTensorMapEncodeTiled rejected k_lm"},
              {&p.tm_vlm, a.v_lm, a.G, a.Hkv, "cuTensorMapEncodeTiled rejected v_lm"}};
  for (int i = 0; i < (a.G > 0 ? 6 : 4); ++i) {
    if (!encode_map(fn, maps[i].m, maps[i].ptr, maps[i].rows, maps[i].H)) {
      *why = maps[i].name;
      return cudaErrorInvalidValue;
    }
  }
  if (a.G == 0) {
    p.tm_klm = p.tm_k;
    p.tm_vlm = p.tm_v;
  }
  p.lse = a.lse;
  p.D = a.D;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.lm_part = a.lm_part;
  p.lm_grad = a.lm_grad;
  p.n = a.n;
  p.window = a.window;
  p.block = a.G > 0 ? a.n / a.G : 1;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.G;
  p.group = a.Hq / a.Hkv;
  p.grad_bf16 = a.grad_bf16;
  p.lm_chunks = a.lm_chunks;
  p.chunk_tiles = a.chunk_tiles;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.status = a.status;
  p.wait_ns = a.wait_limit_ns;

  const int64_t pairs = a.n * a.Hq;
  const unsigned pre_blocks = static_cast<unsigned>((pairs + 7) / 8);
  if (a.out_bf16)
    bwd_preprocess_kernel<true><<<pre_blocks, 256, 0, s>>>(
        a.out, static_cast<const uint16_t*>(a.dout), a.D, a.n, a.Hq);
  else
    bwd_preprocess_kernel<false><<<pre_blocks, 256, 0, s>>>(
        a.out, static_cast<const uint16_t*>(a.dout), a.D, a.n, a.Hq);
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  for (auto* k : {bwd_dkdv_tc_kernel, bwd_dq_tc_kernel}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  const unsigned n_tiles = static_cast<unsigned>((a.n + kT - 1) / kT);
  if (a.G > 0) {
    p.lm_mode = 1;
    dim3 grid(static_cast<unsigned>((a.G + kT - 1) / kT), a.Hkv, a.lm_chunks);
    bwd_dkdv_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    const int64_t per_chunk = 2 * static_cast<int64_t>(a.G) * a.Hkv * kD;
    lm_grad_reduce_kernel<<<static_cast<unsigned>((per_chunk + 255) / 256), 256, 0, s>>>(
        a.lm_part, a.lm_grad, per_chunk, a.lm_chunks);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
  }
  p.lm_mode = 0;
  bwd_dkdv_tc_kernel<<<dim3(n_tiles, a.Hkv, 1), kThreads, kSmemBytes, s>>>(p);
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  bwd_dq_tc_kernel<<<dim3(n_tiles, a.Hq), kThreads, kSmemBytes, s>>>(p);
  return cudaPeekAtLastError();
}

}  // namespace msa
