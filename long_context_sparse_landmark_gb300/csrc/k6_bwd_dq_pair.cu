// K6, pair variant of the dQ kernel of the backward pass (bf16, d = 128),
// run by pairs of CTAs on the two SMs of a TPC that share each tcgen05 MMA
// (`cta_group::2`).  The gradient is the exact one of the forward's
// definition ("Training at 1M+ Token Context", Block-Sparse Flash Attention
// paragraph: the model trains with the sparse pattern): per query row i,
//   P = 2^(S scale log2e - lse log2e),  dS = P (dP - D_i),  dQ = scale dS K,
// over the landmark tiles and the window tiles of the row, as the
// single-CTA dQ kernel in k6_attn_bwd.cu computes it.
//
// Persistent: one cluster per CTA pair that fits on the device loops over
// units, a unit being one 128-row query tile of two query heads (2j, 2j+1)
// of one KV group.  The K/V rings and every barrier phase carry across
// units; Q and dO are refilled once a unit's last S MMA is done, and the
// dQ accumulator is released as soon as the elementwise warps have read it,
// so the next unit's first MMAs overlap the epilogue.
//
// In a unit, CTA rank r holds head 2j + r, its own Q and dO tiles, and its own
// TMEM (S, dQ, two dP buffers, as the single-CTA kernel).  Every MMA is a
// pair MMA with M = 256, issued by the lead CTA: the score products S = Q K^T
// and dP = dO V^T take B = K and V split by key rows (each CTA holds 64 of
// the tile's 128 keys), and dQ += dS K takes B = K split by columns (each
// CTA holds 64 of the 128 head columns, all keys).  So each SM reads half of
// every B operand from shared memory (single-CTA SS MMAs run below the
// tensor rate for lack of shared-memory bandwidth) and one warp issues the
// MMAs of both SMs.
//
// Roles (10 warps per CTA): warps 0-7 elementwise (TMEM lane = row; warps w
// and w + 4 share a row quarter and split the key columns), warp 8 TMA
// producer, warp 9 TMEM allocation (both CTAs) and MMA issue (lead).  Every
// wait is bounded; a wait that runs out sets the CTA's abort flag, which the
// peer also watches, and both CTAs drain and free their tensor memory.
#include <cuda.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "msa_common.cuh"
#include "tc_pair.cuh"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"
#include "tma_map.h"

namespace msa {
namespace {

constexpr int kD = 128;
constexpr int kT = 128;                  // rows per tile (queries or keys)
constexpr int kThreads = 320;
constexpr int kEwWarps = 8;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kChunk = 128 * 128;        // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kTile = 2 * kChunk;        // a 128 x 128 bf16 tile
constexpr int kHalfChunk = 64 * 128;     // 64 rows x 64 bf16
constexpr int kRowsHalf = 2 * kHalfChunk;  // 64 key rows x 128 columns
constexpr int kKStages = 3;              // K is read until the late dQ MMAs
constexpr int kVStages = 2;              // V only by dP
constexpr int kKStage = 2 * kRowsHalf;   // K rows half (scores) + K column half (dQ)
constexpr int kVStage = kRowsHalf;
constexpr uint64_t kBackoffNs = 200;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;
constexpr int kOffDo = kTile;
constexpr int kOffK = 2 * kTile;
constexpr int kOffV = kOffK + kKStages * kKStage;
// bf16 dQ leaves through shared memory: per elementwise warp its 32 rows x
// 64 columns (one 128-byte swizzle span), stored by one bulk tensor copy.
constexpr int kOutStageBytes = 32 * 128;
constexpr int kOffOut = kOffV + kVStages * kVStage;
constexpr int kOffBar = kOffOut + kEwWarps * kOutStageBytes;
// Barriers: "lead" collects bytes or arrivals of both CTAs on the lead's
// copy; "both" is completed on each CTA's copy by a multicast commit.
enum {
  B_FIX = 0,       // lead: Q, dO of both CTAs landed
  B_FULLK0 = 1,    // lead: K stage landed (1..3)
  B_EMPTYK0 = 4,   // both: K stage consumed (4..6)
  B_FULLV0 = 7,    // lead: V stage landed (7, 8)
  B_EMPTYV0 = 9,   // both: V stage consumed (9, 10)
  B_SF = 11,       // both: S and dP of a tile computed
  B_EF = 12,       // lead: dS of an even key tile written (8 warps x 2 CTAs)
  B_ACC = 13,      // both: dQ final
  B_CLEAN = 14,    // both: every MMA done
  B_SFREE = 15,    // lead: every elementwise warp has read S (8 x 2)
  B_QE = 16,       // both: the unit's last S MMA done (Q, dO free)
  B_DQFREE = 17,   // lead: every elementwise warp has read the unit's dQ (8 x 2)
  B_EF1 = 18,      // lead: dS of an odd key tile written (8 x 2); see ef_bar
  kNumBars = 19
};
constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "dQ pair kernel shared memory");

// TMEM columns (per CTA, its own 128 rows): S 0..127, dQ 128..255, dP of
// even / odd key tiles 256..383 / 384..511 (dS of each 32-key chunk packed
// over the chunk's first 16 columns).
constexpr uint32_t kColS = 0;
constexpr uint32_t kColQ = 128;
__device__ __forceinline__ uint32_t col_p(int t) { return 256 + static_cast<uint32_t>(t & 1) * 128; }
// The "dS written" barrier of key tile g, and the phase to wait for.  Tiles
// alternate between two barriers: S(g + 1) needs only every warp's read of
// S(g), so a fast warp may finish tile g + 1 before a slow one has written
// dS(g); with one barrier its arrival could complete tile g's phase and let
// the dQ MMA read dP bits as dS.  Tile g + 2 needs every warp's read of
// S(g + 1), which follows its tile-g arrival, so each barrier's phase counts
// arrivals of one tile only.
__device__ __forceinline__ int ef_bar(uint32_t g) { return (g & 1) ? B_EF1 : B_EF; }
__device__ __forceinline__ uint32_t ef_phase(uint32_t g) { return (g >> 1) & 1; }

struct DqPairParams {
  CUtensorMap tm_q, tm_do;          // [n, Hq, d], 128-row boxes
  CUtensorMap tm_k64, tm_v64;       // [n, Hkv, d], 64-row boxes (key-row halves)
  CUtensorMap tm_k128;              // K, 128-row boxes (one 64-column half)
  CUtensorMap tm_klm64, tm_vlm64, tm_klm128;  // landmarks, same boxes
  CUtensorMap tm_dq;                // dQ when bf16, 32-row boxes (stores)
  const float* L2;                  // [Hq, n_pad] -lse log2e
  const float* D;                   // [Hq, n_pad] -<dO, O>
  void* dq;                         // [n, Hq, d]
  int64_t n, n_pad, window, block;
  int Hq, Hkv, G, group, grad_bf16;
  int n_tiles, units;               // query tiles; units = n_tiles x Hq / 2
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

// One work unit: a 128-row query tile of one head pair.  Units run from the
// last query tile down (the longest windows first), head pairs outermost.
// T depends on the query tile alone, so both CTAs of a pair run as many
// tiles.
struct DqUnit {
  int64_t qr0;
  int h, c, n_lm_tiles, kt_lo, T;
};

__device__ __forceinline__ DqUnit decode_dq_unit(const DqPairParams& p, int u, uint32_t rank) {
  DqUnit w;
  const int qt = p.n_tiles - 1 - (u % p.n_tiles);
  const int hp = u / p.n_tiles;
  w.qr0 = static_cast<int64_t>(qt) * kT;
  w.h = 2 * hp + static_cast<int>(rank);
  w.c = w.h / p.group;  // the same for both CTAs: the group size is even
  // Key tiles of the query tile (the same for both heads): landmark tiles,
  // then the window tiles of its rows.
  const int64_t q_last = min64(w.qr0 + kT, p.n) - 1;
  const int64_t n_lm = visible_landmarks(q_last, p.window, p.block, p.G);
  w.n_lm_tiles = static_cast<int>((n_lm + kT - 1) / kT);
  w.kt_lo = static_cast<int>(max64(w.qr0 - p.window + 1, 0) / kT);
  w.T = w.n_lm_tiles + static_cast<int>(q_last / kT) - w.kt_lo + 1;
  return w;
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_pair_kernel(const __grid_constant__ DqPairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = pair::cta_rank();
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int n_clusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i)
      ptx::mbar_init(bar(i), (i == B_EF || i == B_EF1 || i == B_SFREE || i == B_DQFREE)
                                 ? 2 * kEwWarps
                                 : 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  if (warp == kMmaWarp) {
    pair::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    pair::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  pair::cluster_sync();  // both CTAs' barriers initialised, tensor memory held
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const PairWait ctl{abort_flag, pair::peer_addr(sb + kOffAbort, rank ^ 1u), p.status, p.wait_ns};
  auto lead = [&](int i) -> uint32_t { return pair::peer_addr(bar(i), 0); };

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      bool ok = true;
      uint32_t g = 0;                  // key tiles this cluster has started
      int nfix = 0, nk = 0, nv = 0;    // Q/dO, K and V fills issued
      for (int u = cid; ok && u < p.units; u += n_clusters) {
        const DqUnit w = decode_dq_unit(p, u, rank);
        // Q and dO of the previous unit are free once its last S MMA is done.
        if (nfix >= 1 && !(ok = wait_pair(bar(B_QE), (nfix - 1) & 1, ctl, kBackoffNs))) break;
        if (rank == 0) ptx::mbar_arrive_expect_tx(bar(B_FIX), 2 * 2 * kTile);
        for (int ch = 0; ch < 2; ++ch) {
          (void)MSA_TMA_OK(ch * 64, w.h, w.qr0, kD, p.Hq, p.n, kT, p.status);
          pair::tma_load_3d(sb + kOffQ + ch * kChunk, &p.tm_q, lead(B_FIX), ch * 64, w.h,
                            static_cast<int>(w.qr0));
          pair::tma_load_3d(sb + kOffDo + ch * kChunk, &p.tm_do, lead(B_FIX), ch * 64, w.h,
                            static_cast<int>(w.qr0));
        }
        ++nfix;
        for (int t = 0; t < w.T; ++t, ++g) {
          const bool lm = t < w.n_lm_tiles;
          const int row = lm ? t * kT : (w.kt_lo + t - w.n_lm_tiles) * kT;
          (void)MSA_TMA_OK(0, w.c, row, kD, p.Hkv, lm ? p.G : p.n, kT, p.status);
          const int sk = static_cast<int>(g % kKStages), sv = static_cast<int>(g % kVStages);
          if (g >= kKStages &&
              !(ok = wait_pair(bar(B_EMPTYK0 + sk), ((g / kKStages) - 1) & 1, ctl, kBackoffNs)))
            break;
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar(B_FULLK0 + sk), 2 * kKStage);
          const uint32_t kdst = sb + kOffK + sk * kKStage;
          for (int ch = 0; ch < 2; ++ch)  // key rows 64 rank .. + 64, all columns
            pair::tma_load_3d(kdst + ch * kHalfChunk, lm ? &p.tm_klm64 : &p.tm_k64,
                              lead(B_FULLK0 + sk), ch * 64, w.c,
                              row + 64 * static_cast<int>(rank));
          // all 128 keys, columns 64 rank .. + 64
          pair::tma_load_3d(kdst + kRowsHalf, lm ? &p.tm_klm128 : &p.tm_k128,
                            lead(B_FULLK0 + sk), 64 * static_cast<int>(rank), w.c, row);
          nk = static_cast<int>(g) + 1;
          if (g >= kVStages &&
              !(ok = wait_pair(bar(B_EMPTYV0 + sv), ((g / kVStages) - 1) & 1, ctl, kBackoffNs)))
            break;
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar(B_FULLV0 + sv), 2 * kVStage);
          for (int ch = 0; ch < 2; ++ch)
            pair::tma_load_3d(sb + kOffV + sv * kVStage + ch * kHalfChunk,
                              lm ? &p.tm_vlm64 : &p.tm_v64, lead(B_FULLV0 + sv), ch * 64, w.c,
                              row + 64 * static_cast<int>(rank));
          nv = static_cast<int>(g) + 1;
        }
      }
      // Drain (lead): an armed phase completes once both CTAs' bytes have
      // landed.  After an abort the peer may not have issued its copies of
      // a phase the lead armed; issued copies land within microseconds, so
      // the drain then waits 50 ms per barrier.
      if (rank == 0) {
        const uint64_t lim = *abort_flag ? 50000000ull : kDrainLimitNs;
        if (nfix >= 1) drain_for(bar(B_FIX), (nfix - 1) & 1, p.status, lim);
        for (int st = 0; st < kKStages; ++st) {
          const int last = nk - 1 - ((nk - 1 - st) % kKStages + kKStages) % kKStages;
          if (last >= 0) drain_for(bar(B_FULLK0 + st), (last / kKStages) & 1, p.status, lim);
        }
        for (int st = 0; st < kVStages; ++st) {
          const int last = nv - 1 - ((nv - 1 - st) % kVStages + kVStages) % kVStages;
          if (last >= 0) drain_for(bar(B_FULLV0 + st), (last / kVStages) & 1, p.status, lim);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (lead)
    if (rank == 0) {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(256, kT, false);
      constexpr uint32_t kIdescG = ptx::idesc_bf16_f32(256, kD, true);
      const uint32_t q_lo = ptx::desc_lo(sb + kOffQ, 16);
      const uint32_t do_lo = ptx::desc_lo(sb + kOffDo, 16);
      const uint32_t k_lo = ptx::desc_lo(sb + kOffK, 16);
      const uint32_t v_lo = ptx::desc_lo(sb + kOffV, 16);
      const uint32_t k_mn = ptx::desc_lo(sb + kOffK + kRowsHalf, kChunk);
      // D[128 x 128 per CTA] = A[128 x 128] B[128 x 128]^T: A this CTA's Q or
      // dO, B each CTA's 64 key rows.
      auto scores = [&](uint32_t d, uint32_t a_lo, uint32_t b_lo) {
        pair::mma_ss_x8<(kChunk >> 4), (kHalfChunk >> 4)>(d, a_lo, b_lo, kIdescS, 0u);
      };
      // dP(g) then S(g) of key tile g.  S's columns are free once every
      // elementwise warp has read S(g - 1); dP(g) overwrites dS(g - 2), which
      // the dQ MMA of tile g - 2, issued earlier by this warp, has read.
      auto tile_scores = [&](uint32_t gg) -> bool {
        const int sv = static_cast<int>(gg % kVStages), sk = static_cast<int>(gg % kKStages);
        if (!wait_pair_w(bar(B_FULLV0 + sv), (gg / kVStages) & 1, ctl)) return false;
        ptx::tc_fence_after();
        scores(tmem + col_p(static_cast<int>(gg)), do_lo, v_lo + sv * (kVStage >> 4));
        pair::commit_both(bar(B_EMPTYV0 + sv));  // V(gg) consumed
        if (!wait_pair_w(bar(B_FULLK0 + sk), (gg / kKStages) & 1, ctl)) return false;
        if (gg >= 1 && !wait_pair_w(bar(B_SFREE), (gg - 1) & 1, ctl)) return false;
        ptx::tc_fence_after();
        scores(tmem + kColS, q_lo, k_lo + sk * (kKStage >> 4));
        pair::commit_both(bar(B_SF));
        return true;
      };
      bool ok = true;
      uint32_t g = 0, ul = 0;  // key tiles / units this cluster has processed
      for (int u = cid; ok && u < p.units; u += n_clusters, ++ul) {
        const int T = decode_dq_unit(p, u, 0).T;
        if (!(ok = wait_pair_w(bar(B_FIX), ul & 1, ctl))) break;
        if (!(ok = tile_scores(g))) break;
        if (T == 1) pair::commit_both(bar(B_QE));  // the unit's last S MMA
        for (int t = 0; ok && t < T; ++t) {
          const uint32_t gt = g + t;
          if (t + 1 < T) {
            if (!(ok = tile_scores(gt + 1))) break;
            if (t + 2 == T) pair::commit_both(bar(B_QE));  // the unit's last S MMA
          }
          if (!(ok = wait_pair_w(bar(ef_bar(gt)), ef_phase(gt), ctl))) break;
          // The first dQ MMA of a unit overwrites the accumulator that the
          // previous unit's epilogue reads.
          if (t == 0 && ul >= 1 && !(ok = wait_pair_w(bar(B_DQFREE), (ul - 1) & 1, ctl))) break;
          ptx::tc_fence_after();
          const int sk = static_cast<int>(gt % kKStages);
          pair::mma_ts_chunked_x8(tmem + kColQ, tmem + col_p(static_cast<int>(gt)),
                                  k_mn + sk * (kKStage >> 4), kIdescG, t > 0 ? 1u : 0u);
          pair::commit_both(bar(B_EMPTYK0 + sk));  // K(gt) consumed
        }
        if (!ok) break;
        pair::commit_both(bar(B_ACC));
        g += T;
      }
      pair::commit_both(bar(B_CLEAN));
    }
  } else if (warp < kEwWarps) {
    // ------------------------------------------------------------ elementwise
    const int quarter = warp & 3;  // TMEM lanes (rows) 32 quarter ..
    const int cp = warp >> 2;      // key columns [64 cp, 64 cp + 64) of each tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint64_t c2 = ptx::f2(p.scale_log2, p.scale_log2);
    const uint32_t sfree = lead(B_SFREE), dqfree = lead(B_DQFREE);
    bool ok = true;
    uint32_t g = 0, ul = 0;
    for (int u = cid; ok && u < p.units; u += n_clusters, ++ul) {
      const DqUnit w = decode_dq_unit(p, u, rank);
      const int64_t i = w.qr0 + quarter * 32 + lane;  // query row
      const int64_t st = static_cast<int64_t>(w.h) * p.n_pad + i;
      const bool st_ok = MSA_IN_RANGE(st, 1, static_cast<int64_t>(p.Hq) * p.n_pad, p.status);
      const bool row_ok = i < p.n && st_ok;
      const float nL2 = st_ok ? p.L2[st] : -INFINITY;
      const float nD = st_ok ? p.D[st] : 0.f;
      const uint64_t nL22 = ptx::f2(nL2, nL2);
      const uint64_t nD2 = ptx::f2(nD, nD);
      const int64_t my_lm = visible_landmarks(i, p.window, p.block, p.G);
      const int64_t my_lo = max64(i - p.window + 1, 0);
      for (int t = 0; ok && t < w.T; ++t) {
        const uint32_t gt = g + t;
        int64_t lo, hi;  // valid columns [lo, hi) of this key tile for row i
        if (t < w.n_lm_tiles) {
          lo = 0;
          hi = my_lm - static_cast<int64_t>(t) * kT;
        } else {
          const int64_t kb = static_cast<int64_t>(w.kt_lo + t - w.n_lm_tiles) * kT;
          lo = my_lo - kb;
          hi = i - kb + 1;
        }
        if (!row_ok) hi = lo;
        if (!(ok = wait_pair_w(bar(B_SF), gt & 1, ctl))) break;
        ptx::tc_fence_after();
        const int lo_c = static_cast<int>(max64(0, min64(kT, lo)));
        const int hi_c = static_cast<int>(max64(0, min64(kT, hi)));
        const uint32_t tp = tl + col_p(static_cast<int>(gt));
        // This warp's two 32-column chunks of S and dP, all read before S is
        // released for the next tile's S MMAs.
        float s[2][32], dp[2][32];
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
          ptx::tmem_ld32(tl + kColS + (2 * cp + ci) * 32, s[ci]);
          ptx::tmem_ld32(tp + (2 * cp + ci) * 32, dp[ci]);
        }
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        pair::arrive_cluster_w(sfree);
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
          const int cc = 2 * cp + ci;  // 32-column chunk
          // Masked columns get weight 0, each side on its own in branches
          // uniform across the warp: one compare with a constant and one
          // select per score.
          const int lo_e = lo_c - cc * 32, hi_e = hi_c - cc * 32;
          if (__any_sync(0xffffffffu, lo_e > 0)) {
#pragma unroll
            for (int e = 0; e < 32; ++e) s[ci][e] = e >= lo_e ? s[ci][e] : -INFINITY;
          }
          if (__any_sync(0xffffffffu, hi_e < 32)) {
#pragma unroll
            for (int e = 0; e < 32; ++e) s[ci][e] = e < hi_e ? s[ci][e] : -INFINITY;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            // p = 2^(s scale log2e - lse log2e), dS = p (dP - D)
            float x0, x1;
            ptx::f2_split(ptx::fma2(ptx::f2(s[ci][2 * e], s[ci][2 * e + 1]), c2, nL22), x0, x1);
            const uint64_t pr = ptx::f2(ptx::ex2(x0), ptx::ex2(x1));
            float d0, d1;
            ptx::f2_split(
                ptx::mul2(pr, ptx::add2(ptx::f2(dp[ci][2 * e], dp[ci][2 * e + 1]), nD2)), d0,
                d1);
            pk[e] = ptx::pack_bf16x2(d0, d1);
          }
          ptx::tmem_st16(tp + cc * 32, pk);  // dS over dP columns this warp has read
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        pair::arrive_cluster_w(lead(ef_bar(gt)));
      }
      if (ok) ok = wait_pair_w(bar(B_ACC), ul & 1, ctl);
      if (!ok) break;
      ptx::tc_fence_after();
      // This warp's 64 of the 128 columns, read before the next unit's first
      // dQ MMA may overwrite them; the global stores follow.
      float o[2][32];
      ptx::tmem_ld32(tl + kColQ + (2 * cp) * 32, o[0]);
      ptx::tmem_ld32(tl + kColQ + (2 * cp + 1) * 32, o[1]);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      pair::arrive_cluster_w(dqfree);
      const int64_t off = (i * p.Hq + w.h) * static_cast<int64_t>(kD);
      const bool out_ok =
          !row_ok || MSA_IN_RANGE(off, kD, p.n * p.Hq * static_cast<int64_t>(kD), p.status);
      const int row0 = static_cast<int>(w.qr0) + quarter * 32;
      if (p.grad_bf16 && __all_sync(0xffffffffu, out_ok)) {
        // Staged in shared memory (the 128-byte swizzle of tm_dq's 32 x 64
        // box) and written by one bulk tensor store; rows past n are
        // clipped.  Each thread storing its own row would touch 32 lines
        // per instruction and hold the warp from the next unit's first tile.
        if (row0 < p.n) {
          (void)MSA_TMA_OK(64 * cp, w.h, row0, kD, p.Hq, p.n, 32, p.status);
          const uint32_t stg = sb + kOffOut + static_cast<uint32_t>(warp * kOutStageBytes);
          const uint32_t my = stg + static_cast<uint32_t>(lane * 128);
          if (lane == 0) ptx::bulk_wait_read();  // the buffer's last store has read it
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {  // 16-byte chunk j of row `lane`, swizzled
            const float* c8 = &o[j >> 2][(j & 3) * 8];
            ptx::st_shared_v4(my + static_cast<uint32_t>(((j ^ lane) & 7) << 4),
                              ptx::pack_bf16x2(c8[0] * p.scale, c8[1] * p.scale),
                              ptx::pack_bf16x2(c8[2] * p.scale, c8[3] * p.scale),
                              ptx::pack_bf16x2(c8[4] * p.scale, c8[5] * p.scale),
                              ptx::pack_bf16x2(c8[6] * p.scale, c8[7] * p.scale));
          }
          ptx::fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&p.tm_dq, stg, 64 * cp, w.h, row0);
            ptx::bulk_commit();
          }
        }
      } else if (row_ok && out_ok) {
        store_row(p.dq, off + (2 * cp) * 32, o[0], p.scale, p.grad_bf16);
        store_row(p.dq, off + (2 * cp + 1) * 32, o[1], p.scale, p.grad_bf16);
      }
      g += w.T;
    }
    // This warp's bulk stores of dQ complete before shared memory is released.
    if (lane == 0) ptx::bulk_wait_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) drain_for(bar(B_CLEAN), 0, p.status, kDrainLimitNs);  // the lead's last commit
  ptx::tc_fence_before();
  pair::cluster_sync();  // neither CTA leaves while the other may still address it
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    pair::tmem_dealloc(tmem, 512);
  }
}

constexpr int kMaxDev = 64;
std::mutex g_occ_mu;
int g_max_clusters[kMaxDev] = {};

}  // namespace

bool bwd_dq_pair_supported(const BwdArgs& a) {
  return a.rows == nullptr && a.Hq % 2 == 0 && (a.Hq / a.Hkv) % 2 == 0 &&
         a.n <= (int64_t(1) << 30);
}

cudaError_t launch_bwd_dq_pair(const BwdArgs& a, cudaStream_t s, const char** why) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  DqPairParams p;
  memset(&p, 0, sizeof(p));
  const bool ok = encode_map(fn, &p.tm_q, a.q, a.n, a.Hq, 128) &&
                  encode_map(fn, &p.tm_do, a.dout, a.n, a.Hq, 128) &&
                  encode_map(fn, &p.tm_k64, a.k, a.n, a.Hkv, 64) &&
                  encode_map(fn, &p.tm_k128, a.k, a.n, a.Hkv, 128) &&
                  encode_map(fn, &p.tm_v64, a.v, a.n, a.Hkv, 64) &&
                  (a.G > 0 ? encode_map(fn, &p.tm_klm64, a.k_lm, a.G, a.Hkv, 64) &&
                                 encode_map(fn, &p.tm_klm128, a.k_lm, a.G, a.Hkv, 128) &&
                                 encode_map(fn, &p.tm_vlm64, a.v_lm, a.G, a.Hkv, 64)
                           : true) &&
                  (a.grad_bf16 ? encode_map(fn, &p.tm_dq, a.dq, a.n, a.Hq, 32) : true);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled rejected a tensor of the dQ pair kernel";
    return cudaErrorInvalidValue;
  }
  if (!a.grad_bf16) p.tm_dq = p.tm_q;  // not used: fp32 dQ is stored by the threads
  if (a.G == 0) {  // no landmark tensors read
    p.tm_klm64 = p.tm_k64;
    p.tm_klm128 = p.tm_k128;
    p.tm_vlm64 = p.tm_v64;
  }
  p.L2 = a.stats;
  p.D = a.stats + static_cast<int64_t>(a.Hq) * a.n_pad;
  p.dq = a.dq;
  p.n = a.n;
  p.n_pad = a.n_pad;
  p.window = a.window;
  p.block = a.G > 0 ? a.n / a.G : 1;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.G;
  p.group = a.Hq / a.Hkv;
  p.grad_bf16 = a.grad_bf16;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.wait_ns = a.wait_limit_ns;
  // Function attributes belong to the context: set on every launch.
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t n_tiles = (a.n + kT - 1) / kT;
  const int64_t units = n_tiles * (a.Hq / 2);
  if (units > INT32_MAX) {
    *why = "too many query tiles x head pairs for the dQ pair kernel";
    return cudaErrorInvalidValue;
  }
  p.n_tiles = static_cast<int>(n_tiles);
  p.units = static_cast<int>(units);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) {
    *why = "device ordinal out of range";
    return cudaErrorInvalidDevice;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Persistent: one cluster per CTA pair that fits at once (a property of
  // the device, cached), each looping over units.
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    max_clusters = g_max_clusters[dev];
  }
  if (max_clusters == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    e = cudaOccupancyMaxActiveClusters(&max_clusters, bwd_dq_pair_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) {
      *why = "no CTA pair of the dQ kernel fits on this device";
      return cudaErrorInvalidConfiguration;
    }
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_max_clusters[dev] = max_clusters;
  }
  int64_t clusters = units < max_clusters ? units : max_clusters;
  if (a.max_clusters > 0 && clusters > a.max_clusters) clusters = a.max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  e = cudaLaunchKernelEx(&cfg, bwd_dq_pair_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();
}

}  // namespace msa
