// K2 (tensor-core variant): fused window + landmark attention forward for
// bf16 Q/K/V with d = 128 on sm_103a -- TMA-staged tiles, tcgen05 MMAs with
// fp32 accumulators in tensor memory (TMEM), online softmax in registers.
//
// Method: "Scaling GPU Cluster for Million Token Context", sections "Why
// Sparse Attention Changes the Game" / "What is Flash-MSA Sparse Attention in
// GPU Clusters?" (local window + landmark attention fused in one pass, tiled
// so that the score matrix never reaches HBM; only tiles that hold attended
// pairs are visited, cf. "skip irrelevant pairs").  Row i attends keys
// i-w < j <= i and the landmarks whose whole block lies before that window;
// one softmax over the union.  The running-max/running-sum statistics are
// those a Ring Attention round aggregates ("Training at 1M+ Token Context",
// Ring Attention paragraph); with `partial` set the kernel computes one such
// round's partial against a KV chunk.
//
// Work unit = 128 query rows x 2 query heads of one KV group (GQA: both heads
// read the same K/V tiles, so every K/V tile fetched from L2 feeds two
// 128x128x128 MMA pairs).  One CTA per unit, 12 warps:
//   warp 0      TMA producer: Q tiles once, then K and V tiles through a
//               2-stage ring (landmark tiles first, then window tiles);
//   warp 1      allocates 512 TMEM columns and issues every MMA (the
//               whole warp runs the loop, one elected lane issues):
//               S_s = Q_s K^T (SS: both from shared memory) and
//               O_s += P_s V (TS: P from TMEM, V from shared memory);
//   warps 4-7   softmax of head slot 0 (TMEM lanes 0..127, one row each);
//   warps 8-11  softmax of head slot 1.
// TMEM columns: slot s uses [256s, 256s+128) for S (P overwrites its first
// 64 columns as packed bf16) and [256s+128, 256s+256) for O.
// MMA issue order per tile t: PV_0(t), S_0(t+1), PV_1(t), S_1(t+1), so the
// tensor pipe works on one slot while the other slot's softmax runs.
// S_s(t+1) is issued after PV_s(t), which reads P_s(t) from the same TMEM
// columns; tcgen05 MMAs from one warp execute in issue order.
//
// Softmax: scores are kept in log2 units (scale*log2(e) folded into one FMA);
// the exponent base m is only raised when the row maximum exceeds it by more
// than kTau (then O and l are rescaled in TMEM/registers), so p <= 2^kTau;
// O/l and lse = (m + log2 l) ln 2 are exact for any base.  P enters the PV
// MMA rounded to bf16 and l sums those same rounded values, so each output
// row is an exactly normalised combination of V rows (a key that dominates
// a row then reproduces its V row without the bf16 rounding of its weight).
//
// Every mbarrier wait is bounded (globaltimer); a wait that runs out sets a
// CTA-wide abort flag and the device status word, all roles leave their
// loops, in-flight TMA copies and MMAs are waited for, TMEM is freed, and the
// kernel returns.
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
constexpr int kBM = 128;                 // query rows per slot = TMEM lanes
constexpr int kBN = 128;                 // keys per tile
constexpr int kSlots = 2;                // query heads per CTA
constexpr int kThreads = 384;
constexpr int kChunkBytes = 128 * 128;   // 128 rows x 64 bf16 (one 128-B swizzle span)
constexpr int kTileBytes = 2 * kChunkBytes;  // 128 rows x 128 bf16
constexpr int kStages = 2;
constexpr float kTau = 8.0f;

// Shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kSlots * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
// bf16 O leaves through shared memory: per softmax warp its 32 rows x 64
// columns (one 128-byte swizzle span), stored by one bulk tensor copy.
constexpr int kOutStageBytes = 32 * 128;
constexpr int kOffOut = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffOut + 8 * kOutStageBytes;
constexpr int kNumBars = 14;
constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "attention kernel shared memory");

// Barrier indices.  The K/V ring is organised in pairs: pair g carries V of
// global tile g together with K of tile g+1 (which may be the first tile of
// the next unit), so one barrier tracks both copies and one commit releases
// both buffers.  K of the very first tile of a CTA has its own barrier.
constexpr int BAR_Q = 0;                                 // Q tiles landed
constexpr int BAR_K0 = 1;                                // first K tile landed
__host__ __device__ constexpr int BAR_KVF(int b) { return 2 + b; }  // pair landed
__host__ __device__ constexpr int BAR_KVE(int b) { return 4 + b; }  // pair consumed
__host__ __device__ constexpr int BAR_SF(int s) { return 6 + s; }   // S_s computed
__host__ __device__ constexpr int BAR_PF(int s) { return 8 + s; }   // P_s written
__host__ __device__ constexpr int BAR_OD(int s) { return 10 + s; }  // O_s final
constexpr int BAR_CLEAN = 12;
constexpr int BAR_QE = 13;  // Q buffer free (the unit's last S MMA completed)

struct TcParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_klm;
  CUtensorMap tm_vlm;
  CUtensorMap tm_o;  // O when bf16, 32-row boxes (stores)
  void* out;
  float* lse;
  int64_t n_q, q_start, n_kv, kv_start, window, block, lse_ld;
  int Hq, Hkv, G, group, pairs, n_qtiles, units;
  int out_bf16, partial, merge, band;
  int64_t band_block, band_half;
  const int32_t* sel;
  const int32_t* sel_cnt;
  int top_k, select;
  float scale_log2;
  int* status;
  uint64_t wait_ns;
};

// One work unit: 128 query rows x (up to) 2 heads of one KV group, and the
// key tiles those rows visit (landmark tiles first, then window tiles).
struct Unit {
  int h0, kvh, n_slots, kt_lo, n_lm_tiles, T;
  int64_t qr0;
};

// Unit u in the schedule order: head pair fastest, then query tiles from the
// last one down (the causal partials' heaviest units first), then KV heads.
__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u) {
  Unit w;
  const int pair = u % p.pairs;
  u /= p.pairs;
  const int qt = p.n_qtiles - 1 - (u % p.n_qtiles);
  w.kvh = u / p.n_qtiles;
  w.h0 = w.kvh * p.group + 2 * pair;
  w.n_slots = (2 * pair + 1 < p.group) ? 2 : 1;
  w.qr0 = static_cast<int64_t>(qt) * kBM;
  const int64_t g0 = p.q_start + w.qr0;
  const int64_t g_last = p.q_start + min64(w.qr0 + kBM, p.n_q) - 1;
  const int64_t kv_end = p.kv_start + p.n_kv;
  int64_t j_lo, j_hi;
  if (p.band) {  // union of the rows' bands (whole sequence: kv_start = 0)
    int64_t unused;
    band_keys(g0, p.band_block, p.band_half, p.n_kv, &j_lo, &unused);
    band_keys(g_last, p.band_block, p.band_half, p.n_kv, &unused, &j_hi);
  } else {
    j_lo = max64(g0 - p.window + 1, p.kv_start);
    j_hi = min64(g_last, kv_end - 1);
  }
  w.kt_lo = 0;
  int n_win = 0;
  if (j_hi >= j_lo) {
    w.kt_lo = static_cast<int>((j_lo - p.kv_start) / kBN);
    n_win = static_cast<int>((j_hi - p.kv_start) / kBN) - w.kt_lo + 1;
  }
  if (p.select) {  // the unit's selected key blocks, each block/128 full tiles
    const int64_t ci = static_cast<int64_t>(qt) * p.Hkv + w.kvh;
    const int64_t cnt =
        MSA_IN_RANGE(ci, 1, static_cast<int64_t>(p.n_qtiles) * p.Hkv, p.status)
            ? sel_count_checked(p.sel_cnt[ci], p.top_k,
                                visible_landmarks(g0, p.window, p.block, p.G), p.status)
            : 0;
    w.n_lm_tiles = static_cast<int>(cnt * (p.block / kBN));
  } else {
    const int64_t n_lm = visible_landmarks(g_last, p.window, p.block, p.G);
    w.n_lm_tiles = static_cast<int>((n_lm + kBN - 1) / kBN);
  }
  w.T = w.n_lm_tiles + n_win;
  return w;
}

// Persistent: one CTA per SM walks units blockIdx.x, +gridDim.x, ...  The
// K/V ring, the Q buffer and TMEM carry over from unit to unit, so the next
// unit's Q load and first S MMAs overlap the current unit's epilogue.
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WaitCtl ctl{abort_flag, p.status, p.wait_ns};

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(BAR_Q), 1);
    ptx::mbar_init(bar(BAR_QE), 1);
    ptx::mbar_init(bar(BAR_K0), 1);
    for (int b = 0; b < kStages; ++b) {
      ptx::mbar_init(bar(BAR_KVF(b)), 1);
      ptx::mbar_init(bar(BAR_KVE(b)), 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      ptx::mbar_init(bar(BAR_SF(s)), 1);
      ptx::mbar_init(bar(BAR_PF(s)), 4);  // one arrive per softmax warp
      ptx::mbar_init(bar(BAR_OD(s)), 1);
    }
    ptx::mbar_init(bar(BAR_CLEAN), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Register budget: the producer/MMA warpgroup needs few registers, the
  // two softmax warpgroups hold a 128-score row each.  Launch allocation is
  // 384 x 168; 128 x 96 + 256 x 200 fits in it.  At 200 the softmax keeps a
  // 12-byte spill (3 stores, 1 reload) that only 232 would remove, which
  // would starve the producer; the MMA issue rate, not the softmax, bounds
  // this kernel.  Each role raises or lowers its own budget inside its branch.
  if (warp < 4) {
    ptx::reg_dealloc<96>();
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&p.tm_q);
      ptx::tma_prefetch_desc(&p.tm_k);
      ptx::tma_prefetch_desc(&p.tm_v);
      uint32_t g = 0;       // pairs issued (global tile index)
      uint32_t qn = 0;      // units whose Q was issued
      bool k0 = false;      // first K tile issued
      bool ok = true;
      auto load_tile = [&](const Unit& w, int t, bool is_k, uint32_t dst, uint32_t mbar) {
        const bool lm = t < w.n_lm_tiles;
        int row;
        const CUtensorMap* m;
        if (lm && p.select) {  // tile of a selected block, from K/V themselves
          const int tpb = static_cast<int>(p.block / kBN);
          const int64_t si = (w.qr0 / kBM * p.Hkv + w.kvh) * p.top_k + t / tpb;
          const int64_t blk =
              MSA_IN_RANGE(si, 1, static_cast<int64_t>(p.n_qtiles) * p.Hkv * p.top_k, p.status)
                  ? sel_block_checked(p.sel[si], visible_landmarks(w.qr0, p.window, p.block, p.G),
                                      p.status)
                  : 0;
          row = static_cast<int>(blk * p.block) + (t % tpb) * kBN;
          m = is_k ? &p.tm_k : &p.tm_v;
        } else {
          m = is_k ? (lm ? &p.tm_klm : &p.tm_k) : (lm ? &p.tm_vlm : &p.tm_v);
          row = lm ? t * kBN : (w.kt_lo + t - w.n_lm_tiles) * kBN;
        }
        for (int c = 0; c < 2; ++c) {
          // Box origins are only recorded when out of range: the copy is
          // issued all the same (out-of-range rows read the fill value).
          (void)MSA_TMA_OK(c * 64, w.kvh, row, kD, p.Hkv, lm && !p.select ? p.G : p.n_kv, kBN,
                           p.status);
          ptx::tma_load_3d(dst + c * kChunkBytes, m, mbar, c * 64, w.kvh, row);
        }
      };
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const Unit w = decode_unit(p, u);
        if (w.T == 0) continue;
        // The next unit of this CTA that has tiles: its first K rides with
        // this unit's last V.
        int un = u + gridDim.x;
        Unit nw{};
        while (un < p.units) {
          nw = decode_unit(p, un);
          if (nw.T > 0) break;
          un += gridDim.x;
        }
        const bool has_next = un < p.units;
        // The Q buffer is free once the previous unit's last S MMA is done.
        if (qn > 0 && !(ok = wait_bar(bar(BAR_QE), (qn - 1) & 1, ctl))) break;
        ptx::mbar_arrive_expect_tx(bar(BAR_Q), w.n_slots * kTileBytes);
        for (int s = 0; s < w.n_slots; ++s)
          for (int c = 0; c < 2; ++c) {
            (void)MSA_TMA_OK(c * 64, w.h0 + s, w.qr0, kD, p.Hq, p.n_q, kBM, p.status);
            ptx::tma_load_3d(sb + kOffQ + s * kTileBytes + c * kChunkBytes, &p.tm_q, bar(BAR_Q),
                             c * 64, w.h0 + s, static_cast<int>(w.qr0));
          }
        ++qn;
        // Warm L2 with this CTA's next Q tiles: they are read once, from
        // HBM, exactly when the tensor pipe waits for them.
        if (has_next)
          for (int s = 0; s < nw.n_slots; ++s)
            for (int c = 0; c < 2; ++c)
              ptx::tma_prefetch_3d(&p.tm_q, c * 64, nw.h0 + s, static_cast<int>(nw.qr0));
        if (!k0) {
          ptx::mbar_arrive_expect_tx(bar(BAR_K0), kTileBytes);
          load_tile(w, 0, true, sb + kOffK + (g & 1) * kTileBytes, bar(BAR_K0));
          k0 = true;
        }
        for (int t = 0; t < w.T; ++t, ++g) {
          const int b = g & 1;
          // Pair g refills the buffers of pair g-2.  Pair 1's K buffer held
          // the CTA's first K tile instead, whose release is the first
          // completion of barrier 1; barrier 0's first wait passes at once.
          const uint32_t parity = b == 0 ? ((g >> 1) & 1) ^ 1 : (g >> 1) & 1;
          if (!(ok = wait_bar(bar(BAR_KVE(b)), parity, ctl))) break;
          const bool with_k = (t + 1 < w.T) || has_next;
          ptx::mbar_arrive_expect_tx(bar(BAR_KVF(b)), with_k ? 2 * kTileBytes : kTileBytes);
          load_tile(w, t, false, sb + kOffV + b * kTileBytes, bar(BAR_KVF(b)));
          if (t + 1 < w.T)
            load_tile(w, t + 1, true, sb + kOffK + ((g + 1) & 1) * kTileBytes, bar(BAR_KVF(b)));
          else if (has_next)
            load_tile(nw, 0, true, sb + kOffK + ((g + 1) & 1) * kTileBytes, bar(BAR_KVF(b)));
        }
      }
      // Drain: every copy this thread issued must have landed before exit.
      if (qn > 0) drain_bar(bar(BAR_Q), (qn - 1) & 1, p.status);
      if (k0) drain_bar(bar(BAR_K0), 0, p.status);
      for (int b = 0; b < kStages; ++b) {
        int last = static_cast<int>(g) - 1;
        if (last >= 0 && (last & 1) != b) --last;
        if (last >= 0) drain_bar(bar(BAR_KVF(b)), (last >> 1) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issuing loop; elect.sync picks the lane that
    // issues each tcgen05 instruction.
    {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false);
      constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(kBM, kD, true);
      // Descriptor low halves of every operand base, computed once; per K
      // step the low half advances by a compile-time constant (Q/K: 32 B
      // within a 128-B swizzle row, 16 KB to the second 64-column chunk;
      // V: 16 key rows = 2 KB), see the layouts at the TMA maps.
      const uint32_t q_lo0 = ptx::desc_lo(sb + kOffQ, 16);
      const uint32_t k_lo0 = ptx::desc_lo(sb + kOffK, 16);
      const uint32_t v_lo0 = ptx::desc_lo(sb + kOffV, kChunkBytes);
      constexpr uint32_t kTileLo = kTileBytes >> 4;
      auto issue_s = [&](int slot, uint32_t stage) {
        const uint32_t qa = q_lo0 + slot * kTileLo;
        const uint32_t kb = k_lo0 + stage * kTileLo;
        ptx::mma_ss_x8_w<(kChunkBytes >> 4)>(tmem + slot * 256, qa, kb, kIdescS, 0u);
      };
      auto issue_pv = [&](int slot, uint32_t stage, bool first) {
        const uint32_t vb = v_lo0 + stage * kTileLo;
        ptx::mma_ts_x8_w(tmem + slot * 256 + 128, tmem + slot * 256, vb, kIdescO, first ? 0u : 1u);
      };
      uint32_t g = 0;                 // global tile index (K/V ring position)
      uint32_t qn = 0;                // units processed
      uint32_t sc[kSlots] = {0, 0};   // tiles processed per slot (SF/PF phases)
      bool first = true;              // first unit: K tile 0 has its own barrier
      int pending = -1;               // pair whose K feeds the next unit's S(0)
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
        const Unit w = decode_unit(p, u);
        if (w.T == 0) continue;
        if (!(ok = wait_w(bar(BAR_Q), qn & 1, ctl))) break;
        const bool first_unit = first;
        if (first) {
          if (!(ok = wait_w(bar(BAR_K0), 0, ctl))) break;
          first = false;
        }
        // (Otherwise K of this tile came with the previous unit's last pair,
        // which that unit's last iteration waited for.)
        ptx::tc_fence_after();
        for (int s = 0; s < w.n_slots; ++s) {
          issue_s(s, g & 1);
          ptx::commit_w(bar(BAR_SF(s)));
        }
        // The first K tile's buffer is refilled by pair 1: release it.
        if (first_unit) ptx::commit_w(bar(BAR_KVE(1)));
        if (w.T == 1) ptx::commit_w(bar(BAR_QE));  // the unit's last S MMA
        if (pending >= 0) {
          ptx::commit_w(bar(BAR_KVE(pending & 1)));
          pending = -1;
        }
        for (int t = 0; ok && t < w.T; ++t, ++g) {
          const uint32_t b = g & 1;
          const bool nxt = t + 1 < w.T;
          // Pair g: V of this tile and K of the next one.
          if (!(ok = wait_w(bar(BAR_KVF(b)), (g >> 1) & 1, ctl))) break;
          for (int s = 0; s < w.n_slots; ++s) {
            if (!(ok = wait_w(bar(BAR_PF(s)), (sc[s] + t) & 1, ctl))) break;
            ptx::tc_fence_after();
            // PV_s(t) reads P_s(t) from the S columns; S_s(t+1) overwrites
            // them and is issued after it by this same warp.
            issue_pv(s, b, t == 0);
            if (nxt) {
              issue_s(s, b ^ 1);
              ptx::commit_w(bar(BAR_SF(s)));
            } else {
              ptx::commit_w(bar(BAR_OD(s)));
            }
          }
          if (!ok) break;
          if (t + 2 == w.T) ptx::commit_w(bar(BAR_QE));  // S(T-1) was the last S
          if (nxt)
            ptx::commit_w(bar(BAR_KVE(b)));
          else
            pending = static_cast<int>(g);  // released after the next unit's S(0)
        }
        for (int s = 0; s < w.n_slots; ++s) sc[s] += w.T;
        ++qn;
      }
      if (pending >= 0) ptx::commit_w(bar(BAR_KVE(pending & 1)));
      // Drain: all MMAs issued so far complete before TMEM is released.
      ptx::commit_w(bar(BAR_CLEAN));
      drain_bar(bar(BAR_CLEAN), 0, p.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    ptx::reg_alloc<200>();
    const int slot = (warp - 4) >> 2;
    const int wq = warp & 3;
    const uint32_t tS = tmem + slot * 256 + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tO = tS + 128;
    const int64_t kv_end = p.kv_start + p.n_kv;
    const float sl2 = p.scale_log2;
    uint32_t sc = 0, oc = 0;  // tiles / units this slot has processed
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
      const Unit w = decode_unit(p, u);
      if (slot >= w.n_slots) continue;
      const int64_t i_loc = w.qr0 + wq * 32 + lane;
      const bool row_ok = i_loc < p.n_q;
      const int64_t i = p.q_start + i_loc;
      const int h = w.h0 + slot;
      if (w.T == 0) {  // no key for any row of this unit (partial chunks only)
        const int64_t lse_idx = static_cast<int64_t>(h) * p.lse_ld + i_loc;
        if (row_ok && !p.merge && MSA_IN_RANGE(lse_idx, 1, (p.Hq - 1) * p.lse_ld + p.n_q, p.status))
          p.lse[lse_idx] = -INFINITY;
        continue;
      }
      int64_t my_lo, my_hi;
      if (p.band) {
        band_keys(i, p.band_block, p.band_half, p.n_kv, &my_lo, &my_hi);
      } else {
        my_lo = max64(i - p.window + 1, p.kv_start);
        my_hi = min64(i, kv_end - 1);
      }
      // Selected blocks lie wholly before every row's window: no mask.
      const int64_t my_lm =
          p.select ? INT64_MAX / 2 : visible_landmarks(i, p.window, p.block, p.G);
      float m_used = -INFINITY;
      float l = 0.f;
      for (int t = 0; t < w.T; ++t) {
        ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF(slot)), (sc + t) & 1, ctl));
        if (!ok) break;
        ptx::tc_fence_after();
        float s[128];
        ptx::tmem_ld32(tS + 0, *reinterpret_cast<float(*)[32]>(&s[0]));
        ptx::tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
        ptx::tmem_ld32(tS + 64, *reinterpret_cast<float(*)[32]>(&s[64]));
        ptx::tmem_ld32(tS + 96, *reinterpret_cast<float(*)[32]>(&s[96]));
        ptx::tmem_wait_ld();
        // Valid columns [lo, hi) of this tile for this row.
        int64_t lo, hi;
        if (t < w.n_lm_tiles) {
          lo = 0;
          hi = my_lm - static_cast<int64_t>(t) * kBN;
        } else {
          const int64_t kb = p.kv_start + static_cast<int64_t>(w.kt_lo + t - w.n_lm_tiles) * kBN;
          lo = my_lo - kb;
          hi = my_hi - kb + 1;
        }
        if (!row_ok) hi = lo;
        // Boundary tiles only, each side on its own (one compare with a
        // constant and one select per score); the branches are uniform
        // across the warp.
        const int lo_c = static_cast<int>(max64(0, min64(kBN, lo)));
        const int hi_c = static_cast<int>(max64(0, min64(kBN, hi)));
        if (__builtin_expect(__any_sync(0xffffffffu, lo_c > 0), 0)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = c >= lo_c ? s[c] : -INFINITY;
        }
        if (__builtin_expect(__any_sync(0xffffffffu, hi_c < kBN), 0)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = c < hi_c ? s[c] : -INFINITY;
        }
        // Row maximum: four independent chains of three-input maxima.
        float a0 = fmaxf(s[0], s[1]), a1 = fmaxf(s[2], s[3]);
        float a2 = fmaxf(s[4], s[5]), a3 = fmaxf(s[6], s[7]);
#pragma unroll
        for (int c = 8; c < 128; c += 8) {
          a0 = ptx::max3(a0, s[c], s[c + 1]);
          a1 = ptx::max3(a1, s[c + 2], s[c + 3]);
          a2 = ptx::max3(a2, s[c + 4], s[c + 5]);
          a3 = ptx::max3(a3, s[c + 6], s[c + 7]);
        }
        const float mx = ptx::max3(a0, a1, fmaxf(a2, a3));
        const float m_new = fmaxf(m_used, mx * sl2);
        const bool need = m_new > m_used + kTau;
        if (need) {
          const float alpha = ptx::ex2(m_used - m_new);  // 0 when m_used = -inf
          l *= alpha;
        }
        if (t > 0 && __any_sync(0xffffffffu, need)) {
          const float alpha = need ? ptx::ex2(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            float o[16];
            ptx::tmem_ld16(tO + cc * 16, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha;
            ptx::tmem_st16(tO + cc * 16, *reinterpret_cast<uint32_t(*)[16]>(o));
          }
        }
        if (need) m_used = m_new;
        const float mb = (m_used == -INFINITY) ? 0.f : m_used;
        // p = 2^(s*scale*log2e - m) two at a time (packed FMA), rounded to
        // bf16 pairs for the PV MMA; the denominator sums those same
        // rounded weights (so O is normalised by exactly the weights it was
        // built from), added to four fp32 partial sums as they are.
        const uint64_t c2 = ptx::f2(sl2, sl2);
        const uint64_t nb2 = ptx::f2(-mb, -mb);
        float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint64_t x =
                ptx::fma2(ptx::f2(s[cc * 32 + 2 * e], s[cc * 32 + 2 * e + 1]), c2, nb2);
            float x0, x1;
            ptx::f2_split(x, x0, x1);
            pk[e] = ptx::pack_bf16x2(ptx::ex2(x0), ptx::ex2(x1));
            if (e & 1)
              ptx::acc_bf16x2(l2, l3, pk[e]);
            else
              ptx::acc_bf16x2(l0, l1, pk[e]);
          }
          ptx::tmem_st16(tS + cc * 16, pk);
        }
        l += (l0 + l1) + (l2 + l3);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(BAR_PF(slot)));
      }
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_OD(slot)), oc & 1, ctl));
      if (!ok) break;
      ptx::tc_fence_after();
      // Epilogue.  The TMEM reads of O complete (wait::ld) before this slot
      // arrives for the next unit's first P, which the MMA thread waits for
      // before the next unit's first PV overwrites O.
      const bool has = row_ok && l > 0.f;
      const int64_t lse_idx = static_cast<int64_t>(h) * p.lse_ld + i_loc;
      const int64_t obase = (i_loc * p.Hq + h) * static_cast<int64_t>(kD);
      // Offsets of this row against the extents of O [n_q, Hq, d] and lse
      // [Hq][lse_ld] (checked in the bounds-checked build only).
      const bool io_ok =
          !row_ok ||
          (MSA_IN_RANGE(lse_idx, 1, (p.Hq - 1) * p.lse_ld + p.n_q, p.status) &&
           MSA_IN_RANGE(obase, kD, p.n_q * p.Hq * static_cast<int64_t>(kD), p.status));
      // O = acc * w_new (+ running O * w_run when merging into a running
      // result: lse_run <- ln(e^lse_run + e^lse_p)).
      const float lse_p = has ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      float w_new = has ? 1.f / l : 0.f;
      float w_run = 0.f;
      float lse_out = lse_p;
      if (p.merge && has && io_ok) {
        const float L = p.lse[lse_idx];
        if (L != -INFINITY) {
          const float mx = fmaxf(L, lse_p);
          lse_out = mx + logf(expf(L - mx) + expf(lse_p - mx));
          w_run = expf(L - lse_out);
          w_new *= expf(lse_p - lse_out);
        }
      }
      // bf16 O of a warp whose valid rows all have a key: staged in shared
      // memory (the 128-byte swizzle of tm_o's 32 x 64 box) and written by
      // one bulk tensor store per 64 columns; rows past n_q are clipped.
      const int row0 = static_cast<int>(w.qr0) + wq * 32;
      if (p.out_bf16 && !p.merge && __all_sync(0xffffffffu, (has || !row_ok) && io_ok)) {
        if (row0 < p.n_q) {
          (void)MSA_TMA_OK(0, h, row0, kD, p.Hq, p.n_q, 32, p.status);
          const uint32_t stg = sb + kOffOut + static_cast<uint32_t>((warp - 4) * kOutStageBytes);
          const uint32_t my = stg + static_cast<uint32_t>(lane * 128);
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            float o[64];
            ptx::tmem_ld32(tO + hh * 64, *reinterpret_cast<float(*)[32]>(&o[0]));
            ptx::tmem_ld32(tO + hh * 64 + 32, *reinterpret_cast<float(*)[32]>(&o[32]));
            ptx::tmem_wait_ld();
            if (lane == 0) ptx::bulk_wait_read();  // the buffer's last store has read it
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)  // 16-byte chunk j of row `lane`, swizzled
              ptx::st_shared_v4(my + static_cast<uint32_t>(((j ^ lane) & 7) << 4),
                                ptx::pack_bf16x2(o[8 * j + 0] * w_new, o[8 * j + 1] * w_new),
                                ptx::pack_bf16x2(o[8 * j + 2] * w_new, o[8 * j + 3] * w_new),
                                ptx::pack_bf16x2(o[8 * j + 4] * w_new, o[8 * j + 5] * w_new),
                                ptx::pack_bf16x2(o[8 * j + 6] * w_new, o[8 * j + 7] * w_new));
            ptx::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(&p.tm_o, stg, hh * 64, h, row0);
              ptx::bulk_commit();
            }
          }
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          float o[32];
          ptx::tmem_ld32(tO + cc * 32, o);
          ptx::tmem_wait_ld();
          if (has && io_ok) {
            if (p.out_bf16) {
              uint4* dst =
                  reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + obase + cc * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 q4;
                q4.x = ptx::pack_bf16x2(o[8 * v + 0] * w_new, o[8 * v + 1] * w_new);
                q4.y = ptx::pack_bf16x2(o[8 * v + 2] * w_new, o[8 * v + 3] * w_new);
                q4.z = ptx::pack_bf16x2(o[8 * v + 4] * w_new, o[8 * v + 5] * w_new);
                q4.w = ptx::pack_bf16x2(o[8 * v + 6] * w_new, o[8 * v + 7] * w_new);
                dst[v] = q4;
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + obase + cc * 32);
              if (w_run != 0.f) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  const float4 r = dst[v];
                  dst[v] = make_float4(fmaf(r.x, w_run, o[4 * v] * w_new),
                                       fmaf(r.y, w_run, o[4 * v + 1] * w_new),
                                       fmaf(r.z, w_run, o[4 * v + 2] * w_new),
                                       fmaf(r.w, w_run, o[4 * v + 3] * w_new));
                }
              } else {
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[v] = make_float4(o[4 * v] * w_new, o[4 * v + 1] * w_new, o[4 * v + 2] * w_new,
                                       o[4 * v + 3] * w_new);
              }
            }
          }
        }
      }
      // Rows without a key: -inf (a partial), or untouched (a running merge).
      if (row_ok && io_ok && (has || !p.merge)) p.lse[lse_idx] = lse_out;
      sc += w.T;
      oc += 1;
    }
    // This warp's bulk stores of O complete before shared memory is released.
    if (lane == 0) ptx::bulk_wait_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool attn_tc_supported(int Hq, int Hkv, int d, int in_bf16) {
  (void)Hq;
  (void)Hkv;
  return in_bf16 && d == kD;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s, const char** why) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  const bool ok = encode_map(fn, &p.tm_q, a.q, a.n_q, a.Hq) &&
                  encode_map(fn, &p.tm_k, a.k, a.n_kv, a.Hkv) &&
                  encode_map(fn, &p.tm_v, a.v, a.n_kv, a.Hkv) &&
                  (a.G > 0 && !a.sel ? encode_map(fn, &p.tm_klm, a.k_lm, a.G, a.Hkv) &&
                                           encode_map(fn, &p.tm_vlm, a.v_lm, a.G, a.Hkv)
                                     : true) &&
                  (a.out_bf16 ? encode_map(fn, &p.tm_o, a.out, a.n_q, a.Hq, 32) : true);
  if (!ok) {
    *why = "cuTensorMapEncodeTiled rejected a tensor (alignment or size)";
    return cudaErrorInvalidValue;
  }
  if (!a.out_bf16) p.tm_o = p.tm_q;  // not used: fp32 O is stored by the threads
  if (a.G == 0 || a.sel) {  // no landmark tensors read
    p.tm_klm = p.tm_k;
    p.tm_vlm = p.tm_v;
  }
  p.out = a.out;
  p.lse = a.lse;
  p.n_q = a.n_q;
  p.lse_ld = a.lse_ld;
  p.q_start = a.q_start;
  p.n_kv = a.n_kv;
  p.kv_start = a.kv_start;
  p.window = a.window;
  p.block = a.block;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.G;
  p.group = a.Hq / a.Hkv;
  p.pairs = (p.group + 1) / 2;
  p.n_qtiles = static_cast<int>((a.n_q + kBM - 1) / kBM);
  p.out_bf16 = a.out_bf16;
  p.partial = a.partial;
  p.merge = a.merge;
  p.band = a.band;
  p.band_block = a.band_block;
  p.band_half = a.band_half;
  p.sel = a.sel;
  p.sel_cnt = a.sel_cnt;
  p.top_k = a.top_k;
  p.select = a.sel != nullptr;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.wait_ns = a.wait_limit_ns;

  cudaError_t attr_err = cudaFuncSetAttribute(
      attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t units = static_cast<int64_t>(a.Hkv) * p.pairs * p.n_qtiles;
  p.units = static_cast<int>(units);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t grid = units < sms ? units : sms;
  attn_tc_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, s>>>(p);
  return cudaPeekAtLastError();
}

}  // namespace msa
