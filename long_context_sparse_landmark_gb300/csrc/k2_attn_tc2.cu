// K2, pair variant: fused window + landmark attention forward for bf16
// Q/K/V with d = 128 on sm_103a, run by pairs of CTAs on the two SMs of a
// TPC that share each tcgen05 MMA (`cta_group::2`).
//
// Method: "Scaling GPU Cluster for Million Token Context", sections "Why
// Sparse Attention Changes the Game" / "What is Flash-MSA Sparse Attention in
// GPU Clusters?" (local window + landmark attention fused in one pass, tiled
// so that the score matrix never reaches HBM; only tiles that hold attended
// pairs are visited).  Row i attends keys i-w < j <= i and the landmarks
// whose whole block lies before that window; one softmax over the union.
// The running statistics are those a Ring Attention round aggregates
// ("Training at 1M+ Token Context", Ring Attention paragraph); the partial,
// running-merge, block-band and selected-block modes are those of the
// single-CTA kernel (k2_attn_tc.cu), whose work split, masks, softmax and
// epilogue this kernel keeps: per CTA two head slots of 128 query rows, a
// softmax warpgroup per slot (so two softmax warps share each SM
// sub-partition and hide each other's latencies), P written over its S in
// tensor memory, MMA order PV_0(t), S_0(t+1), PV_1(t), S_1(t+1).
//
// What the pair changes.  A work unit is 128 query rows x 4 query heads of
// one KV group: slot s of CTA rank r holds head h0 + 2s + r.  Every MMA is a
// pair MMA with M = 256 -- slot s of both CTAs in one instruction: A is each
// CTA's own 128 rows (Q, or P from its tensor memory), B is split in half
// between the CTAs (S = Q K^T: each holds 64 of the tile's 128 keys; O += P V:
// each holds 64 of the 128 value columns), D lands in each CTA's tensor
// memory.  So each SM stores and reads half of every K/V tile (the four
// heads share it across the TPC), the shared-memory operand traffic per MMA
// drops from 8 KB to 6 KB for S and from 4 KB to 2 KB for PV (the SS MMAs
// of the single-CTA kernel run below the tensor rate for lack of
// shared-memory bandwidth), and one thread of the lead CTA issues the MMAs
// of both SMs.
// Tensor memory per CTA: slot s uses [256s, 256s+128) for S (P over its
// first 64 columns as packed bf16) and [256s+128, 256s+256) for O.
// O leaves through shared memory: each softmax warp stages its 32 rows in
// a 4 KB buffer and one lane issues bulk tensor stores (a running merge
// first loads the running O box into the buffer the same way).
//
// Roles (12 warps per CTA):
//   warp 0      TMA producer (both CTAs): its own heads' Q tiles, and its
//               half of every K/V tile, through a 4-stage ring; completion
//               bytes are signalled on the lead CTA's barriers;
//   warp 1      tensor-memory allocation (both CTAs); in the lead CTA (rank
//               0) it issues every pair MMA and commit; commits reach both
//               CTAs;
//   warps 4-7   softmax and epilogue of slot 0 (one row per thread);
//   warps 8-11  the same for slot 1.
// A slot whose head is missing on one CTA (odd group size) leaves that
// CTA's warpgroup idle: it keeps the barrier protocol but computes and
// stores nothing.
//
// Every mbarrier wait is bounded (globaltimer); a wait that runs out sets the
// CTA's abort flag and the device status word, both CTAs leave their loops
// (each also watches the peer's flag), in-flight copies and MMAs are waited
// for with a fixed limit, tensor memory is freed, and the kernel returns.
#include <cuda.h>
#include <math.h>
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
constexpr int kBM = 128;                      // query rows per slot = TMEM lanes
constexpr int kBN = 128;                      // keys per tile
constexpr int kSlots = 2;                     // head slots per CTA
constexpr int kThreads = 384;
constexpr int kQChunk = 128 * 128;            // 128 rows x 64 bf16 (one 128-B swizzle span)
constexpr int kQBytes = 2 * kQChunk;          // one head's 128 x 128 Q tile
constexpr int kKChunk = 64 * 128;             // 64 keys x 64 bf16
constexpr int kKBytes = 2 * kKChunk;          // this CTA's half of a K tile
constexpr int kVBytes = 128 * 128;            // 128 keys x this CTA's 64 value columns
constexpr int kStageBytes = kKBytes + kVBytes;
constexpr int kStages = 4;
constexpr float kTau = 8.0f;
constexpr uint32_t kBackoffNs = 200;  // sleep between probes of the producer's waits

// Shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffQ = 0;                                  // Q of slot 0, slot 1
constexpr int kOffKV = kOffQ + kSlots * kQBytes;          // stage s: K half, then V half
// bf16 O leaves through shared memory: per softmax warp its 32 rows x 64
// columns (one 128-byte swizzle span), stored by one bulk tensor copy.
constexpr int kOutStageBytes = 32 * 128;
constexpr int kOffOut = kOffKV + kStages * kStageBytes;
constexpr int kOffBar = kOffOut + 8 * kOutStageBytes;
constexpr int kNumBars = 25;
constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;  // alignment slack
static_assert(kSmemBytes <= 232448, "pair attention kernel shared memory");

// Barriers.  "lead": only the lead CTA's copy is used, and it collects
// arrivals or bytes from both CTAs; "both": each CTA waits on its own copy,
// which a multicast commit of the lead's MMA warp completes.
constexpr int BAR_QF = 0;                                              // lead: Q tiles landed
constexpr int BAR_QE = 1;                                              // both: Q buffer free
__host__ __device__ constexpr int BAR_KVF(int s) { return 2 + s; }     // lead: K/V stage landed
__host__ __device__ constexpr int BAR_KVE(int s) { return 6 + s; }     // both: stage consumed
__host__ __device__ constexpr int BAR_SF(int s) { return 10 + s; }     // both: S of slot s computed
__host__ __device__ constexpr int BAR_PF(int s) { return 12 + s; }     // lead: P of slot s written (8 warps)
__host__ __device__ constexpr int BAR_OD(int s) { return 14 + s; }     // both: O of slot s final
constexpr int BAR_CLEAN = 16;                                          // both: all MMAs done
// local: the running O box that softmax warp w (4..11) loads when merging landed
__host__ __device__ constexpr int BAR_OL(int w) { return 17 + (w - 4); }

struct Tc2Params {
  CUtensorMap tm_q;    // Q, 128-row boxes
  CUtensorMap tm_k;    // K, 64-row boxes (one CTA's half of a tile)
  CUtensorMap tm_v;    // V, 128-row boxes (64 columns: one CTA's half)
  CUtensorMap tm_klm;  // landmark keys, 64-row boxes
  CUtensorMap tm_vlm;  // landmark values, 128-row boxes
  CUtensorMap tm_o;    // O (bf16 or fp32), 32-row boxes (stores)
  void* out;
  float* lse;
  int64_t n_q, q_start, n_kv, kv_start, window, block, lse_ld;
  int Hq, Hkv, G, group, quads, n_qtiles, units;
  int out_bf16, merge, band;
  int64_t band_block, band_half;
  const int32_t* sel;
  const int32_t* sel_cnt;
  int top_k, select;
  float scale_log2;
  int* status;
  uint64_t wait_ns;
};

// One work unit: 128 query rows x (up to) 4 heads of one KV group, and the
// key tiles those rows visit (landmark or selected-block tiles first, then
// window tiles).
struct Unit {
  int h0, kvh, n_heads, n_slots, kt_lo, n_lm_tiles, T;
  int64_t qr0;
};

// Unit u in schedule order: head quad fastest, then query tiles from the
// last one down (the heaviest units of causal partials first), then KV heads.
__device__ __forceinline__ Unit decode_unit(const Tc2Params& p, int u) {
  Unit w;
  const int quad = u % p.quads;
  u /= p.quads;
  const int qt = p.n_qtiles - 1 - (u % p.n_qtiles);
  w.kvh = u / p.n_qtiles;
  w.h0 = w.kvh * p.group + 4 * quad;
  w.n_heads = min(4, p.group - 4 * quad);
  w.n_slots = (w.n_heads + 1) >> 1;
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

__global__ void __launch_bounds__(kThreads, 1) attn_tc2_kernel(const __grid_constant__ Tc2Params p) {
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
    ptx::mbar_init(bar(BAR_QF), 1);
    ptx::mbar_init(bar(BAR_QE), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(BAR_KVF(s)), 1);
      ptx::mbar_init(bar(BAR_KVE(s)), 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      ptx::mbar_init(bar(BAR_SF(s)), 1);
      ptx::mbar_init(bar(BAR_PF(s)), 8);  // 4 softmax warps x 2 CTAs
      ptx::mbar_init(bar(BAR_OD(s)), 1);
    }
    ptx::mbar_init(bar(BAR_CLEAN), 1);
    for (int w = 4; w < 12; ++w) ptx::mbar_init(bar(BAR_OL(w)), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  if (warp == 1) {
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

  // Register budget: 384 x 168 at launch; the producer/MMA warpgroup drops
  // to 96 and the two softmax warpgroups (a 128-score row per thread) rise
  // to 200: 128 x 96 + 256 x 200 <= 384 x 168.
  if (warp < 4) ptx::reg_dealloc<96>();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&p.tm_q);
      ptx::tma_prefetch_desc(&p.tm_k);
      ptx::tma_prefetch_desc(&p.tm_v);
      bool ok = true;
      uint32_t g = 0, ul = 0;
      for (int u = cid; ok && u < p.units; u += n_clusters) {
        const Unit w = decode_unit(p, u);
        if (w.T == 0) continue;
        // The Q buffers are free once the previous unit's last S MMAs are done.
        if (ul >= 1 && !(ok = wait_pair(bar(BAR_QE), (ul - 1) & 1, ctl, kBackoffNs))) break;
        if (rank == 0) ptx::mbar_arrive_expect_tx(bar(BAR_QF), w.n_heads * kQBytes);
        for (int s = 0; s < w.n_slots; ++s)
          if (2 * s + static_cast<int>(rank) < w.n_heads)
            for (int c = 0; c < 2; ++c) {
              // Box origins are only recorded when out of range: the copy is
              // issued all the same (out-of-range rows read the fill value).
              (void)MSA_TMA_OK(c * 64, w.h0 + 2 * s + static_cast<int>(rank), w.qr0, kD, p.Hq,
                               p.n_q, kBM, p.status);
              pair::tma_load_3d(sb + kOffQ + s * kQBytes + c * kQChunk, &p.tm_q, lead(BAR_QF),
                                c * 64, w.h0 + 2 * s + static_cast<int>(rank),
                                static_cast<int>(w.qr0));
            }
        // Warm L2 with this CTA's next Q tiles: they are read once, from HBM.
        for (int un = u + n_clusters; un < p.units; un += n_clusters) {
          const Unit nw = decode_unit(p, un);
          if (nw.T == 0) continue;
          for (int s = 0; s < nw.n_slots; ++s)
            if (2 * s + static_cast<int>(rank) < nw.n_heads)
              for (int c = 0; c < 2; ++c)
                ptx::tma_prefetch_3d(&p.tm_q, c * 64, nw.h0 + 2 * s + static_cast<int>(rank),
                                     static_cast<int>(nw.qr0));
          break;
        }
        for (int t = 0; t < w.T; ++t, ++g) {
          const int s = static_cast<int>(g % kStages);
          if (g >= kStages &&
              !(ok = wait_pair(bar(BAR_KVE(s)), ((g / kStages) - 1) & 1, ctl, kBackoffNs)))
            break;
          if (rank == 0) ptx::mbar_arrive_expect_tx(bar(BAR_KVF(s)), 2 * kStageBytes);
          const bool lm = t < w.n_lm_tiles;
          int row;
          const CUtensorMap* mk;
          const CUtensorMap* mv;
          if (lm && p.select) {  // a selected block's tile, from K/V themselves
            const int tpb = static_cast<int>(p.block / kBN);
            const int64_t si = (w.qr0 / kBM * p.Hkv + w.kvh) * p.top_k + t / tpb;
            const int64_t blk =
                MSA_IN_RANGE(si, 1, static_cast<int64_t>(p.n_qtiles) * p.Hkv * p.top_k, p.status)
                    ? sel_block_checked(p.sel[si],
                                        visible_landmarks(w.qr0, p.window, p.block, p.G),
                                        p.status)
                    : 0;
            row = static_cast<int>(blk * p.block) + (t % tpb) * kBN;
            mk = &p.tm_k;
            mv = &p.tm_v;
          } else {
            mk = lm ? &p.tm_klm : &p.tm_k;
            mv = lm ? &p.tm_vlm : &p.tm_v;
            row = lm ? t * kBN : (w.kt_lo + t - w.n_lm_tiles) * kBN;
          }
          const uint32_t kdst = sb + kOffKV + s * kStageBytes;
          const uint32_t full = lead(BAR_KVF(s));
          const int64_t rows_ext = lm && !p.select ? p.G : p.n_kv;
          (void)rows_ext;
          for (int c = 0; c < 2; ++c) {
            // The tile (not this CTA's half, which may lie wholly past the
            // end of a ragged last tile) must overlap the rows.
            (void)MSA_TMA_OK(c * 64, w.kvh, row, kD, p.Hkv, rows_ext, kBN, p.status);
            pair::tma_load_3d(kdst + c * kKChunk, mk, full, c * 64, w.kvh,
                              row + 64 * static_cast<int>(rank));
          }
          (void)MSA_TMA_OK(64 * static_cast<int>(rank), w.kvh, row, kD, p.Hkv, rows_ext, kBN,
                           p.status);
          pair::tma_load_3d(kdst + kKBytes, mv, full, 64 * static_cast<int>(rank), w.kvh, row);
        }
        ++ul;
      }
      // Drain (lead): every armed phase completes once both CTAs' bytes
      // have landed, so the peer's copies are covered as well.  After an
      // abort the peer may not have issued the copies of a phase the lead
      // armed; copies that were issued land within microseconds, so the
      // drain then waits 50 ms per barrier instead of the full limit.
      if (rank == 0) {
        const uint64_t lim = *abort_flag ? 50000000ull : kDrainLimitNs;
        if (ul >= 1) drain_for(bar(BAR_QF), (ul - 1) & 1, p.status, lim);
        for (int s = 0; s < kStages; ++s) {
          int last = static_cast<int>(g) - 1;
          while (last >= 0 && last % kStages != s) --last;
          if (last >= 0) drain_for(bar(BAR_KVF(s)), (last / kStages) & 1, p.status, lim);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lead)
    if (rank == 0) {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(256, kBN, false);
      constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(256, kD, true);
      const uint32_t q_lo0 = ptx::desc_lo(sb + kOffQ, 16);
      const uint32_t k_lo0 = ptx::desc_lo(sb + kOffKV, 16);
      const uint32_t v_lo0 = ptx::desc_lo(sb + kOffKV + kKBytes, kQChunk);
      auto issue_s = [&](int slot, uint32_t stage) {
        pair::mma_ss_x8<(kQChunk >> 4), (kKChunk >> 4)>(
            tmem + slot * 256, q_lo0 + slot * (kQBytes >> 4), k_lo0 + stage * (kStageBytes >> 4),
            kIdescS, 0u);
      };
      auto issue_pv = [&](int slot, uint32_t stage, bool first) {
        pair::mma_ts_x8(tmem + slot * 256 + 128, tmem + slot * 256,
                        v_lo0 + stage * (kStageBytes >> 4), kIdescO, first ? 0u : 1u);
      };
      bool ok = true;
      uint32_t g = 0, ul = 0;
      uint32_t sc[kSlots] = {0, 0};  // tiles processed per slot (SF / PF phases)
      for (int u = cid; ok && u < p.units; u += n_clusters) {
        const Unit w = decode_unit(p, u);
        if (w.T == 0) continue;
        if (!(ok = wait_pair_w(bar(BAR_QF), ul & 1, ctl))) break;
        if (!(ok = wait_pair_w(bar(BAR_KVF(g % kStages)), (g / kStages) & 1, ctl))) break;
        ptx::tc_fence_after();
        // S(0) of each slot.  Slot s's S columns held P of the previous
        // unit's last tile, which its last PV (issued before, by this same
        // warp) has read.
        for (int s = 0; s < w.n_slots; ++s) {
          issue_s(s, g % kStages);
          pair::commit_both(bar(BAR_SF(s)));
        }
        if (w.T == 1) pair::commit_both(bar(BAR_QE));  // the unit's last S MMAs
        for (int t = 0; ok && t < w.T; ++t) {
          const uint32_t gt = g + t;
          const uint32_t st = gt % kStages;
          const bool nxt = t + 1 < w.T;
          if (nxt && !(ok = wait_pair_w(bar(BAR_KVF((gt + 1) % kStages)), ((gt + 1) / kStages) & 1,
                                        ctl)))
            break;
          for (int s = 0; s < w.n_slots; ++s) {
            // PV_s(t) needs P_s(t) of both CTAs; S_s(t+1) overwrites it and
            // is issued after it by this same warp.
            if (!(ok = wait_pair_w(bar(BAR_PF(s)), (sc[s] + t) & 1, ctl))) break;
            ptx::tc_fence_after();
            issue_pv(s, st, t == 0);
            if (nxt) {
              issue_s(s, (gt + 1) % kStages);
              pair::commit_both(bar(BAR_SF(s)));
            } else {
              pair::commit_both(bar(BAR_OD(s)));
            }
          }
          if (!ok) break;
          if (t + 2 == w.T) pair::commit_both(bar(BAR_QE));  // S(T-1) was the last S
          pair::commit_both(bar(BAR_KVE(st)));
        }
        for (int s = 0; s < w.n_slots; ++s) sc[s] += w.T;
        g += w.T;
        ++ul;
      }
      // Drain: every MMA completes before tensor memory is released.
      pair::commit_both(bar(BAR_CLEAN));
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    ptx::reg_alloc<200>();
    const int slot = (warp - 4) >> 2;
    const int wq = warp & 3;
    const uint32_t tS = tmem + slot * 256 + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tO = tS + 128;
    const int64_t kv_end = p.kv_start + p.n_kv;
    const float sl2 = p.scale_log2;
    const uint32_t pf = lead(BAR_PF(slot));
    uint32_t sc = 0, oc = 0;  // tiles / units this slot has processed
    uint32_t ol_issued = 0, ol_done = 0;  // running-O box loads (merge mode)
    // A unit as this thread's row sees it.  The next unit's is computed while
    // the current unit's last PV runs (its divisions would otherwise sit
    // between the epilogue and the next unit's first softmax).
    struct RowUnit {
      Unit w;
      int h, lo0, hi0, lm0;
      int64_t i_loc;
      bool has, row_ok;
    };
    auto row_unit = [&](int u) -> RowUnit {
      RowUnit r;
      r.w = decode_unit(p, u);
      const int hh = 2 * slot + static_cast<int>(rank);
      r.has = hh < r.w.n_heads;  // this CTA holds a head in this slot
      r.h = r.w.h0 + hh;
      r.i_loc = r.w.qr0 + wq * 32 + lane;
      r.row_ok = r.i_loc < p.n_q;
      const int64_t i = p.q_start + r.i_loc;
      int64_t my_lo, my_hi;
      if (p.band) {
        band_keys(i, p.band_block, p.band_half, p.n_kv, &my_lo, &my_hi);
      } else {
        my_lo = max64(i - p.window + 1, p.kv_start);
        my_hi = min64(i, kv_end - 1);
      }
      // This row's valid columns of tile t are [lo0 - 128 t, hi0 - 128 t)
      // for a window tile and [0, lm0 - 128 t) for a landmark tile, each
      // clamped to [0, 128).  32-bit values keep the tile loop light: with
      // at most 2^29 keys (the launch checks it) lo0 lies in [0, 2^30) and
      // hi0 below it; a very negative hi0 (a row before the chunk) is
      // clamped.  Selected blocks lie wholly before every row's window: no
      // mask.
      const int64_t wbase =
          p.kv_start + static_cast<int64_t>(r.w.kt_lo - r.w.n_lm_tiles) * kBN;
      r.lo0 = static_cast<int>(my_lo - wbase);
      r.hi0 = static_cast<int>(max64(-(int64_t(1) << 30), my_hi - wbase + 1));
      r.lm0 = p.select ? (1 << 30)
                       : static_cast<int>(visible_landmarks(i, p.window, p.block, p.G));
      if (!r.row_ok) {  // no valid column
        r.hi0 = r.lo0 = 1 << 30;
        r.lm0 = 0;
      }
      return r;
    };
    RowUnit nx;
    int nx_u = -1;
    bool ok = true;
    for (int u = cid; ok && u < p.units; u += n_clusters) {
      const RowUnit ru = nx_u == u ? nx : row_unit(u);
      const Unit& w = ru.w;
      if (slot >= w.n_slots) continue;
      const bool has = ru.has;
      const int h = ru.h;
      const int64_t i_loc = ru.i_loc;
      const bool row_ok = ru.row_ok;
      if (w.T == 0) {  // no key for any row of this unit (partial chunks only)
        const int64_t lse_idx = static_cast<int64_t>(h) * p.lse_ld + i_loc;
        if (has && row_ok && !p.merge &&
            MSA_IN_RANGE(lse_idx, 1, (p.Hq - 1) * p.lse_ld + p.n_q, p.status))
          p.lse[lse_idx] = -INFINITY;
        continue;
      }
      const int lo0 = ru.lo0, hi0 = ru.hi0, lm0 = ru.lm0;
      float m_used = -INFINITY;
      float l = 0.f;
      for (int t = 0; t < w.T; ++t) {
        if (!(ok = wait_pair_w(bar(BAR_SF(slot)), (sc + t) & 1, ctl))) break;
        ptx::tc_fence_after();
        if (has) {
          float s[128];
          ptx::tmem_ld32(tS + 0, *reinterpret_cast<float(*)[32]>(&s[0]));
          ptx::tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
          ptx::tmem_ld32(tS + 64, *reinterpret_cast<float(*)[32]>(&s[64]));
          ptx::tmem_ld32(tS + 96, *reinterpret_cast<float(*)[32]>(&s[96]));
          ptx::tmem_wait_ld();
          // Valid columns [lo, hi) of this tile for this row.
          const int lo = t < w.n_lm_tiles ? 0 : lo0 - t * kBN;
          const int hi = (t < w.n_lm_tiles ? lm0 : hi0) - t * kBN;
          // Boundary tiles only, each side on its own (the diagonal and the
          // last landmark tile cut only above, the first window tile only
          // below): one compare with a constant and one select per score.
          // Both branches are uniform across the warp.
          const int lo_c = min(kBN, max(0, lo));
          const int hi_c = min(kBN, max(0, hi));
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
          if (need) l *= ptx::ex2(m_used - m_new);  // 0 when m_used = -inf
          // O holds PV(t-1) complete: S(t), which this warp waited for, was
          // issued after it and tcgen05 MMAs complete in order.
          if (__builtin_expect(t > 0 && __any_sync(0xffffffffu, need), 0)) {
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
          // p = 2^(s*scale*log2e - m), rounded to bf16 pairs for the PV MMA;
          // the denominator sums those same rounded weights.
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
        }
        ptx::tc_fence_before();
        __syncwarp();
        pair::arrive_cluster_w(pf);
        if (t + 1 == w.T && u + n_clusters < p.units) {
          nx_u = u + n_clusters;
          nx = row_unit(nx_u);
        }
      }
      if (ok) ok = wait_pair_w(bar(BAR_OD(slot)), oc & 1, ctl);
      if (!ok) break;
      ptx::tc_fence_after();
      // Epilogue.  The O reads complete (wait::ld) before this slot arrives
      // for the next unit's first P, which the lead waits for before the
      // next unit's first PV overwrites O.
      const bool hv = has && row_ok && l > 0.f;
      const int64_t lse_idx = static_cast<int64_t>(h) * p.lse_ld + i_loc;
      const int64_t obase = (i_loc * p.Hq + h) * static_cast<int64_t>(kD);
      // Offsets of a row this CTA writes, against the extents of O [n_q, Hq,
      // d] and lse [Hq][lse_ld] (checked in the bounds-checked build only).
      const bool io_ok =
          !(has && row_ok) ||
          (MSA_IN_RANGE(lse_idx, 1, (p.Hq - 1) * p.lse_ld + p.n_q, p.status) &&
           MSA_IN_RANGE(obase, kD, p.n_q * p.Hq * static_cast<int64_t>(kD), p.status));
      // O = acc * w_new (+ running O * w_run when merging into a running
      // result: lse_run <- ln(e^lse_run + e^lse_p)).
      const float lse_p = hv ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      float w_new = hv ? 1.f / l : 0.f;
      float w_run = 0.f;
      float lse_out = lse_p;
      if (p.merge && hv && io_ok) {
        const float L = p.lse[lse_idx];
        if (L != -INFINITY) {
          const float mx = fmaxf(L, lse_p);
          lse_out = mx + logf(expf(L - mx) + expf(lse_p - mx));
          w_run = expf(L - lse_out);
          w_new *= expf(lse_p - lse_out);
        }
      }
      // O of a warp whose valid rows all have a key (bf16, or fp32 when not
      // merging into a running result): staged in shared memory (the
      // 128-byte swizzle of tm_o's box: 32 rows x 64 bf16 or 32 fp32) and
      // written by one bulk tensor store per box; rows past n_q are clipped.
      // Stores of global memory from each thread's own row would touch 32
      // lines per instruction and hold the warp in the epilogue.
      const int row0 = static_cast<int>(w.qr0) + wq * 32;
      if (has && p.merge && !p.out_bf16 && __all_sync(0xffffffffu, io_ok)) {
        // Running merge: each 32 x 32 fp32 box of the running O is loaded
        // into the buffer (TMA, this warp's barrier), combined there with
        // this chunk's O row by row, and stored back; rows without a key in
        // this chunk write back what they loaded.
        if (row0 < p.n_q) {
          (void)MSA_TMA_OK(0, h, row0, kD, p.Hq, p.n_q, 32, p.status);
          const uint32_t stg = sb + kOffOut + static_cast<uint32_t>((warp - 4) * kOutStageBytes);
          const uint32_t my = stg + static_cast<uint32_t>(lane * 128);
          const uint32_t lbar = bar(BAR_OL(warp));
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            if (lane == 0) {
              ptx::bulk_wait_read();  // the buffer's last store has read it
              ptx::mbar_arrive_expect_tx(lbar, kOutStageBytes);
              ptx::tma_load_3d(stg, &p.tm_o, lbar, cc * 32, h, row0);
            }
            ++ol_issued;
            float o[32];
            ptx::tmem_ld32(tO + cc * 32, o);
            ptx::tmem_wait_ld();
            if (!(ok = wait_pair_w(lbar, ol_done & 1, ctl))) break;
            ++ol_done;
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16-byte chunk j of row `lane`, swizzled
              const uint32_t a = my + static_cast<uint32_t>(((j ^ lane) & 7) << 4);
              uint32_t r[4];
              ptx::ld_shared_v4(a, r[0], r[1], r[2], r[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float rv = __uint_as_float(r[e]);
                const float nv = w_run != 0.f ? fmaf(rv, w_run, o[4 * j + e] * w_new)
                                              : o[4 * j + e] * w_new;
                r[e] = hv ? __float_as_uint(nv) : r[e];
              }
              ptx::st_shared_v4(a, r[0], r[1], r[2], r[3]);
            }
            ptx::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(&p.tm_o, stg, cc * 32, h, row0);
              ptx::bulk_commit();
            }
          }
          if (!ok) break;
        }
      } else if (has && !p.merge && __all_sync(0xffffffffu, (hv || !row_ok) && io_ok)) {
        const uint32_t stg = sb + kOffOut + static_cast<uint32_t>((warp - 4) * kOutStageBytes);
        const uint32_t my = stg + static_cast<uint32_t>(lane * 128);
        if (row0 < p.n_q && !p.out_bf16) {
          (void)MSA_TMA_OK(0, h, row0, kD, p.Hq, p.n_q, 32, p.status);
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            float o[32];
            ptx::tmem_ld32(tO + cc * 32, o);
            ptx::tmem_wait_ld();
            if (lane == 0) ptx::bulk_wait_read();  // the buffer's last store has read it
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)  // 16-byte chunk j of row `lane`, swizzled
              ptx::st_shared_v4(my + static_cast<uint32_t>(((j ^ lane) & 7) << 4),
                                __float_as_uint(o[4 * j + 0] * w_new),
                                __float_as_uint(o[4 * j + 1] * w_new),
                                __float_as_uint(o[4 * j + 2] * w_new),
                                __float_as_uint(o[4 * j + 3] * w_new));
            ptx::fence_async_shared();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(&p.tm_o, stg, cc * 32, h, row0);
              ptx::bulk_commit();
            }
          }
        } else if (row0 < p.n_q) {
          (void)MSA_TMA_OK(0, h, row0, kD, p.Hq, p.n_q, 32, p.status);
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
          if (hv && io_ok) {
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
      if (has && row_ok && io_ok && (hv || !p.merge)) p.lse[lse_idx] = lse_out;
      sc += w.T;
      oc += 1;
    }
    // This warp's bulk stores of O complete before shared memory is released,
    // and a running-O load left waiting by an abort lands first.
    if (lane == 0) {
      if (ol_issued != ol_done)
        drain_for(bar(BAR_OL(warp)), ol_done & 1, p.status, kDrainLimitNs);
      ptx::bulk_wait_all();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) drain_for(bar(BAR_CLEAN), 0, p.status, kDrainLimitNs);  // the lead's last commit
  ptx::tc_fence_before();
  pair::cluster_sync();  // neither CTA leaves while the other may still address it
  if (warp == 1) {
    ptx::tc_fence_after();
    pair::tmem_dealloc(tmem, 512);
  }
}

constexpr int kMaxDev = 64;
std::mutex g_occ_mu;
int g_max_clusters[kMaxDev] = {};

}  // namespace

bool attn_tc2_supported(int Hq, int Hkv, int d, int in_bf16) {
  return in_bf16 && d == kD && Hkv > 0 && Hq / Hkv >= 2;
}

cudaError_t launch_attn_tc2(const AttnArgs& a, cudaStream_t s, const char** why) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  Tc2Params p;
  memset(&p, 0, sizeof(p));
  const bool lm_maps = a.G > 0 && !a.sel;
  const bool ok = encode_map(fn, &p.tm_q, a.q, a.n_q, a.Hq, 128) &&
                  encode_map(fn, &p.tm_k, a.k, a.n_kv, a.Hkv, 64) &&
                  encode_map(fn, &p.tm_v, a.v, a.n_kv, a.Hkv, 128) &&
                  (lm_maps ? encode_map(fn, &p.tm_klm, a.k_lm, a.G, a.Hkv, 64) &&
                                 encode_map(fn, &p.tm_vlm, a.v_lm, a.G, a.Hkv, 128)
                           : true) &&
                  (a.out_bf16 ? encode_map(fn, &p.tm_o, a.out, a.n_q, a.Hq, 32)
                              : encode_map_f32(fn, &p.tm_o, a.out, a.n_q, a.Hq, 32));
  if (!ok) {
    *why = "cuTensorMapEncodeTiled rejected a tensor (alignment or size)";
    return cudaErrorInvalidValue;
  }
  if (!lm_maps) {  // no landmark tensors read
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
  p.quads = (p.group + 3) / 4;
  p.n_qtiles = static_cast<int>((a.n_q + kBM - 1) / kBM);
  p.out_bf16 = a.out_bf16;
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
  const int64_t units = static_cast<int64_t>(a.Hkv) * p.quads * p.n_qtiles;
  p.units = static_cast<int>(units);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) {
    *why = "device ordinal out of range";
    return cudaErrorInvalidDevice;
  }
  int max_clusters = 0;
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    max_clusters = g_max_clusters[dev];
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
  // Function attributes belong to the context: set on every launch (a
  // cudaDeviceReset in between would drop them); only the occupancy figure,
  // a property of the device, is cached.
  e = cudaFuncSetAttribute(attn_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;
  if (max_clusters == 0) {
    // The register split (setmaxnreg) assumes the launch allocation of
    // 168 registers per thread; refuse to launch a build that differs.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_tc2_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != 168) {
      *why = "pair attention kernel built with an unexpected register count";
      return cudaErrorInvalidConfiguration;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    e = cudaOccupancyMaxActiveClusters(&max_clusters, attn_tc2_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) {
      *why = "no CTA pair of the attention kernel fits on this device";
      return cudaErrorInvalidConfiguration;
    }
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_max_clusters[dev] = max_clusters;
  }
  int64_t clusters = units < max_clusters ? units : max_clusters;
  if (a.max_clusters > 0 && clusters > a.max_clusters) clusters = a.max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  e = cudaLaunchKernelEx(&cfg, attn_tc2_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();
}

}  // namespace msa
