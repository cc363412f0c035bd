// K5: global query rows -- the rows that attend every earlier key in the
// block-sparse pattern of "Training at 1M+ Token Context: Ring Attention,
// YaRN, NTK-Aware Scaling GPU Cost" (Block-Sparse Flash Attention
// paragraph: global tokens attend to all, local tokens to a sliding window,
// compression tokens summarise distant context).  The local rows and their
// compression tokens are the window + landmark attention with 32-token
// blocks; this file computes the few global rows, each attending keys
// j <= its position, and overwrites their O and lse.
//
// Few query rows against many keys: the work is split over the key axis.
// For KV head c the M dimension is the (global row r, query head c*g + hh)
// pairs, m = r*g + hh, so one 128-row M tile holds 128/g global rows that
// all read the same K/V tiles.  Each CTA computes one (key split, M tile,
// KV head) partial -- O normalised by its own sum, and its lse -- into a
// workspace; a merge kernel combines the splits per (row, head) exactly
// (lse = ln sum e^{lse_s}, O = sum e^{lse_s - lse} O_s, the Ring Attention
// combination) and writes the rows of O and lse.
//
// Tensor-core kernel (bf16, d = 128), 6 warps:
//   warps 0-3  load their M row of Q into shared memory (128-byte swizzle,
//              the layout TMA would write), softmax of the S tile rows,
//              epilogue;
//   warp 4     TMA producer of K/V tiles through a 2-stage ring;
//   warp 5     allocates 256 TMEM columns (S: 0..127, P over its first 64;
//              O: 128..255); the warp issues S = Q K^T and O += P V (one elected
//              lane per instruction).
// Per tile: S MMA -> softmax -> P -> PV MMA, in order; S(t+1) is issued
// after PV(t), so the completion of S(t+1) also means PV(t) is done and O
// may be rescaled.  Every wait is bounded as in the attention kernel.
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
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kChunkBytes = 128 * 128;
constexpr int kTileBytes = 2 * kChunkBytes;
constexpr int kThreads = 192;
constexpr float kTau = 8.0f;

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + 2 * kTileBytes;
constexpr int kOffBar = kOffV + 2 * kTileBytes;
enum { BAR_KVF0 = 0, BAR_KVE0 = 2, BAR_SF = 4, BAR_PF = 5, BAR_OF = 6, BAR_CLEAN = 7, kNumBars = 8 };
constexpr int kOffPos = kOffBar + 8 * kNumBars;      // int64 position of each M row
constexpr int kOffTmemSlot = kOffPos + 8 * kBM;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;

struct GrParams {
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const uint16_t* q;  // bf16 bits [n, Hq, 128]
  const int64_t* rows;
  float* o_part;
  float* lse_part;
  int64_t n, Mc, span;
  int Hq, Hkv, group;
  float scale_log2;
  int* status;
  uint64_t wait_ns;
};

// Position of M row m of KV head c (-1: past the end, or an invalid row,
// which is reported).
__device__ __forceinline__ int64_t row_position(const int64_t* rows, int64_t m, int64_t Mc,
                                                int group, int64_t n, int* status) {
  if (m >= Mc) return -1;
  if (!MSA_IN_RANGE(m / group, 1, Mc / group, status)) return -1;
  const int64_t pos = rows[m / group];
  if (pos < 0 || pos >= n) {
    record_status(status, MSA_ERR_INVALID_ARG);
    return -1;
  }
  return pos;
}

__global__ void __launch_bounds__(kThreads, 1)
    global_rows_tc_kernel(const __grid_constant__ GrParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  int64_t* spos = reinterpret_cast<int64_t*>(smem + kOffPos);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };

  const int split = blockIdx.x;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kBM;
  const int c = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t part = static_cast<int64_t>(split) * p.Hkv + c;  // (split, head) slab

  // Positions and the Q tile: thread t < 128 owns M row m0 + t.
  if (threadIdx.x < kBM) {
    const int t = threadIdx.x;
    const int64_t pos = row_position(p.rows, m0 + t, p.Mc, p.group, p.n, p.status);
    spos[t] = pos;
    uint4 g16[16];
    const int h = c * p.group + static_cast<int>((m0 + t) % p.group);
    if (pos >= 0 && MSA_IN_RANGE((pos * p.Hq + h) * static_cast<int64_t>(kD), kD,
                                 p.n * p.Hq * static_cast<int64_t>(kD), p.status)) {
      const uint4* src =
          reinterpret_cast<const uint4*>(p.q + (pos * p.Hq + h) * static_cast<int64_t>(kD));
#pragma unroll
      for (int j = 0; j < 16; ++j) g16[j] = __ldg(src + j);
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) g16[j] = make_uint4(0, 0, 0, 0);
    }
    // 16-byte granule j of row t: chunk j/8, granule (j%8) ^ (t%8).
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<uint4*>(smem + kOffQ + (j >> 3) * kChunkBytes + t * 128 +
                                (((j & 7) ^ (t & 7)) << 4)) = g16[j];
    ptx::fence_async_shared();  // generic-proxy writes -> visible to the MMA
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(BAR_KVF0 + b), 1);
      ptx::mbar_init(bar(BAR_KVE0 + b), 1);
    }
    ptx::mbar_init(bar(BAR_SF), 1);
    ptx::mbar_init(bar(BAR_PF), 4);
    ptx::mbar_init(bar(BAR_OF), 1);
    ptx::mbar_init(bar(BAR_CLEAN), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  __syncthreads();

  // Keys of this split that some row of the tile attends: [key_lo, key_end).
  int64_t max_pos = -1;
  for (int t = 0; t < kBM; ++t) max_pos = max64(max_pos, spos[t]);
  const int64_t key_lo = static_cast<int64_t>(split) * p.span;
  const int64_t key_end = min64(key_lo + p.span, max_pos + 1);
  const int T = key_end > key_lo ? static_cast<int>((key_end - key_lo + kBN - 1) / kBN) : 0;
  if (T == 0) {  // no row of the tile reaches this split
    if (threadIdx.x < kBM && m0 + threadIdx.x < p.Mc &&
        MSA_IN_RANGE(part * p.Mc + m0 + threadIdx.x, 1,
                     static_cast<int64_t>(gridDim.x) * p.Hkv * p.Mc, p.status))
      p.lse_part[part * p.Mc + m0 + threadIdx.x] = -INFINITY;
    return;
  }

  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 256);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  WaitCtl ctl{abort_flag, p.status, p.wait_ns};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&p.tm_k);
      ptx::tma_prefetch_desc(&p.tm_v);
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int b = t & 1;
        if (t >= 2 && !wait_bar(bar(BAR_KVE0 + b), ((t >> 1) - 1) & 1, ctl)) break;
        const uint32_t full = bar(BAR_KVF0 + b);
        ptx::mbar_arrive_expect_tx(full, 2 * kTileBytes);
        const int row = static_cast<int>(key_lo + static_cast<int64_t>(t) * kBN);
        for (int ch = 0; ch < 2; ++ch) {
          // Box origins are only recorded when out of range: the copy is
          // issued all the same (out-of-range rows read the fill value).
          (void)MSA_TMA_OK(ch * 64, c, row, kD, p.Hkv, p.n, kBN, p.status);
          ptx::tma_load_3d(sb + kOffK + b * kTileBytes + ch * kChunkBytes, &p.tm_k, full, ch * 64,
                           c, row);
          ptx::tma_load_3d(sb + kOffV + b * kTileBytes + ch * kChunkBytes, &p.tm_v, full, ch * 64,
                           c, row);
        }
        issued = t + 1;
      }
      // Drain: the last copy issued into each stage has landed.
      for (int b = 0; b < 2; ++b) {
        int last = issued - 1;
        if (last >= 0 && (last & 1) != b) --last;
        if (last >= 0) drain_bar(bar(BAR_KVF0 + b), (last >> 1) & 1, p.status);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // (the whole warp runs the loop; elect.sync picks the issuing lane)
    {
      constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(kBM, kBN, false);
      constexpr uint32_t kIdescO = ptx::idesc_bf16_f32(kBM, kD, true);
      constexpr uint32_t kTileLo = kTileBytes >> 4;
      const uint32_t q_lo = ptx::desc_lo(sb + kOffQ, 16);
      const uint32_t k_lo0 = ptx::desc_lo(sb + kOffK, 16);
      const uint32_t v_lo0 = ptx::desc_lo(sb + kOffV, kChunkBytes);
      bool ok = true;
      for (int t = 0; ok && t < T; ++t) {
        const int b = t & 1;
        if (!(ok = wait_w(bar(BAR_KVF0 + b), (t >> 1) & 1, ctl))) break;
        ptx::tc_fence_after();
        const uint32_t kb = k_lo0 + b * kTileLo;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          ptx::mma_ss_w(tmem, q_lo + off, ptx::kDescHiSw128, kb + off, ptx::kDescHiSw128,
                           kIdescS, kk > 0 ? 1u : 0u);
        }
        ptx::commit_w(bar(BAR_SF));
        if (!(ok = wait_w(bar(BAR_PF), t & 1, ctl))) break;
        ptx::tc_fence_after();
        const uint32_t vb = v_lo0 + b * kTileLo;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          ptx::mma_ts_w(tmem + 128, tmem + kk * 8, vb + ((kk * 2048) >> 4), ptx::kDescHiSw128,
                           kIdescO, (t > 0 || kk > 0) ? 1u : 0u);
        ptx::commit_w(bar(BAR_KVE0 + b));
      }
      if (ok) ptx::commit_w(bar(BAR_OF));
      ptx::commit_w(bar(BAR_CLEAN));
      drain_bar(bar(BAR_CLEAN), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t tS = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t tO = tS + 128;
    const int t_row = threadIdx.x;
    const int64_t m = m0 + t_row;
    const int64_t pos = spos[t_row];
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF), t & 1, ctl));
      if (!ok) break;
      ptx::tc_fence_after();
      float s[128];
      ptx::tmem_ld32(tS + 0, *reinterpret_cast<float(*)[32]>(&s[0]));
      ptx::tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
      ptx::tmem_ld32(tS + 64, *reinterpret_cast<float(*)[32]>(&s[64]));
      ptx::tmem_ld32(tS + 96, *reinterpret_cast<float(*)[32]>(&s[96]));
      ptx::tmem_wait_ld();
      // Keys kb + col with kb + col <= pos are attended.
      const int64_t kb = key_lo + static_cast<int64_t>(t) * kBN;
      const int64_t hi = pos - kb + 1;
      if (hi < kBN) {
        const int hi_c = static_cast<int>(max64(0, hi));
#pragma unroll
        for (int col = 0; col < 128; ++col) s[col] = col < hi_c ? s[col] : -INFINITY;
      }
      float a0 = fmaxf(s[0], s[1]), a1 = fmaxf(s[2], s[3]);
      float a2 = fmaxf(s[4], s[5]), a3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int col = 8; col < 128; col += 8) {
        a0 = ptx::max3(a0, s[col], s[col + 1]);
        a1 = ptx::max3(a1, s[col + 2], s[col + 3]);
        a2 = ptx::max3(a2, s[col + 4], s[col + 5]);
        a3 = ptx::max3(a3, s[col + 6], s[col + 7]);
      }
      const float mx = ptx::max3(a0, a1, fmaxf(a2, a3));
      const float m_new = fmaxf(m_used, mx * sl2);
      const bool need = m_new > m_used + kTau;
      if (need) l *= ptx::ex2(m_used - m_new);  // 0 when m_used = -inf
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
      // P rounded to bf16 for the PV MMA; l sums the rounded weights.
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
      if (lane == 0) ptx::mbar_arrive(bar(BAR_PF));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_OF), 0, ctl));
    if (ok) {
      ptx::tc_fence_after();
      const int64_t all_m = static_cast<int64_t>(gridDim.x) * p.Hkv * p.Mc;
      (void)all_m;
      const bool has = pos >= 0 && l > 0.f &&
                       MSA_IN_RANGE((part * p.Mc + m) * static_cast<int64_t>(kD), kD,
                                    all_m * kD, p.status);
      const float w = has ? 1.f / l : 0.f;
      float* dst = p.o_part + (part * p.Mc + m) * static_cast<int64_t>(kD);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float o[32];
        ptx::tmem_ld32(tO + cc * 32, o);
        ptx::tmem_wait_ld();
        if (has) {
          float4* d4 = reinterpret_cast<float4*>(dst + cc * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            d4[v] = make_float4(o[4 * v] * w, o[4 * v + 1] * w, o[4 * v + 2] * w,
                                o[4 * v + 3] * w);
        }
      }
      if (m < p.Mc && MSA_IN_RANGE(part * p.Mc + m, 1, all_m, p.status))
        p.lse_part[part * p.Mc + m] =
            has ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 256);
  }
}

// ------------------------------------------------------------ CUDA-core path
// One warp per (split, M row, KV head): keys of the split up to the row's
// position, exact online softmax in fp32, lanes split the head dimension.
template <bool kBf16, int D>
__global__ void __launch_bounds__(128)
    global_rows_simt_kernel(const void* q, const void* k, const void* v, const int64_t* rows,
                            float* o_part, float* lse_part, int64_t n, int64_t Mc, int64_t span,
                            int Hq, int Hkv, int group, float scale_log2, int* status) {
  constexpr int E = D / 32;  // elements per lane
  const int split = blockIdx.x;
  const int64_t m = static_cast<int64_t>(blockIdx.y) * 4 + (threadIdx.x >> 5);
  const int c = blockIdx.z;
  const int lane = threadIdx.x & 31;
  if (m >= Mc) return;
  const int64_t part = static_cast<int64_t>(split) * Hkv + c;
  const int64_t pos = row_position(rows, m, Mc, group, n, status);
  const int64_t key_lo = static_cast<int64_t>(split) * span;
  const int64_t key_end = pos < 0 ? key_lo : min64(key_lo + span, pos + 1);
  auto ld = [&](const void* base, int64_t idx) -> float {
    if constexpr (kBf16)
      return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
    else
      return static_cast<const float*>(base)[idx];
  };
  float qv[E], o[E];
  const int h = c * group + static_cast<int>(m % group);
  const bool q_ok = pos >= 0 && MSA_IN_RANGE((pos * Hq + h) * static_cast<int64_t>(D), D,
                                             n * Hq * static_cast<int64_t>(D), status);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qv[e] = q_ok ? ld(q, (pos * Hq + h) * static_cast<int64_t>(D) + lane * E + e) : 0.f;
    o[e] = 0.f;
  }
  float mrun = -INFINITY, l = 0.f;
  for (int64_t j = key_lo; j < key_end; ++j) {
    const int64_t base = (j * Hkv + c) * static_cast<int64_t>(D) + lane * E;
    // The whole key row, so that every lane takes the same branch.
    if (!MSA_IN_RANGE((j * Hkv + c) * static_cast<int64_t>(D), D,
                      n * Hkv * static_cast<int64_t>(D), status))
      break;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) dot = fmaf(qv[e], ld(k, base + e), dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float sc = dot * scale_log2;
    const float m_new = fmaxf(mrun, sc);
    const float alpha = exp2f(mrun - m_new);
    const float pj = exp2f(sc - m_new);
    l = l * alpha + pj;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = fmaf(pj, ld(v, base + e), o[e] * alpha);
    mrun = m_new;
  }
  const int64_t all_m = static_cast<int64_t>(gridDim.x) * Hkv * Mc;
  (void)all_m;
  if (!MSA_IN_RANGE(part * Mc + m, 1, all_m, status)) return;
  const bool has = l > 0.f;
  if (has) {
    const float w = 1.f / l;
    float* dst = o_part + (part * Mc + m) * static_cast<int64_t>(D) + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = o[e] * w;
  }
  if (lane == 0)
    lse_part[part * Mc + m] = has ? (mrun + log2f(l)) * 0.69314718055994530942f : -INFINITY;
}

// ------------------------------------------------------------ merge + scatter
// One warp per (global row, query head): combine the splits' partials and
// write row pos of O and lse.  Invalid rows (already reported) are skipped.
template <int D>
__global__ void __launch_bounds__(128)
    global_rows_merge_kernel(const int64_t* rows, const float* o_part, const float* lse_part,
                             void* out, float* lse, int64_t n, int64_t n_global, int64_t Mc,
                             int n_splits, int Hq, int Hkv, int group, int out_bf16,
                             int* status) {
  constexpr int E = D / 32;
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= n_global * Hq) return;
  const int64_t r = pair / Hq;
  const int h = static_cast<int>(pair % Hq);
  const int c = h / group;
  const int64_t m = r * group + h % group;
  const int64_t pos = rows[r];
  if (pos < 0 || pos >= n) return;
  // Every partial index below is (s * Hkv + c) * Mc + m with s < n_splits.
  if (!MSA_IN_RANGE((static_cast<int64_t>(n_splits - 1) * Hkv + c) * Mc + m, 1,
                    static_cast<int64_t>(n_splits) * Hkv * Mc, status) ||
      !MSA_IN_RANGE((pos * Hq + h) * static_cast<int64_t>(D), D, n * Hq * static_cast<int64_t>(D),
                    status) ||
      !MSA_IN_RANGE(static_cast<int64_t>(h) * n + pos, 1, static_cast<int64_t>(Hq) * n, status))
    return;
  float mx = -INFINITY;
  for (int s = lane; s < n_splits; s += 32)
    mx = fmaxf(mx, lse_part[(static_cast<int64_t>(s) * Hkv + c) * Mc + m]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (mx == -INFINITY) return;  // cannot happen for a valid row (it attends itself)
  float sum = 0.f;
  for (int s = lane; s < n_splits; s += 32) {
    const float L = lse_part[(static_cast<int64_t>(s) * Hkv + c) * Mc + m];
    if (L != -INFINITY) sum += expf(L - mx);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float total = mx + logf(sum);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const int64_t ps = (static_cast<int64_t>(s) * Hkv + c) * Mc + m;
    const float L = lse_part[ps];
    if (L == -INFINITY) continue;
    const float w = expf(L - total);
    const float* src = o_part + ps * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, src[e], acc[e]);
  }
  const int64_t ob = (pos * Hq + h) * static_cast<int64_t>(D) + lane * E;
  if (out_bf16) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = __float2bfloat16_rn(acc[e]);
  } else {
    float* dst = static_cast<float*>(out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = acc[e];
  }
  if (lane == 0) lse[static_cast<int64_t>(h) * n + pos] = total;
}

}  // namespace

cudaError_t launch_global_rows(const GlobalRowsArgs& a, cudaStream_t s, const char** why) {
  const int group = a.Hq / a.Hkv;
  const float sl2 = a.scale * 1.4426950408889634f;
  const int64_t Mc = a.n_global * group;
  const bool tc = a.in_bf16 && a.d == kD;
  if (tc) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) {
      *why = "cuTensorMapEncodeTiled is not available from the driver";
      return cudaErrorNotSupported;
    }
    GrParams p;
    memset(&p, 0, sizeof(p));
    if (!encode_map(fn, &p.tm_k, a.k, a.n, a.Hkv) || !encode_map(fn, &p.tm_v, a.v, a.n, a.Hkv)) {
      *why = "cuTensorMapEncodeTiled rejected a tensor (alignment or size)";
      return cudaErrorInvalidValue;
    }
    p.q = static_cast<const uint16_t*>(a.q);
    p.rows = a.rows;
    p.o_part = a.o_part;
    p.lse_part = a.lse_part;
    p.n = a.n;
    p.Mc = Mc;
    p.span = a.span;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = group;
    p.scale_log2 = sl2;
    p.status = a.status;
    p.wait_ns = a.wait_limit_ns;
    cudaError_t e = cudaFuncSetAttribute(global_rows_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(a.n_splits, static_cast<unsigned>((Mc + kBM - 1) / kBM), a.Hkv);
    global_rows_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  } else {
    dim3 grid(a.n_splits, static_cast<unsigned>((Mc + 3) / 4), a.Hkv);
#define MSA_GR_SIMT(BF, D)                                                                      \
  global_rows_simt_kernel<BF, D><<<grid, 128, 0, s>>>(a.q, a.k, a.v, a.rows, a.o_part,          \
                                                      a.lse_part, a.n, Mc, a.span, a.Hq, a.Hkv, \
                                                      group, sl2, a.status)
    if (a.in_bf16 && a.d == 64) MSA_GR_SIMT(true, 64);
    else if (a.in_bf16) MSA_GR_SIMT(true, 128);
    else if (a.d == 64) MSA_GR_SIMT(false, 64);
    else MSA_GR_SIMT(false, 128);
#undef MSA_GR_SIMT
  }
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  const unsigned mblocks = static_cast<unsigned>((a.n_global * a.Hq + 3) / 4);
  if (a.d == 64)
    global_rows_merge_kernel<64><<<mblocks, 128, 0, s>>>(a.rows, a.o_part, a.lse_part, a.out,
                                                         a.lse, a.n, a.n_global, Mc, a.n_splits,
                                                         a.Hq, a.Hkv, group, a.out_bf16, a.status);
  else
    global_rows_merge_kernel<128><<<mblocks, 128, 0, s>>>(a.rows, a.o_part, a.lse_part, a.out,
                                                          a.lse, a.n, a.n_global, Mc, a.n_splits,
                                                          a.Hq, a.Hkv, group, a.out_bf16, a.status);
  return cudaPeekAtLastError();
}

}  // namespace msa
