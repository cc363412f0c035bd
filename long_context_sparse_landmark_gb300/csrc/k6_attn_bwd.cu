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
//   1. bwd_preprocess_kernel: per-row lse (log2 units) and D (fp32), padded
//      to whole 128-row tiles so that the dK/dV kernel copies them per tile;
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
// Each tensor-core kernel: warps 0-7 elementwise (TMEM lane = row; warps w
// and w + 4 share a row quarter and split the columns), warp 8 TMA
// producer, warp 9 TMEM allocation and MMA issue.  tcgen05 MMAs from one
// warp execute in issue order, which makes overwriting TMEM columns after
// the MMAs that read them safe.
//   dK/dV: TMEM holds two accumulators, so every 128-column tile is handled
//   as two 64-column halves with their own columns: the score-like MMAs of
//   a half land, the elementwise warps turn them into bf16 P / dS in the
//   same columns, the half's gradient MMAs accumulate in TMEM and the next
//   tile's scores of that half follow at once -- the tensor pipe works on
//   one half while the warps process the other.  Q and dO arrive in 64-row
//   halves through a 4-stage ring, each half released by its own MMAs.
//   dQ: one accumulator leaves room for two full-width dP buffers (dS is
//   written over its tile's dP), so the next tile's dP is computed during
//   the elementwise pass and its S as soon as every warp has read this
//   tile's S; K and V come through separate rings (three K stages, since K
//   is read until the late dQ MMAs).
// Every wait is bounded; a wait that runs out aborts the CTA cleanly.
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
constexpr int kHalf = 64;                    // columns per pipelined half
constexpr int kChunkBytes = 128 * 128;       // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kChunkBytes;  // 128 rows x 128 bf16
constexpr uint32_t kTileLo = kTileBytes >> 4;
// Warps: 0-7 elementwise (warps w and w + 4 share TMEM lanes 32(w % 4)..+31,
// i.e. the same 32 rows, and split each tile's columns), 8 TMA producer,
// 9 TMEM allocation and MMA issue.
constexpr int kEwWarps = 8;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory: a fixed pair of tiles (dQ: Q, dO; dK/dV: K, V), then the
// rings.  dK/dV: a 4-stage ring of 64-row halves of the query tiles (Q half,
// dO half; 32 KB a stage): a half is released as soon as its own gradient
// MMAs are done, so each copy has about one whole tile of time to land.
constexpr int kOffFixA = 0;
constexpr int kOffFixB = kTileBytes;
constexpr int kHalfChunk = kChunkBytes / 2;              // 64 rows x 64 bf16
constexpr int kHalfTileBytes = kTileBytes / 2;           // 64 rows x 128 bf16
constexpr int kRing = 4;                                 // dK/dV half-tile stages
constexpr int kOffRing = 2 * kTileBytes;
constexpr int kRingStageBytes = 2 * kHalfTileBytes;      // Q half + dO half
constexpr int kOffBar = kOffRing + kRing * kRingStageBytes;  // 192 KB
enum {
  BAR_FIX = 0,      // fixed tiles landed
  BAR_FULL0 = 1,    // ring stage s landed (1..4)
  BAR_EMPTY0 = 5,   // ring stage s consumed (5..8)
  BAR_SF0 = 9,      // score-like MMAs of half h done (9, 10)
  BAR_EF0 = 11,     // elementwise results of half h written, one arrival per warp (11, 12)
  BAR_ACC = 13,     // gradient accumulators final
  BAR_CLEAN = 14,
  kNumBars = 15
};
// dK/dV: [4 stages][L2, D, positions][64] 4-byte values of the stage's
// queries, bulk-copied: 128-byte aligned (positions only in the gathered
// global-row mode).
constexpr int kOffStats = (kOffBar + 8 * kNumBars + 127) / 128 * 128;
constexpr int kHalfRows = kT / 2;
constexpr int kStatBytes = 3 * kHalfRows * 4;  // one stage's L2, D and position rows
constexpr int kOffTmemSlot = kOffStats + kRing * kStatBytes;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
constexpr int kSmemBytes = kSmemUsed + 1024;

struct BwdParams {
  CUtensorMap tm_q, tm_do, tm_k, tm_v, tm_klm, tm_vlm;
  CUtensorMap tm_q64, tm_do64;  // Q, dO with 64-row boxes (the dK/dV ring)
  const float* L2;    // [Hq, n_pad] -lse * log2(e), -inf past n
  const float* D;     // [Hq, n_pad] -<dO, O>, 0 past n
  void* dq;           // [n, Hq, d]
  void* dk;           // [n, Hkv, d]
  void* dv;
  float* lm_part;     // [chunks][2][G][Hkv][d]
  const float* lm_grad;  // [2][G][Hkv][d]
  // Gathered global-row mode (kernels instantiated with kG = true): the
  // query side is the global rows,
  // M row m = r * group + hh of KV head c at position gpos[m] (-1: padding),
  // tm_q / tm_do map the gathered Qg / dOg [Mp][Hkv][d], L2 / D are
  // [Hkv][Mp]; each row attends every key j <= its position.
  const int* gpos;    // [Mp]
  float* dq_part;     // [n_splits][Hkv][Mp][d]: dQ of the global rows per key split
  float* extra_k;     // [n][Hkv][d]: the global rows' dK / dV, added by the
  float* extra_v;     //   window pass (null outside the global-row backward)
  int64_t n, n_pad, window, block, span, Mp;
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

// Set-up of the dK/dV kernel: barriers, TMEM (512 columns).
__device__ __forceinline__ uint32_t bwd_setup(uint8_t* smem, uint32_t sb, int warp) {
  if (threadIdx.x == 0) {
    ptx::mbar_init(sb + kOffBar + 8 * BAR_FIX, 1);
    for (int b = 0; b < kRing; ++b) {
      ptx::mbar_init(sb + kOffBar + 8 * (BAR_FULL0 + b), 1);
      ptx::mbar_init(sb + kOffBar + 8 * (BAR_EMPTY0 + b), 1);
    }
    for (int h = 0; h < 2; ++h) {
      ptx::mbar_init(sb + kOffBar + 8 * (BAR_SF0 + h), 1);
      ptx::mbar_init(sb + kOffBar + 8 * (BAR_EF0 + h), kEwWarps);
    }
    ptx::mbar_init(sb + kOffBar + 8 * BAR_ACC, 1);
    ptx::mbar_init(sb + kOffBar + 8 * BAR_CLEAN, 1);
    *reinterpret_cast<volatile int*>(smem + kOffAbort) = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(smem + kOffTmemSlot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
}

// Teardown of both kernels: every role done with TMEM, then free it.
__device__ __forceinline__ void bwd_teardown(uint32_t tmem, int warp) {
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Producer of the dK/dV kernel: the fixed pair (K, V) once, then both
// 64-row halves of `iters` query tiles; `coord(it, &map_a, &map_b, &y_a,
// &y_b, &row)` names the tensors (64-row boxes) and coordinates of tile it,
// `stats(it, &l2, &d, &pos)` the tile's statistics rows (positions only in
// the gathered mode).  Half u = 2 it + h goes to ring stage u % kRing.
// Bounds-checked build: a TMA box origin against the tensor its map covers
// -- K / V [n][Hkv], the landmarks [G][Hkv], Q / dO [n][Hq], or in the
// gathered mode the global rows [Mp][Hkv].  Recorded only; the copy is issued
// all the same (out-of-range rows read the fill value).  Empty otherwise.
template <bool kG>
__device__ __forceinline__ void check_box(const BwdParams& p, const CUtensorMap* m, int x, int y,
                                          int64_t z, int box) {
#ifdef MSA_DEBUG_BOUNDS
  int64_t rows;
  int heads;
  if (m == &p.tm_k || m == &p.tm_v) {
    rows = p.n;
    heads = p.Hkv;
  } else if (m == &p.tm_klm || m == &p.tm_vlm) {
    rows = p.G > 0 ? p.G : p.n;
    heads = p.Hkv;
  } else {
    rows = kG ? p.Mp : p.n;
    heads = kG ? p.Hkv : p.Hq;
  }
  (void)MSA_TMA_OK(x, y, z, kD, heads, rows, box, p.status);
#else
  (void)p, (void)m, (void)x, (void)y, (void)z, (void)box;
#endif
}

// Bounds-checked build: `count` 4-byte values at `src` lie in the row
// statistics (L2 / D: [Hq][n_pad], or [Hkv][Mp] gathered; positions [Mp]).
template <bool kG>
__device__ __forceinline__ bool stats_ok(const BwdParams& p, const void* src, int count) {
#ifdef MSA_DEBUG_BOUNDS
  const int64_t ext = kG ? static_cast<int64_t>(p.Hkv) * p.Mp : static_cast<int64_t>(p.Hq) * p.n_pad;
  const char* c = static_cast<const char*>(src);
  const char* bases[3] = {reinterpret_cast<const char*>(p.L2), reinterpret_cast<const char*>(p.D),
                          reinterpret_cast<const char*>(p.gpos)};
  const int64_t exts[3] = {ext, ext, kG ? p.Mp : 0};
  for (int k = 0; k < 3; ++k)
    if (bases[k] && c >= bases[k] && c < bases[k] + 4 * exts[k])
      return MSA_IN_RANGE((c - bases[k]) / 4, count, exts[k], p.status);
  return MSA_IN_RANGE(-1, count, 0, p.status);
#else
  (void)p, (void)src, (void)count;
  return true;
#endif
}

template <bool kG, typename Coord, typename Stats>
__device__ __forceinline__ void produce(uint32_t sb, const CUtensorMap* fa, const CUtensorMap* fb,
                                        int fy, int frow, int iters, Coord coord, Stats stats,
                                        const WaitCtl& ctl, int* status, const BwdParams& p) {
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };
  ptx::mbar_arrive_expect_tx(bar(BAR_FIX), 2 * kTileBytes);
  for (int ch = 0; ch < 2; ++ch) {
    check_box<kG>(p, fa, ch * 64, fy, frow, kT);
    check_box<kG>(p, fb, ch * 64, fy, frow, kT);
    ptx::tma_load_3d(sb + kOffFixA + ch * kChunkBytes, fa, bar(BAR_FIX), ch * 64, fy, frow);
    ptx::tma_load_3d(sb + kOffFixB + ch * kChunkBytes, fb, bar(BAR_FIX), ch * 64, fy, frow);
  }
  int issued = 0;
  for (int u = 0; u < 2 * iters; ++u) {
    const int it = u >> 1, h = u & 1, st = u % kRing;
    if (u >= kRing && !wait_bar(bar(BAR_EMPTY0 + st), ((u / kRing) - 1) & 1, ctl)) break;
    const CUtensorMap *ma, *mb;
    int ya, yb, row;
    coord(it, &ma, &mb, &ya, &yb, &row);
    row += h * kHalfRows;
    const float *sl = nullptr, *sd = nullptr;
    const int* sp = nullptr;
    stats(it, &sl, &sd, &sp);
    const uint32_t full = bar(BAR_FULL0 + st);
    ptx::mbar_arrive_expect_tx(
        full, 2 * kHalfTileBytes + (sl ? 2 * kHalfRows * 4 : 0) + (sp ? kHalfRows * 4 : 0));
    if (sl) {  // this half's per-query lse and D rows (256 bytes each)
      const uint32_t dst = sb + kOffStats + st * kStatBytes;
      // An untiled copy has no bounds of its own: the bounds-checked build
      // skips one whose source leaves the statistics (the stage's wait then
      // runs out and the launch ends with a status).
      if (stats_ok<kG>(p, sl + h * kHalfRows, kHalfRows))
        ptx::bulk_load(dst, sl + h * kHalfRows, kHalfRows * 4, full);
      if (stats_ok<kG>(p, sd + h * kHalfRows, kHalfRows))
        ptx::bulk_load(dst + kHalfRows * 4, sd + h * kHalfRows, kHalfRows * 4, full);
      if (sp && stats_ok<kG>(p, sp + h * kHalfRows, kHalfRows))
        ptx::bulk_load(dst + 2 * kHalfRows * 4, sp + h * kHalfRows, kHalfRows * 4, full);
    }
    const uint32_t base = sb + kOffRing + st * kRingStageBytes;
    for (int ch = 0; ch < 2; ++ch) {
      // The whole query tile (its second half may lie wholly past the end).
      check_box<kG>(p, ma, ch * 64, ya, row - h * kHalfRows, kT);
      check_box<kG>(p, mb, ch * 64, yb, row - h * kHalfRows, kT);
      ptx::tma_load_3d(base + ch * kHalfChunk, ma, full, ch * 64, ya, row);
      ptx::tma_load_3d(base + kHalfTileBytes + ch * kHalfChunk, mb, full, ch * 64, yb, row);
    }
    issued = u + 1;
  }
  drain_bar(bar(BAR_FIX), 0, status);
  for (int st = 0; st < kRing; ++st) {
    const int last = issued - 1 - ((issued - 1 - st) % kRing + kRing) % kRing;
    if (last >= 0) drain_bar(bar(BAR_FULL0 + st), (last / kRing) & 1, status);
  }
}

// Groups of MMAs issued from one asm block with one elect.sync (the whole
// MMA warp calls them; constant descriptor steps inside).  Unlike the
// forward kernel's groups, the operands here may have different chunk
// strides (a 128-row tile against a 64-row ring half) and the TMEM operand
// holds its packed pairs per 32-column chunk.
//
// Eight SS MMAs over K = 128 (steps of 16): both operands K-major
// 128-byte-swizzled tiles whose 64-column chunks are kA / kB descriptor
// units (bytes >> 4) apart; step kk starts kk / 4 chunks in, 32 bytes x
// (kk % 4) into the chunk.  The first MMA overwrites D.
template <uint32_t kA, uint32_t kB>
__device__ __forceinline__ void ss_x8_w(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b64 da, db;\n\t.reg .b32 al, bl;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "mov.b64 da, {%1, %4};\n\tmov.b64 db, {%2, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 0;\n\t"
      "add.u32 al, %1, 2;\n\tadd.u32 bl, %2, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, %1, 4;\n\tadd.u32 bl, %2, 4;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, %1, 6;\n\tadd.u32 bl, %2, 6;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, %1, %5;\n\tadd.u32 bl, %2, %6;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, al, 2;\n\tadd.u32 bl, bl, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, al, 2;\n\tadd.u32 bl, bl, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t"
      "add.u32 al, al, 2;\n\tadd.u32 bl, bl, 2;\n\t"
      "mov.b64 da, {al, %4};\n\tmov.b64 db, {bl, %4};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, 1;\n\t}" ::"r"(d),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "n"(ptx::kDescHiSw128), "n"(kA), "n"(kB)
      : "memory");
}

// TS MMAs over the 32-key chunks of A in tensor memory, two of K = 16 per
// chunk: the packed bf16 pairs of each chunk sit in the first 16 columns of
// that chunk (steps at a, a + 8, a + 32, a + 40, ...); B an MN-major
// 128-byte-swizzled tile, 16 rows (2048 bytes) per step.  The first MMA
// overwrites D unless `accumulate`.
template <int kChunks>
__device__ __forceinline__ void ts_chunked_w(uint32_t d, uint32_t a_tmem, uint32_t b_lo,
                                             uint32_t idesc, uint32_t accumulate) {
  static_assert(kChunks == 2 || kChunks == 4, "2 or 4 chunks");
  if constexpr (kChunks == 2) {
    asm volatile(
        "{\n\t.reg .pred e, p0;\n\t.reg .b64 db;\n\t.reg .b32 at, bl;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "mov.b64 db, {%2, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p0;\n\t"
        "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 32;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 40;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t}" ::"r"(d),
        "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(ptx::kDescHiSw128)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p0;\n\t.reg .b64 db;\n\t.reg .b32 at, bl;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\t"
        "mov.b64 db, {%2, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p0;\n\t"
        "add.u32 at, %1, 8;\n\tadd.u32 bl, %2, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 32;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 40;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 64;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 72;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 96;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t"
        "add.u32 at, %1, 104;\n\tadd.u32 bl, bl, 128;\n\tmov.b64 db, {bl, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [at], db, %3, 1;\n\t}" ::"r"(d),
        "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(ptx::kDescHiSw128)
        : "memory");
  }
}

// Score-like MMAs of one half: D[128 x 64] = A[128 x 128] B[64 x 128]^T,
// 8 SS MMAs (K = 128 in steps of 16); A a fixed 128-row tile, B a 64-row
// half-tile of the ring (64-column chunks 8 KB apart).
__device__ __forceinline__ void mma_scores_half(uint32_t d, uint32_t a_lo, uint32_t b_lo) {
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kT, kHalf, false);
  ss_x8_w<(kChunkBytes >> 4), (kHalfChunk >> 4)>(d, a_lo, b_lo, kIdesc);
}

// Gradient MMAs of one half: D[128 x 128] += A (128 x 64 bf16 in TMEM: the
// packed pairs of each 32-column chunk over the first 16 columns of that
// chunk, i.e. columns a..a+15 and a+32..a+47) B, B a 64-row half-tile of
// the ring read MN-major (K = 64 in steps of 16).
__device__ __forceinline__ void mma_grad_half(uint32_t d, uint32_t a_tmem, uint32_t b_mn,
                                              bool first) {
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kT, kD, true);
  ts_chunked_w<2>(d, a_tmem, b_mn, kIdesc, first ? 0u : 1u);
}

// TMEM columns of the two halves: scores of half h at [64h.. 64h+64) of
// the first 128, the second score-like product at +128; the bf16 results of
// each 32-column chunk overwrite the chunk's own first 16 columns (already
// read by the warp that owns the chunk).
__device__ __forceinline__ uint32_t col_s(int half) { return half * kHalf; }
__device__ __forceinline__ uint32_t col_p(int half) { return 128 + half * kHalf; }

// The MMA issuer's pipeline of the dK/dV kernel over `iters` query tiles
// (run by the whole MMA warp).  Scores of both halves of tile 0; then, as
// the elementwise warps finish each half, that half's gradient MMAs (which
// release its ring stage) followed by the next tile's scores of the same
// half, so the tensor pipe works on one half while the warps process the
// other.  `scores(it, h, stage)` / `grads(it, h, stage)` issue the MMAs.
template <typename Scores, typename Grads>
__device__ __forceinline__ bool mma_pipeline(uint32_t sb, int iters, Scores scores, Grads grads,
                                             const WaitCtl& ctl) {
  auto bar = [&](int i) -> uint32_t { return sb + kOffBar + 8 * i; };
  bool ok = wait_w(bar(BAR_FIX), 0, ctl);
  for (int h = 0; ok && h < 2; ++h) {
    if (!(ok = wait_w(bar(BAR_FULL0 + h), 0, ctl))) break;
    ptx::tc_fence_after();
    scores(0, h, h);
    ptx::commit_w(bar(BAR_SF0 + h));
  }
  for (int it = 0; ok && it < iters; ++it) {
    const bool next = it + 1 < iters;
    for (int h = 0; h < 2; ++h) {
      const int u = 2 * it + h;
      if (!(ok = wait_w(bar(BAR_EF0 + h), it & 1, ctl))) break;
      ptx::tc_fence_after();
      grads(it, h, u % kRing);
      ptx::commit_w(bar(BAR_EMPTY0 + u % kRing));  // this half's stage consumed
      if (next) {
        const int v = u + 2;
        if (!(ok = wait_w(bar(BAR_FULL0 + v % kRing), (v / kRing) & 1, ctl))) break;
        ptx::tc_fence_after();
        scores(it + 1, h, v % kRing);
        ptx::commit_w(bar(BAR_SF0 + h));
      }
    }
  }
  if (ok) ptx::commit_w(bar(BAR_ACC));
  return ok;
}

// --------------------------------------------------------------------- dQ
// The dQ kernel keeps one accumulator (dQ), so its 512 TMEM columns hold S,
// dQ and two full-width dP buffers: S at 0..127, dQ at 128..255, dP of even
// / odd key tiles at 256..383 / 384..511 (the packed dS of each 32-key chunk
// over the first 16 columns of that chunk of its tile's dP).  Score MMAs are
// full width (N = 128).
constexpr uint32_t kDqColS = 0;
constexpr uint32_t kDqColQ = 128;
__device__ __forceinline__ uint32_t dq_col_p(int t) {
  return 256 + static_cast<uint32_t>(t & 1) * 128;
}

// Shared memory of the dQ kernel: Q and dO (fixed), then separate K and V
// rings -- K(t) is read until dQ(t), late in the pipeline, V(t) only by
// dP(t), so K gets three stages and V two (224 KB of tiles in all).
constexpr int kDqKStages = 3;
constexpr int kDqVStages = 2;
constexpr int kDqOffK = 2 * kTileBytes;
constexpr int kDqOffV = kDqOffK + kDqKStages * kTileBytes;
constexpr int kDqOffBar = kDqOffV + kDqVStages * kTileBytes;
enum {
  DQ_FIX = 0,      // Q, dO landed
  DQ_FULLK0 = 1,   // K stage s landed (1..3)
  DQ_EMPTYK0 = 4,  // K stage s consumed (4..6)
  DQ_FULLV0 = 7,   // V stage s landed (7, 8)
  DQ_EMPTYV0 = 9,  // V stage s consumed (9, 10)
  DQ_SF = 11,      // S and dP of a tile computed
  DQ_EF = 12,      // dS of an even tile written, one arrival per elementwise warp
  DQ_ACC = 13,     // dQ final
  DQ_CLEAN = 14,
  DQ_SFREE = 15,   // every elementwise warp has read the tile's S
  DQ_EF1 = 16,     // dS of an odd tile written (see dq_ef)
  kDqNumBars = 17
};
constexpr int kDqOffTmemSlot = kDqOffBar + 8 * kDqNumBars;
constexpr int kDqOffAbort = kDqOffTmemSlot + 8;
constexpr int kDqSmemBytes = kDqOffAbort + 8 + 1024;
static_assert(kDqSmemBytes <= 227 * 1024, "dQ kernel shared memory");

// The "dS written" barrier of tile t, and the phase to wait for.  Tiles
// alternate between two barriers: S(t + 1) needs only every warp's read of
// S(t), so a fast warp may finish tile t + 1 before a slow one has written
// dS(t); with one barrier its arrival could complete tile t's phase.  Tile
// t + 2 needs every warp's read of S(t + 1), which follows its tile-t
// arrival, so each barrier's phase counts arrivals of one tile only.
__device__ __forceinline__ int dq_ef(int t) { return (t & 1) ? DQ_EF1 : DQ_EF; }
__device__ __forceinline__ uint32_t dq_ef_phase(int t) { return (static_cast<uint32_t>(t) >> 1) & 1; }

__device__ __forceinline__ uint32_t dq_setup(uint8_t* smem, uint32_t sb, int warp) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDqNumBars; ++i)
      ptx::mbar_init(sb + kDqOffBar + 8 * i,
                     (i == DQ_EF || i == DQ_EF1 || i == DQ_SFREE) ? kEwWarps : 1);
    *reinterpret_cast<volatile int*>(smem + kDqOffAbort) = 0;
    ptx::fence_mbar_init();
    ptx::fence_async_shared();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(smem + kDqOffTmemSlot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return *reinterpret_cast<uint32_t*>(smem + kDqOffTmemSlot);
}

// Producer of the dQ kernel: Q and dO once, then K(t) and V(t) of every key
// tile into their rings; `coord(t, &map_k, &map_v, &row)` names tile t.
template <bool kG, typename Coord>
__device__ __forceinline__ void dq_produce(uint32_t sb, const CUtensorMap* fq,
                                           const CUtensorMap* fdo, int fy, int frow, int iters,
                                           int c, Coord coord, const WaitCtl& ctl, int* status,
                                           const BwdParams& p) {
  auto bar = [&](int i) -> uint32_t { return sb + kDqOffBar + 8 * i; };
  ptx::mbar_arrive_expect_tx(bar(DQ_FIX), 2 * kTileBytes);
  for (int ch = 0; ch < 2; ++ch) {
    check_box<kG>(p, fq, ch * 64, fy, frow, kT);
    check_box<kG>(p, fdo, ch * 64, fy, frow, kT);
    ptx::tma_load_3d(sb + kOffFixA + ch * kChunkBytes, fq, bar(DQ_FIX), ch * 64, fy, frow);
    ptx::tma_load_3d(sb + kOffFixB + ch * kChunkBytes, fdo, bar(DQ_FIX), ch * 64, fy, frow);
  }
  int nk = 0, nv = 0;  // K / V tiles issued
  for (int t = 0; t < iters; ++t) {
    const CUtensorMap *mk, *mv;
    int row;
    coord(t, &mk, &mv, &row);
    const int sk = t % kDqKStages, sv = t % kDqVStages;
    if (t >= kDqKStages &&
        !wait_bar(bar(DQ_EMPTYK0 + sk), ((t / kDqKStages) - 1) & 1, ctl))
      break;
    ptx::mbar_arrive_expect_tx(bar(DQ_FULLK0 + sk), kTileBytes);
    for (int ch = 0; ch < 2; ++ch) {
      check_box<kG>(p, mk, ch * 64, c, row, kT);
      ptx::tma_load_3d(sb + kDqOffK + sk * kTileBytes + ch * kChunkBytes, mk,
                       bar(DQ_FULLK0 + sk), ch * 64, c, row);
    }
    nk = t + 1;
    if (t >= kDqVStages &&
        !wait_bar(bar(DQ_EMPTYV0 + sv), ((t / kDqVStages) - 1) & 1, ctl))
      break;
    ptx::mbar_arrive_expect_tx(bar(DQ_FULLV0 + sv), kTileBytes);
    for (int ch = 0; ch < 2; ++ch) {
      check_box<kG>(p, mv, ch * 64, c, row, kT);
      ptx::tma_load_3d(sb + kDqOffV + sv * kTileBytes + ch * kChunkBytes, mv,
                       bar(DQ_FULLV0 + sv), ch * 64, c, row);
    }
    nv = t + 1;
  }
  // Drain: every copy issued must have landed before the CTA exits.
  drain_bar(bar(DQ_FIX), 0, status);
  for (int st = 0; st < kDqKStages; ++st) {
    const int last = nk - 1 - ((nk - 1 - st) % kDqKStages + kDqKStages) % kDqKStages;
    if (last >= 0) drain_bar(bar(DQ_FULLK0 + st), (last / kDqKStages) & 1, status);
  }
  for (int st = 0; st < kDqVStages; ++st) {
    const int last = nv - 1 - ((nv - 1 - st) % kDqVStages + kDqVStages) % kDqVStages;
    if (last >= 0) drain_bar(bar(DQ_FULLV0 + st), (last / kDqVStages) & 1, status);
  }
}

// D[128 x 128] = A[128 x 128] B[128 x 128]^T, both K-major: 8 SS MMAs.
__device__ __forceinline__ void mma_scores_full(uint32_t d, uint32_t a_lo, uint32_t b_lo) {
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kT, kT, false);
  ss_x8_w<(kChunkBytes >> 4), (kChunkBytes >> 4)>(d, a_lo, b_lo, kIdesc);
}

// MMA issue order of the dQ kernel (run by the whole MMA warp), tile t's
// elementwise pass running: dP(t+1) into the other dP buffer (its dS(t-1)
// was read by dQ(t-1), issued earlier); S(t+1) as soon as every warp has
// read S(t), at the start of the pass; dQ += dS(t) K(t) once dS(t) is
// written.  Both score products of the next tile are done while the warps
// process this one.
__device__ __forceinline__ bool dq_pipeline(uint32_t sb, uint32_t tmem, int iters,
                                            const WaitCtl& ctl) {
  auto bar = [&](int i) -> uint32_t { return sb + kDqOffBar + 8 * i; };
  constexpr uint32_t kIdescG = ptx::idesc_bf16_f32(kT, kD, true);
  const uint32_t q_lo = ptx::desc_lo(sb + kOffFixA, 16);
  const uint32_t do_lo = ptx::desc_lo(sb + kOffFixB, 16);
  const uint32_t k_lo = ptx::desc_lo(sb + kDqOffK, 16);
  const uint32_t v_lo = ptx::desc_lo(sb + kDqOffV, 16);
  const uint32_t k_mn = ptx::desc_lo(sb + kDqOffK, kChunkBytes);
  bool ok = wait_w(bar(DQ_FIX), 0, ctl) && wait_w(bar(DQ_FULLK0), 0, ctl) &&
            wait_w(bar(DQ_FULLV0), 0, ctl);
  if (!ok) return false;
  ptx::tc_fence_after();
  mma_scores_full(tmem + dq_col_p(0), do_lo, v_lo);  // dP = dO V^T
  ptx::commit_w(bar(DQ_EMPTYV0));
  mma_scores_full(tmem + kDqColS, q_lo, k_lo);       // S  = Q K^T
  ptx::commit_w(bar(DQ_SF));
  for (int t = 0; t < iters; ++t) {
    const bool next = t + 1 < iters;
    if (next) {
      const int sv = (t + 1) % kDqVStages;
      if (!(ok = wait_w(bar(DQ_FULLV0 + sv), ((t + 1) / kDqVStages) & 1, ctl))) break;
      ptx::tc_fence_after();
      mma_scores_full(tmem + dq_col_p(t + 1), do_lo, v_lo + sv * kTileLo);
      ptx::commit_w(bar(DQ_EMPTYV0 + sv));  // V(t+1) consumed
      const int sk = (t + 1) % kDqKStages;
      if (!(ok = wait_w(bar(DQ_FULLK0 + sk), ((t + 1) / kDqKStages) & 1, ctl))) break;
      if (!(ok = wait_w(bar(DQ_SFREE), t & 1, ctl))) break;
      ptx::tc_fence_after();
      mma_scores_full(tmem + kDqColS, q_lo, k_lo + sk * kTileLo);
      ptx::commit_w(bar(DQ_SF));
    }
    if (!(ok = wait_w(bar(dq_ef(t)), dq_ef_phase(t), ctl))) break;
    ptx::tc_fence_after();
    const int sk = t % kDqKStages;
    const uint32_t a = tmem + dq_col_p(t);
    const uint32_t kb = k_mn + sk * kTileLo;
    ts_chunked_w<4>(tmem + kDqColQ, a, kb, kIdescG, t > 0 ? 1u : 0u);
    ptx::commit_w(bar(DQ_EMPTYK0 + sk));  // K(t) consumed
  }
  if (ok) ptx::commit_w(bar(DQ_ACC));
  return ok;
}

// CTA = (query tile, query head).
template <bool kG>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_tc_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + kDqOffBar + 8 * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Window mode: CTA (query tile, head); key tiles = landmark tiles, then the
  // window tiles of the rows.  Gathered mode: CTA (key split, M tile, KV
  // head); key tiles = the split's.
  const int split = kG ? blockIdx.x : 0;
  const int64_t qr0 = static_cast<int64_t>(kG ? blockIdx.y : blockIdx.x) * kT;
  const int h = kG ? 0 : blockIdx.y;
  const int c = kG ? blockIdx.z : h / p.group;
  const int fy = kG ? c : h;  // head coordinate of the fixed Q / dO tiles
  int n_lm_tiles, kt_lo, T;
  if constexpr (kG) {
    const int64_t key_lo = static_cast<int64_t>(split) * p.span;
    const int64_t key_hi = min64(key_lo + p.span, p.n);
    n_lm_tiles = 0;
    kt_lo = static_cast<int>(key_lo / kT);
    T = static_cast<int>((key_hi - key_lo + kT - 1) / kT);
  } else {
    const int64_t q_last = min64(qr0 + kT, p.n) - 1;
    const int64_t n_lm = visible_landmarks(q_last, p.window, p.block, p.G);
    n_lm_tiles = static_cast<int>((n_lm + kT - 1) / kT);
    const int64_t j_lo = max64(qr0 - p.window + 1, 0);
    kt_lo = static_cast<int>(j_lo / kT);
    T = n_lm_tiles + static_cast<int>(q_last / kT) - kt_lo + 1;
  }

  const uint32_t tmem = dq_setup(smem, sb, warp);
  WaitCtl ctl{reinterpret_cast<volatile int*>(smem + kDqOffAbort), p.status, p.wait_ns};

  if (warp == kProdWarp) {
    if (lane == 0) {
      auto coord = [&](int t, const CUtensorMap** mk, const CUtensorMap** mv, int* row) {
        const bool lm = t < n_lm_tiles;
        *mk = lm ? &p.tm_klm : &p.tm_k;
        *mv = lm ? &p.tm_vlm : &p.tm_v;
        *row = lm ? t * kT : (kt_lo + t - n_lm_tiles) * kT;
      };
      dq_produce<kG>(sb, &p.tm_q, &p.tm_do, fy, static_cast<int>(qr0), T, c, coord, ctl,
                     p.status, p);
    }
  } else if (warp == kMmaWarp) {
    dq_pipeline(sb, tmem, T, ctl);
    ptx::commit_w(bar(DQ_CLEAN));
    drain_bar(bar(DQ_CLEAN), 0, p.status);
  } else if (warp < kEwWarps) {
    const int quarter = warp & 3;  // TMEM lanes (rows) 32 quarter ..
    const int cp = warp >> 2;      // key columns [64 cp, 64 cp + 64) of each tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int64_t i_row = qr0 + quarter * 32 + lane;  // query row, or gathered M row
    // Position of the row (its own index outside the gathered mode).
    const int64_t i =
        kG ? (MSA_IN_RANGE(i_row, 1, p.Mp, p.status) ? p.gpos[i_row] : -1) : i_row;
    const int64_t st = kG ? static_cast<int64_t>(c) * p.Mp + i_row
                               : static_cast<int64_t>(h) * p.n_pad + i_row;
    const bool st_ok = MSA_IN_RANGE(
        st, 1, kG ? static_cast<int64_t>(p.Hkv) * p.Mp : static_cast<int64_t>(p.Hq) * p.n_pad,
        p.status);
    const bool row_ok = (kG ? i >= 0 : i < p.n) && st_ok;
    const float nL2 = st_ok ? p.L2[st] : -INFINITY;
    const float nD = st_ok ? p.D[st] : 0.f;
    const uint64_t c2 = ptx::f2(p.scale_log2, p.scale_log2);
    const uint64_t nL22 = ptx::f2(nL2, nL2);
    const uint64_t nD2 = ptx::f2(nD, nD);
    const int64_t my_lm = visible_landmarks(i, p.window, p.block, p.G);
    const int64_t my_lo = max64(i - p.window + 1, 0);
    bool ok = true;
    for (int t = 0; ok && t < T; ++t) {
      int64_t lo, hi;  // valid columns [lo, hi) of this key tile for row i
      if (t < n_lm_tiles) {
        lo = 0;
        hi = my_lm - static_cast<int64_t>(t) * kT;
      } else {
        const int64_t kb = static_cast<int64_t>(kt_lo + t - n_lm_tiles) * kT;
        lo = kG ? 0 : my_lo - kb;  // a global row sees every key j <= i
        hi = i - kb + 1;
      }
      if (!row_ok) hi = lo;
      ok = __all_sync(0xffffffffu, wait_bar(bar(DQ_SF), t & 1, ctl));
      if (!ok) break;
      ptx::tc_fence_after();
      const int lo_c = static_cast<int>(max64(0, min64(kT, lo)));
      const int hi_c = static_cast<int>(max64(0, min64(kT, hi)));
      const uint32_t tp = tl + dq_col_p(t);
      // This warp's two 32-column chunks of S and dP, all read before S is
      // released for the next tile's S MMAs.
      float s[2][32], dp[2][32];
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        ptx::tmem_ld32(tl + kDqColS + (2 * cp + ci) * 32, s[ci]);
        ptx::tmem_ld32(tp + (2 * cp + ci) * 32, dp[ci]);
      }
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(DQ_SFREE));
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
              ptx::mul2(pr, ptx::add2(ptx::f2(dp[ci][2 * e], dp[ci][2 * e + 1]), nD2)), d0, d1);
          pk[e] = ptx::pack_bf16x2(d0, d1);
        }
        ptx::tmem_st16(tp + cc * 32, pk);  // dS over dP columns this warp has read
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(dq_ef(t)));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(DQ_ACC), 0, ctl));
    if (ok) {
      ptx::tc_fence_after();
      // Gathered mode: this split's share of the row's dQ, fp32.
      void* dst = kG ? static_cast<void*>(p.dq_part) : p.dq;
      const int64_t off =
          kG ? ((static_cast<int64_t>(split) * p.Hkv + c) * p.Mp + i_row) * kD
                  : (i_row * p.Hq + h) * static_cast<int64_t>(kD);
      const bool out_ok =
          !row_ok ||
          MSA_IN_RANGE(off, kD,
                       kG ? static_cast<int64_t>(gridDim.x) * p.Hkv * p.Mp * kD
                          : p.n * p.Hq * static_cast<int64_t>(kD),
                       p.status);
#pragma unroll 1
      for (int ci = 0; ci < 2; ++ci) {  // this warp's 64 of the 128 columns
        const int cc = 2 * cp + ci;
        float o[32];
        ptx::tmem_ld32(tl + kDqColQ + cc * 32, o);
        ptx::tmem_wait_ld();
        if (row_ok && out_ok) store_row(dst, off + cc * 32, o, p.scale, kG ? 0 : p.grad_bf16);
      }
    }
  }
  bwd_teardown(tmem, warp);
}

// ------------------------------------------------------------------ dK, dV
// CTA = (key tile or landmark tile, KV head[, query chunk]).  TMEM: S^T of
// query halves 0/1 at 0..63 / 64..127 (P^T over their first 32 columns),
// dP^T at 128..255 (dS^T likewise), dV 256..383, dK 384..511.
template <bool kG>
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
  if constexpr (kG) {  // every M tile of the gathered global rows
    qt_lo = 0;
    qt_hi = p.Mp / kT - 1;
  } else if (p.lm_mode) {
    const int64_t first_row = (kb + 1) * p.block + p.window - 1;  // sees landmark kb
    const int64_t base = first_row / kT;
    qt_lo = base + static_cast<int64_t>(chunk) * p.chunk_tiles;
    qt_hi = min64(base + static_cast<int64_t>(chunk + 1) * p.chunk_tiles, n_qt) - 1;
  } else {
    qt_lo = kb / kT;
    qt_hi = min64(p.n - 1, kb + kT - 1 + p.window - 1) / kT;
  }
  const int hpi = kG ? 1 : p.group;  // heads per query tile (M rows hold them in gmode)
  const int iters = qt_hi >= qt_lo ? static_cast<int>((qt_hi - qt_lo + 1) * hpi) : 0;
  if (iters == 0) {  // landmark chunk beyond the last row: a zero partial
    if (p.lm_mode && threadIdx.x < kT && kb + threadIdx.x < p.G) {
      for (int which = 0; which < 2; ++which) {
        const int64_t o = (((static_cast<int64_t>(chunk) * 2 + which) * p.G + kb + threadIdx.x) *
                               p.Hkv + c) * kD;
        if (!MSA_IN_RANGE(o, kD, static_cast<int64_t>(gridDim.z) * 2 * p.G * p.Hkv * kD,
                          p.status))
          continue;
        float* dst = p.lm_part + o;
        for (int e = 0; e < kD; ++e) dst[e] = 0.f;
      }
    }
    return;
  }

  const uint32_t tmem = bwd_setup(smem, sb, warp);
  WaitCtl ctl{reinterpret_cast<volatile int*>(smem + kOffAbort), p.status, p.wait_ns};

  if (warp == kProdWarp) {
    if (lane == 0) {
      auto coord = [&](int it, const CUtensorMap** ma, const CUtensorMap** mb, int* ya, int* yb,
                       int* row) {
        *ma = &p.tm_q64;
        *mb = &p.tm_do64;
        *ya = *yb = kG ? c : c * p.group + it % p.group;
        *row = static_cast<int>((qt_lo + it / hpi) * kT);
      };
      auto stats = [&](int it, const float** sl, const float** sd, const int** sp) {
        const int64_t row = (qt_lo + it / hpi) * kT;
        const int64_t off = kG ? static_cast<int64_t>(c) * p.Mp + row
                                    : static_cast<int64_t>(c * p.group + it % p.group) * p.n_pad +
                                          row;
        *sl = p.L2 + off;
        *sd = p.D + off;
        if (kG) *sp = p.gpos + row;
      };
      produce<kG>(sb, p.lm_mode ? &p.tm_klm : &p.tm_k, p.lm_mode ? &p.tm_vlm : &p.tm_v, c,
                  static_cast<int>(kb), iters, coord, stats, ctl, p.status, p);
    }
  } else if (warp == kMmaWarp) {  // the whole warp issues (elect.sync inside)
    {
      const uint32_t k_lo = ptx::desc_lo(sb + kOffFixA, 16);
      const uint32_t v_lo = ptx::desc_lo(sb + kOffFixB, 16);
      constexpr uint32_t kStageLo = kRingStageBytes >> 4;
      constexpr uint32_t kDoLo = kHalfTileBytes >> 4;
      const uint32_t r_lo = ptx::desc_lo(sb + kOffRing, 16);            // K-major view
      const uint32_t r_mn = ptx::desc_lo(sb + kOffRing, kHalfChunk);    // MN-major view
      auto scores = [&](int it, int half, int st) {
        (void)it;
        const uint32_t q = r_lo + st * kStageLo;
        mma_scores_half(tmem + col_s(half), k_lo, q);          // S^T  = K Q^T
        mma_scores_half(tmem + col_p(half), v_lo, q + kDoLo);  // dP^T = V dO^T
      };
      auto grads = [&](int it, int half, int st) {
        const uint32_t q = r_mn + st * kStageLo;
        const bool first = it == 0 && half == 0;
        mma_grad_half(tmem + 256, tmem + col_s(half), q + kDoLo, first);  // dV += P^T dO
        mma_grad_half(tmem + 384, tmem + col_p(half), q, first);          // dK += dS^T Q
      };
      mma_pipeline(sb, iters, scores, grads, ctl);
      ptx::commit_w(bar(BAR_CLEAN));
      drain_bar(bar(BAR_CLEAN), 0, p.status);
    }
  } else if (warp < kEwWarps) {
    const int quarter = warp & 3;  // TMEM lanes (rows) 32 quarter ..
    const int cp = warp >> 2;      // query columns [32 cp, 32 cp + 32) of each half
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    // Key (window mode) or landmark (landmark mode) of this row.
    const int64_t j = kb + quarter * 32 + lane;
    const uint64_t c2 = ptx::f2(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int it = 0; ok && it < iters; ++it) {
      const int64_t qr0 = (qt_lo + it / hpi) * kT;
      // Each half's per-query -lse (log2 units) and -D came with its Q / dO
      // stage; the stage has landed once its scores exist, and it is not
      // refilled before this half's results are in.
      // Rows i of this query tile that see key/landmark j: [lo, hi) columns.
      int64_t lo, hi;
      if constexpr (kG) {  // per column below (each M row has its own position)
        lo = 0;
        hi = kT;
      } else if (p.lm_mode) {
        lo = j < p.G ? (j + 1) * p.block + p.window - 1 - qr0 : kT;
        hi = kT;
      } else {
        lo = j - qr0;
        hi = j + p.window - qr0;
      }
      for (int half = 0; half < 2; ++half) {
        const int u = 2 * it + half;
        ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_SF0 + half), it & 1, ctl));
        if (ok)  // completed already; makes the copied rows visible here
          ok = __all_sync(0xffffffffu,
                          wait_bar(bar(BAR_FULL0 + u % kRing), (u / kRing) & 1, ctl));
        if (!ok) break;
        const float* sL =
            reinterpret_cast<const float*>(smem + kOffStats + (u % kRing) * kStatBytes);
        const float* sD = sL + kHalfRows;
        const int* sP = reinterpret_cast<const int*>(sD + kHalfRows);  // gathered mode
        ptx::tc_fence_after();
        const int lo_c = static_cast<int>(max64(0, min64(kHalf, lo - half * kHalf)));
        const int hi_c = static_cast<int>(max64(0, min64(kHalf, hi - half * kHalf)));
        const float4* hL = reinterpret_cast<const float4*>(sL);
        const float4* hD = reinterpret_cast<const float4*>(sD);
        const bool full = lo_c == 0 && hi_c == kHalf;
        {
          const int cc = cp;  // this warp's 32-column chunk of the half
          float s[32], dp[32];
          ptx::tmem_ld32(tl + col_s(half) + cc * 32, s);
          ptx::tmem_ld32(tl + col_p(half) + cc * 32, dp);
          ptx::tmem_wait_ld();
          if (!full) {  // masked columns: weight 0
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int col = cc * 32 + e;
              s[e] = (col >= lo_c && col < hi_c) ? s[e] : -INFINITY;
            }
          }
          if constexpr (kG) {  // global row m sees key j iff j <= its position
            const int* hp = sP + cc * 32;
#pragma unroll
            for (int e = 0; e < 32; ++e) s[e] = j <= hp[e] ? s[e] : -INFINITY;
          }
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const float4 l4 = hL[cc * 8 + q4];  // -lse log2e of 4 queries (broadcast)
            const float4 d4 = hD[cc * 8 + q4];  // -D of the same queries
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int e = 2 * q4 + u;
              const uint64_t nl = u ? ptx::f2(l4.z, l4.w) : ptx::f2(l4.x, l4.y);
              const uint64_t nd = u ? ptx::f2(d4.z, d4.w) : ptx::f2(d4.x, d4.y);
              float x0, x1;
              ptx::f2_split(ptx::fma2(ptx::f2(s[2 * e], s[2 * e + 1]), c2, nl), x0, x1);
              const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
              float d0, d1;
              ptx::f2_split(
                  ptx::mul2(ptx::f2(p0, p1), ptx::add2(ptx::f2(dp[2 * e], dp[2 * e + 1]), nd)),
                  d0, d1);
              pp[e] = ptx::pack_bf16x2(p0, p1);
              dd[e] = ptx::pack_bf16x2(d0, d1);
            }
          }
          ptx::tmem_st16(tl + col_s(half) + cc * 32, pp);  // P^T over columns read above
          ptx::tmem_st16(tl + col_p(half) + cc * 32, dd);  // dS^T likewise
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(BAR_EF0 + half));
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(BAR_ACC), 0, ctl));
    if (ok) {
      ptx::tc_fence_after();
      if constexpr (kG) {  // the global rows' share of dK (scaled) and dV, fp32
        const int64_t off = (j * p.Hkv + c) * static_cast<int64_t>(kD);
        const bool row_ok =
            j < p.n && MSA_IN_RANGE(off, kD, p.n * p.Hkv * static_cast<int64_t>(kD), p.status);
        const int which = cp;  // 0: dK (warps 0-3), 1: dV (warps 4-7)
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          float o[32];
          ptx::tmem_ld32(tl + (which == 0 ? 384 : 256) + cc * 32, o);
          ptx::tmem_wait_ld();
          if (row_ok)
            store_row(which == 0 ? p.extra_k : p.extra_v, off + cc * 32, o,
                      which == 0 ? p.scale : 1.f, 0);
        }
      } else if (p.lm_mode) {
        const int which = cp;  // 0: dK_lm (warps 0-3), 1: dV_lm (warps 4-7)
        const int64_t o =
            (((static_cast<int64_t>(chunk) * 2 + which) * p.G + j) * p.Hkv + c) * kD;
        const bool row_ok =
            j < p.G && MSA_IN_RANGE(o, kD, static_cast<int64_t>(gridDim.z) * 2 * p.G * p.Hkv * kD,
                                    p.status);
        float* dst = p.lm_part + o;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          float o[32];
          ptx::tmem_ld32(tl + (which == 0 ? 384 : 256) + cc * 32, o);
          ptx::tmem_wait_ld();
          if (row_ok) store_row(dst, cc * 32, o, which == 0 ? p.scale : 1.f, 0);
        }
      } else {
        const int64_t off = (j * p.Hkv + c) * static_cast<int64_t>(kD);
        const bool row_ok =
            j < p.n && MSA_IN_RANGE(off, kD, p.n * p.Hkv * static_cast<int64_t>(kD), p.status);
        // The token's share of its landmark's gradient.
        const float* lmk = nullptr;
        const float* lmv = nullptr;
        if (p.G > 0 && row_ok &&
            MSA_IN_RANGE((j / p.block * p.Hkv + c) * kD, kD,
                         static_cast<int64_t>(p.G) * p.Hkv * kD, p.status)) {
          const int64_t l = j / p.block;
          lmk = p.lm_grad + (l * p.Hkv + c) * kD;
          lmv = p.lm_grad + ((static_cast<int64_t>(p.G) + l) * p.Hkv + c) * kD;
        }
        const float invB = 1.f / static_cast<float>(p.block);
        {
          const int which = cp;  // 0: dK (warps 0-3), 1: dV (warps 4-7)
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
            const float* ex = which == 0 ? p.extra_k : p.extra_v;
            if (ex && row_ok) {  // the global rows' share (already scaled)
              const float* exr = ex + off + cc * 32;
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] += exr[e] / w;
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
// Row statistics, stored negated for the packed FMAs that use them:
// nL2[h, i] = -lse[h, i] log2(e) and nD[h, i] = -<dO[i, h], O[i, h]> for
// i < n, -inf and 0 for the padding up to n_pad.  Eight lanes per (row,
// head), 16 elements a lane from 16-byte loads, four pairs a warp.
template <bool kOutBf16>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const void* out, const uint16_t* dout, const float* lse, float* L2,
                          float* D, int64_t n, int64_t n_pad, int Hq, int* status) {
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * 32 + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;  // lane within the pair's 8
  if (pair >= n_pad * Hq) return;  // whole 8-lane groups leave together
  const int64_t i = pair / Hq;
  const int h = static_cast<int>(pair % Hq);
  float acc = 0.f;
  // Rows past n read nothing; a row of O / dO [n][Hq][d] and of lse [Hq][n].
  const bool in_ok = i >= n || (MSA_IN_RANGE(pair * kD, kD, n * Hq * static_cast<int64_t>(kD),
                                             status) &&
                                MSA_IN_RANGE(static_cast<int64_t>(h) * n + i, 1,
                                             static_cast<int64_t>(Hq) * n, status));
  if (i < n && in_ok) {
    const int64_t base = pair * kD + sub * 16;
    const uint4* g4 = reinterpret_cast<const uint4*>(dout + base);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint4 gv = __ldg(g4 + half);
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
      float o[8];
      if constexpr (kOutBf16) {
        const uint4 ov = __ldg(reinterpret_cast<const uint4*>(
                                   static_cast<const uint16_t*>(out) + base) + half);
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          o[2 * k] = __uint_as_float(ow[k] << 16);
          o[2 * k + 1] = __uint_as_float(ow[k] & 0xffff0000u);
        }
      } else {
        const float4* o4 = reinterpret_cast<const float4*>(static_cast<const float*>(out) + base);
        const float4 a = __ldg(o4 + 2 * half), b = __ldg(o4 + 2 * half + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc = fmaf(o[2 * k], __uint_as_float(gw[k] << 16), acc);
        acc = fmaf(o[2 * k + 1], __uint_as_float(gw[k] & 0xffff0000u), acc);
      }
    }
    // The 8 lanes of this pair take the same branches: reduce among them.
    const unsigned gmask = 0xffu << (threadIdx.x & 24);
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(gmask, acc, off);
  }
  if (sub == 0 && in_ok) {
    const int64_t at = static_cast<int64_t>(h) * n_pad + i;
    if (!MSA_IN_RANGE(at, 1, static_cast<int64_t>(Hq) * n_pad, status)) return;
    D[at] = -acc;
    L2[at] = i < n ? -lse[static_cast<int64_t>(h) * n + i] * kLog2e : -INFINITY;
  }
}

// lm_grad[e] = sum over chunks of lm_part[chunk][e] (fixed order).
__global__ void __launch_bounds__(256)
    lm_grad_reduce_kernel(const float* part, float* grad, int64_t per_chunk, int chunks,
                          int* status) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= per_chunk) return;
  if (!MSA_IN_RANGE(static_cast<int64_t>(chunks - 1) * per_chunk + e, 1, chunks * per_chunk,
                    status))
    return;
  float s = 0.f;
  for (int ch = 0; ch < chunks; ++ch) s += part[ch * per_chunk + e];
  grad[e] = s;
}

// True when global row r repeats an earlier row's position (its output is
// that row's; only the first occurrence carries a gradient).
__device__ __forceinline__ bool repeated_row(const int64_t* rows, int64_t r, int64_t pos) {
  for (int64_t q = 0; q < r; ++q)
    if (rows[q] == pos) return true;
  return false;
}

// The window pass gives the global rows no weight: L2 = -inf, D = 0.
__global__ void __launch_bounds__(256)
    suppress_rows_kernel(const int64_t* rows, int64_t n_global, float* L2, float* D, int64_t n,
                         int64_t n_pad, int Hq, int* status) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n_global * Hq) return;
  const int64_t pos = rows[idx / Hq];
  const int h = static_cast<int>(idx % Hq);
  if (pos < 0 || pos >= n) return;
  if (!MSA_IN_RANGE(static_cast<int64_t>(h) * n_pad + pos, 1, static_cast<int64_t>(Hq) * n_pad,
                    status))
    return;
  L2[static_cast<int64_t>(h) * n_pad + pos] = -INFINITY;
  D[static_cast<int64_t>(h) * n_pad + pos] = 0.f;
}

// One warp per (M row m, KV head c): Qg / dOg rows gathered from Q / dO at
// the row's position (lanes 0-15 and 16-31, 16 bytes each), and its
// statistics -lse log2(e) and -<dO, O>; padding, repeated and invalid
// rows (the latter reported) get position -1 and no weight.
template <bool kOutBf16>
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint16_t* q, const uint16_t* dout, const void* out,
                       const float* lse, const int64_t* rows, int64_t Mc, int64_t Mp, int64_t n,
                       int Hq, int Hkv, int group, uint16_t* Qg, uint16_t* dOg, float* gL2,
                       float* gD, int* gpos, int* status) {
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= Mp * Hkv) return;
  const int64_t m = pair / Hkv;
  const int c = static_cast<int>(pair % Hkv);
  int64_t pos = -1;
  if (m < Mc) {
    const int64_t r = m / group;
    pos = rows[r];
    if (pos < 0 || pos >= n) {
      if (lane == 0) record_status(status, MSA_ERR_INVALID_ARG);
      pos = -1;
    } else if (repeated_row(rows, r, pos)) {
      pos = -1;
    }
  }
  const int h = c * group + static_cast<int>(m % group);
  const int64_t dst = (m * Hkv + c) * kD;
  if (!MSA_IN_RANGE(dst, kD, Mp * Hkv * kD, status)) return;  // whole warps leave together
  if (pos >= 0 && !(MSA_IN_RANGE((pos * Hq + h) * kD, kD, n * Hq * kD, status) &&
                    MSA_IN_RANGE(static_cast<int64_t>(h) * n + pos, 1, Hq * n, status)))
    pos = -1;
  const int half = lane >> 4;
  uint4* gdst = reinterpret_cast<uint4*>((half ? dOg : Qg) + dst) + (lane & 15);
  float acc = 0.f;
  if (pos >= 0) {
    const int64_t src = (pos * Hq + h) * kD;
    *gdst = __ldg(reinterpret_cast<const uint4*>((half ? dout : q) + src) + (lane & 15));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t at = src + lane * 4 + e;
      const float o = kOutBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(out)[at])
                               : static_cast<const float*>(out)[at];
      acc = fmaf(o, bf16_bits_to_float(dout[at]), acc);
    }
  } else {
    *gdst = make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    gL2[static_cast<int64_t>(c) * Mp + m] =
        pos >= 0 ? -lse[static_cast<int64_t>(h) * n + pos] * kLog2e : -INFINITY;
    gD[static_cast<int64_t>(c) * Mp + m] = -acc;
    if (c == 0) gpos[m] = static_cast<int>(pos);
  }
}

// One warp per (global row, query head): its dQ = the sum of the key
// splits' shares up to its position, written to row pos of dq.
__global__ void __launch_bounds__(256)
    dq_scatter_kernel(const float* dq_part, const int64_t* rows, int64_t n_global, int64_t Mp,
                      int n_splits, int64_t span, int64_t n, int Hq, int Hkv, int group, void* dq,
                      int grad_bf16, int* status) {
  const int64_t pair = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (pair >= n_global * Hq) return;
  const int64_t r = pair / Hq;
  const int h = static_cast<int>(pair % Hq);
  const int64_t pos = rows[r];
  if (pos < 0 || pos >= n || repeated_row(rows, r, pos)) return;
  const int c = h / group;
  const int64_t m = r * group + h % group;
  if (!MSA_IN_RANGE(((static_cast<int64_t>(n_splits - 1) * Hkv + c) * Mp + m) * kD, kD,
                    static_cast<int64_t>(n_splits) * Hkv * Mp * kD, status) ||
      !MSA_IN_RANGE((pos * Hq + h) * kD, kD, n * Hq * kD, status))
    return;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int sp = 0; sp < n_splits && static_cast<int64_t>(sp) * span <= pos; ++sp) {
    const float4 x = *reinterpret_cast<const float4*>(
        dq_part + ((static_cast<int64_t>(sp) * Hkv + c) * Mp + m) * kD + lane * 4);
    acc[0] += x.x;
    acc[1] += x.y;
    acc[2] += x.z;
    acc[3] += x.w;
  }
  const int64_t off = (pos * Hq + h) * kD + lane * 4;
  if (grad_bf16) {
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(dq) + off;
    for (int e = 0; e < 4; ++e) d[e] = __float2bfloat16_rn(acc[e]);
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(dq) + off) =
        make_float4(acc[0], acc[1], acc[2], acc[3]);
  }
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
  if (!encode_map(fn, &p.tm_q64, a.q, a.n, a.Hq, kHalfRows) ||
      !encode_map(fn, &p.tm_do64, a.dout, a.n, a.Hq, kHalfRows)) {
    *why = "cuTensorMapEncodeTiled rejected q or dout (64-row boxes)";
    return cudaErrorInvalidValue;
  }
  if (a.G == 0) {
    p.tm_klm = p.tm_k;
    p.tm_vlm = p.tm_v;
  }
  p.L2 = a.stats;
  p.D = a.stats + static_cast<int64_t>(a.Hq) * a.n_pad;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.lm_part = a.lm_part;
  p.lm_grad = a.lm_grad;
  p.n = a.n;
  p.n_pad = a.n_pad;
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

  const int64_t pairs = a.n_pad * a.Hq;
  const unsigned pre_blocks = static_cast<unsigned>((pairs + 31) / 32);
  float* L2w = a.stats;
  float* Dw = a.stats + static_cast<int64_t>(a.Hq) * a.n_pad;
  if (a.out_bf16)
    bwd_preprocess_kernel<true><<<pre_blocks, 256, 0, s>>>(
        a.out, static_cast<const uint16_t*>(a.dout), a.lse, L2w, Dw, a.n, a.n_pad, a.Hq,
        a.status);
  else
    bwd_preprocess_kernel<false><<<pre_blocks, 256, 0, s>>>(
        a.out, static_cast<const uint16_t*>(a.dout), a.lse, L2w, Dw, a.n, a.n_pad, a.Hq,
        a.status);
  cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  for (auto* k : {bwd_dkdv_tc_kernel<false>, bwd_dkdv_tc_kernel<true>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  for (auto* k : {bwd_dq_tc_kernel<false>, bwd_dq_tc_kernel<true>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmemBytes);
    if (e != cudaSuccess) return e;
  }
  const unsigned n_tiles = static_cast<unsigned>((a.n + kT - 1) / kT);
  const int group = a.Hq / a.Hkv;
  BwdParams pg;  // the gathered global-row launches
  if (a.rows) {
    suppress_rows_kernel<<<static_cast<unsigned>((a.n_global * a.Hq + 255) / 256), 256, 0, s>>>(
        a.rows, a.n_global, L2w, Dw, a.n, a.n_pad, a.Hq, a.status);
    const unsigned gblocks = static_cast<unsigned>((a.Mp * a.Hkv + 7) / 8);
    if (a.out_bf16)
      gather_rows_kernel<true><<<gblocks, 256, 0, s>>>(
          static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.dout), a.out, a.lse,
          a.rows, a.Mc, a.Mp, a.n, a.Hq, a.Hkv, group, static_cast<uint16_t*>(a.Qg),
          static_cast<uint16_t*>(a.dOg), a.gL2, a.gD, a.gpos, a.status);
    else
      gather_rows_kernel<false><<<gblocks, 256, 0, s>>>(
          static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.dout), a.out, a.lse,
          a.rows, a.Mc, a.Mp, a.n, a.Hq, a.Hkv, group, static_cast<uint16_t*>(a.Qg),
          static_cast<uint16_t*>(a.dOg), a.gL2, a.gD, a.gpos, a.status);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    pg = p;
    if (!encode_map(fn, &pg.tm_q, a.Qg, a.Mp, a.Hkv) ||
        !encode_map(fn, &pg.tm_do, a.dOg, a.Mp, a.Hkv) ||
        !encode_map(fn, &pg.tm_q64, a.Qg, a.Mp, a.Hkv, kHalfRows) ||
        !encode_map(fn, &pg.tm_do64, a.dOg, a.Mp, a.Hkv, kHalfRows)) {
      *why = "cuTensorMapEncodeTiled rejected the gathered rows";
      return cudaErrorInvalidValue;
    }
    pg.L2 = a.gL2;
    pg.D = a.gD;
    pg.gpos = a.gpos;
    pg.Mp = a.Mp;
    pg.span = a.span;
    pg.dq_part = a.dq_part;
    pg.extra_k = a.extra_k;
    pg.extra_v = a.extra_v;
    // The global rows' dK / dV first: the window pass adds them in.
    bwd_dkdv_tc_kernel<true><<<dim3(n_tiles, a.Hkv, 1), kThreads, kSmemBytes, s>>>(pg);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.G > 0) {
    p.lm_mode = 1;
    dim3 grid(static_cast<unsigned>((a.G + kT - 1) / kT), a.Hkv, a.lm_chunks);
    bwd_dkdv_tc_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(p);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    const int64_t per_chunk = 2 * static_cast<int64_t>(a.G) * a.Hkv * kD;
    lm_grad_reduce_kernel<<<static_cast<unsigned>((per_chunk + 255) / 256), 256, 0, s>>>(
        a.lm_part, a.lm_grad, per_chunk, a.lm_chunks, a.status);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
  }
  p.lm_mode = 0;
  p.extra_k = a.rows ? a.extra_k : nullptr;
  p.extra_v = a.rows ? a.extra_v : nullptr;
  bwd_dkdv_tc_kernel<false><<<dim3(n_tiles, a.Hkv, 1), kThreads, kSmemBytes, s>>>(p);
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  if (!a.no_pair && bwd_dq_pair_supported(a)) {
    e = launch_bwd_dq_pair(a, s, why);
  } else {
    bwd_dq_tc_kernel<false><<<dim3(n_tiles, a.Hq), kThreads, kDqSmemBytes, s>>>(p);
    e = cudaPeekAtLastError();
  }
  if (e != cudaSuccess || !a.rows) return e;
  // The global rows' dQ: per key split, then summed into their rows.
  bwd_dq_tc_kernel<true><<<dim3(a.n_splits, static_cast<unsigned>(a.Mp / kT), a.Hkv),
                           kThreads, kDqSmemBytes, s>>>(pg);
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  dq_scatter_kernel<<<static_cast<unsigned>((a.n_global * a.Hq + 7) / 8), 256, 0, s>>>(
      a.dq_part, a.rows, a.n_global, a.Mp, a.n_splits, a.span, a.n, a.Hq, a.Hkv, group, a.dq,
      a.grad_bf16, a.status);
  return cudaPeekAtLastError();
}

}  // namespace msa
