// K2 (CUDA-core variant): fused window + landmark attention with fp32
// arithmetic, for fp32 inputs (and any input the tensor-core kernels do not
// take).  Same method as the tensor-core kernels: one online softmax over the
// visible landmark tiles and the causal window tiles of each query tile
// ("Scaling GPU Cluster for Million Token Context", section "What is
// Flash-MSA Sparse Attention in GPU Clusters?": local window + landmark
// attention fused in one pass, tiled so scores never reach HBM), with the
// running-max / running-sum statistics that "Training at 1M+ Token Context"
// (Ring Attention paragraph) aggregates across rounds.
//
// CTA = 32 query rows of one head, 256 threads.  For d = 64 they form two
// groups of 128 that take alternate key tiles (32 keys), each with its own
// online softmax state, and combine the two states at the end as two key
// chunks combine; for d = 128 one group takes every tile.  The threads of a
// row (8 for d = 64, 16 for d = 128) split its keys and its output columns.
// Per tile, K and V are staged in the group's shared memory as fp32 from
// 16-byte loads, the group's next tile's loads in flight while this one is
// computed; each thread computes the scores of its two rows against its
// keys of the tile (128-bit loads along d, each K vector used for both rows
// and each Q vector for every key of the thread), the threads of a row
// reduce its maximum and sum by shuffles, P goes through shared memory, and
// each thread accumulates its rows' output columns from 128-bit loads of P
// and V.  Scores use the accurate expf; all sums fp32.
#include <math.h>

#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kBQ = 32;            // query rows per CTA
constexpr int kBK = 32;            // keys per tile
constexpr int kThreads = 256;
// Thread groups of a CTA, each on every other key tile, and threads per
// query row: for d = 64 two groups of 128, 8 threads per row (a thread: two
// rows x four keys of a tile, two rows x eight output columns); for d = 128
// one group of 256, 16 threads per row (two rows x two keys, two rows x
// eight columns), which keeps its registers within two CTAs per SM.
__host__ __device__ constexpr int simt_groups(int d) { return d == 64 ? 2 : 1; }
__host__ __device__ constexpr int simt_row_threads(int d) { return d == 64 ? 8 : 16; }

// Barrier of the threads (whole warps) of group g: named barriers 1 and 2
// for two groups of 128, the CTA's for one group.
template <int kGroups>
__device__ __forceinline__ void group_sync(int g) {
  if constexpr (kGroups == 1) {
    __syncthreads();
  } else if (g == 0) {
    asm volatile("bar.sync 1, 128;" ::: "memory");
  } else {
    asm volatile("bar.sync 2, 128;" ::: "memory");
  }
}

// 16 bytes of input (4 fp32 or 8 bf16) widened to fp32 in shared memory.
template <bool kBf16In>
__device__ __forceinline__ void store_vec(float* dst, const uint4 v) {
  if constexpr (kBf16In) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dst[2 * i] = __uint_as_float(w[i] << 16);
      dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    *reinterpret_cast<float4*>(dst) =
        make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                    __uint_as_float(v.w));
  }
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float c) {
  c = fmaf(a.x, b.x, c);
  c = fmaf(a.y, b.y, c);
  c = fmaf(a.z, b.z, c);
  return fmaf(a.w, b.w, c);
}

template <bool kBf16In, int D>
__global__ void __launch_bounds__(kThreads, 2) attn_simt_kernel(const AttnArgs a) {
  constexpr int DP = D + 4;           // padded row (floats) of Q and K: conflict-free 16-B loads
  constexpr int PP = kBK + 4;         // padded row of P
  constexpr int kGroupFloats = kBK * DP + kBK * D + kBQ * PP;
  constexpr int kGroups = simt_groups(D);
  constexpr int kGroupThreads = kThreads / kGroups;
  constexpr int kRowThreads = simt_row_threads(D);  // threads sharing a row: tx
  constexpr int kKeysPerThread = kBK / kRowThreads; // keys tx + kRowThreads j of a tile
  constexpr int kRowsPerThread = kBQ * kRowThreads / kGroupThreads;
  constexpr int kCols = D / kRowThreads;            // output columns per thread
  constexpr int kColStride = 4 * kRowThreads;       // its float4s at kColStride q + 4 tx
  static_assert(kGroupThreads / kRowThreads * kRowsPerThread == kBQ, "rows of a group");
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x;
  const int g = tid / kGroupThreads;  // this thread's group: key tiles g, g + 2, ...
  const int lt = tid % kGroupThreads;
  const int ty = lt / simt_row_threads(D);  // rows kRowsPerThread ty + r
  const int tx = lt % simt_row_threads(D);  // keys tx + kRowThreads j; columns kColStride q + 4 tx
  float* Qs = smem;                                   // [kBQ][DP], shared by both groups
  float* Ks = Qs + kBQ * DP + g * kGroupFloats;       // [kBK][DP], this group's
  float* Vs = Ks + kBK * DP;                          // [kBK][D]
  float* Ps = Vs + kBK * D;                           // [kBQ][PP]

  const int h = blockIdx.y;
  const int c = h / (a.Hq / a.Hkv);
  const int64_t qr0 = static_cast<int64_t>(blockIdx.x) * kBQ;  // local row of the tile
  const int64_t kv_end = a.kv_start + a.n_kv;

  // Extents (elements) of the buffers, as the entry points define them.
  const int64_t q_ext = a.n_q * a.Hq * static_cast<int64_t>(D);
  const int64_t kv_ext = a.n_kv * a.Hkv * static_cast<int64_t>(D);
  const int64_t lm_ext = static_cast<int64_t>(a.G) * a.Hkv * D;
  const int64_t n_qb_all = (a.n_q + kSelQBlock - 1) / kSelQBlock;
  (void)q_ext, (void)kv_ext, (void)lm_ext, (void)n_qb_all;

  // 16-byte vectors: kVE elements each, kVPR per row of d; a 32-row tile is
  // kNVQ vectors per thread of the CTA (Q) or kNV per thread of a group.
  constexpr int kES = kBf16In ? 2 : 4;
  constexpr int kVE = 16 / kES;
  constexpr int kVPR = D / kVE;
  constexpr int kNVQ = kBQ * kVPR / kThreads;
  constexpr int kNV = kBK * kVPR / kGroupThreads;
  static_assert(kNVQ * kThreads == kBQ * kVPR, "query tile vectors per thread");
  static_assert(kNV * kGroupThreads == kBK * kVPR, "key tile vectors per thread");
  const uint8_t* qb8 = static_cast<const uint8_t*>(a.q);

  // Stage the query tile (all threads).
  {
    uint4 qr[kNVQ];
#pragma unroll
    for (int v = 0; v < kNVQ; ++v) {
      const int x = tid + v * kThreads;
      const int64_t row = qr0 + x / kVPR;
      const int64_t off = (row * a.Hq + h) * static_cast<int64_t>(D) + (x % kVPR) * kVE;
      qr[v] = row < a.n_q && MSA_IN_RANGE(off, kVE, q_ext, a.status)
                  ? *reinterpret_cast<const uint4*>(qb8 + off * kES)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < kNVQ; ++v) {
      const int x = tid + v * kThreads;
      store_vec<kBf16In>(Qs + (x / kVPR) * DP + (x % kVPR) * kVE, qr[v]);
    }
  }

  // Key ranges of the whole tile (global positions).
  const int64_t g0 = a.q_start + qr0;
  const int64_t g_last = a.q_start + min64(qr0 + kBQ, a.n_q) - 1;
  int64_t j_lo, j_hi;
  if (a.band) {  // union of the rows' bands (whole sequence: kv_start = 0)
    int64_t unused;
    band_keys(g0, a.band_block, a.band_half, a.n_kv, &j_lo, &unused);
    band_keys(g_last, a.band_block, a.band_half, a.n_kv, &unused, &j_hi);
  } else {
    j_lo = max64(g0 - a.window + 1, a.kv_start);
    j_hi = min64(g_last, kv_end - 1);
  }
  const int64_t n_win = j_hi >= j_lo ? j_hi - j_lo + 1 : 0;
  // Landmark keys, or (select mode) the tokens of the query block's
  // selected key blocks; a 32-row tile lies inside one 128-row query block.
  const int64_t qb = qr0 / kSelQBlock;
  const int64_t n_cand = a.sel ? visible_landmarks(qb * kSelQBlock, a.window, a.block, a.G) : 0;
  const int32_t* sel_list =
      a.sel ? a.sel + (qb * a.Hkv + c) * static_cast<int64_t>(a.top_k) : nullptr;
  const int64_t n_lm =
      a.sel ? (MSA_IN_RANGE(qb * a.Hkv + c, 1, n_qb_all * a.Hkv, a.status)
                   ? sel_count_checked(a.sel_cnt[qb * a.Hkv + c], a.top_k, n_cand, a.status)
                   : 0) * a.block
            : visible_landmarks(g_last, a.window, a.block, a.G);
  const int64_t lm_tiles = (n_lm + kBK - 1) / kBK;
  const int64_t win_tiles = (n_win + kBK - 1) / kBK;

  // This thread's rows and their sets.
  int64_t my_lo[kRowsPerThread], my_hi[kRowsPerThread], my_lm[kRowsPerThread];
  bool row_ok[kRowsPerThread];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    const int64_t i_loc = qr0 + kRowsPerThread * ty + r;
    const int64_t i = a.q_start + i_loc;
    row_ok[r] = i_loc < a.n_q;
    if (a.band) {
      band_keys(i, a.band_block, a.band_half, a.n_kv, &my_lo[r], &my_hi[r]);
    } else {
      my_lo[r] = max64(i - a.window + 1, a.kv_start);
      my_hi[r] = min64(i, kv_end - 1);
    }
    my_lm[r] = a.sel ? n_lm : visible_landmarks(i, a.window, a.block, a.G);
  }

  float o[kRowsPerThread][kCols];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r)
#pragma unroll
    for (int e = 0; e < kCols; ++e) o[r][e] = 0.f;
  float m[kRowsPerThread], l[kRowsPerThread];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
  }

  // K/V vectors of tile t into registers (zeros past the tile's keys); each
  // group loads its own tiles.
  const uint8_t* kb8 = static_cast<const uint8_t*>(a.k);
  const uint8_t* vb8 = static_cast<const uint8_t*>(a.v);
  const uint8_t* klm8 = static_cast<const uint8_t*>(a.k_lm);
  const uint8_t* vlm8 = static_cast<const uint8_t*>(a.v_lm);
  auto load_tile = [&](int64_t t, uint4 (&kr)[kNV], uint4 (&vr)[kNV]) {
    const bool is_lm = t < lm_tiles;
    const int64_t base = is_lm ? t * kBK : j_lo + (t - lm_tiles) * kBK;
    const int64_t limit = is_lm ? n_lm : j_hi + 1;
#pragma unroll
    for (int v = 0; v < kNV; ++v) {
      const int x = lt + v * kGroupThreads;
      const int64_t key = base + x / kVPR;
      const int64_t col = (x % kVPR) * kVE;
      kr[v] = vr[v] = make_uint4(0, 0, 0, 0);
      if (key < limit) {
        if (is_lm && sel_list) {
          const int64_t si = (qb * a.Hkv + c) * static_cast<int64_t>(a.top_k) + key / a.block;
          (void)si;
          const int64_t tok =
              MSA_IN_RANGE(si, 1, n_qb_all * a.Hkv * a.top_k, a.status)
                  ? sel_block_checked(sel_list[key / a.block], n_cand, a.status) * a.block +
                        key % a.block
                  : 0;
          const int64_t off = (tok * a.Hkv + c) * static_cast<int64_t>(D) + col;
          if (MSA_IN_RANGE(off, kVE, kv_ext, a.status)) {
            kr[v] = *reinterpret_cast<const uint4*>(kb8 + off * kES);
            vr[v] = *reinterpret_cast<const uint4*>(vb8 + off * kES);
          }
        } else if (is_lm) {
          const int64_t off = (key * a.Hkv + c) * static_cast<int64_t>(D) + col;
          if (MSA_IN_RANGE(off, kVE, lm_ext, a.status)) {
            kr[v] = *reinterpret_cast<const uint4*>(klm8 + off * kES);
            vr[v] = *reinterpret_cast<const uint4*>(vlm8 + off * kES);
          }
        } else {
          const int64_t off = ((key - a.kv_start) * a.Hkv + c) * static_cast<int64_t>(D) + col;
          if (MSA_IN_RANGE(off, kVE, kv_ext, a.status)) {
            kr[v] = *reinterpret_cast<const uint4*>(kb8 + off * kES);
            vr[v] = *reinterpret_cast<const uint4*>(vb8 + off * kES);
          }
        }
      }
    }
  };

  const int64_t n_tiles = lm_tiles + win_tiles;
  uint4 kr[kNV], vr[kNV];
  if (g < n_tiles) load_tile(g, kr, vr);
  __syncthreads();  // the query tile is staged
  for (int64_t t = g; t < n_tiles; t += kGroups) {
    const bool is_lm = t < lm_tiles;
    const int64_t base = is_lm ? t * kBK : j_lo + (t - lm_tiles) * kBK;  // landmark idx / global key
    group_sync<kGroups>(g);  // this group's previous tile (K, V, P) consumed
#pragma unroll
    for (int v = 0; v < kNV; ++v) {
      const int x = lt + v * kGroupThreads;
      store_vec<kBf16In>(Ks + (x / kVPR) * DP + (x % kVPR) * kVE, kr[v]);
      store_vec<kBf16In>(Vs + (x / kVPR) * D + (x % kVPR) * kVE, vr[v]);
    }
    // The group's next tile's loads are in flight while this one is computed.
    if (t + kGroups < n_tiles) load_tile(t + kGroups, kr, vr);
    group_sync<kGroups>(g);

    // Scores of rows kRowsPerThread ty + r against keys tx + kRowThreads j:
    // 16-byte loads along d, each K vector used for every row of the thread
    // and each Q vector for every key.
    float s[kRowsPerThread][kKeysPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r)
#pragma unroll
      for (int j = 0; j < kKeysPerThread; ++j) s[r][j] = 0.f;
#pragma unroll 4
    for (int dc = 0; dc < D / 4; ++dc) {
      float4 kv[kKeysPerThread];
#pragma unroll
      for (int j = 0; j < kKeysPerThread; ++j)
        kv[j] = *reinterpret_cast<const float4*>(Ks + (tx + kRowThreads * j) * DP + 4 * dc);
#pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r) {
        const float4 qv =
            *reinterpret_cast<const float4*>(Qs + (kRowsPerThread * ty + r) * DP + 4 * dc);
#pragma unroll
        for (int j = 0; j < kKeysPerThread; ++j) s[r][j] = dot4(qv, kv[j], s[r][j]);
      }
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kKeysPerThread; ++j) {
        const int64_t key = base + tx + kRowThreads * j;
        const bool valid = is_lm ? key < my_lm[r] : key >= my_lo[r] && key <= my_hi[r];
        s[r][j] = (valid && row_ok[r]) ? s[r][j] * a.scale : -INFINITY;
        tmax = fmaxf(tmax, s[r][j]);
      }
      // The threads of a row are consecutive lanes of one warp.
#pragma unroll
      for (int off = 1; off < kRowThreads; off <<= 1)
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float m_new = fmaxf(m[r], tmax);
      const float alpha = (m_new == -INFINITY) ? 1.f : expf(m[r] - m_new);  // m = -inf -> 0
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < kKeysPerThread; ++j) {
        const float pj = (m_new == -INFINITY) ? 0.f : expf(s[r][j] - m_new);
        psum += pj;
        Ps[(kRowsPerThread * ty + r) * PP + tx + kRowThreads * j] = pj;
      }
#pragma unroll
      for (int off = 1; off < kRowThreads; off <<= 1)
        psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l[r] = l[r] * alpha + psum;
      m[r] = m_new;
#pragma unroll
      for (int e = 0; e < kCols; ++e) o[r][e] *= alpha;
    }
    __syncwarp();  // a row's P is written and read by the threads of one warp
    // O += P V for this thread's rows and its columns kColStride q + 4 tx .. + 3.
#pragma unroll 2
    for (int kk = 0; kk < kBK; kk += 4) {
      float4 pv[kRowsPerThread];
#pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r)
        pv[r] = *reinterpret_cast<const float4*>(Ps + (kRowsPerThread * ty + r) * PP + kk);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int cq = 0; cq < kCols / 4; ++cq) {
          const float4 vv =
              *reinterpret_cast<const float4*>(Vs + (kk + q) * D + kColStride * cq + 4 * tx);
#pragma unroll
          for (int r = 0; r < kRowsPerThread; ++r) {
            const float p = q == 0 ? pv[r].x : q == 1 ? pv[r].y : q == 2 ? pv[r].z : pv[r].w;
            o[r][4 * cq + 0] = fmaf(p, vv.x, o[r][4 * cq + 0]);
            o[r][4 * cq + 1] = fmaf(p, vv.y, o[r][4 * cq + 1]);
            o[r][4 * cq + 2] = fmaf(p, vv.z, o[r][4 * cq + 2]);
            o[r][4 * cq + 3] = fmaf(p, vv.w, o[r][4 * cq + 3]);
          }
        }
      }
    }
  }

  if constexpr (kGroups == 2) {
    // The two groups' online-softmax states of a row combine as two key
    // chunks do: m = max(m0, m1), l and O each scaled by e^(m_g - m).  Group 1
    // leaves its state in its own K/V buffers, idle by now; group 0 combines
    // it with its own and writes the row.
    __syncthreads();  // both groups' tiles done
    float* xo = Qs + kBQ * DP + kGroupFloats;  // [kBQ][D] O of group 1, then m and l per row
    float* xm = xo + kBQ * D;
    float* xl = xm + kBQ;
    static_assert(kBQ * D + 2 * kBQ <= kBK * DP + kBK * D, "group 1's state fits its K/V buffers");
    if (g == 1) {
  #pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r) {
        const int row = kRowsPerThread * ty + r;
  #pragma unroll
        for (int cq = 0; cq < kCols / 4; ++cq)
          *reinterpret_cast<float4*>(xo + row * D + kColStride * cq + 4 * tx) =
              make_float4(o[r][4 * cq], o[r][4 * cq + 1], o[r][4 * cq + 2], o[r][4 * cq + 3]);
        if (tx == 0) {
          xm[row] = m[r];
          xl[row] = l[r];
        }
      }
    }
    __syncthreads();
    if (g == 1) return;
  #pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      const int row = kRowsPerThread * ty + r;
      const float m1 = xm[row];
      const float mm = fmaxf(m[r], m1);
      const float a0 = m[r] == -INFINITY ? 0.f : expf(m[r] - mm);
      const float a1 = m1 == -INFINITY ? 0.f : expf(m1 - mm);
      l[r] = l[r] * a0 + xl[row] * a1;
      m[r] = mm;
  #pragma unroll
      for (int cq = 0; cq < kCols / 4; ++cq) {
        const float4 x =
            *reinterpret_cast<const float4*>(xo + row * D + kColStride * cq + 4 * tx);
        o[r][4 * cq + 0] = o[r][4 * cq + 0] * a0 + x.x * a1;
        o[r][4 * cq + 1] = o[r][4 * cq + 1] * a0 + x.y * a1;
        o[r][4 * cq + 2] = o[r][4 * cq + 2] * a0 + x.z * a1;
        o[r][4 * cq + 3] = o[r][4 * cq + 3] * a0 + x.w * a1;
      }
    }
  }

  // Epilogue, row by row (group 0).  The threads of a row read the running
  // lse (merge) before its first thread writes the new one.
  const unsigned row_lanes = ((1u << kRowThreads) - 1u)
                             << ((ty % (32 / kRowThreads)) * kRowThreads);
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    if (!row_ok[r]) continue;
    const int64_t i_loc = qr0 + kRowsPerThread * ty + r;
    const int64_t lse_idx = static_cast<int64_t>(h) * a.lse_ld + i_loc;
    const int64_t obase = (i_loc * a.Hq + h) * static_cast<int64_t>(D);
    if (!MSA_IN_RANGE(lse_idx, 1, (a.Hq - 1) * a.lse_ld + a.n_q, a.status)) continue;
    if (!MSA_IN_RANGE(obase, D, q_ext, a.status)) continue;
    if (l[r] == 0.f) {  // no key for this row (only possible for a partial)
      if (a.merge) continue;  // a running merge leaves the row untouched
      if (tx == 0) a.lse[lse_idx] = -INFINITY;
      if (a.partial) continue;
    }
    const float lse_p = l[r] > 0.f ? m[r] + logf(l[r]) : -INFINITY;
    float w_new = l[r] > 0.f ? 1.f / l[r] : 0.f;
    float w_run = 0.f;
    float lse_out = lse_p;
    if (a.merge) {  // lse_run <- ln(e^lse_run + e^lse_p), O <- O w_run + O_p w
      const float L = a.lse[lse_idx];
      if (L != -INFINITY) {
        const float mx = fmaxf(L, lse_p);
        lse_out = mx + logf(expf(L - mx) + expf(lse_p - mx));
        w_run = expf(L - lse_out);
        w_new *= expf(lse_p - lse_out);
      }
    }
#pragma unroll
    for (int cq = 0; cq < kCols / 4; ++cq) {
      const int64_t col = obase + kColStride * cq + 4 * tx;
      if (a.out_bf16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + col;
#pragma unroll
        for (int e = 0; e < 4; ++e) out[e] = __float2bfloat16_rn(o[r][4 * cq + e] * w_new);
      } else {
        float* out = static_cast<float*>(a.out) + col;
        if (w_run != 0.f) {
#pragma unroll
          for (int e = 0; e < 4; ++e) out[e] = fmaf(out[e], w_run, o[r][4 * cq + e] * w_new);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) out[e] = o[r][4 * cq + e] * w_new;
        }
      }
    }
    // Every branch above is uniform over the row's threads (consecutive
    // lanes of one warp), so they meet here.
    __syncwarp(row_lanes);
    if (tx == 0 && l[r] > 0.f) a.lse[lse_idx] = lse_out;
  }
}

template <bool kBf16In, int D>
cudaError_t launch_typed(const AttnArgs& a, cudaStream_t s) {
  const size_t smem =
      sizeof(float) *
      (kBQ * (D + 4) + simt_groups(D) * (kBK * (D + 4) + kBK * D + kBQ * (kBK + 4)));
  cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<kBf16In, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.n_q + kBQ - 1) / kBQ), a.Hq);
  attn_simt_kernel<kBf16In, D><<<grid, kThreads, smem, s>>>(a);
  return cudaPeekAtLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s) {
  if (a.in_bf16) {
    return a.d == 64 ? launch_typed<true, 64>(a, s) : launch_typed<true, 128>(a, s);
  }
  return a.d == 64 ? launch_typed<false, 64>(a, s) : launch_typed<false, 128>(a, s);
}

}  // namespace msa
