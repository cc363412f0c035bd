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
// CTA = 32 query rows of one head, 256 threads; thread (ty, tx) = (tid / 16,
// tid % 16) owns rows 2 ty, 2 ty + 1.  Per 32-key tile, K and V are staged in
// shared memory as fp32 from 16-byte loads, the next tile's loads in flight
// while this one is computed; the thread computes the scores of its two rows
// against keys tx and tx + 16 (a 2 x 2 block, 128-bit loads along d), the 16
// threads of a row (half a warp) reduce its maximum and sum by shuffles, P
// goes through shared memory, and the thread accumulates its rows' output
// columns 4 tx .. 4 tx + 3 (and 64 + 4 tx .. for d = 128) from 128-bit loads
// of P and V.  Scores use the accurate expf; all sums fp32.
#include <math.h>

#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kBQ = 32;
constexpr int kBK = 32;
constexpr int kThreads = 256;
constexpr int kRowsPerThread = 2;

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
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(const AttnArgs a) {
  constexpr int DP = D + 4;           // padded row (floats) of Q and K: conflict-free 16-B loads
  constexpr int PP = kBK + 4;         // padded row of P
  constexpr int kCols = D / 16;       // output columns per thread (4 or 8)
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;                   // [kBQ][DP]
  float* Ks = Qs + kBQ * DP;          // [kBK][DP]
  float* Vs = Ks + kBK * DP;          // [kBK][D]
  float* Ps = Vs + kBK * D;           // [kBQ][PP]

  const int h = blockIdx.y;
  const int c = h / (a.Hq / a.Hkv);
  const int64_t qr0 = static_cast<int64_t>(blockIdx.x) * kBQ;  // local row of the tile
  const int tid = threadIdx.x;
  const int ty = tid >> 4;
  const int tx = tid & 15;
  const int64_t kv_end = a.kv_start + a.n_kv;

  // Extents (elements) of the buffers, as the entry points define them.
  const int64_t q_ext = a.n_q * a.Hq * static_cast<int64_t>(D);
  const int64_t kv_ext = a.n_kv * a.Hkv * static_cast<int64_t>(D);
  const int64_t lm_ext = static_cast<int64_t>(a.G) * a.Hkv * D;
  const int64_t n_qb_all = (a.n_q + kSelQBlock - 1) / kSelQBlock;
  (void)q_ext, (void)kv_ext, (void)lm_ext, (void)n_qb_all;

  // 16-byte vectors: kVE elements each, kVPR per row of d, kNV per thread
  // for a 32-row tile.
  constexpr int kES = kBf16In ? 2 : 4;
  constexpr int kVE = 16 / kES;
  constexpr int kVPR = D / kVE;
  constexpr int kNV = kBK * kVPR / kThreads;
  static_assert(kNV * kThreads == kBK * kVPR, "tile vectors per thread");
  const uint8_t* qb8 = static_cast<const uint8_t*>(a.q);

  // Stage the query tile.
  {
    uint4 qr[kNV];
#pragma unroll
    for (int v = 0; v < kNV; ++v) {
      const int x = tid + v * kThreads;
      const int64_t row = qr0 + x / kVPR;
      const int64_t off = (row * a.Hq + h) * static_cast<int64_t>(D) + (x % kVPR) * kVE;
      qr[v] = row < a.n_q && MSA_IN_RANGE(off, kVE, q_ext, a.status)
                  ? *reinterpret_cast<const uint4*>(qb8 + off * kES)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < kNV; ++v) {
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

  // K/V vectors of tile t into registers (zeros past the tile's keys).
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
      const int x = tid + v * kThreads;
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
  if (n_tiles > 0) load_tile(0, kr, vr);
  for (int64_t t = 0; t < n_tiles; ++t) {
    const bool is_lm = t < lm_tiles;
    const int64_t base = is_lm ? t * kBK : j_lo + (t - lm_tiles) * kBK;  // landmark idx / global key
    __syncthreads();  // previous tile's K/V/P consumed (and Q staged)
#pragma unroll
    for (int v = 0; v < kNV; ++v) {
      const int x = tid + v * kThreads;
      store_vec<kBf16In>(Ks + (x / kVPR) * DP + (x % kVPR) * kVE, kr[v]);
      store_vec<kBf16In>(Vs + (x / kVPR) * D + (x % kVPR) * kVE, vr[v]);
    }
    // The next tile's loads are in flight while this one is computed.
    if (t + 1 < n_tiles) load_tile(t + 1, kr, vr);
    __syncthreads();

    // Scores of rows 4 ty + r against keys tx and tx + 16.
    float s[kRowsPerThread][2];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) s[r][0] = s[r][1] = 0.f;
#pragma unroll 4
    for (int dc = 0; dc < D / 4; ++dc) {
      const float4 k0 = *reinterpret_cast<const float4*>(Ks + tx * DP + 4 * dc);
      const float4 k1 = *reinterpret_cast<const float4*>(Ks + (tx + 16) * DP + 4 * dc);
#pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r) {
        const float4 qv =
            *reinterpret_cast<const float4*>(Qs + (kRowsPerThread * ty + r) * DP + 4 * dc);
        s[r][0] = dot4(qv, k0, s[r][0]);
        s[r][1] = dot4(qv, k1, s[r][1]);
      }
    }
    float alpha[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int64_t key = base + tx + 16 * j;
        const bool valid = is_lm ? key < my_lm[r] : key >= my_lo[r] && key <= my_hi[r];
        s[r][j] = (valid && row_ok[r]) ? s[r][j] * a.scale : -INFINITY;
        tmax = fmaxf(tmax, s[r][j]);
      }
      // The 16 threads of a row are lanes 0-15 or 16-31 of one warp.
#pragma unroll
      for (int off = 1; off < 16; off <<= 1)
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      const float m_new = fmaxf(m[r], tmax);
      alpha[r] = (m_new == -INFINITY) ? 1.f : expf(m[r] - m_new);  // m = -inf -> 0
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float pj = (m_new == -INFINITY) ? 0.f : expf(s[r][j] - m_new);
        psum += pj;
        Ps[(kRowsPerThread * ty + r) * PP + tx + 16 * j] = pj;
      }
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l[r] = l[r] * alpha[r] + psum;
      m[r] = m_new;
#pragma unroll
      for (int e = 0; e < kCols; ++e) o[r][e] *= alpha[r];
    }
    __syncwarp();  // a row's P is written and read by the 16 threads of one warp
#pragma unroll 2
    for (int kk = 0; kk < kBK; kk += 4) {
      float4 pv[kRowsPerThread];
#pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r)
        pv[r] = *reinterpret_cast<const float4*>(Ps + (kRowsPerThread * ty + r) * PP + kk);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int half = 0; half < kCols / 4; ++half) {
          const float4 vv =
              *reinterpret_cast<const float4*>(Vs + (kk + q) * D + 64 * half + 4 * tx);
#pragma unroll
          for (int r = 0; r < kRowsPerThread; ++r) {
            const float p = q == 0 ? pv[r].x : q == 1 ? pv[r].y : q == 2 ? pv[r].z : pv[r].w;
            o[r][4 * half + 0] = fmaf(p, vv.x, o[r][4 * half + 0]);
            o[r][4 * half + 1] = fmaf(p, vv.y, o[r][4 * half + 1]);
            o[r][4 * half + 2] = fmaf(p, vv.z, o[r][4 * half + 2]);
            o[r][4 * half + 3] = fmaf(p, vv.w, o[r][4 * half + 3]);
          }
        }
      }
    }
  }

  // Epilogue, row by row.  The 16 threads of a row read the running lse
  // (merge) before its first thread writes the new one.
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
    for (int half = 0; half < kCols / 4; ++half) {
      const int64_t col = obase + 64 * half + 4 * tx;
      if (a.out_bf16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + col;
#pragma unroll
        for (int e = 0; e < 4; ++e) out[e] = __float2bfloat16_rn(o[r][4 * half + e] * w_new);
      } else {
        float* out = static_cast<float*>(a.out) + col;
        if (w_run != 0.f) {
#pragma unroll
          for (int e = 0; e < 4; ++e) out[e] = fmaf(out[e], w_run, o[r][4 * half + e] * w_new);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) out[e] = o[r][4 * half + e] * w_new;
        }
      }
    }
    // Every branch above is uniform over the row's 16 threads (one half of
    // the warp), so they meet here.
    __syncwarp((ty & 1) ? 0xffff0000u : 0x0000ffffu);
    if (tx == 0 && l[r] > 0.f) a.lse[lse_idx] = lse_out;
  }
}

template <bool kBf16In, int D>
cudaError_t launch_typed(const AttnArgs& a, cudaStream_t s) {
  const size_t smem =
      sizeof(float) * (kBQ * (D + 4) + kBK * (D + 4) + kBK * D + kBQ * (kBK + 4));
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
