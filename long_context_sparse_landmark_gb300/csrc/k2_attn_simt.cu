// K2 (CUDA-core variant): fused window + landmark attention with fp32
// arithmetic, for fp32 inputs (and any input the tensor-core kernel does not
// take).  Same method as the tensor-core kernel: one online softmax over the
// visible landmark tiles and the causal window tiles of each query tile
// ("Scaling GPU Cluster for Million Token Context", section "What is
// Flash-MSA Sparse Attention in GPU Clusters?": local window + landmark
// attention fused in one pass, tiled so scores never reach HBM), with the
// running-max / running-sum statistics that "Training at 1M+ Token Context"
// (Ring Attention paragraph) aggregates across rounds.
//
// CTA = 64 query rows of one head, 256 threads; thread (r, q) = (tid/4,
// tid%4).  Per 32-key tile: K and V staged in shared memory as fp32, each
// thread scores 8 keys of its row, the 4 threads of a row reduce max/sum by
// shuffles, P goes through shared memory, and each thread accumulates d/4
// output columns (interleaved, column 4e+q) in registers.  Scores use the
// accurate expf; all sums are fp32.
#include <math.h>

#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kBQ = 64;
constexpr int kBK = 32;
constexpr int kThreads = 256;

template <bool kBf16In>
__device__ __forceinline__ float ld_in(const void* base, int64_t idx) {
  if constexpr (kBf16In) {
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
  } else {
    return static_cast<const float*>(base)[idx];
  }
}

template <bool kBf16In, int D>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(const AttnArgs a) {
  extern __shared__ float smem[];
  float* Qs = smem;                     // [kBQ][D+1]
  float* Ks = Qs + kBQ * (D + 1);       // [kBK][D+1]
  float* Vs = Ks + kBK * (D + 1);       // [kBK][D]
  float* Ps = Vs + kBK * D;             // [kBQ][kBK+1]

  const int h = blockIdx.y;
  const int c = h / (a.Hq / a.Hkv);
  const int64_t qr0 = static_cast<int64_t>(blockIdx.x) * kBQ;  // local row of the tile
  const int tid = threadIdx.x;
  const int r = tid >> 2;
  const int qd = tid & 3;
  const int64_t i_loc = qr0 + r;
  const bool row_ok = i_loc < a.n_q;
  const int64_t i = a.q_start + i_loc;  // global position
  const int64_t kv_end = a.kv_start + a.n_kv;

  // Extents (elements) of the buffers, as the entry points define them.
  const int64_t q_ext = a.n_q * a.Hq * static_cast<int64_t>(D);
  const int64_t kv_ext = a.n_kv * a.Hkv * static_cast<int64_t>(D);
  const int64_t lm_ext = static_cast<int64_t>(a.G) * a.Hkv * D;
  const int64_t n_qb_all = (a.n_q + kSelQBlock - 1) / kSelQBlock;
  (void)q_ext, (void)kv_ext, (void)lm_ext, (void)n_qb_all;

  // Stage the query tile.
  for (int x = tid; x < kBQ * D; x += kThreads) {
    const int rr = x / D, e = x % D;
    const int64_t row = qr0 + rr;
    const int64_t off = (row * a.Hq + h) * static_cast<int64_t>(D) + e;
    Qs[rr * (D + 1) + e] =
        row < a.n_q && MSA_IN_RANGE(off, 1, q_ext, a.status) ? ld_in<kBf16In>(a.q, off) : 0.f;
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
  // selected key blocks; a 64-row tile lies inside one 128-row query block.
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

  // This row's own sets.
  int64_t my_lo, my_hi;
  if (a.band) {
    band_keys(i, a.band_block, a.band_half, a.n_kv, &my_lo, &my_hi);
  } else {
    my_lo = max64(i - a.window + 1, a.kv_start);
    my_hi = min64(i, kv_end - 1);
  }
  const int64_t my_lm = a.sel ? n_lm : visible_landmarks(i, a.window, a.block, a.G);

  constexpr int DQ = D / 4;
  float o[DQ];
#pragma unroll
  for (int e = 0; e < DQ; ++e) o[e] = 0.f;
  float m = -INFINITY, l = 0.f;

  for (int64_t t = 0; t < lm_tiles + win_tiles; ++t) {
    const bool is_lm = t < lm_tiles;
    const int64_t base = is_lm ? t * kBK : j_lo + (t - lm_tiles) * kBK;  // landmark idx / global key
    const int64_t limit = is_lm ? n_lm : j_hi + 1;
    __syncthreads();  // previous tile's K/V/P fully consumed (and Q staged)
    for (int x = tid; x < kBK * D; x += kThreads) {
      const int kk = x / D, e = x % D;
      const int64_t key = base + kk;
      float kv = 0.f, vv = 0.f;
      if (key < limit) {
        if (is_lm && sel_list) {
          const int64_t si = (qb * a.Hkv + c) * static_cast<int64_t>(a.top_k) + key / a.block;
          const int64_t tok =
              MSA_IN_RANGE(si, 1, n_qb_all * a.Hkv * a.top_k, a.status)
                  ? sel_block_checked(sel_list[key / a.block], n_cand, a.status) * a.block +
                        key % a.block
                  : 0;
          const int64_t off = (tok * a.Hkv + c) * static_cast<int64_t>(D) + e;
          if (MSA_IN_RANGE(off, 1, kv_ext, a.status)) {
            kv = ld_in<kBf16In>(a.k, off);
            vv = ld_in<kBf16In>(a.v, off);
          }
        } else if (is_lm) {
          const int64_t off = (key * a.Hkv + c) * static_cast<int64_t>(D) + e;
          if (MSA_IN_RANGE(off, 1, lm_ext, a.status)) {
            kv = ld_in<kBf16In>(a.k_lm, off);
            vv = ld_in<kBf16In>(a.v_lm, off);
          }
        } else {
          const int64_t off = ((key - a.kv_start) * a.Hkv + c) * static_cast<int64_t>(D) + e;
          if (MSA_IN_RANGE(off, 1, kv_ext, a.status)) {
            kv = ld_in<kBf16In>(a.k, off);
            vv = ld_in<kBf16In>(a.v, off);
          }
        }
      }
      Ks[kk * (D + 1) + e] = kv;
      Vs[kk * D + e] = vv;
    }
    __syncthreads();

    // Scores of keys qd, qd+4, ..., qd+28 for row r.
    float s[kBK / 4];
    float tmax = -INFINITY;
#pragma unroll
    for (int mi = 0; mi < kBK / 4; ++mi) {
      const int kk = qd + 4 * mi;
      const int64_t key = base + kk;
      bool valid;
      if (is_lm) {
        valid = key < my_lm;
      } else {
        valid = key >= my_lo && key <= my_hi;
      }
      float dot = 0.f;
      const float* qrow = Qs + r * (D + 1);
      const float* krow = Ks + kk * (D + 1);
#pragma unroll 16
      for (int e = 0; e < D; ++e) dot = fmaf(qrow[e], krow[e], dot);
      s[mi] = (valid && row_ok) ? dot * a.scale : -INFINITY;
      tmax = fmaxf(tmax, s[mi]);
    }
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
    const float m_new = fmaxf(m, tmax);
    const float alpha = (m_new == -INFINITY) ? 1.f : expf(m - m_new);  // m = -inf -> 0
    float psum = 0.f;
#pragma unroll
    for (int mi = 0; mi < kBK / 4; ++mi) {
      const float p = (m_new == -INFINITY) ? 0.f : expf(s[mi] - m_new);
      psum += p;
      Ps[r * (kBK + 1) + qd + 4 * mi] = p;
    }
    psum += __shfl_xor_sync(0xffffffffu, psum, 1);
    psum += __shfl_xor_sync(0xffffffffu, psum, 2);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int e = 0; e < DQ; ++e) o[e] *= alpha;
    __syncwarp();  // the 4 threads of a row live in one warp
#pragma unroll 4
    for (int kk = 0; kk < kBK; ++kk) {
      const float p = Ps[r * (kBK + 1) + kk];
      const float* vrow = Vs + kk * D;
#pragma unroll
      for (int e = 0; e < DQ; ++e) o[e] = fmaf(p, vrow[4 * e + qd], o[e]);
    }
  }

  if (!row_ok) return;
  const int64_t lse_idx = static_cast<int64_t>(h) * a.lse_ld + i_loc;
  if (!MSA_IN_RANGE(lse_idx, 1, (a.Hq - 1) * a.lse_ld + a.n_q, a.status)) return;
  if (!MSA_IN_RANGE((i_loc * a.Hq + h) * static_cast<int64_t>(D), D, q_ext, a.status)) return;
  if (l == 0.f) {  // no key for this row (only possible for a partial)
    if (a.merge) return;  // a running merge leaves the row untouched
    if (qd == 0) a.lse[lse_idx] = -INFINITY;
    if (a.partial) return;
  }
  const float lse_p = l > 0.f ? m + logf(l) : -INFINITY;
  float w_new = l > 0.f ? 1.f / l : 0.f;
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
  const int64_t obase = (i_loc * a.Hq + h) * static_cast<int64_t>(D);
  if (a.out_bf16) {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + obase;
#pragma unroll
    for (int e = 0; e < DQ; ++e) out[4 * e + qd] = __float2bfloat16_rn(o[e] * w_new);
  } else {
    float* out = static_cast<float*>(a.out) + obase;
    if (w_run != 0.f) {
#pragma unroll
      for (int e = 0; e < DQ; ++e) out[4 * e + qd] = fmaf(out[4 * e + qd], w_run, o[e] * w_new);
    } else {
#pragma unroll
      for (int e = 0; e < DQ; ++e) out[4 * e + qd] = o[e] * w_new;
    }
  }
  // All four threads of the row have read the running lse above; the row's
  // first thread writes it only after the other three are past that read.
  __syncwarp();
  if (qd == 0 && l > 0.f) a.lse[lse_idx] = lse_out;
}

template <bool kBf16In, int D>
cudaError_t launch_typed(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(float) * (kBQ * (D + 1) + kBK * (D + 1) + kBK * D + kBQ * (kBK + 1));
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
