// K3: exact merge of attention partials over disjoint key sets -- the step a
// Ring Attention round takes when it "aggregates softmax statistics"
// ("Training at 1M+ Token Context: Ring Attention, YaRN, NTK-Aware Scaling",
// Ring Attention paragraph):
//     lse = ln sum_p exp(lse_p),   O = sum_p exp(lse_p - lse) * O_p,
// parts with lse_p = -inf (no key in that chunk) are skipped and not read.
//
// Memory-bound streaming pass.  A CTA owns R consecutive rows x all heads,
// which are contiguous in every O_p ([n, Hq, d] layout).  It first loads the
// P x Hq x R log-sum-exps (R consecutive floats per (part, head)), computes
// every row's merged lse and per-part weights into shared memory, then
// streams the O_p slabs with 16-byte loads, weighting and summing in fp32
// registers, and writes O once.
#include <math.h>

#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMergeUnroll = 4;
constexpr int kMergeMaxWeights = 8192;  // floats of shared memory for weights

__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const MergeArgs a, int rows_per_cta) {
  extern __shared__ float wsm[];  // [P][Hq * R] weights
  const int P = a.n_parts;
  const int Hq = a.Hq;
  const int R = rows_per_cta;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R;
  const int rows = static_cast<int>(min64(R, a.n - r0));
  const int HR = Hq * R;

  // Pass 1: merged lse and weights for each (head, row) of the tile.
  for (int x = threadIdx.x; x < HR; x += blockDim.x) {
    const int h = x / R;
    const int r = x % R;
    if (r >= rows) continue;
    const int64_t li = static_cast<int64_t>(h) * a.n + r0 + r;
    if (!MSA_IN_RANGE(li, 1, static_cast<int64_t>(Hq) * a.n, a.status)) continue;
    float mx = -INFINITY;
    for (int p = 0; p < P; ++p) mx = fmaxf(mx, a.lse_parts[p][li]);
    if (mx == -INFINITY) {
      for (int p = 0; p < P; ++p) wsm[p * HR + x] = 0.f;
      a.lse[li] = -INFINITY;
      continue;
    }
    float sum = 0.f;
    for (int p = 0; p < P; ++p) {
      const float l = a.lse_parts[p][li];
      if (l != -INFINITY) sum += expf(l - mx);
    }
    const float total = mx + logf(sum);
    for (int p = 0; p < P; ++p) {
      const float l = a.lse_parts[p][li];
      wsm[p * HR + x] = l == -INFINITY ? -1.f : expf(l - total);  // -1 marks "skip"
    }
    a.lse[li] = total;
  }
  __syncthreads();

  // Pass 2: stream the partial outputs.
  const int d4 = a.d / 4;
  const int64_t tile_f4 = static_cast<int64_t>(rows) * Hq * d4;
  const int64_t base_f4 = r0 * Hq * d4;
  const int64_t all_f4 = a.n * Hq * d4;  // float4s of each O_p and of O
  (void)all_f4;
  for (int64_t f0 = threadIdx.x; f0 < tile_f4; f0 += static_cast<int64_t>(blockDim.x) * kMergeUnroll) {
    float4 acc[kMergeUnroll];
    int widx[kMergeUnroll];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int64_t f = f0 + static_cast<int64_t>(u) * blockDim.x;
      const int64_t rh = f / d4;  // row-major (row, head) index within the tile
      const int r = static_cast<int>(rh / Hq);
      const int h = static_cast<int>(rh % Hq);
      widx[u] = f < tile_f4 ? h * R + r : -1;
    }
    for (int p = 0; p < P; ++p) {
      const float4* src = reinterpret_cast<const float4*>(a.o_parts[p]) + base_f4;
      float4 x[kMergeUnroll];
      float w[kMergeUnroll];
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        const int64_t f = f0 + static_cast<int64_t>(u) * blockDim.x;
        w[u] = widx[u] >= 0 ? wsm[p * HR + widx[u]] : -1.f;
        x[u] = w[u] >= 0.f && MSA_IN_RANGE(base_f4 + f, 1, all_f4, a.status)
                   ? src[f]
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kMergeUnroll; ++u) {
        if (w[u] > 0.f) {
          acc[u].x = fmaf(w[u], x[u].x, acc[u].x);
          acc[u].y = fmaf(w[u], x[u].y, acc[u].y);
          acc[u].z = fmaf(w[u], x[u].z, acc[u].z);
          acc[u].w = fmaf(w[u], x[u].w, acc[u].w);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const int64_t f = f0 + static_cast<int64_t>(u) * blockDim.x;
      if (f >= tile_f4 || !MSA_IN_RANGE(base_f4 + f, 1, all_f4, a.status)) continue;
      if (a.out_bf16) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[u].x, acc[u].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[u].z, acc[u].w);
        uint2 pk = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
        reinterpret_cast<uint2*>(a.out)[base_f4 + f] = pk;
      } else {
        reinterpret_cast<float4*>(a.out)[base_f4 + f] = acc[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s) {
  // Rows per CTA: about 8192 float4 of each part per CTA, bounded by the
  // shared memory that holds P x Hq x R weights.
  const int d4 = a.d / 4;
  int R = static_cast<int>(max64(1, 8192 / (static_cast<int64_t>(a.Hq) * d4)));
  while (R > 1 && static_cast<int64_t>(a.n_parts) * a.Hq * R > kMergeMaxWeights) R /= 2;
  if (static_cast<int64_t>(a.n_parts) * a.Hq * R > kMergeMaxWeights * 4) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(a.n_parts) * a.Hq * R * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(lse_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int64_t blocks = (a.n + R - 1) / R;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), kMergeThreads, smem, s>>>(a, R);
  return cudaPeekAtLastError();
}

}  // namespace msa
