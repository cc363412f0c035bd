// K4: landmark-scored top-k block selection -- the stand-in for the
// hierarchical context index of "Million Token Context Window Optimization:
// What Actually Works", section "The indexing game: smarter context
// management" (score the chunks of the input against the query, attend only
// the top-k chunks plus a history window; a chunk's landmark, its mean key,
// scores it here instead of a BERT embedding).
//
// One CTA per (query block of 128 rows, KV group): it sums the block's
// queries over rows and the group's heads (fp32, 16-byte vector loads, the
// partial sums reduced in a fixed order), scores every key block
// wholly before the window of the block's first row against its landmark
// key, ranks the scores (ties to the lower block index) and writes the
// top-k block indices in ascending order, and their count.
#include <math.h>

#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kSelThreads = 256;

// Sort buffer size of the rank pass: the least power of two >= G.
__host__ __device__ inline int sel_sort_size(int G) {
  int P = 1;
  while (P < G) P <<= 1;
  return P;
}

template <bool kBf16>
__global__ void __launch_bounds__(kSelThreads) block_select_kernel(const SelectArgs a) {
  constexpr int V = kBf16 ? 8 : 4;  // elements per 16-byte load
  extern __shared__ float ssm[];
  float* qsum = ssm;                    // [d]
  float* part = qsum + a.d;             // [kSelThreads * V] partial sums
  float* score = part + kSelThreads * 8;  // [G]
  int* flag = reinterpret_cast<int*>(score + a.G);  // [G]
  const int P = sel_sort_size(a.G);                  // power of two >= G
  float* key = reinterpret_cast<float*>(flag + a.G);  // [P] sort keys
  int* idx = reinterpret_cast<int*>(key + P);         // [P] their block indices
  const int t = blockIdx.x;        // query block
  const int c = blockIdx.y;        // KV group
  const int d = a.d;
  const int g = a.Hq / a.Hkv;
  const int64_t r0 = static_cast<int64_t>(t) * kSelQBlock;
  const int64_t r1 = min64(r0 + kSelQBlock, a.n);

  // Query-block sum over rows and the group's heads: thread (slot, vi)
  // adds 16-byte vector vi of every slots-th (row, head) pair (a row's g
  // heads are contiguous), then the slots are summed in a fixed order.
  {
    const int VP = d / V;                 // vectors per (row, head)
    const int slots = kSelThreads / VP;
    const int vi = threadIdx.x % VP;
    const int ps = threadIdx.x / VP;
    const int64_t npairs = (r1 - r0) * g;
    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = 0.f;
    const uint8_t* qb = static_cast<const uint8_t*>(a.q);
    constexpr int ES = kBf16 ? 2 : 4;
    // (row, head) of pair pr = ps + slots * k, stepped without divisions.
    int64_t i = r0 + ps / g;
    int hh = ps % g;
    const int di = slots / g, dh = slots % g;
#pragma unroll 16
    for (int64_t pr = ps; pr < npairs; pr += slots) {
      const int64_t off = (i * a.Hq + c * g + hh) * static_cast<int64_t>(d) + vi * V;
      const uint4 x = MSA_IN_RANGE(off, V, a.n * a.Hq * static_cast<int64_t>(d), a.status)
                          ? __ldg(reinterpret_cast<const uint4*>(qb + off * ES))
                          : make_uint4(0, 0, 0, 0);
      if constexpr (kBf16) {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[2 * k] += __uint_as_float(w[k] << 16);
          acc[2 * k + 1] += __uint_as_float(w[k] & 0xffff0000u);
        }
      } else {
        acc[0] += __uint_as_float(x.x);
        acc[1] += __uint_as_float(x.y);
        acc[2] += __uint_as_float(x.z);
        acc[3] += __uint_as_float(x.w);
      }
      i += di;
      hh += dh;
      if (hh >= g) {
        hh -= g;
        ++i;
      }
    }
#pragma unroll
    for (int k = 0; k < V; ++k) part[ps * d + vi * V + k] = acc[k];
    __syncthreads();
    for (int e = threadIdx.x; e < d; e += blockDim.x) {
      float s = 0.f;
      for (int q = 0; q < slots; ++q) s += part[q * d + e];
      qsum[e] = s;
    }
    __syncthreads();
  }

  // Candidates: blocks l with (l+1)*bs <= r0 - w + 1.
  // One thread per candidate: its landmark key row in 16-byte loads (all in
  // flight at once), dotted with the query sum read as a shared-memory
  // broadcast, in a fixed order.
  const int64_t n_cand = visible_landmarks(r0, a.window, a.block, a.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t l = threadIdx.x; l < n_cand; l += blockDim.x) {
    constexpr int ES = kBf16 ? 2 : 4;
    const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.k_lm) +
                                                      (l * a.Hkv + c) * static_cast<int64_t>(d) *
                                                          ES);
    float s = 0.f;
    if (!MSA_IN_RANGE((l * a.Hkv + c) * static_cast<int64_t>(d), d,
                      static_cast<int64_t>(a.G) * a.Hkv * d, a.status)) {
      score[l] = -INFINITY;
      continue;
    }
#pragma unroll 4
    for (int v0 = 0; v0 < d / V; ++v0) {
      const uint4 x = __ldg(row + v0);
      const float* qv = qsum + v0 * V;
      if constexpr (kBf16) {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          s = fmaf(qv[2 * k], __uint_as_float(w[k] << 16), s);
          s = fmaf(qv[2 * k + 1], __uint_as_float(w[k] & 0xffff0000u), s);
        }
      } else {
        s = fmaf(qv[0], __uint_as_float(x.x), s);
        s = fmaf(qv[1], __uint_as_float(x.y), s);
        s = fmaf(qv[2], __uint_as_float(x.z), s);
        s = fmaf(qv[3], __uint_as_float(x.w), s);
      }
    }
    // NaN ranks as -inf so that (score, index) stays a total order and
    // exactly min(top_k, n_cand) blocks are chosen.
    score[l] = isnan(s) ? -INFINITY : s;
  }
  __syncthreads();

  // Rank: block l is chosen iff fewer than top_k blocks beat it (higher
  // score, or equal score and lower index), i.e. iff its position in the
  // order (score descending, index ascending) is below top_k.  A bitonic
  // sort of (score, index) over the next power of two gives the order
  // (padding: -inf at indices past the candidates, which sort last).
  const int nc = static_cast<int>(n_cand);
  int pn = 1;
  while (pn < nc) pn <<= 1;
  for (int e = threadIdx.x; e < pn; e += blockDim.x) {
    key[e] = e < nc ? score[e] : -INFINITY;
    idx[e] = e;
  }
  for (int e = threadIdx.x; e < nc; e += blockDim.x) flag[e] = 0;
  __syncthreads();
  for (int kk = 2; kk <= pn; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int e = threadIdx.x; e < pn; e += blockDim.x) {
        const int o = e ^ j;
        if (o > e) {
          const float ka = key[e], kb = key[o];
          const int ia = idx[e], ib = idx[o];
          const bool a_first = ka > kb || (ka == kb && ia < ib);
          if (((e & kk) == 0) != a_first) {  // this run is built in the other order
            key[e] = kb;
            key[o] = ka;
            idx[e] = ib;
            idx[o] = ia;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int e = threadIdx.x; e < a.top_k && e < nc; e += blockDim.x) flag[idx[e]] = 1;
  __syncthreads();

  // Compact the chosen indices in ascending order (one warp, ballots).
  if (warp == 0) {
    int32_t* out = a.sel + (static_cast<int64_t>(t) * a.Hkv + c) * a.top_k;
    int base = 0;
    for (int64_t l0 = 0; l0 < n_cand; l0 += 32) {
      const int64_t l = l0 + lane;
      const bool f = l < n_cand && flag[l];
      const unsigned m = __ballot_sync(0xffffffffu, f);
      const int slot = base + __popc(m & ((1u << lane) - 1u));
      if (f && slot < a.top_k &&
          MSA_IN_RANGE((static_cast<int64_t>(t) * a.Hkv + c) * a.top_k + slot, 1,
                       static_cast<int64_t>(gridDim.x) * a.Hkv * a.top_k, a.status))
        out[slot] = static_cast<int32_t>(l);
      base += __popc(m);
    }
    if (lane == 0 && MSA_IN_RANGE(static_cast<int64_t>(t) * a.Hkv + c, 1,
                                  static_cast<int64_t>(gridDim.x) * a.Hkv, a.status))
      a.cnt[static_cast<int64_t>(t) * a.Hkv + c] = min(base, a.top_k);
  }
}

}  // namespace

size_t block_select_smem(int d, int G) {
  const size_t P = static_cast<size_t>(sel_sort_size(G));
  return sizeof(float) * (static_cast<size_t>(d) + kSelThreads * 8 + G + P) +
         sizeof(int) * (static_cast<size_t>(G) + P);
}

cudaError_t launch_block_select(const SelectArgs& a, cudaStream_t s) {
  const size_t smem = block_select_smem(a.d, a.G);
  const int64_t n_qb = (a.n + kSelQBlock - 1) / kSelQBlock;
  dim3 grid(static_cast<unsigned>(n_qb), a.Hkv);
  if (a.bf16) {
    cudaError_t e = cudaFuncSetAttribute(block_select_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    block_select_kernel<true><<<grid, kSelThreads, smem, s>>>(a);
  } else {
    cudaError_t e = cudaFuncSetAttribute(block_select_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    block_select_kernel<false><<<grid, kSelThreads, smem, s>>>(a);
  }
  return cudaPeekAtLastError();
}

}  // namespace msa
