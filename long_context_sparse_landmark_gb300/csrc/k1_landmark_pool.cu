// K1: landmark pooling.  Landmark l of K (and of V) is the mean over the
// contiguous block of B = n/G tokens [lB, (l+1)B) -- the summary tokens of
// "Scaling GPU Cluster for Million Token Context", section "What is
// Flash-MSA Sparse Attention in GPU Clusters?", made concrete as block means.
//
// Memory-bound: every input byte is read once, the output is G/n of it.
// A token row holds C = Hkv*d contiguous elements, so block l is one
// contiguous [B, C] slab.  One CTA owns (tensor, landmark, 32-lane strip of
// the row); each lane loads 16 bytes per token with a read-only vector load,
// the CTA's warps split the B tokens, accumulate in fp32 registers, and
// reduce across warps in shared memory in a fixed order (deterministic).
#include "msa_common.cuh"

namespace msa {
namespace {

constexpr int kPoolWarps = 8;
constexpr int kPoolUnroll = 8;

template <bool kBf16>
struct Vec {
  static constexpr int N = kBf16 ? 8 : 4;  // elements per 16-byte load
};

template <bool kBf16>
__device__ __forceinline__ void accumulate(float (&acc)[Vec<kBf16>::N], const uint4& x) {
  if constexpr (kBf16) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += __uint_as_float(w[i] << 16);
      acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    acc[0] += __uint_as_float(x.x);
    acc[1] += __uint_as_float(x.y);
    acc[2] += __uint_as_float(x.z);
    acc[3] += __uint_as_float(x.w);
  }
}

template <bool kBf16>
__global__ void __launch_bounds__(kPoolWarps * 32)
    landmark_pool_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                         uint8_t* __restrict__ k_lm, uint8_t* __restrict__ v_lm, int64_t B,
                         int C, int strips, int64_t n, int* status) {
  constexpr int VN = Vec<kBf16>::N;
  constexpr int ES = kBf16 ? 2 : 4;
  __shared__ float red[kPoolWarps][32][VN + 1];

  const int strip = blockIdx.x % strips;
  const int64_t l = blockIdx.x / strips;
  const int tensor = blockIdx.y;  // 0 = K, 1 = V
  const uint8_t* src = tensor == 0 ? k : v;
  uint8_t* dst = tensor == 0 ? k_lm : v_lm;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int col = (strip * 32 + lane) * VN;  // first element of this lane
  const bool active = col < C;               // C % VN == 0 is guaranteed

  float acc[VN];
#pragma unroll
  for (int e = 0; e < VN; ++e) acc[e] = 0.f;

  if (active) {
    const int64_t row_bytes = static_cast<int64_t>(C) * ES;
    const uint8_t* base = src + (l * B) * row_bytes + static_cast<int64_t>(col) * ES;
    for (int64_t r0 = warp; r0 < B; r0 += kPoolWarps * kPoolUnroll) {
      uint4 buf[kPoolUnroll];
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) {
        const int64_t r = r0 + static_cast<int64_t>(u) * kPoolWarps;
        buf[u] = r < B && MSA_IN_RANGE((l * B + r) * row_bytes + static_cast<int64_t>(col) * ES,
                                       16, n * row_bytes, status)
                     ? __ldg(reinterpret_cast<const uint4*>(base + r * row_bytes))
                     : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kPoolUnroll; ++u) accumulate<kBf16>(acc, buf[u]);
    }
  }
#pragma unroll
  for (int e = 0; e < VN; ++e) red[warp][lane][e] = acc[e];
  __syncthreads();
  if (warp == 0 && active) {
    float s[VN];
#pragma unroll
    for (int e = 0; e < VN; ++e) s[e] = 0.f;
    for (int w = 0; w < kPoolWarps; ++w) {
#pragma unroll
      for (int e = 0; e < VN; ++e) s[e] += red[w][lane][e];
    }
    const float fb = static_cast<float>(B);
    uint8_t* out = dst + (l * C + col) * ES;
    if (!MSA_IN_RANGE((l * C + col) * ES, 16,
                      static_cast<int64_t>(gridDim.x / strips) * C * ES, status))
      return;
    if constexpr (kBf16) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(__fdiv_rn(s[2 * i], fb),
                                                 __fdiv_rn(s[2 * i + 1], fb));
        w[i] = *reinterpret_cast<uint32_t*>(&p);
      }
      *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      float4 o = make_float4(__fdiv_rn(s[0], fb), __fdiv_rn(s[1], fb), __fdiv_rn(s[2], fb),
                             __fdiv_rn(s[3], fb));
      *reinterpret_cast<float4*>(out) = o;
    }
  }
}

}  // namespace

cudaError_t launch_landmark_pool(const PoolArgs& a, cudaStream_t s) {
  const int vn = a.bf16 ? 8 : 4;
  const int strips = (a.C / vn + 31) / 32;
  const int64_t B = a.n / a.G;
  dim3 grid(static_cast<unsigned>(static_cast<int64_t>(a.G) * strips), a.v ? 2 : 1);
  dim3 block(kPoolWarps * 32);
  if (a.bf16) {
    landmark_pool_kernel<true><<<grid, block, 0, s>>>(
        static_cast<const uint8_t*>(a.k), static_cast<const uint8_t*>(a.v),
        static_cast<uint8_t*>(a.k_lm), static_cast<uint8_t*>(a.v_lm), B, a.C, strips, a.n,
        a.status);
  } else {
    landmark_pool_kernel<false><<<grid, block, 0, s>>>(
        static_cast<const uint8_t*>(a.k), static_cast<const uint8_t*>(a.v),
        static_cast<uint8_t*>(a.k_lm), static_cast<uint8_t*>(a.v_lm), B, a.C, strips, a.n,
        a.status);
  }
  return cudaPeekAtLastError();
}

}  // namespace msa
