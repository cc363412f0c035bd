// Shared device/host helpers of libmsa (CUDA path only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

#ifdef MSA_DEBUG_BOUNDS
#include <stdio.h>
#endif

namespace msa {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Number of visible landmarks for global row `pos`: the count of blocks l
// with (l+1)*B <= pos - w + 1, i.e. clamp(floor((pos-w+1)/B), 0, G).
__host__ __device__ __forceinline__ int64_t visible_landmarks(int64_t pos, int64_t window,
                                                              int64_t block, int G) {
  if (G <= 0) return 0;
  int64_t x = pos - window + 1;
  if (x < block) return 0;
  int64_t c = x / block;
  return c < G ? c : G;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Range checks of the bounds-checked build.  Compiled with -DMSA_DEBUG_BOUNDS
// (libmsa_debug.so), MSA_IN_RANGE(off, count, extent, status) holds when the
// element (or byte) range [off, off + count) of a plain global access lies in
// [0, extent), the extent the entry point's contract gives that buffer; and
// MSA_TMA_OK(x, y, z, x_ext, y_ext, z_ext, box_z, status) holds when a 3-D
// TMA box origin has x (elements within a row, 16-bit data) 16-byte aligned
// and in [0, x_ext), y (head) in [0, y_ext), and its box_z rows overlapping
// [0, z_ext).  A failed check records MSA_ERR_INVALID_ARG in the status word,
// prints its site once, and the caller skips the access.  In the normal
// build both are the constant true and their arguments are not evaluated.
#ifdef MSA_DEBUG_BOUNDS
__device__ __noinline__ inline void range_fail(const char* file, int line, long long v,
                                               long long lo, long long hi, int* status) {
  if (status == nullptr || atomicCAS(status, 0, MSA_ERR_INVALID_ARG) == 0)
    printf("msa bounds check: %s:%d: %lld outside [%lld, %lld)\n", file, line, v, lo, hi);
}
__device__ __forceinline__ bool in_range(int64_t off, int64_t count, int64_t extent, int* status,
                                         const char* file, int line) {
  if (off >= 0 && count >= 0 && off + count <= extent) return true;
  range_fail(file, line, off < 0 ? off : off + count, 0, extent + 1, status);
  return false;
}
__device__ __forceinline__ bool tma_ok(int x, int y, int64_t z, int x_ext, int y_ext,
                                       int64_t z_ext, int box_z, int* status, const char* file,
                                       int line) {
  if (x % 8 != 0 || x < 0 || x >= x_ext) {
    range_fail(file, line, x, 0, x_ext, status);
    return false;
  }
  if (y < 0 || y >= y_ext) {
    range_fail(file, line, y, 0, y_ext, status);
    return false;
  }
  if (z <= -box_z || z >= z_ext) {
    range_fail(file, line, z, 1 - box_z, z_ext, status);
    return false;
  }
  return true;
}
#define MSA_IN_RANGE(off, count, extent, status) \
  (::msa::in_range((off), (count), (extent), (status), __FILE__, __LINE__))
#define MSA_TMA_OK(x, y, z, x_ext, y_ext, z_ext, box_z, status) \
  (::msa::tma_ok((x), (y), (z), (x_ext), (y_ext), (z_ext), (box_z), (status), __FILE__, __LINE__))
#else
#define MSA_IN_RANGE(off, count, extent, status) true
#define MSA_TMA_OK(x, y, z, x_ext, y_ext, z_ext, box_z, status) true
#endif

// Selection entries are device data the caller may have written: a count
// outside [0, min(top_k, candidates)] or a block index that is not a
// candidate of its query block is clamped into range (count) or replaced by
// block 0 (index) and MSA_ERR_INVALID_ARG recorded, so that no selection
// can make a kernel read outside K and V.
__device__ __forceinline__ int64_t sel_count_checked(int32_t cnt, int top_k, int64_t n_cand,
                                                     int* status) {
  const int64_t hi = min64(top_k, n_cand);
  if (cnt < 0 || cnt > hi) {
    record_status(status, MSA_ERR_INVALID_ARG);
    return cnt < 0 ? 0 : hi;
  }
  return cnt;
}
__device__ __forceinline__ int64_t sel_block_checked(int32_t blk, int64_t n_cand, int* status) {
  if (blk < 0 || blk >= n_cand) {
    record_status(status, MSA_ERR_INVALID_ARG);
    return 0;
  }
  return blk;
}

// Keys of row `pos` under the block-band mask: every key of the blocks
// (size bb) within hw blocks of the row's own, clipped to [0, n_kv).
__host__ __device__ __forceinline__ void band_keys(int64_t pos, int64_t bb, int64_t hw,
                                                   int64_t n_kv, int64_t* lo, int64_t* hi) {
  const int64_t b = pos / bb;
  *lo = max64(0, (b - hw) * bb);
  *hi = min64(n_kv - 1, (b + hw + 1) * bb - 1);
}

// Launch helpers implemented per translation unit; all return cudaError_t of
// the launch (cudaPeekAtLastError) and never synchronise.
struct PoolArgs {
  const void* k;
  const void* v;
  void* k_lm;
  void* v_lm;
  int64_t n;
  int C;  // Hkv * d elements per token
  int G;
  int bf16;
  int* status;  // device status word (range checks of the bounds-checked build)
};
cudaError_t launch_landmark_pool(const PoolArgs& a, cudaStream_t s);

struct MergeArgs {
  const float* o_parts[MSA_MAX_MERGE_PARTS];
  const float* lse_parts[MSA_MAX_MERGE_PARTS];
  int n_parts;
  void* out;
  float* lse;
  int64_t n;
  int Hq;
  int d;
  int out_bf16;
  int* status;  // device status word (range checks of the bounds-checked build)
};
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t s);

struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* k_lm;
  const void* v_lm;
  void* out;
  float* lse;
  int64_t lse_ld;  // row stride of lse [Hq][lse_ld] (0: n_q)
  int64_t n_q;
  int64_t q_start;
  int64_t n_kv;
  int64_t kv_start;
  int Hq;
  int Hkv;
  int d;
  int64_t window;
  int G;
  int64_t block;  // landmark block size B (1 when G == 0)
  float scale;
  int in_bf16;
  int out_bf16;
  int partial;  // rows with no key: lse = -inf, out row untouched
  int merge;    // out/lse hold a running result: merge this partial into it
  int band;     // block-band mask instead of window + landmarks
  int64_t band_block, band_half;
  // Top-k selected key blocks instead of landmarks: sel[t][c][0..cnt[t][c])
  // are the blocks (of `block` tokens) attended by query block t (128 rows)
  // of KV group c, in full, besides the window.
  const int32_t* sel;
  const int32_t* sel_cnt;
  int top_k;
  int* status;  // device status word
  uint64_t wait_limit_ns;
  int max_clusters;  // > 0: the CTA-pair kernel runs on at most this many pairs (test hook)
};
cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s);

// Query rows per selection block (one tensor-core work unit).
constexpr int kSelQBlock = 128;

struct SelectArgs {
  const void* q;
  const void* k_lm;
  int32_t* sel;   // [n_qb, Hkv, top_k]
  int32_t* cnt;   // [n_qb, Hkv]
  int64_t n;
  int Hq, Hkv, d;
  int64_t window;
  int G;
  int64_t block;  // tokens per key block (n / G)
  int top_k;
  int bf16;
  int* status;  // device status word (range checks of the bounds-checked build)
};
cudaError_t launch_block_select(const SelectArgs& a, cudaStream_t s);
size_t block_select_smem(int d, int G);

// Global query rows: each listed row attends every key j <= its position.
// Partials per (key split, KV head, M row m = r*g + hh) go to o_part
// [n_splits, Hkv, n_global*g, d] and lse_part [n_splits, Hkv, n_global*g]
// (fp32); the merge writes rows of out / lse.
struct GlobalRowsArgs {
  const void* q;
  const void* k;
  const void* v;
  const int64_t* rows;
  int64_t n_global;
  void* out;
  float* lse;
  float* o_part;
  float* lse_part;
  int64_t n;
  int Hq, Hkv, d;
  int64_t span;  // keys per split (multiple of 128)
  int n_splits;
  float scale;
  int in_bf16, out_bf16;
  int* status;
  uint64_t wait_limit_ns;
};
cudaError_t launch_global_rows(const GlobalRowsArgs& a, cudaStream_t s, const char** why);

// Backward pass (bf16, d = 128).  Workspace pieces: per-row statistics
// [2][Hq][n_pad] (lse in log2 units, then D; n_pad = n rounded up to 128,
// padding +inf / 0), landmark gradient partials [lm_chunks][2][G][Hkv][d]
// and their sums [2][G][Hkv][d] (fp32).
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* k_lm;
  const void* v_lm;
  const void* out;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* stats;
  float* lm_part;
  float* lm_grad;
  int64_t n, n_pad, window;
  int G, Hq, Hkv;
  float scale;
  int out_bf16, grad_bf16;
  int lm_chunks, chunk_tiles;
  int* status;
  uint64_t wait_limit_ns;
  // Global rows (compression-token pattern; null: none).  Mc = n_global *
  // (Hq / Hkv) gathered M rows, padded to Mp (a multiple of 128); Qg / dOg
  // [Mp][Hkv][d] bf16, gL2 / gD [Hkv][Mp], gpos [Mp]; dq_part
  // [n_splits][Hkv][Mp][d] and extra_k / extra_v [n][Hkv][d] fp32.
  const int64_t* rows;
  int64_t n_global, Mc, Mp, span;
  int n_splits;
  void* Qg;
  void* dOg;
  float* gL2;
  float* gD;
  int* gpos;
  float* dq_part;
  float* extra_k;
  float* extra_v;
  int no_pair;  // 1: the single-CTA dQ kernel even where the pair kernel applies
  int max_clusters;  // > 0: the dQ pair kernel runs on at most this many pairs (test hook)
};
bool attn_bwd_supported(int d, int in_bf16);
cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t s, const char** why);
// The CTA-pair dQ kernel (plain backward, an even number of query heads per
// KV head); launched by launch_attn_bwd.
bool bwd_dq_pair_supported(const BwdArgs& a);
cudaError_t launch_bwd_dq_pair(const BwdArgs& a, cudaStream_t s, const char** why);
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s, const char** why);
bool attn_tc_supported(int Hq, int Hkv, int d, int in_bf16);
// The CTA-pair variant (two SMs share each MMA; query heads per KV head >= 2).
cudaError_t launch_attn_tc2(const AttnArgs& a, cudaStream_t s, const char** why);
bool attn_tc2_supported(int Hq, int Hkv, int d, int in_bf16);

}  // namespace msa
