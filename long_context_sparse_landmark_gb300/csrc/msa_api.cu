// C ABI of libmsa: argument validation, kernel selection and launch.
// Every entry point validates all arguments before enqueueing anything and
// never allocates or synchronises (msa_device_status excepted, which reads
// the status word and says so).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <string>

#include "msa_common.cuh"

#include <nvtx3/nvToolsExt.h>

// Every entry point opens an NVTX range named after itself for the
// duration of the call (host side: argument checks and launches), so that
// profiler timelines group each call's kernels; without a tool attached the
// push and pop cost nanoseconds.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
#define MSA_NVTX_RANGE() NvtxRange msa_nvtx_range_(__func__)

namespace {

thread_local std::string g_last_error;

msa_status fail(msa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

msa_status ok() {
  g_last_error.clear();
  return MSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(msa_dtype d) { return d == MSA_F32 || d == MSA_BF16; }

// Per-device status word written by kernels when a bounded wait runs out.
__device__ int g_device_status;

std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<int> g_force_single_cta{0};
std::atomic<int> g_max_clusters_cap{0};
constexpr uint64_t kDefaultWaitNs = 4000000000ull;

// Address of the status word in the current context, looked up on every
// call: a cached address would dangle after cudaDeviceReset.
msa_status device_status_ptr(int** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_device_status);
  if (e != cudaSuccess)
    return fail(MSA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  *out = static_cast<int*>(p);
  return MSA_OK;
}

// The status word for launches that only record range-check failures of
// the bounds-checked build (null if the lookup fails: those checks then
// only print).
int* status_word() {
  int* p = nullptr;
  return device_status_ptr(&p) == MSA_OK ? p : nullptr;
}

msa_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return ok();
}

// lse_align: alignment the lse pointer needs (16, or 4 where it may point
// into the middle of an [Hq, n] array).
msa_status check_attn_common(const void* q, const void* k, const void* v, const void* out,
                             const float* lse, int Hq, int Hkv, int d, int64_t window,
                             float scale, msa_dtype in_dt, uintptr_t lse_align = 16) {
  if (!q || !k || !v || !out || !lse) return fail(MSA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(lse) & (lse_align - 1)) != 0)
    return fail(MSA_ERR_INVALID_ARG, "tensor pointer not 16-byte aligned (lse: %u)",
                static_cast<unsigned>(lse_align));
  if (Hq < 1 || Hkv < 1) return fail(MSA_ERR_INVALID_ARG, "Hq=%d Hkv=%d must be >= 1", Hq, Hkv);
  if (Hq % Hkv != 0) return fail(MSA_ERR_INVALID_ARG, "Hq=%d not a multiple of Hkv=%d", Hq, Hkv);
  if (window < 1) return fail(MSA_ERR_INVALID_ARG, "window=%lld must be >= 1", (long long)window);
  if (!(scale > 0.f) || !isfinite(scale))
    return fail(MSA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!valid_dtype(in_dt)) return fail(MSA_ERR_INVALID_ARG, "bad input dtype %d", (int)in_dt);
  if (d != 64 && d != 128) return fail(MSA_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
  return MSA_OK;
}

constexpr int64_t kMaxRows = (int64_t(1) << 31) - 256;  // TMA coordinates are 32-bit

msa_status run_attn(const msa::AttnArgs& a0, cudaStream_t stream) {
  msa::AttnArgs a = a0;
  if (a.lse_ld == 0) a.lse_ld = a.n_q;
  msa_status st = device_status_ptr(&a.status);
  if (st != MSA_OK) return st;
  const uint64_t lim = g_wait_limit_ns.load();
  a.wait_limit_ns = lim ? lim : kDefaultWaitNs;
  a.max_clusters = g_max_clusters_cap.load();
  // Selected blocks map to whole 128-key tiles on the tensor-core path.
  const bool tiles_ok = !a.sel || a.block % 128 == 0;
  // The CTA-pair kernel keeps per-row column bounds in 32 bits: up to 2^29
  // keys (longer sequences take the single-CTA kernel).
  const bool pair_sizes = a.n_kv <= (int64_t(1) << 29) && a.n_q <= (int64_t(1) << 29);
  if (tiles_ok && pair_sizes && !g_force_single_cta.load() &&
      msa::attn_tc2_supported(a.Hq, a.Hkv, a.d, a.in_bf16)) {
    const char* why = nullptr;
    cudaError_t e = msa::launch_attn_tc2(a, stream, &why);
    if (e != cudaSuccess && why) return fail(MSA_ERR_CUDA, "tensor-core attention: %s", why);
    return launched(e, "tensor-core attention (CTA pairs)");
  }
  if (tiles_ok && msa::attn_tc_supported(a.Hq, a.Hkv, a.d, a.in_bf16)) {
    const char* why = nullptr;
    cudaError_t e = msa::launch_attn_tc(a, stream, &why);
    if (e != cudaSuccess && why) return fail(MSA_ERR_CUDA, "tensor-core attention: %s", why);
    return launched(e, "tensor-core attention");
  }
  return launched(msa::launch_attn_simt(a, stream), "attention");
}

// Pool the block-mean keys, select each query block's top-k key blocks,
// attend window + selected blocks: three launches on `stream`.
msa_status topk_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                        int64_t n, int Hq, int Hkv, int d, int64_t window, int G, int top_k,
                        float scale, msa_dtype in_dt, msa_dtype out_dt, void* k_lm, int32_t* sel,
                        int32_t* cnt, cudaStream_t stream) {
  msa::PoolArgs pa{k, nullptr, k_lm, nullptr, n, Hkv * d, G, in_dt == MSA_BF16 ? 1 : 0,
                   status_word()};
  msa_status st = launched(msa::launch_landmark_pool(pa, stream), "landmark pool");
  if (st != MSA_OK) return st;
  msa::SelectArgs sa{q, k_lm, sel, cnt, n, Hq, Hkv, d, window, G, n / G, top_k,
                     in_dt == MSA_BF16 ? 1 : 0, status_word()};
  st = launched(msa::launch_block_select(sa, stream), "block select");
  if (st != MSA_OK) return st;
  msa::AttnArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.n_q = n;
  a.n_kv = n;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = window;
  a.G = G;
  a.block = n / G;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = out_dt == MSA_BF16;
  a.sel = sel;
  a.sel_cnt = cnt;
  a.top_k = top_k;
  return run_attn(a, stream);
}

}  // namespace

// Fixed per-device scratch of msa_attn_fwd_topk_noalloc: the block-mean
// keys, the selection and its counts of one call, laid out as the caller
// workspace of msa_attn_fwd_topk.  Nothing in it needs to start at zero:
// every launch writes each byte it later reads (all block-mean keys, every
// count, and the chosen indices below each count) before reading it.
static __device__ __align__(256) uint8_t g_topk_scratch[MSA_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch on the current device, looked up on every
// call (a table lookup once the module is loaded): an address kept from an
// earlier call would dangle after cudaDeviceReset or in another context.
msa_status topk_scratch_ptr(uint8_t** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_topk_scratch);
  if (e != cudaSuccess)
    return fail(MSA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  *out = static_cast<uint8_t*>(p);
  return MSA_OK;
}

}  // namespace

extern "C" {

int msa_version(void) { return 100; }

int msa_debug_bounds_build(void) {
#ifdef MSA_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

const char* msa_last_error_string(void) { return g_last_error.c_str(); }

msa_status msa_landmark_pool(const void* k, const void* v, void* k_lm, void* v_lm, int64_t n,
                             int Hkv, int d, int n_landmarks, msa_dtype dt, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  if (!k || !v || !k_lm || !v_lm) return fail(MSA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_lm) || !aligned16(v_lm))
    return fail(MSA_ERR_INVALID_ARG, "tensor pointer not 16-byte aligned");
  if (n < 1 || Hkv < 1) return fail(MSA_ERR_INVALID_ARG, "n=%lld Hkv=%d", (long long)n, Hkv);
  if (n_landmarks < 1 || n_landmarks > n || n % n_landmarks != 0)
    return fail(MSA_ERR_INVALID_ARG, "G=%d must satisfy 1 <= G <= n and n %% G == 0 (n=%lld)",
                n_landmarks, (long long)n);
  if (!valid_dtype(dt)) return fail(MSA_ERR_INVALID_ARG, "bad dtype %d", (int)dt);
  if (d != 64 && d != 128) return fail(MSA_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
  msa::PoolArgs a{k, v, k_lm, v_lm, n, Hkv * d, n_landmarks, dt == MSA_BF16 ? 1 : 0,
                  status_word()};
  return launched(msa::launch_landmark_pool(a, reinterpret_cast<cudaStream_t>(stream)),
                  "landmark pool");
}

msa_status msa_attn_fwd(const void* q, const void* k, const void* v, const void* k_lm,
                        const void* v_lm, void* out, float* lse, int64_t n, int Hq, int Hkv, int d,
                        int64_t window, int n_landmarks, float scale, msa_dtype in_dt,
                        msa_dtype out_dt, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  if (n_landmarks < 0 || n_landmarks > n || (n_landmarks > 0 && n % n_landmarks != 0))
    return fail(MSA_ERR_INVALID_ARG, "G=%d must satisfy 0 <= G <= n and n %% G == 0 (n=%lld)",
                n_landmarks, (long long)n);
  if (n_landmarks > 0) {
    if (!k_lm || !v_lm) return fail(MSA_ERR_INVALID_ARG, "null landmark pointer with G > 0");
    if (!aligned16(k_lm) || !aligned16(v_lm))
      return fail(MSA_ERR_INVALID_ARG, "landmark pointer not 16-byte aligned");
  }
  msa::AttnArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.k_lm = n_landmarks > 0 ? k_lm : nullptr;
  a.v_lm = n_landmarks > 0 ? v_lm : nullptr;
  a.out = out;
  a.lse = lse;
  a.n_q = n;
  a.q_start = 0;
  a.n_kv = n;
  a.kv_start = 0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = window;
  a.G = n_landmarks;
  a.block = n_landmarks > 0 ? n / n_landmarks : 1;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = out_dt == MSA_BF16;
  a.partial = 0;
  return run_attn(a, reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_attn_fwd_rows(const void* q_rows, const void* k, const void* v, const void* k_lm,
                             const void* v_lm, void* out_rows, float* lse, int64_t lse_ld,
                             int64_t q_start, int64_t n_q, int64_t n, int Hq, int Hkv, int d,
                             int64_t window, int n_landmarks, float scale, msa_dtype in_dt,
                             msa_dtype out_dt, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q_rows, k, v, out_rows, lse, Hq, Hkv, d, window, scale,
                                    in_dt, 4);
  if (st != MSA_OK) return st;
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (n_q < 1 || q_start < 0 || q_start + n_q > n)
    return fail(MSA_ERR_INVALID_ARG, "rows [%lld, %lld) not inside [0, n=%lld)",
                (long long)q_start, (long long)(q_start + n_q), (long long)n);
  if (lse_ld < n_q) return fail(MSA_ERR_INVALID_ARG, "lse_ld=%lld below n_q", (long long)lse_ld);
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  if (n_landmarks < 0 || n_landmarks > n || (n_landmarks > 0 && n % n_landmarks != 0))
    return fail(MSA_ERR_INVALID_ARG, "G=%d must satisfy 0 <= G <= n and n %% G == 0 (n=%lld)",
                n_landmarks, (long long)n);
  if (n_landmarks > 0) {
    if (!k_lm || !v_lm) return fail(MSA_ERR_INVALID_ARG, "null landmark pointer with G > 0");
    if (!aligned16(k_lm) || !aligned16(v_lm))
      return fail(MSA_ERR_INVALID_ARG, "landmark pointer not 16-byte aligned");
  }
  msa::AttnArgs a{};
  a.q = q_rows;
  a.k = k;
  a.v = v;
  a.k_lm = n_landmarks > 0 ? k_lm : nullptr;
  a.v_lm = n_landmarks > 0 ? v_lm : nullptr;
  a.out = out_rows;
  a.lse = lse;
  a.lse_ld = lse_ld;
  a.n_q = n_q;
  a.q_start = q_start;
  a.n_kv = n;
  a.kv_start = 0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = window;
  a.G = n_landmarks;
  a.block = n_landmarks > 0 ? n / n_landmarks : 1;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = out_dt == MSA_BF16;
  return run_attn(a, reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_attn_fwd_band(const void* q, const void* k, const void* v, void* out, float* lse,
                             int64_t n, int Hq, int Hkv, int d, int64_t band_block,
                             int64_t band_half, float scale, msa_dtype in_dt, msa_dtype out_dt,
                             msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, 1, scale, in_dt);
  if (st != MSA_OK) return st;
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  if (band_block < 1 || band_half < 0)
    return fail(MSA_ERR_INVALID_ARG, "band_block=%lld must be >= 1 and band_half=%lld >= 0",
                (long long)band_block, (long long)band_half);
  msa::AttnArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.n_q = n;
  a.q_start = 0;
  a.n_kv = n;
  a.kv_start = 0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = 1;
  a.G = 0;
  a.block = 1;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = out_dt == MSA_BF16;
  a.band = 1;
  a.band_block = band_block;
  a.band_half = band_half;
  return run_attn(a, reinterpret_cast<cudaStream_t>(stream));
}

// Shared checks of the top-k entry points.
static msa_status check_topk(int64_t n, int G, int top_k) {
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (G < 1 || G > n || n % G != 0)
    return fail(MSA_ERR_INVALID_ARG, "G=%d must satisfy 1 <= G <= n and n %% G == 0", G);
  if (G > MSA_MAX_SELECT_BLOCKS)
    return fail(MSA_ERR_UNSUPPORTED, "G=%d key blocks (at most %d)", G, MSA_MAX_SELECT_BLOCKS);
  if (top_k < 1 || top_k > G) return fail(MSA_ERR_INVALID_ARG, "top_k=%d must be in [1, G]", top_k);
  return MSA_OK;
}

msa_status msa_block_select(const void* q, const void* k_lm, int32_t* sel, int32_t* cnt, int64_t n,
                            int Hq, int Hkv, int d, int64_t window, int n_landmarks, int top_k,
                            msa_dtype in_dt, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  if (!q || !k_lm || !sel || !cnt) return fail(MSA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k_lm) || !aligned16(sel) || !aligned16(cnt))
    return fail(MSA_ERR_INVALID_ARG, "tensor pointer not 16-byte aligned");
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(MSA_ERR_INVALID_ARG, "Hq=%d Hkv=%d", Hq, Hkv);
  if (window < 1) return fail(MSA_ERR_INVALID_ARG, "window must be >= 1");
  if (!valid_dtype(in_dt)) return fail(MSA_ERR_INVALID_ARG, "bad input dtype %d", (int)in_dt);
  if (d != 64 && d != 128) return fail(MSA_ERR_UNSUPPORTED, "head dim d=%d (supported: 64, 128)", d);
  msa_status st = check_topk(n, n_landmarks, top_k);
  if (st != MSA_OK) return st;
  msa::SelectArgs a{q, k_lm, sel, cnt, n, Hq, Hkv, d, window, n_landmarks, n / n_landmarks, top_k,
                    in_dt == MSA_BF16 ? 1 : 0, status_word()};
  return launched(msa::launch_block_select(a, reinterpret_cast<cudaStream_t>(stream)),
                  "block select");
}

msa_status msa_attn_fwd_select(const void* q, const void* k, const void* v, const int32_t* sel,
                               const int32_t* cnt, void* out, float* lse, int64_t n, int Hq,
                               int Hkv, int d, int64_t window, int n_landmarks, int top_k,
                               float scale, msa_dtype in_dt, msa_dtype out_dt,
                               msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (!sel || !cnt) return fail(MSA_ERR_INVALID_ARG, "null selection pointer");
  if (!aligned16(sel) || !aligned16(cnt))
    return fail(MSA_ERR_INVALID_ARG, "selection pointer not 16-byte aligned");
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  st = check_topk(n, n_landmarks, top_k);
  if (st != MSA_OK) return st;
  msa::AttnArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.n_q = n;
  a.n_kv = n;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = window;
  a.G = n_landmarks;
  a.block = n / n_landmarks;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = out_dt == MSA_BF16;
  a.sel = sel;
  a.sel_cnt = cnt;
  a.top_k = top_k;
  return run_attn(a, reinterpret_cast<cudaStream_t>(stream));
}

// Workspace layout of msa_attn_fwd_topk: block-mean keys, then the
// selection indices, then the counts, each 256-byte aligned.
struct TopkLayout {
  size_t k_lm, sel, cnt, total;
};

static TopkLayout topk_layout(int64_t n, int Hkv, int d, int G, int top_k, msa_dtype in_dt) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t es = in_dt == MSA_BF16 ? 2 : 4;
  const size_t n_qb = static_cast<size_t>((n + msa::kSelQBlock - 1) / msa::kSelQBlock);
  TopkLayout L;
  L.k_lm = 0;
  L.sel = up(static_cast<size_t>(G) * Hkv * d * es);
  L.cnt = L.sel + up(n_qb * Hkv * top_k * sizeof(int32_t));
  L.total = L.cnt + up(n_qb * Hkv * sizeof(int32_t));
  return L;
}

size_t msa_attn_fwd_topk_workspace_size(int64_t n, int Hkv, int d, int n_landmarks, int top_k,
                                        msa_dtype in_dt) {
  if (Hkv < 1 || d < 1 || !valid_dtype(in_dt) || check_topk(n, n_landmarks, top_k) != MSA_OK)
    return 0;
  return topk_layout(n, Hkv, d, n_landmarks, top_k, in_dt).total;
}

msa_status msa_attn_fwd_topk(const void* q, const void* k, const void* v, void* out, float* lse,
                             int64_t n, int Hq, int Hkv, int d, int64_t window, int n_landmarks,
                             int top_k, float scale, msa_dtype in_dt, msa_dtype out_dt,
                             void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  st = check_topk(n, n_landmarks, top_k);
  if (st != MSA_OK) return st;
  const TopkLayout L = topk_layout(n, Hkv, d, n_landmarks, top_k, in_dt);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MSA_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (workspace_bytes < L.total)
    return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                L.total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return topk_forward(q, k, v, out, lse, n, Hq, Hkv, d, window, n_landmarks, top_k, scale, in_dt,
                      out_dt, ws + L.k_lm, reinterpret_cast<int32_t*>(ws + L.sel),
                      reinterpret_cast<int32_t*>(ws + L.cnt),
                      reinterpret_cast<cudaStream_t>(stream));
}

// The top-k path for callers that cannot allocate device memory: a plain C
// host program that links only this library and holds no allocator of its
// own, or a runtime that must not call cudaMalloc between launches because
// it can synchronise the whole device and stall its other streams.  Same
// kernels and launches as msa_attn_fwd_topk; the intermediates go to the
// fixed scratch above instead of a caller workspace.
msa_status msa_attn_fwd_topk_noalloc(const void* q, const void* k, const void* v, void* out,
                                     float* lse, int64_t n, int Hq, int Hkv, int d,
                                     int64_t window, int n_landmarks, int top_k, float scale,
                                     msa_dtype in_dt, msa_dtype out_dt, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  st = check_topk(n, n_landmarks, top_k);
  if (st != MSA_OK) return st;
  const TopkLayout L = topk_layout(n, Hkv, d, n_landmarks, top_k, in_dt);
  if (L.total > static_cast<size_t>(MSA_NOALLOC_SCRATCH_BYTES))
    return fail(MSA_ERR_UNSUPPORTED,
                "these sizes need %zu bytes of scratch; the fixed scratch holds %zu "
                "(use msa_attn_fwd_topk with a workspace)",
                L.total, static_cast<size_t>(MSA_NOALLOC_SCRATCH_BYTES));
  uint8_t* ws = nullptr;
  st = topk_scratch_ptr(&ws);
  if (st != MSA_OK) return st;
  return topk_forward(q, k, v, out, lse, n, Hq, Hkv, d, window, n_landmarks, top_k, scale, in_dt,
                      out_dt, ws + L.k_lm, reinterpret_cast<int32_t*>(ws + L.sel),
                      reinterpret_cast<int32_t*>(ws + L.cnt),
                      reinterpret_cast<cudaStream_t>(stream));
}

// Key splits and workspace layout of msa_attn_fwd_global_rows: about 152
// (split, M tile, KV head) CTAs -- one wave on GB300's 152 SMs; more,
// shorter splits pay each CTA's set-up more often (measured at 128K with
// 16 global rows: 1024 CTAs 0.239 ms, 512 0.192, 304 0.149, 152 0.129) --
// splits of whole 128-key tiles; partial O, then partial lse, 256-byte
// aligned.
struct GrPlan {
  int64_t Mc, span;
  int n_splits;
  size_t lse_off, total;
};

static GrPlan gr_plan(int64_t n, int64_t n_global, int Hq, int Hkv, int d) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  GrPlan P{};
  P.Mc = n_global * (Hq / Hkv);
  const int64_t mtiles = (P.Mc + 127) / 128;
  const int64_t tiles = (n + 127) / 128;
  const int64_t per_split = mtiles * Hkv;
  int64_t S = (152 + per_split - 1) / per_split;
  S = S < 1 ? 1 : (S > tiles ? tiles : S);
  const int64_t span_tiles = (tiles + S - 1) / S;
  P.span = span_tiles * 128;
  P.n_splits = static_cast<int>((tiles + span_tiles - 1) / span_tiles);
  const size_t slabs = static_cast<size_t>(P.n_splits) * Hkv * static_cast<size_t>(P.Mc);
  P.lse_off = up(slabs * d * sizeof(float));
  P.total = P.lse_off + up(slabs * sizeof(float));
  return P;
}

// Largest n_global * (Hq / Hkv) the launch grids accept.
constexpr int64_t kMaxGlobalM = int64_t(4) * 65535;

static msa_status check_global_rows(int64_t n, int64_t n_global, int Hq, int Hkv) {
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (n_global < 1 || n_global > n)
    return fail(MSA_ERR_INVALID_ARG, "n_global=%lld must be in [1, n]", (long long)n_global);
  if (n_global * (Hq / Hkv) > kMaxGlobalM)
    return fail(MSA_ERR_UNSUPPORTED, "n_global * Hq / Hkv = %lld above %lld",
                (long long)(n_global * (Hq / Hkv)), (long long)kMaxGlobalM);
  return MSA_OK;
}

size_t msa_attn_fwd_global_rows_workspace_size(int64_t n, int64_t n_global, int Hq, int Hkv,
                                               int d) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (d != 64 && d != 128) ||
      check_global_rows(n, n_global, Hq, Hkv) != MSA_OK)
    return 0;
  return gr_plan(n, n_global, Hq, Hkv, d).total;
}

msa_status msa_attn_fwd_global_rows(const void* q, const void* k, const void* v,
                                    const int64_t* rows, int64_t n_global, void* out, float* lse,
                                    int64_t n, int Hq, int Hkv, int d, float scale,
                                    msa_dtype in_dt, msa_dtype out_dt, void* workspace,
                                    size_t workspace_bytes, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, 1, scale, in_dt);
  if (st != MSA_OK) return st;
  if (!rows || (reinterpret_cast<uintptr_t>(rows) & 7u) != 0)
    return fail(MSA_ERR_INVALID_ARG, "rows must be non-null and 8-byte aligned");
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  st = check_global_rows(n, n_global, Hq, Hkv);
  if (st != MSA_OK) return st;
  const GrPlan P = gr_plan(n, n_global, Hq, Hkv, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MSA_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (workspace_bytes < P.total)
    return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                P.total);
  msa::GlobalRowsArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.rows = rows;
  a.n_global = n_global;
  a.out = out;
  a.lse = lse;
  a.o_part = static_cast<float*>(workspace);
  a.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + P.lse_off);
  a.n = n;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.span = P.span;
  a.n_splits = P.n_splits;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = out_dt == MSA_BF16;
  st = device_status_ptr(&a.status);
  if (st != MSA_OK) return st;
  const uint64_t lim = g_wait_limit_ns.load();
  a.wait_limit_ns = lim ? lim : kDefaultWaitNs;
  const char* why = nullptr;
  cudaError_t e = msa::launch_global_rows(a, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && why) return fail(MSA_ERR_CUDA, "global rows: %s", why);
  return launched(e, "global rows");
}

// Workspace layout of msa_attn_bwd: row statistics [2][Hq][n rounded up to
// 128] (lse in log2 units, D), landmark gradient partials
// [chunks][2][G][Hkv][d] and their sums [2][G][Hkv][d] (fp32, 256-byte
// aligned).  Landmark work is split over query chunks so that
// (landmark tile, KV head, chunk) CTAs fill the GPU.
struct BwdPlan {
  int lm_chunks, chunk_tiles;
  size_t part_off, grad_off, total;
};

static BwdPlan bwd_plan(int64_t n, int Hq, int Hkv, int d, int G) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  BwdPlan P{};
  const int64_t n_qt = (n + 127) / 128;
  if (G > 0) {
    // Landmark-mode grid: (landmark tile, KV head, query chunk).  Landmark
    // tile l is seen only by the rows past its blocks, so about half of the
    // CTAs find work; 2048 / per chunks make that several waves of the SMs
    // (a ~256 MB partial buffer whatever G is).
    const int64_t per = ((G + 127) / 128) * static_cast<int64_t>(Hkv);
    int64_t ch = (2048 + per - 1) / per;
    ch = ch < 1 ? 1 : (ch > n_qt ? n_qt : ch);
    P.chunk_tiles = static_cast<int>((n_qt + ch - 1) / ch);
    P.lm_chunks = static_cast<int>((n_qt + P.chunk_tiles - 1) / P.chunk_tiles);
  }
  const size_t lm = 2 * static_cast<size_t>(G) * Hkv * d * sizeof(float);
  P.part_off = up(2 * static_cast<size_t>(Hq) * n_qt * 128 * sizeof(float));
  P.grad_off = P.part_off + up(static_cast<size_t>(P.lm_chunks) * lm);
  P.total = P.grad_off + up(lm);
  return P;
}

static msa_status check_bwd_sizes(int64_t n, int Hq, int Hkv, int d, int G) {
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(MSA_ERR_INVALID_ARG, "Hq=%d Hkv=%d", Hq, Hkv);
  if (G < 0 || G > n || (G > 0 && n % G != 0))
    return fail(MSA_ERR_INVALID_ARG, "G=%d must satisfy 0 <= G <= n and n %% G == 0 (n=%lld)", G,
                (long long)n);
  if (d != 128) return fail(MSA_ERR_UNSUPPORTED, "backward: head dim d=%d (supported: 128)", d);
  return MSA_OK;
}

// Extra workspace of msa_attn_bwd_global_rows after the msa_attn_bwd part:
// gathered Qg / dOg, their statistics and positions, the per-split dQ
// shares and the global rows' dK / dV; key splits as for the forward's
// global rows (about one wave of CTAs).
struct BwdGrPlan {
  int64_t Mc, Mp, span;
  int n_splits;
  size_t qg, dog, gl2, gd, gpos, dq_part, extra_k, extra_v, total;
};

static BwdGrPlan bwd_gr_plan(size_t base, int64_t n, int64_t n_global, int Hq, int Hkv, int d) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  BwdGrPlan P{};
  P.Mc = n_global * (Hq / Hkv);
  P.Mp = (P.Mc + 127) / 128 * 128;
  const int64_t tiles = (n + 127) / 128;
  const int64_t per_split = (P.Mp / 128) * Hkv;
  int64_t S = (152 + per_split - 1) / per_split;
  S = S < 1 ? 1 : (S > tiles ? tiles : S);
  const int64_t span_tiles = (tiles + S - 1) / S;
  P.span = span_tiles * 128;
  P.n_splits = static_cast<int>((tiles + span_tiles - 1) / span_tiles);
  const size_t rows_bytes = static_cast<size_t>(P.Mp) * Hkv * d * 2;
  size_t at = up(base);
  P.qg = at;
  at += up(rows_bytes);
  P.dog = at;
  at += up(rows_bytes);
  P.gl2 = at;
  at += up(static_cast<size_t>(Hkv) * P.Mp * 4);
  P.gd = at;
  at += up(static_cast<size_t>(Hkv) * P.Mp * 4);
  P.gpos = at;
  at += up(static_cast<size_t>(P.Mp) * 4);
  P.dq_part = at;
  at += up(static_cast<size_t>(P.n_splits) * Hkv * P.Mp * d * 4);
  P.extra_k = at;
  at += up(static_cast<size_t>(n) * Hkv * d * 4);
  P.extra_v = at;
  at += up(static_cast<size_t>(n) * Hkv * d * 4);
  P.total = at;
  return P;
}

size_t msa_attn_bwd_workspace_size(int64_t n, int Hq, int Hkv, int d, int n_landmarks) {
  if (check_bwd_sizes(n, Hq, Hkv, d, n_landmarks) != MSA_OK) return 0;
  return bwd_plan(n, Hq, Hkv, d, n_landmarks).total;
}

static msa_status attn_bwd_impl(const void* q, const void* k, const void* v, const void* k_lm,
                                const void* v_lm, const void* out, const float* lse,
                                const void* dout, const int64_t* rows, int64_t n_global, void* dq,
                                void* dk, void* dv, int64_t n, int Hq, int Hkv, int d,
                                int64_t window, int n_landmarks, float scale, msa_dtype in_dt,
                                msa_dtype out_dt, msa_dtype grad_dt, void* workspace,
                                size_t workspace_bytes, msa_stream_t stream) {
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (!dout || !dq || !dk || !dv) return fail(MSA_ERR_INVALID_ARG, "null gradient pointer");
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(MSA_ERR_INVALID_ARG, "gradient pointer not 16-byte aligned");
  if (!valid_dtype(out_dt) || !valid_dtype(grad_dt))
    return fail(MSA_ERR_INVALID_ARG, "bad output/gradient dtype %d/%d", (int)out_dt, (int)grad_dt);
  st = check_bwd_sizes(n, Hq, Hkv, d, n_landmarks);
  if (st != MSA_OK) return st;
  if (in_dt != MSA_BF16)
    return fail(MSA_ERR_UNSUPPORTED, "backward: inputs must be bf16 (tensor-core kernels)");
  if (n_landmarks > 0) {
    if (!k_lm || !v_lm) return fail(MSA_ERR_INVALID_ARG, "null landmark pointer with G > 0");
    if (!aligned16(k_lm) || !aligned16(v_lm))
      return fail(MSA_ERR_INVALID_ARG, "landmark pointer not 16-byte aligned");
  }
  if (rows) {
    if ((reinterpret_cast<uintptr_t>(rows) & 7u) != 0)
      return fail(MSA_ERR_INVALID_ARG, "rows must be 8-byte aligned");
    st = check_global_rows(n, n_global, Hq, Hkv);
    if (st != MSA_OK) return st;
  }
  const BwdPlan P = bwd_plan(n, Hq, Hkv, d, n_landmarks);
  const BwdGrPlan R = rows ? bwd_gr_plan(P.total, n, n_global, Hq, Hkv, d) : BwdGrPlan{};
  const size_t need = rows ? R.total : P.total;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MSA_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (workspace_bytes < need)
    return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  msa::BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.k_lm = n_landmarks > 0 ? k_lm : nullptr;
  a.v_lm = n_landmarks > 0 ? v_lm : nullptr;
  a.out = out;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.stats = reinterpret_cast<float*>(ws);
  a.lm_part = reinterpret_cast<float*>(ws + P.part_off);
  a.lm_grad = reinterpret_cast<float*>(ws + P.grad_off);
  a.n = n;
  a.n_pad = (n + 127) / 128 * 128;
  a.window = window;
  a.G = n_landmarks;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.scale = scale;
  a.out_bf16 = out_dt == MSA_BF16;
  a.grad_bf16 = grad_dt == MSA_BF16;
  a.lm_chunks = P.lm_chunks;
  a.chunk_tiles = P.chunk_tiles;
  if (rows) {
    a.rows = rows;
    a.n_global = n_global;
    a.Mc = R.Mc;
    a.Mp = R.Mp;
    a.span = R.span;
    a.n_splits = R.n_splits;
    a.Qg = ws + R.qg;
    a.dOg = ws + R.dog;
    a.gL2 = reinterpret_cast<float*>(ws + R.gl2);
    a.gD = reinterpret_cast<float*>(ws + R.gd);
    a.gpos = reinterpret_cast<int*>(ws + R.gpos);
    a.dq_part = reinterpret_cast<float*>(ws + R.dq_part);
    a.extra_k = reinterpret_cast<float*>(ws + R.extra_k);
    a.extra_v = reinterpret_cast<float*>(ws + R.extra_v);
  }
  st = device_status_ptr(&a.status);
  if (st != MSA_OK) return st;
  const uint64_t lim = g_wait_limit_ns.load();
  a.wait_limit_ns = lim ? lim : kDefaultWaitNs;
  a.no_pair = g_force_single_cta.load();
  a.max_clusters = g_max_clusters_cap.load();
  const char* why = nullptr;
  cudaError_t e = msa::launch_attn_bwd(a, reinterpret_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && why) return fail(MSA_ERR_CUDA, "backward: %s", why);
  return launched(e, "backward");
}

msa_status msa_attn_bwd(const void* q, const void* k, const void* v, const void* k_lm,
                        const void* v_lm, const void* out, const float* lse, const void* dout,
                        void* dq, void* dk, void* dv, int64_t n, int Hq, int Hkv, int d,
                        int64_t window, int n_landmarks, float scale, msa_dtype in_dt,
                        msa_dtype out_dt, msa_dtype grad_dt, void* workspace,
                        size_t workspace_bytes, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  return attn_bwd_impl(q, k, v, k_lm, v_lm, out, lse, dout, nullptr, 0, dq, dk, dv, n, Hq, Hkv,
                       d, window, n_landmarks, scale, in_dt, out_dt, grad_dt, workspace,
                       workspace_bytes, stream);
}

size_t msa_attn_bwd_global_rows_workspace_size(int64_t n, int64_t n_global, int Hq, int Hkv,
                                               int d, int n_landmarks) {
  if (check_bwd_sizes(n, Hq, Hkv, d, n_landmarks) != MSA_OK ||
      check_global_rows(n, n_global, Hq, Hkv) != MSA_OK)
    return 0;
  return bwd_gr_plan(bwd_plan(n, Hq, Hkv, d, n_landmarks).total, n, n_global, Hq, Hkv, d).total;
}

msa_status msa_attn_bwd_global_rows(const void* q, const void* k, const void* v,
                                    const void* k_lm, const void* v_lm, const void* out,
                                    const float* lse, const void* dout, const int64_t* rows,
                                    int64_t n_global, void* dq, void* dk, void* dv, int64_t n,
                                    int Hq, int Hkv, int d, int64_t window, int n_landmarks,
                                    float scale, msa_dtype in_dt, msa_dtype out_dt,
                                    msa_dtype grad_dt, void* workspace, size_t workspace_bytes,
                                    msa_stream_t stream) {
  MSA_NVTX_RANGE();
  if (!rows) return fail(MSA_ERR_INVALID_ARG, "null rows pointer");
  return attn_bwd_impl(q, k, v, k_lm, v_lm, out, lse, dout, rows, n_global, dq, dk, dv, n, Hq,
                       Hkv, d, window, n_landmarks, scale, in_dt, out_dt, grad_dt, workspace,
                       workspace_bytes, stream);
}

msa_status msa_attn_fwd_partial(const void* q, const void* k_chunk, const void* v_chunk,
                                 float* out_part, float* lse_part, int64_t n_q, int64_t q_start,
                                 int64_t n_kv, int64_t kv_start, int Hq, int Hkv, int d,
                                 int64_t window, float scale, msa_dtype in_dt,
                                 msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st =
      check_attn_common(q, k_chunk, v_chunk, out_part, lse_part, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (n_q < 1 || n_q > kMaxRows || n_kv < 1 || n_kv > kMaxRows)
    return fail(MSA_ERR_INVALID_ARG, "n_q=%lld n_kv=%lld out of range", (long long)n_q,
                (long long)n_kv);
  if (q_start < 0 || kv_start < 0)
    return fail(MSA_ERR_INVALID_ARG, "q_start=%lld kv_start=%lld must be >= 0",
                (long long)q_start, (long long)kv_start);
  msa::AttnArgs a{};
  a.q = q;
  a.k = k_chunk;
  a.v = v_chunk;
  a.out = out_part;
  a.lse = lse_part;
  a.n_q = n_q;
  a.q_start = q_start;
  a.n_kv = n_kv;
  a.kv_start = kv_start;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = window;
  a.G = 0;
  a.block = 1;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = 0;
  a.partial = 1;
  return run_attn(a, reinterpret_cast<cudaStream_t>(stream));
}

msa_status msa_attn_fwd_partial_merge(const void* q, const void* k_chunk, const void* v_chunk,
                                       float* out_run, float* lse_run, int64_t n_q,
                                       int64_t q_start, int64_t n_kv, int64_t kv_start, int Hq,
                                       int Hkv, int d, int64_t window, float scale,
                                       msa_dtype in_dt, msa_stream_t stream) {
  MSA_NVTX_RANGE();
  msa_status st =
      check_attn_common(q, k_chunk, v_chunk, out_run, lse_run, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (n_q < 1 || n_q > kMaxRows || n_kv < 1 || n_kv > kMaxRows)
    return fail(MSA_ERR_INVALID_ARG, "n_q=%lld n_kv=%lld out of range", (long long)n_q,
                (long long)n_kv);
  if (q_start < 0 || kv_start < 0)
    return fail(MSA_ERR_INVALID_ARG, "q_start=%lld kv_start=%lld must be >= 0",
                (long long)q_start, (long long)kv_start);
  msa::AttnArgs a{};
  a.q = q;
  a.k = k_chunk;
  a.v = v_chunk;
  a.out = out_run;
  a.lse = lse_run;
  a.n_q = n_q;
  a.q_start = q_start;
  a.n_kv = n_kv;
  a.kv_start = kv_start;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.window = window;
  a.G = 0;
  a.block = 1;
  a.scale = scale;
  a.in_bf16 = in_dt == MSA_BF16;
  a.out_bf16 = 0;
  a.partial = 1;
  a.merge = 1;
  return run_attn(a, reinterpret_cast<cudaStream_t>(stream));
}

// Row-chunk plan of msa_attn_fwd_host: chunks of `rows` query rows (a
// multiple of 128; default about n/32, at least 4096), and the workspace:
// K and V whole [n, Hkv, d] and the landmarks [G, Hkv, d] in the input
// dtype, Q staging for two chunks, O staging for two chunks in the output
// dtype, the whole lse [Hq, n] fp32; each piece 256-byte aligned.
struct HostPlan {
  int64_t rows;
  size_t k, v, klm, vlm, q[2], o[2], lse, total;
};

static HostPlan host_plan(int64_t n, int Hq, int Hkv, int d, int G, int64_t chunk_rows,
                          msa_dtype in_dt, msa_dtype out_dt) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  HostPlan P{};
  int64_t rows = chunk_rows > 0 ? chunk_rows : msa::max64(4096, (n + 31) / 32);
  rows = msa::max64(128, (rows + 127) / 128 * 128);
  P.rows = rows;
  const int64_t stage = msa::min64(rows, n);
  const size_t es = in_dt == MSA_BF16 ? 2 : 4, eo = out_dt == MSA_BF16 ? 2 : 4;
  const size_t kv = static_cast<size_t>(n) * Hkv * d * es;
  const size_t lm = static_cast<size_t>(G > 0 ? G : 1) * Hkv * d * es;
  size_t at = 0;
  P.k = at;
  at += up(kv);
  P.v = at;
  at += up(kv);
  P.klm = at;
  at += up(lm);
  P.vlm = at;
  at += up(lm);
  for (int b = 0; b < 2; ++b) {
    P.q[b] = at;
    at += up(static_cast<size_t>(stage) * Hq * d * es);
  }
  for (int b = 0; b < 2; ++b) {
    P.o[b] = at;
    at += up(static_cast<size_t>(stage) * Hq * d * eo);
  }
  P.lse = at;
  at += up(static_cast<size_t>(Hq) * n * sizeof(float));
  P.total = at;
  return P;
}

size_t msa_attn_fwd_host_workspace_size(int64_t n, int Hq, int Hkv, int d, int n_landmarks,
                                        int64_t chunk_rows, msa_dtype in_dt, msa_dtype out_dt) {
  if (n < 1 || n > kMaxRows || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || (d != 64 && d != 128) ||
      !valid_dtype(in_dt) || !valid_dtype(out_dt) || n_landmarks < 0 || n_landmarks > n ||
      (n_landmarks > 0 && n % n_landmarks != 0))
    return 0;
  return host_plan(n, Hq, Hkv, d, n_landmarks, chunk_rows, in_dt, out_dt).total;
}

// The window + landmark forward on host buffers: K, V and Q go to the
// device in row chunks on `copy_in`, each chunk's landmarks are pooled and
// its rows attended (msa_attn_fwd_rows) on `stream`, and O comes back on
// `copy_out`, double-buffered, so that the copies overlap the kernels.
// Rows [r0, r1) need only K/V rows below r1 and the landmarks of the blocks
// inside them; when a chunk is not a whole number of landmark blocks, K and
// V are copied and pooled whole before the first chunk instead.
msa_status msa_attn_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse,
                             int64_t n, int Hq, int Hkv, int d, int64_t window, int n_landmarks,
                             float scale, msa_dtype in_dt, msa_dtype out_dt, int64_t chunk_rows,
                             void* workspace, size_t workspace_bytes, msa_stream_t stream,
                             msa_stream_t copy_in, msa_stream_t copy_out) {
  MSA_NVTX_RANGE();
  msa_status st = check_attn_common(q, k, v, out, lse, Hq, Hkv, d, window, scale, in_dt);
  if (st != MSA_OK) return st;
  if (n < 1 || n > kMaxRows) return fail(MSA_ERR_INVALID_ARG, "n=%lld out of range", (long long)n);
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  if (n_landmarks < 0 || n_landmarks > n || (n_landmarks > 0 && n % n_landmarks != 0))
    return fail(MSA_ERR_INVALID_ARG, "G=%d must satisfy 0 <= G <= n and n %% G == 0 (n=%lld)",
                n_landmarks, (long long)n);
  if (chunk_rows < 0) return fail(MSA_ERR_INVALID_ARG, "chunk_rows=%lld", (long long)chunk_rows);
  const HostPlan P = host_plan(n, Hq, Hkv, d, n_landmarks, chunk_rows, in_dt, out_dt);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(MSA_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (workspace_bytes < P.total)
    return fail(MSA_ERR_INVALID_ARG, "workspace of %zu bytes, %zu needed", workspace_bytes,
                P.total);
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const cudaStream_t si = copy_in ? reinterpret_cast<cudaStream_t>(copy_in) : cs;
  const cudaStream_t so = copy_out ? reinterpret_cast<cudaStream_t>(copy_out) : cs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int G = n_landmarks;
  const int64_t blk = G > 0 ? n / G : 1;
  const int64_t rows = P.rows;
  const bool kv_stream = G == 0 || rows % blk == 0;  // K/V and pooling per chunk
  const size_t es = in_dt == MSA_BF16 ? 2 : 4, eo = out_dt == MSA_BF16 ? 2 : 4;
  const size_t tok_kv = static_cast<size_t>(Hkv) * d * es;
  const size_t tok_q = static_cast<size_t>(Hq) * d * es, tok_o = static_cast<size_t>(Hq) * d * eo;
  const uint8_t* hk = static_cast<const uint8_t*>(k);
  const uint8_t* hv = static_cast<const uint8_t*>(v);
  const uint8_t* hq = static_cast<const uint8_t*>(q);
  uint8_t* ho = static_cast<uint8_t*>(out);
  float* dlse = reinterpret_cast<float*>(ws + P.lse);

  // Events: start (prior work on `stream`), K/V whole, and per staging
  // buffer: inputs landed, chunk computed, output copied back.
  cudaEvent_t ev[8] = {};
  int n_ev = 0;
  cudaError_t e = cudaSuccess;
  for (; n_ev < 8 && e == cudaSuccess; ++n_ev)
    e = cudaEventCreateWithFlags(&ev[n_ev], cudaEventDisableTiming);
  auto finish = [&](msa_status result) {
    cudaStreamSynchronize(si);
    cudaStreamSynchronize(cs);
    cudaStreamSynchronize(so);
    for (int i = 0; i < 8; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);
    return result;
  };
  if (e != cudaSuccess) return finish(fail(MSA_ERR_CUDA, "cudaEventCreate: %s", cudaGetErrorString(e)));
  cudaEvent_t ev_start = ev[0], ev_kv = ev[1];
  cudaEvent_t* ev_in = &ev[2];
  cudaEvent_t* ev_done = &ev[4];
  cudaEvent_t* ev_ofree = &ev[6];
  bool have_done[2] = {false, false}, have_ofree[2] = {false, false};
#define MSA_HOST_CHECK(call)                                                                 \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess)                                                                   \
      return finish(fail(MSA_ERR_CUDA, "host path, %s: %s", #call, cudaGetErrorString(e_))); \
  } while (0)
  MSA_HOST_CHECK(cudaEventRecord(ev_start, cs));
  MSA_HOST_CHECK(cudaStreamWaitEvent(si, ev_start, 0));
  MSA_HOST_CHECK(cudaStreamWaitEvent(so, ev_start, 0));
  if (G > 0) {
    // Landmark tiles can reach past the blocks pooled so far; those masked
    // rows must hold finite values (0 times NaN would not vanish in PV).
    const size_t lm_bytes = static_cast<size_t>(G) * tok_kv;
    MSA_HOST_CHECK(cudaMemsetAsync(ws + P.klm, 0, lm_bytes, cs));
    MSA_HOST_CHECK(cudaMemsetAsync(ws + P.vlm, 0, lm_bytes, cs));
  }
  if (!kv_stream) {
    MSA_HOST_CHECK(cudaMemcpyAsync(ws + P.k, hk, n * tok_kv, cudaMemcpyHostToDevice, si));
    MSA_HOST_CHECK(cudaMemcpyAsync(ws + P.v, hv, n * tok_kv, cudaMemcpyHostToDevice, si));
    MSA_HOST_CHECK(cudaEventRecord(ev_kv, si));
    MSA_HOST_CHECK(cudaStreamWaitEvent(cs, ev_kv, 0));
    msa::PoolArgs pa{ws + P.k, ws + P.v, ws + P.klm, ws + P.vlm, n, Hkv * d, G,
                     in_dt == MSA_BF16 ? 1 : 0, status_word()};
    MSA_HOST_CHECK(msa::launch_landmark_pool(pa, cs));
  }
  for (int64_t r0 = 0, c = 0; r0 < n; r0 += rows, ++c) {
    const int64_t r1 = msa::min64(n, r0 + rows), m = r1 - r0;
    const int b = static_cast<int>(c & 1);
    if (have_done[b]) MSA_HOST_CHECK(cudaStreamWaitEvent(si, ev_done[b], 0));
    if (kv_stream) {
      MSA_HOST_CHECK(cudaMemcpyAsync(ws + P.k + r0 * tok_kv, hk + r0 * tok_kv, m * tok_kv,
                                     cudaMemcpyHostToDevice, si));
      MSA_HOST_CHECK(cudaMemcpyAsync(ws + P.v + r0 * tok_kv, hv + r0 * tok_kv, m * tok_kv,
                                     cudaMemcpyHostToDevice, si));
    }
    MSA_HOST_CHECK(cudaMemcpyAsync(ws + P.q[b], hq + r0 * tok_q, m * tok_q,
                                   cudaMemcpyHostToDevice, si));
    MSA_HOST_CHECK(cudaEventRecord(ev_in[b], si));
    MSA_HOST_CHECK(cudaStreamWaitEvent(cs, ev_in[b], 0));
    if (G > 0 && kv_stream) {  // the landmarks of this chunk's (whole) blocks
      const int64_t l0 = r0 / blk, l1 = r1 / blk;
      msa::PoolArgs pa{ws + P.k + r0 * tok_kv, ws + P.v + r0 * tok_kv, ws + P.klm + l0 * tok_kv,
                       ws + P.vlm + l0 * tok_kv, m, Hkv * d, static_cast<int>(l1 - l0),
                       in_dt == MSA_BF16 ? 1 : 0, status_word()};
      MSA_HOST_CHECK(msa::launch_landmark_pool(pa, cs));
    }
    if (have_ofree[b]) MSA_HOST_CHECK(cudaStreamWaitEvent(cs, ev_ofree[b], 0));
    msa::AttnArgs a{};
    a.q = ws + P.q[b];
    a.k = ws + P.k;
    a.v = ws + P.v;
    a.k_lm = G > 0 ? ws + P.klm : nullptr;
    a.v_lm = G > 0 ? ws + P.vlm : nullptr;
    a.out = ws + P.o[b];
    a.lse = dlse + r0;
    a.lse_ld = n;
    a.n_q = m;
    a.q_start = r0;
    a.n_kv = n;
    a.kv_start = 0;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.window = window;
    a.G = G;
    a.block = blk;
    a.scale = scale;
    a.in_bf16 = in_dt == MSA_BF16;
    a.out_bf16 = out_dt == MSA_BF16;
    st = run_attn(a, cs);
    if (st != MSA_OK) return finish(st);
    MSA_HOST_CHECK(cudaEventRecord(ev_done[b], cs));
    have_done[b] = true;
    MSA_HOST_CHECK(cudaStreamWaitEvent(so, ev_done[b], 0));
    MSA_HOST_CHECK(cudaMemcpyAsync(ho + r0 * tok_o, ws + P.o[b], m * tok_o,
                                   cudaMemcpyDeviceToHost, so));
    MSA_HOST_CHECK(cudaEventRecord(ev_ofree[b], so));
    have_ofree[b] = true;
  }
  // lse of every chunk (the last chunk's compute, which `so` waited for,
  // comes after all the others on `stream`).
  MSA_HOST_CHECK(cudaMemcpyAsync(lse, dlse, static_cast<size_t>(Hq) * n * sizeof(float),
                                 cudaMemcpyDeviceToHost, so));
#undef MSA_HOST_CHECK
  return finish(ok());
}

msa_status msa_lse_merge(const float* const* o_parts, const float* const* lse_parts, int n_parts,
                         void* out, float* lse, int64_t n, int Hq, int d, msa_dtype out_dt,
                         msa_stream_t stream) {
  MSA_NVTX_RANGE();
  if (!o_parts || !lse_parts || !out || !lse)
    return fail(MSA_ERR_INVALID_ARG, "null array or output pointer");
  if (n_parts < 1 || n_parts > MSA_MAX_MERGE_PARTS)
    return fail(MSA_ERR_INVALID_ARG, "n_parts=%d (1..%d)", n_parts, MSA_MAX_MERGE_PARTS);
  if (n < 1 || Hq < 1) return fail(MSA_ERR_INVALID_ARG, "n=%lld Hq=%d", (long long)n, Hq);
  if (d < 4 || d % 4 != 0) return fail(MSA_ERR_INVALID_ARG, "d=%d must be a multiple of 4", d);
  if (!valid_dtype(out_dt)) return fail(MSA_ERR_INVALID_ARG, "bad output dtype %d", (int)out_dt);
  if (!aligned16(out) || !aligned16(lse))
    return fail(MSA_ERR_INVALID_ARG, "output pointer not 16-byte aligned");
  msa::MergeArgs a{};
  for (int p = 0; p < n_parts; ++p) {
    if (!o_parts[p] || !lse_parts[p]) return fail(MSA_ERR_INVALID_ARG, "null partial %d", p);
    if (!aligned16(o_parts[p]) || !aligned16(lse_parts[p]))
      return fail(MSA_ERR_INVALID_ARG, "partial %d not 16-byte aligned", p);
    if (static_cast<const void*>(o_parts[p]) == out && (p > 0 || out_dt != MSA_F32))
      return fail(MSA_ERR_INVALID_ARG, "out may alias only o_parts[0], and only with fp32 output");
    if (lse_parts[p] == lse && p > 0)
      return fail(MSA_ERR_INVALID_ARG, "lse may alias only lse_parts[0]");
    a.o_parts[p] = o_parts[p];
    a.lse_parts[p] = lse_parts[p];
  }
  a.n_parts = n_parts;
  a.out = out;
  a.lse = lse;
  a.n = n;
  a.Hq = Hq;
  a.d = d;
  a.out_bf16 = out_dt == MSA_BF16;
  a.status = status_word();
  return launched(msa::launch_lse_merge(a, reinterpret_cast<cudaStream_t>(stream)), "lse merge");
}

int msa_attn_uses_tensor_cores(int Hq, int Hkv, int d, msa_dtype in_dt) {
  return msa::attn_tc_supported(Hq, Hkv, d, in_dt == MSA_BF16) ? 1 : 0;
}

int msa_attn_fwd_topk_uses_tensor_cores(int64_t n, int Hq, int Hkv, int d, int n_landmarks,
                                        msa_dtype in_dt) {
  if (n_landmarks < 1 || n < n_landmarks) return 0;
  // Selected key blocks map to whole 128-key tiles on the tensor-core path.
  const bool tiles_ok = (n / n_landmarks) % 128 == 0;
  return tiles_ok && msa::attn_tc_supported(Hq, Hkv, d, in_dt == MSA_BF16) ? 1 : 0;
}

msa_status msa_device_status(int clear) {
  MSA_NVTX_RANGE();
  int* ptr = nullptr;
  msa_status st = device_status_ptr(&ptr);
  if (st != MSA_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
  int v = 0;
  e = cudaMemcpy(&v, ptr, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (clear) {
    const int zero = 0;
    e = cudaMemcpy(ptr, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(MSA_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
  }
  if (v == MSA_ERR_TIMEOUT) return fail(MSA_ERR_TIMEOUT, "a bounded device wait ran out");
  if (v != 0) return fail(static_cast<msa_status>(v), "device status %d", v);
  return ok();
}

void msa_debug_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }

void msa_debug_force_single_cta(int on) { g_force_single_cta.store(on ? 1 : 0); }

void msa_debug_set_max_clusters(int n) { g_max_clusters_cap.store(n > 0 ? n : 0); }

}  // extern "C"
