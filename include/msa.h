/*
 * msa.h -- C ABI of libmsa: window + landmark sparse attention forward on
 * one GB300 (sm_103a), plus the log-sum-exp merge of Ring Attention partials.
 *
 * The method.  "Scaling GPU Cluster for Million Token Context", sections
 * "Why Sparse Attention Changes the Game" and "What is Flash-MSA Sparse
 * Attention in GPU Clusters?", describe Flash-MSA: every token attends to a
 * local window (4096 tokens there) and to a set of about 512 landmark tokens
 * that summarise distant context, fused in one pass that never materialises
 * the n x n score matrix.  The pages do not define landmarks or the mask;
 * this library fixes them as follows (batch 1, token-major layouts):
 *
 *   Q [n, Hq, d], K and V [n, Hkv, d]; query head h reads KV head
 *   h / (Hq/Hkv) (grouped-query attention, contiguous groups).
 *   Landmark l (0 <= l < G) is the mean of K (resp. V) over the contiguous
 *   block of B = n/G tokens [lB, (l+1)B).
 *   Row i attends keys j with i-w < j <= i, and every landmark l whose whole
 *   block lies before that window: (l+1)B <= i-w+1.
 *   One softmax over the union, scores scale * <q, k>:
 *   O[i,h,:] = sum_x softmax_x * V_x,  lse[h,i] = ln sum_x exp(scale<q,k_x>).
 *
 * Ring Attention ("Training at 1M+ Token Context: Ring Attention, YaRN,
 * NTK-Aware Scaling", Ring Attention paragraph) computes, per round, partial
 * attention of local queries against one contiguous KV block and aggregates
 * the softmax statistics; msa_attn_fwd_partial + msa_lse_merge are those two
 * steps, run on one GPU.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     and 16-byte aligned, unless stated otherwise.  The library never
 *     allocates device memory and never synchronises the stream; all work
 *     is enqueued on `stream` (NULL = legacy default stream) and results are
 *     valid in stream order.
 *   - Arguments are validated before anything is enqueued.  On failure the
 *     call enqueues nothing, returns a status code and records a message
 *     that msa_last_error_string() returns (per calling thread).
 *   - A launch failure returns MSA_ERR_CUDA.  Kernels that wait on
 *     asynchronous copies bound every wait; a wait that runs out makes the
 *     kernel finish early and record MSA_ERR_TIMEOUT in a per-device status
 *     word that msa_device_status() reads.
 *   - lse is always fp32, natural log.
 *   - Outputs and workspaces must not overlap any input, unless an entry
 *     point states otherwise (the running (O, lse) of a merge is both read
 *     and written).  Outputs are written by asynchronous bulk copies from
 *     shared memory as well as by the threads, in no order relative to other
 *     CTAs' reads of the inputs.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *msa_stream_t; /* same object as cudaStream_t */

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or shape */
    MSA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d not 64/128) */
    MSA_ERR_CUDA = 3,        /* CUDA runtime or driver error */
    MSA_ERR_TIMEOUT = 4      /* a bounded device wait ran out */
} msa_status;

typedef enum { MSA_F32 = 0, MSA_BF16 = 1 } msa_dtype;

/* Version as major*10000 + minor*100 + patch. */
int msa_version(void);

/* Message of the last failed call on this thread ("" if none). */
const char *msa_last_error_string(void);

/*
 * Landmark pooling ("Scaling GPU Cluster for Million Token Context",
 * "What is Flash-MSA ...": landmarks summarise distant context; defined here
 * as block means).
 *   k, v       [n, Hkv, d] in dtype `dt`
 *   k_lm, v_lm [G, Hkv, d] in dtype `dt`, written:
 *              k_lm[l,c,:] = (1/B) sum_{j=lB}^{(l+1)B-1} k[j,c,:], B = n/G,
 *              summed in fp32, rounded to `dt` (nearest even).
 * Errors: INVALID_ARG if a pointer is null or not 16-byte aligned, n < 1,
 * Hkv < 1, G < 1, G > n or n % G != 0; UNSUPPORTED if d is not 64 or 128.
 */
msa_status msa_landmark_pool(const void *k, const void *v, void *k_lm,
                             void *v_lm, int64_t n, int Hkv, int d,
                             int n_landmarks, msa_dtype dt,
                             msa_stream_t stream);

/*
 * Fused window + landmark attention forward (the Flash-MSA pass above).
 *   q          [n, Hq, d]  in `in_dt`
 *   k, v       [n, Hkv, d] in `in_dt`
 *   k_lm, v_lm [G, Hkv, d] in `in_dt`: the landmarks msa_landmark_pool
 *              wrote for these k, v (may be NULL iff G == 0)
 *   out        [n, Hq, d]  in `out_dt`, written
 *   lse        [Hq, n] fp32, written (natural log of the softmax denominator)
 *   window     w >= 1 (keys i-w < j <= i); w >= n with G = 0 is causal
 *              attention
 *   scale      score scale (1/sqrt(d) for standard attention)
 * bf16 inputs with d = 128 run on the tensor cores (TMA + tcgen05, fp32
 * accumulation in tensor memory); other inputs run a CUDA-core kernel with
 * fp32 arithmetic.
 * Errors: INVALID_ARG for null/misaligned pointers, n < 1, w < 1, Hq or Hkv
 * < 1, Hq % Hkv != 0, G < 0, G > n, G > 0 with n % G != 0, G > 0 with null
 * landmarks; UNSUPPORTED if d is not 64 or 128.
 */
msa_status msa_attn_fwd(const void *q, const void *k, const void *v,
                        const void *k_lm, const void *v_lm, void *out,
                        float *lse, int64_t n, int Hq, int Hkv, int d,
                        int64_t window, int n_landmarks, float scale,
                        msa_dtype in_dt, msa_dtype out_dt,
                        msa_stream_t stream);

/*
 * msa_attn_fwd restricted to the contiguous query rows [q_start, q_start +
 * n_q): the same window + landmark attention, so that a caller can stream
 * Q and O through the device in row chunks (keys, values and landmarks are
 * the whole sequence's).
 *   q_rows [n_q, Hq, d] = rows q_start.. of Q; k, v [n, Hkv, d]; k_lm, v_lm
 *   [G, Hkv, d]; out_rows [n_q, Hq, d] in `out_dt`; lse: lse[h * lse_ld + r]
 *   receives row q_start + r of head h (lse_ld >= n_q; pass the full [Hq, n]
 *   array offset by q_start and lse_ld = n to fill it chunk by chunk; lse
 *   needs 4-byte alignment only, the other pointers 16).
 * Errors: as msa_attn_fwd, plus INVALID_ARG when the rows do not lie in
 * [0, n) or lse_ld < n_q.
 */
msa_status msa_attn_fwd_rows(const void *q_rows, const void *k, const void *v,
                             const void *k_lm, const void *v_lm, void *out_rows,
                             float *lse, int64_t lse_ld, int64_t q_start,
                             int64_t n_q, int64_t n, int Hq, int Hkv, int d,
                             int64_t window, int n_landmarks, float scale,
                             msa_dtype in_dt, msa_dtype out_dt,
                             msa_stream_t stream);

/* Bytes of device workspace msa_attn_fwd_host needs (0 for invalid sizes):
 * K and V whole, the landmarks, two chunks of Q and of O, the lse; about
 * 2 n Hkv d + 4 chunk_rows Hq d elements plus 4 Hq n bytes. */
size_t msa_attn_fwd_host_workspace_size(int64_t n, int Hq, int Hkv, int d,
                                        int n_landmarks, int64_t chunk_rows,
                                        msa_dtype in_dt, msa_dtype out_dt);

/*
 * msa_landmark_pool + msa_attn_fwd on HOST buffers, for a caller whose
 * sequence lives in host memory (the end-to-end forward whose time
 * "Scaling GPU Cluster for Million Token Context", section "Why Sparse
 * Attention Changes the Game", quotes).  Rows [r0, r1) need only the
 * K/V rows below r1 and the landmarks of the blocks inside them, so K, V
 * and Q go to the device in chunks of chunk_rows rows (rounded up to a
 * multiple of 128; 0 = about n/32, at least 4096) on `copy_in`, each
 * chunk's landmarks are pooled and its rows attended on `stream`, and O
 * comes back on `copy_out`, two chunks in flight, so that the copies
 * overlap the kernels.  When chunk_rows is not a multiple of the landmark
 * block n/G, K and V are copied and pooled whole before the first chunk.
 *   q [n, Hq, d], k, v [n, Hkv, d] in `in_dt`: HOST memory (pinned memory
 *     lets the copies run asynchronously), 16-byte aligned
 *   out [n, Hq, d] in `out_dt`, lse [Hq, n] fp32: HOST memory, written
 *   workspace: DEVICE memory, 256-byte aligned, at least
 *     msa_attn_fwd_host_workspace_size bytes
 *   copy_in, copy_out: streams for the copies (NULL: `stream`, no overlap)
 * Unlike the other entry points this call waits for its streams: out and
 * lse are final when it returns.  It creates and destroys eight CUDA
 * events (no device memory).  The results equal msa_attn_fwd's bit for
 * bit (the same kernels on the same rows).
 * Errors: as msa_attn_fwd, plus INVALID_ARG for a negative chunk_rows or a
 * null, misaligned or too small workspace; MSA_ERR_CUDA if a copy fails.
 */
msa_status msa_attn_fwd_host(const void *q, const void *k, const void *v,
                             void *out, float *lse, int64_t n, int Hq, int Hkv,
                             int d, int64_t window, int n_landmarks, float scale,
                             msa_dtype in_dt, msa_dtype out_dt,
                             int64_t chunk_rows, void *workspace,
                             size_t workspace_bytes, msa_stream_t stream,
                             msa_stream_t copy_in, msa_stream_t copy_out);

/*
 * Block-band attention: the 2-D block-sparse mask of "Million Token Context
 * Window Optimization: What Actually Works", section "The indexing game:
 * smarter context management" (each 128-token block attends to 16 other
 * blocks, left and right).  Row i attends every key j of the blocks within
 * band_half blocks of its own, |floor(j/band_block) - floor(i/band_block)|
 * <= band_half, 0 <= j < n (not causal); one softmax, scores scale*<q,k>.
 * (128-token blocks and 16 neighbours: band_block = 128, band_half = 8.)
 *   q [n, Hq, d], k, v [n, Hkv, d] in `in_dt`; out [n, Hq, d] in `out_dt`;
 *   lse [Hq, n] fp32.
 * Errors: as msa_attn_fwd, plus INVALID_ARG for band_block < 1 or
 * band_half < 0.
 */
msa_status msa_attn_fwd_band(const void *q, const void *k, const void *v,
                             void *out, float *lse, int64_t n, int Hq,
                             int Hkv, int d, int64_t band_block,
                             int64_t band_half, float scale, msa_dtype in_dt,
                             msa_dtype out_dt, msa_stream_t stream);

/* Largest number of key blocks (G) the top-k selection accepts. */
#define MSA_MAX_SELECT_BLOCKS 1024

/*
 * Landmark-scored top-k block selection, standing in for the hierarchical
 * context index of "Million Token Context Window Optimization: What Actually
 * Works", section "The indexing game: smarter context management" (score
 * the input's chunks against the query; attend only the top-k chunks plus a
 * history window).  A chunk is one of G contiguous key blocks of B = n/G
 * tokens and its landmark (mean key, from msa_landmark_pool) scores it.
 * For every query block t of 128 rows and KV group c:
 *   score(l) = sum over rows i of block t, heads h of group c of
 *              <q[i,h], k_lm[l,c]>,
 * defined for the blocks wholly before the window of the block's first row,
 * (l+1)B <= 128t - w + 1.  The min(top_k, #candidates) best blocks are
 * chosen (ties to the lower index; scores summed in fp32).
 *   q    [n, Hq, d] in `in_dt`;  k_lm [G, Hkv, d] in `in_dt`
 *   sel  [ceil(n/128), Hkv, top_k] int32, written: chosen blocks ascending
 *   cnt  [ceil(n/128), Hkv] int32, written: how many were chosen
 * Errors: INVALID_ARG for null/misaligned pointers, Hq % Hkv != 0, w < 1,
 * G < 1, G > n, n % G != 0, top_k < 1 or top_k > G; UNSUPPORTED if d is not
 * 64 or 128 or G > MSA_MAX_SELECT_BLOCKS.
 */
msa_status msa_block_select(const void *q, const void *k_lm, int32_t *sel,
                            int32_t *cnt, int64_t n, int Hq, int Hkv, int d,
                            int64_t window, int n_landmarks, int top_k,
                            msa_dtype in_dt, msa_stream_t stream);

/*
 * Attention over each row's causal window (i-w < j <= i) plus every token
 * of the key blocks msa_block_select chose for its query block; one
 * softmax, scores scale*<q,k>.
 *   q [n, Hq, d], k, v [n, Hkv, d] in `in_dt`; sel, cnt as written by
 *   msa_block_select for the same n, Hkv, G, top_k; out [n, Hq, d] in
 *   `out_dt`; lse [Hq, n] fp32.
 * Errors: as msa_attn_fwd and msa_block_select.  The kernels check the
 * selection they read: a count above min(top_k, candidates) or a block that
 * is not a candidate of its query block is clamped (to that bound / to block
 * 0) and MSA_ERR_INVALID_ARG recorded in the device status word
 * (msa_device_status), so a bad selection never reads outside K and V.
 */
msa_status msa_attn_fwd_select(const void *q, const void *k, const void *v,
                               const int32_t *sel, const int32_t *cnt,
                               void *out, float *lse, int64_t n, int Hq,
                               int Hkv, int d, int64_t window, int n_landmarks,
                               int top_k, float scale, msa_dtype in_dt,
                               msa_dtype out_dt, msa_stream_t stream);

/* Bytes of workspace msa_attn_fwd_topk needs (0 for invalid sizes). */
size_t msa_attn_fwd_topk_workspace_size(int64_t n, int Hkv, int d,
                                        int n_landmarks, int top_k,
                                        msa_dtype in_dt);

/*
 * The whole top-k path in one call: pool the block-mean keys, select each
 * query block's top-k key blocks (msa_block_select), attend window +
 * selected blocks (msa_attn_fwd_select).  The intermediate keys and
 * selection live in the caller's `workspace` (device memory, 256-byte
 * aligned, at least msa_attn_fwd_topk_workspace_size bytes).
 * Errors: as the three steps, plus INVALID_ARG for a null, misaligned or
 * too small workspace.
 */
msa_status msa_attn_fwd_topk(const void *q, const void *k, const void *v,
                             void *out, float *lse, int64_t n, int Hq, int Hkv,
                             int d, int64_t window, int n_landmarks, int top_k,
                             float scale, msa_dtype in_dt, msa_dtype out_dt,
                             void *workspace, size_t workspace_bytes,
                             msa_stream_t stream);

/* Bytes of the fixed device scratch msa_attn_fwd_topk_noalloc uses (16 MiB;
 * the 1M-token layer with 512 blocks, 8 KV heads, d = 128 bf16 and top-50
 * needs 14,417,920). */
#define MSA_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * msa_attn_fwd_topk without a workspace argument, for callers that cannot
 * allocate device memory (a plain C host program holding no allocator, or a
 * runtime that must not call cudaMalloc between launches).  The pages
 * describe no such entry point; it is an interface convenience only, with
 * the same kernels and results as msa_attn_fwd_topk.
 * The intermediates live in one fixed, file-scope device array of
 * MSA_NOALLOC_SCRATCH_BYTES per device; nothing is allocated or freed.
 *   - The array belongs to the library's device code: once that code is
 *     loaded on a device (by the first call of any entry point there), the
 *     device holds its MSA_NOALLOC_SCRATCH_BYTES (16 MiB) whether or not
 *     this entry point is ever called, until the context is destroyed.
 *   - Every call looks up the array's address in the current context (no
 *     address is kept between calls, so a cudaDeviceReset in between is
 *     harmless).  The first call on a device may load the library's device
 *     code; make one call of the library on each device before any stream
 *     capture begins.
 *   - The scratch is shared by every call on a device: calls whose work can
 *     overlap (unordered streams, several host threads) race on it and give
 *     wrong results.  Order them on one stream.
 *   - Nothing in the scratch needs to start at zero.
 * Errors: as msa_attn_fwd_topk; MSA_ERR_UNSUPPORTED (with the sizes in
 * msa_last_error_string) when the sizes need more than
 * MSA_NOALLOC_SCRATCH_BYTES, i.e. msa_attn_fwd_topk_workspace_size above it;
 * MSA_ERR_CUDA if the address lookup fails.
 */
msa_status msa_attn_fwd_topk_noalloc(const void *q, const void *k, const void *v,
                                     void *out, float *lse, int64_t n, int Hq,
                                     int Hkv, int d, int64_t window,
                                     int n_landmarks, int top_k, float scale,
                                     msa_dtype in_dt, msa_dtype out_dt,
                                     msa_stream_t stream);

/*
 * Global query rows of the block-sparse pattern in "Training at 1M+ Token
 * Context: Ring Attention, YaRN, NTK-Aware Scaling GPU Cost" (Block-Sparse
 * Flash Attention paragraph: global tokens attend to all, local tokens to a
 * sliding window, compression tokens summarise distant context).  The local
 * rows are msa_attn_fwd with n_landmarks = n / 32 (one compression token,
 * the mean of K and of V, per 32-token sub-block: 256 per 8192 tokens);
 * this call then overwrites, for every position r in rows[0..n_global),
 * out[r, :, :] and lse[:, r] with attention over every key j <= r (causal,
 * no compression tokens), one softmax.
 *   q [n, Hq, d], k, v [n, Hkv, d] in `in_dt`; rows: device int64 array of
 *   positions (any order; a repeated position is computed twice, same
 *   result); out [n, Hq, d] in `out_dt`, lse [Hq, n] fp32: only the listed
 *   rows are written.
 *   workspace: device memory, 256-byte aligned, at least
 *   msa_attn_fwd_global_rows_workspace_size bytes (per-split partials).
 * Errors: as msa_attn_fwd, plus INVALID_ARG for a null or misaligned rows
 * array or workspace, n_global < 1 or > n, a too small workspace;
 * UNSUPPORTED when n_global * Hq / Hkv exceeds 262140.  A position outside
 * [0, n) in rows is skipped by the kernels and MSA_ERR_INVALID_ARG recorded
 * in the device status word (msa_device_status).
 */
msa_status msa_attn_fwd_global_rows(const void *q, const void *k, const void *v,
                                    const int64_t *rows, int64_t n_global,
                                    void *out, float *lse, int64_t n, int Hq,
                                    int Hkv, int d, float scale,
                                    msa_dtype in_dt, msa_dtype out_dt,
                                    void *workspace, size_t workspace_bytes,
                                    msa_stream_t stream);

/* Bytes of workspace msa_attn_fwd_global_rows needs (0 for invalid sizes). */
size_t msa_attn_fwd_global_rows_workspace_size(int64_t n, int64_t n_global,
                                               int Hq, int Hkv, int d);

/*
 * Backward pass of msa_attn_fwd: the gradients of sum <dout, out> with
 * respect to q, k and v, for training with the sparse pattern (the
 * Block-Sparse Flash Attention paragraph of "Training at 1M+ Token Context:
 * Ring Attention, YaRN, NTK-Aware Scaling GPU Cost" trains with it).  With
 * P recomputed from the forward's lse, D_i = <dout_i, out_i> and
 * dS = P (dout V^T - D): dq = scale dS K, dk = scale dS^T Q, dv = P^T dout,
 * summed over the query heads of each KV group; a landmark's gradient
 * reaches each of the B = n/G tokens it averages divided by B.
 *   q, k, v, k_lm, v_lm as given to msa_attn_fwd (bf16, d = 128);
 *   out [n, Hq, d] (`out_dt`) and lse [Hq, n] fp32 as msa_attn_fwd wrote
 *   them; dout [n, Hq, d] bf16;
 *   dq [n, Hq, d], dk, dv [n, Hkv, d] in `grad_dt`, written;
 *   workspace: device memory, 256-byte aligned, at least
 *   msa_attn_bwd_workspace_size bytes.
 * Errors: as msa_attn_fwd, plus INVALID_ARG for null/misaligned gradient
 * pointers or workspace, a too small workspace; UNSUPPORTED unless the
 * inputs are bf16 with d = 128.
 */
msa_status msa_attn_bwd(const void *q, const void *k, const void *v,
                        const void *k_lm, const void *v_lm, const void *out,
                        const float *lse, const void *dout, void *dq, void *dk,
                        void *dv, int64_t n, int Hq, int Hkv, int d,
                        int64_t window, int n_landmarks, float scale,
                        msa_dtype in_dt, msa_dtype out_dt, msa_dtype grad_dt,
                        void *workspace, size_t workspace_bytes,
                        msa_stream_t stream);

/* Bytes of workspace msa_attn_bwd needs (0 for invalid sizes): about
 * 8 * Hq * n bytes of row statistics, plus, with landmarks, per-query-chunk
 * partial landmark gradients (up to about 256 MiB, fewer chunks for short
 * sequences) and their sum (8 * n_landmarks * Hkv * d bytes). */
size_t msa_attn_bwd_workspace_size(int64_t n, int Hq, int Hkv, int d,
                                   int n_landmarks);

/*
 * Backward pass of the compression-token pattern: msa_attn_fwd (window +
 * n_landmarks compression tokens) followed by msa_attn_fwd_global_rows on
 * rows[0..n_global) -- the pattern the Block-Sparse Flash Attention
 * paragraph of "Training at 1M+ Token Context" trains with.  A global row's
 * output does not depend on the window or the compression tokens and the
 * other rows' do not depend on the global rows' queries, so the gradients
 * are those of msa_attn_bwd with the global rows given no weight, plus
 * those of the global rows' causal attention (every key j <= the row):
 * their dQ rows, and their dK / dV added into every key they see.
 *   Arguments as msa_attn_bwd, plus rows / n_global as given to
 *   msa_attn_fwd_global_rows (out and lse as both forward calls left
 *   them); a repeated position counts once.
 *   workspace: at least msa_attn_bwd_global_rows_workspace_size bytes.
 * Errors: as msa_attn_bwd and msa_attn_fwd_global_rows; a position outside
 * [0, n) is skipped and MSA_ERR_INVALID_ARG recorded in the device status
 * word.
 */
msa_status msa_attn_bwd_global_rows(const void *q, const void *k, const void *v,
                                    const void *k_lm, const void *v_lm,
                                    const void *out, const float *lse,
                                    const void *dout, const int64_t *rows,
                                    int64_t n_global, void *dq, void *dk,
                                    void *dv, int64_t n, int Hq, int Hkv, int d,
                                    int64_t window, int n_landmarks, float scale,
                                    msa_dtype in_dt, msa_dtype out_dt,
                                    msa_dtype grad_dt, void *workspace,
                                    size_t workspace_bytes, msa_stream_t stream);

/* Bytes of workspace msa_attn_bwd_global_rows needs (0 for invalid sizes). */
size_t msa_attn_bwd_global_rows_workspace_size(int64_t n, int64_t n_global,
                                               int Hq, int Hkv, int d,
                                               int n_landmarks);

/*
 * One Ring Attention round's partial: queries at global positions
 * q_start .. q_start+n_q-1 against the contiguous KV chunk at global
 * positions kv_start .. kv_start+n_kv-1, with the causal window mask
 * i-w < j <= i taken in global positions, no landmarks.
 *   q        [n_q, Hq, d]   in `in_dt`
 *   k_chunk, v_chunk [n_kv, Hkv, d] in `in_dt`
 *   out_part [n_q, Hq, d] fp32, written for every row with at least one key
 *   lse_part [Hq, n_q] fp32, written; -inf for a row with no key in the
 *            chunk (its out_part row is then left untouched)
 * Errors: as msa_attn_fwd, plus INVALID_ARG for n_q < 1, n_kv < 1,
 * q_start < 0 or kv_start < 0.
 */
msa_status msa_attn_fwd_partial(const void *q, const void *k_chunk,
                                 const void *v_chunk, float *out_part,
                                 float *lse_part, int64_t n_q, int64_t q_start,
                                 int64_t n_kv, int64_t kv_start, int Hq,
                                 int Hkv, int d, int64_t window, float scale,
                                 msa_dtype in_dt, msa_stream_t stream);

/*
 * One Ring Attention round with its aggregation fused in ("Training at 1M+
 * Token Context", Ring Attention paragraph: each round computes partial
 * attention against one KV block and immediately aggregates the softmax
 * statistics).  Computes the partial of msa_attn_fwd_partial for queries
 * q_start.. against the chunk kv_start.., and merges it into the running
 * result in place:
 *   lse_run <- ln(exp(lse_run) + exp(lse_p)),
 *   out_run <- exp(lse_run_old - lse_run) out_run + exp(lse_p - lse_run) O_p,
 * so the partial never reaches HBM.  Rows with no key in the chunk are left
 * untouched.  A row whose lse_run is -inf takes O_p as is (out_run is not
 * read there), so a fresh run starts from lse_run = -inf and any out_run.
 * After every chunk has been merged (any order), out_run/lse_run equal the
 * single-pass msa_attn_fwd result up to rounding.
 *   q        [n_q, Hq, d] in `in_dt`;  k_chunk, v_chunk [n_kv, Hkv, d]
 *   out_run  [n_q, Hq, d] fp32, read and written
 *   lse_run  [Hq, n_q] fp32, read and written
 * Errors: as msa_attn_fwd_partial.
 */
msa_status msa_attn_fwd_partial_merge(const void *q, const void *k_chunk,
                                       const void *v_chunk, float *out_run,
                                       float *lse_run, int64_t n_q,
                                       int64_t q_start, int64_t n_kv,
                                       int64_t kv_start, int Hq, int Hkv, int d,
                                       int64_t window, float scale,
                                       msa_dtype in_dt, msa_stream_t stream);

/* Largest number of partials msa_lse_merge accepts in one call. */
#define MSA_MAX_MERGE_PARTS 64

/*
 * Exact merge of partial results over disjoint key sets (the aggregation
 * step of a Ring Attention round):
 *   lse = ln sum_p exp(lse_p),   out = sum_p exp(lse_p - lse) * o_p,
 * skipping parts whose lse_p is -inf; a row where every part is -inf gets
 * lse = -inf and out = 0.
 *   o_parts   HOST array of n_parts DEVICE pointers, each [n, Hq, d] fp32
 *   lse_parts HOST array of n_parts DEVICE pointers, each [Hq, n] fp32
 *   out       [n, Hq, d] in `out_dt`, written; with out_dt = MSA_F32 it may
 *             alias o_parts[0] (in-place running accumulation)
 *   lse       [Hq, n] fp32, written; may alias lse_parts[0]
 * Errors: INVALID_ARG for null arrays/pointers, misalignment, n_parts < 1
 * or > MSA_MAX_MERGE_PARTS, n < 1, Hq < 1, d < 4 or d % 4 != 0, or an
 * alias that is not allowed.
 */
msa_status msa_lse_merge(const float *const *o_parts,
                         const float *const *lse_parts, int n_parts,
                         void *out, float *lse, int64_t n, int Hq, int d,
                         msa_dtype out_dt, msa_stream_t stream);

/*
 * 1 in the bounds-checked build of the library (compiled with
 * -DMSA_DEBUG_BOUNDS, shipped as libmsa_debug.so), 0 in the normal one.  In
 * the bounds-checked build every kernel tests each computed global offset
 * against the extent the entry point's contract gives that buffer, and each
 * TMA box origin against its tensor (x 16-byte aligned and inside the row,
 * head in range, box overlapping the rows).  A violation records
 * MSA_ERR_INVALID_ARG in the device status word (msa_device_status), prints
 * the source line once, and the access is skipped (a TMA copy is still
 * issued: out-of-range rows only read the fill value); nothing traps.  The
 * results are otherwise those of the normal build, more slowly.
 */
int msa_debug_bounds_build(void);

/*
 * Which attention kernel msa_attn_fwd, msa_attn_fwd_partial,
 * msa_attn_fwd_band, msa_attn_fwd_rows and msa_attn_fwd_host run for these
 * arguments: 1 = a tensor-core kernel (TMA + tcgen05), 0 = the CUDA-core
 * kernel (fp32 FFMA).  The tensor-core kernels take bf16 inputs with
 * d = 128; fp32 inputs, and bf16 with d = 64, run on CUDA cores (many
 * times slower for bf16).
 */
int msa_attn_uses_tensor_cores(int Hq, int Hkv, int d, msa_dtype in_dt);

/*
 * The same for msa_attn_fwd_topk and msa_attn_fwd_topk_noalloc, whose
 * attention also needs the key block n / n_landmarks to be a whole number
 * of 128-key tiles: 1 = tensor cores, 0 = CUDA cores (also for
 * n_landmarks < 1 or n < n_landmarks, which the call itself refuses).
 */
int msa_attn_fwd_topk_uses_tensor_cores(int64_t n, int Hq, int Hkv, int d,
                                        int n_landmarks, msa_dtype in_dt);

/*
 * Reads (and, if `clear` is nonzero, resets) the status word that the
 * kernels of this library set on the current device when a bounded wait
 * runs out.  Synchronises the device.  Returns MSA_OK, MSA_ERR_TIMEOUT, or
 * MSA_ERR_CUDA if the read itself failed.
 */
msa_status msa_device_status(int clear);

/*
 * Test hook: sets the limit, in nanoseconds, of every bounded wait in the
 * tensor-core kernels for launches made after the call (0 restores the
 * default of 4 s).  A very small limit makes waits run out on purpose, to
 * check that a kernel then finishes early with MSA_ERR_TIMEOUT instead of
 * hanging; with a limit of 1 ns every wait that its first, non-blocking
 * probe does not find complete runs out.  Copies and MMAs already in flight
 * are still waited for with the default limit before a kernel exits.
 */
void msa_debug_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook: with `on` nonzero, launches made after the call run the
 * single-CTA tensor-core kernels even where a CTA-pair kernel applies -- the
 * attention forward (bf16, d = 128, at least two query heads per KV head)
 * and the dQ kernel of msa_attn_bwd (an even number of query heads per KV
 * head) -- so that tests can compare the two; 0 restores the normal
 * choice.  Each pair kernel computes the same arithmetic in the same order
 * as its single-CTA form and gives the same bits.
 */
void msa_debug_force_single_cta(int on);

/*
 * Test hook: with n > 0, launches made after the call run the persistent
 * CTA-pair kernels (the attention forward and the dQ kernel of
 * msa_attn_bwd) on at most n CTA pairs instead of as many as fit on the
 * device, so that each pair works through many units in turn; 0 (or a
 * negative n) restores the normal grid.  Results do not depend on the
 * grid: every unit computes the same arithmetic whichever pair takes it.
 */
void msa_debug_set_max_clusters(int n);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
