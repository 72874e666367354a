/*
 * mla.h — C ABI of libmla.so: Multi-head Latent Attention (MLA) over a latent KV cache,
 * hand-written CUDA for sm_103a (B300).
 *
 * Sources of the operations (page title, section):
 *   [notes]  "MLA前向计算流程" (deepseek-tech-notes, 02-MLA低秩注意力):
 *            §符号 (dimension names), §流程图 (matrix shapes, cache contents),
 *            §三分支计算 ① Query ② Key ③ Value ④ 注意力与输出, §KV Cache 里到底存什么,
 *            V3.1 Hybrid remark (prefill expands K/V per head, decode shares the latent).
 *   [llama]  "从LLaMA到DeepSeek[01] - MLA（上）": §六 (weight absorption by associativity),
 *            §七 (absorption makes per-head products 4x wider; worth it because decode is
 *            memory bound; prefill expands K/V instead).
 *   [atyun]  "多头潜在注意力" article on atyun.com: §RoPE (rotate consecutive pairs),
 *            §多头潜在注意力 (decoupled RoPE key shared by all heads).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor is caller-owned DEVICE memory unless stated otherwise; the library never
 *    allocates device memory. Scratch space is the caller's `ws` buffer, sized by the
 *    matching *_workspace_size query.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *    Host-side validation happens before any launch: a non-MLA_OK status means nothing was
 *    launched. Conditions only visible on the device (an out-of-range cache row, a sequence
 *    length above max_len, a bounded wait that gave up) set a device status word that
 *    mla_get_device_status() reads and clears.
 *  - Matrices are stored [out, in] row-major and applied as y = W x ([notes] §流程图:
 *    W^UQ is [n_h*d_h^C, d_c'], W^QR is [n_h*d_h^R, d_c'], W^KR is [d_h^R, d]).
 *    The head-i block of W^UQ, W^UK and W^UV is rows i*d_h^C..(i+1)*d_h^C-1; the head-i block
 *    of W^QR is rows i*d_h^R..(i+1)*d_h^R-1.
 *  - RoPE rotates consecutive pairs (2k, 2k+1) by pos * rope_base^(-2k/d_h^R), positions
 *    0-based ([atyun] §RoPE; the frequency schedule is the standard one).
 *  - dtype: MLA_BF16 means weights, hidden states, the latent cache and q_c/q_r are bfloat16;
 *    MLA_F32 means all of them are float32. Outputs o are float32 in both cases.
 *  - Pointers to bf16 data must be 16-byte aligned (MLA_ERR_MISALIGNED otherwise); float32
 *    data must be 16-byte aligned too.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent dims          */
  MLA_ERR_UNSUPPORTED = 2,   /* dims outside what the kernels implement                 */
  MLA_ERR_CAPACITY = 3,      /* (device) a cache row index fell outside [0, capacity)   */
  MLA_ERR_MISALIGNED = 4,    /* a pointer is not 16-byte aligned                         */
  MLA_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed                        */
  MLA_ERR_TIMEOUT = 6,       /* (device) a bounded wait inside a kernel gave up          */
  MLA_ERR_WORKSPACE = 7,     /* ws is null or smaller than the workspace query demands   */
  MLA_ERR_LENGTH = 8         /* (device) a sequence length exceeded max_len / max_T      */
} mla_status_t;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype_t;

/* Dimensions in the notation of [notes] §符号. */
typedef struct {
  int32_t d;        /* hidden width d                                  (V2: 5120) */
  int32_t n_h;      /* heads n_h                                       (V2: 128)  */
  int32_t d_hc;     /* per-head content width d_h^C                    (V2: 128)  */
  int32_t d_hr;     /* decoupled RoPE width d_h^R, even                (V2: 64)   */
  int32_t d_c;      /* KV joint latent rank d_c                        (V2: 512)  */
  int32_t d_cq;     /* query latent rank d_c'                          (V2: 1536) */
  float rope_base;  /* RoPE base, e.g. 10000                                     */
  float scale;      /* softmax scale; 0 selects 1/sqrt(d_h^C + d_h^R) ([notes] ④) */
  int32_t dtype;    /* mla_dtype_t                                               */
} mla_dims_t;

/* The seven projection matrices, device pointers, each [out, in] row-major:
 *   W_DQ [d_c', d], W_UQ [n_h*d_h^C, d_c'], W_QR [n_h*d_h^R, d_c'],
 *   W_DKV [d_c, d], W_KR [d_h^R, d], W_UK [n_h*d_h^C, d_c], W_UV [n_h*d_h^C, d_c].
 * A call only reads the matrices its formula uses; the others may be NULL. */
typedef struct {
  const void* W_DQ;
  const void* W_UQ;
  const void* W_QR;
  const void* W_DKV;
  const void* W_KR;
  const void* W_UK;
  const void* W_UV;
} mla_weights_t;

/* The latent cache ([notes] §KV Cache 里到底存什么): one row of d_c + d_h^R values per token,
 * [c^KV_t ; k^R_t], shared by all heads. Sequence b's token at position p lives in row
 * seq_base[b] + p. Rows are contiguous with a pitch of (d_c + d_h^R) elements. */
typedef struct {
  void* rows;               /* [capacity, d_c + d_h^R], dtype per dims                  */
  const int64_t* seq_base;  /* [B] device: first row of each sequence                   */
  int64_t capacity;         /* number of rows in `rows`                                 */
} mla_cache_t;

/* Append tokens to the latent cache ([notes] §三分支计算 ② Key, ③ Value):
 *   c^KV_t = W^DKV h_t,   k^R_t = RoPE(W^KR h_t) at position pos[t],
 *   row seq_base[seq_idx[t]] + pos[t]  <-  [c^KV_t ; k^R_t]   (fp32 accumulation, stored in dtype).
 * h [n, d]; seq_idx [n] and pos [n] are device int32 arrays. Uses W_DKV and W_KR.
 * Rows outside [0, capacity) are skipped and flag MLA_ERR_CAPACITY on the device. */
mla_status_t mla_append_cache(const mla_dims_t* dims, const mla_weights_t* w, const void* h,
                              const int32_t* seq_idx, const int32_t* pos, int32_t n,
                              mla_cache_t* cache, void* stream);

/* Workspace needed by mla_project_q for n tokens. */
mla_status_t mla_project_q_workspace_size(const mla_dims_t* dims, int32_t n, size_t* bytes);

/* Query projection ([notes] §三分支计算 ① Query):
 *   c^Q = W^DQ h,  q^C = W^UQ c^Q split per head,  q^R = RoPE(W^QR c^Q) per head at pos[t].
 * h [n, d]; pos [n] device int32; outputs q_c [n, n_h, d_h^C] and q_r [n, n_h, d_h^R] in dtype.
 * q^R is per head ([notes] §流程图 gives q^R as [128, 64]). c^Q is kept in ws above bf16
 * precision. Uses W_DQ, W_UQ, W_QR. */
mla_status_t mla_project_q(const mla_dims_t* dims, const mla_weights_t* w, const void* h,
                           const int32_t* pos, int32_t n, void* ws, size_t ws_bytes,
                           void* q_c, void* q_r, void* stream);

/* Workspace needed by mla_decode_absorbed for B sequences of at most max_len rows. */
mla_status_t mla_decode_workspace_size(const mla_dims_t* dims, int32_t B, int32_t max_len,
                                       size_t* bytes);

/* Weight-absorbed decode over the latent cache ([llama] §六, [notes] ④ and the V3.1 Hybrid
 * remark), one query token per sequence:
 *   q~_{b,i}  = (W^UK_i)^T q^C_{b,i}                                      (d_c wide)
 *   s_{b,i,j} = (q~_{b,i} . c^KV_j + q^R_{b,i} . k^R_j) * scale,  j = 0..seq_len[b]-1
 *   p = softmax_j(s),  o~_{b,i} = sum_j p_{b,i,j} c^KV_j,  o_{b,i} = W^UV_i o~_{b,i}.
 * The query token's own row is the last attended row (positions 0..seq_len[b]-1, [notes] ④
 * sums j = 1..t). q_c [B, n_h, d_h^C] and q_r [B, n_h, d_h^R] in dtype (RoPE already applied
 * to q_r); seq_len [B] device int32, each in [0, max_len] (0 gives o = 0). Output o
 * [B, n_h, d_h^C] float32. Uses W_UK and W_UV. Sequences are independent; the kernels split
 * long ones across SMs and merge the splits by log-sum-exp. */
mla_status_t mla_decode_absorbed(const mla_dims_t* dims, const mla_weights_t* w,
                                 const void* q_c, const void* q_r, const mla_cache_t* cache,
                                 const int32_t* seq_len, int32_t B, int32_t max_len,
                                 void* ws, size_t ws_bytes, float* o, void* stream);

/* Query projection with the absorption applied ([notes] §三分支计算 ① Query; [llama] §六: W^UQ and
 * W^UK are fixed, so W^UK can be moved onto the query by associativity):
 *   c^Q = W^DQ h,  q~_{t,i} = (W^UK_i)^T (W^UQ_i c^Q)   (d_c wide),  q^R_{t,i} = RoPE(W^QR_i c^Q),
 * without writing q^C to global memory. h [n, d]; pos [n] device int32; outputs q_t
 * [n, n_h, d_c] and q_r [n, n_h, d_h^R] in dtype. Workspace: mla_project_q_workspace_size(n)
 * (c^Q kept above bf16 precision). Uses W_DQ, W_UQ, W_QR, W_UK. Tensor-core path only (V2
 * widths in bf16, mla_fast_path(dims) == 1); other dims return MLA_ERR_UNSUPPORTED. */
mla_status_t mla_project_q_absorbed(const mla_dims_t* dims, const mla_weights_t* w,
                                    const void* h, const int32_t* pos, int32_t n, void* ws,
                                    size_t ws_bytes, void* q_t, void* q_r, void* stream);

/* mla_decode_absorbed for a caller that already holds the absorbed query q~ (for example from
 * mla_project_q_absorbed): q_t [B, n_h, d_c] and q_r [B, n_h, d_h^R] in dtype; the scores,
 * softmax, latent sum and o = W^UV_i o~ are those of mla_decode_absorbed. Workspace:
 * mla_decode_workspace_size(B, max_len). Uses W_UV only. Tensor-core path only; other dims
 * return MLA_ERR_UNSUPPORTED. */
mla_status_t mla_decode_absorbed_latent(const mla_dims_t* dims, const mla_weights_t* w,
                                        const void* q_t, const void* q_r,
                                        const mla_cache_t* cache, const int32_t* seq_len,
                                        int32_t B, int32_t max_len, void* ws, size_t ws_bytes,
                                        float* o, void* stream);

/* Workspace needed by mla_decode_step for B sequences of at most max_len rows. */
mla_status_t mla_decode_step_workspace_size(const mla_dims_t* dims, int32_t B, int32_t max_len,
                                            size_t* bytes);

/* One decode step for B sequences, each with one new token ([notes] §三分支计算 ①–④ with the
 * absorbed decode of [llama] §六): token b of h [B, d] is sequence b's token at position pos[b]
 * (device int32 [B]).
 *   1. the cache row seq_base[b] + pos[b] <- [W^DKV h_b ; RoPE(W^KR h_b)] and c^Q = W^DQ h_b,
 *      in one launch (the three down-projections share their input);
 *   2. q~ and q^R as in mla_project_q_absorbed;
 *   3. the decode of mla_decode_absorbed_latent over seq_len[b] rows (normally pos[b] + 1, so
 *      the new token's own row is the last one attended).
 * Output o [B, n_h, d_h^C] float32. Workspace: mla_decode_step_workspace_size(B, max_len).
 * Uses all seven matrices. Tensor-core path only; other dims return MLA_ERR_UNSUPPORTED (use
 * mla_append_cache, mla_project_q and mla_decode_absorbed). */
mla_status_t mla_decode_step(const mla_dims_t* dims, const mla_weights_t* w, const void* h,
                             const int32_t* pos, mla_cache_t* cache, const int32_t* seq_len,
                             int32_t B, int32_t max_len, void* ws, size_t ws_bytes, float* o,
                             void* stream);

/* Pre-merged absorbed query weights ([llama] §六: W^UQ and W^UK are both fixed, so the
 * product can be formed once, offline): for every head i,
 *   W^UQK_i = (W^UK_i)^T W^UQ_i   [d_c x d_c'],
 * written as W_UQK [n_h*d_c, d_c'] row-major in dtype (head i's block is rows i*d_c ..
 * (i+1)*d_c-1). fp32 accumulation, one rounding to dtype. A one-off: a plain SIMT kernel. At the
 * V2 widths W_UQK is 128*512*1536 values (201 MB in bf16), against 50 MB of W^UQ plus 17 MB of
 * W^UK for the fused two-product path (mla_project_q_absorbed). */
mla_status_t mla_merge_query_absorption(const mla_dims_t* dims, const void* W_UQ,
                                        const void* W_UK, void* W_UQK, void* stream);

/* Query projection with pre-merged weights: c^Q = W^DQ h, q~_{t,i} = W^UQK_i c^Q (one product
 * per head, d_c wide), q^R_{t,i} = RoPE(W^QR_i c^Q). Same inputs, outputs and workspace as
 * mla_project_q_absorbed (q_t [n, n_h, d_c], q_r [n, n_h, d_h^R] in dtype; workspace
 * mla_project_q_workspace_size(n)), with W_UQK from mla_merge_query_absorption in place of
 * W_UQ and W_UK. Uses W_DQ and W_QR from w. Any dims (tensor-core path for the V2 widths in
 * bf16, SIMT otherwise). */
mla_status_t mla_project_q_premerged(const mla_dims_t* dims, const mla_weights_t* w,
                                     const void* W_UQK, const void* h, const int32_t* pos,
                                     int32_t n, void* ws, size_t ws_bytes, void* q_t, void* q_r,
                                     void* stream);

/* Workspace needed by mla_output_projection for n tokens (0 on the SIMT path). */
mla_status_t mla_output_projection_workspace_size(const mla_dims_t* dims, int32_t n,
                                                  size_t* bytes);

/* Output projection ([notes] §三分支计算 ④): u_t = W^O [o_{t,1}; ...; o_{t,n_h}], the per-head
 * outputs of token t concatenated head by head. o [n, n_h, d_h^C] float32 (as mla_decode_* and
 * mla_prefill write it); W_O [d, n_h*d_h^C] row-major in dtype (applied as y = W x); output
 * u [n, d] float32. Accumulation in fp32; on the tensor-core path o enters the MMA as a hi/lo
 * pair of bf16 (o = hi + lo to about 2^-16) held in ws. */
mla_status_t mla_output_projection(const mla_dims_t* dims, const void* W_O, const float* o,
                                   int32_t n, void* ws, size_t ws_bytes, float* u, void* stream);

/* Top-k selection over the latent sequence ([notes] version table, V3.2 + DSA row: MLA is
 * unchanged; an indexer picks top-k positions of the latent sequence and the core attention
 * runs MLA over them). The indexer itself is not defined by the pages: its scores are the
 * caller's input, one float32 per cached position.
 *   scores      [B, score_stride] float32 device, row b valid at positions 0..seq_len[b]-1
 *               (score_stride >= max_len; 4-byte aligned). Scores must not be NaN.
 *   seq_len     [B] device int32, each in [0, max_len] (others flag MLA_ERR_LENGTH and are
 *               clamped).
 *   k           1 .. 2^20.
 *   sel_pos     [B, k] device int32 (output): the positions of the min(k, seq_len[b]) largest
 *               scores of sequence b, in increasing position order; equal scores rank the lower
 *               position first, -0.0 equals +0.0. Entries past sel_count[b] are not written.
 *   sel_count   [B] device int32 (output): min(k, seq_len[b]).
 * The selection is exact (a radix select on the scores' bit patterns), so the result does not
 * depend on the launch configuration. B <= 65535. */
mla_status_t mla_select_topk(const float* scores, int64_t score_stride, const int32_t* seq_len,
                             int32_t B, int32_t max_len, int32_t k, int32_t* sel_pos,
                             int32_t* sel_count, void* stream);

/* Workspace needed by mla_decode_absorbed_sparse for B sequences and k picked rows each. */
mla_status_t mla_decode_sparse_workspace_size(const mla_dims_t* dims, int32_t B, int32_t k,
                                              size_t* bytes);

/* Sparse absorbed decode: mla_select_topk on the caller's scores, then mla_decode_absorbed's
 * computation over the picked rows only, the same picks for every head:
 *   o_{b,i} = W^UV_i sum_{j in S_b} softmax_{j in S_b}(s_{b,i,j}) c^KV_j,  |S_b| = min(k, seq_len[b]).
 * q_c, q_r, cache, seq_len, max_len, o and the weights are as for mla_decode_absorbed; scores,
 * score_stride and k as for mla_select_topk. The picked rows are copied into ws (packed per
 * sequence) and decoded there, so the cache is only read. Rows whose cache index
 * seq_base[b] + position falls outside [0, capacity) flag MLA_ERR_CAPACITY and read as zero.
 * On the tensor-core path (mla_fast_path(dims) == 1), with k >= seq_len[b] for every b, the
 * output equals mla_decode_absorbed's bit for bit. */
mla_status_t mla_decode_absorbed_sparse(const mla_dims_t* dims, const mla_weights_t* w,
                                        const void* q_c, const void* q_r,
                                        const mla_cache_t* cache, const int32_t* seq_len,
                                        int32_t B, int32_t max_len, const float* scores,
                                        int64_t score_stride, int32_t k, void* ws,
                                        size_t ws_bytes, float* o, void* stream);

/* Scratch capacity of mla_decode_absorbed_static, in bytes (32 MiB). */
#define MLA_STATIC_WS_BYTES (32u << 20)

/* mla_decode_absorbed without a caller-provided workspace. The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory themselves, for
 * example a plugin running inside a host framework that owns every device allocation, or a
 * loop that must not call cudaMalloc after start-up because cudaMalloc may synchronise the
 * device. It computes exactly what mla_decode_absorbed computes, with the same kernels, but
 * its scratch is a fixed MLA_STATIC_WS_BYTES array compiled into the library; every GPU that
 * loads the library holds that array until the process exits. The caller still provides
 * q_c, q_r, the cache, seq_len and the output o.
 *  - Problems whose workspace (mla_decode_workspace_size) exceeds MLA_STATIC_WS_BYTES are
 *    rejected with MLA_ERR_WORKSPACE before any launch. At the V2 widths in bf16 the workspace
 *    depends on B alone: up to 31 sequences fit, whatever their lengths. On the SIMT path
 *    (other widths, fp32) it also grows with max_len.
 *  - The first call on a device looks up the array's device address (once per device, with
 *    that device current); make that first call before any stream capture begins. The address
 *    is kept for the life of the process: after the device is reset (cudaDeviceReset, or the
 *    teardown of its primary context) this entry point must not be called again.
 *  - All calls share the one array, which keeps the previous call's contents; the decode
 *    kernels write every scratch byte they later read within the same call (partial results,
 *    their (m, l) and each sequence's slot range), so nothing needs clearing. Calls whose
 *    kernels overlap on the GPU (several streams, several host threads) race on the array:
 *    serialise them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
mla_status_t mla_decode_absorbed_static(const mla_dims_t* dims, const mla_weights_t* w,
                                        const void* q_c, const void* q_r,
                                        const mla_cache_t* cache, const int32_t* seq_len,
                                        int32_t B, int32_t max_len, float* o, void* stream);

/* Workspace needed by mla_prefill for n_tok tokens in B sequences of at most max_T tokens. */
mla_status_t mla_prefill_workspace_size(const mla_dims_t* dims, int32_t n_tok, int32_t B,
                                        int32_t max_T, size_t* bytes);

/* Causal prefill, non-absorbed ([notes] V3.1 Hybrid remark: prefill expands the latent per
 * head, MHA style; [llama] §七): for every token t of sequence b (position p = t - cu_seqlens[b]),
 *   the cache row seq_base[b] + p is written as in mla_append_cache;
 *   q_{t,i} = [q^C_{t,i} ; q^R_{t,i}] as in mla_project_q;
 *   k_{j,i} = [W^UK_i c^KV_j ; k^R_j],  v_{j,i} = W^UV_i c^KV_j, expanded from the stored rows;
 *   o_{t,i} = sum_{j<=p} softmax_j(q_{t,i} . k_{j,i} * scale) v_{j,i}.
 * h [n_tok, d] (sequences packed back to back); cu_seqlens [B+1] device int32 with
 * cu_seqlens[0] = 0 and cu_seqlens[B] = n_tok; every sequence at most max_T tokens.
 * Output o [n_tok, n_h, d_h^C] float32. Uses all seven matrices. */
mla_status_t mla_prefill(const mla_dims_t* dims, const mla_weights_t* w, const void* h,
                         const int32_t* cu_seqlens, int32_t B, int32_t n_tok, int32_t max_T,
                         mla_cache_t* cache, void* ws, size_t ws_bytes, float* o, void* stream);

/* Synchronises `stream`, then returns and clears the device status word (MLA_OK if no kernel
 * flagged anything), or MLA_ERR_CUDA if the stream reports a CUDA error.
 * Debugging aid: with the environment variable MLA_DEBUG set (and not "0") when the library is
 * first used, every kernel launch outside stream capture is followed by a synchronisation of
 * its stream, and a CUDA error or a latched status is printed on stderr with the kernel's name
 * (the status word is not cleared). This serialises the host with the GPU. */
mla_status_t mla_get_device_status(void* stream);

/* Test hook for the bounded device waits (no counterpart on the pages). Arms a one-shot: the
 * next tensor-core decode attention launch (mla_decode_absorbed, mla_decode_absorbed_latent,
 * mla_decode_step or mla_decode_absorbed_static, from any host thread) makes its MMA warp wait
 * for a barrier phase that nothing completes. After limit_ns (1 .. 2e9) the wait gives up, the
 * device status word latches MLA_ERR_TIMEOUT and every CTA stops early, after its TMA copies
 * have landed and its MMAs have completed; that call's output is then undefined. The device
 * stays usable and the next call runs normally. Returns MLA_ERR_INVALID_ARG for limits outside
 * the range. */
mla_status_t mla_debug_arm_wait_timeout(int64_t limit_ns);

/* Static description of a status code. */
const char* mla_status_string(mla_status_t status);

/* Which kernel family serves these dims: 1 = tcgen05/TMA kernels (V2 widths, bf16),
 * 0 = portable SIMT kernels (any widths, fp32 or bf16). For reporting only. */
int32_t mla_fast_path(const mla_dims_t* dims);

/* Launch tracing for measurement (no counterpart on the pages; used to time individual
 * kernels with CUDA events). While armed, each kernel launch the library makes records
 * events[2k] just before and events[2k+1] just after itself on its launch stream, and stores
 * its kernel id in ids[k], for k = 0 .. n_pairs-1; further launches are not recorded.
 * `events` are caller-created cudaEvent_t handles. Host-side state, not thread-safe; arming
 * again resets it. mla_trace_disarm() returns the number of launches recorded. */
mla_status_t mla_trace_arm(void* const* events, int32_t* ids, int32_t n_pairs);
int32_t mla_trace_disarm(void);
const char* mla_kernel_name(int32_t kernel_id);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
