// Internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/mla.h"

namespace mla {

// Kernel ids for launch tracing (names in api.cu).
enum KernelId : int {
  K_APPEND = 0, K_Q_DOWN, K_Q_UP, K_ABSORB, K_DECODE_ATTN, K_DECODE_COMBINE, K_TOKEN_MAP,
  K_PREFILL_APPEND, K_PREFILL_Q_DOWN, K_PREFILL_Q_UP, K_EXPAND_K, K_EXPAND_V, K_PREFILL_ATTN,
  K_DECODE_MERGE, K_UNABSORB, K_Q_ABSORB, K_DOWN, K_OUT_SPLIT, K_OUT_PROJ, K_MERGE_W, K_Q_PREMERGED, K_TOPK, K_GATHER, K_NUM_IDS
};

// Launch tracing (host side): while armed, trace_before/trace_after record caller-owned
// CUDA events around each kernel launch on its stream.
void trace_before(int kernel_id, cudaStream_t st);
void trace_after(cudaStream_t st);

// RAII helper placed around one kernel launch.
struct TraceScope {
  cudaStream_t st;
  TraceScope(int id, cudaStream_t s) : st(s) { trace_before(id, s); }
  ~TraceScope() { trace_after(st); }
};

// Portable SIMT kernels (simt.cu)
mla_status_t simt_append(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                         const int32_t* seq_idx, const int32_t* pos, int n, mla_cache_t* cache,
                         cudaStream_t st);
size_t simt_project_q_ws(const mla_dims_t* d, int n);
mla_status_t simt_project_q(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                            const int32_t* pos, int n, void* ws, void* q_c, void* q_r,
                            cudaStream_t st);
size_t simt_decode_ws(const mla_dims_t* d, int B, int max_len);
size_t simt_decode_smem(const mla_dims_t* d);
mla_status_t simt_decode(const mla_dims_t* d, const mla_weights_t* w, const void* q_c,
                         const void* q_r, const mla_cache_t* cache, const int32_t* seq_len,
                         int B, int max_len, void* ws, float* o, cudaStream_t st);
size_t simt_prefill_ws(const mla_dims_t* d, int n_tok);
size_t simt_prefill_smem(const mla_dims_t* d);
mla_status_t simt_prefill(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                          const int32_t* cu, int B, int n, int max_T, mla_cache_t* cache,
                          void* ws, float* o, cudaStream_t st);

mla_status_t simt_merge_absorption(const mla_dims_t* d, const void* W_UQ, const void* W_UK,
                                   void* W_UQK, cudaStream_t st);
mla_status_t simt_output_projection(const mla_dims_t* d, const void* W_O, const float* o, int n,
                                    float* u, cudaStream_t st);

// Tensor-core kernels (V2 widths, bf16): gemm_tc.cu
size_t tc_output_projection_ws(const mla_dims_t* d, int n);
mla_status_t tc_output_projection(const mla_dims_t* d, const void* W_O, const float* o, int n,
                                  void* ws, float* u, cudaStream_t st);
bool fast_dims(const mla_dims_t* d);
mla_status_t tc_append(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                       const int32_t* seq_idx, const int32_t* pos, int n, mla_cache_t* cache,
                       void* packed, int kid, cudaStream_t st);
mla_status_t tc_down(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                     const int32_t* pos, int n, mla_cache_t* cache, void* cq_hi, void* cq_lo,
                     int kid, cudaStream_t st);
mla_status_t tc_q_down(const mla_dims_t* d, const mla_weights_t* w, const void* h, int n,
                       void* cq_hi, void* cq_lo, int kid, cudaStream_t st);
mla_status_t tc_q_up(const mla_dims_t* d, const mla_weights_t* w, const void* cq_hi,
                     const void* cq_lo, const int32_t* pos, int n, void* q_c, void* q_r,
                     int64_t qc_tok, int64_t qc_head, int64_t qr_tok, int64_t qr_head,
                     bool f16_out, int kid, cudaStream_t st);
mla_status_t tc_absorb(const mla_dims_t* d, const mla_weights_t* w, const void* q_c, int B,
                       void* qt, int kid, cudaStream_t st);

// Fused query up-projection + absorption (V2 widths, bf16): qabsorb_tc.cu
mla_status_t tc_q_absorbed(const mla_dims_t* d, const mla_weights_t* w, const void* cq_hi,
                           const void* cq_lo, const int32_t* pos, int n, void* q_t, void* q_r,
                           cudaStream_t st);

// Tensor-core causal prefill (V2 widths, bf16): prefill_tc.cu
size_t tc_prefill_ws(const mla_dims_t* d, int n_tok);
mla_status_t tc_prefill(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                        const int32_t* cu, int B, int n, int max_T, mla_cache_t* cache, void* ws,
                        float* o, cudaStream_t st);

// Tensor-core absorbed decode (V2 widths, bf16): decode_tc.cu
size_t tc_decode_ws(const mla_dims_t* d, int B);
void arm_decode_wait_timeout(int64_t limit_ns);  // mla_debug_arm_wait_timeout
size_t tc_decode_qt_offset(int B);  // byte offset of the q~ area in the decode workspace
mla_status_t tc_decode(const mla_dims_t* d, const mla_weights_t* w, const void* q_c,
                       const void* q_r, const mla_cache_t* cache, const int32_t* seq_len, int B,
                       int max_len, void* ws, float* o, cudaStream_t st);
// Decode from the absorbed query q~ [B, n_h, d_c] (attention + merge + W^UV): no absorb launch.
// after_q_kernel: the kernel right before it in the stream is the same call's query kernel
// (q~ is its output), so the attention may start early (programmatic dependent launch).
mla_status_t tc_decode_latent(const mla_dims_t* d, const mla_weights_t* w, const void* q_t,
                              const void* q_r, const mla_cache_t* cache, const int32_t* seq_len,
                              int B, int max_len, void* ws, float* o, bool after_q_kernel,
                              cudaStream_t st);
// Top-k selection and row gather for the sparse decode (sparse.cu)
mla_status_t select_topk(const float* scores, int64_t stride, const int32_t* seq_len, int B,
                         int max_len, int k, int32_t* sel_pos, int32_t* sel_count,
                         int64_t* packed_base, cudaStream_t st);
mla_status_t gather_rows(const mla_dims_t* d, const mla_cache_t* cache, const int32_t* sel_pos,
                         const int32_t* sel_count, int B, int k, void* packed, cudaStream_t st);
mla_status_t tc_expand(const void* W, int O, const void* latent, int64_t ld_latent, int K, int n,
                       void* y, bool f16_out, int kid, cudaStream_t st);

}  // namespace mla
