// C ABI of libmla: argument validation, workspace sizing and dispatch to the kernel files.
// The operations are those of "MLA前向计算流程" §三分支计算 ①–④ (see include/mla.h).
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

using namespace mla;

namespace {

mla_status_t check_dims(const mla_dims_t* d) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->d <= 0 || d->n_h <= 0 || d->d_hc <= 0 || d->d_hr <= 0 || d->d_c <= 0 || d->d_cq <= 0)
    return MLA_ERR_INVALID_ARG;
  if (d->dtype != MLA_F32 && d->dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (!(d->rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  // RoPE rotates pairs; the pair-wise epilogues need even content widths too.
  if ((d->d_hr & 1) || (d->d_c & 1) || (d->d_hc & 1)) return MLA_ERR_UNSUPPORTED;
  if (d->d_hr > 2 * kMaxRopePairs) return MLA_ERR_UNSUPPORTED;
  // vectorised row access: 16-byte row pitches of the cache and of every weight row
  const int v = d->dtype == MLA_BF16 ? 8 : 4;
  if ((d->d_c + d->d_hr) % v || d->d % v || d->d_cq % v || d->d_c % v) return MLA_ERR_UNSUPPORTED;
  // SIMT kernels stage a handful of rows in shared memory
  if (simt_decode_smem(d) > 200 * 1024 || simt_prefill_smem(d) > 200 * 1024)
    return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

mla_status_t check_ptr(const void* p) {
  if (!p) return MLA_ERR_INVALID_ARG;
  return aligned16(p) ? MLA_OK : MLA_ERR_MISALIGNED;
}

#define MLA_TRY(x)                       \
  do {                                   \
    mla_status_t s_ = (x);               \
    if (s_ != MLA_OK) return s_;         \
  } while (0)

}  // namespace

namespace mla {
// The tensor-core kernels are specialised to the DeepSeek-V2 head widths (n_h 128, d_h^C 128,
// d_h^R 64, d_c 512) in bf16; d and d_c' only need to be multiples of 64 / 128.
bool fast_dims(const mla_dims_t* d) {
  return d->dtype == MLA_BF16 && d->n_h == 128 && d->d_hc == 128 && d->d_hr == 64 &&
         d->d_c == 512 && d->d % 64 == 0 && d->d_cq % 128 == 0;
}
}  // namespace mla

// ------------------------------------------------------------------ launch tracing
namespace mla {
namespace {
struct TraceState {
  void* const* events = nullptr;
  int32_t* ids = nullptr;
  int32_t n_pairs = 0;
  int32_t count = 0;
  bool armed = false;
};
TraceState g_trace;
const char* const kKernelNames[K_NUM_IDS] = {
    "append", "q_down", "q_up", "absorb", "decode_attn", "decode_combine", "token_map",
    "prefill_append", "prefill_q_down", "prefill_q_up", "expand_k", "expand_v", "prefill_attn",
    "decode_merge", "unabsorb", "q_absorb", "down", "out_split", "out_proj", "merge_w",
    "q_premerged", "topk_select", "gather_rows"};
}  // namespace

namespace {
// MLA_DEBUG (set and not "0", read once per process): after every kernel launch of the library
// outside stream capture, wait for the stream and report a CUDA error or a latched device
// status on stderr with the kernel's name. It serialises the host with the GPU: for debugging.
bool debug_launches() {
  static const bool on = [] {
    const char* e = getenv("MLA_DEBUG");
    return e && *e && strcmp(e, "0") != 0;
  }();
  return on;
}
thread_local int t_last_kernel = -1;

void debug_check(cudaStream_t st) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return;
  const char* name =
      (t_last_kernel >= 0 && t_last_kernel < K_NUM_IDS) ? kKernelNames[t_last_kernel] : "?";
  const cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    fprintf(stderr, "mla: after %s: %s\n", name, cudaGetErrorString(e));
    return;
  }
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) == cudaSuccess && v != 0)
    fprintf(stderr, "mla: after %s: device status %u (%s)\n", name, v,
            mla_status_string((mla_status_t)v));
}
}  // namespace

void trace_before(int kernel_id, cudaStream_t st) {
  t_last_kernel = kernel_id;
  if (!g_trace.armed || g_trace.count >= g_trace.n_pairs) return;
  g_trace.ids[g_trace.count] = kernel_id;
  cudaEventRecord((cudaEvent_t)g_trace.events[2 * g_trace.count], st);
}

void trace_after(cudaStream_t st) {
  if (debug_launches()) debug_check(st);
  if (!g_trace.armed || g_trace.count >= g_trace.n_pairs) return;
  cudaEventRecord((cudaEvent_t)g_trace.events[2 * g_trace.count + 1], st);
  ++g_trace.count;
}
}  // namespace mla

extern "C" {

mla_status_t mla_trace_arm(void* const* events, int32_t* ids, int32_t n_pairs) {
  if (n_pairs < 0 || (n_pairs > 0 && (!events || !ids))) return MLA_ERR_INVALID_ARG;
  g_trace.events = events;
  g_trace.ids = ids;
  g_trace.n_pairs = n_pairs;
  g_trace.count = 0;
  g_trace.armed = n_pairs > 0;
  return MLA_OK;
}

int32_t mla_trace_disarm(void) {
  const int32_t n = g_trace.count;
  g_trace = TraceState();
  return n;
}

const char* mla_kernel_name(int32_t id) {
  return (id >= 0 && id < K_NUM_IDS) ? kKernelNames[id] : "unknown";
}

int32_t mla_fast_path(const mla_dims_t* d) {
  if (check_dims(d) != MLA_OK) return 0;
  return fast_dims(d) ? 1 : 0;
}

mla_status_t mla_append_cache(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                              const int32_t* seq_idx, const int32_t* pos, int32_t n,
                              mla_cache_t* cache, void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || !cache || n < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!seq_idx || !pos || !cache->seq_base || cache->capacity < 0) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(h));
  MLA_TRY(check_ptr(w->W_DKV));
  MLA_TRY(check_ptr(w->W_KR));
  MLA_TRY(check_ptr(cache->rows));
  if (fast_dims(d))
    return tc_append(d, w, h, seq_idx, pos, n, cache, nullptr, K_APPEND, as_stream(stream));
  return simt_append(d, w, h, seq_idx, pos, n, cache, as_stream(stream));
}

mla_status_t mla_project_q_workspace_size(const mla_dims_t* d, int32_t n, size_t* bytes) {
  MLA_TRY(check_dims(d));
  if (!bytes || n < 0) return MLA_ERR_INVALID_ARG;
  // fast path: c^Q as a hi/lo pair of bf16 matrices [n, d_c'] (c^Q = hi + lo to ~2^-16)
  *bytes = fast_dims(d) ? 2 * align_up((size_t)n * d->d_cq * 2, 256) : simt_project_q_ws(d, n);
  return MLA_OK;
}

mla_status_t mla_project_q(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                           const int32_t* pos, int32_t n, void* ws, size_t ws_bytes, void* q_c,
                           void* q_r, void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || n < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!pos) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(h));
  MLA_TRY(check_ptr(w->W_DQ));
  MLA_TRY(check_ptr(w->W_UQ));
  MLA_TRY(check_ptr(w->W_QR));
  MLA_TRY(check_ptr(q_c));
  MLA_TRY(check_ptr(q_r));
  size_t need = 0;
  MLA_TRY(mla_project_q_workspace_size(d, n, &need));
  if (need && (!ws || ws_bytes < need)) return MLA_ERR_WORKSPACE;
  if (need) MLA_TRY(check_ptr(ws));
  if (fast_dims(d)) {
    char* hi = (char*)ws;
    char* lo = hi + align_up((size_t)n * d->d_cq * 2, 256);
    MLA_TRY(tc_q_down(d, w, h, n, hi, lo, K_Q_DOWN, as_stream(stream)));
    return tc_q_up(d, w, hi, lo, pos, n, q_c, q_r, (int64_t)d->n_h * d->d_hc, d->d_hc,
                   (int64_t)d->n_h * d->d_hr, d->d_hr, false, K_Q_UP, as_stream(stream));
  }
  return simt_project_q(d, w, h, pos, n, ws, q_c, q_r, as_stream(stream));
}

mla_status_t mla_decode_workspace_size(const mla_dims_t* d, int32_t B, int32_t max_len,
                                       size_t* bytes) {
  MLA_TRY(check_dims(d));
  if (!bytes || B < 0 || max_len < 0) return MLA_ERR_INVALID_ARG;
  *bytes = fast_dims(d) ? tc_decode_ws(d, B) : simt_decode_ws(d, B, max_len);
  return MLA_OK;
}

mla_status_t mla_decode_absorbed(const mla_dims_t* d, const mla_weights_t* w, const void* q_c,
                                 const void* q_r, const mla_cache_t* cache,
                                 const int32_t* seq_len, int32_t B, int32_t max_len, void* ws,
                                 size_t ws_bytes, float* o, void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || !cache || B < 0 || max_len < 0) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!seq_len || !cache->seq_base || cache->capacity < 0) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(q_c));
  MLA_TRY(check_ptr(q_r));
  MLA_TRY(check_ptr(w->W_UK));
  MLA_TRY(check_ptr(w->W_UV));
  MLA_TRY(check_ptr(o));
  if (max_len > 0) MLA_TRY(check_ptr(cache->rows));
  size_t need = 0;
  MLA_TRY(mla_decode_workspace_size(d, B, max_len, &need));
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  MLA_TRY(check_ptr(ws));
  if (fast_dims(d))
    return tc_decode(d, w, q_c, q_r, cache, seq_len, B, max_len, ws, o, as_stream(stream));
  return simt_decode(d, w, q_c, q_r, cache, seq_len, B, max_len, ws, o, as_stream(stream));
}

mla_status_t mla_project_q_absorbed(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                                    const int32_t* pos, int32_t n, void* ws, size_t ws_bytes,
                                    void* q_t, void* q_r, void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || n < 0) return MLA_ERR_INVALID_ARG;
  if (!fast_dims(d)) return MLA_ERR_UNSUPPORTED;
  if (n == 0) return MLA_OK;
  if (!pos) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(h));
  const void* mats[] = {w->W_DQ, w->W_UQ, w->W_QR, w->W_UK};
  for (const void* p : mats) MLA_TRY(check_ptr(p));
  MLA_TRY(check_ptr(q_t));
  MLA_TRY(check_ptr(q_r));
  size_t need = 0;
  MLA_TRY(mla_project_q_workspace_size(d, n, &need));
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  MLA_TRY(check_ptr(ws));
  char* hi = (char*)ws;
  char* lo = hi + align_up((size_t)n * d->d_cq * 2, 256);
  MLA_TRY(tc_q_down(d, w, h, n, hi, lo, K_Q_DOWN, as_stream(stream)));
  return tc_q_absorbed(d, w, hi, lo, pos, n, q_t, q_r, as_stream(stream));
}

mla_status_t mla_decode_absorbed_latent(const mla_dims_t* d, const mla_weights_t* w,
                                        const void* q_t, const void* q_r,
                                        const mla_cache_t* cache, const int32_t* seq_len,
                                        int32_t B, int32_t max_len, void* ws, size_t ws_bytes,
                                        float* o, void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || !cache || B < 0 || max_len < 0) return MLA_ERR_INVALID_ARG;
  if (!fast_dims(d)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!seq_len || !cache->seq_base || cache->capacity < 0) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(q_t));
  MLA_TRY(check_ptr(q_r));
  MLA_TRY(check_ptr(w->W_UV));
  MLA_TRY(check_ptr(o));
  if (max_len > 0) MLA_TRY(check_ptr(cache->rows));
  size_t need = 0;
  MLA_TRY(mla_decode_workspace_size(d, B, max_len, &need));
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  MLA_TRY(check_ptr(ws));
  return tc_decode_latent(d, w, q_t, q_r, cache, seq_len, B, max_len, ws, o, false,
                          as_stream(stream));
}

namespace {
// Decode-step workspace: the decode workspace (its q~ area holds the absorbed query), then c^Q
// hi, c^Q lo [B, d_c'] and q^R [B, n_h, d_h^R].
struct StepLayout {
  size_t off_hi, off_lo, off_qr, total;
};
StepLayout step_layout(const mla_dims_t* d, int B) {
  StepLayout L;
  L.off_hi = align_up(tc_decode_ws(d, B), 256);
  L.off_lo = align_up(L.off_hi + (size_t)B * d->d_cq * 2, 256);
  L.off_qr = align_up(L.off_lo + (size_t)B * d->d_cq * 2, 256);
  L.total = align_up(L.off_qr + (size_t)B * d->n_h * d->d_hr * 2, 256);
  return L;
}
}  // namespace

mla_status_t mla_decode_step_workspace_size(const mla_dims_t* d, int32_t B, int32_t max_len,
                                            size_t* bytes) {
  MLA_TRY(check_dims(d));
  if (!bytes || B < 0 || max_len < 0) return MLA_ERR_INVALID_ARG;
  if (!fast_dims(d)) return MLA_ERR_UNSUPPORTED;
  *bytes = step_layout(d, B).total;
  return MLA_OK;
}

mla_status_t mla_decode_step(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                             const int32_t* pos, mla_cache_t* cache, const int32_t* seq_len,
                             int32_t B, int32_t max_len, void* ws, size_t ws_bytes, float* o,
                             void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || !cache || B < 0 || max_len < 0) return MLA_ERR_INVALID_ARG;
  if (!fast_dims(d)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!pos || !seq_len || !cache->seq_base || cache->capacity < 0) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(h));
  const void* mats[] = {w->W_DQ, w->W_UQ, w->W_QR, w->W_DKV, w->W_KR, w->W_UK, w->W_UV};
  for (const void* p : mats) MLA_TRY(check_ptr(p));
  MLA_TRY(check_ptr(cache->rows));
  MLA_TRY(check_ptr(o));
  size_t need = 0;
  MLA_TRY(mla_decode_step_workspace_size(d, B, max_len, &need));
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  MLA_TRY(check_ptr(ws));
  const StepLayout L = step_layout(d, B);
  char* wsb = (char*)ws;
  cudaStream_t st = as_stream(stream);
  MLA_TRY(tc_down(d, w, h, pos, B, cache, wsb + L.off_hi, wsb + L.off_lo, K_DOWN, st));
  void* q_t = wsb + tc_decode_qt_offset(B);
  MLA_TRY(tc_q_absorbed(d, w, wsb + L.off_hi, wsb + L.off_lo, pos, B, q_t, wsb + L.off_qr, st));
  return tc_decode_latent(d, w, q_t, wsb + L.off_qr, cache, seq_len, B, max_len, ws, o, true,
                          st);
}

mla_status_t mla_prefill_workspace_size(const mla_dims_t* d, int32_t n_tok, int32_t B,
                                        int32_t max_T, size_t* bytes) {
  MLA_TRY(check_dims(d));
  if (!bytes || n_tok < 0 || B < 0 || max_T < 0) return MLA_ERR_INVALID_ARG;
  *bytes = fast_dims(d) ? tc_prefill_ws(d, n_tok) : simt_prefill_ws(d, n_tok);
  return MLA_OK;
}

mla_status_t mla_prefill(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                         const int32_t* cu_seqlens, int32_t B, int32_t n_tok, int32_t max_T,
                         mla_cache_t* cache, void* ws, size_t ws_bytes, float* o,
                         void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || !cache || B < 0 || n_tok < 0 || max_T < 0) return MLA_ERR_INVALID_ARG;
  if (n_tok == 0 || B == 0) return MLA_OK;
  if (!cu_seqlens || !cache->seq_base || cache->capacity < 0) return MLA_ERR_INVALID_ARG;
  if ((int64_t)max_T * B < n_tok) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(h));
  const void* mats[] = {w->W_DQ, w->W_UQ, w->W_QR, w->W_DKV, w->W_KR, w->W_UK, w->W_UV};
  for (const void* p : mats) MLA_TRY(check_ptr(p));
  MLA_TRY(check_ptr(cache->rows));
  MLA_TRY(check_ptr(o));
  size_t need = 0;
  MLA_TRY(mla_prefill_workspace_size(d, n_tok, B, max_T, &need));
  if (!ws || ws_bytes < need) return MLA_ERR_WORKSPACE;
  MLA_TRY(check_ptr(ws));
  if (fast_dims(d))
    return tc_prefill(d, w, h, cu_seqlens, B, n_tok, max_T, cache, ws, o, as_stream(stream));
  return simt_prefill(d, w, h, cu_seqlens, B, n_tok, max_T, cache, ws, o, as_stream(stream));
}

mla_status_t mla_get_device_status(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return MLA_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return (mla_status_t)v;
}

mla_status_t mla_merge_query_absorption(const mla_dims_t* d, const void* W_UQ, const void* W_UK,
                                        void* W_UQK, void* stream) {
  MLA_TRY(check_dims(d));
  MLA_TRY(check_ptr(W_UQ));
  MLA_TRY(check_ptr(W_UK));
  MLA_TRY(check_ptr(W_UQK));
  return simt_merge_absorption(d, W_UQ, W_UK, W_UQK, as_stream(stream));
}

mla_status_t mla_project_q_premerged(const mla_dims_t* d, const mla_weights_t* w,
                                     const void* W_UQK, const void* h, const int32_t* pos,
                                     int32_t n, void* ws, size_t ws_bytes, void* q_t, void* q_r,
                                     void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || n < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!pos) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_ptr(h));
  MLA_TRY(check_ptr(w->W_DQ));
  MLA_TRY(check_ptr(w->W_QR));
  MLA_TRY(check_ptr(W_UQK));
  MLA_TRY(check_ptr(q_t));
  MLA_TRY(check_ptr(q_r));
  size_t need = 0;
  MLA_TRY(mla_project_q_workspace_size(d, n, &need));
  if (need && (!ws || ws_bytes < need)) return MLA_ERR_WORKSPACE;
  if (need) MLA_TRY(check_ptr(ws));
  // the merged matrix gives each head d_c query columns instead of d_h^C: the query
  // up-projection with that width and W^UQK in place of W^UQ
  mla_dims_t dm = *d;
  dm.d_hc = d->d_c;
  mla_weights_t wm = *w;
  wm.W_UQ = W_UQK;
  cudaStream_t st = as_stream(stream);
  if (fast_dims(d)) {
    char* hi = (char*)ws;
    char* lo = hi + align_up((size_t)n * d->d_cq * 2, 256);
    MLA_TRY(tc_q_down(d, w, h, n, hi, lo, K_Q_DOWN, st));
    return tc_q_up(&dm, &wm, hi, lo, pos, n, q_t, q_r, (int64_t)d->n_h * d->d_c, d->d_c,
                   (int64_t)d->n_h * d->d_hr, d->d_hr, false, K_Q_PREMERGED, st);
  }
  return simt_project_q(&dm, &wm, h, pos, n, ws, q_t, q_r, st);
}

mla_status_t mla_output_projection_workspace_size(const mla_dims_t* d, int32_t n, size_t* bytes) {
  MLA_TRY(check_dims(d));
  if (!bytes || n < 0) return MLA_ERR_INVALID_ARG;
  *bytes = fast_dims(d) ? tc_output_projection_ws(d, n) : 0;
  return MLA_OK;
}

mla_status_t mla_output_projection(const mla_dims_t* d, const void* W_O, const float* o,
                                   int32_t n, void* ws, size_t ws_bytes, float* u,
                                   void* stream) {
  MLA_TRY(check_dims(d));
  if (n < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  MLA_TRY(check_ptr(W_O));
  MLA_TRY(check_ptr(o));
  MLA_TRY(check_ptr(u));
  size_t need = 0;
  MLA_TRY(mla_output_projection_workspace_size(d, n, &need));
  if (need && (!ws || ws_bytes < need)) return MLA_ERR_WORKSPACE;
  if (need) MLA_TRY(check_ptr(ws));
  if (fast_dims(d)) return tc_output_projection(d, W_O, o, n, ws, u, as_stream(stream));
  return simt_output_projection(d, W_O, o, n, u, as_stream(stream));
}

namespace {
// Sparse-decode workspace: picked positions [B, k] int32, their counts [B] int32, the packed
// cache's row bases [B] int64, the packed rows [B * k, d_c + d_h^R], then the decode workspace
// of B sequences of at most k rows.
struct SparseLayout {
  size_t off_count, off_base, off_rows, off_dec, total;
};
SparseLayout sparse_layout(const mla_dims_t* d, int B, int k) {
  SparseLayout L;
  const size_t row_bytes = (size_t)(d->d_c + d->d_hr) * elem_bytes(d);
  L.off_count = align_up((size_t)B * k * 4, 256);
  L.off_base = L.off_count + align_up((size_t)B * 4, 256);
  L.off_rows = L.off_base + align_up((size_t)B * 8, 256);
  L.off_dec = L.off_rows + align_up((size_t)B * k * row_bytes, 256);
  L.total = L.off_dec + (fast_dims(d) ? tc_decode_ws(d, B) : simt_decode_ws(d, B, k));
  return L;
}
constexpr int32_t kMaxTopK = 1 << 20;
}  // namespace

mla_status_t mla_select_topk(const float* scores, int64_t score_stride, const int32_t* seq_len,
                             int32_t B, int32_t max_len, int32_t k, int32_t* sel_pos,
                             int32_t* sel_count, void* stream) {
  if (B < 0 || max_len < 0 || k < 1 || k > kMaxTopK || B > 65535) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!scores || !seq_len || !sel_pos || !sel_count || score_stride < max_len)
    return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scores) & 3u) || (reinterpret_cast<uintptr_t>(sel_pos) & 3u) ||
      (reinterpret_cast<uintptr_t>(sel_count) & 3u))
    return MLA_ERR_MISALIGNED;
  return select_topk(scores, score_stride, seq_len, B, max_len, k, sel_pos, sel_count, nullptr,
                     as_stream(stream));
}

mla_status_t mla_decode_sparse_workspace_size(const mla_dims_t* d, int32_t B, int32_t k,
                                              size_t* bytes) {
  MLA_TRY(check_dims(d));
  if (!bytes || B < 0 || k < 1 || k > kMaxTopK) return MLA_ERR_INVALID_ARG;
  *bytes = sparse_layout(d, B, k).total;
  return MLA_OK;
}

mla_status_t mla_decode_absorbed_sparse(const mla_dims_t* d, const mla_weights_t* w,
                                        const void* q_c, const void* q_r,
                                        const mla_cache_t* cache, const int32_t* seq_len,
                                        int32_t B, int32_t max_len, const float* scores,
                                        int64_t score_stride, int32_t k, void* ws,
                                        size_t ws_bytes, float* o, void* stream) {
  MLA_TRY(check_dims(d));
  if (!w || !cache || B < 0 || max_len < 0 || k < 1 || k > kMaxTopK || B > 65535)
    return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!seq_len || !cache->seq_base || cache->capacity < 0 || !scores || score_stride < max_len)
    return MLA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(scores) & 3u) return MLA_ERR_MISALIGNED;
  MLA_TRY(check_ptr(q_c));
  MLA_TRY(check_ptr(q_r));
  MLA_TRY(check_ptr(w->W_UK));
  MLA_TRY(check_ptr(w->W_UV));
  MLA_TRY(check_ptr(o));
  if (max_len > 0) MLA_TRY(check_ptr(cache->rows));
  const SparseLayout L = sparse_layout(d, B, k);
  if (!ws || ws_bytes < L.total) return MLA_ERR_WORKSPACE;
  MLA_TRY(check_ptr(ws));
  char* base = (char*)ws;
  int32_t* sel = reinterpret_cast<int32_t*>(base);
  int32_t* count = reinterpret_cast<int32_t*>(base + L.off_count);
  int64_t* pbase = reinterpret_cast<int64_t*>(base + L.off_base);
  const cudaStream_t st = as_stream(stream);
  MLA_TRY(select_topk(scores, score_stride, seq_len, B, max_len, k, sel, count, pbase, st));
  MLA_TRY(gather_rows(d, cache, sel, count, B, k, base + L.off_rows, st));
  mla_cache_t packed{base + L.off_rows, pbase, (int64_t)B * k};
  const int kmax = max_len < k ? max_len : k;
  if (fast_dims(d))
    return tc_decode(d, w, q_c, q_r, &packed, count, B, kmax, base + L.off_dec, o, st);
  return simt_decode(d, w, q_c, q_r, &packed, count, B, kmax, base + L.off_dec, o, st);
}

mla_status_t mla_debug_arm_wait_timeout(int64_t limit_ns) {
  if (limit_ns <= 0 || limit_ns > 2000000000ll) return MLA_ERR_INVALID_ARG;
  arm_decode_wait_timeout(limit_ns);
  return MLA_OK;
}

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MLA_ERR_CAPACITY: return "cache row outside [0, capacity)";
    case MLA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "bounded device wait gave up";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_LENGTH: return "sequence length above max_len";
  }
  return "unknown status";
}

}  // extern "C"
