// Portable SIMT kernels of libmla: every step of MLA for any widths, fp32 or bf16 storage,
// fp32 arithmetic. They serve the fp32 workloads and shapes the tensor-core kernels do not
// cover. Formulas: "MLA前向计算流程" §三分支计算 ①–④; absorbed decode: "从LLaMA到DeepSeek[01]
// - MLA（上）" §六.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace mla {

__device__ unsigned int g_status = 0;

// ==================================================================================
// Tiled linear map Y[n, o] = sum_k X[n, k] * W[o, k] (W stored [out, in]) with a fused
// epilogue. W rows [0, O0) come from W0 and rows [O0, O) from W1 (so [W^DKV; W^KR] or
// [W^UQ; W^QR] act as one matrix). X rows may be gathered through xrow[n].
// Each thread produces output pairs (o, o+1) so that RoPE can rotate inside the epilogue.
// ==================================================================================
constexpr int LBM = 64, LBN = 64, LBK = 32;

template <typename TX, typename TW, typename Ep>
__global__ void __launch_bounds__(256) linear_kernel(const TX* __restrict__ X, int64_t ldx,
                                                     const int64_t* __restrict__ xrow, int N,
                                                     const TW* __restrict__ W0, int O0,
                                                     const TW* __restrict__ W1, int O, int K,
                                                     Ep ep) {
  __shared__ float Xs[LBK][LBM + 1];
  __shared__ float Ws[LBK][LBN + 1];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;  // tx: 4 outputs, ty: 4 tokens
  const int n0 = blockIdx.y * LBM, o0 = blockIdx.x * LBN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += LBK) {
    for (int e = tid; e < LBM * LBK; e += 256) {
      const int r = e / LBK, kk = e % LBK;
      const int n = n0 + r, k = k0 + kk;
      float v = 0.f;
      if (n < N && k < K) {
        const int64_t row = xrow ? xrow[n] : (int64_t)n;
        v = to_f(X[row * ldx + k]);
      }
      Xs[kk][r] = v;
    }
    for (int e = tid; e < LBN * LBK; e += 256) {
      const int r = e / LBK, kk = e % LBK;
      const int o = o0 + r, k = k0 + kk;
      float v = 0.f;
      if (o < O && k < K) v = to_f(o < O0 ? W0[(int64_t)o * K + k] : W1[(int64_t)(o - O0) * K + k]);
      Ws[kk][r] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < LBK; ++kk) {
      float xv[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = Xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + ty * 4 + i;
    if (n >= N) continue;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const int o = o0 + tx * 4 + j;
      if (o < O) ep(n, o, acc[i][j], o + 1 < O ? acc[i][j + 1] : 0.f);
    }
  }
}

// Epilogue of the append: [c^KV ; k^R] -> cache row, RoPE on the k^R pairs.
template <typename T>
struct AppendEp {
  T* rows;
  int64_t pitch, capacity;
  const int64_t* seq_base;
  const int32_t* seq_idx;  // null: token n belongs to tok_seq[n]
  const int32_t* pos;
  int d_c;
  RopeFreqs rf;
  __device__ void operator()(int n, int o, float a0, float a1) const {
    const int p = pos[n];
    const int64_t row = seq_base[seq_idx[n]] + p;
    if (row < 0 || row >= capacity) {
      flag_status(MLA_ERR_CAPACITY);
      return;
    }
    if (o >= d_c) {  // k^R pair (2k, 2k+1) of the decoupled RoPE key
      float c, s;
      rope_cs(p, (o - d_c) >> 1, rf, &c, &s);
      const float r0 = a0 * c - a1 * s, r1 = a0 * s + a1 * c;
      a0 = r0;
      a1 = r1;
    }
    T* dst = rows + row * pitch + o;
    dst[0] = from_f<T>(a0);
    dst[1] = from_f<T>(a1);
  }
};

// Epilogue that stores a plain fp32 matrix [N, ldy].
struct StoreF32Ep {
  float* Y;
  int64_t ldy;
  __device__ void operator()(int n, int o, float a0, float a1) const {
    Y[(int64_t)n * ldy + o] = a0;
    Y[(int64_t)n * ldy + o + 1] = a1;
  }
};

// Epilogue of the query up-projection: outputs [0, n_h*d_hc) are q^C, the rest q^R
// (RoPE per head at the token's position). Writes either separate q_c / q_r tensors
// (qc_ld = d_hc, qr_ld = d_hr) or one interleaved [n, n_h, d_hc + d_hr] tensor.
template <typename T>
struct QueryEp {
  T* q_c;
  T* q_r;
  int64_t qc_tok, qc_head, qr_tok, qr_head;  // strides (elements)
  const int32_t* pos;
  int n_h, d_hc, d_hr;
  RopeFreqs rf;
  __device__ void operator()(int n, int o, float a0, float a1) const {
    const int nc = n_h * d_hc;
    if (o < nc) {
      const int i = o / d_hc, e = o % d_hc;
      T* dst = q_c + n * qc_tok + i * qc_head + e;
      dst[0] = from_f<T>(a0);
      dst[1] = from_f<T>(a1);
    } else {
      const int r = o - nc, i = r / d_hr, e = r % d_hr;
      float c, s;
      rope_cs(pos[n], e >> 1, rf, &c, &s);
      T* dst = q_r + n * qr_tok + i * qr_head + e;
      dst[0] = from_f<T>(a0 * c - a1 * s);
      dst[1] = from_f<T>(a0 * s + a1 * c);
    }
  }
};

template <typename TX, typename TW, typename Ep>
static void launch_linear(int kid, const TX* X, int64_t ldx, const int64_t* xrow, int N,
                          const TW* W0, int O0, const TW* W1, int O, int K, Ep ep,
                          cudaStream_t st) {
  if (N <= 0 || O <= 0) return;
  dim3 grid(ceil_div(O, LBN), ceil_div(N, LBM));
  TraceScope ts(kid, st);
  linear_kernel<TX, TW, Ep><<<grid, 256, 0, st>>>(X, ldx, xrow, N, W0, O0, W1, O, K, ep);
}

// ==================================================================================
// Append (§三分支计算 ② Key / ③ Value: the cached [c^KV ; k^R])
// ==================================================================================
template <typename T>
static mla_status_t append_t(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                             const int32_t* seq_idx, const int32_t* pos, int n,
                             mla_cache_t* cache, cudaStream_t st) {
  AppendEp<T> ep{(T*)cache->rows, (int64_t)(d->d_c + d->d_hr), cache->capacity, cache->seq_base,
                 seq_idx, pos, d->d_c, rope_freqs(d)};
  launch_linear<T, T>(K_APPEND, (const T*)h, d->d, nullptr, n, (const T*)w->W_DKV, d->d_c,
                      (const T*)w->W_KR, d->d_c + d->d_hr, d->d, ep, st);
  return launch_status();
}

mla_status_t simt_append(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                         const int32_t* seq_idx, const int32_t* pos, int n, mla_cache_t* cache,
                         cudaStream_t st) {
  if (d->dtype == MLA_BF16)
    return append_t<__nv_bfloat16>(d, w, h, seq_idx, pos, n, cache, st);
  return append_t<float>(d, w, h, seq_idx, pos, n, cache, st);
}

// ==================================================================================
// Query projection (§三分支计算 ① Query); c^Q kept in fp32 in the workspace.
// ==================================================================================
size_t simt_project_q_ws(const mla_dims_t* d, int n) {
  return align_up((size_t)n * d->d_cq * sizeof(float), 256);
}

template <typename T>
static mla_status_t project_q_t(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                                const int32_t* pos, int n, void* ws, void* q_c, void* q_r,
                                cudaStream_t st) {
  float* cq = (float*)ws;
  launch_linear<T, T>(K_Q_DOWN, (const T*)h, d->d, nullptr, n, (const T*)w->W_DQ, d->d_cq,
                      (const T*)w->W_DQ, d->d_cq, d->d, StoreF32Ep{cq, d->d_cq}, st);
  QueryEp<T> ep{(T*)q_c, (T*)q_r, (int64_t)d->n_h * d->d_hc, d->d_hc,
                (int64_t)d->n_h * d->d_hr, d->d_hr, pos, d->n_h, d->d_hc, d->d_hr,
                rope_freqs(d)};
  const int nc = d->n_h * d->d_hc, nr = d->n_h * d->d_hr;
  launch_linear<float, T>(K_Q_UP, cq, d->d_cq, nullptr, n, (const T*)w->W_UQ, nc,
                          (const T*)w->W_QR, nc + nr, d->d_cq, ep, st);
  return launch_status();
}

mla_status_t simt_project_q(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                            const int32_t* pos, int n, void* ws, void* q_c, void* q_r,
                            cudaStream_t st) {
  if (d->dtype == MLA_BF16)
    return project_q_t<__nv_bfloat16>(d, w, h, pos, n, ws, q_c, q_r, st);
  return project_q_t<float>(d, w, h, pos, n, ws, q_c, q_r, st);
}

// ==================================================================================
// Absorbed decode ("从LLaMA到DeepSeek" §六)
//   1. absorb:  q~[b,i,:] = W^UK_i^T q^C[b,i,:]
//   2. split-KV latent attention: per (b, split, head group) online softmax over the
//      split's rows, emitting unnormalised o~, running max m and sum l
//   3. combine: log-sum-exp merge of the splits, then o = W^UV_i o~
// ==================================================================================
template <typename T>
__global__ void __launch_bounds__(256) absorb_kernel(const T* __restrict__ q_c,
                                                     const T* __restrict__ W_UK, int B,
                                                     int n_h, int d_hc, int d_c,
                                                     float* __restrict__ qt) {
  // grid: (ceil(d_c/256), n_h, ceil(B/8)); each thread owns one latent column c for 8 b.
  extern __shared__ float qs[];  // [8][d_hc]
  const int i = blockIdx.y, b0 = blockIdx.z * 8;
  const int c = blockIdx.x * 256 + threadIdx.x;
  const int nb = min(8, B - b0);
  for (int e = threadIdx.x; e < nb * d_hc; e += 256) {
    const int bb = e / d_hc, dd = e % d_hc;
    qs[bb * d_hc + dd] = to_f(q_c[((int64_t)(b0 + bb) * n_h + i) * d_hc + dd]);
  }
  __syncthreads();
  if (c >= d_c) return;
  float acc[8];
#pragma unroll
  for (int bb = 0; bb < 8; ++bb) acc[bb] = 0.f;
  const T* Wi = W_UK + (int64_t)i * d_hc * d_c + c;
  for (int dd = 0; dd < d_hc; ++dd) {
    const float wv = to_f(Wi[(int64_t)dd * d_c]);
#pragma unroll
    for (int bb = 0; bb < 8; ++bb) acc[bb] = fmaf(qs[bb * d_hc + dd], wv, acc[bb]);
  }
  for (int bb = 0; bb < nb; ++bb) qt[((int64_t)(b0 + bb) * n_h + i) * d_c + c] = acc[bb];
}

constexpr int DHG = 8;   // heads per CTA (one warp per head in the softmax step)
constexpr int DTT = 32;  // cache rows per tile

template <typename T>
__global__ void __launch_bounds__(256) decode_attn_kernel(
    const float* __restrict__ qt, const T* __restrict__ q_r, const T* __restrict__ rows,
    const int64_t* __restrict__ seq_base, int64_t capacity, const int32_t* __restrict__ seq_len,
    int max_len, int S, int split_len, int n_h, int d_c, int d_hr, float scale,
    float* __restrict__ part_o, float* __restrict__ part_ml) {
  extern __shared__ float sm[];
  const int R = d_c + d_hr;
  float* qs = sm;                      // [DHG][R]
  float* ts = qs + DHG * R;            // [DTT][R]
  float* ps = ts + DTT * R;            // [DHG][DTT]
  float* os = ps + DHG * DTT;          // [DHG][d_c]
  float* al = os + DHG * d_c;          // [DHG] rescale factors
  const int s_id = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h0 = hg * DHG;
  int L = seq_len[b];
  if (L > max_len || L < 0) {
    if (tid == 0 && s_id == 0) flag_status(MLA_ERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  const int64_t base_row = seq_base[b];
  if (L > 0 && (base_row < 0 || base_row + L > capacity)) {
    if (tid == 0 && s_id == 0) flag_status(MLA_ERR_CAPACITY);
    L = 0;
  }
  const int j_begin = s_id * split_len, j_end = min(L, j_begin + split_len);
  for (int e = tid; e < DHG * R; e += 256) {
    const int hh = e / R, k = e % R;
    const int i = h0 + hh;
    float v = 0.f;
    if (i < n_h)
      v = k < d_c ? qt[((int64_t)b * n_h + i) * d_c + k]
                  : to_f(q_r[((int64_t)b * n_h + i) * d_hr + (k - d_c)]);
    qs[e] = v;
  }
  for (int e = tid; e < DHG * d_c; e += 256) os[e] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // per warp == per head (lane-uniform)
  __syncthreads();
  for (int j0 = j_begin; j0 < j_end; j0 += DTT) {
    const int nt = min(DTT, j_end - j0);
    for (int e = tid; e < DTT * R; e += 256) {
      const int jj = e / R, k = e % R;
      ts[e] = jj < nt ? to_f(rows[(base_row + j0 + jj) * R + k]) : 0.f;
    }
    __syncthreads();
    {  // one score per thread: head tid / DTT, row tid % DTT
      const int hh = tid / DTT, jj = tid % DTT;
      float s = -INFINITY;
      if (jj < nt && h0 + hh < n_h) {
        const float* q = qs + hh * R;
        const float* r = ts + jj * R;
        float acc = 0.f;
        for (int k = 0; k < R; ++k) acc = fmaf(q[k], r[k], acc);
        s = acc * scale;
      }
      ps[hh * DTT + jj] = s;
    }
    __syncthreads();
    {  // warp `warp` updates head `warp`'s running max / sum and turns scores into weights
      const float s = ps[warp * DTT + lane];
      float mx = s;
      for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : __expf(m_run - m_new);
      const float p = (s == -INFINITY) ? 0.f : __expf(s - m_new);
      float sum = p;
      for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run = l_run * alpha + sum;
      m_run = m_new;
      ps[warp * DTT + lane] = p;
      if (lane == 0) al[warp] = alpha;
    }
    __syncthreads();
    for (int e = tid; e < DHG * d_c; e += 256) {
      const int hh = e / d_c, c = e % d_c;
      float acc = os[e] * al[hh];
      const float* p = ps + hh * DTT;
      for (int jj = 0; jj < nt; ++jj) acc = fmaf(p[jj], ts[jj * R + c], acc);
      os[e] = acc;
    }
    __syncthreads();
  }
  const int64_t pbase = ((int64_t)b * S + s_id) * n_h;
  for (int e = tid; e < DHG * d_c; e += 256) {
    const int hh = e / d_c, c = e % d_c;
    if (h0 + hh < n_h) part_o[(pbase + h0 + hh) * d_c + c] = os[e];
  }
  if (lane == 0 && h0 + warp < n_h) {
    part_ml[(pbase + h0 + warp) * 2 + 0] = m_run;
    part_ml[(pbase + h0 + warp) * 2 + 1] = l_run;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) decode_combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_ml, int S, int n_h, int d_c,
    int d_hc, const T* __restrict__ W_UV, float* __restrict__ o) {
  // grid: (n_h, B). Merge the S splits of (b, i) by log-sum-exp, then apply W^UV_i.
  extern __shared__ float ol[];  // [d_c]
  __shared__ float wts[64];
  __shared__ float inv_l;
  const int i = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int64_t pbase = (int64_t)b * S * n_h;
  if (tid == 0) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, part_ml[((pbase + (int64_t)s * n_h) + i) * 2]);
    float Lsum = 0.f;
    for (int s = 0; s < S; ++s) {
      const float m = part_ml[((pbase + (int64_t)s * n_h) + i) * 2];
      const float l = part_ml[((pbase + (int64_t)s * n_h) + i) * 2 + 1];
      const float wgt = (m == -INFINITY) ? 0.f : __expf(m - M);
      if (s < 64) wts[s] = wgt;
      Lsum += wgt * l;
    }
    inv_l = Lsum > 0.f ? 1.f / Lsum : 0.f;
  }
  __syncthreads();
  for (int c = tid; c < d_c; c += 256) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float wgt = wts[s];
      if (wgt != 0.f) acc = fmaf(wgt, part_o[((pbase + (int64_t)s * n_h) + i) * d_c + c], acc);
    }
    ol[c] = acc * inv_l;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int dd = warp; dd < d_hc; dd += 8) {
    const T* wr = W_UV + ((int64_t)i * d_hc + dd) * d_c;
    float acc = 0.f;
    for (int c = lane; c < d_c; c += 32) acc = fmaf(to_f(wr[c]), ol[c], acc);
    for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) o[((int64_t)b * n_h + i) * d_hc + dd] = acc;
  }
}

struct DecodePlan {
  int S, split_len;
  size_t off_qt, off_po, off_pml, total;
};

static DecodePlan decode_plan(const mla_dims_t* d, int B, int max_len) {
  DecodePlan p;
  const int groups = ceil_div(d->n_h, DHG);
  const int base_ctas = max(1, B * groups);
  int S = ceil_div(4 * 148, base_ctas);
  S = max(1, min(S, ceil_div(max(max_len, 1), DTT)));
  S = min(S, 64);
  int split_len = ceil_div(max(max_len, 1), S);
  split_len = ceil_div(split_len, DTT) * DTT;
  S = ceil_div(max(max_len, 1), split_len);
  p.S = S;
  p.split_len = split_len;
  p.off_qt = 0;
  p.off_po = align_up(p.off_qt + (size_t)B * d->n_h * d->d_c * sizeof(float), 256);
  p.off_pml = align_up(p.off_po + (size_t)B * S * d->n_h * d->d_c * sizeof(float), 256);
  p.total = align_up(p.off_pml + (size_t)B * S * d->n_h * 2 * sizeof(float), 256);
  return p;
}

size_t simt_decode_ws(const mla_dims_t* d, int B, int max_len) {
  return decode_plan(d, B, max_len).total;
}

size_t simt_decode_smem(const mla_dims_t* d) {
  const int R = d->d_c + d->d_hr;
  return sizeof(float) * ((size_t)DHG * R + (size_t)DTT * R + DHG * DTT + (size_t)DHG * d->d_c + DHG);
}

template <typename T>
static mla_status_t decode_t(const mla_dims_t* d, const mla_weights_t* w, const void* q_c,
                             const void* q_r, const mla_cache_t* cache, const int32_t* seq_len,
                             int B, int max_len, void* ws, float* o, cudaStream_t st) {
  const DecodePlan p = decode_plan(d, B, max_len);
  char* wsb = (char*)ws;
  float* qt = (float*)(wsb + p.off_qt);
  float* po = (float*)(wsb + p.off_po);
  float* pml = (float*)(wsb + p.off_pml);
  {
    dim3 grid(ceil_div(d->d_c, 256), d->n_h, ceil_div(B, 8));
    TraceScope ts(K_ABSORB, st);
    absorb_kernel<T><<<grid, 256, 8 * d->d_hc * sizeof(float), st>>>(
        (const T*)q_c, (const T*)w->W_UK, B, d->n_h, d->d_hc, d->d_c, qt);
  }
  {
    const size_t smem = simt_decode_smem(d);
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(decode_attn_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
    dim3 grid(p.S, ceil_div(d->n_h, DHG), B);
    TraceScope ts(K_DECODE_ATTN, st);
    decode_attn_kernel<T><<<grid, 256, smem, st>>>(
        qt, (const T*)q_r, (const T*)cache->rows, cache->seq_base, cache->capacity, seq_len,
        max_len, p.S, p.split_len, d->n_h, d->d_c, d->d_hr, softmax_scale(d), po, pml);
  }
  {
    dim3 grid(d->n_h, B);
    TraceScope ts(K_DECODE_COMBINE, st);
    decode_combine_kernel<T><<<grid, 256, d->d_c * sizeof(float), st>>>(
        po, pml, p.S, d->n_h, d->d_c, d->d_hc, (const T*)w->W_UV, o);
  }
  return launch_status();
}

mla_status_t simt_decode(const mla_dims_t* d, const mla_weights_t* w, const void* q_c,
                         const void* q_r, const mla_cache_t* cache, const int32_t* seq_len,
                         int B, int max_len, void* ws, float* o, cudaStream_t st) {
  if (d->dtype == MLA_BF16)
    return decode_t<__nv_bfloat16>(d, w, q_c, q_r, cache, seq_len, B, max_len, ws, o, st);
  return decode_t<float>(d, w, q_c, q_r, cache, seq_len, B, max_len, ws, o, st);
}

// ==================================================================================
// Prefill (non-absorbed, MHA-style expansion; V3.1 Hybrid remark of "MLA前向计算流程")
// ==================================================================================
__global__ void token_map_kernel(const int32_t* __restrict__ cu, int B, int n_tok,
                                 const int64_t* __restrict__ seq_base, int64_t capacity,
                                 int max_T,
                                 int32_t* __restrict__ tok_seq, int32_t* __restrict__ tok_pos,
                                 int64_t* __restrict__ tok_row) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= n_tok) return;
  int lo = 0, hi = B;  // find b with cu[b] <= n < cu[b+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= n) lo = mid; else hi = mid;
  }
  const int p = n - cu[lo];
  if (p >= max_T) flag_status(MLA_ERR_LENGTH);
  int64_t row = seq_base[lo] + p;
  if (row < 0 || row >= capacity) {  // the append flags it; reads fall back to row 0
    flag_status(MLA_ERR_CAPACITY);
    row = 0;
  }
  tok_seq[n] = lo;
  tok_pos[n] = p;
  tok_row[n] = row;
}

constexpr int PBQ = 32, PBK = 32;

template <typename T>
__global__ void __launch_bounds__(256) prefill_attn_kernel(
    const float* __restrict__ Q, const float* __restrict__ KC, const float* __restrict__ V,
    const T* __restrict__ rows, const int64_t* __restrict__ tok_row,
    const int32_t* __restrict__ cu, int n_h, int d_hc, int d_hr, int d_c, float scale,
    float* __restrict__ o) {
  // grid: (q blocks of the longest sequence, n_h, B). Q rows [n, n_h, d_hc + d_hr].
  extern __shared__ float sm[];
  const int dh = d_hc + d_hr;
  float* qs = sm;                  // [PBQ][dh]
  float* ks = qs + PBQ * dh;       // [PBK][dh]
  float* vs = ks + PBK * dh;       // [PBK][d_hc]
  float* ss = vs + PBK * d_hc;     // [PBQ][PBK]
  float* os = ss + PBQ * PBK;      // [PBQ][d_hc]
  float* al = os + PBQ * d_hc;     // [PBQ]
  const int i = blockIdx.y, b = blockIdx.z;
  const int t0 = cu[b], Tq = cu[b + 1] - cu[b];
  const int q0 = blockIdx.x * PBQ;
  if (q0 >= Tq) return;
  const int nq = min(PBQ, Tq - q0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = d_c + d_hr;
  for (int e = tid; e < PBQ * dh; e += 256) {
    const int r = e / dh, k = e % dh;
    qs[e] = r < nq ? Q[((int64_t)(t0 + q0 + r) * n_h + i) * dh + k] : 0.f;
  }
  for (int e = tid; e < PBQ * d_hc; e += 256) os[e] = 0.f;
  // each warp owns 4 query rows: running max / sum for rows warp*4 .. warp*4+3
  float m_run[4], l_run[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) { m_run[r] = -INFINITY; l_run[r] = 0.f; }
  const int k_end = q0 + nq;  // keys 0 .. k_end-1 (causal)
  for (int k0 = 0; k0 < k_end; k0 += PBK) {
    const int nk = min(PBK, k_end - k0);
    __syncthreads();
    for (int e = tid; e < PBK * dh; e += 256) {
      const int r = e / dh, k = e % dh;
      float v = 0.f;
      if (r < nk) {
        const int t = t0 + k0 + r;
        v = k < d_hc ? KC[((int64_t)t * n_h + i) * d_hc + k]
                     : to_f(rows[tok_row[t] * R + d_c + (k - d_hc)]);
      }
      ks[e] = v;
    }
    for (int e = tid; e < PBK * d_hc; e += 256) {
      const int r = e / d_hc, k = e % d_hc;
      vs[e] = r < nk ? V[((int64_t)(t0 + k0 + r) * n_h + i) * d_hc + k] : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < PBQ * PBK; e += 256) {
      const int r = e / PBK, c = e % PBK;
      float s = -INFINITY;
      if (r < nq && c < nk && k0 + c <= q0 + r) {
        float acc = 0.f;
        const float* qq = qs + r * dh;
        const float* kk = ks + c * dh;
        for (int k = 0; k < dh; ++k) acc = fmaf(qq[k], kk[k], acc);
        s = acc * scale;
      }
      ss[e] = s;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      const float s = ss[r * PBK + lane];
      float mx = s;
      for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_run[rr], mx);
      const float alpha = (m_new == -INFINITY) ? 1.f : __expf(m_run[rr] - m_new);
      const float p = (s == -INFINITY) ? 0.f : __expf(s - m_new);
      float sum = p;
      for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l_run[rr] = l_run[rr] * alpha + sum;
      m_run[rr] = m_new;
      ss[r * PBK + lane] = p;
      if (lane == 0) al[r] = alpha;
    }
    __syncthreads();
    for (int e = tid; e < PBQ * d_hc; e += 256) {
      const int r = e / d_hc, c = e % d_hc;
      float acc = os[e] * al[r];
      const float* p = ss + r * PBK;
      for (int kk = 0; kk < nk; ++kk) acc = fmaf(p[kk], vs[kk * d_hc + c], acc);
      os[e] = acc;
    }
  }
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) al[warp * 4 + rr] = l_run[rr] > 0.f ? 1.f / l_run[rr] : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < nq * d_hc; e += 256) {
    const int r = e / d_hc, c = e % d_hc;
    o[((int64_t)(t0 + q0 + r) * n_h + i) * d_hc + c] = os[e] * al[r];
  }
}

struct PrefillPlan {
  size_t off_cq, off_q, off_kc, off_v, off_seq, off_pos, off_row, total;
};

static PrefillPlan prefill_plan(const mla_dims_t* d, int n) {
  PrefillPlan p;
  const size_t dh = d->d_hc + d->d_hr;
  p.off_cq = 0;
  p.off_q = align_up(p.off_cq + (size_t)n * d->d_cq * 4, 256);
  p.off_kc = align_up(p.off_q + (size_t)n * d->n_h * dh * 4, 256);
  p.off_v = align_up(p.off_kc + (size_t)n * d->n_h * d->d_hc * 4, 256);
  p.off_seq = align_up(p.off_v + (size_t)n * d->n_h * d->d_hc * 4, 256);
  p.off_pos = align_up(p.off_seq + (size_t)n * 4, 256);
  p.off_row = align_up(p.off_pos + (size_t)n * 4, 256);
  p.total = align_up(p.off_row + (size_t)n * 8, 256);
  return p;
}

size_t simt_prefill_ws(const mla_dims_t* d, int n_tok) { return prefill_plan(d, n_tok).total; }

size_t simt_prefill_smem(const mla_dims_t* d) {
  const int dh = d->d_hc + d->d_hr;
  return sizeof(float) * ((size_t)PBQ * dh + (size_t)PBK * dh + (size_t)PBK * d->d_hc +
                          PBQ * PBK + (size_t)PBQ * d->d_hc + PBQ);
}

template <typename T>
static mla_status_t prefill_t(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                              const int32_t* cu, int B, int n, int max_T, mla_cache_t* cache,
                              void* ws, float* o, cudaStream_t st) {
  const PrefillPlan p = prefill_plan(d, n);
  char* wsb = (char*)ws;
  float* cq = (float*)(wsb + p.off_cq);
  float* Q = (float*)(wsb + p.off_q);
  float* KC = (float*)(wsb + p.off_kc);
  float* V = (float*)(wsb + p.off_v);
  int32_t* tseq = (int32_t*)(wsb + p.off_seq);
  int32_t* tpos = (int32_t*)(wsb + p.off_pos);
  int64_t* trow = (int64_t*)(wsb + p.off_row);
  const int dh = d->d_hc + d->d_hr;
  {
    TraceScope ts(K_TOKEN_MAP, st);
    token_map_kernel<<<ceil_div(n, 256), 256, 0, st>>>(cu, B, n, cache->seq_base,
                                                        cache->capacity, max_T, tseq,
                                                        tpos, trow);
  }
  // cache rows for every prompt token
  {
    AppendEp<T> ep{(T*)cache->rows, (int64_t)(d->d_c + d->d_hr), cache->capacity,
                   cache->seq_base, tseq, tpos, d->d_c, rope_freqs(d)};
    launch_linear<T, T>(K_PREFILL_APPEND, (const T*)h, d->d, nullptr, n, (const T*)w->W_DKV,
                        d->d_c, (const T*)w->W_KR, d->d_c + d->d_hr, d->d, ep, st);
  }
  // queries: c^Q, then [q^C ; q^R] per head, interleaved [n, n_h, d_hc + d_hr]
  launch_linear<T, T>(K_PREFILL_Q_DOWN, (const T*)h, d->d, nullptr, n, (const T*)w->W_DQ,
                      d->d_cq, (const T*)w->W_DQ, d->d_cq, d->d, StoreF32Ep{cq, d->d_cq}, st);
  {
    QueryEp<float> ep{Q, Q + d->d_hc, (int64_t)d->n_h * dh, dh, (int64_t)d->n_h * dh, dh,
                      tpos, d->n_h, d->d_hc, d->d_hr, rope_freqs(d)};
    const int nc = d->n_h * d->d_hc, nr = d->n_h * d->d_hr;
    launch_linear<float, T>(K_PREFILL_Q_UP, cq, d->d_cq, nullptr, n, (const T*)w->W_UQ, nc,
                            (const T*)w->W_QR, nc + nr, d->d_cq, ep, st);
  }
  // K^C and V expanded per head from the stored latent rows
  {
    const int nc = d->n_h * d->d_hc;
    launch_linear<T, T>(K_EXPAND_K, (const T*)cache->rows, d->d_c + d->d_hr, trow, n,
                        (const T*)w->W_UK, nc, (const T*)w->W_UK, nc, d->d_c,
                        StoreF32Ep{KC, nc}, st);
    launch_linear<T, T>(K_EXPAND_V, (const T*)cache->rows, d->d_c + d->d_hr, trow, n,
                        (const T*)w->W_UV, nc, (const T*)w->W_UV, nc, d->d_c,
                        StoreF32Ep{V, nc}, st);
  }
  {
    const size_t smem = simt_prefill_smem(d);
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(prefill_attn_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
    dim3 grid(ceil_div(max_T, PBQ), d->n_h, B);
    TraceScope ts(K_PREFILL_ATTN, st);
    prefill_attn_kernel<T><<<grid, 256, smem, st>>>(Q, KC, V, (const T*)cache->rows, trow, cu,
                                                     d->n_h, d->d_hc, d->d_hr, d->d_c,
                                                     softmax_scale(d), o);
  }
  return launch_status();
}

mla_status_t simt_prefill(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                          const int32_t* cu, int B, int n, int max_T, mla_cache_t* cache,
                          void* ws, float* o, cudaStream_t st) {
  if (d->dtype == MLA_BF16)
    return prefill_t<__nv_bfloat16>(d, w, h, cu, B, n, max_T, cache, ws, o, st);
  return prefill_t<float>(d, w, h, cu, B, n, max_T, cache, ws, o, st);
}

// ==================================================================================
// Output projection (§三分支计算 ④): u[n, :] = W^O [o_{n,1}; ...; o_{n,n_h}], with o given as
// [n, n_h * d_hc] float32 (the head-major concatenation is the row layout of o).
// ==================================================================================
mla_status_t simt_output_projection(const mla_dims_t* d, const void* W_O, const float* o, int n,
                                    float* u, cudaStream_t st) {
  const int K = d->n_h * d->d_hc;
  if (d->dtype == MLA_BF16)
    launch_linear<float, __nv_bfloat16>(K_OUT_PROJ, o, K, nullptr, n,
                                        (const __nv_bfloat16*)W_O, d->d,
                                        (const __nv_bfloat16*)W_O, d->d, K,
                                        StoreF32Ep{u, d->d}, st);
  else
    launch_linear<float, float>(K_OUT_PROJ, o, K, nullptr, n, (const float*)W_O, d->d,
                                (const float*)W_O, d->d, K, StoreF32Ep{u, d->d}, st);
  return launch_status();
}

// ==================================================================================
// Pre-merged absorbed query weights ("从LLaMA到DeepSeek[01] - MLA（上）" §六: W^UQ and W^UK are
// both fixed, so their product can be formed once): for every head i,
//   W^UQK_i [d_c x d_c'] = (W^UK_i)^T W^UQ_i,
//   out[(i d_c + l) d_c' + c] = sum_d W^UK[i d_hc + d][l] W^UQ[i d_hc + d][c],
// fp32 accumulation, stored in the weights' dtype. A one-off, so a plain tiled kernel: a
// 64 x 64 output tile per block, the shared K dimension d (d_hc) in chunks of 32.
// ==================================================================================
template <typename T>
__global__ void __launch_bounds__(256) merge_absorption_kernel(const T* __restrict__ W_UQ,
                                                               const T* __restrict__ W_UK,
                                                               int d_hc, int d_c, int d_cq,
                                                               T* __restrict__ out) {
  __shared__ float As[32][64 + 1];  // [d][l]
  __shared__ float Bs[32][64 + 1];  // [d][c]
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;  // 4 c-columns x 4 l-rows each
  const int c0 = blockIdx.x * 64, l0 = blockIdx.y * 64, i = blockIdx.z;
  float acc[4][4] = {};
  for (int d0 = 0; d0 < d_hc; d0 += 32) {
    for (int e = tid; e < 32 * 64; e += 256) {
      const int dd = e >> 6, x = e & 63, dr = d0 + dd;
      const int64_t row = (int64_t)i * d_hc + dr;
      As[dd][x] = (dr < d_hc && l0 + x < d_c) ? to_f(W_UK[row * d_c + l0 + x]) : 0.f;
      Bs[dd][x] = (dr < d_hc && c0 + x < d_cq) ? to_f(W_UQ[row * d_cq + c0 + x]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int dd = 0; dd < 32; ++dd) {
      float a[4], b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a[k] = As[dd][ty * 4 + k];
        b[k] = Bs[dd][tx * 4 + k];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int l = l0 + ty * 4 + r;
    if (l >= d_c) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = c0 + tx * 4 + c;
      if (cc < d_cq) out[((int64_t)i * d_c + l) * d_cq + cc] = from_f<T>(acc[r][c]);
    }
  }
}

mla_status_t simt_merge_absorption(const mla_dims_t* d, const void* W_UQ, const void* W_UK,
                                   void* W_UQK, cudaStream_t st) {
  const dim3 grid(ceil_div(d->d_cq, 64), ceil_div(d->d_c, 64), d->n_h);
  TraceScope ts(K_MERGE_W, st);
  if (d->dtype == MLA_BF16)
    merge_absorption_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        (const __nv_bfloat16*)W_UQ, (const __nv_bfloat16*)W_UK, d->d_hc, d->d_c, d->d_cq,
        (__nv_bfloat16*)W_UQK);
  else
    merge_absorption_kernel<float><<<grid, 256, 0, st>>>((const float*)W_UQ, (const float*)W_UK,
                                                         d->d_hc, d->d_c, d->d_cq,
                                                         (float*)W_UQK);
  return launch_status();
}

}  // namespace mla
