// Causal prefill on the tensor cores for the DeepSeek-V2 widths (bf16): the non-absorbed,
// MHA-style expansion that "MLA前向计算流程" prescribes for prefill (V3.1 Hybrid remark) and
// "从LLaMA到DeepSeek[01] - MLA（上）" §七 motivates (many tokens in flight: expand K/V per head
// instead of absorbing):
//   k_{j,i} = [W^UK_i c_j ; k^R_j],  v_{j,i} = W^UV_i c_j,  q_{t,i} = [q^C_{t,i} ; q^R_{t,i}],
//   o_{t,i} = sum_{j <= t} softmax_j(q_{t,i} . k_{j,i} * scale) v_{j,i}   (§三分支计算 ④).
//
// Launch sequence (all tcgen05 kernels except the token map):
//   token map  -> append (cache rows + a packed copy of the latent rows)
//   -> c^Q (bf16) -> [q^C ; q^R] per head (bf16, RoPE in the epilogue)
//   -> K^C = W^UK c (bf16) and V = W^UV c (fp16) per head -> causal attention (this file).
// P and V meet in fp16 (P in [0, 2^8] under the lazy rescale): the rounding of P and V sets this
// path's error, and fp16 keeps three more bits than bf16 at the same MMA rate.
//
// Attention kernel: one CTA per (128-query tile, head, sequence). Blocks are dispatched with all
// query tiles of a head together (heaviest first), so the K/V tiles they share stay in L2.
// Warp 0 streams the query tile once and then, per 128-key tile, K = [K^C | k^R] (3 boxes) and
// V (2 boxes) into two 2-deep rings; warp 1 issues S = Q K^T (K = 192) into one of two TMEM
// score buffers and O += P V with P read from TMEM (the softmax writes P in bf16 over the first
// 64 columns of the score buffer it came from); warps 2..5 run the online softmax, one thread
// query row and column half (two warps per TMEM lane quarter, 64 key columns each), in log2
// units with lazy rescaling of O.
#include <mutex>

#include "internal.h"
#include "tc.cuh"

namespace mla {

using namespace tc;

namespace {

constexpr int kH = 128;       // heads
constexpr int kDC = 512;      // d_c
constexpr int kDQK = 192;     // d_h^C + d_h^R
constexpr int kDV = 128;      // d_h^C
constexpr int kRow = 576;     // latent cache row
constexpr int kBQ = 128;      // queries per tile
constexpr int kBK = 128;      // keys per tile
constexpr int kBox = 128 * 128;  // 128 rows x 64 bf16 (16 KB)
constexpr int kOffQ = 0;                     // 3 boxes
constexpr int kOffK = 3 * kBox;              // 2 stages x 3 boxes
constexpr int kOffV = kOffK + 6 * kBox;      // 2 stages x 2 boxes
constexpr int kOffBar = kOffV + 4 * kBox;    // 13 boxes = 208 KB
constexpr int kThreads = 320;  // 10 warps: 0 TMA, 1 MMA, 2..9 softmax (two per TMEM lane quarter)
constexpr int kSmemBytes = kOffBar + 4096 + 1024;
constexpr uint32_t kColO = 256;  // O: 128 fp32 columns; score buffers at 0 and 128
constexpr float kTau = 8.f;      // lazy rescale threshold (log2 units)

struct Bars {
  uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done;
  uint64_t mma_done;
  uint32_t tmem_slot;
  int abort;
  float row_max[2][2][kBQ];  // [tile parity][column half][row]: partial maxima of the halves
  float row_sum[2][kBQ];     // [column half][row]: final partial row sums
};
static_assert(sizeof(Bars) <= 4096, "barrier block");

// Two probabilities as an fp16 pair (P in [0, 2^8] with the lazy rescale; fp16 keeps 3 more
// mantissa bits than bf16, and V is stored in fp16 to match).
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q,   // Q  [n, 128, 192]
                           const __grid_constant__ CUtensorMap tm_kc,  // K^C [n, 128, 128]
                           const __grid_constant__ CUtensorMap tm_v,   // V  [n, 128, 128] fp16
                           const __grid_constant__ CUtensorMap tm_kr,  // latent rows [n, 576]
                           const int32_t* __restrict__ cu, float scale_log2,
                           float* __restrict__ o) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars& sh = *reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort = &sh.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int qt = gridDim.x - 1 - blockIdx.x;  // heaviest query tiles of a head go first
  const int t0 = cu[b], T = cu[b + 1] - t0;
  if (qt * kBQ >= T) return;
  const int n_kt = qt + 1;  // key tiles 0 .. qt (causal)

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
      mbar_init(&sh.s_full[s], 1);
      mbar_init(&sh.p_full[s], 8);
    }
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.mma_done, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------- TMA producer
    tma_prefetch(&tm_q);
    tma_prefetch(&tm_kc);
    tma_prefetch(&tm_v);
    tma_prefetch(&tm_kr);
    mbar_arrive_expect_tx(&sh.q_full, 3 * kBox);
    for (int k = 0; k < 3; ++k)
      tma_load_3d(smem + kOffQ + k * kBox, &tm_q, &sh.q_full, k * 64, h, t0 + qt * kBQ);
    int k_issued = 0, v_issued = 0;
    for (int kt = 0; kt < n_kt; ++kt) {
      const int s = kt & 1, r = kt >> 1;
      const int y = t0 + kt * kBK;
      if (r > 0 && !mbar_wait(&sh.k_empty[s], (r - 1) & 1, abort)) break;
      uint8_t* kb = smem + kOffK + s * 3 * kBox;
      mbar_arrive_expect_tx(&sh.k_full[s], 3 * kBox);
      tma_load_3d(kb, &tm_kc, &sh.k_full[s], 0, h, y);
      tma_load_3d(kb + kBox, &tm_kc, &sh.k_full[s], 64, h, y);
      tma_load_2d(kb + 2 * kBox, &tm_kr, &sh.k_full[s], kDC, y);
      ++k_issued;
      if (r > 0 && !mbar_wait(&sh.v_empty[s], (r - 1) & 1, abort)) break;
      uint8_t* vb = smem + kOffV + s * 2 * kBox;
      mbar_arrive_expect_tx(&sh.v_full[s], 2 * kBox);
      tma_load_3d(vb, &tm_v, &sh.v_full[s], 0, h, y);
      tma_load_3d(vb + kBox, &tm_v, &sh.v_full[s], 64, h, y);
      ++v_issued;
    }
    // drain: every issued copy must land before the CTA may exit (even after an abort)
    mbar_wait_drain(&sh.q_full, 0);
    for (int kt = (k_issued > 2 ? k_issued - 2 : 0); kt < k_issued; ++kt)
      mbar_wait_drain(&sh.k_full[kt & 1], (kt >> 1) & 1);
    for (int kt = (v_issued > 2 ? v_issued - 2 : 0); kt < v_issued; ++kt)
      mbar_wait_drain(&sh.v_full[kt & 1], (kt >> 1) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_f16(128, kBK, 1, 0, 0);  // A, B K-major
    constexpr uint32_t idesc_o = idesc_f16(128, kDV, 0, 0, 1);  // fp16 P and V; V MN-major
    const uint64_t desc_q = smem_desc(smem_u32(smem + kOffQ), 16, 1024);
    const uint64_t desc_k = smem_desc(smem_u32(smem + kOffK), 16, 1024);
    const uint64_t desc_v = smem_desc(smem_u32(smem + kOffV), kBox, 1024);
    auto issue_s = [&](int kt) -> bool {
      const int s = kt & 1;
      if (!warp_wait(&sh.k_full[s], (kt >> 1) & 1, abort)) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t kd = desc_k + (uint64_t)((s * 3 * kBox) >> 4);
#pragma unroll
        for (int ks = 0; ks < kDQK / 16; ++ks) {
          const uint64_t off = (uint64_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4);
          mma_ss(tmem + s * 128, desc_q + off, kd + off, idesc_s, ks > 0 ? 1u : 0u);
        }
        mma_commit(&sh.s_full[s]);
        mma_commit(&sh.k_empty[s]);
      }
      __syncwarp();
      return true;
    };
    bool ok = warp_wait(&sh.q_full, 0, abort);
    if (ok) {
      tc_fence_after();
      ok = issue_s(0) && (n_kt < 2 || issue_s(1));
    }
    for (int kt = 0; ok && kt < n_kt; ++kt) {
      const int s = kt & 1;
      if (!warp_wait(&sh.p_full[s], (kt >> 1) & 1, abort) ||
          !warp_wait(&sh.v_full[s], (kt >> 1) & 1, abort))
        break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t vd = desc_v + (uint64_t)((s * 2 * kBox) >> 4);
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks)  // P: 8 TMEM columns (16 keys) per step
          mma_ts(tmem + kColO, tmem + s * 128 + ks * 8, vd + (uint64_t)((ks * 2048) >> 4),
                 idesc_o, (kt > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&sh.v_empty[s]);
        mma_commit(&sh.pv_done);
      }
      __syncwarp();
      // the next score tile for this buffer is queued behind PV(kt), which reads P from it
      if (kt + 2 < n_kt && !issue_s(kt + 2)) break;
    }
    // every MMA issued by this CTA completes before its tensor memory is freed
    if (elect_one()) mma_commit(&sh.mma_done);
    __syncwarp();
    mbar_wait_drain(&sh.mma_done, 0);
  } else if (warp >= 2) {
    // ------------------------------------------------------------- softmax warps
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // key columns [64 half, 64 half + 64) of a tile
    const int row = q * 32 + lane;     // query row = TMEM lane
    const int qi = qt * kBQ + row;     // position of this query in its sequence
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    float m_used = -INFINITY, l_half = 0.f;
    // `ok` is warp-uniform; after a failed (timed-out) wait a warp skips all work but still
    // takes part in every named barrier, so that the other softmax warps never block on it
    bool ok = true;
    for (int kt = 0; kt < n_kt; ++kt) {
      const int s = kt & 1;
      float sc[64];
      if (ok) ok = warp_wait(&sh.s_full[s], (kt >> 1) & 1, abort);
      if (ok) {
        tc_fence_after();
        tmem_ld32(lane_base + s * 128 + half * 64, *reinterpret_cast<float(*)[32]>(&sc[0]));
        tmem_ld32(lane_base + s * 128 + half * 64 + 32, *reinterpret_cast<float(*)[32]>(&sc[32]));
        tmem_wait_ld();
        // keys j <= qi inside the sequence: only the diagonal tile and a ragged tail are partial
        const int kmax = min(qi, T - 1) - kt * kBK - half * 64;  // last allowed column index
        if (kt == qt || (kt + 1) * kBK > T) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > kmax) sc[i] = -INFINITY;
        }
        float mx[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
        for (int i = 4; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], sc[i]);
        sh.row_max[kt & 1][half][row] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the two halves of every row
      if (!ok) continue;
      const float mt =
          fmaxf(sh.row_max[kt & 1][0][row], sh.row_max[kt & 1][1][row]) * scale_log2;
      const bool first = kt == 0;
      const float m_new = first ? mt : (mt > m_used + kTau ? mt : m_used);
      const float alpha = (first || m_new == -INFINITY) ? 0.f : ex2(m_used - m_new);
      const float base = m_new == -INFINITY ? 0.f : m_new;  // rows with no key yet
      m_used = m_new;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = ex2(fmaf(sc[2 * k], scale_log2, -base));
        const float p1 = ex2(fmaf(sc[2 * k + 1], scale_log2, -base));
        w[k] = pack2(p0, p1);
        // the row sum is of the rounded P, so the normalisation matches what PV multiplies
        const __half2 pr = *reinterpret_cast<const __half2*>(&w[k]);
        ls[k & 3] += __low2float(pr) + __high2float(pr);
      }
      tmem_st32u(lane_base + s * 128 + half * 32, w);
      l_half = l_half * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      // O may be rescaled only once the previous PV has completed
      if (kt > 0) ok = warp_wait(&sh.pv_done, (kt - 1) & 1, abort);
      if (!ok) continue;
      if (__any_sync(0xffffffffu, !first && alpha != 1.f)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float ov[32];
          tmem_ld32(lane_base + kColO + half * 64 + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) ov[k] *= alpha;
          tmem_st32(lane_base + kColO + half * 64 + c * 32, ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full[s]);
    }
    // row sum = both halves' partial sums (they saw the same sequence of maxima)
    sh.row_sum[half][row] = l_half;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const float l_sum = sh.row_sum[0][row] + sh.row_sum[1][row];
    if (ok && warp_wait(&sh.pv_done, (n_kt - 1) & 1, abort)) {
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      float4* dst =
          reinterpret_cast<float4*>(o + ((int64_t)(t0 + qi) * kH + h) * kDV + half * 64);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float ov[32];
        tmem_ld32(lane_base + kColO + half * 64 + c * 32, ov);
        tmem_wait_ld();
        if (qi < T) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[c * 8 + k] = make_float4(ov[4 * k] * inv_l, ov[4 * k + 1] * inv_l,
                                         ov[4 * k + 2] * inv_l, ov[4 * k + 3] * inv_l);
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Token -> (sequence, position) map of the packed prompt (binary search in cu_seqlens).
__global__ void prefill_token_map_kernel(const int32_t* __restrict__ cu, int B, int n_tok,
                                         int max_T, int32_t* __restrict__ tok_seq,
                                         int32_t* __restrict__ tok_pos) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= n_tok) return;
  int lo = 0, hi = B;  // find b with cu[b] <= n < cu[b+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= n) lo = mid; else hi = mid;
  }
  const int p = n - cu[lo];
  if (p >= max_T) flag_status(MLA_ERR_LENGTH);
  tok_seq[n] = lo;
  tok_pos[n] = p;
}

struct Layout {
  size_t off_seq, off_pos, off_lat, off_hi, off_q, off_kc, off_v, total;
};

Layout layout(const mla_dims_t* d, int n) {
  Layout L;
  L.off_seq = 0;
  L.off_pos = align_up(L.off_seq + (size_t)n * 4, 256);
  L.off_lat = align_up(L.off_pos + (size_t)n * 4, 256);
  L.off_hi = align_up(L.off_lat + (size_t)n * kRow * 2, 256);
  L.off_q = align_up(L.off_hi + (size_t)n * d->d_cq * 2, 256);
  L.off_kc = align_up(L.off_q + (size_t)n * kH * kDQK * 2, 256);
  L.off_v = align_up(L.off_kc + (size_t)n * kH * kDV * 2, 256);
  L.total = align_up(L.off_v + (size_t)n * kH * kDV * 2, 256);
  return L;
}

bool map3(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
          uint32_t box_outer) {
  const uint64_t dims[3] = {inner, mid, outer};
  const uint64_t strides[2] = {inner * 2, inner * mid * 2};
  const uint32_t box[3] = {64, 1, box_outer};
  return make_tmap(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

}  // namespace

size_t tc_prefill_ws(const mla_dims_t* d, int n_tok) { return layout(d, n_tok).total; }

mla_status_t tc_prefill(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                        const int32_t* cu, int B, int n, int max_T, mla_cache_t* cache, void* ws,
                        float* o, cudaStream_t st) {
  const Layout L = layout(d, n);
  char* wsb = (char*)ws;
  int32_t* tseq = (int32_t*)(wsb + L.off_seq);
  int32_t* tpos = (int32_t*)(wsb + L.off_pos);
  void* lat = wsb + L.off_lat;
  void* cq_hi = wsb + L.off_hi;
  __nv_bfloat16* Q = (__nv_bfloat16*)(wsb + L.off_q);
  void* KC = wsb + L.off_kc;
  void* V = wsb + L.off_v;
  {
    TraceScope ts(K_TOKEN_MAP, st);
    prefill_token_map_kernel<<<ceil_div(n, 256), 256, 0, st>>>(cu, B, n, max_T, tseq, tpos);
  }
  mla_status_t s = launch_status();
  if (s != MLA_OK) return s;
  // cache rows for every prompt token (plus a packed copy the expansion and k^R loads read)
  s = tc_append(d, w, h, tseq, tpos, n, cache, lat, K_PREFILL_APPEND, st);
  if (s != MLA_OK) return s;
  // queries: c^Q, then [q^C ; q^R] per head, interleaved [n, n_h, 192]
  // c^Q as one bf16 operand (the error budget of the path is set by P and V, kept in fp16)
  s = tc_q_down(d, w, h, n, cq_hi, nullptr, K_PREFILL_Q_DOWN, st);
  if (s != MLA_OK) return s;
  s = tc_q_up(d, w, cq_hi, nullptr, tpos, n, Q, Q + d->d_hc, (int64_t)kH * kDQK, kDQK,
              (int64_t)kH * kDQK, kDQK, false, K_PREFILL_Q_UP, st);
  if (s != MLA_OK) return s;
  // K^C and V per head from the latent rows
  s = tc_expand(w->W_UK, kH * kDV, lat, kRow, kDC, n, KC, false, K_EXPAND_K, st);
  if (s != MLA_OK) return s;
  s = tc_expand(w->W_UV, kH * kDV, lat, kRow, kDC, n, V, true, K_EXPAND_V, st);  // fp16
  if (s != MLA_OK) return s;
  // causal attention
  CUtensorMap tq, tkc, tv, tkr;
  if (!map3(&tq, Q, kDQK, kH, n, kBQ) || !map3(&tkc, KC, kDV, kH, n, kBK) ||
      !map3(&tv, V, kDV, kH, n, kBK))
    return MLA_ERR_CUDA;
  {
    const uint64_t dims[2] = {(uint64_t)kRow, (uint64_t)n};
    const uint64_t strides[1] = {(uint64_t)kRow * 2};
    const uint32_t box[2] = {64, kBK};
    if (!make_tmap(&tkr, lat, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
      return MLA_ERR_CUDA;
  }
  {
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(prefill_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes) != cudaSuccess)
        return MLA_ERR_CUDA;
      attr_done[dev] = true;
    }
  }
  const float scale_log2 = softmax_scale(d) * 1.4426950408889634f;
  dim3 grid(ceil_div(max_T, kBQ), kH, B);
  TraceScope ts(K_PREFILL_ATTN, st);
  prefill_attn_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, tkc, tv, tkr, cu, scale_log2, o);
  return launch_status();
}

}  // namespace mla
