// Fused query up-projection and absorption for decode, DeepSeek-V2 widths (n_h 128, d_h^C 128,
// d_h^R 64, d_c 512, bf16). "MLA前向计算流程" §三分支计算 ① Query gives
//   q^C_i = W^UQ_i c^Q,   q^R_i = RoPE(W^QR_i c^Q)   (per head, at the token's position),
// and "从LLaMA到DeepSeek[01] - MLA（上）" §六 moves W^UK onto the query by associativity:
//   q~_i = (W^UK_i)^T q^C_i   (d_c = 512 wide),
// so decode attends over the cached latent directly. Here both products run in one kernel and
// q^C never leaves the SM. One CTA per (head i, up to BN tokens), 6 warps:
//   warp 0    TMA producer: 24 chunks of 64 K-columns of [W^UQ_i ; W^QR_i] and of c^Q (a hi/lo
//             bf16 pair), then the 8 tiles of W^UK_i (read MN-major), through one ring
//   warp 1    MMA issuer
//             phase 1: D1 = W^UQ_i [hi ; lo]^T (M = 128) and W^QR_i [hi ; lo]^T (M = 64), each
//                      one MMA of width 2 BN per K-step (the weight slice is read once)
//             phase 2: D2[mt] = (W^UK_i)^T tile mt (M = 128 latent rows) q^C^T, K = 128, into the
//                      tensor-memory columns phase 1 used
//   warps 2-5 epilogue 1: q^C = hi + lo rounded to bf16 into shared memory as phase 2's K-major
//             B operand; q^R = hi + lo rotated by RoPE and stored
//             epilogue 2: q~ rounded to bf16 and stored
// The rounding points are those of the two-launch path (c^Q as hi/lo, q^C and q~ in bf16).
// An M = 64 accumulator holds its rows 16q .. 16q+15 in TMEM lanes 32q .. 32q+15.
#include <mutex>

#include "internal.h"
#include "tc.cuh"

namespace mla {

using namespace tc;

namespace {

constexpr int kH = 128;     // n_h
constexpr int kDHC = 128;   // d_h^C
constexpr int kDHR = 64;    // d_h^R
constexpr int kDC = 512;    // d_c
constexpr int kThreads = 192;

template <int BN>
struct QaLayout {
  static constexpr uint32_t kA0 = 128 * 128;      // W^UQ_i chunk: 128 rows x 64 bf16
  static constexpr uint32_t kA1 = 64 * 128;       // W^QR_i chunk: 64 rows x 64 bf16
  static constexpr uint32_t kB = BN * 128;        // c^Q chunk, one of hi / lo
  static constexpr uint32_t kStage = kA0 + kA1 + 2 * kB;
  static constexpr uint32_t kQc = 2 * BN * 128;   // q^C: 2 K-chunks of BN rows x 128 B
  static constexpr int kStages = (232448 - 1024 - 256 - (int)kQc) / (int)kStage;
  static constexpr uint32_t kOffQc = kStages * kStage;
  static constexpr uint32_t kOffBar = kOffQc + kQc;
  static constexpr uint32_t kBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kTmemCols = 4 * BN;   // D1: 2 x 2BN; D2: 4 x BN (reused)
  static_assert(kStages >= 3 && kStages <= 8, "ring depth");
  static_assert(kStage >= 2 * 8192, "a phase-2 tile (two 8 KB boxes) fits in a stage");
  static_assert(kStage % 1024 == 0 && kOffQc % 1024 == 0, "1 KB alignment");
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    qabsorb_kernel(const __grid_constant__ CUtensorMap tm_uq,  // W^UQ [n_h*128, d_c'], box 64x128
                   const __grid_constant__ CUtensorMap tm_qr,  // W^QR [n_h*64, d_c'], box 64x64
                   const __grid_constant__ CUtensorMap tm_hi,  // c^Q hi [n, d_c'], box 64xBN
                   const __grid_constant__ CUtensorMap tm_lo,  // c^Q lo
                   const __grid_constant__ CUtensorMap tm_uk,  // W^UK [n_h*128, d_c], box 64x64
                   int k_chunks, const int32_t* __restrict__ pos, int n,
                   __nv_bfloat16* __restrict__ q_t, __nv_bfloat16* __restrict__ q_r,
                   RopeFreqs rf) {
  using L = QaLayout<BN>;
  constexpr int S = L::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* empty = full + S;
  uint64_t* d1_full = empty + S;
  uint64_t* qc_ready = d1_full + 1;
  uint64_t* d2_full = qc_ready + 1;
  uint64_t* mma_done = d2_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* qc = smem + L::kOffQc;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.x;
  const int n0 = blockIdx.y * BN;
  const int n1 = k_chunks + 8;  // ring uses: phase 1 chunks, then 4 M-tiles x 2 K-chunks

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(d1_full, 1);
    mbar_init(qc_ready, 4);
    mbar_init(d2_full, 1);
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // c^Q comes from the kernel before this one, which may still be running (programmatic
  // dependent launch): wait for it. Then the attention kernel after this one may be scheduled;
  // it reads the cache rows that the down-projection wrote, complete once this wait returns.
  griddep_wait();
  griddep_launch();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    tma_prefetch(&tm_uq);
    tma_prefetch(&tm_qr);
    tma_prefetch(&tm_hi);
    tma_prefetch(&tm_uk);
    int issued = 0;
    for (int g = 0; g < n1; ++g) {
      const int s = g % S, r = g / S;
      if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort)) break;
      uint8_t* st = smem + s * L::kStage;
      if (g < k_chunks) {
        const int x = g * 64;
        mbar_arrive_expect_tx(&full[s], L::kStage);
        tma_load_2d(st, &tm_uq, &full[s], x, head * kDHC);
        tma_load_2d(st + L::kA0, &tm_qr, &full[s], x, head * kDHR);
        tma_load_2d(st + L::kA0 + L::kA1, &tm_hi, &full[s], x, n0);
        tma_load_2d(st + L::kA0 + L::kA1 + L::kB, &tm_lo, &full[s], x, n0);
      } else {
        // (W^UK_i)^T tile mt, K-chunk kc: rows head*128 + 64 kc .. +63 of W^UK (d_h^C), columns
        // 128 mt .. +127 (latent) as two 64-column boxes, MN-major
        const int t = g - k_chunks, mt = t >> 1, kc = t & 1;
        mbar_arrive_expect_tx(&full[s], 2 * 8192);
        tma_load_2d(st, &tm_uk, &full[s], mt * 128, head * kDHC + kc * 64);
        tma_load_2d(st + 8192, &tm_uk, &full[s], mt * 128 + 64, head * kDHC + kc * 64);
      }
      ++issued;
    }
    // every issued copy lands before the CTA may exit (even after an abort)
    for (int g = (issued > S ? issued - S : 0); g < issued; ++g)
      mbar_wait_drain(&full[g % S], (g / S) & 1);
  } else if (warp == 1) {
    // ---------------- MMA issuer
    constexpr uint32_t id_uq = idesc_f16(128, 2 * BN, 1, 0, 0);
    constexpr uint32_t id_qr = idesc_f16(64, 2 * BN, 1, 0, 0);
    constexpr uint32_t id_uk = idesc_f16(128, BN, 1, 1, 0);  // A (W^UK_i)^T MN-major
    const uint64_t d0 = smem_desc(smem_u32(smem), 16, 1024);
    const uint64_t d0mn = smem_desc(smem_u32(smem), 8192, 1024);
    const uint64_t dqc = smem_desc(smem_u32(qc), 16, 1024);
    bool ok = true;
    for (int g = 0; ok && g < k_chunks; ++g) {
      const int s = g % S;
      if (!(ok = warp_wait(&full[s], (g / S) & 1, abort))) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t base = d0 + (uint64_t)((s * L::kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t b = base + (uint64_t)((L::kA0 + L::kA1 + kk * 32) >> 4);
          const uint32_t acc = (g | kk) != 0 ? 1u : 0u;
          mma_ss(tmem, base + (uint64_t)((kk * 32) >> 4), b, id_uq, acc);
          mma_ss(tmem + 2 * BN, base + (uint64_t)((L::kA0 + kk * 32) >> 4), b, id_qr, acc);
        }
        mma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (ok) {
      if (elect_one()) mma_commit(d1_full);
      __syncwarp();
      // phase 2 reuses D1's columns once the epilogue has read them and written q^C
      ok = warp_wait(qc_ready, 0, abort);
      if (ok) tc_fence_after();
    }
    for (int g = k_chunks; ok && g < n1; ++g) {
      const int s = g % S, t = g - k_chunks, mt = t >> 1, kc = t & 1;
      if (!(ok = warp_wait(&full[s], (g / S) & 1, abort))) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t a = d0mn + (uint64_t)((s * L::kStage) >> 4);
        const uint64_t b = dqc + (uint64_t)((kc * BN * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem + mt * BN, a + (uint64_t)((kk * 2048) >> 4), b + (uint64_t)((kk * 32) >> 4),
                 id_uk, (kc | kk) != 0 ? 1u : 0u);
        mma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (ok) {
      if (elect_one()) mma_commit(d2_full);
      __syncwarp();
    }
    // every MMA issued by this CTA completes before its tensor memory is freed
    if (elect_one()) mma_commit(mma_done);
    __syncwarp();
    mbar_wait_drain(mma_done, 0);
  } else if (warp >= 2) {
    // ---------------- epilogues (warp w reads TMEM lanes 32 (w % 4) .. +31)
    const int q = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    bool ok = warp_wait(d1_full, 0, abort);
    if (ok) {
      tc_fence_after();
      // q^C: lane = feature f of head i; column t = token (hi), BN + t (lo)
      const int f = q * 32 + lane;
      const uint32_t unit = (uint32_t)((f & 63) >> 3), byte = (uint32_t)(f & 7) * 2;
      uint8_t* chunk = qc + (f >> 6) * (BN * 128);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float hi[32], lo[32];
        tmem_ld32(lane_base + c0, hi);
        tmem_ld32(lane_base + BN + c0, lo);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int row = c0 + t;
          *reinterpret_cast<__nv_bfloat16*>(chunk + row * 128 + ((unit ^ (uint32_t)(row & 7)) << 4) +
                                            byte) = __float2bfloat16_rn(hi[t] + lo[t]);
        }
      }
      // q^R: the M = 64 accumulator's row e = 16 q + j sits in lane 32 q + j (j < 16); RoPE
      // pairs (2k, 2k+1) are adjacent lanes
      const int e = 16 * q + (lane & 15);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float hi[32], lo[32];
        tmem_ld32(lane_base + 2 * BN + c0, hi);
        tmem_ld32(lane_base + 3 * BN + c0, lo);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const float v = hi[t] + lo[t];
          const float vp = __shfl_xor_sync(0xffffffffu, v, 1);
          const int tok = n0 + c0 + t;
          if (lane < 16 && tok < n) {
            float c, s;
            rope_cs(pos[tok], e >> 1, rf, &c, &s);
            const float r = (e & 1) ? (vp * s + v * c) : (v * c - vp * s);
            q_r[((int64_t)tok * kH + head) * kDHR + e] = __float2bfloat16_rn(r);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qc_ready);
      ok = warp_wait(d2_full, 0, abort);
    }
    if (ok) {
      tc_fence_after();
      // q~: tile mt, lane = latent column 128 mt + 32 q + lane; column t = token
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(lane_base + mt * BN + c0, v);
          tmem_wait_ld();
          const int l = mt * 128 + q * 32 + lane;
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const int tok = n0 + c0 + t;
            if (tok < n) q_t[((int64_t)tok * kH + head) * kDC + l] = __float2bfloat16_rn(v[t]);
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

bool map2(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return make_tmap(m, base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

template <int BN>
mla_status_t launch_qabsorb(const mla_dims_t* d, const mla_weights_t* w, const void* cq_hi,
                            const void* cq_lo, const int32_t* pos, int n, void* q_t, void* q_r,
                            cudaStream_t st) {
  using L = QaLayout<BN>;
  CUtensorMap tuq, tqr, thi, tlo, tuk;
  if (!map2(&tuq, w->W_UQ, (uint64_t)kH * kDHC, d->d_cq, 128) ||
      !map2(&tqr, w->W_QR, (uint64_t)kH * kDHR, d->d_cq, 64) ||
      !map2(&thi, cq_hi, n, d->d_cq, BN) || !map2(&tlo, cq_lo, n, d->d_cq, BN) ||
      !map2(&tuk, w->W_UK, (uint64_t)kH * kDHC, kDC, 64))
    return MLA_ERR_CUDA;
  static std::mutex mu;
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(qabsorb_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               L::kBytes) != cudaSuccess)
        return MLA_ERR_CUDA;
      attr_done[dev] = true;
    }
  }
  // always right after the c^Q down-projection of the same call: its set-up may overlap the
  // end of that kernel (programmatic dependent launch); it waits before reading c^Q
  TraceScope ts(K_Q_ABSORB, st);
  if (launch_maybe_pdl(qabsorb_kernel<BN>, dim3(kH, ceil_div(n, BN)), dim3(kThreads), L::kBytes,
                       st, true, tuq, tqr, thi, tlo, tuk, d->d_cq / 64, pos, n,
                       (__nv_bfloat16*)q_t, (__nv_bfloat16*)q_r, rope_freqs(d)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

mla_status_t tc_q_absorbed(const mla_dims_t* d, const mla_weights_t* w, const void* cq_hi,
                           const void* cq_lo, const int32_t* pos, int n, void* q_t, void* q_r,
                           cudaStream_t st) {
  if (n <= 0) return MLA_OK;
  if (d->d_cq % 64) return MLA_ERR_UNSUPPORTED;
  if (n <= 32) return launch_qabsorb<32>(d, w, cq_hi, cq_lo, pos, n, q_t, q_r, st);
  return launch_qabsorb<128>(d, w, cq_hi, cq_lo, pos, n, q_t, q_r, st);
}

}  // namespace mla
