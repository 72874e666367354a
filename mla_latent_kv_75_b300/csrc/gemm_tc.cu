// Tensor-core projection GEMM for the MLA projections ("MLA前向计算流程" §三分支计算 ①②③):
//   Y[n, o] = sum_k W[o, k] * X[n, k]      (W stored [out, in], X one token per row)
// computed as D[o, n] = A[o, :] . B[n, :] with A = W (M = output features) and B = X (N =
// tokens), both K-major, bf16 in, fp32 accumulation in tensor memory. One CTA owns a 128 x BN
// output tile: warp 0 streams 64-wide K slices of W and X into a shared-memory ring with TMA,
// warp 1 issues tcgen05.mma, warps 2..5 read the accumulator from TMEM and run the epilogue
// (RoPE on pairs of adjacent output rows, cache-row scatter, dtype conversion).
#include <algorithm>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>

#include "internal.h"
#include "proj_tc.h"
#include "tc.cuh"

namespace mla {

using namespace tc;

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTileA = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxCluster = 8;          // split-K clusters (portable size)

// Shared-memory layout: a ring of stages, each holding one 64-deep K slice of A (16 KB) and of
// the B operand(s) (BN rows each; two with the hi/lo split input), then the barrier block. The
// ring is as deep as fits in ~200 KB (at most 8), so that decode-sized GEMMs (BN = 32) keep
// ~160 KB of weights in flight per SM.
template <int BN, bool kDual, int kMaxStages = 8>
struct ProjSmem {
  static constexpr uint32_t kTileB = BN * 128;
  static constexpr uint32_t kStage = kTileA + (kDual ? 2 : 1) * kTileB;
  static constexpr int kFit = (200 * 1024) / kStage;
  static constexpr int kStages = kFit < kMaxStages ? kFit : kMaxStages;
  static constexpr uint32_t kBars = kStages * kStage;
  static constexpr uint32_t kBytes = kBars + 256;
  static_assert(kBars >= 128 * BN * 4, "split-K receive buffer must fit in the ring");
};

// Operand modes of the projection GEMM.
//   kPlain:     A = [W0; W1] rows (K-major), B = X rows [N, K] (K-major).
//   kGroupedK:  grouped per head: m-tile i belongs to group g = i / mt_group; A rows as in
//               kPlain, B = X[n, g, :] read through a 3-D tensor map (K, groups, N).
//   kGroupedMN: as kGroupedK but A = W^T: A[m, k] = W0[g * K + k, (i % mt_group) * 128 + m],
//               i.e. MN-major (loaded as two 64 x 64 boxes per 64-deep K slice).
enum ProjMode : int { kPlain = 0, kGroupedK = 1, kGroupedMN = 2 };

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c,
                                              float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// One CTA computes a 128 x BN output tile (C = 1; mt_cta consecutive m-tiles per CTA) or, in a
// cluster of C CTAs (2..8, not only powers of two), a 1/C share of the K range of one tile
// (split-K). Split-K partial tiles are reduced through distributed shared memory: CTA c of the
// cluster sums the row pairs [c*64/C, (c+1)*64/C) of all C partials (rows stay in pairs, which
// the RoPE epilogues need) and runs the epilogue on them.
template <int BN, int kMode, bool kDual, int kMaxStages, class Ep>
__global__ void __launch_bounds__(kThreads, kMaxStages <= 4 ? 2 : 1)  // shallow ring: 2 CTAs/SM
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tm_w0,
                     const __grid_constant__ CUtensorMap tm_w1,
                     const __grid_constant__ CUtensorMap tm_w2,
                     const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_x2, int m_tiles0, int m_tiles01,
                     int O, int N, int k_chunks, int mt_group, int mt_cta, int C, Ep ep) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using S = ProjSmem<BN, kDual, kMaxStages>;
  constexpr int kStages = S::kStages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.y * BN;
  const bool split = C > 1;
  const int cl = split ? (int)cluster_ctarank() : 0;
  // The absorb GEMM (the only MN-major use) is followed by the decode attention, launched with
  // programmatic stream serialization: let it be scheduled now (it waits for this grid to
  // complete before it reads q~). Measured: releasing every projection GEMM this way slowed the
  // one-call decode step (the down-projection then lets the fused query kernel in early), so
  // only this one does.
  if constexpr (kMode == kGroupedMN) griddep_launch();
  const int m_first = split ? blockIdx.x / C : blockIdx.x * mt_cta;
  const int n_mt = split ? 1 : mt_cta;
  const int kcp = (k_chunks + C - 1) / C;  // K chunks per cluster rank
  const int kc0 = cl * kcp;
  const int kc_n = min(k_chunks, kc0 + kcp) - kc0;  // >= 1 (C <= k_chunks)
  const int total_chunks = n_mt * kc_n;
  // With the hi/lo input the two B tiles are adjacent in shared memory and one MMA of width
  // 2*BN covers both (the weight slice is read once); the epilogue adds the two halves.
  constexpr int kAccN = kDual ? 2 * BN : BN;  // accumulator columns per output tile
  static_assert(kAccN <= 256, "one MMA is at most 256 columns wide");
  uint32_t tmem_cols = 32;  // a power of two >= the accumulator columns
  while (tmem_cols < (uint32_t)(n_mt * kAccN)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    tma_prefetch(&tm_w0);
    tma_prefetch(&tm_x);
    int issued = 0;
    for (int g = 0; g < total_chunks; ++g) {
      const int i = g / kc_n, kc = kc0 + g % kc_n;
      const int m_tile = m_first + i;
      const int s = g % kStages, r = g / kStages;
      if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort)) break;
      uint8_t* a = smem + s * S::kStage;
      uint8_t* b = a + kTileA;
      mbar_arrive_expect_tx(&full[s], S::kStage);
      const int kx = kc * 64;
      if (kMode == kPlain) {
        // m-tiles [0, m_tiles0) come from W0, [m_tiles0, m_tiles01) from W1, the rest from W2
        const int w_sel = m_tile < m_tiles0 ? 0 : (m_tile < m_tiles01 ? 1 : 2);
        const int w_row = (m_tile - (w_sel == 0 ? 0 : (w_sel == 1 ? m_tiles0 : m_tiles01))) * 128;
        tma_load_2d(a, w_sel == 0 ? &tm_w0 : (w_sel == 1 ? &tm_w1 : &tm_w2), &full[s], kx, w_row);
        tma_load_2d(b, &tm_x, &full[s], kx, n0);
        if (kDual) tma_load_2d(b + S::kTileB, &tm_x2, &full[s], kx, n0);
      } else {
        const int grp = m_tile / mt_group;
        if (kMode == kGroupedK) {
          tma_load_2d(a, &tm_w0, &full[s], kx, m_tile * 128);
        } else {
          const int col = (m_tile % mt_group) * 128, row = grp * k_chunks * 64 + kx;
          tma_load_2d(a, &tm_w0, &full[s], col, row);
          tma_load_2d(a + kTileA / 2, &tm_w0, &full[s], col + 64, row);
        }
        tma_load_3d(b, &tm_x, &full[s], kx, grp, n0);
        if (kDual) tma_load_3d(b + S::kTileB, &tm_x2, &full[s], kx, grp, n0);
      }
      ++issued;
    }
    // drain: every issued copy must land before the CTA may exit (even after an abort)
    for (int g = (issued > kStages ? issued - kStages : 0); g < issued; ++g)
      mbar_wait_drain(&full[g % kStages], (g / kStages) & 1);
  } else if (warp == 1) {
    // ---------------- MMA issuer (one elected lane of the converged warp)
    constexpr uint32_t idesc = idesc_f16(128, kAccN, 1, kMode == kGroupedMN ? 1 : 0, 0);
    const uint64_t a0 = kMode == kGroupedMN ? smem_desc(smem_u32(smem), 8192, 1024)
                                            : smem_desc(smem_u32(smem), 16, 1024);
    const uint64_t b0 = smem_desc(smem_u32(smem) + kTileA, 16, 1024);
    for (int g = 0; g < total_chunks; ++g) {
      const int i = g / kc_n, kc = g % kc_n;
      const int s = g % kStages, r = g / kStages;
      if (!warp_wait(&full[s], r & 1, abort)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t off = (uint64_t)((s * S::kStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t adesc =
              a0 + off + (uint64_t)((kMode == kGroupedMN ? kk * 2048 : kk * 32) >> 4);
          const uint64_t bdesc = b0 + off + (uint64_t)((kk * 32) >> 4);
          mma_ss(tmem + i * kAccN, adesc, bdesc, idesc, (kc | kk) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (elect_one()) mma_commit(done);
    __syncwarp();
  }

  const int q = warp & 3;  // TMEM lane quarter of an epilogue warp
  const bool epi = warp >= 2;
  bool ok = true;
  if (epi) {
    // while the MMAs run: the per-token data the epilogue looks up (positions, row bases)
    for (int n = n0 + lane; n < min(N, n0 + BN); n += 32) ep.warm(n);
    ok = warp_wait(done, 0, abort);
    tc_fence_after();
  }
  if (!split) {
    // ---------------- epilogue: TMEM -> registers -> global
    if (epi && ok) {
#pragma unroll 1
      for (int i = 0; i < n_mt; ++i) {
        const int o = (m_first + i) * 128 + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + i * kAccN + c, v);
          if (kDual) {
            float v2[32];
            tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + i * kAccN + BN + c, v2);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += v2[j];
          }
          tmem_wait_ld();
          float vp[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) vp[j] = __shfl_xor_sync(0xffffffffu, v[j], 1);
          if (o < O) ep.row32(o, n0 + c, N, v, vp);
        }
      }
    }
  } else {
    // ---------------- split-K: all-to-all reduction of the partial tiles through DSMEM
    // CTA c reduces rows [2 * (c*64/C), 2 * ((c+1)*64/C)): at most Rmax rows
    const int Rmax = 2 * ((64 + C - 1) / C);
    float* recv = reinterpret_cast<float*>(smem);  // [C][Rmax][BN], the ring is drained
    __syncthreads();
    cluster_sync();  // every CTA of the cluster finished its MMAs: all rings are free
    if (epi && ok) {
      const int row = q * 32 + lane, pr = row >> 1;
      int dst = pr * C / 64;  // the CTA whose pair range holds pr
      while (dst + 1 < C && (dst + 1) * 64 / C <= pr) ++dst;
      while (dst > 0 && dst * 64 / C > pr) --dst;
      const int rr = row - 2 * (dst * 64 / C);
      const uint32_t base =
          mapa_shared(smem_u32(recv + ((size_t)cl * Rmax + rr) * BN), (uint32_t)dst);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c, v);
        if (kDual) {
          float v2[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + BN + c, v2);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += v2[j];
        }
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_cluster_v4(base + (c + 4 * k) * 4, v[4 * k], v[4 * k + 1], v[4 * k + 2],
                        v[4 * k + 3]);
      }
    }
    cluster_sync();  // all partial rows have arrived
    if (epi) {
      const int ts = threadIdx.x - 64;
      const int p0 = cl * 64 / C, np = (cl + 1) * 64 / C - p0;  // this CTA's row pairs
      for (int e = ts; e < np * BN; e += 128) {
        const int pr = e / BN, col = e % BN;
        float v0 = 0.f, v1 = 0.f;
        for (int src = 0; src < C; ++src) {
          v0 += recv[((size_t)src * Rmax + 2 * pr) * BN + col];
          v1 += recv[((size_t)src * Rmax + 2 * pr + 1) * BN + col];
        }
        const int o = m_first * 128 + 2 * (p0 + pr), n = n0 + col;
        if (n < N && o < O) {
          ep(o, n, v0, v1);
          if (o + 1 < O) ep(o + 1, n, v1, v0);
        }
      }
    }
  }
  if (epi) tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // the MMAs committed to `done` have completed before tensor memory is freed
    mbar_wait_drain(done, 0);
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// Persistent variant of the plain-mode GEMM for many output tiles (prefill-sized N): one CTA
// per SM walks tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... (m-tile fastest, so that the
// CTAs in flight share one activation tile), the TMA ring runs on across tile boundaries, and
// two TMEM accumulators let the epilogue of one tile overlap the MMAs of the next. The epilogue
// (bf16 conversion, RoPE, scattered stores) takes as long as the MMAs at these sizes, so eight
// warps run it: two per TMEM lane quarter, each on half of the tile's columns.
constexpr int kPThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kPEpiWarps = 8;

template <int BN, bool kDual, class Ep>
__global__ void __launch_bounds__(kPThreads, 1)
    proj_gemm_persistent(const __grid_constant__ CUtensorMap tm_w0,
                         const __grid_constant__ CUtensorMap tm_w1,
                         const __grid_constant__ CUtensorMap tm_x,
                         const __grid_constant__ CUtensorMap tm_x2, int m_tiles0, int m_tiles,
                         int n_tiles, int O, int N, int k_chunks, Ep ep) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using S = ProjSmem<BN, kDual>;
  constexpr int kStages = S::kStages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBars);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  constexpr int kAccN = kDual ? 2 * BN : BN;  // hi/lo: one MMA of width 2*BN (see above)
  constexpr uint32_t kCols = 2 * kAccN < 32 ? 32 : 2 * kAccN;
  static_assert(kAccN <= 256, "one MMA is at most 256 columns wide");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_total = m_tiles * n_tiles;
  const int my_tiles = blockIdx.x < n_total ? (n_total - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kPEpiWarps);
    }
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    tma_prefetch(&tm_w0);
    tma_prefetch(&tm_x);
    int g = 0, issued = 0;
    bool ok = true;
    for (int i = 0; ok && i < my_tiles; ++i) {
      const int t = blockIdx.x + i * gridDim.x;
      const int m_tile = t % m_tiles, n0 = (t / m_tiles) * BN;
      const bool from_w1 = m_tile >= m_tiles0;
      const int a_row = (from_w1 ? m_tile - m_tiles0 : m_tile) * 128;
      for (int kc = 0; kc < k_chunks; ++kc, ++g) {
        const int s = g % kStages, r = g / kStages;
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort)) {
          ok = false;
          break;
        }
        uint8_t* a = smem + s * S::kStage;
        uint8_t* b = a + kTileA;
        mbar_arrive_expect_tx(&full[s], S::kStage);
        tma_load_2d(a, from_w1 ? &tm_w1 : &tm_w0, &full[s], kc * 64, a_row);
        tma_load_2d(b, &tm_x, &full[s], kc * 64, n0);
        if (kDual) tma_load_2d(b + S::kTileB, &tm_x2, &full[s], kc * 64, n0);
        ++issued;
      }
    }
    // drain: every issued copy must land before the CTA may exit (even after an abort)
    for (int k = (issued > kStages ? issued - kStages : 0); k < issued; ++k)
      mbar_wait_drain(&full[k % kStages], (k / kStages) & 1);
  } else if (warp == 1) {
    // ---------------- MMA issuer (one elected lane of the converged warp)
    constexpr uint32_t idesc = idesc_f16(128, kAccN, 1, 0, 0);
    const uint64_t a0 = smem_desc(smem_u32(smem), 16, 1024);
    const uint64_t b0 = smem_desc(smem_u32(smem) + kTileA, 16, 1024);
    int g = 0;
    bool ok = true;
    for (int i = 0; ok && i < my_tiles; ++i) {
      const int buf = i & 1;
      // the epilogue has drained this accumulator (passes at once for the first two tiles)
      if (!warp_wait(&acc_empty[buf], ((i >> 1) & 1) ^ 1, abort)) break;
      tc_fence_after();
      for (int kc = 0; kc < k_chunks; ++kc, ++g) {
        const int s = g % kStages, r = g / kStages;
        if (!warp_wait(&full[s], r & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint64_t off = (uint64_t)((s * S::kStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = a0 + off + (uint64_t)((kk * 32) >> 4);
            const uint64_t bdesc = b0 + off + (uint64_t)((kk * 32) >> 4);
            mma_ss(tmem + buf * kAccN, adesc, bdesc, idesc, (kc | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        __syncwarp();
      }
      if (ok) {
        if (elect_one()) mma_commit(&acc_full[buf]);
        __syncwarp();
      }
    }
    // every MMA issued by this CTA completes before its tensor memory is freed
    if (elect_one()) mma_commit(mma_done);
    __syncwarp();
    mbar_wait_drain(mma_done, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue: TMEM -> registers -> global, overlapped with the next tile
    const int q = warp & 3;
    constexpr int kWarpCols = BN >= 64 ? BN / 2 : BN;  // columns per epilogue warp
    const int c_beg = ((warp - 2) >> 2) * kWarpCols;
    for (int i = 0; i < my_tiles; ++i) {
      const int buf = i & 1;
      const int t = blockIdx.x + i * gridDim.x;
      const int m_tile = t % m_tiles, n0 = (t / m_tiles) * BN;
      if (!warp_wait(&acc_full[buf], (i >> 1) & 1, abort)) break;
      tc_fence_after();
      const int o = m_tile * 128 + q * 32 + lane;
#pragma unroll 1
      for (int c = c_beg; c < c_beg + kWarpCols && c < BN; c += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * kAccN + c, v);
        if (kDual) {
          float v2[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * kAccN + BN + c, v2);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += v2[j];
        }
        tmem_wait_ld();
        float vp[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) vp[j] = __shfl_xor_sync(0xffffffffu, v[j], 1);
        if (o < O) ep.row32(o, n0 + c, N, v, vp);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------------- epilogues
// Cache append: rows [0, d_c) of [W^DKV; W^KR] are c^KV, rows [d_c, d_c + d_hr) are k^R,
// rotated by RoPE at the token's position. Optionally also stored to a packed copy. Token n
// belongs to sequence seq_idx[n], or to sequence n when seq_idx is null (a decode step).
struct EpAppend {
  __nv_bfloat16* rows;
  int64_t pitch, capacity;
  const int64_t* seq_base;
  const int32_t* seq_idx;
  const int32_t* pos;
  __nv_bfloat16* packed;  // [N, pitch] or null
  int d_c;
  RopeFreqs rf;
  // Before the accumulator is ready: bring token n's position and row base into L1, so that
  // the epilogue does not wait on the dependent loads seq_idx -> seq_base.
  __device__ void warm(int n) const {
    const int si = seq_idx ? __ldg(seq_idx + n) : n;
    prefetch_l1(seq_base + si);
    prefetch_l1(pos + n);
  }
  __device__ void operator()(int o, int n, float v, float vp) const {
    const int p = pos[n];
    if (o >= d_c) {
      float c, s;
      rope_cs(p, (o - d_c) >> 1, rf, &c, &s);
      v = ((o - d_c) & 1) ? (vp * s + v * c) : (v * c - vp * s);
    }
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    const int64_t row = seq_base[seq_idx ? seq_idx[n] : n] + p;
    if (row < 0 || row >= capacity) {
      flag_status(MLA_ERR_CAPACITY);
    } else {
      rows[row * pitch + o] = b;
    }
    if (packed) packed[(int64_t)n * pitch + o] = b;
  }
  // output row o for tokens nb .. nb+31 (those below N); vp holds the partner rows' values
  __device__ void row32(int o, int nb, int N, const float* v, const float* vp) const {
    const bool rot = o >= d_c;
    const int e = o - d_c;
    const float fh = rot ? rf.hi[e >> 1] : 0.f, fl = rot ? rf.lo[e >> 1] : 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int n = nb + j;
      if (n >= N) break;
      const int p = pos[n];
      float x = v[j];
      if (rot) {
        float c, s;
        rope_cs_f(p, fh, fl, &c, &s);
        x = (e & 1) ? (vp[j] * s + x * c) : (x * c - vp[j] * s);
      }
      const __nv_bfloat16 b = __float2bfloat16_rn(x);
      const int64_t row = seq_base[seq_idx ? seq_idx[n] : n] + p;
      if (row < 0 || row >= capacity)
        flag_status(MLA_ERR_CAPACITY);
      else
        rows[row * pitch + o] = b;
      if (packed) packed[(int64_t)n * pitch + o] = b;
    }
  }
};

// Plain store Y[n * ld + o] in bf16, or as a hi/lo pair of bf16 (v = hi + lo to ~2^-16).
struct EpStoreBF16 {
  __nv_bfloat16* hi;
  __nv_bfloat16* lo;  // null: single bf16
  int64_t ld;
  __device__ void warm(int) const {}
  __device__ void operator()(int o, int n, float v, float) const {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[(int64_t)n * ld + o] = h;
    if (lo) lo[(int64_t)n * ld + o] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
  __device__ void row32(int o, int nb, int N, const float* v, const float*) const {
    __nv_bfloat16* ph = hi + (int64_t)nb * ld + o;
    __nv_bfloat16* pl = lo ? lo + (int64_t)nb * ld + o : nullptr;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (nb + j >= N) break;
      const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
      ph[(int64_t)j * ld] = h;
      if (pl) pl[(int64_t)j * ld] = __float2bfloat16_rn(v[j] - __bfloat162float(h));
    }
  }
};

// Plain store Y[n * ld + o] in fp32.
struct EpStoreF32 {
  float* y;
  int64_t ld;
  __device__ void warm(int) const {}
  __device__ void operator()(int o, int n, float v, float) const { y[(int64_t)n * ld + o] = v; }
  __device__ void row32(int o, int nb, int N, const float* v, const float*) const {
    float* p = y + (int64_t)nb * ld + o;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (nb + j >= N) break;
      p[(int64_t)j * ld] = v[j];
    }
  }
};

// x (float32) -> hi + lo, two bf16 arrays with x = hi + lo to about 2^-16 relative; count is a
// multiple of 4 and the pointers are 16-byte aligned.
__global__ void __launch_bounds__(256) split_hi_lo_kernel(const float4* __restrict__ x,
                                                          uint2* __restrict__ hi,
                                                          uint2* __restrict__ lo, int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = x[i];
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - __low2float(h01), v.y - __high2float(h01));
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - __low2float(h23), v.w - __high2float(h23));
    hi[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
    lo[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
  }
}

// Plain store Y[n * ld + o] in fp16.
struct EpStoreF16 {
  __half* y;
  int64_t ld;
  __device__ void warm(int) const {}
  __device__ void operator()(int o, int n, float v, float) const {
    y[(int64_t)n * ld + o] = __float2half_rn(v);
  }
  __device__ void row32(int o, int nb, int N, const float* v, const float*) const {
    __half* p = y + (int64_t)nb * ld + o;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (nb + j >= N) break;
      p[(int64_t)j * ld] = __float2half_rn(v[j]);
    }
  }
};

// Down-projections of a decode step in one GEMM over [W^DKV; W^KR; W^DQ]: output rows
// [0, d_c + d_hr) are the cache row (EpAppend), rows from q_row0 on are c^Q as a hi/lo pair;
// the rows between (the padding of W^KR's tile) are dropped.
struct EpDown {
  EpAppend app;
  EpStoreBF16 cq;
  int row_end, q_row0;
  __device__ void warm(int n) const { app.warm(n); }
  __device__ void operator()(int o, int n, float v, float vp) const {
    if (o < row_end)
      app(o, n, v, vp);
    else if (o >= q_row0)
      cq(o - q_row0, n, v, vp);
  }
  __device__ void row32(int o, int nb, int N, const float* v, const float* vp) const {
    if (o < row_end)
      app.row32(o, nb, N, v, vp);
    else if (o >= q_row0)
      cq.row32(o - q_row0, nb, N, v, vp);
  }
};



// Query up-projection: rows [0, n_h*d_hc) of [W^UQ; W^QR] are q^C, the rest q^R with RoPE.
template <typename T>
struct EpQuery {
  T* q_c;
  T* q_r;
  int64_t qc_tok, qc_head, qr_tok, qr_head;
  const int32_t* pos;
  int n_h, d_hc, d_hr;
  RopeFreqs rf;
  __device__ void warm(int n) const { prefetch_l1(pos + n); }
  __device__ void operator()(int o, int n, float v, float vp) const {
    const int nc = n_h * d_hc;
    if (o < nc) {
      q_c[n * qc_tok + (o / d_hc) * qc_head + (o % d_hc)] = from_f<T>(v);
    } else {
      const int r = o - nc, i = r / d_hr, e = r % d_hr;
      float c, s;
      rope_cs(pos[n], e >> 1, rf, &c, &s);
      v = (e & 1) ? (vp * s + v * c) : (v * c - vp * s);
      q_r[n * qr_tok + i * qr_head + e] = from_f<T>(v);
    }
  }
  // output row o for tokens nb .. nb+31: the head split, the destination and the RoPE frequency
  // are worked out once per row
  __device__ void row32(int o, int nb, int N, const float* v, const float* vp) const {
    const int nc = n_h * d_hc;
    if (o < nc) {
      T* dst = q_c + (int64_t)nb * qc_tok + (o / d_hc) * qc_head + (o % d_hc);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (nb + j >= N) break;
        dst[(int64_t)j * qc_tok] = from_f<T>(v[j]);
      }
    } else {
      const int r = o - nc, i = r / d_hr, e = r % d_hr;
      const float fh = rf.hi[e >> 1], fl = rf.lo[e >> 1];
      T* dst = q_r + (int64_t)nb * qr_tok + i * qr_head + e;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (nb + j >= N) break;
        float c, s;
        rope_cs_f(pos[nb + j], fh, fl, &c, &s);
        const float x = (e & 1) ? (vp[j] * s + v[j] * c) : (v[j] * c - vp[j] * s);
        dst[(int64_t)j * qr_tok] = from_f<T>(x);
      }
    }
  }
};

bool tmap_rows(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld_elems,
               int box_rows) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)ld_elems * 2};
  const uint32_t box[2] = {64, (uint32_t)box_rows};
  return make_tmap(m, base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// Opt-in shared memory size for a kernel, set once per (function, device).
mla_status_t ensure_smem(const void* fn, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({fn, dev})) return MLA_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return MLA_ERR_CUDA;
  done.insert({fn, dev});
  return MLA_OK;
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

// Clusters of `c` CTAs of kernel `fn` (with `smem` bytes each) that the device holds at once,
// cached per (kernel, size, device); 0 if the query fails.
int max_active_clusters(const void* fn, int c, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int>, int> known;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(fn, c, dev);
  auto it = known.find(key);
  if (it != known.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  known[key] = n;
  return n;
}

// Split-K cluster size: the largest size <= kMaxCluster (any size, not only powers of two)
// whose clusters (one per output tile) are all resident at once, so the grid runs as one wave,
// that leaves every cluster rank at least one K chunk, and whose reduction buffer
// (C x Rmax rows x BN fp32) fits in the drained ring of `ring_bytes`.
int choose_split(int tiles, int k_chunks, int BN, int ring_bytes, const void* fn, int smem) {
  const int sms = sm_count();
  int c = 1;
  for (int n = 2; n <= kMaxCluster && tiles * n <= sms; ++n) {
    const int per = (k_chunks + n - 1) / n;
    if (per * (n - 1) >= k_chunks) continue;  // the last rank would get no K chunk
    if ((size_t)n * 2 * ((64 + n - 1) / n) * BN * 4 > (size_t)ring_bytes) continue;
    if (max_active_clusters(fn, n, smem) < tiles) continue;
    c = n;
  }
  return c;
}

template <int BN, int kMode, bool kDual, int kMaxStages = 8, class Ep>
mla_status_t launch_kernel(const CUtensorMap& tw0, const CUtensorMap& tw1, const CUtensorMap& tw2,
                           const CUtensorMap& tx, const CUtensorMap& tx2, int m_tiles0,
                           int m_tiles01, int O, int N, int k_chunks, int mt_group, int mt_cta,
                           int C, int grid_x, int kid, const Ep& ep, cudaStream_t st) {
  const uint32_t smem = ProjSmem<BN, kDual, kMaxStages>::kBytes + 1024;
  auto kern = proj_gemm_kernel<BN, kMode, kDual, kMaxStages, Ep>;
  mla_status_t s = ensure_smem((const void*)kern, (int)smem);
  if (s != MLA_OK) return s;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, ceil_div(N, BN), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TraceScope ts(kid, st);
  if (cudaLaunchKernelEx(&cfg, kern, tw0, tw1, tw2, tx, tx2, m_tiles0, m_tiles01, O, N, k_chunks,
                         mt_group, mt_cta, C, ep) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

template <int BN, bool kDual, class Ep>
mla_status_t launch_persistent(const CUtensorMap& tw0, const CUtensorMap& tw1,
                               const CUtensorMap& tx, const CUtensorMap& tx2, int m_tiles0,
                               int m_tiles, int O, int N, int k_chunks, int kid, const Ep& ep,
                               cudaStream_t st) {
  const uint32_t smem = ProjSmem<BN, kDual>::kBytes + 1024;
  auto kern = proj_gemm_persistent<BN, kDual, Ep>;
  mla_status_t s = ensure_smem((const void*)kern, (int)smem);
  if (s != MLA_OK) return s;
  const int n_tiles = ceil_div(N, BN);
  const int grid = min(sm_count(), m_tiles * n_tiles);
  TraceScope ts(kid, st);
  kern<<<grid, kPThreads, smem, st>>>(tw0, tw1, tx, tx2, m_tiles0, m_tiles, n_tiles, O, N,
                                      k_chunks, ep);
  return launch_status();
}

template <int BN, class Ep>
mla_status_t launch_proj_bn(const ProjArgs& a, const Ep& ep, cudaStream_t st) {
  CUtensorMap tw0, tw1, tw2, tx, tx2;
  const int m0 = a.O0 / 128;
  if (!tmap_rows(&tw0, a.W0, a.O0, a.K, a.K, 128)) return MLA_ERR_CUDA;
  if (!tmap_rows(&tw1, a.W1 ? a.W1 : a.W0, a.W1 ? a.O1 : a.O0, a.K, a.K, 128)) return MLA_ERR_CUDA;
  if (!tmap_rows(&tw2, a.W2 ? a.W2 : a.W0, a.W2 ? a.O2 : a.O0, a.K, a.K, 128)) return MLA_ERR_CUDA;
  if (!tmap_rows(&tx, a.X, a.N, a.K, a.ldx, BN)) return MLA_ERR_CUDA;
  if (!tmap_rows(&tx2, a.X2 ? a.X2 : a.X, a.N, a.K, a.ldx, BN)) return MLA_ERR_CUDA;
  // a W1 block that is not a multiple of 128 rows is padded to whole tiles (rows read past it
  // are zero), so W2's rows start at output row (m0 + ceil(O1 / 128)) * 128
  const int m01 = m0 + (a.W1 ? ceil_div(a.O1, 128) : 0);
  const int m_tiles = m01 + (a.W2 ? ceil_div(a.O2, 128) : 0);
  const int k_chunks = a.K / 64;
  // split-K kernel of this launch (cluster size chosen against its residency)
  const void* split_fn = (const void*)proj_gemm_kernel<BN, kPlain, false, 8, Ep>;
  int split_smem = (int)ProjSmem<BN, false>::kBytes + 1024;
  int split_ring = (int)ProjSmem<BN, false>::kBars;
  if constexpr (BN <= 128) {  // hi/lo inputs need MMAs of width 2*BN
    if (a.X2) {
      split_fn = (const void*)proj_gemm_kernel<BN, kPlain, true, 8, Ep>;
      split_smem = (int)ProjSmem<BN, true>::kBytes + 1024;
      split_ring = (int)ProjSmem<BN, true>::kBars;
    }
  }
  int C = 1;
  if (m_tiles * ceil_div(a.N, BN) * 2 <= sm_count()) {
    mla_status_t es = ensure_smem(split_fn, split_smem);
    if (es != MLA_OK) return es;
    C = choose_split(m_tiles * ceil_div(a.N, BN), k_chunks, BN, split_ring, split_fn, split_smem);
  }
  const int O = a.W2 ? m01 * 128 + a.O2 : a.O0 + (a.W1 ? a.O1 : 0);
  if (a.W2 && m_tiles * ceil_div(a.N, BN) > sm_count()) return MLA_ERR_UNSUPPORTED;
  if (m_tiles * ceil_div(a.N, BN) > sm_count()) {
    if constexpr (BN == 32)
      if (m_tiles <= 2 * sm_count()) {
        // Decode sizes (one token tile, up to two m-tiles per SM): a 4-deep ring lets two CTAs
        // share an SM, so every m-tile streams its weights at once in a single wave instead of
        // a persistent CTA walking a second tile after the others have finished.
        if (a.X2)
          return launch_kernel<BN, kPlain, true, 4>(tw0, tw1, tw2, tx, tx2, m0, m01, O, a.N,
                                                    k_chunks, 1, 1, 1, m_tiles, a.kid, ep, st);
        return launch_kernel<BN, kPlain, false, 4>(tw0, tw1, tw2, tx, tx2, m0, m01, O, a.N,
                                                   k_chunks, 1, 1, 1, m_tiles, a.kid, ep, st);
      }
    if (a.X2) {
      if constexpr (BN <= 128)  // two accumulators of width 2*BN must fit in tensor memory
        return launch_persistent<BN, true>(tw0, tw1, tx, tx2, m0, m_tiles, O, a.N, k_chunks,
                                           a.kid, ep, st);
      else
        return MLA_ERR_UNSUPPORTED;
    }
    return launch_persistent<BN, false>(tw0, tw1, tx, tx2, m0, m_tiles, O, a.N, k_chunks,
                                        a.kid, ep, st);
  }
  if (a.X2) {
    if constexpr (BN <= 128)  // one MMA covers both halves: 2*BN columns, at most 256
      return launch_kernel<BN, kPlain, true>(tw0, tw1, tw2, tx, tx2, m0, m01, O, a.N, k_chunks, 1,
                                             1, C, m_tiles * C, a.kid, ep, st);
    else
      return MLA_ERR_UNSUPPORTED;
  }
  return launch_kernel<BN, kPlain, false>(tw0, tw1, tw2, tx, tx2, m0, m01, O, a.N, k_chunks, 1, 1,
                                          C, m_tiles * C, a.kid, ep, st);
}

template <class Ep>
mla_status_t launch_proj(const ProjArgs& a, const Ep& ep, cudaStream_t st) {
  if (a.N <= 0) return MLA_OK;
  if (a.K % 64 || a.O0 % 128) return MLA_ERR_UNSUPPORTED;
  if (a.N <= 32) return launch_proj_bn<32>(a, ep, st);
  if (a.N <= 64) return launch_proj_bn<64>(a, ep, st);
  if (a.N <= 128 || a.X2) return launch_proj_bn<128>(a, ep, st);  // hi/lo: 4 ring stages
  return launch_proj_bn<256>(a, ep, st);
}

// Grouped GEMM over heads: Y[n, g*Mg + m] = sum_k A_g[m, k] X[n, g, k] for g < G heads, with
// A_g the head-g block of W ([G*Mg, K] row-major, kGroupedK) or of W^T (W [G*K, Mg]
// row-major, kGroupedMN). X (and X2, accumulated against the same A) is [N, G, K] bf16.
struct GroupArgs {
  const void* W;
  int G, Mg, K;
  const void* X;
  const void* X2;
  int N;
  int kid;
};

template <int BN, int kMode, class Ep>
mla_status_t launch_grouped_bn(const GroupArgs& a, const Ep& ep, cudaStream_t st) {
  CUtensorMap tw, tx, tx2;
  if (kMode == kGroupedK) {
    if (!tmap_rows(&tw, a.W, (int64_t)a.G * a.Mg, a.K, a.K, 128)) return MLA_ERR_CUDA;
  } else {
    if (!tmap_rows(&tw, a.W, (int64_t)a.G * a.K, a.Mg, a.Mg, 64)) return MLA_ERR_CUDA;
  }
  auto map3 = [&](CUtensorMap* m, const void* base) {
    const uint64_t dims[3] = {(uint64_t)a.K, (uint64_t)a.G, (uint64_t)a.N};
    const uint64_t strides[2] = {(uint64_t)a.K * 2, (uint64_t)a.G * a.K * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)BN};
    return make_tmap(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  };
  if (!map3(&tx, a.X) || !map3(&tx2, a.X2 ? a.X2 : a.X)) return MLA_ERR_CUDA;
  const int mt_group = a.Mg / 128;
  int mt_cta = mt_group;
  const int acc_n = a.X2 ? 2 * BN : BN;  // accumulator columns per tile (hi/lo: both halves)
  while (mt_cta * acc_n > 512 || mt_group % mt_cta) --mt_cta;
  const int m_tiles = a.G * mt_group;
  const int k_chunks = a.K / 64;
  if constexpr (BN == 32) if (!a.X2) {
    // Decode sizes, single input (the absorb): a 4-deep ring lets two CTAs share an SM, at most
    // two output tiles per CTA and, with one tile per CTA, split-K clusters over the K range, so
    // that the grid runs as one wave of short-lived CTAs instead of 128 long ones.
    const int sms = sm_count();
    int mtc = mt_group < 2 ? mt_group : 2;
    while (mt_group % mtc) --mtc;
    int C = 1;
    if (mtc == 1)
      while (2 * C <= kMaxCluster && k_chunks % (2 * C) == 0 && k_chunks / (2 * C) >= 2 &&
             m_tiles * 2 * C <= 2 * sms)
        C *= 2;
    const int grid_x = (m_tiles / mtc) * C;
    return launch_kernel<BN, kMode, false, 4>(tw, tw, tw, tx, tx2, m_tiles, m_tiles, a.G * a.Mg,
                                              a.N, k_chunks, mt_group, mtc, C, grid_x, a.kid, ep,
                                              st);
  }
  if (a.X2) {
    if constexpr (BN <= 128)  // one MMA covers both halves: 2*BN columns, at most 256
      return launch_kernel<BN, kMode, true>(tw, tw, tw, tx, tx2, m_tiles, m_tiles, a.G * a.Mg, a.N,
                                            k_chunks, mt_group, mt_cta, 1, m_tiles / mt_cta, a.kid,
                                            ep, st);
    else
      return MLA_ERR_UNSUPPORTED;
  }
  return launch_kernel<BN, kMode, false>(tw, tw, tw, tx, tx2, m_tiles, m_tiles, a.G * a.Mg, a.N,
                                         k_chunks, mt_group, mt_cta, 1, m_tiles / mt_cta, a.kid, ep,
                                         st);
}

template <int kMode, class Ep>
mla_status_t launch_grouped(const GroupArgs& a, const Ep& ep, cudaStream_t st) {
  if (a.N <= 0) return MLA_OK;
  if (a.K % 64 || a.Mg % 128) return MLA_ERR_UNSUPPORTED;
  if (a.N <= 32) return launch_grouped_bn<32, kMode>(a, ep, st);
  if (a.N <= 64) return launch_grouped_bn<64, kMode>(a, ep, st);
  if (a.N <= 128 || a.X2) return launch_grouped_bn<128, kMode>(a, ep, st);  // hi/lo: N <= 256
  return launch_grouped_bn<256, kMode>(a, ep, st);
}

}  // namespace

// ------------------------------------------------------------------------- entry points
mla_status_t tc_append(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                       const int32_t* seq_idx, const int32_t* pos, int n, mla_cache_t* cache,
                       void* packed, int kid, cudaStream_t st) {
  ProjArgs a{};
  a.W0 = w->W_DKV;
  a.O0 = d->d_c;
  a.W1 = w->W_KR;
  a.O1 = d->d_hr;
  a.K = d->d;
  a.X = h;
  a.ldx = d->d;
  a.N = n;
  a.kid = kid;
  EpAppend ep{(__nv_bfloat16*)cache->rows, (int64_t)(d->d_c + d->d_hr), cache->capacity,
              cache->seq_base, seq_idx, pos, (__nv_bfloat16*)packed, d->d_c, rope_freqs(d)};
  return launch_proj(a, ep, st);
}

// Append + c^Q of a decode step ("MLA前向计算流程" §三分支计算 ①②③): token n of h is sequence
// n's token at position pos[n]; one launch streams W^DKV, W^KR and W^DQ once.
mla_status_t tc_down(const mla_dims_t* d, const mla_weights_t* w, const void* h,
                     const int32_t* pos, int n, mla_cache_t* cache, void* cq_hi, void* cq_lo,
                     int kid, cudaStream_t st) {
  ProjArgs a{};
  a.W0 = w->W_DKV;
  a.O0 = d->d_c;
  a.W1 = w->W_KR;
  a.O1 = d->d_hr;
  a.W2 = w->W_DQ;
  a.O2 = d->d_cq;
  a.K = d->d;
  a.X = h;
  a.ldx = d->d;
  a.N = n;
  a.kid = kid;
  const int q_row0 = (d->d_c / 128 + ceil_div(d->d_hr, 128)) * 128;
  EpDown ep{EpAppend{(__nv_bfloat16*)cache->rows, (int64_t)(d->d_c + d->d_hr), cache->capacity,
                     cache->seq_base, nullptr, pos, nullptr, d->d_c, rope_freqs(d)},
            EpStoreBF16{(__nv_bfloat16*)cq_hi, (__nv_bfloat16*)cq_lo, d->d_cq},
            d->d_c + d->d_hr, q_row0};
  return launch_proj(a, ep, st);
}

mla_status_t tc_q_down(const mla_dims_t* d, const mla_weights_t* w, const void* h, int n,
                       void* cq_hi, void* cq_lo, int kid, cudaStream_t st) {
  ProjArgs a{};
  a.W0 = w->W_DQ;
  a.O0 = d->d_cq;
  a.K = d->d;
  a.X = h;
  a.ldx = d->d;
  a.N = n;
  a.kid = kid;
  EpStoreBF16 ep{(__nv_bfloat16*)cq_hi, (__nv_bfloat16*)cq_lo, d->d_cq};
  return launch_proj(a, ep, st);
}

mla_status_t tc_q_up(const mla_dims_t* d, const mla_weights_t* w, const void* cq_hi,
                     const void* cq_lo, const int32_t* pos, int n, void* q_c, void* q_r,
                     int64_t qc_tok, int64_t qc_head, int64_t qr_tok, int64_t qr_head,
                     bool f16_out, int kid, cudaStream_t st) {
  ProjArgs a{};
  a.W0 = w->W_UQ;
  a.O0 = d->n_h * d->d_hc;
  a.W1 = w->W_QR;
  a.O1 = d->n_h * d->d_hr;
  a.K = d->d_cq;
  a.X = cq_hi;
  a.X2 = cq_lo;  // null: c^Q as a single bf16 operand
  a.ldx = d->d_cq;
  a.N = n;
  a.kid = kid;
  if (f16_out) {
    EpQuery<__half> ep{(__half*)q_c, (__half*)q_r, qc_tok, qc_head, qr_tok, qr_head, pos,
                       d->n_h, d->d_hc, d->d_hr, rope_freqs(d)};
    return launch_proj(a, ep, st);
  }
  EpQuery<__nv_bfloat16> ep{(__nv_bfloat16*)q_c, (__nv_bfloat16*)q_r, qc_tok, qc_head, qr_tok,
                            qr_head, pos, d->n_h, d->d_hc, d->d_hr, rope_freqs(d)};
  return launch_proj(a, ep, st);
}

mla_status_t tc_expand(const void* W, int O, const void* latent, int64_t ld_latent, int K, int n,
                       void* y, bool f16_out, int kid, cudaStream_t st) {
  ProjArgs a{};
  a.W0 = W;
  a.O0 = O;
  a.K = K;
  a.X = latent;
  a.ldx = ld_latent;
  a.N = n;
  a.kid = kid;
  if (f16_out) {
    EpStoreF16 ep{(__half*)y, O};
    return launch_proj(a, ep, st);
  }
  EpStoreBF16 ep{(__nv_bfloat16*)y, nullptr, O};
  return launch_proj(a, ep, st);
}

// Output projection ("MLA前向计算流程" §三分支计算 ④): u[n, :] = W^O o[n, :] with o [n, n_h*d_hc]
// float32, applied as one GEMM of K = n_h*d_hc over o's hi/lo bf16 split (o = hi + lo to
// ~2^-16, one MMA of width 2*BN covers both); ws holds the split.
size_t tc_output_projection_ws(const mla_dims_t* d, int n) {
  return 2 * align_up((size_t)n * d->n_h * d->d_hc * 2, 256);
}

mla_status_t tc_output_projection(const mla_dims_t* d, const void* W_O, const float* o, int n,
                                  void* ws, float* u, cudaStream_t st) {
  const int K = d->n_h * d->d_hc;
  char* hi = (char*)ws;
  char* lo = hi + align_up((size_t)n * K * 2, 256);
  const int64_t n4 = (int64_t)n * K / 4;
  {
    TraceScope ts(K_OUT_SPLIT, st);
    split_hi_lo_kernel<<<(int)std::min<int64_t>((n4 + 255) / 256, 4 * 148), 256, 0, st>>>(
        (const float4*)o, (uint2*)hi, (uint2*)lo, n4);
    mla_status_t s = launch_status();
    if (s != MLA_OK) return s;
  }
  ProjArgs a{};
  a.W0 = W_O;
  a.O0 = d->d;
  a.K = K;
  a.X = hi;
  a.X2 = lo;
  a.ldx = K;
  a.N = n;
  a.kid = K_OUT_PROJ;
  EpStoreF32 ep{u, d->d};
  return launch_proj(a, ep, st);
}

// q~[b, i, :] = (W^UK_i)^T q^C[b, i, :]  ("从LLaMA到DeepSeek" §六): per head an MN-major
// [d_c x d_h^C] block of W^UK against the B query rows of that head; bf16 out.
mla_status_t tc_absorb(const mla_dims_t* d, const mla_weights_t* w, const void* q_c, int B,
                       void* qt, int kid, cudaStream_t st) {
  GroupArgs a{w->W_UK, d->n_h, d->d_c, d->d_hc, q_c, nullptr, B, kid};
  EpStoreBF16 ep{(__nv_bfloat16*)qt, nullptr, (int64_t)d->n_h * d->d_c};
  return launch_grouped<kGroupedMN>(a, ep, st);
}

}  // namespace mla
