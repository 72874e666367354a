// Weight-absorbed decode on the tensor cores for the DeepSeek-V2 widths (n_h 128, d_h^C 128,
// d_h^R 64, d_c 512, bf16): "从LLaMA到DeepSeek[01] - MLA（上）" §六 (absorption by
// associativity) and "MLA前向计算流程" §三分支计算 ④ (softmax over j = 1..t, scale
// 1/sqrt(d_h^C + d_h^R)).
//
// Three launches:
//   absorb      q~[b,i,:] = (W^UK_i)^T q^C[b,i,:]        grouped tcgen05 GEMM (gemm_tc.cu)
//   attention   split-KV latent attention, this file     (m, l, O~) partials per segment
//   unabsorb    log-sum-exp merge of the partials, then  o[b,i,:] = W^UV_i o~[b,i,:]
//               (tcgen05, this file)
//
// Attention kernel. All 128 heads form the M dimension of every MMA. The accumulator
// O~ (128 heads x 512 latent columns, fp32) would fill a whole SM's tensor memory, so two CTAs
// (a "pair", on two SMs) share each piece of work: CTA r owns latent columns
// [256 r, 256 r + 256) of O~. Both CTAs stream the full 576-wide cache tile and compute the
// same score tile S = [q~ ; q^R] [c ; k^R]^T (K = 576) themselves: handing a score tile to
// the other SM through distributed shared memory costs more time than recomputing it. Per
// 48-row cache tile, per CTA:
//   TMA     9 boxes of 64 columns x 48 rows into a 3-deep shared-memory ring
//   MMA     S = Q K^T (36 K-steps of 16) into one of two tensor-memory score buffers; later
//           O_r += P V_r (3 K-steps) with P read from tensor memory
//   softmax one thread per head: online softmax in log2 units with lazy rescaling; P in bf16
//           written over the first 24 columns of its own score buffer
// Both CTAs of a pair therefore hold bitwise identical scores and softmax statistics. With two
// score buffers the score MMA of tile t+2 is issued right behind the PV MMA of tile t, so the
// tensor pipe does not wait for the softmax to read a score tile out before the next one can
// be computed. Tensor memory: O_r (256 columns), two score buffers (2 x 48), and the query's K
// columns 0..319 (160 columns of bf16 pairs); K columns 320..575 of the query live in shared
// memory. The tensor pipe executes one thread's MMAs in issue order, so the score MMA of tile
// t+2 overwrites P(t) only after the PV MMA of tile t has read it.
//
// Work split (see pairs_for): whenever it fits, every pair works inside one sequence (sequence
// b gets pairs in proportion to its tile count, each a contiguous share of its tiles, and pair
// p writes slot p), so no pair re-loads the query halfway. Otherwise the cache tiles of all
// sequences form one list and pair p of P takes the contiguous range [p*T/P, (p+1)*T/P); every
// (sequence b, pair p) intersection is a segment writing slot b + p, unique because both ranges
// are ordered. The segments holding a sequence's first and last tile record its slot range for
// the merge.
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "proj_tc.h"
#include "tc.cuh"

namespace mla {

using namespace tc;

namespace {

constexpr int kDC = 512;          // d_c
constexpr int kRowElems = 576;    // d_c + d_h^R
constexpr int kHeads = 128;       // n_h
constexpr int kTile = 48;         // cache rows per tile
constexpr int kStages = 3;
constexpr int kBox = 64 * kTile * 2;   // one TMA box: 64 columns x 48 rows of bf16 (6 KB)
constexpr int kStageBytes = 9 * kBox;  // the whole 576-wide tile
constexpr int kQBox = 64 * kHeads * 2; // 64 query columns x 128 heads (16 KB)
constexpr int kQTmemK = 320;           // query K columns held in tensor memory
constexpr int kQBoxes = (kRowElems - kQTmemK) / 64;  // query boxes in shared memory (4)
constexpr int kOffQb = 0;              // query K columns 320..575
constexpr int kOffStage = kQBoxes * kQBox;
constexpr int kOffBar = kOffStage + kStages * kStageBytes;
constexpr int kThreads = 224;  // 7 warps: 0 TMA (score-only boxes), 1 MMA, 2..5 softmax, 6 TMA (V boxes)
constexpr int kSmemUsed = kOffBar + 256;
constexpr int kSmemBytes = 232448;  // the opt-in maximum; the base is aligned up to 1 KB
constexpr int kMaxPairs = 80;       // partial slots are sized for at most this many CTA pairs
static_assert(kBox % 1024 == 0 && kOffStage % 1024 == 0 && kOffBar % 1024 == 0, "1 KB alignment");
static_assert(kSmemUsed <= kSmemBytes, "shared memory");
static_assert(kQTmemK % 64 == 0, "the shared-memory query part starts on a box boundary");

// tensor-memory columns
constexpr uint32_t kColO = 0;    // O_r: 256 fp32 columns
constexpr uint32_t kColS = 256;  // score buffer i: 48 fp32 columns at kColS + 48 i
constexpr uint32_t kColQ = 352;  // Q K-columns 0..319: 160 columns of bf16 pairs
static_assert(kColS + 2 * kTile <= kColQ && kColQ + kQTmemK / 2 == 512, "tensor-memory map");

constexpr float kTau = 8.f;  // lazy rescale threshold (log2 units): p <= 2^8 between rescales

struct Shared {
  uint64_t full[kStages], empty_a[kStages], empty_b[kStages];
  uint64_t s_full[2], p_full, pv_done, q_full, mma_done, never;
  uint32_t tmem_slot;
  int abort;
  int b0, j0, nt, nospan;
  long long red[8];
};
static_assert(sizeof(Shared) <= 256, "barrier block");

struct SeqInfo {
  int L, n;
  int64_t base;
};

// Length, tile count and first row of sequence b, with the same clamping as the other decode
// kernels: lengths above max_len are cut to max_len; a sequence whose rows leave the cache is
// treated as empty. `flag` latches the matching status.
__device__ __forceinline__ SeqInfo seq_info(const int32_t* __restrict__ seq_len,
                                            const int64_t* __restrict__ seq_base, int b,
                                            int max_len, int64_t capacity, bool flag) {
  int L = seq_len[b];
  const int64_t base = seq_base[b];
  if (L < 0 || L > max_len) {
    if (flag) flag_status(MLA_ERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  if (L > 0 && (base < 0 || base + L > capacity)) {
    if (flag) flag_status(MLA_ERR_CAPACITY);
    L = 0;
  }
  return {L, (L + kTile - 1) / kTile, base};
}

template <int NT>
__device__ __forceinline__ long long block_sum(long long v, long long* red) {
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  long long s = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) s += red[w];
  return s;
}

template <int NT>
__device__ __forceinline__ long long block_excl_scan(long long v, long long* red,
                                                     long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
  for (int off = 1; off < 32; off <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  __syncthreads();
  if (lane == 31) red[warp] = x;
  __syncthreads();
  long long before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) before += red[w];
    tot += red[w];
  }
  *total = tot;
  return before + x - v;
}

__device__ __forceinline__ long long pair_start(int p, long long T, int P) {
  return (long long)p * T / P;
}

// Work split of the tiles over the P CTA pairs.
// Whole-sequence mode, used whenever it fits: sequence b gets k_b = min(n_b, max(1,
// floor(n_b P / T))) pairs, and pair c of them takes tiles [c n_b / k_b, (c+1) n_b / k_b) of
// that sequence alone; pair p writes slot p. No pair then has to re-load the query halfway.
// Otherwise (more non-empty sequences than pairs, or the k_b overflow P): pairs take contiguous
// ranges [p T / P, (p+1) T / P) of the concatenated tile list; each (sequence b, pair p)
// intersection is a segment writing slot b + p.
__device__ __forceinline__ int pairs_for(int n, long long T, int P) {
  if (n <= 0) return 0;
  long long k = (long long)n * P / T;
  if (k < 1) k = 1;
  return (int)(k < n ? k : n);
}

// Walks the tiles of one pair's range sequence by sequence.
struct Cursor {
  int b, j;
  SeqInfo s;
  __device__ void next(const int32_t* seq_len, const int64_t* seq_base, int max_len,
                       int64_t capacity) {
    if (++j < s.n) return;
    j = 0;
    do {
      ++b;
      s = seq_info(seq_len, seq_base, b, max_len, capacity, false);
    } while (s.n == 0);
  }
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------------------------------------------------
// The attention kernel
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_rows,
                          const __grid_constant__ CUtensorMap tm_qt,  // q~ [B*128, 512]
                          const __grid_constant__ CUtensorMap tm_qr,  // q^R [B*128, 64]
                          const __nv_bfloat16* __restrict__ qt,       // [B, 128, 512]
                          const int32_t* __restrict__ seq_len,
                          const int64_t* __restrict__ seq_base, int64_t capacity, int B,
                          int max_len, float scale_log2, float* __restrict__ part_o,
                          float* __restrict__ part_ml, int2* __restrict__ seq_slots,
                          int64_t test_stall_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(smem + kOffBar);
  volatile int* abort = &sh.abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x & 1;  // latent half owned by this CTA
  const int P = gridDim.x / 2, p = blockIdx.x / 2;
  // The merge kernel after this one may be scheduled now: it waits for this grid to complete
  // before it reads anything written here.
  griddep_launch();
  // the aligned layout must fit in the allocation (it does when the base is 1 KB aligned)
  if ((smem - smem_raw) + kSmemUsed > kSmemBytes) {
    if (threadIdx.x == 0) flag_status(MLA_ERR_UNSUPPORTED);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 2);  // one arrival per producer, plus the bytes of all 9 boxes
      mbar_init(&sh.empty_a[s], 1);
      mbar_init(&sh.empty_b[s], 1);
    }
    mbar_init(&sh.s_full[0], 1);
    mbar_init(&sh.s_full[1], 1);
    mbar_init(&sh.p_full, 4);
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.q_full, 4);
    mbar_init(&sh.mma_done, 1);
    mbar_init(&sh.never, 1);  // completed by nobody (the wait-timeout test)
    sh.abort = 0;
    sh.b0 = 0;
    sh.j0 = 0;
    sh.nt = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tm_rows);
    tma_prefetch(&tm_qt);
    tma_prefetch(&tm_qr);
  }

  // ---- plan (see pairs_for): this pair's first (sequence, tile) and tile count
  long long loc_n = 0, loc_ne = 0;
  for (int b = threadIdx.x; b < B; b += kThreads) {
    const int n = seq_info(seq_len, seq_base, b, max_len, capacity, blockIdx.x == 0).n;
    loc_n += n;
    loc_ne += n > 0;
  }
  const long long T = block_sum<kThreads>(loc_n, sh.red);
  const long long NE = block_sum<kThreads>(loc_ne, sh.red);
  long long loc_k = 0;
  if (T > 0)
    for (int b = threadIdx.x; b < B; b += kThreads)
      loc_k += pairs_for(seq_info(seq_len, seq_base, b, max_len, capacity, false).n, T, P);
  const long long K = block_sum<kThreads>(loc_k, sh.red);
  const bool nospan = T > 0 && NE <= P && K <= P;
  if (threadIdx.x == 0) sh.nospan = nospan;
  if (nospan) {
    if (p < K) {
      long long carry = 0;
      for (int b_lo = 0; b_lo < B; b_lo += kThreads) {
        const int b = b_lo + threadIdx.x;
        const int n = b < B ? seq_info(seq_len, seq_base, b, max_len, capacity, false).n : 0;
        const int k = pairs_for(n, T, P);
        long long tot;
        const long long excl = carry + block_excl_scan<kThreads>(k, sh.red, &tot);
        if (k > 0 && excl <= p && p < excl + k) {
          const int c = (int)(p - excl);
          const int j0 = (int)((long long)c * n / k), j1 = (int)((long long)(c + 1) * n / k);
          sh.b0 = b;
          sh.j0 = j0;
          sh.nt = j1 - j0;
        }
        carry += tot;
        if (carry > p) break;
      }
    }
  } else if (T > 0) {
    const long long t_begin = pair_start(p, T, P), t_end = pair_start(p + 1, T, P);
    if (threadIdx.x == 0) sh.nt = (int)(t_end - t_begin);
    if (t_begin < t_end) {
      long long carry = 0;
      for (int b_lo = 0; b_lo < B; b_lo += kThreads) {
        const int b = b_lo + threadIdx.x;
        const int n = b < B ? seq_info(seq_len, seq_base, b, max_len, capacity, false).n : 0;
        long long tot;
        const long long excl = carry + block_excl_scan<kThreads>(n, sh.red, &tot);
        if (n > 0 && excl <= t_begin && t_begin < excl + n) {
          sh.b0 = b;
          sh.j0 = (int)(t_begin - excl);
        }
        carry += tot;
        if (carry > t_begin) break;
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;
  const int nt = sh.nt;
  uint8_t* const qb = smem + kOffQb;

  if (nt > 0 && (warp == 0 || warp == 6) && lane == 0) {
    // ------------------------------------------------------------- TMA producers
    // Warp 0 loads the boxes only the score MMA reads (the other CTA's latent half and the RoPE
    // columns); they are released as soon as the score MMA of their tile completes. Warp 6 loads
    // this CTA's V half, released after the PV MMA. Both walk the same tile sequence.
    const bool v_boxes = warp == 6;
    uint64_t* empty = v_boxes ? sh.empty_b : sh.empty_a;
    Cursor cur{sh.b0, sh.j0, seq_info(seq_len, seq_base, sh.b0, max_len, capacity, false)};
    int issued = 0;
    for (int t = 0; t < nt; ++t) {
      const int s = t % kStages, r = t / kStages;
      if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, abort)) break;
      uint8_t* stage = smem + kOffStage + s * kStageBytes;
      mbar_arrive_expect_tx(&sh.full[s], (v_boxes ? 4 : 5) * kBox);
      const int y = (int)(cur.s.base + (int64_t)cur.j * kTile);
#pragma unroll 1
      for (int k = 0; k < 9; ++k) {
        const bool is_v = (k >> 2) == rank && k < 8;
        if (is_v == v_boxes) tma_load_2d(stage + k * kBox, &tm_rows, &sh.full[s], k * 64, y);
      }
      ++issued;
      if (t + 1 < nt) cur.next(seq_len, seq_base, max_len, capacity);
    }
    // every issued copy lands before the CTA may exit (even after an abort)
    for (int t = (issued > kStages ? issued - kStages : 0); t < issued; ++t)
      mbar_wait_drain(&sh.full[t % kStages], (t / kStages) & 1);
  } else if (nt > 0 && warp == 1) {
    // ------------------------------------------------------------- MMA issuer (one elected
    // lane of a converged warp; the descriptors are precomputed and the K loops unrolled)
    constexpr uint32_t idesc_s = idesc_f16(128, kTile, 1, 0, 0);
    constexpr uint32_t idesc_o = idesc_f16(128, 256, 1, 0, 1);
    // cur: the tile whose PV comes next; ncur: the tile whose score MMA comes next (ns)
    Cursor cur{sh.b0, sh.j0, seq_info(seq_len, seq_base, sh.b0, max_len, capacity, false)};
    Cursor ncur = cur;
    int ns = 0, nseg = 0;  // next score tile, and the segment it belongs to
    const uint64_t desc_qb = smem_desc(smem_u32(qb), 16, 1024);
    const uint64_t desc_st = smem_desc(smem_u32(smem + kOffStage), 16, 1024);
    const uint64_t desc_v = smem_desc(smem_u32(smem + kOffStage + 4 * rank * kBox), kBox, 1024);
    // Score MMA of tile ns into buffer ns & 1. A tile that starts a segment first waits for
    // that segment's query (the softmax loads it once the previous segment's scores are read).
    auto issue_next_s = [&]() -> bool {
      if (ns == 0 || ncur.j == 0) {
        if (ns > 0) ++nseg;
        if (!warp_wait(&sh.q_full, nseg & 1, abort)) return false;
      }
      const int s = ns % kStages;
      if (!warp_wait(&sh.full[s], (ns / kStages) & 1, abort)) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t d_s = tmem + kColS + (uint32_t)((ns & 1) * kTile);
        const uint64_t bst = desc_st + (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < 36; ++ks) {
          const uint64_t bdesc = bst + (uint64_t)(((ks >> 2) * kBox + (ks & 3) * 32) >> 4);
          if (ks < kQTmemK / 16)
            mma_ts(d_s, tmem + kColQ + ks * 8, bdesc, idesc_s, ks > 0 ? 1u : 0u);
          else
            mma_ss(d_s,
                   desc_qb + (uint64_t)((((ks - kQTmemK / 16) >> 2) * kQBox + (ks & 3) * 32) >> 4),
                   bdesc, idesc_s, 1u);
        }
        mma_commit(&sh.s_full[ns & 1]);
        mma_commit(&sh.empty_a[s]);
      }
      __syncwarp();
      if (++ns < nt) ncur.next(seq_len, seq_base, max_len, capacity);
      return true;
    };
    bool ok = true;
    if (test_stall_ns > 0) {
      // Test of the bounded waits: wait for a barrier phase that nothing completes, give up
      // after test_stall_ns, latch MLA_ERR_TIMEOUT and make the CTA's other roles give up too
      // (they drain their own copies and exit).
      const uint64_t t0 = global_ns();
      for (;;) {  // lane 0 polls and decides for the warp
        int state = 0;  // 1: the phase completed, 2: gave up
        if (lane == 0)
          state = mbar_try_wait(&sh.never, 0) ? 1
                                              : (global_ns() - t0 > (uint64_t)test_stall_ns ? 2 : 0);
        state = __shfl_sync(0xffffffffu, state, 0);
        if (state == 1) break;
        if (state == 2) {
          if (lane == 0) {
            flag_status(MLA_ERR_TIMEOUT);
            *abort = 1;
          }
          ok = false;
          break;
        }
      }
    }
    // two score tiles ahead of the first PV
    ok = ok && issue_next_s();
    if (ok && nt > 1) ok = issue_next_s();
    for (int t = 0; ok && t < nt; ++t) {
      const bool seg_first = t == 0 || cur.j == 0;  // O starts from zero
      if (!warp_wait(&sh.p_full, t & 1, abort)) break;
      tc_fence_after();
      if (elect_one()) {
        const uint32_t a_p = tmem + kColS + (uint32_t)((t & 1) * kTile);
        const uint64_t bv = desc_v + (uint64_t)(((t % kStages) * kStageBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks)
          mma_ts(tmem + kColO, a_p + ks * 8, bv + (uint64_t)((ks * 2048) >> 4), idesc_o,
                 (!seg_first || ks > 0) ? 1u : 0u);
        mma_commit(&sh.empty_b[t % kStages]);
        mma_commit(&sh.pv_done);
      }
      __syncwarp();
      // the score MMA of tile t+2 reuses buffer t & 1: issued after PV(t), it runs after it
      if (ns < nt && !issue_next_s()) break;
      if (t + 1 < nt) cur.next(seq_len, seq_base, max_len, capacity);
    }
    // every MMA issued by this CTA completes before its tensor memory is freed
    if (elect_one()) mma_commit(&sh.mma_done);
    __syncwarp();
    mbar_wait_drain(&sh.mma_done, 0);
  } else if (nt > 0 && warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------- softmax warps
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int h = q * 32 + lane;            // head = TMEM lane
    const int ts = threadIdx.x - 64;        // 0..127 among the softmax threads
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);

    // Query of sequence b: K columns 0..319 into tensor memory (two bf16 per column, one
    // thread per head), K columns 320..575 into shared memory by TMA.
    auto load_q = [&](int b) {
      if (ts == 0) {
        mbar_expect_tx(&sh.q_full, kQBoxes * kQBox);
#pragma unroll
        for (int x = kQTmemK; x < kDC; x += 64)
          tma_load_2d(qb + ((x - kQTmemK) / 64) * kQBox, &tm_qt, &sh.q_full, x, b * kHeads);
        tma_load_2d(qb + (kQBoxes - 1) * kQBox, &tm_qr, &sh.q_full, 0, b * kHeads);
      }
      // all 40 loads in flight at once: the query rows come from L2 and the load latency,
      // not the bytes, sets the cost of a segment switch
      const uint4* src = reinterpret_cast<const uint4*>(qt + ((int64_t)b * kHeads + h) * kDC);
      constexpr int kVecs = kQTmemK / 8;
      uint4 v[kVecs];
#pragma unroll
      for (int k = 0; k < kVecs; ++k) v[k] = __ldg(src + k);
#pragma unroll
      for (int c = 0; c < kVecs / 8; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          r[4 * k] = v[c * 8 + k].x;
          r[4 * k + 1] = v[c * 8 + k].y;
          r[4 * k + 2] = v[c * 8 + k].z;
          r[4 * k + 3] = v[c * 8 + k].w;
        }
        tmem_st32u(lane_base + kColQ + c * 32, r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.q_full);
    };

    Cursor cur{sh.b0, sh.j0, seq_info(seq_len, seq_base, sh.b0, max_len, capacity, false)};
    // q~ comes from the kernel before this one (launched with programmatic serialization, this
    // grid may start early): wait for it. The cache rows and the lengths were complete before
    // that kernel started, so the TMA producers need no wait.
    griddep_wait();
    load_q(cur.b);
    float m_used = -INFINITY, l_sum = 0.f;
    int seg_j0 = cur.j;  // first tile of the current segment
    for (int t = 0; t < nt; ++t) {
      const int j = cur.j;
      const int valid = min(kTile, cur.s.L - j * kTile);
      float s[kTile];
      const uint32_t col_s = kColS + (uint32_t)((t & 1) * kTile);  // this tile's score buffer
      if (!warp_wait(&sh.s_full[t & 1], (t >> 1) & 1, abort)) break;
      tc_fence_after();
      tmem_ld32(lane_base + col_s, *reinterpret_cast<float(*)[32]>(&s[0]));
      tmem_ld16(lane_base + col_s + 32, &s[32]);
      tmem_wait_ld();

      // online softmax in log2 units with lazy rescaling
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < kTile; ++i)
        if (i < valid) mx[i & 3] = fmaxf(mx[i & 3], s[i]);
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
      const bool first = t == 0 || j == 0;  // first tile of a segment
      const float m_new = first ? mt : (mt > m_used + kTau ? mt : m_used);
      const float alpha = first ? 0.f : ex2(m_used - m_new);
      m_used = m_new;

      // P in bf16 (and its row sum) while the previous tile's PV may still run
      uint32_t w[kTile / 2];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < kTile / 2; ++k) {
        const int i = 2 * k;
        const float p0 = i < valid ? ex2(fmaf(s[i], scale_log2, -m_used)) : 0.f;
        const float p1 = i + 1 < valid ? ex2(fmaf(s[i + 1], scale_log2, -m_used)) : 0.f;
        w[k] = pack_bf16(p0, p1);
        const __nv_bfloat162 pb = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
        ls[k & 3] += __low2float(pb) + __high2float(pb);
      }
      l_sum = l_sum * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));

      // P over the first 24 columns of this tile's own score buffer (already read out), the
      // A operand of the PV MMA; the previous tile's PV reads the other buffer meanwhile
      tmem_st16u(lane_base + col_s, *reinterpret_cast<const uint32_t(*)[16]>(&w[0]));
      tmem_st8u(lane_base + col_s + 16, *reinterpret_cast<const uint32_t(*)[8]>(&w[16]));
      // O is free once the previous tile's PV has completed
      if (t > 0 && !warp_wait(&sh.pv_done, (t - 1) & 1, abort)) break;
      if (__any_sync(0xffffffffu, alpha != 1.f && !first)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float o[32];
          tmem_ld32(lane_base + kColO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(lane_base + kColO + c * 32, o);
        }
        tmem_wait_st();
      }
      tmem_wait_st();
      if (valid < kTile) {
        // rows past the sequence end may hold anything (even NaN): zero them in the V operand
        uint8_t* v0 = smem + kOffStage + (t % kStages) * kStageBytes + 4 * rank * kBox;
        const int n16 = (kTile - valid) * 8;  // 16-byte chunks per box
        for (int e = ts; e < 4 * n16; e += 128) {
          const int box = e / n16, r = e % n16;
          *reinterpret_cast<uint4*>(v0 + box * kBox + valid * 128 + r * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full);

      if (j + 1 == cur.s.n || t + 1 == nt) {
        // end of a segment (end of the sequence or of this pair's range): the next
        // sequence's query first, then O_r and (m, l) to the segment's partial slot
        const int b_done = cur.b, n_done = cur.s.n;
        if (t + 1 < nt) {
          cur.next(seq_len, seq_base, max_len, capacity);
          load_q(cur.b);
        }
        if (!warp_wait(&sh.pv_done, t & 1, abort)) break;
        tc_fence_after();
        const int64_t slot = sh.nospan ? (int64_t)p : (int64_t)b_done + p;
        float4* dst = reinterpret_cast<float4*>(part_o + (slot * kHeads + h) * kDC + rank * 256);
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float o[32];
          tmem_ld32(lane_base + kColO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[c * 8 + k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
        if (rank == 0) {
          part_ml[slot * 256 + h] = m_used;
          part_ml[slot * 256 + 128 + h] = l_sum;
          // the segments holding a sequence's first and last tile record its slot range
          if (ts == 0) {
            if (seg_j0 == 0) seq_slots[b_done].x = (int)slot;
            if (j + 1 == n_done) seq_slots[b_done].y = (int)slot;
          }
        }
        seg_j0 = 0;
        tc_fence_before();
        m_used = -INFINITY;
        l_sum = 0.f;
      } else if (t + 1 < nt) {
        cur.next(seq_len, seq_base, max_len, capacity);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------------------------------
// Merge + un-absorb: o[b,i,:] = W^UV_i o~[b,i,:], with o~ the log-sum-exp merge of the
// sequence's partial results, o~ = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s (m in log2
// units). One CTA per (head i, 64 sequences), 16 warps:
//   - the head's [128 x 512] block of W^UV streams through a 4-deep ring of 64-column chunks
//     (TMA): thread 0 loads the first four while the partials are merged, warp 8 the rest as
//     the MMAs free the ring;
//   - the warps merge the partials in teams: with n sequences in the CTA, G = 16 / n warps (a
//     power of two, at least 1) share a sequence, each taking every G-th slot of its range and
//     keeping an online (max, sum, O) in registers, four slots' loads in flight at a time; a
//     team combines its members through shared memory. Lane l owns latent columns 4l + 128j
//     (j < 4), so each partial row is one contiguous 512-byte warp load;
//   - o~ is written as a hi/lo pair of bf16 (o~ = hi + lo to about 2^-16) straight into the
//     K-major, 128-byte-swizzled B operand: rows 0..63 hold hi, rows 64..127 lo;
//   - one thread issues D[128 features x 128] = W^UV_i [hi ; lo]^T (32 K-steps of 16);
//   - eight warps add the two halves of each column and store o (one feature per lane).
// The slot range of sequence b, [seq_slots[b].x, seq_slots[b].y], was recorded by the attention
// kernel; every slot in it holds a segment of b.
// ------------------------------------------------------------------------------------------
constexpr int kUnBN = 64;                              // sequences per CTA
constexpr int kUnWarps = 16;
constexpr int kUnThreads = 32 * kUnWarps;
constexpr int kUnABox = 128 * 128;                     // 128 rows x 64 bf16: one K chunk of A
constexpr int kUnAStages = 4;
constexpr int kUnBChunk = 2 * kUnBN * 128;             // one 64-wide K chunk of [hi ; lo]
constexpr int kUnOffB = kUnAStages * kUnABox;          // A ring: 64 KB
constexpr int kUnOffTeam = kUnOffB + 8 * kUnBChunk;    // B: 128 KB
constexpr int kUnTeamFloats = 4 * 128 + 4;             // per warp: O (512), max, sum (16 B rows)
constexpr int kUnOffBar = kUnOffTeam + kUnWarps * kUnTeamFloats * 4;
constexpr int kUnSmem = kUnOffBar + 128 + 1024;
constexpr int kMergeVec = kDC / 128;                   // float4 groups per lane
static_assert(kUnOffB % 1024 == 0 && kUnOffTeam % 16 == 0 && kUnTeamFloats % 4 == 0, "alignment");
static_assert(kUnSmem <= 232448, "shared memory");

__global__ void __launch_bounds__(kUnThreads, 1)
    decode_unabsorb_kernel(const __grid_constant__ CUtensorMap tm_wuv,  // W^UV [n_h*128, 512]
                           const float* __restrict__ part_o, const float* __restrict__ part_ml,
                           const int2* __restrict__ seq_slots, int n_slots,
                           const int32_t* __restrict__ seq_len,
                           const int64_t* __restrict__ seq_base, int64_t capacity, int B,
                           int max_len, float* __restrict__ o) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + kUnOffBar);
  uint64_t* a_empty = a_full + kUnAStages;
  uint64_t* done = a_empty + kUnAStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* team = reinterpret_cast<float*>(smem + kUnOffTeam);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x;  // head
  const int b0 = blockIdx.y * kUnBN;
  const int nb = min(kUnBN, B - b0);

  if (threadIdx.x == 0) {
    for (int k = 0; k < kUnAStages; ++k) {
      mbar_init(&a_full[k], 1);
      mbar_init(&a_empty[k], 1);
    }
    mbar_init(done, 1);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    tma_prefetch(&tm_wuv);
    for (int k = 0; k < kUnAStages; ++k) {
      mbar_arrive_expect_tx(&a_full[k], kUnABox);
      tma_load_2d(smem + k * kUnABox, &tm_wuv, &a_full[k], k * 64, i * 128);
    }
  }
  // the partial results come from the attention kernel (this grid may start before it ends)
  griddep_wait();

  // ---- merge in teams of G warps per sequence
  int G = 1;
  while (G * 2 * nb <= kUnWarps) G *= 2;
  const int teams = kUnWarps / G, g = warp % G;
  const int rounds = (nb + teams - 1) / teams;
  auto bits = [](__nv_bfloat162 x) { return *reinterpret_cast<const uint32_t*>(&x); };
  for (int rd = 0; rd < rounds; ++rd) {
    const int r = rd * teams + warp / G;  // sequence within the CTA
    float4 acc[kMergeVec];
#pragma unroll
    for (int j = 0; j < kMergeVec; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    float M = -INFINITY, L = 0.f;
    if (r < nb && seq_info(seq_len, seq_base, b0 + r, max_len, capacity, false).n > 0) {
      const int2 rg = seq_slots[b0 + r];
      if (rg.x < 0 || rg.y < rg.x || rg.y >= n_slots) {
        if (lane == 0) flag_status(MLA_ERR_UNSUPPORTED);  // not written by the attention kernel
      } else {
        // slots rg.x + g, rg.x + g + G, ...: four at a time, all their loads in flight
        for (int s0 = rg.x + g; s0 <= rg.y; s0 += 4 * G) {
          float mv[4], lv[4];
          float4 v[4][kMergeVec];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int sl = s0 + u * G;
            mv[u] = -INFINITY;
            lv[u] = 0.f;
#pragma unroll
            for (int j = 0; j < kMergeVec; ++j) v[u][j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (sl <= rg.y) {
              mv[u] = __ldg(part_ml + (int64_t)sl * 256 + i);
              lv[u] = __ldg(part_ml + (int64_t)sl * 256 + 128 + i);
              const float4* src =
                  reinterpret_cast<const float4*>(part_o + ((int64_t)sl * kHeads + i) * kDC) + lane;
#pragma unroll
              for (int j = 0; j < kMergeVec; ++j) v[u][j] = __ldg(src + 32 * j);
            }
          }
          const float mx = fmaxf(fmaxf(mv[0], mv[1]), fmaxf(mv[2], mv[3]));
          const float Mn = fmaxf(M, mx);
          const float sc = M == -INFINITY ? 0.f : exp2f(M - Mn);
          L *= sc;
#pragma unroll
          for (int j = 0; j < kMergeVec; ++j) {
            acc[j].x *= sc;
            acc[j].y *= sc;
            acc[j].z *= sc;
            acc[j].w *= sc;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float w = mv[u] == -INFINITY ? 0.f : exp2f(mv[u] - Mn);
            L = fmaf(w, lv[u], L);
#pragma unroll
            for (int j = 0; j < kMergeVec; ++j) {
              acc[j].x = fmaf(w, v[u][j].x, acc[j].x);
              acc[j].y = fmaf(w, v[u][j].y, acc[j].y);
              acc[j].z = fmaf(w, v[u][j].z, acc[j].z);
              acc[j].w = fmaf(w, v[u][j].w, acc[j].w);
            }
          }
          M = Mn;
        }
      }
    }
    if (G > 1) {
      // team members hand (M, L, O) to the team's first warp through shared memory
      float* mine = team + warp * kUnTeamFloats;
#pragma unroll
      for (int j = 0; j < kMergeVec; ++j)
        *reinterpret_cast<float4*>(mine + 4 * lane + 128 * j) = acc[j];
      if (lane == 0) {
        mine[512] = M;
        mine[513] = L;
      }
      __syncthreads();
      if (g == 0) {
        float Mt = -INFINITY;
        for (int k = 0; k < G; ++k) Mt = fmaxf(Mt, team[(warp + k) * kUnTeamFloats + 512]);
#pragma unroll
        for (int j = 0; j < kMergeVec; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        L = 0.f;
        for (int k = 0; k < G; ++k) {
          const float* t = team + (warp + k) * kUnTeamFloats;
          const float w = t[512] == -INFINITY ? 0.f : exp2f(t[512] - Mt);
          L = fmaf(w, t[513], L);
#pragma unroll
          for (int j = 0; j < kMergeVec; ++j) {
            const float4 x = *reinterpret_cast<const float4*>(t + 4 * lane + 128 * j);
            acc[j].x = fmaf(w, x.x, acc[j].x);
            acc[j].y = fmaf(w, x.y, acc[j].y);
            acc[j].z = fmaf(w, x.z, acc[j].z);
            acc[j].w = fmaf(w, x.w, acc[j].w);
          }
        }
      }
    }
    if (g == 0 && r < kUnBN) {
      // o~ -> hi/lo bf16 rows r and 64 + r of the B operand. Columns 4l + 128j sit in K chunk
      // 2j + l/16, 16-byte unit (l % 16) / 2 (swizzled by the row), half l % 2.
      const float inv_l = L > 0.f ? 1.f / L : 0.f;
      const uint32_t unit = (uint32_t)((lane & 15) >> 1);
      const uint32_t sw = ((unit ^ (uint32_t)(r & 7)) << 4) + (lane & 1) * 8;  // (64 + r) & 7 == r & 7
#pragma unroll
      for (int j = 0; j < kMergeVec; ++j) {
        const float v0 = acc[j].x * inv_l, v1 = acc[j].y * inv_l;
        const float v2 = acc[j].z * inv_l, v3 = acc[j].w * inv_l;
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v0, v1);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(v2, v3);
        const __nv_bfloat162 l01 =
            __floats2bfloat162_rn(v0 - __low2float(h01), v1 - __high2float(h01));
        const __nv_bfloat162 l23 =
            __floats2bfloat162_rn(v2 - __low2float(h23), v3 - __high2float(h23));
        uint8_t* chunk = smem + kUnOffB + (2 * j + (lane >> 4)) * kUnBChunk;
        *reinterpret_cast<uint2*>(chunk + r * 128 + sw) = make_uint2(bits(h01), bits(h23));
        *reinterpret_cast<uint2*>(chunk + (kUnBN + r) * 128 + sw) =
            make_uint2(bits(l01), bits(l23));
      }
    }
    if (G > 1) __syncthreads();  // the team buffer is reused by the next round
  }
  fence_proxy_async_smem();
  __syncthreads();

  // ---- D[f, n] = sum_k W^UV_i[f, k] B[n, k]: 8 chunks x 4 K-steps; chunks 4..7 of A are
  // loaded into the ring as the first four are consumed
  if (warp == 0) {
    bool ok = true;
    for (int kc = 0; kc < 8 && ok; ++kc) {
      ok = warp_wait(&a_full[kc % kUnAStages], (kc / kUnAStages) & 1, abort);
      if (!ok) break;
      tc_fence_after();
      if (elect_one()) {
        constexpr uint32_t idesc = idesc_f16(128, 2 * kUnBN, 1, 0, 0);
        const uint64_t ad = smem_desc(smem_u32(smem + (kc % kUnAStages) * kUnABox), 16, 1024);
        const uint64_t bd = smem_desc(smem_u32(smem + kUnOffB + kc * kUnBChunk), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem, ad + (uint64_t)((kk * 32) >> 4), bd + (uint64_t)((kk * 32) >> 4), idesc,
                 (kc | kk) != 0 ? 1u : 0u);
        mma_commit(&a_empty[kc % kUnAStages]);
      }
      __syncwarp();
    }
    if (elect_one()) mma_commit(done);
    __syncwarp();
  } else if (warp == 8 && lane == 0) {  // not an epilogue warp
    int issued = kUnAStages;
    for (int kc = kUnAStages; kc < 8; ++kc) {
      if (!mbar_wait(&a_empty[kc % kUnAStages], 0, abort)) break;
      mbar_arrive_expect_tx(&a_full[kc % kUnAStages], kUnABox);
      tma_load_2d(smem + (kc % kUnAStages) * kUnABox, &tm_wuv, &a_full[kc % kUnAStages], kc * 64,
                  i * 128);
      ++issued;
    }
    // every issued copy lands before the CTA may exit (even after an abort)
    for (int kc = issued - kUnAStages; kc < issued; ++kc)
      mbar_wait_drain(&a_full[kc % kUnAStages], (kc / kUnAStages) & 1);
  }
  // ---- epilogue: lane = output feature; warp w reads columns [32 (w/4), +32) of hi and lo
  if (warp < 8 && warp_wait(done, 0, abort)) {
    tc_fence_after();
    const int c0 = (warp >> 2) * 32;
    float hi[32], lo[32];
    tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + c0, hi);
    tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + kUnBN + c0, lo);
    tmem_wait_ld();
    const int f = (warp & 3) * 32 + lane;
#pragma unroll
    for (int r = 0; r < 32; ++r)
      if (c0 + r < nb) o[((int64_t)(b0 + c0 + r) * kHeads + i) * 128 + f] = hi[r] + lo[r];
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 0) {
    mbar_wait_drain(done, 0);  // the MMAs have completed before tensor memory is freed
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
struct Layout {
  size_t off_qt, off_part, off_ml, off_rng, total;
};

Layout layout(int B) {
  Layout L;
  const size_t slots = (size_t)B + kMaxPairs;
  L.off_qt = 0;
  L.off_part = align_up(L.off_qt + (size_t)B * kHeads * kDC * 2, 256);
  L.off_ml = align_up(L.off_part + slots * kDC * kHeads * 4, 256);
  L.off_rng = align_up(L.off_ml + slots * 256 * 4, 256);
  L.total = align_up(L.off_rng + (size_t)B * sizeof(int2), 256);
  return L;
}

constexpr int kMaxDevices = 64;

// One-shot wait-timeout test (mla_debug_arm_wait_timeout): consumed by the next launch.
std::atomic<int64_t> g_test_stall_ns{0};
std::mutex g_mu;
int g_pairs[kMaxDevices] = {};

// Number of CTA pairs resident at once on the current device (one CTA per SM), capped at
// kMaxPairs. Set up once per device.
mla_status_t attn_pairs(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_pairs[dev]) {
    if (cudaFuncSetAttribute(decode_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return MLA_ERR_CUDA;
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_attn_tc_kernel, kThreads,
                                                      kSmemBytes) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        per_sm < 1)
      return MLA_ERR_CUDA;
    int n = per_sm * sms / 2;
    if (n < 1) return MLA_ERR_UNSUPPORTED;
    if (n > kMaxPairs) n = kMaxPairs;
    // MLA_DECODE_PAIRS (read once per device) lowers the pair count, for tests and tuning
    const char* e = getenv("MLA_DECODE_PAIRS");
    if (e && atoi(e) >= 1 && atoi(e) < n) n = atoi(e);
    g_pairs[dev] = n;
  }
  *out = g_pairs[dev];
  return MLA_OK;
}

// Opt-in shared memory of the merge + un-absorb kernel, set once per device.
mla_status_t unabsorb_setup() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  static bool done[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(g_mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(decode_unabsorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kUnSmem) != cudaSuccess)
      return MLA_ERR_CUDA;
    done[dev] = true;
  }
  return MLA_OK;
}

}  // namespace

size_t tc_decode_ws(const mla_dims_t*, int B) { return layout(B).total; }
void arm_decode_wait_timeout(int64_t limit_ns) { g_test_stall_ns.store(limit_ns); }
size_t tc_decode_qt_offset(int B) { return layout(B).off_qt; }

mla_status_t tc_decode(const mla_dims_t* d, const mla_weights_t* w, const void* q_c,
                       const void* q_r, const mla_cache_t* cache, const int32_t* seq_len, int B,
                       int max_len, void* ws, float* o, cudaStream_t st) {
  // 1. q~ = (W^UK_i)^T q^C_i into the workspace, then the latent decode
  void* qt = (char*)ws + layout(B).off_qt;
  const mla_status_t s = tc_absorb(d, w, q_c, B, qt, K_ABSORB, st);
  if (s != MLA_OK) return s;
  return tc_decode_latent(d, w, qt, q_r, cache, seq_len, B, max_len, ws, o, true, st);
}

mla_status_t tc_decode_latent(const mla_dims_t* d, const mla_weights_t* w, const void* q_t,
                              const void* q_r, const mla_cache_t* cache, const int32_t* seq_len,
                              int B, int max_len, void* ws, float* o, bool after_q_kernel,
                              cudaStream_t st) {
  const Layout L = layout(B);
  char* wsb = (char*)ws;
  const __nv_bfloat16* qt = (const __nv_bfloat16*)q_t;
  float* part = (float*)(wsb + L.off_part);
  float* ml = (float*)(wsb + L.off_ml);
  int2* rng = (int2*)(wsb + L.off_rng);
  int pairs = 0;
  mla_status_t s = attn_pairs(&pairs);
  if (s != MLA_OK) return s;

  // 2. attention over the latent cache
  if (max_len > 0 && cache->capacity > 0) {
    CUtensorMap tm_rows, tm_qt, tm_qr;
    {
      const uint64_t dims[2] = {(uint64_t)kRowElems, (uint64_t)cache->capacity};
      const uint64_t strides[1] = {(uint64_t)kRowElems * 2};
      const uint32_t box[2] = {64, (uint32_t)kTile};
      if (!make_tmap(&tm_rows, cache->rows, 2, dims, strides, box,
                     CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return MLA_ERR_CUDA;
    }
    {
      const uint64_t dims[2] = {(uint64_t)kDC, (uint64_t)B * kHeads};
      const uint64_t strides[1] = {(uint64_t)kDC * 2};
      const uint32_t box[2] = {64, (uint32_t)kHeads};
      if (!make_tmap(&tm_qt, q_t, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return MLA_ERR_CUDA;
    }
    {
      const uint64_t dims[2] = {64, (uint64_t)B * kHeads};
      const uint64_t strides[1] = {64 * 2};
      const uint32_t box[2] = {64, (uint32_t)kHeads};
      if (!make_tmap(&tm_qr, q_r, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
        return MLA_ERR_CUDA;
    }
    const float scale_log2 = softmax_scale(d) * 1.4426950408889634f;
    // With the query kernel of the same call right before it, the attention may start early
    // (programmatic dependent launch): its set-up, work split and first cache loads overlap the
    // end of that kernel. As the first kernel of a call it starts normally, since then the
    // kernel before it may have written the cache or the lengths.
    TraceScope ts(K_DECODE_ATTN, st);
    if (launch_maybe_pdl(decode_attn_tc_kernel, dim3(2 * pairs), dim3(kThreads), kSmemBytes, st,
                         after_q_kernel, tm_rows, tm_qt, tm_qr, qt, seq_len, cache->seq_base,
                         cache->capacity, B, max_len, scale_log2, part, ml, rng,
                         (int64_t)g_test_stall_ns.exchange(0)) != cudaSuccess)
      return MLA_ERR_CUDA;
  }

  // 3. merge the partials of each sequence and apply W^UV_i (o = 0 for empty sequences)
  CUtensorMap tm_wuv;
  {
    const uint64_t dims[2] = {(uint64_t)kDC, (uint64_t)kHeads * 128};
    const uint64_t strides[1] = {(uint64_t)kDC * 2};
    const uint32_t box[2] = {64, 128};
    if (!make_tmap(&tm_wuv, w->W_UV, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
      return MLA_ERR_CUDA;
  }
  s = unabsorb_setup();
  if (s != MLA_OK) return s;
  // always after a kernel of the same call; it reads only weights before griddep_wait
  TraceScope ts(K_UNABSORB, st);
  if (launch_maybe_pdl(decode_unabsorb_kernel, dim3(kHeads, ceil_div(B, kUnBN)), dim3(kUnThreads),
                       kUnSmem, st, true, tm_wuv, (const float*)part, (const float*)ml,
                       (const int2*)rng, B + kMaxPairs, seq_len, cache->seq_base,
                       max_len > 0 ? cache->capacity : (int64_t)0, B, max_len, o) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace mla
