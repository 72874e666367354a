// Top-k sparse selection over the latent sequence before the decode ("MLA前向计算流程",
// version table, V3.2 + DSA row: MLA itself is unchanged; an indexer picks top-k positions
// of the latent sequence and the core attention runs MLA over the picked rows only).
//
// The indexer is not defined by the pages, so its scores are an input: one fp32 score per
// cached position. Two kernels:
//   topk_select_kernel  one cluster of 1-8 CTAs per sequence: an exact radix select of the k-th
//                       largest score (four 8-bit passes over order-preserving keys; histograms
//                       per warp, totalled per CTA and over the cluster through distributed
//                       shared memory), then an order-preserving compaction that writes the
//                       picked positions in increasing order. Equal scores rank the lower
//                       position first; -0.0 equals +0.0.
//   gather_rows_kernel  one warp per picked row: copies the row out of the cache into a
//                       packed per-sequence block (sequence b at rows b*k ...), 16 bytes per
//                       lane access, so that the unchanged decode kernels read it as a dense
//                       cache.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace mla {

using namespace tc;

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kKeysPerThread = 32;  // at most this many consecutive positions per thread
constexpr int kSelMaxCluster = 8;  // CTAs per sequence at most
constexpr int kSelSlice = 16384;   // positions per CTA that set the cluster size

// Order-preserving map of an fp32 bit pattern to uint32: a larger score gives a larger key,
// and both zeros give the same key.
__device__ __forceinline__ uint32_t score_key(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) == 0) return 0x80000000u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// A load from another CTA's shared memory. Callers issue a batch of these before using any
// result, so that their latencies overlap.
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Block-wide exclusive scan of one 32-bit value per thread (kSelThreads threads); also
// returns the block total. `tmp` holds kSelWarps + 1 words.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* tmp,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kSelWarps ? tmp[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < kSelWarps) tmp[lane] = wi - w;  // exclusive prefix of each warp
    if (lane == kSelWarps - 1) tmp[kSelWarps] = wi;
  }
  __syncthreads();
  const uint32_t r = tmp[warp] + incl - v;
  *total = tmp[kSelWarps];
  __syncthreads();  // tmp is reused by the next call
  return r;
}

// One cluster of C CTAs per sequence (blockIdx.y), C = ceil(max_len / 16384) up to 8 (one CTA
// for short sequences: then no cluster exchange at all); CTA c of the cluster owns the
// contiguous slice [c*S, min(L, (c+1)*S)) of positions, S = ceil(L / C). Thread t of
// a CTA holds R <= 32 consecutive positions of each 512 R-position round of its slice, in
// registers (kept across the passes when the slice is one round, re-read from L2 otherwise).
//  - radix select, four 8-bit passes, most significant first: every CTA counts the keys that
//    match the prefix found so far into warp-private shared-memory histograms (two buffers,
//    so that one is cleared while the other is counted), totals them per CTA, and after a
//    cluster barrier every CTA sums the cluster's totals through distributed shared memory and
//    finds the same bin: the one holding the `need`-th largest remaining key;
//  - the result: T, the key of the k-th largest score, and `need`, how many keys equal to T
//    are picked (the lowest positions among them);
//  - each CTA counts its keys above T and equal to T; a second cluster exchange gives every
//    CTA the counts of the slices before its own, and an order-preserving block scan writes
//    the picked positions in increasing order.
__global__ void __launch_bounds__(kSelThreads, 1)
topk_select_kernel(const float* __restrict__ scores, int64_t stride,
                   const int32_t* __restrict__ seq_len, int max_len, int k,
                   int32_t* __restrict__ sel_pos, int32_t* __restrict__ sel_count,
                   int64_t* __restrict__ packed_base) {
  __shared__ uint32_t hist[2][kSelWarps][256];  // per warp, double-buffered over the passes
  __shared__ uint32_t hist_cta[2][256];  // this CTA's totals, double-buffered over the passes
  __shared__ uint32_t cnt_cta[2];        // this CTA's keys above T and equal to T
  __shared__ uint32_t scan_tmp[kSelWarps + 1];
  __shared__ uint32_t s_prefix, s_need, s_gt0, s_eq0;
  const int b = blockIdx.y;
  const int c = (int)cluster_ctarank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = seq_len[b];
  if (L < 0 || L > max_len) {
    if (c == 0 && tid == 0) flag_status(MLA_ERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  const float* row = scores + (int64_t)b * stride;
  int32_t* out = sel_pos + (int64_t)b * k;
  if (c == 0 && tid == 0) {
    sel_count[b] = min(L, k);
    if (packed_base) packed_base[b] = (int64_t)b * k;
  }
  const int C = (int)gridDim.x;  // the cluster spans the grid's x dimension
  const int S = (L + C - 1) / C;
  const int s0 = min(L, c * S), s1 = min(L, s0 + S);
  if (L <= k) {  // every position is picked (the same branch for the whole cluster)
    for (int j = s0 + tid; j < s1; j += kSelThreads) out[j] = j;
    return;
  }
  // R consecutive positions per thread (R <= 32, all threads busy on short slices), in
  // rounds of 512 R positions; R and the round count may differ between the CTAs
  const int n_slice = s1 - s0;
  const int R = min(kKeysPerThread, max(1, (n_slice + kSelThreads - 1) / kSelThreads));
  const int chunk = kSelThreads * R;
  const int rounds = (n_slice + chunk - 1) / chunk;
  uint32_t kk[kKeysPerThread];
  auto load_round = [&](int r) {
    const int j0 = s0 + r * chunk + tid * R;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; ++i)
      kk[i] = (i < R && j0 + i < s1) ? score_key(__ldg(row + j0 + i)) : 0u;
  };
  if (rounds == 1) load_round(0);

  // barrier over the cluster (over the CTA alone when it is the whole cluster)
  auto sync_all = [&]() {
    if (C > 1)
      cluster_sync();
    else
      __syncthreads();
  };

  // ---- radix select
  uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
  for (int i = tid; i < kSelWarps * 256; i += kSelThreads) (&hist[0][0][0])[i] = 0u;
  __syncthreads();
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass, buf = pass & 1;
#pragma unroll 1
    for (int r = 0; r < rounds; ++r) {
      if (rounds > 1) load_round(r);
      const int j0 = s0 + r * chunk + tid * R;
#pragma unroll
      for (int i = 0; i < kKeysPerThread; ++i) {
        if (i >= R) break;
        if (j0 + i < s1 && (kk[i] & mask) == prefix)
          atomicAdd(&hist[buf][warp][(kk[i] >> shift) & 255u], 1u);
      }
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) t += hist[buf][w][tid];
      hist_cta[buf][tid] = t;
    }
    // the other histogram buffer (last read in the previous pass) for the next pass
    for (int i = tid; i < kSelWarps * 256; i += kSelThreads) (&hist[buf ^ 1][0][0])[i] = 0u;
    sync_all();  // every CTA's totals of this pass are visible to the cluster
    // totals over the cluster, then the bin holding the need-th largest key: lane l of warp 0
    // owns bins 255-8l down to 248-8l (every CTA computes the same answer)
    if (warp == 0) {
      // all 64 remote loads in flight before any is used
      uint32_t rv[8][kSelMaxCluster];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t a = smem_u32(&hist_cta[buf][255 - 8 * lane - q]);
#pragma unroll
        for (int rk = 0; rk < kSelMaxCluster; ++rk)
          rv[q][rk] = rk < C ? ld_cluster_u32(mapa_shared(a, rk)) : 0u;
      }
      uint32_t cb[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t t = 0;
#pragma unroll
        for (int rk = 0; rk < kSelMaxCluster; ++rk) t += rv[q][rk];
        cb[q] = t;
        sum += t;
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      const uint32_t reach = __ballot_sync(0xffffffffu, incl >= need);
      const int owner = __ffs(reach) - 1;  // reach != 0: need <= keys matching the prefix
      if (lane == owner) {
        uint32_t above = incl - sum;
        int q = 0;
        for (; q < 7; ++q) {
          if (above + cb[q] >= need) break;
          above += cb[q];
        }
        s_prefix = prefix | ((uint32_t)(255 - 8 * lane - q) << shift);
        s_need = need - above;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;  // key of the k-th largest score

  // ---- this CTA's counts, then the counts of the slices before it
  uint32_t n_gt = 0, n_eq = 0;
#pragma unroll 1
  for (int r = 0; r < rounds; ++r) {
    if (rounds > 1) load_round(r);
    const int j0 = s0 + r * chunk + tid * R;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; ++i) {
      if (i >= R) break;
      n_gt += (j0 + i < s1 && kk[i] > T);
      n_eq += (j0 + i < s1 && kk[i] == T);
    }
  }
  // per-CTA totals can exceed 2^16 over several rounds: two scans rather than one packed one
  uint32_t tot_gt, tot_eq;
  block_exclusive_scan(n_gt, scan_tmp, &tot_gt);
  block_exclusive_scan(n_eq, scan_tmp, &tot_eq);
  if (tid == 0) {
    cnt_cta[0] = tot_gt;
    cnt_cta[1] = tot_eq;
  }
  sync_all();
  if (warp == 0) {  // lane rk < c reads CTA rk's counts; a warp sum adds them
    uint32_t g = 0, e = 0;
    if (lane < c) {
      g = ld_cluster_u32(mapa_shared(smem_u32(&cnt_cta[0]), lane));
      e = ld_cluster_u32(mapa_shared(smem_u32(&cnt_cta[1]), lane));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if (lane == 0) {
      s_gt0 = g;
      s_eq0 = e;
    }
  }
  __syncthreads();

  // ---- compaction in position order: keys above T, then the first `need` keys equal to T
  uint32_t gt_before = s_gt0, eq_before = s_eq0;
#pragma unroll 1
  for (int r = 0; r < rounds; ++r) {
    if (rounds > 1) load_round(r);
    const int j0 = s0 + r * chunk + tid * R;
    uint32_t g_n = 0, e_n = 0;
#pragma unroll
    for (int i = 0; i < kKeysPerThread; ++i) {
      if (i >= R) break;
      g_n += (j0 + i < s1 && kk[i] > T);
      e_n += (j0 + i < s1 && kk[i] == T);
    }
    uint32_t rt;
    const uint32_t ex = block_exclusive_scan(g_n | (e_n << 16), scan_tmp, &rt);
    uint32_t g = gt_before + (ex & 0xffffu), e = eq_before + (ex >> 16);
#pragma unroll
    for (int i = 0; i < kKeysPerThread; ++i) {
      if (i >= R || j0 + i >= s1) break;
      if (kk[i] > T) {
        out[g + min(e, need)] = j0 + i;
        ++g;
      } else if (kk[i] == T) {
        if (e < need) out[g + e] = j0 + i;
        ++e;
      }
    }
    gt_before += rt & 0xffffu;
    eq_before += rt >> 16;
  }
  if (C > 1) cluster_sync();  // no CTA leaves while another may still read its shared memory
}

template <int kRowVecs>  // 16-byte vectors per cache row
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ rows, const int64_t* __restrict__ seq_base,
                   int64_t capacity, const int32_t* __restrict__ sel_pos,
                   const int32_t* __restrict__ sel_count, int k, uint4* __restrict__ packed) {
  const int b = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= k || i >= sel_count[b]) return;
  const int64_t src = seq_base[b] + sel_pos[(int64_t)b * k + i];
  uint4* dst = packed + ((int64_t)b * k + i) * kRowVecs;
  if (src < 0 || src >= capacity) {
    if (lane == 0) flag_status(MLA_ERR_CAPACITY);
    for (int v = lane; v < kRowVecs; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* s = rows + src * kRowVecs;
  uint4 r[(kRowVecs + 31) / 32];
#pragma unroll
  for (int q = 0; q < (kRowVecs + 31) / 32; ++q)
    if (q * 32 + lane < kRowVecs) r[q] = __ldg(s + q * 32 + lane);
#pragma unroll
  for (int q = 0; q < (kRowVecs + 31) / 32; ++q)
    if (q * 32 + lane < kRowVecs) dst[q * 32 + lane] = r[q];
}

// Generic row width (any multiple of 16 bytes).
__global__ void __launch_bounds__(256)
gather_rows_any_kernel(const uint4* __restrict__ rows, int row_vecs,
                       const int64_t* __restrict__ seq_base, int64_t capacity,
                       const int32_t* __restrict__ sel_pos, const int32_t* __restrict__ sel_count,
                       int k, uint4* __restrict__ packed) {
  const int b = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= k || i >= sel_count[b]) return;
  const int64_t src = seq_base[b] + sel_pos[(int64_t)b * k + i];
  uint4* dst = packed + ((int64_t)b * k + i) * row_vecs;
  if (src < 0 || src >= capacity) {
    if (lane == 0) flag_status(MLA_ERR_CAPACITY);
    for (int v = lane; v < row_vecs; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* s = rows + src * row_vecs;
  for (int v = lane; v < row_vecs; v += 32) dst[v] = __ldg(s + v);
}

}  // namespace

mla_status_t select_topk(const float* scores, int64_t stride, const int32_t* seq_len, int B,
                         int max_len, int k, int32_t* sel_pos, int32_t* sel_count,
                         int64_t* packed_base, cudaStream_t st) {
  TraceScope tr(K_TOPK, st);
  const int C = std::min(kSelMaxCluster, std::max(1, (max_len + kSelSlice - 1) / kSelSlice));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, B, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, topk_select_kernel, scores, stride, seq_len, max_len, k, sel_pos,
                         sel_count, packed_base) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
  return launch_status();
}

mla_status_t gather_rows(const mla_dims_t* d, const mla_cache_t* cache, const int32_t* sel_pos,
                         const int32_t* sel_count, int B, int k, void* packed, cudaStream_t st) {
  const int row_bytes = (d->d_c + d->d_hr) * (int)elem_bytes(d);
  const int vecs = row_bytes / 16;
  const dim3 grid((unsigned)ceil_div(k, 8), (unsigned)B);
  TraceScope tr(K_GATHER, st);
  if (vecs == 72)  // the V2 row: 576 bf16
    gather_rows_kernel<72><<<grid, 256, 0, st>>>(
        reinterpret_cast<const uint4*>(cache->rows), cache->seq_base, cache->capacity, sel_pos,
        sel_count, k, reinterpret_cast<uint4*>(packed));
  else
    gather_rows_any_kernel<<<grid, 256, 0, st>>>(
        reinterpret_cast<const uint4*>(cache->rows), vecs, cache->seq_base, cache->capacity,
        sel_pos, sel_count, k, reinterpret_cast<uint4*>(packed));
  return launch_status();
}

}  // namespace mla
