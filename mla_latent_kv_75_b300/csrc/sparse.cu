// Top-k sparse selection over the latent sequence before the decode ("MLA前向计算流程",
// version table, V3.2 + DSA row: MLA itself is unchanged; an indexer picks top-k positions
// of the latent sequence and the core attention runs MLA over the picked rows only).
//
// The indexer is not defined by the pages, so its scores are an input: one fp32 score per
// cached position. Two kernels:
//   topk_select_kernel  one CTA per sequence: an exact radix select of the k-th largest
//                       score (four 8-bit passes over order-preserving keys, warp-private
//                       shared-memory histograms), then an order-preserving compaction that
//                       writes the picked positions in increasing order. Equal scores rank the
//                       lower position first; -0.0 equals +0.0.
//   gather_rows_kernel  one warp per picked row: copies the row out of the cache into a
//                       packed per-sequence block (sequence b at rows b*k ...), 16 bytes per
//                       lane access, so that the unchanged decode kernels read it as a dense
//                       cache.
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kPerThread = 8;                      // consecutive positions per thread (compaction)
constexpr int kChunk = kSelThreads * kPerThread;   // positions per compaction round

// Order-preserving map of an fp32 bit pattern to uint32: a larger score gives a larger key,
// and both zeros give the same key.
__device__ __forceinline__ uint32_t score_key(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) == 0) return 0x80000000u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

__global__ void __launch_bounds__(kSelThreads)
topk_select_kernel(const float* __restrict__ scores, int64_t stride,
                   const int32_t* __restrict__ seq_len, int max_len, int k,
                   int32_t* __restrict__ sel_pos, int32_t* __restrict__ sel_count,
                   int64_t* __restrict__ packed_base) {
  __shared__ uint32_t hist[kSelWarps][256];
  __shared__ uint32_t scan_tmp[kSelWarps + 1];
  __shared__ uint32_t s_prefix, s_need;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int L = seq_len[b];
  if (L < 0 || L > max_len) {
    if (tid == 0) flag_status(MLA_ERR_LENGTH);
    L = L < 0 ? 0 : max_len;
  }
  const float* row = scores + (int64_t)b * stride;
  int32_t* out = sel_pos + (int64_t)b * k;
  if (tid == 0) {
    sel_count[b] = min(L, k);
    if (packed_base) packed_base[b] = (int64_t)b * k;
  }
  if (L <= k) {  // every position is picked
    for (int j = tid; j < L; j += kSelThreads) out[j] = j;
    return;
  }

  // ---- radix select: the key of the k-th largest score, and how many keys equal to it
  // are needed (the lowest positions among them)
  uint32_t prefix = 0, mask = 0, need = (uint32_t)k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kSelWarps * 256; i += kSelThreads) (&hist[0][0])[i] = 0u;
    __syncthreads();
    for (int j0 = 0; j0 < L; j0 += 32 * kSelThreads) {
      // 32 scores per thread per round: contiguous per warp, so each load instruction
      // reads 128 consecutive bytes
#pragma unroll 4
      for (int u = 0; u < 32; ++u) {
        const int j = j0 + (u * kSelWarps + warp) * 32 + lane;
        const bool ok = j < L;
        const uint32_t key = ok ? score_key(__ldg(row + j)) : 0u;
        const bool hit = ok && (key & mask) == prefix;
        const uint32_t bin = (key >> shift) & 255u;
        // lanes with the same bin add once (ties would otherwise serialise the atomics)
        const uint32_t act = __ballot_sync(0xffffffffu, hit);
        if (hit) {
          const uint32_t peers = __match_any_sync(act, bin);
          if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[warp][bin], __popc(peers));
        }
      }
    }
    __syncthreads();
    // total per bin over the warps, then the bin holding the need-th largest key: lane l
    // of warp 0 owns bins 255-8l down to 248-8l
    if (warp == 0) {
      uint32_t c[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int bin = 255 - 8 * lane - q;
        uint32_t t = 0;
        for (int w = 0; w < kSelWarps; ++w) t += hist[w][bin];
        c[q] = t;
        s += t;
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      const uint32_t reach = __ballot_sync(0xffffffffu, incl >= need);
      const int owner = __ffs(reach) - 1;  // reach != 0: need <= keys matching the prefix
      if (lane == owner) {
        uint32_t above = incl - s;
        int q = 0;
        for (; q < 7; ++q) {
          if (above + c[q] >= need) break;
          above += c[q];
        }
        const uint32_t bin = (uint32_t)(255 - 8 * lane - q);
        s_prefix = prefix | (bin << shift);
        s_need = need - above;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // key of the k-th largest score
  // ---- compaction in position order: keys above T, then the first `need` keys equal to T
  uint32_t gt_before = 0, eq_before = 0;
#pragma unroll 1
  for (int c0 = 0; c0 < L; c0 += kChunk) {
    const int j0 = c0 + tid * kPerThread;
    uint32_t kk[kPerThread];
    uint32_t n_gt = 0, n_eq = 0;
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int j = j0 + u;
      kk[u] = j < L ? score_key(__ldg(row + j)) : 0u;
      n_gt += (j < L && kk[u] > T);
      n_eq += (j < L && kk[u] == T);
    }
    // one scan of both counts (each below 2^16 per round)
    uint32_t tot;
    const uint32_t ex = block_exclusive_scan(n_gt | (n_eq << 16), scan_tmp, &tot);
    uint32_t g = gt_before + (ex & 0xffffu), e = eq_before + (ex >> 16);
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int j = j0 + u;
      if (j >= L) break;
      if (kk[u] > T) {
        out[g + min(e, need)] = j;
        ++g;
      } else if (kk[u] == T) {
        if (e < need) out[g + e] = j;
        ++e;
      }
    }
    gt_before += tot & 0xffffu;
    eq_before += tot >> 16;
  }
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
  topk_select_kernel<<<B, kSelThreads, 0, st>>>(scores, stride, seq_len, max_len, k, sel_pos,
                                                sel_count, packed_base);
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
