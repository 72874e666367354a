// Absorbed decode whose scratch is a fixed array inside the library, for callers that cannot
// allocate device memory (the pages have no counterpart; see mla_decode_absorbed_static in
// include/mla.h). The arithmetic is mla_decode_absorbed's: this file only supplies the scratch.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kStaticWsBytes = MLA_STATIC_WS_BYTES;
constexpr int kMaxDevices = 64;

// The scratch. Device code could name it directly; host code must use the address that
// cudaGetSymbolAddress returns (the host-side symbol is only a stand-in, not a device address).
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticWsBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
mla_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_absorbed_static(const mla_dims_t* dims, const mla_weights_t* w,
                                                   const void* q_c, const void* q_r,
                                                   const mla_cache_t* cache,
                                                   const int32_t* seq_len, int32_t B,
                                                   int32_t max_len, float* o, void* stream) {
  size_t need = 0;
  mla_status_t s = mla_decode_workspace_size(dims, B, max_len, &need);
  if (s != MLA_OK) return s;
  if (need > kStaticWsBytes) return MLA_ERR_WORKSPACE;
  void* ws = nullptr;
  s = scratch_address(&ws);
  if (s != MLA_OK) return s;
  return mla_decode_absorbed(dims, w, q_c, q_r, cache, seq_len, B, max_len, ws, kStaticWsBytes,
                             o, stream);
}
