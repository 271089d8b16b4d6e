// Offline decode that allocates nothing (ctcpb_decode_offline_noalloc).
//
// Some callers cannot call cudaMalloc at all: plugins of engines that own the
// device heap and forbid allocations from outside it, and real-time paths that
// may not block in the allocator.  For them the decode's workspace lives in a
// file-scope device array of fixed size that every device loading this
// library holds until the process exits.
//
// Host code cannot use the array's name as a device address (it names a host
// stand-in), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, and caches it (the
// cached address does not survive cudaDeviceReset).
#include <mutex>

#include "ctcpb.h"
#include "ctcpb_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[CTCPB_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device; null until looked up

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CTCPB_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CTCPB_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CTCPB_OK;
}

}  // namespace

extern "C" int ctcpb_decode_offline_noalloc(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b,
                                            int64_t stride_t, const int32_t* seq_lengths, int B, int T, int V,
                                            int32_t* out_tokens, int32_t* out_lengths, float* out_scores,
                                            int out_len, ctcpb_stream_t stream) {
  size_t need = 0;
  int rc = ctcpb_workspace_size(cfg, B, T, V, &need);  // also validates the configuration
  if (rc != CTCPB_OK) return rc;
  if (need > (size_t)CTCPB_NOALLOC_SCRATCH_BYTES) return CTCPB_ESIZE;
  void* ws = nullptr;
  if ((rc = scratch_address(&ws)) != CTCPB_OK) return rc;
  // Every per-call value the decode reads is written earlier in the same call
  // (its first stage resets the per-row state), so the array's contents from
  // an earlier call never leak into this one.
  return ctcpb_decode_offline(cfg, log_prob, stride_b, stride_t, seq_lengths, B, T, V, ws,
                              (size_t)CTCPB_NOALLOC_SCRATCH_BYTES, out_tokens, out_lengths, out_scores, out_len,
                              stream);
}

// The status word of the array's header: the CTCPB_DEV_* bits of the last
// decode on the current device (synchronises the device).
extern "C" int ctcpb_noalloc_read_status(uint32_t* device_status) {
  if (!device_status) return CTCPB_ENULL;
  void* ws = nullptr;
  int rc = scratch_address(&ws);
  if (rc != CTCPB_OK) return rc;
  return ctcpb_read_status(ws, device_status);
}
