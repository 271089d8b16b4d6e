// Host-side launchers of the decoder kernels (ctcpb_kernels.cu).
#pragma once

#include <mutex>

#include "ctcpb_internal.cuh"

namespace ctcpb {

// Raise kernel K's dynamic shared-memory limit to at least `bytes` on the
// current device.  The limit is an attribute of the kernel on each device, so
// it is set once per device (and again when a launch needs more); the mutex
// makes first launches from several host threads safe.
template <auto K>
cudaError_t smem_optin(size_t bytes) {
  constexpr int kDevices = 128;
  static std::mutex mu;
  static size_t done[kDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  const bool known = dev >= 0 && dev < kDevices;
  if (known && done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && known) done[dev] = bytes;
  return e;
}

cudaError_t launch_init(const View& st, cudaStream_t s);
// Every row's label-boost hash table from compressed-row (row_ptr, tokens, bonus) device arrays.
cudaError_t launch_boost_build(const View& st, const int* row_ptr, const int* tokens, const float* bonus,
                               cudaStream_t s);
// Speech-masked streaming: the tile's selected chunk rows per stream.
cudaError_t launch_select_tile(const View& st, const uint8_t* mask, long long mstride, const int* nframes,
                               int chunk_T, int tile_start, int tile_len, cudaStream_t s);
// The same selection by the blank threshold (lp[b, j, blank] < log_thr, section 3.5) of the chunk.
cudaError_t launch_select_tile_thr(const View& st, const float* lp, long long sb, long long stt, float log_thr,
                                   const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s);
// Frames of each row in each chunk of F frames, for the host-buffer decode: plan [nchunks][B].
cudaError_t launch_host_plan(const int* lens, int B, int T, int F, int nchunks, int* plan, cudaStream_t s);
cudaError_t launch_init_select(const View& st, const float* lp, long long sb, long long stt, const int* lens, int T,
                               int mode, float log_thr, int* sel, int* nsel, cudaStream_t s);
cudaError_t launch_select(const View& st, const float* lp, long long sb, long long stt, const int* lens, int T,
                          int mode, float log_thr, int* sel, int* nsel, cudaStream_t s);
cudaError_t launch_prepass(const View& st, const float* lp, long long sb, long long stt, int mode,
                           const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s);
cudaError_t launch_prepass_rows(const float* lp, long long stride_r, int R, int V, int blank, int L, int* ids,
                                float* lps, int* cnt, float* lpb, float* flp, int* fid, cudaStream_t s);
cudaError_t launch_step(const View& st, const float* lp, long long sb, long long stt, int mode, const int* nframes,
                        int chunk_T, int tile_start, int tile_len, cudaStream_t s);
// Pre-pass and steps of one tile in a single cooperative launch (the pre-pass
// publishes records that the step warps consume as they arrive).  Returns
// cudaErrorNotSupported, launching nothing and leaving no error pending, when
// the problem or the device does not allow it (a cooperative grid too large
// for the device included); the caller then launches the two kernels one
// after the other.  Any other error is a real failure.
cudaError_t launch_fused(const View& st, const float* lp, long long sb, long long stt, int mode, const int* nframes,
                         int chunk_T, int tile_start, int tile_len, cudaStream_t s);
bool rank_tma_ok(const float* lp, long long s1, long long s2, int V, int L);
int rank_tma_warps(int V);

// The warp-per-row step kernel takes flat storage, beam <= 16 and a ranked
// record of at most 32 + 8*68 bytes (list length <= 66).
bool step_warp_fits(const Layout& lay);
cudaError_t launch_step_warp(const View& st, const float* lp, long long sb, long long stt, int mode,
                             const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s);
cudaError_t launch_output(const View& st, int nbest, int* out_tokens, int* out_lengths, float* out_scores,
                          int out_len, cudaStream_t s);

}  // namespace ctcpb
