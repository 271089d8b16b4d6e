// C ABI of the decoder (include/ctcpb.h): argument validation on the host,
// workspace/state layout, and the launch sequence of each call.
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "ctcpb.h"
#include "ctcpb_internal.cuh"
#include "ctcpb_kernels.h"

using namespace ctcpb;

namespace {

bool finite_or_inf(float x) { return !std::isnan(x); }

// Section 11 / 13: refuse out-of-range configurations.
int check_cfg(const ctcpb_config* c, int V) {
  if (!c) return CTCPB_ENULL;
  if (V < 2 || V > kMaxV) return CTCPB_EINVAL;
  if (c->beam < 1 || c->beam > kMaxBeam) return CTCPB_EINVAL;
  if (c->nbest < 1 || c->nbest > c->beam) return CTCPB_EINVAL;
  if (c->blank_id < 0 || c->blank_id >= V) return CTCPB_EINVAL;
  if (c->paged != 0 && c->paged != 1) return CTCPB_EINVAL;
  if (c->paged && (c->page_size < 1 || c->page_size > 1024)) return CTCPB_EINVAL;
  if (c->list_len < 0) return CTCPB_EINVAL;
  if (!finite_or_inf(c->blank_threshold)) return CTCPB_EINVAL;
  if (c->word_boundary != 0 && c->word_boundary != 1) return CTCPB_EINVAL;
  if (c->word_boundary && (c->space_id < 0 || c->space_id >= V)) return CTCPB_EINVAL;
  if (c->max_boost < 0 || c->max_boost > kMaxBoost) return CTCPB_EINVAL;
  return CTCPB_OK;
}

int offline_cap(const ctcpb_config* c, int T) {
  const int t = T > 1 ? T : 1;
  // no hypothesis can hold more labels than frames: a larger cap never binds
  return (c->max_seq_len > 0 && c->max_seq_len < t) ? c->max_seq_len : t;
}

int space_of(const ctcpb_config* c) { return c->word_boundary ? c->space_id : -1; }

int stream_cap(const ctcpb_config* c) { return c->max_seq_len > 0 ? c->max_seq_len : kStreamDefaultCap; }

Layout offline_layout(const ctcpb_config* c, int B, int T, int V) {
  return make_layout(B, V, c->beam, offline_cap(c, T), c->paged, c->paged ? c->page_size : 16, c->blank_id,
                     default_list_len(c->beam, V, c->list_len), T > 0 ? T : 1, T > 0 ? T : 1, space_of(c),
                     c->max_boost);
}

Layout stream_layout(const ctcpb_config* c, int B, int V) {
  // T_sel = kStreamTile: the selection holds one tile's chunk rows (speech-masked streaming)
  return make_layout(B, V, c->beam, stream_cap(c), c->paged, c->paged ? c->page_size : 16, c->blank_id,
                     default_list_len(c->beam, V, c->list_len), kStreamTile, kStreamTile, space_of(c),
                     c->max_boost);
}

int check_buf(const void* p, size_t have, size_t need) {
  if (!p) return CTCPB_ENULL;
  if (((uintptr_t)p & 255u) != 0) return CTCPB_EALIGN;
  if (have < need) return CTCPB_ESIZE;
  return CTCPB_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? CTCPB_OK : CTCPB_ECUDA; }

// A label-boost argument: boosting configured, every array given.
int check_boost(const ctcpb_config* c, const ctcpb_boost* bo) {
  if (c->max_boost < 1) return CTCPB_EINVAL;
  if (!bo || !bo->row_ptr || !bo->tokens || !bo->bonus) return CTCPB_ENULL;
  return CTCPB_OK;
}

#define TRY(x)                      \
  do {                              \
    cudaError_t e_ = (x);           \
    if (e_ != cudaSuccess) return CTCPB_ECUDA; \
  } while (0)

// Pre-pass and steps of one tile in one cooperative launch when the device and
// the problem allow it; CTCPB_NO_FUSE=1 in the environment turns it off.
// Returns 1 when launched, 0 when not available (the caller launches the two
// kernels one after the other), CTCPB_ECUDA on a real CUDA failure.
int try_fused(const View& st, const float* lp, long long sb, long long stt, int mode, const int* nframes,
              int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  static const bool off = [] {
    const char* e = std::getenv("CTCPB_NO_FUSE");
    return e && e[0] == '1';
  }();
  if (off) return 0;
  const cudaError_t e = launch_fused(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
  if (e == cudaSuccess) return 1;
  return e == cudaErrorNotSupported ? 0 : CTCPB_ECUDA;
}

#define FUSED_OR_TWO_KERNELS(st, lp, sb, stt, mode, nf, cT, t0, tl, s)                     \
  do {                                                                                    \
    const int f_ = try_fused(st, lp, sb, stt, mode, nf, cT, t0, tl, s);                    \
    if (f_ < 0) return f_;                                                                \
    if (f_ == 0) {                                                                        \
      TRY(launch_prepass(st, lp, sb, stt, mode, nf, cT, t0, tl, s));                       \
      TRY(launch_step(st, lp, sb, stt, mode, nf, cT, t0, tl, s));                          \
    }                                                                                     \
  } while (0)

}  // namespace

extern "C" {

const char* ctcpb_status_string(int s) {
  switch (s) {
    case CTCPB_OK: return "ok";
    case CTCPB_EINVAL: return "invalid dimension or configuration value";
    case CTCPB_ENULL: return "required pointer is NULL";
    case CTCPB_EALIGN: return "workspace/state pointer is not 256-byte aligned";
    case CTCPB_ESIZE: return "workspace/state buffer is smaller than its size query";
    case CTCPB_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

int ctcpb_lse_table(float* out, int n) {
  static constexpr FCoef kTable = make_fcoef();
  if (n < 0) return CTCPB_EINVAL;
  if (n > 0 && !out) return CTCPB_ENULL;
  for (int i = 0; i < n && i < kFCoef; ++i) out[i] = kTable.c[i];
  return kFCoef;
}

int ctcpb_list_len(const ctcpb_config* cfg, int V) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  return default_list_len(cfg->beam, V, cfg->list_len);
}

int ctcpb_workspace_size(const ctcpb_config* cfg, int B, int T, int V, size_t* bytes) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (!bytes) return CTCPB_ENULL;
  if (B < 0 || T < 0) return CTCPB_EINVAL;
  *bytes = offline_layout(cfg, B, T, V).total;
  return CTCPB_OK;
}

}  // extern "C"

namespace {

// The offline decode stages; boost (may be null) is built right after the init.
int decode_offline_impl(const ctcpb_config* cfg, const ctcpb_boost* boost, const float* log_prob, int64_t stride_b,
                        int64_t stride_t, const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                        int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                        uint32_t stage_mask, ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (boost && (rc = check_boost(cfg, boost))) return rc;
  if (B < 0 || T < 0 || out_len < 0) return CTCPB_EINVAL;
  if (stage_mask & ~CTCPB_STAGE_ALL) return CTCPB_EINVAL;
  if (B == 0) return CTCPB_OK;
  if (stride_t < V || stride_b < V) return CTCPB_EINVAL;
  if ((T > 0 && !log_prob) || !out_lengths || !out_scores || (out_len > 0 && !out_tokens)) return CTCPB_ENULL;
  const Layout lay = offline_layout(cfg, B, T, V);
  if ((rc = check_buf(ws, ws_bytes, lay.total))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  View st{(char*)ws, lay};
  const float thr = cfg->blank_threshold;
  const int mode = thr >= 1.0f ? 0 : (thr > 0.0f ? 1 : 2);
  const float log_thr = mode == 1 ? (float)std::log((double)thr) : 0.0f;
  // the reset and the selection share a launch when both run
  const bool init_select = (stage_mask & CTCPB_STAGE_INIT) && (stage_mask & CTCPB_STAGE_SELECT) && T > 0;
  if (init_select)
    TRY(launch_init_select(st, log_prob, stride_b, stride_t, seq_lengths, T, mode, log_thr, st.sel(), st.nsel(), s));
  else if (stage_mask & CTCPB_STAGE_INIT)
    TRY(launch_init(st, s));
  if ((stage_mask & CTCPB_STAGE_INIT) && boost)
    TRY(launch_boost_build(st, boost->row_ptr, boost->tokens, boost->bonus, s));
  if (T > 0) {
    if ((stage_mask & CTCPB_STAGE_SELECT) && !init_select)
      TRY(launch_select(st, log_prob, stride_b, stride_t, seq_lengths, T, mode, log_thr, st.sel(), st.nsel(), s));
    const bool both = (stage_mask & CTCPB_STAGE_RANK) && (stage_mask & CTCPB_STAGE_STEPS);
    const int fused = both ? try_fused(st, log_prob, stride_b, stride_t, 0, nullptr, 0, 0, T, s) : 0;
    if (fused < 0) return fused;
    if (fused == 0) {
      if (stage_mask & CTCPB_STAGE_RANK) TRY(launch_prepass(st, log_prob, stride_b, stride_t, 0, nullptr, 0, 0, T, s));
      if (stage_mask & CTCPB_STAGE_STEPS) TRY(launch_step(st, log_prob, stride_b, stride_t, 0, nullptr, 0, 0, T, s));
    }
  }
  if (stage_mask & CTCPB_STAGE_OUTPUT)
    TRY(launch_output(st, cfg->nbest, out_tokens, out_lengths, out_scores, out_len, s));
  return CTCPB_OK;
}

}  // namespace

extern "C" {

int ctcpb_decode_offline_staged(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                                const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                                int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                                uint32_t stage_mask, ctcpb_stream_t stream) {
  return decode_offline_impl(cfg, nullptr, log_prob, stride_b, stride_t, seq_lengths, B, T, V, ws, ws_bytes,
                             out_tokens, out_lengths, out_scores, out_len, stage_mask, stream);
}

int ctcpb_decode_offline_boosted(const ctcpb_config* cfg, const ctcpb_boost* boost, const float* log_prob,
                                 int64_t stride_b, int64_t stride_t, const int32_t* seq_lengths, int B, int T,
                                 int V, void* ws, size_t ws_bytes, int32_t* out_tokens, int32_t* out_lengths,
                                 float* out_scores, int out_len, ctcpb_stream_t stream) {
  return decode_offline_impl(cfg, boost, log_prob, stride_b, stride_t, seq_lengths, B, T, V, ws, ws_bytes,
                             out_tokens, out_lengths, out_scores, out_len, CTCPB_STAGE_ALL, stream);
}

int ctcpb_decode_offline(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                         const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                         int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                         ctcpb_stream_t stream) {
  return ctcpb_decode_offline_staged(cfg, log_prob, stride_b, stride_t, seq_lengths, B, T, V, ws, ws_bytes,
                                     out_tokens, out_lengths, out_scores, out_len, CTCPB_STAGE_ALL, stream);
}

int ctcpb_state_size(const ctcpb_config* cfg, int B, int V, size_t* bytes) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (!bytes) return CTCPB_ENULL;
  if (B < 0) return CTCPB_EINVAL;
  *bytes = stream_layout(cfg, B, V).total;
  return CTCPB_OK;
}

int ctcpb_stream_init(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                      ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (B < 0) return CTCPB_EINVAL;
  const Layout lay = stream_layout(cfg, B, V);
  if ((rc = check_buf(state, state_bytes, lay.total))) return rc;
  View st{(char*)state, lay};
  return cuda_rc(launch_init(st, (cudaStream_t)stream));
}

int ctcpb_stream_set_boost(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                           const ctcpb_boost* boost, ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if ((rc = check_boost(cfg, boost))) return rc;
  if (B < 0) return CTCPB_EINVAL;
  const Layout lay = stream_layout(cfg, B, V);
  if ((rc = check_buf(state, state_bytes, lay.total))) return rc;
  View st{(char*)state, lay};
  return cuda_rc(launch_boost_build(st, boost->row_ptr, boost->tokens, boost->bonus, (cudaStream_t)stream));
}

int ctcpb_stream_step_chunk(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                            const float* lp_chunk, int64_t stride_b, int64_t stride_t, const int32_t* n_frames,
                            int chunk_T, ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (B < 0 || chunk_T < 0) return CTCPB_EINVAL;
  if (B == 0 || chunk_T == 0) return CTCPB_OK;
  if (stride_t < V || stride_b < V) return CTCPB_EINVAL;
  if (!lp_chunk) return CTCPB_ENULL;
  const Layout lay = stream_layout(cfg, B, V);
  if ((rc = check_buf(state, state_bytes, lay.total))) return rc;
  View st{(char*)state, lay};
  cudaStream_t s = (cudaStream_t)stream;
  for (int t0 = 0; t0 < chunk_T; t0 += kStreamTile) {
    const int tl = chunk_T - t0 < kStreamTile ? chunk_T - t0 : kStreamTile;
    FUSED_OR_TWO_KERNELS(st, lp_chunk, stride_b, stride_t, 1, n_frames, chunk_T, t0, tl, s);
  }
  return CTCPB_OK;
}

int ctcpb_stream_step_chunk_masked(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V,
                                   const float* lp_chunk, int64_t stride_b, int64_t stride_t,
                                   const int32_t* n_frames, const uint8_t* is_speech, int64_t mask_stride,
                                   int chunk_T, ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (B < 0 || chunk_T < 0) return CTCPB_EINVAL;
  if (B == 0 || chunk_T == 0) return CTCPB_OK;
  if (stride_t < V || stride_b < V || mask_stride < chunk_T) return CTCPB_EINVAL;
  if (!lp_chunk || !is_speech) return CTCPB_ENULL;
  const Layout lay = stream_layout(cfg, B, V);
  if ((rc = check_buf(state, state_bytes, lay.total))) return rc;
  View st{(char*)state, lay};
  cudaStream_t s = (cudaStream_t)stream;
  for (int t0 = 0; t0 < chunk_T; t0 += kStreamTile) {
    const int tl = chunk_T - t0 < kStreamTile ? chunk_T - t0 : kStreamTile;
    TRY(launch_select_tile(st, is_speech, mask_stride, n_frames, chunk_T, t0, tl, s));
    FUSED_OR_TWO_KERNELS(st, lp_chunk, stride_b, stride_t, 2, n_frames, chunk_T, t0, tl, s);
  }
  return CTCPB_OK;
}

int ctcpb_stream_step(const ctcpb_config* cfg, void* state, size_t state_bytes, int B, int V, const float* lp_frame,
                      int64_t stride_b, const uint8_t* is_speech, ctcpb_stream_t stream) {
  // a chunk of one frame; its frame stride is never stepped over, so it is
  // given the row stride, which keeps the row addresses' alignment the same
  if (!is_speech)
    return ctcpb_stream_step_chunk(cfg, state, state_bytes, B, V, lp_frame, stride_b, stride_b, nullptr, 1, stream);
  return ctcpb_stream_step_chunk_masked(cfg, state, state_bytes, B, V, lp_frame, stride_b, stride_b, nullptr,
                                        is_speech, 1, 1, stream);
}

int ctcpb_read_state(const ctcpb_config* cfg, const void* state, size_t state_bytes, int B, int V,
                     int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                     ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (B < 0 || out_len < 0) return CTCPB_EINVAL;
  if (B == 0) return CTCPB_OK;
  if (!out_lengths || !out_scores || (out_len > 0 && !out_tokens)) return CTCPB_ENULL;
  const Layout lay = stream_layout(cfg, B, V);
  if ((rc = check_buf(state, state_bytes, lay.total))) return rc;
  View st{(char*)state, lay};
  return cuda_rc(launch_output(st, cfg->nbest, out_tokens, out_lengths, out_scores, out_len, (cudaStream_t)stream));
}

int ctcpb_read_status(const void* ws_or_state, uint32_t* device_status) {
  if (!ws_or_state || !device_status) return CTCPB_ENULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return CTCPB_ECUDA;
  Header h;
  if (cudaMemcpy(&h, ws_or_state, sizeof(Header), cudaMemcpyDeviceToHost) != cudaSuccess) return CTCPB_ECUDA;
  *device_status = h.status;
  return CTCPB_OK;
}

int ctcpb_read_counters(const void* ws_or_state, uint32_t counters[6]) {
  if (!ws_or_state || !counters) return CTCPB_ENULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return CTCPB_ECUDA;
  Header h;
  if (cudaMemcpy(&h, ws_or_state, sizeof(Header), cudaMemcpyDeviceToHost) != cudaSuccess) return CTCPB_ECUDA;
  for (int i = 0; i < 5; ++i) counters[i] = h.counters[i];
  counters[5] = h.fused_launches;
  return CTCPB_OK;
}

int ctcpb_select_frames(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                        const int32_t* seq_lengths, int B, int T, int V, int32_t* sel, int32_t* nsel,
                        ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (B < 0 || T < 0) return CTCPB_EINVAL;
  if (B == 0) return CTCPB_OK;
  if (stride_t < V || stride_b < V) return CTCPB_EINVAL;
  if ((T > 0 && (!log_prob || !sel)) || !nsel) return CTCPB_ENULL;
  Layout lay{};
  lay.B = B;
  lay.V = V;
  lay.blank = cfg->blank_id;
  View st{nullptr, lay};
  const float thr = cfg->blank_threshold;
  const int mode = thr >= 1.0f ? 0 : (thr > 0.0f ? 1 : 2);
  const float log_thr = mode == 1 ? (float)std::log((double)thr) : 0.0f;
  return cuda_rc(launch_select(st, log_prob, stride_b, stride_t, seq_lengths, T, mode, log_thr, sel, nsel,
                               (cudaStream_t)stream));
}

int ctcpb_topk_prepass(const ctcpb_config* cfg, const float* log_prob, int64_t stride_r, int R, int V, int32_t* ids,
                       float* lps, int32_t* cnt, float* lpb, float* front_lp, int32_t* front_id,
                       ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (R < 0 || stride_r < V) return CTCPB_EINVAL;
  if (R == 0) return CTCPB_OK;
  if (!log_prob || !ids || !lps || !cnt || !lpb || !front_lp || !front_id) return CTCPB_ENULL;
  const int L = default_list_len(cfg->beam, V, cfg->list_len);
  return cuda_rc(launch_prepass_rows(log_prob, stride_r, R, V, cfg->blank_id, L, ids, lps, cnt, lpb, front_lp,
                                     front_id, (cudaStream_t)stream));
}

}  // extern "C"

// ------------------------------------------------------------------ host-buffer offline decode
namespace {

constexpr size_t kHostSegment = 1u << 20;  // bytes of a row a chunk copies at least: host-to-device
                                           // copies run at full speed from about 1 MB per segment
constexpr int kHostBufs = 3;             // chunk buffers in the workspace
constexpr int kCopyStreams = 1;          // chunks arrive in order (the copy bandwidth is shared, not added)

// Workspace of ctcpb_decode_offline_host: a decode state with streaming tiles
// and the offline cap, the row lengths, the per-chunk frame counts, the chunk
// buffers [kHostBufs][B][F][V] and the device outputs.
struct HostLayout {
  Layout st;
  int F, nchunks;
  size_t o_lens, o_plan, o_buf, buf_elems, o_tok, o_len, o_sc, total;
};

HostLayout host_layout(const ctcpb_config* c, int B, int T, int V, int out_len) {
  HostLayout h{};
  h.st = make_layout(B, V, c->beam, offline_cap(c, T), c->paged, c->paged ? c->page_size : 16, c->blank_id,
                     default_list_len(c->beam, V, c->list_len), kStreamTile, kStreamTile, space_of(c),
                     c->max_boost);
  // frames per chunk: whole streaming tiles covering >= kHostSegment bytes of a row
  const size_t row_bytes = 4 * (size_t)V;
  int F = (int)((kHostSegment + row_bytes - 1) / row_bytes);
  F = (F + kStreamTile - 1) / kStreamTile * kStreamTile;
  h.F = T < F ? (T > 0 ? T : 1) : F;
  h.nchunks = T > 0 ? (T + h.F - 1) / h.F : 0;
  size_t off = h.st.total;
  auto take = [&](size_t bytes) {
    const size_t at = align_up(off, 256);
    off = at + bytes;
    return at;
  };
  const size_t nb = (size_t)B * c->nbest;
  h.o_lens = take(4 * (size_t)B);
  h.o_plan = take(4 * (size_t)B * (size_t)(h.nchunks > 0 ? h.nchunks : 1));
  h.buf_elems = (size_t)B * h.F * V;
  h.o_buf = take(4 * h.buf_elems * kHostBufs);
  h.o_tok = take(4 * nb * (size_t)(out_len > 0 ? out_len : 0));
  h.o_len = take(4 * nb);
  h.o_sc = take(4 * nb);
  h.total = align_up(off, 256);
  return h;
}

// The copy streams and the events that order them against the decode, one
// set per device, made on first use and kept for the process.
struct HostRes {
  cudaStream_t cs[kCopyStreams];
  cudaEvent_t start, lens, ready[kHostBufs], done[kHostBufs];
};

std::mutex g_host_mu;

HostRes* host_res(int dev) {
  static HostRes res[64];
  static bool made[64];
  if (dev < 0 || dev >= 64) return nullptr;
  if (!made[dev]) {
    HostRes& r = res[dev];
    const unsigned ef = cudaEventDisableTiming;
    bool ok = true;
    for (int i = 0; i < kCopyStreams; ++i) ok = ok && cudaStreamCreateWithFlags(&r.cs[i], cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&r.start, ef) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&r.lens, ef) == cudaSuccess;
    for (int i = 0; i < kHostBufs; ++i) {
      ok = ok && cudaEventCreateWithFlags(&r.ready[i], ef) == cudaSuccess;
      ok = ok && cudaEventCreateWithFlags(&r.done[i], ef) == cudaSuccess;
    }
    if (!ok) return nullptr;
    made[dev] = true;
  }
  return &res[dev];
}

}  // namespace

extern "C" {

int ctcpb_host_workspace_size(const ctcpb_config* cfg, int B, int T, int V, int out_len, size_t* bytes) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (!bytes) return CTCPB_ENULL;
  if (B < 0 || T < 0 || out_len < 0) return CTCPB_EINVAL;
  *bytes = host_layout(cfg, B, T, V, out_len).total;
  return CTCPB_OK;
}

// The frames go to the device chunk by chunk on the copy streams; `stream`
// decodes chunk c (the streaming tile path, every frame or the frames the
// blank threshold keeps) once its copies are done, and chunk c's buffer is
// copied into again only after that decode.  Row b's chunk c holds its frames
// [cF, cF + F) that are below len_b; the others are never read.
}  // extern "C"

namespace {

int decode_offline_host_impl(const ctcpb_config* cfg, const ctcpb_boost* boost, const float* log_prob,
                             int64_t stride_b, int64_t stride_t, const int32_t* seq_lengths, int B, int T, int V,
                             void* ws, size_t ws_bytes, int32_t* out_tokens, int32_t* out_lengths, float* out_scores,
                             int out_len, ctcpb_stream_t stream) {
  int rc = check_cfg(cfg, V);
  if (rc) return rc;
  if (boost && (rc = check_boost(cfg, boost))) return rc;
  if (B < 0 || T < 0 || out_len < 0) return CTCPB_EINVAL;
  if (B == 0) return CTCPB_OK;
  if (T > 0 && (stride_t < V || stride_b < V)) return CTCPB_EINVAL;
  if ((T > 0 && !log_prob) || !out_lengths || !out_scores || (out_len > 0 && !out_tokens)) return CTCPB_ENULL;
  const HostLayout hl = host_layout(cfg, B, T, V, out_len);
  if ((rc = check_buf(ws, ws_bytes, hl.total))) return rc;
  int dev = 0;
  TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostRes* R = host_res(dev);
  if (!R) return CTCPB_ECUDA;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  View st{base, hl.st};
  int* lens_d = (int*)(base + hl.o_lens);
  int* plan = (int*)(base + hl.o_plan);
  float* bufs = (float*)(base + hl.o_buf);
  int* tok_d = (int*)(base + hl.o_tok);
  int* len_d = (int*)(base + hl.o_len);
  float* sc_d = (float*)(base + hl.o_sc);
  const int F = hl.F;
  std::vector<int> len_h(B);
  for (int b = 0; b < B; ++b) {
    const int L = seq_lengths ? seq_lengths[b] : T;
    len_h[b] = L < 0 ? 0 : (L > T ? T : L);
  }
  auto frames = [&](int b, int c0) {
    const int f = len_h[b] - c0;
    return f < 0 ? 0 : (f > F ? F : f);
  };

  // the copies start after the caller's earlier work on `stream`
  TRY(cudaEventRecord(R->start, s));
  for (int i = 0; i < kCopyStreams; ++i) TRY(cudaStreamWaitEvent(R->cs[i], R->start, 0));
  if (seq_lengths) {
    TRY(cudaMemcpyAsync(lens_d, seq_lengths, 4 * (size_t)B, cudaMemcpyHostToDevice, R->cs[0]));
    TRY(cudaEventRecord(R->lens, R->cs[0]));
    TRY(cudaStreamWaitEvent(s, R->lens, 0));
  }
  TRY(launch_host_plan(seq_lengths ? lens_d : nullptr, B, T, F, hl.nchunks, plan, s));
  TRY(launch_init(st, s));
  if (boost) TRY(launch_boost_build(st, boost->row_ptr, boost->tokens, boost->bonus, s));

  const float thr = cfg->blank_threshold;
  // every frame (mode 1), or the frames the threshold keeps (mode 2; thr <= 0 keeps none)
  const bool all = thr >= 1.0f;
  const float log_thr = thr > 0.0f ? (float)std::log((double)thr) : -FLT_MAX;
  const long long dsb = (long long)F * V;  // chunk buffer [B][F][V]
  const bool merge = stride_t == V && stride_b >= dsb;
  for (int c = 0; c < hl.nchunks; ++c) {
    const int k = c % kHostBufs, c0 = c * F;
    cudaStream_t cs = R->cs[c % kCopyStreams];
    float* buf = bufs + (size_t)k * hl.buf_elems;
    TRY(cudaStreamWaitEvent(cs, R->done[k], 0));  // the buffer's previous chunk is decoded
    for (int b = 0; b < B;) {
      const int n = frames(b, c0);
      if (n == 0) {
        ++b;
        continue;
      }
      const float* src = log_prob + (size_t)b * (size_t)stride_b + (size_t)c0 * (size_t)stride_t;
      if (n == F && merge) {  // a run of rows whose whole chunk is valid: one copy
        int e = b + 1;
        while (e < B && frames(e, c0) == F) ++e;
        TRY(cudaMemcpy2DAsync(buf + (size_t)b * dsb, (size_t)dsb * 4, src, (size_t)stride_b * 4, (size_t)dsb * 4,
                              (size_t)(e - b), cudaMemcpyHostToDevice, cs));
        b = e;
      } else {
        TRY(cudaMemcpy2DAsync(buf + (size_t)b * dsb, (size_t)V * 4, src, (size_t)stride_t * 4, (size_t)V * 4,
                              (size_t)n, cudaMemcpyHostToDevice, cs));
        ++b;
      }
    }
    TRY(cudaEventRecord(R->ready[k], cs));
    TRY(cudaStreamWaitEvent(s, R->ready[k], 0));
    const int* nf = plan + (size_t)c * B;
    const int mode = all ? 1 : 2;
    for (int t0 = 0; t0 < F; t0 += kStreamTile) {  // the chunk's streaming tiles
      const int tl = F - t0 < kStreamTile ? F - t0 : kStreamTile;
      if (!all) TRY(launch_select_tile_thr(st, buf, dsb, V, log_thr, nf, F, t0, tl, s));
      FUSED_OR_TWO_KERNELS(st, buf, dsb, V, mode, nf, F, t0, tl, s);
    }
    TRY(cudaEventRecord(R->done[k], s));
  }
  TRY(launch_output(st, cfg->nbest, tok_d, len_d, sc_d, out_len, s));
  const size_t nb = (size_t)B * cfg->nbest;
  TRY(cudaMemcpyAsync(out_lengths, len_d, 4 * nb, cudaMemcpyDeviceToHost, s));
  TRY(cudaMemcpyAsync(out_scores, sc_d, 4 * nb, cudaMemcpyDeviceToHost, s));
  if (out_len > 0) TRY(cudaMemcpyAsync(out_tokens, tok_d, 4 * nb * (size_t)out_len, cudaMemcpyDeviceToHost, s));
  return CTCPB_OK;
}

}  // namespace

extern "C" {

int ctcpb_decode_offline_host(const ctcpb_config* cfg, const float* log_prob, int64_t stride_b, int64_t stride_t,
                              const int32_t* seq_lengths, int B, int T, int V, void* ws, size_t ws_bytes,
                              int32_t* out_tokens, int32_t* out_lengths, float* out_scores, int out_len,
                              ctcpb_stream_t stream) {
  return decode_offline_host_impl(cfg, nullptr, log_prob, stride_b, stride_t, seq_lengths, B, T, V, ws, ws_bytes,
                                  out_tokens, out_lengths, out_scores, out_len, stream);
}

int ctcpb_decode_offline_host_boosted(const ctcpb_config* cfg, const ctcpb_boost* boost, const float* log_prob,
                                      int64_t stride_b, int64_t stride_t, const int32_t* seq_lengths, int B, int T,
                                      int V, void* ws, size_t ws_bytes, int32_t* out_tokens, int32_t* out_lengths,
                                      float* out_scores, int out_len, ctcpb_stream_t stream) {
  return decode_offline_host_impl(cfg, boost, log_prob, stride_b, stride_t, seq_lengths, B, T, V, ws, ws_bytes,
                                  out_tokens, out_lengths, out_scores, out_len, stream);
}

}  // extern "C"
