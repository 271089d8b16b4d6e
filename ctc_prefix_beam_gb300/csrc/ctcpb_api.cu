// C ABI of the decoder (include/ctcpb.h): argument validation on the host,
// workspace/state layout, and the launch sequence of each call.
#include <cmath>
#include <cstdint>
#include <cstdlib>

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
bool try_fused(const View& st, const float* lp, long long sb, long long stt, int mode, const int* nframes,
               int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  static const bool off = [] {
    const char* e = std::getenv("CTCPB_NO_FUSE");
    return e && e[0] == '1';
  }();
  if (off) return false;
  if (launch_fused(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s) == cudaSuccess) return true;
  cudaGetLastError();  // a refused cooperative launch: take the two-kernel path
  return false;
}

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
  if (stage_mask & CTCPB_STAGE_INIT) {
    TRY(launch_init(st, s));
    if (boost) TRY(launch_boost_build(st, boost->row_ptr, boost->tokens, boost->bonus, s));
  }
  if (T > 0) {
    const float thr = cfg->blank_threshold;
    const int mode = thr >= 1.0f ? 0 : (thr > 0.0f ? 1 : 2);
    const float log_thr = mode == 1 ? (float)std::log((double)thr) : 0.0f;
    if (stage_mask & CTCPB_STAGE_SELECT)
      TRY(launch_select(st, log_prob, stride_b, stride_t, seq_lengths, T, mode, log_thr, st.sel(), st.nsel(), s));
    const bool both = (stage_mask & CTCPB_STAGE_RANK) && (stage_mask & CTCPB_STAGE_STEPS);
    if (!(both && try_fused(st, log_prob, stride_b, stride_t, 0, nullptr, 0, 0, T, s))) {
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
    if (try_fused(st, lp_chunk, stride_b, stride_t, 1, n_frames, chunk_T, t0, tl, s)) continue;
    TRY(launch_prepass(st, lp_chunk, stride_b, stride_t, 1, n_frames, chunk_T, t0, tl, s));
    TRY(launch_step(st, lp_chunk, stride_b, stride_t, 1, n_frames, chunk_T, t0, tl, s));
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
    if (try_fused(st, lp_chunk, stride_b, stride_t, 2, n_frames, chunk_T, t0, tl, s)) continue;
    TRY(launch_prepass(st, lp_chunk, stride_b, stride_t, 2, n_frames, chunk_T, t0, tl, s));
    TRY(launch_step(st, lp_chunk, stride_b, stride_t, 2, n_frames, chunk_T, t0, tl, s));
  }
  return CTCPB_OK;
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
