// Vocabulary pre-pass ("GPU CTC Prefix Beam Search Decoder", section 3.4.7):
// for every decoded frame, the first L non-blank live labels by (log-prob
// desc, label asc), the blank log-prob and the next label ("front").
//
// One warp per frame row, 16 warps per block, a persistent grid of one block
// per SM: many rows in flight per SM keep HBM streaming.  A row is read with
// coalesced 16-byte loads (L2-resident for the second pass).  Ranking (exact):
//   1. each lane keeps the maxima of two disjoint halves of its labels (the
//      x,y and the z,w components of its float4 slices) in four independent
//      max chains: 64 distinct labels;
//   2. tau = the K-th largest of those 64 values, K = L + 1: at least K labels
//      score >= tau, so the top K all do;
//   3. every label >= tau is compacted (warp ballots) into shared memory;
//   4. each compacted label's rank = how many compacted keys beat it; the
//      first L go to the list, rank L is the front.
// Rows that are not 16-byte aligned, lists longer than 511 labels, and
// compactions past the buffer use the plain per-warp ranking (rank_row).
#include "ctcpb_rank.cuh"
#include "ctcpb_kernels.h"

namespace ctcpb {

namespace {
static int grid_for(long long items_per_warp_units, int warps_per_block) {
  long long blocks = (items_per_warp_units + warps_per_block - 1) / warps_per_block;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}
}  // namespace

// Warps (one 16-byte aligned row buffer each) that fit 200 KB of shared memory
// (the fused launch; the stand-alone pre-pass takes what the device allows).
int rank_tma_warps(int V) {
  int w = (int)((200u * 1024u) / rank_tma_per_warp(V));
  return w > 16 ? 16 : w;
}

// Records for the decode: item (b, s) ranks the frame of row b's step s.
// mode 0 (offline): frame sel[b][s], s < nsel[b].
// mode 1 (streaming): chunk row tile_start + s, s < frames of row b in the tile.
__global__ void __launch_bounds__(256) k_prepass(View st, const float* __restrict__ lp, long long sb, long long stt,
                                                 int mode, const int* __restrict__ nframes, int chunk_T,
                                                 int tile_start, int tile_len) {
  __shared__ u64 bufs[8][kRankCap];
  const Layout& Ly = st.lay;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const long long gw = (long long)blockIdx.x * nw + wid;
  const long long tw = (long long)gridDim.x * nw;
  const long long items = (long long)Ly.B * tile_len;
  for (long long it = gw; it < items; it += tw) {
    const int b = (int)(it % Ly.B);
    const int s = (int)(it / Ly.B);
    const float* row;
    if (mode != 1) {
      if (s >= st.nsel()[b]) continue;
      const int t = st.sel()[(size_t)b * Ly.T_sel + s];
      row = lp + (long long)b * sb + (long long)t * stt;
    } else {
      int nf = nframes ? nframes[b] : chunk_T;
      nf = nf < 0 ? 0 : (nf > chunk_T ? chunk_T : nf);
      if (tile_start + s >= nf) continue;
      row = lp + (long long)b * sb + (long long)(tile_start + s) * stt;
    }
    char* r = st.rec(b, s);
    RecHdr* h = (RecHdr*)r;
    if (lane == 0) h->t = mode != 1 ? st.sel()[(size_t)b * Ly.T_sel + s] : tile_start + s;
    const BoostTab bt{Ly.hcap > 0 ? st.bkey(b) : nullptr, Ly.hcap > 0 ? st.bval(b) : nullptr, Ly.hcap - 1};
    rank_row(row, Ly.V, Ly.blank, Ly.L, bufs[wid], lane, rec_ids(r), rec_lps(r, Ly.Lpad), &h->cnt, &h->lpb,
             &h->front_lp, &h->front_id, bt);
  }
}

// Stand-alone pre-pass over R rows (the ctcpb_topk_prepass entry point).
__global__ void __launch_bounds__(256) k_prepass_rows(const float* __restrict__ lp, long long stride_r, int R, int V,
                                                      int blank, int L, int* ids, float* lps, int* cnt, float* lpb,
                                                      float* flp, int* fid) {
  __shared__ u64 bufs[8][kRankCap];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  for (long long r = (long long)blockIdx.x * nw + wid; r < R; r += (long long)gridDim.x * nw) {
    rank_row(lp + r * stride_r, V, blank, L, bufs[wid], lane, ids + r * L, lps + r * L, cnt + r, lpb + r, flp + r,
             fid + r);
  }
}


namespace {

template <class Items>
__global__ void __launch_bounds__(512, 1) k_rank_tma(Items items, int V, int blank, int L, u32* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  rank_tma_body_e<Items, 2>(items, V, blank, L, status, smem, blockIdx.x, gridDim.x, blockDim.x >> 5);
}

// Lists of 64..255 labels: a larger threshold pool (E maxima per lane) and up
// to 8 warps a block, so the registers are not capped at 128.
template <class Items, int E>
__global__ void __launch_bounds__(256, 1) k_rank_tma_big(Items items, int V, int blank, int L, u32* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  rank_tma_body_e<Items, E>(items, V, blank, L, status, smem, blockIdx.x, gridDim.x, blockDim.x >> 5);
}


template <class Items>
cudaError_t launch_rank_tma(const Items& items, long long nitems, int V, int blank, int L, u32* status,
                            cudaStream_t s) {
  const int E = L + 1 <= 64 ? 2 : (L + 1 <= 128 ? 4 : (L + 1 <= 256 ? 8 : 16));
  int wpb = rank_tma_warps(V);
  {  // as many row buffers as the device's largest block allocation holds
    int dev = 0, maxsm = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess) {
      const int w = (int)((size_t)maxsm / rank_tma_per_warp(V));
      if (w > wpb) wpb = w > 16 ? 16 : w;
    }
  }
  if (E > 2 && wpb > 8) wpb = 8;
  const size_t smem = rank_tma_per_warp(V) * wpb;
  const void* fn = E == 2    ? (const void*)k_rank_tma<Items>
                  : E == 4  ? (const void*)k_rank_tma_big<Items, 4>
                  : E == 8  ? (const void*)k_rank_tma_big<Items, 8>
                            : (const void*)k_rank_tma_big<Items, 16>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (nitems + wpb - 1) / wpb;
  if (blocks > sms) blocks = sms;
  if (blocks < 1) blocks = 1;
  if (E == 2)
    k_rank_tma<Items><<<(int)blocks, 32 * wpb, smem, s>>>(items, V, blank, L, status);
  else if (E == 4)
    k_rank_tma_big<Items, 4><<<(int)blocks, 32 * wpb, smem, s>>>(items, V, blank, L, status);
  else if (E == 8)
    k_rank_tma_big<Items, 8><<<(int)blocks, 32 * wpb, smem, s>>>(items, V, blank, L, status);
  else
    k_rank_tma_big<Items, 16><<<(int)blocks, 32 * wpb, smem, s>>>(items, V, blank, L, status);
  return cudaGetLastError();
}

}  // namespace

// The staged path needs 16-byte aligned rows of a multiple of 4 labels, one of
// which fits a warp's share of shared memory, and lists of at most 511 labels.
bool rank_tma_ok(const float* lp, long long s1, long long s2, int V, int L) {
  return ((uintptr_t)lp & 15u) == 0 && (s1 & 3) == 0 && (s2 & 3) == 0 && (V & 3) == 0 && V >= 4 &&
         L + 1 <= 512 && rank_tma_warps(V) >= 1;
}

cudaError_t launch_prepass_tma(const View& st, const float* lp, long long sb, long long stt, int mode,
                               const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  RecItems items{st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len};
  return launch_rank_tma(items, (long long)st.lay.B * tile_len, st.lay.V, st.lay.blank, st.lay.L,
                         &st.hdr()->status, s);
}

cudaError_t launch_prepass_rows_tma(const float* lp, long long stride_r, int R, int V, int blank, int L, int* ids,
                                    float* lps, int* cnt, float* lpb, float* flp, int* fid, cudaStream_t s) {
  RowItems items{lp, stride_r, R, L, ids, cnt, fid, lps, lpb, flp};
  return launch_rank_tma(items, (long long)R, V, blank, L, nullptr, s);
}

static cudaError_t launch_prepass_plain(const View& st, const float* lp, long long sb, long long stt, int mode,
                           const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  long long items = (long long)st.lay.B * tile_len;
  if (items == 0) return cudaSuccess;
  k_prepass<<<grid_for(items, 8), 256, 0, s>>>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len);
  return cudaGetLastError();
}

static cudaError_t launch_prepass_rows_plain(const float* lp, long long stride_r, int R, int V, int blank, int L, int* ids,
                                float* lps, int* cnt, float* lpb, float* flp, int* fid, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  k_prepass_rows<<<grid_for(R, 8), 256, 0, s>>>(lp, stride_r, R, V, blank, L, ids, lps, cnt, lpb, flp, fid);
  return cudaGetLastError();
}


cudaError_t launch_prepass(const View& st, const float* lp, long long sb, long long stt, int mode,
                           const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  if ((long long)st.lay.B * tile_len == 0) return cudaSuccess;
  if (rank_tma_ok(lp, sb, stt, st.lay.V, st.lay.L))
    return launch_prepass_tma(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
  return launch_prepass_plain(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
}

cudaError_t launch_prepass_rows(const float* lp, long long stride_r, int R, int V, int blank, int L, int* ids,
                                float* lps, int* cnt, float* lpb, float* flp, int* fid, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  if (rank_tma_ok(lp, stride_r, 0, V, L))
    return launch_prepass_rows_tma(lp, stride_r, R, V, blank, L, ids, lps, cnt, lpb, flp, fid, s);
  return launch_prepass_rows_plain(lp, stride_r, R, V, blank, L, ids, lps, cnt, lpb, flp, fid, s);
}

}  // namespace ctcpb
