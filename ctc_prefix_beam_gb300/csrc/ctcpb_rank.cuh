// Vocabulary pre-pass building blocks ("GPU CTC Prefix Beam Search Decoder",
// section 3.4.7), shared by the stand-alone pre-pass kernels and the fused
// pre-pass + step kernel: the plain per-warp ranking and the staged ranking
// of one shared-memory row per warp.
#pragma once

#include "ctcpb_async.cuh"
#include "ctcpb_internal.cuh"
#include "ctcpb_sort.cuh"

namespace ctcpb {
namespace {

#define FULL 0xffffffffu
template <int NT>
__device__ __forceinline__ void gsync() {
  if (NT == 32)
    __syncwarp();
  else
    __syncthreads();
}
template <int NT>
__device__ void bitonic_desc(u64* a, int P, int tid) {
  for (int k = 2; k <= P; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += NT) {
        int ixj = i ^ j;
        if (ixj > i) {
          u64 x = a[i], y = a[ixj];
          bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) {
            a[i] = y;
            a[ixj] = x;
          }
        }
      }
      gsync<NT>();
    }
}
__device__ __forceinline__ u64 warp_max_u64(u64 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    u64 w = __shfl_xor_sync(FULL, v, o);
    v = w > v ? w : v;
  }
  return v;
}
__device__ __forceinline__ int pow2_at_least(int n, int lo) {
  int p = lo;
  while (p < n) p <<= 1;
  return p;
}
// ---- plain per-warp ranking (any alignment, any list length)
// Rank one frame row by one warp: the first L live non-blank labels by
// (lp desc, id asc), the blank log-prob and the label after the list.
//
// Exact top-(L+1) selection:
//   1. each lane keeps its top-2 label keys over labels lane, lane+32, ...;
//   2. the (L+1)-th largest of these 64 keys is a lower bound tau of the
//      (L+1)-th largest key of the row (they are distinct labels);
//   3. every label with key >= tau is compacted into shared memory and the
//      compacted set is sorted; it contains the top L+1 by construction;
//   4. if the compacted set would overflow `lcap`, the warp falls back to
//      L+1 rounds of "largest key below the previous one".
constexpr int kRankCap = 512;  // shared keys per ranking warp

// A row's label-boost table (keys null: no boosting).
struct BoostTab {
  const int* keys;
  const float* vals;
  int hmask;
};

// Label c's ranking key, by its log-prob as emitted (boosted when bt.keys).
__device__ __forceinline__ u64 label_key_at(const float* __restrict__ row, int c, int V, int blank,
                                            const BoostTab& bt) {
  if (c >= V || c == blank) return 0ull;
  float v = rdlp(row[c]);
  if (bt.keys) v = dadd(v, boost_of(bt.keys, bt.vals, bt.hmask, c));
  return v > CTCPB_NEG ? lab_key(v, c) : 0ull;
}

__device__ void rank_row(const float* __restrict__ row, int V, int blank, int L, u64* buf, int lane,
                         int* o_ids, float* o_lps, int* o_cnt, float* o_lpb, float* o_flp, int* o_fid,
                         const BoostTab& bt = BoostTab{nullptr, nullptr, 0}) {
  const int K = L + 1;
  u64 tau = 0ull;
  if (K <= 64) {
    u64 k1 = 0ull, k2 = 0ull;
    for (int c = lane; c < V; c += 32) {
      u64 key = label_key_at(row, c, V, blank, bt);
      if (key > k2) {
        if (key > k1) {
          k2 = k1;
          k1 = key;
        } else {
          k2 = key;
        }
      }
    }
    buf[lane] = k1;
    buf[lane + 32] = k2;
    __syncwarp();
    bitonic_desc<32>(buf, 64, lane);
    tau = buf[K - 1];
    __syncwarp();
  }
  int n = 0;
  bool ovf = false;
  for (int c0 = 0; c0 < V; c0 += 32) {
    const int c = c0 + lane;
    u64 key = label_key_at(row, c, V, blank, bt);
    bool take = key != 0ull && key >= tau;
    unsigned m = __ballot_sync(FULL, take);
    int tot = __popc(m);
    if (n + tot > kRankCap) {
      ovf = true;
      break;
    }
    if (take) buf[n + __popc(m & ((1u << lane) - 1u))] = key;
    n += tot;
  }
  __syncwarp();
  if (!ovf) {
    const int P = pow2_at_least(n, 32);
    for (int i = n + lane; i < P; i += 32) buf[i] = 0ull;
    __syncwarp();
    bitonic_desc<32>(buf, P, lane);
  } else {
    u64 prev = ~0ull;
    n = 0;
    for (int r = 0; r < K; ++r) {
      u64 best = 0ull;
      for (int c = lane; c < V; c += 32) {
        u64 key = label_key_at(row, c, V, blank, bt);
        if (key < prev && key > best) best = key;
      }
      best = warp_max_u64(best);
      if (best == 0ull) break;
      if (lane == 0) buf[r] = best;
      prev = best;
      n = r + 1;
    }
    __syncwarp();
  }
  const int cnt = n < L ? n : L;
  for (int i = lane; i < L; i += 32) {
    if (i < cnt) {
      u64 kk = buf[i];
      o_ids[i] = (int)(~(u32)kk);
      o_lps[i] = fkey_inv((u32)(kk >> 32));
    } else {
      o_ids[i] = -1;
      o_lps[i] = CTCPB_NEG;
    }
  }
  if (lane == 0) {
    *o_cnt = cnt;
    *o_lpb = rdlp(row[blank]);
    if (n > L) {
      *o_flp = fkey_inv((u32)(buf[L] >> 32));
      *o_fid = (int)(~(u32)buf[L]);
    } else {
      *o_flp = CTCPB_NEG;
      *o_fid = -1;
    }
  }
  __syncwarp();
}

#define RFULL 0xffffffffu
constexpr int kCandCap = 512;          // compacted labels per warp (= rank_row's buffer)
// Where one ranked row goes.
struct RankDst {
  int* ids;
  float* lps;
  int* cnt;
  float* lpb;
  float* flp;
  int* fid;
  int* tout;
  int t;
  u32* flag;  // set (release) once the record is complete; null: none
  BoostTab boost;  // the frame's row's label boosts (keys null: none)
};

// Items of the decode: (row b, step s), frame-major, records in the state.
struct RecItems {
  View st;
  const float* lp;
  long long sb, stt;
  int mode;
  const int* nframes;
  int chunk_T, tile_start, tile_len;
  u32* flags;  // per-record ready flags [B][tile] when a consumer runs concurrently, else null
  __device__ long long count() const { return (long long)st.lay.B * tile_len; }
  // is item `it` a decoded frame? then its row and frame index
  __device__ bool probe(long long it, const float** row, int* t) const {
    const int B = st.lay.B;
    const int b = (int)(it % B), s = (int)(it / B);
    if (mode != 1) {  // offline (frame index) or masked streaming (chunk row), from the selection
      if (s >= st.nsel()[b]) return false;
      *t = st.sel()[(size_t)b * st.lay.T_sel + s];
    } else {
      int nf = nframes ? nframes[b] : chunk_T;
      nf = nf < 0 ? 0 : (nf > chunk_T ? chunk_T : nf);
      if (tile_start + s >= nf) return false;
      *t = tile_start + s;
    }
    *row = lp + (long long)b * sb + (long long)(*t) * stt;
    return true;
  }
  __device__ RankDst dst(long long it, int t) const {
    const int B = st.lay.B;
    const int b = (int)(it % B), s = (int)(it / B);
    char* r = st.rec(b, s);
    RecHdr* h = (RecHdr*)r;
    const bool bo = st.lay.hcap > 0;
    return RankDst{rec_ids(r),  rec_lps(r, st.lay.Lpad), &h->cnt, &h->lpb, &h->front_lp, &h->front_id, &h->t, t,
                   flags ? flags + (size_t)b * st.lay.tile + s : nullptr,
                   BoostTab{bo ? st.bkey(b) : nullptr, bo ? st.bval(b) : nullptr, st.lay.hcap - 1}};
  }
};

// Independent rows (the ctcpb_topk_prepass entry point).
struct RowItems {
  const float* lp;
  long long stride;
  int R, L;
  int *ids, *cnt, *fid;
  float *lps, *lpb, *flp;
  __device__ long long count() const { return R; }
  __device__ bool probe(long long r, const float** row, int* t) const {
    *row = lp + r * stride;
    *t = 0;
    return true;
  }
  __device__ RankDst dst(long long r, int t) const {
    return RankDst{ids + r * L, lps + r * L, cnt + r, lpb + r, flp + r, fid + r, nullptr, t, nullptr,
                   BoostTab{nullptr, nullptr, 0}};
  }
};

// Passes 1-3 over one staged row (all lanes): compacts every label that can
// be in the top L+1 into `cand`; returns their count, or -1 when they
// overflow the buffer.  `row`: 16-byte aligned shared memory, V % 4 == 0, the
// blank already replaced by -inf.
// Passes 1-2: tau = the K-th largest of a pool of 32*E label maxima, one per
// disjoint label subset (E = 2: the x,y and z,w halves of each lane's float4
// slices; 4: each component; 8: each component of the even and of the odd
// rounds; 16: each component of rounds 0, 1, 2, 3 mod 4), so at least K
// labels score >= tau and the top K all do.  K <= 32*E.
template <int E>
__device__ __forceinline__ float pool_tau(const float4* __restrict__ r4, int V4, int K, int lane) {
  float m[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) m[e] = -INFINITY;
  if (E == 16) {
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int q = lane; q < V4; q += 128) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 x = q + 32 * u < V4 ? r4[q + 32 * u] : ninf;
        m[4 * u] = fmaxf(m[4 * u], x.x);
        m[4 * u + 1] = fmaxf(m[4 * u + 1], x.y);
        m[4 * u + 2] = fmaxf(m[4 * u + 2], x.z);
        m[4 * u + 3] = fmaxf(m[4 * u + 3], x.w);
      }
    }
  } else if (E == 8) {
#pragma unroll 2
    for (int q = lane; q < V4; q += 64) {
      const float4 x = r4[q];
      const float4 y = q + 32 < V4 ? r4[q + 32] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      m[0] = fmaxf(m[0], x.x); m[1] = fmaxf(m[1], x.y); m[2] = fmaxf(m[2], x.z); m[3] = fmaxf(m[3], x.w);
      m[4] = fmaxf(m[4], y.x); m[5] = fmaxf(m[5], y.y); m[6] = fmaxf(m[6], y.z); m[7] = fmaxf(m[7], y.w);
    }
  } else {
#pragma unroll 4
    for (int q = lane; q < V4; q += 32) {
      const float4 x = r4[q];
      m[0] = fmaxf(m[0], x.x); m[1] = fmaxf(m[1], x.y); m[2] = fmaxf(m[2], x.z); m[3] = fmaxf(m[3], x.w);
    }
    if (E == 2) {
      m[0] = fmaxf(m[0], m[1]);
      m[1] = fmaxf(m[2], m[3]);
    }
  }
  u32 pool[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float v = m[e] + 0.0f;
    pool[e] = v > CTCPB_NEG ? fkey(v) : 0u;
  }
  warp_sort_desc<E>(pool, lane);
  u32 pk = pool[0];
#pragma unroll
  for (int e = 1; e < E; ++e)
    if (((K - 1) >> 5) == e) pk = pool[e];
  const u32 kth = __shfl_sync(RFULL, pk, (K - 1) & 31);
  return kth != 0u ? fkey_inv(kth) : -FLT_MAX;
}

template <int E>
__device__ int rank_gather(const float* __restrict__ row, int V, int L, u64* cand, int lane) {
  const int K = L + 1;
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int V4 = V >> 2;
  const float tauf = pool_tau<E>(r4, V4, K, lane);
  // 3. every live label >= tau, four float4 per lane per round, compacted by
  // an exclusive scan of the lanes' hit counts
  int n = 0;
  for (int q0 = 0; q0 < V4; q0 += 128) {
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int qq = q0 + 32 * u + lane;
      x[u] = qq < V4 ? r4[qq] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    u32 hit = 0u;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      hit |= (u32)(x[u].x >= tauf && x[u].x > CTCPB_NEG) << (4 * u);
      hit |= (u32)(x[u].y >= tauf && x[u].y > CTCPB_NEG) << (4 * u + 1);
      hit |= (u32)(x[u].z >= tauf && x[u].z > CTCPB_NEG) << (4 * u + 2);
      hit |= (u32)(x[u].w >= tauf && x[u].w > CTCPB_NEG) << (4 * u + 3);
    }
    if (!__any_sync(RFULL, hit != 0u)) continue;
    const int cntl = __popc(hit);
    int incl = cntl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(RFULL, incl, o);
      if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(RFULL, incl, 31);
    if (n + total > kCandCap) return -1;
    int pos = n + incl - cntl;
    if (hit != 0u) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int b = (q0 + 32 * u + lane) << 2;
        if (hit & (1u << (4 * u))) cand[pos++] = lab_key(x[u].x + 0.0f, b);
        if (hit & (2u << (4 * u))) cand[pos++] = lab_key(x[u].y + 0.0f, b + 1);
        if (hit & (4u << (4 * u))) cand[pos++] = lab_key(x[u].z + 0.0f, b + 2);
        if (hit & (8u << (4 * u))) cand[pos++] = lab_key(x[u].w + 0.0f, b + 3);
      }
    }
    n += total;
  }
  __syncwarp();
  return n;
}

// Write rank r's label (r < L: list, r == L: front).
__device__ __forceinline__ void put_ranked(u64 key, int r, int L, const RankDst& d) {
  if (key == 0ull) return;
  if (r < L) {
    d.ids[r] = (int)(~(u32)key);
    d.lps[r] = fkey_inv((u32)(key >> 32));
  } else if (r == L) {
    *d.fid = (int)(~(u32)key);
    *d.flp = fkey_inv((u32)(key >> 32));
  }
}

// Pass 4 (all lanes): rank the n compacted labels and write the row's list.
template <int E>
__device__ void rank_finish(const u64* cand, int n, int L, float lpb, int lane, const RankDst& d) {
  const int cnt = n < L ? n : L;
  if (n <= 64) {
    u64 v[2] = {lane < n ? cand[lane] : 0ull, lane + 32 < n ? cand[lane + 32] : 0ull};
    warp_sort_desc<2>(v, lane);
    put_ranked(v[0], lane, L, d);
    put_ranked(v[1], lane + 32, L, d);
  } else if (n <= 128) {
    u64 v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = lane + 32 * e < n ? cand[lane + 32 * e] : 0ull;
    warp_sort_desc<4>(v, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) put_ranked(v[e], lane + 32 * e, L, d);
  } else if (E >= 8 && n <= 256) {
    u64 v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = lane + 32 * e < n ? cand[lane + 32 * e] : 0ull;
    warp_sort_desc<8>(v, lane);
#pragma unroll
    for (int e = 0; e < 8; ++e) put_ranked(v[e], lane + 32 * e, L, d);
  } else if (E >= 16 && n <= 512) {
    u64 v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = lane + 32 * e < n ? cand[lane + 32 * e] : 0ull;
    warp_sort_desc<16>(v, lane);
#pragma unroll
    for (int e = 0; e < 16; ++e) put_ranked(v[e], lane + 32 * e, L, d);
  } else {
    for (int e = lane; e < n; e += 32) {
      const u64 me = cand[e];
      int rk = 0, rk2 = 0;
      int j = 0;
      for (; j + 1 < n; j += 2) {
        rk += cand[j] > me;
        rk2 += cand[j + 1] > me;
      }
      if (j < n) rk += cand[j] > me;
      put_ranked(me, rk + rk2, L, d);
    }
  }
  for (int i = cnt + lane; i < L; i += 32) {
    d.ids[i] = -1;
    d.lps[i] = CTCPB_NEG;
  }
  if (lane == 0) {
    *d.cnt = cnt;
    *d.lpb = lpb;
    if (n <= L) {
      *d.flp = CTCPB_NEG;
      *d.fid = -1;
    }
    if (d.tout) *d.tout = d.t;
  }
  __syncwarp();
}

// The lean ranking of one staged row for lists of K = L + 1 <= 64 labels
// (used up to kLeanK)
// (all lanes).  Every step is a short, mostly independent instruction stream,
// so a warp ranks a row in a few hundred cycles:
//   1. each lane takes the maxima of two disjoint halves of its labels (the
//      x,y and the z,w components of its float4 slices): 64 maxima of 64
//      distinct labels;
//   2. tau = the K-th largest of them, by counting: every lane reads the 64
//      maxima from shared memory (broadcast) and keeps its maxima that have at
//      least K maxima >= them; the largest such is tau.  At least K labels
//      score >= tau, so the top K all do;
//   3. each lane tests its float4 slices by their maxima against tau (one
//      compare each, no branch) into a bit mask, then reads the few slices
//      with a hit again and appends their labels >= tau to its own column of
//      `cand` (at most kLaneHits each, no cross-lane traffic); one scan packs
//      the columns into a contiguous list;
//   4. each packed key's rank = how many packed keys are larger (keys are
//      distinct: they hold the label); ranks below L fill the list, rank L is
//      the front.
// Returns false, having written nothing, when a lane collects more than
// kLaneHits labels (near-constant rows); the caller then ranks the row the
// general way.
constexpr int kLaneHits = 8;
// The lean ranking serves lists of K = L + 1 <= 32 labels; with longer lists
// more labels pass tau and counting every pair costs more than a sort.
constexpr int kLeanK = 32;
template <class Release>
__device__ __forceinline__ bool rank_lean(const float* __restrict__ row, int V, int L, u64* cand, float lpb,
                                          int lane, const RankDst& d, Release&& release_row) {
  const int K = L + 1;
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int V4 = V >> 2;
  // 1. two maxima per lane, four independent chains
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
  int q = lane;
  for (; q + 32 < V4; q += 64) {
    const float4 x = r4[q], y = r4[q + 32];
    m0 = fmaxf(m0, fmaxf(x.x, x.y));
    m1 = fmaxf(m1, fmaxf(x.z, x.w));
    m2 = fmaxf(m2, fmaxf(y.x, y.y));
    m3 = fmaxf(m3, fmaxf(y.z, y.w));
  }
  if (q < V4) {
    const float4 x = r4[q];
    m0 = fmaxf(m0, fmaxf(x.x, x.y));
    m1 = fmaxf(m1, fmaxf(x.z, x.w));
  }
  const float a = fmaxf(m0, m2) + 0.0f, b = fmaxf(m1, m3) + 0.0f;
  const u32 ka = a > CTCPB_NEG ? fkey(a) : 0u, kb = b > CTCPB_NEG ? fkey(b) : 0u;
  // 2. tau by counting (the pool lives in the packed-list half of cand)
  u32* pool = reinterpret_cast<u32*>(cand + 32 * kLaneHits);
  pool[lane] = ka;
  pool[32 + lane] = kb;
  __syncwarp();
  int ga0 = 0, ga1 = 0, gb0 = 0, gb1 = 0;
  const uint4* p4 = reinterpret_cast<const uint4*>(pool);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint4 v = p4[i];
    ga0 += (int)(v.x >= ka) + (int)(v.y >= ka);
    ga1 += (int)(v.z >= ka) + (int)(v.w >= ka);
    gb0 += (int)(v.x >= kb) + (int)(v.y >= kb);
    gb1 += (int)(v.z >= kb) + (int)(v.w >= kb);
  }
  u32 mine = 0u;
  if (ka != 0u && ga0 + ga1 >= K) mine = ka;
  if (kb != 0u && gb0 + gb1 >= K && kb > mine) mine = kb;
  const u32 tk = __reduce_max_sync(RFULL, mine);
  const float tauf = tk != 0u ? fkey_inv(tk) : -FLT_MAX;  // fewer than K live maxima: every live label
  // 3. this lane's labels >= tau into its column of cand
  int h = 0;
  const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  // a label is taken iff v >= t2: t2 = tau, or the least float above NEG when
  // tau is NEG (fewer than K live maxima), so dead labels and NaN never pass
  const float t2 = fmaxf(tauf, __int_as_float(0xff7ffffe));
  // Each round tests four of the lane's float4 slices by their maxima (one
  // compare each) into a bit mask; every eighth round (and the last) the few
  // slices with a hit are read again and their labels taken.
  const int nrounds = (V4 + 127) >> 7;
  u32 fm = 0u;
  int r0 = 0;  // round of mask bit 0
  for (int r = 0; r < nrounds; ++r) {
    const int q0 = lane + 128 * r;
    float4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = q0 + 32 * u < V4 ? r4[q0 + 32 * u] : ninf;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      fm |= (u32)(fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)) >= t2) << (4 * (r - r0) + u);
    if (r - r0 == 7 || r == nrounds - 1) {
      for (; fm; fm &= fm - 1u) {
        const int bit = __ffs(fm) - 1;
        const int q = lane + 128 * (r0 + (bit >> 2)) + 32 * (bit & 3);
        const float4 y = r4[q];
        const float v[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          if (v[cc] >= t2) {
            if (h < kLaneHits) cand[32 * h + lane] = lab_key(v[cc] + 0.0f, 4 * q + cc);
            ++h;
          }
      }
      r0 = r + 1;
    }
  }
  if (__any_sync(RFULL, h > kLaneHits)) return false;
  release_row();  // the row buffer is not read again: its next row may start arriving
  int incl = h;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(RFULL, incl, o);
    if (lane >= o) incl += y;
  }
  const int n = __shfl_sync(RFULL, incl, 31);
  u64* packed = cand + 32 * kLaneHits;
  __syncwarp();  // the pool is read by every lane before it is overwritten
  for (int j = 0, pos = incl - h; j < h; ++j, ++pos) packed[pos] = cand[32 * j + lane];
  __syncwarp();
  // 4. rank by counting; ranks 0..L-1 form the list, rank L is the front
  for (int i = lane; i < n; i += 32) {
    const u64 me = packed[i];
    int r0 = 0, r1 = 0;
    const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(packed);
    int j = 0;
    for (; j + 1 < n; j += 2) {
      const ulonglong2 v = k2[j >> 1];
      r0 += (int)(v.x > me);
      r1 += (int)(v.y > me);
    }
    if (j < n) r0 += (int)(packed[j] > me);
    put_ranked(me, r0 + r1, L, d);
  }
  const int cnt = n < L ? n : L;
  for (int i = cnt + lane; i < L; i += 32) {
    d.ids[i] = -1;
    d.lps[i] = CTCPB_NEG;
  }
  if (lane == 0) {
    *d.cnt = cnt;
    *d.lpb = lpb;
    if (n <= L) {
      *d.flp = CTCPB_NEG;
      *d.fid = -1;
    }
    if (d.tout) *d.tout = d.t;
  }
  __syncwarp();
  return true;
}

__host__ __device__ inline size_t rank_tma_per_warp(int V) {
  return align_up((size_t)V * 4, 128) + (size_t)kCandCap * 8 + 16;
}

// The ranking of one block: warps 0..nwb-1 each own a row buffer in `smem`;
// (vblock, nvblocks) is this block's place among the blocks that rank.  The
// next row's bulk copy is issued as soon as the current row's passes have read
// the buffer, so it overlaps pass 4.
template <class Items, int E>
__device__ __forceinline__ void rank_tma_body_e(const Items& items, int V, int blank, int L, u32* status,
                                                unsigned char* smem, int vblock, int nvblocks, int nwb) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (wid >= nwb) return;
  const size_t per_warp = align_up((size_t)V * 4, 128) + (size_t)kCandCap * 8 + 16;
  unsigned char* base = smem + per_warp * wid;
  float* buf = reinterpret_cast<float*>(base);
  u64* cand = reinterpret_cast<u64*>(base + align_up((size_t)V * 4, 128));
  u64* bar = cand + kCandCap;
  if (lane == 0) {
    mbar_init(bar);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();
  const unsigned bytes = (unsigned)V * 4u;
  const long long total = items.count();
  const long long stride = (long long)nvblocks * nwb;
  unsigned phase = 0u;
  // This warp's items are it0, it0 + stride, ...; lane j resolves the j-th of
  // the next 32 in parallel, so finding the next row costs no dependent loads.
  long long batch = (long long)vblock * nwb + wid;
  long long my_it = 0;
  const float* my_row = nullptr;
  int my_t = 0;
  unsigned vmask = 0u;
  auto refill = [&]() {
    while (vmask == 0u && batch < total) {
      my_it = batch + (long long)lane * stride;
      const bool ok = my_it < total && items.probe(my_it, &my_row, &my_t);
      vmask = __ballot_sync(RFULL, ok);
      batch += 32 * stride;
    }
  };
  // next valid item (all lanes): returns false when the warp's items are done
  auto advance = [&](long long* it, const float** row, int* t) -> bool {
    refill();
    if (vmask == 0u) return false;
    const int j = __ffs(vmask) - 1;
    vmask &= vmask - 1u;
    *it = __shfl_sync(RFULL, my_it, j);
    *row = reinterpret_cast<const float*>(__shfl_sync(RFULL, reinterpret_cast<unsigned long long>(my_row), j));
    *t = __shfl_sync(RFULL, my_t, j);
    return true;
  };
  long long it = 0;
  const float* row = nullptr;
  int t = 0;
  bool have = advance(&it, &row, &t);
  if (have && lane == 0) {
    mbar_arrive_tx(bar, bytes);
    bulk_g2s(buf, row, bytes, bar);
  }
  while (have) {
    if (!mbar_wait(bar, phase)) {
      if (lane == 0 && status) atomicOr(status, CTCPB_DEV_TIMEOUT);
      // A warp has one bulk copy in flight at most (the next row's is issued
      // only after this one is read), and it issues no other after a timeout.
      // Before the warp retires, that copy must land in its shared memory:
      // wait for it again, each wait bounded, the last giving up for good.
      for (int i = 0; i < kExitWaits && !mbar_wait(bar, phase); ++i) {
      }
      return;
    }
    phase ^= 1u;
    const RankDst dc = items.dst(it, t);
    const float rawb = buf[blank];
    const float lpb = rdlp(rawb);
    __syncwarp();
    if (lane == 0) buf[blank] = -INFINITY;  // the blank is not a label of the list
    if (dc.boost.keys) {  // rank the labels as emitted: add the row's bonuses (never the blank's)
      for (int i = lane; i <= dc.boost.hmask; i += 32) {
        const int c = dc.boost.keys[i];
        if (c >= 0) buf[c] = dadd(rdlp(buf[c]), dc.boost.vals[i]);
      }
    }
    __syncwarp();
    // the next row's bulk copy, issued once every lane is done reading the buffer
    bool issued = false;
    auto next_copy = [&]() {
      __syncwarp();
      have = advance(&it, &row, &t);
      if (have && lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        mbar_arrive_tx(bar, bytes);
        bulk_g2s(buf, row, bytes, bar);
      }
      issued = true;
    };
    // lists up to 31 labels: the lean ranking, which issues the next copy as
    // soon as its passes over the row are done and has written the record when
    // it succeeds; otherwise (and for longer lists) the general one
    const bool lean = E == 2 && L + 1 <= kLeanK && rank_lean(buf, V, L, cand, lpb, lane, dc, next_copy);
    const int n = lean ? 0 : rank_gather<E>(buf, V, L, cand, lane);
    if (n < 0) {  // constant or near-constant row: plain ranking of the staged row
      if (lane == 0) buf[blank] = rawb;
      __syncwarp();
      rank_row(buf, V, blank, L, cand, lane, dc.ids, dc.lps, dc.cnt, dc.lpb, dc.flp, dc.fid);
      if (dc.tout && lane == 0) *dc.tout = dc.t;
    }
    if (!issued) next_copy();
    if (!lean && n >= 0) rank_finish<E>(cand, n, L, lpb, lane, dc);
    if (dc.flag) {  // publish the record: every lane's stores, then the flag
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release_u32(dc.flag, 1u);
    }
    __syncwarp();
  }
}


// The staged ranking with the threshold pool sized for K = L + 1 <= 512.
template <class Items>
__device__ __forceinline__ void rank_tma_body(const Items& items, int V, int blank, int L, u32* status,
                                              unsigned char* smem, int vblock, int nvblocks, int nwb) {
  if (L + 1 <= 64)
    rank_tma_body_e<Items, 2>(items, V, blank, L, status, smem, vblock, nvblocks, nwb);
  else if (L + 1 <= 128)
    rank_tma_body_e<Items, 4>(items, V, blank, L, status, smem, vblock, nvblocks, nwb);
  else if (L + 1 <= 256)
    rank_tma_body_e<Items, 8>(items, V, blank, L, status, smem, vblock, nvblocks, nwb);
  else
    rank_tma_body_e<Items, 16>(items, V, blank, L, status, smem, vblock, nvblocks, nwb);
}

// The same for lists of at most 127 labels (the fused pre-pass + steps launch).
template <class Items>
__device__ __forceinline__ void rank_tma_body_small(const Items& items, int V, int blank, int L, u32* status,
                                                    unsigned char* smem, int vblock, int nvblocks, int nwb) {
  if (L + 1 <= 64)
    rank_tma_body_e<Items, 2>(items, V, blank, L, status, smem, vblock, nvblocks, nwb);
  else
    rank_tma_body_e<Items, 4>(items, V, blank, L, status, smem, vblock, nvblocks, nwb);
}

}  // namespace
}  // namespace ctcpb
