// Warp-per-row decode steps for beam <= 16 (flat token storage).
//
// One warp owns one row for the whole call and keeps the beam in registers:
// lane k holds hypothesis k.  Per step ("GPU CTC Prefix Beam Search Decoder",
// sections 3.3-3.4.6):
//   * blank slot of every hypothesis (3.4.2) with the stay path (3.4.1) and
//     the merge fold of 3.4.3, on lanes 0..nlive-1;
//   * round 1: a staircase of each hypothesis' best listed labels on the other
//     lanes (hypothesis k gets q_k labels, (k+1)(q_k+1) kept small: the best
//     `beam` of a sum of two sorted lists lie under such a staircase), with the
//     repeat path (c = last, pb only) in the slot of its label; the 32
//     candidates are ranked by counting;
//   * the ranking is PROVEN exact when every candidate left out scores below
//     the beam-th kept one: hypothesis k's left-out labels score at most
//     add(lp[next listed label], A_k), its unlisted ones add(front, A_k), so
//     it suffices that `beam` candidates score above the largest such bound;
//   * round 2 (the proof failed): the beam-th kept score tau is a lower bound
//     of the true one, so the candidates that matter are exactly those scoring
//     >= tau; each hypothesis counts its listed labels >= tau (the list is
//     sorted) and, if they fit in 32 lanes, they are ranked again -- exact;
//   * otherwise every candidate >= tau of the frame, unlisted labels included,
//     is collected and sorted (warp_collect_select).
// Prefix merges are tracked through the winners' sources (no token reads):
// if j extends source s and i is s's blank winner, l_j = l_i + last_j; two
// blank winners inherit their sources' relation.  The one remaining case (a
// blank winner whose parent prefix was rebuilt by an extension) is proposed
// by 32-bit prefix hashes and confirmed by comparing stored tokens.
// Tokens: every step appends (source slot, token) per winner to a ring in
// shared memory; every kRing steps (and at the end of the call) the ring is
// materialised into the flat double-buffered rows: each hypothesis' row in the
// other parity = its origin row's prefix + the labels it gained in the window.
// lp[t][last] for step s+1 is gathered at the top of step s over every label
// that can be "last" then (the current lasts and step s's list) into
// shared memory by 4-byte asynchronous copies, so the loads overlap step s.
// Ranked-frame records are loaded from L2 into registers one step ahead
// (header broadcast, list position = lane), their frame index two steps
// ahead for the gather; every register copied at the end of a step was loaded
// a whole step earlier.
#include "ctcpb_async.cuh"
#include "ctcpb_internal.cuh"
#include "ctcpb_kernels.h"
#include "ctcpb_rank.cuh"
#include "ctcpb_sort.cuh"

namespace ctcpb {
namespace {

#define WFULL 0xffffffffu

// Optional per-phase cycle accounting (build with -DCTCPB_PHASE_PROF).
#ifdef CTCPB_PHASE_PROF
#define PHASE_MARK(i)                 \
  do {                                \
    const long long now_ = clock64(); \
    prof[i] += (u64)(now_ - prof_t0); \
    prof_t0 = now_;                   \
  } while (0)
#else
#define PHASE_MARK(i) \
  do {                \
  } while (0)
#endif

constexpr int kRing = 128;            // steps of history between materialisations
constexpr int kWPC = 4;               // rows (warps) per block
constexpr int kGenCap = 512;          // keys of the exhaustive selection
constexpr int kGath = 128;            // gathered log-probs per frame (beam + L <= 98)
constexpr int kMaxRec = 32 + 8 * 68;  // record bytes for lists of L <= 66 labels
constexpr u32 kH32 = 2166136261u;     // prefix hash of the empty prefix
constexpr u32 kGold = 0x9e3779b9u;
constexpr int kBlankWin = 1 << 30;    // flag bit of a blank winner in its slot's gained-label count

struct __align__(16) WarpSmem {
  u64 keys[kGenCap];
  u32 hist[kRing][32];
  char rec1[kMaxRec];  // the current record, copied for the slow selection
  float A[32], bpb[32], bpnb[32], scb[32], rep[32];
  int last[32], len[32];
  int bw[32];
  int fold_i[32], fold_c[32];
  int nfold, nkeys;
  // Both tables are word-major ([word][slot]) so that 32 lanes writing or
  // reading 16-byte words of different slots hit different banks.
  int4 st[2][32];   // bookkeeping of hypothesis k, read by the candidates extending it
  int4 nst[3][32];  // the new hypothesis of slot r, written by the candidate ranked r
  u32 fk[32];       // fold key of slot j: (i << 20 | last_j) when l_j = l_i + last_j
  u32 hk[32];       // prefix hash keys of the extension winners
  float gath[2][kGath];  // lp[t][slot] of the next step, slot = hypothesis or beam + list position
};

struct __align__(16) Tables {
  float fc[kFCoef];             // the coefficients of log(1 + e^-d) (dlse)
  unsigned short qmap[33][32];  // nlive -> lane -> (hyp << 8 | list position), 0xffff: none
  unsigned char qcnt[33][32];  // nlive -> hyp -> listed labels of that hyp in the round-1 set
};
static_assert(sizeof(Tables) % 16 == 0, "tables copy as 16-byte words");


// 32-bit prefix hash (FNV-1a step).  Equal prefixes hash equal; a collision
// only costs an extra exact comparison.
__device__ __forceinline__ u32 h32(u32 h, int c) { return (h ^ (u32)c) * 16777619u; }

__device__ __forceinline__ int wpow2(int n, int lo) {
  int p = lo;
  while (p < n) p <<= 1;
  return p;
}

__device__ __noinline__ void warp_bitonic(u64* a, int P, int lane) {
  for (int k = 2; k <= P; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = lane; i < P; i += 32) {
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
      __syncwarp();
    }
}

// Sort W.keys[0 .. m) descending, m = 32 + W.nkeys (the keys after m, up to
// the next power of two, are zero): in registers up to 128 keys, else in
// shared memory.
__device__ __noinline__ void sort_keys(WarpSmem& W, int m, int lane) {
  if (m <= 64) {
    u64 v[2] = {W.keys[lane], W.keys[32 + lane]};
    warp_sort_desc<2>(v, lane);
    W.keys[lane] = v[0];
    W.keys[32 + lane] = v[1];
  } else if (m <= 128) {
    u64 v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = W.keys[lane + 32 * e];
    warp_sort_desc<4>(v, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) W.keys[lane + 32 * e] = v[e];
  } else {
    const int P = wpow2(m, 64);
    for (int i = m + lane; i < P; i += 32) W.keys[i] = 0ull;
    __syncwarp();
    warp_bitonic(W.keys, P, lane);
  }
  __syncwarp();
}

// Staircase tables for every nlive (compile-time constant): hypothesis k of n
// live ones gets q_k list positions, one per hypothesis first (a frame whose
// best label extends every hypothesis needs each of them in the set), then
// greedily by the smallest (k+1)(q_k+1).
constexpr Tables make_tables() {
  Tables tb{};
  const FCoef f = make_fcoef();
  for (int i = 0; i < kFCoef; ++i) tb.fc[i] = f.c[i];
  for (int n = 0; n <= 32; ++n) {
    unsigned char q[32] = {};
    for (int k = 0; k < 32; ++k) tb.qmap[n][k] = 0xffff;
    int l = n;
    for (int k = 0; k < n && l < 32; ++k, ++l) {
      tb.qmap[n][l] = (unsigned short)(k << 8);
      q[k] = 1;
    }
    for (; l < 32 && n > 0; ++l) {
      int best = 0, bv = 1 << 30;
      for (int k = 0; k < n; ++k) {
        const int v = (k + 1) * (q[k] + 1);
        if (v < bv) {
          bv = v;
          best = k;
        }
      }
      tb.qmap[n][l] = (unsigned short)((best << 8) | q[best]);
      q[best]++;
    }
    for (int k = 0; k < 32; ++k) tb.qcnt[n][k] = q[k];
  }
  return tb;
}
__device__ const Tables g_tables = make_tables();

// Append `key` (if nonzero and >= thr) to the candidate buffer W.keys[32 ..];
// the first 32 entries hold the running best after each compaction.
__device__ __forceinline__ void push_key(WarpSmem& W, u64 key, u64 thr, int lane) {
  const bool take = key != 0ull && key >= thr;
  const unsigned m = __ballot_sync(WFULL, take);
  if (m == 0u) return;
  const int base = W.nkeys;
  if (take) W.keys[32 + base + __popc(m & ((1u << lane) - 1u))] = key;
  __syncwarp();
  if (lane == 0) W.nkeys = base + __popc(m);
  __syncwarp();
  if (base + __popc(m) > kGenCap - 64) {  // compact: keep the best 32 at the front
    warp_bitonic(W.keys, kGenCap, lane);
    for (int i = 32 + lane; i < kGenCap; i += 32) W.keys[i] = 0ull;
    if (lane == 0) W.nkeys = 0;
    __syncwarp();
  }
}

// Every candidate of the step with key >= thr, the frame's unlisted labels
// included when the list cannot bound them, sorted; W.keys[0..beam) holds the
// best.  Returns how many are live, plus 1 << 16 when the frame's unlisted
// labels were scanned.
__device__ __noinline__ int warp_collect_select(WarpSmem& W, const char* rec, int Lpad, int n, int beam, int cap,
                                                int blank, int V, const float* __restrict__ row, int lane, u64 thr,
                                                BoostTab bt) {
  const RecHdr* h = (const RecHdr*)rec;
  const int cnt = h->cnt;
  const int* ids = (const int*)(rec + 32);
  const float* lps = (const float*)(rec + 32 + 4 * Lpad);
  const int nfold = W.nfold;
  int scanned = 0;
  for (int i = lane; i < kGenCap; i += 32) W.keys[i] = 0ull;
  if (lane == 0) W.nkeys = 0;
  __syncwarp();
  // blank slots and repeat candidates, one hypothesis per lane
  for (int k0 = 0; k0 < n; k0 += 32) {
    const int k = k0 + lane;
    u64 kb = 0ull, kr = 0ull;
    if (k < n) {
      if (W.scb[k] > CTCPB_NEG) kb = cand_key(W.scb[k], k, blank);
      bool ok = W.rep[k] > CTCPB_NEG;
      for (int f = 0; f < nfold && ok; ++f) ok = !(W.fold_i[f] == k && W.fold_c[f] == W.last[k]);
      if (ok) kr = cand_key(W.rep[k], k, W.last[k]);
    }
    push_key(W, kb, thr, lane);
    push_key(W, kr, thr, lane);
  }
  // listed labels, one hypothesis at a time, one list position per lane; a
  // hypothesis whose best listed label scores below thr has none to add (the
  // list is sorted)
  const u32 thr_hi = (u32)(thr >> 32);
  const float lp0 = cnt > 0 ? lps[0] : CTCPB_NEG;
  for (int k = 0; k < n; ++k) {
    const int L = W.len[k], lastk = W.last[k];
    const float Ak = W.A[k];
    if (fkey(dadd(lp0, Ak)) < thr_hi) continue;
    for (int p0 = 0; p0 < cnt; p0 += 32) {
      const int p = p0 + lane;
      u64 key = 0ull;
      if (p < cnt && L < cap) {
        const int c = ids[p];
        bool ok = !(L > 0 && c == lastk);
        for (int f = 0; f < nfold && ok; ++f) ok = !(W.fold_i[f] == k && W.fold_c[f] == c);
        const float sc = dadd(lps[p], Ak);
        if (ok && sc > CTCPB_NEG) key = cand_key(sc, k, c);
      }
      push_key(W, key, thr, lane);
    }
  }
  const float front_lp = h->front_lp;
  if (front_lp > CTCPB_NEG) {
    // the running beam-th key so far bounds what an unlisted label must reach
    const int P = wpow2(32 + W.nkeys, 64);
    sort_keys(W, 32 + W.nkeys, lane);
    for (int i = 32 + lane; i < P; i += 32) W.keys[i] = 0ull;
    if (lane == 0) W.nkeys = 0;
    __syncwarp();
    int nw = 0;
    for (int w = 0; w < beam; ++w) nw += W.keys[w] != 0ull;
    const u64 kb = nw == beam ? W.keys[beam - 1] : 0ull;
    if (kb > thr) thr = kb & 0xffffffff00000000ull;
    bool bad = false;
    float amax = CTCPB_NEG;
    if (lane < n && W.len[lane] < cap) {
      const float u = dadd(front_lp, W.A[lane]);
      bad = u > CTCPB_NEG && ((u64)fkey(u) << 32) >= thr;
      amax = W.A[lane];
    }
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(WFULL, amax, o));
    if (__any_sync(WFULL, bad)) {
      scanned = 1;
      const u64 kfront = lab_key(front_lp, h->front_id);
      for (int c0 = 0; c0 < V; c0 += 128) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + 32 * u + lane;
          v[u] = c < V ? rdlp(row[c]) : CTCPB_NEG;
          // labels as emitted: the list ranks them by the boosted log-prob
          if (bt.keys && c < V) v[u] = dadd(v[u], boost_of(bt.keys, bt.vals, bt.hmask, c));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + 32 * u + lane;
          // an unlisted label worth scoring: reaches thr for the best hypothesis
          const bool q = c < V && c != blank && v[u] > CTCPB_NEG && lab_key(v[u], c) <= kfront &&
                         ((u64)fkey(dadd(v[u], amax)) << 32) >= thr;
          for (unsigned m = __ballot_sync(WFULL, q); m; m &= m - 1) {
            const int src = __ffs(m) - 1;
            const int cc = __shfl_sync(WFULL, c, src);
            const float vv = __shfl_sync(WFULL, v[u], src);
            u64 key = 0ull;
            if (lane < n) {
              const int L = W.len[lane];
              bool ok = L < cap && !(L > 0 && cc == W.last[lane]);
              for (int f = 0; f < nfold && ok; ++f) ok = !(W.fold_i[f] == lane && W.fold_c[f] == cc);
              const float sc = dadd(vv, W.A[lane]);
              if (ok && sc > CTCPB_NEG) key = cand_key(sc, lane, cc);
            }
            push_key(W, key, thr, lane);
          }
        }
      }
    }
  }
  sort_keys(W, 32 + W.nkeys, lane);
  int nw = 0;
  for (int w = 0; w < beam; ++w) nw += W.keys[w] != 0ull;
  return nw | (scanned << 16);
}

// Rank of this lane's key among the warp's 32 keys (larger key = better),
// counting the larger score keys; equal scores among the kept ones (two kept
// lanes with one rank) are resolved on the full key (score, source slot, token).
__device__ __forceinline__ int warp_rank(u32 hi, u32 lo, bool live, int beam) {
  // four independent counts, so the compares do not form one dependent chain
  int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    r0 += (int)(__shfl_sync(WFULL, hi, j) > hi);
    r1 += (int)(__shfl_sync(WFULL, hi, j + 1) > hi);
    r2 += (int)(__shfl_sync(WFULL, hi, j + 2) > hi);
    r3 += (int)(__shfl_sync(WFULL, hi, j + 3) > hi);
  }
  int r = (r0 + r1) + (r2 + r3);
  const bool in = live && r < beam;
  const u32 orr = __reduce_or_sync(WFULL, in ? (1u << r) : 0u);
  if (__popc(orr) != __popc(__ballot_sync(WFULL, in))) {
    r = 0;
#pragma unroll 4
    for (int j = 0; j < 32; ++j) {
      const u32 hj = __shfl_sync(WFULL, hi, j), lj = __shfl_sync(WFULL, lo, j);
      r += (int)((hj > hi) || (hj == hi && lj > lo));
    }
  }
  return r;
}

// Bit j set when a[j] == key, for j < cnt (<= KB) of the words of a (16-byte
// aligned shared memory): KB/4 broadcast reads, no branches.
template <int KB>
__device__ __forceinline__ unsigned smem_match(const u32* a, u32 key, int cnt) {
  const uint4* a4 = reinterpret_cast<const uint4*>(a);
  unsigned m = 0u;
#pragma unroll
  for (int q = 0; q < KB / 4; ++q) {
    const uint4 v = a4[q];
    m |= ((unsigned)(v.x == key) << (4 * q)) | ((unsigned)(v.y == key) << (4 * q + 1)) |
         ((unsigned)(v.z == key) << (4 * q + 2)) | ((unsigned)(v.w == key) << (4 * q + 3));
  }
  return cnt >= 32 ? m : (m & ((1u << cnt) - 1u));
}

// Round 2 of the step selection: hypothesis k's first ck_k listed labels are
// every listed candidate of k scoring >= sstar (the list is sorted).  Returns
// -1 when they do not fit the lanes after the n blank slots or the list cannot
// bound what it leaves out; else this lane's candidate as
// (valid << 16 | k << 8 | list position).
__device__ __noinline__ int round2_plan(float A, int len, bool live, float my_lp, int cnt, int n, int cap,
                                        float front_lp, u32 sstar, int lane) {
  const int lim = cnt < 32 ? cnt : 32;
  int ck = 0;
  for (int k = 0; k < n; ++k) {
    const float a = __shfl_sync(WFULL, A, k);
    const int lk = __shfl_sync(WFULL, len, k);
    const bool p = lane < lim && fkey(dadd(my_lp, a)) >= sstar;
    const int c = lk < cap ? __popc(__ballot_sync(WFULL, p)) : 0;
    if (lane == k) ck = c;
  }
  // the list must bound everything it leaves out
  bool over = false;
  if (live && ck == lim && len < cap) {
    if (cnt > 32)
      over = true;
    else if (front_lp > CTCPB_NEG && fkey(dadd(front_lp, A)) >= sstar)
      over = true;
  }
  int pre = ck;  // inclusive prefix over hypotheses
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(WFULL, pre, o);
    if (lane >= o) pre += v;
  }
  const int total = __shfl_sync(WFULL, pre, n > 0 ? n - 1 : 0);
  if (__any_sync(WFULL, over) || n + total > 32) return -1;
  int qk = 0, qp = 0;
  const int idx = lane - n;
  for (int k = 0; k < n; ++k) {
    const int e = __shfl_sync(WFULL, pre, k);
    const int c = __shfl_sync(WFULL, ck, k);
    if (idx >= e - c && idx < e) {
      qk = k;
      qp = idx - (e - c);
    }
  }
  const bool valid = lane >= n && idx < total;
  return ((valid ? 1 : 0) << 16) | (qk << 8) | qp;
}

// Materialise the history ring (steps win0..s_last) into the other parity of
// the flat rows: each hypothesis' row = its origin row's first lo labels + the
// nnew labels it gained in the window.  rows[p]: this row's hypotheses in
// parity p, ldseq labels apart.  prefixes = false writes only the gained
// labels and leaves the prefixes in the old parity (a pending prefix, copied
// later by a call with an empty window and prefixes = true).
__device__ __noinline__ void flush_rows(WarpSmem& W, int* rows0, int* rows1, int ldseq, int lane, int nlive, int blank,
                                        int par, int win0, int s_last, int origin, int lo, int nnew, bool prefixes) {
  int* const from_rows = par ? rows1 : rows0;
  int* const to_rows = par ? rows0 : rows1;
  int slot = lane, rem = nnew;
  for (int r = s_last - win0; r >= 0; --r) {
    const u32 e = W.hist[r][slot & 31];
    const int tk = (int)(e & 0xffffffu);
    if (lane < nlive && tk != blank) {
      --rem;
      to_rows[(size_t)lane * ldseq + lo + rem] = tk;
    }
    slot = (int)(e >> 24);
  }
  // origin prefixes, four rows at a time with every load issued before the stores
  for (int w0 = 0; prefixes && w0 < nlive; w0 += 4) {
    int4 v[4][2];
    int nv[4], o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int w = w0 + u < nlive ? w0 + u : w0;
      o[u] = w0 + u < nlive ? __shfl_sync(WFULL, origin, w) : -1;
      const int c = __shfl_sync(WFULL, lo, w);
      nv[u] = o[u] >= 0 ? (c >> 2) : 0;
      const int4* from = o[u] >= 0 ? reinterpret_cast<const int4*>(from_rows + (size_t)o[u] * ldseq) : nullptr;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (lane + 32 * i < nv[u]) v[u][i] = from[lane + 32 * i];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (o[u] < 0) continue;
      int4* to = reinterpret_cast<int4*>(to_rows + (size_t)(w0 + u) * ldseq);
      const int4* from = reinterpret_cast<const int4*>(from_rows + (size_t)o[u] * ldseq);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (lane + 32 * i < nv[u]) to[lane + 32 * i] = v[u][i];
      for (int x = 64 + lane; x < nv[u]; x += 32) to[x] = from[x];
      const int c = __shfl_sync(WFULL, lo, w0 + u);
      if (lane < (c & 3))
        to_rows[(size_t)(w0 + u) * ldseq + (nv[u] << 2) + lane] = from_rows[(size_t)o[u] * ldseq + (nv[u] << 2) + lane];
    }
  }
  __syncwarp();
}

// A step candidate: score, source slot, token, gathered-slot index of its
// next-step lp[last] (-1: read it directly).
struct Cand {
  float cs;
  int src, tok, gl;
};

// This lane's candidate: its hypothesis' blank slot (lane < n, score scB) or
// listed label qp of hypothesis qk; folded candidates (some live j has
// l_j = l_k + c) are dead.
template <int KB>
__device__ __forceinline__ Cand make_cand(const WarpSmem& W, bool valid, int qk, int qp, float A, int last, int len,
                                          float Rrep, int my_id, float my_lp, float scB, int n, int cnt, int cap,
                                          int beam, int blank, bool anyfold, int lane) {
  const float Ak = __shfl_sync(WFULL, A, qk);
  const int lastk = __shfl_sync(WFULL, last, qk);
  const int lenk = __shfl_sync(WFULL, len, qk);
  const float Rk = __shfl_sync(WFULL, Rrep, qk);
  const int cq = __shfl_sync(WFULL, my_id, qp);
  const float lq = __shfl_sync(WFULL, my_lp, qp);
  Cand c;
  c.cs = lane < n ? scB : CTCPB_NEG;
  c.src = lane < n ? lane : 0;
  c.tok = blank;
  c.gl = lane < n ? lane : -1;
  if (lane >= n && valid && qp < cnt && lenk < cap) {
    c.src = qk;
    c.tok = cq;
    if (lenk > 0 && cq == lastk) {  // the repeat path: pb only
      c.cs = Rk;
      c.gl = qk;
    } else {
      c.cs = dadd(lq, Ak);
      c.gl = beam + qp < kGath ? beam + qp : -1;
    }
    if (anyfold && c.cs > CTCPB_NEG && smem_match<KB>(W.fk, ((u32)c.src << 20) | (u32)c.tok, n) != 0u)
      c.cs = CTCPB_NEG;
  }
  return c;
}

// New slot r := candidate c (source bookkeeping from W.st), its history entry
// in ring row hrow.  nm: the new slot's merge source.
__device__ __forceinline__ void commit_slot(WarpSmem& W, int r, const Cand& c, bool isb, float bpb, float bpnb,
                                            bool gap, int nm, int hrow) {
  const int4 s0 = W.st[0][c.src], s1 = W.st[1][c.src];
  float npb = isb ? bpb : CTCPB_NEG, npnb = isb ? bpnb : c.cs;
  if (gap) {
    npb = c.cs;
    npnb = CTCPB_NEG;
  }
  W.hist[hrow][r] = ((u32)c.src << 24) | ((u32)c.tok & 0xffffffu);
  W.nst[0][r] = make_int4(__float_as_int(npb), __float_as_int(npnb), __float_as_int(c.cs), isb ? s0.x : c.tok);
  W.nst[1][r] = make_int4(isb ? s0.y : s0.y + 1, isb ? s0.z : (int)h32((u32)s0.z, c.tok), isb ? s0.w : s0.z, s1.x);
  // the labels gained since the last token-store write, and bit 30: a blank winner
  W.nst[2][r] = make_int4(s1.y, (s1.z + (isb ? 0 : 1)) | (isb ? kBlankWin : 0), c.gl, nm);
  // prefix key of an extension winner for the merge check (a blank winner's
  // dummy can only cause an extra exact comparison)
  W.hk[r] = isb ? 0xffffffffu : (h32((u32)s0.z, c.tok) ^ ((u32)(s0.y + 1) * kGold));
}

// The exhaustive selection when the frame's list bounds every unlisted label:
// the candidates scoring at least thr (blank slots, repeats, listed
// extensions) are compacted into W.keys with the running count in a register,
// then each lane ranks its keys by counting the larger ones (the keys are
// distinct: no two candidates share a source slot and a token).  Leaves the
// winners in order in W.keys[0 .. nw) and returns nw, or -1 when
// warp_collect_select must run instead: more than kFastKeys candidates, or an
// unlisted label that could still reach the beam.
constexpr int kFastKeys = 128;
__device__ __noinline__ int fast_exhaustive(WarpSmem& W, const char* rec, int Lpad, u64 thr, float A, int last,
                                               int len, bool live, float Rrep, float scB, int mi, int n, int cap,
                                               int beam, int blank, int lane) {
  const RecHdr* h = (const RecHdr*)rec;
  const int cnt = h->cnt;
  const int* ids = (const int*)(rec + 32);
  const float* lps = (const float*)(rec + 32 + 4 * Lpad);
  const unsigned lt = (1u << lane) - 1u;
  int base = 0;  // keys written so far (the same in every lane)
  // slot j absorbs the extension (mi_j, last_j): it is not a candidate of its own
  const unsigned folds = __ballot_sync(WFULL, live && mi >= 0);
  bool rep_folded = false;
  for (unsigned f = folds; f; f &= f - 1u) {
    const int j = __ffs(f) - 1;
    const int ij = __shfl_sync(WFULL, mi, j), cj = __shfl_sync(WFULL, last, j);  // every lane shuffles
    rep_folded |= ij == lane && cj == last;
  }
  {
    const u64 kb = (live && scB > CTCPB_NEG) ? cand_key(scB, lane, blank) : 0ull;
    const u64 kr = (live && Rrep > CTCPB_NEG && !rep_folded) ? cand_key(Rrep, lane, last) : 0ull;
    const bool tb = kb != 0ull && kb >= thr, tr = kr != 0ull && kr >= thr;
    const unsigned mb = __ballot_sync(WFULL, tb), mr = __ballot_sync(WFULL, tr);
    if (tb) W.keys[__popc(mb & lt)] = kb;
    if (tr) W.keys[__popc(mb) + __popc(mr & lt)] = kr;
    base = __popc(mb) + __popc(mr);
  }
  for (int p0 = 0; p0 < cnt; p0 += 32) {
    const int p = p0 + lane;
    const bool pv = p < cnt;
    const int c = pv ? ids[p] : -1;
    const float v = pv ? lps[p] : CTCPB_NEG;
    unsigned fk = 0u;  // hypotheses whose extension by c a fold absorbs
    for (unsigned f = folds; f; f &= f - 1u) {
      const int j = __ffs(f) - 1;
      const int ij = __shfl_sync(WFULL, mi, j), cj = __shfl_sync(WFULL, last, j);
      if (cj == c) fk |= 1u << ij;
    }
    for (int k = 0; k < n; ++k) {
      const float a = __shfl_sync(WFULL, A, k);
      const int lk = __shfl_sync(WFULL, len, k), tk = __shfl_sync(WFULL, last, k);
      const float sc = dadd(v, a);
      const bool ok = pv && lk < cap && !(lk > 0 && c == tk) && ((fk >> k) & 1u) == 0u && sc > CTCPB_NEG;
      const u64 key = ok ? cand_key(sc, k, c) : 0ull;
      const bool take = ok && key >= thr;
      const unsigned m = __ballot_sync(WFULL, take);
      const int at = base + __popc(m & lt);
      if (take && at < kFastKeys) W.keys[at] = key;
      base += __popc(m);
    }
  }
  if (base > kFastKeys) return -1;
  __syncwarp();
  const int m = base;
  u64 x[kFastKeys / 32];
  int r[kFastKeys / 32];
#pragma unroll
  for (int i = 0; i < kFastKeys / 32; ++i) {
    const int q = lane + 32 * i;
    x[i] = q < m ? W.keys[q] : 0ull;
    r[i] = 0;
  }
  for (int t = 0; t < m; ++t) {
    const u64 y = W.keys[t];
#pragma unroll
    for (int i = 0; i < kFastKeys / 32; ++i) r[i] += (int)(y > x[i]);
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kFastKeys / 32; ++i)
    if (x[i] != 0ull && r[i] < beam) W.keys[r[i]] = x[i];
  __syncwarp();
  const int nw = m < beam ? m : beam;
  // an unlisted label scores at most front_lp: it must stay below the beam-th key
  const float front_lp = h->front_lp;
  if (front_lp > CTCPB_NEG) {
    u64 t2 = thr;
    if (nw == beam && W.keys[beam - 1] > t2) t2 = W.keys[beam - 1] & 0xffffffff00000000ull;
    bool bad = false;
    if (live && len < cap) {
      const float u = dadd(front_lp, A);
      bad = u > CTCPB_NEG && ((u64)fkey(u) << 32) >= t2;
    }
    if (__any_sync(WFULL, bad)) return -1;
  }
  return nw;
}

// The selection when the first candidate set did not prove it: round 2 (every
// listed candidate scoring >= sstar, when they fit the warp), else the
// exhaustive selection.  Writes the winners' new slots like the fast path.
// Returns nw | exhaustive << 8 | frame scanned << 9.
template <int KB>
__device__ __forceinline__ int slow_select(WarpSmem& W, const char* Rc, const float* row, u32 sstar, int nw1, float A,
                                        int last, int len, bool live, float Rrep, int my_id, float my_lp, float scB,
                                        float bpb, float bpnb, int mi, bool anyfold, int n, int cnt, int cap, int beam,
                                        int blank, int V, int Lpad, bool gap, int hrow, int lane, BoostTab bt) {
  const RecHdr* hd = (const RecHdr*)Rc;
  if (nw1 == beam) {
    const int plan = round2_plan(A, len, live, my_lp, cnt, n, cap, hd->front_lp, sstar, lane);
    if (plan >= 0) {
      const Cand c = make_cand<KB>(W, (plan >> 16) != 0, (plan >> 8) & 0xff, plan & 0xff, A, last, len, Rrep, my_id,
                                   my_lp, scB, n, cnt, cap, beam, blank, anyfold, lane);
      const bool clive = c.cs > CTCPB_NEG;
      const u32 hi = clive ? fkey(c.cs) : 0u;
      const int r = warp_rank(hi, clive ? ~(((u32)c.src << 20) | (u32)c.tok) : 0u, clive, beam);
      const bool won = clive && r < beam;
      const int nw = __popc(__ballot_sync(WFULL, won));
      const int mq = lane < n ? mi : c.src;
      const int nm = __shfl_sync(WFULL, won ? r : -1, mq < 0 ? 0 : mq);
      if (won) commit_slot(W, r, c, lane < n, bpb, bpnb, gap, mq < 0 ? -1 : nm, hrow);
      return nw;
    }
  }
  // ---- exhaustive selection over the frame's list
  if (live) {
    W.A[lane] = A;
    W.bpb[lane] = bpb;
    W.bpnb[lane] = bpnb;
    W.scb[lane] = scB;
    W.rep[lane] = Rrep;
    W.last[lane] = last;
    W.len[lane] = len;
  }
  const unsigned fmm = __ballot_sync(WFULL, mi >= 0);
  if (mi >= 0) {
    const int f = __popc(fmm & ((1u << lane) - 1u));
    W.fold_i[f] = mi;
    W.fold_c[f] = last;
  }
  if (lane == 0) W.nfold = __popc(fmm);
  W.bw[lane] = -1;
  __syncwarp();
  const u64 thr = nw1 == beam ? ((u64)sstar << 32) : 0ull;
  int res = fast_exhaustive(W, Rc, Lpad, thr, A, last, len, live, Rrep, scB, mi, n, cap, beam, blank, lane);
  if (res < 0) res = warp_collect_select(W, Rc, Lpad, n, beam, cap, blank, V, row, lane, thr, bt);
  const int nw = res & 0xffff;
  const u64 key = lane < nw ? W.keys[lane] : 0ull;
  const int gsrc = ck_src(key), gtk = ck_tok(key);
  const bool gisb = gtk == blank;
  if (lane < nw && gisb) W.bw[gsrc] = lane;
  __syncwarp();
  if (lane < nw) {
    Cand c;
    c.cs = ck_score(key);
    c.src = gsrc;
    c.tok = gtk;
    const int4 s0 = W.st[0][gsrc], s1 = W.st[1][gsrc];
    c.gl = (gisb || (s0.y > 0 && gtk == s0.x)) ? gsrc : -1;
    const int gm = gisb ? (s1.w >= 0 ? W.bw[s1.w] : -1) : W.bw[gsrc];
    commit_slot(W, lane, c, gisb, gisb ? W.bpb[gsrc] : CTCPB_NEG, gisb ? W.bpnb[gsrc] : CTCPB_NEG, gap, gm, hrow);
  }
  return nw | (1 << 8) | ((res >> 16) << 9);
}

}  // namespace

// ----------------------------------------------------------------------------
constexpr long long kFlagSpins = 1ll << 20;  // bounded wait for published records (about 1 s)

// The steps of rows row_block*kWPC + warp (warps 0..kWPC-1 of the block; the
// block's other warps only help build the tables).  KB: beam bucket (8 or 16),
// the bound of the per-hypothesis compares.  BOOST: the rows have label-boost
// tables.  flags: the records' ready flags when the pre-pass runs concurrently
// (null: the records are complete).
template <int KB, bool BOOST>
__device__ __forceinline__ void step_warp_body(const View& st, const float* __restrict__ lp, long long sb,
                                               long long stt, int mode, const int* __restrict__ nframes,
                                               int chunk_T, int tile_start, int tile_len, unsigned char* smem,
                                               int row_block, u32* flags) {
  Tables& tb = *reinterpret_cast<Tables*>(smem);
  const int wid = threadIdx.x >> 5;
  WarpSmem& W = reinterpret_cast<WarpSmem*>(smem + align_up(sizeof(Tables), 16))[wid < kWPC ? wid : 0];
  // per step warp: its row's pending prefixes are in place (set by a helper warp)
  volatile int* pend_done = reinterpret_cast<int*>(smem + align_up(sizeof(Tables), 16) + kWPC * sizeof(WarpSmem));
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < (int)(sizeof(Tables) / 16); i += blockDim.x)
    reinterpret_cast<int4*>(&tb)[i] = reinterpret_cast<const int4*>(&g_tables)[i];
  if (threadIdx.x < kWPC) pend_done[threadIdx.x] = 0;
  __syncthreads();

  const Layout& Ly = st.lay;
  if (wid >= kWPC) {
    // A helper warp: the prefixes that the previous call left in the other
    // parity of the row of step warp wid - kWPC, copied while that warp waits
    // for its first ranked records.  (Repeating the copy is harmless, so it
    // does not matter whether the step warp decodes anything in this call.)
    const int hw = wid - kWPC, hb = row_block * kWPC + hw;
    if (hw < kWPC && hb < Ly.B) {
      const RowHdr rh = st.rows()[hb];
      if (rh.pending && (mode == 0 || header_matches(st))) {
        const size_t hrb = (size_t)hb * Ly.beam;
        const int po = lane < rh.nlive ? st.porg()[hrb + lane] : -1;
        const int pl = lane < rh.nlive ? st.plo()[hrb + lane] : 0;
        flush_rows(W, st.clist(0, hb, 0), st.clist(1, hb, 0), Ly.ldseq, lane, rh.nlive, Ly.blank, rh.parity ^ 1, 0,
                   -1, po, pl, 0, true);
      }
      __threadfence_block();
      if (lane == 0) pend_done[hw] = 1;
    }
    return;
  }
  const int b = row_block * kWPC + wid;
  if (b >= Ly.B) return;
  // the row's label-boost table (keys null: no boosting; BOOST instantiations only)
  const BoostTab bt{BOOST ? st.bkey(b) : nullptr, BOOST ? st.bval(b) : nullptr, Ly.hcap - 1};
  const int beam = Ly.beam, cap = Ly.cap, blank = Ly.blank, V = Ly.V, Lpad = Ly.Lpad;
  const int space = Ly.space;  // word-boundary label, -1: none
  const float NEG = CTCPB_NEG;

  if (mode != 0) {
    const Header* hd = st.hdr();
    bool ok = hd->magic == kMagic && hd->version == kVersion && hd->B == Ly.B && hd->V == Ly.V &&
              hd->beam == Ly.beam && hd->cap == Ly.cap && hd->paged == Ly.paged &&
              hd->page_size == Ly.page_size && hd->blank == Ly.blank && hd->list_len == Ly.L &&
              hd->tile == Ly.tile && hd->space == Ly.space && hd->hcap == Ly.hcap;
    if (!ok) {
      if (lane == 0) atomicOr(&st.hdr()->status, CTCPB_DEV_HEADER);
      return;
    }
  }
  // mode 0: offline (frame list); 1: streaming, every frame of the tile;
  // 2: streaming with a speech mask (the tile's selected chunk rows)
  int nsteps, nft = 0;  // nft: the tile's frames of this stream, skipped ones included
  if (mode != 0) {
    int nf = nframes ? nframes[b] : chunk_T;
    nf = nf < 0 ? 0 : (nf > chunk_T ? chunk_T : nf);
    nft = nf - tile_start;
    nft = nft < 0 ? 0 : (nft > tile_len ? tile_len : nft);
  }
  nsteps = mode == 1 ? nft : st.nsel()[b];
  if (nsteps == 0) {
    if (mode == 2 && lane == 0) st.rows()[b].tcount += nft;  // every frame of the tile was skipped
    return;
  }

  const RowHdr rh0 = st.rows()[b];
  int step = rh0.step, t_prev = rh0.t_prev, nlive = rh0.nlive, par = rh0.parity;
  const int tcount = rh0.tcount;
  const size_t rb = (size_t)b * beam;
  float pb = NEG, pnb = NEG, sc = NEG;
  int last = blank, len = 0, msrc = -1;
  u32 h = 0u, hp = 0u;
  if (lane < nlive) {
    pb = st.pb()[rb + lane];
    pnb = st.pnb()[rb + lane];
    sc = st.sc()[rb + lane];
    last = st.last()[rb + lane];
    len = st.len()[rb + lane];
    h = (u32)st.h()[rb + lane];
    hp = (u32)st.hp()[rb + lane];
    msrc = st.msrc()[rb + lane];
  }
  int origin = lane, lo = len, nnew = 0, gl = -1;
  // BOOST: the first two slots of the last label's probe sequence, loaded a
  // step before they are used and without a branch on the loaded values (a
  // branch would wait for the loads); a label further along is looked up then
  int bk0 = -1, bk1 = -1;
  float bv0 = 0.0f, bv1 = 0.0f;
  auto bonus_prefetch = [&](bool want) {
    const int h0 = boost_slot(want ? last : 0, bt.hmask), h1 = (h0 + 1) & bt.hmask;
    bk0 = want ? __ldg(bt.keys + h0) : -1;
    bk1 = want ? __ldg(bt.keys + h1) : -1;
    bv0 = want ? __ldg(bt.vals + h0) : 0.0f;
    bv1 = want ? __ldg(bt.vals + h1) : 0.0f;
  };
  if (BOOST) bonus_prefetch(lane < nlive && len > 0);
  int win0 = 0;  // call step index of the ring's first entry
  u32 c_steps = 0, c_fb = 0, c_gen = 0, c_scan = 0, c_hash = 0;
#ifdef CTCPB_PHASE_PROF
  u64 prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  long long prof_t0 = clock64();
#endif
  const float* lpb_row = lp + (long long)b * sb;
  char* const rec_g = st.rec(b, 0);  // this row's records, rec_bytes apart
  const unsigned rbytes = (unsigned)Ly.rec_bytes;
  u32* const rflags = flags ? flags + (size_t)b * Ly.tile : nullptr;
  int s_pub = rflags ? 0 : nsteps;  // records [0, s_pub) are known to be published
  // all lanes: make sure records [0, s_end) are published.  Lane j acquires
  // the flag of record s_pub + j, so one pass covers up to 32 records.
  auto await_records = [&](int s_end) -> bool {
    for (long long spin = 0; s_pub < s_end; ++spin) {
      if (spin >= kFlagSpins) return false;
      const int r = s_pub + lane;
      const bool set = r >= nsteps || ld_acquire_u32(rflags + r) != 0u;
      const unsigned m = __ballot_sync(WFULL, set);
      s_pub += (m == WFULL) ? 32 : __ffs(~m) - 1;
      if (s_pub < s_end) __nanosleep(64);
    }
    __syncwarp();
    return true;
  };
  // record of step s in registers (L2 loads: records may be written by other
  // SMs during this launch)
  struct RecR {
    int cnt, t, id;
    float lpb, flp, lp;
  };
  auto rec_t = [&](int s) -> int { return __ldcg(reinterpret_cast<const int*>(rec_g + (size_t)s * rbytes + 16)); };
  auto load_rec = [&](int s) -> RecR {
    const char* g = rec_g + (size_t)s * rbytes;
    const int4 h0 = __ldcg(reinterpret_cast<const int4*>(g));  // cnt, front id, lp[blank], front lp
    RecR r;
    r.cnt = h0.x;
    r.lpb = __int_as_float(h0.z);
    r.flp = __int_as_float(h0.w);
    r.t = __ldcg(reinterpret_cast<const int*>(g + 16));
    // list position `lane` (lanes past the list read position 0; see my_id)
    const int p = lane < Ly.L ? lane : 0;
    r.id = __ldcg(reinterpret_cast<const int*>(g + 32) + p);
    r.lp = __ldcg(reinterpret_cast<const float*>(g + 32 + 4 * Lpad) + p);
    return r;
  };
  // a wait ran out: report it, let this warp's copies in flight land
  auto bail = [&]() {
    if (lane == 0) atomicOr(&st.hdr()->status, CTCPB_DEV_TIMEOUT);
    cp_wait_all();
  };

  // Materialise the ring into the other parity of the flat rows.
  int* const rows0 = st.clist(0, b, 0);
  int* const rows1 = st.clist(1, b, 0);
  // Before the rows are first written or compared: the helper warp has put
  // the previous call's pending prefixes in place (a bounded wait).  Blocks
  // without helper warps (the stand-alone step kernel) copy them here.
  const bool helpers = (int)blockDim.x >= 64 * kWPC;
  if (rh0.pending && !helpers) {
    const int po = lane < nlive ? st.porg()[rb + lane] : -1;
    const int pl = lane < nlive ? st.plo()[rb + lane] : 0;
    flush_rows(W, rows0, rows1, Ly.ldseq, lane, nlive, blank, par ^ 1, 0, -1, po, pl, 0, true);
  }
  bool pend_wait = rh0.pending != 0 && helpers;
  auto wait_pending = [&]() {
    if (!pend_wait) return;
    pend_wait = false;
    long long spin = 0;
    while (pend_done[wid] == 0 && spin < kFlagSpins) {
      __nanosleep(64);
      ++spin;
    }
    if (spin >= kFlagSpins && lane == 0) atomicOr(&st.hdr()->status, CTCPB_DEV_TIMEOUT);
    __threadfence_block();
    __syncwarp();
  };
  auto flush = [&](int s_last) {
    wait_pending();
    flush_rows(W, rows0, rows1, Ly.ldseq, lane, nlive, blank, par, win0, s_last, origin, lo, nnew, true);
    par ^= 1;
    origin = lane;
    lo = len;
    nnew = 0;
    win0 = s_last + 1;
  };

  if (!await_records(nsteps < 2 ? nsteps : 2)) {
    bail();
    return;
  }
  RecR cur = load_rec(0);                   // the record of step s
  int t1 = nsteps > 1 ? rec_t(1) : 0;      // frame index of step s+1

  for (int s = 0; s < nsteps; ++s) {
    PHASE_MARK(7);
    // the record of step s+1 and the frame index of step s+2
    if (s + 2 < nsteps && !await_records(s + 3)) {
      bail();
      return;
    }
    // unconditional loads (clamped to a published record): a select on the
    // loaded values would wait for them here
    const RecR nx = load_rec(s + 1 < nsteps ? s + 1 : s);
    const int t2 = rec_t(s + 2 < nsteps ? s + 2 : s);
    if (rflags && lane == 0) rflags[s] = 0u;  // consumed: the slot is free for the next tile
    PHASE_MARK(0);
    const int cnt = cur.cnt;
    const float lpb = cur.lpb;
    const int my_id = lane < Ly.L ? cur.id : -1;
    const float my_lp = lane < Ly.L ? cur.lp : NEG;
    const int t = mode == 0 ? cur.t : (mode == 1 ? tcount + s : tcount + cur.t - tile_start);
    const float* row = lpb_row + (long long)(mode != 1 ? cur.t : tile_start + s) * stt;
    const bool gap = t > t_prev + 1;
    const bool live = lane < nlive;
    // lp[t][last] of this lane's hypothesis, gathered by the previous step
    cp_wait_all();
    __syncwarp();
    const float gcur = gl >= 0 ? W.gath[s & 1][gl] : 0.0f;
    // lp[t_{s+1}][x] for every label x that can be "last" at step s+1: the
    // current lasts (slot k) and this step's list (slot beam + position)
    if (s + 1 < nsteps) {
      const float* row1 = lpb_row + (long long)(mode != 1 ? t1 : tile_start + s + 1) * stt;
      float* gdst = W.gath[(s + 1) & 1];
      if (live && len > 0) cp_async4(gdst + lane, row1 + last);
      if (lane < cnt && beam + lane < kGath) cp_async4(gdst + beam + lane, row1 + my_id);
      cp_commit();
    }

    int nw;
    bool isb_w = false;
    if (step == 0) {
      // ---- section 3.3
      const int nb = beam > 1 ? beam - 1 : 1;
      const int ntok = cap >= 1 ? (nb < cnt ? nb : cnt) : 0;
      const bool empty_live = beam > 1 && lpb > NEG;
      if (lane < ntok) {
        pb = gap ? my_lp : NEG;
        pnb = gap ? NEG : my_lp;
        sc = my_lp;
        last = my_id;
        len = 1;
        h = h32(kH32, my_id);
        hp = kH32;
        msrc = empty_live ? ntok : -1;
        W.hist[s - win0][lane] = ((u32)lane << 24) | (u32)my_id;
      } else if (lane == ntok && empty_live) {
        pb = lpb;
        pnb = NEG;
        sc = lpb;
        last = blank;
        len = 0;
        h = kH32;
        hp = 0u;
        msrc = -1;
        W.hist[s - win0][lane] = ((u32)lane << 24) | (u32)blank;
      }
      nw = ntok + (empty_live ? 1 : 0);
      origin = -1;
      lo = 0;
      nnew = lane < ntok ? 1 : 0;
      gl = -1;
    } else {
      // ---- sections 3.4.1-3.4.3 on lanes 0..nlive-1
      const int mi = live ? msrc : -1;
      // (i, last) names the candidate this slot absorbs; a unique dummy otherwise
      const u32 foldk = mi >= 0 ? (((u32)mi << 20) | (u32)last) : (0x80000000u | (u32)lane);
      if (live) {
        W.st[0][lane] = make_int4(last, len, (int)h, (int)hp);
        W.st[1][lane] = make_int4(origin, lo, nnew, msrc);
      }
      W.fk[lane] = foldk;
      __syncwarp();
      PHASE_MARK(1);
      const float A = sc;
      const float pbx = gap ? A : pb;  // collapsed-blank correction: lse(pb, pnb) is the stored score
      const float pnbx = gap ? NEG : pnb;
      float lpl = NEG;
      {
        const bool gathered = s >= 1 && gl >= 0;
        if (live && len > 0) lpl = gathered ? rdlp(gcur) : rdlp(__ldg(row + last));
      }
      // the last label emitted again (the repeat path, a fold) carries its bonus
      float lple = lpl;
      if (BOOST && live && len > 0) {
        float bon = 0.0f;  // an empty slot ends the probe: not boosted
        if (bk0 == last)
          bon = bv0;
        else if (bk0 >= 0 && bk1 == last)
          bon = bv1;
        else if (bk0 >= 0 && bk1 >= 0)
          bon = boost_of(bt.keys, bt.vals, bt.hmask, last);
        lple = dadd(lpl, bon);
      }
      const float bpb = dadd(lpb, A);
      // (a space-ending beam has no stay path: every space frame is a token)
      const float stay = (live && len > 0 && !gap && last != space) ? dadd(lpl, pnbx) : NEG;
      const int mil = mi < 0 ? 0 : mi;
      const float A_i = __shfl_sync(WFULL, A, mil);
      const float pb_i = __shfl_sync(WFULL, pbx, mil);
      const int last_i = __shfl_sync(WFULL, last, mil);
      const int len_i = __shfl_sync(WFULL, len, mil);
      const bool rep_i = mi >= 0 && len_i > 0 && last_i == last && last != space;
      // the extension of l_i folded into this blank slot (NEG when there is none)
      const float mterm = mi >= 0 ? dadd(lple, rep_i ? pb_i : A_i) : NEG;
      // candidate (k, last): the repeat path (pb only); the word-boundary label
      // extends from both paths
      const float Rrep = (live && len > 0 && len < cap) ? dadd(lple, last == space ? A : pbx) : NEG;
      const int n = nlive;
      // blank slot (3.4.1-3.4.3), branch-free so it overlaps the candidates below
      const bool anyfold = __any_sync(WFULL, mi >= 0);
      const float bpnb = anyfold ? dlse(tb.fc, stay, mterm) : stay;  // dlse(stay, NEG) == stay
      const float scB = live ? dlse(tb.fc, bpb, bpnb) : NEG;
      // proof bound of this hypothesis: what its best label outside the set scores
      float bnd = NEG;
      {
        const int q = live ? tb.qcnt[n][lane] : 0;
        const float nxt = __shfl_sync(WFULL, my_lp, q & 31);
        if (live && len < cap) {
          if (q < cnt)
            bnd = dadd(nxt, A);
          else if (cur.flp > NEG)
            bnd = dadd(cur.flp, A);
        }
      }

      // the largest bound (0: none), for the proof below
      const u32 bmax = __reduce_max_sync(WFULL, bnd > NEG ? fkey(bnd) : 0u);
      // ---- round 1: the staircase
      const unsigned short qm = lane >= n ? tb.qmap[n][lane] : (unsigned short)0xffff;
      const Cand c = make_cand<KB>(W, qm != 0xffff, qm == 0xffff ? 0 : (qm >> 8), qm == 0xffff ? 0 : (qm & 31), A,
                                   last, len, Rrep, my_id, my_lp, scB, n, cnt, cap, beam, blank, anyfold, lane);
      const bool clive = c.cs > NEG;
      const u32 hi = clive ? fkey(c.cs) : 0u;
      // The ranking is proven exact when no hypothesis can reach the beam-th
      // kept score with a label left out of the set: there is no bound, or at
      // least `beam` live candidates score above the largest bound.  This
      // needs only the scores, so it runs beside the ranking.
      const bool proven = bmax == 0u || __popc(__ballot_sync(WFULL, clive && hi > bmax)) >= beam;
      const int r = warp_rank(hi, clive ? ~(((u32)c.src << 20) | (u32)c.tok) : 0u, clive, beam);
      const bool won = clive && r < beam;
      nw = __popc(__ballot_sync(WFULL, won));
      PHASE_MARK(2);
      // ---- section 3.4.5: the candidate ranked r writes new slot r, before
      // the proof is known (an unproven step rewrites the slots)
      {
        const int mq = lane < n ? mi : c.src;
        const int nm = __shfl_sync(WFULL, won ? r : -1, mq < 0 ? 0 : mq);
        if (won) commit_slot(W, r, c, lane < n, bpb, bpnb, gap, mq < 0 ? -1 : nm, s - win0);
      }
      PHASE_MARK(3);
      if (!proven) {
        // the beam-th kept score: round 2's threshold
        const unsigned lastm = __ballot_sync(WFULL, won && r == beam - 1);
        const u32 sstar = __shfl_sync(WFULL, hi, lastm ? __ffs(lastm) - 1 : 0);
        // the record, for the slow selection, into shared memory
        const int4* rg = reinterpret_cast<const int4*>(rec_g + (size_t)s * rbytes);
        for (int i = lane; i < (int)(rbytes / 16); i += 32) reinterpret_cast<int4*>(W.rec1)[i] = __ldcg(rg + i);
        __syncwarp();  // (also: the optimistic slots are written before they are rewritten)
        ++c_fb;
        const int res = slow_select<KB>(W, W.rec1, row, sstar, nw, A, last, len, live, Rrep, my_id, my_lp, scB, bpb, bpnb,
                                        mi, anyfold, n, cnt, cap, beam, blank, V, Lpad, gap, s - win0, lane, bt);
        nw = res & 0xff;
        c_gen += (u32)((res >> 8) & 1);
        c_scan += (u32)((res >> 9) & 1);
      }
      __syncwarp();
      PHASE_MARK(4);
      if (lane < nw) {
        const int4 n0 = W.nst[0][lane], n1 = W.nst[1][lane], n2 = W.nst[2][lane];
        pb = __int_as_float(n0.x);
        pnb = __int_as_float(n0.y);
        sc = __int_as_float(n0.z);
        last = n0.w;
        len = n1.x;
        h = (u32)n1.y;
        hp = (u32)n1.z;
        origin = n1.w;
        lo = n2.x;
        nnew = n2.y & ~kBlankWin;
        gl = n2.z;
        msrc = n2.w;
        isb_w = (n2.y & kBlankWin) != 0;
      } else {
        msrc = -1;
      }
    }

    // ---- the one merge relation the sources cannot show: a blank winner
    // whose parent prefix equals an extension winner (hash proposal, exact check)
    nlive = nw;
    if (BOOST) bonus_prefetch(lane < nw && len > 0);
    {
      const bool wl = lane < nw;
      const bool want = wl && step > 0 && isb_w && msrc < 0 && len >= 1;
      {
        const unsigned match = smem_match<KB>(W.hk, hp ^ ((u32)(len - 1) * kGold), nw);
        const bool cand = want && match != 0u;
        if (__any_sync(WFULL, cand)) {
          ++c_hash;
          flush(s);  // tokens of every hypothesis into the flat rows
          for (unsigned mj = __ballot_sync(WFULL, cand); mj; mj &= mj - 1) {
            const int j = __ffs(mj) - 1;
            const unsigned gj = __shfl_sync(WFULL, match, j);
            const int Lj = __shfl_sync(WFULL, len, j);
            for (unsigned mi2 = gj; mi2; mi2 &= mi2 - 1) {
              const int i = __ffs(mi2) - 1;
              const int* ri = st.clist(par, b, i);
              const int* rj = st.clist(par, b, j);
              bool mism = false;
              for (int x = lane; x < Lj - 1; x += 32) mism |= ri[x] != rj[x];
              if (!__any_sync(WFULL, mism)) {
                if (lane == j) msrc = i;
                break;
              }
            }
          }
        }
      }
    }
    PHASE_MARK(5);
    t_prev = t;
    ++step;
    ++c_steps;
    cur = nx;
    t1 = t2;
    PHASE_MARK(6);
    if (s - win0 + 1 == kRing && s + 1 < nsteps) flush(s);
  }
  cp_wait_all();
  __syncwarp();
  // the gained labels only; the prefixes stay pending in the old parity (the
  // next call or the N-best gather reads them from there)
  wait_pending();
  flush_rows(W, rows0, rows1, Ly.ldseq, lane, nlive, blank, par, win0, nsteps - 1, origin, lo, nnew, false);
  if (lane < nlive) {
    st.porg()[rb + lane] = origin;
    st.plo()[rb + lane] = lo;
  }
  par ^= 1;

  if (lane < beam) {
    st.pb()[rb + lane] = pb;
    st.pnb()[rb + lane] = pnb;
    st.sc()[rb + lane] = sc;
    st.last()[rb + lane] = last;
    st.len()[rb + lane] = len;
    st.h()[rb + lane] = h;
    st.hp()[rb + lane] = hp;
    st.msrc()[rb + lane] = msrc;
  }
  if (lane == 0) {
    atomicAdd(&st.hdr()->counters[0], c_steps);
    atomicAdd(&st.hdr()->counters[1], c_fb);
    atomicAdd(&st.hdr()->counters[2], c_gen);
    atomicAdd(&st.hdr()->counters[3], c_scan);
    atomicAdd(&st.hdr()->counters[4], c_hash);
#ifdef CTCPB_PHASE_PROF
    for (int i = 0; i < 8; ++i) atomicAdd(&st.hdr()->phase_cycles[i], prof[i]);
#endif
    RowHdr rr = rh0;
    rr.step = step;
    rr.tcount = mode == 0 ? rh0.tcount : tcount + nft;
    rr.t_prev = t_prev;
    rr.nlive = nlive;
    rr.parity = par;
    rr.pending = 1;
    st.rows()[b] = rr;
  }
}

template <int KB, bool BOOST>
__global__ void __launch_bounds__(32 * kWPC, 1) k_step_warp(View st, const float* __restrict__ lp, long long sb,
                                                         long long stt, int mode, const int* __restrict__ nframes,
                                                         int chunk_T, int tile_start, int tile_len) {
  extern __shared__ __align__(128) unsigned char smem[];
  step_warp_body<KB, BOOST>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, smem, blockIdx.x, nullptr);
}

// Pre-pass and steps in one cooperative launch: blocks [0, nsb) run the rows'
// steps, the others rank frames (frame-major) and publish each record with a
// release flag that the step warps acquire before copying it.  Every block is
// resident at once (cooperative launch), so the waits always end; each one is
// bounded all the same.
template <int KB, bool BOOST>
__global__ void __launch_bounds__(256, 1) k_fused(View st, const float* __restrict__ lp, long long sb, long long stt,
                                                  int mode, const int* __restrict__ nframes, int chunk_T,
                                                  int tile_start, int tile_len, int nsb, int rank_warps) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(&st.hdr()->fused_launches, 1u);
  if ((int)blockIdx.x < nsb) {
    step_warp_body<KB, BOOST>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, smem, blockIdx.x,
                              st.rflag());
  } else {
    RecItems items{st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, st.rflag()};
    rank_tma_body_small(items, st.lay.V, st.lay.blank, st.lay.L, &st.hdr()->status, smem, (int)blockIdx.x - nsb,
                  (int)gridDim.x - nsb, rank_warps);
  }
}

// beam <= 16: with more live hypotheses the 32-lane candidate set leaves too
// few lanes for extensions to prove a selection (the block kernel is faster
// from beam 17 on: 9.2 vs 17.4 ms at beam 20 on the bpe workload).
bool step_warp_fits(const Layout& lay) {
  return lay.beam <= 16 && !lay.paged && lay.rec_bytes <= (size_t)kMaxRec;
}

size_t step_warp_smem_bytes() { return align_up(sizeof(Tables), 16) + kWPC * sizeof(WarpSmem) + 16 * kWPC; }

template <int KB, bool BOOST>
static cudaError_t launch_kb(const View& st, const float* lp, long long sb, long long stt, int mode,
                             const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  const size_t smem = step_warp_smem_bytes();
  cudaError_t e = smem_optin<k_step_warp<KB, BOOST>>(smem);
  if (e != cudaSuccess) return e;
  const int blocks = (st.lay.B + kWPC - 1) / kWPC;
  k_step_warp<KB, BOOST><<<blocks, 32 * kWPC, smem, s>>>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len);
  return cudaGetLastError();
}

cudaError_t launch_step_warp(const View& st, const float* lp, long long sb, long long stt, int mode,
                             const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  // label boosting has instantiations of its own, so the plain kernels carry none of its code
  const bool bo = st.lay.hcap > 0;
  if (st.lay.beam <= 8)
    return bo ? launch_kb<8, true>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s)
              : launch_kb<8, false>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
  return bo ? launch_kb<16, true>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s)
            : launch_kb<16, false>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
}

template <int KB, bool BOOST>
static cudaError_t launch_fused_kb(const View& st, const float* lp, long long sb, long long stt, int mode,
                                  const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  const Layout& Ly = st.lay;
  int dev = 0, coop = 0, sms = 0, maxsm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  int rw = rank_tma_warps(Ly.V);
  if (rw > 8) rw = 8;
  const size_t rank_smem = rank_tma_per_warp(Ly.V) * (size_t)rw;
  const size_t smem = rank_smem > step_warp_smem_bytes() ? rank_smem : step_warp_smem_bytes();
  if (!coop || rw < 1 || smem > (size_t)maxsm) return cudaErrorNotSupported;
  e = smem_optin<k_fused<KB, BOOST>>(smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_fused<KB, BOOST>, 256, smem);
  if (e != cudaSuccess) return e;
  const int grid = per_sm * sms;
  int nsb = (Ly.B + kWPC - 1) / kWPC;
  if (per_sm < 1 || nsb + 8 > grid) return cudaErrorNotSupported;  // keep at least 8 ranking blocks
  View stv = st;
  void* args[] = {&stv, (void*)&lp, &sb, &stt, &mode, (void*)&nframes, &chunk_T, &tile_start, &tile_len, &nsb, &rw};
  e = cudaLaunchCooperativeKernel((const void*)k_fused<KB, BOOST>, grid, 256, args, smem, s);
  if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported) {
    cudaGetLastError();  // this launch's own refusal, just recorded: consume it
    return cudaErrorNotSupported;
  }
  return e;
}

cudaError_t launch_fused(const View& st, const float* lp, long long sb, long long stt, int mode, const int* nframes,
                         int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  if (!step_warp_fits(st.lay) || !rank_tma_ok(lp, sb, stt, st.lay.V, st.lay.L)) return cudaErrorNotSupported;
  const bool bo = st.lay.hcap > 0;
  if (st.lay.beam <= 8)
    return bo ? launch_fused_kb<8, true>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s)
              : launch_fused_kb<8, false>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
  return bo ? launch_fused_kb<16, true>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s)
            : launch_fused_kb<16, false>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
}

}  // namespace ctcpb
