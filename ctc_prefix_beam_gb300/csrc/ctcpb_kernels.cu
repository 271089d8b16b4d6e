// Kernels of the GB300 CTC prefix beam search decoder.
//
// Paths follow "GPU CTC Prefix Beam Search Decoder" (OASR docs):
//   k_init      state reset (section 3.7's memsets, section 8's init)
//   k_select    frame selection by blank threshold, ordered compaction (3.5)
//   k_prepass   per-frame vocabulary ranking, hoisted out of the serial loop
//               (3.4.7): the first L non-blank labels by (lp desc, id asc)
//   k_step      one block per row: step-0 seeding (3.3), extension scoring
//               (3.4.1-3.4.2), prefix merge (3.4.3), top-beam selection
//               (3.4.4-3.4.5 / 3.4.6) and the token store update (flat
//               double-buffered rows or paged prefix-shared pages, 3.4.5, 4.2)
//   k_output    N-best gather (3.6)
#include <cstdio>
#include <cstring>

#include "ctcpb_async.cuh"
#include "ctcpb_internal.cuh"
#include "ctcpb_kernels.h"
#include "ctcpb_sort.cuh"

namespace ctcpb {

#define FULL 0xffffffffu

// Optional per-phase cycle accounting of the block step kernel (build with
// -DCTCPB_PHASE_PROF): thread 0's clock between marks, summed over rows.
#ifdef CTCPB_PHASE_PROF
#define BPHASE(i)                     \
  do {                                \
    const long long now_ = clock64(); \
    prof[i] += (u64)(now_ - prof_t0); \
    prof_t0 = now_;                   \
  } while (0)
#else
#define BPHASE(i) \
  do {            \
  } while (0)
#endif

// ------------------------------------------------------------------ helpers

template <int NT>
__device__ __forceinline__ void gsync() {
  if (NT == 32)
    __syncwarp();
  else
    __syncthreads();
}

template <int NT>
__device__ __forceinline__ bool g_any(bool p) {
  if (NT == 32) {
    return __any_sync(FULL, p);
  } else {
    return __syncthreads_or(p) != 0;
  }
}

// Bitonic sort (descending) of P keys, P a power of two, by a group of NT
// threads (a warp when NT == 32).  Ends with a group barrier.
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

// Block-wide descending ranks of 2*NT keys held two per thread (0: no key;
// the other keys are distinct).  Each warp sorts its 64 keys in registers
// (lane l then holds places l and l + 32 of its run) and writes the run to
// run[64 w ..]; a key's rank is its place in its own run plus, for every
// other run, the number of keys above it there (branch-free binary search).
// Ends with the keys in v (sorted within the warp) and their ranks in r.
template <int NT>
__device__ __forceinline__ void block_rank2(u64 (&v)[2], int (&r)[2], u64* run, int tid) {
  const int lane = tid & 31, w = tid >> 5;
  warp_sort_desc<2>(v, lane);
  r[0] = lane;
  r[1] = lane + 32;
  if (NT > 32) {
    run[64 * w + lane] = v[0];
    run[64 * w + 32 + lane] = v[1];
    gsync<NT>();
#pragma unroll
    for (int o = 1; o < NT / 32; ++o) {
      const u64* other = run + 64 * ((w + o) % (NT / 32));
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int c = 0;  // keys of `other` above v[e]: other is descending
#pragma unroll
        for (int step = 32; step >= 1; step >>= 1) c += other[c + step - 1] > v[e] ? step : 0;
        c += other[c] > v[e] ? 1 : 0;  // all 64 above
        r[e] += c;
      }
    }
  }
}

__device__ __forceinline__ int pow2_at_least(int n, int lo) {
  int p = lo;
  while (p < n) p <<= 1;
  return p;
}

__device__ __forceinline__ void set_status(const View& st, u32 bit) { atomicOr(&st.hdr()->status, bit); }

// ------------------------------------------------------------------ init

// The reset, spread over the launch's threads.
__device__ __forceinline__ void init_body(const View& st) {
  const Layout& L = st.lay;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthr = (size_t)gridDim.x * blockDim.x;
  if (tid == 0) {
    Header* h = st.hdr();
    h->magic = kMagic;
    h->version = kVersion;
    h->B = L.B; h->V = L.V; h->beam = L.beam; h->cap = L.cap; h->paged = L.paged;
    h->page_size = L.page_size; h->blank = L.blank; h->list_len = L.L; h->tile = L.tile; h->space = L.space;
    h->status = 0u;
    for (int i = 0; i < 5; ++i) h->counters[i] = 0u;
    for (int i = 0; i < 8; ++i) h->phase_cycles[i] = 0ull;
    h->fused_launches = 0u;
    h->hcap = L.hcap;
  }
  for (size_t b = tid; b < (size_t)L.B; b += nthr) {
    RowHdr r;
    r.step = 0; r.tcount = 0; r.t_prev = -1; r.nlive = 0; r.parity = 0; r.pending = 0;
    r.pad[0] = r.pad[1] = 0;
    st.rows()[b] = r;
    if (L.paged) {
      st.ptop()[b] = 0;
      st.pnext()[b] = 0;
    }
  }
  {
    const size_t nf = (size_t)L.B * L.tile;
    u32* rf = st.rflag();
    for (size_t i = tid; i < nf; i += nthr) rf[i] = 0u;
  }
  if (L.hcap > 0) {  // no label is boosted until a table is set
    const size_t nk = (size_t)L.B * L.hcap;
    int* bk = (int*)(st.base + L.o_bkey);
    for (size_t i = tid; i < nk; i += nthr) bk[i] = -1;
  }
  if (L.paged) {
    const size_t nt = 2 * (size_t)L.B * L.beam * L.max_lp;
    int* bt = (int*)(st.base + L.o_btab);
    for (size_t i = tid; i < nt; i += nthr) bt[i] = -1;
    const size_t np = (size_t)L.B * L.ppr;
    int* rc = (int*)(st.base + L.o_refc);
    for (size_t i = tid; i < np; i += nthr) rc[i] = 0;
  }
}

__global__ void k_init(View st) { init_body(st); }

// ------------------------------------------------------------------ label boosts
// Row b's label-boost hash table from entries [row_ptr[b], row_ptr[b+1]) of
// (tokens, bonus), taken in order by one thread (so a repeated label keeps its
// first bonus whatever the launch).  Rejected entries set CTCPB_DEV_BOOST.
__global__ void __launch_bounds__(64) k_boost_build(View st, const int* __restrict__ row_ptr,
                                                    const int* __restrict__ tokens, const float* __restrict__ bonus) {
  const Layout& L = st.lay;
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= L.B) return;
  if (!header_matches(st)) {
    set_status(st, CTCPB_DEV_HEADER);
    return;
  }
  const int hm = L.hcap - 1;
  int* keys = st.bkey(b);
  float* vals = st.bval(b);
  for (int i = 0; i <= hm; ++i) {
    keys[i] = -1;
    vals[i] = 0.0f;
  }
  const int lo = row_ptr[b], hi = row_ptr[b + 1];
  bool bad = lo < 0 || hi < lo;
  int n = 0;
  for (int e = bad ? hi : lo; e < hi; ++e) {
    const int c = tokens[e];
    const float v = bonus[e];
    if (n >= L.max_boost || c < 0 || c >= L.V || c == L.blank || !(fabsf(v) <= kMaxBonus)) {
      bad = true;
      continue;
    }
    int i = boost_slot(c, hm);
    while (keys[i] >= 0 && keys[i] != c) i = (i + 1) & hm;  // n < hcap / 2: an empty slot exists
    if (keys[i] == c) {
      bad = true;
      continue;
    }
    keys[i] = c;
    vals[i] = v;
    ++n;
  }
  if (bad) set_status(st, CTCPB_DEV_BOOST);
}

// ------------------------------------------------------------------ host-buffer decode plan
// plan[c * B + b] = the frames of row b in chunk c (chunks of F frames):
// clamp(len_b - c F, 0, F), len_b = clamp(lens[b], 0, T) (T when lens is null).
__global__ void k_host_plan(const int* __restrict__ lens, int B, int T, int F, int nchunks, int* __restrict__ plan) {
  const long long n = (long long)nchunks * B;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(i / B), b = (int)(i - (long long)c * B);
    int L = lens ? lens[b] : T;
    L = L < 0 ? 0 : (L > T ? T : L);
    int f = L - c * F;
    plan[i] = f < 0 ? 0 : (f > F ? F : f);
  }
}

// ------------------------------------------------------------------ select
// Section 3.5: keep t < len_b iff lp[b,t,blank] < log_thr (mode 1), all
// frames (mode 0) or none (mode 2); ordered compaction with warp ballots.
// Row b's selection by one block of 256 threads.
__device__ __forceinline__ void select_row(const View& st, int b, const float* __restrict__ lp, long long sb,
                                           long long stt, const int* __restrict__ lens, int T, int mode,
                                           float log_thr, int* __restrict__ sel, int* __restrict__ nsel) {
  __shared__ int wcount[8];
  __shared__ int base_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int len_b = lens ? lens[b] : T;
  len_b = len_b < 0 ? 0 : (len_b > T ? T : len_b);
  const int blank = st.lay.blank;
  if (tid == 0) base_s = 0;
  __syncthreads();
  for (int t0 = 0; t0 < T; t0 += 256) {
    const int t = t0 + tid;
    bool keep = false;
    if (t < len_b) {
      if (mode == 0)
        keep = true;
      else if (mode == 1)
        keep = rdlp(lp[(long long)b * sb + (long long)t * stt + blank]) < log_thr;
    }
    unsigned m = __ballot_sync(FULL, keep);
    if (lane == 0) wcount[wid] = __popc(m);
    __syncthreads();
    int off = base_s;
    for (int w = 0; w < wid; ++w) off += wcount[w];
    if (keep) sel[(size_t)b * T + off + __popc(m & ((1u << lane) - 1u))] = t;
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int w = 0; w < 8; ++w) tot += wcount[w];
      base_s += tot;
    }
    __syncthreads();
  }
  const int n = base_s;
  for (int i = n + tid; i < T; i += 256) sel[(size_t)b * T + i] = -1;
  if (tid == 0) nsel[b] = n;
}

__global__ void __launch_bounds__(256) k_select(View st, const float* __restrict__ lp, long long sb, long long stt,
                                                const int* __restrict__ lens, int T, int mode, float log_thr,
                                                int* __restrict__ sel, int* __restrict__ nsel) {
  select_row(st, blockIdx.x, lp, sb, stt, lens, T, mode, log_thr, sel, nsel);
}

// The reset and the selection in one launch (they touch disjoint memory):
// blocks b < B also select row b.
__global__ void __launch_bounds__(256) k_init_select(View st, const float* __restrict__ lp, long long sb,
                                                     long long stt, const int* __restrict__ lens, int T, int mode,
                                                     float log_thr, int* __restrict__ sel, int* __restrict__ nsel) {
  init_body(st);
  if ((int)blockIdx.x < st.lay.B) select_row(st, blockIdx.x, lp, sb, stt, lens, T, mode, log_thr, sel, nsel);
}

// Speech-masked streaming: the chunk rows of tile [tile_start, tile_start +
// tile_len) that stream b decodes (mask != 0), in order, into sel/nsel.  One
// warp per stream.
// Without a mask the rows are kept by the blank threshold of section 3.5
// instead: lp[b, j, blank] < log_thr, read from the chunk (lp, sb, stt).
__global__ void __launch_bounds__(32) k_select_tile(View st, const uint8_t* __restrict__ mask, long long mstride,
                                                    const float* __restrict__ lp, long long sb, long long stt,
                                                    float log_thr, const int* __restrict__ nframes, int chunk_T,
                                                    int tile_start, int tile_len) {
  const int b = blockIdx.x, lane = threadIdx.x;
  int nf = nframes ? nframes[b] : chunk_T;
  nf = nf < 0 ? 0 : (nf > chunk_T ? chunk_T : nf);
  const int end = tile_start + tile_len < nf ? tile_start + tile_len : nf;
  int* sel = st.sel() + (size_t)b * st.lay.T_sel;
  int n = 0;
  for (int j0 = tile_start; j0 < end; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false;
    if (j < end)
      keep = mask ? mask[(long long)b * mstride + j] != 0
                  : rdlp(lp[(long long)b * sb + (long long)j * stt + st.lay.blank]) < log_thr;
    const unsigned m = __ballot_sync(FULL, keep);
    if (keep) sel[n + __popc(m & ((1u << lane) - 1u))] = j;
    n += __popc(m);
  }
  if (lane == 0) st.nsel()[b] = n;
}

// ------------------------------------------------------------------ step
//
// One block of NT threads owns one row for the whole call.  The beam state of
// the row lives in shared memory between steps; tokens live in the state
// buffer (flat rows or pages).
template <int NT>
struct StepSmem {
  float fc[kFCoef];  // the coefficients of log(1 + e^-d) (dlse)
  // current hypotheses, slot order
  float pb[NT], pnb[NT], sc[NT];
  int last[NT], len[NT];
  u64 h[NT], hp[NT];
  // per step
  float A[NT], pbg[NT], lpl[NT], lple[NT], bpb[NT], bpnb[NT], rep[NT];  // lple: lp[last] as emitted (boosted)
  int into[NT], repdead[NT];
  // next hypotheses
  float npb[NT], npnb[NT], nsc[NT];
  int nlast[NT], nlen[NT], nsrc[NT], ntok[NT];
  u64 nh[NT], nhp[NT];
  // the ranked-frame records of this step and the next (raw copies: header,
  // ids, log-probs), and lp[frame][last] of every slot for those steps
  static constexpr int kRecMax = 32 + 8 * ((kMaxList + 3) / 4 * 4);
  alignas(16) unsigned char rec[2][kRecMax];
  float lplf[2][NT];
  // the step's list positions by label: key (decode step + 1) << 32 | label
  // (older steps' keys read as empty), open addressing
  static constexpr int kLpos = 1024;  // a power of two >= 2 * list length
  u64 lpkey[kLpos];
  int lpval[kLpos];
  u32 excl[NT][(kMaxList + 31) / 32];
  int xu_k[NT], xu_c[NT];
  int pi[2 * NT], pj[2 * NT];
  int dfree[NT];
  u64 top2[2 * NT];  // each hypothesis' best two candidate keys
  // merge sources: slot i with l_k = l_i + last_k (or -1), tracked through the winners' sources
  int msrc[NT], nmsrc[NT], bw[NT];
  u64 hkey[2 * NT];   // the extension winners' prefix hashes (open addressing) ...
  int hval[2 * NT];   // ... and their slots (-1: empty)
  int npg[2][NT];     // paged: pages held by slot w of each parity's block table
  // the step history since the token store was last written (ring row r =
  // step win0 + r, entry w = source slot << 24 | token of winner w), and per
  // slot the stored slot it descends from and how many of its labels that
  // slot holds
  static constexpr int R = kBlockRing;
  u32 hist[R][NT];
  int org[NT], lo[NT], norg[NT], nlo[NT];
  int uc[8 * NT];      // frame scan: unlisted labels that can reach the threshold ...
  float uv[8 * NT];    // ... and their log-probs
  u64 tau;  // the step's selection threshold
  int nw, npairs, nxu, nkeys, ndfree, nuc;
  int ptop, pnext;  // the row's page pool: LIFO top and bump pointer (paged)
};

__device__ const FCoef g_fcoef = make_fcoef();

template <int NT>
size_t step_smem_bytes(int sortcap) {
  return align_up(sizeof(StepSmem<NT>), 16) + (size_t)sortcap * sizeof(u64);
}

struct TokenStore {
  View st;
  int b;
  __device__ __forceinline__ int get(int par, int k, int x) const {
    if (!st.lay.paged) return st.clist(par, b, k)[x];
    const int ps = st.lay.page_size;
    const int phys = st.btab(par, b, k)[x / ps];
    return phys >= 0 ? st.page(b, phys)[x % ps] : -1;
  }
};

// The row's page pool (only the row's block touches it): the LIFO top and the
// bump pointer live in shared memory during a call, the stack in the state.
// Allocate one page: LIFO pool first, then the bump pointer.  Allocations and
// releases never run in the same phase of a step.
__device__ int page_alloc(const View& st, int b, int* ptop, int* pnext) {
  const int pos = atomicSub(ptop, 1) - 1;  // may go below zero; the phase end clamps it
  if (pos >= 0) {
    if (pos >= st.lay.ppr) {
      set_status(st, CTCPB_DEV_OVERFLOW);
      return -1;
    }
    return st.pool(b)[pos];
  }
  const int phys = atomicAdd(pnext, 1);
  if (phys >= st.lay.ppr) {
    set_status(st, CTCPB_DEV_PAGES);
    return -1;
  }
  return phys;
}

__device__ __forceinline__ void page_push(const View& st, int b, int phys, int* ptop) {
  const int pos = atomicAdd(ptop, 1);
  if (pos < st.lay.ppr)
    st.pool(b)[pos] = phys;
  else
    set_status(st, CTCPB_DEV_OVERFLOW);
}

// Flat rows: write every next slot w < nw into the rows of parity par ^ 1 --
// its origin row's first nlo[w] labels (parity par) followed by the labels it
// gained in ring rows 0..nrows-1, found by walking its sources backwards --
// then make each slot its own origin.  Ends with a group barrier.
template <int NT>
__device__ void flush_flat(StepSmem<NT>& S, const View& st, int b, int par, int nrows, int nw, int blank, int tid) {
  const int to = par ^ 1;
  const int lw = st.lay.ldseq >> 2;  // 16-byte words per row
  // whole words of the origin prefixes, four independent copies in flight
  for (int i0 = 0; i0 < nw * lw; i0 += 4 * NT) {
    int4 v[4];
    int dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * NT + tid;
      dst[u] = -1;
      if (i < nw * lw) {
        const int w = i / lw, x = i - w * lw;
        const int o = S.norg[w];
        if (o >= 0 && 4 * x + 4 <= S.nlo[w]) {
          v[u] = reinterpret_cast<const int4*>(st.clist(par, b, o))[x];
          dst[u] = i;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] >= 0) {
        const int w = dst[u] / lw, x = dst[u] - w * lw;
        reinterpret_cast<int4*>(st.clist(to, b, w))[x] = v[u];
      }
  }
  // every word copy has read its slot's origin and length before the owners
  // below reset them
  gsync<NT>();
  // the prefix tail after the last whole word, then the gained labels
  for (int w = tid; w < nw; w += NT) {
    const int o = S.norg[w], l0 = S.nlo[w];
    int* row = st.clist(to, b, w);
    if (o >= 0) {
      const int* from = st.clist(par, b, o);
      for (int x = l0 & ~3; x < l0; ++x) row[x] = from[x];
    }
    int slot = w, rem = S.nlen[w] - l0;
    for (int r = nrows - 1; r >= 0 && rem > 0; --r) {
      const u32 e = S.hist[r][slot];
      const int tk = (int)(e & 0xffffffu);
      if (tk != blank) row[l0 + --rem] = tk;
      slot = (int)(e >> 24);
    }
    S.norg[w] = w;
    S.nlo[w] = S.nlen[w];
  }
  gsync<NT>();
}

// Paged storage: the same write into the block tables of parity par ^ 1.
// Slot w's table takes its origin's pages (parity par; reference counts change
// only for entries that differ from what the slot held), then the labels it
// gained go to a copy of the origin's partial last page (the origin's table
// still holds the original) and to new pages.  Ends with a group barrier.
template <int NT>
__device__ void flush_paged(StepSmem<NT>& S, const View& st, int b, int par, int nrows, int nw, int blank, int tid) {
  const int to = par ^ 1, ps = st.lay.page_size, beam = st.lay.beam;
  int* refc = st.refc(b);
  // pass A: acquire (a thread per slot)
  for (int w = tid; w < nw; w += NT) {
    const int o = S.norg[w];
    const int nn = o >= 0 ? (S.nlo[w] + ps - 1) / ps : 0, no = S.npg[to][w];
    const int* bs = st.btab(par, b, o >= 0 ? o : 0);
    const int* bd = st.btab(to, b, w);
#pragma unroll 4
    for (int x = 0; x < nn; ++x) {
      const int nv = bs[x], ov = x < no ? bd[x] : -1;
      if (nv >= 0 && nv != ov) atomicAdd(&refc[nv], 1);
    }
  }
  if (tid == 0) S.ndfree = 0;
  gsync<NT>();
  // pass B: release what changed, install the origin's pages
  for (int w = tid; w < beam; w += NT) {
    const int o = w < nw ? S.norg[w] : -1;
    const int nn = o >= 0 ? (S.nlo[w] + ps - 1) / ps : 0, no = S.npg[to][w];
    const int* bs = st.btab(par, b, o >= 0 ? o : 0);
    int* bd = st.btab(to, b, w);
    const int m = nn > no ? nn : no;
#pragma unroll 4
    for (int x = 0; x < m; ++x) {
      const int nv = x < nn ? bs[x] : -1, ov = x < no ? bd[x] : -1;
      if (ov >= 0 && ov != nv && atomicSub(&refc[ov], 1) == 1) page_push(st, b, ov, &S.ptop);
      bd[x] = nv;
    }
    S.npg[to][w] = nn;
  }
  gsync<NT>();
  // pass C: pages for the gained labels, then the labels (ring walk)
  for (int w = tid; w < nw; w += NT) {
    const int l0 = S.nlo[w], l1 = S.nlen[w];
    if (l1 > l0) {
      int* bd = st.btab(to, b, w);
      const int x0 = l0 / ps, off = l0 - x0 * ps;
      bool ok = true;  // false: a shared page could not be copied; nothing is written into it
      if (off != 0) {
        const int phys = bd[x0];
        if (phys >= 0) {
          const int nph = page_alloc(st, b, &S.ptop, &S.pnext);
          if (nph >= 0) {
            const int* from = st.page(b, phys);
            int* top = st.page(b, nph);
            for (int y = 0; y < off; ++y) top[y] = from[y];
            refc[nph] = 1;
            bd[x0] = nph;
            if (atomicSub(&refc[phys], 1) == 1) S.dfree[atomicAdd(&S.ndfree, 1)] = phys;
          } else {
            ok = false;
          }
        }
      }
      int xe = (l1 - 1) / ps;  // the table ends at the first page that could not be had
      for (int y = off != 0 ? x0 + 1 : x0; y <= xe; ++y) {
        const int phys = page_alloc(st, b, &S.ptop, &S.pnext);
        if (phys < 0) {
          xe = y - 1;
          break;
        }
        refc[phys] = 1;
        bd[y] = phys;
      }
      S.npg[to][w] = xe + 1;
      int slot = w, rem = l1 - l0;
      for (int r = nrows - 1; r >= 0 && rem > 0; --r) {
        const u32 e = S.hist[r][slot];
        const int tk = (int)(e & 0xffffffu);
        if (tk != blank) {
          const int pos = l0 + --rem, y = pos / ps;
          const int phys = bd[y];
          if (phys >= 0 && (ok || y != x0)) st.page(b, phys)[pos - y * ps] = tk;
        }
        slot = (int)(e >> 24);
      }
    }
    S.norg[w] = w;
    S.nlo[w] = l1;
  }
  gsync<NT>();
  if (tid == 0 && S.ptop < 0) S.ptop = 0;  // allocations past an empty pool
  gsync<NT>();
  for (int q = tid; q < S.ndfree; q += NT) page_push(st, b, S.dfree[q], &S.ptop);
  gsync<NT>();
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) k_step(View st, const float* __restrict__ lp, long long sb, long long stt,
                                             int mode, const int* __restrict__ nframes, int chunk_T,
                                             int tile_start, int tile_len, int sortcap) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  StepSmem<NT>& S = *reinterpret_cast<StepSmem<NT>*>(smem_raw);
  u64* keys = reinterpret_cast<u64*>(smem_raw + align_up(sizeof(StepSmem<NT>), 16));
  const Layout& Ly = st.lay;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int beam = Ly.beam, cap = Ly.cap, blank = Ly.blank, V = Ly.V;
  const int space = Ly.space;  // word-boundary label, -1: none
  const float NEG = CTCPB_NEG;
  // the row's label-boost table (null: no boosting)
  const int* bkeys = Ly.hcap > 0 ? st.bkey(b) : nullptr;
  const float* bvals = Ly.hcap > 0 ? st.bval(b) : nullptr;
  const int hmask = Ly.hcap - 1;

  if (mode != 0) {
    const Header* hd = st.hdr();
    bool ok = hd->magic == kMagic && hd->version == kVersion && hd->B == Ly.B && hd->V == Ly.V &&
              hd->beam == Ly.beam && hd->cap == Ly.cap && hd->paged == Ly.paged &&
              hd->page_size == Ly.page_size && hd->blank == Ly.blank && hd->list_len == Ly.L &&
              hd->tile == Ly.tile && hd->space == Ly.space && hd->hcap == Ly.hcap;
    if (!ok) {
      if (tid == 0) set_status(st, CTCPB_DEV_HEADER);
      return;
    }
  }

  RowHdr* rh = st.rows() + b;
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
    if (mode == 2 && tid == 0) rh->tcount += nft;  // every frame of the tile was skipped
    return;
  }

  int step = rh->step, tcount = rh->tcount, t_prev = rh->t_prev, nlive = rh->nlive, par = rh->parity;
  const size_t rb = (size_t)b * beam;
  for (int k = tid; k < beam; k += NT) {
    S.pb[k] = st.pb()[rb + k];
    S.pnb[k] = st.pnb()[rb + k];
    S.sc[k] = st.sc()[rb + k];
    S.last[k] = st.last()[rb + k];
    S.len[k] = st.len()[rb + k];
    S.h[k] = st.h()[rb + k];
    S.hp[k] = st.hp()[rb + k];
    S.msrc[k] = st.msrc()[rb + k];
    S.org[k] = k;
    S.lo[k] = S.len[k];
  }
  int win0 = 0;  // flat rows: the call step of ring row 0
  if (Ly.paged) {
    for (int k = tid; k < 2 * beam; k += NT) {
      const int pp = k / beam, w = k - pp * beam;
      const int* bt = st.btab(pp, b, w);
      int n = 0;
      while (n < Ly.max_lp && bt[n] >= 0) ++n;
      S.npg[pp][w] = n;
    }
  }
  TokenStore tok{st, b};
  const int M = sortcap - NT;  // candidates per selection chunk
  // decode steps, unlisted-label scans, overflow (chunked) selections,
  // hash-proposed merges confirmed
  u32 c_steps = 0, c_scan = 0, c_exh = 0, c_hash = 0;
#ifdef CTCPB_PHASE_PROF
  u64 prof[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  long long prof_t0 = clock64();
#endif
  if (Ly.paged && tid == 0) {
    S.ptop = st.ptop()[b];
    S.pnext = st.pnext()[b];
  }
  for (int i = tid; i < S.kLpos; i += NT) S.lpkey[i] = 0ull;
  for (int i = tid; i < kFCoef; i += NT) S.fc[i] = g_fcoef.c[i];
  gsync<NT>();

  // Asynchronous copies that step s waits for at its start: its record into
  // rec[s & 1] (issued at the start of step s-1) and lp[its frame][last] of
  // its n slots into lplf[s & 1] (issued once step s-1 has chosen them:
  // lasts/lens are the slots' last labels and lengths).
  const int rwords = (int)(Ly.rec_bytes >> 4);
  auto prefetch_rec = [&](int s) {
    const char* src = st.rec(b, s);
    unsigned char* dst = S.rec[s & 1];
    for (int i = tid; i < rwords; i += NT) cp_async16(dst + 16 * i, src + 16 * i);
    cp_commit();
  };
  auto prefetch_lpl = [&](int s, int srow, int n, const int* lasts, const int* lens) {
    const float* frow = lp + (long long)b * sb + (long long)srow * stt;
    for (int k = tid; k < n; k += NT)
      if (lens[k] > 0) cp_async4(&S.lplf[s & 1][k], frow + lasts[k]);
    cp_commit();
  };
  auto srow_of = [&](int s) { return mode != 1 ? st.sel()[(size_t)b * Ly.T_sel + s] : tile_start + s; };
  int srow_next = srow_of(0);  // the batch or chunk row of the coming step
  prefetch_rec(0);
  prefetch_lpl(0, srow_next, nlive, S.last, S.len);

  for (int s = 0; s < nsteps; ++s) {
    const int srow = srow_next;  // batch or chunk row
    const int t = mode == 0 ? srow : (mode == 1 ? tcount + s : tcount + srow - tile_start);
    const float* row = lp + (long long)b * sb + (long long)srow * stt;
    cp_wait_all();
    gsync<NT>();
    if (s + 1 < nsteps) prefetch_rec(s + 1);  // rec[(s+1) & 1] was step s-1's, done
    if (s + 1 < nsteps) srow_next = srow_of(s + 1);  // used at the winners: its load has time
    BPHASE(0);
    const unsigned char* rbuf = S.rec[s & 1];
    const RecHdr& rhd = *reinterpret_cast<const RecHdr*>(rbuf);
    const int* ids = reinterpret_cast<const int*>(rbuf + 32);
    const float* lps = reinterpret_cast<const float*>(rbuf + 32 + 4 * Ly.Lpad);
    const float* lplf = S.lplf[s & 1];
    const float rec_lpb = rhd.lpb, front_lp = rhd.front_lp;
    const int front_id = rhd.front_id;
    const bool gap = t > t_prev + 1;
    const int cnt = rhd.cnt;

    if (step == 0) {
      // ---- section 3.3: seed the top (beam-1) labels, then the empty prefix
      const int nb = beam > 1 ? beam - 1 : 1;
      const int ntok = cap >= 1 ? (nb < cnt ? nb : cnt) : 0;
      const bool empty_live = beam > 1 && rec_lpb > NEG;
      for (int k = tid; k < beam; k += NT) {
        if (k < ntok) {
          const int c = ids[k];
          const float v = lps[k];
          S.npb[k] = gap ? v : NEG;
          S.npnb[k] = gap ? NEG : v;
          S.nsc[k] = v;
          S.nlast[k] = c;
          S.nlen[k] = 1;
          S.nh[k] = hmix(kH0, c);
          S.nhp[k] = kH0;
          S.ntok[k] = c;
          S.nsrc[k] = -1;
          S.nmsrc[k] = empty_live ? ntok : -1;  // l_k = empty prefix + c
        } else if (k == ntok && empty_live) {
          S.npb[k] = rec_lpb;
          S.npnb[k] = NEG;
          S.nsc[k] = rec_lpb;
          S.nlast[k] = blank;
          S.nlen[k] = 0;
          S.nh[k] = kH0;
          S.nhp[k] = 0ull;
          S.ntok[k] = blank;
          S.nsrc[k] = -1;
          S.nmsrc[k] = -1;
        }
      }
      if (tid == 0) S.nw = ntok + (empty_live ? 1 : 0);
      gsync<NT>();
      const int nw = S.nw;
      for (int k = tid; k < nw; k += NT) {
        S.hist[s - win0][k] = (u32)S.ntok[k] & 0xffffffu;
        S.norg[k] = -1;
        S.nlo[k] = 0;
      }
      gsync<NT>();
    } else {
      // ---- section 3.4: collapsed-blank correction, extension and blank slots
      for (int k = tid; k < nlive; k += NT) {
        float pb = S.pb[k], pnb = S.pnb[k];
        if (gap) {
          pb = dlse(S.fc, pb, pnb);
          pnb = NEG;
        }
        const float A = dlse(S.fc, pb, pnb);
        const int L = S.len[k];
        const float lpl = L > 0 ? rdlp(lplf[k]) : NEG;
        // the last label emitted again (the repeat path, a merge fold) carries its bonus
        const float lple = (L > 0 && bkeys) ? dadd(lpl, boost_of(bkeys, bvals, hmask, S.last[k])) : lpl;
        S.A[k] = A;
        S.pbg[k] = pb;
        S.lpl[k] = lpl;
        S.lple[k] = lple;
        S.bpb[k] = dadd(rec_lpb, A);
        // a space-ending beam has no stay path, and its candidate (k, last)
        // extends from both paths (every space frame is a token)
        const bool spc = S.last[k] == space;
        S.bpnb[k] = (L > 0 && !gap && !spc) ? dadd(lpl, pnb) : NEG;
        S.rep[k] = (L > 0 && L < cap) ? dadd(lple, spc ? A : pb) : NEG;
        S.repdead[k] = 0;
        // section 3.4.3: pairs (i shorter, j longer) with l_j = l_i + last_j,
        // known from the merge sources tracked through the previous steps
        S.into[k] = S.msrc[k];
        for (int w = 0; w < (kMaxList + 31) / 32; ++w) S.excl[k][w] = 0u;
      }
      for (int k = tid; k < NT; k += NT) S.bw[k] = -1;
      // the list positions by label, for the folds (short lists are searched)
      const u64 stamp = (u64)(step + 1);
      const bool lpos = cnt > 96;
      for (int p = tid; lpos && p < cnt; p += NT) {
        const int c = ids[p];
        int h = (int)(((u32)c * 0x9E3779B1u) & (u32)(S.kLpos - 1));
        for (int n = 0; n < S.kLpos; ++n) {  // the table is at most half full
          const u64 old = S.lpkey[h];
          if ((old >> 32) != stamp && atomicCAS(&S.lpkey[h], old, (stamp << 32) | (u32)c) == old) {
            S.lpval[h] = p;
            break;
          }
          if ((S.lpkey[h] >> 32) == stamp) h = (h + 1) & (S.kLpos - 1);
        }
      }
      if (tid == 0) {
        S.npairs = 0;
        S.nxu = 0;
        S.nkeys = 0;
      }
      gsync<NT>();
      // fold (i, last_j) into j's blank slot; drop the folded candidate
      for (int j = tid; j < nlive; j += NT) {
        const int i = S.into[j];
        if (i < 0) continue;
        const int c = S.last[j];
        const bool same = S.len[i] > 0 && S.last[i] == c;  // the folded candidate is i's (i, last) entry
        const bool rep_i = same && c != space;
        const float ext = rep_i ? dadd(S.lple[j], S.pbg[i]) : dadd(S.lple[j], S.A[i]);
        S.bpnb[j] = dlse(S.fc, S.bpnb[j], ext);
        if (same) {
          S.repdead[i] = 1;
        } else {
          int p = -1;  // c's list position
          if (!lpos) {
            for (int q = 0; q < cnt; ++q)
              if (ids[q] == c) {
                p = q;
                break;
              }
          }
          for (int h = (int)(((u32)c * 0x9E3779B1u) & (u32)(S.kLpos - 1)), n = 0; lpos && n < S.kLpos;
               h = (h + 1) & (S.kLpos - 1), ++n) {
            const u64 k2 = S.lpkey[h];
            if ((k2 >> 32) != stamp) break;
            if ((u32)k2 == (u32)c) {
              p = S.lpval[h];
              break;
            }
          }
          if (p >= 0) {
            atomicOr(&S.excl[i][p >> 5], 1u << (p & 31));
          } else {
            int u = atomicAdd(&S.nxu, 1);
            S.xu_k[u] = i;
            S.xu_c[u] = c;
          }
        }
      }
      gsync<NT>();
      BPHASE(1);

      // ---- sections 3.4.4-3.4.6: best `beam` candidates over
      // {blank slot, repeat slot, listed labels} of every live hypothesis.
      // Thread k = hypothesis k (nlive <= beam <= NT).  Its listed candidates
      // score in list order, so its keys are (blank, repeat, listed ones in
      // order).  tau = the beam-th largest of every hypothesis' best two keys
      // is at most the beam-th largest key of the step (those are distinct
      // candidates), so the winners are among the candidates >= tau.
      auto blank_key = [&](int k) -> u64 {
        const float sc = dlse(S.fc, S.bpb[k], S.bpnb[k]);
        return sc > NEG ? cand_key(sc, k, blank) : 0ull;
      };
      auto rep_key = [&](int k) -> u64 {
        const int L = S.len[k];
        return (L > 0 && L < cap && !S.repdead[k] && S.rep[k] > NEG) ? cand_key(S.rep[k], k, S.last[k]) : 0ull;
      };
      auto list_key = [&](int k, int p) -> u64 {  // 0: not a candidate
        const int L = S.len[k];
        const int c = ids[p];
        if (L < cap && !(L > 0 && c == S.last[k]) && !((S.excl[k][p >> 5] >> (p & 31)) & 1u)) {
          const float sc = dadd(lps[p], S.A[k]);
          if (sc > NEG) return cand_key(sc, k, c);
        }
        return 0ull;
      };
      bool selected = false;
      int nsel = 0;  // the winners, when the rank paths selected (keys are nonzero and distinct)
      {
        u64 kb = 0ull, kr = 0ull, ka = 0ull, kc = 0ull;
        if (tid < nlive) {
          kb = blank_key(tid);
          kr = rep_key(tid);
          for (int p = 0, got = 0; p < cnt && got < 2; ++p) {
            const u64 key = list_key(tid, p);
            if (key) {
              if (got == 0) ka = key; else kc = key;
              ++got;
            }
          }
        }
        // best two of {kb, kr, ka, kc}
        u64 m1 = kb > kr ? kb : kr, m2 = kb > kr ? kr : kb;
        if (ka > m1) { m2 = m1; m1 = ka; } else if (ka > m2) { m2 = ka; }
        if (kc > m1) { m2 = m1; m1 = kc; } else if (kc > m2) { m2 = kc; }
        if (tid == 0) {
          S.nkeys = 0;
          S.tau = 0ull;  // every live key when fewer than beam are live
        }
        // tau: the key that exactly beam-1 of the 2 nlive keys exceed (live
        // keys are distinct: score, source, token).  Up to 128 keys each
        // counts the keys above it; more are sorted per warp and searched.
        if (2 * nlive <= 128) {
          S.top2[2 * tid] = m1;
          S.top2[2 * tid + 1] = m2;
          gsync<NT>();
          if (tid < nlive) {
            int r1 = 0, r2 = 0;
            for (int j = 0; j < 2 * nlive; ++j) {
              const u64 y = S.top2[j];
              r1 += y > m1 ? 1 : 0;
              r2 += y > m2 ? 1 : 0;
            }
            if (m1 != 0ull && r1 == beam - 1) S.tau = m1;
            if (m2 != 0ull && r2 == beam - 1) S.tau = m2;
          }
        } else {
          gsync<NT>();
          u64 v2[2] = {m1, m2};
          int r2[2];
          block_rank2<NT>(v2, r2, S.top2, tid);
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (v2[e] != 0ull && r2[e] == beam - 1) S.tau = v2[e];
        }
        gsync<NT>();
        const u64 tau = S.tau;
        // every candidate >= tau (the listed ones stop at the first below tau)
        const int cap_keys = sortcap;
        if (tid < nlive) {
          const u64 c0 = blank_key(tid), c1 = rep_key(tid);
          if (c0 && c0 >= tau) { const int q = atomicAdd(&S.nkeys, 1); if (q < cap_keys) keys[q] = c0; }
          if (c1 && c1 >= tau) { const int q = atomicAdd(&S.nkeys, 1); if (q < cap_keys) keys[q] = c1; }
          for (int p = 0; p < cnt; ++p) {
            const u64 key = list_key(tid, p);
            if (!key) continue;
            // scores fall along the list; equal scores may come in any token order
            if ((key >> 32) < (tau >> 32)) break;
            if (key < tau) continue;
            const int q = atomicAdd(&S.nkeys, 1);
            if (q < cap_keys) keys[q] = key;
          }
        }
        gsync<NT>();
        const int nk = S.nkeys;
        if (nk <= NT) {
          // the best beam in order by rank: each key counts the keys above it
          const u64 mk = tid < nk ? keys[tid] : 0ull;
          int mr = 0;
          for (int j = 0; j < nk; ++j) mr += keys[j] > mk ? 1 : 0;
          gsync<NT>();
          if (mk != 0ull && mr < beam) keys[mr] = mk;
          // the rest of the first NT slots holds no key (a frame scan sorts them)
          for (int i = (nk < beam ? nk : beam) + tid; i < NT; i += NT) keys[i] = 0ull;
          selected = true;
          nsel = nk < beam ? nk : beam;
        } else if (nk <= 2 * NT) {
          // the best beam in order: block-wide ranks of the collected keys
          u64 v2[2];
          int r2[2];
          const int i0 = 64 * (tid >> 5) + (tid & 31);
          v2[0] = i0 < nk ? keys[i0] : 0ull;
          v2[1] = i0 + 32 < nk ? keys[i0 + 32] : 0ull;
          block_rank2<NT>(v2, r2, S.top2, tid);
          gsync<NT>();  // every key is read before the first is placed
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (v2[e] != 0ull && r2[e] < beam) keys[r2[e]] = v2[e];
          // the rest of the first NT slots holds no key (a frame scan sorts them)
          for (int i = (nk < beam ? nk : beam) + tid; i < NT; i += NT) keys[i] = 0ull;
          selected = true;
          nsel = nk < beam ? nk : beam;
        } else if (nk <= 4 * NT) {
          // the best beam in order by rank: each key counts the keys above it
          u64 mk[4];
          int mr[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = tid + u * NT;
            mk[u] = i < nk ? keys[i] : 0ull;
            mr[u] = 0;
          }
          for (int j = 0; j < nk; ++j) {
            const u64 y = keys[j];
#pragma unroll
            for (int u = 0; u < 4; ++u) mr[u] += y > mk[u] ? 1 : 0;
          }
          gsync<NT>();
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (mk[u] != 0ull && mr[u] < beam) keys[mr[u]] = mk[u];
          // the rest of the first NT slots holds no key (a frame scan sorts them)
          for (int i = (nk < beam ? nk : beam) + tid; i < NT; i += NT) keys[i] = 0ull;
          selected = true;
        } else if (nk <= cap_keys) {
          const int P = pow2_at_least(nk > beam ? nk : beam, 2 * NT);
          for (int i = nk + tid; i < P; i += NT) keys[i] = 0ull;
          gsync<NT>();
          bitonic_desc<NT>(keys, P, tid);
          selected = true;
        }
        gsync<NT>();
        if (tid == 0) S.nkeys = 0;
        gsync<NT>();
      }
      c_exh += selected ? 0u : 1u;
      const int stride = cnt + 2;
      const int NC = selected ? 0 : nlive * stride;  // the chunked sort of every candidate (overflow only)
      if (!selected)
        for (int i = tid; i < NT; i += NT) keys[i] = 0ull;
      for (int base = 0; base < NC; base += M) {
        const int m = (NC - base) < M ? (NC - base) : M;
        for (int x = tid; x < m; x += NT) {
          const int g = base + x;
          const int k = g / stride, r = g - k * stride;
          u64 key = 0ull;
          const int L = S.len[k];
          if (r == 0) {
            const float sc = dlse(S.fc, S.bpb[k], S.bpnb[k]);
            if (sc > NEG) key = cand_key(sc, k, blank);
          } else if (r == 1) {
            if (L > 0 && L < cap && !S.repdead[k] && S.rep[k] > NEG) key = cand_key(S.rep[k], k, S.last[k]);
          } else {
            const int p = r - 2;
            const int c = ids[p];
            if (L < cap && !(L > 0 && c == S.last[k]) && !((S.excl[k][p >> 5] >> (p & 31)) & 1u)) {
              const float sc = dadd(lps[p], S.A[k]);
              if (sc > NEG) key = cand_key(sc, k, c);
            }
          }
          keys[NT + x] = key;
        }
        const int P = pow2_at_least(NT + m, 2 * NT);
        for (int i = NT + m + tid; i < P; i += NT) keys[i] = 0ull;
        gsync<NT>();
        bitonic_desc<NT>(keys, P, tid);
      }
      int nw = nsel;
      if (nsel == 0)
        for (int w = 0; w < beam; ++w) nw += keys[w] != 0ull;
      BPHASE(2);

      // ---- the list proves the selection unless an unlisted label could
      // reach the beam: then rank every unlisted label of this frame
      if (front_lp > NEG) {
        const u32 sstar = nw == beam ? (u32)(keys[beam - 1] >> 32) : 0u;
        bool bad = false;
        for (int k = tid; k < nlive; k += NT) {
          if (S.len[k] < cap) {
            const float u = dadd(front_lp, S.A[k]);
            if (u > NEG && (nw < beam || fkey(u) >= sstar)) bad = true;
          }
        }
        const bool need = g_any<NT>(bad);
        if (need) {
          ++c_scan;
          // One pass over the frame: an unlisted label is worth scoring only
          // if it reaches the threshold with the largest A of a hypothesis
          // that can grow (adding is monotone), so only those labels are
          // kept and then paired with every hypothesis.
          u64 thr = nw == beam ? (keys[beam - 1] & 0xffffffff00000000ull) : 0ull;
          const u64 kfront = lab_key(front_lp, front_id);
          float amax = NEG;
          for (int k = 0; k < nlive; ++k)
            if (S.len[k] < cap) amax = fmaxf(amax, S.A[k]);
          if (tid == 0) S.nuc = 0;
          gsync<NT>();
          for (int c0 = 0; c0 < V; c0 += 4 * NT) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + u * NT + tid;
              v[u] = c < V ? rdlp(row[c]) : NEG;
            }
            if (bkeys) {  // labels as emitted: the list ranks them by the boosted log-prob
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * NT + tid;
                if (c < V) v[u] = dadd(v[u], boost_of(bkeys, bvals, hmask, c));
              }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + u * NT + tid;
              if (c < V && c != blank && v[u] > NEG && lab_key(v[u], c) <= kfront &&
                  ((u64)fkey(dadd(v[u], amax)) << 32) >= thr) {
                const int q = atomicAdd(&S.nuc, 1);  // < 8 NT: flushed above 4 NT
                S.uc[q] = c;
                S.uv[q] = v[u];
              }
            }
            gsync<NT>();
            const int nl = S.nuc;
            const bool last_round = c0 + 4 * NT >= V;
            if (nl > 4 * NT || (last_round && nl > 0)) {
              // pair the kept labels with every hypothesis, NT pairs a round
              const int items = nlive * nl;
              for (int base = 0; base < items; base += NT) {
                const int x = base + tid;
                if (x < items) {
                  const int k = x / nl, j = x - k * nl;
                  const int c = S.uc[j], L = S.len[k];
                  if (L < cap && !(L > 0 && c == S.last[k])) {
                    bool ex = false;
                    for (int u = 0; u < S.nxu; ++u) ex |= (S.xu_k[u] == k && S.xu_c[u] == c);
                    const float sc = dadd(S.uv[j], S.A[k]);
                    if (!ex && sc > NEG) {
                      const u64 key = cand_key(sc, k, c);
                      if (key >= thr) keys[NT + atomicAdd(&S.nkeys, 1)] = key;
                    }
                  }
                }
                gsync<NT>();
                const int nk = S.nkeys;
                gsync<NT>();  // every thread has read nk before the next round adds to it
                if (nk > M - NT) {
                  const int P = pow2_at_least(NT + nk, 2 * NT);
                  for (int i = NT + nk + tid; i < P; i += NT) keys[i] = 0ull;
                  gsync<NT>();
                  bitonic_desc<NT>(keys, P, tid);
                  if (tid == 0) S.nkeys = 0;
                  gsync<NT>();
                  if (keys[beam - 1] != 0ull) {
                    const u64 kb = keys[beam - 1] & 0xffffffff00000000ull;
                    thr = kb > thr ? kb : thr;
                  }
                }
              }
              if (tid == 0) S.nuc = 0;
              gsync<NT>();
            }
          }
          const int nk = S.nkeys;
          if (nk > 0) {
            const int P = pow2_at_least(NT + nk, 2 * NT);
            for (int i = NT + nk + tid; i < P; i += NT) keys[i] = 0ull;
            gsync<NT>();
            bitonic_desc<NT>(keys, P, tid);
          }
          gsync<NT>();
          if (tid == 0) S.nkeys = 0;
          gsync<NT>();
          nw = 0;
          for (int w = 0; w < beam; ++w) nw += keys[w] != 0ull;
        }
      }

      BPHASE(3);
      // ---- section 3.4.5: the winners become the next hypotheses
      for (int w = tid; w < nw; w += NT) {
        const u64 key = keys[w];
        const float score = ck_score(key);
        const int src = ck_src(key), tk = ck_tok(key);
        if (tk == blank) {
          S.npb[w] = S.bpb[src];
          S.npnb[w] = S.bpnb[src];
          S.nlast[w] = S.last[src];
          S.nlen[w] = S.len[src];
          S.nh[w] = S.h[src];
          S.nhp[w] = S.hp[src];
        } else {
          S.npb[w] = NEG;
          S.npnb[w] = score;
          S.nlast[w] = tk;
          S.nlen[w] = S.len[src] + 1;
          S.nh[w] = hmix(S.h[src], tk);
          S.nhp[w] = S.h[src];
        }
        if (gap) {
          S.npb[w] = score;
          S.npnb[w] = NEG;
        }
        S.nsc[w] = score;
        S.nsrc[w] = src;
        S.ntok[w] = tk;
        // the new slot of each source's blank winner
        if (tk == blank) S.bw[src] = w;
        // token store: the winner's (source, token) into the ring; the rows
        // or pages are written at a flush
        S.hist[s - win0][w] = ((u32)src << 24) | ((u32)tk & 0xffffffu);
        S.norg[w] = S.org[src];
        S.nlo[w] = S.lo[src];
      }
      for (int i = tid; i < 2 * NT; i += NT) {
        S.hval[i] = -1;
        S.hkey[i] = 0ull;
      }
      if (tid == 0) {
        S.nw = nw;
        S.ndfree = 0;
      }
      gsync<NT>();
      // every winner's merge source: a blank winner keeps its source's
      // relation, an extension of source s relates to s's blank winner
      for (int w = tid; w < nw; w += NT) {
        const int src = S.nsrc[w];
        S.nmsrc[w] = S.ntok[w] == blank ? (S.msrc[src] >= 0 ? S.bw[S.msrc[src]] : -1) : S.bw[src];
        if (S.ntok[w] != blank) {  // the extension winners by prefix hash, for the check below
          const u64 key = S.nh[w];
          for (int q = 0; q < 2 * NT; ++q) {
            const int slot = (int)((key + (u64)q) & (u64)(2 * NT - 1));
            if (atomicCAS(&S.hval[slot], -1, w) == -1) {
              S.hkey[slot] = key;
              break;
            }
          }
        }
      }
      if (tid == 0) S.npairs = 0;
      gsync<NT>();
      BPHASE(4);
    }

    // the next step's lp[last] of the slots just chosen
    if (s + 1 < nsteps) prefetch_lpl(s + 1, srow_next, S.nw, S.nlast, S.nlen);
    BPHASE(5);
    // ---- the one merge relation the sources cannot show: a blank winner whose
    // parent prefix was just rebuilt by an extension winner (prefix hash
    // proposal, confirmed on the stored tokens)
    int npairs = 0;
    if (step > 0) {
      const int nw = S.nw;
      for (int j = tid; j < nw; j += NT) {
        if (S.ntok[j] != blank || S.nmsrc[j] >= 0 || S.nlen[j] < 1) continue;
        const u64 key = S.nhp[j];
        for (int q = 0; q < 2 * NT; ++q) {
          const int slot = (int)((key + (u64)q) & (u64)(2 * NT - 1));
          const int i = S.hval[slot];
          if (i < 0) break;
          if (S.hkey[slot] == key && S.nlen[i] == S.nlen[j] - 1) {
            const int pq = atomicAdd(&S.npairs, 1);
            if (pq < 2 * NT) {
              S.pi[pq] = i;
              S.pj[pq] = j;
            }
          }
        }
      }
      gsync<NT>();
      npairs = S.npairs < 2 * NT ? S.npairs : 2 * NT;
    }
    // the token store is written when the ring is full, at the call's last
    // step, and before tokens are compared
    if (s - win0 + 1 == S.R || s + 1 == nsteps || npairs > 0) {
      if (Ly.paged)
        flush_paged<NT>(S, st, b, par, s - win0 + 1, S.nw, blank, tid);
      else
        flush_flat<NT>(S, st, b, par, s - win0 + 1, S.nw, blank, tid);
      par ^= 1;
      win0 = s + 1;
    }
    if (npairs > 0) {
      const int tp = par;  // the parity holding the next slots' tokens
      for (int pq = 0; pq < npairs; ++pq) {
        const int i = S.pi[pq], j = S.pj[pq];
        const int Li = S.nlen[i];
        bool mism = false;
        for (int x = tid; x < Li; x += NT) mism |= tok.get(tp, i, x) != tok.get(tp, j, x);
        const bool same = !g_any<NT>(mism);
        c_hash += same ? 1u : 0u;
        if (same && tid == 0) S.nmsrc[j] = i;
      }
      gsync<NT>();
    }

    BPHASE(6);
    // ---- commit
    const int nw = S.nw;
    for (int k = tid; k < nw; k += NT) {
      S.pb[k] = S.npb[k];
      S.pnb[k] = S.npnb[k];
      S.sc[k] = S.nsc[k];
      S.last[k] = S.nlast[k];
      S.len[k] = S.nlen[k];
      S.h[k] = S.nh[k];
      S.hp[k] = S.nhp[k];
      S.msrc[k] = S.nmsrc[k];
      S.org[k] = S.norg[k];
      S.lo[k] = S.nlo[k];
    }
    gsync<NT>();
    nlive = nw;
    t_prev = t;
    ++step;
    ++c_steps;
    BPHASE(7);
  }

  for (int k = tid; k < beam; k += NT) {
    st.pb()[rb + k] = S.pb[k];
    st.pnb()[rb + k] = S.pnb[k];
    st.sc()[rb + k] = S.sc[k];
    st.last()[rb + k] = S.last[k];
    st.len()[rb + k] = S.len[k];
    st.h()[rb + k] = S.h[k];
    st.hp()[rb + k] = S.hp[k];
    st.msrc()[rb + k] = S.msrc[k];
  }
  if (tid == 0) {
    Header* hd = st.hdr();
    atomicAdd(&hd->counters[0], c_steps);
    if (c_scan) {
      atomicAdd(&hd->counters[1], c_scan);  // the list could not bound the unlisted labels
      atomicAdd(&hd->counters[3], c_scan);
    }
    if (c_exh) atomicAdd(&hd->counters[2], c_exh);
    if (c_hash) atomicAdd(&hd->counters[4], c_hash);
#ifdef CTCPB_PHASE_PROF
    for (int i = 0; i < 8; ++i) atomicAdd(&hd->phase_cycles[i], prof[i]);
#endif
    if (Ly.paged) {
      st.ptop()[b] = S.ptop;
      st.pnext()[b] = S.pnext;
    }
    rh->step = step;
    rh->tcount = mode == 0 ? rh->tcount : tcount + nft;
    rh->t_prev = t_prev;
    rh->nlive = nlive;
    rh->parity = par;
  }
}

// ------------------------------------------------------------------ output
// Section 3.6: the first nbest hypotheses after a stable sort by score.  Block
// (b, n) writes row b's n-th: it finds the slot of rank n, then copies its
// labels, so the rows' N best are written side by side.
__global__ void __launch_bounds__(128) k_output(View st, int nbest, int* __restrict__ out_tokens,
                                                int* __restrict__ out_lengths, float* __restrict__ out_scores,
                                                int out_len) {
  __shared__ float scs[kMaxBeam];
  __shared__ int slot_n;
  const Layout& Ly = st.lay;
  const int b = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
  const RowHdr rh = st.rows()[b];
  const int beam = Ly.beam;
  const bool never = rh.step == 0;
  const int nlive = never ? 0 : rh.nlive;
  const size_t o = (size_t)b * nbest + n;
  int* dst = out_tokens + o * (size_t)out_len;
  if (n >= nlive) {  // a dead slot (the whole block)
    for (int x = tid; x < out_len; x += blockDim.x) dst[x] = -1;
    if (tid == 0) {
      const bool empty_row = never && n == 0;
      out_lengths[o] = 0;
      out_scores[o] = empty_row ? 0.0f : CTCPB_NEG;
    }
    return;
  }
  for (int k = tid; k < nlive; k += blockDim.x) scs[k] = st.sc()[(size_t)b * beam + k];
  __syncthreads();
  for (int k = tid; k < nlive; k += blockDim.x) {
    int r = 0;
    const float v = scs[k];
    for (int j = 0; j < nlive; ++j) r += (scs[j] > v) || (scs[j] == v && j < k);
    if (r == n) slot_n = k;  // ranks are a permutation: exactly one slot
  }
  __syncthreads();
  const int k = slot_n;
  TokenStore tok{st, b};
  // flat storage left by the warp kernel: a slot's first plo labels may still
  // be in the other buffer (row porg)
  const bool pend = !Ly.paged && rh.pending != 0;
  const int L = st.len()[(size_t)b * beam + k];
  const int plo = pend ? st.plo()[(size_t)b * beam + k] : 0;
  const int org = pend ? st.porg()[(size_t)b * beam + k] : 0;
  const int* pre = plo > 0 ? st.clist(rh.parity ^ 1, b, org) : nullptr;
  for (int x = tid; x < out_len; x += blockDim.x) dst[x] = x < L ? (x < plo ? pre[x] : tok.get(rh.parity, k, x)) : -1;
  if (tid == 0) {
    out_lengths[o] = L;
    out_scores[o] = scs[k];
  }
}

// ------------------------------------------------------------------ launchers

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

cudaError_t launch_init(const View& st, cudaStream_t s) {
  k_init<<<grid_for((long long)st.lay.B * st.lay.beam * 2 + 1, 8), 256, 0, s>>>(st);
  return cudaGetLastError();
}

cudaError_t launch_boost_build(const View& st, const int* row_ptr, const int* tokens, const float* bonus,
                               cudaStream_t s) {
  if (st.lay.B == 0 || st.lay.hcap == 0) return cudaSuccess;
  k_boost_build<<<(st.lay.B + 63) / 64, 64, 0, s>>>(st, row_ptr, tokens, bonus);
  return cudaGetLastError();
}

cudaError_t launch_init_select(const View& st, const float* lp, long long sb, long long stt, const int* lens, int T,
                               int mode, float log_thr, int* sel, int* nsel, cudaStream_t s) {
  const int gi = grid_for((long long)st.lay.B * st.lay.beam * 2 + 1, 8);
  const int grid = st.lay.B > gi ? st.lay.B : gi;
  k_init_select<<<grid, 256, 0, s>>>(st, lp, sb, stt, lens, T, mode, log_thr, sel, nsel);
  return cudaGetLastError();
}

cudaError_t launch_select(const View& st, const float* lp, long long sb, long long stt, const int* lens, int T,
                          int mode, float log_thr, int* sel, int* nsel, cudaStream_t s) {
  if (st.lay.B == 0) return cudaSuccess;
  k_select<<<st.lay.B, 256, 0, s>>>(st, lp, sb, stt, lens, T, mode, log_thr, sel, nsel);
  return cudaGetLastError();
}

static_assert(sizeof(StepSmem<128>) + 4096 * sizeof(u64) <= 227 * 1024, "block step kernel shared memory");
static_assert(sizeof(StepSmem<32>) + 1024 * sizeof(u64) <= 227 * 1024, "block step kernel shared memory");

template <int NT>
static cudaError_t launch_step_t(const View& st, const float* lp, long long sb, long long stt, int mode,
                                 const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  const int sortcap = NT == 32 ? 1024 : 4096;
  // records are copied whole into shared memory in 16-byte words
  if (st.lay.rec_bytes > (size_t)StepSmem<NT>::kRecMax || (st.lay.rec_bytes & 15) != 0) return cudaErrorInvalidValue;
  const size_t smem = step_smem_bytes<NT>(sortcap);
  cudaError_t e = smem_optin<k_step<NT>>(smem);
  if (e != cudaSuccess) return e;
  k_step<NT><<<st.lay.B, NT, smem, s>>>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, sortcap);
  return cudaGetLastError();
}

cudaError_t launch_step(const View& st, const float* lp, long long sb, long long stt, int mode, const int* nframes,
                        int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  if (st.lay.B == 0) return cudaSuccess;
  if (step_warp_fits(st.lay))  // beam <= 16, flat storage, short lists
    return launch_step_warp(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
  if (st.lay.beam <= 32) return launch_step_t<32>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
  return launch_step_t<128>(st, lp, sb, stt, mode, nframes, chunk_T, tile_start, tile_len, s);
}

cudaError_t launch_select_tile(const View& st, const uint8_t* mask, long long mstride, const int* nframes,
                               int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  if (st.lay.B == 0) return cudaSuccess;
  k_select_tile<<<st.lay.B, 32, 0, s>>>(st, mask, mstride, nullptr, 0, 0, 0.0f, nframes, chunk_T, tile_start,
                                        tile_len);
  return cudaGetLastError();
}

cudaError_t launch_select_tile_thr(const View& st, const float* lp, long long sb, long long stt, float log_thr,
                                   const int* nframes, int chunk_T, int tile_start, int tile_len, cudaStream_t s) {
  if (st.lay.B == 0) return cudaSuccess;
  k_select_tile<<<st.lay.B, 32, 0, s>>>(st, nullptr, 0, lp, sb, stt, log_thr, nframes, chunk_T, tile_start,
                                        tile_len);
  return cudaGetLastError();
}

cudaError_t launch_host_plan(const int* lens, int B, int T, int F, int nchunks, int* plan, cudaStream_t s) {
  const long long n = (long long)nchunks * B;
  if (n == 0) return cudaSuccess;
  const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  k_host_plan<<<blocks, 256, 0, s>>>(lens, B, T, F, nchunks, plan);
  return cudaGetLastError();
}

cudaError_t launch_output(const View& st, int nbest, int* out_tokens, int* out_lengths, float* out_scores,
                          int out_len, cudaStream_t s) {
  if (st.lay.B == 0) return cudaSuccess;
  if (nbest <= 0) return cudaSuccess;
  k_output<<<dim3((unsigned)st.lay.B, (unsigned)nbest), 128, 0, s>>>(st, nbest, out_tokens, out_lengths, out_scores,
                                                                      out_len);
  return cudaGetLastError();
}

}  // namespace ctcpb
