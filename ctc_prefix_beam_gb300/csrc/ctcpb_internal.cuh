// Internal definitions of the GB300 CTC prefix beam search decoder:
// workspace/state layout (host + device) and the float32 arithmetic.
#pragma once

#include <cfloat>
#include <cstddef>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "ctcpb.h"

namespace ctcpb {

typedef unsigned long long u64;
typedef unsigned int u32;

constexpr int kMaxBeam = 128;                 // section 11: beam 1..128
constexpr int kMaxList = 2 * kMaxBeam + 2;    // section 3.4.6: K_all <= 2*beam+2
constexpr int kMaxV = 1 << 20;                // labels fit the 20-bit token field of a rank key
constexpr int kStreamTile = 64;               // frames ranked per pre-pass tile when streaming
constexpr int kBlockRing = 64;                // block step kernel: steps between token-store writes
constexpr int kMaxBoost = 4096;               // boosted labels per row
constexpr float kMaxBonus = 1e6f;             // largest bonus magnitude
constexpr int kStreamDefaultCap = 4096;       // section 11: STREAMING_MAX_SEQ_LEN
constexpr u32 kMagic = 0x42504354u;           // "TCPB"
constexpr u32 kVersion = 3u;

// ---------------------------------------------------------------- layout
//
// One "decode state" serves both the offline workspace (tile = T, one record
// per decoded step) and a streaming state (tile = kStreamTile, records reused
// per chunk tile).  Every slab is 256-byte aligned; offsets are from the base.
struct Header {
  u32 magic, version;
  int32_t B, V, beam, cap, paged, page_size, blank, list_len, tile, space;
  u32 status;  // CTCPB_DEV_* bits
  u32 counters[5];  // decode steps, unproven first sets, exhaustive selections, full-frame scans,
                    // hash-proposed merges
  u64 phase_cycles[8];  // CTCPB_PHASE_PROF builds: clock64 cycles per step phase, summed over rows
  u32 fused_launches;   // pre-pass + steps launches made as one cooperative kernel
  int32_t hcap;         // label-boost hash slots per row (0: no boosting)
  u32 pad1[28];
};
static_assert(sizeof(Header) == 256, "header is 256 bytes");

struct RowHdr {
  int32_t step;    // decode steps done (0: the row has not decoded a frame yet)
  int32_t tcount;  // frames consumed (streaming) -- the next frame index
  int32_t t_prev;  // frame index of the last decoded step (-1 before the first)
  int32_t nlive;   // live hypotheses in slots [0, nlive)
  int32_t parity;  // token buffer holding the current hypotheses
  // flat storage: 1 when each slot k's first plo[k] labels are still in the
  // other buffer, at row porg[k] (the warp step kernel leaves them there at
  // the end of a call and copies them at the start of the next)
  int32_t pending;
  int32_t pad[2];
};

struct Layout {
  int B, V, beam, cap, paged, page_size, blank, L, Lpad, tile;
  int space;   // word-boundary label (sections 3.4.1/3.4.2), -1: none
  int ldseq;   // flat: labels per hypothesis row
  int max_lp;  // paged: logical pages per hypothesis
  int ppr;     // paged: physical pages per row
  int T_sel;   // selection entries per row: offline T (frames); streaming kStreamTile (one tile's chunk rows)
  int max_boost, hcap;  // boosted labels per row and hash slots per row (a power of two, 0: no boosting)
  size_t rec_bytes;
  size_t o_rows, o_pb, o_pnb, o_sc, o_last, o_len, o_h, o_hp, o_msrc;
  size_t o_clist, o_porg, o_plo, o_pages, o_btab, o_refc, o_pool, o_ptop, o_pnext;
  size_t o_recs, o_rflag, o_sel, o_nsel, o_bkey, o_bval, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Labels ranked per frame: default min(2*beam+2, V-1) (section 3.4.6's K_all
// bound).  A requested length below `beam` is raised to `beam`, because step 0
// seeds beam-1 labels straight from the list (section 3.3).
inline int default_list_len(int beam, int V, int list_len) {
  int L = list_len > 0 ? list_len : 2 * beam + 2;
  if (L < beam) L = beam;
  if (L > V - 1) L = V - 1;
  if (L > kMaxList) L = kMaxList;
  return L < 1 ? 1 : L;
}

// Build the layout.  tile = records per row; T_sel = selection list length
// (offline T, 0 when streaming).
inline Layout make_layout(int B, int V, int beam, int cap, int paged, int page_size, int blank, int L,
                          int tile, int T_sel, int space = -1, int max_boost = 0) {
  Layout o{};
  o.space = (space >= 0 && space != blank) ? space : -1;
  o.B = B; o.V = V; o.beam = beam; o.cap = cap; o.paged = paged; o.page_size = page_size;
  o.blank = blank; o.L = L; o.Lpad = (int)align_up((size_t)L, 4); o.tile = tile; o.T_sel = T_sel;
  o.ldseq = (int)align_up((size_t)cap, 16);
  o.max_lp = paged ? (cap + page_size - 1) / page_size : 0;
  // a row's pages at a token-store write: the tables written at the previous
  // write (<= max_lp pages a slot) and each slot's pages for the labels it
  // gained since, at most kBlockRing of them (one partial page copied)
  const int gain_pages = (kBlockRing + page_size - 1) / page_size + 1;
  o.ppr = paged ? beam * (o.max_lp + (gain_pages < o.max_lp ? gain_pages : o.max_lp)) : 0;
  o.rec_bytes = align_up(32 + 8 * (size_t)o.Lpad, 32);
  o.max_boost = max_boost > 0 ? max_boost : 0;
  o.hcap = 0;
  if (o.max_boost > 0) {  // open addressing at load <= 1/2
    o.hcap = 2;
    while (o.hcap < 2 * o.max_boost) o.hcap <<= 1;
  }
  const size_t A = 256;
  size_t off = sizeof(Header);
  auto take = [&](size_t bytes) { size_t at = align_up(off, A); off = at + bytes; return at; };
  const size_t nb = (size_t)B * beam;
  o.o_rows = take(sizeof(RowHdr) * (size_t)B);
  o.o_pb = take(4 * nb);
  o.o_pnb = take(4 * nb);
  o.o_sc = take(4 * nb);
  o.o_last = take(4 * nb);
  o.o_len = take(4 * nb);
  o.o_h = take(8 * nb);
  o.o_hp = take(8 * nb);
  o.o_msrc = take(4 * nb);
  if (!paged) {
    o.o_clist = take(4 * 2 * nb * (size_t)o.ldseq);
    o.o_porg = take(4 * nb);
    o.o_plo = take(4 * nb);
  } else {
    o.o_pages = take(4 * (size_t)B * o.ppr * (size_t)page_size);
    o.o_btab = take(4 * 2 * nb * (size_t)o.max_lp);
    o.o_refc = take(4 * (size_t)B * o.ppr);
    o.o_pool = take(4 * (size_t)B * o.ppr);
    o.o_ptop = take(4 * (size_t)B);
    o.o_pnext = take(4 * (size_t)B);
  }
  o.o_recs = take(o.rec_bytes * (size_t)B * tile);
  o.o_rflag = take(4 * (size_t)B * tile);
  if (T_sel > 0) {
    o.o_sel = take(4 * (size_t)B * T_sel);
    o.o_nsel = take(4 * (size_t)B);
  }
  if (o.hcap > 0) {
    o.o_bkey = take(4 * (size_t)B * o.hcap);
    o.o_bval = take(4 * (size_t)B * o.hcap);
  }
  o.total = align_up(off, A);
  return o;
}

// Typed views of a state buffer.
struct View {
  char* base;
  Layout lay;
  __host__ __device__ Header* hdr() const { return (Header*)base; }
  __host__ __device__ RowHdr* rows() const { return (RowHdr*)(base + lay.o_rows); }
  __host__ __device__ float* pb() const { return (float*)(base + lay.o_pb); }
  __host__ __device__ float* pnb() const { return (float*)(base + lay.o_pnb); }
  __host__ __device__ float* sc() const { return (float*)(base + lay.o_sc); }
  __host__ __device__ int* last() const { return (int*)(base + lay.o_last); }
  __host__ __device__ int* len() const { return (int*)(base + lay.o_len); }
  __host__ __device__ u64* h() const { return (u64*)(base + lay.o_h); }
  __host__ __device__ u64* hp() const { return (u64*)(base + lay.o_hp); }
  // merge source: slot i with l_k = l_i + last(l_k), or -1 (kept by the warp kernel)
  __host__ __device__ int* msrc() const { return (int*)(base + lay.o_msrc); }
  // flat token rows: clist[par][b][k][ldseq]
  __host__ __device__ int* clist(int par, int b, int k) const {
    return (int*)(base + lay.o_clist) + (((size_t)par * lay.B + b) * lay.beam + k) * (size_t)lay.ldseq;
  }
  // flat: a pending prefix's row in the other buffer and its length, [B][beam]
  __host__ __device__ int* porg() const { return (int*)(base + lay.o_porg); }
  __host__ __device__ int* plo() const { return (int*)(base + lay.o_plo); }
  // paged storage, per-row partitions of ppr pages
  __host__ __device__ int* page(int b, int phys) const {
    return (int*)(base + lay.o_pages) + ((size_t)b * lay.ppr + phys) * (size_t)lay.page_size;
  }
  __host__ __device__ int* btab(int par, int b, int k) const {
    return (int*)(base + lay.o_btab) + (((size_t)par * lay.B + b) * lay.beam + k) * (size_t)lay.max_lp;
  }
  __host__ __device__ int* refc(int b) const { return (int*)(base + lay.o_refc) + (size_t)b * lay.ppr; }
  __host__ __device__ int* pool(int b) const { return (int*)(base + lay.o_pool) + (size_t)b * lay.ppr; }
  __host__ __device__ int* ptop() const { return (int*)(base + lay.o_ptop); }
  __host__ __device__ int* pnext() const { return (int*)(base + lay.o_pnext); }
  // pre-pass records: rec(b, s)
  __host__ __device__ char* rec(int b, int s) const {
    return base + lay.o_recs + ((size_t)b * lay.tile + s) * lay.rec_bytes;
  }
  // record ready flags [B][tile]: set by the pre-pass, cleared by the step
  // kernel once it has copied the record (only when the two run concurrently)
  // label-boost hash table of row b: hcap (label, bonus) slots, label -1 empty
  __host__ __device__ int* bkey(int b) const { return (int*)(base + lay.o_bkey) + (size_t)b * lay.hcap; }
  __host__ __device__ float* bval(int b) const { return (float*)(base + lay.o_bval) + (size_t)b * lay.hcap; }
  __host__ __device__ u32* rflag() const { return (u32*)(base + lay.o_rflag); }
  __host__ __device__ int* sel() const { return (int*)(base + lay.o_sel); }
  __host__ __device__ int* nsel() const { return (int*)(base + lay.o_nsel); }
};

// Pre-pass record: one ranked frame.
struct RecHdr {
  int32_t cnt;       // labels in the list
  int32_t front_id;  // first label after the list (-1: none live)
  float lpb;         // blank log-prob
  float front_lp;    // its log-prob (-FLT_MAX: none)
  int32_t t;         // frame index of the step (offline: the kept frame)
  int32_t pad[3];
};
static_assert(sizeof(RecHdr) == 32, "record header is 32 bytes");
__host__ __device__ inline int* rec_ids(char* r) { return (int*)(r + 32); }
__host__ __device__ inline float* rec_lps(char* r, int Lpad) { return (float*)(r + 32 + 4 * (size_t)Lpad); }

// ---------------------------------------------------------------- arithmetic
//
// The decoder's float32 log-semiring ("GPU CTC Prefix Beam Search Decoder",
// section 3: logsumexp(a,b) = max + log(1 + exp(-|a-b|)), NEG_INF = -FLT_MAX),
// written with explicit round-to-nearest intrinsics so nothing is contracted.
//   dF(d)     log(1 + e^-d) for d >= 0: on each of 96 segments [k/4, (k+1)/4)
//             the degree-5 Taylor polynomial of the function about the
//             segment's midpoint d_k = k/4 + 1/8, in u = d - d_k, by Horner's
//             rule; 0 for d >= 24 (where it is below 4e-11).
//   dlse      max(a,b) + dF(|a-b|).
//   dadd      max(a+b, NEG): a product of probabilities, clamped to NEG.
// The coefficients are the float32 roundings of F^(n)(d_k) / n!.  They are
// computed at compile time (make_fcoef) in double: F' = -s with s =
// 1/(1 + e^d) and ds/dd = s^2 - s, so each derivative is a polynomial in s;
// exp and log1p come from their series (cx_exp, cx_log1p).  The kernels copy
// the table into shared memory and pass it to dlse.
#define CTCPB_NEG (-FLT_MAX)

constexpr int kFSeg = 96, kFDeg = 5, kFCoef = kFSeg * (kFDeg + 1);
struct FCoef {
  float c[kFCoef];  // segment-major: c[6k + n]
};

// e^x for |x| <= 25: x = n ln2 + r, |r| <= ln2/2, the Taylor series of e^r to
// r^24, times 2^n.
constexpr double cx_exp(double x) {
  const double ln2 = 0.693147180559945309417232121458;
  const double t = x / ln2;
  const int n = (int)(t >= 0.0 ? t + 0.5 : t - 0.5);
  const double r = x - n * ln2;
  double term = 1.0, sum = 1.0;
  for (int i = 1; i <= 24; ++i) {
    term = term * r / i;
    sum += term;
  }
  double p = 1.0;
  for (int i = 0; i < (n >= 0 ? n : -n); ++i) p *= 2.0;
  return n >= 0 ? sum * p : sum / p;
}

// log(1 + y) for y in [0, 1]: 2 atanh(t), t = y / (2 + y) <= 1/3, the odd
// series to t^49 (stopping once a term is below 1e-60 of the first, which
// also keeps the compile-time evaluation clear of underflow).
constexpr double cx_log1p(double y) {
  const double t = y / (2.0 + y), t2 = t * t;
  double pw = t, sum = 0.0;
  for (int j = 0; j < 25 && pw > t * 1e-60; ++j) {
    sum += pw / (2 * j + 1);
    pw *= t2;
  }
  return 2.0 * sum;
}

constexpr FCoef make_fcoef() {
  FCoef f{};
  for (int k = 0; k < kFSeg; ++k) {
    const double d0 = k * 0.25 + 0.125;
    const double s = 1.0 / (1.0 + cx_exp(d0));
    f.c[6 * k] = (float)cx_log1p(cx_exp(-d0));
    double P[kFDeg + 2] = {0.0, -1.0, 0.0, 0.0, 0.0, 0.0, 0.0};  // F' = -s, coefficients of s^i
    double fact = 1.0;
    for (int n = 1; n <= kFDeg; ++n) {
      double v = 0.0;
      for (int i = kFDeg + 1; i >= 0; --i) v = v * s + P[i];
      fact *= n;
      f.c[6 * k + n] = (float)(v / fact);
      double Q[kFDeg + 2] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};  // d/dd P(s) = P'(s) (s^2 - s)
      for (int i = 1; i <= kFDeg; ++i) {
        Q[i + 1] += i * P[i];
        Q[i] -= i * P[i];
      }
      for (int i = 0; i < kFDeg + 2; ++i) P[i] = Q[i];
    }
  }
  return f;
}

__device__ __forceinline__ float dF(const float* __restrict__ fc, float d) {
  const bool far = !(d < 24.0f);  // NaN too
  const int k = far ? 0 : (int)__fmul_rn(d, 4.0f);
  const float u = __fsub_rn(d, __fadd_rn(__fmul_rn((float)k, 0.25f), 0.125f));
  const float* c = fc + 6 * k;
  float p = c[5];
  p = __fmaf_rn(p, u, c[4]);
  p = __fmaf_rn(p, u, c[3]);
  p = __fmaf_rn(p, u, c[2]);
  p = __fmaf_rn(p, u, c[1]);
  p = __fmaf_rn(p, u, c[0]);
  return far ? 0.0f : p;
}

// fc: the coefficient table (shared memory).
__device__ __forceinline__ float dlse(const float* __restrict__ fc, float a, float b) {
  float m = fmaxf(a, b);
  float d = fabsf(__fsub_rn(a, b));
  return __fadd_rn(m, dF(fc, d));
}

__device__ __forceinline__ float dadd(float a, float b) { return fmaxf(__fadd_rn(a, b), CTCPB_NEG); }

// Read a log-prob: NaN and -inf become NEG, -0 becomes +0.
__device__ __forceinline__ float rdlp(float raw) { return __fadd_rn(fmaxf(raw, CTCPB_NEG), 0.0f); }

// Does the state's header describe this layout?  (A state initialised with
// another configuration or size must not be written through this one.)
__device__ __forceinline__ bool header_matches(const View& st) {
  const Header* hd = st.hdr();
  const Layout& Ly = st.lay;
  return hd->magic == kMagic && hd->version == kVersion && hd->B == Ly.B && hd->V == Ly.V && hd->beam == Ly.beam &&
         hd->cap == Ly.cap && hd->paged == Ly.paged && hd->page_size == Ly.page_size && hd->blank == Ly.blank &&
         hd->list_len == Ly.L && hd->tile == Ly.tile && hd->space == Ly.space && hd->hcap == Ly.hcap;
}

// Home slot of label c in a label-boost table of hmask + 1 slots.
__host__ __device__ __forceinline__ int boost_slot(int c, int hmask) { return (int)(((u32)c * 0x9E3779B1u) & (u32)hmask); }

// The bonus of label c in a row's label-boost table (0 when c is not boosted):
// linear probing from its home slot to the label or an empty slot (the table
// is at most half full, so one exists).
__device__ __forceinline__ float boost_of(const int* __restrict__ keys, const float* __restrict__ vals, int hmask,
                                          int c) {
  for (int i = boost_slot(c, hmask), n = 0; n <= hmask; i = (i + 1) & hmask, ++n) {
    const int k = keys[i];
    if (k == c) return vals[i];
    if (k < 0) break;
  }
  return 0.0f;
}

// Order-preserving unsigned image of a float (larger float -> larger key).
__host__ __device__ __forceinline__ u32 fkey(float f) {
#ifdef __CUDA_ARCH__
  u32 u = __float_as_uint(f);
#else
  u32 u;
  memcpy(&u, &f, 4);
#endif
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(u32 k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Rank key of a pre-pass label: larger = (higher log-prob, then smaller id).
// 0 marks "not a live label".
__device__ __forceinline__ u64 lab_key(float lp, int c) {
  return ((u64)fkey(lp) << 32) | (u32)(~(u32)c);
}

// Rank key of a step candidate: larger = (higher score, then smaller source
// slot, then smaller token); 0 marks a dead candidate.
__device__ __forceinline__ u64 cand_key(float score, int src, int tok) {
  return ((u64)fkey(score) << 32) | (u32)(~(((u32)src << 20) | (u32)tok));
}
__device__ __forceinline__ float ck_score(u64 k) { return fkey_inv((u32)(k >> 32)); }
__device__ __forceinline__ int ck_src(u64 k) { return (int)((~(u32)k) >> 20); }
__device__ __forceinline__ int ck_tok(u64 k) { return (int)((~(u32)k) & 0xfffffu); }

// Prefix hash: h(empty) = kH0, h(l + c) = mix(h(l), c).  Used only to find
// candidate pairs for the exact prefix comparison of section 3.4.3.
constexpr u64 kH0 = 0x6a09e667f3bcc909ull;
__device__ __forceinline__ u64 hmix(u64 h, int c) {
  u64 x = h ^ ((u64)(u32)c * 0x9e3779b97f4a7c15ull + 0x632be59bd9b4e019ull);
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ull;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebull;
  x ^= x >> 31;
  return x;
}

}  // namespace ctcpb
