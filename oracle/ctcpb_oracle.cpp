// CPU oracle for batched CTC prefix beam search -- TEST INFRASTRUCTURE ONLY.
//
// Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
// call this library.  It shares no code, header, table or constant generator
// with the CUDA decoder: every formula below is restated from the method's
// description ("GPU CTC Prefix Beam Search Decoder", OASR docs, section 3) and
// from mathematics.  It is deliberately plain and slow: every step scores the
// whole beam x vocabulary table, merges by comparing stored prefixes, and ranks
// with a library sort.
//
// Arithmetic.  The method stores its log-probabilities in float32 (log_prob is
// float32; pprev is a float2; score is a float), so the oracle computes in
// float32 with a fixed operation order.  Build with -ffp-contract=off and
// without -ffast-math: fused multiply-adds appear only where fmaf() is written.
//
//   NEG          = -FLT_MAX, the additive identity of the log semiring
//                  (section 3, the logsumexp definition).
//   add(a, b)    = max(a + b, NEG)          -- a product of probabilities
//   lse(a, b)    = max(a,b) + F(|a-b|)      -- section 3's logsumexp
//   F(d)         = log(1 + e^-d) for d >= 0, piecewise: on each of 96
//                  segments [k/4, (k+1)/4), k = 0..95, the degree-5 Taylor
//                  polynomial of F about the segment's midpoint d_k = k/4 +
//                  1/8, in u = d - d_k, evaluated by Horner's rule with fmaf;
//                  F(d) = 0 for d >= 24 (F(24) < 4e-11).  Its coefficients are
//                  the float32 roundings of F^(n)(d_k) / n!, computed once in
//                  double from libm's exp and log1p: F' = -s with s =
//                  1/(1 + e^d), and ds/dd = s^2 - s, so every derivative is a
//                  polynomial in s.
//   lp read      = max(raw, NEG) + 0.0f (clamps -inf/NaN to NEG, -0 to +0).
//
// Decoding follows section 3 of the page:
//   3.3   step 0 seeds the top (beam-1) non-blank labels (beam 1: one label)
//         by (log-prob desc, id asc), then the empty prefix in the last slot;
//         a skipped lead-in puts each label's mass in its blank slot.
//   3.4   collapsed-blank correction when frames were skipped (t > t_prev+1):
//         prev = (lse(pb, pnb), NEG) before the step, winners = (score, NEG)
//         after it (3.4.5).
//   3.4.1 non-blank extension: c != last -> lp[c] + lse(pb, pnb);
//         c == last -> lp[c] + pb; the stay path lp[last] + pnb goes to the
//         beam's own blank slot.
//   3.4.2 blank slot: pb' = lp[blank] + lse(pb, pnb); pnb' = stay, or NEG for
//         the empty prefix or after a gap.
//   3.4.3 merge: if len_j = len_i + 1 and l_j starts with l_i, candidate
//         (i, last_j) is folded into j's blank slot (pnb'_j = lse(pnb'_j, .))
//         and dropped.
//   3.4.4/5 score = lse(pb', pnb'); keep the best `beam` live candidates.
//   8, 14 a speech mask skips the frames it marks 0 exactly like the blank
//         threshold does (streaming decodes compare against it).
//   3.4.1/3.4.2 with a word-boundary label (space_id): its extension always
//         uses lse(pb, pnb) -- every space frame is a token of its own -- and a
//         space-ending beam gets no stay contribution.
//   Token boosting (the per-utterance word-boosting table of "GPU-Accelerated
//         WFST Beam Search Decoder for CTC-based Speech Recognition", applied
//         to CTC labels at the first page's section 15 extension point, where
//         scores are added before the top-K): each row gives every label a
//         bonus (0 when it is not boosted).  A label an extension emits scores
//         lp'[c] = add(lp[c], bonus[c]) in place of lp[c] -- in the step-0
//         ranking, the 3.4.1 extensions (repeat path included) and the 3.4.3
//         folds -- while the blank and the stay path, which emit no label,
//         keep lp.  Without pruning a prefix then scores log P(l) plus the sum
//         of its labels' bonuses.
// Readings where the page is silent or inconsistent:
//   * ties rank by (score desc, source slot asc, token asc), blank's token is
//     blank_id; a candidate with score <= NEG is dead and never kept;
//   * a hypothesis whose length equals the cap max_seq_len has no non-blank
//     extensions (its blank/stay slot still applies);
//   * frames are kept iff lp[blank] < log(threshold) (section 3.5), threshold
//     >= 1 keeps all frames and <= 0 keeps none (section 13);
//   * a row with no kept frame returns the empty prefix with score 0 in slot 0
//     and dead slots after it (section 13);
//   * output: the first nbest slots after a stable sort by score (desc);
//     dead slots have length 0, score NEG and tokens -1; tokens past out_len
//     are cut while the length still reports the full count (section 13).

#include <algorithm>
#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

constexpr float NEG = -FLT_MAX;

// The coefficient table of F: c[k][n] = F^(n)(d_k) / n! rounded to float.
constexpr int kSeg = 96, kDeg = 5;
constexpr float kFMax = 24.0f;

struct FTable {
  float c[kSeg][kDeg + 1];
  FTable() {
    for (int k = 0; k < kSeg; ++k) {
      const double d0 = k * 0.25 + 0.125;
      const double s = 1.0 / (1.0 + std::exp(d0));
      c[k][0] = (float)std::log1p(std::exp(-d0));
      // P[i]: coefficient of s^i in the current derivative, starting at F' = -s
      double P[kDeg + 2] = {0.0, -1.0};
      double fact = 1.0;
      for (int n = 1; n <= kDeg; ++n) {
        double v = 0.0;
        for (int i = kDeg + 1; i >= 0; --i) v = v * s + P[i];
        fact *= n;
        c[k][n] = (float)(v / fact);
        // d/dd P(s) = P'(s) (s^2 - s)
        double Q[kDeg + 2] = {};
        for (int i = 1; i <= kDeg; ++i) {
          Q[i + 1] += i * P[i];
          Q[i] -= i * P[i];
        }
        for (int i = 0; i <= kDeg + 1; ++i) P[i] = Q[i];
      }
    }
  }
};
const FTable& ftable() {
  static const FTable t;
  return t;
}

// log(1 + e^-d) for d >= 0.
float fF(float d) {
  if (!(d < kFMax)) return 0.0f;
  const int k = (int)(d * 4.0f);
  const float u = d - ((float)k * 0.25f + 0.125f);
  const float* c = ftable().c[k];
  float p = c[5];
  p = std::fmaf(p, u, c[4]);
  p = std::fmaf(p, u, c[3]);
  p = std::fmaf(p, u, c[2]);
  p = std::fmaf(p, u, c[1]);
  p = std::fmaf(p, u, c[0]);
  return p;
}

float lse(float a, float b) {
  float m = std::fmax(a, b);
  float d = std::fabs(a - b);
  return m + fF(d);
}

float add(float a, float b) { return std::fmax(a + b, NEG); }

float rd(const float* p) { return std::fmax(*p, NEG) + 0.0f; }

struct Hyp {
  std::vector<int32_t> pre;
  float pb, pnb;
  float score() const { return lse(pb, pnb); }
  int32_t last(int blank) const { return pre.empty() ? blank : pre.back(); }
};

struct Cand {
  float score;
  int32_t src, tok;
  float pb, pnb;
};

// ranking: score desc, then source slot asc, then token asc
bool better(const Cand& x, const Cand& y) {
  if (x.score != y.score) return x.score > y.score;
  if (x.src != y.src) return x.src < y.src;
  return x.tok < y.tok;
}

struct Args {
  const float* lp;
  int64_t sb, st;
  const int32_t* lens;
  int B, T, V, beam, nbest, blank, cap;
  float thr;
  int32_t* out_tokens;
  int32_t* out_lengths;
  float* out_scores;
  int out_len;
  const uint8_t* mask;  // [B, T] speech mask (0: skip the frame), or null
  int space;            // word-boundary label, or -1
  const float* boost;   // [B, V] label bonuses (0: not boosted), or null
};

bool keep_frame(float lpb, float thr, float log_thr) {
  if (thr >= 1.0f) return true;
  if (!(thr > 0.0f)) return false;
  return lpb < log_thr;
}

float log_threshold(float thr) {
  if (thr >= 1.0f || !(thr > 0.0f)) return NEG;
  return (float)std::log((double)thr);
}

// A label's log-prob as an emitted label: add(lp, bonus) when the row boosts
// labels (bonus 0 leaves lp unchanged: lp is never -0).
float emitted(const float* row, int c, const float* bonus) {
  return bonus ? add(rd(row + c), bonus[c]) : rd(row + c);
}

// Non-blank live labels of one frame in (lp desc, id asc) order, lp as emitted.
void ranked_labels(const float* row, int V, int blank, const float* bonus,
                   std::vector<std::pair<float, int32_t>>& out) {
  out.clear();
  for (int c = 0; c < V; ++c) {
    if (c == blank) continue;
    float v = emitted(row, c, bonus);
    if (v > NEG) out.push_back({v, c});
  }
  std::sort(out.begin(), out.end(), [](const std::pair<float, int32_t>& a, const std::pair<float, int32_t>& b) {
    if (a.first != b.first) return a.first > b.first;
    return a.second < b.second;
  });
}

void decode_row(const Args& a, int b) {
  const float* base = a.lp + (int64_t)b * a.sb;
  auto row = [&](int t) { return base + (int64_t)t * a.st; };
  const float log_thr = log_threshold(a.thr);
  int len_b = std::min(std::max(a.lens ? a.lens[b] : a.T, 0), a.T);
  const float* bonus = a.boost ? a.boost + (int64_t)b * a.V : nullptr;

  // section 3.5: ordered list of kept frames.  A speech mask (sections 8, 14
  // and 15: frames the caller marks as non-speech bypass the decoder, like
  // frames skipped by the blank threshold) removes frames as well.
  std::vector<int> sel;
  for (int t = 0; t < len_b; ++t)
    if (keep_frame(rd(row(t) + a.blank), a.thr, log_thr) && (!a.mask || a.mask[(int64_t)b * a.T + t] != 0))
      sel.push_back(t);

  std::vector<Hyp> beams;
  if (sel.empty()) {
    beams.push_back(Hyp{{}, 0.0f, NEG});
  } else {
    // ---- step 0 (section 3.3)
    const int t0 = sel[0];
    const bool gap0 = t0 > 0;
    const int nb = a.beam > 1 ? a.beam - 1 : 1;
    std::vector<std::pair<float, int32_t>> ranked;
    ranked_labels(row(t0), a.V, a.blank, bonus, ranked);
    if (a.cap >= 1) {
      for (int k = 0; k < nb && k < (int)ranked.size(); ++k) {
        float v = ranked[k].first;
        Hyp h{{ranked[k].second}, gap0 ? v : NEG, gap0 ? NEG : v};
        beams.push_back(h);
      }
    }
    if (a.beam > 1) {
      float lpb = rd(row(t0) + a.blank);
      if (lpb > NEG) beams.push_back(Hyp{{}, lpb, NEG});
    }

    // ---- steps s >= 1 (section 3.4)
    std::vector<Cand> cands;
    for (size_t s = 1; s < sel.size(); ++s) {
      const int t = sel[s];
      const bool gap = t > sel[s - 1] + 1;
      const float* lpt = row(t);
      const int K = (int)beams.size();
      if (K == 0) break;
      // collapsed-blank correction of the previous probabilities
      std::vector<float> pb(K), pnb(K), A(K);
      for (int k = 0; k < K; ++k) {
        pb[k] = beams[k].pb;
        pnb[k] = beams[k].pnb;
        if (gap) {
          pb[k] = lse(pb[k], pnb[k]);
          pnb[k] = NEG;
        }
        A[k] = lse(pb[k], pnb[k]);
      }
      // section 3.4.3 pair condition: into[j] = i when l_j = l_i + last(l_j)
      std::vector<int> into(K, -1);
      for (int j = 0; j < K; ++j)
        for (int i = 0; i < K; ++i) {
          const auto& li = beams[i].pre;
          const auto& lj = beams[j].pre;
          if (lj.size() == li.size() + 1 && std::equal(li.begin(), li.end(), lj.begin())) into[j] = i;
        }
      std::vector<std::vector<int32_t>> folded(K);  // labels of beam i folded away
      for (int j = 0; j < K; ++j)
        if (into[j] >= 0) folded[into[j]].push_back(beams[j].last(a.blank));

      const float lpb = rd(lpt + a.blank);
      // sections 3.4.1/3.4.2 with a word-boundary label: the space extension
      // always takes lp[space] + lse(pb, pnb) (it never repeats into the
      // previous space), so a space-ending beam has no stay contribution
      const int space = (a.space >= 0 && a.space != a.blank) ? a.space : -1;
      cands.clear();
      for (int k = 0; k < K; ++k) {
        const Hyp& h = beams[k];
        const int32_t last = h.last(a.blank);
        const bool empty = h.pre.empty();
        // section 3.4.2 blank slot, with section 3.4.1's stay contribution
        float bpb = add(lpb, A[k]);
        float bpnb = (!empty && !gap && last != space) ? add(rd(lpt + last), pnb[k]) : NEG;
        if (into[k] >= 0) {
          // section 3.4.3: fold candidate (i, last_k) into this blank slot; its
          // value is the section 3.4.1 table entry, which takes the repeat
          // path (pb only) when last_k is also the last label of l_i
          int i = into[k];
          const bool rep = !beams[i].pre.empty() && beams[i].pre.back() == last && last != space;
          const float v = emitted(lpt, last, bonus);
          float ext = rep ? add(v, pb[i]) : add(v, A[i]);
          bpnb = lse(bpnb, ext);
        }
        float sc = lse(bpb, bpnb);
        if (sc > NEG) cands.push_back(Cand{sc, k, a.blank, bpb, bpnb});
        if ((int)h.pre.size() >= a.cap) continue;
        // section 3.4.1 non-blank extensions
        for (int c = 0; c < a.V; ++c) {
          if (c == a.blank) continue;
          if (std::find(folded[k].begin(), folded[k].end(), c) != folded[k].end()) continue;
          float v = emitted(lpt, c, bonus);
          float ext = (!empty && c == last && c != space) ? add(v, pb[k]) : add(v, A[k]);
          if (ext > NEG) cands.push_back(Cand{ext, k, c, NEG, ext});
        }
      }
      // section 3.4.4/3.4.5: keep the best `beam`
      size_t keep = std::min(cands.size(), (size_t)a.beam);
      if (cands.size() > keep) std::nth_element(cands.begin(), cands.begin() + keep, cands.end(), better);
      std::sort(cands.begin(), cands.begin() + keep, better);
      std::vector<Hyp> next;
      next.reserve(keep);
      for (size_t w = 0; w < keep; ++w) {
        const Cand& c = cands[w];
        Hyp h;
        h.pre = beams[c.src].pre;
        if (c.tok != a.blank) h.pre.push_back(c.tok);
        if (gap) {
          h.pb = c.score;
          h.pnb = NEG;
        } else {
          h.pb = c.pb;
          h.pnb = c.pnb;
        }
        next.push_back(std::move(h));
      }
      beams.swap(next);
    }
  }

  // ---- output (sections 3.6 and 13)
  std::vector<int> order(beams.size());
  std::vector<float> sc(beams.size());
  for (size_t k = 0; k < beams.size(); ++k) {
    order[k] = (int)k;
    sc[k] = beams[k].score();
  }
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return sc[x] > sc[y]; });
  for (int n = 0; n < a.nbest; ++n) {
    int32_t* tok = a.out_tokens + ((int64_t)b * a.nbest + n) * a.out_len;
    for (int i = 0; i < a.out_len; ++i) tok[i] = -1;
    int64_t o = (int64_t)b * a.nbest + n;
    if (n < (int)order.size()) {
      const Hyp& h = beams[order[n]];
      a.out_lengths[o] = (int32_t)h.pre.size();
      a.out_scores[o] = sc[order[n]];
      for (int i = 0; i < (int)h.pre.size() && i < a.out_len; ++i) tok[i] = h.pre[i];
    } else {
      a.out_lengths[o] = 0;
      a.out_scores[o] = NEG;
    }
  }
}

void for_rows(int B, int threads, const std::function<void(int)>& fn) {
  if (threads <= 0) threads = (int)std::thread::hardware_concurrency();
  threads = std::max(1, std::min(threads, B));
  std::atomic<int> next{0};
  auto work = [&]() {
    for (int b; (b = next.fetch_add(1)) < B;) fn(b);
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < threads; ++i) pool.emplace_back(work);
  work();
  for (auto& th : pool) th.join();
}
}  // namespace

extern "C" {

float ctcpb_oracle_F(float d) { return fF(d); }
// The 96 x 6 coefficients of F, segment-major.
void ctcpb_oracle_F_coefficients(float* out) {
  for (int k = 0; k < kSeg; ++k)
    for (int n = 0; n <= kDeg; ++n) out[k * (kDeg + 1) + n] = ftable().c[k][n];
}
float ctcpb_oracle_lse(float a, float b) { return lse(a, b); }
float ctcpb_oracle_add(float a, float b) { return add(a, b); }
float ctcpb_oracle_log_threshold(float thr) { return log_threshold(thr); }

void ctcpb_oracle_map(int which, const float* a, const float* b, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    switch (which) {
      case 0: out[i] = fF(a[i]); break;
      case 2: out[i] = lse(a[i], b[i]); break;
      default: out[i] = add(a[i], b[i]); break;
    }
  }
}

// Section 3.5: kept frames of each row, in order.  sel is [B, T], nsel is [B].
int ctcpb_oracle_select_frames(const float* lp, int64_t sb, int64_t st, const int32_t* lens, int B, int T,
                               int blank, float thr, int32_t* sel, int32_t* nsel) {
  const float log_thr = log_threshold(thr);
  for (int b = 0; b < B; ++b) {
    int len_b = std::min(std::max(lens ? lens[b] : T, 0), T);
    int n = 0;
    for (int t = 0; t < len_b; ++t)
      if (keep_frame(rd(lp + b * sb + (int64_t)t * st + blank), thr, log_thr)) sel[(int64_t)b * T + n++] = t;
    for (int i = n; i < T; ++i) sel[(int64_t)b * T + i] = -1;
    nsel[b] = n;
  }
  return 0;
}

// The ranked non-blank labels of each of R frame rows ([R, V], row stride st):
// the first C by (lp desc, id asc), their count, the blank log-prob, and the
// next label after them (front) or (NEG, -1) when there is none.
int ctcpb_oracle_frame_lists(const float* lp, int64_t st, int R, int V, int blank, int C, int32_t* ids,
                             float* lps, int32_t* cnt, float* lpb, float* front_lp, int32_t* front_id) {
  std::vector<std::pair<float, int32_t>> ranked;
  for (int r = 0; r < R; ++r) {
    const float* row = lp + (int64_t)r * st;
    ranked_labels(row, V, blank, nullptr, ranked);
    int n = std::min((int)ranked.size(), C);
    for (int i = 0; i < C; ++i) {
      ids[(int64_t)r * C + i] = i < n ? ranked[i].second : -1;
      lps[(int64_t)r * C + i] = i < n ? ranked[i].first : NEG;
    }
    cnt[r] = n;
    lpb[r] = rd(row + blank);
    if ((int)ranked.size() > C) {
      front_lp[r] = ranked[C].first;
      front_id[r] = ranked[C].second;
    } else {
      front_lp[r] = NEG;
      front_id[r] = -1;
    }
  }
  return 0;
}

// Offline decode of B rows.  cap >= 1 is the per-hypothesis token cap; mask
// ([B, T] uint8, may be null) skips every frame marked 0; space_id (-1: none)
// is the word-boundary label; boost ([B, V] float, may be null) holds each
// row's label bonuses.
// Outputs: tokens [B, nbest, out_len], lengths [B, nbest], scores [B, nbest].
int ctcpb_oracle_decode(const float* lp, int64_t sb, int64_t st, const int32_t* lens, int B, int T, int V,
                        int beam, int nbest, int blank, int cap, float thr, int threads, int32_t* out_tokens,
                        int32_t* out_lengths, float* out_scores, int out_len, const uint8_t* mask,
                        int space_id, const float* boost) {
  if (B < 0 || T < 0 || V < 2 || beam < 1 || nbest < 1 || nbest > beam || blank < 0 || blank >= V || cap < 1 ||
      out_len < 0)
    return -1;
  Args a{lp, sb, st, lens, B, T, V, beam, nbest, blank, cap, thr, out_tokens, out_lengths, out_scores, out_len,
         mask, space_id, boost};
  for_rows(B, threads, [&](int b) { decode_row(a, b); });
  return 0;
}

}  // extern "C"
