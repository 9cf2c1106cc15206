// Speculative-sampling residual draw for sm_103a ("Accelerating Large
// Language Model Decoding with Speculative Sampling", section 4.2 "Modified
// Rejection Sampling"): at the first rejected position j, one token is drawn
// from max(0, p_j - q_j) normalised, by inverse CDF in vocabulary order.
//
// Runs after the row kernel in SpS mode, which wrote the first rejected
// position of every prompt (or -1) and each row's log-sum-exp to about 1e-7.
// Without top-p, three launches, each over what the one before it left:
//   sps_fast_kernel:  one CTA per (8192-logit chunk, prompt), p_v and q_v in
//                     fp32 with a proven bound E on the residual CDF's error;
//                     the last CTA of the prompt draws when u R lies farther
//                     than 2E from both edges of the chosen token, which makes
//                     that token the exact one, and queues the prompt
//                     otherwise;
//   sps_ff_kernel:    the queued prompts in float-float: each CTA sums p_v and
//                     q_v against the row kernel's log-sum-exps (provisional
//                     shifts) and the residual at ratio 1; the last CTA of the
//                     prompt turns those into the exact normalisers and chunk
//                     masses, picks the chunk and the element.  Where the
//                     shifts' ratio or the close calls (|p_v - q_v| <= tau
//                     q_v) could move the masses by more than 2e-10 of the
//                     residual mass, the prompt is queued again;
//   sps_retry_kernel: the same pass with the exact log-sum-exps as shifts.
// A prompt with no residual mass or a non-finite row takes the two-pass route
// below in one CTA.  With top-p, two launches:
//   sps_stats_kernel:    float-float log-sum-exp of rows p_j and q_j, so that
//                        p_v and q_v are known to ~1e-10 relative;
//   sps_residual_kernel: per-chunk residual mass; the last CTA of the prompt
//                        picks the chunk and the element.
// CTAs of prompts with no rejection exit at once.
//
// Under a temperature T the rows are s l with s = fl32(1/T); under top-p each
// of p_j and q_j is restricted to its nucleus {l >= thr} (the thresholds the
// nucleus kernel left in the rows' results) and renormalised.
#include <cmath>

#include "row_common.cuh"
#include "kernels.h"
#include "smcsd.h"

namespace smcsd {

// The residual kernels' chunk: kSpsNV 16-byte vectors per thread (half the
// row kernels' chunk), so that both rows' chunks fit in few registers and
// four CTAs share an SM.
constexpr int kSpsNV = 2;
template <typename T> struct SpsGeom {
  static constexpr int kEPV = LogitTraits<T>::kPerVec;
  static constexpr int kEPT = kSpsNV * kEPV;
  static constexpr int kCH = kThreads * kEPT;
  static constexpr int kESZ = sizeof(T) == 4 ? 4 : 2;
};

int sps_chunks_per_row(int dtype, int V) {
  const int ch = dtype == SMC_BF16 ? SpsGeom<bf16_tag>::kCH : SpsGeom<float>::kCH;
  return (V + ch - 1) / ch;
}

// The fp32 pass's chunk: kNV 16-byte vectors per thread and row, all in
// flight at once (twice the residual kernels' chunk).
template <typename T> struct FastGeom {
  static constexpr int kEPV = LogitTraits<T>::kPerVec;
  static constexpr int kNV = 4;
  static constexpr int kEPT = kNV * kEPV;
  static constexpr int kCH = kThreads * kEPT;
  static constexpr int kESZ = sizeof(T) == 4 ? 4 : 2;
  static constexpr int kLaneTerms = kEPT / 2;  // terms in each fp32 lane sum
};

static int sps_fast_chunks_per_row(int dtype, int V) {
  const int ch = dtype == SMC_BF16 ? FastGeom<bf16_tag>::kCH : FastGeom<float>::kCH;
  return (V + ch - 1) / ch;
}

struct SpsArgs {
  const char *target, *draft;
  int B, K, V, nch;
  int nchf;      // chunks of the fp32 pass (FastGeom)
  float tscale;  // s = 1/T
  int topp;      // nonzero: thresholds in ws.results[row].tok
  uint64_t seed;
  uint32_t step;
  int32_t *tokens_out;
  Workspace ws;
};

// The nucleus thresholds of rows p_j and q_j of prompt b (-inf: every logit).
__device__ __forceinline__ void sps_thresholds(const SpsArgs &a, int b, int jr, float *thr_p,
                                               float *thr_q) {
  const float kAll = kNegInf;
  if (!a.topp) { *thr_p = *thr_q = kAll; return; }
  const size_t base = static_cast<size_t>(b) * (2 * a.K + 1);
  *thr_p = __int_as_float(__ldcg(&a.ws.results[base + jr].tok));
  *thr_q = __int_as_float(__ldcg(&a.ws.results[base + a.K + 1 + jr].tok));
}

// exp(s x - L) for a float-float L, with s x taken exactly (two_prod).
__device__ __forceinline__ ff prob_term_s(float x, float s, ff big_l, const float2 *tab) {
  if (!(x > kNegInf)) return {0.f, 0.f};
  const ff sx = two_prod(s, x);
  const ff d = two_sum(sx.hi, -big_l.hi);
  return accurate_exp(d.hi, d.lo + (sx.lo - big_l.lo), tab);
}

// One row's chunk sum of exp(s (x - mc)) over the kept logits x[], mc their
// maximum: two logits at a time on the packed pipes (BonusPairSum), or, when
// mc is too large for the pair path's lower bound, by scalar terms.
template <typename T, int EPT>
__device__ __forceinline__ ff chunk_weight_sum(const float (&x)[EPT], float mc, float s,
                                               const float *th, const float *tl,
                                               const float2 *tab) {
  constexpr float kInf = -kNegInf;
  if (!(mc > kNegInf && mc < kInf)) return {0.f, 0.f};
  BonusPairSum ps;
  if (ps.init(mc, s, 40.f / s)) {
    const bool fast = sizeof(T) == 2 && BonusPairSum::fast_diff_ok(mc, 40.f / s);
    if (s == 1.f) {
      if (fast) {
#pragma unroll
        for (int e = 0; e < EPT; e += 2) ps.add<true, true>(x[e], x[e + 1], th, tl);
      } else {
#pragma unroll
        for (int e = 0; e < EPT; e += 2) ps.add<true, false>(x[e], x[e + 1], th, tl);
      }
    } else {
      if (fast) {
#pragma unroll
        for (int e = 0; e < EPT; e += 2) ps.add<false, true>(x[e], x[e + 1], th, tl);
      } else {
#pragma unroll
        for (int e = 0; e < EPT; e += 2) ps.add<false, false>(x[e], x[e + 1], th, tl);
      }
    }
    return ps.total();
  }
  ff S0{0.f, 0.f}, S1{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    if (e & 1) ff_accum(S1, weight_term(x[e], mc, s, tab));
    else ff_accum(S0, weight_term(x[e], mc, s, tab));
  }
  return ff_add(ff_norm(S0), ff_norm(S1));
}


// Shared memory of the SpS kernels.
struct SpsSmem {
  float2 tab[64];
  float th[64], tl[64];
  float red[2 * kWarps];
  float2 ffs[kWarps];
  float4 rec[2 * kWarps];
  float tred[8][kThreads];  // the one-pass CTA's per-thread sums, for warp 0 to add
  int ints[2 * kWarps];
  int last, sel, mode;
  float sel_m;
  float fcp, fe2;       // the fp32 pass's normaliser and doubled error bound
  int fsel;             // the fp32 pass's drawn token, or -1
  ff rem, lp, lq, total;
};

// Rows p_j and q_j of prompt b, element size esz.
__device__ __forceinline__ void sps_rows(const SpsArgs &a, int b, int jr, int esz,
                                         const char **prow, const char **qrow) {
  *prow = a.target + (static_cast<size_t>(b) * (a.K + 1) + jr) * static_cast<size_t>(a.V) * esz;
  *qrow = a.draft + (static_cast<size_t>(b) * a.K + jr) * static_cast<size_t>(a.V) * esz;
}

// Chunk c of rows p_j and q_j: each row's kept maximum mc and float-float sum
// of exp(s (x - mc)) over its kept logits, to sps_part_pq[(b nch + c) 2 + r]
// (r = 0: p, 1: q) as (mc, sum hi, sum lo, 0).  All threads call it.
template <typename T, bool VEC>
__device__ void stats_chunk(const SpsArgs &a, int b, int jr, int c, float thr_p, float thr_q,
                            SpsSmem &sm) {
  using G = SpsGeom<T>;
  const int tid = threadIdx.x;
  const int64_t c0 = static_cast<int64_t>(c) * G::kCH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - c0));
  const char *rows[2];
  sps_rows(a, b, jr, G::kESZ, &rows[0], &rows[1]);
  const float thr[2] = {thr_p, thr_q};
  // both rows' chunks in flight at once; logits outside a nucleus weigh 0
  float x[2][G::kEPT];
  load_chunk<T, VEC, kSpsNV>(rows[0] + c0 * G::kESZ, n_valid, x[0]);
  load_chunk<T, VEC, kSpsNV>(rows[1] + c0 * G::kESZ, n_valid, x[1]);
  float m[2] = {kNegInf, kNegInf};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
#pragma unroll
    for (int e = 0; e < G::kEPT; ++e) {
      if (!(x[r][e] >= thr[r])) x[r][e] = kNegInf;
      m[r] = fmaxf(m[r], x[r][e]);
    }
  }
  const float mcp = block_max(m[0], sm.red);
  const float mcq = block_max(m[1], sm.red);  // (block_max's barriers also cover the tables)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float mc = r == 0 ? mcp : mcq;
    const ff S = block_ff_sum(
        chunk_weight_sum<T, G::kEPT>(x[r], mc, a.tscale, sm.th, sm.tl, sm.tab), sm.ffs);
    if (tid == 0) {
      a.ws.sps_part_pq[(static_cast<size_t>(b) * a.nch + c) * 2 + r] = make_float4(mc, S.hi, S.lo, 0.f);
    }
  }
}

// Run by one full warp once every chunk's stats_chunk is visible: the
// float-float log-sum-exps of the kept parts of rows p_j and q_j (-inf for an
// empty one), to sps_stats[b] and returned.
__device__ void stats_combine(const SpsArgs &a, int b, const float2 *tab, ff *lp, ff *lq) {
  const int lane = threadIdx.x & 31;
  float lse[2][2];
  for (int r = 0; r < 2; ++r) {
    float M = kNegInf;
    for (int cc = lane; cc < a.nch; cc += 32) {
      M = fmaxf(M, __ldcg(&a.ws.sps_part_pq[(static_cast<size_t>(b) * a.nch + cc) * 2 + r].x));
    }
    M = warp_max(M);
    ff tot{0.f, 0.f};
    for (int c0w = 0; c0w < a.nch; c0w += 32) {
      const int cc = c0w + lane;
      ff val{0.f, 0.f};
      if (cc < a.nch && M > kNegInf) {
        const float4 q = __ldcg(&a.ws.sps_part_pq[(static_cast<size_t>(b) * a.nch + cc) * 2 + r]);
        if (q.x > kNegInf) val = ff_mul(ff{q.y, q.z}, ff_norm(weight_term(q.x, M, a.tscale, tab)));
      }
      tot = ff_add(tot, warp_ff_sum(val));
    }
    // log of the (kept) mass of exp(s l): s M (exact, as a pair) + log(total)
    const ff l = (M > kNegInf && tot.hi > 0.f)
                     ? ff_add(two_prod(a.tscale, M), ff_log(ff_norm(tot), tab))
                     : ff{kNegInf, 0.f};
    lse[r][0] = l.hi;
    lse[r][1] = l.lo;
  }
  if (lane == 0) a.ws.sps_stats[b] = make_float4(lse[0][0], lse[0][1], lse[1][0], lse[1][1]);
  *lp = ff{lse[0][0], lse[0][1]};
  *lq = ff{lse[1][0], lse[1][1]};
}

// max(0, p_v - q_v) for logits xp, xq, each probability zero outside its
// nucleus.
__device__ __forceinline__ ff residual_of(float xp, float xq, float s, ff lp, ff lq, float thr_p,
                                          float thr_q, const float2 *tab) {
  const ff p = xp >= thr_p ? ff_norm(prob_term_s(xp, s, lp, tab)) : ff{0.f, 0.f};
  const ff q = xq >= thr_q ? ff_norm(prob_term_s(xq, s, lq, tab)) : ff{0.f, 0.f};
  const ff d = ff_sub(p, q);
  return d.hi > 0.f ? d : ff{0.f, 0.f};
}

// Running float-float sums of nonnegative packed pairs: the heads start at 2,
// above any single addend, so the fast two-sum is exact at every addition.
struct PairAcc {
  unsigned long long h, l;
  __device__ __forceinline__ void init() {
    h = f2dup(2.f);
    l = 0ull;
  }
  __device__ __forceinline__ void add(unsigned long long xh, unsigned long long xl) {
    const unsigned long long s2 = add2(h, xh);
    l = add2(l, add2(sub2(xh, sub2(s2, h)), xl));
    h = s2;
  }
  __device__ __forceinline__ ff total() const {
    float a0, a1, o0, o1;
    f2unpack(h, a0, a1);
    f2unpack(l, o0, o1);
    ff r0 = two_sum(a0, -2.f), r1 = two_sum(a1, -2.f);
    r0.lo += o0;
    r1.lo += o1;
    return ff_add(ff_norm(r0), ff_norm(r1));
  }
};

// d = p - q of packed float-float pairs, normalised (NH, NL).
__device__ __forceinline__ void packed_diff(unsigned long long PH, unsigned long long PL,
                                            unsigned long long QH, unsigned long long QL,
                                            unsigned long long *NH, unsigned long long *NL) {
  const unsigned long long DH = sub2(PH, QH);
  const unsigned long long BB = sub2(DH, PH);
  const unsigned long long DE = sub2(sub2(PH, sub2(DH, BB)), add2(QH, BB));
  const unsigned long long DL = add2(DE, sub2(PL, QL));
  *NH = add2(DH, DL);
  *NL = sub2(DL, sub2(*NH, DH));
}

// Chunk c's residual mass sum_v max(0, p_v - q_v) in float-float, for exact
// log-sum-exps lp, lq of the kept rows, to sps_part_r[b nch + c].  All threads
// call it (the tables staged).
template <typename T, bool VEC>
__device__ void residual_chunk(const SpsArgs &a, int b, int jr, int c, ff lp, ff lq,
                               float thr_p, float thr_q, SpsSmem &sm) {
  using G = SpsGeom<T>;
  const int tid = threadIdx.x;
  const int64_t c0 = static_cast<int64_t>(c) * G::kCH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - c0));
  const char *prow, *qrow;
  sps_rows(a, b, jr, G::kESZ, &prow, &qrow);
  float xp[G::kEPT], xq[G::kEPT];
  load_chunk<T, VEC, kSpsNV>(prow + c0 * G::kESZ, n_valid, xp);
  load_chunk<T, VEC, kSpsNV>(qrow + c0 * G::kESZ, n_valid, xq);
  // p and q two logits at a time on the packed pipes, and the residual
  // max(0, p - q) of each in float-float as residual_of takes it: logits
  // outside a nucleus are set to -inf first (they then weigh about e^-59
  // instead of 0, far below what can move a draw)
  ShiftedExp ep, eq;
  ep.init(a.tscale, lp);
  eq.init(a.tscale, lq);
  const bool live = lp.hi > kNegInf && lq.hi > kNegInf;
  ff R{0.f, 0.f};
  if (live) {
    PairAcc acc;
    acc.init();
#pragma unroll
    for (int e = 0; e < G::kEPT; e += 2) {
      unsigned long long PH, PL, QH, QL, NH, NL;
      ep.eval(xp[e] >= thr_p ? xp[e] : kNegInf, xp[e + 1] >= thr_p ? xp[e + 1] : kNegInf, sm.th,
              sm.tl, &PH, &PL);
      eq.eval(xq[e] >= thr_q ? xq[e] : kNegInf, xq[e + 1] >= thr_q ? xq[e + 1] : kNegInf, sm.th,
              sm.tl, &QH, &QL);
      packed_diff(PH, PL, QH, QL, &NH, &NL);
      float h0, h1, l0, l1;
      f2unpack(NH, h0, h1);
      f2unpack(NL, l0, l1);
      acc.add(f2pack(h0 > 0.f ? h0 : 0.f, h1 > 0.f ? h1 : 0.f),
              f2pack(h0 > 0.f ? l0 : 0.f, h1 > 0.f ? l1 : 0.f));
    }
    R = acc.total();
  } else {
    ff R0{0.f, 0.f}, R1{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < G::kEPT; ++e) {
      const ff d = residual_of(xp[e], xq[e], a.tscale, lp, lq, thr_p, thr_q, sm.tab);
      if (d.hi > 0.f) {
        if (e & 1) ff_accum(R1, d);
        else ff_accum(R0, d);
      }
    }
    R = ff_add(ff_norm(R0), ff_norm(R1));
  }
  R = block_ff_sum(R, sm.ffs);
  if (tid == 0) a.ws.sps_part_r[static_cast<size_t>(b) * a.nch + c] = make_float2(R.hi, R.lo);
}

// The residual draw inside chunk [c0, c0 + len) of rows p_j and q_j, by the
// whole CTA, with exact log-sum-exps lp, lq: thread t takes the kEPT
// consecutive elements from t kEPT, evaluates their residuals
// max(0, p - q) two at a time on the packed pipes and keeps them in
// registers; a block scan of the threads' sums finds the thread whose run
// passes `target` (in the chunk's absolute units), which walks its own terms.
// Past the chunk's total (rounding), the last element with a residual.
// Elements whose p is zero (outside p's nucleus, -inf, past the row) weigh 0.
template <typename T, bool VEC>
__device__ __noinline__ int select_residual_in_chunk(const SpsArgs &a, const char *prow, const char *qrow,
                                        int64_t c0, int len, ff target, ff lp, ff lq,
                                        float thr_p, float thr_q, SpsSmem &sm) {
  using G = SpsGeom<T>;
  using Tr = LogitTraits<T>;
  constexpr int E = G::kEPT;
  const int tid = threadIdx.x;
  const int beg = tid * E;
  float xp[E], xq[E];
  if (VEC && beg + E <= len) {
    const uint4 *vp = reinterpret_cast<const uint4 *>(prow + (c0 + beg) * G::kESZ);
    const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + (c0 + beg) * G::kESZ);
#pragma unroll
    for (int i = 0; i < kSpsNV; ++i) {
      const uint4 up = __ldcg(vp + i), uq = __ldcg(vq + i);
#pragma unroll
      for (int e = 0; e < G::kEPV; ++e) {
        xp[i * G::kEPV + e] = Tr::at(up, e);
        xq[i * G::kEPV + e] = Tr::at(uq, e);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool in = beg + e < len;
      xp[e] = in ? Tr::scalar(prow, c0 + beg + e) : kNegInf;
      xq[e] = in ? Tr::scalar(qrow, c0 + beg + e) : kNegInf;
    }
  }
  ShiftedExp ep, eq;
  ep.init(a.tscale, lp);
  eq.init(a.tscale, lq);
  unsigned long long rh[E / 2], rl[E / 2];
  ff part{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    unsigned long long PH, PL, QH, QL, NH, NL;
    const bool k0 = xp[e] >= thr_p && xp[e] > kNegInf, k1 = xp[e + 1] >= thr_p && xp[e + 1] > kNegInf;
    ep.eval(k0 ? xp[e] : kNegInf, k1 ? xp[e + 1] : kNegInf, sm.th, sm.tl, &PH, &PL);
    eq.eval(xq[e] >= thr_q ? xq[e] : kNegInf, xq[e + 1] >= thr_q ? xq[e + 1] : kNegInf, sm.th,
            sm.tl, &QH, &QL);
    packed_diff(PH, PL, QH, QL, &NH, &NL);
    float h0, h1, l0, l1;
    f2unpack(NH, h0, h1);
    f2unpack(NL, l0, l1);
    const bool p0 = k0 && h0 > 0.f, p1 = k1 && h1 > 0.f;
    rh[e / 2] = f2pack(p0 ? h0 : 0.f, p1 ? h1 : 0.f);
    rl[e / 2] = f2pack(p0 ? l0 : 0.f, p1 ? l1 : 0.f);
    part = ff_add(part, ff_norm(ff{p0 ? h0 : 0.f, p0 ? l0 : 0.f}));
    part = ff_add(part, ff_norm(ff{p1 ? h1 : 0.f, p1 ? l1 : 0.f}));
  }
  ff total;
  const ff incl = block_ff_scan(part, sm.ffs, &total);
  const ff excl = ff_sub(incl, part);
  int cand = 0x7fffffff, last_pos = -1, first_pos = -1;
  ff run = excl;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    float h0, h1, l0, l1;
    f2unpack(rh[e / 2], h0, h1);
    f2unpack(rl[e / 2], l0, l1);
    if (h0 > 0.f) {
      last_pos = beg + e;
      if (first_pos < 0) first_pos = beg + e;
      run = ff_add(run, ff_norm(ff{h0, l0}));
      if (cand == 0x7fffffff && ff_gt(run, target)) cand = beg + e;
    }
    if (h1 > 0.f) {
      last_pos = beg + e + 1;
      if (first_pos < 0) first_pos = beg + e + 1;
      run = ff_add(run, ff_norm(ff{h1, l1}));
      if (cand == 0x7fffffff && ff_gt(run, target)) cand = beg + e + 1;
    }
  }
  // a thread whose run starts past the target (rounding) takes its first term
  if (part.hi > 0.f && ff_gt(excl, target)) cand = first_pos;
  if (!(part.hi > 0.f)) cand = 0x7fffffff;
  cand = block_min_i(cand, sm.ints);
  if (cand == 0x7fffffff) cand = -block_min_i(-last_pos, sm.ints);  // max over threads
  return cand < 0 ? -1 : static_cast<int>(c0 + cand);
}

// The draw once every chunk's residual mass is in sps_part_r (and, for the
// fallback below, every chunk's stats_chunk in sps_part_pq), run by the whole
// CTA: u from Philox (purpose RESIDUAL) picks the chunk by the chunk masses,
// then the element by a rescan of the chunk with exact residuals.  With no
// residual mass (p_j == q_j up to rounding) the token is drawn from p_j.
// Writes the token; `total` is the residual mass when already summed, else
// negative.
template <typename T, bool VEC>
__device__ __noinline__ void residual_select(const SpsArgs &a, int b, int jr, ff lp, ff lq, float thr_p,
                                float thr_q, ff total_in, SpsSmem &sm) {
  using G = SpsGeom<T>;
  using Tr = LogitTraits<T>;
  const int tid = threadIdx.x;
  const char *prow, *qrow;
  sps_rows(a, b, jr, G::kESZ, &prow, &qrow);
  if (tid < 32) {
    const int lane = tid;
    const float2 *pr = a.ws.sps_part_r + static_cast<size_t>(b) * a.nch;
    ff total = total_in;
    if (!(total.hi >= 0.f)) {
      total = ff{0.f, 0.f};
      for (int c0w = 0; c0w < a.nch; c0w += 32) {
        const int cc = c0w + lane;
        ff val{0.f, 0.f};
        if (cc < a.nch) val = ff{__ldcg(&pr[cc].x), __ldcg(&pr[cc].y)};
        total = ff_add(total, warp_ff_sum(val));
      }
    }
    const float u = philox_uniform(a.seed, a.step, b, jr, SMC_PURPOSE_RESIDUAL);
    ff rem{0.f, 0.f};
    int sel, mode;
    float sel_m = 0.f;
    if (total.hi > 0.f) {
      mode = 0;  // residual mass, absolute units in every chunk
      sel = warp_find_chunk(a.nch, ff_mul_f(total, u),
                            [&](int cc, ff *val, ff *f) {
                              *val = ff{__ldcg(&pr[cc].x), __ldcg(&pr[cc].y)};
                            },
                            &rem);
    } else {
      mode = 1;  // no residual mass (p_j == q_j up to rounding): draw from p_j
      const float4 *pq = a.ws.sps_part_pq + static_cast<size_t>(b) * a.nch * 2;
      float M = kNegInf;
      for (int cc = lane; cc < a.nch; cc += 32) M = fmaxf(M, __ldcg(&pq[cc * 2].x));
      M = warp_max(M);
      auto chunk_mass = [&](int cc, ff *val, ff *f) {
        const float4 q = __ldcg(&pq[cc * 2]);
        if (q.x > kNegInf) {
          *f = ff_norm(weight_term(q.x, M, a.tscale, sm.tab));
          *val = ff_mul(ff{q.y, q.z}, *f);
        }
      };
      ff ptot{0.f, 0.f};
      for (int c0w = 0; c0w < a.nch; c0w += 32) {
        const int cc = c0w + lane;
        ff val{0.f, 0.f}, f{1.f, 0.f};
        if (cc < a.nch) chunk_mass(cc, &val, &f);
        ptot = ff_add(ptot, warp_ff_sum(val));
      }
      sel = warp_find_chunk(a.nch, ff_mul_f(ptot, u), chunk_mass, &rem);
      if (sel >= 0) sel_m = __ldcg(&pq[sel * 2].x);
    }
    if (lane == 0) {
      sm.sel = sel;
      sm.mode = mode;
      sm.sel_m = sel_m;
      sm.rem = rem;
    }
  }
  __syncthreads();
  const int sel = sm.sel;
  int tok = -1;
  if (sel >= 0) {
    const int64_t sc0 = static_cast<int64_t>(sel) * G::kCH;
    const int len = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - sc0));
    if (sm.mode == 0) {
      tok = select_residual_in_chunk<T, VEC>(a, prow, qrow, sc0, len, sm.rem, lp, lq, thr_p,
                                             thr_q, sm);
    } else {
      const float cm = sm.sel_m;
      tok = block_select_in_chunk(
          sc0, len, sm.rem,
          [&](int64_t i) {
            const float x = Tr::scalar(prow, i);
            return x >= thr_p ? weight_term(x, cm, a.tscale, sm.tab) : ff{0.f, 0.f};
          },
          sm.ffs, sm.ints);
    }
  }
  if (tid == 0) a.tokens_out[static_cast<size_t>(b) * (a.K + 1) + jr] = tok;
}

// The two-pass route for one prompt, run by one whole CTA: stats_chunk over
// every chunk, the exact log-sum-exps, residual_chunk over every chunk, the
// draw.
template <typename T, bool VEC>
__device__ __noinline__ void sps_two_pass_one_cta(const SpsArgs &a, int b, int jr, float thr_p, float thr_q,
                                     SpsSmem &sm) {
  for (int cc = 0; cc < a.nch; ++cc) stats_chunk<T, VEC>(a, b, jr, cc, thr_p, thr_q, sm);
  __syncthreads();
  if (threadIdx.x < 32) {
    ff lp, lq;
    stats_combine(a, b, sm.tab, &lp, &lq);
    if (threadIdx.x == 0) {
      sm.lp = lp;
      sm.lq = lq;
    }
  }
  __syncthreads();
  const ff lp = sm.lp, lq = sm.lq;
  for (int cc = 0; cc < a.nch; ++cc) residual_chunk<T, VEC>(a, b, jr, cc, lp, lq, thr_p, thr_q, sm);
  __syncthreads();
  residual_select<T, VEC>(a, b, jr, lp, lq, thr_p, thr_q, ff{-1.f, 0.f}, sm);
}

__device__ __forceinline__ void sps_stage_tables(SpsSmem &sm) {
  stage_exp2_table(sm.tab);
  stage_exp2_split(sm.th, sm.tl);
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) sps_stats_kernel(const SpsArgs a) {
  __shared__ SpsSmem sm;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the acceptance scan's results
  // the residual pass may launch once every CTA has started; it waits for
  // this grid before it reads the statistics
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int jr = a.ws.sps_rej[b];
  if (jr < 0) return;
  sps_stage_tables(sm);
  float thr_p, thr_q;
  sps_thresholds(a, b, jr, &thr_p, &thr_q);
  stats_chunk<T, VEC>(a, b, jr, c, thr_p, thr_q, sm);
  if (tid == 0) {
    __threadfence();
    sm.last = atomicAdd(&a.ws.sps_ticket_a[b], 1u) == static_cast<unsigned>(a.nch - 1);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (tid < 32) {
    ff lp, lq;
    stats_combine(a, b, sm.tab, &lp, &lq);
    if (tid == 0) a.ws.sps_ticket_a[b] = 0u;
  }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) sps_residual_kernel(const SpsArgs a) {
  __shared__ SpsSmem sm;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  // the next call's row pass may launch once every CTA has started: it
  // writes only its own copy of the row partials and counters
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the statistics
  const int jr = a.ws.sps_rej[b];
  if (jr < 0) return;
  sps_stage_tables(sm);
  const float4 st = a.ws.sps_stats[b];
  const ff lp{st.x, st.y}, lq{st.z, st.w};
  float thr_p, thr_q;
  sps_thresholds(a, b, jr, &thr_p, &thr_q);
  __syncthreads();  // tables staged
  residual_chunk<T, VEC>(a, b, jr, c, lp, lq, thr_p, thr_q, sm);
  if (tid == 0) {
    __threadfence();
    sm.last = atomicAdd(&a.ws.sps_ticket_b[b], 1u) == static_cast<unsigned>(a.nch - 1);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (tid == 0) a.ws.sps_ticket_b[b] = 0u;
  residual_select<T, VEC>(a, b, jr, lp, lq, thr_p, thr_q, ff{-1.f, 0.f}, sm);
}

// Appends prompt b to a queue of capacity cap (one entry per prompt and call;
// the bound only keeps a workspace left half-used by a failed call in range).
__device__ __forceinline__ void queue_push(unsigned *n, int32_t *list, int cap, int b) {
  const unsigned slot = atomicAdd(n, 1u);
  if (slot < static_cast<unsigned>(cap)) list[slot] = b;
}

// The one-pass route's tolerances.  tau bounds the ratio error it accepts
// (|rho - 1| <= tau / 2) and sets the close-call band |p_v - q_v| <= tau q_v;
// the chunk masses may move by at most kSpsMassBound of the residual mass.
// The first pass shifts by the row kernel's log-sum-exps (about 1e-7); the
// retry pass by exact ones.
constexpr float kSpsTauFirst = 4e-6f;
constexpr float kSpsTauRetry = 1e-8f;
constexpr float kSpsMassBound = 2e-10f;

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Chunk c of prompt b without top-p, with P_v = exp(s x_v - lp0) and
// Q_v = exp(s y_v - lq0) for shifts lp0, lq0 near the rows' log-sum-exps
// (p_v = P_v / sum P, q_v = Q_v / sum Q): the float-float sums of P and Q,
// the residual at ratio 1, R1 = sum max(0, P - Q), the Q-mass where P > Q
// (AQ) and the Q-mass of the close calls (CQ), to
// sps_part_pq[(b nch + c) 2 + {0, 1}].  The prompt's last CTA (ticket) sets
// cp = 1 / sum P, cq = 1 / sum Q; chunk c's residual mass is
// cp R1 + (cp - cq) AQ, exact but for close calls, which move it by at most
// |cp - cq| CQ.  If that bound or the ratio is out of range: on the first
// pass the prompt is queued for the retry pass with the exact log-sum-exps
// (sps_stats); on the retry pass, or when no residual is left or a shift is
// not finite, the CTA takes the two-pass route alone.
template <typename T, bool VEC>
__device__ void onepass_chunk(const SpsArgs &a, int b, int jr, int c, ff lp0, ff lq0, bool retry,
                              unsigned *ticket, SpsSmem &sm) {
  using G = SpsGeom<T>;
  constexpr float kInf = -kNegInf;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float tau = retry ? kSpsTauRetry : kSpsTauFirst;
  const bool live = fabsf(lp0.hi) < kInf && fabsf(lq0.hi) < kInf;
  const int64_t c0 = static_cast<int64_t>(c) * G::kCH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - c0));
  const char *prow, *qrow;
  sps_rows(a, b, jr, G::kESZ, &prow, &qrow);
  float xp[G::kEPT], xq[G::kEPT];
  load_chunk<T, VEC, kSpsNV>(prow + c0 * G::kESZ, n_valid, xp);
  load_chunk<T, VEC, kSpsNV>(qrow + c0 * G::kESZ, n_valid, xq);
  __syncthreads();  // tables staged; the previous prompt's shared state read
  ff sp{0.f, 0.f}, sq{0.f, 0.f}, r1{0.f, 0.f};
  float aq = 0.f, cq = 0.f;
  if (live) {
    ShiftedExp ep, eq;
    ep.init(a.tscale, lp0);
    eq.init(a.tscale, lq0);
    PairAcc accp, accq, accr;
    accp.init();
    accq.init();
    accr.init();
    unsigned long long aq2 = 0ull, cq2 = 0ull;
#pragma unroll
    for (int e = 0; e < G::kEPT; e += 2) {
      unsigned long long PH, PL, QH, QL, NH, NL;
      ep.eval(xp[e], xp[e + 1], sm.th, sm.tl, &PH, &PL);
      eq.eval(xq[e], xq[e + 1], sm.th, sm.tl, &QH, &QL);
      accp.add(PH, PL);
      accq.add(QH, QL);
      packed_diff(PH, PL, QH, QL, &NH, &NL);
      float h0, h1, l0, l1, q0, q1;
      f2unpack(NH, h0, h1);
      f2unpack(NL, l0, l1);
      f2unpack(QH, q0, q1);
      accr.add(f2pack(h0 > 0.f ? h0 : 0.f, h1 > 0.f ? h1 : 0.f),
               f2pack(h0 > 0.f ? l0 : 0.f, h1 > 0.f ? l1 : 0.f));
      aq2 = add2(aq2, f2pack(h0 > 0.f ? q0 : 0.f, h1 > 0.f ? q1 : 0.f));
      cq2 = add2(cq2, f2pack(fabsf(h0) <= tau * q0 ? q0 : 0.f, fabsf(h1) <= tau * q1 ? q1 : 0.f));
    }
    sp = accp.total();
    sq = accq.total();
    r1 = accr.total();
    float a0, a1;
    f2unpack(aq2, a0, a1);
    aq = a0 + a1;
    f2unpack(cq2, a0, a1);
    cq = a0 + a1;
  }
  // the CTA's sums, by warp 0 alone: each lane adds kWarps threads' values
  // from shared memory, then the warp's lanes by shuffles
  sm.tred[0][tid] = sp.hi;
  sm.tred[1][tid] = sp.lo;
  sm.tred[2][tid] = sq.hi;
  sm.tred[3][tid] = sq.lo;
  sm.tred[4][tid] = r1.hi;
  sm.tred[5][tid] = r1.lo;
  sm.tred[6][tid] = aq;
  sm.tred[7][tid] = cq;
  __syncthreads();
  if (warp == 0) {
    ff tsp{0.f, 0.f}, tsq{0.f, 0.f}, tr1{0.f, 0.f};
    float taq = 0.f, tcq = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int t = lane + 32 * w;
      tsp = ff_add(tsp, ff{sm.tred[0][t], sm.tred[1][t]});
      tsq = ff_add(tsq, ff{sm.tred[2][t], sm.tred[3][t]});
      tr1 = ff_add(tr1, ff{sm.tred[4][t], sm.tred[5][t]});
      taq += sm.tred[6][t];
      tcq += sm.tred[7][t];
    }
    tsp = warp_ff_sum(tsp);
    tsq = warp_ff_sum(tsq);
    tr1 = warp_ff_sum(tr1);
    taq = warp_sum_f(taq);
    tcq = warp_sum_f(tcq);
    if (lane == 0) {
      float4 *rec = a.ws.sps_part_pq + (static_cast<size_t>(b) * a.nch + c) * 2;
      rec[0] = make_float4(tsp.hi, tsp.lo, tsq.hi, tsq.lo);
      rec[1] = make_float4(tr1.hi, tr1.lo, taq, tcq);
      __threadfence();
      sm.last = atomicAdd(ticket + b, 1u) == static_cast<unsigned>(a.nch - 1);
    }
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (tid < 32) {
    const float4 *rec = a.ws.sps_part_pq + static_cast<size_t>(b) * a.nch * 2;
    ff tp{0.f, 0.f}, tq{0.f, 0.f};
    float cqs = 0.f;
    for (int cc = lane; cc < a.nch; cc += 32) {
      const float4 u0 = __ldcg(rec + 2 * cc), u1 = __ldcg(rec + 2 * cc + 1);
      tp = ff_add(tp, ff{u0.x, u0.y});
      tq = ff_add(tq, ff{u0.z, u0.w});
      cqs += u1.w;
    }
    tp = warp_ff_sum(tp);
    tq = warp_ff_sum(tq);
    cqs = warp_sum_f(cqs);
    const bool shifts_ok = live && tp.hi > 0.f && tp.hi < kInf && tq.hi > 0.f && tq.hi < kInf;
    bool fast = false;
    ff total{0.f, 0.f};
    if (shifts_ok) {
      const ff cp = ff_div(ff{1.f, 0.f}, tp), cqn = ff_div(ff{1.f, 0.f}, tq);
      const ff dc = ff_sub(cp, cqn);
      float2 *pr = a.ws.sps_part_r + static_cast<size_t>(b) * a.nch;
      for (int cc = lane; cc < a.nch; cc += 32) {
        const float4 u1 = __ldcg(rec + 2 * cc + 1);
        ff rc = ff_add(ff_mul(cp, ff{u1.x, u1.y}), ff_mul_f(dc, u1.z));
        if (!(rc.hi > 0.f)) rc = ff{0.f, 0.f};
        pr[cc] = make_float2(rc.hi, rc.lo);
        total = ff_add(total, rc);
      }
      total = warp_ff_sum(total);
      const float rho_m1 = ff_sub(ff_div(tp, tq), ff{1.f, 0.f}).hi;
      fast = fabsf(rho_m1) <= 0.5f * tau && total.hi > 0.f && total.hi < kInf &&
             fabsf(dc.hi) * cqs <= kSpsMassBound * total.hi;
      __syncwarp();
    }
    if (lane == 0) {
      const ff lp = ff_add(lp0, ff_log(tp, sm.tab)), lq = ff_add(lq0, ff_log(tq, sm.tab));
      // 0: draw now; 1: queue for the retry pass; 2: two-pass route here
      sm.mode = fast ? 0 : (!retry && shifts_ok && total.hi > 0.f) ? 1 : 2;
      sm.total = total;
      sm.lp = lp;
      sm.lq = lq;
      ticket[b] = 0u;
      if (sm.mode == 1) {
        a.ws.sps_stats[b] = make_float4(lp.hi, lp.lo, lq.hi, lq.lo);
        queue_push(a.ws.sps_retry_n, a.ws.sps_retry, a.B, b);
      }
    }
  }
  __syncthreads();
  const int mode = sm.mode;
  if (mode == 0) {
    residual_select<T, VEC>(a, b, jr, sm.lp, sm.lq, kNegInf, kNegInf, sm.total, sm);
  } else if (mode == 2) {
    sps_two_pass_one_cta<T, VEC>(a, b, jr, kNegInf, kNegInf, sm);
  }
}

// Retry pass over the queued prompts, shifts exact: CTA (c, k) takes chunk c
// of queue entries k, k + gridDim.y, ...  The grid's last CTA clears the
// queue.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) sps_retry_kernel(const SpsArgs a) {
  __shared__ SpsSmem sm;
  // The next call's row pass may launch now and stream beside this pass: it
  // writes only its own copy of the row partials and counters, and lets its
  // own dependents launch only after this grid has ended.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the first pass's queue
  // the float-float pass, and with it the fp32 pass, has finished
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.ws.sps_ff_n = 0u;
  const unsigned n = min(__ldcg(a.ws.sps_retry_n), static_cast<unsigned>(a.B));
  if (n > 0u) sps_stage_tables(sm);
  for (unsigned k = blockIdx.y; k < n; k += gridDim.y) {
    const int b = __ldcg(a.ws.sps_retry + k);
    // an entry left by a call that failed between its launches is skipped
    if (b < 0 || b >= a.B) continue;
    const int jr = a.ws.sps_rej[b];
    if (jr < 0 || jr >= a.K) continue;
    const float4 st = __ldcg(a.ws.sps_stats + b);
    onepass_chunk<T, VEC>(a, b, jr, blockIdx.x, ff{st.x, st.y}, ff{st.z, st.w}, true,
                          a.ws.sps_ticket_b, sm);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.ws.sps_retry_done, 1u) == gridDim.x * gridDim.y - 1u) {
      *a.ws.sps_retry_n = 0u;
      *a.ws.sps_retry_done = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// The fp32 first pass (no top-p), ahead of sps_onepass_kernel.  Each
// probability is taken in fp32 against the row kernel's log-sum-exp L:
// P_v = 2^y_v, y_v = log2(e) (s x_v - L), with t = s x - L.hi by one FMA,
// y = t log2(e) - L.lo log2(e) by another and 2^y by the hardware
// approximation.  Per element
//   |P^_v - P_v| <= P^_v (kArgErr |y_v| + kEx2Err):
// the two roundings of y and the rounding of log2(e) move y by at most three
// units in the last place of |y| (ln 2 of that through 2^y), and kEx2Err is
// twice the 2-ulp accuracy CUDA documents for its exp2 approximation.  Below
// 2^-126 the approximation flushes to 0, which no bound here can notice.
// Lane sums are sequential fp32 sums of kLaneTerms non-negative terms (as many
// units of their value); everything after them is float-float.
//
// With those, the prompt's last CTA bounds by E the distance between the
// computed residual CDF and the exact one at every vocabulary prefix, and the
// distance between its target u R and the exact one:
//   E = 1.05 (2 kArgErr (B_p + B_q) / min(S_p, S_q) + 4 kEx2Err
//             + kFastRoundUnits u + |cp - cq| S_q),
// S the sums of P^ and Q^, B the sums of P^ |y| and Q^ |y|, cp = 1 / S_p,
// cq = 1 / S_q.  The weights are cp max(P^ - Q^, 0).  Each row's element
// errors count twice (once in the terms, once in the normaliser); the lane
// sums, the normalisers' division and the roundings of the weights take at
// most kFastRoundUnits units; and weighing Q^ by cp instead of cq moves each
// weight by at most |cp - cq| Q^_v (max is 1-Lipschitz).  The CTA draws only
// when u R lies farther than 2E from both edges of the chosen token's
// interval: that token is then the exact one.  The prompts it leaves (the
// draws that land among tokens narrower than about E, about one in five on
// the serving rows) go to a queue for sps_ff_kernel.
constexpr float kU32 = 0x1p-24f;
constexpr float kArgErr = 2.09f * kU32;
constexpr float kEx2Err = 0x1p-21f;
constexpr float kFastRoundUnits = 64.f;  // >= 3 kLaneTerms + 12 for either dtype
static_assert(3 * FastGeom<bf16_tag>::kLaneTerms + 12 <= 64, "rounding budget");

// 2^(log2(e) (s x - L)) two logits at a time, in fp32, and |y| for the bound.
struct FastShiftedExp {
  unsigned long long s2, nlh, l2e, nll;
  float lbx;
  bool s1;

  __device__ __forceinline__ void init(float s, ff big_l) {
    s1 = s == 1.f;
    s2 = f2dup(s);
    nlh = f2dup(-big_l.hi);
    l2e = f2dup(kLog2e);
    nll = f2dup(-big_l.lo * kLog2e);
    lbx = (big_l.hi - 140.f) / s;  // below it 2^y flushes to 0 (NaN logits too)
  }

  // lbx rounded down to a bfloat16, for clamping packed bf16 logits
  __device__ __forceinline__ uint32_t lbx_bf16x2() const {
    uint32_t bits = __float_as_uint(lbx) & 0xffff0000u;
    if (__uint_as_float(bits) > lbx) bits += 0x10000u;  // negative: one step down
    return bits | (bits >> 16);
  }

  // P = 2^y and y for logits x0, x1; kClamped: already at least lbx.
  template <bool kClamped>
  __device__ __forceinline__ void eval(float x0, float x1, float *p0, float *p1, float *y0,
                                       float *y1) const {
    const unsigned long long X =
        kClamped ? f2pack(x0, x1) : f2pack(fmaxf(x0, lbx), fmaxf(x1, lbx));
    const unsigned long long T = s1 ? add2(X, nlh) : fma2(s2, X, nlh);
    f2unpack(fma2(T, l2e, nll), *y0, *y1);
    *p0 = fast_exp2(*y0);
    *p1 = fast_exp2(*y1);
  }
};

// The fp32 pass's weights for elements [c0 + g, c0 + g + n) of rows p_j and
// q_j, n = SpsGeom<T>::kEPT (elements at or past len weigh 0):
// cp max(D_v, 0), D_v = P^_v - Q^_v, as the chunk sums took them.
template <typename T, bool VEC>
__device__ __forceinline__ void fast_group_weights(const char *prow, const char *qrow,
                                                   int64_t c0, int len, int g,
                                                   const FastShiftedExp &fp,
                                                   const FastShiftedExp &fq, float cp,
                                                   float (&v)[SpsGeom<T>::kEPT]) {
  using G = SpsGeom<T>;
  using Tr = LogitTraits<T>;
  constexpr int E = G::kEPT;
  float xp[E], xq[E];
  if (VEC && g + E <= len) {
    const uint4 *vp = reinterpret_cast<const uint4 *>(prow + (c0 + g) * G::kESZ);
    const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + (c0 + g) * G::kESZ);
#pragma unroll
    for (int i = 0; i < kSpsNV; ++i) {
      const uint4 up = __ldcg(vp + i), uq = __ldcg(vq + i);
#pragma unroll
      for (int e = 0; e < G::kEPV; ++e) {
        xp[i * G::kEPV + e] = Tr::at(up, e);
        xq[i * G::kEPV + e] = Tr::at(uq, e);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool in = g + e < len;
      xp[e] = in ? Tr::scalar(prow, c0 + g + e) : kNegInf;
      xq[e] = in ? Tr::scalar(qrow, c0 + g + e) : kNegInf;
    }
  }
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    float p0, p1, q0, q1, y0, y1, d0, d1;
    fp.eval<false>(xp[e], xp[e + 1], &p0, &p1, &y0, &y1);
    fq.eval<false>(xq[e], xq[e + 1], &q0, &q1, &y0, &y1);
    f2unpack(sub2(f2pack(p0, p1), f2pack(q0, q1)), d0, d1);
    v[e] = cp * fmaxf(d0, 0.f);
    v[e + 1] = cp * fmaxf(d1, 0.f);
  }
}

// The fp32 pass's draw inside chunk [c0, c0 + len) of rows p_j and q_j, by
// the whole CTA: thread t takes the FastGeom<T>::kEPT consecutive elements
// from t kEPT, sums their weights, and after a block scan walks them again.
// Running sums are float-float.  Returns the first element whose running sum
// passes `target` (chunk units) when its interval holds
// [target - e2, target + e2], else -1.
template <typename T, bool VEC>
__device__ __noinline__ int fast_select_in_chunk(const char *prow, const char *qrow, int64_t c0,
                                                 int len, ff target, float e2,
                                                 const FastShiftedExp &fp,
                                                 const FastShiftedExp &fq, float cp,
                                                 SpsSmem &sm) {
  constexpr int E = SpsGeom<T>::kEPT;
  constexpr int kGroups = FastGeom<T>::kEPT / E;
  const int tid = threadIdx.x;
  const int beg = tid * FastGeom<T>::kEPT;
  ff part{0.f, 0.f};
#pragma unroll 1
  for (int g = 0; g < kGroups; ++g) {
    float v[E];
    fast_group_weights<T, VEC>(prow, qrow, c0, len, beg + g * E, fp, fq, cp, v);
#pragma unroll
    for (int e = 0; e < E; ++e) part = ff_add(part, ff{v[e], 0.f});
  }
  ff total;
  const ff incl = block_ff_scan(part, sm.ffs, &total);
  ff run = ff_sub(incl, part), before{0.f, 0.f}, after{0.f, 0.f};
  int cand = 0x7fffffff;
#pragma unroll 1
  for (int g = 0; g < kGroups && cand == 0x7fffffff; ++g) {
    float v[E];
    fast_group_weights<T, VEC>(prow, qrow, c0, len, beg + g * E, fp, fq, cp, v);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (v[e] != 0.f && cand == 0x7fffffff) {
        const ff prev = run;
        run = ff_add(run, ff{v[e], 0.f});
        if (ff_gt(run, target)) {
          cand = beg + g * E + e;
          before = prev;
          after = run;
        }
      }
    }
  }
  if (tid == 0) sm.fsel = -1;
  const int win = block_min_i(cand, sm.ints);  // its barriers order the store above
  if (win != 0x7fffffff && cand == win) {
    const bool ok = ff_sub(target, before).hi > e2 && ff_sub(after, target).hi > e2;
    sm.fsel = ok ? static_cast<int>(c0 + cand) : -1;
  }
  __syncthreads();
  return sm.fsel;
}

// One CTA per (fp32 chunk, prompt) without top-p: the chunk's sums of P^, Q^
// and D+ = max(D, 0) and the bound sum P^ |y| + Q^ |y| to
// sps_part_pq[(b nchf + c) 2 + {0, 1}]; the prompt's last CTA (ticket) draws
// when E settles the token, else queues the prompt for the float-float pass.
// Every vector of the chunk is requested before any arithmetic, bf16 logits
// are clamped two at a time, and the four sums are added by four warps at
// once.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) sps_fast_kernel(const SpsArgs a) {
  __shared__ SpsSmem sm;
  using G = FastGeom<T>;
  using Tr = LogitTraits<T>;
  constexpr float kInf = -kNegInf;
  constexpr bool kPackedClamp = VEC && sizeof(T) == 2;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the acceptance scan's results
  // the float-float pass may launch once every CTA has started; it waits for
  // this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int jr = a.ws.sps_rej[b];
  if (jr < 0) return;
  const char *prow, *qrow;
  sps_rows(a, b, jr, G::kESZ, &prow, &qrow);
  const int64_t c0 = static_cast<int64_t>(c) * G::kCH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - c0));
  uint4 rawp[G::kNV], rawq[G::kNV];
  if (VEC) {
    const uint4 *vp = reinterpret_cast<const uint4 *>(prow + c0 * G::kESZ);
    const uint4 *vq = reinterpret_cast<const uint4 *>(qrow + c0 * G::kESZ);
#pragma unroll
    for (int i = 0; i < G::kNV; ++i) {
      const int vi = i * kThreads + tid;
      const bool in = vi * G::kEPV < n_valid;
      rawp[i] = in ? ld_stream16(vp + vi) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
      rawq[i] = in ? ld_stream16(vq + vi) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
    }
  }
  const RowResult *res = a.ws.results + static_cast<size_t>(b) * (2 * a.K + 1);
  const float4 rp = __ldcg(reinterpret_cast<const float4 *>(res + jr));
  const float4 rq = __ldcg(reinterpret_cast<const float4 *>(res + a.K + 1 + jr));
  const ff lp0{rp.x, rp.z}, lq0{rq.x, rq.z};
  const bool live = fabsf(lp0.hi) < kInf && fabsf(lq0.hi) < kInf;
  FastShiftedExp fp, fq;
  fp.init(a.tscale, lp0);
  fq.init(a.tscale, lq0);
  float sp = 0.f, sq = 0.f, r1 = 0.f, bnd = 0.f;
  if (live) {
    const uint32_t lbp = fp.lbx_bf16x2(), lbq = fq.lbx_bf16x2();
    unsigned long long SP = 0ull, SQ = 0ull, R1 = 0ull;
#pragma unroll
    for (int i = 0; i < G::kNV; ++i) {
      const int vi = i * kThreads + tid;
      float xp[G::kEPV], xq[G::kEPV];
      if (kPackedClamp) {
        // -inf past the row (the fill above) and NaN become the clamp too
        uint4 wp = rawp[i], wq = rawq[i];
        wp.x = bmax2(wp.x, lbp); wp.y = bmax2(wp.y, lbp);
        wp.z = bmax2(wp.z, lbp); wp.w = bmax2(wp.w, lbp);
        wq.x = bmax2(wq.x, lbq); wq.y = bmax2(wq.y, lbq);
        wq.z = bmax2(wq.z, lbq); wq.w = bmax2(wq.w, lbq);
#pragma unroll
        for (int e = 0; e < G::kEPV; ++e) {
          xp[e] = Tr::at(wp, e);
          xq[e] = Tr::at(wq, e);
        }
      } else {
#pragma unroll
        for (int e = 0; e < G::kEPV; ++e) {
          const int idx = vi * G::kEPV + e;
          if (VEC) {
            const bool in = vi * G::kEPV < n_valid;
            xp[e] = in ? Tr::at(rawp[i], e) : kNegInf;
            xq[e] = in ? Tr::at(rawq[i], e) : kNegInf;
          } else {
            xp[e] = idx < n_valid ? Tr::scalar(prow, c0 + idx) : kNegInf;
            xq[e] = idx < n_valid ? Tr::scalar(qrow, c0 + idx) : kNegInf;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < G::kEPV; e += 2) {
        float p0, p1, q0, q1, yp0, yp1, yq0, yq1, d0, d1;
        fp.eval<kPackedClamp>(xp[e], xp[e + 1], &p0, &p1, &yp0, &yp1);
        fq.eval<kPackedClamp>(xq[e], xq[e + 1], &q0, &q1, &yq0, &yq1);
        const unsigned long long P = f2pack(p0, p1), Q = f2pack(q0, q1);
        SP = add2(SP, P);
        SQ = add2(SQ, Q);
        f2unpack(sub2(P, Q), d0, d1);
        R1 = add2(R1, f2pack(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
        bnd = fmaf(p0, fabsf(yp0), bnd);
        bnd = fmaf(p1, fabsf(yp1), bnd);
        bnd = fmaf(q0, fabsf(yq0), bnd);
        bnd = fmaf(q1, fabsf(yq1), bnd);
      }
    }
    float a0, a1;
    f2unpack(SP, a0, a1);
    sp = a0 + a1;
    f2unpack(SQ, a0, a1);
    sq = a0 + a1;
    f2unpack(R1, a0, a1);
    r1 = a0 + a1;
  }
  // the CTA's four sums, one per warp: warps 0-2 add S_p, S_q and D+ in
  // float-float, warp 3 the bound sum
  sm.tred[0][tid] = sp;
  sm.tred[1][tid] = sq;
  sm.tred[2][tid] = r1;
  sm.tred[3][tid] = bnd;
  __syncthreads();
  if (warp < 3) {
    ff t{0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t = ff_add(t, ff{sm.tred[warp][lane + 32 * w], 0.f});
    t = warp_ff_sum(t);
    if (lane == 0) sm.ffs[warp] = make_float2(t.hi, t.lo);
  } else if (warp == 3) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += sm.tred[3][lane + 32 * w];
    t = warp_sum_f(t);
    if (lane == 0) sm.red[0] = t;
  }
  __syncthreads();
  if (tid == 0) {
    float4 *rec = a.ws.sps_part_pq + (static_cast<size_t>(b) * a.nchf + c) * 2;
    rec[0] = make_float4(sm.ffs[0].x, sm.ffs[0].y, sm.ffs[1].x, sm.ffs[1].y);
    rec[1] = make_float4(sm.ffs[2].x, sm.ffs[2].y, 0.f, sm.red[0]);
    __threadfence();
    sm.last = atomicAdd(a.ws.sps_ticket_a + b, 1u) == static_cast<unsigned>(a.nchf - 1);
  }
  __syncthreads();
  if (!sm.last) return;
  __threadfence();
  if (warp == 0) {
    const float4 *rec = a.ws.sps_part_pq + static_cast<size_t>(b) * a.nchf * 2;
    ff tp{0.f, 0.f}, tq{0.f, 0.f};
    float tb = 0.f;
    for (int cc = lane; cc < a.nchf; cc += 32) {
      const float4 u0 = __ldcg(rec + 2 * cc), u1 = __ldcg(rec + 2 * cc + 1);
      tp = ff_add(tp, ff{u0.x, u0.y});
      tq = ff_add(tq, ff{u0.z, u0.w});
      tb += u1.w;
    }
    tp = warp_ff_sum(tp);
    tq = warp_ff_sum(tq);
    tb = warp_sum_f(tb);
    bool ok = live && tp.hi > 0.f && tp.hi < kInf && tq.hi > 0.f && tq.hi < kInf && tb < kInf;
    int sel = -1;
    ff rem{0.f, 0.f};
    float cp = 0.f, e2 = 0.f;
    if (ok) {
      cp = 1.f / tp.hi;
      // the weights are cp max(D, 0): against max(0, cp P^ - cq Q^) that
      // moves each by at most |cp - cq| Q^ (max is 1-Lipschitz)
      const float dc = cp - 1.f / tq.hi;
      const float err = 1.05f * (2.f * kArgErr * tb / fminf(tp.hi, tq.hi) + 4.f * kEx2Err +
                                 kFastRoundUnits * kU32 + 1.001f * fabsf(dc) * tq.hi);
      e2 = 2.f * err;
      auto chunk_mass = [&](int cc, ff *val, ff *f) {
        const float4 u1 = __ldcg(rec + 2 * cc + 1);
        const ff rc = ff_mul_f(ff{u1.x, u1.y}, cp);
        *val = rc.hi > 0.f ? rc : ff{0.f, 0.f};
      };
      ff total{0.f, 0.f};
      for (int c0w = 0; c0w < a.nchf; c0w += 32) {
        const int cc = c0w + lane;
        ff val{0.f, 0.f}, f{1.f, 0.f};
        if (cc < a.nchf) chunk_mass(cc, &val, &f);
        total = ff_add(total, warp_ff_sum(val));
      }
      ok = e2 < kInf && total.hi > 2.f * e2;
      if (ok) {
        const float u = philox_uniform(a.seed, a.step, b, jr, SMC_PURPOSE_RESIDUAL);
        sel = warp_find_chunk(a.nchf, ff_mul_f(total, u), chunk_mass, &rem);
        ok = sel >= 0;
      }
    }
    if (lane == 0) {
      sm.mode = ok ? 0 : 1;
      sm.sel = sel;
      sm.rem = rem;
      sm.fcp = cp;
      sm.fe2 = e2;
      a.ws.sps_ticket_a[b] = 0u;
    }
  }
  __syncthreads();
  int tok = -1;
  if (sm.mode == 0) {
    const int64_t sc0 = static_cast<int64_t>(sm.sel) * G::kCH;
    const int len = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - sc0));
    tok = fast_select_in_chunk<T, VEC>(prow, qrow, sc0, len, sm.rem, sm.fe2, fp, fq, sm.fcp, sm);
  }
  if (tid == 0) {
    if (tok >= 0) a.tokens_out[static_cast<size_t>(b) * (a.K + 1) + jr] = tok;
    else queue_push(a.ws.sps_ff_n, a.ws.sps_ff, a.B, b);
  }
}

// The float-float pass over the prompts the fp32 pass left, shifts from the
// row kernel: CTA (c, k) takes chunk c of queue entries k, k + gridDim.y, ...
// Its own close calls go on to the retry pass, which clears this queue.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) sps_ff_kernel(const SpsArgs a) {
  __shared__ SpsSmem sm;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the fp32 pass's queue
  // the retry pass may launch once every CTA has started; it waits for this
  // grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const unsigned n = min(__ldcg(a.ws.sps_ff_n), static_cast<unsigned>(a.B));
  if (n <= blockIdx.y) return;
  sps_stage_tables(sm);
  for (unsigned k = blockIdx.y; k < n; k += gridDim.y) {
    const int b = __ldcg(a.ws.sps_ff + k);
    // an entry left by a call that failed between its launches is skipped
    if (b < 0 || b >= a.B) continue;
    const int jr = a.ws.sps_rej[b];
    if (jr < 0 || jr >= a.K) continue;
    const RowResult *res = a.ws.results + static_cast<size_t>(b) * (2 * a.K + 1);
    const float4 rp = __ldcg(reinterpret_cast<const float4 *>(res + jr));
    const float4 rq = __ldcg(reinterpret_cast<const float4 *>(res + a.K + 1 + jr));
    onepass_chunk<T, VEC>(a, b, jr, blockIdx.x, ff{rp.x, rp.z}, ff{rq.x, rq.z}, false,
                          a.ws.sps_ticket_a, sm);
  }
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kSpsRetryCtas = 8;  // queue entries the retry grid takes at once
constexpr int kSpsFfCtas = 64;    // queue entries the float-float grid takes at once

template <typename T, bool VEC>
static void launch_sps_kernels(const SpsArgs &a, bool topp, dim3 g, cudaStream_t stream) {
  // every kernel with programmatic dependent launch: each waits for the grid
  // before it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (topp) {
    cfg.gridDim = g;
    if (cudaLaunchKernelEx(&cfg, sps_stats_kernel<T, VEC>, a) != cudaSuccess) return;
    (void)cudaLaunchKernelEx(&cfg, sps_residual_kernel<T, VEC>, a);
  } else {
    cfg.gridDim = dim3(a.nchf, g.y);
    if (cudaLaunchKernelEx(&cfg, sps_fast_kernel<T, VEC>, a) != cudaSuccess) return;
    cfg.gridDim = dim3(g.x, min(static_cast<int>(g.y), kSpsFfCtas));
    if (cudaLaunchKernelEx(&cfg, sps_ff_kernel<T, VEC>, a) != cudaSuccess) return;
    cfg.gridDim = dim3(g.x, min(static_cast<int>(g.y), kSpsRetryCtas));
    (void)cudaLaunchKernelEx(&cfg, sps_retry_kernel<T, VEC>, a);
  }
}

cudaError_t launch_sps_residual(const Shape &s, const void *target, const void *draft,
                                int32_t *tokens_out, const Workspace &ws, cudaStream_t stream) {
  SpsArgs a{};
  a.target = static_cast<const char *>(target);
  a.draft = static_cast<const char *>(draft);
  a.B = s.B; a.K = s.K; a.V = s.V;
  a.nch = sps_chunks_per_row(s.dtype, s.V);
  a.nchf = sps_fast_chunks_per_row(s.dtype, s.V);
  a.tscale = s.tscale;
  a.topp = s.top_p < 1.f;
  a.seed = s.seed; a.step = s.step;
  a.tokens_out = tokens_out;
  a.ws = ws;
  const int esz = s.dtype == SMC_BF16 ? 2 : 4;
  const bool vec = aligned16(target) && aligned16(draft) && (static_cast<long long>(s.V) * esz) % 16 == 0;
  const dim3 g(a.nch, s.B);
  if (s.dtype == SMC_BF16) {
    if (vec) launch_sps_kernels<bf16_tag, true>(a, a.topp != 0, g, stream);
    else launch_sps_kernels<bf16_tag, false>(a, a.topp != 0, g, stream);
  } else {
    if (vec) launch_sps_kernels<float, true>(a, a.topp != 0, g, stream);
    else launch_sps_kernels<float, false>(a, a.topp != 0, g, stream);
  }
  return cudaGetLastError();
}

}  // namespace smcsd
