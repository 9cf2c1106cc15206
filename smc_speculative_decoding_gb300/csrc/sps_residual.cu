// Speculative-sampling residual draw for sm_103a ("Accelerating Large
// Language Model Decoding with Speculative Sampling", section 4.2 "Modified
// Rejection Sampling"): at the first rejected position j, one token is drawn
// from max(0, p_j - q_j) normalised, by inverse CDF in vocabulary order.
//
// Runs after the row kernel in SpS mode, which wrote the first rejected
// position of every prompt (or -1).  Two launches over (chunk, prompt):
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

struct SpsArgs {
  const char *target, *draft;
  int B, K, V, nch;
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

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) sps_stats_kernel(const SpsArgs a) {
  using G = SpsGeom<T>;
  __shared__ float s_red[2 * kWarps];
  __shared__ float2 s_ff[kWarps];
  __shared__ float2 s_tab[64];
  __shared__ float s_th[64], s_tl[64];
  __shared__ int s_last;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int jr = a.ws.sps_rej[b];
  if (jr < 0) return;
  stage_exp2_table(s_tab);
  stage_exp2_split(s_th, s_tl);
  const int64_t c0 = static_cast<int64_t>(c) * G::kCH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - c0));
  const char *rows[2] = {
      a.target + (static_cast<size_t>(b) * (a.K + 1) + jr) * static_cast<size_t>(a.V) * G::kESZ,
      a.draft + (static_cast<size_t>(b) * a.K + jr) * static_cast<size_t>(a.V) * G::kESZ};
  float thr[2];
  sps_thresholds(a, b, jr, &thr[0], &thr[1]);
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
  const float mcp = block_max(m[0], s_red);
  const float mcq = block_max(m[1], s_red);  // (the table is staged: block_max has barriers)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float mc = r == 0 ? mcp : mcq;
    const ff S = block_ff_sum(chunk_weight_sum<T, G::kEPT>(x[r], mc, a.tscale, s_th, s_tl, s_tab),
                              s_ff);
    if (tid == 0) a.ws.sps_part_pq[(static_cast<size_t>(b) * a.nch + c) * 2 + r] = make_float4(mc, S.hi, S.lo, 0.f);
  }
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(&a.ws.sps_ticket_a[b], 1u) == static_cast<unsigned>(a.nch - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < 32) {
    const int lane = tid;
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
          if (q.x > kNegInf) val = ff_mul(ff{q.y, q.z}, ff_norm(weight_term(q.x, M, a.tscale, s_tab)));
        }
        tot = ff_add(tot, warp_ff_sum(val));
      }
      // log of the (kept) mass of exp(s l): s M (exact, as a pair) + log(total)
      const ff l = (M > kNegInf && tot.hi > 0.f)
                       ? ff_add(two_prod(a.tscale, M), ff_log(ff_norm(tot), s_tab))
                       : ff{kNegInf, 0.f};
      lse[r][0] = l.hi;
      lse[r][1] = l.lo;
    }
    if (lane == 0) {
      a.ws.sps_stats[b] = make_float4(lse[0][0], lse[0][1], lse[1][0], lse[1][1]);
      a.ws.sps_ticket_a[b] = 0u;
    }
  }
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

template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads) sps_residual_kernel(const SpsArgs a) {
  using G = SpsGeom<T>;
  using Tr = LogitTraits<T>;
  __shared__ float2 s_ff[kWarps];
  __shared__ float2 s_tab[64];
  __shared__ float s_th[64], s_tl[64];
  __shared__ int s_int[2 * kWarps];
  __shared__ int s_last;
  __shared__ int s_sel;
  __shared__ int s_mode;
  __shared__ float s_sel_m;
  __shared__ ff s_rem;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  const int jr = a.ws.sps_rej[b];
  if (jr < 0) return;
  stage_exp2_table(s_tab);
  stage_exp2_split(s_th, s_tl);
  const float4 st = a.ws.sps_stats[b];
  const ff lp{st.x, st.y}, lq{st.z, st.w};
  float thr_p, thr_q;
  sps_thresholds(a, b, jr, &thr_p, &thr_q);
  const int64_t c0 = static_cast<int64_t>(c) * G::kCH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - c0));
  const char *prow = a.target + (static_cast<size_t>(b) * (a.K + 1) + jr) * static_cast<size_t>(a.V) * G::kESZ;
  const char *qrow = a.draft + (static_cast<size_t>(b) * a.K + jr) * static_cast<size_t>(a.V) * G::kESZ;
  float xp[G::kEPT], xq[G::kEPT];
  load_chunk<T, VEC, kSpsNV>(prow + c0 * G::kESZ, n_valid, xp);
  load_chunk<T, VEC, kSpsNV>(qrow + c0 * G::kESZ, n_valid, xq);
  __syncthreads();  // tables staged
  // p and q two logits at a time on the packed pipes, and the residual
  // max(0, p - q) of each in float-float as residual_of takes it: logits
  // outside a nucleus are set to -inf first (they then weigh about e^-59
  // instead of 0, far below what can move a draw); the running sums start at
  // 2, above any residual (<= 1), so the fast two-sum is exact at every
  // addition
  ShiftedExp ep, eq;
  ep.init(a.tscale, lp);
  eq.init(a.tscale, lq);
  const bool live = lp.hi > kNegInf && lq.hi > kNegInf;
  ff R0{0.f, 0.f}, R1{0.f, 0.f};
  if (live) {
    unsigned long long acc = f2dup(2.f), alo = 0ull;
#pragma unroll
    for (int e = 0; e < G::kEPT; e += 2) {
      unsigned long long PH, PL, QH, QL;
      ep.eval(xp[e] >= thr_p ? xp[e] : kNegInf, xp[e + 1] >= thr_p ? xp[e + 1] : kNegInf, s_th,
              s_tl, &PH, &PL);
      eq.eval(xq[e] >= thr_q ? xq[e] : kNegInf, xq[e + 1] >= thr_q ? xq[e + 1] : kNegInf, s_th,
              s_tl, &QH, &QL);
      // d = p - q: two-sum of the heads, the tails after, then normalised
      const unsigned long long DH = sub2(PH, QH);
      const unsigned long long BB = sub2(DH, PH);
      const unsigned long long DE = sub2(sub2(PH, sub2(DH, BB)), add2(QH, BB));
      const unsigned long long DL = add2(DE, sub2(PL, QL));
      const unsigned long long NH = add2(DH, DL);
      const unsigned long long NL = sub2(DL, sub2(NH, DH));
      float h0, h1, l0, l1;
      f2unpack(NH, h0, h1);
      f2unpack(NL, l0, l1);
      const unsigned long long RH = f2pack(h0 > 0.f ? h0 : 0.f, h1 > 0.f ? h1 : 0.f);
      const unsigned long long RL = f2pack(h0 > 0.f ? l0 : 0.f, h1 > 0.f ? l1 : 0.f);
      const unsigned long long S2 = add2(acc, RH);
      alo = add2(alo, add2(sub2(RH, sub2(S2, acc)), RL));
      acc = S2;
    }
    float a0, a1, o0, o1;
    f2unpack(acc, a0, a1);
    f2unpack(alo, o0, o1);
    R0 = two_sum(a0, -2.f);
    R1 = two_sum(a1, -2.f);
    R0.lo += o0;
    R1.lo += o1;
  } else {
#pragma unroll
    for (int e = 0; e < G::kEPT; ++e) {
      const ff d = residual_of(xp[e], xq[e], a.tscale, lp, lq, thr_p, thr_q, s_tab);
      if (d.hi > 0.f) {
        if (e & 1) ff_accum(R1, d);
        else ff_accum(R0, d);
      }
    }
  }
  const ff R = block_ff_sum(ff_add(ff_norm(R0), ff_norm(R1)), s_ff);
  if (tid == 0) {
    a.ws.sps_part_r[static_cast<size_t>(b) * a.nch + c] = make_float2(R.hi, R.lo);
    __threadfence();
    s_last = atomicAdd(&a.ws.sps_ticket_b[b], 1u) == static_cast<unsigned>(a.nch - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < 32) {
    const int lane = tid;
    const float2 *pr = a.ws.sps_part_r + static_cast<size_t>(b) * a.nch;
    ff total{0.f, 0.f};
    for (int c0w = 0; c0w < a.nch; c0w += 32) {
      const int cc = c0w + lane;
      ff val{0.f, 0.f};
      if (cc < a.nch) val = ff{__ldcg(&pr[cc].x), __ldcg(&pr[cc].y)};
      total = ff_add(total, warp_ff_sum(val));
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
          *f = ff_norm(weight_term(q.x, M, a.tscale, s_tab));
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
      s_sel = sel;
      s_mode = mode;
      s_sel_m = sel_m;
      s_rem = rem;
      a.ws.sps_ticket_b[b] = 0u;
    }
  }
  __syncthreads();
  const int sel = s_sel;
  int tok = -1;
  if (sel >= 0) {
    const int64_t sc0 = static_cast<int64_t>(sel) * G::kCH;
    const int len = static_cast<int>(min(static_cast<int64_t>(G::kCH), a.V - sc0));
    if (s_mode == 0) {
      tok = block_select_in_chunk(
          sc0, len, s_rem,
          [&](int64_t i) {
            return residual_of(Tr::scalar(prow, i), Tr::scalar(qrow, i), a.tscale, lp, lq, thr_p,
                               thr_q, s_tab);
          },
          s_ff, s_int);
    } else {
      const float cm = s_sel_m;
      tok = block_select_in_chunk(
          sc0, len, s_rem,
          [&](int64_t i) {
            const float x = Tr::scalar(prow, i);
            return x >= thr_p ? weight_term(x, cm, a.tscale, s_tab) : ff{0.f, 0.f};
          },
          s_ff, s_int);
    }
  }
  if (tid == 0) a.tokens_out[static_cast<size_t>(b) * (a.K + 1) + jr] = tok;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_sps_residual(const Shape &s, const void *target, const void *draft,
                                int32_t *tokens_out, const Workspace &ws, cudaStream_t stream) {
  SpsArgs a{};
  a.target = static_cast<const char *>(target);
  a.draft = static_cast<const char *>(draft);
  a.B = s.B; a.K = s.K; a.V = s.V;
  a.nch = sps_chunks_per_row(s.dtype, s.V);
  a.tscale = s.tscale;
  a.topp = s.top_p < 1.f;
  a.seed = s.seed; a.step = s.step;
  a.tokens_out = tokens_out;
  a.ws = ws;
  const int esz = s.dtype == SMC_BF16 ? 2 : 4;
  const bool vec = aligned16(target) && aligned16(draft) && (static_cast<long long>(s.V) * esz) % 16 == 0;
  dim3 g(a.nch, s.B), blk(kThreads);
  if (s.dtype == SMC_BF16) {
    if (vec) {
      sps_stats_kernel<bf16_tag, true><<<g, blk, 0, stream>>>(a);
      sps_residual_kernel<bf16_tag, true><<<g, blk, 0, stream>>>(a);
    } else {
      sps_stats_kernel<bf16_tag, false><<<g, blk, 0, stream>>>(a);
      sps_residual_kernel<bf16_tag, false><<<g, blk, 0, stream>>>(a);
    }
  } else {
    if (vec) {
      sps_stats_kernel<float, true><<<g, blk, 0, stream>>>(a);
      sps_residual_kernel<float, true><<<g, blk, 0, stream>>>(a);
    } else {
      sps_stats_kernel<float, false><<<g, blk, 0, stream>>>(a);
      sps_residual_kernel<float, false><<<g, blk, 0, stream>>>(a);
    }
  }
  return cudaGetLastError();
}

}  // namespace smcsd
