// Row-level device helpers shared by the step kernel and the SpS residual
// kernels: chunk streaming, sampling-weight terms, and the two stages of an
// inverse-CDF draw in vocabulary order (which chunk, then which element).
#pragma once

#include "device_common.cuh"

namespace smcsd {

constexpr int kNV = 4;  // 16-byte vectors per thread per chunk

template <typename T> struct ChunkGeom {
  static constexpr int kEPV = LogitTraits<T>::kPerVec;
  static constexpr int kEPT = kNV * kEPV;          // logits per thread
  static constexpr int kCH = kThreads * kEPT;      // logits per chunk
  static constexpr int kESZ = sizeof(T) == 4 ? 4 : 2;
};

// Stream `n_valid` logits of a chunk starting at `chunk_base` into x[]
// (positions past n_valid read as -inf).  VEC: 16-byte streaming loads,
// requires a 16-byte aligned base and n_valid a multiple of the vector width.
// Element x[i*EPV + e] is logit (i*kThreads + tid)*EPV + e of the chunk (VEC)
// or logit i*kThreads + tid (scalar path); order does not matter to callers.
// NV: 16-byte vectors per thread (the chunk holds kThreads * NV of them).
template <typename T, bool VEC, int NV = kNV>
__device__ __forceinline__ void load_chunk(const char *chunk_base, int n_valid,
                                           float (&x)[NV * LogitTraits<T>::kPerVec]) {
  using Tr = LogitTraits<T>;
  constexpr int EPV = ChunkGeom<T>::kEPV;
  const int tid = threadIdx.x;
  if (VEC) {
    const uint4 *base = reinterpret_cast<const uint4 *>(chunk_base);
    uint4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int vi = i * kThreads + tid;
      v[i] = vi * EPV < n_valid ? ld_stream16(base + vi) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const bool ok = (i * kThreads + tid) * EPV < n_valid;
#pragma unroll
      for (int e = 0; e < EPV; ++e) x[i * EPV + e] = ok ? Tr::at(v[i], e) : kNegInf;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NV * EPV; ++i) {
      const int idx = i * kThreads + tid;
      x[i] = idx < n_valid ? Tr::scalar(chunk_base, idx) : kNegInf;
    }
  }
}

// exp(alpha (x - m)) as a float pair, accurate to ~3e-10 relative; -inf -> 0.
// x - m is taken exactly (two_sum): even for bf16 logits the difference is
// not always a float (a logit 2^-16 times smaller than the max, say).
__device__ __forceinline__ ff weight_term(float x, float m, float alpha, const float2 *tab) {
  if (!(x > kNegInf)) return {0.f, 0.f};
  const ff s = two_sum(x, -m);
  ff ad = two_prod(alpha, s.hi);
  ad.lo = fmaf(alpha, s.lo, ad.lo);
  return accurate_exp(ad.hi, ad.lo, tab);
}

// exp(x - L) for a float-float L: exp((x - L.hi) - L.lo).
__device__ __forceinline__ ff prob_term(float x, ff big_l, const float2 *tab) {
  if (!(x > kNegInf)) return {0.f, 0.f};
  const ff s = two_sum(x, -big_l.hi);
  return accurate_exp(s.hi, s.lo - big_l.lo, tab);
}


// ---------------------------------------------------------------------------
// Sampling weights as exact fixed-point integers.
//
// weight_fixed returns exp(alpha (x - ref)) for x <= ref in units of 2^-50,
// rounded to an integer: the exponential is evaluated in float-float (about
// 3e-10 relative) and each of its two float parts is converted exactly, so a
// sum of these integers is order-independent and exact, and a prefix sum can
// be compared with a target without rounding.  Weights below 2^-60 are 0, so
// -inf (and NaN) logits weigh 0.  A sum of 2^12 weights stays below 2^63.
// ---------------------------------------------------------------------------
constexpr int kFixBits = 50;

__device__ __forceinline__ long long weight_fixed(float x, float ref, float alpha,
                                                  const float2 *tab) {
  const ff s = two_sum(x, -ref);              // x - ref exactly
  ff ad = two_prod(alpha, s.hi);
  ad.lo = fmaf(alpha, s.lo, ad.lo);
  const float yh = ad.hi * kLog2eHi;
  const float yl = fmaf(ad.hi, kLog2eHi, -yh) + fmaf(ad.hi, kLog2eLo, ad.lo * kLog2eHi);
  const bool live = yh > -60.f;               // false for -inf and NaN
  const float yc = fmaxf(yh, -60.f);
  constexpr float kShift = 12582912.f;        // 1.5 * 2^23: rounds yc*64 into the low bits
  const float t = fmaf(yc, 64.f, kShift);
  const float k = t - kShift;
  const int ki = __float_as_int(t) - 0x4B400000;
  const float r = fmaf(k, -0.015625f, yc) + yl;  // y - ki/64, |r| <= 1/128 + tiny
  float q = fmaf(r, kC4, kC3);
  q = fmaf(r, q, kC2);
  q = fmaf(r, q, kC1Lo);
  const float p = fmaf(r, kC1Hi, r * q);      // 2^r - 1
  const float2 tv = tab[ki & 63];             // 2^(j/64), float-float
  const float lo = fmaf(tv.x, p, fmaf(tv.y, p, tv.y));
  const float sc = __int_as_float(((ki >> 6) + kFixBits + 127) << 23);  // 2^(n + kFixBits)
  const long long v = float_to_ll_rn(tv.x * sc) + float_to_ll_rn(lo * sc);
  return live ? v : 0ll;
}

// ---------------------------------------------------------------------------
// Sampling-weight sums of a bonus row, two logits at a time on the packed
// fp32x2 pipes (f32x2 add / sub / mul / fma).
//
// add() evaluates exp(alpha (x - ref)) for two logits x <= ref the way
// weight_fixed does (x - ref exactly by two_sum; y = alpha (x - ref) log2(e)
// as a float pair; 2^y = 2^n * 2^(j/64) * 2^r; 2^r - 1 by its Taylor
// polynomial to r^3, whose remainder is below 4e-11 for |r| <= 1/128), about
// 3e-10 relative, and adds them to a float-float running sum per half.
// Logits below lb = ref - 40/alpha (also -inf and NaN) are raised to lb, so
// they weigh e^-40 instead of less; init() reports whether lb is usable
// (false when ref is so large that ref - 40/alpha rounds to ref).  The
// running sums start at 2, above any single weight (<= 1), so fast_two_sum
// is exact at every addition; total() removes the offset.
// ---------------------------------------------------------------------------
struct BonusPairSum {
  unsigned long long acc, lo;        // packed running sums: head, tail
  unsigned long long nref, al, nal;  // -ref, alpha, -alpha in both halves
  float lb;

  // For bf16 logits x and their bf16 maximum ref, with every x at or above
  // ref - span: x - ref fails to be a float only when x and ref differ in
  // magnitude by 2^15 or more.  When |ref| >= span * 2^-13 that can only be a
  // tiny x, so -ref is the larger operand and the fast two-sum is exact.
  // (Logits raised to lb contribute about e^-40 and need no exact difference.)
  __device__ __forceinline__ static bool fast_diff_ok(float ref, float span) {
    return fabsf(ref) >= span * 0x1p-13f;
  }

  __device__ __forceinline__ bool init(float ref, float alpha, float span) {
    acc = f2dup(2.f);
    lo = 0ull;
    nref = f2dup(-ref);
    al = f2dup(alpha);
    nal = f2dup(-alpha);
    lb = ref - span;
    return lb < ref && lb > kNegInf;
  }

  // ALPHA1: the caller guarantees alpha == 1, so a = d needs no product.
  // FAST_DIFF: the caller guarantees fast_diff_ok(): x - ref then needs only
  // the three-operation exact difference (fast two-sum with -ref leading).
  template <bool ALPHA1, bool FAST_DIFF>
  __device__ __forceinline__ void add(float x0, float x1, const float *th, const float *tl) {
    constexpr float kShift = 12582912.f;  // 1.5 * 2^23: rounds 64 y into the low bits
    const unsigned long long X = f2pack(fmaxf(x0, lb), fmaxf(x1, lb));
    // d = x - ref as S + SE, exactly
    const unsigned long long S = add2(X, nref);
    unsigned long long SE;
    if (FAST_DIFF) {
      SE = sub2(X, sub2(S, nref));
    } else {
      const unsigned long long BB = sub2(S, X);
      SE = add2(sub2(X, sub2(S, BB)), sub2(nref, BB));
    }
    // a = alpha d as AH + AL
    unsigned long long AH = S, AL = SE;
    if (!ALPHA1) {
      AH = mul2(al, S);
      const unsigned long long NAE = fma2(nal, S, AH);  // minus the rounding error of AH
      AL = sub2(mul2(al, SE), NAE);
    }
    // y = a log2(e) as YH - NYL
    const unsigned long long YH = mul2(AH, f2dup(kLog2eHi));
    const unsigned long long NYE = fma2(AH, f2dup(-kLog2eHi), YH);
    const unsigned long long NYL =
        fma2(AH, f2dup(-kLog2eLo), fma2(AL, f2dup(-kLog2eHi), NYE));
    // y = ki/64 + r
    const unsigned long long T = fma2(YH, f2dup(64.f), f2dup(kShift));
    const unsigned long long K = sub2(T, f2dup(kShift));
    const unsigned long long R = sub2(fma2(K, f2dup(-0.015625f), YH), NYL);
    unsigned long long Q = fma2(R, f2dup(kC3), f2dup(kC2));
    Q = fma2(R, Q, f2dup(kC1Lo));
    const unsigned long long P = fma2(R, f2dup(kC1Hi), mul2(R, Q));  // 2^r - 1
    float t0, t1;
    f2unpack(T, t0, t1);
    const int k0 = __float_as_int(t0) - 0x4B400000, k1 = __float_as_int(t1) - 0x4B400000;
    const int j0 = k0 & 63, j1 = k1 & 63;
    const unsigned long long TH = f2pack(th[j0], th[j1]), TL = f2pack(tl[j0], tl[j1]);
    const unsigned long long LO = fma2(TH, P, fma2(TL, P, TL));  // 2^(j/64) 2^r - head
    const unsigned long long SC = f2pack(__int_as_float(((k0 >> 6) + 127) << 23),
                                         __int_as_float(((k1 >> 6) + 127) << 23));
    const unsigned long long HT = mul2(TH, SC), LT = mul2(LO, SC);
    const unsigned long long S2 = add2(acc, HT);
    lo = add2(lo, add2(sub2(HT, sub2(S2, acc)), LT));
    acc = S2;
  }

  // This lane's sum of the weights it added, as a float-float value.
  __device__ __forceinline__ ff total() const {
    float a0, a1, l0, l1;
    f2unpack(acc, a0, a1);
    f2unpack(lo, l0, l1);
    ff e = two_sum(a0, -2.f), o = two_sum(a1, -2.f);
    e.lo += l0;
    o.lo += l1;
    return ff_add(ff_norm(e), ff_norm(o));
  }
};

// ---------------------------------------------------------------------------
// exp(s x - L) for two logits at a time on the packed fp32x2 pipes, for a
// scale s > 0 and a float-float L shared by both (a row's log-sum-exp, so
// that the result is a probability): the method of BonusPairSum::add with
// the offset L in place of a float reference.  s x is taken exactly
// (two-product), s x - L.hi exactly (two-sum), L.lo joins the tail, y =
// (s x - L) log2(e) as a float pair, and 2^y = 2^n 2^(j/64) 2^r, about 3e-10
// relative.  The result is a float pair per logit, head and tail packed,
// unnormalised.  Logits with s x - L below -59 (also -inf and NaN) are raised
// to that bound, so they weigh about e^-59 instead of less: masking a logit
// to 0 is the caller's.
// ---------------------------------------------------------------------------
struct ShiftedExp {
  unsigned long long s2, ns2, nlh, nll;
  float lbx;
  bool s1;

  __device__ __forceinline__ void init(float s, ff big_l) {
    s1 = s == 1.f;
    s2 = f2dup(s);
    ns2 = f2dup(-s);
    nlh = f2dup(-big_l.hi);
    nll = f2dup(-big_l.lo);
    lbx = (big_l.hi - 59.f) / s;
  }

  __device__ __forceinline__ void eval(float x0, float x1, const float *th, const float *tl,
                                       unsigned long long *out_h, unsigned long long *out_l) const {
    constexpr float kShift = 12582912.f;  // 1.5 * 2^23: rounds 64 y into the low bits
    const unsigned long long X = f2pack(fmaxf(x0, lbx), fmaxf(x1, lbx));
    // s x as SH - NSE, exactly
    unsigned long long SH = X, NSE = 0ull;
    if (!s1) {
      SH = mul2(s2, X);
      NSE = fma2(ns2, X, SH);
    }
    // d = s x - L as DH + DL: two-sum of SH and -L.hi, then the tails
    const unsigned long long DH = add2(SH, nlh);
    const unsigned long long BB = sub2(DH, SH);
    const unsigned long long DE = add2(sub2(SH, sub2(DH, BB)), sub2(nlh, BB));
    const unsigned long long DL = add2(sub2(DE, NSE), nll);
    // y = d log2(e) as YH - NYL
    const unsigned long long YH = mul2(DH, f2dup(kLog2eHi));
    const unsigned long long NYE = fma2(DH, f2dup(-kLog2eHi), YH);
    const unsigned long long NYL =
        fma2(DH, f2dup(-kLog2eLo), fma2(DL, f2dup(-kLog2eHi), NYE));
    // y = ki/64 + r
    const unsigned long long T = fma2(YH, f2dup(64.f), f2dup(kShift));
    const unsigned long long K = sub2(T, f2dup(kShift));
    const unsigned long long R = sub2(fma2(K, f2dup(-0.015625f), YH), NYL);
    unsigned long long Q = fma2(R, f2dup(kC3), f2dup(kC2));
    Q = fma2(R, Q, f2dup(kC1Lo));
    const unsigned long long P = fma2(R, f2dup(kC1Hi), mul2(R, Q));  // 2^r - 1
    float t0, t1;
    f2unpack(T, t0, t1);
    const int k0 = __float_as_int(t0) - 0x4B400000, k1 = __float_as_int(t1) - 0x4B400000;
    const int j0 = k0 & 63, j1 = k1 & 63;
    const unsigned long long TH = f2pack(th[j0], th[j1]), TL = f2pack(tl[j0], tl[j1]);
    const unsigned long long LO = fma2(TH, P, fma2(TL, P, TL));  // 2^(j/64) 2^r - head
    const unsigned long long SC = f2pack(__int_as_float(((k0 >> 6) + 127) << 23),
                                         __int_as_float(((k1 >> 6) + 127) << 23));
    *out_h = mul2(TH, SC);
    *out_l = mul2(LO, SC);
  }
};

// The 2^(j/64) table as separate head and tail arrays in shared memory.
__device__ __forceinline__ void stage_exp2_split(float *th, float *tl) {
  if (threadIdx.x < 64) {
    const float2 v = kExp2Tab[threadIdx.x];
    th[threadIdx.x] = v.x;
    tl[threadIdx.x] = v.y;
  }
}

__device__ __forceinline__ long long shfl_xor_ll(long long v, int o) {
  return __shfl_xor_sync(0xffffffffu, v, o);
}
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += shfl_xor_ll(v, o);
  return v;
}
__device__ __forceinline__ long long warp_incl_scan_ll(long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long w = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += w;
  }
  return v;
}
// A non-negative float-float value times 2^kFixBits, rounded to an integer.
__device__ __forceinline__ long long ff_to_fixed(ff a) {
  const float sc = __int_as_float((kFixBits + 127) << 23);
  return float_to_ll_rn(a.hi * sc) + float_to_ll_rn(a.lo * sc);
}
// A fixed-point integer (units of 2^-kFixBits) as a float-float value.
__device__ __forceinline__ ff fixed_to_ff(long long v) {
  const float hi = __ll2float_rn(v);
  const long long rest = v - __float2ll_rn(hi);
  const float sc = __int_as_float((127 - kFixBits) << 23);
  return fast_two_sum(hi * sc, __ll2float_rn(rest) * sc);
}

__device__ __forceinline__ ff warp_ff_incl_scan(ff v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ff w{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
    if (lane >= o) v = ff_add(w, v);
  }
  return v;
}

__device__ __forceinline__ float block_sum_f(float v, float *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = lane < kWarps ? scratch[lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ ff shfl_ff(ff v, int src) {
  return ff{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// Stage 1 of an inverse-CDF draw, run by one full warp.  chunk(c, &val, &f)
// gives chunk c's mass `val` in absolute units and the factor `f` from the
// chunk's own units to absolute ones.  Finds the first chunk with positive
// mass whose inclusive prefix exceeds `target` and returns it with the
// remaining target in that chunk's units; if rounding leaves none, returns
// the last chunk with positive mass and its full mass (the draw then takes
// its last element).  Returns -1 when no chunk has mass.
template <typename ChunkFn>
__device__ int warp_find_chunk(int nch, ff target, ChunkFn chunk, ff *rem_local) {
  const int lane = threadIdx.x & 31;
  ff carry{0.f, 0.f};
  int sel = -1, last = -1;
  ff sel_excl{0.f, 0.f}, sel_f{1.f, 0.f}, last_val{0.f, 0.f}, last_f{1.f, 0.f};
  for (int c0w = 0; c0w < nch && sel < 0; c0w += 32) {
    const int c = c0w + lane;
    ff val{0.f, 0.f}, f{1.f, 0.f};
    if (c < nch) chunk(c, &val, &f);
    const ff incl = ff_add(carry, warp_ff_incl_scan(val));
    const ff excl = ff_sub(incl, val);
    const bool pos = c < nch && val.hi > 0.f;
    const unsigned hit = __ballot_sync(0xffffffffu, pos && ff_gt(incl, target));
    const unsigned any = __ballot_sync(0xffffffffu, pos);
    if (hit) {
      const int src = __ffs(hit) - 1;
      sel = c0w + src;
      sel_excl = shfl_ff(excl, src);
      sel_f = shfl_ff(f, src);
    } else if (any) {
      const int src = 31 - __clz(any);
      last = c0w + src;
      last_val = shfl_ff(val, src);
      last_f = shfl_ff(f, src);
    }
    carry = shfl_ff(incl, 31);
  }
  if (sel >= 0) {
    *rem_local = ff_div(ff_sub(target, sel_excl), sel_f);
    return sel;
  }
  *rem_local = last >= 0 ? ff_div(last_val, last_f) : ff{0.f, 0.f};
  return last;
}

// Stage 2, run by the whole CTA: inside chunk [c0, c0+len), the first element
// with a positive weight whose running sum exceeds `target` (in the chunk's
// units); if rounding leaves none, the last positive element.  Thread t scans
// the contiguous segment [t*seg, (t+1)*seg).  term(i) is the weight of
// vocabulary index i.  Returns the vocabulary index, or -1 with no mass.
template <typename TermFn>
__device__ int block_select_in_chunk(int64_t c0, int len, ff target, TermFn term,
                                     float2 *s_ff, int *s_int) {
  const int seg = (len + kThreads - 1) / kThreads;
  const int beg = min(static_cast<int>(threadIdx.x) * seg, len);
  const int end = min(beg + seg, len);
  ff part{0.f, 0.f};
  int last_pos = -1, first_pos = -1;
  for (int e = beg; e < end; ++e) {
    const ff t = term(c0 + e);
    if (t.hi > 0.f) {
      last_pos = e;
      if (first_pos < 0) first_pos = e;
    }
    ff_accum(part, t);
  }
  part = ff_norm(part);
  ff total;
  const ff incl = block_ff_scan(part, s_ff, &total);
  const ff excl = ff_sub(incl, part);
  int cand = 0x7fffffff;
  if (part.hi > 0.f) {
    if (ff_gt(excl, target)) {
      cand = first_pos;                 // target below this segment (rounding)
    } else if (ff_gt(incl, target)) {
      ff run = excl;
      for (int e = beg; e < end; ++e) {
        const ff t = term(c0 + e);
        run = ff_add(run, ff_norm(t));
        if (t.hi > 0.f && ff_gt(run, target)) { cand = e; break; }
      }
      if (cand == 0x7fffffff) cand = last_pos;
    }
  }
  cand = block_min_i(cand, s_int);
  if (cand == 0x7fffffff) cand = -block_min_i(-last_pos, s_int);  // max over threads
  return cand < 0 ? -1 : static_cast<int>(c0 + cand);
}

}  // namespace smcsd
