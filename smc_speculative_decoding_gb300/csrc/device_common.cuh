// Device building blocks shared by the SMC-SD kernels: Philox4x32-10,
// float-float arithmetic, the accurate exp2 used by sampling sums, vector
// loads of logit chunks, and block-wide reductions and scans.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "exp2_table.cuh"

namespace smcsd {

constexpr int kThreads = 256;            // threads per CTA of every kernel here
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): word 0 of one block.
// Counter (step, stream, position, purpose), key (seed lo, seed hi).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += kW0; k1 += kW1; }
    const uint32_t hi0 = __umulhi(kM0, c0), lo0 = kM0 * c0;
    const uint32_t hi1 = __umulhi(kM1, c2), lo1 = kM1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return c0;
}

// u in [0, 1) on the 2^-24 lattice; exact in fp32 and fp64.
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t step, uint32_t stream,
                                                uint32_t position, uint32_t purpose) {
  const uint32_t x = philox_word0(step, stream, position, purpose,
                                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  return static_cast<float>(x >> 8) * 0x1p-24f;
}

// ---------------------------------------------------------------------------
// float-float arithmetic (Knuth two-sum, Dekker fast-two-sum, FMA two-product).
// Relies on IEEE fp32 with no reassociation (the build does not use fast-math).
// ---------------------------------------------------------------------------
struct ff { float hi, lo; };

__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}
__device__ __forceinline__ ff fast_two_sum(float a, float b) {  // needs |a| >= |b| or a == 0
  const float s = a + b;
  return {s, b - (s - a)};
}
__device__ __forceinline__ ff two_prod(float a, float b) {
  const float p = a * b;
  return {p, fmaf(a, b, -p)};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  s.lo += a.lo + b.lo;
  return fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff{-b.hi, -b.lo}); }
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  ff p = two_prod(a.hi, b.hi);
  p.lo += a.hi * b.lo + a.lo * b.hi;
  return fast_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  ff p = two_prod(a.hi, b);
  p.lo = fmaf(a.lo, b, p.lo);
  return fast_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q1 = a.hi / b.hi;
  const ff r = ff_sub(a, ff_mul_f(b, q1));
  const float q2 = r.hi / b.hi;
  return fast_two_sum(q1, q2);
}
// a > b, exact on the represented values (both normalised).
__device__ __forceinline__ bool ff_gt(ff a, ff b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

// ---------------------------------------------------------------------------
// Accurate 2^y for y = yh + yl <= ~0, as an unnormalised float pair with
// relative error about 3e-10: y = n + j/64 + r, |r| <= 1/128;
// 2^(j/64) from a float-float table, 2^r - 1 from its Taylor polynomial.
// `tab` points at the table staged in shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ ff accurate_exp2(float yh, float yl, const float2 *tab) {
  // below 2^-120 the weight is taken as 0 (and -inf or NaN inputs give 0;
  // NaN rows are reported separately)
  const bool live = yh > -120.f;
  const float yc = fmaxf(yh, -120.f);
  // round yc*64 to an integer ki with the 1.5*2^23 shift: the low mantissa
  // bits of t then hold ki, a multiple-of-64 offset from the shift's pattern
  constexpr float kShift = 12582912.f;               // 1.5 * 2^23
  const float t = fmaf(yc, 64.f, kShift);
  const float k = t - kShift;                        // ki as a float, exact
  const int bits = __float_as_int(t) - 0x4B400000;   // ki
  const float rh = fmaf(k, -0.015625f, yc);          // exact: y - ki/64
  const float r = rh + yl;
  const int j = bits & 63;
  const int n = bits >> 6;                           // floor(ki / 64)
  float q = fmaf(r, kC4, kC3);
  q = fmaf(r, q, kC2);
  q = fmaf(r, q, kC1Lo);
  const float p = fmaf(r, kC1Hi, r * q);             // 2^r - 1
  const float2 tv = tab[j];
  const float lo = fmaf(tv.x, p, fmaf(tv.y, p, tv.y));
  const float sc = __int_as_float((n + 127) << 23);  // 2^n, n >= -120
  return live ? ff{tv.x * sc, lo * sc} : ff{0.f, 0.f};
}

// 2^(log2(e) * d) for d given as a float pair (d, dl): exp(d + dl).
__device__ __forceinline__ ff accurate_exp(float d, float dl, const float2 *tab) {
  const float yh = d * kLog2eHi;
  const float yl = fmaf(d, kLog2eHi, -yh) + fmaf(d, kLog2eLo, dl * kLog2eHi);
  return accurate_exp2(yh, yl, tab);
}

// ff_add, ff_sub and ff_mul_f that pass an infinite or NaN operand through
// as a plain float (the float-float forms would turn an infinite head into
// NaN): -inf stays -inf, so a weight of 0 stays 0.
__device__ __forceinline__ ff ff_add_x(ff a, ff b) {
  return (isfinite(a.hi) && isfinite(b.hi)) ? ff_add(a, b) : ff{a.hi + b.hi, 0.f};
}
__device__ __forceinline__ ff ff_sub_x(ff a, ff b) { return ff_add_x(a, ff{-b.hi, -b.lo}); }
__device__ __forceinline__ ff ff_mul_fx(ff a, float f) {
  return isfinite(a.hi) ? ff_mul_f(a, f) : ff{a.hi * f, 0.f};
}

// log(x) of a float-float x >= 2^-100 (normalised), as a float-float value
// about 1e-9 from the exact logarithm: y0 = logf(x.hi), then one Newton step
// with the accurate exponential, log x = y0 + log(x e^-y0), where x e^-y0 =
// 1 + r with |r| ~ 1e-7, so log(1 + r) = r - r^2/2 to far below the exp's
// own 3e-10.
__device__ __forceinline__ ff ff_log(ff x, const float2 *tab) {
  const float y0 = logf(x.hi);
  const ff e = accurate_exp(-y0, 0.f, tab);
  const ff p = ff_mul(x, fast_two_sum(e.hi, e.lo));  // x e^-y0, close to 1
  const float r = (p.hi - 1.f) + p.lo;                // p.hi - 1 is exact (Sterbenz)
  return fast_two_sum(y0, fmaf(-0.5f * r, r, r));
}
__device__ __forceinline__ ff ff_log_f(float x, const float2 *tab) {
  return ff_log(ff{x, 0.f}, tab);
}

// A row's log-sum-exp ts*M + log(S) as a float-float value, from its largest
// logit M and S = sum exp(ts (l - M)) (S >= 1 when M is finite).  Rows with a
// non-finite M or S (errors reported elsewhere) get the plain fp32 value.
__device__ __forceinline__ ff row_lse(float ts, float M, float S, const float2 *tab) {
  if (!(isfinite(M) && S >= 1.f && S < __int_as_float(0x7f800000))) {
    return ff{ts * M + logf(S), 0.f};
  }
  return ff_add(two_prod(ts, M), ff_log_f(S, tab));
}

// Accumulate an unnormalised pair into a running float-float sum.
__device__ __forceinline__ void ff_accum(ff &acc, ff t) {
  ff s = two_sum(acc.hi, t.hi);
  acc.hi = s.hi;
  acc.lo += s.lo + t.lo;
}
__device__ __forceinline__ ff ff_norm(ff a) { return fast_two_sum(a.hi, a.lo); }

// round(f) to the nearest integer, ties away from zero, for |f| < 2^62
// (larger magnitudes, infinities and NaN are not handled), decoded from the
// float's sign, exponent and significand on the integer pipes: this GPU runs
// 64-bit float-to-integer conversions on its narrow fp64 pipe.
__device__ __forceinline__ long long float_to_ll_rn(float f) {
  const uint32_t b = __float_as_uint(f);
  const int e = min(static_cast<int>((b >> 23) & 0xffu) - 150, 38);  // |f| = m 2^e
  const uint32_t m = (b & 0x7fffffu) | 0x800000u;
  unsigned long long mag;
  if (e >= 0) {
    mag = static_cast<unsigned long long>(m) << e;
  } else {
    const int s = -e;  // the last kept bit is bit s of m; add half of it
    mag = s > 24 ? 0ull : static_cast<unsigned long long>((m + (1u << (s - 1))) >> s);
  }
  const long long v = static_cast<long long>(mag);
  return (b >> 31) ? -v : v;
}

__device__ __forceinline__ void stage_exp2_table(float2 *s_tab) {
  if (threadIdx.x < 64) s_tab[threadIdx.x] = kExp2Tab[threadIdx.x];
}

// ---------------------------------------------------------------------------
// Fast-path exp2 (MUFU) and logit widening.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed pairs of fp32 (one 64-bit register pair) for the sm_100+ f32x2 ops.
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2dup(float a) { return f2pack(a, a); }
// Lane-wise max of two packed bfloat16 pairs that propagates NaN.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
// Lane-wise max of two packed bfloat16 pairs (NaN yields the other operand).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 16-byte streaming load that bypasses L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <typename T> struct LogitTraits;
template <> struct LogitTraits<float> {
  static constexpr int kPerVec = 4;               // logits per 16-byte vector
  __device__ __forceinline__ static float at(const uint4 &v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  __device__ __forceinline__ static float scalar(const void *row, int64_t i) {
    return __ldg(static_cast<const float *>(row) + i);
  }
};
struct bf16_tag {};
template <> struct LogitTraits<bf16_tag> {
  static constexpr int kPerVec = 8;
  __device__ __forceinline__ static float at(const uint4 &v, int e) {
    const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
  }
  __device__ __forceinline__ static float scalar(const void *row, int64_t i) {
    const uint16_t b = __ldg(static_cast<const unsigned short *>(row) + i);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
};

// ---------------------------------------------------------------------------
// Block-wide reductions and scans over kThreads threads.  `scratch` is shared
// memory of at least 2*kWarps words.  All threads must call them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float block_max(float v, float *scratch) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = lane < kWarps ? scratch[lane] : kNegInf;
  return warp_max(v);
}

__device__ __forceinline__ ff warp_ff_sum(ff v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ff w{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    v = ff_add(v, w);
  }
  return v;
}
__device__ __forceinline__ ff block_ff_sum(ff v, float2 *scratch) {
  v = warp_ff_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = make_float2(v.hi, v.lo);
  __syncthreads();
  ff w = lane < kWarps ? ff{scratch[lane].x, scratch[lane].y} : ff{0.f, 0.f};
  return warp_ff_sum(w);
}

// Inclusive float-float scan across the block in thread order.
__device__ __forceinline__ ff block_ff_scan(ff v, float2 *scratch, ff *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    ff w{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
    if (lane >= o) v = ff_add(w, v);
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = make_float2(v.hi, v.lo);
  __syncthreads();
  ff base{0.f, 0.f};
  ff all{0.f, 0.f};
  for (int w = 0; w < kWarps; ++w) {
    const ff s{scratch[w].x, scratch[w].y};
    if (w < warp) base = ff_add(base, s);
    all = ff_add(all, s);
  }
  *total = all;
  return ff_add(base, v);
}

// Exclusive scan of ints in thread order; *total gets the sum.
__device__ __forceinline__ int block_excl_scan_i(int v, int *scratch, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int w = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += w;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  int base = 0, all = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) base += scratch[w];
    all += scratch[w];
  }
  *total = all;
  return base + x - v;
}
// Exclusive CTA-wide prefix sum of a 64-bit value; *total gets the sum.
// scratch: kWarps words of shared memory.  All threads must call it.
__device__ __forceinline__ long long block_excl_scan_ll(long long v, long long *scratch,
                                                        long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  long long base = 0, all = 0;
  for (int w = 0; w < kWarps; ++w) {
    const long long s = scratch[w];
    if (w < warp) base += s;
    all += s;
  }
  *total = all;
  return base + x - v;
}

__device__ __forceinline__ int block_min_i(int v, int *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = lane < kWarps ? scratch[lane] : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}


// ---------------------------------------------------------------------------
// mbarrier and bulk-copy (TMA, non-tensor) primitives, sm_90+ PTX.
// Every wait is bounded: it gives up after `limit` polls and returns false.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// try_wait suspends the thread until the phase completes or about
// `suspend_ns` nanoseconds pass, so a waiting warp issues few instructions.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity,
                                              uint32_t suspend_ns = 20000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  return false;
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to shared memory; completion is signalled on `bar` as tx bytes.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// A hint to bring [p, p + bytes) into L2: the 16-byte-aligned part of the
// range, by one bulk prefetch (no data moves to the SM; nothing to wait for).
__device__ __forceinline__ void prefetch_l2(const void *p, size_t bytes) {
  const unsigned long long a0 = reinterpret_cast<unsigned long long>(p);
  const unsigned long long s = (a0 + 15ull) & ~15ull, e = (a0 + bytes) & ~15ull;
  if (e > s) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s),
                 "r"(static_cast<unsigned>(e - s))
                 : "memory");
  }
}

// 64-bit stores and loads at gpu scope.  An aligned 64-bit access is single-
// copy atomic, so a value and its tag written in one such store are seen
// together or not at all, with no fence.
__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// The GPU's global timer, in nanoseconds.
__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A named CTA barrier (id 1..15) over `n` threads, a multiple of 32: only
// the warps that take part wait for one another.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Counters that one kernel's CTAs raise and a concurrent kernel's CTAs wait
// on (gpu scope).  add_release publishes the calling thread's earlier writes
// with the increment; a thread whose acquire load reads the count sees them.
__device__ __forceinline__ void add_release_gpu(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// atomicAdd on a shared counter with acquire-release semantics at CTA scope:
// the calling thread's earlier writes (global ones too) happen before any
// later add's observer, and this add sees what earlier adders published.
__device__ __forceinline__ unsigned atom_add_acq_rel_cta(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(static_cast<unsigned>(__cvta_generic_to_shared(p))), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits until *p reaches `target`: at most `limit` polls, backing off to
// about a microsecond between them.  False when it gave up.
__device__ __forceinline__ bool wait_count(const unsigned *p, unsigned target, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ld_acquire_gpu(p) >= target) return true;
    __nanosleep(i < 64 ? 32 : 1024);
  }
  return ld_acquire_gpu(p) >= target;
}

// Asynchronous 4-byte global-to-shared copy (cp.async): issued without
// waiting; cp_async_wait_all waits for the calling thread's copies (a CTA
// barrier after it makes them visible to the other threads).
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Device status word: OR in error bits (never traps, never waits).
__device__ __forceinline__ void raise_status(unsigned *status, unsigned bits) {
  atomicOr(status, bits);
}

}  // namespace smcsd
