// Top-p (nucleus) restriction of the step's rows for sm_103a: the kernel
// smc_step_ex runs after the row combine when top_p < 1.
#include <cmath>
#include <type_traits>

#include <cuda_bf16.h>

#include "row_common.cuh"
#include "kernels.h"
#include "smcsd.h"
#include "step_args.cuh"

namespace smcsd {

// Variants for a CTA of NT threads (NT a multiple of 32, at most 1024);
// scratch holds NT / 32 words.  All threads must call them.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Exclusive prefix sum in thread order; *total gets the sum.  scratch holds
// NT / 32 + 1 words: warp 0 scans the warp totals in place.
template <int NT>
__device__ __forceinline__ unsigned long long block_excl_scan_u64(unsigned long long v,
                                                                  unsigned long long *scratch,
                                                                  unsigned long long *total) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long t = lane < W ? scratch[lane] : 0ull;
    unsigned long long c = t;
#pragma unroll
    for (int o = 1; o < W; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) c += y;
    }
    if (lane < W) scratch[lane] = c - t;
    if (lane == W - 1) scratch[W] = c;
  }
  __syncthreads();
  *total = scratch[W];
  return scratch[warp] + x - v;
}
template <int NT>
__device__ __forceinline__ int block_max_int(int v, int *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = lane < NT / 32 ? scratch[lane] : -0x7fffffff - 1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int NT>
__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, int *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = static_cast<int>(v);
  __syncthreads();
  v = lane < NT / 32 ? static_cast<uint32_t>(scratch[lane]) : 0xffffffffu;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
template <int NT>
__device__ __forceinline__ uint32_t block_or_u32(uint32_t v, int *scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = static_cast<int>(v);
  __syncthreads();
  v = lane < NT / 32 ? static_cast<uint32_t>(scratch[lane]) : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
template <int NT>
__device__ __forceinline__ float block_max_nt(float v, float *scratch) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  v = lane < NT / 32 ? scratch[lane] : kNegInf;
  return warp_max(v);
}


// ---------------------------------------------------------------------------
// Top-p (nucleus) restriction of every row, after the row combine: one CTA of
// kToppThreads threads per row, two CTAs per SM (so that the rows being read
// a second time are still in L2).  With pi = softmax(s l), a token is kept
// iff the mass of the tokens strictly more likely than it is below top_p
// (tokens of equal logit go together), so the kept set is {l >= l*} for a
// threshold logit l*, found as an order-preserving 32-bit key v* of l*.
//
// Main path (mass bins).  The first pass streams the row from HBM and puts
// every logit into one of kToppMassBins bins by rn(-8 log2 pi): bins of 1/8
// of a binary order of pi, in decreasing order of the logit (the last bin
// also takes everything below 2^-48).  Within its bin, a logit's mass is
// quantised relative to the bin's top, q = rn(pi 2^(b/8) 2^qb) with pi
// 2^(b/8) in [2^-1/16, 2^1/16] (a relative error below 2^-(qb+1) / 0.95),
// and added as a 32-bit shared atomic to a (bin, lane) cell: each lane owns
// a column of cells, so a warp's adds never share a bank, and qb is chosen
// so that no cell can overflow.  A bin's mass is then (sum q) 2^(26 - b/8)
// in units of 2^-(26 + qb), exact integers throughout, so every sum is
// order-independent.  A scan over the bins finds the threshold bin b*: the
// lowest non-empty bin whose mass above stays below top_p times the total.
// The second pass copies the keys and q of b*'s logits into shared memory,
// and a radix select over those keys, 8 bits at a time from their highest
// differing bit, finds v* inside b*.  A threshold bin with more than
// kToppListCap logits, or rows long enough that qb would fall below 18, take
// the exact path instead.
//
// The first pass is tried first on the likely logits only: those with
// pi >= 2^-16, which fill bins 0 .. kToppHighBins - 1 completely, while a
// 16-byte group without one costs four packed compares.  They are also
// listed in shared memory (each thread its own, up to kToppHighBytes in all),
// and the total is taken as 1
// (the row's log-sum-exp, right to about 1e-7, well inside the 1e-5 near-tie
// margin of the nucleus).  If those bins already hold top_p of the mass, b*
// is among them and the second pass reads the list instead of the row;
// otherwise the full first pass runs, and the second pass reads the row
// again (mostly from L2).
//
// Exact path (radix select over the whole row).  Radix digits of 12 bits
// then 4 (bf16) or 10 + 10 (fp32) over the keys; each pass histograms the
// fixed-point mass round(pi 2^40) (lowest bit set, so a bin holding a finite
// logit reads non-empty) of the logits under the prefix chosen so far, as a
// 32-bit shared atomic on a low word whose carry goes to a high word.
//
// Either way log(kept / total) is added to the row's log-sum-exp; a drafted
// token outside the target's nucleus gets logit -inf (weight 0), one outside
// the draft's nucleus is reported (SMC_DEV_BAD_TOKEN: it could not have
// been drawn).  The bonus row's token is redrawn by inverse CDF over the
// kept tokens in exact integer weights, exp(s (l - ref)) in units of 2^-38
// (about 3e-10 relative; ref = lse / s on the main path, the row's max on
// the exact path): the row is cut into up to kToppEntries runs of 128 G
// consecutive 16-byte groups, each warp sums the kept weights of whole
// runs, a scan over the runs finds the one the draw lands in, and a
// block-wide scan over that run's logits finds the token.
// ---------------------------------------------------------------------------
constexpr int kToppThreads = 512;
constexpr int kToppWarps = kToppThreads / 32;
constexpr int kToppUnroll = 4;       // 16-byte groups in flight per thread
constexpr int kToppMassBins = 384;   // mass bins: pi from 1 down to 2^-48
constexpr int kToppListCap = 2048;   // logits of the threshold bin held in shared memory
constexpr int kToppBins = 4096;      // exact path: bins of the first radix digit (12 bits)
constexpr int kToppEntries = 4096;   // runs of a bonus row summed in the first pass
constexpr int kToppHighBins = 128;   // mass bins of pi >= 2^-16, which the first attempt fills
constexpr int kToppHighBytes = 32768;  // shared memory of the list of those bins' logits
constexpr int kToppQueue = 64;         // 16-byte groups each warp queues for them
constexpr int kToppPrefetchAhead = 2;  // iterations of that pass brought into L2 ahead

// 2^(26 - j/8) rounded to an integer, j = 0..7: the fractional part of a
// mass bin's scale.
__device__ const unsigned kToppFrac[8] = {67108864u, 61539100u, 56431603u, 51748008u,
                                          47453133u, 43514715u, 39903169u, 36591368u};

struct ToppScalars {
  unsigned long long above, kept, base, bin_above, in_above, in_kept;
  long long tok;
  uint32_t prefix;
  int sel, n, nh_over;
  float xlo, xhi;
  uint32_t lo2, hi2;
  int klo, nk;  // direct mode: the 16-bit keys klo .. klo + nk - 1 of bf16 bin b*
  bool last_bin;
};
struct ToppShared {
  uint32_t cell[kToppMassBins * 32];  // mass cells; then the list, or the exact path's buffers
  float2 tab[64];
  uint32_t hq[256], hc[256], hh[256];
  unsigned long long u64s[kToppWarps + 1];
  int ints[kToppWarps];
  float fl[kToppWarps];
  unsigned frac[8];
  ToppScalars s;
};
// Dynamic shared memory: ToppShared, then the first attempt's list of logits
// (kToppHighBytes), then the warps' queues of 16-byte groups.
constexpr size_t kToppHighOff = (sizeof(ToppShared) + 15) / 16 * 16;
constexpr size_t kToppQueueOff = kToppHighOff + kToppHighBytes;
constexpr size_t kToppSmemBytes = kToppQueueOff + sizeof(uint4) * kToppQueue * kToppWarps;
static_assert(sizeof(uint32_t) * kToppMassBins * 32 >= sizeof(unsigned long long) * kToppBins,
              "the exact path's histogram and runs fit in the cells");
static_assert(kToppMassBins * 32 >= 2 * kToppListCap, "the list fits in the cells");

// An order-preserving 32-bit key of a logit; -0 and +0 (equal logits) share
// the key of +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The logit whose key is k (the inverse of order_key, +0 for the key of 0).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Digits of the exact path's radix select for the logit type T.
template <typename T> struct ToppDigits {
  static constexpr int kPasses = sizeof(T) == 4 ? 3 : 2;
  static constexpr int kKeyBits = sizeof(T) == 4 ? 32 : 16;  // significant key bits
  __device__ __forceinline__ static int width(int pass) {
    return pass == 0 ? 12 : (sizeof(T) == 4 ? 10 : 4);
  }
  static constexpr uint32_t kNegInfWord = sizeof(T) == 4 ? 0xff800000u : 0xff80ff80u;
};

// Group g of a row: logits [g E, g E + E) as one 16-byte word (E = 8 bf16 or
// 4 fp32); logits at or past V read as -inf.  VEC: rows are 16-byte aligned
// and V is a multiple of E, so the group is one vector load.  Group and logit
// indices fit in 32 bits (V <= 2^24).
template <typename T, bool VEC>
__device__ __forceinline__ uint4 topp_group(const char *rowp, int g, int V) {
  if (VEC) return ld_stream16(rowp + static_cast<size_t>(g) * 16);
  uint32_t w[4];
  if (sizeof(T) == 4) {
    const float *r = reinterpret_cast<const float *>(rowp);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = g * 4 + e;
      w[e] = i < V ? __float_as_uint(__ldg(r + i)) : 0xff800000u;
    }
  } else {
    const unsigned short *r = reinterpret_cast<const unsigned short *>(rowp);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = g * 8 + 2 * e;
      const uint32_t lo = i < V ? __ldg(r + i) : 0xff80u;
      const uint32_t hi = i + 1 < V ? __ldg(r + i + 1) : 0xff80u;
      w[e] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Calls f(v) for every group of the row (as one 16-byte word), kToppUnroll
// groups in flight per thread; thread t takes the groups g = t mod
// kToppThreads.
template <typename T, bool VEC, typename F>
__device__ __forceinline__ void topp_for_each_group(const char *rowp, int V, F f) {
  constexpr int E = LogitTraits<T>::kPerVec;
  const int ng = (V + E - 1) / E;
  for (int g0 = threadIdx.x; g0 < ng; g0 += kToppThreads * kToppUnroll) {
    uint4 v[kToppUnroll];
#pragma unroll
    for (int u = 0; u < kToppUnroll; ++u) {
      const int g = g0 + u * kToppThreads;
      if (g < ng) v[u] = topp_group<T, VEC>(rowp, g, V);
    }
#pragma unroll
    for (int u = 0; u < kToppUnroll; ++u) {
      if (g0 + u * kToppThreads >= ng) break;
      f(v[u]);
    }
  }
}

// Calls f(x) for every logit of the row.
template <typename T, bool VEC, typename F>
__device__ __forceinline__ void topp_for_each(const char *rowp, int V, F f) {
  topp_for_each_group<T, VEC>(rowp, V, [&](const uint4 &v) {
#pragma unroll
    for (int e = 0; e < LogitTraits<T>::kPerVec; ++e) f(LogitTraits<T>::at(v, e));
  });
}

// The same, two consecutive logits at a time: f(x0, x1).
template <typename T, bool VEC, typename F>
__device__ __forceinline__ void topp_for_each_pair(const char *rowp, int V, F f) {
  topp_for_each_group<T, VEC>(rowp, V, [&](const uint4 &v) {
#pragma unroll
    for (int e = 0; e < LogitTraits<T>::kPerVec; e += 2)
      f(LogitTraits<T>::at(v, e), LogitTraits<T>::at(v, e + 1));
  });
}

// Lane-wise min of two packed bfloat16 pairs (NaN yields the other operand).
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The largest logit of a group (NaN ignored; -inf for an all-NaN group).
template <typename T>
__device__ __forceinline__ float group_max(const uint4 &v) {
  if (sizeof(T) == 4)
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  const uint32_t m = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
  return fmaxf(bf16_lo(m), bf16_hi(m));
}

// Whether any logit of a group lies in [lo, hi].  For bf16 groups lo2 and
// hi2 are the bounds as packed bf16 pairs (rounded outwards) and the test
// takes four packed compares; NaN is in no interval.
template <typename T>
__device__ __forceinline__ bool group_hits(const uint4 &v, float lo, float hi, uint32_t lo2,
                                           uint32_t hi2) {
  if (sizeof(T) == 4) {
    bool any = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = LogitTraits<T>::at(v, e);
      any |= x >= lo && x <= hi;
    }
    return any;
  }
  uint32_t m = 0;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t ge, le;
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ge) : "r"(w[k]), "r"(lo2));
    asm("set.le.u32.bf16x2 %0, %1, %2;" : "=r"(le) : "r"(w[k]), "r"(hi2));
    m |= ge & le;
  }
  return m != 0u;
}

// Whether any logit of a group is at least lo (lo2: lo as a packed bf16 pair,
// for bf16 groups two packed compares per word); NaN is never.
template <typename T>
__device__ __forceinline__ bool group_any_ge(const uint4 &v, float lo, uint32_t lo2) {
  if (sizeof(T) == 4) {
    return __uint_as_float(v.x) >= lo || __uint_as_float(v.y) >= lo ||
           __uint_as_float(v.z) >= lo || __uint_as_float(v.w) >= lo;
  }
  uint32_t m = 0, ge;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ge) : "r"(v.x), "r"(lo2));
  m |= ge;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ge) : "r"(v.y), "r"(lo2));
  m |= ge;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ge) : "r"(v.z), "r"(lo2));
  m |= ge;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(ge) : "r"(v.w), "r"(lo2));
  m |= ge;
  return m != 0u;
}

// The bonus row's draw over the kept logits {x >= thr} (none unless live):
// the first whose inclusive prefix of weight(x) (exact integers) exceeds
// floor(u total); -1 with no weight.  The row is cut into runs of 128 G
// consecutive groups (at most kToppEntries runs); each warp sums whole runs,
// reading kToppUnroll * 32 consecutive groups at a time, and skips any group
// whose largest logit is below thr.
template <typename T, bool VEC, typename WeightF>
__device__ long long topp_bonus_draw(const StepArgs &a, int part, const char *rowp, bool live,
                                     float thr, WeightF weight, ToppShared &sh) {
  using Tr = LogitTraits<T>;
  constexpr int E = Tr::kPerVec;
  constexpr int kRun = 32 * kToppUnroll;  // groups per warp read, and per run when G = 1
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const int ng = (V + E - 1) / E;
  const int G = (ng + kRun * kToppEntries - 1) / (kRun * kToppEntries);
  const int gpr = kRun * G;  // groups per run
  const int ne = (ng + gpr - 1) / gpr;
  const int rpw = (ne + kToppWarps - 1) / kToppWarps;  // runs per warp
  unsigned long long *const s_run = reinterpret_cast<unsigned long long *>(sh.cell);
  __syncthreads();  // the cells' previous contents are no longer read
  if (tid == 0) { sh.s.sel = -1; sh.s.tok = -1; }
  // warp w sums runs [w rpw, (w + 1) rpw); its trip counts are warp-uniform
  for (int r = warp * rpw; r < min(ne, (warp + 1) * rpw); ++r) {
    unsigned long long acc = 0;
    if (live) {
      const int r1 = min(ng, (r + 1) * gpr);
      for (int g0 = r * gpr + lane; g0 < r1; g0 += kRun) {
        uint4 v[kToppUnroll];
#pragma unroll
        for (int u = 0; u < kToppUnroll; ++u) {
          const int g = g0 + 32 * u;
          v[u] = g < r1 ? topp_group<T, VEC>(rowp, g, V)
                        : make_uint4(ToppDigits<T>::kNegInfWord, ToppDigits<T>::kNegInfWord,
                                     ToppDigits<T>::kNegInfWord, ToppDigits<T>::kNegInfWord);
        }
#pragma unroll
        for (int u = 0; u < kToppUnroll; ++u) {
          if (!(group_max<T>(v[u]) >= thr)) continue;
          uint32_t m = 0;
#pragma unroll
          for (int e = 0; e < E; ++e)
            if (Tr::at(v[u], e) >= thr) m |= 1u << e;
          while (m) {
            const int e = __ffs(m) - 1;
            m &= m - 1;
            acc += weight(Tr::at(v[u], e));
          }
        }
      }
    }
    acc = warp_sum_u64(acc);
    if (lane == 0) s_run[r] = acc;
  }
  __syncthreads();
  // the run the draw lands in
  const int c = (ne + kToppThreads - 1) / kToppThreads;
  unsigned long long sum = 0;
  for (int i = 0; i < c; ++i) {
    const int d = tid * c + i;
    if (d < ne) sum += s_run[d];
  }
  unsigned long long total_w;
  const unsigned long long excl_w = block_excl_scan_u64<kToppThreads>(sum, sh.u64s, &total_w);
  const float u = philox_uniform(a.seed, a.step, part, a.bonus_position, a.bonus_purpose);
  const unsigned long long u24 = static_cast<unsigned long long>(u * 16777216.f);
  // floor(total * u), exactly: u = u24 / 2^24
  const unsigned long long target = __umul64hi(total_w, u24 << 40);
  if (total_w > 0) {
    unsigned long long run = excl_w;
    for (int i = 0; i < c; ++i) {
      const int d = tid * c + i;
      if (d >= ne) break;
      const unsigned long long w = s_run[d];
      if (w > 0 && run <= target && target < run + w) { sh.s.sel = d; sh.s.base = run; }
      run += w;
    }
  }
  __syncthreads();
  const int sel = sh.s.sel;
  if (sel >= 0) {
    // the token within the run, by a block-wide scan in index order
    unsigned long long rem = target - sh.s.base;
    const int i0 = sel * gpr * E;
    const int i1 = min(V, i0 + gpr * E);
    for (int base = i0; base < i1; base += kToppThreads) {
      const int i = base + tid;
      unsigned long long w = 0;
      if (i < i1) {
        const float x = Tr::scalar(rowp, i);
        if (x >= thr) w = weight(x);
      }
      unsigned long long tot;
      const unsigned long long ex = block_excl_scan_u64<kToppThreads>(w, sh.u64s, &tot);
      if (w > 0 && ex <= rem && rem < ex + w) sh.s.tok = i;
      if (rem < tot) break;  // the same for every thread
      rem -= tot;
    }
  }
  __syncthreads();
  return sh.s.tok;
}

// log(kept / total) for 64-bit fixed-point masses, in float (each part
// converted through its two 32-bit halves; about 2e-7 absolute); 0 without
// mass.  One thread calls it.
__device__ __forceinline__ float topp_log_ratio(unsigned long long kept, unsigned long long total) {
  if (kept == 0 || total == 0) return 0.f;
  auto to_f = [](unsigned long long v) {
    return fmaf(__uint2float_rn(static_cast<uint32_t>(v >> 32)), 4294967296.f,
                __uint2float_rn(static_cast<uint32_t>(v)));
  };
  return logf(to_f(kept) / to_f(total));
}

// The row of this CTA: the bonus rows (one per particle, the costliest) take
// the first CTAs, so that their extra work is not left for the last wave;
// the other 2K rows of each particle follow in order.
__device__ __forceinline__ int topp_row(const StepArgs &a) {
  const int rpp = 2 * a.K + 1;
  const int parts = a.B * a.N;
  const int b = blockIdx.x;
  if (b < parts) return b * rpp + a.K;
  const int f = b - parts, part = f / (2 * a.K), jj = f - part * (2 * a.K);
  return part * rpp + (jj < a.K ? jj : jj + 1);
}

// Writes a row's nucleus result: the log kept mass on its log-sum-exp(s), for
// a drafted position the check of its token, and the threshold logit thr
// (kept: l >= thr) in the row's otherwise unused token slot, where the
// speculative-sampling residual reads it.
template <typename T, typename KeptF>
__device__ __forceinline__ void topp_finish_fast(const StepArgs &a, int row, int part, int j,
                                                 const char *rowp, float log_z, KeptF kept,
                                                 float thr) {
  using Tr = LogitTraits<T>;
  RowResult r = a.ws.results[row];
  r.tok = __float_as_int(thr);
  const int tok = a.tokens[static_cast<size_t>(part) * a.K + (j < a.K ? j : j - a.K - 1)];
  if (tok >= 0 && tok < a.V && !kept(Tr::scalar(rowp, tok))) {
    if (j < a.K) r.g = kNegInf;                         // outside the target's nucleus
    else raise_status(a.ws.status, SMC_DEV_BAD_TOKEN);  // could not have been drafted
  }
  // a log-sum-exp row's result holds its value as a float pair (lse, lse_alpha)
  const ff lse = ff_add(ff{r.lse, r.lse_alpha}, ff{log_z, 0.f});
  r.lse = lse.hi;
  r.lse_alpha = lse.lo;
  a.ws.results[row] = r;
}

// Main path; returns false (and writes nothing) when the row needs the exact
// path.  The return value is the same in every thread.
template <typename T, bool VEC>
__device__ bool topp_mass_bins(const StepArgs &a, unsigned long long p64, int qb, ToppShared &sh,
                               unsigned char *hlist, uint4 *queue) {
  constexpr int NT = kToppThreads;
  const int tid = threadIdx.x, lane = tid & 31;
  const int row = topp_row(a);
  const int rpp = 2 * a.K + 1;
  const int part = row / rpp, j = row - part * rpp;
  const char *rowp = row_base<T>(a, row);
  const float lse = a.ws.results[row].lse;
  const float l2s = a.tscale * kLog2e, l2lse = lse * kLog2e;
  // 2^(qb - 149), a subnormal: r times it is a subnormal whose bits are
  // rn(r 2^qb) (r 2^qb < 2^23), since fp32 arithmetic here keeps subnormals
  const float qsc = __int_as_float(1 << qb);
  uint32_t *const cell = sh.cell;
  if (tid < 8) sh.frac[tid] = kToppFrac[tid];
  // Logits are first clamped to [x_lo, x_hi]: x_lo puts log2 pi at -47.5 or
  // above (-inf, NaN and the far tail then weigh about 2^-47.5, negligible),
  // x_hi at 1/32 or below.  Every finite logit lies below x_hi, since it is
  // at most lse / s.  For bf16 rows both bounds are bf16 values (x_lo rounded
  // up, x_hi down), so the clamp is exact on the packed pairs.  Then
  // y = log2 pi lies in [-47.5, 1/32], and t = 1.5 2^23 + rn(-8 y) holds the
  // bin, 0..380, in its low bits.  That needs |log2 lse| below 4096, where
  // the rounding of the bounds moves y by at most 5e-4, and finite bounds;
  // other rows (logits in the thousands, or a log-sum-exp that is not finite,
  // which the row pass reports) take the exact path.
  float x_lo = (l2lse - 47.5f) / l2s, x_hi = (l2lse + 0.03125f) / l2s;
  if (sizeof(T) != 4) {
    x_lo = __bfloat162float(__float2bfloat16_ru(x_lo));
    x_hi = __bfloat162float(__float2bfloat16_rd(x_hi));
  }
  if (!(fabsf(l2lse) < 4096.f && fabsf(x_lo) < 3e38f && fabsf(x_hi) < 3e38f)) return false;
  constexpr float kMagicB = 12582912.f;   // 1.5 2^23
  auto mass_bin = [&](float x, float &y, float &t) -> uint32_t {
    y = __fmaf_rn(fminf(fmaxf(x, x_lo), x_hi), l2s, -l2lse);
    t = __fmaf_rn(y, -8.f, kMagicB);
    return static_cast<uint32_t>(__float_as_int(t) - 0x4B400000);
  };
  // pi relative to the top of its bin, rn(pi 2^(b/8) 2^qb), from y and t
  auto quantise = [&](float y, float t) -> uint32_t {
    const float r = fast_exp2(__fmaf_rn(t - kMagicB, 0.125f, y));  // in [2^-1/16, 2^1/16]
    return __float_as_uint(__fmul_rn(r, qsc));
  };

  // ---- pass 1 (HBM): the (bin, lane) cells ----------------------------------
  // First attempt: only the logits with pi >= 2^-16 (x >= x_c) are binned and
  // listed in shared memory; every logit of bins 0 .. kToppHighBins - 1 is
  // among them, and the total is 1 (the row's log-sum-exp).  Most 16-byte
  // groups hold no such logit and cost four packed compares.  If those bins
  // hold less than top_p of the mass, the full pass below bins every logit.
  float x_c = (l2lse - 16.f) / l2s;
  if (sizeof(T) != 4) x_c = __bfloat162float(__float2bfloat16_rd(x_c));
  const uint32_t c16 = __float_as_uint(x_c) >> 16;
  const uint32_t XC2 = c16 | (c16 << 16);
  auto clear_cells = [&](int n_bins) {
    for (int i = tid; i < n_bins * 32; i += NT) cell[i] = 0u;
    if (tid == 0) { sh.s.n = 0; sh.s.nh_over = 0; }
    __syncthreads();
  };
  clear_cells(kToppHighBins + 8);  // the first attempt's logits reach bin 129 at most
  using HighT = typename std::conditional<sizeof(T) == 4, uint32_t, uint16_t>::type;
  constexpr int kHighPerThread = kToppHighBytes / (NT * static_cast<int>(sizeof(HighT)));
  HighT *const hstore = reinterpret_cast<HighT *>(hlist);
  auto high_bits = [](float x) -> HighT {
    return static_cast<HighT>(sizeof(T) == 4 ? __float_as_uint(x) : __float_as_uint(x) >> 16);
  };
  auto high_value = [](HighT u) -> float {
    return __uint_as_float(sizeof(T) == 4 ? static_cast<uint32_t>(u) : static_cast<uint32_t>(u) << 16);
  };
  int n_high = 0;
  {
    // A group that holds such a logit is queued in its warp's shared-memory
    // queue (positions from a ballot; every lane runs every iteration, groups
    // past the row being empty), and 32 queued groups are binned at a time, one
    // per lane, so that the warp's instructions are spent on full groups.
    // Each thread lists the logits it bins, entry k at k NT + tid (bf16 rows
    // keep the 16-bit values); a thread with more than kHighPerThread of them
    // marks the list incomplete.
    const int warp = tid >> 5;
    uint4 *const wq = queue + warp * kToppQueue;
    constexpr int E = LogitTraits<T>::kPerVec;
    const int ng = (a.V + E - 1) / E;
    auto bin_queued = [&](int count) {  // lanes below count take slots 0 .. count - 1
      __syncwarp();
      if (lane < count) {
        const uint4 g = wq[lane];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float x = LogitTraits<T>::at(g, e);
          if (x >= x_c) {
            float y, t;
            const uint32_t b = mass_bin(x, y, t);
            atomicAdd(&cell[(b << 5) + lane], quantise(y, t));
            if (n_high < kHighPerThread) hstore[n_high * NT + tid] = high_bits(x);
            ++n_high;
          }
        }
      }
      __syncwarp();
    };
    int qn = 0;  // groups in the queue, the same in every lane
    // the row's next groups go into L2 kToppPrefetchAhead iterations ahead
    // (one bulk prefetch per iteration, by thread 0), so that the loads below
    // meet L2 latency rather than HBM's
    constexpr int kIt = NT * kToppUnroll;  // groups per iteration
    auto prefetch_groups = [&](int g_from) {
      if (VEC && tid == 0 && g_from < ng) {
        prefetch_l2(rowp + static_cast<size_t>(g_from) * 16,
                    static_cast<size_t>(min(kIt, ng - g_from)) * 16);
      }
    };
    for (int k = 0; k < kToppPrefetchAhead; ++k) prefetch_groups(k * kIt);
    for (int g0 = 0; g0 < ng; g0 += kIt) {
      prefetch_groups(g0 + kToppPrefetchAhead * kIt);
      uint4 v[kToppUnroll];
      bool in[kToppUnroll];
#pragma unroll
      for (int u = 0; u < kToppUnroll; ++u) {
        const int g = g0 + u * NT + tid;
        in[u] = g < ng;
        if (in[u]) v[u] = topp_group<T, VEC>(rowp, g, a.V);
      }
#pragma unroll
      for (int u = 0; u < kToppUnroll; ++u) {
        const bool hit = in[u] && group_any_ge<T>(v[u], x_c, XC2);
        const unsigned bal = __ballot_sync(0xffffffffu, hit);
        if (hit) wq[qn + __popc(bal & ((1u << lane) - 1u))] = v[u];
        qn += __popc(bal);
        if (qn >= 32) {
          bin_queued(32);
          if (lane < qn - 32) wq[lane] = wq[32 + lane];
          qn -= 32;
        }
      }
    }
    bin_queued(qn);
    if (n_high > kHighPerThread) sh.s.nh_over = 1;
  }
  __syncthreads();
  // bin masses in units of 2^-(26 + qb), in decreasing order of the logit;
  // first those of the first attempt's bins, against a total of 1
  auto bin_masses = [&](int n_bins, unsigned long long *Q, unsigned long long *m) {
    *Q = 0;
    *m = 0;
    if (tid < n_bins) {
#pragma unroll 8
      for (int l = 0; l < 32; ++l) *Q += cell[tid * 32 + ((l + lane) & 31)];
      *m = (*Q * sh.frac[tid & 7]) >> (tid >> 3);
    }
  };
  unsigned long long Q, m, total;
  bin_masses(kToppHighBins, &Q, &m);
  unsigned long long above = block_excl_scan_u64<NT>(m, sh.u64s, &total);
  const bool high = total >= __umul64hi(1ull << (26 + qb), p64);
  if (high) {
    total = 1ull << (26 + qb);
  } else {
    // the full pass: every logit, with the same arithmetic as mass_bin and
    // quantise, two logits at a time on the packed fp32x2 pipes (bf16 pairs
    // clamped with packed bf16 min / max)
    clear_cells(kToppMassBins);
    {
      const unsigned long long L2S = f2dup(l2s), NL2LSE = f2dup(-l2lse), M8 = f2dup(-8.f),
                               MB = f2dup(kMagicB), EIGHTH = f2dup(0.125f), QSC = f2dup(qsc);
      // cell index of bin b for this lane, b 32 + lane, from t's bits directly
      // (modulo 2^32: the bias cancels)
      const uint32_t lane_bias = static_cast<uint32_t>(lane) - (0x4B400000u << 5);
      auto add_pair = [&](float x0, float x1) {
        const unsigned long long Y = fma2(f2pack(x0, x1), L2S, NL2LSE);
        const unsigned long long Tt = fma2(Y, M8, MB);
        float t0, t1;
        f2unpack(Tt, t0, t1);
        float e0, e1;
        f2unpack(fma2(sub2(Tt, MB), EIGHTH, Y), e0, e1);
        float q0, q1;
        f2unpack(mul2(f2pack(fast_exp2(e0), fast_exp2(e1)), QSC), q0, q1);
        atomicAdd(&cell[(__float_as_uint(t0) << 5) + lane_bias], __float_as_uint(q0));
        atomicAdd(&cell[(__float_as_uint(t1) << 5) + lane_bias], __float_as_uint(q1));
      };
      if (sizeof(T) == 4) {
        topp_for_each_pair<T, VEC>(rowp, a.V, [&](float x0, float x1) {
          add_pair(fminf(fmaxf(x0, x_lo), x_hi), fminf(fmaxf(x1, x_lo), x_hi));
        });
      } else {
        const uint32_t lo16 = __float_as_uint(x_lo) >> 16, hi16 = __float_as_uint(x_hi) >> 16;
        const uint32_t LO2 = lo16 | (lo16 << 16), HI2 = hi16 | (hi16 << 16);
        topp_for_each_group<T, VEC>(rowp, a.V, [&](const uint4 &v) {
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t c = bmin2(bmax2(w[k], LO2), HI2);  // NaN takes the bound
            add_pair(bf16_lo(c), bf16_hi(c));
          }
        });
      }
    }
    __syncthreads();
    bin_masses(kToppMassBins, &Q, &m);
    above = block_excl_scan_u64<NT>(m, sh.u64s, &total);
  }
  // (in the first attempt only bins 0 .. kToppHighBins - 1 are complete)
  const int n_bins = high ? kToppHighBins : kToppMassBins;
  const unsigned long long limit = __umul64hi(total, p64);  // floor(top_p total)
  const bool cand = tid < n_bins && Q > 0 && above < limit;
  const int bstar = block_max_int<NT>(cand ? tid : -1, sh.ints);
  if (bstar < 0) return false;  // an empty or non-finite row: the exact path reports it
  if (tid == bstar) sh.s.bin_above = above;
  if (tid == 0) {
    // A superset of bin b*'s logits as an interval [x_lo, x_hi]: its members
    // have -8 y within 1/2 of b*, y = log2 pi rounded once (an error below
    // 2^-18 for |y| < 64), so x l2s - l2lse lies within 1/16 + 2^-10 of
    // -b*/8; widened by 1e-5 relative for the rounding of the bounds.  The list below still
    // checks every logit's bin.
    const float bf = static_cast<float>(bstar);
    const float xl = (l2lse - fmaf(bf, 0.125f, 0.0625f + 0x1p-10f)) / l2s;
    const float xh = (l2lse - fmaf(bf, 0.125f, -0.0625f - 0x1p-10f)) / l2s;
    const float slack = 1e-6f * fabsf(l2lse) / l2s;  // the rounding of l2lse - c
    sh.s.xlo = xl - 1e-5f * (fabsf(xl) + 1.f) - slack;
    sh.s.xhi = xh + 1e-5f * (fabsf(xh) + 1.f) + slack;
    // the same bounds as bf16, rounded outwards, in both halves of a word
    const uint32_t lb = __bfloat16_as_ushort(__float2bfloat16_rd(sh.s.xlo));
    const uint32_t hb = __bfloat16_as_ushort(__float2bfloat16_ru(sh.s.xhi));
    sh.s.lo2 = lb | (lb << 16);
    sh.s.hi2 = hb | (hb << 16);
    // bf16: a per-key histogram when b*'s interval spans at most 256 keys
    const int klo = static_cast<int>(order_key(__uint_as_float(lb << 16)) >> 16);
    const int khi = static_cast<int>(order_key(__uint_as_float(hb << 16)) >> 16);
    sh.s.klo = klo;
    sh.s.nk = sizeof(T) != 4 && bstar != kToppMassBins - 1 && khi - klo < 256 ? khi - klo + 1 : 0;
    // the last bin also holds everything below it, -inf and NaN included
    sh.s.last_bin = bstar == kToppMassBins - 1;
  }
  if (tid < 256) { sh.hq[tid] = 0u; sh.hc[tid] = 0u; sh.hh[tid] = 0u; }
  __syncthreads();  // every cell has been read: they hold the list from here on

  // ---- pass 2: the threshold bin's keys and quantised masses ----------------
  uint32_t *const lkey = cell;
  uint32_t *const lq = cell + kToppListCap;
  const float xlo = sh.s.xlo, xhi = sh.s.xhi;
  const uint32_t lo2 = sh.s.lo2, hi2 = sh.s.hi2;
  const bool last_bin = sh.s.last_bin;
  const int klo = sh.s.klo, nk = sh.s.nk;
  // the threshold bin's logits, from the list of the first attempt when it
  // holds them all, else from the row (L2)
  auto take = [&](float x) {
    float y, t;
    if ((last_bin || (x >= xlo && x <= xhi)) && mass_bin(x, y, t) == static_cast<uint32_t>(bstar)) {
      const uint32_t q = quantise(y, t);
      if (nk > 0) {
        // x lies in [xlo, xhi], so its key lies in [klo, klo + nk)
        const int d = static_cast<int>(order_key(x) >> 16) - klo;
        const uint32_t old = atomicAdd(&sh.hq[d], q);
        if (old + q < q) atomicAdd(&sh.hh[d], 1u);  // the carry out of the low word
        atomicAdd(&sh.hc[d], 1u);
      } else {
        const int idx = atomicAdd(&sh.s.n, 1);
        if (idx < kToppListCap) {
          lkey[idx] = order_key(x);
          lq[idx] = q;
        }
      }
    }
  };
  if (high && !sh.s.nh_over) {
    for (int k = 0; k < n_high; ++k) take(high_value(hstore[k * NT + tid]));
  } else {
    topp_for_each_group<T, VEC>(rowp, a.V, [&](const uint4 &v) {
      // almost no group holds a logit of the interval
      if (!last_bin && !group_hits<T>(v, xlo, xhi, lo2, hi2)) return;
#pragma unroll
      for (int e = 0; e < LogitTraits<T>::kPerVec; ++e) take(LogitTraits<T>::at(v, e));
    });
  }
  __syncthreads();
  const unsigned long long bin_above = sh.s.bin_above;
  const unsigned fr = sh.frac[bstar & 7];
  const int bsh = bstar >> 3;
  auto to_mass = [&](unsigned long long s) { return (s * fr) >> bsh; };
  uint32_t vstar;
  unsigned long long in_kept;
  if (nk > 0) {
    // ---- the threshold key from the per-key histogram, keys descending ------
    const int d = nk - 1 - tid;  // thread tid takes key klo + nk - 1 - tid
    const unsigned long long hv =
        tid < nk ? (static_cast<unsigned long long>(sh.hh[d]) << 32) | sh.hq[d] : 0ull;
    unsigned long long tot_unused;
    const unsigned long long ex = block_excl_scan_u64<NT>(hv, sh.u64s, &tot_unused);
    const bool c = tid < nk && sh.hc[d] > 0u && bin_above + to_mass(ex) < limit;
    const int best = block_max_int<NT>(c ? tid : -1, sh.ints);
    if (best < 0) return false;  // an empty threshold bin (not reached)
    if (tid == best) {
      const uint32_t k16 = static_cast<uint32_t>(klo + d);
      // the 32-bit key of that bf16 logit: low half 0 (positive) or 1s (negative)
      sh.s.prefix = (k16 << 16) | ((k16 & 0x8000u) ? 0u : 0xffffu);
      sh.s.in_kept = ex + hv;
    }
    __syncthreads();
    vstar = sh.s.prefix;
    in_kept = sh.s.in_kept;
  } else {
    const int n = sh.s.n;
    if (n > kToppListCap || n == 0) return false;  // the exact path

    // ---- otherwise a radix select over the list of the bin's logits -------------
    // the bits in which the list's keys differ: [lb, hb]
    uint32_t kmin = 0xffffffffu;
    unsigned long long qsum = 0;
    for (int i = tid; i < n; i += NT) {
      kmin = min(kmin, lkey[i]);
      qsum += lq[i];
    }
    kmin = block_min_u32<NT>(kmin, sh.ints);
    uint32_t diff = 0u;
    for (int i = tid; i < n; i += NT) diff |= lkey[i] ^ kmin;
    diff = block_or_u32<NT>(diff, sh.ints);
    unsigned long long qtot;
    block_excl_scan_u64<NT>(qsum, sh.u64s, &qtot);
    const int hb = diff == 0u ? -1 : 31 - __clz(diff);
    const int lb = diff == 0u ? 0 : __ffs(diff) - 1;
    uint32_t prefix = hb == 31 ? 0u : (kmin >> (hb + 1));
    unsigned long long in_above = 0;
    in_kept = qtot;
    for (int top = hb; top >= lb; top -= 8) {
      const int w = min(8, top + 1 - lb), sh_lo = top + 1 - w;
      const int nb = 1 << w;
      if (tid < 256) { sh.hq[tid] = 0u; sh.hc[tid] = 0u; }
      __syncthreads();
      for (int i = tid; i < n; i += NT) {
        const uint32_t key = lkey[i];
        if (top == 31 || (key >> (top + 1)) == prefix) {
          const uint32_t d = (key >> sh_lo) & static_cast<uint32_t>(nb - 1);
          atomicAdd(&sh.hq[d], lq[i]);
          atomicAdd(&sh.hc[d], 1u);
        }
      }
      __syncthreads();
      const int dd = nb - 1 - tid;  // thread tid takes digit nb - 1 - tid (descending)
      const unsigned long long hv = tid < nb ? sh.hq[dd] : 0ull;
      unsigned long long tot_unused;
      const unsigned long long ex = block_excl_scan_u64<NT>(hv, sh.u64s, &tot_unused);
      const bool c = tid < nb && sh.hc[dd] > 0u && bin_above + to_mass(in_above + ex) < limit;
      const int best = block_max_int<NT>(c ? tid : -1, sh.ints);
      if (best < 0) return false;  // not reached: the bin's largest key is always a candidate
      if (tid == best) {
        sh.s.prefix = (prefix << w) | static_cast<uint32_t>(dd);
        sh.s.in_above = in_above + ex;
        sh.s.in_kept = in_above + ex + hv;
      }
      __syncthreads();
      prefix = sh.s.prefix;
      in_above = sh.s.in_above;
      in_kept = sh.s.in_kept;
    }
    // the bits below lb are the same in every key of the list
    vstar = hb < 0 ? kmin : (prefix << lb) | (kmin & ((1u << lb) - 1u));
  }
  const unsigned long long kept_mass = bin_above + to_mass(in_kept);
  // keys order logits as floats do, with -0 = +0; NaN is never kept
  const float thr = key_value(vstar);
  auto kept = [&](float x) { return x >= thr; };
  if (j != a.K) {
    if (tid == 0) topp_finish_fast<T>(a, row, part, j, rowp, topp_log_ratio(kept_mass, total), kept, thr);
    return true;
  }
  // the bonus row: exact weights exp(s x - lse) = exp(s (x - lse / s)), as on
  // the exact path (units of 2^-38; their sum is about 2^38), so that a draw
  // can differ from exact arithmetic only within about 1e-9 of a boundary
  stage_exp2_table(sh.tab);
  __syncthreads();
  const float ref = lse / a.tscale;
  auto weight = [&](float x) -> unsigned long long {
    return static_cast<unsigned long long>(weight_fixed(x, ref, a.balpha, sh.tab) >> 12);
  };
  const long long tok = topp_bonus_draw<T, VEC>(a, part, rowp, true, thr, weight, sh);
  if (tid == 0) {
    const float log_z = topp_log_ratio(kept_mass, total);
    RowResult r = a.ws.results[row];
    r.lse += log_z;
    r.lse_alpha += log_z;
    r.tok = static_cast<int>(tok);
    a.ws.results[row] = r;
  }
  return true;
}

// Exact path: a radix select over the whole row's keys.
template <typename T, bool VEC>
__device__ void topp_exact(const StepArgs &a, unsigned long long p64, ToppShared &sh) {
  using Tr = LogitTraits<T>;
  using Dg = ToppDigits<T>;
  constexpr int kShift = 12;  // bonus weights in units of 2^-(kFixBits - kShift)
  uint32_t *const s_lo = sh.cell;
  uint32_t *const s_hi = s_lo + kToppBins;
  const int tid = threadIdx.x;
  const int row = topp_row(a);
  const int rpp = 2 * a.K + 1;
  const int part = row / rpp, j = row - part * rpp;
  const bool bonus = j == a.K;
  const char *rowp = row_base<T>(a, row);
  const float lse = a.ws.results[row].lse;
  const float l2s = a.tscale * kLog2e, l2lse = lse * kLog2e;
  if (bonus) stage_exp2_table(sh.tab);

  // adds round(pi 2^40), lowest bit set, for the finite logit x to bin b
  auto add_mass = [&](uint32_t b, float x) {
    const float pm = fminf(fast_exp2(fmaf(x, l2s, -l2lse)), 2.f);  // pi, about 1e-7 relative
    const unsigned long long fx = static_cast<unsigned long long>(float_to_ll_rn(pm * 0x1p40f)) | 1ull;
    const uint32_t lo = static_cast<uint32_t>(fx);
    const uint32_t old = atomicAdd(&s_lo[b], lo);
    const uint32_t hi = static_cast<uint32_t>(fx >> 32) + (old + lo < lo ? 1u : 0u);
    if (hi) atomicAdd(&s_hi[b], hi);
  };

  float mx = kNegInf;
  uint32_t prefix = 0;
  int consumed = 0;  // key bits fixed so far
  unsigned long long total = 0, above = 0;
  bool ok = true;
#pragma unroll 1
  for (int pass = 0; pass < Dg::kPasses; ++pass) {
    const int width = Dg::width(pass);
    const int nb = 1 << width;
    const int shift = 32 - consumed - width;
    for (int b = tid; b < nb; b += kToppThreads) s_lo[b] = s_hi[b] = 0u;
    __syncthreads();
    if (pass == 0) {
      topp_for_each<T, VEC>(rowp, a.V, [&](float x) {
        mx = fmaxf(mx, x);
        if (x > kNegInf && x < -kNegInf) add_mass(order_key(x) >> shift, x);
      });
    } else {
      topp_for_each<T, VEC>(rowp, a.V, [&](float x) {
        const uint32_t key = order_key(x);
        if ((key >> (shift + width)) == prefix && x > kNegInf && x < -kNegInf)
          add_mass((key >> shift) & static_cast<uint32_t>(nb - 1), x);
      });
    }
    __syncthreads();
    // bins in descending key order: thread tid takes positions
    // [tid c, tid c + c), position d being bin nb - 1 - d
    const int c = (nb + kToppThreads - 1) / kToppThreads;
    unsigned long long sum = 0;
    for (int i = 0; i < c; ++i) {
      const int d = tid * c + i;
      if (d < nb) sum += (static_cast<unsigned long long>(s_hi[nb - 1 - d]) << 32) | s_lo[nb - 1 - d];
    }
    unsigned long long tot;
    const unsigned long long excl = block_excl_scan_u64<kToppThreads>(sum, sh.u64s, &tot);
    if (pass == 0) total = tot;
    const unsigned long long limit = __umul64hi(total, p64);  // floor(top_p total)
    // the lowest candidate: a non-empty bin whose mass above is below limit
    int best = -1;
    unsigned long long best_a = 0, best_v = 0, run = above + excl;
    for (int i = 0; i < c; ++i) {
      const int d = tid * c + i;
      if (d >= nb) break;
      const unsigned long long m =
          (static_cast<unsigned long long>(s_hi[nb - 1 - d]) << 32) | s_lo[nb - 1 - d];
      if (m > 0 && run < limit) { best = d; best_a = run; best_v = m; }
      run += m;
    }
    const int bd = block_max_int<kToppThreads>(best, sh.ints);
    if (bd >= 0 && best == bd) {
      sh.s.prefix = (prefix << width) | static_cast<uint32_t>(nb - 1 - bd);
      sh.s.above = best_a;
      sh.s.kept = best_a + best_v;
    }
    __syncthreads();
    if (bd < 0) { ok = false; break; }  // an empty or non-finite row (reported elsewhere)
    prefix = sh.s.prefix;
    above = sh.s.above;
    consumed += width;
  }
  // kept: logits at or above the threshold key (nothing when the select failed)
  const unsigned long long kept_mass = ok ? sh.s.kept : 0ull;
  // the threshold logit: the key prefix, padded with zero bits
  const float thr = key_value(prefix << (32 - Dg::kKeyBits));
  auto kept = [&](float x) { return ok && x >= thr; };
  if (!bonus) {
    if (tid == 0)
      topp_finish_fast<T>(a, row, part, j, rowp, topp_log_ratio(kept_mass, total), kept,
                          ok ? thr : -kNegInf);
    return;
  }
  // ---- bonus row: weights exp(s (x - M)) in exact fixed point ---------------
  const float M = block_max_nt<kToppThreads>(mx, sh.fl);
  const bool live = ok && M > kNegInf && M < -kNegInf;
  auto weight = [&](float x) -> unsigned long long {
    return static_cast<unsigned long long>(weight_fixed(x, M, a.balpha, sh.tab) >> kShift);
  };
  const long long tok = topp_bonus_draw<T, VEC>(a, part, rowp, live, thr, weight, sh);
  if (tid == 0) {
    const float log_z = topp_log_ratio(kept_mass, total);
    RowResult r = a.ws.results[row];
    r.lse += log_z;
    r.lse_alpha += log_z;
    r.tok = static_cast<int>(tok);
    a.ws.results[row] = r;
  }
}

// qb > 0: the mass-bin path with quantisation bits qb, falling back to the
// exact path row by row; qb == 0: the exact path for every row.  p64 =
// top_p 2^64.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kToppThreads, 2)
topp_kernel(const StepArgs a, unsigned long long p64, int qb) {
  extern __shared__ __align__(16) unsigned char topp_smem[];
  ToppShared &sh = *reinterpret_cast<ToppShared *>(topp_smem);
  // programmatic dependent launch: the row combine's log-sum-exps first; the
  // tail may launch once every CTA of this grid has started (it waits for
  // this grid before it reads the nucleus results)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (qb > 0) {
    if (topp_mass_bins<T, VEC>(a, p64, qb, sh, topp_smem + kToppHighOff,
                               reinterpret_cast<uint4 *>(topp_smem + kToppQueueOff))) {
      return;
    }
    __syncthreads();
  }
  topp_exact<T, VEC>(a, p64, sh);
}

// The nucleus kernel.  Its quantisation bits qb keep every (bin, lane) cell
// of the mass-bin path below 2^32: a cell takes at most 16 threads' logits,
// each q at most 2^qb 2^(1/16); below 18 bits the exact path takes every row.
template <typename T, bool VEC>
static cudaError_t launch_topp_t(const StepArgs &a, float top_p, long long rows,
                                 cudaStream_t stream) {
  constexpr int E = LogitTraits<T>::kPerVec;
  const long long ng = (static_cast<long long>(a.V) + E - 1) / E;
  const long long n_cell = (kToppThreads / 32) * ((ng + kToppThreads - 1) / kToppThreads) * E;
  int lg = 0;
  while ((1ll << lg) < n_cell) ++lg;
  int qb = 31 - lg < 20 ? 31 - lg : 20;
  if (qb < 18) qb = 0;
  const unsigned long long p64 =
      static_cast<unsigned long long>(std::ldexp(static_cast<double>(top_p), 64));
  const size_t smem = kToppSmemBytes;
  cudaError_t e = allow_dyn_smem(topp_kernel<T, VEC>, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(kToppThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topp_kernel<T, VEC>, a, p64, qb);
}

cudaError_t launch_topp(const StepArgs &a, int dtype, float top_p, long long rows,
                        cudaStream_t stream) {
  const int esz = dtype == SMC_BF16 ? 2 : 4;
  const bool vec = aligned16(a.target) && aligned16(a.draft) &&
                   (static_cast<long long>(a.V) * esz) % 16 == 0;
  if (dtype == SMC_BF16)
    return vec ? launch_topp_t<bf16_tag, true>(a, top_p, rows, stream)
               : launch_topp_t<bf16_tag, false>(a, top_p, rows, stream);
  return vec ? launch_topp_t<float, true>(a, top_p, rows, stream)
             : launch_topp_t<float, false>(a, top_p, rows, stream);
}

}  // namespace smcsd
