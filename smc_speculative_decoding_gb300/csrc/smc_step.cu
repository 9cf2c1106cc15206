// SMC-SD step kernels for sm_103a.
//
// One step ("Faster LLM Inference via Sequential Monte Carlo", section 2
// "核心流程": Score & Bonus, Reweight, Resample; "系统优化设计": KV pointer
// exchange) runs as three kernels chained by programmatic dependent launch:
//
//   row_stream_kernel  every target and draft row once, through a shared-
//                      memory ring filled by bulk copies: per (item, warp)
//                      partial (max, sum of exp) of the log-sum-exp rows, and
//                      per (chunk, warp) float-float sums of the bonus row's
//                      sampling weights;
//   finish_kernel      one warp per row: log-sum-exp and the drafted token's
//                      logit, or for the bonus row the inverse-CDF draw (which
//                      unit from the unit sums, then which element by an exact
//                      fixed-point rescan of that unit);
//   tail_kernel        one CTA per prompt: weight update, normalisation, ESS,
//                      systematic resampling, token emission, KV remap; in SpS
//                      mode the acceptance scan instead.
//
// Rows that are not 16-byte aligned (V * bytes per logit not a multiple of
// 16, or a misaligned base pointer) take step_rows_kernel instead: one CTA per
// (row, 16 KB chunk) with plain loads, and the last CTA of a row (atomic
// ticket) combines it.  smc_resample and kv_blocktable_remap run the tail's
// pieces alone (resample_kernel, kv_remap_kernel).  With top_p < 1 the
// nucleus kernel (topp.cu) runs between the row combine and the tail.
#include <atomic>
#include <cmath>

#include "row_common.cuh"
#include "kernels.h"
#include "smcsd.h"
#include "step_args.cuh"

namespace smcsd {

int chunk_elems(int dtype) { return kThreads * kNV * (dtype == SMC_BF16 ? 8 : 4); }
int chunks_per_row(int dtype, int V) {
  const int ch = chunk_elems(dtype);
  return (V + ch - 1) / ch;
}


// Blocks that hold `len` tokens (64-bit, so a corrupt length cannot overflow).
// ---------------------------------------------------------------------------
// Normalise one prompt's log-weights, compute ESS and, below the threshold,
// resample systematically.  The log-weights arrive as float-float values
// (the fp32 state plus this step's increment, unrounded) and everything
// stays float-float on the fp32 pipes (this GPU's fp64 rate is far lower).
// With e_i = exp(lw_i - max) by the accurate exponential (about 3e-10),
// S = sum e and Q = sum e^2, the normalised weights are w = e / S, so
//   ESS = 1 / sum w^2 = S^2 / Q,  resample iff S^2 < tau N Q,
// and ancestor a_i = min{j : C_j > (u0 + i)/N} with C the prefix of w is
// the first j whose prefix of e exceeds (u0 + i) S / N: no division on the
// critical path.  u0 is the step's resampling uniform of the prompt and rN
// the float-float 1/N, both computed by the caller ahead of time.  The
// block version serves any N <= 256; thread i < N holds lw_i and, on
// return, s_anc[i] holds the ancestor of particle i.  `tab` is the 2^(j/64)
// table in shared memory.
// ---------------------------------------------------------------------------
struct ResampleResult { bool resampled; float ess; };

// Smallest j in [0, n) with c[j] > pt, clamped to n-1 (c as float-float).
__device__ __forceinline__ int first_above(const float2 *c, int n, ff pt) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ff_gt(ff{c[mid].x, c[mid].y}, pt)) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Weight e = exp(lw - m) of one particle (0 for -inf or invalid).
__device__ __forceinline__ ff particle_mass(ff lw, float m, bool use, const float2 *tab) {
  if (!use) return ff{0.f, 0.f};
  const ff d = ff_sub(lw, ff{m, 0.f});
  return ff_norm(accurate_exp(d.hi, d.lo, tab));
}

// The resampling inputs that do not depend on the weights: the prompt's
// uniform u0 and 1/N as a float-float value.
struct ResampleKey { float u0; ff rn; };
__device__ __forceinline__ ResampleKey resample_key(uint64_t seed, uint32_t step, int b, int N) {
  return {philox_uniform(seed, step, b, 0, SMC_PURPOSE_RESAMPLE),
          ff_div(ff{1.f, 0.f}, ff{static_cast<float>(N), 0.f})};
}

// ESS = S^2 / Q and the decision S^2 < tau N Q.
__device__ __forceinline__ bool resample_decision(ff S, ff Q, float ess_frac, int N, bool ok,
                                                  float *ess) {
  const ff s2 = ff_mul(S, S);
  *ess = ff_div(s2, Q).hi;
  return ok && ff_gt(ff_mul(two_prod(ess_frac, static_cast<float>(N)), Q), s2);
}

__device__ __noinline__ ResampleResult normalise_resample(int N, ff lw, bool valid,
                                                          float ess_frac,
                                             ResampleKey key, unsigned *status, int *s_anc,
                                             float2 *s_c, float2 *s_red, const float2 *tab) {
  constexpr float kInf = -kNegInf;
  unsigned bits = 0;
  if (valid && (isnan(lw.hi) || lw.hi == kInf)) bits |= SMC_DEV_NONFINITE;
  const float m = block_max(valid && !isnan(lw.hi) ? lw.hi : kNegInf,
                            reinterpret_cast<float *>(s_red));
  const bool ok = m > kNegInf && m < kInf;
  if (threadIdx.x == 0 && m == kNegInf) bits |= SMC_DEV_ALL_ZERO_WEIGHT;
  if (bits) raise_status(status, bits);
  const ff e = particle_mass(lw, m, valid && ok, tab);
  const ff S = block_ff_sum(e, s_red);
  const ff Q = block_ff_sum(ff_mul(e, e), s_red);
  float ess;
  const bool resample = resample_decision(S, Q, ess_frac, N, ok, &ess);
  int anc = threadIdx.x;
  if (resample) {
    ff total;
    const ff c = block_ff_scan(e, s_red, &total);
    if (valid) s_c[threadIdx.x] = make_float2(c.hi, c.lo);
    __syncthreads();
    if (valid) {
      const ff pt = ff_mul(ff_mul(two_sum(key.u0, static_cast<float>(threadIdx.x)), S), key.rn);
      anc = first_above(s_c, N, pt);
    }
  }
  if (valid) s_anc[threadIdx.x] = anc;
  __syncthreads();
  return {resample, ess};
}

// The same for N <= 32, by warp 0 alone with shuffles (no CTA barrier).
__device__ ResampleResult normalise_resample_warp(int N, ff lw, bool valid, float ess_frac,
                                                  ResampleKey key, unsigned *status, int *s_anc,
                                                  float2 *s_c, const float2 *tab) {
  constexpr float kInf = -kNegInf;
  const int lane = threadIdx.x & 31;
  unsigned bits = 0;
  if (valid && (isnan(lw.hi) || lw.hi == kInf)) bits |= SMC_DEV_NONFINITE;
  const float m = warp_max(valid && !isnan(lw.hi) ? lw.hi : kNegInf);
  const bool ok = m > kNegInf && m < kInf;
  if (lane == 0 && m == kNegInf) bits |= SMC_DEV_ALL_ZERO_WEIGHT;
  if (bits) raise_status(status, bits);
  const ff e = particle_mass(lw, m, valid && ok, tab);
  // S = sum e and Q = sum e^2, the two butterflies interleaved
  ff S = e, Q = ff_mul(e, e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff s2{__shfl_xor_sync(0xffffffffu, S.hi, o), __shfl_xor_sync(0xffffffffu, S.lo, o)};
    const ff q2{__shfl_xor_sync(0xffffffffu, Q.hi, o), __shfl_xor_sync(0xffffffffu, Q.lo, o)};
    S = ff_add(S, s2);
    Q = ff_add(Q, q2);
  }
  float ess;
  const bool resample = resample_decision(S, Q, ess_frac, N, ok, &ess);
  int anc = lane;
  if (resample) {
    const ff c = warp_ff_incl_scan(e);
    if (valid) s_c[lane] = make_float2(c.hi, c.lo);
    __syncwarp();
    if (valid) {
      const ff pt = ff_mul(ff_mul(two_sum(key.u0, static_cast<float>(lane)), S), key.rn);
      anc = first_above(s_c, N, pt);
    }
  }
  if (valid) s_anc[lane] = anc;
  __syncwarp();
  return {resample, ess};
}

// ---------------------------------------------------------------------------
// Block-table remap by ancestors and append of n_append tokens, one prompt,
// one CTA.  Reference counts count table references; the free stack of prompt
// b is free_list[b*P .. b*P + free_top[b]).  See smcsd.h (kv_blocktable_remap).
//
// The scratch holds a copy of the prompt's tables and token counts and a
// cleared freed-block bitmap, in shared memory (staged) or in workspace
// scratch.  Staged, it also holds copies of the prompt's reference counts,
// of free_top and of the top kStackPre entries of the free stack, all read
// while the weights are computed, so that the remap itself waits on no
// global load; `delta` collects each block's net count change and then the
// list of blocks freed by this remap.  s_nb holds each particle's used block
// count.  Loops run a warp per particle and a lane per table slot, so no
// index needs a division.
// ---------------------------------------------------------------------------
constexpr int kStackPre = 512;

struct KvScratch {
  int *old_t;      // [N*T]
  int *old_l;      // [N]
  unsigned *bits;  // [ceil(P/32)]
  int *rc;         // [P]  staged: reference counts of the prompt's pool (else null)
  int *delta;      // [P]  staged: count changes, then the freed blocks (else null)
  int *stk;        // [kStackPre] staged: stk[k] = free stack entry k below the top
  int *top0;       // [1]  staged: free_top at copy-in
};

// dst[i] = src[i] for i in [0, n), by thread t of nt, with kB loads in
// flight per thread before the first store.
__device__ __forceinline__ void copy_batched(int *dst, const int32_t *src, int n, int t, int nt) {
  constexpr int kB = 16;
  for (int base = t; base < n; base += nt * kB) {
    int v[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = base + u * nt;
      v[u] = i < n ? __ldcg(src + i) : 0;
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = base + u * nt;
      if (i < n) dst[i] = v[u];
    }
  }
}

// Copy prompt b's state into the scratch and clear the bitmap, using threads
// [t0, t0 + nt) of the CTA; no barrier inside.
__device__ void kv_copy_in(const KvArgs &kv, int b, int N, const KvScratch &sc, int t0, int nt) {
  const int T = kv.T, P = kv.P;
  const int words = (P + 31) / 32;
  const int t = static_cast<int>(threadIdx.x) - t0;
  if (t < 0 || t >= nt) return;
  int top = 0;
  if (sc.rc) top = __ldcg(kv.free_top + b);  // every thread; one transaction per warp
  copy_batched(sc.old_t, kv.tables + static_cast<size_t>(b) * N * T, N * T, t, nt);
  copy_batched(sc.old_l, kv.seq_len + static_cast<size_t>(b) * N, N, t, nt);
  for (int w = t; w < words; w += nt) sc.bits[w] = 0u;
  if (sc.rc) {
    const int32_t *stack = kv.free_list + static_cast<size_t>(b) * P;
    copy_batched(sc.rc, kv.refcount + static_cast<size_t>(b) * P, P, t, nt);
    for (int k = t; k < P; k += nt) sc.delta[k] = 0;
    if (t == 0) *sc.top0 = top;
    const int n_pre = (top >= 0 && top <= P) ? min(top, kStackPre) : 0;
    for (int k = t; k < n_pre; k += nt) sc.stk[k] = __ldcg(stack + top - 1 - k);
  }
}

// The staged copy-in of kv_copy_in, by asynchronous copies that the caller
// waits for later (cp_async_wait_all, then a CTA barrier): prompt b's tables,
// token counts and reference counts; the freed-block bitmap and the count
// changes are cleared.  The free stack's top entries need free_top first and
// come separately (kv_copy_stack_async).  All threads of the CTA call it.
__device__ void kv_copy_in_async(const KvArgs &kv, int b, int N, const KvScratch &sc) {
  const int T = kv.T, P = kv.P;
  const int words = (P + 31) / 32;
  const int t = threadIdx.x;
  const int32_t *tables = kv.tables + static_cast<size_t>(b) * N * T;
  for (int i = t; i < N * T; i += kThreads) cp_async4(sc.old_t + i, tables + i);
  const int32_t *len = kv.seq_len + static_cast<size_t>(b) * N;
  for (int i = t; i < N; i += kThreads) cp_async4(sc.old_l + i, len + i);
  const int32_t *rc = kv.refcount + static_cast<size_t>(b) * P;
  for (int i = t; i < P; i += kThreads) cp_async4(sc.rc + i, rc + i);
  for (int w = t; w < words; w += kThreads) sc.bits[w] = 0u;
  for (int k = t; k < P; k += kThreads) sc.delta[k] = 0;
}

// The top kStackPre entries of prompt b's free stack (stk[k] = entry k below
// the top `top`) and the top itself, by asynchronous copies.
__device__ void kv_copy_stack_async(const KvArgs &kv, int b, int top, const KvScratch &sc) {
  const int P = kv.P;
  const int32_t *stack = kv.free_list + static_cast<size_t>(b) * P;
  if (threadIdx.x == 0) *sc.top0 = top;
  const int n_pre = (top >= 0 && top <= P) ? min(top, kStackPre) : 0;
  for (int k = threadIdx.x; k < n_pre; k += kThreads) cp_async4(sc.stk + k, stack + top - 1 - k);
}

// L2 prefetch of what a prompt's remap stages: tables, token counts,
// reference counts, the free stack and its top.
__device__ __forceinline__ void kv_prefetch_l2(const KvArgs &kv, int b, int N) {
  const size_t nt = static_cast<size_t>(N) * kv.T, p = static_cast<size_t>(kv.P);
  prefetch_l2(kv.tables + b * nt, nt * sizeof(int32_t));
  prefetch_l2(kv.refcount + b * p, p * sizeof(int32_t));
  prefetch_l2(kv.free_list + b * p, p * sizeof(int32_t));
  prefetch_l2(kv.seq_len + static_cast<size_t>(b) * N, static_cast<size_t>(N) * sizeof(int32_t));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(kv.free_top + b));
}

// The count update of a remap whose copy of the tables lives in workspace
// scratch (prompts too large to stage in shared memory): global atomics, new
// references first, so that no count touches 0 before every increment is in.
// Out of line: shapes that stage in shared memory never run it.  Returns
// false (with *s_flag set) when a block id lies outside the prompt's pool.
// All threads of the CTA call it.
__device__ __noinline__ bool kv_remap_unstaged(const KvArgs &kv, int N, const int *s_anc,
                                               const int *s_nb, const KvScratch &sc, int lo_id,
                                               int32_t *tables, int32_t *seq_len,
                                               volatile int *s_flag) {
  const int T = kv.T, P = kv.P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  auto in_pool = [&](int blk) { return blk >= lo_id && blk < lo_id + P; };
  for (int i = warp; i < N; i += kWarps) {
    for (int t = lane; t < s_nb[i]; t += 32) {
      if (!in_pool(sc.old_t[i * T + t])) *s_flag = 1;
    }
  }
  __syncthreads();
  if (*s_flag) return false;
  for (int i = warp; i < N; i += kWarps) {
    const int a = s_anc[i];
    const int nb_new = s_nb[a], nb_old = s_nb[i];
    for (int t = lane; t < nb_new; t += 32) {
      const int blk = sc.old_t[a * T + t];
      if (!(t < nb_old && sc.old_t[i * T + t] == blk)) atomicAdd(&kv.refcount[blk], 1);
    }
  }
  __syncthreads();
  for (int i = warp; i < N; i += kWarps) {
    const int a = s_anc[i];
    const int nb_new = s_nb[a], nb_old = s_nb[i];
    for (int t = lane; t < T; t += 32) {
      const int nv = sc.old_t[a * T + t];
      if (t < nb_old) {
        const int blk = sc.old_t[i * T + t];
        if (!(t < nb_new && nv == blk)) {
          if (atomicSub(&kv.refcount[blk], 1) == 1) {
            const int rel = blk - lo_id;
            atomicOr(&sc.bits[rel >> 5], 1u << (rel & 31));
          }
        }
      }
      tables[i * T + t] = nv;
    }
  }
  for (int i = tid; i < N; i += kThreads) seq_len[i] = sc.old_l[s_anc[i]];
  __syncthreads();
  return true;
}

// Shared state of one prompt's remap (kv_prepare, kv_remap_append).
struct KvSmem {
  int nb[SMC_MAX_N];     // used blocks of each particle before the remap
  int otail[SMC_MAX_N];  // its partially filled last block, -1 when it has none
  int ntail[SMC_MAX_N];  // the same after the remap (append of more than 32 particles)
  int ired[2 * kWarps];
  long long ll[kWarps];
  int bad;               // kv_prepare's findings: kBadState | kBadId | kBadTail
  int top_old;           // free_top before the remap
  int n_freed;           // blocks the remap pushed
  int flag;              // the unstaged remap's error flag
  int t_common;          // first table slot at which the particles' tables differ
};
constexpr int kBadState = 1;  // a token count outside [0, T*block_size] or free_top outside [0, P]
constexpr int kBadId = 2;     // a used block outside the prompt's pool
constexpr int kBadTail = 4;   // a partially filled last block outside the pool

// What the remap and the append read of the state before the remap, by
// threads [t0, t0 + nt) of the CTA with no barrier inside (ks.bad must be 0
// and ks.t_common T beforehand, kv_prepare_init; the caller's barrier
// publishes the rest): each particle's used block count and partial tail
// block, free_top, the checks of the ids, and the first table slot at which
// two particles differ (in the block id or in whether the slot is used).
// Every used block of every particle is checked, so that a remap can take
// any of them without checking again.  Below t_common every particle holds
// the same blocks (the shared prefix), so no remap changes a table or a
// count there.
__device__ __forceinline__ void kv_prepare_init(KvSmem &ks, int T) {
  ks.bad = 0;
  ks.t_common = T;
}

__device__ void kv_prepare(const KvArgs &kv, int b, int N, const KvScratch &sc, KvSmem &ks,
                           int t0, int nt) {
  const int t = static_cast<int>(threadIdx.x) - t0;
  if (t < 0 || t >= nt) return;
  const int T = kv.T, P = kv.P;
  const unsigned bs = static_cast<unsigned>(kv.block_size);
  const int lo_id = b * P;
  const long long cap = static_cast<long long>(T) * kv.block_size;  // tokens a full table holds
  auto in_pool = [&](int blk) { return blk >= lo_id && blk < lo_id + P; };
  int bad = 0;
  if (t == 0) {
    const int top0 = sc.rc ? *sc.top0 : __ldcg(kv.free_top + b);
    ks.top_old = top0;
    if (top0 < 0 || top0 > P) bad |= kBadState;
  }
  for (int i = t; i < N; i += nt) {
    const int len = sc.old_l[i];
    int nb = 0, tail = -1;
    if (len < 0 || len > cap) {
      bad |= kBadState;
    } else {
      nb = static_cast<int>((static_cast<unsigned>(len) + bs - 1u) / bs);
      if (static_cast<unsigned>(len) % bs) {
        tail = sc.old_t[i * T + nb - 1];
        if (!in_pool(tail)) bad |= kBadTail;
      }
    }
    ks.nb[i] = nb;
    ks.otail[i] = tail;
  }
  named_bar_sync(2, nt);  // ks.nb of every particle
  // every slot (i, s): consecutive threads on consecutive particles at one
  // slot, each thread's pairs kept apart by nt; the first slot at which a
  // particle differs from particle 0 bounds t_common
  const int nb0 = ks.nb[0];
  const int di = nt % N, ds = nt / N;
  int i = t % N, s = t / N, first = T;
  while (s < T) {
    const int v = sc.old_t[i * T + s];
    const bool used = s < ks.nb[i];
    if (used && !in_pool(v)) bad |= kBadId;
    if (s < first && (v != sc.old_t[s] || used != (s < nb0))) first = s;
    i += di;
    s += ds;
    if (i >= N) {
      i -= N;
      ++s;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
  if ((t & 31) == 0 && first < T) atomicMin(&ks.t_common, first);
  if (bad) atomicOr(&ks.bad, bad);
}

// Exclusive warp scan of v (all lanes); *total gets the warp's sum.
__device__ __forceinline__ int warp_excl_scan_i(int v, int *total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// ceil(a / b) for a >= 0, b >= 1, by a 32-bit division when the operands
// allow (a 64-bit division costs several hundred cycles).
__device__ __forceinline__ long long ceil_div_nonneg(long long a, int b) {
  const unsigned long long n = static_cast<unsigned long long>(a) + static_cast<unsigned>(b) - 1ull;
  if (n < 4294967296ull) return static_cast<unsigned>(n) / static_cast<unsigned>(b);
  return static_cast<long long>(n / static_cast<unsigned long long>(b));
}

// Remap of prompt b's block tables by the ancestors s_anc (when resampled)
// and append of n_append tokens to every particle, by the whole CTA.  With
// `prepared`, kv_prepare has run on the staged state (all threads passed a
// barrier since); with `copied`, the state is already in `sc`.
//
// Staged state: the pushed blocks are listed in shared memory and go back as
// one range, and each remapped table goes back as one contiguous row segment
// (past the shared prefix).  Global stores are the expensive part of this
// latency-bound code (on GB300 each warp-wide store instruction occupies the
// SM for about 40 cycles, coalesced or not), so only changed counts are
// stored.
__device__ void kv_remap_append(const KvArgs &kv, int b, int N, const int *s_anc, bool resampled,
                                int n_append, const Workspace &ws, KvSmem &ks,
                                const KvScratch &sc, bool copied, bool prepared) {
  const int T = kv.T, bs = kv.block_size, P = kv.P;
  const int lo_id = b * P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int words = (P + 31) / 32;
  const bool staged = sc.rc != nullptr;
  int32_t *tables = kv.tables + static_cast<size_t>(b) * N * T;
  int32_t *seq_len = kv.seq_len + static_cast<size_t>(b) * N;
  int32_t *stack = kv.free_list + static_cast<size_t>(b) * P;
  auto in_pool = [&](int blk) { return blk >= lo_id && blk < lo_id + P; };
  auto fail = [&]() {
    if (tid == 0) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
  };
  if (!copied) kv_copy_in(kv, b, N, sc, 0, kThreads);
  if (!prepared) {
    if (tid == 0) kv_prepare_init(ks, T);
    __syncthreads();
    kv_prepare(kv, b, N, sc, ks, 0, kThreads);
  }
  if (tid == 0) {
    kv.n_cow[b] = 0;
    ks.n_freed = 0;
    ks.flag = 0;
  }
  __syncthreads();
  {
    const int bad = ks.bad;
    if ((bad & kBadState) || (bad & (resampled ? kBadId : kBadTail))) {
      fail();
      return;
    }
  }
  const int top_old = ks.top_old;

  if (resampled) {
    if (staged) {
      // net reference-count change per block in shared memory: a slot whose
      // block changes gives +1 to the new block and -1 to the old one; then
      // a pass over the same slots applies the changes, and a count reaching
      // 0 frees the block.  Only slots from t_common on can change.  Slot
      // (i, t) sits at idx = t N + i, so consecutive threads take consecutive
      // particles at one slot (blocks appended in the same step sit N ids
      // apart along a table: a warp along one table would send its updates to
      // two banks).  Each thread's slots advance by kThreads; their loads are
      // issued in batches of kU before the updates.
      constexpr int kU = 4;
      const int tc = ks.t_common;
      const int di = kThreads % N, dt = kThreads / N;
      int i = tid % N, t = tc + tid / N;
      while (t < T) {
        int nv[kU], ov[kU];
        bool upd[kU], hn[kU], ho[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          upd[u] = false;
          if (t < T) {
            const int anc = s_anc[i];
            upd[u] = anc != i;  // a particle that is its own ancestor keeps its table
            nv[u] = sc.old_t[anc * T + t];
            ov[u] = sc.old_t[i * T + t];
            hn[u] = t < ks.nb[anc];
            ho[u] = t < ks.nb[i];
          }
          i += di;
          t += dt;
          if (i >= N) {
            i -= N;
            ++t;
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (!upd[u]) continue;
          if (hn[u] && !(ho[u] && ov[u] == nv[u])) atomicAdd(&sc.delta[nv[u] - lo_id], 1);
          if (ho[u] && !(hn[u] && nv[u] == ov[u])) atomicSub(&sc.delta[ov[u] - lo_id], 1);
        }
      }
      // the new tables: row segments [t_common, T) of the ancestors, a warp a row
      for (int p = warp; p < N; p += kWarps) {
        const int anc = s_anc[p];
        if (anc == p) continue;
        for (int s2 = tc + lane; s2 < T; s2 += 32) tables[p * T + s2] = sc.old_t[anc * T + s2];
      }
      for (int p = tid; p < N; p += kThreads) seq_len[p] = sc.old_l[s_anc[p]];
      __syncthreads();
      // every block whose count changed is an old block at a slot from
      // t_common on; the first thread to reach it takes its change
      i = tid % N;
      t = tc + tid / N;
      for (; t < T;) {
        if (t < ks.nb[i]) {
          const int k = sc.old_t[i * T + t] - lo_id;
          const int d = atomicExch(&sc.delta[k], 0);
          if (d != 0) {
            const int nr = sc.rc[k] + d;
            kv.refcount[lo_id + k] = nr;
            if (nr == 0) atomicOr(&sc.bits[k >> 5], 1u << (k & 31));
          }
        }
        i += di;
        t += dt;
        if (i >= N) {
          i -= N;
          ++t;
        }
      }
      __syncthreads();
    } else {
      if (!kv_remap_unstaged(kv, N, s_anc, ks.nb, sc, lo_id, tables, seq_len, &ks.flag)) {
        fail();
        return;
      }
    }
    // push the freed blocks in ascending id order: staged, listed in `delta`
    // (whose counts are spent) and written back as one range; else straight
    // to the stack
    int top = top_old;
    for (int w0 = 0; w0 < words; w0 += kThreads) {
      const int w = w0 + tid;
      unsigned fb = w < words ? sc.bits[w] : 0u;
      int total;
      int pos = top + block_excl_scan_i(__popc(fb), ks.ired, &total);
      if (fb) sc.bits[w] = 0u;
      while (fb) {
        const int bit = __ffs(fb) - 1;
        fb &= fb - 1;
        if (pos < P) {
          if (staged) sc.delta[pos - top_old] = lo_id + w * 32 + bit;
          else stack[pos] = lo_id + w * 32 + bit;
        }
        ++pos;
      }
      top += total;
    }
    if (top > P) {  // counts did not match the tables
      fail();
      return;
    }
    if (tid == 0) {
      kv.free_top[b] = top;
      ks.n_freed = top - top_old;
    }
    __syncthreads();
    if (staged) {
      for (int k = tid; k < top - top_old; k += kThreads) stack[top_old + k] = sc.delta[k];
    }
  }

  // ---- append: particle i's table is now row src(i) of the copy ----------
  // (errors go to ks.flag: 1 bad block, 2 table overflow, 4 pool exhausted)
  const int n_freed = ks.n_freed;
  const int top = top_old + n_freed;
  auto pop = [&](int k) -> int {
    if (!staged) return stack[top - 1 - k];
    if (k < n_freed) return sc.delta[n_freed - 1 - k];
    const int j = k - n_freed;
    return j < kStackPre ? sc.stk[j] : stack[top_old - 1 - j];
  };
  // particle p's part of the append; k = its first pop, cidx its fork's pair
  auto append_one = [&](int p, int src, int len, int nb, int tail, int fork, int grow, int k,
                        int cidx) {
    if (fork) {
      const int d = pop(k);
      ++k;
      if (in_pool(d)) {
        int32_t *pair = kv.cow_pairs + (static_cast<size_t>(b) * N + cidx) * 2;
        pair[0] = tail;
        pair[1] = d;
        tables[p * T + nb - 1] = d;
        kv.refcount[d] = 1;
        atomicSub(&kv.refcount[tail], 1);
      } else {
        atomicOr(&ks.flag, 1);
      }
    }
    for (int g = 0; g < grow; ++g) {
      const int d = pop(k);
      ++k;
      if (in_pool(d)) {
        tables[p * T + nb + g] = d;
        kv.refcount[d] = 1;
      } else {
        atomicOr(&ks.flag, 1);
      }
    }
    seq_len[p] = static_cast<int>(len + n_append);
  };
  const bool warp_append = N <= 32 && staged;
  if (n_append > 0 && warp_append) {
    // one warp: no CTA barrier
    if (warp == 0) {
      const bool valid = lane < N;
      const int src = valid ? (resampled ? s_anc[lane] : lane) : 0;
      const int len = valid ? sc.old_l[src] : 0;
      const int nb = valid ? ks.nb[src] : 0;
      const int tail = valid ? ks.otail[src] : -1;
      // a shared partial tail stays with its lowest particle; the others fork
      const unsigned peers = __match_any_sync(0xffffffffu, tail >= 0 ? tail : -1 - lane);
      const int fork = (tail >= 0 && __ffs(peers) - 1 != lane) ? 1 : 0;
      const long long nb2 = valid ? ceil_div_nonneg(static_cast<long long>(len) + n_append, bs) : 0;
      int n_forks, total_pops;
      const int grow = (valid && nb2 <= T) ? static_cast<int>(nb2) - nb : 0;
      const int cidx = warp_excl_scan_i(fork, &n_forks);
      const int off = warp_excl_scan_i(fork + grow, &total_pops);
      if (__any_sync(0xffffffffu, nb2 > T)) {
        if (lane == 0) ks.flag = 2;
      } else if (total_pops > top) {
        if (lane == 0) ks.flag = 4;
      } else {
        if (valid) append_one(lane, src, len, nb, tail, fork, grow, off, cidx);
        if (lane == 0) {
          kv.free_top[b] = top - total_pops;
          kv.n_cow[b] = n_forks;
        }
      }
    }
    __syncthreads();
  } else if (n_append > 0) {
    const bool valid = tid < N;
    const int src = valid ? (resampled ? s_anc[tid] : tid) : 0;
    int len = 0, nb = 0, tail = -1;
    if (valid) {
      len = sc.old_l[src];
      nb = ks.nb[src];
      tail = ks.otail[src];
      ks.ntail[tid] = tail;
    }
    __syncthreads();
    int fork = 0;
    if (valid && tail >= 0) {
      for (int i2 = 0; i2 < tid; ++i2) {
        if (ks.ntail[i2] == tail) { fork = 1; break; }
      }
    }
    const long long nb2 = valid ? ceil_div_nonneg(static_cast<long long>(len) + n_append, bs) : 0;
    const bool overflow = __syncthreads_or(valid && nb2 > T) != 0;
    const int grow = (valid && !overflow) ? static_cast<int>(nb2) - nb : 0;
    // one scan of (forks, pops) packed in 64 bits: forks high, pops low
    long long both_total;
    const long long both = block_excl_scan_ll((static_cast<long long>(fork) << 32) | (fork + grow),
                                              ks.ll, &both_total);
    const int off = static_cast<int>(both & 0xffffffffll);
    const int cidx = static_cast<int>(both >> 32);
    const int total_pops = static_cast<int>(both_total & 0xffffffffll);
    const int n_forks = static_cast<int>(both_total >> 32);
    if (overflow) {
      if (tid == 0) ks.flag = 2;
    } else if (total_pops > top) {
      if (tid == 0) ks.flag = 4;
    } else {
      if (valid) append_one(tid, src, len, nb, tail, fork, grow, off, cidx);
      if (tid == 0) {
        kv.free_top[b] = top - total_pops;
        kv.n_cow[b] = n_forks;
      }
    }
    __syncthreads();
  }
  if (tid == 0 && n_append > 0) {
    const int f = ks.flag;
    if (f & 1) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
    if (f & 2) raise_status(ws.status, SMC_DEV_TABLE_OVERFLOW);
    if (f & 4) raise_status(ws.status, SMC_DEV_POOL_EXHAUSTED);
  }
}

// Shared-memory words a staged remap needs, and whether a shape fits.
__host__ __device__ inline size_t kv_stage_words(int N, int T, int P) {
  return static_cast<size_t>(N) * T + N + (P + 31) / 32 + 2 * static_cast<size_t>(P) +
         kStackPre + 1;
}
constexpr size_t kKvStageMaxBytes = 96 * 1024;

// Scratch of a remap: staged in `dyn` shared memory, or workspace scratch.
__device__ inline KvScratch kv_scratch(const KvArgs &kv, int b, int N, const Workspace &ws,
                                       int *dyn, bool staged) {
  KvScratch sc{};
  if (staged) {
    const int P = kv.P;
    sc.old_t = dyn;
    sc.old_l = dyn + static_cast<size_t>(N) * kv.T;
    sc.bits = reinterpret_cast<unsigned *>(sc.old_l + N);
    sc.rc = reinterpret_cast<int *>(sc.bits + (P + 31) / 32);
    sc.delta = sc.rc + P;
    sc.stk = sc.delta + P;
    sc.top0 = sc.stk + kStackPre;
  } else {
    sc.old_t = ws.kv_old_tables + static_cast<size_t>(b) * N * kv.T;
    sc.old_l = ws.kv_old_len + static_cast<size_t>(b) * N;
    sc.bits = ws.kv_bitmap + static_cast<size_t>(b) * ((kv.P + 31) / 32);
  }
  return sc;
}

// ---------------------------------------------------------------------------
// Prompt tails.
// ---------------------------------------------------------------------------
constexpr int kTailTokens = 2048;  // drafted tokens of a prompt staged in shared memory

struct TailSmem {
  int tok[kTailTokens];
  float2 c[SMC_MAX_N];
  float2 red[2 * kWarps];
  float2 tab[64];
  int anc[SMC_MAX_N];
  int bonus[SMC_MAX_N];
  int ired[2 * kWarps];
  KvSmem ks;
};

// Stages what a prompt's tail reads that no kernel of this step writes: the
// KV state (in shared memory when `sc` is staged, else in workspace scratch),
// the drafted tokens and the incoming log-weight of particle tid (returned);
// *top receives the prompt's free_top.  Called before the wait on the row
// kernels.  Staged copies are asynchronous: the caller issues the stack's
// copy (tail_prefetch_stack, once *top has arrived) and waits for them all
// (cp_async_wait_all) before prompt_tail.
__device__ float tail_prefetch(const StepArgs &a, int b, TailSmem &sm, const KvScratch &sc,
                               int *top) {
  const int N = a.N, K = a.K;
  const int tid = threadIdx.x;
  stage_exp2_table(sm.tab);
  *top = 0;
  if (a.use_kv) {
    if (sc.rc) {
      kv_copy_in_async(a.kv, b, N, sc);
      *top = __ldcg(a.kv.free_top + b);
    } else {
      kv_copy_in(a.kv, b, N, sc, 0, kThreads);
    }
  }
  if (N * K <= kTailTokens) {
    const int32_t *tok = a.tokens + static_cast<size_t>(b) * N * K;
    for (int i = tid; i < N * K; i += kThreads) cp_async4(sm.tok + i, tok + i);
  }
  return tid < N ? __ldcg(a.out.log_weights + static_cast<size_t>(b) * N + tid) : 0.f;
}

__device__ __forceinline__ void tail_prefetch_stack(const StepArgs &a, int b, int top,
                                                    const KvScratch &sc) {
  if (a.use_kv && sc.rc) kv_copy_stack_async(a.kv, b, top, sc);
}

// A prompt's weights once every particle's increment is known: thread i < N
// holds lwf = the incoming log-weight plus this step's increment (float-float,
// unrounded); sm.tab holds the 2^(j/64) table; key = resample_key(seed, step,
// b, N).  Normalisation, ESS, systematic resampling (ancestors in sm.anc) and
// the emission of each particle's K drafted tokens, taken from its ancestor;
// the bonus slot of each output is the caller's.  With `sc` (the staged KV
// state), kv_prepare also runs: on warps 1.. while warp 0 takes the weights
// (N <= 32), else after them.  All threads of the CTA call it, after
// tail_prefetch; all get whether the prompt resampled.
__device__ bool prompt_weights(const StepArgs &a, int b, TailSmem &sm, ff lwf, ResampleKey key,
                               const KvScratch *sc) {
  const int N = a.N, K = a.K;
  const int tid = threadIdx.x;
  const bool small = N <= 32;
  const bool tok_staged = N * K <= kTailTokens;
  __shared__ int s_res;
  const bool valid = tid < N;
  const int part = b * N + tid;
  if (tid == 0) kv_prepare_init(sm.ks, a.use_kv ? a.kv.T : 0);
  cp_async_wait_all();  // this thread's staged copies
  __syncthreads();      // everyone's: sm.tok, the KV stage; and sm.tab
  // with N <= 32, warp 0 alone does the weights (shuffles, no CTA barrier)
  if (small ? tid < 32 : true) {
    const ResampleResult rr =
        small ? normalise_resample_warp(N, lwf, valid, a.ess_frac, key, a.ws.status, sm.anc, sm.c,
                                        sm.tab)
              : normalise_resample(N, lwf, valid, a.ess_frac, key, a.ws.status, sm.anc, sm.c,
                                   sm.red, sm.tab);
    if (valid) {
      const int anc = sm.anc[tid];
      a.out.log_weights[part] = rr.resampled ? 0.f : lwf.hi;
      a.out.ancestors[part] = anc;
      int32_t *dst = a.out.tokens_out + static_cast<size_t>(part) * (K + 1);
      if (tok_staged) {
        const int *srcp = sm.tok + anc * K;
#pragma unroll 4
        for (int k = 0; k < K; ++k) dst[k] = srcp[k];
      } else {
        const int32_t *srcp = a.tokens + static_cast<size_t>(b * N + anc) * K;
#pragma unroll 4
        for (int k = 0; k < K; ++k) dst[k] = srcp[k];
      }
    }
    if (tid == 0) {
      a.out.ess[b] = rr.ess;
      a.out.resampled[b] = rr.resampled ? 1 : 0;
      s_res = rr.resampled ? 1 : 0;
    }
  } else if (sc) {
    kv_prepare(a.kv, b, N, *sc, sm.ks, 32, kThreads - 32);
  }
  __syncthreads();
  if (!small && sc) kv_prepare(a.kv, b, N, *sc, sm.ks, 0, kThreads);  // published by the remap's barrier
  return s_res != 0;
}

// The prompt's tail with every particle's weight and bonus token known
// (sm.bonus[i]: particle i's): prompt_weights, the bonus slots, and the KV
// remap with append.
__device__ void prompt_tail(const StepArgs &a, int b, TailSmem &sm, ff lwf, ResampleKey key,
                            const KvScratch &sc) {
  const int N = a.N, K = a.K;
  const int tid = threadIdx.x;
  const bool res = prompt_weights(a, b, sm, lwf, key, a.use_kv ? &sc : nullptr);
  if (tid < N) {
    a.out.tokens_out[static_cast<size_t>(b * N + tid) * (K + 1) + K] = sm.bonus[sm.anc[tid]];
  }
  if (a.use_kv) kv_remap_append(a.kv, b, N, sm.anc, res, K + 1, a.ws, sm.ks, sc, true, true);
}

// Runs in tail_kernel, launched with programmatic dependent launch while the
// row combine still runs.  The KV state, the incoming log-weights and the
// drafted tokens were all written before this step's first kernel, so they
// are read before waiting for the combine; only the row results are read
// after.  The increment is summed in float-float from the rows' results (a
// log-sum-exp row's result holds its value as a float pair, head and tail).
__device__ void smc_tail(const StepArgs &a, int b, TailSmem &sm, int *dyn, bool kv_staged) {
  const int N = a.N, K = a.K, rpp = 2 * K + 1;
  const int tid = threadIdx.x;
  const KvScratch sc = a.use_kv ? kv_scratch(a.kv, b, N, a.ws, dyn, kv_staged) : KvScratch{};
  int top = 0;
  const float lw0 = tail_prefetch(a, b, sm, sc, &top);
  tail_prefetch_stack(a, b, top, sc);
  const ResampleKey key = resample_key(a.seed, a.step, b, N);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the next step's rows
  ff lwf{0.f, 0.f};
  if (tid < N) {
    const int part = b * N + tid;
    const RowResult *r = a.ws.results + static_cast<size_t>(part) * rpp;
    const float4 rb = __ldcg(reinterpret_cast<const float4 *>(r + K));
    ff delta{0.f, 0.f};
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
      const float4 rp = __ldcg(reinterpret_cast<const float4 *>(r + k));
      const float4 rq = __ldcg(reinterpret_cast<const float4 *>(r + K + 1 + k));
      const ff lp = ff_sub_x(ff{rp.y, 0.f}, ff{rp.x, rp.z});  // log p of the drafted token
      const ff lq = ff_sub_x(ff{rq.y, 0.f}, ff{rq.x, rq.z});  // log q of it
      delta = ff_add_x(delta, ff_sub_x(ff_mul_fx(lp, a.alpha), lq));
    }
    if (a.alpha != 1.f) {
      delta = ff_add_x(delta, ff_sub_x(ff{rb.z, 0.f}, ff_mul_fx(ff{rb.x, 0.f}, a.alpha)));
    }
    if (a.potential) delta = ff_add_x(delta, ff{__ldcg(a.potential + part), 0.f});
    sm.bonus[tid] = __float_as_int(rb.w);
    lwf = ff_add_x(ff{lw0, 0.f}, delta);
  }
  prompt_tail(a, b, sm, lwf, key, sc);
}

__device__ void sps_tail(const StepArgs &a, int b, TailSmem &sm) {
  const int K = a.K, rpp = 2 * K + 1;
  const int tid = threadIdx.x;
  const RowResult *r = a.ws.results + static_cast<size_t>(b) * rpp;
  int cand = 0x7fffffff;
  if (tid < K) {
    const float4 rp = __ldcg(reinterpret_cast<const float4 *>(r + tid));
    const float4 rq = __ldcg(reinterpret_cast<const float4 *>(r + K + 1 + tid));
    const float ratio = expf((rp.y - rp.x) - (rq.y - rq.x));
    const float u = philox_uniform(a.seed, a.step, b, tid, SMC_PURPOSE_ACCEPT);
    if (!(u < ratio)) cand = tid;
  }
  int j = block_min_i(cand, sm.ired);
  if (j > K) j = K;
  const int bonus = __float_as_int(__ldcg(reinterpret_cast<const float4 *>(r + K)).w);
  if (tid <= K) {
    int v = -1;
    if (tid < j) v = a.tokens[static_cast<size_t>(b) * K + tid];
    else if (tid == j && j == K) v = bonus;
    a.out.tokens_out[static_cast<size_t>(b) * (K + 1) + tid] = v;
  }
  if (tid == 0) {
    a.out.n_emitted[b] = j + 1;
    a.ws.sps_rej[b] = j < K ? j : -1;
  }
}

// ---------------------------------------------------------------------------
// The row kernel.
// ---------------------------------------------------------------------------
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) step_rows_kernel(const StepArgs a) {
  using Tr = LogitTraits<T>;
  using G = ChunkGeom<T>;
  constexpr int EPT = G::kEPT;
  constexpr int CH = G::kCH;
  constexpr int ESZ = G::kESZ;

  __shared__ float s_red[2 * kWarps];
  __shared__ float2 s_ff[kWarps];
  __shared__ float2 s_tab[64];
  __shared__ int s_int[2 * kWarps];
  __shared__ int s_last;
  __shared__ ff s_target;
  __shared__ int s_sel_chunk;
  __shared__ float s_sel_m;

  const int tid = threadIdx.x;
  const int work = blockIdx.x;
  const int row = work / a.nch;
  const int chunk = work - row * a.nch;
  const int rpp = 2 * a.K + 1;
  const int part = row / rpp;
  const int j = row - part * rpp;
  const bool is_bonus = j == a.K;
  const char *rowp = j <= a.K
      ? a.target + (static_cast<size_t>(part) * (a.K + 1) + j) * static_cast<size_t>(a.V) * ESZ
      : a.draft + (static_cast<size_t>(part) * a.K + (j - a.K - 1)) * static_cast<size_t>(a.V) * ESZ;
  const int64_t c0 = static_cast<int64_t>(chunk) * CH;
  const int n_valid = static_cast<int>(min(static_cast<int64_t>(CH), a.V - c0));

  // ---- stream the chunk and reduce it -------------------------------------
  float x[EPT];
  load_chunk<T, VEC>(rowp + c0 * ESZ, n_valid, x);
  stage_exp2_table(s_tab);  // read by the bonus sums and by the row combine

  float m = kNegInf;
#pragma unroll
  for (int e = 0; e < EPT; ++e) m = fmaxf(m, x[e]);
  const float mc = block_max(m, s_red);  // chunk max: the reference of its sums
  const bool finite_ref = mc > kNegInf && mc < -kNegInf;

  float s = 0.f;
  ff S{0.f, 0.f};
  const float l2s = a.tscale * kLog2e;  // log2(e) of the scaled logits
  if (!is_bonus) {
    if (finite_ref) {
      const float mb = mc * l2s;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < EPT; e += 2) {
        s0 += fast_exp2(fmaf(x[e], l2s, -mb));
        s1 += fast_exp2(fmaf(x[e + 1], l2s, -mb));
      }
      s = s0 + s1;            // NaN logits propagate here and are reported at combine
    } else if (mc == -kNegInf) {
      s = __int_as_float(0x7fc00000);  // a +inf logit: NaN marks the row
    }
  } else {
    bool bad = false;
#pragma unroll
    for (int e = 0; e < EPT; ++e) bad |= !(x[e] < -kNegInf);  // NaN or +inf
    if (bad) raise_status(a.ws.status, SMC_DEV_NONFINITE);
    if (finite_ref) {
      const float mb = mc * l2s;
      const bool need_fast = a.bonus_lse;
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        ff_accum(S, weight_term(x[e], mc, a.balpha, s_tab));
        if (need_fast) s += fast_exp2(fmaf(x[e], l2s, -mb));
      }
    }
    S = ff_norm(S);
  }
  s = block_sum_f(s, s_red);
  if (is_bonus) S = block_ff_sum(S, s_ff);
  if (tid == 0) {
    a.ws.partials[work] = RowPartial{mc, s, S.hi, S.lo};
    __threadfence();
    const unsigned t = atomicAdd(&a.ws.row_ticket[row], 1u);
    s_last = t == static_cast<unsigned>(a.nch - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of the row: combine the chunk partials ----------------------
  __threadfence();
  if (tid == 0) a.ws.row_ticket[row] = 0u;
  const RowPartial *pp = a.ws.partials + static_cast<size_t>(row) * a.nch;
  const int lane = tid & 31, warp = tid >> 5;
  if (!is_bonus) {
    if (warp == 0) {
      float M = kNegInf;
      for (int c = lane; c < a.nch; c += 32) M = fmaxf(M, __ldcg(&pp[c].m));
      M = warp_max(M);
      float sum = 0.f;
      for (int c = lane; c < a.nch; c += 32) {
        const float cm = __ldcg(&pp[c].m), cs = __ldcg(&pp[c].s);
        if (cm > kNegInf) sum += cs * expf(a.tscale * (cm - M));
        else if (cs != 0.f) sum += cs;  // NaN marker of a chunk holding +inf
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        unsigned bits = 0;
        float g = __int_as_float(0x7fc00000);
        if (M == kNegInf) bits |= SMC_DEV_EMPTY_ROW;
        else if (!(sum < -kNegInf) || M == -kNegInf) bits |= SMC_DEV_NONFINITE;
        const ff lse = row_lse(a.tscale, M, sum, s_tab);
        const int k = j < a.K ? j : j - a.K - 1;
        const int tok = a.tokens[static_cast<size_t>(part) * a.K + k];
        if (tok < 0 || tok >= a.V) bits |= SMC_DEV_BAD_TOKEN;
        else g = a.tscale * Tr::scalar(rowp, tok);
        if (bits) raise_status(a.ws.status, bits);
        a.ws.results[row] = RowResult{lse.hi, g, lse.lo, -1};  // lse as head and tail
      }
    }
  } else {
    // bonus row: float-float mass per chunk in absolute units (reference M),
    // then the inverse-CDF draw: which chunk, then which element.
    const float alpha = a.balpha;
    if (warp == 0) {
      float M = kNegInf;
      for (int c = lane; c < a.nch; c += 32) M = fmaxf(M, __ldcg(&pp[c].m));
      M = warp_max(M);
      const bool ok = M > kNegInf && M < -kNegInf;
      auto chunk_mass = [&](int c, ff *val, ff *f) {
        const float cm = __ldcg(&pp[c].m);
        if (ok && cm > kNegInf) {
          *f = ff_norm(weight_term(cm, M, alpha, s_tab));  // exp(alpha (m_c - M))
          *val = ff_mul(ff{__ldcg(&pp[c].shi), __ldcg(&pp[c].slo)}, *f);
        }
      };
      float fast = 0.f;
      ff total{0.f, 0.f};
      for (int c0w = 0; c0w < a.nch; c0w += 32) {
        const int c = c0w + lane;
        ff val{0.f, 0.f}, f{1.f, 0.f};
        if (c < a.nch) {
          chunk_mass(c, &val, &f);
          const float cm = __ldcg(&pp[c].m);
          if (ok && cm > kNegInf) fast += __ldcg(&pp[c].s) * expf(a.tscale * (cm - M));
        }
        total = ff_add(total, warp_ff_sum(val));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) fast += __shfl_xor_sync(0xffffffffu, fast, o);
      const float u = philox_uniform(a.seed, a.step, part, a.bonus_position, a.bonus_purpose);
      ff rem{0.f, 0.f};
      const int sel = ok ? warp_find_chunk(a.nch, ff_mul_f(total, u), chunk_mass, &rem) : -1;
      if (lane == 0) {
        s_sel_chunk = sel;
        s_sel_m = sel >= 0 ? __ldcg(&pp[sel].m) : 0.f;
        s_target = rem;
        float lse, lse_alpha;
        if (ok) {
          lse_alpha = ff_add(two_prod(alpha, M), ff_log(total, s_tab)).hi;
          lse = a.bonus_lse ? row_lse(a.tscale, M, fast, s_tab).hi : lse_alpha;
        } else {
          lse = lse_alpha = M == kNegInf ? kNegInf : __int_as_float(0x7fc00000);
          raise_status(a.ws.status, M == kNegInf ? SMC_DEV_EMPTY_ROW : SMC_DEV_NONFINITE);
        }
        a.ws.results[row] = RowResult{lse, 0.f, lse_alpha, -1};
      }
    }
    __syncthreads();
    const int sel = s_sel_chunk;
    int tok = -1;
    if (sel >= 0) {
      const float cm = s_sel_m;
      const int64_t sc0 = static_cast<int64_t>(sel) * CH;
      const int len = static_cast<int>(min(static_cast<int64_t>(CH), a.V - sc0));
      tok = block_select_in_chunk(
          sc0, len, s_target,
          [&](int64_t i) { return weight_term(Tr::scalar(rowp, i), cm, alpha, s_tab); },
          s_ff, s_int);
    }
    if (tid == 0) {
      a.ws.results[row].tok = tok;
      if (a.mode == 2) a.out.tokens_out[part] = tok;
    }
  }
}

// ---------------------------------------------------------------------------
// Streaming row kernel (shapes whose rows are 16-byte aligned).
//
// Persistent CTAs, two per SM, each with 8 consumer warps and 1 producer
// warp.  The producer claims work from two atomic queues, alternating: items
// of G consecutive 32 KB chunks of one target or draft row (the log-sum-exp
// rows), and single chunks of the bonus rows (target row K, whose sampling
// weights cost far more arithmetic per logit).  It streams each chunk into a
// ring of kStages shared-memory slots with one bulk copy (cp.async.bulk,
// completion counted in bytes on the slot's mbarrier), as far ahead as the
// ring allows.  Consumer warp w owns the contiguous eighth w of every chunk:
// it copies its part to registers, releases the slot, and folds the logits
// into a running (max, sum of exp) pair per lane (MUFU ex2, packed f32x2
// arithmetic); at an item's end the warp writes one partial per (item,
// warp).  For a bonus chunk the warp instead sums the sampling weights of
// its range relative to the range's max in float-float (BonusPairSum) and
// writes one unit partial.  No CTA-wide barrier after set-up; every wait is
// bounded and reports SMC_DEV_TIMEOUT when it gives up.
// ---------------------------------------------------------------------------
constexpr int kStages = 3;
constexpr int kChunkBytes = 32768;      // one ring slot: 16384 bf16 or 8192 fp32 logits
constexpr int kConsumerWarps = 8;
constexpr int kStreamThreads = (kConsumerWarps + 1) * 32;
constexpr uint32_t kWaitLimit = 1u << 18;  // polls; each may suspend up to 20 us

enum : int { kSlotFirst = 1, kSlotLast = 2, kSlotEnd = 4 };

// item: the index, within its row, of the work item the chunk belongs to
// (where the item's partials go); for bonus rows, the chunk itself.
struct SlotMeta { int row, part, j, chunk, n, flags, item, pad; };

// Logits per ring slot and per 16-byte vector of the streaming kernel.
template <typename T> struct StreamGeom {
  static constexpr int kESZ = sizeof(T) == 4 ? 4 : 2;
  static constexpr int kEPV = 16 / kESZ;
  static constexpr int kCH = kChunkBytes / kESZ;
  static constexpr int kWCH = kCH / kConsumerWarps;  // logits of one consumer warp's range
};

// Non-bonus rows are numbered rf = particle * 2K + (target positions 0..K-1,
// then draft positions 0..K-1).  Rows rf < R1 are cut into ipr items of G
// chunks; the last rows, rf >= R1, into single-chunk items, so that the work
// queue ends in small pieces and the CTAs run out of work at nearly the same
// time.
struct StreamArgs {
  StepArgs a;
  int snch;           // ring-slot chunks per row: ceil(V / StreamGeom<T>::kCH)
  float wspan;        // 40 / balpha: logits further below a range's max weigh e^-40
  int G;              // chunks per work item of a non-bonus row rf < R1
  int ipr;            // work items per non-bonus row rf < R1
  int R1;             // non-bonus rows cut into G-chunk items
  int n_items1;       // R1 * ipr: the queue's G-chunk items come first
  int n_fast_items;   // all non-bonus items
  int n_bonus_items;  // bonus rows * snch (one chunk per item)
  int signal_rows;    // nonzero: each CTA adds 1 to ws.rows_done once its partials are out
  int row_grid;       // CTAs of the streaming kernel
  unsigned long long *clk;  // step-clock hook (smc_set_step_clock), or null
  unsigned *clk_ctr;
  int clk_cap;
};

// Partial slots (work items) of non-bonus row rf.
__host__ __device__ __forceinline__ int items_of_row(const StreamArgs &sa, int rf) {
  return rf < sa.R1 ? sa.ipr : sa.snch;
}

constexpr size_t stream_dyn_smem() {
  return static_cast<size_t>(kStages) * kChunkBytes + 2 * kStages * sizeof(uint64_t) +
         kStages * sizeof(SlotMeta);
}


template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 2) row_stream_kernel(const StreamArgs sa) {
  using Gm = StreamGeom<T>;
  constexpr int EPV = Gm::kEPV;                       // logits per 16-byte vector
  constexpr int CH = Gm::kCH;                         // logits per chunk
  constexpr int ESZ = Gm::kESZ;
  constexpr int WCH = Gm::kWCH;                       // logits per warp range
  constexpr int VPL = WCH / EPV / 32;                 // vectors per lane per chunk
  constexpr float kInf = -kNegInf;
  const StepArgs &a = sa.a;

  extern __shared__ __align__(128) unsigned char dyn_smem[];
  uint4 *bufs = reinterpret_cast<uint4 *>(dyn_smem);
  uint64_t *full = reinterpret_cast<uint64_t *>(dyn_smem + kStages * kChunkBytes);
  uint64_t *empty = full + kStages;
  SlotMeta *meta = reinterpret_cast<SlotMeta *>(empty + kStages);
  __shared__ float s_th[64], s_tl[64];
  __shared__ unsigned s_exited;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rpp = 2 * a.K + 1;

  // Launched with programmatic dependent launch.  The producer reads only the
  // logits and claims work from this call's copy of the queue counters, so it
  // starts its copies at once; the consumers start at once in the plain step
  // and wait for the previous grid elsewhere (see below).
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init_fence();
    s_exited = 0u;
  }
  stage_exp2_split(s_th, s_tl);
  __syncthreads();  // the only CTA-wide barrier

  // ---- producer warp -----------------------------------------------------------
  // Work comes from two queues: items of G chunks of the non-bonus rows, and
  // single chunks of the bonus rows (whose weights cost far more to compute).
  // The producer interleaves them in about the proportion of the whole step
  // (2K non-bonus chunks per bonus chunk), so that every CTA mixes
  // streaming-bound and arithmetic-bound chunks evenly; bonus chunks are
  // taken 8/7 as often, so that their queue drains before the other and the
  // kernel ends on cheap chunks.
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const int rest = rpp - 1;  // non-bonus rows per particle
      int row = 0, first = 0, chunk = 0, end = 0, item = 0;
      int fast_chunks = 0, n_bonus = 0;
      bool have = false, fast_done = sa.n_fast_items == 0, bonus_done = sa.n_bonus_items == 0;
      // each queue's next claim is issued one item ahead, so that the
      // atomic's round trip overlaps the copies of the current item
      unsigned next_fast = fast_done ? 0u : atomicAdd(&a.ws.work_counter[0], 1u);
      unsigned next_bonus = bonus_done ? 0u : atomicAdd(&a.ws.work_counter[1], 1u);
      // near the end of the queues (bonus queue empty, under two fast items
      // per CTA left) at most two chunks stay in flight: the last items go to
      // whichever CTAs are ready, and each CTA has less queued when they run dry
      const unsigned tail_from = static_cast<unsigned>(
          max(0, sa.n_fast_items - 2 * static_cast<int>(gridDim.x)));
      for (int i = 0;; ++i) {
        const int slot = i % kStages;
        if (i >= kStages &&
            !mbar_wait(&empty[slot], static_cast<uint32_t>(i / kStages - 1) & 1u, kWaitLimit)) {
          raise_status(a.ws.status, SMC_DEV_TIMEOUT);
          meta[slot].flags = kSlotEnd;  // consumers time out on this slot too
          break;
        }
        if (i >= 2 && bonus_done && next_fast >= tail_from) {
          // the chunk issued two iterations ago has been consumed (its slot is
          // not refilled before the next iteration, so the parity is exact)
          const int i2 = i - 2;
          if (!mbar_wait(&empty[i2 % kStages], static_cast<uint32_t>(i2 / kStages) & 1u,
                         kWaitLimit)) {
            raise_status(a.ws.status, SMC_DEV_TIMEOUT);
            meta[slot].flags = kSlotEnd;
            break;
          }
        }
        while (!have || chunk >= end) {
          have = false;
          if (fast_done && bonus_done) break;
          const bool take_bonus =
              !bonus_done && (fast_done || n_bonus * 2 * a.K * 7 < fast_chunks * 8);
          if (take_bonus) {
            const unsigned id = next_bonus;
            if (id >= static_cast<unsigned>(sa.n_bonus_items)) { bonus_done = true; continue; }
            next_bonus = atomicAdd(&a.ws.work_counter[1], 1u);
            ++n_bonus;
            const int part = static_cast<int>(id) / sa.snch;
            row = part * rpp + a.K;
            first = static_cast<int>(id) - part * sa.snch;
            end = first + 1;
            item = first;
          } else {
            const unsigned id = next_fast;
            if (id >= static_cast<unsigned>(sa.n_fast_items)) { fast_done = true; continue; }
            next_fast = atomicAdd(&a.ws.work_counter[0], 1u);
            int rf;
            if (static_cast<int>(id) < sa.n_items1) {
              rf = static_cast<int>(id) / sa.ipr;
              item = static_cast<int>(id) - rf * sa.ipr;
              first = item * sa.G;
              end = min(first + sa.G, sa.snch);
            } else {
              const int i2 = static_cast<int>(id) - sa.n_items1;
              const int r2 = i2 / sa.snch;
              rf = sa.R1 + r2;
              item = first = i2 - r2 * sa.snch;
              end = first + 1;
            }
            fast_chunks += end - first;
            const int part = rf / rest, jj = rf - part * rest;
            row = part * rpp + (jj < a.K ? jj : jj + 1);
          }
          chunk = first;
          have = true;
        }
        if (!have) {
          SlotMeta &mt = meta[slot];
          mt.row = -1; mt.part = 0; mt.j = 0; mt.chunk = 0; mt.n = 0; mt.flags = kSlotEnd;
          mbar_arrive(&full[slot]);
          // the queues are drained: the dependent kernel may launch, so that its
          // CTAs take SMs as this kernel's CTAs leave them.  (After this grid's
          // own wait, so that it never launches before the previous step ends.)
          asm volatile("griddepcontrol.wait;" ::: "memory");
          asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
          // the queues are drained, so the step's tail comes within a few
          // microseconds: bring a prompt's KV state into L2 for it
          if (a.mode == 0 && a.use_kv) {
            for (int b = static_cast<int>(blockIdx.x); b < a.B; b += static_cast<int>(gridDim.x)) {
              kv_prefetch_l2(a.kv, b, a.N);
            }
          }
          break;
        }
        const int64_t c0 = static_cast<int64_t>(chunk) * CH;
        const int n = static_cast<int>(min(static_cast<int64_t>(CH), a.V - c0));
        SlotMeta &mt = meta[slot];
        mt.row = row;
        mt.part = row / rpp;
        mt.j = row - mt.part * rpp;
        mt.chunk = chunk;
        mt.n = n;
        mt.flags = (chunk == first ? kSlotFirst : 0) | (chunk + 1 == end ? kSlotLast : 0);
        mt.item = item;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(n * ESZ));
        bulk_copy_g2s(bufs + static_cast<size_t>(slot) * (kChunkBytes / 16),
                      row_base<T>(a, row) + c0 * ESZ, static_cast<uint32_t>(n * ESZ), &full[slot]);
        ++chunk;
      }
    }
    return;
  }

  // ---- consumer warps --------------------------------------------------------
  if (sa.clk && blockIdx.x == 0 && tid == 0) {  // the step-clock hook: this step starts
    const unsigned k = atomicAdd(sa.clk_ctr, 1u);
    if (k < static_cast<unsigned>(sa.clk_cap)) sa.clk[k] = global_timer_ns();
  }
  // The consumers write only what the previous call's kernels have finished
  // reading once that call let this grid launch (an SMC step's prompt kernel
  // once the weights are in, or its tail once it has waited for the nucleus
  // and the row combine; a verify's residual retry pass; the draft sampler's
  // row combine once it has waited for its row pass): the (item, warp)
  // partials and this call's copy of the bonus partials and counters
  // (consecutive calls alternate copies).  So they stream at once, and wait
  // for the previous call only before they let the next kernels launch.
  const float l2s = a.tscale * kLog2e;  // log2(e) of the scaled logits
  float m_t = kNegInf, s_t = 0.f;  // this lane's running (max, sum exp) over the item
  for (int i = 0;; ++i) {
    const int slot = i % kStages;
    const uint32_t par = static_cast<uint32_t>(i / kStages) & 1u;
    if (!mbar_wait(&full[slot], par, kWaitLimit)) {
      raise_status(a.ws.status, SMC_DEV_TIMEOUT);
      break;
    }
    const SlotMeta mt = meta[slot];
    if (mt.flags & kSlotEnd) break;
    const int row = mt.row;
    const int part = mt.part;
    const int j = mt.j;
    const bool is_bonus = j == a.K;
    const bool fast = !is_bonus || a.bonus_lse;
    if (mt.flags & kSlotFirst) { m_t = kNegInf; s_t = 0.f; }

    // this warp's range of the chunk: logits [warp*WCH, (warp+1)*WCH).  A
    // vector past the chunk's valid logits reads as -inf.
    constexpr uint32_t kNegInfBits = sizeof(T) == 4 ? 0xff800000u : 0xff80ff80u;
    uint4 q[VPL];
    const uint4 *buf = bufs + static_cast<size_t>(slot) * (kChunkBytes / 16) + warp * (WCH / EPV);
    if (mt.n == CH) {  // a full chunk: every vector is valid
#pragma unroll
      for (int v = 0; v < VPL; ++v) q[v] = buf[v * 32 + lane];
    } else {
      const int wbase = warp * WCH;
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const bool ok = wbase + (v * 32 + lane) * EPV < mt.n;
        q[v] = ok ? buf[v * 32 + lane]
                  : make_uint4(kNegInfBits, kNegInfBits, kNegInfBits, kNegInfBits);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done reading the slot

    // the words of my vectors: 2 bf16 or 1 fp32 logit each
    const uint32_t *wd = reinterpret_cast<const uint32_t *>(q);
    constexpr int NW = VPL * 4;
    // chunk max; for the bonus row NaN-propagating, since a NaN or +inf
    // anywhere in it is an error
    float cm;
    if (sizeof(T) == 4) {
      cm = __uint_as_float(wd[0]);
      if (is_bonus) {
#pragma unroll
        for (int k = 1; k < NW; ++k) cm = fmax_nan(cm, __uint_as_float(wd[k]));
      } else {
#pragma unroll
        for (int k = 1; k < NW; ++k) cm = fmaxf(cm, __uint_as_float(wd[k]));
      }
    } else {
      uint32_t mw = wd[0];
      if (is_bonus) {
#pragma unroll
        for (int k = 1; k < NW; ++k) mw = bmax2_nan(mw, wd[k]);
        cm = fmax_nan(bf16_lo(mw), bf16_hi(mw));
      } else {
#pragma unroll
        for (int k = 1; k < NW; ++k) mw = bmax2(mw, wd[k]);
        cm = fmaxf(bf16_lo(mw), bf16_hi(mw));
      }
    }
    if (is_bonus && !(cm < kInf)) {
      raise_status(a.ws.status, SMC_DEV_NONFINITE);
      cm = kNegInf;  // the outputs are unspecified now; keep the arithmetic finite
    }
    if (fast) {
      if (cm > m_t) {
        if (m_t > kNegInf) s_t *= fast_exp2((m_t - cm) * l2s);
        m_t = cm;
      }
      if (m_t > kNegInf && m_t < kInf) {
        const float mb = m_t * l2s;
        const unsigned long long l2 = f2pack(l2s, l2s), nmb = f2pack(-mb, -mb);
        unsigned long long acc = 0ull;
        if (sizeof(T) == 4) {
#pragma unroll
          for (int k = 0; k < NW; k += 2) {
            float y0, y1;
            f2unpack(fma2(f2pack(__uint_as_float(wd[k]), __uint_as_float(wd[k + 1])), l2, nmb), y0, y1);
            acc = add2(acc, f2pack(fast_exp2(y0), fast_exp2(y1)));
          }
        } else {
#pragma unroll
          for (int k = 0; k < NW; ++k) {
            float y0, y1;
            f2unpack(fma2(f2pack(bf16_lo(wd[k]), bf16_hi(wd[k])), l2, nmb), y0, y1);
            acc = add2(acc, f2pack(fast_exp2(y0), fast_exp2(y1)));
          }
        }
        float a0, a1;
        f2unpack(acc, a0, a1);
        s_t += a0 + a1;  // NaN logits propagate and are reported at the row combine
      } else if (m_t == kInf) {
        s_t = __int_as_float(0x7fc00000);
      }
    }
    if (is_bonus) {
      // this unit's reference is its max logit; the weights relative to it
      // are summed in float-float
      const float ref = warp_max(cm);
      ff usum{0.f, 0.f};
      int flag = 0;
      if (ref > kNegInf) {
        BonusPairSum bs;
        if (bs.init(ref, a.balpha, sa.wspan)) {
          if (sizeof(T) == 4) {
            // fp32 logits: the general path only (the power-sampling case)
#pragma unroll
            for (int k = 0; k < NW; k += 2)
              bs.add<false, false>(__uint_as_float(wd[k]), __uint_as_float(wd[k + 1]), s_th, s_tl);
          } else if (a.balpha == 1.f && BonusPairSum::fast_diff_ok(ref, sa.wspan)) {
#pragma unroll
            for (int k = 0; k < NW; ++k)
              bs.add<true, true>(bf16_lo(wd[k]), bf16_hi(wd[k]), s_th, s_tl);
          } else {
#pragma unroll
            for (int k = 0; k < NW; ++k)
              bs.add<false, false>(bf16_lo(wd[k]), bf16_hi(wd[k]), s_th, s_tl);
          }
          usum = warp_ff_sum(bs.total());
        } else {
          flag = 1;  // ref too large for the clamp: the finish kernel sums this unit
        }
      }
      if (lane == 0) {
        a.ws.bonus_part[(static_cast<size_t>(part) * sa.snch + mt.chunk) * kConsumerWarps + warp] =
            make_int4(__float_as_int(ref), __float_as_int(usum.hi), __float_as_int(usum.lo), flag);
      }
    }

    if (!(mt.flags & kSlotLast)) continue;

    // ---- end of this warp's share of a work item: its partial -----------------
    if (fast) {
      const float M = warp_max(m_t);
      float contrib = 0.f;
      if (m_t > kNegInf && M < kInf) contrib = s_t * fast_exp2((m_t - M) * l2s);
      else if (s_t != 0.f) contrib = s_t;  // NaN marker
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) contrib += __shfl_xor_sync(0xffffffffu, contrib, o);
      if (lane == 0) {
        a.ws.item_part[(static_cast<size_t>(row) * sa.snch + mt.item) * kConsumerWarps + warp] =
            make_float2(M, contrib);
      }
    }
  }

  // ---- consumer exit: publish the CTA's partials; reset the work counters ----
  // Each warp's lane 0 wrote the warp's partials; the CTA-scope acquire-release
  // adds order them before the last warp's gpu-scope release of rows_done,
  // which the plain step's particle kernel waits on.
  if (lane == 0) {
    if (atom_add_acq_rel_cta(&s_exited, 1u) == kConsumerWarps - 1) {
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous call has ended
      if (sa.signal_rows) add_release_gpu(a.ws.rows_done, 1u);
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      __threadfence();
      if (atomicAdd(a.ws.exit_counter, 1u) == gridDim.x - 1) {
        a.ws.work_counter[0] = 0u;
        a.ws.work_counter[1] = 0u;
        *a.ws.exit_counter = 0u;
      }
    }
  }
}


// ---------------------------------------------------------------------------
// CTA-wide inverse-CDF selection inside the range [r0, r0 + len) of a row, in
// exact fixed-point arithmetic: the first element with a positive weight
// weight_fixed(l, ref) whose inclusive prefix exceeds `target`; if none does
// (the target at or past the range's total), the last positive element; -1
// with no mass.  Thread t holds the one 16-byte vector [t*EPT, (t+1)*EPT)
// (EPT logits); r0 and len are multiples of EPT, len <= kThreads * EPT, and
// the row is 16-byte aligned.  All threads must call it; all get the result.
// ---------------------------------------------------------------------------
template <typename T, int EPT>
__device__ int block_select_fixed(const char *rowp, int64_t r0, int len, long long target,
                                  float ref, float alpha, const float2 *tab,
                                  long long *s_ll, int *s_i) {
  using Tr = LogitTraits<T>;
  static_assert(EPT == Tr::kPerVec, "one 16-byte vector per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int beg = tid * EPT;
  long long w[EPT];
  long long part = 0;
  const bool have = beg < len;
  const uint4 v = have ? *reinterpret_cast<const uint4 *>(rowp + (r0 + beg) * StreamGeom<T>::kESZ)
                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    w[e] = have ? weight_fixed(Tr::at(v, e), ref, alpha, tab) : 0ll;
    part += w[e];
  }
  // block inclusive scan of the per-thread sums
  const long long incl_w = warp_incl_scan_ll(part);
  if (lane == 31) s_ll[warp] = incl_w;
  __syncthreads();
  long long base = 0;
  for (int k = 0; k < warp; ++k) base += s_ll[k];
  const long long incl = base + incl_w;
  int cand = 0x7fffffff, last = -1;
  long long run = incl - part;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    run += w[e];
    if (w[e] > 0) {
      last = beg + e;
      if (cand == 0x7fffffff && run > target) cand = beg + e;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  }
  if (lane == 0) {
    s_i[warp] = cand;
    s_i[kWarps + warp] = last;
  }
  __syncthreads();
  int c = 0x7fffffff, l = -1;
#pragma unroll
  for (int k = 0; k < kWarps; ++k) {
    c = min(c, s_i[k]);
    l = max(l, s_i[kWarps + k]);
  }
  __syncthreads();  // s_ll and s_i may be reused by the caller
  if (c == 0x7fffffff) c = l;
  return c < 0 ? -1 : static_cast<int>(r0 + c);
}

// ---------------------------------------------------------------------------
// A row's log-sum-exp pieces from the streaming kernel's (item, warp)
// partials, by an aligned group of G lanes: M the row's largest logit and S
// the fp32 sum of exp(tscale (l - M)) (NaN marks a NaN or +inf logit).  Every
// lane of the group gets both; all 32 lanes of the warp must call it (each
// group on its own row, or with act false).  rf: the row's non-bonus number,
// or -1 for a bonus row (one item a chunk).
// ---------------------------------------------------------------------------
template <int G>
__device__ __forceinline__ void group_row_stats(const StreamArgs &sa, int row, int rf, bool act,
                                                float *out_m, float *out_s) {
  constexpr float kInf = -kNegInf;
  const StepArgs &a = sa.a;
  const int sub = threadIdx.x & (G - 1);
  float lm = kNegInf, ls = 0.f;
  if (act) {
    const float2 *ip = a.ws.item_part + static_cast<size_t>(row) * sa.snch * kConsumerWarps;
    const int n_ip = (rf < 0 ? sa.snch : items_of_row(sa, rf)) * kConsumerWarps;
#pragma unroll 4
    for (int c = sub; c < n_ip; c += G) {
      const float2 pv = __ldcg(ip + c);
      if (pv.x > lm) {
        if (lm > kNegInf && pv.x < kInf) ls *= expf(a.tscale * (lm - pv.x));
        else if (pv.x == kInf) ls = 0.f;
        lm = pv.x;
      }
      if (pv.x > kNegInf && lm < kInf) ls += pv.y * expf(a.tscale * (pv.x - lm));
      else if (pv.y != 0.f) ls += pv.y;  // NaN marker
    }
  }
  float fM = lm;
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) fM = fmaxf(fM, __shfl_xor_sync(0xffffffffu, fM, o));
  float fS = (lm > kNegInf && fM < kInf) ? ls * expf(a.tscale * (lm - fM)) : ls;
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) fS += __shfl_xor_sync(0xffffffffu, fS, o);
  *out_m = fM;
  *out_s = fS;
}

__device__ __forceinline__ void fast_row_stats(const StreamArgs &sa, int row, int rf,
                                               float *out_m, float *out_s) {
  group_row_stats<32>(sa, row, rf, true, out_m, out_s);
}

// Where a bonus row's inverse-CDF draw falls, found by bonus_select_warp: the
// unit (-1 when the row has no mass), the remaining target inside it in the
// unit's own fixed-point scale, the unit's reference logit, and the row's
// log-sum-exps of tscale*l (lse) and of balpha*l (lse_alpha).
struct BonusSel { long long target; int sel; float ref; ff lse, lse_alpha; };

// Units whose largest logit was too large for the streaming kernel's clamp
// (flag set) are summed here instead, in exact fixed point, by one warp.
// Rare, so kept out of line: the draw's usual path stays short.
template <typename T>
__device__ __noinline__ void bonus_resum_flagged(const StreamArgs &sa, const char *rowp,
                                                 int4 *bp, int n_units, const float2 *tab) {
  using Tr = LogitTraits<T>;
  constexpr int CH = StreamGeom<T>::kCH;
  constexpr int WCH = StreamGeom<T>::kWCH;
  const int lane = threadIdx.x & 31;
  for (int q = 0; q < n_units; ++q) {
    const int4 pv = bp[q];
    if (pv.w == 0) continue;
    const float ref = __int_as_float(pv.x);
    const int c = q / kConsumerWarps, w = q - c * kConsumerWarps;
    const int64_t r0 = static_cast<int64_t>(c) * CH + static_cast<int64_t>(w) * WCH;
    const int len = static_cast<int>(min(static_cast<int64_t>(WCH), sa.a.V - r0));
    long long sum = 0;
    for (int i = lane; i < len; i += 32) {
      sum += weight_fixed(Tr::scalar(rowp, r0 + i), ref, sa.a.balpha, tab);
    }
    const ff v = fixed_to_ff(warp_sum_ll(sum));
    __syncwarp();
    if (lane == 0) bp[q] = make_int4(pv.x, __float_as_int(v.hi), __float_as_int(v.lo), 0);
    __syncwarp();
  }
  __threadfence_block();
}

// Unit selection for rows of more than 64 units, by one warp: masses
// computed on demand in blocks of 32, the total first, then the scan
// (warp_find_chunk).  Out of line, like the rare paths.
__device__ __noinline__ void bonus_select_long(const StreamArgs &sa, const int4 *bp,
                                               int n_units, float u, const float2 *tab, int *sel,
                                               float *out_m, ff *out_total, ff *rem) {
  constexpr float kInf = -kNegInf;
  const int lane = threadIdx.x & 31;
  const float alpha = sa.a.balpha;
  float M = kNegInf;
  for (int q = lane; q < n_units; q += 32) M = fmaxf(M, __int_as_float(bp[q].x));
  M = warp_max(M);
  const bool ok = M > kNegInf && M < kInf;
  auto unit_mass = [&](int q, ff *val, ff *f) {
    const int4 pv = bp[q];
    const float ref = __int_as_float(pv.x);
    if (ok && ref > kNegInf) {
      *f = ff_norm(weight_term(ref, M, alpha, tab));  // exp(alpha (ref - M))
      *val = ff_mul(ff{__int_as_float(pv.y), __int_as_float(pv.z)}, *f);
    }
  };
  ff total{0.f, 0.f};
  for (int q0 = 0; q0 < n_units; q0 += 32) {
    ff val{0.f, 0.f}, f{1.f, 0.f};
    if (q0 + lane < n_units) unit_mass(q0 + lane, &val, &f);
    total = ff_add(total, warp_ff_sum(val));
  }
  *sel = ok ? warp_find_chunk(n_units, ff_mul_f(total, u), unit_mass, rem) : -1;
  *out_m = M;
  *out_total = total;
}

// Stage 1 of a bonus-row draw, by one full warp (no CTA barrier), from the
// streaming kernel's unit sums: units are (chunk, warp) ranges of WCH
// logits in vocabulary order, each with its largest logit as reference and
// the float-float sum of its weights exp(balpha (l - ref)).  Which unit holds
// u times the total comes from a float-float scan of the units' masses (two
// units a lane for rows of at most 64 units, else bonus_select_long).  u is
// the draw's uniform (bonus_uniform).  fM and fS are the row's fast
// log-sum-exp pieces (used when alpha != 1).  With need_lse the row's
// log-sum-exps go to out->lse and out->lse_alpha.  Lane 0 writes *out.
__device__ __forceinline__ float bonus_uniform(const StepArgs &a, int part) {
  return philox_uniform(a.seed, a.step, part, a.bonus_position, a.bonus_purpose);
}

template <typename T>
__device__ void bonus_select_warp(const StreamArgs &sa, int part, const char *rowp, float u,
                                  float fM, float fS, bool need_lse, const float2 *tab,
                                  BonusSel *out) {
  constexpr float kInf = -kNegInf;
  constexpr unsigned kAll = 0xffffffffu;
  const StepArgs &a = sa.a;
  const int lane = threadIdx.x & 31;
  const float alpha = a.balpha;
  int4 *bp = a.ws.bonus_part + static_cast<size_t>(part) * sa.snch * kConsumerWarps;
  const int n_units = sa.snch * kConsumerWarps;
  int sel = -1;
  float M = kNegInf, ref = 0.f;
  ff total{0.f, 0.f}, rem{0.f, 0.f};
  if (n_units <= 64) {
    // units 2*lane and 2*lane + 1, adjacent in vocabulary order
    const int q0 = 2 * lane, q1 = q0 + 1;
    const int4 neg = make_int4(__float_as_int(kNegInf), 0, 0, 0);
    int4 p0 = q0 < n_units ? bp[q0] : neg, p1 = q1 < n_units ? bp[q1] : neg;
    if (__any_sync(kAll, (p0.w | p1.w) != 0)) {
      bonus_resum_flagged<T>(sa, rowp, bp, n_units, tab);
      p0 = q0 < n_units ? bp[q0] : neg;
      p1 = q1 < n_units ? bp[q1] : neg;
    }
    const float r0 = __int_as_float(p0.x), r1 = __int_as_float(p1.x);
    M = warp_max(fmaxf(r0, r1));
    const bool ok = M > kNegInf && M < kInf;
    ff v0{0.f, 0.f}, v1{0.f, 0.f}, f0{1.f, 0.f}, f1{1.f, 0.f};
    if (ok && r0 > kNegInf) {
      f0 = ff_norm(weight_term(r0, M, alpha, tab));  // exp(alpha (ref - M))
      v0 = ff_mul(ff{__int_as_float(p0.y), __int_as_float(p0.z)}, f0);
    }
    if (ok && r1 > kNegInf) {
      f1 = ff_norm(weight_term(r1, M, alpha, tab));
      v1 = ff_mul(ff{__int_as_float(p1.y), __int_as_float(p1.z)}, f1);
    }
    const ff pair = ff_add(v0, v1);
    const ff incl = warp_ff_incl_scan(pair);  // through unit q1
    total = shfl_ff(incl, 31);
    const ff excl = ff_sub(incl, pair);       // before unit q0
    const ff c0 = ff_add(excl, v0);           // through unit q0
    const ff target = ff_mul_f(total, u);
    const bool pos0 = v0.hi > 0.f, pos1 = v1.hi > 0.f;
    const bool hit0 = pos0 && ff_gt(c0, target), hit1 = pos1 && ff_gt(incl, target);
    const unsigned hits = __ballot_sync(kAll, hit0 || hit1);
    const unsigned any = __ballot_sync(kAll, pos0 || pos1);
    if (ok && any) {
      // the first unit whose prefix exceeds the target; past the total
      // (rounding), the last unit with mass, taken whole
      const int src = hits ? __ffs(hits) - 1 : 31 - __clz(any);
      const bool first_half = hits ? hit0 : !pos1;
      const bool h0 = __shfl_sync(kAll, first_half, src);
      const ff ex = h0 ? excl : c0;  // the chosen unit's exclusive prefix
      const ff val = h0 ? v0 : v1, f = h0 ? f0 : f1;
      const ff l_rem = hits ? ff_div(ff_sub(target, ex), f) : ff_div(val, f);
      rem = shfl_ff(l_rem, src);
      ref = __shfl_sync(kAll, h0 ? r0 : r1, src);
      sel = 2 * src + (h0 ? 0 : 1);
    }
  } else {
    bool flagged = false;
    for (int q = lane; q < n_units; q += 32) flagged |= bp[q].w != 0;
    if (__any_sync(kAll, flagged)) bonus_resum_flagged<T>(sa, rowp, bp, n_units, tab);
    bonus_select_long(sa, bp, n_units, u, tab, &sel, &M, &total, &rem);
    if (sel >= 0) ref = __int_as_float(bp[sel].x);
  }
  if (lane == 0) {
    const bool ok = M > kNegInf && M < kInf;
    out->sel = sel;
    out->target = ff_to_fixed(rem);
    out->ref = ref;
    if (!need_lse) {
      out->lse = out->lse_alpha = ff{0.f, 0.f};
      if (!ok) raise_status(a.ws.status, M == kNegInf ? SMC_DEV_EMPTY_ROW : SMC_DEV_NONFINITE);
    } else if (ok) {
      out->lse_alpha = ff_add(two_prod(alpha, M), ff_log(total, tab));
      out->lse = a.bonus_lse ? row_lse(a.tscale, fM, fS, tab) : out->lse_alpha;
    } else {
      const float v = M == kNegInf ? kNegInf : __int_as_float(0x7fc00000);
      out->lse = out->lse_alpha = ff{v, 0.f};
      raise_status(a.ws.status, M == kNegInf ? SMC_DEV_EMPTY_ROW : SMC_DEV_NONFINITE);
    }
  }
}

// Stage 2, by the whole CTA: the element of the selected unit, by an exact
// fixed-point rescan of its WCH logits (block_select_fixed); -1 when the row
// has no mass.  All threads must call it, with `s` visible to every thread;
// every thread gets the token.
template <typename T>
__device__ __forceinline__ int bonus_rescan(const StreamArgs &sa, const char *rowp,
                                            const BonusSel &s, const float2 *tab,
                                            long long *s_ll, int *s_i) {
  constexpr int CH = StreamGeom<T>::kCH;
  constexpr int WCH = StreamGeom<T>::kWCH;
  const int sel = s.sel;
  if (sel < 0) return -1;  // uniform across the CTA
  const int c = sel / kConsumerWarps, w = sel - c * kConsumerWarps;
  const int64_t r0 = static_cast<int64_t>(c) * CH + static_cast<int64_t>(w) * WCH;
  const int len = static_cast<int>(max(static_cast<int64_t>(0),
                                       min(static_cast<int64_t>(WCH), sa.a.V - r0)));
  return block_select_fixed<T, WCH / kThreads>(rowp, r0, len, s.target, s.ref, sa.a.balpha, tab,
                                               s_ll, s_i);
}

// ---------------------------------------------------------------------------
// Row combine after the streaming kernel, launched with programmatic
// dependent launch (it waits for the streaming kernel before reading its
// partials).  The first n_fast_ctas CTAs take the log-sum-exp rows, one warp
// per row: the row's log-sum-exp from its (item, warp) partials and the
// drafted token's logit.  Each further CTA takes one bonus row: warp 0
// finds the unit (bonus_select_warp), then the whole CTA the element
// (bonus_rescan).  Used by the verify, the draft sampler and the nucleus
// path; the plain SMC step takes particle_kernel and prompt_kernel instead.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) finish_kernel(const StreamArgs sa, int n_fast_ctas) {
  using Tr = LogitTraits<T>;
  constexpr float kInf = -kNegInf;
  const StepArgs &a = sa.a;
  __shared__ float2 s_tab[64];
  __shared__ BonusSel s_sel;
  __shared__ long long s_ll[kWarps];
  __shared__ int s_i[2 * kWarps];
  stage_exp2_table(s_tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rpp = 2 * a.K + 1;
  const bool bonus_cta = static_cast<int>(blockIdx.x) >= n_fast_ctas;
  int row, part, j, rfi = -1;
  bool live = true;
  if (!bonus_cta) {
    const long long n_fast_rows = static_cast<long long>(a.B) * a.N * 2 * a.K;
    const long long rf = static_cast<long long>(blockIdx.x) * kWarps + warp;
    live = rf < n_fast_rows;
    rfi = live ? static_cast<int>(rf) : 0;
    part = live ? static_cast<int>(rf / (2 * a.K)) : 0;
    const int jj = live ? static_cast<int>(rf - static_cast<long long>(part) * 2 * a.K) : 0;
    j = jj < a.K ? jj : jj + 1;
  } else {
    part = static_cast<int>(blockIdx.x) - n_fast_ctas;
    j = a.K;
  }
  row = part * rpp + j;
  const bool is_bonus = j == a.K;
  const bool fast = !is_bonus || a.bonus_lse;
  const char *rowp = row_base<T>(a, row);
  // the drafted token and its logit are inputs of the step: gathered while
  // the streaming kernel still runs
  int gtok = 0;
  float gv = 0.f, u = 0.f;
  if (is_bonus && warp == 0) u = bonus_uniform(a, part);
  if (!is_bonus && live && lane == 0) {
    gtok = a.tokens[static_cast<size_t>(part) * a.K + (j < a.K ? j : j - a.K - 1)];
    gv = (gtok < 0 || gtok >= a.V) ? __int_as_float(0x7fc00000) : a.tscale * Tr::scalar(rowp, gtok);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (!live) return;

  // fast log-sum-exp pieces of the row (for a bonus row, warp 0's are used)
  float fM = kNegInf, fS = 0.f;
  if (fast && (!is_bonus || warp == 0)) fast_row_stats(sa, row, is_bonus ? -1 : rfi, &fM, &fS);
  if (!is_bonus) {
    if (lane == 0) {
      unsigned bits = 0;
      if (fM == kNegInf) bits |= SMC_DEV_EMPTY_ROW;
      else if (!(fS < kInf) || fM == kInf) bits |= SMC_DEV_NONFINITE;
      const ff lse = row_lse(a.tscale, fM, fS, s_tab);
      if (gtok < 0 || gtok >= a.V) bits |= SMC_DEV_BAD_TOKEN;
      if (bits) raise_status(a.ws.status, bits);
      a.ws.results[row] = RowResult{lse.hi, gv, lse.lo, -1};  // lse as head and tail
    }
    return;
  }
  if (warp == 0) bonus_select_warp<T>(sa, part, rowp, u, fM, fS, true, s_tab, &s_sel);
  __syncthreads();
  const int tok = bonus_rescan<T>(sa, rowp, s_sel, s_tab, s_ll, s_i);
  if (threadIdx.x == 0) {
    a.ws.results[row] = RowResult{s_sel.lse.hi, 0.f, s_sel.lse_alpha.hi, tok};
    if (a.mode == 2) a.out.tokens_out[part] = tok;
  }
}

// ---------------------------------------------------------------------------
// Epilogue of a plain SMC step on the streaming path: particle_kernel (one CTA
// per particle) and prompt_kernel (one CTA per prompt) run side by side.
//
// particle_kernel, launched with programmatic dependent launch after the
// streaming kernel, waits for it, then: warps 1.. combine the particle's 2K
// log-sum-exp rows from their (item, warp) partials and sum its weight
// increment in float-float, while warp 0 locates the bonus draw
// (bonus_select_warp); then the whole CTA rescans the unit (bonus_rescan).
// Each warp's part of the increment goes out at once as tagged 64-bit records
// (publish_part; warp 0's part, the bonus row's log-sum-exps, only with
// alpha != 1): prompt_kernel's thread i polls particle i's records until all
// carry the call's tag and adds the incoming log-weight and the potential
// itself, so no barrier or fence sits between a warp's rows and the prompt.
// The bonus token goes to the bonus row's result, followed by a release
// increment of the prompt's bonus_done counter.
// ---------------------------------------------------------------------------
constexpr uint32_t kCountWaitLimit = 1u << 20;  // polls of about 1 us: about a second

// A warp's part of a particle's weight increment, stored as two tagged 64-bit
// records (head, tail) that prompt_kernel polls: a value and its call's tag in
// one single-copy-atomic store, so no fence is needed.
__device__ __forceinline__ void publish_part(const StepArgs &a, int part, int warp, ff d) {
  unsigned long long *rec = a.ws.wrec + static_cast<size_t>(part) * kWrecPerParticle + 2 * warp;
  const unsigned long long tag = static_cast<unsigned long long>(a.call_tag) << 32;
  st_relaxed_gpu_u64(rec, tag | __float_as_uint(d.hi));
  st_relaxed_gpu_u64(rec + 1, tag | __float_as_uint(d.lo));
}

template <typename T>
__global__ void __launch_bounds__(kThreads) particle_kernel(const StreamArgs sa) {
  using Tr = LogitTraits<T>;
  constexpr float kInf = -kNegInf;
  constexpr unsigned kAll = 0xffffffffu;
  const StepArgs &a = sa.a;
  __shared__ float2 s_tab[64];
  __shared__ BonusSel s_sel;
  __shared__ long long s_ll[kWarps];
  __shared__ int s_i[2 * kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = blockIdx.x;
  const int K = a.K, rpp = 2 * K + 1, nr = 2 * K;
  const char *bonus_rowp = row_base<T>(a, part * rpp + K);
  // the prompt kernel may launch once every particle CTA has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  stage_exp2_table(s_tab);
  // the log-sum-exp rows go to groups of kG lanes of warps 1..: group
  // g = (w - 1) 32/kG + lane/kG takes rows g, g + n_grp, ...
  constexpr int kG = 8, kGpw = 32 / kG;
  constexpr int n_grp = (kWarps - 1) * kGpw;
  const int grp = (warp - 1) * kGpw + lane / kG, sub = lane & (kG - 1);
  // inputs of the step, read while the streaming kernel still runs: the
  // drafted tokens and their logits (lane q kG + r of warp w >= 1 holds row
  // (w - 1) kGpw + q + n_grp r), the incoming log-weight and the potential
  const int jj_l = (warp - 1) * kGpw + lane / kG + n_grp * sub;
  int gtok = 0;
  float gv = 0.f;
  if (warp > 0 && jj_l < nr) {
    const int j = jj_l < K ? jj_l : jj_l + 1;
    gtok = a.tokens[static_cast<size_t>(part) * K + (jj_l < K ? jj_l : jj_l - K)];
    gv = (gtok < 0 || gtok >= a.V) ? __int_as_float(0x7fc00000)
                                   : a.tscale * Tr::scalar(row_base<T>(a, part * rpp + j), gtok);
  }
  const float u = warp == 0 ? bonus_uniform(a, part) : 0.f;
  // every streaming CTA's partials are out once rows_done reaches the grid
  // (bounded; this grid launches only after every streaming CTA has started)
  __shared__ int s_rows_ok;
  if (threadIdx.x == 0) {
    s_rows_ok = wait_count(a.ws.rows_done, static_cast<unsigned>(sa.row_grid), kCountWaitLimit);
  }
  __syncthreads();
  if (!s_rows_ok) {
    if (threadIdx.x == 0) raise_status(a.ws.status, SMC_DEV_TIMEOUT);
    return;
  }

  if (warp == 0) {
    float fM = kNegInf, fS = 0.f;
    if (a.bonus_lse) fast_row_stats(sa, part * rpp + K, -1, &fM, &fS);
    bonus_select_warp<T>(sa, part, bonus_rowp, u, fM, fS, a.bonus_lse, s_tab, &s_sel);
    if (a.bonus_lse && lane == 0) {
      // alpha != 1: the bonus row's log-sum-exps enter the increment
      publish_part(a, part, 0, ff_sub_x(s_sel.lse_alpha, ff_mul_fx(s_sel.lse, a.alpha)));
    }
  } else {
    ff d{0.f, 0.f};
    unsigned bits = 0;
#pragma unroll 1
    for (int r = 0; (warp - 1) * kGpw + n_grp * r < nr; ++r) {  // uniform across the warp
      const int jj = grp + n_grp * r;
      const bool act = jj < nr;
      const int j = jj < K ? jj : jj + 1;
      float fM, fS;
      group_row_stats<kG>(sa, part * rpp + j, part * nr + jj, act, &fM, &fS);
      const int src = (lane & ~(kG - 1)) + r;
      const int t = __shfl_sync(kAll, gtok, src);
      const float g = __shfl_sync(kAll, gv, src);
      if (act && sub == 0) {
        if (fM == kNegInf) bits |= SMC_DEV_EMPTY_ROW;
        else if (!(fS < kInf) || fM == kInf) bits |= SMC_DEV_NONFINITE;
        if (t < 0 || t >= a.V) bits |= SMC_DEV_BAD_TOKEN;
        const ff l = ff_sub_x(ff{g, 0.f}, row_lse(a.tscale, fM, fS, s_tab));  // log p or log q
        d = jj < K ? ff_add_x(d, ff_mul_fx(l, a.alpha)) : ff_sub_x(d, l);
      }
    }
    // the warp's groups, summed into lane 0 (other lanes hold zeros)
#pragma unroll
    for (int o = kG; o < 32; o <<= 1) {
      d = ff_add_x(d, ff{__shfl_xor_sync(kAll, d.hi, o), __shfl_xor_sync(kAll, d.lo, o)});
    }
    if (bits) raise_status(a.ws.status, bits);
    if (lane == 0) publish_part(a, part, warp, d);
  }
  __syncthreads();
  const int tok = bonus_rescan<T>(sa, bonus_rowp, s_sel, s_tab, s_ll, s_i);
  if (threadIdx.x == 0) {
    a.ws.results[static_cast<size_t>(part) * rpp + K].tok = tok;
    add_release_gpu(a.ws.bonus_done + part / a.N, 1u);
  }
}

// prompt_kernel, launched with programmatic dependent launch after
// particle_kernel, never waits for that grid to finish: it stages the KV
// state and the drafted tokens, waits (bounded) until all N particles of its
// prompt have published their weights, lets the next step's row pass launch,
// normalises, resamples and remaps the KV state, and only then waits for the
// bonus tokens to emit them.  It resets its prompt's counters.  A wait that
// gives up raises SMC_DEV_TIMEOUT and leaves the prompt's outputs unwritten.
__global__ void __launch_bounds__(kThreads, 1) prompt_kernel(const StepArgs a, int kv_staged) {
  __shared__ TailSmem sm;
  __shared__ int s_ok;
  extern __shared__ int dyn_i[];
  const int b = blockIdx.x, N = a.N, K = a.K, rpp = 2 * K + 1;
  const int tid = threadIdx.x;
  const KvScratch sc = a.use_kv ? kv_scratch(a.kv, b, N, a.ws, dyn_i, kv_staged != 0) : KvScratch{};
  int top = 0;
  const float lw0 = tail_prefetch(a, b, sm, sc, &top);
  tail_prefetch_stack(a, b, top, sc);
  const float pot = (a.potential && tid < N) ? __ldcg(a.potential + b * N + tid) : 0.f;
  const ResampleKey key = resample_key(a.seed, a.step, b, N);
  // thread i < N polls particle i's weight records until every one carries
  // this call's tag (bounded), and sums them with the incoming log-weight
  ff lwf{0.f, 0.f};
  bool ok = true;
  if (tid < N) {
    const unsigned long long *rec =
        a.ws.wrec + static_cast<size_t>(b * N + tid) * kWrecPerParticle;
    const int w0 = a.bonus_lse ? 0 : 1;
    ok = false;
    for (uint32_t it = 0; it < kCountWaitLimit; ++it) {
      unsigned long long v[kWrecPerParticle];
      bool all = true;
#pragma unroll
      for (int k = 0; k < kWrecPerParticle; ++k) {
        v[k] = k >= 2 * w0 ? ld_relaxed_gpu_u64(rec + k) : 0ull;
        if (k >= 2 * w0 && static_cast<uint32_t>(v[k] >> 32) != a.call_tag) all = false;
      }
      if (all) {
        ff d{0.f, 0.f};
#pragma unroll
        for (int w = 0; w < kWrecPerParticle / 2; ++w) {
          if (w >= w0) {
            d = ff_add_x(d, ff{__uint_as_float(static_cast<uint32_t>(v[2 * w])),
                               __uint_as_float(static_cast<uint32_t>(v[2 * w + 1]))});
          }
        }
        lwf = ff_add_x(ff{lw0, 0.f}, ff_add_x(d, ff{pot, 0.f}));
        ok = true;
        break;
      }
      __nanosleep(it < 64 ? 32 : 1024);
    }
  }
  if (__syncthreads_or(!ok)) {
    if (tid == 0) raise_status(a.ws.status, SMC_DEV_TIMEOUT);
    cp_async_wait_all();
    return;
  }
  // Every particle of this prompt has read its row partials.  The next
  // step's streaming kernel may launch now and stream beside this tail: it
  // writes nothing this step's kernels still read (the bonus partials and
  // counters alternate between calls), and it lets its own dependents launch
  // only after this grid has ended.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const RowResult *res = a.ws.results + static_cast<size_t>(b) * N * rpp;
  const bool resampled = prompt_weights(a, b, sm, lwf, key, a.use_kv ? &sc : nullptr);
  if (a.use_kv) kv_remap_append(a.kv, b, N, sm.anc, resampled, K + 1, a.ws, sm.ks, sc, true, true);
  if (tid == 0) s_ok = wait_count(a.ws.bonus_done + b, static_cast<unsigned>(N), kCountWaitLimit);
  __syncthreads();
  if (!s_ok) {
    if (tid == 0) raise_status(a.ws.status, SMC_DEV_TIMEOUT);
    return;
  }
  if (tid < N) {
    const int anc = sm.anc[tid];
    a.out.tokens_out[static_cast<size_t>(b * N + tid) * (K + 1) + K] =
        __ldcg(&res[static_cast<size_t>(anc) * rpp + K].tok);
  }
  if (tid == 0) {
    a.ws.bonus_done[b] = 0u;
    // the last prompt CTA past its waits: every particle CTA has passed its
    // wait on rows_done, which can start again from 0
    if (atomicAdd(a.ws.tail_ticket, 1u) == gridDim.x - 1) {
      *a.ws.rows_done = 0u;
      *a.ws.tail_ticket = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// Per-prompt tail, one CTA per prompt: weights, ESS, resampling, emission and
// KV remap (SMC mode), or the acceptance scan (SpS mode).  Launched after a
// row kernel; with programmatic dependent launch it may start early and
// waits here until the row kernel has finished and its results are visible.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) tail_kernel(const StepArgs a, int kv_staged) {
  __shared__ TailSmem sm;
  extern __shared__ int dyn_i[];
  if (a.mode == 0) {
    smc_tail(a, blockIdx.x, sm, dyn_i, kv_staged != 0);  // waits inside
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the residual pass may launch now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    sps_tail(a, blockIdx.x, sm);
  }
}

// ---------------------------------------------------------------------------
// Standalone resampling and remap kernels: one CTA per prompt.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
resample_kernel(int N, float ess_frac, uint64_t seed, uint32_t step, float *log_weights,
                int32_t *ancestors, float *ess, int32_t *resampled, unsigned *status) {
  __shared__ TailSmem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const bool valid = tid < N;
  const float lwf = valid ? log_weights[static_cast<size_t>(b) * N + tid] : 0.f;
  stage_exp2_table(sm.tab);
  __syncthreads();
  const ResampleResult rr = normalise_resample(N, ff{lwf, 0.f}, valid, ess_frac,
                                               resample_key(seed, step, b, N), status, sm.anc,
                                               sm.c, sm.red, sm.tab);
  if (valid) {
    log_weights[static_cast<size_t>(b) * N + tid] = rr.resampled ? 0.f : lwf;
    ancestors[static_cast<size_t>(b) * N + tid] = sm.anc[tid];
  }
  if (tid == 0) {
    ess[b] = rr.ess;
    resampled[b] = rr.resampled ? 1 : 0;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
kv_remap_kernel(int N, KvArgs kv, const int32_t *ancestors, const int32_t *resampled,
                int n_append, Workspace ws, int kv_staged) {
  __shared__ TailSmem sm;
  extern __shared__ int dyn_i[];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const bool res = resampled[b] != 0;
  if (tid < N) {
    int a = res ? ancestors[static_cast<size_t>(b) * N + tid] : tid;
    if (a < 0 || a >= N) {
      raise_status(ws.status, SMC_DEV_BAD_BLOCK);
      a = tid;
    }
    sm.anc[tid] = a;
  }
  __syncthreads();
  kv_remap_append(kv, b, N, sm.anc, res, n_append, ws, sm.ks,
                  kv_scratch(kv, b, N, ws, dyn_i, kv_staged != 0), false, false);
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------

// Resident CTAs of the streaming kernel per SM and the SM count of the
// current device (queried once per device).
template <typename T>
static cudaError_t stream_geometry(int *sms, int *per_sm) {
  constexpr int kMaxDev = 64;
  static int cache_sms[kMaxDev], cache_bps[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int slot = dev < kMaxDev ? dev : kMaxDev - 1;
  if (dev >= kMaxDev || cache_sms[slot] == 0) {
    e = cudaFuncSetAttribute(row_stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(stream_dyn_smem()));
    if (e != cudaSuccess) return e;
    int n = 0, b = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, row_stream_kernel<T>, kStreamThreads,
                                                      stream_dyn_smem());
    if (e != cudaSuccess) return e;
    cache_sms[slot] = n;
    cache_bps[slot] = b > 0 ? b : 1;
  }
  *sms = cache_sms[slot];
  *per_sm = cache_bps[slot];
  return cudaSuccess;
}

static cudaEvent_t g_rows_begin = nullptr, g_rows_end = nullptr;
static unsigned long long *g_clk = nullptr;
static unsigned *g_clk_ctr = nullptr;
static int g_clk_cap = 0;

void set_step_clock(unsigned long long *stamps, unsigned *counter, int capacity) {
  g_clk = stamps;
  g_clk_ctr = counter;
  g_clk_cap = capacity;
}

void set_row_timing_events(cudaEvent_t begin, cudaEvent_t end) {
  g_rows_begin = begin;
  g_rows_end = end;
}

// Dynamic shared memory for a staged KV remap, or 0 when it does not fit.
static size_t kv_stage_bytes(int N, const KvArgs *kv) {
  if (!kv) return 0;
  const size_t bytes = kv_stage_words(N, kv->T, kv->P) * sizeof(int);
  return bytes <= kKvStageMaxBytes ? bytes : 0;
}

// The kernels that stage a KV remap in dynamic shared memory take up to
// kKvStageMaxBytes of it on top of their static shared memory; they are
// opted into that maximum once per device, so that every staged size fits
// (and concurrent launches never lower the limit under one another).
//
// The epilogue kernels also ask for the largest shared-memory carveout.  An
// SM changes its L1/shared split only when it is idle, so a small-footprint
// kernel given a small carveout would keep the next kernel's large-footprint
// CTAs (the prompt tails, the next step's streaming CTAs) off every SM it
// occupies until it drains.
static cudaError_t configure_kernels() {
  constexpr int kMaxDev = 64;
  static std::atomic<bool> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const int bytes = static_cast<int>(kKvStageMaxBytes);
  const cudaFuncAttribute attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if ((e = cudaFuncSetAttribute(tail_kernel, attr, bytes)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kv_remap_kernel, attr, bytes)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(prompt_kernel, attr, bytes)) != cudaSuccess) return e;
  const cudaFuncAttribute co = cudaFuncAttributePreferredSharedMemoryCarveout;
  const int full = cudaSharedmemCarveoutMaxShared;
  const void *epilogue[] = {
      reinterpret_cast<const void *>(tail_kernel),
      reinterpret_cast<const void *>(prompt_kernel),
      reinterpret_cast<const void *>(particle_kernel<float>),
      reinterpret_cast<const void *>(particle_kernel<bf16_tag>),
      reinterpret_cast<const void *>(finish_kernel<float>),
      reinterpret_cast<const void *>(finish_kernel<bf16_tag>),
      reinterpret_cast<const void *>(row_stream_kernel<float>),
      reinterpret_cast<const void *>(row_stream_kernel<bf16_tag>)};
  for (const void *f : epilogue) {
    if ((e = cudaFuncSetAttribute(f, co, full)) != cudaSuccess) return e;
  }
  if (dev < kMaxDev) done[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

// A launch with programmatic stream serialisation: the kernel may start
// before the one ahead of it in the stream has finished, and waits
// (griddepcontrol.wait, or on workspace counters) before reading its results.
// Used in place: cfg points at attr.
struct PdlLaunch {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  PdlLaunch(unsigned grid, unsigned block, size_t dyn, cudaStream_t stream) {
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  PdlLaunch(const PdlLaunch &) = delete;
};

// The plain SMC step's epilogue: particle_kernel, then prompt_kernel, which
// runs alongside it.
template <typename T>
static cudaError_t launch_particle_epilogue(const StreamArgs &sa, cudaStream_t stream) {
  const StepArgs &a = sa.a;
  const size_t dyn = a.use_kv ? kv_stage_bytes(a.N, &a.kv) : 0;
  cudaError_t e = configure_kernels();
  if (e != cudaSuccess) return e;
  {
    PdlLaunch l(static_cast<unsigned>(a.B * a.N), kThreads, 0, stream);
    e = cudaLaunchKernelEx(&l.cfg, particle_kernel<T>, sa);
    if (e != cudaSuccess) return e;
  }
  PdlLaunch l(static_cast<unsigned>(a.B), kThreads, dyn, stream);
  return cudaLaunchKernelEx(&l.cfg, prompt_kernel, a, dyn > 0 ? 1 : 0);
}

// The streaming kernel, then either the plain step's epilogue (when
// `fuse_tail` is set; *tail_done is then set) or the row combine
// (finish_kernel), after which the caller launches the tail.
template <typename T>
static cudaError_t launch_stream(const StepArgs &a, long long rows, cudaStream_t stream,
                                 bool fuse_tail, bool *tail_done) {
  int sms = 0, per_sm = 0;
  cudaError_t e = stream_geometry<T>(&sms, &per_sm);
  if (e != cudaSuccess) return e;
  const long long grid_max = static_cast<long long>(sms) * per_sm;
  StreamArgs sa{};
  sa.a = a;
  sa.snch = static_cast<int>((static_cast<long long>(a.V) + StreamGeom<T>::kCH - 1) /
                             StreamGeom<T>::kCH);
  sa.wspan = 40.f / a.balpha;
  const long long total_chunks = rows * sa.snch;
  // about twelve work items per resident CTA, each 1..8 chunks, split evenly
  // over a row (short items keep the CTAs' finishing times close together)
  const long long g = total_chunks / (grid_max * 12);
  const int g0 = static_cast<int>(g < 1 ? 1 : (g > 8 ? 8 : g));
  sa.ipr = (sa.snch + g0 - 1) / g0;
  sa.G = (sa.snch + sa.ipr - 1) / sa.ipr;
  const long long parts = rows / (2 * a.K + 1);
  const long long fast_rows = parts * 2 * a.K;
  // the queue's last non-bonus rows go in single-chunk items: about five
  // halves of a chunk per resident CTA at the end
  long long r2 = sa.G > 1 ? (5 * grid_max / 2 + sa.snch - 1) / sa.snch : 0;
  if (r2 > fast_rows) r2 = fast_rows;
  sa.R1 = static_cast<int>(fast_rows - r2);
  sa.n_items1 = sa.R1 * sa.ipr;
  sa.n_fast_items = static_cast<int>(sa.n_items1 + r2 * sa.snch);
  sa.n_bonus_items = static_cast<int>(parts * sa.snch);
  const long long n_items = static_cast<long long>(sa.n_fast_items) + sa.n_bonus_items;
  const long long grid = grid_max < n_items ? grid_max : n_items;
  sa.signal_rows = fuse_tail ? 1 : 0;
  sa.row_grid = static_cast<int>(grid);
  sa.clk = g_clk;
  sa.clk_ctr = g_clk_ctr;
  sa.clk_cap = g_clk_cap;
  if (g_rows_begin && (e = cudaEventRecord(g_rows_begin, stream)) != cudaSuccess) return e;
  {
    // programmatic dependent launch: when the kernel before it in the stream
    // lets its dependents start early (the step's own epilogue or tail does),
    // the CTAs become resident while it runs and wait at their first
    // instruction for its completion, so no launch gap separates two steps
    PdlLaunch l(static_cast<unsigned>(grid), kStreamThreads, stream_dyn_smem(), stream);
    e = cudaLaunchKernelEx(&l.cfg, row_stream_kernel<T>, sa);
    if (e != cudaSuccess) return e;
  }
  if (g_rows_end && (e = cudaEventRecord(g_rows_end, stream)) != cudaSuccess) return e;
  if (fuse_tail) {
    *tail_done = true;
    return launch_particle_epilogue<T>(sa, stream);
  }
  // log-sum-exp rows: one warp each; bonus rows: one CTA each
  const int n_fast_ctas = static_cast<int>((fast_rows + kWarps - 1) / kWarps);
  PdlLaunch l(static_cast<unsigned>(n_fast_ctas + parts), kThreads, 0, stream);
  return cudaLaunchKernelEx(&l.cfg, finish_kernel<T>, sa, n_fast_ctas);
}


static cudaError_t launch_tail(const StepArgs &a, cudaStream_t stream) {
  const size_t dyn = a.use_kv ? kv_stage_bytes(a.N, &a.kv) : 0;
  cudaError_t e = configure_kernels();
  if (e != cudaSuccess) return e;
  PdlLaunch l(static_cast<unsigned>(a.B), kThreads, dyn, stream);
  return cudaLaunchKernelEx(&l.cfg, tail_kernel, a, dyn > 0 ? 1 : 0);
}

// The row pass (streaming or per-chunk kernel, then the row combine).  With
// `fuse_tail`, the streaming path may also run the per-prompt tail
// (*tail_done is then set).
static cudaError_t launch_rows(const StepArgs &a, int dtype, long long rows, cudaStream_t stream,
                               bool fuse_tail = false, bool *tail_done = nullptr) {
  bool dummy = false;
  if (!tail_done) tail_done = &dummy;
  *tail_done = false;
  cudaError_t e = configure_kernels();
  if (e != cudaSuccess) return e;
  const int esz = dtype == SMC_BF16 ? 2 : 4;
  // bulk copies need 16-byte aligned rows and chunk sizes: aligned bases and V*esz % 16 == 0
  const bool vec = aligned16(a.target) && aligned16(a.draft) &&
                   (static_cast<long long>(a.V) * esz) % 16 == 0;
  if (vec) {
    e = dtype == SMC_BF16 ? launch_stream<bf16_tag>(a, rows, stream, fuse_tail, tail_done)
                          : launch_stream<float>(a, rows, stream, fuse_tail, tail_done);
  } else {
    const long long grid = rows * a.nch;
    dim3 g(static_cast<unsigned>(grid)), blk(kThreads);
    if (g_rows_begin && (e = cudaEventRecord(g_rows_begin, stream)) != cudaSuccess) return e;
    if (dtype == SMC_BF16) step_rows_kernel<bf16_tag, false><<<g, blk, 0, stream>>>(a);
    else step_rows_kernel<float, false><<<g, blk, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess && g_rows_end) e = cudaEventRecord(g_rows_end, stream);
  }
  return e;
}

// A tag for each call, never 0 (so zeroed records never match).
static uint32_t next_call_tag() {
  static std::atomic<uint32_t> counter{0};
  uint32_t t = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
  if (t == 0u) t = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
  return t;
}

static StepArgs step_args(const Shape &s, int mode, const Workspace &ws) {
  StepArgs a{};
  a.call_tag = next_call_tag();
  a.B = s.B; a.N = s.N; a.K = s.K; a.V = s.V;
  a.nch = chunks_per_row(s.dtype, s.V);
  a.mode = mode;
  a.alpha = s.alpha; a.ess_frac = s.ess_frac; a.seed = s.seed; a.step = s.step;
  a.tscale = s.tscale;
  a.balpha = s.alpha * s.tscale;  // fp32 product, as the oracle takes it
  a.bonus_lse = mode != 2 && s.alpha != 1.f;
  a.bonus_purpose = SMC_PURPOSE_BONUS;
  a.bonus_position = s.K;
  a.potential = s.potential;
  a.ws = ws;
  return a;
}

cudaError_t launch_step_rows(const Shape &s, int mode, const void *target, const void *draft,
                             const int32_t *tokens, const StepOutputs &out, const KvArgs *kv,
                             const Workspace &ws, cudaStream_t stream) {
  StepArgs a = step_args(s, mode, ws);
  a.target = static_cast<const char *>(target);
  a.draft = static_cast<const char *>(draft);
  a.tokens = tokens;
  a.out = out;
  a.use_kv = kv != nullptr;
  if (kv) a.kv = *kv;
  const long long rows = static_cast<long long>(s.B) * s.N * (2 * s.K + 1);
  bool tail_done = false;
  cudaError_t e = launch_rows(a, s.dtype, rows, stream, mode == 0 && s.top_p >= 1.f, &tail_done);
  if (e != cudaSuccess) return e;
  if (tail_done) return cudaGetLastError();
  if (s.top_p < 1.f) {
    e = launch_topp(a, s.dtype, s.top_p, rows, stream);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  e = launch_tail(a, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self-test of the bounded waits: one thread runs the counter wait
// (wait_count, as the epilogue kernels use it) or the mbarrier wait
// (mbar_wait, as the streaming kernel's ring uses it) against a condition
// nothing satisfies, for `limit` polls, and raises SMC_DEV_TIMEOUT.
// words[0] is the status word; words[1] the counter (0, never raised).
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(unsigned *words, int kind, unsigned limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  bool ok;
  if (kind == 0) {
    ok = wait_count(words + 1, 1u, limit);
  } else {
    mbar_init(&bar, 1);
    mbar_init_fence();
    ok = mbar_wait(&bar, 0u, limit);  // phase 0 never completes: nothing arrives
  }
  if (!ok) raise_status(words, SMC_DEV_TIMEOUT);
}

cudaError_t launch_selftest_wait(unsigned *words, int kind, unsigned limit, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(words, kind, limit);
  return cudaGetLastError();
}

cudaError_t launch_draft_sample(const Shape &s, const void *logits, int position,
                                int32_t *tokens_out, const Workspace &ws, cudaStream_t stream) {
  Shape s0 = s;
  s0.K = 0;  // one row per particle, and it is the sampled ("bonus") row
  StepArgs a = step_args(s0, 2, ws);
  a.target = static_cast<const char *>(logits);
  a.draft = static_cast<const char *>(logits);
  a.bonus_purpose = SMC_PURPOSE_DRAFT;
  a.bonus_position = position;
  a.out.tokens_out = tokens_out;
  return launch_rows(a, s.dtype, static_cast<long long>(s.B) * s.N, stream);
}

// Per prompt b (one CTA): blocks of its pool with a positive reference count,
// and the blocks its particles' token counts fill without sharing.
__global__ void __launch_bounds__(kThreads) kv_usage_kernel(int N, KvArgs kv, int32_t *used,
                                                            int32_t *unshared) {
  __shared__ int s_red[2 * kWarps];
  const int b = blockIdx.x;
  int u = 0, w = 0;
  for (int k = threadIdx.x; k < kv.P; k += kThreads) {
    u += __ldcg(kv.refcount + static_cast<size_t>(b) * kv.P + k) > 0;
  }
  for (int i = threadIdx.x; i < N; i += kThreads) {
    const long long len = __ldcg(kv.seq_len + static_cast<size_t>(b) * N + i);
    w += len > 0 ? static_cast<int>((len + kv.block_size - 1) / kv.block_size) : 0;
  }
  int tu, tw;
  block_excl_scan_i(u, s_red, &tu);
  block_excl_scan_i(w, s_red, &tw);
  if (threadIdx.x == 0) {
    used[b] = tu;
    unshared[b] = tw;
  }
}

cudaError_t launch_kv_usage(const Shape &s, const KvArgs &kv, int32_t *used, int32_t *unshared,
                            cudaStream_t stream) {
  kv_usage_kernel<<<s.B, kThreads, 0, stream>>>(s.N, kv, used, unshared);
  return cudaGetLastError();
}

cudaError_t launch_resample(const Shape &s, float *log_weights, int32_t *ancestors, float *ess,
                            int32_t *resampled, const Workspace &ws, cudaStream_t stream) {
  resample_kernel<<<s.B, kThreads, 0, stream>>>(s.N, s.ess_frac, s.seed, s.step, log_weights,
                                                ancestors, ess, resampled, ws.status);
  return cudaGetLastError();
}

cudaError_t launch_kv_remap(const Shape &s, const KvArgs &kv, const int32_t *ancestors,
                            const int32_t *resampled, int n_append, const Workspace &ws,
                            cudaStream_t stream) {
  const size_t dyn = kv_stage_bytes(s.N, &kv);
  cudaError_t e = configure_kernels();
  if (e != cudaSuccess) return e;
  kv_remap_kernel<<<s.B, kThreads, dyn, stream>>>(s.N, kv, ancestors, resampled, n_append, ws,
                                                   dyn > 0 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace smcsd
