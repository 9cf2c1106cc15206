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
// resample systematically.  fp32 throughout (FP64 is a slow path on this
// GPU, and the row statistics feeding the weights are fp32-accurate).  The
// block version serves any N <= 256; thread i < N holds lw_i and, on return,
// s_anc[i] holds the ancestor of particle i.
// ---------------------------------------------------------------------------
struct ResampleResult { bool resampled; float ess; };

// Smallest j in [0, n) with c[j] > pt, clamped to n-1.
__device__ __forceinline__ int first_above(const float *c, int n, float pt) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (c[mid] > pt) hi = mid; else lo = mid + 1;
  }
  return lo;
}

__device__ __forceinline__ float block_scan_f(float v, float *scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float w = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += w;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  float base = 0.f;
  for (int w = 0; w < warp; ++w) base += scratch[w];
  return base + v;
}

__device__ ResampleResult normalise_resample(int b, int N, float lw, bool valid, float ess_frac,
                                             uint64_t seed, uint32_t step, unsigned *status,
                                             int *s_anc, float *s_c, float *s_red) {
  constexpr float kInf = -kNegInf;
  unsigned bits = 0;
  if (valid && (isnan(lw) || lw == kInf)) bits |= SMC_DEV_NONFINITE;
  const float m = block_max(valid && !isnan(lw) ? lw : kNegInf, s_red);
  const bool ok = m > kNegInf && m < kInf;
  if (threadIdx.x == 0 && m == kNegInf) bits |= SMC_DEV_ALL_ZERO_WEIGHT;
  if (bits) raise_status(status, bits);
  const float e = (valid && ok) ? expf(lw - m) : 0.f;
  const float big_l = m + logf(block_sum_f(e, s_red));
  const float w = (valid && ok) ? expf(lw - big_l) : 0.f;
  const float ess = 1.f / block_sum_f(w * w, s_red);
  const bool resample = ok && ess < ess_frac * static_cast<float>(N);
  int anc = threadIdx.x;
  if (resample) {
    const float c = block_scan_f(w, s_red);
    if (valid) s_c[threadIdx.x] = c;
    __syncthreads();
    if (valid) {
      const float u0 = philox_uniform(seed, step, b, 0, SMC_PURPOSE_RESAMPLE);
      anc = first_above(s_c, N, (u0 + static_cast<float>(threadIdx.x)) / static_cast<float>(N));
    }
  }
  if (valid) s_anc[threadIdx.x] = anc;
  __syncthreads();
  return {resample, ess};
}

// The same for N <= 32, by warp 0 alone with shuffles (no CTA barrier).
__device__ ResampleResult normalise_resample_warp(int b, int N, float lw, bool valid,
                                                  float ess_frac, uint64_t seed, uint32_t step,
                                                  unsigned *status, int *s_anc, float *s_c) {
  constexpr float kInf = -kNegInf;
  const int lane = threadIdx.x & 31;
  unsigned bits = 0;
  if (valid && (isnan(lw) || lw == kInf)) bits |= SMC_DEV_NONFINITE;
  const float m = warp_max(valid && !isnan(lw) ? lw : kNegInf);
  const bool ok = m > kNegInf && m < kInf;
  if (lane == 0 && m == kNegInf) bits |= SMC_DEV_ALL_ZERO_WEIGHT;
  if (bits) raise_status(status, bits);
  float e = (valid && ok) ? expf(lw - m) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
  const float big_l = m + logf(e);
  const float w = (valid && ok) ? expf(lw - big_l) : 0.f;
  float w2 = w * w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w2 += __shfl_xor_sync(0xffffffffu, w2, o);
  const float ess = 1.f / w2;
  const bool resample = ok && ess < ess_frac * static_cast<float>(N);
  int anc = lane;
  if (resample) {
    float c = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) c += v;
    }
    if (valid) s_c[lane] = c;
    __syncwarp();
    if (valid) {
      const float u0 = philox_uniform(seed, step, b, 0, SMC_PURPOSE_RESAMPLE);
      anc = first_above(s_c, N, (u0 + static_cast<float>(lane)) / static_cast<float>(N));
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

__device__ void kv_remap_append(const KvArgs &kv, int b, int N, const int *s_anc, bool resampled,
                                int n_append, const Workspace &ws, int *s_i, int *s_tail,
                                int *s_nb, const KvScratch &sc, bool copied) {
  __shared__ int s_flag, s_top_old, s_n_freed;
  __shared__ long long s_ll[kWarps];
  const int T = kv.T, bs = kv.block_size, P = kv.P;
  const int lo_id = b * P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int words = (P + 31) / 32;
  const bool staged = sc.rc != nullptr;
  int32_t *tables = kv.tables + static_cast<size_t>(b) * N * T;
  int32_t *seq_len = kv.seq_len + static_cast<size_t>(b) * N;
  int32_t *stack = kv.free_list + static_cast<size_t>(b) * P;
  const long long cap = static_cast<long long>(T) * bs;  // tokens a full table holds
  if (!copied) kv_copy_in(kv, b, N, sc, 0, kThreads);
  if (!staged && tid == 0) {
    const int top0 = kv.free_top[b];
    s_top_old = top0;
    s_flag = (top0 < 0 || top0 > P) ? 1 : 0;
    kv.n_cow[b] = 0;
  }
  __syncthreads();
  if (staged && tid == 0) {
    const int top0 = *sc.top0;
    s_top_old = top0;
    s_flag = (top0 < 0 || top0 > P) ? 1 : 0;
    kv.n_cow[b] = 0;
  }
  if (tid == 0) s_n_freed = 0;
  __syncthreads();
  auto in_pool = [&](int blk) { return blk >= lo_id && blk < lo_id + P; };
  auto fail = [&]() {
    if (tid == 0) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
  };
  if (s_flag) { fail(); return; }
  // used blocks of every (pre-remap) particle; a bad count is an error
  for (int i = tid; i < N; i += kThreads) {
    const int len = sc.old_l[i];
    if (len < 0 || len > cap) {
      s_flag = 1;
      s_nb[i] = 0;
    } else {
      s_nb[i] = static_cast<int>((static_cast<long long>(len) + bs - 1) / bs);
    }
  }
  __syncthreads();
  if (s_flag) { fail(); return; }

  if (resampled) {
    if (staged) {
      // net reference-count change per block in shared memory, then one pass
      // over the pool applies it; a count reaching 0 frees the block.  Every
      // used slot of every old table is seen here (as ov of its particle),
      // so the pool check of the ids happens in the same pass; a slot whose
      // value does not change is not rewritten.
      for (int i = warp; i < N; i += kWarps) {
        const int a = s_anc[i];
        const int nb_new = s_nb[a], nb_old = s_nb[i];
        for (int t = lane; t < T; t += 32) {
          const int nv = sc.old_t[a * T + t];
          const int ov = sc.old_t[i * T + t];
          const bool has_new = t < nb_new, has_old = t < nb_old;
          if ((has_new && !in_pool(nv)) || (has_old && !in_pool(ov))) {
            s_flag = 1;
            continue;
          }
          if (has_new && !(has_old && ov == nv)) atomicAdd(&sc.delta[nv - lo_id], 1);
          if (has_old && !(has_new && nv == ov)) atomicSub(&sc.delta[ov - lo_id], 1);
          if (nv != ov) tables[i * T + t] = nv;
        }
      }
      for (int i = tid; i < N; i += kThreads) seq_len[i] = sc.old_l[s_anc[i]];
      __syncthreads();
      if (s_flag) { fail(); return; }
      for (int k = tid; k < P; k += kThreads) {
        const int d = sc.delta[k];
        if (d != 0) {
          const int nr = sc.rc[k] + d;
          kv.refcount[lo_id + k] = nr;
          if (nr == 0) atomicOr(&sc.bits[k >> 5], 1u << (k & 31));
        }
      }
      __syncthreads();
    } else {
      for (int i = warp; i < N; i += kWarps) {
        for (int t = lane; t < s_nb[i]; t += 32) {
          if (!in_pool(sc.old_t[i * T + t])) s_flag = 1;
        }
      }
      __syncthreads();
      if (s_flag) { fail(); return; }
      // new references first, so no count touches 0 before every increment is in
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
    }
    // push freed blocks in ascending id order (staged: also list them in
    // `delta`, whose counts are spent)
    int top = s_top_old;
    for (int w0 = 0; w0 < words; w0 += kThreads) {
      const int w = w0 + tid;
      unsigned fb = w < words ? sc.bits[w] : 0u;
      int total;
      int pos = top + block_excl_scan_i(__popc(fb), s_i, &total);
      if (fb) sc.bits[w] = 0u;
      while (fb) {
        const int bit = __ffs(fb) - 1;
        fb &= fb - 1;
        if (pos < P) {
          stack[pos] = lo_id + w * 32 + bit;
          if (staged) sc.delta[pos - s_top_old] = lo_id + w * 32 + bit;
        }
        ++pos;
      }
      top += total;
    }
    if (top > P) s_flag = 1;  // counts did not match the tables
    __syncthreads();
    if (tid == 0) {
      kv.free_top[b] = min(top, P);
      s_n_freed = min(top, P) - s_top_old;
    }
    if (s_flag) { fail(); return; }
    __syncthreads();
  }
  if (n_append <= 0) return;

  // ---- append: particle i's table is now row src(i) of the copy -----------
  const bool valid = tid < N;
  const int src = valid ? (resampled ? s_anc[tid] : tid) : 0;
  int len = 0, nb = 0, tail = -1;
  if (valid) {
    len = sc.old_l[src];
    nb = s_nb[src];
    if (len % bs) {
      tail = sc.old_t[src * T + nb - 1];
      if (!in_pool(tail)) s_flag = 1;
    }
    s_tail[tid] = tail;
  }
  __syncthreads();
  if (s_flag) { fail(); return; }
  int fork = 0;
  if (valid && tail >= 0) {
    for (int i2 = 0; i2 < tid; ++i2) {
      if (s_tail[i2] == tail) { fork = 1; break; }
    }
  }
  const long long nb2 = valid ? (static_cast<long long>(len) + n_append + bs - 1) / bs : 0;
  if (valid && nb2 > T) s_flag = 2;
  const int grow = (valid && nb2 <= T) ? static_cast<int>(nb2) - nb : 0;
  // one scan of (forks, pops) packed in 64 bits: forks high, pops low
  long long both_total;
  const long long both = block_excl_scan_ll((static_cast<long long>(fork) << 32) | (fork + grow),
                                            s_ll, &both_total);
  const int off = static_cast<int>(both & 0xffffffffll);
  const int cidx = static_cast<int>(both >> 32);
  const int total_pops = static_cast<int>(both_total & 0xffffffffll);
  const int n_forks = static_cast<int>(both_total >> 32);
  const int n_freed = s_n_freed, top_old = s_top_old;
  const int top = top_old + n_freed;
  __syncthreads();
  if (s_flag == 2) {
    if (tid == 0) raise_status(ws.status, SMC_DEV_TABLE_OVERFLOW);
    return;
  }
  if (total_pops > top) {
    if (tid == 0) raise_status(ws.status, SMC_DEV_POOL_EXHAUSTED);
    return;
  }
  // the k-th pop from the top: this remap's freed blocks first (the last
  // pushed on top), then the stack as it was
  auto pop = [&](int k) -> int {
    if (!staged) return stack[top - 1 - k];
    if (k < n_freed) return sc.delta[n_freed - 1 - k];
    const int j = k - n_freed;
    return j < kStackPre ? sc.stk[j] : stack[top_old - 1 - j];
  };
  if (valid) {
    int k = off;
    if (fork) {
      const int d = pop(k);
      ++k;
      if (in_pool(d)) {
        int32_t *pair = kv.cow_pairs + (static_cast<size_t>(b) * N + cidx) * 2;
        pair[0] = tail;
        pair[1] = d;
        tables[tid * T + nb - 1] = d;
        kv.refcount[d] = 1;
        atomicSub(&kv.refcount[tail], 1);
      } else {
        raise_status(ws.status, SMC_DEV_BAD_BLOCK);
      }
    }
    for (int g = 0; g < grow; ++g) {
      const int d = pop(k);
      ++k;
      if (in_pool(d)) {
        tables[tid * T + nb + g] = d;
        kv.refcount[d] = 1;
      } else {
        raise_status(ws.status, SMC_DEV_BAD_BLOCK);
      }
    }
    seq_len[tid] = static_cast<int>(len + n_append);
  }
  if (tid == 0) {
    kv.free_top[b] = top - total_pops;
    kv.n_cow[b] = n_forks;
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
  float c[SMC_MAX_N];
  float red[2 * kWarps];
  int anc[SMC_MAX_N];
  int bonus[SMC_MAX_N];
  int tail[SMC_MAX_N];
  int nb[SMC_MAX_N];
  int ired[2 * kWarps];
};

// Runs in tail_kernel, launched with programmatic dependent launch while the
// finish kernel still runs.  The KV state, the incoming log-weights and the
// drafted tokens were all written before this step's first kernel, so they
// are read before waiting for the finish kernel; only the row results are
// read after.
__device__ void smc_tail(const StepArgs &a, int b, TailSmem &sm, int *dyn, bool kv_staged) {
  const int N = a.N, K = a.K, rpp = 2 * K + 1;
  const int tid = threadIdx.x;
  const bool small = N <= 32;
  __shared__ int s_res;
  const KvScratch sc = a.use_kv ? kv_scratch(a.kv, b, N, a.ws, dyn, kv_staged) : KvScratch{};
  if (a.use_kv) kv_copy_in(a.kv, b, N, sc, 0, kThreads);
  const bool tok_staged = N * K <= kTailTokens;
  if (tok_staged) {
    copy_batched(sm.tok, a.tokens + static_cast<size_t>(b) * N * K, N * K, tid, kThreads);
  }
  const bool valid = tid < N;
  const int part = b * N + tid;
  const float lw0 = valid ? __ldcg(a.out.log_weights + part) : 0.f;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tok_staged) __syncthreads();  // sm.tok complete
  // with N <= 32, warp 0 alone does the weights (shuffles, no CTA barrier)
  const bool weights_thread = small ? tid < 32 : true;
  if (weights_thread) {
    float lwf = 0.f;
    if (valid) {
      const RowResult *r = a.ws.results + static_cast<size_t>(part) * rpp;
      const float4 rb = __ldcg(reinterpret_cast<const float4 *>(r + K));
      float delta = 0.f;
#pragma unroll 4
      for (int k = 0; k < K; ++k) {
        const float4 rp = __ldcg(reinterpret_cast<const float4 *>(r + k));
        const float4 rq = __ldcg(reinterpret_cast<const float4 *>(r + K + 1 + k));
        delta += a.alpha * (rp.y - rp.x) - (rq.y - rq.x);
      }
      if (a.alpha != 1.f) delta += rb.z - a.alpha * rb.x;
      if (a.potential) delta += __ldcg(a.potential + part);
      sm.bonus[tid] = __float_as_int(rb.w);
      lwf = lw0 + delta;
    }
    const ResampleResult rr =
        small ? normalise_resample_warp(b, N, lwf, valid, a.ess_frac, a.seed, a.step, a.ws.status,
                                        sm.anc, sm.c)
              : normalise_resample(b, N, lwf, valid, a.ess_frac, a.seed, a.step, a.ws.status,
                                   sm.anc, sm.c, sm.red);
    if (valid) {
      const int anc = sm.anc[tid];
      a.out.log_weights[part] = rr.resampled ? 0.f : lwf;
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
      dst[K] = sm.bonus[anc];
    }
    if (tid == 0) {
      a.out.ess[b] = rr.ess;
      a.out.resampled[b] = rr.resampled ? 1 : 0;
      s_res = rr.resampled ? 1 : 0;
    }
  }
  __syncthreads();
  if (a.use_kv) {
    kv_remap_append(a.kv, b, N, sm.anc, s_res != 0, K + 1, a.ws, sm.ired, sm.tail, sm.nb, sc,
                    true);
  }
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
  if (is_bonus) stage_exp2_table(s_tab);

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
        const float lse = a.tscale * M + logf(sum);
        const int k = j < a.K ? j : j - a.K - 1;
        const int tok = a.tokens[static_cast<size_t>(part) * a.K + k];
        if (tok < 0 || tok >= a.V) bits |= SMC_DEV_BAD_TOKEN;
        else g = a.tscale * Tr::scalar(rowp, tok);
        if (bits) raise_status(a.ws.status, bits);
        a.ws.results[row] = RowResult{lse, g, 0.f, -1};
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
          const double lt = log(ff_to_double(total));
          lse_alpha = static_cast<float>(static_cast<double>(alpha) * M + lt);
          lse = a.bonus_lse ? a.tscale * M + logf(fast) : lse_alpha;
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

struct SlotMeta { int row, part, j, chunk, n, flags, pad0, pad1; };

// Logits per ring slot and per 16-byte vector of the streaming kernel.
template <typename T> struct StreamGeom {
  static constexpr int kESZ = sizeof(T) == 4 ? 4 : 2;
  static constexpr int kEPV = 16 / kESZ;
  static constexpr int kCH = kChunkBytes / kESZ;
  static constexpr int kWCH = kCH / kConsumerWarps;  // logits of one consumer warp's range
};

struct StreamArgs {
  StepArgs a;
  int snch;           // ring-slot chunks per row: ceil(V / StreamGeom<T>::kCH)
  float wspan;        // 40 / balpha: logits further below a range's max weigh e^-40
  int G;              // chunks per work item of a non-bonus row
  int ipr;            // work items per non-bonus row
  int n_fast_items;   // non-bonus rows * ipr
  int n_bonus_items;  // bonus rows * snch (one chunk per item)
};

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
  __shared__ int s_exited;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rpp = 2 * a.K + 1;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init_fence();
    s_exited = 0;
  }
  stage_exp2_split(s_th, s_tl);
  __syncthreads();  // the only CTA-wide barrier

  // ---- producer warp -----------------------------------------------------------
  // Work comes from two queues: items of G chunks of the non-bonus rows, and
  // single chunks of the bonus rows (whose weights cost far more to compute).
  // The producer interleaves them in the proportion of the whole step (2K
  // non-bonus chunks per bonus chunk), so that every CTA, all through the
  // kernel, mixes streaming-bound and arithmetic-bound chunks evenly.
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      const int rest = rpp - 1;  // non-bonus rows per particle
      int row = 0, first = 0, chunk = 0, end = 0;
      int n_fast = 0, n_bonus = 0;
      bool have = false, fast_done = sa.n_fast_items == 0, bonus_done = sa.n_bonus_items == 0;
      // each queue's next claim is issued one item ahead, so that the
      // atomic's round trip overlaps the copies of the current item
      unsigned next_fast = fast_done ? 0u : atomicAdd(&a.ws.work_counter[0], 1u);
      unsigned next_bonus = bonus_done ? 0u : atomicAdd(&a.ws.work_counter[1], 1u);
      for (int i = 0;; ++i) {
        const int slot = i % kStages;
        if (i >= kStages &&
            !mbar_wait(&empty[slot], static_cast<uint32_t>(i / kStages - 1) & 1u, kWaitLimit)) {
          raise_status(a.ws.status, SMC_DEV_TIMEOUT);
          meta[slot].flags = kSlotEnd;  // consumers time out on this slot too
          break;
        }
        while (!have || chunk >= end) {
          have = false;
          if (fast_done && bonus_done) break;
          const bool take_bonus =
              !bonus_done && (fast_done || n_bonus * 2 * a.K < n_fast * sa.G);
          if (take_bonus) {
            const unsigned id = next_bonus;
            if (id >= static_cast<unsigned>(sa.n_bonus_items)) { bonus_done = true; continue; }
            next_bonus = atomicAdd(&a.ws.work_counter[1], 1u);
            ++n_bonus;
            const int part = static_cast<int>(id) / sa.snch;
            row = part * rpp + a.K;
            first = static_cast<int>(id) - part * sa.snch;
            end = first + 1;
          } else {
            const unsigned id = next_fast;
            if (id >= static_cast<unsigned>(sa.n_fast_items)) { fast_done = true; continue; }
            next_fast = atomicAdd(&a.ws.work_counter[0], 1u);
            ++n_fast;
            const int rf = static_cast<int>(id) / sa.ipr;
            const int g = static_cast<int>(id) - rf * sa.ipr;
            const int part = rf / rest, jj = rf - (rf / rest) * rest;
            row = part * rpp + (jj < a.K ? jj : jj + 1);
            first = g * sa.G;
            end = min(first + sa.G, sa.snch);
          }
          chunk = first;
          have = true;
        }
        if (!have) {
          SlotMeta &mt = meta[slot];
          mt.row = -1; mt.part = 0; mt.j = 0; mt.chunk = 0; mt.n = 0; mt.flags = kSlotEnd;
          mbar_arrive(&full[slot]);
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
        const int g = is_bonus ? mt.chunk : mt.chunk / sa.G;
        a.ws.item_part[(static_cast<size_t>(row) * sa.snch + g) * kConsumerWarps + warp] =
            make_float2(M, contrib);
      }
    }
  }

  // ---- consumer exit: let the finish kernel launch; reset the work counters ---
  if (lane == 0) {
    if (atomicAdd(&s_exited, 1) == kConsumerWarps - 1) {
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
// Row combine after the streaming kernel, launched with programmatic
// dependent launch (it waits for the streaming kernel before reading its
// partials).  The first n_fast_ctas CTAs take the log-sum-exp rows, one warp
// per row: the row's log-sum-exp from its (item, warp) partials and the
// drafted token's logit.  Each further CTA takes one bonus row: warp 0 finds
// which (chunk, warp) unit holds u times the total from the units'
// float-float sums, then the whole CTA rescans that unit in exact fixed
// point to find the element (inverse CDF in vocabulary order).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kThreads) finish_kernel(const StreamArgs sa, int n_fast_ctas) {
  using Tr = LogitTraits<T>;
  constexpr int CH = StreamGeom<T>::kCH;
  constexpr int WCH = StreamGeom<T>::kWCH;
  constexpr float kInf = -kNegInf;
  const StepArgs &a = sa.a;
  __shared__ float2 s_tab[64];
  __shared__ long long s_ll[kWarps];
  __shared__ int s_i[2 * kWarps];
  __shared__ long long s_target;
  __shared__ int s_sel;
  __shared__ float s_ref;
  __shared__ float s_red[2 * kWarps];
  __shared__ float2 s_f2[kWarps];
  stage_exp2_table(s_tab);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rpp = 2 * a.K + 1;
  const bool bonus_cta = static_cast<int>(blockIdx.x) >= n_fast_ctas;
  int row, part, j;
  bool live = true;
  if (!bonus_cta) {
    const long long n_fast_rows = static_cast<long long>(a.B) * a.N * 2 * a.K;
    const long long rf = static_cast<long long>(blockIdx.x) * kWarps + warp;
    live = rf < n_fast_rows;
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
  float gv = 0.f;
  if (!is_bonus && live && lane == 0) {
    gtok = a.tokens[static_cast<size_t>(part) * a.K + (j < a.K ? j : j - a.K - 1)];
    gv = (gtok < 0 || gtok >= a.V) ? __int_as_float(0x7fc00000) : a.tscale * Tr::scalar(rowp, gtok);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (!live) return;

  // fast log-sum-exp pieces of the row (every warp of a bonus CTA computes
  // them; only warp 0's are used)
  float fM = kNegInf, fS = 0.f;
  if (fast) {
    const float2 *ip = a.ws.item_part + static_cast<size_t>(row) * sa.snch * kConsumerWarps;
    const int n_ip = (is_bonus ? sa.snch : sa.ipr) * kConsumerWarps;
    float lm = kNegInf, ls = 0.f;
#pragma unroll 4
    for (int c = lane; c < n_ip; c += 32) {
      const float2 pv = ip[c];
      if (pv.x > lm) {
        if (lm > kNegInf && pv.x < kInf) ls *= expf(a.tscale * (lm - pv.x));
        else if (pv.x == kInf) ls = 0.f;
        lm = pv.x;
      }
      if (pv.x > kNegInf && lm < kInf) ls += pv.y * expf(a.tscale * (pv.x - lm));
      else if (pv.y != 0.f) ls += pv.y;  // NaN marker
    }
    fM = warp_max(lm);
    fS = (lm > kNegInf && fM < kInf) ? ls * expf(a.tscale * (lm - fM)) : ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) fS += __shfl_xor_sync(0xffffffffu, fS, o);
  }
  if (!is_bonus) {
    if (lane == 0) {
      unsigned bits = 0;
      if (fM == kNegInf) bits |= SMC_DEV_EMPTY_ROW;
      else if (!(fS < kInf) || fM == kInf) bits |= SMC_DEV_NONFINITE;
      const float lse = a.tscale * fM + logf(fS);
      if (gtok < 0 || gtok >= a.V) bits |= SMC_DEV_BAD_TOKEN;
      if (bits) raise_status(a.ws.status, bits);
      a.ws.results[row] = RowResult{lse, gv, 0.f, -1};
    }
    return;
  }

  // ---- bonus row: units are (chunk, warp) ranges of WCH logits in vocabulary
  // order, each with its max as reference and the float-float sum of its
  // weights relative to it
  const float alpha = a.balpha;
  int4 *bp = a.ws.bonus_part + static_cast<size_t>(part) * sa.snch * kConsumerWarps;
  const int n_units = sa.snch * kConsumerWarps;
  // rows of up to kThreads units: thread q holds unit q from here on
  int4 pv_own = threadIdx.x < n_units ? bp[threadIdx.x]
                                      : make_int4(__float_as_int(kNegInf), 0, 0, 0);
  bool flagged = pv_own.w != 0;
  for (int q = kThreads + threadIdx.x; q < n_units; q += kThreads) flagged |= bp[q].w != 0;
  if (__syncthreads_or(flagged)) {
    // a unit whose max was too large for the streaming kernel's clamp (flag
    // set) is summed here instead, in exact fixed point (rare)
    if (warp == 0) {
      for (int q = 0; q < n_units; ++q) {
        const int4 pv = bp[q];
        if (pv.w == 0) continue;
        const float ref = __int_as_float(pv.x);
        const int c = q / kConsumerWarps, w = q - c * kConsumerWarps;
        const int64_t r0 = static_cast<int64_t>(c) * CH + static_cast<int64_t>(w) * WCH;
        const int len = static_cast<int>(min(static_cast<int64_t>(WCH), a.V - r0));
        long long sum = 0;
        for (int i = lane; i < len; i += 32) sum += weight_fixed(Tr::scalar(rowp, r0 + i), ref, alpha, s_tab);
        const ff v = fixed_to_ff(warp_sum_ll(sum));
        __syncwarp();
        if (lane == 0) bp[q] = make_int4(pv.x, __float_as_int(v.hi), __float_as_int(v.lo), 0);
        __syncwarp();
      }
    }
    __syncthreads();
    if (threadIdx.x < n_units) pv_own = bp[threadIdx.x];
  }
  const float u = philox_uniform(a.seed, a.step, part, a.bonus_position, a.bonus_purpose);
  if (n_units <= kThreads) {
    // one unit per thread: its mass relative to the row's largest reference
    // M, a CTA-wide inclusive prefix, and the first unit whose prefix exceeds
    // u times the total
    const int q = threadIdx.x;
    const int4 pv = pv_own;
    const float ref = __int_as_float(pv.x);
    const float M = block_max(ref, s_red);
    const bool ok = M > kNegInf && M < kInf;
    ff val{0.f, 0.f}, f{1.f, 0.f};
    if (ok && ref > kNegInf) {
      f = ff_norm(weight_term(ref, M, alpha, s_tab));  // exp(alpha (ref - M))
      val = ff_mul(ff{__int_as_float(pv.y), __int_as_float(pv.z)}, f);
    }
    ff total;
    const ff incl = block_ff_scan(val, s_f2, &total);
    const ff target = ff_mul_f(total, u);
    const bool pos = val.hi > 0.f;
    const bool hit = pos && ff_gt(incl, target);
    const int first = block_min_i(hit ? q : 0x7fffffff, s_i);
    const int last = -block_min_i(pos ? -q : 1, s_i);  // largest positive unit, or -1
    const int sel = !ok ? -1 : (first != 0x7fffffff ? first : last);
    if (q == sel) {
      // the remaining target in the unit's own units; past the total
      // (rounding), the unit's whole mass
      const ff rem = first != 0x7fffffff ? ff_div(ff_sub(target, ff_sub(incl, val)), f)
                                         : ff_div(val, f);
      s_target = ff_to_fixed(rem);
      s_ref = ref;
    }
    if (q == 0) {
      s_sel = sel;
      float lse, lse_alpha;
      if (ok) {
        lse_alpha = alpha * M + (logf(total.hi) + total.lo / total.hi);
        lse = a.bonus_lse ? a.tscale * fM + logf(fS) : lse_alpha;
      } else {
        lse = lse_alpha = M == kNegInf ? kNegInf : __int_as_float(0x7fc00000);
        raise_status(a.ws.status, M == kNegInf ? SMC_DEV_EMPTY_ROW : SMC_DEV_NONFINITE);
      }
      a.ws.results[row] = RowResult{lse, 0.f, lse_alpha, -1};
    }
  } else if (warp == 0) {
    // longer rows: warp 0 computes unit masses on demand
    float M = kNegInf;
    for (int q = lane; q < n_units; q += 32) M = fmaxf(M, __int_as_float(bp[q].x));
    M = warp_max(M);
    const bool ok = M > kNegInf && M < kInf;
    auto unit_mass = [&](int q, ff *val, ff *f) {
      const int4 pv = bp[q];
      const float ref = __int_as_float(pv.x);
      if (ok && ref > kNegInf) {
        *f = ff_norm(weight_term(ref, M, alpha, s_tab));  // exp(alpha (ref - M))
        *val = ff_mul(ff{__int_as_float(pv.y), __int_as_float(pv.z)}, *f);
      }
    };
    ff total{0.f, 0.f};
    for (int q0 = 0; q0 < n_units; q0 += 32) {
      ff val{0.f, 0.f}, f{1.f, 0.f};
      if (q0 + lane < n_units) unit_mass(q0 + lane, &val, &f);
      total = ff_add(total, warp_ff_sum(val));
    }
    ff rem{0.f, 0.f};
    const int sel = ok ? warp_find_chunk(n_units, ff_mul_f(total, u), unit_mass, &rem) : -1;
    if (lane == 0) {
      s_sel = sel;
      s_target = ff_to_fixed(rem);
      s_ref = sel >= 0 ? __int_as_float(bp[sel].x) : 0.f;
      float lse, lse_alpha;
      if (ok) {
        lse_alpha = alpha * M + (logf(total.hi) + total.lo / total.hi);
        lse = a.bonus_lse ? a.tscale * fM + logf(fS) : lse_alpha;
      } else {
        lse = lse_alpha = M == kNegInf ? kNegInf : __int_as_float(0x7fc00000);
        raise_status(a.ws.status, M == kNegInf ? SMC_DEV_EMPTY_ROW : SMC_DEV_NONFINITE);
      }
      a.ws.results[row] = RowResult{lse, 0.f, lse_alpha, -1};
    }
  }
  __syncthreads();
  const int sel = s_sel;
  if (sel < 0) {  // uniform across the CTA
    if (a.mode == 2 && threadIdx.x == 0) a.out.tokens_out[part] = -1;
    return;
  }
  const int c = sel / kConsumerWarps, w = sel - c * kConsumerWarps;
  const int64_t r0 = static_cast<int64_t>(c) * CH + static_cast<int64_t>(w) * WCH;
  const int len = static_cast<int>(max(static_cast<int64_t>(0),
                                       min(static_cast<int64_t>(WCH), a.V - r0)));
  const int tok = block_select_fixed<T, WCH / kThreads>(rowp, r0, len, s_target, s_ref, alpha,
                                                         s_tab, s_ll, s_i);
  if (threadIdx.x == 0) {
    a.ws.results[row].tok = tok;
    if (a.mode == 2) a.out.tokens_out[part] = tok;
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
  const ResampleResult rr = normalise_resample(b, N, lwf, valid, ess_frac, seed, step, status,
                                               sm.anc, sm.c, sm.red);
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
  kv_remap_append(kv, b, N, sm.anc, res, n_append, ws, sm.ired, sm.tail, sm.nb,
                  kv_scratch(kv, b, N, ws, dyn_i, kv_staged != 0), false);
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

void set_row_timing_events(cudaEvent_t begin, cudaEvent_t end) {
  g_rows_begin = begin;
  g_rows_end = end;
}

template <typename T>
static cudaError_t launch_stream(const StepArgs &a, long long rows, cudaStream_t stream) {
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
  sa.n_fast_items = static_cast<int>(parts * 2 * a.K * sa.ipr);
  sa.n_bonus_items = static_cast<int>(parts * sa.snch);
  const long long n_items = static_cast<long long>(sa.n_fast_items) + sa.n_bonus_items;
  const long long grid = grid_max < n_items ? grid_max : n_items;
  if (g_rows_begin && (e = cudaEventRecord(g_rows_begin, stream)) != cudaSuccess) return e;
  row_stream_kernel<T><<<static_cast<unsigned>(grid), kStreamThreads, stream_dyn_smem(), stream>>>(sa);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (g_rows_end && (e = cudaEventRecord(g_rows_end, stream)) != cudaSuccess) return e;
  // log-sum-exp rows: one warp each; bonus rows: one CTA each
  const long long fast_rows = parts * 2 * a.K;
  const int n_fast_ctas = static_cast<int>((fast_rows + kWarps - 1) / kWarps);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_fast_ctas + parts));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, finish_kernel<T>, sa, n_fast_ctas);
}

// The per-prompt tail, launched with programmatic dependent launch so that it
// can be scheduled while the row kernel drains.
// Dynamic shared memory for a staged KV remap, or 0 when it does not fit.
static size_t kv_stage_bytes(int N, const KvArgs *kv) {
  if (!kv) return 0;
  const size_t bytes = kv_stage_words(N, kv->T, kv->P) * sizeof(int);
  return bytes <= kKvStageMaxBytes ? bytes : 0;
}


static cudaError_t launch_tail(const StepArgs &a, cudaStream_t stream) {
  const size_t dyn = a.use_kv ? kv_stage_bytes(a.N, &a.kv) : 0;
  cudaError_t e = allow_dyn_smem(tail_kernel, dyn);
  if (e != cudaSuccess) return e;
  const int staged = dyn > 0 ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tail_kernel, a, staged);
}

// The row pass (streaming or per-chunk kernel, then the row combine).
static cudaError_t launch_rows(const StepArgs &a, int dtype, long long rows, cudaStream_t stream) {
  const int esz = dtype == SMC_BF16 ? 2 : 4;
  // bulk copies need 16-byte aligned rows and chunk sizes: aligned bases and V*esz % 16 == 0
  const bool vec = aligned16(a.target) && aligned16(a.draft) &&
                   (static_cast<long long>(a.V) * esz) % 16 == 0;
  cudaError_t e;
  if (vec) {
    e = dtype == SMC_BF16 ? launch_stream<bf16_tag>(a, rows, stream)
                          : launch_stream<float>(a, rows, stream);
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

static StepArgs step_args(const Shape &s, int mode, const Workspace &ws) {
  StepArgs a{};
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
  cudaError_t e = launch_rows(a, s.dtype, rows, stream);
  if (e != cudaSuccess) return e;
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
  cudaError_t e = allow_dyn_smem(kv_remap_kernel, dyn);
  if (e != cudaSuccess) return e;
  kv_remap_kernel<<<s.B, kThreads, dyn, stream>>>(s.N, kv, ancestors, resampled, n_append, ws,
                                                   dyn > 0 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace smcsd
