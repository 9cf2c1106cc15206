// SMC-SD step kernels for sm_103a.
//
// step_rows_kernel: one CTA per (row, chunk) of the logits.  It streams one
// chunk of a target or draft row with 16-byte loads, reduces it to the chunk
// max and sum of exp (fp32, MUFU ex2), and for the bonus row (target row K)
// also to the float-float sum of the sampling weights exp(alpha (l - m)).
// The last CTA to finish a row (atomic ticket, no waiting) combines the chunk
// partials into the row's log-sum-exp, gathers the drafted token's logit, and
// for the bonus row draws the bonus token by inverse CDF in vocabulary order.
// The last row of a prompt then runs the prompt's tail in the same CTA:
// importance-weight update, normalisation, ESS, systematic resampling, token
// emission and the KV block-table remap ("Faster LLM Inference via Sequential
// Monte Carlo", section 2 "核心流程" and "系统优化设计").  In SpS mode the tail
// instead runs the acceptance scan of speculative sampling.
#include <cmath>

#include "row_common.cuh"
#include "kernels.h"
#include "smcsd.h"

namespace smcsd {

int chunk_elems(int dtype) { return kThreads * kNV * (dtype == SMC_BF16 ? 8 : 4); }
int chunks_per_row(int dtype, int V) {
  const int ch = chunk_elems(dtype);
  return (V + ch - 1) / ch;
}

struct StepArgs {
  const char *target, *draft;
  const int32_t *tokens;
  int B, N, K, V, nch, mode, use_kv;
  float alpha, ess_frac;
  uint64_t seed;
  uint32_t step;
  Workspace ws;
  StepOutputs out;
  KvArgs kv;
};

// Blocks that hold `len` tokens (64-bit, so a corrupt length cannot overflow).
__device__ __forceinline__ long long nblk(long long len, int bs) { return (len + bs - 1) / bs; }

// ---------------------------------------------------------------------------
// Normalise one prompt's log-weights, compute ESS and, below the threshold,
// resample systematically.  Thread i < N holds lw_i.  On return s_anc[i]
// holds the ancestor of particle i for every i < N.
// ---------------------------------------------------------------------------
struct ResampleResult { bool resampled; double ess; };

__device__ ResampleResult normalise_resample(int b, int N, double lw, bool valid, float ess_frac,
                                             uint64_t seed, uint32_t step, unsigned *status,
                                             int *s_anc, double *s_c, double *s_dred) {
  const double kInf = __longlong_as_double(0x7ff0000000000000ll);
  unsigned bits = 0;
  if (valid && (isnan(lw) || lw == kInf)) bits |= SMC_DEV_NONFINITE;
  const double m = block_max_d(valid && !isnan(lw) ? lw : -kInf, s_dred);
  const bool ok = m > -kInf && m < kInf;
  if (threadIdx.x == 0 && m == -kInf) bits |= SMC_DEV_ALL_ZERO_WEIGHT;
  if (bits) raise_status(status, bits);
  const double e = (valid && ok) ? exp(lw - m) : 0.0;
  const double se = block_sum_d(e, s_dred);
  const double big_l = m + log(se);
  const double w = (valid && ok) ? exp(lw - big_l) : 0.0;
  const double w2 = block_sum_d(w * w, s_dred);
  const double ess = 1.0 / w2;
  const bool resample = ok && ess < static_cast<double>(ess_frac) * N;
  int anc = threadIdx.x;
  if (resample) {
    const double c = block_scan_d(w, s_dred);
    if (valid) s_c[threadIdx.x] = c;
    __syncthreads();
    if (valid) {
      const double u0 = philox_uniform(seed, step, b, 0, SMC_PURPOSE_RESAMPLE);
      const double pt = (u0 + threadIdx.x) / N;
      int lo = 0, hi = N - 1;            // smallest j with c_j > pt, clamped to N-1
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_c[mid] > pt) hi = mid; else lo = mid + 1;
      }
      anc = lo;
    }
  }
  if (valid) s_anc[threadIdx.x] = anc;
  __syncthreads();
  return {resample, ess};
}

// ---------------------------------------------------------------------------
// Block-table remap by ancestors and append of n_append tokens, one prompt,
// one CTA.  Reference counts count table references; the free stack of prompt
// b is free_list[b*P .. b*P + free_top[b]).  See smcsd.h (kv_blocktable_remap).
// ---------------------------------------------------------------------------
__device__ void kv_remap_append_block(const KvArgs &kv, int b, int N, const int *s_anc,
                                      bool resampled, int n_append, const Workspace &ws,
                                      int *s_i, int *s_tail) {
  __shared__ int s_flag;
  const int T = kv.T, bs = kv.block_size, P = kv.P;
  const int lo_id = b * P;
  const int tid = threadIdx.x;
  int32_t *tables = kv.tables + static_cast<size_t>(b) * N * T;
  int32_t *seq_len = kv.seq_len + static_cast<size_t>(b) * N;
  int32_t *stack = kv.free_list + static_cast<size_t>(b) * P;
  if (tid == 0) {
    const int top0 = kv.free_top[b];
    s_flag = (top0 < 0 || top0 > P) ? 1 : 0;
    kv.n_cow[b] = 0;
  }
  __syncthreads();
  if (s_flag) {
    if (tid == 0) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
    return;
  }
  auto in_pool = [&](int blk) { return blk >= lo_id && blk < lo_id + P; };

  if (resampled) {
    int32_t *old_t = ws.kv_old_tables + static_cast<size_t>(b) * N * T;
    int32_t *old_l = ws.kv_old_len + static_cast<size_t>(b) * N;
    for (int idx = tid; idx < N * T; idx += kThreads) old_t[idx] = tables[idx];
    for (int i = tid; i < N; i += kThreads) {
      const int len = seq_len[i];
      old_l[i] = len;
      if (len < 0 || nblk(len, bs) > T) s_flag = 1;
    }
    __syncthreads();
    for (int idx = tid; idx < N * T; idx += kThreads) {
      const int i = idx / T, t = idx - (idx / T) * T;
      const int len = old_l[i];
      if (len >= 0 && t < nblk(len, bs) && !in_pool(old_t[idx])) s_flag = 1;
    }
    __syncthreads();
    if (s_flag) {
      if (tid == 0) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
      return;
    }
    // new references first, so no count touches 0 before every increment is in
    for (int idx = tid; idx < N * T; idx += kThreads) {
      const int i = idx / T, t = idx - (idx / T) * T;
      const int a = s_anc[i];
      const int nb_new = static_cast<int>(nblk(old_l[a], bs));
      const int nb_old = static_cast<int>(nblk(old_l[i], bs));
      if (t < nb_new) {
        const int blk = old_t[a * T + t];
        if (!(t < nb_old && old_t[idx] == blk)) atomicAdd(&kv.refcount[blk], 1);
      }
    }
    __syncthreads();
    unsigned *bitmap = ws.kv_bitmap + static_cast<size_t>(b) * ((P + 31) / 32);
    for (int idx = tid; idx < N * T; idx += kThreads) {
      const int i = idx / T, t = idx - (idx / T) * T;
      const int a = s_anc[i];
      const int nb_new = static_cast<int>(nblk(old_l[a], bs));
      const int nb_old = static_cast<int>(nblk(old_l[i], bs));
      if (t < nb_old) {
        const int blk = old_t[idx];
        if (!(t < nb_new && old_t[a * T + t] == blk)) {
          if (atomicSub(&kv.refcount[blk], 1) == 1) {
            const int rel = blk - lo_id;
            atomicOr(&bitmap[rel >> 5], 1u << (rel & 31));
          }
        }
      }
      tables[idx] = old_t[a * T + t];
    }
    for (int i = tid; i < N; i += kThreads) seq_len[i] = old_l[s_anc[i]];
    __syncthreads();
    // push freed blocks in ascending id order
    const int words = (P + 31) / 32;
    int top = kv.free_top[b];
    for (int w0 = 0; w0 < words; w0 += kThreads) {
      const int w = w0 + tid;
      unsigned bits = w < words ? bitmap[w] : 0u;
      int total;
      int pos = top + block_excl_scan_i(__popc(bits), s_i, &total);
      if (bits) bitmap[w] = 0u;
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        if (pos < P) stack[pos] = lo_id + w * 32 + bit;
        ++pos;
      }
      top += total;
    }
    if (top > P) s_flag = 1;                 // counts did not match the tables
    __syncthreads();
    if (tid == 0) kv.free_top[b] = min(top, P);
    if (s_flag) {
      if (tid == 0) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
      return;
    }
    __syncthreads();
  }
  if (n_append <= 0) return;

  // ---- append: fork shared partial tails, then grow ------------------------
  const bool valid = tid < N;
  int len = 0, nb = 0, tail = -1;
  if (valid) {
    len = seq_len[tid];
    if (len < 0 || nblk(len, bs) > T) {
      s_flag = 1;
    } else {
      nb = static_cast<int>(nblk(len, bs));
      if (len % bs) {
        tail = tables[tid * T + nb - 1];
        if (!in_pool(tail)) s_flag = 1;
      }
    }
    s_tail[tid] = tail;
  }
  __syncthreads();
  if (s_flag) {
    if (tid == 0) raise_status(ws.status, SMC_DEV_BAD_BLOCK);
    return;
  }
  int fork = 0;
  if (valid && tail >= 0) {
    for (int i2 = 0; i2 < tid; ++i2) {
      if (s_tail[i2] == tail) { fork = 1; break; }
    }
  }
  const long long nb2 = valid ? nblk(static_cast<long long>(len) + n_append, bs) : 0;
  if (valid && nb2 > T) s_flag = 2;
  const int grow = (valid && nb2 <= T) ? static_cast<int>(nb2) - nb : 0;
  int total_pops, n_forks;
  const int off = block_excl_scan_i(fork + grow, s_i, &total_pops);
  const int cidx = block_excl_scan_i(fork, s_i, &n_forks);
  const int top = kv.free_top[b];
  __syncthreads();
  if (s_flag == 2) {
    if (tid == 0) raise_status(ws.status, SMC_DEV_TABLE_OVERFLOW);
    return;
  }
  if (total_pops > top) {
    if (tid == 0) raise_status(ws.status, SMC_DEV_POOL_EXHAUSTED);
    return;
  }
  if (valid) {
    int k = off;
    if (fork) {
      const int d = stack[top - 1 - k];
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
      const int d = stack[top - 1 - k];
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

// ---------------------------------------------------------------------------
// Prompt tails.
// ---------------------------------------------------------------------------
struct TailSmem {
  double c[SMC_MAX_N];
  double dred[kWarps];
  int anc[SMC_MAX_N];
  int bonus[SMC_MAX_N];
  int tail[SMC_MAX_N];
  int ired[2 * kWarps];
};

__device__ void smc_tail(const StepArgs &a, int b, TailSmem &sm) {
  const int N = a.N, K = a.K, rpp = 2 * K + 1;
  const int tid = threadIdx.x;
  const bool valid = tid < N;
  float lwf = 0.f;
  if (valid) {
    const int part = b * N + tid;
    const RowResult *r = a.ws.results + static_cast<size_t>(part) * rpp;
    double delta = 0.0;
    for (int k = 0; k < K; ++k) {
      const float4 rp = __ldcg(reinterpret_cast<const float4 *>(r + k));
      const float4 rq = __ldcg(reinterpret_cast<const float4 *>(r + K + 1 + k));
      delta += static_cast<double>(a.alpha) * (static_cast<double>(rp.y) - rp.x)
             - (static_cast<double>(rq.y) - rq.x);
    }
    const float4 rb = __ldcg(reinterpret_cast<const float4 *>(r + K));
    if (a.alpha != 1.f) delta += static_cast<double>(rb.z) - static_cast<double>(a.alpha) * rb.x;
    sm.bonus[tid] = __float_as_int(rb.w);
    lwf = static_cast<float>(static_cast<double>(a.out.log_weights[part]) + delta);
  }
  const ResampleResult rr = normalise_resample(b, N, lwf, valid, a.ess_frac, a.seed, a.step,
                                               a.ws.status, sm.anc, sm.c, sm.dred);
  if (valid) {
    const int part = b * N + tid;
    const int anc = sm.anc[tid];
    a.out.log_weights[part] = rr.resampled ? 0.f : lwf;
    a.out.ancestors[part] = anc;
    int32_t *dst = a.out.tokens_out + static_cast<size_t>(part) * (K + 1);
    const int32_t *src = a.tokens + static_cast<size_t>(b * N + anc) * K;
    for (int k = 0; k < K; ++k) dst[k] = src[k];
    dst[K] = sm.bonus[anc];
  }
  if (tid == 0) {
    a.out.ess[b] = static_cast<float>(rr.ess);
    a.out.resampled[b] = rr.resampled ? 1 : 0;
  }
  if (a.use_kv) {
    kv_remap_append_block(a.kv, b, N, sm.anc, rr.resampled, K + 1, a.ws, sm.ired, sm.tail);
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
    const double ratio = exp((static_cast<double>(rp.y) - rp.x) - (static_cast<double>(rq.y) - rq.x));
    const double u = philox_uniform(a.seed, a.step, b, tid, SMC_PURPOSE_ACCEPT);
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
  constexpr bool kExactDiff = sizeof(T) != 4;  // bf16 logits

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
  if (!is_bonus) {
    if (finite_ref) {
      const float mb = mc * kLog2e;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < EPT; e += 2) {
        s0 += fast_exp2(fmaf(x[e], kLog2e, -mb));
        s1 += fast_exp2(fmaf(x[e + 1], kLog2e, -mb));
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
      const float mb = mc * kLog2e;
      const bool need_fast = a.alpha != 1.f;
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        ff_accum(S, weight_term<kExactDiff>(x[e], mc, a.alpha, s_tab));
        if (need_fast) s += fast_exp2(fmaf(x[e], kLog2e, -mb));
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
        if (cm > kNegInf) sum += cs * expf(cm - M);
        else if (cs != 0.f) sum += cs;  // NaN marker of a chunk holding +inf
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        unsigned bits = 0;
        float g = __int_as_float(0x7fc00000);
        if (M == kNegInf) bits |= SMC_DEV_EMPTY_ROW;
        else if (!(sum < -kNegInf) || M == -kNegInf) bits |= SMC_DEV_NONFINITE;
        const float lse = M + logf(sum);
        const int k = j < a.K ? j : j - a.K - 1;
        const int tok = a.tokens[static_cast<size_t>(part) * a.K + k];
        if (tok < 0 || tok >= a.V) bits |= SMC_DEV_BAD_TOKEN;
        else g = Tr::scalar(rowp, tok);
        if (bits) raise_status(a.ws.status, bits);
        a.ws.results[row] = RowResult{lse, g, 0.f, -1};
      }
    }
  } else {
    // bonus row: float-float mass per chunk in absolute units (reference M),
    // then the inverse-CDF draw: which chunk, then which element.
    const float alpha = a.alpha;
    if (warp == 0) {
      float M = kNegInf;
      for (int c = lane; c < a.nch; c += 32) M = fmaxf(M, __ldcg(&pp[c].m));
      M = warp_max(M);
      const bool ok = M > kNegInf && M < -kNegInf;
      auto chunk_mass = [&](int c, ff *val, ff *f) {
        const float cm = __ldcg(&pp[c].m);
        if (ok && cm > kNegInf) {
          *f = ff_norm(weight_term<false>(cm, M, alpha, s_tab));  // exp(alpha (m_c - M))
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
          if (ok && cm > kNegInf) fast += __ldcg(&pp[c].s) * expf(cm - M);
        }
        total = ff_add(total, warp_ff_sum(val));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) fast += __shfl_xor_sync(0xffffffffu, fast, o);
      const float u = philox_uniform(a.seed, a.step, part, a.K, SMC_PURPOSE_BONUS);
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
          lse = alpha != 1.f ? M + logf(fast) : lse_alpha;
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
          [&](int64_t i) { return weight_term<kExactDiff>(Tr::scalar(rowp, i), cm, alpha, s_tab); },
          s_ff, s_int);
    }
    if (tid == 0) a.ws.results[row].tok = tok;
  }

  // ---- last row of the prompt: the prompt's tail ---------------------------
  __syncthreads();
  const int b = part / a.N;
  if (tid == 0) {
    __threadfence();
    const unsigned t = atomicAdd(&a.ws.prompt_ticket[b], 1u);
    s_last = t == static_cast<unsigned>(a.N * rpp - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) a.ws.prompt_ticket[b] = 0u;
  __shared__ TailSmem tail_sm;
  if (a.mode == 0) smc_tail(a, b, tail_sm);
  else sps_tail(a, b, tail_sm);
}

// ---------------------------------------------------------------------------
// Standalone resampling and remap kernels: one CTA per prompt.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
resample_kernel(int N, float ess_frac, uint64_t seed, uint32_t step, float *log_weights,
                int32_t *ancestors, float *ess, int32_t *resampled, unsigned *status) {
  __shared__ TailSmem sm;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const bool valid = tid < N;
  const float lwf = valid ? log_weights[static_cast<size_t>(b) * N + tid] : 0.f;
  const ResampleResult rr = normalise_resample(b, N, lwf, valid, ess_frac, seed, step, status,
                                               sm.anc, sm.c, sm.dred);
  if (valid) {
    log_weights[static_cast<size_t>(b) * N + tid] = rr.resampled ? 0.f : lwf;
    ancestors[static_cast<size_t>(b) * N + tid] = sm.anc[tid];
  }
  if (tid == 0) {
    ess[b] = static_cast<float>(rr.ess);
    resampled[b] = rr.resampled ? 1 : 0;
  }
}

__global__ void __launch_bounds__(kThreads)
kv_remap_kernel(int N, KvArgs kv, const int32_t *ancestors, const int32_t *resampled,
                int n_append, Workspace ws) {
  __shared__ TailSmem sm;
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
  kv_remap_append_block(kv, b, N, sm.anc, res, n_append, ws, sm.ired, sm.tail);
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_step_rows(const Shape &s, int mode, const void *target, const void *draft,
                             const int32_t *tokens, const StepOutputs &out, const KvArgs *kv,
                             const Workspace &ws, cudaStream_t stream) {
  StepArgs a{};
  a.target = static_cast<const char *>(target);
  a.draft = static_cast<const char *>(draft);
  a.tokens = tokens;
  a.B = s.B; a.N = s.N; a.K = s.K; a.V = s.V;
  a.nch = chunks_per_row(s.dtype, s.V);
  a.mode = mode;
  a.alpha = s.alpha; a.ess_frac = s.ess_frac; a.seed = s.seed; a.step = s.step;
  a.ws = ws;
  a.out = out;
  a.use_kv = kv != nullptr;
  if (kv) a.kv = *kv;
  const long long rows = static_cast<long long>(s.B) * s.N * (2 * s.K + 1);
  const long long grid = rows * a.nch;
  const int esz = s.dtype == SMC_BF16 ? 2 : 4;
  const bool vec = aligned16(target) && aligned16(draft) &&
                   (static_cast<long long>(s.V) * esz) % 16 == 0;
  dim3 g(static_cast<unsigned>(grid)), blk(kThreads);
  if (s.dtype == SMC_BF16) {
    if (vec) step_rows_kernel<bf16_tag, true><<<g, blk, 0, stream>>>(a);
    else step_rows_kernel<bf16_tag, false><<<g, blk, 0, stream>>>(a);
  } else {
    if (vec) step_rows_kernel<float, true><<<g, blk, 0, stream>>>(a);
    else step_rows_kernel<float, false><<<g, blk, 0, stream>>>(a);
  }
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
  kv_remap_kernel<<<s.B, kThreads, 0, stream>>>(s.N, kv, ancestors, resampled, n_append, ws);
  return cudaGetLastError();
}

}  // namespace smcsd
