// C ABI of libsmcsd.so (declared in include/smcsd.h): argument validation,
// workspace layout and kernel launches.  No allocation, no synchronisation
// except in smc_device_status.
#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "kernels.h"
#include "smcsd.h"

namespace smcsd {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t carve_workspace(const Shape &s, int T, int P, void *base, Workspace *ws) {
  const size_t rows = static_cast<size_t>(s.B) * s.N * (2 * s.K + 1);
  const size_t nch = static_cast<size_t>(chunks_per_row(s.dtype, s.V));
  const size_t words = P > 0 ? static_cast<size_t>(P + 31) / 32 : 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  // region that must start at zero (counters and the freed-block bitmap)
  const size_t o_status = take(sizeof(unsigned));
  const size_t o_wr = take(sizeof(unsigned long long) * s.B * s.N * kWrecPerParticle);
  const size_t o_bd = take(sizeof(unsigned) * s.B);
  const size_t o_rt = take(sizeof(unsigned) * rows);
  const size_t o_sa = take(sizeof(unsigned) * s.B);
  const size_t o_sb = take(sizeof(unsigned) * s.B);
  const size_t o_bm = take(sizeof(unsigned) * s.B * words);
  const size_t o_wc = take(sizeof(unsigned) * 2 * kCounterWords);
  const size_t zero_bytes = off;
  // scratch that every call overwrites before reading
  const size_t o_part = take(sizeof(RowPartial) * rows * nch);
  const size_t o_ip = take(sizeof(float2) * rows * nch * 8);
  const size_t bp_half = static_cast<size_t>(s.B) * s.N * nch * 8;
  const size_t o_bp = take(sizeof(int4) * 2 * bp_half);
  const size_t o_res = take(sizeof(RowResult) * rows);
  const size_t o_rej = take(sizeof(int32_t) * s.B);
  const size_t o_sst = take(sizeof(float4) * s.B);
  const size_t snch = static_cast<size_t>(sps_chunks_per_row(s.dtype, s.V));
  const size_t o_spq = take(sizeof(float4) * s.B * snch * 2);
  const size_t o_spr = take(sizeof(float2) * s.B * snch);
  const size_t o_srt = take(sizeof(int32_t) * s.B);
  const size_t o_sff = take(sizeof(int32_t) * s.B);
  const size_t o_kt = take(sizeof(int32_t) * static_cast<size_t>(s.B) * s.N * (T > 0 ? T : 0));
  const size_t o_kl = take(sizeof(int32_t) * static_cast<size_t>(s.B) * s.N);
  if (ws && base) {
    char *p = static_cast<char *>(base);
    ws->status = reinterpret_cast<unsigned *>(p + o_status);
    ws->wrec = reinterpret_cast<unsigned long long *>(p + o_wr);
    ws->bonus_done = reinterpret_cast<unsigned *>(p + o_bd);
    ws->row_ticket = reinterpret_cast<unsigned *>(p + o_rt);
    ws->sps_ticket_a = reinterpret_cast<unsigned *>(p + o_sa);
    ws->sps_ticket_b = reinterpret_cast<unsigned *>(p + o_sb);
    ws->kv_bitmap = reinterpret_cast<unsigned *>(p + o_bm);
    ws->work_counter = reinterpret_cast<unsigned *>(p + o_wc);
    ws->exit_counter = ws->work_counter + 2;
    ws->rows_done = ws->work_counter + 3;
    ws->tail_ticket = ws->work_counter + 4;
    ws->sps_retry_n = ws->work_counter + 5;
    ws->sps_retry_done = ws->work_counter + 6;
    ws->sps_ff_n = ws->work_counter + 7;
    ws->partials = reinterpret_cast<RowPartial *>(p + o_part);
    ws->item_part = reinterpret_cast<float2 *>(p + o_ip);
    ws->bonus_part = reinterpret_cast<int4 *>(p + o_bp);
    ws->results = reinterpret_cast<RowResult *>(p + o_res);
    ws->sps_rej = reinterpret_cast<int32_t *>(p + o_rej);
    ws->sps_stats = reinterpret_cast<float4 *>(p + o_sst);
    ws->sps_part_pq = reinterpret_cast<float4 *>(p + o_spq);
    ws->sps_part_r = reinterpret_cast<float2 *>(p + o_spr);
    ws->sps_retry = reinterpret_cast<int32_t *>(p + o_srt);
    ws->sps_ff = reinterpret_cast<int32_t *>(p + o_sff);
    ws->kv_old_tables = reinterpret_cast<int32_t *>(p + o_kt);
    ws->kv_old_len = reinterpret_cast<int32_t *>(p + o_kl);
    ws->zero_bytes = zero_bytes;
    ws->bonus_part_half = bp_half;
  }
  return off;
}

void use_workspace_copy(Workspace *ws, unsigned which) {
  if (!which) return;
  ws->work_counter += kCounterWords;
  ws->exit_counter += kCounterWords;
  ws->rows_done += kCounterWords;
  ws->tail_ticket += kCounterWords;
  ws->sps_retry_n += kCounterWords;
  ws->sps_retry_done += kCounterWords;
  ws->sps_ff_n += kCounterWords;
  ws->bonus_part += ws->bonus_part_half;
}

// Consecutive steps on one workspace take alternate copies, so that a step's
// row pass may start while the previous step's tail still reads its own.
unsigned next_workspace_copy(const void *base) {
  static std::mutex mu;
  static std::unordered_map<const void *, unsigned> calls;
  std::lock_guard<std::mutex> lock(mu);
  return calls[base]++ & 1u;
}

static bool shape_ok(const smc_params *p) {
  if (!p) return false;
  if (p->B < 1 || p->N < 1 || p->N > SMC_MAX_N || p->K < 1 || p->K > SMC_MAX_K) return false;
  if (p->V < 1 || p->V > SMC_MAX_V) return false;
  if (!(std::isfinite(p->alpha) && p->alpha > 0.f)) return false;
  if (!std::isfinite(p->ess_frac)) return false;
  const double rows = static_cast<double>(p->B) * p->N * (2 * p->K + 1);
  const double grid = rows * chunks_per_row(p->dtype == SMC_BF16 ? 1 : 0, p->V);
  return grid < 2147483647.0;
}

static bool kv_ok(const smc_params *p, const smc_kv *kv) {
  if (!kv) return true;
  if (kv->T < 1 || kv->block_size < 1 || kv->P < 1) return false;
  if (static_cast<double>(p->B) * kv->P >= 2147483647.0) return false;
  if (static_cast<double>(p->N) * kv->T >= 2147483647.0) return false;
  return kv->tables && kv->seq_len && kv->refcount && kv->free_list && kv->free_top &&
         kv->cow_pairs && kv->n_cow;
}

static Shape to_shape(const smc_params *p) {
  Shape s{};
  s.B = p->B; s.N = p->N; s.K = p->K; s.V = p->V;
  s.dtype = p->dtype;
  s.alpha = p->alpha; s.ess_frac = p->ess_frac;
  s.seed = p->seed; s.step = p->step;
  s.tscale = 1.f;
  s.potential = nullptr;
  s.top_p = 1.f;
  return s;
}

static KvArgs to_kv(const smc_kv *kv) {
  KvArgs k{};
  k.tables = kv->tables; k.seq_len = kv->seq_len; k.refcount = kv->refcount;
  k.free_list = kv->free_list; k.free_top = kv->free_top; k.cow_pairs = kv->cow_pairs;
  k.n_cow = kv->n_cow; k.T = kv->T; k.block_size = kv->block_size; k.P = kv->P;
  return k;
}

// Validates the workspace and carves it; returns SMC_OK or an error.
static int32_t prepare_ws(const smc_params *p, const smc_kv *kv, void *workspace, size_t ws_bytes,
                          Workspace *ws) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return SMC_ERR_WORKSPACE;
  const Shape s = to_shape(p);
  const size_t need = carve_workspace(s, kv ? kv->T : 0, kv ? kv->P : 0, nullptr, nullptr);
  if (ws_bytes < need) return SMC_ERR_WORKSPACE;
  carve_workspace(s, kv ? kv->T : 0, kv ? kv->P : 0, workspace, ws);
  use_workspace_copy(ws, next_workspace_copy(workspace));
  return SMC_OK;
}

}  // namespace smcsd

using namespace smcsd;

extern "C" {

int32_t smc_abi_version(void) { return SMCSD_ABI_VERSION; }

const char *smc_strerror(int32_t code) {
  switch (code) {
    case SMC_OK: return "ok";
    case SMC_ERR_ARG: return "invalid argument (null pointer, size out of range or bad shape)";
    case SMC_ERR_DTYPE: return "unsupported logit dtype";
    case SMC_ERR_WORKSPACE: return "workspace null, misaligned or smaller than smc_workspace_bytes()";
    case SMC_ERR_LAUNCH: return "kernel launch failed";
    case SMC_ERR_CUDA: return "CUDA runtime call failed";
    case SMC_DEV_BAD_TOKEN: return "device: drafted token outside [0, V)";
    case SMC_DEV_NONFINITE: return "device: NaN/+inf logit or log-weight";
    case SMC_DEV_EMPTY_ROW: return "device: logit row is -inf everywhere";
    case SMC_DEV_ALL_ZERO_WEIGHT: return "device: every particle of a prompt has weight 0";
    case SMC_DEV_POOL_EXHAUSTED: return "device: free block stack exhausted";
    case SMC_DEV_TABLE_OVERFLOW: return "device: block table too short";
    case SMC_DEV_BAD_BLOCK: return "device: block id outside its prompt's pool or bad KV state";
    case SMC_DEV_TIMEOUT: return "device: a bounded wait gave up; re-initialise the workspace";
    default: return code > 0 ? "device: several status bits set" : "unknown error";
  }
}

size_t smc_workspace_bytes(const smc_params *p, const smc_kv *kv) {
  if (!shape_ok(p) || (p->dtype != SMC_F32 && p->dtype != SMC_BF16)) return 0;
  if (kv && (kv->T < 1 || kv->P < 1)) return 0;
  return carve_workspace(to_shape(p), kv ? kv->T : 0, kv ? kv->P : 0, nullptr, nullptr);
}

int32_t smc_workspace_init(void *workspace, size_t ws_bytes, void *stream) {
  if (!workspace) return SMC_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    return SMC_ERR_CUDA;
  }
  return SMC_OK;
}

int32_t smc_device_status(void *workspace, int32_t clear, int32_t *out_bits, void *stream) {
  if (!workspace || !out_bits) return SMC_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned bits = 0;
  if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    return SMC_ERR_CUDA;
  }
  *out_bits = static_cast<int32_t>(bits);
  if (clear && cudaMemsetAsync(workspace, 0, sizeof(unsigned), st) != cudaSuccess) return SMC_ERR_CUDA;
  return SMC_OK;
}

int32_t smc_set_row_timing_events(void *rows_begin, void *rows_end) {
  if ((rows_begin == nullptr) != (rows_end == nullptr)) return SMC_ERR_ARG;
  set_row_timing_events(static_cast<cudaEvent_t>(rows_begin),
                        static_cast<cudaEvent_t>(rows_end));
  return SMC_OK;
}

int32_t smc_selftest_bounded_wait(void *workspace, size_t ws_bytes, int32_t kind,
                                  int32_t poll_limit, void *stream) {
  if (!workspace || ws_bytes < 2 * sizeof(unsigned) || (kind != 0 && kind != 1) ||
      poll_limit < 1) {
    return SMC_ERR_ARG;
  }
  if (launch_selftest_wait(static_cast<unsigned *>(workspace), kind,
                           static_cast<unsigned>(poll_limit),
                           static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    return SMC_ERR_LAUNCH;
  }
  return SMC_OK;
}

int32_t smc_set_step_clock(uint64_t *stamps, uint32_t *counter, int32_t capacity) {
  if (stamps && (!counter || capacity < 1)) return SMC_ERR_ARG;
  set_step_clock(reinterpret_cast<unsigned long long *>(stamps), counter, stamps ? capacity : 0);
  return SMC_OK;
}

}  // extern "C"

namespace smcsd {

int32_t check_step_args(const smc_params *p, const void *target_logits,
                        const void *draft_logits, const int32_t *draft_tokens,
                        const float *log_weights, const int32_t *tokens_out,
                        const int32_t *ancestors, const float *ess, const int32_t *resampled,
                        const smc_kv *kv) {
  if (!p) return SMC_ERR_ARG;
  if (p->dtype != SMC_F32 && p->dtype != SMC_BF16) return SMC_ERR_DTYPE;
  if (!shape_ok(p) || !kv_ok(p, kv)) return SMC_ERR_ARG;
  if (!target_logits || !draft_logits || !draft_tokens || !log_weights || !tokens_out ||
      !ancestors || !ess || !resampled) {
    return SMC_ERR_ARG;
  }
  return SMC_OK;
}

static int32_t step_impl(const smc_params *p, const smc_step_opts *opts,
                         const void *target_logits, const void *draft_logits,
                         const int32_t *draft_tokens, float *log_weights, int32_t *tokens_out,
                         int32_t *ancestors, float *ess, int32_t *resampled, const smc_kv *kv,
                         void *workspace, size_t ws_bytes, void *stream) {
  const int32_t arg_rc = check_step_args(p, target_logits, draft_logits, draft_tokens,
                                         log_weights, tokens_out, ancestors, ess, resampled, kv);
  if (arg_rc != SMC_OK) return arg_rc;
  Shape s = to_shape(p);
  if (opts) {
    if (opts->reserved[0] != 0 || opts->reserved[1] != 0) return SMC_ERR_ARG;
    if (!(opts->top_p > 0.f && opts->top_p <= 1.f)) return SMC_ERR_ARG;
    if (opts->top_p < 1.f && p->alpha != 1.f) return SMC_ERR_ARG;
    s.top_p = opts->top_p;
    const float t = opts->temperature;
    if (!(std::isfinite(t) && t > 0.f)) return SMC_ERR_ARG;
    s.tscale = 1.f / t;
    const float balpha = s.alpha * s.tscale;
    if (!(std::isfinite(s.tscale) && s.tscale > 0.f && std::isfinite(balpha) && balpha > 0.f)) {
      return SMC_ERR_ARG;
    }
    s.potential = opts->log_potential;
  }
  Workspace ws{};
  const int32_t rc = prepare_ws(p, kv, workspace, ws_bytes, &ws);
  if (rc != SMC_OK) return rc;
  StepOutputs out{};
  out.log_weights = log_weights;
  out.tokens_out = tokens_out;
  out.ancestors = ancestors;
  out.resampled = resampled;
  out.ess = ess;
  KvArgs k{};
  if (kv) k = to_kv(kv);
  const cudaError_t e = launch_step_rows(s, 0, target_logits, draft_logits, draft_tokens,
                                         out, kv ? &k : nullptr, ws,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMC_OK : SMC_ERR_LAUNCH;
}

}  // namespace smcsd

extern "C" {

int32_t smc_step(const smc_params *p, const void *target_logits, const void *draft_logits,
                 const int32_t *draft_tokens, float *log_weights, int32_t *tokens_out,
                 int32_t *ancestors, float *ess, int32_t *resampled, const smc_kv *kv,
                 void *workspace, size_t ws_bytes, void *stream) {
  return step_impl(p, nullptr, target_logits, draft_logits, draft_tokens, log_weights,
                   tokens_out, ancestors, ess, resampled, kv, workspace, ws_bytes, stream);
}

int32_t smc_step_ex(const smc_params *p, const smc_step_opts *opts,
                    const void *target_logits, const void *draft_logits,
                    const int32_t *draft_tokens, float *log_weights, int32_t *tokens_out,
                    int32_t *ancestors, float *ess, int32_t *resampled, const smc_kv *kv,
                    void *workspace, size_t ws_bytes, void *stream) {
  return step_impl(p, opts, target_logits, draft_logits, draft_tokens, log_weights,
                   tokens_out, ancestors, ess, resampled, kv, workspace, ws_bytes, stream);
}

int32_t smc_draft_sample(const smc_params *p, const void *draft_logits, int32_t position,
                         int32_t *tokens_out, void *workspace, size_t ws_bytes,
                         void *stream) {
  if (!p) return SMC_ERR_ARG;
  if (p->dtype != SMC_F32 && p->dtype != SMC_BF16) return SMC_ERR_DTYPE;
  smc_params q = *p;
  q.K = 1;  // not used; the workspace needs only what K = 1 needs
  if (!shape_ok(&q) || position < 0 || !draft_logits || !tokens_out) return SMC_ERR_ARG;
  Workspace ws{};
  const int32_t rc = prepare_ws(&q, nullptr, workspace, ws_bytes, &ws);
  if (rc != SMC_OK) return rc;
  const cudaError_t e = launch_draft_sample(to_shape(&q), draft_logits, position, tokens_out, ws,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMC_OK : SMC_ERR_LAUNCH;
}

int32_t smc_kv_usage(const smc_params *p, const smc_kv *kv, int32_t *used_blocks,
                     int32_t *unshared_blocks, void *stream) {
  if (!p || !kv || p->B < 1 || p->N < 1 || p->N > SMC_MAX_N || !kv_ok(p, kv) ||
      !used_blocks || !unshared_blocks) {
    return SMC_ERR_ARG;
  }
  const cudaError_t e = launch_kv_usage(to_shape(p), to_kv(kv), used_blocks, unshared_blocks,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMC_OK : SMC_ERR_LAUNCH;
}

int32_t smc_resample(const smc_params *p, float *log_weights, int32_t *ancestors, float *ess,
                     int32_t *resampled, void *workspace, size_t ws_bytes, void *stream) {
  if (!p) return SMC_ERR_ARG;
  if (p->dtype != SMC_F32 && p->dtype != SMC_BF16) return SMC_ERR_DTYPE;
  if (!shape_ok(p) || !log_weights || !ancestors || !ess || !resampled) return SMC_ERR_ARG;
  Workspace ws{};
  const int32_t rc = prepare_ws(p, nullptr, workspace, ws_bytes, &ws);
  if (rc != SMC_OK) return rc;
  const cudaError_t e = launch_resample(to_shape(p), log_weights, ancestors, ess, resampled, ws,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMC_OK : SMC_ERR_LAUNCH;
}

int32_t kv_blocktable_remap(const smc_params *p, const smc_kv *kv, const int32_t *ancestors,
                            const int32_t *resampled, int32_t n_append, void *workspace,
                            size_t ws_bytes, void *stream) {
  if (!p) return SMC_ERR_ARG;
  if (p->dtype != SMC_F32 && p->dtype != SMC_BF16) return SMC_ERR_DTYPE;
  if (!shape_ok(p) || !kv || !kv_ok(p, kv) || !ancestors || !resampled || n_append < 0) {
    return SMC_ERR_ARG;
  }
  Workspace ws{};
  const int32_t rc = prepare_ws(p, kv, workspace, ws_bytes, &ws);
  if (rc != SMC_OK) return rc;
  const cudaError_t e = launch_kv_remap(to_shape(p), to_kv(kv), ancestors, resampled, n_append, ws,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SMC_OK : SMC_ERR_LAUNCH;
}

int32_t sps_verify(const smc_params *p, const void *target_logits, const void *draft_logits,
                   const int32_t *draft_tokens, int32_t *tokens_out, int32_t *n_emitted,
                   void *workspace, size_t ws_bytes, void *stream) {
  return sps_verify_ex(p, target_logits, draft_logits, draft_tokens, tokens_out, n_emitted,
                       nullptr, workspace, ws_bytes, stream);
}

int32_t sps_verify_ex(const smc_params *p, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, int32_t *tokens_out, int32_t *n_emitted,
                      const smc_step_opts *opts, void *workspace, size_t ws_bytes,
                      void *stream) {
  if (!p) return SMC_ERR_ARG;
  if (p->dtype != SMC_F32 && p->dtype != SMC_BF16) return SMC_ERR_DTYPE;
  if (!shape_ok(p) || p->N != 1 || p->alpha != 1.f || p->B > 65535) return SMC_ERR_ARG;
  if (!target_logits || !draft_logits || !draft_tokens || !tokens_out || !n_emitted) {
    return SMC_ERR_ARG;
  }
  Shape s = to_shape(p);
  if (opts) {
    if (opts->reserved[0] != 0 || opts->reserved[1] != 0) return SMC_ERR_ARG;
    if (opts->log_potential) return SMC_ERR_ARG;  // one particle: no weights to tilt
    if (!(opts->top_p > 0.f && opts->top_p <= 1.f)) return SMC_ERR_ARG;
    s.top_p = opts->top_p;
    const float t = opts->temperature;
    if (!(std::isfinite(t) && t > 0.f)) return SMC_ERR_ARG;
    s.tscale = 1.f / t;
    if (!(std::isfinite(s.tscale) && s.tscale > 0.f)) return SMC_ERR_ARG;
  }
  Workspace ws{};
  const int32_t rc = prepare_ws(p, nullptr, workspace, ws_bytes, &ws);
  if (rc != SMC_OK) return rc;
  StepOutputs out{};
  out.tokens_out = tokens_out;
  out.n_emitted = n_emitted;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_step_rows(s, 1, target_logits, draft_logits, draft_tokens, out, nullptr,
                                   ws, st);
  if (e != cudaSuccess) return SMC_ERR_LAUNCH;
  e = launch_sps_residual(s, target_logits, draft_logits, tokens_out, ws, st);
  return e == cudaSuccess ? SMC_OK : SMC_ERR_LAUNCH;
}

}  // extern "C"
