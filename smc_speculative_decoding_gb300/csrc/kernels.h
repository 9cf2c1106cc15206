// Internal interface between the C-ABI layer (api.cu) and the kernels.
// Host-only declarations; no CUDA types beyond cudaStream_t.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "smcsd.h"

namespace smcsd {

// smc_step's host-side argument checks (shape, dtype, KV struct, null
// pointers): SMC_OK or the error code smc_step would return.
int32_t check_step_args(const smc_params *p, const void *target_logits,
                        const void *draft_logits, const int32_t *draft_tokens,
                        const float *log_weights, const int32_t *tokens_out,
                        const int32_t *ancestors, const float *ess, const int32_t *resampled,
                        const smc_kv *kv);

// Per-(row, chunk) partial of a vocabulary reduction: chunk max m, fast fp32
// sum s of exp(l - m), and the float-float sum (shi, slo) of the sampling
// weights exp(alpha (l - m)) (bonus rows only).
struct RowPartial { float m, s, shi, slo; };

// Per-row result: log-sum-exp, gathered logit of the drafted token, the
// log-sum-exp of alpha*l (bonus rows), and the bonus token (bonus rows).
struct RowResult { float lse, g, lse_alpha; int32_t tok; };

struct KvArgs {
  int32_t *tables, *seq_len, *refcount, *free_list, *free_top, *cow_pairs, *n_cow;
  int32_t T, block_size, P;
};

// Workspace carve-up shared by every entry point.
constexpr int kWrecPerParticle = 16;  // two 64-bit records for each of 8 warps
constexpr int kCounterWords = 8;      // one copy of the counters, work_counter[0] on

struct Workspace {
  unsigned *status;          // [1]  device status bits
  unsigned long long *wrec;  // [B*N * kWrecPerParticle] tagged weight records (plain step):
                             // (call tag << 32) | float bits, head and tail per warp
  unsigned *bonus_done;      // [B]  particles of the prompt whose bonus token is published
  unsigned *row_ticket;      // [rows]
  unsigned *sps_ticket_a;    // [B]
  unsigned *sps_ticket_b;    // [B]
  unsigned *kv_bitmap;       // [B * ceil(P/32)]
  unsigned *work_counter;    // [2]  next fast-row item, next bonus chunk (streaming kernel)
  unsigned *exit_counter;    // [1]  CTAs of the streaming kernel that finished
  unsigned *rows_done;       // [1]  streaming CTAs whose partials are published (plain step)
  unsigned *tail_ticket;     // [1]  prompt CTAs past their waits (plain step)
  unsigned *sps_retry_n;     // [1]  prompts queued for the SpS retry pass
  unsigned *sps_retry_done;  // [1]  retry-pass CTAs that finished
  unsigned *sps_ff_n;        // [1]  prompts queued for the float-float pass
  int32_t *sps_retry;        // [B]  the queued prompts
  int32_t *sps_ff;           // [B]  prompts the fp32 pass left to the float-float pass
  RowPartial *partials;      // [rows * nch]  (per-chunk kernel)
  float2 *item_part;         // [rows * nch * 8]  (m, s) per work item and warp (streaming kernel)
  int4 *bonus_part;          // [B * N * nch * 8] (ref bits, fixed-point sum lo, hi, -)
                             // per chunk and warp
  RowResult *results;        // [rows]
  int32_t *sps_rej;          // [B]  first rejected position, -1 if none
  float4 *sps_stats;         // [B]  precise (lse_p hi, lo, lse_q hi, lo) of row j
  float4 *sps_part_pq;       // [B * snch * 2] per-chunk stats of rows p_j, q_j (SpS chunks)
  float2 *sps_part_r;        // [B * snch]     per-chunk residual mass
  int32_t *kv_old_tables;    // [B * N * T]
  int32_t *kv_old_len;       // [B * N]
  size_t zero_bytes;         // bytes from the start that must start at zero
  size_t bonus_part_half;    // int4s in one of the two bonus_part buffers
};

struct Shape {
  int B, N, K, V, dtype;     // dtype 0 = f32, 1 = bf16
  float alpha, ess_frac;
  uint64_t seed;
  uint32_t step;
  float tscale;              // 1/T of a temperature T (1: none)
  const float *potential;    // [B*N] log-potential increments, or null
  float top_p;               // nucleus mass (1: none)
};

// Elements per chunk of the row reductions for a dtype.
int chunk_elems(int dtype);
int chunks_per_row(int dtype, int V);
int sps_chunks_per_row(int dtype, int V);  // chunks of the SpS residual kernels

// Lays out `base` for the shape; returns the bytes needed (base may be null).
// The counters (work_counter .. sps_ff_n) and bonus_part come twice; the
// carve points at the first copy, use_workspace_copy(ws, 1) at the second.
size_t carve_workspace(const Shape &s, int T, int P, void *base, Workspace *ws);
void use_workspace_copy(Workspace *ws, unsigned which);
// Alternates 0, 1, 0, ... over the calls that use the workspace at `base`.
unsigned next_workspace_copy(const void *base);

struct StepOutputs {
  float *log_weights;
  int32_t *tokens_out, *ancestors, *resampled, *n_emitted;
  float *ess;
};

// mode 0: SMC step; mode 1: SpS verify (first launch); mode 2: draft
// sampler (K = 0: every row is a bonus row, drawn into out.tokens_out).
cudaError_t launch_step_rows(const Shape &s, int mode, const void *target, const void *draft,
                             const int32_t *tokens, const StepOutputs &out, const KvArgs *kv,
                             const Workspace &ws, cudaStream_t stream);
// One token per row of `logits` [rows, V] from softmax(alpha l), by inverse
// CDF with the DRAFT uniform of (seed, step, row, position).
cudaError_t launch_draft_sample(const Shape &s, const void *logits, int position,
                                int32_t *tokens_out, const Workspace &ws, cudaStream_t stream);
// Per prompt: blocks with a positive reference count, and the blocks the
// particles' token counts fill without sharing.
cudaError_t launch_kv_usage(const Shape &s, const KvArgs &kv, int32_t *used, int32_t *unshared,
                            cudaStream_t stream);
cudaError_t launch_resample(const Shape &s, float *log_weights, int32_t *ancestors, float *ess,
                            int32_t *resampled, const Workspace &ws, cudaStream_t stream);
cudaError_t launch_kv_remap(const Shape &s, const KvArgs &kv, const int32_t *ancestors,
                            const int32_t *resampled, int n_append, const Workspace &ws,
                            cudaStream_t stream);
// Events recorded around the row pass of every later step (null: none).
void set_row_timing_events(cudaEvent_t begin, cudaEvent_t end);
void set_step_clock(unsigned long long *stamps, unsigned *counter, int capacity);
cudaError_t launch_selftest_wait(unsigned *words, int kind, unsigned limit, cudaStream_t stream);

cudaError_t launch_sps_residual(const Shape &s, const void *target, const void *draft,
                                int32_t *tokens_out, const Workspace &ws, cudaStream_t stream);

}  // namespace smcsd
