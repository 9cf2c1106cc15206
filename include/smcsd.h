/*
 * smcsd.h -- C ABI of libsmcsd.so: the per-step particle update of Sequential
 * Monte Carlo speculative decoding (SMC-SD) and single-particle
 * speculative-sampling verification, on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow these pages:
 *   [SMC]  "Faster LLM Inference via Sequential Monte Carlo" (gist.science
 *          explainer; zh section 2 "核心流程" / es section 2 "Metodología:
 *          SMC-SD"): N particles, K drafted tokens each; Score & Bonus,
 *          Reweight by the target/draft ratio, ESS, Resample below a
 *          threshold; always K+1 tokens per particle per step.
 *          Section 2 "系统优化设计" / "Ventajas Sistémicas": KV cache managed on
 *          resampling by pointer exchange and reference counts, no KV copy,
 *          shared prefixes.  Section 3 "通用性扩展": unnormalised targets such
 *          as p^alpha (power sampling).
 *   [SpS]  "Accelerating Large Language Model Decoding with Speculative
 *          Sampling" (blog notes; sections 1 and 4.2 "Modified Rejection
 *          Sampling"): accept drafted tokens with probability min(1, p/q),
 *          resample from max(0, p - q) at the first rejection.
 *
 * Conventions for every entry point
 *   - All array arguments are DEVICE pointers owned by the caller, row-major
 *     and contiguous, unless stated otherwise.  Parameter structs are HOST
 *     pointers, read during the call only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream: it validates its
 *     arguments on the host, launches kernels, and returns without syncing.
 *   - The library allocates no memory.  Scratch space is the caller's
 *     `workspace`, sized by smc_workspace_bytes(), 256-byte aligned, and
 *     zero-filled once before first use (smc_workspace_init).  Each call
 *     leaves the workspace's counters zero again, so it can be reused by the
 *     next call on the same stream without clearing, by calls of the same
 *     entry point and shape (the layout depends on both; another shape or
 *     entry point takes its own workspace, or smc_workspace_init first).  Two
 *     calls that run concurrently must not share a workspace.  Consecutive
 *     steps on one workspace may overlap on the GPU (a step's first kernel
 *     starts while the previous step's last kernel finishes); the library
 *     orders everything they share.
 *   - The library's kernels are launched with programmatic dependent launch,
 *     and the row pass reads its logits as soon as it starts.  So the kernel
 *     before a call in the stream must not let its dependents start before
 *     it has written the inputs (griddepcontrol.launch_dependents /
 *     cudaTriggerProgrammaticLaunchCompletion ahead of its last stores): put
 *     an event wait or any ordinary launch between them if it does.  Kernels
 *     that never trigger early (the default) are waited for in full.
 *   - Return value: SMC_OK or a negative SMC_ERR_* code for a host-side
 *     failure (nothing was launched).  Conditions only the GPU can see (a bad
 *     token id, a non-finite logit, an exhausted block pool ...) set bits of a
 *     status word inside the workspace; read them with smc_device_status().
 *     When a status bit is set the outputs of that call are unspecified.
 *     No kernel traps, and every wait inside a kernel is bounded: a bad input
 *     never hangs or faults the GPU.
 *   - Logits: `dtype` SMC_F32 (IEEE fp32) or SMC_BF16 (bfloat16 stored as
 *     16-bit words).  Arithmetic is fp32 with fp32 accumulation, except the
 *     sampling sums (bonus and residual tokens), which are carried in
 *     float-float (about 48 significant bits) so that the drawn token agrees
 *     with an exact-arithmetic sampler except on genuine near ties.
 *     sps_verify first tries each residual draw in fp32 with a proven bound
 *     on its error, and keeps that draw only when the bound shows it is the
 *     exact one; every other residual draw is made in float-float.
 *   - Randomness: Philox4x32-10, key (seed mod 2^32, seed >> 32), counter
 *     (step, stream, position, purpose); u = (word0 >> 8) * 2^-24.  Streams
 *     and purposes are listed with each entry point.
 */
#ifndef SMCSD_H
#define SMCSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMCSD_ABI_VERSION 1

/* ---- host-side return codes ------------------------------------------- */
#define SMC_OK             0
#define SMC_ERR_ARG       (-1)   /* NULL pointer, size out of range, bad shape */
#define SMC_ERR_DTYPE     (-2)   /* dtype is neither SMC_F32 nor SMC_BF16      */
#define SMC_ERR_WORKSPACE (-3)   /* workspace NULL, too small or misaligned    */
#define SMC_ERR_LAUNCH    (-4)   /* a kernel launch was rejected by CUDA       */
#define SMC_ERR_CUDA      (-5)   /* a CUDA runtime call failed                 */

/* ---- device status bits (smc_device_status) ---------------------------- */
#define SMC_DEV_BAD_TOKEN        0x01  /* drafted token id outside [0, V)          */
#define SMC_DEV_NONFINITE        0x02  /* NaN/+inf logit, or NaN/+inf log-weight   */
#define SMC_DEV_EMPTY_ROW        0x04  /* a logit row that is -inf everywhere      */
#define SMC_DEV_ALL_ZERO_WEIGHT  0x08  /* every particle of a prompt has weight 0  */
#define SMC_DEV_POOL_EXHAUSTED   0x10  /* free-block stack cannot cover an append  */
#define SMC_DEV_TABLE_OVERFLOW   0x20  /* a particle would need more than T blocks */
#define SMC_DEV_BAD_BLOCK        0x40  /* a block id outside its prompt's pool, or a
                                          negative or oversized token count      */
#define SMC_DEV_TIMEOUT          0x80  /* a bounded wait for a bulk copy gave up;
                                          re-initialise the workspace            */

/* ---- limits ------------------------------------------------------------ */
#define SMC_MAX_N  256        /* particles per prompt                           */
#define SMC_MAX_K  64         /* drafted tokens per particle                    */
#define SMC_MAX_V  (1 << 24)  /* vocabulary size                                */

/* ---- Philox purposes (4th counter word) -------------------------------- */
#define SMC_PURPOSE_DRAFT     0  /* stream b*N+n, position k (smc_draft_sample)  */
#define SMC_PURPOSE_BONUS     1  /* stream b*N+n, position K                     */
#define SMC_PURPOSE_ACCEPT    2  /* stream b, position k (sps_verify)            */
#define SMC_PURPOSE_RESIDUAL  3  /* stream b, position j (sps_verify)            */
#define SMC_PURPOSE_RESAMPLE  4  /* stream b, position 0                         */

typedef enum { SMC_F32 = 0, SMC_BF16 = 1 } smc_dtype;

/* Shape and scalars of one step. */
typedef struct {
  int32_t B;          /* prompts (independent problems), >= 1                   */
  int32_t N;          /* particles per prompt, 1..SMC_MAX_N                     */
  int32_t K;          /* drafted tokens per particle, 1..SMC_MAX_K              */
  int32_t V;          /* vocabulary size, 1..SMC_MAX_V                          */
  int32_t dtype;      /* smc_dtype of both logit tensors                        */
  float alpha;        /* target exponent: the target is p^alpha (1 = plain p),
                         finite and > 0                                          */
  float ess_frac;     /* resample iff ESS < ess_frac * N (strict)               */
  uint64_t seed;      /* Philox key                                             */
  uint32_t step;      /* Philox counter word 0; callers advance it per step     */
} smc_params;

/* Paged KV block tables of all prompts (see kv_blocktable_remap).  Every
 * pointer is device memory, int32.  Block ids are global: prompt b owns ids
 * b*P .. b*P+P-1. */
typedef struct {
  int32_t *tables;     /* [B, N, T] block id per table slot, -1 past the used  */
  int32_t *seq_len;    /* [B, N]    tokens held by each particle               */
  int32_t *refcount;   /* [B * P]   table references to each block             */
  int32_t *free_list;  /* [B, P]    prompt b's LIFO stack of free ids          */
  int32_t *free_top;   /* [B]       entries on prompt b's stack                */
  int32_t *cow_pairs;  /* [B, N, 2] out: (src, dst) blocks to copy, in order   */
  int32_t *n_cow;      /* [B]       out: pairs written for prompt b            */
  int32_t T;           /* table slots per particle, >= 1                       */
  int32_t block_size;  /* tokens per block, >= 1                               */
  int32_t P;           /* pool blocks per prompt, >= 1                         */
} smc_kv;

/* Library ABI version (SMCSD_ABI_VERSION of the build). */
int32_t smc_abi_version(void);

/* Human-readable text of a return code or of a device status word. */
const char *smc_strerror(int32_t code);

/* Bytes of workspace that smc_step, sps_verify, smc_resample and
 * kv_blocktable_remap need for shape `p` and, when `kv` is not NULL, for its
 * T and P.  Returns 0 when the shape is invalid. */
size_t smc_workspace_bytes(const smc_params *p, const smc_kv *kv);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). */
int32_t smc_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/* Reads the device status word of `workspace` into *out_bits (host memory):
 * a bitwise OR of SMC_DEV_* over every call since it was last cleared.
 * Synchronises `stream`.  When `clear` is non-zero the word is reset to 0. */
int32_t smc_device_status(void *workspace, int32_t clear, int32_t *out_bits,
                          void *stream);

/* Measurement hook (no counterpart in the pages).  While set, every later
 * smc_step, smc_step_ex, smc_step_noalloc, sps_verify, sps_verify_ex and
 * smc_draft_sample records `rows_begin` on its
 * stream just before the row pass (the kernel that streams the target and
 * draft rows) and `rows_end` just after it, so a caller can time the
 * vocabulary reduction alone with cudaEventElapsedTime.  Both are
 * cudaEvent_t handles passed as void*, created and owned by the caller and
 * created without cudaEventDisableTiming; NULL, NULL (the initial state)
 * turns the hook off.  Recording `rows_end` separates the row pass from the
 * kernels after it, which otherwise start while it drains, so a step timed
 * with the hook on runs slightly longer.  One process-wide setting; set it
 * from the thread that makes the calls.  Returns SMC_OK, or SMC_ERR_ARG when
 * exactly one of the two is NULL. */
int32_t smc_set_row_timing_events(void *rows_begin, void *rows_end);

/* Measurement hook with no counterpart in the pages: a device-side clock of
 * step starts.  When `stamps` is not NULL, every later call's streaming row
 * kernel takes k = (*counter)++ once the kernel before it in the stream has
 * finished, and writes the GPU's global nanosecond timer to stamps[k] if
 * k < capacity.  So consecutive stamps of back-to-back steps differ by the
 * step's period, measured without putting any stream operation between the
 * steps (an event recorded between two steps delays the second one's
 * launch).  `stamps` (uint64 [capacity]) and `counter` (one uint32, set to 0
 * by the caller) are device memory owned by the caller; NULL turns the hook
 * off.  Only the streaming row kernel writes stamps (rows 16-byte aligned
 * with V * element size a multiple of 16).  One process-wide setting; set it
 * from the thread that makes the calls.  Returns SMC_OK, or SMC_ERR_ARG when
 * `stamps` is not NULL and `counter` is NULL or capacity < 1. */
int32_t smc_set_step_clock(uint64_t *stamps, uint32_t *counter, int32_t capacity);

/* Self-test of failure detection, with no counterpart in the pages: runs one
 * of the library's bounded waits against a condition that nothing satisfies,
 * so that it gives up after `poll_limit` polls and raises SMC_DEV_TIMEOUT in
 * the status word, as a real wait that times out does.  kind 0: the counter
 * wait of the step's epilogue kernels (each poll backs off up to about a
 * microsecond); kind 1: the mbarrier wait of the streaming kernel's ring.
 * `workspace` is device memory of at least 8 bytes, zeroed beforehand
 * (smc_workspace_init): its first word is the status word read by
 * smc_device_status, its second a counter that stays 0.  No kernel traps
 * or faults; the context stays usable.  Returns SMC_OK once queued,
 * SMC_ERR_ARG on a bad argument, SMC_ERR_LAUNCH if the launch fails. */
int32_t smc_selftest_bounded_wait(void *workspace, size_t ws_bytes, int32_t kind,
                                  int32_t poll_limit, void *stream);

/* One SMC-SD step for B prompts x N particles ([SMC] section 2).
 *
 * target_logits [B, N, K+1, V]  row k < K scores drafted token k, row K is the
 *                               bonus distribution.
 * draft_logits  [B, N, K, V]    row k is the distribution token k was drawn from.
 * draft_tokens  [B, N, K] int32 drafted tokens x_k.
 * log_weights   [B, N] fp32, in/out: unnormalised log-weights.
 * Outputs (device): tokens_out [B, N, K+1] int32, ancestors [B, N] int32,
 *                   ess [B] fp32, resampled [B] int32 (0/1).
 * kv (host struct of device pointers) may be NULL; when given, the step also
 * runs kv_blocktable_remap's remap and appends K+1 tokens to every particle.
 *
 * Per particle (b, n):  lse_k = log sum_v exp(l_{k,v}) of each row;
 *   delta = sum_{k<K} [alpha (lp_k[x_k] - lseP_k) - (lq_k[x_k] - lseQ_k)]
 *         + (alpha != 1 ? lse(alpha lp_K) - alpha lseP_K : 0);
 *   log_weights += delta;  bonus = inverse-CDF draw, in vocabulary order, from
 *   softmax(alpha lp_K) with u(step, b*N+n, K, BONUS).
 * Per prompt b:  w = softmax(log_weights), ESS = 1 / sum w^2;  if
 *   ESS < ess_frac*N: systematic resampling with u0(step, b, 0, RESAMPLE),
 *   ancestor a_i = min{j : sum_{t<=j} w_t > (u0+i)/N}, and log_weights := 0;
 *   else a_i = i.  tokens_out[b,i] = (x[b,a_i,0..K-1], bonus[b,a_i]).
 * ess[b] is the ESS before resampling. */
int32_t smc_step(const smc_params *p, const void *target_logits,
                 const void *draft_logits, const int32_t *draft_tokens,
                 float *log_weights, int32_t *tokens_out, int32_t *ancestors,
                 float *ess, int32_t *resampled, const smc_kv *kv,
                 void *workspace, size_t ws_bytes, void *stream);

/* Per-call settings of smc_step_ex. */
typedef struct {
  const float *log_potential;  /* DEVICE [B, N] fp32, or NULL: a per-particle
                                  log-potential increment added to delta (a log
                                  reward ratio, or -inf for a particle that
                                  breaks a constraint); NaN or +inf sets
                                  SMC_DEV_NONFINITE                             */
  float temperature;           /* T > 0, finite (1 = none): p and q are
                                  softmax(l / T) wherever they are scored or
                                  sampled; every logit is multiplied by the
                                  fp32 value of 1/T                             */
  float top_p;                 /* nucleus mass in (0, 1] (1 = none); below 1
                                  needs p->alpha == 1                           */
  int32_t reserved[2];         /* must be 0                                     */
} smc_step_opts;

/* smc_step with per-call settings ([SMC] section 3, "通用性扩展": the target
 * may be reweighted by rewards or constraints; [SpS] section 6: decoding at
 * temperature and nucleus settings).  opts may be NULL (= smc_step).  With
 * temperature T and multiplier s = fl32(1/T): every lse and gathered logit
 * is taken of s*l, the bonus is drawn from softmax(fl32(alpha*s) * l_K), and
 * the drafted tokens are taken to come from the tempered draft.  With top_p
 * < 1: each row's distribution pi = softmax(s*l) is restricted to its
 * nucleus (token v kept iff the mass of tokens with a larger logit is below
 * top_p; equal logits go together) and renormalised; a drafted token outside
 * the target's nucleus gives its particle weight 0, one outside the draft's
 * nucleus sets SMC_DEV_BAD_TOKEN; the bonus is drawn from the target's
 * nucleus.  Each row is then read twice more (four times for fp32 logits).
 * With a log-potential phi: delta += phi[b, n] before normalisation.
 * Everything else, and every argument, is as for smc_step. */
int32_t smc_step_ex(const smc_params *p, const smc_step_opts *opts,
                    const void *target_logits, const void *draft_logits,
                    const int32_t *draft_tokens, float *log_weights, int32_t *tokens_out,
                    int32_t *ancestors, float *ess, int32_t *resampled, const smc_kv *kv,
                    void *workspace, size_t ws_bytes, void *stream);

/* The sampling half of one drafted position of the Extend stage ([SMC]
 * section 2: the draft model extends every particle by K tokens, one
 * position at a time).  draft_logits [B, N, V] (the draft's next-token
 * logits of every particle); tokens_out [B, N] int32: x ~ softmax(alpha * l)
 * by inverse CDF in vocabulary order with u(step, b*N+n, position, DRAFT).
 * p->alpha is the draft's inverse temperature (1 = sample q itself); p->K and
 * p->ess_frac are not used; `position` is the drafted position 0..K-1.  The
 * workspace is one sized by smc_workspace_bytes(p, NULL) for the same B, N,
 * V and dtype.  A row that is -inf everywhere gives token -1 and
 * SMC_DEV_EMPTY_ROW; NaN or +inf gives SMC_DEV_NONFINITE. */
int32_t smc_draft_sample(const smc_params *p, const void *draft_logits, int32_t position,
                         int32_t *tokens_out, void *workspace, size_t ws_bytes,
                         void *stream);

/* KV-cache accounting ([SMC] section 2, "系统优化设计": prefix sharing and
 * pointer exchange shrink the KV cache).  For each prompt b: used_blocks[b] =
 * blocks of its pool with a positive reference count; unshared_blocks[b] =
 * sum over its particles of ceil(seq_len / block_size), the blocks N
 * unshared copies would hold.  1 - used/unshared is the saving.  Both outputs
 * are device int32 [B]; p supplies B and N.  Reads the state only. */
int32_t smc_kv_usage(const smc_params *p, const smc_kv *kv, int32_t *used_blocks,
                     int32_t *unshared_blocks, void *stream);

/* Normalise, ESS and systematic resampling alone ([SMC] section 2, Resample),
 * for callers that computed the weights themselves.  log_weights [B, N] fp32
 * in/out (reset to 0 where resampled); ancestors [B, N] int32; ess [B] fp32;
 * resampled [B] int32.  Same rule and uniforms as smc_step. */
int32_t smc_resample(const smc_params *p, float *log_weights,
                     int32_t *ancestors, float *ess, int32_t *resampled,
                     void *workspace, size_t ws_bytes, void *stream);

/* Block-table remap by ancestors, then append n_append tokens per particle
 * ([SMC] section 2, KV Cache 优化: pointer exchange + reference counts).
 *
 * For each prompt b with resampled[b] != 0: particle i takes ancestor a_i's
 * table and token count; each new table reference adds 1 to its block's
 * count and each old one subtracts 1; blocks that reach 0 are pushed on
 * prompt b's free stack in ascending id order.  Then, when n_append > 0,
 * every particle grows by n_append tokens: a partially filled tail block held
 * by several particles stays with the lowest index and every other holder
 * pops a fresh block and records (src, dst) in cow_pairs (the caller copies
 * that block's KV; no KV data is touched here); further blocks are popped in
 * ascending particle order.  Popped blocks get count 1.  If the prompt's pops
 * exceed its stack (SMC_DEV_POOL_EXHAUSTED) or a particle would need more
 * than T blocks (SMC_DEV_TABLE_OVERFLOW), that prompt's append is skipped.
 * ancestors [B, N] int32 and resampled [B] int32 are device arrays (as written
 * by smc_resample).  p supplies B and N. */
int32_t kv_blocktable_remap(const smc_params *p, const smc_kv *kv,
                            const int32_t *ancestors, const int32_t *resampled,
                            int32_t n_append, void *workspace, size_t ws_bytes,
                            void *stream);

/* Speculative-sampling verify of B prompts with one particle each ([SpS]
 * section 4.2; p->N must be 1, p->alpha must be 1, p->B at most 65535).
 *
 * target_logits [B, K+1, V], draft_logits [B, K, V], draft_tokens [B, K].
 * For k = 0..K-1: accept x_k iff u(step, b, k, ACCEPT) < p_k(x_k)/q_k(x_k).
 * At the first rejection j: draw one token by inverse CDF from
 * max(0, p_j - q_j) (or from p_j should that have no mass) with
 * u(step, b, j, RESIDUAL); n_emitted = j+1.  If all are accepted: draw the
 * bonus token from p_K with u(step, b, K, BONUS); n_emitted = K+1.
 * Outputs: tokens_out [B, K+1] int32 (-1 past n_emitted), n_emitted [B]. */
int32_t sps_verify(const smc_params *p, const void *target_logits,
                   const void *draft_logits, const int32_t *draft_tokens,
                   int32_t *tokens_out, int32_t *n_emitted, void *workspace,
                   size_t ws_bytes, void *stream);

/* sps_verify under a temperature and a top-p nucleus ([SpS] section 6
 * evaluates the method at several temperatures and with nucleus sampling).
 * opts may be NULL (sps_verify itself); otherwise opts->log_potential must be
 * NULL (SMC_ERR_ARG: one particle has no weight to tilt), and temperature and
 * top_p are as for smc_step_ex: p and q become softmax(l / T) restricted to
 * their top-p nuclei and renormalised, and the acceptance rule, the residual
 * max(0, p_j - q_j) and the bonus draw run on those.  A drafted token outside
 * the draft's nucleus sets SMC_DEV_BAD_TOKEN; one outside the target's
 * nucleus is always rejected.  Arguments, outputs and errors otherwise as
 * sps_verify. */
int32_t sps_verify_ex(const smc_params *p, const void *target_logits,
                      const void *draft_logits, const int32_t *draft_tokens,
                      int32_t *tokens_out, int32_t *n_emitted,
                      const smc_step_opts *opts, void *workspace, size_t ws_bytes,
                      void *stream);


/* ---- allocation-free variant of smc_step -------------------------------
 * No counterpart in the pages: a deployment convenience.  For callers that
 * cannot allocate device memory themselves (a plugin inside a serving
 * runtime whose allocator owns the GPU's memory, or a loop where cudaMalloc,
 * which may synchronise the device, is not allowed) and so have no
 * workspace to pass.  Same operation, arguments and outputs as smc_step,
 * without workspace arguments: the scratch is a fixed array of
 * SMC_NOALLOC_WS_BYTES bytes in the library's own device memory, which every
 * GPU that loads the library holds until the process exits.  Calls no
 * allocating routine.
 *   - Shapes whose smc_workspace_bytes(p, kv) exceeds SMC_NOALLOC_WS_BYTES
 *     are rejected with SMC_ERR_WORKSPACE before anything is launched.
 *   - status_bits: DEVICE pointer to one int32, written (asynchronously, on
 *     `stream`) with this call's SMC_DEV_* bits.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture.  If the library's device code is not yet
 *     loaded on that device (lazy module loading), the lookup loads it, which
 *     reserves the array: make the first call before a host allocator
 *     reserves the device's free memory, or use eager module loading.
 *   - The address is kept for the life of the process: a device reset
 *     (cudaDeviceReset) is not supported.
 *   - Every argument check of smc_step runs before anything is queued; when
 *     a non-zero code is returned, *status_bits is left unwritten.
 *   - Every call on a device shares the one array; each call clears the
 *     parts that must start at zero.  Calls whose GPU work overlaps (issued
 *     on different streams without ordering) race on the array. */
#define SMC_NOALLOC_WS_BYTES (8u << 20)
int32_t smc_step_noalloc(const smc_params *p, const void *target_logits,
                         const void *draft_logits, const int32_t *draft_tokens,
                         float *log_weights, int32_t *tokens_out, int32_t *ancestors,
                         float *ess, int32_t *resampled, const smc_kv *kv,
                         int32_t *status_bits, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SMCSD_H */
