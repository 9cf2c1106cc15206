// smc_step_noalloc: smc_step for callers that cannot hand the library any
// device scratch memory.
//
// Some callers cannot allocate device memory on their own: a plugin inside a
// serving runtime whose allocator owns all of the GPU's memory, or a
// latency-critical loop where a cudaMalloc (which may synchronise the device)
// is not allowed after start-up.  They have no workspace to pass, so this
// entry point uses a fixed scratch array that lives in the library's own
// device memory instead: the array below, SMC_NOALLOC_WS_BYTES bytes, which
// every GPU that loads the library holds until the process exits.
//
// Host code cannot use the array's name as a device address: on the host it
// names a stand-in, not device memory.  The device address is fetched once
// per device with cudaGetSymbolAddress, with that device current, on the
// first call made while it is current; that first call should therefore come
// before any stream capture.  If the library's device code has not been
// loaded on that device yet (lazy module loading), that lookup loads it, and
// loading reserves the array: make the first call before a host allocator
// takes the device's free memory, or load with eager module loading.  The
// address is kept for the life of the process, so a device reset
// (cudaDeviceReset), after which the array may move, is not supported.  All calls on a device share the one array and
// each call leaves its contents behind, so the counters that must start at
// zero are cleared at the start of every call, and two calls whose work
// overlaps on the GPU (on different streams) race on the array and must not
// be issued.
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "smcsd.h"

namespace smcsd {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_ws[SMC_NOALLOC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;                        // held only while a slot is first filled
std::atomic<void *> g_noalloc_addr[kMaxDevices];  // device address of g_noalloc_ws per device

// Device address of the scratch array on the current device: read without a
// lock once known, looked up under the lock on the first call.
int32_t noalloc_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMC_ERR_CUDA;
  void *p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    p = g_noalloc_addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) {
        return SMC_ERR_CUDA;
      }
      g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return SMC_OK;
}

}  // namespace
}  // namespace smcsd

extern "C" int32_t smc_step_noalloc(const smc_params *p, const void *target_logits,
                                    const void *draft_logits, const int32_t *draft_tokens,
                                    float *log_weights, int32_t *tokens_out, int32_t *ancestors,
                                    float *ess, int32_t *resampled, const smc_kv *kv,
                                    int32_t *status_bits, void *stream) {
  using namespace smcsd;
  // every check smc_step makes, before anything is queued on the stream
  const int32_t arg_rc = check_step_args(p, target_logits, draft_logits, draft_tokens,
                                         log_weights, tokens_out, ancestors, ess, resampled, kv);
  if (arg_rc != SMC_OK) return arg_rc;
  if (!status_bits) return SMC_ERR_ARG;
  const size_t need = smc_workspace_bytes(p, kv);
  if (need == 0) return SMC_ERR_ARG;
  if (need > SMC_NOALLOC_WS_BYTES) return SMC_ERR_WORKSPACE;  // shape too large for the array
  void *ws = nullptr;
  int32_t rc = noalloc_scratch(&ws);
  if (rc != SMC_OK) return rc;
  Shape s{};
  s.B = p->B; s.N = p->N; s.K = p->K; s.V = p->V; s.dtype = p->dtype;
  Workspace w{};
  carve_workspace(s, kv ? kv->T : 0, kv ? kv->P : 0, ws, &w);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // counters, tickets, bitmap and this call's status word start at zero
  if (cudaMemsetAsync(ws, 0, w.zero_bytes, st) != cudaSuccess) return SMC_ERR_CUDA;
  rc = smc_step(p, target_logits, draft_logits, draft_tokens, log_weights, tokens_out, ancestors,
                ess, resampled, kv, ws, SMC_NOALLOC_WS_BYTES, stream);
  if (rc != SMC_OK) return rc;
  if (cudaMemcpyAsync(status_bits, w.status, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) !=
      cudaSuccess) {
    return SMC_ERR_CUDA;
  }
  return SMC_OK;
}
