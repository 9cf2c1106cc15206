// Arguments of the step's row kernels, shared by the translation units that
// launch them (smc_step.cu, topp.cu).
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

#include "kernels.h"
#include "row_common.cuh"

namespace smcsd {

struct StepArgs {
  const char *target, *draft;
  const int32_t *tokens;
  int B, N, K, V, nch, mode, use_kv;
  float alpha, ess_frac;
  float tscale;               // 1/T: every logit is scaled by it
  float balpha;               // exponent of the bonus distribution: alpha * tscale
  bool bonus_lse;             // the bonus row's own log-sum-exp is needed (alpha != 1)
  int bonus_purpose, bonus_position;  // Philox purpose and position of the bonus draw
  const float *potential;     // [B*N] log-potential increments, or null
  uint64_t seed;
  uint32_t step;
  uint32_t call_tag;          // nonzero, different for every call (tags the weight records)
  Workspace ws;
  StepOutputs out;
  KvArgs kv;
};

// The logit row `row` of the step: for particle part = row / (2K+1) and
// j = row mod (2K+1), target position j for j <= K, else draft position
// j - K - 1.
template <typename T>
__device__ __forceinline__ const char *row_base(const StepArgs &a, int row) {
  const int rpp = 2 * a.K + 1;
  const int part = row / rpp, j = row - part * rpp;
  constexpr int ESZ = ChunkGeom<T>::kESZ;
  return j <= a.K
      ? a.target + (static_cast<size_t>(part) * (a.K + 1) + j) * static_cast<size_t>(a.V) * ESZ
      : a.draft + (static_cast<size_t>(part) * a.K + (j - a.K - 1)) * static_cast<size_t>(a.V) * ESZ;
}

static inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Opts a kernel into `bytes` of dynamic shared memory.  A launch whose static
// plus dynamic shared memory exceeds 48 KB needs this even when the dynamic
// part alone does not, so it is set whenever a kernel takes any.
template <typename K>
static inline cudaError_t allow_dyn_smem(K kernel, size_t bytes) {
  if (bytes == 0) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

// The top-p restriction of every row after the row combine (topp.cu).
cudaError_t launch_topp(const StepArgs &a, int dtype, float top_p, long long rows,
                        cudaStream_t stream);

}  // namespace smcsd
