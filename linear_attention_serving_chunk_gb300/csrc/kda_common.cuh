// Shared device helpers of the KDA CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Chunk length of the chunkwise-parallel prefill and the sub-tile height.
// The lower bound gmin = -5 keeps exp(-16 * gmin) = e^80 below the bf16 /
// fp32 maximum (~e^88.7), so a 16-token sub-tile can be rescaled by its own
// reference without overflow ("Kimi K3 Technical Report - Open Frontier
// Intelligence", sec. 2.1.1, Fig. 3).
constexpr int kChunk = 64;
constexpr int kSub = 16;
constexpr int kSubTiles = kChunk / kSub;

__device__ __forceinline__ float bf2f(kda_bf16 x) {
  return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

__device__ __forceinline__ kda_bf16 f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<kda_bf16 *>(&b);
}

// Per-step decay factor exp(g) of one key channel, g = gmin * sigmoid(eA * z)
// with eA = exp(A_h) (report page, sec. 2.1.1).  z = +inf gives exp(gmin),
// z = -inf gives 1.
__device__ __forceinline__ float decay_factor(float gmin, float eA, float z) {
  const float sig = 1.0f / (1.0f + expf(-eA * z));
  return expf(gmin * sig);
}

}  // namespace kda
