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

// Token range [b, e) of sequence s from a device cu_seqlens array, checked
// before use: 0 <= cu[s] <= cu[s + 1] <= total.  A malformed pair gives the
// empty range and false (the caller records KDA_ERR_SHAPE), so no access
// outside [0, total) follows from it.
__device__ __forceinline__ bool seq_range(const int32_t *cu, int s, int64_t total, int64_t &b,
                                          int64_t &e) {
  const int64_t x = cu[s], y = cu[s + 1];
  if (x < 0 || x > y || y > total) {
    b = e = 0;
    return false;
  }
  b = x;
  e = y;
  return true;
}

// First snapshot row of sequence s (length len) from snap_offsets, checked:
// the sequence's rows [offs[s], offs[s + 1]) must hold exactly len / 64
// snapshots inside [0, offs[n_seq]) (the rows the caller allocated).  -1 if
// not (the caller then writes no snapshot for s and records KDA_ERR_SHAPE).
__device__ __forceinline__ int64_t snap_first_row(const int64_t *offs, int s, int n_seq,
                                                  int64_t len) {
  const int64_t a = offs[s], b = offs[s + 1], rows = offs[n_seq];
  if (a < 0 || b - a != len / 64 || b > rows) return -1;
  return a;
}

// Per-step decay factor exp(g) of one key channel, g = gmin * sigmoid(eA * z)
// with eA = exp(A_h) (report page, sec. 2.1.1).  z = +inf gives exp(gmin),
// z = -inf gives 1.
__device__ __forceinline__ float decay_factor(float gmin, float eA, float z) {
  const float sig = 1.0f / (1.0f + expf(-eA * z));
  return expf(gmin * sig);
}

}  // namespace kda
