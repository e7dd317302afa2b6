// Restore chunk-boundary states into state slots (prefix caching: "state-aware
// prefix caching" in "Kimi K3 Technical Report - Open Frontier Intelligence",
// Key claims / Infrastructure).  A pure HBM copy: each (row, head) state of
// dk*dv fp32 is read once and written once with 16-byte vectors.
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
snapshot_restore_kernel(const float *__restrict__ snaps, int64_t n_rows,
                        const int64_t *__restrict__ src_idx, float *__restrict__ pool,
                        int n_slots, const int32_t *__restrict__ dst_slots, int H,
                        int state_vec4, int *status) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int64_t row = src_idx[b];
  const int32_t slot = dst_slots[b];
  if (row < 0 || row >= n_rows || slot < 0 || slot >= n_slots) {  // skipped, recorded
    if (threadIdx.x == 0) atomicOr(status, KDA_ERR_SHAPE);
    return;
  }
  const float4 *src = reinterpret_cast<const float4 *>(snaps) +
                      (static_cast<size_t>(row) * H + h) * state_vec4;
  float4 *dst = reinterpret_cast<float4 *>(pool) +
                (static_cast<size_t>(slot) * H + h) * state_vec4;
  for (int x = threadIdx.x; x < state_vec4; x += kCopyThreads) __stcs(dst + x, __ldcs(src + x));
}

}  // namespace

cudaError_t snapshot_restore_launch(const float *snaps, int64_t n_rows, const int64_t *src_idx,
                                    float *pool, int n_slots, const int32_t *dst_slots, int n,
                                    int H, int dk, int dv, int *status, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(n), static_cast<unsigned>(H));
  snapshot_restore_kernel<<<grid, kCopyThreads, 0, stream>>>(
      snaps, n_rows, src_idx, pool, n_slots, dst_slots, H, dk * dv / 4, status);
  return cudaGetLastError();
}

}  // namespace kda
