// Segment-parallel scan of the KDA state for long sequences with few
// (sequence, head) chains (the single-GPU form of what the report page calls
// "KDA Context Parallelism", Key claims / Infrastructure).
//
// The recurrence is affine in the state: over one segment of chunks,
// S_out = M S_in + N, with N the segment's state when it starts from zero and
// M = prod_chunks (Diag(e^{G_last}) - K'^T Wk) its dk x dk transition (the
// state reached from S_in = I with v = 0).  Both come from the tensor-core
// prefill kernel run over every segment at once; this kernel then chains the
// segments of each (sequence, head) in fp32:
//
//   S_start[0] = S0,   S_start[g + 1] = M_g S_start[g] + N_g,
//
// and the prefill kernel runs once more from the segment start states to
// produce the outputs and snapshots.  Work per segment here is one
// 128 x 128 x 128 fp32 product (2.1 MFLOP), negligible next to the prefill.
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kScanThreads = 256;
constexpr int kD = 128;

// One CTA per (sequence, head).  States, M and N use the [rows, H, dk, dv]
// layout with rows = sequence * n_segs + segment.
__global__ void __launch_bounds__(kScanThreads)
segment_combine_kernel(const float *__restrict__ M, const float *__restrict__ N,
                       const float *__restrict__ S0, float *__restrict__ S_start,
                       float *__restrict__ S_final, int n_segs, int H) {
  extern __shared__ float4 scan_smem[];
  float *Sc = reinterpret_cast<float *>(scan_smem);  // current state [dk][dv]
  const int s = blockIdx.y, h = blockIdx.x, tid = threadIdx.x;
  const size_t sz = static_cast<size_t>(kD) * kD;
  for (int x = tid; x < kD * kD; x += kScanThreads)
    Sc[x] = S0 ? S0[(static_cast<size_t>(s) * H + h) * sz + x] : 0.f;
  __syncthreads();
  // thread -> rows i0 = tid / 2 (one row), columns j0 .. j0 + 63
  const int i0 = tid >> 1, j0 = (tid & 1) * 64;
  for (int g = 0; g < n_segs; ++g) {
    const size_t row = (static_cast<size_t>(s) * n_segs + g) * H + h;
    float4 *start = reinterpret_cast<float4 *>(S_start + row * sz);
    const float4 *cur = reinterpret_cast<const float4 *>(Sc);
    for (int x = tid; x < kD * kD / 4; x += kScanThreads) start[x] = cur[x];
    float acc[64];
    const float *Nrow = N + row * sz + static_cast<size_t>(i0) * kD + j0;
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = Nrow[j];
    const float *Mrow = M + row * sz + static_cast<size_t>(i0) * kD;
    for (int k = 0; k < kD; ++k) {
      const float m = Mrow[k];
      const float4 *srow = reinterpret_cast<const float4 *>(Sc + k * kD + j0);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 v = srow[j];
        acc[4 * j] += m * v.x;
        acc[4 * j + 1] += m * v.y;
        acc[4 * j + 2] += m * v.z;
        acc[4 * j + 3] += m * v.w;
      }
    }
    __syncthreads();  // every thread has read the old state
#pragma unroll
    for (int j = 0; j < 64; ++j) Sc[i0 * kD + j0 + j] = acc[j];
    __syncthreads();
  }
  if (S_final) {
    float4 *dst = reinterpret_cast<float4 *>(S_final + (static_cast<size_t>(s) * H + h) * sz);
    const float4 *cur = reinterpret_cast<const float4 *>(Sc);
    for (int x = tid; x < kD * kD / 4; x += kScanThreads) dst[x] = cur[x];
  }
}

}  // namespace

cudaError_t segment_combine_launch(const float *M, const float *N, const float *S0,
                                   float *S_start, float *S_final, int n_seq, int n_segs, int H,
                                   cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kD) * kD * sizeof(float);
  cudaError_t err = cudaFuncSetAttribute(segment_combine_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const dim3 grid(static_cast<unsigned>(H), static_cast<unsigned>(n_seq));
  segment_combine_kernel<<<grid, kScanThreads, smem, stream>>>(M, N, S0, S_start, S_final,
                                                               n_segs, H);
  return cudaGetLastError();
}

}  // namespace kda
