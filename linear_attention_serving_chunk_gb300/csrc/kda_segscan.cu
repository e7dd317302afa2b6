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
// 128 x 128 x 128 fp32 product (2.1 MFLOP), split over 8 CTAs per chain.
#include "kda_common.cuh"

namespace kda {

namespace {

constexpr int kScanThreads = 256;
constexpr int kD = 128;
constexpr int kCols = 16;           // state columns per CTA (the columns never mix)
constexpr int kLd = kD + 4;         // padded row of the staged M (16-byte aligned rows)
constexpr size_t kMBytes = static_cast<size_t>(kD) * kLd * sizeof(float);
constexpr size_t kCombineSmem = 2 * kMBytes + static_cast<size_t>(kD) * kCols * sizeof(float);

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One CTA per (16 state columns, head, sequence); states, M and N use the
// [rows, H, dk, dv] layout with rows = sequence * n_segs + segment.  Column j
// of S_start[g + 1] = M_g S_start[g] + N_g depends only on column j of
// S_start[g], so the 128 columns of a chain run as 8 independent CTAs.  M_g is
// staged in shared memory (rows padded to 132 floats), the next segment's
// copy in flight while this one is used.  Thread (rg, cg) accumulates rows
// rg and rg + 64, columns 4 cg .. 4 cg + 3, over k in ascending order.
__global__ void __launch_bounds__(kScanThreads)
segment_combine_kernel(const float *__restrict__ M, const float *__restrict__ N,
                       const float *__restrict__ S0, float *__restrict__ S_start,
                       float *__restrict__ S_final, int n_segs, int H) {
  extern __shared__ float4 scan_smem[];
  float *Mb = reinterpret_cast<float *>(scan_smem);  // [2][kD][kLd]
  float *Sc = Mb + 2 * kD * kLd;                     // current columns [kD][kCols]
  const int col0 = blockIdx.x * kCols, h = blockIdx.y, s = blockIdx.z, tid = threadIdx.x;
  const size_t sz = static_cast<size_t>(kD) * kD;
  auto state_row = [&](int g) { return (static_cast<size_t>(s) * n_segs + g) * H + h; };
  auto stage_m = [&](int g, int buf) {  // M_g -> Mb[buf]: 4096 16-byte copies
    const float *src = M + state_row(g) * sz;
    float *dst = Mb + buf * kD * kLd;
    for (int x = tid; x < kD * kD / 4; x += kScanThreads) {
      const int r = x >> 5, c4 = x & 31;
      cp_async16(dst + r * kLd + 4 * c4, src + r * kD + 4 * c4);
    }
    cp_async_commit();
  };
  if (n_segs > 0) stage_m(0, 0);
  for (int x = tid; x < kD * kCols; x += kScanThreads) {
    const int r = x / kCols, c = x % kCols;
    Sc[x] = S0 ? S0[(static_cast<size_t>(s) * H + h) * sz + static_cast<size_t>(r) * kD + col0 + c]
               : 0.f;
  }
  const int rg = tid >> 2, cg = tid & 3;
  for (int g = 0; g < n_segs; ++g) {
    const size_t row = state_row(g);
    __syncthreads();  // Sc holds S_start[g]
    for (int x = tid; x < kD * kCols / 4; x += kScanThreads) {
      const int r = x >> 2, c4 = x & 3;
      reinterpret_cast<float4 *>(S_start + row * sz + static_cast<size_t>(r) * kD + col0)[c4] =
          reinterpret_cast<const float4 *>(Sc)[x];
    }
    if (g + 1 < n_segs) {
      stage_m(g + 1, (g + 1) & 1);
      cp_async_wait<1>();  // M_g is in; M_{g+1} may still be in flight
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const float *Ms = Mb + (g & 1) * kD * kLd;
    float acc[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float4 n4 = *reinterpret_cast<const float4 *>(
          N + row * sz + static_cast<size_t>(rg + 64 * r) * kD + col0 + 4 * cg);
      acc[r][0] = n4.x; acc[r][1] = n4.y; acc[r][2] = n4.z; acc[r][3] = n4.w;
    }
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
      const float4 m0 = *reinterpret_cast<const float4 *>(Ms + rg * kLd + k);
      const float4 m1 = *reinterpret_cast<const float4 *>(Ms + (rg + 64) * kLd + k);
      const float ma[2][4] = {{m0.x, m0.y, m0.z, m0.w}, {m1.x, m1.y, m1.z, m1.w}};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 s4 = *reinterpret_cast<const float4 *>(Sc + (k + kk) * kCols + 4 * cg);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          acc[r][0] += ma[r][kk] * s4.x;
          acc[r][1] += ma[r][kk] * s4.y;
          acc[r][2] += ma[r][kk] * s4.z;
          acc[r][3] += ma[r][kk] * s4.w;
        }
      }
    }
    __syncthreads();  // every thread has read the old state
#pragma unroll
    for (int r = 0; r < 2; ++r)
      *reinterpret_cast<float4 *>(Sc + (rg + 64 * r) * kCols + 4 * cg) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
  __syncthreads();
  if (S_final) {
    for (int x = tid; x < kD * kCols / 4; x += kScanThreads) {
      const int r = x >> 2, c4 = x & 3;
      reinterpret_cast<float4 *>(S_final + (static_cast<size_t>(s) * H + h) * sz +
                                 static_cast<size_t>(r) * kD + col0)[c4] =
          reinterpret_cast<const float4 *>(Sc)[x];
    }
  }
}

}  // namespace

cudaError_t segment_combine_launch(const float *M, const float *N, const float *S0,
                                   float *S_start, float *S_final, int n_seq, int n_segs, int H,
                                   cudaStream_t stream) {
  cudaError_t err = cudaFuncSetAttribute(segment_combine_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kCombineSmem));
  if (err != cudaSuccess) return err;
  const dim3 grid(static_cast<unsigned>(kD / kCols), static_cast<unsigned>(H),
                  static_cast<unsigned>(n_seq));
  segment_combine_kernel<<<grid, kScanThreads, kCombineSmem, stream>>>(M, N, S0, S_start,
                                                                       S_final, n_segs, H);
  return cudaGetLastError();
}

}  // namespace kda
