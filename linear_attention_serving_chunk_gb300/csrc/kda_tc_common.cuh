// Shared-memory helpers of the tcgen05 prefill kernels: typed access to the
// dynamic shared memory by shared-window address, bf16 / fp16 packing, rows
// of fp32 values to and from 128-byte-swizzled fp16 tiles, and the issue of
// one product as a chain of tcgen05.mma K-steps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_sm100.cuh"

namespace kda {
namespace tcx {

using namespace sm100;

constexpr uint32_t KiB = 1024;
constexpr uint32_t REG64 = 8 * KiB;    // one 64-column region of a 64-row 2-byte tile
constexpr uint32_t REG128 = 16 * KiB;  // one 64-column region of a 128-row 2-byte tile

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// Shared memory seen by the threads: plain C++ accesses (so the compiler can
// schedule and overlap them) addressed by the same 32-bit shared-window
// addresses the descriptors and TMA use.
struct Smem {
  uint8_t *base;
  uint32_t sb;
  __device__ __forceinline__ uint8_t *ptr(uint32_t a) const { return base + (a - sb); }
  __device__ __forceinline__ uint32_t &u32(uint32_t a) const {
    return *reinterpret_cast<uint32_t *>(ptr(a));
  }
  __device__ __forceinline__ float &f32(uint32_t a) const {
    return *reinterpret_cast<float *>(ptr(a));
  }
  __device__ __forceinline__ uint2 &u64(uint32_t a) const {
    return *reinterpret_cast<uint2 *>(ptr(a));
  }
  __device__ __forceinline__ uint4 &u128(uint32_t a) const {
    return *reinterpret_cast<uint4 *>(ptr(a));
  }
  __device__ __forceinline__ unsigned short &u16(uint32_t a) const {
    return *reinterpret_cast<unsigned short *>(ptr(a));
  }
};

// Write 32 fp32 values (columns [32 q4, 32 q4 + 32) of `row`) as fp16 into a
// 128-byte-swizzled tile whose 64-column regions are `region` bytes apart.
__device__ __forceinline__ void store_row32_f16(const Smem &S, uint32_t tile, int row, int q4,
                                                uint32_t region, const float (&v)[32],
                                                float scale) {
  const uint32_t base =
      tile + static_cast<uint32_t>(q4 >> 1) * region + static_cast<uint32_t>(row) * 128u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t pos = static_cast<uint32_t>((4 * (q4 & 1) + j) ^ (row & 7)) << 4;
    S.u128(base + pos) = make_uint4(pack_f16x2(scale * v[8 * j + 0], scale * v[8 * j + 1]),
                                    pack_f16x2(scale * v[8 * j + 2], scale * v[8 * j + 3]),
                                    pack_f16x2(scale * v[8 * j + 4], scale * v[8 * j + 5]),
                                    pack_f16x2(scale * v[8 * j + 6], scale * v[8 * j + 7]));
  }
}

// Write 16 fp32 values (columns [16 c4, 16 c4 + 16) of `row`, c4 = 0..3) as
// fp16 into a 64-column, 128-byte-swizzled tile.
__device__ __forceinline__ void store_row16_f16(const Smem &S, uint32_t tile, int row, int c4,
                                                const float (&v)[16], float scale) {
  const uint32_t base = tile + static_cast<uint32_t>(row) * 128u;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t pos = static_cast<uint32_t>((2 * c4 + j) ^ (row & 7)) << 4;
    S.u128(base + pos) = make_uint4(pack_f16x2(scale * v[8 * j + 0], scale * v[8 * j + 1]),
                                    pack_f16x2(scale * v[8 * j + 2], scale * v[8 * j + 3]),
                                    pack_f16x2(scale * v[8 * j + 4], scale * v[8 * j + 5]),
                                    pack_f16x2(scale * v[8 * j + 6], scale * v[8 * j + 7]));
  }
}

// Add the 16 fp16 values at columns [16 c4, 16 c4 + 16) of `row` of a
// 64-column, 128-byte-swizzled tile to v.
__device__ __forceinline__ void add_row16_f16(const Smem &S, uint32_t tile, int row, int c4,
                                              float (&v)[16]) {
  const uint32_t base = tile + static_cast<uint32_t>(row) * 128u;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t pos = static_cast<uint32_t>((2 * c4 + j) ^ (row & 7)) << 4;
    const uint4 w = S.u128(base + pos);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[e]));
      v[8 * j + 2 * e] += f.x;
      v[8 * j + 2 * e + 1] += f.y;
    }
  }
}

// Add the 32 fp16 values at columns [32 q4, 32 q4 + 32) of `row` of a
// 128-byte-swizzled tile (regions `region` bytes apart) to v.
__device__ __forceinline__ void add_row32_f16(const Smem &S, uint32_t tile, int row, int q4,
                                              uint32_t region, float (&v)[32]) {
  const uint32_t base =
      tile + static_cast<uint32_t>(q4 >> 1) * region + static_cast<uint32_t>(row) * 128u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t pos = static_cast<uint32_t>((4 * (q4 & 1) + j) ^ (row & 7)) << 4;
    const uint4 w = S.u128(base + pos);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[e]));
      v[8 * j + 2 * e] += f.x;
      v[8 * j + 2 * e + 1] += f.y;
    }
  }
}

// One K-step of a product: K-steps of 16 elements (8 for tf32, the same 32
// bytes).  K-major operands advance 32 bytes per step inside a 128-byte row
// and jump one region per 4 steps; MN-major operands advance 2048 bytes (16
// rows) per step and find their 64-element MN blocks `region` apart.
// A single thread issues the MMAs, and each waits for its descriptors: so the
// descriptor of the operand base is built once (the same for every step of a
// product) and the step's offset is added to its 14-bit address field, which
// cannot carry for shared-memory addresses below 256 KiB.
__device__ __forceinline__ void issue_mma_step(uint32_t d_tmem, uint32_t a_base, bool a_mn,
                                               uint32_t a_region, uint32_t b_base, bool b_mn,
                                               uint32_t b_region, int ks, uint32_t idesc,
                                               uint32_t accumulate, bool tf32 = false) {
  const uint32_t a_off = a_mn ? static_cast<uint32_t>(ks) * 2048u
                              : static_cast<uint32_t>(ks >> 2) * a_region +
                                    static_cast<uint32_t>(ks & 3) * 32u;
  const uint32_t b_off = b_mn ? static_cast<uint32_t>(ks) * 2048u
                              : static_cast<uint32_t>(ks >> 2) * b_region +
                                    static_cast<uint32_t>(ks & 3) * 32u;
  const uint64_t ad = sw128_desc(a_base, a_mn ? a_region : 16u, 1024u) + (a_off >> 4);
  const uint64_t bd = sw128_desc(b_base, b_mn ? b_region : 16u, 1024u) + (b_off >> 4);
  if (tf32)
    mma_tf32(d_tmem, ad, bd, idesc, accumulate);
  else
    mma_f16(d_tmem, ad, bd, idesc, accumulate);
}

// Issue the MMAs of one product, K-step by K-step into one accumulator.
__device__ __forceinline__ void issue_mma(uint32_t d_tmem, uint32_t a_base, bool a_mn,
                                          uint32_t a_region, uint32_t b_base, bool b_mn,
                                          uint32_t b_region, int ksteps, uint32_t idesc,
                                          uint32_t accumulate, bool tf32 = false) {
#pragma unroll
  for (int ks = 0; ks < ksteps; ++ks)
    issue_mma_step(d_tmem, a_base, a_mn, a_region, b_base, b_mn, b_region, ks, idesc,
                   (ks > 0 || accumulate) ? 1u : 0u, tf32);
}

// Host: the driver's cuTensorMapEncodeTiled, looked up once per process
// (nullptr if the driver does not provide it).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn tensor_map_encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &ptr, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return nullptr;
  }();
  return fn;
}

}  // namespace tcx
}  // namespace kda
