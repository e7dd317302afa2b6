// Chunk preparation of the two-pass tensor-core prefill: everything in a
// chunk that does not depend on the state, for every (chunk, head) of the
// batch at once, written as one record per (chunk, head) (kda_split.cuh) for
// the sequential state pass.
//
// Algebra ("Kimi K3 Technical Report - Open Frontier Intelligence", sec. 2.1
// chunkwise-parallel form, sec. 2.1.1 / Fig. 3 bounded decay), for one chunk
// of 64 tokens r with per-step decays a_r = e^{g_r} (per key channel) and
// inclusive cumulative log-decay G_r:
//
//   A_kk[r][i] = beta_r sum_c k_r k_i e^{G_r - G_i}    (i < r)
//   P[r][i]    =        sum_c q_r k_i e^{G_r - G_i}    (i <= r)
//   T = (I + A_kk)^{-1},  T' = T diag(beta),  Wk = T' (K e^G),  U = T' V
//   record: [-Wk ; -Q e^G], K' = K e^{G_last - G}, U, -P, gamma = e^{G_last}
//
// Every causal tile is a dense matmul.  The chunk is cut into four 16-token
// sub-tiles R.  With F_r the decay product from the start of r's sub-tile
// through r, Lam_R the sub-tile's total and B_i = Lam_J / F_i the product
// after i to the end of its sub-tile J:
//
//  - an off-diagonal tile (i in J < R <= r's sub-tile) factors as
//      e^{G_r - G_i} = F_r * prod_{J<M<R} Lam_M * B_i,
//    every factor <= 1: the tiles run on the tcgen05 tensor cores with fp16
//    operands [k_r F_r ; q_r F_r] (B) and k_i B_i prod Lam (A, one stacked
//    block of rows per R), fp32 accumulation in TMEM;
//  - a diagonal tile (i, r in one sub-tile) needs e^{G_r - G_i} = F_r / F_i,
//    whose second factor reaches e^{-16 gmin} = e^80 -- the lower bound
//    gmin = -5 is what keeps it inside the 8-bit exponent range.  These four
//    16 x 16 tiles run as warp-level tf32 MMAs (m16n8k8) whose fragments are
//    exactly the elements each thread holds: no operand goes through shared
//    memory.
//
// The element mapping follows the m16n8k8 fragment layout: warp w owns
// sub-tile R = w / 2 and the key channels 64 (w % 2) .. + 63; lane (g, t)
// owns tokens 16R + g and 16R + g + 8 and, for k-step s = 0..7, channels
// 64 (w % 2) + 8s + 2t and + 1.  The running products along the tokens of a
// sub-tile are shuffle scans over g.
//
// Per task (persistent CTAs, two per SM: 256 threads, 108 KB of shared
// memory, 256 TMEM columns each):
//   TMA    z (prefetched while the previous chunk runs), q and k, v (after
//          the operand build)
//   SIMT   gate, scans, sub-tile totals; then every operand (packed fp32x2
//          arithmetic over each thread's channel pairs): [KE ; QE] and the
//          stacked Kc (fp16, shared memory), -K e^G (bf16, over k), and
//          -Q e^G, K' (fp16, straight to the record); diagonal tiles by mma.sync
//   MMA    off-diagonal A_kk / P tiles (M128 N128 K128, fp16)
//   SIMT   A_kk to shared memory (fp32, transposed), -P to the record;
//          T by diagonal-block column updates, then block forward
//          substitution for the off-diagonal blocks in three levels of
//          16 x 16 products; T' = T diag(beta) as bf16 hi | lo
//   MMA    T'(-K e^G) and T'V, each one M128 N128 K128 product with hi and lo
//          concatenated along K (bf16)
//   SIMT   -Wk and U (fp16) to the record
// Every mbarrier wait is bounded; a wait that gives up records
// KDA_ERR_TIMEOUT and the CTA stops cleanly.
#include "kda_common.cuh"
#include "kda_pdl.cuh"
#include "kda_sm100.cuh"
#include "kda_split.cuh"
#include "kda_tc_common.cuh"

namespace kda {

namespace {

using namespace sm100;
using namespace tcx;

constexpr int CP_THREADS = 256;

// Shared-memory map (byte offsets from the 1024-aligned dynamic base).
constexpr uint32_t SM_Q = 0;              // q tile [64 tok x 128] bf16, then v
constexpr uint32_t SM_K = 16 * KiB;       // k tile, rewritten in place as -K e^G (bf16, MN-major)
constexpr uint32_t SM_Z = 32 * KiB;       // z tile (the next chunk's once the scans have read it)
constexpr uint32_t SM_KQ = 48 * KiB;      // [KE ; QE] fp16 K-major, 128 rows; then scratch
constexpr uint32_t SM_KC = 80 * KiB;      // stacked Kc fp16 K-major, 96 rows
constexpr uint32_t KC_REGION = 12 * KiB;  // its two 64-channel regions
// T' = T diag(beta) as bf16 hi (K columns 0..63) | lo (64..127), K-major, in
// the Kc tile once the off-diagonal MMA has read it.  Its M = 128 operand
// reads rows 64..127 of each region too (they only feed unused rows of D):
// those of the lo region end 24 KiB after SM_TP, inside the Kc tile.
constexpr uint32_t SM_TP = SM_KC;
// scratch of the triangular inverse, in the [KE ; QE] tile once the off-diagonal MMA is done
constexpr uint32_t SM_AKK = SM_KQ;                     // fp32 [64][68]: A_kk transposed, [i][r]
constexpr uint32_t SM_TD = SM_AKK + 64 * 68 * 4;       // fp32 [4][16][17]: diagonal blocks of T
constexpr uint32_t SM_XS = SM_TD + 4 * 16 * 17 * 4;    // fp32 [10][16][17]: block products
static_assert(SM_XS + 10 * 16 * 17 * 4 <= SM_KC, "inverse scratch overflows the KE/QE tile");
static_assert(6 * 16 * 17 * 4 <= 64 * 68 * 4, "level-2 blocks overflow the A_kk tile");
constexpr uint32_t SM_MISC = 104 * KiB;
constexpr uint32_t MS_BAR_Z = SM_MISC;            // mbarriers: z in, q/k in, v in, MMA done
constexpr uint32_t MS_BAR_QK = SM_MISC + 8;
constexpr uint32_t MS_BAR_V = SM_MISC + 16;
constexpr uint32_t MS_BAR_MMA = SM_MISC + 24;
constexpr uint32_t MS_TMEM = SM_MISC + 32;
constexpr uint32_t MS_TASK = SM_MISC + 64;        // 3 task slots of 32 bytes
constexpr uint32_t MS_BETA = SM_MISC + 160;       // [64] fp32
constexpr uint32_t MS_LAM = SM_MISC + 416;        // [64 channel pairs][4 sub-tiles][2] fp32
constexpr uint32_t MS_NSQ = MS_LAM + 128 * 16;    // [64 tok][2 halves] (k.k, q.q) partial sums
// The M = 128 Kc operand reads 128 rows of each region: its second region's
// unused rows 96..127 end 28 KiB after SM_KC, so the allocation reaches there.
constexpr uint32_t CP_SMEM_BYTES = SM_KC + KC_REGION + 16 * KiB;
static_assert(MS_NSQ + 64 * 2 * 8 <= CP_SMEM_BYTES, "misc area");
static_assert(CP_SMEM_BYTES <= 110 * KiB, "two CTAs per SM");

constexpr uint32_t TILE = 16 * KiB;  // a [64 tok x 128] 2-byte tile (two 8 KiB regions)
constexpr uint32_t TM_COLS = 256;
constexpr uint32_t TM_WK = 0;        // off-diagonal A_kk/P, then T'(-K e^G) = -Wk
constexpr uint32_t TM_U = 128;       // T'V

constexpr uint32_t kWaitPolls = 1u << 24;
constexpr int kTmaThread = 96;       // lane 0 of warp 3 (idle in both TMEM read-outs)
constexpr int kTaskThread = 224;     // lane 0 of warp 7 (idle in both TMEM read-outs)

constexpr uint32_t ID_OFF = idesc_mma(128, 128, kFmtF16, kFmtF16, 0, 0);   // K-major x K-major
constexpr uint32_t ID_TPROD = idesc_mma(128, 128, kFmtBF16, kFmtBF16, 0, 1);

struct CpParams {
  const kda_bf16 *beta;
  const float *A;
  float gmin;
  const int32_t *cu_seqlens;   // or NULL: equal lengths fixed_len
  const int32_t *chunk_start;  // varlen: first chunk of each sequence, [n_seq + 1]
  const int2 *chunk_info;      // varlen: first token and length of every chunk
  int64_t fixed_len;
  int n_seq, H, h0, hg;        // heads h0 .. h0 + hg - 1 of H
  unsigned pre;
  uint8_t *rec;                // records [chunk][head in group]
  int *status;
};

__device__ __forceinline__ uint32_t tf32_rna(float x) {
  return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}

// Raw bf16 global load kept where it is written (a prefetch the compiler must
// not sink to its use), predicated inside the instruction: raw keeps its
// value when `take` is 0, so no select waits for the load here.
__device__ __forceinline__ void ldg_u16_prefetch(unsigned short &raw, const kda_bf16 *ptr,
                                                 int take) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p ld.global.nc.u16 %0, [%1];\n\t}"
      : "+h"(raw)
      : "l"(ptr), "r"(take));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(gmin * sigmoid(eA * z)) with c1 = -eA log2(e), c2 = gmin log2(e).
__device__ __forceinline__ float fast_decay2(float c1, float c2, float z) {
  return ex2_approx(c2 * rcp_approx(1.0f + ex2_approx(c1 * z)));
}

__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(a, b);
  const float2 h = unpack_bf16x2(hi);
  lo = pack_bf16x2(a - h.x, b - h.y);
}

__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One warp: C[16x16] (two 16x8 fragments) += X[16x16] Y[16x16] in tf32, X and
// Y fp32 in shared memory (row strides ldx, ldy); XT / YT: given transposed.
template <bool XT = false, bool YT = false>
__device__ __forceinline__ void warp_mma16(const float *X, int ldx, const float *Y, int ldy,
                                           float (&c)[2][4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  auto xa = [&](int row, int col) { return XT ? X[col * ldx + row] : X[row * ldx + col]; };
  auto yb = [&](int row, int col) { return YT ? Y[col * ldy + row] : Y[row * ldy + col]; };
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int k0 = 8 * ks;
    const uint32_t a0 = tf32_rna(xa(g, k0 + t)), a1 = tf32_rna(xa(g + 8, k0 + t));
    const uint32_t a2 = tf32_rna(xa(g, k0 + t + 4)), a3 = tf32_rna(xa(g + 8, k0 + t + 4));
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
      mma_m16n8k8_tf32(c[nt], a0, a1, a2, a3, tf32_rna(yb(k0 + t, 8 * nt + g)),
                       tf32_rna(yb(k0 + t + 4, 8 * nt + g)));
  }
}

// 4 x 4 transpose of 32-bit words across the four lanes t = lane & 3 of a
// quad: lane t holds x[j] = W[j][t] and ends with x[j] = W[t][j].
__device__ __forceinline__ void quad_transpose(uint32_t (&x)[4], int t) {
  {
    const bool hi = (t & 2) != 0;
    const uint32_t s0 = hi ? x[0] : x[2], s1 = hi ? x[1] : x[3];
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 2);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 2);
    if (hi) { x[0] = r0; x[1] = r1; } else { x[2] = r0; x[3] = r1; }
  }
  {
    const bool odd = (t & 1) != 0;
    const uint32_t s0 = odd ? x[0] : x[1], s1 = odd ? x[2] : x[3];
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
    if (odd) { x[0] = r0; x[2] = r1; } else { x[1] = r0; x[3] = r1; }
  }
}

// Byte offset of the 16-byte chunk `ch` (8 two-byte elements) of row r in a
// 128-byte-swizzled tile (one 64-element region).
__device__ __forceinline__ uint32_t chunk_off(int r, int ch) {
  return static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(ch ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(CP_THREADS, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_v,
                  const CpParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const Smem S{smem, sb};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((sb & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
    if (tid == 0) atomicOr(p.status, KDA_ERR_UNSUPPORTED);
    return;
  }
  // a dependent launch: the inputs, the chunk table and the workspace (the
  // previous head group's state pass reads it) are only touched from here on
  grid_launch_dependents();
  grid_dependency_wait();
  const int H = p.H;
  const int64_t cps = p.cu_seqlens ? 0 : (p.fixed_len + 63) / 64;
  const int64_t n_tasks =
      (p.cu_seqlens ? static_cast<int64_t>(p.chunk_start[p.n_seq]) : p.n_seq * cps) * p.hg;
  const int n_iter = n_tasks > static_cast<int64_t>(blockIdx.x)
                         ? static_cast<int>((n_tasks - blockIdx.x + gridDim.x - 1) / gridDim.x)
                         : 0;

  // Task n of this CTA: global task blockIdx.x + n * gridDim.x = chunk-major,
  // head-minor.  Resolved two tasks ahead into a three-slot ring by one thread
  // of a warp that is idle at that point; a varlen chunk's first token and
  // length come from the chunk table (one load, beside that of A).
  auto put_task = [&](int n) {
    const int64_t task = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(n) * gridDim.x;
    const int64_t c = task / p.hg;
    const int hh = p.h0 + static_cast<int>(task % p.hg);
    int64_t t0, L;
    if (p.cu_seqlens) {
      const int2 ci = p.chunk_info[c];
      t0 = ci.x;
      L = ci.y;
    } else {
      const int64_t q = c / cps;
      t0 = q * p.fixed_len + 64 * (c - q * cps);
      L = min(static_cast<int64_t>(64), (q + 1) * p.fixed_len - t0);
    }
    const uint32_t slot = sb + MS_TASK + 32u * static_cast<uint32_t>(n % 3);
    S.u128(slot) = make_uint4(static_cast<uint32_t>(t0), static_cast<uint32_t>(t0 >> 32),
                              static_cast<uint32_t>(L), static_cast<uint32_t>(hh));
    S.f32(slot + 16) = -__expf(p.A[hh]) * 1.4426950408889634f;
  };
  struct Task {
    int64_t t0;
    int L, h;
    float dc1;
  };
  auto task_of = [&](int n) -> Task {
    const uint32_t slot = sb + MS_TASK + 32u * static_cast<uint32_t>(n % 3);
    const uint4 w = S.u128(slot);
    return {static_cast<int64_t>((static_cast<uint64_t>(w.y) << 32) | w.x), static_cast<int>(w.z),
            static_cast<int>(w.w), S.f32(slot + 16)};
  };

  const uint32_t bar_z = sb + MS_BAR_Z, bar_qk = sb + MS_BAR_QK, bar_v = sb + MS_BAR_V,
                 bar_mma = sb + MS_BAR_MMA;
  if (tid == 0) {
    mbar_init(bar_z, 1);
    mbar_init(bar_qk, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_v);
  }
  if (tid == kTaskThread) {
    if (n_iter > 0) put_task(0);
    if (n_iter > 1) put_task(1);
  }
  if (warp == 0) {
    tmem_alloc(sb + MS_TMEM, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + MS_TMEM);

  // Loads: z on its own barrier (the next chunk's z comes in as soon as this
  // chunk's scans have read it), q and k together (once this chunk's T'
  // products are done), v once the operand build has read q.
  auto load2 = [&](uint32_t dst, const CUtensorMap *map, int n, uint32_t bar) {
    const Task tk = task_of(n);
    tma_load_3d(dst, map, 0, tk.h, static_cast<int>(tk.t0), bar);
    tma_load_3d(dst + REG64, map, 64, tk.h, static_cast<int>(tk.t0), bar);
  };
  auto issue_z = [&](int n) {
    mbar_expect_tx(bar_z, TILE);
    load2(sb + SM_Z, &tm_z, n, bar_z);
  };
  auto issue_qk = [&](int n) {
    mbar_expect_tx(bar_qk, 2 * TILE);
    load2(sb + SM_Q, &tm_q, n, bar_qk);
    load2(sb + SM_K, &tm_k, n, bar_qk);
  };
  auto issue_v = [&](int n) {
    mbar_expect_tx(bar_v, TILE);
    load2(sb + SM_Q, &tm_v, n, bar_v);
  };
  if (tid == kTmaThread && n_iter > 0) {
    issue_z(0);
    issue_qk(0);
  }
  bool z_pending = n_iter > 0, qk_pending = n_iter > 0, v_pending = false;
  bool mma_pending = false, aborted = false;
  uint32_t mma_phase = 0;
  float range_max = 0.f;

  auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait_bounded(bar, parity, kWaitPolls);
    if (__syncthreads_or(ok ? 0 : 1)) {
      if (tid == 0) atomicOr(p.status, KDA_ERR_TIMEOUT);
      return false;
    }
    return true;
  };
  auto wait_mma = [&]() -> bool {
    const bool ok = wait_all(bar_mma, mma_phase);
    if (ok) {
      mma_phase ^= 1u;
      mma_pending = false;
    }
    tc_fence_after();
    return ok;
  };

  // Element mapping (see the header): sub-tile R, channel half hc, fragment (g, t).
  const int R = warp >> 1, hc = warp & 1, g = lane >> 2, t = lane & 3;
  const int ra = 16 * R + g, rb = ra + 8;               // this thread's two tokens
  const uint32_t reg = static_cast<uint32_t>(hc) * REG64;  // 64-channel region of a [64 x 128] tile
  const float c2 = p.gmin * 1.4426950408889634f;
  const bool l2n = (p.pre & KDA_PRE_L2NORM_QK) != 0;
  const int quad = warp & 3;                            // TMEM lane quadrant of this warp
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);

  for (int n = 0; n < n_iter && !aborted; ++n) {
    const Task tk = task_of(n);
    const int L = tk.L, h = tk.h;
    const int64_t task = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(n) * gridDim.x;
    uint8_t *rec = p.rec + static_cast<size_t>(task) * kRecBytes;
    // this chunk's beta (raw bits, widened after the operand build)
    unsigned short beta_raw = 0;
    if (tid < 64)
      ldg_u16_prefetch(beta_raw, p.beta + static_cast<size_t>(tk.t0 + min(tid, L - 1)) * H + h,
                       tid < L);

    if (!wait_all(bar_z, n & 1)) { aborted = true; break; }
    z_pending = false;

    // ---- phase 1: gate, running products along the tokens, sub-tile totals --------------
    // F[s][0..3] = (ra, c), (ra, c + 1), (rb, c), (rb, c + 1) for c = 64 hc + 8 s + 2 t.
    float F[8][4];
    const bool ina = ra < L, inb = rb < L;
    // four k-steps at a time: 16 independent gate values, then each scan round
    // over all 16, so the shuffle and transcendental latencies overlap
#pragma unroll
    for (int s0 = 0; s0 < 8; s0 += 4) {
      float x[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t off = reg + static_cast<uint32_t>(4 * t);
        const float2 za = unpack_bf16x2(S.u32(sb + SM_Z + off + chunk_off(ra, s0 + u)));
        const float2 zb = unpack_bf16x2(S.u32(sb + SM_Z + off + chunk_off(rb, s0 + u)));
        x[u][0] = ina ? fast_decay2(tk.dc1, c2, za.x) : 1.f;
        x[u][1] = ina ? fast_decay2(tk.dc1, c2, za.y) : 1.f;
        x[u][2] = inb ? fast_decay2(tk.dc1, c2, zb.x) : 1.f;
        x[u][3] = inb ? fast_decay2(tk.dc1, c2, zb.y) : 1.f;
      }
      // inclusive products over g (lanes 4 apart) for tokens ra and rb separately
#pragma unroll
      for (int d = 1; d < 8; d <<= 1) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float y = __shfl_up_sync(0xffffffffu, x[u][e], 4 * d);
            if (g >= d) x[u][e] *= y;
          }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // tokens rb continue from the product of all eight ra tokens (held at g = 7)
        const float ta0 = __shfl_sync(0xffffffffu, x[u][0], 28 + t);
        const float ta1 = __shfl_sync(0xffffffffu, x[u][1], 28 + t);
        F[s0 + u][0] = x[u][0];
        F[s0 + u][1] = x[u][1];
        F[s0 + u][2] = x[u][2] * ta0;
        F[s0 + u][3] = x[u][3] * ta1;
        if (g == 7) {  // the sub-tile's totals Lam_R of channels c, c + 1, as one pair
          const int c = 64 * hc + 8 * (s0 + u) + 2 * t;
          S.u64(sb + MS_LAM + 32 * (c >> 1) + 8 * R) =
              make_uint2(__float_as_uint(F[s0 + u][2]), __float_as_uint(F[s0 + u][3]));
        }
      }
    }
    // q and k (loaded since the previous chunk's T' products); the barrier also
    // ends every read of z: the next chunk's z may come in
    if (!wait_all(bar_qk, n & 1)) { aborted = true; break; }
    qk_pending = false;
    if (tid == kTmaThread && n + 1 < n_iter) issue_z(n + 1);
    z_pending = n + 1 < n_iter;
    if (l2n) {
      // sums of squares of this warp's 64 channels of tokens ra, rb (k and q)
      float ska = 0.f, skb = 0.f, sqa = 0.f, sqb = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = reg + static_cast<uint32_t>(4 * t);
        const float2 ka = unpack_bf16x2(S.u32(sb + SM_K + off + chunk_off(ra, s)));
        const float2 kb = unpack_bf16x2(S.u32(sb + SM_K + off + chunk_off(rb, s)));
        const float2 qa = unpack_bf16x2(S.u32(sb + SM_Q + off + chunk_off(ra, s)));
        const float2 qb = unpack_bf16x2(S.u32(sb + SM_Q + off + chunk_off(rb, s)));
        ska += ka.x * ka.x + ka.y * ka.y;
        skb += kb.x * kb.x + kb.y * kb.y;
        sqa += qa.x * qa.x + qa.y * qa.y;
        sqb += qb.x * qb.x + qb.y * qb.y;
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        ska += __shfl_xor_sync(0xffffffffu, ska, o);
        skb += __shfl_xor_sync(0xffffffffu, skb, o);
        sqa += __shfl_xor_sync(0xffffffffu, sqa, o);
        sqb += __shfl_xor_sync(0xffffffffu, sqb, o);
      }
      if (t == 0) {
        S.u64(sb + MS_NSQ + 16 * ra + 8 * hc) = make_uint2(__float_as_uint(ska), __float_as_uint(sqa));
        S.u64(sb + MS_NSQ + 16 * rb + 8 * hc) = make_uint2(__float_as_uint(skb), __float_as_uint(sqb));
      }
    }
    __syncthreads();  // B1: totals (and norms) in

    // ---- phase 2: operands ------------------------------------------------------------------
    float nka = 1.f, nkb = 1.f, nqa = 1.f, nqb = 1.f;  // 1 / ||row|| with the pre-op
    if (l2n) {
      const uint4 a = S.u128(sb + MS_NSQ + 16 * ra), b = S.u128(sb + MS_NSQ + 16 * rb);
      const float kka = __uint_as_float(a.x) + __uint_as_float(a.z);
      const float qqa = __uint_as_float(a.y) + __uint_as_float(a.w);
      const float kkb = __uint_as_float(b.x) + __uint_as_float(b.z);
      const float qqb = __uint_as_float(b.y) + __uint_as_float(b.w);
      nka = kka > 0.f ? rsqrtf(kka) : 0.f;
      nqa = qqa > 0.f ? rsqrtf(qqa) : 0.f;
      nkb = kkb > 0.f ? rsqrtf(kkb) : 0.f;
      nqb = qqb > 0.f ? rsqrtf(qqb) : 0.f;
    }
    if (!ina) { nka = 0.f; nqa = 0.f; }  // tokens past the chunk's end: zero rows
    if (!inb) { nkb = 0.f; nqb = 0.f; }
    float dacc[4][4];  // diagonal tile: n-tiles KE(ra), KE(rb), QE(ra), QE(rb)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) dacc[i][e] = 0.f;
    // channel pairs (c, c + 1) in packed fp32x2 arithmetic: every factor below is
    // per channel, so the pairs need no duplication
    auto mul2 = [](float2 a, float2 b) { return __fmul2_rn(a, b); };
    const float2 nk2a = make_float2(nka, nka), nk2b = make_float2(nkb, nkb);
    const float2 nq2a = make_float2(nqa, nqa), nq2b = make_float2(nqb, nqb);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int c = 64 * hc + 8 * s + 2 * t;
      const uint32_t off = reg + static_cast<uint32_t>(4 * t);
      float2 ka = unpack_bf16x2(S.u32(sb + SM_K + off + chunk_off(ra, s)));
      float2 kb = unpack_bf16x2(S.u32(sb + SM_K + off + chunk_off(rb, s)));
      float2 qa = unpack_bf16x2(S.u32(sb + SM_Q + off + chunk_off(ra, s)));
      float2 qb = unpack_bf16x2(S.u32(sb + SM_Q + off + chunk_off(rb, s)));
      if (l2n || !ina || !inb) {  // the pre-op's norms; zero rows past the chunk's end
        ka = mul2(ka, nk2a);
        kb = mul2(kb, nk2b);
        qa = mul2(qa, nq2a);
        qb = mul2(qb, nq2b);
      }
      // sub-tile totals Lam_M of channels c, c + 1 (pairs)
      const float4 l01 = *reinterpret_cast<const float4 *>(S.ptr(sb + MS_LAM + 32 * (c >> 1)));
      const float4 l23 = *reinterpret_cast<const float4 *>(S.ptr(sb + MS_LAM + 32 * (c >> 1) + 16));
      const float2 lam[4] = {make_float2(l01.x, l01.y), make_float2(l01.z, l01.w),
                             make_float2(l23.x, l23.y), make_float2(l23.z, l23.w)};
      float2 pre = make_float2(1.f, 1.f), post = pre;  // prod_{M<R}, prod_{M>R}
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if (m < R) pre = mul2(pre, lam[m]);
        if (m > R) post = mul2(post, lam[m]);
      }
      const float2 lr = R == 0 ? lam[0] : R == 1 ? lam[1] : R == 2 ? lam[2] : lam[3];
      const float2 fa = make_float2(F[s][0], F[s][1]), fb = make_float2(F[s][2], F[s][3]);
      const float2 ia = make_float2(rcp_approx(fa.x), rcp_approx(fa.y));
      const float2 ib = make_float2(rcp_approx(fb.x), rcp_approx(fb.y));
      // KE = k F, QE = q F (<= 1): the off-diagonal B operand, rows tok / 64 + tok
      const float2 kea = mul2(ka, fa), keb = mul2(kb, fb), qea = mul2(qa, fa), qeb = mul2(qb, fb);
      const uint32_t kq = sb + SM_KQ + static_cast<uint32_t>(hc) * TILE + static_cast<uint32_t>(4 * t);
      S.u32(kq + chunk_off(ra, s)) = pack_f16x2(kea.x, kea.y);
      S.u32(kq + chunk_off(rb, s)) = pack_f16x2(keb.x, keb.y);
      S.u32(kq + chunk_off(64 + ra, s)) = pack_f16x2(qea.x, qea.y);
      S.u32(kq + chunk_off(64 + rb, s)) = pack_f16x2(qeb.x, qeb.y);
      // -K e^G = -KE prod_{M<R} Lam (bf16, B operand of T'(-K e^G) = -Wk, the
      // record's sign): each thread overwrites exactly the k elements it has just read
      const float2 npre = make_float2(-pre.x, -pre.y);
      const float2 nka2 = mul2(kea, npre), nkb2 = mul2(keb, npre);
      S.u32(sb + SM_K + off + chunk_off(ra, s)) = pack_bf16x2(nka2.x, nka2.y);
      S.u32(sb + SM_K + off + chunk_off(rb, s)) = pack_bf16x2(nkb2.x, nkb2.y);
      // -Q e^G and K' = k B prod_{M>R} Lam (record words; B = Lam_R / F)
      const float2 ba = mul2(lr, ia), bb = mul2(lr, ib);
      const float2 kba = mul2(ka, ba), kbb = mul2(kb, bb);
      // record rows: -Q e^G in A3 rows 64 + tok (two regions of 128 rows), K'
      // in KP (two regions of 64 rows); the four lanes t of a quad write one
      // 16-byte chunk together
      {
        uint8_t *a3 = rec + kRecA3 + hc * 16384 + 4 * t;
        uint8_t *kp = rec + kRecKP + hc * 8192 + 4 * t;
        const float2 nqa2 = mul2(qea, npre), nqb2 = mul2(qeb, npre);
        const float2 kpa = mul2(kba, post), kpb = mul2(kbb, post);
        *reinterpret_cast<uint32_t *>(a3 + chunk_off(64 + ra, s)) = pack_f16x2(nqa2.x, nqa2.y);
        *reinterpret_cast<uint32_t *>(a3 + chunk_off(64 + rb, s)) = pack_f16x2(nqb2.x, nqb2.y);
        *reinterpret_cast<uint32_t *>(kp + chunk_off(ra, s)) = pack_f16x2(kpa.x, kpa.y);
        *reinterpret_cast<uint32_t *>(kp + chunk_off(rb, s)) = pack_f16x2(kpb.x, kpb.y);
      }
      // Kc rows of the later sub-tiles R' > R: k B prod_{R<M<R'} Lam, stacked at
      // rows 0 (R' = 1, 16 rows), 16 (R' = 2, 32 rows), 48 (R' = 3, 48 rows)
      {
        float2 mm = make_float2(1.f, 1.f);
#pragma unroll
        for (int rp = 1; rp < 4; ++rp) {
          if (rp > R) {
            if (rp > R + 1) mm = mul2(mm, rp - 1 == 1 ? lam[1] : rp - 1 == 2 ? lam[2] : lam[3]);
            const int base = rp == 1 ? 0 : rp == 2 ? 16 : 48;
            const uint32_t kc = sb + SM_KC + static_cast<uint32_t>(hc) * KC_REGION +
                                static_cast<uint32_t>(4 * t);
            const float2 xa = mul2(kba, mm), xb = mul2(kbb, mm);
            S.u32(kc + chunk_off(base + ra, s)) = pack_f16x2(xa.x, xa.y);
            S.u32(kc + chunk_off(base + rb, s)) = pack_f16x2(xb.x, xb.y);
          }
        }
      }
      // diagonal tile by mma.sync: A = k / F (rows ra, rb), B = [KE | QE] (tokens ra, rb)
      {
        const float2 kia = mul2(ka, ia), kib = mul2(kb, ib);
        const uint32_t a0 = tf32_rna(kia.x), a1 = tf32_rna(kib.x);
        const uint32_t a2 = tf32_rna(kia.y), a3 = tf32_rna(kib.y);
        mma_m16n8k8_tf32(dacc[0], a0, a1, a2, a3, tf32_rna(kea.x), tf32_rna(kea.y));
        mma_m16n8k8_tf32(dacc[1], a0, a1, a2, a3, tf32_rna(keb.x), tf32_rna(keb.y));
        mma_m16n8k8_tf32(dacc[2], a0, a1, a2, a3, tf32_rna(qea.x), tf32_rna(qea.y));
        mma_m16n8k8_tf32(dacc[3], a0, a1, a2, a3, tf32_rna(qeb.x), tf32_rna(qeb.y));
      }
      // gamma = prod_M Lam_M per key channel (one writer per channel)
      if (R == 0 && g == 0) {
        float* gam = reinterpret_cast<float *>(rec + kRecG);
        *reinterpret_cast<float2 *>(gam + c) = mul2(mul2(lam[0], lam[1]), mul2(lam[2], lam[3]));
      }
    }
    if (tid < 64) {  // this chunk's beta (logits through a sigmoid with the pre-op)
      const float bn = __uint_as_float(static_cast<uint32_t>(beta_raw) << 16);
      const float b = (p.pre & KDA_PRE_SIGMOID_BETA) ? 1.0f / (1.0f + __expf(-bn)) : bn;
      S.f32(sb + MS_BETA + 4 * tid) = tid < L ? b : 0.f;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();  // B2: operands in; q, k are read out

    // ---- off-diagonal A_kk / P tiles on the tensor cores; v streams into the q tile --------
    if (tid == 0) {
      tc_fence_after();
      issue_mma(tmem + TM_WK, sb + SM_KC, false, KC_REGION, sb + SM_KQ, false, TILE, 8, ID_OFF,
                0);
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (tid == kTmaThread) issue_v(n);
    v_pending = true;
    if (!wait_mma()) { aborted = true; break; }
    // the Kc tile is consumed: T' starts at zero there (the inverse writes the
    // lower triangle only; the barriers below order these stores before it)
    for (int x = tid; x < 1024; x += CP_THREADS) S.u128(sb + SM_TP + 16 * x) = make_uint4(0, 0, 0, 0);

    // ---- read-outs: A_kk (transposed, fp32) to shared memory, -P to the record --------------
    // TMEM lane m is stacked row m of Kc: sub-tile R' = 1 for m < 16, 2 for m < 48,
    // 3 for m < 96 (lanes 96..127 carry nothing); its columns r of sub-tile R'
    // hold A_kk / beta_r (KE part, columns 16 R' ..) and P (QE part, 64 + 16 R' ..).
    if (quad < 3) {
      const int m = quad * 32 + lane;
      const int rp = m < 16 ? 1 : m < 48 ? 2 : 3;
      const int i = m - (rp == 1 ? 0 : rp == 2 ? 16 : 48);
      const int wbase = quad == 0 ? 16 : quad == 1 ? 32 : 48;  // the warp's 32-column window
      const bool upper = (16 * rp - wbase) != 0;               // this lane's 16 in the upper half
      float w[32];
      tmem_ld32(t_lane + TM_WK + (warp < 4 ? 0 : 64) + wbase, w);
      tmem_wait_ld();
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = upper ? w[16 + j] : w[j];
      if (warp < 4) {  // A_kk[r][i] = beta_r D[i][r] into row i of the transposed tile
        const uint32_t row = sb + SM_AKK + 4u * static_cast<uint32_t>(i * 68 + 16 * rp);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 b = *reinterpret_cast<const float4 *>(S.ptr(sb + MS_BETA + 4 * (16 * rp + 4 * j)));
          S.u128(row + 16 * j) = make_uint4(
              __float_as_uint(b.x * v[4 * j]), __float_as_uint(b.y * v[4 * j + 1]),
              __float_as_uint(b.z * v[4 * j + 2]), __float_as_uint(b.w * v[4 * j + 3]));
        }
      } else {  // -P[r][i], r in sub-tile R' (all below the diagonal): record row i, chunks 2R', 2R'+1
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          *reinterpret_cast<uint4 *>(rec + kRecP + chunk_off(i, 2 * rp + cc)) = make_uint4(
              pack_f16x2(-v[8 * cc + 0], -v[8 * cc + 1]), pack_f16x2(-v[8 * cc + 2], -v[8 * cc + 3]),
              pack_f16x2(-v[8 * cc + 4], -v[8 * cc + 5]), pack_f16x2(-v[8 * cc + 6], -v[8 * cc + 7]));
      }
    }
    // diagonal tiles: the two channel halves' partial sums meet in the block scratch
    float *xs = reinterpret_cast<float *>(S.ptr(sb + SM_XS));  // [4 R][16 values][32 lanes]
    if (hc == 1) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) xs[(R * 16 + 4 * nt + e) * 32 + lane] = dacc[nt][e];
    }
    tc_fence_before();
    __syncthreads();  // B3
    if (hc == 0) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) dacc[nt][e] += xs[(R * 16 + 4 * nt + e) * 32 + lane];
      // fragment (nt, e): token i = ra (e < 2) or rb (e >= 2), token
      // r = 16 R + 8 (nt & 1) + 2 t + (e & 1); nt < 2: A_kk / beta_r, nt >= 2: P
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e < 2 ? ra : rb, r = 16 * R + 8 * nt + 2 * t + (e & 1);
          S.f32(sb + SM_AKK + 4 * (i * 68 + r)) = S.f32(sb + MS_BETA + 4 * r) * dacc[nt][e];
        }
      // -P row i, chunk (16 R + 8 (nt - 2)) / 8: lanes t hold its words 2t..2t+1 -> transpose
      uint32_t pw[4];
      pw[0] = pack_f16x2(ra <= 16 * R + 2 * t ? -dacc[2][0] : 0.f, ra <= 16 * R + 2 * t + 1 ? -dacc[2][1] : 0.f);
      pw[1] = pack_f16x2(rb <= 16 * R + 2 * t ? -dacc[2][2] : 0.f, rb <= 16 * R + 2 * t + 1 ? -dacc[2][3] : 0.f);
      pw[2] = pack_f16x2(ra <= 16 * R + 8 + 2 * t ? -dacc[3][0] : 0.f,
                         ra <= 16 * R + 9 + 2 * t ? -dacc[3][1] : 0.f);
      pw[3] = pack_f16x2(rb <= 16 * R + 8 + 2 * t ? -dacc[3][2] : 0.f,
                         rb <= 16 * R + 9 + 2 * t ? -dacc[3][3] : 0.f);
      // word j of the quad is (row, chunk) = (ra, 2R), (rb, 2R), (ra, 2R + 1), (rb, 2R + 1)
      quad_transpose(pw, t);
      const int prow = (t & 1) ? rb : ra, pch = 2 * R + (t >> 1);
      *reinterpret_cast<uint4 *>(rec + kRecP + chunk_off(prow, pch)) =
          make_uint4(pw[0], pw[1], pw[2], pw[3]);
    } else {
      // -P is zero for i above r: rows ra, rb, chunks 0 .. 2R - 1 (the earlier sub-tiles)
      for (int x = t; x < 4 * R; x += 4) {
        const int prow = (x & 1) ? rb : ra, pch = x >> 1;
        *reinterpret_cast<uint4 *>(rec + kRecP + chunk_off(prow, pch)) = make_uint4(0, 0, 0, 0);
      }
    }
    __syncthreads();  // B4: A_kk complete

    // ---- T = (I + A_kk)^{-1}: diagonal 16 x 16 blocks by column updates --------------------
    // T' = T diag(beta) as bf16 hi (K columns 0..63) | lo (64..127) of the A tile at SM_K.
    auto put_tp = [&](int r, int col, float v) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      const uint32_t o = sw128_off(r, col, REG64);
      S.u16(sb + SM_TP + o) = *reinterpret_cast<const unsigned short *>(&hi);
      S.u16(sb + SM_TP + REG64 + o) = *reinterpret_cast<const unsigned short *>(&lo);
    };
    {
      // column jc of the inverse of diagonal block Rd: four lanes per column,
      // lane rq holds rows rq, rq + 4, rq + 8, rq + 12; x[m] passed by shuffle
      const int Rd = warp >> 1, jc = 8 * (warp & 1) + (lane >> 2), rq = lane & 3, o = 16 * Rd;
      float x[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = (rq + 4 * k == jc) ? 1.f : 0.f;
#pragma unroll
      for (int mm = 0; mm < 15; ++mm) {
        const float xm = __shfl_sync(0xffffffffu, x[mm >> 2], (lane & ~3) | (mm & 3));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = rq + 4 * k;
          if (r > mm) x[k] -= S.f32(sb + SM_AKK + 4 * ((o + mm) * 68 + o + r)) * xm;
        }
      }
      const float bj = S.f32(sb + MS_BETA + 4 * (o + jc));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = rq + 4 * k;
        S.f32(sb + SM_TD + 4 * ((Rd * 16 + r) * 17 + jc)) = x[k];
        if (r >= jc) put_tp(o + r, o + jc, x[k] * bj);
      }
    }
    __syncthreads();  // B5
    // Off-diagonal blocks: with D = blockdiag(T_RR) and E = D A_off (E_RJ =
    // T_RR A_RJ, strictly block-lower, E^4 = 0), block forward substitution
    // T_RJ = -sum_{J<=M<R} E_RM T_MJ in three dependent levels, with
    // Y_RJ = E_RJ T_JJ and N_31 = E_32 E_21 - E_31:
    //   level 1: E_RJ (six blocks);
    //   level 2: T_10 = -Y_10, T_21 = -Y_21, T_32 = -Y_32; Y_20, Y_31, Y_30, N_31;
    //   level 3: T_20 = E_21 Y_10 - Y_20, T_31 = E_32 Y_21 - Y_31,
    //            T_30 = E_32 Y_20 - N_31 Y_10 - Y_30.
    {
      const float *akk = reinterpret_cast<const float *>(S.ptr(sb + SM_AKK));
      const float *td = reinterpret_cast<const float *>(S.ptr(sb + SM_TD));
      float *bs = reinterpret_cast<float *>(S.ptr(sb + SM_XS));  // E_RJ: 6 blocks of [16][17]
      // level 2 results, in the A_kk tile (read for the last time by level 1)
      float *ys = reinterpret_cast<float *>(S.ptr(sb + SM_AKK));
      auto blk = [&](int i) { return bs + i * 16 * 17; };
      auto yblk = [&](int i) { return ys + i * 16 * 17; };
      auto tdiag = [&](int Rr) { return td + Rr * 16 * 17; };
      // fragment element (nt, hh, e) of a 16 x 16 block: row g + 8 hh, column 8 nt + 2 t + e
      auto frag_off = [&](int nt, int hh) { return (g + 8 * hh) * 17 + 8 * nt + 2 * t; };
      auto put16 = [&](float *dst, const float (&c)[2][4], const float *sub) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int oo = frag_off(nt, hh);
            dst[oo] = c[nt][2 * hh] - (sub ? sub[oo] : 0.f);
            dst[oo + 1] = c[nt][2 * hh + 1] - (sub ? sub[oo + 1] : 0.f);
          }
      };
      auto put_t = [&](int Rr, int J, const float (&c)[2][4], float sgn) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int col = 16 * J + 8 * nt + 2 * t;
          const float b0 = sgn * S.f32(sb + MS_BETA + 4 * col);
          const float b1 = sgn * S.f32(sb + MS_BETA + 4 * (col + 1));
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t hi, lo;
            split_bf16x2(c[nt][2 * hh] * b0, c[nt][2 * hh + 1] * b1, hi, lo);
            const uint32_t o = sw128_off(16 * Rr + g + 8 * hh, col, REG64);
            S.u32(sb + SM_TP + o) = hi;
            S.u32(sb + SM_TP + REG64 + o) = lo;
          }
        }
      };
      float c[2][4];
      auto zero = [&](float (&x)[2][4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e >> 1][e & 1] = x[e >> 1][2 + (e & 1)] = 0.f;
      };
      zero(c);
      if (warp < 6) {  // level 1: E_RJ = T_RR A_RJ (A_kk stored transposed)
        const int Rr = warp == 0 ? 1 : warp < 3 ? 2 : 3;
        const int J = warp == 0 ? 0 : warp < 3 ? warp - 1 : warp - 3;
        warp_mma16<false, true>(tdiag(Rr), 17, akk + (16 * J) * 68 + 16 * Rr, 68, c, lane);
        put16(blk(warp), c, nullptr);  // blocks E_10, E_20, E_21, E_30, E_31, E_32
      }
      __syncthreads();
      // One product call site per level (operands picked per warp), so the
      // loop body stays small enough for the instruction caches.
      if (warp < 7) {  // level 2: Y_10, Y_21, Y_32, Y_20, Y_31, Y_30, E_32 E_21
        zero(c);
        const int xi = warp == 0 ? 0 : warp == 1 ? 2 : warp == 2 ? 5 : warp == 3 ? 1 : warp == 4 ? 4
                     : warp == 5 ? 3 : 5;
        const float *Y = warp == 6 ? blk(2)
                                   : tdiag(warp == 1 || warp == 4 ? 1 : warp == 2 ? 2 : 0);
        warp_mma16(blk(xi), 17, Y, 17, c, lane);
        if (warp < 3) put_t(warp + 1, warp, c, -1.f);  // T_10, T_21, T_32
        // kept for level 3: Y_10, Y_21, Y_20, Y_31, Y_30 in slots 0..4, N_31 in slot 5
        if (warp != 2) put16(yblk(warp < 2 ? warp : warp - 1), c, warp == 6 ? blk(4) : nullptr);
      }
      __syncthreads();
      if (warp < 3) {  // level 3: T_20, T_31, T_30
        zero(c);
        warp_mma16(blk(warp == 0 ? 2 : 5), 17, yblk(warp), 17, c, lane);
        const float *ysub = yblk(warp == 0 ? 2 : warp == 1 ? 3 : 4);
        float c2[2][4];
        zero(c2);
        if (warp == 2) warp_mma16(yblk(5), 17, yblk(0), 17, c2, lane);  // N_31 Y_10
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int oo = frag_off(nt, hh);
            c[nt][2 * hh] -= c2[nt][2 * hh] + ysub[oo];
            c[nt][2 * hh + 1] -= c2[nt][2 * hh + 1] + ysub[oo + 1];
          }
        put_t(warp == 0 ? 2 : 3, warp == 1 ? 1 : 0, c, 1.f);
      }
    }
    fence_proxy_async();  // T' was written by the threads above
    tc_fence_before();
    {
      const bool v_ok = mbar_wait_bounded(bar_v, n & 1, kWaitPolls);
      if (__syncthreads_or(v_ok ? 0 : 1)) {
        if (tid == 0) atomicOr(p.status, KDA_ERR_TIMEOUT);
        aborted = true;
        break;
      }
      v_pending = false;
    }

    // ---- -Wk = T'(-K e^G) -> TMEM 0..127, U = T'V -> 128..255 (hi | lo along K) -------------
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        // A: T' K-major, K-step ks in region ks / 4 (hi, then lo); B: MN-major
        // rows 16 (ks % 4) .. of -K e^G and of v (the same 64 tokens twice)
        const uint32_t a_off = static_cast<uint32_t>(ks >> 2) * REG64 + static_cast<uint32_t>(ks & 3) * 32u;
        const uint32_t b_off = static_cast<uint32_t>(ks & 3) * 2048u;
        const uint64_t ad = sw128_desc(sb + SM_TP, 16u, 1024u) + (a_off >> 4);
        const uint64_t bk = sw128_desc(sb + SM_K, REG64, 1024u) + (b_off >> 4);
        const uint64_t bv = sw128_desc(sb + SM_Q, REG64, 1024u) + (b_off >> 4);
        mma_f16(tmem + TM_WK, ad, bk, ID_TPROD, ks > 0 ? 1u : 0u);
        mma_f16(tmem + TM_U, ad, bv, ID_TPROD, ks > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!wait_mma()) { aborted = true; break; }
    // v (in the q tile) and -K e^G (in the k tile) are consumed: the next task's q, k
    if (tid == kTmaThread && n + 1 < n_iter) issue_qk(n + 1);
    qk_pending = n + 1 < n_iter;

    // ---- -Wk (lanes 0..63, columns 0..127) and U (columns 128..255) to the record ---------
    // (warps 2, 3, 6, 7 reach no TMEM lane below 64: one of them resolves task n + 2)
    if (tid == kTaskThread && n + 2 < n_iter) put_task(n + 2);
    if (quad < 2) {
      const int r = quad * 32 + lane;
      const bool is_u = warp >= 4;
      // two 32-column loads per wait: columns 64 h .. + 63 are region h
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[2][32];
        tmem_ld32(t_lane + (is_u ? TM_U : TM_WK) + 64 * h, v[0]);
        tmem_ld32(t_lane + (is_u ? TM_U : TM_WK) + 64 * h + 32, v[1]);
        tmem_wait_ld();
        if (is_u) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            range_max = fmaxf(range_max, fmaxf(fabsf(v[0][j]), fabsf(v[1][j])));
        }
        uint8_t *base = is_u ? rec + kRecU + h * 8192 : rec + kRecA3 + h * 16384;
#pragma unroll
        for (int hq = 0; hq < 2; ++hq)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(base + chunk_off(r, 4 * hq + j)) = make_uint4(
                pack_f16x2(v[hq][8 * j + 0], v[hq][8 * j + 1]), pack_f16x2(v[hq][8 * j + 2], v[hq][8 * j + 3]),
                pack_f16x2(v[hq][8 * j + 4], v[hq][8 * j + 5]), pack_f16x2(v[hq][8 * j + 6], v[hq][8 * j + 7]));
      }
    }
    tc_fence_before();
    __syncthreads();  // the TMEM columns are read before the next task's MMAs
  }

  // Drain anything still in flight (bounded) before TMEM and shared memory go.
  if (aborted && tid == 0) {
    if (mma_pending) mbar_wait_bounded(bar_mma, mma_phase, kWaitPolls);
    if (z_pending) mbar_wait_bounded(bar_z, 0, kWaitPolls) || mbar_wait_bounded(bar_z, 1, kWaitPolls);
    if (qk_pending) mbar_wait_bounded(bar_qk, 0, kWaitPolls) || mbar_wait_bounded(bar_qk, 1, kWaitPolls);
    if (v_pending) mbar_wait_bounded(bar_v, 0, kWaitPolls) || mbar_wait_bounded(bar_v, 1, kWaitPolls);
  }
  tc_fence_before();
  if (__syncthreads_or(range_max > 65504.f ? 1 : 0) && tid == 0) atomicOr(p.status, KDA_ERR_RANGE);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

bool make_map(CUtensorMap *m, const void *base, int64_t total, int H, int d) {
  EncodeTiledFn fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(total)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(d) * 2 * H};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Persistent grid: two CTAs per SM, each taking (chunk, head) tasks in turn.
cudaError_t chunk_prep_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                              const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                              const int32_t *cu_seqlens, const int32_t *chunk_start,
                              const int2 *chunk_info, int n_seq, int64_t total_tokens,
                              int64_t fixed_len, int H, int dk, int dv, int h0, int hg,
                              int64_t max_tasks, uint8_t *rec, int *status, unsigned pre,
                              int n_sms, cudaStream_t stream) {
  CUtensorMap mq, mk, mz, mv;
  if (!make_map(&mq, q, total_tokens, H, dk) || !make_map(&mk, k, total_tokens, H, dk) ||
      !make_map(&mz, z, total_tokens, H, dk) || !make_map(&mv, v, total_tokens, H, dv))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(chunk_prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(CP_SMEM_BYTES));
  if (err != cudaSuccess) return err;
  CpParams prm{beta, A, gmin, cu_seqlens, chunk_start, chunk_info, fixed_len, n_seq, H, h0,
               hg, pre, rec, status};
  const int64_t ctas = max_tasks < 2LL * n_sms ? max_tasks : 2LL * n_sms;
  if (ctas <= 0) return cudaSuccess;
  return launch_pdl(chunk_prep_kernel, dim3(static_cast<unsigned>(ctas)), dim3(CP_THREADS),
                    CP_SMEM_BYTES, stream, mq, mk, mz, mv, prm);
}

}  // namespace kda
