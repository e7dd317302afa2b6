// Chunkwise-parallel KDA prefill on the sm_103a tensor cores (tcgen05 + TMEM,
// operands staged by TMA), dk, dv in {64, 128}, chunk C = 64.
//
// The kernels are laid out for 128 key and 128 value channels.  A head of 64
// channels runs through the same tiles: its tensor maps have 64 channels, so
// the TMA box over channels 64..127 lies wholly out of bounds and arrives as
// zeros.  Zero key / query channels add nothing to any product, and zero
// value columns keep their state columns and outputs at zero; the state is
// read and written only inside [dk, dv].
//
// Algebra ("Kimi K3 Technical Report - Open Frontier Intelligence", sec. 2.1
// chunkwise-parallel form, sec. 2.1.1 / Fig. 3 bounded decay): for one chunk
// with inclusive cumulative log-decay G_r and chunk-start state S,
//
//   A_kk = strict_lower(diag(beta) (K e^G)(K e^-G)^T),  T = (I + A_kk)^{-1}
//   T'   = T diag(beta),   Wk = T' (K e^G),   U = T' V,   W = U - Wk S
//   P    = tril((Q e^G)(K e^-G)^T),  O = (Q e^G) S + P W
//   S'   = Diag(e^{G_last}) S + (K e^{G_last - G})^T W
//
// Every causal tile of A_kk and P, the diagonal ones included, is one dense
// MMA.  The chunk is split into four 16-row sub-tiles; for the rows of
// sub-tile R the reference is the cumulative decay just before R, so the row
// factor e^{G_r - G_ref} is <= 1 and the column factor e^{G_ref - G_i} is at
// most e^{-16 gmin} = e^80: the lower bound gmin = -5 is what keeps these
// reciprocal factors inside the 8-bit-exponent (bf16 / fp32) range.  The
// transposed products D[i, r] = Khat_R[i] . [K_R e^{G - G_ref}; Q_R e^{G - G_ref}][r]
// are issued two sub-tiles per M = 128 MMA.
//
// Operand precision: the A_kk / P products need the 8-bit exponent range
// (factors up to e^80) and more than bf16's 8-bit mantissa (outputs are
// heavy-tailed and P feeds them directly), so they run as kind::tf32
// (10-bit mantissa, operands rounded to nearest).  T' K~ and T' V use bf16
// operands (V arrives as bf16) with T' = T diag(beta) split into bf16 hi + lo
// tiles, two accumulating MMAs each: the diagonal of T' is beta itself, the
// main write strength, and rounding it to bf16 alone moves the outputs by a
// few 1e-2 RMS.  The state-dependent products use fp16 operands (11-bit
// mantissa; |S|, |W|, |Wk| stay far below 65504 for unit keys and beta in
// [0, 1]).
//
// Per chunk (one CTA per (sequence, head), 512 threads, chunks in order):
//   TMA     q -> A3 lower half, z -> ZB, k -> KB, v -> VB (next chunk's q/z
//           double-buffered, k/v refilled as soon as their MMAs finish)
//   SIMT    gate exp(g), per-sub-tile running products, then every scaled
//           operand in place: k -> K e^G, q -> -(Q e^G), z -> K e^{G_last-G}
//   MMA     A_kk and P (2 x M128 N64 K128, tf32); T on the CUDA cores (the
//           16x16 diagonal blocks by column updates in fp32, the others as
//           (I - E + E^2 - E^3) D with warp-level tf32 products); Wk = T' K~
//           and U = T' V (M128 N128 K64; U lands in the output accumulator D1)
//   serial  D1 += [-Wk; -Q~] S_fp16  (W in rows 0..63, -Q~S in rows 64..127)
//           S_tm = e^{G_last} S_tm + K'^T W   (fp32 state kept in TMEM)
//           D1 += [0; -P] W                   (-O in rows 64..127)
//
// Sizes: shared memory 226 KB (1 CTA / SM), TMEM 384 of 512 columns.
// Every mbarrier wait is bounded; a wait that gives up records
// KDA_ERR_TIMEOUT in the status word and the CTA stops cleanly.
#include "kda_common.cuh"
#include "kda_sm100.cuh"
#include "kda_split.cuh"
#include "kda_tc_common.cuh"

namespace kda {

namespace {

using namespace sm100;
using namespace tcx;

constexpr int TC_THREADS = 512;
constexpr int TD = 128;  // dk = dv handled by this kernel

// Shared-memory map, byte offsets from the (1024-aligned) dynamic base.
constexpr uint32_t SM_A3 = 0;                     // 2 x 32 KiB: [-Wk ; q -> -Q~], K-major
constexpr uint32_t SM_ZB = 64 * KiB;              // 2 x 16 KiB: z -> K'   [tok x dk]
constexpr uint32_t SM_KB = 96 * KiB;              // 16 KiB: k -> K~       [tok x dk]
constexpr uint32_t SM_VB = 112 * KiB;             // 16 KiB: v             [tok x dv]
constexpr uint32_t SM_AP = 128 * KiB;             // 96 KiB work region
constexpr uint32_t SM_APA = SM_AP;                // tf32 [Khat_2p ; Khat_2p+1]   128 x 128
constexpr uint32_t SM_APB = SM_AP + 64 * KiB;     // tf32 [KE_2p; QE_2p; KE_2p+1; QE_2p+1] 64 x 128
constexpr uint32_t SM_AKK = SM_AP;                // fp32 [64][68] A_kk transposed: [i][r] (after the AP MMAs)
constexpr uint32_t SM_TF = SM_AP + 64 * 68 * 4;   // fp32 [64][65] T
constexpr uint32_t SM_TY = SM_AP + 34 * KiB;      // fp32 [10][16][17] block products
constexpr uint32_t SM_SBF = SM_AP;                // [dk x dv] S in fp16, MN-major (after T')
constexpr uint32_t SM_A5 = SM_AP + 48 * KiB;      // [128 x 64] MN-major: [X ; -P] (X unused)
// T' = T diag(beta) as bf16 hi + lo, two [128 x 64] K-major tiles:
// TP = [hi ; 0], TPL = [lo ; 0] (rows 64..127 of D1 carry -O).
constexpr uint32_t SM_TP = SM_AP + 64 * KiB;
constexpr uint32_t SM_TPL = SM_AP + 80 * KiB;
constexpr uint32_t SM_WBF = SM_AP + 64 * KiB;     // [tok x dv] W in fp16 (after T' is used)

constexpr uint32_t SM_MISC = 224 * KiB;
constexpr uint32_t MS_BAR_QZ = SM_MISC + 0;       // 2 mbarriers
constexpr uint32_t MS_BAR_K = SM_MISC + 16;
constexpr uint32_t MS_BAR_MMA = SM_MISC + 24;
constexpr uint32_t MS_TMEM = SM_MISC + 32;
constexpr uint32_t MS_BAR_V = SM_MISC + 40;
constexpr uint32_t MS_BETA = SM_MISC + 64;        // 64 fp32
constexpr uint32_t MS_LAM = SM_MISC + 320;        // [4][128] fp32 sub-tile decay totals
constexpr uint32_t MS_NRM = MS_LAM + 4 * TD * 4;  // [64][2] fp32 1/||k_r||, 1/||q_r|| (pre-op)
constexpr uint32_t TC_SMEM_BYTES = MS_NRM + 64 * 8;
static_assert(SM_TF + 64 * 65 * 4 <= SM_TY, "T scratch overlaps");
static_assert(SM_TY + 10 * 16 * 17 * 4 <= SM_A5, "block scratch overlaps A5");
static_assert(TC_SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t A3_BYTES = 32 * KiB;
constexpr uint32_t TILE_BYTES = 16 * KiB;   // a [64 tok x 128] bf16 tile
// tf32 tiles: 32-column regions of 128-byte rows
constexpr uint32_t APA_REG = 128 * 128;     // 128 rows
constexpr uint32_t APB_REG = 64 * 128;      // 64 rows

// TMEM columns.
constexpr uint32_t TM_AP = 0;     // A_kk / P products, later Wk
constexpr uint32_t TM_D1 = 128;   // U -> W (rows 0..63), -O (rows 64..127)
constexpr uint32_t TM_S = 256;    // fp32 state S (row = key channel)

constexpr uint32_t TM_COLS = 512;

constexpr uint32_t kWaitPolls = 1u << 24;
// TMA loads are issued by lane 0 of warp 4 (a warp with no output stores),
// the MMAs by thread 0.
constexpr int kTmaThread = 128;

// Instruction descriptors (fp32 accumulation).
constexpr uint32_t ID_AP = idesc_mma(128, 64, kFmtTF32, kFmtTF32, 0, 0);      // A_kk / P
constexpr uint32_t ID_TPROD = idesc_mma(128, 128, kFmtBF16, kFmtBF16, 0, 1);  // T' K~, T' V
constexpr uint32_t ID_KMN = idesc_mma(128, 128, kFmtF16, kFmtF16, 0, 1);      // K-major x MN
constexpr uint32_t ID_MNMN = idesc_mma(128, 128, kFmtF16, kFmtF16, 1, 1);     // MN x MN

struct TcParams {
  const kda_bf16 *beta;
  const float *A;
  float gmin;
  const int32_t *cu_seqlens;
  int64_t fixed_len;
  int64_t total;  // tokens of the batch (bounds every cu_seqlens entry)
  int H;
  const float *S0;
  kda_bf16 *o;
  float *S_final;
  float *snaps;
  const int64_t *snap_offsets;
  int *status;
  const int32_t *slots;  // S0 / S_final row of sequence s: slots[s] (state pool), or s
  int n_slots;           // rows of the state pool (slots are checked against it)
  int dk, dv;            // 64 or 128 each (the tiles always hold 128)
  int test_stall;        // KDA_TEST_STALL: give up on an unarmed wait first
  int zero_v;       // 1: treat v as zero (U = 0) and do not read it
  int s0_identity;  // 1: start every chain from S0 = I (dk = dv) instead of S0
  unsigned pre;     // KDA_PRE_* input pre-ops (L2-normalise q, k; sigmoid of beta)
  int n_seq;
};

// Round fp32 to tf32 (nearest, ties away from zero) on the integer ALU: add
// half a unit of the 10-bit mantissa, clear the 13 low bits.  (Values here are
// finite and far below FLT_MAX, so the carry into the exponent is exact.)
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}

// Raw bf16 global load kept where it is written (a prefetch the compiler must
// not sink to its use); the caller widens the bits where it uses them, so the
// load's latency is not waited for here.
__device__ __forceinline__ unsigned short ldg_u16_pinned(const kda_bf16 *ptr) {
  unsigned short raw;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(raw) : "l"(ptr));
  return raw;
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

// Per-step decay exp(gmin * sigmoid(eA * z)) with the base-2 constants folded
// in: c1 = -eA log2(e), c2 = gmin log2(e).  z = +inf gives e^gmin, z = -inf 1.
__device__ __forceinline__ float fast_decay2(float c1, float c2, float z) {
  return ex2_approx(c2 * rcp_approx(1.0f + ex2_approx(c1 * z)));
}

// (a, b) as bf16 pairs hi = bf16(a, b), lo = bf16((a, b) - hi): hi + lo
// carries about 16 mantissa bits.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(a, b);
  const float2 h = unpack_bf16x2(hi);
  lo = pack_bf16x2(a - h.x, b - h.y);
}

// Warp-level D(16x8) += A(16x8) B(8x8) in tf32 with fp32 accumulation.
__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One warp: C[16x16] (two 16x8 fragments) += X[16x16] Y[16x16] with X and Y
// fp32 in shared memory (row strides ldx, ldy floats); with XT, X is given
// transposed (X[g][k] at X[k * ldx + g]), with YT likewise Y.
template <bool XT = false, bool YT = false>
__device__ __forceinline__ void warp_mma16(const float *X, int ldx, const float *Y, int ldy,
                                           float (&c)[2][4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  auto xa = [&](int row, int col) { return XT ? X[col * ldx + row] : X[row * ldx + col]; };
  auto yb = [&](int row, int col) { return YT ? Y[col * ldy + row] : Y[row * ldy + col]; };
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    const int k0 = 8 * ks;
    const uint32_t a[4] = {tf32_rna(xa(g, k0 + t)), tf32_rna(xa(g + 8, k0 + t)),
                           tf32_rna(xa(g, k0 + t + 4)), tf32_rna(xa(g + 8, k0 + t + 4))};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
      mma_m16n8k8_tf32(c[nt], a, tf32_rna(yb(k0 + t, 8 * nt + g)),
                       tf32_rna(yb(k0 + t + 4, 8 * nt + g)));
  }
}

// One CTA per (sequence, head) chain, the whole chunk step, chunks in order.
__global__ void __launch_bounds__(TC_THREADS, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_v,
                  const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const Smem S{smem, sb};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, s = blockIdx.y;
  const int H = p.H;

  if ((sb & 1023u) != 0) {  // the swizzled layouts need 1024-byte alignment
    if (tid == 0) atomicOr(p.status, KDA_ERR_UNSUPPORTED);
    return;
  }

  int64_t t_begin = 0, t_end = 0;
  bool shape_bad = false;  // a device-side index was malformed (KDA_ERR_SHAPE)
  int slot = s;
  if (p.slots) {
    slot = p.slots[s];
    if (slot < 0 || slot >= p.n_slots) {  // nothing of this sequence is touched
      if (tid == 0) atomicOr(p.status, KDA_ERR_SHAPE);
      return;
    }
  }
  if (p.cu_seqlens) {
    if (!seq_range(p.cu_seqlens, s, p.total, t_begin, t_end)) shape_bad = true;
  } else {
    t_begin = static_cast<int64_t>(s) * p.fixed_len;
    t_end = t_begin + p.fixed_len;
  }
  int n_chunks = static_cast<int>((t_end - t_begin + 63) / 64);  // iterations of this CTA
  // Iteration n's chunk: first token and length.
  struct Task {
    int64_t t0;
    int L, h;
  };
  auto task_of = [&](int n) -> Task {
    const int64_t t0 = t_begin + 64LL * n;
    return {t0, static_cast<int>(min(static_cast<int64_t>(64), t_end - t0)), h};
  };
  int64_t snap_row = 0;
  bool want_snaps = p.snaps != nullptr;
  if (want_snaps) {
    snap_row = p.snap_offsets ? snap_first_row(p.snap_offsets, s, p.n_seq, t_end - t_begin)
                              : static_cast<int64_t>(s) * (p.fixed_len / 64);
    if (snap_row < 0) {
      want_snaps = false;
      shape_bad = true;
    }
  }
  const float kLog2e = 1.4426950408889634f;
  const float dc1 = -__expf(p.A[h]) * kLog2e;
  const float dc2 = p.gmin * kLog2e;
  const int DK = p.dk, DV = p.dv;
  const size_t state_off = (static_cast<size_t>(slot) * H + h) * DK * DV;

  const uint32_t bar_qz0 = sb + MS_BAR_QZ, bar_k = sb + MS_BAR_K, bar_v = sb + MS_BAR_V,
                 bar_mma = sb + MS_BAR_MMA;
  if (tid == 0) {
    mbar_init(bar_qz0, 1);
    mbar_init(bar_qz0 + 8, 1);
    mbar_init(bar_k, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_z);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(sb + MS_TMEM, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + MS_TMEM);

  // TMEM read-outs: a warp reaches the 32 lanes of its quadrant; the 16 warps
  // split the columns in quarters.
  const int quad = warp & 3, q4 = warp >> 2;
  const int trow = quad * 32 + lane;  // TMEM lane = matrix row
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);

  // Test hook: a wait that nothing arms gives up before anything is issued.
  bool aborted = false;
  if (p.test_stall) {
    const bool ok = mbar_wait_bounded(bar_mma, 0, 1u << 10);
    if (__syncthreads_or(ok ? 0 : 1)) {
      if (tid == 0) atomicOr(p.status, KDA_ERR_TIMEOUT);
      aborted = true;
      n_chunks = 0;
    }
  }

  // Initial state -> TMEM (row trow, columns [32 q4, 32 q4 + 32)); rows and
  // columns beyond dk, dv are zero.
  const bool row_in = trow < DK, cols_in = 32 * q4 < DV;
  {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      v[j] = p.s0_identity ? (trow == 32 * q4 + j ? 1.f : 0.f)
             : (p.S0 && row_in && cols_in)
                 ? p.S0[state_off + static_cast<size_t>(trow) * DV + 32 * q4 + j]
                 : 0.f;
    tmem_st32(t_lane + TM_S + 32 * q4, v);
    tmem_wait_st();
  }

  auto issue_qz = [&](int n) {  // q -> A3[n&1] lower half, z -> ZB[n&1]
    const int par = n & 1;
    const Task tk = task_of(n);
    const int t0 = static_cast<int>(tk.t0), h = tk.h;
    const uint32_t bar = bar_qz0 + 8 * par;
    mbar_expect_tx(bar, 2 * TILE_BYTES);
    const uint32_t a3 = sb + SM_A3 + par * A3_BYTES;
    tma_load_3d(a3 + 64 * 128, &tm_q, 0, h, t0, bar);
    tma_load_3d(a3 + REG128 + 64 * 128, &tm_q, 64, h, t0, bar);
    const uint32_t zb = sb + SM_ZB + par * TILE_BYTES;
    tma_load_3d(zb, &tm_z, 0, h, t0, bar);
    tma_load_3d(zb + REG64, &tm_z, 64, h, t0, bar);
  };
  // k is refilled as soon as the operand build has read it (K~ goes to A3),
  // v once T'V is done; each has its own barrier.
  auto issue_k = [&](int n) {
    const Task tk = task_of(n);
    const int t0 = static_cast<int>(tk.t0), h = tk.h;
    mbar_expect_tx(bar_k, TILE_BYTES);
    tma_load_3d(sb + SM_KB, &tm_k, 0, h, t0, bar_k);
    tma_load_3d(sb + SM_KB + REG64, &tm_k, 64, h, t0, bar_k);
  };
  auto issue_v = [&](int n) {
    const Task tk = task_of(n);
    const int t0 = static_cast<int>(tk.t0), h = tk.h;
    mbar_expect_tx(bar_v, TILE_BYTES);
    tma_load_3d(sb + SM_VB, &tm_v, 0, h, t0, bar_v);
    tma_load_3d(sb + SM_VB + REG64, &tm_v, 64, h, t0, bar_v);
  };

  // bit b: a q / z load into parity b is in flight (a bit mask, not an array
  // indexed by the parity, which would live in local memory)
  uint32_t qz_pending = 0;
  bool k_pending = false, v_pending = false, mma_pending = false;
  unsigned short beta_raw = 0;  // bf16 bits of this thread's beta, one chunk ahead
  if (tid < 64 && n_chunks > 0) {
    const Task tk = task_of(0);
    if (tid < tk.L) beta_raw = p.beta[static_cast<size_t>(tk.t0 + tid) * H + tk.h];
  }
  // A full chunk's snapshot is written from the next chunk's state read-out
  // (or after the last chunk): the row it goes to, or -1.
  int64_t snap_pending = -1;
  uint32_t mma_phase = 0;
  float range_max = 0.f;  // largest magnitude sent through an fp16 operand

  // Wait helper: every thread polls; the CTA agrees on the outcome.
  auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait_bounded(bar, parity, kWaitPolls);
    const int bad = __syncthreads_or(ok ? 0 : 1);
    if (bad) {
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

  if (tid == kTmaThread && n_chunks > 0) {
    issue_qz(0);
    issue_k(0);
    if (!p.zero_v) issue_v(0);
  }
  qz_pending = n_chunks > 0 ? 1u : 0u;
  k_pending = (n_chunks > 0);
  v_pending = n_chunks > 0 && !p.zero_v;

  // Element-phase mapping: channel pair cp (channels c0, c0 + 1), sub-tile R,
  // and half hf of the sub-tile's rows.  Thread rows, in order, are
  //   r(j) = 16 R + 4 hf + (j & 3) + 8 (j >> 2),  j = 0..7,
  // i.e. the two 4-row segments hf and 2 + hf of the sub-tile; the partner
  // holding the other two segments is lane ^ 16.  A row's swizzle phase is
  // 4 hf + (j & 3), so the two half-warps touch disjoint banks.
  const int hf = lane >> 4;
  const int cp = (warp & 3) * 16 + (lane & 15), R = warp >> 2;
  const int c0 = 2 * cp;
  uint32_t sw16[4], sw32[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int ph = 4 * hf + t;
    sw16[t] = (static_cast<uint32_t>(((c0 >> 3) & 7) ^ ph) << 4) + static_cast<uint32_t>(c0 & 7) * 2u;
    sw32[t] = (static_cast<uint32_t>(((c0 >> 2) & 7) ^ ph) << 4) + static_cast<uint32_t>(c0 & 3) * 4u;
  }
  const uint32_t rg16_64 = static_cast<uint32_t>(c0 >> 6) * REG64;    // 64-row 2-byte tiles
  const uint32_t rg16_128 = static_cast<uint32_t>(c0 >> 6) * REG128;  // 128-row 2-byte tiles
  const uint32_t rg32_a = static_cast<uint32_t>(c0 >> 5) * APA_REG;   // tf32 APA
  const uint32_t rg32_b = static_cast<uint32_t>(c0 >> 5) * APB_REG;   // tf32 APB
  const int rbase = 16 * R + 4 * hf;
  for (int n = 0; n < n_chunks && !aborted; ++n) {
    const int par = n & 1;
    const Task tk = task_of(n);
    const int64_t t0 = tk.t0;
    const int L = tk.L;
    const uint32_t a3 = sb + SM_A3 + par * A3_BYTES;
    const uint32_t zb = sb + SM_ZB + par * TILE_BYTES;

    // Prefetch the next chunk's q and z into the other parity buffers.  (The
    // threads that last wrote those buffers fenced their generic-proxy
    // writes before the barrier that ended the previous chunk.)
    if (tid == kTmaThread && n + 1 < n_chunks) issue_qz(n + 1);
    if (n + 1 < n_chunks) qz_pending |= 1u << (par ^ 1);
    // beta of this chunk was loaded one chunk ahead (logits pass through a sigmoid)
    if (tid < 64) {
      const float bn = __uint_as_float(static_cast<uint32_t>(beta_raw) << 16);
      const float b = (p.pre & KDA_PRE_SIGMOID_BETA) ? 1.0f / (1.0f + __expf(-bn)) : bn;
      S.f32(sb + MS_BETA + 4 * tid) = tid < L ? b : 0.f;
    }
    if (!wait_all(bar_qz0 + 8 * par, (n >> 1) & 1)) { aborted = true; break; }
    qz_pending &= ~(1u << par);

    // ---- element phase A: decay factors and their running products ---------------------
    float ef0[8], ef1[8], eb0[8], eb1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = rbase + (j & 3) + 8 * (j >> 2);
      if (r < L) {
        const float2 zz =
            unpack_bf16x2(S.u32(zb + rg16_64 + static_cast<uint32_t>(r) * 128u + sw16[j & 3]));
        ef0[j] = fast_decay2(dc1, dc2, zz.x);
        ef1[j] = fast_decay2(dc1, dc2, zz.y);
      } else {
        ef0[j] = 1.f;
        ef1[j] = 1.f;
      }
    }
    // segment-local backward products (rows after j inside its 4-row segment)
#pragma unroll
    for (int sg = 0; sg < 2; ++sg) {
      eb0[4 * sg + 3] = 1.f;
      eb1[4 * sg + 3] = 1.f;
#pragma unroll
      for (int j = 2; j >= 0; --j) {
        eb0[4 * sg + j] = eb0[4 * sg + j + 1] * ef0[4 * sg + j + 1];
        eb1[4 * sg + j] = eb1[4 * sg + j + 1] * ef1[4 * sg + j + 1];
      }
#pragma unroll
      for (int j = 1; j < 4; ++j) {
        ef0[4 * sg + j] *= ef0[4 * sg + j - 1];
        ef1[4 * sg + j] *= ef1[4 * sg + j - 1];
      }
    }
    {
      // Segment totals of the whole sub-tile: T_hf, T_2+hf here, the others at lane ^ 16.
      const float ta0 = ef0[3], tb0 = ef0[7], ta1 = ef1[3], tb1 = ef1[7];
      const float pa0 = __shfl_xor_sync(0xffffffffu, ta0, 16);
      const float pb0 = __shfl_xor_sync(0xffffffffu, tb0, 16);
      const float pa1 = __shfl_xor_sync(0xffffffffu, ta1, 16);
      const float pb1 = __shfl_xor_sync(0xffffffffu, tb1, 16);
      // segments in row order: s0 = (hf0, A), s1 = (hf1, A), s2 = (hf0, B), s3 = (hf1, B)
      const float s00 = hf ? pa0 : ta0, s10 = hf ? ta0 : pa0, s20 = hf ? pb0 : tb0, s30 = hf ? tb0 : pb0;
      const float s01 = hf ? pa1 : ta1, s11 = hf ? ta1 : pa1, s21 = hf ? pb1 : tb1, s31 = hf ? tb1 : pb1;
      // prefix before and suffix after each of this thread's segments
      const float preA0 = hf ? s00 : 1.f, preB0 = hf ? s00 * s10 * s20 : s00 * s10;
      const float preA1 = hf ? s01 : 1.f, preB1 = hf ? s01 * s11 * s21 : s01 * s11;
      const float sufA0 = hf ? s20 * s30 : s10 * s20 * s30, sufB0 = hf ? 1.f : s30;
      const float sufA1 = hf ? s21 * s31 : s11 * s21 * s31, sufB1 = hf ? 1.f : s31;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ef0[j] *= preA0;
        ef1[j] *= preA1;
        eb0[j] *= sufA0;
        eb1[j] *= sufA1;
        ef0[4 + j] *= preB0;
        ef1[4 + j] *= preB1;
        eb0[4 + j] *= sufB0;
        eb1[4 + j] *= sufB1;
      }
      if (hf == 0) {
        S.f32(sb + MS_LAM + 4 * (R * TD + c0)) = s00 * s10 * s20 * s30;
        S.f32(sb + MS_LAM + 4 * (R * TD + c0 + 1)) = s01 * s11 * s21 * s31;
      }
    }
    // the next chunk's beta, issued while the store queue is quiet
    if (tid < 64) {
      beta_raw = 0;
      if (n + 1 < n_chunks) {
        const Task nx = task_of(n + 1);
        if (tid < nx.L)
          beta_raw = ldg_u16_pinned(p.beta + static_cast<size_t>(nx.t0 + tid) * H + nx.h);
      }
    }
    if (!wait_all(bar_k, n & 1)) { aborted = true; break; }  // also orders the Lam table
    k_pending = false;
    if (L < 64) {
      // A partial chunk: rows L..63 of k and q hold other tokens (or the TMA
      // fill); zero them once, so that the operand passes need no per-row test.
      // A row is 2 x 128 bytes in each tile (two 64-channel regions).
      for (int x = tid; x < (64 - L) * 32; x += TC_THREADS) {
        const int r = L + (x >> 5), c = x & 31;
        const uint32_t reg = static_cast<uint32_t>((c >> 3) & 1), ch = static_cast<uint32_t>(c & 7);
        const uint32_t addr =
            c < 16 ? sb + SM_KB + reg * REG64 + static_cast<uint32_t>(r) * 128u + ch * 16u
                   : a3 + reg * REG128 + static_cast<uint32_t>(64 + r) * 128u + ch * 16u;
        S.u128(addr) = make_uint4(0, 0, 0, 0);
      }
      __syncthreads();
    }

    const bool l2n = (p.pre & KDA_PRE_L2NORM_QK) != 0;
    if (l2n) {
      // Raw q and k: 1 / ||k_r||, 1 / ||q_r|| of every row (fp32) into MS_NRM;
      // phase B multiplies them in, so the normalised rows are never rounded
      // back to bf16 (their rounding alone moves the outputs by ~2.4e-2 RMS).
      // Sums of squares: this thread's two channels, its half-warp (16
      // channel pairs), then the 4 warps of the sub-tile through a table in
      // the other parity's A3 rows 0..15, which hold nothing during this chunk.
      const uint32_t tab = sb + SM_A3 + (par ^ 1) * A3_BYTES;  // [64 rows][4 warps][k, q]
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = rbase + (j & 3) + 8 * (j >> 2);
        const uint32_t o16 = static_cast<uint32_t>(r) * 128u + sw16[j & 3];
        const float2 kk = unpack_bf16x2(S.u32(sb + SM_KB + rg16_64 + o16));
        const float2 qq = unpack_bf16x2(S.u32(a3 + rg16_128 + 64 * 128 + o16));
        float sk = kk.x * kk.x + kk.y * kk.y, sq = qq.x * qq.x + qq.y * qq.y;
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) {
          sk += __shfl_xor_sync(0xffffffffu, sk, off);
          sq += __shfl_xor_sync(0xffffffffu, sq, off);
        }
        if ((lane & 15) == 0)
          S.u64(tab + static_cast<uint32_t>(r * 4 + (warp & 3)) * 8u) =
              make_uint2(__float_as_uint(sk), __float_as_uint(sq));
      }
      __syncthreads();
      if (tid < 64) {
        float tk = 0.f, tq = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint2 e = S.u64(tab + static_cast<uint32_t>(tid * 4 + w) * 8u);
          tk += __uint_as_float(e.x);
          tq += __uint_as_float(e.y);
        }
        S.u64(sb + MS_NRM + 8 * tid) = make_uint2(__float_as_uint(tk > 0.f ? rsqrtf(tk) : 0.f),
                                                 __float_as_uint(tq > 0.f ? rsqrtf(tq) : 0.f));
      }
      __syncthreads();
    }

    // ---- element phase B: scaled operands, one row-block pair at a time -----------------
    // Pass pp builds the tf32 operands of sub-tiles {2pp, 2pp+1} and runs their
    // M128 x N64 x K128 MMA; the second pass also rewrites k, q, z in place.
    // The tf32 operands are rounded to nearest (truncation would bias the
    // 128-term sums).
    {
      float l0[4], l1[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        l0[m] = S.f32(sb + MS_LAM + 4 * (m * TD + c0));
        l1[m] = S.f32(sb + MS_LAM + 4 * (m * TD + c0 + 1));
      }
      float x0 = 1.f, x1 = 1.f, y0 = 1.f, y1 = 1.f;  // prod_{M<R} Lam, prod_{M>R} Lam
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if (m < R) { x0 *= l0[m]; x1 *= l1[m]; }
        if (m > R) { y0 *= l0[m]; y1 *= l1[m]; }
      }
      // column factors of Khat_{R'} for R' >= R (this thread's rows are sub-tile
      // R), as scalars: an array indexed by the pass would live in local memory
      auto colf = [&](int rp, const float (&l)[4]) {
        float a = 1.f;
#pragma unroll
        for (int m = 0; m < 4; ++m)
          if (m > R && m < rp) a *= l[m];
        const float lr = R == 0 ? l[0] : R == 1 ? l[1] : R == 2 ? l[2] : l[3];
        return (rp == R) ? rcp_approx(lr) : a;
      };
      const float f0_0 = colf(0, l0), f0_1 = colf(1, l0), f0_2 = colf(2, l0), f0_3 = colf(3, l0);
      const float f1_0 = colf(0, l1), f1_1 = colf(1, l1), f1_2 = colf(2, l1), f1_3 = colf(3, l1);
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if (2 * pp + 1 >= R) {
          // column factors of the two Khat blocks of this pass
          const float fa0 = pp ? f0_2 : f0_0, fa1 = pp ? f1_2 : f1_0;
          const float fb0 = pp ? f0_3 : f0_1, fb1 = pp ? f1_3 : f1_1;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = rbase + (j & 3) + 8 * (j >> 2);
            const uint32_t ro = static_cast<uint32_t>(r) * 128u;
            const uint32_t o16 = ro + sw16[j & 3];
            const uint32_t o32 = ro + sw32[j & 3];
            const uint32_t a_kb = sb + SM_KB + rg16_64 + o16;
            const uint32_t a_q = a3 + rg16_128 + 64 * 128 + o16;
            const uint32_t a_z = zb + rg16_64 + o16;
            float2 kk = unpack_bf16x2(S.u32(a_kb));
            float2 qq = unpack_bf16x2(S.u32(a_q));
            if (l2n) {
              const uint2 nr = S.u64(sb + MS_NRM + 8 * r);
              kk.x *= __uint_as_float(nr.x);
              kk.y *= __uint_as_float(nr.x);
              qq.x *= __uint_as_float(nr.y);
              qq.y *= __uint_as_float(nr.y);
            }
            const float ke0 = kk.x * ef0[j], ke1 = kk.y * ef1[j];
            const float qe0 = qq.x * ef0[j], qe1 = qq.y * ef1[j];
            const float kb0 = kk.x * eb0[j], kb1 = kk.y * eb1[j];
            if ((R >> 1) == pp) {
              // rows 32 lb + (r - 16R) (KE) and +16 (QE), lb = R - 2pp:
              // byte offset r * 128 + 2048 R - 8192 pp, same swizzle phase as r
              const uint32_t ab = sb + SM_APB + rg32_b + o32 + 2048u * R - 8192u * pp;
              S.u64(ab) = make_uint2(tf32_rna(ke0), tf32_rna(ke1));
              S.u64(ab + 16 * 128) = make_uint2(tf32_rna(qe0), tf32_rna(qe1));
            }
            if (2 * pp >= R)
              S.u64(sb + SM_APA + rg32_a + o32) = make_uint2(tf32_rna(kb0 * fa0), tf32_rna(kb1 * fa1));
            S.u64(sb + SM_APA + rg32_a + 64 * 128 + o32) =
                make_uint2(tf32_rna(kb0 * fb0), tf32_rna(kb1 * fb1));
            if (pp == 1) {
              // K~ into A3 rows 0..63 (free until -Wk), so k can be refilled now;
              // -Q~ over q, K' over z
              S.u32(a3 + rg16_128 + o16) = pack_bf16x2(ke0 * x0, ke1 * x1);
              S.u32(a_q) = pack_f16x2(-qe0 * x0, -qe1 * x1);
              S.u32(a_z) = pack_f16x2(kb0 * y0, kb1 * y1);
            }
          }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
          tc_fence_after();
          issue_mma(tmem + TM_AP + 64 * pp, sb + SM_APA, false, APA_REG, sb + SM_APB, false,
                    APB_REG, 16, ID_AP, 0, true);
          mma_commit(bar_mma);
        }
        if (pp == 1) {  // every read of k is done: the next chunk's k
          if (tid == kTmaThread && n + 1 < n_chunks) issue_k(n + 1);
          if (n + 1 < n_chunks) k_pending = true;
        }
        mma_pending = true;
        if (!wait_mma()) break;
      }
      if (mma_pending) { aborted = true; break; }
    }

    // Zero what the T blocks do not write: the upper triangles of the T' hi /
    // lo tiles (in the single pass also their rows 64..127, as U's rows
    // 64..127 start -O).  The read-out below writes all of -P itself, zeros
    // included, and the first block X of [X ; -P] only feeds D1 rows that
    // are never read after M5; so no barrier is needed before it.
    for (int x = tid; x < 1024; x += TC_THREADS) {
      S.u128(sb + SM_TP + 16 * x) = make_uint4(0, 0, 0, 0);
      S.u128(sb + SM_TPL + 16 * x) = make_uint4(0, 0, 0, 0);
    }
    {
      // Pair q4 >> 1 of the products: lanes < 64 (rows i of Khat_2pair) hold
      // columns [0, 32), lanes >= 64 (Khat_2pair+1) columns [32, 64); the
      // first 16 of them are A_kk / beta, the next 16 P.  q4 & 1 picks which.
      const int pair = q4 >> 1, sub = q4 & 1;
      float v[16];
      tmem_ld16(t_lane + TM_AP + 64 * pair + (quad >= 2 ? 32 : 0) + 16 * sub, v);
      tmem_wait_ld();
      const int i = trow & 63;
      const int Rb = 2 * pair + (quad >= 2 ? 1 : 0);  // sub-tile of the rows r
      if (sub == 0 && i < 16 * Rb + 16) {
        {
          // A_kk[r][i] = beta_r D[i][r] into row i of the transposed tile (the
          // entries with i >= r are never read)
          const uint32_t row = sb + SM_AKK + 4u * static_cast<uint32_t>(i * 68 + 16 * Rb);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 b = *reinterpret_cast<const float4 *>(
                S.ptr(sb + MS_BETA + 4 * (16 * Rb + 4 * j)));
            S.u128(row + 16 * j) = make_uint4(
                __float_as_uint(b.x * v[4 * j]), __float_as_uint(b.y * v[4 * j + 1]),
                __float_as_uint(b.z * v[4 * j + 2]), __float_as_uint(b.w * v[4 * j + 3]));
          }
        }
      } else if (sub == 1) {
        {
          // -P[r][i] (zero above the diagonal) into K-row i of the MN-major
          // [X ; -P] tile: the r's of -P are the second 64-element MN block;
          // every (i, 16 r's) is written by exactly one thread
          float pv[16];
#pragma unroll
          for (int nn = 0; nn < 16; ++nn) pv[nn] = (i <= 16 * Rb + nn) ? -v[nn] : 0.f;
          const uint32_t row = sb + SM_A5 + REG64 + static_cast<uint32_t>(i) * 128u;
#pragma unroll
          for (int c = 0; c < 2; ++c)
            S.u128(row + (static_cast<uint32_t>((2 * Rb + c) ^ (i & 7)) << 4)) =
                make_uint4(pack_f16x2(pv[8 * c], pv[8 * c + 1]),
                           pack_f16x2(pv[8 * c + 2], pv[8 * c + 3]),
                           pack_f16x2(pv[8 * c + 4], pv[8 * c + 5]),
                           pack_f16x2(pv[8 * c + 6], pv[8 * c + 7]));
        }
      }
    }
    __syncthreads();

    // ---- T = (I + A_kk)^{-1}: diagonal 16x16 blocks, then off-diagonal by distance ------
    // T' hi / lo at byte offset `off` of the [128 x 64] tiles (row r < 64, see SM_TP).
    auto put_tp16 = [&](uint32_t off, unsigned short hi, unsigned short lo) {
      S.u16(sb + SM_TP + off) = hi;
      S.u16(sb + SM_TPL + off) = lo;
    };
    auto put_tp32 = [&](uint32_t off, uint32_t hi, uint32_t lo) {
      S.u32(sb + SM_TP + off) = hi;
      S.u32(sb + SM_TPL + off) = lo;
    };
    {
      // Column jc of the inverse of diagonal block Rd by column updates (once
      // x[m] is final, subtract A[r][m] x[m] from every later row r): eight
      // lanes per column, each holding rows rq and rq + 8; x[m] is passed
      // along by shuffle.  Every CTA thread takes part (64 columns x 8 lanes).
      const int Rd = warp >> 2, jc = 4 * (warp & 3) + (lane >> 3), rq = lane & 7, o = 16 * Rd;
      float a0[7], a1[15];  // A[rq][m] (m < rq), A[rq + 8][m] (m < rq + 8), zero elsewhere
#pragma unroll
      for (int m = 0; m < 15; ++m) {
        const float e1 = S.f32(sb + SM_AKK + 4 * ((o + m) * 68 + o + rq + 8));
        a1[m] = (m < rq + 8) ? e1 : 0.f;
        if (m < 7) {
          const float e0 = S.f32(sb + SM_AKK + 4 * ((o + m) * 68 + o + rq));
          a0[m] = (m < rq) ? e0 : 0.f;
        }
      }
      float x0 = (rq == jc) ? 1.f : 0.f, x1 = (rq + 8 == jc) ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 15; ++m) {
        const float xm = __shfl_sync(0xffffffffu, m < 8 ? x0 : x1, m & 7, 8);
        if (m < 7) x0 -= a0[m] * xm;
        x1 -= a1[m] * xm;
      }
      const float bj = S.f32(sb + MS_BETA + 4 * (o + jc));
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = rq + 8 * hr;
        const float xr = hr ? x1 : x0;
        S.f32(sb + SM_TF + 4 * ((o + r) * 65 + o + jc)) = xr;
        if (r >= jc) {  // T' = T diag(beta) as bf16 hi + lo (the upper triangle stays zero)
          const float tv = xr * bj;
          const __nv_bfloat16 hi = __float2bfloat16_rn(tv);
          const __nv_bfloat16 lo = __float2bfloat16_rn(tv - __bfloat162float(hi));
          put_tp16(sw128_off(o + r, o + jc, REG128), *reinterpret_cast<const unsigned short *>(&hi),
                   *reinterpret_cast<const unsigned short *>(&lo));
        }
      }
    }
    __syncthreads();
    // Off-diagonal blocks.  With D = blockdiag(T_RR) (the diagonal inverses
    // above) and E = D A_off (E_RJ = T_RR A_RJ, strictly block-lower, E^4 = 0):
    //   I + A_kk = D^-1 (I + E),  T = (I - E + E^2 - E^3) D,
    // so with N = I - E + E^2 - E^3, block by block
    //   N_10 = -E_10, N_21 = -E_21, N_32 = -E_32,
    //   N_20 = E_21 E_10 - E_20,  N_31 = E_32 E_21 - E_31,
    //   N_30 = E_31 E_10 - E_30 - E_32 N_20,      and  T_RJ = N_RJ T_JJ.
    // Four levels of single 16 x 16 products on up to six warps.  Only the
    // diagonal T blocks are read again, so the off-diagonal ones go straight
    // to T' (bf16 hi + lo).
    {
      const int g = lane >> 2, t = lane & 3;
      const float *akk = reinterpret_cast<const float *>(S.ptr(sb + SM_AKK));
      const float *tf = reinterpret_cast<const float *>(S.ptr(sb + SM_TF));
      float *xs = reinterpret_cast<float *>(S.ptr(sb + SM_TY));  // 10 blocks of [16][17]
      // block slots: E_10, E_20, E_21, E_30, E_31, E_32, N_20, N_31, E_31 E_10, N_30
      auto blk = [&](int i) { return xs + i * 16 * 17; };
      auto tdiag = [&](int R) { return tf + R * (16 * 65 + 16); };  // T_RR
      // c (two 16x8 fragments) -> fp32 [16][17] block, minus the block `sub` if given
      auto put16 = [&](float *dst, const float (&c)[2][4], const float *sub) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int o = (g + 8 * h) * 17 + 8 * nt + 2 * t;
            dst[o] = c[nt][2 * h] - (sub ? sub[o] : 0.f);
            dst[o + 1] = c[nt][2 * h + 1] - (sub ? sub[o + 1] : 0.f);
          }
        }
      };
      // T_RJ = sgn c as T' = T diag(beta) in bf16 hi + lo
      auto put_t = [&](int R, int J, const float (&c)[2][4], float sgn) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int col = 16 * J + 8 * nt + 2 * t;
          const float b0 = sgn * S.f32(sb + MS_BETA + 4 * col);
          const float b1 = sgn * S.f32(sb + MS_BETA + 4 * (col + 1));
          uint32_t hi, lo;
          split_bf16x2(c[nt][0] * b0, c[nt][1] * b1, hi, lo);
          put_tp32(sw128_off(16 * R + g, col, REG128), hi, lo);
          split_bf16x2(c[nt][2] * b0, c[nt][3] * b1, hi, lo);
          put_tp32(sw128_off(16 * R + g + 8, col, REG128), hi, lo);
        }
      };
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (warp < 6) {  // level 1: E_RJ = T_RR A_RJ (A_kk is stored transposed)
        const int R = warp == 0 ? 1 : warp < 3 ? 2 : 3;
        const int J = warp == 0 ? 0 : warp < 3 ? warp - 1 : warp - 3;
        warp_mma16<false, true>(tdiag(R), 65, akk + (16 * J) * 68 + 16 * R, 68, c, lane);
        put16(blk(warp), c, nullptr);
      }
      __syncthreads();
      if (warp < 6) {  // level 2
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e >> 1][e & 1] = c[e >> 1][2 + (e & 1)] = 0.f;
        switch (warp) {
          case 0: warp_mma16(blk(0), 17, tdiag(0), 65, c, lane); put_t(1, 0, c, -1.f); break;
          case 1: warp_mma16(blk(2), 17, tdiag(1), 65, c, lane); put_t(2, 1, c, -1.f); break;
          case 2: warp_mma16(blk(5), 17, tdiag(2), 65, c, lane); put_t(3, 2, c, -1.f); break;
          case 3: warp_mma16(blk(2), 17, blk(0), 17, c, lane); put16(blk(6), c, blk(1)); break;
          case 4: warp_mma16(blk(5), 17, blk(2), 17, c, lane); put16(blk(7), c, blk(4)); break;
          default: warp_mma16(blk(4), 17, blk(0), 17, c, lane); put16(blk(8), c, nullptr); break;
        }
      }
      __syncthreads();
      if (warp < 3) {  // level 3
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e >> 1][e & 1] = c[e >> 1][2 + (e & 1)] = 0.f;
        switch (warp) {
          case 0: warp_mma16(blk(6), 17, tdiag(0), 65, c, lane); put_t(2, 0, c, 1.f); break;
          case 1: warp_mma16(blk(7), 17, tdiag(1), 65, c, lane); put_t(3, 1, c, 1.f); break;
          default:
            // N_30 = (E_31 E_10 - E_30) - E_32 N_20: the product enters with a minus sign
            warp_mma16(blk(5), 17, blk(6), 17, c, lane);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int o = (g + 8 * h) * 17 + 8 * nt + 2 * t;
                blk(9)[o] = (blk(8)[o] - blk(3)[o]) - c[nt][2 * h];
                blk(9)[o + 1] = (blk(8)[o + 1] - blk(3)[o + 1]) - c[nt][2 * h + 1];
              }
            break;
        }
      }
      __syncthreads();
      if (warp == 0) {  // level 4: T_30 = N_30 T_00
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e >> 1][e & 1] = c[e >> 1][2 + (e & 1)] = 0.f;
        warp_mma16(blk(9), 17, tdiag(0), 65, c, lane);
        put_t(3, 0, c, 1.f);
      }
    }
    fence_proxy_async();  // T' was written by the T blocks above
    tc_fence_before();
    {
      // v of this chunk (loaded a chunk ahead) must be in before T'V
      const bool v_ok = p.zero_v || mbar_wait_bounded(bar_v, n & 1, kWaitPolls);
      if (__syncthreads_or(v_ok ? 0 : 1)) {
        if (tid == 0) atomicOr(p.status, KDA_ERR_TIMEOUT);
        aborted = true;
        break;
      }
      v_pending = false;
    }

    // ---- Wk = T' K~ -> TM_AP,  U = T' V -> D1 ---------------------------------------------
    if (tid == 0) {
      tc_fence_after();
      // T'K~ and T'V interleaved K-step by K-step (independent accumulators)
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // T' hi, then T' lo
        const uint32_t tp = h ? sb + SM_TPL : sb + SM_TP;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t acc = (h > 0 || ks > 0) ? 1u : 0u;
          issue_mma_step(tmem + TM_AP, tp, false, REG128, a3, true, REG128, ks, ID_TPROD, acc);
          if (!p.zero_v)
            issue_mma_step(tmem + TM_D1, tp, false, REG128, sb + SM_VB, true, REG64, ks,
                           ID_TPROD, acc);
        }
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!wait_mma()) { aborted = true; break; }
    if (!p.zero_v) {  // the next chunk's v
      if (tid == kTmaThread && n + 1 < n_chunks) issue_v(n + 1);
      if (n + 1 < n_chunks) v_pending = true;
    }


    // -Wk -> A3 rows 0..63;  S (fp32, TMEM) -> fp16 S for the MMA, then S *= e^{G_last}.
    {
      float v[32];
      if (quad < 2) {
        tmem_ld32(t_lane + TM_AP + 32 * q4, v);
        tmem_wait_ld();
        store_row32_f16(S, a3, trow, q4, REG128, v, -1.f);
      }
      tmem_ld32(t_lane + TM_S + 32 * q4, v);
      tmem_wait_ld();
      if (snap_pending >= 0) {
        // The state after the previous (full) chunk.  Each warp stages its
        // 32 x 32 fp32 tile (4 KiB, float4 slots swizzled by row) in the work
        // region, then stores it so that every instruction writes four whole
        // 128-byte rows.  Warps 0..7 use [0, 32 KiB) (not yet the fp16 S),
        // warps 8..15 [64 KiB, 96 KiB) (T' is consumed, W not yet written).
        // A warp whose tile lies beyond dk or dv has nothing to store.
        if (row_in && cols_in) {
          const uint32_t tile = sb + SM_AP + (warp < 8 ? warp : warp + 8) * 4096u;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            S.u128(tile + lane * 128u + (static_cast<uint32_t>(j ^ (lane & 7)) << 4)) =
                make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                           __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
          __syncwarp();
          float *base = p.snaps + (static_cast<size_t>(snap_pending) * H + h) * DK * DV +
                        static_cast<size_t>(quad * 32) * DV + 32 * q4;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + (lane >> 3), c = lane & 7;
            const uint4 w = S.u128(tile + r * 128u + (static_cast<uint32_t>(c ^ (r & 7)) << 4));
            __stcs(reinterpret_cast<float4 *>(base + static_cast<size_t>(r) * DV) + c,
                   make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                               __uint_as_float(w.w)));
          }
        }
        snap_pending = -1;
        __syncthreads();  // staging tiles are read before the fp16 S overwrites them
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) range_max = fmaxf(range_max, fabsf(v[j]));
      store_row32_f16(S, sb + SM_SBF, trow, q4, REG128, v, 1.f);
      float gam = 1.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) gam *= S.f32(sb + MS_LAM + 4 * (m * TD + trow));
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= gam;
      tmem_st32(t_lane + TM_S + 32 * q4, v);
      tmem_wait_st();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- D1 += [-Wk; -Q~] S: W (rows 0..63), -Q~ S (rows 64..127) --------------------------
    if (tid == 0) {
      tc_fence_after();
      // with zero v there is no U: this product initialises D1
      issue_mma(tmem + TM_D1, a3, false, REG128, sb + SM_SBF, true, REG128, 8, ID_KMN,
                p.zero_v ? 0u : 1u);
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!wait_mma()) { aborted = true; break; }
    if (quad < 2) {
      float v[32];
      tmem_ld32(t_lane + TM_D1 + 32 * q4, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) range_max = fmaxf(range_max, fabsf(v[j]));
      store_row32_f16(S, sb + SM_WBF, trow, q4, REG64, v, 1.f);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- S += K'^T W;  D1 += [0; -P] W -------------------------------------------------------
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // the two products interleaved
        issue_mma_step(tmem + TM_S, zb, true, REG64, sb + SM_WBF, true, REG64, ks, ID_MNMN, 1);
        issue_mma_step(tmem + TM_D1, sb + SM_A5, true, REG64, sb + SM_WBF, true, REG64, ks,
                       ID_MNMN, 1);
      }
      mma_commit(bar_mma);
    }
    mma_pending = true;
    if (!wait_mma()) { aborted = true; break; }

    // ---- outputs: o = -D1 rows 64..127; snapshot of the new state ----------------------------
    if (quad >= 2) {
      const int r = trow - 64;
      float v[32];
      tmem_ld32(t_lane + TM_D1 + 32 * q4, v);
      tmem_wait_ld();
      if (r < L && p.o && cols_in) {
        uint4 *dst = reinterpret_cast<uint4 *>(
            p.o + (static_cast<size_t>(t0 + r) * H + h) * DV + 32 * q4);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_uint4(pack_bf16x2(-v[8 * j + 0], -v[8 * j + 1]),
                              pack_bf16x2(-v[8 * j + 2], -v[8 * j + 3]),
                              pack_bf16x2(-v[8 * j + 4], -v[8 * j + 5]),
                              pack_bf16x2(-v[8 * j + 6], -v[8 * j + 7]));
      }
    }
    if (want_snaps && L == 64) snap_pending = snap_row;
    if (L == 64) ++snap_row;
    tc_fence_before();
    __syncthreads();
  }

  if (!aborted && (p.S_final || snap_pending >= 0)) {
    float v[32];
    tmem_ld32(t_lane + TM_S + 32 * q4, v);
    tmem_wait_ld();
    if (p.S_final && row_in && cols_in) {
      float4 *dst = reinterpret_cast<float4 *>(p.S_final + state_off +
                                               static_cast<size_t>(trow) * DV + 32 * q4);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    if (snap_pending >= 0 && row_in && cols_in) {
      float4 *dst = reinterpret_cast<float4 *>(
          p.snaps + (static_cast<size_t>(snap_pending) * H + h) * DK * DV +
          static_cast<size_t>(trow) * DV + 32 * q4);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        __stcs(dst + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
    }
  }

  // Drain anything still in flight (bounded) before TMEM is released.
  if (aborted && tid == 0) {
    if (mma_pending) mbar_wait_bounded(bar_mma, mma_phase, kWaitPolls);
    for (int b = 0; b < 2; ++b)
      if ((qz_pending >> b) & 1u) mbar_wait_bounded(bar_qz0 + 8 * b, 0, kWaitPolls) ||
                             mbar_wait_bounded(bar_qz0 + 8 * b, 1, kWaitPolls);
    if (k_pending) mbar_wait_bounded(bar_k, 0, kWaitPolls) || mbar_wait_bounded(bar_k, 1, kWaitPolls);
    if (v_pending) mbar_wait_bounded(bar_v, 0, kWaitPolls) || mbar_wait_bounded(bar_v, 1, kWaitPolls);
  }
  tc_fence_before();
  if (__syncthreads_or(range_max > 65504.f ? 1 : 0) && tid == 0)
    atomicOr(p.status, KDA_ERR_RANGE);
  if (shape_bad && tid == 0) atomicOr(p.status, KDA_ERR_SHAPE);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
}

// 3-D map over a [total, H, d] bf16 tensor: box = 64 channels x 1 head x 64
// tokens.  With d = 64 the box at channel 64 lies outside the tensor and
// TMA fills it with zeros.
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

bool prefill_tc_supported(int dk, int dv, int64_t total_tokens) {
  return (dk == 64 || dk == TD) && (dv == 64 || dv == TD) && total_tokens > 0 &&
         total_tokens < (1LL << 31);
}

cudaError_t prefill_tc_launch(const kda_bf16 *q, const kda_bf16 *k, const kda_bf16 *v,
                              const kda_bf16 *z, const kda_bf16 *beta, const float *A, float gmin,
                              const int32_t *cu_seqlens, int n_seq, int64_t total_tokens,
                              int64_t fixed_len, int H, int dk, int dv, const float *S0,
                              kda_bf16 *o, float *S_final, float *snaps,
                              const int64_t *snap_offsets, int *status, int zero_v,
                              int s0_identity, const int32_t *slots, int n_slots, unsigned pre,
                              int test_stall, cudaStream_t stream) {
  CUtensorMap mq, mk, mz, mv;
  if (!make_map(&mq, q, total_tokens, H, dk) || !make_map(&mk, k, total_tokens, H, dk) ||
      !make_map(&mz, z, total_tokens, H, dk) ||
      !make_map(&mv, zero_v ? k : v, total_tokens, H, zero_v ? dk : dv))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(TC_SMEM_BYTES));
  if (err != cudaSuccess) return err;
  TcParams prm{beta, A, gmin, cu_seqlens, fixed_len, total_tokens, H, S0, o, S_final, snaps,
               snap_offsets, status, slots, n_slots, dk, dv, test_stall, zero_v, s0_identity,
               pre, n_seq};
  const dim3 grid(static_cast<unsigned>(H), static_cast<unsigned>(n_seq));
  prefill_tc_kernel<<<grid, TC_THREADS, TC_SMEM_BYTES, stream>>>(mq, mk, mz, mv, prm);
  return cudaGetLastError();
}


}  // namespace kda
